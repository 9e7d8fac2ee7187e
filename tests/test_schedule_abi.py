"""CPU tests of the C-ABI library: exported symbols, host scheduler bit-exact
against the oracle's mask-derived tile set, dual-end / zigzag ownership,
argument validation.  No kernel is launched (no GPU needed)."""
import ctypes

import numpy as np
import pytest

from block_diffusion_lm_gb300 import csbp
from block_diffusion_lm_gb300.inputs import WORKLOADS
from oracle import csbp_oracle as O


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_diffusion_lm_gb300 import build
    build.build()


def expand(words, info, P):
    """Work list -> (fwd set, bwd set, fwd costs, bwd costs) of
    (q_stream, q_tile, kv_stream, kv_tile, full, part) tuples."""
    h = words[:16]
    assert h[0] == 0x43534250 and h[1] == 1
    off_ft, off_fs, off_bt, off_bs, total = (int(x) for x in h[11:16])
    assert total == len(words)
    fwd, bwd, fc, bc = set(), set(), [], []
    seen = set()
    for t in range(info.n_fwd_tasks):
        qs, qt, part, sb, sc, cost = (int(x) for x in words[off_ft + 8 * t: off_ft + 8 * t + 6])
        fc.append(cost)
        n = 0
        for s in range(sb, sb + sc):
            ks, b, e, fl = (int(x) for x in words[off_fs + 4 * s: off_fs + 4 * s + 4])
            for kt in range(b, e):
                key = (qs, qt, ks, kt)
                assert key not in seen  # every tile pair appears once
                seen.add(key)
                fwd.add(key + (not (fl & 1), part))
                n += 1
        assert n == cost
    for t in range(info.n_bwd_tasks):
        ks, kt, part, sb, sc, cost = (int(x) for x in words[off_bt + 8 * t: off_bt + 8 * t + 6])
        bc.append(cost)
        n = 0
        for s in range(sb, sb + sc):
            qs, b, e, fl = (int(x) for x in words[off_bs + 4 * s: off_bs + 4 * s + 4])
            for qt in range(b, e):
                bwd.add((qs, qt, ks, kt, not (fl & 1), part))
                n += 1
        assert n == cost
    return fwd, bwd, fc, bc


def fwd_order_keys(words, info):
    """(part, q_tile, q_stream) of every forward task, in list order."""
    off_ft = int(words[11])
    out = []
    for t in range(info.n_fwd_tasks):
        qs, qt, part = (int(x) for x in words[off_ft + 8 * t: off_ft + 8 * t + 3])
        out.append((max(part, 0), qt, qs))
    return out


def assert_fwd_order(words, info, fc, W):
    """Forward tasks are heaviest first; with a sliding window (near-equal
    costs) they run in (part, query tile, copy) order instead, so a CTA's
    two tasks are the clean and corrupted tiles at one position, which read
    the same window of clean key tiles."""
    if W == 0:
        assert fc == sorted(fc, reverse=True)
    else:
        keys = fwd_order_keys(words, info)
        assert keys == sorted(keys)


def test_library_exports_every_declared_symbol():
    L = csbp.lib()
    names = csbp.header_functions()
    assert set(names) >= {"csbp_block_schedule", "csbp_attn_fwd", "csbp_attn_bwd",
                          "csbp_lse_merge"}
    for n in names:
        assert hasattr(L, n), n
    assert L.csbp_version() >= 200
    for code, name in csbp.STATUS.items():
        assert L.csbp_status_string(code)


SWEEP = [
    # L, M, T, P, has_clean
    (256, 16, 32, 1, True), (256, 32, 32, 1, True), (256, 64, 32, 1, True),
    (512, 16, 64, 2, True), (512, 8, 32, 4, True), (480, 16, 32, 1, True),   # ragged tail
    (256, 1, 32, 1, True), (256, 256, 32, 1, True), (256, 16, 32, 1, False),
    (512, 16, 32, 2, False), (200, 8, 32, 1, True), (384, 128, 128, 1, True),
    (1024, 64, 128, 1, True), (1024, 32, 128, 4, True), (1040, 16, 128, 1, True),
]
SWEEP = [s + (0, False) for s in SWEEP] + [
    # L, M, T, P, has_clean, window, token-causal clean
    (256, 16, 32, 1, True, 0, True), (480, 16, 32, 1, True, 0, True),
    (256, 16, 32, 1, True, 40, False), (256, 16, 32, 1, True, 33, True),
    (512, 16, 32, 2, True, 100, False), (512, 8, 32, 4, True, 64, True),
    (480, 32, 32, 1, False, 50, False), (256, 64, 32, 1, True, 1, False),
    (256, 1, 32, 1, True, 17, True), (1040, 16, 128, 1, True, 300, True),
    (1024, 64, 128, 1, True, 128, False), (1024, 32, 128, 4, True, 129, False),
    (384, 128, 128, 1, True, 1000, True),
]


def random_sweep(n, seed):
    """Seeded valid problems: ragged tails (P = 1), P up to 4, unit to
    256-token blocks, any window from one token to wider than the sequence,
    both clean-query modes, drafter shapes."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        T = int(rng.choice([32, 64, 128]))
        M = int(rng.choice([1, 2, 4, 8, 16, 32, 64, 128, 256]))
        P = int(rng.choice([1, 1, 2, 3, 4]))
        B = int(rng.integers(1, 1200 // M + 1))
        L = B * M
        if L < 2 or L > 1200:
            continue
        if P > 1 and (B % (2 * P) != 0 or (L // (2 * P)) % T != 0):
            continue
        W = 0 if rng.random() < 0.3 else int(rng.integers(1, L + 40))
        out.append((L, M, T, P, bool(rng.random() < 0.8), W, bool(rng.random() < 0.5)))
    return out


@pytest.mark.parametrize("L,M,T,P,clean,W,causal", SWEEP + random_sweep(40, 2026))
def test_schedule_matches_oracle_tile_set_bit_exactly(L, M, T, P, clean, W, causal):
    prob = csbp.make_problem(1, L, M, 2, 1, 64, P=P, has_clean_queries=clean, tile=T,
                             window=W, clean_causal=causal)
    bo, co, words, info = csbp.block_schedule(prob)
    fwd, bwd, fc, bc = expand(words, info, P)
    want = O.tile_pairs(L, M, T, T, P, clean, W, causal)
    if P == 1:
        got_fwd = {x[:5] + ((1 if x[2] == 1 else 0),) for x in fwd}
        assert all(x[5] == -1 for x in fwd)
    else:
        got_fwd = fwd
    assert got_fwd == want
    got_bwd = {x for x in bwd}
    if P == 1:
        got_bwd = {x[:5] + ((1 if x[2] == 1 else 0),) for x in bwd}
    assert got_bwd == want
    assert info.tile_pairs == len(want)
    # forward: heaviest first (by position under a window); backward: heaviest first
    assert_fwd_order(words, info, fc, W)
    assert bc == sorted(bc, reverse=True)
    # every key tile of both copies has exactly one backward task
    nT = -(-L // T)
    assert info.n_bwd_tasks == 2 * nT


@pytest.mark.parametrize("L,M,P", [(64, 4, 2), (128, 4, 4), (96, 4, 3), (4096, 32, 8)])
def test_ownership_matches_oracle(L, M, P):
    prob = csbp.make_problem(1, L, M, 1, 1, 64, P=P, tile=16 if L < 4096 else 128)
    if (L // (2 * P)) % prob.tile_kv:
        prob.tile_q = prob.tile_kv = 4
    bo, co, _, _ = csbp.block_schedule(prob)
    np.testing.assert_array_equal(bo, O.block_owner(L, M, P))
    np.testing.assert_array_equal(co, O.chunk_owner(L, P))


@pytest.mark.parametrize("name", ["tiny", "dense14b", "sharded", "long"])
def test_full_size_schedules_closed_form(name):
    """Tile-pair count nT(nT+1)+nT at the workload sizes (M < 128), and equal
    tile counts per clean shard under the zigzag pairing."""
    w = WORKLOADS[name]
    prob = csbp.make_problem(w.batch, w.L, w.M, w.Hq, w.Hkv, w.d, P=w.P,
                             has_clean_queries=w.has_clean_queries)
    _, _, words, info = csbp.block_schedule(prob)
    nT = w.L // 128
    assert info.tile_pairs == nT * (nT + 1) + nT
    if w.P > 1:
        fwd, _, _, _ = expand(words, info, w.P)
        per = np.zeros(w.P + 1, np.int64)
        for x in fwd:
            per[x[5]] += 1
        assert np.all(per[:w.P] == per[0])
        assert per[w.P] == nT


def test_drafter_schedule_count():
    """Corrupted queries only, L = 2^20, M = 16: nT(nT+1)/2 + nT tile pairs
    (clean tiles 0..t plus the own corrupted tile per query tile)."""
    w = WORKLOADS["drafter"]
    prob = csbp.make_problem(1, w.L, w.M, w.Hq, w.Hkv, w.d, has_clean_queries=False)
    info = csbp.ScheduleInfo()
    st = csbp.lib().csbp_block_schedule(ctypes.byref(prob), None, None, None, 0,
                                        ctypes.byref(info))
    assert st == -6  # capacity query
    nT = w.L // 128
    assert info.tile_pairs == nT * (nT + 1) // 2 + nT
    assert info.n_bwd_tasks == 2 * nT
    # with backward windows of 512 query tiles: clean key tile kt is read by
    # query tiles kt .. nT-1, i.e. by ceil((nT - kt) / 512) windows;
    # corrupted key tiles by their own query tile only
    c = 512
    prob.bwd_chunk = c
    st = csbp.lib().csbp_block_schedule(ctypes.byref(prob), None, None, None, 0,
                                        ctypes.byref(info))
    assert st == -6
    assert info.n_bwd_tasks == sum(-(-m // c) for m in range(1, nT + 1)) + nT
    assert info.n_bwd_tasks == c * (nT // c) * (nT // c + 1) // 2 + nT


def test_windowed_full_size_schedule_count():
    """L = 16384, M = 32, window 1024 = 8 key tiles: query tile t of either
    copy touches clean key tiles max(0, t-8) .. t, and corrupted query tiles
    their own corrupted tile as well."""
    w = WORKLOADS["window1k"]
    prob = csbp.make_problem(w.batch, w.L, w.M, w.Hq, w.Hkv, w.d, window=w.window)
    _, _, _, info = csbp.block_schedule(prob)
    nT, wt = w.L // 128, w.window // 128
    per_stream = sum(min(t + 1, wt + 1) for t in range(nT))
    assert info.tile_pairs == 2 * per_stream + nT
    assert info.n_bwd_tasks == 2 * nT


@pytest.mark.parametrize("field,value,code", [
    ("M", 3, -1),            # L % M != 0
    ("Hkv", 3, -1),          # Hq % Hkv != 0
    ("d", 96, -2),           # unsupported head dim
    ("P", 3, -2),            # B % 2P != 0
    ("scale", 0.0, -1),
    ("L", 0, -1),
    ("has_clean_queries", 2, -1),
    ("window", -1, -1),
    ("clean_causal", 2, -1),
])
def test_schedule_rejects_invalid_problems(field, value, code):
    prob = csbp.make_problem(1, 1024, 64, 4, 2, 64)
    setattr(prob, field, value)
    info = csbp.ScheduleInfo()
    st = csbp.lib().csbp_block_schedule(ctypes.byref(prob), None, None, None, 0, ctypes.byref(info))
    assert st == code


def test_workspace_sizes():
    prob = csbp.make_problem(2, 1024, 64, 4, 2, 128, P=4)
    rows = 2 * 1024
    fwd = csbp.workspace_bytes(prob, 0)
    bwd = csbp.workspace_bytes(prob, 1)
    assert fwd >= 256 + 5 * 2 * rows * 4 * 128 * 4 + 5 * 2 * rows * 4 * 4
    assert bwd >= 256 + 2 * rows * 4 * 4 + 2 * rows * 4 * 128 * 4
    prob.d = 96
    assert csbp.workspace_bytes(prob, 0) == 0


def test_entry_points_reject_bad_arguments_without_launching():
    """Null pointers and misalignment are refused before anything is enqueued
    (no CUDA call is made on these paths, so this runs without a GPU)."""
    L = csbp.lib()
    prob = csbp.make_problem(1, 1024, 64, 2, 2, 64)
    info = csbp.ScheduleInfo()
    inp = csbp.Inputs()
    assert L.csbp_attn_fwd(ctypes.byref(prob), ctypes.byref(inp), None, ctypes.byref(info),
                           None, None, None, None, 0, None) == -1
    assert L.csbp_attn_bwd(ctypes.byref(prob), None, None, ctypes.byref(info), *([None] * 12),
                           0, None) == -1
    arr = (ctypes.c_void_p * 1)(None)
    assert L.csbp_lse_merge(0, arr, arr, 16, 2, 64, None, None, None) == -1
    assert L.csbp_lse_merge(1, arr, arr, 16, 2, 64, None, None, None) == -1
    # fp32 LSE pointers must be 4-byte aligned; sizes must stay below 2^39
    # elements (checked without overflow)
    g16 = ctypes.c_void_p(0x10000)
    ok = (ctypes.c_void_p * 1)(0x10000)
    odd = (ctypes.c_void_p * 1)(0x10002)
    assert L.csbp_lse_merge(1, ok, odd, 16, 2, 64, g16, g16, None) == -1
    assert L.csbp_lse_merge(1, ok, ok, 16, 2, 64, g16, ctypes.c_void_p(0x10001), None) == -1
    assert L.csbp_lse_merge(1, ok, ok, 1 << 62, 2, 64, g16, g16, None) == -1
    assert L.csbp_lse_merge(1, ok, ok, 1 << 30, 4, 128, g16, g16, None) == -1
    # misaligned (odd) pointers
    bad = ctypes.c_void_p(0x1001)
    inp = csbp.Inputs(bad, bad, bad, bad, bad, bad)
    assert L.csbp_attn_fwd(ctypes.byref(prob), ctypes.byref(inp), bad, ctypes.byref(info),
                           bad, bad, bad, bad, 1 << 20, None) == -1


def test_input_strides_are_checked_before_launching():
    """Token and batch strides of csbp_inputs: the contiguous default (0) and
    packed-QKV views pass (the call then stops at the too-small workspace,
    before any CUDA call); strides that break the header's rules are refused."""
    L = csbp.lib()
    prob = csbp.make_problem(2, 1024, 64, 4, 2, 64)  # Hq*d = 256, Hkv*d = 128
    info = csbp.ScheduleInfo()
    assert L.csbp_block_schedule(ctypes.byref(prob), None, None, None, 0,
                                 ctypes.byref(info)) == -6  # counts and key only
    g = ctypes.c_void_p(0x10000)

    def fwd(tok, bat):
        inp = csbp.Inputs(g, g, g, g, g, g, (ctypes.c_int64 * 6)(*tok),
                          (ctypes.c_int64 * 6)(*bat))
        return L.csbp_attn_fwd(ctypes.byref(prob), ctypes.byref(inp), g, ctypes.byref(info),
                               g, g, g, g, 16, None)

    def bwd(tok, bat):
        inp = csbp.Inputs(g, g, g, g, g, g, (ctypes.c_int64 * 6)(*tok),
                          (ctypes.c_int64 * 6)(*bat))
        return L.csbp_attn_bwd(ctypes.byref(prob), ctypes.byref(inp), g, ctypes.byref(info),
                               *([g] * 12), 16, None)

    packed = (4 + 2 * 2) * 64  # [L][Hq + 2 Hkv][d]
    zero = [0] * 6
    assert fwd(zero, zero) == -3 and bwd(zero, zero) == -3
    assert fwd([packed] * 6, [1024 * packed] * 6) == -3
    assert bwd([packed] * 6, [1024 * packed + 64] * 6) == -3
    assert fwd([0, 128, 128, 0, 128, 128], zero) == -3  # k/v at their own H*d
    for tok, bat in [
        ([248, 0, 0, 0, 0, 0], zero),              # q token stride below Hq*d
        ([0, 0, 0, 0, 120, 0], zero),              # k token stride below Hkv*d
        ([0, packed + 4, 0, 0, 0, 0], zero),       # not a multiple of 8 elements
        ([0, 0, -8, 0, 0, 0], zero),               # negative
        ([0, 0, 0, 1 << 39, 0, 0], zero),          # past the TMA stride range
        ([0, 0, 0, 0, 1 << 62, 0], zero),          # L x stride would overflow int64
        ([0, 0, 0, 0, 0, (1 << 39) // 1024 + 8], zero),  # one batch entry past 2^39
        ([packed] * 6, [1024 * packed - 8] + [0] * 5),  # batch entries overlap
        (zero, [0, 0, 0, 0, 0, 1024 * 128 + 4]),   # batch stride not a multiple of 8
        (zero, [0, -1024 * 128, 0, 0, 0, 0]),      # negative batch stride
    ]:
        assert fwd(tok, bat) == -1, (tok, bat)
        assert bwd(tok, bat) == -1, (tok, bat)
    # with one batch entry the batch stride is not read (a negative one is
    # still malformed)
    prob.batch = 1
    assert fwd(zero, [8] * 6) == -3
    assert fwd(zero, [-8] + [0] * 5) == -1


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_every_workload_passes_input_validation(name):
    """Every benchmark and test workload, with contiguous and with packed-QKV
    strides, passes the argument checks of both entry points (the calls
    then stop at a deliberately small workspace, before any CUDA call)."""
    w = WORKLOADS[name]
    L = csbp.lib()
    prob = csbp.make_problem(w.batch, w.L, w.M, w.Hq, w.Hkv, w.d, P=w.P,
                             has_clean_queries=w.has_clean_queries, window=w.window,
                             clean_causal=w.clean_causal)
    info = csbp.ScheduleInfo()
    assert L.csbp_block_schedule(ctypes.byref(prob), None, None, None, 0,
                                 ctypes.byref(info)) == -6  # counts and key only
    g = ctypes.c_void_p(0x10000)
    packed = (w.Hq + 2 * w.Hkv) * w.d
    for tok, bat in (([0] * 6, [0] * 6), ([packed] * 6, [w.L * packed] * 6)):
        inp = csbp.Inputs(g, g, g, g, g, g, (ctypes.c_int64 * 6)(*tok),
                          (ctypes.c_int64 * 6)(*bat))
        assert L.csbp_attn_fwd(ctypes.byref(prob), ctypes.byref(inp), g, ctypes.byref(info),
                               g, g, g, g, 16, None) == -3
        assert L.csbp_attn_bwd(ctypes.byref(prob), ctypes.byref(inp), g, ctypes.byref(info),
                               *([g] * 12), 16, None) == -3


@pytest.mark.parametrize("batch,L,Hq,d", [(1, 1 << 30, 1024, 128), (1 << 20, 1 << 20, 8, 64),
                                          ((1 << 31) - 1, (1 << 31) - 1, 8, 128)])
def test_problems_past_2_39_elements_are_unsupported(batch, L, Hq, d):
    """No tensor may reach 2^39 elements (1 TiB of bf16): such problems are
    refused up front, so no element or byte count can overflow int64."""
    prob = csbp.make_problem(batch, L, 1, Hq, Hq, d)
    assert csbp.workspace_bytes(prob, 0) == 0 and csbp.workspace_bytes(prob, 1) == 0
    info = csbp.ScheduleInfo()
    assert csbp.lib().csbp_block_schedule(ctypes.byref(prob), None, None, None, 0,
                                          ctypes.byref(info)) == -2


@pytest.mark.parametrize("field,value", [("L", 2048), ("M", 32), ("P", 1), ("window", 100),
                                         ("clean_causal", 1), ("bwd_chunk", 2),
                                         ("has_clean_queries", 0)])
def test_a_list_built_for_another_problem_is_refused(field, value):
    """The info of a work list carries a fingerprint of the problem fields
    the list depends on; changing any of them makes both entry points refuse
    the list before any CUDA call, while batch, heads and the scale do not
    matter to it."""
    L = csbp.lib()
    prob = csbp.make_problem(2, 1024, 64, 4, 2, 64, P=2)
    _, _, _, info = csbp.block_schedule(prob)
    g = ctypes.c_void_p(0x10000)
    inp = csbp.Inputs(g, g, g, g, g, g)

    def calls(p):
        return (L.csbp_attn_fwd(ctypes.byref(p), ctypes.byref(inp), g, ctypes.byref(info),
                                g, g, g, g, 16, None),
                L.csbp_attn_bwd(ctypes.byref(p), ctypes.byref(inp), g, ctypes.byref(info),
                                *([g] * 12), 16, None))

    assert calls(prob) == (-3, -3)
    other = csbp.make_problem(2, 1024, 64, 4, 2, 64, P=2)
    setattr(other, field, value)
    assert calls(other) == (-1, -1)
    same_list = csbp.make_problem(1, 1024, 64, 8, 1, 128, P=2, scale=0.3)
    assert calls(same_list) == (-3, -3)


def random_windowed_sweep(n, seed):
    """Random problems of `random_sweep` with at least two query tiles and a
    backward window of 1 .. nT - 1 tiles."""
    rng = np.random.default_rng(seed)
    out = []
    for L, M, T, P, clean, W, causal in random_sweep(4 * n, seed):
        nT = -(-L // T)
        if nT >= 2 and len(out) < n:
            out.append((L, M, T, P, clean, W, causal, int(rng.integers(1, nT))))
    return out


@pytest.mark.parametrize("L,M,T,P,clean,W,causal,chunk", [
    (1024, 16, 128, 1, True, 0, False, 2), (1024, 32, 128, 1, False, 0, False, 3),
    (1152, 64, 128, 1, True, 300, True, 1), (512, 16, 32, 1, True, 0, False, 5),
    (1040, 16, 128, 1, True, 0, True, 4),
] + random_windowed_sweep(20, 2027))
def test_windowed_backward_tasks_partition_the_tile_set(L, M, T, P, clean, W, causal, chunk):
    """With a query-tile window smaller than the tile count, every backward
    task covers one window (counted from the last query tile), flags its
    dK/dV for fp32 accumulation, and the tasks together hold every allowed
    (query tile, key tile) pair exactly once; windows run in order, heaviest
    first within a window."""
    prob = csbp.make_problem(1, L, M, 2, 1, 64, P=P, has_clean_queries=clean, tile=T,
                             window=W, clean_causal=causal, bwd_chunk=chunk)
    _, _, words, info = csbp.block_schedule(prob)
    h = words[:16]
    off_bt, off_bs = int(h[13]), int(h[14])
    nT = -(-L // T)
    want = {x[:4] for x in O.tile_pairs(L, M, T, T, P, clean, W, causal)}
    seen = []
    order = []
    for t in range(info.n_bwd_tasks):
        ks, kt, part, sb, sc, cost, flags, win = (int(x) for x in
                                                  words[off_bt + 8 * t: off_bt + 8 * t + 8])
        assert flags == 1
        lo, hi = max(0, nT - (win + 1) * chunk), nT - win * chunk
        n = 0
        for s in range(sb, sb + sc):
            qs, b, e, fl = (int(x) for x in words[off_bs + 4 * s: off_bs + 4 * s + 4])
            assert lo <= b < e <= hi
            for qt in range(b, e):
                seen.append((qs, qt, ks, kt))
                n += 1
        assert n == cost
        order.append((win, -cost))
    assert len(seen) == len(set(seen))
    assert set(seen) == want
    assert order == sorted(order)


def test_backward_is_not_windowed_below_the_window():
    """Up to `bwd_chunk` query tiles per key tile the list keeps one task per
    key tile, with bf16 dK/dV written directly (flags 0)."""
    prob = csbp.make_problem(1, 1024, 16, 2, 1, 64, bwd_chunk=8)
    _, _, words, info = csbp.block_schedule(prob)
    off_bt = int(words[13])
    assert info.n_bwd_tasks == 2 * 8
    assert all(int(words[off_bt + 8 * t + 6]) == 0 for t in range(info.n_bwd_tasks))
    prob.bwd_chunk = -1
    assert csbp.workspace_bytes(prob, 1) == 0


def test_wait_selftest_refuses_bad_arguments_without_launching():
    L = csbp.lib()
    good = ctypes.c_void_p(0x10000)
    assert L.csbp_wait_selftest(1_000_000, None, None) == -1          # no workspace
    assert L.csbp_wait_selftest(1_000_000, ctypes.c_void_p(0x10008), None) == -1  # misaligned
    assert L.csbp_wait_selftest(10, good, None) == -1                 # budget too short
    assert L.csbp_wait_selftest(3_000_000_000, good, None) == -1      # budget too long


def test_entry_points_refuse_a_small_workspace_without_launching():
    L = csbp.lib()
    prob = csbp.make_problem(1, 1024, 64, 2, 2, 64, P=2)
    _, _, _, info = csbp.block_schedule(prob)
    g = ctypes.c_void_p(0x10000)
    inp = csbp.Inputs(g, g, g, g, g, g)
    need_f, need_b = csbp.workspace_bytes(prob, 0), csbp.workspace_bytes(prob, 1)
    assert need_f > 0 and need_b > 0
    assert L.csbp_attn_fwd(ctypes.byref(prob), ctypes.byref(inp), g, ctypes.byref(info),
                           g, g, g, g, need_f - 1, None) == -3
    assert L.csbp_attn_bwd(ctypes.byref(prob), ctypes.byref(inp), g, ctypes.byref(info),
                           *([g] * 12), need_b - 1, None) == -3


RANK_CASES = [s for s in SWEEP + random_sweep(40, 2026) if s[3] > 1]


@pytest.mark.parametrize("L,M,T,P,clean,W,causal", RANK_CASES)
def test_per_rank_lists_partition_the_tile_set_by_query_owner(L, M, T, P, clean, W, causal):
    """A CSBP rank's list (per_rank = 1) holds exactly the mask's tile pairs
    whose query tile lies in one of the rank's two clean chunks (the oracle's
    zigzag chunk owner; the corrupted blocks of such a tile all belong to the
    rank too), with the same full/partial flags and key parts; the forward is
    one fused task per owned query tile; every key tile keeps a backward
    task; and the ranks' lists partition the single-GPU list."""
    want = O.tile_pairs(L, M, T, T, P, clean, W, causal)
    chunk = L // (2 * P)
    co = O.chunk_owner(L, P)
    bo = O.block_owner(L, M, P)
    nT = -(-L // T)
    union = set()
    for r in range(P):
        prob = csbp.make_problem(1, L, M, 2, 1, 64, P=P, has_clean_queries=clean, tile=T,
                                 window=W, clean_causal=causal, rank=r)
        _, _, words, info = csbp.block_schedule(prob)
        fwd, bwd, fc, bc = expand(words, info, P)
        owned = {qt for qt in range(nT) if co[(qt * T) // chunk] == r}
        for qt in owned:  # the corrupted blocks of an owned tile are the rank's
            assert set(bo[qt * T // M:min((qt + 1) * T, L) // M]) <= {r}
        mine = {x for x in want if x[1] in owned}
        assert all(x[5] == -1 for x in fwd)
        assert {x[:5] for x in fwd} == {x[:5] for x in mine}
        assert bwd == mine
        assert info.tile_pairs == len(mine)
        assert info.n_bwd_tasks == 2 * nT
        assert_fwd_order(words, info, fc, W)
        assert bc == sorted(bc, reverse=True)
        assert not (union & mine)
        union |= mine
    assert union == want


def test_per_rank_needs_shards_and_a_rank_in_range():
    for P, rank, per_rank, ok in [(1, 0, 1, False), (2, 2, 1, False), (2, -1, 1, False),
                                  (2, 1, 0, False), (2, 1, 1, True), (4, 0, 2, False)]:
        prob = csbp.make_problem(1, 1024, 32, 2, 1, 64, P=P)
        prob.per_rank, prob.rank = per_rank, rank
        info = csbp.ScheduleInfo()
        st = csbp.lib().csbp_block_schedule(ctypes.byref(prob), None, None, None, 0,
                                            ctypes.byref(info))
        assert (st == -6) == ok, (P, rank, per_rank, st)   # CSBP_ERR_CAPACITY: size query
        if not ok:
            assert st == -1
    # a rank's list is refused for the whole-sequence problem, and vice versa
    a = csbp.make_problem(1, 1024, 32, 2, 1, 64, P=2)
    b = csbp.make_problem(1, 1024, 32, 2, 1, 64, P=2, rank=1)
    c = csbp.make_problem(1, 1024, 32, 2, 1, 64, P=2, rank=0)
    keys = {csbp.block_schedule(x)[3].problem_key for x in (a, b, c)}
    assert len(keys) == 3
    # a rank's forward needs no partials: status word only
    assert csbp.workspace_bytes(b, 0) == 256 < csbp.workspace_bytes(a, 0)
    assert csbp.workspace_bytes(b, 1) == csbp.workspace_bytes(a, 1)
