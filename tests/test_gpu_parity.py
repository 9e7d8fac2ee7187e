"""GPU parity: the CUDA path through the C-ABI against the float64 oracle.

Tolerances (bf16 inputs, fp32 accumulation): O max-abs <= 1e-2; dQ, dK, dV
relative Frobenius <= 1e-2; LSE abs <= 1e-3.  Small cases compare every
element; the full-size workloads compare seeded samples of query rows (O,
LSE, dQ) and of keys (dK, dV) that the oracle computes one by one, plus the
exact whole-tensor invariants sum_j dK_j = 0 and sum_j dV_j = sum dO.
"""
import numpy as np
import pytest
import torch

from block_diffusion_lm_gb300 import csbp
from block_diffusion_lm_gb300.inputs import WORKLOADS, Workload, make_inputs, to_f64
from oracle import csbp_oracle as O

pytestmark = pytest.mark.gpu

TOL_O = 1e-2
TOL_REL = 1e-2
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from block_diffusion_lm_gb300 import build
    build.build()


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def run_gpu(w: Workload, L=None, seed=None, P=None, bwd_chunk=0):
    L = w.L if L is None else L
    t = make_inputs(w, "cuda", seed=seed, L=L)
    attn = csbp.BlockDiffusionAttention(w.batch, L, w.M, w.Hq, w.Hkv, w.d,
                                        P=w.P if P is None else P,
                                        has_clean_queries=w.has_clean_queries,
                                        window=w.window, clean_causal=w.clean_causal,
                                        bwd_chunk=bwd_chunk)
    out = attn.forward(t)
    g = attn.backward(t, out)
    attn.check()
    torch.cuda.synchronize()
    return t, out, g


SMALL = [
    WORKLOADS["tiny"],
    Workload("gqa_ragged", 1, 400, 16, 4, 2, 128, seed=11),
    Workload("batch2", 2, 384, 32, 2, 1, 128, seed=12),
    Workload("drafter_small", 1, 512, 16, 4, 1, 128, has_clean_queries=False, seed=13),
    Workload("block_eq_tile", 1, 512, 128, 2, 2, 64, seed=14),
    Workload("block_gt_tile", 1, 512, 256, 2, 1, 128, seed=15),
    Workload("token_blocks", 1, 256, 1, 2, 2, 64, seed=16),
    Workload("kscale", 1, 384, 32, 4, 1, 128, k_scale_range=(0.5, 2.0), seed=17),
    Workload("single_partial_tile", 1, 48, 16, 2, 1, 128, seed=18),
    Workload("sharded_small", 1, 1024, 16, 4, 2, 128, P=2, seed=19),
    Workload("sharded_p4", 1, 2048, 32, 2, 1, 128, P=4, seed=20),
    Workload("drafter_sharded", 1, 1024, 16, 2, 1, 64, P=2, has_clean_queries=False, seed=21),
    # sliding window (keys less than W positions back) and token-causal clean queries
    Workload("win_gqa", 1, 512, 16, 4, 2, 128, window=100, seed=22),
    Workload("causal_clean", 1, 384, 32, 2, 1, 128, clean_causal=True, seed=23),
    Workload("win_causal_ragged", 1, 400, 16, 4, 2, 64, window=150, clean_causal=True, seed=24),
    Workload("win_sharded", 1, 1024, 16, 4, 2, 128, P=2, window=200, seed=25),
    Workload("win_drafter", 1, 512, 16, 4, 1, 128, has_clean_queries=False, window=64, seed=26),
    Workload("win_one", 1, 256, 8, 2, 1, 128, window=1, clean_causal=True, seed=27),
    Workload("win_tokens", 1, 256, 1, 2, 2, 64, window=37, seed=28),
    Workload("win_tile_multiple", 1, 1024, 32, 2, 1, 128, window=256, clean_causal=True, seed=29),
    # blocks spanning several tiles
    Workload("block512_small", 1, 1536, 512, 2, 1, 128, seed=34),
    Workload("block1024_gqa", 1, 2048, 1024, 4, 2, 64, seed=35),
    Workload("block384_ragged_tiles", 1, 1152, 384, 2, 2, 128, seed=36),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_cases_match_oracle_elementwise(w):
    _check_against_oracle(w)


# the backward in query-tile windows (fp32 dK/dV accumulation), forced on
# small problems by a window of a few query tiles
WINDOWED = [
    (WORKLOADS["tiny"], 3),
    (Workload("gqa_ragged_w", 1, 400, 16, 4, 2, 128, seed=40), 1),
    (Workload("drafter_small_w", 1, 512, 16, 4, 1, 128, has_clean_queries=False, seed=41), 2),
    (Workload("win_causal_w", 1, 640, 16, 4, 2, 64, window=150, clean_causal=True, seed=42), 2),
    (Workload("sharded_w", 1, 1024, 16, 4, 2, 128, P=2, seed=43), 3),
    (Workload("batch2_w", 2, 384, 32, 2, 1, 128, seed=44), 1),
]


@pytest.mark.parametrize("w,chunk", WINDOWED, ids=[f"{w.name}-c{c}" for w, c in WINDOWED])
def test_windowed_backward_matches_oracle_elementwise(w, chunk):
    _check_against_oracle(w, bwd_chunk=chunk)


def _check_against_oracle(w, bwd_chunk=0):
    t, (oc, ox, lse), g = run_gpu(w, bwd_chunk=bwd_chunk)
    for b in range(w.batch):
        f = {k: (to_f64(v[b]) if v is not None else None) for k, v in t.items()}
        Oc, Ox, Z = O.bd_attention_fwd(f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"],
                                       f["k_corr"], f["v_corr"], w.M, w.scale, w.window,
                                       w.clean_causal)
        G = O.bd_attention_bwd(f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"],
                               f["k_corr"], f["v_corr"], f["do_clean"], f["do_corr"], w.M, w.scale,
                               w.window, w.clean_causal)
        gl = to_f64(lse[b])
        assert np.abs(to_f64(ox[b]) - Ox).max() <= TOL_O
        assert np.abs(gl[1] - Z[1]).max() <= TOL_LSE
        if w.has_clean_queries:
            assert np.abs(to_f64(oc[b]) - Oc).max() <= TOL_O
            assert np.abs(gl[0] - Z[0]).max() <= TOL_LSE
        names = ["dq_corr", "dk_clean", "dv_clean", "dk_corr", "dv_corr"]
        if w.has_clean_queries:
            names.append("dq_clean")
        for k in names:
            want = G[k]
            got = to_f64(g[k][b])
            if np.linalg.norm(want) == 0:
                # an exactly cancelling gradient (a row or key with one
                # partner: dS = P (dP - D) = 0) leaves only rounding residue
                assert np.abs(got).max() <= TOL_O, k
            else:
                assert rel_fro(got, want) <= TOL_REL, (k, rel_fro(got, want))


@pytest.mark.parametrize("pad_heads,extra_tokens,clean", [(0, 0, True), (1, 3, True),
                                                         (0, 5, False)])
def test_packed_qkv_views_match_contiguous_inputs_and_oracle(pad_heads, extra_tokens, clean):
    """q, k and v of each copy as views into one packed [batch][L'][Hq + 2 Hkv
    (+ pad)][d] buffer: token stride (Hq + 2 Hkv + pad) d, batch stride
    L' (Hq + 2 Hkv + pad) d with L' >= L.  The forward is bit-identical to the
    contiguous inputs' (the same data through other tensor maps); the
    gradients agree to fp32 summation order; both match the oracle."""
    w = Workload("packed", 2, 512, 16, 4, 2, 128, has_clean_queries=clean, seed=50)
    t = make_inputs(w, "cuda")
    attn = csbp.BlockDiffusionAttention(w.batch, w.L, w.M, w.Hq, w.Hkv, w.d,
                                        has_clean_queries=clean)
    ref_o = attn.forward(t)
    ref_g = attn.backward(t, ref_o)
    Ht = w.Hq + 2 * w.Hkv + pad_heads
    v = dict(t)
    for copy in ("clean", "corr"):
        buf = torch.zeros(w.batch, w.L + extra_tokens, Ht, w.d, dtype=torch.bfloat16,
                          device="cuda")
        spans = {"q": (0, w.Hq), "k": (w.Hq, w.Hq + w.Hkv), "v": (w.Hq + w.Hkv, w.Hq + 2 * w.Hkv)}
        for x, (a, b) in spans.items():
            if t[f"{x}_{copy}"] is None:
                continue
            buf[:, :w.L, a:b] = t[f"{x}_{copy}"]
            v[f"{x}_{copy}"] = buf[:, :w.L, a:b]
            assert not v[f"{x}_{copy}"].is_contiguous()
    out = attn.forward(v)
    g = attn.backward(v, out)
    attn.check()
    torch.cuda.synchronize()
    for a, b in zip(out, ref_o):
        # LSE rows of an absent clean-query stream are NaN in both
        assert (a is None and b is None) or bool(((a == b) | (a.isnan() & b.isnan())).all())
    for k, r in ref_g.items():
        if r is not None:
            assert ((g[k].double() - r.double()).norm() / r.double().norm()).item() <= 1e-5, k
    for b in range(w.batch):
        f = {k: (to_f64(x[b]) if x is not None else None) for k, x in t.items()}
        _, Ox, Z = O.bd_attention_fwd(f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"],
                                      f["k_corr"], f["v_corr"], w.M, w.scale)
        assert np.abs(to_f64(out[1][b]) - Ox).max() <= TOL_O
        assert np.abs(to_f64(out[2][b])[1] - Z[1]).max() <= TOL_LSE
        G = O.bd_attention_bwd(f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"],
                               f["k_corr"], f["v_corr"], f["do_clean"], f["do_corr"], w.M, w.scale)
        for k in ("dq_corr", "dk_clean", "dv_clean"):
            assert rel_fro(to_f64(g[k][b]), G[k]) <= TOL_REL, k


def test_sharded_equals_unsharded_on_gpu():
    """Per-shard partials + LSE merge (P=4) reproduce the fused unsharded pass."""
    w = Workload("shard_vs_fused", 1, 2048, 16, 4, 2, 128, P=4, seed=30)
    _, (oc1, ox1, z1), g1 = run_gpu(w, P=1)
    _, (oc4, ox4, z4), g4 = run_gpu(w, P=4)
    assert (ox1.float() - ox4.float()).abs().max().item() <= 2 ** -7
    assert (oc1.float() - oc4.float()).abs().max().item() <= 2 ** -7
    assert (z1 - z4).abs().max().item() <= 1e-4
    for k in ("dq_clean", "dq_corr", "dk_clean", "dv_clean", "dk_corr", "dv_corr"):
        a, b = g1[k].double(), g4[k].double()
        assert ((a - b).norm() / b.norm()).item() <= 1e-2, k


def test_repeat_calls_are_deterministic_in_forward():
    w = Workload("repeat", 1, 512, 32, 2, 1, 128, seed=31)
    t = make_inputs(w, "cuda")
    attn = csbp.BlockDiffusionAttention(1, 512, 32, 2, 1, 128)
    a = attn.forward(t)
    b = attn.forward(t)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[0], b[0]) and torch.equal(a[2], b[2])


def test_kernel_timing_records_one_pair_per_call():
    w = Workload("timing", 1, 512, 32, 2, 1, 128, seed=33)
    t = make_inputs(w, "cuda")
    attn = csbp.BlockDiffusionAttention(1, 512, 32, 2, 1, 128)
    out = attn.forward(t)
    attn.backward(t, out)
    torch.cuda.synchronize()
    csbp.kernel_timing(True)
    for _ in range(3):
        out = attn.forward(t, out=out)
        attn.backward(t, out)
    csbp.kernel_timing(False)
    attn.forward(t, out=out)  # not recorded
    fwd_ms, n_fwd, bwd_ms, n_bwd = csbp.kernel_timing_read()
    assert (n_fwd, n_bwd) == (3, 3)
    assert fwd_ms > 0.0 and bwd_ms > 0.0
    attn.check()


# ------------------------------------------------------------------ full size
def _invariants(w, t, g):
    """sum_j dK_j = 0 per KV head; sum_j dV_j = sum of the group's dO rows."""
    G = w.Hq // w.Hkv
    dk = g["dk_clean"].double().sum(dim=1) + g["dk_corr"].double().sum(dim=1)  # [b, Hkv, d]
    dv = g["dv_clean"].double().sum(dim=1) + g["dv_corr"].double().sum(dim=1)
    do = t["do_corr"].double().sum(dim=1)
    if t["do_clean"] is not None:
        do = do + t["do_clean"].double().sum(dim=1)
    do = do.view(w.batch, w.Hkv, G, w.d).sum(dim=2)
    dk_scale = g["dk_clean"].double().abs().sum(dim=1).max().item()
    assert dk.abs().max().item() <= 2e-3 * dk_scale
    assert ((dv - do).norm() / do.norm()).item() <= 1e-2


class _HostView:
    """bf16 host tensor [L, H, d] that hands the oracle float32 numpy slices on
    indexing (exact up-cast), so only the slices it touches are converted."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        return self.t[idx].to(torch.float32).numpy()


def _sampled_check(w, t, out, g, rows_per_head, n_keys, walk_keys, walk_heads, seed):
    oc, ox, lse = out
    rng = np.random.default_rng(seed)
    L = w.L
    fv = {k: (_HostView(v[0].cpu()) if v is not None else None) for k, v in t.items()}
    streams = [0, 1] if w.has_clean_queries else [1]
    samples = []
    for h in range(w.Hq):
        for _ in range(rows_per_head):
            samples.append((int(rng.choice(streams)), int(rng.integers(0, L)), h))
    ref = O.sampled_rows(fv["q_clean"], fv["k_clean"], fv["v_clean"], fv["q_corr"], fv["k_corr"],
                         fv["v_corr"], fv["do_clean"], fv["do_corr"], w.M, w.scale, samples,
                         w.window, w.clean_causal)
    o_err, z_err = 0.0, 0.0
    dq_got, dq_want = [], []
    for (qs, i, h), (o, z, D, dq) in ref.items():
        og = (oc if qs == 0 else ox)[0, i, h].double().cpu().numpy()
        o_err = max(o_err, float(np.abs(og - o).max()))
        z_err = max(z_err, abs(lse[0, qs, h, i].item() - z))
        dq_got.append(g["dq_clean" if qs == 0 else "dq_corr"][0, i, h].double().cpu().numpy())
        dq_want.append(dq)
    assert o_err <= TOL_O, o_err
    assert z_err <= TOL_LSE, z_err
    assert rel_fro(np.array(dq_got), np.array(dq_want)) <= TOL_REL
    # keys: corrupted keys (read by their own block), late clean keys (read
    # by the last blocks) and clean keys whose backward task walks many query
    # tiles (the readers of clean key j are every later query row, so its
    # dK/dV sum over the longest walks of the kernel); each compared
    # element-wise, per key
    keys = []
    for _ in range(n_keys):
        g_ = int(rng.integers(0, w.Hkv))
        keys.append((1, int(rng.integers(0, L)), g_))
        keys.append((0, int(rng.integers(L - 2 * w.M, L - w.M)), g_))
    walk = set()
    for g_ in rng.choice(w.Hkv, size=walk_heads, replace=False):
        for pos in walk_keys:
            j = (pos if pos >= 0 else L + pos) + int(rng.integers(0, w.M))
            keys.append((0, j, int(g_)))
            walk.add((0, j, int(g_)))
    kref = O.sampled_keys(fv["q_clean"], fv["k_clean"], fv["v_clean"], fv["q_corr"], fv["k_corr"],
                          fv["v_corr"], fv["do_clean"], fv["do_corr"], w.M, w.scale, keys,
                          w.window, w.clean_causal)
    got_k, want_k, got_v, want_v = [], [], [], []
    for (ks, j, gg), (dk, dv) in kref.items():
        sfx = "clean" if ks == 0 else "corr"
        a_k = g["dk_" + sfx][0, j, gg].double().cpu().numpy()
        a_v = g["dv_" + sfx][0, j, gg].double().cpu().numpy()
        if (ks, j, gg) in walk:
            # each walk key on its own: a dropped (query tile, key tile)
            # contribution of a long walk shows in that key's row
            assert rel_fro(a_k, dk) <= TOL_REL, (ks, j, gg, rel_fro(a_k, dk))
            assert rel_fro(a_v, dv) <= TOL_REL, (ks, j, gg, rel_fro(a_v, dv))
        got_k.append(a_k)
        got_v.append(a_v)
        want_k.append(dk)
        want_v.append(dv)
    assert rel_fro(np.array(got_k), np.array(want_k)) <= TOL_REL
    assert rel_fro(np.array(got_v), np.array(want_v)) <= TOL_REL


# name, query rows per head, random (corrupted, late clean) key pairs, clean
# key positions whose tasks walk many query tiles (negative: from the end;
# one key of each block that starts there), KV heads they are drawn on, seed.
# The walk keys cost the oracle their readers' full rows (about 1.5 minutes
# of host time each beyond the 16K sequences): the early and middle ones are
# affordable on the 16K sequences only, where a block-0 key's task walks
# every query tile of both copies; the longer workloads take a key 8,192
# (sharded), 2,048 (long) or 1,024 (drafter) positions before the end,
# walks of 512, 256 and 32 query-tile steps under the KV-head-major CTA order.
FULL_SIZE = [
    ("dense14b", 256, 8, (0, 4096, 8192), 2, 101),
    ("sharded", 64, 4, (-8192,), 1, 102),
    ("long", 64, 4, (-2048,), 1, 103),
    ("drafter", 32, 2, (-1024,), 1, 104),
    ("window1k", 64, 8, (0, 8192), 2, 105),
    ("block1024", 32, 8, (0, 8192), 1, 106),
]


@pytest.mark.parametrize("name,rows,keys,walk,walk_heads,seed", FULL_SIZE,
                         ids=[c[0] for c in FULL_SIZE])
def test_full_size_workloads_sampled(name, rows, keys, walk, walk_heads, seed):
    w = WORKLOADS[name]
    t, out, g = run_gpu(w)
    _invariants(w, t, g)
    _sampled_check(w, t, out, g, rows, keys, walk, walk_heads, seed=seed)
    del t, out, g
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n,rows,Hq,d", [(1, 300, 2, 64), (2, 257, 4, 128), (3, 128, 1, 128),
                                         (9, 1000, 2, 64)])
def test_lse_merge_entry_point_matches_oracle(n, rows, Hq, d):
    """csbp_lse_merge on its own: n fp32 partials with random LSEs, some parts
    empty for some rows (z = -inf) and row 0 empty in every part, against the
    oracle's two-part merge folded over the parts."""
    g = torch.Generator().manual_seed(100 * n + rows)
    o_parts = [torch.randn(rows, Hq, d, generator=g) for _ in range(n)]
    z_parts = [3.0 * torch.randn(Hq, rows, generator=g) for _ in range(n)]
    for z in z_parts:
        z[torch.rand(Hq, rows, generator=g) < 0.2] = float("-inf")
        z[:, 0] = float("-inf")
    o_out = torch.empty(rows, Hq, d, dtype=torch.bfloat16, device="cuda")
    z_out = torch.empty(Hq, rows, dtype=torch.float32, device="cuda")
    csbp.lse_merge([o.cuda() for o in o_parts], [z.cuda() for z in z_parts], o_out, z_out)
    torch.cuda.synchronize()
    ref_o, ref_z = O.lse_merge([o.double().numpy().reshape(rows * Hq, d) for o in o_parts],
                               [z.double().numpy().T.reshape(rows * Hq) for z in z_parts])
    got_o = to_f64(o_out).reshape(rows * Hq, d)
    got_z = to_f64(z_out).T.reshape(rows * Hq)
    # bf16 output: rounding grows with |O|, which reaches ~4.5 for these
    # unit-normal partials (attention outputs stay near 1)
    assert np.all(np.abs(got_o - ref_o) <= TOL_O + 2.0 ** -8 * np.abs(ref_o))
    finite = np.isfinite(ref_z)
    assert np.array_equal(finite, np.isfinite(got_z))
    assert np.abs(got_z[finite] - ref_z[finite]).max() <= 1e-5 * max(1.0, np.abs(ref_z[finite]).max())
    assert np.all(got_o[~finite] == 0)


# ----------------------------------------------------------------- fp8 inputs
def test_e4m3_decode_is_bit_exact_against_the_oracle():
    """csbp_e4m3_to_bf16 on every E4M3 code (a ragged length, so the scalar
    tail runs too) and several scales, bit for bit against the oracle's
    decoding from the format definition (NaN where the code is NaN)."""
    n = 256 * 37 + 5
    codes = (torch.arange(n, dtype=torch.int64) * 7 % 256).to(torch.uint8)
    for scale in (1.0, 2.0 ** -5, 128.0, 0.3, -1.7):
        got = csbp.e4m3_to_bf16(codes.cuda(), scale).double().cpu().numpy()
        want = O.e4m3_to_bf16(codes.numpy(), scale)
        nan = np.isnan(want)
        assert np.array_equal(nan, np.isnan(got)), scale
        assert np.array_equal(got[~nan], want[~nan]), scale


E4M3_CASES = [Workload("e4m3_small", 1, 512, 32, 4, 2, 128, seed=70, e4m3=True),
              Workload("e4m3_drafter", 1, 384, 16, 2, 1, 64, has_clean_queries=False,
                       k_scale_range=(0.5, 2.0), seed=71, e4m3=True)]


@pytest.mark.parametrize("w", E4M3_CASES, ids=[w.name for w in E4M3_CASES])
def test_e4m3_inputs_through_the_attention_match_the_oracle(w):
    """Q, K, V and dO kept in fp8 E4M3 with power-of-two scales: decoded on
    the GPU, then the same attention entry points; the oracle decodes the
    same bytes itself, so both sides see identical bf16 values."""
    from block_diffusion_lm_gb300.inputs import make_inputs_e4m3
    codes, scales = make_inputs_e4m3(w, "cuda")
    t = {k: (csbp.e4m3_to_bf16(c, scales[k]) if c is not None else None)
         for k, c in codes.items()}
    attn = csbp.BlockDiffusionAttention(w.batch, w.L, w.M, w.Hq, w.Hkv, w.d,
                                        has_clean_queries=w.has_clean_queries)
    oc, ox, lse = attn.forward(t)
    g = attn.backward(t, (oc, ox, lse))
    attn.check()
    torch.cuda.synchronize()
    f = {k: (O.e4m3_to_bf16(c[0].cpu().numpy(), scales[k]) if c is not None else None)
         for k, c in codes.items()}
    args = (f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"], f["k_corr"], f["v_corr"])
    Oc, Ox, Z = O.bd_attention_fwd(*args, w.M, w.scale)
    G = O.bd_attention_bwd(*args, f["do_clean"], f["do_corr"], w.M, w.scale)
    assert np.abs(to_f64(ox[0]) - Ox).max() <= TOL_O
    assert np.abs(to_f64(lse[0])[1] - Z[1]).max() <= TOL_LSE
    names = ["dq_corr", "dk_clean", "dv_clean", "dk_corr", "dv_corr"]
    if w.has_clean_queries:
        assert np.abs(to_f64(oc[0]) - Oc).max() <= TOL_O
        names.append("dq_clean")
    for k in names:
        assert rel_fro(to_f64(g[k][0]), G[k]) <= TOL_REL, k
