"""Pins for the float64 oracle, against facts fixed by the pages and by
mathematics rather than by the oracle itself: hand-worked fixtures, closed
forms, special cases that reduce to a library routine (torch SDPA in float64),
finite differences, and the invariants the pages state in words.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import csbp_oracle as O
from conftest import read_golden

CLEAN, CORR = O.CLEAN, O.CORR


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def make(L, Hq, Hkv, d, seed=0, clean=True):
    r = np.random.default_rng(seed)
    t = {n: r.standard_normal((L, Hq if n.startswith(("q", "do")) else Hkv, d))
         for n in ("qc", "kc", "vc", "qx", "kx", "vx", "doc", "dox")}
    if not clean:
        t["qc"] = None
        t["doc"] = None
    return t


# ---------------------------------------------------------------- mask
def test_mask_matches_hand_written_fixture():
    rows = read_golden("mask_L6_M2.txt")
    want = np.array([[c == "1" for c in r.replace(" ", "")] for r in rows])
    assert want.shape == (12, 12)
    np.testing.assert_array_equal(O.bd_mask(6, 2), want)


def test_forward_matches_hand_worked_fixture():
    """O and LSE of all four rows of a two-block, one-token-per-block problem
    whose scores are logs of small integers, and every gradient for dO = 1,
    worked out by hand."""
    rows = [[float(x) for x in r.split()] for r in read_golden("attention_L2_M1.txt")]
    inp, want, grads = np.array(rows[:2]), np.array(rows[2:4]), np.array(rows[4:6])
    qc, kc, vc, qx, kx, vx = (inp[:, c].reshape(2, 1, 1) for c in range(6))
    Oc, Ox, lse = O.bd_attention_fwd(qc, kc, vc, qx, kx, vx, M=1, scale=1.0)
    np.testing.assert_allclose(Oc[:, 0, 0], want[:, 0], atol=1e-14)
    np.testing.assert_allclose(lse[CLEAN, 0], want[:, 1], atol=1e-14)
    np.testing.assert_allclose(Ox[:, 0, 0], want[:, 2], atol=1e-14)
    np.testing.assert_allclose(lse[CORR, 0], want[:, 3], atol=1e-14)
    ones = np.ones((2, 1, 1))
    G = O.bd_attention_bwd(qc, kc, vc, qx, kx, vx, ones, ones, M=1, scale=1.0)
    for c, name in enumerate(("dq_clean", "dk_clean", "dv_clean", "dq_corr", "dk_corr",
                              "dv_corr")):
        np.testing.assert_allclose(G[name][:, 0, 0], grads[:, c], atol=1e-14, err_msg=name)


def test_mask_agrees_with_scalar_predicate_and_rows():
    L, M = 12, 3
    A = O.bd_mask(L, M)
    for qs, i, ks, j in itertools.product((0, 1), range(L), (0, 1), range(L)):
        assert A[qs * L + i, ks * L + j] == O.allowed(qs, i, ks, j, M)
    for qs, i in itertools.product((0, 1), range(L)):
        np.testing.assert_array_equal(O.mask_row(qs, i, L, M), A[qs * L + i])


def test_every_row_reads_at_least_one_block():
    for L, M in ((16, 4), (16, 1), (16, 16)):
        A = O.bd_mask(L, M)
        assert A.sum(axis=1).min() >= M


def test_masked_attention_matches_torch_sdpa_with_explicit_mask():
    L, M, d = 16, 4, 8
    A = O.bd_mask(L, M)
    q, k, v = rnd((2 * L, d), 1), rnd((2 * L, d), 2), rnd((2 * L, d), 3)
    o, _ = O.masked_attention(q, k, v, A, 0.3)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=torch.from_numpy(A)[None], scale=0.3)[0].numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-13)


# ------------------------------------------------ special cases / closed forms
def test_single_block_is_two_independent_full_attentions():
    """M = L (B = 1): clean and corrupted copies each attend bidirectionally
    to themselves; corrupted queries see no clean key."""
    L, d, Hq = 8, 4, 2
    t = make(L, Hq, Hq, d, seed=5)
    Oc, Ox, lse = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"],
                                     M=L, scale=0.5)
    for h in range(Hq):
        for q, k, v, got in ((t["qc"], t["kc"], t["vc"], Oc), (t["qx"], t["kx"], t["vx"], Ox)):
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[:, h])[None], torch.from_numpy(k[:, h])[None],
                torch.from_numpy(v[:, h])[None], scale=0.5)[0].numpy()
            np.testing.assert_allclose(got[:, h], ref, atol=1e-13)


def test_unit_blocks_make_clean_stream_token_causal():
    """M = 1: clean queries reduce to textbook (inclusive) causal attention."""
    L, d = 10, 4
    t = make(L, 1, 1, d, seed=6)
    Oc, _, _ = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"],
                                  M=1, scale=0.7)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(t["qc"][:, 0])[None], torch.from_numpy(t["kc"][:, 0])[None],
        torch.from_numpy(t["vc"][:, 0])[None], is_causal=True, scale=0.7)[0].numpy()
    np.testing.assert_allclose(Oc[:, 0], ref, atol=1e-13)


def test_unit_blocks_corrupted_row_reads_own_token_and_earlier_clean():
    """M = 1: corrupted query i = softmax over {clean keys < i} U {corrupted key i}."""
    L, d = 7, 3
    t = make(L, 1, 1, d, seed=7)
    _, Ox, _ = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"],
                                  M=1, scale=1.0)
    for i in range(L):
        keys = np.concatenate([t["kc"][:i, 0], t["kx"][i:i + 1, 0]])
        vals = np.concatenate([t["vc"][:i, 0], t["vx"][i:i + 1, 0]])
        s = keys @ t["qx"][i, 0]
        p = np.exp(s - s.max())
        p /= p.sum()
        np.testing.assert_allclose(Ox[i, 0], p @ vals, atol=1e-13)


def test_zero_queries_give_log_of_visible_key_count():
    """Q = 0: every allowed logit is 0, so LSE_i = ln(n_i) with n_i = M (b_i + 1)
    for both copies, and O_i = mean of the visible V rows."""
    L, M, d = 24, 4, 4
    t = make(L, 2, 1, d, seed=8)
    z = np.zeros_like(t["qc"])
    Oc, Ox, lse = O.bd_attention_fwd(z, t["kc"], t["vc"], z, t["kx"], t["vx"], M, 0.5)
    n = M * (np.arange(L) // M + 1)
    for st in (CLEAN, CORR):
        for h in range(2):
            np.testing.assert_allclose(lse[st, h], np.log(n), atol=1e-14)
    for i in range(L):
        b = i // M
        np.testing.assert_allclose(Oc[i, 0], t["vc"][: (b + 1) * M, 0].mean(0), atol=1e-13)
        vis = np.concatenate([t["vc"][: b * M, 0], t["vx"][b * M:(b + 1) * M, 0]])
        np.testing.assert_allclose(Ox[i, 1], vis.mean(0), atol=1e-13)


def test_zero_queries_closed_form_dq():
    """Q = 0: P_ij = 1/n_i over visible keys, so
    dQ_i = scale * sum_j P_ij (dP_ij - D_i) K_j with dP_ij = dO_i . V_j."""
    L, M, d = 12, 3, 3
    t = make(L, 1, 1, d, seed=9)
    z = np.zeros_like(t["qc"])
    g = O.bd_attention_bwd(z, t["kc"], t["vc"], z, t["kx"], t["vx"], t["doc"], t["dox"], M, 0.9)
    for i in range(L):
        b = i // M
        K = t["kc"][: (b + 1) * M, 0]
        V = t["vc"][: (b + 1) * M, 0]
        dp = V @ t["doc"][i, 0]
        D = dp.mean()
        want = 0.9 * ((dp - D)[:, None] * K).mean(0)
        np.testing.assert_allclose(g["dq_clean"][i, 0], want, atol=1e-13)


def test_constant_values_give_constant_output():
    L, M, d = 16, 4, 5
    t = make(L, 2, 2, d, seed=10)
    c = np.arange(d, dtype=np.float64) - 2.0
    vc = np.broadcast_to(c, t["vc"].shape).copy()
    Oc, Ox, _ = O.bd_attention_fwd(t["qc"], t["kc"], vc, t["qx"], t["kx"], vc.copy(), M, 0.4)
    np.testing.assert_allclose(Oc, np.broadcast_to(c, Oc.shape), atol=1e-13)
    np.testing.assert_allclose(Ox, np.broadcast_to(c, Ox.shape), atol=1e-13)


# ------------------------------------------------------------ backward
@pytest.mark.parametrize("M,Hkv,clean", [(2, 1, True), (4, 2, True), (8, 1, True), (2, 2, False)])
def test_backward_matches_central_finite_differences(M, Hkv, clean):
    L, Hq, d, scale = 16, 2, 4, 0.6
    t = make(L, Hq, Hkv, d, seed=11 + M, clean=clean)

    def f(tt):
        Oc, Ox, _ = O.bd_attention_fwd(tt["qc"], tt["kc"], tt["vc"], tt["qx"], tt["kx"],
                                       tt["vx"], M, scale)
        val = (Ox * tt["dox"]).sum()
        if clean:
            val += (Oc * tt["doc"]).sum()
        return val

    g = O.bd_attention_bwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"],
                           t["doc"], t["dox"], M, scale)
    names = {"qx": "dq_corr", "kc": "dk_clean", "vc": "dv_clean", "kx": "dk_corr",
             "vx": "dv_corr"}
    if clean:
        names["qc"] = "dq_clean"
    rng = np.random.default_rng(0)
    eps = 1e-5
    for src, gname in names.items():
        for _ in range(6):
            idx = tuple(rng.integers(0, s) for s in t[src].shape)
            tp = {k: (None if v is None else v.copy()) for k, v in t.items()}
            tm = {k: (None if v is None else v.copy()) for k, v in t.items()}
            tp[src][idx] += eps
            tm[src][idx] -= eps
            fd = (f(tp) - f(tm)) / (2 * eps)
            an = g[gname][idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (src, idx, fd, an)


def test_backward_sum_invariants():
    """sum_j dK_j = 0 per KV head (rows of dS sum to zero) and
    sum_j dV_j = sum over the group's query rows of dO_i."""
    L, M, d, Hq, Hkv = 32, 4, 6, 4, 2
    t = make(L, Hq, Hkv, d, seed=21)
    g = O.bd_attention_bwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"],
                           t["doc"], t["dox"], M, 0.35)
    dk = g["dk_clean"].sum(0) + g["dk_corr"].sum(0)
    dv = g["dv_clean"].sum(0) + g["dv_corr"].sum(0)
    np.testing.assert_allclose(dk, 0.0, atol=1e-12)
    G = Hq // Hkv
    for kvh in range(Hkv):
        want = sum(t["doc"][:, h].sum(0) + t["dox"][:, h].sum(0) for h in range(kvh * G, (kvh + 1) * G))
        np.testing.assert_allclose(dv[kvh], want, atol=1e-12)


# ------------------------------------------------------ block separability
def test_corrupted_block_output_ignores_other_blocks_corrupted_kv():
    L, M, d = 16, 4, 4
    t = make(L, 2, 1, d, seed=30)
    _, Ox, _ = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], M, 0.5)
    b = 2
    kx, vx = t["kx"].copy(), t["vx"].copy()
    for other in (0, 1, 3):
        kx[other * M:(other + 1) * M] += 10.0 * rnd((M, 1, d), other)
        vx[other * M:(other + 1) * M] -= 5.0
    _, Ox2, _ = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], kx, vx, M, 0.5)
    np.testing.assert_array_equal(Ox[b * M:(b + 1) * M], Ox2[b * M:(b + 1) * M])
    assert not np.array_equal(Ox[:M], Ox2[:M])


# ---------------------------------------------------------- BP equivalence
def test_block_parallel_gradients_sum_to_whole_sequence_gradient():
    """Owners compute the loss of their own query rows only (corrupted rows of
    their blocks, clean rows of their clean chunks); the owners' losses and
    gradients sum to the whole-sequence objective f = sum O o dO and its VJP."""
    L, M, d, Hq, Hkv, P = 32, 4, 4, 2, 1, 2
    t = make(L, Hq, Hkv, d, seed=40)
    full = O.bd_attention_bwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"],
                              t["doc"], t["dox"], M, 0.5)
    Oc, Ox, _ = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], M, 0.5)
    f_full = (Oc * t["doc"]).sum() + (Ox * t["dox"]).sum()
    owner = O.block_owner(L, M, P)
    f_sum = 0.0
    acc = {k: np.zeros_like(v) for k, v in full.items() if k != "D"}
    for r in range(P):
        rows = np.repeat(owner == r, M)
        doc = np.where(rows[:, None, None], t["doc"], 0.0)
        dox = np.where(rows[:, None, None], t["dox"], 0.0)
        f_sum += (Oc * doc).sum() + (Ox * dox).sum()
        g = O.bd_attention_bwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"],
                               doc, dox, M, 0.5)
        for k in acc:
            acc[k] += g[k]
    assert abs(f_sum - f_full) <= 1e-12 * abs(f_full)
    for k in acc:
        np.testing.assert_allclose(acc[k], full[k], atol=1e-12)


# ------------------------------------------------------------- LSE merge
def test_lse_merge_hand_worked_fixture():
    for line in read_golden("lse_merge_two_parts.txt"):
        v = [float(x) for x in line.split()]
        z1, z2, o1, o2, z, o = v[0], v[1], v[2:5], v[5:8], v[8], v[9:12]
        om, zm = O.lse_merge_pair(np.array([o1]), np.array([z1]), np.array([o2]), np.array([z2]))
        np.testing.assert_allclose(om[0], o, atol=1e-15)
        assert abs(zm[0] - z) < 1e-15


@pytest.mark.parametrize("n_parts", [1, 2, 3, 8])
def test_lse_merge_over_random_partitions_equals_unsharded(n_parts):
    L, M, d = 32, 4, 6
    A = O.bd_mask(L, M)
    q, k, v = rnd((2 * L, d), 50), rnd((2 * L, d), 51), rnd((2 * L, d), 52)
    o_ref, z_ref = O.masked_attention(q, k, v, A, 0.45)
    lab = np.random.default_rng(n_parts).integers(0, n_parts + 1, size=A.shape)  # label n_parts = dropped
    lab = np.where(lab == n_parts, 0, lab)  # every key belongs to some part; part sizes random, some empty rows
    parts = [O.masked_attention(q, k, v, A & (lab == s), 0.45) for s in range(n_parts)]
    o, z = O.lse_merge([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(z, z_ref, atol=1e-12)
    # merge order does not matter
    perm = np.random.default_rng(9).permutation(n_parts)
    o2, z2 = O.lse_merge([parts[s][0] for s in perm], [parts[s][1] for s in perm])
    np.testing.assert_allclose(o2, o_ref, atol=1e-12)
    np.testing.assert_allclose(z2, z_ref, atol=1e-12)


@pytest.mark.parametrize("P,clean,W,causal", [
    (1, True, 0, False), (2, True, 0, False), (4, True, 0, False), (2, False, 0, False),
    # windows leave most shards empty for most rows (z = -inf parts)
    (2, True, 5, False), (4, True, 3, True), (4, False, 7, True), (2, True, 0, True),
])
def test_sharded_forward_equals_unsharded(P, clean, W, causal):
    L, M, d, Hq, Hkv = 32, 2, 4, 4, 2
    t = make(L, Hq, Hkv, d, seed=60 + P + W, clean=clean)
    Oc, Ox, lse = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], M, 0.5,
                                     W, causal)
    Oc2, Ox2, lse2, (op, zp) = O.bd_attention_fwd_sharded(
        t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], M, 0.5, P, W, causal)
    np.testing.assert_allclose(Ox2, Ox, atol=1e-12)
    if clean:
        np.testing.assert_allclose(Oc2, Oc, atol=1e-12)
        np.testing.assert_allclose(lse2, lse, atol=1e-12)
    else:
        np.testing.assert_allclose(lse2[1], lse[1], atol=1e-12)
    # clean queries never read the own-block part
    assert np.all(np.isneginf(zp[P, CLEAN]))


# ------------------------------------------------------- dual-end pairing
def test_dual_end_owner_fixture():
    rows = read_golden("dual_end_owner_B8_P2.txt")
    bo = [int(x) for x in rows[0].split()]
    co = [int(x) for x in rows[1].split()]
    np.testing.assert_array_equal(O.block_owner(16, 2, 2), bo)
    np.testing.assert_array_equal(O.chunk_owner(16, 2), co)


@pytest.mark.parametrize("L,M,P", [(64, 4, 2), (64, 2, 4), (128, 4, 4), (96, 4, 3), (64, 8, 1)])
def test_dual_end_pairing_equalises_work_exactly(L, M, P):
    B = L // M
    owner = O.block_owner(L, M, P)
    # pages: block b and block B-1-b (0-based) share a rank
    for b in range(B):
        assert owner[b] == owner[B - 1 - b]
    for clean in (True, False):
        brute = O.pair_counts_from_mask(L, M, P, owner, clean)
        assert np.all(brute == brute[0]), brute
        np.testing.assert_array_equal(brute, O.pair_counts_per_owner(L, M, P, owner, clean))
    if P > 1:
        contiguous = np.repeat(np.arange(P), B // P).astype(np.int32)
        neg = O.pair_counts_from_mask(L, M, P, contiguous)
        assert len(set(neg.tolist())) == P  # strictly increasing: unbalanced


def test_allowed_pairs_closed_form():
    """Allowed pairs per head = L(L+M) (clean + corrupted queries), from
    sum_b M(M + bM) + sum_b M(b+1)M."""
    for L, M in ((32, 4), (48, 3), (64, 64), (16, 1)):
        A = O.bd_mask(L, M)
        assert A.sum() == L * (L + M) == O.allowed_pairs_per_head(L, M)
        assert A[L:].sum() == L * (L + M) // 2 == O.allowed_pairs_per_head(L, M, False)


# ---------------------------------------------------------- tile schedule
def test_tile_pairs_count_closed_form():
    """With M | T and M < T: clean q tile t needs clean kv tiles 0..t; corrupted
    q tile t needs clean tiles 0..t (t partial) plus corrupted tile t, so the
    count is nT(nT+1) + nT.  With M = T the corrupted diagonal clean tile is
    empty: nT(nT+1)."""
    for L, M, T in ((256, 16, 32), (512, 32, 64), (256, 32, 32)):
        nT = L // T
        s = O.tile_pairs(L, M, T, T)
        want = nT * (nT + 1) + (nT if M < T else 0)
        assert len(s) == want
        full = sum(1 for e in s if e[4])
        # every off-diagonal (kv < q) tile is full; with M < T the diagonal tiles
        # are partial, with M = T the clean-clean and corrupted-corrupted
        # diagonal tiles are single whole blocks, hence full
        assert full == nT * (nT - 1) + (2 * nT if M == T else 0)


def test_tile_pairs_shards_get_equal_tile_counts():
    L, M, T, P = 512, 8, 32, 4
    s = O.tile_pairs(L, M, T, T, P)
    per = np.zeros(P + 1, int)
    for e in s:
        per[e[5]] += 1
    assert np.all(per[:P] == per[0])


# -------------------------------------------------- sampled evaluation
def test_sampled_rows_and_keys_agree_with_full_oracle():
    L, M, d, Hq, Hkv = 32, 4, 4, 4, 2
    t = make(L, Hq, Hkv, d, seed=70)
    Oc, Ox, lse = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], M, 0.5)
    g = O.bd_attention_bwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"],
                           t["doc"], t["dox"], M, 0.5)
    samples = [(CLEAN, 0, 0), (CLEAN, 31, 3), (CORR, 5, 1), (CORR, 30, 2), (CORR, 0, 0),
               (CLEAN, 17, 0), (CORR, 12, 0), (CLEAN, 3, 0)]
    for chunk in (None, 1, 2):
        r = O.sampled_rows(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"],
                           t["doc"], t["dox"], M, 0.5, samples, chunk_rows=chunk)
        assert len(r) == len(samples)
        for (qs, i, h), (o, z, D, dq) in r.items():
            np.testing.assert_allclose(o, (Oc if qs == CLEAN else Ox)[i, h], atol=1e-13)
            assert abs(z - lse[qs, h, i]) < 1e-13
            assert abs(D - g["D"][qs, h, i]) < 1e-13
            np.testing.assert_allclose(dq, g["dq_clean" if qs == CLEAN else "dq_corr"][i, h],
                                       atol=1e-13)
    ks = [(CLEAN, 0, 0), (CLEAN, 29, 1), (CORR, 7, 1), (CORR, 16, 0)]
    # one chunk of readers, and chunks of 1, 3 and 7 rows (ragged last chunk)
    for chunk in (None, 1, 3, 7):
        r = O.sampled_keys(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"],
                           t["doc"], t["dox"], M, 0.5, ks, chunk_rows=chunk)
        for (st, j, kvh), (dk, dv) in r.items():
            sfx = "clean" if st == CLEAN else "corr"
            np.testing.assert_allclose(dk, g["dk_" + sfx][j, kvh], atol=1e-12)
            np.testing.assert_allclose(dv, g["dv_" + sfx][j, kvh], atol=1e-12)
    # drafter shape: no clean queries read the clean keys
    g2 = O.bd_attention_bwd(None, t["kc"], t["vc"], t["qx"], t["kx"], t["vx"],
                            None, t["dox"], M, 0.5)
    r = O.sampled_keys(None, t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], None, t["dox"], M,
                       0.5, ks, chunk_rows=5)
    for (st, j, kvh), (dk, dv) in r.items():
        sfx = "clean" if st == CLEAN else "corr"
        np.testing.assert_allclose(dk, g2["dk_" + sfx][j, kvh], atol=1e-12)
        np.testing.assert_allclose(dv, g2["dv_" + sfx][j, kvh], atol=1e-12)


def test_mask_rows_equal_the_rows_of_the_mask():
    """The vectorised row mask of the sampled evaluators equals `mask_row`
    (and so `bd_mask`) row by row, for every option."""
    rng = np.random.default_rng(71)
    for L, M, W, causal in [(48, 4, 0, False), (48, 8, 0, True), (64, 4, 9, False),
                            (64, 16, 23, True), (30, 1, 5, False)]:
        rows = [(int(rng.integers(0, 2)), int(rng.integers(0, L))) for _ in range(40)]
        got = O.mask_rows(rows, L, M, W, causal)
        want = np.stack([O.mask_row(qs, i, L, M, W, causal) for qs, i in rows])
        assert np.array_equal(got, want)
        A = O.bd_mask(L, M, W, causal)
        assert np.array_equal(got, np.stack([A[qs * L + i] for qs, i in rows]))


# ------------------------------------------------------- planted mistakes
def test_pins_catch_planted_mask_mistakes(monkeypatch):
    """Plant plausible mask errors in the oracle and check the fixture pin fails."""
    rows = read_golden("mask_L6_M2.txt")
    want = np.array([[c == "1" for c in r.replace(" ", "")] for r in rows])
    good = O.bd_mask

    def inclusive_clean_for_corrupted(L, M):      # b_j <= b_i instead of <
        A = good(L, M)
        b = np.arange(L) // M
        A[L:, :L] = b[None, :] <= b[:, None]
        return A

    def token_causal_clean(L, M):                  # token-causal instead of block-causal
        A = good(L, M)
        A[:L, :L] = np.tri(L, dtype=bool)
        return A

    for bad in (inclusive_clean_for_corrupted, token_causal_clean):
        assert not np.array_equal(bad(6, 2), want)


def test_pins_catch_planted_backward_mistake(monkeypatch):
    """Dropping D from dS (a plausible slip) breaks the dK sum invariant."""
    real = O.masked_attention_bwd

    def no_D(q, k, v, allow, scale, do):
        dq, dk, dv, D = real(q, k, v, allow, scale, do)
        s = scale * (np.asarray(q) @ np.asarray(k).T)
        s = np.where(allow, s, -np.inf)
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        ds = p * (np.asarray(do) @ np.asarray(v).T)
        return scale * ds @ k, scale * ds.T @ q, dv, D

    monkeypatch.setattr(O, "masked_attention_bwd", no_D)
    L, M, d = 16, 4, 4
    t = make(L, 1, 1, d, seed=80)
    g = O.bd_attention_bwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"],
                           t["doc"], t["dox"], M, 0.5)
    dk = g["dk_clean"].sum(0) + g["dk_corr"].sum(0)
    assert np.abs(dk).max() > 1e-3


def test_lse_merge_of_parts_that_read_no_key():
    """A row every part left empty (z = -inf) merges to O = 0, z = -inf for
    any number of parts, as the two-part merge defines it; one empty part
    among others has weight 0."""
    o = np.array([[1.0, 2.0], [3.0, 4.0]])
    z = np.array([-np.inf, 0.5])
    for n in (1, 2, 3):
        om, zm = O.lse_merge([o] * n, [z] * n)
        assert np.all(om[0] == 0) and zm[0] == -np.inf
        np.testing.assert_allclose(om[1], o[1])
        np.testing.assert_allclose(zm[1], 0.5 + np.log(n))
    om, zm = O.lse_merge([o, 5 * o], [np.array([-np.inf, -np.inf]), z])
    np.testing.assert_allclose(om[1], 5 * o[1])
    assert zm[1] == 0.5
