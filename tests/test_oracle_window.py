"""Pins for the oracle's sliding-window and token-causal clean options, against
facts that do not come from the oracle: a mask worked out by hand, reductions
to textbook causal and sliding-window attention (torch SDPA in float64 with a
band mask built from triangles), a window too wide to matter, a one-token
window, finite differences, and a planted off-by-one window that the SDPA pin
must catch.

Reading (where the pages only name 1,024-token sliding-window layers): a
window W keeps, of the keys the block rules allow, those less than W positions
before the query (positions within each copy).
"""
import numpy as np
import pytest
import torch

from oracle import csbp_oracle as O
from conftest import read_golden


def make(L, Hq, Hkv, d, seed=0, clean=True):
    r = np.random.default_rng(seed)
    t = {n: r.standard_normal((L, Hq if n.startswith(("q", "do")) else Hkv, d))
         for n in ("qc", "kc", "vc", "qx", "kx", "vx", "doc", "dox")}
    if not clean:
        t["qc"] = None
        t["doc"] = None
    return t


def band(L, W):
    """Textbook sliding-window causal mask: key j <= query i and j > i - W."""
    ones = torch.ones(L, L, dtype=torch.bool)
    return torch.tril(ones) & ~torch.tril(ones, diagonal=-W)


def sdpa(q, k, v, mask, scale):
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=mask[None], scale=scale)[0].numpy()


def test_windowed_masks_match_hand_written_fixture():
    """Both clean-query variants, every scalar predicate and every row agree
    with a mask worked out by hand (L=8, M=4, W=3)."""
    rows = read_golden("mask_L8_M4_W3.txt")
    want = np.array([[c == "1" for c in r.replace(" ", "")] for r in rows])
    assert want.shape == (32, 16)
    for k, causal in enumerate((False, True)):
        ref = want[16 * k:16 * (k + 1)]
        np.testing.assert_array_equal(O.bd_mask(8, 4, 3, causal), ref)
        for qs in (0, 1):
            for i in range(8):
                np.testing.assert_array_equal(O.mask_row(qs, i, 8, 4, 3, causal), ref[qs * 8 + i])
                for ks in (0, 1):
                    for j in range(8):
                        assert O.allowed(qs, i, ks, j, 4, 3, causal) == ref[qs * 8 + i, ks * 8 + j]


@pytest.mark.parametrize("W", [1, 3, 7, 40])
def test_token_causal_windowed_clean_stream_is_textbook_sliding_window(W):
    L, d, scale = 24, 5, 0.5
    t = make(L, 1, 1, d, seed=W)
    Oc, _, _ = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], M=4,
                                  scale=scale, window=W, clean_causal=True)
    ref = sdpa(t["qc"][:, 0], t["kc"][:, 0], t["vc"][:, 0], band(L, W), scale)
    np.testing.assert_allclose(Oc[:, 0], ref, atol=1e-13)


@pytest.mark.parametrize("W", [2, 5, 11])
def test_unit_blocks_windowed_corrupted_row_is_own_token_plus_window_of_clean(W):
    """M = 1: corrupted row i reads its own token and the clean tokens
    i-W+1 .. i-1: SDPA over [clean; own] keys with the band mask shifted by one."""
    L, d, scale = 20, 4, 0.6
    t = make(L, 1, 1, d, seed=30 + W)
    _, Ox, _ = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], M=1,
                                  scale=scale, window=W)
    for i in range(L):
        lo = max(0, i - W + 1)
        keys = np.concatenate([t["kc"][lo:i, 0], t["kx"][i:i + 1, 0]])
        vals = np.concatenate([t["vc"][lo:i, 0], t["vx"][i:i + 1, 0]])
        ref = sdpa(t["qx"][i:i + 1, 0], keys, vals, torch.ones(1, len(keys), dtype=torch.bool),
                   scale)
        np.testing.assert_allclose(Ox[i, 0], ref[0], atol=1e-13)


def test_block_rules_stay_under_token_causal_with_unit_blocks():
    """With M = 1 block-causal and token-causal clean attention coincide."""
    assert np.array_equal(O.bd_mask(12, 1), O.bd_mask(12, 1, clean_causal=True))
    A, C = O.bd_mask(16, 4), O.bd_mask(16, 4, clean_causal=True)
    assert np.all(C <= A) and np.any(A & ~C)


@pytest.mark.parametrize("clean_causal", [False, True])
def test_window_wider_than_the_sequence_changes_nothing(clean_causal):
    L, M = 32, 4
    t = make(L, 2, 1, 4, seed=5)
    a = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], M, 0.4,
                           clean_causal=clean_causal)
    b = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], M, 0.4,
                           window=2 * L, clean_causal=clean_causal)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_one_token_window_leaves_each_row_its_own_key_and_later_block_keys():
    """W = 1 bounds only how far back a key may lie: a clean (token-causal)
    row reads only itself, so O = V and LSE = scale q.k; a corrupted row
    reads its own token and the later tokens of its block (bidirectional),
    so the last row of each block reads only itself."""
    L, M, d, scale = 16, 4, 6, 0.3
    t = make(L, 2, 2, d, seed=9)
    Oc, Ox, lse = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], M,
                                     scale, window=1, clean_causal=True)
    np.testing.assert_allclose(Oc, t["vc"], atol=1e-13)
    np.testing.assert_allclose(lse[0], scale * np.einsum("lhd,lhd->hl", t["qc"], t["kc"]),
                               atol=1e-13)
    for i in range(L):
        end = (i // M + 1) * M
        for h in range(2):
            ref = sdpa(t["qx"][i:i + 1, h], t["kx"][i:end, h], t["vx"][i:end, h],
                       torch.ones(1, end - i, dtype=torch.bool), scale)
            np.testing.assert_allclose(Ox[i, h], ref[0], atol=1e-13)
        if end == i + 1:
            np.testing.assert_allclose(Ox[i], t["vx"][i], atol=1e-13)


@pytest.mark.parametrize("W,causal,clean", [(3, False, True), (6, True, True), (5, False, False)])
def test_windowed_backward_matches_central_finite_differences(W, causal, clean):
    L, M, Hq, Hkv, d, scale = 16, 4, 2, 1, 4, 0.6
    t = make(L, Hq, Hkv, d, seed=40 + W, clean=clean)

    def f(tt):
        Oc, Ox, _ = O.bd_attention_fwd(tt["qc"], tt["kc"], tt["vc"], tt["qx"], tt["kx"],
                                       tt["vx"], M, scale, W, causal)
        val = (Ox * tt["dox"]).sum()
        if clean:
            val += (Oc * tt["doc"]).sum()
        return val

    g = O.bd_attention_bwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], t["doc"],
                           t["dox"], M, scale, W, causal)
    names = {"qx": "dq_corr", "kc": "dk_clean", "vc": "dv_clean", "kx": "dk_corr", "vx": "dv_corr"}
    if clean:
        names["qc"] = "dq_clean"
    rng = np.random.default_rng(1)
    eps = 1e-5
    for src, gname in names.items():
        for _ in range(5):
            idx = tuple(rng.integers(0, s) for s in t[src].shape)
            tp = {k: (None if v is None else v.copy()) for k, v in t.items()}
            tm = {k: (None if v is None else v.copy()) for k, v in t.items()}
            tp[src][idx] += eps
            tm[src][idx] -= eps
            fd = (f(tp) - f(tm)) / (2 * eps)
            an = g[gname][idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (src, idx, fd, an)


def test_windowed_sampled_rows_and_keys_agree_with_full_oracle():
    L, M, W = 32, 4, 9
    t = make(L, 2, 1, 4, seed=77)
    Oc, Ox, lse = O.bd_attention_fwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], M,
                                     0.5, W, True)
    g = O.bd_attention_bwd(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], t["doc"],
                           t["dox"], M, 0.5, W, True)
    rows = [(0, 3, 0), (1, 17, 1), (0, 31, 1), (1, 0, 0)]
    got = O.sampled_rows(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], t["doc"],
                         t["dox"], M, 0.5, rows, W, True)
    for (qs, i, h), (o, z, _, dq) in got.items():
        np.testing.assert_allclose(o, (Oc if qs == 0 else Ox)[i, h], atol=1e-12)
        np.testing.assert_allclose(z, lse[qs, h, i], atol=1e-12)
        np.testing.assert_allclose(dq, g["dq_clean" if qs == 0 else "dq_corr"][i, h], atol=1e-12)
    keys = [(0, 30, 0), (1, 5, 0), (0, 2, 0)]
    got = O.sampled_keys(t["qc"], t["kc"], t["vc"], t["qx"], t["kx"], t["vx"], t["doc"],
                         t["dox"], M, 0.5, keys, W, True, chunk_rows=4)
    for (ks, j, gg), (dk, dv) in got.items():
        np.testing.assert_allclose(dk, g["dk_clean" if ks == 0 else "dk_corr"][j, gg], atol=1e-12)
        np.testing.assert_allclose(dv, g["dv_clean" if ks == 0 else "dv_corr"][j, gg], atol=1e-12)


def test_window_pair_count_matches_the_mask():
    for L, M, W, causal, clean in [(64, 4, 7, False, True), (64, 8, 5, True, True),
                                   (96, 4, 13, False, False), (128, 16, 100, True, True)]:
        A = O.bd_mask(L, M, W, causal)
        n = int(A[L:].sum()) + (int(A[:L].sum()) if clean else 0)
        assert n == O.allowed_pairs_per_head(L, M, clean, W, causal)


def test_sdpa_pin_catches_a_planted_off_by_one_window(monkeypatch):
    """An oracle whose window keeps i - j <= W (one key too many) fails the
    textbook sliding-window pin."""
    good = O.bd_mask

    def inclusive_window(L, M, window=0, clean_causal=False):
        return good(L, M, window + 1 if window > 0 else 0, clean_causal)

    monkeypatch.setattr(O, "bd_mask", inclusive_window)
    with pytest.raises(AssertionError):
        test_token_causal_windowed_clean_stream_is_textbook_sliding_window(3)
