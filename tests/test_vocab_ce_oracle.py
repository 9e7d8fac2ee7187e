"""Pins for the LM-head cross-entropy oracle, against facts that do not come
from the oracle: a three-row example worked by hand, torch's own cross-entropy and autograd in float64, the
zero-head closed form, shift invariance, exact invariants, central finite
differences, ignored rows, and a planted mistake the torch pin must catch."""
import numpy as np
import pytest
import torch

from oracle import vocab_ce_oracle as C
from conftest import read_golden


def make(N, Dm, V, seed, ignore=0.0, sigma=None):
    r = np.random.default_rng(seed)
    H = r.standard_normal((N, Dm))
    W = r.standard_normal((V, Dm)) * (sigma if sigma is not None else 2.0 / np.sqrt(Dm))
    t = r.integers(0, V, N)
    if ignore > 0:
        t[r.random(N) < ignore] = -1
    return H, W, t


@pytest.mark.parametrize("N,Dm,V,ignore,head", [(7, 5, 11, 0.0, True), (33, 16, 64, 0.3, True),
                                                (20, 8, 40, 0.5, False), (64, 24, 300, 0.0, True)])
def test_matches_torch_cross_entropy_and_autograd(N, Dm, V, ignore, head):
    H, W, t = make(N, Dm, V, seed=N + V, ignore=ignore, sigma=0.7)
    s = 1.0 / max(1, int((t >= 0).sum()))
    loss, lse, dH, dW = C.vocab_ce(H, W, t, s, head_grad=head)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    z = Ht @ Wt.T
    ref = torch.nn.functional.cross_entropy(z, torch.tensor(t), ignore_index=-1, reduction="none")
    np.testing.assert_allclose(loss, ref.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(z, dim=1).detach().numpy(), atol=1e-12)
    (s * ref.sum()).backward()
    np.testing.assert_allclose(dH, Ht.grad.numpy(), atol=1e-12)
    if head:
        np.testing.assert_allclose(dW, Wt.grad.numpy(), atol=1e-12)
    else:
        assert dW is None


def test_matches_hand_worked_fixture():
    """Three rows (one ignored) over a three-word vocabulary whose logits are
    logs of small integers, worked out by hand."""
    lines = [[float(x) for x in ln.split()] for ln in read_golden("vocab_ce_three_rows.txt")]
    W = np.array(lines[0])[:, None]
    s = lines[1][0]
    rows = np.array(lines[2:5])
    H, t = rows[:, :1], rows[:, 1].astype(np.int64)
    loss, lse, dH, dW = C.vocab_ce(H, W, t, s)
    np.testing.assert_allclose(lse, rows[:, 2], atol=1e-14)
    np.testing.assert_allclose(loss, rows[:, 3], atol=1e-14)
    np.testing.assert_allclose(dH[:, 0], rows[:, 4], atol=1e-14)
    np.testing.assert_allclose(dW[:, 0], lines[5], atol=1e-14)
    l2, z2, d2 = C.vocab_ce_rows(H, W, t, s, [2, 0])
    np.testing.assert_allclose(z2, rows[[2, 0], 2], atol=1e-14)
    np.testing.assert_allclose(l2, rows[[2, 0], 3], atol=1e-14)
    np.testing.assert_allclose(d2[:, 0], rows[[2, 0], 4], atol=1e-14)


def test_zero_head_closed_form():
    """W = 0: every logit is 0, so lse = loss = ln V, dH = 0 and
    dW_v = s sum_i (1/V - [t_i = v]) h_i."""
    N, Dm, V, s = 12, 6, 9, 0.25
    H, _, t = make(N, Dm, V, seed=3)
    loss, lse, dH, dW = C.vocab_ce(H, np.zeros((V, Dm)), t, s)
    np.testing.assert_allclose(lse, np.log(V), atol=1e-14)
    np.testing.assert_allclose(loss, np.log(V), atol=1e-14)
    np.testing.assert_array_equal(dH, 0.0)
    want = np.zeros((V, Dm))
    for i in range(N):
        want += H[i] / V
        want[t[i]] -= H[i]
    np.testing.assert_allclose(dW, s * want, atol=1e-13)


def test_shift_of_every_head_row_moves_lse_not_loss():
    """Adding one vector u to every row of W adds h_i.u to all logits of row
    i: lse moves by h_i.u, loss and dH do not change."""
    H, W, t = make(16, 8, 30, seed=5)
    u = np.random.default_rng(6).standard_normal(8)
    a = C.vocab_ce(H, W, t, 0.1)
    b = C.vocab_ce(H, W + u, t, 0.1)
    np.testing.assert_allclose(b[1] - a[1], H @ u, atol=1e-12)
    np.testing.assert_allclose(b[0], a[0], atol=1e-12)
    np.testing.assert_allclose(b[2], a[2], atol=1e-12)


def test_gradient_invariants():
    """Each row's softmax minus one-hot sums to 0: sum_v dW_v = 0 and
    dH_i = s (E_p[W] - W_t)."""
    H, W, t = make(40, 12, 70, seed=7, ignore=0.2)
    s = 0.5
    _, lse, dH, dW = C.vocab_ce(H, W, t, s)
    np.testing.assert_allclose(dW.sum(axis=0), 0.0, atol=1e-12)
    P = np.exp(H @ W.T - lse[:, None])
    for i in range(40):
        want = s * (P[i] @ W - W[t[i]]) if t[i] >= 0 else np.zeros(12)
        np.testing.assert_allclose(dH[i], want, atol=1e-12)


def test_central_finite_differences():
    N, Dm, V, s = 6, 4, 10, 0.3
    H, W, t = make(N, Dm, V, seed=8, sigma=0.8)
    t[2] = -1
    _, _, dH, dW = C.vocab_ce(H, W, t, s)

    def f(Hx, Wx):
        return s * C.vocab_ce(Hx, Wx, t, s, head_grad=False)[0].sum()

    eps = 1e-6
    rng = np.random.default_rng(9)
    for _ in range(12):
        i, k = rng.integers(0, N), rng.integers(0, Dm)
        Hp, Hm = H.copy(), H.copy()
        Hp[i, k] += eps
        Hm[i, k] -= eps
        assert abs((f(Hp, W) - f(Hm, W)) / (2 * eps) - dH[i, k]) < 1e-8
        v = rng.integers(0, V)
        Wp, Wm = W.copy(), W.copy()
        Wp[v, k] += eps
        Wm[v, k] -= eps
        assert abs((f(H, Wp) - f(H, Wm)) / (2 * eps) - dW[v, k]) < 1e-8


def test_ignored_rows_contribute_nothing():
    H, W, t = make(24, 8, 50, seed=10)
    t2 = t.copy()
    t2[[1, 5, 6]] = -1
    loss, _, dH, dW = C.vocab_ce(H, W, t2, 0.2)
    assert np.all(loss[[1, 5, 6]] == 0) and np.all(dH[[1, 5, 6]] == 0)
    keep = np.setdiff1d(np.arange(24), [1, 5, 6])
    _, _, _, dW_keep = C.vocab_ce(H[keep], W, t[keep], 0.2)
    np.testing.assert_allclose(dW, dW_keep, atol=1e-13)


def test_targets_past_the_vocabulary_are_ignored_rows():
    """A target >= V reads as an ignored row: the same outputs as target -1,
    and dW as if the row were absent."""
    H, W, t = make(20, 6, 30, seed=12)
    a, b = t.copy(), t.copy()
    a[[2, 9, 17]] = [30, 31, 10 ** 6]
    b[[2, 9, 17]] = -1
    ra = C.vocab_ce(H, W, a, 0.3)
    rb = C.vocab_ce(H, W, b, 0.3)
    for x, y in zip(ra, rb):
        np.testing.assert_array_equal(x, y)
    assert np.all(ra[0][[2, 9, 17]] == 0) and np.all(ra[2][[2, 9, 17]] == 0)
    keep = np.setdiff1d(np.arange(20), [2, 9, 17])
    np.testing.assert_allclose(ra[3], C.vocab_ce(H[keep], W, t[keep], 0.3)[3], atol=1e-13)


def test_sampled_rows_equal_the_full_evaluation():
    H, W, t = make(50, 8, 64, seed=11, ignore=0.2)
    loss, lse, dH, _ = C.vocab_ce(H, W, t, 0.1)
    rows = [0, 7, 49, 13]
    l2, z2, d2 = C.vocab_ce_rows(H, W, t, 0.1, rows)
    np.testing.assert_allclose(l2, loss[rows], atol=1e-13)
    np.testing.assert_allclose(z2, lse[rows], atol=1e-13)
    np.testing.assert_allclose(d2, dH[rows], atol=1e-13)


def test_torch_pin_catches_a_planted_missing_one_hot(monkeypatch):
    """An oracle that forgets to subtract the one-hot target from the
    softmax gives dH = s E_p[W]: the autograd pin must fail."""
    real_exp = np.exp

    def vocab_ce_no_onehot(H, W, target, grad_scale, head_grad=True):
        H = np.asarray(H, np.float64)
        W = np.asarray(W, np.float64)
        Z = H @ W.T
        m = Z.max(axis=1, keepdims=True)
        lse = (m + np.log(real_exp(Z - m).sum(axis=1, keepdims=True)))[:, 0]
        rows = np.arange(H.shape[0])
        loss = lse - Z[rows, target]
        G = grad_scale * real_exp(Z - lse[:, None])
        return loss, lse, G @ W, G.T @ H

    monkeypatch.setattr(C, "vocab_ce", vocab_ce_no_onehot)
    with pytest.raises(AssertionError):
        test_matches_torch_cross_entropy_and_autograd(7, 5, 11, 0.0, True)
