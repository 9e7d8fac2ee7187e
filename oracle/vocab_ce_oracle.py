"""Float64 CPU oracle for the streamed LM-head cross-entropy.

TEST INFRASTRUCTURE ONLY: tests, the package's smoke check and the benchmark's
CPU-baseline leg call this module; the library never does, and nothing here
is shared with the CUDA path.

What it computes ([Project] "Library", tables "Speculative Decoding
Optimizations" and "Block Diffusion Optimizations", row "Vocabulary loss":
rows are streamed through the LM head in token chunks and the cross-entropy
is taken without the full-sequence logits ever existing; for the drafter the
head is frozen):

    z_i      = W h_i                         logits of row i over the vocabulary
    lse_i    = log sum_v exp(z_iv)
    loss_i   = lse_i - z_{i, t_i}            (0 for an ignored row: t_i outside [0, V))
    g_i      = s (softmax(z_i) - e_{t_i})     (0 for an ignored row)
    dH_i     = g_i W                          gradient of s * sum_i loss_i
    dW       = sum_i g_i^T h_i                (only when the head is trained)

with s the caller's gradient scale (for example 1 / number of counted rows).
The pages give no target encoding.  The reading here is the usual
ignore-index convention, widened to every value outside [0, V): negative
targets (padding, the clean half of a block-diffusion sequence) and any
target past the vocabulary.

The chunking is a memory schedule, not part of the arithmetic, so the oracle
has none.  Every row's outputs depend on that row alone, which is what lets
the tests evaluate sampled rows of full-size problems one by one.
"""
import numpy as np


def vocab_ce(H, W, target, grad_scale, head_grad=True):
    """Loss, LSE, dH and (optionally) dW for rows H [N, Dm] against the head
    W [V, Dm] with integer targets [N] (outside [0, V) = ignored row).

    Returns (loss [N], lse [N], dH [N, Dm], dW [V, Dm] or None), float64.
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    t = np.asarray(target, dtype=np.int64)
    n = H.shape[0]
    Z = H @ W.T
    m = Z.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(Z - m).sum(axis=1, keepdims=True)))[:, 0]
    valid = (t >= 0) & (t < W.shape[0])
    rows = np.arange(n)
    zt = np.where(valid, Z[rows, np.where(valid, t, 0)], 0.0)
    loss = np.where(valid, lse - zt, 0.0)
    G = np.exp(Z - lse[:, None])
    G[rows[valid], t[valid]] -= 1.0
    G[~valid] = 0.0
    G *= grad_scale
    dH = G @ W
    dW = G.T @ H if head_grad else None
    return loss, lse, dH, dW


def vocab_ce_rows(H, W, target, grad_scale, rows):
    """loss, lse and dH of the listed rows only (each row stands alone)."""
    rows = np.asarray(rows, dtype=np.int64)
    loss, lse, dH, _ = vocab_ce(np.asarray(H[rows], dtype=np.float64), W,
                                np.asarray(target)[rows], grad_scale, head_grad=False)
    return loss, lse, dH
