"""Float64 CPU oracle for two-copy block-diffusion attention (CSBP per-rank math).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module; only the test suite, the smoke check and the CPU-baseline
leg of the benchmark use it.  It shares no code with the CUDA library.

Every function is the plain definition written out in float64 NumPy, in the
order and notation of the pages it follows (the row- and key-sampled
evaluators for long sequences use float64 PyTorch CPU ops, which run their
element-wise passes on every host core):

* [Blog] "CSBP 完全拆解：块并行如何让长上下文扩散语言模型少传无效 KV"
  (pinghaoyang.com.cn), sections
    - "块扩散模型到底多了哪一种并行机会"  (block partition x = (x^(1)..x^(B)),
      M = L/B, factorisation p(x) = prod_b p(x^(b) | x^(<b)))
    - "传统上下文并行为什么会传错东西"  (O_r = softmax(Q_r K^T / sqrt(d_h) + M_r) V;
      a corrupted query of block b needs exactly [K_b; K^clean_<b], [V_b; V^clean_<b])
    - "BP：把损坏块留在本地"  (L_r = sum_{b in B_r} L_b, sum_r grad L_r = grad L)
    - "CSBP：BP 管损坏块，CP 管干净上下文"  (O_b = Attn(Q_b, [K_b; K^clean_<b],
      [V_b; V^clean_<b]); corrupted grads stay local, clean dK/dV go to the
      clean-shard owner)
    - "在线 softmax 合并：为什么分两段算仍是同一个注意力"  (m = max(z1, z2),
      w_i = e^(z_i - m), O = (w1 O1 + w2 O2)/(w1 + w2), z = m + log(w1 + w2))
    - "负载均衡：为什么要首尾块配对"  (block b paired with block B+1-b;
      zigzag pairing of early and late clean chunks)
* [Project] "Block Parallelism for Efficient Distributed Long-Context Diffusion
  Language Model Training" (Turbo-dLLM project page), sections "Method"
  (corrupted K/V are read only by their own block) and "Load balancing:
  pairing early and late blocks" (block b and block B+1-b share a rank; the
  same early-late pairing shards the clean sequence; every pair does
  identical work).
* [Wiki] "CSBP: stop sharding by token position, start sharding by what the
  loss actually needs", "TL;DR" (a length-L example runs as 2L positions: a
  clean copy and a corrupted copy).

Readings taken where the pages are silent (each is also listed in the design
notes): clean queries attend block-causally over the clean copy (b_j <= b_i);
clean queries never read corrupted keys; GQA maps query head h to KV head
h // (Hq / Hkv); the LSE is the natural log of the softmax denominator; blocks
map to shards through 2P contiguous clean chunks, shard r owning chunks r and
2P-1-r; a sharded forward takes one partial per clean shard plus one "own"
(corrupted own-block) partial for every query row.

Positions are 0-based inside each copy; block id blk(i) = i // M.
Stream 0 = clean copy, stream 1 = corrupted copy.
"""
from __future__ import annotations

import numpy as np

CLEAN = 0
CORR = 1


# --------------------------------------------------------------------------
# Mask  ([Blog] "传统上下文并行为什么会传错东西" and "CSBP：BP 管损坏块，CP 管干净上下文";
#        [Project] "Method")
# --------------------------------------------------------------------------
def allowed(q_stream: int, i: int, k_stream: int, j: int, M: int, window: int = 0,
            clean_causal: bool = False) -> bool:
    """Scalar mask predicate: may query (q_stream, i) read key (k_stream, j)?

    corrupted q -> corrupted k : same block (bidirectional inside the block)
    corrupted q -> clean k     : strictly earlier block  (K^clean_<b)
    clean q     -> clean k     : same or earlier block   (block-causal reading);
                                 with clean_causal, j <= i (token-causal)
    clean q     -> corrupted k : never (corrupted K/V are read by their own
                                 block only)

    window > 0 keeps, of those keys, the ones less than `window` positions
    before the query (i - j < window, positions within each copy): the
    sliding-window attention layers of [Blog] "实验数字：256K 上下文下的主结果"
    (25 of DiffusionGemma's 30 layers use a 1,024-token window) and [Project]
    "Where does the time go? Attention traffic at 256K"; reading: the window
    bounds only how far back a key may lie, the block rules above still apply.
    """
    bi, bj = i // M, j // M
    if q_stream == CORR and k_stream == CORR:
        ok = bj == bi
    elif q_stream == CORR and k_stream == CLEAN:
        ok = bj < bi
    elif q_stream == CLEAN and k_stream == CLEAN:
        ok = (j <= i) if clean_causal else (bj <= bi)
    else:
        ok = False
    return ok and (window <= 0 or i - j < window)


def bd_mask(L: int, M: int, window: int = 0, clean_causal: bool = False) -> np.ndarray:
    """Explicit boolean mask A[2L, 2L] over (query, key) positions.

    Rows/cols 0..L-1 are the clean copy, L..2L-1 the corrupted copy.  Built
    from the block ids (and positions) by broadcasting the cases of `allowed`.
    """
    if L % M != 0:
        raise ValueError("L must be a multiple of the block size M")
    pos = np.arange(L)
    b = pos // M
    bq, bk = b[:, None], b[None, :]
    A = np.zeros((2 * L, 2 * L), dtype=bool)
    if clean_causal:
        A[:L, :L] = pos[None, :] <= pos[:, None]   # clean q, clean k (token-causal)
    else:
        A[:L, :L] = bk <= bq                        # clean q, clean k (block-causal)
    A[:L, L:] = False             # clean q, corrupted k
    A[L:, :L] = bk < bq           # corrupted q, clean k
    A[L:, L:] = bk == bq          # corrupted q, corrupted k
    if window > 0:
        near = (pos[:, None] - pos[None, :]) < window
        A &= np.tile(near, (2, 2))
    return A


def mask_row(q_stream: int, i: int, L: int, M: int, window: int = 0,
             clean_causal: bool = False) -> np.ndarray:
    """Row (q_stream, i) of `bd_mask`, length 2L (clean keys then corrupted)."""
    pos = np.arange(L)
    b = pos // M
    bi = i // M
    row = np.zeros(2 * L, dtype=bool)
    if q_stream == CLEAN:
        row[:L] = (pos <= i) if clean_causal else (b <= bi)
    else:
        row[:L] = b < bi
        row[L:] = b == bi
    if window > 0:
        near = (i - pos) < window
        row[:L] &= near
        row[L:] &= near
    return row


# --------------------------------------------------------------------------
# Scaled softmax attention over an explicit mask
# ([Blog] "传统上下文并行为什么会传错东西": O = softmax(Q K^T / sqrt(d_h) + M) V)
# --------------------------------------------------------------------------
def masked_attention(q, k, v, allow, scale):
    """q [Nq,d], k/v [Nk,d], allow [Nq,Nk] bool -> (O [Nq,d], lse [Nq]).

    Rows with no allowed key get O = 0 and lse = -inf (an empty part of a
    partition; used by the sharded forward).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    s = scale * (q @ k.T)
    s = np.where(allow, s, -np.inf)
    m = s.max(axis=1)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    p = np.exp(s - m_safe[:, None])            # exp(-inf) = 0 off the mask
    l = p.sum(axis=1)
    l_safe = np.where(empty, 1.0, l)
    o = (p @ v) / l_safe[:, None]
    o[empty] = 0.0
    lse = np.where(empty, -np.inf, m_safe + np.log(l_safe))
    return o, lse


def masked_attention_bwd(q, k, v, allow, scale, do):
    """Analytic VJP of `masked_attention` for upstream gradient dO.

    P = softmax(S), dV = P^T dO, dP = dO V^T, D_i = sum_j P_ij dP_ij,
    dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
    Returns (dQ, dK, dV, D).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    s = scale * (q @ k.T)
    s = np.where(allow, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    p = e / np.where(l > 0, l, 1.0)
    dv = p.T @ do
    dp = do @ v.T
    D = (p * dp).sum(axis=1)
    ds = p * (dp - D[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, D


# --------------------------------------------------------------------------
# Two-copy block-diffusion attention, multi-head with GQA
# --------------------------------------------------------------------------
def _stack_streams(x_clean, x_corr):
    """[L,H,d] clean and corrupted -> [2L,H,d] (clean first)."""
    return np.concatenate([np.asarray(x_clean, np.float64),
                           np.asarray(x_corr, np.float64)], axis=0)


def bd_attention_fwd(qc, kc, vc, qx, kx, vx, M, scale, window=0, clean_causal=False):
    """Full forward of two-copy block-diffusion attention.

    Inputs [L, H, d] (H = Hq for q, Hkv for k/v); qc may be None for the
    corrupted-queries-only (drafter) workload.  Returns
    (Oc [L,Hq,d] or None, Ox [L,Hq,d], lse [2,Hq,L] with NaN rows for an absent
    clean query stream).
    """
    L, Hkv, d = np.shape(kc)
    Hq = np.shape(qx)[1]
    G = Hq // Hkv
    A = bd_mask(L, M, window, clean_causal)
    K = _stack_streams(kc, kx)
    V = _stack_streams(vc, vx)
    has_clean = qc is not None
    Oc = np.zeros((L, Hq, d)) if has_clean else None
    Ox = np.zeros((L, Hq, d))
    lse = np.full((2, Hq, L), np.nan)
    for h in range(Hq):
        g = h // G
        if has_clean:
            o, z = masked_attention(np.asarray(qc, np.float64)[:, h], K[:, g], V[:, g],
                                    A[:L], scale)
            Oc[:, h], lse[0, h] = o, z
        o, z = masked_attention(np.asarray(qx, np.float64)[:, h], K[:, g], V[:, g],
                                A[L:], scale)
        Ox[:, h], lse[1, h] = o, z
    return Oc, Ox, lse


def bd_attention_bwd(qc, kc, vc, qx, kx, vx, doc, dox, M, scale, window=0, clean_causal=False):
    """Analytic backward of `bd_attention_fwd`.

    Returns dict with dq_clean, dq_corr, dk_clean, dv_clean, dk_corr, dv_corr
    (dK/dV summed over the G query heads of each KV head) and D [2,Hq,L].
    Clean dK/dV collect contributions from clean queries (same or later block)
    and corrupted queries (later blocks); corrupted dK/dV only from queries of
    their own block ([Blog] "CSBP：BP 管损坏块，CP 管干净上下文", backward paragraph).
    """
    L, Hkv, d = np.shape(kc)
    Hq = np.shape(qx)[1]
    G = Hq // Hkv
    A = bd_mask(L, M, window, clean_causal)
    K = _stack_streams(kc, kx)
    V = _stack_streams(vc, vx)
    has_clean = qc is not None
    if has_clean:
        Q = _stack_streams(qc, qx)
        dO = _stack_streams(doc, dox)
        rows = slice(0, 2 * L)
    else:
        Q = np.concatenate([np.zeros((L, Hq, d)), np.asarray(qx, np.float64)], 0)
        dO = np.concatenate([np.zeros((L, Hq, d)), np.asarray(dox, np.float64)], 0)
        rows = slice(L, 2 * L)
    dQ = np.zeros((2 * L, Hq, d))
    dK = np.zeros((2 * L, Hkv, d))
    dV = np.zeros((2 * L, Hkv, d))
    D = np.full((2, Hq, L), np.nan)
    for h in range(Hq):
        g = h // G
        dq, dk, dv, Dh = masked_attention_bwd(Q[rows, h], K[:, g], V[:, g], A[rows],
                                              scale, dO[rows, h])
        dQ[rows, h] = dq
        dK[:, g] += dk
        dV[:, g] += dv
        if has_clean:
            D[0, h], D[1, h] = Dh[:L], Dh[L:]
        else:
            D[1, h] = Dh
    return {
        "dq_clean": dQ[:L] if has_clean else None, "dq_corr": dQ[L:],
        "dk_clean": dK[:L], "dv_clean": dV[:L],
        "dk_corr": dK[L:], "dv_corr": dV[L:], "D": D,
    }


# --------------------------------------------------------------------------
# Log-sum-exp merge  ([Blog] "在线 softmax 合并：为什么分两段算仍是同一个注意力")
# --------------------------------------------------------------------------
def lse_merge_pair(o1, z1, o2, z2):
    """Merge two normalised partial outputs over disjoint key sets.

    m = max(z1, z2); w_i = exp(z_i - m); O = (w1 O1 + w2 O2) / (w1 + w2);
    z = m + log(w1 + w2).  A part with z = -inf has w = 0 (it read no key).
    o* [rows, ...], z* [rows].
    """
    z1 = np.asarray(z1, np.float64)
    z2 = np.asarray(z2, np.float64)
    m = np.maximum(z1, z2)
    both_empty = ~np.isfinite(m)
    m_safe = np.where(both_empty, 0.0, m)
    w1 = np.exp(z1 - m_safe)
    w2 = np.exp(z2 - m_safe)
    wsum = w1 + w2
    wsum_safe = np.where(both_empty, 1.0, wsum)
    shape = (-1,) + (1,) * (np.ndim(o1) - 1)
    o = (w1.reshape(shape) * o1 + w2.reshape(shape) * o2) / wsum_safe.reshape(shape)
    o = np.where(both_empty.reshape(shape), 0.0, o)
    z = np.where(both_empty, -np.inf, m_safe + np.log(wsum_safe))
    return o, z


def lse_merge(o_parts, z_parts):
    """Merge n partials by applying the two-part merge left to right.  A row
    that no part read a key for (every z = -inf) merges to O = 0, z = -inf,
    the two-part rule's convention, also when n = 1."""
    o, z = np.asarray(o_parts[0], np.float64), np.asarray(z_parts[0], np.float64)
    for s in range(1, len(o_parts)):
        o, z = lse_merge_pair(o, z, np.asarray(o_parts[s], np.float64), z_parts[s])
    empty = ~np.isfinite(z)
    o = np.where(empty.reshape((-1,) + (1,) * (np.ndim(o) - 1)), 0.0, o)
    return o, z


# --------------------------------------------------------------------------
# Block / clean-chunk ownership: dual-end pairing and zigzag clean sharding
# ([Blog] "负载均衡：为什么要首尾块配对"; [Project] "Load balancing: pairing early
#  and late blocks")
# --------------------------------------------------------------------------
def chunk_owner(L: int, P: int) -> np.ndarray:
    """Owner shard of each of the 2P contiguous clean chunks (length L/(2P)).

    Shard r owns chunk r and chunk 2P-1-r: the early/late (zigzag) pairing.
    """
    if L % (2 * P) != 0:
        raise ValueError("L must be a multiple of 2P")
    owner = np.empty(2 * P, dtype=np.int32)
    for r in range(P):
        owner[r] = r
        owner[2 * P - 1 - r] = r
    return owner


def block_owner(L: int, M: int, P: int) -> np.ndarray:
    """Owner shard of each corrupted block: the owner of the clean chunk that
    holds the block's first position.  With B % 2P == 0 this pairs block b
    with block B-1-b (0-based), i.e. the pages' b with B+1-b (1-based)."""
    B = L // M
    if L % M != 0 or B % (2 * P) != 0:
        raise ValueError("need L % M == 0 and B % 2P == 0")
    cl = L // (2 * P)
    co = chunk_owner(L, P)
    return np.array([co[(b * M) // cl] for b in range(B)], dtype=np.int32)


def pair_counts_per_owner(L, M, P, owner_of_block, has_clean_queries=True):
    """Allowed (query, key) pairs charged to each owner when owner r computes
    every query row of the blocks it owns (both copies), over all keys."""
    B = L // M
    counts = np.zeros(P, dtype=np.int64)
    for b in range(B):
        r = owner_of_block[b]
        # corrupted queries of block b: M own + b*M clean keys each
        counts[r] += M * (M + b * M)
        if has_clean_queries:
            # clean queries of block b: (b+1)*M clean keys each
            counts[r] += M * ((b + 1) * M)
    return counts


def pair_counts_from_mask(L, M, P, owner_of_block, has_clean_queries=True):
    """Brute-force version of `pair_counts_per_owner` from the explicit mask."""
    A = bd_mask(L, M)
    counts = np.zeros(P, dtype=np.int64)
    per_row = A.sum(axis=1)
    for i in range(L):
        r = owner_of_block[i // M]
        if has_clean_queries:
            counts[r] += per_row[i]
        counts[r] += per_row[L + i]
    return counts


# --------------------------------------------------------------------------
# Sharded forward: per-part partial attention merged by LSE
# ([Blog] "在线 softmax 合并" implementation schedule steps 2-4, generalised to
#  one partial per clean shard plus the corrupted own-block part)
# --------------------------------------------------------------------------
def key_parts(L: int, P: int) -> np.ndarray:
    """Part id of each of the 2L keys: clean key j -> owner of its chunk,
    corrupted key -> part P ("own")."""
    co = chunk_owner(L, P)
    cl = L // (2 * P)
    part = np.empty(2 * L, dtype=np.int32)
    part[:L] = co[np.arange(L) // cl]
    part[L:] = P
    return part


def bd_attention_fwd_sharded(qc, kc, vc, qx, kx, vx, M, scale, P, window=0, clean_causal=False):
    """Forward via P+1 partials per query row and the LSE merge.

    Returns (Oc, Ox, lse, partials) where partials = (o_parts [P+1,2,L,Hq,d],
    z_parts [P+1,2,Hq,L]); a part that holds no allowed key of a row has
    z = -inf and O = 0.
    """
    L, Hkv, d = np.shape(kc)
    Hq = np.shape(qx)[1]
    G = Hq // Hkv
    A = bd_mask(L, M, window, clean_causal)
    K = _stack_streams(kc, kx)
    V = _stack_streams(vc, vx)
    part = key_parts(L, P)
    has_clean = qc is not None
    o_parts = np.zeros((P + 1, 2, L, Hq, d))
    z_parts = np.full((P + 1, 2, Hq, L), -np.inf)
    streams = [(CLEAN, qc), (CORR, qx)] if has_clean else [(CORR, qx)]
    for s in range(P + 1):
        in_part = part == s
        for st, q in streams:
            rows = A[:L] if st == CLEAN else A[L:]
            for h in range(Hq):
                g = h // G
                o, z = masked_attention(np.asarray(q, np.float64)[:, h], K[:, g], V[:, g],
                                        rows & in_part[None, :], scale)
                o_parts[s, st, :, h] = o
                z_parts[s, st, h] = z
    Oc = np.zeros((L, Hq, d)) if has_clean else None
    Ox = np.zeros((L, Hq, d))
    lse = np.full((2, Hq, L), np.nan)
    for st in ([CLEAN, CORR] if has_clean else [CORR]):
        for h in range(Hq):
            o, z = lse_merge([o_parts[s, st, :, h] for s in range(P + 1)],
                             [z_parts[s, st, h] for s in range(P + 1)])
            if st == CLEAN:
                Oc[:, h] = o
            else:
                Ox[:, h] = o
            lse[st, h] = z
    return Oc, Ox, lse, (o_parts, z_parts)


# --------------------------------------------------------------------------
# Tile schedule derived from the mask
# --------------------------------------------------------------------------
def tile_pairs(L, M, Tq, Tkv, P=1, has_clean_queries=True, window=0, clean_causal=False):
    """Set of (q_stream, q_tile, kv_stream, kv_tile, full, part) over every
    (query-tile, key-tile) pair holding at least one allowed entry.

    full = every entry of the tile is allowed.  part = owner shard of the
    clean chunk holding the key tile (clean keys) or P (corrupted keys).
    Requires Tkv to divide L/(2P) so a key tile lies in one chunk.
    """
    if (L // (2 * P)) % Tkv != 0 and P > 1:
        raise ValueError("Tkv must divide L/(2P)")
    A = bd_mask(L, M, window, clean_causal)
    if P == 1:
        part = np.concatenate([np.zeros(L, np.int32), np.ones(L, np.int32)])
    else:
        part = key_parts(L, P)
    nq = -(-L // Tq)
    nk = -(-L // Tkv)
    out = set()
    qstreams = [CLEAN, CORR] if has_clean_queries else [CORR]
    for qs in qstreams:
        for qt in range(nq):
            r0, r1 = qs * L + qt * Tq, qs * L + min((qt + 1) * Tq, L)
            for ks in (CLEAN, CORR):
                for kt in range(nk):
                    c0, c1 = ks * L + kt * Tkv, ks * L + min((kt + 1) * Tkv, L)
                    blk = A[r0:r1, c0:c1]
                    if blk.any():
                        out.add((qs, qt, ks, kt, bool(blk.all()), int(part[c0])))
    return out


# --------------------------------------------------------------------------
# Row / key sampled evaluation for long sequences
#
# The same definitions as `masked_attention` / `masked_attention_bwd`, for a
# subset of rows or keys of sequences too long for the explicit 2L x 2L mask.
# They run in float64 PyTorch CPU ops, whose element-wise passes use every
# host core (the NumPy ones run on one), on chunks of rows at a time.
# --------------------------------------------------------------------------
def mask_rows(rows, L: int, M: int, window: int = 0, clean_causal: bool = False) -> np.ndarray:
    """Rows [(q_stream, i)] of `bd_mask` as one bool array [len(rows), 2L]
    (the rules of `mask_row`, evaluated for all the rows at once)."""
    qs = np.array([r[0] for r in rows], dtype=np.int64)[:, None]
    i = np.array([r[1] for r in rows], dtype=np.int64)[:, None]
    pos = np.arange(L, dtype=np.int64)[None, :]
    b, bi = pos // M, i // M
    clean_rule = (pos <= i) if clean_causal else (b <= bi)
    left = np.where(qs == CLEAN, clean_rule, b < bi)           # clean keys
    right = (qs == CORR) & (b == bi)                           # corrupted keys
    if window > 0:
        near = (i - pos) < window
        left &= near
        right &= near
    return np.concatenate([left, right], axis=1)


def _kv_of_head(kc, kx, vc, vx, g):
    """[2L, d] float64 K and V of KV head g, clean keys first."""
    K = np.concatenate([np.asarray(kc[:, g], np.float64), np.asarray(kx[:, g], np.float64)], 0)
    V = np.concatenate([np.asarray(vc[:, g], np.float64), np.asarray(vx[:, g], np.float64)], 0)
    return K, V


def _gather_rows(qc, qx, doc, dox, rows, h):
    """Query and dO vectors [len(rows), d] of rows [(q_stream, i)] for query
    head h (one indexing per copy)."""
    n = len(rows)
    d = np.shape(qx)[2]
    q = np.empty((n, d))
    do = np.empty((n, d))
    for stream, (qsrc, dsrc) in ((CLEAN, (qc, doc)), (CORR, (qx, dox))):
        at = [n_ for n_, (qs, _) in enumerate(rows) if qs == stream]
        if at:
            idx = np.array([rows[n_][1] for n_ in at], dtype=np.int64)
            q[at] = np.asarray(qsrc[idx, h], np.float64)
            do[at] = np.asarray(dsrc[idx, h], np.float64)
    return q, do


def _t64(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))


def _tbool(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=bool))


def _softmax_rows_t(q, K, V, allow, scale, want_p=True):
    """`masked_attention` in float64 torch for rows with at least one allowed
    key: q [n,d], K/V [m,d], allow [n,m] bool -> (P [n,m] or None, O [n,d],
    lse [n])."""
    s = (q @ K.T) * scale
    s.masked_fill_(~allow, float("-inf"))
    m = s.amax(dim=1, keepdim=True)
    e = s.sub_(m).exp_()               # exp(-inf) = 0 off the mask
    l = e.sum(dim=1, keepdim=True)
    o = (e @ V) / l
    return (e.div_(l) if want_p else None), o, (m + l.log()).squeeze(1)


def _default_chunk(L):
    """Rows per chunk so that a chunk's [rows, 2L] float64 arrays stay
    within about 1 GB each."""
    return int(max(8, min(1024, (1 << 27) // (2 * L))))


def _chunk_keys(allow, K, V, L):
    """The keys a chunk of mask rows may read: in each copy, the range from
    its first to its last allowed key (keys inside the range that no row
    reads stay masked).  Returns (K_u, V_u, allow_u) as torch tensors."""
    import torch
    parts = []
    for c in (0, 1):
        hit = np.flatnonzero(allow[:, c * L:(c + 1) * L].any(axis=0))
        if hit.size:
            parts.append((c * L + int(hit[0]), c * L + int(hit[-1]) + 1))
    Ku = torch.cat([K[a:b] for a, b in parts])
    Vu = torch.cat([V[a:b] for a, b in parts])
    au = np.concatenate([allow[:, a:b] for a, b in parts], axis=1)
    return Ku, Vu, _tbool(au)


def sampled_rows(qc, kc, vc, qx, kx, vx, doc, dox, M, scale, samples, window=0,
                 clean_causal=False, chunk_rows=None):
    """Exact O, lse, D and dQ for sampled query rows.

    samples: iterable of (q_stream, i, h).  Each row depends only on itself,
    the full K/V of its KV head and dO_i: P_i = softmax over its allowed keys,
    O_i = P_i V, D_i = dO_i . O_i, dS_ij = P_ij (dO_i . v_j - D_i),
    dQ_i = scale sum_j dS_ij k_j.  Rows of one head go through in chunks
    against the keys some row of the chunk may read.  Returns dict keyed by
    the sample tuple -> (o [d], lse, D, dq [d]).
    """
    L, Hkv, d = np.shape(kc)
    Hq = np.shape(qx)[1]
    G = Hq // Hkv
    chunk_rows = chunk_rows or _default_chunk(L)
    by_head = {}
    for (qs, i, h) in samples:
        by_head.setdefault(h, []).append((qs, i))
    out = {}
    for g in range(Hkv):
        heads = [h for h in range(g * G, (g + 1) * G) if h in by_head]
        if not heads:
            continue
        K, V = (_t64(x) for x in _kv_of_head(kc, kx, vc, vx, g))
        for h in heads:
            rows_h = by_head[h]
            for c0 in range(0, len(rows_h), chunk_rows):
                rows = rows_h[c0:c0 + chunk_rows]
                allow = mask_rows(rows, L, M, window, clean_causal)
                Ku, Vu, au = _chunk_keys(allow, K, V, L)
                q, do = (_t64(x) for x in _gather_rows(qc, qx, doc, dox, rows, h))
                p, o, lse = _softmax_rows_t(q, Ku, Vu, au, scale)
                D = (do * o).sum(dim=1)
                ds = p * (do @ Vu.T - D[:, None])
                dq = scale * (ds @ Ku)
                for r, (qs, i) in enumerate(rows):
                    out[(qs, i, h)] = (o[r].numpy(), float(lse[r]), float(D[r]), dq[r].numpy())
        del K, V
    return out


def readers_of_key(k_stream, j, L, M, has_clean_queries=True, window=0, clean_causal=False):
    """All query rows (q_stream, i) whose mask row allows key (k_stream, j)."""
    bj = j // M
    out = []
    if k_stream == CORR:
        out += [(CORR, i) for i in range(bj * M, (bj + 1) * M)]
    else:
        if has_clean_queries:
            out += [(CLEAN, i) for i in range(bj * M, L)]
        out += [(CORR, i) for i in range((bj + 1) * M, L)]
    if window > 0 or clean_causal:  # the block rules above give a superset
        out = [(qs, i) for qs, i in out if allowed(qs, i, k_stream, j, M, window, clean_causal)]
    return out


def sampled_keys(qc, kc, vc, qx, kx, vx, doc, dox, M, scale, samples, window=0,
                 clean_causal=False, chunk_rows=None):
    """Exact dK, dV for sampled keys (k_stream, j, g).

    dK_j = scale sum_i dS_ij q_i and dV_j = sum_i P_ij dO_i, summed over every
    query row i that reads key j and over the G query heads of KV head g, with
    P_ij = exp(S_ij - lse_i), dP_ij = dO_i . v_j, D_i = dO_i . O_i (the same
    sum_j P_ij dP_ij as in `masked_attention_bwd`, since O_i = sum_j P_ij v_j)
    and dS_ij = P_ij (dP_ij - D_i).  Each reader's lse_i and O_i come from its
    own complete masked softmax, so the union of the sampled keys' readers
    goes through in chunks of `chunk_rows` rows, each against the keys that
    some row of the chunk may read (the other columns of its mask rows are
    all False).  The cost is that of the readers' full rows: an early clean
    key is read by almost every row of the sequence.
    """
    import torch
    L, Hkv, d = np.shape(kc)
    Hq = np.shape(qx)[1]
    G = Hq // Hkv
    has_clean = qc is not None
    chunk_rows = chunk_rows or _default_chunk(L)
    by_g = {}
    for (ks, j, g) in samples:
        by_g.setdefault(g, []).append((ks, j))
    out = {}
    for g, keys in by_g.items():
        readers = sorted({r for ks, j in keys
                          for r in readers_of_key(ks, j, L, M, has_clean, window, clean_causal)})
        K, V = (_t64(x) for x in _kv_of_head(kc, kx, vc, vx, g))
        cols = np.array([ks * L + j for ks, j in keys], dtype=np.int64)
        Kc, Vc = K[cols], V[cols]
        dk = torch.zeros(len(keys), d, dtype=torch.float64)
        dv = torch.zeros(len(keys), d, dtype=torch.float64)
        for c0 in range(0, len(readers), chunk_rows):
            rows = readers[c0:c0 + chunk_rows]
            allow = mask_rows(rows, L, M, window, clean_causal)
            Ku, Vu, au = _chunk_keys(allow, K, V, L)
            ac = _tbool(allow[:, cols])
            for h in range(g * G, (g + 1) * G):
                q, do = (_t64(x) for x in _gather_rows(qc, qx, doc, dox, rows, h))
                _, o, lse = _softmax_rows_t(q, Ku, Vu, au, scale, want_p=False)
                D = (do * o).sum(dim=1)
                p = torch.where(ac, ((q @ Kc.T) * scale - lse[:, None]).exp(),
                                torch.zeros((), dtype=torch.float64))
                ds = p * (do @ Vc.T - D[:, None])
                dk += scale * (ds.T @ q)
                dv += p.T @ do
        for n, (ks, j) in enumerate(keys):
            out[(ks, j, g)] = (dk[n].numpy(), dv[n].numpy())
        del K, V
    return out


# --------------------------------------------------------------------------
# fp8 inputs: OCP 8-bit floating point, variant E4M3
# (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
#  holds the subnormals; no infinities; S.1111.111 is NaN)
# --------------------------------------------------------------------------
def e4m3_value(code: int) -> float:
    """The real number an E4M3 byte encodes, from the format definition."""
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 array -> the nearest bfloat16 values (ties to even), as
    float64: keep the top 16 bits of the float32 pattern after adding half an
    ulp of bf16 plus the tie-breaking bit; NaN stays NaN."""
    x = np.asarray(x, np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    out = rounded.astype(np.uint32).view(np.float32).astype(np.float64)
    out[np.isnan(x)] = np.nan
    return out


def e4m3_to_bf16(codes, scale: float) -> np.ndarray:
    """bf16 values (as float64) of scale * value(code): the product in fp32
    (one IEEE multiply of two fp32 numbers is the exact product rounded to
    fp32), then rounded to bf16, nearest even."""
    table = np.array([e4m3_value(c) for c in range(256)], np.float64)
    v = table[np.asarray(codes, np.uint8)]
    prod = (v.astype(np.float32) * np.float32(scale)).astype(np.float32)
    return round_to_bf16(prod)


# --------------------------------------------------------------------------
# Useful (mask-allowed) work
# ([Blog] "CSBP：BP 管损坏块，CP 管干净上下文": CP and CSBP compute the same legal
#  pairs, Theta(L^2) in total)
# --------------------------------------------------------------------------
def allowed_pairs_per_head(L, M, has_clean_queries=True, window=0, clean_causal=False):
    """Number of allowed (query, key) pairs for one query head."""
    B = L // M
    if window <= 0 and not clean_causal:
        corr = sum(M * (M + b * M) for b in range(B))
        clean = sum(M * ((b + 1) * M) for b in range(B)) if has_clean_queries else 0
        return corr + clean
    # per query row, each key set is one range of positions [lo, hi)
    i = np.arange(L, dtype=np.int64)
    b = i // M
    w_lo = np.maximum(0, i - window + 1) if window > 0 else np.zeros(L, np.int64)
    n = np.maximum(0, b * M - w_lo)                                   # corrupted q, clean k
    n += np.maximum(0, (b + 1) * M - np.maximum(b * M, w_lo))         # corrupted q, own block
    if has_clean_queries:
        hi = (i + 1) if clean_causal else (b + 1) * M
        n += np.maximum(0, hi - w_lo)                                 # clean q, clean k
    return int(n.sum())
