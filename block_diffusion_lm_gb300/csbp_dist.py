"""CSBP's exchange layer: one process per GPU, each owning one rank's shard.

The method ("CSBP 完全拆解" blog, section "在线 softmax 合并：为什么分两段算仍是同一个
注意力", implementation schedule; Turbo-dLLM project page, section "Library",
row "Collectives") exchanges exactly two things between ranks:

* forward: an all-gather of every rank's clean K/V shard, so each rank holds
  the whole clean copy (the clean prefix any of its corrupted blocks reads);
* backward: a reduce-scatter of the clean dK/dV, summed over the ranks whose
  queries read each clean key and delivered to the key's owner.

Corrupted Q/K/V and their gradients never move: a corrupted block is read
only by its own queries, which live on the same rank.

Ownership is the library's (csbp_block_schedule): the clean sequence is cut
into 2P chunks of L/(2P) tokens, rank r owns chunks r and 2P-1-r (dual-end
pairing, "负载均衡：为什么要首尾块配对"), and a corrupted block belongs to the
owner of the chunk that holds it.  A rank's local tensors hold its two
chunks back to back, [batch, 2C, H, d] with C = L/(2P), chunk r first.

Each rank computes with the library's per-rank problem (csbp_problem
per_rank = 1): its query rows against the gathered clean copy and its own
corrupted blocks.  The collectives are plain torch.distributed calls
(all_gather_into_tensor, reduce_scatter_tensor); the clean dK/dV addends are
summed in fp32 and rounded to bf16 once, at the owner.  The gathered K/V and
the full-length buffers the per-rank kernels address are placed in
sequence order on every rank (L positions, owned rows filled in, the rest
never read by that rank's kernels).

What runs here is host orchestration only; every step of the attention runs
in the library's kernels.  The data movement is exercised by CPU process
groups (gloo) in the tests; on GPUs the same calls run over NCCL.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import csbp


@dataclass(frozen=True)
class ShardLayout:
    """Who owns which clean chunk: from the library's schedule builder."""

    L: int
    M: int
    P: int
    chunk_owner: tuple  # owner rank of each of the 2P clean chunks

    @staticmethod
    def build(L: int, M: int, P: int, tile: int = 128) -> "ShardLayout":
        prob = csbp.make_problem(1, L, M, 1, 1, 64, P=P, tile=tile)
        _, co, _, _ = csbp.block_schedule(prob)
        return ShardLayout(L, M, P, tuple(int(x) for x in co))

    @property
    def chunk(self) -> int:
        return self.L // (2 * self.P)

    def chunks_of(self, rank: int):
        """The two chunks rank owns, in local order."""
        return [c for c in range(2 * self.P) if self.chunk_owner[c] == rank]

    def positions_of(self, rank: int) -> np.ndarray:
        """Sequence positions of the rank's local rows, in local order."""
        C = self.chunk
        return np.concatenate([np.arange(c * C, (c + 1) * C) for c in self.chunks_of(rank)])


def _ranks(group):
    import torch.distributed as dist
    return dist.get_rank(group), dist.get_world_size(group)


def scatter_local_rows(layout: ShardLayout, rank: int, local, full):
    """Write a rank's local rows [batch, 2C, ...] into a sequence-order
    buffer [batch, L, ...] (the other rows are left as they are)."""
    C = layout.chunk
    for n, c in enumerate(layout.chunks_of(rank)):
        full[:, c * C:(c + 1) * C] = local[:, n * C:(n + 1) * C]
    return full


def gather_local_rows(layout: ShardLayout, rank: int, full):
    """The rank's local rows [batch, 2C, ...] of a sequence-order tensor."""
    import torch
    C = layout.chunk
    return torch.cat([full[:, c * C:(c + 1) * C] for c in layout.chunks_of(rank)], dim=1)


def all_gather_clean_kv(layout: ShardLayout, k_local, v_local, group=None):
    """Forward exchange: every rank's clean K and V shards [batch, 2C, Hkv, d]
    -> the whole clean copy [batch, L, Hkv, d] on every rank, in sequence
    order (one all-gather of K and V packed together)."""
    import torch
    import torch.distributed as dist
    rank, world = _ranks(group)
    if world != layout.P:
        raise ValueError(f"the group has {world} ranks, the layout {layout.P} shards")
    kv = torch.stack([k_local, v_local]).contiguous()           # [2, b, 2C, Hkv, d]
    # the collective concatenates the ranks' tensors along dim 0
    got = torch.empty((world * 2,) + tuple(kv.shape[1:]), dtype=kv.dtype, device=kv.device)
    dist.all_gather_into_tensor(got, kv, group=group)
    got = got.view((world,) + tuple(kv.shape))
    b, _, Hkv, d = k_local.shape
    full = torch.empty((2, b, layout.L, Hkv, d), dtype=kv.dtype, device=kv.device)
    C = layout.chunk
    for r in range(world):
        for n, c in enumerate(layout.chunks_of(r)):
            full[:, :, c * C:(c + 1) * C] = got[r, :, :, n * C:(n + 1) * C]
    return full[0], full[1]


def reduce_scatter_clean_grads(layout: ShardLayout, dk_full, dv_full, group=None):
    """Backward exchange: this rank's addend of the clean dK and dV for the
    whole clean copy [batch, L, Hkv, d] -> the sums over every rank of the
    rows this rank owns [batch, 2C, Hkv, d] (one reduce-scatter in fp32, the
    result rounded to the addends' dtype once)."""
    import torch
    import torch.distributed as dist
    rank, world = _ranks(group)
    if world != layout.P:
        raise ValueError(f"the group has {world} ranks, the layout {layout.P} shards")
    # destination-major: block s holds the rows rank s owns, in its local order
    send = torch.stack([torch.stack([gather_local_rows(layout, s, dk_full),
                                     gather_local_rows(layout, s, dv_full)])
                        for s in range(world)]).to(torch.float32).contiguous()
    recv = torch.empty(send.shape[1:], dtype=torch.float32, device=send.device)
    # the collective splits its input along dim 0, one slice per rank
    dist.reduce_scatter_tensor(recv, send.view((-1,) + tuple(send.shape[2:])), group=group)
    return recv[0].to(dk_full.dtype), recv[1].to(dv_full.dtype)


class CSBPRank:
    """One rank of a CSBP job: local shards in, local outputs and gradients
    out, with the two exchanges around the library's per-rank kernels.

    Local tensors are [batch, 2C, H, d] bf16 (the rank's two chunks, chunk
    `rank` first): q/k/v and dO of both copies (no clean q / dO without clean
    queries).  forward() returns the local (o_clean or None, o_corr,
    lse [batch, 2, Hq, 2C]); backward() the local dQ of the query copies, the
    local corrupted dK/dV, and the clean dK/dV of the rows this rank owns
    summed over all ranks.
    """

    def __init__(self, batch, L, M, Hq, Hkv, d, P, rank, group=None, device="cuda",
                 scale=None, compute=None, has_clean_queries=True, window=0,
                 clean_causal=False):
        """`compute`: the per-rank attention (forward / backward /
        alloc_outputs / alloc_grads of csbp.BlockDiffusionAttention); by
        default the library's, for this rank's query rows."""
        import torch
        self.layout = ShardLayout.build(L, M, P)
        self.rank, self.group = rank, group
        self.has_clean = has_clean_queries
        self.attn = compute if compute is not None else csbp.BlockDiffusionAttention(
            batch, L, M, Hq, Hkv, d, P=P, scale=scale, device=device, rank=rank,
            has_clean_queries=has_clean_queries, window=window, clean_causal=clean_causal)
        q_shape, kv_shape = (batch, L, Hq, d), (batch, L, Hkv, d)
        z = lambda s: torch.zeros(s, dtype=torch.bfloat16, device=device)  # noqa: E731
        # sequence-order buffers the per-rank kernels address (rows the rank
        # does not own are never read)
        self.full = {"q_corr": z(q_shape), "k_corr": z(kv_shape), "v_corr": z(kv_shape),
                     "do_corr": z(q_shape)}
        if has_clean_queries:
            self.full["q_clean"] = z(q_shape)
            self.full["do_clean"] = z(q_shape)
        self.out = self.attn.alloc_outputs()
        self.grads = self.attn.alloc_grads()

    def forward(self, local: dict, stream=None):
        lay, r = self.layout, self.rank
        k_full, v_full = all_gather_clean_kv(lay, local["k_clean"], local["v_clean"], self.group)
        for n in ("q_clean", "q_corr", "k_corr", "v_corr"):
            if n in self.full:
                scatter_local_rows(lay, r, local[n], self.full[n])
        self.inputs = {**{n: self.full.get(n) for n in ("q_clean", "q_corr", "k_corr", "v_corr")},
                       "k_clean": k_full, "v_clean": v_full}
        oc, ox, lse = self.attn.forward(self.inputs, out=self.out, stream=stream)
        C = lay.chunk
        lse_local = np.concatenate([np.arange(c * C, (c + 1) * C) for c in lay.chunks_of(r)])
        return (gather_local_rows(lay, r, oc) if oc is not None else None,
                gather_local_rows(lay, r, ox), lse[..., lse_local])

    def backward(self, local_do: dict, stream=None):
        lay, r = self.layout, self.rank
        for n in ("do_clean", "do_corr"):
            if n in self.full:
                scatter_local_rows(lay, r, local_do[n], self.full[n])
        t = {**self.inputs, "do_clean": self.full.get("do_clean"), "do_corr": self.full["do_corr"]}
        g = self.attn.backward(t, self.out, grads=self.grads, stream=stream)
        dk, dv = reduce_scatter_clean_grads(lay, g["dk_clean"], g["dv_clean"], self.group)
        local = {n: (gather_local_rows(lay, r, g[n]) if g.get(n) is not None else None)
                 for n in ("dq_clean", "dq_corr", "dk_corr", "dv_corr")}
        local["dk_clean"], local["dv_clean"] = dk, dv
        return local
