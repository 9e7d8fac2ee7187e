"""CSBP's exchange layer (block_diffusion_lm_gb300.csbp_dist) on CPU process
groups: 2 and 4 gloo ranks on 127.0.0.1, no GPU.

* The shard layout comes from the library's schedule builder and equals the
  oracle's zigzag chunk ownership.
* The all-gather gives every rank the whole clean K/V copy, bit for bit, in
  sequence order; corrupted tensors are never sent.
* The reduce-scatter gives each rank, for the clean rows it owns, the sum of
  every rank's addend (exact on values representable in bf16).
* The whole orchestration -- gather, a per-rank attention over the rank's
  own query rows, reduce-scatter -- reproduces the float64 oracle of the
  unsharded sequence on every rank.  The per-rank attention is injected: the
  oracle on the rank's sequence-order buffers (rows the rank does not own
  hold zeros, so they add nothing), since a CPU test cannot run the
  library's kernels; the GPU tests run the same per-rank problems through
  the library.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from block_diffusion_lm_gb300 import csbp_dist as D
from oracle import csbp_oracle as O


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_lm_gb300 import build
    build.build()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _spawn(fn, world, *args):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_entry, args=(fn, r, world, port, q, args)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
    codes = [p.exitcode for p in procs]
    res = {}
    while not q.empty():
        r, v = q.get(timeout=10)
        res[r] = v
    assert codes == [0] * world, (codes, res)
    assert sorted(res) == list(range(world)), res
    for r, v in res.items():
        assert not (isinstance(v, str) and v.startswith("FAIL")), (r, v)
    return res


def _entry(fn, rank, world, port, q, args):
    import traceback

    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.set_num_threads(1)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, fn(rank, world, *args)))
    except Exception:  # reported to the parent, which fails the test
        q.put((rank, "FAIL " + traceback.format_exc()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("L,M,P", [(256, 8, 2), (512, 16, 4), (1024, 32, 4), (4096, 64, 8)])
def test_layout_is_the_oracle_zigzag_ownership(L, M, P):
    lay = D.ShardLayout.build(L, M, P, tile=32 if L // (2 * P) % 128 else 128)
    assert list(lay.chunk_owner) == list(O.chunk_owner(L, P))
    pos = np.concatenate([lay.positions_of(r) for r in range(P)])
    assert sorted(pos.tolist()) == list(range(L))          # a partition of the sequence
    for r in range(P):
        assert lay.chunks_of(r) == [r, 2 * P - 1 - r]
        # every corrupted block inside the rank's rows belongs to the rank
        blocks = np.unique(lay.positions_of(r) // M)
        assert set(O.block_owner(L, M, P)[blocks].tolist()) == {r}


def _gather_case(rank, world, L, M, Hkv, d):
    lay = D.ShardLayout.build(L, M, world, tile=32)
    g = torch.Generator().manual_seed(5)
    k = torch.randn(2, L, Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(2, L, Hkv, d, generator=g).to(torch.bfloat16)
    kf, vf = D.all_gather_clean_kv(lay, D.gather_local_rows(lay, rank, k),
                                   D.gather_local_rows(lay, rank, v))
    return "ok" if torch.equal(kf, k) and torch.equal(vf, v) else "FAIL gathered copy differs"


@pytest.mark.parametrize("world", [2, 4])
def test_all_gather_gives_every_rank_the_whole_clean_copy(world):
    _spawn(_gather_case, world, 512, 16, 2, 8)


def _rs_case(rank, world, L, M, Hkv, d):
    lay = D.ShardLayout.build(L, M, world, tile=32)
    # addends: small integers, exact in bf16 and in an fp32 sum
    addend = lambda r: torch.randint(-8, 9, (1, L, Hkv, d), generator=torch.Generator().manual_seed(100 + r))  # noqa: E731,E501
    dk = addend(rank).to(torch.bfloat16)
    dv = (2 * addend(rank)).to(torch.bfloat16)
    gk, gv = D.reduce_scatter_clean_grads(lay, dk, dv)
    total = sum(addend(r).to(torch.float64) for r in range(world))
    want_k = D.gather_local_rows(lay, rank, total)
    ok = torch.equal(gk.double(), want_k) and torch.equal(gv.double(), 2 * want_k)
    ok = ok and gk.dtype == torch.bfloat16 and gk.shape == (1, 2 * lay.chunk, Hkv, d)
    return "ok" if ok else "FAIL reduce-scatter sum differs"


@pytest.mark.parametrize("world", [2, 4])
def test_reduce_scatter_delivers_each_owner_the_sum_of_every_rank(world):
    _spawn(_rs_case, world, 512, 16, 2, 8)


class _OracleRankCompute:
    """A rank's attention on CPU, for the test: the float64 oracle over the
    rank's sequence-order buffers, rounded to bf16 like the library's
    outputs.  Rows the rank does not own hold zero q, K/V and dO there, so
    they contribute nothing to the clean dK/dV addend; only owned rows of
    O, LSE and dQ are read back."""

    def __init__(self, L, M, Hq, Hkv, d, scale, window=0, clean_causal=False):
        self.L, self.M, self.Hq, self.Hkv, self.d, self.scale = L, M, Hq, Hkv, d, scale
        self.window, self.clean_causal = window, clean_causal

    def alloc_outputs(self):
        sh = (1, self.L, self.Hq, self.d)
        return (torch.empty(sh, dtype=torch.bfloat16), torch.empty(sh, dtype=torch.bfloat16),
                torch.empty(1, 2, self.Hq, self.L))

    def alloc_grads(self):
        return {}

    def forward(self, t, out=None, stream=None):
        f = {k: (v[0].double().numpy() if v is not None else None) for k, v in t.items()}
        oc, ox, lse = O.bd_attention_fwd(f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"],
                                         f["k_corr"], f["v_corr"], self.M, self.scale,
                                         self.window, self.clean_causal)
        if oc is not None:
            out[0][0] = torch.from_numpy(oc).to(torch.bfloat16)
        out[1][0] = torch.from_numpy(ox).to(torch.bfloat16)
        out[2][0] = torch.from_numpy(lse).float()
        return (out[0] if oc is not None else None, out[1], out[2])

    def backward(self, t, out, grads=None, stream=None):
        f = {k: (v[0].double().numpy() if v is not None else None) for k, v in t.items()}
        g = O.bd_attention_bwd(f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"],
                               f["k_corr"], f["v_corr"], f["do_clean"], f["do_corr"], self.M,
                               self.scale, self.window, self.clean_causal)
        return {k: (torch.from_numpy(g[k])[None].to(torch.bfloat16) if g.get(k) is not None
                    else None)
                for k in ("dq_clean", "dq_corr", "dk_clean", "dv_clean", "dk_corr", "dv_corr")}


def _inputs(L, Hq, Hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    shapes = {"q_clean": Hq, "k_clean": Hkv, "v_clean": Hkv, "q_corr": Hq, "k_corr": Hkv,
              "v_corr": Hkv, "do_clean": Hq, "do_corr": Hq}
    return {k: torch.randn(1, L, h, d, generator=g).to(torch.bfloat16) for k, h in shapes.items()}


def _e2e_case(rank, world, L, M, Hq, Hkv, d, clean=True, window=0, causal=False):
    scale = d ** -0.5
    full = _inputs(L, Hq, Hkv, d, seed=9)
    if not clean:
        full["q_clean"] = full["do_clean"] = None
    node = D.CSBPRank(1, L, M, Hq, Hkv, d, world, rank, device="cpu",
                      compute=_OracleRankCompute(L, M, Hq, Hkv, d, scale, window, causal),
                      has_clean_queries=clean, window=window, clean_causal=causal)
    lay = node.layout
    local = {k: (D.gather_local_rows(lay, rank, v) if v is not None else None)
             for k, v in full.items()}
    oc, ox, lse = node.forward(local)
    grads = node.backward({"do_clean": local["do_clean"], "do_corr": local["do_corr"]})
    # the unsharded sequence, float64
    f = {k: (v[0].double().numpy() if v is not None else None) for k, v in full.items()}
    Oc, Ox, Z = O.bd_attention_fwd(f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"],
                                   f["k_corr"], f["v_corr"], M, scale, window, causal)
    G = O.bd_attention_bwd(f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"], f["k_corr"],
                           f["v_corr"], f["do_clean"], f["do_corr"], M, scale, window, causal)
    pos = lay.positions_of(rank)

    def rel(a, b):
        return float(np.linalg.norm(a - b) / np.linalg.norm(b))

    errs = {
        "o_corr": np.abs(ox[0].double().numpy() - Ox[pos]).max(),
        "lse": np.abs(lse[0, 1].double().numpy() - Z[1][:, pos]).max(),
    }
    names = ["dq_corr", "dk_corr", "dv_corr", "dk_clean", "dv_clean"]
    if clean:
        errs["o_clean"] = np.abs(oc[0].double().numpy() - Oc[pos]).max()
        errs["lse_clean"] = np.abs(lse[0, 0].double().numpy() - Z[0][:, pos]).max()
        names.append("dq_clean")
    else:
        assert oc is None and grads["dq_clean"] is None
    for k in names:
        errs[k] = rel(grads[k][0].double().numpy(), G[k][pos])
    bad = {k: v for k, v in errs.items() if not v <= (1e-3 if k.startswith("lse") else 1e-2)}
    return "ok" if not bad else f"FAIL {bad}"


@pytest.mark.parametrize("world", [2, 4])
def test_gather_rank_attention_reduce_scatter_equals_the_unsharded_oracle(world):
    _spawn(_e2e_case, world, 1024, 16, 4, 2, 16)


@pytest.mark.parametrize("world,clean,window,causal", [(2, False, 0, False), (4, True, 200, True)])
def test_exchange_layer_with_corrupted_queries_only_and_a_window(world, clean, window, causal):
    """The drafter shape (no clean queries: the clean copy is context only)
    and a sliding window with token-causal clean queries, through the same
    gather / per-rank attention / reduce-scatter."""
    _spawn(_e2e_case, world, 1024, 16, 4, 2, 16, clean, window, causal)


def test_layout_refuses_a_group_of_the_wrong_size():
    lay = D.ShardLayout.build(256, 8, 4, tile=32)
    res = _spawn(_wrong_size_case, 2, lay)
    assert all(v == "ok" for v in res.values())


def _wrong_size_case(rank, world, lay):
    try:
        D.all_gather_clean_kv(lay, torch.zeros(1, 64, 1, 8), torch.zeros(1, 64, 1, 8))
    except ValueError:
        return "ok"
    return "FAIL accepted a 2-rank group for a 4-shard layout"
