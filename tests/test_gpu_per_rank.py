"""GPU parity of the per-rank problems (csbp_problem.per_rank = 1): each CSBP
rank's query rows through the C-ABI, the ranks run one after another on one
GPU (no collective; the clean dK/dV addends are summed on the host, as the
owner reduce-scatter would).

Against the float64 oracle of the unsharded sequence:
* O, LSE and dQ of the rank's rows (the oracle's zigzag chunk owner), and its
  corrupted blocks' dK/dV, match the unsharded values;
* the rank's clean dK/dV addend matches the oracle's VJP with dO kept on the
  rank's rows only, and the addends of all ranks sum to the unsharded clean
  dK/dV;
* rows the rank does not own are never read: they hold NaN in q, dO and the
  corrupted K/V, and every result stays finite; dQ and the corrupted dK/dV
  of those rows come out zero.
Tolerances as in the other parity tests.
"""
import numpy as np
import pytest
import torch

from block_diffusion_lm_gb300 import csbp
from block_diffusion_lm_gb300.inputs import Workload, make_inputs, to_f64
from oracle import csbp_oracle as O

pytestmark = pytest.mark.gpu

TOL_O, TOL_REL, TOL_LSE = 1e-2, 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from block_diffusion_lm_gb300 import build
    build.build()


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


CASES = [
    (Workload("rank_p2", 1, 1024, 16, 4, 2, 128, seed=60), 2),
    (Workload("rank_p4", 1, 2048, 32, 4, 1, 128, seed=61), 4),
    (Workload("rank_drafter", 1, 1024, 16, 2, 1, 64, has_clean_queries=False, seed=62), 2),
    (Workload("rank_window", 1, 2048, 16, 4, 2, 128, window=300, clean_causal=True, seed=63), 4),
]


@pytest.mark.parametrize("w,P", CASES, ids=[c[0].name for c in CASES])
def test_ranks_reproduce_the_unsharded_sequence(w, P):
    t = make_inputs(w, "cuda")
    f = {k: (to_f64(v[0]) if v is not None else None) for k, v in t.items()}
    args = (f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"], f["k_corr"], f["v_corr"])
    Oc, Ox, Z = O.bd_attention_fwd(*args, w.M, w.scale, w.window, w.clean_causal)
    G = O.bd_attention_bwd(*args, f["do_clean"], f["do_corr"], w.M, w.scale, w.window,
                           w.clean_causal)
    C = w.L // (2 * P)
    co = O.chunk_owner(w.L, P)
    clean = w.has_clean_queries
    dk_sum = np.zeros_like(G["dk_clean"])
    dv_sum = np.zeros_like(G["dv_clean"])
    for r in range(P):
        mine = np.concatenate([np.arange(c * C, (c + 1) * C) for c in range(2 * P) if co[c] == r])
        other = np.setdiff1d(np.arange(w.L), mine)
        # rows the rank does not own: never read, so poison them
        tr = dict(t)
        for k in ("q_clean", "q_corr", "k_corr", "v_corr", "do_clean", "do_corr"):
            if tr[k] is not None:
                tr[k] = tr[k].clone()
                tr[k][:, torch.as_tensor(other, device="cuda")] = float("nan")
        attn = csbp.BlockDiffusionAttention(1, w.L, w.M, w.Hq, w.Hkv, w.d, P=P,
                                            has_clean_queries=clean, window=w.window,
                                            clean_causal=w.clean_causal, rank=r)
        oc, ox, lse = attn.forward(tr)
        g = attn.backward(tr, (oc, ox, lse))
        attn.check()
        torch.cuda.synchronize()
        # owned rows equal the unsharded sequence's
        assert np.abs(to_f64(ox[0])[mine] - Ox[mine]).max() <= TOL_O
        assert np.abs(to_f64(lse[0])[1][:, mine] - Z[1][:, mine]).max() <= TOL_LSE
        assert rel_fro(to_f64(g["dq_corr"][0])[mine], G["dq_corr"][mine]) <= TOL_REL
        if clean:
            assert np.abs(to_f64(oc[0])[mine] - Oc[mine]).max() <= TOL_O
            assert np.abs(to_f64(lse[0])[0][:, mine] - Z[0][:, mine]).max() <= TOL_LSE
            assert rel_fro(to_f64(g["dq_clean"][0])[mine], G["dq_clean"][mine]) <= TOL_REL
            assert np.all(to_f64(g["dq_clean"][0])[other] == 0)
        assert np.all(to_f64(g["dq_corr"][0])[other] == 0)
        for k in ("dk_corr", "dv_corr"):
            got = to_f64(g[k][0])
            assert rel_fro(got[mine], G[k][mine]) <= TOL_REL, k
            assert np.all(got[other] == 0), k
        # the rank's clean dK/dV addend: the VJP with dO on its rows only
        do_c = None if f["do_clean"] is None else f["do_clean"].copy()
        do_x = f["do_corr"].copy()
        do_x[other] = 0
        if do_c is not None:
            do_c[other] = 0
        Gr = O.bd_attention_bwd(*args, do_c, do_x, w.M, w.scale, w.window, w.clean_causal)
        for k in ("dk_clean", "dv_clean"):
            got = to_f64(g[k][0])
            assert np.isfinite(got).all(), k
            assert rel_fro(got, Gr[k]) <= TOL_REL, (k, r, rel_fro(got, Gr[k]))
        dk_sum += to_f64(g["dk_clean"][0])
        dv_sum += to_f64(g["dv_clean"][0])
    assert rel_fro(dk_sum, G["dk_clean"]) <= TOL_REL
    assert rel_fro(dv_sum, G["dv_clean"]) <= TOL_REL


def test_full_size_sharded_ranks_sampled():
    """The sharded workload (L = 65,536, P = 8) as eight ranks on one GPU:
    each rank's problem runs on the whole inputs with every row it does not
    own poisoned (NaN); its owned rows of O, LSE and dQ are checked on seeded
    samples against the oracle, and the eight clean dK/dV addends, summed as
    the owner reduce-scatter would (fp32), on seeded keys and through the
    exact whole-tensor invariants (sum_j dK_j = 0, sum_j dV_j = sum dO)."""
    from block_diffusion_lm_gb300.inputs import WORKLOADS
    w = WORKLOADS["sharded"]
    P = w.P
    t = make_inputs(w, "cuda")
    L = w.L
    C = L // (2 * P)
    co = O.chunk_owner(L, P)
    rng = np.random.default_rng(301)
    fv = {k: (_HostView(v[0].cpu()) if v is not None else None) for k, v in t.items()}
    dk_sum = torch.zeros(L, w.Hkv, w.d, dtype=torch.float32, device="cuda")
    dv_sum = torch.zeros_like(dk_sum)
    dk_corr_sum = torch.zeros_like(dk_sum)   # each rank writes its own blocks, zeros elsewhere
    dv_corr_sum = torch.zeros_like(dk_sum)
    corr_keys = []
    for r in range(P):
        mine = np.concatenate([np.arange(c * C, (c + 1) * C) for c in range(2 * P) if co[c] == r])
        other = torch.as_tensor(np.setdiff1d(np.arange(L), mine), device="cuda")
        tr = dict(t)
        for k in ("q_clean", "q_corr", "k_corr", "v_corr", "do_clean", "do_corr"):
            tr[k] = tr[k].clone()
            tr[k][:, other] = float("nan")
        attn = csbp.BlockDiffusionAttention(1, L, w.M, w.Hq, w.Hkv, w.d, P=P, rank=r)
        oc, ox, lse = attn.forward(tr)
        g = attn.backward(tr, (oc, ox, lse))
        attn.check()
        # owned rows: 4 per head, both copies
        samples = [(int(rng.integers(0, 2)), int(rng.choice(mine)), h)
                   for h in range(w.Hq) for _ in range(4)]
        ref = O.sampled_rows(fv["q_clean"], fv["k_clean"], fv["v_clean"], fv["q_corr"],
                             fv["k_corr"], fv["v_corr"], fv["do_clean"], fv["do_corr"], w.M,
                             w.scale, samples)
        dq_got, dq_want = [], []
        for (qs, i, h), (o, z, _, dq) in ref.items():
            og = (oc if qs == 0 else ox)[0, i, h].double().cpu().numpy()
            assert np.abs(og - o).max() <= TOL_O, (r, qs, i, h)
            assert abs(lse[0, qs, h, i].item() - z) <= TOL_LSE, (r, qs, i, h)
            dq_got.append(g["dq_clean" if qs == 0 else "dq_corr"][0, i, h].double().cpu().numpy())
            dq_want.append(dq)
        assert rel_fro(np.array(dq_got), np.array(dq_want)) <= TOL_REL, r
        assert torch.isfinite(g["dk_clean"]).all() and torch.isfinite(g["dv_clean"]).all()
        dk_sum += g["dk_clean"][0].float()
        dv_sum += g["dv_clean"][0].float()
        dk_corr_sum += g["dk_corr"][0].float()
        dv_corr_sum += g["dv_corr"][0].float()
        # corrupted keys of this rank's blocks: complete on this rank alone
        for _ in range(2):
            j = int(rng.choice(mine))
            gg = int(rng.integers(0, w.Hkv))
            corr_keys.append(((1, j, gg), g["dk_corr"][0, j, gg].double().cpu().numpy(),
                              g["dv_corr"][0, j, gg].double().cpu().numpy()))
        del tr, attn, g, oc, ox, lse
        torch.cuda.empty_cache()
    # the reduce-scattered clean dK/dV: late clean keys (readers: the last two
    # blocks) on seeded KV heads, plus the whole-tensor invariants
    keys = [(0, int(rng.integers(L - 2 * w.M, L - w.M)), int(rng.integers(0, w.Hkv)))
            for _ in range(4)] + [k for k, _, _ in corr_keys]
    kref = O.sampled_keys(fv["q_clean"], fv["k_clean"], fv["v_clean"], fv["q_corr"],
                          fv["k_corr"], fv["v_corr"], fv["do_clean"], fv["do_corr"], w.M, w.scale,
                          keys)
    got_k, want_k, got_v, want_v = [], [], [], []
    corr = {k: (a, b) for k, a, b in corr_keys}
    for (ks, j, gg), (dk, dv) in kref.items():
        if ks == 0:
            got_k.append(dk_sum[j, gg].double().cpu().numpy())
            got_v.append(dv_sum[j, gg].double().cpu().numpy())
        else:
            got_k.append(corr[(ks, j, gg)][0])
            got_v.append(corr[(ks, j, gg)][1])
        want_k.append(dk)
        want_v.append(dv)
    assert rel_fro(np.array(got_k), np.array(want_k)) <= TOL_REL
    assert rel_fro(np.array(got_v), np.array(want_v)) <= TOL_REL
    # exact whole-tensor invariants over every key of both copies:
    # sum_j dK_j = 0 and sum_j dV_j = sum of the group's dO rows
    G = w.Hq // w.Hkv
    dk_tot = dk_sum.double().sum(0) + dk_corr_sum.double().sum(0)
    dv_tot = dv_sum.double().sum(0) + dv_corr_sum.double().sum(0)
    do = (t["do_clean"][0].double().sum(0) + t["do_corr"][0].double().sum(0)).view(w.Hkv, G, w.d)
    do = do.sum(1)
    assert dk_tot.abs().max().item() <= 2e-3 * dk_sum.double().abs().sum(0).max().item()
    assert ((dv_tot - do).norm() / do.norm()).item() <= 1e-2


class _HostView:
    """bf16 host tensor [L, H, d] that hands the oracle float32 numpy slices."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        return self.t[idx].to(torch.float32).numpy()
