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
