"""The allocation-free backward entry point (csbp_attn_bwd_noalloc).

It exists for callers that cannot call cudaMalloc (plugin or custom-op
interfaces that receive only input and output buffers, runtimes whose memory
pool forbids outside allocations, paths that cannot take cudaMalloc's
implicit device synchronisation): its scratch is a fixed 64 MiB array in the
library's device memory instead of a caller workspace.  These tests call it
through the C-ABI and check it, on two calls in a row, against the regular
entry point (csbp_attn_bwd with a caller workspace) and against the float64
oracle, so stale contents left in the shared scratch by the first call would
show up in the second; after each call its own status query must report no
timed-out device wait.  This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_diffusion_lm_gb300 import csbp
from block_diffusion_lm_gb300.inputs import Workload, make_inputs, to_f64
from oracle import csbp_oracle as O

TOL_REL = 1e-2


@pytest.fixture(scope="module")
def _lib():
    from block_diffusion_lm_gb300 import build
    build.build()
    return csbp.lib()


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward_on_two_calls(_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = Workload("noalloc", 1, 1024, 32, 4, 2, 128, seed=41)
    t = make_inputs(w, "cuda")
    attn = csbp.BlockDiffusionAttention(1, w.L, w.M, w.Hq, w.Hkv, w.d)
    assert csbp.workspace_bytes(attn.problem, 1) <= 64 << 20
    out = attn.forward(t)
    ref = attn.backward(t, out)
    attn.check()
    torch.cuda.synchronize()
    f = {k: to_f64(v[0]) for k, v in t.items()}
    want = O.bd_attention_bwd(f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"],
                              f["k_corr"], f["v_corr"], f["do_clean"], f["do_corr"], w.M, w.scale)
    for _ in range(2):
        g = attn.alloc_grads()
        for v in g.values():
            v.fill_(float("nan"))
        csbp.attn_bwd_noalloc(attn.problem, t, attn.work_dev, attn.info, out[0], out[1], out[2],
                              t["do_clean"], t["do_corr"], g)
        csbp.attn_bwd_noalloc_status()  # synchronises; raises on a timed-out wait
        for k, r in ref.items():
            a, b = g[k].double(), r.double()
            assert torch.isfinite(a).all(), k
            assert ((a - b).norm() / b.norm()).item() <= TOL_REL, k
            got = to_f64(g[k][0])
            assert np.linalg.norm(got - want[k]) / np.linalg.norm(want[k]) <= TOL_REL, k


def test_noalloc_rejects_problems_beyond_its_scratch(_lib):
    """A problem needing more than the 64 MiB scratch is refused before any
    CUDA call (so this runs without a GPU too)."""
    prob = csbp.make_problem(1, 65536, 64, 32, 8, 128)
    assert csbp.workspace_bytes(prob, 1) > 64 << 20
    info = csbp.ScheduleInfo()
    st = _lib.csbp_attn_bwd_noalloc(ctypes.byref(prob), None, None, ctypes.byref(info),
                                    *([None] * 11), None)
    assert st == -3  # CSBP_ERR_WORKSPACE
