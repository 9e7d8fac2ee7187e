"""The allocation-free backward entry point (csbp_attn_bwd_noalloc).

It exists for callers that cannot call cudaMalloc (plugin or custom-op
interfaces that receive only input and output buffers, runtimes whose memory
pool forbids outside allocations, paths that cannot take cudaMalloc's
implicit device synchronisation): its scratch is a fixed 64 MiB array in the
library's device memory instead of a caller workspace.  These tests call it
through the C-ABI and check it against the regular entry point
(csbp_attn_bwd with a caller workspace) on two calls in a row, so stale
contents left in the shared scratch by the first call would show up in the
second.  This file is named to be collected last.
"""
import ctypes

import pytest
import torch

from block_diffusion_lm_gb300 import csbp
from block_diffusion_lm_gb300.inputs import Workload, make_inputs

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
    for _ in range(2):
        g = attn.alloc_grads()
        for v in g.values():
            v.fill_(float("nan"))
        csbp.attn_bwd_noalloc(attn.problem, t, attn.work_dev, attn.info, out[0], out[1], out[2],
                              t["do_clean"], t["do_corr"], g)
        torch.cuda.synchronize()
        for k, r in ref.items():
            a, b = g[k].double(), r.double()
            assert torch.isfinite(a).all(), k
            assert ((a - b).norm() / b.norm()).item() <= TOL_REL, k


def test_noalloc_rejects_problems_beyond_its_scratch(_lib):
    """A problem needing more than the 64 MiB scratch is refused before any
    CUDA call (so this runs without a GPU too)."""
    prob = csbp.make_problem(1, 65536, 64, 32, 8, 128)
    assert csbp.workspace_bytes(prob, 1) > 64 << 20
    info = csbp.ScheduleInfo()
    st = _lib.csbp_attn_bwd_noalloc(ctypes.byref(prob), None, None, ctypes.byref(info),
                                    *([None] * 11), None)
    assert st == -3  # CSBP_ERR_WORKSPACE
