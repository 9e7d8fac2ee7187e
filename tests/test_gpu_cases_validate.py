"""Every problem the GPU tests and the benchmark run (attention and the
LM-head cross-entropy) passes the library's host-side argument checks, on
the CPU.  Each is built through the binding
(schedule, info and fingerprint as a GPU run builds them); both entry points
are then called with placeholder 16-byte-aligned pointers and a workspace
one byte short, so they stop at CSBP_ERR_WORKSPACE after every other check,
before any CUDA call."""
import ctypes

import pytest

from block_diffusion_lm_gb300 import csbp
from block_diffusion_lm_gb300.inputs import CE_WORKLOADS, WORKLOADS, CeWorkload, Workload

import test_gpu_debug_checks as dbg
import test_gpu_parity as par
import test_gpu_vocab_ce as gce

CASES = ([(w, 0) for w in par.SMALL] + list(par.WINDOWED) + list(dbg.CASES)
         + [(w, 0) for w in WORKLOADS.values()]
         + [(Workload("packed", 2, 512, 16, 4, 2, 128, has_clean_queries=c, seed=50), 0)
            for c in (True, False)])


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_lm_gb300 import build
    build.build()


@pytest.mark.parametrize("w,chunk", CASES, ids=[f"{w.name}-c{c}" for w, c in CASES])
def test_problem_passes_every_host_check(w, chunk):
    # the calls BlockDiffusionAttention makes, without its device workspaces
    prob = csbp.make_problem(w.batch, w.L, w.M, w.Hq, w.Hkv, w.d, w.P, w.has_clean_queries,
                             window=w.window, clean_causal=w.clean_causal, bwd_chunk=chunk)
    _, _, _, info = csbp.block_schedule(prob)
    L = csbp.lib()
    g = ctypes.c_void_p(0x10000)
    packed = (w.Hq + 2 * w.Hkv) * w.d
    need_f = csbp.workspace_bytes(prob, 0)
    need_b = csbp.workspace_bytes(prob, 1)
    assert need_f > 0 and need_b > 0
    for tok in (0, packed):
        inp = csbp.Inputs(g, g, g, g, g, g, (ctypes.c_int64 * 6)(*[tok] * 6),
                          (ctypes.c_int64 * 6)(*[w.L * tok] * 6))
        assert L.csbp_attn_fwd(ctypes.byref(prob), ctypes.byref(inp), g, ctypes.byref(info),
                               g, g, g, g, need_f - 1, None) == -3
        assert L.csbp_attn_bwd(ctypes.byref(prob), ctypes.byref(inp), g, ctypes.byref(info),
                               *([g] * 12), need_b - 1, None) == -3


CE_CASES = (list(gce.SMALL) + list(CE_WORKLOADS.values())
            + [CeWorkload("ce_out_of_range", 300, 128, 1024, seed=2030),
               CeWorkload("ce_rechunk", 1000, 256, 2048, chunk=128, seed=2020)])


@pytest.mark.parametrize("w", CE_CASES, ids=[w.name for w in CE_CASES])
def test_cross_entropy_problem_passes_every_host_check(w):
    p = csbp.make_ce_problem(w.N, w.Dm, w.V, w.chunk, w.head_grad, 0.5)
    n = csbp.ce_workspace_bytes(p)
    assert n > 0
    g = ctypes.c_void_p(0x10000)
    dw = g if w.head_grad else None
    assert csbp.lib().csbp_vocab_ce(ctypes.byref(p), g, g, g, g, g, g, dw, g, n - 1,
                                    None) == -3
