"""Every problem the GPU tests and the benchmark run passes the library's
host-side argument checks, on the CPU.  Each is built through the binding
(schedule, info and fingerprint as a GPU run builds them); both entry points
are then called with placeholder 16-byte-aligned pointers and a workspace
one byte short, so they stop at CSBP_ERR_WORKSPACE after every other check,
before any CUDA call."""
import ctypes

import pytest

from block_diffusion_lm_gb300 import csbp
from block_diffusion_lm_gb300.inputs import WORKLOADS, Workload

import test_gpu_debug_checks as dbg
import test_gpu_parity as par

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
