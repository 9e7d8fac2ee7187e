"""CPU checks of the LM-head cross-entropy's C-ABI: workspace sizing and the
argument checks that run before anything is enqueued (no CUDA call is made
on these paths, so they need no GPU)."""
import ctypes

import pytest

from block_diffusion_lm_gb300 import csbp


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_lm_gb300 import build
    build.build()


def test_workspace_bytes_cover_logits_g_and_partials():
    p = csbp.make_ce_problem(16384, 5120, 131072, 8192, True, 1.0 / 16384)
    C, V = 8192, 131072
    want = 256 + C * V * 4 + C * V * 2 + C * (V // 256) * 8 + C * 4
    assert want <= csbp.ce_workspace_bytes(p) <= want + 4 * 256
    # the chunk never exceeds the rows (rounded up to a 128-row tile)
    small = csbp.make_ce_problem(300, 192, 1600, 0, True, 0.1)
    C = 384
    assert csbp.ce_workspace_bytes(small) >= 256 + C * 1600 * 6


@pytest.mark.parametrize("field,value", [
    ("rows", 0), ("rows", 1 << 62), ("rows", (1 << 39) // 256 + 1), ("d_model", 96), ("d_model", 0), ("vocab", 100), ("vocab", 1 << 25),
    ("chunk_rows", 100), ("chunk_rows", -128), ("head_grad", 2), ("grad_scale", float("inf")),
])
def test_invalid_problems_have_no_workspace_and_are_refused(field, value):
    p = csbp.make_ce_problem(1000, 256, 4096)
    setattr(p, field, value)
    assert csbp.ce_workspace_bytes(p) == 0
    good = ctypes.c_void_p(0x10000)
    st = csbp.lib().csbp_vocab_ce(ctypes.byref(p), good, good, good, good, good, good, good,
                                  good, 1 << 40, None)
    assert st == -1


def test_pointer_and_workspace_checks():
    L = csbp.lib()
    p = csbp.make_ce_problem(1000, 256, 4096, 0, True, 0.01)
    good = ctypes.c_void_p(0x10000)
    bad = ctypes.c_void_p(0x10008)  # 8-byte aligned only
    n = csbp.ce_workspace_bytes(p)
    args = [good] * 8
    for i in range(8):
        a = list(args)
        a[i] = None
        assert L.csbp_vocab_ce(ctypes.byref(p), *a, n, None) == -1, i
        a[i] = bad
        assert L.csbp_vocab_ce(ctypes.byref(p), *a, n, None) == -1, i
    # frozen head: dw must be NULL
    p.head_grad = 0
    assert L.csbp_vocab_ce(ctypes.byref(p), *args, n, None) == -1
    p.head_grad = 1
    assert L.csbp_vocab_ce(ctypes.byref(p), *args, n - 1, None) == -3
