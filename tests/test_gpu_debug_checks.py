"""The debug build (kernels compiled with work-list record checks): valid
problems run to oracle tolerance with a clean status, and a planted bad
record (a segment running past the last tile) is refused by the CTA that
would use it, reported as CSBP_ERR_DEVICE, before that CTA touches memory.
A bad segment is also safe without the check: its tiles lie outside the
tensors, where TMA loads read zeros and stores are clipped."""
import numpy as np
import pytest
import torch

from block_diffusion_lm_gb300 import csbp
from block_diffusion_lm_gb300.inputs import Workload, make_inputs, to_f64
from oracle import csbp_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _debug_library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from block_diffusion_lm_gb300 import build
    build.build(debug=True)
    csbp.use_library(csbp.DEBUG_LIB_PATH)
    yield
    csbp.use_library()


CASES = [
    (Workload("dbg_ragged", 1, 400, 16, 4, 2, 128, seed=60), 0),
    (Workload("dbg_sharded", 1, 1024, 16, 4, 2, 128, P=2, seed=61), 0),
    (Workload("dbg_window", 1, 640, 16, 4, 2, 64, window=150, clean_causal=True, seed=62), 2),
]


@pytest.mark.parametrize("w,chunk", CASES, ids=[w.name for w, _ in CASES])
def test_debug_build_runs_valid_problems(w, chunk):
    t = make_inputs(w, "cuda")
    attn = csbp.BlockDiffusionAttention(1, w.L, w.M, w.Hq, w.Hkv, w.d, P=w.P,
                                        window=w.window, clean_causal=w.clean_causal,
                                        bwd_chunk=chunk)
    out = attn.forward(t)
    g = attn.backward(t, out)
    attn.check()
    torch.cuda.synchronize()
    f = {k: to_f64(v[0]) for k, v in t.items()}
    Oc, Ox, _ = O.bd_attention_fwd(f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"],
                                   f["k_corr"], f["v_corr"], w.M, w.scale, w.window,
                                   w.clean_causal)
    assert np.abs(to_f64(out[1][0]) - Ox).max() <= 1e-2
    assert np.abs(to_f64(out[0][0]) - Oc).max() <= 1e-2
    G = O.bd_attention_bwd(f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"], f["k_corr"],
                           f["v_corr"], f["do_clean"], f["do_corr"], w.M, w.scale, w.window,
                           w.clean_causal)
    got = to_f64(g["dk_clean"][0])
    assert np.linalg.norm(got - G["dk_clean"]) <= 1e-2 * np.linalg.norm(G["dk_clean"])


@pytest.mark.parametrize("which", ["fwd", "bwd"])
def test_debug_build_refuses_a_bad_work_record(which):
    w = Workload("dbg_bad", 1, 512, 16, 2, 1, 128, seed=63)
    t = make_inputs(w, "cuda")
    attn = csbp.BlockDiffusionAttention(1, w.L, w.M, w.Hq, w.Hkv, w.d)
    words = attn.work_host.copy()
    off_segs = int(words[12] if which == "fwd" else words[14])
    nT = -(-w.L // 128)
    words[off_segs + 2] = nT + 3  # first segment of the list now runs past the last tile
    attn.work_dev = torch.from_numpy(words).to("cuda")
    out = attn.forward(t)
    if which == "bwd":
        attn.check()  # the forward read an intact list
        attn.backward(t, out)
    with pytest.raises(csbp.CsbpError) as e:
        attn.check()
    assert e.value.status == -7  # CSBP_ERR_DEVICE
    attn.check()  # cleared; the context is still usable
