"""Failure detection on the GPU without a GPU fault: a bounded device wait on
a barrier that nothing ever arrives on gives up after its budget, the host
reads CSBP_ERR_TIMEOUT through the status word, and the same context then
runs the attention path correctly."""
import time

import numpy as np
import pytest
import torch

from block_diffusion_lm_gb300 import csbp
from block_diffusion_lm_gb300.inputs import Workload, make_inputs, to_f64
from oracle import csbp_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from block_diffusion_lm_gb300 import build
    build.build()


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    csbp.wait_selftest(5_000_000, ws)  # 5 ms budget
    with pytest.raises(csbp.CsbpError) as e:
        csbp.check_status(ws)
    assert e.value.status == -5  # CSBP_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    csbp.check_status(ws)  # the status word was cleared

    w = Workload("after_timeout", 1, 256, 32, 2, 1, 64, seed=50)
    t = make_inputs(w, "cuda")
    attn = csbp.BlockDiffusionAttention(1, w.L, w.M, w.Hq, w.Hkv, w.d)
    oc, ox, lse = attn.forward(t)
    attn.check()
    torch.cuda.synchronize()
    f = {k: to_f64(v[0]) for k, v in t.items()}
    Oc, Ox, _ = O.bd_attention_fwd(f["q_clean"], f["k_clean"], f["v_clean"], f["q_corr"],
                                   f["k_corr"], f["v_corr"], w.M, w.scale)
    assert np.abs(to_f64(ox[0]) - Ox).max() <= 1e-2
    assert np.abs(to_f64(oc[0]) - Oc).max() <= 1e-2
