"""GPU parity of the streamed LM-head cross-entropy through the C-ABI against
the float64 oracle.

Tolerances (bf16 inputs, fp32 logits and accumulation, bf16 g): loss and
LSE abs <= 1e-3; dH and dW relative Frobenius <= 1e-2 (exactly-zero
references: max-abs <= 1e-6).  Small cases compare every element; the
full-size workloads compare seeded sample rows the oracle evaluates one by
one, plus the exact invariant sum_v dW_v = 0.
"""
import numpy as np
import pytest
import torch

from block_diffusion_lm_gb300 import csbp
from block_diffusion_lm_gb300.inputs import CE_WORKLOADS, CeWorkload, make_ce_inputs
from oracle import vocab_ce_oracle as C

pytestmark = pytest.mark.gpu

TOL_LOSS = 1e-3
TOL_REL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from block_diffusion_lm_gb300 import build
    build.build()


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def close(got, want, name):
    if np.linalg.norm(want) == 0:
        assert np.abs(got).max() <= 1e-6, name
    else:
        assert rel_fro(got, want) <= TOL_REL, (name, rel_fro(got, want))


def run_gpu(w: CeWorkload, chunk=None, head_grad=None):
    x = make_ce_inputs(w, "cuda")
    ce = csbp.VocabCrossEntropy(w.N, w.Dm, w.V, w.chunk if chunk is None else chunk,
                                w.head_grad if head_grad is None else head_grad, x["grad_scale"])
    out = ce(x["h"], x["w"], x["target"])
    ce.check()
    torch.cuda.synchronize()
    return x, out


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


SMALL = [
    CE_WORKLOADS["ce_tiny"],                                                  # 3 chunks, ragged
    CeWorkload("ce_frozen", 1000, 256, 4096, head_grad=False, ignore_frac=0.1, seed=2010),
    CeWorkload("ce_chunks", 1024, 512, 8192, chunk=384, seed=2011),
    CeWorkload("ce_one_row", 1, 64, 64, seed=2012),
    CeWorkload("ce_ragged", 257, 320, 4160, chunk=256, ignore_frac=0.5, seed=2013),
    CeWorkload("ce_all_ignored", 130, 128, 512, ignore_frac=1.0, seed=2014),
    CeWorkload("ce_wide_head", 640, 1024, 2048, seed=2015),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_cases_match_oracle_elementwise(w):
    x, (loss, lse, dh, dw) = run_gpu(w)
    t = x["target"].cpu().numpy()
    rl, rz, rdh, rdw = C.vocab_ce(f64(x["h"]), f64(x["w"]), t, x["grad_scale"], w.head_grad)
    assert np.abs(f64(loss) - rl).max() <= TOL_LOSS
    assert np.abs(f64(lse) - rz).max() <= TOL_LOSS
    close(f64(dh), rdh, "dh")
    if w.head_grad:
        close(f64(dw), rdw, "dw")
    else:
        assert dw is None


def test_targets_outside_the_vocabulary_are_ignored():
    """Targets past the vocabulary (V, V + 100, INT32_MAX) and negative ones
    other than -1 mark ignored rows, as the header states."""
    w = CeWorkload("ce_out_of_range", 300, 128, 1024, seed=2030)
    x = make_ce_inputs(w, "cuda")
    tgt = x["target"]
    tgt[::7] = w.V
    tgt[3::11] = w.V + 100
    tgt[5] = 2 ** 31 - 1
    tgt[6] = -(2 ** 31)
    ce = csbp.VocabCrossEntropy(w.N, w.Dm, w.V, w.chunk, True, x["grad_scale"])
    loss, lse, dh, dw = ce(x["h"], x["w"], tgt)
    ce.check()
    torch.cuda.synchronize()
    t = tgt.cpu().numpy()
    rl, rz, rdh, rdw = C.vocab_ce(f64(x["h"]), f64(x["w"]), t, x["grad_scale"])
    ignored = (t < 0) | (t >= w.V)
    assert np.all(f64(loss)[ignored] == 0) and np.all(f64(dh)[ignored] == 0)
    assert np.abs(f64(loss) - rl).max() <= TOL_LOSS
    assert np.abs(f64(lse) - rz).max() <= TOL_LOSS
    close(f64(dh), rdh, "dh")
    close(f64(dw), rdw, "dw")


def test_chunking_changes_nothing_per_row():
    """Rows are independent: loss, LSE and dH are bit-identical whatever the
    chunk size; dW differs only by fp32 summation order across chunks."""
    w = CeWorkload("ce_rechunk", 1000, 256, 2048, seed=2020)
    _, a = run_gpu(w, chunk=128)
    _, b = run_gpu(w, chunk=1024)
    for i in range(3):
        assert torch.equal(a[i], b[i])
    assert rel_fro(f64(a[3]), f64(b[3])) <= 1e-5


def test_frozen_head_gives_the_same_dh():
    w = CeWorkload("ce_frozen_vs_trained", 512, 256, 2048, seed=2021)
    _, a = run_gpu(w, head_grad=True)
    _, b = run_gpu(w, head_grad=False)
    assert torch.equal(a[2], b[2]) and b[3] is None


def _sampled(w, n_rows, seed):
    x, (loss, lse, dh, dw) = run_gpu(w)
    rng = np.random.default_rng(seed)
    rows = rng.choice(w.N, size=n_rows, replace=False)
    W = x["w"].cpu().to(torch.float64).numpy()
    H = x["h"].cpu()
    t = x["target"].cpu().numpy()
    rl, rz, rdh = C.vocab_ce_rows(_Rows(H), W, t, x["grad_scale"], rows)
    assert np.abs(f64(loss[rows]) - rl).max() <= TOL_LOSS
    assert np.abs(f64(lse[rows]) - rz).max() <= TOL_LOSS
    assert rel_fro(f64(dh[rows]), rdh) <= TOL_REL
    if w.head_grad:
        s = dw.double().sum(dim=0)
        assert (s.norm() / dw.double().norm()).item() <= 1e-2


class _Rows:
    """bf16 host matrix that hands the oracle float64 rows on indexing."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, idx):
        return self.t[torch.as_tensor(idx)].to(torch.float64).numpy()


@pytest.mark.parametrize("name,rows,seed", [("lmhead14b", 12, 301), ("lmhead_frozen", 12, 302)])
def test_full_size_sampled_rows(name, rows, seed):
    _sampled(CE_WORKLOADS[name], rows, seed)
    torch.cuda.empty_cache()
