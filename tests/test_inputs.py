"""The benchmark's useful-FLOP count: Workload.pairs_per_head and
keys_of_row (used by the CPU baseline) against the oracle's explicit mask,
for every mask option; and the seeded inputs are reproducible."""
import numpy as np
import pytest
import torch

from block_diffusion_lm_gb300.inputs import (CE_WORKLOADS, WORKLOADS, Workload, make_ce_inputs,
                                             make_inputs)
from oracle import csbp_oracle as O

CASES = [
    Workload("a", 1, 256, 16, 2, 1, 64),
    Workload("b", 1, 256, 16, 2, 1, 64, has_clean_queries=False),
    Workload("c", 1, 320, 32, 2, 1, 64, window=70),
    Workload("d", 1, 320, 32, 2, 1, 64, clean_causal=True),
    Workload("e", 1, 384, 8, 2, 1, 64, window=41, clean_causal=True),
    Workload("f", 1, 256, 16, 2, 1, 64, window=1, has_clean_queries=False),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_pair_counts_match_the_mask(w):
    A = O.bd_mask(w.L, w.M, w.window, w.clean_causal)
    L = w.L
    corr = A[L:].sum(axis=1)
    clean = A[:L].sum(axis=1)
    want = int(corr.sum()) + (int(clean.sum()) if w.has_clean_queries else 0)
    assert w.pairs_per_head() == want
    assert [w.keys_of_row(1, i) for i in range(L)] == corr.tolist()
    if w.has_clean_queries:
        assert [w.keys_of_row(0, i) for i in range(L)] == clean.tolist()


def test_useful_flops_of_the_dense_layer():
    w = WORKLOADS["dense14b"]
    assert w.pairs_per_head() == w.L * (w.L + w.M)
    assert w.useful_fwd_flops() == 4.0 * w.d * w.L * (w.L + w.M) * w.Hq
    assert w.useful_bwd_flops() == 2.5 * w.useful_fwd_flops()


def test_inputs_are_seeded_and_bf16():
    w = WORKLOADS["tiny"]
    a, b = make_inputs(w, "cpu"), make_inputs(w, "cpu")
    for k in a:
        assert a[k].dtype == torch.bfloat16 and a[k].shape[1] == w.L
        assert torch.equal(a[k], b[k])
    c = make_inputs(w, "cpu", seed=w.seed + 1)
    assert not torch.equal(a["q_corr"], c["q_corr"])
    x, y = make_ce_inputs(CE_WORKLOADS["ce_tiny"], "cpu"), make_ce_inputs(CE_WORKLOADS["ce_tiny"], "cpu")
    assert torch.equal(x["h"], y["h"]) and torch.equal(x["target"], y["target"])
    n_valid = int((x["target"] >= 0).sum())
    assert 0 < n_valid < CE_WORKLOADS["ce_tiny"].N and x["grad_scale"] == 1.0 / n_valid
