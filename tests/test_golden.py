"""The oracle against its stored record on the tiny decode layer
(tests/golden/tiny_layer_m4_seed0.json, written by tests/golden/make_golden.py
from the oracle alone).  Integer results must match exactly; floating-point
results within a few units in the last place of float64, or one bf16 step
for the bf16 outputs, so that another platform's exp/BLAS rounding does not
fail the record while any change to the arithmetic does."""

from __future__ import annotations

import json
import os

import numpy as np

from tests.golden import make_golden


def test_oracle_matches_its_golden_record_on_the_tiny_layer():
    with open(make_golden.PATH) as f:
        gold = json.load(f)
    now = make_golden.compute()
    for key in ("topk_ids", "sorted_routes", "expert_offsets", "columns", "redrawn_tokens"):
        assert now[key] == gold[key], key
    np.testing.assert_allclose(now["topk_weights"], gold["topk_weights"], rtol=1e-12, atol=0)
    for key in ("out", "residual_out"):
        a, b = np.asarray(now[key]), np.asarray(gold[key])
        # bf16 values: equal, or one bf16 step (2^-7 relative) apart
        assert np.all(np.abs(a - b) <= np.abs(b) * 2.0 ** -7), key
    for key in ("out_row_sum", "out_row_sumsq", "residual_out_row_sum"):
        np.testing.assert_allclose(now[key], gold[key], rtol=1e-3, atol=1e-3)


def test_golden_record_is_consistent():
    with open(make_golden.PATH) as f:
        gold = json.load(f)
    ids = np.asarray(gold["topk_ids"])
    M, k = ids.shape
    # routing weights: normalised over the selected experts, then x routed_scaling (2.5)
    np.testing.assert_allclose(np.asarray(gold["topk_weights"]).sum(axis=1), 2.5, rtol=1e-12)
    # the route order is a permutation of the expanded indices, grouped by expert
    sr = gold["sorted_routes"]
    assert sorted(sr) == list(range(M * k))
    off = gold["expert_offsets"]
    for e in range(len(off) - 1):
        grp = sr[off[e]:off[e + 1]]
        assert all(ids.reshape(-1)[r] == e for r in grp)
        assert grp == sorted(grp)  # stable: expanded index ascending within an expert
    assert os.path.getsize(make_golden.PATH) < 16384
