"""The seeded input recipe: routing statistics of the benchmark workloads
(active experts, rows per expert) recomputed from the generator and pinned, so
that a change to the generator cannot pass unnoticed (the measured numbers and
the committed profiles were taken on these inputs)."""
from __future__ import annotations

import numpy as np
import pytest

import synth


@pytest.mark.parametrize("name,active,max_rows,min_rows,top5,light", [
    ("decode_w2", 29, 2, 1, [2, 2, 2, 1, 1], (29, 32)),
    ("decode_w4_T1", 8, 1, 1, [1, 1, 1, 1, 1], (8, 8)),
    ("prefill_w2_zipf", 142, 1990, 1, [1990, 1788, 1538, 1285, 1176], (80, 210)),
    ("prefill_w4_g64", 256, 296, 210, [296, 295, 295, 294, 291], (0, 0)),
])
def test_routing_statistics(name, active, max_rows, min_rows, top5, light):
    w = synth.get(name)
    ids, weights = synth.make_routing(w, 0)
    assert ids.shape == (w.T, w.topk) and ids.dtype == np.int32
    assert weights.shape == (w.T, w.topk) and weights.dtype == np.float32
    counts = np.bincount(ids.ravel(), minlength=w.E)
    assert int((counts > 0).sum()) == active
    assert int(counts.max()) == max_rows
    assert int(counts[counts > 0].min()) == min_rows
    assert sorted(counts.tolist(), reverse=True)[:5] == top5
    # experts of at most 8 rows (the light-expert launches of 2-bit prefill
    # batches): how many, and their rows
    few = (counts > 0) & (counts <= 8)
    assert (int(few.sum()), int(counts[few].sum())) == light
    # top-k: distinct experts per token, weights renormalised, descending
    assert all(len(set(r)) == w.topk for r in ids.tolist())
    assert np.allclose(weights.sum(axis=1), 1.0, atol=1e-6)
    assert (np.diff(weights, axis=1) <= 0).all()
