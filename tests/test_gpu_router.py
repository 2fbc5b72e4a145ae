"""The router kernel (softmax over the experts with an optional logit bias,
top-k with ties to the lower index, renormalisation) through the C ABI,
against the oracle's router.

The chosen experts must be bit-exact.  The weights are fp32 in the kernel
(exp of the fp32 difference to the largest chosen score, summed over the k
chosen in choice order) and fp64 rounded to fp32 in the oracle; with scores
within 16 of each other (N(0,1) logits plus at most a 6.1 Zipf bias) the
fp32 difference, expf's 2-ulp error, the k-term sum and the division keep
the relative error under 2e-6, the stated tolerance.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

W_REL_TOL = 2e-6


@pytest.fixture(scope="module")
def moe():
    import wna16_grouped_gemm_gb300 as m
    from wna16_grouped_gemm_gb300 import build
    build.build()
    m.load_library()
    return m


def _check(moe, oracle, logits, k, bias=None, what=""):
    lg = torch.from_numpy(logits).cuda()
    b = None if bias is None else torch.from_numpy(bias).cuda()
    ids, w = moe.route_topk(lg, k, b)
    torch.cuda.synchronize()
    rid, rw = oracle.route_topk(logits, k, bias)
    gid, gw = ids.cpu().numpy(), w.cpu().numpy()
    assert np.array_equal(gid, rid), what
    rel = np.abs(gw.astype(np.float64) - rw) / np.abs(rw)
    print(what, "max rel weight error", float(rel.max()), "exact", float((gw == rw).mean()))
    assert rel.max() <= W_REL_TOL, what
    return gid, gw


@pytest.mark.parametrize("name", ["tiny_w2", "decode_w2", "decode_w4_T1", "prefill_w2_zipf", "prefill_w4_g64"])
def test_router_workloads(moe, oracle, name):
    """The routing of every workload (softmax top-k of N(0,1) logits, with the
    Zipf(1.1) popularity bias for the 2048-token prefill) from its logits; the
    chosen experts are also exactly the ones the seeded generator gave the
    forward."""
    w = synth.get(name)
    logits, bias = synth.make_logits(w, 0)
    gid, gw = _check(moe, oracle, logits, w.topk, bias, name)
    ids, wts = synth.make_routing(w, 0)
    assert np.array_equal(gid, ids)
    assert np.max(np.abs(gw.astype(np.float64) - wts) / wts) <= W_REL_TOL


@pytest.mark.parametrize("T,E,k", [(100, 1024, 32), (37, 33, 5), (9, 5, 5), (64, 64, 1), (300, 256, 8)])
def test_router_shapes(moe, oracle, T, E, k):
    rng = np.random.default_rng(T + E + k)
    _check(moe, oracle, rng.standard_normal((T, E), dtype=np.float32), k, None, f"T={T} E={E} k={k}")


def test_router_ties_go_to_the_lower_index(moe, oracle):
    """Scores rounded to quarters: many equal scores inside every token's top-k."""
    rng = np.random.default_rng(5)
    logits = (np.round(rng.standard_normal((257, 256)) * 4) / 4).astype(np.float32)
    logits[0] = 0.0                                   # all equal: experts 0..k-1
    gid, gw = _check(moe, oracle, logits, 8, None, "ties")
    assert gid[0].tolist() == list(range(8)) and np.all(gw[0] == np.float32(0.125))


def test_router_bias_and_empty(moe, oracle):
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((50, 16), dtype=np.float32)
    bias = np.zeros(16, np.float32)
    bias[:12] = -1e4                                   # only experts 12..15 can win
    gid, _ = _check(moe, oracle, logits, 4, bias, "bias")
    assert np.all(np.sort(gid, axis=1) == np.arange(12, 16))
    ids, w = moe.route_topk(torch.empty(0, 16, dtype=torch.float32, device="cuda"), 4)
    assert ids.shape == (0, 4) and w.shape == (0, 4)
