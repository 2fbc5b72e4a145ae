"""The sharded shapes of the path on one GPU, through the C ABI, against the
oracle.

* Tensor parallel (the pages' deployment: TP 4 over the intermediate
  dimension): one GPU's share is the forward with N/4 = 512; its output is
  that rank's partial (the ranks' outputs are summed across GPUs), here
  compared with the oracle's forward at the same shapes.
* Expert parallel: each rank holds a contiguous range of experts and writes
  an fp32 partial output for the slots routed to them; the ranks' partials,
  summed in rank order in fp32 and rounded to BF16, are the oracle's
  expert-parallel profile.  The ranks run one after the other on the one GPU.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import wna16_grouped_gemm_gb300 as m
    from wna16_grouped_gemm_gb300 import build
    build.build()
    m.load_library()
    return m


@pytest.mark.parametrize("name", ["decode_w2_tp4", "prefill_w2_zipf_tp4"])
def test_tp4_share_matches_oracle(moe, oracle, name):
    w = synth.get(name)
    inp = synth.make_all(w, 0)
    d = gu.to_dev(inp)
    ws = moe.alloc_workspace(w.T, w.K, w.N, w.E, w.topk, w.bits)
    out = moe.forward(d["x"], d["topk_ids"], d["topk_weights"], d["w13_packed"], d["w13_scales"], d["w2_packed"],
                      d["w2_scales"], bits=w.bits, group_size=w.g13, group_size_w2=w.g2, swiglu_limit=w.swiglu_limit,
                      workspace=ws)
    assert moe.read_status(ws) == moe.OK
    ref = oracle.forward(inp["x"], inp["ids"], inp["weights"], inp["w13_packed"], inp["w13_scales"],
                         inp["w2_packed"], inp["w2_scales"], bits=w.bits, group_size=w.g13, group_size_w2=w.g2,
                         swiglu_limit=w.swiglu_limit)
    gu.assert_close(gu.host_bits(out), ref, name)


def _ep_case(name):
    if name == "moderate_w4":
        return synth.Workload("moderate_w4", T=512, K=1024, N=512, E=8, topk=2, bits=4, g13=128, g2=64,
                              scale_lo=0.001, scale_hi=0.005)
    return synth.get(name)


@pytest.mark.parametrize("name,ranks", [("decode_w2", 2), ("decode_w4", 4), ("moderate_w4", 2), ("tiny_w2", 3)])
def test_expert_parallel_partials(moe, oracle, name, ranks):
    w = _ep_case(name)
    inp = synth.make_all(w, 0)
    d = gu.to_dev(inp)
    bounds = np.linspace(0, w.E, ranks + 1).astype(int)
    ref_out, _, y_ref = oracle.forward(inp["x"], inp["ids"], inp["weights"], inp["w13_packed"], inp["w13_scales"],
                                       inp["w2_packed"], inp["w2_scales"], bits=w.bits, group_size=w.g13,
                                       group_size_w2=w.g2, swiglu_limit=w.swiglu_limit, return_intermediates=True)
    gpu_parts, ref_parts = [], []
    for r in range(ranks):
        b, e = int(bounds[r]), int(bounds[r + 1])
        loc = {k: d[k][b:e] for k in ("w13_packed", "w13_scales", "w2_packed", "w2_scales")}
        ws = moe.alloc_workspace(w.T, w.K, w.N, e - b, w.topk, w.bits)
        part = moe.forward_partial(d["x"], d["topk_ids"], d["topk_weights"], loc["w13_packed"], loc["w13_scales"],
                                   loc["w2_packed"], loc["w2_scales"], expert_begin=b, E_total=w.E, bits=w.bits,
                                   group_size=w.g13, group_size_w2=w.g2, swiglu_limit=w.swiglu_limit, workspace=ws)
        assert moe.read_status(ws) == moe.OK
        gpu_parts.append(part.cpu().numpy())
        ref_parts.append(oracle.combine_partial(inp["ids"], inp["weights"], y_ref, (b, e)))
        # a slot of another rank contributes nothing: rows whose experts are all remote are exactly 0
        remote = ~((inp["ids"] >= b) & (inp["ids"] < e)).any(axis=1)
        assert np.all(gpu_parts[-1][remote] == 0.0)
        g, rf = gpu_parts[-1].astype(np.float64), ref_parts[-1].astype(np.float64)
        rel = np.sqrt(((g - rf) ** 2).sum() / max((rf ** 2).sum(), 1e-300))
        print(name, "rank", r, "partial rel-L2", rel)
        assert rel <= gu.REL_L2
    # ranks summed in rank order in fp32, then BF16
    s = gpu_parts[0].astype(np.float32)
    for p in gpu_parts[1:]:
        s = s + p.astype(np.float32)
    got = torch.from_numpy(s).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    gu.assert_close(got, oracle.sum_partials(ref_parts), f"{name} EP x{ranks} (profile)")
    gu.assert_close(got, ref_out, f"{name} EP x{ranks} (single-device oracle)")
