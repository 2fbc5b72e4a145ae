"""The bounds-checked build (libwna16_moe_debug.so, compiled with
-DWNA16_DEBUG) on the GPU: every plan runs with its index checks on, leaves the
status word at OK (no computed index fell outside its buffer) and gives the
same bits as the release build."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    import wna16_grouped_gemm_gb300 as moe
    from wna16_grouped_gemm_gb300 import binding, build
    build.build()
    build.build(debug=True)
    return moe, moe.load_library(), binding.load_debug_library()


def _small(T, K, N, E, topk, bits, g13, g2, zipf=0.0):
    return synth.Workload("dbg", T=T, K=K, N=N, E=E, topk=topk, bits=bits, g13=g13, g2=g2,
                          scale_lo=0.005 if bits == 2 else 0.001, scale_hi=0.02 if bits == 2 else 0.005,
                          zipf_s=zipf)


CASES = {
    "tiny_w2": synth.get("tiny_w2"),
    "decode_w2": synth.get("decode_w2"),                         # group-accumulate, offset codes, split K
    "decode_w4_T1": synth.get("decode_w4_T1"),
    "decode_w2_T64": synth.get("decode_w2_T64"),                 # group-accumulate without split
    "w4_prefill_tiles_g64": _small(700, 1024, 512, 4, 2, 4, 128, 64),
    "w2_g32_tiles64": _small(96, 1024, 512, 4, 2, 2, 32, 32),
    "w4_chunked_route": _small(1200, 512, 256, 16, 8, 4, 128, 128),   # 9600 slots: routed by chunks
    "w4_paired_k_splits": _small(300, 4096, 256, 3, 1, 4, 128, 128),  # w13 K splits on CTA pairs
    "w2_light_experts": _small(1024, 4096, 512, 64, 4, 2, 128, 128, zipf=1.1),          # light-expert launches
    "w2_light_experts_chunked": _small(2200, 4096, 512, 64, 4, 2, 128, 128, zipf=1.1),  # ... chunked routing
}


def _forward(lib, moe, w, d, ws, out):
    P = ctypes.c_void_p
    rc = lib.wna16_moe_forward(P(d["x"].data_ptr()), P(d["topk_ids"].data_ptr()), P(d["topk_weights"].data_ptr()),
                               P(d["w13_packed"].data_ptr()), P(d["w13_scales"].data_ptr()),
                               P(d["w2_packed"].data_ptr()), P(d["w2_scales"].data_ptr()), w.T, w.K, w.N, w.E, w.topk,
                               w.g13, w.g2, w.bits, ctypes.c_float(w.swiglu_limit), P(out.data_ptr()),
                               P(ws.data_ptr()), ws.numel(), P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.wna16_moe_last_error().decode()
    st = ctypes.c_int(99)
    assert lib.wna16_moe_read_status(P(ws.data_ptr()), ctypes.byref(st),
                                     P(torch.cuda.current_stream().cuda_stream)) == 0
    return st.value


@pytest.mark.parametrize("name", list(CASES))
def test_debug_build_matches_release(libs, name):
    moe, rel, dbg = libs
    w = CASES[name]
    d = gu.to_dev(synth.make_all(w, 0))
    outs, stats = [], []
    for lib in (rel, dbg):
        ws = moe.alloc_workspace(w.T, w.K, w.N, w.E, w.topk, w.bits)
        out = torch.full((w.T, w.K), float("nan"), dtype=torch.bfloat16, device="cuda")
        stats.append(_forward(lib, moe, w, d, ws, out))
        outs.append(gu.host_bits(out))
    assert stats == [moe.OK, moe.OK], stats
    assert np.array_equal(outs[0], outs[1])
