"""The allocation-free forward, through the C ABI, on the GPU.

Some callers cannot allocate device memory once they are running (their
device memory is all owned by another allocator, or their latency-critical
path must not risk an allocation failing or synchronising the device);
`wna16_moe_forward_noalloc` serves them with its scratch in a static device
array inside the library.  This test checks that two calls in a row -- the
second one finding the first one's data still in that array -- each give
the same bits as the regular workspace entry point (both run the same
deterministic plan, so the outputs must be identical, well inside the parity
tolerance), and that a size too large for the array is refused on the host.

The file name sorts last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _noalloc(lib, d, w, out):
    P = ctypes.c_void_p
    return lib.wna16_moe_forward_noalloc(
        P(d["x"].data_ptr()), P(d["topk_ids"].data_ptr()), P(d["topk_weights"].data_ptr()),
        P(d["w13_packed"].data_ptr()), P(d["w13_scales"].data_ptr()), P(d["w2_packed"].data_ptr()),
        P(d["w2_scales"].data_ptr()), w.T, w.K, w.N, w.E, w.topk, w.g13, w.g2, w.bits, ctypes.c_float(w.swiglu_limit),
        P(out.data_ptr()), P(torch.cuda.current_stream().cuda_stream))


def test_noalloc_forward_matches_workspace_forward_twice():
    import wna16_grouped_gemm_gb300 as moe
    from wna16_grouped_gemm_gb300 import build
    build.build()
    lib = moe.load_library()
    lib.wna16_moe_forward_noalloc.restype = ctypes.c_int

    # two different batches: the decode workload (2-bit) and a W4 batch with ragged experts
    cases = [(synth.get("decode_w2"), 0),
             (synth.Workload("w4_batch", T=37, K=512, N=256, E=4, topk=2, bits=4, g13=128, g2=128,
                             scale_lo=0.001, scale_hi=0.005), 5)]
    for w, seed in cases:
        d = gu.to_dev(synth.make_all(w, seed))
        ref = moe.forward(d["x"], d["topk_ids"], d["topk_weights"], d["w13_packed"], d["w13_scales"],
                          d["w2_packed"], d["w2_scales"], bits=w.bits, group_size=w.g13, group_size_w2=w.g2,
                          swiglu_limit=w.swiglu_limit)
        out = torch.full((w.T, w.K), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = _noalloc(lib, d, w, out)
        assert rc == moe.OK, lib.wna16_moe_last_error().decode()
        torch.cuda.synchronize()
        got, want = gu.host_bits(out), gu.host_bits(ref)
        gu.assert_close(got, want, f"noalloc {w.name}")
        assert np.array_equal(got, want), f"noalloc {w.name}: not bit-identical to the workspace forward"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import wna16_grouped_gemm_gb300 as moe
    lib = moe.load_library()
    w = synth.get("prefill_w4_g64")          # needs about 1.3 GB of scratch
    d = gu.to_dev(synth.make_all(synth.get("tiny_w2")))
    fake = dict(d)
    out = torch.empty(1, dtype=torch.bfloat16, device="cuda")
    rc = _noalloc(lib, fake, w, out)
    assert rc == moe.ERR_WORKSPACE_TOO_SMALL
    assert "scratch" in lib.wna16_moe_last_error().decode()
