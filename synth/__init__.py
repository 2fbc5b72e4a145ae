"""Seeded synthetic inputs for the WNA16 routed-MoE forward.

This module is shared by the tests, the oracle runs and the CUDA path; it
holds none of the method's arithmetic (no unpacking, dequantisation, GEMM,
SwiGLU or combine).  It only draws numbers:

* one ``numpy.random.Generator(PCG64)`` per input, spawned from
  ``SeedSequence(seed)`` in a fixed order: router logits, x, w13 words,
  w13 scales, w2 words, w2 scales;
* router logits N(0, 1) in fp32 (plus an optional popularity bias), turned
  into top-k ids and renormalised weights in fp64 (ties to the lower
  expert index), stored as int32 / fp32 -- these are *inputs* of the forward;
* x ~ N(0, 1) in fp32, rounded to BF16 (torch's round-to-nearest-even);
* packed weight words uniform over all 2^32 values: every b-bit field of a
  uniform word is uniform over [0, 2^b), i.e. the codes are uniform over
  {-2..1} (2-bit) or {-8..7} (4-bit) whatever the in-word field order;
* FP16 scales uniform on [lo, hi] in fp64, rounded to FP16.

The workloads are those of the pages' serving setting (DeepSeek-V4-Flash
routed experts: hidden 4096, intermediate 2048, 256 experts, top-8; decode
with 4 concurrent sequences, prefill in chunks of 2048 tokens), synthetic
because no checkpoint or dataset is used.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    K: int           # hidden size (input dim of w13, output dim of w2)
    N: int           # intermediate size
    E: int
    topk: int
    bits: int
    g13: int
    g2: int
    scale_lo: float
    scale_hi: float
    zipf_s: float = 0.0   # >0: logit bias -s*ln(e+1) (expert e has popularity rank e+1)
    swiglu_limit: float = 7.0

    @property
    def R(self) -> int:
        return self.T * self.topk

    def with_tokens(self, T: int) -> "Workload":
        return dataclasses.replace(self, T=T, name=f"{self.name}_T{T}")


WORKLOADS = {
    # tiny W2A16 indexed MoE, parity only
    "tiny_w2": Workload("tiny_w2", T=16, K=256, N=128, E=8, topk=2, bits=2, g13=128, g2=128,
                        scale_lo=0.005, scale_hi=0.02),
    # decode: 4 concurrent sequences, one step, W2A16 g128
    "decode_w2": Workload("decode_w2", T=4, K=4096, N=2048, E=256, topk=8, bits=2, g13=128,
                          g2=128, scale_lo=0.005, scale_hi=0.02),
    # decode W4A16 g128 (timed at T=1 and T=4)
    "decode_w4": Workload("decode_w4", T=4, K=4096, N=2048, E=256, topk=8, bits=4, g13=128,
                          g2=128, scale_lo=0.001, scale_hi=0.005),
    # prefill chunk of 2048 tokens, W2A16 g128, Zipf(1.1) expert popularity
    "prefill_w2_zipf": Workload("prefill_w2_zipf", T=2048, K=4096, N=2048, E=256, topk=8, bits=2,
                                g13=128, g2=128, scale_lo=0.005, scale_hi=0.02, zipf_s=1.1),
    # large prefill, 8192 tokens, W4A16 with w13 g128 and w2 g64, uniform routing
    "prefill_w4_g64": Workload("prefill_w4_g64", T=8192, K=4096, N=2048, E=256, topk=8, bits=4,
                               g13=128, g2=64, scale_lo=0.001, scale_hi=0.005),
}
# one GPU's share of the tensor-parallel deployment the pages measure (TP 4
# over the intermediate dimension: w13 rows and w2 columns split four ways)
WORKLOADS["decode_w2_tp4"] = dataclasses.replace(WORKLOADS["decode_w2"], name="decode_w2_tp4", N=512)
WORKLOADS["prefill_w2_zipf_tp4"] = dataclasses.replace(WORKLOADS["prefill_w2_zipf"], name="prefill_w2_zipf_tp4", N=512)


def get(name: str) -> Workload:
    """A named workload; "<name>_T<tokens>" changes the token count and
    "<name>_E<experts>_T<tokens>" also the expert count (a smaller problem of
    the same shape, e.g. for a profiler capture)."""
    if name in WORKLOADS:
        return WORKLOADS[name]
    base, _, t = name.rpartition("_T")
    if base in WORKLOADS and t.isdigit():
        return WORKLOADS[base].with_tokens(int(t))
    b2, _, e = base.rpartition("_E")
    if b2 in WORKLOADS and e.isdigit() and t.isdigit():
        w = dataclasses.replace(WORKLOADS[b2], E=int(e), name=name)
        return dataclasses.replace(w, T=int(t))
    raise KeyError(name)


def _streams(seed: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(6)]


def route_topk(logits: np.ndarray, topk: int):
    """Softmax over experts, top-k (ties -> lower index), renormalised; fp64."""
    z = logits.astype(np.float64)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :topk]
    w = np.take_along_axis(p, order, axis=1)
    w /= w.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 array -> BF16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def make_logits(w: Workload, seed: int = 0):
    """Router logits fp32 [T, E] ~ N(0, 1) and the popularity bias fp32 [E]
    (-s*ln(e+1) for a Zipf(s) workload, else None)."""
    rng = _streams(seed)[0]
    logits = rng.standard_normal((w.T, w.E), dtype=np.float32)
    bias = None
    if w.zipf_s:
        bias = (-w.zipf_s * np.log(np.arange(1, w.E + 1, dtype=np.float64))).astype(np.float32)
    return logits, bias


def make_routing(w: Workload, seed: int = 0):
    logits, bias = make_logits(w, seed)
    if bias is not None:
        logits = logits + bias
    return route_topk(logits, w.topk)


def make_x(w: Workload, seed: int = 0) -> np.ndarray:
    rng = _streams(seed)[1]
    return to_bf16_bits(rng.standard_normal((w.T, w.K), dtype=np.float32))


def _words(rng, shape) -> np.ndarray:
    return rng.integers(0, 1 << 32, size=shape, dtype=np.uint32).view(np.int32)


def _scales(rng, shape, lo, hi) -> np.ndarray:
    return rng.uniform(lo, hi, size=shape).astype(np.float16)


def make_weights(w: Workload, seed: int = 0):
    """(w13_packed int32 [E,2N,K/p], w13_scales fp16 [E,2N,K/g13],
        w2_packed int32 [E,K,N/p], w2_scales fp16 [E,K,N/g2])."""
    s = _streams(seed)
    p = 32 // w.bits
    w13p = _words(s[2], (w.E, 2 * w.N, w.K // p))
    w13s = _scales(s[3], (w.E, 2 * w.N, w.K // w.g13), w.scale_lo, w.scale_hi)
    w2p = _words(s[4], (w.E, w.K, w.N // p))
    w2s = _scales(s[5], (w.E, w.K, w.N // w.g2), w.scale_lo, w.scale_hi)
    return w13p, w13s, w2p, w2s


def make_all(w: Workload, seed: int = 0) -> dict:
    ids, wts = make_routing(w, seed)
    w13p, w13s, w2p, w2s = make_weights(w, seed)
    return dict(x=make_x(w, seed), ids=ids, weights=wts, w13_packed=w13p, w13_scales=w13s,
                w2_packed=w2p, w2_scales=w2s)


def random_codes(rng: np.random.Generator, shape, bits: int) -> np.ndarray:
    """Uniform signed codes in [-2^(b-1), 2^(b-1)) as int8 (for pack tests)."""
    half = 1 << (bits - 1)
    return rng.integers(-half, half, size=shape, dtype=np.int8)


def make_quant_inputs(rows: int, K: int, seed: int = 0):
    """Source weights for the quantiser, fp32 [rows, K]: N(0, 0.02^2) with 1 %
    of the entries eight times larger (heavy-tailed, like decoded expert
    weights), and an importance vector fp32 [K] (per input channel, the mean
    squared activation of a calibration set: log-normal, exp(N(0, 1)))."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))
    w = rng.standard_normal((rows, K), dtype=np.float32) * np.float32(0.02)
    out = rng.random((rows, K)) < 0.01
    w[out] *= np.float32(8.0)
    imp = np.exp(rng.standard_normal(K)).astype(np.float32)
    return w, imp
