"""Pins of the CPU oracle to things other than itself (CPU only).

Each pin checks the oracle against a fact fixed by the pages' format
definition or by mathematics: hand-decoded words, exact rational rounding,
closed-form SwiGLU cases, a library routine (numpy stable sort, torch
matmul/silu) on a special case, invariants (zero codes, scale doubling,
relabelling, token permutation) and a pure-Python brute force on tiny inputs.
``test_every_planted_mistake_is_caught`` plants each plausible bug in the
oracle and checks that at least one pin fails.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

import synth
from tests import independent as ind

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def _tiny_case(bits, T=3, K=64, N=32, E=3, topk=2, g13=16, g2=16, seed=11, scale=(0.05, 0.3)):
    rng = np.random.default_rng(seed)
    p = 32 // bits
    w13p = rng.integers(0, 1 << 32, size=(E, 2 * N, K // p), dtype=np.uint32).view(np.int32)
    w2p = rng.integers(0, 1 << 32, size=(E, K, N // p), dtype=np.uint32).view(np.int32)
    w13s = rng.uniform(*scale, size=(E, 2 * N, K // g13)).astype(np.float16)
    w2s = rng.uniform(*scale, size=(E, K, N // g2)).astype(np.float16)
    x = synth.to_bf16_bits(rng.standard_normal((T, K), dtype=np.float32))
    logits = rng.standard_normal((T, E), dtype=np.float32)
    ids, wts = synth.route_topk(logits, topk)
    return dict(x=x, ids=ids, weights=wts, w13_packed=w13p, w13_scales=w13s, w2_packed=w2p,
                w2_scales=w2s, K=K, N=N, E=E, topk=topk, g13=g13, g2=g2, bits=bits)


def _run(oracle, c, limit=7.0, **kw):
    return oracle.forward(c["x"], c["ids"], c["weights"], c["w13_packed"], c["w13_scales"],
                          c["w2_packed"], c["w2_scales"], bits=c["bits"], group_size=c["g13"],
                          group_size_w2=c["g2"], swiglu_limit=limit, **kw)


def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- pins

def pin_fp16_decode(oracle):
    """fp16 -> double equals numpy's float16 conversion for every pattern."""
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = allbits.view(np.float16).astype(np.float64)
    for b in list(range(0, 1 << 16, 97)) + [0x0001, 0x03FF, 0x0400, 0x7BFF, 0x8001, 0xFBFF, 0x3C00]:
        if np.isnan(ref[b]):
            continue
        assert oracle.fp16_to_double(b) == ref[b], hex(b)


def pin_bf16_rounding(oracle):
    """One-step RNE to bf16: exact-rational reference and torch's fp32->bf16."""
    rng = np.random.default_rng(5)
    vals = list(rng.standard_normal(300) * np.exp(rng.uniform(-20, 20, 300)))
    # ties and near-ties around 1: 1 + 2^-8 is a tie (-> 1.0, even); a hair above goes up
    vals += [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -30, -(1 + 2.0 ** -8),
             2.0 ** -130, 3 * 2.0 ** -134, 3.3895313892515355e38, 3.4e38, 1e-45]
    for v in vals:
        assert oracle.bf16_rne(v) == ind.bf16_bits_exact(v), v
    f32 = rng.standard_normal(2000).astype(np.float32)
    tb = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for v, b in zip(f32, tb):
        assert oracle.bf16_rne(float(v)) == int(b)


def pin_hand_words(oracle):
    with open(os.path.join(GOLDEN, "packed_words.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        bits = c["bits"]
        p = 32 // bits
        word = np.array([[int(c["word"], 16)]], dtype=np.uint32).view(np.int32)
        got = oracle.unpack(word, p, bits)[0].tolist()
        assert got == c["codes"], c
        assert oracle.pack(np.array([c["codes"]], np.int8), bits).view(np.uint32)[0, 0] == int(c["word"], 16)


def pin_pack_roundtrip(oracle):
    rng = np.random.default_rng(3)
    for bits in (2, 4):
        codes = synth.random_codes(rng, (7, 128), bits)
        words = oracle.pack(codes, bits)
        assert np.array_equal(oracle.unpack(words, 128, bits), codes)
        raw = rng.integers(0, 1 << 32, size=(5, 8), dtype=np.uint32).view(np.int32)
        K = 8 * 32 // bits
        assert np.array_equal(oracle.pack(oracle.unpack(raw, K, bits), bits), raw)
        # independent Python unpacking agrees
        for r in range(5):
            ref = []
            for wi in range(8):
                ref += ind.py_unpack_word(int(raw[r, wi]), bits)
            assert oracle.unpack(raw[r:r + 1], K, bits)[0].tolist() == ref


def pin_dequant(oracle):
    """bf16(code*scale) with exact rational rounding; W2 == code*bf16(scale)."""
    rng = np.random.default_rng(7)
    for bits, group in ((2, 32), (4, 16), (4, 64)):
        K = 128
        p = 32 // bits
        words = rng.integers(0, 1 << 32, size=(4, K // p), dtype=np.uint32).view(np.int32)
        scales = rng.uniform(0.001, 0.02, size=(4, K // group)).astype(np.float16)
        got = oracle.dequant(words, scales, K, group, bits)
        sbits = scales.view(np.uint16)
        for r in range(4):
            codes = []
            for wi in range(K // p):
                codes += ind.py_unpack_word(int(words[r, wi]), bits)
            for k in range(K):
                from fractions import Fraction
                s = Fraction(ind.fp16_value(int(sbits[r, k // group])))
                assert got[r, k] == ind.bf16_bits_exact(codes[k] * s), (bits, r, k)
                if bits == 2:
                    sb = ind.bf16_value(ind.bf16_bits_exact(s))
                    assert ind.bf16_value(int(got[r, k])) == codes[k] * sb


def pin_route(oracle):
    rng = np.random.default_rng(9)
    for R, E in ((64, 8), (1000, 37), (7, 256)):
        ids = rng.integers(0, E, size=R).astype(np.int32)
        counts, offsets, perm, inv = oracle.route(ids, E)
        assert np.array_equal(counts, np.bincount(ids, minlength=E))
        assert offsets[0] == 0 and offsets[-1] == R
        assert np.array_equal(perm, np.argsort(ids, kind="stable"))
        assert np.array_equal(inv[perm], np.arange(R))


def pin_zero_codes(oracle):
    """All-zero codes (stored 0xAAAAAAAA / 0x88888888) give exactly +0."""
    for bits, word in ((2, 0xAAAAAAAA), (4, 0x88888888)):
        c = _tiny_case(bits)
        c["w13_packed"] = np.full_like(c["w13_packed"], np.uint32(word).view(np.int32))
        c["w2_packed"] = np.full_like(c["w2_packed"], np.uint32(word).view(np.int32))
        out = _run(oracle, c)
        assert np.all(out == 0), bits


def pin_brute_force(oracle):
    """Pure-Python loops on tiny inputs give the same bits (fp64 mode)."""
    for bits in (2, 4):
        c = _tiny_case(bits, T=2, K=32, N=16, E=3, topk=2, g13=8, g2=8)
        got = _run(oracle, c)
        ref = ind.brute_force_forward(
            c["x"], c["ids"], c["weights"], c["w13_packed"], c["w13_scales"].view(np.uint16),
            c["w2_packed"], c["w2_scales"].view(np.uint16), c["K"], c["N"], c["E"], c["topk"],
            c["g13"], c["g2"], bits, 7.0)
        assert np.array_equal(got, ref), bits


def pin_fp32_mode(oracle):
    """The fp32 accumulation mode equals the same loops written with numpy
    binary32 scalars (every product and sum rounded).  SiLU's exponential
    comes from two different binary32 implementations (libm and numpy), so a
    rare one-ulp difference of h is allowed to show through."""
    for bits in (2, 4):
        c = _tiny_case(bits, T=2, K=32, N=16, E=3, topk=2, g13=8, g2=8)
        got = _run(oracle, c, accum="fp32")
        ref = ind.brute_force_forward(
            c["x"], c["ids"], c["weights"], c["w13_packed"], c["w13_scales"].view(np.uint16),
            c["w2_packed"], c["w2_scales"].view(np.uint16), c["K"], c["N"], c["E"], c["topk"],
            c["g13"], c["g2"], bits, 7.0, fp32=True)
        diff = np.abs(got.astype(np.int32) - ref.astype(np.int32))
        assert diff.max() <= 1 and (diff == 0).mean() >= 0.95, (bits, diff.max(), (diff == 0).mean())


def pin_given_h(oracle):
    """With h given, the oracle runs the down projection and the combine only:
    the pure-Python loops fed the same h give the same bits."""
    for bits in (2, 4):
        c = _tiny_case(bits, T=2, K=32, N=16, E=3, topk=2, g13=8, g2=8)
        rng = np.random.default_rng(17)
        h = synth.to_bf16_bits(rng.standard_normal((2 * 2, 16), dtype=np.float32))
        got = _run(oracle, c, h_in=h)
        ref = ind.brute_force_forward(
            c["x"], c["ids"], c["weights"], c["w13_packed"], c["w13_scales"].view(np.uint16),
            c["w2_packed"], c["w2_scales"].view(np.uint16), c["K"], c["N"], c["E"], c["topk"],
            c["g13"], c["g2"], bits, 7.0, h_in=h)
        assert np.array_equal(got, ref), bits


def _dense_mlp_torch(c, limit):
    """One expert, top-1, weight 1: a plain dense SwiGLU MLP in torch fp64 on the
    dequantised weights (numpy unpacking, torch bf16 rounding)."""
    bits = c["bits"]
    p = 32 // bits

    def deq(words, scales, group):
        w = words.view(np.uint32)[..., None] >> (bits * np.arange(p, dtype=np.uint32))
        codes = (w & ((1 << bits) - 1)).astype(np.int64).reshape(words.shape[0], -1) - (1 << (bits - 1))
        s = np.repeat(scales.astype(np.float64), group, axis=1)
        prod = torch.from_numpy(codes.astype(np.float64) * s).to(torch.float32)  # exact
        return prod.to(torch.bfloat16).to(torch.float64)

    W13 = deq(c["w13_packed"][0], c["w13_scales"][0], c["g13"])
    W2 = deq(c["w2_packed"][0], c["w2_scales"][0], c["g2"])
    x = torch.from_numpy(_bf16_to_f64(c["x"]))
    N = c["N"]
    gu = x @ W13.T
    g, u = gu[:, :N], gu[:, N:]
    h = (torch.nn.functional.silu(torch.clamp(g, max=limit)) * torch.clamp(u, -limit, limit))
    h = h.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    y = (h @ W2.T).to(torch.float32).to(torch.bfloat16)
    return y.view(torch.int16).numpy().view(np.uint16)


def pin_dense_mlp(oracle):
    for bits in (2, 4):
        c = _tiny_case(bits, T=6, K=64, N=32, E=1, topk=1, g13=16, g2=32, scale=(0.05, 0.4))
        c["ids"] = np.zeros((6, 1), np.int32)
        c["weights"] = np.ones((6, 1), np.float32)
        got = _run(oracle, c, limit=7.0)
        ref = _dense_mlp_torch(c, 7.0)
        # torch rounds through fp32 (two roundings); allow a rare one-ulp flip
        diff = np.abs(got.astype(np.int32) - ref.astype(np.int32))
        assert diff.max() <= 1 and (diff == 0).mean() > 0.97, (bits, diff.max(), (diff == 0).mean())
        assert np.abs(_bf16_to_f64(got)).max() > 0


def _clamp_case(gate_code, gate_scale, up_code, up_scale):
    """E=1, top-1, K=N=16, 2-bit, group 16: x = e_0, so g = gate_code*gate_scale,
    u = up_code*up_scale in row 0, every other h is 0, and each w2 row copies h_0."""
    K = N = 16
    bits = 2

    def word(code0):
        codes = np.zeros((1, 16), np.int8)
        codes[0, 0] = code0
        return codes

    import oracle as o
    zero = o.pack(np.zeros((1, 16), np.int8), bits)[0, 0]
    w13 = np.full((1, 2 * N, 1), zero, np.int32)
    w13[0, 0, 0] = o.pack(word(gate_code), bits)[0, 0]
    w13[0, N, 0] = o.pack(word(up_code), bits)[0, 0]
    w13s = np.ones((1, 2 * N, 1), np.float16)
    w13s[0, 0, 0] = gate_scale
    w13s[0, N, 0] = up_scale
    w2 = np.full((1, K, 1), o.pack(word(1), bits)[0, 0], np.int32)
    w2s = np.ones((1, K, 1), np.float16)
    x = np.zeros((1, K), np.float32)
    x[0, 0] = 1.0
    return dict(x=synth.to_bf16_bits(x), ids=np.zeros((1, 1), np.int32), weights=np.ones((1, 1), np.float32),
                w13_packed=w13, w13_scales=w13s, w2_packed=w2, w2_scales=w2s, K=K, N=N, E=1, topk=1,
                g13=16, g2=16, bits=bits)


def pin_clamp_closed_form(oracle):
    L = 7.0
    silu = lambda z: z / (1.0 + math.exp(-z))  # noqa: E731
    cases = [
        ((1, 10.0, 1, 1.0), silu(7.0) * 1.0),      # gate 10 is clamped to 7
        ((1, 1.0, -1, 10.0), silu(1.0) * -7.0),    # up -10 is clamped to -7
        ((-1, 10.0, 1, 1.0), silu(-10.0) * 1.0),   # gate -10 is not clamped
        ((1, 2.0, 1, 8.0), silu(2.0) * 7.0),       # up 8 is clamped to 7
        ((1, 0.5, -2, 1.5), silu(0.5) * -3.0),     # inside the limits
    ]
    for args, h0 in cases:
        c = _clamp_case(*args)
        out = _run(oracle, c, limit=L)
        expect = ind.bf16_bits_exact(ind.bf16_value(ind.bf16_bits_exact(h0)))
        assert np.all(out[0] == expect), (args, out[0][:2], expect)
    # no limit (+inf): gate 10 passes through
    c = _clamp_case(1, 10.0, 1, 1.0)
    out = _run(oracle, c, limit=float("inf"))
    assert np.all(out[0] == ind.bf16_bits_exact(silu(10.0)))


def pin_scale_doubling(oracle):
    for bits in (2, 4):
        c = _tiny_case(bits, T=4, K=64, N=32, E=3, topk=2)
        out = _run(oracle, c)
        c2 = dict(c)
        c2["w2_scales"] = (c["w2_scales"].astype(np.float32) * 2).astype(np.float16)
        out2 = _run(oracle, c2)
        assert np.array_equal(_bf16_to_f64(out2), 2 * _bf16_to_f64(out))


def pin_relabel_and_token_permutation(oracle):
    for bits in (2, 4):
        c = _tiny_case(bits, T=5, K=64, N=32, E=4, topk=2)
        out = _run(oracle, c)
        sigma = np.array([2, 0, 3, 1])        # new label of old expert e is sigma[e]
        c2 = dict(c)
        for key in ("w13_packed", "w13_scales", "w2_packed", "w2_scales"):
            arr = np.empty_like(c[key])
            arr[sigma] = c[key]
            c2[key] = arr
        c2["ids"] = sigma[c["ids"]].astype(np.int32)
        assert np.array_equal(_run(oracle, c2), out)
        tp = np.array([3, 0, 4, 2, 1])
        c3 = dict(c, x=c["x"][tp], ids=c["ids"][tp], weights=c["weights"][tp])
        assert np.array_equal(_run(oracle, c3), out[tp])


def pin_split_routing_weight(oracle):
    """Two slots on the same expert with weights 0.25 and 0.75 equal one slot of
    weight 1 (the sum w*y + (1-w)*y is exact here), and weight 0.5 halves it."""
    for bits in (2, 4):
        c = _tiny_case(bits, T=3, K=64, N=32, E=3, topk=2)
        c1 = dict(c, ids=c["ids"][:, :1].copy(), weights=np.ones((3, 1), np.float32), topk=1)
        one = _run(oracle, c1)
        c2 = dict(c, ids=np.repeat(c["ids"][:, :1], 2, axis=1),
                  weights=np.tile(np.array([[0.25, 0.75]], np.float32), (3, 1)))
        assert np.array_equal(_run(oracle, c2), one)
        c3 = dict(c1, weights=np.full((3, 1), 0.5, np.float32))
        assert np.array_equal(_bf16_to_f64(_run(oracle, c3)), 0.5 * _bf16_to_f64(one))


def pin_router(oracle):
    """Router: ids are numpy's stable argsort of the fp32 scores (ties to the
    lower index); weights match scipy's softmax renormalised over the chosen
    experts; closed forms (k = 1 gives weight 1, all-equal scores give 1/k in
    index order, two scores ln 3 apart give 3/4 and 1/4, k = E is the full
    softmax); a constant shift changes nothing; a bias of -1e4 removes an
    expert."""
    from scipy.special import softmax
    rng = np.random.default_rng(21)
    for T, E, k, with_bias in ((5, 8, 2, False), (7, 64, 8, True), (3, 256, 8, True), (2, 5, 5, False)):
        lg = rng.standard_normal((T, E), dtype=np.float32)
        bias = (-1.1 * np.log(np.arange(1, E + 1))).astype(np.float32) if with_bias else None
        ids, w = oracle.route_topk(lg, k, bias)
        z = lg + (bias if with_bias else np.float32(0))
        assert z.dtype == np.float32
        assert np.array_equal(ids, np.argsort(-z, axis=1, kind="stable")[:, :k])
        p = softmax(z.astype(np.float64), axis=1)
        sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
        ref = (sel / sel.sum(axis=1, keepdims=True)).astype(np.float32)
        assert np.max(np.abs(w.astype(np.float64) - ref) / ref) <= 2 * 2.0 ** -24, (T, E, k)
        assert np.all(np.abs(w.sum(axis=1) - 1.0) <= k * 2.0 ** -24)
        if k == E:
            assert np.allclose(w, softmax(z.astype(np.float64), axis=1)[np.arange(T)[:, None], ids], rtol=3e-7)
        # an exact constant shift (scores are multiples of 2^-10 below 16)
        q = np.round(lg * 1024) / 1024
        a = oracle.route_topk(q.astype(np.float32), k, bias)
        b = oracle.route_topk((q + 3.0).astype(np.float32), k, bias)
        assert np.array_equal(a[0], b[0])
        assert np.max(np.abs(a[1].astype(np.float64) - b[1])) <= 2.0 ** -23
    ids, w = oracle.route_topk(np.zeros((2, 6), np.float32), 3)
    assert ids.tolist() == [[0, 1, 2], [0, 1, 2]] and np.all(w == np.float32(1 / 3))
    ids, w = oracle.route_topk(np.array([[0.5, -2.0, 0.7, 0.1]], np.float32), 1)
    assert ids.tolist() == [[2]] and w[0, 0] == 1.0
    lg = np.array([[-3.0, 1.0, 1.0 - math.log(3.0), -5.0]], np.float32)
    ids, w = oracle.route_topk(lg, 2)
    assert ids.tolist() == [[1, 2]]
    assert abs(float(w[0, 0]) - 0.75) <= 2e-7 and abs(float(w[0, 1]) - 0.25) <= 2e-7
    bias = np.zeros(6, np.float32)
    bias[[0, 1, 2]] = -1e4
    ids, _ = oracle.route_topk(np.zeros((1, 6), np.float32), 3, bias)
    assert ids.tolist() == [[3, 4, 5]]


def pin_ep_profile(oracle):
    """Expert-parallel profile: an expert range with no routed slot gives +0;
    a top-1 slot of weight 1 gives its y exactly; partials over disjoint
    ranges that cover all experts add up (fp32) to the partial over all of
    them; BF16 of the all-expert partial equals the single-device output but
    for rare double-rounding cases; the rank sum adds in rank order in fp32
    (numpy float32 arithmetic) and rounds like torch's fp32 -> bf16."""
    for bits in (2, 4):
        c = _tiny_case(bits, T=5, K=64, N=32, E=4, topk=2)
        out, _, y = _run(oracle, c, return_intermediates=True)
        E = c["E"]
        assert np.all(oracle.combine_partial(c["ids"], c["weights"], y, (E, E)) == 0.0)
        unused = [e for e in range(E) if e not in set(c["ids"].ravel().tolist())]
        for e in unused:
            assert np.all(oracle.combine_partial(c["ids"], c["weights"], y, (e, e + 1)) == 0.0)
        full = oracle.combine_partial(c["ids"], c["weights"], y, (0, E))
        parts = [oracle.combine_partial(c["ids"], c["weights"], y, r) for r in ((0, 1), (1, 3), (3, E))]
        s = (parts[0] + parts[1]) + parts[2]
        mag = np.abs(parts[0]).astype(np.float64) + np.abs(parts[1]) + np.abs(parts[2])
        assert np.all(np.abs(s.astype(np.float64) - full) <= 4 * 2.0 ** -24 * mag)
        fb = torch.from_numpy(full).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        diff = np.abs(fb.astype(np.int32) - out.astype(np.int32))
        assert diff.max() <= 1 and (diff == 0).mean() >= 0.99
        got = oracle.sum_partials(parts)
        ref32 = (parts[0].astype(np.float32) + parts[1].astype(np.float32)) + parts[2].astype(np.float32)
        assert np.array_equal(got, torch.from_numpy(ref32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    c = _tiny_case(2, T=3, K=64, N=32, E=3, topk=1)
    c["weights"] = np.ones((3, 1), np.float32)
    _, _, y = _run(oracle, c, return_intermediates=True)
    p = oracle.combine_partial(c["ids"], c["weights"], y, (0, 3))
    assert np.array_equal(p, _bf16_to_f64(y).astype(np.float32))
    assert np.all(oracle.sum_partials([p, -p]) == 0)


def pin_fp16_rounding(oracle):
    """One-step RNE to binary16 equals numpy's double -> half conversion."""
    rng = np.random.default_rng(31)
    vals = list(rng.standard_normal(400) * np.exp(rng.uniform(-20, 12, 400)))
    vals += [65504.0, 65519.99, 65520.0, 70000.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14,
             (2.0 ** -14) * (1 - 2.0 ** -12), 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, -0.0, 0.0]
    with np.errstate(over="ignore"):
        for v in vals:
            assert oracle.fp16_rne(v) == int(np.array(v, np.float64).astype(np.float16).view(np.uint16)), v


def _q_case(rows=6, K=256, seed=41, scale=0.02):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((rows, K)) * scale).astype(np.float32)
    w[:, 5] *= 6.0                     # an outlier column
    imp = np.exp(rng.standard_normal(K)).astype(np.float32)
    return w, imp


def pin_quantizer(oracle):
    """Quantiser: weights that are exactly code x scale come back exactly;
    the searched scale never has a larger weighted error than plain RTN (f = 1
    is a candidate); the packed words and scales, dequantised by the forward's
    own dequantisation, reproduce the reconstruction the errors were measured
    on; scaling w by 8 scales the scales by 8 and the errors by 64 exactly;
    a one-hot importance picks the candidate best for that one weight (checked
    in exact rational arithmetic over all 31 candidates); an all-zero group
    gets scale 0 and code 0."""
    from fractions import Fraction
    for bits in (2, 4):
        lo, hi = -(1 << (bits - 1)), (1 << (bits - 1)) - 1
        p = 32 // bits
        rng = np.random.default_rng(bits)
        # (a) exact representability, plain RTN
        codes = rng.integers(lo, hi + 1, size=(3, 128)).astype(np.int8)
        codes[:, 7] = lo
        sv = np.array([1.25 * 2.0 ** -6, 1.5 * 2.0 ** -9, 0.375], np.float16)   # products exact in BF16
        w = (codes.astype(np.float32) * sv.astype(np.float32)[:, None]).astype(np.float32)
        pk, sc, m = oracle.quantize(w, bits, 128, None, search=False)
        assert np.array_equal(sc.view(np.uint16)[:, 0], sv.view(np.uint16))
        assert np.array_equal(oracle.unpack(pk, 128, bits), codes)
        assert np.all(m[:, 0] == 0) and np.all(m[:, 1] == 0)
        w, imp = _q_case()
        for g in (32, 128):
            pk0, sc0, m0 = oracle.quantize(w, bits, g, imp, search=False)
            pk1, sc1, m1 = oracle.quantize(w, bits, g, imp, search=True)
            assert np.all(m1[:, 0] <= m0[:, 0]) and m1[:, 0].sum() < m0[:, 0].sum()
            # (c) consistency with the forward's dequantisation
            for pk_, sc_, m_ in ((pk0, sc0, m0), (pk1, sc1, m1)):
                deq = _bf16_to_f64(oracle.dequant(pk_, sc_, w.shape[1], g, bits))
                d = w.astype(np.float64) - deq
                assert np.allclose(m_[:, 1], (d * d).sum(axis=1), rtol=1e-12, atol=0)
                assert np.allclose(m_[:, 0], (imp * d * d).sum(axis=1), rtol=1e-12, atol=0)
                assert np.allclose(m_[:, 3], (w.astype(np.float64) ** 2).sum(axis=1), rtol=1e-12)
            # (d) power-of-two homogeneity
            pk8, sc8, m8 = oracle.quantize(w * np.float32(8), bits, g, imp, search=True)
            assert np.array_equal(pk8, pk1)
            assert np.array_equal(sc8.astype(np.float64), 8 * sc1.astype(np.float64))
            assert np.array_equal(m8, 64 * m1)
        # (e) one-hot importance, exact arithmetic over the candidates
        wg = w[:1, :128]
        k0 = 5
        onehot = np.zeros(128, np.float32)
        onehot[k0] = 1.0
        _, sc, _ = oracle.quantize(wg, bits, 128, onehot, search=True)
        mx = Fraction(float(np.abs(wg).max()))

        def err(sf):
            s = Fraction(sf)
            q = max(lo, min(hi, round(Fraction(float(np.float32(wg[0, k0]) / np.float32(sf))))))
            return abs(Fraction(float(wg[0, k0])) - Fraction(ind.bf16_value(ind.bf16_bits_exact(q * s))))
        cands = []
        for i in range(31):
            f = np.float32(10 + i) / np.float32(20)
            s0 = np.float32(float(mx)) / np.float32(1 << (bits - 1))
            cands.append(float(np.float16(np.float32(s0 * f))))
        best = min(err(c) for c in cands)
        assert err(float(sc[0, 0])) == best, bits
        # (g) an all-zero group
        z = np.zeros((1, 128), np.float32)
        pkz, scz, mz = oracle.quantize(z, bits, 128, imp[:128], search=True)
        assert scz[0, 0] == 0 and np.all(oracle.unpack(pkz, 128, bits) == 0) and np.all(mz == 0)
        assert p * pkz.shape[1] == 128


PINS = [pin_fp16_decode, pin_bf16_rounding, pin_hand_words, pin_pack_roundtrip, pin_dequant,
        pin_route, pin_zero_codes, pin_brute_force, pin_dense_mlp, pin_clamp_closed_form,
        pin_scale_doubling, pin_relabel_and_token_permutation, pin_split_routing_weight, pin_fp32_mode,
        pin_given_h, pin_router, pin_ep_profile, pin_fp16_rounding, pin_quantizer]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(clean_oracle, pin):
    pin(clean_oracle)


@pytest.mark.parametrize("mutation", sorted(__import__("oracle").MUTATIONS))
def test_every_planted_mistake_is_caught(clean_oracle, mutation):
    clean_oracle.set_mutation(mutation)
    failed = []
    for pin in PINS:
        try:
            pin(clean_oracle)
        except (AssertionError, Exception) as exc:  # noqa: B014 - any failure counts
            failed.append((pin.__name__, type(exc).__name__))
    assert failed, f"no pin caught mutation {mutation}"


def test_fp32_mode_close_to_fp64(clean_oracle):
    c = _tiny_case(4, T=8, K=256, N=128, E=4, topk=2, g13=128, g2=64)
    a = _run(clean_oracle, c)
    b = _run(clean_oracle, c, accum="fp32")
    diff = np.abs(a.astype(np.int32) - b.astype(np.int32))
    assert (diff == 0).mean() > 0.95 and diff.max() <= 2


def test_token_subset_matches_full(clean_oracle):
    c = _tiny_case(2, T=6, K=64, N=32, E=3, topk=2)
    full = _run(clean_oracle, c)
    sub = _run(clean_oracle, c, tokens=np.array([4, 1]))
    assert np.array_equal(sub, full[[4, 1]])


def test_out_of_range_id_is_an_error(clean_oracle):
    c = _tiny_case(2)
    c["ids"] = c["ids"].copy()
    c["ids"][0, 0] = c["E"]
    with pytest.raises(clean_oracle.OracleError):
        _run(clean_oracle, c)
