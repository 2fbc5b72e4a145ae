"""Independent pure-Python restatements used to pin the oracle (tests only).

These are written separately from ``oracle/wna16_oracle.c`` with different
techniques (exact rational arithmetic for rounding, Python integer bit
operations for unpacking, plain Python loops for the forward) so that a
mistake in the oracle does not repeat here.  They are slow and only run on
tiny inputs.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


def bf16_bits_exact(v) -> int:
    """Nearest bfloat16 of the real number ``v`` (int/float/Fraction), ties to
    even, computed in exact rational arithmetic; returns the bit pattern."""
    v = Fraction(v)
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    # exponent e with 2^e <= a < 2^(e+1)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = max(e - 7, -133)                       # quantum: 8 significant bits
    scaled = a / (Fraction(2) ** q)
    n = math.floor(scaled)
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = Fraction(n) * Fraction(2) ** q
    if r > Fraction(2) ** 127 * Fraction(255, 128):
        return sign | 0x7F80
    f32 = np.array([float(r)], np.float32)      # exact: r has <= 8 significant bits
    return sign | int(f32.view(np.uint32)[0] >> 16)


def bf16_value(bits: int) -> float:
    return float(np.array([bits << 16], np.uint32).view(np.float32)[0])


def fp16_value(bits: int) -> float:
    return float(np.array([bits], np.uint16).view(np.float16)[0])


def py_unpack_word(word: int, bits: int):
    """Codes of one INT32 word, element order = field order LSB-first."""
    w = word & 0xFFFFFFFF
    p = 32 // bits
    mask = (1 << bits) - 1
    return [((w >> (bits * j)) & mask) - (1 << (bits - 1)) for j in range(p)]


def py_dequant_matrix(packed, scales_bits, K, group, bits):
    """Dequantised weights as Python floats (list of rows)."""
    p = 32 // bits
    out = []
    for r in range(len(packed)):
        codes = []
        for wi in range(K // p):
            codes += py_unpack_word(int(packed[r][wi]), bits)
        row = []
        for k in range(K):
            s = Fraction(fp16_value(int(scales_bits[r][k // group])))
            row.append(bf16_value(bf16_bits_exact(codes[k] * s)))
        out.append(row)
    return out


def brute_force_forward(x_bits, ids, wts, w13p, w13s_bits, w2p, w2s_bits, K, N, E, topk,
                        g13, g2, bits, limit, fp32=False, h_in=None):
    """Plain loops over tokens, slots, rows and columns; sums in ascending
    order, in fp64 (default) or, with ``fp32``, in IEEE binary32 with every
    product and every addition rounded (numpy float32 scalars; SiLU's
    exponential in binary32 too); BF16 rounding of the weights, h, y and out.
    With ``h_in`` (BF16 bits per slot t*topk + j, [T*topk, N]) the gate/up
    projection and SwiGLU are skipped and h_in is used as h."""
    f32 = np.float32
    T = len(x_bits)
    W13 = None if h_in is not None else [py_dequant_matrix(w13p[e], w13s_bits[e], K, g13, bits) for e in range(E)]
    W2 = [py_dequant_matrix(w2p[e], w2s_bits[e], N, g2, bits) for e in range(E)]
    out = []
    for t in range(T):
        xs = [bf16_value(int(b)) for b in x_bits[t]]
        ys = []
        for j in range(topk):
            e = int(ids[t][j])
            h = []
            for n in range(N):
                if h_in is not None:
                    h.append(bf16_value(int(h_in[t * topk + j][n])))
                    continue
                if fp32:
                    g = f32(0.0)
                    u = f32(0.0)
                    for k in range(K):
                        g = f32(g + f32(f32(W13[e][n][k]) * f32(xs[k])))
                        u = f32(u + f32(f32(W13[e][N + n][k]) * f32(xs[k])))
                    gc = min(g, f32(limit))
                    uc = max(f32(-limit), min(u, f32(limit)))
                    val = float(f32(f32(gc / f32(f32(1.0) + np.exp(f32(-gc)))) * uc))
                else:
                    g = 0.0
                    u = 0.0
                    for k in range(K):
                        g += W13[e][n][k] * xs[k]
                    for k in range(K):
                        u += W13[e][N + n][k] * xs[k]
                    gc = min(g, limit)
                    uc = max(-limit, min(u, limit))
                    val = gc / (1.0 + math.exp(-gc)) * uc
                h.append(bf16_value(bf16_bits_exact(val)))
            y = []
            for m in range(K):
                if fp32:
                    acc = f32(0.0)
                    for n in range(N):
                        acc = f32(acc + f32(f32(W2[e][m][n]) * f32(h[n])))
                    acc = float(acc)
                else:
                    acc = 0.0
                    for n in range(N):
                        acc += W2[e][m][n] * h[n]
                y.append(bf16_value(bf16_bits_exact(acc)))
            ys.append(y)
        row = []
        for m in range(K):
            if fp32:
                acc = f32(0.0)
                for j in range(topk):
                    acc = f32(acc + f32(f32(wts[t][j]) * f32(ys[j][m])))
                acc = float(acc)
            else:
                acc = 0.0
                for j in range(topk):
                    acc += float(np.float32(wts[t][j])) * ys[j][m]
            row.append(bf16_bits_exact(acc))
        out.append(row)
    return np.array(out, dtype=np.uint16)
