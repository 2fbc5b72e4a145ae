"""CPU oracle for the WNA16 routed-expert MoE forward (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The CUDA product path never
imports it and shares no code with it; the arithmetic lives in
``wna16_oracle.c`` (plain C, built with gcc), and this module only marshals
numpy arrays into it.

Every function here follows the definition in ``wna16_oracle.c``; see the
header of that file for the passages of the pages each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wna16_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

# Planted-mistake switches (see the enum in wna16_oracle.c); tests only.
MUTATIONS = {
    "msb_first": 1,
    "code_offset": 2,
    "gate_up_swap": 3,
    "no_clamp": 4,
    "group_axis": 5,
    "w2_transpose": 6,
    "no_route_weight": 7,
    "unstable_perm": 8,
    "silu_sign": 9,
    "topk_tie_high": 10,
    "topk_no_renorm": 11,
    "topk_no_bias": 12,
    "q_no_importance": 13,
    "q_clamp_high": 14,
}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` with gcc (OpenMP)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    lib.oracle_set_mutation.argtypes = [I]
    lib.oracle_set_mutation.restype = I
    lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_fp16_to_double.restype = ctypes.c_double
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_bf16_rne.argtypes = [ctypes.c_double]
    lib.oracle_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_pack.argtypes = [P, I64, I64, I, P]
    lib.oracle_pack.restype = I
    lib.oracle_unpack.argtypes = [P, I64, I64, I, P]
    lib.oracle_unpack.restype = I
    lib.oracle_dequant.argtypes = [P, P, I64, I64, I64, I, P]
    lib.oracle_dequant.restype = I
    lib.oracle_route.argtypes = [P, I64, I64, P, P, P, P]
    lib.oracle_route.restype = I
    lib.oracle_forward.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64, I, I64, I64, I,
                                   ctypes.c_float, I, P, I64, P, P, P, P]
    lib.oracle_forward.restype = I
    lib.oracle_combine_partial.argtypes = [P, P, P, I64, I64, I, I64, I64, P]
    lib.oracle_combine_partial.restype = I
    lib.oracle_sum_partials.argtypes = [P, I, I64, P]
    lib.oracle_sum_partials.restype = I
    lib.oracle_fp16_rne.argtypes = [ctypes.c_double]
    lib.oracle_fp16_rne.restype = ctypes.c_uint16
    lib.oracle_quantize.argtypes = [P, I64, I64, P, I, I64, I, P, P, P]
    lib.oracle_quantize.restype = I
    lib.oracle_route_topk.argtypes = [P, P, I64, I64, I, P, P]
    lib.oracle_route_topk.restype = I
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = I
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(ValueError):
    pass


def set_mutation(name: str | None) -> None:
    """Plant a known mistake in the oracle (None restores the correct oracle)."""
    code = 0 if name is None else MUTATIONS[name]
    if _load().oracle_set_mutation(code) != 0:
        raise OracleError(name)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def fp16_to_double(h: int) -> float:
    return float(_load().oracle_fp16_to_double(h))


def bf16_to_double(b: int) -> float:
    return float(_load().oracle_bf16_to_double(b))


def bf16_rne(v: float) -> int:
    """Nearest bfloat16 (ties to even) of a double, as its 16-bit pattern."""
    return int(_load().oracle_bf16_rne(float(v)))


def fp16_rne(v: float) -> int:
    """Nearest binary16 (ties to even) of a double, as its 16-bit pattern."""
    return int(_load().oracle_fp16_rne(float(v)))


def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    """int8 codes [rows, K] -> int32 words [rows, K*bits/32]."""
    codes = _c(codes, np.int8)
    rows, K = codes.shape
    out = np.empty((rows, K * bits // 32), np.int32)
    if _load().oracle_pack(_ptr(codes), rows, K, bits, _ptr(out)) != 0:
        raise OracleError("pack: bad bits / K / code range")
    return out


def unpack(packed: np.ndarray, K: int, bits: int) -> np.ndarray:
    packed = _c(packed, np.int32)
    rows = packed.shape[0]
    out = np.empty((rows, K), np.int8)
    if _load().oracle_unpack(_ptr(packed), rows, K, bits, _ptr(out)) != 0:
        raise OracleError("unpack: bad bits / K")
    return out


def dequant(packed: np.ndarray, scales_fp16: np.ndarray, K: int, group: int, bits: int) -> np.ndarray:
    """Dequantised BF16 weights [rows, K] as uint16 bit patterns."""
    packed = _c(packed, np.int32)
    scales = _c(scales_fp16, np.float16).view(np.uint16)
    rows = packed.shape[0]
    out = np.empty((rows, K), np.uint16)
    if _load().oracle_dequant(_ptr(packed), _ptr(scales), rows, K, group, bits, _ptr(out)) != 0:
        raise OracleError("dequant: bad arguments")
    return out


def route(ids: np.ndarray, E: int):
    """Routing lists for flat slots f = t*topk + j: (counts, offsets, perm, inv)."""
    ids = _c(ids, np.int32).reshape(-1)
    R = ids.size
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(R, np.int32)
    inv = np.empty(R, np.int32)
    if _load().oracle_route(_ptr(ids), R, E, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv)) != 0:
        raise OracleError("route: expert id out of range")
    return counts, offsets, perm, inv


def forward(x_bf16: np.ndarray, ids: np.ndarray, weights: np.ndarray,
            w13_packed: np.ndarray, w13_scales: np.ndarray,
            w2_packed: np.ndarray, w2_scales: np.ndarray,
            *, bits: int, group_size: int, group_size_w2: int | None = None,
            swiglu_limit: float = 7.0, accum: str = "fp64", tokens=None,
            return_intermediates: bool = False, h_in: np.ndarray | None = None):
    """Oracle forward.  ``x_bf16`` is uint16 [T, K] (BF16 bit patterns);
    returns BF16 bit patterns ``out`` [n_tok, K] (and h [n_tok*topk, N],
    y [n_tok*topk, K] in slot order when ``return_intermediates``).
    With ``h_in`` (BF16 bits [n_tok*topk, N], slot order) the gate/up
    projection and SwiGLU are skipped and ``h_in`` is used as h."""
    x = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    wts = _c(weights, np.float32)
    w13p = _c(w13_packed, np.int32)
    w13s = _c(w13_scales, np.float16).view(np.uint16)
    w2p = _c(w2_packed, np.int32)
    w2s = _c(w2_scales, np.float16).view(np.uint16)
    T, K = x.shape
    topk = ids.shape[1]
    E = w13p.shape[0]
    N = w13p.shape[1] // 2
    g2 = group_size if not group_size_w2 else group_size_w2
    tok = None if tokens is None else _c(tokens, np.int64)
    n_tok = T if tok is None else tok.size
    out = np.empty((n_tok, K), np.uint16)
    h = np.empty((n_tok * topk, N), np.uint16) if return_intermediates else None
    y = np.empty((n_tok * topk, K), np.uint16) if return_intermediates else None
    hin = None
    if h_in is not None:
        hin = _c(h_in, np.uint16)
        if hin.shape != (n_tok * topk, N):
            raise OracleError(f"h_in must be [{n_tok * topk}, {N}]")
    rc = _load().oracle_forward(
        _ptr(x), _ptr(ids), _ptr(wts), _ptr(w13p), _ptr(w13s), _ptr(w2p), _ptr(w2s),
        T, K, N, E, topk, group_size, g2, bits, float(swiglu_limit),
        0 if accum == "fp64" else 1, _ptr(tok), n_tok, _ptr(hin), _ptr(out), _ptr(h), _ptr(y))
    if rc != 0:
        raise OracleError("forward: bad arguments or expert id out of range")
    if return_intermediates:
        return out, h, y
    return out


def route_topk(logits: np.ndarray, k: int, bias: np.ndarray | None = None):
    """Router: softmax of (logits + bias) over the experts, the top k (ties to
    the lower expert index), renormalised.  logits fp32 [T, E], bias fp32 [E]
    or None; returns (ids int32 [T, k], weights fp32 [T, k])."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    b = None if bias is None else _c(bias, np.float32)
    if b is not None and b.shape != (E,):
        raise OracleError("bias must be [E]")
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    if _load().oracle_route_topk(_ptr(lg), _ptr(b), T, E, k, _ptr(ids), _ptr(w)) != 0:
        raise OracleError("route_topk: k must be in [1, E]")
    return ids, w


def combine_partial(ids: np.ndarray, weights: np.ndarray, y_bf16: np.ndarray, expert_range) -> np.ndarray:
    """Expert-parallel partial output of one rank: fp32 [n, K] = sum over the
    slots routed to experts in [begin, end) of w * y (fp64, rounded once to
    fp32), slots in order.  y is the BF16 bits of the down projection per
    slot t*topk + j ([n*topk, K], e.g. forward(..., return_intermediates=True))."""
    ids = _c(ids, np.int32)
    wts = _c(weights, np.float32)
    y = _c(y_bf16, np.uint16)
    n, topk = ids.shape
    K = y.shape[1]
    if y.shape[0] != n * topk:
        raise OracleError("y must be [n*topk, K]")
    out = np.empty((n, K), np.float32)
    b, e = expert_range
    if _load().oracle_combine_partial(_ptr(ids), _ptr(wts), _ptr(y), n, K, topk, int(b), int(e), _ptr(out)) != 0:
        raise OracleError("combine_partial: bad arguments")
    return out


def sum_partials(partials) -> np.ndarray:
    """bf16 bits of the fp32 sum of the ranks' partial outputs, ranks added in order."""
    p = _c(np.stack(partials), np.float32)
    P = p.shape[0]
    out = np.empty(p.shape[1:], np.uint16)
    if _load().oracle_sum_partials(_ptr(p), P, int(np.prod(p.shape[1:])), _ptr(out)) != 0:
        raise OracleError("sum_partials: bad arguments")
    return out


def quantize(w: np.ndarray, bits: int, group: int, importance: np.ndarray | None = None, search: bool = True):
    """Symmetric RTN quantiser with an importance-weighted scale search (the
    definition in wna16_oracle.c).  w fp32 [rows, K], importance fp32 [K] or
    None; returns (packed int32 [rows, K*bits/32], scales fp16 [rows, K/group],
    metrics fp64 [rows, 4]: weighted error, unweighted error, sum a w^2, sum w^2)."""
    wa = _c(w, np.float32)
    rows, K = wa.shape
    imp = None if importance is None else _c(importance, np.float32)
    if imp is not None and imp.shape != (K,):
        raise OracleError("importance must be [K]")
    packed = np.empty((rows, K * bits // 32), np.int32)
    scales = np.empty((rows, K // group), np.uint16)
    metrics = np.empty((rows, 4), np.float64)
    if _load().oracle_quantize(_ptr(wa), rows, K, _ptr(imp), bits, group, 1 if search else 0, _ptr(packed),
                               _ptr(scales), _ptr(metrics)) != 0:
        raise OracleError("quantize: bad arguments")
    return packed, scales.view(np.float16), metrics
