"""Thin Python binding of ``libwna16_moe.so`` (argument marshalling only).

Every function takes torch CUDA tensors, checks dtype / shape / contiguity,
and passes raw device pointers plus the current CUDA stream to the C ABI
declared in ``include/wna16_moe.h``.  All computation happens in the
library's sm_103a kernels; if the library is missing, loading fails loudly
(there is no fallback implementation).
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libwna16_moe.so")
DEBUG_LIB_PATH = os.path.join(HERE, "libwna16_moe_debug.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "wna16_moe.h")

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE_TOO_SMALL = -3
ERR_CUDA = -4
ERR_BAD_ROUTING = -5
ERR_DEVICE_TIMEOUT = -6
ERR_INDEX = -7

_lib = None
_debug_lib = None


class Wna16Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"wna16 error {code}: {msg}")
        self.code = code


def exported_names_in_header() -> list[str]:
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"WNA16_API\s+[\w\s\*]+?\b(wna16_\w+)\s*\(", text)


def load_library(path: str = LIB_PATH):
    """Load the CUDA library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = _open(path)
    return _lib


def load_debug_library():
    """The bounds-checked build of the same library (built with
    build.build(debug=True)): same entry points, and an index that falls
    outside its buffer sets the status word to ERR_INDEX instead of touching
    memory out of bounds."""
    global _debug_lib
    if _debug_lib is None:
        _debug_lib = _open(DEBUG_LIB_PATH)
    return _debug_lib


def _open(path: str):
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with wna16_grouped_gemm_gb300.build.build() "
                           "(there is no non-CUDA implementation)")
    lib = ctypes.CDLL(path)
    P, I64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    SZ = ctypes.c_size_t
    lib.wna16_moe_last_error.restype = ctypes.c_char_p
    lib.wna16_moe_last_error.argtypes = []
    lib.wna16_moe_workspace_size.restype = SZ
    lib.wna16_moe_workspace_size.argtypes = [I64, I64, I64, I64, I, I]
    lib.wna16_moe_pack.restype = I
    lib.wna16_moe_pack.argtypes = [P, I64, I64, I, P, P]
    lib.wna16_moe_forward.restype = I
    lib.wna16_moe_forward.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64, I, I, I, I, F, P, P, SZ, P]
    lib.wna16_moe_read_status.restype = I
    lib.wna16_moe_read_status.argtypes = [P, ctypes.POINTER(ctypes.c_int), P]
    lib.wna16_moe_route.restype = I
    lib.wna16_moe_route.argtypes = [P, I64, I, I64, I64, I64, I, P, P, P, P, P, SZ, P]
    lib.wna16_moe_w13.restype = I
    lib.wna16_moe_w13.argtypes = [P, P, P, P, I64, I64, I64, I64, I, I, I, F, P, P, SZ, P]
    lib.wna16_moe_w2.restype = I
    lib.wna16_moe_w2.argtypes = [P, P, P, I64, I64, I64, I64, I, I, I, P, P, SZ, P]
    lib.wna16_moe_forward_noalloc.restype = I
    lib.wna16_moe_forward_noalloc.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64, I, I, I, I, F, P, P]
    lib.wna16_moe_check_wait_timeout.restype = I
    lib.wna16_moe_check_wait_timeout.argtypes = [P, SZ, I64, P]
    lib.wna16_moe_launches_last_forward.restype = I
    lib.wna16_moe_launches_last_forward.argtypes = []
    lib.wna16_moe_profile.restype = I
    lib.wna16_moe_profile.argtypes = [I]
    lib.wna16_moe_profile_read.restype = I
    lib.wna16_moe_profile_read.argtypes = [ctypes.POINTER(ctypes.c_float), I]
    lib.wna16_moe_forward_partial.restype = I
    lib.wna16_moe_forward_partial.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64, I64, I64, I, I, I, I, F, P,
                                              P, SZ, P]
    lib.wna16_moe_quantize.restype = I
    lib.wna16_moe_quantize.argtypes = [P, I64, I64, P, I, I, I, P, P, P, P]
    lib.wna16_moe_route_topk.restype = I
    lib.wna16_moe_route_topk.argtypes = [P, P, I64, I64, I, P, P, P]
    lib.wna16_moe_combine.restype = I
    lib.wna16_moe_combine.argtypes = [P, P, I64, I64, I, I64, I64, I, P, P, SZ, P]
    return lib


def _check(rc: int):
    if rc != OK:
        raise Wna16Error(rc, load_library().wna16_moe_last_error().decode())


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str, ndim: int | None = None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def workspace_size(T: int, K: int, N: int, E: int, topk: int, bits: int) -> int:
    return int(load_library().wna16_moe_workspace_size(T, K, N, E, topk, bits))


def alloc_workspace(T: int, K: int, N: int, E: int, topk: int, bits: int, device="cuda") -> torch.Tensor:
    n = workspace_size(T, K, N, E, topk, bits)
    if n == 0:
        raise Wna16Error(ERR_UNSUPPORTED, "unsupported sizes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def pack(codes: torch.Tensor, bits: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """int8 codes [..., K] -> int32 words [..., K*bits/32]."""
    _need(codes, torch.int8, "codes")
    K = codes.shape[-1]
    rows = codes.numel() // K if K else 0
    if out is None:
        out = torch.empty(*codes.shape[:-1], K * bits // 32, dtype=torch.int32, device=codes.device)
    _need(out, torch.int32, "out")
    _check(load_library().wna16_moe_pack(_ptr(codes), rows, K, bits, _ptr(out), _stream(stream)))
    return out


def _dims(x, ids, w13_packed, w2_packed, bits):
    T, K = x.shape
    topk = ids.shape[1]
    E = w13_packed.shape[0]
    N = w13_packed.shape[1] // 2
    if ids.shape[0] != T:
        raise ValueError("topk_ids must be [T, topk]")
    p = 32 // bits
    if tuple(w13_packed.shape) != (E, 2 * N, K // p):
        raise ValueError(f"w13_packed must be [E, 2N, K/p] = {(E, 2 * N, K // p)}, got {tuple(w13_packed.shape)}")
    if w2_packed is not None and tuple(w2_packed.shape) != (E, K, N // p):
        raise ValueError(f"w2_packed must be [E, K, N/p] = {(E, K, N // p)}, got {tuple(w2_packed.shape)}")
    return T, K, N, E, topk


def forward(x, topk_ids, topk_weights, w13_packed, w13_scales, w2_packed, w2_scales, *, bits: int,
            group_size: int, group_size_w2: int = 0, swiglu_limit: float = 7.0, out=None, workspace=None,
            stream=None) -> torch.Tensor:
    """The routed-expert WNA16 MoE forward; returns out bf16 [T, K]."""
    _need(x, torch.bfloat16, "x", 2)
    _need(topk_ids, torch.int32, "topk_ids", 2)
    _need(topk_weights, torch.float32, "topk_weights", 2)
    _need(w13_packed, torch.int32, "w13_packed", 3)
    _need(w2_packed, torch.int32, "w2_packed", 3)
    _need(w13_scales, torch.float16, "w13_scales", 3)
    _need(w2_scales, torch.float16, "w2_scales", 3)
    T, K, N, E, topk = _dims(x, topk_ids, w13_packed, w2_packed, bits)
    if out is None:
        out = torch.empty(T, K, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out", 2)
    if workspace is None:
        workspace = alloc_workspace(T, K, N, E, topk, bits, x.device)
    rc = load_library().wna16_moe_forward(
        _ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(w13_packed), _ptr(w13_scales), _ptr(w2_packed),
        _ptr(w2_scales), T, K, N, E, topk, group_size, group_size_w2, bits, float(swiglu_limit), _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc)
    return out


def forward_partial(x, topk_ids, topk_weights, w13_local, w13_scales_local, w2_local, w2_scales_local, *,
                    expert_begin: int, E_total: int, bits: int, group_size: int, group_size_w2: int = 0,
                    swiglu_limit: float = 7.0, out=None, workspace=None, stream=None) -> torch.Tensor:
    """Expert-parallel partial forward over the local experts [expert_begin,
    expert_begin + E_local) (the weight tensors hold those experts only);
    returns the fp32 partial output [T, K] (unrounded, to be summed across
    ranks in rank order and then rounded to BF16)."""
    _need(x, torch.bfloat16, "x", 2)
    _need(topk_ids, torch.int32, "topk_ids", 2)
    _need(topk_weights, torch.float32, "topk_weights", 2)
    _need(w13_local, torch.int32, "w13_local", 3)
    _need(w2_local, torch.int32, "w2_local", 3)
    _need(w13_scales_local, torch.float16, "w13_scales_local", 3)
    _need(w2_scales_local, torch.float16, "w2_scales_local", 3)
    T, K = x.shape
    topk = topk_ids.shape[1]
    E_local = w13_local.shape[0]
    N = w13_local.shape[1] // 2
    p = 32 // bits
    if tuple(w13_local.shape) != (E_local, 2 * N, K // p) or tuple(w2_local.shape) != (E_local, K, N // p):
        raise ValueError("local weight shapes must be [E_local, 2N, K/p] and [E_local, K, N/p]")
    if out is None:
        out = torch.empty(T, K, dtype=torch.float32, device=x.device)
    _need(out, torch.float32, "out", 2)
    if workspace is None:
        workspace = alloc_workspace(T, K, N, E_local, topk, bits, x.device)
    _check(load_library().wna16_moe_forward_partial(
        _ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(w13_local), _ptr(w13_scales_local), _ptr(w2_local),
        _ptr(w2_scales_local), T, K, N, E_total, expert_begin, E_local, topk, group_size, group_size_w2, bits,
        float(swiglu_limit), _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def forward_noalloc(x, topk_ids, topk_weights, w13_packed, w13_scales, w2_packed, w2_scales, *, bits: int,
                    group_size: int, group_size_w2: int = 0, swiglu_limit: float = 7.0, out=None,
                    stream=None) -> torch.Tensor:
    """The forward with the library's static scratch instead of a workspace
    (for callers that cannot allocate device memory while running); same
    results as forward().  Calls that overlap on the GPU race on that scratch."""
    _need(x, torch.bfloat16, "x", 2)
    _need(topk_ids, torch.int32, "topk_ids", 2)
    _need(topk_weights, torch.float32, "topk_weights", 2)
    _need(w13_packed, torch.int32, "w13_packed", 3)
    _need(w2_packed, torch.int32, "w2_packed", 3)
    _need(w13_scales, torch.float16, "w13_scales", 3)
    _need(w2_scales, torch.float16, "w2_scales", 3)
    T, K, N, E, topk = _dims(x, topk_ids, w13_packed, w2_packed, bits)
    if out is None:
        out = torch.empty(T, K, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out", 2)
    _check(load_library().wna16_moe_forward_noalloc(
        _ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(w13_packed), _ptr(w13_scales), _ptr(w2_packed),
        _ptr(w2_scales), T, K, N, E, topk, group_size, group_size_w2, bits, float(swiglu_limit), _ptr(out),
        _stream(stream)))
    return out


def route_topk(logits, topk: int, bias=None, ids=None, weights=None, stream=None):
    """Router: (topk_ids int32 [T, topk], topk_weights fp32 [T, topk]) from
    fp32 logits [T, E] (+ bias [E]): softmax, top-k (ties to the lower
    index), renormalised."""
    _need(logits, torch.float32, "logits", 2)
    T, E = logits.shape
    if bias is not None:
        _need(bias, torch.float32, "bias", 1)
    if ids is None:
        ids = torch.empty(T, topk, dtype=torch.int32, device=logits.device)
    if weights is None:
        weights = torch.empty(T, topk, dtype=torch.float32, device=logits.device)
    _need(ids, torch.int32, "ids", 2)
    _need(weights, torch.float32, "weights", 2)
    _check(load_library().wna16_moe_route_topk(_ptr(logits), _ptr(bias), T, E, topk, _ptr(ids), _ptr(weights),
                                               _stream(stream)))
    return ids, weights


def quantize(w, bits: int, group_size: int = 128, importance=None, search: bool = True, metrics: bool = True,
             stream=None):
    """Symmetric RTN with an importance-weighted scale search: fp32 w
    [rows, K] (+ importance [K]) -> (packed int32 [rows, K*bits/32], scales
    fp16 [rows, K/group_size], metrics fp64 [rows, 4] or None)."""
    _need(w, torch.float32, "w", 2)
    rows, K = w.shape
    if importance is not None:
        _need(importance, torch.float32, "importance", 1)
    packed = torch.empty(rows, K * bits // 32, dtype=torch.int32, device=w.device)
    scales = torch.empty(rows, K // group_size, dtype=torch.float16, device=w.device)
    met = torch.empty(rows, 4, dtype=torch.float64, device=w.device) if metrics else None
    _check(load_library().wna16_moe_quantize(_ptr(w), rows, K, _ptr(importance), bits, group_size,
                                             1 if search else 0, _ptr(packed), _ptr(scales), _ptr(met),
                                             _stream(stream)))
    return packed, scales, met


STAGES = ("route", "gather", "w13", "w2", "combine")


def profile(slots: int) -> None:
    """Record per-stage CUDA events in the next forwards on this thread (ring of
    `slots` forwards; 0 turns it off)."""
    _check(load_library().wna16_moe_profile(int(slots)))


def profile_read(n: int = 1) -> list[dict]:
    """Stage durations (ms) of the last n profiled forwards, oldest first (waits for them)."""
    ms = (ctypes.c_float * (5 * n))()
    _check(load_library().wna16_moe_profile_read(ms, n))
    return [dict(zip(STAGES, [float(ms[5 * i + j]) for j in range(5)])) for i in range(n)]


def check_wait_timeout(workspace: torch.Tensor, limit_us: int, stream=None) -> None:
    """Run one bounded device wait that nothing completes; it leaves
    ERR_DEVICE_TIMEOUT in the workspace status word (see read_status)."""
    _check(load_library().wna16_moe_check_wait_timeout(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                                       int(limit_us), _stream(stream)))


def launches_last_forward() -> int:
    """Kernels the last forward on this thread launched."""
    return int(load_library().wna16_moe_launches_last_forward())


def read_status(workspace: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int(0)
    _check(load_library().wna16_moe_read_status(_ptr(workspace), ctypes.byref(v), _stream(stream)))
    return v.value


def route(topk_ids, E: int, K: int, N: int, bits: int, workspace=None, stream=None):
    """Routing lists (counts [E], offsets [E+1], perm [R], inv [R]) as int32 CUDA tensors."""
    _need(topk_ids, torch.int32, "topk_ids", 2)
    T, topk = topk_ids.shape
    R = T * topk
    dev = topk_ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(max(R, 1), dtype=torch.int32, device=dev)[:R]
    inv = torch.empty(max(R, 1), dtype=torch.int32, device=dev)[:R]
    if workspace is None:
        workspace = alloc_workspace(T, K, N, E, topk, bits, dev)
    _check(load_library().wna16_moe_route(_ptr(topk_ids), T, topk, E, K, N, bits, _ptr(counts), _ptr(offsets),
                                          _ptr(perm), _ptr(inv), _ptr(workspace), workspace.numel(),
                                          _stream(stream)))
    return counts, offsets, perm, inv


def w13(x, topk_ids, w13_packed, w13_scales, *, bits: int, group_size: int, swiglu_limit: float = 7.0,
        workspace=None, stream=None) -> torch.Tensor:
    """h bf16 [R, N] in permuted order (route + gather + w13 GEMM + SwiGLU)."""
    _need(x, torch.bfloat16, "x", 2)
    _need(topk_ids, torch.int32, "topk_ids", 2)
    _need(w13_packed, torch.int32, "w13_packed", 3)
    _need(w13_scales, torch.float16, "w13_scales", 3)
    T, K, N, E, topk = _dims(x, topk_ids, w13_packed, None, bits)
    h = torch.empty(T * topk, N, dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = alloc_workspace(T, K, N, E, topk, bits, x.device)
    _check(load_library().wna16_moe_w13(_ptr(x), _ptr(topk_ids), _ptr(w13_packed), _ptr(w13_scales), T, K, N, E,
                                        topk, group_size, bits, float(swiglu_limit), _ptr(h), _ptr(workspace),
                                        workspace.numel(), _stream(stream)))
    return h


def w2(h, w2_packed, w2_scales, *, T: int, topk: int, bits: int, group_size_w2: int, workspace,
       stream=None) -> torch.Tensor:
    """y bf16 [R, K] = W2 h for permuted rows (routing lists must be in `workspace`)."""
    _need(h, torch.bfloat16, "h", 2)
    _need(w2_packed, torch.int32, "w2_packed", 3)
    _need(w2_scales, torch.float16, "w2_scales", 3)
    E, K, _ = w2_packed.shape
    N = h.shape[1]
    y = torch.empty(T * topk, K, dtype=torch.bfloat16, device=h.device)
    _check(load_library().wna16_moe_w2(_ptr(h), _ptr(w2_packed), _ptr(w2_scales), T, K, N, E, topk, group_size_w2,
                                       bits, _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream)))
    return y


def combine(y, topk_weights, *, E: int, N: int, bits: int, workspace, stream=None) -> torch.Tensor:
    """out bf16 [T, K] from y [R, K] in permuted order (inverse map in `workspace`)."""
    _need(y, torch.bfloat16, "y", 2)
    _need(topk_weights, torch.float32, "topk_weights", 2)
    T, topk = topk_weights.shape
    K = y.shape[1]
    out = torch.empty(T, K, dtype=torch.bfloat16, device=y.device)
    _check(load_library().wna16_moe_combine(_ptr(y), _ptr(topk_weights), T, K, topk, E, N, bits, _ptr(out),
                                            _ptr(workspace), workspace.numel(), _stream(stream)))
    return out
