"""C ABI checks that need no GPU: the library builds, loads, exports every
symbol the header declares, and rejects bad arguments on the host before any
CUDA call (so these run on a machine without a GPU)."""
from __future__ import annotations

import ctypes
import math

import pytest

from wna16_grouped_gemm_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = binding.exported_names_in_header()
    assert len(names) == 17, names
    for n in names:
        assert hasattr(lib, n), n


def test_kernels_are_built_for_sm103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)


# fake device pointers: never dereferenced, because validation fails first
A16 = ctypes.c_void_p(0x10000)
A8 = ctypes.c_void_p(0x10008)


def _fwd(lib, *, x=A16, out=ctypes.c_void_p(0x90000), T=4, K=4096, N=2048, E=256, topk=8, g=128, g2=0, bits=2,
         limit=7.0, ws=ctypes.c_void_p(0x100000), ws_bytes=1 << 40, ids=A16, w=A16, w13=A16, w2=A16):
    return lib.wna16_moe_forward(x, ids, w, w13, A16, w2, A16, T, K, N, E, topk, g, g2, bits, limit, out, ws,
                                 ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bits=3), binding.ERR_UNSUPPORTED),
    (dict(bits=8), binding.ERR_UNSUPPORTED),
    (dict(K=100), binding.ERR_UNSUPPORTED),
    (dict(N=96), binding.ERR_UNSUPPORTED),
    (dict(g=16), binding.ERR_UNSUPPORTED),
    (dict(g=96), binding.ERR_UNSUPPORTED),
    (dict(g=48), binding.ERR_UNSUPPORTED),
    (dict(g2=192), binding.ERR_UNSUPPORTED),
    (dict(topk=9, E=8), binding.ERR_INVALID_ARG),
    (dict(E=2048), binding.ERR_UNSUPPORTED),
    (dict(T=-1), binding.ERR_INVALID_ARG),
    (dict(limit=0.0), binding.ERR_INVALID_ARG),
    (dict(limit=-1.0), binding.ERR_INVALID_ARG),
    (dict(limit=math.nan), binding.ERR_INVALID_ARG),
    (dict(x=None), binding.ERR_INVALID_ARG),
    (dict(x=A8), binding.ERR_INVALID_ARG),
    (dict(ids=None), binding.ERR_INVALID_ARG),
    (dict(w13=A8), binding.ERR_INVALID_ARG),
    (dict(out=ctypes.c_void_p(0x10000 + 4096)), binding.ERR_INVALID_ARG),   # overlaps x
    (dict(ws=None), binding.ERR_INVALID_ARG),
    (dict(ws=ctypes.c_void_p(0x100010)), binding.ERR_INVALID_ARG),          # not 256-aligned
    (dict(ws_bytes=1024), binding.ERR_WORKSPACE_TOO_SMALL),
])
def test_forward_rejects_on_host(lib, kw, code):
    assert _fwd(lib, **kw) == code
    assert lib.wna16_moe_last_error().decode() != ""


def test_empty_batch_is_a_no_op(lib):
    assert _fwd(lib, T=0, x=None, out=None, ws=None, ids=None) == binding.OK


def test_workspace_size(lib):
    assert lib.wna16_moe_workspace_size(4, 4096, 2048, 256, 8, 2) > 0
    assert lib.wna16_moe_workspace_size(4, 4096, 2048, 256, 8, 3) == 0
    assert lib.wna16_moe_workspace_size(4, 100, 2048, 256, 8, 2) == 0
    big = lib.wna16_moe_workspace_size(8192, 4096, 2048, 256, 8, 4)
    # permuted x, h and y dominate: R*(K + N + K)*2 bytes
    R = 8192 * 8
    assert big >= R * (4096 + 2048 + 4096) * 2


def test_workspace_holds_split_k_partials_and_corrections(lib):
    """Decode W2 (T=4, top-8 over 256 experts): 16-token tiles, at most
    min(R, E) + R/16 + 1 = 35 tiles, so 560 units per GEMM, split 4 ways; the
    partial sums take splits x row tiles x R x 256 fp32 (2 MiB for either
    GEMM) and the offset-code corrections R x (K + N) / 128 fp32, on top of
    the permuted x, h and y."""
    T, K, N, E, topk = 4, 4096, 2048, 256, 8
    R = T * topk
    partial = 4 * (N // 128) * R * 256 * 4
    assert partial == 4 * (K // 256) * R * 256 * 4 == 2 << 20
    corrections = R * (K + N) // 128 * 4
    need = R * (K + N + K) * 2 + partial + corrections
    assert lib.wna16_moe_workspace_size(T, K, N, E, topk, 2) >= need


def test_pack_rejects_on_host(lib):
    assert lib.wna16_moe_pack(A16, 4, 64, 3, A16, None) == binding.ERR_UNSUPPORTED
    assert lib.wna16_moe_pack(A16, 4, 60, 2, A16, None) == binding.ERR_INVALID_ARG
    assert lib.wna16_moe_pack(None, 4, 64, 2, A16, None) == binding.ERR_INVALID_ARG
    assert lib.wna16_moe_pack(A16, 0, 64, 2, A16, None) == binding.OK


def test_stage_entry_points_reject_on_host(lib):
    assert lib.wna16_moe_route(A16, 4, 8, 256, 4096, 2048, 3, None, None, None, None, A16, 1 << 40,
                               None) == binding.ERR_UNSUPPORTED
    assert lib.wna16_moe_w13(A16, A16, A16, A16, 4, 4096, 2048, 256, 8, 16, 2, 7.0, A16, A16, 1 << 40,
                             None) == binding.ERR_UNSUPPORTED
    assert lib.wna16_moe_w2(A16, A16, A16, 4, 4096, 2048, 256, 8, 128, 2, A16, A16, 16, None) == \
        binding.ERR_WORKSPACE_TOO_SMALL
    assert lib.wna16_moe_combine(A16, A16, 4, 4096, 8, 256, 2048, 2, A16, None, 1 << 40, None) == \
        binding.ERR_INVALID_ARG


def test_wait_timeout_check_rejects_on_host(lib):
    assert lib.wna16_moe_check_wait_timeout(None, 16, 1000, None) == binding.ERR_INVALID_ARG
    assert lib.wna16_moe_check_wait_timeout(A16, 2, 1000, None) == binding.ERR_INVALID_ARG
    assert lib.wna16_moe_check_wait_timeout(A16, 16, 0, None) == binding.ERR_INVALID_ARG
    assert lib.wna16_moe_check_wait_timeout(A16, 16, 10_000_000, None) == binding.ERR_INVALID_ARG


def test_profile_read_without_forward_is_an_error(lib):
    assert lib.wna16_moe_profile_read(None, 1) == binding.ERR_INVALID_ARG
    assert lib.wna16_moe_profile(-1) == binding.ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    saved = binding._lib
    try:
        binding._lib = None
        with pytest.raises(RuntimeError, match="missing"):
            binding.load_library(str(tmp_path / "nope.so"))
    finally:
        binding._lib = saved


def test_partial_forward_rejects_on_host(lib):
    P = ctypes.c_void_p
    f = lib.wna16_moe_forward_partial

    def call(E_total=256, begin=0, E_local=128, topk=8, out=P(0x90000)):
        return f(A16, A16, A16, A16, A16, A16, A16, 4, 4096, 2048, E_total, begin, E_local, topk, 128, 0, 2,
                 ctypes.c_float(7.0), out, P(0x100000), 1 << 40, None)
    assert call(begin=200) == binding.ERR_INVALID_ARG          # range past E_total
    assert call(begin=-1) == binding.ERR_INVALID_ARG
    assert call(E_local=300) == binding.ERR_INVALID_ARG         # more local experts than exist
    assert call(topk=300) == binding.ERR_INVALID_ARG            # topk > E_total
    assert call(out=None) == binding.ERR_INVALID_ARG
    assert call(out=P(0x10000 + 4096)) == binding.ERR_INVALID_ARG   # fp32 out overlaps x


def test_router_rejects_on_host(lib):
    P = ctypes.c_void_p
    f = lib.wna16_moe_route_topk
    assert f(A16, None, 4, 256, 33, A16, A16, None) == binding.ERR_INVALID_ARG     # topk > 32
    assert f(A16, None, 4, 8, 9, A16, A16, None) == binding.ERR_INVALID_ARG       # topk > E
    assert f(A16, None, 4, 2048, 8, A16, A16, None) == binding.ERR_UNSUPPORTED    # E > 1024
    assert f(None, None, 4, 256, 8, A16, A16, None) == binding.ERR_INVALID_ARG
    assert f(A16, P(0x10002), 4, 256, 8, A16, A16, None) == binding.ERR_INVALID_ARG  # misaligned bias
    assert f(None, None, 0, 256, 8, None, None, None) == binding.OK


def test_quantize_rejects_on_host(lib):
    P = ctypes.c_void_p
    f = lib.wna16_moe_quantize
    assert f(A16, 4, 4096, None, 3, 128, 1, A16, A16, None, None) == binding.ERR_UNSUPPORTED      # bits
    assert f(A16, 4, 4096, None, 2, 48, 1, A16, A16, None, None) == binding.ERR_UNSUPPORTED       # group
    assert f(A16, 4, 4096, None, 2, 16, 1, A16, A16, None, None) == binding.ERR_UNSUPPORTED       # 256 groups
    assert f(A8, 4, 4096, None, 2, 128, 1, A16, A16, None, None) == binding.ERR_INVALID_ARG       # w alignment
    assert f(A16, 4, 4096, None, 2, 128, 2, A16, A16, None, None) == binding.ERR_INVALID_ARG      # search flag
    assert f(A16, 4, 4096, P(0x10004), 2, 128, 1, A16, A16, None, None) == binding.ERR_INVALID_ARG
    assert f(None, 0, 4096, None, 2, 128, 1, None, None, None, None) == binding.OK


def test_debug_library_exports_the_same_symbols():
    """The bounds-checked build is the same library with index checks on."""
    build.build(debug=True)
    dbg = binding.load_debug_library()
    for n in binding.exported_names_in_header():
        assert hasattr(dbg, n), n
