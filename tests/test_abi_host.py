"""The C ABI on the host: the library loads, exports every entry point that
include/moe_route.h declares, and rejects bad arguments with status codes
before touching CUDA (so these run on a machine without a GPU; no compute is
launched, every pointer below is a fake address that is never dereferenced).
"""
import ctypes
import os
import re

import pytest
import torch

import combine_moe_route_02_gb300 as moe

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_route.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA = 0, 1, 2, 3, 4, 5

A = 0x10000   # a 16-byte aligned fake device address
A2 = 0x20000
A3 = 0x30000
A4 = 0x40000


@pytest.fixture(scope="module")
def L():
    moe.build()
    return moe.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("moe_route", "moe_dispatch", "moe_combine", "moe_dispatch_workspace_size",
              "moe_status_string"):
        assert s in syms
    assert set(syms) == set(moe.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    for s in declared_symbols():
        assert hasattr(L, s), s
    assert L.moe_abi_version() == moe.ABI_VERSION


def test_status_strings(L):
    for code in range(8):
        s = moe.status_string(code)
        assert s.startswith("MOE_")
    assert "unknown" in moe.status_string(99)


def route(L, X=A, W=A2, bias=None, N=16, H=64, E=16, K=2, idx=A3, w=A4, algo=0):
    return L.moe_route_ex(X, W, bias, N, H, E, K, 1, idx, w, None, algo, None)


def test_route_validation(L):
    assert route(L, N=0) == OK                     # no tokens: nothing to do
    assert route(L, E=0) == INVALID
    assert route(L, E=257) == INVALID
    assert route(L, K=0) == INVALID
    assert route(L, K=17, E=32) == INVALID
    assert route(L, K=5, E=4) == INVALID
    assert route(L, N=-1) == INVALID
    assert route(L, X=None) == INVALID
    assert route(L, idx=None) == INVALID
    assert route(L, H=0) == INVALID
    assert route(L, H=12) == MISALIGNED
    assert route(L, X=A + 8) == MISALIGNED
    assert route(L, W=A2 + 2) == MISALIGNED
    assert route(L, algo=7) == INVALID
    assert route(L, N=2**31, K=1) == INVALID       # N*K must stay below 2^31


def dispatch(L, idx=A, X=None, N=16, H=64, E=16, K=2, counts=A2, offsets=A3, row_map=A4,
             src=None, xp=None, xq=None, xs=None, ws=None, ws_bytes=0):
    return L.moe_dispatch(idx, X, N, H, E, K, counts, offsets, row_map, src, xp, xq, xs, None,
                          ws, ws_bytes, None)


def test_dispatch_validation(L):
    assert L.moe_dispatch_workspace_size(1 << 20, 64, 8) >= 256 + 64 * 4
    ws = L.moe_dispatch_workspace_size(16, 16, 2)
    assert dispatch(L, ws=A, ws_bytes=ws - 4) == WORKSPACE                 # too small
    assert dispatch(L, ws=None, ws_bytes=ws) == WORKSPACE                  # size without a buffer
    assert dispatch(L, ws=A + 16, ws_bytes=ws) == MISALIGNED               # 256-byte alignment
    assert dispatch(L, E=0) == INVALID
    assert dispatch(L, K=0) == INVALID
    assert dispatch(L, counts=None) == INVALID
    assert dispatch(L, idx=None) == INVALID
    assert dispatch(L, row_map=None) == INVALID
    assert dispatch(L, xp=A) == INVALID                           # output rows without X
    assert dispatch(L, X=A, xp=None) == INVALID                   # X without any output
    assert dispatch(L, X=A, xp=A2 + 4) == MISALIGNED
    assert dispatch(L, X=A, H=12, xp=A) == MISALIGNED
    assert dispatch(L, X=A, H=192, xq=A, xs=None) == INVALID      # fp8 codes need scales
    assert dispatch(L, X=A, H=192, xq=A, xs=A2) == INVALID        # H % 128 != 0
    assert dispatch(L, idx=A + 2) == MISALIGNED
    assert dispatch(L, N=-5) == INVALID


def test_permute_and_combine_validation(L):
    assert L.moe_permute(A, A2, 0, 64, 2, A3, None, None, None, None) == OK
    assert L.moe_permute(None, A2, 8, 64, 2, A3, None, None, None, None) == INVALID
    assert L.moe_permute(A, A2, 8, 64, 2, None, None, None, None, None) == INVALID
    assert L.moe_permute(A, A2, 8, 64, 0, A3, None, None, None, None) == INVALID
    assert L.moe_permute(A, A2, 8, 64, 2, A3 + 8, None, None, None, None) == MISALIGNED
    assert L.moe_combine(A, A2, A3, 0, 64, 2, A4, None, None) == OK
    assert L.moe_combine(None, A2, A3, 8, 64, 2, A4, None, None) == INVALID
    assert L.moe_combine(A, A2, A3, 8, 64, 17, A4, None, None) == INVALID
    assert L.moe_combine(A, A2, A3, 8, 60, 2, A4, None, None) == MISALIGNED
    assert L.moe_combine(A, A2, A3, 8, 64, 2, A4 + 8, None, None) == MISALIGNED
    # block-scale format: fp32 scales need 4-byte alignment, UE8M0 bytes none; other formats are refused
    assert L.moe_permute_ex(A, A2, 8, 128, 2, A3, A4, A + 2, 0, None, None) == MISALIGNED
    assert L.moe_permute_ex(A, A2, 8, 128, 2, A3, A4, A, 2, None, None) == INVALID
    assert L.moe_permute_ex(A, A2, 0, 128, 2, A3, A4, A, 7, None, None) == INVALID
    assert L.moe_dispatch_ex(A, A2, 8, 128, 16, 2, A3, A4, A, A2, A3, A4, A, 5, None, None, 0, None) == INVALID
    # router statistics: argument checks before any CUDA call
    assert L.moe_route_stats(A, A2, None, 16, 64, 16, 2, 1, A3, A4, A + 2, None, None, 0, None) == MISALIGNED
    assert L.moe_route_stats(A, A2, None, 16, 64, 16, 17, 1, A3, A4, None, None, None, 0, None) == INVALID
    assert L.moe_route_stats(A, A2, None, 16, 64, 16, 2, 1, A3, A4, None, None, None, 9, None) == INVALID
    assert L.moe_load_stats(A, 0, None, 0, ctypes.c_float(1e-3), A2, None) == INVALID
    assert L.moe_load_stats(A, 257, None, 0, ctypes.c_float(1e-3), A2, None) == INVALID
    assert L.moe_load_stats(None, 16, None, 0, ctypes.c_float(1e-3), A2, None) == INVALID
    assert L.moe_load_stats(A, 16, None, 0, ctypes.c_float(1e-3), A2 + 2, None) == MISALIGNED
    # expert-parallel metadata: ep_size must divide E; the workspace is required
    ep = lambda R, ws=0x60000, nb=1 << 20: L.moe_dispatch_ep(A, None, 8, 0, 16, 2, R, A, A2, A3, A4, A, A2, A3, A4,
                                                             A, None, None, ws, nb, None)
    assert ep(0) == INVALID and ep(3) == INVALID and ep(32) == INVALID
    assert ep(4, ws=None, nb=0) == WORKSPACE
    assert ep(4, ws=0x60000 + 16) == MISALIGNED
    R = 0x50000
    assert L.moe_combine_residual(A, A2, A3, R, 0, 64, 2, A4, None, None) == OK
    assert L.moe_combine_residual(A, A2, A3, None, 8, 64, 2, A4, None, None) == INVALID
    assert L.moe_combine_residual(A, A2, A3, R + 8, 8, 64, 2, A4, None, None) == MISALIGNED
    assert L.moe_combine_residual(None, A2, A3, R, 8, 64, 2, A4, None, None) == INVALID
    assert L.moe_combine_residual(A, A2, A3, R, 8, 64, 0, A4, None, None) == INVALID


def route_dispatch(L, X=A, W=A2, N=16, H=64, E=16, K=2, idx=A3, w=A4, counts=A, offsets=A2, row_map=A3,
                   src=None, xp=None, ws=0x100000, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = L.moe_dispatch_workspace_size(N, E, K)
    n = ctypes.c_int(-1)
    code = L.moe_route_dispatch(X, W, None, N, H, E, K, 1, idx, w, counts, offsets, row_map, src, xp, None, ws,
                                ws_bytes, ctypes.byref(n), None)
    assert n.value == 0          # nothing launched on a rejected call
    return code


def test_route_dispatch_validation(L):
    assert route_dispatch(L, E=0) == INVALID
    assert route_dispatch(L, K=17, E=32) == INVALID
    assert route_dispatch(L, N=-1) == INVALID
    assert route_dispatch(L, H=0) == INVALID
    assert route_dispatch(L, counts=None) == INVALID
    assert route_dispatch(L, ws=None) == WORKSPACE
    assert route_dispatch(L, ws_bytes=64) == WORKSPACE
    assert route_dispatch(L, ws=0x100000 + 16) == MISALIGNED
    assert route_dispatch(L, X=None) == INVALID
    assert route_dispatch(L, row_map=None) == INVALID
    assert route_dispatch(L, H=12) == MISALIGNED
    assert route_dispatch(L, X=A + 8) == MISALIGNED
    assert route_dispatch(L, xp=A4 + 4) == MISALIGNED
    assert route_dispatch(L, src=A + 2) == MISALIGNED


def noalloc_fn(L):
    f = L.moe_dispatch_noalloc
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.argtypes = [P, P, I64, I32, I32, I32, P, P, P, P, P, P, P, P, P]
    f.restype = I32
    return f


def noalloc(L, idx=A, X=None, N=16, H=64, E=16, K=2, counts=A2, offsets=A3, row_map=A4,
            src=None, xp=None, xq=None, xs=None, st=None):
    return noalloc_fn(L)(idx, X, N, H, E, K, counts, offsets, row_map, src, xp, xq, xs, st, None)


def test_noalloc_validation(L):
    # moe_dispatch_noalloc runs moe_dispatch's argument checks before any CUDA
    # call: on this machine (no GPU) any CUDA call would fail with MOE_ERR_CUDA,
    # so each code below also shows that nothing reached CUDA or a stream
    assert noalloc(L, idx=A + 2) == MISALIGNED
    assert noalloc(L, row_map=A4 + 2) == MISALIGNED
    assert noalloc(L, st=A + 2) == MISALIGNED
    assert noalloc(L, X=A, xp=A2 + 4) == MISALIGNED
    assert noalloc(L, X=A + 8, xp=A2) == MISALIGNED
    assert noalloc(L, X=A, H=12, xp=A) == MISALIGNED
    assert noalloc(L, X=A, H=128, xq=A, xs=A2 + 2) == MISALIGNED   # fp32 scales need 4-byte alignment
    assert noalloc(L, E=0) == INVALID
    assert noalloc(L, K=17, E=32) == INVALID
    assert noalloc(L, N=-1) == INVALID
    assert noalloc(L, counts=None) == INVALID
    assert noalloc(L, idx=None) == INVALID
    assert noalloc(L, xp=A) == INVALID                           # output rows without X
    assert noalloc(L, X=A, H=192, xq=A, xs=A2) == INVALID        # H % 128 != 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_call_without_gpu_fails_loudly(L):
    # arguments pass validation, then the first CUDA call fails: MOE_ERR_CUDA, no crash
    assert route(L) == CUDA
    assert L.moe_combine(A, A2, A3, 8, 64, 2, A4, None, None) == CUDA
    assert L.moe_combine_residual(A, A2, A3, 0x50000, 8, 64, 2, A4, None, None) == CUDA
    assert L.moe_load_stats(A, 16, None, 0, ctypes.c_float(1e-3), A2, None) == CUDA
    assert L.moe_route_dispatch(A, A2, None, 16, 64, 16, 2, 1, A3, A4, A, A2, A3, None, None, None, 0x100000,
                                L.moe_dispatch_workspace_size(16, 16, 2), None, None) == CUDA
    # UE8M0 scale bytes need no alignment: the call passes validation (then fails on CUDA)
    assert L.moe_permute_ex(A, A2, 8, 128, 2, A3, A4, A + 2, 1, None, None) == CUDA
    # a valid no-allocation dispatch reaches its first CUDA call only after the checks
    assert noalloc(L) == CUDA


def test_binding_refuses_cpu_tensors():
    X = torch.zeros(4, 64, dtype=torch.bfloat16)
    W = torch.zeros(64, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        moe.route(X, W, 2)


def test_binding_checks_status_word_and_workspace():
    # the status word and the workspace reach the kernels as raw pointers: a host
    # tensor is refused before the library is called, and a workspace's size is
    # its byte count whatever its dtype
    assert moe._status_ptr(None) is None
    with pytest.raises(ValueError, match="CUDA"):
        moe._status_ptr(torch.zeros(1, dtype=torch.int32))
    assert moe._workspace_arg(None) == (None, 0)
    with pytest.raises(ValueError, match="CUDA"):
        moe._workspace_arg(torch.zeros(64, dtype=torch.int32))


def test_binding_status_word_pointer(monkeypatch):
    # with the device checks stubbed out (no GPU here), an accepted status word
    # is passed as its own data pointer
    monkeypatch.setattr(moe, "_need", lambda t, name, dtype, shape=None: t)
    st = torch.zeros(1, dtype=torch.int32)
    assert moe._status_ptr(st).value == st.data_ptr()
    with pytest.raises(ValueError, match="at least one"):
        moe._status_ptr(torch.zeros(0, dtype=torch.int32))


def test_product_does_not_import_oracle():
    # the product path (package + CUDA sources) never imports, links or loads the oracle
    here = os.path.dirname(moe.__file__)
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#include\s+.*oracle)|_oracle\.so", re.M)
    for root, _, files in os.walk(here):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f), errors="ignore").read()
                assert not pat.search(text), f
