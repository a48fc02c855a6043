"""GB300 (sm_103a) MoE routing hot path: route -> dispatch -> permute -> combine.

A thin ctypes binding over the C ABI of ``libmoe_route_gb300.so`` (declared in
``include/moe_route.h``).  This module only marshals arguments: it checks
dtypes, devices and contiguity, allocates outputs with torch when the caller
does not pass them, and hands raw device pointers plus the current CUDA stream
to the library.  Every step of the path runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback -- if the library is missing the calls
raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

from . import _build

__all__ = [
    "build", "lib", "MoeError", "route", "route_stats", "load_stats", "dispatch", "dispatch_ep", "permute",
    "combine", "dispatch_workspace_size", "dispatch_workspace", "status_string", "ROUTE_AUTO", "ROUTE_TCGEN05",
    "ROUTE_SIMT", "SCALE_FP32", "SCALE_UE8M0", "Dispatch", "DispatchEP", "route_dispatch",
]

MOE_OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_MISALIGNED = 3
ERR_WORKSPACE = 4
ERR_CUDA = 5
ERR_TIMEOUT = 6
ERR_BAD_INDEX = 7

ROUTE_AUTO = 0
ROUTE_TCGEN05 = 1
ROUTE_SIMT = 2
_ALGOS = {"auto": ROUTE_AUTO, "tcgen05": ROUTE_TCGEN05, "simt": ROUTE_SIMT}

ABI_VERSION = 1
EXPORTED_SYMBOLS = (
    "moe_route", "moe_route_ex", "moe_dispatch_workspace_size", "moe_dispatch",
    "moe_permute", "moe_combine", "moe_status_string", "moe_abi_version", "moe_dispatch_noalloc",
    "moe_combine_residual", "moe_dispatch_ex", "moe_permute_ex", "moe_route_stats", "moe_load_stats",
    "moe_dispatch_ep", "moe_route_dispatch",
)

SCALE_FP32, SCALE_UE8M0 = 0, 1
_SCALE_FORMATS = {"fp32": SCALE_FP32, "ue8m0": SCALE_UE8M0}


def _scale_format(name: str) -> int:
    if name not in _SCALE_FORMATS:
        raise ValueError(f"scale_format must be one of {sorted(_SCALE_FORMATS)}")
    return _SCALE_FORMATS[name]


def _scale_dtype(name: str):
    return torch.uint8 if name == "ue8m0" else torch.float32

_lib = None


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)}")


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a) and return its path."""
    return _build.build(force=force)


def lib():
    """The loaded shared library (ctypes.CDLL) with argument types set."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB_PATH):
        raise RuntimeError(
            f"CUDA library {_build.LIB_PATH} is not built; run combine_moe_route_02_gb300.build() "
            "(there is no CPU fallback)")
    L = ctypes.CDLL(_build.LIB_PATH)
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    L.moe_route.argtypes = [P, P, P, I64, I32, I32, I32, I32, P, P, P, P]
    L.moe_route.restype = I32
    L.moe_route_ex.argtypes = [P, P, P, I64, I32, I32, I32, I32, P, P, P, I32, P]
    L.moe_route_ex.restype = I32
    L.moe_dispatch_workspace_size.argtypes = [I64, I32, I32]
    L.moe_dispatch_workspace_size.restype = SZ
    L.moe_dispatch.argtypes = [P, P, I64, I32, I32, I32, P, P, P, P, P, P, P, P, P, SZ, P]
    L.moe_dispatch.restype = I32
    L.moe_permute.argtypes = [P, P, I64, I32, I32, P, P, P, P, P]
    L.moe_permute.restype = I32
    L.moe_combine.argtypes = [P, P, P, I64, I32, I32, P, P, P]
    L.moe_combine.restype = I32
    L.moe_combine_residual.argtypes = [P, P, P, P, I64, I32, I32, P, P, P]
    L.moe_combine_residual.restype = I32
    L.moe_route_stats.argtypes = [P, P, P, I64, I32, I32, I32, I32, P, P, P, P, P, I32, P]
    L.moe_route_stats.restype = I32
    L.moe_load_stats.argtypes = [P, I32, P, I64, ctypes.c_float, P, P]
    L.moe_load_stats.restype = I32
    L.moe_dispatch_ep.argtypes = [P, P, I64, I32, I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]
    L.moe_dispatch_ep.restype = I32
    L.moe_dispatch_ex.argtypes = [P, P, I64, I32, I32, I32, P, P, P, P, P, P, P, I32, P, P, SZ, P]
    L.moe_dispatch_ex.restype = I32
    L.moe_permute_ex.argtypes = [P, P, I64, I32, I32, P, P, P, I32, P, P]
    L.moe_permute_ex.restype = I32
    L.moe_route_dispatch.argtypes = [P, P, P, I64, I32, I32, I32, I32, P, P, P, P, P, P, P, P, P, SZ,
                                     ctypes.POINTER(ctypes.c_int), P]
    L.moe_route_dispatch.restype = I32
    L.moe_status_string.argtypes = [I32]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_abi_version.argtypes = []
    L.moe_abi_version.restype = I32
    if L.moe_abi_version() != ABI_VERSION:
        raise RuntimeError("libmoe_route_gb300.so ABI version mismatch; rebuild it")
    _lib = L
    return L


def status_string(code: int) -> str:
    try:
        return lib().moe_status_string(int(code)).decode()
    except RuntimeError:
        return f"moe_status {code}"


def _check(code: int, where: str):
    if code != MOE_OK:
        raise MoeError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _status_ptr(status: Optional[torch.Tensor]):
    """The device status word (one int32 on the current device), or None."""
    if status is None:
        return None
    _need(status, "status", torch.int32)
    if status.numel() < 1:
        raise ValueError("status must hold at least one int32")
    return _ptr(status)


def _workspace_arg(ws: Optional[torch.Tensor]):
    """(pointer, size in bytes) of a workspace tensor of any dtype, or (None, 0)."""
    if ws is None:
        return None, 0
    if not isinstance(ws, torch.Tensor) or not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if ws.device.index != torch.cuda.current_device():
        raise ValueError(f"workspace is on {ws.device}, but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()}")
    return _ptr(ws), ws.numel() * ws.element_size()


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.device.index != torch.cuda.current_device():
        # the library launches on the current device and takes raw pointers
        raise ValueError(f"{name} is on {t.device}, but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()} (select it with torch.cuda.device)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def route(X: torch.Tensor, W_gate: torch.Tensor, K: int, bias: Optional[torch.Tensor] = None,
          renorm: bool = True, algo: str = "auto", topk_idx=None, topk_w=None, status=None,
          stream=None):
    """Fused router: returns (topk_idx int32 [N,K], topk_w fp32 [N,K])."""
    N, H = X.shape
    E = W_gate.shape[1]
    _need(X, "X", torch.bfloat16)
    _need(W_gate, "W_gate", torch.bfloat16, (H, E))
    if bias is not None:
        _need(bias, "bias", torch.float32, (E,))
    if topk_idx is None:
        topk_idx = torch.empty((N, K), dtype=torch.int32, device=X.device)
    if topk_w is None:
        topk_w = torch.empty((N, K), dtype=torch.float32, device=X.device)
    _need(topk_idx, "topk_idx", torch.int32, (N, K))
    _need(topk_w, "topk_w", torch.float32, (N, K))
    code = lib().moe_route_ex(_ptr(X), _ptr(W_gate), _ptr(bias), N, H, E, K, int(bool(renorm)),
                              _ptr(topk_idx), _ptr(topk_w), _status_ptr(status), _ALGOS[algo], _stream(stream))
    _check(code, "moe_route")
    return topk_idx, topk_w


def route_stats(X: torch.Tensor, W_gate: torch.Tensor, K: int, bias: Optional[torch.Tensor] = None,
                renorm: bool = True, algo: str = "auto", want_lse: bool = True, want_counts: bool = True,
                status=None, stream=None):
    """Fused router with its statistics: returns (topk_idx, topk_w, lse fp32 [N] or None,
    expert_counts int32 [E] or None)."""
    N, H = X.shape
    E = W_gate.shape[1]
    _need(X, "X", torch.bfloat16)
    _need(W_gate, "W_gate", torch.bfloat16, (H, E))
    if bias is not None:
        _need(bias, "bias", torch.float32, (E,))
    dev = X.device
    topk_idx = torch.empty((N, K), dtype=torch.int32, device=dev)
    topk_w = torch.empty((N, K), dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev) if want_lse else None
    counts = torch.empty(E, dtype=torch.int32, device=dev) if want_counts else None
    code = lib().moe_route_stats(_ptr(X), _ptr(W_gate), _ptr(bias), N, H, E, K, int(bool(renorm)),
                                 _ptr(topk_idx), _ptr(topk_w), _ptr(lse), _ptr(counts), _status_ptr(status),
                                 _ALGOS[algo], _stream(stream))
    _check(code, "moe_route_stats")
    return topk_idx, topk_w, lse, counts


def load_stats(expert_counts: torch.Tensor, lse: Optional[torch.Tensor] = None, z_coef: float = 1e-3,
               out=None, stream=None) -> torch.Tensor:
    """Expert-load statistics: fp32 [4] = (max/mean, p95/mean, z_loss, mean)."""
    _need(expert_counts, "expert_counts", torch.int32)
    E = expert_counts.shape[0]
    N = 0
    if lse is not None:
        _need(lse, "lse", torch.float32)
        N = lse.shape[0]
    if out is None:
        out = torch.empty(4, dtype=torch.float32, device=expert_counts.device)
    _need(out, "stats", torch.float32, (4,))
    code = lib().moe_load_stats(_ptr(expert_counts), E, _ptr(lse), N, float(z_coef), _ptr(out), _stream(stream))
    _check(code, "moe_load_stats")
    return out


@dataclass
class Dispatch:
    expert_counts: torch.Tensor
    expert_offsets: torch.Tensor
    row_map: torch.Tensor
    src_slot: Optional[torch.Tensor]
    X_perm: Optional[torch.Tensor] = None
    X_fp8: Optional[torch.Tensor] = None
    X_scale: Optional[torch.Tensor] = None


def dispatch_workspace_size(N: int, E: int, K: int) -> int:
    return int(lib().moe_dispatch_workspace_size(N, E, K))


_workspaces = {}


def dispatch_workspace(E: int, device=None, stream=None) -> torch.Tensor:
    """A zeroed workspace for moe_dispatch, cached per (device, stream, E).

    The library keeps grid-barrier counters in it: they must start at zero and
    every completed call leaves them at zero, so one workspace serves any
    number of calls issued on one stream (calls that overlap on the GPU must
    not share a workspace)."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if stream is None:
        stream = torch.cuda.current_stream(device)
    key = (device.index, stream.cuda_stream, E)
    ws = _workspaces.get(key)
    if ws is None:
        # zero-filled on the stream that will use it, so the first call there is
        # ordered after the fill
        with torch.cuda.stream(stream):
            ws = torch.zeros(dispatch_workspace_size(0, E, 1), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def _fresh_workspace(E: int, device, stream) -> torch.Tensor:
    """The cached workspace of (device, stream, E) with its 256-byte grid-barrier
    header cleared on `stream` first.  A completed call leaves the counters at
    zero, but one whose bounded barrier wait ran out (MOE_ERR_TIMEOUT) does not;
    clearing them before every call keeps such a call from corrupting the next."""
    ws = dispatch_workspace(E, device, stream)
    s = torch.cuda.current_stream(ws.device) if stream is None else stream
    with torch.cuda.stream(s):
        ws[:256].zero_()
    return ws


def dispatch(topk_idx: torch.Tensor, E: int, X: Optional[torch.Tensor] = None, fp8: bool = False,
             bf16: bool = True, want_src_slot: bool = True, out: Optional[Dispatch] = None,
             workspace: Optional[torch.Tensor] = None, fused: bool = True, status=None,
             stream=None, scale_format: str = "fp32") -> Dispatch:
    """Counting-sort dispatch (+ optional row permute / E4M3 quantise).

    fused=True (default) passes a workspace (a cached zeroed one unless
    given), which selects the one-launch cooperative kernel (for row copies of
    256 MiB or more: that kernel for the metadata, then the permute kernel);
    fused=False passes no workspace, which selects the single-cluster metadata
    kernel followed by the permute kernel.  scale_format "fp32" (float scales) or "ue8m0" (one
    exponent byte per 1x128 block) selects the E4M3 block-scale output."""
    fmt = _scale_format(scale_format)
    N, K = topk_idx.shape
    _need(topk_idx, "topk_idx", torch.int32)
    dev = topk_idx.device
    H = 0
    if X is not None:
        _need(X, "X", torch.bfloat16)
        if X.shape[0] != N:
            raise ValueError("X and topk_idx disagree on N")
        H = X.shape[1]
    if out is None:
        out = Dispatch(
            expert_counts=torch.empty(E, dtype=torch.int32, device=dev),
            expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
            row_map=torch.empty(N * K, dtype=torch.int32, device=dev),
            src_slot=torch.empty(N * K, dtype=torch.int32, device=dev) if want_src_slot else None,
            X_perm=torch.empty((N * K, H), dtype=torch.bfloat16, device=dev) if (X is not None and bf16) else None,
            X_fp8=torch.empty((N * K, H), dtype=torch.uint8, device=dev) if (X is not None and fp8) else None,
            X_scale=torch.empty((N * K, H // 128), dtype=_scale_dtype(scale_format), device=dev)
            if (X is not None and fp8) else None,
        )
    if not fused:
        workspace = None
    elif workspace is None:
        workspace = _fresh_workspace(E, dev, stream)
    has_x = X is not None
    code = lib().moe_dispatch_ex(
        _ptr(topk_idx), _ptr(X), N, H, E, K, _ptr(out.expert_counts), _ptr(out.expert_offsets),
        _ptr(out.row_map), _ptr(out.src_slot), _ptr(out.X_perm) if has_x else None,
        _ptr(out.X_fp8) if has_x else None, _ptr(out.X_scale) if has_x else None, fmt,
        _status_ptr(status), *_workspace_arg(workspace), _stream(stream))
    _check(code, "moe_dispatch_ex")
    return out


def route_dispatch(X: torch.Tensor, W_gate: torch.Tensor, K: int, bias: Optional[torch.Tensor] = None,
                   renorm: bool = True, permute: bool = True, want_src_slot: bool = True, topk_idx=None,
                   topk_w=None, out: Optional[Dispatch] = None, workspace: Optional[torch.Tensor] = None,
                   status=None, stream=None):
    """Router, then the counting-sort dispatch of its ids with a bf16 row copy
    (moe_route_dispatch): one launch where the router runs split-K, else the two
    calls.  Returns (topk_idx, topk_w, Dispatch, kernels launched)."""
    N, H = X.shape
    E = W_gate.shape[1]
    _need(X, "X", torch.bfloat16)
    _need(W_gate, "W_gate", torch.bfloat16, (H, E))
    if bias is not None:
        _need(bias, "bias", torch.float32, (E,))
    dev = X.device
    if topk_idx is None:
        topk_idx = torch.empty((N, K), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((N, K), dtype=torch.float32, device=dev)
    _need(topk_idx, "topk_idx", torch.int32, (N, K))
    _need(topk_w, "topk_w", torch.float32, (N, K))
    if out is None:
        out = Dispatch(
            expert_counts=torch.empty(E, dtype=torch.int32, device=dev),
            expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
            row_map=torch.empty(N * K, dtype=torch.int32, device=dev),
            src_slot=torch.empty(N * K, dtype=torch.int32, device=dev) if want_src_slot else None,
            X_perm=torch.empty((N * K, H), dtype=torch.bfloat16, device=dev) if permute else None,
        )
    if workspace is None:
        workspace = _fresh_workspace(E, dev, stream)
    launches = ctypes.c_int(0)
    code = lib().moe_route_dispatch(
        _ptr(X), _ptr(W_gate), _ptr(bias), N, H, E, K, int(bool(renorm)), _ptr(topk_idx), _ptr(topk_w),
        _ptr(out.expert_counts), _ptr(out.expert_offsets), _ptr(out.row_map), _ptr(out.src_slot),
        _ptr(out.X_perm), _status_ptr(status), *_workspace_arg(workspace), ctypes.byref(launches),
        _stream(stream))
    _check(code, "moe_route_dispatch")
    return topk_idx, topk_w, out, launches.value


@dataclass
class DispatchEP:
    expert_counts: torch.Tensor
    expert_offsets: torch.Tensor
    row_map: torch.Tensor
    rank_counts: torch.Tensor
    rank_offsets: torch.Tensor
    send_token: torch.Tensor
    slot_send_row: torch.Tensor
    expand_idx: torch.Tensor
    send_meta: torch.Tensor
    X_send: Optional[torch.Tensor] = None


def dispatch_ep(topk_idx: torch.Tensor, E: int, ep_size: int, X: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None, status=None, stream=None) -> DispatchEP:
    """Expert-parallel dispatch metadata with token deduplication (moe_dispatch_ep).
    send_token / X_send have N*min(K, ep_size) rows; rank_offsets[-1] of them are used."""
    N, K = topk_idx.shape
    _need(topk_idx, "topk_idx", torch.int32)
    dev = topk_idx.device
    H = 0
    if X is not None:
        _need(X, "X", torch.bfloat16)
        if X.shape[0] != N:
            raise ValueError("X and topk_idx disagree on N")
        H = X.shape[1]
    if ep_size < 1 or E % ep_size != 0:
        raise ValueError("ep_size must divide E")
    R, P = ep_size, E // ep_size
    rows = N * min(K, R)
    i32 = dict(dtype=torch.int32, device=dev)
    out = DispatchEP(
        expert_counts=torch.empty(E, **i32), expert_offsets=torch.empty(E + 1, **i32),
        row_map=torch.empty(N * K, **i32), rank_counts=torch.empty(R, **i32),
        rank_offsets=torch.empty(R + 1, **i32), send_token=torch.empty(max(rows, 1), **i32),
        slot_send_row=torch.empty(N * K, **i32), expand_idx=torch.empty(N * K, **i32),
        send_meta=torch.empty((R, P + 1), **i32),
        X_send=torch.empty((rows, H), dtype=torch.bfloat16, device=dev) if X is not None else None)
    if workspace is None:
        workspace = _fresh_workspace(E, dev, stream)
    code = lib().moe_dispatch_ep(
        _ptr(topk_idx), _ptr(X), N, H, E, K, ep_size, _ptr(out.expert_counts), _ptr(out.expert_offsets),
        _ptr(out.row_map), _ptr(out.rank_counts), _ptr(out.rank_offsets), _ptr(out.send_token),
        _ptr(out.slot_send_row), _ptr(out.expand_idx), _ptr(out.send_meta), _ptr(out.X_send), _status_ptr(status),
        *_workspace_arg(workspace), _stream(stream))
    _check(code, "moe_dispatch_ep")
    return out


def permute(X: torch.Tensor, row_map: torch.Tensor, K: int, bf16: bool = True, fp8: bool = False,
            X_perm=None, X_fp8=None, X_scale=None, status=None, stream=None, scale_format: str = "fp32"):
    """Row permute: returns (X_perm, X_fp8, X_scale) (entries None when not requested);
    X_scale is fp32, or uint8 UE8M0 bytes with scale_format="ue8m0"."""
    fmt = _scale_format(scale_format)
    N, H = X.shape
    _need(X, "X", torch.bfloat16)
    _need(row_map, "row_map", torch.int32, (N * K,))
    dev = X.device
    if bf16 and X_perm is None:
        X_perm = torch.empty((N * K, H), dtype=torch.bfloat16, device=dev)
    if fp8 and X_fp8 is None:
        X_fp8 = torch.empty((N * K, H), dtype=torch.uint8, device=dev)
        X_scale = torch.empty((N * K, H // 128), dtype=_scale_dtype(scale_format), device=dev)
    code = lib().moe_permute_ex(_ptr(X), _ptr(row_map), N, H, K, _ptr(X_perm), _ptr(X_fp8), _ptr(X_scale), fmt,
                                _status_ptr(status), _stream(stream))
    _check(code, "moe_permute_ex")
    return X_perm, X_fp8, X_scale


def combine(Y: torch.Tensor, row_map: torch.Tensor, topk_w: torch.Tensor, out=None, status=None,
            stream=None, residual=None) -> torch.Tensor:
    """Weighted gather back to token order: out bf16 [N,H]; with `residual`
    (bf16 [N,H]) the residual is added before the bf16 rounding
    (moe_combine_residual).  `out` may be `residual` itself (in place)."""
    N, K = topk_w.shape
    H = Y.shape[1]
    _need(Y, "Y", torch.bfloat16, (N * K, H))
    _need(row_map, "row_map", torch.int32, (N * K,))
    _need(topk_w, "topk_w", torch.float32)
    if out is None:
        out = torch.empty((N, H), dtype=torch.bfloat16, device=Y.device)
    _need(out, "out", torch.bfloat16, (N, H))
    if residual is None:
        code = lib().moe_combine(_ptr(Y), _ptr(row_map), _ptr(topk_w), N, H, K, _ptr(out), _status_ptr(status),
                                 _stream(stream))
        _check(code, "moe_combine")
    else:
        _need(residual, "residual", torch.bfloat16, (N, H))
        code = lib().moe_combine_residual(_ptr(Y), _ptr(row_map), _ptr(topk_w), _ptr(residual), N, H, K,
                                          _ptr(out), _status_ptr(status), _stream(stream))
        _check(code, "moe_combine_residual")
    return out
