"""CPU oracle for the MoE routing hot path (route -> dispatch -> permute -> combine).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` are the only
callers.  The product path (the CUDA library and its Python binding) never
imports this package, and this package imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, fp64); this module compiles it
with gcc on first use and wraps it for numpy arrays.  Every function cites the
page passage it follows in ``oracle.c``.

Parity status: every function here is pinned by ``tests/test_oracle.py``
(brute force on tiny inputs, closed forms, library cross-checks, invariants and
the hand-derived fixtures in ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
BAD_ARG = 1
BAD_INDEX = 7


def build(force: bool = False) -> str:
    """Compile oracle.c into _oracle.so (portable C11, OpenMP over tokens)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_route.argtypes = [P, P, P, I64, I64, I64, I64, ctypes.c_int, P, P, P, P]
        lib.oracle_dispatch.argtypes = [P, I64, I64, I64, P, P, P, P]
        lib.oracle_permute.argtypes = [P, P, I64, I64, I64, P, P, P]
        lib.oracle_combine.argtypes = [P, P, P, I64, I64, I64, P]
        lib.oracle_combine_residual.argtypes = [P, P, P, P, I64, I64, I64, P]
        lib.oracle_expert_fixture.argtypes = [P, P, I64, I64, I64, P]
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_e4m3_satfinite.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_e4m3_satfinite.restype = ctypes.c_uint8
        lib.oracle_dispatch_ep.argtypes = [P, I64, I64, I64, I64, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_logsumexp.argtypes = [P, I64, I64, P]
        lib.oracle_load_stats.argtypes = [P, I64, P, I64, ctypes.c_double, P]
        lib.oracle_ue8m0_block_scale.argtypes = [ctypes.c_double]
        lib.oracle_ue8m0_block_scale.restype = ctypes.c_uint8
        lib.oracle_permute_ue8m0.argtypes = [P, P, I64, I64, I64, P, P]
        lib.oracle_fp8_block_scale.argtypes = [ctypes.c_double]
        lib.oracle_fp8_block_scale.restype = ctypes.c_float
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != OK:
        raise OracleError(f"{what} failed with code {rc}")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's OpenMP loops from now on (the default is every host core)."""
    _load().oracle_set_num_threads(int(n))


def route(X_bits, W_bits, bias=None, K=1, renorm=True, want_logits=False, want_probs=False):
    """Route every token: returns (topk_idx int32 [N,K], topk_w f32 [N,K][, logits f64][, probs f64]).

    X_bits: uint16 bf16 bits [N,H]; W_bits: uint16 bf16 bits [H,E]; bias: f32 [E] or None.
    """
    lib = _load()
    X = _c(X_bits, np.uint16)
    W = _c(W_bits, np.uint16)
    N, H = X.shape
    H2, E = W.shape
    if H2 != H:
        raise ValueError("X and W disagree on H")
    b = None if bias is None else _c(bias, np.float32)
    idx = np.empty((N, K), np.int32)
    w = np.empty((N, K), np.float32)
    logits = np.empty((N, E), np.float64) if want_logits else None
    probs = np.empty((N, E), np.float64) if want_probs else None
    _check(lib.oracle_route(_ptr(X), _ptr(W), _ptr(b), N, H, E, K, int(bool(renorm)),
                            _ptr(idx), _ptr(w), _ptr(logits), _ptr(probs)), "oracle_route")
    out = [idx, w]
    if want_logits:
        out.append(logits)
    if want_probs:
        out.append(probs)
    return tuple(out)


def logsumexp(logits):
    """Per-token log-sum-exp of fp64 logits [N,E] (NaN as -inf): fp64 [N]."""
    lib = _load()
    L = _c(logits, np.float64)
    N, E = L.shape
    out = np.empty(N, np.float64)
    _check(lib.oracle_logsumexp(_ptr(L), N, E, _ptr(out)), "oracle_logsumexp")
    return out


def load_stats(counts, lse=None, z_coef=1e-3):
    """Expert-load statistics: (max/mean, p95/mean, z_loss, mean) as fp64."""
    lib = _load()
    c = _c(counts, np.int32)
    l = None if lse is None else _c(lse, np.float64)
    out = np.empty(4, np.float64)
    _check(lib.oracle_load_stats(_ptr(c), c.shape[0], _ptr(l), 0 if l is None else l.shape[0],
                                 float(z_coef), _ptr(out)), "oracle_load_stats")
    return out


def dispatch(topk_idx, E):
    """Stable counting-sort metadata: returns (counts [E], offsets [E+1], row_map [N*K], src_slot [N*K])."""
    lib = _load()
    idx = _c(topk_idx, np.int32)
    N, K = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    row_map = np.empty(N * K, np.int32)
    src_slot = np.empty(N * K, np.int32)
    _check(lib.oracle_dispatch(_ptr(idx), N, E, K, _ptr(counts), _ptr(offsets),
                               _ptr(row_map), _ptr(src_slot)), "oracle_dispatch")
    return counts, offsets, row_map, src_slot


def dispatch_ep(topk_idx, E, ep_size):
    """Expert-parallel dispatch metadata with dedup: returns a dict of counts, offsets,
    row_map, src_slot, rank_counts, rank_offsets, send_token (rank_offsets[-1] rows),
    slot_send_row, expand_idx, send_meta [R, P+1]."""
    lib = _load()
    idx = _c(topk_idx, np.int32)
    N, K = idx.shape
    R = ep_size
    P = E // R if R > 0 else 0
    out = dict(counts=np.empty(E, np.int32), offsets=np.empty(E + 1, np.int32),
               row_map=np.empty(N * K, np.int32), src_slot=np.empty(N * K, np.int32),
               rank_counts=np.empty(R, np.int32), rank_offsets=np.empty(R + 1, np.int32),
               send_token=np.empty(max(N * min(K, R), 1), np.int32),
               slot_send_row=np.empty(N * K, np.int32), expand_idx=np.empty(N * K, np.int32),
               send_meta=np.empty((R, P + 1), np.int32))
    _check(lib.oracle_dispatch_ep(_ptr(idx), N, E, K, R, *(_ptr(out[k]) for k in (
        "counts", "offsets", "row_map", "src_slot", "rank_counts", "rank_offsets", "send_token",
        "slot_send_row", "expand_idx", "send_meta"))), "oracle_dispatch_ep")
    out["send_token"] = out["send_token"][:out["rank_offsets"][-1]]
    return out


def permute(X_bits, row_map, K, fp8=False):
    """Row permute (+ optional E4M3 1x128 quantise): returns Xp bits [, Xq uint8, Xs f32]."""
    lib = _load()
    X = _c(X_bits, np.uint16)
    rm = _c(row_map, np.int32)
    N, H = X.shape
    Xp = np.empty((N * K, H), np.uint16)
    Xq = np.empty((N * K, H), np.uint8) if fp8 else None
    Xs = np.empty((N * K, H // 128), np.float32) if fp8 else None
    _check(lib.oracle_permute(_ptr(X), _ptr(rm), N, H, K, _ptr(Xp), _ptr(Xq), _ptr(Xs)),
           "oracle_permute")
    return (Xp, Xq, Xs) if fp8 else Xp


def permute_ue8m0(X_bits, row_map, K):
    """E4M3 copy with UE8M0 block scales: returns Xq uint8 [N*K,H], Xs uint8 [N*K,H/128]."""
    lib = _load()
    X = _c(X_bits, np.uint16)
    rm = _c(row_map, np.int32)
    N, H = X.shape
    Xq = np.empty((N * K, H), np.uint8)
    Xs = np.empty((N * K, H // 128), np.uint8)
    _check(lib.oracle_permute_ue8m0(_ptr(X), _ptr(rm), N, H, K, _ptr(Xq), _ptr(Xs)), "oracle_permute_ue8m0")
    return Xq, Xs


def ue8m0_block_scale(amax):
    """UE8M0 scale byte of one block with absolute maximum `amax`."""
    return int(_load().oracle_ue8m0_block_scale(float(amax)))


def combine(Y_bits, row_map, topk_w):
    """Weighted gather back to token order: returns out bf16 bits [N,H]."""
    lib = _load()
    Y = _c(Y_bits, np.uint16)
    rm = _c(row_map, np.int32)
    w = _c(topk_w, np.float32)
    N, K = w.shape
    H = Y.shape[1]
    out = np.empty((N, H), np.uint16)
    _check(lib.oracle_combine(_ptr(Y), _ptr(rm), _ptr(w), N, H, K, _ptr(out)), "oracle_combine")
    return out


def combine_residual(Y_bits, row_map, topk_w, residual_bits):
    """forward_aggregate: weighted gather plus the residual, one bf16 rounding: bits [N,H]."""
    lib = _load()
    Y = _c(Y_bits, np.uint16)
    rm = _c(row_map, np.int32)
    w = _c(topk_w, np.float32)
    R = _c(residual_bits, np.uint16)
    N, K = w.shape
    H = Y.shape[1]
    if R.shape != (N, H):
        raise ValueError("residual must be [N,H]")
    out = np.empty((N, H), np.uint16)
    _check(lib.oracle_combine_residual(_ptr(Y), _ptr(rm), _ptr(w), _ptr(R), N, H, K, _ptr(out)),
           "oracle_combine_residual")
    return out


def expert_fixture(Xp_bits, offsets):
    """Synthetic expert outputs: Y[p] = bf16(fl32(Xp[p] * fl32(1 + e(p)/E)))."""
    lib = _load()
    Xp = _c(Xp_bits, np.uint16)
    off = _c(offsets, np.int32)
    rows, H = Xp.shape
    E = off.shape[0] - 1
    Y = np.empty_like(Xp)
    _check(lib.oracle_expert_fixture(_ptr(Xp), _ptr(off), E, rows, H, _ptr(Y)),
           "oracle_expert_fixture")
    return Y


def bf16_to_f64(b: int) -> float:
    return float(_load().oracle_bf16_to_f64(int(b)))


def f64_to_bf16(x: float) -> int:
    return int(_load().oracle_f64_to_bf16(float(x)))


def e4m3_to_f64(c: int) -> float:
    return float(_load().oracle_e4m3_to_f64(int(c)))


def f64_to_e4m3(x: float) -> int:
    return int(_load().oracle_f64_to_e4m3_satfinite(float(x)))


def fp8_block_scale(amax: float) -> float:
    return float(_load().oracle_fp8_block_scale(float(amax)))


def bf16_bits_to_f64_array(bits) -> np.ndarray:
    """Vector form of the exact bf16 -> fp64 widening (pure numpy)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_path(X_bits, W_bits, bias, K, renorm=True, fp8=False):
    """The whole path on the CPU: route, dispatch, permute, fixture, combine.

    Returns a dict of every intermediate (numpy arrays).
    """
    E = W_bits.shape[1]
    idx, w = route(X_bits, W_bits, bias, K, renorm)
    counts, offsets, row_map, src_slot = dispatch(idx, E)
    if fp8:
        Xp, Xq, Xs = permute(X_bits, row_map, K, fp8=True)
    else:
        Xp, Xq, Xs = permute(X_bits, row_map, K), None, None
    Y = expert_fixture(Xp, offsets)
    out = combine(Y, row_map, w)
    return dict(topk_idx=idx, topk_w=w, counts=counts, offsets=offsets, row_map=row_map,
                src_slot=src_slot, Xp=Xp, Xq=Xq, Xs=Xs, Y=Y, out=out)
