"""moe_dispatch_noalloc, the dispatch entry point for callers that cannot
allocate device memory while they dispatch (a fixed up-front memory plan, a
context where cudaMalloc would block or synchronise the device, a C caller
without a device allocator).  It runs the same one-launch dispatch as
moe_dispatch but on scratch memory compiled into the library, so the caller
passes only inputs and outputs.

What is checked, through the C ABI:
  * two calls in a row give exactly the outputs of moe_dispatch with a
    caller-provided workspace, so a call's result does not depend on what an
    earlier call left in the shared scratch array; the shapes cover the
    one-launch copy, the E4M3 copy and a row copy large enough (>= 256 MiB)
    to run in a launch of its own;
  * after a first call of each shape, further calls leave the device's free
    memory unchanged (cudaMemGetInfo): the entry point allocates nothing;
  * the size limit ceil(N / min(N, SMs)) * K <= 16384 at its exact boundary
    (accepted, checked against moe_dispatch) and one token past it (refused
    with MOE_ERR_UNSUPPORTED before any launch), with K = 3.
This file is named to be collected last.
"""
import ctypes

import pytest
import torch

import combine_moe_route_02_gb300 as moe
import moe_inputs as mi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def noalloc():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    moe.build()
    f = moe.lib().moe_dispatch_noalloc
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.argtypes = [P, P, I64, I32, I32, I32, P, P, P, P, P, P, P, P, P]
    f.restype = I32
    return f


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _outputs(N, H, E, K, fp8, rows, dev):
    return dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                row_map=torch.empty(N * K, dtype=torch.int32, device=dev),
                src_slot=torch.empty(N * K, dtype=torch.int32, device=dev),
                Xp=torch.empty((N * K, H), dtype=torch.bfloat16, device=dev) if rows else None,
                Xq=torch.empty((N * K, H), dtype=torch.uint8, device=dev) if fp8 else None,
                Xs=torch.empty((N * K, H // 128), dtype=torch.float32, device=dev) if fp8 else None,
                st=torch.zeros(1, dtype=torch.int32, device=dev))


def _call(noalloc, idx, X, N, H, E, K, o):
    return noalloc(_ptr(idx), _ptr(X), N, H, E, K, _ptr(o["counts"]), _ptr(o["offsets"]), _ptr(o["row_map"]),
                   _ptr(o["src_slot"]), _ptr(o["Xp"]), _ptr(o["Xq"]), _ptr(o["Xs"]), _ptr(o["st"]),
                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _assert_same(o, ref, N, K, fp8):
    assert o["st"].item() == 0, moe.status_string(o["st"].item())
    assert torch.equal(o["counts"], ref.expert_counts)
    assert torch.equal(o["offsets"], ref.expert_offsets)
    assert torch.equal(o["row_map"], ref.row_map)
    assert torch.equal(o["src_slot"], ref.src_slot)
    if o["Xp"] is not None:
        assert torch.equal(o["Xp"].view(torch.int16), ref.X_perm.view(torch.int16))
    if fp8:
        assert torch.equal(o["Xq"], ref.X_fp8)
        assert torch.equal(o["Xs"], ref.X_scale)
    assert int(o["counts"].sum()) == N * K


@pytest.mark.parametrize("N,H,E,K,fp8", [
    (4096, 1024, 64, 2, False),      # rows copied inside the one launch
    (2048, 2048, 128, 8, True),      # bf16 rows and E4M3 codes + scales
    (16384, 4096, 64, 2, False),     # 384 MiB row copy: its own launch of the permute kernel
])
def test_noalloc_matches_workspace_dispatch_on_two_calls(noalloc, N, H, E, K, fp8):
    dev = torch.device("cuda")
    X = mi.random_bf16((N, H), seed=N + H).to(dev)
    idx = mi.random_topk_idx(N, E, K, seed=N + E).to(dev)
    ref = moe.dispatch(idx, E, X, fp8=fp8)     # the existing entry point, workspace from the caller
    o = _outputs(N, H, E, K, fp8, True, dev)
    for call in range(3):
        if call == 2:
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
        for t in o.values():
            if t is not None:
                t.fill_(-1 if t.dtype == torch.int32 else 0)
        o["st"].zero_()
        rc = _call(noalloc, idx, X, N, H, E, K, o)
        assert rc == 0, moe.status_string(rc)
        torch.cuda.synchronize()
        if call == 2:
            # the first call of this shape may have loaded kernel code; later ones allocate nothing
            assert torch.cuda.mem_get_info()[0] == free_before
        _assert_same(o, ref, N, K, fp8)


def test_noalloc_size_limit_boundary(noalloc):
    dev = torch.device("cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    K, E = 3, 16
    tok_per = 16384 // K                 # 5461 tokens x 3 = 16383 slots per CTA
    N = tok_per * sms                    # the largest N with ceil(N / SMs) * K <= 16384
    idx = mi.random_topk_idx(N, E, K, seed=7).to(dev)
    ref = moe.dispatch(idx, E)           # metadata only
    o = _outputs(N, 0, E, K, False, False, dev)
    rc = _call(noalloc, idx, None, N, 0, E, K, o)
    assert rc == 0, moe.status_string(rc)
    torch.cuda.synchronize()
    _assert_same(o, ref, N, K, False)
    # one token more: a CTA would hold 5462 x 3 = 16386 slots -- refused before any launch
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: the call returns first
    rc = noalloc(fake, None, N + 1, 64, E, K, fake, fake, fake, None, None, None, None, None, None)
    assert rc == moe.ERR_UNSUPPORTED


def test_noalloc_rejects_sizes_beyond_its_scratch(noalloc):
    # more than 16384 slots per CTA with one CTA per SM: refused before any launch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N, K = 16384 * sms + 1, 1
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: the call returns first
    rc = noalloc(fake, None, N, 64, 8, K, fake, fake, fake, None, None, None, None, None, None)
    assert rc == moe.ERR_UNSUPPORTED
