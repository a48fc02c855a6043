"""moe_dispatch_noalloc, the dispatch entry point for callers that cannot
allocate device memory while they dispatch (a fixed up-front memory plan, a
context where cudaMalloc would block or synchronise the device, a C caller
without a device allocator).  It runs the same one-launch dispatch as
moe_dispatch but on scratch memory compiled into the library, so the caller
passes only inputs and outputs.

The check: through the C ABI, two calls in a row (the second one finds the
scratch holding the first call's contents) must give exactly the outputs of
moe_dispatch with a caller-provided workspace.  This file is named to be
collected last.
"""
import ctypes

import numpy as np
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


def test_noalloc_matches_workspace_dispatch_on_two_calls(noalloc):
    dev = torch.device("cuda")
    for N, H, E, K, fp8 in [(4096, 1024, 64, 2, False), (2048, 2048, 128, 8, True)]:
        X = mi.random_bf16((N, H), seed=N + H).to(dev)
        idx = mi.random_topk_idx(N, E, K, seed=N + E).to(dev)
        ref = moe.dispatch(idx, E, X, fp8=fp8)     # the existing entry point, workspace from the caller
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        row_map = torch.empty(N * K, dtype=torch.int32, device=dev)
        src_slot = torch.empty(N * K, dtype=torch.int32, device=dev)
        Xp = torch.empty((N * K, H), dtype=torch.bfloat16, device=dev)
        Xq = torch.empty((N * K, H), dtype=torch.uint8, device=dev) if fp8 else None
        Xs = torch.empty((N * K, H // 128), dtype=torch.float32, device=dev) if fp8 else None
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        rc = noalloc(_ptr(idx), _ptr(X), N, H, E, K, _ptr(counts), _ptr(offsets), _ptr(row_map), _ptr(src_slot),
                     _ptr(Xp), _ptr(Xq), _ptr(Xs), _ptr(st),
                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, moe.status_string(rc)
        torch.cuda.synchronize()
        assert st.item() == 0, moe.status_string(st.item())
        assert torch.equal(counts, ref.expert_counts)
        assert torch.equal(offsets, ref.expert_offsets)
        assert torch.equal(row_map, ref.row_map)
        assert torch.equal(src_slot, ref.src_slot)
        assert torch.equal(Xp.view(torch.int16), ref.X_perm.view(torch.int16))
        if fp8:
            assert torch.equal(Xq, ref.X_fp8)
            assert torch.equal(Xs, ref.X_scale)
        assert int(counts.sum()) == N * K


def test_noalloc_rejects_sizes_beyond_its_scratch(noalloc):
    # more than 16384 slots per CTA with one CTA per SM: refused before any launch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N, K = 16384 * sms + 1, 1
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: the call returns first
    rc = noalloc(fake, None, N, 64, 8, K, fake, fake, fake, None, None, None, None, None, None)
    assert rc == moe.ERR_UNSUPPORTED
