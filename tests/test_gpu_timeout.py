"""Failure detection on the GPU without a fault.

The one-launch dispatch waits at a grid barrier whose spin is bounded (2 s of
%globaltimer).  Here the barrier's arrive counter starts at 0xFFFFFFFF: each
CTA adds its arrival before it polls, so the counter runs from 0 to G-1 and can
never reach G -- the wait cannot complete, the way a flag that nothing sets
cannot.  Every CTA gives up at the bound, records MOE_ERR_TIMEOUT in the status
word and returns before it writes any output; the context stays usable.  The
one-launch route + dispatch has the same kind of barrier after its router phase
and is tested the same way.
"""
import time

import numpy as np
import pytest
import torch

import combine_moe_route_02_gb300 as moe
import moe_inputs as mi
import oracle
from parity_util import compare_topk

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    moe.build()
    moe.lib()


def test_dispatch_grid_barrier_timeout_reports_status():
    N, H, E, K = 4000, 256, 16, 2
    idx = mi.random_topk_idx(N, E, K, seed=1).to(DEV)
    X = mi.random_bf16((N, H), seed=2).to(DEV)
    ws = torch.zeros(moe.dispatch_workspace_size(N, E, K), dtype=torch.uint8, device=DEV)
    ws.view(torch.int32)[0] = -1          # arrive counter 0xFFFFFFFF: the barrier can never open
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.time()
    moe.dispatch(idx, E, X, workspace=ws, status=st)
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert st.item() == moe.ERR_TIMEOUT, moe.status_string(st.item())
    assert 1.5 < waited < 30.0
    # the same context still dispatches correctly with a clean workspace
    st.zero_()
    d = moe.dispatch(idx, E, X, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _, _, r, _ = oracle.dispatch(idx.cpu().numpy(), E)
    assert np.array_equal(d.row_map.cpu().numpy(), r)


def test_route_dispatch_grid_barrier_timeout_reports_status():
    # the one-launch route + dispatch waits at the same kind of bounded grid barrier
    # after its router phase; with the arrive counter at 0xFFFFFFFF every CTA gives up
    N, H, E, K = 2048, 1024, 64, 2
    X, W, _ = mi.make_route_inputs(N, H, E, 3)
    Xd, Wd = X.to(DEV), W.to(DEV)
    ws = torch.zeros(moe.dispatch_workspace_size(N, E, K), dtype=torch.uint8, device=DEV)
    ws.view(torch.int32)[0] = -1
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.time()
    idx, tw, d, n = moe.route_dispatch(Xd, Wd, K, workspace=ws, status=st)
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert n == 1                                   # the fused launch ran
    assert st.item() == moe.ERR_TIMEOUT, moe.status_string(st.item())
    assert 1.5 < waited < 30.0
    # the router part completed before the barrier: its ids and weights match the oracle
    r_idx, r_w, L, P = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), None, K, True, want_logits=True,
                                    want_probs=True)
    compare_topk(idx.cpu().numpy(), tw.cpu().numpy(), r_idx, r_w, L, P, True)
    # the same context still works with a clean workspace
    st.zero_()
    idx, tw, d, n = moe.route_dispatch(Xd, Wd, K, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0 and n == 1
    _, _, r, _ = oracle.dispatch(idx.cpu().numpy(), E)
    assert np.array_equal(d.row_map.cpu().numpy(), r)
