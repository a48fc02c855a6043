"""Failure detection on the GPU without a fault.

The one-launch dispatch waits at a grid barrier whose spin is bounded (2 s of
%globaltimer).  Here the barrier's arrive counter starts at 0xFFFFFFFF: each
CTA adds its arrival before it polls, so the counter runs from 0 to G-1 and can
never reach G -- the wait cannot complete, the way a flag that nothing sets
cannot.  Every CTA gives up at the bound, records MOE_ERR_TIMEOUT in the status
word and returns before it writes any output; the context stays usable.
"""
import time

import numpy as np
import pytest
import torch

import combine_moe_route_02_gb300 as moe
import moe_inputs as mi
import oracle

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
