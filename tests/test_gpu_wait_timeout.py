"""A bounded device wait that runs out: the error path, on a real GPU.

Every spin of the expert kernel gives up after a time limit, latches
MOE_ERR_TIMEOUT with the site of the wait, and takes the kernel's abort path
(the other warps leave their waits, copies in flight land, tensor memory is
freed).  The test builds the library's wait-test variant (waits give up after
1 ms; one down unit can be told to wait for a readiness count no kernel
reaches -- a flag that nothing sets), makes that wait run out on the tiny
workload, checks the reported status and site, and then checks that the next
normal call on the same device and workspace matches the oracle.  Nothing
here faults or hangs the GPU: the wait is bounded and the kernel returns.
"""
import ctypes
import os

import numpy as np
import pytest

import moe_inputs as mi
import mxfp4_mixture_experts_route_gb300 as moe
import oracle as O
from libmoe_util import device_block, ensure_built

pytestmark = pytest.mark.gpu

SITE_TILE_READY = 2     # the token producer's wait for its tile's h rows


@pytest.fixture(scope="module")
def waitlib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    from mxfp4_mixture_experts_route_gb300.build import WAIT_TEST_LIB, build_wait_test_library
    if not os.path.exists(WAIT_TEST_LIB):
        build_wait_test_library()
    L = moe.load_library(WAIT_TEST_LIB)
    L.moe_test_unreachable_wait.argtypes = [ctypes.c_int]
    L.moe_test_unreachable_wait.restype = ctypes.c_int
    return L


def _forward(L, blk):
    import torch
    s, p = blk.shape, (lambda t: None if t is None else t.data_ptr())
    rc = L.moe_forward(ctypes.byref(s), p(blk.x), p(blk.w_gate), p(blk.bias), p(blk.logit_off),
                       p(blk.w13), p(blk.w13s), p(blk.w2), p(blk.w2s), p(blk.norm_w), p(blk.ids),
                       p(blk.weights), p(blk.out), p(blk.ws), blk.ws.numel(),
                       torch.cuda.current_stream().cuda_stream)
    assert rc == moe.MOE_OK
    det = ctypes.c_int32(0)
    st = L.moe_device_status(p(blk.ws), ctypes.byref(det), torch.cuda.current_stream().cuda_stream)
    return st, det.value


def test_wait_runs_out_and_the_next_call_is_correct(waitlib):
    inp = mi.make_inputs(mi.CONFIGS[0])
    blk = device_block(inp)
    waitlib.moe_test_unreachable_wait(1)
    try:
        st, det = _forward(waitlib, blk)
    finally:
        waitlib.moe_test_unreachable_wait(0)
    assert st == moe.MOE_ERR_TIMEOUT and det == SITE_TILE_READY, (st, det)
    # the status was cleared by the read; the context and the workspace are usable
    for _ in range(2):
        st, det = _forward(waitlib, blk)
        assert st == moe.MOE_OK, (st, det)
        rids, rw, rout, _ = O.moe_forward(inp)
        assert np.array_equal(blk.ids.cpu().numpy(), rids)
        assert O.parity_error(blk.out.cpu().numpy(), rout) <= 1e-2
