"""moe_forward_noalloc: the block for callers that cannot allocate device memory.

Such a caller (an operator or plugin interface that is handed only its inputs
and outputs, an application whose memory pool owns the whole GPU, a serving
loop that must never call cudaMalloc) has no workspace to pass.  This entry
point runs the same kernels on a static 32 MiB scratch array inside the
library.  The GPU test calls it through the C ABI twice in a row, with
different inputs, and checks each result against moe_forward's on the same
inputs, with the tolerances of the other parity tests.  This file is named so
that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import moe_inputs as mi
import mxfp4_mixture_experts_route_gb300 as moe
from libmoe_util import device_block, ensure_built, shape_of

OUT_TOL = 1e-2
W_TOL = 1e-5


def _noalloc(L, blk, x):
    import torch
    s = blk.shape
    ids = torch.full((s.S, s.k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((s.S, s.k), dtype=torch.float32, device="cuda")
    out = torch.zeros((s.S, s.d), dtype=torch.float32, device="cuda")
    status = torch.full((2,), 12345, dtype=torch.int32, device="cuda")
    p = lambda t: None if t is None else t.data_ptr()
    rc = L.moe_forward_noalloc(ctypes.byref(s), p(x), p(blk.w_gate), p(blk.bias), p(blk.logit_off),
                               p(blk.w13), p(blk.w13s), p(blk.w2), p(blk.w2s), p(blk.norm_w), p(ids),
                               p(w), p(out), p(status), torch.cuda.current_stream().cuda_stream)
    assert rc == moe.MOE_OK, moe.strerror(rc)
    torch.cuda.current_stream().synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), out.cpu().numpy(), status.cpu().numpy()


@pytest.mark.gpu
def test_noalloc_matches_forward_on_two_calls_in_a_row():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = ensure_built()
    cfg = mi.CONFIGS[1]
    inp = mi.make_inputs(cfg)
    blk = device_block(inp)
    # a second step input: other rows of x, same weights
    x2 = torch.as_tensor(mi.gen_x(cfg, seed=1)).view(torch.bfloat16).cuda()
    for x in (blk.x, x2):
        ids_r, w_r, out_r = [t.cpu().numpy().copy() for t in blk.forward(x)]
        moe.check_device_status(blk.ws, "moe_forward")
        ids, w, out, status = _noalloc(L, blk, x)
        assert list(status) == [moe.MOE_OK, 0]
        assert np.array_equal(ids, ids_r)
        assert np.max(np.abs(w - w_r) / np.abs(w_r)) <= W_TOL
        err = np.max(np.abs(out - out_r)) / np.max(np.abs(out_r))
        assert err <= OUT_TOL, err


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # host-side size check: nothing is enqueued, no device is touched
    L = ensure_built()
    s = shape_of(mi.CONFIGS[3])
    assert moe.workspace_bytes(s) > 32 << 20
    rc = L.moe_forward_noalloc(ctypes.byref(s), *([0x1000] * 13), None, None)
    assert rc == moe.MOE_ERR_WORKSPACE
