"""moe_forward_noalloc: the block for callers that cannot allocate device memory.

Such a caller (an operator or plugin interface that is handed only its inputs
and outputs, an application whose memory pool owns the whole GPU, a serving
loop that must never call cudaMalloc) has no workspace to pass.  This entry
point runs the same kernels on a static 32 MiB scratch array inside the
library, which keeps whatever the previous call left in it.

The GPU test calls it through the C ABI on a sequence of calls that share the
array: two in a row on the same shape with different inputs, a larger shape, a
shape with the per-pick norm, then smaller shapes again (so that anything read
from a previous call's leftovers would show).  Each result must equal
moe_forward's on the same inputs bit for bit (ids, weights and out): both run
the same kernels on the same inputs, so any difference is a read of stale
scratch.  This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import moe_inputs as mi
import mxfp4_mixture_experts_route_gb300 as moe
from libmoe_util import device_block, ensure_built, shape_of

NORM_CFG = mi.MoEConfig("norm_s17", S=17, d=256, E=40, k=8, I=128, post_norm=True)


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
def test_noalloc_equals_forward_on_calls_in_a_row():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = ensure_built()
    blocks = {}

    def block(cfg):
        if cfg.name not in blocks:
            blocks[cfg.name] = device_block(mi.make_inputs(cfg, 1, use_stored_attempts=False)
                                            if cfg is NORM_CFG else mi.make_inputs(cfg))
        return blocks[cfg.name]

    c0, c1, c2 = mi.CONFIGS[0], mi.CONFIGS[1], mi.CONFIGS[2]
    x1b = torch.as_tensor(mi.gen_x(c1, seed=1)).view(torch.bfloat16).cuda()
    # (workload, input rows): S = 8 twice in a row, then a larger workspace
    # (S = 32), the per-pick norm, and smaller shapes after larger ones
    seq = [(c1, None), (c1, x1b), (c2, None), (NORM_CFG, None), (c0, None), (c1, x1b)]
    assert moe.workspace_bytes(shape_of(c2)) > moe.workspace_bytes(shape_of(c1))
    for cfg, x in seq:
        blk = block(cfg)
        x = blk.x if x is None else x
        ids_r, w_r, out_r = [t.cpu().numpy().copy() for t in blk.forward(x)]
        moe.check_device_status(blk.ws, "moe_forward")
        ids, w, out, status = _noalloc(L, blk, x)
        assert list(status) == [moe.MOE_OK, 0], cfg.name
        assert np.array_equal(ids, ids_r), cfg.name
        assert np.array_equal(w, w_r), cfg.name
        assert np.array_equal(out, out_r), cfg.name


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # host-side size check: nothing is enqueued, no device is touched
    L = ensure_built()
    s = shape_of(mi.CONFIGS[3])
    assert moe.workspace_bytes(s) > 32 << 20
    # 12 tensor pointers, then status and stream
    rc = L.moe_forward_noalloc(ctypes.byref(s), *([0x1000] * 12), None, None)
    assert rc == moe.MOE_ERR_WORKSPACE


def test_noalloc_argument_checks_match_forward():
    # the argument checks run before the scratch array is looked up, with
    # moe_forward's codes
    L = ensure_built()
    s = shape_of(mi.CONFIGS[0])
    good = [0x1000 * (i + 1) for i in range(12)]
    null_x = [None] + good[1:]
    odd_out = good[:11] + [good[11] + 4]
    for args, code in ((null_x, moe.MOE_ERR_INVALID_ARG), (odd_out, moe.MOE_ERR_ALIGNMENT)):
        assert L.moe_forward_noalloc(ctypes.byref(s), *args, None, None) == code
        fwd = args + [0x100000, moe.workspace_bytes(s), None]
        assert L.moe_forward(ctypes.byref(s), *fwd) == code
