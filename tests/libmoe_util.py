"""Shared helpers of the libmoe tests: build-on-demand and device uploads."""
import os

import numpy as np

import moe_inputs as mi
import mxfp4_mixture_experts_route_gb300 as moe


def ensure_built():
    if not os.path.exists(moe.LIB_PATH):
        from mxfp4_mixture_experts_route_gb300.build import build_library
        build_library()
    return moe.lib()


def shape_of(cfg: mi.MoEConfig) -> moe.MoEShape:
    return moe.MoEShape.of(cfg.S, cfg.d, cfg.E, cfg.k, cfg.I, post_norm=cfg.post_norm,
                           logit_offset=bool(cfg.zipf), norm_eps=cfg.norm_eps)


def device_block(inp: mi.MoEInputs) -> moe.DeviceWeights:
    return moe.DeviceWeights(shape_of(inp.cfg), inp.x, inp.w_gate, inp.bias, inp.logit_off,
                             inp.w13, inp.w13s, inp.w2, inp.w2s, inp.norm_w)


def gpu_forward(inp: mi.MoEInputs):
    blk = device_block(inp)
    ids, w, out = blk.forward()
    moe.check_device_status(blk.ws, "forward")
    return ids.cpu().numpy(), w.cpu().numpy(), out.cpu().numpy().astype(np.float64)
