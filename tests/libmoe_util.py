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
    """(ids, weights, out fp64, the router's fp32 logits) of one moe_forward."""
    import torch
    blk = device_block(inp)
    ids, w, out = blk.forward()
    moe.check_device_status(blk.ws, "forward")
    L = moe.read_region(blk.shape, blk.ws, moe.MOE_WS_LOGITS, torch.float32).numpy().reshape(inp.cfg.S, inp.cfg.E)
    return ids.cpu().numpy(), w.cpu().numpy(), out.cpu().numpy().astype(np.float64), L


def check_routing_weights(L_gpu, x_bits, w_gate_bits, logit_off, ids, w, rows=None):
    """The routing weights are w_j = s_j / sum s over the picks, s = sigmoid of
    the fp32 logits.  The logits' last bits depend on the order of the fp32
    sums (K split over CTAs, the tensor core's accumulation; the kda page lets
    split-K reductions differ only in order), so what is unique is checked:

      * the GPU's logits against the exact dot products, within the error of an
        fp32 sum of K exact products in any order: K * 2^-23 * sum_i |x_i w_i|
        (twice the unit roundoff, in case an adder truncates), plus one
        rounding of the offset add;
      * the weights against those logits, renormalised in fp64: within 2e-6
        relative (the device's sigmoid and division in fp32)."""
    import oracle as O
    rows = np.arange(L_gpu.shape[0]) if rows is None else np.asarray(rows)
    xf, wf = O.bf16_to_f64(x_bits[rows]), O.bf16_to_f64(w_gate_bits)
    exact = xf @ wf.T
    K = xf.shape[1]
    bound = K * 2.0 ** -23 * (np.abs(xf) @ np.abs(wf).T)
    if logit_off is not None:
        exact = exact + np.asarray(logit_off, np.float64)[None, :]
        bound = bound + 2.0 ** -23 * (np.abs(exact) + 1.0)
    Lg = L_gpu[rows].astype(np.float64)
    assert np.all(np.abs(Lg - exact) <= bound), float(np.max(np.abs(Lg - exact) / bound))
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(Lg, ids[rows].astype(np.int64), 1)))
    want = s / s.sum(1, keepdims=True)
    err = float(np.max(np.abs(w[rows] - want) / want))
    assert err <= 2e-6, err
