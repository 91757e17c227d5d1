"""The latent-MoE layer (moe_latent_forward) against the oracle, through the C ABI.

Bars as for the block: routing ids bit-exact, routing weights through the
router's fp32 logits (check_routing_weights), out max|out - ref| / max|ref|
<= 1e-2.  The GPU rounds the layer's
intermediate activations (the latent rows, the normalised latent output, the
shared expert's silu(g) * u) to bf16, the dense products' operand type, with
fp32 sums; the oracle keeps fp64 throughout.
"""
import numpy as np
import pytest

import moe_inputs as mi
import mxfp4_mixture_experts_route_gb300 as moe
import oracle as O
from libmoe_util import check_routing_weights, ensure_built
from oracle.gap_tables import enforce_gap

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _device(inp):
    cfg = inp.cfg
    shape = moe.LatentShape.of(cfg.S, cfg.H, cfg.LAT, cfg.E, cfg.k, cfg.I, cfg.SI,
                               logit_offset=bool(cfg.zipf), norm_eps=cfg.norm_eps)
    return moe.DeviceLatentWeights(shape, inp.x, inp.w_gate, inp.bias, inp.logit_off, inp.w_ld, inp.w13,
                                   inp.w13s, inp.w2, inp.w2s, inp.ln_w, inp.w_up, inp.w_sgu, inp.w_sd)


def _check(inp, blk):
    import torch
    ids, w, out = [t.cpu().numpy() for t in blk.forward()]
    moe.check_device_status(blk.ws, "latent forward")
    cfg = inp.cfg
    # the router's workspace (over H) opens the layer's workspace
    rshape = moe.MoEShape.of(cfg.S, cfg.H, cfg.E, cfg.k, cfg.I, logit_offset=bool(cfg.zipf))
    Lg = moe.read_region(rshape, blk.ws, moe.MOE_WS_LOGITS, torch.float32).numpy().reshape(cfg.S, cfg.E)
    rids, rw, rout, _ = O.latent_forward(inp)
    assert np.array_equal(ids, rids), "routing ids differ"
    check_routing_weights(Lg, inp.x, inp.w_gate, inp.logit_off, ids, w)
    err = O.parity_error(out, rout)
    assert err <= OUT_TOL, f"out parity {err:.3e}"
    return out


CASES = [
    mi.LatentConfig("lg_s3_noshared", S=3, H=384, LAT=256, E=16, k=2, I=256, SI=0),
    mi.LatentConfig("lg_s20_zipf", S=20, H=256, LAT=384, E=12, k=3, I=128, SI=256, zipf=1.1),
    mi.LatentConfig("lg_s1", S=1, H=128, LAT=128, E=4, k=1, I=128, SI=128),
    # E a multiple of 128: the router's rows join the latent-down launch
    # (with the shared gate/up: three products of x in one launch; without it, two)
    mi.LatentConfig("lg_s5_router_part", S=5, H=256, LAT=256, E=128, k=4, I=128, SI=256),
    mi.LatentConfig("lg_s2_router_part_noshared", S=2, H=384, LAT=128, E=256, k=2, I=256, SI=0, zipf=1.1),
    # more than 32 tokens: the top-k kernel, then up to 128 picks the fused
    # sort + gather after its wait (the latent rows are the call's own), above
    # that the counting sort and the per-token gather
    mi.LatentConfig("lg_s40_k3", S=40, H=256, LAT=256, E=16, k=3, I=128, SI=128),
    mi.LatentConfig("lg_s48_k4", S=48, H=256, LAT=384, E=12, k=4, I=128, SI=0),
]


@pytest.mark.parametrize("ci", [0, 1])
def test_latent_workloads(ci):
    inp = mi.make_latent_inputs(mi.LATENT_CONFIGS[ci])
    _check(inp, _device(inp))


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_latent_shapes(cfg):
    inp = mi.make_latent_inputs(cfg, 1, attempts=enforce_gap(cfg.router(), 1), use_stored_attempts=False)
    _check(inp, _device(inp))


def test_latent_calls_are_repeatable():
    """Two calls with other work in between give identical bytes."""
    import torch
    inp = mi.make_latent_inputs(mi.LATENT_CONFIGS[0])
    blk = _device(inp)
    a = [t.cpu().numpy().copy() for t in blk.forward()]
    torch.empty(256 << 20, dtype=torch.uint8, device="cuda").zero_()
    b = [t.cpu().numpy().copy() for t in blk.forward()]
    moe.check_device_status(blk.ws, "latent forward")
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
