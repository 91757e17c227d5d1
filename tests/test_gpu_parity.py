"""GPU path vs the CPU oracle, through the C ABI (needs a GB300).

Bars: routing ids bit-exact; routing weights within 1e-5 relative; outputs
max|out - ref| / max|ref| <= 1e-2 (the expert GEMMs take x exactly, as two
e4m3 halves under a block scale, and h to about 9 significant bits; the
oracle keeps fp64 throughout).
"""
import numpy as np
import pytest

import moe_inputs as mi
import mxfp4_mixture_experts_route_gb300 as moe
import oracle as O
from libmoe_util import device_block, ensure_built, gpu_forward, shape_of
from oracle.gap_tables import enforce_gap

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
W_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _check(inp, ids, w, out, rows=None):
    rows = np.arange(inp.cfg.S) if rows is None else np.asarray(rows)
    rids, rw, rout, _ = O.moe_forward(inp, rows)
    assert np.array_equal(ids[rows], rids), "routing ids differ"
    assert np.max(np.abs(w[rows] - rw) / rw) <= W_TOL
    err = O.parity_error(out[rows], rout)
    assert err <= OUT_TOL, f"out parity {err:.3e}"
    return err


def _gap_inputs(cfg, seed):
    return mi.make_inputs(cfg, seed, attempts=enforce_gap(cfg, seed), use_stored_attempts=False)


@pytest.mark.parametrize("ci", [0, 1, 2])
def test_configs_full(ci):
    inp = mi.make_inputs(mi.CONFIGS[ci])
    ids, w, out = gpu_forward(inp)
    _check(inp, ids, w, out)


def test_config3_sampled():
    cfg = mi.CONFIGS[3]
    inp = mi.make_inputs(cfg)
    ids, w, out = gpu_forward(inp)
    # every token's routing exactly; outputs on a sample of tokens
    L = O.router_logits(inp.x, inp.w_gate, inp.logit_off)
    rids, rw = O.route(L, inp.bias, cfg.k)
    assert np.array_equal(ids, rids)
    assert np.max(np.abs(w - rw) / rw) <= W_TOL
    _check(inp, ids, w, out, rows=[0, 17, 63, 64, 100, 127])


def test_config4_sampled():
    cfg = mi.CONFIGS[4]
    inp = mi.make_inputs(cfg)
    ids, w, out = gpu_forward(inp)
    L = O.router_logits(inp.x, inp.w_gate, inp.logit_off)
    rids, rw = O.route(L, inp.bias, cfg.k)
    assert np.array_equal(ids, rids)
    assert np.max(np.abs(w - rw) / rw) <= W_TOL
    _check(inp, ids, w, out, rows=[0, 1, 2047, 4095])


SMALL = [
    mi.MoEConfig("s1", S=1, d=128, E=8, k=1, I=128),
    mi.MoEConfig("s3", S=3, d=384, E=16, k=2, I=256),
    mi.MoEConfig("s17", S=17, d=256, E=40, k=8, I=128, post_norm=True),
    mi.MoEConfig("s33", S=33, d=512, E=12, k=3, I=384, zipf=1.1),
    mi.MoEConfig("kE", S=5, d=128, E=4, k=4, I=128),
    mi.MoEConfig("s70", S=70, d=256, E=8, k=2, I=256),      # > NT picks per expert
    mi.MoEConfig("s160", S=160, d=256, E=8, k=2, I=128),    # 32-pick tiles (40 picks per expert)
    mi.MoEConfig("maxEk", S=4, d=256, E=512, k=16, I=128),  # E and k at their maxima
    mi.MoEConfig("maxd", S=2, d=16384, E=8, k=2, I=128),    # d at its maximum (two gather passes)
    mi.MoEConfig("maxI", S=2, d=256, E=4, k=1, I=8192),     # I at its maximum
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c.name for c in SMALL])
def test_small_shapes(cfg):
    inp = _gap_inputs(cfg, 1)
    ids, w, out = gpu_forward(inp)
    _check(inp, ids, w, out)


def test_route_then_experts_separately():
    import torch
    inp = mi.make_inputs(mi.CONFIGS[0])
    blk = device_block(inp)
    s = blk.shape
    moe.route(s, blk.x, blk.w_gate, blk.bias, blk.logit_off, blk.ids, blk.weights, blk.ws)
    # experts on the oracle's ids / weights (reversed pick order: any order is allowed)
    L = O.router_logits(inp.x, inp.w_gate)
    rids, rw = O.route(L, inp.bias, inp.cfg.k)
    ids_t = torch.as_tensor(rids[:, ::-1].copy()).cuda()
    w_t = torch.as_tensor(rw[:, ::-1].astype(np.float32).copy()).cuda()
    moe.experts(s, blk.x, ids_t, w_t, blk.w13, blk.w13s, blk.w2, blk.w2s, blk.norm_w, blk.out, blk.ws)
    moe.check_device_status(blk.ws)
    assert np.array_equal(blk.ids.cpu().numpy(), rids)
    _, _, rout, _ = O.moe_forward(inp)
    assert O.parity_error(blk.out.cpu().numpy(), rout) <= OUT_TOL


def test_one_expert_takes_every_token():
    cfg = mi.MoEConfig("hot", S=40, d=256, E=8, k=2, I=128)
    inp = mi.make_inputs(cfg, 2, use_stored_attempts=False)
    inp.bias = np.zeros(cfg.E, np.float32)
    inp.bias[3] = 5.0           # expert 3 wins every token; 40 picks > NT
    inp.bias[6] = 4.0
    ids, w, out = gpu_forward(inp)
    assert np.all(ids == np.array([3, 6]))
    _check(inp, ids, w, out)


def test_bad_ids_latch_status():
    import torch
    inp = mi.make_inputs(mi.CONFIGS[0])
    blk = device_block(inp)
    s = blk.shape
    ids = torch.tensor([[0, 1]] * 8, dtype=torch.int32).cuda()
    ids[2, 1] = 9          # out of range
    ids[5, 1] = 0          # repeated within token 5
    w = torch.full((8, 2), 0.5, dtype=torch.float32).cuda()
    moe.experts(s, blk.x, ids, w, blk.w13, blk.w13s, blk.w2, blk.w2s, None, blk.out, blk.ws)
    rc, det = moe.device_status(blk.ws)
    assert rc == moe.MOE_ERR_BAD_IDS and det in (2 * 2 + 1, 5 * 2 + 1)
    out = blk.out.cpu().numpy()
    assert np.all(np.isfinite(out))
    # the valid picks still contribute: token 2 = 0.5 * expert 0 only
    xf = O.bf16_to_f64(inp.x)
    y0 = O.expert_ffn(xf[2:3], inp.w13[0], inp.w13s[0], inp.w2[0], inp.w2s[0])[0]
    assert O.parity_error(out[2], 0.5 * y0) <= OUT_TOL
    assert moe.device_status(blk.ws)[0] == moe.MOE_OK      # cleared


def test_bad_scale_latches_status():
    # e8m0 255 is NaN (OCP MX v1.0); it is reported, not silently used
    inp = mi.make_inputs(mi.CONFIGS[0])
    inp.w2s = inp.w2s.copy()
    inp.w2s[:, 7, 1] = 255
    blk = device_block(inp)
    blk.forward()
    rc, det = moe.device_status(blk.ws)
    assert rc == moe.MOE_ERR_BAD_SCALE and det == 255


@pytest.mark.parametrize("shift13,shift2", [(24, -24), (-20, 20), (40, -40)])
def test_scale_range(shift13, shift2):
    # every e8m0 byte 0..254 is a valid scale: gate_up scales moved up (down)
    # by 2^shift13 and the down scales back, so h spans a very different range
    # from y (kept well inside fp32: h grows as 2^(2 shift13)); the routing is
    # unchanged
    inp = mi.make_inputs(mi.CONFIGS[0])
    inp.w13s = np.clip(inp.w13s.astype(np.int64) + shift13, 0, 254).astype(np.uint8)
    inp.w2s = np.clip(inp.w2s.astype(np.int64) + shift2, 0, 254).astype(np.uint8)
    ids, w, out = gpu_forward(inp)
    _check(inp, ids, w, out)


@pytest.mark.parametrize("ci,pinned", [(1, True), (1, False), (2, True), (3, True)])
def test_forward_host_matches_forward(ci, pinned):
    """Host buffers: small pinned ones are read and written in place by the
    kernels (all four at S = 8, ids and weights at S = 32), the others are
    staged through the workspace; either way the bytes equal moe_forward's."""
    import torch
    inp = mi.make_inputs(mi.CONFIGS[ci])
    blk = device_block(inp)
    ids, w, out = [t.cpu().numpy() for t in blk.forward()]
    s = blk.shape

    def host(t):
        return t.pin_memory() if pinned else t

    xh = host(torch.as_tensor(inp.x).view(torch.bfloat16).clone())
    oh = host(torch.empty((s.S, s.d), dtype=torch.float32))
    ih = host(torch.empty((s.S, s.k), dtype=torch.int32))
    wh = host(torch.empty((s.S, s.k), dtype=torch.float32))
    moe.forward_host(s, xh, blk.w_gate, blk.bias, blk.logit_off, blk.w13, blk.w13s, blk.w2, blk.w2s,
                     blk.norm_w, ih, wh, oh, blk.ws)
    torch.cuda.current_stream().synchronize()
    moe.check_device_status(blk.ws)
    assert np.array_equal(ih.numpy(), ids) and np.array_equal(wh.numpy(), w)
    assert np.array_equal(oh.numpy(), out)


@pytest.mark.parametrize("ci", [2, 3])
def test_repeat_calls_are_deterministic(ci):
    """Synchronised calls with other work on the stream in between (a write
    larger than L2) give identical bytes: every kernel reads its predecessors'
    outputs coherently, whatever the caches hold from the previous call."""
    import torch
    inp = mi.make_inputs(mi.CONFIGS[ci])
    blk = device_block(inp)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ref = None
    for _ in range(6):
        flush.zero_()
        got = [t.cpu().numpy().copy() for t in blk.forward()]
        moe.check_device_status(blk.ws, "repeat")
        if ref is None:
            ref = got
        for u, v in zip(got, ref):
            assert np.array_equal(u, v)


@pytest.mark.parametrize("ci", [0, 1, 2, 3])
def test_back_to_back_calls_with_different_routing(ci):
    """Calls enqueued one after another on one stream, with nothing between
    them, overlap on the device (each kernel may start before its predecessor
    ends, and the expert kernel before the token gather ends).  Four inputs with
    different routing, each called many times in turn into fresh outputs, must
    give exactly what each gives alone."""
    import torch
    inp = mi.make_inputs(mi.CONFIGS[ci])
    blk = device_block(inp)
    s = blk.shape
    xs = [blk.x, blk.x.roll(1, 0).contiguous(), blk.x.flip(1).contiguous(), (-blk.x).contiguous()]

    def outs():
        return (torch.empty((s.S, s.k), dtype=torch.int32, device="cuda"),
                torch.empty((s.S, s.k), dtype=torch.float32, device="cuda"),
                torch.empty((s.S, s.d), dtype=torch.float32, device="cuda"))

    def call(x, o):
        moe.forward(s, x, blk.w_gate, blk.bias, blk.logit_off, blk.w13, blk.w13s, blk.w2, blk.w2s,
                    blk.norm_w, *o, blk.ws)

    refs = []
    for x in xs:
        o = outs()
        call(x, o)
        torch.cuda.synchronize()
        moe.check_device_status(blk.ws, "alone")
        refs.append(o)
    rounds = 12 if ci < 3 else 4
    got = []
    for _ in range(rounds):
        for v, x in enumerate(xs):
            o = outs()
            call(x, o)
            got.append((v, o))
    torch.cuda.synchronize()
    moe.check_device_status(blk.ws, "back to back")
    for v, o in got:
        for a, b in zip(o, refs[v]):
            assert torch.equal(a, b), f"input {v} differs when enqueued back to back"
