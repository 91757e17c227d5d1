"""The token quantiser's precision claim, checked on the GPU's own output.

The expert GEMMs take each bf16 token row x as two e4m3 rows under one e8m0
scale 2^(s - 127) per 32 elements (the tensor core's block-scaled 8-bit
operand).  The claim (the gather kernel's contract): s is chosen so that the
block's largest magnitude M lies in [128, 256) * 2^(s - 127) (s clamped to
1..247), hi = e4m3(x / 2^(s-127)) and lo = e4m3(x / 2^(s-127) - hi), so that
  * (hi + lo) * 2^(s-127) == x exactly for every |x| >= 2^-9 M, and
  * |(hi + lo) * 2^(s-127) - x| <= 2^-17 M below that.
Why: with M / 2^(s-127) >= 2^7 and |x| >= 2^-9 M, a = x / 2^(s-127) has its 8
significant bits at or above 2^-9 (e4m3's subnormal step), hi keeps the top 4
and the remainder a - hi (at most 4 more bits, same step or coarser) is exact
in e4m3; below, lo rounds at the 2^-9 step, an error of at most 2^-10, i.e.
2^-17 of M / 2^(s-127).

The test builds token rows whose 32-element blocks hit the edges of that
claim -- a block maximum at a power of two and just below one, elements 2^8,
2^9 and 2^10 below the maximum, bf16 values with all 8 significant bits set,
an all-zero block, very large and very small blocks -- runs the block, reads
the gathered rows back from the workspace and decodes them here with an e4m3
decoder written from the OCP 8-bit floating point specification (E4M3: 1 sign,
4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal,
m/8 * 2^-6; S.1111.111 is NaN).
"""
import numpy as np
import pytest

import moe_inputs as mi
import mxfp4_mixture_experts_route_gb300 as moe
from libmoe_util import device_block, ensure_built


def e4m3_value(code):
    c = np.asarray(code, np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    ex = (c >> 3) & 15
    man = c & 7
    mag = np.where(ex == 0, man / 8.0 * 2.0 ** -6, (1.0 + man / 8.0) * np.exp2(ex - 7.0))
    mag = np.where((ex == 15) & (man == 7), np.nan, mag)
    return sign * mag


def test_e4m3_decoder_spec_values():
    assert e4m3_value(0x38) == 1.0 and e4m3_value(0xB8) == -1.0
    assert e4m3_value(0x7E) == 448.0                    # largest finite
    assert e4m3_value(0x08) == 2.0 ** -6                # smallest normal
    assert e4m3_value(0x01) == 2.0 ** -9                # smallest subnormal
    assert e4m3_value(0x07) == 7 * 2.0 ** -9
    assert np.isnan(e4m3_value(0x7F)) and e4m3_value(0x00) == 0.0


def _bf16(v):
    return mi.f32_to_bf16_bits(np.asarray(v, np.float32))


def _edge_rows(S, d, rng):
    """[S, d] bf16 bits: every 32-element block one of the edge patterns."""
    f = np.zeros((S, d), np.float64)
    nb = d // 32
    for t in range(S):
        for b in range(nb):
            kind = (t * nb + b) % 9
            sgn = rng.choice([-1.0, 1.0], 32)
            m = rng.integers(128, 256, 32) / 128.0          # 8 significant bits in [1, 2)
            if kind == 0:      # maximum exactly a power of two, elements 2^8, 2^9, 2^10 below it
                M = 2.0 ** int(rng.integers(-8, 8))
                v = sgn * m * M * 2.0 ** -rng.integers(0, 12, 32)
                v[:4] = [M, M * 2.0 ** -8, -M * 2.0 ** -9, M * 2.0 ** -10]
                v[4] = M * (1 + 2 ** -7) * 2.0 ** -9        # just above the exact range's edge
                v[5] = M * (2 - 2 ** -7) * 2.0 ** -10       # just below it
            elif kind == 1:    # maximum just below a power of two (8 bits all set)
                M = (2 - 2 ** -7) * 2.0 ** int(rng.integers(-8, 8))
                v = sgn * m * M / 2 * 2.0 ** -rng.integers(0, 12, 32)
                v[0] = -M
            elif kind == 2:    # all 8 significant bits set everywhere, spread over 2^10
                v = sgn * (2 - 2 ** -7) * 2.0 ** -rng.integers(0, 11, 32)
            elif kind == 3:
                v = np.zeros(32)
            elif kind == 4:    # very large block
                v = sgn * m * 2.0 ** (40 - rng.integers(0, 14, 32))
            elif kind == 5:    # very small block
                v = sgn * m * 2.0 ** (-40 - rng.integers(0, 14, 32))
            elif kind == 6:    # one element, the rest zero
                v = np.zeros(32)
                v[int(rng.integers(0, 32))] = -m[0] * 3.0
            elif kind == 7:    # elements far below the maximum (the inexact range)
                v = sgn * m * 2.0 ** -rng.integers(9, 24, 32)
                v[0] = 1.5
            else:              # a plain N(0, 1) block
                v = rng.standard_normal(32)
            f[t, 32 * b:32 * b + 32] = v
    bits = _bf16(f)
    return bits


def _check_rows(xrow, hi, lo, scale_of_block):
    """One token row x (fp64) against its e4m3 hi / lo rows and block scales."""
    n_exact = n_below = 0
    for b in range(len(xrow) // 32):
        xb = xrow[32 * b:32 * b + 32]
        M = np.max(np.abs(xb))
        byte = int(scale_of_block(b))
        want = 1 if M == 0 else int(np.clip(np.frexp(M)[1] - 1 + 127 - 7, 1, 247))
        assert byte == want, (b, byte, want)
        v = (hi[32 * b:32 * b + 32] + lo[32 * b:32 * b + 32]) * 2.0 ** (byte - 127)
        assert np.all(np.isfinite(v))
        exact = np.abs(xb) >= M * 2.0 ** -9
        assert np.array_equal(v[exact], xb[exact]), b
        assert np.all(np.abs(v[~exact] - xb[~exact]) <= M * 2.0 ** -17), b
        n_exact += int(exact.sum())
        n_below += int((~exact).sum())
    return n_exact, n_below


def _edge_block(cfg, seed):
    inp = mi.make_inputs(cfg)
    inp.x = _edge_rows(cfg.S, cfg.d, np.random.default_rng(seed))
    return inp, device_block(inp)


@pytest.mark.gpu
def test_gathered_token_rows_meet_the_precision_claim():
    """The gather kernel's rows (moe_experts: the picks' rows in sorted order)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    cfg = mi.CONFIGS[0]           # S = 8, d = 256, E = 8, k = 2
    inp, blk = _edge_block(cfg, 7)
    s = blk.shape
    moe.route(s, blk.x, blk.w_gate, blk.bias, blk.logit_off, blk.ids, blk.weights, blk.ws)
    moe.experts(s, blk.x, blk.ids, blk.weights, blk.w13, blk.w13s, blk.w2, blk.w2s, blk.norm_w, blk.out, blk.ws)
    moe.check_device_status(blk.ws, "route + experts")
    P, d = cfg.S * cfg.k, cfg.d
    pos = moe.read_region(s, blk.ws, moe.MOE_WS_POS, torch.int32).numpy()
    xq = moe.read_region(s, blk.ws, moe.MOE_WS_XQ).numpy().reshape(2 * P, d)
    xs = moe.read_region(s, blk.ws, moe.MOE_WS_XS).numpy().reshape(-1, P + 64, 16)
    x = mi.bf16_bits_to_f32(inp.x).astype(np.float64)
    n_exact = n_below = 0
    for p in range(P):
        t, r = p // cfg.k, int(pos[p])
        e, b = _check_rows(x[t], e4m3_value(xq[2 * r]), e4m3_value(xq[2 * r + 1]),
                           lambda blk_i: xs[blk_i // 8, r, blk_i % 8])
        n_exact += e
        n_below += b
    assert n_exact > 1000 and n_below > 100
