"""Pins of the latent-MoE layer oracle (oracle.latent_forward; CPU only).

Nothing here re-evaluates the oracle's own code.  The layer is checked against:
  * a pure-Python brute force on tiny layers (loops over every sum, the MXFP4
    decode read from the published e2m1 table, a full sort of the experts),
    with and without the shared expert, with the hidden and latent widths
    equal (so that a transposed projection still has the right shape and must
    be caught by value) and different;
  * a reduction to the pinned block: with permutation matrices as the latent
    down and up projections and no shared expert, the layer is the block on
    permuted token rows, normalised and permuted back;
  * invariants: the latent norm removes any scale of the routed output (w2
    scales + 1), and a shared expert with zero gate rows contributes nothing.
"""
import math

import numpy as np
import pytest

import moe_inputs as mi
import oracle as O
import test_oracle as T


def _f(b):
    return T._bf16_to_float(b)


def _silu(v):
    return v / (1.0 + math.exp(-v))


def _brute_latent(inp):
    """Every sum a Python loop (math.fsum), every value from its encoding."""
    cfg = inp.cfg
    S, H, LAT, E, k, I, SI = cfg.S, cfg.H, cfg.LAT, cfg.E, cfg.k, cfg.I, cfg.SI
    xs = [[_f(b) for b in row] for row in inp.x]
    wg = [[_f(b) for b in row] for row in inp.w_gate]
    wld = [[_f(b) for b in row] for row in inp.w_ld]
    wup = [[_f(b) for b in row] for row in inp.w_up]
    W13 = [[T._brute_dequant_row(inp.w13[e][r], inp.w13s[e][r]) for r in range(2 * I)] for e in range(E)]
    W2 = [[T._brute_dequant_row(inp.w2[e][m], inp.w2s[e][m]) for m in range(LAT)] for e in range(E)]
    ids, outs = [], []
    for t in range(S):
        logit = [float(np.float32(math.fsum(xs[t][c] * wg[e][c] for c in range(H)))) for e in range(E)]
        s = [1.0 / (1.0 + math.exp(-z)) for z in logit]
        top = sorted(range(E), key=lambda e: (s[e] + float(inp.bias[e]), -e), reverse=True)[:k]
        top.sort()
        tot = math.fsum(s[e] for e in top)
        xl = [math.fsum(xs[t][c] * wld[i][c] for c in range(H)) for i in range(LAT)]
        yl = [0.0] * LAT
        for e in top:
            h = [_silu(math.fsum(W13[e][i][c] * xl[c] for c in range(LAT))) *
                 math.fsum(W13[e][I + i][c] * xl[c] for c in range(LAT)) for i in range(I)]
            for m in range(LAT):
                yl[m] += s[e] / tot * math.fsum(W2[e][m][i] * h[i] for i in range(I))
        r = math.sqrt(math.fsum(v * v for v in yl) / LAT + cfg.norm_eps)
        zl = [yl[m] / r * float(inp.ln_w[m]) for m in range(LAT)]
        out = [math.fsum(zl[m] * wup[i][m] for m in range(LAT)) for i in range(H)]
        if SI:
            wsgu = [[_f(b) for b in row] for row in inp.w_sgu]
            wsd = [[_f(b) for b in row] for row in inp.w_sd]
            hs = [_silu(math.fsum(xs[t][c] * wsgu[j][c] for c in range(H))) *
                  math.fsum(xs[t][c] * wsgu[SI + j][c] for c in range(H)) for j in range(SI)]
            out = [out[i] + math.fsum(hs[j] * wsd[i][j] for j in range(SI)) for i in range(H)]
        ids.append(top)
        outs.append(out)
    return np.array(ids), np.array(outs)


BRUTE = [
    mi.LatentConfig("lb_square", S=2, H=64, LAT=64, E=4, k=2, I=32, SI=4),
    mi.LatentConfig("lb_wide", S=2, H=96, LAT=64, E=5, k=2, I=32, SI=8),
    mi.LatentConfig("lb_noshared", S=2, H=64, LAT=64, E=4, k=1, I=32, SI=0),
]


@pytest.mark.parametrize("cfg", BRUTE, ids=[c.name for c in BRUTE])
def test_latent_brute_force_tiny(cfg):
    inp = mi.make_latent_inputs(cfg, seed=5, use_stored_attempts=False)
    ids, w, out, _ = O.latent_forward(inp)
    bids, bout = _brute_latent(inp)
    assert np.array_equal(ids, bids)
    assert np.max(np.abs(out - bout)) <= 1e-12 * np.max(np.abs(bout))


def _perm_bits(perm):
    n = len(perm)
    m = np.zeros((n, n), np.float32)
    m[np.arange(n), perm] = 1.0          # row i picks column perm[i]
    return mi.f32_to_bf16_bits(m)


def test_permutation_projections_reduce_to_the_block():
    cfg = mi.LatentConfig("lperm", S=3, H=128, LAT=128, E=6, k=2, I=64, SI=0)
    inp = mi.make_latent_inputs(cfg, seed=9, use_stored_attempts=False)
    rng = np.random.default_rng(3)
    pi, sigma = rng.permutation(128), rng.permutation(128)
    inp.w_ld, inp.w_up = _perm_bits(pi), _perm_bits(sigma)
    ids, w, out, _ = O.latent_forward(inp)
    # the block (pinned in test_oracle) on x with columns permuted by pi,
    # routed on x itself; its RMSNorm; columns permuted by sigma
    L = O.router_logits(inp.x, inp.w_gate)
    rids, rw = O.route(L, inp.bias, cfg.k)
    assert np.array_equal(ids, rids)
    yl = O.experts_combine(O.bf16_to_f64(inp.x)[:, pi], rids, rw, inp.w13, inp.w13s, inp.w2, inp.w2s)
    zl = yl / np.sqrt(np.mean(yl * yl, axis=1, keepdims=True) + cfg.norm_eps) * inp.ln_w
    want = zl[:, sigma]
    assert np.max(np.abs(out - want)) <= 1e-12 * np.max(np.abs(want))


def test_latent_norm_removes_the_routed_scale():
    cfg = mi.LATENT_CONFIGS[0].__class__(**{**mi.LATENT_CONFIGS[0].__dict__, "norm_eps": 0.0})   # exact without eps
    inp = mi.make_latent_inputs(cfg)
    _, _, out, _ = O.latent_forward(inp)
    inp.w2s = (inp.w2s.astype(np.int64) + 1).astype(np.uint8)      # every expert output doubles
    _, _, out2, _ = O.latent_forward(inp)
    assert np.max(np.abs(out2 - out)) <= 1e-12 * np.max(np.abs(out))


def test_shared_expert_with_zero_gate_adds_nothing():
    cfg = mi.LATENT_CONFIGS[0]
    inp = mi.make_latent_inputs(cfg)
    inp.w_sgu = inp.w_sgu.copy()
    inp.w_sgu[:cfg.SI] = 0                  # silu(0) = 0
    _, _, out, _ = O.latent_forward(inp)
    inp.w_sgu, inp.w_sd = None, None
    _, _, routed, _ = O.latent_forward(mi.LatentInputs(**{**inp.__dict__, "cfg": cfg.__class__(
        **{**cfg.__dict__, "SI": 0})}))
    assert np.array_equal(out, routed)
