"""Pins of the CPU oracle (no GPU).

Nothing here re-evaluates the oracle's own formulas.  Each function of
``oracle.moe_oracle`` is checked against one of:
  * published values: the OCP MX v1.0 e2m1 and e8m0 tables and hand-worked
    MXFP4 rows (tests/golden/, each file cites its source);
  * closed forms worked out by hand (one-token experts, the fp32 rounding of a
    logit, RMSNorm of a constant vector, ties in the top-k);
  * an independent brute force on tiny inputs: pure-Python loops, the decode
    read from the golden table, a full sort of all experts, every expert
    evaluated densely on every token and then selected;
  * invariants: weights sum to 1, expert relabelling, linearity in the w2
    scale, scale invariance of the post-expert norm, unpicked experts do not
    matter, rows are independent.
"""
import math

import numpy as np
import pytest

import moe_inputs as mi
import oracle as O
from conftest import golden_path


def _read_table(name):
    rows = []
    for line in open(golden_path(name)):
        line = line.split("#")[0].strip()
        if line:
            a, b = line.split()
            rows.append((int(a), float(b)))
    return rows


E2M1 = dict(_read_table("e2m1_codes.txt"))


# ---------------------------------------------------------------------------
# element decodes against the published tables
# ---------------------------------------------------------------------------
def test_e2m1_table():
    codes = np.arange(16)
    got = O.e2m1_value(codes)
    want = np.array([E2M1[c] for c in codes])
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))     # code 8 is -0.0


def test_e8m0_cases():
    for b, v in _read_table("e8m0_cases.txt"):
        got = float(O.e8m0_value(np.array([b]))[0])
        if math.isnan(v):
            assert math.isnan(got)
        else:
            assert got == v, (b, got, v)


def test_dequant_worked_rows():
    for line in open(golden_path("mxfp4_worked.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        bts, scs, vals = [p.split() for p in line.split("|")]
        nblk = len(scs)
        packed = np.zeros((1, 16 * nblk), np.uint8)
        packed[0, :len(bts)] = [int(b, 16) for b in bts]
        scales = np.array([[int(s) for s in scs]], np.uint8)
        got = O.dequant_mxfp4(packed, scales)[0]
        want = np.array([float(v) for v in vals])
        assert np.array_equal(got[:len(want)], want), (line, got[:len(want)])
        assert np.array_equal(np.signbit(got[:len(want)]), np.signbit(want))
        assert np.all(got[len(want):] == 0)


# ---------------------------------------------------------------------------
# router closed forms
# ---------------------------------------------------------------------------
def _bf16(a):
    return mi.f32_to_bf16_bits(np.asarray(a, np.float32))


def test_logit_is_exact_sum_rounded_once_to_fp32():
    # 2**24 + 1 + 1: a left-to-right fp32 sum gives 2**24 (each +1 is a tie to
    # even), the exact sum 16777218 is representable in fp32.
    x = _bf16([[1.0, 1.0, 1.0]])
    w = _bf16([[2.0 ** 24, 1.0, 1.0]])
    L = O.router_logits(x, w)
    assert L.dtype == np.float32 and L[0, 0] == np.float32(16777218.0)
    # fp32 offset added after the rounding
    L = O.router_logits(x, w, np.array([-2.0], np.float32))
    assert L[0, 0] == np.float32(16777216.0)


def test_route_closed_form_and_ties():
    # logits 0 -> sigmoid 0.5 everywhere; equal selection scores pick the
    # lowest ids; weights are 1/k.
    L = np.zeros((2, 6), np.float32)
    ids, w = O.route(L, np.zeros(6, np.float32), 3)
    assert ids.tolist() == [[0, 1, 2], [0, 1, 2]]
    assert np.allclose(w, 1 / 3, rtol=0, atol=1e-15)
    # the bias only selects; the weights use the unbiased sigmoid
    L = np.array([[0.0, math.log(3.0), 0.0, -math.log(3.0)]], np.float32)
    bias = np.array([0.0, 0.0, 0.0, 0.6], np.float32)
    ids, w = O.route(L, bias, 2)
    # sel = 0.5, 0.75, 0.5, 0.25+0.6=0.85 -> picks {1, 3}; s = 0.75, 0.25
    s1 = 1 / (1 + math.exp(-float(np.float32(math.log(3.0)))))
    s3 = 1 / (1 + math.exp(float(np.float32(math.log(3.0)))))
    assert ids.tolist() == [[1, 3]]
    assert np.allclose(w[0], [s1 / (s1 + s3), s3 / (s1 + s3)], rtol=1e-15)
    assert abs(w[0, 0] - 0.75) < 1e-7
    g = O.score_gap(L, bias, 2)
    assert abs(g[0] - (0.75 - 0.5)) < 1e-7


# ---------------------------------------------------------------------------
# expert closed forms (one token, x = e_0)
# ---------------------------------------------------------------------------
def _pack(codes):
    codes = np.asarray(codes, np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def _one_expert_case(gate_code_even, gate_code_odd, up_code, down_codes, d=32, I=32):
    """x = e_0.  Gate row r: element 0 has the code for r even/odd, the rest 0;
    up rows: every element ``up_code``; down row m: every element down_codes[m]."""
    gate = np.zeros((I, d), np.uint8)
    gate[0::2, 0] = gate_code_even
    gate[1::2, 0] = gate_code_odd
    gate[:, 5] = 9                       # -0.5 at column 5: x[5] = 0 so it must not matter
    up = np.full((I, d), up_code, np.uint8)
    w13 = _pack(np.concatenate([gate, up]))[None]
    w13s = np.full((1, 2 * I, d // 32), 127, np.uint8)
    down = np.repeat(np.asarray(down_codes, np.uint8)[:, None], I, axis=1)
    w2 = _pack(down)[None]
    w2s = np.full((1, d, I // 32), 127, np.uint8)
    x = np.zeros((1, d))
    x[0, 0] = 1.0
    return x, w13, w13s, w2, w2s


def test_expert_closed_form():
    d = I = 32
    down_codes = [m % 8 for m in range(d)]                 # row m: e2m1(m % 8)
    x, w13, w13s, w2, w2s = _one_expert_case(2, 6, 4, down_codes)
    # g_r = 1 (r even) or 4 (r odd); u_r = 2 * sum_c x_c = 2
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))
    h_even, h_odd = 1.0 * sig(1.0) * 2.0, 4.0 * sig(4.0) * 2.0
    hsum = (I // 2) * (h_even + h_odd)
    mag = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    want = np.array([mag[m % 8] * hsum for m in range(d)])
    y = O.expert_ffn(x, w13[0], w13s[0], w2[0], w2s[0])[0]
    assert np.allclose(y, want, rtol=1e-14, atol=0)
    # negative gate: g = -1 (code 10) -> silu(-1) = -sigmoid(-1)
    x, w13, w13s, w2, w2s = _one_expert_case(10, 10, 4, [1] * d)
    y = O.expert_ffn(x, w13[0], w13s[0], w2[0], w2s[0])[0]
    assert np.allclose(y, I * 0.5 * (-sig(-1.0)) * 2.0, rtol=1e-14)


def test_scale_blocks_along_k():
    # d = 64: two scale blocks; only block 1 is scaled by 2**3.  x = e_40.
    d, I = 64, 32
    gate = np.full((I, d), 2, np.uint8)                    # 1.0
    up = np.full((I, d), 2, np.uint8)
    w13 = _pack(np.concatenate([gate, up]))[None]
    w13s = np.full((1, 2 * I, 2), 127, np.uint8)
    w13s[0, :, 1] = 130
    w2 = _pack(np.full((d, I), 2, np.uint8))[None]
    w2s = np.full((1, d, 1), 127, np.uint8)
    x = np.zeros((1, d))
    x[0, 40] = 1.0
    y = O.expert_ffn(x, w13[0], w13s[0], w2[0], w2s[0])[0]
    g = 8.0
    assert np.allclose(y, I * g / (1 + math.exp(-g)) * g, rtol=1e-14)


def test_post_norm_closed_form():
    c, eps = 3.0, 1e-6
    y = np.full((1, 16), -c)
    wn = np.linspace(0.5, 1.5, 16)
    got = O.post_expert_norm(y, wn, eps)[0]
    assert np.allclose(got, -c / math.sqrt(c * c + eps) * wn, rtol=1e-15)


# ---------------------------------------------------------------------------
# brute force on tiny inputs (independent pure-Python evaluation)
# ---------------------------------------------------------------------------
def _bf16_to_float(b):
    return float(mi.bf16_bits_to_f32(np.array([b], np.uint16))[0])


def _brute_dequant_row(packed_row, scale_row):
    vals = []
    for j, byte in enumerate(packed_row):
        for code in (int(byte) & 15, int(byte) >> 4):
            vals.append(E2M1[code])
    return [v * 2.0 ** (int(scale_row[i // 32]) - 127) for i, v in enumerate(vals)]


def _brute_forward(inp):
    cfg = inp.cfg
    S, d, E, k, I = cfg.S, cfg.d, cfg.E, cfg.k, cfg.I
    xs = [[_bf16_to_float(b) for b in row] for row in inp.x]
    wg = [[_bf16_to_float(b) for b in row] for row in inp.w_gate]
    W13 = [[_brute_dequant_row(inp.w13[e][r], inp.w13s[e][r]) for r in range(2 * I)] for e in range(E)]
    W2 = [[_brute_dequant_row(inp.w2[e][m], inp.w2s[e][m]) for m in range(d)] for e in range(E)]
    # every expert on every token
    Y = [[None] * E for _ in range(S)]
    for t in range(S):
        for e in range(E):
            h = []
            for i in range(I):
                g = sum(W13[e][i][c] * xs[t][c] for c in range(d))
                u = sum(W13[e][I + i][c] * xs[t][c] for c in range(d))
                h.append(g / (1.0 + math.exp(-g)) * u)
            Y[t][e] = [sum(W2[e][m][i] * h[i] for i in range(I)) for m in range(d)]
    ids, ws, outs = [], [], []
    for t in range(S):
        logit = []
        for e in range(E):
            acc = math.fsum(xs[t][c] * wg[e][c] for c in range(d))
            acc = float(np.float32(acc))
            if inp.logit_off is not None:
                acc = float(np.float32(np.float32(acc) + inp.logit_off[e]))
            logit.append(acc)
        s = [1.0 / (1.0 + math.exp(-z)) for z in logit]
        sel = [(s[e] + float(inp.bias[e]), -e) for e in range(E)]
        top = sorted(range(E), key=lambda e: sel[e], reverse=True)[:k]
        top.sort()
        tot = sum(s[e] for e in top)
        w = [s[e] / tot for e in top]
        ys = []
        for e in top:
            y = Y[t][e]
            if cfg.post_norm:
                r = math.sqrt(sum(v * v for v in y) / d + cfg.norm_eps)
                y = [y[m] / r * float(inp.norm_w[m]) for m in range(d)]
            ys.append(y)
        outs.append([sum(w[j] * ys[j][m] for j in range(k)) for m in range(d)])
        ids.append(top)
        ws.append(w)
    return np.array(ids), np.array(ws), np.array(outs)


@pytest.mark.parametrize("post_norm,zipf", [(False, 0.0), (True, 0.0), (False, 1.1)])
def test_brute_force_tiny(post_norm, zipf):
    cfg = mi.MoEConfig("brute", S=3, d=64, E=5, k=2, I=64, post_norm=post_norm, zipf=zipf)
    inp = mi.make_inputs(cfg, seed=11, use_stored_attempts=False)
    ids, w, out, _ = O.moe_forward(inp)
    bids, bw, bout = _brute_forward(inp)
    assert np.array_equal(ids, bids)
    assert np.allclose(w, bw, rtol=1e-13, atol=0)
    assert np.max(np.abs(out - bout)) <= 1e-12 * np.max(np.abs(bout))


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def small():
    cfg = mi.MoEConfig("small", S=6, d=128, E=24, k=3, I=64)
    return mi.make_inputs(cfg, seed=3, use_stored_attempts=False)


def test_weights_sum_to_one(small):
    _, w, _, _ = O.moe_forward(small)
    assert np.all(np.abs(w.sum(1) - 1) <= 1e-15)
    assert np.all(w > 0)


def test_expert_relabelling(small):
    perm = np.random.default_rng(0).permutation(small.cfg.E)       # new id -> old id
    inv = np.argsort(perm)
    relab = mi.MoEInputs(**{**small.__dict__})
    relab.w_gate, relab.bias = small.w_gate[perm], small.bias[perm]
    relab.w13, relab.w13s, relab.w2, relab.w2s = (small.w13[perm], small.w13s[perm],
                                                  small.w2[perm], small.w2s[perm])
    ids0, w0, out0, _ = O.moe_forward(small)
    ids1, w1, out1, _ = O.moe_forward(relab)
    for t in range(small.cfg.S):
        old = perm[ids1[t]]
        order = np.argsort(old)
        assert np.array_equal(old[order], ids0[t])
        assert np.allclose(w1[t][order], w0[t], rtol=1e-15)
    assert np.allclose(out1, out0, rtol=1e-13, atol=1e-12 * np.abs(out0).max())
    assert np.array_equal(inv[perm], np.arange(small.cfg.E))


def test_down_scale_linearity(small):
    # +1 on every w2 scale byte doubles every expert output exactly
    _, _, out0, _ = O.moe_forward(small)
    two = mi.MoEInputs(**{**small.__dict__})
    two.w2s = (small.w2s + 1).astype(np.uint8)
    _, _, out1, _ = O.moe_forward(two)
    assert np.array_equal(out1, 2 * out0)


def test_post_norm_scale_invariance(small):
    # with eps = 0 the RMSNorm output does not depend on the scale of y
    cfg = small.cfg.with_(post_norm=True, norm_eps=0.0)
    a = mi.MoEInputs(**{**small.__dict__, "cfg": cfg, "norm_w": mi.gen_norm_w(cfg, 3)})
    b = mi.MoEInputs(**{**a.__dict__})
    b.w2s = (a.w2s + 3).astype(np.uint8)
    _, _, oa, _ = O.moe_forward(a)
    _, _, ob, _ = O.moe_forward(b)
    assert np.allclose(oa, ob, rtol=1e-12, atol=1e-12 * np.abs(oa).max())


def test_unpicked_experts_do_not_matter(small):
    ids, _, out0, _ = O.moe_forward(small)
    unused = sorted(set(range(small.cfg.E)) - set(ids.ravel().tolist()))
    assert unused, "fixture should leave an expert unpicked"
    c = mi.MoEInputs(**{**small.__dict__})
    c.w13 = small.w13.copy()
    c.w2 = small.w2.copy()
    c.w13[unused] ^= 0x5A
    c.w2[unused] ^= 0xA5
    _, _, out1, _ = O.moe_forward(c)
    assert np.array_equal(out0, out1)


def test_rows_are_independent(small):
    ids, w, out, L = O.moe_forward(small)
    rows = np.array([4, 1])
    ids2, w2, out2, L2 = O.moe_forward(small, rows)
    assert np.array_equal(ids2, ids[rows]) and np.array_equal(L2, L[rows])
    assert np.allclose(out2, out[rows], rtol=1e-14, atol=1e-12 * np.abs(out).max())


def test_one_hot_router_is_dense_expert():
    cfg = mi.MoEConfig("onehot", S=4, d=64, E=6, k=1, I=32)
    inp = mi.make_inputs(cfg, seed=5, use_stored_attempts=False)
    inp.w_gate = np.zeros_like(inp.w_gate)           # logits 0 -> s = 0.5
    inp.bias = np.zeros(cfg.E, np.float32)
    inp.bias[4] = 0.05
    ids, w, out, _ = O.moe_forward(inp)
    assert np.all(ids == 4) and np.all(w == 1.0)
    # the dense expert by explicit matrices: W1 = rows 0..I-1, W3 = rows I..2I-1
    W13 = O.dequant_mxfp4(inp.w13[4], inp.w13s[4])
    W2 = O.dequant_mxfp4(inp.w2[4], inp.w2s[4])
    X = O.bf16_to_f64(inp.x)
    for t in range(cfg.S):
        g = W13[:cfg.I] @ X[t]
        u = W13[cfg.I:] @ X[t]
        y = W2 @ (g * (1 / (1 + np.exp(-g))) * u)
        assert np.allclose(out[t], y, rtol=1e-14, atol=1e-12 * np.abs(y).max())


def test_stored_gap_tables_hold():
    from oracle.gap_tables import enforce_gap  # noqa: F401  (the writer of the table)
    for cfg in mi.CONFIGS[:4]:
        inp_x = mi.gen_x(cfg, 0, mi.stored_attempts(cfg, 0))
        L = O.router_logits(inp_x, mi.gen_w_gate(cfg, 0), mi.gen_logit_offset(cfg, 0))
        assert O.score_gap(L, mi.gen_bias(cfg, 0), cfg.k).min() >= cfg.gap, cfg.name
