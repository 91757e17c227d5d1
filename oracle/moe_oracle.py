"""CPU oracle of the routed MXFP4 mixture-of-experts block -- TEST INFRASTRUCTURE.

Only the test suite, the smoke check and the CPU-baseline leg of the benchmark
use this module.  The CUDA library never imports, links or calls it, and it
shares no code with the CUDA path (its only shared dependency is the seeded
input generator ``moe_inputs``, which holds no arithmetic of the block).

Everything here is the plain definition of the block, evaluated in fp64, with
one exception that the pages fix: the router logits are fp32 values (the k3
page, stage A, gives the router's logits in fp32).  They are formed as the exact fp64 dot
product rounded once to fp32.

Pages cited (vLLM API documentation):
  k3  = vllm.models.muse_spark.amd.mono.kernels.k3 -- stage list (A, route,
        C/D, E) and the summaries of route_token, mx_chunk, fp4_mma, dn_loads.
  k5  = vllm.models.muse_spark.amd.mono.kernels.k5 -- stage HA: fp32 router,
        top 8, ids and weights handed to the expert stage.
  k2  = vllm.models.kimi_k3.amd.specialized_decode.mono.layer -- K2b's latent
        MoE and the k2_launch argument list (w_gate, bias, w13, w13s, w2, w2s,
        out [S, 7168]).
  kda = vllm.models.kimi_k3.amd.specialized_decode.mono.attention.kda -- the
        numerical contract (split-K reductions may differ only in order).

Readings where the pages are silent (the plainest reading in each case):
  * e2m1 / e8m0 follow the OCP Microscaling Formats (MX) v1.0 specification:
    e2m1 = 1 sign, 2 exponent (bias 1), 1 mantissa bit, no inf/NaN; e8m0 =
    2**(byte - 127), byte 255 = NaN.  One scale per 32 consecutive K-elements.
  * packed layout: row-major, K contiguous; byte j of a row holds element 2j in
    its low nibble and 2j+1 in its high nibble; scales are [rows, K/32].
  * w13 rows 0..I-1 are the gate projection (w1), rows I..2I-1 the up (w3).
  * activation: SiLU(gate) * up.
  * routing: s = sigmoid(logit); the k experts with the largest s + bias are
    picked (ties -> lower expert id); weights are the unbiased s of the picks
    renormalised to sum to 1; picks are reported in ascending expert id.
  * post-expert norm (workload 3): RMSNorm y * rsqrt(mean(y^2) + eps) * w_n.
  * out[t] = sum over picks j (ascending id) of w_j * y_j.

Parity status: every function below is pinned by tests/test_oracle.py against
values that do not come from this file (see the header of that test file).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# ----------------------------------------------------------------------------
# MX element decodes (OCP MX v1.0, sections 5.3.3 "FP4" and 5.4.1 "E8M0")
# ----------------------------------------------------------------------------


def e2m1_value(code: np.ndarray) -> np.ndarray:
    """Value of 4-bit e2m1 codes (fp64): sign bit 3, exponent bits 2..1 with
    bias 1, mantissa bit 0; exponent 0 is the subnormal 0.5 * m."""
    code = np.asarray(code, dtype=np.int64)
    sign = (code >> 3) & 1
    ex = (code >> 1) & 3
    man = code & 1
    mag = np.where(ex == 0, 0.5 * man, np.ldexp(1.0 + 0.5 * man, ex - 1))
    return np.where(sign == 1, -mag, mag)


def e8m0_value(byte: np.ndarray) -> np.ndarray:
    """Value of e8m0 scale bytes: 2**(byte - 127); 255 encodes NaN."""
    b = np.asarray(byte, dtype=np.int64)
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 127))


def _byte_pair_table() -> np.ndarray:
    """[256, 2] fp64: the two e2m1 values held by each packed byte (low nibble
    = element 2j, high nibble = element 2j+1)."""
    b = np.arange(256)
    return np.stack([e2m1_value(b & 0x0F), e2m1_value(b >> 4)], axis=1)


_PAIR = _byte_pair_table()


def dequant_mxfp4(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """[R, K/2] packed e2m1 + [R, K/32] e8m0 -> fp64 [R, K].

    k3 page, mx_chunk: rows x K of an MXFP4 [*, k] weight and its e8m0 scales
    (here the plain row-major layout; the vLLM shuffle is not reproduced).
    Element (r, c) = e2m1(code of element c) * 2**(scales[r, c // 32] - 127)."""
    packed = np.asarray(packed, dtype=np.uint8)
    R, Kh = packed.shape
    vals = np.take(_PAIR, packed, axis=0).reshape(R, (2 * Kh) // 32, 32)
    sc = e8m0_value(scales)                 # [R, K/32]
    return (vals * sc[:, :, None]).reshape(R, 2 * Kh)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# router (k3 stage A + route; k5 HA; k2_launch w_gate / bias)
# ----------------------------------------------------------------------------


def router_logits(x_bits: np.ndarray, w_gate_bits: np.ndarray,
                  logit_off: np.ndarray | None = None) -> np.ndarray:
    """fp32 router logits L[t, e] = x[t] . w_gate[e] (+ offset[e]).

    The bf16 x bf16 products are exact in fp64 and the fp64 sum is rounded once
    to fp32 (the pages' logits are fp32).  A per-expert offset, when given, is
    added in fp32 after that rounding."""
    L = bf16_to_f64(x_bits) @ bf16_to_f64(w_gate_bits).T
    L = L.astype(np.float32)
    if logit_off is not None:
        L = (L + np.asarray(logit_off, np.float32)[None, :]).astype(np.float32)
    return L


def sigmoid(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def routing_scores(L32: np.ndarray, bias: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(s, sel): s = sigmoid(L) and the selection score sel = s + bias, fp64."""
    s = sigmoid(L32)
    return s, s + np.asarray(bias, np.float64)[None, :]


def route(L32: np.ndarray, bias: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Sigmoid top-k (k3 route_token: sigmoid scores; k5 stage HA: top 8, ids
    and weights).  Returns ids [S, k] int32 in ascending expert order and the
    renormalised weights [S, k] fp64."""
    s, sel = routing_scores(L32, bias)
    S, E = s.shape
    ids = np.empty((S, k), np.int32)
    w = np.empty((S, k), np.float64)
    for t in range(S):
        # descending sel; equal sel -> lower expert id first (stable sort on -sel)
        order = np.argsort(-sel[t], kind="stable")
        top = np.sort(order[:k])
        ids[t] = top
        w[t] = s[t, top] / s[t, top].sum()
    return ids, w


def score_gap(L32: np.ndarray, bias: np.ndarray, k: int) -> np.ndarray:
    """Per token: sel of the k-th pick minus sel of the (k+1)-th (inf if k == E)."""
    _, sel = routing_scores(L32, bias)
    if k >= sel.shape[1]:
        return np.full(sel.shape[0], np.inf)
    srt = -np.sort(-sel, axis=1)
    return srt[:, k - 1] - srt[:, k]


# ----------------------------------------------------------------------------
# experts (k3 stages C, D, E; k2 K2b "ug", "down")
# ----------------------------------------------------------------------------


def silu(g: np.ndarray) -> np.ndarray:
    """SiLU(g) = g * sigmoid(g), with sigmoid(g) = (1 + tanh(g / 2)) / 2: the
    same function, written so that no exponential overflows for large |g|."""
    g = np.asarray(g, dtype=np.float64)
    return g * 0.5 * (1.0 + np.tanh(0.5 * g))


def expert_ffn(xf: np.ndarray, w13: np.ndarray, w13s: np.ndarray,
               w2: np.ndarray, w2s: np.ndarray) -> np.ndarray:
    """One expert on rows xf [n, d] (fp64): y = W2 (silu(W1 x) * (W3 x)).

    w13 [2I, d/2] / w13s [2I, d/32]; w2 [d, I/2] / w2s [d, I/32]."""
    W13 = dequant_mxfp4(w13, w13s)           # [2I, d]
    I = W13.shape[0] // 2
    g = xf @ W13[:I].T                        # [n, I]
    u = xf @ W13[I:].T
    h = silu(g) * u
    W2 = dequant_mxfp4(w2, w2s)               # [d, I]
    return h @ W2.T                           # [n, d]


def post_expert_norm(y: np.ndarray, norm_w: np.ndarray, eps: float) -> np.ndarray:
    """Per-pick RMSNorm of an expert output (k3 stage E: a norm of each pick's output)."""
    ms = np.mean(y * y, axis=-1, keepdims=True)
    return y / np.sqrt(ms + eps) * np.asarray(norm_w, np.float64)


def experts_combine(xf: np.ndarray, ids: np.ndarray, w: np.ndarray,
                    w13, w13s, w2, w2s, norm_w=None, eps: float = 1e-6,
                    return_y: bool = False):
    """out[t] = sum_j w[t, j] * [norm](y_{t,j}), y_{t,j} = expert ids[t, j] on x[t].

    Experts are dequantised one at a time (k3 stage E: per-pick norm and
    weighted sum).  Summation over j follows the ascending-id pick order."""
    S, k = ids.shape
    d = xf.shape[1]
    y = np.zeros((S, k, d), np.float64)

    def one_expert(e):
        tt, jj = np.nonzero(ids == e)
        y[tt, jj] = expert_ffn(xf[tt], w13[e], w13s[e], w2[e], w2s[e])

    # experts are independent; a thread pool only overlaps their numpy calls
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        list(ex.map(one_expert, np.unique(ids)))
    if norm_w is not None:
        y = post_expert_norm(y, norm_w, eps)
    out = np.zeros((S, d), np.float64)
    for j in range(k):
        out += w[:, j:j + 1] * y[:, j]
    return (out, y) if return_y else out


def moe_forward(inp, tokens: np.ndarray | None = None):
    """The whole block on an ``moe_inputs.MoEInputs``.

    Returns (ids [n, k] int32, w [n, k] fp64, out [n, d] fp64, logits [n, E] fp32)
    for the rows ``tokens`` (default: all rows).  Rows are independent, so a
    subset is evaluated exactly as in the full call."""
    cfg = inp.cfg
    rows = np.arange(cfg.S) if tokens is None else np.asarray(tokens)
    xb = inp.x[rows]
    L = router_logits(xb, inp.w_gate, inp.logit_off)
    ids, w = route(L, inp.bias, cfg.k)
    out = experts_combine(bf16_to_f64(xb), ids, w, inp.w13, inp.w13s, inp.w2, inp.w2s,
                          inp.norm_w if cfg.post_norm else None, cfg.norm_eps)
    return ids, w, out, L


# ----------------------------------------------------------------------------
# the latent-MoE layer around the block (k2 page, K2b: router parts, latent
# parts, route, ug / down, lnorm, up; shared gate/up, its activation, shared
# down; k2_launch w_gate, bias, w_ld, w_sgu, w_sd, w13, w13s, w2, w2s, ln_w,
# w_up, out [S, 7168])
# ----------------------------------------------------------------------------


def dense(xf: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """x [n, K] (fp64) times a bf16 weight [N, K] transposed: [n, N]."""
    return xf @ bf16_to_f64(w_bits).T


def shared_expert(xf: np.ndarray, w_sgu: np.ndarray, w_sd: np.ndarray) -> np.ndarray:
    """The shared expert on rows xf [n, H]: (silu(x Wg^T) * (x Wu^T)) Wd^T, with
    w_sgu = [Wg; Wu] (gate rows first, as w13) and w_sd = Wd [H, SI]."""
    SI = w_sgu.shape[0] // 2
    gu = dense(xf, w_sgu)
    return dense(silu(gu[:, :SI]) * gu[:, SI:], w_sd)


def latent_forward(inp, tokens: np.ndarray | None = None):
    """The latent-MoE layer on a ``moe_inputs.LatentInputs``, in fp64 (fp32
    logits).  Returns (ids, w, out [n, H], logits) for the rows ``tokens``.

      routing  on x (the router parts read the layer input)
      xl       = x . w_ld^T                       (latent parts)
      yl       = sum_j w_j expert_j(xl)            (ug, down: the block at d = LAT)
      zl       = RMSNorm(yl) * ln_w                (lnorm)
      out      = zl . w_up^T + shared_expert(x)   (up; shared gate/up, down)"""
    cfg = inp.cfg
    rows = np.arange(cfg.S) if tokens is None else np.asarray(tokens)
    xb = inp.x[rows]
    L = router_logits(xb, inp.w_gate, inp.logit_off)
    ids, w = route(L, inp.bias, cfg.k)
    xf = bf16_to_f64(xb)
    xl = dense(xf, inp.w_ld)
    yl = experts_combine(xl, ids, w, inp.w13, inp.w13s, inp.w2, inp.w2s)
    zl = post_expert_norm(yl, inp.ln_w, cfg.norm_eps)
    out = dense(zl, inp.w_up)
    if cfg.SI:
        out = out + shared_expert(xf, inp.w_sgu, inp.w_sd)
    return ids, w, out, L


def parity_error(out_gpu: np.ndarray, out_ref: np.ndarray) -> float:
    """max |out - ref| / max |ref| -- the output parity measure."""
    ref = np.asarray(out_ref, np.float64)
    return float(np.max(np.abs(np.asarray(out_gpu, np.float64) - ref)) / np.max(np.abs(ref)))
