"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in the oracle (monkeypatched for the duration of
the case only) and checks that at least one pin of tests/test_oracle.py fails.
"""
import numpy as np
import pytest

import oracle
import oracle.moe_oracle as M
import test_oracle as T

_ORIG = {n: getattr(M, n) for n in ("dequant_mxfp4", "route", "e2m1_value")}


def _swapped_nibbles(packed, scales):
    p = np.asarray(packed, np.uint8)
    return _ORIG["dequant_mxfp4"](((p >> 4) | (p << 4)).astype(np.uint8), scales)


def _gate_up_swapped(xf, w13, w13s, w2, w2s):
    W13 = M.dequant_mxfp4(w13, w13s)
    I = W13.shape[0] // 2
    g, u = xf @ W13[:I].T, xf @ W13[I:].T
    return (M.silu(u) * g) @ M.dequant_mxfp4(w2, w2s).T


def _w2_transposed_blocks(xf, w13, w13s, w2, w2s):
    W13 = M.dequant_mxfp4(w13, w13s)
    I = W13.shape[0] // 2
    h = M.silu(xf @ W13[:I].T) * (xf @ W13[I:].T)
    W2 = M.dequant_mxfp4(w2, w2s)
    return h @ W2[::-1].T


def _biased_weights(L32, bias, k):
    s, sel = M.routing_scores(L32, bias)
    ids = np.sort(np.argsort(-sel, axis=1, kind="stable")[:, :k], axis=1).astype(np.int32)
    w = np.take_along_axis(sel, ids, 1)
    return ids, w / w.sum(1, keepdims=True)


def _no_renorm(L32, bias, k):
    ids, w = _ORIG["route"](L32, bias, k)
    s, _ = M.routing_scores(L32, bias)
    return ids, np.take_along_axis(s, ids.astype(np.int64), 1)


def _fp32_accumulation(x_bits, w_gate_bits, logit_off=None):
    L = M.bf16_to_f64(x_bits).astype(np.float32) @ M.bf16_to_f64(w_gate_bits).astype(np.float32).T
    if logit_off is not None:
        L = L + logit_off[None, :]
    return L.astype(np.float32)


def _norm_without_weight(y, norm_w, eps):
    return y / np.sqrt(np.mean(y * y, axis=-1, keepdims=True) + eps)


def _e8m0_bias_128(byte):
    b = np.asarray(byte, dtype=np.int64)
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 128))


def _e2m1_subnormal_as_one(code):
    v = _ORIG["e2m1_value"](code)
    c = np.asarray(code)
    return np.where((c & 7) == 1, np.where(c >> 3, -1.0, 1.0), v)


MUTATIONS = {
    "nibble order": ("dequant_mxfp4", _swapped_nibbles),
    "gate/up swapped": ("expert_ffn", _gate_up_swapped),
    "w2 rows reversed": ("expert_ffn", _w2_transposed_blocks),
    "weights from biased score": ("route", _biased_weights),
    "weights not renormalised": ("route", _no_renorm),
    "fp32 logit accumulation": ("router_logits", _fp32_accumulation),
    "norm weight dropped": ("post_expert_norm", _norm_without_weight),
    "e8m0 bias": ("e8m0_value", _e8m0_bias_128),
    "e2m1 subnormal": ("e2m1_value", _e2m1_subnormal_as_one),
}

PINS = [
    T.test_e2m1_table, T.test_e8m0_cases, T.test_dequant_worked_rows,
    T.test_logit_is_exact_sum_rounded_once_to_fp32, T.test_route_closed_form_and_ties,
    T.test_expert_closed_form, T.test_scale_blocks_along_k, T.test_post_norm_closed_form,
    lambda: T.test_brute_force_tiny(False, 0.0), lambda: T.test_brute_force_tiny(True, 0.0),
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    fname, fake = MUTATIONS[name]
    orig = getattr(M, fname)
    monkeypatch.setattr(M, fname, fake)
    monkeypatch.setattr(oracle, fname, fake)
    if fname == "e2m1_value":
        monkeypatch.setattr(M, "_PAIR", np.stack([fake(np.arange(256) & 15), fake(np.arange(256) >> 4)], 1))
    failed = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed.append(getattr(pin, "__name__", "brute"))
    assert failed, f"no pin caught the planted mistake '{name}' in {orig.__name__}"


# ---------------------------------------------------------------------------
# the latent-MoE layer (tests/test_oracle_latent.py's pins)
# ---------------------------------------------------------------------------
import test_oracle_latent as TL  # noqa: E402

_ORIG_L = {n: getattr(M, n) for n in ("dense", "shared_expert")}


def _shared_gate_up_swapped(xf, w_sgu, w_sd):
    SI = w_sgu.shape[0] // 2
    gu = _ORIG_L["dense"](xf, w_sgu)
    return _ORIG_L["dense"](M.silu(gu[:, SI:]) * gu[:, :SI], w_sd)


def _shared_sigmoid(xf, w_sgu, w_sd):
    SI = w_sgu.shape[0] // 2
    gu = _ORIG_L["dense"](xf, w_sgu)
    return _ORIG_L["dense"](M.sigmoid(gu[:, :SI]) * gu[:, SI:], w_sd)


def _shared_dropped(xf, w_sgu, w_sd):
    return np.zeros((xf.shape[0], w_sd.shape[0]))


def _dense_square_transposed(xf, w_bits):
    W = M.bf16_to_f64(w_bits)
    return xf @ W if W.shape[0] == W.shape[1] else xf @ W.T


LATENT_MUTATIONS = {
    "shared gate/up swapped": ("shared_expert", _shared_gate_up_swapped),
    "shared activation sigmoid": ("shared_expert", _shared_sigmoid),
    "shared expert dropped": ("shared_expert", _shared_dropped),
    "projection not transposed": ("dense", _dense_square_transposed),
    "latent norm weight dropped": ("post_expert_norm", _norm_without_weight),
}

LATENT_PINS = [lambda c=c: TL.test_latent_brute_force_tiny(c) for c in TL.BRUTE] + [
    TL.test_permutation_projections_reduce_to_the_block, TL.test_shared_expert_with_zero_gate_adds_nothing,
]


@pytest.mark.parametrize("name", sorted(LATENT_MUTATIONS))
def test_latent_pins_catch_mutation(name, monkeypatch):
    fname, fake = LATENT_MUTATIONS[name]
    monkeypatch.setattr(M, fname, fake)
    monkeypatch.setattr(oracle, fname, fake)
    failed = 0
    for pin in LATENT_PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed, f"no latent pin caught the planted mistake '{name}'"
