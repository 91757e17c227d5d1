"""Seeded synthetic inputs for the routed MXFP4 mixture-of-experts block.

This module is shared by the CPU oracle (``oracle/``) and the CUDA path (tests,
``bench.py``).  It holds the random-number stream, the value distributions and
the storage encodings of the inputs (bf16 bit patterns, packed e2m1 nibbles,
e8m0 scale bytes) -- and none of the block's arithmetic: no router, no top-k,
no dequantisation, no expert math.

Random stream
-------------
Every tensor draws from its own counter-based stream built on SplitMix64
(G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014; the 64-bit finaliser with the constants published there)::

    key(seed, tensor, attempt) = mix(mix(mix(seed + G) + tensor*G) + attempt*G)
    draw(key, i)               = mix(key + (i + 1)*G)        (G = 0x9E3779B97F4A7C15)

All arithmetic is modulo 2**64.  ``attempt`` is only non-zero for rows of x that
were re-drawn to enforce the routing-score gap (see ``attempts`` below).

Distributions (the five workloads in ``CONFIGS``)
-------------------------------------------------
* x ~ N(0, 1), rounded to bf16 (Box-Muller from draws 2i and 2i+1, fp64 ->
  fp32 -> bf16, round to nearest even at each step).
* router weight ``w_gate`` ~ N(0, 1/d), rounded the same way.
* router ``bias`` ~ U(-0.1, 0.1), fp32.
* ``w13`` [E, 2I, d/2] and ``w2`` [E, d, I/2]: uniform random bytes, i.e. both
  e2m1 nibbles uniform over the 16 codes.  Byte j of a row holds K-elements 2j
  (low nibble) and 2j+1 (high nibble).
* ``w13s`` [E, 2I, d/32] and ``w2s`` [E, d, I/32]: e8m0 bytes 127 + U{-6..-2}.
* post-expert norm weight ~ U(0.5, 1.5), fp32 (workload 3 only).
* Zipf(1.1) logit offset (workload 4 only): a seeded random ranking of the
  experts, offset[e] = -1.1 * ln(rank[e]), fp32.

The gap between the k-th and (k+1)-th routing score is enforced by re-drawing
rows of x with a higher ``attempt`` counter.  Which rows need it is decided by
the oracle (it needs the router's arithmetic); the resulting per-row counters
for seed 0 are stored beside this file in ``gap_attempts.json``.
"""
from __future__ import annotations

import json
import math
import os
from dataclasses import dataclass, field

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
MASK64 = (1 << 64) - 1

# tensor ids of the per-tensor streams
T_X, T_W_GATE, T_BIAS, T_W13, T_W13S, T_W2, T_W2S, T_NORM_W, T_ZIPF = range(1, 10)
# the latent-MoE layer's dense weights
T_W_LD, T_W_UP, T_LN_W, T_W_SGU, T_W_SD = range(10, 15)

# e8m0 bytes 127 + U{-6..-2}
SCALE_LO, SCALE_N = 121, 5


@dataclass(frozen=True)
class MoEConfig:
    """One workload: S token rows, hidden d, E experts, top-k, intermediate I."""
    name: str
    S: int
    d: int
    E: int
    k: int
    I: int
    post_norm: bool = False
    zipf: float = 0.0          # Zipf exponent of the per-expert logit offset (0 = none)
    norm_eps: float = 1e-6
    gap: float = 1e-3          # minimum score gap between pick k and pick k+1

    def with_(self, **kw) -> "MoEConfig":
        d = dict(self.__dict__)
        d.update(kw)
        return MoEConfig(**d)


CONFIGS = [
    MoEConfig("tiny", S=8, d=256, E=8, k=2, I=128),
    MoEConfig("verify_latent_s8", S=8, d=4096, E=256, k=8, I=512),
    MoEConfig("verify_s32", S=32, d=4096, E=256, k=8, I=1024),
    MoEConfig("wide_s128_postnorm", S=128, d=7168, E=256, k=8, I=2048, post_norm=True),
    MoEConfig("prefill_s4096_zipf", S=4096, d=7168, E=256, k=8, I=2048, zipf=1.1),
]


# ----------------------------------------------------------------------------
# SplitMix64 counter stream (vectorised, modulo 2**64)
# ----------------------------------------------------------------------------
def _mix_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def _mix_arr(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z *= np.uint64(0xBF58476D1CE4E5B9)
    z ^= z >> np.uint64(27)
    z *= np.uint64(0x94D049BB133111EB)
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, tensor: int, attempt: int = 0) -> int:
    k = _mix_int(seed + GOLDEN)
    k = _mix_int(k + tensor * GOLDEN)
    return _mix_int(k + attempt * GOLDEN)


def draws(key: int, start: int, n: int) -> np.ndarray:
    """Draws start .. start+n-1 of the stream ``key`` as uint64."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + i * np.uint64(GOLDEN)
        return _mix_arr(z)


def uniform01(u: np.ndarray) -> np.ndarray:
    """uint64 draws -> fp64 in [0, 1) from the top 53 bits."""
    return (u >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(key: int, start: int, n: int) -> np.ndarray:
    """n standard normals (Box-Muller, cosine branch) from draws 2i, 2i+1."""
    u = draws(key, 2 * start, 2 * n).reshape(n, 2)
    u1 = 1.0 - uniform01(u[:, 0])           # (0, 1]
    u2 = uniform01(u[:, 1])
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def random_bytes(key: int, byte_start: int, nbytes: int) -> np.ndarray:
    """Bytes byte_start .. byte_start+nbytes-1 of the stream (little-endian draws)."""
    w0 = byte_start // 8
    w1 = (byte_start + nbytes + 7) // 8
    b = draws(key, w0, w1 - w0).astype("<u8").view(np.uint8)
    off = byte_start - 8 * w0
    return b[off:off + nbytes]


# ----------------------------------------------------------------------------
# storage encodings
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern (uint16), round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------
# tensors
# ----------------------------------------------------------------------------
def gen_x(cfg: MoEConfig, seed: int = 0, attempts: np.ndarray | None = None) -> np.ndarray:
    """x [S, d] as bf16 bits.  Row t is drawn from stream (seed, X, attempts[t])."""
    S, d = cfg.S, cfg.d
    att = np.zeros(S, np.int64) if attempts is None else np.asarray(attempts, np.int64)
    z = normal(stream_key(seed, T_X, 0), 0, S * d).astype(np.float32)
    out = f32_to_bf16_bits(z).reshape(S, d)
    redo = np.nonzero(att != 0)[0]
    for t in redo:
        out[t] = gen_x_rows(cfg, seed, np.array([t]), int(att[t]))[0]
    return out


def gen_x_rows(cfg: MoEConfig, seed: int, rows: np.ndarray, attempt: int) -> np.ndarray:
    """Rows ``rows`` of x drawn at ``attempt`` (bf16 bits) -- used by gap enforcement."""
    key = stream_key(seed, T_X, int(attempt))
    out = np.empty((len(rows), cfg.d), np.uint16)
    for i, t in enumerate(rows):
        out[i] = f32_to_bf16_bits(normal(key, int(t) * cfg.d, cfg.d).astype(np.float32))
    return out


def gen_w_gate(cfg: MoEConfig, seed: int = 0) -> np.ndarray:
    z = normal(stream_key(seed, T_W_GATE), 0, cfg.E * cfg.d) / math.sqrt(cfg.d)
    return f32_to_bf16_bits(z.astype(np.float32)).reshape(cfg.E, cfg.d)


def gen_bias(cfg: MoEConfig, seed: int = 0) -> np.ndarray:
    u = uniform01(draws(stream_key(seed, T_BIAS), 0, cfg.E))
    return (-0.1 + 0.2 * u).astype(np.float32)


def gen_logit_offset(cfg: MoEConfig, seed: int = 0) -> np.ndarray | None:
    if not cfg.zipf:
        return None
    order = np.argsort(draws(stream_key(seed, T_ZIPF), 0, cfg.E), kind="stable")
    rank = np.empty(cfg.E, np.int64)
    rank[order] = np.arange(1, cfg.E + 1)
    return (-cfg.zipf * np.log(rank.astype(np.float64))).astype(np.float32)


def gen_norm_w(cfg: MoEConfig, seed: int = 0) -> np.ndarray | None:
    if not cfg.post_norm:
        return None
    u = uniform01(draws(stream_key(seed, T_NORM_W), 0, cfg.d))
    return (0.5 + u).astype(np.float32)


def _gen_packed(key: int, E: int, rows: int, K: int, out: np.ndarray | None) -> np.ndarray:
    per_e = rows * (K // 2)
    if out is None:
        out = np.empty((E, rows, K // 2), np.uint8)
    for e in range(E):
        out[e] = random_bytes(key, e * per_e, per_e).reshape(rows, K // 2)
    return out


def _gen_scales(key: int, E: int, rows: int, K: int, out: np.ndarray | None) -> np.ndarray:
    per_e = rows * (K // 32)
    if out is None:
        out = np.empty((E, rows, K // 32), np.uint8)
    for e in range(E):
        u = draws(key, e * per_e, per_e)
        out[e] = (SCALE_LO + (u % np.uint64(SCALE_N))).astype(np.uint8).reshape(rows, K // 32)
    return out


def gen_w13(cfg: MoEConfig, seed: int = 0, out=None) -> np.ndarray:
    """w13 [E, 2I, d/2] packed e2m1: rows 0..I-1 gate (w1), rows I..2I-1 up (w3)."""
    return _gen_packed(stream_key(seed, T_W13), cfg.E, 2 * cfg.I, cfg.d, out)


def gen_w13s(cfg: MoEConfig, seed: int = 0, out=None) -> np.ndarray:
    return _gen_scales(stream_key(seed, T_W13S), cfg.E, 2 * cfg.I, cfg.d, out)


def gen_w2(cfg: MoEConfig, seed: int = 0, out=None) -> np.ndarray:
    """w2 [E, d, I/2] packed e2m1."""
    return _gen_packed(stream_key(seed, T_W2), cfg.E, cfg.d, cfg.I, out)


def gen_w2s(cfg: MoEConfig, seed: int = 0, out=None) -> np.ndarray:
    return _gen_scales(stream_key(seed, T_W2S), cfg.E, cfg.d, cfg.I, out)


# ----------------------------------------------------------------------------
# stored gap-enforcement counters (written by oracle/gap_tables.py)
# ----------------------------------------------------------------------------
_GAP_FILE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "gap_attempts.json")


def stored_attempts(cfg: MoEConfig, seed: int = 0) -> np.ndarray | None:
    """Per-row attempt counters for (cfg, seed) if the table holds them, else None."""
    if not os.path.exists(_GAP_FILE):
        return None
    with open(_GAP_FILE) as f:
        tab = json.load(f)
    ent = tab.get(f"{cfg.name}/seed{seed}")
    if ent is None or ent["shape"] != [cfg.S, cfg.d, cfg.E, cfg.k]:
        return None
    att = np.zeros(cfg.S, np.int64)
    for r, a in zip(ent["rows"], ent["attempts"]):
        att[r] = a
    return att


@dataclass
class MoEInputs:
    cfg: MoEConfig
    seed: int
    x: np.ndarray                 # [S, d] bf16 bits (uint16)
    w_gate: np.ndarray            # [E, d] bf16 bits
    bias: np.ndarray              # [E] fp32
    logit_off: np.ndarray | None  # [E] fp32
    w13: np.ndarray               # [E, 2I, d/2] uint8
    w13s: np.ndarray              # [E, 2I, d/32] uint8
    w2: np.ndarray                # [E, d, I/2] uint8
    w2s: np.ndarray               # [E, d, I/32] uint8
    norm_w: np.ndarray | None     # [d] fp32
    attempts: np.ndarray = field(default=None)


def make_inputs(cfg: MoEConfig, seed: int = 0, attempts: np.ndarray | None = None,
                use_stored_attempts: bool = True) -> MoEInputs:
    """All inputs of one workload.  ``attempts`` (per row of x) defaults to the
    stored gap table when it covers (cfg, seed), else all zero."""
    if attempts is None and use_stored_attempts:
        attempts = stored_attempts(cfg, seed)
    if attempts is None:
        attempts = np.zeros(cfg.S, np.int64)
    return MoEInputs(
        cfg=cfg, seed=seed,
        x=gen_x(cfg, seed, attempts),
        w_gate=gen_w_gate(cfg, seed),
        bias=gen_bias(cfg, seed),
        logit_off=gen_logit_offset(cfg, seed),
        w13=gen_w13(cfg, seed), w13s=gen_w13s(cfg, seed),
        w2=gen_w2(cfg, seed), w2s=gen_w2s(cfg, seed),
        norm_w=gen_norm_w(cfg, seed),
        attempts=np.asarray(attempts, np.int64),
    )


def expert_weight_bytes(cfg: MoEConfig) -> int:
    """Bytes of one expert's w13 + w2 with their e8m0 scales (3 I d 17/32)."""
    return 3 * cfg.I * cfg.d * 17 // 32


# ----------------------------------------------------------------------------
# the latent-MoE layer around the block (k2 page, K2b)
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class LatentConfig:
    """One latent-MoE layer workload: S tokens of hidden size H, routed on x;
    the routed experts work at the latent width LAT (their d); a shared expert
    of intermediate size SI (0: none)."""
    name: str
    S: int
    H: int
    LAT: int
    E: int
    k: int
    I: int
    SI: int
    zipf: float = 0.0
    norm_eps: float = 1e-6
    gap: float = 1e-3

    def router(self) -> MoEConfig:
        """The routing workload: x [S, H], w_gate [E, H], bias (and the gap)."""
        return MoEConfig(self.name, S=self.S, d=self.H, E=self.E, k=self.k, I=self.I, zipf=self.zipf,
                         norm_eps=self.norm_eps, gap=self.gap)

    def block(self) -> MoEConfig:
        """The routed experts at d = LAT (their w13 / w2 and scales)."""
        return MoEConfig(self.name + "/experts", S=self.S, d=self.LAT, E=self.E, k=self.k, I=self.I,
                         norm_eps=self.norm_eps, gap=self.gap)


LATENT_CONFIGS = [
    LatentConfig("latent_tiny", S=8, H=512, LAT=256, E=8, k=2, I=128, SI=128),
    # the verify-step latent MoE (d = LAT = 4096, I = 512) inside a Kimi-sized
    # layer (H = 7168) with a shared expert of 2 SI = 1536 gate/up rows
    LatentConfig("latent_s8_shared", S=8, H=7168, LAT=4096, E=256, k=8, I=512, SI=768),
]


def _normal_bf16(key: int, n: int, std: float) -> np.ndarray:
    return f32_to_bf16_bits((normal(key, 0, n) * std).astype(np.float32))


@dataclass
class LatentInputs:
    cfg: LatentConfig
    seed: int
    x: np.ndarray                 # [S, H] bf16 bits
    w_gate: np.ndarray            # [E, H] bf16 bits
    bias: np.ndarray              # [E] fp32
    logit_off: np.ndarray | None  # [E] fp32
    w_ld: np.ndarray              # [LAT, H] bf16 bits
    w13: np.ndarray               # [E, 2I, LAT/2] uint8
    w13s: np.ndarray              # [E, 2I, LAT/32] uint8
    w2: np.ndarray                # [E, LAT, I/2] uint8
    w2s: np.ndarray               # [E, LAT, I/32] uint8
    ln_w: np.ndarray              # [LAT] fp32
    w_up: np.ndarray              # [H, LAT] bf16 bits
    w_sgu: np.ndarray | None      # [2 SI, H] bf16 bits (gate rows, then up rows)
    w_sd: np.ndarray | None       # [H, SI] bf16 bits
    attempts: np.ndarray = field(default=None)


def make_latent_inputs(cfg: LatentConfig, seed: int = 0, attempts: np.ndarray | None = None,
                       use_stored_attempts: bool = True) -> LatentInputs:
    """All inputs of one latent layer.  x, w_gate, bias and the Zipf offset are
    the routing workload's (cfg.router()); the experts' tensors those of
    cfg.block(); dense weights ~ N(0, 1/fan-in) in bf16, ln_w ~ U(0.5, 1.5)."""
    r, b = cfg.router(), cfg.block()
    if attempts is None and use_stored_attempts:
        attempts = stored_attempts(r, seed)
    if attempts is None:
        attempts = np.zeros(cfg.S, np.int64)
    H, LAT, SI = cfg.H, cfg.LAT, cfg.SI
    ln_u = uniform01(draws(stream_key(seed, T_LN_W), 0, LAT))
    return LatentInputs(
        cfg=cfg, seed=seed,
        x=gen_x(r, seed, attempts), w_gate=gen_w_gate(r, seed), bias=gen_bias(r, seed),
        logit_off=gen_logit_offset(r, seed),
        w_ld=_normal_bf16(stream_key(seed, T_W_LD), LAT * H, 1.0 / math.sqrt(H)).reshape(LAT, H),
        w13=gen_w13(b, seed), w13s=gen_w13s(b, seed), w2=gen_w2(b, seed), w2s=gen_w2s(b, seed),
        ln_w=(0.5 + ln_u).astype(np.float32),
        w_up=_normal_bf16(stream_key(seed, T_W_UP), H * LAT, 1.0 / math.sqrt(LAT)).reshape(H, LAT),
        w_sgu=_normal_bf16(stream_key(seed, T_W_SGU), 2 * SI * H, 1.0 / math.sqrt(H)).reshape(2 * SI, H)
        if SI else None,
        w_sd=_normal_bf16(stream_key(seed, T_W_SD), H * SI, 1.0 / math.sqrt(SI)).reshape(H, SI) if SI else None,
        attempts=np.asarray(attempts, np.int64),
    )


def latent_dense_bytes(cfg: LatentConfig) -> int:
    """Bytes of the layer's dense bf16 weights: router, latent down, up and the
    shared expert."""
    return 2 * (cfg.E * cfg.H + 2 * cfg.LAT * cfg.H + 3 * cfg.SI * cfg.H)
