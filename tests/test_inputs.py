"""Seeded generator: stream definition, encodings and distributions (CPU)."""
import numpy as np

import moe_inputs as mi


def test_splitmix64_published_outputs():
    # SplitMix64 seeded with 0: the first outputs of the reference generator
    # (Steele, Lea, Flood 2014; the constants of its 64-bit finaliser).
    d = mi.draws(0, 0, 3)
    assert [int(v) for v in d] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_draws_are_counter_based():
    key = mi.stream_key(7, mi.T_W13)
    a = mi.draws(key, 0, 100)
    b = mi.draws(key, 37, 20)
    assert np.array_equal(a[37:57], b)
    rb = mi.random_bytes(key, 5, 11)
    assert np.array_equal(rb, a[:2].astype("<u8").view(np.uint8)[5:16])


def test_bf16_rounding_nearest_even():
    f = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 1.0 + 2**-9], np.float32)
    assert list(mi.f32_to_bf16_bits(f)) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F80]
    assert np.array_equal(mi.bf16_bits_to_f32(np.array([0x3F80, 0xC020], np.uint16)),
                          np.array([1.0, -2.5], np.float32))


def test_distributions_tiny():
    cfg = mi.CONFIGS[0]
    inp = mi.make_inputs(cfg)
    assert inp.x.shape == (8, 256) and inp.w13.shape == (8, 256, 128)
    assert inp.w13s.shape == (8, 256, 8) and inp.w2.shape == (8, 256, 64) and inp.w2s.shape == (8, 256, 4)
    assert set(np.unique(inp.w13s)) <= set(range(121, 126))
    assert np.all((inp.bias >= -0.1) & (inp.bias < 0.1))
    assert inp.logit_off is None and inp.norm_w is None


def test_normal_moments():
    z = mi.normal(mi.stream_key(0, mi.T_X), 0, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01


def test_nibbles_uniform():
    b = mi.random_bytes(mi.stream_key(0, mi.T_W2), 0, 1 << 18)
    nib = np.concatenate([b & 15, b >> 4])
    cnt = np.bincount(nib, minlength=16) / len(nib)
    assert np.all(np.abs(cnt - 1 / 16) < 0.003)


def test_zipf_offsets_and_norm_weight():
    off = mi.gen_logit_offset(mi.CONFIGS[4])
    assert off.shape == (256,) and np.isclose(off.max(), 0.0)
    assert np.allclose(np.sort(-off), 1.1 * np.log(np.arange(1, 257)), atol=1e-5)
    nw = mi.gen_norm_w(mi.CONFIGS[3])
    assert nw.shape == (7168,) and nw.min() >= 0.5 and nw.max() < 1.5


def test_attempts_only_change_their_rows():
    cfg = mi.CONFIGS[1].with_(d=256)
    a0 = mi.gen_x(cfg, 0, np.zeros(cfg.S, np.int64))
    att = np.zeros(cfg.S, np.int64)
    att[3] = 2
    a1 = mi.gen_x(cfg, 0, att)
    assert np.array_equal(np.delete(a0, 3, 0), np.delete(a1, 3, 0))
    assert not np.array_equal(a0[3], a1[3])
