"""Pins of the oracle's layer parts (CPU only): bf16 rounding, RMSNorm, the
[out][in] projection, rotate-half RoPE, FP8-cache attention and SiLU.

Each is checked against closed forms with literal numbers, invariants, or a
library routine -- chosen so that a dropped term, a wrong sign or index, a
transposed operand or a wrong scale fails at least one test.
"""
import math

import numpy as np
import torch

import oracle
import synth

COS1, SIN1 = 0.5403023058681398, 0.8414709848078965  # cos(1), sin(1)
LN3 = 1.0986122886681098


# ------------------------------------------------------------------- bf16
def test_bf16_round_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * 10, rng.standard_normal(2000) * 1e-30]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    L = oracle.lib()
    got = np.array([L.oracle_double_to_bf16(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_round_is_nearest_for_doubles():
    rng = np.random.default_rng(2)
    L = oracle.lib()
    for x in rng.standard_normal(3000) * 3:
        b = L.oracle_double_to_bf16(float(x))
        v = L.oracle_bf16_to_double(b)
        up = L.oracle_bf16_to_double(b + 1)
        dn = L.oracle_bf16_to_double(b - 1)
        assert abs(v - x) <= abs(up - x) and abs(v - x) <= abs(dn - x)
    # an exact tie between 1 and the next bf16 (1 + 2^-7) goes to the even one
    assert L.oracle_double_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    assert L.oracle_double_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_closed_form_and_gain():
    one = np.full(2, 0x3F80, dtype=np.uint16)  # bf16 1.0
    two = np.full(2, 0x4000, dtype=np.uint16)  # bf16 2.0
    out = oracle.rmsnorm(np.array([3.0, 4.0]), one, 0.0)
    assert np.allclose(out, [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=1e-15)
    out_eps = oracle.rmsnorm(np.array([3.0, 4.0]), one, 0.5)
    assert np.allclose(out_eps, [3 / math.sqrt(13.0), 4 / math.sqrt(13.0)], rtol=1e-15)
    assert np.allclose(oracle.rmsnorm(np.array([3.0, 4.0]), two, 0.0), 2 * out, rtol=1e-15)


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(3)
    r = rng.standard_normal(4096) * 7
    g = np.full(4096, 0x3F80, dtype=np.uint16)
    out = oracle.rmsnorm(r, g, 0.0)
    assert abs(math.sqrt(np.mean(out ** 2)) - 1.0) < 1e-13
    assert np.allclose(oracle.rmsnorm(r * 1000.0, g, 0.0), out, rtol=1e-13)


# ------------------------------------------------------------- projection
def test_matvec_one_hot_selects_column_of_out_in_matrix():
    rng = np.random.default_rng(4)
    W = synth.f32_to_bf16_bits(rng.standard_normal((7, 13)).astype(np.float32))
    Wf = synth.bf16_bits_to_f32(W).astype(np.float64)
    for j in (0, 5, 12):
        x = np.zeros(13)
        x[j] = 1.0
        assert np.array_equal(oracle.matvec(W, x), Wf[:, j])
    x = rng.standard_normal(13)
    assert np.allclose(oracle.matvec(W, x), Wf @ x, rtol=1e-14, atol=1e-14)


# ------------------------------------------------------------------- RoPE
def test_rope_identity_at_position_zero():
    rng = np.random.default_rng(5)
    v = rng.standard_normal(128)
    assert np.array_equal(oracle.rope(v, 0), v)


def test_rope_rotate_half_pairing_and_frequencies():
    D = 128
    # theta_0 = 1: at pos 1, e_0 -> cos(1) e_0 + sin(1) e_64
    e0 = np.zeros(D); e0[0] = 1.0
    out = oracle.rope(e0, 1)
    exp = np.zeros(D); exp[0] = COS1; exp[64] = SIN1
    assert np.allclose(out, exp, atol=1e-15)
    # e_64 -> -sin e_0 + cos e_64
    e64 = np.zeros(D); e64[64] = 1.0
    out = oracle.rope(e64, 1)
    exp = np.zeros(D); exp[0] = -SIN1; exp[64] = COS1
    assert np.allclose(out, exp, atol=1e-15)
    # theta_32 = 10000^(-64/128) = 0.01: at pos 100 the angle is 1
    e32 = np.zeros(D); e32[32] = 1.0
    out = oracle.rope(e32, 100)
    exp = np.zeros(D); exp[32] = COS1; exp[96] = SIN1
    assert np.allclose(out, exp, atol=1e-12)
    # D = 64: theta_16 = 10000^(-32/64) = 0.01 as well
    e16 = np.zeros(64); e16[16] = 1.0
    out = oracle.rope(e16, 100)
    exp = np.zeros(64); exp[16] = COS1; exp[48] = SIN1
    assert np.allclose(out, exp, atol=1e-12)


def test_rope_norm_and_relative_position():
    rng = np.random.default_rng(6)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for p in (1, 17, 2999):
        assert abs(np.linalg.norm(oracle.rope(q, p)) - np.linalg.norm(q)) < 1e-12
    a = oracle.rope(q, 50) @ oracle.rope(k, 20)
    b = oracle.rope(q, 1030) @ oracle.rope(k, 1000)
    assert abs(a - b) < 1e-10


# -------------------------------------------------------------- attention
def _codes(vals):
    return oracle.e4m3_encode(np.asarray(vals, dtype=np.float32))


def test_attention_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(8)
    D, T = 64, 40
    dec = oracle.e4m3_decode_all()
    krow = _codes(rng.standard_normal(D))
    kc = np.tile(krow, (T, 1))
    ks = np.full(T, 0.37, dtype=np.float32)
    vc = _codes(rng.standard_normal((T, D)) * 20).reshape(T, D)
    vs = (rng.random(T) + 0.5).astype(np.float32)
    q = rng.standard_normal(D) * 3
    for pos in (0, 9, T - 1):
        o = oracle.attention_head(q, kc, ks, vc, vs, pos)
        exp = np.mean(dec[vc[:pos + 1]] * vs[:pos + 1, None].astype(np.float64), axis=0)
        assert np.allclose(o, exp, rtol=1e-13, atol=1e-13)
    # q = 0 gives uniform weights whatever the keys
    kc2 = _codes(rng.standard_normal((T, D))).reshape(T, D)
    o = oracle.attention_head(np.zeros(D), kc2, ks, vc, vs, 9)
    exp = np.mean(dec[vc[:10]] * vs[:10, None].astype(np.float64), axis=0)
    assert np.allclose(o, exp, rtol=1e-13, atol=1e-13)


def test_attention_self_only_at_position_zero_and_ignores_later_slots():
    rng = np.random.default_rng(9)
    D, T = 128, 8
    dec = oracle.e4m3_decode_all()
    kc = _codes(rng.standard_normal((T, D))).reshape(T, D)
    vc = _codes(rng.standard_normal((T, D))).reshape(T, D)
    ks = np.ones(T, dtype=np.float32)
    vs = np.full(T, 0.5, dtype=np.float32)
    kc[1:] = 0x7F  # NaN codes and scales beyond pos must never be read
    vc[1:] = 0x7F
    ks[1:] = np.nan
    vs[1:] = np.nan
    o = oracle.attention_head(rng.standard_normal(D), kc, ks, vc, vs, 0)
    assert np.array_equal(o, dec[vc[0]] * 0.5)


def test_attention_softmax_scale_is_inverse_sqrt_head_dim_and_uses_key_scales():
    # Two slots, D = 64 (sqrt 8).  Slot 0's key is e_0 with code 1.0 and key
    # scale 2; q = 4 ln3 e_0, so its score is 4 ln3 * 2 / 8 = ln 3 against 0
    # for slot 1: weights 3/4 and 1/4.
    D = 64
    dec = oracle.e4m3_decode_all()
    kc = np.zeros((2, D), dtype=np.uint8)
    kc[0, 0] = 0x38
    ks = np.array([2.0, 5.0], dtype=np.float32)
    vc = np.zeros((2, D), dtype=np.uint8)
    vc[0, :] = 0x38   # 1.0
    vc[1, :] = 0x40   # 2.0
    vs = np.array([1.0, 3.0], dtype=np.float32)
    q = np.zeros(D); q[0] = 4 * LN3
    o = oracle.attention_head(q, kc, ks, vc, vs, 1)
    assert np.allclose(o, 0.75 * 1.0 + 0.25 * 2.0 * 3.0, rtol=1e-14)
    assert dec[0x40] == 2.0


def test_attention_single_dominant_key_returns_its_value():
    rng = np.random.default_rng(10)
    D, T = 64, 30
    dec = oracle.e4m3_decode_all()
    kc = np.zeros((T, D), dtype=np.uint8)
    kc[17, 3] = 0x7E  # 448 in dim 3 for slot 17 only
    ks = np.ones(T, dtype=np.float32)
    vc = _codes(rng.standard_normal((T, D))).reshape(T, D)
    vs = (rng.random(T) + 0.1).astype(np.float32)
    q = np.zeros(D); q[3] = 10.0
    o = oracle.attention_head(q, kc, ks, vc, vs, T - 1)
    assert np.allclose(o, dec[vc[17]] * vs[17], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------- SiLU
def test_silu_closed_forms():
    L = oracle.lib()
    assert L.oracle_silu(0.0) == 0.0
    assert abs(L.oracle_silu(LN3) - 0.75 * LN3) < 1e-15
    assert abs(L.oracle_silu(-LN3) - (-0.25 * LN3)) < 1e-15
