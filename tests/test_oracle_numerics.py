"""Pins of the oracle's arithmetic: bf16 rounding, RoPE, attention.

Each check is tied to something other than the oracle itself: a library
routine (torch's fp32->bf16 cast, torch's scaled_dot_product_attention),
textbook constants, closed forms of softmax, or brute force."""
import math

import numpy as np
import pytest
import torch

from oracle import ff_oracle as fo


# ---------------------------------------------------------------- bf16 -----

def test_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000),
                        rng.standard_normal(1000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = fo.f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(ref, got)


def test_bf16_single_rounding_from_fp64():
    # 1 + 2^-8 + 2^-30: one rounding gives 1 + 2^-7; rounding through fp32 first
    # would drop 2^-30 and then tie to even at 1.0.
    v = np.array([1 + 2.0 ** -8 + 2.0 ** -30, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8 + 2.0 ** -30)])
    assert list(fo.f64_to_bf16_bits(v)) == [0x3F81, 0x3F80, 0x3F82, 0xBF81]


def test_bf16_overflow_and_subnormal():
    v = np.array([3.4e38, -3.4e38, fo.BF16_MAX, 2.0 ** -130, 2.0 ** -133, 2.0 ** -134,
                  1.5 * 2.0 ** -134, 0.0, -0.0, np.inf])
    assert list(fo.f64_to_bf16_bits(v)) == [0x7F80, 0xFF80, 0x7F7F, 0x0008, 0x0001, 0x0000,
                                            0x0001, 0x0000, 0x8000, 0x7F80]


def test_bf16_roundtrip_all_patterns():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = fo.bf16_bits_to_f64(b)
    ok = ~np.isnan(v)
    assert np.array_equal(fo.f64_to_bf16_bits(v[ok]), b[ok])


# ---------------------------------------------------------------- RoPE -----

def test_rope_split():
    assert fo.rope_axis_dims(128) == (44, 42, 42)
    assert fo.rope_axis_dims(64) == (24, 20, 20)
    ax = fo.rope_pair_axis(128)
    assert ax[21] == (0, 21, 44) and ax[22] == (1, 0, 42) and ax[43] == (2, 0, 42) and ax[63] == (2, 20, 42)


def _rand_bits(shape, seed):
    x = np.random.default_rng(seed).standard_normal(shape)
    return fo.f64_to_bf16_bits(x)


def test_rope_origin_is_identity():
    k = _rand_bits((16, 3, 128), 2)
    pos = np.zeros((16, 3), np.int64)
    assert np.array_equal(fo.rope_k_bits(k, pos, 128, 10000.0), k)


def test_rope_textbook_values_and_sign():
    # pair 0 (time axis, j = 0, omega = 1) at t = 1: angle 1 rad.
    cos1, sin1 = 0.5403023058681398, 0.8414709848078965
    x = np.zeros((2, 1, 128))
    x[0, 0, 0] = 1.0          # (1, 0) -> (cos 1, sin 1)
    x[1, 0, 1] = 1.0          # (0, 1) -> (-sin 1, cos 1)
    pos = np.array([[1, 0, 0], [1, 0, 0]])
    c, s = fo.rope_cos_sin(pos, 128, 10000.0)
    y = fo.rope_rotate_f64(x, c, s)
    assert y[0, 0, 0] == pytest.approx(cos1, abs=1e-16) and y[0, 0, 1] == pytest.approx(sin1, abs=1e-16)
    assert y[1, 0, 0] == pytest.approx(-sin1, abs=1e-16) and y[1, 0, 1] == pytest.approx(cos1, abs=1e-16)


def test_rope_axes_and_frequencies():
    x = np.random.default_rng(3).standard_normal((3, 1, 128))
    pos = np.array([[0, 1, 0], [0, 0, 1], [1, 0, 0]])
    c, s = fo.rope_cos_sin(pos, 128, 10000.0)
    y = fo.rope_rotate_f64(x, c, s)
    moved = [np.flatnonzero(np.abs(y[r, 0] - x[r, 0]) > 0) // 2 for r in range(3)]
    assert set(moved[0]) == set(range(22, 43))       # y axis -> pairs 22..42
    assert set(moved[1]) == set(range(43, 64))       # x axis -> pairs 43..63
    assert set(moved[2]) == set(range(0, 22))        # t axis -> pairs 0..21
    # frequency of time pair j: theta^(-2j/44); pair 5 at t = 1 -> exp(-ln(1e4) * 10 / 44)
    ang = math.exp(-math.log(10000.0) * 10 / 44)
    assert c[2, 5] == pytest.approx(math.cos(ang), abs=1e-15)
    assert s[2, 5] == pytest.approx(math.sin(ang), abs=1e-15)
    # row pair 22 + 3 at y = 1 -> exp(-ln(1e4) * 6 / 42)
    ang = math.exp(-math.log(10000.0) * 6 / 42)
    assert s[0, 25] == pytest.approx(math.sin(ang), abs=1e-15)


def test_rope_preserves_pair_norm():
    x = np.random.default_rng(4).standard_normal((50, 2, 64))
    pos = np.random.default_rng(5).integers(0, 300, (50, 3))
    c, s = fo.rope_cos_sin(pos, 64, 10000.0)
    y = fo.rope_rotate_f64(x, c, s)
    n0 = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n1 = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.allclose(n0, n1, rtol=1e-13, atol=1e-13)


def test_rope_relative_position():
    # <R_m q, R_n k> depends only on m - n (per axis).
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    m, n, r = np.array([[7, 3, 11]]), np.array([[2, 9, 4]]), np.array([[1, 2, 3]])

    def dot(a, b):
        ca, sa = fo.rope_cos_sin(a, 128, 10000.0)
        cb, sb = fo.rope_cos_sin(b, 128, 10000.0)
        return float(np.sum(fo.rope_rotate_f64(q, ca, sa) * fo.rope_rotate_f64(k, cb, sb)))

    assert dot(m, n) == pytest.approx(dot(m - r, n - r), abs=1e-12)
    assert dot(m, n) != pytest.approx(dot(m, n + 1), abs=1e-6)


# ----------------------------------------------------------- attention -----

def _qkv(nq, nk, h, d, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((nq, h, d)), rng.standard_normal((nk, h, d)), rng.standard_normal((nk, h, d))


def test_attention_matches_torch_sdpa():
    q, k, v = _qkv(37, 53, 3, 64, 7)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).permute(1, 0, 2), torch.from_numpy(k).permute(1, 0, 2),
        torch.from_numpy(v).permute(1, 0, 2)).permute(1, 0, 2).numpy()
    assert np.allclose(fo.attention_f64(q, k, v), ref, atol=1e-12, rtol=0)


def test_attention_identical_keys_give_mean_v():
    q, k, v = _qkv(9, 17, 2, 64, 8)
    k[:] = k[0]
    o = fo.attention_f64(q, k, v)
    assert np.allclose(o, v.mean(axis=0, keepdims=True), atol=1e-12, rtol=0)


def test_attention_single_key_and_row_sums():
    q, k, v = _qkv(5, 1, 2, 64, 9)
    assert np.allclose(fo.attention_f64(q, k, v), np.broadcast_to(v, (5, 2, 64)), atol=1e-15)
    q, k, v = _qkv(5, 40, 2, 64, 10)
    assert np.allclose(fo.attention_f64(q, k, np.ones_like(v)), 1.0, atol=1e-14)


def test_attention_key_permutation_invariance():
    q, k, v = _qkv(6, 30, 2, 64, 11)
    p = np.random.default_rng(12).permutation(30)
    assert np.allclose(fo.attention_f64(q, k, v), fo.attention_f64(q, k[p], v[p]), atol=1e-13)


def test_attention_duplicate_keys_shift_logit_by_log_n():
    # gist.science summary of FAST-AR, TempCache, Lemma 5.1: n identical keys with averaged
    # values behave as one key whose logit is raised by ln n.
    q, k, v = _qkv(4, 10, 1, 64, 13)
    n = 3
    k_dup = np.concatenate([k, np.repeat(k[:1], n - 1, axis=0)])
    v_dup = np.concatenate([v, np.repeat(v[:1], n - 1, axis=0)])
    o_dup = fo.attention_f64(q, k_dup, v_dup)
    logits = (q[:, 0] @ k[:, 0].T) / 8.0
    logits[:, 0] += math.log(n)
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    w /= w.sum(axis=1, keepdims=True)
    assert np.allclose(o_dup[:, 0], w @ v[:, 0], atol=1e-13)


def test_attention_bruteforce_agrees():
    q, k, v = _qkv(6, 11, 2, 16, 14)
    bf = np.array(fo.attention_bruteforce(q.tolist(), k.tolist(), v.tolist()))
    assert np.allclose(fo.attention_f64(q, k, v), bf, atol=1e-12, rtol=0)
