"""Pins of the CPU oracle against things the pages and the mathematics fix.

Each test checks one oracle function against a closed form, an invariant, a
special case that reduces to a textbook/library routine, brute force on a tiny
input, or the hand-worked values in tests/golden/.  No test re-types the
function it pins.
"""
import cmath
import math
import os
import struct

import numpy as np
import pytest
import scipy.special

from oracle import decoder as od
from workloads import f32_to_bf16_bits, tiny_config

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- bf16 storage
def test_bf16_rounding_hand_values():
    # 1 + 2^-8 is halfway between 1 (0x3F80) and 1 + 2^-7 (0x3F81): ties to even -> 0x3F80
    # 1 + 3*2^-8 is halfway between 0x3F81 and 0x3F82: ties to even -> 0x3F82
    vals = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.5, 0.0, 1 + 2 ** -8 + 2 ** -20])
    want = np.array([0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000, 0x3F81], dtype=np.uint16)
    assert np.array_equal(od.f64_to_bf16_bits(vals), want)
    assert np.array_equal(od.bf16_to_f64(want[:4]), [1.0, 1.0, 1 + 2 ** -6, -2.5])


def test_bf16_rounding_agrees_with_generator_rounding():
    # two independent implementations (frexp/rint vs integer bit rounding) on float32 inputs
    r = np.random.default_rng(1)
    x = (r.standard_normal(100000) * 10.0 ** r.integers(-8, 8, 100000)).astype(np.float32)
    assert np.array_equal(od.f64_to_bf16_bits(x.astype(np.float64)), f32_to_bf16_bits(x))


# ----------------------------------------------------------------- int4 dequant
def _bf16_py(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def test_dequant_brute_force_tiny():
    r = np.random.default_rng(2)
    N, K, g = 3, 256, 128
    q = r.integers(0, 16, (N, K), dtype=np.uint8)
    s = f32_to_bf16_bits(r.uniform(0.002, 0.02, (N, K // g)).astype(np.float32))
    z = f32_to_bf16_bits((r.standard_normal((N, K // g)) * 0.005).astype(np.float32))
    W = od.dequant_int4(q, s, z, g)
    for n in range(N):
        for k in range(K):
            want = (int(q[n, k]) - 8) * _bf16_py(s[n, k // g]) + _bf16_py(z[n, k // g])
            assert W[n, k] == pytest.approx(want, rel=0, abs=1e-15)


def test_int4_linear_special_cases():
    N, K, g = 4, 256, 128
    s = f32_to_bf16_bits(np.full((N, K // g), 0.5, np.float32))
    zero = np.zeros((N, K // g), np.uint16)
    x = np.random.default_rng(3).standard_normal((2, K))
    # q = 8, z = 0 -> W = 0 -> y = 0
    q = np.full((N, K), 8, np.uint8)
    assert np.all(od.int4_linear(x, q, s, zero, g) == 0.0)
    # one code 9 at (n, k) -> y[:, n] = x[:, k] * s
    q2 = q.copy()
    q2[2, 130] = 9
    y = od.int4_linear(x, q2, s, zero, g)
    assert np.allclose(y[:, 2], 0.5 * x[:, 130]) and np.all(y[:, [0, 1, 3]] == 0)
    # a one-hot input selects column k of W
    r = np.random.default_rng(4)
    q3 = r.integers(0, 16, (N, K), dtype=np.uint8)
    z3 = f32_to_bf16_bits((r.standard_normal((N, K // g)) * 0.005).astype(np.float32))
    e = np.zeros((1, K))
    e[0, 200] = 1.0
    col = od.int4_linear(e, q3, s, z3, g)[0]
    assert np.allclose(col, (q3[:, 200].astype(float) - 8) * 0.5 + od.bf16_to_f64(z3[:, 1]))


# ----------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_vector_closed_form():
    c, eps = 3.0, 1e-6
    w = f32_to_bf16_bits(np.array([1.0, 2.0, 0.5, -1.0], np.float32))
    out = od.rmsnorm(np.full(4, c), w, eps)
    assert np.allclose(out, c / math.sqrt(c * c + eps) * np.array([1.0, 2.0, 0.5, -1.0]), rtol=1e-15)


def test_rmsnorm_unit_rms_and_scale_invariance():
    x = np.random.default_rng(5).standard_normal((3, 64))
    ones = f32_to_bf16_bits(np.ones(64, np.float32))
    y = od.rmsnorm(x, ones, 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-14)
    assert np.allclose(od.rmsnorm(7.5 * x, ones, 0.0), y, rtol=1e-13)


# ----------------------------------------------------------------- M-RoPE
def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "mrope_d6_theta8.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            p = line.split()
            rows.append((p[0], [int(v) for v in p[1:4]], [float(v) for v in p[4:10]],
                         [float(v) for v in p[10:16]]))
    return rows


@pytest.mark.parametrize("case", _golden_rows(), ids=lambda c: c[0])
def test_mrope_hand_worked(case):
    _, pos, x, want = case
    out = od.mrope(np.array(x), pos, head_dim=6, theta=8.0, sections=(1, 1, 1))
    assert np.allclose(out, want, rtol=0, atol=1e-12)


def _mrope_complex(x, pos, d, theta, sections):
    """Independent formulation: pair (x_i, x_{i+d/2}) as x_i + j x_{i+d/2}, times e^{j angle}."""
    axes = [0] * sections[0] + [1] * sections[1] + [2] * sections[2]
    out = np.empty(d)
    for i in range(d // 2):
        zc = complex(x[i], x[i + d // 2]) * cmath.exp(1j * pos[axes[i]] * theta ** (-2.0 * i / d))
        out[i], out[i + d // 2] = zc.real, zc.imag
    return out


def test_mrope_matches_complex_rotation_distinct_axes():
    r = np.random.default_rng(6)
    d, sections = 128, (16, 24, 24)
    for pos in ([5, 900, 37], [0, 0, 1], [1023, 512, 7]):
        x = r.standard_normal(d)
        assert np.allclose(od.mrope(x, pos, d, 1e6, sections), _mrope_complex(x, pos, d, 1e6, sections),
                           rtol=0, atol=1e-12)


def test_mrope_equal_ids_is_1d_rope_and_norm_preserving():
    r = np.random.default_rng(7)
    d = 64
    x = r.standard_normal((3, d))
    out = od.mrope(x, [41, 41, 41], d, 1e6, (8, 12, 12))
    for h in range(3):
        ref = _mrope_complex(x[h], [41, 41, 41], d, 1e6, (32, 0, 0))   # 1-D RoPE: every freq on one axis
        assert np.allclose(out[h], ref, atol=1e-12)
    pair_norm = lambda v: v[..., :d // 2] ** 2 + v[..., d // 2:] ** 2
    assert np.allclose(pair_norm(out), pair_norm(x), rtol=1e-13)
    assert np.array_equal(od.mrope(x, [0, 0, 0], d, 1e6, (8, 12, 12)), x)


# ----------------------------------------------------------------- attention
def test_attention_single_token_returns_v():
    r = np.random.default_rng(8)
    q = r.standard_normal((4, 16))
    K = r.standard_normal((2, 1, 16))
    V = r.standard_normal((2, 1, 16))
    out = od.decode_attention(q, K, V)
    assert np.allclose(out, V[[0, 0, 1, 1], 0], rtol=1e-15)


def test_attention_equal_keys_mean_of_v_and_gqa_mapping():
    r = np.random.default_rng(9)
    q = r.standard_normal((4, 8))
    K = np.repeat(r.standard_normal((2, 1, 8)), 5, axis=1)    # 5 identical keys per KV head
    V = r.standard_normal((2, 5, 8))
    out = od.decode_attention(q, K, V)
    assert np.allclose(out, V.mean(axis=1)[[0, 0, 1, 1]], rtol=1e-13)


def test_attention_matches_library_softmax():
    r = np.random.default_rng(10)
    q = r.standard_normal((16, 128))
    K = r.standard_normal((8, 37, 128))
    V = r.standard_normal((8, 37, 128))
    out = od.decode_attention(q, K, V)
    for i in range(16):
        p = scipy.special.softmax(K[i // 2] @ q[i] / math.sqrt(128))
        assert math.isclose(p.sum(), 1.0, rel_tol=1e-14)
        assert np.allclose(out[i], p @ V[i // 2], rtol=1e-12)


def test_lse_merge_of_splits_equals_single_pass():
    r = np.random.default_rng(11)
    q = r.standard_normal((2, 64))
    K = r.standard_normal((1, 50, 64)) * 2
    V = r.standard_normal((1, 50, 64))
    full = od.decode_attention(q, K, V)
    for cuts in ([0, 50], [0, 17, 50], [0, 1, 2, 30, 49, 50]):
        outs, lses = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            sc = q @ K[0, a:b].T / 8.0
            lses.append(scipy.special.logsumexp(sc, axis=-1))
            outs.append(od.decode_attention(q, K[:, a:b], V[:, a:b]))
        assert np.allclose(od.merge_partials(outs, lses), full, rtol=1e-12, atol=1e-14)


def test_attention_lse_matches_library_logsumexp():
    r = np.random.default_rng(13)
    q = r.standard_normal((4, 32))
    K = r.standard_normal((2, 23, 32)) * 3
    V = r.standard_normal((2, 23, 32))
    out, lse = od.attention_with_lse(q, K, V)
    assert np.allclose(out, od.decode_attention(q, K, V), rtol=1e-14)
    for i in range(4):
        assert math.isclose(lse[i], scipy.special.logsumexp(K[i // 2] @ q[i] / math.sqrt(32)), rel_tol=1e-14)


@pytest.mark.parametrize("P,T", [(0, 5), (1, 1), (400, 100), (37, 3)])
def test_cascade_equals_attention_over_the_concatenation(P, T):
    """The pages' claim: prefix + suffix + LSE merge is mathematically single-pass attention
    over [prefix; suffix] (here in float64, so equal to rounding)."""
    r = np.random.default_rng(14 + P)
    q = r.standard_normal((16, 128))
    Kp, Vp = r.standard_normal((8, P, 128)), r.standard_normal((8, P, 128))
    Ks, Vs = r.standard_normal((8, T, 128)), r.standard_normal((8, T, 128))
    full = od.decode_attention(q, np.concatenate([Kp, Ks], axis=1), np.concatenate([Vp, Vs], axis=1))
    assert np.allclose(od.cascade_attention(q, Kp, Vp, Ks, Vs), full, rtol=1e-11, atol=1e-13)


def test_cascade_dominant_part_wins():
    """A prefix whose scores dwarf the suffix's returns the prefix's attention (and vice
    versa): the merge weights are exp(lse_part - max lse)."""
    r = np.random.default_rng(15)
    q = np.ones((2, 16))
    Kp = np.full((1, 3, 16), 4.0)
    Vp = r.standard_normal((1, 3, 16))
    Ks = np.full((1, 2, 16), -4.0)
    Vs = r.standard_normal((1, 2, 16))
    out = od.cascade_attention(q, Kp, Vp, Ks, Vs)
    assert np.allclose(out, Vp[0].mean(axis=0), rtol=1e-12)
    out = od.cascade_attention(q, Ks, Vs, Kp, Vp)
    assert np.allclose(out, Vp[0].mean(axis=0), rtol=1e-12)


# ----------------------------------------------------------------- argmax
def test_argmax_lowest_index_and_nan():
    assert od.argmax_lowest(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    assert od.argmax_lowest(np.array([np.nan, 1.0, np.nan, 0.5])) == 1
    assert od.argmax_lowest(np.array([-np.inf, -np.inf])) == 0
    r = np.random.default_rng(12)
    for _ in range(20):
        v = r.standard_normal(1000)
        assert od.argmax_lowest(v) == int(np.argmax(v))


def test_silu_closed_form():
    x = np.array([-3.0, 0.0, 2.0])
    assert np.allclose(od.silu(x), x * scipy.special.expit(x), rtol=1e-15)


def test_attention_is_invariant_to_permuting_cached_positions_and_linear_in_v():
    """softmax(q K^T / sqrt(d)) V does not depend on the order of the cached positions (K and V
    permuted together) and is linear in V — a K/V index mix-up or a stray nonlinearity breaks
    one of them."""
    r = np.random.default_rng(21)
    nq, nkv, d, T = 4, 2, 16, 37
    q = r.standard_normal((nq, d))
    K = r.standard_normal((nkv, T, d))
    V = r.standard_normal((nkv, T, d))
    V2 = r.standard_normal((nkv, T, d))
    out = od.decode_attention(q, K, V)
    perm = r.permutation(T)
    assert np.allclose(od.decode_attention(q, K[:, perm], V[:, perm]), out, rtol=1e-12, atol=1e-14)
    assert not np.allclose(od.decode_attention(q, K[:, perm], V), out)          # permuting V alone matters
    lin = od.decode_attention(q, K, 2.5 * V - 0.75 * V2)
    assert np.allclose(lin, 2.5 * out - 0.75 * od.decode_attention(q, K, V2), rtol=1e-12, atol=1e-13)


def test_int4_linear_is_linear_in_x():
    r = np.random.default_rng(22)
    N, K = 24, 256
    q = r.integers(0, 16, (N, K), dtype=np.uint8)
    s = od.f64_to_bf16_bits(r.uniform(0.002, 0.02, (N, K // 128)))
    z = od.f64_to_bf16_bits(r.normal(0, 0.005, (N, K // 128)))
    x1, x2 = r.standard_normal((2, K)), r.standard_normal((2, K))
    y = od.int4_linear(1.5 * x1 - 2.0 * x2, q, s, z, 128)
    assert np.allclose(y, 1.5 * od.int4_linear(x1, q, s, z, 128) - 2.0 * od.int4_linear(x2, q, s, z, 128),
                       rtol=1e-12, atol=1e-12)
