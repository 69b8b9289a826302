"""Pins for the oracle's RMSNorm, neox RoPE and cache append (CPU only).

Each test fixes the oracle against mathematics independent of its code:
closed forms, invariants of the definition, or a separately formulated
restatement (RoPE as complex multiplication).  Source of the operation:
InfiniLM PR #585, section "概述 / Summary", item 2 (fused per-head RMSNorm +
full-rotary RoPE on the Qwen3 paged path) and item 1 (BSHD paged cache).
"""

import math
import os

import numpy as np
import pytest

from oracle import (bf16_bits_to_f64, f64_to_bf16_bits, norm_rope_append,
                    rms_norm, rope_neox)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line)
    return rows


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_hand_example():
    # x = (3, 4): mean(x^2) = 12.5; gamma = (1, 2); eps = 0.
    y = rms_norm(np.array([3.0, 4.0]), np.array([1.0, 2.0]), 0.0)
    r = math.sqrt(12.5)
    assert np.allclose(y, [3.0 / r, 8.0 / r], rtol=0, atol=1e-15)


def test_rmsnorm_golden():
    for row in _load_golden("rmsnorm_closed_form.txt"):
        xs, gs, eps, ys = row.split("|")
        x = np.array([float(t) for t in xs.split()])
        g = np.array([float(t) for t in gs.split()])
        y = np.array([float(t) for t in ys.split()])
        assert np.allclose(rms_norm(x, g, float(eps)), y, rtol=1e-14, atol=1e-14)


def test_rmsnorm_unit_gain_rms_closed_form():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 128)) * 3.0
    eps = 1e-6
    y = rms_norm(x, np.ones(128), eps)
    ms = np.mean(x * x, axis=-1)
    assert np.allclose(np.mean(y * y, axis=-1), ms / (ms + eps), rtol=1e-13)


def test_rmsnorm_scale_invariance_and_zero():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 64))
    g = 1 + 0.1 * rng.standard_normal(64)
    assert np.allclose(rms_norm(5.0 * x, g, 0.0), rms_norm(x, g, 0.0), rtol=1e-13)
    z = rms_norm(np.zeros((2, 8)), np.ones(8), 1e-6)
    assert np.all(z == 0.0)


# --------------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 128))
    assert np.array_equal(rope_neox(x, np.zeros(5), 1e6), x)


def test_rope_hand_example_pairs_and_frequencies():
    # D = 4, theta = 100: inv_freq = (1, 100^(-1/2)) = (1, 0.1).
    # neox pairs are (0, 2) and (1, 3).
    x = np.array([1.0, 1.0, 0.0, 0.0])
    y = rope_neox(x, np.array(10.0), 100.0)
    want = [math.cos(10.0), math.cos(1.0), math.sin(10.0), math.sin(1.0)]
    assert np.allclose(y, want, rtol=0, atol=1e-14)
    # rotation direction: (0, 1) in the first pair goes to (-sin, cos)
    y = rope_neox(np.array([0.0, 0.0, 1.0, 0.0]), np.array(10.0), 100.0)
    assert np.allclose(y, [-math.sin(10.0), 0.0, math.cos(10.0), 0.0], atol=1e-14)


def test_rope_golden():
    for row in _load_golden("rope_closed_form.txt"):
        xs, pos, theta, ys = row.split("|")
        x = np.array([float(t) for t in xs.split()])
        y = np.array([float(t) for t in ys.split()])
        assert np.allclose(rope_neox(x, np.array(float(pos)), float(theta)), y,
                           rtol=0, atol=1e-13)


def test_rope_equals_complex_rotation():
    # Independent formulation: z_i = x_i + i x_{i+D/2} multiplied by e^{i a_i}.
    rng = np.random.default_rng(4)
    D = 128
    x = rng.standard_normal((6, D))
    pos = np.array([0, 1, 7, 511, 8195, 32767], np.float64)
    theta = 1e6
    a = pos[:, None] * np.array([theta ** (-(2.0 * i) / D) for i in range(D // 2)])[None, :]
    z = (x[:, : D // 2] + 1j * x[:, D // 2:]) * np.exp(1j * a)
    want = np.concatenate([z.real, z.imag], axis=1)
    assert np.allclose(rope_neox(x, pos, theta), want, rtol=0, atol=1e-11)


def test_rope_norm_and_relative_position():
    rng = np.random.default_rng(5)
    D = 128
    q = rng.standard_normal(D)
    k = rng.standard_normal(D)
    for m, n in [(3, 1), (1000, 17), (32767, 30000)]:
        rq, rk = rope_neox(q, np.array(m), 1e6), rope_neox(k, np.array(n), 1e6)
        # pair norms preserved
        assert np.allclose(rq[: D // 2] ** 2 + rq[D // 2:] ** 2,
                           q[: D // 2] ** 2 + q[D // 2:] ** 2, rtol=1e-12)
        # <R(m) q, R(n) k> depends on m - n only
        d1 = rq @ rk
        d2 = rope_neox(q, np.array(m + 5), 1e6) @ rope_neox(k, np.array(n + 5), 1e6)
        d3 = rope_neox(q, np.array(m - n), 1e6) @ k
        assert abs(d1 - d2) < 1e-9 and abs(d1 - d3) < 1e-9


# ----------------------------------------------------------- fused + append

def _bits(x):
    return f64_to_bf16_bits(np.asarray(x, np.float64))


def _small_case(seed=6, T=5, Hq=4, Hkv=2, D=16, NB=6, bs=4):
    rng = np.random.default_rng(seed)
    q = _bits(rng.standard_normal((T, Hq, D)))
    k = _bits(rng.standard_normal((T, Hkv, D)))
    v = _bits(rng.standard_normal((T, Hkv, D)))
    gq = _bits(1 + 0.1 * rng.standard_normal(D))
    gk = _bits(1 + 0.1 * rng.standard_normal(D))
    pos = np.array([0, 3, 17, 40, 9], np.int64)[:T]
    sentinel = np.uint16(0x7FBF)     # a NaN pattern no computation produces
    kc = np.full((NB, bs, Hkv, D), sentinel, np.uint16)
    vc = np.full((NB, bs, Hkv, D), sentinel, np.uint16)
    return q, k, v, gq, gk, pos, kc, vc, bs


def test_append_places_exactly_the_mapped_slots():
    q, k, v, gq, gk, pos, kc, vc, bs = _small_case()
    NB = kc.shape[0]
    slots = np.array([5, -1, 23, 0, NB * bs], np.int64)   # -1 and NB*bs are skipped
    qh, kc2, vc2, _, _ = norm_rope_append(q, k, v, pos, slots, gq, gk, 1e6, 1e-6, kc, vc, bs)
    written = np.zeros((NB, bs), bool)
    for t, s in enumerate(slots):
        if 0 <= s < NB * bs:
            written[s // bs, s % bs] = True
            assert np.array_equal(vc2[s // bs, s % bs], v[t])          # v unchanged (R8)
    changed_k = np.any(kc2 != kc, axis=(2, 3))
    changed_v = np.any(vc2 != vc, axis=(2, 3))
    assert np.array_equal(changed_k, written)
    assert np.array_equal(changed_v, written)
    # inputs not modified
    assert np.all(kc == np.uint16(0x7FBF))


def test_fused_equals_unfused_chain():
    q, k, v, gq, gk, pos, kc, vc, bs = _small_case(seed=7)
    slots = np.array([1, 2, 3, 4, 5], np.int64)
    qh, kc2, _, k_hat, q_hat = norm_rope_append(q, k, v, pos, slots, gq, gk, 1e6, 1e-6, kc, vc, bs)
    # unfused chain written from the definitions, step by step, per head
    eps = float(np.float32(1e-6))
    for t in range(q.shape[0]):
        for h in range(q.shape[1]):
            x = bf16_bits_to_f64(q[t, h])
            ms = sum(float(a) * float(a) for a in x) / len(x)
            y = x / math.sqrt(ms + eps) * bf16_bits_to_f64(gq)
            D = len(x)
            out = np.empty(D)
            for i in range(D // 2):
                a = float(pos[t]) * (1e6 ** (-2.0 * i / D))
                out[i] = y[i] * math.cos(a) - y[i + D // 2] * math.sin(a)
                out[i + D // 2] = y[i + D // 2] * math.cos(a) + y[i] * math.sin(a)
            assert np.allclose(out, q_hat[t, h], rtol=1e-12, atol=1e-12)
            assert np.array_equal(f64_to_bf16_bits(out), qh[t, h])
        s = slots[t]
        for h in range(k.shape[1]):
            assert np.array_equal(kc2[s // bs, s % bs, h], f64_to_bf16_bits(k_hat[t, h]))


def test_rounding_is_once_after_rope():
    # the stored result is the rounding of the float64 value, not of a
    # value that was rounded to bf16 after the norm
    q, k, v, gq, gk, pos, kc, vc, bs = _small_case(seed=8)
    slots = np.arange(5, dtype=np.int64)
    qh, _, _, _, q_hat = norm_rope_append(q, k, v, pos, slots, gq, gk, 1e6, 1e-6, kc, vc, bs)
    assert np.array_equal(qh, f64_to_bf16_bits(q_hat))
    err = np.abs(bf16_bits_to_f64(qh) - q_hat)
    ulp = np.ldexp(1.0, np.frexp(np.abs(q_hat))[1] - 8)
    assert np.all(err <= 0.5 * ulp + 1e-300)


@pytest.mark.parametrize("pos", [0, 1, 8195, 32767])
def test_fused_output_norm_matches_gain(pos):
    # with unit gain the normalised, rotated head has RMS sqrt(ms/(ms+eps))
    rng = np.random.default_rng(9)
    D = 128
    q = _bits(rng.standard_normal((1, 1, D)))
    ones = _bits(np.ones(D))
    kc = np.zeros((1, 16, 1, D), np.uint16)
    _, _, _, _, q_hat = norm_rope_append(q, q, q, np.array([pos]), np.array([-1]),
                                         ones, ones, 1e6, 1e-6, kc, kc, 16)
    x = bf16_bits_to_f64(q)[0, 0]
    ms = np.mean(x * x)
    eps = float(np.float32(1e-6))
    assert np.isclose(np.mean(q_hat[0, 0] ** 2), ms / (ms + eps), rtol=1e-12)
