"""Pins of the CPU oracle's Llama-3-scaled RoPE and its bf16 rounding (no GPU).

Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "The path of
one inference", step (3): init_rope_frequencies(HEAD_DIM, MAX_SEQ_LEN,
500000, 32, 1, 4, 8192); "What is in the box": the RoPE row (Llama 3
scaling, ropeKernel_llama3).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

D = 64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "llama3_rope_bands.json")


def _base(i, theta=500000.0):
    return theta ** (-(2.0 * i) / D)


def test_band_structure_at_the_pages_arguments():
    inv = oracle.llama3_inv_freq()
    assert inv.shape == (32,)
    for i in range(32):
        lam = 2 * math.pi / _base(i)
        if lam < 8192 / 4:                       # high-frequency band: unchanged
            assert inv[i] == _base(i)
        elif lam > 8192 / 1:                     # low-frequency band: divided by factor 32
            assert inv[i] == _base(i) / 32
        else:                                    # blend band: strictly between
            assert _base(i) / 32 < inv[i] < _base(i)
    assert np.all(np.diff(inv) < 0)


def test_band_values_worked_by_hand():
    """Values worked by hand from the published Llama 3.1 rescaling at the
    pages' arguments (fixture cites its derivation)."""
    g = json.load(open(GOLDEN))
    inv = oracle.llama3_inv_freq()
    for i_str, spec in g["values"].items():
        i = int(i_str)
        assert inv[i] == pytest.approx(spec["inv_freq"], rel=spec["rel_tol"])
    kept = [i for i in range(32) if inv[i] == _base(i)]
    divided = [i for i in range(32) if inv[i] == _base(i) / 32]
    assert kept == g["unchanged"]
    assert divided == g["divided_by_factor"]


def test_blend_endpoints_are_continuous_and_midpoint_is_half():
    two_pi = 2 * math.pi
    f_hi = two_pi / 2048.0            # wavelength exactly original/high
    assert oracle.llama3_scale_freq(f_hi) == pytest.approx(f_hi, rel=1e-15)
    f_lo = two_pi / 8192.0            # wavelength exactly original/low
    assert oracle.llama3_scale_freq(f_lo) == pytest.approx(f_lo / 32, rel=1e-15)
    f_mid = two_pi / (8192.0 / 2.5)   # smoothing weight exactly 1/2
    assert oracle.llama3_scale_freq(f_mid) == pytest.approx(f_mid * (0.5 + 0.5 / 32), rel=1e-14)


def test_factor_one_reduces_to_plain_rope_as_complex_rotation():
    """With factor 1 the rescaling is the identity, and rotate-half RoPE is
    multiplication of x[i] + i*x[i+32] by exp(i * pos * theta^(-2i/64))."""
    rng = np.random.default_rng(1)
    inv = np.array([oracle.llama3_scale_freq(_base(i), factor=1.0) for i in range(32)])
    np.testing.assert_allclose(inv, np.array([_base(i) for i in range(32)]), rtol=1e-15, atol=0)
    for pos in (0, 1, 7, 1000, 32767):
        x = rng.standard_normal(D)
        z = (x[:32] + 1j * x[32:]) * np.exp(1j * pos * inv)
        y = oracle.rope_rotate(x, pos, inv)
        np.testing.assert_allclose(y[:32], z.real, rtol=0, atol=1e-12)
        np.testing.assert_allclose(y[32:], z.imag, rtol=0, atol=1e-12)


def test_position_zero_is_identity_and_norm_is_kept():
    rng = np.random.default_rng(2)
    inv = oracle.llama3_inv_freq()
    x = rng.standard_normal(D)
    assert np.array_equal(oracle.rope_rotate(x, 0, inv), x)
    for pos in (1, 17, 4096, 32768):
        y = oracle.rope_rotate(x, pos, inv)
        assert np.linalg.norm(y) == pytest.approx(np.linalg.norm(x), rel=1e-14)


def test_pairing_and_sign_on_basis_vectors():
    inv = oracle.llama3_inv_freq()
    pos = 3
    for i in (0, 15, 31):
        e = np.zeros(D)
        e[i] = 1.0
        y = oracle.rope_rotate(e, pos, inv)
        assert y[i] == pytest.approx(math.cos(pos * inv[i]), abs=1e-15)
        assert y[i + 32] == pytest.approx(math.sin(pos * inv[i]), abs=1e-15)
        assert np.count_nonzero(y) == 2
        e = np.zeros(D)
        e[i + 32] = 1.0
        y = oracle.rope_rotate(e, pos, inv)
        assert y[i] == pytest.approx(-math.sin(pos * inv[i]), abs=1e-15)
        assert y[i + 32] == pytest.approx(math.cos(pos * inv[i]), abs=1e-15)


def test_rotations_compose():
    rng = np.random.default_rng(4)
    inv = oracle.llama3_inv_freq()
    x = rng.standard_normal(D)
    for a, b in ((3, 5), (100, 2000), (8191, 1)):
        ab = oracle.rope_rotate(oracle.rope_rotate(x, a, inv), b, inv)
        np.testing.assert_allclose(ab, oracle.rope_rotate(x, a + b, inv), rtol=0, atol=1e-11)


def test_float_to_bf16_matches_torch_rounding():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(4000).astype(np.float32),
                        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 65504.0, 3.0e38], dtype=np.float32)])
    ours = oracle.f64_to_bf16(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def _exact_bf16(x: float) -> int:
    """Round a double to bf16 exactly with rational arithmetic (normal range)."""
    if x == 0.0:
        return 0x8000 if math.copysign(1.0, x) < 0 else 0
    sign = 0x8000 if x < 0 else 0
    fx = Fraction(abs(x))
    e = math.floor(math.log2(abs(x)))
    while Fraction(2) ** e > fx:
        e -= 1
    while Fraction(2) ** (e + 1) <= fx:
        e += 1
    ulp = Fraction(2) ** (e - 7)
    q, r = divmod(fx, ulp)
    if r > ulp / 2 or (r == ulp / 2 and q % 2 == 1):
        q += 1
    val = q * ulp
    f = np.float32(float(val))                  # exactly representable
    bits = int(np.array([f]).view(np.uint32)[0]) >> 16
    return sign | (bits & 0x7FFF)


def test_double_to_bf16_is_correctly_rounded_near_ties():
    """Doubles a hair off a bf16 half-way point must round away from the
    tie the way the exact value says (no double rounding through float)."""
    rng = np.random.default_rng(6)
    xs = []
    for _ in range(300):
        hi = int(rng.integers(0x3F00, 0x4100))
        lo = (np.array([hi << 16], dtype=np.uint32).view(np.float32)[0]).astype(np.float64)
        up = (np.array([(hi + 1) << 16], dtype=np.uint32).view(np.float32)[0]).astype(np.float64)
        mid = (lo + up) / 2
        for eps in (-1e-12, 1e-12, 0.0):
            xs.append(mid * (1 + eps))
    xs += list(rng.standard_normal(500) * 3)
    for x in xs:
        assert oracle.f64_to_bf16(np.array([x]))[0] == _exact_bf16(float(x)), x
