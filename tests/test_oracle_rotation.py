"""Pins for the oracle's Canalized Rotation and Omni-Token Scaling.

Each check ties the oracle to something other than itself: a library
construction of the Hadamard matrix, an independently written radix-2 fast
transform, closed forms (H e0, H H^T = d I) and the invariants the pages state
(orthogonality keeps q.k; scaling gives unit norm and keeps the norm).
Sources: "OScaR: The Occam's Razor for Extreme KV Cache Quantization in LLMs
and Beyond" (reading notes), II. Method, Step One / Step Two.
"""
import math

import numpy as np
import pytest
import scipy.linalg

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth

D = 128


def _fht_radix2(x: np.ndarray) -> np.ndarray:
    """In-place butterfly fast Walsh-Hadamard transform (natural order),
    written independently of the oracle's dense matrix."""
    y = np.array(x, dtype=np.float64, copy=True)
    h = 1
    while h < y.shape[-1]:
        for i in range(0, y.shape[-1], 2 * h):
            a = y[..., i:i + h].copy()
            b = y[..., i + h:i + 2 * h].copy()
            y[..., i:i + h] = a + b
            y[..., i + h:i + 2 * h] = a - b
        h *= 2
    return y / math.sqrt(y.shape[-1])


def _rand_bits(seed, n):
    return synth.gen_bf16(seed, 1, [0], [0], 0, n)[0, 0]


def test_hadamard_matches_scipy_sylvester():
    H = O.sylvester_hadamard(D)
    np.testing.assert_array_equal(H * math.sqrt(D), scipy.linalg.hadamard(D).astype(np.float64))


def test_hadamard_matches_kronecker_power():
    h2 = np.array([[1.0, 1.0], [1.0, -1.0]])
    H = np.array([[1.0]])
    for _ in range(7):
        H = np.kron(H, h2)
    np.testing.assert_array_equal(O.sylvester_hadamard(D) * math.sqrt(D), H)


def test_unnormalised_hadamard_gram_is_d_identity_exactly():
    Hu = np.rint(O.sylvester_hadamard(D) * math.sqrt(D)).astype(np.int64)
    assert set(np.unique(Hu)) == {-1, 1}
    np.testing.assert_array_equal(Hu @ Hu.T, D * np.eye(D, dtype=np.int64))


def test_rotate_q_equals_radix2_fht():
    bits = _rand_bits(11, 16)
    got = O.rotate_q(bits)
    ref = _fht_radix2(O.bf16_to_f64(bits))
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_rotation_round_trip_is_identity():
    bits = _rand_bits(12, 8)
    q = O.bf16_to_f64(bits)
    qr = O.rotate_q(bits)
    np.testing.assert_allclose(qr @ O.sylvester_hadamard(D).T, q, atol=1e-12)


def test_hadamard_of_e0_is_flat():
    e0 = np.zeros(D, dtype=np.uint16)
    e0[0] = 0x3F80  # bf16 1.0
    np.testing.assert_allclose(O.rotate_q(e0), np.full(D, 1 / math.sqrt(D)), atol=1e-15)


def test_joint_rotation_keeps_dot_products():
    q = _rand_bits(13, 32)
    k = _rand_bits(14, 32)
    raw = np.sum(O.bf16_to_f64(q) * O.bf16_to_f64(k), axis=-1)
    rot = np.sum(O.rotate_q(q) * O.rotate_q(k), axis=-1)
    np.testing.assert_allclose(rot, raw, rtol=1e-12, atol=1e-12)


def test_scaling_gives_unit_norm_and_keeps_norm():
    k = synth.gen_bf16(15, 1, [0], [0], 0, 64, chan_factor=synth.channel_factors([5, 38], 20.0),
                       tok_factor=synth.sink_token_factors(1, 0, 64))[0, 0]
    rk = O.rotate_scale_k(k)
    np.testing.assert_allclose(np.linalg.norm(rk.k_hat, axis=-1), 1.0, atol=1e-12)
    # orthogonality: the stored norm is the raw key's norm
    np.testing.assert_allclose(rk.norm, np.linalg.norm(O.bf16_to_f64(k), axis=-1), rtol=1e-12)
    # stored forms are the nearest bf16 / fp16
    kb = O.bf16_to_f64(rk.k_hat_bf16)
    ulp = np.spacing(np.abs(kb).astype(np.float32)).astype(np.float64) * 2 ** 16
    assert np.all(np.abs(kb - rk.k_hat) <= 0.5 * ulp + 1e-300)
    assert np.all(np.abs(rk.norm_f16.astype(np.float64) - rk.norm)
                  <= 0.5 * np.spacing(rk.norm_f16).astype(np.float64))
    # the sink tokens (x0.05) come out at unit norm like the rest
    assert rk.norm[0] < 0.1 * rk.norm[10]


def test_zero_key_keeps_zero():
    rk = O.rotate_scale_k(np.zeros((2, D), dtype=np.uint16))
    assert np.all(rk.k_hat == 0) and np.all(rk.norm == 0)
    assert np.all(rk.k_hat_bf16 == 0)


def test_ablation_flags():
    k = _rand_bits(16, 4)
    kr = O.bf16_to_f64(k)
    no_scale = O.rotate_scale_k(k, O.NO_SCALE)
    np.testing.assert_allclose(no_scale.k_hat, _fht_radix2(kr), atol=1e-12)
    np.testing.assert_array_equal(no_scale.norm, 1.0)
    no_rot = O.rotate_scale_k(k, O.NO_ROTATE)
    np.testing.assert_allclose(no_rot.k_hat, kr / np.linalg.norm(kr, axis=-1, keepdims=True),
                               atol=1e-15)
    both = O.rotate_scale_k(k, O.NO_ROTATE | O.NO_SCALE)
    np.testing.assert_array_equal(both.k_hat_bf16, k)


@pytest.mark.parametrize("x, want", [
    (1.0 + 2.0 ** -8, 0x3F80),                      # tie -> even (1.0)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),                  # tie -> even (1 + 2^-6)
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),         # just above the tie: up
    (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
    (2.0 ** -130, 0x0000 | 0x0008),                 # bf16 subnormal region (exact)
])
def test_f64_to_bf16_direct_rounding(x, want):
    # (1 + 2^-8 + 2^-40) rounds up directly but would tie through fp32.
    assert int(O.f64_to_bf16(np.array([x]))[0]) == want


def test_f64_to_bf16_agrees_with_fp32_rne_on_fp32_values():
    import torch
    x = np.random.default_rng(0).standard_normal(4096).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(O.f64_to_bf16(x.astype(np.float64)), want)


def test_f16_rounding_is_nearest_even():
    got = O.f_to_f16(np.array([1 + 2.0 ** -11, 1 + 2.0 ** -11 + 2.0 ** -30, 1 + 3 * 2.0 ** -11]))
    np.testing.assert_array_equal(got.astype(np.float64), [1.0, 1 + 2.0 ** -10, 1 + 2 * 2.0 ** -10])
