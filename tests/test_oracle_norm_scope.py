"""Pins for the oracle's norm-scope and target-norm variants of Omni-Token
Scaling.

* All-heads norm ("OScaR: The Occam's Razor for Extreme KV Cache Quantization
  in LLMs and Beyond" reading notes, II. Method, Notation: the key of token i
  spans all heads, n_i = ||k_i||; Step Two: the norm is taken across all
  heads).  Checked against: the unit total energy of the scaled keys; the
  norm of the raw, unrotated keys over all heads (H is orthogonal, so the
  rotated and raw norms agree; this route never applies H); the per-head
  variant, to which it reduces bit for bit with one head and from which each
  head differs only by the factor ||k_h|| / n_i.
* Target norm (the scaling target that "OScaR：面向大模型及多模态LLM极限KV缓存
  量化的奥卡姆剃刀", 独立分析的弱点 (1), says an appendix ablates): stored norm x
  k_hat reproduces the rotated key whatever the target; a power-of-two target
  leaves every INT2 code unchanged and scales the steps and zeros exactly
  (min-max quantisation is scale-equivariant, and such products are exact).
* End to end: with the whole prompt in the residual window, attention over
  either variant's cache equals plain bf16 attention up to the bf16 / fp16
  rounding of the stored keys and norms (rotation invariance, Step One).
"""
import math

import numpy as np
import pytest

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth

TAU = 1 / math.sqrt(128)
HKV = 4


def _keys(seed, T, Hkv=HKV):
    """[Hkv][T][128] raw keys with outlier channels, sink tokens and heads of
    very different sizes (head h scaled by 4^h), so that the all-heads norm
    differs from every head's own."""
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    tf = synth.sink_token_factors(1, 0, T)
    k = synth.gen_bf16(seed, Hkv, [0], range(Hkv), 0, T, chan_factor=cf, tok_factor=tf)[0]
    x = O.bf16_to_f64(k) * (4.0 ** np.arange(Hkv))[:, None, None]
    return O.f64_to_bf16(x)          # exact: powers of two


@pytest.mark.parametrize("flags", [O.NORM_ALL_HEADS, O.NORM_ALL_HEADS | O.NO_ROTATE])
def test_all_heads_unit_total_energy_and_raw_norm(flags):
    k = _keys(301, 64)
    rk = O.rotate_scale_k(k, flags)
    # every token's scaled keys have unit energy over all heads together
    np.testing.assert_allclose(np.sum(rk.k_hat ** 2, axis=(0, 2)), 1.0, rtol=1e-12)
    # the stored norm is the raw keys' norm over all heads, the same in every head
    raw = np.sqrt(np.sum(O.bf16_to_f64(k) ** 2, axis=(0, 2)))
    for h in range(HKV):
        np.testing.assert_allclose(rk.norm[h], raw, rtol=1e-12)
    assert np.all(rk.norm_f16 == rk.norm_f16[0])


def test_all_heads_relation_to_per_head():
    k = _keys(302, 32)
    allh = O.rotate_scale_k(k, O.NORM_ALL_HEADS)
    own = O.rotate_scale_k(k, 0)
    # k_hat of head h under the all-heads norm = its own unit key x ||k_h|| / n
    ratio = own.norm / allh.norm
    np.testing.assert_allclose(allh.k_hat, own.k_hat * ratio[..., None], rtol=1e-12, atol=1e-300)
    # head norms are 4^h apart, so the small heads are far below unit norm
    assert np.all(np.linalg.norm(allh.k_hat[0], axis=-1) < 0.05)
    # with a single head the two scopes are the same computation
    one = k[:1]
    np.testing.assert_array_equal(O.rotate_scale_k(one, O.NORM_ALL_HEADS).k_hat_bf16,
                                  O.rotate_scale_k(one, 0).k_hat_bf16)
    np.testing.assert_array_equal(O.rotate_scale_k(one, O.NORM_ALL_HEADS).norm_f16,
                                  O.rotate_scale_k(one, 0).norm_f16)


def test_all_heads_zero_token_and_zero_head():
    k = _keys(303, 4)
    k[:, 1, :] = 0                      # token 1 zero in every head
    k[2, 2, :] = 0                      # token 2 zero in head 2 only
    rk = O.rotate_scale_k(k, O.NORM_ALL_HEADS)
    assert np.all(rk.k_hat[:, 1] == 0) and np.all(rk.norm[:, 1] == 0)
    assert np.all(rk.k_hat[2, 2] == 0) and rk.norm[2, 2] > 0
    np.testing.assert_allclose(np.sum(rk.k_hat[:, 2] ** 2), 1.0, rtol=1e-12)


@pytest.mark.parametrize("flags", [0, O.NORM_ALL_HEADS])
@pytest.mark.parametrize("target", [1.0, 0.37, 3.0, 2.0 ** -3])
def test_target_reconstructs_rotated_key(flags, target):
    k = _keys(304, 32)
    rk = O.rotate_scale_k(k, flags, target)
    rotated = O.bf16_to_f64(k) @ O.sylvester_hadamard().T
    np.testing.assert_allclose(rk.norm[..., None] * rk.k_hat, rotated, rtol=1e-12, atol=1e-12)
    if not flags:
        np.testing.assert_allclose(np.linalg.norm(rk.k_hat, axis=-1), target, rtol=1e-12)


@pytest.mark.parametrize("flags", [0, O.NORM_ALL_HEADS])
@pytest.mark.parametrize("j", [-3, 2])
def test_power_of_two_target_keeps_codes(flags, j):
    k = _keys(305, 64)
    base = O.rotate_scale_k(k, flags)
    scaled = O.rotate_scale_k(k, flags, 2.0 ** j)
    np.testing.assert_array_equal(O.bf16_to_f64(scaled.k_hat_bf16),
                                  O.bf16_to_f64(base.k_hat_bf16) * 2.0 ** j)
    np.testing.assert_array_equal(scaled.norm_f16.astype(np.float64),
                                  base.norm_f16.astype(np.float64) * 2.0 ** -j)
    for h in range(HKV):
        a = O.quantize_k(base.k_hat_bf16[h])
        b = O.quantize_k(scaled.k_hat_bf16[h])
        np.testing.assert_array_equal(a.codes, b.codes)
        np.testing.assert_array_equal(b.step16.astype(np.float64),
                                      a.step16.astype(np.float64) * 2.0 ** j)
        np.testing.assert_array_equal(b.zero16.astype(np.float64),
                                      a.zero16.astype(np.float64) * 2.0 ** j)


@pytest.mark.parametrize("flags, target", [(O.NORM_ALL_HEADS, 1.0), (0, 0.37),
                                           (O.NORM_ALL_HEADS, 3.0)])
def test_residual_only_matches_bf16_attention(flags, target):
    T = 80
    k = _keys(306, T)
    v = synth.gen_bf16(307, HKV, [0], range(HKV), 0, T)[0]
    q = synth.gen_bf16(308, HKV, [0], range(HKV), 0, 1)[0, :, 0]
    caches = O.build_row_caches(k, v, 0, flags, target)
    for h, c in enumerate(caches):
        assert c.n_packed == 0 and c.n_res == T
        got = c.decode(O.rotate_q(q[h]), TAU)
        want = O.bf16_attention(q[h][None], k[h], v[h], TAU)
        # stored key = bf16(k_hat) x fp16(norm): relative error per element
        # <= 2^-8 + 2^-11 of the head's own key; first-order softmax bound
        qn = np.linalg.norm(O.bf16_to_f64(q[h]))
        n = np.linalg.norm(O.bf16_to_f64(k[h]), axis=-1).max()
        bound = 2 * TAU * qn * n * (2 ** -8 + 2 ** -11) * np.abs(O.bf16_to_f64(v[h])).max()
        assert np.abs(got - want).max() <= bound


def test_row_caches_stream_like_one_shot():
    """append_row with flush-before-append stores what build_row_caches
    stores for the same tokens (blocks align to 32)."""
    T = 128 + 40
    k = _keys(309, T)
    v = synth.gen_bf16(310, HKV, [0], range(HKV), 0, T)[0]
    P0 = 32
    s = O.build_row_caches(k[:, :P0 + 128], v[:, :P0 + 128], P0, O.NORM_ALL_HEADS, 0.37)
    for t in range(P0 + 128, T):
        O.append_row(s, k[:, t], v[:, t])
    one = O.build_row_caches(k, v, P0 + 128, O.NORM_ALL_HEADS, 0.37)
    for a, b in zip(s, one):
        assert a.n_packed == b.n_packed == P0 + 128 and a.n_res == b.n_res == T - P0 - 128
        np.testing.assert_array_equal(a.packed_k().codes, b.packed_k().codes)
        np.testing.assert_array_equal(a.packed_k().step16, b.packed_k().step16)
        np.testing.assert_array_equal(a.packed_norm16(), b.packed_norm16())
        np.testing.assert_array_equal(np.stack(a.res_k_bf16), np.stack(b.res_k_bf16))
