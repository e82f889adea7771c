"""Pins for the oracle's decode attention over the packed + residual cache.

* closed-form softmax on a hand-built case (tests/golden/attention_closed_form.json);
* a lossless special case: with both ablation flags on and every quantisation
  group holding only the levels {-1.5, -0.5, 0.5, 1.5} (both extremes
  present), INT2 storage is exact, so the cache's attention must equal plain
  attention on the same bf16 K, V;
* rotation invariance with an empty packed region ("OScaR: The Occam's Razor
  for Extreme KV Cache Quantization in LLMs and Beyond", II. Method, Step One:
  the two rotations cancel in q.k) up to the stated bf16/fp16 rounding;
* the flush invariant: streaming appends with flush-before-append give the
  same packed codes as quantising the same prefix in one go (news article on
  arXiv 2605.19660, 三: the residual cache is batch-quantised every 128 tokens).
"""
import json
import math
import os

import numpy as np

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")
TAU = 1 / math.sqrt(128)


def test_closed_form_softmax():
    with open(os.path.join(GOLD, "attention_closed_form.json")) as f:
        g = json.load(f)
    q = np.zeros((1, 128))
    q[0, 0] = math.sqrt(128)                      # tau * q.k == k[0]
    keys = np.zeros((3, 128))
    keys[:, 0] = [math.log(w) for w in g["weights_unnormalised"]]
    vals = np.zeros((3, 128))
    for i, row in enumerate(g["values_first4"]):
        vals[i, :4] = row
    o = O.attention(q, keys, vals, TAU)
    np.testing.assert_allclose(o[0, :4], g["expected_first4"], rtol=0, atol=1e-15)
    assert np.all(o[0, 4:] == 0)


def test_dequant_worked_examples():
    q = O.QuantK(codes=np.array([[2] + [0] * 127] * 32, np.uint8),
                 step16=np.full((1, 128), 0.5, np.float16),
                 zero16=np.full((1, 128), -1.0, np.float16))
    k = O.dequant_k(q, np.full(32, 3.0, np.float16))
    assert k[0, 0] == 0.0 and k[0, 1] == -3.0
    v = O.dequant_v(O.QuantV(np.array([[3, 1] + [0] * 126], np.uint8),
                             np.array([0.25], np.float16), np.array([-0.5], np.float16)))
    assert v[0, 0] == 0.25 and v[0, 1] == -0.25 and v[0, 2] == -0.5


def _lossless_kv(T, seed):
    """K, V whose every group holds only {-1.5, -0.5, 0.5, 1.5} and both ends."""
    lv = np.array([-1.5, -0.5, 0.5, 1.5])
    r = synth.splitmix64(seed, np.arange(2 * T * 128)).reshape(2, T, 128)
    k = lv[(r[0] % np.uint64(4)).astype(np.int64)]
    v = lv[(r[1] % np.uint64(4)).astype(np.int64)]
    k[0::32, :] = -1.5                 # every (block, channel) group spans the range
    k[1::32, :] = 1.5
    v[:, 0], v[:, 1] = -1.5, 1.5       # every token group spans the range
    return O.f64_to_bf16(k), O.f64_to_bf16(v)


def test_lossless_special_case_equals_plain_attention():
    flags = O.NO_ROTATE | O.NO_SCALE
    T, P = 1024 + 200, 1024 - 64
    k, v = _lossless_kv(T, 21)
    q = synth.gen_bf16(22, 4, [0], [0, 1, 2, 3], 0, 1)[0, :, 0]
    c = O.HeadCache(flags=flags)
    c.quantize_prefix(k[:P], v[:P])
    for t in range(P, T):
        c.append(k[t], v[t])
    assert c.n_packed > P          # some flushes happened
    keys, vals = c.keys_values()
    np.testing.assert_array_equal(keys, O.bf16_to_f64(k))
    np.testing.assert_array_equal(vals, O.bf16_to_f64(v))
    got = c.decode(O.rotate_q(q, flags), TAU)
    want = O.bf16_attention(q, k, v, TAU)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_residual_only_matches_bf16_attention_up_to_rounding():
    T = 96
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    k = synth.gen_bf16(31, 1, [0], [0], 0, T, chan_factor=cf,
                       tok_factor=synth.sink_token_factors(1, 0, T))[0, 0]
    v = synth.gen_bf16(32, 1, [0], [0], 0, T, tok_factor=synth.sink_token_factors(1, 0, T))[0, 0]
    q = synth.gen_bf16(33, 1, [0], [0], 0, 2)[0, 0]
    c = O.build_head_cache(k[:T], v[:T], n_packed=0)
    assert c.n_packed == 0 and c.n_res == T
    got = c.decode(O.rotate_q(q), TAU)
    want = O.bf16_attention(q, k, v, TAU)
    # Only the bf16 key and fp16 norm rounding differ: |d score| <= tau*|q|*n*(2^-8 + 2^-11)
    # and the output moves by at most 2*max|d score|*max|v| (first-order softmax bound).
    qn = np.linalg.norm(O.bf16_to_f64(q), axis=-1).max()
    n = np.linalg.norm(O.bf16_to_f64(k), axis=-1).max()
    bound = 2 * TAU * qn * n * (2 ** -8 + 2 ** -11) * np.abs(O.bf16_to_f64(v)).max()
    assert np.abs(got - want).max() <= bound


def test_streaming_flush_equals_one_shot_prefix():
    T = 3 * 128 + 17
    k = synth.gen_bf16(41, 1, [0], [0], 0, T)[0, 0]
    v = synth.gen_bf16(42, 1, [0], [0], 0, T)[0, 0]
    s = O.HeadCache()
    for t in range(T):
        s.append(k[t], v[t])
    P = 128 * ((T - 1) // 128)
    assert s.n_packed == P and s.n_res == T - P and 1 <= s.n_res <= 128
    one = O.build_head_cache(k[:P + 0], v[:P], n_packed=P)
    a, b = s.packed_k(), one.packed_k()
    np.testing.assert_array_equal(a.codes, b.codes)
    np.testing.assert_array_equal(a.step16, b.step16)
    np.testing.assert_array_equal(a.zero16, b.zero16)
    np.testing.assert_array_equal(s.packed_norm16(), one.packed_norm16())
    np.testing.assert_array_equal(s.packed_v().codes, one.packed_v().codes)


def test_empty_cache_and_single_token():
    c = O.HeadCache()
    q = synth.gen_bf16(51, 1, [0], [0], 0, 1)[0, 0]
    assert np.all(c.decode(O.rotate_q(q), TAU) == 0)
    k = synth.gen_bf16(52, 1, [0], [0], 0, 1)[0, 0]
    v = synth.gen_bf16(53, 1, [0], [0], 0, 1)[0, 0]
    c.append(k[0], v[0])
    # a single token gets weight 1: the output is that token's value
    np.testing.assert_array_equal(c.decode(O.rotate_q(q), TAU)[0], O.bf16_to_f64(v[0]))
