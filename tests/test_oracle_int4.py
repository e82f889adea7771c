"""Pins for the oracle's INT4 option (16 levels instead of 4; the pages fix
only INT2 — "OScaR：面向大模型及多模态LLM极限KV缓存量化的奥卡姆剃刀", 局限与改进
(1), names other bit widths as unstudied — so the formula is the same
min-max quantiser with (max - min)/15 as the step).

* Lossless special case: with both ablation flags on and every group
  holding only the 16 exactly representable levels -7.5, -6.5, ..., 7.5
  (both extremes present), INT4 storage is exact and the cache's attention
  equals plain attention on the same bf16 K, V.
* Each group's minimum gets code 0 and its maximum code 15; the closed-form
  error bound |x~ - x| <= step/2 + fp16 rounding holds, with a step 1/5 of
  the INT2 step of the same group.
* The packed-word layouts against hand-worked cases
  (tests/golden/layout_words_int4.json).
* Streaming appends with flush-before-append equal one-shot quantisation.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")
TAU = 1 / math.sqrt(128)
LEVELS16 = np.arange(16) - 7.5


def _khat(seed, n):
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    k = synth.gen_bf16(seed, 1, [0], [0], 0, n, chan_factor=cf,
                       tok_factor=synth.sink_token_factors(1, 0, n))[0, 0]
    return O.rotate_scale_k(k).k_hat_bf16


def test_lossless_special_case():
    flags = O.NO_ROTATE | O.NO_SCALE
    T, P = 1024 + 200, 1024 - 64
    r = synth.splitmix64(601, np.arange(2 * T * 128)).reshape(2, T, 128)
    k = LEVELS16[(r[0] % np.uint64(16)).astype(np.int64)]
    v = LEVELS16[(r[1] % np.uint64(16)).astype(np.int64)]
    k[0::32, :], k[1::32, :] = -7.5, 7.5          # every (block, channel) group spans the range
    v[:, 0], v[:, 1] = -7.5, 7.5                  # every token group spans the range
    kb, vb = O.f64_to_bf16(k), O.f64_to_bf16(v)
    q = synth.gen_bf16(602, 4, [0], [0, 1, 2, 3], 0, 1)[0, :, 0]
    c = O.HeadCache(flags=flags, bits=4)
    c.quantize_prefix(kb[:P], vb[:P])
    for t in range(P, T):
        c.append(kb[t], vb[t])
    assert c.n_packed > P
    keys, vals = c.keys_values()
    np.testing.assert_array_equal(keys, k)
    np.testing.assert_array_equal(vals, v)
    got = c.decode(O.rotate_q(q, flags), TAU)
    want = O.bf16_attention(q, kb, vb, TAU)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)
    assert int(c.packed_k().codes.max()) == 15


def test_extremes_and_error_bound():
    kh = _khat(603, 128)
    q4, q2 = O.quantize_k(kh, bits=4), O.quantize_k(kh, bits=2)
    x = O.bf16_to_f64(kh)
    ch = np.arange(128)
    for j in range(4):
        xs, cs = x[32 * j:32 * j + 32], q4.codes[32 * j:32 * j + 32]
        assert np.all(cs[xs.argmin(axis=0), ch] == 0)
        assert np.all(cs[xs.argmax(axis=0), ch] == 15)
    # INT4 step = range / 15 = INT2 step / 5, up to the fp16 roundings
    np.testing.assert_allclose(q4.step16.astype(np.float64) * 5, q2.step16.astype(np.float64),
                               rtol=2e-3)
    back = O.dequant_k(q4, np.ones(128, np.float16))
    step = np.repeat(q4.step16.astype(np.float64), 32, axis=0)
    u = np.repeat(np.spacing(np.abs(q4.step16)).astype(np.float64), 32, axis=0)
    uz = np.repeat(np.spacing(np.abs(q4.zero16)).astype(np.float64), 32, axis=0)
    assert np.all(np.abs(back - x) <= step / 2 + 7.5 * u + 0.5 * uz + 1e-12)
    v = synth.gen_bf16(604, 1, [0], [0], 0, 64)[0, 0]
    qv = O.quantize_v(v, bits=4)
    assert qv.codes.max() == 15 and np.all(qv.codes.max(axis=1) == 15)


def test_key_word_layout_golden():
    with open(os.path.join(GOLD, "layout_words_int4.json")) as f:
        gold = json.load(f)
    codes = np.fromfunction(lambda t, c: c % 16, (32, 128), dtype=np.int64).astype(np.uint8)
    w = O.pack_k_words4(codes)
    assert np.all(w[:, 0::2] == np.uint32(int(gold["k_word_even_w_codes_c_mod_16"], 16)))
    assert np.all(w[:, 1::2] == np.uint32(int(gold["k_word_odd_w_codes_c_mod_16"], 16)))
    one = np.zeros((32, 128), np.uint8)
    one[0, 13] = 5
    w = O.pack_k_words4(one)
    case = gold["k_word_ch13_code5"]
    assert w[0, case["word"]] == np.uint32(int(case["value"], 16))
    assert w.sum() == w[0, case["word"]]


def test_value_word_layout_golden():
    with open(os.path.join(GOLD, "layout_words_int4.json")) as f:
        gold = json.load(f)
    for case in gold["v_single_code_cases"]:
        codes = np.zeros((32, 128), np.uint8)
        codes[case["token"], case["channel"]] = 1
        w = O.pack_v_words4(codes)[0]
        assert list(np.nonzero(w)[0]) == [case["word"]]
        assert int(w[case["word"]]) == 1 << case["bit"]
    # every code bit lands once
    rng = np.random.default_rng(8)
    codes = rng.integers(0, 16, size=(64, 128)).astype(np.uint8)
    w = O.pack_v_words4(codes)
    assert sum(bin(int(x)).count("1") for x in w.ravel()) == \
        sum(bin(int(c)).count("1") for c in codes.ravel())


@pytest.mark.parametrize("g", [32, 128])
def test_streaming_equals_one_shot(g):
    T = 3 * 128 + 17
    k = synth.gen_bf16(605, 1, [0], [0], 0, T)[0, 0]
    v = synth.gen_bf16(606, 1, [0], [0], 0, T)[0, 0]
    s = O.HeadCache(group=g, bits=4)
    for t in range(T):
        s.append(k[t], v[t])
    P = 128 * ((T - 1) // 128)
    one = O.build_head_cache(k[:P], v[:P], n_packed=P, group=g, bits=4)
    np.testing.assert_array_equal(s.packed_k().codes, one.packed_k().codes)
    np.testing.assert_array_equal(s.packed_k().step16, one.packed_k().step16)
    np.testing.assert_array_equal(s.packed_v().codes, one.packed_v().codes)
