"""Pins for the oracle's INT2 quantiser and the packed word layouts.

INT2 means four levels ("OScaR：面向大模型及多模态LLM极限KV缓存量化的奥卡姆剃刀",
前置知识, per-channel quantisation with step Δ and zero z; news article on
arXiv 2605.19660, Q&A Q1: "only four distinguishable levels").  The checks
are properties any correct asymmetric min-max round-to-nearest quantiser has:
at most four codes, min -> 0 and max -> 3, nearest-level choice (brute
force over the four levels), the half-step error bound, ties to even, and the
per-block / per-token grouping.  The layout goldens are derived by hand from
the layout definition in include/oscar.h.
"""
import json
import os

import numpy as np

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _groups(seed, n_groups, size=32, scale=None):
    x = synth.normal_f32(seed, np.arange(n_groups * size)).reshape(n_groups, size)
    if scale is not None:
        x = (x * np.asarray(scale, np.float32)[:, None]).astype(np.float32)
    # values the cache can hold are bf16
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(x))


def test_four_levels_and_extremes():
    x = _groups(1, 200, scale=np.geomspace(1e-3, 1e3, 200))
    codes, step, zero = O.quantize_groups(x)
    assert codes.max() <= 3
    for g in range(x.shape[0]):
        assert len(np.unique(codes[g])) <= 4
        assert codes[g][np.argmin(x[g])] == 0
        assert codes[g][np.argmax(x[g])] == 3
    np.testing.assert_array_equal(zero, x.min(axis=1))
    # min is reconstructed exactly and max within one fp32 ulp (fp32 params)
    rec_min = zero + np.float32(0) * step
    np.testing.assert_array_equal(rec_min, x.min(axis=1))
    rec_max = (zero.astype(np.float64) + 3 * step.astype(np.float64))
    assert np.all(np.abs(rec_max - x.max(axis=1)) <= np.spacing(np.abs(x.max(axis=1)))
                  + np.spacing(np.abs(zero)) + 3 * np.spacing(step))


def test_code_is_a_nearest_level_brute_force():
    x = _groups(2, 300, scale=np.geomspace(1e-2, 1e2, 300))
    codes, step, zero = O.quantize_groups(x)
    lv = zero[:, None, None].astype(np.float64) + step[:, None, None].astype(np.float64) * np.arange(4)
    dist = np.abs(x[:, :, None].astype(np.float64) - lv)
    chosen = np.take_along_axis(dist, codes[:, :, None].astype(np.int64), axis=2)[..., 0]
    best = dist.min(axis=2)
    # the fp32 division can only blur exact ties by an ulp of (x - z)/Δ
    slack = 4 * np.spacing(np.float32(4.0)) * step[:, None].astype(np.float64)
    assert np.all(chosen <= best + slack)


def test_error_bound_with_stored_fp16_params():
    x = _groups(3, 200)
    codes, step, zero = O.quantize_groups(x)
    s16 = step.astype(np.float16).astype(np.float64)
    z16 = zero.astype(np.float16).astype(np.float64)
    rec = codes * s16[:, None] + z16[:, None]
    bound = (step.astype(np.float64) / 2 + 3 * np.abs(s16 - step) + np.abs(z16 - zero))[:, None]
    assert np.all(np.abs(rec - x) <= bound * (1 + 1e-6))


def test_ties_round_to_even_and_constant_group():
    x = np.array([[0.0, 0.5, 1.5, 2.5, 3.0, 1.0, 2.0, 0.0]], dtype=np.float32)
    codes, step, zero = O.quantize_groups(x)
    assert step[0] == 1.0 and zero[0] == 0.0
    np.testing.assert_array_equal(codes[0], [0, 0, 2, 2, 3, 1, 2, 0])
    c, s, z = O.quantize_groups(np.full((1, 32), 0.75, np.float32))
    assert s[0] == 0 and z[0] == np.float32(0.75) and np.all(c == 0)


def test_key_blocks_are_per_channel_per_32_tokens():
    n = 96
    base = synth.gen_bf16(4, 1, [0], [0], 0, n)[0, 0]
    x = synth.bf16_bits_to_f32(base).astype(np.float64)
    # give every (block, channel) its own offset: the parameters must follow
    off = np.arange(3)[:, None] * 100.0 + np.arange(128)[None, :]
    xs = x + np.repeat(off, 32, axis=0)
    bits = O.f64_to_bf16(xs)
    q = O.quantize_k(bits)
    vals = O.bf16_to_f64(bits).reshape(3, 32, 128)
    np.testing.assert_array_equal(q.zero16, vals.min(axis=1).astype(np.float16))
    for blk in range(3):
        c, s, z = O.quantize_groups(vals[blk].T.astype(np.float32))
        np.testing.assert_array_equal(q.codes[32 * blk:32 * blk + 32], c.T)


def test_value_groups_are_per_token():
    bits = synth.gen_bf16(5, 1, [0], [0], 0, 64)[0, 0]
    q = O.quantize_v(bits)
    vals = O.bf16_to_f64(bits)
    np.testing.assert_array_equal(q.zero16, vals.min(axis=1).astype(np.float16))
    assert all(len(np.unique(q.codes[t])) <= 4 for t in range(64))


def test_key_word_layout_golden():
    with open(os.path.join(GOLD, "layout_words.json")) as f:
        gold = json.load(f)
    codes = np.fromfunction(lambda t, c: c % 4, (32, 128), dtype=np.int64).astype(np.uint8)
    words = O.pack_k_words(codes)
    assert np.all(words == np.uint32(int(gold["k_words_c_mod_4"], 16)))
    one = np.zeros((32, 128), np.uint8)
    one[0, 17] = 3           # word 1, j=1 (odd) -> bit 16
    w = O.pack_k_words(one)
    assert w[0, 1] == np.uint32(int(gold["k_word_ch17_code3"], 16)) and w.sum() == w[0, 1]


def test_value_word_layout_golden():
    with open(os.path.join(GOLD, "layout_words.json")) as f:
        gold = json.load(f)
    # one code set at a time, location from the definition worked by hand
    for case in gold["v_single_code_cases"]:
        codes = np.zeros((32, 128), np.uint8)
        codes[case["token"], case["channel"]] = 1
        w = O.pack_v_words(codes)[0]
        nz = np.nonzero(w)[0]
        assert list(nz) == [case["word"]]
        assert int(w[case["word"]]) == 1 << case["bit"]


def test_value_word_layout_is_a_bijection():
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 4, size=(64, 128)).astype(np.uint8)
    w = O.pack_v_words(codes)
    # every code bit lands once: total popcount is preserved
    pop = sum(bin(int(v)).count("1") for v in w.ravel())
    assert pop == sum(bin(int(c)).count("1") for c in codes.ravel())
