"""Pins for the oracle's larger key groups (a channel's step and zero shared by
64 or 128 tokens instead of 32; "OScaR：面向大模型及多模态LLM极限KV缓存量化的奥卡姆剃刀",
局限与改进 (1), names the larger groups as not studied; 方法步骤详情 (2) gives
the per-channel block quantisation itself).

* Groups compose: a 64-token group's zero is the smaller of its two 32-token
  halves' zeros (rounding to fp16 is monotone, so this holds exactly), and
  its step is at least each half's step.
* A constructed case whose 32-token blocks hold, per channel, one of the
  four exactly representable levels {-1.5, -0.5, 0.5, 1.5}: groups of 32
  and 128 reproduce the input exactly, the 128-token codes are the level
  indices, and each 64-token group codes its lower level 0 and its upper
  level 3 (a group boundary in the wrong place, or channels and tokens
  swapped, gives other codes).
* The closed-form error bound |x~ - x| <= step/2 + the fp16 rounding of
  step and zero, for random rotated keys.
* Streaming appends with flush-before-append equal one-shot quantisation,
  and the lossless special case gives plain attention, at every group size.
"""
import math

import numpy as np
import pytest

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth

TAU = 1 / math.sqrt(128)
LEVELS = np.array([-1.5, -0.5, 0.5, 1.5])


def _khat(seed, n):
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    k = synth.gen_bf16(seed, 1, [0], [0], 0, n, chan_factor=cf,
                       tok_factor=synth.sink_token_factors(1, 0, n))[0, 0]
    return O.rotate_scale_k(k).k_hat_bf16


def test_groups_compose():
    kh = _khat(501, 256)
    q32, q64, q128 = (O.quantize_k(kh, g) for g in (32, 64, 128))
    assert q64.step16.shape == (4, 128) and q128.step16.shape == (2, 128)
    np.testing.assert_array_equal(q64.zero16, np.minimum(q32.zero16[0::2], q32.zero16[1::2]))
    np.testing.assert_array_equal(q128.zero16, np.minimum(q64.zero16[0::2], q64.zero16[1::2]))
    assert np.all(q64.step16 >= np.maximum(q32.step16[0::2], q32.step16[1::2]))
    assert np.all(q128.step16 >= np.maximum(q64.step16[0::2], q64.step16[1::2]))
    # each group's extremes get codes 0 and 3 (every group here is live)
    x = O.bf16_to_f64(kh)
    for g, q in ((64, q64), (128, q128)):
        for j in range(256 // g):
            xs, cs = x[j * g:(j + 1) * g], q.codes[j * g:(j + 1) * g]
            ch = np.arange(128)
            assert np.all(cs[xs.argmin(axis=0), ch] == 0)
            assert np.all(cs[xs.argmax(axis=0), ch] == 3)


def test_block_levels_exact_at_every_group_size():
    """Block b of channel c holds level (b + c) % 4 for all its 32 tokens."""
    n = 256
    idx = (np.arange(n)[:, None] // 32 + np.arange(128)[None, :]) % 4
    kh = O.f64_to_bf16(LEVELS[idx])
    for g in (32, 128):
        q = O.quantize_k(kh, g)
        back = O.dequant_k(q, np.ones(n, np.float16))
        np.testing.assert_array_equal(back, LEVELS[idx])
    # a 64-group holds two adjacent levels: the lower gets code 0, the upper 3
    q64 = O.quantize_k(kh, 64)
    lo_blk = (idx[0::32][0::2] > idx[0::32][1::2])         # [group][ch]: block 1 lower?
    want = np.where(np.repeat(np.repeat(lo_blk, 2, axis=0), 32, axis=0)
                    == (np.arange(n)[:, None] // 32 % 2 == 1), 0, 3)
    np.testing.assert_array_equal(q64.codes, want)
    q128 = O.quantize_k(kh, 128)
    np.testing.assert_array_equal(q128.codes, idx)         # levels span every 128-group
    assert np.all(q128.zero16 == -1.5) and np.all(q128.step16 == 1.0)
    q32 = O.quantize_k(kh, 32)
    assert np.all(q32.codes == 0) and np.all(q32.step16 == 0)   # constant blocks
    s, z = q128.block_params()
    assert s.shape == (8, 128) and np.all(z == -1.5)


@pytest.mark.parametrize("g", [64, 128])
def test_error_bound(g):
    kh = _khat(502, 384)
    q = O.quantize_k(kh, g)
    x = O.bf16_to_f64(kh)
    back = O.dequant_k(q, np.ones(384, np.float16))
    step = np.repeat(q.step16.astype(np.float64), g, axis=0)
    # the fp16 step and zero are within half an fp16 ulp of their fp32 values,
    # and a code c <= 3 multiplies the step's error
    u = np.spacing(np.abs(q.step16)).astype(np.float64)
    uz = np.spacing(np.abs(q.zero16)).astype(np.float64)
    bound = step / 2 + 1.5 * np.repeat(u, g, axis=0) + 0.5 * np.repeat(uz, g, axis=0) + 1e-12
    assert np.all(np.abs(back - x) <= bound)


@pytest.mark.parametrize("g", [64, 128])
def test_streaming_equals_one_shot(g):
    T = 3 * 128 + 17
    k = synth.gen_bf16(503, 1, [0], [0], 0, T)[0, 0]
    v = synth.gen_bf16(504, 1, [0], [0], 0, T)[0, 0]
    s = O.HeadCache(group=g)
    for t in range(T):
        s.append(k[t], v[t])
    P = 128 * ((T - 1) // 128)
    one = O.build_head_cache(k[:P], v[:P], n_packed=P, group=g)
    a, b = s.packed_k(), one.packed_k()
    assert a.group == b.group == g
    np.testing.assert_array_equal(a.codes, b.codes)
    np.testing.assert_array_equal(a.step16, b.step16)
    np.testing.assert_array_equal(a.zero16, b.zero16)


@pytest.mark.parametrize("g", [64, 128])
def test_lossless_special_case(g):
    flags = O.NO_ROTATE | O.NO_SCALE
    T, P = 1024 + 200, 896
    r = synth.splitmix64(505, np.arange(2 * T * 128)).reshape(2, T, 128)
    k = LEVELS[(r[0] % np.uint64(4)).astype(np.int64)]
    v = LEVELS[(r[1] % np.uint64(4)).astype(np.int64)]
    k[0::32, :], k[1::32, :] = -1.5, 1.5        # every group spans the range
    v[:, 0], v[:, 1] = -1.5, 1.5
    kb, vb = O.f64_to_bf16(k), O.f64_to_bf16(v)
    q = synth.gen_bf16(506, 4, [0], [0, 1, 2, 3], 0, 1)[0, :, 0]
    c = O.HeadCache(flags=flags, group=g)
    c.quantize_prefix(kb[:P], vb[:P])
    for t in range(P, T):
        c.append(kb[t], vb[t])
    keys, vals = c.keys_values()
    np.testing.assert_array_equal(keys, k)
    np.testing.assert_array_equal(vals, v)
    got = c.decode(O.rotate_q(q, flags), TAU)
    want = O.bf16_attention(q, kb, vb, TAU)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)
