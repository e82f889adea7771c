"""The rule the INT2 group kernels use to form codes, checked on the host
against the definition.

The quantiser's code of a = fl(x - mn) (both fp32) is rint(fl(a / step))
with round-half-even throughout ("OScaR：面向大模型及多模态LLM极限KV缓存量化的
奥卡姆剃刀", 前置知识: asymmetric quantisation with step Δ and zero z).  The
kernels count thresholds instead: code >= j + 1 iff a >= A_j, with A_j the
fp32 rounding upward of m_j * step (exact in fp64), m_j = h - u-/2 when
j + 1 is even and h + u+/2 (strictly above) when odd, h = j + 1/2 and u-,
u+ the fp32 spacings below and above h.  This test derives m_j from exact
rationals and checks, for random steps (normal and subnormal) and for a
values at, around and far from each threshold, that the threshold count
equals the definition; and, on bf16 key groups and value tokens with ties
and tiny steps, that it equals the oracle's codes.
"""
import math
from fractions import Fraction

import numpy as np
import pytest


def _spacing(h, below):
    e = math.floor(math.log2(h))
    if below and h == Fraction(2) ** e:
        return Fraction(2) ** (e - 24)
    return Fraction(2) ** (e - 23)


def _factor(j):
    h = Fraction(2 * j + 1, 2)
    if (j + 1) % 2 == 0:
        return h - _spacing(h, True) / 2
    return h + _spacing(h, False) / 2


def _f32_up(x: Fraction) -> np.float32:
    f = np.float32(float(x))                 # nearest (x is exact in fp64 here)
    if not np.isfinite(f):                   # beyond the largest fp32: rounds up to inf
        return f
    if Fraction(float(f)) < x:
        f = np.nextafter(f, np.float32(np.inf))
    return f


def _threshold(step: np.float32, j: int) -> np.float32:
    b = _factor(j) * Fraction(float(step))
    up = _f32_up(b)
    if (j + 1) % 2 == 1 and np.isfinite(up) and Fraction(float(up)) == b:
        up = np.nextafter(up, np.float32(np.inf))
    return up


def _code(a: np.float32, step: np.float32, levels: int) -> int:
    t = np.float32(a) / np.float32(step)     # IEEE fp32 division
    return int(min(max(np.rint(t), 0), levels))


@pytest.mark.parametrize("bits", [2, 4])
def test_threshold_count_equals_definition(bits):
    levels = (1 << bits) - 1
    rng = np.random.default_rng(5 + bits)
    steps = [np.float32(s) for s in
             list(rng.uniform(1e-3, 10.0, 40)) + [0.25, 1 / 3, 3.0 / 64, 1e-30, 2.0 ** -133,
                                                   3 * 2.0 ** -140, 1e30]]
    n_checked = 0
    with np.errstate(over="ignore"):
        for s in steps:
            if not np.isfinite(s) or s == 0:
                continue
            A = [_threshold(s, j) for j in range(levels)]
            assert all(A[i] <= A[i + 1] for i in range(levels - 1))
            cands = []
            for Aj in A:
                f = Aj
                for _ in range(4):
                    f = np.nextafter(f, np.float32(0))
                g = f
                for _ in range(9):                  # A_j - 4 ulp .. A_j + 4 ulp
                    cands.append(g)
                    g = np.nextafter(g, np.float32(np.inf))
            cands += list((rng.uniform(0, levels, 64) * s).astype(np.float32))
            for a in cands:
                if not np.isfinite(a) or a < 0:
                    continue
                want = _code(a, s, levels)
                got = sum(1 for Aj in A if a >= Aj)
                assert got == want, (float(s), float(a), got, want)
                n_checked += 1
    assert n_checked > 1000


def test_factors_are_exact_in_fp64():
    for j in range(15):
        m = _factor(j)
        assert Fraction(float(m)) == m              # the kernels hold m as a double
        assert m.denominator <= 2 ** 26 and m * 2 ** 26 % 1 == 0


def test_threshold_count_equals_oracle_codes():
    """The rule against the oracle's quantiser on bf16 data: key groups of 32
    tokens per channel and value tokens, with random, tied and tiny-step
    groups; the count of thresholds at or below fl(x - zero) is the oracle's
    code everywhere."""
    from oracle import oscar_oracle as O
    rng = np.random.default_rng(21)
    x = rng.standard_normal((64, 128))
    x[0:32, 0:16] = (rng.integers(0, 7, (32, 16)) * 0.125 - 0.375)     # exact half levels
    x[32:64, 16] = rng.integers(0, 4, 32) * 2.0 ** -133                # step 2^-133
    x[5, :] = rng.integers(0, 7, 128) * 0.25 - 0.75                    # a tied value token
    xb = O.f64_to_bf16(x)
    xf = O.bf16_to_f64(xb).astype(np.float32)
    for axis, groups in (("k", xf.reshape(2, 32, 128).transpose(0, 2, 1).reshape(-1, 32)),
                         ("v", xf)):
        codes, step, zero = O.quantize_groups(groups)
        for g in range(groups.shape[0]):
            if not step[g] > 0:
                assert np.all(codes[g] == 0)
                continue
            A = [_threshold(np.float32(step[g]), j) for j in range(3)]
            a = (groups[g] - zero[g]).astype(np.float32)
            got = sum((a >= Aj).astype(np.int64) for Aj in A)
            np.testing.assert_array_equal(got, codes[g].astype(np.int64), err_msg=f"{axis} {g}")


def _f32_down(x: Fraction) -> np.float32:
    f = np.float32(float(x))
    if not np.isfinite(f):                   # beyond the largest fp32: rounds down to it
        return np.float32(np.finfo(np.float32).max)
    if Fraction(float(f)) > x:
        f = np.nextafter(f, np.float32(-np.inf))
    return f


def _threshold_fp32_form(step: np.float32, j: int) -> np.float32:
    """The kernels' fp32 form of A_j, step by step: m_j = h + d, h = j + 1/2,
    d = +-2^-k; c = fl(d * s) in fp32; the fused multiply-add h * s + c
    rounded up (and down, for the strict case); steps below 2^-100 scaled
    by 2^64 first and the results scaled back with the same rounding."""
    h = np.float32(j + 0.5)
    d = np.float32(float(_factor(j) - Fraction(2 * j + 1, 2)))
    tiny = step < np.float32(2.0 ** -100)
    s = np.float32(step * np.float32(2.0 ** 64)) if tiny else step
    c = np.float32(d * s)                                # fp32 multiply
    exact = Fraction(float(h)) * Fraction(float(s)) + Fraction(float(c))
    up, dn = _f32_up(exact), _f32_down(exact)
    if tiny:
        up = _f32_up(Fraction(float(up)) * Fraction(1, 2 ** 64))
        dn = _f32_down(Fraction(float(dn)) * Fraction(1, 2 ** 64))
    if (j + 1) % 2 == 0:
        return up
    return np.nextafter(up, np.float32(np.inf)) if dn == up else up


def test_fp32_form_of_the_thresholds_equals_the_rule():
    """The fp32 fused multiply-add form the kernels use gives the same A_j as
    the exact rule, for normal, tiny-normal, subnormal and huge steps and the
    edge of the scaling (2^-100)."""
    rng = np.random.default_rng(77)
    bits = np.concatenate([
        rng.integers(0x00000001, 0x00800000, 300),       # subnormal
        rng.integers(0x00800000, 0x0d800000, 300),       # normal below 2^-100
        rng.integers(0x0d000000, 0x0e800000, 300),       # around 2^-100
        rng.integers(0x0e800000, 0x7f000000, 600),       # normal
        rng.integers(0x7f000000, 0x7f800000, 100),       # huge (products may overflow)
        np.array([1, 2, 3, 0x00800000, 0x0d800000, 0x0d7fffff, 0x3eaaaaab, 0x7f7fffff]),
    ]).astype(np.uint32)
    with np.errstate(over="ignore"):
        for b in bits:
            s = np.array([b], dtype=np.uint32).view(np.float32)[0]
            for j in range(3):
                want, got = _threshold(s, j), _threshold_fp32_form(s, j)
                assert want.view(np.uint32) == got.view(np.uint32), (hex(int(b)), j, want, got)
