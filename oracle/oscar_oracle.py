"""OScaR oracle: a plain, slow CPU statement of what the decode path computes.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA path and imports nothing from the package; it takes plain numpy
arrays (bf16 values are passed as their uint16 bit patterns).

Precision: fp64 everywhere, except the INT2 quantiser, whose parameters and
code decision are fp32 with one rounding per operation (the quotient
(x - zero) / step rounded half to even; the pages fix no precision for it),
and the stored side arrays, which are rounded to fp16 / bf16 as the cache
format stores them.

Sources (page title and section):
* [rainbus] "OScaR：面向大模型及多模态LLM极限KV缓存量化的奥卡姆剃刀"
  (paper.rainbus.top summary): 方法步骤详情 (method step details), 前置知识
  (per-channel quantisation, Hadamard/FHT), 论文图表 (figure of the KIVI block
  layout with the R=128 residual window).
* [notes] "OScaR: The Occam's Razor for Extreme KV Cache Quantization in LLMs
  and Beyond" (reading notes, yingwang.github.io): II. Method (Notation; Step
  One: Canalized Rotation; Step Two: Omni-Token Scaling; End-to-End Flow).
* [news] news article on arXiv 2605.19660 (animattoys.com): 二 (the two steps),
  三 (three kernels, packed cache + residual cache, rsqrt).

Where the pages are silent or ambiguous, these readings shape the arithmetic
here: Sylvester (natural order) Hadamard of size 128 with entries
+-1/sqrt(128); the norm is per (token, KV head) unless NORM_ALL_HEADS asks for
the norm over all heads; keys are scaled to a target norm (1 unless given)
and the stored norm is n / target; asymmetric min-max INT2 with step
(max-min)/3 (INT4, an option: (max-min)/15), zero = min, round half to even,
codes from the fp32 parameters before their fp16 rounding; key groups of 32
tokens (64 or 128 as an option); a constant group stores step 0 and codes 0;
a zero key keeps k_hat = 0 and norm 0; flush-before-append.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

D = 128          # head_dim
G = 32           # key quantisation block (tokens sharing a channel's step/zero)
R = 128          # residual window
NO_ROTATE = 1    # ablation: skip Canalized Rotation
NO_SCALE = 2     # ablation: skip Omni-Token Scaling
NORM_ALL_HEADS = 4   # norm-scope variant: one norm per token over all KV heads


# --------------------------------------------------------------------------
# number formats (plain rounding definitions)
# --------------------------------------------------------------------------

def bf16_to_f64(u) -> np.ndarray:
    u = np.asarray(u, dtype=np.uint16)
    return (u.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round fp64 directly to bf16 (8 significant bits), nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    b = x.view(np.uint64)
    shift = np.uint64(52 - 7)
    lsb = (b >> shift) & np.uint64(1)
    r = ((b + (np.uint64(1) << (shift - np.uint64(1))) - np.uint64(1) + lsb) >> shift) << shift
    y = r.view(np.float64).astype(np.float32)          # exact: 8 significant bits
    return (y.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def f_to_f16(x) -> np.ndarray:
    """Round to IEEE binary16 (nearest, ties to even)."""
    return np.asarray(x).astype(np.float16)


# --------------------------------------------------------------------------
# Canalized Rotation  ([notes] II. Step One; [rainbus] 前置知识 Hadamard/FHT)
# --------------------------------------------------------------------------

def sylvester_hadamard(d: int = D) -> np.ndarray:
    """Orthonormal Hadamard matrix: H[i, j] = (-1)^popcount(i & j) / sqrt(d).

    Entries are +-1/sqrt(d) and H is orthogonal ([notes] Step One).  The pages
    name no ordering; the natural (Sylvester) order is the one the fast
    transform's Kronecker factorisation produces.
    """
    i = np.arange(d)[:, None]
    j = np.arange(d)[None, :]
    bits = np.bitwise_and(i, j)
    parity = np.zeros_like(bits)
    while np.any(bits):
        parity ^= bits & 1
        bits >>= 1
    return np.where(parity == 1, -1.0, 1.0) / math.sqrt(d)


_H = sylvester_hadamard(D)


def rotate_q(q_bits: np.ndarray, flags: int = 0) -> np.ndarray:
    """Query side of the rotation: q' = H q, applied to every [..., 128] vector.

    The same H as the keys, so q'.k' = q.k ([notes] Step One, "Query-side
    symmetric processing"; [rainbus] 方法步骤详情 item (1)).  The softmax scale is
    not applied here.  Dense mat-vec in fp64, no fast transform.
    """
    q = bf16_to_f64(q_bits)
    if flags & NO_ROTATE:
        return q
    return q @ _H.T


@dataclass
class RotatedKeys:
    k_hat: np.ndarray        # fp64 [..., 128], before bf16 rounding
    k_hat_bf16: np.ndarray   # uint16 [..., 128], what the cache stores
    norm: np.ndarray         # fp64 [...]
    norm_f16: np.ndarray     # float16 [...]


def rotate_scale_k(k_bits: np.ndarray, flags: int = 0, target: float = 1.0) -> RotatedKeys:
    """Canalized Rotation then Omni-Token Scaling of raw keys [..., 128].

    k' = H k ([notes] Step One, K' = K.H with H symmetric); s = sum k'^2,
    n = sqrt(s); k_hat = k' / n so every token has unit L2 norm, and n is kept
    to be multiplied back at dequantisation ([notes] Step Two; [news] 二, the
    norm is stored as a tag and restored at decode).  A zero key keeps
    k_hat = 0 and n = 0.  With NO_SCALE, k_hat = k' and n = 1.

    NORM_ALL_HEADS: k_bits is [Hkv, ..., 128], heads first, and n of a token
    is the norm of its rotated keys over all heads together ([notes] II,
    Notation: k_i in R^{H d_h}, n_i = ||k_i||; Step Two: the norm across all
    heads); every head's key is divided by it and stores it.

    target: the keys are scaled to norm `target` instead of 1 and the stored
    norm is n / target, so stored norm x k_hat = k' either way (the scaling
    target that [rainbus] 独立分析的弱点 (1) says an appendix ablates).
    """
    k = bf16_to_f64(k_bits)
    kr = k if flags & NO_ROTATE else k @ _H.T
    if flags & NO_SCALE:
        n = np.ones(kr.shape[:-1])
        return RotatedKeys(kr, f64_to_bf16(kr), n, f_to_f16(n))
    s = np.sum(kr * kr, axis=-1)
    if flags & NORM_ALL_HEADS:
        s = np.broadcast_to(np.sum(s, axis=0, keepdims=True), s.shape)
    n = np.sqrt(s)
    safe = np.where(n > 0, n, 1.0)
    kh = np.where((n > 0)[..., None], kr * (target / safe)[..., None], 0.0)
    stored = n / target
    return RotatedKeys(kh, f64_to_bf16(kh), stored, f_to_f16(stored))


# --------------------------------------------------------------------------
# INT2 quantiser ([rainbus] 前置知识 per-channel quantisation with step Δ and
# zero z; 方法步骤详情: K per-channel blocks of G=32 tokens (larger groups as
# an option), V per token)
# --------------------------------------------------------------------------

def quantize_groups(x: np.ndarray, bits: int = 2):
    """Asymmetric min-max quantisation over the last axis of ``x`` (fp32).

    L = 2^bits - 1 steps (INT2: 3, INT4: 15), levels z + c*Δ with
    c in {0..L}: z = min, Δ = (max - min)/L, the code is
    round-half-even((x - z)/Δ) clamped to [0, L].  All in fp32, one rounding
    per operation, in this order.  A constant group gets Δ = 0 and codes 0.
    Returns (codes uint8, step fp32, zero fp32).
    """
    L = (1 << bits) - 1
    x = np.asarray(x, dtype=np.float32)
    mn = x.min(axis=-1).astype(np.float32)
    mx = x.max(axis=-1).astype(np.float32)
    d = (mx - mn).astype(np.float32)
    step = (d / np.float32(L)).astype(np.float32)
    live = mx > mn
    safe = np.where(live, step, np.float32(1.0)).astype(np.float32)
    t = ((x - mn[..., None]).astype(np.float32) / safe[..., None]).astype(np.float32)
    codes = np.clip(np.rint(t), 0, L).astype(np.uint8)
    codes = np.where(live[..., None], codes, np.uint8(0)).astype(np.uint8)
    step = np.where(live, step, np.float32(0.0)).astype(np.float32)
    return codes, step, mn


@dataclass
class QuantK:
    codes: np.ndarray    # uint8 [n][128]
    step16: np.ndarray   # float16 [n/group][128]
    zero16: np.ndarray   # float16 [n/group][128]
    group: int = G       # tokens sharing a channel's step and zero

    def block_params(self):
        """(step16, zero16) per 32-token block, as the cache's records carry
        them: each group's parameters repeated over its group/32 blocks."""
        r = self.group // G
        return np.repeat(self.step16, r, axis=0), np.repeat(self.zero16, r, axis=0)


@dataclass
class QuantV:
    codes: np.ndarray    # uint8 [n][128]
    step16: np.ndarray   # float16 [n]
    zero16: np.ndarray   # float16 [n]


def quantize_k(k_hat_bits: np.ndarray, group: int = G, bits: int = 2) -> QuantK:
    """Block-wise per-channel INT2 for keys [n][128], n a multiple of group.

    Each channel of each group of ``group`` consecutive tokens has its own
    step and zero ([rainbus] 方法步骤详情 item (2); [notes] Notation).  The
    pages use groups of 32; 64 and 128 are the larger groups that [rainbus]
    局限与改进 (1) lists as not studied.
    """
    n = k_hat_bits.shape[0]
    assert group in (32, 64, 128) and n % group == 0
    x = bf16_to_f64(k_hat_bits).astype(np.float32)          # exact
    xb = x.reshape(n // group, group, D).transpose(0, 2, 1)  # [grp][ch][tok]
    codes, step, zero = quantize_groups(xb, bits)
    return QuantK(codes.transpose(0, 2, 1).reshape(n, D).copy(),
                  f_to_f16(step), f_to_f16(zero), group)


def quantize_v(v_bits: np.ndarray, bits: int = 2) -> QuantV:
    """Per-token INT2 (or INT4) for values [n][128] ([rainbus] 方法步骤详情
    item (3))."""
    x = bf16_to_f64(v_bits).astype(np.float32)
    codes, step, zero = quantize_groups(x, bits)
    return QuantV(codes, f_to_f16(step), f_to_f16(zero))


def dequant_k(q: QuantK, norm16: np.ndarray) -> np.ndarray:
    """k_tilde = (c*Δ + z) * n in fp64 with the stored fp16 parameters: the
    inverse quantisation followed by the inverse token scaling ([notes]
    End-to-End Flow, "dequantized and inverse-scaled")."""
    n = q.codes.shape[0]
    s = np.repeat(q.step16.astype(np.float64), q.group, axis=0)
    z = np.repeat(q.zero16.astype(np.float64), q.group, axis=0)
    return (q.codes.astype(np.float64) * s + z) * norm16.astype(np.float64)[:n, None]


def dequant_v(q: QuantV) -> np.ndarray:
    return (q.codes.astype(np.float64) * q.step16.astype(np.float64)[:, None]
            + q.zero16.astype(np.float64)[:, None])


# --------------------------------------------------------------------------
# Packed word layouts (the cache format; 16 two-bit codes per 32-bit word)
# --------------------------------------------------------------------------

def pack_k_words(codes: np.ndarray) -> np.ndarray:
    """Key codes [n][128] -> uint32 [n][8].

    Word w of a token holds channels 16w..16w+15; channel 16w+j sits at bit
    2*(j//2) + 16*(j%2): even channels in the low half-word, odd channels in
    the high half-word, in channel order.
    """
    n = codes.shape[0]
    out = np.zeros((n, 8), dtype=np.uint32)
    for w in range(8):
        for j in range(16):
            pos = 2 * (j // 2) + 16 * (j % 2)
            out[:, w] |= codes[:, 16 * w + j].astype(np.uint32) << np.uint32(pos)
    return out


def pack_v_words(codes: np.ndarray) -> np.ndarray:
    """Value codes [n][128] (n a multiple of 32) -> uint32 [n/32][256].

    Per block of 32 tokens, word index = 128*kh + 4*lane + 2*p + hh with
    kh, p, hh in {0, 1}, lane = 4*g + t (g in 0..7, t in 0..3).  The low
    half-word holds token 16*kh + 2*t + 8*p, the high half-word token + 1;
    slot k (bits 2k..2k+1 of each half) holds channel g + 8*(8*hh + k).
    """
    n = codes.shape[0]
    assert n % 32 == 0
    out = np.zeros((n // 32, 256), dtype=np.uint32)
    for kh in range(2):
        for lane in range(32):
            g, t = lane // 4, lane % 4
            for p in range(2):
                for hh in range(2):
                    widx = 128 * kh + 4 * lane + 2 * p + hh
                    tok = 16 * kh + 2 * t + 8 * p
                    for k in range(8):
                        ch = g + 8 * (8 * hh + k)
                        lo = codes[tok::32, ch].astype(np.uint32) << np.uint32(2 * k)
                        hi = codes[tok + 1::32, ch].astype(np.uint32) << np.uint32(16 + 2 * k)
                        out[:, widx] |= lo | hi
    return out


def pack_k_words4(codes: np.ndarray) -> np.ndarray:
    """INT4 key codes [n][128] -> uint32 [n][16].

    Word w of a token holds channels 8w..8w+7; channel 8w+j sits at bit
    4*(j//2) + 16*(j%2): even channels in the low half-word, odd channels in
    the high half-word, in channel order.
    """
    n = codes.shape[0]
    out = np.zeros((n, 16), dtype=np.uint32)
    for w in range(16):
        for j in range(8):
            pos = 4 * (j // 2) + 16 * (j % 2)
            out[:, w] |= codes[:, 8 * w + j].astype(np.uint32) << np.uint32(pos)
    return out


def pack_v_words4(codes: np.ndarray) -> np.ndarray:
    """INT4 value codes [n][128] (n a multiple of 32) -> uint32 [n/32][512].

    Per block of 32 tokens, word index = 256*kh + 128*p + 4*lane + hh with
    kh, p in {0, 1}, hh in {0..3}, lane = 4*g + t (g in 0..7, t in 0..3).
    The low half-word holds token 16*kh + 2*t + 8*p, the high half-word
    token + 1; slot k (bits 4k..4k+3 of each half) holds channel
    g + 8*(4*hh + k).
    """
    n = codes.shape[0]
    assert n % 32 == 0
    out = np.zeros((n // 32, 512), dtype=np.uint32)
    for kh in range(2):
        for lane in range(32):
            g, t = lane // 4, lane % 4
            for p in range(2):
                for hh in range(4):
                    widx = 256 * kh + 128 * p + 4 * lane + hh
                    tok = 16 * kh + 2 * t + 8 * p
                    for k in range(4):
                        ch = g + 8 * (4 * hh + k)
                        lo = codes[tok::32, ch].astype(np.uint32) << np.uint32(4 * k)
                        hi = codes[tok + 1::32, ch].astype(np.uint32) << np.uint32(16 + 4 * k)
                        out[:, widx] |= lo | hi
    return out


def pack_words(codes: np.ndarray, bits: int, kind: str) -> np.ndarray:
    """The cache's packed words of key (kind "k") or value ("v") codes."""
    if bits == 2:
        return pack_k_words(codes) if kind == "k" else pack_v_words(codes)
    return pack_k_words4(codes) if kind == "k" else pack_v_words4(codes)


# --------------------------------------------------------------------------
# Attention (fp64)
# --------------------------------------------------------------------------

def attention(q: np.ndarray, keys: np.ndarray, values: np.ndarray, tau: float) -> np.ndarray:
    """softmax(tau * q.K^T) V for q [g][128], keys/values [T][128]; no mask
    (a decode step sees the whole cache).  Max-subtracted, fp64."""
    if keys.shape[0] == 0:
        return np.zeros((q.shape[0], values.shape[1]))
    sc = tau * (q @ keys.T)
    sc -= sc.max(axis=-1, keepdims=True)
    p = np.exp(sc)
    return (p @ values) / p.sum(axis=-1, keepdims=True)


def bf16_attention(q_bits, k_bits, v_bits, tau: float) -> np.ndarray:
    """Unquantised attention on bf16 q, K, V (no rotation, no scaling)."""
    return attention(bf16_to_f64(q_bits), bf16_to_f64(k_bits), bf16_to_f64(v_bits), tau)


# --------------------------------------------------------------------------
# The cache of one (sequence, KV head) and the streaming state machine
# ([news] 三: packed cache of INT2 codes + parameters + norm tags, residual
# cache of the newest tokens in 16 bit, batch quantisation when 128 have
# accumulated; [rainbus] 论文图表 Fig. 2(c))
# --------------------------------------------------------------------------

@dataclass
class HeadCache:
    flags: int = 0
    target: float = 1.0
    group: int = G       # key group size (tokens sharing step and zero)
    bits: int = 2        # code width: 2 (the method) or 4
    k_codes: list = field(default_factory=list)   # QuantK per quantised chunk
    k_norm16: list = field(default_factory=list)
    v_q: list = field(default_factory=list)
    res_k_bf16: list = field(default_factory=list)   # uint16 [128] each
    res_norm16: list = field(default_factory=list)
    res_v_bf16: list = field(default_factory=list)

    @property
    def n_packed(self) -> int:
        return sum(q.codes.shape[0] for q in self.k_codes)

    @property
    def n_res(self) -> int:
        return len(self.res_k_bf16)

    def quantize_prefix(self, k_raw_bits: np.ndarray, v_bits: np.ndarray):
        """Rotate, scale and quantise a block-aligned run of tokens."""
        assert k_raw_bits.shape[0] % self.group == 0
        rk = self._rotate(k_raw_bits)
        self._pack(rk.k_hat_bf16, rk.norm_f16, v_bits)

    def _rotate(self, k_raw_bits):
        # a per-head norm; the all-heads norm needs every head (build_row_caches)
        assert not self.flags & NORM_ALL_HEADS
        return rotate_scale_k(k_raw_bits, self.flags, self.target)

    def _pack(self, k_hat_bits, norm16, v_bits):
        self.k_codes.append(quantize_k(k_hat_bits, self.group, self.bits))
        self.k_norm16.append(np.asarray(norm16, dtype=np.float16))
        self.v_q.append(quantize_v(v_bits, self.bits))

    def append(self, k_raw_bits: np.ndarray, v_bits: np.ndarray):
        """One decode token.  Flush-before-append: a full residual (128
        tokens) is quantised as four blocks first, so the newest token always
        stays 16-bit."""
        rk = self._rotate(k_raw_bits[None, :])
        self.append_scaled(rk.k_hat_bf16[0], rk.norm_f16[0], v_bits)

    def append_scaled(self, k_hat_bf16, norm16, v_bits):
        """append() of a key already rotated and scaled (flush first if full)."""
        if self.n_res == R:
            self.flush()
        self.res_k_bf16.append(np.asarray(k_hat_bf16, dtype=np.uint16))
        self.res_norm16.append(np.float16(norm16))
        self.res_v_bf16.append(np.asarray(v_bits, dtype=np.uint16))

    def push_residual(self, k_raw_bits: np.ndarray, v_bits: np.ndarray):
        """Place up to 128 prompt tokens in the residual window (no flush)."""
        assert self.n_res + k_raw_bits.shape[0] <= R
        rk = self._rotate(k_raw_bits)
        self._push_scaled(rk, v_bits)

    def _push_scaled(self, rk, v_bits):
        for i in range(rk.k_hat_bf16.shape[0]):
            self.res_k_bf16.append(rk.k_hat_bf16[i])
            self.res_norm16.append(rk.norm_f16[i])
            self.res_v_bf16.append(np.asarray(v_bits[i], dtype=np.uint16))

    def flush(self):
        assert self.n_res == R
        self._pack(np.stack(self.res_k_bf16), np.array(self.res_norm16, dtype=np.float16),
                   np.stack(self.res_v_bf16))
        self.res_k_bf16, self.res_norm16, self.res_v_bf16 = [], [], []

    # -- views -------------------------------------------------------------
    def packed_k(self) -> QuantK:
        if not self.k_codes:
            return QuantK(np.zeros((0, D), np.uint8), np.zeros((0, D), np.float16),
                          np.zeros((0, D), np.float16), self.group)
        return QuantK(np.concatenate([q.codes for q in self.k_codes]),
                      np.concatenate([q.step16 for q in self.k_codes]),
                      np.concatenate([q.zero16 for q in self.k_codes]), self.group)

    def packed_norm16(self) -> np.ndarray:
        if not self.k_norm16:
            return np.zeros(0, np.float16)
        return np.concatenate(self.k_norm16)

    def packed_v(self) -> QuantV:
        if not self.v_q:
            return QuantV(np.zeros((0, D), np.uint8), np.zeros(0, np.float16),
                          np.zeros(0, np.float16))
        return QuantV(np.concatenate([q.codes for q in self.v_q]),
                      np.concatenate([q.step16 for q in self.v_q]),
                      np.concatenate([q.zero16 for q in self.v_q]))

    def keys_values(self):
        """All cached keys (rotated basis, norm restored) and values, fp64."""
        kq, vq = self.packed_k(), self.packed_v()
        keys = [dequant_k(kq, self.packed_norm16())]
        vals = [dequant_v(vq)]
        if self.n_res:
            keys.append(bf16_to_f64(np.stack(self.res_k_bf16))
                        * np.array(self.res_norm16, dtype=np.float64)[:, None])
            vals.append(bf16_to_f64(np.stack(self.res_v_bf16)))
        return np.concatenate(keys), np.concatenate(vals)

    def decode(self, q_rot: np.ndarray, tau: float) -> np.ndarray:
        """Attention of the g rotated query heads [g][128] over this cache."""
        keys, vals = self.keys_values()
        return attention(np.atleast_2d(q_rot), keys, vals, tau)


def build_head_cache(k_raw_bits, v_bits, n_packed: int, flags: int = 0,
                     target: float = 1.0, group: int = G, bits: int = 2) -> HeadCache:
    """Prompt of T tokens: the first ``n_packed`` (a multiple of the key
    group) are quantised, the remaining T - n_packed (at most 128) stay in the
    residual."""
    T = k_raw_bits.shape[0]
    assert n_packed % group == 0 and 0 <= T - n_packed <= R
    c = HeadCache(flags=flags, target=target, group=group, bits=bits)
    if n_packed:
        c.quantize_prefix(k_raw_bits[:n_packed], v_bits[:n_packed])
    if T > n_packed:
        c.push_residual(k_raw_bits[n_packed:], v_bits[n_packed:])
    return c


def build_row_caches(k_raw_bits, v_bits, n_packed: int, flags: int = 0,
                     target: float = 1.0, group: int = G, bits: int = 2) -> list:
    """build_head_cache for every KV head of one sequence, k_raw_bits and
    v_bits [Hkv][T][128]: the keys of all heads are rotated and scaled
    together, which the all-heads norm needs, then each head is quantised
    and filled on its own."""
    Hkv, T = k_raw_bits.shape[0], k_raw_bits.shape[1]
    assert n_packed % group == 0 and 0 <= T - n_packed <= R
    rk = rotate_scale_k(k_raw_bits, flags, target)
    caches = []
    for h in range(Hkv):
        c = HeadCache(flags=flags, target=target, group=group, bits=bits)
        if n_packed:
            c._pack(rk.k_hat_bf16[h, :n_packed], rk.norm_f16[h, :n_packed], v_bits[h, :n_packed])
        if T > n_packed:
            c._push_scaled(RotatedKeys(rk.k_hat[h, n_packed:], rk.k_hat_bf16[h, n_packed:],
                                       rk.norm[h, n_packed:], rk.norm_f16[h, n_packed:]),
                           v_bits[h, n_packed:])
        caches.append(c)
    return caches


def append_row(caches: list, k_raw_bits, v_bits):
    """One decode token for every KV head of a sequence (k_raw_bits, v_bits
    [Hkv][128]): rotated and scaled together, then appended head by head
    (flush-before-append)."""
    c0 = caches[0]
    rk = rotate_scale_k(np.asarray(k_raw_bits)[:, None, :], c0.flags, c0.target)
    for h, c in enumerate(caches):
        c.append_scaled(rk.k_hat_bf16[h, 0], rk.norm_f16[h, 0], v_bits[h])
