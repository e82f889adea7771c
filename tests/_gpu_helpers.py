"""Shared helpers of the GPU parity tests (test infrastructure).

Data flows one way only: inputs are drawn by the shared generator, the oracle
builds its own cache and results from them, and oracle-built inputs may be
uploaded to the GPU; nothing the GPU computes is ever fed to the oracle.
"""
import functools
import math

import numpy as np
import torch

from oracle import oscar_oracle as O

TAU = 1.0 / math.sqrt(128)
MAX_ABS = 2e-3     # attention tolerance: max-abs error
REL_L2 = 1e-3      # and relative L2 error, per (sequence, query head) vector


def bits_to_bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_tensor_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def f16_tensor_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def attn_errors(gpu: np.ndarray, ref: np.ndarray):
    """(max-abs, worst per-vector relative L2) over [..., 128] vectors."""
    d = np.asarray(gpu, np.float64) - np.asarray(ref, np.float64)
    num = np.linalg.norm(d.reshape(-1, 128), axis=1)
    den = np.linalg.norm(np.asarray(ref, np.float64).reshape(-1, 128), axis=1)
    rel = np.where(den > 0, num / np.maximum(den, 1e-300), num)
    return float(np.abs(d).max()), float(rel.max())


def assert_attention_close(gpu, ref, what=""):
    ma, rl = attn_errors(gpu, ref)
    assert ma <= MAX_ABS and rl <= REL_L2, f"{what}: max-abs {ma:.3e}, rel-L2 {rl:.3e}"
    return ma, rl


def upload_oracle_cache(cache, heads: dict, flags: int = 0, norm_target: float = 0.0,
                        key_group: int = 0):
    """Writes oracle HeadCaches {(b, h): HeadCache} into a KVCache (same
    n_packed / n_res for every row), using the oracle's own packing; the
    cache takes the flags and target norm the oracle built them with."""
    P = R = None
    for (b, h), hc in heads.items():
        kq, vq = hc.packed_k(), hc.packed_v()
        p = kq.codes.shape[0]
        r = hc.n_res
        assert (P is None or P == p) and (R is None or R == r)
        P, R = p, r
        if p:
            nb = p // 32
            put = lambda name, arr: cache.field(name)[b, h, :nb].copy_(
                torch.from_numpy(np.ascontiguousarray(arr)))
            bits = getattr(cache, "bits", 2)
            put("k_codes", O.pack_words(kq.codes, bits, "k").reshape(nb, 128 * bits)
                .view(np.int32))
            put("v_codes", O.pack_words(vq.codes, bits, "v").view(np.int32))
            ks16, kz16 = kq.block_params()
            put("k_scale", ks16)
            put("k_zero", kz16)
            put("k_norm", hc.packed_norm16().reshape(nb, 4, 8))
            put("v_scale", vq.step16.reshape(nb, 4, 8))
            put("v_zero", vq.zero16.reshape(nb, 4, 8))
        if r:
            cache.k_res[b, h, :r] = bits_to_bf16_tensor(np.stack(hc.res_k_bf16))
            cache.v_res[b, h, :r] = bits_to_bf16_tensor(np.stack(hc.res_v_bf16))
            cache.k_res_norm[b, h, :r] = torch.from_numpy(np.array(hc.res_norm16, np.float16))
    cache.struct.n_packed = P or 0
    cache.struct.n_res = R or 0
    cache.struct.flags = flags
    cache.struct.norm_target = norm_target
    cache.struct.key_group = key_group
    return cache


def code_mismatches(a_words: np.ndarray, b_words: np.ndarray) -> int:
    """Number of 2-bit fields that differ between two uint32 word arrays."""
    x = (np.asarray(a_words).view(np.uint32) ^ np.asarray(b_words).view(np.uint32))
    x = (x | (x >> np.uint32(1))) & np.uint32(0x55555555)
    return int(sum(bin(int(v)).count("1") for v in x.ravel() if v))


@functools.lru_cache(maxsize=None)
def _key_field_map(bits: int):
    """(word, shift) of every channel in a token's packed key words, found by
    packing one-hot code arrays with the oracle's own packer."""
    where = []
    for c in range(128):
        x = np.zeros((32, 128), np.uint8)
        x[0, c] = 1
        w = np.asarray(O.pack_words(x, bits, "k")).view(np.uint32).reshape(-1)
        i = int(np.flatnonzero(w)[0])
        where.append((i, int(w[i]).bit_length() - 1))
    return tuple(where)


def unpack_key_codes(words: np.ndarray, bits: int) -> np.ndarray:
    """Key codes uint8 [n][128] from packed key words [n][4*bits] (uint32)."""
    w = np.asarray(words).view(np.uint32).reshape(words.shape[0], -1)
    mask = np.uint32((1 << bits) - 1)
    out = np.empty((w.shape[0], 128), np.uint8)
    for c, (i, sh) in enumerate(_key_field_map(bits)):
        out[:, c] = (w[:, i] >> np.uint32(sh)) & mask
    return out


def bf16_ulps(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place between two bf16 bit arrays
    (as ordered integers, in which -0 and +0 coincide)."""
    def ordered(u):
        u = np.asarray(u).astype(np.int64)
        return np.where(u & 0x8000, 0x8000 - u, u)
    return np.abs(ordered(a) - ordered(b))


def traced_key_check(L, cache, b: int, h: int, k_raw_bits: np.ndarray, v_bits: np.ndarray,
                     hc, flags: int = 0, bits: int = 2, target: float = 0.0, what: str = ""):
    """Traces every key code of row (b, h) of a GPU-built cache instead of
    bounding their number.

    The oracle and the GPU start from the same raw keys; only their rotated,
    scaled keys k_hat can differ (the GPU divides by an rsqrt, the oracle by an
    exact fp64 norm; the rotation gate bounds that at one bf16 ulp).  So:
     1. the GPU's k_hat of the row (oscar_rotate_scale_k on the raw keys) is
        within one bf16 ulp of the oracle's k_hat everywhere;
     2. quantising that GPU k_hat with the GPU's own quantiser
        (oscar_quantize_kv) reproduces the row's records byte for byte, so the
        fused prefill and the appends quantised exactly that k_hat;
     3. every (key group, channel) whose inputs are equal on both sides has
        the oracle's codes, step and zero bit for bit, and every differing
        code lies in a group that holds a differing input.
    Nothing computed on the GPU is fed to the oracle.  k_raw_bits / v_bits are
    the row's raw keys and values [T][128] in token order; with the all-heads
    norm (OSCAR_NORM_ALL_HEADS) they are the sequence's [Hkv][T][128], since a
    token's norm then spans every head.  Returns (differing codes, groups
    with a differing input)."""
    n = cache.n_packed
    nb = n // 32
    G = cache.key_group
    all_heads = bool(flags & O.NORM_ALL_HEADS)
    kr = np.ascontiguousarray(k_raw_bits[..., :n, :])
    vr = np.ascontiguousarray(v_bits[..., :n, :])
    H = kr.shape[0] if all_heads else 1
    rk = O.rotate_scale_k(kr, flags, target or 1.0)
    k_or = rk.k_hat_bf16[h] if all_heads else rk.k_hat_bf16
    kd = bits_to_bf16_tensor(kr.reshape(1, H, n, 128))
    vd = bits_to_bf16_tensor(vr.reshape(1, H, n, 128))
    kh = torch.empty_like(kd)
    nrm = torch.empty((1, H, n), dtype=torch.float16, device="cuda")
    L.rotate_scale_k(kd, kh, nrm, 1, H, n, in_T=n, out_T=n, flags=flags, norm_target=target)
    solo = L.KVCache(1, H, n, flags=flags, bits=bits, key_group=G, norm_target=target)
    L.quantize_kv(solo, kh, nrm, vd, src_T=n, n_tok=n)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    hs = h if all_heads else 0
    # 2. the row's records are the GPU quantiser applied to the GPU's k_hat
    assert torch.equal(solo.packed[0, hs, :nb], cache.packed[b, h, :nb]), f"{what}: records"
    # 1. k_hat within one bf16 ulp of the oracle's, or, where the rotated value
    #    cancels to nearly zero, within the fp32 rounding of the transform
    #    (2^-24 of the token's largest element): the GPU rotates in fp32, the
    #    oracle in exact fp64
    k_gpu = bf16_tensor_to_bits(kh)[0, hs]
    a, c = O.bf16_to_f64(k_gpu), O.bf16_to_f64(k_or)
    ulps = bf16_ulps(k_gpu, k_or)
    floor = 2.0 ** -24 * np.abs(c).max(axis=-1, keepdims=True)
    ok = (ulps <= 1) | (np.abs(a - c) <= floor)
    assert ok.all(), f"{what}: k_hat differs by {ulps[~ok].max()} ulp beyond the fp32 floor"
    # 3. groups with identical inputs are bit-exact; differences stay in the others
    kq = hc.packed_k()
    # an input differs where the bit patterns differ (so -0 against +0 counts)
    grp_in = (k_gpu != k_or).reshape(n // G, G, 128).any(axis=1)       # [group][channel]
    grp_in = np.repeat(grp_in, G // 32, axis=0)                         # [block][channel]
    got_codes = unpack_key_codes(cache.tokens("k_codes")[b, h, :n].cpu().numpy(), bits)
    diff = (got_codes != kq.codes).reshape(nb, 32, 128)
    assert not (diff & ~grp_in[:, None, :]).any(), f"{what}: code differs where inputs agree"
    ks16, kz16 = kq.block_params()
    gs = f16_tensor_to_np(cache.field("k_scale")[b, h, :nb])
    gz = f16_tensor_to_np(cache.field("k_zero")[b, h, :nb])
    same = ~grp_in
    assert np.array_equal(gs.view(np.uint16)[same], ks16.view(np.uint16)[same]), f"{what}: step"
    assert np.array_equal(gz.view(np.uint16)[same], kz16.view(np.uint16)[same]), f"{what}: zero"
    return int(diff.sum()), int(grp_in.sum())
