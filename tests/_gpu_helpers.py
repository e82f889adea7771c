"""Shared helpers of the GPU parity tests (test infrastructure).

Data flows one way only: inputs are drawn by the shared generator, the oracle
builds its own cache and results from them, and oracle-built inputs may be
uploaded to the GPU; nothing the GPU computes is ever fed to the oracle.
"""
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
