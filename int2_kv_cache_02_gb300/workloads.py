"""The decode workloads: shapes and seeded synthetic structure.

Each workload is one attention layer's KV cache for B sequences, drawn with
the generator of ``synth.py`` (numpy on the CPU, the same numbers on the GPU).
Structure follows the token-norm-imbalance patterns the pages describe: a few
channel outliers in K, attention-sink tokens with low K and V norm, and for
the mixed-modality stream norm jumps at segment boundaries plus rare
high-norm tokens.  Shapes are Qwen3-8B-like (32 query / 8 KV heads) and
Qwen3-Omni-30B-A3B-like (32 / 4) layers, head_dim 128.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import synth

OUTLIER_CHANNELS = (5, 38, 77, 110)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    T0: int            # cached tokens before the first decode step
    n_packed: int      # of which quantised (multiple of 32); T0 - n_packed <= 128 stay bf16
    steps: int         # decode steps that append one token each
    chan_factor_value: float
    mixed_modality: bool
    seed_base: int

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def n_res(self) -> int:
        return self.T0 - self.n_packed

    # seeds of the separate streams
    @property
    def seed_k(self) -> int:
        return self.seed_base + 1

    @property
    def seed_v(self) -> int:
        return self.seed_base + 2

    @property
    def seed_q(self) -> int:
        return self.seed_base + 3

    @property
    def seed_seg(self) -> int:
        return self.seed_base + 5

    def chan_factor(self) -> np.ndarray:
        return synth.channel_factors(OUTLIER_CHANNELS, self.chan_factor_value)

    def tok_factors(self, b_idx, t0: int, n_t: int):
        """(k_factor, v_factor) fp32 [len(b_idx)][n_t] for positions t0.."""
        b_idx = np.atleast_1d(np.asarray(b_idx))
        if self.mixed_modality:
            return synth.mixed_modality_factors(self.seed_seg, b_idx, t0, n_t,
                                                T_hint=self.T0 + self.steps)
        f = synth.sink_token_factors(len(b_idx), t0, n_t)
        return f, f.copy()

    def t_cap(self, extra_steps: int = 0) -> int:
        """Capacity covering the prompt and every flush of steps + extra_steps."""
        res, packed = self.n_res, self.n_packed
        for _ in range(self.steps + extra_steps):
            if res == 128:
                packed += 128
                res = 0
            res += 1
        return max(packed, 32)

    # -- CPU (numpy) draws of any slice -------------------------------------
    def k_bits(self, b_idx, h_idx, t0: int, n_t: int) -> np.ndarray:
        kf, _ = self.tok_factors(b_idx, t0, n_t)
        return synth.gen_bf16(self.seed_k, self.Hkv, b_idx, h_idx, t0, n_t,
                              chan_factor=self.chan_factor(), tok_factor=kf)

    def v_bits(self, b_idx, h_idx, t0: int, n_t: int) -> np.ndarray:
        _, vf = self.tok_factors(b_idx, t0, n_t)
        return synth.gen_bf16(self.seed_v, self.Hkv, b_idx, h_idx, t0, n_t, tok_factor=vf)

    def q_bits(self, b_idx, hq_idx, step: int) -> np.ndarray:
        """Query of decode step ``step`` (position = step in the query stream)."""
        return synth.gen_bf16(self.seed_q, self.Hq, b_idx, hq_idx, step, 1)[:, :, 0]


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_1k", B=1, Hq=1, Hkv=1, T0=1024, n_packed=992, steps=0,
                 chan_factor_value=20.0, mixed_modality=False, seed_base=1000),
        Workload("qwen3_8b_32k", B=8, Hq=32, Hkv=8, T0=32768, n_packed=32640, steps=1,
                 chan_factor_value=15.0, mixed_modality=False, seed_base=2000),
        Workload("long_stream_128k", B=1, Hq=32, Hkv=8, T0=131072, n_packed=130944, steps=256,
                 chan_factor_value=20.0, mixed_modality=False, seed_base=3000),
        Workload("batch48_128k", B=48, Hq=32, Hkv=8, T0=131072, n_packed=130944, steps=256,
                 chan_factor_value=20.0, mixed_modality=False, seed_base=4000),
        Workload("omni_tni_64k", B=16, Hq=32, Hkv=4, T0=65536, n_packed=65408, steps=256,
                 chan_factor_value=15.0, mixed_modality=True, seed_base=5000),
    ]
}


# ---------------------------------------------------------------------------
# GPU side: draw the inputs on the device and build the cache through the
# library's own calls.
# ---------------------------------------------------------------------------

def draw_kv_cuda(wl: Workload, t0: int, n_t: int, device="cuda"):
    """Raw bf16 K and V [B][Hkv][n_t][128] of positions t0.. on the device."""
    import torch
    K = torch.empty((wl.B, wl.Hkv, n_t, 128), dtype=torch.bfloat16, device=device)
    V = torch.empty_like(K)
    kf, vf = wl.tok_factors(np.arange(wl.B), t0, n_t)
    cf = torch.from_numpy(wl.chan_factor()).to(device)
    synth.gen_bf16_cuda(K, wl.seed_k, wl.Hkv, 0, t0, n_t, chan_factor=cf,
                        tok_factor=torch.from_numpy(kf).to(device))
    synth.gen_bf16_cuda(V, wl.seed_v, wl.Hkv, 0, t0, n_t,
                        tok_factor=torch.from_numpy(vf).to(device))
    return K, V


def draw_q_cuda(wl: Workload, step: int, device="cuda"):
    import torch
    q = torch.empty((wl.B, wl.Hq, 1, 128), dtype=torch.bfloat16, device=device)
    synth.gen_bf16_cuda(q, wl.seed_q, wl.Hq, 0, step, 1)
    return q.view(wl.B, wl.Hq, 128)


def build_cache_cuda(wl: Workload, K, V, flags: int = 0, T_cap: int | None = None,
                     chunk: int = 8192, device="cuda", fused: bool = True,
                     norm_target: float = 0.0, bits: int = 0):
    """Prompt of T0 tokens -> OScaR cache: rotate + scale + quantise the first
    n_packed tokens, then append the remaining ones to the residual window.
    fused=True does the first part in one oscar_prefill_kv call; fused=False
    takes the two-call path (oscar_rotate_scale_k into a bf16 staging buffer,
    then oscar_quantize_kv), in chunks."""
    import torch
    from . import oscar
    T_cap = T_cap if T_cap is not None else wl.t_cap()
    cache = oscar.KVCache(wl.B, wl.Hkv, T_cap, flags=flags, device=device,
                          norm_target=norm_target, bits=bits)
    T_stride = K.shape[2]
    if fused:
        if wl.n_packed:
            oscar.prefill_kv(cache, K, V, n_tok=wl.n_packed, in_T=T_stride)
    else:
        prefill_two_call(cache, K, V, wl.n_packed, chunk=chunk, device=device)
    if wl.n_res:
        kr = K[:, :, wl.n_packed:wl.T0].contiguous()
        vr = V[:, :, wl.n_packed:wl.T0].contiguous()
        oscar.append_kv(cache, kr, vr, n_tok=wl.n_res)
    return cache


def prefill_two_call(cache, K, V, n_tok: int, chunk: int = 8192, device="cuda"):
    """Tokens [0, n_tok) of raw K, V [B][Hkv][T][128] into the packed cache
    through the two-call path: oscar_rotate_scale_k into a bf16 staging
    buffer, then oscar_quantize_kv, in chunks (the cache's flags and target
    norm apply)."""
    import torch
    from . import oscar
    B, Hkv, T_stride = K.shape[0], K.shape[1], K.shape[2]
    chunk = min(chunk, max(32, n_tok))
    stage = torch.empty((B, Hkv, chunk, 128), dtype=torch.bfloat16, device=device)
    norm = torch.empty((B, Hkv, chunk), dtype=torch.float16, device=device)
    vstage = torch.empty_like(stage)
    for t0 in range(0, n_tok, chunk):
        n = min(chunk, n_tok - t0)
        oscar.rotate_scale_k(_offset(K, t0), stage, norm, B, Hkv, n, in_T=T_stride,
                             out_T=chunk, flags=cache.flags, norm_target=cache.norm_target)
        vstage[:, :, :n].copy_(V[:, :, t0:t0 + n])
        oscar.quantize_kv(cache, stage, norm, vstage, src_T=chunk, n_tok=n)


class _Offset:
    """A device pointer into a contiguous tensor at token offset t0 (rows keep
    their full stride, as the C ABI's in_T argument expects)."""

    def __init__(self, base, t0: int):
        self.base, self.t0 = base, t0
        self.is_cuda = True

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return self.base.data_ptr() + self.t0 * 128 * self.base.element_size()


def _offset(t, t0: int):
    return _Offset(t, t0)


# ---------------------------------------------------------------------------
# Needle variant of a workload, for the accuracy report: a few keys per row
# point at the row's queries, so that attention concentrates on them (in the
# spirit of the pages' needle-in-a-haystack retrieval runs) and the output of
# bf16 attention is far from zero.  Input structure only: no step of the
# method is computed here.
# ---------------------------------------------------------------------------

N_NEEDLES = 4
NEEDLE_MARGINS = (6.0, 5.0, 4.0, 3.0)   # nats above ln(context) for needles 0..3


def needle_keys(wl: Workload, b: int, h: int, step: int = 0):
    """(positions int [N_NEEDLES], raw bf16 key bits uint16 [N_NEEDLES][128])
    for row (b, h).  Needle i points along the mean of the row's query group
    at decode step `step`, tilted by a seeded random tenth, with the length
    that gives it a softmax score of ln(context) + NEEDLE_MARGINS[i] (nats,
    averaged over the group's heads): the needles take nearly all of the
    attention, in graded shares, and the rest of the context keeps a little.
    Positions are seeded, distinct, inside the packed prefix and clear of its
    first block (the attention sinks)."""
    g = wl.g
    q = synth.bf16_bits_to_f32(wl.q_bits([b], range(h * g, (h + 1) * g), step)[0])
    q = q.astype(np.float64)
    u = q.sum(axis=0)
    u /= np.linalg.norm(u)
    tau = 1.0 / np.sqrt(128.0)
    seed = wl.seed_base + 7
    row = b * wl.Hkv + h
    lo, hi = 32, max(33, wl.n_packed - 32)
    r = synth.splitmix64(seed, np.arange(row * 64, row * 64 + 64)).astype(np.uint64)
    pos, seen = [], set()
    for x in r:
        p = lo + int(x % np.uint64(hi - lo))
        if p not in seen:
            seen.add(p)
            pos.append(p)
        if len(pos) == N_NEEDLES:
            break
    tilt = synth.normal_f32(seed + 1, np.arange(row * N_NEEDLES * 128,
                                                (row + 1) * N_NEEDLES * 128))
    tilt = tilt.astype(np.float64).reshape(N_NEEDLES, 128)
    tilt /= np.linalg.norm(tilt, axis=1, keepdims=True)
    dirs = u[None, :] + 0.1 * tilt
    dirs /= np.linalg.norm(dirs, axis=1, keepdims=True)
    target = np.log(wl.T0) + np.asarray(NEEDLE_MARGINS[:N_NEEDLES])
    per_unit = tau * (dirs @ q.T).mean(axis=1)            # score of a unit-length needle
    keys = dirs * (target / per_unit)[:, None]
    return np.array(pos), synth.f32_to_bf16_bits(keys.astype(np.float32))


def plant_needles(wl: Workload, k_bits: np.ndarray, b: int, h: int, t0: int = 0):
    """Row (b, h)'s raw key bits [n_t][128] for positions t0.. with the needles
    written in (a copy)."""
    out = np.array(k_bits, copy=True)
    pos, keys = needle_keys(wl, b, h)
    for p, k in zip(pos, keys):
        if t0 <= p < t0 + out.shape[0]:
            out[p - t0] = k
    return out


def plant_needles_cuda(wl: Workload, K):
    """Writes every row's needles into raw keys K [B][Hkv][T][128] on the device."""
    import torch
    for b in range(wl.B):
        for h in range(wl.Hkv):
            pos, keys = needle_keys(wl, b, h)
            kt = torch.from_numpy(keys.view(np.int16)).view(torch.bfloat16).to(K.device)
            K[b, h, torch.from_numpy(pos).to(K.device)] = kt
    return K
