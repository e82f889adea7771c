"""Seeded synthetic inputs shared by the CUDA path and the oracle.

This module holds no arithmetic of the method: it only draws numbers.  It is
the one piece of code that both sides may use (the oracle tests draw their
inputs here, and the GPU draws the same numbers with the kernel declared in
``include/oscar_synth.h``, which implements the same definition below).

Definition (both implementations follow it bit for bit)
------------------------------------------------------
* ``splitmix64`` (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014; the 64-bit finaliser popularised by Vigna) used as a
  counter-based generator: output ``n`` of stream ``seed`` is
  ``mix(seed + (n + 1) * 0x9E3779B97F4A7C15)`` in wrapping 64-bit arithmetic,
  with ``mix(z) = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
  z *= 0x94D049BB133111EB; z ^= z >> 31``.
* A standard-normal-like value per element (Irwin-Hall of twelve 16-bit
  uniforms): element counter ``e`` takes outputs ``3e, 3e+1, 3e+2``, splits each
  into four 16-bit fields, sums the twelve fields and subtracts ``6 * 65536``.
  The integer is converted to fp32 (exact: |v| < 2^20) and multiplied by 2^-16
  (exact).  Mean 0, variance 1.
* Structure: the fp32 value is multiplied (fp32, round to nearest even) by the
  channel factor, then by the token factor, then rounded to bf16 (RNE).
* Element counter for a [B][H][T][128] tensor: ``((b*H + h) * 2^32 + t) * 128 + c``
  so a token's value does not depend on the tensor's allocated length, and
  positions appended later in a stream continue the same sequence.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)
D = 128  # head_dim

_U64 = np.uint64


def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> _U64(30))
    z = z * M1
    z = z ^ (z >> _U64(27))
    z = z * M2
    return z ^ (z >> _U64(31))


def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """Output number ``counters`` of the splitmix64 stream ``seed`` (uint64)."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(_U64(seed & 0xFFFFFFFFFFFFFFFF) + (c + _U64(1)) * GAMMA)


def normal_int(seed: int, elem: np.ndarray) -> np.ndarray:
    """Irwin-Hall integer (sum of twelve 16-bit fields minus 6*65536), int64."""
    e = np.asarray(elem, dtype=np.uint64)
    acc = np.zeros(e.shape, dtype=np.int64)
    with np.errstate(over="ignore"):
        for j in range(3):
            r = splitmix64(seed, e * _U64(3) + _U64(j))
            for f in range(4):
                acc += ((r >> _U64(16 * f)) & _U64(0xFFFF)).astype(np.int64)
    return acc - 6 * 65536


def normal_f32(seed: int, elem: np.ndarray) -> np.ndarray:
    return normal_int(seed, elem).astype(np.float32) * np.float32(2.0 ** -16)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); finite inputs only."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + _U64(0x7FFF) + ((b >> _U64(16)) & _U64(1))) >> _U64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def element_counter(b, h, t, c, H: int) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint64)
    h = np.asarray(h, dtype=np.uint64)
    t = np.asarray(t, dtype=np.uint64)
    c = np.asarray(c, dtype=np.uint64)
    return ((b * _U64(H) + h) * _U64(1 << 32) + t) * _U64(D) + c


def gen_bf16(seed: int, H: int, b_idx, h_idx, t0: int, n_t: int,
             chan_factor: np.ndarray | None = None,
             tok_factor: np.ndarray | None = None) -> np.ndarray:
    """bf16 bits of shape [len(b_idx)][len(h_idx)][n_t][128].

    ``tok_factor`` is indexed [b][t - t0] with b the position inside ``b_idx``
    (shape [len(b_idx)][n_t]); ``chan_factor`` has 128 entries.
    """
    b_idx = np.atleast_1d(np.asarray(b_idx))
    h_idx = np.atleast_1d(np.asarray(h_idx))
    bb, hh, tt, cc = np.meshgrid(b_idx, h_idx, np.arange(t0, t0 + n_t), np.arange(D),
                                 indexing="ij")
    x = normal_f32(seed, element_counter(bb, hh, tt, cc, H))
    if chan_factor is not None:
        x = (x * np.asarray(chan_factor, dtype=np.float32)[None, None, None, :]).astype(np.float32)
    if tok_factor is not None:
        tf = np.asarray(tok_factor, dtype=np.float32)
        x = (x * tf[:, None, :, None]).astype(np.float32)
    return f32_to_bf16_bits(x)


# --------------------------------------------------------------------------
# Structure tables (token-norm imbalance patterns and channel outliers).
# Pure data: which tokens / channels get which fp32 factor.
# --------------------------------------------------------------------------

SINK_FACTOR = np.float32(0.05)


def channel_factors(channels, factor) -> np.ndarray:
    f = np.ones(D, dtype=np.float32)
    for c in channels:
        f[c] = np.float32(factor)
    return f


def sink_token_factors(n_b: int, t0: int, n_t: int, n_sink: int = 4) -> np.ndarray:
    """Tokens 0..n_sink-1 of each sequence scaled by 0.05 (attention sinks)."""
    t = np.arange(t0, t0 + n_t)
    f = np.where(t < n_sink, SINK_FACTOR, np.float32(1.0)).astype(np.float32)
    return np.broadcast_to(f, (n_b, n_t)).copy()


SEG_LEVELS = (np.float32(0.1), np.float32(1.0), np.float32(10.0))


def segments(seed: int, b: int, T: int, lo: int = 512, hi: int = 4096):
    """Segment starts and level indices for sequence ``b`` covering [0, T)."""
    starts, levels = [], []
    pos, i, prev = 0, 0, -1
    while pos < T:
        r = splitmix64(seed, np.array([(b << 20) * 2 + 2 * i, (b << 20) * 2 + 2 * i + 1],
                                      dtype=np.uint64))
        length = lo + int(r[0] % np.uint64(hi - lo + 1))
        if prev < 0:
            lev = int(r[1] % np.uint64(3))
        else:
            lev = (prev + 1 + int(r[1] % np.uint64(2))) % 3
        starts.append(pos)
        levels.append(lev)
        prev = lev
        pos += length
        i += 1
    return np.array(starts, dtype=np.int64), np.array(levels, dtype=np.int64)


def mixed_modality_factors(seed: int, b_idx, t0: int, n_t: int, T_hint: int,
                           n_sink: int = 4, outlier_per_mille: int = 1,
                           outlier_factor: float = 30.0):
    """Token factors for the mixed-modality stream.

    K factor = segment level (0.1 / 1 / 10, changing at every boundary)
               x 30 for about 0.1 % of tokens x 0.05 for the first 4 tokens of
               each segment; V factor = 0.05 on those segment-start tokens.
    Returns (k_factor, v_factor), each fp32 [len(b_idx)][n_t].
    """
    b_idx = np.atleast_1d(np.asarray(b_idx))
    kf = np.empty((len(b_idx), n_t), dtype=np.float32)
    vf = np.empty((len(b_idx), n_t), dtype=np.float32)
    t = np.arange(t0, t0 + n_t, dtype=np.int64)
    for i, b in enumerate(b_idx):
        starts, levels = segments(seed, int(b), max(T_hint, t0 + n_t))
        seg = np.searchsorted(starts, t, side="right") - 1
        level = np.array(SEG_LEVELS, dtype=np.float32)[levels[seg]]
        in_seg = t - starts[seg]
        sink = np.where(in_seg < n_sink, SINK_FACTOR, np.float32(1.0)).astype(np.float32)
        r = splitmix64(seed + 7, (np.uint64(int(b)) << np.uint64(32)) + t.astype(np.uint64))
        outl = np.where(r % np.uint64(1000) < np.uint64(outlier_per_mille),
                        np.float32(outlier_factor), np.float32(1.0)).astype(np.float32)
        kf[i] = (level * outl).astype(np.float32) * sink
        vf[i] = sink
    return kf, vf


# --------------------------------------------------------------------------
# The same generator on the GPU (liboscar_synth.so, include/oscar_synth.h).
# --------------------------------------------------------------------------

_synth_lib = None


def _synth():
    global _synth_lib
    if _synth_lib is None:
        import ctypes
        import os
        from . import _build
        path = _build.lib_path("liboscar_synth.so")
        if not os.path.exists(path):
            raise ImportError(f"liboscar_synth.so is not built ({path})")
        lib = ctypes.CDLL(path)
        c = ctypes
        lib.oscar_synth_bf16.restype = c.c_int
        lib.oscar_synth_bf16.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int,
                                         c.c_int, c.c_ulonglong, c.c_void_p, c.c_void_p,
                                         c.c_void_p]
        _synth_lib = lib
    return _synth_lib


def gen_bf16_cuda(out, seed: int, H: int, b0: int, t0: int, n_t: int,
                  chan_factor=None, tok_factor=None, stream=None):
    """Fills the bf16 device tensor ``out`` [nB][H][out_T][128] (tokens
    [0, n_t) of each row) with the same values as ``gen_bf16``.
    ``chan_factor`` / ``tok_factor`` are device fp32 tensors or None."""
    import ctypes
    import torch
    assert out.is_cuda and out.dtype == torch.bfloat16 and out.is_contiguous()
    nB, Hh, out_T = out.shape[0], out.shape[1], out.shape[2]
    assert Hh == H
    s = stream if stream is not None else torch.cuda.current_stream()
    cf = ctypes.c_void_p(chan_factor.data_ptr()) if chan_factor is not None else None
    tf = ctypes.c_void_p(tok_factor.data_ptr()) if tok_factor is not None else None
    rc = _synth().oscar_synth_bf16(ctypes.c_void_p(out.data_ptr()), nB, H, b0, out_T, t0, n_t,
                                   seed & 0xFFFFFFFFFFFFFFFF, cf, tf, ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError(f"oscar_synth_bf16 failed ({rc})")
