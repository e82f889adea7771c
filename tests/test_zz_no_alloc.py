"""The allocation-free decode entry point, checked against the regular one.

oscar_decode_attention_static_ws exists for callers that cannot allocate
device memory, for example a serving loop that forbids cudaMalloc once it is
warmed up, or a plug-in whose host runtime owns every device buffer and lends
it no allocator.  It keeps the split-K partials in a static array inside the
library, so its results must match oscar_decode_attention (which uses a
caller-provided workspace) on the same cache and queries, call after call.

This file is collected last on purpose and must pass both alone in a fresh
process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth
from tests._gpu_helpers import TAU, assert_attention_close, upload_oracle_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from int2_kv_cache_02_gb300 import _build
    _build.build()
    from int2_kv_cache_02_gb300 import oscar
    return oscar


def _cache(L, B=2, Hkv=2, T=2048 + 77, P=2048, seed=900):
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    tf = synth.sink_token_factors(B, 0, T)
    k = synth.gen_bf16(seed, Hkv, range(B), range(Hkv), 0, T, chan_factor=cf, tok_factor=tf)
    v = synth.gen_bf16(seed + 1, Hkv, range(B), range(Hkv), 0, T, tok_factor=tf)
    heads = {(b, h): O.build_head_cache(k[b, h], v[b, h], P)
             for b in range(B) for h in range(Hkv)}
    return upload_oracle_cache(L.KVCache(B, Hkv, P), heads)


def _qrot(L, B, Hq, seed):
    qb = synth.gen_bf16(seed, Hq, range(B), range(Hq), 0, 1)[:, :, 0]
    q = torch.from_numpy(qb.view(np.int16)).view(torch.bfloat16).cuda()
    qr = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    L.rotate_q(q, qr)
    return qr


@pytest.mark.parametrize("Hq", [8, 24])          # groups of 4, and of 12 (two slices)
@pytest.mark.parametrize("splits", [0, 5])
def test_static_scratch_matches_workspace_entry_on_two_calls(L, splits, Hq):
    B, Hkv = 2, 2
    cache = _cache(L)
    ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, cache.n_packed, splits))
    for call, seed in enumerate((910, 911)):          # two calls in a row, new queries
        qr = _qrot(L, B, Hq, seed)
        want = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
        L.decode_attention(cache, qr, Hq, TAU, want, ws, num_splits=splits)
        got = torch.full((B, Hq, 128), float("nan"), device="cuda")
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        st = L.library().oscar_decode_attention_static_ws(
            ctypes.byref(cache.struct), ctypes.c_void_p(qr.data_ptr()), Hq, TAU,
            ctypes.c_void_p(got.data_ptr()), splits,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, st
        torch.cuda.synchronize()
        if call > 0:
            # Once the library's module is loaded (first call), a call takes
            # no device memory: the driver's free memory is unchanged.
            assert torch.cuda.mem_get_info()[0] == free0
        assert L.device_status() == 0
        assert_attention_close(got.cpu().numpy(), want.cpu().numpy(), f"call {call}")


def test_static_scratch_rejects_oversized_requests(L):
    B, Hq = 2, 8
    cache = _cache(L, seed=920)
    qr = _qrot(L, B, Hq, 921)
    out = torch.zeros((B, Hq, 128), dtype=torch.float32, device="cuda")
    # 2 x 8 x 4097 partial records of 528 bytes exceed the 16 MiB array
    st = L.library().oscar_decode_attention_static_ws(
        ctypes.byref(cache.struct), ctypes.c_void_p(qr.data_ptr()), Hq, TAU,
        ctypes.c_void_p(out.data_ptr()), 4096, None)
    assert st == 5                                     # OSCAR_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 0)                         # nothing was launched


def test_static_scratch_lowers_an_automatic_split_count_that_does_not_fit(L):
    """With num_splits = 0 the planner's split count is lowered to the largest
    one whose partial records and row counters fit in the static array; the
    output then equals the workspace entry's at that count, bit for bit, on
    two calls in a row.  The shape is chosen so that the planned count does
    not fit (batch 128 or more, 32 query / 8 KV heads, 32K packed tokens)."""
    Hkv, Hq, P = 8, 32, 32768
    limit = 16 << 20
    for B in (128, 160, 192, 256):
        S_plan = L.decode_num_splits(B, Hkv, Hq, P)
        if L.decode_workspace_bytes(B, Hkv, Hq, P, S_plan) > limit:
            break
    else:
        raise AssertionError("no batch up to 256 needs more than the static array")
    S = max(s for s in range(1, S_plan)
            if L.decode_workspace_bytes(B, Hkv, Hq, P, s) <= limit)
    # A cache of random codes with finite, plausible steps, zeros and norms:
    # both entry points read the same bytes, so no oracle is needed here.
    g = torch.Generator(device="cuda").manual_seed(930)
    cache = L.KVCache(B, Hkv, P)
    cache.packed.copy_(torch.randint(0, 256, cache.packed.shape, dtype=torch.uint8,
                                     device="cuda", generator=g))
    for name, lo, hi in (("k_scale", 0.05, 0.4), ("k_zero", -1.0, -0.5), ("k_norm", 8.0, 14.0),
                         ("v_scale", 0.5, 1.0), ("v_zero", -2.0, -1.5)):
        cache.field(name).uniform_(lo, hi, generator=g)
    cache.struct.n_packed = P
    ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, P, S))
    for call, seed in enumerate((931, 932)):
        qr = _qrot(L, B, Hq, seed)
        want = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
        L.decode_attention(cache, qr, Hq, TAU, want, ws, num_splits=S)
        got = torch.full((B, Hq, 128), float("nan"), device="cuda")
        st = L.library().oscar_decode_attention_static_ws(
            ctypes.byref(cache.struct), ctypes.c_void_p(qr.data_ptr()), Hq, TAU,
            ctypes.c_void_p(got.data_ptr()), 0,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, st
        torch.cuda.synchronize()
        assert L.device_status() == 0
        assert torch.isfinite(want).all()
        assert torch.equal(got, want), f"call {call}: static entry did not use {S} splits"
    del cache
    torch.cuda.empty_cache()
