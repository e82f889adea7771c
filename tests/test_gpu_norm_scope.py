"""Norm-scope and target-norm variants of Omni-Token Scaling on the GPU
against the oracle.

* Rotation gate: oscar_rotate_scale_k with OSCAR_NORM_ALL_HEADS and / or a
  target norm; k_hat within 1 bf16 ulp of the oracle's fp64 value, the
  stored norm within 2 fp16 ulp (zero tokens and a zero head included).
* The fused prefill equals the two-call path byte for byte under each
  variant (both form the all-heads sum the same way).
* Attention gate: the decode over an oracle-built cache of each variant
  (max-abs <= 2e-3 and rel-L2 <= 1e-3), and over a cache built on the GPU
  by prefill + streaming appends across a flush, against the oracle's own
  pipeline on the same draws.
Sources: "OScaR: The Occam's Razor for Extreme KV Cache Quantization in LLMs
and Beyond" (reading notes), II. Method, Notation and Step Two (the norm
across all heads); "OScaR：面向大模型及多模态LLM极限KV缓存量化的奥卡姆剃刀",
独立分析的弱点 (1) (the scaling target).
"""
import numpy as np
import pytest
import torch

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth
from tests._gpu_helpers import (TAU, assert_attention_close, bf16_tensor_to_bits,
                                bits_to_bf16_tensor, code_mismatches, f16_tensor_to_np, traced_key_check,
                                upload_oracle_cache)

pytestmark = pytest.mark.gpu

VARIANTS = [(O.NORM_ALL_HEADS, 1.0), (0, 0.37), (O.NORM_ALL_HEADS, 3.0),
            (O.NORM_ALL_HEADS | O.NO_ROTATE, 1.0)]


@pytest.fixture(scope="module")
def L():
    from int2_kv_cache_02_gb300 import _build
    _build.build()
    from int2_kv_cache_02_gb300 import oscar
    return oscar


def _sync_ok(L):
    torch.cuda.synchronize()
    assert L.device_status() == 0


def _keys(seed, B, Hkv, T0, T):
    """bf16 bits [B][Hkv][T][128]: outlier channels, sinks, and head h
    scaled by 4^-h, so that the all-heads norm differs from each head's own
    and the last heads' k_hat lie far below unit norm (1/64 for h = 3) while
    every head's scores stay of ordinary size."""
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    tf = synth.sink_token_factors(B, T0, T)
    k = synth.gen_bf16(seed, Hkv, range(B), range(Hkv), T0, T, chan_factor=cf, tok_factor=tf)
    x = O.bf16_to_f64(k) * (4.0 ** -np.arange(Hkv))[None, :, None, None]
    return O.f64_to_bf16(x)


def _ulp_bf16(x):
    x = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 7)


@pytest.mark.parametrize("flags, target", VARIANTS)
def test_rotate_scale_k_gate(L, flags, target):
    B, H, T = 2, 4, 70
    bits = _keys(1201, B, H, 0, T)
    bits[0, :, 7] = 0                 # a token that is zero in every head
    bits[1, 2, 9] = 0                 # a token that is zero in one head only
    k = bits_to_bf16_tensor(bits)
    k_hat = torch.empty((B, H, T + 5, 128), dtype=torch.bfloat16, device="cuda")
    norm = torch.zeros((B, H, T + 5), dtype=torch.float16, device="cuda")
    L.rotate_scale_k(k, k_hat, norm, B, H, T, in_T=T, out_T=T + 5, out_t0=5, flags=flags,
                     norm_target=target)
    _sync_ok(L)
    for b in range(B):
        ref = O.rotate_scale_k(bits[b], flags, target)     # heads first
        got = O.bf16_to_f64(bf16_tensor_to_bits(k_hat[b])[:, 5:])
        err = np.abs(got - ref.k_hat)
        assert np.all(err <= _ulp_bf16(ref.k_hat) + 2.0 ** -133), \
            float((err / _ulp_bf16(ref.k_hat)).max())
        n_got = f16_tensor_to_np(norm[b])[:, 5:].astype(np.float64)
        ulp16 = np.spacing(np.abs(ref.norm).astype(np.float16)).astype(np.float64)
        assert np.all(np.abs(n_got - ref.norm) <= 2 * ulp16)
    assert torch.all(k_hat[0, :, 5 + 7] == 0) and torch.all(norm[0, :, 5 + 7] == 0)
    # a head that is zero keeps k_hat = 0; it stores the token's all-heads
    # norm under that scope, its own (zero) norm otherwise
    assert torch.all(k_hat[1, 2, 5 + 9] == 0)
    assert (norm[1, 2, 5 + 9] > 0) == bool(flags & O.NORM_ALL_HEADS)


@pytest.mark.parametrize("flags, target", VARIANTS)
def test_fused_prefill_equals_two_call_path(L, flags, target):
    from int2_kv_cache_02_gb300 import workloads as W
    B, Hkv, T = 2, 4, 320
    k = bits_to_bf16_tensor(_keys(1202, B, Hkv, 0, T))
    v = bits_to_bf16_tensor(synth.gen_bf16(1203, Hkv, range(B), range(Hkv), 0, T))
    fused = L.KVCache(B, Hkv, T, flags=flags, norm_target=target)
    split = L.KVCache(B, Hkv, T, flags=flags, norm_target=target)
    L.prefill_kv(fused, k, v, n_tok=T)
    W.prefill_two_call(split, k, v, T, chunk=96)
    _sync_ok(L)
    assert torch.equal(fused.packed, split.packed)


@pytest.mark.parametrize("g", [1, 4, 8])
@pytest.mark.parametrize("flags, target", VARIANTS)
def test_decode_over_oracle_cache(L, g, flags, target):
    B, Hkv = 2, 4       # heads 4^-h apart: the smallest k_hat ~1/64 of unit norm
    Hq = Hkv * g
    T, P = 1024 + 77, 1024
    k = _keys(1204, B, Hkv, 0, T)
    v = synth.gen_bf16(1205, Hkv, range(B), range(Hkv), 0, T,
                       tok_factor=synth.sink_token_factors(B, 0, T))
    heads = {}
    for b in range(B):
        for h, hc in enumerate(O.build_row_caches(k[b], v[b], P, flags, target)):
            heads[(b, h)] = hc
    cache = upload_oracle_cache(L.KVCache(B, Hkv, P), heads, flags, target)
    qbits = synth.gen_bf16(1206, Hq, range(B), range(Hq), 0, 1)[:, :, 0]
    qrot = O.rotate_q(qbits, flags)
    qr = torch.from_numpy(qrot.astype(np.float32)).cuda()
    for S in (0, 3):
        ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, P, S))
        out = torch.full((B, Hq, 128), float("nan"), device="cuda")
        L.decode_attention(cache, qr, Hq, TAU, out, ws, num_splits=S)
        _sync_ok(L)
        got = out.cpu().numpy()
        for b in range(B):
            ref = np.concatenate([heads[(b, h)].decode(qrot[b, h * g:(h + 1) * g], TAU)
                                  for h in range(Hkv)])
            assert_attention_close(got[b], ref, f"b={b} S={S}")


@pytest.mark.parametrize("flags, target", [(O.NORM_ALL_HEADS, 1.0), (O.NORM_ALL_HEADS, 0.37)])
def test_pipeline_prefill_append_decode(L, flags, target):
    """GPU prefill of a prompt, then streaming appends across a flush, then
    decode; the oracle runs its own pipeline on the same draws."""
    B, Hkv, g = 2, 4, 4
    Hq = Hkv * g
    P0, steps = 512, 200
    T = P0 + steps
    kb = _keys(1207, B, Hkv, 0, T)
    vb = synth.gen_bf16(1208, Hkv, range(B), range(Hkv), 0, T)
    k, v = bits_to_bf16_tensor(kb), bits_to_bf16_tensor(vb)
    cache = L.KVCache(B, Hkv, 1024, flags=flags, norm_target=target)
    L.prefill_kv(cache, k, v, n_tok=P0)
    for t in range(P0, T):
        L.append_kv(cache, k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous(), n_tok=1)
    _sync_ok(L)
    oracle = []
    for b in range(B):
        row = O.build_row_caches(kb[b, :, :P0], vb[b, :, :P0], P0, flags, target)
        for t in range(P0, T):
            O.append_row(row, kb[b, :, t], vb[b, :, t])
        oracle.append(row)
    assert cache.n_packed == oracle[0][0].n_packed and cache.n_res == oracle[0][0].n_res
    for b in range(B):
        for h in range(Hkv):
            hc = oracle[b][h]
            # every key code traced to its inputs (the all-heads norm reads
            # the token's keys in every head)
            rows_k = kb[b] if flags & O.NORM_ALL_HEADS else kb[b, h]
            rows_v = vb[b] if flags & O.NORM_ALL_HEADS else vb[b, h]
            traced_key_check(L, cache, b, h, rows_k, rows_v, hc, flags=flags, target=target,
                             what=f"flags {flags} target {target} row {(b, h)}")
            gotv = cache.field("v_codes")[b, h, :cache.n_packed // 32].cpu().numpy()
            assert np.array_equal(gotv.reshape(-1).view(np.uint32),
                                  O.pack_v_words(hc.packed_v().codes).reshape(-1))
    qbits = synth.gen_bf16(1209, Hq, range(B), range(Hq), 0, 1)[:, :, 0]
    qrot = O.rotate_q(qbits, flags)
    qr = torch.from_numpy(qrot.astype(np.float32)).cuda()
    ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, cache.n_packed, 0))
    out = torch.empty((B, Hq, 128), device="cuda")
    L.decode_attention(cache, qr, Hq, TAU, out, ws)
    _sync_ok(L)
    got = out.cpu().numpy()
    for b in range(B):
        ref = np.concatenate([oracle[b][h].decode(qrot[b, h * g:(h + 1) * g], TAU)
                              for h in range(Hkv)])
        assert_attention_close(got[b], ref, f"b={b}")
