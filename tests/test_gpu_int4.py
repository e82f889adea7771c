"""The INT4 option (16 levels, the 4800-byte record) on the GPU against the
oracle.  The pages fix only INT2 ("OScaR：面向大模型及多模态LLM极限KV缓存量化的
奥卡姆剃刀", 局限与改进 (1), names other widths as unstudied); the quantiser is
the same min-max formula with (max - min)/15 as the step.

* Quantisation gate: codes, every record's step / zero, norms and value
  parameters bit-exact on identical bf16 inputs, with a planted constant
  group and exact ties at every half level, at key groups of 32 and 128.
* The fused prefill equals the two-call path byte for byte.
* Attention gate over oracle-built INT4 caches for g in {1, 4, 8}, split
  counts {planned, 3}, with the per-head and the all-heads norm; the
  lossless 16-level case against plain attention; the GPU pipeline
  (prefill + appends across a flush + decode) against the oracle's; the
  paged cache equal to the contiguous one.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth
from tests._gpu_helpers import (TAU, assert_attention_close, bits_to_bf16_tensor,
                                code_mismatches, traced_key_check, upload_oracle_cache)

pytestmark = pytest.mark.gpu
LEVELS16 = np.arange(16) - 7.5


@pytest.fixture(scope="module")
def L():
    from int2_kv_cache_02_gb300 import _build
    _build.build()
    from int2_kv_cache_02_gb300 import oscar
    return oscar


def _sync_ok(L):
    torch.cuda.synchronize()
    assert L.device_status() == 0


@pytest.mark.parametrize("g", [32, 128])
def test_quantize_bit_exact(L, g):
    B, H, T = 2, 2, max(160, 2 * g)
    T = T // g * g
    cf = synth.channel_factors([5, 38, 77, 110], 15.0)
    tf = synth.sink_token_factors(B, 0, T)
    kraw = synth.gen_bf16(1401, H, range(B), range(H), 0, T, chan_factor=cf, tok_factor=tf)
    vraw = synth.gen_bf16(1402, H, range(B), range(H), 0, T, tok_factor=tf)
    rk = O.rotate_scale_k(kraw)
    khat, vb = rk.k_hat_bf16.copy(), vraw.copy()
    khat[1, 1, g:2 * g, 3] = O.f64_to_bf16(np.full(g, 0.25))          # constant key group
    ties = np.resize(np.arange(31) * 0.5, g)                          # 0, 0.5, ..., 15: every tie
    ties[0], ties[1] = 0.0, 15.0
    khat[1, 1, 0:g, 9] = O.f64_to_bf16(ties)
    vb[1, 1, 5, :] = O.f64_to_bf16(np.full(128, -0.75))                 # constant value token
    vb[1, 1, 6, :] = O.f64_to_bf16(np.resize(np.arange(31) * 0.5, 128))  # value ties
    # steps of 2^-133 (the reciprocal overflows fp32): a key channel, a value token
    tiny = np.resize(np.arange(16.0), 128) * 2.0 ** -133
    khat[0, 1, 0:g, 17] = O.f64_to_bf16(tiny[:g])
    vb[0, 1, 9, :] = O.f64_to_bf16(tiny)
    cache = L.KVCache(B, H, T + 128, key_group=g, bits=4)
    L.quantize_kv(cache, bits_to_bf16_tensor(khat), torch.from_numpy(rk.norm_f16).cuda(),
                  bits_to_bf16_tensor(vb), src_T=T, n_tok=g)
    L.quantize_kv(cache, bits_to_bf16_tensor(np.ascontiguousarray(khat[:, :, g:])),
                  torch.from_numpy(np.ascontiguousarray(rk.norm_f16[:, :, g:])).cuda(),
                  bits_to_bf16_tensor(np.ascontiguousarray(vb[:, :, g:])), src_T=T - g,
                  n_tok=T - g)
    _sync_ok(L)
    assert cache.n_packed == T
    for b in range(B):
        for h in range(H):
            kq, vq = O.quantize_k(khat[b, h], g, bits=4), O.quantize_v(vb[b, h], bits=4)
            np.testing.assert_array_equal(
                cache.tokens("k_codes")[b, h, :T].cpu().numpy().view(np.uint32),
                O.pack_k_words4(kq.codes))
            np.testing.assert_array_equal(
                cache.field("v_codes")[b, h, :T // 32].cpu().numpy().view(np.uint32),
                O.pack_v_words4(vq.codes))
            ks16, kz16 = kq.block_params()
            for name, want in [("k_scale", ks16), ("k_zero", kz16)]:
                got = cache.field(name)[b, h, :T // 32].cpu().numpy()
                np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))
            for name, want in [("v_scale", vq.step16), ("v_zero", vq.zero16),
                               ("k_norm", rk.norm_f16[b, h])]:
                got = cache.tokens(name)[b, h, :T].cpu().numpy()
                np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))
    assert int(O.quantize_k(khat[1, 1], g, bits=4).codes.max()) == 15


@pytest.mark.parametrize("flags", [0, O.NORM_ALL_HEADS])
def test_fused_prefill_equals_two_call_path(L, flags):
    from int2_kv_cache_02_gb300 import workloads as W
    B, Hkv, T = 2, 4, 320
    cf = synth.channel_factors([5, 38], 20.0)
    k = bits_to_bf16_tensor(synth.gen_bf16(1403, Hkv, range(B), range(Hkv), 0, T, chan_factor=cf))
    v = bits_to_bf16_tensor(synth.gen_bf16(1404, Hkv, range(B), range(Hkv), 0, T))
    fused = L.KVCache(B, Hkv, T, flags=flags, bits=4)
    split = L.KVCache(B, Hkv, T, flags=flags, bits=4)
    L.prefill_kv(fused, k, v, n_tok=T)
    W.prefill_two_call(split, k, v, T, chunk=96)
    _sync_ok(L)
    assert torch.equal(fused.packed, split.packed)


@pytest.mark.parametrize("g", [1, 4, 8])
@pytest.mark.parametrize("flags", [0, O.NORM_ALL_HEADS])
def test_decode_over_oracle_cache(L, g, flags):
    B, Hkv = 2, 2
    Hq = Hkv * g
    T, P = 1024 + 77, 1024
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    tf = synth.sink_token_factors(B, 0, T)
    k = synth.gen_bf16(1405, Hkv, range(B), range(Hkv), 0, T, chan_factor=cf, tok_factor=tf)
    v = synth.gen_bf16(1406, Hkv, range(B), range(Hkv), 0, T, tok_factor=tf)
    heads = {}
    for b in range(B):
        for h, hc in enumerate(O.build_row_caches(k[b], v[b], P, flags, bits=4)):
            heads[(b, h)] = hc
    cache = upload_oracle_cache(L.KVCache(B, Hkv, P, bits=4), heads, flags)
    qbits = synth.gen_bf16(1407, Hq, range(B), range(Hq), 0, 1)[:, :, 0]
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


def test_lossless_equals_plain_attention(L):
    """Both ablation flags on, every group holding only the 16 exact levels:
    INT4 storage is exact, so the decode must match fp64 attention on the
    bf16 K, V to within fp32 accumulation."""
    flags = O.NO_ROTATE | O.NO_SCALE
    B, Hkv, g = 1, 2, 4
    Hq = Hkv * g
    T, P = 1024 + 40, 1024
    r = synth.splitmix64(1408, np.arange(2 * Hkv * T * 128)).reshape(2, Hkv, T, 128)
    k = LEVELS16[(r[0] % np.uint64(16)).astype(np.int64)]
    v = LEVELS16[(r[1] % np.uint64(16)).astype(np.int64)]
    k[:, 0::32, :], k[:, 1::32, :] = -7.5, 7.5
    v[:, :, 0], v[:, :, 1] = -7.5, 7.5
    kb, vb = O.f64_to_bf16(k), O.f64_to_bf16(v)
    heads = {(0, h): O.build_head_cache(kb[h], vb[h], P, flags, bits=4) for h in range(Hkv)}
    cache = upload_oracle_cache(L.KVCache(B, Hkv, P, flags=flags, bits=4), heads, flags)
    q = synth.gen_bf16(1409, Hq, [0], range(Hq), 0, 1)[0, :, 0]
    qr = torch.from_numpy(O.rotate_q(q, flags)[None].astype(np.float32)).cuda()
    ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, P, 0))
    out = torch.empty((B, Hq, 128), device="cuda")
    L.decode_attention(cache, qr, Hq, TAU, out, ws)
    _sync_ok(L)
    got = out.cpu().numpy()[0]
    for h in range(Hkv):
        want = O.bf16_attention(q[h * g:(h + 1) * g], kb[h], vb[h], TAU)
        assert np.abs(got[h * g:(h + 1) * g] - want).max() <= 1e-4


def test_pipeline_prefill_append_decode(L):
    B, Hkv, gq = 2, 2, 4
    Hq = Hkv * gq
    P0, steps = 384, 200
    T = P0 + steps
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    tf = synth.sink_token_factors(B, 0, T)
    kb = synth.gen_bf16(1410, Hkv, range(B), range(Hkv), 0, T, chan_factor=cf, tok_factor=tf)
    vb = synth.gen_bf16(1411, Hkv, range(B), range(Hkv), 0, T, tok_factor=tf)
    k, v = bits_to_bf16_tensor(kb), bits_to_bf16_tensor(vb)
    cache = L.KVCache(B, Hkv, 1024, bits=4)
    L.prefill_kv(cache, k, v, n_tok=P0)
    for t in range(P0, T):
        L.append_kv(cache, k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous(), n_tok=1)
    _sync_ok(L)
    heads = {}
    for b in range(B):
        for h in range(Hkv):
            hc = O.build_head_cache(kb[b, h, :P0], vb[b, h, :P0], P0, bits=4)
            for t in range(P0, T):
                hc.append(kb[b, h, t], vb[b, h, t])
            heads[(b, h)] = hc
    assert (cache.n_packed, cache.n_res) == (heads[(0, 0)].n_packed, heads[(0, 0)].n_res)
    for (b, h), hc in heads.items():
        # every key code traced to its inputs (16 levels)
        traced_key_check(L, cache, b, h, kb[b, h], vb[b, h], hc, bits=4,
                         what=f"INT4 row {(b, h)}")
        gotv = cache.field("v_codes")[b, h, :cache.n_packed // 32].cpu().numpy()
        assert np.array_equal(gotv.reshape(-1).view(np.uint32),
                              O.pack_v_words4(hc.packed_v().codes).reshape(-1))
    qbits = synth.gen_bf16(1412, Hq, range(B), range(Hq), 0, 1)[:, :, 0]
    qrot = O.rotate_q(qbits)
    qr = torch.from_numpy(qrot.astype(np.float32)).cuda()
    ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, cache.n_packed, 0))
    out = torch.empty((B, Hq, 128), device="cuda")
    L.decode_attention(cache, qr, Hq, TAU, out, ws)
    _sync_ok(L)
    got = out.cpu().numpy()
    for b in range(B):
        ref = np.concatenate([heads[(b, h)].decode(qrot[b, h * gq:(h + 1) * gq], TAU)
                              for h in range(Hkv)])
        assert_attention_close(got[b], ref, f"b={b}")


def test_paged_equals_contiguous(L):
    Hkv = 2
    prompts = [(256, 30), (96, 0)]
    steps = 140
    B = len(prompts)
    T_all = max(p + a for p, a in prompts) + steps
    k = synth.gen_bf16(1413, Hkv, range(B), range(Hkv), 0, T_all,
                       chan_factor=synth.channel_factors([5, 38], 20.0))
    v = synth.gen_bf16(1414, Hkv, range(B), range(Hkv), 0, T_all)
    kd, vd = bits_to_bf16_tensor(k), bits_to_bf16_tensor(v)
    max_blocks = (T_all + 255) // 32 + 8
    paged = L.PagedKVCache(B, Hkv, max_blocks, n_pages=B * max_blocks, bits=4)
    rng = np.random.default_rng(11)
    paged.map_blocks(0, 0, order=list(rng.permutation(B * max_blocks)))
    for b in range(B):
        paged.map_blocks(b, max_blocks)
    n_tok = torch.tensor([p for p, _ in prompts], dtype=torch.int32, device="cuda")
    L.paged_prefill_kv(paged, kd, vd, n_tok, max(p for p, _ in prompts), in_T=T_all)
    conts = []
    for b, (p, _) in enumerate(prompts):
        c = L.KVCache(1, Hkv, max_blocks * 32, bits=4)
        L.prefill_kv(c, kd[b:b + 1].contiguous(), vd[b:b + 1].contiguous(), n_tok=p, in_T=T_all)
        conts.append(c)
    pos = [p for p, _ in prompts]
    end = [p + a + steps for p, a in prompts]
    while any(pos[b] < end[b] for b in range(B)):
        act = [1 if pos[b] < end[b] else 0 for b in range(B)]
        kn = torch.stack([kd[b, :, min(pos[b], T_all - 1)] for b in range(B)]).contiguous()
        vn = torch.stack([vd[b, :, min(pos[b], T_all - 1)] for b in range(B)]).contiguous()
        L.paged_append_kv(paged, kn, vn, torch.tensor(act, dtype=torch.int32, device="cuda"))
        for b in range(B):
            if act[b]:
                L.append_kv(conts[b], kn[b:b + 1].contiguous(), vn[b:b + 1].contiguous(), n_tok=1)
                pos[b] += 1
    _sync_ok(L)
    n_packed, n_res = paged.lengths()
    for b in range(B):
        c = conts[b]
        assert (n_packed[b], n_res[b]) == (c.n_packed, c.n_res), b
        for h in range(Hkv):
            for j in range(c.n_packed // 32):
                assert torch.equal(paged.record(b, h, j), c.packed[0, h, j]), (b, h, j)
    # and the paged decode reads INT4 pages: equal to the contiguous decode
    Hq = 4 * Hkv
    qr = torch.randn((B, Hq, 128), generator=torch.Generator().manual_seed(3)).cuda()
    maxp = max(c.n_packed for c in conts)
    ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, maxp, 0))
    out = torch.empty((B, Hq, 128), device="cuda")
    L.paged_decode_attention(paged, qr, Hq, TAU, maxp, out, ws)
    for b in range(B):
        ws1 = L.alloc_workspace(L.decode_workspace_bytes(1, Hkv, Hq, conts[b].n_packed, 0))
        o1 = torch.empty((1, Hq, 128), device="cuda")
        L.decode_attention(conts[b], qr[b:b + 1].contiguous(), Hq, TAU, o1, ws1)
        _sync_ok(L)
        assert torch.allclose(out[b], o1[0], rtol=0, atol=1e-5)
