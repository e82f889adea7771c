"""Larger key groups (64 and 128 tokens sharing a channel's step and zero) on
the GPU against the oracle ("OScaR：面向大模型及多模态LLM极限KV缓存量化的
奥卡姆剃刀", 局限与改进 (1): larger groups as the untested direction; 方法步骤
详情 (2): the per-channel block quantisation).

* Quantisation gate: on identical bf16 inputs (with planted constant
  groups and exact ties) codes, every record's step / zero (the group's,
  repeated over its 32-token records), norms and value parameters are
  bit-exact; quantised in two calls so the packed offset is exercised.
* The fused prefill equals the two-call path byte for byte.
* Attention gate over a cache the GPU built by prefill + streaming appends
  across flushes, against the oracle's pipeline on the same draws; the
  paged cache equals the contiguous one under the same group size.
"""
import numpy as np
import pytest
import torch

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth
from tests._gpu_helpers import (TAU, assert_attention_close, bits_to_bf16_tensor,
                                code_mismatches, traced_key_check)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from int2_kv_cache_02_gb300 import _build
    _build.build()
    from int2_kv_cache_02_gb300 import oscar
    return oscar


def _sync_ok(L):
    torch.cuda.synchronize()
    assert L.device_status() == 0


def _planted(khat, vb, g):
    """A constant key group and exact ties inside the second group."""
    kb, vv = khat.copy(), vb.copy()
    kb[g:2 * g, 3] = O.f64_to_bf16(np.full(g, 0.25))
    ties = np.resize(np.array([0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 3.0]), g)
    kb[g:2 * g, 9] = O.f64_to_bf16(ties)
    vv[5, :] = O.f64_to_bf16(np.full(128, -0.75))
    return kb, vv


@pytest.mark.parametrize("g", [64, 128])
def test_quantize_bit_exact(L, g):
    B, H, T = 2, 2, 3 * g
    cf = synth.channel_factors([5, 38, 77, 110], 15.0)
    tf = synth.sink_token_factors(B, 0, T)
    kraw = synth.gen_bf16(1301, H, range(B), range(H), 0, T, chan_factor=cf, tok_factor=tf)
    vraw = synth.gen_bf16(1302, H, range(B), range(H), 0, T, tok_factor=tf)
    rk = O.rotate_scale_k(kraw)
    khat, vb = rk.k_hat_bf16.copy(), vraw.copy()
    khat[1, 1], vb[1, 1] = _planted(khat[1, 1], vb[1, 1], g)
    cache = L.KVCache(B, H, T + 128, key_group=g)
    norm = torch.from_numpy(rk.norm_f16).cuda()
    L.quantize_kv(cache, bits_to_bf16_tensor(khat), norm, bits_to_bf16_tensor(vb), src_T=T,
                  n_tok=g)
    L.quantize_kv(cache, bits_to_bf16_tensor(np.ascontiguousarray(khat[:, :, g:])),
                  torch.from_numpy(np.ascontiguousarray(rk.norm_f16[:, :, g:])).cuda(),
                  bits_to_bf16_tensor(np.ascontiguousarray(vb[:, :, g:])), src_T=T - g,
                  n_tok=2 * g)
    _sync_ok(L)
    assert cache.n_packed == T
    for b in range(B):
        for h in range(H):
            kq, vq = O.quantize_k(khat[b, h], g), O.quantize_v(vb[b, h])
            np.testing.assert_array_equal(
                cache.tokens("k_codes")[b, h, :T].cpu().numpy().view(np.uint32),
                O.pack_k_words(kq.codes))
            np.testing.assert_array_equal(
                cache.field("v_codes")[b, h, :T // 32].cpu().numpy().view(np.uint32),
                O.pack_v_words(vq.codes))
            ks16, kz16 = kq.block_params()
            for name, want in [("k_scale", ks16), ("k_zero", kz16)]:
                got = cache.field(name)[b, h, :T // 32].cpu().numpy()
                np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))
            for name, want in [("v_scale", vq.step16), ("v_zero", vq.zero16),
                               ("k_norm", rk.norm_f16[b, h])]:
                got = cache.tokens(name)[b, h, :T].cpu().numpy()
                np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))
            assert torch.all(cache.packed[b, h, T // 32:] == 0)


@pytest.mark.parametrize("g, flags", [(64, 0), (128, 0), (128, O.NORM_ALL_HEADS)])
def test_fused_prefill_equals_two_call_path(L, g, flags):
    from int2_kv_cache_02_gb300 import workloads as W
    B, Hkv, T = 2, 4, 512
    cf = synth.channel_factors([5, 38], 20.0)
    k = bits_to_bf16_tensor(synth.gen_bf16(1303, Hkv, range(B), range(Hkv), 0, T, chan_factor=cf))
    v = bits_to_bf16_tensor(synth.gen_bf16(1304, Hkv, range(B), range(Hkv), 0, T))
    fused = L.KVCache(B, Hkv, T, flags=flags, key_group=g)
    split = L.KVCache(B, Hkv, T, flags=flags, key_group=g)
    L.prefill_kv(fused, k, v, n_tok=T)
    W.prefill_two_call(split, k, v, T, chunk=2 * g)
    _sync_ok(L)
    assert torch.equal(fused.packed, split.packed)


@pytest.mark.parametrize("g", [64, 128])
def test_pipeline_prefill_append_decode(L, g):
    """Prefill of a prompt, streaming appends across two flushes, decode; the
    oracle runs its own pipeline on the same draws with the same group."""
    B, Hkv, gq = 2, 2, 4
    Hq = Hkv * gq
    P0, steps = 2 * g + 128, 300
    T = P0 + steps
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    tf = synth.sink_token_factors(B, 0, T)
    kb = synth.gen_bf16(1305, Hkv, range(B), range(Hkv), 0, T, chan_factor=cf, tok_factor=tf)
    vb = synth.gen_bf16(1306, Hkv, range(B), range(Hkv), 0, T, tok_factor=tf)
    k, v = bits_to_bf16_tensor(kb), bits_to_bf16_tensor(vb)
    cache = L.KVCache(B, Hkv, 1024, key_group=g)
    L.prefill_kv(cache, k, v, n_tok=P0)
    for t in range(P0, T):
        L.append_kv(cache, k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous(), n_tok=1)
    _sync_ok(L)
    heads = {}
    for b in range(B):
        for h in range(Hkv):
            hc = O.build_head_cache(kb[b, h, :P0], vb[b, h, :P0], P0, group=g)
            for t in range(P0, T):
                hc.append(kb[b, h, t], vb[b, h, t])
            heads[(b, h)] = hc
    hc0 = heads[(0, 0)]
    assert (cache.n_packed, cache.n_res) == (hc0.n_packed, hc0.n_res)
    assert cache.n_packed == P0 + 256
    for (b, h), hc in heads.items():
        # every key code traced to its inputs (groups of g tokens)
        traced_key_check(L, cache, b, h, kb[b, h], vb[b, h], hc, what=f"G={g} row {(b, h)}")
        gotv = cache.field("v_codes")[b, h, :cache.n_packed // 32].cpu().numpy()
        assert np.array_equal(gotv.reshape(-1).view(np.uint32),
                              O.pack_v_words(hc.packed_v().codes).reshape(-1))
    qbits = synth.gen_bf16(1307, Hq, range(B), range(Hq), 0, 1)[:, :, 0]
    qrot = O.rotate_q(qbits)
    qr = torch.from_numpy(qrot.astype(np.float32)).cuda()
    for S in (0, 3):
        ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, cache.n_packed, S))
        out = torch.empty((B, Hq, 128), device="cuda")
        L.decode_attention(cache, qr, Hq, TAU, out, ws, num_splits=S)
        _sync_ok(L)
        got = out.cpu().numpy()
        for b in range(B):
            ref = np.concatenate([heads[(b, h)].decode(qrot[b, h * gq:(h + 1) * gq], TAU)
                                  for h in range(Hkv)])
            assert_attention_close(got[b], ref, f"b={b} S={S}")


def test_paged_prefill_and_append_equal_contiguous(L):
    g, Hkv = 128, 2
    prompts = [(256, 30), (128, 0), (0, 0)]
    steps = 140
    B = len(prompts)
    T_all = max(p + a for p, a in prompts) + steps
    k = synth.gen_bf16(1308, Hkv, range(B), range(Hkv), 0, T_all,
                       chan_factor=synth.channel_factors([5, 38], 20.0))
    v = synth.gen_bf16(1309, Hkv, range(B), range(Hkv), 0, T_all)
    kd, vd = bits_to_bf16_tensor(k), bits_to_bf16_tensor(v)
    max_blocks = (T_all + 255) // 32 + 8
    paged = L.PagedKVCache(B, Hkv, max_blocks, n_pages=B * max_blocks, key_group=g)
    rng = np.random.default_rng(9)
    paged.map_blocks(0, 0, order=list(rng.permutation(B * max_blocks)))
    for b in range(B):
        paged.map_blocks(b, max_blocks)
    n_tok = torch.tensor([p for p, _ in prompts], dtype=torch.int32, device="cuda")
    L.paged_prefill_kv(paged, kd, vd, n_tok, max(p for p, _ in prompts), in_T=T_all)
    conts = []
    for b, (p, _) in enumerate(prompts):
        c = L.KVCache(1, Hkv, max_blocks * 32, key_group=g)
        if p:
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
            r = c.n_res
            assert torch.equal(paged.k_res[b, h, :r], c.k_res[0, h, :r])
