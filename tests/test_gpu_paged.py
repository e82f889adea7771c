"""The paged cache (oscar_paged_cache): sequences of different lengths whose
32-token blocks sit in pages of a shared pool, found through a block table.

* Decode against the oracle: per-sequence oracle caches (different packed
  and residual lengths, an empty sequence, a residual-only one) are written
  into pages in a shuffled order; every sequence's attention must match the
  oracle's within the attention gate.
* Prefill and append against the contiguous calls: each sequence is also
  built alone in an oscar_cache with oscar_prefill_kv / oscar_append_kv (the
  paths the parity gates check against the oracle); every record reached
  through the block table, every residual slot and every length must be
  identical.
* A page id outside the pool is reported in the status word; nothing
  outside the pool is read.
"""
import numpy as np
import pytest
import torch

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth
from tests._gpu_helpers import (TAU, assert_attention_close, bits_to_bf16_tensor)

pytestmark = pytest.mark.gpu

DEVICE_STATUS = 7


@pytest.fixture(scope="module")
def L():
    from int2_kv_cache_02_gb300 import _build
    _build.build()
    from int2_kv_cache_02_gb300 import oscar
    return oscar


def _per_token(a):
    """A block's per-token array [32] in the record's order 4*(t%8) + t//8."""
    return np.ascontiguousarray(np.asarray(a).reshape(4, 8).T.reshape(32))


def _write_record(rec, kq, vq, norm16, j):
    """Block j of an oracle head cache into a 2752-byte record view."""
    t = slice(32 * j, 32 * j + 32)
    ks16, kz16 = kq.block_params()
    parts = [O.pack_k_words(kq.codes[t]).reshape(-1).view(np.uint8),
             O.pack_v_words(vq.codes[t]).reshape(-1).view(np.uint8),
             ks16[j].view(np.uint8), kz16[j].view(np.uint8),
             _per_token(norm16[t]).view(np.uint8),
             _per_token(vq.step16[t]).view(np.uint8), _per_token(vq.zero16[t]).view(np.uint8)]
    rec.copy_(torch.from_numpy(np.concatenate(parts)))


@pytest.mark.parametrize("g", [1, 3, 4, 8, 16])
def test_paged_decode_matches_oracle(L, g):
    Hkv = 2
    Hq = Hkv * g
    lens = [(1024 + 40, 1024), (2336 + 128, 2336), (100, 0), (0, 0), (320 + 1, 320)]
    B = len(lens)
    max_blocks = 80
    cache = L.PagedKVCache(B, Hkv, max_blocks, n_pages=200)
    rng = np.random.default_rng(5)
    order = list(rng.permutation(200))
    heads = {}
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    for b, (T, P) in enumerate(lens):
        cache.map_blocks(b, P // 32, order=order if b == 0 else None)
        if T == 0:
            continue
        tf = synth.sink_token_factors(1, 0, T)
        k = synth.gen_bf16(980 + b, Hkv, [0], range(Hkv), 0, T, chan_factor=cf, tok_factor=tf)
        v = synth.gen_bf16(990 + b, Hkv, [0], range(Hkv), 0, T, tok_factor=tf)
        for h in range(Hkv):
            hc = O.build_head_cache(k[0, h], v[0, h], P)
            heads[(b, h)] = hc
            if P:
                kq, vq = hc.packed_k(), hc.packed_v()
                norm16 = hc.packed_norm16()
                for j in range(P // 32):
                    _write_record(cache.record(b, h, j), kq, vq, norm16, j)
            r = hc.n_res
            if r:
                cache.k_res[b, h, :r] = bits_to_bf16_tensor(np.stack(hc.res_k_bf16))
                cache.v_res[b, h, :r] = bits_to_bf16_tensor(np.stack(hc.res_v_bf16))
                cache.k_res_norm[b, h, :r] = torch.from_numpy(np.array(hc.res_norm16, np.float16))
    cache.n_packed_d.copy_(torch.tensor([P for _, P in lens], dtype=torch.int32))
    cache.n_res_d.copy_(torch.tensor([T - P for T, P in lens], dtype=torch.int32))
    qbits = synth.gen_bf16(999, Hq, range(B), range(Hq), 0, 1)[:, :, 0]
    qrot = O.rotate_q(qbits, 0)
    qr = torch.from_numpy(qrot.astype(np.float32)).cuda()
    max_packed = max(P for _, P in lens)
    for S in (0, 1, 5):
        ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, max_packed, S))
        out = torch.full((B, Hq, 128), float("nan"), device="cuda")
        L.paged_decode_attention(cache, qr, Hq, TAU, max_packed, out, ws, num_splits=S)
        torch.cuda.synchronize()
        assert L.device_status() == 0
        got = out.cpu().numpy()
        for b, (T, P) in enumerate(lens):
            if T == 0:
                assert np.all(got[b] == 0)
                continue
            ref = np.concatenate([heads[(b, h)].decode(qrot[b, h * g:(h + 1) * g], TAU)
                                  for h in range(Hkv)])
            assert_attention_close(got[b], ref, f"sequence {b}, splits {S}")


@pytest.mark.parametrize("flags, target", [(0, 0.0), (O.NORM_ALL_HEADS, 0.37)])
def test_paged_prefill_and_append_equal_contiguous(L, flags, target):
    Hkv = 2
    prompts = [(1024, 40), (640, 0), (0, 0), (96, 130)]   # (prefill tokens, appended tokens)
    steps = 140                                           # decode steps after the prompt
    B = len(prompts)
    T_all = max(p + a for p, a in prompts) + steps
    k = synth.gen_bf16(1100, Hkv, range(B), range(Hkv), 0, T_all,
                       chan_factor=synth.channel_factors([5, 38], 20.0))
    v = synth.gen_bf16(1101, Hkv, range(B), range(Hkv), 0, T_all)
    kd, vd = bits_to_bf16_tensor(k), bits_to_bf16_tensor(v)
    max_blocks = (T_all + 127) // 32 + 8
    paged = L.PagedKVCache(B, Hkv, max_blocks, n_pages=B * max_blocks, flags=flags,
                           norm_target=target)
    rng = np.random.default_rng(7)
    paged.map_blocks(0, 0, order=list(rng.permutation(B * max_blocks)))
    for b in range(B):
        paged.map_blocks(b, max_blocks)
    n_tok = torch.tensor([p for p, _ in prompts], dtype=torch.int32, device="cuda")
    max_tok = max(max(p for p, _ in prompts), 32)
    L.paged_prefill_kv(paged, kd, vd, n_tok, max_tok, in_T=T_all)
    conts = []
    for b, (p, a) in enumerate(prompts):
        c = L.KVCache(1, Hkv, max_blocks * 32, flags=flags, norm_target=target)
        if p:
            L.prefill_kv(c, kd[b:b + 1].contiguous(), vd[b:b + 1].contiguous(), n_tok=p, in_T=T_all)
        conts.append(c)
    # per-sequence appends: the prompt remainder, then `steps` decode tokens
    pos = [p for p, _ in prompts]
    end = [p + a + steps for p, a in prompts]
    for i in range(max(end)):
        act = [1 if pos[b] < end[b] else 0 for b in range(B)]
        if not any(act):
            break
        kn = torch.stack([kd[b, :, min(pos[b], T_all - 1)] for b in range(B)]).contiguous()
        vn = torch.stack([vd[b, :, min(pos[b], T_all - 1)] for b in range(B)]).contiguous()
        L.paged_append_kv(paged, kn, vn, torch.tensor(act, dtype=torch.int32, device="cuda"))
        for b in range(B):
            if act[b]:
                L.append_kv(conts[b], kn[b:b + 1].contiguous(), vn[b:b + 1].contiguous(), n_tok=1)
                pos[b] += 1
    torch.cuda.synchronize()
    assert L.device_status() == 0
    n_packed, n_res = paged.lengths()
    for b in range(B):
        c = conts[b]
        assert (n_packed[b], n_res[b]) == (c.n_packed, c.n_res), b
        for h in range(Hkv):
            for j in range(c.n_packed // 32):
                assert torch.equal(paged.record(b, h, j), c.packed[0, h, j]), (b, h, j)
            r = c.n_res
            assert torch.equal(paged.k_res[b, h, :r], c.k_res[0, h, :r])
            assert torch.equal(paged.v_res[b, h, :r], c.v_res[0, h, :r])
            assert torch.equal(paged.k_res_norm[b, h, :r], c.k_res_norm[0, h, :r])


def test_paged_bad_page_is_reported(L):
    B, Hkv, Hq = 1, 2, 8
    cache = L.PagedKVCache(B, Hkv, 4, n_pages=4)
    cache.map_blocks(0, 2)
    cache.block_table[0, 1] = 4          # outside the pool of 4 pages
    cache.n_packed_d.fill_(64)
    qr = torch.randn((B, Hq, 128), device="cuda")
    ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, 64, 1))
    out = torch.zeros((B, Hq, 128), device="cuda")
    L.paged_decode_attention(cache, qr, Hq, TAU, 64, out, ws, num_splits=1)
    assert L.device_status() == DEVICE_STATUS
    assert L.device_status() == 0


def test_paged_batch48_variable_lengths_sampled(L):
    """Full size, as the benchmark's paged measurement runs it: 48 sequences of
    the batch48_128k prompt cut to lengths drawn in [n/4, n], pages handed
    out in a shuffled order, one appended token each, the planned split
    count; sampled (sequence, head) rows against the oracle."""
    from int2_kv_cache_02_gb300 import workloads as W
    wl = W.WORKLOADS["batch48_128k"]
    rng = np.random.default_rng(12345)
    n_tok = [int(x) // 32 * 32 for x in rng.integers(wl.n_packed // 4, wl.n_packed + 1, size=wl.B)]
    blocks = [n // 32 + 4 for n in n_tok]
    pc = L.PagedKVCache(wl.B, wl.Hkv, max(blocks), n_pages=sum(blocks))
    pc.map_blocks(0, 0, order=list(rng.permutation(sum(blocks))))
    for b in range(wl.B):
        pc.map_blocks(b, blocks[b])
    K, V = W.draw_kv_cuda(wl, 0, wl.T0)
    L.paged_prefill_kv(pc, K, V, torch.tensor(n_tok, dtype=torch.int32, device="cuda"),
                       max(n_tok), in_T=wl.T0)
    del K, V
    Kn, Vn = W.draw_kv_cuda(wl, wl.T0, 1)
    L.paged_append_kv(pc, Kn[:, :, 0].contiguous(), Vn[:, :, 0].contiguous())
    del Kn, Vn
    q = W.draw_q_cuda(wl, 0)
    qr = torch.empty((wl.B, wl.Hq, 128), dtype=torch.float32, device="cuda")
    L.rotate_q(q, qr)
    maxp = max(n_tok)
    S = L.decode_num_splits(wl.B, wl.Hkv, wl.Hq, maxp)
    ws = L.alloc_workspace(L.decode_workspace_bytes(wl.B, wl.Hkv, wl.Hq, maxp, S))
    out = torch.empty((wl.B, wl.Hq, 128), dtype=torch.float32, device="cuda")
    L.paged_decode_attention(pc, qr, wl.Hq, TAU, maxp, out, ws, num_splits=S)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    got = out.cpu().numpy()
    g = wl.g
    shortest = int(np.argmin(n_tok))
    for b, h in [(shortest, 1), (11, 6)]:
        n = n_tok[b]
        kb = wl.k_bits([b], [h], 0, n)[0, 0]
        vb = wl.v_bits([b], [h], 0, n)[0, 0]
        hc = O.build_head_cache(kb, vb, n)
        hc.append(wl.k_bits([b], [h], wl.T0, 1)[0, 0, 0], wl.v_bits([b], [h], wl.T0, 1)[0, 0, 0])
        qbits = wl.q_bits([b], range(h * g, (h + 1) * g), 0)[0]
        ref = hc.decode(O.rotate_q(qbits), TAU)
        assert_attention_close(got[b, h * g:(h + 1) * g], ref, f"paged row {(b, h)}, n {n}")
