"""A decode step over the paged cache captured in a CUDA graph.

The paged cache keeps its per-sequence lengths in device memory and the
library's calls only enqueue work on the caller's stream, so one decode
step (rotate the query, append the new token with its flush, decode and
combine) can be captured once and replayed: every replay advances the
lengths on the device.  The replayed steps must give bit-for-bit the outputs
of the same steps run eagerly, across residual flushes.
"""
import numpy as np
import pytest
import torch

from int2_kv_cache_02_gb300 import synth
from tests._gpu_helpers import TAU, bits_to_bf16_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from int2_kv_cache_02_gb300 import _build
    _build.build()
    from int2_kv_cache_02_gb300 import oscar
    return oscar


def _make(L, B, Hkv, T_pre, max_blocks, kd, vd):
    c = L.PagedKVCache(B, Hkv, max_blocks, n_pages=B * max_blocks)
    for b in range(B):
        c.map_blocks(b, max_blocks)
    n_tok = torch.full((B,), T_pre, dtype=torch.int32, device="cuda")
    L.paged_prefill_kv(c, kd, vd, n_tok, T_pre)
    return c


def test_paged_decode_step_in_a_cuda_graph(L):
    B, Hkv, g = 3, 2, 4
    Hq = Hkv * g
    T_pre, steps = 256, 260                       # two residual flushes on the way
    T_all = T_pre + steps
    kb = synth.gen_bf16(1501, Hkv, range(B), range(Hkv), 0, T_all,
                        chan_factor=synth.channel_factors([5, 38], 20.0))
    vb = synth.gen_bf16(1502, Hkv, range(B), range(Hkv), 0, T_all)
    qb = synth.gen_bf16(1503, Hq, range(B), range(Hq), 0, steps)
    kd, vd = bits_to_bf16_tensor(kb), bits_to_bf16_tensor(vb)
    qd = bits_to_bf16_tensor(qb)                  # [B][Hq][steps][128]
    max_blocks = (T_all + 128) // 32 + 4
    max_packed = (max_blocks - 4) * 32
    S = L.decode_num_splits(B, Hkv, Hq, max_packed)
    ws_bytes = L.decode_workspace_bytes(B, Hkv, Hq, max_packed, S)

    def step(c, q, k_new, v_new, qr, out, ws):
        L.rotate_q(q, qr)
        L.paged_append_kv(c, k_new, v_new)
        L.paged_decode_attention(c, qr, Hq, TAU, max_packed, out, ws, num_splits=S)

    # eager
    ce = _make(L, B, Hkv, T_pre, max_blocks, kd, vd)
    qr = torch.empty((B, Hq, 128), device="cuda")
    out = torch.empty((B, Hq, 128), device="cuda")
    ws = L.alloc_workspace(ws_bytes)
    eager = []
    for i in range(steps):
        step(ce, qd[:, :, i].contiguous(), kd[:, :, T_pre + i].contiguous(),
             vd[:, :, T_pre + i].contiguous(), qr, out, ws)
        eager.append(out.clone())
    torch.cuda.synchronize()
    assert L.device_status() == 0

    # captured once, replayed with the inputs copied into static buffers
    cg = _make(L, B, Hkv, T_pre, max_blocks, kd, vd)
    q_s = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    k_s = torch.empty((B, Hkv, 128), dtype=torch.bfloat16, device="cuda")
    v_s = torch.empty_like(k_s)
    qr_g = torch.empty((B, Hq, 128), device="cuda")
    out_g = torch.empty((B, Hq, 128), device="cuda")
    ws_g = L.alloc_workspace(ws_bytes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(cg, q_s, k_s, v_s, qr_g, out_g, ws_g)
    # capturing enqueues nothing: the cache is still at its prefill state
    n_packed, n_res = cg.lengths()
    assert n_packed == [T_pre] * B and n_res == [0] * B
    for i in range(steps):
        q_s.copy_(qd[:, :, i])
        k_s.copy_(kd[:, :, T_pre + i])
        v_s.copy_(vd[:, :, T_pre + i])
        graph.replay()
        assert torch.equal(out_g, eager[i]), i
    torch.cuda.synchronize()
    assert L.device_status() == 0
    assert cg.lengths() == ce.lengths()
    n_packed, n_res = cg.lengths()
    assert n_packed[0] == T_pre + 256 and n_res[0] == steps - 256
