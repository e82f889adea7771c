"""The fused prefill (oscar_prefill_kv: rotation, scaling, quantisation and
packing in one pass) against the two-call path (oscar_rotate_scale_k into a
bf16 staging buffer, then oscar_quantize_kv), whose two steps the parity
gates check against the oracle one by one.  Both paths run the same
per-token arithmetic, so every byte of the packed cache must agree.  The
full-size pipeline tests in test_gpu_parity.py build their caches through
the fused path and compare codes and attention with the oracle.
"""
import numpy as np
import pytest
import torch

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth, workloads as W
from tests._gpu_helpers import bits_to_bf16_tensor, traced_key_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from int2_kv_cache_02_gb300 import _build
    _build.build()
    from int2_kv_cache_02_gb300 import oscar
    return oscar


def _both(L, wl, flags=0):
    K, V = W.draw_kv_cuda(wl, 0, wl.T0)
    fused = W.build_cache_cuda(wl, K, V, flags=flags, fused=True)
    split = W.build_cache_cuda(wl, K, V, flags=flags, fused=False)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    assert fused.n_packed == split.n_packed and fused.n_res == split.n_res
    return fused, split


def test_fused_prefill_equals_two_call_path(L):
    fused, split = _both(L, W.WORKLOADS["qwen3_8b_32k"])
    assert torch.equal(fused.packed, split.packed)
    assert torch.equal(fused.k_res, split.k_res) and torch.equal(fused.v_res, split.v_res)


@pytest.mark.parametrize("flags", [O.NO_ROTATE, O.NO_SCALE, O.NO_ROTATE | O.NO_SCALE])
def test_fused_prefill_ablation_flags(L, flags):
    fused, split = _both(L, W.WORKLOADS["tiny_1k"], flags=flags)
    assert torch.equal(fused.packed, split.packed)


def test_fused_prefill_strided_rows_and_offset(L):
    """Two calls into one cache (the second at packed offset 64), sources
    whose rows hold more tokens than are quantised."""
    B, Hkv, T = 2, 3, 160
    k = synth.gen_bf16(970, Hkv, range(B), range(Hkv), 0, T,
                       chan_factor=synth.channel_factors([5, 38], 20.0))
    v = synth.gen_bf16(971, Hkv, range(B), range(Hkv), 0, T)
    kd, vd = bits_to_bf16_tensor(k), bits_to_bf16_tensor(v)
    cache = L.KVCache(B, Hkv, 256)
    L.prefill_kv(cache, kd, vd, n_tok=64, in_T=T)
    L.prefill_kv(cache, kd[:, :, 64:].contiguous(), vd[:, :, 64:].contiguous(), n_tok=96)
    torch.cuda.synchronize()
    assert cache.n_packed == 160 and L.device_status() == 0
    for b in range(B):
        for h in range(Hkv):
            hc = O.build_head_cache(k[b, h], v[b, h], 160)
            # every key code traced to its inputs: groups whose k_hat agrees
            # with the oracle's are bit-exact, the rest are what the GPU
            # quantiser gives for the GPU's own k_hat
            traced_key_check(L, cache, b, h, k[b, h], v[b, h], hc, what=f"row {(b, h)}")
            gotv = cache.field("v_codes")[b, h, :5].cpu().numpy().view(np.uint32)
            assert np.array_equal(gotv.reshape(-1),
                                  O.pack_v_words(hc.packed_v().codes).reshape(-1))
