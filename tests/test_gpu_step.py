"""The fused decode step (oscar_decode_step) against the separate calls.

One step of the decode path is rotate_q, the append of the new token (with
the flush of a full residual window first) and the fused decode attention
("OScaR：面向大模型及多模态LLM极限KV缓存量化的奥卡姆剃刀", 方法步骤详情; news article on
arXiv 2605.19660, 三: kernels ① and ③).  oscar_decode_step does the three in
one launch, with the rotation and scaling done by the same device code, so
its outputs and the cache it leaves must equal those of rotate_q +
append_kv + decode_attention bit for bit, step after step and across
flushes.  The separate calls are themselves checked against the oracle
(test_gpu_parity.py and the other -m gpu files).
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

TAU = 128 ** -0.5


@pytest.fixture(scope="module")
def L():
    from int2_kv_cache_02_gb300 import _build
    _build.build()
    from int2_kv_cache_02_gb300 import oscar
    return oscar


def _randn_bf16(g, *shape, scale=1.0):
    return (torch.randn(*shape, generator=g, device="cuda") * scale).to(torch.bfloat16)


CASES = [  # (group size g, code bits, flags, norm target, key group)
    (1, 0, 0, 0.0, 0),
    (2, 0, 0, 0.0, 0),
    (4, 0, 0, 0.0, 0),
    (8, 0, 0, 0.0, 0),
    (4, 4, 0, 0.0, 0),
    (8, 4, 0, 0.0, 128),
    (4, 0, 4, 0.0, 0),           # all-heads norm
    (8, 0, 4, 0.0, 64),
    (4, 0, 1 | 2, 0.0, 0),       # neither rotation nor scaling
    (4, 0, 1, 3.0, 0),           # scaling only, target norm 3
    (3, 0, 0, 0.0, 0),           # a padding head in the 4-head form
    (6, 0, 0, 0.0, 0),           # two padding heads in the 8-head form
    (16, 0, 0, 0.0, 0),          # two slices of 8 heads per KV head
    (12, 4, 0, 0.0, 0),
]


@pytest.mark.parametrize("g,bits,flags,target,kg", CASES)
def test_fused_step_equals_separate_calls(L, g, bits, flags, target, kg):
    B, Hkv, P, R0, steps = 2, 2, 1024, 100, 160     # flushes at steps 28 and 156
    Hq = g * Hkv
    T_cap = P + 128 + 256
    gen = torch.Generator(device="cuda").manual_seed(1000 + 17 * g + bits + 3 * flags + kg)
    k = _randn_bf16(gen, B, Hkv, P + R0, 128)
    v = _randn_bf16(gen, B, Hkv, P + R0, 128)
    k[:, :, 5] *= 20                                  # an outlier channel
    caches = []
    for _ in range(2):
        c = L.KVCache(B, Hkv, T_cap, flags=flags, norm_target=target, key_group=kg, bits=bits)
        L.prefill_kv(c, k, v, n_tok=P)
        L.append_kv(c, k[:, :, P:].contiguous(), v[:, :, P:].contiguous(), n_tok=R0)
        caches.append(c)
    sep, fused = caches
    ws_a = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, T_cap, 64))
    ws_b = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, T_cap, 64))
    qr = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    out_a = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    out_b = torch.empty_like(out_a)
    flushes = 0
    for i in range(steps):
        q = _randn_bf16(gen, B, Hq, 128)
        kn = _randn_bf16(gen, B, Hkv, 128)
        vn = _randn_bf16(gen, B, Hkv, 128)
        flushes += sep.n_res == 128
        L.rotate_q(q, qr, flags=flags)
        L.append_kv(sep, kn, vn, n_tok=1)
        L.decode_attention(sep, qr, Hq, TAU, out_a, ws_a)
        out_b.fill_(float("nan"))
        L.decode_step(fused, q, kn, vn, Hq, TAU, out_b, ws_b)
        assert (fused.n_packed, fused.n_res) == (sep.n_packed, sep.n_res), i
        assert torch.equal(out_a, out_b), f"step {i}: max diff {(out_a - out_b).abs().max()}"
    torch.cuda.synchronize()
    assert L.device_status() == 0
    assert flushes == 2
    for name in ("packed", "k_res", "v_res", "k_res_norm"):
        assert torch.equal(getattr(sep, name), getattr(fused, name)), name


def test_fused_step_on_an_empty_residual_and_with_fixed_splits(L):
    """The first step after a prefill of whole blocks (no residual token yet)
    and explicit split counts, including more splits than blocks."""
    B, Hkv, g, P = 1, 2, 4, 256
    Hq = g * Hkv
    gen = torch.Generator(device="cuda").manual_seed(77)
    k = _randn_bf16(gen, B, Hkv, P, 128)
    v = _randn_bf16(gen, B, Hkv, P, 128)
    for splits in (1, 3, 20):
        sep = L.KVCache(B, Hkv, P + 128)
        fused = L.KVCache(B, Hkv, P + 128)
        for c in (sep, fused):
            L.prefill_kv(c, k, v, n_tok=P)
        ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, P + 128, splits))
        qr = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
        out_a = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
        out_b = torch.empty_like(out_a)
        for _ in range(3):
            q = _randn_bf16(gen, B, Hq, 128)
            kn = _randn_bf16(gen, B, Hkv, 128)
            vn = _randn_bf16(gen, B, Hkv, 128)
            L.rotate_q(q, qr)
            L.append_kv(sep, kn, vn, n_tok=1)
            L.decode_attention(sep, qr, Hq, TAU, out_a, ws, num_splits=splits)
            L.decode_step(fused, q, kn, vn, Hq, TAU, out_b, ws, num_splits=splits)
            assert torch.equal(out_a, out_b), splits
        torch.cuda.synchronize()
        assert L.device_status() == 0
