"""GPU parity of the CUDA path against the oracle, through the C ABI.

Gates (tolerances fixed by the decode-path contract):
* rotation: k_hat within 1 bf16 ulp of the oracle's exact value, the norm
  within 2 fp16 ulp, q' within 1e-6 relative;
* quantisation: codes, steps, zeros and norms bit-exact when both sides
  quantise the same bf16 inputs (the oracle's rotated keys are uploaded);
* attention: max-abs <= 2e-3 and relative L2 <= 1e-3 per query head, both on
  an oracle-built cache and end to end from the same raw inputs.
Sizes span several tiles and a ragged tail; the full-size workloads are
checked on sampled (sequence, KV head) rows in the launch configuration the
benchmark uses.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth
from tests._gpu_helpers import (TAU, assert_attention_close, attn_errors, bf16_tensor_to_bits,
                                bits_to_bf16_tensor, code_mismatches, f16_tensor_to_np,
                                traced_key_check, upload_oracle_cache)

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


# --------------------------------------------------------------------------
# generator
# --------------------------------------------------------------------------

def test_gpu_generator_matches_numpy(L):
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    tf = synth.sink_token_factors(2, 100, 70) * np.float32(3.0)
    out = torch.empty((2, 3, 80, 128), dtype=torch.bfloat16, device="cuda")
    synth.gen_bf16_cuda(out, 77, 3, 5, 100, 70, chan_factor=torch.from_numpy(cf).cuda(),
                        tok_factor=torch.from_numpy(tf).cuda())
    got = bf16_tensor_to_bits(out)[:, :, :70]
    want = synth.gen_bf16(77, 3, [5, 6], [0, 1, 2], 100, 70, chan_factor=cf, tok_factor=tf)
    np.testing.assert_array_equal(got, want)


# --------------------------------------------------------------------------
# rotation gates
# --------------------------------------------------------------------------

def _ulp_bf16(x):
    x = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 7)


@pytest.mark.parametrize("flags", [0, O.NO_ROTATE, O.NO_SCALE, O.NO_ROTATE | O.NO_SCALE])
def test_rotate_scale_k_gate(L, flags):
    B, H, T = 2, 3, 200
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    tf = synth.sink_token_factors(B, 0, T)
    bits = synth.gen_bf16(101, H, range(B), range(H), 0, T, chan_factor=cf, tok_factor=tf)
    bits[0, 0, 7] = 0                                   # a zero key
    k = bits_to_bf16_tensor(bits)
    k_hat = torch.empty((B, H, T + 5, 128), dtype=torch.bfloat16, device="cuda")
    norm = torch.zeros((B, H, T + 5), dtype=torch.float16, device="cuda")
    L.rotate_scale_k(k, k_hat, norm, B, H, T, in_T=T, out_T=T + 5, out_t0=5, flags=flags)
    _sync_ok(L)
    ref = O.rotate_scale_k(bits, flags)
    got = O.bf16_to_f64(bf16_tensor_to_bits(k_hat)[:, :, 5:])
    err = np.abs(got - ref.k_hat)
    assert np.all(err <= _ulp_bf16(ref.k_hat) + 2.0 ** -133), float((err / _ulp_bf16(ref.k_hat)).max())
    n_got = f16_tensor_to_np(norm)[:, :, 5:].astype(np.float64)
    ulp16 = np.spacing(np.abs(ref.norm).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(n_got - ref.norm) <= 2 * ulp16)
    assert np.all(got[0, 0, 7] == 0) and (flags & O.NO_SCALE or n_got[0, 0, 7] == 0)


@pytest.mark.parametrize("flags", [0, O.NO_ROTATE])
def test_rotate_q_gate(L, flags):
    B, Hq = 3, 8
    bits = synth.gen_bf16(102, Hq, range(B), range(Hq), 0, 1)[:, :, 0]
    q = bits_to_bf16_tensor(bits)
    qr = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    L.rotate_q(q, qr, flags=flags)
    _sync_ok(L)
    ref = O.rotate_q(bits, flags)
    got = qr.cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() <= 1e-6 * np.abs(ref).max()


# --------------------------------------------------------------------------
# quantisation gate: bit-exact on identical inputs
# --------------------------------------------------------------------------

def _special_blocks(k_hat_bits, v_bits):
    """Plant degenerate groups and exact ties into the inputs."""
    kb = k_hat_bits.copy()
    vb = v_bits.copy()
    kb[32:64, 3] = O.f64_to_bf16(np.full(32, 0.25))          # constant key channel in block 1
    ties = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 3.0] + [1.0] * 25)
    kb[64:96, 9] = O.f64_to_bf16(ties)                        # ties 0.5/1.5/2.5 in block 2
    vb[5, :] = O.f64_to_bf16(np.full(128, -0.75))             # constant value token
    vb[6, :] = O.f64_to_bf16(np.resize(ties, 128))            # ties in a value token
    # steps of 2^-133 (bf16 subnormal levels), whose reciprocal overflows
    # fp32: a key channel in block 3 and a value token; and a value token
    # with step 2^-126, the smallest normal one
    levels = np.array([0.0, 1.0, 2.0, 3.0, 2.0, 1.0, 3.0, 0.0])
    kb[96:128, 20] = O.f64_to_bf16(np.resize(levels, 32) * 2.0 ** -133)
    vb[7, :] = O.f64_to_bf16(np.resize(levels, 128) * 2.0 ** -133)
    vb[8, :] = O.f64_to_bf16(np.resize(levels, 128) * 2.0 ** -126)
    return kb, vb


def test_quantize_bit_exact(L):
    B, H, T = 2, 2, 160
    cf = synth.channel_factors([5, 38, 77, 110], 15.0)
    tf = synth.sink_token_factors(B, 0, T)
    kraw = synth.gen_bf16(201, H, range(B), range(H), 0, T, chan_factor=cf, tok_factor=tf)
    vraw = synth.gen_bf16(202, H, range(B), range(H), 0, T, tok_factor=tf)
    rk = O.rotate_scale_k(kraw)
    khat = rk.k_hat_bf16.copy()
    vb = vraw.copy()
    khat[1, 1], vb[1, 1] = _special_blocks(khat[1, 1], vb[1, 1])
    T_cap = 256
    cache = L.KVCache(B, H, T_cap)
    # quantise in two calls to exercise the packed offset
    L.quantize_kv(cache, bits_to_bf16_tensor(khat), torch.from_numpy(rk.norm_f16).cuda(),
                  bits_to_bf16_tensor(vb), src_T=T, n_tok=64)
    k2 = np.ascontiguousarray(khat[:, :, 64:])
    L.quantize_kv(cache, bits_to_bf16_tensor(k2), torch.from_numpy(np.ascontiguousarray(rk.norm_f16[:, :, 64:])).cuda(),
                  bits_to_bf16_tensor(np.ascontiguousarray(vb[:, :, 64:])), src_T=T - 64, n_tok=96)
    _sync_ok(L)
    assert cache.n_packed == 160
    for b in range(B):
        for h in range(H):
            kq, vq = O.quantize_k(khat[b, h]), O.quantize_v(vb[b, h])
            np.testing.assert_array_equal(
                cache.tokens("k_codes")[b, h, :T].cpu().numpy().view(np.uint32),
                O.pack_k_words(kq.codes))
            np.testing.assert_array_equal(
                cache.field("v_codes")[b, h, :T // 32].cpu().numpy().view(np.uint32),
                O.pack_v_words(vq.codes))
            for name, want in [("k_scale", kq.step16), ("k_zero", kq.zero16)]:
                got = cache.field(name)[b, h, :T // 32].cpu().numpy()
                np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))
            for name, want in [("v_scale", vq.step16), ("v_zero", vq.zero16),
                               ("k_norm", rk.norm_f16[b, h])]:
                got = cache.tokens(name)[b, h, :T].cpu().numpy()
                np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))
            # the untouched tail of the capacity stays zero
            assert torch.all(cache.packed[b, h, T // 32:] == 0)


def _tie_blocks(n_blocks, seed):
    """Keys and values of one head whose codes sit on exact ties and next to
    absorbed values: every block mixes (i) levels mn + k s / 2 (k = 0..6,
    every half level an exact quotient) for a step s that is a power of two,
    a multiple of 3 or neither, (ii) tiny values beside a large zero, where
    fl(x - mn) absorbs x, and (iii) random bf16 noise."""
    rng = np.random.default_rng(seed)
    T = 32 * n_blocks
    k = rng.standard_normal((T, 128)) * 0.1
    v = rng.standard_normal((T, 128))
    for b in range(n_blocks):
        r = slice(32 * b, 32 * b + 32)
        s = [0.25, 0.375, 0.3, 3.0 / 64][b % 4]
        mn = [-0.5, 0.125, -1.0, 2.0][b % 4]
        half = mn + np.arange(7) * s / 2
        k[r, 0:40] = half[rng.integers(0, 7, (32, 40))]
        k[r, 0:40][0], k[r, 0:40][1] = mn, mn + 3 * s          # every channel spans [mn, mn + 3s]
        v[32 * b:32 * b + 16, :] = half[rng.integers(0, 7, (16, 128))]
        v[32 * b:32 * b + 16, 0], v[32 * b:32 * b + 16, 1] = mn, mn + 3 * s
        # absorption: zero -1000, max 1000, the rest within 1e-3 of 0
        k[r, 60] = rng.uniform(-1e-3, 1e-3, 32)
        k[32 * b, 60], k[32 * b + 1, 60] = -1000.0, 1000.0
        v[32 * b + 20, :] = rng.uniform(-1e-3, 1e-3, 128)
        v[32 * b + 20, 0], v[32 * b + 20, 1] = -1000.0, 1000.0
        v[32 * b + 21, :] = rng.choice([-1000.0, 0.0, 1000.0, 5e-4, -5e-4], 128)
    return O.f64_to_bf16(k), O.f64_to_bf16(v)


def _exact_ties(x_bits, bits, keys):
    """Quotients (x - mn) / step (fp32, as the quantiser forms them) that are
    exactly k + 1/2."""
    x = O.bf16_to_f64(x_bits).astype(np.float32)
    xs = x.reshape(-1, 32, 128) if keys else x[:, None, :]
    ax = 1 if keys else 2
    mn, mx = xs.min(ax, keepdims=True), xs.max(ax, keepdims=True)
    st = ((mx - mn) / np.float32((1 << bits) - 1)).astype(np.float32)
    t = ((xs - mn) / np.where(mx > mn, st, np.float32(1))).astype(np.float32)
    return int(((t - np.floor(t)) == 0.5).sum())


@pytest.mark.parametrize("bits", [2, 4])
def test_quantize_ties_and_absorption_bit_exact(L, bits):
    B, H, nb = 1, 1, 8
    kb, vb = _tie_blocks(nb, 77 + bits)
    T = 32 * nb
    norm = np.ones((B, H, T), np.float16)
    cache = L.KVCache(B, H, T, bits=bits)
    L.quantize_kv(cache, bits_to_bf16_tensor(kb[None, None]), torch.from_numpy(norm).cuda(),
                  bits_to_bf16_tensor(vb[None, None]), src_T=T, n_tok=T)
    _sync_ok(L)
    kq, vq = O.quantize_k(kb, bits=bits), O.quantize_v(vb, bits=bits)
    # the construction does put thousands of quotients exactly on half levels
    assert _exact_ties(kb, bits, keys=True) > 1000 and _exact_ties(vb, bits, keys=False) > 1000
    assert int(kq.codes.max()) == (1 << bits) - 1
    np.testing.assert_array_equal(cache.tokens("k_codes")[0, 0, :T].cpu().numpy().view(np.uint32),
                                  O.pack_words(kq.codes, bits, "k"))
    np.testing.assert_array_equal(cache.field("v_codes")[0, 0, :nb].cpu().numpy().view(np.uint32),
                                  O.pack_words(vq.codes, bits, "v"))
    for name, want in [("k_scale", kq.step16), ("k_zero", kq.zero16)]:
        got = cache.field(name)[0, 0, :nb].cpu().numpy()
        np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))
    for name, want in [("v_scale", vq.step16), ("v_zero", vq.zero16)]:
        got = cache.tokens(name)[0, 0, :T].cpu().numpy()
        np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))


# --------------------------------------------------------------------------
# attention gate on an oracle-built cache
# --------------------------------------------------------------------------

def _oracle_heads(seed, B, Hkv, T, P, flags=0, chan=20.0, sinks=True):
    cf = synth.channel_factors([5, 38, 77, 110], chan)
    tf = synth.sink_token_factors(B, 0, T) if sinks else None
    k = synth.gen_bf16(seed, Hkv, range(B), range(Hkv), 0, T, chan_factor=cf, tok_factor=tf)
    v = synth.gen_bf16(seed + 1, Hkv, range(B), range(Hkv), 0, T, tok_factor=tf)
    return {(b, h): O.build_head_cache(k[b, h], v[b, h], P, flags)
            for b in range(B) for h in range(Hkv)}, k, v


def _decode_vs_oracle(L, heads, B, Hq, Hkv, T_cap, seed_q, flags=0, splits=(0,)):
    g = Hq // Hkv
    cache = upload_oracle_cache(L.KVCache(B, Hkv, T_cap, flags), heads, flags)
    qbits = synth.gen_bf16(seed_q, Hq, range(B), range(Hq), 0, 1)[:, :, 0]
    qrot = O.rotate_q(qbits, flags)
    ref = np.stack([np.concatenate([heads[(b, h)].decode(qrot[b, h * g:(h + 1) * g], TAU)
                                    for h in range(Hkv)]) for b in range(B)])
    qr = torch.from_numpy(qrot.astype(np.float32)).cuda()
    outs = []
    for S in splits:
        ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, cache.n_packed, S))
        out = torch.full((B, Hq, 128), float("nan"), device="cuda")
        L.decode_attention(cache, qr, Hq, TAU, out, ws, num_splits=S)
        _sync_ok(L)
        got = out.cpu().numpy()
        assert_attention_close(got, ref, f"splits={S}")
        outs.append(got)
    return outs, ref


# groups of 1, 2, 4 and 8 heads run whole; 3 takes the 4-head form with one
# padding head, 5..7 the 8-head form, 12 and 16 two slices of 8 per KV head
@pytest.mark.parametrize("g", [1, 2, 3, 4, 5, 6, 7, 8, 12, 16])
def test_decode_on_oracle_cache_all_groups(L, g):
    B, Hkv, T, P = 2, 2, 2048 + 77, 2048
    heads, _, _ = _oracle_heads(300 + g, B, Hkv, T, P)
    _decode_vs_oracle(L, heads, B, g * Hkv, Hkv, 2112, 310 + g, splits=(1, 2, 7, 0))


@pytest.mark.parametrize("g", [1, 3, 4, 6, 8, 16])
@pytest.mark.parametrize("R", [128, 127, 64, 31])
def test_decode_residual_window_fills(L, g, R):
    """The residual CTA over windows of 31 to 128 tokens: each warp's slice
    of the window full, partial or empty (groups of 8 take a token per lane,
    smaller groups four tokens per warp step)."""
    B, Hkv, P = 2, 2, 1024
    heads, _, _ = _oracle_heads(380 + g + R, B, Hkv, P + R, P)
    _decode_vs_oracle(L, heads, B, g * Hkv, Hkv, P + 128, 390 + g, splits=(3, 0))


@pytest.mark.parametrize("g", [1, 2, 4, 5, 8, 16])
def test_decode_with_many_splits(L, g):
    """More splits than blocks and more than 64 partials per combining warp:
    splits of one block or none (empty partials), and the combine's path for
    partials beyond the first 64 of a warp."""
    B, Hkv, T, P = 1, 2, 4096 + 40, 4096
    heads, _, _ = _oracle_heads(360 + g, B, Hkv, T, P)
    _decode_vs_oracle(L, heads, B, g * Hkv, Hkv, 4096, 370 + g, splits=(100, 300))


def test_split_invariance(L):
    B, Hkv, Hq, T, P = 1, 2, 8, 4096 + 128, 4096
    heads, _, _ = _oracle_heads(320, B, Hkv, T, P)
    outs, ref = _decode_vs_oracle(L, heads, B, Hq, Hkv, 4096, 321, splits=(1, 2, 7, 13, 0))
    for o in outs[1:]:
        d = np.linalg.norm(o - outs[0]) / np.linalg.norm(outs[0])
        assert d <= 1e-6


def test_workspace_reuse_across_split_counts_and_shapes(L):
    """The decode workspace is a header of row counters (zero between calls)
    then the split-K partials.  A zeroed workspace whose partial area holds
    arbitrary bytes, and one that calls with other split counts and another
    cache shape used in between, give the same output bit for bit as a fresh
    one; a non-zero counter is reported in the status word."""
    B, Hkv, Hq, T, P = 1, 2, 8, 4096 + 128, 4096
    heads, _, _ = _oracle_heads(330, B, Hkv, T, P)
    cache = upload_oracle_cache(L.KVCache(B, Hkv, 4096), heads)
    qbits = synth.gen_bf16(331, Hq, range(B), range(Hq), 0, 1)[:, :, 0]
    qr = torch.from_numpy(O.rotate_q(qbits).astype(np.float32)).cuda()
    nbytes = L.decode_workspace_bytes(B, Hkv, Hq, P, 64)
    header = 65536                                    # u32 counters, in 4-byte words
    want = {}
    for S in (13, 2, 7):
        ws = L.alloc_workspace(nbytes)
        want[S] = torch.empty((B, Hq, 128), device="cuda")
        L.decode_attention(cache, qr, Hq, TAU, want[S], ws, num_splits=S)
    shared = L.alloc_workspace(nbytes)
    g = torch.Generator(device="cuda").manual_seed(332)
    part = shared.view(torch.int32)[header:]
    part.copy_(torch.randint(-2**31, 2**31 - 1, (part.numel(),), dtype=torch.int32,
                             device="cuda", generator=g))
    other = upload_oracle_cache(L.KVCache(2, 1, 4096), {(b, 0): heads[(0, b)] for b in range(2)})
    other_out = torch.empty((2, 4, 128), device="cuda")
    for S in (13, 2, 7, 13, 2, 7):
        got = torch.full((B, Hq, 128), float("nan"), device="cuda")
        L.decode_attention(cache, qr, Hq, TAU, got, shared, num_splits=S)
        _sync_ok(L)
        assert torch.equal(got, want[S]), f"splits {S}"
        # another shape between the calls, on the same workspace
        L.decode_attention(other, qr.reshape(2, 4, 128).contiguous(), 4, TAU, other_out,
                           shared, num_splits=5)
        _sync_ok(L)
    assert torch.count_nonzero(shared.view(torch.int32)[:header]) == 0
    # a counter left non-zero (a workspace never zeroed) is reported
    shared.view(torch.int32)[1] = 3
    L.decode_attention(cache, qr, Hq, TAU, got, shared, num_splits=2)
    torch.cuda.synchronize()
    assert L.device_status() != 0


@pytest.mark.parametrize("T,P", [(96, 0), (1024, 1024), (32, 32), (33, 32), (1, 0)])
def test_decode_edge_sizes(L, T, P):
    B, Hkv, Hq = 1, 2, 8
    heads, _, _ = _oracle_heads(330 + T, B, Hkv, T, P)
    _decode_vs_oracle(L, heads, B, Hq, Hkv, max(32, P), 331, splits=(0, 3))


@pytest.mark.parametrize("Hq", [32, 96])   # groups of 4, and of 12 (two rows per KV head)
def test_decode_at_the_row_limit(L, Hq):
    """As many rows as the workspace has arrival counters (65536): every
    row's counter is taken and left at zero (a second call at the same split
    count is bit-identical, with a clean status word), the split counts agree
    on every row, and sampled rows match the oracle."""
    Hkv, P, R = 8, 32, 8
    g = Hq // Hkv
    B = 65536 // (Hkv * (2 if g > 8 else 1))
    T = P + R
    k = torch.empty((B, Hkv, T, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    synth.gen_bf16_cuda(k, 600, Hkv, 0, 0, T)
    synth.gen_bf16_cuda(v, 601, Hkv, 0, 0, T)
    cache = L.KVCache(B, Hkv, P)
    L.prefill_kv(cache, k, v, n_tok=P)
    L.append_kv(cache, k[:, :, P:].contiguous(), v[:, :, P:].contiguous(), n_tok=R)
    del k, v
    qb = torch.empty((B, Hq, 1, 128), dtype=torch.bfloat16, device="cuda")
    synth.gen_bf16_cuda(qb, 602, Hq, 0, 0, 1)
    qr = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    L.rotate_q(qb[:, :, 0].contiguous(), qr)
    ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, P, 2))
    outs = []
    for S in (1, 2, 1):
        out = torch.full((B, Hq, 128), float("nan"), device="cuda")
        L.decode_attention(cache, qr, Hq, TAU, out, ws, num_splits=S)
        _sync_ok(L)
        outs.append(out)
    assert torch.equal(outs[0], outs[2])
    d = (torch.linalg.vector_norm(outs[1] - outs[0]) / torch.linalg.vector_norm(outs[0])).item()
    assert d <= 1e-6, d
    for b, h in [(0, 0), (B // 2 + 1, 3), (B - 1, Hkv - 1)]:
        kb = synth.gen_bf16(600, Hkv, [b], [h], 0, T)[0, 0]
        vb = synth.gen_bf16(601, Hkv, [b], [h], 0, T)[0, 0]
        qbits = synth.gen_bf16(602, Hq, [b], range(h * g, (h + 1) * g), 0, 1)[0, :, 0]
        ref = O.build_head_cache(kb, vb, P).decode(O.rotate_q(qbits), TAU)
        got = outs[0][b, h * g:(h + 1) * g].cpu().numpy()
        assert_attention_close(got[None], ref[None], f"row ({b}, {h})")


def test_decode_empty_cache_gives_zeros(L):
    cache = L.KVCache(1, 2, 64)
    qr = torch.randn((1, 8, 128), device="cuda")
    ws = L.alloc_workspace(L.decode_workspace_bytes(1, 2, 8, 0, 2))
    out = torch.full((1, 8, 128), float("nan"), device="cuda")
    L.decode_attention(cache, qr, 8, TAU, out, ws, num_splits=2)
    _sync_ok(L)
    assert torch.all(out == 0)


@pytest.mark.parametrize("flags", [O.NO_ROTATE, O.NO_SCALE, O.NO_ROTATE | O.NO_SCALE])
def test_decode_ablation_flags(L, flags):
    B, Hkv, Hq, T, P = 1, 2, 8, 1024 + 40, 1024
    heads, _, _ = _oracle_heads(340 + flags, B, Hkv, T, P, flags=flags)
    _decode_vs_oracle(L, heads, B, Hq, Hkv, 1024, 341, flags=flags, splits=(0,))


def test_decode_lossless_case_equals_plain_attention(L):
    """INT2 storage is exact here, so the kernel must match bf16 attention."""
    flags = O.NO_ROTATE | O.NO_SCALE
    lv = np.array([-1.5, -0.5, 0.5, 1.5])
    T, P, Hq = 1024 + 60, 1024, 4
    r = synth.splitmix64(350, np.arange(2 * T * 128)).reshape(2, T, 128)
    k = lv[(r[0] % np.uint64(4)).astype(np.int64)]
    v = lv[(r[1] % np.uint64(4)).astype(np.int64)]
    k[0::32], k[1::32] = -1.5, 1.5
    v[:, 0], v[:, 1] = -1.5, 1.5
    kb, vb = O.f64_to_bf16(k), O.f64_to_bf16(v)
    heads = {(0, 0): O.build_head_cache(kb, vb, P, flags)}
    outs, ref = _decode_vs_oracle(L, heads, 1, Hq, 1, 1024, 351, flags=flags, splits=(0,))
    q = synth.gen_bf16(351, Hq, [0], range(Hq), 0, 1)[0, :, 0]
    plain = O.bf16_attention(q, kb, vb, TAU)
    assert_attention_close(outs[0][0], plain, "lossless")


# --------------------------------------------------------------------------
# end to end: GPU pipeline vs oracle pipeline from the same raw inputs
# --------------------------------------------------------------------------

def _pipeline(L, wl_name, rows, flags=0, steps=None, check_codes=True, bits=2):
    from int2_kv_cache_02_gb300 import workloads as W
    wl = W.WORKLOADS[wl_name]
    steps = wl.steps if steps is None else steps
    K, V = W.draw_kv_cuda(wl, 0, wl.T0)
    cache = W.build_cache_cuda(wl, K, V, flags=flags, T_cap=wl.t_cap(steps - wl.steps), bits=bits)
    del K, V
    if steps:
        Kn, Vn = W.draw_kv_cuda(wl, wl.T0, steps)
        for i in range(steps):
            L.append_kv(cache, Kn[:, :, i].contiguous(), Vn[:, :, i].contiguous(), n_tok=1)
        del Kn, Vn
    step = max(steps - 1, 0)
    q = W.draw_q_cuda(wl, step)
    qr = torch.empty((wl.B, wl.Hq, 128), dtype=torch.float32, device="cuda")
    L.rotate_q(q, qr, flags=flags)
    S = L.decode_num_splits(wl.B, wl.Hkv, wl.Hq, cache.n_packed)
    ws = L.alloc_workspace(L.decode_workspace_bytes(wl.B, wl.Hkv, wl.Hq, cache.n_packed, S))
    out = torch.empty((wl.B, wl.Hq, 128), dtype=torch.float32, device="cuda")
    L.decode_attention(cache, qr, wl.Hq, TAU, out, ws, num_splits=S)
    _sync_ok(L)
    out = out.cpu().numpy()
    g = wl.g
    worst = (0.0, 0.0)
    for (b, h) in rows:
        T_all = wl.T0 + steps
        kb = wl.k_bits([b], [h], 0, T_all)[0, 0]
        vb = wl.v_bits([b], [h], 0, T_all)[0, 0]
        hc = O.build_head_cache(kb[:wl.T0], vb[:wl.T0], wl.n_packed, flags, bits=bits)
        for t in range(wl.T0, T_all):
            hc.append(kb[t], vb[t])
        assert hc.n_packed == cache.n_packed and hc.n_res == cache.n_res
        qbits = wl.q_bits([b], range(h * g, (h + 1) * g), step)[0]
        ref = hc.decode(O.rotate_q(qbits, flags), TAU)
        ma, rl = assert_attention_close(out[b, h * g:(h + 1) * g], ref, f"{wl_name} row {(b, h)}")
        worst = (max(worst[0], ma), max(worst[1], rl))
        if check_codes:
            # every key code traced to its inputs (no count allowance): groups
            # whose k_hat agrees with the oracle's are bit-exact, the others
            # hold exactly what the GPU quantiser gives for the GPU's k_hat
            n_diff, n_grp = traced_key_check(L, cache, b, h, kb, vb, hc, flags=flags, bits=bits,
                                             what=f"{wl_name} row {(b, h)}")
            print(f"{wl_name} row {(b, h)}: {n_diff} key codes differ from the oracle's own, "
                  f"all inside {n_grp} (block, channel) groups whose k_hat differs by 1 ulp")
            vq = hc.packed_v()
            gotv = cache.field("v_codes")[b, h, :cache.n_packed // 32].cpu().numpy().view(np.uint32)
            assert code_mismatches(gotv, O.pack_words(vq.codes, bits, "v")) == 0
    return worst


def test_pipeline_tiny(L):
    _pipeline(L, "tiny_1k", [(0, 0)])


@pytest.mark.parametrize("flags", [O.NO_ROTATE, O.NO_SCALE])
def test_pipeline_tiny_ablations(L, flags):
    _pipeline(L, "tiny_1k", [(0, 0)], flags=flags)


def test_pipeline_qwen3_8b_32k_sampled(L):
    _pipeline(L, "qwen3_8b_32k", [(0, 0), (7, 5)])


def test_pipeline_long_stream_128k_sampled(L):
    _pipeline(L, "long_stream_128k", [(0, 3)])


def test_pipeline_batch48_128k_sampled(L):
    _pipeline(L, "batch48_128k", [(0, 0), (17, 3), (31, 5), (47, 7)], steps=1)


def test_pipeline_batch48_128k_int4_sampled(L):
    """The INT4 option at the benchmark's full size and launch configuration."""
    _pipeline(L, "batch48_128k", [(0, 0), (29, 6)], steps=1, bits=4)


def test_pipeline_omni_tni_64k_sampled(L):
    _pipeline(L, "omni_tni_64k", [(0, 0), (15, 3)])


def test_streaming_flush_equals_one_shot_on_gpu(L):
    """Appending tokens one by one (with flushes) and quantising the same
    prefix in one call give identical packed words."""
    from int2_kv_cache_02_gb300 import workloads as W
    B, Hkv, T = 2, 2, 3 * 128 + 9
    cf = synth.channel_factors([5], 20.0)
    kb = synth.gen_bf16(360, Hkv, range(B), range(Hkv), 0, T, chan_factor=cf)
    vb = synth.gen_bf16(361, Hkv, range(B), range(Hkv), 0, T)
    K, V = bits_to_bf16_tensor(kb), bits_to_bf16_tensor(vb)
    a = L.KVCache(B, Hkv, 512)
    for t in range(T):
        L.append_kv(a, K[:, :, t].contiguous(), V[:, :, t].contiguous())
    b_ = L.KVCache(B, Hkv, 512)
    L.append_kv(b_, K, V, n_tok=T)
    _sync_ok(L)
    P = 128 * ((T - 1) // 128)
    assert a.n_packed == b_.n_packed == P and a.n_res == b_.n_res == T - P
    stage = torch.empty((B, Hkv, P, 128), dtype=torch.bfloat16, device="cuda")
    norm = torch.empty((B, Hkv, P), dtype=torch.float16, device="cuda")
    L.rotate_scale_k(K, stage, norm, B, Hkv, P, in_T=T, out_T=P)
    c = L.KVCache(B, Hkv, 512)
    L.quantize_kv(c, stage, norm, V[:, :, :P].contiguous(), src_T=P, n_tok=P)
    _sync_ok(L)
    for x in (a, b_):
        assert torch.equal(x.packed[:, :, :P // 32], c.packed[:, :, :P // 32])
    assert torch.equal(a.k_res[:, :, :T - P], b_.k_res[:, :, :T - P])
    assert torch.equal(a.v_res[:, :, :T - P], b_.v_res[:, :, :T - P])


# --------------------------------------------------------------------------
# the bf16 comparison kernel
# --------------------------------------------------------------------------

@pytest.mark.parametrize("g,T,S", [(1, 1000, 0), (4, 4097, 0), (4, 4097, 3), (8, 777, 2),
                                   (2, 64, 1), (4, 1, 1), (3, 1000, 0), (6, 500, 2),
                                   (12, 300, 3), (16, 777, 0)])
def test_bf16_decode_parity(L, g, T, S):
    B, Hkv = 2, 2
    Hq = g * Hkv
    kb = synth.gen_bf16(400 + g, Hkv, range(B), range(Hkv), 0, T,
                        chan_factor=synth.channel_factors([5, 38], 20.0))
    vb = synth.gen_bf16(401 + g, Hkv, range(B), range(Hkv), 0, T)
    qb = synth.gen_bf16(402 + g, Hq, range(B), range(Hq), 0, 1)[:, :, 0]
    Ts = T + 3
    K = torch.zeros((B, Hkv, Ts, 128), dtype=torch.bfloat16, device="cuda")
    V = torch.zeros_like(K)
    K[:, :, :T] = bits_to_bf16_tensor(kb)
    V[:, :, :T] = bits_to_bf16_tensor(vb)
    q = bits_to_bf16_tensor(qb)
    Sx = S if S else 64
    ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, T, Sx))
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    L.bf16_decode_attention(q, K, V, B, Hq, Hkv, T, Ts, TAU, out, ws, num_splits=S)
    _sync_ok(L)
    ref = np.stack([np.concatenate([O.bf16_attention(qb[b, h * g:(h + 1) * g], kb[b, h], vb[b, h], TAU)
                                    for h in range(Hkv)]) for b in range(B)])
    assert_attention_close(out.cpu().numpy(), ref, f"bf16 g={g} T={T}")


def test_kernel_launch_counter_moves(L):
    n0 = L.kernel_launches()
    q = torch.zeros((1, 1, 128), dtype=torch.bfloat16, device="cuda")
    qr = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    L.rotate_q(q, qr)
    _sync_ok(L)
    assert L.kernel_launches() == n0 + 1
