"""Host-side checks of the C ABI: the libraries build for sm_103a, load, export
every symbol the headers declare, and reject bad arguments before launching
anything.  No kernel runs here.

The validation cases pass made-up device addresses that must never reach a
kernel; they are skipped where a GPU is present so that a validation bug can
never turn into a launch with a bad pointer.
"""
import ctypes
import os
import re

import pytest
import torch

from int2_kv_cache_02_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = {"liboscar.so": "oscar.h", "liboscar_synth.so": "oscar_synth.h"}

no_gpu_only = pytest.mark.skipif(torch.cuda.is_available(),
                                 reason="fake-pointer validation runs only without a GPU")


@pytest.fixture(scope="module")
def libs():
    paths = _build.build()
    return {k: ctypes.CDLL(v) for k, v in paths.items()}


def _declared(header: str) -> list[str]:
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(oscar_\w+)\s*\(", text, flags=re.M)))


def test_headers_declare_the_documented_calls():
    names = _declared("oscar.h")
    for want in ["oscar_rotate_q", "oscar_rotate_scale_k", "oscar_quantize_kv",
                 "oscar_append_kv", "oscar_decode_attention", "oscar_bf16_decode_attention",
                 "oscar_decode_workspace_bytes", "oscar_decode_num_splits",
                 "oscar_device_status", "oscar_status_string", "oscar_kernel_launches",
                 "oscar_selftest_wait_timeout", "oscar_prefill_kv", "oscar_paged_prefill_kv",
                 "oscar_paged_append_kv", "oscar_paged_decode_attention", "oscar_decode_step",
                 "oscar_decode_plan_splits"]:
        assert want in names
    assert _declared("oscar_synth.h") == ["oscar_synth_bf16"]


@pytest.mark.parametrize("lib", sorted(HEADERS))
def test_every_declared_symbol_is_exported(libs, lib):
    for name in _declared(HEADERS[lib]):
        assert hasattr(libs[lib], name), f"{lib} does not export {name}"


def test_status_strings(libs):
    f = libs["liboscar.so"].oscar_status_string
    f.restype = ctypes.c_char_p
    seen = {f(i) for i in range(8)}
    assert len(seen) == 8 and f(99) == b"unknown status"


# --------------------------------------------------------------------------
# validation (made-up addresses, no device)
# --------------------------------------------------------------------------

FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


def _cache(**kw):
    from int2_kv_cache_02_gb300.oscar import OscarCacheStruct
    s = OscarCacheStruct()
    s.B, s.Hkv, s.T_cap = kw.get("B", 2), kw.get("Hkv", 2), kw.get("T_cap", 256)
    for i, name in enumerate(["packed", "k_res", "v_res", "k_res_norm"]):
        setattr(s, name, kw.get(name, FAKE + 0x100000 * i))
    s.n_packed, s.n_res, s.flags = kw.get("n_packed", 0), kw.get("n_res", 0), kw.get("flags", 0)
    s.norm_target = kw.get("norm_target", 0.0)
    s.key_group = kw.get("key_group", 0)
    s.bits = kw.get("bits", 0)
    return s


@no_gpu_only
def test_rotate_validation():
    from int2_kv_cache_02_gb300 import oscar as O
    L = O.library()
    P = ctypes.c_void_p
    assert L.oscar_rotate_q(None, P(FAKE), 1, 1, 0, None) == 1
    assert L.oscar_rotate_q(P(FAKE + 8), P(FAKE), 1, 1, 0, None) == 3
    assert L.oscar_rotate_q(P(FAKE), P(FAKE), 1, 1, 8, None) == 1          # unknown flag
    assert L.oscar_rotate_q(P(FAKE), P(FAKE), 0, 1, 0, None) == 1
    assert L.oscar_rotate_scale_k(P(FAKE), 4, P(FAKE), P(FAKE), 8, 6, 1, 1, 4, 0, 0.0, None) == 1
    assert L.oscar_rotate_scale_k(P(FAKE), 2, P(FAKE), P(FAKE), 8, 0, 1, 1, 4, 0, 0.0, None) == 1
    assert L.oscar_rotate_scale_k(P(FAKE), 4, P(FAKE + 2), P(FAKE), 8, 0, 1, 1, 4, 0, 0.0,
                                  None) == 3
    assert L.oscar_rotate_scale_k(P(FAKE), 4, P(FAKE), P(FAKE), 8, 0, 1, 1, 4, 8, 0.0, None) == 1
    # target norm outside [2^-8, 2^8], negative or NaN
    for t in (1e-3, 300.0, -1.0, float("nan"), float("inf")):
        assert L.oscar_rotate_scale_k(P(FAKE), 4, P(FAKE), P(FAKE), 8, 0, 1, 1, 4, 0, t,
                                      None) == 1


@no_gpu_only
def test_cache_validation_and_state_untouched():
    from int2_kv_cache_02_gb300 import oscar as O
    L = O.library()
    P = ctypes.c_void_p
    bad_cap = _cache(T_cap=100)
    assert L.oscar_quantize_kv(ctypes.byref(bad_cap), None, None, None, 0, 0, None) == 1
    misaligned = _cache(packed=FAKE + 4)
    assert L.oscar_quantize_kv(ctypes.byref(misaligned), None, None, None, 0, 0, None) == 3
    c = _cache()
    # flush needs a full residual window
    assert L.oscar_quantize_kv(ctypes.byref(c), None, None, None, 0, 0, None) == 1
    # non-multiple of 32, and too many tokens for the capacity
    assert L.oscar_quantize_kv(ctypes.byref(c), P(FAKE), P(FAKE), P(FAKE), 64, 48, None) == 1
    assert L.oscar_quantize_kv(ctypes.byref(c), P(FAKE), P(FAKE), P(FAKE), 512, 512, None) == 4
    # packed tokens must precede residual ones
    c2 = _cache(n_res=3)
    assert L.oscar_quantize_kv(ctypes.byref(c2), P(FAKE), P(FAKE), P(FAKE), 64, 64, None) == 1
    # append needing a flush that does not fit: nothing launched, struct unchanged
    full = _cache(n_packed=256, n_res=128)
    assert L.oscar_append_kv(ctypes.byref(full), P(FAKE), P(FAKE), 1, None) == 4
    assert full.n_packed == 256 and full.n_res == 128
    st = _cache(n_packed=128, n_res=128)
    assert L.oscar_append_kv(ctypes.byref(st), P(FAKE), P(FAKE), 200, None) == 4
    assert st.n_packed == 128 and st.n_res == 128
    assert c.n_packed == 0 and c.n_res == 0
    # scaling variants: unknown flag bit, target norm out of range
    for bad in (_cache(flags=8), _cache(norm_target=512.0), _cache(norm_target=-1.0),
                _cache(norm_target=float("nan"))):
        assert L.oscar_prefill_kv(ctypes.byref(bad), P(FAKE), P(FAKE), 64, 64, None) == 1
        assert L.oscar_append_kv(ctypes.byref(bad), P(FAKE), P(FAKE), 1, None) == 1
        assert L.oscar_decode_attention_static_ws(ctypes.byref(bad), P(FAKE), 2, 0.1, P(FAKE),
                                                  1, None) == 1
        assert bad.n_packed == 0 and bad.n_res == 0
    # key groups: only 32 (0), 64, 128; n_packed and quantised runs multiples of it
    for bad in (_cache(key_group=48), _cache(key_group=256), _cache(key_group=64, n_packed=32),
                _cache(key_group=128, n_packed=64)):
        assert L.oscar_prefill_kv(ctypes.byref(bad), P(FAKE), P(FAKE), 64, 64, None) == 1
        # both decode entry points apply the same cache checks
        assert L.oscar_decode_attention(ctypes.byref(bad), P(FAKE), 2, 0.1, P(FAKE), 1, P(FAKE),
                                        1 << 20, None) == 1
        assert L.oscar_decode_attention_static_ws(ctypes.byref(bad), P(FAKE), 2, 0.1, P(FAKE),
                                                  1, None) == 1
    for bad in (_cache(bits=3), _cache(bits=8), _cache(bits=1)):
        assert L.oscar_prefill_kv(ctypes.byref(bad), P(FAKE), P(FAKE), 64, 64, None) == 1
        assert L.oscar_decode_attention_static_ws(ctypes.byref(bad), P(FAKE), 2, 0.1, P(FAKE),
                                                  1, None) == 1
    g128 = _cache(key_group=128)
    assert L.oscar_prefill_kv(ctypes.byref(g128), P(FAKE), P(FAKE), 64, 64, None) == 1
    assert L.oscar_quantize_kv(ctypes.byref(g128), P(FAKE), P(FAKE), P(FAKE), 192, 192, None) == 1
    assert g128.n_packed == 0


@no_gpu_only
def test_prefill_validation():
    from int2_kv_cache_02_gb300 import oscar as O
    L = O.library()
    P = ctypes.c_void_p
    c = _cache()
    assert L.oscar_prefill_kv(ctypes.byref(c), None, P(FAKE), 64, 64, None) == 1
    assert L.oscar_prefill_kv(ctypes.byref(c), P(FAKE + 8), P(FAKE), 64, 64, None) == 3
    assert L.oscar_prefill_kv(ctypes.byref(c), P(FAKE), P(FAKE), 64, 48, None) == 1   # not x32
    assert L.oscar_prefill_kv(ctypes.byref(c), P(FAKE), P(FAKE), 32, 64, None) == 1   # in_T < n_tok
    assert L.oscar_prefill_kv(ctypes.byref(c), P(FAKE), P(FAKE), 512, 512, None) == 4 # capacity
    c2 = _cache(n_res=5)
    assert L.oscar_prefill_kv(ctypes.byref(c2), P(FAKE), P(FAKE), 64, 64, None) == 1
    assert c.n_packed == 0 and c2.n_packed == 0


def _paged(**kw):
    from int2_kv_cache_02_gb300.oscar import OscarPagedCacheStruct
    s = OscarPagedCacheStruct()
    s.B, s.Hkv = kw.get("B", 2), kw.get("Hkv", 2)
    s.max_blocks, s.n_pages = kw.get("max_blocks", 8), kw.get("n_pages", 16)
    for i, name in enumerate(["pages", "block_table", "n_packed", "n_res", "k_res", "v_res",
                              "k_res_norm"]):
        setattr(s, name, kw.get(name, FAKE + 0x100000 * i))
    s.flags = kw.get("flags", 0)
    s.norm_target = kw.get("norm_target", 0.0)
    s.key_group = kw.get("key_group", 0)
    s.bits = kw.get("bits", 0)
    return s


@no_gpu_only
def test_paged_validation():
    from int2_kv_cache_02_gb300 import oscar as O
    L = O.library()
    P = ctypes.c_void_p
    bad = _paged(n_pages=0)
    assert L.oscar_paged_append_kv(ctypes.byref(bad), P(FAKE), P(FAKE), None, None) == 1
    mis = _paged(pages=FAKE + 8)
    assert L.oscar_paged_append_kv(ctypes.byref(mis), P(FAKE), P(FAKE), None, None) == 3
    for bad in (_paged(flags=8), _paged(norm_target=1e-3), _paged(key_group=96), _paged(bits=3)):
        assert L.oscar_paged_append_kv(ctypes.byref(bad), P(FAKE), P(FAKE), None, None) == 1
    g128 = _paged(key_group=128)
    assert L.oscar_paged_prefill_kv(ctypes.byref(g128), P(FAKE), P(FAKE), 64, P(FAKE), 64,
                                    None) == 1          # max_tok not a multiple of the group
    c = _paged()
    assert L.oscar_paged_prefill_kv(ctypes.byref(c), P(FAKE), P(FAKE), 64, P(FAKE), 48, None) == 1
    assert L.oscar_paged_prefill_kv(ctypes.byref(c), P(FAKE), P(FAKE), 512, P(FAKE), 512,
                                    None) == 4          # more blocks than a table row
    assert L.oscar_paged_decode_attention(ctypes.byref(c), P(FAKE), 34, 0.1, 64, P(FAKE), 0,
                                          P(FAKE), 1 << 20, None) == 2      # group of 17
    assert L.oscar_paged_decode_attention(ctypes.byref(c), P(FAKE), 5, 0.1, 64, P(FAKE), 0,
                                          P(FAKE), 1 << 20, None) == 2      # not a multiple
    assert L.oscar_paged_decode_attention(ctypes.byref(c), P(FAKE), 8, 0.1, 33, P(FAKE), 0,
                                          P(FAKE), 1 << 20, None) == 1
    assert L.oscar_paged_decode_attention(ctypes.byref(c), P(FAKE), 8, 0.1, 64, P(FAKE), 2,
                                          P(FAKE), 10, None) == 5
    # a block table of 2^31 entries or more (the kernels index it in 32 bits)
    big = _paged(B=2, max_blocks=1 << 30)
    assert L.oscar_paged_append_kv(ctypes.byref(big), P(FAKE), P(FAKE), None, None) == 2
    assert L.oscar_paged_decode_attention(ctypes.byref(big), P(FAKE), 8, 0.1, 64, P(FAKE), 0,
                                          P(FAKE), 1 << 20, None) == 2


@no_gpu_only
def test_decode_validation():
    from int2_kv_cache_02_gb300 import oscar as O
    L = O.library()
    P = ctypes.c_void_p
    c = _cache(Hkv=2)
    # a query group above 16 heads, or Hq not a multiple of Hkv, is not supported
    assert L.oscar_decode_attention(ctypes.byref(c), P(FAKE), 34, 0.1, P(FAKE), 0, P(FAKE),
                                    1 << 30, None) == 2
    assert L.oscar_decode_attention(ctypes.byref(c), P(FAKE), 7, 0.1, P(FAKE), 0, P(FAKE),
                                    1 << 30, None) == 2
    # groups of 9..16 take two rows per KV head: 32769 KV heads of 12 query
    # heads are over the 65536 row counters, 32769 of 8 are not
    big = _cache(B=1, Hkv=32769)
    assert L.oscar_decode_attention(ctypes.byref(big), P(FAKE), 12 * 32769, 0.1, P(FAKE), 1,
                                    P(FAKE), 1 << 40, None) == 2
    assert L.oscar_decode_attention(ctypes.byref(big), P(FAKE), 8 * 32769, 0.1, P(FAKE), 1,
                                    P(FAKE), 4, None) == 5
    # workspace missing / too small
    assert L.oscar_decode_attention(ctypes.byref(c), P(FAKE), 8, 0.1, P(FAKE), 4, None,
                                    1 << 30, None) == 5
    need = L.oscar_decode_workspace_bytes(2, 2, 8, 0, 4)
    # a fixed header of 65536 u32 row counters, then partial records of 132 floats
    assert need == 65536 * 4 + 2 * 8 * 5 * 132 * 4
    assert L.oscar_decode_workspace_bytes(3, 3, 6, 0, 1) == 65536 * 4 + 3 * 6 * 2 * 528
    assert L.oscar_decode_attention(ctypes.byref(c), P(FAKE), 8, 0.1, P(FAKE), 4, P(FAKE),
                                    need - 1, None) == 5
    assert L.oscar_decode_attention(ctypes.byref(c), P(FAKE), 8, float("nan"), P(FAKE), 4,
                                    P(FAKE), need, None) == 1
    # bf16 comparison kernel
    assert L.oscar_bf16_decode_attention(P(FAKE), P(FAKE), P(FAKE), 1, 4, 2, 100, 50, 0.1,
                                         P(FAKE), 1, P(FAKE), 1 << 20, None) == 1
    assert L.oscar_bf16_decode_attention(P(FAKE), P(FAKE), P(FAKE), 1, 5, 2, 100, 100, 0.1,
                                         P(FAKE), 1, P(FAKE), 1 << 20, None) == 2
    assert L.oscar_bf16_decode_attention(P(FAKE), P(FAKE), P(FAKE), 1, 4, 2, 100, 100, 0.1,
                                         P(FAKE), 2, P(FAKE), 100, None) == 5


def test_selftest_validation(libs):
    # rejected on the host before any device call: safe with or without a GPU
    f = libs["liboscar.so"].oscar_selftest_wait_timeout
    f.argtypes = [ctypes.c_uint, ctypes.c_void_p]
    assert f(0, None) == 1
    assert f((1 << 20) + 1, None) == 1


@no_gpu_only
def test_synth_validation(libs):
    f = libs["liboscar_synth.so"].oscar_synth_bf16
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_ulonglong, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p]
    assert f(None, 1, 1, 0, 4, 0, 4, 1, None, None, None) == 1
    assert f(FAKE + 2, 1, 1, 0, 4, 0, 4, 1, None, None, None) == 1
    assert f(FAKE, 1, 1, 0, 2, 0, 4, 1, None, None, None) == 1


@no_gpu_only
def test_decode_step_validation_leaves_the_cache_untouched():
    """The fused decode step checks everything (arguments, alignment, the
    flush's capacity, the workspace) before it launches anything, and leaves
    the cache's counts as they were when a check fails."""
    from int2_kv_cache_02_gb300 import oscar as O
    L = O.library()
    P = ctypes.c_void_p
    ws = 1 << 30

    def step(c, q=FAKE, k=FAKE, v=FAKE, Hq=4, out=FAKE, splits=1, wsb=ws):
        return L.oscar_decode_step(ctypes.byref(c), P(q), P(k), P(v), Hq, 0.1, P(out), splits,
                                   P(FAKE + 0x1000000), wsb, None)

    c = _cache(n_packed=64, n_res=5)
    assert step(c, q=0) == 1
    assert step(c, k=0) == 1
    assert step(c, v=0) == 1
    assert step(c, out=0) == 1
    assert step(c, Hq=0) == 1
    assert step(c, splits=-1) == 1
    assert step(c, k=FAKE + 8) == 3
    assert step(c, q=FAKE + 4) == 3
    assert step(c, Hq=34) == 2                               # group of 17
    assert step(c, Hq=5) == 2                                # not a multiple of Hkv
    assert step(c, wsb=16) == 5                              # workspace too small
    assert c.n_packed == 64 and c.n_res == 5
    full = _cache(n_packed=256, n_res=128)                   # the flush would not fit
    assert step(full) == 4
    assert full.n_packed == 256 and full.n_res == 128
    for bad in (_cache(flags=8), _cache(norm_target=-1.0), _cache(key_group=48)):
        assert step(bad) == 1
        assert bad.n_packed == 0 and bad.n_res == 0
