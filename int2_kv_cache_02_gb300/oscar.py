"""Python binding of liboscar (include/oscar.h): argument marshalling only.

Every computation runs in the CUDA kernels of liboscar.so; this module turns
torch tensors into device pointers, keeps the oscar_cache struct, and raises
OscarError on a non-OK status.  Importing it fails loudly if the library has
not been built (``__graft_entry__.build()`` or ``python -m
int2_kv_cache_02_gb300._build``): there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
from ctypes import POINTER, c_float, c_int, c_size_t, c_uint, c_ulonglong, c_void_p

import torch

from . import _build

D, G, R = 128, 32, 128
NO_ROTATE, NO_SCALE, NORM_ALL_HEADS = 1, 2, 4

_STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "ALIGNMENT", 4: "CAPACITY",
           5: "WORKSPACE", 6: "CUDA", 7: "DEVICE_STATUS"}


class OscarError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, status)} "
                         f"({_lib.oscar_status_string(status).decode()})")


class OscarCacheStruct(ctypes.Structure):
    _fields_ = [("B", c_int), ("Hkv", c_int), ("T_cap", c_int),
                ("packed", c_void_p),
                ("k_res", c_void_p), ("v_res", c_void_p), ("k_res_norm", c_void_p),
                ("n_packed", c_int), ("n_res", c_int), ("flags", c_uint),
                ("norm_target", c_float), ("key_group", c_int), ("bits", c_int)]


class OscarPagedCacheStruct(ctypes.Structure):
    _fields_ = [("B", c_int), ("Hkv", c_int), ("max_blocks", c_int), ("n_pages", c_int),
                ("pages", c_void_p), ("block_table", c_void_p),
                ("n_packed", c_void_p), ("n_res", c_void_p),
                ("k_res", c_void_p), ("v_res", c_void_p), ("k_res_norm", c_void_p),
                ("flags", c_uint), ("norm_target", c_float), ("key_group", c_int),
                ("bits", c_int)]


BLOCK_BYTES = 2752
BLOCK_BYTES_INT4 = 4800
# byte ranges of the fields of one 32-token block record (include/oscar.h)
RECORD_FIELDS = {"k_codes": (0, 1024), "v_codes": (1024, 2048), "k_scale": (2048, 2304),
                 "k_zero": (2304, 2560), "k_norm": (2560, 2624), "v_scale": (2624, 2688),
                 "v_zero": (2688, 2752)}
# the INT4 record: twice the code bytes, the same side arrays after them
RECORD_FIELDS_INT4 = {"k_codes": (0, 2048), "v_codes": (2048, 4096), "k_scale": (4096, 4352),
                      "k_zero": (4352, 4608), "k_norm": (4608, 4672), "v_scale": (4672, 4736),
                      "v_zero": (4736, 4800)}
PER_TOKEN_FIELDS = ("k_norm", "v_scale", "v_zero")


def record_bytes(bits: int = 2) -> int:
    return BLOCK_BYTES_INT4 if bits == 4 else BLOCK_BYTES


def _load() -> ctypes.CDLL:
    path = _build.lib_path("liboscar.so")
    if not os.path.exists(path):
        raise ImportError(f"liboscar.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P = POINTER(OscarCacheStruct)
    PP = POINTER(OscarPagedCacheStruct)
    sig = {
        "oscar_rotate_q": (c_int, [c_void_p, c_void_p, c_int, c_int, c_uint, c_void_p]),
        "oscar_rotate_scale_k": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_int, c_int,
                                         c_int, c_int, c_int, c_uint, c_float, c_void_p]),
        "oscar_quantize_kv": (c_int, [P, c_void_p, c_void_p, c_void_p, c_int, c_int, c_void_p]),
        "oscar_append_kv": (c_int, [P, c_void_p, c_void_p, c_int, c_void_p]),
        "oscar_prefill_kv": (c_int, [P, c_void_p, c_void_p, c_int, c_int, c_void_p]),
        "oscar_paged_prefill_kv": (c_int, [PP, c_void_p, c_void_p, c_int, c_void_p, c_int,
                                           c_void_p]),
        "oscar_paged_append_kv": (c_int, [PP, c_void_p, c_void_p, c_void_p, c_void_p]),
        "oscar_paged_decode_attention": (c_int, [PP, c_void_p, c_int, c_float, c_int, c_void_p,
                                                 c_int, c_void_p, c_size_t, c_void_p]),
        "oscar_decode_attention": (c_int, [P, c_void_p, c_int, c_float, c_void_p, c_int,
                                           c_void_p, c_size_t, c_void_p]),
        "oscar_decode_attention_static_ws": (c_int, [P, c_void_p, c_int, c_float, c_void_p,
                                                     c_int, c_void_p]),
        "oscar_decode_step": (c_int, [P, c_void_p, c_void_p, c_void_p, c_int, c_float, c_void_p,
                                      c_int, c_void_p, c_size_t, c_void_p]),
        "oscar_decode_num_splits": (c_int, [c_int, c_int, c_int, c_int]),
        "oscar_decode_plan_splits": (c_int, [ctypes.c_longlong, ctypes.c_longlong, c_int, c_int]),
        "oscar_decode_workspace_bytes": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
        "oscar_bf16_decode_attention": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int,
                                                c_int, c_int, c_int, c_float, c_void_p, c_int,
                                                c_void_p, c_size_t, c_void_p]),
        "oscar_device_status": (c_int, [c_void_p]),
        "oscar_selftest_wait_timeout": (c_int, [c_uint, c_void_p]),
        "oscar_status_string": (ctypes.c_char_p, [c_int]),
        "oscar_kernel_launches": (c_ulonglong, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("liboscar takes device tensors")
    if not t.is_contiguous():
        raise ValueError("liboscar takes contiguous tensors")
    return c_void_p(t.data_ptr())


def _stream(stream) -> c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(st: int, where: str):
    if st != 0:
        raise OscarError(st, where)


# ---------------------------------------------------------------------------
# the cache
# ---------------------------------------------------------------------------

class KVCache:
    """Caller-owned device buffers of one layer's OScaR cache plus the
    oscar_cache struct that points at them (layouts in include/oscar.h)."""

    def __init__(self, B: int, Hkv: int, T_cap: int, flags: int = 0, device=None,
                 norm_target: float = 0.0, key_group: int = 0, bits: int = 0):
        if T_cap % G:
            raise ValueError("T_cap must be a multiple of 32")
        dev = torch.device(device if device is not None else "cuda")
        self.packed = torch.zeros((B, Hkv, T_cap // G, record_bytes(bits)), dtype=torch.uint8,
                                  device=dev)
        self.k_res = torch.zeros((B, Hkv, R, D), dtype=torch.bfloat16, device=dev)
        self.v_res = torch.zeros((B, Hkv, R, D), dtype=torch.bfloat16, device=dev)
        self.k_res_norm = torch.zeros((B, Hkv, R), dtype=torch.float16, device=dev)
        s = OscarCacheStruct()
        s.B, s.Hkv, s.T_cap = B, Hkv, T_cap
        for name in ("packed", "k_res", "v_res", "k_res_norm"):
            setattr(s, name, getattr(self, name).data_ptr())
        s.n_packed, s.n_res, s.flags, s.norm_target = 0, 0, flags, norm_target
        s.key_group = key_group
        s.bits = bits
        self.struct = s

    B = property(lambda self: self.struct.B)
    Hkv = property(lambda self: self.struct.Hkv)
    T_cap = property(lambda self: self.struct.T_cap)
    n_packed = property(lambda self: self.struct.n_packed)
    n_res = property(lambda self: self.struct.n_res)
    flags = property(lambda self: self.struct.flags)
    norm_target = property(lambda self: self.struct.norm_target)
    key_group = property(lambda self: self.struct.key_group or 32)
    bits = property(lambda self: self.struct.bits or 2)

    def ref(self):
        return ctypes.byref(self.struct)

    def field(self, name: str) -> torch.Tensor:
        """Writable view of one record field for every block:
        [B][Hkv][T_cap/32][n] with n = 256 words (codes; INT4: 512) or 128 halves (key
        step / zero); the per-token arrays (k_norm, v_scale, v_zero) as
        [B][Hkv][T_cap/32][4][8], element [j][i] = token 8j + i of the block."""
        lo, hi = (RECORD_FIELDS_INT4 if self.bits == 4 else RECORD_FIELDS)[name]
        raw = self.packed[..., lo:hi]
        if name.endswith("codes"):
            return raw.view(torch.int32)
        f = raw.view(torch.float16)
        if name in PER_TOKEN_FIELDS:
            # stored at 4 (t % 8) + t // 8: an [8][4] array, read transposed
            return f.unflatten(-1, (8, 4)).transpose(-1, -2)
        return f

    def tokens(self, name: str) -> torch.Tensor:
        """A copy of a field in token order: key codes [B][Hkv][T_cap][8]
        (INT4: [..][16]); norms and value step / zero [B][Hkv][T_cap]; value
        codes and key step / zero stay per block ([B][Hkv][T_cap/32][n])."""
        f = self.field(name)
        if name == "k_codes":
            return f.reshape(self.B, self.Hkv, self.T_cap, 4 * self.bits)
        if name in PER_TOKEN_FIELDS:
            return f.reshape(self.B, self.Hkv, self.T_cap)
        return f.clone()

    def nbytes(self) -> int:
        return sum(getattr(self, n).numel() * getattr(self, n).element_size()
                   for n in ("packed", "k_res", "v_res", "k_res_norm"))


class PagedKVCache:
    """Caller-owned device buffers of a paged cache (oscar_paged_cache):
    a pool of n_pages pages (each one 2752-byte record per KV head for 32
    tokens), the block table [B][max_blocks] (page ids, -1 = unmapped),
    per-sequence lengths n_packed[B], n_res[B] on the device, and the
    per-(b, h) residual windows.  Pages are handed out by the host-side
    allocator below; the device kernels only follow the table."""

    def __init__(self, B: int, Hkv: int, max_blocks: int, n_pages: int, flags: int = 0,
                 device=None, norm_target: float = 0.0, key_group: int = 0, bits: int = 0):
        dev = torch.device(device if device is not None else "cuda")
        self.pages = torch.zeros((n_pages, Hkv, record_bytes(bits)), dtype=torch.uint8,
                                 device=dev)
        self.block_table = torch.full((B, max_blocks), -1, dtype=torch.int32, device=dev)
        self.n_packed_d = torch.zeros(B, dtype=torch.int32, device=dev)
        self.n_res_d = torch.zeros(B, dtype=torch.int32, device=dev)
        self.k_res = torch.zeros((B, Hkv, R, D), dtype=torch.bfloat16, device=dev)
        self.v_res = torch.zeros((B, Hkv, R, D), dtype=torch.bfloat16, device=dev)
        self.k_res_norm = torch.zeros((B, Hkv, R), dtype=torch.float16, device=dev)
        s = OscarPagedCacheStruct()
        s.B, s.Hkv, s.max_blocks, s.n_pages, s.flags = B, Hkv, max_blocks, n_pages, flags
        s.norm_target = norm_target
        s.key_group = key_group
        s.bits = bits
        s.pages = self.pages.data_ptr()
        s.block_table = self.block_table.data_ptr()
        s.n_packed = self.n_packed_d.data_ptr()
        s.n_res = self.n_res_d.data_ptr()
        for name in ("k_res", "v_res", "k_res_norm"):
            setattr(s, name, getattr(self, name).data_ptr())
        self.struct = s
        self._free = list(range(n_pages))
        self._table_host = [[-1] * max_blocks for _ in range(B)]

    B = property(lambda self: self.struct.B)
    Hkv = property(lambda self: self.struct.Hkv)
    max_blocks = property(lambda self: self.struct.max_blocks)
    n_pages = property(lambda self: self.struct.n_pages)
    flags = property(lambda self: self.struct.flags)

    def ref(self):
        return ctypes.byref(self.struct)

    def map_blocks(self, b: int, n_blocks: int, order=None):
        """Gives sequence b pages for its logical blocks 0..n_blocks-1 (those
        not mapped yet), taking free pages in `order` (a permutation of page
        ids, for tests) or in pool order."""
        if order is not None:
            free = set(self._free)
            self._free = [p for p in order if p in free]
        row = self._table_host[b]
        for j in range(n_blocks):
            if row[j] < 0:
                if not self._free:
                    raise OscarError(4, "PagedKVCache.map_blocks: page pool exhausted")
                row[j] = self._free.pop(0)
        self.block_table[b].copy_(torch.tensor(row, dtype=torch.int32))

    def page_of(self, b: int, block: int) -> int:
        return self._table_host[b][block]

    def record(self, b: int, h: int, block: int) -> torch.Tensor:
        """View of the 2752-byte record of (b, h, logical block)."""
        return self.pages[self.page_of(b, block), h]

    def lengths(self):
        """(n_packed, n_res) per sequence, read back from the device."""
        return self.n_packed_d.cpu().tolist(), self.n_res_d.cpu().tolist()


# ---------------------------------------------------------------------------
# the calls (same names as the C ABI, without the oscar_ prefix)
# ---------------------------------------------------------------------------

def rotate_q(q: torch.Tensor, q_rot: torch.Tensor, flags: int = 0, stream=None):
    B, Hq = q.shape[0], q.shape[1]
    _check(_lib.oscar_rotate_q(_ptr(q), _ptr(q_rot), B, Hq, flags, _stream(stream)),
           "oscar_rotate_q")


def rotate_scale_k(k: torch.Tensor, k_hat: torch.Tensor, norm: torch.Tensor, B: int, Hkv: int,
                   n_tok: int, in_T: int, out_T: int, out_t0: int = 0, flags: int = 0,
                   stream=None, norm_target: float = 0.0):
    _check(_lib.oscar_rotate_scale_k(_ptr(k), in_T, _ptr(k_hat), _ptr(norm), out_T, out_t0,
                                     B, Hkv, n_tok, flags, norm_target, _stream(stream)),
           "oscar_rotate_scale_k")


def prefill_kv(cache: KVCache, k: torch.Tensor, v: torch.Tensor, n_tok: int, in_T: int = 0,
               stream=None):
    """Fused rotate + scale + quantise of tokens [0, n_tok) of raw bf16 keys
    and values [B][Hkv][in_T][128] into the packed cache (advances n_packed)."""
    in_T = in_T or k.shape[2]
    _check(_lib.oscar_prefill_kv(cache.ref(), _ptr(k), _ptr(v), in_T, n_tok, _stream(stream)),
           "oscar_prefill_kv")


def paged_prefill_kv(cache: PagedKVCache, k: torch.Tensor, v: torch.Tensor,
                     n_tok: torch.Tensor, max_tok: int, in_T: int = 0, stream=None):
    """Fused prefill of sequence b's tokens [0, n_tok[b]) (device int32 [B],
    multiples of 32, <= max_tok) into its next logical blocks."""
    in_T = in_T or k.shape[2]
    _check(_lib.oscar_paged_prefill_kv(cache.ref(), _ptr(k), _ptr(v), in_T, _ptr(n_tok),
                                       max_tok, _stream(stream)), "oscar_paged_prefill_kv")


def paged_append_kv(cache: PagedKVCache, k_new: torch.Tensor, v_new: torch.Tensor,
                    active: torch.Tensor | None = None, stream=None):
    """One new token [B][Hkv][128] for every sequence with active[b] != 0."""
    _check(_lib.oscar_paged_append_kv(cache.ref(), _ptr(k_new), _ptr(v_new), _ptr(active),
                                      _stream(stream)), "oscar_paged_append_kv")


def paged_decode_attention(cache: PagedKVCache, q_rot: torch.Tensor, Hq: int,
                           softmax_scale: float, max_packed: int, out: torch.Tensor,
                           workspace: torch.Tensor, num_splits: int = 0, stream=None):
    _check(_lib.oscar_paged_decode_attention(cache.ref(), _ptr(q_rot), Hq, softmax_scale,
                                             max_packed, _ptr(out), num_splits, _ptr(workspace),
                                             workspace.numel() * workspace.element_size(),
                                             _stream(stream)), "oscar_paged_decode_attention")


def quantize_kv(cache: KVCache, k_hat=None, k_norm=None, v=None, src_T: int = 0,
                n_tok: int = 0, stream=None):
    _check(_lib.oscar_quantize_kv(cache.ref(), _ptr(k_hat), _ptr(k_norm), _ptr(v), src_T, n_tok,
                                  _stream(stream)), "oscar_quantize_kv")


def append_kv(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, n_tok: int = 1,
              stream=None):
    _check(_lib.oscar_append_kv(cache.ref(), _ptr(k_new), _ptr(v_new), n_tok, _stream(stream)),
           "oscar_append_kv")


def decode_num_splits(B: int, Hkv: int, Hq: int, n_packed: int) -> int:
    return int(_lib.oscar_decode_num_splits(B, Hkv, Hq, n_packed))


def decode_plan_splits(rows: int, n_blocks: int, ctas_per_sm: int, sms: int) -> int:
    return int(_lib.oscar_decode_plan_splits(rows, n_blocks, ctas_per_sm, sms))


def decode_workspace_bytes(B: int, Hkv: int, Hq: int, n_packed: int, num_splits: int = 0) -> int:
    return int(_lib.oscar_decode_workspace_bytes(B, Hkv, Hq, n_packed, num_splits))


def alloc_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A decode workspace of at least nbytes, zeroed: its header of row
    counters must start at zero, and every decode call leaves it zero."""
    return torch.zeros(max(16, (nbytes + 15) // 16 * 16) // 4, dtype=torch.float32,
                       device=device if device is not None else "cuda")


def decode_attention(cache: KVCache, q_rot: torch.Tensor, Hq: int, softmax_scale: float,
                     out: torch.Tensor, workspace: torch.Tensor, num_splits: int = 0,
                     stream=None):
    _check(_lib.oscar_decode_attention(cache.ref(), _ptr(q_rot), Hq, softmax_scale, _ptr(out),
                                       num_splits, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream)), "oscar_decode_attention")


def decode_step(cache: KVCache, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                Hq: int, softmax_scale: float, out: torch.Tensor, workspace: torch.Tensor,
                num_splits: int = 0, stream=None):
    """One decode step in one launch: rotate the raw queries q (bf16
    [B][Hq][128]), append the new token (k_new, v_new bf16 [B][Hkv][128];
    a full window is flushed first) and attend; equals rotate_q + append_kv +
    decode_attention bit for bit.  Advances the cache's residual count."""
    _check(_lib.oscar_decode_step(cache.ref(), _ptr(q), _ptr(k_new), _ptr(v_new), Hq,
                                  softmax_scale, _ptr(out), num_splits, _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)),
           "oscar_decode_step")


def decode_attention_static_ws(cache: KVCache, q_rot: torch.Tensor, Hq: int,
                               softmax_scale: float, out: torch.Tensor, num_splits: int = 0,
                               stream=None):
    """decode_attention for callers that cannot allocate: the split-K partials
    use the library's own static device array (no workspace argument)."""
    _check(_lib.oscar_decode_attention_static_ws(cache.ref(), _ptr(q_rot), Hq, softmax_scale,
                                                 _ptr(out), num_splits, _stream(stream)),
           "oscar_decode_attention_static_ws")


def bf16_decode_attention(q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, B: int, Hq: int,
                          Hkv: int, T: int, T_stride: int, softmax_scale: float,
                          out: torch.Tensor, workspace: torch.Tensor, num_splits: int = 0,
                          stream=None):
    _check(_lib.oscar_bf16_decode_attention(_ptr(q), _ptr(K), _ptr(V), B, Hq, Hkv, T, T_stride,
                                            softmax_scale, _ptr(out), num_splits,
                                            _ptr(workspace),
                                            workspace.numel() * workspace.element_size(),
                                            _stream(stream)), "oscar_bf16_decode_attention")


def selftest_wait_timeout(iterations: int = 256, stream=None):
    """Launches the bounded-wait self-test: a wait that can never complete
    gives up after `iterations` polls and sets the device status word."""
    _check(_lib.oscar_selftest_wait_timeout(iterations, _stream(stream)),
           "oscar_selftest_wait_timeout")


def device_status(stream=None) -> int:
    return int(_lib.oscar_device_status(_stream(stream)))


def kernel_launches() -> int:
    return int(_lib.oscar_kernel_launches())


def default_scale() -> float:
    return 1.0 / math.sqrt(D)
