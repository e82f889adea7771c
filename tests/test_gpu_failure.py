"""Failure detection on the GPU without a fault.

Every wait in the decode kernels polls its mbarrier a bounded number of
times; a wait that gives up sets a bit in the device status word and the
kernel returns instead of hanging.  Here a wait that can never complete (an
mbarrier nothing arrives at) is made to run out on purpose: the status word
must report it, reading it must clear it, and the context must stay usable
for a regular decode afterwards.
"""
import time

import numpy as np
import pytest
import torch

from oracle import oscar_oracle as O
from int2_kv_cache_02_gb300 import synth
from tests._gpu_helpers import TAU, assert_attention_close, upload_oracle_cache

pytestmark = pytest.mark.gpu

DEVICE_STATUS = 7   # OSCAR_ERR_DEVICE_STATUS


@pytest.fixture(scope="module")
def L():
    from int2_kv_cache_02_gb300 import _build
    _build.build()
    from int2_kv_cache_02_gb300 import oscar
    return oscar


def test_bounded_wait_gives_up_and_reports(L):
    assert L.device_status() == 0
    t0 = time.time()
    L.selftest_wait_timeout(256)
    assert L.device_status() == DEVICE_STATUS
    assert L.device_status() == 0          # reading clears the word
    assert time.time() - t0 < 60


def test_context_stays_usable_after_a_timeout(L):
    L.selftest_wait_timeout(64)
    assert L.device_status() == DEVICE_STATUS
    B, Hkv, Hq, T, P = 1, 2, 8, 1024 + 50, 1024
    cf = synth.channel_factors([5, 38, 77, 110], 20.0)
    k = synth.gen_bf16(940, Hkv, range(B), range(Hkv), 0, T, chan_factor=cf)
    v = synth.gen_bf16(941, Hkv, range(B), range(Hkv), 0, T)
    heads = {(0, h): O.build_head_cache(k[0, h], v[0, h], P) for h in range(Hkv)}
    cache = upload_oracle_cache(L.KVCache(B, Hkv, P), heads)
    qbits = synth.gen_bf16(942, Hq, range(B), range(Hq), 0, 1)[:, :, 0]
    qrot = O.rotate_q(qbits, 0)
    g = Hq // Hkv
    ref = np.concatenate([heads[(0, h)].decode(qrot[0, h * g:(h + 1) * g], TAU)
                          for h in range(Hkv)])[None]
    qr = torch.from_numpy(qrot.astype(np.float32)).cuda()
    ws = L.alloc_workspace(L.decode_workspace_bytes(B, Hkv, Hq, cache.n_packed, 3))
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    L.decode_attention(cache, qr, Hq, TAU, out, ws, num_splits=3)
    assert L.device_status() == 0
    assert_attention_close(out.cpu().numpy(), ref, "decode after a timeout")
