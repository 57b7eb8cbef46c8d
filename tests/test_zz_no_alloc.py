"""pkv_attention_noalloc, the attention call for callers that cannot allocate
device memory (services with a device-memory footprint fixed at start-up,
hosts whose own allocator the library must not bypass, loops that cannot take
the synchronisation of a cudaMalloc).  It keeps its scratch in a static
device array instead of a cudaMalloc'd workspace; its results must match
pkv_attention's.

This file is collected last on purpose: if it fails, a run that stops at
the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_attention_05_gb300 as pkv
from paged_kv_attention_05_gb300 import workloads as W

FAKE = 0x10000


def test_refuses_a_batch_beyond_the_static_scratch():
    """Host-side check, before any device work: 4096 requests x 8 KV heads x
    the longest block-table rows need far more than the 32 MiB array."""
    lib = pkv.load()
    fn = lib.pkv_attention_noalloc
    i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [vp, i64, i64, i32, vp, vp, i64, i32, i32, i32, vp, vp, vp, i64, i32, f32, vp,
                   i64, vp]
    rc = fn(FAKE, 4096, 4096, 32, FAKE, FAKE, 100000, 16, 8, 128, FAKE, FAKE, FAKE, 32768, 4096,
            0.088, FAKE, 4096, None)
    assert rc == -2


def test_refuses_kv_heads_beyond_the_unit_packing():
    """Host-side check, as pkv_attention's: a decode unit packs the KV head in
    16 bits, so num_kv_heads above 32767 is refused before any device work."""
    lib = pkv.load()
    fn = lib.pkv_attention_noalloc
    i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [vp, i64, i64, i32, vp, vp, i64, i32, i32, i32, vp, vp, vp, i64, i32, f32, vp,
                   i64, vp]
    hkv = 65536
    rc = fn(FAKE, hkv * 128, 1, hkv, FAKE, FAKE, 10, 16, hkv, 128, FAKE, FAKE, FAKE, 1, 1,
            0.088, FAKE, hkv * 128, None)
    assert rc == -2


def _ref_and_noalloc(step):
    from gpu_util import DeviceStep, assert_close, to_host_bits
    ds = DeviceStep(step)
    ds.write()
    ds.attention()                      # the allocating entry point
    assert pkv.pkv_get_error() == 0
    ref = ds.out_f64()
    n = int(step.query_start_loc[-1])
    for call in range(2):               # two calls in a row on the shared array
        out = torch.empty_like(ds.out)
        out.view(torch.int16).fill_(W.BF16_NAN)
        pkv.pkv_attention_noalloc(ds.q, ds.key_cache, ds.value_cache, ds.qsl, ds.seq_lens,
                                  ds.block_table, step.num_reqs, step.scale, out)
        torch.cuda.synchronize()
        got = W.bf16_to_f32(to_host_bits(out)).astype(np.float64)
        assert_close(got[:n], ref[:n], "no-alloc call %d" % call)
        assert np.isnan(got[n:]).all()


@pytest.mark.gpu
def test_matches_pkv_attention_mixed_batch():
    step = W.build(W.custom([0, 700, 1500, 33, 0], [40, 1, 1, 130, 1], 16, 4, seed=404,
                            pad_tokens=3))
    _ref_and_noalloc(step)


@pytest.mark.gpu
def test_matches_pkv_attention_split_decode():
    step = W.build(W.subset(W.spec("gqa_decode"), 4))   # 8193 keys: split over several units
    _ref_and_noalloc(step)
