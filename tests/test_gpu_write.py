"""pkv_write on the GPU against the oracle's write: whole caches, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_05_gb300 as pkv
from paged_kv_attention_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu

from gpu_util import DeviceStep, to_dev, to_host_bits  # noqa: E402


def _expected_caches(step):
    kc, vc = step.key_cache.copy(), step.value_cache.copy()
    assert oracle.write(step.k, step.v, kc, vc, step.slot_mapping) == 0
    return kc, vc


@pytest.mark.parametrize("name", ["tiny_mixed", "mixed_chunked", "gqa_decode", "large_prefill"])
def test_write_bit_exact_whole_cache(name):
    step = W.build(W.spec(name))
    ek, ev = _expected_caches(step)
    ds = DeviceStep(step)
    ds.write()
    assert pkv.pkv_get_error() == 0
    assert torch.equal(ds.key_cache.view(torch.int16), to_dev(ek).view(torch.int16))
    assert torch.equal(ds.value_cache.view(torch.int16), to_dev(ev).view(torch.int16))


@pytest.mark.parametrize("hkv", [1, 2, 5, 8, 32, 48])
def test_write_small_ragged_with_pads(hkv):
    """Rows of 1 to 48 KV heads: a part of a warp's 2 KB piece, one piece,
    several, and a last piece partly filled."""
    spec = W.custom([3, 17, 0], [5, 1, 33], 2 * hkv, hkv, seed=100 + hkv, pad_tokens=7)
    step = W.build(spec)
    ek, ev = _expected_caches(step)
    ds = DeviceStep(step)
    ds.write()
    assert pkv.pkv_get_error() == 0
    assert np.array_equal(to_host_bits(ds.key_cache), ek)
    assert np.array_equal(to_host_bits(ds.value_cache), ev)


def test_write_out_of_range_slot_flagged_and_skipped():
    step = W.build(W.custom([0], [4], 2, 2, seed=5))
    step.slot_mapping[2] = step.key_cache.shape[0] * 16 + 3    # past the pool
    ek, ev = step.key_cache.copy(), step.value_cache.copy()
    assert oracle.write(step.k, step.v, ek, ev, step.slot_mapping) == oracle.ERR_SLOT_RANGE
    ds = DeviceStep(step)
    ds.write()
    assert pkv.pkv_get_error() == pkv.DEV_ERR_BITS["SLOT_RANGE"]
    assert pkv.pkv_get_error() == 0     # read clears
    assert np.array_equal(to_host_bits(ds.key_cache), ek)
    assert np.array_equal(to_host_bits(ds.value_cache), ev)


def test_write_all_pads_touches_nothing():
    step = W.build(W.custom([20], [3], 4, 4, seed=6))
    step.slot_mapping[:] = -1
    ds = DeviceStep(step)
    before_k = to_host_bits(ds.key_cache)
    ds.write()
    assert pkv.pkv_get_error() == 0
    assert np.array_equal(to_host_bits(ds.key_cache), before_k)
