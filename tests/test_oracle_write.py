"""Pins the oracle's cache write: brute force over the whole cache, pads,
out-of-range slots and strided (fused-qkv) rows."""
import numpy as np

import oracle
from paged_kv_attention_05_gb300 import workloads as W

BS, D = 16, 128


def _brute_write(k, v, kc, vc, slots):
    """Token by token: slot -> (slot // 16, slot % 16), whole [hkv, D] rows."""
    kc, vc = kc.copy(), vc.copy()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        kc[s // BS, s % BS] = k[t]
        vc[s // BS, s % BS] = v[t]
    return kc, vc


def test_write_equals_brute_force_over_whole_cache():
    rng = np.random.default_rng(1)
    nb, hkv, n = 12, 4, 40
    kc = rng.integers(0, 1 << 16, size=(nb, BS, hkv, D), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(nb, BS, hkv, D), dtype=np.uint16)
    k = rng.integers(0, 1 << 16, size=(n, hkv, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(n, hkv, D), dtype=np.uint16)
    slots = rng.permutation(nb * BS)[:n].astype(np.int64)
    slots[[3, 17, 39]] = -1
    ek, ev = _brute_write(k, v, kc, vc, slots)
    assert oracle.write(k, v, kc, vc, slots) == 0
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def test_pad_tokens_never_touch_the_cache():
    rng = np.random.default_rng(2)
    kc = rng.integers(0, 1 << 16, size=(5, BS, 2, D), dtype=np.uint16)
    vc = kc.copy()
    before = kc.copy()
    k = rng.integers(0, 1 << 16, size=(6, 2, D), dtype=np.uint16)
    slots = np.full(6, -1, dtype=np.int64)
    assert oracle.write(k, k, kc, vc, slots) == 0
    assert np.array_equal(kc, before) and np.array_equal(vc, before)


def test_out_of_range_slot_is_skipped_and_reported():
    rng = np.random.default_rng(3)
    kc = np.zeros((2, BS, 1, D), dtype=np.uint16)
    vc = kc.copy()
    k = rng.integers(1, 1 << 15, size=(3, 1, D), dtype=np.uint16)
    slots = np.array([0, 2 * BS, 31], dtype=np.int64)   # middle one is past the pool
    err = oracle.write(k, k, kc, vc, slots)
    assert err == oracle.ERR_SLOT_RANGE
    assert np.array_equal(kc[0, 0], k[0]) and np.array_equal(kc[1, 15], k[2])
    assert int((kc != 0).any(axis=(2, 3)).sum()) == 2


def test_write_from_fused_qkv_rows_of_trace_step():
    step = W.build(W.spec("tiny_mixed"))
    assert not step.k.flags.c_contiguous            # row views of the fused qkv
    kc, vc = step.key_cache.copy(), step.value_cache.copy()
    ek, ev = _brute_write(np.ascontiguousarray(step.k), np.ascontiguousarray(step.v),
                          kc, vc, step.slot_mapping)
    assert oracle.write(step.k, step.v, kc, vc, step.slot_mapping) == 0
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)
    # the 300 scheduled tokens land at 300 distinct slots; the 4 pads nowhere
    assert int((step.slot_mapping >= 0).sum()) == 300
    assert (step.slot_mapping[300:] == -1).all()
