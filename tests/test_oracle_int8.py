"""Pins for the oracle's int8 KV cache (one fp32 scale per cache, symmetric
codes clamp(rne(x / scale), -127, 127)): closed forms of the code, the
round-trip bound, the write placement shared with the bf16 write, and the
attention reducing to the (already pinned) bf16 attention whenever code *
scale is exactly a bf16 value."""
import numpy as np
import pytest

import oracle
from paged_kv_attention_05_gb300 import workloads as W


def _codes(x, scale):
    """int8 codes of float32 values through the oracle's write (one token,
    one head, d = len(x))."""
    d = len(x)
    k = W.bf16_bits(np.asarray(x, dtype=np.float32)).reshape(1, 1, d)
    kc = np.zeros((1, 16, 1, d), dtype=np.int8)
    vc = np.zeros_like(kc)
    assert oracle.write_int8(k, k, kc, vc, np.array([3], dtype=np.int64), scale, scale) == 0
    assert np.array_equal(kc, vc)
    return kc[0, 3, 0].astype(np.int64)


def test_codes_of_exact_multiples_ties_and_clamp():
    s = 0.0625  # 2^-4: every c * s with |c| <= 127 is exact in bf16 and fp32
    c = np.arange(-127, 128)
    assert np.array_equal(_codes(c * s, s), c)
    # half-way values round to the even neighbour: 0.5 -> 0, 1.5 -> 2, -2.5 -> -2
    assert _codes(np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5]) * s, s).tolist() == [0, 2, 2, 0, -2, -2]
    # beyond +-127.5 steps the code saturates symmetrically (never -128)
    assert _codes(np.array([128, 200, -128, -1e30, 1e30]) * s, s).tolist() == [127, 127, -127, -127, 127]
    # NaN input stores code 0 (the reading taken where the pages are silent)
    assert _codes(np.array([np.nan, 1.0]), 1.0).tolist() == [0, 1]


def test_round_trip_error_is_at_most_half_a_step():
    rng = np.random.default_rng(5)
    for s in (0.01, 0.037, 1.0 / 30):
        x = W.bf16_to_f32(W.bf16_bits(rng.uniform(-127 * s, 127 * s, 512).astype(np.float32)))
        c = _codes(x, s)
        sf = np.float64(np.float32(s))
        err = np.abs(c * sf - x.astype(np.float64))
        # half a step, plus the rounding of the fp32 division x / s
        assert (err <= 0.5 * sf + np.abs(x.astype(np.float64)) * 2.0 ** -23).all()
        # and no code is off by one: the other neighbour is always farther
        assert (np.abs((c - np.sign(x - c * sf)) * sf - x) >= err - 1e-12).all()
        assert np.abs(c).max() <= 127


def test_write_places_codes_where_the_bf16_write_places_values():
    step = W.build(W.custom([20, 0, 37], [5, 33, 1], 4, 2, seed=9, pad_tokens=3))
    kb, vb = step.key_cache.copy(), step.value_cache.copy()
    assert oracle.write(step.k, step.v, kb, vb, step.slot_mapping) == 0
    k8 = np.zeros(step.key_cache.shape, dtype=np.int8)
    v8 = np.zeros_like(k8)
    assert oracle.write_int8(step.k, step.v, k8, v8, step.slot_mapping, 0.05, 0.03) == 0
    written = np.zeros(k8.shape[:2], dtype=bool)
    for s in step.slot_mapping:
        if s >= 0:
            written[s // 16, s % 16] = True
    # where the bf16 write put a row, the int8 write put that row's codes
    kx = W.bf16_to_f32(kb[written]).astype(np.float64)
    vx = W.bf16_to_f32(vb[written]).astype(np.float64)
    saturated = 0
    for c8, x, sc in ((k8, kx, 0.05), (v8, vx, 0.03)):
        sf = np.float64(np.float32(sc))
        c = c8[written].astype(np.float64)
        inside = np.abs(x) <= 127 * sf
        assert (np.abs(c * sf - x) <= 0.5 * sf + np.abs(x) * 2.0 ** -23)[inside].all()
        assert (c[~inside] == 127 * np.sign(x[~inside])).all()
        saturated += int((~inside).sum())
    assert saturated > 0  # the clamp is exercised (|v| > 127 * 0.03 occurs)
    assert not k8[~written].any() and not v8[~written].any()
    # an out-of-range slot is reported and skipped, as in the bf16 write
    bad = step.slot_mapping.copy()
    bad[0] = k8.shape[0] * 16
    assert oracle.write_int8(step.k, step.v, k8, v8, bad, 0.05, 0.03) == oracle.ERR_SLOT_RANGE


def _int8_step(seed, ks, vs):
    """A mixed step whose int8 caches hold random codes and whose bf16 caches
    hold exactly code * scale (scales are powers of two)."""
    step = W.build(W.custom([40, 0, 17, 70], [1, 20, 3, 1], 8, 2, seed=seed))
    rng = np.random.default_rng(seed)
    k8 = rng.integers(-127, 128, step.key_cache.shape).astype(np.int8)
    v8 = rng.integers(-127, 128, step.value_cache.shape).astype(np.int8)
    kb = W.bf16_bits((k8 * np.float32(ks)).astype(np.float32))
    vb = W.bf16_bits((v8 * np.float32(vs)).astype(np.float32))
    return step, k8, v8, kb, vb


def test_attention_over_codes_equals_bf16_attention_over_their_values():
    ks, vs = 2.0 ** -5, 2.0 ** -3
    step, k8, v8, kb, vb = _int8_step(31, ks, vs)
    a = (step.q, step.query_start_loc, step.seq_lens, step.block_table, step.num_reqs, step.scale)
    ref, e1 = oracle.attention(a[0], kb, vb, *a[1:])
    got, e2 = oracle.attention_int8(a[0], k8, v8, ks, vs, *a[1:])
    assert e1 == e2 == 0
    n = int(step.query_start_loc[-1])
    assert np.abs(got[:n] - ref[:n]).max() <= 1e-12 * max(1.0, np.abs(ref[:n]).max())
    assert np.isnan(got[n:]).all()


def test_value_scale_scales_the_output_and_key_scale_trades_with_softmax_scale():
    ks, vs = 0.013, 0.021
    step, k8, v8, _, _ = _int8_step(32, ks, vs)
    a = (step.query_start_loc, step.seq_lens, step.block_table, step.num_reqs)
    base, _ = oracle.attention_int8(step.q, k8, v8, ks, vs, *a, step.scale)
    twice, _ = oracle.attention_int8(step.q, k8, v8, ks, 2 * vs, *a, step.scale)
    n = int(step.query_start_loc[-1])
    np.testing.assert_allclose(twice[:n], 2 * base[:n], rtol=1e-12, atol=1e-15)
    # K = code * ks under softmax scale t  ==  K = code * (2 ks) under t / 2
    other, _ = oracle.attention_int8(step.q, k8, v8, 2 * ks, vs, *a, step.scale / 2)
    np.testing.assert_allclose(other[:n], base[:n], rtol=1e-9, atol=1e-12)
