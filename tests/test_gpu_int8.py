"""int8 KV cache on the GPU against the float64 oracle: the quantising write
bit for bit (codes, clamp, NaN), and decode-path attention over the codes
(every head grouping, splits, multi-token decode) within the tolerance;
requests too long for the decode path are reported and left unwritten."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_05_gb300 as pkv
from paged_kv_attention_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu

from gpu_util import DeviceStep, assert_close  # noqa: E402

KS, VS = 0.03, 0.04   # |x| > 127 * scale (about 3.8 and 5.1 for N(0, 1) data) saturates


def _history_codes(step):
    """The bf16 history caches as int8 codes (stale NaN slots become 0)."""
    nb, bs, hkv, d = step.key_cache.shape
    k8 = np.zeros((nb, bs, hkv, d), dtype=np.int8)
    v8 = np.zeros_like(k8)
    flat_k = step.key_cache.reshape(nb * bs, hkv, d)
    flat_v = step.value_cache.reshape(nb * bs, hkv, d)
    assert oracle.write_int8(flat_k, flat_v, k8, v8, np.arange(nb * bs, dtype=np.int64),
                             KS, VS) == 0
    return k8, v8


def run_int8(step, what, expect_err=0):
    k8, v8 = _history_codes(step)
    rk, rv = k8.copy(), v8.copy()
    assert oracle.write_int8(step.k, step.v, rk, rv, step.slot_mapping, KS, VS) == 0
    ref, err = oracle.attention_int8(step.q, rk, rv, KS, VS, step.query_start_loc,
                                     step.seq_lens, step.block_table, step.num_reqs, step.scale)
    assert err == 0
    ds = DeviceStep(step)
    dk, dv = torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda()
    pkv.pkv_write_int8(ds.k, ds.v, dk, dv, ds.slot_mapping, KS, VS)
    assert pkv.pkv_get_error() == 0
    assert np.array_equal(dk.cpu().numpy(), rk) and np.array_equal(dv.cpu().numpy(), rv), \
        "int8 write differs from the oracle's codes"
    pkv.pkv_attention_int8(ds.q, dk, dv, KS, VS, ds.qsl, ds.seq_lens, ds.block_table,
                           step.num_reqs, step.scale, ds.out)
    assert pkv.pkv_get_error() == expect_err
    got = ds.out_f64()
    return ds, got, ref


def _check_all(step, got, ref, what):
    n = int(step.query_start_loc[-1])
    assert_close(got[:n], ref[:n], what)
    assert np.isnan(got[n:]).all()


def test_int8_write_codes_clamp_and_nan():
    step = W.build(W.custom([20, 0, 37], [5, 33, 1], 8, 2, seed=41, pad_tokens=3))
    # plant special values in the new rows: NaN -> 0, +-inf and large -> +-127
    step.k[0, 0, :4] = W.bf16_bits(np.array([np.nan, np.inf, -np.inf, 1e3], dtype=np.float32))
    step.v[1, 1, 5:8] = W.bf16_bits(np.array([-1e3, 127.5 * 0.04, -0.02], dtype=np.float32))
    k8, v8 = _history_codes(step)
    rk, rv = k8.copy(), v8.copy()
    assert oracle.write_int8(step.k, step.v, rk, rv, step.slot_mapping, KS, VS) == 0
    ds = DeviceStep(step)
    dk, dv = torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda()
    pkv.pkv_write_int8(ds.k, ds.v, dk, dv, ds.slot_mapping, KS, VS)
    assert pkv.pkv_get_error() == 0
    assert np.array_equal(dk.cpu().numpy(), rk) and np.array_equal(dv.cpu().numpy(), rv)
    s0 = int(step.slot_mapping[0])
    assert rk[s0 // 16, s0 % 16, 0, :4].tolist() == [0, 127, -127, 127]


@pytest.mark.parametrize("hq,hkv,qn", [(8, 8, 1), (32, 8, 1), (32, 1, 1), (64, 2, 1),
                                       (48, 2, 1), (20, 1, 1), (8, 8, 4), (16, 4, 2),
                                       (12, 4, 5), (8, 1, 2), (17, 1, 1), (56, 2, 1)])
def test_int8_decode(hq, hkv, qn):
    ctx = [0, 1, 15, 16, 63, 200, 1023, 2100, 5000]
    step = W.build(W.custom(ctx, [qn] * len(ctx), hq, hkv, seed=hq * 7 + hkv + qn))
    ds, got, ref = run_int8(step, "int8 decode")
    _check_all(step, got, ref, "int8 decode hq=%d hkv=%d qn=%d" % (hq, hkv, qn))


@pytest.mark.parametrize("hq,hkv", [(32, 1), (8, 2)])
def test_int8_decode_queries_with_large_offset_and_spread(hq, hkv):
    """Queries 3 + 4 * N(0, 1): every score of a row carries a large common
    part and the softmax is sharp.  The kernels feed the codes to the MMAs as
    code + 1152, which adds 1152 * sum(q) to each score of a row and 1152 * L
    to the output sums before both are taken out; this checks that nothing of
    it shows at the tolerance, with and without splits."""
    ctx = [0, 17, 300, 2100, 5000, 9000]
    step = W.build(W.custom(ctx, [1] * len(ctx), hq, hkv, seed=4747 + hq))
    q = W.bf16_to_f32(step.q)
    step.q[...] = W.bf16_bits((3.0 + 4.0 * q).astype(np.float32))
    ds, got, ref = run_int8(step, "int8 shifted queries")
    _check_all(step, got, ref, "int8 decode, shifted queries hq=%d hkv=%d" % (hq, hkv))


@pytest.mark.parametrize("hq,hkv", [(32, 1), (24, 1)])
def test_int8_decode_several_units_per_worker(hq, hkv):
    """About 2,400 short requests and two long split ones over int8 codes:
    every warp of the two-tile kernel takes two or three units in turn, so
    the query buffer is refilled by TMA after the previous unit's fragments
    were read from it and the page ring's phases carry over."""
    rng = np.random.default_rng(4048 + hq)
    ctx = [int(c) for c in rng.integers(16, 300, size=2400)] + [5000, 9000]
    step = W.build(W.custom(ctx, [1] * len(ctx), hq, hkv, seed=hq * 17 + 3))
    ds, got, ref = run_int8(step, "int8 several units per worker")
    _check_all(step, got, ref, "int8 decode, several units per worker, hq=%d hkv=%d" % (hq, hkv))


def test_int8_long_requests_split_and_merge():
    step = W.build(W.custom([9000, 3, 16384], [1, 1, 1], 32, 8, seed=43))
    ds, got, ref = run_int8(step, "int8 split")
    _check_all(step, got, ref, "int8 split decode")


def test_int8_prefill_class_requests_are_reported_and_skipped():
    step = W.build(W.custom([100, 0, 50], [1, 40, 2], 8, 2, seed=44))
    ds, got, ref = run_int8(step, "int8 mixed", expect_err=pkv.DEV_ERR_BITS["INT8_PREFILL"])
    q = step.query_start_loc
    for r, ok in ((0, True), (1, False), (2, True)):
        rows = slice(int(q[r]), int(q[r + 1]))
        if ok:
            assert_close(got[rows], ref[rows], "int8 decode rows of request %d" % r)
        else:
            assert np.isnan(got[rows]).all(), "rows of the skipped request were written"


def test_int8_mha_decode_subset_full_lengths():
    step = W.build(W.subset(W.spec("mha_decode"), 24))
    ds, got, ref = run_int8(step, "int8 mha_decode subset")
    _check_all(step, got, ref, "int8 mha_decode subset")


@pytest.mark.parametrize("name", ["mha_decode", "gqa_decode", "mqa_long_decode"])
def test_int8_decode_full_size(name):
    """The bench's decode workloads at full size, every output row checked."""
    step = W.build(W.spec(name))
    ds, got, ref = run_int8(step, "int8 " + name)
    _check_all(step, got, ref, "int8 " + name)


def test_int8_split_size_does_not_change_the_result():
    """As for the bf16 cache: the same four decode requests over the same
    codes, alone (one wave of 64-key units) and as the first requests of a
    204-request batch (longer units), both within the tolerance of the
    oracle and within 1e-3 + one bf16 ulp of each other (P is rounded to fp16
    before P.V and the splits move each probability's reference max)."""
    ctx = [3000, 1500, 700, 9000] + [4096] * 200
    step = W.build(W.custom(ctx, [1] * len(ctx), 8, 2, seed=4343))
    ds, got, ref = run_int8(step, "int8 batch")
    in_batch = got[:4]
    k8, v8 = _history_codes(step)
    dk, dv = torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda()
    pkv.pkv_write_int8(ds.k, ds.v, dk, dv, ds.slot_mapping, KS, VS)
    alone = torch.empty_like(ds.out)
    alone.view(torch.int16).fill_(W.BF16_NAN)
    pkv.pkv_attention_int8(ds.q, dk, dv, KS, VS, ds.qsl, ds.seq_lens, ds.block_table, 4,
                           step.scale, alone)
    assert pkv.pkv_get_error() == 0
    by_itself = W.bf16_to_f32(alone.view(torch.int16).cpu().numpy().view(np.uint16))
    by_itself = by_itself.astype(np.float64)
    assert np.isnan(by_itself[4:]).all()
    by_itself = by_itself[:4]
    assert_close(in_batch, ref[:4], "int8 in the batch")
    assert_close(by_itself, ref[:4], "int8 alone")
    diff = np.abs(in_batch - by_itself)
    assert (diff <= 1e-3 + 2.0 ** -7 * np.maximum(np.abs(in_batch), np.abs(by_itself))).all(), \
        float(diff.max())
