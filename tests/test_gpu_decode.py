"""Decode attention (one query token per request) on the GPU against the
float64 oracle: small batches spanning several tiles, splits and ragged
tails for every head grouping; the full-size decode workloads; invariances."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_05_gb300 as pkv
from paged_kv_attention_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu

from gpu_util import DeviceStep, assert_close  # noqa: E402


def run_and_check(step, what):
    kc, vc = step.key_cache.copy(), step.value_cache.copy()
    assert oracle.write(step.k, step.v, kc, vc, step.slot_mapping) == 0
    ref, err = oracle.attention(step.q, kc, vc, step.query_start_loc, step.seq_lens,
                                step.block_table, step.num_reqs, step.scale)
    assert err == 0
    ds = DeviceStep(step)
    ds.write()
    ds.attention()
    assert pkv.pkv_get_error() == 0
    got = ds.out_f64()
    n = int(step.query_start_loc[-1])
    assert_close(got[:n], ref[:n], what)
    assert np.isnan(got[n:]).all(), "rows past the last request must not be written"
    return ds, got


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (8, 1), (16, 1), (32, 1), (32, 8), (12, 4)])
def test_decode_small_batches(hq, hkv):
    ctx = [0, 1, 15, 16, 63, 64, 65, 200, 1023, 1500, 2100]
    step = W.build(W.custom(ctx, [1] * len(ctx), hq, hkv, seed=hq * 100 + hkv))
    run_and_check(step, "decode hq=%d hkv=%d" % (hq, hkv))


@pytest.mark.parametrize("hq,hkv", [(17, 1), (40, 2), (24, 1), (64, 2)])
def test_decode_groups_above_16(hq, hkv):
    """Groups of 17 to 32 heads: a warp pair per unit, one 16-row tile each
    (the second tile partly filled below 32 heads), sharing the page ring;
    short requests, a page-aligned one and long ones split over several
    units."""
    ctx = [0, 15, 16, 300, 4095, 9000]
    step = W.build(W.custom(ctx, [1] * len(ctx), hq, hkv, seed=hq * 7 + hkv))
    run_and_check(step, "decode hq=%d hkv=%d" % (hq, hkv))


@pytest.mark.parametrize("hq,hkv", [(32, 1), (24, 1)])
def test_decode_groups_above_16_several_units_per_worker(hq, hkv):
    """About 2,400 short requests and two long split ones: with one unit per
    request, every warp pair takes two or three units in turn, so the unit
    hand-over through the pair's mailbox, the page ring's phases carried
    from unit to unit and the query fragments loaded per unit all run."""
    rng = np.random.default_rng(2024 + hq)
    ctx = [int(c) for c in rng.integers(16, 300, size=2400)] + [5000, 9000]
    step = W.build(W.custom(ctx, [1] * len(ctx), hq, hkv, seed=hq * 13 + 5))
    run_and_check(step, "decode, several units per worker, hq=%d hkv=%d" % (hq, hkv))


def test_decode_long_requests_split_and_merge():
    ctx = [5000, 9000, 3, 4097]
    step = W.build(W.custom(ctx, [1] * 4, 32, 8, seed=77))
    run_and_check(step, "split decode")


def test_decode_bit_identical_under_block_permutation():
    ctx = [700, 1800, 33]
    outs = []
    for seed in (1, 2):
        spec = W.custom(ctx, [1, 1, 1], 16, 4, seed=90)
        step = W.build(spec)
        # same values, different physical placement: permute the pool
        rng = np.random.default_rng(seed)
        perm = rng.permutation(step.key_cache.shape[0]).astype(np.int32)
        inv = np.argsort(perm).astype(np.int32)
        step.key_cache = step.key_cache[inv]
        step.value_cache = step.value_cache[inv]
        bt = step.block_table
        step.block_table = np.where(bt >= 0, perm[np.clip(bt, 0, None)], -1).astype(np.int32)
        sm = step.slot_mapping
        step.slot_mapping = np.where(sm >= 0, perm[sm // 16].astype(np.int64) * 16 + sm % 16, -1)
        ds, got = run_and_check(step, "permuted %d" % seed)
        outs.append(ds.out.view(torch.int16).cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("name", ["mha_decode", "gqa_decode", "mqa_long_decode"])
def test_decode_full_size(name):
    step = W.build(W.spec(name))
    run_and_check(step, name)


# Multi-token decode (speculative / multi-token steps): a request whose query
# tokens x heads of one KV head fit 16 rows (32 for groups above 16) runs in
# the decode kernel with a causal mask inside its own tokens.
@pytest.mark.parametrize("hq,hkv,qn", [(4, 4, 2), (4, 4, 5), (4, 4, 16), (8, 4, 8),
                                       (8, 2, 4), (16, 2, 2), (32, 1, 1), (12, 4, 5)])
def test_multi_token_decode(hq, hkv, qn):
    # ctx 253, 2045, 767 with qn up to 16: the last 256-key split starts after
    # the first token's last visible key, so that row sees nothing there
    ctx = [0, 3, 16, 253, 767, 2045, 1500]
    step = W.build(W.custom(ctx, [qn] * len(ctx), hq, hkv, seed=hq * 31 + qn))
    run_and_check(step, "multi-token decode hq=%d hkv=%d qn=%d" % (hq, hkv, qn))


@pytest.mark.parametrize("hq,hkv", [(4, 4), (16, 4), (32, 4), (64, 2)])
def test_decode_prefill_boundary(hq, hkv):
    """q_len at the decode row cap and one past it, in one batch with single
    tokens and long prefills."""
    G = hq // hkv
    cap = 16 if G <= 16 else 32
    at = max(cap // G, 1)
    q_len = [1, at, at + 1, 1, 200, at, 3, 130]
    ctx = [900, 40, 5000, 0, 17, 2300, 64, 0]
    step = W.build(W.custom(ctx, q_len, hq, hkv, seed=5 + G))
    run_and_check(step, "decode/prefill boundary hq=%d hkv=%d" % (hq, hkv))


def test_multi_token_decode_long_split():
    ctx = [9000, 4093, 12000]
    step = W.build(W.custom(ctx, [4, 4, 4], 16, 4, seed=61))
    run_and_check(step, "multi-token split decode")


def test_shared_prefix_blocks():
    """Requests whose block tables start with the same physical blocks (a
    shared prompt prefix): every reader sees the shared pages; new tokens are
    written past the shared part."""
    ctx = [600, 650, 700, 610]
    q_len = [1, 4, 40, 1]
    step = W.build(W.custom(ctx, q_len, 16, 4, seed=808))
    shared = 600 // 16          # whole pages below every request's ctx
    for r in range(1, 4):
        step.block_table[r, :shared] = step.block_table[0, :shared]
    run_and_check(step, "shared prefix")


def test_decode_longest_request():
    """A request at the longest supported length (a block-table row of 32,768
    blocks, 524,288 keys: the most splits of one request, all merged) next to
    a short one."""
    ctx = [32768 * 16 - 1, 40]
    step = W.build(W.custom(ctx, [1, 1], 8, 1, seed=71, num_blocks=32768 + 8, bt_width=32768))
    run_and_check(step, "longest request decode")


def test_split_size_does_not_change_the_result():
    """The same four decode requests, on the same cache, split two ways: alone
    (one wave of 64-key units) and as the first requests of a 204-request
    batch (384-key units).  Both match the oracle; against each other they
    differ only by rounding: the splits change each probability's reference
    max, and P is rounded to bf16 (2^-9 relative) before P.V, then the output
    to bf16 (one ulp, 2^-7 relative)."""
    ctx = [3000, 1500, 700, 9000] + [4096] * 200
    step = W.build(W.custom(ctx, [1] * len(ctx), 8, 2, seed=4242))
    ds = DeviceStep(step)
    ds.write()
    ds.attention()                       # all 204 requests
    alone = torch.empty_like(ds.out)
    alone.view(torch.int16).fill_(W.BF16_NAN)
    pkv.pkv_attention(ds.q, ds.key_cache, ds.value_cache, ds.qsl, ds.seq_lens, ds.block_table,
                      4, step.scale, alone)
    assert pkv.pkv_get_error() == 0
    in_batch = ds.out_f64()[:4]
    by_itself = W.bf16_to_f32(alone.view(torch.int16).cpu().numpy().view(np.uint16))
    by_itself = by_itself.astype(np.float64)
    assert np.isnan(by_itself[4:]).all()
    by_itself = by_itself[:4]
    kc, vc = step.key_cache.copy(), step.value_cache.copy()
    assert oracle.write(step.k, step.v, kc, vc, step.slot_mapping) == 0
    rows = np.repeat(np.arange(4, dtype=np.int64), 8)
    heads = np.tile(np.arange(8, dtype=np.int32), 4)
    ref, err = oracle.attention_sampled(step.q, kc, vc, step.query_start_loc, step.seq_lens,
                                        step.block_table, step.num_reqs, step.scale, rows, heads)
    assert err == 0
    ref = ref.reshape(4, 8, 128)
    assert_close(in_batch, ref, "in the batch")
    assert_close(by_itself, ref, "alone")
    diff = np.abs(in_batch - by_itself)
    assert (diff <= 1e-3 + 2.0 ** -7 * np.maximum(np.abs(in_batch), np.abs(by_itself))).all(), \
        float(diff.max())
