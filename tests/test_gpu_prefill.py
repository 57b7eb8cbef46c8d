"""Prefill and chunked-prefill attention (query_len > 1) and mixed batches on
the GPU against the float64 oracle: ragged query tiles, chunks continuing a
cached prompt, every head grouping, the trace step, the mixed 512-token batch
and the large prefill (sampled rows)."""
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


@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 1), (8, 2), (6, 3)])
def test_prefill_single_tile_and_ragged(hq, hkv):
    step = W.build(W.custom([0, 0, 0], [2, 17, 128], hq, hkv, seed=hq * 31 + hkv))
    run_and_check(step, "prefill hq=%d hkv=%d" % (hq, hkv))


def test_prefill_odd_group_single_head_items():
    """Hq / Hkv = 3: every work item carries one query tile, and the second
    tile's softmax warps stand by; prompts of several key tiles and a chunk
    after a cached context."""
    step = W.build(W.custom([0, 300, 0], [700, 150, 65], 12, 4, seed=303))
    run_and_check(step, "odd group")


def test_prefill_many_one_tile_items():
    """Two hundred short prompts (17 to 60 rows, one 64-key tile each): the
    score cursor of the MMA issuer runs up to two items ahead of P.V, across
    item boundaries, through the four-slot item ring and both Q buffers."""
    rng = np.random.default_rng(17)
    n = rng.integers(17, 61, 200).tolist()
    step = W.build(W.custom([0] * 200, n, 2, 2, seed=1717, pad_tokens=1))
    run_and_check(step, "one-tile items")


def test_prefill_rows_alone_and_in_a_large_batch():
    """Batch-composition invariance of the prefill path: four requests (a
    chunk after a 1024-token context, a 300-token prompt, a chunk after 100
    cached tokens, a 20-token prompt) computed in a step of their own (few
    work items, most SMs idle) and again at the head of a batch with 24 more
    prompts (hundreds of items, other tiles on every SM).  Both runs are
    checked against the oracle and against each other."""
    small_ctx, small_n = [1024, 0, 100, 0], [224, 300, 60, 20]
    small = W.build(W.custom(small_ctx, small_n, 16, 4, seed=909, pad_tokens=2))
    _, got_small = run_and_check(small, "prefill alone")
    rng = np.random.default_rng(910)
    extra = 24
    big = W.build(W.custom(small_ctx + [0] * extra, small_n + rng.integers(200, 257, extra).tolist(),
                           16, 4, seed=909, pad_tokens=2))
    # the shared requests get the same inputs in both runs
    n_small = int(small.query_start_loc[-1])
    big.qkv[:n_small] = small.qkv[:n_small]
    for r in range(len(small_ctx)):
        full, part = divmod(small_ctx[r], 16)
        for b in range(full + (1 if part else 0)):
            big.key_cache[big.block_table[r, b]] = small.key_cache[small.block_table[r, b]]
            big.value_cache[big.block_table[r, b]] = small.value_cache[small.block_table[r, b]]
    _, got_big = run_and_check(big, "prefill in a large batch")
    assert_close(got_small[:n_small], got_big[:n_small], "alone vs in a large batch")


def test_prefill_many_query_and_key_tiles():
    step = W.build(W.custom([0, 0], [300, 513], 4, 2, seed=12))
    run_and_check(step, "multi-tile prefill")


@pytest.mark.parametrize("ctx,n", [(1, 5), (15, 2), (16, 16), (100, 129), (1024, 224), (250, 7)])
def test_chunk_continuing_a_cached_prompt(ctx, n):
    step = W.build(W.custom([ctx, 3], [n, 40], 8, 2, seed=ctx + n))
    run_and_check(step, "chunk ctx=%d n=%d" % (ctx, n))


def test_trace_step_mixed():
    ds, got = run_and_check(W.build(W.spec("tiny_mixed")), "tiny_mixed")


def test_mixed_chunked_512_tokens():
    run_and_check(W.build(W.spec("mixed_chunked")), "mixed_chunked")


def test_mixed_decode_and_prefill_interleaved():
    ctx = [0, 700, 0, 33, 1500, 0]
    q_len = [40, 1, 1, 130, 1, 260]
    step = W.build(W.custom(ctx, q_len, 16, 4, seed=44, pad_tokens=5))
    run_and_check(step, "interleaved")


def test_two_chunks_match_one_prefill():
    """448 prompt tokens as one prefill vs 224 + 224 with the second chunk
    continuing the first: same rows (both within tolerance of the oracle and
    of each other)."""
    whole = W.build(W.custom([0], [448], 8, 2, seed=55))
    _, a = run_and_check(whole, "whole")
    two = W.build(W.custom([0, 224], [224, 224], 8, 2, seed=55))
    # same prompt: reuse the whole prefill's q/k/v rows and place the second
    # chunk's history (the first chunk) in its cache like the first request's
    two.qkv[:] = whole.qkv
    two.q = two.qkv[:, :8 * 128].reshape(448, 8, 128)
    two.k = two.qkv[:, 8 * 128:10 * 128].reshape(448, 2, 128)
    two.v = two.qkv[:, 10 * 128:].reshape(448, 2, 128)
    kc, vc = two.key_cache, two.value_cache
    for j in range(224):
        blk = two.block_table[1, j // 16]
        kc[blk, j % 16] = whole.k[j]
        vc[blk, j % 16] = whole.v[j]
    _, b = run_and_check(two, "two chunks")
    # chunk 2's rows equal the whole prefill's rows 224..447
    diff = np.abs(a[224:448] - b[224:448])
    assert (diff <= 1e-2 + 1e-2 * np.abs(a[224:448])).all()


def test_prefill_bit_identical_under_block_permutation():
    outs = []
    for seed in (3, 4):
        step = W.build(W.custom([100, 0], [60, 200], 8, 2, seed=66))
        rng = np.random.default_rng(seed)
        perm = rng.permutation(step.key_cache.shape[0]).astype(np.int32)
        inv = np.argsort(perm).astype(np.int32)
        step.key_cache = step.key_cache[inv]
        step.value_cache = step.value_cache[inv]
        bt = step.block_table
        step.block_table = np.where(bt >= 0, perm[np.clip(bt, 0, None)], -1).astype(np.int32)
        sm = step.slot_mapping
        step.slot_mapping = np.where(sm >= 0, perm[sm // 16].astype(np.int64) * 16 + sm % 16, -1)
        ds, _ = run_and_check(step, "permuted %d" % seed)
        outs.append(ds.out.view(torch.int16).cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


def test_large_prefill_sampled_rows():
    step = W.build(W.spec("large_prefill"))
    kc, vc = step.key_cache.copy(), step.value_cache.copy()
    assert oracle.write(step.k, step.v, kc, vc, step.slot_mapping) == 0
    ds = DeviceStep(step)
    ds.write()
    ds.attention()
    assert pkv.pkv_get_error() == 0
    got = ds.out_f64()
    rng = np.random.default_rng(0)
    # rows at tile edges and in the ragged parts of every request, all heads
    rows = []
    for r in range(step.num_reqs):
        q0 = int(step.query_start_loc[r])
        rows += [q0, q0 + 1, q0 + 127, q0 + 128, q0 + 1023, q0 + 2047]
        rows += (q0 + rng.integers(0, 2048, 4)).tolist()
    rows = np.repeat(np.array(rows, dtype=np.int64), 4)
    heads = rng.integers(0, step.spec.hq, rows.shape[0]).astype(np.int32)
    ref, err = oracle.attention_sampled(step.q, kc, vc, step.query_start_loc, step.seq_lens,
                                        step.block_table, step.num_reqs, step.scale, rows, heads)
    assert err == 0
    assert_close(got[rows, heads], ref, "large_prefill sampled")
    assert np.isfinite(got).all()


def test_large_prefill_one_whole_request():
    """The full large_prefill step (8 prompts of 2048 tokens, Hq 64 / Hkv 8,
    causal) on the GPU, and one of its requests compared element by element:
    all 2048 rows x 64 heads x 128 columns, i.e. every query tile, every
    head pair and every diagonal key tile of the launch's geometry."""
    step = W.build(W.spec("large_prefill"))
    kc, vc = step.key_cache.copy(), step.value_cache.copy()
    assert oracle.write(step.k, step.v, kc, vc, step.slot_mapping) == 0
    ds = DeviceStep(step)
    ds.write()
    ds.attention()
    assert pkv.pkv_get_error() == 0
    got = ds.out_f64()
    r = 5
    qsl = step.query_start_loc
    q0, q1 = int(qsl[r]), int(qsl[r + 1])
    sub_qsl = np.array([q0, q1], dtype=np.int32)
    ref, err = oracle.attention(step.q, kc, vc, sub_qsl, step.seq_lens[r:r + 1],
                                step.block_table[r:r + 1], 1, step.scale)
    assert err == 0
    assert_close(got[q0:q1], ref[q0:q1], "large_prefill request %d" % r)
    assert np.isfinite(got).all()


def test_prefill_scores_growing_along_the_keys():
    """Scores that rise steadily along the keys (by about 2^8 in the log2
    domain every 128 keys): the running maximum grows past the rescale
    threshold inside most key tiles, so the max pass, the reload of the scores
    and the rescale of O run on most tiles, next to tiles that take the
    single-pass route."""
    step = W.build(W.custom([600, 0], [300, 700], 4, 2, seed=21))
    u = np.full(128, 0.5, dtype=np.float32)
    step.q[:] = W.bf16_bits(u)[None, None, :]
    R = step.num_reqs
    for r in range(R):
        ctx = int(step.seq_lens[r]) - int(step.query_start_loc[r + 1] - step.query_start_loc[r])
        for pos in range(int(step.seq_lens[r])):
            kv = W.bf16_bits(u * np.float32(pos / 64.0))
            if pos < ctx:
                blk = step.block_table[r, pos // 16]
                step.key_cache[blk, pos % 16, :, :] = kv[None, :]
            else:
                step.k[step.query_start_loc[r] + pos - ctx, :, :] = kv[None, :]
    run_and_check(step, "growing scores")


def test_prefill_chunk_after_long_context():
    """A 200-row chunk continuing a 32,768-token cached prompt: items of 258
    key tiles, the steady state of the prefill kernel, next to a decode."""
    step = W.build(W.custom([32768, 900], [200, 1], 8, 2, seed=73))
    run_and_check(step, "prefill after a long context")


def test_more_requests_than_one_plan_pass():
    """2,600 requests: the step plan takes them in passes of 1,024, carrying
    every offset (decode units by length class, split pairs, partial rows,
    prefill tiles) from one pass to the next.  Decodes of 1 to 4 tokens and
    prefill chunks are spread over all three passes."""
    rng = np.random.default_rng(2600)
    n = 2600
    kind = rng.choice(3, size=n, p=[0.9, 0.07, 0.03])  # decode, multi-token decode, chunk
    q_len = np.where(kind == 0, 1, np.where(kind == 1, rng.integers(2, 5, n),
                                            rng.integers(20, 200, n)))
    ctx = np.where(kind == 2, rng.integers(0, 300, n), rng.integers(1, 160, n))
    step = W.build(W.custom(ctx.tolist(), q_len.tolist(), 4, 2, seed=2600, pad_tokens=3))
    run_and_check(step, "2600 requests")
