"""Pins the float64 oracle's paged attention to what the pages and the
mathematics fix: the dense textbook form (numpy and torch's float64 SDPA), the
key counts of the forward-pass trace, closed forms and invariances."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import blocks, brute
from paged_kv_attention_05_gb300 import workloads as W

D = 128
BS = 16


def _bits(x):
    return W.bf16_bits(np.asarray(x, dtype=np.float32))


def _f(bits):
    return W.bf16_to_f32(bits).astype(np.float64)


def paged_batch(hist_k, hist_v, q_rows, hkv, rng, num_blocks=None, bt_extra=2):
    """Lays contiguous per-request K/V ([L_r, hkv, D] bf16 bits) into a
    shuffled block pool and returns the oracle inputs.  q_rows: list of
    [n_r, hq, D] bf16 bits.  The cache is NaN everywhere no key lives."""
    R = len(hist_k)
    need = [blocks.blocks_needed(k.shape[0]) for k in hist_k]
    nb = num_blocks or (sum(need) + 5)
    perm = rng.permutation(nb).astype(np.int32)
    width = max(need + [1]) + bt_extra
    bt = np.full((R, width), -1, dtype=np.int32)
    kc = np.full((nb, BS, hkv, D), W.BF16_NAN, dtype=np.uint16)
    vc = kc.copy()
    used = 0
    for r in range(R):
        bt[r, :need[r]] = perm[used:used + need[r]]
        used += need[r]
        for j in range(hist_k[r].shape[0]):
            kc[bt[r, j // BS], j % BS] = hist_k[r][j]
            vc[bt[r, j // BS], j % BS] = hist_v[r][j]
    q = np.concatenate(q_rows, axis=0)
    qsl = np.zeros(R + 1, dtype=np.int32)
    qsl[1:] = np.cumsum([x.shape[0] for x in q_rows])
    seq_lens = np.array([k.shape[0] for k in hist_k], dtype=np.int32)
    return q, kc, vc, qsl, seq_lens, bt


def random_case(ctx, q_len, hq, hkv, seed, std=1.0):
    rng = np.random.default_rng(seed)
    hk, hv, qs = [], [], []
    for c, n in zip(ctx, q_len):
        hk.append(_bits(rng.standard_normal((c + n, hkv, D)) * std))
        hv.append(_bits(rng.standard_normal((c + n, hkv, D)) * std))
        qs.append(_bits(rng.standard_normal((n, hq, D)) * std))
    return hk, hv, qs, rng


@pytest.mark.parametrize("hq,hkv", [(4, 4), (4, 2), (4, 1), (6, 3)])
def test_paged_oracle_equals_dense_brute_force(hq, hkv):
    ctx, q_len = [0, 5, 37, 16], [7, 1, 4, 16]
    hk, hv, qs, rng = random_case(ctx, q_len, hq, hkv, seed=hq * 10 + hkv)
    q, kc, vc, qsl, sl, bt = paged_batch(hk, hv, qs, hkv, rng)
    scale = 1 / math.sqrt(D)
    out, err = oracle.attention(q, kc, vc, qsl, sl, bt, len(ctx), scale)
    assert err == 0
    for r in range(len(ctx)):
        ref = brute.dense_causal_attention(_f(qs[r]), _f(hk[r]), _f(hv[r]), ctx[r], scale)
        np.testing.assert_allclose(out[qsl[r]:qsl[r + 1]], ref, rtol=1e-12, atol=1e-13)


def test_paged_oracle_equals_torch_sdpa_float64():
    hq, hkv = 8, 2
    ctx, q_len = [3, 0, 20], [5, 9, 1]
    hk, hv, qs, rng = random_case(ctx, q_len, hq, hkv, seed=11)
    q, kc, vc, qsl, sl, bt = paged_batch(hk, hv, qs, hkv, rng)
    scale = 0.07
    out, err = oracle.attention(q, kc, vc, qsl, sl, bt, len(ctx), scale)
    assert err == 0
    for r in range(len(ctx)):
        n, L = q_len[r], ctx[r] + q_len[r]
        qt = torch.from_numpy(_f(qs[r])).permute(1, 0, 2)            # [hq, n, D]
        kt = torch.from_numpy(_f(hk[r])).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
        vt = torch.from_numpy(_f(hv[r])).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
        mask = torch.arange(L)[None, :] <= (ctx[r] + torch.arange(n))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, attn_mask=mask, scale=scale).permute(1, 0, 2).numpy()
        np.testing.assert_allclose(out[qsl[r]:qsl[r + 1]], ref, rtol=1e-11, atol=1e-12)


def test_single_key_returns_its_value_exactly():
    hq, hkv = 4, 2
    hk, hv, qs, rng = random_case([0, 0], [1, 1], hq, hkv, seed=3)
    q, kc, vc, qsl, sl, bt = paged_batch(hk, hv, qs, hkv, rng)
    out, err = oracle.attention(q, kc, vc, qsl, sl, bt, 2, 1 / math.sqrt(D))
    assert err == 0
    for r in range(2):
        for h in range(hq):
            assert np.array_equal(out[r, h], _f(hv[r][0, h // 2]))


def test_trace_key_counts_through_equal_keys():
    """All keys equal -> uniform weights over the visible keys.  With value
    dim 0 = key position, the output is the mean visible position
    (ctx + i) / 2, which pins how many keys each row reads: 541, 130 and
    298 + causal for the three requests of the forward-pass trace."""
    with open(os.path.join(os.path.dirname(__file__), "golden", "forward_pass_trace.json")) as f:
        g = json.load(f)
    ctx, q_len = g["num_computed_tokens"], g["num_scheduled_tokens"]
    hq, hkv = 4, 2
    rng = np.random.default_rng(5)
    hk, hv, qs = [], [], []
    for c, n in zip(ctx, q_len):
        L = c + n
        key = _bits(rng.standard_normal((1, hkv, D)))
        hk.append(np.repeat(key, L, axis=0))
        val = np.zeros((L, hkv, D), dtype=np.float32)
        val[:, :, 0] = np.arange(L)[:, None]   # rounded to bf16; the mean uses the rounded values
        val[:, :, 1] = 1.0
        hv.append(_bits(val))
        qs.append(_bits(rng.standard_normal((n, hq, D))))
    q, kc, vc, qsl, sl, bt = paged_batch(hk, hv, qs, hkv, rng)
    out, err = oracle.attention(q, kc, vc, qsl, sl, bt, 3, 1 / math.sqrt(D))
    assert err == 0
    for r in range(3):
        pos_bf16 = _f(hv[r][:, 0, 0])
        for i in range(q_len[r]):
            visible = ctx[r] + i + 1
            row = out[qsl[r] + i]
            np.testing.assert_allclose(row[:, 0], pos_bf16[:visible].mean(), rtol=1e-12)
            np.testing.assert_allclose(row[:, 1], 1.0, rtol=1e-12)
        # the last row of each request reads exactly keys_read keys
        assert ctx[r] + q_len[r] == g["keys_read"][r]


def test_one_hot_scores_select_one_value_row():
    hq, hkv, L = 2, 1, 40
    rng = np.random.default_rng(9)
    target = 23
    key = np.zeros((L, hkv, D), dtype=np.float32)
    key[target, 0, 0] = 1.0
    val = rng.standard_normal((L, hkv, D)).astype(np.float32)
    qv = np.zeros((1, hq, D), dtype=np.float32)
    qv[0, :, 0] = 64.0
    hk, hv, qs = [_bits(key)], [_bits(val)], [_bits(qv)]
    q, kc, vc, qsl, sl, bt = paged_batch(hk, hv, qs, hkv, rng)
    out, err = oracle.attention(q, kc, vc, qsl, sl, bt, 1, 16.0)   # score gap 1024
    assert err == 0
    np.testing.assert_allclose(out[0, 0], _f(hv[0][target, 0]), rtol=0, atol=1e-300)


def test_block_permutation_changes_nothing():
    hq, hkv = 4, 2
    ctx, q_len = [50, 3], [1, 30]
    hk, hv, qs, _ = random_case(ctx, q_len, hq, hkv, seed=21)
    outs = []
    for seed in range(3):
        q, kc, vc, qsl, sl, bt = paged_batch(hk, hv, qs, hkv, np.random.default_rng(seed),
                                             num_blocks=40)
        outs.append(oracle.attention(q, kc, vc, qsl, sl, bt, 2, 0.09)[0])
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_gqa_equals_mha_with_repeated_kv_heads():
    hq, hkv = 6, 2
    ctx, q_len = [17, 0], [1, 12]
    hk, hv, qs, rng = random_case(ctx, q_len, hq, hkv, seed=31)
    q, kc, vc, qsl, sl, bt = paged_batch(hk, hv, qs, hkv, rng)
    gqa = oracle.attention(q, kc, vc, qsl, sl, bt, 2, 0.1)[0]
    hk2 = [np.repeat(x, hq // hkv, axis=1) for x in hk]
    hv2 = [np.repeat(x, hq // hkv, axis=1) for x in hv]
    q, kc, vc, qsl, sl, bt = paged_batch(hk2, hv2, qs, hq, rng)
    mha = oracle.attention(q, kc, vc, qsl, sl, bt, 2, 0.1)[0]
    assert np.array_equal(gqa, mha)


def test_request_order_does_not_matter():
    hq, hkv = 4, 1
    ctx, q_len = [10, 0, 33], [1, 8, 2]
    hk, hv, qs, rng = random_case(ctx, q_len, hq, hkv, seed=41)
    q, kc, vc, qsl, sl, bt = paged_batch(hk, hv, qs, hkv, rng)
    a = oracle.attention(q, kc, vc, qsl, sl, bt, 3, 0.1)[0]
    order = [2, 0, 1]
    q, kc, vc, qsl2, sl, bt = paged_batch([hk[i] for i in order], [hv[i] for i in order],
                                          [qs[i] for i in order], hkv, rng)
    b = oracle.attention(q, kc, vc, qsl2, sl, bt, 3, 0.1)[0]
    for new, old in enumerate(order):
        assert np.array_equal(b[qsl2[new]:qsl2[new + 1]], a[qsl[old]:qsl[old + 1]])


def test_two_chunks_equal_one_prefill():
    """A 448-token prompt as one prefill, or as a 224-token chunk then a
    224-token chunk with 224 tokens cached, gives the same rows."""
    hq, hkv, n = 2, 1, 448
    rng = np.random.default_rng(51)
    k = _bits(rng.standard_normal((n, hkv, D)))
    v = _bits(rng.standard_normal((n, hkv, D)))
    qq = _bits(rng.standard_normal((n, hq, D)))
    q, kc, vc, qsl, sl, bt = paged_batch([k], [v], [qq], hkv, rng)
    whole = oracle.attention(q, kc, vc, qsl, sl, bt, 1, 0.088)[0]
    q, kc, vc, qsl, sl, bt = paged_batch([k[:224], k], [v[:224], v], [qq[:224], qq[224:]], hkv, rng)
    parts = oracle.attention(q, kc, vc, qsl, sl, bt, 2, 0.088)[0]
    assert np.array_equal(parts, whole)


def test_rows_outside_requests_untouched():
    hq, hkv = 4, 2
    hk, hv, qs, rng = random_case([4], [3], hq, hkv, seed=61)
    q, kc, vc, qsl, sl, bt = paged_batch(hk, hv, qs, hkv, rng)
    q = np.concatenate([q, _bits(np.ones((4, hq, D)))], axis=0)   # 4 padding rows
    out, err = oracle.attention(q, kc, vc, qsl, sl, bt, 1, 0.1)
    assert err == 0
    assert np.isfinite(out[:3]).all() and np.isnan(out[3:]).all()


def test_invalid_requests_are_skipped_and_reported():
    hq, hkv = 2, 1
    hk, hv, qs, rng = random_case([5, 5, 5, 5], [2, 2, 2, 2], hq, hkv, seed=71)
    q, kc, vc, qsl, sl, bt = paged_batch(hk, hv, qs, hkv, rng, bt_extra=0)
    nb = kc.shape[0]
    cases = []
    sl1 = sl.copy(); sl1[1] = 1                        # seq_len < query_len
    cases.append((qsl, sl1, bt, 1, oracle.ERR_SEQ_LEN))
    bt2 = bt.copy(); bt2[2, 0] = nb                    # block id out of range
    cases.append((qsl, sl, bt2, 2, oracle.ERR_BLOCK_ID))
    sl3 = sl.copy(); sl3[3] = 40                       # row too short for seq_len
    cases.append((qsl, sl3, bt, 3, oracle.ERR_BT_WIDTH))
    qsl4 = qsl.copy(); qsl4[2] = 1                     # decreasing start locations
    cases.append((qsl4, sl, bt, None, oracle.ERR_QSL))
    good, _ = oracle.attention(q, kc, vc, qsl, sl, bt, 4, 0.1)
    for qs_, sl_, bt_, bad, bit in cases:
        out, err = oracle.attention(q, kc, vc, qs_, sl_, bt_, 4, 0.1)
        assert err & bit
        if bad is not None:
            assert np.isnan(out[qs_[bad]:qs_[bad + 1]]).all()
            for r in range(4):
                if r != bad:
                    assert np.array_equal(out[qs_[r]:qs_[r + 1]], good[qsl[r]:qsl[r + 1]])


def test_sampled_rows_match_full_batch():
    step = W.build(W.custom([30, 0, 7], [1, 20, 3], 8, 2, seed=81))
    kc, vc = step.key_cache.copy(), step.value_cache.copy()
    oracle.write(step.k, step.v, kc, vc, step.slot_mapping)
    full, err = oracle.attention(step.q, kc, vc, step.query_start_loc, step.seq_lens,
                                 step.block_table, step.num_reqs, step.scale)
    assert err == 0
    rows = np.array([0, 1, 5, 20, 23], dtype=np.int64)
    heads = np.array([7, 0, 3, 5, 2], dtype=np.int32)
    samp, err = oracle.attention_sampled(step.q, kc, vc, step.query_start_loc, step.seq_lens,
                                         step.block_table, step.num_reqs, step.scale, rows, heads)
    assert err == 0
    for s in range(len(rows)):
        assert np.array_equal(samp[s], full[rows[s], heads[s]])


def test_workload_history_plus_write_is_a_valid_cache():
    """After the step's write, every key position < seq_len of every request
    is finite and every slot outside them is still NaN."""
    step = W.build(W.spec("tiny_mixed"))
    kc, vc = step.key_cache.copy(), step.value_cache.copy()
    assert oracle.write(step.k, step.v, kc, vc, step.slot_mapping) == 0
    live = np.zeros(kc.shape[:2], dtype=bool)
    for r in range(step.num_reqs):
        for j in range(int(step.seq_lens[r])):
            live[step.block_table[r, j // BS], j % BS] = True
    kf = W.bf16_to_f32(kc)
    assert np.isfinite(kf[live]).all()
    assert np.isnan(kf[~live]).all()
    out, err = oracle.attention(step.q, kc, vc, step.query_start_loc, step.seq_lens,
                                step.block_table, step.num_reqs, step.scale)
    assert err == 0
    assert np.isfinite(out[:300]).all() and np.isnan(out[300:]).all()
