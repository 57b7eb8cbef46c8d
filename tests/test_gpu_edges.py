"""Degenerate steps on the GPU: requests with no query tokens this step, a
step with no requests and no tokens at all, and a first token that sees only
itself (whose output is its own V row, bit for bit)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_05_gb300 as pkv
from paged_kv_attention_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu

from gpu_util import DeviceStep, assert_close, to_host_bits  # noqa: E402


def test_requests_with_no_query_tokens():
    """Zero-token requests (query_start_loc repeats) between, before and after
    decodes and a prefill chunk, one of them with a long cached context: they
    produce no row and change nothing, the others match the oracle."""
    ctx = [300, 40, 5000, 0, 2000, 7, 64]
    q_len = [0, 1, 0, 150, 3, 0, 1]
    step = W.build(W.custom(ctx, q_len, 8, 2, seed=808, pad_tokens=2))
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
    assert n == sum(q_len)
    assert_close(got[:n], ref[:n], "zero-token requests")
    assert np.isnan(got[n:]).all()


def test_empty_step():
    """No tokens and no requests: every call returns without error and
    writes nothing."""
    hq, hkv, d = 8, 2, 128
    kc = torch.zeros((4, 16, hkv, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.empty((0, hkv, d), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((0, hq, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((0, hq, d), dtype=torch.bfloat16, device="cuda")
    slots = torch.empty((0,), dtype=torch.int64, device="cuda")
    qsl = torch.zeros((1,), dtype=torch.int32, device="cuda")
    seq_lens = torch.empty((0,), dtype=torch.int32, device="cuda")
    bt = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    pkv.pkv_write(k, k, kc, vc, slots)
    pkv.pkv_attention(q, kc, vc, qsl, seq_lens, bt, 0, d ** -0.5, out)
    k8 = torch.zeros((4, 16, hkv, d), dtype=torch.int8, device="cuda")
    v8 = torch.zeros_like(k8)
    pkv.pkv_write_int8(k, k, k8, v8, slots, 0.03, 0.03)
    pkv.pkv_attention_int8(q, k8, v8, 0.03, 0.03, qsl, seq_lens, bt, 0, d ** -0.5, out)
    pkv.pkv_attention_noalloc(q, kc, vc, qsl, seq_lens, bt, 0, d ** -0.5, out)
    pkv.pkv_plan(0, hq, hkv, qsl, seq_lens, 4, 0)
    pkv.pkv_attention_planned(q, kc, vc, bt, d ** -0.5, out)
    torch.cuda.synchronize()
    assert pkv.pkv_get_error() == 0
    assert not kc.any() and not vc.any() and not k8.any() and not v8.any()


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (32, 1)])
def test_first_token_sees_only_itself(hq, hkv):
    """Prompts of one token with nothing cached: one visible key, softmax
    weight exactly 1, so every head's output is its KV head's new V row,
    bit for bit, whatever the scores."""
    step = W.build(W.custom([0] * 5, [1] * 5, hq, hkv, seed=hq + hkv, std=3.0))
    ds = DeviceStep(step)
    ds.write()
    ds.attention()
    assert pkv.pkv_get_error() == 0
    got = to_host_bits(ds.out)[:5].reshape(5, hq, 128)
    v = step.v.reshape(-1, hkv, 128)[:5]
    G = hq // hkv
    for h in range(hq):
        assert np.array_equal(got[:, h], v[:, h // G]), "head %d" % h


def test_steps_back_to_back_without_a_sync():
    """Four different steps enqueued one after another on one stream with no
    host synchronisation between them: each step's plan rewrites the work
    lists at the same workspace addresses, and the prefill grid reads them
    beside the running decode grid (without waiting for it).  Every step's
    rows must match its own oracle: nothing read is left over from the step
    before."""
    specs = [W.custom([700, 0, 33], [1, 200, 1], 16, 4, seed=1201, pad_tokens=1),
             W.custom([0, 1500, 9, 0], [300, 1, 1, 17], 16, 4, seed=1202),
             W.custom([4000] * 6, [1] * 6, 16, 4, seed=1203),
             W.custom([100, 0, 2048, 5], [129, 64, 1, 1], 16, 4, seed=1204, pad_tokens=3)]
    steps, refs, dss = [], [], []
    for sp in specs:
        step = W.build(sp)
        kc, vc = step.key_cache.copy(), step.value_cache.copy()
        assert oracle.write(step.k, step.v, kc, vc, step.slot_mapping) == 0
        ref, err = oracle.attention(step.q, kc, vc, step.query_start_loc, step.seq_lens,
                                    step.block_table, step.num_reqs, step.scale)
        assert err == 0
        steps.append(step)
        refs.append(ref)
        dss.append(DeviceStep(step))
    # room for the largest of the four, so that no call grows the workspace
    # (growing it synchronises the device)
    pkv.pkv_reserve_workspace(max(st.num_reqs for st in steps),
                              max(st.qkv.shape[0] for st in steps),
                              max(st.block_table.shape[1] for st in steps), 16, 4)
    torch.cuda.synchronize()
    for ds in dss:               # enqueued back to back, one stream, no sync
        ds.write()
        ds.attention()
    assert pkv.pkv_get_error() == 0
    for i, (step, ref, ds) in enumerate(zip(steps, refs, dss)):
        got = ds.out_f64()
        n = int(step.query_start_loc[-1])
        assert_close(got[:n], ref[:n], "step %d of four" % i)
        assert np.isnan(got[n:]).all()


@pytest.mark.parametrize("name", ["tiny_mixed", "mixed_chunked"])
def test_many_mixed_steps_back_to_back(name):
    """Twenty thousand steps of a small mixed batch enqueued back to back,
    the error word read once at the end.  In these steps a prefill CTA often
    takes two items in a row, the second with a single key tile, while the
    decode grid keeps HBM busy and the epilogue warps' stores are slow: the
    softmax warps may then finish the second item before the epilogue warps
    have waited for the first one's row sums, and each item's signal must
    still be told apart (a wait that missed it would give up after its time
    limit and set PKV_DEV_ERR_TIMEOUT).  The last step's rows match the
    oracle."""
    step = W.build(W.spec(name))
    kc, vc = step.key_cache.copy(), step.value_cache.copy()
    assert oracle.write(step.k, step.v, kc, vc, step.slot_mapping) == 0
    ref, err = oracle.attention(step.q, kc, vc, step.query_start_loc, step.seq_lens,
                                step.block_table, step.num_reqs, step.scale)
    assert err == 0
    ds = DeviceStep(step)
    ds.write()
    ds.attention()
    torch.cuda.synchronize()
    assert pkv.pkv_get_error() == 0
    for _ in range(20000):
        ds.write()
        ds.attention()
    torch.cuda.synchronize()
    assert pkv.pkv_get_error() == 0
    n = int(step.query_start_loc[-1])
    got = ds.out_f64()
    assert_close(got[:n], ref[:n], name + " after 20000 steps")
