"""One step plan serving several layers (pkv_plan + pkv_attention_planned):
bit-identical to per-layer pkv_attention, a snapshot of the metadata (later
changes of query_start_loc / seq_lens do not reach the kernels), refused
without a plan or with another head geometry, and capturable in a CUDA graph
together with the layers."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_05_gb300 as pkv
from paged_kv_attention_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu

from gpu_util import DeviceStep, assert_close  # noqa: E402


def _layers(n, seed=700):
    spec = W.custom([0, 700, 33, 1500, 0, 2300], [40, 1, 130, 1, 3, 1], 16, 4, seed=seed,
                    pad_tokens=2)
    steps = [W.build(W.StepSpec(spec.name, spec.ctx, spec.q_len, spec.hq, spec.hkv,
                                spec.num_blocks, spec.seed + 100 * l, pad_tokens=spec.pad_tokens))
             for l in range(n)]
    return steps, [DeviceStep(s) for s in steps]


def _eager(devs):
    outs = []
    for ds in devs:
        ds.write()
        ds.attention()
        outs.append(ds.out.clone())
    assert pkv.pkv_get_error() == 0
    return outs


def _planned(ds, stream=None):
    pkv.pkv_attention_planned(ds.q, ds.key_cache, ds.value_cache, ds.block_table,
                              ds.step.scale, ds.out, stream=stream)


def test_one_plan_serves_every_layer():
    steps, devs = _layers(4)
    eager = _eager(devs)
    s0, d0 = steps[0], devs[0]
    for ds in devs:
        ds.out.view(torch.int16).fill_(W.BF16_NAN)
    pkv.pkv_plan(d0.q.shape[0], s0.spec.hq, s0.spec.hkv, d0.qsl, d0.seq_lens,
                 d0.block_table.shape[1], s0.num_reqs)
    for ds in devs:
        _planned(ds)
    assert pkv.pkv_get_error() == 0
    n = int(s0.query_start_loc[-1])
    for l, ds in enumerate(devs):
        assert torch.equal(ds.out.view(torch.int16), eager[l].view(torch.int16)), "layer %d" % l
        assert torch.isnan(ds.out[n:].float()).all()
    # and against the float64 oracle for one layer
    kc, vc = steps[2].key_cache.copy(), steps[2].value_cache.copy()
    oracle.write(steps[2].k, steps[2].v, kc, vc, steps[2].slot_mapping)
    ref, _ = oracle.attention(steps[2].q, kc, vc, steps[2].query_start_loc, steps[2].seq_lens,
                              steps[2].block_table, steps[2].num_reqs, steps[2].scale)
    assert_close(devs[2].out_f64()[:n], ref[:n], "planned layer 2")


def test_plan_is_a_snapshot_of_the_metadata():
    steps, devs = _layers(1, seed=720)
    eager = _eager(devs)
    ds, s0 = devs[0], steps[0]
    pkv.pkv_plan(ds.q.shape[0], s0.spec.hq, s0.spec.hkv, ds.qsl, ds.seq_lens,
                 ds.block_table.shape[1], s0.num_reqs)
    # the metadata arrays change after planning (here: to values that would
    # point far outside every buffer); the planned call must not see them
    ds.qsl.fill_(1 << 30)
    ds.seq_lens.fill_(1 << 30)
    ds.out.view(torch.int16).fill_(W.BF16_NAN)
    _planned(ds)
    assert pkv.pkv_get_error() == 0
    assert torch.equal(ds.out.view(torch.int16), eager[0].view(torch.int16))


def test_planned_call_is_refused_without_a_plan_or_with_other_heads():
    steps, devs = _layers(1, seed=740)
    ds, s0 = devs[0], steps[0]
    pkv.pkv_plan(ds.q.shape[0], s0.spec.hq, s0.spec.hkv, ds.qsl, ds.seq_lens,
                 ds.block_table.shape[1], s0.num_reqs)
    q8 = torch.zeros((ds.q.shape[0], 8, 128), dtype=torch.bfloat16, device="cuda")
    out8 = torch.zeros_like(q8)
    with pytest.raises(pkv.PkvError):   # 8 query heads against a plan for 16
        pkv.pkv_attention_planned(q8, ds.key_cache, ds.value_cache, ds.block_table, 0.1, out8)
    # a workspace reallocation drops the plan
    pkv.pkv_reserve_workspace(50000, 200000, ds.block_table.shape[1] * 4, s0.spec.hq,
                              s0.spec.hkv)
    with pytest.raises(pkv.PkvError):
        _planned(ds)


def test_plan_and_layers_in_one_cuda_graph():
    steps, devs = _layers(3, seed=760)
    eager = _eager(devs)
    s0, d0 = steps[0], devs[0]
    pkv.pkv_reserve_workspace(s0.num_reqs, d0.q.shape[0], d0.block_table.shape[1], s0.spec.hq,
                              s0.spec.hkv)
    for ds in devs:
        ds.out.view(torch.int16).fill_(W.BF16_NAN)
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            pkv.pkv_plan(d0.q.shape[0], s0.spec.hq, s0.spec.hkv, d0.qsl, d0.seq_lens,
                         d0.block_table.shape[1], s0.num_reqs, stream=stream)
            for ds in devs:
                pkv.pkv_write(ds.k, ds.v, ds.key_cache, ds.value_cache, ds.slot_mapping,
                              stream=stream)
                _planned(ds, stream=stream)
    torch.cuda.current_stream().wait_stream(stream)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert pkv.pkv_get_error() == 0
    for l, ds in enumerate(devs):
        assert torch.equal(ds.out.view(torch.int16), eager[l].view(torch.int16)), "layer %d" % l
