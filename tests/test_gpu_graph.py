"""A whole multi-layer step captured in one CUDA graph: with the workspace
reserved beforehand, pkv_write + pkv_attention enqueue no allocation and no
host synchronisation, so the layers of a step ("Tour: One forward pass",
stop 7: the 32-layer loop; stop 5: one attention metadata object shared by
all layers) can be captured and replayed.  Replays must reproduce the eager
results exactly (same kernels, same inputs)."""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_05_gb300 as pkv
from paged_kv_attention_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu

from gpu_util import DeviceStep, assert_close  # noqa: E402


def test_capture_layers_in_a_cuda_graph_and_replay():
    layers = 4
    spec = W.custom([0, 700, 33, 1500, 0], [40, 1, 130, 1, 1], 16, 4, seed=515, pad_tokens=2)
    steps = [W.build(W.StepSpec(spec.name, spec.ctx, spec.q_len, spec.hq, spec.hkv,
                                spec.num_blocks, spec.seed + 100 * l, pad_tokens=spec.pad_tokens))
             for l in range(layers)]
    devs = [DeviceStep(s) for s in steps]
    # eager reference, layer by layer (each layer its own cache and q/k/v)
    eager = []
    for ds in devs:
        ds.write()
        ds.attention()
        eager.append(ds.out.clone())
    assert pkv.pkv_get_error() == 0
    s0 = steps[0]
    pkv.pkv_reserve_workspace(s0.num_reqs, s0.q.shape[0], s0.block_table.shape[1], spec.hq, spec.hkv)
    for ds in devs:   # fresh outputs and the pre-write caches again
        ds.out.view(torch.int16).fill_(W.BF16_NAN)
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for ds in devs:
                pkv.pkv_write(ds.k, ds.v, ds.key_cache, ds.value_cache, ds.slot_mapping,
                              stream=stream)
                pkv.pkv_attention(ds.q, ds.key_cache, ds.value_cache, ds.qsl, ds.seq_lens,
                                  ds.block_table, ds.step.num_reqs, ds.step.scale, ds.out,
                                  stream=stream)
    torch.cuda.current_stream().wait_stream(stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert pkv.pkv_get_error() == 0
    n = int(s0.query_start_loc[-1])
    for l, ds in enumerate(devs):
        assert torch.equal(ds.out.view(torch.int16), eager[l].view(torch.int16)), "layer %d" % l
        kc, vc = steps[l].key_cache.copy(), steps[l].value_cache.copy()
        oracle.write(steps[l].k, steps[l].v, kc, vc, steps[l].slot_mapping)
        ref, _ = oracle.attention(steps[l].q, kc, vc, steps[l].query_start_loc,
                                  steps[l].seq_lens, steps[l].block_table, steps[l].num_reqs,
                                  steps[l].scale)
        assert_close(ds.out_f64()[:n], ref[:n], "graph layer %d" % l)


_REFUSAL_SCRIPT = r"""
import sys
sys.path[:0] = [sys.argv[1], sys.argv[2]]
import torch
import paged_kv_attention_05_gb300 as pkv
from paged_kv_attention_05_gb300 import workloads as W
from gpu_util import DeviceStep
spec = W.custom([5000], [1], 32, 1, seed=616)   # MQA, long: a big partial buffer
ds = DeviceStep(W.build(spec))
ds.write()
ds.attention()   # eager first: the device state and a small workspace exist
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
stream = torch.cuda.Stream()
big = 4096   # far more requests than this process reserved for
qsl = torch.zeros(big + 1, dtype=torch.int32, device="cuda")
sl = torch.zeros(big, dtype=torch.int32, device="cuda")
# the widest block table: 4096 x 2048 split units alone need 256 MiB
bt = torch.zeros((big, 32768), dtype=torch.int32, device="cuda")
torch.cuda.synchronize()
try:
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            pkv.pkv_attention(ds.q, ds.key_cache, ds.value_cache, qsl, sl, bt, big,
                              ds.step.scale, ds.out, stream=stream)
except pkv.PkvError as e:
    torch.cuda.synchronize()
    print("refused:", e)
    sys.exit(0)
print("not refused")
sys.exit(1)
"""


def test_capture_without_reserved_workspace_is_refused_cleanly():
    """A capture that would need a larger workspace fails on the host with an
    error (no allocation inside capture), not with a broken graph.  Run in a
    fresh process: the workspace only grows, so an earlier test's reservation
    in this process could already cover the request."""
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    r = subprocess.run([sys.executable, "-c", _REFUSAL_SCRIPT, root, here],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "refused:" in r.stdout
