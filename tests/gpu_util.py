"""Helpers shared by the GPU parity tests: move a seeded workload to the
device, run the library's two calls, and compare with the float64 oracle."""
import numpy as np
import torch

import paged_kv_attention_05_gb300 as pkv
from paged_kv_attention_05_gb300 import workloads as W

ATOL = 1e-2   # |gpu - ref| <= ATOL + RTOL * |ref|, elementwise (bf16 in, fp32 accumulate)
RTOL = 1e-2


def to_dev(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit array -> CUDA bfloat16 tensor (same bytes)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceStep:
    """A workload resident on the GPU; q/k/v are row views of one fused qkv."""

    def __init__(self, step: W.Step, nan_out=True):
        s = step.spec
        d = s.head_size
        self.step = step
        self.qkv = to_dev(step.qkv)
        rows = step.qkv.shape[0]
        self.q = self.qkv[:, :s.hq * d].view(rows, s.hq, d)
        self.k = self.qkv[:, s.hq * d:(s.hq + s.hkv) * d].view(rows, s.hkv, d)
        self.v = self.qkv[:, (s.hq + s.hkv) * d:].view(rows, s.hkv, d)
        self.key_cache = to_dev(step.key_cache)
        self.value_cache = to_dev(step.value_cache)
        self.slot_mapping = torch.from_numpy(step.slot_mapping).cuda()
        self.qsl = torch.from_numpy(step.query_start_loc).cuda()
        self.seq_lens = torch.from_numpy(step.seq_lens).cuda()
        self.block_table = torch.from_numpy(step.block_table).cuda()
        self.out = torch.empty((rows, s.hq, d), dtype=torch.bfloat16, device="cuda")
        if nan_out:
            self.out.view(torch.int16).fill_(W.BF16_NAN)

    def write(self):
        pkv.pkv_write(self.k, self.v, self.key_cache, self.value_cache, self.slot_mapping)

    def attention(self):
        pkv.pkv_attention(self.q, self.key_cache, self.value_cache, self.qsl, self.seq_lens,
                          self.block_table, self.step.num_reqs, self.step.scale, self.out)

    def out_f64(self) -> np.ndarray:
        return W.bf16_to_f32(to_host_bits(self.out)).astype(np.float64)


def assert_close(gpu: np.ndarray, ref: np.ndarray, what=""):
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d of %d elements outside %g + %g|ref| (max err %g); first %s"
                             % (what, int(bad.sum()), bad.size, ATOL, RTOL, float(np.nanmax(err)),
                                [(tuple(i), float(gpu[tuple(i)]), float(ref[tuple(i)]))
                                 for i in idx]))
