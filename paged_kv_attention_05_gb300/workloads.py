"""Seeded synthetic inputs for the paged-KV attention step.

This module builds inputs only: request lengths, block tables, the step's new
q/k/v rows, a KV cache holding each request's history, and the slot of every
new token.  It computes no attention and writes no cache through the method's
scatter; both the CUDA library's tests and the float64 oracle read the same
arrays from here, and neither side imports the other.

The workloads follow the five step shapes this library is measured on (block
size 16, head size 128, bf16 values, scale 1/sqrt(128)):

  tiny_mixed       3 requests as in "Tour: One forward pass" (stop 1: 540,
                   129 and 0 tokens cached; 1, 1 and 298 scheduled), 300
                   tokens padded to 304 with four pad slots at -1 (stop 4),
                   Hq 32 / Hkv 8, pool of 128 blocks in seeded random order.
  mha_decode       256 decodes, cached lengths uniform in [512, 4096],
                   Hq = Hkv = 32.  The pool is 40,000 blocks: a 20,000-block
                   pool cannot hold ~37,000 distinct blocks drawn without
                   replacement.
  gqa_decode       128 decodes at 8192 cached tokens, Hq 32 / Hkv 8,
                   pool 70,000 blocks.
  mixed_chunked    64 decodes (cached uniform in [256, 2048]) then two
                   224-token prefill chunks continuing prompts with 1024 and
                   0 cached tokens (512 tokens), Hq 32 / Hkv 8, pool 8192.
  large_prefill    8 prompts of 2048 tokens, nothing cached, Hq 64 / Hkv 8,
                   values N(0, 0.5^2), pool 4096.
  mqa_long_decode  32 decodes at 32,768 cached tokens, Hq 32 / Hkv 1,
                   pool 70,000.

Recipe.  Lengths and block assignments come from
``numpy.random.Generator(PCG64(seed))`` with seed 1000, 1010, 1020, 1030,
1040, 1050 in the order above; tensor values from ``PCG64(seed + 1)``.  Values are float32 normal draws rounded to bf16 by
round-to-nearest-even.  Large tensors are filled with windows of one
16 Mi-value pool of such draws, each window starting at a seeded random
offset (the values stay N(0, sigma^2) and reproducible, and a 10 GB cache is
built at memcpy speed instead of RNG speed).  Each request's physical blocks
are the next entries of one seeded permutation of the pool, so no block is
shared.  The cache holds random history at positions < num_computed of each
request; every other slot (the tail of the last block, blocks past it, blocks
no request owns) holds the bf16 NaN pattern 0x7FC0, so any read outside a
request's keys shows up.  Block-table entries past a request's last block
are -1.  q/k/v are row views of one fused [T, (Hq + 2 Hkv) * 128] qkv array,
as the model's projection produces them ("Tour: One forward pass", stop 9).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

HEAD_SIZE = 128
BLOCK_SIZE = 16
BF16_NAN = 0x7FC0
_POOL = 1 << 24


@dataclasses.dataclass
class StepSpec:
    name: str
    ctx: list            # cached tokens per request (num_computed_tokens)
    q_len: list          # scheduled tokens per request
    hq: int
    hkv: int
    num_blocks: int      # physical blocks in the pool
    seed: int            # metadata seed; tensor values use seed + 1
    pad_tokens: int = 0  # padding rows after the last request (slot -1)
    std: float = 1.0
    head_size: int = HEAD_SIZE
    block_size: int = BLOCK_SIZE
    bt_width: int | None = None  # block-table row width; default: max needed

    @property
    def num_reqs(self) -> int:
        return len(self.ctx)

    @property
    def seq_lens(self):
        return [c + n for c, n in zip(self.ctx, self.q_len)]

    @property
    def num_tokens(self) -> int:
        return int(sum(self.q_len))

    @property
    def num_rows(self) -> int:
        return self.num_tokens + self.pad_tokens

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_size)

    def blocks_of(self, r: int) -> int:
        return -(-self.seq_lens[r] // self.block_size)

    def kv_bytes(self) -> int:
        """KV bytes a step reads once per KV head: every visible key and
        value row of every request, bf16."""
        return sum(self.seq_lens) * self.hkv * self.head_size * 2 * 2


CONFIG_NAMES = ["tiny_mixed", "mha_decode", "gqa_decode", "mixed_chunked",
                "large_prefill", "mqa_long_decode"]


def spec(name: str) -> StepSpec:
    """The named workload (lengths drawn from its metadata seed)."""
    if name == "tiny_mixed":
        return StepSpec(name, [540, 129, 0], [1, 1, 298], 32, 8, 128, 1000, pad_tokens=4)
    if name == "mha_decode":
        rng = np.random.Generator(np.random.PCG64(1010))
        ctx = rng.integers(512, 4096, size=256, endpoint=True).tolist()
        return StepSpec(name, ctx, [1] * 256, 32, 32, 40000, 1010)
    if name == "gqa_decode":
        return StepSpec(name, [8192] * 128, [1] * 128, 32, 8, 70000, 1020)
    if name == "mixed_chunked":
        rng = np.random.Generator(np.random.PCG64(1030))
        ctx = rng.integers(256, 2048, size=64, endpoint=True).tolist()
        return StepSpec(name, ctx + [1024, 0], [1] * 64 + [224, 224], 32, 8, 8192, 1030)
    if name == "large_prefill":
        return StepSpec(name, [0] * 8, [2048] * 8, 64, 8, 4096, 1040, std=0.5)
    if name == "mqa_long_decode":
        return StepSpec(name, [32768] * 32, [1] * 32, 32, 1, 70000, 1050)
    raise KeyError(name)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
            >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


class _Values:
    """Seeded bf16 N(0, std^2) values: direct draws for small requests,
    windows of a fixed pool of draws for large ones."""

    def __init__(self, seed: int, std: float):
        self.rng = np.random.Generator(np.random.PCG64(seed))
        self.std = std
        self._pool = None

    def draw(self, n: int) -> np.ndarray:
        return bf16_bits(self.rng.standard_normal(n, dtype=np.float32) * np.float32(self.std))

    def pool(self) -> np.ndarray:
        if self._pool is None:
            self._pool = self.draw(_POOL)
        return self._pool

    def fill(self, out2d: np.ndarray) -> None:
        """Fills a [rows, width] uint16 array (width <= 64 Ki)."""
        rows, width = out2d.shape
        if rows * width <= (1 << 20):
            out2d[...] = self.draw(rows * width).reshape(rows, width)
            return
        pool = self.pool()
        starts = self.rng.integers(0, _POOL - width, size=rows)
        for i in range(rows):
            s = int(starts[i])
            out2d[i] = pool[s:s + width]


@dataclasses.dataclass
class Step:
    spec: StepSpec
    qkv: np.ndarray           # uint16 [rows, (hq + 2 hkv) * d]
    q: np.ndarray             # uint16 view [rows, hq, d]
    k: np.ndarray             # uint16 view [rows, hkv, d]
    v: np.ndarray             # uint16 view [rows, hkv, d]
    key_cache: np.ndarray     # uint16 [num_blocks, bs, hkv, d], history only
    value_cache: np.ndarray
    slot_mapping: np.ndarray  # int64 [rows]
    query_start_loc: np.ndarray  # int32 [num_reqs + 1]
    seq_lens: np.ndarray      # int32 [num_reqs]
    block_table: np.ndarray   # int32 [num_reqs, bt_width]

    @property
    def num_reqs(self) -> int:
        return self.spec.num_reqs

    @property
    def scale(self) -> float:
        return self.spec.scale


def build(s: StepSpec, with_cache: bool = True) -> Step:
    """Materialises a workload.  ``with_cache=False`` leaves the caches as
    zero-size arrays (metadata and q/k/v only)."""
    R, bs, d = s.num_reqs, s.block_size, s.head_size
    meta = np.random.Generator(np.random.PCG64(s.seed))
    need = [s.blocks_of(r) for r in range(R)]
    width = s.bt_width or max(need + [1])
    assert width >= max(need + [0])
    assert sum(need) <= s.num_blocks, "pool too small for distinct blocks"
    perm = meta.permutation(s.num_blocks).astype(np.int32)
    block_table = np.full((R, width), -1, dtype=np.int32)
    used = 0
    for r in range(R):
        block_table[r, :need[r]] = perm[used:used + need[r]]
        used += need[r]

    qsl = np.zeros(R + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(s.q_len)
    seq_lens = np.asarray(s.seq_lens, dtype=np.int32)

    # the slot of each new token: its request's block for that position,
    # offset inside the block; pad rows at -1
    rows = s.num_rows
    slot_mapping = np.full(rows, -1, dtype=np.int64)
    for r in range(R):
        pos = np.arange(s.ctx[r], s.ctx[r] + s.q_len[r], dtype=np.int64)
        slot_mapping[qsl[r]:qsl[r + 1]] = block_table[r, pos // bs].astype(np.int64) * bs + pos % bs

    vals = _Values(s.seed + 1, s.std)
    qkv = np.empty((rows, (s.hq + 2 * s.hkv) * d), dtype=np.uint16)
    if rows:
        vals.fill(qkv)
    q = qkv[:, :s.hq * d].reshape(rows, s.hq, d)
    k = qkv[:, s.hq * d:(s.hq + s.hkv) * d].reshape(rows, s.hkv, d)
    v = qkv[:, (s.hq + s.hkv) * d:].reshape(rows, s.hkv, d)

    if with_cache:
        shape = (s.num_blocks, bs, s.hkv, d)
        caches = []
        for _ in range(2):
            c = np.empty(shape, dtype=np.uint16)
            vals.fill(c.reshape(s.num_blocks, bs * s.hkv * d))
            caches.append(c)
        history = np.zeros((s.num_blocks, bs), dtype=bool)
        for r in range(R):
            full, part = divmod(s.ctx[r], bs)
            history[block_table[r, :full]] = True
            if part:
                history[block_table[r, full], :part] = True
        flat_mask = ~history.reshape(-1)
        for c in caches:
            c.reshape(s.num_blocks * bs, s.hkv * d)[flat_mask] = BF16_NAN
        key_cache, value_cache = caches
    else:
        key_cache = np.empty((0, bs, s.hkv, d), dtype=np.uint16)
        value_cache = np.empty((0, bs, s.hkv, d), dtype=np.uint16)

    return Step(s, qkv, q, k, v, key_cache, value_cache, slot_mapping, qsl, seq_lens,
                block_table)


def custom(ctx, q_len, hq, hkv, num_blocks=None, seed=7, pad_tokens=0, std=1.0,
           bt_width=None) -> StepSpec:
    """A small workload with explicit lengths, for parity and edge-case tests."""
    need = sum(-(-(c + n) // BLOCK_SIZE) for c, n in zip(ctx, q_len))
    nb = num_blocks if num_blocks is not None else max(need + need // 2 + 3, 4)
    return StepSpec("custom", list(ctx), list(q_len), hq, hkv, nb, seed,
                    pad_tokens=pad_tokens, std=std, bt_width=bt_width)


def subset(s: StepSpec, n_reqs: int) -> StepSpec:
    """The first n_reqs requests of a workload, with a pool 10% larger than
    they need (same seeds, same shapes per request)."""
    ctx, q_len = s.ctx[:n_reqs], s.q_len[:n_reqs]
    need = sum(-(-(c + n) // s.block_size) for c, n in zip(ctx, q_len))
    return StepSpec(s.name, ctx, q_len, s.hq, s.hkv, need + need // 10 + 1, s.seed,
                    pad_tokens=s.pad_tokens if n_reqs >= s.num_reqs else 0, std=s.std,
                    head_size=s.head_size, block_size=s.block_size, bt_width=s.bt_width)
