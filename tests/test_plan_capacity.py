"""The workspace bound against what the step plan writes (CPU only).

The plan kernel lists decode units (request, KV head, key range), split pairs,
split-KV partial rows and prefill tiles into the device workspace; the host
sizes that workspace before the plan runs, without reading the device
metadata.  If the bound were ever too small the plan reports
PKV_DEV_ERR_CAPACITY and runs nothing, so this test checks the bound itself:
for seeded random batches a plain Python loop counts the entries of the plan
the kernel would make, for every split-chunk choice the kernel can take, and
each count must fit the capacities pkv_workspace_size reports for the
batch's sizes.

"Tour: One forward pass", stop 5: the attention metadata (query_start_loc,
seq_lens, block table) the plan reads; "vLLM MHA Code Path: From QKV to Paged
KV Cache", "Prefill and decode share an interface": a request's phase is told
from its query and sequence lengths only.
"""
import numpy as np
import pytest

import paged_kv_attention_05_gb300 as pkv

SMS = 152


def rows_cap(group):
    """Query rows one decode unit carries (query tokens x heads of a group)."""
    return 16 if group <= 16 else 32


def plan_counts(ctx, q_len, hq, hkv, workers, caps):
    """Entries of the plan for one batch: the split chunk chosen as the plan
    kernel chooses it (about four units per decode worker, whole 64-key
    tiles, between max(256, 32 G) and 2048 keys; shorter where every pair's
    splits fit one wave of workers and the workspace holds them; longer, by
    less than twice, where that makes one wave instead of more; in the first
    case a chunk of 256 keys or more is cut at whole 16-key pages), then the
    units, split pairs, partial rows and prefill tiles of that chunk."""
    G = hq // hkv
    decs, pres = [], []
    for c, n in zip(ctx, q_len):
        if n == 0:
            continue
        (decs if n * G <= rows_cap(G) else pres).append((c + n, n))
    chunk = 2048
    if decs:
        total = sum(L for L, _ in decs)
        pairs = len(decs) * hkv
        lmax = max(L for L, _ in decs)
        rmax = max(n * G for _, n in decs)
        want = -(-total * hkv // (workers * 4))
        want = -(-want // 64) * 64
        lo = max(256, 32 * G)
        chunk = min(max(want, lo), 2048)
        if pairs * -(-lmax // chunk) <= workers:
            per_pair = workers // pairs
            c1 = -(-lmax // per_pair)
            c = -(-c1 // 64) * 64
            if c >= 256:
                c = max(-(-c1 // 16) * 16, 256)
            else:
                per = min(per_pair, caps["decode_units"] // pairs,
                          caps["partial_rows"] // (pairs * max(rmax, 1)))
                c2 = -(-lmax // per) if per >= 1 else 256
                c2 = -(-c2 // 64) * 64
                c = max(c2, c) if c2 < 256 else 256
            chunk = min(chunk, c)
        elif pairs <= workers:
            # one wave of somewhat longer units instead of two waves
            per_pair = workers // pairs
            c = -(-lmax // per_pair)
            c = -(-c // 64) * 64
            if c <= 2048 and c < 2 * chunk:
                chunk = c
    units = parts = split_pairs = 0
    for L, n in decs:
        ns = -(-L // chunk)
        units += ns * hkv
        if ns > 1:
            parts += ns * hkv * n * G
            split_pairs += hkv
    tiles = sum(-(-n // 128) for _, n in pres)
    return {"chunk": chunk, "decode_units": units, "partial_rows": parts,
            "split_pairs": split_pairs, "prefill_tiles": tiles}


def random_batch(rng, kind):
    hq, hkv = [(32, 32), (32, 8), (32, 1), (64, 8), (16, 4), (40, 5), (32, 2)][
        rng.integers(0, 7)]
    G = hq // hkv
    R = int(rng.integers(1, 64 if kind == "small" else 400))
    ctx, q_len = [], []
    for _ in range(R):
        u = rng.random()
        if u < 0.6:                                   # single-token decode
            q = 1
        elif u < 0.75:                                # multi-token decode
            q = int(rng.integers(1, max(2, rows_cap(G) // G + 1)))
        else:                                         # prefill chunk
            q = int(rng.integers(2, 3000))
        c = int(rng.integers(0, 70000 if kind != "small" else 3000))
        ctx.append(c)
        q_len.append(q)
    return ctx, q_len, hq, hkv


@pytest.mark.parametrize("kind", ["small", "large"])
def test_workspace_holds_every_plan(kind):
    rng = np.random.Generator(np.random.PCG64(4242 if kind == "small" else 4343))
    for _ in range(150):
        ctx, q_len, hq, hkv = random_batch(rng, kind)
        q_rows = sum(q_len) + int(rng.integers(0, 8))     # padded rows past the last request
        need = max(-(-(c + n) // 16) for c, n in zip(ctx, q_len))
        width = need + int(rng.integers(0, 40))
        caps = pkv.pkv_workspace_size(len(ctx), q_rows, width, hq, hkv, SMS)
        for workers in (caps["decode_workers"], caps["decode_workers_int8"]):
            got = plan_counts(ctx, q_len, hq, hkv, workers, caps)
            for key in ("decode_units", "partial_rows", "split_pairs", "prefill_tiles"):
                assert got[key] <= caps[key], (key, got, caps, ctx, q_len, hq, hkv)


def test_one_wave_small_batches_split_below_256_keys_within_capacity():
    """The small-batch branch: every pair's splits fit one wave, so the plan
    may cut chunks shorter than 256 keys; the workspace's one-wave room must
    hold what that makes (three requests of the trace step; a single long
    decode; 8 MQA decodes)."""
    cases = [([540, 129, 0], [1, 1, 298], 32, 8), ([20000], [1], 32, 8),
             ([32768] * 8, [1] * 8, 32, 1), ([100, 200, 300], [4, 4, 4], 16, 4)]
    short = 0
    for ctx, q_len, hq, hkv in cases:
        width = max(-(-(c + n) // 16) for c, n in zip(ctx, q_len))
        caps = pkv.pkv_workspace_size(len(ctx), sum(q_len), width, hq, hkv, SMS)
        got = plan_counts(ctx, q_len, hq, hkv, caps["decode_workers"], caps)
        short += got["chunk"] < 256
        for key in ("decode_units", "partial_rows", "split_pairs", "prefill_tiles"):
            assert got[key] <= caps[key], (key, got, caps)
    assert short >= 3   # the branch is exercised (the MQA case keeps 256-key chunks)


def test_capacities_grow_with_the_bound_and_match_the_byte_count():
    a = pkv.pkv_workspace_size(16, 4096, 128, 32, 8, SMS)
    b = pkv.pkv_workspace_size(32, 8192, 256, 32, 8, SMS)
    for key in ("decode_units", "partial_rows", "split_pairs", "prefill_tiles", "bytes"):
        assert b[key] >= a[key]
    # units of 32 bytes, prefill entries and pairs of 32, partial rows of
    # 130 fp32: the byte count covers every list
    lists = 32 * (b["decode_units"] + b["prefill_tiles"] + b["split_pairs"])
    assert b["bytes"] >= lists + 520 * b["partial_rows"]
    assert b["decode_workers"] == 8 * SMS


def test_workspace_size_rejects_bad_sizes():
    with pytest.raises(pkv.PkvError):
        pkv.pkv_workspace_size(4, 16, 4, 30, 8, SMS)   # heads not a multiple
    with pytest.raises(pkv.PkvError):
        pkv.pkv_workspace_size(4, 16, 4, 32, 8, 0)     # no SMs
