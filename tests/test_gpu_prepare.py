"""pkv_prepare_step (positions, seq_lens, gathered block table, slot mapping)
against the oracle's block arithmetic: the forward-pass trace's printed
values and random batches, bit for bit."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_05_gb300 as pkv
from oracle import blocks

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "forward_pass_trace.json")


def run(qsl, num_computed, pbt, idx, n_padded):
    R = len(num_computed)
    d = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).cuda()
    positions = torch.full((n_padded,), -77, dtype=torch.int64, device="cuda")
    seq_lens = torch.zeros(R, dtype=torch.int32, device="cuda")
    slots = torch.zeros(n_padded, dtype=torch.int64, device="cuda")
    bt = torch.zeros((R, pbt.shape[1]), dtype=torch.int32, device="cuda")
    pkv.pkv_prepare_step(d(qsl, np.int32), d(num_computed, np.int32), d(pbt, np.int32), R,
                         n_padded, positions, seq_lens, slots, bt,
                         idx_mapping=None if idx is None else d(idx, np.int32))
    assert pkv.pkv_get_error() == 0
    return positions.cpu().numpy(), seq_lens.cpu().numpy(), slots.cpu().numpy(), bt.cpu().numpy()


def expected(qsl, num_computed, pbt, idx, n_padded):
    R = len(num_computed)
    rows = np.arange(R) if idx is None else np.asarray(idx)
    bt = pbt[rows]
    pos, sl = blocks.positions_and_seq_lens(qsl, num_computed, R, n_padded, pad_value=-77)
    sm = blocks.slot_mappings(bt, qsl, pos, R, n_padded)
    return pos, sl, sm, bt


def test_trace_step_values():
    with open(GOLDEN) as f:
        g = json.load(f)
    rng = np.random.default_rng(3)
    pbt = np.full((1024, 40), -1, dtype=np.int32)       # persistent rows, slots 1021..1023 used
    ids = rng.permutation(128).astype(np.int32)
    pbt[1023, :34], pbt[1022, :9], pbt[1021, :19] = ids[:34], ids[34:43], ids[43:62]
    idx = np.array([1023, 1022, 1021], dtype=np.int32)
    qsl = np.array(g["query_start_loc"], dtype=np.int32)
    got = run(qsl, g["num_computed_tokens"], pbt, idx, g["num_tokens_padded"])
    exp = expected(qsl, g["num_computed_tokens"], pbt, idx, g["num_tokens_padded"])
    for a, b in zip(got, exp):
        assert np.array_equal(a, b)
    pos, sl, sm, bt = got
    assert pos[:4].tolist() == g["positions_first"] and pos[299] == g["positions_R3_last"]
    assert (pos[300:] == -77).all()                      # padding rows not written
    assert sl.tolist() == g["seq_lens"]
    assert sm[g["pad_rows"]].tolist() == [g["pad_slot_id"]] * 4
    assert sm[0] == bt[0, 33] * 16 + 12 and sm[1] == bt[1, 8] * 16 + 1


@pytest.mark.parametrize("seed", [0, 1])
def test_random_batches(seed):
    rng = np.random.default_rng(seed)
    R, width = 77, 130
    q_len = rng.integers(0, 40, R)
    q_len[rng.random(R) < 0.5] = 1
    num_computed = rng.integers(0, 1900, R)
    qsl = np.zeros(R + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_len)
    pbt = rng.integers(0, 100000, (300, width)).astype(np.int32)
    idx = rng.permutation(300)[:R].astype(np.int32)
    n_padded = int(qsl[-1]) + 13
    got = run(qsl, num_computed, pbt, idx, n_padded)
    exp = expected(qsl, num_computed, pbt, idx, n_padded)
    for a, b in zip(got, exp):
        assert np.array_equal(a, b)
