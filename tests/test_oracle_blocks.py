"""Pins the oracle's block/slot arithmetic to the values the pages print."""
import json
import os

import numpy as np

from oracle import blocks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_trace_block_count_and_last_block():
    g = _load("forward_pass_trace.json")
    bs = g["block_size"]
    assert blocks.blocks_needed(g["prompt_len_R3"], bs) == g["blocks_in_R3_row"]
    assert blocks.last_block_fill(g["prompt_len_R3"], bs) == g["R3_last_block_tokens"]
    first, last = g["R3_block_indexes"]
    assert blocks.position_to_block(0, bs)[0] == first
    assert blocks.position_to_block(g["positions_R3_last"], bs)[0] == last


def test_trace_position_to_block():
    g = _load("forward_pass_trace.json")
    for pos, bi, off in g["position_to_block"]:
        assert blocks.position_to_block(pos, g["block_size"]) == (bi, off)


def test_trace_query_start_loc_positions_seq_lens():
    g = _load("forward_pass_trace.json")
    qsl = blocks.query_start_loc(g["num_scheduled_tokens"], 1024, g["num_actual_tokens"])
    assert qsl[:4].tolist() == g["query_start_loc"]
    assert (qsl[4:] == g["query_start_loc_buffer_fill"]).all()
    pos, seq_lens = blocks.positions_and_seq_lens(qsl, g["num_computed_tokens"], 3,
                                                  g["num_tokens_padded"])
    assert seq_lens.tolist() == g["seq_lens"]
    assert pos[:4].tolist() == g["positions_first"]
    assert pos[299] == g["positions_R3_last"]
    q_lens = np.diff(qsl[:4])
    assert int(q_lens.max()) == g["max_query_len"]
    assert int(seq_lens.max()) == g["max_seq_len"]
    assert int(qsl[3]) == g["num_actual_tokens"]


def test_trace_slot_mapping_pads_and_values():
    g = _load("forward_pass_trace.json")
    bs = g["block_size"]
    qsl = np.array(g["query_start_loc"], dtype=np.int32)
    pos, seq_lens = blocks.positions_and_seq_lens(qsl, g["num_computed_tokens"], 3,
                                                  g["num_tokens_padded"])
    # any block ids will do: the page derives only block index and offset
    rng = np.random.default_rng(0)
    ids = rng.permutation(128).astype(np.int32)
    bt = np.full((3, 40), -1, dtype=np.int32)
    bt[0, :34], bt[1, :9], bt[2, :19] = ids[:34], ids[34:43], ids[43:62]
    sm = blocks.slot_mappings(bt, qsl, pos, 3, g["num_tokens_padded"], bs)
    assert sm.dtype == np.int64 and sm.shape == (g["num_tokens_padded"],)
    assert sm[g["pad_rows"]].tolist() == [g["pad_slot_id"]] * 4
    assert sm[0] == bt[0, 33] * bs + 12
    assert sm[1] == bt[1, 8] * bs + 1
    # R3: 298 tokens in blocks 0..18, the last one holds 10 tokens
    r3 = sm[2:300]
    assert r3[0] == bt[2, 0] * bs and r3[-1] == bt[2, 18] * bs + 9
    assert len(set((r3 // bs).tolist())) == 19
    assert int((r3 // bs == bt[2, 18]).sum()) == 10


def test_block_manager_35_token_example():
    g = _load("block_manager_examples.json")
    p = g["prompt_35"]
    bs = g["block_size"]
    assert blocks.blocks_needed(p["prompt_len"], bs) == p["blocks"] == len(p["block_table"])
    assert blocks.blocks_at_admission(p["prompt_len"], bs) == p["blocks"]
    for bi, (t0, t1) in enumerate(p["block_tokens"]):
        assert blocks.position_to_block(t0, bs) == (bi, 0)
        assert blocks.position_to_block(t1, bs) == (bi, bs - 1)
    # after the prompt: 3 slots of block 89 in use (positions 32..34); the
    # page's slot list ends at 89*16+2
    assert blocks.last_block_fill(35, bs) == 3
    bi, off = blocks.position_to_block(34, bs)
    assert blocks.slot(p["block_table"][bi], off, bs) == blocks.slot(*g["slot_of_A_last"], bs)
    # once the first decode token is written (seq_len 36) the page's "first
    # 4 slots used" holds, still in 3 blocks
    assert blocks.blocks_needed(36, bs) == 3
    assert blocks.last_block_fill(36, bs) == p["last_block_slots_as_printed"]


def test_block_count_formulas_agree_and_differ_where_expected():
    g = _load("block_manager_examples.json")
    bs = g["block_size"]
    for n, expect in g["num_required_blocks_formula_examples"]:
        assert blocks.blocks_at_admission(n, bs) == expect
    assert blocks.blocks_needed(298, bs) == blocks.blocks_at_admission(298, bs) == 19
    assert blocks.blocks_needed(35, bs) == blocks.blocks_at_admission(35, bs) == 3
    # multiples of the block size: the admission formula reserves one more
    assert blocks.blocks_needed(32, bs) == 2 and blocks.blocks_at_admission(32, bs) == 3
    for n in range(1, 200):
        extra = blocks.blocks_at_admission(n, bs) - blocks.blocks_needed(n, bs)
        assert extra == (1 if n % bs == 0 else 0)


def test_block_mem_formula():
    g = _load("block_manager_examples.json")["block_mem"]
    b = blocks.block_mem_bytes(g["num_layers"], g["num_kv_heads"], g["head_size"],
                               g["block_size"], g["elem_bytes"])
    assert b == g["bytes"] == 8388608
    assert round(b / 1e6, 1) == g["printed_approx_MB"]


def test_packed_batch_example():
    g = _load("block_manager_examples.json")["packed_batch"]
    n_sched = g["prompt_lens"] + [1] * len(g["decode_positions"])
    num_computed = [0] * len(g["prompt_lens"]) + g["decode_positions"]
    qsl = blocks.query_start_loc(n_sched, len(n_sched), sum(n_sched))
    assert int(qsl[-1]) == g["input_ids_len"]
    pos, seq_lens = blocks.positions_and_seq_lens(qsl, num_computed, len(n_sched), int(qsl[-1]))
    assert seq_lens.tolist() == g["seq_lens"]
    ctx = (seq_lens - np.diff(qsl)).tolist()
    assert ctx == g["context_lens"]
    assert pos[:35].tolist() == list(range(35)) and pos[-1] == 5
