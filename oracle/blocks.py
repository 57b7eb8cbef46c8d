"""Block and slot arithmetic of the paged KV cache, as the pages print it.

Test infrastructure (see the package docstring).  Each function restates one
rule from the pages; ``tests/test_oracle_blocks.py`` pins them against the
values the pages print.
"""
import numpy as np


def blocks_needed(seq_len: int, block_size: int = 16) -> int:
    """Blocks that hold ``seq_len`` tokens: ceil(seq_len / block_size).

    "Tour: One forward pass", stop 1: R3's 298-token prompt gets a block-table
    row of ceil(298 / 16) = 19 block ids."""
    return -(-int(seq_len) // int(block_size))


def blocks_at_admission(prompt_len: int, block_size: int = 16) -> int:
    """The older scheduler's reservation at admission: prompt_len // bs + 1.

    "vLLM 推理全流程深度解析" (vLLM inference deep dive), scheduler section
    (num_required_blocks).  It equals ``blocks_needed`` unless prompt_len is a
    multiple of the block size, where it reserves one block more."""
    return int(prompt_len) // int(block_size) + 1


def last_block_fill(seq_len: int, block_size: int = 16) -> int:
    """Tokens held by the last of a request's blocks (seq_len > 0)."""
    nb = blocks_needed(seq_len, block_size)
    return int(seq_len) - (nb - 1) * int(block_size)


def position_to_block(position: int, block_size: int = 16):
    """(block index in the request's row, offset inside the block).

    "Tour: One forward pass", stop 4: position 540 -> block index 33,
    offset 12; position 129 -> block index 8, offset 1."""
    return int(position) // int(block_size), int(position) % int(block_size)


def slot(block_number: int, offset: int, block_size: int = 16) -> int:
    """Physical slot of a token: block_number * block_size + offset (stop 4)."""
    return int(block_number) * int(block_size) + int(offset)


def block_mem_bytes(num_layers: int, num_kv_heads: int, head_size: int,
                    block_size: int, elem_bytes: int) -> int:
    """Bytes of one block id across all layers, K and V together:
    2 * num_layers * num_kv_heads * head_size * block_size * sizeof(elem).

    "vLLM 推理全流程深度解析", block-manager section (block_mem)."""
    return 2 * num_layers * num_kv_heads * head_size * block_size * elem_bytes


def query_start_loc(num_scheduled, max_num_reqs: int, num_tokens: int):
    """int32 [max_num_reqs + 1]: 0, the running sum of the scheduled tokens,
    then every entry past num_reqs set to num_tokens (non-decreasing).

    "Tour: One forward pass", stop 3 (prepare_inputs)."""
    n = len(num_scheduled)
    out = np.empty(max_num_reqs + 1, dtype=np.int32)
    out[0] = 0
    acc = 0
    for r in range(n):
        acc += int(num_scheduled[r])
        out[r + 1] = acc
    out[n + 1:] = num_tokens
    return out


def positions_and_seq_lens(qsl, num_computed, num_reqs: int, num_tokens_padded: int,
                           pad_value: int = -1):
    """positions int64 [num_tokens_padded] and seq_lens int32 [num_reqs].

    Token t of request r sits at num_computed[r] + (t - qsl[r]);
    seq_len = num_computed + query_len.  Padding rows are not written by the
    page's kernel; here they hold ``pad_value``.
    "Tour: One forward pass", stop 3 (prepare_pos_seq_lens)."""
    positions = np.full(num_tokens_padded, pad_value, dtype=np.int64)
    seq_lens = np.empty(num_reqs, dtype=np.int32)
    for r in range(num_reqs):
        q0, q1 = int(qsl[r]), int(qsl[r + 1])
        for t in range(q0, q1):
            positions[t] = int(num_computed[r]) + (t - q0)
        seq_lens[r] = int(num_computed[r]) + (q1 - q0)
    return positions, seq_lens


PAD_SLOT_ID = -1


def slot_mappings(block_table, qsl, positions, num_reqs: int, num_tokens_padded: int,
                  block_size: int = 16):
    """int64 [num_tokens_padded]: each scheduled token's slot
    block_table[r][pos // bs] * bs + pos % bs; rows past the last request's
    tokens get PAD_SLOT_ID = -1.

    "Tour: One forward pass", stop 4 (compute_slot_mappings)."""
    out = np.full(num_tokens_padded, PAD_SLOT_ID, dtype=np.int64)
    for r in range(num_reqs):
        for t in range(int(qsl[r]), int(qsl[r + 1])):
            bi, off = position_to_block(positions[t], block_size)
            out[t] = slot(block_table[r][bi], off, block_size)
    return out
