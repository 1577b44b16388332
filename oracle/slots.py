"""Slot arithmetic of the paged KV cache, as the pages state it.

Test infrastructure only (see the package docstring).
"""
from __future__ import annotations


def slot_of(block_id: int, block_size: int, loc: int) -> int:
    """[UML] §1 Step2: a slot's global index is blockID * blockSize + loc, where
    loc is the token's offset inside its block (worked example 25*4+2 = 102)."""
    return block_id * block_size + loc


def get_slots(block_ids: list[int], block_size: int, seq_len: int) -> list[int]:
    """[UML] §3.2 "KV cache的写入函数": the slots of a whole sequence are every slot
    of each block but the last, then the first seq_len-(n-1)*block_size slots
    of the last block."""
    slots: list[int] = []
    for b in block_ids[:-1]:
        first = b * block_size
        slots.extend(range(first, first + block_size))
    tail = seq_len - (len(block_ids) - 1) * block_size
    first = block_ids[-1] * block_size
    slots.extend(range(first, first + tail))
    return slots


def num_blocks(num_tokens: int, block_size: int) -> int:
    """[SRC2] sequence.py, Sequence.num_blocks: blocks a sequence occupies,
    rounded up."""
    return (num_tokens + block_size - 1) // block_size


def last_block_num_tokens(num_tokens: int, block_size: int) -> int:
    """[SRC2] sequence.py, Sequence.last_block_num_tokens: tokens held by the
    last block (600 tokens with 256-slot blocks -> 88)."""
    return num_tokens - (num_blocks(num_tokens, block_size) - 1) * block_size


def needs_new_block(num_tokens_after_append: int, num_table_blocks: int,
                    block_size: int) -> bool:
    """[SRC2] scheduler.py decode stage: a block is appended to the table only
    when the current last block is full, i.e. when the appended token would
    not fit in the blocks the table already has."""
    return num_tokens_after_append > num_table_blocks * block_size


def decode_slot(block_table: list[int], num_tokens: int, block_size: int) -> int:
    """The slot of a decode step's new token: it sits at position num_tokens-1
    of its sequence, in logical block (num_tokens-1)//block_size at offset
    (num_tokens-1)%block_size ([UML] §1 Step2 formula; [LIFE] §3.3.2 slot_mapping
    is one slot per flattened token)."""
    pos = num_tokens - 1
    return slot_of(block_table[pos // block_size], block_size, pos % block_size)


def prefill_metadata(seqs, block_size: int):
    """[LIFE] §3.3.2 prepare_prefill: flattens the scheduled tokens of several
    sequences.  `seqs` is a list of (num_cached_tokens, num_scheduled_tokens,
    block_table).  Returns positions, cu_seqlens_q, cu_seqlens_k and
    slot_mapping: token t of a sequence sits at position num_cached+t, its KV
    goes to the slot of that position ([UML] §1 Step2), cu_seqlens_q are the
    prefix sums of scheduled counts and cu_seqlens_k those of
    num_cached+scheduled ([UML] §3.2 format list)."""
    positions, slots = [], []
    cu_q, cu_k = [0], [0]
    for cached, sched, table in seqs:
        for t in range(sched):
            p = cached + t
            positions.append(p)
            slots.append(slot_of(table[p // block_size], block_size, p % block_size))
        cu_q.append(cu_q[-1] + sched)
        cu_k.append(cu_k[-1] + cached + sched)
    return positions, cu_q, cu_k, slots


def chunk_rounds(num_tokens: int, num_cached_tokens: int, budget: int):
    """[LIFE] §3.1 / [SRC2] Sequence walkthrough: each round computes
    min(remaining, budget) tokens starting at num_cached_tokens, then
    num_cached_tokens advances by that count.  Returns (start, count) pairs."""
    rounds = []
    cached = num_cached_tokens
    while cached < num_tokens:
        n = min(num_tokens - cached, budget)
        rounds.append((cached, n))
        cached += n
    return rounds
