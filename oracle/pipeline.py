"""Oracle-side construction of a decode step's cache state (test infrastructure).

Runs the host steps of one decode iteration with the oracle's own pieces, in
the order of the per-iteration algorithm box of "079｜vLLM 与 PagedAttention"
(wq-win.github.io, §3): room for the next token (new block or copy-on-write of
a shared tail), copy, write the new keys/values, then attend.

The pool starts filled with a NaN bit pattern, so any slot that no token owns
reads as NaN.
"""

from __future__ import annotations

import numpy as np

from .block_manager import BlockManager
from .cache_ops import copy_blocks, reshape_and_cache


def pool_demand(context_lens, block_size: int) -> int:
    """Blocks the batch needs without sharing: sum of ceil(L / B)."""
    return int(sum(-(-int(L) // block_size) for L in context_lens))


def empty_pool(num_blocks: int, block_size: int, num_kv_heads: int, head_size: int,
               poison: int):
    shape = (num_blocks, block_size, num_kv_heads, head_size)
    return np.full(shape, poison, np.uint16), np.full(shape, poison, np.uint16)


def build_decode_state(batch, num_blocks: int, free_order, poison: int):
    """Prefill L-1 tokens of each sequence, then one decode append per sequence.

    Returns a dict with the block manager, both caches, the padded block tables
    (int32, -1 past each table), the prefill slot mapping and the decode step's
    slot mapping (one new token per sequence, the last row of its token data).
    """
    B = batch.block_size
    bm = BlockManager(num_blocks, B, free_order)
    kc, vc = empty_pool(num_blocks, B, batch.num_kv_heads, batch.head_size, poison)
    S = batch.num_seqs
    pre_slots = np.full(batch.total_tokens, -1, np.int64)
    for s in range(S):
        L = int(batch.context_lens[s])
        bm.allocate(s, L - 1)
        o = int(batch.offsets[s])
        pre_slots[o:o + L - 1] = bm.slots(s)
    reshape_and_cache(batch.k_tokens, batch.v_tokens, kc, vc, pre_slots)
    new_slots = np.empty(S, np.int64)
    for s in range(S):
        slot, cow = bm.append_slot(s)
        assert cow is None
        new_slots[s] = slot
    last = batch.offsets[1:] - 1
    reshape_and_cache(batch.k_tokens[last], batch.v_tokens[last], kc, vc, new_slots)
    tables = bm.padded_tables(range(S))
    return dict(bm=bm, k_cache=kc, v_cache=vc, block_tables=tables,
                prefill_slots=pre_slots, new_slots=new_slots,
                new_k=batch.k_tokens[last], new_v=batch.v_tokens[last])


def build_shared_prefix_state(batch, num_blocks: int, free_order, poison: int):
    """Beam groups: prefill each group's prefix once, fork it to every beam,
    then append every beam's tail one decode step at a time (all sequences in
    index order within a step). Copy-on-write pairs are applied before the
    tail tokens are written.
    """
    B = batch.block_size
    bm = BlockManager(num_blocks, B, free_order)
    kc, vc = empty_pool(num_blocks, B, batch.num_kv_heads, batch.head_size, poison)
    G, beams = batch.num_groups, batch.beams
    pre_slots = np.full(int(batch.prefix_offsets[-1]), -1, np.int64)
    for g in range(G):
        lead = g * beams
        bm.allocate(lead, int(batch.prefix_lens[g]))
        o = int(batch.prefix_offsets[g])
        pre_slots[o:o + int(batch.prefix_lens[g])] = bm.slots(lead)
        for b in range(1, beams):
            bm.fork(lead, lead + b)
    reshape_and_cache(batch.prefix_k, batch.prefix_v, kc, vc, pre_slots)
    tail_slots = np.full(int(batch.tail_offsets[-1]), -1, np.int64)
    cow_pairs = []
    max_tail = int(batch.tail_lens.max())
    for i in range(max_tail):
        for s in range(batch.num_seqs):
            if int(batch.tail_lens[s]) > i:
                slot, cow = bm.append_slot(s)
                tail_slots[int(batch.tail_offsets[s]) + i] = slot
                if cow is not None:
                    cow_pairs.append(cow)
    copy_blocks(kc, vc, cow_pairs)
    reshape_and_cache(batch.tail_k, batch.tail_v, kc, vc, tail_slots)
    S = batch.num_seqs
    context_lens = np.array([int(batch.prefix_lens[s // beams]) + int(batch.tail_lens[s])
                             for s in range(S)], np.int32)
    tables = bm.padded_tables(range(S))
    return dict(bm=bm, k_cache=kc, v_cache=vc, block_tables=tables,
                context_lens=context_lens, prefill_slots=pre_slots,
                tail_slots=tail_slots, cow_pairs=np.array(cow_pairs, np.int64).reshape(-1, 2))
