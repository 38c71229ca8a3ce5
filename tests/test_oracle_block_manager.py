"""Pins of the oracle block manager: the pages' worked examples (tests/golden),
the ceil(L/B) and tail-waste closed forms, the mean-waste identity, the free
list order, atomic failure, reference counting and copy-on-write rules."""

import json
import os
import random
from fractions import Fraction

import pytest

from oracle.block_manager import BlockManager, BlockManagerStateError, OutOfBlocks

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def test_worked_example_b4():
    ex = GOLD["b4_lengths_5_9"]
    bm = BlockManager(64, ex["block_size"])
    for i, L in enumerate(ex["lengths"]):
        bm.allocate(i, L)
    assert [len(bm.table(i)) for i in range(2)] == ex["blocks"]
    slots = sum(len(bm.table(i)) * ex["block_size"] for i in range(2))
    assert slots == ex["slots_total"]
    assert sum(ex["lengths"]) == ex["slots_used"]
    assert slots - sum(ex["lengths"]) == ex["slots_empty"]
    cont = ex["contiguous_reservation_per_request"] * len(ex["lengths"])
    assert cont == ex["contiguous_slots_total"]
    assert cont - sum(ex["lengths"]) == ex["contiguous_slots_empty"]


def test_worked_example_b16_growth():
    ex = GOLD["b16_lengths_17_31_32"]
    B = ex["block_size"]
    bm = BlockManager(64, B)
    for i, L in enumerate(ex["lengths"]):
        bm.allocate(i, L)
    assert [len(bm.table(i)) * B for i in range(3)] == ex["slots_each"]
    waste = [len(bm.table(i)) * B - L for i, L in enumerate(ex["lengths"])]
    assert waste == ex["waste"] and sum(waste) == ex["waste_total"]
    free0 = bm.num_free()
    for _ in range(ex["first_request_grows_by"]):
        bm.append_slot(0)
    assert (bm.num_free() != free0) == ex["new_block_needed_after_growth"]
    assert bm.length(0) == 31
    bm.append_slot(0)                                   # the 32nd token still fits
    assert bm.num_free() == free0 and bm.length(0) == ex["new_block_needed_after_crossing"]
    bm.append_slot(0)                                   # crossing 32 takes a block
    assert bm.num_free() == free0 - 1


@pytest.mark.parametrize("B", [1, 2, 3, 4, 8, 16, 128])
def test_block_count_and_waste_closed_form(B):
    for L in range(0, 400):
        bm = BlockManager(512, B)
        bm.allocate(0, L)
        n = len(bm.table(0))
        brute = 0
        while brute * B < L:                            # smallest n with n*B >= L
            brute += 1
        assert n == brute
        w = n * B - L
        if L > 0:
            assert GOLD["waste_bounds"]["lower"] <= w <= B - GOLD["waste_bounds"]["upper_is_block_size_minus"]


@pytest.mark.parametrize("B", [4, 8, 16, 32])
def test_mean_waste_when_length_mod_b_uniform(B):
    K = 7
    total = Fraction(0)
    for L in range(1, K * B + 1):
        bm = BlockManager(K + 1, B)
        bm.allocate(0, L)
        total += len(bm.table(0)) * B - L
    assert total / (K * B) == Fraction(B - 1, 2)


def test_free_list_pops_from_the_end_and_returns_in_order():
    bm = BlockManager(10, 4)
    assert bm.allocate(0, 9) == [9, 8, 7]
    assert bm.allocate(1, 1) == [6]
    bm.free_seq(0)
    assert bm.free[-3:] == [9, 8, 7]
    assert bm.allocate(2, 4) == [7]                     # last released first
    bm2 = BlockManager(5, 4, free_order=[3, 0, 4, 1, 2])
    assert bm2.allocate(0, 8) == [2, 1]


def test_out_of_blocks_changes_nothing():
    bm = BlockManager(4, 4)
    bm.allocate(0, 9)
    snap = (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()}, dict(bm.lens))
    with pytest.raises(OutOfBlocks):
        bm.allocate(1, 5)
    with pytest.raises(BlockManagerStateError):
        bm.allocate(0, 1)
    assert snap == (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()}, dict(bm.lens))
    bm.allocate(1, 4)
    bm.append_slot(0)
    bm.append_slot(0)
    bm.append_slot(0)                                   # 12 tokens: 3 blocks full
    snap = (list(bm.free), list(bm.ref), dict(bm.lens))
    with pytest.raises(OutOfBlocks):
        bm.append_slot(0)
    assert snap == (list(bm.free), list(bm.ref), dict(bm.lens))


def test_fork_then_write_copies_only_a_partial_tail():
    B = 4
    bm = BlockManager(16, B)
    bm.allocate(0, 6)                                   # blocks [15, 14], tail holds 2
    bm.fork(0, 1)
    assert bm.ref[15] == 2 and bm.ref[14] == 2
    slot, cow = bm.append_slot(1)                       # child writes the shared tail
    assert cow == (14, 13) and bm.table(1) == [15, 13] and slot == 13 * B + 2
    assert bm.ref[14] == 1 and bm.ref[15] == 2
    slot, cow = bm.append_slot(0)                       # parent is now alone on 14
    assert cow is None and slot == 14 * B + 2
    # full blocks are never copied: a fork at a block boundary shares, then grows
    bm.allocate(5, 8)
    bm.fork(5, 6)
    _, c1 = bm.append_slot(5)
    _, c2 = bm.append_slot(6)
    assert c1 is None and c2 is None and bm.table(5)[:2] == bm.table(6)[:2]


def test_beam_group_copies_all_but_the_last_writer():
    bm = BlockManager(64, 16)
    bm.allocate(0, 16 * 3 + 5)
    for b in (1, 2, 3):
        bm.fork(0, b)
    tail = bm.table(0)[3]
    cows = [bm.append_slot(b)[1] for b in range(4)]
    assert [c is not None for c in cows] == [True, True, True, False]
    assert all(c[0] == tail for c in cows[:3])
    assert bm.table(3)[3] == tail and bm.ref[tail] == 1


def test_reclaim_only_at_zero():
    bm = BlockManager(8, 2)
    bm.allocate(0, 4)
    bm.fork(0, 1)
    bm.free_seq(0)
    assert bm.num_free() == 6
    bm.free_seq(1)
    assert bm.num_free() == 8
    with pytest.raises(BlockManagerStateError):
        bm.free_seq(1)


def test_invariants_under_random_operations():
    rng = random.Random(11)
    for trial in range(20):
        N, B = rng.randint(4, 60), rng.choice([1, 2, 4, 8, 16])
        bm = BlockManager(N, B, free_order=rng.sample(range(N), N))
        live, nxt = [], 0
        for _ in range(300):
            op = rng.random()
            try:
                if op < 0.3 or not live:
                    bm.allocate(nxt, rng.randint(0, 3 * B)); live.append(nxt); nxt += 1
                elif op < 0.45:
                    bm.fork(rng.choice(live), nxt); live.append(nxt); nxt += 1
                elif op < 0.85:
                    bm.append_slot(rng.choice(live))
                else:
                    s = rng.choice(live); bm.free_seq(s); live.remove(s)
            except OutOfBlocks:
                pass
            refs = [0] * N
            for s in live:
                for b in bm.table(s):
                    refs[b] += 1
                assert len(bm.table(s)) == -(-bm.length(s) // B)
            assert refs == bm.ref
            assert len(set(bm.free)) == len(bm.free)
            assert set(bm.free) == {b for b in range(N) if refs[b] == 0}


def test_tiny_workload_counts():
    """The tiny decode batch (B=4, lengths 5, 9, 17, 31): 2+3+5+8 = 18 blocks,
    72 slots, 62 used, tail waste 3+3+3+1 = 10, by the w(L) closed form."""
    from workloads import TINY_LENS
    bm = BlockManager(64, 4)
    for s, L in enumerate(TINY_LENS):
        bm.allocate(s, L)
    n = [len(bm.table(s)) for s in range(4)]
    assert n == [2, 3, 5, 8] and sum(n) * 4 == 72 and sum(TINY_LENS) == 62
    assert [k * 4 - L for k, L in zip(n, TINY_LENS)] == [3, 3, 3, 1]


def test_pool_bytes_follow_the_kv_size_formula():
    """M_KV = 2 * layers * T * H_kv * d_h * s ("KV cache 有多大", §2 of the review):
    a one-layer pool of num_blocks*B token slots holds exactly that many bytes."""
    import numpy as np
    from oracle.pipeline import empty_pool
    for (N, B, Hkv, d) in [(64, 4, 4, 64), (10, 16, 40, 128), (3, 128, 8, 128)]:
        kc, vc = empty_pool(N, B, Hkv, d, 0x7E00)
        assert kc.nbytes + vc.nbytes == 2 * 1 * (N * B) * Hkv * d * 2


def test_swap_moves_a_group_and_keeps_sharing():
    """Swap out a beam group (4 sequences sharing a prefix): each distinct block
    gets one destination block, sharing is kept, the source blocks return to
    the source free list only when nothing references them."""
    gpu, cpu = BlockManager(32, 4), BlockManager(16, 4)
    gpu.allocate(0, 10)                                 # 3 blocks, tail holds 2
    for b in (1, 2, 3):
        gpu.fork(0, b)
    for b in range(4):
        gpu.append_slot(b)                              # 3 copy-on-write tails + 1 in place
    gpu.allocate(9, 5)                                  # bystander
    before = {s: gpu.table(s) for s in range(4)}
    distinct = sorted({b for t in before.values() for b in t})
    pairs = gpu.swap([0, 1, 2, 3], cpu)
    assert sorted(p[0] for p in pairs) == distinct
    assert len({p[1] for p in pairs}) == len(pairs) == 2 + 4  # shared prefix blocks once
    m = dict(pairs)
    for s in range(4):
        assert cpu.table(s) == [m[b] for b in before[s]]
        assert cpu.length(s) == 11
    assert cpu.ref[m[before[0][0]]] == 4                # shared prefix block
    assert gpu.num_free() == 32 - 2                     # only the bystander remains
    back = cpu.swap([0, 1, 2, 3], gpu)
    assert len(back) == len(pairs) and cpu.num_free() == 16
    for s in range(4):
        assert len(gpu.table(s)) == 3


def test_swap_is_all_or_nothing():
    gpu, cpu = BlockManager(16, 4), BlockManager(2, 4)
    gpu.allocate(0, 12)
    snap = (list(gpu.free), list(gpu.ref), list(cpu.free))
    with pytest.raises(OutOfBlocks):
        gpu.swap([0], cpu)
    assert snap == (list(gpu.free), list(gpu.ref), list(cpu.free))
    with pytest.raises(BlockManagerStateError):
        gpu.swap([0, 0], cpu)


def test_fnv1a64_published_vectors():
    from oracle.block_manager import fnv1a64
    assert fnv1a64(b"") == 0xcbf29ce484222325
    assert fnv1a64(b"a") == 0xaf63dc4c8601ec8c
    assert fnv1a64(b"foobar") == 0x85944171f73967e8


def test_prefix_cache_reuses_full_prompt_blocks():
    bm = BlockManager(32, 4)
    prompt = list(range(100, 111))                    # 11 tokens: 2 full blocks + 3
    assert bm.allocate_prefix(0, prompt) == 0         # nothing cached yet
    assert bm.allocate_prefix(1, prompt) == 8         # both full blocks reused
    assert bm.table(1)[:2] == bm.table(0)[:2] and bm.table(1)[2] != bm.table(0)[2]
    assert bm.ref[bm.table(0)[0]] == 2 and bm.ref[bm.table(0)[2]] == 1
    # same second-block tokens after a different first block: no hit (chained hash)
    other = [7, 7, 7, 7] + prompt[4:8]
    assert bm.allocate_prefix(2, other) == 0
    assert bm.table(2)[1] != bm.table(0)[1]
    # a prompt sharing only the first block
    assert bm.allocate_prefix(3, prompt[:4] + [1, 2, 3, 4, 5]) == 4


def test_prefix_cache_keeps_freed_blocks_until_evicted():
    bm = BlockManager(6, 4)
    a = [1, 2, 3, 4, 5, 6, 7, 8]                     # 2 full blocks
    bm.allocate_prefix(0, a)
    bm.free_seq(0)
    assert bm.num_free() == 6 and len(bm.free) == 4 and len(bm.evictable) == 2
    assert bm.allocate_prefix(1, a) == 8              # revived from the cache
    bm.free_seq(1)
    bm.allocate(2, 16)                                # takes the 4 free blocks ...
    bm.allocate(3, 4)                                 # ... then evicts the oldest cached one
    assert len(bm.evictable) == 1 and len(bm.cached) == 1
    bm.free_seq(3)
    assert bm.allocate_prefix(4, a) == 0              # the chain is broken at block 0
