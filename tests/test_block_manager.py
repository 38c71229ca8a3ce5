"""The library's C++ block manager against the oracle's Python one: identical
tables, slots, copy-on-write pairs, reference counts and free lists for the
same operation sequence, bit for bit; and its own error behaviour."""

import random

import numpy as np
import pytest

import paged_kv_cache_118_gb300 as pk
from oracle.block_manager import BlockManager as RefBM
from oracle.block_manager import BlockManagerStateError, OutOfBlocks
from workloads import free_order, gqa_prefix


def same_state(bm, ref, live):
    assert bm.num_free() == ref.num_free()
    assert list(bm.free_list()) == ref.free
    for b in range(ref.num_blocks):
        assert bm.refcount(b) == ref.ref[b]
    for s in live:
        assert list(bm.table(s)) == ref.table(s)
        assert bm.length(s) == ref.length(s)
        assert list(bm.slots(s)) == ref.slots(s)


@pytest.mark.parametrize("seed", range(12))
def test_random_operations_match_oracle(seed):
    rng = random.Random(seed)
    N, B = rng.randint(4, 80), rng.choice([1, 2, 4, 8, 16, 32])
    order = free_order(N, seed)
    bm, ref = pk.BlockManager(N, B, order), RefBM(N, B, order)
    live, nxt = [], 0
    for _ in range(400):
        op = rng.random()
        if op < 0.25 or not live:
            n = rng.randint(0, 3 * B)
            try:
                ref.allocate(nxt, n)
                ok = True
            except OutOfBlocks:
                ok = False
            if ok:
                bm.allocate(nxt, n)
                live.append(nxt)
            else:
                with pytest.raises(pk.PagedKVError) as e:
                    bm.allocate(nxt, n)
                assert e.value.status == pk.PKV_ENOMEM
            nxt += 1
        elif op < 0.4:
            p = rng.choice(live)
            ref.fork(p, nxt); bm.fork(p, nxt); live.append(nxt); nxt += 1
        elif op < 0.7:
            s = rng.choice(live)
            try:
                want = ref.append_slot(s)
            except OutOfBlocks:
                with pytest.raises(pk.PagedKVError) as e:
                    bm.append_slot(s)
                assert e.value.status == pk.PKV_ENOMEM
            else:
                assert bm.append_slot(s) == want
        elif op < 0.85:
            batch = [rng.choice(live) for _ in range(rng.randint(1, 6))]
            snap = (list(ref.free), list(ref.ref), {k: list(v) for k, v in ref.tables.items()},
                    dict(ref.lens))
            try:
                want = [ref.append_slot(s) for s in batch]
            except OutOfBlocks:
                ref.free, ref.ref, ref.tables, ref.lens = snap   # all or nothing
                with pytest.raises(pk.PagedKVError) as e:
                    bm.append_slots(batch)
                assert e.value.status == pk.PKV_ENOMEM
            else:
                slots, cow = bm.append_slots(batch)
                assert list(slots) == [w[0] for w in want]
                assert [tuple(c) for c in cow] == [w[1] for w in want if w[1] is not None]
        else:
            s = rng.choice(live)
            ref.free_seq(s); bm.free_seq(s); live.remove(s)
        same_state(bm, ref, live)


def test_beam_groups_match_oracle_and_copy_three_of_four():
    pb = gqa_prefix(seed=1, groups=5, beams=4, prefix_tokens=48, max_tail=20)
    N = 120
    order = free_order(N, 4)
    bm, ref = pk.BlockManager(N, 16, order), RefBM(N, 16, order)
    for g in range(pb.num_groups):
        for m in (bm, ref):
            m.allocate(4 * g, int(pb.prefix_lens[g]))
            for b in range(1, 4):
                m.fork(4 * g, 4 * g + b)
    seqs = list(range(pb.num_seqs))
    slots, cow = bm.append_slots(seqs)
    want = [ref.append_slot(s) for s in seqs]
    assert list(slots) == [w[0] for w in want]
    assert len(cow) == 3 * pb.num_groups
    same_state(bm, ref, seqs)


def test_error_statuses():
    bm = pk.BlockManager(4, 4)
    bm.allocate(1, 5)
    for fn, args, status in [(bm.allocate, (1, 1), pk.PKV_ESTATE),
                             (bm.allocate, (2, 9), pk.PKV_ENOMEM),
                             (bm.fork, (7, 8), pk.PKV_ESTATE),
                             (bm.fork, (1, 1), pk.PKV_ESTATE),
                             (bm.append_slot, (9,), pk.PKV_ESTATE),
                             (bm.free_seq, (9,), pk.PKV_ESTATE)]:
        with pytest.raises(pk.PagedKVError) as e:
            fn(*args)
        assert e.value.status == status
    assert bm.length(9) == -1 and bm.refcount(99) == -1
    with pytest.raises(pk.PagedKVError):
        pk.BlockManager(4, 4, free_order=[0, 1, 1, 2])
    tabs, lens = bm.fill_tables([1], 4)
    assert list(tabs[0]) == [3, 2, -1, -1] and list(lens) == [5]
    with pytest.raises(pk.PagedKVError) as e:
        bm.fill_tables([1], 1)
    assert e.value.status == pk.PKV_ERANGE


@pytest.mark.parametrize("seed", range(6))
def test_swap_matches_oracle(seed):
    rng = random.Random(100 + seed)
    B = rng.choice([2, 4, 16])
    N, M = 60, 40
    og, oc = free_order(N, seed), free_order(M, seed + 7)
    gpu, cpu = pk.BlockManager(N, B, og), pk.BlockManager(M, B, oc)
    rg, rc = RefBM(N, B, og), RefBM(M, B, oc)
    nxt = 0
    groups = []
    for _ in range(5):                      # beam groups sharing a partial prefix
        lead, L = nxt, rng.randint(0, 3 * B)
        for m in (gpu, rg):
            m.allocate(lead, L)
        members = [lead]
        for j in range(rng.randint(0, 3)):
            for m in (gpu, rg):
                m.fork(lead, nxt + 1 + j)
            members.append(nxt + 1 + j)
        for s in members:
            if rng.random() < 0.7:
                assert gpu.append_slot(s) == rg.append_slot(s)
        nxt += len(members)
        groups.append(members)
    for g in groups:                          # out, then back in, comparing each time
        for (src, dst, rs, rd) in ((gpu, cpu, rg, rc), (cpu, gpu, rc, rg)):
            try:
                want = rs.swap(g, rd)
            except OutOfBlocks:
                with pytest.raises(pk.PagedKVError) as e:
                    src.swap(g, dst)
                assert e.value.status == pk.PKV_ENOMEM
                continue
            got = src.swap(g, dst)
            assert [tuple(p) for p in got] == want
            live_src = [s for gg in groups for s in gg if s in rs.tables]
            live_dst = [s for gg in groups for s in gg if s in rd.tables]
            same_state(src, rs, live_src)
            same_state(dst, rd, live_dst)


def test_swap_errors():
    a, b, c = pk.BlockManager(8, 4), pk.BlockManager(2, 4), pk.BlockManager(8, 8)
    a.allocate(0, 12)
    with pytest.raises(pk.PagedKVError) as e:
        a.swap([0], b)
    assert e.value.status == pk.PKV_ENOMEM
    assert a.num_free() == 5 and b.num_free() == 2
    with pytest.raises(pk.PagedKVError) as e:
        a.swap([0], c)
    assert e.value.status == pk.PKV_EINVAL
    with pytest.raises(pk.PagedKVError) as e:
        a.swap([7], b)
    assert e.value.status == pk.PKV_ESTATE
    a.allocate(1, 0)                          # empty table: nothing to copy
    assert len(a.swap([1], b)) == 0 and b.length(1) == 0


@pytest.mark.parametrize("seed", range(8))
def test_prefix_cache_matches_oracle(seed):
    rng = random.Random(300 + seed)
    N, B = rng.randint(20, 60), rng.choice([2, 4, 8])
    order = free_order(N, seed)
    bm, ref = pk.BlockManager(N, B, order), RefBM(N, B, order)
    prompts = [[rng.randint(0, 3) for _ in range(rng.randint(0, 4 * B))] for _ in range(6)]
    live, nxt = [], 0
    for _ in range(150):
        op = rng.random()
        if op < 0.45 or not live:
            base = rng.choice(prompts)
            toks = base[:rng.randint(0, len(base))] + [rng.randint(0, 3) for _ in range(rng.randint(0, B))]
            try:
                want = ref.allocate_prefix(nxt, toks)
            except OutOfBlocks:
                with pytest.raises(pk.PagedKVError) as e:
                    bm.allocate_prefix(nxt, toks)
                assert e.value.status == pk.PKV_ENOMEM
            else:
                assert bm.allocate_prefix(nxt, toks) == want
                live.append(nxt)
            nxt += 1
        elif op < 0.6:
            s = rng.choice(live)
            try:
                want = ref.append_slot(s)
            except OutOfBlocks:
                with pytest.raises(pk.PagedKVError):
                    bm.append_slot(s)
            else:
                assert bm.append_slot(s) == want
        elif op < 0.7:
            p = rng.choice(live)
            ref.fork(p, nxt); bm.fork(p, nxt); live.append(nxt); nxt += 1
        else:
            s = rng.choice(live)
            ref.free_seq(s); bm.free_seq(s); live.remove(s)
        same_state(bm, ref, live)
        assert bm.num_cached() == len(ref.cached)
