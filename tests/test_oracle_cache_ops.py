"""Pins of the oracle's cache writes: the scatter puts every token where the
gather through the block table finds it again, padding slots are skipped,
out-of-range slots are refused; copy_blocks copies exactly the named blocks."""

import numpy as np
import pytest

from oracle.attention import gather_sequence
from oracle.block_manager import BlockManager
from oracle.cache_ops import copy_blocks, reshape_and_cache
from workloads import normal_bits


def test_scatter_then_gather_round_trip():
    rng = np.random.default_rng(0)
    B, Hkv, d, N = 4, 3, 8, 40
    bm = BlockManager(N, B, free_order=rng.permutation(N))
    lens = [1, 4, 5, 13, 16]
    kc = np.full((N, B, Hkv, d), 0x7E00, np.uint16)
    vc = kc.copy()
    toks = []
    for s, L in enumerate(lens):
        bm.allocate(s, L)
        k = normal_bits(rng, (L, Hkv, d), "f16")
        v = normal_bits(rng, (L, Hkv, d), "f16")
        reshape_and_cache(k, v, kc, vc, np.array(bm.slots(s), np.int64))
        toks.append((k, v))
    for s, L in enumerate(lens):
        assert np.array_equal(gather_sequence(kc, bm.table(s), L, B), toks[s][0])
        assert np.array_equal(gather_sequence(vc, bm.table(s), L, B), toks[s][1])
    # every slot that no token owns still holds the poison pattern
    owned = {sl for s in range(len(lens)) for sl in bm.slots(s)}
    flat = kc.reshape(N * B, Hkv, d)
    for sl in range(N * B):
        if sl not in owned:
            assert np.all(flat[sl] == 0x7E00)


def test_scatter_skips_padding_and_refuses_out_of_range():
    kc = np.zeros((2, 2, 1, 4), np.uint16)
    vc = kc.copy()
    k = np.arange(12, dtype=np.uint16).reshape(3, 1, 4)
    reshape_and_cache(k, k, kc, vc, np.array([3, -1, 0]))
    assert np.array_equal(kc[1, 1, 0], k[0, 0]) and np.array_equal(kc[0, 0, 0], k[2, 0])
    assert kc.sum() == k[0].sum() + k[2].sum()
    with pytest.raises(IndexError):
        reshape_and_cache(k[:1], k[:1], kc, vc, np.array([4]))


def test_copy_blocks_copies_named_blocks_only():
    rng = np.random.default_rng(1)
    kc = rng.integers(0, 1 << 16, (10, 4, 2, 8), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, (10, 4, 2, 8), dtype=np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    copy_blocks(kc, vc, [(1, 7), (1, 8), (3, 2)])
    for src, dst in [(1, 7), (1, 8), (3, 2)]:
        assert np.array_equal(kc[dst], k0[src]) and np.array_equal(vc[dst], v0[src])
    for b in (0, 1, 3, 4, 5, 6, 9):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])
    with pytest.raises(ValueError):
        copy_blocks(kc, vc, [(1, 2), (2, 3)])
    with pytest.raises(ValueError):
        copy_blocks(kc, vc, [(1, 2), (3, 2)])


def test_swap_blocks_copies_between_pools():
    from oracle.cache_ops import swap_blocks
    rng = np.random.default_rng(2)
    gk = rng.integers(0, 1 << 16, (8, 4, 2, 8), dtype=np.uint16)
    gv = rng.integers(0, 1 << 16, (8, 4, 2, 8), dtype=np.uint16)
    hk = np.zeros((5, 4, 2, 8), np.uint16)
    hv = np.zeros_like(hk)
    swap_blocks(gk, gv, hk, hv, [(7, 0), (2, 4)])
    assert np.array_equal(hk[0], gk[7]) and np.array_equal(hv[4], gv[2])
    assert not hk[1:4].any()
    with pytest.raises(ValueError):
        swap_blocks(gk, gv, hk, hv, [(1, 2), (3, 2)])
