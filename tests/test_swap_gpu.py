"""swap_blocks on the GPU: copies between the device pool and a pinned host
pool (swap space), bitwise against the oracle, and a preemption round trip —
swap a sequence group out, let other sequences take its blocks, swap it back
into different blocks — that leaves the attention output unchanged bit for bit."""

import numpy as np
import pytest
import torch

import paged_kv_cache_118_gb300 as pk
from oracle.cache_ops import swap_blocks as oracle_swap
from oracle.pipeline import pool_demand
from parity import dev, gpu_decode_state
from workloads import decode_batch, free_order

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("n_pairs", [1, 9, 1100])
def test_swap_blocks_device_host_bitwise(n_pairs):
    rng = np.random.default_rng(n_pairs)
    G, H = n_pairs + 7, n_pairs + 3
    gk_h = rng.integers(0, 1 << 16, (G, 16, 4, 128), dtype=np.uint16)
    gv_h = rng.integers(0, 1 << 16, (G, 16, 4, 128), dtype=np.uint16)
    gk, gv = dev(gk_h, "bf16"), dev(gv_h, "bf16")
    hk = torch.zeros((H, 16, 4, 128), dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    out_pairs = np.stack([rng.permutation(G)[:n_pairs], rng.permutation(H)[:n_pairs]], 1)
    pk.pkv_swap_blocks(hk, hv, gk, gv, out_pairs)            # device -> host
    torch.cuda.synchronize()
    hk_want = np.zeros((H, 16, 4, 128), np.uint16)
    hv_want = np.zeros_like(hk_want)
    oracle_swap(gk_h, gv_h, hk_want, hv_want, out_pairs)
    assert np.array_equal(_bits(hk), hk_want) and np.array_equal(_bits(hv), hv_want)
    in_pairs = np.stack([out_pairs[:, 1], rng.permutation(G)[:n_pairs]], 1)
    pk.pkv_swap_blocks(gk, gv, hk, hv, in_pairs)              # host -> device
    torch.cuda.synchronize()
    oracle_swap(hk_want, hv_want, gk_h, gv_h, in_pairs)
    assert np.array_equal(_bits(gk), gk_h) and np.array_equal(_bits(gv), gv_h)


def test_swap_rejects_bad_pairs():
    gk = torch.zeros((4, 16, 4, 128), dtype=torch.bfloat16, device="cuda")
    hk = torch.zeros((4, 16, 4, 128), dtype=torch.bfloat16).pin_memory()
    with pytest.raises(pk.PagedKVError) as e:
        pk.pkv_swap_blocks(hk, hk, gk, gk, [(0, 4)])
    assert e.value.status == pk.PKV_ERANGE
    with pytest.raises(pk.PagedKVError) as e:
        pk.pkv_swap_blocks(hk, hk, gk, gk, [(0, 1), (2, 1)])
    assert e.value.status == pk.PKV_EINVAL


def test_preempt_and_resume_round_trip():
    batch = decode_batch("t", (300, 40, 1500, 77), 8, 2, 128, 16, "bf16", seed=31)
    n = 2 * pool_demand(batch.context_lens, 16) + 8   # room to swap back into other blocks
    cache, tables, ctx = gpu_decode_state(batch, n, free_order(n, 5))
    q = dev(batch.q, "bf16")
    before = cache.attend(q, tables, ctx, float(batch.scale)).clone()
    M = 300
    hk = torch.empty((M, 16, 2, 128), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    cpu = pk.BlockManager(M, 16, free_order(M, 6))
    group = [1, 2]
    pairs = cache.bm.swap(group, cpu)
    pk.pkv_swap_blocks(hk, hv, cache.k_cache, cache.v_cache, pairs)
    torch.cuda.synchronize()
    # the freed GPU blocks go to another sequence and are overwritten
    freed = torch.as_tensor(pairs[:, 0], dtype=torch.long, device="cuda")
    cache.k_cache[freed] = float("nan")
    cache.v_cache[freed] = float("nan")
    cache.bm.allocate(99, 16 * len(pairs))
    pairs_in = cpu.swap(group, cache.bm)
    assert set(pairs_in[:, 1]).isdisjoint(set(pairs[:, 0]))
    pk.pkv_swap_blocks(cache.k_cache, cache.v_cache, hk, hv, pairs_in)
    tables2, ctx2 = cache.tables(range(4))
    after = cache.attend(q, tables2, ctx2, float(batch.scale))
    torch.cuda.synchronize()
    assert torch.equal(before, after)
    assert cache.err.item() == 0
