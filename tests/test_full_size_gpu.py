"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (block size 16 or the sweep's, 512-token partitions, output in the
input dtype): sampled sequences against the oracle (all heads of each), plus
what holds at any size — bit-exact tables, pools and copy pairs against the
oracle's host pipeline, bit-identical outputs across block sizes."""

import math

import numpy as np
import pytest
import torch

from oracle.attention import paged_attention_decode as oracle_decode
from oracle.block_manager import BlockManager as RefBM
from oracle.pipeline import build_decode_state, build_shared_prefix_state, pool_demand
from parity import (assert_close, dev, gpu_decode_state, oracle_sampled, sample_seqs)
from workloads import (LLAMA_BLOCK_SIZES, free_order, gqa_prefix, llama13b, longctx, mqa,
                       opt13b, poison_bits)

pytestmark = pytest.mark.gpu


def _pool(lens, B):
    return int(math.ceil(1.2 * pool_demand(lens, B)))


def _tables_match_oracle(batch, n, order, tables):
    """The oracle block manager, driven with the same operations, gives the
    same tables bit for bit."""
    ref = RefBM(n, batch.block_size, order)
    for s in range(batch.num_seqs):
        ref.allocate(s, int(batch.context_lens[s]) - 1)
    for s in range(batch.num_seqs):
        ref.append_slot(s)
    assert np.array_equal(tables.cpu().numpy(), ref.padded_tables(range(batch.num_seqs),
                                                                   tables.shape[1]))


def test_opt13b_full():
    batch = opt13b(0)
    n = _pool(batch.context_lens, 16)
    order = free_order(n, 0)
    cache, tables, ctx = gpu_decode_state(batch, n, order, poison=True)
    ref = build_decode_state(batch, n, order, poison_bits("f16"))
    assert np.array_equal(tables.cpu().numpy(), ref["block_tables"])
    assert np.array_equal(cache.k_cache.view(torch.int16).cpu().numpy().view(np.uint16),
                          ref["k_cache"])
    assert np.array_equal(cache.v_cache.view(torch.int16).cpu().numpy().view(np.uint16),
                          ref["v_cache"])
    out = cache.attend(dev(batch.q, "f16"), tables, ctx, float(batch.scale))
    torch.cuda.synchronize()
    seqs = sample_seqs(batch.context_lens, 8, 0)
    want = oracle_decode(batch.q, ref["k_cache"], ref["v_cache"], ref["block_tables"],
                         batch.context_lens, 16, batch.scale, "f16", seqs=seqs)
    assert_close(out[seqs], want[seqs], "f16")
    assert cache.err.item() == 0


def test_llama13b_block_size_sweep_full():
    outs = []
    base = llama13b(0, block_size=16)
    seqs = sample_seqs(base.context_lens, 4, 1)
    want = oracle_sampled(base, seqs)
    for B in LLAMA_BLOCK_SIZES:
        batch = base
        batch.block_size = B
        n = _pool(batch.context_lens, B)
        order = free_order(n, B)
        cache, tables, ctx = gpu_decode_state(batch, n, order, poison=False)
        _tables_match_oracle(batch, n, order, tables)
        out = cache.attend(dev(batch.q, "f16"), tables, ctx, float(batch.scale))
        torch.cuda.synchronize()
        for s in seqs:
            assert_close(out[s], want[s], "f16")
        assert cache.err.item() == 0
        outs.append(out.cpu())
        del cache, tables, ctx, out
        torch.cuda.empty_cache()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    base.block_size = 16


def test_gqa_shared_prefix_full():
    from paged_kv_cache_118_gb300.cache import PagedKVCache
    pb = gqa_prefix(0)
    S = pb.num_seqs
    lens_logical = [int(pb.prefix_lens[s // 4]) + int(pb.tail_lens[s]) for s in range(S)]
    unique = pool_demand(pb.prefix_lens, 16) + pool_demand(pb.tail_lens + 16, 16)
    n = int(math.ceil(1.2 * unique))
    order = free_order(n, 0)
    ref = build_shared_prefix_state(pb, n, order, poison_bits("bf16"))
    cache = PagedKVCache(n, 16, 8, 128, torch.bfloat16, free_order=order)
    for g in range(pb.num_groups):
        a, b = pb.prefix_offsets[g], pb.prefix_offsets[g + 1]
        cache.prefill([4 * g], [b - a], dev(pb.prefix_k[a:b], "bf16"),
                      dev(pb.prefix_v[a:b], "bf16"))
        for j in range(1, 4):
            cache.fork(4 * g, 4 * g + j)
    cows = []
    for i in range(int(pb.tail_lens.max())):
        seqs = [s for s in range(S) if pb.tail_lens[s] > i]
        rows = pb.tail_offsets[seqs] + i
        _, cow = cache.append(seqs, dev(pb.tail_k[rows], "bf16"), dev(pb.tail_v[rows], "bf16"))
        cows += [tuple(c) for c in cow]
    assert len(cows) == 192 and cows == [tuple(c) for c in ref["cow_pairs"]]
    tables, ctx = cache.tables(range(S))
    assert np.array_equal(tables.cpu().numpy(), ref["block_tables"])
    assert list(ctx.cpu().numpy()) == lens_logical
    assert np.array_equal(cache.k_cache.view(torch.int16).cpu().numpy().view(np.uint16),
                          ref["k_cache"])
    assert np.array_equal(cache.v_cache.view(torch.int16).cpu().numpy().view(np.uint16),
                          ref["v_cache"])
    out = cache.attend(dev(pb.q, "bf16"), tables, ctx, float(pb.scale))
    torch.cuda.synchronize()
    seqs = sample_seqs(np.array(lens_logical), 8, 2)
    want = oracle_decode(pb.q, ref["k_cache"], ref["v_cache"], ref["block_tables"],
                         ref["context_lens"], 16, pb.scale, "bf16", seqs=seqs)
    assert_close(out[seqs], want[seqs], "bf16")
    assert cache.err.item() == 0


def test_longctx_full():
    batch = longctx(0)
    n = _pool(batch.context_lens, 16)
    order = free_order(n, 0)
    cache, tables, ctx = gpu_decode_state(batch, n, order, poison=True)
    _tables_match_oracle(batch, n, order, tables)
    out = cache.attend(dev(batch.q, "bf16"), tables, ctx, float(batch.scale))
    out32 = torch.empty(out.shape, dtype=torch.float32, device="cuda")
    cache.attend(dev(batch.q, "bf16"), tables, ctx, float(batch.scale), out=out32)
    torch.cuda.synchronize()
    seqs = [0, 4, 7]                       # 32k, 128k, 40k tokens
    want = oracle_sampled(batch, seqs)
    for s in seqs:
        assert_close(out[s], want[s], "bf16")
        assert_close(out32[s], want[s], "bf16")
    assert cache.err.item() == 0


def test_mqa_full():
    """64 query heads on one KV head (the tensor-memory path): sampled
    sequences against the oracle, both output types."""
    batch = mqa(0)
    n = _pool(batch.context_lens, 16)
    order = free_order(n, 0)
    cache, tables, ctx = gpu_decode_state(batch, n, order, poison=True)
    _tables_match_oracle(batch, n, order, tables)
    out = cache.attend(dev(batch.q, "bf16"), tables, ctx, float(batch.scale))
    out32 = torch.empty(out.shape, dtype=torch.float32, device="cuda")
    cache.attend(dev(batch.q, "bf16"), tables, ctx, float(batch.scale), out=out32)
    torch.cuda.synchronize()
    seqs = sample_seqs(batch.context_lens, 6, 1)
    want = oracle_sampled(batch, seqs)
    for s in seqs:
        assert_close(out[s], want[s], "bf16")
        assert_close(out32[s], want[s], "bf16")
    assert cache.err.item() == 0
