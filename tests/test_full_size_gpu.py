"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (block size 16 or the sweep's, the default partitions, output in the
input dtype), and with fp32 outputs held to the plain bound: EVERY sequence
and head of each batch against the oracle, element by element. Also what
holds at any size: bit-exact tables, pools and copy pairs against the
oracle's host pipeline, and bit-identical outputs across block sizes.

The long-context batch also runs at its stated 512-token partitions (1232
partitions, up to 256 partials per row for the merge).

The oracle is one fp64 mat-vec per (sequence, head); it runs on a pool of
host threads (tests/parity.py, ``oracle_all``).
"""

import functools
import math

import numpy as np
import pytest
import torch

from oracle.attention import paged_attention_decode as oracle_decode
from oracle.block_manager import BlockManager as RefBM
from oracle.pipeline import build_decode_state, build_shared_prefix_state, pool_demand
from parity import (assert_close, dev, gpu_decode_state, oracle_all, record_max_err,
                    stack_oracle)
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


def _check_all(name, cache, q, tables, ctx, scale, want, dtype, partition_tokens=0):
    """Both output types of one decode call against the oracle, every element;
    and the same call again, bit for bit (every CTA must derive the same work
    list, whatever order its threads run in)."""
    out = cache.attend(q, tables, ctx, scale, partition_tokens=partition_tokens)
    out32 = torch.empty(out.shape, dtype=torch.float32, device="cuda")
    cache.attend(q, tables, ctx, scale, out=out32, partition_tokens=partition_tokens)
    again = torch.empty_like(out32)
    cache.attend(q, tables, ctx, scale, out=again, partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    assert torch.equal(again, out32)
    record_max_err(f"{name} ({dtype} out)", assert_close(out, want, dtype))
    record_max_err(f"{name} (fp32 out)", assert_close(out32, want, dtype))
    assert cache.err.item() == 0
    return out


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
    want = stack_oracle(oracle_all(batch), range(batch.num_seqs))
    _check_all("opt13b", cache, dev(batch.q, "f16"), tables, ctx, float(batch.scale), want, "f16")


def test_llama13b_block_size_sweep_full():
    outs = []
    base = llama13b(0, block_size=16)
    want = stack_oracle(oracle_all(base), range(base.num_seqs))   # the same for every B
    for B in LLAMA_BLOCK_SIZES:
        batch = base
        batch.block_size = B
        n = _pool(batch.context_lens, B)
        order = free_order(n, B)
        cache, tables, ctx = gpu_decode_state(batch, n, order, poison=False)
        _tables_match_oracle(batch, n, order, tables)
        out = _check_all(f"llama13b B={B}", cache, dev(batch.q, "f16"), tables, ctx,
                         float(batch.scale), want, "f16")
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
    # every beam against the oracle on the oracle's own shared-prefix pool
    want = _oracle_threads(lambda s: oracle_decode(
        pb.q, ref["k_cache"], ref["v_cache"], ref["block_tables"], ref["context_lens"], 16,
        pb.scale, "bf16", seqs=[s])[s], S)
    _check_all("gqa_prefix", cache, dev(pb.q, "bf16"), tables, ctx, float(pb.scale), want, "bf16")


def _oracle_threads(fn, n, workers=8):
    import concurrent.futures as cf
    with cf.ThreadPoolExecutor(workers) as ex:
        return np.stack(list(ex.map(fn, range(n))))


@functools.lru_cache(maxsize=1)
def _longctx():
    batch = longctx(0)
    return batch, stack_oracle(oracle_all(batch, max_workers=4), range(batch.num_seqs))


@pytest.mark.parametrize("partition_tokens", [0, 512])
def test_longctx_full(partition_tokens):
    """0: the default for so long a table (1024-token partitions, what bench.py
    times by default); 512: the workload's stated partitions, 1232 of them,
    up to 256 partials per row in the merge."""
    import paged_kv_cache_118_gb300 as pk
    batch, want = _longctx()
    n = _pool(batch.context_lens, 16)
    order = free_order(n, 0)
    cache, tables, ctx = gpu_decode_state(batch, n, order, poison=True)
    _tables_match_oracle(batch, n, order, tables)
    pt = pk.pkv_decode_partition_tokens(batch.num_seqs, 32, 8, 128, tables.shape[1], 16,
                                        partition_tokens)
    assert pt == (1024 if partition_tokens == 0 else 512)
    if pt == 512:
        parts = sum(-(-int(L) // 512) for L in batch.context_lens)
        assert parts == 1232 and -(-int(batch.context_lens.max()) // 512) == 256
    _check_all(f"longctx partitions={pt}", cache, dev(batch.q, "bf16"), tables, ctx,
               float(batch.scale), want, "bf16", partition_tokens=partition_tokens)


def test_mqa_full():
    """64 query heads on one KV head (the tensor-memory path): every sequence
    against the oracle, both output types."""
    batch = mqa(0)
    n = _pool(batch.context_lens, 16)
    order = free_order(n, 0)
    cache, tables, ctx = gpu_decode_state(batch, n, order, poison=True)
    _tables_match_oracle(batch, n, order, tables)
    want = stack_oracle(oracle_all(batch), range(batch.num_seqs))
    _check_all("mqa", cache, dev(batch.q, "bf16"), tables, ctx, float(batch.scale), want, "bf16")
