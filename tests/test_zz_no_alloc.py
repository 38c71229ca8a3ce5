"""The allocation-free decode entry point, for callers that cannot allocate
device memory (a plugin given only its input and output buffers, or a serving
loop that must not call cudaMalloc once it runs): it takes no workspace and
keeps its partials in a fixed array inside the library.

Checked through the C ABI against the regular entry point, which takes a
caller workspace, on calls in a row with different batches (the array keeps
the previous call's contents when the next one runs). Both entry points run
the same deterministic kernels on the same inputs, so their outputs must be
identical bit for bit: a read of stale or foreign rows of the shared array
would show up even where it stayed inside the attention tolerance. The test
needs nothing from other tests: it passes alone in a fresh process and after
them. Its file is collected after the others, so that a run which stops at
the first failure has run every other test first.
"""

import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_118_gb300 as pk
from oracle.pipeline import pool_demand
from parity import dev, gpu_decode_state
from workloads import decode_batch, free_order

pytestmark = pytest.mark.gpu


def _noalloc(out, q, cache, tables, ctx, scale, pt=0):
    S, H, D = q.shape
    nb, B, Hkv, _ = cache.k_cache.shape
    return pk.lib.pkv_paged_attention_decode_noalloc(
        out.data_ptr(), pk.PKV_F32 if out.dtype == torch.float32 else pk.PKV_BF16 if
        out.dtype == torch.bfloat16 else pk.PKV_F16, q.data_ptr(), cache.k_cache.data_ptr(),
        cache.v_cache.data_ptr(), pk.PKV_BF16 if q.dtype == torch.bfloat16 else pk.PKV_F16,
        tables.data_ptr(), ctx.data_ptr(), S, H, Hkv, D, nb, B, tables.shape[1], float(scale),
        pt, cache.err.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _case(lens, H, Hkv, B, dt, seed):
    batch = decode_batch("n", lens, H, Hkv, 128, B, dt, seed=seed)
    n = pool_demand(batch.context_lens, B) + 5
    cache, tables, ctx = gpu_decode_state(batch, n, free_order(n, seed))
    return batch, cache, tables, ctx


def test_matches_workspace_entry_point_twice_in_a_row():
    cases = [((3000, 17, 900, 1, 2048, 513), 32, 8, 16, "bf16", 1),
             ((40, 700, 1500), 40, 40, 32, "f16", 2),
             ((1200, 5, 333), 64, 1, 16, "bf16", 3)]          # 64 heads per KV head: tcgen05
    runs = []
    for lens, H, Hkv, B, dt, seed in cases:
        batch, cache, tables, ctx = _case(lens, H, Hkv, B, dt, seed)
        q = dev(batch.q, dt)
        need = pk.pkv_decode_workspace_size(batch.num_seqs, H, Hkv, 128, tables.shape[1], B)
        assert need <= pk.NOALLOC_SCRATCH_BYTES
        want = cache.attend(q, tables, ctx, float(batch.scale)).clone()
        runs.append((batch, cache, tables, ctx, q, want, dt))
    torch.cuda.synchronize()
    outs = []
    for batch, cache, tables, ctx, q, want, dt in runs:      # two calls in a row
        got = torch.full_like(want, float("nan"))
        assert _noalloc(got, q, cache, tables, ctx, batch.scale) == pk.PKV_OK
        outs.append(got)
    torch.cuda.synchronize()
    for (batch, cache, tables, ctx, q, want, dt), got in zip(runs, outs):
        assert torch.equal(got, want), (got.float() - want.float()).abs().max().item()
        assert cache.err.item() == 0


def test_refuses_batches_beyond_the_built_in_scratch():
    batch, cache, tables, ctx = _case((64,), 8, 8, 16, "f16", 3)
    q = dev(batch.q, "f16")
    out = torch.zeros_like(q)
    # a table wide enough that the partials would not fit: rows of 128 floats + (m, l),
    # in partitions of the default size for so wide a table (1024 tokens)
    parts = pk.NOALLOC_SCRATCH_BYTES // (8 * (128 * 4 + 8)) + 1
    width = parts * 1024 // 16
    assert pk.pkv_decode_partition_tokens(1, 8, 8, 128, width, 16) == 1024
    wide = torch.full((1, width), -1, dtype=torch.int32, device="cuda")
    wide[0, :tables.shape[1]] = tables[0]
    assert pk.pkv_decode_workspace_size(1, 8, 8, 128, width, 16) > pk.NOALLOC_SCRATCH_BYTES
    assert _noalloc(out, q, cache, wide, ctx, batch.scale) == pk.PKV_EWORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 0)
