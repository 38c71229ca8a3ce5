"""Failure detection on the GPU, without a fault: a pipeline wait that runs out.

Every wait of the decode kernels on an mbarrier has a time limit, after which
the kernel flags PKV_DEVERR_TIMEOUT, lets its copies and tensor-core products
in flight finish, frees its tensor memory and returns. The library's test hook
pkv_test_decode_wait_timeout runs the tensor-memory decode path (64 query heads
on one KV head) with a 2 ms limit and its softmax warps waiting, at their first
unit, on a barrier that nothing completes; the waits of the MMA thread and the
copy warp, which depend on them, then run out too. The call must come back with
the flag set, and a normal call right after it must be correct: that kernel
allocates all of the SM's tensor memory, so it also shows that the aborted one
freed it.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_118_gb300 as pk
from oracle.pipeline import pool_demand
from parity import assert_close, dev, gpu_decode_state, oracle_all, stack_oracle
from workloads import decode_batch, free_order

pytestmark = pytest.mark.gpu


def _hook(out, q, cache, tables, ctx, scale, ws, err, limit_ns):
    S, H, D = q.shape
    nb, B, Hkv, _ = cache.k_cache.shape
    return pk.lib.pkv_test_decode_wait_timeout(
        out.data_ptr(), pk.PKV_F32, q.data_ptr(), cache.k_cache.data_ptr(),
        cache.v_cache.data_ptr(), pk.PKV_BF16, tables.data_ptr(), ctx.data_ptr(), S, H, Hkv, D,
        nb, B, tables.shape[1], float(scale), 0, ws.data_ptr(), ws.numel(), err.data_ptr(),
        limit_ns, torch.cuda.current_stream().cuda_stream)


def test_wait_runs_out_then_next_call_is_correct():
    batch = decode_batch("mqa_small", (700, 1, 2048, 333, 64, 1500), 64, 1, 128, 16, "bf16", seed=5)
    n = pool_demand(batch.context_lens, 16) + 7
    cache, tables, ctx = gpu_decode_state(batch, n, free_order(n, 5))
    q = dev(batch.q, "bf16")
    want = stack_oracle(oracle_all(batch), range(batch.num_seqs))
    scale = float(batch.scale)
    ws = cache.workspace(batch.num_seqs, 64, tables.shape[1])
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")

    cache.attend(q, tables, ctx, scale, out=out)           # the path works before
    torch.cuda.synchronize()
    assert_close(out, want, "bf16")
    assert cache.err.item() == 0

    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _hook(out, q, cache, tables, ctx, scale, ws, err, 2_000_000) == pk.PKV_OK
    torch.cuda.synchronize()                                 # the call came back
    assert err.item() & pk.PKV_DEVERR_TIMEOUT

    for _ in range(2):                                       # and the device is sound
        again = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        cache.attend(q, tables, ctx, scale, out=again)
        torch.cuda.synchronize()
        assert_close(again, want, "bf16")
        assert cache.err.item() == 0
