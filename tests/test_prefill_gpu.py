"""Chunked-prefill attention on the GPU against the fp64 oracle: varied chunk
sizes (one token, ragged, several row tiles, the whole prompt), MHA and GQA,
d = 64 / 128, fp16 / bf16, block sizes 8..128, fp32 outputs held to the
stated bound; bad chunk lengths reported."""

import numpy as np
import pytest
import torch

import paged_kv_cache_118_gb300 as pk
from oracle.pipeline import build_decode_state, pool_demand
from oracle.prefill import paged_attention_prefill
from parity import TORCH_DTYPE, assert_close, dev, gpu_decode_state, record_max_err
from workloads import decode_batch, free_order, normal_bits, poison_bits

pytestmark = pytest.mark.gpu

CASES = [
    # lens, chunks, H, H_kv, D, B, dtype
    ((100, 37, 1, 700), (1, 37, 1, 300), 8, 8, 128, 16, "f16"),
    ((513, 64, 2049), (200, 64, 130), 32, 8, 128, 16, "bf16"),
    ((90, 300), (90, 17), 4, 2, 64, 8, "f16"),
    ((1500, 33), (129, 5), 16, 2, 128, 32, "bf16"),
    ((640,), (640,), 64, 1, 64, 128, "bf16"),
    ((77, 400, 9), (3, 65, 9), 40, 40, 128, 64, "f16"),
    # 128 query heads per KV head (one token per query tile), 256-row blocks,
    # and a whole 1000-token prompt over 8-row blocks at d = 128
    ((300, 50), (300, 7), 128, 1, 64, 16, "bf16"),
    ((600, 70), (600, 70), 8, 2, 128, 256, "f16"),
    ((1000,), (1000,), 8, 8, 128, 8, "bf16"),
    # more work items than SMs, so CTAs claim items from the counter and run
    # several in turn: 12 sequences x 16 KV heads x 2 query blocks (MHA,
    # chunks of 0, 1 and up to 300 tokens, so some items are empty), and
    # 4-way GQA over 10 sequences with up to 4 query blocks each
    ((620, 610, 700, 333, 900, 640, 777, 1200, 301, 512, 450, 1000),
     (300, 0, 1, 333, 299, 250, 17, 300, 300, 256, 257, 129), 16, 16, 64, 16, "f16"),
    ((800, 1024, 260, 999, 512, 700, 1300, 257, 640, 900),
     (256, 255, 1, 200, 64, 65, 256, 257, 128, 190), 32, 8, 128, 16, "bf16"),
]


def _run(case, seed=0):
    lens, chunks, H, Hkv, D, B, dt = case
    batch = decode_batch("p", lens, H, Hkv, D, B, dt, seed=seed + len(lens))
    n = pool_demand(batch.context_lens, B) + 9
    order = free_order(n, seed)
    cache, tables, ctx = gpu_decode_state(batch, n, order)
    ref = build_decode_state(batch, n, order, poison_bits(dt))
    starts = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = normal_bits(np.random.default_rng(seed + 99), (int(starts[-1]), H, D), dt)
    want = paged_attention_prefill(q, ref["k_cache"], ref["v_cache"], ref["block_tables"],
                                   batch.context_lens, starts, B, batch.scale, dt)
    qd = dev(q, dt)
    qsd = torch.from_numpy(starts).cuda()
    ws = pk.prefill_workspace()
    for od in (TORCH_DTYPE[dt], torch.float32):
        out = torch.full(qd.shape, float("nan"), dtype=od, device="cuda")
        pk.pkv_paged_attention_prefill(out, qd, cache.k_cache, cache.v_cache, tables, ctx, qsd,
                                       max(chunks), B, float(batch.scale), workspace=ws,
                                       err_flag=cache.err)
        torch.cuda.synchronize()
        err = assert_close(out, want, dt)
        record_max_err(f"prefill {dt} lens={lens} chunks={chunks} H={H}/{Hkv} d={D} B={B} "
                       f"({'fp32' if od == torch.float32 else dt} out)", err)
        if od == torch.float32:
            # the same call again, bit for bit, whichever CTA claims which item
            again = torch.empty_like(out)
            pk.pkv_paged_attention_prefill(again, qd, cache.k_cache, cache.v_cache, tables, ctx,
                                           qsd, max(chunks), B, float(batch.scale),
                                           workspace=ws, err_flag=cache.err)
            torch.cuda.synchronize()
            assert torch.equal(again, out)
    assert cache.err.item() == 0


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_prefill_against_oracle(case):
    _run(case)


def test_bad_chunk_is_reported_and_skipped():
    batch = decode_batch("p", (40, 50), 4, 4, 64, 16, "f16", seed=3)
    n = pool_demand(batch.context_lens, 16) + 2
    cache, tables, ctx = gpu_decode_state(batch, n, free_order(n, 1))
    starts = torch.tensor([0, 10, 70], dtype=torch.int32, device="cuda")   # 60 > L = 50
    q = torch.randn(70, 4, 64, dtype=torch.float16, device="cuda")
    out = torch.zeros_like(q)
    pk.pkv_paged_attention_prefill(out, q, cache.k_cache, cache.v_cache, tables, ctx, starts,
                                   60, 16, 0.125, err_flag=cache.err)
    torch.cuda.synchronize()
    assert cache.err.item() & pk.PKV_DEVERR_CONTEXT
    assert torch.all(out[10:] == 0) and torch.all(torch.isfinite(out[:10]))
    assert not torch.all(out[:10] == 0)


def test_rows_past_the_end_of_q_are_reported_and_skipped():
    """A chunk whose rows would run past the end of q (query_start[s] + C >
    the rows of q) is skipped and reported; the other sequences are computed."""
    batch = decode_batch("p", (40, 100), 4, 4, 64, 16, "f16", seed=3)
    n = pool_demand(batch.context_lens, 16) + 2
    cache, tables, ctx = gpu_decode_state(batch, n, free_order(n, 1))
    starts = torch.tensor([0, 10, 70], dtype=torch.int32, device="cuda")   # 70 > 65 rows
    q = torch.randn(65, 4, 64, dtype=torch.float16, device="cuda")
    out = torch.zeros_like(q)
    pk.pkv_paged_attention_prefill(out, q, cache.k_cache, cache.v_cache, tables, ctx, starts,
                                   60, 16, 0.125, err_flag=cache.err)
    torch.cuda.synchronize()
    assert cache.err.item() & pk.PKV_DEVERR_CONTEXT
    assert torch.all(out[10:] == 0) and torch.all(torch.isfinite(out[:10]))
    assert not torch.all(out[:10] == 0)


@pytest.mark.parametrize("od", [torch.float16, torch.float32])
def test_output_aligned_to_16_bytes_only(od):
    """An output 16-byte but not 32-byte aligned takes the 16-byte stores: the
    same values, bit for bit, as a 32-byte aligned output."""
    batch = decode_batch("p", (300, 129), 8, 2, 128, 16, "f16", seed=5)
    n = pool_demand(batch.context_lens, 16) + 2
    cache, tables, ctx = gpu_decode_state(batch, n, free_order(n, 2))
    starts = torch.tensor([0, 100, 229], dtype=torch.int32, device="cuda")
    q = torch.randn(229, 8, 128, dtype=torch.float16, device="cuda")
    aligned = torch.empty(q.shape, dtype=od, device="cuda")
    pad = 16 // aligned.element_size()
    big = torch.empty(aligned.numel() + pad, dtype=od, device="cuda")
    shifted = big[pad:].view(q.shape)
    assert shifted.data_ptr() % 16 == 0 and shifted.data_ptr() % 32 != 0
    for out in (aligned, shifted):
        pk.pkv_paged_attention_prefill(out, q, cache.k_cache, cache.v_cache, tables, ctx, starts,
                                       129, 16, float(batch.scale), err_flag=cache.err)
    torch.cuda.synchronize()
    assert cache.err.item() == 0
    assert torch.equal(aligned, shifted)
