"""Shared pieces of the GPU parity tests: moving the generator's bit patterns
to the device, running a decode step through the library, and the tolerance.

Tolerance (attention outputs): the kernels accumulate in fp32; the stated
bound is a max-abs error of 2e-3 (fp16) / 8e-3 (bf16) against the fp64
oracle. An fp32 output is held to that bound as it is. An output rounded to
fp16/bf16 also carries the rounding of the result itself, up to half an ulp
of the format at the value's magnitude, which for bf16 outputs above 2 alone
exceeds 8e-3; so those are held to bound + half an ulp of |oracle|.
"""

import numpy as np
import torch

from paged_kv_cache_118_gb300.cache import PagedKVCache

TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}
BOUND = {"f16": 2e-3, "bf16": 8e-3}
MANT = {torch.float16: (10, -14), torch.bfloat16: (7, -126)}


def dev(bits: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        TORCH_DTYPE[dtype]).cuda()


def half_ulp(x: np.ndarray, tdtype) -> np.ndarray:
    mant, emin = MANT[tdtype]
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** emin)))
    return 0.5 * np.exp2(e - mant)


def assert_close(gpu: torch.Tensor, ref: np.ndarray, dtype: str):
    """Element-wise check of a GPU attention output against the oracle."""
    got = gpu.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape
    mask = ~np.isnan(ref)
    assert np.all(np.isfinite(got[mask])), "non-finite output"
    err = np.abs(got - ref)[mask]
    tol = BOUND[dtype] + (0.0 if gpu.dtype == torch.float32 else half_ulp(ref, gpu.dtype)[mask])
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} elements off, max err {err.max():.3e}"
    return float(err.max()) if err.size else 0.0


def gpu_decode_state(batch, num_blocks, order, poison=True):
    """Prefill L-1 tokens per sequence, append the newest token of each, build
    the device tables — all through the library (block manager + kernels)."""
    cache = PagedKVCache(num_blocks, batch.block_size, batch.num_kv_heads, batch.head_size,
                         TORCH_DTYPE[batch.dtype], free_order=order, poison=poison)
    S = batch.num_seqs
    lens = batch.context_lens.astype(np.int64)
    last = batch.offsets[1:] - 1
    keep = np.ones(batch.total_tokens, bool)
    keep[last] = False
    cache.prefill(range(S), lens - 1, dev(batch.k_tokens[keep], batch.dtype),
                  dev(batch.v_tokens[keep], batch.dtype))
    cache.append(list(range(S)), dev(batch.k_tokens[last], batch.dtype),
                 dev(batch.v_tokens[last], batch.dtype))
    tables, ctx = cache.tables(range(S))
    return cache, tables, ctx


def sub_batch(batch, s):
    """Sequence s of a DecodeBatch as a batch of its own (same bits)."""
    from workloads import DecodeBatch
    a, b = int(batch.offsets[s]), int(batch.offsets[s + 1])
    return DecodeBatch(batch.name, batch.dtype, batch.num_heads, batch.num_kv_heads,
                       batch.head_size, batch.block_size, batch.scale,
                       batch.context_lens[s:s + 1].copy(), batch.q[s:s + 1],
                       batch.k_tokens[a:b], batch.v_tokens[a:b],
                       np.array([0, b - a], np.int64), batch.seed)


def oracle_sampled(batch, seqs):
    """Oracle outputs [H, D] for the sampled sequences, each computed from a
    pool of its own (placement does not change the result)."""
    from oracle.attention import paged_attention_decode
    from oracle.pipeline import build_decode_state, pool_demand
    from workloads import free_order, poison_bits
    out = {}
    for s in seqs:
        sb = sub_batch(batch, s)
        n = pool_demand(sb.context_lens, sb.block_size) + 2
        st = build_decode_state(sb, n, free_order(n, s), poison_bits(sb.dtype))
        out[s] = paged_attention_decode(sb.q, st["k_cache"], st["v_cache"], st["block_tables"],
                                        sb.context_lens, sb.block_size, sb.scale, sb.dtype)[0]
    return out


def _available_bytes() -> int:
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 16 << 30


def oracle_all(batch, seqs=None, max_workers=8):
    """Oracle outputs [H, D] of every sequence (or of ``seqs``), each computed
    from a pool of its own, by a pool of threads (numpy's array operations
    release the interpreter lock). The number of threads is bounded by host
    memory: the oracle widens a sequence's keys and values to float64, with
    temporaries of about eight times their element count each."""
    import concurrent.futures as cf
    seqs = list(range(batch.num_seqs)) if seqs is None else list(seqs)
    longest = int(max(batch.context_lens[s] for s in seqs))
    per_seq = longest * batch.num_kv_heads * batch.head_size * 8 * 8 * 2
    workers = max(1, min(max_workers, len(seqs), _available_bytes() // 2 // max(per_seq, 1)))
    out = {}
    with cf.ThreadPoolExecutor(workers) as ex:
        for part in ex.map(lambda s: oracle_sampled(batch, [s]), seqs):
            out.update(part)
    return out


def stack_oracle(want: dict, seqs) -> np.ndarray:
    return np.stack([want[s] for s in seqs])


def record_max_err(name: str, err: float) -> None:
    """Keep the largest error seen per check; written as JSON to the path in
    PKV_PARITY_REPORT (if set) so that a run can report it."""
    import json
    import os
    RECORDED[name] = max(err, RECORDED.get(name, 0.0))
    path = os.environ.get("PKV_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump(RECORDED, f, indent=1, sort_keys=True)


RECORDED: dict = {}


def sample_seqs(lens, k, seed):
    """Shortest, longest, median and k-3 seeded others."""
    order = np.argsort(lens, kind="stable")
    pick = {int(order[0]), int(order[-1]), int(order[len(order) // 2])}
    rng = np.random.default_rng(seed)
    while len(pick) < min(k, len(lens)):
        pick.add(int(rng.integers(len(lens))))
    return sorted(pick)
