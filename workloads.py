"""Seeded synthetic inputs for paged decode attention.

This module only draws random numbers and rounds them to the 16-bit storage
formats. It holds none of the method's arithmetic: no block counting, no slot
mapping, no softmax. The oracle-side tests, the CUDA-side tests, ``bench.py``
and the smoke check all take their inputs from here, so that both sides see
identical bits.

Every array of 16-bit values is returned as ``uint16`` bit patterns together
with a dtype tag (``"f16"`` IEEE binary16 or ``"bf16"`` bfloat16).

The five workload shapes follow the decode batches that the PagedAttention
pages measure on (the paper review's "Table 1" setup section: OPT-13B and
LLaMA-13B, chat-style request lengths, beam search / shared prefixes, long
contexts). The pages' own datasets (ShareGPT, Alpaca) are not used: seeded
length distributions stand in for them.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F16_NAN = 0x7E00
BF16_NAN = 0x7FC0
DTYPES = ("f16", "bf16")


def poison_bits(dtype: str) -> int:
    """A quiet-NaN bit pattern of the storage format, used to fill cache slots
    that no token owns: any read of such a slot turns the output into NaN."""
    return F16_NAN if dtype == "f16" else BF16_NAN


def round_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the 16-bit format, round-to-nearest-even.

    Returns uint16 bit patterns. bfloat16 keeps the upper 16 bits of the
    float32 encoding after adding half an ulp (with the tie going to even);
    binary16 uses numpy's own conversion, which is also round-to-nearest-even.
    The inputs never hold NaN.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32).astype(np.uint64)
        lsb = (u >> 16) & 1
        return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def _streams(seed: int, n: int) -> list[np.random.Generator]:
    """Independent generators for the separate draws of one workload, so that
    changing the size of one draw does not shift the others."""
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def normal_bits(rng: np.random.Generator, shape, dtype: str,
                outlier_frac: float = 0.0, outlier_scale: float = 8.0,
                chunk_rows: int = 1 << 16) -> np.ndarray:
    """N(0,1) values rounded to ``dtype``; shape = (rows, heads, dim).

    With ``outlier_frac`` > 0, each (row, head) vector is multiplied by
    ``outlier_scale`` before rounding with that probability (Bernoulli per
    vector). Generated in row chunks to bound host memory.
    """
    rows = shape[0]
    inner = tuple(shape[1:])
    out = np.empty(shape, dtype=np.uint16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = rng.standard_normal((r1 - r0,) + inner, dtype=np.float32)
        if outlier_frac > 0.0:
            hit = rng.random((r1 - r0,) + inner[:1]) < outlier_frac
            x[hit] *= np.float32(outlier_scale)
        out[r0:r1] = round_to_storage(x, dtype)
    return out


def free_order(num_blocks: int, seed: int) -> np.ndarray:
    """Seeded permutation of the physical block ids 0..num_blocks-1.

    It is the initial content of the block manager's free list ("seeded random
    block placement"): the order in which physical blocks are handed out.
    """
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0xB10C]))
    return rng.permutation(num_blocks).astype(np.int32)


@dataclass
class DecodeBatch:
    """One decode step's inputs for a batch of independent sequences.

    ``context_lens[s]`` is the number of tokens sequence ``s`` attends over,
    its newest token included. The keys/values of sequence ``s``'s tokens, in
    position order, are rows ``offsets[s]:offsets[s+1]`` of ``k_tokens`` /
    ``v_tokens`` (shape [total_tokens, num_kv_heads, head_size]); the last row
    of each sequence is the token written in this step.
    """

    name: str
    dtype: str
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    scale: np.float32
    context_lens: np.ndarray
    q: np.ndarray
    k_tokens: np.ndarray
    v_tokens: np.ndarray
    offsets: np.ndarray
    seed: int = 0
    notes: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def total_tokens(self) -> int:
        return int(self.offsets[-1])


def decode_batch(name: str, context_lens, num_heads: int, num_kv_heads: int,
                 head_size: int, block_size: int, dtype: str, seed: int,
                 outlier_frac: float = 0.0) -> DecodeBatch:
    """Draw q, K and V for the given per-sequence context lengths.

    Values are N(0,1) rounded to ``dtype``. Keys may carry outliers (see
    ``normal_bits``). ``scale`` = 1/sqrt(head_size) computed in float32.
    """
    lens = np.asarray(context_lens, dtype=np.int32)
    if lens.ndim != 1 or lens.size == 0 or lens.min() < 1:
        raise ValueError("context lengths must be a non-empty list of positive ints")
    offsets = np.zeros(lens.size + 1, dtype=np.int64)
    np.cumsum(lens, out=offsets[1:])
    g_q, g_k, g_v = _streams(seed, 3)
    q = normal_bits(g_q, (lens.size, num_heads, head_size), dtype)
    k = normal_bits(g_k, (int(offsets[-1]), num_kv_heads, head_size), dtype,
                    outlier_frac=outlier_frac)
    v = normal_bits(g_v, (int(offsets[-1]), num_kv_heads, head_size), dtype)
    scale = np.float32(1.0) / np.sqrt(np.float32(head_size))
    return DecodeBatch(name, dtype, num_heads, num_kv_heads, head_size, block_size,
                       np.float32(scale), lens, q, k, v, offsets, seed)


# --------------------------------------------------------------------------
# The five decode workloads
# --------------------------------------------------------------------------

TINY_LENS = (5, 9, 17, 31)
TINY_POOL_BLOCKS = 64
LONGCTX_LENS_K = (32, 48, 64, 96, 128, 128, 80, 40)
LLAMA_BLOCK_SIZES = (8, 16, 32, 64, 128)


def tiny(seed: int = 0) -> DecodeBatch:
    """4 sequences of lengths {5, 9, 17, 31}; 4 heads = 4 KV heads, head_dim 64,
    block_size 4, fp16; the pool holds 64 physical blocks."""
    return decode_batch("tiny", TINY_LENS, 4, 4, 64, 4, "f16", seed)


def opt13b_lengths(num_seqs: int, seed: int) -> np.ndarray:
    """Chat-style request lengths: lognormal around a median of 600 tokens
    (sigma 0.8), rounded and clipped to [1, 2048]."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x0913]))
    x = rng.lognormal(mean=math.log(600.0), sigma=0.8, size=num_seqs)
    return np.clip(np.rint(x), 1, 2048).astype(np.int32)


def opt13b(seed: int = 0, num_seqs: int = 64) -> DecodeBatch:
    """OPT-13B-shaped decode: 40 heads MHA, head_dim 128, block_size 16, fp16,
    a batch of 64 with lognormal lengths."""
    return decode_batch("opt13b", opt13b_lengths(num_seqs, seed), 40, 40, 128, 16,
                        "f16", seed)


def llama13b_lengths(num_seqs: int, seed: int, max_len: int = 4096) -> np.ndarray:
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x11A3A]))
    return rng.integers(1, max_len, size=num_seqs, endpoint=True).astype(np.int32)


def llama13b(seed: int = 0, block_size: int = 16, num_seqs: int = 128,
             max_len: int = 4096) -> DecodeBatch:
    """LLaMA-13B-shaped decode: 40 heads MHA, head_dim 128, fp16, a batch of
    128 with lengths uniform in [1, 4096]. The token data does not depend on
    ``block_size``, so the block-size sweep sees the same values."""
    return decode_batch(f"llama13b_b{block_size}", llama13b_lengths(num_seqs, seed, max_len),
                        40, 40, 128, block_size, "f16", seed)


def longctx(seed: int = 0, scale_k: int = 1024) -> DecodeBatch:
    """Long-context decode: 32 query heads / 8 KV heads, head_dim 128, bf16,
    block_size 16, lengths {32k, 48k, 64k, 96k, 128k, 128k, 80k, 40k}; 1% of the
    key vectors are scaled x8 before rounding."""
    lens = [n * scale_k for n in LONGCTX_LENS_K]
    return decode_batch("longctx", lens, 32, 8, 128, 16, "bf16", seed, outlier_frac=0.01)


def mqa(seed: int = 0, num_seqs: int = 128) -> DecodeBatch:
    """Multi-query decode: 64 query heads sharing one KV head, head_dim 128,
    bf16, block_size 16, a batch of 128 with lengths uniform in [1, 4096]."""
    return decode_batch("mqa", llama13b_lengths(num_seqs, seed), 64, 1, 128, 16, "bf16", seed)


@dataclass
class SharedPrefixBatch:
    """Beam groups that share a prefix of physical blocks.

    Group ``g`` holds ``prefix_lens[g]`` shared tokens (rows
    ``prefix_offsets[g]:prefix_offsets[g+1]`` of ``prefix_k``/``prefix_v``).
    Beam ``b`` of group ``g`` (sequence index ``g*beams + b``) then appends
    ``tail_lens[g*beams+b]`` tokens of its own (rows of ``tail_k``/``tail_v``)
    and decodes with query ``q[g*beams+b]``.
    """

    name: str
    dtype: str
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    scale: np.float32
    beams: int
    prefix_lens: np.ndarray
    prefix_offsets: np.ndarray
    prefix_k: np.ndarray
    prefix_v: np.ndarray
    tail_lens: np.ndarray
    tail_offsets: np.ndarray
    tail_k: np.ndarray
    tail_v: np.ndarray
    q: np.ndarray
    seed: int = 0

    @property
    def num_groups(self) -> int:
        return int(self.prefix_lens.shape[0])

    @property
    def num_seqs(self) -> int:
        return int(self.tail_lens.shape[0])


def gqa_prefix(seed: int = 0, groups: int = 64, beams: int = 4, prefix_tokens: int = 1024,
               max_partial: int = 15, max_tail: int = 512,
               partial: bool = True) -> SharedPrefixBatch:
    """GQA shared-prefix decode: 32 query heads / 8 KV heads, head_dim 128,
    bf16, block_size 16; ``groups`` groups of ``beams`` beams. Each group shares
    ``prefix_tokens`` + r_g tokens (r_g uniform in [1, max_partial], or 0 when
    ``partial`` is False) and each beam appends a tail of 1..max_tail tokens."""
    H, H_kv, d, B, dtype = 32, 8, 128, 16, "bf16"
    _, g_pk, g_pv, g_tk, g_tv, g_q = _streams(seed, 6)
    prefix_lens, tail_lens = gqa_prefix_lengths(seed, groups, beams, prefix_tokens, max_partial,
                                                max_tail, partial)
    p_off = np.zeros(groups + 1, np.int64)
    np.cumsum(prefix_lens, out=p_off[1:])
    t_off = np.zeros(groups * beams + 1, np.int64)
    np.cumsum(tail_lens, out=t_off[1:])
    pk = normal_bits(g_pk, (int(p_off[-1]), H_kv, d), dtype)
    pv = normal_bits(g_pv, (int(p_off[-1]), H_kv, d), dtype)
    tk = normal_bits(g_tk, (int(t_off[-1]), H_kv, d), dtype)
    tv = normal_bits(g_tv, (int(t_off[-1]), H_kv, d), dtype)
    q = normal_bits(g_q, (groups * beams, H, d), dtype)
    scale = np.float32(1.0) / np.sqrt(np.float32(d))
    return SharedPrefixBatch("gqa_prefix", dtype, H, H_kv, d, B, np.float32(scale), beams,
                             prefix_lens, p_off, pk, pv, tail_lens, t_off, tk, tv, q, seed)


def gqa_prefix_lengths(seed: int = 0, groups: int = 64, beams: int = 4,
                       prefix_tokens: int = 1024, max_partial: int = 15, max_tail: int = 512,
                       partial: bool = True):
    """The shared-prefix workload's lengths alone (the draws ``gqa_prefix``
    makes first, from the same stream): per group the shared tokens
    ``prefix_tokens`` + r_g, per beam its tail length."""
    g_len = _streams(seed, 6)[0]
    r = g_len.integers(1, max_partial, size=groups, endpoint=True) if partial else np.zeros(groups, np.int64)
    prefix_lens = (prefix_tokens + r).astype(np.int32)
    tail_lens = g_len.integers(1, max_tail, size=groups * beams, endpoint=True).astype(np.int32)
    return prefix_lens, tail_lens


def new_tokens(num_seqs: int, num_kv_heads: int, head_size: int, dtype: str,
               seed: int, step: int = 0):
    """Keys and values of one freshly decoded token per sequence, for a decode
    step that appends to the cache: uint16 [num_seqs, num_kv_heads, head_size]."""
    g_k, g_v = _streams(seed * 1_000_003 + step + 17, 2)
    return (normal_bits(g_k, (num_seqs, num_kv_heads, head_size), dtype),
            normal_bits(g_v, (num_seqs, num_kv_heads, head_size), dtype))


def queries(num_seqs: int, num_heads: int, head_size: int, dtype: str, seed: int,
            step: int = 0) -> np.ndarray:
    """Decode queries for one step: uint16 [num_seqs, num_heads, head_size]."""
    (g,) = _streams(seed * 1_000_033 + step + 29, 1)
    return normal_bits(g, (num_seqs, num_heads, head_size), dtype)
