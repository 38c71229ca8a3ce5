"""Paged decode attention in float64 (oracle; test infrastructure only).

What it computes — single-query attention of each sequence over its whole
cached history, with one softmax denominator shared by all blocks:

    Z = sum_j sum_{u in S_j} exp(s_u),   o = sum_j sum_{u in S_j} exp(s_u) v_u / Z,
    s_u = scale * q . k_u

("079｜vLLM 与 PagedAttention" review of Kwon et al. 2023, wq-win.github.io, §2,
sub-section "分块以后，注意力仍需对整个历史归一化": S_j is the set of valid
positions of block j; every block shares the global denominator; the last,
partly filled block's empty positions are masked; the kernel reads blocks
through the block table in the sequence's own order.)

How: the plain definition, in the gather-then-attend shape of the
``PagedAttention.forward`` walk-through on "vLLM 推理引擎：PagedAttention 与
KVCache 管理" (gitcode.csdn.net, §3 "PagedAttention 核心算法"): take the first
ceil(L/B) entries of the sequence's block table, gather those physical blocks,
flatten them to token rows, keep the first L rows (this drops the unfilled
tail of the last block), then evaluate the softmax over all L scores at once
with the maximum subtracted (the stable evaluation of the same quotient).

Readings where the pages are silent (each listed in the design notes):
* the newest token is part of the context: ``context_lens[s]`` counts it;
* query head h reads KV head floor(h / (H / H_kv)) (grouped-query attention
  with contiguous groups);
* ``scale`` is the float32 the caller passes, widened exactly to float64;
* the cache layout is [num_blocks, block_size, num_kv_heads, head_size] and
  ``q`` is [num_seqs, num_heads, head_size], as in the walk-through's comments.
"""

import numpy as np

from .formats import decode_bits


def blocks_for(context_len: int, block_size: int) -> int:
    """Number of blocks that hold ``context_len`` tokens: ceil(L / B)."""
    return -(-int(context_len) // int(block_size))


def kv_head_of(h: int, num_heads: int, num_kv_heads: int) -> int:
    """KV head read by query head ``h``: contiguous groups of H / H_kv heads."""
    return h // (num_heads // num_kv_heads)


def gather_sequence(cache_bits: np.ndarray, table_row: np.ndarray, context_len: int,
                    block_size: int) -> np.ndarray:
    """The sequence's cached rows in position order: [L, H_kv, d] (uint16 bits).

    Only the first ceil(L/B) table entries are read; each must name a physical
    block of the pool.
    """
    n = blocks_for(context_len, block_size)
    ids = np.asarray(table_row[:n], dtype=np.int64)
    if ids.size != n or ids.min() < 0 or ids.max() >= cache_bits.shape[0]:
        raise IndexError("block table entry outside the pool")
    blocks = cache_bits[ids]                      # [n, B, H_kv, d]
    rows = blocks.reshape(n * block_size, *cache_bits.shape[2:])
    return rows[:context_len]


def softmax_weights(scores: np.ndarray) -> np.ndarray:
    """exp(s_u) / sum_u exp(s_u) over the last axis, evaluated with the maximum
    subtracted (the quotient is unchanged)."""
    m = scores.max(axis=-1, keepdims=True)
    e = np.exp(scores - m)
    return e / e.sum(axis=-1, keepdims=True)


def attend_sequence(q_bits: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                    table_row: np.ndarray, context_len: int, block_size: int,
                    scale: float, dtype: str) -> np.ndarray:
    """Decode attention of one sequence: q [H, d] bits -> o [H, d] float64."""
    num_heads = q_bits.shape[0]
    num_kv_heads = k_cache.shape[2]
    K = decode_bits(gather_sequence(k_cache, table_row, context_len, block_size), dtype)
    V = decode_bits(gather_sequence(v_cache, table_row, context_len, block_size), dtype)
    Q = decode_bits(q_bits, dtype)
    s64 = float(np.float32(scale))
    out = np.empty((num_heads, Q.shape[1]), dtype=np.float64)
    for h in range(num_heads):
        g = kv_head_of(h, num_heads, num_kv_heads)
        scores = s64 * (K[:, g, :] @ Q[h])        # [L]
        w = softmax_weights(scores)
        out[h] = w @ V[:, g, :]
    return out


def paged_attention_decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                           block_tables: np.ndarray, context_lens: np.ndarray,
                           block_size: int, scale: float, dtype: str,
                           seqs=None) -> np.ndarray:
    """Decode attention of a batch: out[s, h, :] in float64.

    q: uint16 [S, H, d]; k_cache, v_cache: uint16 [num_blocks, B, H_kv, d];
    block_tables: int32 [S, max_blocks] (entries past ceil(L/B) are ignored);
    context_lens: int32 [S]. With ``seqs`` given, only those rows are computed
    and the others are NaN (for sampled checks of large batches).
    """
    S, H, d = q.shape
    if k_cache.shape[1] != block_size or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape does not match block_size")
    if H % k_cache.shape[2] != 0:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    out = np.full((S, H, d), np.nan, dtype=np.float64)
    for s in (range(S) if seqs is None else seqs):
        L = int(context_lens[s])
        if L < 1:
            raise ValueError("a decode query attends over at least one token")
        out[s] = attend_sequence(q[s], k_cache, v_cache, block_tables[s], L,
                                 block_size, scale, dtype)
    return out
