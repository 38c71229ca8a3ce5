"""Paged chunked-prefill attention in float64 (oracle; test infrastructure only).

What it computes: a sequence with L tokens in its cache receives a chunk of C
new query tokens, the last C of the L (their keys and values are already
written). Query i of the chunk sits at position p_i = L - C + i and attends over
positions 0..p_i of its own sequence, with one softmax denominator:

    o_i = sum_{u <= p_i} exp(s_u) v_u / sum_{u <= p_i} exp(s_u),   s_u = scale * q_i . k_u

(chunked prefill: zhy-blog.vercel.app §4 — a long prompt is split into chunks
processed in order, each chunk's mask set by its position in the prompt and
attending to the cache the earlier chunks left; "079｜vLLM 与 PagedAttention"
§3 algorithm box — prefill for new prompts, paged attention over the cache).
Decode is the case C = 1. Keys are read through the block table as in
``attention.gather_sequence``; query head h reads KV head floor(h / (H/H_kv)).

Queries of all sequences are packed: rows query_start[s] .. query_start[s+1]-1
of ``q`` ([total_queries, H, d]) belong to sequence s.
"""

import numpy as np

from .attention import gather_sequence, kv_head_of, softmax_weights
from .formats import decode_bits


def causal_visibility(context_len: int, chunk: int) -> np.ndarray:
    """[C, L] booleans: query i (position L - C + i) sees key positions <= its own."""
    pos = context_len - chunk + np.arange(chunk)
    return np.arange(context_len)[None, :] <= pos[:, None]


def prefill_sequence(q_bits: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                     table_row: np.ndarray, context_len: int, block_size: int, scale: float,
                     dtype: str) -> np.ndarray:
    """One sequence's chunk: q [C, H, d] bits -> o [C, H, d] float64."""
    C, H, _ = q_bits.shape
    L = int(context_len)
    if C < 1 or C > L:
        raise ValueError("a chunk holds 1..L of the sequence's last tokens")
    Hkv = k_cache.shape[2]
    K = decode_bits(gather_sequence(k_cache, table_row, L, block_size), dtype)
    V = decode_bits(gather_sequence(v_cache, table_row, L, block_size), dtype)
    Q = decode_bits(q_bits, dtype)
    s64 = float(np.float32(scale))
    visible = causal_visibility(L, C)                          # [C, L]
    out = np.empty(Q.shape, dtype=np.float64)
    for h in range(H):
        g = kv_head_of(h, H, Hkv)
        scores = s64 * (Q[:, h, :] @ K[:, g, :].T)              # [C, L]
        scores = np.where(visible, scores, -np.inf)
        out[:, h, :] = softmax_weights(scores) @ V[:, g, :]
    return out


def paged_attention_prefill(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                            block_tables: np.ndarray, context_lens: np.ndarray,
                            query_start: np.ndarray, block_size: int, scale: float,
                            dtype: str, seqs=None) -> np.ndarray:
    """Chunked prefill for a batch: out [total_queries, H, d] float64 (rows of
    sequences not in ``seqs`` are NaN when ``seqs`` is given)."""
    out = np.full(q.shape, np.nan, dtype=np.float64)
    for s in (range(len(context_lens)) if seqs is None else seqs):
        a, b = int(query_start[s]), int(query_start[s + 1])
        if b > a:
            out[a:b] = prefill_sequence(q[a:b], k_cache, v_cache, block_tables[s],
                                        int(context_lens[s]), block_size, scale, dtype)
    return out
