"""Cache writes of the decode step (oracle; test infrastructure only).

* reshape_and_cache — each new token's key and value go to its slot: physical
  block slot // B, row slot % B. The pages only say that a new token is written
  into the sequence's tail block ("079｜vLLM 与 PagedAttention", wq-win.github.io,
  §2 "共享与写时复制" and the §3 per-iteration algorithm box); the slot number
  is block_table[p // B] * B + p % B for position p. A negative slot means
  "no write" (padding).
* copy_blocks — copy-on-write: before a sequence writes into a block that
  another sequence still references, the block's keys and values are copied to
  a fresh block and only this branch's table is remapped (same review, §2
  "共享与写时复制" and "一次分叉什么时候真的要复制缓存块"; "vLLM 推理引擎"
  gitcode.csdn.net overview of Copy-on-Write).

* swap_blocks — the copies of a swap: block src of one pool (K and V) becomes
  block dst of another pool ("079｜vLLM 与 PagedAttention" §3 algorithm box;
  "PagedAttention 内存管理深度解析", "Swap 机制").

All are bitwise copies, written as plain loops.
"""

import numpy as np


def reshape_and_cache(k: np.ndarray, v: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                      slot_mapping: np.ndarray) -> None:
    """In place: k_cache[slot // B, slot % B] = k[t] (same for v) for every token t.

    k, v: [num_tokens, H_kv, d]; caches: [num_blocks, B, H_kv, d]; slot_mapping:
    int64 [num_tokens]. Raises IndexError for a slot past the pool.
    """
    block_size = k_cache.shape[1]
    capacity = k_cache.shape[0] * block_size
    for t in range(k.shape[0]):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        if slot >= capacity:
            raise IndexError(f"slot {slot} outside a pool of {capacity} slots")
        blk, row = divmod(slot, block_size)
        k_cache[blk, row] = k[t]
        v_cache[blk, row] = v[t]


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, pairs) -> None:
    """In place: for each (src, dst), block dst of both caches becomes a copy of
    block src. No dst may appear twice, and no dst may also be a src."""
    pairs = [(int(s), int(d)) for s, d in pairs]
    dsts = [d for _, d in pairs]
    if len(set(dsts)) != len(dsts) or set(dsts) & {s for s, _ in pairs}:
        raise ValueError("copy_blocks pairs overlap")
    snapshot_k = {s: k_cache[s].copy() for s, _ in pairs}
    snapshot_v = {s: v_cache[s].copy() for s, _ in pairs}
    for src, dst in pairs:
        k_cache[dst] = snapshot_k[src]
        v_cache[dst] = snapshot_v[src]


def swap_blocks(src_k: np.ndarray, src_v: np.ndarray, dst_k: np.ndarray, dst_v: np.ndarray,
                pairs) -> None:
    """In place: dst pool block d becomes a copy of src pool block s for each
    (s, d). Destinations must be distinct."""
    pairs = [(int(s), int(d)) for s, d in pairs]
    if len({d for _, d in pairs}) != len(pairs):
        raise ValueError("swap destinations repeat")
    for s, d in pairs:
        dst_k[d] = src_k[s]
        dst_v[d] = src_v[s]
