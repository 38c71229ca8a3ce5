"""A paged KV cache on one GPU and the host steps of a decode iteration.

Holds the two block pools (torch device memory), the library's host block
manager and small pinned staging buffers, and issues the library calls of one
decode iteration in the order of the per-iteration algorithm box of
"079｜vLLM 与 PagedAttention" (wq-win.github.io, §3): room for the next token
(new block, or copy-on-write of a shared tail) → copy_blocks → write the new
keys/values (reshape_and_cache) → paged attention. Nothing here computes: every
step is a call through the C ABI.
"""

from __future__ import annotations

import numpy as np
import torch

from . import (BlockManager, decode_workspace, pkv_copy_blocks, pkv_paged_attention_decode,
               pkv_reshape_and_cache)

_NAN_BITS = {torch.float16: 0x7E00, torch.bfloat16: 0x7FC0}


class PagedKVCache:
    def __init__(self, num_blocks: int, block_size: int, num_kv_heads: int, head_size: int,
                 dtype=torch.float16, device="cuda", free_order=None, poison: bool = True):
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.num_kv_heads, self.head_size = int(num_kv_heads), int(head_size)
        self.dtype, self.device = dtype, torch.device(device)
        shape = (num_blocks, block_size, num_kv_heads, head_size)
        self.k_cache = torch.empty(shape, dtype=dtype, device=self.device)
        self.v_cache = torch.empty(shape, dtype=dtype, device=self.device)
        if poison:   # slots no token owns read as NaN
            for c in (self.k_cache, self.v_cache):
                c.view(torch.int16).fill_(_NAN_BITS[dtype])
        self.bm = BlockManager(num_blocks, block_size, free_order)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        self._ws = None

    # ---- host -> device staging ------------------------------------------------
    def _upload(self, arr: np.ndarray) -> torch.Tensor:
        host = torch.from_numpy(np.ascontiguousarray(arr)).pin_memory()
        return host.to(self.device, non_blocking=True)

    # ---- sequence lifecycle --------------------------------------------------
    def prefill(self, seqs, lens, k: torch.Tensor, v: torch.Tensor) -> None:
        """New sequences seqs[i] holding lens[i] tokens whose keys/values are
        consecutive rows of k, v ([sum(lens), H_kv, D], device)."""
        slots = []
        for s, n in zip(seqs, lens):
            self.bm.allocate(int(s), int(n))
            if n:
                slots.append(self.bm.slots(int(s)))
        if slots:
            sl = self._upload(np.concatenate(slots))
            pkv_reshape_and_cache(k, v, self.k_cache, self.v_cache, sl, self.err)

    def fork(self, parent: int, child: int) -> None:
        self.bm.fork(parent, child)

    def append(self, seqs, k: torch.Tensor, v: torch.Tensor):
        """One new token per entry of seqs (rows of k, v, [n, H_kv, D]): make
        room (copy-on-write where a tail is shared), copy, write. Returns the
        (slots, cow_pairs) the block manager produced."""
        slots, cow = self.bm.append_slots(seqs)
        if len(cow):
            pkv_copy_blocks(self.k_cache, self.v_cache, cow)
        pkv_reshape_and_cache(k, v, self.k_cache, self.v_cache, self._upload(slots), self.err)
        return slots, cow

    def free(self, seq: int) -> None:
        self.bm.free_seq(seq)

    # ---- attention -------------------------------------------------------------
    def tables(self, seqs, width: int | None = None):
        """Device block tables (int32, padded with -1) and context lengths."""
        if width is None:
            width = max(1, max(-(-self.bm.length(int(s)) // self.block_size) for s in seqs))
        tab, lens = self.bm.fill_tables(seqs, width)
        return self._upload(tab), self._upload(lens)

    def workspace(self, num_seqs, num_heads, max_blocks, partition_tokens=0) -> torch.Tensor:
        from . import pkv_decode_workspace_size
        need = pkv_decode_workspace_size(num_seqs, num_heads, self.num_kv_heads, self.head_size,
                                         max_blocks, self.block_size, partition_tokens)
        if self._ws is None or self._ws.numel() < need:
            self._ws = decode_workspace(num_seqs, num_heads, self.num_kv_heads, self.head_size,
                                        max_blocks, self.block_size, partition_tokens,
                                        self.device)
        return self._ws

    def attend(self, q: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
               scale: float, out: torch.Tensor | None = None, partition_tokens: int = 0):
        if out is None:
            out = torch.empty_like(q)
        ws = self.workspace(q.shape[0], q.shape[1], block_tables.shape[1], partition_tokens)
        pkv_paged_attention_decode(out, q, self.k_cache, self.v_cache, block_tables,
                                   context_lens, self.block_size, scale, ws, partition_tokens,
                                   self.err)
        return out
