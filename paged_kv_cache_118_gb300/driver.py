"""Host decode-step driver: the per-iteration loop of the method without a model.

Follows the algorithm box of "079｜vLLM 与 PagedAttention" (wq-win.github.io,
§3), one iteration per `step()`:

  1. drop finished sequences (their block references go; blocks whose count
     reaches zero are reclaimed, or kept evictable in the prefix cache);
  2. resume preempted sequences whose blocks fit again (swap in);
  3. admit waiting requests that fit, reusing cached prompt blocks (prefix
     cache, zhy-blog.vercel.app §2.2(5)) and writing only the uncached tokens;
  4. make room for every running sequence's next token; when blocks run short,
     preempt the most recently admitted sequence by swapping it out to the CPU
     pool (§3: "swap out"; recomputation needs a model and is not modelled);
  5. append (new blocks, copy-on-write of shared tails), write the new keys and
     values, and run paged attention for the running sequences.

Keys, values and queries come from the caller (``kv_source(seq, positions)`` ->
(k, v) device tensors [n, H_kv, D]; ``q_source(seq, position)`` -> [H, D]),
standing in for a model's projections. Every GPU step is a call through the C
ABI; the bookkeeping here is host logic only.
"""

from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field

import numpy as np
import torch

from . import BlockManager, PagedKVError, PKV_ENOMEM, pkv_swap_blocks
from .cache import PagedKVCache


@dataclass
class Request:
    seq: int
    prompt: list
    max_new_tokens: int
    generated: int = 0
    admitted_at: int = -1

    @property
    def length(self) -> int:
        return len(self.prompt) + self.generated


@dataclass
class StepResult:
    seqs: list = field(default_factory=list)      # running sequences attended this step
    out: torch.Tensor | None = None               # [len(seqs), H, D]
    context_lens: list = field(default_factory=list)
    admitted: list = field(default_factory=list)
    cached_tokens: dict = field(default_factory=dict)
    preempted: list = field(default_factory=list)
    resumed: list = field(default_factory=list)
    finished: list = field(default_factory=list)
    cow_pairs: int = 0


class DecodeLoop:
    def __init__(self, num_gpu_blocks: int, num_cpu_blocks: int, block_size: int,
                 num_heads: int, num_kv_heads: int, head_size: int, dtype, scale: float,
                 kv_source, q_source, device="cuda"):
        self.gpu = PagedKVCache(num_gpu_blocks, block_size, num_kv_heads, head_size, dtype,
                                device)
        self.cpu_bm = BlockManager(num_cpu_blocks, block_size)
        shape = (num_cpu_blocks, block_size, num_kv_heads, head_size)
        self.cpu_k = torch.empty(shape, dtype=dtype).pin_memory()
        self.cpu_v = torch.empty(shape, dtype=dtype).pin_memory()
        self.B, self.H, self.D, self.scale = block_size, num_heads, head_size, scale
        self.kv_source, self.q_source = kv_source, q_source
        self.waiting: deque[Request] = deque()
        self.running: list[Request] = []
        self.swapped: deque[Request] = deque()
        self.t = 0

    def add_request(self, seq: int, prompt, max_new_tokens: int) -> None:
        self.waiting.append(Request(int(seq), list(prompt), int(max_new_tokens)))

    def idle(self) -> bool:
        return not (self.waiting or self.running or self.swapped)

    # -- helpers -----------------------------------------------------------
    def _blocks(self, n: int) -> int:
        return -(-n // self.B)

    def _room_for_next(self, reqs) -> int:
        """Blocks the next token of each request can take (a new block at a
        block boundary; a shared tail may need one more for copy-on-write)."""
        need = 0
        for r in reqs:
            L = self.gpu.bm.length(r.seq)
            if L % self.B == 0:
                need += 1
            else:
                tail = self.gpu.bm.table(r.seq)[L // self.B]
                need += self.gpu.bm.refcount(tail) > 1
        return need

    def _swap_out(self, r: Request) -> None:
        pairs = self.gpu.bm.swap([r.seq], self.cpu_bm)
        pkv_swap_blocks(self.cpu_k, self.cpu_v, self.gpu.k_cache, self.gpu.v_cache, pairs)
        self.running.remove(r)
        self.swapped.append(r)

    def _swap_in(self, r: Request) -> None:
        pairs = self.cpu_bm.swap([r.seq], self.gpu.bm)
        pkv_swap_blocks(self.gpu.k_cache, self.gpu.v_cache, self.cpu_k, self.cpu_v, pairs)
        self.running.append(r)

    # -- one iteration -----------------------------------------------------
    def step(self) -> StepResult:
        res = StepResult()
        # 1. finished sequences leave
        for r in [r for r in self.running if r.generated >= r.max_new_tokens]:
            self.gpu.free(r.seq)
            self.running.remove(r)
            res.finished.append(r.seq)
        # 2. resume preempted sequences, oldest first, while their blocks fit
        while self.swapped:
            r = self.swapped[0]
            if self._blocks(r.length) + 1 > self.gpu.bm.num_free() - self._room_for_next(self.running):
                break
            self.swapped.popleft()
            self._swap_in(r)
            res.resumed.append(r.seq)
        # 3. admit waiting requests that fit, through the prefix cache
        while self.waiting and not self.swapped:
            r = self.waiting[0]
            spare = self.gpu.bm.num_free() - self._room_for_next(self.running)
            if self._blocks(len(r.prompt)) + 1 > spare:
                break
            self.waiting.popleft()
            cached = self.gpu.bm.allocate_prefix(r.seq, r.prompt)
            if cached < len(r.prompt):
                pos = np.arange(cached, len(r.prompt))
                k, v = self.kv_source(r.seq, pos)
                slots = self.gpu.bm.slots(r.seq, cached, len(pos))
                from . import pkv_reshape_and_cache
                pkv_reshape_and_cache(k, v, self.gpu.k_cache, self.gpu.v_cache,
                                      self.gpu._upload(slots), self.gpu.err)
            r.admitted_at = self.t
            self.running.append(r)
            res.admitted.append(r.seq)
            res.cached_tokens[r.seq] = cached
        # 4. room for the next token of every running sequence; preempt if short
        while self.running and self._room_for_next(self.running) > self.gpu.bm.num_free():
            victim = max(self.running, key=lambda x: (x.admitted_at, x.seq))
            self._swap_out(victim)
            res.preempted.append(victim.seq)
        if not self.running:
            self.t += 1
            return res
        # 5. append, copy-on-write, write the new token, attend
        seqs = [r.seq for r in self.running]
        pos = [r.length for r in self.running]
        kv = [self.kv_source(s, np.array([p])) for s, p in zip(seqs, pos)]
        k = torch.cat([a for a, _ in kv])
        v = torch.cat([b for _, b in kv])
        try:
            _, cow = self.gpu.append(seqs, k, v)
        except PagedKVError as e:            # cannot happen after step 4
            if e.status == PKV_ENOMEM:
                raise RuntimeError("block accounting out of step") from e
            raise
        for r in self.running:
            r.generated += 1
        q = torch.stack([self.q_source(s, p) for s, p in zip(seqs, pos)])
        tables, ctx = self.gpu.tables(seqs)
        res.out = self.gpu.attend(q, tables, ctx, self.scale)
        res.seqs, res.context_lens, res.cow_pairs = seqs, [p + 1 for p in pos], len(cow)
        self.t += 1
        return res
