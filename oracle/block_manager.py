"""Block manager of the paged KV cache (oracle; test infrastructure only).

Sources, in the order the rules are taken from them:

* free list: "PagedAttention 内存管理深度解析" (deepinsea.top), "分页机制设计"
  BlockManager sketch — the free list starts as the list of all block ids, a
  request takes ceil(n/B) blocks by popping from the end, fails without side
  effects when too few are free, and its blocks are appended back on release.
  Here the initial list may be a seeded permutation ("seeded random block
  placement"); popping from the end stays the rule.
* reference counts, fork and copy-on-write: "079｜vLLM 与 PagedAttention"
  (wq-win.github.io), §2 "共享与写时复制" (each physical block carries a
  reference count; a branch that must write into a tail block still referenced
  by others first copies it and remaps only its own table; a block is reclaimed
  only when its count reaches zero), §2 "一次分叉什么时候真的要复制缓存块"
  (full blocks stay shared; only the partly filled tail is ever copied) and the
  §3 per-iteration algorithm box (check whether the next token needs a new
  block; copy a shared tail before writing).
* tail waste: same review, §2 "块大小决定有多少无法借给别人的尾部空间":
  a sequence of L tokens holds B*ceil(L/B) slots.
* swapping: same review, §3 algorithm box (when memory runs short, preempt a
  sequence group and swap its cache out; on resumption swap it back in) and
  zhy-blog.vercel.app §3.3 (the swapped queue holds requests whose KV blocks
  moved to CPU memory); "PagedAttention 内存管理深度解析" (deepinsea.top),
  "Swap 机制" (a CPU swap space of blocks). A swap moves a group of sequences
  from one pool's manager to another's: every distinct block they reference is
  given one block in the destination (blocks shared inside the group stay
  shared), the sequences leave the source, and the (source, destination) block
  pairs to copy come back in order of first reference.

* prefix caching: zhy-blog.vercel.app §2.2(5) — every KV block is kept in a
  hash table keyed by a hash of the block's tokens and all the tokens before
  it; a new request looks its prefix up and reuses the blocks it finds.
  Readings: only full blocks of a prompt are registered (a partial tail will
  be written to and is never shared); reuse stops at the first miss (a later
  block's KV needs every block before it); a registered block whose count
  drops to zero stays cached and evictable, least recently freed first, until
  a fresh allocation finds the free list empty; the hash is 64-bit FNV-1a
  (offset basis 14695981039346656037, prime 1099511628211, over bytes) of the
  previous block's hash (8 bytes, little-endian) followed by the block's token
  ids (4 bytes each, little-endian), the first block's "previous hash" being 0.

Readings (listed in the design notes): when several sequences share a tail and
append in turn, each writer that still sees a count above one takes a copy;
the last one (count one) writes in place. Freed blocks go back to the free list
in the sequence's logical order. The GPU/CPU fallback allocation of the
gitcode.csdn.net sketch is not the method (swap is a preemption path) and is
not modelled: running out of blocks is an error.
"""

from __future__ import annotations


class OutOfBlocks(RuntimeError):
    """Too few free blocks; nothing was changed."""


class BlockManagerStateError(RuntimeError):
    """Unknown or duplicate sequence id, or a bad block id."""


FNV_OFFSET = 14695981039346656037
FNV_PRIME = 1099511628211
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes, h: int = FNV_OFFSET) -> int:
    """64-bit FNV-1a: for every byte, xor it in, then multiply by the prime."""
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & MASK64
    return h


def block_hashes(token_ids, block_size: int) -> list[int]:
    """Chained hashes of the full blocks of a token sequence."""
    out, prev = [], 0
    for j in range(len(token_ids) // block_size):
        data = prev.to_bytes(8, "little") + b"".join(
            int(t).to_bytes(4, "little", signed=True)
            for t in token_ids[j * block_size:(j + 1) * block_size])
        prev = fnv1a64(data)
        out.append(prev)
    return out


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if num_blocks < 1 or block_size < 1:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = range(num_blocks) if free_order is None else [int(x) for x in free_order]
        self.free = list(order)
        if sorted(self.free) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of 0..num_blocks-1")
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}
        self.cached: dict[int, int] = {}      # block hash -> block
        self.hash_of: dict[int, int] = {}     # block -> its registered hash
        self.evictable: list[int] = []        # cached blocks with count 0, oldest first

    # -- queries ---------------------------------------------------------
    def blocks_needed(self, num_tokens: int) -> int:
        return -(-int(num_tokens) // self.block_size)

    def num_free(self) -> int:
        """Blocks an allocation can take: the free list and evictable cached blocks."""
        return len(self.free) + len(self.evictable)

    def _take(self) -> int:
        """A fresh block: from the free list, else the least recently freed cached one."""
        if self.free:
            b = self.free.pop()
        else:
            b = self.evictable.pop(0)
            del self.cached[self.hash_of.pop(b)]
        self.ref[b] = 1
        return b

    def table(self, seq: int) -> list[int]:
        self._known(seq)
        return list(self.tables[seq])

    def length(self, seq: int) -> int:
        self._known(seq)
        return self.lens[seq]

    def slot(self, seq: int, pos: int) -> int:
        """Physical slot of position ``pos``: table[pos // B] * B + pos % B."""
        t = self.tables[seq]
        return t[pos // self.block_size] * self.block_size + pos % self.block_size

    def slots(self, seq: int) -> list[int]:
        return [self.slot(seq, p) for p in range(self.lens[seq])]

    # -- operations ------------------------------------------------------
    def allocate(self, seq: int, num_tokens: int) -> list[int]:
        """Give a new sequence room for ``num_tokens`` tokens."""
        if seq in self.tables:
            raise BlockManagerStateError(f"sequence {seq} already allocated")
        if num_tokens < 0:
            raise ValueError("negative token count")
        need = self.blocks_needed(num_tokens)
        if need > self.num_free():
            raise OutOfBlocks(f"need {need} blocks, {self.num_free()} free")
        ids = [self._take() for _ in range(need)]
        self.tables[seq] = ids
        self.lens[seq] = int(num_tokens)
        return list(ids)

    def fork(self, parent: int, child: int) -> None:
        """``child`` shares every block of ``parent`` (reference count + 1)."""
        self._known(parent)
        if child in self.tables:
            raise BlockManagerStateError(f"sequence {child} already allocated")
        ids = list(self.tables[parent])
        for b in ids:
            self.ref[b] += 1
        self.tables[child] = ids
        self.lens[child] = self.lens[parent]

    def append_slot(self, seq: int):
        """Room for one more token of ``seq``.

        Returns (slot, cow) where cow is None or the (src, dst) block pair whose
        contents must be copied before the token is written.
        """
        self._known(seq)
        L = self.lens[seq]
        t = self.tables[seq]
        cow = None
        if L % self.block_size == 0:              # tail full (or no block yet)
            if not self.num_free():
                raise OutOfBlocks("no free block for the next token")
            t.append(self._take())
        else:
            tail = t[L // self.block_size]
            if self.ref[tail] > 1:                # shared partial tail: copy on write
                if not self.num_free():
                    raise OutOfBlocks("no free block for copy-on-write")
                b = self._take()
                self.ref[tail] -= 1
                t[L // self.block_size] = b
                cow = (tail, b)
        self.lens[seq] = L + 1
        return self.slot(seq, L), cow

    def free_seq(self, seq: int) -> None:
        """Drop ``seq``'s references; blocks whose count reaches zero go back to
        the free list, in the sequence's logical order."""
        self._known(seq)
        for b in self.tables[seq]:
            if self.ref[b] < 1:
                raise BlockManagerStateError(f"reference count of block {b} underflows")
            self.ref[b] -= 1
            if self.ref[b] == 0:
                if b in self.hash_of:
                    self.evictable.append(b)      # keep its contents for later hits
                else:
                    self.free.append(b)
        del self.tables[seq]
        del self.lens[seq]

    def allocate_prefix(self, seq: int, token_ids) -> int:
        """A new sequence holding the prompt ``token_ids``, reusing cached blocks
        of the longest cached prefix of full blocks. Returns how many leading
        tokens already have their keys/values in the cache."""
        if seq in self.tables:
            raise BlockManagerStateError(f"sequence {seq} already allocated")
        n = len(token_ids)
        hashes = block_hashes(token_ids, self.block_size)
        hits = []
        for h in hashes:
            b = self.cached.get(h)
            if b is None:
                break
            hits.append(b)
        revived = sum(1 for b in hits if self.ref[b] == 0)
        fresh = self.blocks_needed(n) - len(hits)
        if fresh > self.num_free() - revived:
            raise OutOfBlocks(f"need {fresh} blocks, {self.num_free() - revived} free")
        for b in hits:
            if self.ref[b] == 0:
                self.evictable.remove(b)
            self.ref[b] += 1
        table = list(hits)
        for j in range(len(hits), self.blocks_needed(n)):
            b = self._take()
            if j < len(hashes):                   # a full block: registered for later hits
                self.cached[hashes[j]] = b
                self.hash_of[b] = hashes[j]
            table.append(b)
        self.tables[seq] = table
        self.lens[seq] = n
        return len(hits) * self.block_size

    def swap(self, seqs, dst: "BlockManager"):
        """Move ``seqs`` (a sequence group) from this pool to ``dst``.

        All or nothing: raises OutOfBlocks (nothing changed) if ``dst`` has
        fewer free blocks than the group references distinct blocks. Returns
        the (source block, destination block) pairs to copy.
        """
        seqs = [int(x) for x in seqs]
        if len(set(seqs)) != len(seqs):
            raise BlockManagerStateError("a sequence appears twice in the group")
        for x in seqs:
            self._known(x)
            if x in dst.tables:
                raise BlockManagerStateError(f"sequence {x} already in the destination pool")
        if dst.block_size != self.block_size:
            raise ValueError("pools differ in block size")
        distinct = []
        for x in seqs:
            for b in self.tables[x]:
                if b not in distinct:
                    distinct.append(b)
        if len(distinct) > dst.num_free():
            raise OutOfBlocks(f"need {len(distinct)} blocks, {dst.num_free()} free")
        mapping = {}
        for b in distinct:
            mapping[b] = dst._take()
            dst.ref[mapping[b]] = 0
        for x in seqs:
            table = [mapping[b] for b in self.tables[x]]
            for b in table:
                dst.ref[b] += 1
            dst.tables[x] = table
            dst.lens[x] = self.lens[x]
        for x in seqs:
            self.free_seq(x)
        return [(b, mapping[b]) for b in distinct]

    # -- helpers ---------------------------------------------------------
    def padded_tables(self, seqs, width: int | None = None):
        """int32 [len(seqs), width] tables padded with -1."""
        import numpy as np
        rows = [self.tables[s] for s in seqs]
        w = max((len(r) for r in rows), default=0) if width is None else width
        out = np.full((len(rows), max(w, 1)), -1, dtype=np.int32)
        for i, r in enumerate(rows):
            out[i, :len(r)] = r
        return out

    def _known(self, seq: int) -> None:
        if seq not in self.tables:
            raise BlockManagerStateError(f"unknown sequence {seq}")
