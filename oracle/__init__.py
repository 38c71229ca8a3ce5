"""Oracle for paged decode attention — TEST INFRASTRUCTURE, not the product.

A plain, slow, obviously correct CPU restatement of what the PagedAttention
hot path computes, in float64. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s ``cpu_baseline`` / reference leg may import, call or execute
anything in this package. The product path (the CUDA library and its Python
binding) never reaches it, and this package imports nothing of the product.

Modules:
  formats        binary16 / bfloat16 bit patterns -> float64, from the formats' definitions
  attention      decode attention: gather through the block table, then one global softmax
  cache_ops      reshape_and_cache (slot scatter), copy_blocks (copy-on-write copy),
                 swap_blocks (copies between a GPU pool and a CPU pool)
  block_manager  free list, reference counts, fork, append with copy-on-write, swap

Parity status of every function is pinned by ``tests/test_oracle_*.py`` except
where a function's docstring says "parity unpinned".
"""

from .formats import decode_bits  # noqa: F401
from .attention import paged_attention_decode, attend_sequence  # noqa: F401
from .cache_ops import reshape_and_cache, copy_blocks, swap_blocks  # noqa: F401
from .block_manager import BlockManager, OutOfBlocks, BlockManagerStateError  # noqa: F401
