"""pagedkv — paged KV-cache decode attention on GB300 (sm_103a).

A thin Python binding over the C ABI of ``libpagedkv.so`` (declared in
``include/pagedkv.h``). The functions here keep the C names and only marshal
arguments: torch tensors become device pointers and sizes, the current torch
stream becomes the CUDA stream. Every step of the computation runs in the
library's CUDA kernels (or, for the block manager, its C++ host code).

Importing this package loads the library and raises if it has not been built
(``python paged_kv_cache_118_gb300/build.py``); there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedkv.so")

PKV_OK, PKV_EINVAL, PKV_ENOMEM, PKV_ERANGE, PKV_ECUDA, PKV_ESTATE, PKV_EWORKSPACE = range(7)
PKV_F16, PKV_BF16, PKV_F32 = 0, 1, 2
PKV_DEVERR_BLOCK_ID, PKV_DEVERR_CONTEXT, PKV_DEVERR_SLOT, PKV_DEVERR_TIMEOUT = 1, 2, 4, 8

_DTYPE = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16, torch.float32: PKV_F32}

_c_int, _c_i64, _c_sz, _c_f, _vp = (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                     ctypes.c_float, ctypes.c_void_p)

# name -> (restype, argtypes); the exported symbols of include/pagedkv.h
SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [_c_int]),
    "pkv_version": (ctypes.c_char_p, []),
    "pkv_decode_workspace_size": (_c_sz, [_c_int] * 7),
    "pkv_decode_partition_tokens": (_c_int, [_c_int] * 7),
    "pkv_paged_attention_decode": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _c_int, _vp, _vp,
                                            _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                            _c_int, _c_f, _c_int, _vp, _c_sz, _vp, _vp]),
    "pkv_paged_attention_decode_noalloc": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _c_int, _vp,
                                                    _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                                    _c_int, _c_int, _c_f, _c_int, _vp, _vp]),
    "pkv_test_decode_wait_timeout": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _c_int, _vp, _vp,
                                              _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                              _c_int, _c_f, _c_int, _vp, _c_sz, _vp,
                                              ctypes.c_uint64, _vp]),
    "pkv_prefill_workspace_size": (_c_sz, []),
    "pkv_paged_attention_prefill": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _c_int, _vp, _vp, _vp,
                                             _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                             _c_int, _c_int, _c_int, _c_f, _vp, _c_sz, _vp, _vp]),
    "pkv_reshape_and_cache": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                       _c_int, _c_int, _c_int, _vp, _vp]),
    "pkv_copy_blocks": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_sz, _vp]),
    "pkv_swap_blocks": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_sz, _vp]),
    "pkv_bm_swap": (_c_int, [_vp, _vp, _vp, _c_int, _vp, _c_int, _vp]),
    "pkv_bm_create": (_vp, [_c_int, _c_int, _vp]),
    "pkv_bm_destroy": (None, [_vp]),
    "pkv_bm_allocate": (_c_int, [_vp, _c_i64, _c_i64]),
    "pkv_bm_fork": (_c_int, [_vp, _c_i64, _c_i64]),
    "pkv_bm_append_slot": (_c_int, [_vp, _c_i64, _vp, _vp, _vp]),
    "pkv_bm_append_slots": (_c_int, [_vp, _vp, _c_int, _vp, _vp, _vp]),
    "pkv_bm_free": (_c_int, [_vp, _c_i64]),
    "pkv_bm_allocate_prefix": (_c_int, [_vp, _c_i64, _vp, _c_i64, _vp]),
    "pkv_bm_num_cached": (_c_int, [_vp]),
    "pkv_bm_num_free": (_c_int, [_vp]),
    "pkv_bm_refcount": (_c_int, [_vp, ctypes.c_int32]),
    "pkv_bm_length": (_c_i64, [_vp, _c_i64]),
    "pkv_bm_block_table": (_c_int, [_vp, _c_i64, _vp, _c_int, _vp]),
    "pkv_bm_fill_tables": (_c_int, [_vp, _vp, _c_int, _vp, _c_int, _vp]),
    "pkv_bm_slots": (_c_int, [_vp, _c_i64, _c_i64, _c_i64, _vp]),
    "pkv_bm_free_list": (_c_int, [_vp, _vp, _c_int]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python paged_kv_cache_118_gb300/build.py` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class PagedKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib.pkv_status_string(status).decode()} (status {status})")


def _check(status: int, where: str) -> None:
    if status != PKV_OK:
        raise PagedKVError(status, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _need_cuda(*ts):
    d0 = None
    for t in ts:
        if t is None:
            continue
        d = t.device
        if d0 is None:
            d0 = d
        if d != d0 or d.type != "cuda":
            if d.type != "cuda" or d0.type != "cuda":
                raise ValueError("pagedkv kernels take CUDA tensors")
            raise ValueError(f"pagedkv tensors must share one device, got {d0} and {d}")


# ---------------------------------------------------------------- argument checks
# The C ABI sees only pointers and sizes, so every shape, dtype and layout fact
# the kernels rely on is checked here first: a tensor of the wrong type or shape
# would otherwise be read or written past its end.

_KV_DTYPES = (torch.float16, torch.bfloat16)


def _require(cond: bool, where: str, what: str) -> None:
    if not cond:
        raise ValueError(f"{where}: {what}")


def _contiguous(where: str, **ts) -> None:
    for name, t in ts.items():
        if t is not None:
            _require(t.is_contiguous(), where, f"{name} must be contiguous")


def _check_caches(where: str, k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
    _require(k_cache.dim() == 4, where,
             "k_cache must be [num_blocks, block_size, num_kv_heads, head_size]")
    _require(tuple(v_cache.shape) == tuple(k_cache.shape), where,
             f"v_cache shape {tuple(v_cache.shape)} != k_cache shape {tuple(k_cache.shape)}")
    _require(k_cache.dtype in _KV_DTYPES and v_cache.dtype == k_cache.dtype, where,
             "caches must both be float16 or both bfloat16")
    _contiguous(where, k_cache=k_cache, v_cache=v_cache)


def _check_int(where: str, name: str, t: torch.Tensor, dtype, shape) -> None:
    _require(t.dtype == dtype, where, f"{name} must be {dtype}, got {t.dtype}")
    _require(tuple(t.shape) == tuple(shape), where,
             f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    _require(t.is_contiguous(), where, f"{name} must be contiguous")


def _check_err(where: str, err_flag) -> None:
    if err_flag is not None:
        _require(err_flag.dtype == torch.int32 and err_flag.numel() >= 1, where,
                 "err_flag must be an int32 tensor of at least one element")


_I32, _I64 = torch.int32, torch.int64


def _caches_ok(k_cache, v_cache) -> bool:
    ks = k_cache.shape
    kd = k_cache.dtype
    return (len(ks) == 4 and v_cache.shape == ks and (kd is torch.float16 or kd is torch.bfloat16)
            and v_cache.dtype is kd and k_cache.is_contiguous() and v_cache.is_contiguous())


def _err_ok(err_flag) -> bool:
    return err_flag is None or (err_flag.dtype is _I32 and err_flag.numel() >= 1)


def _decode_ok(out, q, k_cache, v_cache, block_tables, context_lens, block_size,
               err_flag) -> bool:
    """Every fact _check_decode checks, as one cheap expression (the wrappers
    run on every decode call; the detailed checks only run when this fails)."""
    if not _caches_ok(k_cache, v_cache):
        return False
    ks, qs, bs = k_cache.shape, q.shape, block_tables.shape
    return (len(qs) == 3 and q.dtype is k_cache.dtype and qs[2] == ks[3] and qs[1] % ks[2] == 0
            and block_size == ks[1] and out.shape == qs and out.dtype in _DTYPE
            and len(bs) == 2 and block_tables.dtype is _I32 and bs[0] == qs[0]
            and context_lens.dtype is _I32 and context_lens.shape == (qs[0],)
            and q.is_contiguous() and out.is_contiguous() and block_tables.is_contiguous()
            and context_lens.is_contiguous() and _err_ok(err_flag))


def _check_decode(where: str, out, q, k_cache, v_cache, block_tables, context_lens,
                  block_size, err_flag) -> None:
    if _decode_ok(out, q, k_cache, v_cache, block_tables, context_lens, block_size, err_flag):
        return
    _check_caches(where, k_cache, v_cache)
    nb, B, Hkv, D = k_cache.shape
    _require(q.dim() == 3, where, "q must be [num_seqs, num_heads, head_size]")
    S, H, Dq = q.shape
    _require(q.dtype == k_cache.dtype, where, f"q dtype {q.dtype} != cache dtype {k_cache.dtype}")
    _require(Dq == D, where, f"q head_size {Dq} != cache head_size {D}")
    _require(H % Hkv == 0, where, f"num_heads {H} is not a multiple of num_kv_heads {Hkv}")
    _require(int(block_size) == B, where, f"block_size {block_size} != cache block size {B}")
    _require(tuple(out.shape) == tuple(q.shape), where,
             f"out shape {tuple(out.shape)} != q shape {tuple(q.shape)}")
    _require(out.dtype in _DTYPE, where, f"out dtype {out.dtype} is not float16/bfloat16/float32")
    _require(block_tables.dim() == 2, where, "block_tables must be [num_seqs, max_blocks_per_seq]")
    _check_int(where, "block_tables", block_tables, torch.int32, (S, block_tables.shape[1]))
    _check_int(where, "context_lens", context_lens, torch.int32, (S,))
    _contiguous(where, q=q, out=out)
    _check_err(where, err_flag)
    raise ValueError(f"{where}: arguments rejected")


# ---------------------------------------------------------------- kernels

def pkv_decode_partition_tokens(num_seqs: int, num_heads: int, num_kv_heads: int,
                                head_size: int, max_blocks_per_seq: int, block_size: int,
                                partition_tokens: int = 0) -> int:
    """The partition size a decode call with these arguments uses (0 = the default)."""
    return int(lib.pkv_decode_partition_tokens(num_seqs, num_heads, num_kv_heads, head_size,
                                               max_blocks_per_seq, block_size, partition_tokens))


def pkv_decode_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int,
                              head_size: int, max_blocks_per_seq: int, block_size: int,
                              partition_tokens: int = 0) -> int:
    return int(lib.pkv_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size,
                                             max_blocks_per_seq, block_size, partition_tokens))


def decode_workspace(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq,
                     block_size, partition_tokens=0, device="cuda") -> torch.Tensor:
    """A caller-owned scratch buffer of the size the decode call needs."""
    n = pkv_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size,
                                  max_blocks_per_seq, block_size, partition_tokens)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def prefill_workspace(device="cuda") -> torch.Tensor:
    """A caller-owned scratch buffer of the size the prefill call needs."""
    return torch.empty(lib.pkv_prefill_workspace_size(), dtype=torch.uint8, device=device)


def pkv_paged_attention_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                               v_cache: torch.Tensor, block_tables: torch.Tensor,
                               context_lens: torch.Tensor, block_size: int, scale: float,
                               workspace: torch.Tensor, partition_tokens: int = 0,
                               err_flag: torch.Tensor | None = None, stream=None) -> None:
    """out[s, h] = softmax attention of q[s, h] over sequence s's paged history.

    q, out: [num_seqs, num_heads, head_size]; caches: [num_blocks, block_size,
    num_kv_heads, head_size]; block_tables: int32 [num_seqs, max_blocks_per_seq];
    context_lens: int32 [num_seqs]; workspace: bytes from decode_workspace().
    """
    where = "pkv_paged_attention_decode"
    _check_decode(where, out, q, k_cache, v_cache, block_tables, context_lens, block_size,
                  err_flag)
    _contiguous(where, workspace=workspace)
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, workspace, err_flag)
    S, H, D = q.shape
    nb, B, Hkv, _ = k_cache.shape
    st = lib.pkv_paged_attention_decode(
        _ptr(out), _DTYPE[out.dtype], _ptr(q), _ptr(k_cache), _ptr(v_cache), _DTYPE[q.dtype],
        _ptr(block_tables), _ptr(context_lens), S, H, Hkv, D, nb, block_size,
        block_tables.shape[1], float(scale), partition_tokens, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(err_flag), _stream(stream))
    _check(st, "pkv_paged_attention_decode")


NOALLOC_SCRATCH_BYTES = 8 << 20


def pkv_paged_attention_decode_noalloc(out: torch.Tensor, q: torch.Tensor,
                                       k_cache: torch.Tensor, v_cache: torch.Tensor,
                                       block_tables: torch.Tensor, context_lens: torch.Tensor,
                                       block_size: int, scale: float, partition_tokens: int = 0,
                                       err_flag: torch.Tensor | None = None, stream=None) -> None:
    """pkv_paged_attention_decode without a workspace argument, for callers that
    cannot allocate device memory: the partials go to the library's built-in
    NOALLOC_SCRATCH_BYTES array (shared by all calls; keep calls on one stream)."""
    _check_decode("pkv_paged_attention_decode_noalloc", out, q, k_cache, v_cache, block_tables,
                  context_lens, block_size, err_flag)
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, err_flag)
    S, H, D = q.shape
    nb, B, Hkv, _ = k_cache.shape
    st = lib.pkv_paged_attention_decode_noalloc(
        _ptr(out), _DTYPE[out.dtype], _ptr(q), _ptr(k_cache), _ptr(v_cache), _DTYPE[q.dtype],
        _ptr(block_tables), _ptr(context_lens), S, H, Hkv, D, nb, block_size,
        block_tables.shape[1], float(scale), partition_tokens, _ptr(err_flag), _stream(stream))
    _check(st, "pkv_paged_attention_decode_noalloc")


def pkv_paged_attention_prefill(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                v_cache: torch.Tensor, block_tables: torch.Tensor,
                                context_lens: torch.Tensor, query_start: torch.Tensor,
                                max_query_len: int, block_size: int, scale: float,
                                workspace: torch.Tensor | None = None,
                                err_flag: torch.Tensor | None = None, stream=None) -> None:
    """Causal attention of each sequence's query chunk (its last C tokens) over
    its paged history. q, out: [total_queries, num_heads, head_size];
    query_start: int32 [num_seqs + 1]; workspace: uint8, at least
    pkv_prefill_workspace_size() bytes (prefill_workspace() makes one; the
    call allocates one when it is None)."""
    where = "pkv_paged_attention_prefill"
    _check_caches(where, k_cache, v_cache)
    nb, B, Hkv, D = k_cache.shape
    _require(q.dim() == 3 and q.shape[2] == D, where, "q must be [total_queries, num_heads, head_size]")
    _require(q.dtype == k_cache.dtype, where, f"q dtype {q.dtype} != cache dtype {k_cache.dtype}")
    _require(q.shape[1] % Hkv == 0, where, "num_heads is not a multiple of num_kv_heads")
    _require(int(block_size) == B, where, f"block_size {block_size} != cache block size {B}")
    _require(tuple(out.shape) == tuple(q.shape), where, "out must have q's shape")
    _require(out.dtype in _DTYPE, where, f"out dtype {out.dtype} is not float16/bfloat16/float32")
    S = context_lens.shape[0] if context_lens.dim() == 1 else -1
    _check_int(where, "context_lens", context_lens, torch.int32, (S,))
    _require(block_tables.dim() == 2, where, "block_tables must be [num_seqs, max_blocks_per_seq]")
    _check_int(where, "block_tables", block_tables, torch.int32, (S, block_tables.shape[1]))
    _check_int(where, "query_start", query_start, torch.int32, (S + 1,))
    _contiguous(where, q=q, out=out)
    _check_err(where, err_flag)
    if workspace is not None:
        _require(workspace.dtype == torch.uint8 and workspace.is_contiguous(), where,
                 "workspace must be a contiguous uint8 tensor")
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, query_start, err_flag,
               workspace)
    if workspace is None:
        workspace = prefill_workspace(out.device)
    _, H, D = q.shape
    st = lib.pkv_paged_attention_prefill(
        _ptr(out), _DTYPE[out.dtype], _ptr(q), _ptr(k_cache), _ptr(v_cache), _DTYPE[q.dtype],
        _ptr(block_tables), _ptr(context_lens), _ptr(query_start), context_lens.shape[0], H,
        Hkv, D, nb, block_size, block_tables.shape[1], int(max_query_len), q.shape[0],
        float(scale), _ptr(workspace), workspace.numel(), _ptr(err_flag), _stream(stream))
    _check(st, "pkv_paged_attention_prefill")


def pkv_reshape_and_cache(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                          err_flag: torch.Tensor | None = None, stream=None) -> None:
    """k_cache[slot // B, slot % B] = k[t] (and v) for every token t with slot >= 0."""
    kshape = k.shape
    if not (_caches_ok(k_cache, v_cache) and len(kshape) == 3 and v.shape == kshape
            and kshape[1:] == k_cache.shape[2:] and k.dtype is k_cache.dtype
            and v.dtype is k_cache.dtype and slot_mapping.dtype is _I64
            and slot_mapping.shape == kshape[:1] and slot_mapping.is_contiguous()
            and k.is_contiguous() and v.is_contiguous() and _err_ok(err_flag)):
        where = "pkv_reshape_and_cache"
        _check_caches(where, k_cache, v_cache)
        _require(k.dim() == 3 and tuple(v.shape) == tuple(k.shape), where,
                 "k and v must both be [num_tokens, num_kv_heads, head_size]")
        _require(tuple(k.shape[1:]) == tuple(k_cache.shape[2:]), where,
                 f"k rows {tuple(k.shape[1:])} != cache rows {tuple(k_cache.shape[2:])}")
        _require(k.dtype == k_cache.dtype and v.dtype == k_cache.dtype, where,
                 f"k/v dtype must be the cache dtype {k_cache.dtype}")
        _check_int(where, "slot_mapping", slot_mapping, torch.int64, (k.shape[0],))
        _contiguous(where, k=k, v=v)
        _check_err(where, err_flag)
        raise ValueError(f"{where}: arguments rejected")
    _need_cuda(k, v, k_cache, v_cache, slot_mapping, err_flag)
    T, Hkv, D = k.shape
    nb, B = k_cache.shape[:2]
    st = lib.pkv_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(slot_mapping), T, Hkv, D, nb, B, _DTYPE[k.dtype],
                                   _ptr(err_flag), _stream(stream))
    _check(st, "pkv_reshape_and_cache")


def pkv_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst_pairs,
                    stream=None) -> None:
    """Copy-on-write: block dst of both caches becomes a copy of block src.

    src_dst_pairs: host int32 array-like [n, 2]."""
    import numpy as np
    _check_caches("pkv_copy_blocks", k_cache, v_cache)
    _need_cuda(k_cache, v_cache)
    pairs = np.ascontiguousarray(np.asarray(src_dst_pairs, dtype=np.int32).reshape(-1, 2))
    block_bytes = k_cache[0].numel() * k_cache.element_size()
    st = lib.pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), pairs.ctypes.data, pairs.shape[0],
                             k_cache.shape[0], block_bytes, _stream(stream))
    _check(st, "pkv_copy_blocks")


def pkv_swap_blocks(dst_k: torch.Tensor, dst_v: torch.Tensor, src_k: torch.Tensor,
                    src_v: torch.Tensor, src_dst_pairs, stream=None) -> None:
    """dst pool block d = src pool block s for each (s, d); either pool may be a
    pinned host tensor (swap space)."""
    import numpy as np
    where = "pkv_swap_blocks"
    _check_caches(where, src_k, src_v)
    _check_caches(where, dst_k, dst_v)
    _require(tuple(dst_k.shape[1:]) == tuple(src_k.shape[1:]) and dst_k.dtype == src_k.dtype,
             where, "source and destination pools must have the same block shape and dtype")
    for t in (dst_k, dst_v, src_k, src_v):
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError("swap pools must be CUDA tensors or pinned host tensors")
    pairs = np.ascontiguousarray(np.asarray(src_dst_pairs, dtype=np.int32).reshape(-1, 2))
    block_bytes = src_k[0].numel() * src_k.element_size()
    st = lib.pkv_swap_blocks(_ptr(dst_k), _ptr(dst_v), _ptr(src_k), _ptr(src_v),
                             pairs.ctypes.data, pairs.shape[0], src_k.shape[0], dst_k.shape[0],
                             block_bytes, _stream(stream))
    _check(st, "pkv_swap_blocks")


# ---------------------------------------------------------------- block manager

class BlockManager:
    """Handle on the library's host block manager (pkv_bm_*)."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        import numpy as np
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = None
        if free_order is not None:
            order = np.ascontiguousarray(np.asarray(free_order, dtype=np.int32))
            if order.shape != (num_blocks,):
                raise ValueError("free_order must hold num_blocks ids")
        self._h = lib.pkv_bm_create(num_blocks, block_size,
                                    None if order is None else order.ctypes.data)
        if not self._h:
            raise PagedKVError(PKV_EINVAL, "pkv_bm_create")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib.pkv_bm_destroy(h)
            self._h = None

    def allocate(self, seq: int, num_tokens: int) -> None:
        _check(lib.pkv_bm_allocate(self._h, seq, num_tokens), "pkv_bm_allocate")

    def allocate_prefix(self, seq: int, token_ids) -> int:
        """A new sequence holding the prompt token_ids, sharing cached blocks of
        its prefix; returns the number of leading tokens already cached."""
        import numpy as np
        toks = np.ascontiguousarray(np.asarray(token_ids, dtype=np.int32))
        cached = ctypes.c_int64()
        _check(lib.pkv_bm_allocate_prefix(self._h, seq, toks.ctypes.data, toks.shape[0],
                                          ctypes.byref(cached)), "pkv_bm_allocate_prefix")
        return cached.value

    def num_cached(self) -> int:
        return int(lib.pkv_bm_num_cached(self._h))

    def fork(self, parent: int, child: int) -> None:
        _check(lib.pkv_bm_fork(self._h, parent, child), "pkv_bm_fork")

    def append_slot(self, seq: int):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib.pkv_bm_append_slot(self._h, seq, ctypes.byref(slot), ctypes.byref(src),
                                      ctypes.byref(dst)), "pkv_bm_append_slot")
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def append_slots(self, seqs):
        """Batch append (all or nothing): returns (slots int64 [n], cow int32 [k, 2])."""
        import numpy as np
        seqs = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        n = seqs.shape[0]
        slots = np.empty(n, np.int64)
        cow = np.empty((max(n, 1), 2), np.int32)
        k = ctypes.c_int()
        _check(lib.pkv_bm_append_slots(self._h, seqs.ctypes.data, n, slots.ctypes.data,
                                       cow.ctypes.data, ctypes.byref(k)), "pkv_bm_append_slots")
        return slots, cow[:k.value]

    def free_seq(self, seq: int) -> None:
        _check(lib.pkv_bm_free(self._h, seq), "pkv_bm_free")

    def swap(self, seqs, dst: "BlockManager"):
        """Move a sequence group to another pool's manager; returns the
        (src block, dst block) pairs to copy (int32 [k, 2])."""
        import numpy as np
        seqs = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        n = ctypes.c_int()
        st = lib.pkv_bm_swap(self._h, dst._h, seqs.ctypes.data, seqs.shape[0], None, 0,
                             ctypes.byref(n))
        if st == PKV_OK:                      # nothing to copy: the swap is done
            return np.empty((0, 2), np.int32)
        if st != PKV_ERANGE:
            _check(st, "pkv_bm_swap")
        pairs = np.empty((max(n.value, 1), 2), np.int32)
        _check(lib.pkv_bm_swap(self._h, dst._h, seqs.ctypes.data, seqs.shape[0],
                               pairs.ctypes.data, pairs.shape[0], ctypes.byref(n)),
               "pkv_bm_swap")
        return pairs[:n.value]

    def num_free(self) -> int:
        return int(lib.pkv_bm_num_free(self._h))

    def refcount(self, block: int) -> int:
        return int(lib.pkv_bm_refcount(self._h, block))

    def length(self, seq: int) -> int:
        return int(lib.pkv_bm_length(self._h, seq))

    def table(self, seq: int):
        import numpy as np
        n = ctypes.c_int()
        lib.pkv_bm_block_table(self._h, seq, None, 0, ctypes.byref(n))
        out = np.empty(max(n.value, 1), np.int32)
        _check(lib.pkv_bm_block_table(self._h, seq, out.ctypes.data, out.shape[0],
                                      ctypes.byref(n)), "pkv_bm_block_table")
        return out[:n.value]

    def fill_tables(self, seqs, width: int):
        """(tables int32 [n, width] padded with -1, context_lens int32 [n])."""
        import numpy as np
        seqs = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        n = seqs.shape[0]
        out = np.empty((n, width), np.int32)
        lens = np.empty(n, np.int32)
        _check(lib.pkv_bm_fill_tables(self._h, seqs.ctypes.data, n, out.ctypes.data, width,
                                      lens.ctypes.data), "pkv_bm_fill_tables")
        return out, lens

    def slots(self, seq: int, first: int = 0, count: int | None = None):
        import numpy as np
        if count is None:
            count = self.length(seq) - first
        out = np.empty(max(count, 1), np.int64)
        _check(lib.pkv_bm_slots(self._h, seq, first, count, out.ctypes.data), "pkv_bm_slots")
        return out[:count]

    def free_list(self):
        import numpy as np
        n = lib.pkv_bm_free_list(self._h, None, 0)
        out = np.empty(max(n, 1), np.int32)
        lib.pkv_bm_free_list(self._h, out.ctypes.data, n)
        return out[:n]
