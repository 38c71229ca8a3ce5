"""The Python binding rejects tensors the C ABI cannot describe safely.

The library sees only pointers and sizes, so a tensor of the wrong dtype,
shape or layout would be read or written past its end by the kernels. Each
wrapper checks these facts before anything crosses the ABI and raises
ValueError; these tests run on the CPU (CPU tensors with one fact wrong are
refused for that fact, and CPU tensors that are right in every other way are
refused for not being on a CUDA device).
"""

import pytest
import torch

import paged_kv_cache_118_gb300 as pk

S, H, HKV, D, NB, B, W = 3, 8, 2, 64, 10, 16, 4


def _decode_args(**over):
    a = dict(out=torch.empty(S, H, D, dtype=torch.float16),
             q=torch.empty(S, H, D, dtype=torch.float16),
             k_cache=torch.empty(NB, B, HKV, D, dtype=torch.float16),
             v_cache=torch.empty(NB, B, HKV, D, dtype=torch.float16),
             block_tables=torch.zeros(S, W, dtype=torch.int32),
             context_lens=torch.ones(S, dtype=torch.int32),
             block_size=B, scale=0.125,
             workspace=torch.empty(1024, dtype=torch.uint8))
    a.update(over)
    return a


@pytest.mark.parametrize("over, msg", [
    (dict(q=torch.empty(S, H, D, dtype=torch.bfloat16)), "q dtype"),
    (dict(q=torch.empty(S, H, 128, dtype=torch.float16),
          out=torch.empty(S, H, 128, dtype=torch.float16)), "head_size"),
    (dict(block_size=8), "block_size"),
    (dict(block_tables=torch.zeros(S, W, dtype=torch.int64)), "block_tables must be torch.int32"),
    (dict(block_tables=torch.zeros(S + 1, W, dtype=torch.int32)), "block_tables must have shape"),
    (dict(context_lens=torch.ones(S, dtype=torch.int64)), "context_lens must be torch.int32"),
    (dict(context_lens=torch.ones(S + 2, dtype=torch.int32)), "context_lens must have shape"),
    (dict(v_cache=torch.empty(NB, B, HKV + 1, D, dtype=torch.float16)), "v_cache shape"),
    (dict(v_cache=torch.empty(NB, B, HKV, D, dtype=torch.bfloat16)), "caches must both be"),
    (dict(out=torch.empty(S, H + 1, D, dtype=torch.float16)), "out shape"),
    (dict(out=torch.empty(S, H, D, dtype=torch.float64)), "out dtype"),
    (dict(q=torch.empty(S, D, H, dtype=torch.float16).transpose(1, 2)), "q must be contiguous"),
    (dict(q=torch.empty(S, 3, D, dtype=torch.float16),
          out=torch.empty(S, 3, D, dtype=torch.float16)), "multiple of num_kv_heads"),
    (dict(k_cache=torch.empty(NB, HKV, B, D, dtype=torch.float16).transpose(1, 2),
          v_cache=torch.empty(NB, HKV, B, D, dtype=torch.float16).transpose(1, 2)),
     "contiguous"),
])
def test_decode_rejects(over, msg):
    a = _decode_args(**over)
    with pytest.raises(ValueError, match=msg):
        pk.pkv_paged_attention_decode(**a)


def test_decode_noalloc_rejects_int64_tables():
    a = _decode_args(block_tables=torch.zeros(S, W, dtype=torch.int64))
    del a["workspace"]
    with pytest.raises(ValueError, match="block_tables must be torch.int32"):
        pk.pkv_paged_attention_decode_noalloc(**a)


def test_decode_err_flag_must_be_int32():
    with pytest.raises(ValueError, match="err_flag"):
        pk.pkv_paged_attention_decode(**_decode_args(), err_flag=torch.zeros(1, dtype=torch.int64))


def test_decode_wants_cuda_once_everything_else_is_right():
    with pytest.raises(ValueError, match="CUDA tensors"):
        pk.pkv_paged_attention_decode(**_decode_args())


def _rc_args(**over):
    T = 5
    a = dict(k=torch.empty(T, HKV, D, dtype=torch.float16),
             v=torch.empty(T, HKV, D, dtype=torch.float16),
             k_cache=torch.empty(NB, B, HKV, D, dtype=torch.float16),
             v_cache=torch.empty(NB, B, HKV, D, dtype=torch.float16),
             slot_mapping=torch.zeros(T, dtype=torch.int64))
    a.update(over)
    return a


@pytest.mark.parametrize("over, msg", [
    (dict(slot_mapping=torch.zeros(5, dtype=torch.int32)), "slot_mapping must be torch.int64"),
    (dict(slot_mapping=torch.zeros(4, dtype=torch.int64)), "slot_mapping must have shape"),
    (dict(k=torch.empty(5, HKV + 1, D, dtype=torch.float16),
          v=torch.empty(5, HKV + 1, D, dtype=torch.float16)), "k rows"),
    (dict(k=torch.empty(5, HKV, 2 * D, dtype=torch.float16),
          v=torch.empty(5, HKV, 2 * D, dtype=torch.float16)), "k rows"),
    (dict(v=torch.empty(6, HKV, D, dtype=torch.float16)), "k and v"),
    (dict(k=torch.empty(5, HKV, D, dtype=torch.bfloat16),
          v=torch.empty(5, HKV, D, dtype=torch.bfloat16)), "cache dtype"),
    (dict(k=torch.empty(5, D, HKV, dtype=torch.float16).transpose(1, 2)), "k must be contiguous"),
])
def test_reshape_and_cache_rejects(over, msg):
    with pytest.raises(ValueError, match=msg):
        pk.pkv_reshape_and_cache(**_rc_args(**over))


def test_reshape_and_cache_wants_cuda():
    with pytest.raises(ValueError, match="CUDA tensors"):
        pk.pkv_reshape_and_cache(**_rc_args())


def _pf_args(**over):
    Tq = 7
    a = dict(out=torch.empty(Tq, H, D, dtype=torch.float16),
             q=torch.empty(Tq, H, D, dtype=torch.float16),
             k_cache=torch.empty(NB, B, HKV, D, dtype=torch.float16),
             v_cache=torch.empty(NB, B, HKV, D, dtype=torch.float16),
             block_tables=torch.zeros(S, W, dtype=torch.int32),
             context_lens=torch.ones(S, dtype=torch.int32),
             query_start=torch.zeros(S + 1, dtype=torch.int32),
             max_query_len=4, block_size=B, scale=0.125)
    a.update(over)
    return a


@pytest.mark.parametrize("over, msg", [
    (dict(query_start=torch.zeros(S, dtype=torch.int32)), "query_start must have shape"),
    (dict(query_start=torch.zeros(S + 1, dtype=torch.int64)), "query_start must be torch.int32"),
    (dict(block_tables=torch.zeros(S, W, dtype=torch.int64)), "block_tables must be torch.int32"),
    (dict(q=torch.empty(7, H, D, dtype=torch.bfloat16)), "q dtype"),
    (dict(block_size=32), "block_size"),
])
def test_prefill_rejects(over, msg):
    with pytest.raises(ValueError, match=msg):
        pk.pkv_paged_attention_prefill(**_pf_args(**over))


def test_prefill_rejects_a_wrong_workspace():
    with pytest.raises(ValueError, match="workspace"):
        pk.pkv_paged_attention_prefill(**_pf_args(), workspace=torch.empty(16, dtype=torch.int32))


def test_copy_blocks_rejects_mismatched_caches():
    k = torch.empty(NB, B, HKV, D, dtype=torch.float16)
    with pytest.raises(ValueError, match="v_cache shape"):
        pk.pkv_copy_blocks(k, torch.empty(NB, B, HKV, 2 * D, dtype=torch.float16), [[0, 1]])
    with pytest.raises(ValueError, match="CUDA tensors"):
        pk.pkv_copy_blocks(k, torch.empty_like(k), [[0, 1]])


def test_swap_blocks_rejects_mismatched_pools():
    src = torch.empty(NB, B, HKV, D, dtype=torch.float16)
    dst = torch.empty(NB, B, HKV, D, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="same block shape"):
        pk.pkv_swap_blocks(dst, torch.empty_like(dst), src, torch.empty_like(src), [[0, 1]])
