"""Pins of the chunked-prefill oracle: a one-token chunk is the (pinned) decode
oracle bit for bit; a whole-prompt chunk is torch's causal SDPA; a chunk at
the end of a context is SDPA with an explicit causal mask; chunks computed
one after another give what one chunk over the union gives."""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle.attention import paged_attention_decode
from oracle.formats import decode_bits
from oracle.pipeline import build_decode_state, pool_demand
from oracle.prefill import paged_attention_prefill, prefill_sequence
from workloads import decode_batch, free_order, normal_bits, poison_bits


def _state(lens, H, Hkv, d, B, dt, seed):
    batch = decode_batch("p", lens, H, Hkv, d, B, dt, seed=seed)
    n = pool_demand(batch.context_lens, B) + 5
    return batch, build_decode_state(batch, n, free_order(n, seed), poison_bits(dt))


def _sdpa(qb, kb, vb, dt, scale, mask):
    q = torch.from_numpy(decode_bits(qb, dt)).permute(1, 0, 2)[None]     # [1, H, C, d]
    k = torch.from_numpy(decode_bits(kb, dt)).permute(1, 0, 2)[None]
    v = torch.from_numpy(decode_bits(vb, dt)).permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=torch.from_numpy(mask),
                                       scale=scale, enable_gqa=q.shape[1] != k.shape[1])
    return o[0].permute(1, 0, 2).numpy()


def test_one_token_chunk_is_decode():
    batch, st = _state((5, 40, 129), 8, 2, 64, 16, "bf16", 1)
    starts = np.arange(4)
    got = paged_attention_prefill(batch.q, st["k_cache"], st["v_cache"], st["block_tables"],
                                  batch.context_lens, starts, 16, batch.scale, "bf16")
    want = paged_attention_decode(batch.q, st["k_cache"], st["v_cache"], st["block_tables"],
                                  batch.context_lens, 16, batch.scale, "bf16")
    assert np.array_equal(got, want)


@pytest.mark.parametrize("C", [1, 9, 64, 100])
def test_chunk_matches_masked_sdpa(C):
    L = 100
    batch, st = _state((L,), 6, 3, 64, 8, "f16", C)
    rng = np.random.default_rng(C)
    q = normal_bits(rng, (C, 6, 64), "f16")
    got = prefill_sequence(q, st["k_cache"], st["v_cache"], st["block_tables"][0], L, 8,
                           batch.scale, "f16")
    pos = L - C + np.arange(C)
    mask = np.arange(L)[None, :] <= pos[:, None]
    want = _sdpa(q, batch.k_tokens, batch.v_tokens, "f16", float(batch.scale), mask)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    if C == L:                                            # the whole prompt: plain causal
        qt = torch.from_numpy(decode_bits(q, "f16")).permute(1, 0, 2)[None]
        kt = torch.from_numpy(decode_bits(batch.k_tokens, "f16")).permute(1, 0, 2)[None]
        vt = torch.from_numpy(decode_bits(batch.v_tokens, "f16")).permute(1, 0, 2)[None]
        o = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=float(batch.scale),
                                           enable_gqa=True)[0].permute(1, 0, 2).numpy()
        np.testing.assert_allclose(got, o, rtol=0, atol=1e-12)


def test_chunks_in_order_equal_one_chunk():
    L = 90
    batch, st = _state((L,), 4, 4, 64, 16, "bf16", 4)
    q = normal_bits(np.random.default_rng(9), (50, 4, 64), "bf16")
    whole = prefill_sequence(q, st["k_cache"], st["v_cache"], st["block_tables"][0], L, 16,
                             batch.scale, "bf16")
    a = prefill_sequence(q[:20], st["k_cache"], st["v_cache"], st["block_tables"][0], L - 30, 16,
                         batch.scale, "bf16")
    b = prefill_sequence(q[20:], st["k_cache"], st["v_cache"], st["block_tables"][0], L, 16,
                         batch.scale, "bf16")
    np.testing.assert_allclose(np.concatenate([a, b]), whole, rtol=0, atol=1e-12)


def test_planted_mistake_no_causal_mask_is_caught(monkeypatch):
    import oracle.prefill as pf
    L = 40
    batch, st = _state((L,), 4, 2, 64, 8, "f16", 5)
    q = normal_bits(np.random.default_rng(1), (10, 4, 64), "f16")
    monkeypatch.setattr(pf, "causal_visibility", lambda L_, C_: np.ones((C_, L_), bool))
    got = pf.prefill_sequence(q, st["k_cache"], st["v_cache"], st["block_tables"][0], L, 8,
                              batch.scale, "f16")
    pos = L - 10 + np.arange(10)
    mask = np.arange(L)[None, :] <= pos[:, None]
    want = _sdpa(q, batch.k_tokens, batch.v_tokens, "f16", float(batch.scale), mask)
    assert not np.allclose(got, want, atol=1e-6)
