"""Pins of the oracle's decode attention against what the pages and the
mathematics fix, independently of the oracle's own code:

* closed forms: one token (o = v0), equal keys or zero query (o = mean v),
  two tokens (logistic weights, scipy's expit);
* a library routine: torch's scaled_dot_product_attention (float64, CPU) on the
  contiguous token data, which involves no block table at all;
* invariants from the pages: relabelling physical blocks changes nothing
  (the kernel reads blocks in the sequence's own order), shared-prefix tables
  give the same output as private copies;
* planted mistakes in the oracle (per-block softmax, unmasked tail, wrong
  head grouping, missing scale, wrong table walk) each fail one of the pins.
"""

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import oracle.attention as att
from oracle.formats import decode_bits
from oracle.pipeline import build_decode_state, build_shared_prefix_state, pool_demand
from workloads import decode_batch, free_order, gqa_prefix, poison_bits

CASES = [
    # lens, H, H_kv, d, B, dtype
    ((1, 2, 3, 17, 40, 64), 4, 4, 64, 4, "f16"),
    ((5, 33, 64, 100), 8, 2, 128, 16, "bf16"),
    ((7, 129, 31, 8), 4, 1, 64, 8, "f16"),
    ((300, 1, 45), 6, 3, 128, 32, "bf16"),
]


def _state(batch, seed=1, extra=7):
    n = pool_demand(batch.context_lens, batch.block_size) + extra
    return build_decode_state(batch, n, free_order(n, seed), poison_bits(batch.dtype))


def _oracle(batch, st):
    return att.paged_attention_decode(batch.q, st["k_cache"], st["v_cache"], st["block_tables"],
                                      batch.context_lens, batch.block_size, batch.scale, batch.dtype)


def _sdpa(batch):
    """torch SDPA on each sequence's contiguous keys/values (no block table)."""
    out = np.empty((batch.num_seqs, batch.num_heads, batch.head_size))
    for s in range(batch.num_seqs):
        a, b = int(batch.offsets[s]), int(batch.offsets[s + 1])
        q = torch.from_numpy(decode_bits(batch.q[s], batch.dtype))[None, :, None, :]
        k = torch.from_numpy(decode_bits(batch.k_tokens[a:b], batch.dtype)).permute(1, 0, 2)[None]
        v = torch.from_numpy(decode_bits(batch.v_tokens[a:b], batch.dtype)).permute(1, 0, 2)[None]
        o = F.scaled_dot_product_attention(q, k, v, scale=float(batch.scale),
                                           enable_gqa=batch.num_heads != batch.num_kv_heads)
        out[s] = o[0, :, 0, :].numpy()
    return out


@pytest.mark.parametrize("case", CASES)
def test_matches_library_attention(case):
    lens, H, Hkv, d, B, dt = case
    batch = decode_batch("t", lens, H, Hkv, d, B, dt, seed=3)
    got = _oracle(batch, _state(batch))
    ref = _sdpa(batch)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_single_token_returns_its_value():
    batch = decode_batch("t", (1, 1, 1), 8, 2, 64, 16, "bf16", seed=4)
    got = _oracle(batch, _state(batch))
    v = decode_bits(batch.v_tokens, "bf16")            # [3, H_kv, d]
    for s in range(3):
        for h in range(8):
            assert np.array_equal(got[s, h], v[s, h // 4])


def test_equal_keys_or_zero_query_average_the_values():
    batch = decode_batch("t", (37, 5), 4, 4, 64, 8, "f16", seed=5)
    batch.k_tokens[:] = batch.k_tokens[0]             # every key identical
    got = _oracle(batch, _state(batch))
    v = decode_bits(batch.v_tokens, "f16")
    for s in range(2):
        a, b = batch.offsets[s], batch.offsets[s + 1]
        np.testing.assert_allclose(got[s], v[a:b].mean(axis=0), rtol=0, atol=1e-13)
    batch = decode_batch("t", (37, 5), 4, 4, 64, 8, "f16", seed=6)
    batch.q[:] = 0
    got = _oracle(batch, _state(batch))
    v = decode_bits(batch.v_tokens, "f16")
    for s in range(2):
        a, b = batch.offsets[s], batch.offsets[s + 1]
        np.testing.assert_allclose(got[s], v[a:b].mean(axis=0), rtol=0, atol=1e-13)


def test_two_tokens_logistic_weights():
    batch = decode_batch("t", (2, 2), 2, 1, 64, 4, "bf16", seed=7)
    got = _oracle(batch, _state(batch))
    k = decode_bits(batch.k_tokens, "bf16")
    v = decode_bits(batch.v_tokens, "bf16")
    q = decode_bits(batch.q, "bf16")
    sc = float(batch.scale)
    for s in range(2):
        a = batch.offsets[s]
        for h in range(2):
            d0 = sc * float(q[s, h] @ k[a, 0])
            d1 = sc * float(q[s, h] @ k[a + 1, 0])
            w0 = scipy.special.expit(d0 - d1)
            want = w0 * v[a, 0] + (1.0 - w0) * v[a + 1, 0]
            np.testing.assert_allclose(got[s, h], want, rtol=0, atol=1e-13)


def test_output_within_value_hull():
    batch = decode_batch("t", (50, 3, 90), 4, 2, 64, 16, "f16", seed=8)
    got = _oracle(batch, _state(batch))
    v = decode_bits(batch.v_tokens, "f16")
    for s in range(3):
        a, b = batch.offsets[s], batch.offsets[s + 1]
        for h in range(4):
            lo = v[a:b, h // 2].min(axis=0)
            hi = v[a:b, h // 2].max(axis=0)
            assert np.all(got[s, h] >= lo - 1e-12) and np.all(got[s, h] <= hi + 1e-12)


def test_relabelling_physical_blocks_changes_nothing():
    batch = decode_batch("t", (5, 9, 17, 31), 4, 4, 64, 4, "f16", seed=9)
    st = _state(batch, extra=20)
    base = _oracle(batch, st)
    n = st["k_cache"].shape[0]
    perm = np.random.default_rng(0).permutation(n)      # old id i -> new id perm[i]
    kc = np.empty_like(st["k_cache"]); kc[perm] = st["k_cache"]
    vc = np.empty_like(st["v_cache"]); vc[perm] = st["v_cache"]
    tab = st["block_tables"].copy()
    tab[tab >= 0] = perm[tab[tab >= 0]]
    got = att.paged_attention_decode(batch.q, kc, vc, tab, batch.context_lens, 4,
                                     batch.scale, "f16")
    assert np.array_equal(got, base)


def test_shared_prefix_equals_private_copies():
    pb = gqa_prefix(seed=2, groups=3, beams=4, prefix_tokens=64, max_partial=15, max_tail=40)
    n = 200
    st = build_shared_prefix_state(pb, n, free_order(n, 3), poison_bits(pb.dtype))
    shared = att.paged_attention_decode(pb.q, st["k_cache"], st["v_cache"], st["block_tables"],
                                        st["context_lens"], pb.block_size, pb.scale, pb.dtype)
    # the same token data laid out as private sequences (no sharing, no copies)
    lens, ks, vs = [], [], []
    for s in range(pb.num_seqs):
        g = s // pb.beams
        pa, pz = pb.prefix_offsets[g], pb.prefix_offsets[g + 1]
        ta, tz = pb.tail_offsets[s], pb.tail_offsets[s + 1]
        ks.append(np.concatenate([pb.prefix_k[pa:pz], pb.tail_k[ta:tz]]))
        vs.append(np.concatenate([pb.prefix_v[pa:pz], pb.tail_v[ta:tz]]))
        lens.append(len(ks[-1]))
    priv = decode_batch("p", lens, pb.num_heads, pb.num_kv_heads, pb.head_size, pb.block_size,
                        pb.dtype, seed=0)
    priv.k_tokens = np.concatenate(ks); priv.v_tokens = np.concatenate(vs); priv.q = pb.q
    assert np.array_equal(priv.context_lens, st["context_lens"])
    private = _oracle(priv, _state(priv))
    assert np.array_equal(shared, private)
    assert len(st["cow_pairs"]) == 3 * 3          # beams-1 copies per group


# ---- planted mistakes: each must be caught by a pin above --------------------

def _per_block_softmax(q_bits, k_cache, v_cache, table_row, L, B, scale, dtype):
    """The rejected variant: softmax inside each block, block results added."""
    H = q_bits.shape[0]
    Hkv = k_cache.shape[2]
    K = decode_bits(att.gather_sequence(k_cache, table_row, L, B), dtype)
    V = decode_bits(att.gather_sequence(v_cache, table_row, L, B), dtype)
    Q = decode_bits(q_bits, dtype)
    out = np.zeros((H, Q.shape[1]))
    for h in range(H):
        g = h // (H // Hkv)
        for j0 in range(0, L, B):
            s = float(np.float32(scale)) * (K[j0:j0 + B, g] @ Q[h])
            out[h] += att.softmax_weights(s) @ V[j0:j0 + B, g]
    return out


def _no_tail_mask(cache_bits, table_row, L, B):
    n = -(-L // B)
    return cache_bits[np.asarray(table_row[:n])].reshape(n * B, *cache_bits.shape[2:])


def _walk_whole_row(cache_bits, table_row, L, B):
    ids = np.asarray(table_row)
    ids = np.where(ids < 0, 0, ids)
    return cache_bits[ids].reshape(-1, *cache_bits.shape[2:])[:L]


@pytest.mark.parametrize("mutant", ["per_block", "no_mask", "head_mod", "no_scale", "reverse_blocks"])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    if mutant == "per_block":
        monkeypatch.setattr(att, "attend_sequence", _per_block_softmax)
    elif mutant == "no_mask":
        monkeypatch.setattr(att, "gather_sequence", _no_tail_mask)
    elif mutant == "head_mod":
        monkeypatch.setattr(att, "kv_head_of", lambda h, H, Hkv: h % Hkv)
    elif mutant == "no_scale":
        orig = att.softmax_weights
        monkeypatch.setattr(att, "softmax_weights", lambda s: orig(s * 8.0))
    elif mutant == "reverse_blocks":
        def rev(cache_bits, table_row, L, B):
            n = -(-L // B)
            return _walk_whole_row(cache_bits, np.asarray(table_row[:n])[::-1], L, B)
        monkeypatch.setattr(att, "gather_sequence", rev)
    caught = 0
    for case in CASES:
        lens, H, Hkv, d, B, dt = case
        batch = decode_batch("t", lens, H, Hkv, d, B, dt, seed=3)
        got = _oracle(batch, _state(batch))
        ref = _sdpa(batch)
        if not np.all(np.isfinite(got)) or not np.allclose(got, ref, rtol=0, atol=1e-12):
            caught += 1
    assert caught >= 1
