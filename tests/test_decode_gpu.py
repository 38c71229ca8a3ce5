"""GPU parity: the library's kernels against the fp64 oracle, element by
element, on seeded inputs that span several tiles, partitions and ragged
tails; invariances that must hold bitwise; device-side error reporting."""

import numpy as np
import pytest
import torch

import paged_kv_cache_118_gb300 as pk
from oracle.attention import paged_attention_decode as oracle_decode
from oracle.cache_ops import copy_blocks as oracle_copy
from oracle.pipeline import build_decode_state, build_shared_prefix_state, pool_demand
from parity import TORCH_DTYPE, assert_close, dev, gpu_decode_state
from workloads import decode_batch, free_order, gqa_prefix, poison_bits, tiny

pytestmark = pytest.mark.gpu


def run_case(batch, pt=0, extra=13, seed=1, out_dtypes=("same", "f32")):
    n = pool_demand(batch.context_lens, batch.block_size) + extra
    order = free_order(n, seed)
    ref = build_decode_state(batch, n, order, poison_bits(batch.dtype))
    cache, tables, ctx = gpu_decode_state(batch, n, order)
    # the block manager and both scatters agree bit for bit
    assert np.array_equal(tables.cpu().numpy(), ref["block_tables"])
    assert np.array_equal(ctx.cpu().numpy(), batch.context_lens)
    assert np.array_equal(cache.k_cache.view(torch.int16).cpu().numpy().view(np.uint16),
                          ref["k_cache"])
    assert np.array_equal(cache.v_cache.view(torch.int16).cpu().numpy().view(np.uint16),
                          ref["v_cache"])
    want = oracle_decode(batch.q, ref["k_cache"], ref["v_cache"], ref["block_tables"],
                         batch.context_lens, batch.block_size, batch.scale, batch.dtype)
    q = dev(batch.q, batch.dtype)
    outs = {}
    for od in out_dtypes:
        out = torch.empty(q.shape, dtype=q.dtype if od == "same" else torch.float32,
                          device="cuda")
        cache.attend(q, tables, ctx, float(batch.scale), out=out, partition_tokens=pt)
        torch.cuda.synchronize()
        assert_close(out, want, batch.dtype)
        outs[od] = out
    assert cache.err.item() == 0
    return outs, cache, tables, ctx


def test_tiny_config():
    batch = tiny(0)
    outs, *_ = run_case(batch, extra=64 - 18)


CASES = [
    # lens, H, H_kv, D, B, dtype, partition_tokens
    ((1, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1000, 2048), 40, 40, 128, 16, "f16", 512),
    ((1, 100, 513, 1537, 3000), 32, 8, 128, 16, "bf16", 512),
    ((3, 64, 65, 700), 8, 8, 64, 8, "f16", 64),
    ((2, 33, 95, 250), 6, 2, 64, 32, "bf16", 32),
    ((1, 300, 257, 1024), 16, 2, 128, 64, "f16", 256),
    ((7, 900, 4097), 10, 2, 128, 128, "bf16", 4096),
    ((95, 96, 97, 300), 4, 2, 128, 8, "f16", 96),
    ((129, 300, 64), 4, 4, 64, 128, "bf16", 32),
    ((5000,), 8, 1, 128, 16, "bf16", 0),
    ((1, 2, 3, 70), 4, 2, 64, 1, "f16", 64),
    ((33, 257, 600), 8, 8, 128, 256, "bf16", 512),
    ((6, 45), 4, 4, 128, 2, "bf16", 32),
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_against_oracle(case):
    lens, H, Hkv, D, B, dt, pt = case
    batch = decode_batch("t", lens, H, Hkv, D, B, dt, seed=len(lens) + H)
    run_case(batch, pt=pt)


def test_large_batch_uses_the_plain_work_list():
    """More than 1024 sequences: units are numbered (partition, sequence, head
    slice) with empty ones skipped instead of a compact list."""
    lens = np.random.default_rng(7).integers(1, 700, size=1100)
    batch = decode_batch("t", lens, 4, 2, 64, 16, "bf16", seed=8)
    run_case(batch, pt=256)


def test_outlier_keys_long_context():
    """1% of the keys x8: softmax weights nearly one-hot in places."""
    batch = decode_batch("t", (2500, 6000, 700), 32, 8, 128, 16, "bf16", seed=3,
                         outlier_frac=0.01)
    run_case(batch)


def test_block_size_sweep_identical_outputs():
    """Same token data placed in pools of block size 8..128: the outputs agree
    bit for bit (tiles of 32 tokens and 512-token partitions do not depend on
    the block size) and each matches the oracle."""
    outs = []
    for B in (8, 16, 32, 64, 128):
        batch = decode_batch("t", (1, 77, 513, 1400, 2049), 40, 40, 128, B, "f16", seed=11)
        o, *_ = run_case(batch, seed=B)
        outs.append(o["f32"].cpu())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_physical_placement_does_not_matter():
    batch = decode_batch("t", (40, 555, 1111), 8, 2, 128, 16, "bf16", seed=12)
    a, *_ = run_case(batch, seed=1, extra=40)
    b, *_ = run_case(batch, seed=2, extra=40)
    assert torch.equal(a["same"], b["same"]) and torch.equal(a["f32"], b["f32"])


def test_shared_prefix_copy_on_write_pipeline():
    """Beam groups: prefill once, fork, append tails step by step with
    copy-on-write; tables, copy pairs and pools match the oracle's pipeline
    bit for bit; outputs match the oracle and equal private copies bitwise."""
    pb = gqa_prefix(seed=5, groups=6, beams=4, prefix_tokens=256, max_tail=70)
    n = 400
    order = free_order(n, 9)
    ref = build_shared_prefix_state(pb, n, order, poison_bits(pb.dtype))
    from paged_kv_cache_118_gb300.cache import PagedKVCache
    cache = PagedKVCache(n, pb.block_size, pb.num_kv_heads, pb.head_size, torch.bfloat16,
                         free_order=order)
    for g in range(pb.num_groups):
        a, b = pb.prefix_offsets[g], pb.prefix_offsets[g + 1]
        cache.prefill([g * pb.beams], [b - a], dev(pb.prefix_k[a:b], "bf16"),
                      dev(pb.prefix_v[a:b], "bf16"))
        for j in range(1, pb.beams):
            cache.fork(g * pb.beams, g * pb.beams + j)
    cows = []
    for i in range(int(pb.tail_lens.max())):
        seqs = [s for s in range(pb.num_seqs) if pb.tail_lens[s] > i]
        rows = pb.tail_offsets[seqs] + i
        _, cow = cache.append(seqs, dev(pb.tail_k[rows], "bf16"), dev(pb.tail_v[rows], "bf16"))
        cows += [tuple(c) for c in cow]
    assert cows == [tuple(c) for c in ref["cow_pairs"]]
    assert len(cows) == 3 * pb.num_groups
    tables, ctx = cache.tables(range(pb.num_seqs))
    assert np.array_equal(tables.cpu().numpy(), ref["block_tables"])
    assert np.array_equal(ctx.cpu().numpy(), ref["context_lens"])
    assert np.array_equal(cache.k_cache.view(torch.int16).cpu().numpy().view(np.uint16),
                          ref["k_cache"])
    want = oracle_decode(pb.q, ref["k_cache"], ref["v_cache"], ref["block_tables"],
                         ref["context_lens"], 16, pb.scale, "bf16")
    q = dev(pb.q, "bf16")
    shared = cache.attend(q, tables, ctx, float(pb.scale))
    torch.cuda.synchronize()
    assert_close(shared, want, "bf16")
    # private copies of the same tokens
    lens, ks, vs = [], [], []
    for s in range(pb.num_seqs):
        g = s // pb.beams
        pa, pz = pb.prefix_offsets[g], pb.prefix_offsets[g + 1]
        ta, tz = pb.tail_offsets[s], pb.tail_offsets[s + 1]
        ks.append(np.concatenate([pb.prefix_k[pa:pz], pb.tail_k[ta:tz]]))
        vs.append(np.concatenate([pb.prefix_v[pa:pz], pb.tail_v[ta:tz]]))
        lens.append(len(ks[-1]))
    priv = PagedKVCache(sum(-(-L // 16) for L in lens) + 3, 16, 8, 128, torch.bfloat16,
                        free_order=free_order(sum(-(-L // 16) for L in lens) + 3, 4))
    priv.prefill(range(pb.num_seqs), lens, dev(np.concatenate(ks), "bf16"),
                 dev(np.concatenate(vs), "bf16"))
    pt, pc = priv.tables(range(pb.num_seqs))
    private = priv.attend(q, pt, pc, float(pb.scale))
    torch.cuda.synchronize()
    assert torch.equal(shared, private)
    assert cache.err.item() == 0 and priv.err.item() == 0


def test_no_partial_prefix_means_no_copies():
    pb = gqa_prefix(seed=6, groups=3, beams=4, prefix_tokens=64, max_tail=5, partial=False)
    ref = build_shared_prefix_state(pb, 100, free_order(100, 1), poison_bits("bf16"))
    assert len(ref["cow_pairs"]) == 0


def test_reshape_and_cache_padding_and_range_errors():
    kc = torch.zeros(4, 8, 2, 64, dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.randn(3, 2, 64, dtype=torch.float16, device="cuda")
    v = torch.randn_like(k)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.tensor([5, -1, 32], dtype=torch.int64, device="cuda")
    pk.pkv_reshape_and_cache(k, v, kc, vc, slots, err)
    torch.cuda.synchronize()
    assert torch.equal(kc.view(-1, 2, 64)[5], k[0]) and torch.equal(vc.view(-1, 2, 64)[5], v[0])
    assert int((kc != 0).any(dim=(1, 2, 3)).sum()) == 1
    assert err.item() & pk.PKV_DEVERR_SLOT


@pytest.mark.parametrize("n_pairs", [1, 7, 1500])
def test_copy_blocks_bitwise(n_pairs):
    rng = np.random.default_rng(n_pairs)
    nb = 2 * n_pairs + 5
    kc_h = rng.integers(0, 1 << 16, (nb, 16, 8, 128), dtype=np.uint16)
    vc_h = rng.integers(0, 1 << 16, (nb, 16, 8, 128), dtype=np.uint16)
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:n_pairs], perm[n_pairs:2 * n_pairs]], 1)
    kc, vc = dev(kc_h, "bf16"), dev(vc_h, "bf16")
    pk.pkv_copy_blocks(kc, vc, pairs)
    oracle_copy(kc_h, vc_h, pairs)
    torch.cuda.synchronize()
    assert np.array_equal(kc.view(torch.int16).cpu().numpy().view(np.uint16), kc_h)
    assert np.array_equal(vc.view(torch.int16).cpu().numpy().view(np.uint16), vc_h)


@pytest.mark.parametrize("heads", [(4, 4), (64, 1)], ids=["mha", "tcgen05"])
def test_decode_flags_bad_block_ids_and_lengths(heads):
    """Both the warp-level path and the tensor-memory path (64 query heads on
    one KV head) report a bad block id and an out-of-range length, and give
    the bad sequence a zero row."""
    batch = decode_batch("t", (40, 70, 20), heads[0], heads[1], 64, 16, "f16", seed=21)
    n = 20
    cache, tables, ctx = gpu_decode_state(batch, n, free_order(n, 0))
    q = dev(batch.q, "f16")
    good = cache.attend(q, tables, ctx, float(batch.scale)).clone()
    bad_tab = tables.clone()
    bad_tab[1, 2] = n + 5                       # outside the pool
    bad_ctx = ctx.clone()
    bad_ctx[2] = tables.shape[1] * 16 + 1       # longer than its table
    cache.err.zero_()
    out = cache.attend(q, bad_tab, bad_ctx, float(batch.scale))
    torch.cuda.synchronize()
    e = cache.err.item()
    assert e & pk.PKV_DEVERR_BLOCK_ID and e & pk.PKV_DEVERR_CONTEXT and not e & pk.PKV_DEVERR_TIMEOUT
    assert torch.equal(out[0], good[0])         # untouched sequence
    assert torch.all(out[2] == 0)               # invalid length -> zeros


def shared_tables(sizes, prefix_tokens, B, seed, diverge=0.25, max_tail=100):
    """Beam groups at the table level: the sequences of a group name the same
    physical blocks for their first prefix_tokens // B blocks (some beams only
    for a random shorter run of them), then blocks of their own. Returns the
    tables (-1 padded), context lengths and the number of physical blocks,
    placed by a seeded permutation."""
    rng = np.random.default_rng(seed)
    nbp = prefix_tokens // B
    rows, lens, nxt = [], [], 0
    for n in sizes:
        shared = list(range(nxt, nxt + nbp))
        nxt += nbp
        for _ in range(n):
            L = nbp * B + int(rng.integers(1, max_tail, endpoint=True))
            keep = nbp if rng.random() >= diverge else int(rng.integers(0, nbp + 1))
            own = -(-L // B) - keep
            rows.append(shared[:keep] + list(range(nxt, nxt + own)))
            nxt += own
            lens.append(L)
    place = rng.permutation(nxt + 5)
    w = max(len(r) for r in rows)
    tables = np.full((len(rows), w), -1, np.int32)
    for i, r in enumerate(rows):
        tables[i, :len(r)] = place[r]
    return tables, np.array(lens, np.int32), nxt + 5


def privatize(tables, k, v, B):
    """The same token data with every block of every sequence copied to a block
    of its own (no two sequences share one)."""
    rows, srcs = [], []
    for r in tables:
        ids = [int(x) for x in r if x >= 0]
        rows.append(list(range(len(srcs), len(srcs) + len(ids))))
        srcs += ids
    pt = np.full(tables.shape, -1, np.int32)
    for i, r in enumerate(rows):
        pt[i, :len(r)] = r
    return pt, k[srcs], v[srcs]


SHARED_CASES = [
    # beams per group, prefix tokens, H, H_kv, D, B, dtype, partition_tokens
    ((3, 5, 1, 4, 2, 7), 300, 32, 8, 128, 16, "bf16", 64),     # 4 heads: 4 sequences a unit
    ((4, 4, 4, 4, 4, 4), 1040, 32, 8, 128, 16, "bf16", 512),
    ((2, 9, 3, 11), 520, 16, 8, 128, 32, "f16", 128),          # 2 heads: 8 sequences a unit
    ((3, 3, 2, 6), 256, 64, 8, 64, 8, "f16", 64),              # 8 heads: 2 sequences a unit
    ((5, 4), 200, 32, 2, 128, 16, "bf16", 32),                 # 16 heads in two slices of 8
    ((6, 1, 6), 192, 24, 4, 128, 64, "bf16", 64),              # 6 heads: 2 sequences a unit
]


@pytest.mark.parametrize("case", SHARED_CASES, ids=[f"s{i}" for i in range(len(SHARED_CASES))])
def test_shared_prefix_runs(case):
    """Sequences whose blocks for a partition are the same physical blocks are
    served together on the tensor path: the outputs match the oracle, and equal
    bit for bit those of the same data with no block shared."""
    sizes, P, H, Hkv, D, B, dt, pt = case
    tables, lens, nb = shared_tables(sizes, P, B, seed=sum(sizes) + H)
    rng = np.random.default_rng(len(sizes) * 7 + D)
    from workloads import normal_bits
    kc = normal_bits(rng, (nb, B, Hkv, D), dt)
    vc = normal_bits(rng, (nb, B, Hkv, D), dt)
    q = normal_bits(rng, (len(lens), H, D), dt)
    scale = np.float32(1.0) / np.sqrt(np.float32(D))
    want = oracle_decode(q, kc, vc, tables, lens, B, scale, dt)
    ptab, pk_, pv_ = privatize(tables, kc, vc, B)
    outs = []
    for tab, k, v in ((tables, kc, vc), (ptab, pk_, pv_)):
        out = torch.empty(q.shape, dtype=TORCH_DTYPE[dt], device="cuda")
        tt = torch.from_numpy(tab).cuda()
        ws = pk.decode_workspace(len(lens), H, Hkv, D, tab.shape[1], B, pt)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pk.pkv_paged_attention_decode(out, dev(q, dt), dev(k, dt), dev(v, dt), tt,
                                      torch.from_numpy(lens).cuda(), B, float(scale), ws,
                                      partition_tokens=pt, err_flag=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert_close(out, want, dt)
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


TC_CASES = [
    # lens, H, H_kv, D, B, dtype, partition_tokens: groups of 32..128 query heads
    # per KV head run on the tensor-memory path
    ((1, 63, 64, 65, 700, 1500), 64, 2, 128, 16, "bf16", 512),
    ((5, 300, 2049), 64, 2, 128, 32, "f16", 256),
    ((77, 1000, 2), 64, 1, 64, 8, "bf16", 64),
    ((3, 129, 4100), 128, 1, 128, 128, "f16", 0),
    ((33, 70, 130), 32, 1, 64, 64, "f16", 128),
    ((20, 1024, 517), 96, 3, 128, 16, "bf16", 512),
    # 64-key tiles gathered from blocks of 8, 16 and 64 rows, two 128-byte
    # lines per row; one group of 128 heads (a single copy of the query rows)
    ((9, 200, 1031), 64, 1, 128, 8, "f16", 128),
    ((17, 1500, 64), 128, 1, 128, 16, "bf16", 512),
    ((50, 640, 3), 32, 1, 128, 64, "bf16", 256),
    # a long context: the default 1024-token partitions, 40 partials per row
    # (the four-warp reduce); one copy of 128 heads at d = 64; blocks of 256
    # rows (tiles inside one block)
    ((40000, 5, 33000), 64, 1, 128, 16, "bf16", 0),
    ((7, 777), 128, 1, 64, 32, "bf16", 256),
    ((1, 2, 3, 4, 100, 513), 64, 1, 128, 256, "f16", 512),
]


@pytest.mark.parametrize("case", TC_CASES, ids=[f"tc{i}" for i in range(len(TC_CASES))])
def test_large_groups_against_oracle(case):
    lens, H, Hkv, D, B, dt, pt = case
    batch = decode_batch("t", lens, H, Hkv, D, B, dt, seed=len(lens) + H + D)
    run_case(batch, pt=pt)


def test_large_groups_many_sequences():
    """More sequences than the compact work list takes: every (partition,
    sequence, KV head) is numbered and the empty ones are skipped."""
    rng = np.random.default_rng(5)
    lens = tuple(int(x) for x in rng.integers(1, 200, 1100))
    batch = decode_batch("t", lens, 32, 1, 64, 16, "f16", seed=6)
    run_case(batch, pt=64)


def test_large_groups_outlier_keys():
    """Nearly one-hot softmax rows on the tensor-memory path (rescales of the
    output rows in tensor memory)."""
    batch = decode_batch("t", (3000, 700, 129), 64, 2, 128, 16, "bf16", seed=21,
                         outlier_frac=0.02)
    run_case(batch)
