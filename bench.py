#!/usr/bin/env python
"""Paged decode attention benchmark: KV GB/s, fraction of HBM peak, decode tokens/s.

Workload (default): the OPT-13B-shaped decode batch — 64 sequences, 40 heads
(MHA), head_dim 128, block_size 16, fp16, lognormal context lengths (median
600, sigma 0.8, clipped to [1, 2048], seed 0), block placement from a seeded
permutation, pool sized 1.2x the demand. A step is one decode iteration of a
40-layer model's attention: one batch append in the host block manager (new
blocks / copy-on-write), the upload of slots, tables and lengths, then for
every layer reshape_and_cache of the new token and paged decode attention over
that layer's own pool. Every layer's pool is a separate 1.3 GB region, so each
step reads ~42 GB of cache — far more than L2 (no flush needed).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--block-size B] [--partition-tokens P]

Prints one JSON line (rank 0). ``--impl reference`` times the fp64 CPU oracle
on the host cores on a bounded sample of the same workload.

The default run (1 GPU) adds a ``per_config`` object: every workload of the
set measured the same way, each with fewer layers where its pools are large
(every step still reads far more than L2): the tiny batch (latency only), the
LLaMA-13B-shaped batch at each block size 8..128, the GQA shared-prefix batch,
the long-context batch at 512- and 1024-token partitions, and the 64-heads-per-
KV-head batch. Their key and value data are drawn on the device (torch's
generator, N(0, 1) rounded to the storage type, 1% of key vectors x8 for the
long-context batch) with the workloads' own lengths, shapes and block
placement: drawing several GB on the host would take minutes.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode KV GB/s & fraction of GB300 HBM peak; decode tokens/s per config"
FALLBACK_HBM_GBS = 6800.0
CONFIGS = {
    # name: layers of the model whose decode iteration one step runs
    "opt13b": dict(layers=40),
    "llama13b": dict(layers=40),
    "gqa_prefix": dict(layers=16),
    "longctx": dict(layers=8),
    "mqa": dict(layers=16),
}
# The default run's per-config measurements: (key, config, block size,
# partition tokens, layers). Layers are chosen so that a step reads several
# GB (far more than L2) while the pools stay well inside HBM.
PER_CONFIG = [("llama13b_b%d" % b, "llama13b", b, 0, 4) for b in (8, 16, 32, 64, 128)] + [
    ("gqa_prefix", "gqa_prefix", 16, 0, 16),
    ("longctx_p512", "longctx", 16, 512, 8),
    ("longctx_p1024", "longctx", 16, 1024, 8),
    ("mqa", "mqa", 16, 0, 16),
]


# ---------------------------------------------------------------- helpers

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x: float, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as td
    if not (td.is_available() and td.is_initialized()) or td.get_world_size() == 1:
        return float(x)
    t = torch.tensor([x], dtype=torch.float64, device=device or "cpu")
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(bytes_per_rank: int, world: int, ms_max: float) -> float:
    """Weak scaling: every rank processes its own batch of the same size, so
    the job moves world x bytes_per_rank in the slowest rank's time."""
    return bytes_per_rank * world / (ms_max * 1e-3) / 1e9


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(config: str, bytes_per_launch: float):
    """DRAM bytes per decode launch, from the committed ncu summary of this
    workload, if it was taken on the kernel source as it is now (the summary
    names the source file and records its sha256). The captured launch's
    traffic is scaled to this run's launch by the ratio of algorithmic bytes
    (same batch, a few tokens longer or shorter)."""
    path = os.path.join(ROOT, "profiles", f"decode_partition_{config}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"source_sha256:\s*([0-9a-f]{64})\s*\((\S+)", text)
    t = re.search(r"captured_traffic_bytes:\s*([0-9]+)", text)
    a = re.search(r"captured_algorithmic_bytes:\s*([0-9]+)", text)
    if not (m and t and a):
        return None
    src = os.path.join(ROOT, m.group(2))
    if not os.path.exists(src):
        return None
    cur = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if m.group(1) != cur:
        return None
    return round(float(t.group(1)) * bytes_per_launch / float(a.group(1)))


def profile_key(args, B, pt):
    """Name of the ncu summary of a workload (profiles/decode_partition_<key>.md):
    the block size for the LLaMA-shaped sweep, the partition size for the
    long-context batch."""
    if args.config == "llama13b":
        return f"llama13b_b{B}"
    if args.config == "longctx":
        return f"longctx_p{pt}"
    return args.config


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"pkv_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index),
                                          f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        rows = [r.split(", ") for r in open(self.path).read().strip().splitlines() if r]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[2]))
                smax.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        busy = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": float(np.median(busy)) if busy else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- our arm

def workload_shape(name, seed, block_size=0):
    """Lengths and dimensions of a workload, without drawing its token data
    (block_size 0: the workload's own, 16)."""
    import workloads as wl
    B = block_size or 16
    if name == "opt13b":
        return wl.opt13b_lengths(64, seed), 40, 40, 128, B, "f16"
    if name == "llama13b":
        return wl.llama13b_lengths(128, seed), 40, 40, 128, B, "f16"
    if name == "longctx":
        return np.array([n * 1024 for n in wl.LONGCTX_LENS_K], np.int32), 32, 8, 128, B, "bf16"
    if name == "mqa":
        return wl.llama13b_lengths(128, seed), 64, 1, 128, B, "bf16"
    if name == "gqa_prefix":
        pl, tl = wl.gqa_prefix_lengths(seed)
        lens = np.array([int(pl[s // 4]) + int(tl[s]) for s in range(256)], np.int32)
        return lens, 32, 8, 128, B, "bf16"
    raise ValueError(name)


def device_tokens(n, Hkv, D, tdt, gen, dev, outlier_frac=0.0, chunk=1 << 16):
    """n token rows [n, Hkv, D] of N(0, 1) values rounded to tdt, drawn on the
    device; with outlier_frac > 0 a (token, head) vector is x8 with that
    probability (the long-context workload's keys)."""
    import torch
    out = torch.empty((n, Hkv, D), dtype=tdt, device=dev)
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        x = torch.randn((b - a, Hkv, D), generator=gen, device=dev, dtype=torch.float32)
        if outlier_frac > 0.0:
            hit = torch.rand((b - a, Hkv, 1), generator=gen, device=dev) < outlier_frac
            x = torch.where(hit, x * 8.0, x)
        out[a:b] = x.to(tdt)
    return out


def make_workload(name, seed, block_size=16):
    import workloads as wl
    if name == "opt13b":
        return wl.opt13b(seed)
    if name == "llama13b":
        return wl.llama13b(seed, block_size=block_size)
    if name == "longctx":
        return wl.longctx(seed)
    if name == "mqa":
        return wl.mqa(seed)
    raise ValueError(name)


def decode_bytes(ctx, H, Hkv, D, out_bytes):
    """Algorithmic bytes of one decode call: every cached key and value read
    once, the queries read and the outputs written once."""
    S = len(ctx)
    return int(np.sum(ctx, dtype=np.int64)) * 2 * Hkv * D * 2 + S * H * D * 2 + S * H * D * out_bytes


def setup_pools(args, rank, dev, layers, total_steps):
    """Pools of every layer filled with the workload's cached tokens through the
    library (block manager + reshape_and_cache [+ copy_blocks]); returns the
    state the timed decode steps start from."""
    import torch
    import paged_kv_cache_118_gb300 as pk
    import workloads as wl

    seed = args.seed + rank
    devv = getattr(args, "device_values", False)
    gen = None
    if devv:
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
    if args.config == "gqa_prefix":
        pl, tl = wl.gqa_prefix_lengths(seed)
        beams, groups = 4, len(pl)
        S, H, Hkv, D, B = groups * beams, 32, 8, 128, 16
        tdt = torch.bfloat16
        p_off = np.concatenate([[0], np.cumsum(pl)]).astype(np.int64)
        t_off = np.concatenate([[0], np.cumsum(tl)]).astype(np.int64)
        L0 = np.array([int(pl[s // beams]) + int(tl[s]) + 1 for s in range(S)], np.int64)
        unique = int(np.sum(-(-pl // B))) + int(np.sum(-(-(tl + B + total_steps) // B)))
        num_blocks = int(math.ceil(1.2 * unique))
        bm = pk.BlockManager(num_blocks, B, wl.free_order(num_blocks, seed))
        pre = []
        for g in range(groups):
            bm.allocate(g * beams, int(pl[g]))
            pre.append(bm.slots(g * beams))
            for j in range(1, beams):
                bm.fork(g * beams, g * beams + j)
        tail_slots = np.full(int(t_off[-1]), -1, np.int64)
        cows = []
        for i in range(int(tl.max())):
            seqs = np.nonzero(tl > i)[0]
            sl, cow = bm.append_slots(seqs)
            tail_slots[t_off[seqs] + i] = sl
            cows.append(cow)
        cows = np.concatenate(cows)
        kc = torch.empty((layers, num_blocks, B, Hkv, D), dtype=tdt, device=dev)
        vc = torch.empty_like(kc)
        if devv:
            src = [(np.concatenate(pre), lambda: device_tokens(int(p_off[-1]), Hkv, D, tdt, gen, dev)),
                   (tail_slots, lambda: device_tokens(int(t_off[-1]), Hkv, D, tdt, gen, dev))]
        else:
            pb = wl.gqa_prefix(seed)
            up = lambda a: torch.from_numpy(a.view(np.int16)).view(tdt).to(dev)
            src = [(np.concatenate(pre), lambda: up(pb.prefix_k), lambda: up(pb.prefix_v)),
                   (tail_slots, lambda: up(pb.tail_k), lambda: up(pb.tail_v))]
        for i, part in enumerate(src):
            d_sl = torch.from_numpy(part[0]).to(dev)
            kt = part[1]()
            vt = part[1]() if devv else part[2]()
            for l in range(layers):
                if i == 1:
                    pk.pkv_copy_blocks(kc[l], vc[l], cows)
                pk.pkv_reshape_and_cache(kt, vt, kc[l], vc[l], d_sl)
            del kt, vt, d_sl
        # tokens of shared (full) blocks are read by several beams but stored once
        refs = np.array([bm.refcount(b) for b in range(num_blocks)])
        shared_extra = int(np.sum(np.maximum(refs - 1, 0))) * B
        scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
        info = dict(dtype="bf16", scale=scale, cow_pairs=int(len(cows)), groups=groups,
                    beams=beams)
    else:
        lens, H, Hkv, D, B, dname = workload_shape(args.config, seed, args.block_size)
        if getattr(args, "seqs", 0):
            if not getattr(args, "device_values", False):
                raise SystemExit("--seqs needs --device-values")
            lens = lens[:args.seqs]
        S = len(lens)
        tdt = torch.float16 if dname == "f16" else torch.bfloat16
        L0 = lens.astype(np.int64)                          # context at the first step
        final = L0 + total_steps
        num_blocks = int(math.ceil(1.2 * int(np.sum(-(-final // B)))))
        bm = pk.BlockManager(num_blocks, B, wl.free_order(num_blocks, seed))
        kc = torch.empty((layers, num_blocks, B, Hkv, D), dtype=tdt, device=dev)
        vc = torch.empty_like(kc)
        # prefill L-1 tokens of every sequence into every layer's pool
        slots = []
        for s in range(S):
            bm.allocate(s, int(L0[s]) - 1)
            if L0[s] > 1:
                slots.append(bm.slots(s))
        d_slots = torch.from_numpy(np.concatenate(slots)).to(dev)
        if devv:
            n = int(np.sum(L0 - 1))
            of = 0.01 if args.config == "longctx" else 0.0
            kp = device_tokens(n, Hkv, D, tdt, gen, dev, outlier_frac=of)
            vp = device_tokens(n, Hkv, D, tdt, gen, dev)
        else:
            batch = make_workload(args.config, seed, B)
            keep = np.ones(batch.total_tokens, bool)
            keep[batch.offsets[1:] - 1] = False
            kp = torch.from_numpy(batch.k_tokens[keep].view(np.int16)).view(tdt).to(dev)
            vp = torch.from_numpy(batch.v_tokens[keep].view(np.int16)).view(tdt).to(dev)
        for l in range(layers):
            pk.pkv_reshape_and_cache(kp, vp, kc[l], vc[l], d_slots)
        del kp, vp, d_slots
        shared_extra = 0
        info = dict(dtype=dname, scale=float(np.float32(1.0) / np.sqrt(np.float32(D))))
    torch.cuda.synchronize()
    width = int(np.max(-(-(L0 + total_steps) // B)))
    return dict(bm=bm, kc=kc, vc=vc, S=S, H=H, Hkv=Hkv, D=D, B=B, tdt=tdt, L0=L0,
                width=width, num_blocks=num_blocks, shared_extra=shared_extra, **info)


def run_ours(args, rank, world, local_rank):
    import torch
    import paged_kv_cache_118_gb300 as pk
    import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    layers = args.layers or CONFIGS[args.config]["layers"]
    pt = args.partition_tokens
    total_steps = 2 * (args.warmup + args.steps) + 1
    st = setup_pools(args, rank, dev, layers, total_steps)
    bm, kc, vc = st["bm"], st["kc"], st["vc"]
    S, H, Hkv, D, B, tdt, L0, width = (st[k] for k in ("S", "H", "Hkv", "D", "B", "tdt", "L0",
                                                       "width"))
    num_blocks = st["num_blocks"]
    dtype_name = st["dtype"]
    scale = st["scale"]

    # per-layer step inputs (resident), and pinned host copies for the e2e run
    qh = np.stack([wl.queries(S, H, D, dtype_name, args.seed, l) for l in range(layers)])
    nk, nv = zip(*[wl.new_tokens(S, Hkv, D, dtype_name, args.seed, l) for l in range(layers)])
    host = {n: torch.from_numpy(np.stack(a).view(np.int16) if n != "q" else a.view(np.int16))
            .view(tdt).pin_memory() for n, a in (("q", qh), ("k", nk), ("v", nv))}
    q = host["q"].to(dev)
    knew, vnew = host["k"].to(dev), host["v"].to(dev)
    out = torch.empty_like(q)
    out_host = torch.empty(out.shape, dtype=tdt).pin_memory()
    ws = pk.decode_workspace(S, H, Hkv, D, width, B, pt, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    seq_ids = np.arange(S, dtype=np.int64)
    d_tab = torch.empty((S, width), dtype=torch.int32, device=dev)
    d_lens = torch.empty(S, dtype=torch.int32, device=dev)
    d_new = torch.empty(S, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream()
    launches = [0]
    ctx_log = []
    ev_pairs = []

    # events of the timed region's decode calls, created up front (creating
    # them inside the layer loop costs host time the GPU may wait for)
    ev_pool = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps * layers)]

    def step(timed_kernels: bool, before=None, after=None):
        new_slots, cow = bm.append_slots(seq_ids)                       # host block manager
        tab, lens = bm.fill_tables(seq_ids, width)
        d_new.copy_(torch.from_numpy(new_slots).pin_memory(), non_blocking=True)
        d_tab.copy_(torch.from_numpy(tab).pin_memory(), non_blocking=True)
        d_lens.copy_(torch.from_numpy(lens).pin_memory(), non_blocking=True)
        ctx_log.append(lens.astype(np.int64))
        for l in range(layers):
            if before is not None:
                before(l)
            if len(cow):
                pk.pkv_copy_blocks(kc[l], vc[l], cow)
                launches[0] += -(-len(cow) // 1024)
            pk.pkv_reshape_and_cache(knew[l], vnew[l], kc[l], vc[l], d_new, err)
            if timed_kernels:
                a, b = ev_pool[len(ev_pairs)]
                a.record(stream)
            pk.pkv_paged_attention_decode(out[l], q[l], kc[l], vc[l], d_tab, d_lens, B,
                                          scale, ws, pt, err)
            if timed_kernels:
                b.record(stream)
                ev_pairs.append((a, b))
            if after is not None:
                after(l)
            launches[0] += 3

    dist = world > 1
    if dist:
        import torch.distributed as td

    def barrier():
        if dist:
            td.barrier()
        torch.cuda.synchronize()


    # ---- device-resident run
    for _ in range(args.warmup):
        step(False)
    clocks = ClockSampler(local_rank)
    if rank == 0:
        clocks.start()
    ctx_log.clear()
    ev_pairs.clear()
    launches[0] = 0
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step(True)
    t1.record(stream)
    barrier()
    clk = clocks.stop() if rank == 0 else None
    ms = max_over_ranks(t0.elapsed_time(t1), dev)
    out_bytes = 2
    # unique bytes: a token stored once but read by several beams counts once
    shared_bytes = st["shared_extra"] * 2 * Hkv * D * 2
    logical_call = [decode_bytes(c, H, Hkv, D, out_bytes) for c in ctx_log]
    per_call = [b - shared_bytes for b in logical_call]
    step_bytes = sum(per_call) * layers
    value = whole_job_gbps(step_bytes, world, ms)
    dec_ms = [a.elapsed_time(b) for a, b in ev_pairs]
    achieved = (sum(per_call) * layers) / (sum(dec_ms) * 1e-3) / 1e9
    n_launches = launches[0]
    tokens_s = S * args.steps * world / (ms * 1e-3)
    assert err.item() == 0, f"device error flag {err.item()}"

    # ---- end-to-end: host inputs in, host outputs back, inside the timed region.
    # As a serving pipeline would: the layers' q and new K/V go up on a copy
    # stream and their outputs come down on another, a group of layers at a
    # time (four groups per step), so a group waits only for its own inputs;
    # events keep a buffer from being refilled (or an output overwritten)
    # before the previous step has used (or read back) it.
    e2e = None
    if not args.no_e2e:
        for _ in range(args.warmup):
            step(False)
        ctx_log.clear()
        up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ng = min(4, layers)
        bounds = [layers * g // ng for g in range(ng + 1)]          # group g: layers [b_g, b_g+1)
        group_of = [g for g in range(ng) for _ in range(bounds[g], bounds[g + 1])]
        ev_in = [torch.cuda.Event() for _ in range(ng)]
        ev_used = [torch.cuda.Event() for _ in range(ng)]
        ev_read = [torch.cuda.Event() for _ in range(ng)]
        later = [False]

        def before(l):
            g = group_of[l]
            if l == bounds[g]:
                stream.wait_event(ev_in[g])
                if later[0]:
                    stream.wait_event(ev_read[g])

        def after(l):
            g = group_of[l]
            if l == bounds[g + 1] - 1:
                a, b = bounds[g], bounds[g + 1]
                ev_used[g].record(stream)
                down.wait_event(ev_used[g])
                with torch.cuda.stream(down):
                    out_host[a:b].copy_(out[a:b], non_blocking=True)
                ev_read[g].record(down)

        barrier()
        w0 = time.perf_counter()
        t0.record(stream)
        up.wait_stream(stream)
        down.wait_stream(stream)
        for _ in range(args.steps):
            with torch.cuda.stream(up):
                for g in range(ng):
                    a, b = bounds[g], bounds[g + 1]
                    if later[0]:
                        up.wait_event(ev_used[g])
                    q[a:b].copy_(host["q"][a:b], non_blocking=True)
                    knew[a:b].copy_(host["k"][a:b], non_blocking=True)
                    vnew[a:b].copy_(host["v"][a:b], non_blocking=True)
                    ev_in[g].record(up)
            step(False, before, after)
            later[0] = True
        stream.wait_stream(down)
        t1.record(stream)
        barrier()
        ms_e2e = max_over_ranks(max(t0.elapsed_time(t1), (time.perf_counter() - w0) * 1e3), dev)
        e_bytes = sum(decode_bytes(c, H, Hkv, D, out_bytes) - shared_bytes
                      for c in ctx_log) * layers
        h2d = (q.numel() + knew.numel() + vnew.numel()) * 2 + S * (8 + 4 + 4 * width)
        e2e = {"value": round(whole_job_gbps(e_bytes, world, ms_e2e), 2), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(out.numel() * 2)}

    peak, peak_kind = load_peaks()
    traffic = profile_traffic(profile_key(args, B, pk.pkv_decode_partition_tokens(
        S, H, Hkv, D, width, B, pt)), float(np.mean(per_call)))
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_name, "data": "synthetic",
        "config": {"workload": f"{args.config}_decode", "num_seqs": S, "num_heads": H,
                   "num_kv_heads": Hkv, "head_size": D, "block_size": B, "layers": layers,
                   "context_tokens_first_step": int(L0.sum()), "partition_tokens": pk.pkv_decode_partition_tokens(S, H, Hkv, D, width, B, pt),
                   "num_blocks": num_blocks, "seed": args.seed,
                   **({"first_seqs": args.seqs} if getattr(args, "seqs", 0) else {}),
                   "l2": "inputs larger than L2 (each step reads every layer's pool)",
                   "values": ("drawn on the device (torch generator)"
                              if getattr(args, "device_values", False) else
                              "workloads.py generators (host)"),
                   **({"groups": st["groups"], "beams": st["beams"],
                       "cow_pairs": st["cow_pairs"]} if "groups" in st else {})},
        "decode_tokens_per_s": round(tokens_s, 1),
        "logical_GBps": round(sum(logical_call) * layers * world / (ms * 1e-3) / 1e9, 2),
        "frac_of_hbm_peak": round(value / peak, 4),
        "roofline": {"bound": "hbm", "kernel": "paged decode attention (partition + reduce)",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": traffic,
                     "bytes_per_launch": int(np.mean(per_call)),
                     "launch_us": round(1e3 * float(np.mean(dec_ms)), 2)},
        "e2e": e2e, "gpu_launches": n_launches, "clocks": clk,
    }
    del kc, vc
    return line


# ---------------------------------------------------------------- swap measurement

def run_swap(args):
    """swap_blocks bandwidth: the whole opt13b batch's blocks (one layer's pool)
    out to a pinned host pool and back into other device blocks, against
    contiguous cudaMemcpyAsync copies of the same number of bytes."""
    import torch
    import paged_kv_cache_118_gb300 as pk
    import workloads as wl
    batch = make_workload("opt13b", args.seed)
    B, Hkv, D = batch.block_size, batch.num_kv_heads, batch.head_size
    L0 = batch.context_lens.astype(np.int64)
    demand = int(np.sum(-(-L0 // B)))
    n = 2 * demand + 8
    bm = pk.BlockManager(n, B, wl.free_order(n, args.seed))
    for s in range(batch.num_seqs):
        bm.allocate(s, int(L0[s]))
    dev = torch.device("cuda")
    kc = torch.empty((n, B, Hkv, D), dtype=torch.float16, device=dev)
    vc = torch.empty_like(kc)
    kc.view(torch.int16).random_(-30000, 30000)
    vc.view(torch.int16).random_(-30000, 30000)
    hk = torch.empty((demand + 8, B, Hkv, D), dtype=torch.float16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    cpu = pk.BlockManager(demand + 8, B, wl.free_order(demand + 8, args.seed + 1))
    seqs = list(range(batch.num_seqs))
    out_pairs = bm.swap(seqs, cpu)
    in_pairs = cpu.swap(seqs, bm)              # bookkeeping only: the timed copies repeat
    nbytes = 2 * len(out_pairs) * kc[0].numel() * 2
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, reps):
        fn()
        torch.cuda.synchronize()
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    reps = max(3, args.steps // 4)
    t_out = timed(lambda: pk.pkv_swap_blocks(hk, hv, kc, vc, out_pairs), reps)
    t_in = timed(lambda: pk.pkv_swap_blocks(kc, vc, hk, hv, in_pairs), reps)
    flat_d = kc.view(-1)[: nbytes // 4]
    flat_h = hk.view(-1)[: nbytes // 4]
    t_d2h = timed(lambda: (flat_h.copy_(flat_d, non_blocking=True),
                           hv.view(-1)[: nbytes // 4].copy_(vc.view(-1)[: nbytes // 4],
                                                            non_blocking=True)), reps)
    t_h2d = timed(lambda: (flat_d.copy_(flat_h, non_blocking=True),
                           vc.view(-1)[: nbytes // 4].copy_(hv.view(-1)[: nbytes // 4],
                                                            non_blocking=True)), reps)
    gbs = lambda t: round(nbytes / (t * 1e-3) / 1e9, 1)
    return {"op": "swap_blocks", "metric": "swap GB/s (blocks copied per second)",
            "unit": "GB/s", "bytes_per_swap": nbytes, "pairs": int(len(out_pairs)),
            "swap_out": gbs(t_out), "swap_in": gbs(t_in),
            "memcpy_d2h_same_bytes": gbs(t_d2h), "memcpy_h2d_same_bytes": gbs(t_h2d),
            "frac_of_memcpy": {"out": round(t_d2h / t_out, 3), "in": round(t_h2d / t_in, 3)},
            "config": {"workload": "opt13b one layer", "block_size": B,
                       "block_bytes_k_plus_v": 2 * kc[0].numel() * 2}}


# ---------------------------------------------------------------- chunked prefill

def run_prefill(args):
    """Chunked-prefill attention throughput: 16 LLaMA-13B-shaped sequences
    (40 heads, d = 128, fp16, B = 16) whose last 512 tokens of a 2k..4k-token
    context form the query chunk. FLOPs are the causal ones: 4 d H per (query,
    visible key) pair."""
    import torch
    import paged_kv_cache_118_gb300 as pk
    import workloads as wl
    from paged_kv_cache_118_gb300.cache import PagedKVCache
    rng = np.random.default_rng(args.seed)
    S, H, Hkv, D, B, C = 16, 40, 40, 128, 16, 512
    lens = rng.integers(2048, 4096, size=S, endpoint=True).astype(np.int64)
    n = int(np.sum(-(-lens // B))) + 8
    cache = PagedKVCache(n, B, Hkv, D, torch.float16, free_order=wl.free_order(n, args.seed),
                         poison=False)
    k = torch.randn(int(lens.sum()), Hkv, D, dtype=torch.float16, device="cuda")
    v = torch.randn_like(k)
    cache.prefill(range(S), lens, k, v)
    del k, v
    tables, ctx = cache.tables(range(S))
    starts = torch.arange(0, (S + 1) * C, C, dtype=torch.int32, device="cuda")
    q = torch.randn(S * C, H, D, dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    scale = 1.0 / math.sqrt(D)
    visible = sum(int(np.sum(L - C + np.arange(C) + 1)) for L in lens)
    flops = 4 * D * H * visible
    ws = pk.prefill_workspace()
    call = lambda: pk.pkv_paged_attention_prefill(out, q, cache.k_cache, cache.v_cache, tables,
                                                  ctx, starts, C, B, scale, workspace=ws,
                                                  err_flag=cache.err)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(5, args.steps)
    a.record()
    for _ in range(reps):
        call()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    assert cache.err.item() == 0
    tflops = flops / (ms * 1e-3) / 1e12
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {"bf16_tflops": 1900.0}
    peak = float(peaks.get("bf16_tflops", 1900.0))
    return {"op": "prefill", "metric": "chunked-prefill attention TFLOP/s", "unit": "TFLOP/s",
            "value": round(tflops, 1), "ms": round(ms, 4),
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "peak_source": "measured bf16 dense GEMM (fp16 runs at the same rate)"},
            "config": {"workload": "llama13b-shaped chunked prefill", "num_seqs": S,
                       "chunk": C, "context": "U[2048, 4096]", "num_heads": H,
                       "num_kv_heads": Hkv, "head_size": D, "block_size": B, "dtype": "f16"}}


# ---------------------------------------------------------------- host block manager

def run_blockmgr(args):
    """Host costs of the block manager's per-iteration work (the library's C++
    through its C ABI; microseconds per call, median of repeats)."""
    import paged_kv_cache_118_gb300 as pk
    import workloads as wl
    rng = np.random.default_rng(args.seed)
    lens = wl.opt13b_lengths(64, args.seed)
    out = {}

    def med(fn, reps=50):
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            fn()
            ts.append(time.perf_counter() - t0)
        return round(1e6 * float(np.median(ts)), 2)

    n = 2 * int(np.sum(-(-lens // 16))) + 4096
    bm = pk.BlockManager(n, 16, wl.free_order(n, args.seed))
    for s in range(64):
        bm.allocate(s, int(lens[s]))
    seqs = np.arange(64, dtype=np.int64)
    out["append_slots_64_seqs_us"] = med(lambda: bm.append_slots(seqs))
    width = int(np.max(-(-(lens + 200) // 16)))
    out["fill_tables_64_seqs_us"] = med(lambda: bm.fill_tables(seqs, width))
    prompt = rng.integers(0, 32000, 2048).astype(np.int32)
    pc = pk.BlockManager(8192, 16)
    ids = iter(range(10 ** 6))
    out["allocate_prefix_2048_tokens_miss_us"] = med(lambda: pc.allocate_prefix(
        next(ids), rng.integers(0, 32000, 2048).astype(np.int32)), reps=20)
    pc.allocate_prefix(next(ids), prompt)
    out["allocate_prefix_2048_tokens_hit_us"] = med(lambda: pc.allocate_prefix(next(ids), prompt),
                                                    reps=20)
    cpu = pk.BlockManager(n, 16)
    t0 = time.perf_counter()
    pairs = bm.swap(list(range(32)), cpu)
    out["swap_32_seqs_bookkeeping_us"] = round(1e6 * (time.perf_counter() - t0), 2)
    out["swap_32_seqs_pairs"] = int(len(pairs))
    return {"op": "block_manager", "metric": "host microseconds per call", "unit": "us",
            "results": out, "config": {"workload": "opt13b lengths, block_size 16"}}


# ---------------------------------------------------------------- oracle (CPU) arm

def _oracle_worker(args):
    """Spawned process: build the oracle's state for a share of the sequences
    (untimed), then time oracle decode steps (append + scatter + attention)
    until the time budget is used."""
    cfg, seed, seqs, budget_s, min_reps, block_size, max_tokens = args
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    sys.path.insert(0, ROOT)
    import workloads as wl
    from oracle.attention import paged_attention_decode
    from oracle.cache_ops import reshape_and_cache
    from oracle.pipeline import build_decode_state, pool_demand
    all_lens, H, Hkv, D, B, dtype = workload_shape(cfg, seed, block_size)
    lens = np.minimum(all_lens[seqs], max_tokens) if max_tokens else all_lens[seqs]
    sub = wl.decode_batch("sample", lens, H, Hkv, D, B, dtype, seed + 1000 * seqs[0],
                          outlier_frac=0.01 if cfg == "longctx" else 0.0)
    max_reps = max(min_reps, 2048)           # the pool holds this many appended tokens
    n = pool_demand(lens + max_reps, sub.block_size) + 8
    st = build_decode_state(sub, n, wl.free_order(n, seed), wl.poison_bits(sub.dtype))
    bm, kc, vc = st["bm"], st["k_cache"], st["v_cache"]
    nk, nv = wl.new_tokens(len(seqs), sub.num_kv_heads, sub.head_size, sub.dtype, seed, 0)
    done_bytes, reps, t0 = 0, 0, time.perf_counter()
    while reps < min_reps or (time.perf_counter() - t0 < budget_s and reps < max_reps):
        new_slots = np.array([bm.append_slot(s)[0] for s in range(len(seqs))], np.int64)
        reshape_and_cache(nk, nv, kc, vc, new_slots)
        ctx = np.array([bm.length(s) for s in range(len(seqs))], np.int64)
        tables = bm.padded_tables(range(len(seqs)))
        paged_attention_decode(sub.q, kc, vc, tables, ctx, sub.block_size, sub.scale, sub.dtype)
        done_bytes += decode_bytes(ctx, sub.num_heads, sub.num_kv_heads, sub.head_size, 2)
        reps += 1
    return done_bytes, time.perf_counter() - t0, reps


def oracle_throughput(cfg, seed, budget_s, min_reps=1, block_size=0):
    """Oracle GB/s on all host cores: the batch's sequences dealt round-robin
    to one spawned worker per core; each times whole oracle decode steps of
    its share for about ``budget_s`` seconds."""
    return oracle_throughputs([(cfg, block_size)], seed, budget_s, min_reps, 0)[0]


def oracle_throughputs(cases, seed, budget_s, min_reps=1, one_seq_tokens=0):
    """oracle_throughput of several (config, block size) cases through one
    pool of spawned workers (one per core); returns one
    (GB/s, workers, reps, wall seconds) per case. With one_seq_tokens > 0 each
    worker takes a single sequence of the batch (spread over it), its context
    capped at that many tokens: a bounded sample of a large batch."""
    cores = os.cpu_count() or 1
    jobs, spans = [], []
    for cfg, bs in cases:
        n_seqs = len(workload_shape(cfg, seed, bs)[0])
        workers = min(cores, n_seqs)
        spans.append((len(jobs), workers))
        shares = ([[w * n_seqs // workers] for w in range(workers)] if one_seq_tokens else
                  [list(range(w, n_seqs, workers)) for w in range(workers)])
        jobs += [(cfg, seed, sh, budget_s, min_reps, bs, one_seq_tokens) for sh in shares]
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_worker, jobs, chunksize=1)
    out = []
    for first, workers in spans:
        r = res[first:first + workers]
        wall = max(x[1] for x in r)
        out.append((sum(x[0] for x in r) / wall / 1e9, workers, min(x[2] for x in r), wall))
    return out


def run_reference(args, rank):
    """The oracle as it stands, timed on the host cores: each step is one
    bounded sample — a single layer's decode step of the whole batch."""
    gbs, cores, reps, wall = oracle_throughput(args.config, args.seed, budget_s=0.0,
                                               min_reps=args.warmup + args.steps,
                                               block_size=args.block_size)
    sample = (f"{args.config} batch, one layer per step, {reps} oracle decode steps "
              f"(append + reshape_and_cache + fp64 attention) over {cores} spawn workers")
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * wall / max(reps, 1), 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.config}_decode", "seed": args.seed},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- tiny batch latency

def run_tiny(args):
    """The tiny batch (4 sequences of 5..31 tokens, 4 heads, d = 64, B = 4,
    fp16; ~64 KB of cache, resident in L2): decode-call latency only. One call
    between two synchronisations (CUDA events around it), and the mean per
    call when calls are queued back to back."""
    import torch
    import paged_kv_cache_118_gb300 as pk
    import workloads as wl
    from paged_kv_cache_118_gb300.cache import PagedKVCache
    b = wl.tiny(args.seed)
    order = wl.free_order(wl.TINY_POOL_BLOCKS, args.seed)
    cache = PagedKVCache(wl.TINY_POOL_BLOCKS, b.block_size, b.num_kv_heads, b.head_size,
                         torch.float16, free_order=order)
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.float16).cuda()
    cache.prefill(range(b.num_seqs), b.context_lens, up(b.k_tokens), up(b.v_tokens))
    tables, ctx = cache.tables(range(b.num_seqs))
    q = up(b.q)
    out = torch.empty_like(q)
    ws = cache.workspace(b.num_seqs, b.num_heads, tables.shape[1])
    call = lambda: pk.pkv_paged_attention_decode(out, q, cache.k_cache, cache.v_cache, tables,
                                                 ctx, b.block_size, float(b.scale), ws, 0,
                                                 cache.err)
    for _ in range(20):
        call()
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    single = []
    for _ in range(200):
        a.record()
        call()
        e.record()
        torch.cuda.synchronize()
        single.append(a.elapsed_time(e) * 1e3)
    n = 1000
    a.record()
    for _ in range(n):
        call()
    e.record()
    torch.cuda.synchronize()
    assert cache.err.item() == 0
    return {"metric": "decode call latency (L2-resident; no roofline claim)", "unit": "us",
            "latency_us": round(float(np.median(single)), 2),
            "latency_us_p90": round(float(np.percentile(single, 90)), 2),
            "back_to_back_us_per_call": round(a.elapsed_time(e) * 1e3 / n, 2),
            "gpu_launches_per_call": 2,
            "config": {"workload": "tiny_decode", "num_seqs": b.num_seqs,
                       "context_lens": [int(x) for x in b.context_lens],
                       "num_heads": b.num_heads, "num_kv_heads": b.num_kv_heads,
                       "head_size": b.head_size, "block_size": b.block_size,
                       "pool_blocks": wl.TINY_POOL_BLOCKS, "dtype": "f16"}}


# ---------------------------------------------------------------- every workload

def _summary(line):
    """The per-config fields of a bench line."""
    keep = ("value", "unit", "ms_per_step", "decode_tokens_per_s", "logical_GBps",
            "frac_of_hbm_peak", "roofline", "e2e", "gpu_launches", "clocks", "config", "dtype",
            "steps", "warmup")
    return {k: line[k] for k in keep if k in line}


def run_per_config(args, cpu):
    """Every workload measured like the headline one (see PER_CONFIG); cpu maps
    a key to its oracle baseline. A failure in one entry is recorded there and
    does not stop the others."""
    import torch
    out = {}
    try:
        out["tiny"] = run_tiny(args)
    except Exception as e:          # pragma: no cover - reported in the line
        out["tiny"] = {"error": f"{type(e).__name__}: {e}"}
    for key, cfg, bs, pt, layers in PER_CONFIG:
        sub = argparse.Namespace(**vars(args))
        sub.config, sub.block_size, sub.partition_tokens, sub.layers = cfg, bs, pt, layers
        sub.steps, sub.warmup = args.per_config_steps, 3
        sub.device_values = True
        try:
            line = _summary(run_ours(sub, 0, 1, 0))
            line["cpu_baseline"] = cpu.get(key)
            out[key] = line
        except Exception as e:      # pragma: no cover - reported in the line
            out[key] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    return out


def per_config_cpu(args):
    """Oracle baselines of the per-config entries (one spawn pool; a share of
    each batch per worker for about args.per_config_cpu_budget seconds).
    Longctx at 512 and 1024 partitions share one: the oracle has no partitions."""
    cases, keys = [], []
    for key, cfg, bs, pt, layers in PER_CONFIG:
        if (cfg, bs) not in cases:
            cases.append((cfg, bs))
        keys.append((key, cases.index((cfg, bs))))
    cap = 8192
    res = oracle_throughputs(cases, args.seed, args.per_config_cpu_budget, one_seq_tokens=cap)
    out = {}
    for key, i in keys:
        gbs, cores, reps, wall = res[i]
        cfg, bs = cases[i]
        out[key] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                    "sample": f"{cfg} batch (block size {bs}): one sequence per worker, spread "
                              f"over the batch, context capped at {cap} tokens; {reps}+ oracle "
                              f"decode steps (append + reshape_and_cache + fp64 attention) per "
                              f"worker, {wall:.1f} s on {cores} spawn workers"}
    return out


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(CONFIGS), default="opt13b")
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--partition-tokens", type=int, default=0)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--block-size", type=int, default=0,
                    help="block size of the workload (0: its own, 16); llama13b sweeps 8..128")
    ap.add_argument("--seqs", type=int, default=0,
                    help="only the first N sequences of the batch (smaller profiling cases)")
    ap.add_argument("--device-values", action="store_true",
                    help="draw the cached keys/values on the device (as the per-config runs do)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-config measurements of the default run")
    ap.add_argument("--per-config-steps", type=int, default=10)
    ap.add_argument("--per-config-cpu-budget", type=float, default=2.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--op", choices=["decode", "swap", "blockmgr", "prefill", "tiny"],
                    default="decode",
                    help="decode: the headline measurement; swap: swap_blocks bandwidth; "
                         "blockmgr: host costs of the block manager; prefill: chunked-prefill "
                         "attention; tiny: decode-call latency of the tiny batch")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = dist_env()

    if args.op == "swap":
        if rank == 0:
            print(json.dumps(run_swap(args)), flush=True)
        return
    if args.op == "prefill":
        if rank == 0:
            print(json.dumps(run_prefill(args)), flush=True)
        return
    if args.op == "blockmgr":
        if rank == 0:
            print(json.dumps(run_blockmgr(args)), flush=True)
        return
    if args.op == "tiny":
        if rank == 0:
            print(json.dumps(run_tiny(args)), flush=True)
        return

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank)), flush=True)
        return

    per_config = (world == 1 and not args.no_per_config and args.config == "opt13b"
                  and args.block_size in (0, 16) and args.partition_tokens == 0
                  and args.layers == 0 and args.seqs == 0)
    cpu = None
    cpu_per = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # before the first GPU call: the oracle pools are spawned, not forked
        if per_config:
            cpu_per = per_config_cpu(args)
        gbs, cores, reps, wall = oracle_throughput(args.config, args.seed, args.cpu_budget,
                                                   block_size=args.block_size)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{args.config} batch, one layer, {reps}+ oracle decode steps per "
                         f"worker (append + reshape_and_cache + fp64 attention), "
                         f"{wall:.1f} s on {cores} spawn workers"}
    if world > 1:
        import torch
        import torch.distributed as td
        torch.cuda.set_device(local_rank)
        td.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    line["cpu_baseline"] = cpu
    if per_config and rank == 0:
        import torch
        torch.cuda.empty_cache()
        line["per_config"] = {"opt13b": dict(_summary(line), cpu_baseline=cpu),
                              **run_per_config(args, cpu_per)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as td
        td.destroy_process_group()


if __name__ == "__main__":
    main()
