"""The host decode-step driver end to end on the GPU: admission through the
prefix cache, appends with new blocks, preemption by swap-out when the pool
runs short, resumption by swap-in, and paged attention every iteration — each
attended sequence checked against the oracle over its whole context."""

import numpy as np
import pytest
import torch

from oracle.attention import attend_sequence
from parity import TORCH_DTYPE, assert_close
from workloads import poison_bits, round_to_storage

pytestmark = pytest.mark.gpu

B, H, HKV, D, DT = 4, 4, 2, 64, "bf16"


def _row(key):
    """Seeded N(0,1) row [H_kv, D] for a key tuple, rounded to bf16 bits."""
    rng = np.random.default_rng(list(key))
    return round_to_storage(rng.standard_normal((HKV, D), dtype=np.float32), DT)


class Source:
    """Keys/values: a prompt row depends only on (token, position), so equal
    prompt prefixes have equal cache contents; generated rows on (seq, position)."""

    def __init__(self, prompts):
        self.prompts = prompts
        self.k, self.v = {}, {}

    def rows(self, seq, p):
        if (seq, p) not in self.k:
            pr = self.prompts[seq]
            key = (1, pr[p], p) if p < len(pr) else (2, seq, p)
            self.k[(seq, p)] = _row(key + (0,))
            self.v[(seq, p)] = _row(key + (1,))
        return self.k[(seq, p)], self.v[(seq, p)]

    def kv(self, seq, positions):
        ks, vs = zip(*[self.rows(seq, int(p)) for p in positions])
        to = lambda a: torch.from_numpy(np.stack(a).view(np.int16)).view(TORCH_DTYPE[DT]).cuda()
        return to(ks), to(vs)

    def q_bits(self, seq, p):
        rng = np.random.default_rng([3, seq, p])
        return round_to_storage(rng.standard_normal((H, D), dtype=np.float32), DT)

    def q(self, seq, p):
        return torch.from_numpy(self.q_bits(seq, p).view(np.int16)).view(TORCH_DTYPE[DT]).cuda()

    def oracle(self, seq, L, scale):
        n = -(-L // B)
        kc = np.full((n, B, HKV, D), poison_bits(DT), np.uint16)
        vc = kc.copy()
        for p in range(L):
            kc[p // B, p % B], vc[p // B, p % B] = self.rows(seq, p)
        return attend_sequence(self.q_bits(seq, L - 1), kc, vc, np.arange(n), L, B, scale, DT)


def test_driver_iterations_match_oracle():
    from paged_kv_cache_118_gb300.driver import DecodeLoop
    rng = np.random.default_rng(0)
    shared = list(rng.integers(0, 50, 12))
    prompts = {0: shared + [1, 2], 1: shared + [3], 2: shared[:8] + [9, 9, 9], 3: [5] * 6,
               4: shared + [1, 2], 5: list(rng.integers(0, 50, 17))}
    src = Source(prompts)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    loop = DecodeLoop(num_gpu_blocks=22, num_cpu_blocks=64, block_size=B, num_heads=H,
                      num_kv_heads=HKV, head_size=D, dtype=torch.bfloat16, scale=scale,
                      kv_source=src.kv, q_source=src.q)
    for s, pr in prompts.items():
        loop.add_request(s, pr, max_new_tokens=12 + 3 * s)
    events = {"preempted": 0, "resumed": 0, "cached": 0, "checked": 0}
    for _ in range(200):
        if loop.idle():
            break
        res = loop.step()
        events["preempted"] += len(res.preempted)
        events["resumed"] += len(res.resumed)
        events["cached"] += sum(res.cached_tokens.values())
        if res.out is not None:
            torch.cuda.synchronize()
            for i, (s, L) in enumerate(zip(res.seqs, res.context_lens)):
                assert_close(res.out[i], src.oracle(s, L, scale), DT)
                events["checked"] += 1
    assert loop.idle()
    assert loop.gpu.err.item() == 0
    assert events["cached"] >= 8 + 12 + 12          # requests 1, 2 and 4 reuse cached blocks
    assert events["preempted"] >= 1 and events["resumed"] == events["preempted"]
    assert events["checked"] > 50
