"""The C ABI: libpagedkv.so loads, exports every function include/pagedkv.h
declares, and refuses bad arguments on the host before touching the GPU."""

import ctypes
import os
import re

import pytest

import paged_kv_cache_118_gb300 as pk

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 20
    raw = ctypes.CDLL(pk.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert set(names) == set(pk.SIGNATURES), set(names) ^ set(pk.SIGNATURES)


def test_status_strings_and_version():
    for s in range(7):
        assert pk.lib.pkv_status_string(s)
    assert b"unknown" in pk.lib.pkv_status_string(99)
    assert b"sm_103a" in pk.lib.pkv_version()


def _default_partition(S, H, Hkv, D, mb, B):
    """The default partition as the header states it: 1024 tokens when
    S * Hkv * ceil(max/1024) reaches 1024 for query groups of 2 to 16 heads per
    KV head (B >= 8), or 256 for groups of 32/64/128 (the tensor-memory path,
    which takes 2048 when S * Hkv * ceil(max/2048) reaches 256 and a partition
    holds at most 254 blocks); else 512, or 1024 for tables of 32768 tokens or
    more."""
    group = H // Hkv
    units = S * Hkv * -(-(mb * B) // 1024)
    tc = group >= 32 and 128 % group == 0 and D in (64, 128) and B >= 8 and 1024 // B + 2 <= 256
    if tc:
        if S * Hkv * -(-(mb * B) // 2048) >= 256 and 2048 // B + 2 <= 256:
            return 2048
        return 1024 if units >= 256 or mb * B >= 32768 else 512
    warp_tensor = 2 <= group and B >= 8
    if warp_tensor and units >= 1024:
        return 1024
    return 1024 if mb * B >= 32768 else 512


def test_workspace_size_formula():
    # rows = S * H * ceil(max_blocks * B / partition); each row holds D floats and an
    # (m, l) pair (the pairs padded to 16 bytes), then a 16-byte work counter
    for S, H, Hkv, D, mb, B, pt in [(64, 40, 40, 128, 128, 16, 512), (8, 32, 8, 128, 8192, 16, 512),
                                    (3, 4, 4, 64, 5, 4, 32), (1, 1, 1, 64, 1, 8, 0),
                                    (8, 32, 8, 128, 8192, 16, 0), (64, 40, 40, 128, 128, 16, 0),
                                    (256, 32, 8, 128, 98, 16, 0), (16, 32, 8, 128, 98, 16, 0),
                                    (128, 64, 1, 128, 256, 16, 0), (256, 32, 8, 128, 98, 4, 0),
                                    (16, 128, 4, 64, 40, 32, 0), (16, 32, 1, 128, 40, 16, 1024),
                                    (128, 64, 1, 128, 512, 8, 0), (96, 64, 1, 128, 256, 16, 0)]:
        eff = pt or _default_partition(S, H, Hkv, D, mb, B)
        assert pk.pkv_decode_partition_tokens(S, H, Hkv, D, mb, B, pt) == eff
        parts = -(-(mb * B) // eff)
        rows = S * H * parts
        assert (pk.pkv_decode_workspace_size(S, H, Hkv, D, mb, B, pt)
                == rows * D * 4 + -(-rows * 8 // 16) * 16 + 16)
    # the shared-prefix batch (256 beams, 32/8 heads) takes 1024-token partitions,
    # the same heads over 16 sequences 512, MHA 512; 64 heads on one KV head
    # 2048 over 128 sequences of up to 4096 tokens (1024 with 8-row blocks, whose
    # 2048-token partitions would hold 256 blocks; 1024 over 96 sequences), 512
    # over 16
    assert pk.pkv_decode_partition_tokens(256, 32, 8, 128, 98, 16, 0) == 1024
    assert pk.pkv_decode_partition_tokens(16, 32, 8, 128, 98, 16, 0) == 512
    assert pk.pkv_decode_partition_tokens(64, 40, 40, 128, 128, 16, 0) == 512
    assert pk.pkv_decode_partition_tokens(128, 64, 1, 128, 256, 16, 0) == 2048
    assert pk.pkv_decode_partition_tokens(128, 64, 1, 128, 512, 8, 0) == 1024
    assert pk.pkv_decode_partition_tokens(96, 64, 1, 128, 256, 16, 0) == 1024
    assert pk.pkv_decode_partition_tokens(16, 64, 1, 128, 256, 16, 0) == 512
    assert pk.pkv_decode_workspace_size(4, 8, 0, 128, 10, 16, 0) == 0


def _decode_status(**over):
    a = dict(out=16, out_dtype=0, q=16, k=16, v=16, kv_dtype=0, bt=16, cl=16, S=2, H=4, Hkv=4,
             D=64, nb=8, B=16, mb=4, scale=0.125, pt=0, ws=16, wsb=1 << 20, err=None)
    a.update(over)
    return pk.lib.pkv_paged_attention_decode(a["out"], a["out_dtype"], a["q"], a["k"], a["v"],
                                             a["kv_dtype"], a["bt"], a["cl"], a["S"], a["H"],
                                             a["Hkv"], a["D"], a["nb"], a["B"], a["mb"],
                                             a["scale"], a["pt"], a["ws"], a["wsb"], a["err"],
                                             None)


@pytest.mark.parametrize("over", [
    dict(q=None), dict(out=None), dict(ws=None), dict(kv_dtype=2), dict(out_dtype=7),
    dict(D=96), dict(D=256), dict(H=6, Hkv=4), dict(B=12), dict(B=512), dict(pt=48),
    dict(pt=8192), dict(S=-1), dict(nb=0), dict(mb=0), dict(q=24), dict(k=8),
    dict(scale=float("nan")), dict(S=70000)])
def test_decode_rejects_bad_arguments_on_host(over):
    assert _decode_status(**over) == pk.PKV_EINVAL


def test_decode_rejects_small_workspace_and_accepts_empty_batch():
    assert _decode_status(wsb=100) == pk.PKV_EWORKSPACE
    assert _decode_status(S=0, q=None) == pk.PKV_OK


def test_copy_blocks_host_validation():
    import numpy as np
    def st(pairs, nb=10, bb=4096, k=16, v=16):
        p = np.asarray(pairs, np.int32).reshape(-1, 2)
        return pk.lib.pkv_copy_blocks(k, v, p.ctypes.data, p.shape[0], nb, bb, None)
    assert st([(1, 10)]) == pk.PKV_ERANGE
    assert st([(-1, 2)]) == pk.PKV_ERANGE
    assert st([(1, 2), (3, 2)]) == pk.PKV_EINVAL      # duplicate destination
    assert st([(1, 2), (2, 3)]) == pk.PKV_EINVAL      # a destination is also a source
    assert st([(1, 2)], bb=100) == pk.PKV_EINVAL
    assert st([(1, 2)], k=8) == pk.PKV_EINVAL
    assert pk.lib.pkv_copy_blocks(16, 16, None, 0, 10, 4096, None) == pk.PKV_OK


def test_reshape_and_cache_host_validation():
    f = pk.lib.pkv_reshape_and_cache
    assert f(16, 16, 16, 16, 16, 0, 4, 64, 8, 16, 0, None, None) == pk.PKV_OK
    assert f(16, 16, 16, 16, None, 3, 4, 64, 8, 16, 0, None, None) == pk.PKV_EINVAL
    assert f(16, 16, 16, 16, 16, 3, 4, 60, 8, 16, 0, None, None) == pk.PKV_EINVAL
    assert f(16, 16, 16, 16, 16, 3, 4, 64, 8, 16, 2, None, None) == pk.PKV_EINVAL
    assert f(16, 24, 16, 16, 16, 3, 4, 64, 8, 16, 0, None, None) == pk.PKV_EINVAL


def _prefill_status(**over):
    a = dict(out=16, out_dtype=0, q=16, k=16, v=16, kv_dtype=0, bt=16, cl=16, qs=16, S=2, H=8,
             Hkv=8, D=128, nb=8, B=16, mb=4, mq=64, tq=64, scale=0.125, ws=16, ws_bytes=16,
             err=None)
    a.update(over)
    return pk.lib.pkv_paged_attention_prefill(a["out"], a["out_dtype"], a["q"], a["k"], a["v"],
                                              a["kv_dtype"], a["bt"], a["cl"], a["qs"], a["S"],
                                              a["H"], a["Hkv"], a["D"], a["nb"], a["B"], a["mb"],
                                              a["mq"], a["tq"], a["scale"], a["ws"], a["ws_bytes"],
                                              a["err"], None)


@pytest.mark.parametrize("over", [
    dict(q=None), dict(qs=None), dict(kv_dtype=2), dict(out_dtype=7), dict(D=96), dict(B=4),
    dict(B=12), dict(B=512), dict(H=24, Hkv=8), dict(H=6, Hkv=4), dict(mq=0), dict(S=-1),
    dict(scale=0.0), dict(scale=-0.125), dict(scale=float("inf")), dict(out=24),
    dict(ws=None), dict(ws=24), dict(ws_bytes=8), dict(tq=-1)])
def test_prefill_rejects_bad_arguments_on_host(over):
    """Host checks: head size 64/128, block sizes 8..256 (powers of two), a
    query-head group that divides the 128 rows of a query tile, a positive
    finite scale, 16-byte aligned buffers, a workspace of the stated size."""
    assert _prefill_status(**over) == pk.PKV_EINVAL


def test_prefill_accepts_an_empty_batch():
    assert _prefill_status(S=0, q=None) == pk.PKV_OK


def test_prefill_workspace_size():
    """One claim counter, padded to 16 bytes."""
    assert pk.lib.pkv_prefill_workspace_size() == 16
    assert pk.prefill_workspace("cpu").numel() == 16


def test_wait_timeout_hook_refuses_other_paths_and_bad_limits():
    """The failure-path test hook runs only the tensor-memory decode path, with a
    limit from 1 us to 1 s and an error flag to report through; everything else
    is refused before anything is queued."""
    f = pk.lib.pkv_test_decode_wait_timeout
    args = lambda H, Hkv, err, lim: (16, 0, 16, 16, 16, 1, 16, 16, 2, H, Hkv, 128, 8, 16, 4,
                                     0.125, 0, 16, 1 << 20, err, lim, None)
    assert f(*args(4, 4, 16, 2_000_000)) == pk.PKV_EINVAL       # not the tensor-memory path
    assert f(*args(64, 1, None, 2_000_000)) == pk.PKV_EINVAL    # no error flag
    assert f(*args(64, 1, 16, 10)) == pk.PKV_EINVAL             # limit below 1 us
    assert f(*args(64, 1, 16, 2 * 10 ** 9)) == pk.PKV_EINVAL    # above 1 s
