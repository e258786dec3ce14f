"""The C-ABI library loads and exports every entry point include/kvq.h declares (no GPU
needed: only symbol lookup and the pure host helpers are exercised)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    from int8_kv_cache_quant_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)
    names = declared_symbols()
    assert len(names) >= 10
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_host_helpers_without_gpu():
    import int8_kv_cache_quant_gb300 as k
    L = k.lib()
    assert L.kvq_version() == 1
    assert L.kvq_status_string(4) == b"workspace missing or too small"
    # pageable host memory (and NULL) is never reported as device-accessible
    import ctypes
    import numpy as np
    buf = np.zeros(64, np.uint8)
    assert L.kvq_device_accessible(ctypes.c_void_p(buf.ctypes.data)) == 0
    assert L.kvq_device_accessible(None) == 0
    # workspace sizes are pure host arithmetic
    # automatic split size: the workspace is the bound for its smallest split (64 keys)
    assert k.kvq_decode_workspace_bytes(1, 24, 32768, 256) == 512 * 24 * 256 * 4 + 512 * 24 * 16
    assert k.kvq_decode_workspace_bytes(1, 24, 32768, 256, split_rows=512) == 64 * 24 * 256 * 4 + 64 * 24 * 16
    # the automatic rule: one wave of resident CTAs (one per SM at head_dim 256, two at 128) for
    # few (sequence, KV head) units, 2048-key splits for a large batch; never below 64 keys
    assert k.kvq_decode_auto_split_rows(1, 4, 256, 32768, 152) == 864   # 38 splits x 4 = 152 CTAs
    assert k.kvq_decode_auto_split_rows(1, 4, 128, 32768, 152) == 432   # 76 x 4 = 304 (two per SM)
    assert k.kvq_decode_auto_split_rows(64, 8, 128, 16384, 152) == 2048
    assert k.kvq_decode_auto_split_rows(1, 4, 256, 4096, 152) == 112   # 37 splits x 4 = 148 CTAs
    assert k.kvq_decode_auto_split_rows(1, 4, 256, 1024, 152) == 64    # 16 x 4: four pages per CTA
    assert k.kvq_decode_auto_split_rows(1, 1, 256, 1 << 20, 152) == 1712
    assert k.kvq_decode_auto_split_rows(0, 4, 256, 4096, 152) == 0
    assert k.kvq_decode_auto_split_rows(1, 4, 192, 4096, 152) == 0
    # automatic route: one split (ctx within the smallest automatic split) is the single-CTA
    # route; beyond it the split route may be taken
    assert k.kvq_decode_workspace_bytes(1, 24, 64, 256) == 0
    assert k.kvq_decode_workspace_bytes(1, 24, 1024, 256) == 16 * 24 * 256 * 4 + 16 * 24 * 16
    # the pages' threshold route: ctx <= 2048 takes the single-CTA route
    assert k.kvq_decode_workspace_bytes(1, 24, 1024, 256, route_threshold=2048) == 0
    # verify: the decode workspace of batch * n_rows query rows
    assert k.kvq_verify_workspace_bytes(2, 4, 24, 32768, 256, split_rows=512) == \
        k.kvq_decode_workspace_bytes(8, 24, 32768, 256, split_rows=512)
    assert k.kvq_verify_workspace_bytes(2, 0, 24, 32768, 256) == 0
    # prefill: Q codes | Q scales | widened K and V of 256 tiles x 4 KV heads (2 bytes per code) |
    # their key and value scales
    # | with a full tile of history, room for the key-range split: per unit (16 query tiles x 24
    # heads) 128 rows of numerators and (m, l), and two counters
    tiles = 4 * ((30720 + 2048 + 127) // 128)
    units = 16 * 24
    assert k.kvq_prefill_workspace_bytes(2048, 24, 4, 30720, 256) == (
        2048 * 24 * 256 + 2048 * 24 * 4 + 2 * tiles * 128 * 256 * 2 + 2 * tiles * 128 * 4
        + units * 128 * 256 * 4 + units * 128 * 2 * 4 + units * 2 * 4)
    tiles = 4 * ((100 + 2048 + 127) // 128)  # history below one tile: no split region
    assert k.kvq_prefill_workspace_bytes(2048, 24, 4, 100, 256) == (
        2048 * 24 * 256 + 2048 * 24 * 4 + 2 * tiles * 128 * 256 * 2 + 2 * tiles * 128 * 4)
    # more than 16384 units (here 512 query tiles x 64 heads) never split: no split region
    tiles = 8 * ((4096 + 65536 + 127) // 128)
    assert k.kvq_prefill_workspace_bytes(65536, 64, 8, 4096, 128) == (
        65536 * 64 * 128 + 65536 * 64 * 4 + 2 * tiles * 128 * 128 * 2 + 2 * tiles * 128 * 4)
    assert k.kvq_prefill_split_tiles(65536, 64, 4096, 152) == 0
    # the split choice (host-only simulation of the dispatch onto one CTA per SM)
    assert k.kvq_prefill_split_tiles(2048, 24, 30720, 152) == 32
    assert k.kvq_prefill_split_tiles(2048, 24, 100, 152) == 0       # no full tile of history
    assert k.kvq_prefill_split_tiles(1, 24, 30000, 152) == 128      # 24 one-tile-row units
    assert k.kvq_prefill_split_tiles(130, 6, 200, 152) == 0         # too few tiles to split
    assert k.kvq_prefill_split_tiles(4096, 24, 4096, 152) == 0      # five waves: the split does not pay
    assert k.kvq_prefill_split_tiles(0, 24, 30720, 152) == 0
    assert k.kvq_prefill_split_tiles(2048, 24, 30720, 0) == 0
    # the kernel's preconditions for any split it is given: a full tile of history, and a lead
    # segment of at least one tile in every unit (r < the shortest unit's tile count)
    import numpy as np
    rng = np.random.default_rng(5)
    for _ in range(300):
        T = int(rng.integers(1, 9000))
        hq = int(rng.choice([1, 4, 6, 8, 12, 24, 32, 64]))
        hist = int(rng.integers(0, 140000))
        sms = int(rng.choice([1, 8, 132, 148, 152]))
        r = k.kvq_prefill_split_tiles(T, hq, hist, sms)
        shortest = (hist + min(127, T - 1)) // 128 + 1
        assert r == 0 or (hist >= 128 and 1 <= r < shortest), (T, hq, hist, sms, r)
    assert k.kvq_prefill_workspace_bytes(2048, 24, 4, -1, 256) == 0
    # first chunk: fp16 Q (2 bytes per element) | Q scales | fp16 K and V pieces of the chunk's tiles | scales
    tiles1 = 4 * ((4096 + 127) // 128)
    q16 = 4096 * 24 * 256 * 2
    assert k.kvq_prefill_first_workspace_bytes(4096, 24, 4, 256) == (
        q16 + 4096 * 24 * 4 + 2 * tiles1 * 128 * 256 * 2 + 2 * tiles1 * 128 * 4)
    assert k.kvq_prefill_first_workspace_bytes(4096, 24, 4, 192) == 0
    # sparse: one gather record (K row | V row | 2 scales | valid | pad) per page, KV head and slot
    assert k.kvq_sparse_workspace_bytes(2048, 1, 256) == 2048 * 16 * (2 * 256 + 16)
    assert k.kvq_sparse_workspace_bytes(100, 2, 128) == 100 * 2 * 16 * (2 * 128 + 16)
    assert k.kvq_sparse_workspace_bytes(0, 1, 256) == 0 and k.kvq_sparse_workspace_bytes(8, 1, 192) == 0


def test_invalid_arguments_rejected_before_launch():
    import int8_kv_cache_quant_gb300 as k
    L = k.lib()
    c = k.kvq._Cache(16, 16, 16, 16, 4, 16, 4, 192)  # head_dim 192 unsupported
    assert L.kvq_quant_write(ctypes.byref(c), 16, 16, 1, 16, 16, 16, 1, 1, None) == 2
    c = k.kvq._Cache(16, 16, 16, 16, 4, 8, 4, 256)  # block size 8 unsupported
    assert L.kvq_quant_write(ctypes.byref(c), 16, 16, 1, 16, 16, 16, 1, 1, None) == 2
    c = k.kvq._Cache(17, 16, 16, 16, 4, 16, 4, 256)  # misaligned K
    assert L.kvq_quant_write(ctypes.byref(c), 16, 16, 1, 16, 16, 16, 1, 1, None) == 3
    c = k.kvq._Cache(16, 16, 16, 16, 4, 16, 4, 256)
    assert L.kvq_quant_write(ctypes.byref(c), None, 16, 1, 16, 16, 16, 1, 1, None) == 1
    # decode: Hq not a multiple of Hkv; group above 16; workspace too small
    assert L.kvq_attn_decode_int8kv(ctypes.byref(c), 16, 1, 6, 16, 4, 16, 100, 1.0, 16, None, 0,
                                    None, None) == 1
    assert L.kvq_attn_decode_int8kv(ctypes.byref(c), 16, 1, 68, 16, 4, 16, 100, 1.0, 16, None, 0,
                                    None, None) == 2
    assert L.kvq_attn_decode_int8kv(ctypes.byref(c), 16, 1, 8, 16, 4000, 16, 60000, 1.0, 16, None,
                                    0, None, None) == 4
    # verify: more than 48 rows per (sequence, KV head); more than 65535 (sequence, row) pairs;
    # no rows
    assert L.kvq_attn_verify_int8kv(ctypes.byref(c), 16, 1, 7, 32, 16, 4, 16, 100, 1.0, 16, None, 0,
                                    None, None) == 2    # group 8 x 7 rows = 56
    assert L.kvq_attn_verify_int8kv(ctypes.byref(c), 16, 20000, 4, 8, 16, 4, 16, 100, 1.0, 16, None, 0,
                                    None, None) == 2
    assert L.kvq_attn_verify_int8kv(ctypes.byref(c), 16, 1, 0, 8, 16, 4, 16, 100, 1.0, 16, None, 0,
                                    None, None) == 1
    # sparse: group above 16; workspace missing or too small
    assert L.kvq_attn_sparse_int8kv(ctypes.byref(c), 16, 4, 68, 16, 16, 16, 8, 1.0, 16, 16, 1 << 20, None) == 2
    assert L.kvq_attn_sparse_int8kv(ctypes.byref(c), 16, 4, 48, 16, 16, 16, 8, 1.0, 16, None, 0, None) == 4
    assert L.kvq_attn_sparse_int8kv(ctypes.byref(c), 16, 4, 48, 16, 16, 16, 8, 1.0, 16, 16, 100, None) == 4
    # prefill: the softmax scale must be finite and positive (the kernel's exp2 relies on it)
    for bad in (0.0, -0.5, float("inf"), float("nan")):
        assert L.kvq_attn_prefill_int8(ctypes.byref(c), 16, 16, 8, 0, 16, 1, bad, 16, 16, 1 << 30,
                                       None) == 1


def test_host_tensors_refused_before_launch():
    import pytest
    # a kernel handed a pageable host pointer would fault, so the binding refuses CPU tensors
    # (outside the decode calls' zero-copy arguments, which must be mapped page-locked memory)
    import numpy as np
    import torch

    import int8_kv_cache_quant_gb300 as k
    cache = k.KVCache(4, 1, 128, device="cpu")
    rows = torch.zeros((2, 1, 128), dtype=torch.bfloat16)
    idx = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError):
        k.kvq_quant_write(cache, rows, rows, idx, idx, torch.zeros((1, 4), dtype=torch.int32))
    with pytest.raises(ValueError):
        k.kvq.kvq_attn_prefill_int8(cache, rows.view(2, 1, 128), 0, torch.zeros(4, dtype=torch.int32), 0.1,
                                    out=torch.zeros((2, 1, 128)), workspace=torch.zeros(1 << 20, dtype=torch.uint8))
    # the cache itself: its four tensors are checked like every other argument
    with pytest.raises(ValueError):
        cache.struct()
    # a pageable tensor is not device-accessible
    assert not k.kvq_device_accessible(torch.from_numpy(np.zeros(16, np.float32)))
