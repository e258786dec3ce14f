"""Pages past 2^31 bytes of the cache.

A pool of 150,000 pages at 4 KV heads and head_dim 256 holds 2.46 GB of K codes (and as much of
V), so a page above 131,072 starts past byte 2^31 of each array: every address the kernels form
from a page id must be 64-bit.  Each entry point runs once on the workload's own small pool and
once with its block table moved to the top of the large pool.  Gates: the outputs, and the codes
and scales written, are bit-identical between the two; the decode output also matches the
oracle's FP64 reference."""
import numpy as np
import pytest

import workloads as W
from helpers import host_cache_from, norm_max_err, to_bf16_tensor, to_i32

pytestmark = pytest.mark.gpu

POOL = 150_000
HKV, D = 4, 256
assert POOL * HKV * D * 16 > 2 ** 31 + 2 ** 28  # the top pages sit well past byte 2^31


@pytest.fixture(scope="module")
def kvq():
    import int8_kv_cache_quant_gb300 as k
    k.lib()
    return k


@pytest.fixture(scope="module")
def big(kvq):
    return kvq.KVCache(POOL, HKV, D)


def _fill(kvq, cache, w, table):
    kvq.kvq_quant_write(cache, to_bf16_tensor(w["k_fill"]), to_bf16_tensor(w["v_fill"]), to_i32(w["fill_seq"]),
                        to_i32(w["fill_pos"]), to_i32(table))


def _high(w):
    t = w["block_table"]  # rows padded with -1 past each sequence's last page
    return np.where(t >= 0, t + (POOL - w["num_blocks"]), -1).astype(np.int32)


def _same(a, b):
    return np.array_equal(np.asarray(a).view(np.uint32), np.asarray(b).view(np.uint32))


def _pages_equal(small, big, table_small, table_big):
    keep = table_small.ravel() >= 0
    ts, tb = table_small.ravel()[keep], table_big.ravel()[keep]
    import torch
    ts_t, tb_t = torch.from_numpy(ts.astype(np.int64)).cuda(), torch.from_numpy(tb.astype(np.int64)).cuda()
    for name in ("k", "v", "k_scale", "v_scale"):
        a = getattr(small, name).index_select(0, ts_t)
        b = getattr(big, name).index_select(0, tb_t)
        assert torch.equal(a.view(torch.int8) if a.dtype != torch.int8 else a,
                           b.view(torch.int8) if b.dtype != torch.int8 else b), name


def test_decode_and_fused_step_on_top_pages(kvq, oracle, big):
    w = W.make("decode_b64", seed=1200, batch=3, ctx_range=(300, 3000), hq=24, hkv=HKV, d=D)
    small = kvq.KVCache(w["num_blocks"], HKV, D)
    hi = _high(w)
    _fill(kvq, small, w, w["block_table"])
    _fill(kvq, big, w, hi)
    _pages_equal(small, big, w["block_table"], hi)
    q, ctx = to_bf16_tensor(w["q"]), to_i32(w["ctx_lens"])
    for route in (1, 2):
        a = kvq.kvq_attn_decode_int8kv(small, q, to_i32(w["block_table"]), ctx, w["max_ctx"], w["softmax_scale"],
                                       force_route=route).cpu().numpy()
        b = kvq.kvq_attn_decode_int8kv(big, q, to_i32(hi), ctx, w["max_ctx"], w["softmax_scale"],
                                       force_route=route).cpu().numpy()
        assert _same(a, b), route
    ref = oracle.decode_f64(host_cache_from(w, oracle), w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    assert norm_max_err(b, ref) <= 1e-4
    # the fused step rewrites each sequence's newest token into its top page
    kn, vn = to_bf16_tensor(w["k_new"]), to_bf16_tensor(w["v_new"])
    a = kvq.kvq_decode_step_int8kv(small, kn, vn, q, to_i32(w["block_table"]), ctx, w["max_ctx"],
                                   w["softmax_scale"]).cpu().numpy()
    b = kvq.kvq_decode_step_int8kv(big, kn, vn, q, to_i32(hi), ctx, w["max_ctx"], w["softmax_scale"]).cpu().numpy()
    assert _same(a, b)
    _pages_equal(small, big, w["block_table"], hi)
    assert kvq.kvq_device_status() == 0


def test_prefill_and_first_chunk_on_top_pages(kvq, big):
    w = W.make("prefill_32k", seed=1210, history=1500, chunk=300, hq=8, hkv=HKV, d=D)
    small = kvq.KVCache(w["num_blocks"], HKV, D)
    hi = _high(w)
    _fill(kvq, small, w, w["block_table"])
    _fill(kvq, big, w, hi)
    q = to_bf16_tensor(w["q"])
    a = kvq.kvq_attn_prefill_int8(small, q, w["history"], to_i32(w["block_table"][0]), w["softmax_scale"])
    b = kvq.kvq_attn_prefill_int8(big, q, w["history"], to_i32(hi[0]), w["softmax_scale"])
    assert _same(a.cpu().numpy(), b.cpu().numpy())
    # the first chunk writes its K/V through its own pre-pass
    T = 400
    kf, vf = to_bf16_tensor(w["k_fill"][:T]), to_bf16_tensor(w["v_fill"][:T])
    qf = to_bf16_tensor(W.normal_bf16(np.random.default_rng(1211), (T, 8, D)))
    small2 = kvq.KVCache(w["num_blocks"], HKV, D)
    a = kvq.kvq_attn_prefill_first_bf16(small2, qf, kf, vf, to_i32(w["block_table"][0]), w["softmax_scale"])
    b = kvq.kvq_attn_prefill_first_bf16(big, qf, kf, vf, to_i32(hi[0]), w["softmax_scale"])
    assert _same(a.cpu().numpy(), b.cpu().numpy())
    n = (T + 15) // 16
    _pages_equal(small2, big, w["block_table"][0][:n], hi[0][:n])
    assert kvq.kvq_device_status() == 0


def test_sparse_on_top_pages(kvq, big):
    w = W.make("sparse_32k", seed=1220, ctx=2000, n_queries=30, n_sample=400, hq=8, hkv=HKV)
    small = kvq.KVCache(w["num_blocks"], HKV, D)
    hi = _high(w)
    _fill(kvq, small, w, w["block_table"])
    _fill(kvq, big, w, hi)
    q, offs, cells = to_bf16_tensor(w["q"]), to_i32(w["cell_offsets"]), to_i32(w["cells"])
    a = kvq.kvq_attn_sparse_int8kv(small, q, offs, cells, to_i32(w["block_table"][0]), w["softmax_scale"])
    b = kvq.kvq_attn_sparse_int8kv(big, q, offs, cells, to_i32(hi[0]), w["softmax_scale"])
    assert _same(a.cpu().numpy(), b.cpu().numpy())
    assert kvq.kvq_device_status() == 0
