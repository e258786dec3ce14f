"""kvq_attn_decode_int8kv_noalloc: the decode entry point for callers that cannot allocate
device memory (its split-K partials live in a fixed scratch array inside the library).

Called through the C ABI and checked against the regular entry point, which takes a
caller-allocated workspace, on two calls in a row (the scratch array keeps the previous
call's contents; each call must still give the regular result).  This file is collected last
so that a run that stops at the first failure has already run every other test.
"""
import numpy as np
import pytest

import workloads as W
from helpers import gpu_cache_from, norm_max_err, to_bf16_tensor, to_i32

pytestmark = pytest.mark.gpu

DESIGN_TOL = 1e-4  # the tolerance the decode tests use


def test_noalloc_decode_matches_workspace_decode_twice():
    import torch

    import int8_kv_cache_quant_gb300 as kvq
    kvq.lib()
    # split route at the decode_32k geometry (24 query / 4 KV heads, head_dim 256), two
    # sequences of different lengths, shuffled pages
    w = W.make("decode_b64", seed=901, batch=2, ctx_range=(3000, 6000), hq=24, hkv=4, d=256)
    cache, bt = gpu_cache_from(w, kvq)
    ctx = to_i32(w["ctx_lens"])
    need = kvq.kvq_decode_workspace_bytes(w["batch"], w["hq"], w["max_ctx"], w["d"])
    assert 0 < need <= kvq.kvq.NOALLOC_SCRATCH_BYTES
    for call in range(2):
        rng = np.random.default_rng(950 + call)
        q = to_bf16_tensor(W.normal_bf16(rng, (w["batch"], w["hq"], w["d"])))
        ref = kvq.kvq_attn_decode_int8kv(cache, q, bt, ctx, w["max_ctx"], w["softmax_scale"]).cpu().numpy()
        out = torch.full((w["batch"], w["hq"], w["d"]), float("nan"), dtype=torch.float32, device="cuda")
        kvq.kvq_attn_decode_int8kv_noalloc(cache, q, bt, ctx, w["max_ctx"], w["softmax_scale"], out)
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        assert norm_max_err(got, ref) <= DESIGN_TOL, (call, norm_max_err(got, ref))
    assert kvq.kvq_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    import torch

    import int8_kv_cache_quant_gb300 as kvq
    kvq.lib()
    cache = kvq.KVCache(4, 8, 128)
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((64, 4096), dtype=torch.int32, device="cuda")
    ctx = torch.zeros(64, dtype=torch.int32, device="cuda")
    out = torch.zeros((64, 32, 128), dtype=torch.float32, device="cuda")
    assert kvq.kvq_decode_workspace_bytes(64, 32, 65536, 128) > kvq.kvq.NOALLOC_SCRATCH_BYTES
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_attn_decode_int8kv_noalloc(cache, q, bt, ctx, 65536, 0.1, out)
    assert e.value.status == 4


def test_noalloc_limit_applies_to_the_split_it_takes():
    """A shape whose partials at the smallest automatic split (the bound kvq_decode_workspace_bytes
    states) exceed the scratch array, but whose partials at the split size this GPU takes fit:
    accepted, and equal to the regular entry point's result."""
    import torch

    import int8_kv_cache_quant_gb300 as kvq
    kvq.lib()
    w = W.make("decode_32k", seed=903, batch=1, ctx=32768, hq=48, hkv=6, d=256)
    assert kvq.kvq_decode_workspace_bytes(1, 48, 32768, 256) > kvq.kvq.NOALLOC_SCRATCH_BYTES
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    split = kvq.kvq_decode_auto_split_rows(1, 6, 256, 32768, sms)
    assert kvq.kvq_decode_workspace_bytes(1, 48, 32768, 256, split_rows=split) <= kvq.kvq.NOALLOC_SCRATCH_BYTES
    cache, bt = gpu_cache_from(w, kvq)
    q, ctx = to_bf16_tensor(w["q"]), to_i32(w["ctx_lens"])
    ref = kvq.kvq_attn_decode_int8kv(cache, q, bt, ctx, w["max_ctx"], w["softmax_scale"]).cpu().numpy()
    out = torch.full((1, 48, 256), float("nan"), dtype=torch.float32, device="cuda")
    kvq.kvq_attn_decode_int8kv_noalloc(cache, q, bt, ctx, w["max_ctx"], w["softmax_scale"], out)
    assert norm_max_err(out.cpu().numpy(), ref) <= DESIGN_TOL
    assert kvq.kvq_device_status() == 0
