"""kvq_attn_decode_int8kv on the GPU against the oracle (FP64 Part A).

Gates: the spec acceptance is <= 5e-3 normalised max-abs error against the FP64
reference over the dequantised K/V (and <= 2e-3 against the int8-emulated output, which for
decode is the same Part A: decode quantises neither Q nor P).  The design itself keeps
~22-bit softmax weights (fp16 hi + lo) and fp32 accumulation, so errors land near 1e-6;
DESIGN_TOL = 1e-4 catches regressions well inside the gate.
"""
import numpy as np
import pytest

import workloads as W
from helpers import gpu_cache_from, host_cache_from, norm_max_err, sample_units, to_bf16_tensor, to_i32

pytestmark = pytest.mark.gpu

GATE = 2e-3
DESIGN_TOL = 1e-4


@pytest.fixture(scope="module")
def kvq():
    import int8_kv_cache_quant_gb300 as k
    k.lib()
    return k


def _run(kvq, w, **opts):
    cache, bt = gpu_cache_from(w, kvq)
    q = to_bf16_tensor(w["q"])
    ctx = to_i32(w["ctx_lens"])
    out = kvq.kvq_attn_decode_int8kv(cache, q, bt, ctx, w["max_ctx"], w["softmax_scale"], **opts)
    return out.cpu().numpy(), cache, bt


@pytest.mark.parametrize("route", [1, 2])
@pytest.mark.parametrize("ctx", [1, 15, 17, 511, 513, 1000])
def test_small_contexts_both_routes(kvq, oracle, route, ctx):
    w = W.make("decode_32k", seed=200 + ctx, batch=2, ctx=ctx, hq=24, hkv=4, d=256)
    got, _, _ = _run(kvq, w, force_route=route)
    hc = host_cache_from(w, oracle)
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    err = norm_max_err(got, ref)
    assert err <= GATE and err <= DESIGN_TOL, err
    assert kvq.kvq_device_status() == 0


@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (128, 8, 1), (256, 16, 2), (128, 4, 4),
                                      (128, 32, 2), (256, 12, 1), (256, 16, 1)])
def test_head_geometries(kvq, oracle, d, hq, hkv):
    """GQA groups 1..8 take the one-row kernel; 12 and 16 take the rows kernel with the group's
    heads as its rows (two 8-row n-tiles)."""
    w = W.make("decode_b64", seed=300 + hq, batch=5, ctx_range=(1, 1500), hq=hq, hkv=hkv, d=d)
    hc = host_cache_from(w, oracle)
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    for route in (1, 2):
        got, _, _ = _run(kvq, w, force_route=route, split_rows=128)
        err = norm_max_err(got, ref)
        assert err <= DESIGN_TOL, (route, err)


@pytest.mark.parametrize("split", [16, 64, 512, 2048])
def test_split_size_invariance(kvq, oracle, split):
    w = W.make("decode_b64", seed=400, batch=3, ctx_range=(900, 3000), hq=24, hkv=4, d=256)
    got, _, _ = _run(kvq, w, force_route=2, split_rows=split)
    hc = host_cache_from(w, oracle)
    ref = oracle.decode_split_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"], split)
    assert norm_max_err(got, ref) <= DESIGN_TOL


def test_zero_context_and_mixed_lengths(kvq, oracle):
    w = W.make("decode_b64", seed=401, batch=4, ctx_range=(100, 700), hq=8, hkv=2, d=128)
    w["ctx_lens"] = w["ctx_lens"].copy()
    w["ctx_lens"][1] = 0
    got, _, _ = _run(kvq, w, force_route=2, split_rows=64)
    assert not got[1].any()
    hc = host_cache_from(w, oracle)
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    assert norm_max_err(got, ref) <= DESIGN_TOL


def test_bad_block_is_flagged_not_faulted(kvq):
    w = W.make("decode_32k", seed=402, batch=1, ctx=64, hq=6, hkv=1, d=128)
    cache, bt = gpu_cache_from(w, kvq)
    kvq.kvq_device_status()
    bad = bt.clone()
    bad[0, 2] = 10 ** 6
    q = to_bf16_tensor(w["q"])
    out = kvq.kvq_attn_decode_int8kv(cache, q, bad, to_i32(w["ctx_lens"]), 64, w["softmax_scale"])
    flags = kvq.kvq_device_status()
    assert flags & kvq.kvq.DEV_BAD_BLOCK
    assert np.isfinite(out.cpu().numpy()).all()


@pytest.mark.parametrize("route", [None, 1])
def test_decode_1k_full(kvq, oracle, route):
    """Workload decode_1k: ctx 1024, contiguous cache, on the automatic route (split-K with the
    GPU-sized split: 64-key splits on 152 SMs, then the merge) and forced onto the single-CTA
    route: every output against FP64."""
    w = W.make("decode_1k")
    got, _, _ = _run(kvq, w) if route is None else _run(kvq, w, force_route=route)
    hc = host_cache_from(w, oracle)
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    err = norm_max_err(got, ref)
    print("decode_1k normalised max err", err)
    assert err <= GATE and err <= DESIGN_TOL


def test_decode_32k_full(kvq, oracle):
    """Workload decode_32k at full size at the split size its configuration states (split-K with
    512-key splits, shuffled pages, K outliers; the benchmark's own call, the fused step with the
    automatic split, is checked in full in test_gpu_step.py): every output against FP64."""
    w = W.make("decode_32k")
    got, _, _ = _run(kvq, w, split_rows=w["split_rows"])
    hc = host_cache_from(w, oracle)
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    err = norm_max_err(got, ref)
    print("decode_32k normalised max err", err)
    assert err <= GATE and err <= DESIGN_TOL


def test_decode_128k_fused_step(kvq, oracle):
    """A 131072-token context (the decode_32k geometry, four times longer: 272 MB of K/V) through
    the fused step, which writes the newest token inside stage 1: every output against FP64,
    and the rewritten token's codes and scales against the oracle's quantiser."""
    w = W.make("decode_32k", seed=1300, ctx=131072)
    cache, bt = gpu_cache_from(w, kvq)
    kvq.kvq_quant_write(cache, to_bf16_tensor(np.zeros_like(w["k_new"])), to_bf16_tensor(np.zeros_like(w["v_new"])),
                        to_i32(w["new_seq"]), to_i32(w["new_pos"]), bt)  # the step must write these rows
    out = kvq.kvq_decode_step_int8kv(cache, to_bf16_tensor(w["k_new"]), to_bf16_tensor(w["v_new"]),
                                     to_bf16_tensor(w["q"]), bt, to_i32(w["ctx_lens"]), w["max_ctx"],
                                     w["softmax_scale"]).cpu().numpy()
    hc = host_cache_from(w, oracle)
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    err = norm_max_err(out, ref)
    print("decode 128k fused step normalised max err", err)
    assert err <= GATE and err <= DESIGN_TOL
    page = int(w["block_table"][0][(131072 - 1) // 16])
    assert np.array_equal(cache.k[page].cpu().numpy(), hc.k[page])
    assert np.array_equal(cache.v_scale[page].cpu().numpy().view(np.uint32), hc.v_scale[page].view(np.uint32))
    assert kvq.kvq_device_status() == 0


def test_decode_b64_full_sampled(kvq, oracle):
    """Workload decode_b64 at full size (64 sequences, ctx up to 16384, head_dim 128) with the
    step's kv_quant_write of one new token per sequence; sampled (sequence, head) outputs."""
    import torch
    w = W.make("decode_b64")
    cache, bt = gpu_cache_from(w, kvq)
    rng = np.random.default_rng(9)
    kn = W.normal_bf16(rng, (w["batch"], w["hkv"], w["d"]))
    vn = W.normal_bf16(rng, (w["batch"], w["hkv"], w["d"]))
    kvq.kvq_quant_write(cache, to_bf16_tensor(kn), to_bf16_tensor(vn), to_i32(w["new_seq"]),
                        to_i32(w["new_pos"]), bt)
    out = kvq.kvq_attn_decode_int8kv(cache, to_bf16_tensor(w["q"]), bt, to_i32(w["ctx_lens"]),
                                     w["max_ctx"], w["softmax_scale"]).cpu().numpy()
    hc = host_cache_from(w, oracle)
    oracle.kv_quant_write(hc, kn, vn, w["new_seq"], w["new_pos"], w["block_table"])
    units = sample_units(w["batch"], w["hq"], 96, seed=10)
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"], units=units)
    got = out.reshape(-1, w["d"])[units]
    err = norm_max_err(got, ref)
    print("decode_b64 normalised max err (sampled)", err)
    assert err <= GATE and err <= DESIGN_TOL
    del torch


def test_ctx_above_max_ctx_is_clamped_and_reported(kvq, oracle):
    """A ctx_lens entry above the host bound max_ctx (but within the pages its block-table row
    maps) breaks the call's contract: both routes clamp it to max_ctx, set KVQ_DEV_BAD_POS, and
    agree with the FP64 reference over max_ctx keys."""
    w = W.make("decode_32k", seed=1400, batch=2, ctx=1000, hq=8, hkv=2, d=128)
    cache, bt = gpu_cache_from(w, kvq)
    hc = host_cache_from(w, oracle)
    max_ctx = 900
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], np.full(2, max_ctx, np.int32), w["softmax_scale"])
    q, ctx = to_bf16_tensor(w["q"]), to_i32(w["ctx_lens"])
    kvq.kvq_device_status()
    for route in (1, 2):
        got = kvq.kvq_attn_decode_int8kv(cache, q, bt, ctx, max_ctx, w["softmax_scale"], force_route=route,
                                         split_rows=256).cpu().numpy()
        assert kvq.kvq_device_status() & kvq.kvq.DEV_BAD_POS, route
        assert norm_max_err(got, ref) <= DESIGN_TOL, route


def test_gqa_group_above_16_is_refused(kvq):
    import torch
    cache = kvq.KVCache(4, 2, 128)
    q = torch.zeros((1, 34, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    ctx = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_attn_decode_int8kv(cache, q, bt, ctx, 64, 0.1)
    assert e.value.status == 2  # KVQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("d", [128, 256])
def test_many_units_few_splits_merge(kvq, oracle, d):
    """A batch with many (sequence, query head) units and a few splits each takes the
    warp-per-unit merge: against FP64, and ctx 0 rows give zeros."""
    w = W.make("decode_b64", seed=330 + d, batch=24, ctx_range=(300, 2000), hq=24, hkv=4, d=d)
    w["ctx_lens"][3] = 0
    got, _, _ = _run(kvq, w, force_route=2, split_rows=256)
    hc = host_cache_from(w, oracle)
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    assert np.all(got[3] == 0)
    assert norm_max_err(got, ref) <= DESIGN_TOL
    assert kvq.kvq_device_status() == 0
