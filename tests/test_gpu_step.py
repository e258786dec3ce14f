"""kvq_decode_step_int8kv (the fused step: write each sequence's newest tokens, then attend)
on the GPU.

The cache starts with every token except the step's new ones; after the call it must equal,
bit for bit, the oracle's cache with all tokens written by the oracle's quantiser, and the
output must match the oracle's FP64 decode / verify (design tolerance 1e-4, acceptance
2e-3) and the unfused kvq_quant_write + attention path on the same cache."""
import numpy as np
import pytest

import workloads as W
from helpers import host_cache_from, norm_max_err, to_bf16_tensor, to_i32

pytestmark = pytest.mark.gpu

DESIGN_TOL = 1e-4


@pytest.fixture(scope="module")
def kvq():
    import int8_kv_cache_quant_gb300 as k
    k.lib()
    return k


def _cache_without_new(kvq, w):
    """Device cache holding every token of the workload but each sequence's newest nq."""
    nq = w["nq"]
    last = w["ctx_lens"][w["fill_seq"]] - nq
    keep = w["fill_pos"] < last
    cache = kvq.KVCache(w["num_blocks"], w["hkv"], w["d"])
    bt = to_i32(w["block_table"])
    kvq.kvq_quant_write(cache, to_bf16_tensor(w["k_fill"][keep]), to_bf16_tensor(w["v_fill"][keep]),
                        to_i32(w["fill_seq"][keep]), to_i32(w["fill_pos"][keep]), bt)
    return cache, bt


def _new_rows(w):
    B, nq = w["batch"], w["nq"]
    shape = (B, nq, w["hkv"], w["d"])
    return w["k_new"].reshape(shape), w["v_new"].reshape(shape)


def _check_cache(cache, hc):
    assert np.array_equal(cache.k.cpu().numpy(), hc.k)
    assert np.array_equal(cache.v.cpu().numpy(), hc.v)
    assert np.array_equal(cache.k_scale.cpu().numpy().view(np.uint32), hc.k_scale.view(np.uint32))
    assert np.array_equal(cache.v_scale.cpu().numpy().view(np.uint32), hc.v_scale.view(np.uint32))


@pytest.mark.parametrize("nq,d,hq,hkv,route", [(1, 128, 32, 8, 2), (1, 256, 24, 4, 1), (1, 256, 24, 4, 2),
                                               (4, 256, 24, 4, 2), (3, 128, 8, 2, 1), (6, 128, 16, 2, 2),
                                               (1, 256, 32, 2, 2), (3, 128, 32, 2, 1)])
def test_step_writes_and_attends(kvq, oracle, nq, d, hq, hkv, route):
    w = W.make("decode_b64", seed=700 + nq + d + route, batch=5, ctx_range=(nq, 1500), hq=hq, hkv=hkv, d=d, nq=nq)
    cache, bt = _cache_without_new(kvq, w)
    kn, vn = _new_rows(w)
    q = w["q"] if nq > 1 else w["q"][:, None]
    out = kvq.kvq_decode_step_int8kv(cache, to_bf16_tensor(kn), to_bf16_tensor(vn), to_bf16_tensor(q), bt,
                                     to_i32(w["ctx_lens"]), w["max_ctx"], w["softmax_scale"], force_route=route,
                                     split_rows=128).cpu().numpy()
    assert kvq.kvq_device_status() == 0
    hc = host_cache_from(w, oracle)
    _check_cache(cache, hc)
    ref = oracle.verify_f64(hc, q, w["block_table"], w["ctx_lens"], w["softmax_scale"])
    assert norm_max_err(out, ref) <= DESIGN_TOL
    # the unfused path on the now complete cache gives the same bits
    sep = kvq.kvq_attn_verify_int8kv(cache, to_bf16_tensor(q), bt, to_i32(w["ctx_lens"]), w["max_ctx"],
                                     w["softmax_scale"], force_route=route, split_rows=128).cpu().numpy()
    assert np.array_equal(out, sep)


def test_one_token_step_3d_and_decode_32k_shape(kvq, oracle):
    """The benchmark's call in full: the fused step at workload decode_32k (ctx 32768, 24/4,
    head_dim 256, shuffled pages, K outliers) with the automatic split and no option set, the new
    token the last of the last split.  The rewritten cache bit for bit, and all 24 heads against
    FP64."""
    w = W.make("decode_32k")
    cache, bt = _cache_without_new(kvq, w)
    kn, vn = _new_rows(w)
    out = kvq.kvq_decode_step_int8kv(cache, to_bf16_tensor(kn[:, 0]), to_bf16_tensor(vn[:, 0]),
                                     to_bf16_tensor(w["q"]), bt, to_i32(w["ctx_lens"]), w["max_ctx"],
                                     w["softmax_scale"]).cpu().numpy()
    assert out.shape == (1, w["hq"], w["d"])
    assert kvq.kvq_device_status() == 0
    hc = host_cache_from(w, oracle)
    _check_cache(cache, hc)
    dec = kvq.kvq_attn_decode_int8kv(cache, to_bf16_tensor(w["q"]), bt, to_i32(w["ctx_lens"]), w["max_ctx"],
                                     w["softmax_scale"]).cpu().numpy()
    assert np.array_equal(out, dec)
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    err = norm_max_err(out, ref)
    print("decode_32k fused step (automatic split), all heads: normalised max err", err)
    assert err <= DESIGN_TOL


def test_step_with_short_context_writes_nothing_and_flags(kvq):
    # a sequence shorter than its new-token count has no valid positions for them
    w = W.make("decode_b64", seed=720, batch=2, ctx_range=(40, 40), hq=8, hkv=2, d=128, nq=3)
    cache, bt = _cache_without_new(kvq, w)
    before_k, before_v = cache.k.cpu().numpy(), cache.v.cpu().numpy()
    kn, vn = _new_rows(w)
    ctx = w["ctx_lens"].copy()
    ctx[1] = 2
    kvq.kvq_decode_step_int8kv(cache, to_bf16_tensor(kn), to_bf16_tensor(vn), to_bf16_tensor(w["q"]), bt,
                               to_i32(ctx), 40, w["softmax_scale"], force_route=1)
    st = kvq.kvq_device_status()
    assert st & 0x2  # KVQ_DEV_BAD_POS
    # sequence 1 wrote nothing; sequence 0 wrote its 3 tokens (positions 37..39)
    after_k, after_v = cache.k.cpu().numpy(), cache.v.cpu().numpy()
    pages1 = w["block_table"][1][w["block_table"][1] >= 0]
    assert np.array_equal(after_k[pages1], before_k[pages1])
    assert np.array_equal(after_v[pages1], before_v[pages1])
    p0 = w["block_table"][0][39 // 16]
    assert not np.array_equal(after_k[p0], before_k[p0])


def test_decode_b64_fused_step_full_sampled(kvq, oracle):
    """decode_b64 at full size (64 sequences, ctx up to 16384, 32/8 heads, head_dim 128) through
    the fused step, as bench.py times it: a fresh new token per sequence is written by stage 1;
    the pages holding them match the oracle's writer bit for bit, and sampled outputs match FP64."""
    from helpers import gpu_cache_from, sample_units
    w = W.make("decode_b64")
    cache, bt = gpu_cache_from(w, kvq)
    rng = np.random.default_rng(730)
    kn = W.normal_bf16(rng, (w["batch"], w["hkv"], w["d"]))
    vn = W.normal_bf16(rng, (w["batch"], w["hkv"], w["d"]))
    out = kvq.kvq_decode_step_int8kv(cache, to_bf16_tensor(kn), to_bf16_tensor(vn), to_bf16_tensor(w["q"]), bt,
                                     to_i32(w["ctx_lens"]), w["max_ctx"], w["softmax_scale"]).cpu().numpy()
    assert kvq.kvq_device_status() == 0
    hc = host_cache_from(w, oracle)
    oracle.kv_quant_write(hc, kn, vn, w["new_seq"], w["new_pos"], w["block_table"])
    pages = w["block_table"][w["new_seq"], w["new_pos"] // 16]
    for name in ("k", "v", "k_scale", "v_scale"):
        got = getattr(cache, name)[torch_index(pages)].cpu().numpy()
        assert np.array_equal(got.view(np.uint8), getattr(hc, name)[pages].view(np.uint8)), name
    units = sample_units(w["batch"], w["hq"], 96, seed=731)
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"], units=units)
    assert norm_max_err(out.reshape(-1, w["d"])[units], ref) <= DESIGN_TOL


def torch_index(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).cuda()


def test_one_token_step_far_into_a_warps_pages(kvq, oracle):
    """Single route at head_dim 256 with a context long enough that the new token's page is
    past the first 32 pages of its warp (the page id then comes from the block table, not the
    warp's window): the rewritten cache bit for bit, the output against FP64 and bit-identical to
    plain decode on the completed cache."""
    w = W.make("decode_32k", seed=741, batch=1, ctx=6000, hq=24, hkv=4, d=256)
    assert (w["ctx_lens"][0] - 1) // 16 // 8 >= 32
    cache, bt = _cache_without_new(kvq, w)
    kn, vn = _new_rows(w)
    args = (bt, to_i32(w["ctx_lens"]), w["max_ctx"], w["softmax_scale"])
    out = kvq.kvq_decode_step_int8kv(cache, to_bf16_tensor(kn[:, 0]), to_bf16_tensor(vn[:, 0]),
                                     to_bf16_tensor(w["q"]), *args, force_route=1).cpu().numpy()
    assert kvq.kvq_device_status() == 0
    hc = host_cache_from(w, oracle)
    _check_cache(cache, hc)
    dec = kvq.kvq_attn_decode_int8kv(cache, to_bf16_tensor(w["q"]), *args, force_route=1).cpu().numpy()
    assert np.array_equal(out, dec)
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    assert norm_max_err(out, ref) <= DESIGN_TOL


@pytest.mark.parametrize("route", [1, 2])
def test_one_token_step_on_an_unmapped_page(kvq, route):
    """The new token's page has no valid block-table entry: nothing is written, KVQ_DEV_BAD_BLOCK
    is reported, and the output is that of plain decode, which skips the same page."""
    import torch
    w = W.make("decode_32k", seed=742, batch=1, ctx=3000, hq=24, hkv=4, d=256)
    cache, _ = _cache_without_new(kvq, w)
    table = w["block_table"].copy()
    table[0, (w["ctx_lens"][0] - 1) // 16] = w["num_blocks"] + 5
    bt = to_i32(table)
    before = [t.clone() for t in (cache.k, cache.v, cache.k_scale, cache.v_scale)]
    kn, vn = _new_rows(w)
    args = (bt, to_i32(w["ctx_lens"]), w["max_ctx"], w["softmax_scale"])
    out = kvq.kvq_decode_step_int8kv(cache, to_bf16_tensor(kn[:, 0]), to_bf16_tensor(vn[:, 0]),
                                     to_bf16_tensor(w["q"]), *args, force_route=route, split_rows=512).cpu().numpy()
    assert kvq.kvq_device_status() & 0x1  # KVQ_DEV_BAD_BLOCK
    for t0, t1 in zip(before, (cache.k, cache.v, cache.k_scale, cache.v_scale)):
        assert torch.equal(t0, t1)
    dec = kvq.kvq_attn_decode_int8kv(cache, to_bf16_tensor(w["q"]), *args, force_route=route,
                                     split_rows=512).cpu().numpy()
    kvq.kvq_device_status()
    assert np.isfinite(out).all()
    assert np.array_equal(out, dec)
