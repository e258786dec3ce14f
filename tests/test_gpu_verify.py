"""kvq_attn_verify_int8kv (nq query rows per sequence, causal among the nq newest tokens) on
the GPU against the oracle's FP64 verify decode.

Same gates as plain decode: <= 2e-3 normalised max-abs error (the acceptance bar), and the
design tolerance 1e-4 (the kernel keeps ~22-bit softmax weights and fp32 accumulation).
The row counts G * nq cover one to six 8-row n-tiles (warp teams of one to six warps)."""
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


def _case(seed, nq, batch, ctx_range, hq, hkv, d):
    return W.make("decode_b64", seed=seed, batch=batch, ctx_range=ctx_range, hq=hq, hkv=hkv, d=d, nq=nq)


def _run(kvq, w, **opts):
    cache, bt = gpu_cache_from(w, kvq)
    out = kvq.kvq_attn_verify_int8kv(cache, to_bf16_tensor(w["q"]), bt, to_i32(w["ctx_lens"]), w["max_ctx"],
                                     w["softmax_scale"], **opts)
    return out.cpu().numpy()


# (G, nq) -> rows = G * nq: 8 (1 tile), 16, 24, 36 (5 tiles), 48 (6 tiles), 2 x 3 = 6
@pytest.mark.parametrize("d,hq,hkv,nq", [(128, 8, 2, 2), (128, 8, 2, 4), (128, 32, 8, 6), (256, 24, 4, 3),
                                         (256, 24, 4, 6), (256, 16, 2, 6), (256, 2, 1, 3)])
def test_rows_and_geometries_both_routes(kvq, oracle, d, hq, hkv, nq):
    w = _case(500 + hq + nq, nq, 3, (1, 1400), hq, hkv, d)
    hc = host_cache_from(w, oracle)
    ref = oracle.verify_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    for route in (1, 2):
        got = _run(kvq, w, force_route=route, split_rows=128)
        err = norm_max_err(got, ref)
        assert err <= GATE and err <= DESIGN_TOL, (route, err)
    assert kvq.kvq_device_status() == 0


@pytest.mark.parametrize("split", [16, 48, 512])
def test_split_boundaries_inside_the_verified_tokens(kvq, oracle, split):
    # contexts that put a split boundary among the nq newest tokens: some splits hold keys
    # for only some rows
    w = _case(520, 5, 4, (700, 700), 12, 2, 256)  # 700 tokens filled; the lengths below are shorter
    w["ctx_lens"] = np.array([16 * 20 + 2, 48 * 9 + 3, 515, 640], np.int32)
    w["max_ctx"] = int(w["ctx_lens"].max())
    hc = host_cache_from(w, oracle)
    ref = oracle.verify_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    got = _run(kvq, w, force_route=2, split_rows=split)
    assert norm_max_err(got, ref) <= DESIGN_TOL


def test_contexts_shorter_than_the_rows(kvq, oracle):
    # ctx < nq: the first rows see no key and give zeros; ctx 0 gives zeros everywhere
    w = _case(521, 4, 4, (40, 40), 8, 2, 128)
    w["ctx_lens"] = np.array([2, 0, 4, 33], np.int32)
    w["max_ctx"] = 33
    hc = host_cache_from(w, oracle)
    ref = oracle.verify_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    for route in (1, 2):
        got = _run(kvq, w, force_route=route, split_rows=16)
        assert not got[0, :2].any() and not got[1].any()
        assert norm_max_err(got, ref) <= DESIGN_TOL, route
    assert kvq.kvq_device_status() == 0


def test_one_row_is_plain_decode(kvq):
    w = _case(522, 1, 3, (100, 2000), 24, 4, 256)
    cache, bt = gpu_cache_from(w, kvq)
    q = to_bf16_tensor(w["q"])
    ctx = to_i32(w["ctx_lens"])
    dec = kvq.kvq_attn_decode_int8kv(cache, q, bt, ctx, w["max_ctx"], w["softmax_scale"], split_rows=256)
    ver = kvq.kvq_attn_verify_int8kv(cache, q[:, None], bt, ctx, w["max_ctx"], w["softmax_scale"],
                                     split_rows=256)
    assert np.array_equal(dec.cpu().numpy(), ver[:, 0].cpu().numpy())


def test_verify_32k_full_size_sampled(kvq, oracle):
    """The verify_32k workload (ctx 32768, 4 rows, 24/4, d 256) in the bench's launch
    configuration (automatic split), on sampled (row, head) units."""
    w = W.make("verify_32k")
    cache, bt = gpu_cache_from(w, kvq)
    got = kvq.kvq_attn_verify_int8kv(cache, to_bf16_tensor(w["q"]), bt, to_i32(w["ctx_lens"]), w["max_ctx"],
                                     w["softmax_scale"]).cpu().numpy()
    hc = host_cache_from(w, oracle)
    units = sample_units(w["nq"], w["hq"], 24, seed=523)
    ref = oracle.verify_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"], units=units)
    err = norm_max_err(got.reshape(-1, w["d"])[units], ref)
    assert err <= DESIGN_TOL, err
    assert kvq.kvq_device_status() == 0
