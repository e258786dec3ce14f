"""kvq_quant_write on the GPU against the oracle: codes and scales bit-exact."""
import numpy as np
import pytest

import workloads as W
from helpers import gpu_cache_from, host_cache_from, to_bf16_tensor, to_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import int8_kv_cache_quant_gb300 as k
    k.lib()
    return k


def _assert_cache_equal(gc, hc):
    assert np.array_equal(gc.k.cpu().numpy(), hc.k)
    assert np.array_equal(gc.v.cpu().numpy(), hc.v)
    assert np.array_equal(gc.k_scale.cpu().numpy().view(np.uint32), hc.k_scale.view(np.uint32))
    assert np.array_equal(gc.v_scale.cpu().numpy().view(np.uint32), hc.v_scale.view(np.uint32))


@pytest.mark.parametrize("d,hkv,ctx", [(256, 4, 333), (128, 8, 517), (256, 1, 40), (128, 2, 16)])
def test_bit_exact_random(kvq, oracle, d, hkv, ctx):
    w = W.make("decode_32k", seed=100 + d + ctx, batch=1, ctx=ctx, hkv=hkv, hq=hkv, d=d)
    gc, _ = gpu_cache_from(w, kvq)
    hc = host_cache_from(w, oracle)
    assert kvq.kvq_device_status() == 0
    _assert_cache_equal(gc, hc)


def test_bit_exact_edge_rows(kvq, oracle):
    # zero rows, hand-worked tie rows, huge and tiny magnitudes, one-hot rows
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "quant_rows_handworked.json")))
    d, hkv = 128, 1
    rows = []
    for r in g["rows"]:
        rows.append(np.tile(np.asarray(r["x"], np.float32), d // 16))
    rng = np.random.default_rng(5)
    rows.append(rng.standard_normal(d).astype(np.float32) * 1e30)
    rows.append(rng.standard_normal(d).astype(np.float32) * 1e-30)
    rows.append(rng.standard_normal(d).astype(np.float32) * 1e-38)  # bf16 subnormals
    oh = np.zeros(d, np.float32)
    oh[17] = -3.0
    rows.append(oh)
    rows.append(np.zeros(d, np.float32))
    x = W.f32_to_bf16_bits(np.stack(rows))[:, None, :]
    T = x.shape[0]
    w = dict(num_blocks=2, hkv=hkv, d=d, k_fill=x, v_fill=x[::-1].copy(),
             fill_seq=np.zeros(T, np.int32), fill_pos=np.arange(T, dtype=np.int32),
             block_table=np.array([[1, 0]], np.int32))
    gc, _ = gpu_cache_from(w, kvq)
    hc = host_cache_from(w, oracle)
    _assert_cache_equal(gc, hc)
    codes, scales = oracle.quant_rows(x[:3, 0, :16])
    assert codes[0].tolist() == g["rows"][0]["codes"]


def test_out_of_range_tokens_are_skipped_and_flagged(kvq):
    d, hkv = 128, 2
    cache = kvq.KVCache(2, hkv, d)
    rng = np.random.default_rng(7)
    x = W.normal_bf16(rng, (4, hkv, d))
    bt = to_i32(np.array([[0, 7]], np.int32))  # page 7 does not exist
    kvq.kvq_device_status()  # clear
    kvq.kvq_quant_write(cache, to_bf16_tensor(x), to_bf16_tensor(x), to_i32([0, 3, 0, 0]),
                        to_i32([0, 0, 20, 99]), bt)
    flags = kvq.kvq_device_status()
    assert flags & kvq.kvq.DEV_BAD_SEQ and flags & kvq.kvq.DEV_BAD_BLOCK and flags & kvq.kvq.DEV_BAD_POS
    # only token 0 (seq 0, pos 0 -> page 0 slot 0) was written
    k = cache.k.cpu().numpy()
    assert k[0, :, :, 0, :].any() and not k[0, :, :, 1:, :].any() and not k[1].any()


def test_batched_new_tokens_like_decode_step(kvq, oracle):
    # one new token per sequence into a shuffled shared pool (the batched decode step)
    w = W.make("decode_b64", seed=77, batch=16, ctx_range=(20, 300))
    gc, bt = gpu_cache_from(w, kvq)
    hc = host_cache_from(w, oracle)
    # overwrite each sequence's last token with fresh values on both sides
    rng = np.random.default_rng(8)
    kn = W.normal_bf16(rng, (16, w["hkv"], w["d"]), outlier_p=0.05)
    vn = W.normal_bf16(rng, (16, w["hkv"], w["d"]))
    kvq.kvq_quant_write(gc, to_bf16_tensor(kn), to_bf16_tensor(vn), to_i32(w["new_seq"]),
                        to_i32(w["new_pos"]), bt)
    oracle.kv_quant_write(hc, kn, vn, w["new_seq"], w["new_pos"], w["block_table"])
    _assert_cache_equal(gc, hc)
