"""kvq_rope_quant_write (the fused producer with RoPE) and kvq_attn_prefill_int8_qcodes on the
GPU.  Gates: K/V codes and scales, Q codes, Q scales and the rotated bf16 Q bit-exact against
the oracle's producer; the Q-codes prefill identical to the prefill that quantises Q itself when
both see the same codes."""
import numpy as np
import pytest

import workloads as W
from helpers import to_bf16_tensor, to_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import int8_kv_cache_quant_gb300 as k
    k.lib()
    return k


def _rope_table(max_pos, r, base=1.0e6):
    inv = base ** (-np.arange(0, r, 2, dtype=np.float64) / r)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


@pytest.mark.parametrize("d,hq,hkv,rot", [(256, 24, 4, 256), (256, 6, 1, 128), (128, 32, 8, 128), (128, 8, 2, 64)])
def test_rope_quant_write_bit_exact(kvq, oracle, d, hq, hkv, rot):
    import torch
    rng = np.random.default_rng(900 + d + rot)
    T, max_pos = 77, 4096
    # distinct positions (distinct slots); two out of range: no K/V write, zero Q outputs
    pos = rng.choice(max_pos, size=T, replace=False).astype(np.int32)
    pos[5], pos[9] = max_pos + 3, -1
    seq = np.zeros(T, np.int32)
    n_blocks = max_pos // 16 + 1
    table = rng.permutation(n_blocks).astype(np.int32)[None, :]
    q = W.normal_bf16(rng, (T, hq, d))
    k = W.normal_bf16(rng, (T, hkv, d), outlier_p=0.01)
    v = W.normal_bf16(rng, (T, hkv, d))
    cs = _rope_table(max_pos, rot)

    cache = kvq.KVCache(n_blocks, hkv, d)
    qc, qs, qr = kvq.kvq_rope_quant_write(cache, to_bf16_tensor(q), to_bf16_tensor(k), to_bf16_tensor(v),
                                          to_i32(seq), to_i32(pos), to_i32(table),
                                          torch.from_numpy(cs).cuda(), rot)
    st = kvq.kvq_device_status()
    hc = oracle.HostCache(n_blocks, hkv, d)
    skipped, rqc, rqs, rqr = oracle.rope_quant_write(hc, q, k, v, seq, pos, table, cs, rot)
    assert skipped == 2 and st != 0  # the two bad positions were flagged
    assert np.array_equal(cache.k.cpu().numpy(), hc.k)
    assert np.array_equal(cache.v.cpu().numpy(), hc.v)
    assert np.array_equal(cache.k_scale.cpu().numpy().view(np.uint32), hc.k_scale.view(np.uint32))
    assert np.array_equal(cache.v_scale.cpu().numpy().view(np.uint32), hc.v_scale.view(np.uint32))
    assert np.array_equal(qc.cpu().numpy(), rqc)
    assert np.array_equal(qs.cpu().numpy().view(np.uint32), rqs.view(np.uint32))
    assert np.array_equal(qr.cpu().view(torch.int16).numpy().view(np.uint16), rqr)


@pytest.mark.parametrize("d,c", [(256, 0.70710677), (128, 0.3), (256, 0.9)])
def test_rope_quant_near_half_integer_quotients(kvq, oracle, d, c):
    """Rotated fp32 rows whose quotients x / scale sit a hair away from half-integers: rows of
    integer values in [-254, 254] with amax 254 (so x / scale would be x / 2 exactly), rotated by a
    table whose cosine is the constant c and whose sine is 0, so that every element becomes
    RN(x * c) and the scale RN(RN(254 c) / 127).  Most odd x then land within a few 1e-6 of a
    half-integer, where the rule's fast path must hand the code to the IEEE division.  Gate: codes,
    scales and rotated rows bit-exact against the oracle's producer."""
    import torch
    rng = np.random.default_rng(int(d + 1000 * c))
    T, hq, hkv, max_pos = 48, 8, 2, 64

    def rows(shape):
        x = rng.integers(-254, 255, size=shape).astype(np.float32)
        x[..., 0] = np.where(rng.random(shape[:-1]) < 0.5, 254.0, -254.0)
        return W.f32_to_bf16_bits(x)  # integers up to 256 are exact in bf16

    q, k, v = rows((T, hq, d)), rows((T, hkv, d)), rows((T, hkv, d))
    cs = np.zeros((max_pos, d), np.float32)
    cs[:, : d // 2] = np.float32(c)
    pos = np.arange(T, dtype=np.int32)
    seq = np.zeros(T, np.int32)
    table = np.arange(max_pos // 16, dtype=np.int32)[None, :]
    # how many quotients the fast path must leave to the division (the test's reason to exist)
    xr = W.bf16_bits_to_f32(q) * np.float32(c)
    scale = (np.abs(xr).max(axis=-1, keepdims=True) / np.float32(127.0)).astype(np.float32)
    quo = xr.astype(np.float64) / scale.astype(np.float64)
    near = np.abs(np.abs(quo - np.floor(quo)) - 0.5) < 3.0e-5
    assert near.sum() > 1000, near.sum()

    cache = kvq.KVCache(max_pos // 16, hkv, d)
    qc, qs, qr = kvq.kvq_rope_quant_write(cache, to_bf16_tensor(q), to_bf16_tensor(k), to_bf16_tensor(v),
                                          to_i32(seq), to_i32(pos), to_i32(table), torch.from_numpy(cs).cuda(), d)
    assert kvq.kvq_device_status() == 0
    hc = oracle.HostCache(max_pos // 16, hkv, d)
    skipped, rqc, rqs, rqr = oracle.rope_quant_write(hc, q, k, v, seq, pos, table, cs, d)
    assert skipped == 0
    assert np.array_equal(cache.k.cpu().numpy(), hc.k)
    assert np.array_equal(cache.v.cpu().numpy(), hc.v)
    assert np.array_equal(cache.k_scale.cpu().numpy().view(np.uint32), hc.k_scale.view(np.uint32))
    assert np.array_equal(cache.v_scale.cpu().numpy().view(np.uint32), hc.v_scale.view(np.uint32))
    assert np.array_equal(qc.cpu().numpy(), rqc)
    assert np.array_equal(qs.cpu().numpy().view(np.uint32), rqs.view(np.uint32))
    assert np.array_equal(qr.cpu().view(torch.int16).numpy().view(np.uint16), rqr)


def test_rope_quant_write_without_q(kvq, oracle):
    import torch
    rng = np.random.default_rng(950)
    T, d, hkv, max_pos = 40, 256, 4, 640
    pos = rng.choice(max_pos, size=T, replace=False).astype(np.int32)
    table = np.arange(max_pos // 16, dtype=np.int32)[None, :]
    k = W.normal_bf16(rng, (T, hkv, d))
    v = W.normal_bf16(rng, (T, hkv, d))
    cs = _rope_table(max_pos, d)
    cache = kvq.KVCache(max_pos // 16, hkv, d)
    out = kvq.kvq_rope_quant_write(cache, None, to_bf16_tensor(k), to_bf16_tensor(v), to_i32(np.zeros(T, np.int32)),
                                   to_i32(pos), to_i32(table), torch.from_numpy(cs).cuda(), d)
    assert out == (None, None, None)
    hc = oracle.HostCache(max_pos // 16, hkv, d)
    oracle.rope_quant_write(hc, None, k, v, np.zeros(T, np.int32), pos, table, cs, d)
    assert np.array_equal(cache.k.cpu().numpy(), hc.k) and np.array_equal(cache.v.cpu().numpy(), hc.v)
    assert kvq.kvq_device_status() == 0


@pytest.mark.parametrize("history,T,d,hq,hkv", [(300, 77, 128, 8, 2), (1000, 300, 256, 12, 2)])
def test_prefill_qcodes_equals_prefill(kvq, history, T, d, hq, hkv):
    w = W.make("prefill_32k", seed=960 + T, history=history, chunk=T, hq=hq, hkv=hkv, d=d)
    from helpers import gpu_cache_from
    cache, bt = gpu_cache_from(w, kvq)
    q = to_bf16_tensor(w["q"])
    ref = kvq.kvq_attn_prefill_int8(cache, q, w["history"], bt[0], w["softmax_scale"]).cpu().numpy()
    codes, scales = kvq.kvq_debug_prefill_q_codes(q)
    got = kvq.kvq_attn_prefill_int8_qcodes(cache, codes, scales, w["history"], bt[0], w["softmax_scale"]).cpu().numpy()
    assert np.array_equal(got, ref)
    assert kvq.kvq_device_status() == 0
