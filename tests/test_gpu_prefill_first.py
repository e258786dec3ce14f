"""kvq_attn_prefill_first_bf16 (the first prefill chunk: high-precision causal attention over
the chunk's own bf16 Q/K/V, with the chunk's K/V written into the int8 cache) on the GPU.

Gates: the cache after the call equals the oracle's quantiser bit for bit; the output is
within 5e-3 (normalised max-abs) of the oracle's FP64 attention over the bf16 values (the bar
for outputs checked against FP64), and within the design tolerance 2e-3.  Q, K and V reach the
tensor cores exactly (power-of-two scaled fp16); the softmax weights of each 128-key tile go in
as fp16 w / max w, each rounded by at most 2^-12 of itself.  The largest normalised errors sit
in the first rows of a chunk: they average only a few V rows, so their outputs are large next
to the RMS of all outputs, which the long rows' averaging keeps small (measured 1.2e-3 at a
130-token chunk)."""
import numpy as np
import pytest

import workloads as W
from helpers import norm_max_err, sample_units, to_bf16_tensor, to_i32

pytestmark = pytest.mark.gpu

GATE = 5e-3
DESIGN_TOL = 2e-3


@pytest.fixture(scope="module")
def kvq():
    import int8_kv_cache_quant_gb300 as k
    k.lib()
    return k


def _case(seed, T, hq, hkv, d, outlier_p=0.0):
    rng = np.random.default_rng(seed)
    n_blocks = (T + 15) // 16 + 3
    table = rng.permutation(n_blocks).astype(np.int32)
    q = W.normal_bf16(rng, (T, hq, d))
    k = W.normal_bf16(rng, (T, hkv, d), outlier_p=outlier_p)
    v = W.normal_bf16(rng, (T, hkv, d))
    return table, n_blocks, q, k, v


def _run(kvq, table, n_blocks, q, k, v, scale):
    T, hq, d = q.shape
    cache = kvq.KVCache(n_blocks, k.shape[1], d)
    out = kvq.kvq_attn_prefill_first_bf16(cache, to_bf16_tensor(q), to_bf16_tensor(k), to_bf16_tensor(v),
                                          to_i32(table), scale).cpu().numpy()
    return cache, out


@pytest.mark.parametrize("T,hq,hkv,d", [(130, 6, 1, 256), (300, 8, 2, 128), (1, 4, 4, 256), (257, 24, 4, 256),
                                        (128, 32, 8, 128)])
def test_first_chunk_attention_and_cache(kvq, oracle, T, hq, hkv, d):
    table, nb, q, k, v = _case(600 + T + hq, T, hq, hkv, d, outlier_p=0.01)
    scale = 1.0 / np.sqrt(d)
    cache, out = _run(kvq, table, nb, q, k, v, scale)
    assert kvq.kvq_device_status() == 0
    ref = oracle.prefill_first_f64(q, k, v, scale)
    err = norm_max_err(out, ref)
    assert err <= GATE and err <= DESIGN_TOL, err
    hc = oracle.HostCache(nb, hkv, d)
    oracle.kv_quant_write(hc, k, v, np.zeros(T, np.int32), np.arange(T, dtype=np.int32), table[None, :])
    assert np.array_equal(cache.k.cpu().numpy(), hc.k) and np.array_equal(cache.v.cpu().numpy(), hc.v)
    assert np.array_equal(cache.k_scale.cpu().numpy().view(np.uint32), hc.k_scale.view(np.uint32))
    assert np.array_equal(cache.v_scale.cpu().numpy().view(np.uint32), hc.v_scale.view(np.uint32))


def test_first_chunk_wide_dynamic_range(kvq, oracle):
    # Q and K rows scaled by powers of two in 2^-8 .. 2^8 (logits up to ~2^12) and V rows in
    # 2^-20 .. 2^20, over several 128-key tiles: each row's fp16 image is exact after its
    # power-of-two scale, and O's unit only grows, so the result tracks FP64 whatever the
    # magnitudes of the rows
    table, nb, q, k, v = _case(640, 700, 8, 2, 128)
    rng = np.random.default_rng(641)
    for x, span in ((q, 8), (k, 8), (v, 20)):
        f = W.bf16_bits_to_f32(x) * (2.0 ** rng.integers(-span, span + 1, size=x.shape[:2]))[..., None].astype(np.float32)
        x[...] = W.f32_to_bf16_bits(f)
    scale = 1.0 / np.sqrt(128) * 2.0 ** -8
    _, out = _run(kvq, table, nb, q, k, v, scale)
    ref = oracle.prefill_first_f64(q, k, v, scale)
    assert norm_max_err(out, ref) <= DESIGN_TOL


def test_first_then_int8_chunk_continue_the_sequence(kvq, oracle):
    # the first chunk writes the cache that the next (int8) chunk reads as its history
    rng = np.random.default_rng(650)
    T1, T2, hq, hkv, d = 384, 200, 12, 2, 256
    n_blocks = (T1 + T2 + 15) // 16
    table = rng.permutation(n_blocks).astype(np.int32)
    q1 = W.normal_bf16(rng, (T1, hq, d))
    k = W.normal_bf16(rng, (T1 + T2, hkv, d))
    v = W.normal_bf16(rng, (T1 + T2, hkv, d))
    q2 = W.normal_bf16(rng, (T2, hq, d))
    scale = 1.0 / 16
    cache = kvq.KVCache(n_blocks, hkv, d)
    bt = to_i32(table)
    kvq.kvq_attn_prefill_first_bf16(cache, to_bf16_tensor(q1), to_bf16_tensor(k[:T1]), to_bf16_tensor(v[:T1]), bt,
                                    scale)
    kvq.kvq_quant_write(cache, to_bf16_tensor(k[T1:]), to_bf16_tensor(v[T1:]), to_i32(np.zeros(T2, np.int32)),
                        to_i32(np.arange(T1, T1 + T2, dtype=np.int32)), bt[None, :])
    out2 = kvq.kvq_attn_prefill_int8(cache, to_bf16_tensor(q2), T1, bt, scale).cpu().numpy()
    hc = oracle.HostCache(n_blocks, hkv, d)
    oracle.kv_quant_write(hc, k, v, np.zeros(T1 + T2, np.int32), np.arange(T1 + T2, dtype=np.int32), table[None, :])
    ref = oracle.prefill_int8_emul(hc, q2, T1, table, scale)
    assert norm_max_err(out2, ref) <= 2e-3


def test_first_chunk_4k_sampled(kvq, oracle):
    """A 4096-token first chunk at 24 query / 4 KV heads, head_dim 256 (the page's 0 + 4K chunk),
    sampled (token, head) outputs against FP64."""
    table, nb, q, k, v = _case(660, 4096, 24, 4, 256)
    scale = 1.0 / 16
    _, out = _run(kvq, table, nb, q, k, v, scale)
    units = sample_units(4096, 24, 48, seed=661)
    ref = oracle.prefill_first_f64(q, k, v, scale, units=units)
    err = norm_max_err(out.reshape(-1, 256)[units], ref)
    assert err <= DESIGN_TOL, err
    assert kvq.kvq_device_status() == 0
