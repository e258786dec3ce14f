"""kvq_attn_prefill_int8 on the GPU against the oracle's int8 emulation.

Gates: Q codes and the int32 QK score tiles bit-exact; outputs within 2e-3
normalised max-abs of the int8-emulated output.  The P-code decisions are taken with the
same fp32 operations on both sides, so the expected difference is only the fp32 vs double
accumulation of l and of the numerator (~1e-6); DESIGN_TOL = 1e-4 catches regressions.
Against the FP64 reference (Part A) the method's own error (7-bit P codes, int8 Q) is a few
percent of the output RMS; that figure is printed, not gated.
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


def _case(seed, history, T, hq=6, hkv=1, d=256, **kw):
    return W.make("prefill_32k", seed=seed, history=history, chunk=T, hq=hq, hkv=hkv, d=d, **kw)


@pytest.mark.parametrize("d", [128, 256])
def test_q_codes_bit_exact(kvq, oracle, d):
    w = _case(600 + d, history=0, T=77, hq=4, hkv=2, d=d)
    codes, scales = kvq.kvq_debug_prefill_q_codes(to_bf16_tensor(w["q"]))
    rc, rs = oracle.quant_rows(w["q"])
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("d,hq,hkv,q_head,q0,k0,nk", [
    (256, 6, 1, 0, 0, 0, 128),
    (256, 6, 1, 5, 40, 128, 256),
    (128, 8, 2, 3, 0, 0, 256),
    (128, 4, 4, 2, 100, 256, 128),
])
def test_qk_int32_tile_bit_exact(kvq, oracle, d, hq, hkv, q_head, q0, k0, nk):
    w = _case(610 + q0 + k0, history=400, T=200, hq=hq, hkv=hkv, d=d)
    cache, bt = gpu_cache_from(w, kvq)
    q_codes, _ = kvq.kvq_debug_prefill_q_codes(to_bf16_tensor(w["q"]))
    s = kvq.kvq_debug_prefill_qk_int32(cache, q_codes, bt[0], q_head, q0, k0, nk).cpu().numpy()
    hc = host_cache_from(w, oracle)
    ref = oracle.prefill_qk_int32(q_codes.cpu().numpy(), hc, w["block_table"][0], q_head, q0, 128, k0, nk)
    assert np.array_equal(s, ref)


def _prefill(kvq, w):
    cache, bt = gpu_cache_from(w, kvq)
    out = kvq.kvq_attn_prefill_int8(cache, to_bf16_tensor(w["q"]), w["history"], bt[0], w["softmax_scale"])
    return out.cpu().numpy()


@pytest.mark.parametrize("history,T,d,hq,hkv", [
    (0, 1, 256, 6, 1),
    (0, 130, 256, 6, 1),
    (128, 128, 256, 6, 1),
    (300, 77, 128, 8, 2),
    (1000, 300, 256, 12, 2),
    (4095, 257, 128, 4, 4),
])
def test_prefill_matches_int8_emulation(kvq, oracle, history, T, d, hq, hkv):
    w = _case(700 + history + T, history=history, T=T, hq=hq, hkv=hkv, d=d)
    got = _prefill(kvq, w)
    hc = host_cache_from(w, oracle)
    emul = oracle.prefill_int8_emul(hc, w["q"], history, w["block_table"][0], w["softmax_scale"])
    err = norm_max_err(got, emul)
    ref = oracle.prefill_ref_f64(hc, w["q"], history, w["block_table"][0], w["softmax_scale"])
    print("prefill h=%d T=%d: vs emulation %.3g, vs FP64 %.3g" % (history, T, err, norm_max_err(got, ref)))
    assert err <= GATE and err <= DESIGN_TOL, err
    assert kvq.kvq_device_status() == 0


def test_prefill_outlier_keys_and_wide_scores(kvq, oracle):
    # K outliers and a large softmax scale make tiles with very different P scales and
    # rows whose maximum moves late: exercises the O rescaling across tiles.
    w = _case(720, history=900, T=140, hq=6, hkv=1, d=256, k_outlier_p=0.02)
    w["softmax_scale"] = 0.4
    got = _prefill(kvq, w)
    hc = host_cache_from(w, oracle)
    emul = oracle.prefill_int8_emul(hc, w["q"], w["history"], w["block_table"][0], w["softmax_scale"])
    assert norm_max_err(got, emul) <= DESIGN_TOL


def _n_sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("history,T,d,hq,hkv,wide", [
    (1200, 1024, 256, 6, 1, False),  # long units: tails start at the history's last full tile
    (2000, 1, 128, 24, 4, False),    # a one-token chunk: 24 units become 48 CTAs
    (5000, 700, 128, 32, 8, False),
    (3000, 300, 256, 12, 2, True),   # outlier keys and a large scale: segment maxima far apart
])
def test_prefill_key_range_split(kvq, oracle, history, T, d, hq, hkv, wide):
    """Shapes whose units run as a lead and a tail segment on this GPU (the second segment to
    finish merges the two partial softmax results): against the int8 emulation."""
    assert kvq.kvq_prefill_split_tiles(T, hq, history, _n_sms()) > 0
    w = _case(760 + history + T, history=history, T=T, hq=hq, hkv=hkv, d=d,
              **({"k_outlier_p": 0.02} if wide else {}))
    if wide:
        w["softmax_scale"] = 0.4
    got = _prefill(kvq, w)
    hc = host_cache_from(w, oracle)
    emul = oracle.prefill_int8_emul(hc, w["q"], history, w["block_table"][0], w["softmax_scale"])
    err = norm_max_err(got, emul)
    print("split prefill h=%d T=%d: vs emulation %.3g" % (history, T, err))
    assert err <= GATE and err <= DESIGN_TOL, err
    assert kvq.kvq_device_status() == 0


def test_prefill_32k_full_sampled(kvq, oracle):
    """Workload prefill_32k at full size (2048 queries after 30720 history, 24/4 heads,
    head_dim 256, shuffled pages) in the benchmark's launch configuration (on 152 SMs its
    units are split into lead and tail segments); sampled (token, head) outputs against the
    int8 emulation."""
    w = W.make("prefill_32k")
    got = _prefill(kvq, w)
    hc = host_cache_from(w, oracle)
    units = sample_units(w["n_tokens"], w["hq"], 48, seed=12)
    emul = oracle.prefill_int8_emul(hc, w["q"], w["history"], w["block_table"][0], w["softmax_scale"],
                                    units=units)
    ref = oracle.prefill_ref_f64(hc, w["q"], w["history"], w["block_table"][0], w["softmax_scale"],
                                 units=units)
    g = got.reshape(-1, w["d"])[units]
    err = norm_max_err(g, emul)
    print("prefill_32k sampled: vs emulation %.3g, vs FP64 %.3g" % (err, norm_max_err(g, ref)))
    assert err <= GATE and err <= DESIGN_TOL


def test_prefill_long_history_sampled(kvq, oracle):
    """2048 queries after 122880 history keys (the prefill_32k geometry at four times the
    context: 976 key tiles per head), split into lead and tail segments on this GPU; sampled
    (token, head) outputs against the int8 emulation."""
    w = W.make("prefill_32k", seed=1310, history=122880)
    got = _prefill(kvq, w)
    hc = host_cache_from(w, oracle)
    units = sample_units(w["n_tokens"], w["hq"], 24, seed=1311)
    emul = oracle.prefill_int8_emul(hc, w["q"], w["history"], w["block_table"][0], w["softmax_scale"],
                                    units=units)
    err = norm_max_err(got.reshape(-1, w["d"])[units], emul)
    print("prefill 2048 @ 125k sampled: vs emulation %.3g" % err)
    assert err <= GATE and err <= DESIGN_TOL
    assert kvq.kvq_device_status() == 0
