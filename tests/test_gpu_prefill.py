"""kvq_attn_prefill_int8 on the GPU against the oracle.

Two gates on every output, each independent of the other:
  * the method (its plain definition): against the FP64 attention over the dequantised Q
    codes and the dequantised cache with exact softmax arithmetic (oracle.prefill_qdeq_f64),
    every element within the per-tile P re-quantisation bound that the oracle returns beside
    it, sum_t min(w_t, ps_tile / 2) |v8_t| / l, plus the fp32 rounding slack 3e-5 * mag
    (mag = sum_t p_t |v^_t| / l).  This check does not depend on how the P codes are decided
    in fp32 (exp2 polynomial, tile-maximum basis, rounding trick): a kernel that fed a wrong
    tile, key, scale or code into the contractions falls outside it.
  * the specification (the int8 emulation, Part B, which takes every P-code decision with the
    kernel's fp32 operations): within 2e-3 normalised max-abs (the acceptance gate), and
    within DESIGN_TOL = 1e-4, which catches a single flipped code.
Q codes and the int32 QK score tiles of the production kernel are bit-exact.  The distance to
the FP64 reference over the bf16 Q (Part A; the method's own error, int8 Q and 7-bit P codes,
a few percent of the output RMS) is printed, not gated.
"""
import numpy as np
import pytest

import workloads as W
from helpers import gpu_cache_from, host_cache_from, norm_max_err, sample_units, to_bf16_tensor, to_i32

pytestmark = pytest.mark.gpu

GATE = 2e-3
DESIGN_TOL = 1e-4
SLACK = 3e-5  # fp32 rounding of the kernel's weights and sums, relative to mag


def check_method_bound(got, ref, bound, mag, what):
    """Every element of got within the P re-quantisation bound of the FP64 definition."""
    got = np.asarray(got, np.float64).reshape(ref.shape)
    excess = np.abs(got - ref) - (bound * (1 + 1e-5) + SLACK * mag)
    share = float(np.divide(np.abs(got - ref), bound, out=np.zeros_like(bound), where=bound > 0).max())
    print("%s: |got - FP64(Q codes)| / bound: max %.3f" % (what, share))
    assert excess.max() <= 0, (what, float(excess.max()), np.unravel_index(np.argmax(excess), excess.shape))


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


def _qk_window_ref(oracle, q_codes, hc, bt_row, n_keys, q_head, q0, k0, nk):
    """Exact integer S of the window from the oracle; keys at or past n_keys are zero (the
    production kernel's operands there are zero rows)."""
    ref = np.zeros((128, nk), np.int32)
    real = max(0, min(nk, n_keys - k0))
    if real:
        ref[:, :real] = oracle.prefill_qk_int32(q_codes, hc, bt_row, q_head, q0, 128, k0, real)
    return ref


# (history, T, d, hq, hkv, q_head, q0, k0, nk, split_tiles): which tiles of the unit the window holds
QK_CASES = [
    (400, 200, 256, 6, 1, 0, 0, 0, 640, 0),      # history tiles 0-2, diagonal tiles 3-4, ragged tile 4
    (400, 200, 256, 6, 1, 5, 128, 384, 256, 0),  # second query tile (rows past T), diagonal + ragged
    (1000, 300, 128, 8, 2, 3, 0, 512, 512, 4),   # forced split: lead's last tile 4, tail's first tile 5
    (1000, 300, 256, 12, 2, 7, 256, 640, 512, 3),  # forced split at head_dim 256, a later query tile
    (0, 130, 128, 4, 4, 2, 0, 0, 128, 0),        # no history: the diagonal tile alone
    (1200, 1024, 256, 6, 1, 4, 896, 1024, 1280, -1),  # the split this GPU chooses (if any)
]


@pytest.mark.parametrize("history,T,d,hq,hkv,q_head,q0,k0,nk,split", QK_CASES)
def test_qk_int32_production_kernel_bit_exact(kvq, oracle, history, T, d, hq, hkv, q_head, q0, k0, nk, split):
    """The int32 score tiles of the production attention kernel (its own operand pieces from
    the widening pre-pass, Q widened into tensor memory, the tcgen05 QK issue), copied out of
    tensor memory as the softmax threads load them: bit-exact against the oracle's integer QK.
    The same call's output equals the int8 emulation, and with the call's own split it is the
    output of kvq_attn_prefill_int8 bit for bit."""
    w = _case(610 + history + q0 + k0, history=history, T=T, hq=hq, hkv=hkv, d=d)
    cache, bt = gpu_cache_from(w, kvq)
    q_codes, q_scales = kvq.kvq_debug_prefill_q_codes(to_bf16_tensor(w["q"]))
    s, out = kvq.kvq_debug_prefill_qk_int32(cache, q_codes, q_scales, history, bt[0], w["softmax_scale"], q_head,
                                            q0, k0, nk, split_tiles=split)
    hc = host_cache_from(w, oracle)
    ref = _qk_window_ref(oracle, q_codes.cpu().numpy(), hc, w["block_table"][0], history + T, q_head, q0, k0, nk)
    s = s.cpu().numpy()
    assert np.array_equal(s, ref), np.argwhere(s != ref)[:5]
    assert np.abs(ref).max() > 0
    emul = oracle.prefill_int8_emul(hc, w["q"], history, w["block_table"][0], w["softmax_scale"])
    assert norm_max_err(out.cpu().numpy(), emul) <= DESIGN_TOL
    if split == -1:
        plain = kvq.kvq_attn_prefill_int8(cache, to_bf16_tensor(w["q"]), history, bt[0], w["softmax_scale"])
        assert np.array_equal(out.cpu().numpy().view(np.uint32), plain.cpu().numpy().view(np.uint32))
    assert kvq.kvq_device_status() == 0


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
    check_method_bound(got, *oracle.prefill_qdeq_f64(hc, w["q"], history, w["block_table"][0], w["softmax_scale"]),
                       "prefill h=%d T=%d" % (history, T))
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
    check_method_bound(got, *oracle.prefill_qdeq_f64(hc, w["q"], w["history"], w["block_table"][0],
                                                     w["softmax_scale"]), "outlier keys")


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
    check_method_bound(got, *oracle.prefill_qdeq_f64(hc, w["q"], history, w["block_table"][0], w["softmax_scale"]),
                       "split prefill h=%d T=%d" % (history, T))
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
    check_method_bound(g, *oracle.prefill_qdeq_f64(hc, w["q"], w["history"], w["block_table"][0], w["softmax_scale"],
                                                   units=units), "prefill_32k sampled")


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
    check_method_bound(got.reshape(-1, w["d"])[units],
                       *oracle.prefill_qdeq_f64(hc, w["q"], w["history"], w["block_table"][0], w["softmax_scale"],
                                                units=units), "prefill 2048 @ 125k sampled")
    assert kvq.kvq_device_status() == 0
