"""The quantisation rule on the GPU against the oracle's, over every bf16 value.

The rule every cache writer and the prefill Q quantisation share (amax, scale = amax / 127,
code = clamp(rint(x / scale)), IEEE fp32 quotients).  These rows run every finite bf16 value x
with |x| <= amax through it for amax values that cover exact ties (amax 127, scale 1: every
half-integer is a tie and must round to even), scales across the exponent range, the largest
bf16 value, and subnormal scales.  Gate: codes and scales bit-identical to the oracle."""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import int8_kv_cache_quant_gb300 as k
    k.lib()
    return k


def _all_finite_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = W.bf16_bits_to_f32(bits)
    return bits[np.isfinite(f)], f[np.isfinite(f)]


def _rows_for(amax_bits, d):
    """Rows of d bf16 values: the amax element first, then values with |x| <= amax."""
    bits, f = _all_finite_bf16()
    amax = float(W.bf16_bits_to_f32(np.array([amax_bits], np.uint16))[0])
    sel = bits[np.abs(f) <= amax]
    per = d - 1
    n = (len(sel) + per - 1) // per
    body = np.zeros(n * per, np.uint16)
    body[:len(sel)] = sel
    rows = np.concatenate([np.full((n, 1), amax_bits, np.uint16), body.reshape(n, per)], axis=1)
    return rows


AMAX = [127.0, 1.0, 0.5, 3.0, 100.0, 1.0e-3, 7.25e12, 2.0 ** -60, 2.0 ** 60, 3.3895314e38,
        1.0e-28, 1.0e-36, 2.0 ** -126]


@pytest.mark.parametrize("d", [256, 128])
def test_rule_bit_exact_over_all_bf16(kvq, oracle, d):
    import torch
    rows = np.concatenate([_rows_for(int(W.f32_to_bf16_bits(np.array([a], np.float32))[0]), d) for a in AMAX])
    q = rows[:, None, :]  # [T][1][d]
    qt = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    codes, scales = kvq.kvq_debug_prefill_q_codes(qt)
    ref_codes, ref_scales = oracle.quant_rows(q)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_scales.view(np.uint32))
    got = codes.cpu().numpy()
    bad = np.argwhere(got != ref_codes)
    assert len(bad) == 0, (len(bad), bad[:5])


@pytest.mark.parametrize("d", [256, 128])
def test_rule_non_finite_rows(kvq, oracle, d):
    """Rows holding inf, -inf or NaN beside finite values, and a NaN in an otherwise zero row.
    The rule as written decides them: amax ignores NaN, an infinite amax gives an infinite scale,
    so finite values quantise to 0 and inf / inf = NaN clamps to -127; a zero amax gives zeros.
    Gate: codes and scales bit-identical to the oracle."""
    import torch
    rng = np.random.default_rng(4242 + d)
    inf, nan = np.float32(np.inf), np.float32(np.nan)
    rows = []
    for special in ([inf], [-inf], [nan], [inf, nan], [inf, -inf], [nan, nan]):
        x = rng.normal(size=d).astype(np.float32) * 3
        pos = rng.choice(d, size=len(special), replace=False)
        x[pos] = special
        rows.append(x)
    z = np.zeros(d, np.float32)
    z[7] = nan
    rows.append(z)
    bits = W.f32_to_bf16_bits(np.stack(rows))
    bits[np.isnan(np.stack(rows))] = 0x7FC0  # a quiet NaN pattern in bf16
    q = bits[:, None, :]
    qt = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    codes, scales = kvq.kvq_debug_prefill_q_codes(qt)
    ref_codes, ref_scales = oracle.quant_rows(q)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_scales.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), ref_codes)
