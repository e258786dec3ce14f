"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than its own formula: numbers
printed on the pages (tests/golden/, each with its citation), hand-worked cases, closed
forms of special inputs, invariants (split size, permutation, sub-problem consistency)
and brute force.  The oracle's arithmetic is in oracle/kvq_oracle.cpp.
"""
import json
import os

import numpy as np
import pytest

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf16(x):
    return W.f32_to_bf16_bits(np.asarray(x, np.float32))


def make_cache(oracle, k_bf16, v_bf16, table=None, num_blocks=None):
    """Write tokens 0..T-1 of one sequence (k/v bf16 [T][Hkv][D]) into a fresh cache."""
    T, H, D = k_bf16.shape
    nb = (T + 15) // 16
    if table is None:
        table = np.arange(nb, dtype=np.int32)
    if num_blocks is None:
        num_blocks = int(max(table.max() + 1, nb))
    c = oracle.HostCache(num_blocks, H, D)
    skipped = oracle.kv_quant_write(c, k_bf16, v_bf16, np.zeros(T, np.int32),
                                    np.arange(T, dtype=np.int32), table[None, :])
    assert skipped == 0
    return c, table


# --------------------------------------------------------------------------- bytes

def test_bytes_per_token_match_page(oracle):
    g = golden("dcu_kv_bytes.json")
    H, D = g["n_kv_heads"], g["head_dim"]
    assert oracle.bf16_kv_bytes_per_token(H, D) == g["bf16_kv_bytes"]
    assert oracle.kv_bytes_per_token(H, D) == g["int8_kv_total_bytes"]
    assert 2 * H * D == g["int8_kv_code_bytes"] and 2 * H * 4 == g["fp32_scale_bytes"]
    assert round(100 * g["int8_kv_total_bytes"] / g["bf16_kv_bytes"], 2) == g["ratio_percent_printed"]
    assert round(g["bf16_kv_bytes"] / g["int8_kv_total_bytes"], 2) == g["read_speedup_printed"]


def test_cache_layout_holds_exactly_the_page_byte_count(oracle):
    # The documented layout stores exactly the page's per-token bytes (no padding).
    g = golden("dcu_kv_bytes.json")
    c = oracle.HostCache(8, g["n_kv_heads"], g["head_dim"])
    total = c.k.nbytes + c.v.nbytes + c.k_scale.nbytes + c.v_scale.nbytes
    assert total == 8 * 16 * g["int8_kv_total_bytes"]


# --------------------------------------------------------------------------- quantisation

def test_quant_handworked_rows(oracle):
    g = golden("quant_rows_handworked.json")
    for row in g["rows"]:
        x = bf16(row["x"])
        assert np.array_equal(W.bf16_bits_to_f32(x), np.asarray(row["x"], np.float32))
        codes, scale = oracle.quant_rows(x[None, :])
        assert scale[0] == np.float32(row["scale"])
        assert codes[0].tolist() == row["codes"]


@pytest.mark.parametrize("k", [-9, -3, 0, 2, 7])
def test_quant_exhaustive_bf16_with_exact_scale(oracle, k):
    # amax = 127 * 2^k makes scale = 2^k exact, so each code is round-half-even(x / 2^k)
    # computed exactly in binary64; check every bf16 value in [-amax, amax].
    amax = np.float32(127.0 * 2.0 ** k)
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = W.bf16_bits_to_f32(allbits)
    ok = np.isfinite(vals) & (np.abs(vals) <= amax)
    xs = allbits[ok]
    n = 256
    pad = (-len(xs)) % (n - 1)
    xs = np.concatenate([xs, np.zeros(pad, np.uint16)])
    rows = xs.reshape(-1, n - 1)
    amax_bits = bf16([amax])[0]
    rows = np.concatenate([rows, np.full((rows.shape[0], 1), amax_bits, np.uint16)], axis=1)
    codes, scales = oracle.quant_rows(rows)
    assert np.all(scales == np.float32(2.0 ** k))
    expect = np.array([round(float(v) / 2.0 ** k) for v in W.bf16_bits_to_f32(rows).ravel()],
                      dtype=np.int64).reshape(rows.shape)
    assert np.array_equal(codes.astype(np.int64), expect)


def test_quant_properties_random(oracle):
    rng = np.random.default_rng(1)
    x = W.normal_bf16(rng, (4096, 128), outlier_p=0.02)
    codes, scales = oracle.quant_rows(x)
    xf = W.bf16_bits_to_f32(x).astype(np.float64)
    amax = np.abs(xf).max(axis=1)
    # the largest element maps to +-127; codes stay in [-127, 127]
    assert np.all(np.abs(codes).max(axis=1) == 127)
    assert codes.min() >= -127
    # scale is amax / 127 to fp32 precision
    assert np.allclose(scales.astype(np.float64), amax / 127.0, rtol=2 ** -23, atol=0)
    # round to nearest: each code is within 1/2 (plus fp32 slack) of x * 127 / amax
    err = np.abs(codes - xf * 127.0 / amax[:, None])
    assert err.max() <= 0.5 + 1e-5
    # odd symmetry and monotonicity
    neg = x ^ np.uint16(0x8000)
    codes_neg, _ = oracle.quant_rows(neg)
    assert np.array_equal(codes_neg, -codes)
    order = np.argsort(xf, axis=1, kind="stable")
    assert np.all(np.diff(np.take_along_axis(codes.astype(np.int32), order, axis=1), axis=1) >= 0)


def test_quant_zero_row(oracle):
    codes, scales = oracle.quant_rows(np.zeros((3, 64), np.uint16))
    assert np.all(codes == 0) and np.all(scales == 0)


# --------------------------------------------------------------------------- cache write

def test_kv_quant_write_layout_round_trip(oracle):
    rng = np.random.default_rng(2)
    T, H, D = 53, 3, 128
    k = W.normal_bf16(rng, (T, H, D))
    v = W.normal_bf16(rng, (T, H, D))
    table = rng.permutation(8).astype(np.int32)[:4]
    c, _ = make_cache(oracle, k, v, table=table, num_blocks=8)
    kc, ks = oracle.quant_rows(k)
    vc, vs = oracle.quant_rows(v)
    for t in range(T):
        page, slot = table[t // 16], t % 16
        for h in range(H):
            # read back through the array axes [page][head][d/16][slot][d%16] etc.
            assert np.array_equal(c.k[page, h, :, slot, :].reshape(D), kc[t, h])
            assert np.array_equal(c.v[page, h, :, slot], vc[t, h])
            assert c.k_scale[page, h, slot] == ks[t, h]
            assert c.v_scale[page, h, slot] == vs[t, h]
    # pages not in the table stay untouched
    unused = sorted(set(range(8)) - set(table.tolist()))
    assert not c.k[unused].any() and not c.v[unused].any()


def test_kv_quant_write_skips_out_of_range(oracle):
    c = oracle.HostCache(2, 1, 128)
    k = np.zeros((4, 1, 128), np.uint16)
    table = np.array([[0, 5]], np.int32)  # page 5 does not exist
    skipped = oracle.kv_quant_write(c, k, k, np.array([0, 1, 0, 0], np.int32),
                                    np.array([0, 0, 20, 40], np.int32), table)
    # seq 1 does not exist; pos 20 maps to page 5; pos 40 is past the table
    assert skipped == 3


# --------------------------------------------------------------------------- Part A decode

def test_two_key_worked_example(oracle):
    g = golden("two_key_softmax.json")
    D = 16
    k = np.zeros((2, 1, D), np.float32)
    v = np.zeros((2, 1, D), np.float32)
    k[0, 0, 0], k[1, 0, 0] = 1.0, -1.0
    v[0, 0, 1], v[1, 0, 2] = 1.0, 1.0
    c, table = make_cache(oracle, bf16(k), bf16(v))
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = 1.0
    out = oracle.decode_f64(c, bf16(q), table[None, :], np.array([2], np.int32), 1.0)
    assert np.allclose(out[0, 0], g["expected_out"], atol=g["tolerance"], rtol=0)
    sc = g["scaled_case"]
    out = oracle.decode_f64(c, bf16(q), table[None, :], np.array([2], np.int32),
                            sc["softmax_scale"])
    assert np.allclose(out[0, 0], sc["expected_out"], atol=g["tolerance"], rtol=0)


def test_equal_scores_constant_v_gives_v(oracle):
    # all K codes equal -> all scores equal; V rows identical -> output is exactly v^.
    rng = np.random.default_rng(3)
    T, H, D, Hq = 37, 2, 128, 6
    k = np.tile(W.normal_bf16(rng, (1, H, D)), (T, 1, 1))
    vrow = W.normal_bf16(rng, (1, H, D))
    v = np.tile(vrow, (T, 1, 1))
    c, table = make_cache(oracle, k, v)
    q = W.normal_bf16(rng, (1, Hq, D))
    out = oracle.decode_f64(c, q, table[None, :], np.array([T], np.int32), 1 / np.sqrt(D))
    vc, vs = oracle.quant_rows(vrow)
    vhat = vc[0].astype(np.float64) * vs[0][:, None].astype(np.float64)
    for h in range(Hq):
        assert np.array_equal(out[0, h], vhat[h // 3])


def test_ctx_one_gives_v0_and_ctx_zero_gives_zeros(oracle):
    rng = np.random.default_rng(4)
    H, D = 1, 256
    k = W.normal_bf16(rng, (5, H, D))
    v = W.normal_bf16(rng, (5, H, D))
    c, table = make_cache(oracle, k, v)
    q = W.normal_bf16(rng, (2, 4, D))
    bt = np.stack([table, table])
    out = oracle.decode_f64(c, q, bt, np.array([1, 0], np.int32), 0.0625)
    vc, vs = oracle.quant_rows(v[0])
    vhat = vc[0].astype(np.float64) * np.float64(vs[0])
    assert np.array_equal(out[0, 0], vhat) and np.array_equal(out[0, 3], vhat)
    assert not out[1].any()


def test_dominant_key(oracle):
    # one key aligned with q and a huge softmax scale: output -> that key's v^.
    rng = np.random.default_rng(5)
    T, D = 40, 128
    k = W.normal_bf16(rng, (T, 1, D))
    v = W.normal_bf16(rng, (T, 1, D))
    q = k[17:18].copy()
    c, table = make_cache(oracle, k, v)
    out = oracle.decode_f64(c, q, table[None, :], np.array([T], np.int32), 50.0)
    vc, vs = oracle.quant_rows(v[17])
    assert np.allclose(out[0, 0], vc[0] * np.float64(vs[0]), atol=1e-9)


def test_permutation_invariance(oracle):
    # the same tokens stored in a different order (and pages) give the same output
    rng = np.random.default_rng(6)
    T, H, D = 48, 2, 128
    k = W.normal_bf16(rng, (T, H, D))
    v = W.normal_bf16(rng, (T, H, D))
    q = W.normal_bf16(rng, (1, 4, D))
    c1, t1 = make_cache(oracle, k, v)
    perm = rng.permutation(T)
    c2, t2 = make_cache(oracle, k[perm], v[perm], table=np.array([2, 0, 1], np.int32))
    o1 = oracle.decode_f64(c1, q, t1[None, :], np.array([T], np.int32), 0.1)
    o2 = oracle.decode_f64(c2, q, t2[None, :], np.array([T], np.int32), 0.1)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("split", [1, 7, 16, 512, 1000])
def test_split_merge_invariance(oracle, split):
    rng = np.random.default_rng(7)
    B, T, H, D, Hq = 2, 1000, 2, 128, 4
    w = W.make("decode_b64", seed=11, batch=B, ctx_range=(300, T), hq=Hq, hkv=H, d=D)
    c = oracle.HostCache(w["num_blocks"], H, D)
    oracle.kv_quant_write(c, w["k_fill"], w["v_fill"], w["fill_seq"], w["fill_pos"],
                          w["block_table"])
    ref = oracle.decode_f64(c, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    got = oracle.decode_split_f64(c, w["q"], w["block_table"], w["ctx_lens"],
                                  w["softmax_scale"], split)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_units_sampling_matches_full(oracle):
    w = W.make("decode_b64", seed=12, batch=3, ctx_range=(20, 90), hq=8, hkv=2, d=128)
    c = oracle.HostCache(w["num_blocks"], 2, 128)
    oracle.kv_quant_write(c, w["k_fill"], w["v_fill"], w["fill_seq"], w["fill_pos"],
                          w["block_table"])
    full = oracle.decode_f64(c, w["q"], w["block_table"], w["ctx_lens"], 0.1)
    units = np.array([0, 5, 9, 23], np.int64)
    part = oracle.decode_f64(c, w["q"], w["block_table"], w["ctx_lens"], 0.1, units=units)
    assert np.array_equal(part, full.reshape(-1, 128)[units])


# --------------------------------------------------------------------------- verify decode

def _verify_case(oracle, seed, ctx, nq, hq, hkv, d):
    """Sequences b = 0.. with ctx[b] tokens in shuffled pages of one cache; returns the cache,
    the block table, the logical K/V (bf16 bits [b][t][Hkv][D]) and q [B][nq][Hq][D]."""
    rng = np.random.default_rng(seed)
    B = len(ctx)
    mb = max((c + 15) // 16 for c in ctx)
    pages = rng.permutation(B * mb).astype(np.int32)
    table = pages.reshape(B, mb)
    cache = oracle.HostCache(B * mb, hkv, d)
    ks, vs = [], []
    for b, n in enumerate(ctx):
        k = W.normal_bf16(rng, (n, hkv, d), outlier_p=0.02)
        v = W.normal_bf16(rng, (n, hkv, d))
        assert oracle.kv_quant_write(cache, k, v, np.full(n, b, np.int32), np.arange(n, dtype=np.int32),
                                     table) == 0
        ks.append(k)
        vs.append(v)
    q = W.normal_bf16(rng, (B, nq, hq, d))
    return cache, table, ks, vs, q


def test_verify_brute_force_causal_rows(oracle):
    # numpy from the quantisation rule alone: row i of sequence b sees keys t <= ctx - nq + i;
    # the second sequence is shorter than nq (its first row sees no key: zeros)
    ctx, nq, hq, hkv, d, scale = [37, 2, 16], 3, 6, 2, 128, 0.09
    cache, table, ks, vs, q = _verify_case(oracle, 31, ctx, nq, hq, hkv, d)
    out = oracle.verify_f64(cache, q, table, np.array(ctx, np.int32), scale)
    G = hq // hkv
    qf = W.bf16_bits_to_f32(q).astype(np.float64)
    for b, n in enumerate(ctx):
        kc, ksc = oracle.quant_rows(ks[b])
        vc, vsc = oracle.quant_rows(vs[b])
        kh = kc.astype(np.float64) * ksc[..., None].astype(np.float64)   # [n][Hkv][D]
        vh = vc.astype(np.float64) * vsc[..., None].astype(np.float64)
        for i in range(nq):
            nk = max(0, min(n, n - nq + 1 + i))
            for h in range(hq):
                if nk == 0:
                    assert not out[b, i, h].any()
                    continue
                s = scale * (kh[:nk, h // G] @ qf[b, i, h])
                p = np.exp(s - s.max())
                ref = (p / p.sum()) @ vh[:nk, h // G]
                assert np.allclose(out[b, i, h], ref, rtol=1e-11, atol=1e-13), (b, i, h)


def test_verify_rows_equal_prefill_chunk_and_decode(oracle):
    # the nq verify rows of a sequence are the causal chunk of nq queries after ctx - nq
    # history keys; with nq = 1 verify is plain decode
    ctx, nq, hq, hkv, d, scale = [70, 41], 4, 8, 2, 256, 0.0625
    cache, table, _, _, q = _verify_case(oracle, 32, ctx, nq, hq, hkv, d)
    out = oracle.verify_f64(cache, q, table, np.array(ctx, np.int32), scale)
    for b, n in enumerate(ctx):
        ref = oracle.prefill_ref_f64(cache, q[b], n - nq, table[b], scale)
        assert np.array_equal(out[b], ref)
    one = oracle.verify_f64(cache, q[:, :1], table, np.array(ctx, np.int32), scale)
    dec = oracle.decode_f64(cache, q[:, 0], table, np.array(ctx, np.int32), scale)
    assert np.array_equal(one[:, 0], dec)
    units = np.array([0, 9, 31, 40, 63], np.int64)
    part = oracle.verify_f64(cache, q, table, np.array(ctx, np.int32), scale, units=units)
    assert np.array_equal(part, out.reshape(-1, d)[units])


# --------------------------------------------------------------------------- first prefill chunk

def test_prefill_first_brute_force(oracle):
    # numpy over the bf16 values: row i is softmax over keys 0..i (causal), GQA 3
    rng = np.random.default_rng(41)
    T, Hq, Hkv, D, scale = 19, 6, 2, 128, 0.07
    q, k, v = (W.normal_bf16(rng, (T, h, D)) for h in (Hq, Hkv, Hkv))
    out = oracle.prefill_first_f64(q, k, v, scale)
    qf, kf, vf = (W.bf16_bits_to_f32(x).astype(np.float64) for x in (q, k, v))
    for i in range(T):
        for h in range(Hq):
            s = scale * (kf[:i + 1, h // 3] @ qf[i, h])
            p = np.exp(s - s.max())
            assert np.allclose(out[i, h], (p / p.sum()) @ vf[:i + 1, h // 3], rtol=1e-12, atol=1e-14)


def test_prefill_first_closed_forms(oracle):
    # row 0 sees only key 0: output is v_0 exactly; with every K row equal the weights are
    # uniform, so row i is the mean of v_0..v_i
    rng = np.random.default_rng(42)
    T, Hq, D = 9, 4, 256
    k = np.tile(W.normal_bf16(rng, (1, 1, D)), (T, 1, 1))
    v = W.normal_bf16(rng, (T, 1, D))
    q = W.normal_bf16(rng, (T, Hq, D))
    out = oracle.prefill_first_f64(q, k, v, 1 / 16)
    vf = W.bf16_bits_to_f32(v).astype(np.float64)[:, 0]
    for h in range(Hq):
        assert np.array_equal(out[0, h], vf[0])
    for i in range(T):
        assert np.allclose(out[i, 2], vf[:i + 1].mean(axis=0), rtol=1e-13, atol=1e-15)
    units = np.array([0, 7, 35], np.int64)
    assert np.array_equal(oracle.prefill_first_f64(q, k, v, 1 / 16, units=units), out.reshape(-1, D)[units])


# --------------------------------------------------------------------------- prefill

def _prefill_case(oracle, seed, history, T, hq=4, hkv=2, d=128, **kw):
    w = W.make("prefill_32k", seed=seed, history=history, chunk=T, hq=hq, hkv=hkv, d=d, **kw)
    c = oracle.HostCache(w["num_blocks"], hkv, d)
    oracle.kv_quant_write(c, w["k_fill"], w["v_fill"], w["fill_seq"], w["fill_pos"],
                          w["block_table"])
    return w, c


def test_prefill_rows_equal_decode_at_their_position(oracle):
    w, c = _prefill_case(oracle, 21, history=70, T=9)
    bt = w["block_table"][0]
    out = oracle.prefill_ref_f64(c, w["q"], w["history"], bt, w["softmax_scale"])
    for i in range(w["n_tokens"]):
        dec = oracle.decode_f64(c, w["q"][i:i + 1], bt[None, :],
                                np.array([w["history"] + i + 1], np.int32), w["softmax_scale"])
        assert np.array_equal(out[i], dec[0])


def test_qk_int32_brute_force(oracle):
    w, c = _prefill_case(oracle, 22, history=200, T=40, hq=6, hkv=2, d=256)
    bt = w["block_table"][0]
    _, qc, qs = oracle.prefill_int8_emul(c, w["q"], w["history"], bt, w["softmax_scale"],
                                         want_q_codes=True)
    kc, _ = oracle.quant_rows(w["k_fill"])  # [ctx][Hkv][D], logical order
    for h in (0, 4):
        s = oracle.prefill_qk_int32(qc, c, bt, h, 8, 40, 32, 200)
        expect = np.zeros((40, 200), np.int64)
        nrows = w["n_tokens"] - 8
        expect[:nrows] = qc[8:, h].astype(np.int64) @ kc[32:232, h // 3].astype(np.int64).T
        assert np.array_equal(s.astype(np.int64), expect)


def test_q_codes_equal_row_quantisation(oracle):
    w, c = _prefill_case(oracle, 23, history=10, T=7)
    _, qc, qs = oracle.prefill_int8_emul(c, w["q"], 10, w["block_table"][0], 0.1,
                                         want_q_codes=True)
    rc, rs = oracle.quant_rows(w["q"])
    assert np.array_equal(qc, rc) and np.array_equal(qs, rs)


def test_int8_emul_single_tile_equal_weights_is_exact(oracle):
    # all K codes zero -> all scores equal; one V scale for every token; one tile holds
    # every key -> every P code is 127 and Part B equals the mean of v^ = Part A.
    rng = np.random.default_rng(8)
    T, hist, D = 20, 60, 128
    ctx = T + hist
    k = np.zeros((ctx, 1, D), np.uint16)
    v = W.normal_bf16(rng, (ctx, 1, D))
    v[:, 0, 0] = bf16([4.0])[0]  # same amax in every row -> same V scale
    v[:, 0, 1:] = W.f32_to_bf16_bits(np.clip(W.bf16_bits_to_f32(v[:, 0, 1:]), -3.9, 3.9))
    c, table = make_cache(oracle, k, v)
    q = W.normal_bf16(rng, (T, 2, D))
    a = oracle.prefill_ref_f64(c, q, hist, table, 0.1)
    b = oracle.prefill_int8_emul(c, q, hist, table, 0.1, pv_tile=128)
    # exact up to the fp32 rounding of w = p * sV (2^-24 relative)
    assert np.allclose(b, a, rtol=2e-7, atol=1e-12)


def test_int8_emul_tiles_are_aligned_at_absolute_multiples_of_128(oracle):
    # Equal scores (K codes zero); keys 0..127 have V scale a, keys 128.. have V scale
    # a/2.  With one P scale per absolute 128-key tile every code is 127 and Part B is
    # exact; a tile straddling key 128 (or one scale per row) would give codes 64 there.
    rng = np.random.default_rng(13)
    hist, T, D = 200, 56, 128
    ctx = hist + T
    k = np.zeros((ctx, 1, D), np.uint16)
    vf = rng.uniform(-0.9, 0.9, size=(ctx, 1, D)).astype(np.float32)
    vf[128:] *= 0.5
    vf[:128, 0, 0], vf[128:, 0, 0] = 1.0, 0.5  # row amax 1 (keys < 128) and 1/2 (the rest)
    v = W.f32_to_bf16_bits(vf)
    c, table = make_cache(oracle, k, v)
    q = W.normal_bf16(rng, (T, 2, D))
    a = oracle.prefill_ref_f64(c, q, hist, table, 0.1)
    b = oracle.prefill_int8_emul(c, q, hist, table, 0.1, pv_tile=128)
    assert np.allclose(b, a, rtol=2e-7, atol=1e-12)
    # the same data with 96-key tiles mixes the two scales and is no longer exact
    b96 = oracle.prefill_int8_emul(c, q, hist, table, 0.1, pv_tile=96)
    assert np.abs(b96 - a).max() > 1e-4


def test_int8_emul_tile_order_does_not_change_the_codes(oracle):
    # Rows that see every history key attend over the same (key, value) set whichever order
    # the history's 128-key tiles come in.  Each tile's P codes are decided from the tile
    # alone (relative to its own maximum score), so exchanging two whole tiles leaves every
    # code, and the output up to double rounding, unchanged.  Decided relative to the
    # running maximum instead, the fp32 codes would differ in near-tie cases (a rounding flip
    # moves a row by ~1e-3 of the output RMS), so this pins the decision basis.
    rng = np.random.default_rng(17)
    hist, T, H, G, D = 512, 64, 2, 4, 128
    ctx = hist + T
    k = W.normal_bf16(rng, (ctx, H, D), 0.01)
    v = W.normal_bf16(rng, (ctx, H, D))
    q = W.normal_bf16(rng, (T, H * G, D))
    perm = np.arange(ctx)
    perm[0:128], perm[256:384] = np.arange(256, 384), np.arange(0, 128)  # tiles 0 and 2 exchanged
    c1, table = make_cache(oracle, k, v)
    c2, _ = make_cache(oracle, k[perm], v[perm])
    a = oracle.prefill_int8_emul(c1, q, hist, table, 0.3)
    b = oracle.prefill_int8_emul(c2, q, hist, table, 0.3)
    rms = np.sqrt((a ** 2).mean())
    assert np.abs(a - b).max() <= 1e-12 * rms
    # and the exchange is real: a row at position 300 sees only part of tile 2, so its
    # visible key set, and its output, change
    a1 = oracle.prefill_int8_emul(c1, q[:1], 300, table, 0.3)
    b1 = oracle.prefill_int8_emul(c2, q[:1], 300, table, 0.3)
    assert np.abs(a1 - b1).max() > 1e-3 * rms


def test_int8_emul_error_within_p_quantisation_bound(oracle):
    # Q chosen exactly representable by its codes (amax = 127/128, values on the 2^-7
    # grid), so the scores of Part A and Part B agree; the only difference is the
    # per-tile P code rounding, bounded per output element by
    #   sum_tiles ps/2 * sum_t |v8_t[d]| / l.
    rng = np.random.default_rng(9)
    hist, T, H, D, Hq = 300, 30, 1, 128, 2
    ctx = hist + T
    k = W.normal_bf16(rng, (ctx, H, D))
    v = W.normal_bf16(rng, (ctx, H, D))
    c, table = make_cache(oracle, k, v)
    qi = rng.integers(-127, 128, size=(T, Hq, D))
    qi[:, :, 0] = 127
    q = bf16(qi.astype(np.float32) / 128.0)
    scale = 1 / np.sqrt(D)
    a = oracle.prefill_ref_f64(c, q, hist, table, scale)
    b = oracle.prefill_int8_emul(c, q, hist, table, scale)
    vc, vs = oracle.quant_rows(v)
    kc, ks = oracle.quant_rows(k)
    for i in range(T):
        for h in range(Hq):
            nk = hist + i + 1
            s = (qi[i, h].astype(np.float64) / 128.0) @ (kc[:nk, 0].astype(np.float64).T) \
                * ks[:nk, 0] * scale
            p = np.exp(s - s.max())
            wts = p * vs[:nk, 0]
            bound = np.zeros(D)
            for t0 in range(0, nk, 128):
                sl = slice(t0, min(nk, t0 + 128))
                ps = wts[sl].max() / 127.0
                bound += ps / 2 * np.abs(vc[sl, 0]).sum(axis=0)
            bound /= p.sum()
            # slack for the fp32 scores and the exp2 polynomial (relative error < 5e-6)
            slack = 1e-5 * np.abs(a[i, h]).max() + 1e-12
            assert np.all(np.abs(b[i, h] - a[i, h]) <= bound + slack)
    # the method's own error (7-bit P codes) is a few percent of the output RMS here
    rms = np.sqrt((a ** 2).mean())
    assert np.abs(b - a).max() / rms < 0.1


# --------------------------------------------------------------------------- prefill, Q dequantised (FP64)

def test_qdeq_equals_part_a_when_q_is_exactly_its_codes(oracle):
    # Q rows on the 2^-7 grid with amax 127/128 are exactly code * scale (scale = 1/128), so
    # the Q-dequantised reference must equal Part A over the bf16 Q.
    rng = np.random.default_rng(21)
    hist, T, H, D, Hq = 200, 20, 2, 128, 4
    k = W.normal_bf16(rng, (hist + T, H, D))
    v = W.normal_bf16(rng, (hist + T, H, D))
    c, table = make_cache(oracle, k, v)
    qi = rng.integers(-127, 128, size=(T, Hq, D))
    qi[:, :, 3] = -127
    q = bf16(qi.astype(np.float32) / 128.0)
    a = oracle.prefill_ref_f64(c, q, hist, table, 0.2)
    b, bound, mag = oracle.prefill_qdeq_f64(c, q, hist, table, 0.2)
    assert np.abs(a - b).max() <= 1e-12 * np.abs(a).max()
    # mag bounds |out| (triangle inequality), bound is positive and far below mag
    assert np.all(np.abs(b) <= mag * (1 + 1e-12))
    assert np.all(bound > 0) and np.all(bound <= mag)


def test_qdeq_single_key_closed_form(oracle):
    # Row 0 of a chunk with no history sees key 0 alone: p = 1, l = 1, out = v^_0, and the
    # bound is (sV / 127) / 2 * |v8_0| = |v^_0| / 254, mag = |v^_0|.
    rng = np.random.default_rng(22)
    D = 256
    k = W.normal_bf16(rng, (3, 1, D))
    v = W.normal_bf16(rng, (3, 1, D))
    c, table = make_cache(oracle, k, v)
    q = W.normal_bf16(rng, (3, 2, D))
    out, bound, mag = oracle.prefill_qdeq_f64(c, q, 0, table, 1 / 16)
    vc, vs = oracle.quant_rows(v)
    v0 = vc[0, 0].astype(np.float64) * np.float64(vs[0, 0])
    for h in range(2):
        assert np.array_equal(out[0, h], v0)
        assert np.allclose(bound[0, h], np.abs(v0) / 254, rtol=1e-15, atol=0)
        assert np.array_equal(mag[0, h], np.abs(v0))


def test_qdeq_bound_is_per_tile_at_absolute_multiples_of_128(oracle):
    # Zero K rows give every key the same score (p = 1, l = n).  Keys of tile 0 (positions
    # 0..127) get V rows of amax 1 (sV = 1/127), keys of tile 1 amax 64: each tile's P scale is
    # its own sV / 127, every weight of a tile is 127 of its P scale (min(w, ps / 2) = ps / 2), so
    # bound = (sum_tiles sV_tile * sum_{t in tile} |v8_t|) / (254 n).  One scale for the whole
    # row, or tiles counted from the row's first key, would give another number.
    rng = np.random.default_rng(23)
    hist, T, D = 150, 2, 128
    n = hist + T
    k = np.zeros((n, 1, D), np.uint16)
    vf = rng.uniform(-1, 1, size=(n, 1, D)).astype(np.float32)
    vf[:, 0, 0] = 1.0
    vf[128:] *= 64.0
    v = bf16(vf)
    c, table = make_cache(oracle, k, v)
    q = W.normal_bf16(rng, (T, 1, D))
    out, bound, _ = oracle.prefill_qdeq_f64(c, q, hist, table, 0.1)
    vc, vs = oracle.quant_rows(v)
    assert vs[0, 0] == np.float32(1 / 127) and vs[130, 0] == np.float32(64 / 127)
    for i in range(T):
        nk = hist + i + 1
        expect = (np.float64(vs[0, 0]) * np.abs(vc[:128, 0].astype(np.float64)).sum(axis=0) +
                  np.float64(vs[128, 0]) * np.abs(vc[128:nk, 0].astype(np.float64)).sum(axis=0)) / (254 * nk)
        assert np.allclose(bound[i, 0], expect, rtol=1e-12, atol=0)
        vhat = vc[:nk, 0].astype(np.float64) * vs[:nk, 0, None].astype(np.float64)
        assert np.allclose(out[i, 0], vhat.mean(axis=0), rtol=1e-12, atol=1e-15)


def test_int8_emul_within_the_qdeq_bound(oracle):
    # Part B differs from the Q-dequantised reference only by the per-tile P rounding (and
    # fp32 arithmetic): every element within bound + 2e-5 * mag, on N(0,1) inputs with a ragged
    # last tile, and on K outliers with a large softmax scale (tiles with very different P
    # scales).
    for seed, hist, T, outl, scale in ((24, 300, 40, 0.0, 1 / np.sqrt(128)), (25, 900, 20, 0.02, 0.4)):
        w, c = _prefill_case(oracle, seed, history=hist, T=T, hq=4, hkv=2, d=128, k_outlier_p=outl)
        emul = oracle.prefill_int8_emul(c, w["q"], hist, w["block_table"][0], scale)
        ref, bound, mag = oracle.prefill_qdeq_f64(c, w["q"], hist, w["block_table"][0], scale)
        excess = np.abs(emul - ref) - (bound + 2e-5 * mag)
        assert excess.max() <= 0, excess.max()
        # the bound is not vacuous: the method's error reaches a visible share of it
        assert (np.abs(emul - ref) / bound).max() > 0.1


def test_int8_emul_uniform_v_close_to_v(oracle):
    rng = np.random.default_rng(10)
    hist, T, D = 140, 12, 128
    ctx = hist + T
    k = W.normal_bf16(rng, (ctx, 1, D))
    vrow = W.normal_bf16(rng, (1, 1, D))
    v = np.tile(vrow, (ctx, 1, 1))
    c, table = make_cache(oracle, k, v)
    q = W.normal_bf16(rng, (T, 3, D))
    b = oracle.prefill_int8_emul(c, q, hist, table, 1 / np.sqrt(D))
    vc, vs = oracle.quant_rows(vrow)
    vhat = vc[0, 0] * np.float64(vs[0, 0])
    # sum of quantised weights / sum of exact weights is within 1/254 per tile of 1
    assert np.allclose(b, vhat[None, None, :], rtol=1 / 200, atol=1e-12)


def test_exp2_det_coefficients_are_the_minimax_fit(oracle):
    # The polynomial's four coefficients are the ones the committed Remez fit produces (rounded to
    # fp32): the fit is the minimax relative error of 2^f on [-1/2, 1/2] with constant term 1.
    from oracle import fit_exp2_poly as fit
    c, err = fit.remez()
    assert 2.7e-6 < err < 2.9e-6
    src = open(os.path.join(os.path.dirname(GOLDEN), "..", "oracle", "kvq_oracle.cpp")).read()
    body = src[src.index("float exp2_det(float x) {"):]
    body = body[:body.index("\n}\n")]
    for ci in np.asarray(c, np.float32):
        assert ("%.9gf" % ci) in body, ci
    # and the fitted polynomial's error, exactly evaluated, is its minimax value
    grid = np.linspace(-0.5, 0.5, 100001)
    assert np.abs(fit._err(np.asarray(c, np.float32).astype(np.float64), grid)).max() < 2.9e-6


def test_exp2_det_against_exp2(oracle):
    import math
    xs = np.concatenate([np.linspace(-124.9, 0.0, 20001), -np.arange(0, 125, dtype=np.float64),
                         np.linspace(-1, 1, 2001)])
    for x in xs.astype(np.float32):
        got = oracle.exp2_det(float(x))
        ref = 2.0 ** float(x)
        assert abs(got - ref) <= 5e-6 * ref, (x, got, ref)
    for n in range(-125, 2):  # integers: f = 0, polynomial is exactly 1
        assert oracle.exp2_det(float(n)) == 2.0 ** n
    # below -125 the argument is clamped: 2^-125 (NaN is clamped the same way)
    for x in (-125.5, -126.0, -1000.0, float("-inf"), float("nan")):
        assert oracle.exp2_det(x) == 2.0 ** -125, x


# --------------------------------------------------------------------------- sparse

def test_sparse_full_cells_equal_causal_reference(oracle):
    w, c = _prefill_case(oracle, 31, history=50, T=6, hq=6, hkv=1, d=256)
    bt = w["block_table"][0]
    T, hist = w["n_tokens"], w["history"]
    offsets = np.zeros(T + 1, np.int32)
    cells = []
    for i in range(T):
        cells.append(np.arange(hist + i + 1, dtype=np.int32))
        offsets[i + 1] = offsets[i] + hist + i + 1
    cells = np.concatenate(cells)
    ref = oracle.prefill_ref_f64(c, w["q"], hist, bt, w["softmax_scale"])
    got = oracle.sparse_f64(c, w["q"], offsets, cells, bt, w["softmax_scale"])
    assert np.array_equal(got, ref)


def test_sparse_single_cell_and_empty(oracle):
    rng = np.random.default_rng(12)
    T, D = 30, 128
    k = W.normal_bf16(rng, (T, 1, D))
    v = W.normal_bf16(rng, (T, 1, D))
    c, table = make_cache(oracle, k, v)
    q = W.normal_bf16(rng, (2, 2, D))
    offsets = np.array([0, 1, 1], np.int32)
    cells = np.array([13], np.int32)
    out = oracle.sparse_f64(c, q, offsets, cells, table, 0.1)
    vc, vs = oracle.quant_rows(v[13])
    assert np.array_equal(out[0, 1], vc[0] * np.float64(vs[0]))
    assert not out[1].any()


def test_sparse_workload_matches_page_shape():
    g = golden("qsa_cells.json")
    w = W.make("sparse_32k", n_queries=16)
    off, cells = w["cell_offsets"], w["cells"]
    counts = np.diff(off)
    assert np.all(counts == g["cells_per_query"]) and g["sampled"] + g["tail"] == g["cells_per_query"]
    assert w["hq"] // w["hkv"] == g["q_heads_per_kv_head"] and w["d"] == g["head_dim"]
    for i, p in enumerate(w["positions"]):
        cl = cells[off[i]:off[i + 1]]
        assert np.all(np.diff(cl) > 0) and cl[-1] == p and cl[-3] == p - 2 and cl[0] >= 0


# --------------------------------------------------------------------------- fused producer (RoPE)

def _rope_table(max_pos, r, base=10000.0):
    inv = base ** (-np.arange(0, r, 2, dtype=np.float64) / r)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def _identity_table(max_pos, r):
    return np.concatenate([np.ones((max_pos, r // 2)), np.zeros((max_pos, r // 2))], axis=1).astype(np.float32)


def test_rope_identity_table_is_the_plain_producer(oracle):
    rng = np.random.default_rng(21)
    T, H, Hq, D = 37, 2, 6, 128
    k = W.normal_bf16(rng, (T, H, D), outlier_p=0.02)
    v = W.normal_bf16(rng, (T, H, D))
    q = W.normal_bf16(rng, (T, Hq, D))
    table = np.arange(3, dtype=np.int32)
    c1, _ = make_cache(oracle, k, v, table=table, num_blocks=3)
    c2 = oracle.HostCache(3, H, D)
    skipped, qc, qs, qr = oracle.rope_quant_write(c2, q, k, v, np.zeros(T, np.int32), np.arange(T, dtype=np.int32),
                                                  table[None, :], _identity_table(64, D), D)
    assert skipped == 0
    for a, b in ((c1.k, c2.k), (c1.v, c2.v), (c1.k_scale, c2.k_scale), (c1.v_scale, c2.v_scale)):
        assert np.array_equal(a, b)
    rc, rs = oracle.quant_rows(q)
    assert np.array_equal(qc, rc) and np.array_equal(qs.view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(qr, q)


def test_rope_quarter_and_half_turns_are_exact(oracle):
    # head_dim 16, rotary_dim 8: pairs (i, i + 4) turned by 0, 90, 180, 270 degrees; the turned
    # values are sign changes and swaps of bf16 values, so the expected row is exact:
    # (x1, x2) -> (x1 cos - x2 sin, x2 cos + x1 sin)
    D, r = 16, 8
    x = np.array([1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 16], np.float32) * 0.25
    cs = np.array([[1, 0, -1, 0, 0, 1, 0, -1]], np.float32)  # cos for the 4 pairs, then sin
    expect = x.copy()
    expect[0], expect[4] = x[0], x[4]        # 0 degrees
    expect[1], expect[5] = -x[5], x[1]       # 90
    expect[2], expect[6] = -x[2], -x[6]      # 180
    expect[3], expect[7] = x[7], -x[3]       # 270
    c = oracle.HostCache(1, 1, D)
    kb = bf16(x)[None, None, :]
    skipped, qc, qs, qr = oracle.rope_quant_write(c, kb, kb, kb, np.zeros(1, np.int32), np.zeros(1, np.int32),
                                                  np.zeros((1, 1), np.int32), cs, r)
    assert skipped == 0
    assert np.array_equal(qr[0, 0], bf16(expect))
    ec, es = oracle.quant_rows(bf16(expect)[None, :])
    assert np.array_equal(qc[0, 0], ec[0]) and qs[0, 0] == es[0]
    assert np.array_equal(c.k[0, 0, :, 0, :].reshape(D), ec[0]) and c.k_scale[0, 0, 0] == es[0]
    # V is not rotated
    vc, vs = oracle.quant_rows(kb[0])
    assert np.array_equal(c.v[0, 0, :, 0], vc[0]) and c.v_scale[0, 0, 0] == vs[0]


def test_rope_keeps_pair_norms_and_depends_on_relative_position(oracle):
    rng = np.random.default_rng(22)
    D, Hq, T = 128, 1, 12
    base = W.normal_bf16(rng, (1, Hq, D))
    q = np.repeat(base, T, axis=0)  # the same vector at positions 0, 7, 14, ...
    pos = (np.arange(T) * 7).astype(np.int32)
    cs = _rope_table(128, D)
    c = oracle.HostCache(8, 1, D)
    _, _, _, qr = oracle.rope_quant_write(c, q, q[:, :1], q[:, :1], np.zeros(T, np.int32), pos,
                                          np.arange(8, dtype=np.int32)[None, :], cs, D)
    x = W.bf16_bits_to_f32(base[0, 0]).astype(np.float64)
    rot = W.bf16_bits_to_f32(qr[:, 0]).astype(np.float64)
    h = D // 2
    # each pair keeps its length (bf16 rounding of the output: 2^-8 relative)
    n0 = x[:h] ** 2 + x[h:] ** 2
    for t in range(T):
        n1 = rot[t, :h] ** 2 + rot[t, h:] ** 2
        assert np.all(np.abs(n1 - n0) <= 2 ** -7 * n0 + 1e-6)
    # <R_m x, R_n x> depends on m - n only: positions (0, 7) vs (35, 42), (14, 28) vs (49, 63)
    scale = float(x @ x)
    for (a, b), (cc, dd) in (((0, 1), (5, 6)), ((2, 4), (7, 9)), ((1, 3), (8, 10))):
        assert abs(rot[a] @ rot[b] - rot[cc] @ rot[dd]) <= 2e-2 * scale


def test_rope_partial_rotary_and_bad_positions(oracle):
    rng = np.random.default_rng(23)
    D, Hq, T = 256, 3, 5
    q = W.normal_bf16(rng, (T, Hq, D))
    k = W.normal_bf16(rng, (T, 1, D))
    c = oracle.HostCache(1, 1, D)
    pos = np.array([0, 3, 9, 10, -1], np.int32)  # max_pos 10: the last two are out of range
    skipped, qc, qs, qr = oracle.rope_quant_write(c, q, k, k, np.zeros(T, np.int32), pos,
                                                  np.zeros((1, 1), np.int32), _rope_table(10, D // 2), D // 2)
    assert skipped == 2
    assert np.array_equal(qr[:3, :, D // 2:], q[:3, :, D // 2:])   # dims past rotary_dim untouched
    assert not qr[3:].any() and not qc[3:].any() and not qs[3:].any()
    assert np.array_equal(qr[0], q[0])                               # position 0 is the identity
