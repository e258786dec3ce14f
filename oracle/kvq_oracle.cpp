// kvq_oracle.cpp — CPU oracle for attention over an INT8-quantised paged K/V cache.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the CUDA path
// is checked against.  Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline
// / reference legs may load it.  It shares no code, header, table or constant with the
// CUDA library: it reads the same documented cache layout through its own index
// functions below.
//
// Two parts:
//   Part A  an FP64 reference attention over the dequantised cache (k^ = code * scale).
//   Part B  an exact emulation of the int8 arithmetic of the prefill path: int8 Q,
//           exact integer QK, per-tile re-quantised P, exact integer PV per tile.
// Sources (page title, section):
//   [DCU]  "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化": §1.1 byte counts,
//          §1.3 score / output composition, §2.1 quantisation rule, §2.3 layout,
//          §3.2 one online softmax over history + chunk, §3.3 fragment code.
//   [DOT4] "dot4-flash-attention" README: "Tile Inner Loop (pseudocode)" (online
//          softmax), split-K stage 1 + stage 2 (512-row splits, merge).
//   [QSA]  "#3381 ... prompt QSA attention without the decode kernel's split and merge":
//          per-query selected cell lists.
//
// Parity status per function (what pins it is in tests/test_oracle_pins.py):
//   oracle_quant_rows          pinned (hand-worked golden rows, closed-form properties)
//   oracle_kv_quant_write      pinned (layout round trip, byte counts of [DCU] §1.1)
//   oracle_rope_quant_write    pinned (identity table = plain producer; quarter and half turns
//                              exact; norm of each rotated pair; relative-position property;
//                              dims past rotary_dim untouched)
//   oracle_decode_f64          pinned (closed forms: equal scores, ctx 1, two keys)
//   oracle_decode_split_f64    pinned (equals the unsplit result for every split size)
//   oracle_prefill_ref_f64     pinned (last row equals decode; closed forms)
//   oracle_prefill_int8_emul   pinned (reduces to Part A when one tile holds every key
//                              and all weights are equal; uniform V; error bound)
//   oracle_prefill_qk_int32    pinned (brute-force integer dot products)
//   oracle_sparse_f64          pinned (full cell set equals the causal prefill reference)
//
// Build: g++ -O2 -std=c++17 -fPIC -shared -pthread -ffp-contract=off (oracle/build.py).
// No fast-math: the quantisation decisions below are IEEE fp32 and must round exactly.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

extern "C" {

typedef struct oracle_cache {
  int8_t* k;
  int8_t* v;
  float* k_scale;
  float* v_scale;
  int32_t num_blocks;
  int32_t block_size;
  int32_t n_kv_heads;
  int32_t head_dim;
} oracle_cache;

}  // extern "C"

namespace {

// ---- value helpers -----------------------------------------------------------------

float bf16_to_float(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// ---- cache layout ([DCU] §2.3, scales head-major) -------------------------------------
// K: [page][head][d/16][slot][d%16], V: [page][head][d][slot], scales: [page][head][slot].

size_t k_offset(const oracle_cache& c, int page, int head, int d, int slot) {
  size_t chunk = static_cast<size_t>(d / 16);
  size_t inner = static_cast<size_t>(d % 16);
  size_t ph = static_cast<size_t>(page) * c.n_kv_heads + head;
  return ((ph * (c.head_dim / 16) + chunk) * c.block_size + slot) * 16 + inner;
}

size_t v_offset(const oracle_cache& c, int page, int head, int d, int slot) {
  size_t ph = static_cast<size_t>(page) * c.n_kv_heads + head;
  return (ph * c.head_dim + d) * c.block_size + slot;
}

size_t scale_offset(const oracle_cache& c, int page, int head, int slot) {
  size_t ph = static_cast<size_t>(page) * c.n_kv_heads + head;
  return ph * c.block_size + slot;
}

// Physical (page, slot) of logical position `pos` through one block-table row.
struct Slot {
  int page;
  int slot;
};

Slot locate(const oracle_cache& c, const int32_t* bt_row, int pos) {
  return Slot{bt_row[pos / c.block_size], pos % c.block_size};
}

// Dequantised K and V rows of one (token, KV head) in double.
void load_kv(const oracle_cache& c, const int32_t* bt_row, int pos, int head,
             std::vector<double>& kd, std::vector<double>& vd) {
  Slot s = locate(c, bt_row, pos);
  double ks = c.k_scale[scale_offset(c, s.page, head, s.slot)];
  double vs = c.v_scale[scale_offset(c, s.page, head, s.slot)];
  for (int d = 0; d < c.head_dim; ++d) {
    kd[d] = static_cast<double>(c.k[k_offset(c, s.page, head, d, s.slot)]) * ks;
    vd[d] = static_cast<double>(c.v[v_offset(c, s.page, head, d, s.slot)]) * vs;
  }
}

// ---- B1: per-row symmetric absmax quantisation ([DCU] §2.1) -------------------------
// amax = max|x|; scale = amax / 127 (fp32); code = clamp(round(x / scale), -127, 127).
// Reading: "round" is round-to-nearest-even (the IEEE default); both divisions are IEEE
// fp32 as in the page's fragment code (§3.3 uses 127.0f); amax == 0 gives scale 0 and
// zero codes (the page asks for a safe scale or an all-zero output).
void quant_row_f32(const float* x, int n, int8_t* codes, float* scale_out) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) amax = std::max(amax, std::fabs(x[i]));
  float scale = amax / 127.0f;
  *scale_out = scale;
  for (int i = 0; i < n; ++i) {
    if (amax == 0.0f) {
      codes[i] = 0;
      continue;
    }
    float r = x[i] / scale;
    float q = std::nearbyint(r);
    q = std::fmin(std::fmax(q, -127.0f), 127.0f);
    codes[i] = static_cast<int8_t>(q);
  }
}

// B1 on a bf16 row (the values are exact in fp32).
void quant_row(const uint16_t* x, int n, int8_t* codes, float* scale_out) {
  std::vector<float> xf(n);
  for (int i = 0; i < n; ++i) xf[i] = bf16_to_float(x[i]);
  quant_row_f32(xf.data(), n, codes, scale_out);
}

// fp32 -> bf16 bits, round to nearest even (NaN stays a quiet NaN).
uint16_t float_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return static_cast<uint16_t>((u >> 16) | 0x40u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// Rotary position embedding of one row in place (fp32), the reading of [DCU] §2.2's
// "apply_rope(q, position)": the rotate-half form over the first r = rotary_dim dims, with
// cs = the table row of the position, cos of the r/2 frequencies then their sin:
//   x1 = x[i], x2 = x[i + r/2] (i < r/2):  x[i] = fma(x1, c, -(x2 * s)),
//                                          x[i + r/2] = fma(x2, c, x1 * s).
// Dims at or past r are unchanged.  This operation order is the specification.
void rope_row(float* x, const float* cs, int r) {
  const int h = r / 2;
  for (int i = 0; i < h; ++i) {
    const float c = cs[i], sn = cs[h + i];
    const float x1 = x[i], x2 = x[i + h];
    x[i] = std::fma(x1, c, -(x2 * sn));
    x[i + h] = std::fma(x2, c, x1 * sn);
  }
}

// Deterministic base-2 exponential shared, as a specification, by the oracle and the
// CUDA prefill kernel (each has its own code): the argument is clamped to [-125, 125] (with the
// fmax / fmin rule, so NaN becomes -125), then Cody-Waite range reduction x = n + f with
// n = rint(x), f in [-1/2, 1/2], 2^f by a degree-4 polynomial with constant term 1 whose other
// four coefficients minimise the largest relative error of 2^f on [-1/2, 1/2] (2.82e-6; found,
// and rounded to fp32, by oracle/fit_exp2_poly.py), in Horner form with fp32 fma, and scaling
// by 2^n.  Relative error against 2^x is below 3.6e-6 on [-125, 125] (fit error plus fp32
// rounding); integers are exact (f = 0 gives p = 1); below -125 the result is 2^-125.  It
// exists so that the P-code decisions below are the same fp32 decisions on both sides.
float exp2_det(float x) {
  x = std::fmin(std::fmax(x, -125.0f), 125.0f);
  const float magic = 12582912.0f;  // 1.5 * 2^23: x + magic rounds x to an integer
  float t = x + magic;
  float n = t - magic;
  float f = x - n;
  float p = std::fma(0.00958285294f, f, 0.0559064262f);
  p = std::fma(p, f, 0.240240991f);
  p = std::fma(p, f, 0.693124175f);
  p = std::fma(p, f, 1.0f);
  int ni = static_cast<int>(n);
  uint32_t bits = static_cast<uint32_t>(ni + 127) << 23;
  float scale2;
  std::memcpy(&scale2, &bits, sizeof scale2);
  return p * scale2;
}

// fp32 constant c2 = softmax_scale * log2(e) as both sides form it.
float score_log2_scale(float softmax_scale) { return softmax_scale * 1.44269504088896341f; }

// ---- thread helper -------------------------------------------------------------------

template <class F>
void parallel_for(int64_t n, int n_threads, F fn) {
  if (n_threads <= 0) n_threads = static_cast<int>(std::thread::hardware_concurrency());
  if (n_threads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> pool;
  int t = static_cast<int>(std::min<int64_t>(n_threads, n));
  for (int w = 0; w < t; ++w) {
    pool.emplace_back([&]() {
      for (int64_t i = next++; i < n; i = next++) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

// ---- Part A: attention of one query row over an explicit key list, FP64 ---------------
// s_t = scale * (q . k^_t);  p = softmax over the listed keys;  o = sum_t p_t v^_t.
// [DOT4] "Tile Inner Loop" computes the same quantity with an online softmax; the plain
// definition is written here.
void attend_f64(const oracle_cache& c, const int32_t* bt_row, const double* q, int head,
                const int32_t* keys, int n_keys, double scale, double* out) {
  const int D = c.head_dim;
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (n_keys <= 0) return;
  std::vector<double> kd(D), vd(D), s(n_keys);
  double m = -INFINITY;
  for (int j = 0; j < n_keys; ++j) {
    load_kv(c, bt_row, keys[j], head, kd, vd);
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q[d] * kd[d];
    s[j] = scale * dot;
    m = std::max(m, s[j]);
  }
  double l = 0.0;
  for (int j = 0; j < n_keys; ++j) {
    double p = std::exp(s[j] - m);
    l += p;
    load_kv(c, bt_row, keys[j], head, kd, vd);
    for (int d = 0; d < D; ++d) out[d] += p * vd[d];
  }
  for (int d = 0; d < D; ++d) out[d] /= l;
}

void bf16_row_to_double(const uint16_t* src, int n, double* dst) {
  for (int i = 0; i < n; ++i) dst[i] = bf16_to_float(src[i]);
}

}  // namespace

extern "C" {

// The deterministic exp2 of the prefill P-code decisions (exposed for its pins).
float oracle_exp2_det(float x) { return exp2_det(x); }

// Bytes per token and layer of the int8 cache: K and V codes plus one fp32 scale each
// per KV head ([DCU] §1.1: 2*4*256*1 + 2*4*4 = 2080 at 4 KV heads x 256).
int64_t oracle_kv_bytes_per_token(int32_t n_kv_heads, int32_t head_dim) {
  return 2LL * n_kv_heads * head_dim * 1 + 2LL * n_kv_heads * 4;
}

// Bytes per token and layer of a bf16 K/V cache ([DCU] §1.1: 2*4*256*2 = 4096).
int64_t oracle_bf16_kv_bytes_per_token(int32_t n_kv_heads, int32_t head_dim) {
  return 2LL * n_kv_heads * head_dim * 2;
}

// B1 on `rows` rows of n bf16 values each.
void oracle_quant_rows(const uint16_t* x, int64_t rows, int32_t n, int8_t* codes,
                       float* scales) {
  for (int64_t r = 0; r < rows; ++r) quant_row(x + r * n, n, codes + r * n, scales + r);
}

// Producer step ([DCU] §2.2-2.3): quantise each new (token, KV head) row of K and V and
// place codes and scale at the token's physical slot.  Out-of-range tokens are skipped.
// Returns the number of skipped tokens.
int32_t oracle_kv_quant_write(oracle_cache* cache, const uint16_t* k_new,
                              const uint16_t* v_new, int32_t n_tokens,
                              const int32_t* seq_idx, const int32_t* pos,
                              const int32_t* block_table, int32_t num_seqs,
                              int32_t max_blocks_per_seq) {
  const oracle_cache& c = *cache;
  const int H = c.n_kv_heads, D = c.head_dim;
  std::vector<int8_t> codes(D);
  int32_t skipped = 0;
  for (int i = 0; i < n_tokens; ++i) {
    int s = seq_idx[i], p = pos[i];
    if (s < 0 || s >= num_seqs || p < 0 || p / c.block_size >= max_blocks_per_seq) {
      ++skipped;
      continue;
    }
    int page = block_table[static_cast<int64_t>(s) * max_blocks_per_seq + p / c.block_size];
    if (page < 0 || page >= c.num_blocks) {
      ++skipped;
      continue;
    }
    int slot = p % c.block_size;
    for (int h = 0; h < H; ++h) {
      float sc;
      const uint16_t* krow = k_new + (static_cast<int64_t>(i) * H + h) * D;
      quant_row(krow, D, codes.data(), &sc);
      for (int d = 0; d < D; ++d) c.k[k_offset(c, page, h, d, slot)] = codes[d];
      c.k_scale[scale_offset(c, page, h, slot)] = sc;
      const uint16_t* vrow = v_new + (static_cast<int64_t>(i) * H + h) * D;
      quant_row(vrow, D, codes.data(), &sc);
      for (int d = 0; d < D; ++d) c.v[v_offset(c, page, h, d, slot)] = codes[d];
      c.v_scale[scale_offset(c, page, h, slot)] = sc;
    }
  }
  return skipped;
}

// The fused producer ([DCU] §2.2: read Q/K/V, apply RoPE to Q and K, reduce absmax, quantise,
// write the paged int8 K/V and their scales, quantise Q once): for token i at position pos[i],
// the rows of K and Q are rotated by rope_row with table row cos_sin[pos[i]], then every row
// (Q, rotated K, V) is quantised by B1 (quant_row_f32).  K/V go to the token's slot as in
// oracle_kv_quant_write; Q gives q_codes [T][Hq][D], q_scales [T][Hq] and the rotated row
// rounded to bf16 q_rot [T][Hq][D] (each output may be NULL; q may be NULL).  A token whose
// position is outside [0, max_pos) writes no K/V and zero Q outputs; an invalid sequence or
// page skips only the K/V write.  Returns the number of tokens whose K/V were not written.
int32_t oracle_rope_quant_write(oracle_cache* cache, const uint16_t* q, int32_t n_q_heads,
                                const uint16_t* k_new, const uint16_t* v_new, int32_t n_tokens,
                                const int32_t* seq_idx, const int32_t* pos, const int32_t* block_table,
                                int32_t num_seqs, int32_t max_blocks_per_seq, const float* cos_sin,
                                int32_t max_pos, int32_t rotary_dim, int8_t* q_codes, float* q_scales,
                                uint16_t* q_rot) {
  const oracle_cache& c = *cache;
  const int H = c.n_kv_heads, D = c.head_dim;
  std::vector<int8_t> codes(D);
  std::vector<float> row(D);
  int32_t skipped = 0;
  for (int i = 0; i < n_tokens; ++i) {
    const int p = pos[i];
    const bool pos_ok = p >= 0 && p < max_pos;
    const float* cs = pos_ok ? cos_sin + static_cast<int64_t>(p) * rotary_dim : nullptr;
    // Q: rotate, quantise, round the rotated row to bf16
    for (int h = 0; q && h < n_q_heads; ++h) {
      const int64_t u = static_cast<int64_t>(i) * n_q_heads + h;
      float sc = 0.0f;
      if (pos_ok) {
        for (int d = 0; d < D; ++d) row[d] = bf16_to_float(q[u * D + d]);
        rope_row(row.data(), cs, rotary_dim);
        quant_row_f32(row.data(), D, codes.data(), &sc);
      } else {
        std::fill(row.begin(), row.end(), 0.0f);
        std::fill(codes.begin(), codes.end(), 0);
      }
      if (q_codes) std::memcpy(q_codes + u * D, codes.data(), D);
      if (q_scales) q_scales[u] = sc;
      if (q_rot)
        for (int d = 0; d < D; ++d) q_rot[u * D + d] = float_to_bf16(row[d]);
    }
    const int s = seq_idx[i];
    if (!pos_ok || s < 0 || s >= num_seqs || p / c.block_size >= max_blocks_per_seq) {
      ++skipped;
      continue;
    }
    const int page = block_table[static_cast<int64_t>(s) * max_blocks_per_seq + p / c.block_size];
    if (page < 0 || page >= c.num_blocks) {
      ++skipped;
      continue;
    }
    const int slot = p % c.block_size;
    for (int h = 0; h < H; ++h) {
      float sc;
      const uint16_t* krow = k_new + (static_cast<int64_t>(i) * H + h) * D;
      for (int d = 0; d < D; ++d) row[d] = bf16_to_float(krow[d]);
      rope_row(row.data(), cs, rotary_dim);
      quant_row_f32(row.data(), D, codes.data(), &sc);
      for (int d = 0; d < D; ++d) c.k[k_offset(c, page, h, d, slot)] = codes[d];
      c.k_scale[scale_offset(c, page, h, slot)] = sc;
      const uint16_t* vrow = v_new + (static_cast<int64_t>(i) * H + h) * D;
      quant_row(vrow, D, codes.data(), &sc);
      for (int d = 0; d < D; ++d) c.v[v_offset(c, page, h, d, slot)] = codes[d];
      c.v_scale[scale_offset(c, page, h, slot)] = sc;
    }
  }
  return skipped;
}


// Every attention function below works on "units" (row, query head): unit u stands for
// row u / n_q_heads and query head u % n_q_heads, where a row is a sequence (decode), a
// chunk token (prefill) or a query (sparse).  With units == NULL all rows * n_q_heads
// units are computed and out is [rows][n_q_heads][D]; otherwise out is [n_units][D] in
// the order of `units` (sampled checks of full-size workloads).

static int64_t unit_at(const int64_t* units, int64_t j) { return units ? units[j] : j; }

// Part A, decode: one query per sequence over keys [0, ctx_lens[b]).
void oracle_decode_f64(const oracle_cache* cache, const uint16_t* q, int32_t batch,
                       int32_t n_q_heads, const int32_t* block_table,
                       int32_t max_blocks_per_seq, const int32_t* ctx_lens, double scale,
                       const int64_t* units, int32_t n_units, double* out,
                       int32_t n_threads) {
  const oracle_cache& c = *cache;
  const int D = c.head_dim, G = n_q_heads / c.n_kv_heads;
  int64_t n = units ? n_units : static_cast<int64_t>(batch) * n_q_heads;
  parallel_for(n, n_threads, [&](int64_t j) {
    int64_t u = unit_at(units, j);
    int b = static_cast<int>(u / n_q_heads), h = static_cast<int>(u % n_q_heads);
    std::vector<double> qd(D);
    bf16_row_to_double(q + u * D, D, qd.data());
    std::vector<int32_t> keys(ctx_lens[b]);
    for (int t = 0; t < ctx_lens[b]; ++t) keys[t] = t;
    attend_f64(c, block_table + static_cast<int64_t>(b) * max_blocks_per_seq, qd.data(),
               h / G, keys.data(), ctx_lens[b], scale, out + j * D);
  });
}

// Part A, verify decode (the multi-row decode of [DOT4] "Future Work", MTP verify with nq
// query rows per sequence; "ROCm/RDNA4 (gfx1201) vLLM ..." row-shape routing, spec-verify
// with 2-6 rows): sequence b holds ctx_lens[b] keys, the last nq of them the tokens being
// verified; query row i of b sits at position ctx - nq + i and sees keys
// t < ctx - nq + 1 + i (causal among the nq tokens; none when that bound is <= 0).
// q and out are [batch][nq][n_q_heads][D]; unit u = (b * nq + i) * n_q_heads + h.
void oracle_verify_f64(const oracle_cache* cache, const uint16_t* q, int32_t batch,
                       int32_t nq, int32_t n_q_heads, const int32_t* block_table,
                       int32_t max_blocks_per_seq, const int32_t* ctx_lens, double scale,
                       const int64_t* units, int32_t n_units, double* out,
                       int32_t n_threads) {
  const oracle_cache& c = *cache;
  const int D = c.head_dim, G = n_q_heads / c.n_kv_heads;
  int64_t n = units ? n_units : static_cast<int64_t>(batch) * nq * n_q_heads;
  parallel_for(n, n_threads, [&](int64_t j) {
    int64_t u = unit_at(units, j);
    int h = static_cast<int>(u % n_q_heads);
    int64_t row = u / n_q_heads;
    int i = static_cast<int>(row % nq), b = static_cast<int>(row / nq);
    std::vector<double> qd(D);
    bf16_row_to_double(q + u * D, D, qd.data());
    int nk = std::min(ctx_lens[b], ctx_lens[b] - nq + 1 + i);
    if (nk < 0) nk = 0;
    std::vector<int32_t> keys(nk);
    for (int t = 0; t < nk; ++t) keys[t] = t;
    attend_f64(c, block_table + static_cast<int64_t>(b) * max_blocks_per_seq, qd.data(),
               h / G, keys.data(), nk, scale, out + j * D);
  });
}

// B5, decode through split-K ([DOT4] stage 1 + stage 2): each split of `split_rows` keys
// yields (m_s, l_s, acc_s) with acc_s = sum_t e^{s_t - m_s} v^_t; the merge takes
// M = max m_s, l = sum l_s e^{m_s - M}, o = sum acc_s e^{m_s - M} / l.
void oracle_decode_split_f64(const oracle_cache* cache, const uint16_t* q, int32_t batch,
                             int32_t n_q_heads, const int32_t* block_table,
                             int32_t max_blocks_per_seq, const int32_t* ctx_lens,
                             double scale, int32_t split_rows, double* out,
                             int32_t n_threads) {
  const oracle_cache& c = *cache;
  const int D = c.head_dim, G = n_q_heads / c.n_kv_heads;
  parallel_for(static_cast<int64_t>(batch) * n_q_heads, n_threads, [&](int64_t u) {
    int b = static_cast<int>(u / n_q_heads), h = static_cast<int>(u % n_q_heads);
    const int32_t* bt = block_table + static_cast<int64_t>(b) * max_blocks_per_seq;
    int ctx = ctx_lens[b];
    std::vector<double> qd(D), kd(D), vd(D);
    bf16_row_to_double(q + u * D, D, qd.data());
    std::vector<double> ms, ls;
    std::vector<std::vector<double>> accs;
    for (int t0 = 0; t0 < ctx; t0 += split_rows) {
      int t1 = std::min(ctx, t0 + split_rows);
      std::vector<double> s(t1 - t0);
      double m = -INFINITY;
      for (int t = t0; t < t1; ++t) {
        load_kv(c, bt, t, h / G, kd, vd);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * kd[d];
        s[t - t0] = scale * dot;
        m = std::max(m, s[t - t0]);
      }
      double l = 0.0;
      std::vector<double> acc(D, 0.0);
      for (int t = t0; t < t1; ++t) {
        double p = std::exp(s[t - t0] - m);
        l += p;
        load_kv(c, bt, t, h / G, kd, vd);
        for (int d = 0; d < D; ++d) acc[d] += p * vd[d];
      }
      ms.push_back(m);
      ls.push_back(l);
      accs.push_back(acc);
    }
    double* o = out + u * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (ms.empty()) return;
    double M = *std::max_element(ms.begin(), ms.end());
    double l = 0.0;
    for (size_t i = 0; i < ms.size(); ++i) {
      double w = std::exp(ms[i] - M);
      l += ls[i] * w;
      for (int d = 0; d < D; ++d) o[d] += accs[i][d] * w;
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
  });
}

// The first prefill chunk ([DCU] §3.1: no history to read; the chunk runs the high-precision
// attention while the producer writes its K/V as int8): causal attention of the chunk over its
// own bf16 K/V, before any quantisation.  Query i sees keys t <= i.  q [T][Hq][D], k and v
// [T][Hkv][D] (bf16 bits); unit u = i * Hq + h.
void oracle_prefill_first_f64(const uint16_t* q, const uint16_t* k, const uint16_t* v, int32_t n_tokens,
                              int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, double scale,
                              const int64_t* units, int32_t n_units, double* out, int32_t n_threads) {
  const int D = head_dim, Hq = n_q_heads, Hkv = n_kv_heads, G = Hq / Hkv;
  int64_t n = units ? n_units : static_cast<int64_t>(n_tokens) * Hq;
  parallel_for(n, n_threads, [&](int64_t j) {
    int64_t u = unit_at(units, j);
    const int i = static_cast<int>(u / Hq), h = static_cast<int>(u % Hq), kvh = h / G;
    std::vector<double> qd(D), s(i + 1);
    bf16_row_to_double(q + u * D, D, qd.data());
    double m = -INFINITY;
    for (int t = 0; t <= i; ++t) {
      const uint16_t* kr = k + (static_cast<int64_t>(t) * Hkv + kvh) * D;
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qd[d] * bf16_to_float(kr[d]);
      s[t] = scale * dot;
      m = std::max(m, s[t]);
    }
    double l = 0.0;
    double* o = out + j * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int t = 0; t <= i; ++t) {
      const double p = std::exp(s[t] - m);
      l += p;
      const uint16_t* vr = v + (static_cast<int64_t>(t) * Hkv + kvh) * D;
      for (int d = 0; d < D; ++d) o[d] += p * bf16_to_float(vr[d]);
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
  });
}

// Part A, prefill chunk ([DCU] §3.2): query i at position history + i sees keys
// t <= history + i, history and chunk alike.
void oracle_prefill_ref_f64(const oracle_cache* cache, const uint16_t* q, int32_t n_tokens,
                            int32_t n_q_heads, int32_t history, const int32_t* bt_row,
                            double scale, const int64_t* units, int32_t n_units, double* out,
                            int32_t n_threads) {
  const oracle_cache& c = *cache;
  const int D = c.head_dim, G = n_q_heads / c.n_kv_heads;
  int64_t n = units ? n_units : static_cast<int64_t>(n_tokens) * n_q_heads;
  parallel_for(n, n_threads, [&](int64_t j) {
    int64_t u = unit_at(units, j);
    int i = static_cast<int>(u / n_q_heads), h = static_cast<int>(u % n_q_heads);
    std::vector<double> qd(D);
    bf16_row_to_double(q + u * D, D, qd.data());
    int nk = history + i + 1;
    std::vector<int32_t> keys(nk);
    for (int t = 0; t < nk; ++t) keys[t] = t;
    attend_f64(c, bt_row, qd.data(), h / G, keys.data(), nk, scale, out + j * D);
  });
}

// The method's prefill with exact softmax arithmetic ([DCU] §1.3, §3.3; §2.1 for Q): Q is
// quantised per (token, query head) by B1 and enters as its dequantised value
// q^ = q_code * sQ; the attention is then the plain definition in double,
//   s_t = scale * (q^ . k^_t),  p_t = exp(s_t - max s),  l = sum_t p_t,
//   out[d] = sum_t p_t v^_t[d] / l,
// with no P quantisation.  Beside it, per output element, the largest change that the
// per-tile P re-quantisation of the method can make to it:
//   w_t = p_t * sV_t;  per tile of pv_tile keys at absolute multiples of pv_tile,
//   ps_j = max_{t in tile} w_t / 127;  the code of w_t is rint(w_t / ps_j), so ps_j * code
//   differs from w_t by at most ps_j / 2, and by exactly w_t when w_t < ps_j / 2 (code 0);
//   the numerator multiplies that difference by the integer v8_t[d]:
//   bound[d] = sum_t min(w_t, ps_{j(t)} / 2) * |v8_t[d]| / l,
// and mag[d] = sum_t p_t |v^_t[d]| / l, the scale of the output's own rounding errors (an
// implementation whose weights carry a relative error e moves the output by at most about
// e * mag[d]).  bound and mag may be null.
void oracle_prefill_qdeq_f64(const oracle_cache* cache, const uint16_t* q, int32_t n_tokens, int32_t n_q_heads,
                             int32_t history, const int32_t* bt_row, double scale, int32_t pv_tile,
                             const int64_t* units, int32_t n_units, double* out, double* bound, double* mag,
                             int32_t n_threads) {
  const oracle_cache& c = *cache;
  const int D = c.head_dim, G = n_q_heads / c.n_kv_heads;
  int64_t n = units ? n_units : static_cast<int64_t>(n_tokens) * n_q_heads;
  parallel_for(n, n_threads, [&](int64_t j) {
    int64_t u = unit_at(units, j);
    int i = static_cast<int>(u / n_q_heads), h = static_cast<int>(u % n_q_heads);
    int kvh = h / G;
    std::vector<int8_t> q8(D);
    float sq;
    quant_row(q + u * D, D, q8.data(), &sq);
    std::vector<double> qd(D);
    for (int d = 0; d < D; ++d) qd[d] = static_cast<double>(q8[d]) * static_cast<double>(sq);
    const int nk = history + i + 1;
    std::vector<double> s(nk), kd(D), vd(D);
    double m = -INFINITY;
    for (int t = 0; t < nk; ++t) {
      load_kv(c, bt_row, t, kvh, kd, vd);
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qd[d] * kd[d];
      s[t] = scale * dot;
      m = std::max(m, s[t]);
    }
    double l = 0.0;
    std::vector<double> o(D, 0.0), b(D, 0.0), a(D, 0.0), p(pv_tile), w(pv_tile);
    for (int t0 = 0; t0 < nk; t0 += pv_tile) {
      const int t1 = std::min(nk, t0 + pv_tile);
      double wmax = 0.0;
      for (int t = t0; t < t1; ++t) {
        Slot sl = locate(c, bt_row, t);
        p[t - t0] = std::exp(s[t] - m);
        w[t - t0] = p[t - t0] * c.v_scale[scale_offset(c, sl.page, kvh, sl.slot)];
        wmax = std::max(wmax, w[t - t0]);
      }
      const double half_ps = (wmax / 127.0) / 2.0;
      for (int t = t0; t < t1; ++t) {
        Slot sl = locate(c, bt_row, t);
        const double sv = c.v_scale[scale_offset(c, sl.page, kvh, sl.slot)];
        const double e = std::min(w[t - t0], half_ps);
        l += p[t - t0];
        for (int d = 0; d < D; ++d) {
          const double v8 = c.v[v_offset(c, sl.page, kvh, d, sl.slot)];
          o[d] += p[t - t0] * (v8 * sv);
          a[d] += p[t - t0] * std::fabs(v8 * sv);
          b[d] += e * std::fabs(v8);
        }
      }
    }
    for (int d = 0; d < D; ++d) {
      out[j * D + d] = o[d] / l;
      if (bound) bound[j * D + d] = b[d] / l;
      if (mag) mag[j * D + d] = a[d] / l;
    }
  });
}

// B2: exact integer QK for one window, no mask: s_out[r][j] = sum_d q8[q0+r][h][d] *
// k8[k0+j][h/G][d] for r < nq, j < nk; rows at or past n_tokens give 0.
void oracle_prefill_qk_int32(const int8_t* q_codes, int32_t n_tokens, int32_t n_q_heads,
                             const oracle_cache* cache, const int32_t* bt_row,
                             int32_t q_head, int32_t q0, int32_t nq, int32_t k0, int32_t nk,
                             int32_t* s_out) {
  const oracle_cache& c = *cache;
  const int D = c.head_dim, G = n_q_heads / c.n_kv_heads, kvh = q_head / G;
  for (int r = 0; r < nq; ++r) {
    int i = q0 + r;
    for (int j = 0; j < nk; ++j) {
      int64_t acc = 0;
      if (i < n_tokens) {
        Slot s = locate(c, bt_row, k0 + j);
        const int8_t* qr = q_codes + (static_cast<int64_t>(i) * n_q_heads + q_head) * D;
        for (int d = 0; d < D; ++d)
          acc += static_cast<int64_t>(qr[d]) * c.k[k_offset(c, s.page, kvh, d, s.slot)];
      }
      s_out[static_cast<int64_t>(r) * nk + j] = static_cast<int32_t>(acc);
    }
  }
}

// Part B, prefill chunk with the int8 arithmetic of [DCU] §1.3 / §3.3, the page's
// fragment code taken step by step in fp32:
//   Q codes by B1 per (token, query head);  S_t = sum_d q8 k8 (exact integer);
//   a = sQ * c2 (c2 = softmax_scale * log2 e);  y_t = S_t * sK_t  (log2-domain score a*y_t);
//   tiles of `pv_tile` keys at absolute multiples of pv_tile, over the visible keys of the
//   tile:
//     t_j = (max_t y_t) * a                               the tile's own maximum
//     p_t = exp2_det(fma(y_t, a, -t_j))                   p relative to t_j
//     w_t = p_t * sV_t                                   sV folded into the weight
//     r_j = 127 / max_t w_t;  c_t = rint(w_t * r_j) in [0, 127] (one rounding, fma)
//     numerator_j = ps_j * sum_t c_t v8_t with ps_j = max_t w_t / 127, sum exact
//   out = sum_j numerator_j 2^{t_j - M} / sum_j (sum_t p_t) 2^{t_j - M}, M the row maximum,
//   this final combination in double (accumulated with an online maximum, exact in double).
//   l sums the unquantised p.
// Readings (the page is silent): one P scale per (query row, tile); tiles aligned at
// absolute key positions; l from the unquantised weights; exp by exp2_det so that both
// sides decide each code with the same fp32 operations.  The page takes p relative to the
// online running maximum; the maximum cancels in w / max w, so the codes are the same in
// exact arithmetic, and taking the fp32 decision relative to the tile's own maximum makes
// each tile's codes a function of that tile alone (independent of the order in which the
// tiles are visited, or of how the key range is divided between workers).  q_codes_out ([n_tokens][n_q_heads][D]) and q_scales_out
// ([n_tokens][n_q_heads]) may be null; they are written for every token and head.
void oracle_prefill_int8_emul(const oracle_cache* cache, const uint16_t* q, int32_t n_tokens,
                              int32_t n_q_heads, int32_t history, const int32_t* bt_row,
                              float softmax_scale, int32_t pv_tile, const int64_t* units,
                              int32_t n_units, double* out, int8_t* q_codes_out,
                              float* q_scales_out, int32_t n_threads) {
  const oracle_cache& c = *cache;
  const int D = c.head_dim, G = n_q_heads / c.n_kv_heads;
  const float c2 = score_log2_scale(softmax_scale);
  if (q_codes_out || q_scales_out) {
    std::vector<int8_t> q8(D);
    for (int64_t u = 0; u < static_cast<int64_t>(n_tokens) * n_q_heads; ++u) {
      float sq;
      quant_row(q + u * D, D, q8.data(), &sq);
      if (q_codes_out) std::memcpy(q_codes_out + u * D, q8.data(), D);
      if (q_scales_out) q_scales_out[u] = sq;
    }
  }
  int64_t n = units ? n_units : static_cast<int64_t>(n_tokens) * n_q_heads;
  parallel_for(n, n_threads, [&](int64_t j) {
    int64_t u = unit_at(units, j);
    int i = static_cast<int>(u / n_q_heads), h = static_cast<int>(u % n_q_heads);
    int kvh = h / G;
    std::vector<int8_t> q8(D);
    float sq;
    quant_row(q + u * D, D, q8.data(), &sq);
    const float a = sq * c2;
    int nk = history + i + 1;
    std::vector<float> y(pv_tile), w(pv_tile), p(pv_tile);
    std::vector<int64_t> tile_sum(D);
    std::vector<double> num(D, 0.0);
    double l = 0.0;
    float m = -INFINITY;
    for (int t0 = 0; t0 < nk; t0 += pv_tile) {
      int t1 = std::min(nk, t0 + pv_tile);
      float ymax = -INFINITY;
      for (int t = t0; t < t1; ++t) {
        Slot s = locate(c, bt_row, t);
        int64_t acc = 0;
        for (int d = 0; d < D; ++d)
          acc += static_cast<int64_t>(q8[d]) * c.k[k_offset(c, s.page, kvh, d, s.slot)];
        y[t - t0] = static_cast<float>(acc) * c.k_scale[scale_offset(c, s.page, kvh, s.slot)];
        ymax = std::max(ymax, y[t - t0]);
      }
      // The tile's codes c = rint(127 w / max w) do not depend on the maximum that p is taken
      // relative to (it cancels in w / max w); the fp32 decisions are taken relative to the
      // tile's own maximum t = max(y) * a, so each tile's codes follow from the tile alone.
      // beta = 2^(t - m) then moves the tile's P scale and its sum of p onto the running
      // maximum m (in double).
      const float m_tile = ymax * a;
      float m_new = std::max(m, m_tile);
      // rescale what was accumulated relative to the previous maximum (exact in double)
      double alpha = (m == -INFINITY) ? 0.0 : std::exp2(static_cast<double>(m) - m_new);
      const double beta = std::exp2(static_cast<double>(m_tile) - m_new);
      l *= alpha;
      for (int d = 0; d < D; ++d) num[d] *= alpha;
      m = m_new;
      float wmax = 0.0f;
      double psum = 0.0;
      for (int t = t0; t < t1; ++t) {
        Slot s = locate(c, bt_row, t);
        p[t - t0] = exp2_det(std::fma(y[t - t0], a, -m_tile));
        psum += p[t - t0];
        w[t - t0] = p[t - t0] * c.v_scale[scale_offset(c, s.page, kvh, s.slot)];
        wmax = std::max(wmax, w[t - t0]);
      }
      l += psum * beta;
      if (!(wmax > 0.0f)) continue;  // every weight of the tile is zero: codes all zero
      const float r = 127.0f / wmax;
      std::fill(tile_sum.begin(), tile_sum.end(), 0);
      for (int t = t0; t < t1; ++t) {
        const float magic = 12582912.0f;
        float code = std::fma(w[t - t0], r, magic) - magic;
        code = std::fmin(std::fmax(code, 0.0f), 127.0f);
        int64_t ci = static_cast<int64_t>(code);
        if (ci == 0) continue;
        Slot s = locate(c, bt_row, t);
        for (int d = 0; d < D; ++d) tile_sum[d] += ci * c.v[v_offset(c, s.page, kvh, d, s.slot)];
      }
      double ps = static_cast<double>(wmax) / 127.0 * beta;
      for (int d = 0; d < D; ++d) num[d] += ps * static_cast<double>(tile_sum[d]);
    }
    double* o = out + j * D;
    for (int d = 0; d < D; ++d) o[d] = num[d] / l;
  });
}

// Part A, sparse prompt attention ([QSA]): query i attends to
// cells[offsets[i] .. offsets[i+1]) (logical positions through bt_row).
void oracle_sparse_f64(const oracle_cache* cache, const uint16_t* q, int32_t n_queries,
                       int32_t n_q_heads, const int32_t* offsets, const int32_t* cells,
                       const int32_t* bt_row, double scale, const int64_t* units,
                       int32_t n_units, double* out, int32_t n_threads) {
  const oracle_cache& c = *cache;
  const int D = c.head_dim, G = n_q_heads / c.n_kv_heads;
  int64_t n = units ? n_units : static_cast<int64_t>(n_queries) * n_q_heads;
  parallel_for(n, n_threads, [&](int64_t j) {
    int64_t u = unit_at(units, j);
    int i = static_cast<int>(u / n_q_heads), h = static_cast<int>(u % n_q_heads);
    std::vector<double> qd(D);
    bf16_row_to_double(q + u * D, D, qd.data());
    attend_f64(c, bt_row, qd.data(), h / G, cells + offsets[i], offsets[i + 1] - offsets[i],
               scale, out + j * D);
  });
}

}  // extern "C"
