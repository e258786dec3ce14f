// sparse.cu — sparse prompt attention over the int8 paged K/V cache.
//
// Method: "#3381 [Engine] STRATA_PROMPT_ATTN_RDNA2=1 ... prompt QSA attention without the
// decode kernel's split and merge", sections "Problem and result" and "Approach": one block
// per (query, KV head) walks all of the query's selected cells with an online softmax, with
// no per-chunk scratch and no merge pass over HBM; the GQA group shares each gathered K/V row.
//
// GB300 design.
// * Gather records (pre-pass).  The cache keeps V dimension-major inside a page ([DCU] §2.3:
//   [page][head][dim][slot], chosen for dense PV), so one cell's V row is 256 single bytes at a
//   16-byte stride: every cell would pull its page's whole 4 KB V block through L2.  A pre-pass
//   rewrites the sequence's pages once into token-major records, one per (logical page, KV
//   head, slot): [K codes D][V codes D][k_scale][v_scale][valid][pad], 2D + 16 bytes.  Each
//   selected cell is then one contiguous bulk copy, and the record stride (33 or 17 units of
//   16 bytes) keeps the ldmatrix rows of 8 cells in 8 distinct bank groups.
// * Attention (sparse_chunk_kernel, below): one CTA of four warps per (query, KV head) walks the
//   cells in 64-cell chunks with the page's blocked fold: the chunk's scores give the chunk
//   maximum, the chunk's sums start from zero relative to the updated maximum, and they are folded
//   into the running sums with one fma each.  QK and PV run on mma.sync with the int8 codes widened
//   exactly to fp16 (each code once per query), the weights as fp16 hi + lo parts.
#include "kvq_dev.cuh"
#include "kvq_launch.h"

namespace kvq {

namespace {

constexpr float kLog2eS = 1.4426950408889634f;

template <int D>
struct SparseRec {
  static constexpr int kBytes = 2 * D + 16;  // K | V | k_scale | v_scale | valid | pad
  static constexpr int kV = D;
  static constexpr int kScales = 2 * D;
};

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// byte selectors: bytes (0, 2) and (1, 3) of a word into the low bytes of two halves
constexpr uint32_t kSelB02 = 0x4240u;
constexpr uint32_t kSelB13 = 0x4341u;

}  // namespace

// Pre-pass: the gather records of logical page blockIdx.x, KV head blockIdx.y.
template <int D>
__global__ void __launch_bounds__(256) sparse_prep_kernel(SparseArgs a) {
  using R = SparseRec<D>;
  __shared__ __align__(16) uint8_t vt[D * KVQ_BLOCK_SIZE];  // the page's V block, [dim][slot]
  const int lp = blockIdx.x, kvh = blockIdx.y, t = threadIdx.x;
  uint8_t* out = a.records + ((static_cast<long long>(lp) * a.n_kv_heads + kvh) * KVQ_BLOCK_SIZE) * R::kBytes;
  const int page = a.block_table_row[lp];
  const bool valid = page >= 0 && page < a.num_blocks;
  if (!valid) {
    if (t < KVQ_BLOCK_SIZE)
      *reinterpret_cast<int4*>(out + t * R::kBytes + R::kScales) = make_int4(0, 0, 0, 0);
    return;
  }
  const long long ph = static_cast<long long>(page) * a.n_kv_heads + kvh;
  if (t < D) {
    // K: the 16-byte piece (chunk j, slot s) of [page][head][D/16][16][16] to record s at 16 j
    const int j = t / KVQ_BLOCK_SIZE, s = t % KVQ_BLOCK_SIZE;
    const int4 kp = __ldg(reinterpret_cast<const int4*>(a.k + (ph * (D / 16) + j) * 256 + s * 16));
    *reinterpret_cast<int4*>(out + s * R::kBytes + j * 16) = kp;
    // V: dimension row t (16 slots) into shared memory
    *reinterpret_cast<int4*>(vt + t * 16) = __ldg(reinterpret_cast<const int4*>(a.v + (ph * D + t) * KVQ_BLOCK_SIZE));
  }
  if (t < KVQ_BLOCK_SIZE) {
    const float ks = a.k_scale[ph * KVQ_BLOCK_SIZE + t], vs = a.v_scale[ph * KVQ_BLOCK_SIZE + t];
    *reinterpret_cast<int4*>(out + t * R::kBytes + R::kScales) =
        make_int4(__float_as_int(ks), __float_as_int(vs), 1, 0);
  }
  __syncthreads();
  if (t < D) {
    // V of slot s, dims 16 db .. 16 db + 15, gathered from the [dim][slot] block; consecutive
    // threads take consecutive slots, so a warp's byte reads of one dim share a word (the other
    // order put the 16 dims' reads of a warp in one bank)
    const int s = t % KVQ_BLOCK_SIZE, db = t / KVQ_BLOCK_SIZE;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      w[q] = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) w[q] |= static_cast<uint32_t>(vt[(db * 16 + q * 4 + e) * 16 + s]) << (8 * e);
    }
    *reinterpret_cast<int4*>(out + s * R::kBytes + R::kV + db * 16) =
        make_int4(static_cast<int>(w[0]), static_cast<int>(w[1]), static_cast<int>(w[2]), static_cast<int>(w[3]));
  }
}

// ============================================================================ chunked attention
// [QSA] "Approach": the query's cells are walked in 64-cell chunks; each chunk's scores give the
// chunk maximum, the running maximum moves to max(m, chunk max), the chunk's weights are summed
// from zero relative to it (l_c, acc_c), and the chunk is folded into the running sums with one
// fma each: l = fma(l, alpha, l_c), acc = fma(acc, alpha, acc_c), alpha = 2^(m_old - m_new).
// One CTA of four warps per (query, KV head); chunk c sits in buffer c % NBUF.
// * QK: warp w scores the chunk's cells 16 w .. 16 w + 15 against every head of the group (cells
//   on M, heads on N of mma.sync m16n8k16, the int8 K codes widened once and used for each 8-head
//   n-tile).  The four warps then agree on each head's chunk maximum through shared memory.
// * Weights: warp w turns its cells' scores into W = 2^(z - m_z) (z = s + log2 sV: the second
//   running maximum keeps W in [0, 1] whatever the V scales are) and l_c's part, and leaves W as
//   fp16 hi + lo PV B-fragments in shared memory.
// * PV: warp w multiplies all 64 weights into head dims w D/4 .. (w + 1) D/4 - 1 (dims on M via the
//   ldmatrix.trans V^T fragments of the token-major records, the V codes widened once), from a
//   zero chunk accumulator, and folds it into its running O^T.
// Every K and V code is therefore widened once per query, and the four warps' accumulators are
// disjoint: the CTA needs no merge at the end.
template <int D, int NHT, int NBUF>
struct ChunkSmem {
  static constexpr int kCells = 64;
  static constexpr int kBufBytes = kCells * SparseRec<D>::kBytes;
  static constexpr int kQOffset = NBUF * kBufBytes;         // Q^T fragments, NHT n-tiles
  static constexpr int kWOffset = kQOffset + NHT * D * 16;  // W fragments [tile][n-tile][32 lanes] x 4 words
  static constexpr int kRedOffset = kWOffset + 4 * NHT * 4 * 32 * 4;  // [3][NHT * 8 heads][warp] floats
  static constexpr int kCqOffset = kRedOffset + 3 * 4 * NHT * 8 * 4;
  static constexpr int kMaskOffset = kCqOffset + NHT * 8 * 4;         // [NBUF][warp] copied-cell masks
  static constexpr int kBarOffset = (kMaskOffset + NBUF * 4 * 4 + 7) / 8 * 8;  // full [NBUF], empty [NBUF]
  static constexpr int kTotal = kBarOffset + 2 * NBUF * 8;
  static_assert(kQOffset % 16 == 0 && kWOffset % 16 == 0 && kRedOffset % 16 == 0, "ldmatrix / vector alignment");
  static_assert(kTotal <= 227 * 1024, "shared memory of one CTA");
};

// bar.sync on barrier 1 of the CTA's 128 threads, returning the OR of pred over them
__device__ __forceinline__ bool chunk_bar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, 128, q;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void chunk_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// FI: the test-only fault injection and wait budget of kvq_debug_fault_inject are compiled in
// (a separate instantiation, so that the production kernel keeps its registers).
template <int D, int NHT, int NBUF, bool FI>
__global__ void __launch_bounds__(128, NBUF == 1 ? 4 : 2) sparse_chunk_kernel(SparseArgs a) {
  using L = ChunkSmem<D, NHT, NBUF>;
  using R = SparseRec<D>;
  constexpr int RB = R::kBytes;
  constexpr int NH = NHT * 8;     // heads of the group, padded to whole n-tiles
  constexpr int NDB = D / 128;    // 32-dim blocks of a warp's quarter of the head dimension
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  uint8_t* q_s = smem + L::kQOffset;
  uint4* wx = reinterpret_cast<uint4*>(smem + L::kWOffset);
  float* red = reinterpret_cast<float*>(smem + L::kRedOffset);
  float* cq_s = reinterpret_cast<float*>(smem + L::kCqOffset);
  uint32_t* cmask = reinterpret_cast<uint32_t*>(smem + L::kMaskOffset);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  uint64_t* empty = full + NBUF;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x, kvh = blockIdx.y;
  const int Hq = a.n_q_heads, G = Hq / a.n_kv_heads;

  grid_dep_wait();  // the records come from the pre-pass
  const int c_begin = a.cell_offsets[i], c_end = a.cell_offsets[i + 1];
  const int n_cells = max(0, c_end - c_begin);
  const int n_chunks = (n_cells + L::kCells - 1) / L::kCells;
  float* out_q = a.out + (static_cast<long long>(i) * Hq + kvh * G) * D;
  if (n_chunks == 0) {
    for (int e = threadIdx.x; e < G * D; e += blockDim.x) out_q[e] = 0.0f;
    return;
  }
  if (threadIdx.x == 0) {
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&full[b], 4);
      mbar_init(&empty[b], 4);
    }
    mbar_fence_init();
  }
  __syncthreads();

  // Warp w copies cells 16 w + l (lane l < 16) of each chunk.  Their positions are loaded NBUF
  // chunks ahead of the copies (pos_q[c % NBUF] holds chunk c's), so no copy waits on an index load.
  auto load_pos = [&](int c) {
    const int cell = c_begin + c * L::kCells + warp * 16 + lane;
    return (c < n_chunks && lane < 16 && cell < c_end) ? __ldg(a.cells + cell) : -1;
  };
  int pos_q[NBUF];
#pragma unroll
  for (int b = 0; b < NBUF; ++b) pos_q[b] = load_pos(b);
  int n_issued = 0;
  // test-only fault injection: the first CTA leaves chunk 1 un-issued (no copy and no arrival: the
  // chunk's barrier never completes and nothing is in flight for it), so the bounded waits run out
  const bool skip_one = FI && a.fault == 3 && blockIdx.x == 0 && blockIdx.y == 0;
  const long long budget = FI ? a.wait_budget : kWaitBudgetCycles;
  auto issue = [&](int c) {
    const int b = c % NBUF;
    int pos = -1;
#pragma unroll
    for (int d = 0; d < NBUF; ++d)
      if (d == b) {
        pos = pos_q[d];
        pos_q[d] = load_pos(c + NBUF);
      }
    const int cell = c_begin + c * L::kCells + warp * 16 + lane;
    bool ok = false;
    long long rec = 0;
    if (lane < 16 && cell < c_end) {
      if (pos >= 0 && pos / KVQ_BLOCK_SIZE < a.n_blocks_row) {
        ok = true;
        rec = ((static_cast<long long>(pos / KVQ_BLOCK_SIZE) * a.n_kv_heads + kvh) * KVQ_BLOCK_SIZE +
               pos % KVQ_BLOCK_SIZE) * RB;
      } else {
        set_status(a.status, KVQ_DEV_BAD_CELL);
      }
    }
    const uint32_t m = __ballot_sync(0xffffffffu, ok);
    if (skip_one && c == 1) {
      ++n_issued;
      return;
    }
    if (lane == 0) {
      cmask[b * 4 + warp] = m;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&full[b], __popc(m) * RB);
    }
    __syncwarp();
    if (ok) bulk_g2s(ring + b * L::kBufBytes + (warp * 16 + lane) * RB, a.records + rec, RB, &full[b]);
    ++n_issued;
  };
  for (int c = 0; c < min(NBUF, n_chunks); ++c) issue(c);

  // ---- Q^T fragments (as decode): row r = head r of the group, fp16 q * 2^e per head
  for (int h = warp; h < NH; h += 4) {
    const bool real = h < G;
    uint8_t* q_tile = q_s + (h >> 3) * (D * 16);
    const int hr = h & 7;
    constexpr int PER = D / 32;
    float x[PER];
    const uint16_t* qrow = static_cast<const uint16_t*>(a.q) + (static_cast<long long>(i) * Hq + kvh * G + (real ? h : 0)) * D + lane * PER;
    if constexpr (PER == 8) {
      const uint4 raw = real ? __ldg(reinterpret_cast<const uint4*>(qrow)) : make_uint4(0, 0, 0, 0);
      const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w4[e] << 16);
        x[2 * e + 1] = __uint_as_float(w4[e] & 0xFFFF0000u);
      }
    } else {
      const uint2 raw = real ? __ldg(reinterpret_cast<const uint2*>(qrow)) : make_uint2(0, 0);
      const uint32_t w2[2] = {raw.x, raw.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        x[2 * e] = __uint_as_float(w2[e] << 16);
        x[2 * e + 1] = __uint_as_float(w2[e] & 0xFFFF0000u);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    int ex = amax > 0.f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127 : 0;
    ex = max(-100, min(ex, 127));
    const float qs = __uint_as_float(static_cast<uint32_t>(127 + 14 - ex) << 23);
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int d = lane * PER + e;
      const int j = d >> 4, w = d & 15, cc = w >> 2, bb = w & 3;
      const int half = bb >> 1, el = 2 * cc + (bb & 1);
      *reinterpret_cast<__half*>(q_tile + ((j * 2 + half) * 8 + hr) * 16 + el * 2) = __float2half_rn(x[e] * qs);
    }
    if (lane == 0) cq_s[h] = a.softmax_scale * kLog2eS / qs;
  }
  __syncthreads();

  const int g = lane >> 2, c4 = lane & 3;
  // running statistics of this thread's heads nt * 8 + 2 c4 + e (the same in all four warps)
  float ms[NHT][2], mz[NHT][2], lsum[NHT][2], cq[NHT][2];
  float o_acc[2 * NDB][NHT][4];
#pragma unroll
  for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      ms[nt][e] = -INFINITY;
      mz[nt][e] = -INFINITY;
      lsum[nt][e] = 0.f;
      cq[nt][e] = cq_s[nt * 8 + 2 * c4 + e];
    }
#pragma unroll
  for (int t = 0; t < 2 * NDB; ++t)
#pragma unroll
    for (int nt = 0; nt < NHT; ++nt) o_acc[t][nt][0] = o_acc[t][nt][1] = o_acc[t][nt][2] = o_acc[t][nt][3] = 0.f;

  const int mi = lane >> 3, r = lane & 7;
  const uint32_t k_lane_off = ((mi & 1) * 8 + r) * RB + (mi >> 1) * 16;
  const uint32_t v_lane_off = ((mi >> 1) * 8 + r) * RB + R::kV + (mi & 1) * 16;
  const uint32_t q_lane_off = static_cast<uint32_t>(smem_u32(q_s)) + mi * 128 + r * 16;
  float* red_s = red;                  // [NH][warp] chunk maxima of the scores
  float* red_z = red + 4 * NH;         // [NH][warp] chunk maxima of z
  float* red_l = red + 8 * NH;         // [NH][warp] parts of l_c

  int c = 0;
  bool failed = false;
  for (; c < n_chunks; ++c) {
    const int b = c % NBUF;
    const bool got = mbar_wait(&full[b], (c / NBUF) & 1, a.status, budget);
    const uint8_t* buf = ring + b * L::kBufBytes;
    const uint32_t bbase = smem_u32(buf);
    const uint32_t tbase = bbase + warp * 16 * RB;  // this warp's 16 cells

    // ---- S^T = K * Q^T for this warp's cells, every head
    float S[NHT][4];
    {
      float sa[NHT][4], sb[NHT][4];
#pragma unroll
      for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[nt][e] = sb[nt][e] = 0.f;
#pragma unroll
      for (int jj = 0; jj < D / 32; ++jj) {
        uint32_t r0, r1, r2, r3, a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(tbase + jj * 32 + k_lane_off, r0, r1, r2, r3);
        i8x4_to_h2x2(r0, kSelB01, kSelB23, a0, a2);
        i8x4_to_h2x2(r1, kSelB01, kSelB23, a1, a3);
        i8x4_to_h2x2(r2, kSelB01, kSelB23, b0, b2);
        i8x4_to_h2x2(r3, kSelB01, kSelB23, b1, b3);
#pragma unroll
        for (int nt = 0; nt < NHT; ++nt) {
          uint32_t q0, q1, q2, q3;
          ldsm_x4(q_lane_off + nt * (D * 16) + jj * 512, q0, q1, q2, q3);
          mma_f16_16816(sa[nt], a0, a1, a2, a3, q0, q1);
          mma_f16_16816(sb[nt], b0, b1, b2, b3, q2, q3);
        }
      }
#pragma unroll
      for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) S[nt][e] = sa[nt][e] + sb[nt][e];
    }
    // ---- scores and this tile's maxima per head
    const uint32_t m = cmask[b * 4 + warp];
    const int4 t0 = *reinterpret_cast<const int4*>(buf + (warp * 16 + g) * RB + R::kScales);
    const int4 t1 = *reinterpret_cast<const int4*>(buf + (warp * 16 + g + 8) * RB + R::kScales);
    const bool c0 = ((m >> g) & 1) != 0, c1 = ((m >> (g + 8)) & 1) != 0;
    if (got && ((c0 && t0.z == 0) || (c1 && t1.z == 0))) set_status(a.status, KVQ_DEV_BAD_BLOCK);
    const bool v0 = c0 && t0.z != 0, v1 = c1 && t1.z != 0;
    const float sk0 = __int_as_float(t0.x), sk1 = __int_as_float(t1.x);
    const float lv0 = v0 ? fast_log2(__int_as_float(t0.y)) : -INFINITY;
    const float lv1 = v1 ? fast_log2(__int_as_float(t1.y)) : -INFINITY;
    float sc[NHT][4], zc[NHT][4];
#pragma unroll
    for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sc[nt][e] = v0 ? S[nt][e] * sk0 * cq[nt][e] : -INFINITY;
        sc[nt][2 + e] = v1 ? S[nt][2 + e] * sk1 * cq[nt][e] : -INFINITY;
        zc[nt][e] = sc[nt][e] + lv0;
        zc[nt][2 + e] = sc[nt][2 + e] + lv1;
        float tms = fmaxf(sc[nt][e], sc[nt][2 + e]), tmz = fmaxf(zc[nt][e], zc[nt][2 + e]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          tms = fmaxf(tms, __shfl_xor_sync(0xffffffffu, tms, off));
          tmz = fmaxf(tmz, __shfl_xor_sync(0xffffffffu, tmz, off));
        }
        if (g == 0) {
          red_s[(nt * 8 + 2 * c4 + e) * 4 + warp] = tms;
          red_z[(nt * 8 + 2 * c4 + e) * 4 + warp] = tmz;
        }
      }
    // every warp's maxima are in place, and every warp leaves together if a wait ran out
    if (chunk_bar_or(!got)) {
      failed = true;
      break;
    }
    // ---- the chunk maximum, the weights relative to the updated maximum, l_c's part
    float ms_new[NHT][2], mz_new[NHT][2];
    uint32_t wf[NHT][4];
#pragma unroll
    for (int nt = 0; nt < NHT; ++nt) {
      float w[2][2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int hd = nt * 8 + 2 * c4 + e;
        const float4 vs4 = *reinterpret_cast<const float4*>(red_s + hd * 4);
        const float4 vz4 = *reinterpret_cast<const float4*>(red_z + hd * 4);
        const float cs = fmaxf(fmaxf(vs4.x, vs4.y), fmaxf(vs4.z, vs4.w));
        const float cz = fmaxf(fmaxf(vz4.x, vz4.y), fmaxf(vz4.z, vz4.w));
        ms_new[nt][e] = fmaxf(ms[nt][e], cs);
        mz_new[nt][e] = fmaxf(mz[nt][e], cz);
        const float msr = ms_new[nt][e] == -INFINITY ? 0.f : ms_new[nt][e];
        const float mzr = mz_new[nt][e] == -INFINITY ? 0.f : mz_new[nt][e];
        float lp = fast_exp2(sc[nt][e] - msr) + fast_exp2(sc[nt][2 + e] - msr);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) lp += __shfl_xor_sync(0xffffffffu, lp, off);
        if (g == 0) red_l[hd * 4 + warp] = lp;
        w[0][e] = fast_exp2(zc[nt][e] - mzr);      // cell g
        w[1][e] = fast_exp2(zc[nt][2 + e] - mzr);  // cell g + 8
      }
      // W as fp16 hi + lo parts, transposed to the PV B layout (cells on K, heads on N)
      const uint32_t h0 = pack_half2(w[0][0], w[0][1]);
      const uint32_t h1 = pack_half2(w[1][0], w[1][1]);
      const __half2 hh0 = *reinterpret_cast<const __half2*>(&h0);
      const __half2 hh1 = *reinterpret_cast<const __half2*>(&h1);
      const uint32_t l0 = pack_half2(w[0][0] - __low2float(hh0), w[0][1] - __high2float(hh0));
      const uint32_t l1 = pack_half2(w[1][0] - __low2float(hh1), w[1][1] - __high2float(hh1));
      wf[nt][0] = movmatrix_trans(h0);
      wf[nt][1] = movmatrix_trans(h1);
      wf[nt][2] = movmatrix_trans(l0);
      wf[nt][3] = movmatrix_trans(l1);
    }
#pragma unroll
    for (int nt = 0; nt < NHT; ++nt) wx[(warp * NHT + nt) * 32 + lane] = make_uint4(wf[nt][0], wf[nt][1], wf[nt][2], wf[nt][3]);
    chunk_bar();  // every warp's W fragments and l_c parts are in place
    // ---- the fold of l: l = fma(l, alpha, l_c)
#pragma unroll
    for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int hd = nt * 8 + 2 * c4 + e;
        const float4 vl4 = *reinterpret_cast<const float4*>(red_l + hd * 4);
        const float lc = (vl4.x + vl4.y) + (vl4.z + vl4.w);
        const float al = ms[nt][e] == -INFINITY ? 0.f : fast_exp2(ms[nt][e] - ms_new[nt][e]);
        lsum[nt][e] = fmaf(lsum[nt][e], al, lc);
        ms[nt][e] = ms_new[nt][e];
      }
    // ---- acc_c = V^T W over the chunk's 64 cells for this warp's dims, from zero; then the fold.
    // One 32-dim block at a time (its two m-tiles' chunk accumulators over the four 16-cell
    // tiles, then their fold), so that only one block's accumulators are live.
    float al[NHT][2];
#pragma unroll
    for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        al[nt][e] = mz[nt][e] == -INFINITY ? 0.f : fast_exp2(mz[nt][e] - mz_new[nt][e]);
        mz[nt][e] = mz_new[nt][e];
      }
#pragma unroll
    for (int db = 0; db < NDB; ++db) {
      float acc_c[2][NHT][4];
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int nt = 0; nt < NHT; ++nt) acc_c[t][nt][0] = acc_c[t][nt][1] = acc_c[t][nt][2] = acc_c[t][nt][3] = 0.f;
#pragma unroll
      for (int tile = 0; tile < 4; ++tile) {
        uint32_t bf[NHT][4];
#pragma unroll
        for (int nt = 0; nt < NHT; ++nt) {
          const uint4 wv = wx[(tile * NHT + nt) * 32 + lane];
          bf[nt][0] = wv.x;
          bf[nt][1] = wv.y;
          bf[nt][2] = wv.z;
          bf[nt][3] = wv.w;
        }
        uint32_t r0, r1, r2, r3, e0, e1, e2, e3, o0, o1, o2, o3;
        ldsm_x4_trans(bbase + tile * 16 * RB + v_lane_off + (warp * NDB + db) * 32, r0, r1, r2, r3);
        i8x4_to_h2x2(r0, kSelB02, kSelB13, e0, o0);  // cells 0..7, dims + 0..15
        i8x4_to_h2x2(r1, kSelB02, kSelB13, e1, o1);  // cells 0..7, dims + 16..31
        i8x4_to_h2x2(r2, kSelB02, kSelB13, e2, o2);  // cells 8..15, dims + 0..15
        i8x4_to_h2x2(r3, kSelB02, kSelB13, e3, o3);  // cells 8..15, dims + 16..31
#pragma unroll
        for (int nt = 0; nt < NHT; ++nt) {
          mma_f16_16816(acc_c[0][nt], e0, e1, e2, e3, bf[nt][0], bf[nt][1]);
          mma_f16_16816(acc_c[0][nt], e0, e1, e2, e3, bf[nt][2], bf[nt][3]);
          mma_f16_16816(acc_c[1][nt], o0, o1, o2, o3, bf[nt][0], bf[nt][1]);
          mma_f16_16816(acc_c[1][nt], o0, o1, o2, o3, bf[nt][2], bf[nt][3]);
        }
      }
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            o_acc[2 * db + t][nt][e] = fmaf(o_acc[2 * db + t][nt][e], al[nt][e], acc_c[t][nt][e]);
            o_acc[2 * db + t][nt][2 + e] = fmaf(o_acc[2 * db + t][nt][2 + e], al[nt][e], acc_c[t][nt][2 + e]);
          }
    }
    // ---- this warp is done with the buffer: refill it with chunk c + NBUF once all four are
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[b]);
    if (c + NBUF < n_chunks) {
      bool freed = true;
      if (lane == 0) freed = mbar_wait(&empty[b], (c / NBUF) & 1, a.status, budget);
      if (__shfl_sync(0xffffffffu, freed ? 1 : 0, 0)) issue(c + NBUF);
    }
  }
  if (failed) {
    // a wait ran out (KVQ_DEV_TIMEOUT is set): the copies issued from this chunk on land before the
    // CTA exits (bounded waits), and the query's rows are written as zeros
    if (lane == 0)
      for (int cc = c; cc < n_issued; ++cc) mbar_wait(&full[cc % NBUF], (cc / NBUF) & 1, a.status, budget);
    __syncwarp();
    for (int e = lane; e < G * (D / 4); e += 32) out_q[(e / (D / 4)) * D + warp * (D / 4) + e % (D / 4)] = 0.0f;
    return;
  }
  // ---- out = O 2^(m_z - m_s) / l for this warp's dims
#pragma unroll
  for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int hd = nt * 8 + 2 * c4 + e;
      if (hd >= G) continue;
      const float fin = (lsum[nt][e] > 0.f && mz[nt][e] != -INFINITY) ? fast_exp2(mz[nt][e] - ms[nt][e]) / lsum[nt][e] : 0.f;
#pragma unroll
      for (int t = 0; t < 2 * NDB; ++t) {
        // M-tile t = 2 db + odd: row g <-> dim 32 db + odd + 2 g, row g + 8 <-> that + 16
        const int d0 = warp * (D / 4) + (t >> 1) * 32 + (t & 1) + 2 * g;
        out_q[hd * D + d0] = o_acc[t][nt][e] * fin;
        out_q[hd * D + d0 + 16] = o_acc[t][nt][2 + e] * fin;
      }
    }
}

size_t sparse_workspace_bytes(int n_blocks_row, int n_kv_heads, int head_dim) {
  return static_cast<size_t>(n_blocks_row) * n_kv_heads * KVQ_BLOCK_SIZE * (2 * head_dim + 16);
}

template <int D, int NHT, int NBUF>
static cudaError_t launch_sparse_chunk(const SparseArgs& a, cudaStream_t stream) {
  using L = ChunkSmem<D, NHT, NBUF>;
  auto kern = (a.fault != 0 || a.wait_budget != kWaitBudgetCycles) ? sparse_chunk_kernel<D, NHT, NBUF, true>
                                                                    : sparse_chunk_kernel<D, NHT, NBUF, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(a.n_queries, a.n_kv_heads), dim3(128), L::kTotal, stream, a);
}

template <int D>
static cudaError_t launch_sparse_d(const SparseArgs& a, cudaStream_t stream) {
  sparse_prep_kernel<D><<<dim3(a.n_blocks_row, a.n_kv_heads), 256, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // One chunk buffer: four CTAs per SM at head_dim 256, whose copies and compute interleave
  // (measured at sparse_32k: 0.527 ms, against 0.628 ms for two buffers and two CTAs per SM).
  const int G = a.n_q_heads / a.n_kv_heads;
  if (G <= 8) return launch_sparse_chunk<D, 1, 1>(a, stream);
  return launch_sparse_chunk<D, 2, 1>(a, stream);
}

cudaError_t launch_sparse(const SparseArgs& a, cudaStream_t stream) {
  if (a.head_dim == 256) return launch_sparse_d<256>(a, stream);
  return launch_sparse_d<128>(a, stream);
}

}  // namespace kvq
