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
// * Attention.  As decode's stage 1 with cells for page slots: teams of NT warps (NT = ceil(G /
//   8)) stream 16-cell tiles through DEPTH-stage rings of bulk copies on mbarriers; warp nt of
//   a team holds query heads 8nt..8nt+7.  QK: S^T = K * Q^T on mma.sync m16n8k16 (cells on M,
//   heads on N) with the int8 codes widened to integer-valued fp16 (exact).  PV: O^T += V^T * W
//   with the V^T fragments taken straight from the token-major records by ldmatrix.trans: for an
//   8-cell x 16-dim block a lane receives V[2c][2g], V[2c][2g+1], V[2c+1][2g], V[2c+1][2g+1]
//   (c = lane % 4, g = lane / 4), and byte selectors (0, 2) / (1, 3) split that into the A
//   fragments of an even-dimension and an odd-dimension M-tile.  W = p * sV is split into fp16
//   hi + lo parts (two MMAs), and a second running maximum carries log2 sV, as in decode.
// * Precision: fp32 accumulation throughout; the page's chunked fold ("summed from zero and
//   folded with one fma") only changes fp32 rounding, and the tests hold the result to 1e-4 of
//   the FP64 reference.
#include "kvq_dev.cuh"
#include "kvq_launch.h"

namespace kvq {

namespace {

constexpr float kLog2eS = 1.4426950408889634f;
constexpr int kTile = 16;                 // cells per tile (M of the QK MMA, K of the PV MMA)
constexpr float kLazyRescaleS = 8.0f;     // keep a running maximum until a tile exceeds it by 2^8

template <int D>
struct SparseRec {
  static constexpr int kBytes = 2 * D + 16;  // K | V | k_scale | v_scale | valid | pad
  static constexpr int kV = D;
  static constexpr int kScales = 2 * D;
};

template <int D, int NT, int NTEAM, int DEPTH>
struct SparseSmem {
  static constexpr int kWarps = NT * NTEAM;
  static constexpr int kRows = NT * 8;
  static constexpr int kStageBytes = kTile * SparseRec<D>::kBytes;
  static constexpr int kStages = NTEAM * DEPTH;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kQOffset = kRingBytes;
  static constexpr int kQBytes = NT * D * 16;
  static constexpr int kBarOffset = kQOffset + kQBytes;            // full [team][DEPTH], empty [team][DEPTH]
  static constexpr int kMaskOffset = kBarOffset + 2 * kStages * 8;  // copied-cell mask per stage
  static constexpr int kCqOffset = kMaskOffset + kStages * 4;
  static constexpr int kTotal = kCqOffset + kRows * 4;
  static constexpr int kMergeBytes = (kWarps * 8 * (D + 4) + kWarps * 8 * 4 + kWarps * 8 + kRows * 4) * 4;
  static_assert(kMergeBytes <= kRingBytes, "merge scratch must fit in the ring");
  static_assert(kTotal <= 227 * 1024, "shared memory of one CTA");
  static_assert(kQOffset % 16 == 0 && kBarOffset % 8 == 0, "ldmatrix / mbarrier alignment");
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
    // V of slot s, dims 16 db .. 16 db + 15, gathered from the [dim][slot] block
    const int s = t / (D / 16), db = t % (D / 16);
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

// One CTA per (query, KV head): NTEAM teams of NT warps; team p takes tiles p, p + NTEAM, ... of
// the query's cell list; warp nt of a team holds query heads 8 nt .. 8 nt + 7 of the group.
template <int D, int NT, int NTEAM, int DEPTH>
__global__ void __launch_bounds__(NT * NTEAM * 32, 2) sparse_kernel(SparseArgs a) {
  using L = SparseSmem<D, NT, NTEAM, DEPTH>;
  using R = SparseRec<D>;
  constexpr int NW = L::kWarps;
  constexpr int RB = R::kBytes;
  constexpr int NMT = D / 16;  // 16-dim M-tiles of O^T
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  uint8_t* q_s = smem + L::kQOffset;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  uint64_t* empty = full + L::kStages;
  uint32_t* cmask = reinterpret_cast<uint32_t*>(smem + L::kMaskOffset);
  float* cq_s = reinterpret_cast<float*>(smem + L::kCqOffset);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p = warp / NT, nt = warp % NT;
  const int i = blockIdx.x, kvh = blockIdx.y;
  const int Hq = a.n_q_heads, G = Hq / a.n_kv_heads;

  grid_dep_wait();  // the records come from the pre-pass
  const int c_begin = a.cell_offsets[i], c_end = a.cell_offsets[i + 1];
  const int n_cells = max(0, c_end - c_begin);
  const int n_tiles = (n_cells + kTile - 1) / kTile;
  if (n_tiles == 0) {
    for (int e = threadIdx.x; e < G * D; e += blockDim.x)
      a.out[(static_cast<long long>(i) * Hq + kvh * G + e / D) * D + e % D] = 0.0f;
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&full[s], 1);
      if (NT > 1) mbar_init(&empty[s], NT);
    }
    mbar_fence_init();
  }
  __syncthreads();

  const int npp = (p < n_tiles) ? (n_tiles - p + NTEAM - 1) / NTEAM : 0;  // tiles of this team
  uint64_t* pfull = full + p * DEPTH;
  uint64_t* pempty = empty + p * DEPTH;
  uint32_t* pmask = cmask + p * DEPTH;
  uint8_t* pring = ring + p * DEPTH * L::kStageBytes;

  // Cell positions of the team's tiles, loaded DEPTH tiles ahead of their copies (lane l < 16
  // holds cell l of a tile; pos_q[k % DEPTH] holds tile k's): the tiles are issued in order, so
  // the index load of tile k + DEPTH goes out right after tile k's copies and has DEPTH tiles of
  // work to arrive, instead of stalling the issuing warp on a memory round trip every tile.
  auto load_pos = [&](int k) {
    const int cb = c_begin + (p + k * NTEAM) * kTile;
    return (k < npp && lane < kTile && cb + lane < c_end) ? __ldg(a.cells + cb + lane) : -1;
  };
  int pos_q[DEPTH];
#pragma unroll
  for (int k = 0; k < DEPTH; ++k) pos_q[k] = nt == 0 ? load_pos(k) : -1;
  // the issuing warp, collectively: copy the records of tile k's cells into its slot (lane l < 16
  // copies cell l); cells outside the list or the mapped range are not copied and are masked
  auto issue = [&](int k) {
    const int s = k % DEPTH;
    const int cb = c_begin + (p + k * NTEAM) * kTile;
    int pos = -1;
#pragma unroll
    for (int d = 0; d < DEPTH; ++d)
      if (d == s) {
        pos = pos_q[d];
        pos_q[d] = load_pos(k + DEPTH);
      }
    bool ok = false;
    long long rec = 0;
    if (lane < kTile && cb + lane < c_end) {
      if (pos >= 0 && pos / KVQ_BLOCK_SIZE < a.n_blocks_row) {
        ok = true;
        rec = ((static_cast<long long>(pos / KVQ_BLOCK_SIZE) * a.n_kv_heads + kvh) * KVQ_BLOCK_SIZE +
               pos % KVQ_BLOCK_SIZE) * RB;
      } else {
        set_status(a.status, KVQ_DEV_BAD_CELL);
      }
    }
    const uint32_t m = __ballot_sync(0xffffffffu, ok);
    if (lane == 0) {
      pmask[s] = m;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&pfull[s], __popc(m) * RB);
    }
    __syncwarp();
    if (ok) bulk_g2s(pring + s * L::kStageBytes + lane * RB, a.records + rec, RB, &pfull[s]);
  };
  if (nt == 0)
    for (int k = 0; k < min(DEPTH, npp); ++k) issue(k);

  // ---- Q^T fragments (as decode): row r = head r of the group, fp16 q * 2^e per head
  for (int h = warp; h < L::kRows; h += NW) {
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

  const int g = lane >> 2, c = lane & 3;
  float o_acc[NMT][4];
#pragma unroll
  for (int t = 0; t < NMT; ++t) o_acc[t][0] = o_acc[t][1] = o_acc[t][2] = o_acc[t][3] = 0.f;
  float ms[2] = {-INFINITY, -INFINITY}, mz[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};
  const float cq0 = cq_s[nt * 8 + 2 * c], cq1 = cq_s[nt * 8 + 2 * c + 1];

  // per-lane ldmatrix offsets.  K: matrix mi = lane / 8 holds cells 8 (mi & 1) + r of dim chunk
  // (mi >> 1) of the chunk pair; V (transposed load): cells 8 (mi >> 1) + r, dims 16 (mi & 1).
  const int mi = lane >> 3, r = lane & 7;
  const uint32_t k_lane_off = ((mi & 1) * 8 + r) * RB + (mi >> 1) * 16;
  const uint32_t v_lane_off = ((mi >> 1) * 8 + r) * RB + R::kV + (mi & 1) * 16;
  const uint32_t q_lane_off = static_cast<uint32_t>(smem_u32(q_s)) + nt * (D * 16) + mi * 128 + r * 16;

  int k = 0;
  for (; k < npp; ++k) {
    const int s = k % DEPTH;
    const bool got = mbar_wait(&pfull[s], (k / DEPTH) & 1, a.status);
    const uint8_t* st = pring + s * L::kStageBytes;
    const uint32_t sbase = smem_u32(st);

    // ---- S^T = K * Q^T over the head dimension
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int jj = 0; jj < D / 32; ++jj) {
      uint32_t r0, r1, r2, r3, a0, a1, a2, a3, q0, q1, q2, q3;
      ldsm_x4(sbase + jj * 32 + k_lane_off, r0, r1, r2, r3);
      ldsm_x4(q_lane_off + jj * 512, q0, q1, q2, q3);
      i8x4_to_h2x2(r0, kSelB01, kSelB23, a0, a2);
      i8x4_to_h2x2(r1, kSelB01, kSelB23, a1, a3);
      mma_f16_16816(sa, a0, a1, a2, a3, q0, q1);
      i8x4_to_h2x2(r2, kSelB01, kSelB23, a0, a2);
      i8x4_to_h2x2(r3, kSelB01, kSelB23, a1, a3);
      mma_f16_16816(sb, a0, a1, a2, a3, q2, q3);
    }
    if (!__all_sync(0xffffffffu, got)) break;
    const float S[4] = {sa[0] + sb[0], sa[1] + sb[1], sa[2] + sb[2], sa[3] + sb[3]};

    // ---- online softmax over the tile's cells g and g + 8
    const uint32_t m = pmask[s];
    const int4 t0 = *reinterpret_cast<const int4*>(st + g * RB + R::kScales);
    const int4 t1 = *reinterpret_cast<const int4*>(st + (g + 8) * RB + R::kScales);
    const bool c0 = ((m >> g) & 1) != 0, c1 = ((m >> (g + 8)) & 1) != 0;
    if ((c0 && t0.z == 0) || (c1 && t1.z == 0)) set_status(a.status, KVQ_DEV_BAD_BLOCK);
    const bool v0 = c0 && t0.z != 0, v1 = c1 && t1.z != 0;
    const float sk0 = __int_as_float(t0.x), sk1 = __int_as_float(t1.x);
    const float lv0 = v0 ? fast_log2(__int_as_float(t0.y)) : -INFINITY;
    const float lv1 = v1 ? fast_log2(__int_as_float(t1.y)) : -INFINITY;
    float w[2][2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float cqe = e ? cq1 : cq0;
      const float s0 = v0 ? S[e] * sk0 * cqe : -INFINITY;
      const float s1 = v1 ? S[2 + e] * sk1 * cqe : -INFINITY;
      const float z0 = s0 + lv0, z1 = s1 + lv1;
      float tms = fmaxf(s0, s1), tmz = fmaxf(z0, z1);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        tms = fmaxf(tms, __shfl_xor_sync(0xffffffffu, tms, off));
        tmz = fmaxf(tmz, __shfl_xor_sync(0xffffffffu, tmz, off));
      }
      if (tms > ms[e] + kLazyRescaleS) {
        lsum[e] *= (ms[e] == -INFINITY) ? 0.f : fast_exp2(ms[e] - tms);
        ms[e] = tms;
      }
      if (tmz > mz[e] + kLazyRescaleS) {
        const float az = (mz[e] == -INFINITY) ? 0.f : fast_exp2(mz[e] - tmz);
#pragma unroll
        for (int t = 0; t < NMT; ++t) {
          o_acc[t][e] *= az;
          o_acc[t][2 + e] *= az;
        }
        mz[e] = tmz;
      }
      const float msr = (ms[e] == -INFINITY) ? 0.f : ms[e];
      const float mzr = (mz[e] == -INFINITY) ? 0.f : mz[e];
      lsum[e] += fast_exp2(s0 - msr) + fast_exp2(s1 - msr);
      w[0][e] = fast_exp2(z0 - mzr);
      w[1][e] = fast_exp2(z1 - mzr);
    }
    // W fragments (cells on K, heads on N): hi + lo fp16 parts
    const uint32_t h0 = pack_half2(w[0][0], w[0][1]);
    const uint32_t h1 = pack_half2(w[1][0], w[1][1]);
    const __half2 hh0 = *reinterpret_cast<const __half2*>(&h0);
    const __half2 hh1 = *reinterpret_cast<const __half2*>(&h1);
    const uint32_t l0 = pack_half2(w[0][0] - __low2float(hh0), w[0][1] - __high2float(hh0));
    const uint32_t l1 = pack_half2(w[1][0] - __low2float(hh1), w[1][1] - __high2float(hh1));
    const uint32_t bh0 = movmatrix_trans(h0), bh1 = movmatrix_trans(h1);
    const uint32_t bl0 = movmatrix_trans(l0), bl1 = movmatrix_trans(l1);

    // ---- O^T += V^T * W: per 32-dim block, an even-dimension and an odd-dimension M-tile
#pragma unroll
    for (int db = 0; db < D / 32; ++db) {
      uint32_t r0, r1, r2, r3, e0, e1, e2, e3, o0, o1, o2, o3;
      ldsm_x4_trans(sbase + v_lane_off + db * 32, r0, r1, r2, r3);
      i8x4_to_h2x2(r0, kSelB02, kSelB13, e0, o0);  // cells 0..7, dims 32 db + 0..15
      i8x4_to_h2x2(r1, kSelB02, kSelB13, e1, o1);  // cells 0..7, dims 32 db + 16..31
      i8x4_to_h2x2(r2, kSelB02, kSelB13, e2, o2);  // cells 8..15, dims 32 db + 0..15
      i8x4_to_h2x2(r3, kSelB02, kSelB13, e3, o3);  // cells 8..15, dims 32 db + 16..31
      mma_f16_16816(o_acc[2 * db], e0, e1, e2, e3, bh0, bh1);
      mma_f16_16816(o_acc[2 * db], e0, e1, e2, e3, bl0, bl1);
      mma_f16_16816(o_acc[2 * db + 1], o0, o1, o2, o3, bh0, bh1);
      mma_f16_16816(o_acc[2 * db + 1], o0, o1, o2, o3, bl0, bl1);
    }
    __syncwarp();
    if constexpr (NT == 1) {
      if (k + DEPTH < npp) issue(k + DEPTH);
    } else {
      if (lane == 0) mbar_arrive(&pempty[s]);
      if (nt == 0 && k + DEPTH < npp) {
        bool freed = true;
        if (lane == 0) freed = mbar_wait(&pempty[s], (k / DEPTH) & 1, a.status);
        if (__shfl_sync(0xffffffffu, freed ? 1 : 0, 0)) issue(k + DEPTH);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 2; ++e) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) lsum[e] += __shfl_xor_sync(0xffffffffu, lsum[e], off);
  }

  // ------------------------------------------------------------ merge the teams
  __syncthreads();  // every issued copy was waited for: the ring is free
  constexpr int RS = D + 4;
  float* mo = reinterpret_cast<float*>(smem);   // [NW][8][RS]
  float* mstat = mo + NW * 8 * RS;              // [NW][8][4]
  float* mw = mstat + NW * 8 * 4;               // [rows][NTEAM]
  float* mfin = mw + NW * 8;                    // [rows][4]
#pragma unroll
  for (int t = 0; t < NMT; ++t) {
    // M-tile t = 2 db + odd: row g <-> dim 32 db + odd + 2 g, row g + 8 <-> dim 32 db + 16 + odd + 2 g
    const int d0 = (t >> 1) * 32 + (t & 1) + 2 * g;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      mo[(warp * 8 + 2 * c + e) * RS + d0] = o_acc[t][e];
      mo[(warp * 8 + 2 * c + e) * RS + d0 + 16] = o_acc[t][2 + e];
    }
  }
  if (g == 0) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float* stt = mstat + (warp * 8 + 2 * c + e) * 4;
      stt[0] = ms[e];
      stt[1] = mz[e];
      stt[2] = lsum[e];
    }
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int hh = threadIdx.x;
    float Ms = -INFINITY, Mz = -INFINITY;
    for (int q2 = 0; q2 < NTEAM; ++q2) {
      Ms = fmaxf(Ms, mstat[(q2 * L::kRows + hh) * 4 + 0]);
      Mz = fmaxf(Mz, mstat[(q2 * L::kRows + hh) * 4 + 1]);
    }
    float lsum_all = 0.f;
    for (int q2 = 0; q2 < NTEAM; ++q2) {
      const float* stt = mstat + (q2 * L::kRows + hh) * 4;
      if (Ms != -INFINITY && stt[0] != -INFINITY) lsum_all += stt[2] * fast_exp2(stt[0] - Ms);
      mw[hh * NTEAM + q2] = (Mz != -INFINITY && stt[1] != -INFINITY) ? fast_exp2(stt[1] - Mz) : 0.f;
    }
    mfin[hh * 4 + 3] = (lsum_all > 0.f && Mz != -INFINITY) ? fast_exp2(Mz - Ms) / lsum_all : 0.f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int hh = idx / D, d = idx % D;
    float o = 0.f;
#pragma unroll
    for (int q2 = 0; q2 < NTEAM; ++q2) o = fmaf(mo[(q2 * L::kRows + hh) * RS + d], mw[hh * NTEAM + q2], o);
    a.out[(static_cast<long long>(i) * Hq + kvh * G + hh) * D + d] = o * mfin[hh * 4 + 3];
  }
}

size_t sparse_workspace_bytes(int n_blocks_row, int n_kv_heads, int head_dim) {
  return static_cast<size_t>(n_blocks_row) * n_kv_heads * KVQ_BLOCK_SIZE * (2 * head_dim + 16);
}

template <int D, int NT>
static cudaError_t launch_sparse_attn(const SparseArgs& a, cudaStream_t stream) {
  // four teams, three stages each: two CTAs per SM, so one CTA's start-up and merge overlap
  // the other's streaming (measured at sparse_32k: 0.668 ms, against 0.742 ms for one CTA of
  // eight teams per SM and 0.77-1.07 ms for the other shapes tried)
  constexpr int NTEAM = 4;
  constexpr int DEPTH = 3;
  using L = SparseSmem<D, NT, NTEAM, DEPTH>;
  auto kern = sparse_kernel<D, NT, NTEAM, DEPTH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(a.n_queries, a.n_kv_heads), dim3(L::kWarps * 32), L::kTotal, stream, a);
}

template <int D>
static cudaError_t launch_sparse_d(const SparseArgs& a, cudaStream_t stream) {
  sparse_prep_kernel<D><<<dim3(a.n_blocks_row, a.n_kv_heads), 256, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int G = a.n_q_heads / a.n_kv_heads;
  if (G <= 8) return launch_sparse_attn<D, 1>(a, stream);
  return launch_sparse_attn<D, 2>(a, stream);
}

cudaError_t launch_sparse(const SparseArgs& a, cudaStream_t stream) {
  if (a.head_dim == 256) return launch_sparse_d<256>(a, stream);
  return launch_sparse_d<128>(a, stream);
}

}  // namespace kvq
