// decode.cu — decode attention over the int8 paged K/V cache, one query per sequence.
//
// Method: "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" §3.3 (locate the paged
// int8 K/V, QK on the int8 codes, scale restore and online softmax, PV, partition merge;
// no dequantised K/V tensor), §1.2 (decode is bound by the K/V read); "dot4-flash-attention"
// README route table (one CTA per head for short contexts; split-K stage 1 over 512-row
// splits emitting partial max / sum / acc, stage 2 merging them with the online-softmax
// rule); "ROCm/RDNA4 (gfx1201) vLLM ..." ("Don't re-read what a group shares": the GQA
// group is folded into the matrix dimension so each K/V page is read once per KV head).
//
// GB300 design.
// * Grid over (split, KV head, sequence); one producer warp streams whole (page, head)
//   blocks of K and V (4 KB each at head_dim 256, contiguous in the cache layout) and
//   their 64-byte scale runs into a shared-memory ring with 1-D bulk copies (TMA) behind
//   full/empty mbarriers.  Consumer warps each own whole pages of the ring.
// * QK and PV of a 16-token page run on the tensor cores (mma.sync m16n8k16, fp32
//   accumulate) with the int8 codes widened to integer-valued fp16 in registers (exact:
//   |code| <= 127).  S^T = K * Q^T puts the 16 tokens on M and the GQA group (<= 8 heads)
//   on N; O^T = V^T * W puts 16 head dimensions on M.  This keeps the FP32 pipe free: at
//   GQA 6 x head_dim 256 a CUDA-core FMA decode needs ~11 us of FMA issue per 68 MB of
//   K/V on GB300, more than the ~10 us the bytes take at the measured HBM rate.
// * Q is bf16, scaled per head by a power of two into fp16 range (exact for bf16 values);
//   the softmax weight W = p * sV of each token is split into fp16 hi + lo parts, two MMAs,
//   so PV keeps ~22 bits.  log2(sV) is folded into a second running maximum so that W
//   stays in [0, 1] whatever the V scales are.
// * Split route: each CTA writes (m_s, m_z, l, acc[D]) per query head; stage 2 merges.
#include "kvq_dev.cuh"
#include "kvq_launch.h"

namespace kvq {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Token order of the 16 rows of the S^T tile (see the fragment-layout notes in the
// kernel): rows 0..7 and 8..15 each hit eight distinct 16-byte bank groups, and after the
// 8x8 transposes every thread holds the weights of the four consecutive tokens its V
// fragment covers.
__device__ __forceinline__ int row_token(int row) {
  // rows 0..7 -> 0,1,4,5,10,11,14,15 ; rows 8..15 -> 2,3,6,7,8,9,12,13
  const int r = row & 7;
  const int base = (r >> 1) * 4 + (r & 1);  // 0,1,4,5,8,9,12,13
  const int hi = row >> 3;
  // first half adds 2 for r >= 4 (10,11,14,15); second half adds 2 for r < 4 (2,3,6,7)
  return base + (((r >= 4) != (hi != 0)) ? 2 : 0);
}

template <int D, int NW, int STAGES>
struct DecodeSmem {
  static constexpr int kKvBytes = D * KVQ_BLOCK_SIZE;            // one (page, head) of K or V
  static constexpr int kStageBytes = 2 * kKvBytes + 2 * 64;      // K, V, k_scale, v_scale
  static constexpr int kRingBytes = STAGES * kStageBytes;
  static constexpr int kBarOffset = kRingBytes;
  static constexpr int kFlagOffset = kBarOffset + 2 * STAGES * 8;
  static constexpr int kTotal = kFlagOffset + STAGES * 4;
  static constexpr int kMergeBytes = NW * 8 * (D + 4) * 4;       // per-warp O and stats
  static_assert(kMergeBytes <= kRingBytes, "merge scratch must fit in the ring");
  static_assert(STAGES % NW == 0, "each stage belongs to one consumer warp");
};

}  // namespace

template <int D, int NW, int STAGES, bool SPLIT>
__global__ void __launch_bounds__((NW + 1) * 32) decode_stage1_kernel(DecodeArgs a) {
  using L = DecodeSmem<D, NW, STAGES>;
  constexpr int KB = L::kKvBytes;
  constexpr int NCH = D / 16;  // 16-dim chunks
  constexpr int NMT = D / 16;  // 16-dim m-tiles of O^T
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  uint64_t* empty = full + STAGES;
  int* stage_ok = reinterpret_cast<int*>(smem + L::kFlagOffset);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int Hq = a.n_q_heads, G = Hq / a.n_kv_heads;

  int ctx = a.ctx_lens[b];
  const int cap = a.max_blocks_per_seq * KVQ_BLOCK_SIZE;
  if (ctx > cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(a.status, KVQ_DEV_BAD_POS);
    ctx = cap;
  }
  if (ctx < 0) ctx = 0;
  const int t_begin = SPLIT ? static_cast<int>(blockIdx.x) * a.split_rows : 0;
  const int t_end = SPLIT ? min(ctx, t_begin + a.split_rows) : ctx;
  const int n_pages = (t_end > t_begin) ? (t_end - t_begin + KVQ_BLOCK_SIZE - 1) / KVQ_BLOCK_SIZE : 0;

  if (n_pages == 0) {
    // No keys in this range: the single route writes zeros; an empty split writes nothing
    // (stage 2 only reads splits that start below ctx).
    if (!SPLIT) {
      for (int i = threadIdx.x; i < G * D; i += blockDim.x)
        a.out[(static_cast<long long>(b) * Hq + kvh * G + i / D) * D + i % D] = 0.0f;
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer warp
    const int32_t* bt = a.block_table + static_cast<long long>(b) * a.max_blocks_per_seq + t_begin / KVQ_BLOCK_SIZE;
    bool alive = true;
    for (int j0 = 0; j0 < n_pages && alive; j0 += 32) {
      int pg = -1;
      if (j0 + lane < n_pages) pg = __ldg(bt + j0 + lane);
      const int cnt = min(32, n_pages - j0);
      for (int jj = 0; jj < cnt; ++jj) {
        const int j = j0 + jj;
        const int page = __shfl_sync(0xffffffffu, pg, jj);
        const int s = j % STAGES;
        int ok_wait = 1;
        if (lane == 0 && j >= STAGES) ok_wait = mbar_wait(&empty[s], ((j / STAGES) - 1) & 1, a.status);
        ok_wait = __shfl_sync(0xffffffffu, ok_wait, 0);
        if (!ok_wait) {
          alive = false;
          break;
        }
        if (lane == 0) {
          const bool ok = page >= 0 && page < a.num_blocks;
          stage_ok[s] = ok ? 1 : 0;
          if (ok) {
            uint8_t* st = ring + s * L::kStageBytes;
            const long long ph = static_cast<long long>(page) * a.n_kv_heads + kvh;
            mbar_arrive_expect_tx(&full[s], 2 * KB + 128);
            bulk_g2s(st, a.k + ph * KB, KB, &full[s]);
            bulk_g2s(st + KB, a.v + ph * KB, KB, &full[s]);
            bulk_g2s(st + 2 * KB, a.k_scale + ph * KVQ_BLOCK_SIZE, 64, &full[s]);
            bulk_g2s(st + 2 * KB + 64, a.v_scale + ph * KVQ_BLOCK_SIZE, 64, &full[s]);
          } else {
            set_status(a.status, KVQ_DEV_BAD_BLOCK);
            mbar_arrive(&full[s]);
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ consumer warps
  const int g = lane >> 2, c = lane & 3;
  float o_acc[NMT][4];
  float ms[2] = {-INFINITY, -INFINITY}, mz[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};
  if (warp > 0) {
    const int cw = warp - 1;
#pragma unroll
    for (int i = 0; i < NMT; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;

    // Q^T fragments: head g of the group, dims 16j + 4c .. 16j + 4c + 3 of chunk j (the
    // chunk's k-slots (2c, 2c+1, 2c+8, 2c+9) carry dims (4c, 4c+1, 4c+2, 4c+3)).
    uint32_t qb[NCH][2];
    float qscale_self = 1.0f;
    {
      const bool real = g < G;
      const uint16_t* qrow = static_cast<const uint16_t*>(a.q) +
                             (static_cast<long long>(b) * Hq + kvh * G + (real ? g : 0)) * D;
      float qv[NCH][4];
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const uint2 raw = real ? __ldg(reinterpret_cast<const uint2*>(qrow + 16 * j + 4 * c)) : make_uint2(0, 0);
        qv[j][0] = __uint_as_float(raw.x << 16);
        qv[j][1] = __uint_as_float(raw.x & 0xFFFF0000u);
        qv[j][2] = __uint_as_float(raw.y << 16);
        qv[j][3] = __uint_as_float(raw.y & 0xFFFF0000u);
#pragma unroll
        for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(qv[j][i]));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      // power of two that brings max|q| into [2^14, 2^15): exact for bf16 inputs
      int e = amax > 0.f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127 : 0;
      e = max(-100, min(e, 127));
      qscale_self = __uint_as_float(static_cast<uint32_t>(127 + 14 - e) << 23);
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        qb[j][0] = pack_half2(qv[j][0] * qscale_self, qv[j][1] * qscale_self);
        qb[j][1] = pack_half2(qv[j][2] * qscale_self, qv[j][3] * qscale_self);
      }
    }
    // score factor of this thread's two heads 2c, 2c+1: softmax_scale * log2(e) / qscale
    float cq[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float qs = __shfl_sync(0xffffffffu, qscale_self, (2 * c + i) * 4);
      cq[i] = a.softmax_scale * kLog2e / qs;
    }

    // per-lane ldmatrix offsets
    const int mi = lane >> 3, r = lane & 7;
    const uint32_t k_lane_off = (mi >> 1) * 256 + row_token((mi & 1) * 8 + r) * 16;
    const uint32_t v_lane_off = lane * 16;
    const int tk0 = row_token(g), tk1 = row_token(g + 8);
    const uint32_t selA = (c < 2) ? kSelB01 : kSelB23;
    const uint32_t selB = (c < 2) ? kSelB23 : kSelB01;

    for (int j = cw; j < n_pages; j += NW) {
      const int s = j % STAGES;
      if (!mbar_wait(&full[s], (j / STAGES) & 1, a.status)) break;
      uint8_t* st = ring + s * L::kStageBytes;
      const uint32_t kbase = smem_u32(st);
      const uint32_t vbase = kbase + KB;
      const float* sks = reinterpret_cast<const float*>(st + 2 * KB);
      const float* svs = reinterpret_cast<const float*>(st + 2 * KB + 64);
      const bool page_ok = stage_ok[s] != 0;
      const int tpage = t_begin + j * KVQ_BLOCK_SIZE;

      // ---- S^T = K * Q^T over the head dimension
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int jj = 0; jj < NCH / 2; ++jj) {
        uint32_t r0, r1, r2, r3, a0, a1, a2, a3;
        ldsm_x4(kbase + jj * 512 + k_lane_off, r0, r1, r2, r3);
        i8x4_to_h2x2(r0, kSelB01, kSelB23, a0, a2);
        i8x4_to_h2x2(r1, kSelB01, kSelB23, a1, a3);
        mma_f16_16816(sa, a0, a1, a2, a3, qb[2 * jj][0], qb[2 * jj][1]);
        i8x4_to_h2x2(r2, kSelB01, kSelB23, a0, a2);
        i8x4_to_h2x2(r3, kSelB01, kSelB23, a1, a3);
        mma_f16_16816(sb, a0, a1, a2, a3, qb[2 * jj + 1][0], qb[2 * jj + 1][1]);
      }
      // rows g (token tk0) and g + 8 (token tk1); columns = heads 2c, 2c + 1
      const bool v0 = page_ok && (tpage + tk0 < t_end);
      const bool v1 = page_ok && (tpage + tk1 < t_end);
      const float sk0 = sks[tk0], sk1 = sks[tk1];
      const float lv0 = v0 ? fast_log2(svs[tk0]) : -INFINITY;
      const float lv1 = v1 ? fast_log2(svs[tk1]) : -INFINITY;
      float s2[2][2], z[2][2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        s2[0][i] = v0 ? (sa[i] + sb[i]) * sk0 * cq[i] : -INFINITY;
        s2[1][i] = v1 ? (sa[2 + i] + sb[2 + i]) * sk1 * cq[i] : -INFINITY;
        z[0][i] = s2[0][i] + lv0;
        z[1][i] = s2[1][i] + lv1;
      }
      float w[2][2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float tms = fmaxf(s2[0][i], s2[1][i]);
        float tmz = fmaxf(z[0][i], z[1][i]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          tms = fmaxf(tms, __shfl_xor_sync(0xffffffffu, tms, off));
          tmz = fmaxf(tmz, __shfl_xor_sync(0xffffffffu, tmz, off));
        }
        const float ms_new = fmaxf(ms[i], tms);
        const float mz_new = fmaxf(mz[i], tmz);
        const float msr = (ms_new == -INFINITY) ? 0.f : ms_new;
        const float mzr = (mz_new == -INFINITY) ? 0.f : mz_new;
        const float as = fast_exp2(ms[i] - msr);
        const float az = fast_exp2(mz[i] - mzr);
        lsum[i] = lsum[i] * as + fast_exp2(s2[0][i] - msr) + fast_exp2(s2[1][i] - msr);
        w[0][i] = fast_exp2(z[0][i] - mzr);
        w[1][i] = fast_exp2(z[1][i] - mzr);
        ms[i] = ms_new;
        mz[i] = mz_new;
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
          o_acc[mt][i] *= az;
          o_acc[mt][2 + i] *= az;
        }
      }
      // ---- W fragments: hi + lo fp16 parts, transposed to the PV B layout
      const uint32_t h0 = pack_half2(w[0][0], w[0][1]);
      const uint32_t h1 = pack_half2(w[1][0], w[1][1]);
      const __half2 hh0 = *reinterpret_cast<const __half2*>(&h0);
      const __half2 hh1 = *reinterpret_cast<const __half2*>(&h1);
      const uint32_t l0 = pack_half2(w[0][0] - __low2float(hh0), w[0][1] - __high2float(hh0));
      const uint32_t l1 = pack_half2(w[1][0] - __low2float(hh1), w[1][1] - __high2float(hh1));
      const uint32_t bh0 = movmatrix_trans(h0), bh1 = movmatrix_trans(h1);
      const uint32_t bl0 = movmatrix_trans(l0), bl1 = movmatrix_trans(l1);

      // ---- O^T += V^T * W
#pragma unroll
      for (int gg = 0; gg < D / 32; ++gg) {
        uint32_t r0, r1, r2, r3, a0, a1, a2, a3;
        ldsm_x4(vbase + gg * 512 + v_lane_off, r0, r1, r2, r3);
        i8x4_to_h2x2(r0, selA, selB, a0, a2);
        i8x4_to_h2x2(r1, selA, selB, a1, a3);
        mma_f16_16816(o_acc[2 * gg], a0, a1, a2, a3, bh0, bh1);
        mma_f16_16816(o_acc[2 * gg], a0, a1, a2, a3, bl0, bl1);
        i8x4_to_h2x2(r2, selA, selB, a0, a2);
        i8x4_to_h2x2(r3, selA, selB, a1, a3);
        mma_f16_16816(o_acc[2 * gg + 1], a0, a1, a2, a3, bh0, bh1);
        mma_f16_16816(o_acc[2 * gg + 1], a0, a1, a2, a3, bl0, bl1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // l over all tokens of the warp for heads 2c, 2c + 1
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) lsum[i] += __shfl_xor_sync(0xffffffffu, lsum[i], off);
    }
  }

  // ------------------------------------------------------------ merge the consumer warps
  __syncthreads();  // every fill was waited for by its consumer: the ring is free
  float* mo = reinterpret_cast<float*>(smem);                 // [NW][8][D]
  float* mstat = mo + NW * 8 * D;                              // [NW][8][4]
  if (warp > 0) {
    const int cw = warp - 1;
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) {
      const int d0 = mt * 16 + g;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        mo[(cw * 8 + 2 * c + i) * D + d0] = o_acc[mt][i];
        mo[(cw * 8 + 2 * c + i) * D + d0 + 8] = o_acc[mt][2 + i];
      }
    }
    if (g == 0) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float* st = mstat + (cw * 8 + 2 * c + i) * 4;
        st[0] = ms[i];
        st[1] = mz[i];
        st[2] = lsum[i];
      }
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int hh = idx / D, d = idx % D;
    float Ms = -INFINITY, Mz = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < NW; ++w2) {
      Ms = fmaxf(Ms, mstat[(w2 * 8 + hh) * 4 + 0]);
      Mz = fmaxf(Mz, mstat[(w2 * 8 + hh) * 4 + 1]);
    }
    float lsum_all = 0.f, o = 0.f;
    if (Ms != -INFINITY) {
#pragma unroll
      for (int w2 = 0; w2 < NW; ++w2) {
        const float* st = mstat + (w2 * 8 + hh) * 4;
        if (st[0] != -INFINITY) lsum_all += st[2] * fast_exp2(st[0] - Ms);
        if (Mz != -INFINITY && st[1] != -INFINITY) o += mo[(w2 * 8 + hh) * D + d] * fast_exp2(st[1] - Mz);
      }
    }
    const int h = kvh * G + hh;
    if (SPLIT) {
      const long long pu = (static_cast<long long>(b) * Hq + h) * a.n_split + blockIdx.x;
      a.part_acc[pu * D + d] = o;
      if (d == 0) {
        a.part_stats[pu * 4 + 0] = Ms;
        a.part_stats[pu * 4 + 1] = Mz;
        a.part_stats[pu * 4 + 2] = lsum_all;
        a.part_stats[pu * 4 + 3] = 0.f;
      }
    } else {
      float res = 0.f;
      if (lsum_all > 0.f && Mz != -INFINITY) res = o * fast_exp2(Mz - Ms) / lsum_all;
      a.out[(static_cast<long long>(b) * Hq + h) * D + d] = res;
    }
  }
}

// Stage 2: log-sum-exp merge of the splits of one (sequence, query head).
//   M_s = max m_s, M_z = max m_z;  l = sum l_s 2^{m_s - M_s};  o = sum acc_s 2^{m_z - M_z};
//   out = o 2^{M_z - M_s} / l.  The per-split weights are computed once into shared memory.
template <int D>
__global__ void __launch_bounds__(D) decode_merge_kernel(DecodeArgs a) {
  extern __shared__ float wts[];  // [n_split] weights for acc, then [n_split] for l
  __shared__ float red[2][32];
  const int h = blockIdx.x, b = blockIdx.y, Hq = a.n_q_heads;
  int ctx = a.ctx_lens[b];
  ctx = max(0, min(ctx, a.max_blocks_per_seq * KVQ_BLOCK_SIZE));
  const int n = min(a.n_split, (ctx + a.split_rows - 1) / a.split_rows);
  const long long pu0 = (static_cast<long long>(b) * Hq + h) * a.n_split;
  const float* stats = a.part_stats + pu0 * 4;
  float Ms = -INFINITY, Mz = -INFINITY;
  for (int s = threadIdx.x; s < n; s += blockDim.x) {
    Ms = fmaxf(Ms, stats[s * 4 + 0]);
    Mz = fmaxf(Mz, stats[s * 4 + 1]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Ms = fmaxf(Ms, __shfl_xor_sync(0xffffffffu, Ms, off));
    Mz = fmaxf(Mz, __shfl_xor_sync(0xffffffffu, Mz, off));
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = Ms;
    red[1][threadIdx.x >> 5] = Mz;
  }
  __syncthreads();
  Ms = -INFINITY;
  Mz = -INFINITY;
  for (int i = 0; i < static_cast<int>(blockDim.x + 31) / 32; ++i) {
    Ms = fmaxf(Ms, red[0][i]);
    Mz = fmaxf(Mz, red[1][i]);
  }
  float lpart = 0.f;
  for (int s = threadIdx.x; s < n; s += blockDim.x) {
    const float ms = stats[s * 4 + 0], mz = stats[s * 4 + 1], l = stats[s * 4 + 2];
    wts[s] = (Mz != -INFINITY && mz != -INFINITY) ? fast_exp2(mz - Mz) : 0.f;
    lpart += (Ms != -INFINITY && ms != -INFINITY) ? l * fast_exp2(ms - Ms) : 0.f;
  }
  __syncthreads();  // red[] reused below
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lpart += __shfl_xor_sync(0xffffffffu, lpart, off);
  if ((threadIdx.x & 31) == 0) red[0][threadIdx.x >> 5] = lpart;
  __syncthreads();
  float l = 0.f;
  for (int i = 0; i < static_cast<int>(blockDim.x + 31) / 32; ++i) l += red[0][i];
  const int d = threadIdx.x;
  const float* acc = a.part_acc + pu0 * D + d;
  float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
  int s = 0;
  for (; s + 4 <= n; s += 4) {
    o0 += acc[(s + 0) * D] * wts[s + 0];
    o1 += acc[(s + 1) * D] * wts[s + 1];
    o2 += acc[(s + 2) * D] * wts[s + 2];
    o3 += acc[(s + 3) * D] * wts[s + 3];
  }
  for (; s < n; ++s) o0 += acc[s * D] * wts[s];
  const float o = (o0 + o1) + (o2 + o3);
  float res = 0.f;
  if (l > 0.f && Mz != -INFINITY) res = o * fast_exp2(Mz - Ms) / l;
  a.out[(static_cast<long long>(b) * Hq + h) * D + d] = res;
}

size_t decode_workspace_bytes(int batch, int n_q_heads, int max_ctx, int head_dim, int split_rows) {
  const long long n_split = (static_cast<long long>(max_ctx) + split_rows - 1) / split_rows;
  const long long units = static_cast<long long>(batch) * n_q_heads * n_split;
  const long long acc = units * head_dim * 4;
  const long long stats = units * 4 * 4;
  return static_cast<size_t>(((acc + 255) / 256) * 256 + stats);
}

template <int D, int NW, int STAGES, bool SPLIT>
static cudaError_t launch_stage1(const DecodeArgs& a, dim3 grid, cudaStream_t stream) {
  using L = DecodeSmem<D, NW, STAGES>;
  auto kern = decode_stage1_kernel<D, NW, STAGES, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
  if (e != cudaSuccess) return e;
  kern<<<grid, (NW + 1) * 32, L::kTotal, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, DecodeRoute route, cudaStream_t stream) {
  if (route == DecodeRoute::kSingle) {
    dim3 grid(1, a.n_kv_heads, a.batch);
    if (a.head_dim == 256) return launch_stage1<256, 8, 24, false>(a, grid, stream);
    return launch_stage1<128, 8, 32, false>(a, grid, stream);
  }
  dim3 grid(a.n_split, a.n_kv_heads, a.batch);
  cudaError_t e;
  if (a.head_dim == 256)
    e = launch_stage1<256, 4, 12, true>(a, grid, stream);
  else
    e = launch_stage1<128, 4, 16, true>(a, grid, stream);
  if (e != cudaSuccess) return e;
  const size_t wbytes = static_cast<size_t>(a.n_split) * sizeof(float);
  dim3 g2(a.n_q_heads, a.batch);
  if (a.head_dim == 256) {
    if (wbytes > 48 * 1024) {
      e = cudaFuncSetAttribute(decode_merge_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(wbytes));
      if (e != cudaSuccess) return e;
    }
    decode_merge_kernel<256><<<g2, 256, wbytes, stream>>>(a);
  } else {
    if (wbytes > 48 * 1024) {
      e = cudaFuncSetAttribute(decode_merge_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(wbytes));
      if (e != cudaSuccess) return e;
    }
    decode_merge_kernel<128><<<g2, 128, wbytes, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kvq
