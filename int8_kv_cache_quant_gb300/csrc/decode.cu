// decode.cu — decode attention over the int8 paged K/V cache: one query per sequence, or nq
// query rows per sequence (speculative / MTP verify, causal among the nq newest tokens).
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
// * Grid over (split, KV head, sequence).  Each of the CTA's eight warps takes whole pages
//   (warp w: pages w, w + 8, ...) and streams each (page, head) block of K and V (4 KB each
//   at head_dim 256, contiguous in the cache layout) and its two 64-byte scale runs into its
//   own DEPTH-stage shared-memory ring with 1-D bulk copies (TMA) completing on mbarriers;
//   it refills a slot as soon as it has read the page in it.  A warp does QK, the online
//   softmax and PV of a page over the whole head dimension: no exchange with another warp
//   and no softmax computed twice.  The warps' partial results are merged at the end of the
//   CTA.
// * QK and PV of a 16-token page run on the tensor cores (mma.sync m16n8k16, fp32
//   accumulate) with the int8 codes widened to integer-valued fp16 in registers (exact:
//   |code| <= 127).  S^T = K * Q^T puts the 16 tokens on M and the GQA group (<= 8 heads; a
//   larger group, up to 16, takes the rows path below with its heads as the rows)
//   on N; O^T = V^T * W puts 16 head dimensions on M.  This keeps the FP32 pipe free: at
//   GQA 6 x head_dim 256 a CUDA-core FMA decode needs ~11 us of FMA issue per 68 MB of
//   K/V on GB300, more than the ~10 us the bytes take at the measured HBM rate.
// * Q is bf16, scaled per head by a power of two into fp16 range (exact for bf16 values);
//   the softmax weight W = p * sV of each token is split into fp16 hi + lo parts, two MMAs,
//   so PV keeps ~22 bits.  log2(sV) is folded into a second running maximum so that W
//   stays in [0, 1] whatever the V scales are.
// * Split route: each CTA writes (m_s, m_z, l, acc[D]) per query head; stage 2 merges.
// * Verify rows ([DOT4] "Future Work": MTP verify at nq = 2-4; "ROCm/RDNA4 (gfx1201) vLLM
//   ..." row-shape routing: spec-verify with 2-6 rows): the nq query rows of a sequence
//   join the GQA group on the N side, rows = G * nq (row r = query i * G + head).  A warp
//   holds one 8-row n-tile of S^T and O^T; NT = ceil(rows / 8) warps form a team that shares
//   one page ring, so each K/V page is still read from HBM once for all nq rows ("Redundancy
//   is a currency": the byte-bound decode does not re-stream K per row tile).  A slot is
//   refilled once every warp of its team has arrived on the slot's empty barrier.
// * Fused decode step ("gfx936 ..." §4.2 measures decode together with the producer; §2.2
//   writes the new token's K/V in the producer): with k_new / v_new given, the nq newest
//   tokens of each sequence are quantised (quant_rule.cuh, the kvq_quant_write rule) and
//   written into their page, before its bulk copy, by the warp that will issue that copy (a
//   proxy fence orders the generic stores before the copy's reads).  Only that warp's team
//   reads the page, so no other CTA or launch has to wait for the write; the write sits in the
//   CTA's prologue, off the page loop.  One new token at head_dim 256: the owning warp stores the
//   codes without waiting for them and writes them into its landed shared-memory copy of the
//   page instead (see PATCH below).
#include <type_traits>

#include "kvq_dev.cuh"
#include "kvq_launch.h"
#include "quant_rule.cuh"

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

// NTEAM teams of NT warps; each team streams its pages through DEPTH private stages.
template <int D, int NT, int NTEAM, int DEPTH>
struct DecodeSmem {
  static constexpr int kWarps = NT * NTEAM;
  static constexpr int kRows = NT * 8;                            // query rows of the CTA (padded)
  static constexpr int kKvBytes = D * KVQ_BLOCK_SIZE;             // one (page, head) of K or V
  static constexpr int kStageBytes = 2 * kKvBytes + 2 * 64;       // K, V, k_scale, v_scale
  static constexpr int kStages = NTEAM * DEPTH;                   // DEPTH private stages per team
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kQOffset = kRingBytes;                     // Q^T fragments (fp16)
  static constexpr int kQBytes = NT * D * 16;                     // per n-tile: D/16 chunks x 2 x 8 rows x 16 B
  static constexpr int kBarOffset = kQOffset + kQBytes;           // full [team][DEPTH], then empty [team][DEPTH]
  static constexpr int kFlagOffset = kBarOffset + (NT > 1 ? 2 : 1) * kStages * 8;  // page-ok flags [team][DEPTH]
  static constexpr int kCqOffset = kFlagOffset + kStages * 4;     // score factor per row
  static constexpr int kFailOffset = kCqOffset + kRows * 4;       // a warp's bounded wait ran out
  static constexpr int kTotal = kFailOffset + 16;
  static constexpr int kMergeBytes = (kWarps * 8 * (D + 4) + kWarps * 8 * 4 + kWarps * 8 + kRows * 4) * 4;
  static_assert(kMergeBytes <= kRingBytes, "merge scratch must fit in the ring");
  static_assert(kWarps >= 8 && kWarps <= 16, "8..16 warps");
  static_assert(kTotal <= 227 * 1024, "shared memory of one CTA");
  static_assert(kQOffset % 16 == 0 && kBarOffset % 8 == 0, "ldmatrix / mbarrier alignment");
};

constexpr float kLazyRescale = 8.0f;  // keep a running maximum until the tile exceeds it by 2^8

}  // namespace

// Fused step, warp-collective: quantise the new tokens at positions lo, lo + step, ... < hi
// (token j of sequence b at position first_new + j) and store them into `page`, then order
// those stores before the async-proxy bulk copy of the page that is issued later.
template <int D>
__device__ __forceinline__ void write_new_tokens(const DecodeArgs& a, int b, int kvh, int nq, int page, int lo,
                                                 int hi, int step, int first_new, int lane) {
  constexpr int P = D / 32;
  const long long ph = static_cast<long long>(page) * a.n_kv_heads + kvh;
  for (int t = lo; t < hi; t += step) {
    const long long row = ((static_cast<long long>(b) * nq + (t - first_new)) * a.n_kv_heads + kvh) * D + lane * P;
    const int slot = t % KVQ_BLOCK_SIZE;
    float xk[P], xv[P];
    uint32_t packed[P / 4];
    // both rows before any store (the stores could alias the inputs as far as the compiler knows)
    load_bf16_lane(static_cast<const uint16_t*>(a.k_new) + row, xk);
    load_bf16_lane(static_cast<const uint16_t*>(a.v_new) + row, xv);
    const float sk = quant_rule_warp_packed(xk, packed);
    store_k_codes<D>(a.k, ph, slot, lane, packed);
    const float sv = quant_rule_warp_packed(xv, packed);
    store_v_codes<D>(a.v, ph, slot, lane, packed);
    if (lane == 0) {
      a.k_scale[ph * KVQ_BLOCK_SIZE + slot] = sk;
      a.v_scale[ph * KVQ_BLOCK_SIZE + slot] = sv;
    }
  }
  // the stores above, then the bulk copy that reads them (async proxy)
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
}

// Stage 1.  CTA = NTEAM teams of NT warps over the key range of one (split, KV head,
// sequence); team p takes pages p, p + NTEAM, ... of the range through its own DEPTH-stage
// ring, and warp nt of the team accumulates S^T, the softmax statistics and O^T of query rows
// 8 nt .. 8 nt + 7 over the whole head dimension.  MROW: more than one query row per sequence
// (the causal bound among the rows applies); without it nq is 1 at compile time.  WRITE: the
// fused step's write of the new tokens is compiled in (and runs when a.k_new is set).
template <int D, int NT, int NTEAM, int DEPTH, bool SPLIT, bool MROW, bool WRITE>
__global__ void __launch_bounds__(NT * NTEAM * 32, (D == 128 && NT * NTEAM == 8) ? 2 : 1)
    decode_stage1_kernel(DecodeArgs a) {
  using L = DecodeSmem<D, NT, NTEAM, DEPTH>;
  constexpr int NW = L::kWarps;
  constexpr int KB = L::kKvBytes;
  constexpr int NCH_H = D / 16;  // 16-dim chunks of the head dimension (whole, one warp)
  constexpr int NMT_H = D / 16;  // 16-dim m-tiles of O^T
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  uint8_t* q_s = smem + L::kQOffset;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  uint64_t* empty = full + L::kStages;
  int* stage_ok = reinterpret_cast<int*>(smem + L::kFlagOffset);
  float* cq_s = reinterpret_cast<float*>(smem + L::kCqOffset);
  volatile int* cta_failed = reinterpret_cast<volatile int*>(smem + L::kFailOffset);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p = warp / NT;   // team: takes whole pages
  const int nt = warp % NT;  // n-tile of query rows of this warp
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int Hq = a.n_q_heads, G = Hq / a.n_kv_heads;
  const int nq = MROW ? a.nq : 1, R = G * nq;  // query rows of this (sequence, KV head)

  grid_dep_wait();  // inputs may come from the previous kernel of the stream
  const int t_begin = SPLIT ? static_cast<int>(blockIdx.x) * a.split_rows : 0;
  const int32_t* bt = a.block_table + static_cast<long long>(b) * a.max_blocks_per_seq + t_begin / KVQ_BLOCK_SIZE;
  // The team's first 32 page ids are read together with ctx (not after it): entries past the
  // sequence's pages are read but not used; the row bound keeps every read inside the table.
  int pg = -1;
  {
    const int first = t_begin / KVQ_BLOCK_SIZE + p + lane * NTEAM;
    if (nt == 0 && first < a.max_blocks_per_seq) pg = __ldg(bt + p + lane * NTEAM);
  }
  int ctx = a.ctx_lens[b];
  // The query rows are requested next, ahead of every page copy: a load issued after the first
  // copies queues behind tens of megabytes of them, and no page can be used before Q is set up
  // (which would leave the copies' slots full and HBM idle once they have landed).  Warp w holds
  // rows w, w + NW, ... of the Q^T set-up below.
  constexpr int PER = D / 32;  // dims per lane
  constexpr int kQPerWarp = (L::kRows + NW - 1) / NW;
  uint4 qraw[kQPerWarp];
#pragma unroll
  for (int i = 0; i < kQPerWarp; ++i) {
    const int h = warp + i * NW;
    const bool real = h < R;
    const int qi = (MROW && real) ? h / G : 0, hh = !MROW ? h : real ? h % G : 0;
    const uint16_t* qrow = static_cast<const uint16_t*>(a.q) +
                           ((static_cast<long long>(b) * nq + qi) * Hq + kvh * G + hh) * D + lane * PER;
    qraw[i] = make_uint4(0, 0, 0, 0);
    if (real) {
      if constexpr (PER == 8) {
        qraw[i] = __ldg(reinterpret_cast<const uint4*>(qrow));
      } else {
        const uint2 r2 = __ldg(reinterpret_cast<const uint2*>(qrow));
        qraw[i].x = r2.x;
        qraw[i].y = r2.y;
      }
    }
  }
  // keys this call may read: what the block-table row maps, and the host's bound max_ctx (the
  // split route's grid and workspace are sized by it); a longer ctx is clamped to it, on both
  // routes, and reported
  const int cap = min(a.max_blocks_per_seq * KVQ_BLOCK_SIZE, a.max_ctx);
  // fused step: the new tokens are written only when their positions are all mapped
  const bool write_new = WRITE && a.k_new != nullptr && ctx >= nq && ctx <= cap;
  if (ctx > cap || (WRITE && a.k_new != nullptr && ctx < nq)) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(a.status, KVQ_DEV_BAD_POS);
    ctx = min(ctx, cap);
  }
  if (ctx < 0) ctx = 0;
  const int t_end = SPLIT ? min(ctx, t_begin + a.split_rows) : ctx;
  const int n_pages = (t_end > t_begin) ? (t_end - t_begin + KVQ_BLOCK_SIZE - 1) / KVQ_BLOCK_SIZE : 0;
  // One new token (plain decode, single-warp teams, head_dim 256): the owning warp requests the
  // token's bf16 K/V rows now, quantises them after the Q set-up and stores the codes to the cache
  // with no fence, and writes the same codes into its shared-memory copy of the page once that copy
  // has landed (the copy may read the slot before or after the stores; the patch makes it right
  // either way).  Nothing on the way to the page's copy waits for the write, which otherwise held
  // the owning warp (the last CTA's) about 4 us behind the others.  At head_dim 128 (two CTAs per
  // SM) the write before the copy measured faster, so it stays there.
  constexpr bool PATCH = WRITE && !MROW && NT == 1 && D == 256;
  using RowRaw = typename std::conditional<PATCH && PER == 8, uint4, uint2>::type;
  int k_w = -1;  // PATCH: this warp's page index holding the new token, or -1
  int pr_w = 0;
  RowRaw raw_k{}, raw_v{};
  if constexpr (PATCH) {
    const int tok = ctx - 1;  // nq = 1: the new token's position
    if (write_new && tok >= t_begin && tok < t_end) {
      pr_w = (tok - t_begin) / KVQ_BLOCK_SIZE;
      if (pr_w % NTEAM == p) {
        k_w = pr_w / NTEAM;
        const long long row = (static_cast<long long>(b) * a.n_kv_heads + kvh) * D + lane * PER;
        // volatile: the loads go out here, ahead of the copies, not where their values are used
        const uint16_t* pk = static_cast<const uint16_t*>(a.k_new) + row;
        const uint16_t* pv = static_cast<const uint16_t*>(a.v_new) + row;
        if constexpr (PER == 8) {
          asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(raw_k.x), "=r"(raw_k.y), "=r"(raw_k.z), "=r"(raw_k.w) : "l"(pk));
          asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(raw_v.x), "=r"(raw_v.y), "=r"(raw_v.z), "=r"(raw_v.w) : "l"(pv));
        } else {
          asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(raw_k.x), "=r"(raw_k.y) : "l"(pk));
          asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(raw_v.x), "=r"(raw_v.y) : "l"(pv));
        }
      }
    }
  }
  if constexpr (WRITE && !PATCH) {
    // fused step: warp 0 of a CTA whose range holds new tokens pulls their bf16 K/V rows into L2
    // now, so the write in the prologue below finds them there
    if (write_new && warp == 0) {
      const int lo = max(ctx - nq, t_begin);
      for (int t = lo + (lane >> 4); t < t_end; t += 2) {
        const long long row = ((static_cast<long long>(b) * nq + (t - (ctx - nq))) * a.n_kv_heads + kvh) * D;
        const char* src = static_cast<const char*>((lane & 8) ? a.v_new : a.k_new) + row * 2 + (lane & 7) * (D / 4);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
      }
    }
  }

  if (n_pages == 0) {
    // No keys in this range: the single route writes zeros; an empty split writes nothing
    // (stage 2 only reads splits that start below ctx).
    if (!SPLIT) {
      for (int i = threadIdx.x; i < R * D; i += blockDim.x) {
        const int r = i / D;
        a.out[((static_cast<long long>(b) * nq + r / G) * Hq + kvh * G + r % G) * D + i % D] = 0.0f;
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&full[s], 1);
      if (NT > 1) mbar_init(&empty[s], NT);
    }
    *cta_failed = 0;
    mbar_fence_init();
  }
  __syncthreads();  // the barriers are initialised before any copy completes on them

  const int npp = (p < n_pages) ? (n_pages - p + NTEAM - 1) / NTEAM : 0;  // pages of this team
  uint64_t* pfull = full + p * DEPTH;
  uint64_t* pempty = empty + p * DEPTH;
  int* pok = stage_ok + p * DEPTH;
  uint8_t* pring = ring + p * DEPTH * L::kStageBytes;

  // page ids of this team (read by its issuing warp, nt = 0), a window of 32 in its lanes
  // (lane i <-> page k = wb + i)
  int wb = 0;
  if (lane >= npp) pg = -1;
  int n_issued = 0;  // pages of the team whose copies the issuing warp has issued
  // test-only fault injection: the first team of CTA 0 leaves its second page un-issued (no copy
  // in flight, its full barrier never completes), so its bounded waits run out
  const bool skip_one = a.fault == 1 && p == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
  // the issuing warp, collectively: issue the copy of the team's page k into its slot
  auto issue = [&](int k) {
    while (k >= wb + 32) {
      wb += 32;
      pg = (wb + lane < npp) ? __ldg(bt + p + (wb + lane) * NTEAM) : -1;
    }
    const int page = __shfl_sync(0xffffffffu, pg, k - wb);
    ++n_issued;
    if (lane == 0 && !(skip_one && k == 1)) {
      const int s = k % DEPTH;
      const bool ok = page >= 0 && page < a.num_blocks;
      pok[s] = ok ? 1 : 0;
      if (ok) {
        uint8_t* st = pring + s * L::kStageBytes;
        const long long ph = static_cast<long long>(page) * a.n_kv_heads + kvh;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&pfull[s], 2 * KB + 128);
        bulk_g2s(st, a.k + ph * KB, KB, &pfull[s]);
        bulk_g2s(st + KB, a.v + ph * KB, KB, &pfull[s]);
        bulk_g2s(st + 2 * KB, a.k_scale + ph * KVQ_BLOCK_SIZE, 64, &pfull[s]);
        bulk_g2s(st + 2 * KB + 64, a.v_scale + ph * KVQ_BLOCK_SIZE, 64, &pfull[s]);
      } else {
        set_status(a.status, KVQ_DEV_BAD_BLOCK);
        mbar_arrive(&pfull[s]);
      }
    }
  };
  // Fused step: the team that owns a page holding new tokens (positions ctx - nq .. ctx - 1)
  // writes them before that page's copy is issued.  A page among the team's first copies is
  // written by the issuing warp before it issues them.  A later page (k >= DEPTH) is written
  // after the CTA's Q set-up, just before the page loop, by all NT warps of the team (warp nt
  // takes tokens nt, nt + NT, ...): each warp's stores and proxy fence precede its arrivals on
  // the empty barriers, and the issuing warp copies page k only after acquiring one of them.
  // The page loop has no write in it.
  auto write_team_pages = [&](bool first_batch) {
    if constexpr (WRITE && !PATCH) {
      if (!write_new) return;
      const int first_new = ctx - nq;
      const int lo_all = max(first_new, t_begin);
      if (lo_all >= t_end) return;
      for (int pr = (lo_all - t_begin) / KVQ_BLOCK_SIZE; pr < n_pages; ++pr) {
        if (pr % NTEAM != p || ((pr / NTEAM) < DEPTH) != first_batch) continue;
        const int tp = t_begin + pr * KVQ_BLOCK_SIZE;
        const int page = __ldg(bt + pr);
        const int lo = max(tp, first_new), hi = min(tp + KVQ_BLOCK_SIZE, t_end);
        const int w0 = first_batch ? 0 : nt, step = first_batch ? 1 : NT;
        if (page >= 0 && page < a.num_blocks && lo + w0 < hi)
          write_new_tokens<D>(a, b, kvh, nq, page, lo + w0, hi, step, first_new, lane);
      }
    }
  };
  // The first copies go out before Q is set up (its rows were requested first), so their HBM
  // latency overlaps the set-up.
  if (nt == 0) {
    write_team_pages(true);
    for (int k = 0; k < min(DEPTH, npp); ++k) issue(k);
  }

  // ---- Q^T fragments: row r = i * G + hh (query row i of the sequence, head hh of the
  // group) is prepared by warp r mod NW; rows past G * nq are zeros.  The fp16 values are
  // q * 2^e (e brings max|q| into [2^14, 2^15): exact for bf16).  Per n-tile of 8 rows,
  // chunk j (16 dims) is two 8 x 8 b16 matrices, rows = query rows, whose columns are the
  // k-slots of the MMA: slots (2c, 2c+1) carry dims (4c, 4c+1) and slots (2c+8, 2c+9) carry
  // dims (4c+2, 4c+3).
#pragma unroll
  for (int iq = 0; iq < kQPerWarp; ++iq) {
    const int h = warp + iq * NW;
    if (h >= L::kRows) break;
    uint8_t* q_tile = q_s + (h >> 3) * (D * 16);
    const int hr = h & 7;
    float x[PER];
    const uint32_t w4[4] = {qraw[iq].x, qraw[iq].y, qraw[iq].z, qraw[iq].w};
#pragma unroll
    for (int i = 0; i < PER / 2; ++i) {
      x[2 * i] = __uint_as_float(w4[i] << 16);
      x[2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    int e = amax > 0.f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127 : 0;
    e = max(-100, min(e, 127));
    const float qs = __uint_as_float(static_cast<uint32_t>(127 + 14 - e) << 23);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int d = lane * PER + i;
      const int j = d >> 4, w = d & 15, c = w >> 2, bb = w & 3;
      const int half = bb >> 1, el = 2 * c + (bb & 1);
      *reinterpret_cast<__half*>(q_tile + ((j * 2 + half) * 8 + hr) * 16 + el * 2) = __float2half_rn(x[i] * qs);
    }
    if (lane == 0) cq_s[h] = a.softmax_scale * kLog2e / qs;
  }
  __syncthreads();
  write_team_pages(false);
  // PATCH: the new token's codes and scales, kept for the shared-memory patch
  uint32_t kpk[PER / 4], vpk[PER / 4];
  float w_sk = 0.f, w_sv = 0.f;
  bool w_ok = false;
  if constexpr (PATCH) {
    if (k_w >= 0) {  // warp-uniform
      float xk[PER], xv[PER];
      {
        uint32_t wk[PER / 2], wv[PER / 2];
        if constexpr (PER == 8) {
          wk[0] = raw_k.x; wk[1] = raw_k.y; wk[2] = raw_k.z; wk[3] = raw_k.w;
          wv[0] = raw_v.x; wv[1] = raw_v.y; wv[2] = raw_v.z; wv[3] = raw_v.w;
        } else {
          wk[0] = raw_k.x; wk[1] = raw_k.y;
          wv[0] = raw_v.x; wv[1] = raw_v.y;
        }
#pragma unroll
        for (int i = 0; i < PER / 2; ++i) {
          xk[2 * i] = __uint_as_float(wk[i] << 16);
          xk[2 * i + 1] = __uint_as_float(wk[i] & 0xFFFF0000u);
          xv[2 * i] = __uint_as_float(wv[i] << 16);
          xv[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
        }
      }
      w_sk = quant_rule_warp_packed(xk, kpk);
      w_sv = quant_rule_warp_packed(xv, vpk);
      // the page: from the issuing window (page k <-> lane k) when it holds it
      const int page = (k_w < 32) ? __shfl_sync(0xffffffffu, pg, k_w) : __ldg(bt + pr_w);
      w_ok = page >= 0 && page < a.num_blocks;
      if (w_ok) {
        const long long ph = static_cast<long long>(page) * a.n_kv_heads + kvh;
        const int slot = (ctx - 1) % KVQ_BLOCK_SIZE;
        store_k_codes<D>(a.k, ph, slot, lane, kpk);
        store_v_codes<D>(a.v, ph, slot, lane, vpk);
        if (lane == 0) {
          a.k_scale[ph * KVQ_BLOCK_SIZE + slot] = w_sk;
          a.v_scale[ph * KVQ_BLOCK_SIZE + slot] = w_sv;
        }
      }
    }
  }


  const int g = lane >> 2, c = lane & 3;
  float o_acc[NMT_H][4];
#pragma unroll
  for (int i = 0; i < NMT_H; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
  float ms[2] = {-INFINITY, -INFINITY}, mz[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};
  const float cq0 = cq_s[nt * 8 + 2 * c], cq1 = cq_s[nt * 8 + 2 * c + 1];
  // key bound of this thread's two rows: row i of the sequence sees keys t < ctx - nq + 1 + i
  int lim[2] = {t_end, t_end};
  if constexpr (MROW) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = nt * 8 + 2 * c + i;
      if (r < R) lim[i] = min(t_end, ctx - nq + 1 + r / G);
    }
  }

  // per-lane ldmatrix offsets: K rows are tokens (in row_token order), Q^T rows are heads,
  // V rows are head dimensions
  const int mi = lane >> 3, r = lane & 7;
  const uint32_t k_lane_off = (mi >> 1) * 256 + row_token((mi & 1) * 8 + r) * 16;
  const uint32_t q_lane_off = static_cast<uint32_t>(smem_u32(q_s)) + nt * (D * 16) + mi * 128 + r * 16;
  const uint32_t v_lane_off = lane * 16;
  const int tk0 = row_token(g), tk1 = row_token(g + 8);
  const uint32_t selA = (c < 2) ? kSelB01 : kSelB23;
  const uint32_t selB = (c < 2) ? kSelB23 : kSelB01;

  int k_fail = npp;  // the page whose wait ran out (npp: none)
  for (int k = 0; k < npp; ++k) {
    const int s = k % DEPTH;
    const bool got = mbar_wait(&pfull[s], (k / DEPTH) & 1, a.status, a.wait_budget);
    uint8_t* st = pring + s * L::kStageBytes;
    if constexpr (PATCH) {
      if (k == k_w) {  // warp-uniform: the new token's slot of this copy gets its codes
        if (w_ok) {
          const int slot = (ctx - 1) % KVQ_BLOCK_SIZE, d0 = lane * PER;
          uint8_t* kd = st + ((d0 / 16) * KVQ_BLOCK_SIZE + slot) * 16 + (d0 % 16);
          if constexpr (PER == 8) *reinterpret_cast<uint2*>(kd) = make_uint2(kpk[0], kpk[1]);
          else *reinterpret_cast<uint32_t*>(kd) = kpk[0];
#pragma unroll
          for (int i = 0; i < PER; ++i)
            st[KB + (d0 + i) * KVQ_BLOCK_SIZE + slot] = static_cast<uint8_t>((vpk[i / 4] >> (8 * (i % 4))) & 0xFFu);
          if (lane == 0) {
            reinterpret_cast<float*>(st + 2 * KB)[slot] = w_sk;
            reinterpret_cast<float*>(st + 2 * KB + 64)[slot] = w_sv;
          }
          // a later copy into this slot comes after these generic writes
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
      }
    }
    const uint32_t kbase = smem_u32(st);
    const uint32_t vbase = kbase + KB;
    const float* sks = reinterpret_cast<const float*>(st + 2 * KB);
    const float* svs = reinterpret_cast<const float*>(st + 2 * KB + 64);

    // ---- S^T = K * Q^T over the head dimension
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int jj = 0; jj < NCH_H / 2; ++jj) {
      uint32_t r0, r1, r2, r3, a0, a1, a2, a3, q0, q1, q2, q3;
      ldsm_x4(kbase + jj * 512 + k_lane_off, r0, r1, r2, r3);
      ldsm_x4(q_lane_off + jj * 512, q0, q1, q2, q3);
      i8x4_to_h2x2(r0, kSelB01, kSelB23, a0, a2);
      i8x4_to_h2x2(r1, kSelB01, kSelB23, a1, a3);
      mma_f16_16816(sa, a0, a1, a2, a3, q0, q1);
      i8x4_to_h2x2(r2, kSelB01, kSelB23, a0, a2);
      i8x4_to_h2x2(r3, kSelB01, kSelB23, a1, a3);
      mma_f16_16816(sb, a0, a1, a2, a3, q2, q3);
    }
    if (!__all_sync(0xffffffffu, got)) {  // the warp leaves together
      k_fail = k;
      break;
    }
    const float S[4] = {sa[0] + sb[0], sa[1] + sb[1], sa[2] + sb[2], sa[3] + sb[3]};

    // ---- online softmax
    const bool page_ok = pok[s] != 0;
    const int tpage = t_begin + (p + k * NTEAM) * KVQ_BLOCK_SIZE;
    const int t0 = tpage + tk0, t1 = tpage + tk1;
    const bool v0 = page_ok && (t0 < t_end);
    const bool v1 = page_ok && (t1 < t_end);
    const float sk0 = sks[tk0], sk1 = sks[tk1];
    const float lv0 = v0 ? fast_log2(svs[tk0]) : -INFINITY;
    const float lv1 = v1 ? fast_log2(svs[tk1]) : -INFINITY;
    float w[2][2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float cqi = i ? cq1 : cq0;
      const float s0 = (v0 && (!MROW || t0 < lim[i])) ? S[i] * sk0 * cqi : -INFINITY;
      const float s1 = (v1 && (!MROW || t1 < lim[i])) ? S[2 + i] * sk1 * cqi : -INFINITY;
      const float z0 = s0 + lv0, z1 = s1 + lv1;
      float tms = fmaxf(s0, s1), tmz = fmaxf(z0, z1);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        tms = fmaxf(tms, __shfl_xor_sync(0xffffffffu, tms, off));
        tmz = fmaxf(tmz, __shfl_xor_sync(0xffffffffu, tmz, off));
      }
      // lazy references: move them only when the tile exceeds them by 2^8
      if (tms > ms[i] + kLazyRescale) {
        lsum[i] *= (ms[i] == -INFINITY) ? 0.f : fast_exp2(ms[i] - tms);
        ms[i] = tms;
      }
      if (tmz > mz[i] + kLazyRescale) {
        const float az = (mz[i] == -INFINITY) ? 0.f : fast_exp2(mz[i] - tmz);
#pragma unroll
        for (int mt = 0; mt < NMT_H; ++mt) {
          o_acc[mt][i] *= az;
          o_acc[mt][2 + i] *= az;
        }
        mz[i] = tmz;
      }
      const float msr = (ms[i] == -INFINITY) ? 0.f : ms[i];
      const float mzr = (mz[i] == -INFINITY) ? 0.f : mz[i];
      lsum[i] += fast_exp2(s0 - msr) + fast_exp2(s1 - msr);
      w[0][i] = fast_exp2(z0 - mzr);
      w[1][i] = fast_exp2(z1 - mzr);
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

    // ---- O^T += V^T * W over the head dimension
#pragma unroll
    for (int gg = 0; gg < NMT_H / 2; ++gg) {
      uint32_t r0, r1, r2, r3, a0, a1, a2, a3;
      ldsm_x4(vbase + v_lane_off + gg * 512, r0, r1, r2, r3);
      i8x4_to_h2x2(r0, selA, selB, a0, a2);
      i8x4_to_h2x2(r1, selA, selB, a1, a3);
      mma_f16_16816(o_acc[2 * gg], a0, a1, a2, a3, bh0, bh1);
      mma_f16_16816(o_acc[2 * gg], a0, a1, a2, a3, bl0, bl1);
      i8x4_to_h2x2(r2, selA, selB, a0, a2);
      i8x4_to_h2x2(r3, selA, selB, a1, a3);
      mma_f16_16816(o_acc[2 * gg + 1], a0, a1, a2, a3, bh0, bh1);
      mma_f16_16816(o_acc[2 * gg + 1], a0, a1, a2, a3, bl0, bl1);
    }
    // this page's slot is read: refill it with the team's page k + DEPTH
    __syncwarp();
    if constexpr (NT == 1) {
      if (k + DEPTH < npp) issue(k + DEPTH);
    } else {
      if (lane == 0) mbar_arrive(&pempty[s]);
      if (nt == 0 && k + DEPTH < npp) {
        // every warp of the team has read the slot (the (k / DEPTH)-th phase of its empty barrier)
        bool freed = true;
        if (lane == 0) freed = mbar_wait(&pempty[s], (k / DEPTH) & 1, a.status, a.wait_budget);
        if (__shfl_sync(0xffffffffu, freed ? 1 : 0, 0)) issue(k + DEPTH);
      }
    }
  }
  if (k_fail < npp) {
    // A wait ran out: the CTA's result is dropped (below).  The issuing warp first waits, again
    // with the budget, for the copies it issued past that page, so that none lands in shared
    // memory after the ring is reused or the CTA exits.
    if (lane == 0) {
      *cta_failed = 1;
      if (nt == 0)
        for (int kk = k_fail; kk < n_issued; ++kk) mbar_wait(&pfull[kk % DEPTH], (kk / DEPTH) & 1, a.status, a.wait_budget);
    }
    __syncwarp();
  }
  // l over all tokens of the warp for heads 2c, 2c + 1
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) lsum[i] += __shfl_xor_sync(0xffffffffu, lsum[i], off);
  }

  // ------------------------------------------------------------ merge the warps
  grid_dep_trigger();  // the stage-2 merge may start launching
  __syncthreads();  // every issued copy was waited for by its warp: the ring is free
  if (*cta_failed) {
    // a bounded wait ran out (KVQ_DEV_TIMEOUT is set): this range contributes nothing; the single
    // route writes zeros, a split writes an empty partial that the merge skips
    for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
      const int hh = idx / D, d = idx % D;
      const long long orow = MROW ? (static_cast<long long>(b) * nq + hh / G) * Hq + kvh * G + hh % G
                                  : static_cast<long long>(b) * Hq + kvh * G + hh;
      if (SPLIT) {
        const long long pu = orow * a.n_split + blockIdx.x;
        a.part_acc[pu * D + d] = 0.0f;
        if (d == 0) {
          a.part_stats[pu * 4 + 0] = -INFINITY;
          a.part_stats[pu * 4 + 1] = -INFINITY;
          a.part_stats[pu * 4 + 2] = 0.0f;
          a.part_stats[pu * 4 + 3] = 0.0f;
        }
      } else {
        a.out[orow * D + d] = 0.0f;
      }
    }
    return;
  }
  constexpr int RS = D + 4;                                     // padded row: no bank conflicts
  // slot of (team, row r) = team * 8 NT + r = warp * 8 + (r mod 8) for the warp holding r
  float* mo = reinterpret_cast<float*>(smem);                   // [NW][8][RS]
  float* mstat = mo + NW * 8 * RS;                              // [NW][8][4]
  float* mw = mstat + NW * 8 * 4;                               // [rows][NTEAM] weights of the teams' O
  float* mfin = mw + NW * 8;                                    // [rows][4]: Ms, Mz, l, final factor
#pragma unroll
  for (int mt = 0; mt < NMT_H; ++mt) {
    const int d0 = mt * 16 + g;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mo[(warp * 8 + 2 * c + i) * RS + d0] = o_acc[mt][i];
      mo[(warp * 8 + 2 * c + i) * RS + d0 + 8] = o_acc[mt][2 + i];
    }
  }
  if (g == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float* stt = mstat + (warp * 8 + 2 * c + i) * 4;
      stt[0] = ms[i];
      stt[1] = mz[i];
      stt[2] = lsum[i];
    }
  }
  __syncthreads();
  if (threadIdx.x < R) {
    // per row: the teams' maxima, the merged l and one weight per team (exp once per team)
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
    mfin[hh * 4 + 0] = Ms;
    mfin[hh * 4 + 1] = Mz;
    mfin[hh * 4 + 2] = lsum_all;
    mfin[hh * 4 + 3] = (lsum_all > 0.f && Mz != -INFINITY) ? fast_exp2(Mz - Ms) / lsum_all : 0.f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
    const int hh = idx / D, d = idx % D;
    float o = 0.f;
#pragma unroll
    for (int q2 = 0; q2 < NTEAM; ++q2) o = fmaf(mo[(q2 * L::kRows + hh) * RS + d], mw[hh * NTEAM + q2], o);
    // output row: query row hh / G of the sequence, query head kvh * G + hh % G
    const long long orow = MROW ? (static_cast<long long>(b) * nq + hh / G) * Hq + kvh * G + hh % G
                                : static_cast<long long>(b) * Hq + kvh * G + hh;
    if (SPLIT) {
      const long long pu = orow * a.n_split + blockIdx.x;
      a.part_acc[pu * D + d] = o;
      if (d == 0) {
        a.part_stats[pu * 4 + 0] = mfin[hh * 4 + 0];
        a.part_stats[pu * 4 + 1] = mfin[hh * 4 + 1];
        a.part_stats[pu * 4 + 2] = mfin[hh * 4 + 2];
        a.part_stats[pu * 4 + 3] = 0.f;
      }
    } else {
      a.out[orow * D + d] = o * mfin[hh * 4 + 3];
    }
  }
}

// The K/V stream of the stage-1 kernel alone (measurement entry point kvq_debug_stream_floor): the
// same grid, the same eight warps with their three-stage rings, the same bulk copies of the same
// pages in the same order, and no arithmetic.  Its duration is what streaming one launch's pages
// costs on this GPU by itself (launch, ramp-up and tail included), the floor of stage 1.
template <int D>
__global__ void __launch_bounds__(256, D == 128 ? 2 : 1) decode_stream_kernel(DecodeArgs a) {
  constexpr int NTEAM = 8, DEPTH = 3;
  using L = DecodeSmem<D, 1, NTEAM, DEPTH>;
  constexpr int KB = L::kKvBytes;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.y, b = blockIdx.z;
  grid_dep_wait();
  const int t_begin = static_cast<int>(blockIdx.x) * a.split_rows;
  const int32_t* bt = a.block_table + static_cast<long long>(b) * a.max_blocks_per_seq + t_begin / KVQ_BLOCK_SIZE;
  int pg = -1;
  if (t_begin / KVQ_BLOCK_SIZE + warp + lane * NTEAM < a.max_blocks_per_seq) pg = __ldg(bt + warp + lane * NTEAM);
  const int ctx = max(0, min(a.ctx_lens[b], min(a.max_blocks_per_seq * KVQ_BLOCK_SIZE, a.max_ctx)));
  const int t_end = min(ctx, t_begin + a.split_rows);
  const int n_pages = (t_end > t_begin) ? (t_end - t_begin + KVQ_BLOCK_SIZE - 1) / KVQ_BLOCK_SIZE : 0;
  if (n_pages == 0) return;
  if (threadIdx.x == 0) {
    for (int st = 0; st < L::kStages; ++st) mbar_init(&full[st], 1);
    mbar_fence_init();
  }
  __syncthreads();
  const int npp = (warp < n_pages) ? (n_pages - warp + NTEAM - 1) / NTEAM : 0;
  uint64_t* pfull = full + warp * DEPTH;
  uint8_t* pring = smem + warp * DEPTH * L::kStageBytes;
  if (lane >= npp) pg = -1;
  int wb = 0, n_issued = 0;
  auto issue = [&](int k) {
    while (k >= wb + 32) {
      wb += 32;
      pg = (wb + lane < npp) ? __ldg(bt + warp + (wb + lane) * NTEAM) : -1;
    }
    const int page = __shfl_sync(0xffffffffu, pg, k - wb);
    ++n_issued;
    if (lane == 0) {
      const int st = k % DEPTH;
      if (page >= 0 && page < a.num_blocks) {
        uint8_t* dst = pring + st * L::kStageBytes;
        const long long ph = static_cast<long long>(page) * a.n_kv_heads + kvh;
        mbar_arrive_expect_tx(&pfull[st], 2 * KB + 128);
        bulk_g2s(dst, a.k + ph * KB, KB, &pfull[st]);
        bulk_g2s(dst + KB, a.v + ph * KB, KB, &pfull[st]);
        bulk_g2s(dst + 2 * KB, a.k_scale + ph * KVQ_BLOCK_SIZE, 64, &pfull[st]);
        bulk_g2s(dst + 2 * KB + 64, a.v_scale + ph * KVQ_BLOCK_SIZE, 64, &pfull[st]);
      } else {
        set_status(a.status, KVQ_DEV_BAD_BLOCK);
        mbar_arrive(&pfull[st]);
      }
    }
  };
  for (int k = 0; k < min(DEPTH, npp); ++k) issue(k);
  for (int k = 0; k < npp; ++k) {
    const bool got = mbar_wait(&pfull[k % DEPTH], (k / DEPTH) & 1, a.status, a.wait_budget);
    if (!__all_sync(0xffffffffu, got)) {
      // the copies issued past this page land before the CTA exits
      if (lane == 0)
        for (int kk = k; kk < n_issued; ++kk) mbar_wait(&pfull[kk % DEPTH], (kk / DEPTH) & 1, a.status, a.wait_budget);
      __syncwarp();
      break;
    }
    if (k + DEPTH < npp) issue(k + DEPTH);
  }
}

cudaError_t launch_stream_floor(const DecodeArgs& a, cudaStream_t stream) {
  dim3 grid(a.n_split, a.n_kv_heads, a.batch);
  if (a.head_dim == 256) {
    using L = DecodeSmem<256, 1, 8, 3>;
    cudaError_t e = cudaFuncSetAttribute(decode_stream_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_stream_kernel<256>, grid, dim3(256), L::kTotal, stream, a);
  }
  using L = DecodeSmem<128, 1, 8, 3>;
  cudaError_t e = cudaFuncSetAttribute(decode_stream_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_stream_kernel<128>, grid, dim3(256), L::kTotal, stream, a);
}

// Stage 2: log-sum-exp merge of the splits of one (sequence, query row, query head).
//   M_s = max m_s, M_z = max m_z;  l = sum l_s 2^{m_s - M_s};  o = sum acc_s 2^{m_z - M_z};
//   out = o 2^{M_z - M_s} / l.  The per-split weights are computed once into shared memory
// ("ROCm/RDNA4 (gfx1201) vLLM ...", "The reduce is not free": one cooperative pass, each
// exponential once per split).  One CTA per (query head, sequence, 64-dim column block), so that
// a small batch still spreads over many SMs; 256 threads = 16 split groups x 16 threads of 4
// dims; each thread keeps 8 independent loads in flight.
constexpr int kMergeThreads = 256;
constexpr int kMergeCols = 64;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(DecodeArgs a) {
  constexpr int TPG = kMergeCols / 4;           // threads per split group (4 dims each)
  constexpr int NG = kMergeThreads / TPG;       // split groups
  constexpr int PRE = 8;                        // partials per thread loaded before the weights
  extern __shared__ float wts[];                // [n_split] weights of the partial accumulators
  __shared__ float red[2][kMergeThreads / 32];
  __shared__ __align__(16) float4 part[NG][TPG];
  // blockIdx.y = b * nq + i: query row i of sequence b
  const int h = blockIdx.x, row = blockIdx.y, b = row / a.nq, Hq = a.n_q_heads, col0 = blockIdx.z * kMergeCols;
  const long long pu0 = (static_cast<long long>(row) * Hq + h) * a.n_split;
  const float* stats = a.part_stats + pu0 * 4;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int grp = tid / TPG, dq = tid % TPG;
  const float4* acc = reinterpret_cast<const float4*>(a.part_acc + pu0 * D + col0) + dq;
  grid_dep_wait();  // the partials come from stage 1
  // The first PRE partials of this thread and its split's statistics are loaded together with
  // ctx, before the number of live splits is known: the reads stay inside the grid's n_split
  // slots, and slots past the live ones are never used.
  float4 v[PRE];
#pragma unroll
  for (int u = 0; u < PRE; ++u)
    if (grp + u * NG < a.n_split) v[u] = acc[static_cast<long long>(grp + u * NG) * (D / 4)];
  float4 st0 = make_float4(-INFINITY, -INFINITY, 0.f, 0.f);
  if (tid < a.n_split) st0 = reinterpret_cast<const float4*>(stats)[tid];
  int ctx = a.ctx_lens[b];
  ctx = max(0, min(ctx, min(a.max_blocks_per_seq * KVQ_BLOCK_SIZE, a.max_ctx)));
  const int n = min(a.n_split, (ctx + a.split_rows - 1) / a.split_rows);

  float Ms = tid < n ? st0.x : -INFINITY, Mz = tid < n ? st0.y : -INFINITY;
  for (int s = tid + kMergeThreads; s < n; s += kMergeThreads) {
    Ms = fmaxf(Ms, stats[s * 4 + 0]);
    Mz = fmaxf(Mz, stats[s * 4 + 1]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Ms = fmaxf(Ms, __shfl_xor_sync(0xffffffffu, Ms, off));
    Mz = fmaxf(Mz, __shfl_xor_sync(0xffffffffu, Mz, off));
  }
  if (lane == 0) {
    red[0][wid] = Ms;
    red[1][wid] = Mz;
  }
  __syncthreads();
  Ms = -INFINITY;
  Mz = -INFINITY;
#pragma unroll
  for (int i = 0; i < kMergeThreads / 32; ++i) {
    Ms = fmaxf(Ms, red[0][i]);
    Mz = fmaxf(Mz, red[1][i]);
  }
  float lpart = 0.f;
  for (int s = tid; s < n; s += kMergeThreads) {
    const float4 st = s == tid ? st0 : reinterpret_cast<const float4*>(stats)[s];
    wts[s] = (Mz != -INFINITY && st.y != -INFINITY) ? fast_exp2(st.y - Mz) : 0.f;
    lpart += (Ms != -INFINITY && st.x != -INFINITY) ? st.z * fast_exp2(st.x - Ms) : 0.f;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lpart += __shfl_xor_sync(0xffffffffu, lpart, off);
  __syncthreads();  // red[] and wts[] reuse
  if (lane == 0) red[0][wid] = lpart;
  __syncthreads();
  float l = 0.f;
#pragma unroll
  for (int i = 0; i < kMergeThreads / 32; ++i) l += red[0][i];

  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int u = 0; u < PRE; ++u) {
    const int s = grp + u * NG;
    if (s < n) {
      const float wgt = wts[s];
      o.x = fmaf(v[u].x, wgt, o.x);
      o.y = fmaf(v[u].y, wgt, o.y);
      o.z = fmaf(v[u].z, wgt, o.z);
      o.w = fmaf(v[u].w, wgt, o.w);
    }
  }
  int s = grp + PRE * NG;
  for (; s + 7 * NG < n; s += 8 * NG) {
    float4 w8[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) w8[u] = acc[static_cast<long long>(s + u * NG) * (D / 4)];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float wgt = wts[s + u * NG];
      o.x = fmaf(w8[u].x, wgt, o.x);
      o.y = fmaf(w8[u].y, wgt, o.y);
      o.z = fmaf(w8[u].z, wgt, o.z);
      o.w = fmaf(w8[u].w, wgt, o.w);
    }
  }
  for (; s < n; s += NG) {
    const float4 w1 = acc[static_cast<long long>(s) * (D / 4)];
    const float wgt = wts[s];
    o.x = fmaf(w1.x, wgt, o.x);
    o.y = fmaf(w1.y, wgt, o.y);
    o.z = fmaf(w1.z, wgt, o.z);
    o.w = fmaf(w1.w, wgt, o.w);
  }
  part[grp][dq] = o;
  __syncthreads();
  if (grp == 0) {
    float4 t = part[0][dq];
#pragma unroll
    for (int g2 = 1; g2 < NG; ++g2) {
      const float4 u = part[g2][dq];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    const float sc = (l > 0.f && Mz != -INFINITY) ? fast_exp2(Mz - Ms) / l : 0.f;
    reinterpret_cast<float4*>(a.out + (static_cast<long long>(row) * Hq + h) * D + col0)[dq] =
        make_float4(t.x * sc, t.y * sc, t.z * sc, t.w * sc);
  }
}

// Stage 2 for many (query row, head) units with few splits each (a large batch): one warp per
// unit, the splits' statistics in its lanes and their weights passed by shuffles, each lane
// combining D / 32 head dimensions of every split.  No shared memory and no block barrier, and
// a CTA of eight warps takes eight units, so the grid stays within a wave where the per-(unit,
// 64-dim block) CTAs of decode_merge_kernel would take several.  The same rule as that kernel.
constexpr int kMergeWarpMaxSplits = 32;

template <int D>
__global__ void __launch_bounds__(256) decode_merge_warp_kernel(DecodeArgs a) {
  constexpr int PER = D / 32;  // dims per lane
  const int lane = threadIdx.x & 31;
  const int Hq = a.n_q_heads;
  const long long unit = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);  // row * Hq + h
  grid_dep_wait();  // the partials come from stage 1
  if (unit >= static_cast<long long>(a.batch) * a.nq * Hq) return;  // warp-uniform
  const int row = static_cast<int>(unit / Hq), b = row / a.nq;
  int ctx = a.ctx_lens[b];
  ctx = max(0, min(ctx, min(a.max_blocks_per_seq * KVQ_BLOCK_SIZE, a.max_ctx)));
  const int n = min(a.n_split, (ctx + a.split_rows - 1) / a.split_rows);
  const long long pu0 = unit * a.n_split;
  float4 st = make_float4(-INFINITY, -INFINITY, 0.f, 0.f);
  if (lane < n) st = reinterpret_cast<const float4*>(a.part_stats)[pu0 + lane];
  float Ms = st.x, Mz = st.y;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Ms = fmaxf(Ms, __shfl_xor_sync(0xffffffffu, Ms, off));
    Mz = fmaxf(Mz, __shfl_xor_sync(0xffffffffu, Mz, off));
  }
  float l = (Ms != -INFINITY && st.x != -INFINITY) ? st.z * fast_exp2(st.x - Ms) : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  const float wgt = (Mz != -INFINITY && st.y != -INFINITY) ? fast_exp2(st.y - Mz) : 0.f;  // split `lane`
  float o[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) o[i] = 0.f;
  const float* acc = a.part_acc + pu0 * D + lane * PER;
  for (int s0 = 0; s0 < n; s0 += 8) {
    float4 v[8][PER / 4];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (s0 + u < n)
#pragma unroll
        for (int i = 0; i < PER / 4; ++i) v[u][i] = *reinterpret_cast<const float4*>(acc + static_cast<long long>(s0 + u) * D + 4 * i);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float w = __shfl_sync(0xffffffffu, wgt, (s0 + u) & 31);
      if (s0 + u < n)
#pragma unroll
        for (int i = 0; i < PER / 4; ++i) {
          o[4 * i + 0] = fmaf(v[u][i].x, w, o[4 * i + 0]);
          o[4 * i + 1] = fmaf(v[u][i].y, w, o[4 * i + 1]);
          o[4 * i + 2] = fmaf(v[u][i].z, w, o[4 * i + 2]);
          o[4 * i + 3] = fmaf(v[u][i].w, w, o[4 * i + 3]);
        }
    }
  }
  const float sc = (l > 0.f && Mz != -INFINITY) ? fast_exp2(Mz - Ms) / l : 0.f;
  float* dst = a.out + unit * D + lane * PER;
#pragma unroll
  for (int i = 0; i < PER / 4; ++i)
    *reinterpret_cast<float4*>(dst + 4 * i) = make_float4(o[4 * i] * sc, o[4 * i + 1] * sc, o[4 * i + 2] * sc, o[4 * i + 3] * sc);
}

size_t decode_workspace_bytes(int batch, int n_q_heads, int max_ctx, int head_dim, int split_rows) {
  const long long n_split = (static_cast<long long>(max_ctx) + split_rows - 1) / split_rows;
  const long long units = static_cast<long long>(batch) * n_q_heads * n_split;
  const long long acc = units * head_dim * 4;
  const long long stats = units * 4 * 4;
  return static_cast<size_t>(((acc + 255) / 256) * 256 + stats);
}

template <int D, int NT, bool SPLIT, bool MROW = true, bool WRITE = true>
static cudaError_t launch_stage1(const DecodeArgs& a, dim3 grid, cudaStream_t stream) {
  // One n-tile: 8 single-warp teams x 3 stages.  More rows: up to 16 warps in as many teams
  // as fit (pages in flight per SM), each ring 24 / NTEAM deep.
  constexpr int NTEAM = NT == 1 ? 8 : 16 / NT;
  constexpr int DEPTH = 24 / NTEAM;
  using L = DecodeSmem<D, NT, NTEAM, DEPTH>;
  auto kern = decode_stage1_kernel<D, NT, NTEAM, DEPTH, SPLIT, MROW, WRITE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
  if (e != cudaSuccess) return e;
  if (a.ev_begin && (e = cudaEventRecord(a.ev_begin, stream)) != cudaSuccess) return e;
  if ((e = launch_pdl(kern, grid, dim3(L::kWarps * 32), L::kTotal, stream, a)) != cudaSuccess) return e;
  if (a.ev_end && (e = cudaEventRecord(a.ev_end, stream)) != cudaSuccess) return e;
  return cudaSuccess;
}

template <int D, bool SPLIT>
static cudaError_t launch_stage1_rows(const DecodeArgs& a, dim3 grid, cudaStream_t stream) {
  if (a.nq == 1 && a.n_q_heads / a.n_kv_heads <= 8) {  // plain decode, or the fused one-token step
    if (a.k_new) return launch_stage1<D, 1, SPLIT, false, true>(a, grid, stream);
    return launch_stage1<D, 1, SPLIT, false, false>(a, grid, stream);
  }
  const int rows = (a.n_q_heads / a.n_kv_heads) * a.nq;
  switch ((rows + 7) / 8) {
    case 1: return launch_stage1<D, 1, SPLIT>(a, grid, stream);
    case 2: return launch_stage1<D, 2, SPLIT>(a, grid, stream);
    case 3: return launch_stage1<D, 3, SPLIT>(a, grid, stream);
    case 4: return launch_stage1<D, 4, SPLIT>(a, grid, stream);
    case 5: return launch_stage1<D, 5, SPLIT>(a, grid, stream);
    case 6: return launch_stage1<D, 6, SPLIT>(a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(const DecodeArgs& a, DecodeRoute route, cudaStream_t stream, int* launched) {
  *launched = route == DecodeRoute::kSingle ? 1 : 2;
  if (route == DecodeRoute::kSingle) {
    dim3 grid(1, a.n_kv_heads, a.batch);
    if (a.head_dim == 256) return launch_stage1_rows<256, false>(a, grid, stream);
    return launch_stage1_rows<128, false>(a, grid, stream);
  }
  dim3 grid(a.n_split, a.n_kv_heads, a.batch);
  cudaError_t e;
  if (a.head_dim == 256)
    e = launch_stage1_rows<256, true>(a, grid, stream);
  else
    e = launch_stage1_rows<128, true>(a, grid, stream);
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>(a.batch) * a.nq * a.n_q_heads;
  if (a.n_split <= kMergeWarpMaxSplits && units >= 512) {
    // many units, few splits each: a warp per unit
    const dim3 gw(static_cast<unsigned>((units + 7) / 8));
    e = a.head_dim == 256 ? launch_pdl(decode_merge_warp_kernel<256>, gw, dim3(256), 0, stream, a)
                          : launch_pdl(decode_merge_warp_kernel<128>, gw, dim3(256), 0, stream, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  const size_t wbytes = static_cast<size_t>(a.n_split) * sizeof(float);
  dim3 g2(a.n_q_heads, a.batch * a.nq, a.head_dim / kMergeCols);
  if (a.head_dim == 256) {
    if (wbytes > 48 * 1024) {
      e = cudaFuncSetAttribute(decode_merge_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(wbytes));
      if (e != cudaSuccess) return e;
    }
    e = launch_pdl(decode_merge_kernel<256>, g2, dim3(kMergeThreads), wbytes, stream, a);
  } else {
    if (wbytes > 48 * 1024) {
      e = cudaFuncSetAttribute(decode_merge_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(wbytes));
      if (e != cudaSuccess) return e;
    }
    e = launch_pdl(decode_merge_kernel<128>, g2, dim3(kMergeThreads), wbytes, stream, a);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvq
