// prefill.cu — chunked causal prefill over the int8 paged K/V cache on the 5th-generation
// tensor cores.
//
// Method: "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" §3.2 (a non-first prefill
// chunk: INT8 Q, history and chunk K/V in one online softmax), §1.3 and the §3.3 fragment
// code (Score = MMA_int8(Q, K^T) * sQ * sK / sqrt(d); each token's sV folded into the softmax
// weight; the weights re-quantised per block with scale absmax / 127; Output += MMA_int8(P,
// V) * p_scale), §2.1 (Q quantised per (token, head) by the same absmax rule).
//
// GB300 design.
// * sm_103a has no tcgen05 kind::i8, so the int8 codes are widened to integer-valued fp16 and
//   the contractions use tcgen05.mma kind::f16 with fp32 accumulators in tensor memory.  This
//   is exact: every QK partial sum is an integer of magnitude at most 256 * 127 * 127 < 2^24,
//   every per-tile PV sum at most 128 * 127 * 127 < 2^24.
// * Three kernels per call, chained by programmatic dependent launch: Q codes (q_quant_kernel),
//   a pre-pass that widens each (KV head, 128-key tile) of the cache once into the exact byte
//   image of the attention kernel's shared-memory operands (kv_widen_kernel), and the attention
//   (prefill_tma_kernel).
// * Attention: one CTA per (128 query rows, query head), longest units first.  A producer lane
//   brings the widened K and V pieces through a ring of 16 KB shared-memory slots by bulk copy;
//   one MMA warp issues QK (A = Q, held in tensor memory as fp16 pairs, B = a K piece) into a
//   single S buffer, and PV (A = the P codes in shared memory, B = V pieces) into O in tensor
//   memory.  16 softmax warps, four threads per query row (each owns 32 keys of the tile and a
//   quarter of the O columns), load S into registers, free the S buffer, and run the online
//   softmax and the per-tile P re-quantisation.
// * Every P-code decision is taken in fp32 relative to the tile's own maximum score, with a
//   specified exp2 (exp2_det), so the codes of a tile depend on that tile alone and are
//   reproducible off the GPU; the running maximum only rescales the tile's P scale and sum.
// * A unit's key range may run as two CTAs (a lead and a tail segment); the segment that
//   finishes second merges the two partial results, in an order that does not depend on which
//   finished first.
#include <algorithm>
#include <functional>
#include <vector>

#include "kvq_dev.cuh"
#include "kvq_launch.h"
#include "quant_rule.cuh"
#include "tcgen05.cuh"

namespace kvq {

// ============================================================================ Q quantisation
// Per (token, query head): the kvq_quant_write rule applied to Q ("gfx936 ..." §2.1, §2.2:
// the query is quantised once and reused).  One warp per row, the shared rule of every cache
// writer (IEEE fp32 quotients, round to nearest even).
template <int D>
__global__ void __launch_bounds__(256) q_quant_kernel(PrefillArgs a) {
  constexpr int kPerLane = D / 32;
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(a.n_tokens) * a.n_q_heads) return;
  float x[kPerLane];
  load_bf16_lane(static_cast<const uint16_t*>(a.q) + row * D + lane * kPerLane, x);
  uint32_t packed[kPerLane / 4];
  const float scale = quant_rule_warp_packed(x, packed);
  int8_t* dst = a.q_codes + row * D + lane * kPerLane;
  if constexpr (kPerLane == 8) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  }
  if (lane == 0 && a.q_scales) a.q_scales[row] = scale;
}

namespace {

constexpr float kLog2eP = 1.44269504088896341f;
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23

// Packed fp32 pairs (add / mul / fma .rn.f32x2): each lane is rounded exactly like the scalar
// operation, so these give the same bits as __fadd_rn / __fmul_rn / __fmaf_rn per element with
// half the instructions.
struct f2 {
  unsigned long long v;
};
__device__ __forceinline__ f2 mk2(float x, float y) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(x), "f"(y));
  return r;
}
// one half of a pair: the unpacking mov names both halves and the other one is dropped
#pragma nv_diag_suppress 550
__device__ __forceinline__ float lo2(f2 a) {
  float x, y;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(a.v));
  return x;
}
__device__ __forceinline__ float hi2(f2 a) {
  float x, y;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(a.v));
  return y;
}
#pragma nv_diag_default 550
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
  f2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}

// The specified exp2 of the P-code decisions (the same function, step for step, as the CPU
// reference): the argument clamped to [-125, 125] (fmaxf / fminf: NaN becomes -125), Cody-Waite
// reduction x = n + f with n = rint(x), 2^f by the degree-4 polynomial with constant term 1 whose
// other coefficients minimise the largest relative error of 2^f on [-1/2, 1/2] (2.82e-6; Horner,
// fp32 fma), times 2^n.
// Here on a pair, the same operations per element, for arguments x <= 0 up to one rounding (the
// attention kernels pass x = fma(y, a, -m) with m >= fl(ymax * a) >= fl(y * a) and a >= 0, so
// the clamp at +125 never acts and is left out): n = rint(x) through the 1.5 * 2^23 magic sum t,
// f = x - n (exact), the polynomial p in [0.70, 1.42], and p * 2^n as an exponent-field add: the
// product is normal for n in [-125, 0], so it equals bits(p) + n * 2^23, and n * 2^23 ==
// bits(t) * 2^23 (mod 2^32) because bits(t) = 0x4B400000 + n and 0x4B400000 * 2^23 == 0 (mod 2^32).
__device__ __forceinline__ f2 exp2_det2(f2 xin) {
  const f2 x = mk2(fmaxf(lo2(xin), -125.0f), fmaxf(hi2(xin), -125.0f));
  const f2 magic = mk2(kMagic, kMagic);
  const f2 t = add2(x, magic);
  const f2 n = sub2(t, magic);
  const f2 f = sub2(x, n);
  f2 p = fma2(mk2(0.00958285294f, 0.00958285294f), f, mk2(0.0559064262f, 0.0559064262f));
  p = fma2(p, f, mk2(0.240240991f, 0.240240991f));
  p = fma2(p, f, mk2(0.693124175f, 0.693124175f));
  p = fma2(p, f, mk2(1.0f, 1.0f));
  const uint32_t r0 = __float_as_uint(lo2(p)) + (__float_as_uint(lo2(t)) << 23);
  const uint32_t r1 = __float_as_uint(hi2(p)) + (__float_as_uint(hi2(t)) << 23);
  return mk2(__uint_as_float(r0), __uint_as_float(r1));
}

// 16 int8 codes (one int4) -> two 16-byte chunks of 8 fp16 (exact integer values).
__device__ __forceinline__ void widen16(const int4 raw, uint4& c0, uint4& c1) {
  uint32_t lo, hi;
  i8x4_to_h2x2(static_cast<uint32_t>(raw.x), kSelB01, kSelB23, lo, hi);
  c0.x = lo;
  c0.y = hi;
  i8x4_to_h2x2(static_cast<uint32_t>(raw.y), kSelB01, kSelB23, lo, hi);
  c0.z = lo;
  c0.w = hi;
  i8x4_to_h2x2(static_cast<uint32_t>(raw.z), kSelB01, kSelB23, lo, hi);
  c1.x = lo;
  c1.y = hi;
  i8x4_to_h2x2(static_cast<uint32_t>(raw.w), kSelB01, kSelB23, lo, hi);
  c1.z = lo;
  c1.w = hi;
}

__device__ __forceinline__ void sts128(uint8_t* p, const uint4& v) { *reinterpret_cast<uint4*>(p) = v; }

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t s = smem_u32(p);
  return p + (((s + 1023u) & ~1023u) - s);
}

}  // namespace

// ============================================================================ K/V widening pre-pass
// The attention kernel reads every K/V tile of its KV head once per (query tile, query head);
// widening the int8 codes to fp16 there would repeat the same work for every query head of the
// group and every query tile.  So one pass per prefill call widens each (KV head, 128-key tile)
// once, into the exact byte image of the attention kernel's shared-memory operands (128-byte
// swizzle, K-major), cut into 16 KB pieces that one bulk copy each brings in:
//   K tile: piece a (a < D/64) = head dims 64a .. 64a+63 of the 128 keys (rows = keys);
//   V tile: piece kh * (D/128) + dh = keys 64kh .. 64kh+63 (the K extent of the PV MMA) of head
//           dims 128dh .. 128dh+127 (rows = dims);
// plus the tile's key and value scales (fp32 [128] each).  Keys at or past the context, and keys
// on pages outside the pool, get zero codes and zero scales.
constexpr int kPieceBytes = 16384;

template <int D>
__global__ void __launch_bounds__(256) kv_widen_kernel(PrefillArgs a) {
  grid_dep_wait();  // the chunk's own K/V were written by the previous kernels of the stream
  const int j = blockIdx.x, kvh = blockIdx.y, tid = threadIdx.x;
  const int n_keys = a.history_len + a.n_tokens;
  __shared__ int page_s[8];
  if (tid < 8) {
    const int key0 = 128 * j + 16 * tid;
    int page = -1;
    if (key0 < n_keys) {
      const int bi = key0 / KVQ_BLOCK_SIZE;
      if (bi < a.n_blocks_row) page = a.block_table_row[bi];
      if (page < 0 || page >= a.num_blocks) {
        set_status(a.status, KVQ_DEV_BAD_BLOCK);
        page = -1;
      }
    }
    page_s[tid] = page;
  }
  if (a.split_tail > 0 && j == 0 && kvh == 0) {
    // the attention's split units meet through these counters: zero them before the trigger
    // below lets the attention grid read them
    const int n_units = ((a.n_tokens + 127) / 128) * a.n_q_heads;
    for (int u = tid; u < n_units; u += 256) {
      a.part_cnt[u] = 0u;
      a.part_ready[u] = 0u;
    }
  }
  __syncthreads();
  const long long tile = static_cast<long long>(kvh) * a.n_kv_tiles + j;
  uint8_t* kdst = a.kw + tile * (D / 64) * kPieceBytes;
  uint8_t* vdst = a.vw + tile * (D / 64) * kPieceBytes;
  // K: item i = (key n, 16-dim chunk c16); one key's chunk is 16 bytes of the
  // [page][head][D/16][slot][16] cache block.  The four chunks that fill one 128-byte row of a
  // piece (c16 = 4a .. 4a + 3 for key n) go to four adjacent lanes, so a warp's stores cover
  // whole rows (8 keys x 128 bytes) and its loads four 128-byte runs.
  for (int i = tid; i < 128 * (D / 16); i += 256) {
    const int n = (i >> 2) & 127, c16 = ((i >> 9) << 2) | (i & 3);
    const int page = page_s[n >> 4];
    int4 raw = make_int4(0, 0, 0, 0);
    if (page >= 0 && 128 * j + n < n_keys)
      raw = __ldg(reinterpret_cast<const int4*>(
          a.k + ((static_cast<long long>(page) * a.n_kv_heads + kvh) * (D / 16) + c16) * 256 + (n & 15) * 16));
    uint4 c0, c1;
    widen16(raw, c0, c1);
    uint8_t* piece = kdst + (c16 >> 2) * kPieceBytes;
    const int cc = (c16 & 3) * 2;
    sts128(piece + tc::sw128_off(n, cc), c0);  // global stores (same helper, generic address)
    sts128(piece + tc::sw128_off(n, cc + 1), c1);
  }
  // V: item i = (dim d, page pl); the 16 keys of page pl for dim d are 16 bytes of the
  // [page][head][D][slot] cache block.  The four pages that fill one 128-byte row of a piece
  // (pl = 4b .. 4b + 3 for dim d) go to four adjacent lanes.  Keys past the context carry
  // whatever the slot holds: their P codes are zero, and int8 codes are finite, so they add
  // nothing.
  for (int i = tid; i < 8 * D; i += 256) {
    const int pl = ((i / (4 * D)) << 2) | (i & 3), d = (i >> 2) % D;
    const int page = page_s[pl];
    int4 raw = make_int4(0, 0, 0, 0);
    if (page >= 0)
      raw = __ldg(reinterpret_cast<const int4*>(
          a.v + ((static_cast<long long>(page) * a.n_kv_heads + kvh) * D + d) * KVQ_BLOCK_SIZE));
    uint4 c0, c1;
    widen16(raw, c0, c1);
    uint8_t* piece = vdst + ((pl >> 2) * (D / 128) + (d >> 7)) * kPieceBytes;
    const int cc = (pl & 3) * 2;
    sts128(piece + tc::sw128_off(d & 127, cc), c0);
    sts128(piece + tc::sw128_off(d & 127, cc + 1), c1);
  }
  if (tid < 128) {
    const int n = tid, page = page_s[n >> 4];
    float sk = 0.0f, sv = 0.0f;
    if (page >= 0 && 128 * j + n < n_keys) {
      const long long idx = (static_cast<long long>(page) * a.n_kv_heads + kvh) * KVQ_BLOCK_SIZE + (n & 15);
      sk = a.k_scale[idx];
      sv = a.v_scale[idx];
    }
    a.skw[tile * 128 + n] = sk;
    a.svw[tile * 128 + n] = sv;
  }
  // Only now: an attention CTA made resident early would hold most of an SM's registers while
  // it waits for this grid.
  grid_dep_trigger();
}

// ============================================================================ first chunk (high precision)
// "gfx936 ..." §3.1: the first prefill chunk has no history to read; it runs the high-precision
// attention over its own bf16 Q/K/V while the producer writes its K/V as int8 for the chunks
// and decode steps that follow.  Here the same attention kernel runs on fp16 operands: a row x
// of Q, K or V becomes x * 2^(14 - e) with e the exponent of max |x| (so max |x| * 2^(14 - e) lies
// in [2^14, 2^15)), exact for every bf16 value within 2^29 of the row's maximum, and its scale
// is 2^(e - 14).  The int8 codes and the fp16 operands are made by one pass over the chunk.

// 2^(e - 14) and its inverse for a row maximum amax (1 for amax = 0), exponents clamped.
__device__ __forceinline__ void pow2_scales(float amax, float& to_f16, float& back) {
  int e = amax > 0.f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127 : 14;
  e = max(-100, min(e, 100));
  to_f16 = __uint_as_float(static_cast<uint32_t>(127 + 14 - e) << 23);
  back = __uint_as_float(static_cast<uint32_t>(127 + e - 14) << 23);
}

// P fp32 values (this lane's elements of a row) to fp16 after scaling, packed in pairs.
template <int P>
__device__ __forceinline__ void to_f16_pairs(const float (&x)[P], float s, uint32_t (&h)[P / 2]) {
#pragma unroll
  for (int e = 0; e < P / 2; ++e) h[e] = pack_half2(x[2 * e] * s, x[2 * e + 1] * s);
}

// Q rows to fp16 (one warp per (token, query head) row).
template <int D>
__global__ void __launch_bounds__(256) q_pack_f16_kernel(PrefillArgs a) {
  constexpr int P = D / 32;
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(a.n_tokens) * a.n_q_heads) return;
  grid_dep_wait();
  float x[P];
  load_bf16_lane(static_cast<const uint16_t*>(a.q) + row * D + lane * P, x);
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < P; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  float to_f16, back;
  pow2_scales(amax, to_f16, back);
  uint32_t hq[P / 2];
  to_f16_pairs(x, to_f16, hq);
  uint16_t* dst = a.q_f16 + row * D + lane * P;
  if constexpr (P == 8) *reinterpret_cast<uint4*>(dst) = make_uint4(hq[0], hq[1], hq[2], hq[3]);
  else *reinterpret_cast<uint2*>(dst) = make_uint2(hq[0], hq[1]);
  if (lane == 0) a.q_scales[row] = back;
}

// One CTA per (16 keys of the chunk's 128-key tiles, KV head), one warp per key t: its K and V
// rows are (1) quantised by the kvq_quant_write rule into the cache slot of position t (V codes
// staged so that a full page leaves in 16-byte stores), and (2) turned into fp16 with their
// power-of-two scales: K straight into row t % 128 of its tile's operand pieces, V through
// shared memory into the group's two 8-key chunks of each dimension row (rows = dims): the
// layout kv_widen_kernel writes.  Keys from the chunk's end to the end of its last tile get zero
// rows and zero scales (the attention multiplies masked keys' V by zero, so those rows must not
// hold stale NaN bits).
constexpr int kPackGroup = 16;

template <int D>
__global__ void __launch_bounds__(kPackGroup * 32) first_pack_kernel(PrefillArgs a) {
  constexpr int P = D / 32;
  __shared__ __align__(16) int8_t vq[kPackGroup][D];    // V codes for the cache
  __shared__ __align__(16) uint16_t vh[kPackGroup][D];  // V as fp16 for the pieces
  __shared__ long long tok_ph[kPackGroup];
  __shared__ int tok_slot[kPackGroup];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g0 = blockIdx.x * kPackGroup, kvh = blockIdx.y;
  const int T = a.n_tokens;
  const int j = g0 / 128;  // tile of this group
  const long long tile = static_cast<long long>(kvh) * a.n_kv_tiles + j;
  uint8_t* kdst = a.kw + tile * (D / 64) * kPieceBytes;
  uint8_t* vdst = a.vw + tile * (D / 64) * kPieceBytes;
  grid_dep_wait();  // Q packing and the chunk's rows come from the preceding kernels
  {
    const int k = warp, t = g0 + k, n = t % 128;
    float xk[P], xv[P];
    float sk = 0.f, sv = 0.f;
    long long ph = -1;
    int slot = 0;
    if (t < T) {
      const long long row = (static_cast<long long>(t) * a.n_kv_heads + kvh) * D + lane * P;
      load_bf16_lane(static_cast<const uint16_t*>(a.k_src) + row, xk);
      load_bf16_lane(static_cast<const uint16_t*>(a.v_src) + row, xv);
      // (1) the int8 cache write (the fused producer's part)
      const int bi = t / KVQ_BLOCK_SIZE;
      const int page = bi < a.n_blocks_row ? a.block_table_row[bi] : -1;
      if (page >= 0 && page < a.num_blocks) {
        ph = static_cast<long long>(page) * a.n_kv_heads + kvh;
        slot = t % KVQ_BLOCK_SIZE;
        uint32_t packed[P / 4];
        const float ck = quant_rule_warp_packed(xk, packed);
        store_k_codes<D>(a.k, ph, slot, lane, packed);
        const float cv = quant_rule_warp_packed(xv, packed);
        if constexpr (P == 8) *reinterpret_cast<uint2*>(&vq[k][lane * P]) = make_uint2(packed[0], packed[1]);
        else *reinterpret_cast<uint32_t*>(&vq[k][lane * P]) = packed[0];
        if (lane == 0) {
          a.k_scale[ph * KVQ_BLOCK_SIZE + slot] = ck;
          a.v_scale[ph * KVQ_BLOCK_SIZE + slot] = cv;
        }
      } else if (lane == 0) {
        set_status(a.status, KVQ_DEV_BAD_BLOCK);
      }
      // (2) fp16 operands
      float mk = 0.f, mv = 0.f;
#pragma unroll
      for (int e = 0; e < P; ++e) {
        mk = fmaxf(mk, fabsf(xk[e]));
        mv = fmaxf(mv, fabsf(xv[e]));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, off));
        mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, off));
      }
      float tk, tv;
      pow2_scales(mk, tk, sk);
      pow2_scales(mv, tv, sv);
#pragma unroll
      for (int e = 0; e < P; ++e) {
        xk[e] *= tk;
        xv[e] *= tv;
      }
    } else {
#pragma unroll
      for (int e = 0; e < P; ++e) xk[e] = xv[e] = 0.f;
    }
    if (lane == 0) {
      tok_ph[k] = ph;
      tok_slot[k] = slot;
    }
    uint32_t hk[P / 2], hv[P / 2];
    to_f16_pairs(xk, 1.0f, hk);
    to_f16_pairs(xv, 1.0f, hv);
    // K piece d / 64, row n, 16-byte chunk (d % 64) / 8 (this lane's P dims start at d = lane * P)
    const int d0 = lane * P;
    uint8_t* kp = kdst + (d0 / 64) * kPieceBytes + tc::sw128_off(n, (d0 % 64) / 8) + (d0 % 8) * 2;
    if constexpr (P == 8) *reinterpret_cast<uint4*>(kp) = make_uint4(hk[0], hk[1], hk[2], hk[3]);
    else *reinterpret_cast<uint2*>(kp) = make_uint2(hk[0], hk[1]);
    if constexpr (P == 8) *reinterpret_cast<uint4*>(&vh[k][d0]) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    else *reinterpret_cast<uint2*>(&vh[k][d0]) = make_uint2(hv[0], hv[1]);
    if (lane == 0) {
      a.skw[tile * 128 + n] = sk;
      a.svw[tile * 128 + n] = sv;
    }
  }
  __syncthreads();
  // V codes into the cache: one 16-byte store per dimension when the 16 keys fill a page in order
  bool full = true;
#pragma unroll
  for (int k = 0; k < kPackGroup; ++k) full = full && tok_ph[k] == tok_ph[0] && tok_slot[k] == k;
  full = full && tok_ph[0] >= 0;
  if (full) {
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
      uint32_t w[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        w[q4] = static_cast<uint32_t>(static_cast<uint8_t>(vq[4 * q4][d])) |
                (static_cast<uint32_t>(static_cast<uint8_t>(vq[4 * q4 + 1][d])) << 8) |
                (static_cast<uint32_t>(static_cast<uint8_t>(vq[4 * q4 + 2][d])) << 16) |
                (static_cast<uint32_t>(static_cast<uint8_t>(vq[4 * q4 + 3][d])) << 24);
      *reinterpret_cast<uint4*>(a.v + (tok_ph[0] * D + d) * KVQ_BLOCK_SIZE) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    for (int it = threadIdx.x; it < kPackGroup * D; it += blockDim.x) {
      const int k = it / D, d = it % D;
      const long long ph = tok_ph[k];
      if (ph >= 0) a.v[(ph * D + d) * KVQ_BLOCK_SIZE + tok_slot[k]] = vq[k][d];
    }
  }
  // V pieces: this group's keys are 8-key chunks c0 and c0 + 1 of key half kh; item = (dim, chunk)
  const int kh = (g0 % 128) / 64, c0 = (g0 % 64) / 8;
  for (int it = threadIdx.x; it < 2 * D; it += blockDim.x) {
    const int d = it >> 1, cc = it & 1;
    const int pc = kh * (D / 128) + d / 128;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = static_cast<uint32_t>(vh[8 * cc + 2 * e][d]) | (static_cast<uint32_t>(vh[8 * cc + 2 * e + 1][d]) << 16);
    *reinterpret_cast<uint4*>(vdst + pc * kPieceBytes + tc::sw128_off(d % 128, c0 + cc)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  grid_dep_trigger();
}

// ============================================================================ warp-specialised prefill
// One CTA per (128 query rows, query head), 18 warps:
//   warps 0-15  softmax: thread (row r, part p = warp / 4) owns keys 32p .. 32p+31 of row r's S
//               row and O columns p*D/4 .. (p+1)*D/4 - 1; the four parts of a row (warps w, w+4,
//               w+8, w+12: the same tensor-memory lanes) exchange their partial maxima through
//               shared memory at their own named barrier.  They also widen Q at the start.
//   warp 16     MMA issue and tensor-memory allocation: the whole warp runs the loop and one
//               elected lane issues, so the descriptors stay on the uniform datapath (the MMA
//               warp shares its SM sub-partition with four busy softmax warps; fewer instructions
//               per MMA keep the tensor pipe fed).  PV uses N = head_dim, one MMA per k-step.
//   warp 17     bulk-copy producer (lane 0): the widened K/V pieces through a ring of 16 KB
//               shared-memory slots in the order the MMAs consume them, and the scales.
// Tensor memory: S (128 columns) | Q (head_dim / 2 columns of fp16 pairs, the A operand of QK) |
// O (head_dim columns).  Q in tensor memory leaves QK reading only K from shared memory: with A
// and B both there a 128 x 128 x 16 MMA needs the whole shared-memory bandwidth, which the
// ring's bulk copies also use.  S is single-buffered: each softmax thread loads its S_j into
// registers and releases the buffer at once, so QK_{j+1} overlaps the rest of the tile's softmax.
// The P codes go to one of two shared-memory tiles (the A operand of PV).
// A P code c is stored as the fp16 bit pattern c, i.e. the subnormal c * 2^-24: its two bytes
// come straight from the rounding sum fma(w, r, 1.5 * 2^23), whose low byte is c.  The products
// c * v * 2^-24 and their sums are exact in fp32 (a power-of-two scaling of the integer sums), so
// O holds 2^-24 * sum_tiles (ps_tile / ps_ref) * PV_tile, and the epilogue multiplies by 2^24.
// Per tile j: MMA: QK_j (after s_free(j-1), pieces of K_j) -> commit s_full; then PV_{j-1} (after
// p_full, pieces of V_{j-1}, P tile (j-1) % 2) -> commit pv_done; every piece's slot is released
// by a commit after its MMAs.  Softmax: S_j after s_full and the scales -> arrive s_free; P_j
// (into P tile j % 2, last read by PV_{j-2}) and the O rescale after pv_done(j-1) -> arrive p_full.
namespace {

constexpr int kRingSlots = 8;  // one K tile and one V tile: keeps each V piece pair in adjacent slots
constexpr int kScaleBufs = 4;

template <int D>
struct PrefillTmaSmem {
  static constexpr int offP = 0;                                        // 2 P tiles [128 x 128] fp16
  static constexpr int kPBytes = 2 * kPieceBytes;                        // two 64-key atom columns
  static constexpr int offRing = offP + 2 * kPBytes;                    // kRingSlots pieces
  static constexpr int offScale = offRing + kRingSlots * kPieceBytes;   // [buf][k, v][128] fp32
  static constexpr int offRed = offScale + kScaleBufs * 2 * 128 * 4;    // [exchange][part][128]
  static constexpr int offBar = offRed + 2 * 4 * 128 * 4;
  static constexpr int kNumBars = 2 * kRingSlots + 2 * kScaleBufs + 6;
  static constexpr int offFlag = offBar + kNumBars * 8;                 // abort flag, TMEM base
  static constexpr int kBytes = offFlag + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTmemCols = 512;  // S | Q | O
  static constexpr uint32_t kQCol = 128;      // Q codes as fp16 pairs: D/2 columns
  static constexpr uint32_t kOCol = 256;
};

// mbarrier indices
constexpr int kBarFull = 0;                            // [kRingSlots] piece landed (tx)
constexpr int kBarEmpty = kBarFull + kRingSlots;       // [kRingSlots] piece consumed (commit)
constexpr int kBarSclFull = kBarEmpty + kRingSlots;    // [kScaleBufs] scales landed (tx)
constexpr int kBarSclFree = kBarSclFull + kScaleBufs;  // [kScaleBufs] scales read (softmax)
constexpr int kBarS0 = kBarSclFree + kScaleBufs;       // S_j complete (+0), S_j loaded by the softmax (+1)
constexpr int kBarPvDone = kBarS0 + 2;
constexpr int kBarPFull = kBarPvDone + 1;
constexpr int kBarQFull = kBarPFull + 1;
constexpr int kBarDrain = kBarQFull + 1;

constexpr int kSoftmaxThreads = 512;
constexpr int kMmaWarp = kSoftmaxThreads / 32;
constexpr int kPrefillThreads = kSoftmaxThreads + 64;

// Bounded wait that also gives up as soon as another thread of the CTA has given up.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, unsigned int* status,
                                              volatile int* abort_flag, long long budget) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) {
      set_status(status, KVQ_DEV_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ bool elect_one() {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r));
  return r != 0;
}

__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also returns the OR of `pred` over its `count` threads: every thread of
// the group takes the same decision.
__device__ __forceinline__ bool named_bar_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, %2, %3, q;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait for a flag that another CTA of the same grid sets.  The prefill waits only on a
// CTA that has already announced itself in its epilogue, so the flag comes within microseconds.
__device__ __forceinline__ void wait_flag(const unsigned int* flag, unsigned int* status, long long budget) {
  const long long t0 = clock64();
  while (ld_acquire_gpu(flag) == 0u) {
    if (clock64() - t0 > budget) {
      set_status(status, KVQ_DEV_TIMEOUT);
      return;
    }
    __nanosleep(64);
  }
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float max4_col(const float* p, int row) {
  return fmaxf(fmaxf(p[row], p[128 + row]), fmaxf(p[256 + row], p[384 + row]));
}

}  // namespace

// HP: the first chunk in high precision (fp16 Q with a power-of-two scale per row, the
// chunk's K/V as fp16 pieces with power-of-two scales per key, P as fp16 w / max w per tile)
// in place of the int8 Q, K/V and P codes; everything else is the same kernel.
// DBG (test entry point kvq_debug_prefill_qk_int32): the same int8 kernel, which also copies
// the raw integer scores S of the requested (query head, query tile, key window) out of tensor
// memory as each softmax thread loads them; nothing else changes.
template <int D, bool HP, bool DBG = false>
__global__ void __launch_bounds__(kPrefillThreads, 1) prefill_tma_kernel(PrefillArgs a) {
  using L = PrefillTmaSmem<D>;
  constexpr int OCOLS = D / 4;   // O columns per softmax thread
  constexpr int NP = D / 64;     // pieces per K tile and per V tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* ps_smem = sm + L::offP;
  uint8_t* ring = sm + L::offRing;
  float* scale_s = reinterpret_cast<float*>(sm + L::offScale);  // [buf][0: k, 1: v][128]
  float* red = reinterpret_cast<float*>(sm + L::offRed);        // [exchange][part][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::offBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::offFlag);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::offFlag + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // longest first: unit u takes query tile n_qt - 1 - u / Hq of head u % Hq, so the CTAs with the
  // most key tiles start in the first wave and the short ones fill the last.  With the key range
  // split, blocks [0, n_units) run the units' lead segments and blocks [n_units, 2 n_units) their
  // (short) tail segments, which fill the SMs the last wave of lead segments leaves idle.
  const int n_qt = (a.n_tokens + 127) / 128;
  const int n_units = n_qt * a.n_q_heads;
  const bool split = !HP && a.split_tail > 0;
  const bool tail_seg = split && static_cast<int>(blockIdx.x) >= n_units;
  const int unit = tail_seg ? static_cast<int>(blockIdx.x) - n_units : static_cast<int>(blockIdx.x);
  const int h = unit % a.n_q_heads;
  const int q0 = (n_qt - 1 - unit / a.n_q_heads) * 128;
  const int Hq = a.n_q_heads, G = Hq / a.n_kv_heads, kvh = h / G;
  const int T = a.n_tokens;
  const int n_keys = a.history_len + T;
  const int last_pos = a.history_len + min(q0 + 127, T - 1);
  // key tiles [j_begin, j_begin + nt) of this CTA.  The tail starts at a tile no later than the
  // last one inside the history, so its first tile holds a key that every row of the unit sees
  // (the running maximum starts finite in both segments); the host keeps js >= 1.
  int j_begin = 0, nt = last_pos / 128 + 1;
  if (split) {
    const int js = min(nt - a.split_tail, a.history_len / 128);
    if (tail_seg) {
      j_begin = js;
      nt -= js;
    } else {
      nt = js;
    }
  }
  // first tile of this head and segment: the producer's loads count from here, while the
  // barrier phases and buffers count the segment's own tiles from 0
  const long long tile0 = static_cast<long long>(kvh) * a.n_kv_tiles + j_begin;

  grid_dep_wait();  // Q codes, widened K/V and scales come from the preceding kernels
  if (warp == kMmaWarp) tc::tmem_alloc(tmem_slot, L::kTmemCols);
  if (tid == 0) {
    for (int s = 0; s < kRingSlots; ++s) {
      mbar_init(&bars[kBarFull + s], 1);
      mbar_init(&bars[kBarEmpty + s], 1);
    }
    for (int s = 0; s < kScaleBufs; ++s) {
      mbar_init(&bars[kBarSclFull + s], 1);
      mbar_init(&bars[kBarSclFree + s], kSoftmaxThreads);
    }
    mbar_init(&bars[kBarS0], 1);
    mbar_init(&bars[kBarS0 + 1], kSoftmaxThreads);
    mbar_init(&bars[kBarPvDone], 1);
    mbar_init(&bars[kBarPFull], kSoftmaxThreads);
    mbar_init(&bars[kBarQFull], kSoftmaxThreads);
    mbar_init(&bars[kBarDrain], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp < kMmaWarp) {
    // ================================================================ softmax warps
    const int row = tid & 127, part = tid >> 7;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int gbar = 1 + (warp & 3);  // named barrier of the four warps on these lanes
    const bool row_real = q0 + row < T;
    // the row's position and the key count, counted from this CTA's first key
    const int pos_r = a.history_len + q0 + row - 128 * j_begin;
    const int n_keys_seg = n_keys - 128 * j_begin;
    {
      // Q: this thread's D/4 dims of its row as fp16 pairs into tensor memory, the A operand of
      // QK (lane = row, dim d in column kQCol + d / 2, even dims in the low half): the int8
      // codes widened, or (HP) the fp16 row as it is
      uint32_t qw[D / 8];
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const int c16 = part * NP + i;
        uint4 c0, c1;
        if constexpr (HP) {
          const uint16_t* src_h = a.q_f16 + (static_cast<long long>(q0 + row) * Hq + h) * D;
          c0 = make_uint4(0, 0, 0, 0);
          c1 = make_uint4(0, 0, 0, 0);
          if (row_real) {
            c0 = __ldg(reinterpret_cast<const uint4*>(src_h + 16 * c16));
            c1 = __ldg(reinterpret_cast<const uint4*>(src_h + 16 * c16 + 8));
          }
        } else {
          const int8_t* src = a.q_codes + (static_cast<long long>(q0 + row) * Hq + h) * D;
          int4 raw = make_int4(0, 0, 0, 0);
          if (row_real) raw = __ldg(reinterpret_cast<const int4*>(src + 16 * c16));
          widen16(raw, c0, c1);
        }
        qw[8 * i + 0] = c0.x;
        qw[8 * i + 1] = c0.y;
        qw[8 * i + 2] = c0.z;
        qw[8 * i + 3] = c0.w;
        qw[8 * i + 4] = c1.x;
        qw[8 * i + 5] = c1.y;
        qw[8 * i + 6] = c1.z;
        qw[8 * i + 7] = c1.w;
      }
      if constexpr (D == 256) {
        tc::st_32x32b_x32(tmem + lane_base + L::kQCol + 32 * part, qw);
      } else {
        tc::st_32x32b_x16(tmem + lane_base + L::kQCol + 16 * part, qw);
      }
      tc::wait_st();
      tc::fence_before_sync();
      mbar_arrive(&bars[kBarQFull]);
    }
    const float c2 = __fmul_rn(a.softmax_scale, kLog2eP);
    const float a_row = row_real ? __fmul_rn(a.q_scales[static_cast<long long>(q0 + row) * Hq + h], c2) : 0.0f;
    float m = -INFINITY, l_part = 0.0f, ps_ref = 0.0f;
    bool started = false;
    const uint32_t tm_o = tmem + lane_base + L::kOCol + part * OCOLS;
    {
      uint32_t z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
      for (int c = 0; c < OCOLS / 32; ++c) tc::st_32x32b_x32(tm_o + 32 * c, z);
      tc::wait_st();
    }
    float* red_max = red;             // exchange 1: [part][row]
    float* red_wmax = red + 4 * 128;  // exchange 2
    bool failed = false;  // a wait of this thread gave up; the group leaves together below
    for (int j = 0; j < nt; ++j) {
      const int b = j & 1, sb = j & (kScaleBufs - 1);
      failed |= !wait_or_abort(&bars[kBarS0], j & 1, a.status, abort_flag, a.wait_budget);
      tc::fence_after_sync();
      uint32_t sv[32];
      tc::ld_32x32b_x32(tmem + lane_base + 32 * part, sv);
      failed |= !wait_or_abort(&bars[kBarSclFull + sb], (j / kScaleBufs) & 1, a.status, abort_flag, a.wait_budget);
      tc::wait_ld();
      if constexpr (DBG) {
        // this thread's 32 scores of key tile j_begin + j, when the tile lies in the window
        const int k_abs = 128 * (j_begin + j);
        if (h == a.dbg_q_head && q0 == a.dbg_q0 && k_abs >= a.dbg_k0 && k_abs < a.dbg_k0 + a.dbg_nk) {
          int32_t* dst = a.dbg_s_out + static_cast<long long>(row) * a.dbg_nk + (k_abs - a.dbg_k0) + 32 * part;
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<int4*>(dst + e) =
                make_int4(__float2int_rn(__uint_as_float(sv[e])), __float2int_rn(__uint_as_float(sv[e + 1])),
                          __float2int_rn(__uint_as_float(sv[e + 2])), __float2int_rn(__uint_as_float(sv[e + 3])));
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&bars[kBarS0 + 1]);  // S_j is in registers: the next QK may overwrite it
      const float4* sk_t = reinterpret_cast<const float4*>(scale_s + (sb * 2 + 0) * 128 + 32 * part);
      const float4* sv_t = reinterpret_cast<const float4*>(scale_s + (sb * 2 + 1) * 128 + 32 * part);
      // visible keys of this row in this tile, counted from the start of this thread's part
      const int lim = min(min(pos_r - 128 * j + 1, n_keys_seg - 128 * j), 128) - 32 * part;
      float ym0 = -INFINITY, ym1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 32; n += 4) {
        const float4 k4 = sk_t[n >> 2];
        const f2 ya = mul2(mk2(__uint_as_float(sv[n]), __uint_as_float(sv[n + 1])), mk2(k4.x, k4.y));
        const f2 yb = mul2(mk2(__uint_as_float(sv[n + 2]), __uint_as_float(sv[n + 3])), mk2(k4.z, k4.w));
        sv[n] = __float_as_uint(lo2(ya));
        sv[n + 1] = __float_as_uint(hi2(ya));
        sv[n + 2] = __float_as_uint(lo2(yb));
        sv[n + 3] = __float_as_uint(hi2(yb));
        ym0 = fmax3(ym0, lo2(ya), hi2(ya));
        ym1 = fmax3(ym1, lo2(yb), hi2(yb));
      }
      float ymax = fmaxf(ym0, ym1);
      if (lim < 32) {  // only tiles on the diagonal or past the context carry masked keys
        ymax = -INFINITY;
#pragma unroll
        for (int n = 0; n < 32; ++n) {
          const float y = (n < lim) ? __uint_as_float(sv[n]) : -INFINITY;
          sv[n] = __float_as_uint(y);
          ymax = fmaxf(ymax, y);
        }
      }
      red_max[part * 128 + row] = ymax;
      tc::fence_before_sync();
      if (named_bar_or(gbar, 128, failed)) break;  // the four parts of these rows leave together
      tc::fence_after_sync();
      // the tile's own maximum (fmaxf turns the NaN of a fully masked row times a zero a_row
      // into -inf) and the running maximum
      const float m_tile = fmaxf(__fmul_rn(max4_col(red_max, row), a_row), -INFINITY);
      const float m_new = fmaxf(m, m_tile);
      const float alpha = (m == -INFINITY) ? 0.0f : fast_exp2(m - m_new);
      // int8: p is taken relative to the tile's own maximum, so the P codes rint(127 w / max w)
      // are decided from the tile alone, whichever tiles came before it in this CTA (the key
      // range may be split between CTAs); beta = 2^(m_tile - m_new) moves the tile's P scale
      // and sum of p onto the running maximum.  The first-chunk path keeps p relative to the
      // running maximum (its P unit only grows).
      const float m_ref = HP ? m_new : m_tile;
      const float beta = HP ? 1.0f : (m_tile == -INFINITY ? 0.0f : fast_exp2(m_tile - m_new));
      f2 psum = mk2(0.0f, 0.0f);
      float wm0 = 0.0f, wm1 = 0.0f;
      const f2 a2 = mk2(a_row, a_row), nm2 = mk2(-m_ref, -m_ref);
      // p of the four keys n .. n+3, w = p * sV back into sv, and the running sums; masked keys
      // (only on tiles that carry them: the diagonal and past the context) get p = 0
      auto pass2_step = [&](int n, bool masked) {
        const float4 v4 = sv_t[n >> 2];
        f2 pa = exp2_det2(fma2(mk2(__uint_as_float(sv[n]), __uint_as_float(sv[n + 1])), a2, nm2));
        f2 pb = exp2_det2(fma2(mk2(__uint_as_float(sv[n + 2]), __uint_as_float(sv[n + 3])), a2, nm2));
        if (masked) {
          pa = mk2(n < lim ? lo2(pa) : 0.0f, n + 1 < lim ? hi2(pa) : 0.0f);
          pb = mk2(n + 2 < lim ? lo2(pb) : 0.0f, n + 3 < lim ? hi2(pb) : 0.0f);
        }
        psum = add2(psum, add2(pa, pb));
        const f2 wa = mul2(pa, mk2(v4.x, v4.y));
        const f2 wb = mul2(pb, mk2(v4.z, v4.w));
        sv[n] = __float_as_uint(lo2(wa));
        sv[n + 1] = __float_as_uint(hi2(wa));
        sv[n + 2] = __float_as_uint(lo2(wb));
        sv[n + 3] = __float_as_uint(hi2(wb));
        wm0 = fmax3(wm0, lo2(wa), hi2(wa));
        wm1 = fmax3(wm1, lo2(wb), hi2(wb));
      };
      if (lim < 32) {
#pragma unroll
        for (int n = 0; n < 32; n += 4) pass2_step(n, true);
      } else {
#pragma unroll
        for (int n = 0; n < 32; n += 4) pass2_step(n, false);
      }
      const float wmax = fmaxf(wm0, wm1);
      mbar_arrive(&bars[kBarSclFree + sb]);  // this tile's scales are no longer read
      l_part = l_part * alpha + (lo2(psum) + hi2(psum)) * beta;
      m = m_new;
      red_wmax[part * 128 + row] = wmax;
      tc::fence_before_sync();
      named_bar(gbar, 128);
      tc::fence_after_sync();
      const float wmax_row = max4_col(red_wmax, row);
      // reference scale of O and the factor that moves O onto this tile's P scale (the same
      // decisions in all four parts of the row)
      float f = 1.0f;
      bool codes_on = wmax_row > 0.0f;
      const float ps_new = HP ? wmax_row : __fdiv_rn(wmax_row, 127.0f) * beta;
      if constexpr (HP) {
        // fp16 P needs no per-tile unit: O's unit ps_ref only grows (to a tile whose largest
        // weight exceeds it), and a tile below it goes in as w / ps_ref <= 1, so O never grows.
        // ps_ref stays a normal number: it starts at a tile holding the running maximum (a
        // weight p * sV with p = 1), and it only decays (by alpha < 1) on a tile that holds a new
        // maximum, whose own weight then bounds it from below.
        if (!started) {
          if (codes_on) {
            started = true;
            ps_ref = wmax_row;
          }
        } else {
          const float dec = ps_ref * alpha;
          if (wmax_row > dec) {
            f = dec / wmax_row;
            ps_ref = wmax_row;
          } else {
            ps_ref = dec;
          }
        }
      } else if (!started) {
        if (codes_on) {
          started = true;
          ps_ref = ps_new;
        }
      } else if (codes_on) {
        const float fr = ps_ref * alpha / ps_new;
        if (fr > 1.8446744e19f) {  // 2^64: the tile is negligible against what O holds; drop it
          codes_on = false;
          ps_ref *= alpha;
        } else {
          f = fr;
          ps_ref = ps_new;
        }
      } else {
        ps_ref *= alpha;
      }
      uint32_t pk[16];
      if constexpr (HP) {
        // P = w / ps_ref in [0, 1] as fp16 (round to nearest), two per 32-bit column
        const float rr = (codes_on && ps_ref > 0.0f) ? __fdiv_rn(1.0f, ps_ref) : 0.0f;
        const f2 r2 = mk2(rr, rr);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const f2 c = mul2(mk2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), r2);
          pk[e] = pack_half2(lo2(c), hi2(c));
        }
      } else {
        // c = rint(w * r) with one rounding, as the low byte of fma(w, r, 1.5 * 2^23) (w <= wmax
        // keeps c in [0, 127]; r = 0 gives c = 0); two codes per 32-bit column
        const float rr = codes_on ? __fdiv_rn(127.0f, wmax_row) : 0.0f;
        const f2 r2 = mk2(rr, rr), mg = mk2(kMagic, kMagic);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const f2 c = fma2(mk2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), r2, mg);
          pk[e] = __byte_perm(__float_as_uint(lo2(c)), __float_as_uint(hi2(c)), 0x5410u);
        }
      }
      // O must hold PV_{j-1} before it is rescaled (and P_{j-1} must be consumed: it is)
      if (j > 0) {
        failed |= !wait_or_abort(&bars[kBarPvDone], (j - 1) & 1, a.status, abort_flag, a.wait_budget);
        tc::fence_after_sync();
      }
      {
        // P codes of keys 32 part .. 32 part + 31: four 16-byte chunks of row `row` in atom column
        // part / 2 of P buffer b (buffer b was last read by PV_{j-2}, complete by pv_done(j-1))
        uint8_t* pa = ps_smem + b * L::kPBytes + (part >> 1) * kPieceBytes;
        const int cb = (part & 1) * 4;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          sts128(pa + tc::sw128_off(row, cb + q4), make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]));
      }
      if (__any_sync(0xffffffffu, f != 1.0f)) {
        const f2 f2v = mk2(f, f);
#pragma unroll
        for (int c = 0; c < OCOLS / 32; ++c) {
          uint32_t o[32];
          tc::ld_32x32b_x32(tm_o + 32 * c, o);
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const f2 r = mul2(mk2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), f2v);
            o[e] = __float_as_uint(lo2(r));
            o[e + 1] = __float_as_uint(hi2(r));
          }
          tc::st_32x32b_x32(tm_o + 32 * c, o);
        }
      }
      tc::wait_st();
      tc::fence_proxy_async_smem();  // the P codes are read by the tensor core
      tc::fence_before_sync();
      mbar_arrive(&bars[kBarPFull]);
    }
    // ---- epilogue: out = O * 2^24 * ps_ref / l (l summed over the four parts; HP: no 2^24)
    if (!*abort_flag) {
      wait_or_abort(&bars[kBarPvDone], (nt - 1) & 1, a.status, abort_flag, a.wait_budget);
      tc::fence_after_sync();
    }
    red_max[part * 128 + row] = l_part;
    named_bar(gbar, 128);
    const float l = (red_max[row] + red_max[128 + row]) + (red_max[256 + row] + red_max[384 + row]);
    constexpr float kOUnit = HP ? 1.0f : 16777216.0f;  // the P codes' 2^-24 unit (int8 path)
    // The result tile goes out through shared memory: each thread puts its row's D/4 columns
    // into a staging tile (the P tiles and the ring, idle once the last PV is done; rows padded
    // by 16 bytes so that a warp's 32 rows hit distinct banks), then each warp copies whole rows
    // with 512-byte coalesced accesses.  Stored straight from registers, every warp store would
    // touch 32 rows a head-row stride apart.
    constexpr int kStageStride = D + 4;
    static_assert(128 * kStageStride * 4 <= L::offScale - L::offP, "the staging tile fits in the P tiles and the ring");
    float* stage = reinterpret_cast<float*>(sm + L::offP);
    float* my = stage + row * kStageStride + part * OCOLS;
    volatile unsigned int* bcast = reinterpret_cast<volatile unsigned int*>(sm + L::offFlag + 8);
    // After an abort the producer may still have copies landing in the ring: no staging then
    // (the status word already reports the failure).  One decision for all 512 threads.
    if (tid == 0) bcast[0] = *abort_flag ? 2u : (split ? atomicAdd(a.part_cnt + unit, 1u) : 0u);
    tc::fence_proxy_async_smem();  // the tensor core's reads of these bytes come before our writes
    named_bar(5, kSoftmaxThreads);
    const unsigned int decision = bcast[0];
    auto stage_o = [&](float scale) {
#pragma unroll
      for (int c = 0; c < OCOLS / 32; ++c) {
        uint32_t o[32];
        tc::ld_32x32b_x32(tm_o + 32 * c, o);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(my + 32 * c + e) =
              make_float4(__uint_as_float(o[e]) * scale, __uint_as_float(o[e + 1]) * scale,
                          __uint_as_float(o[e + 2]) * scale, __uint_as_float(o[e + 3]) * scale);
      }
    };
    // warp w moves staged rows 8w .. 8w + 7 (those below n_rows) to dst0 + row * dst_stride
    auto store_rows = [&](float* dst0, long long dst_stride, int n_rows) {
#pragma unroll 1
      for (int rr = 0; rr < 8; ++rr) {
        const int r = warp * 8 + rr;
        if (r < n_rows) {
          const float4* src = reinterpret_cast<const float4*>(stage + r * kStageStride);
          float4* dst = reinterpret_cast<float4*>(dst0 + r * dst_stride);
#pragma unroll
          for (int i = lane; i < D / 4; i += 32) dst[i] = src[i];
        }
      }
    };
    float* out0 = a.out + (static_cast<long long>(q0) * Hq + h) * D;
    const int n_real = min(128, T - q0);
    if (decision == 2u) {
      // aborted: nothing is written
    } else if (!split) {
      stage_o((started && l > 0.0f) ? ps_ref / l * kOUnit : 0.0f);
      named_bar(5, kSoftmaxThreads);
      store_rows(out0, static_cast<long long>(Hq) * D, n_real);
    } else if (decision == 0u) {
      // The unit's two segments meet here, and this one arrived first: it leaves its numerator
      // n = O * 2^24 * ps_ref and its (m, l) in the workspace and publishes them.
      const long long prow = static_cast<long long>(unit) * 128 + row;
      stage_o(started ? ps_ref * kOUnit : 0.0f);
      if (part == 0) {
        a.part_ml[2 * prow] = m;
        a.part_ml[2 * prow + 1] = l;
      }
      named_bar(5, kSoftmaxThreads);
      store_rows(a.part + static_cast<long long>(unit) * 128 * D, D, 128);
      __threadfence();
      named_bar(5, kSoftmaxThreads);
      if (tid == 0) {
        __threadfence();
        atomicExch(a.part_ready + unit, 1u);
      }
    } else {
      // The second segment: moves both numerators onto the larger maximum M (s = 2^(m - M)) and
      // writes out = (n_lead s_lead + n_tail s_tail) / (l_lead s_lead + l_tail s_tail).  The
      // terms are taken in lead, tail order whichever segment arrived second, and this segment's
      // own n is rounded exactly as the first one's was, so the result does not depend on the
      // order in which the two segments finished.
      const long long prow = static_cast<long long>(unit) * 128 + row;
      if (tid == 0) wait_flag(a.part_ready + unit, a.status, a.wait_budget);
      named_bar(5, kSoftmaxThreads);
      __threadfence();
#pragma unroll 1
      for (int rr = 0; rr < 8; ++rr) {  // the first segment's numerator rows, coalesced, into the stage
        const int r = warp * 8 + rr;
        const float4* src = reinterpret_cast<const float4*>(a.part + (static_cast<long long>(unit) * 128 + r) * D);
        float4* dst = reinterpret_cast<float4*>(stage + r * kStageStride);
#pragma unroll
        for (int i = lane; i < D / 4; i += 32) dst[i] = __ldcg(src + i);
      }
      const float m2 = __ldcg(a.part_ml + 2 * prow), l2 = __ldcg(a.part_ml + 2 * prow + 1);
      named_bar(5, kSoftmaxThreads);
      const float m_lead = tail_seg ? m2 : m, m_tail = tail_seg ? m : m2;
      const float l_lead = tail_seg ? l2 : l, l_tail = tail_seg ? l : l2;
      const float mx = fmaxf(m_lead, m_tail);
      const float s_lead = (m_lead == -INFINITY) ? 0.0f : exp2f(m_lead - mx);
      const float s_tail = (m_tail == -INFINITY) ? 0.0f : exp2f(m_tail - mx);
      const float lt = __fadd_rn(__fmul_rn(l_lead, s_lead), __fmul_rn(l_tail, s_tail));
      const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
      const float own = started ? ps_ref * kOUnit : 0.0f;
      auto comb = [&](float o_bits_f, float n_other) {
        const float n_own = __fmul_rn(o_bits_f, own);
        const float nl = tail_seg ? n_other : n_own, ntl = tail_seg ? n_own : n_other;
        return __fmul_rn(__fadd_rn(__fmul_rn(nl, s_lead), __fmul_rn(ntl, s_tail)), inv);
      };
#pragma unroll
      for (int c = 0; c < OCOLS / 32; ++c) {
        uint32_t o[32];
        tc::ld_32x32b_x32(tm_o + 32 * c, o);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float4* sp = reinterpret_cast<float4*>(my + 32 * c + e);
          const float4 n2 = *sp;
          *sp = make_float4(comb(__uint_as_float(o[e]), n2.x), comb(__uint_as_float(o[e + 1]), n2.y),
                            comb(__uint_as_float(o[e + 2]), n2.z), comb(__uint_as_float(o[e + 3]), n2.w));
        }
      }
      named_bar(5, kSoftmaxThreads);
      store_rows(out0, static_cast<long long>(Hq) * D, n_real);
    }
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issue (the whole warp
    // runs the loop, one elected lane issues): descriptors stay on the uniform datapath and a
    // piece's k-steps differ only in the start-address field (+32 bytes = +2 per step).
    const uint64_t pd0 = tc::sdesc_sw128(smem_u32(ps_smem)), rd0 = tc::sdesc_sw128(smem_u32(ring));
    constexpr uint32_t idesc = tc::idesc_f16_f32(128, 128);
    const uint32_t tm_o = tmem + L::kOCol;
    int slot = 0;
    uint32_t ph = 0;
    bool ok = __all_sync(0xffffffffu, wait_or_abort(&bars[kBarQFull], 0, a.status, abort_flag, a.wait_budget));
    for (int j = 0; ok && j <= nt; ++j) {
      if (j < nt) {
        // S is single-buffered: QK_j overwrites it once every softmax thread has loaded S_{j-1}
        if (j >= 1) ok = __all_sync(0xffffffffu, wait_or_abort(&bars[kBarS0 + 1], (j - 1) & 1, a.status, abort_flag, a.wait_budget));
        for (int qa = 0; ok && qa < NP; ++qa) {
          ok = __all_sync(0xffffffffu, wait_or_abort(&bars[kBarFull + slot], ph, a.status, abort_flag, a.wait_budget));
          if (!ok) break;
          if (elect_one()) {
            tc::fence_after_sync();
            const uint64_t kd = rd0 + static_cast<uint64_t>((slot * kPieceBytes) >> 4);
#pragma unroll
            for (int s = 0; s < 4; ++s)
              tc::mma_f16_ts(tmem, tmem + L::kQCol + 32 * qa + 8 * s, kd + 2 * s, idesc, (qa | s) ? 1u : 0u);
            tc::commit(&bars[kBarEmpty + slot]);
            if (qa == NP - 1) tc::commit(&bars[kBarS0]);
          }
          __syncwarp();
          if (++slot == kRingSlots) {
            slot = 0;
            ph ^= 1u;
          }
        }
      }
      if (ok && j >= 1) {
        // PV_{j-1}: for each 64-key half kh, the D/128 pieces of V rows (head dims) sit in adjacent
        // slots, so one N = D MMA per k-step covers all of O.
        const int jp = j - 1, bp = jp & 1;
        constexpr uint32_t idesc_pv = tc::idesc_f16_f32(128, D);
        ok = __all_sync(0xffffffffu, wait_or_abort(&bars[kBarPFull], jp & 1, a.status, abort_flag, a.wait_budget));
        for (int kh = 0; ok && kh < 2; ++kh) {
          const int s0 = slot;
          for (int dh = 0; ok && dh < D / 128; ++dh) {
            ok = __all_sync(0xffffffffu, wait_or_abort(&bars[kBarFull + slot], ph, a.status, abort_flag, a.wait_budget));
            if (++slot == kRingSlots) {
              slot = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          if (elect_one()) {
            tc::fence_after_sync();
            const uint64_t vd = rd0 + static_cast<uint64_t>((s0 * kPieceBytes) >> 4);
            const uint64_t pd = pd0 + static_cast<uint64_t>((bp * L::kPBytes + kh * kPieceBytes) >> 4);
#pragma unroll
            for (int s = 0; s < 4; ++s)
              tc::mma_f16_ss(tm_o, pd + 2 * s, vd + 2 * s, idesc_pv, 1u);
#pragma unroll
            for (int dh = 0; dh < D / 128; ++dh) tc::commit(&bars[kBarEmpty + s0 + dh]);
            if (kh == 1) tc::commit(&bars[kBarPvDone]);
          }
          __syncwarp();
        }
      }
    }
    // every MMA this warp issued has completed before the CTA releases tensor memory
    if (elect_one()) {
      tc::commit(&bars[kBarDrain]);
      mbar_wait(&bars[kBarDrain], 0, a.status, a.wait_budget);
    }
    __syncwarp();
  } else if (lane == 0) {
    // ================================================================ bulk-copy producer (one thread)
    int slot = 0, fills = 0;
    uint32_t ph = 0;
    bool ok = true;
    // test-only fault injection: CTA 0 leaves its fourth piece un-issued (no copy in flight, its
    // full barrier never completes), so the MMA warp's bounded wait on it runs out
    const bool skip_one = a.fault == 2 && blockIdx.x == 0;
    auto push = [&](const uint8_t* src) {
      if (fills >= kRingSlots && !wait_or_abort(&bars[kBarEmpty + slot], ph ^ 1u, a.status, abort_flag, a.wait_budget)) {
        ok = false;
        return;
      }
      if (!(skip_one && fills == 3)) {
        mbar_arrive_expect_tx(&bars[kBarFull + slot], kPieceBytes);
        bulk_g2s(ring + slot * kPieceBytes, src, kPieceBytes, &bars[kBarFull + slot]);
      }
      ++fills;
      if (++slot == kRingSlots) {
        slot = 0;
        ph ^= 1u;
      }
    };
    int scl_loads = 0;
    auto push_scales = [&](int j) {
      const int sb = j & (kScaleBufs - 1);
      if (j >= kScaleBufs &&
          !wait_or_abort(&bars[kBarSclFree + sb], ((j - kScaleBufs) / kScaleBufs) & 1, a.status, abort_flag, a.wait_budget)) {
        ok = false;
        return;
      }
      mbar_arrive_expect_tx(&bars[kBarSclFull + sb], 1024);
      bulk_g2s(scale_s + sb * 256, a.skw + (tile0 + j) * 128, 512, &bars[kBarSclFull + sb]);
      bulk_g2s(scale_s + sb * 256 + 128, a.svw + (tile0 + j) * 128, 512, &bars[kBarSclFull + sb]);
      ++scl_loads;
    };
    for (int j = 0; ok && j <= nt; ++j) {
      if (j < nt) {
        const uint8_t* kt = a.kw + (tile0 + j) * NP * kPieceBytes;
        for (int qa = 0; ok && qa < NP; ++qa) push(kt + qa * kPieceBytes);
        if (ok) push_scales(j);
      }
      if (j >= 1) {
        const uint8_t* vt = a.vw + (tile0 + j - 1) * NP * kPieceBytes;
        for (int qv = 0; ok && qv < NP; ++qv) push(vt + qv * kPieceBytes);
      }
    }
    // Copies still in flight (only after an abort) land before the CTA exits: wait for the
    // last fill of every slot and the last load of every scale buffer.
    for (int i = (fills > kRingSlots ? fills - kRingSlots : 0); i < fills; ++i)
      mbar_wait(&bars[kBarFull + i % kRingSlots], (i / kRingSlots) & 1, a.status, a.wait_budget);
    for (int i = (scl_loads > kScaleBufs ? scl_loads - kScaleBufs : 0); i < scl_loads; ++i)
      mbar_wait(&bars[kBarSclFull + i % kScaleBufs], (i / kScaleBufs) & 1, a.status, a.wait_budget);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, L::kTmemCols);
  }
}

// ============================================================================ launchers
// Workspace: int8 Q codes | Q scales | widened K tiles | widened V tiles | K scales | V scales,
// and for an int8 chunk with at least one full tile of history (whose key range may be split)
// the split units' numerators | (m, l) | arrival counters and ready flags (each part starting on
// a 1024-byte boundary of the workspace).
static long long round1k(long long x) { return (x + 1023) / 1024 * 1024; }

// Above this many units (128 query rows x one query head) the last wave is a small share of the
// call and the key range is never split, so no workspace is reserved for it either.
constexpr long long kMaxSplitUnits = 16384;

PrefillWorkspace prefill_workspace(int n_tokens, int n_q_heads, int n_kv_heads, int history_len, int head_dim,
                                   int q_elem_bytes) {
  PrefillWorkspace w{};
  w.n_kv_tiles = static_cast<int>((static_cast<long long>(history_len) + n_tokens + 127) / 128);
  const long long tiles = static_cast<long long>(n_kv_heads) * w.n_kv_tiles;
  w.off_q_scales = round1k(static_cast<long long>(n_tokens) * n_q_heads * head_dim * q_elem_bytes);
  w.off_kw = w.off_q_scales + round1k(static_cast<long long>(n_tokens) * n_q_heads * 4);
  w.off_vw = w.off_kw + tiles * 128 * head_dim * 2;
  w.off_skw = w.off_vw + tiles * 128 * head_dim * 2;
  w.off_svw = w.off_skw + tiles * 128 * 4;
  w.bytes = w.off_svw + tiles * 128 * 4;
  const long long units = static_cast<long long>((n_tokens + 127) / 128) * n_q_heads;
  w.can_split = q_elem_bytes == 1 && history_len >= 128 && units <= kMaxSplitUnits;
  if (w.can_split) {
    w.off_part = round1k(w.bytes);
    w.off_part_ml = w.off_part + round1k(units * 128 * head_dim * 4);
    w.off_part_flags = w.off_part_ml + round1k(units * 128 * 2 * 4);
    w.bytes = w.off_part_flags + units * 2 * 4;
  }
  return w;
}

// The split choice models the attention grid as list scheduling in block order onto one CTA
// slot per SM (the hardware hands the next block to the first SM that frees): a CTA costs its
// key tiles plus a fixed start-up and epilogue cost, and a split segment also pays for writing
// or reading the partial result.  Costs are in units of one key tile's time; the two constants
// were fitted to the measured call time of a 2048-query chunk after 30720 keys (24 query /
// 4 KV heads, head_dim 256) on 152 SMs at tail lengths 0, 16, 24, 32, 40, 48 and 64 tiles
// (within 0.5% at each), and agree with per-CTA timestamps (about 5 tiles of start-up and
// epilogue per CTA).
int prefill_split_tail(int n_tokens, int n_q_heads, int history_len, int n_sms) {
  if (n_tokens <= 0 || n_q_heads <= 0 || history_len < 128 || n_sms <= 0) return 0;
  const int n_qt = (n_tokens + 127) / 128;
  const long long units = static_cast<long long>(n_qt) * n_q_heads;
  if (units > kMaxSplitUnits) return 0;
  constexpr double kCtaCost = 6.0, kCombineCost = 1.0;
  const int h_tiles = history_len / 128;
  auto tiles_of = [&](int qt) { return (history_len + std::min(128 * qt + 127, n_tokens - 1)) / 128 + 1; };
  std::vector<double> slots;
  auto makespan = [&](int r) {
    slots.assign(static_cast<size_t>(n_sms), 0.0);  // a min-heap of the SMs' free times
    auto run = [&](double cost) {
      std::pop_heap(slots.begin(), slots.end(), std::greater<double>());
      slots.back() += cost;
      std::push_heap(slots.begin(), slots.end(), std::greater<double>());
    };
    for (int seg = 0; seg < (r > 0 ? 2 : 1); ++seg)
      for (long long u = 0; u < units; ++u) {
        const int n = tiles_of(n_qt - 1 - static_cast<int>(u / n_q_heads));
        const int js = std::min(n - r, h_tiles);
        const int len = r == 0 ? n : (seg == 0 ? js : n - js);
        run(len + kCtaCost + (r > 0 ? kCombineCost : 0.0));
      }
    return *std::max_element(slots.begin(), slots.end());
  };
  const int max_r = tiles_of(0) - 1;  // every lead segment keeps at least one tile
  double best = makespan(0);
  int best_r = 0;
  for (int r : {8, 16, 24, 32, 48, 64, 96, 128}) {
    if (r > max_r) break;
    const double m = makespan(r);
    if (m < best) {
      best = m;
      best_r = r;
    }
  }
  return best_r;
}

cudaError_t launch_prefill_q_quant(const PrefillArgs& a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.n_tokens) * a.n_q_heads;
  const long long blocks = (rows + 7) / 8;
  if (a.head_dim == 256)
    q_quant_kernel<256><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  else
    q_quant_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

template <int D, bool HP, bool DBG = false>
static cudaError_t launch_attention(const PrefillArgs& a, cudaStream_t stream) {
  using L = PrefillTmaSmem<D>;
  auto kern = prefill_tma_kernel<D, HP, DBG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid(((a.n_tokens + 127) / 128) * a.n_q_heads * (!HP && a.split_tail > 0 ? 2 : 1));
  return launch_pdl(kern, grid, dim3(kPrefillThreads), L::kAlloc, stream, a);
}

template <int D, bool DBG>
static cudaError_t launch_prefill_d(const PrefillArgs& a, cudaStream_t stream) {
  cudaError_t e = launch_pdl(kv_widen_kernel<D>, dim3(a.n_kv_tiles, a.n_kv_heads), dim3(256), 0, stream, a);
  if (e != cudaSuccess) return e;
  return launch_attention<D, false, DBG>(a, stream);
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  return a.head_dim == 256 ? launch_prefill_d<256, false>(a, stream) : launch_prefill_d<128, false>(a, stream);
}

cudaError_t launch_prefill_qk_debug(const PrefillArgs& a, cudaStream_t stream) {
  return a.head_dim == 256 ? launch_prefill_d<256, true>(a, stream) : launch_prefill_d<128, true>(a, stream);
}

template <int D>
static cudaError_t launch_prefill_first_d(const PrefillArgs& a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.n_tokens) * a.n_q_heads;
  cudaError_t e = launch_pdl(q_pack_f16_kernel<D>, dim3(static_cast<unsigned>((rows + 7) / 8)), dim3(256), 0, stream, a);
  if (e != cudaSuccess) return e;
  e = launch_pdl(first_pack_kernel<D>, dim3(a.n_kv_tiles * (128 / kPackGroup), a.n_kv_heads), dim3(kPackGroup * 32), 0,
                 stream, a);
  if (e != cudaSuccess) return e;
  return launch_attention<D, true>(a, stream);
}

cudaError_t launch_prefill_first(const PrefillArgs& a, cudaStream_t stream) {
  return a.head_dim == 256 ? launch_prefill_first_d<256>(a, stream) : launch_prefill_first_d<128>(a, stream);
}

}  // namespace kvq
