// quant_rule.cuh — the per-(token, head) absmax int8 rule on one row held by a warp, and the
// stores of a row's codes into the paged cache layout.  Shared by every kernel that writes
// the cache (kvq_quant_write, the fused RoPE producer, the fused decode step), so the codes
// and scales are the same bits whichever kernel writes them.
//
// Method: "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" §2.1 (amax = max|x|,
// scale = amax / 127, q = clamp(round(x / scale), -127, 127)) and §2.3 (K in 16-element
// head-dimension chunks with the tokens of a chunk adjacent, V token-contiguous per dimension).
// Scales are IEEE fp32 quotients (__fdiv_rn), codes the nearest-even rounding of the IEEE
// quotient x / scale (computed through a reciprocal where that provably gives the same code).
#pragma once

#include <cstdint>

#include "kvq_dev.cuh"

namespace kvq {

// P consecutive bf16 values of a row (this lane's elements) to fp32.  src 4 * P-byte aligned.
template <int P>
__device__ __forceinline__ void load_bf16_lane(const uint16_t* src, float (&x)[P]) {
  static_assert(P == 8 || P == 4, "head_dim 256 or 128 over 32 lanes");
  if constexpr (P == 8) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src));
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(src));
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

// The quantisation rule over the warp's row (32 lanes x P values): returns the row's scale and
// this lane's codes, four to a word (element 4w in the low byte of word w).  An all-zero row gives
// scale 0 and codes 0.
template <int P>
__device__ __forceinline__ float quant_rule_warp_packed(const float (&x)[P], uint32_t (&packed)[P / 4]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < P; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = __fdiv_rn(amax, 127.0f);
  if (amax == 0.0f) {  // the same in every lane
#pragma unroll
    for (int w = 0; w < P / 4; ++w) packed[w] = 0u;
    return scale;
  }
  // code = rint(RN(x / scale)), taken as c = rint(y) with y = RN(x * r) and r the hardware
  // reciprocal of scale (at most 1 ulp from 1 / scale).  y then lies within |x / scale| * 1.5 *
  // 2^-23 (< 2.3e-5, since |x / scale| <= 127 (1 + 2^-23)) of the exact quotient and RN(x / scale)
  // within 7.6e-6 of it, so c is the rule's code unless y is within 3.1e-5 of a half-integer.
  // c comes from the rounding sum s = RN(y + 1.5 * 2^23) (nearest, ties to even, for |y| < 2^22):
  // c = s - 1.5 * 2^23 exactly, and bits(s) = 0x4B400000 + c, whose low byte is the code.
  // t = y - c is exact (c is the integer nearest y), and |t| > 1/2 - 2^-14 marks the elements near
  // a half-integer with room to spare (it would still hold for an r 3 ulp off), and non-finite y
  // (where r overflows or the input is not finite); there the IEEE division decides, clamped.
  constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
  constexpr float kNearHalf = 0.49993896484375f;  // 1/2 - 2^-14
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(scale));
  bool exact_needed = false;
#pragma unroll
  for (int w = 0; w < P / 4; ++w) {
    uint32_t sb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float y = __fmul_rn(x[4 * w + j], r);
      const float sr = __fadd_rn(y, kRound);
      exact_needed |= !(fabsf(__fsub_rn(y, __fsub_rn(sr, kRound))) <= kNearHalf);  // false for NaN
      sb[j] = __float_as_uint(sr);
    }
    packed[w] = __byte_perm(__byte_perm(sb[0], sb[1], 0x0040u), __byte_perm(sb[2], sb[3], 0x0040u), 0x5410u);
  }
  if (__any_sync(0xffffffffu, exact_needed)) {
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const float y = __fmul_rn(x[i], r);
      if (!(fabsf(__fsub_rn(y, __fsub_rn(__fadd_rn(y, kRound), kRound))) <= kNearHalf)) {
        const float ce = fminf(fmaxf(rintf(__fdiv_rn(x[i], scale)), -127.0f), 127.0f);
        const uint32_t sh = 8u * (i % 4);
        packed[i / 4] = (packed[i / 4] & ~(0xFFu << sh)) | ((static_cast<uint32_t>(static_cast<int>(ce)) & 0xFFu) << sh);
      }
    }
  }
  return scale;
}

// K codes of one token into its slot: [page][head][d/16][slot][16].  Lane l's dims l*P .. l*P+P-1
// lie in chunk (l*P)/16 at byte (l*P)%16 of the 16-byte row.  ph = page * n_kv_heads + head.
template <int D>
__device__ __forceinline__ void store_k_codes(int8_t* k, long long ph, int slot, int lane,
                                              const uint32_t (&packed)[D / 128]) {
  constexpr int P = D / 32;
  const int d0 = lane * P;
  int8_t* dst = k + ((ph * (D / 16) + d0 / 16) * KVQ_BLOCK_SIZE + slot) * 16 + (d0 % 16);
  if constexpr (P == 8) *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  else *reinterpret_cast<uint32_t*>(dst) = packed[0];
}

// V codes of one token into its slot: [page][head][d][slot], one byte per dimension.
template <int D>
__device__ __forceinline__ void store_v_codes(int8_t* v, long long ph, int slot, int lane,
                                              const uint32_t (&packed)[D / 128]) {
  constexpr int P = D / 32;
  int8_t* dst = v + (ph * D + lane * P) * KVQ_BLOCK_SIZE + slot;
#pragma unroll
  for (int i = 0; i < P; ++i) dst[i * KVQ_BLOCK_SIZE] = static_cast<int8_t>(packed[i / 4] >> (8 * (i % 4)));
}

}  // namespace kvq
