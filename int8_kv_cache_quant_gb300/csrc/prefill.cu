// prefill.cu — chunked causal prefill over the int8 paged K/V cache (placeholder: the Q
// quantisation step only; the tensor-core attention kernel follows).
#include "kvq_dev.cuh"
#include "kvq_launch.h"

namespace kvq {

// Q quantisation per (token, query head): the kvq_quant_write rule applied to Q
// ("gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" §2.1, §2.2: the query is quantised
// once and reused).  One warp per row; IEEE fp32 divisions, round to nearest even.
template <int D>
__global__ void __launch_bounds__(256) q_quant_kernel(PrefillArgs a) {
  constexpr int kPerLane = D / 32;
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(a.n_tokens) * a.n_q_heads) return;
  const uint16_t* src = static_cast<const uint16_t*>(a.q) + row * D + lane * kPerLane;
  float x[kPerLane];
  if constexpr (kPerLane == 8) {
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
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = __fdiv_rn(amax, 127.0f);
  uint32_t packed[kPerLane / 4];
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    float c = 0.0f;
    if (amax != 0.0f) {
      c = rintf(__fdiv_rn(x[i], scale));
      c = fminf(fmaxf(c, -127.0f), 127.0f);
    }
    const uint32_t byte = static_cast<uint32_t>(static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(c))));
    if (i % 4 == 0) packed[i / 4] = 0;
    packed[i / 4] |= byte << (8 * (i % 4));
  }
  int8_t* dst = a.q_codes + row * D + lane * kPerLane;
  if constexpr (kPerLane == 8) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  }
  if (lane == 0 && a.q_scales) a.q_scales[row] = scale;
}

size_t prefill_workspace_bytes(int n_tokens, int n_q_heads, int head_dim) {
  const long long codes = static_cast<long long>(n_tokens) * n_q_heads * head_dim;
  const long long scales = static_cast<long long>(n_tokens) * n_q_heads * 4;
  return static_cast<size_t>(((codes + 255) / 256) * 256 + scales);
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

cudaError_t launch_prefill(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_prefill_qk_debug(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace kvq
