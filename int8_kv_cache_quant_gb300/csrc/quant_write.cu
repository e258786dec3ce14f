// quant_write.cu — fused per-(token, KV head) absmax int8 quantisation of new K/V rows
// into the paged cache: codes and fp32 scale in one kernel.
//
// Method: "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" §2.1 (quantisation rule:
// amax = max|x|, scale = amax / 127, q = clamp(round(x / scale), -127, 127)), §2.2 (one
// producer kernel: quantise and write the paged cache and the scale, no bf16 write-back),
// §2.3 (K in 16-element head-dimension chunks with the tokens of a chunk adjacent, V
// token-contiguous per dimension).
//
// Mapping: one warp per (token, KV head, K|V) row.  The row (head_dim bf16 values) is read
// with one vector load per lane and quantised by the warp (quant_rule.cuh: warp-shuffle amax,
// IEEE fp32 divisions, round to nearest even), so the codes and scales are bit-identical to
// the reference rule.  K codes go out as 8- or 4-byte stores into the [chunk][slot][16] rows;
// V codes are one byte per dimension into [dim][slot].
#include <cuda_bf16.h>

#include "kvq_dev.cuh"
#include "kvq_launch.h"
#include "quant_rule.cuh"

namespace kvq {

template <int D>
__global__ void __launch_bounds__(256) quant_write_kernel(QuantWriteArgs a) {
  constexpr int kPerLane = D / 32;  // 8 (D = 256) or 4 (D = 128) values per lane
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int H = a.n_kv_heads;
  const long long n_rows = static_cast<long long>(a.n_tokens) * H * 2;
  if (row >= n_rows) return;
  const int is_v = static_cast<int>(row & 1);
  const long long th = row >> 1;
  const int tok = static_cast<int>(th / H);
  const int h = static_cast<int>(th % H);

  grid_dep_wait();     // the new rows may come from the previous kernel of the stream
  grid_dep_trigger();  // the attention kernel may start launching; it waits for this grid
  const int seq = a.seq_idx[tok];
  const int pos = a.pos[tok];
  if (seq < 0 || seq >= a.num_seqs) {
    if (lane == 0) set_status(a.status, KVQ_DEV_BAD_SEQ);
    return;
  }
  if (pos < 0 || pos / KVQ_BLOCK_SIZE >= a.max_blocks_per_seq) {
    if (lane == 0) set_status(a.status, KVQ_DEV_BAD_POS);
    return;
  }
  const int page = a.block_table[static_cast<long long>(seq) * a.max_blocks_per_seq + pos / KVQ_BLOCK_SIZE];
  if (page < 0 || page >= a.num_blocks) {
    if (lane == 0) set_status(a.status, KVQ_DEV_BAD_BLOCK);
    return;
  }
  const int slot = pos % KVQ_BLOCK_SIZE;

  const uint16_t* src = static_cast<const uint16_t*>(is_v ? a.v_new : a.k_new) +
                        (static_cast<long long>(tok) * H + h) * D + lane * kPerLane;
  float x[kPerLane];
  load_bf16_lane(src, x);
  int8_t q[kPerLane];
  const float scale = quant_rule_warp(x, q);

  const long long ph = static_cast<long long>(page) * H + h;
  if (!is_v) {
    uint32_t packed[kPerLane / 4];
    pack_codes(q, packed);
    store_k_codes<D>(a.k, ph, slot, lane, packed);
    if (lane == 0) a.k_scale[ph * KVQ_BLOCK_SIZE + slot] = scale;
  } else {
    store_v_codes<D>(a.v, ph, slot, lane, q);
    if (lane == 0) a.v_scale[ph * KVQ_BLOCK_SIZE + slot] = scale;
  }
}

cudaError_t launch_quant_write(const QuantWriteArgs& a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.n_tokens) * a.n_kv_heads * 2;
  const int warps_per_block = 8;
  const long long blocks = (rows + warps_per_block - 1) / warps_per_block;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (a.head_dim == 256) return launch_pdl(quant_write_kernel<256>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, a);
  return launch_pdl(quant_write_kernel<128>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, a);
}

// ============================================================================ fused producer
// "gfx936 ..." §2.2 (one producer kernel: read Q/K/V, apply RoPE to Q and K, reduce absmax,
// quantise, write the paged int8 K/V and scales, quantise Q once for the attention that
// follows).  The rotation is the rotate-half form over the first r = rotary_dim dims with the
// caller's table row cs = cos_sin[pos] (cos of the r/2 frequencies, then their sin):
//   dim i < r/2 (partner i + r/2):      out = fma(x_i, c_i, -(x_{i+r/2} * s_i))
//   dim i + r/2 (partner i):            out = fma(x_{i+r/2}, c_i, x_i * s_i)
// in fp32 with exactly these roundings, then the quantisation rule of quant_write_kernel on the
// fp32 row.  One warp per (token, row) with rows = the token's Hq query heads, then Hkv K heads,
// then Hkv V heads; lane l holds dims l*P .. l*P+P-1 (P = D/32), so the partner of a dim is the
// same element of lane l +- (r/2)/P (r/2 is a multiple of P).
template <int D>
__global__ void __launch_bounds__(256) rope_quant_write_kernel(RopeQuantArgs a) {
  constexpr int P = D / 32;
  const int lane = threadIdx.x & 31;
  const int Hq = a.q ? a.n_q_heads : 0, H = a.kv.n_kv_heads;
  const int rows_per_token = Hq + 2 * H;
  const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(a.kv.n_tokens) * rows_per_token) return;
  const int tok = static_cast<int>(row / rows_per_token);
  const int r = static_cast<int>(row % rows_per_token);
  const int kind = r < Hq ? 0 : (r < Hq + H ? 1 : 2);  // 0 Q, 1 K, 2 V
  const int h = kind == 0 ? r : (kind == 1 ? r - Hq : r - Hq - H);

  grid_dep_wait();     // the rows may come from the previous kernel of the stream
  grid_dep_trigger();  // the attention kernel may start launching; it waits for this grid
  const int p = a.kv.pos[tok];
  const bool pos_ok = p >= 0 && p < a.max_pos;

  const uint16_t* src = kind == 0 ? static_cast<const uint16_t*>(a.q) + (static_cast<long long>(tok) * Hq + h) * D
                        : static_cast<const uint16_t*>(kind == 1 ? a.kv.k_new : a.kv.v_new) +
                              (static_cast<long long>(tok) * H + h) * D;
  src += lane * P;
  float x[P];
  load_bf16_lane(src, x);
  // ---- RoPE (Q and K; the warp takes the branch together: kind is uniform)
  if (kind != 2 && pos_ok) {
    const int half = a.rotary_dim / 2, shift = half / P;
    const int d0 = lane * P;
    const bool first = d0 < half, rotated = d0 < a.rotary_dim;
    const int partner = rotated ? (first ? lane + shift : lane - shift) : lane;
    const float* cs = a.cos_sin + static_cast<long long>(p) * a.rotary_dim;
    const int fi = first ? d0 : d0 - half;  // frequency index of this lane's first dim
#pragma unroll
    for (int e = 0; e < P; ++e) {
      const float other = __shfl_sync(0xffffffffu, x[e], partner);
      if (rotated) {
        const float c = __ldg(cs + fi + e), sn = __ldg(cs + half + fi + e);
        x[e] = first ? __fmaf_rn(x[e], c, -__fmul_rn(other, sn)) : __fmaf_rn(x[e], c, __fmul_rn(other, sn));
      }
    }
  }
  if (!pos_ok) {
#pragma unroll
    for (int e = 0; e < P; ++e) x[e] = 0.0f;
  }
  // ---- the quantisation rule (as quant_write_kernel)
  int8_t qc[P];
  const float scale = quant_rule_warp(x, qc);
  uint32_t packed[P / 4];
  pack_codes(qc, packed);

  if (kind == 0) {
    const long long u = static_cast<long long>(tok) * Hq + h;
    if (a.q_codes) {
      int8_t* dst = a.q_codes + u * D + lane * P;
      if constexpr (P == 8) *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
      else *reinterpret_cast<uint32_t*>(dst) = packed[0];
    }
    if (a.q_scales && lane == 0) a.q_scales[u] = scale;
    if (a.q_rot) {
      uint32_t b[P / 2];
#pragma unroll
      for (int i = 0; i < P / 2; ++i) {
        const __nv_bfloat162 v2 = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        b[i] = *reinterpret_cast<const uint32_t*>(&v2);
      }
      uint16_t* dst = a.q_rot + u * D + lane * P;
      if constexpr (P == 8) *reinterpret_cast<uint4*>(dst) = make_uint4(b[0], b[1], b[2], b[3]);
      else *reinterpret_cast<uint2*>(dst) = make_uint2(b[0], b[1]);
    }
    return;
  }
  // ---- K or V row into the token's slot
  const int seq = a.kv.seq_idx[tok];
  if (!pos_ok || p / KVQ_BLOCK_SIZE >= a.kv.max_blocks_per_seq) {
    if (lane == 0) set_status(a.kv.status, KVQ_DEV_BAD_POS);
    return;
  }
  if (seq < 0 || seq >= a.kv.num_seqs) {
    if (lane == 0) set_status(a.kv.status, KVQ_DEV_BAD_SEQ);
    return;
  }
  const int page = a.kv.block_table[static_cast<long long>(seq) * a.kv.max_blocks_per_seq + p / KVQ_BLOCK_SIZE];
  if (page < 0 || page >= a.kv.num_blocks) {
    if (lane == 0) set_status(a.kv.status, KVQ_DEV_BAD_BLOCK);
    return;
  }
  const int slot = p % KVQ_BLOCK_SIZE;
  const long long ph = static_cast<long long>(page) * H + h;
  if (kind == 1) {
    store_k_codes<D>(a.kv.k, ph, slot, lane, packed);
    if (lane == 0) a.kv.k_scale[ph * KVQ_BLOCK_SIZE + slot] = scale;
  } else {
    store_v_codes<D>(a.kv.v, ph, slot, lane, qc);
    if (lane == 0) a.kv.v_scale[ph * KVQ_BLOCK_SIZE + slot] = scale;
  }
}

cudaError_t launch_rope_quant_write(const RopeQuantArgs& a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.kv.n_tokens) * ((a.q ? a.n_q_heads : 0) + 2 * a.kv.n_kv_heads);
  const long long blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (a.kv.head_dim == 256)
    return launch_pdl(rope_quant_write_kernel<256>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, a);
  return launch_pdl(rope_quant_write_kernel<128>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, a);
}

}  // namespace kvq
