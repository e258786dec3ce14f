// quant_write.cu — fused per-(token, KV head) absmax int8 quantisation of new K/V rows
// into the paged cache: codes and fp32 scale in one kernel.
//
// Method: "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" §2.1 (quantisation rule:
// amax = max|x|, scale = amax / 127, q = clamp(round(x / scale), -127, 127)), §2.2 (one
// producer kernel: quantise and write the paged cache and the scale, no bf16 write-back),
// §2.3 (K in 16-element head-dimension chunks with the tokens of a chunk adjacent, V
// token-contiguous per dimension).
//
// Mapping: a block per (16 consecutive tokens, KV head), a warp per token row.  The row
// (head_dim bf16 values) is read with one vector load per lane and quantised by the warp
// (quant_rule.cuh: warp-shuffle amax, IEEE fp32 divisions, round to nearest even), so the codes
// and scales are bit-identical to the reference rule.  K codes go out as 8- or 4-byte stores
// into the [chunk][slot][16] rows; V codes go through shared memory so that a page filled by 16
// tokens of the block is written dim by dim in 16-byte stores.
#include <cuda_bf16.h>

#include "kvq_dev.cuh"
#include "kvq_launch.h"
#include "quant_rule.cuh"

namespace kvq {

// One block per (group of 16 consecutive input tokens, KV head); warp w quantises the K and V
// rows of token w of the group.  K codes go straight to their slots (8- or 4-byte
// stores into the [chunk][slot][16] rows).  V codes are staged in shared memory: when the 16
// tokens fill one page in slot order (a prefill chunk aligned to a page), each head dimension's
// 16 slots leave as one 16-byte store into the page's [dim][slot] block; otherwise (decode
// steps, scattered or unaligned tokens) each code leaves as a single byte, as its row dictates.
constexpr int kGroup = 16;

template <int D>
__global__ void __launch_bounds__(kGroup * 32) quant_write_kernel(QuantWriteArgs a) {
  constexpr int P = D / 32;  // 8 (D = 256) or 4 (D = 128) values per lane
  __shared__ __align__(16) int8_t vs[kGroup][D];
  __shared__ long long tok_ph[kGroup];  // page * n_kv_heads + head, -1: not written
  __shared__ int tok_slot[kGroup];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g0 = blockIdx.x * kGroup, h = blockIdx.y, H = a.n_kv_heads;

  grid_dep_wait();     // the new rows may come from the previous kernel of the stream
  grid_dep_trigger();  // the attention kernel may start launching; it waits for this grid
  {
    const int k = warp;  // one token per warp
    const int tok = g0 + k;
    long long ph = -1;
    int slot = 0;
    if (tok < a.n_tokens) {
      const int seq = a.seq_idx[tok];
      const int pos = a.pos[tok];
      if (seq < 0 || seq >= a.num_seqs) {
        if (lane == 0) set_status(a.status, KVQ_DEV_BAD_SEQ);
      } else if (pos < 0 || pos / KVQ_BLOCK_SIZE >= a.max_blocks_per_seq) {
        if (lane == 0) set_status(a.status, KVQ_DEV_BAD_POS);
      } else {
        const int page = a.block_table[static_cast<long long>(seq) * a.max_blocks_per_seq + pos / KVQ_BLOCK_SIZE];
        if (page < 0 || page >= a.num_blocks) {
          if (lane == 0) set_status(a.status, KVQ_DEV_BAD_BLOCK);
        } else {
          ph = static_cast<long long>(page) * H + h;
          slot = pos % KVQ_BLOCK_SIZE;
        }
      }
    }
    if (lane == 0) {
      tok_ph[k] = ph;
      tok_slot[k] = slot;
    }
    if (ph >= 0) {  // warp-uniform
      const long long row = (static_cast<long long>(tok) * H + h) * D + lane * P;
      float xk[P], xv[P];
      load_bf16_lane(static_cast<const uint16_t*>(a.k_new) + row, xk);
      load_bf16_lane(static_cast<const uint16_t*>(a.v_new) + row, xv);
      uint32_t packed[P / 4];
      const float sk = quant_rule_warp_packed(xk, packed);
      store_k_codes<D>(a.k, ph, slot, lane, packed);
      const float sv = quant_rule_warp_packed(xv, packed);
      if constexpr (P == 8) *reinterpret_cast<uint2*>(&vs[k][lane * P]) = make_uint2(packed[0], packed[1]);
      else *reinterpret_cast<uint32_t*>(&vs[k][lane * P]) = packed[0];
      if (lane == 0) {
        a.k_scale[ph * KVQ_BLOCK_SIZE + slot] = sk;
        a.v_scale[ph * KVQ_BLOCK_SIZE + slot] = sv;
      }
    }
  }
  __syncthreads();
  // one page in slot order?
  bool full = true;
#pragma unroll
  for (int k = 0; k < kGroup; ++k) full = full && tok_ph[k] == tok_ph[0] && tok_slot[k] == k;
  full = full && tok_ph[0] >= 0;
  if (full) {
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
      uint32_t w[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        w[q4] = static_cast<uint32_t>(static_cast<uint8_t>(vs[4 * q4][d])) |
                (static_cast<uint32_t>(static_cast<uint8_t>(vs[4 * q4 + 1][d])) << 8) |
                (static_cast<uint32_t>(static_cast<uint8_t>(vs[4 * q4 + 2][d])) << 16) |
                (static_cast<uint32_t>(static_cast<uint8_t>(vs[4 * q4 + 3][d])) << 24);
      *reinterpret_cast<uint4*>(a.v + (tok_ph[0] * D + d) * KVQ_BLOCK_SIZE) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    for (int it = threadIdx.x; it < kGroup * D; it += blockDim.x) {
      const int k = it / D, d = it % D;
      const long long ph = tok_ph[k];
      if (ph >= 0) a.v[(ph * D + d) * KVQ_BLOCK_SIZE + tok_slot[k]] = vs[k][d];
    }
  }
}

cudaError_t launch_quant_write(const QuantWriteArgs& a, cudaStream_t stream) {
  const long long groups = (static_cast<long long>(a.n_tokens) + kGroup - 1) / kGroup;
  if (groups > 0x7fffffffLL || a.n_kv_heads > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(groups), a.n_kv_heads);
  if (a.head_dim == 256) return launch_pdl(quant_write_kernel<256>, grid, dim3(kGroup * 32), 0, stream, a);
  return launch_pdl(quant_write_kernel<128>, grid, dim3(kGroup * 32), 0, stream, a);
}

// ============================================================================ fused producer
// "gfx936 ..." §2.2 (one producer kernel: read Q/K/V, apply RoPE to Q and K, reduce absmax,
// quantise, write the paged int8 K/V and scales, quantise Q once for the attention that
// follows).  The rotation is the rotate-half form over the first r = rotary_dim dims with the
// caller's table row cs = cos_sin[pos] (cos of the r/2 frequencies, then their sin):
//   dim i < r/2 (partner i + r/2):      out = fma(x_i, c_i, -(x_{i+r/2} * s_i))
//   dim i + r/2 (partner i):            out = fma(x_{i+r/2}, c_i, x_i * s_i)
// in fp32 with exactly these roundings, then the quantisation rule of quant_write_kernel on the
// fp32 row.  A warp per (token, K/V head), or per (token, group of q_heads_per_warp query heads);
// lane l holds dims l*P .. l*P+P-1 (P = D/32), so the partner of a dim is the same element of lane
// l +- (r/2)/P (r/2 is a multiple of P).
// The rotation of this lane's P elements of a Q or K row at position p (rotate-half form above).
template <int P>
__device__ __forceinline__ void rope_lane(float (&x)[P], const RopeQuantArgs& a, int p, int lane) {
  const int half = a.rotary_dim / 2, shift = half / P;
  const int d0 = lane * P;
  const bool first = d0 < half, rotated = d0 < a.rotary_dim;
  const int partner = rotated ? (first ? lane + shift : lane - shift) : lane;
  const float* cs = a.cos_sin + static_cast<long long>(p) * a.rotary_dim;
  const int fi = first ? d0 : d0 - half;  // frequency index of this lane's first dim
  // the table row is 16-byte aligned at every lane's first frequency (cos_sin is 16-byte aligned
  // and rotary_dim / 2 is a multiple of P, hence of 4)
#pragma unroll
  for (int i = 0; i < P / 4; ++i) {
    float o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = __shfl_sync(0xffffffffu, x[4 * i + j], partner);
    if (rotated) {
      // -(o * s) == o * (-s) exactly, so the sign goes onto the table value
      const float4 c4 = __ldg(reinterpret_cast<const float4*>(cs + fi) + i);
      float4 s4 = __ldg(reinterpret_cast<const float4*>(cs + half + fi) + i);
      if (first) s4 = make_float4(-s4.x, -s4.y, -s4.z, -s4.w);
      x[4 * i] = __fmaf_rn(x[4 * i], c4.x, __fmul_rn(o[0], s4.x));
      x[4 * i + 1] = __fmaf_rn(x[4 * i + 1], c4.y, __fmul_rn(o[1], s4.y));
      x[4 * i + 2] = __fmaf_rn(x[4 * i + 2], c4.z, __fmul_rn(o[2], s4.z));
      x[4 * i + 3] = __fmaf_rn(x[4 * i + 3], c4.w, __fmul_rn(o[3], s4.w));
    }
  }
}

// The query side: warp w of a block takes token g0 + w and the block's q_heads_per_warp query
// heads, loading its lane's table values once for all of them and each next row before it works on
// the current one.
template <int D>
__device__ __forceinline__ void rope_q_rows(const RopeQuantArgs& a, int tok, int h0, int lane) {
  constexpr int P = D / 32;
  const int Hq = a.n_q_heads;
  const int h1 = min(Hq, h0 + a.q_heads_per_warp);
  const int p = a.kv.pos[tok];
  const bool pos_ok = p >= 0 && p < a.max_pos;
  const int half = a.rotary_dim / 2, shift = half / P;
  const int d0 = lane * P;
  const bool first = d0 < half, rotated = d0 < a.rotary_dim;
  const int partner = rotated ? (first ? lane + shift : lane - shift) : lane;
  // cos and sin of this lane's dims; the sin carries the rotation's sign for the first half
  // (-(o * s) == o * (-s) exactly)
  float cf[P], sf[P];
  if (pos_ok && rotated) {
    const float* cs = a.cos_sin + static_cast<long long>(p) * a.rotary_dim + (first ? d0 : d0 - half);
#pragma unroll
    for (int i = 0; i < P / 4; ++i) {
      const float4 c4 = __ldg(reinterpret_cast<const float4*>(cs) + i);
      const float4 s4 = __ldg(reinterpret_cast<const float4*>(cs + half) + i);
      cf[4 * i] = c4.x;
      cf[4 * i + 1] = c4.y;
      cf[4 * i + 2] = c4.z;
      cf[4 * i + 3] = c4.w;
      sf[4 * i] = first ? -s4.x : s4.x;
      sf[4 * i + 1] = first ? -s4.y : s4.y;
      sf[4 * i + 2] = first ? -s4.z : s4.z;
      sf[4 * i + 3] = first ? -s4.w : s4.w;
    }
  }
  using Raw = typename std::conditional<P == 8, uint4, uint2>::type;
  const uint16_t* qrow = static_cast<const uint16_t*>(a.q) + static_cast<long long>(tok) * Hq * D + d0;
  Raw nxt = __ldg(reinterpret_cast<const Raw*>(qrow + h0 * D));
  for (int h = h0; h < h1; ++h) {
    const Raw raw = nxt;
    if (h + 1 < h1) nxt = __ldg(reinterpret_cast<const Raw*>(qrow + (h + 1) * D));
    float x[P];
    uint32_t w[P / 2];
    if constexpr (P == 8) {
      w[0] = raw.x; w[1] = raw.y; w[2] = raw.z; w[3] = raw.w;
    } else {
      w[0] = raw.x; w[1] = raw.y;
    }
#pragma unroll
    for (int i = 0; i < P / 2; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    // ---- rotate, quantise, codes + scale + rotated bf16 row
    if (pos_ok) {
      // the partner's element e is element e of lane `partner`: its bf16 pairs move as they are
#pragma unroll
      for (int i = 0; i < P / 2; ++i) {
        const uint32_t ow = __shfl_sync(0xffffffffu, w[i], partner);
        if (rotated) {
          x[2 * i] = __fmaf_rn(x[2 * i], cf[2 * i], __fmul_rn(__uint_as_float(ow << 16), sf[2 * i]));
          x[2 * i + 1] = __fmaf_rn(x[2 * i + 1], cf[2 * i + 1], __fmul_rn(__uint_as_float(ow & 0xFFFF0000u), sf[2 * i + 1]));
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < P; ++e) x[e] = 0.0f;
    }
    uint32_t packed[P / 4];
    const float scale = quant_rule_warp_packed(x, packed);
    const long long u = static_cast<long long>(tok) * Hq + h;
    if (a.q_codes) {
      int8_t* dst = a.q_codes + u * D + d0;
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
      uint16_t* dst = a.q_rot + u * D + d0;
      if constexpr (P == 8) *reinterpret_cast<uint4*>(dst) = make_uint4(b[0], b[1], b[2], b[3]);
      else *reinterpret_cast<uint2*>(dst) = make_uint2(b[0], b[1]);
    }
  }
}

// One block per (group of 16 consecutive tokens, slot r): r < n_qg is the query heads
// q_heads_per_warp * r .. (Q outputs), r >= n_qg is KV head r - n_qg (the K row rotated into its cache
// slot, the V row staged in shared memory and written page-wise as in quant_write_kernel).  Warp w
// takes token w.
template <int D>
__global__ void __launch_bounds__(kGroup * 32, 2) rope_quant_write_kernel(RopeQuantArgs a) {
  constexpr int P = D / 32;
  __shared__ __align__(16) int8_t vs[kGroup][D];
  __shared__ long long tok_ph[kGroup];
  __shared__ int tok_slot[kGroup];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qg = a.q ? (a.n_q_heads + a.q_heads_per_warp - 1) / a.q_heads_per_warp : 0, H = a.kv.n_kv_heads;
  const int g0 = blockIdx.x * kGroup, r = blockIdx.y;
  const bool is_q = r < n_qg;
  const int h = is_q ? r : r - n_qg;

  grid_dep_wait();     // the rows may come from the previous kernel of the stream
  grid_dep_trigger();  // the attention kernel may start launching; it waits for this grid
  if (is_q) {  // block-uniform; the query side has no block barrier
    if (g0 + warp < a.kv.n_tokens) rope_q_rows<D>(a, g0 + warp, h * a.q_heads_per_warp, lane);
    return;
  }
  {
    const int k = warp;  // one token per warp
    const int tok = g0 + k;
    long long ph = -1;
    int slot = 0;
    if (tok < a.kv.n_tokens) {
      const int p = a.kv.pos[tok];
      const bool pos_ok = p >= 0 && p < a.max_pos;
      {
        // ---- K and V rows of KV head h into the token's slot
        const int seq = a.kv.seq_idx[tok];
        if (!pos_ok || p / KVQ_BLOCK_SIZE >= a.kv.max_blocks_per_seq) {
          if (lane == 0) set_status(a.kv.status, KVQ_DEV_BAD_POS);
        } else if (seq < 0 || seq >= a.kv.num_seqs) {
          if (lane == 0) set_status(a.kv.status, KVQ_DEV_BAD_SEQ);
        } else {
          const int page = a.kv.block_table[static_cast<long long>(seq) * a.kv.max_blocks_per_seq + p / KVQ_BLOCK_SIZE];
          if (page < 0 || page >= a.kv.num_blocks) {
            if (lane == 0) set_status(a.kv.status, KVQ_DEV_BAD_BLOCK);
          } else {
            ph = static_cast<long long>(page) * H + h;
            slot = p % KVQ_BLOCK_SIZE;
          }
        }
        if (ph >= 0) {  // warp-uniform
          const long long row = (static_cast<long long>(tok) * H + h) * D + lane * P;
          float xk[P], xv[P];
          load_bf16_lane(static_cast<const uint16_t*>(a.kv.k_new) + row, xk);
          load_bf16_lane(static_cast<const uint16_t*>(a.kv.v_new) + row, xv);
          rope_lane(xk, a, p, lane);
          uint32_t packed[P / 4];
          const float sk = quant_rule_warp_packed(xk, packed);
          store_k_codes<D>(a.kv.k, ph, slot, lane, packed);
          const float sv = quant_rule_warp_packed(xv, packed);
          if constexpr (P == 8) *reinterpret_cast<uint2*>(&vs[k][lane * P]) = make_uint2(packed[0], packed[1]);
          else *reinterpret_cast<uint32_t*>(&vs[k][lane * P]) = packed[0];
          if (lane == 0) {
            a.kv.k_scale[ph * KVQ_BLOCK_SIZE + slot] = sk;
            a.kv.v_scale[ph * KVQ_BLOCK_SIZE + slot] = sv;
          }
        }
      }
    }
    if (lane == 0) {
      tok_ph[k] = ph;
      tok_slot[k] = slot;
    }
  }
  __syncthreads();
  bool full = true;
#pragma unroll
  for (int k = 0; k < kGroup; ++k) full = full && tok_ph[k] == tok_ph[0] && tok_slot[k] == k;
  full = full && tok_ph[0] >= 0;
  if (full) {
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
      uint32_t w[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        w[q4] = static_cast<uint32_t>(static_cast<uint8_t>(vs[4 * q4][d])) |
                (static_cast<uint32_t>(static_cast<uint8_t>(vs[4 * q4 + 1][d])) << 8) |
                (static_cast<uint32_t>(static_cast<uint8_t>(vs[4 * q4 + 2][d])) << 16) |
                (static_cast<uint32_t>(static_cast<uint8_t>(vs[4 * q4 + 3][d])) << 24);
      *reinterpret_cast<uint4*>(a.kv.v + (tok_ph[0] * D + d) * KVQ_BLOCK_SIZE) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    for (int it = threadIdx.x; it < kGroup * D; it += blockDim.x) {
      const int k = it / D, d = it % D;
      const long long ph = tok_ph[k];
      if (ph >= 0) a.kv.v[(ph * D + d) * KVQ_BLOCK_SIZE + tok_slot[k]] = vs[k][d];
    }
  }
}

cudaError_t launch_rope_quant_write(const RopeQuantArgs& a_in, cudaStream_t stream) {
  RopeQuantArgs a = a_in;
  // Many tokens: a warp takes several query heads of its token (the table row is read once for
  // them and the next row's load overlaps the current row); few tokens: one head per warp, so
  // that the rows still spread over the GPU.
  a.q_heads_per_warp = a.kv.n_tokens >= 512 ? 8 : 1;
  const long long groups = (static_cast<long long>(a.kv.n_tokens) + kGroup - 1) / kGroup;
  const int slots = (a.q ? (a.n_q_heads + a.q_heads_per_warp - 1) / a.q_heads_per_warp : 0) + a.kv.n_kv_heads;
  if (groups > 0x7fffffffLL || slots > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(groups), slots);
  if (a.kv.head_dim == 256) return launch_pdl(rope_quant_write_kernel<256>, grid, dim3(kGroup * 32), 0, stream, a);
  return launch_pdl(rope_quant_write_kernel<128>, grid, dim3(kGroup * 32), 0, stream, a);
}

}  // namespace kvq
