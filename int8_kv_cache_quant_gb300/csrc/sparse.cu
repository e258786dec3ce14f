// sparse.cu — sparse prompt attention over the int8 paged K/V cache.
//
// Method: "#3381 [Engine] STRATA_PROMPT_ATTN_RDNA2=1 ... prompt QSA attention without the
// decode kernel's split and merge", sections "Problem and result" and "Approach": one block
// per (query, KV head) walks all of the query's selected cells in 64-cell chunks with an
// online softmax, with no per-chunk scratch and no merge pass; the value phase takes 4 head
// dimensions per thread; each chunk's softmax sum and value sums start from zero (relative
// to the updated maximum) and are folded into the running sums with one fma each, so the
// summation is blocked like a split path's.
//
// GB300 mapping: a CTA of 64 threads serves one (query, KV head) and every query head of
// its GQA group (12 at the page's geometry).  Score phase: thread j owns cell j of the
// chunk, reads the cell's K row as sixteen 16-byte loads (the K layout keeps 16 dims of a
// token contiguous) and dots it with the group's Q rows held in shared memory.  Value
// phase: thread t owns dims 4t..4t+3 and accumulates every head of the group.  FP32
// arithmetic on the CUDA cores throughout; the working set (17 MB of cache at ctx 32768,
// head_dim 256, one KV head) stays in L2.
#include "kvq_dev.cuh"
#include "kvq_launch.h"

namespace kvq {

namespace {
constexpr int kChunk = 64;  // cells per chunk, = threads per CTA
constexpr float kLog2eS = 1.4426950408889634f;
}  // namespace

template <int D, int G>
__global__ void __launch_bounds__(kChunk) sparse_kernel(SparseArgs a) {
  static_assert(D / 4 == kChunk || D / 4 == kChunk / 2, "value phase maps 4 dims per thread");
  constexpr int NVT = D / 4;  // threads active in the value phase
  __shared__ __align__(16) float q_s[G][D];
  __shared__ float w_s[G][kChunk];
  __shared__ float red_s[2][G];
  __shared__ int page_s[kChunk];
  __shared__ int slot_s[kChunk];

  const int i = blockIdx.x;   // query
  const int kvh = blockIdx.y;
  const int tid = threadIdx.x;
  const int Hq = a.n_q_heads;
  const float c2 = a.softmax_scale * kLog2eS;

  for (int e = tid; e < G * D; e += kChunk) {
    const int hh = e / D, d = e % D;
    const uint16_t qb = static_cast<const uint16_t*>(a.q)[(static_cast<long long>(i) * Hq + kvh * G + hh) * D + d];
    q_s[hh][d] = bf16_bits_to_float(qb) * c2;  // scores in the log2 domain
  }
  const int c_begin = a.cell_offsets[i];
  const int c_end = a.cell_offsets[i + 1];

  float m[G], l[G], acc[G][4];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    m[hh] = -INFINITY;
    l[hh] = 0.f;
    acc[hh][0] = acc[hh][1] = acc[hh][2] = acc[hh][3] = 0.f;
  }
  __syncthreads();

  for (int base = c_begin; base < c_end; base += kChunk) {
    const int n = min(kChunk, c_end - base);
    // ---- score phase: thread tid owns cell base + tid
    float s[G];
    bool valid = false;
    int page = 0, slot = 0;
    if (tid < n) {
      const int pos = a.cells[base + tid];
      if (pos >= 0 && pos / KVQ_BLOCK_SIZE < a.n_blocks_row) {
        page = a.block_table_row[pos / KVQ_BLOCK_SIZE];
        slot = pos % KVQ_BLOCK_SIZE;
        valid = page >= 0 && page < a.num_blocks;
        if (!valid) set_status(a.status, KVQ_DEV_BAD_BLOCK);
      } else {
        set_status(a.status, KVQ_DEV_BAD_CELL);
      }
    }
    page_s[tid] = valid ? page : -1;
    slot_s[tid] = slot;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) s[hh] = 0.f;
    float sk = 0.f, sv = 0.f;
    if (valid) {
      const long long ph = static_cast<long long>(page) * a.n_kv_heads + kvh;
      const int8_t* krow = a.k + ph * D * KVQ_BLOCK_SIZE + slot * 16;
      sk = a.k_scale[ph * KVQ_BLOCK_SIZE + slot];
      sv = a.v_scale[ph * KVQ_BLOCK_SIZE + slot];
#pragma unroll 4
      for (int ch = 0; ch < D / 16; ++ch) {
        const int4 raw = __ldg(reinterpret_cast<const int4*>(krow + ch * 256));
        const int w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
          float kf[4];
#pragma unroll
          for (int bi = 0; bi < 4; ++bi) kf[bi] = static_cast<float>(static_cast<int8_t>(w4[wi] >> (8 * bi)));
          const int d0 = ch * 16 + wi * 4;
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            const float4 qv = *reinterpret_cast<const float4*>(&q_s[hh][d0]);
            s[hh] = fmaf(kf[0], qv.x, s[hh]);
            s[hh] = fmaf(kf[1], qv.y, s[hh]);
            s[hh] = fmaf(kf[2], qv.z, s[hh]);
            s[hh] = fmaf(kf[3], qv.w, s[hh]);
          }
        }
      }
    }
    // chunk maximum per head (two warps)
    float alpha[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      s[hh] = valid ? s[hh] * sk : -INFINITY;
      float mx = s[hh];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if ((tid & 31) == 0) red_s[tid >> 5][hh] = mx;
    }
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float m_new = fmaxf(m[hh], fmaxf(red_s[0][hh], red_s[1][hh]));
      const float mr = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[hh] = fast_exp2(m[hh] - mr);
      m[hh] = m_new;
      const float p = fast_exp2(s[hh] - mr);
      w_s[hh][tid] = p * sv;  // sV folded into the value weights
      // chunk-local softmax sum, from zero
      float ps = p;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      s[hh] = ps;  // reuse: warp partial of the chunk sum
    }
    __syncthreads();  // red_s reads done before reuse; w_s written
    if ((tid & 31) == 0) {
#pragma unroll
      for (int hh = 0; hh < G; ++hh) red_s[tid >> 5][hh] = s[hh];
    }
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < G; ++hh) l[hh] = fmaf(l[hh], alpha[hh], red_s[0][hh] + red_s[1][hh]);

    // ---- value phase: thread tid owns dims 4*tid .. 4*tid + 3
    if (tid < NVT) {
      float ca[G][4];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) ca[hh][0] = ca[hh][1] = ca[hh][2] = ca[hh][3] = 0.f;
      const int d0 = 4 * tid;
#pragma unroll 2
      for (int j = 0; j < n; ++j) {
        const int pg = page_s[j];
        if (pg < 0) continue;
        const int8_t* vcol = a.v + (static_cast<long long>(pg) * a.n_kv_heads + kvh) * D * KVQ_BLOCK_SIZE +
                             d0 * KVQ_BLOCK_SIZE + slot_s[j];
        float vf[4];
#pragma unroll
        for (int bi = 0; bi < 4; ++bi) vf[bi] = static_cast<float>(__ldg(vcol + bi * KVQ_BLOCK_SIZE));
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float wv = w_s[hh][j];
          ca[hh][0] = fmaf(wv, vf[0], ca[hh][0]);
          ca[hh][1] = fmaf(wv, vf[1], ca[hh][1]);
          ca[hh][2] = fmaf(wv, vf[2], ca[hh][2]);
          ca[hh][3] = fmaf(wv, vf[3], ca[hh][3]);
        }
      }
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[hh][e] = fmaf(acc[hh][e], alpha[hh], ca[hh][e]);
      }
    }
    __syncthreads();  // w_s, page_s, red_s reused by the next chunk
  }

  if (tid < NVT) {
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float inv = (l[hh] > 0.f) ? 1.0f / l[hh] : 0.f;
      float4 o = make_float4(acc[hh][0] * inv, acc[hh][1] * inv, acc[hh][2] * inv, acc[hh][3] * inv);
      *reinterpret_cast<float4*>(a.out + (static_cast<long long>(i) * Hq + kvh * G + hh) * D + 4 * tid) = o;
    }
  }
}

template <int D>
static cudaError_t launch_sparse_d(const SparseArgs& a, int G, dim3 grid, cudaStream_t stream) {
  switch (G) {
    case 1: sparse_kernel<D, 1><<<grid, kChunk, 0, stream>>>(a); break;
    case 2: sparse_kernel<D, 2><<<grid, kChunk, 0, stream>>>(a); break;
    case 4: sparse_kernel<D, 4><<<grid, kChunk, 0, stream>>>(a); break;
    case 6: sparse_kernel<D, 6><<<grid, kChunk, 0, stream>>>(a); break;
    case 8: sparse_kernel<D, 8><<<grid, kChunk, 0, stream>>>(a); break;
    case 12: sparse_kernel<D, 12><<<grid, kChunk, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_sparse(const SparseArgs& a, cudaStream_t stream) {
  const int G = a.n_q_heads / a.n_kv_heads;
  dim3 grid(a.n_queries, a.n_kv_heads);
  if (a.head_dim == 256) return launch_sparse_d<256>(a, G, grid, stream);
  return launch_sparse_d<128>(a, G, grid, stream);
}

}  // namespace kvq
