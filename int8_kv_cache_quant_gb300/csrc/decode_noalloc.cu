// decode_noalloc.cu — kvq_attn_decode_int8kv_noalloc: the decode call for callers that
// cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc at the point where they run decode: code that
// executes under an allocator that forbids new allocations (a captured or replayed region
// whose memory plan is fixed in advance), plugin hosts that hand out only the tensors they
// own, or runtimes that reserve all device memory up front.  kvq_attn_decode_int8kv needs a
// caller-provided workspace for its split-K partials; this entry point instead keeps that
// scratch in a fixed array inside the library (kvq_noalloc_scratch below), which every GPU
// that loads the library holds until the process exits.  Inputs and outputs are still the
// caller's.
#include <cstdint>
#include <mutex>

#include "kvq.h"
#include "kvq_launch.h"

namespace {

// Scratch of the split route's partials (per (sequence, query head, split): acc[head_dim]
// plus 4 statistics).  KVQ_NOALLOC_SCRATCH_BYTES in kvq.h states its size.
static __device__ __align__(256) unsigned char kvq_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once per device.  In
// host code `kvq_noalloc_scratch` names a host-side stand-in, not device memory: only the
// address returned by cudaGetSymbolAddress may be handed to a kernel.
int scratch_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, kvq_noalloc_scratch) != cudaSuccess || p == nullptr) return KVQ_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" int kvq_attn_decode_int8kv_noalloc(const kvq_cache* cache, const void* q, int32_t batch,
                                              int32_t n_q_heads, const int32_t* block_table,
                                              int32_t max_blocks_per_seq, const int32_t* ctx_lens,
                                              int32_t max_ctx, float softmax_scale, float* out,
                                              const kvq_decode_opts* opts, void* stream) {
  // Same validation and kernels as kvq_attn_decode_int8kv; only the workspace differs.  The
  // limit applies to the partials of the split this call actually takes (the automatic split
  // size of this GPU unless opts sets one), not to the bound kvq_decode_workspace_bytes states.
  if (!cache) return KVQ_ERR_INVALID_ARG;
  kvq::DecodePlan plan;
  const int st0 = kvq::decode_plan(cache, batch, 1, n_q_heads, max_ctx > 0 ? max_ctx : 1, opts, &plan);
  if (st0 != KVQ_OK) return st0;
  if (plan.bytes > static_cast<size_t>(KVQ_NOALLOC_SCRATCH_BYTES)) return KVQ_ERR_WORKSPACE;
  void* ws = nullptr;
  const int st = scratch_ptr(&ws);
  if (st != KVQ_OK) return st;
  return kvq_attn_decode_int8kv(cache, q, batch, n_q_heads, block_table, max_blocks_per_seq, ctx_lens,
                                max_ctx, softmax_scale, out, ws, KVQ_NOALLOC_SCRATCH_BYTES, opts, stream);
}
