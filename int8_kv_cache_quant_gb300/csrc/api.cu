// api.cu — the C ABI of libkvq (include/kvq.h): host-side validation, routing and launch.
// Every entry point checks its arguments before launching anything, allocates nothing and
// never synchronises (except kvq_device_status).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "kvq.h"
#include "kvq_dev.cuh"
#include "kvq_launch.h"

namespace {

// Device status word (KVQ_DEV_* bits), one per device that loads the library.
__device__ unsigned int g_kvq_status = 0;

constexpr int kMaxDevices = 64;
unsigned int* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;

// Device address of the status word on the current device, looked up once per device.
unsigned int* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kvq_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  return g_status_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int check_cache(const kvq_cache* c) {
  if (!c || !c->k || !c->v || !c->k_scale || !c->v_scale) return KVQ_ERR_INVALID_ARG;
  if (c->num_blocks <= 0 || c->n_kv_heads <= 0) return KVQ_ERR_INVALID_ARG;
  if (c->block_size != KVQ_BLOCK_SIZE) return KVQ_ERR_UNSUPPORTED;
  if (c->head_dim != 128 && c->head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  if (!aligned16(c->k) || !aligned16(c->v) || !aligned16(c->k_scale) || !aligned16(c->v_scale))
    return KVQ_ERR_MISALIGNED;
  return KVQ_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

kvq_decode_opts decode_defaults(const kvq_decode_opts* o) {
  kvq_decode_opts r = {0, 0, 0, nullptr, nullptr, nullptr};  // split_rows 0: sized to the GPU; route 0: automatic
  if (o) {
    if (o->split_rows > 0) r.split_rows = o->split_rows;
    if (o->route_threshold > 0) r.route_threshold = o->route_threshold;
    r.force_route = o->force_route;
    r.stage1_event_begin = o->stage1_event_begin;
    r.stage1_event_end = o->stage1_event_end;
    r.launches = o->launches;
  }
  return r;
}

constexpr int kMaxSplits = 16384;

// Test-only fault injection (kvq_debug_fault_inject): the mode and the wait budget that the
// kernels launched from now on receive.
std::atomic<int> g_fault_mode{0};
std::atomic<long long> g_wait_budget{kvq::kWaitBudgetCycles};

}  // namespace

namespace kvq {
int debug_fault_mode() { return g_fault_mode.load(std::memory_order_relaxed); }
long long debug_wait_budget() { return g_wait_budget.load(std::memory_order_relaxed); }
}  // namespace kvq

extern "C" {

int kvq_version(void) { return KVQ_ABI_VERSION; }

const char* kvq_status_string(int s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported shape or option";
    case KVQ_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KVQ_ERR_CUDA: return "CUDA launch or runtime error";
    default: return "unknown status";
  }
}

int kvq_debug_fault_inject(int32_t mode, int64_t wait_budget_cycles) {
  if (mode < 0 || mode > 3) return KVQ_ERR_INVALID_ARG;
  g_wait_budget.store(wait_budget_cycles > 0 ? static_cast<long long>(wait_budget_cycles) : kvq::kWaitBudgetCycles);
  g_fault_mode.store(mode);
  return KVQ_OK;
}

int kvq_device_status(uint32_t* flags_out, void* stream) {
  if (!flags_out) return KVQ_ERR_INVALID_ARG;
  *flags_out = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_kvq_status, sizeof v) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_kvq_status, &zero, sizeof zero) != cudaSuccess) return KVQ_ERR_CUDA;
  *flags_out = v;
  return KVQ_OK;
}

int kvq_quant_write(const kvq_cache* cache, const void* k_new, const void* v_new, int32_t n_tokens,
                    const int32_t* seq_idx, const int32_t* pos, const int32_t* block_table,
                    int32_t num_seqs, int32_t max_blocks_per_seq, void* stream) {
  int st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (n_tokens < 0 || num_seqs <= 0 || max_blocks_per_seq <= 0) return KVQ_ERR_INVALID_ARG;
  if (n_tokens == 0) return KVQ_OK;
  if (!k_new || !v_new || !seq_idx || !pos || !block_table) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_MISALIGNED;
  if (!aligned4(seq_idx) || !aligned4(pos) || !aligned4(block_table)) return KVQ_ERR_MISALIGNED;
  kvq::QuantWriteArgs a{};
  a.k = cache->k;
  a.v = cache->v;
  a.k_scale = cache->k_scale;
  a.v_scale = cache->v_scale;
  a.num_blocks = cache->num_blocks;
  a.n_kv_heads = cache->n_kv_heads;
  a.head_dim = cache->head_dim;
  a.k_new = k_new;
  a.v_new = v_new;
  a.n_tokens = n_tokens;
  a.seq_idx = seq_idx;
  a.pos = pos;
  a.block_table = block_table;
  a.num_seqs = num_seqs;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.status = status_ptr();
  return cuda_status(kvq::launch_quant_write(a, static_cast<cudaStream_t>(stream)));
}

int kvq_rope_quant_write(const kvq_cache* cache, const void* q, int32_t n_q_heads, const void* k_new,
                         const void* v_new, int32_t n_tokens, const int32_t* seq_idx, const int32_t* pos,
                         const int32_t* block_table, int32_t num_seqs, int32_t max_blocks_per_seq,
                         const float* cos_sin, int32_t max_pos, int32_t rotary_dim, int8_t* q_codes,
                         float* q_scales, void* q_rot, void* stream) {
  int st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (n_tokens < 0 || num_seqs <= 0 || max_blocks_per_seq <= 0 || max_pos <= 0) return KVQ_ERR_INVALID_ARG;
  if (n_tokens == 0) return KVQ_OK;
  if (!k_new || !v_new || !seq_idx || !pos || !block_table || !cos_sin) return KVQ_ERR_INVALID_ARG;
  if (q && n_q_heads <= 0) return KVQ_ERR_INVALID_ARG;
  const int D = cache->head_dim;
  if (rotary_dim <= 0 || rotary_dim > D || rotary_dim % 2 != 0 || (rotary_dim / 2) % (D / 32) != 0)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(cos_sin)) return KVQ_ERR_MISALIGNED;
  if ((q && !aligned16(q)) || (q_rot && !aligned16(q_rot))) return KVQ_ERR_MISALIGNED;
  if (q_codes && reinterpret_cast<uintptr_t>(q_codes) % 8 != 0) return KVQ_ERR_MISALIGNED;
  if ((q_scales && !aligned4(q_scales)) || !aligned4(seq_idx) || !aligned4(pos) || !aligned4(block_table))
    return KVQ_ERR_MISALIGNED;
  kvq::RopeQuantArgs r{};
  r.kv.k = cache->k;
  r.kv.v = cache->v;
  r.kv.k_scale = cache->k_scale;
  r.kv.v_scale = cache->v_scale;
  r.kv.num_blocks = cache->num_blocks;
  r.kv.n_kv_heads = cache->n_kv_heads;
  r.kv.head_dim = D;
  r.kv.k_new = k_new;
  r.kv.v_new = v_new;
  r.kv.n_tokens = n_tokens;
  r.kv.seq_idx = seq_idx;
  r.kv.pos = pos;
  r.kv.block_table = block_table;
  r.kv.num_seqs = num_seqs;
  r.kv.max_blocks_per_seq = max_blocks_per_seq;
  r.kv.status = status_ptr();
  r.q = q;
  r.n_q_heads = q ? n_q_heads : 0;
  r.cos_sin = cos_sin;
  r.max_pos = max_pos;
  r.rotary_dim = rotary_dim;
  r.q_codes = q_codes;
  r.q_scales = q_scales;
  r.q_rot = static_cast<uint16_t*>(q_rot);
  return cuda_status(kvq::launch_rope_quant_write(r, static_cast<cudaStream_t>(stream)));
}

// Smallest split the automatic rule chooses: the workspace bound when split_rows is 0.
constexpr int kAutoSplitMinRows = 4 * KVQ_BLOCK_SIZE;

// Whether the split route may be taken, from host arguments alone (sizes the workspace).  The
// automatic route splits only when the split size leaves more than one split, and the automatic
// split size is never below kAutoSplitMinRows keys.
static bool decode_split_route(const kvq_decode_opts& o, int32_t max_ctx) {
  if (o.force_route == 1) return false;
  if (o.force_route == 2) return true;
  if (o.route_threshold > 0) return max_ctx > o.route_threshold;
  const int rows = o.split_rows > 0 ? o.split_rows : kAutoSplitMinRows;
  return max_ctx > rows;
}

int32_t kvq_decode_auto_split_rows(int32_t batch, int32_t n_kv_heads, int32_t head_dim, int32_t max_ctx,
                                   int32_t n_sms) {
  if (batch <= 0 || n_kv_heads <= 0 || max_ctx <= 0 || n_sms <= 0) return 0;
  if (head_dim != 128 && head_dim != 256) return 0;
  const long long slots = static_cast<long long>(n_sms) * (head_dim == 256 ? 1 : 2);  // resident stage-1 CTAs
  const long long units = static_cast<long long>(batch) * n_kv_heads;
  const long long pages = (static_cast<long long>(max_ctx) + KVQ_BLOCK_SIZE - 1) / KVQ_BLOCK_SIZE;
  long long split_pages;
  if (units * ((pages + 31) / 32) > 2 * slots) {
    split_pages = std::min(128LL, std::max(32LL, units * pages / (4 * slots)));
  } else {
    const long long per_unit = std::max(1LL, slots / units);
    split_pages = std::max(4LL, (pages + per_unit - 1) / per_unit);
  }
  return static_cast<int32_t>(split_pages * KVQ_BLOCK_SIZE);
}

static int device_sm_count() {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

size_t kvq_decode_workspace_bytes(int32_t batch, int32_t n_q_heads, int32_t max_ctx,
                                  int32_t head_dim, const kvq_decode_opts* opts) {
  const kvq_decode_opts o = decode_defaults(opts);
  if (batch <= 0 || n_q_heads <= 0 || max_ctx <= 0 || head_dim <= 0 || o.split_rows < 0) return 0;
  if (!decode_split_route(o, max_ctx)) return 0;
  const int rows = o.split_rows > 0 ? o.split_rows : kAutoSplitMinRows;
  return kvq::decode_workspace_bytes(batch, n_q_heads, max_ctx, head_dim, rows);
}

size_t kvq_verify_workspace_bytes(int32_t batch, int32_t n_rows, int32_t n_q_heads, int32_t max_ctx,
                                  int32_t head_dim, const kvq_decode_opts* opts) {
  if (batch <= 0 || n_rows <= 0 || static_cast<long long>(batch) * n_rows > INT32_MAX) return 0;
  return kvq_decode_workspace_bytes(batch * n_rows, n_q_heads, max_ctx, head_dim, opts);
}

}  // extern "C"

namespace kvq {
int decode_plan(const kvq_cache* cache, int32_t batch, int32_t nq, int32_t n_q_heads, int32_t max_ctx,
                const kvq_decode_opts* opts, DecodePlan* plan) {
  if (!cache || batch <= 0 || nq <= 0 || n_q_heads <= 0 || cache->n_kv_heads <= 0) return KVQ_ERR_INVALID_ARG;
  if (cache->head_dim != 128 && cache->head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  kvq_decode_opts o = decode_defaults(opts);
  if (o.split_rows % KVQ_BLOCK_SIZE != 0 || o.force_route < 0 || o.force_route > 2) return KVQ_ERR_INVALID_ARG;
  const int mc = max_ctx > 0 ? max_ctx : 1;
  bool split = decode_split_route(o, mc);
  if (split && o.split_rows == 0) {
    const int sms = device_sm_count();
    if (sms <= 0) return KVQ_ERR_CUDA;
    o.split_rows = kvq_decode_auto_split_rows(batch, cache->n_kv_heads, cache->head_dim, mc, sms);
  }
  // automatic route: one split would be the single-CTA route plus a merge
  if (split && o.force_route == 0 && o.route_threshold == 0 && mc <= o.split_rows) split = false;
  plan->split = split;
  plan->split_rows = o.split_rows;
  plan->n_split = 1;
  plan->bytes = 0;
  if (split) {
    const long long n_split = (static_cast<long long>(mc) + o.split_rows - 1) / o.split_rows;
    if (n_split > kMaxSplits) return KVQ_ERR_UNSUPPORTED;
    plan->n_split = static_cast<int>(n_split);
    plan->bytes = decode_workspace_bytes(batch * nq, n_q_heads, mc, cache->head_dim, o.split_rows);
  }
  return KVQ_OK;
}
}  // namespace kvq

extern "C" {

// Decode with nq query rows per sequence (nq = 1: plain decode); with k_new / v_new, the fused
// step that first writes each sequence's nq newest tokens into the cache.
static int decode_rows(const kvq_cache* cache, const void* k_new, const void* v_new, const void* q, int32_t batch,
                       int32_t nq, int32_t n_q_heads, const int32_t* block_table, int32_t max_blocks_per_seq,
                       const int32_t* ctx_lens, int32_t max_ctx, float softmax_scale, float* out, void* workspace,
                       size_t workspace_bytes, const kvq_decode_opts* opts, void* stream) {
  int st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!q || !block_table || !ctx_lens || !out) return KVQ_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return KVQ_ERR_INVALID_ARG;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return KVQ_ERR_MISALIGNED;
  if (batch <= 0 || nq <= 0 || n_q_heads <= 0 || max_blocks_per_seq <= 0 || max_ctx < 0) return KVQ_ERR_INVALID_ARG;
  // stage 1 puts the sequences on grid z, the merge puts (sequence, row) on grid y
  if (static_cast<long long>(batch) * nq > 65535) return KVQ_ERR_UNSUPPORTED;
  if (n_q_heads % cache->n_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  const int G = n_q_heads / cache->n_kv_heads;
  if (G > 16 || static_cast<long long>(G) * nq > KVQ_VERIFY_MAX_ROWS) return KVQ_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(out)) return KVQ_ERR_MISALIGNED;
  if (!aligned4(block_table) || !aligned4(ctx_lens)) return KVQ_ERR_MISALIGNED;
  const int mc = max_ctx > 0 ? max_ctx : 1;
  const kvq_decode_opts o = decode_defaults(opts);
  if (o.split_rows % KVQ_BLOCK_SIZE != 0 || o.force_route < 0 || o.force_route > 2) return KVQ_ERR_INVALID_ARG;
  // the workspace rule is pure host arithmetic (kvq_decode_workspace_bytes), checked before the GPU is asked
  if (decode_split_route(o, mc) && !workspace) return KVQ_ERR_WORKSPACE;
  kvq::DecodePlan plan;
  st = kvq::decode_plan(cache, batch, nq, n_q_heads, mc, opts, &plan);
  if (st != KVQ_OK) return st;
  const bool split = plan.split;
  kvq::DecodeArgs a{};
  a.k = cache->k;
  a.v = cache->v;
  a.k_scale = cache->k_scale;
  a.v_scale = cache->v_scale;
  a.num_blocks = cache->num_blocks;
  a.n_kv_heads = cache->n_kv_heads;
  a.head_dim = cache->head_dim;
  a.q = q;
  a.batch = batch;
  a.nq = nq;
  a.n_q_heads = n_q_heads;
  a.block_table = block_table;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.ctx_lens = ctx_lens;
  a.max_ctx = mc;
  a.softmax_scale = softmax_scale;
  a.k_new = k_new;
  a.v_new = v_new;
  a.out = out;
  a.split_rows = plan.split_rows;
  a.status = status_ptr();
  a.ev_begin = static_cast<cudaEvent_t>(o.stage1_event_begin);
  a.ev_end = static_cast<cudaEvent_t>(o.stage1_event_end);
  a.wait_budget = kvq::debug_wait_budget();
  a.fault = kvq::debug_fault_mode();
  if (split) {
    const long long n_split = plan.n_split;
    if (!workspace || workspace_bytes < plan.bytes) return KVQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return KVQ_ERR_MISALIGNED;
    a.n_split = static_cast<int>(n_split);
    const long long units = static_cast<long long>(batch) * nq * n_q_heads * n_split;
    const long long acc_bytes = ((units * cache->head_dim * 4 + 255) / 256) * 256;
    a.part_acc = static_cast<float*>(workspace);
    a.part_stats = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_bytes);
    int launched = 0;
    const int rc = cuda_status(kvq::launch_decode(a, kvq::DecodeRoute::kSplit, static_cast<cudaStream_t>(stream), &launched));
    if (o.launches) *o.launches = launched;
    return rc;
  }
  a.n_split = 1;
  int launched = 0;
  const int rc = cuda_status(kvq::launch_decode(a, kvq::DecodeRoute::kSingle, static_cast<cudaStream_t>(stream), &launched));
  if (o.launches) *o.launches = launched;
  return rc;
}

int kvq_attn_decode_int8kv(const kvq_cache* cache, const void* q, int32_t batch, int32_t n_q_heads,
                           const int32_t* block_table, int32_t max_blocks_per_seq,
                           const int32_t* ctx_lens, int32_t max_ctx, float softmax_scale, float* out,
                           void* workspace, size_t workspace_bytes, const kvq_decode_opts* opts,
                           void* stream) {
  return decode_rows(cache, nullptr, nullptr, q, batch, 1, n_q_heads, block_table, max_blocks_per_seq, ctx_lens,
                     max_ctx, softmax_scale, out, workspace, workspace_bytes, opts, stream);
}

int kvq_attn_verify_int8kv(const kvq_cache* cache, const void* q, int32_t batch, int32_t n_rows,
                           int32_t n_q_heads, const int32_t* block_table, int32_t max_blocks_per_seq,
                           const int32_t* ctx_lens, int32_t max_ctx, float softmax_scale, float* out,
                           void* workspace, size_t workspace_bytes, const kvq_decode_opts* opts,
                           void* stream) {
  return decode_rows(cache, nullptr, nullptr, q, batch, n_rows, n_q_heads, block_table, max_blocks_per_seq,
                     ctx_lens, max_ctx, softmax_scale, out, workspace, workspace_bytes, opts, stream);
}

int kvq_decode_step_int8kv(const kvq_cache* cache, const void* k_new, const void* v_new, const void* q,
                           int32_t batch, int32_t n_new, int32_t n_q_heads, const int32_t* block_table,
                           int32_t max_blocks_per_seq, const int32_t* ctx_lens, int32_t max_ctx,
                           float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                           const kvq_decode_opts* opts, void* stream) {
  if (!k_new || !v_new) return KVQ_ERR_INVALID_ARG;
  return decode_rows(cache, k_new, v_new, q, batch, n_new, n_q_heads, block_table, max_blocks_per_seq, ctx_lens,
                     max_ctx, softmax_scale, out, workspace, workspace_bytes, opts, stream);
}

size_t kvq_prefill_workspace_bytes(int32_t n_tokens, int32_t n_q_heads, int32_t n_kv_heads, int32_t history_len,
                                   int32_t head_dim) {
  if (n_tokens <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || history_len < 0 || head_dim <= 0) return 0;
  return static_cast<size_t>(kvq::prefill_workspace(n_tokens, n_q_heads, n_kv_heads, history_len, head_dim).bytes);
}

static kvq::PrefillArgs prefill_args(const kvq_cache* cache, const void* q, int32_t n_tokens,
                                     int32_t n_q_heads, int32_t history_len,
                                     const int32_t* block_table_row, int32_t n_blocks_row,
                                     float softmax_scale, float* out, void* workspace) {
  kvq::PrefillArgs a{};
  a.k = cache->k;
  a.v = cache->v;
  a.k_scale = cache->k_scale;
  a.v_scale = cache->v_scale;
  a.num_blocks = cache->num_blocks;
  a.n_kv_heads = cache->n_kv_heads;
  a.head_dim = cache->head_dim;
  a.q = q;
  a.n_tokens = n_tokens;
  a.n_q_heads = n_q_heads;
  a.history_len = history_len;
  a.block_table_row = block_table_row;
  a.n_blocks_row = n_blocks_row;
  a.softmax_scale = softmax_scale;
  a.out = out;
  if (workspace) {
    const kvq::PrefillWorkspace w =
        kvq::prefill_workspace(n_tokens, n_q_heads, cache->n_kv_heads, history_len, cache->head_dim);
    char* base = static_cast<char*>(workspace);
    a.q_codes = reinterpret_cast<int8_t*>(base);
    a.q_scales = reinterpret_cast<float*>(base + w.off_q_scales);
    a.n_kv_tiles = w.n_kv_tiles;
    a.kw = reinterpret_cast<uint8_t*>(base + w.off_kw);
    a.vw = reinterpret_cast<uint8_t*>(base + w.off_vw);
    a.skw = reinterpret_cast<float*>(base + w.off_skw);
    a.svw = reinterpret_cast<float*>(base + w.off_svw);
    if (w.can_split) {
      a.part = reinterpret_cast<float*>(base + w.off_part);
      a.part_ml = reinterpret_cast<float*>(base + w.off_part_ml);
      a.part_cnt = reinterpret_cast<unsigned int*>(base + w.off_part_flags);
      a.part_ready = a.part_cnt + static_cast<long long>((n_tokens + 127) / 128) * n_q_heads;
      a.split_tail = kvq::prefill_split_tail(n_tokens, n_q_heads, history_len, device_sm_count());
    }
  }
  a.status = status_ptr();
  a.wait_budget = kvq::debug_wait_budget();
  a.fault = kvq::debug_fault_mode();
  return a;
}

int32_t kvq_device_accessible(const void* p) {
  if (!p) return 0;
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    (void)cudaGetLastError();  // not a sticky error: clear it so the caller's next check is clean
    return 0;
  }
  if (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged) return 1;
  return attr.type == cudaMemoryTypeHost && attr.devicePointer == p ? 1 : 0;
}

int32_t kvq_prefill_split_tiles(int32_t n_tokens, int32_t n_q_heads, int32_t history_len, int32_t n_sms) {
  return kvq::prefill_split_tail(n_tokens, n_q_heads, history_len, n_sms);
}

int kvq_attn_prefill_int8(const kvq_cache* cache, const void* q, int32_t n_tokens, int32_t n_q_heads,
                          int32_t history_len, const int32_t* block_table_row, int32_t n_blocks_row,
                          float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                          void* stream) {
  int st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!q || !block_table_row || !out) return KVQ_ERR_INVALID_ARG;
  if (n_tokens <= 0 || n_q_heads <= 0 || history_len < 0 || n_blocks_row <= 0) return KVQ_ERR_INVALID_ARG;
  if (n_q_heads % cache->n_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || !std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if (static_cast<long long>(history_len) + n_tokens > static_cast<long long>(n_blocks_row) * KVQ_BLOCK_SIZE)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned4(block_table_row)) return KVQ_ERR_MISALIGNED;
  const size_t need = kvq_prefill_workspace_bytes(n_tokens, n_q_heads, cache->n_kv_heads, history_len,
                                                  cache->head_dim);
  if (!workspace || workspace_bytes < need) return KVQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KVQ_ERR_MISALIGNED;
  kvq::PrefillArgs a = prefill_args(cache, q, n_tokens, n_q_heads, history_len, block_table_row,
                                    n_blocks_row, softmax_scale, out, workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = kvq::launch_prefill_q_quant(a, s);
  if (e != cudaSuccess) return e == cudaErrorNotSupported ? KVQ_ERR_UNSUPPORTED : KVQ_ERR_CUDA;
  e = kvq::launch_prefill(a, s);
  if (e != cudaSuccess) return e == cudaErrorNotSupported ? KVQ_ERR_UNSUPPORTED : KVQ_ERR_CUDA;
  return KVQ_OK;
}

size_t kvq_prefill_first_workspace_bytes(int32_t n_tokens, int32_t n_q_heads, int32_t n_kv_heads,
                                         int32_t head_dim) {
  if (n_tokens <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || (head_dim != 128 && head_dim != 256)) return 0;
  return static_cast<size_t>(kvq::prefill_workspace(n_tokens, n_q_heads, n_kv_heads, 0, head_dim, 2).bytes);
}

int kvq_attn_prefill_first_bf16(const kvq_cache* cache, const void* q, const void* k_new, const void* v_new,
                                int32_t n_tokens, int32_t n_q_heads, const int32_t* block_table_row,
                                int32_t n_blocks_row, float softmax_scale, float* out, void* workspace,
                                size_t workspace_bytes, void* stream) {
  int st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!q || !k_new || !v_new || !block_table_row || !out) return KVQ_ERR_INVALID_ARG;
  if (n_tokens <= 0 || n_q_heads <= 0 || n_blocks_row <= 0) return KVQ_ERR_INVALID_ARG;
  if (n_q_heads % cache->n_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || !std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if (static_cast<long long>(n_tokens) > static_cast<long long>(n_blocks_row) * KVQ_BLOCK_SIZE)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out) || !aligned4(block_table_row))
    return KVQ_ERR_MISALIGNED;
  const kvq::PrefillWorkspace w = kvq::prefill_workspace(n_tokens, n_q_heads, cache->n_kv_heads, 0, cache->head_dim, 2);
  if (!workspace || workspace_bytes < static_cast<size_t>(w.bytes)) return KVQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KVQ_ERR_MISALIGNED;
  kvq::PrefillArgs a = prefill_args(cache, q, n_tokens, n_q_heads, 0, block_table_row, n_blocks_row,
                                    softmax_scale, out, nullptr);
  char* base = static_cast<char*>(workspace);
  a.q_f16 = reinterpret_cast<uint16_t*>(base);
  a.q_scales = reinterpret_cast<float*>(base + w.off_q_scales);
  a.n_kv_tiles = w.n_kv_tiles;
  a.kw = reinterpret_cast<uint8_t*>(base + w.off_kw);
  a.vw = reinterpret_cast<uint8_t*>(base + w.off_vw);
  a.skw = reinterpret_cast<float*>(base + w.off_skw);
  a.svw = reinterpret_cast<float*>(base + w.off_svw);
  a.k_src = k_new;
  a.v_src = v_new;
  return cuda_status(kvq::launch_prefill_first(a, static_cast<cudaStream_t>(stream)));
}

int kvq_attn_prefill_int8_qcodes(const kvq_cache* cache, const int8_t* q_codes, const float* q_scales,
                                 int32_t n_tokens, int32_t n_q_heads, int32_t history_len,
                                 const int32_t* block_table_row, int32_t n_blocks_row, float softmax_scale,
                                 float* out, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!q_codes || !q_scales || !block_table_row || !out) return KVQ_ERR_INVALID_ARG;
  if (n_tokens <= 0 || n_q_heads <= 0 || history_len < 0 || n_blocks_row <= 0) return KVQ_ERR_INVALID_ARG;
  if (n_q_heads % cache->n_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || !std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if (static_cast<long long>(history_len) + n_tokens > static_cast<long long>(n_blocks_row) * KVQ_BLOCK_SIZE)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q_codes) || !aligned4(q_scales) || !aligned16(out) || !aligned4(block_table_row))
    return KVQ_ERR_MISALIGNED;
  const size_t need = kvq_prefill_workspace_bytes(n_tokens, n_q_heads, cache->n_kv_heads, history_len,
                                                  cache->head_dim);
  if (!workspace || workspace_bytes < need) return KVQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KVQ_ERR_MISALIGNED;
  kvq::PrefillArgs a = prefill_args(cache, nullptr, n_tokens, n_q_heads, history_len, block_table_row,
                                    n_blocks_row, softmax_scale, out, workspace);
  a.q_codes = const_cast<int8_t*>(q_codes);
  a.q_scales = const_cast<float*>(q_scales);
  return cuda_status(kvq::launch_prefill(a, static_cast<cudaStream_t>(stream)));
}

size_t kvq_sparse_workspace_bytes(int32_t n_blocks_row, int32_t n_kv_heads, int32_t head_dim) {
  if (n_blocks_row <= 0 || n_kv_heads <= 0 || (head_dim != 128 && head_dim != 256)) return 0;
  return kvq::sparse_workspace_bytes(n_blocks_row, n_kv_heads, head_dim);
}

int kvq_attn_sparse_int8kv(const kvq_cache* cache, const void* q, int32_t n_queries, int32_t n_q_heads,
                           const int32_t* cell_offsets, const int32_t* cells,
                           const int32_t* block_table_row, int32_t n_blocks_row, float softmax_scale,
                           float* out, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!q || !cell_offsets || !cells || !block_table_row || !out) return KVQ_ERR_INVALID_ARG;
  if (n_queries <= 0 || n_q_heads <= 0 || n_blocks_row <= 0) return KVQ_ERR_INVALID_ARG;
  if (cache->n_kv_heads > 65535) return KVQ_ERR_UNSUPPORTED;  // grid y of both kernels
  if (n_q_heads % cache->n_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  const int G = n_q_heads / cache->n_kv_heads;
  if (G > 16) return KVQ_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < kvq::sparse_workspace_bytes(n_blocks_row, cache->n_kv_heads, cache->head_dim))
    return KVQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KVQ_ERR_MISALIGNED;
  if (!aligned16(q) || !aligned16(out)) return KVQ_ERR_MISALIGNED;
  if (!aligned4(cell_offsets) || !aligned4(cells) || !aligned4(block_table_row)) return KVQ_ERR_MISALIGNED;
  kvq::SparseArgs a{};
  a.k = cache->k;
  a.v = cache->v;
  a.k_scale = cache->k_scale;
  a.v_scale = cache->v_scale;
  a.num_blocks = cache->num_blocks;
  a.n_kv_heads = cache->n_kv_heads;
  a.head_dim = cache->head_dim;
  a.q = q;
  a.n_queries = n_queries;
  a.n_q_heads = n_q_heads;
  a.cell_offsets = cell_offsets;
  a.cells = cells;
  a.block_table_row = block_table_row;
  a.n_blocks_row = n_blocks_row;
  a.softmax_scale = softmax_scale;
  a.out = out;
  a.records = static_cast<uint8_t*>(workspace);
  a.status = status_ptr();
  a.wait_budget = kvq::debug_wait_budget();
  a.fault = kvq::debug_fault_mode();
  return cuda_status(kvq::launch_sparse(a, static_cast<cudaStream_t>(stream)));
}

int kvq_debug_stream_floor(const kvq_cache* cache, int32_t batch, const int32_t* block_table,
                           int32_t max_blocks_per_seq, const int32_t* ctx_lens, int32_t max_ctx, int32_t split_rows,
                           void* stream) {
  int st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!block_table || !ctx_lens || batch <= 0 || batch > 65535 || max_blocks_per_seq <= 0 || max_ctx <= 0)
    return KVQ_ERR_INVALID_ARG;
  if (split_rows < 0 || split_rows % KVQ_BLOCK_SIZE != 0) return KVQ_ERR_INVALID_ARG;
  if (!aligned4(block_table) || !aligned4(ctx_lens)) return KVQ_ERR_MISALIGNED;
  if (split_rows == 0) {
    const int sms = device_sm_count();
    if (sms <= 0) return KVQ_ERR_CUDA;
    split_rows = kvq_decode_auto_split_rows(batch, cache->n_kv_heads, cache->head_dim, max_ctx, sms);
  }
  const long long n_split = (static_cast<long long>(max_ctx) + split_rows - 1) / split_rows;
  if (n_split > kMaxSplits) return KVQ_ERR_UNSUPPORTED;
  kvq::DecodeArgs a{};
  a.k = cache->k;
  a.v = cache->v;
  a.k_scale = cache->k_scale;
  a.v_scale = cache->v_scale;
  a.num_blocks = cache->num_blocks;
  a.n_kv_heads = cache->n_kv_heads;
  a.head_dim = cache->head_dim;
  a.batch = batch;
  a.block_table = block_table;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.ctx_lens = ctx_lens;
  a.max_ctx = max_ctx;
  a.split_rows = split_rows;
  a.n_split = static_cast<int>(n_split);
  a.status = status_ptr();
  a.wait_budget = kvq::debug_wait_budget();
  return cuda_status(kvq::launch_stream_floor(a, static_cast<cudaStream_t>(stream)));
}

int kvq_debug_prefill_q_codes(const void* q, int32_t n_tokens, int32_t n_q_heads, int32_t head_dim,
                              int8_t* q_codes, float* q_scales, void* stream) {
  if (!q || !q_codes || !q_scales || n_tokens <= 0 || n_q_heads <= 0) return KVQ_ERR_INVALID_ARG;
  if (head_dim != 128 && head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(q_codes) || !aligned4(q_scales)) return KVQ_ERR_MISALIGNED;
  kvq::PrefillArgs a{};
  a.head_dim = head_dim;
  a.q = q;
  a.n_tokens = n_tokens;
  a.n_q_heads = n_q_heads;
  a.q_codes = q_codes;
  a.q_scales = q_scales;
  a.status = status_ptr();
  return cuda_status(kvq::launch_prefill_q_quant(a, static_cast<cudaStream_t>(stream)));
}

int kvq_debug_prefill_qk_int32(const kvq_cache* cache, const int8_t* q_codes, const float* q_scales,
                               int32_t n_tokens, int32_t n_q_heads, int32_t history_len,
                               const int32_t* block_table_row, int32_t n_blocks_row, float softmax_scale,
                               int32_t split_tiles, int32_t q_head, int32_t q0, int32_t k0, int32_t nk,
                               int32_t* s_out, float* out, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!q_codes || !q_scales || !block_table_row || !s_out || !out) return KVQ_ERR_INVALID_ARG;
  if (n_tokens <= 0 || n_q_heads <= 0 || history_len < 0 || n_blocks_row <= 0) return KVQ_ERR_INVALID_ARG;
  if (n_q_heads % cache->n_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || !std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if (static_cast<long long>(history_len) + n_tokens > static_cast<long long>(n_blocks_row) * KVQ_BLOCK_SIZE)
    return KVQ_ERR_INVALID_ARG;
  // the window: one unit (query tile q0 / 128 of q_head) and whole key tiles it computes
  if (q_head < 0 || q_head >= n_q_heads || q0 < 0 || q0 >= n_tokens || q0 % 128 != 0) return KVQ_ERR_INVALID_ARG;
  const long long unit_tiles = (static_cast<long long>(history_len) + std::min(q0 + 127, n_tokens - 1)) / 128 + 1;
  if (k0 < 0 || nk <= 0 || k0 % 128 != 0 || nk % 128 != 0 || k0 + static_cast<long long>(nk) > 128 * unit_tiles)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q_codes) || !aligned4(q_scales) || !aligned16(out) || !aligned16(s_out) || !aligned4(block_table_row))
    return KVQ_ERR_MISALIGNED;
  const size_t need = kvq_prefill_workspace_bytes(n_tokens, n_q_heads, cache->n_kv_heads, history_len,
                                                  cache->head_dim);
  if (!workspace || workspace_bytes < need) return KVQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KVQ_ERR_MISALIGNED;
  kvq::PrefillArgs a = prefill_args(cache, nullptr, n_tokens, n_q_heads, history_len, block_table_row,
                                    n_blocks_row, softmax_scale, out, workspace);
  if (split_tiles >= 0) {
    // a forced split: every lead segment keeps at least one tile, as the automatic choice does
    const long long shortest = (static_cast<long long>(history_len) + std::min(127, n_tokens - 1)) / 128 + 1;
    const bool can = kvq::prefill_workspace(n_tokens, n_q_heads, cache->n_kv_heads, history_len, cache->head_dim)
                         .can_split;
    if (split_tiles > 0 && (!can || split_tiles > shortest - 1)) return KVQ_ERR_INVALID_ARG;
    a.split_tail = split_tiles;
  }
  a.q_codes = const_cast<int8_t*>(q_codes);
  a.q_scales = const_cast<float*>(q_scales);
  a.dbg_q_head = q_head;
  a.dbg_q0 = q0;
  a.dbg_k0 = k0;
  a.dbg_nk = nk;
  a.dbg_s_out = s_out;
  cudaError_t e = kvq::launch_prefill_qk_debug(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return e == cudaErrorNotSupported ? KVQ_ERR_UNSUPPORTED : KVQ_ERR_CUDA;
  return KVQ_OK;
}

}  // extern "C"
