// kvq_launch.h — internal launcher interface between the C ABI (api.cu) and the kernels.
// Host-side validation happens in api.cu; the launchers assume valid arguments.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "kvq.h"

namespace kvq {

struct QuantWriteArgs {
  int8_t* k;
  int8_t* v;
  float* k_scale;
  float* v_scale;
  int num_blocks, n_kv_heads, head_dim;
  const void* k_new;
  const void* v_new;
  int n_tokens;
  const int32_t* seq_idx;
  const int32_t* pos;
  const int32_t* block_table;
  int num_seqs, max_blocks_per_seq;
  unsigned int* status;
};
cudaError_t launch_quant_write(const QuantWriteArgs& a, cudaStream_t stream);

// Fused producer: RoPE on Q and K, the quantisation rule on Q, K and V; K/V into the cache.
struct RopeQuantArgs {
  QuantWriteArgs kv;      // the cache, k_new / v_new, tokens, slots
  const void* q;          // bf16 [T][Hq][D] or nullptr
  int n_q_heads;
  const float* cos_sin;   // fp32 [max_pos][rotary_dim]: cos of rotary_dim / 2 frequencies, then sin
  int max_pos, rotary_dim;
  int8_t* q_codes;        // [T][Hq][D] or nullptr
  float* q_scales;        // [T][Hq] or nullptr
  uint16_t* q_rot;        // bf16 [T][Hq][D] or nullptr
  int q_heads_per_warp;   // set by launch_rope_quant_write
};
cudaError_t launch_rope_quant_write(const RopeQuantArgs& a, cudaStream_t stream);

// Decode: nq query rows per sequence (1 for plain decode; row i sees keys
// t < ctx - nq + 1 + i).  Stage 1 (both routes) walks a key range of one (sequence, KV head)
// for all G * nq rows; the single-CTA route writes `out` directly, the split route writes
// partials that stage 2 merges.
struct DecodeArgs {
  int8_t* k;          // the cache (written only by the fused step)
  int8_t* v;
  float* k_scale;
  float* v_scale;
  int num_blocks, n_kv_heads, head_dim;
  const void* q;  // bf16 [B][nq][Hq][D]
  int batch, nq, n_q_heads;
  const int32_t* block_table;
  int max_blocks_per_seq;
  const int32_t* ctx_lens;
  int max_ctx;
  float softmax_scale;
  // fused step: bf16 [B][nq][Hkv][D] K / V of each sequence's nq newest tokens, quantised
  // into the cache by stage 1 before it reads their page; nullptr for attention only
  const void* k_new;
  const void* v_new;
  float* out;          // fp32 [B][nq][Hq][D]
  float* part_acc;     // fp32 [B][nq][Hq][n_split][D]  (split route)
  float* part_stats;   // fp32 [B][nq][Hq][n_split][4]  (split route: m_s, m_z, l, unused)
  int split_rows;      // keys per split (split route); ignored by the single route
  int n_split;         // splits per sequence in the grid (split route)
  unsigned int* status;
  cudaEvent_t ev_begin;  // optional events around the stage-1 launch
  cudaEvent_t ev_end;
  // bounded waits: budget in SM clock cycles; fault: test-only injection (kvq_debug_fault_inject),
  // 1 = CTA 0's first team does not issue the copy of its second page
  long long wait_budget;
  int fault;
};
enum class DecodeRoute { kSingle = 1, kSplit = 2 };
// Test-only fault injection and wait budget of the kernels launched next (kvq_debug_fault_inject).
int debug_fault_mode();
long long debug_wait_budget();
size_t decode_workspace_bytes(int batch, int n_q_heads, int max_ctx, int head_dim, int split_rows);
// The route, split size and workspace bytes a decode call with these (checked) arguments takes:
// the automatic split size of this GPU when opts->split_rows is 0.  A kvq_status.
struct DecodePlan {
  bool split;
  int split_rows, n_split;
  size_t bytes;
};
int decode_plan(const kvq_cache* cache, int32_t batch, int32_t nq, int32_t n_q_heads, int32_t max_ctx,
                const kvq_decode_opts* opts, DecodePlan* plan);
cudaError_t launch_decode(const DecodeArgs& a, DecodeRoute route, cudaStream_t stream, int* launched);
// the stage-1 kernel's K/V stream alone, split route geometry (kvq_debug_stream_floor)
cudaError_t launch_stream_floor(const DecodeArgs& a, cudaStream_t stream);

struct SparseArgs {
  const int8_t* k;
  const int8_t* v;
  const float* k_scale;
  const float* v_scale;
  int num_blocks, n_kv_heads, head_dim;
  const void* q;  // bf16 [N][Hq][D]
  int n_queries, n_q_heads;
  const int32_t* cell_offsets;
  const int32_t* cells;
  const int32_t* block_table_row;
  int n_blocks_row;
  float softmax_scale;
  float* out;
  uint8_t* records;  // workspace: gather records [n_blocks_row][Hkv][16][2D + 16]
  unsigned int* status;
  long long wait_budget;  // SM clock cycles a bounded wait may take
  int fault;              // test-only fault injection (kvq_debug_fault_inject), 0: none
};
size_t sparse_workspace_bytes(int n_blocks_row, int n_kv_heads, int head_dim);
cudaError_t launch_sparse(const SparseArgs& a, cudaStream_t stream);

struct PrefillArgs {
  int8_t* k;          // the cache (written only by the first-chunk pass)
  int8_t* v;
  float* k_scale;
  float* v_scale;
  int num_blocks, n_kv_heads, head_dim;
  const void* q;  // bf16 [T][Hq][D]
  int n_tokens, n_q_heads, history_len;
  const int32_t* block_table_row;
  int n_blocks_row;
  float softmax_scale;
  float* out;        // fp32 [T][Hq][D]
  int8_t* q_codes;   // workspace int8 [T][Hq][D]
  float* q_scales;   // workspace fp32 [T][Hq]
  // first chunk in high precision: fp16 Q (q * 2^e per row) in place of the codes, and the
  // chunk's own bf16 K/V [T][Hkv][D] (also written into the int8 cache by the pre-pass)
  uint16_t* q_f16;   // workspace fp16 [T][Hq][D]
  const void* k_src;
  const void* v_src;
  // workspace: K/V of every (KV head, 128-key tile) widened to the attention kernel's
  // shared-memory operand image, and the tiles' key / value scales
  int n_kv_tiles;
  uint8_t* kw;       // [Hkv][n_kv_tiles][D/64 pieces of 16 KB]
  uint8_t* vw;       // [Hkv][n_kv_tiles][D/64 pieces of 16 KB]
  float* skw;        // [Hkv][n_kv_tiles][128]
  float* svw;        // [Hkv][n_kv_tiles][128]
  unsigned int* status;
  // key-range split (int8 path): with split_tail > 0 each unit (128 query rows, query head) runs
  // as two CTAs, a lead segment (key tiles [0, js)) and a tail segment (tiles [js, n_tiles)),
  // js = min(n_tiles - split_tail, history_len / 128); whichever finishes first leaves its
  // numerator and (m, l) in part / part_ml, and the other merges them into out
  int split_tail;
  float* part;               // workspace fp32 [units][128][D]
  float* part_ml;            // workspace fp32 [units][128][2]
  unsigned int* part_cnt;    // workspace [units]: segments arrived (zeroed by the widen pass)
  unsigned int* part_ready;  // workspace [units]: the first segment's values are written
  // debug QK tile (kvq_debug_prefill_qk_int32)
  int dbg_q_head, dbg_q0, dbg_k0, dbg_nk;
  int32_t* dbg_s_out;
  // bounded waits: budget in SM clock cycles; fault: test-only injection (kvq_debug_fault_inject),
  // 2 = the producer of attention CTA 0 does not issue its fourth piece copy
  long long wait_budget;
  int fault;
};
struct PrefillWorkspace {
  int n_kv_tiles;
  long long off_q_scales, off_kw, off_vw, off_skw, off_svw;
  long long off_part, off_part_ml, off_part_flags;  // only when the key range may be split
  bool can_split;
  long long bytes;
};
PrefillWorkspace prefill_workspace(int n_tokens, int n_q_heads, int n_kv_heads, int history_len, int head_dim,
                                   int q_elem_bytes = 1);
// Tail length (in 128-key tiles) of the key-range split of the int8 prefill at this shape on
// n_sms SMs, 0 for no split: the choice that minimises the modelled finish time of the
// longest-first dispatch (one attention CTA per SM).
int prefill_split_tail(int n_tokens, int n_q_heads, int history_len, int n_sms);
cudaError_t launch_prefill_q_quant(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);
// first chunk: Q to fp16, the chunk's K/V into the cache and into fp16 operand pieces, then the
// attention in high precision (fp16 P)
cudaError_t launch_prefill_first(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_qk_debug(const PrefillArgs& a, cudaStream_t stream);

}  // namespace kvq
