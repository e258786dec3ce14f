/*
 * kvq.h — C ABI of libkvq: attention over an INT8-quantised, paged K/V cache,
 * hand-written CUDA for NVIDIA GB300 (sm_103a).
 *
 * Sources of the method (cited by page title and section):
 *   [DCU]   "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" (INT8 KV and INT8
 *           MMAC attention on a gfx936 DCU), sections 1.1-1.3, 2.1-2.3, 3.2-3.3, 5.4.
 *   [DOT4]  "dot4-flash-attention" README (INT8 DOT4 FlashAttention for llama.cpp HIP):
 *           route table, "Tile Inner Loop (pseudocode)", split-K stage 1 + stage 2.
 *   [QSA]   "#3381 [Engine] STRATA_PROMPT_ATTN_RDNA2=1 ... prompt QSA attention without
 *           the decode kernel's split and merge": sections "Problem and result", "Approach".
 *   [RDNA4] "ROCm/RDNA4 (gfx1201) vLLM: native HIP kernels ...": "Segments, split-K and
 *           tile shape", "The reduce is not free".
 *
 * Conventions shared by every call
 *   - Every pointer argument named as "device" is device memory of the current CUDA
 *     device, owned by the caller.  The library allocates nothing, keeps no per-call
 *     state and never synchronises, except kvq_device_status().
 *   - Zero-copy host buffers: the decode calls (kvq_attn_decode_int8kv,
 *     kvq_attn_verify_int8kv, kvq_decode_step_int8kv) also take q, k_new, v_new and out in
 *     page-locked host memory mapped into the device's address space (cudaHostAlloc, or
 *     cudaHostRegister with the mapped flag, under unified addressing: the pointer the host
 *     uses is the one the device uses).  The kernels then read the step's inputs and write
 *     its result across the host link themselves, overlapped with the K/V stream, so a
 *     step needs no separate host-device copies.  kvq_device_accessible() tells such a
 *     pointer from pageable host memory, which a kernel cannot read: the library cannot
 *     detect that case on the device, so a caller that may hold either checks first.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - bf16 tensors are passed as raw 16-bit patterns (const void*).
 *   - Outputs of the attention calls are fp32 (a bf16 output would add up to 2^-9
 *     relative rounding error by itself).
 *   - Return value: a kvq_status.  Host-side checks run before any launch; on an error
 *     nothing is launched and no output is touched.  Problems that only the device can
 *     see (a block-table entry out of range, a cell index out of range, a bounded wait
 *     that ran out) set bits in the device status word (KVQ_DEV_*), the offending unit
 *     is skipped (its output is left as zeros where the call writes one), and the
 *     kernel never traps.  Read and clear those bits with kvq_device_status().
 *
 * Cache layout in HBM (one layer; KVQ_BLOCK_SIZE = 16 tokens per page).  Token at
 * logical position p of sequence s lives in physical page
 * block_table[s * max_blocks_per_seq + p / 16], slot p % 16.  The K and V layouts are
 * the ones printed in [DCU] §2.3: K in 16-element head-dimension chunks with the
 * tokens of a chunk adjacent, V token-contiguous per head dimension.  Scales are
 * stored head-major ([page][head][slot]) rather than [page][slot][head] so that the
 * 16 scales of one (page, head) are one contiguous 64-byte run.
 *     k       int8  [num_blocks][n_kv_heads][head_dim/16][16 slots][16]
 *     v       int8  [num_blocks][n_kv_heads][head_dim][16 slots]
 *     k_scale fp32  [num_blocks][n_kv_heads][16 slots]
 *     v_scale fp32  [num_blocks][n_kv_heads][16 slots]
 * One (page, head) of K or V is head_dim*16 contiguous bytes (4096 B at head_dim 256).
 * Per token and layer this is 2*Hkv*D + 2*Hkv*4 bytes: 2080 B at 4 KV heads x 256
 * against 4096 B for bf16 K/V ([DCU] §1.1).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_ABI_VERSION 1
#define KVQ_BLOCK_SIZE 16          /* tokens per cache page */
#define KVQ_PV_TILE 128            /* keys per P re-quantisation tile in prefill */

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, Hq % Hkv != 0, ... */
  KVQ_ERR_UNSUPPORTED = 2, /* head_dim not in {128, 256}, block_size != 16, ... */
  KVQ_ERR_MISALIGNED = 3,  /* a device pointer is not 16-byte aligned */
  KVQ_ERR_WORKSPACE = 4,   /* workspace missing or smaller than the *_workspace_bytes size */
  KVQ_ERR_CUDA = 5         /* a launch failed (cudaGetLastError after the launch) */
} kvq_status;

/*
 * kvq_device_accessible — 1 when p can be dereferenced by the kernels of the current device:
 * device memory, managed memory, or page-locked host memory whose device address is p itself;
 * 0 otherwise (NULL, pageable host memory, no device).  Host only, no synchronisation.
 */
int32_t kvq_device_accessible(const void* p);

/* Device status bits (sticky until read by kvq_device_status). */
#define KVQ_DEV_BAD_BLOCK 0x1u /* a block-table entry is outside [0, num_blocks) */
#define KVQ_DEV_BAD_POS 0x2u   /* a position / length exceeds what the block table maps */
#define KVQ_DEV_TIMEOUT 0x4u   /* a bounded mbarrier wait ran out; the CTA returned early */
#define KVQ_DEV_BAD_CELL 0x8u  /* a sparse cell index is negative or past the mapped range */
#define KVQ_DEV_BAD_SEQ 0x10u  /* a seq_idx is outside [0, num_seqs) */

typedef struct kvq_cache {
  int8_t* k;          /* device, layout above */
  int8_t* v;          /* device, layout above */
  float* k_scale;     /* device, layout above */
  float* v_scale;     /* device, layout above */
  int32_t num_blocks; /* physical pages */
  int32_t block_size; /* must be KVQ_BLOCK_SIZE */
  int32_t n_kv_heads;
  int32_t head_dim;   /* 128 or 256 */
} kvq_cache;

/*
 * kvq_quant_write — fused per-(token, KV head) absmax quantisation of new K and V rows
 * into the paged int8 cache, codes and scales in one kernel ([DCU] §2.1 rule, §2.2
 * fused producer, §2.3 layout).  For every row x (head_dim values of one token and one
 * KV head, K and V separately):
 *     amax = max |x|;  scale = amax / 127 (fp32, IEEE round-to-nearest);
 *     code = clamp(rint(x / scale), -127, 127) (fp32 IEEE division, ties to even);
 *     amax == 0 gives scale 0 and all-zero codes.
 *   k_new, v_new : device bf16 [n_tokens][n_kv_heads][head_dim]
 *   seq_idx, pos : device int32 [n_tokens]; token i goes to sequence seq_idx[i],
 *                  logical position pos[i]
 *   block_table  : device int32 [num_seqs][max_blocks_per_seq]
 * A token whose seq_idx, position or page is out of range is skipped and sets
 * KVQ_DEV_BAD_SEQ / KVQ_DEV_BAD_POS / KVQ_DEV_BAD_BLOCK.  Tokens must target distinct
 * slots (two tokens writing one slot race).
 */
int kvq_quant_write(const kvq_cache* cache, const void* k_new, const void* v_new,
                    int32_t n_tokens, const int32_t* seq_idx, const int32_t* pos,
                    const int32_t* block_table, int32_t num_seqs,
                    int32_t max_blocks_per_seq, void* stream);

/*
 * kvq_rope_quant_write — the fused producer ([DCU] §2.2: one kernel reads Q/K/V, applies
 * RoPE to Q and K, reduces absmax, quantises, writes the paged int8 K/V and their scales,
 * and quantises Q once for the attention that follows).  For token i at position pos[i]:
 *   RoPE (the pages name apply_rope(q, position); the reading is the rotate-half form over
 *   the first r = rotary_dim dims with the caller's table row cs = cos_sin[pos[i]], the cos
 *   of the r/2 frequencies then their sin), in fp32 with exactly these roundings:
 *     dim j < r/2:       out = fma(x_j, cs[j], -(x_{j+r/2} * cs[r/2 + j]))
 *     dim j + r/2:       out = fma(x_{j+r/2}, cs[j], x_j * cs[r/2 + j])
 *     dims >= r unchanged;
 *   then each K row (rotated), V row (not rotated) and Q row (rotated) is quantised by the
 *   kvq_quant_write rule.  K/V codes and scales go to the token's slot as in
 *   kvq_quant_write; Q gives q_codes, q_scales and the rotated row rounded to bf16 (q_rot).
 *   q        : device bf16 [n_tokens][n_q_heads][head_dim], or NULL (no Q outputs)
 *   cos_sin  : device fp32 [max_pos][rotary_dim], 16-byte aligned
 *   rotary_dim: even, <= head_dim, (rotary_dim / 2) a multiple of head_dim / 32
 *   q_codes  : device int8 [n_tokens][n_q_heads][head_dim] or NULL (8-byte aligned)
 *   q_scales : device fp32 [n_tokens][n_q_heads] or NULL
 *   q_rot    : device bf16 [n_tokens][n_q_heads][head_dim] or NULL (16-byte aligned)
 * A token whose position is outside [0, max_pos) writes no K/V (KVQ_DEV_BAD_POS) and zero
 * Q outputs; an invalid sequence or page skips the K/V write as in kvq_quant_write.
 */
int kvq_rope_quant_write(const kvq_cache* cache, const void* q, int32_t n_q_heads,
                         const void* k_new, const void* v_new, int32_t n_tokens,
                         const int32_t* seq_idx, const int32_t* pos, const int32_t* block_table,
                         int32_t num_seqs, int32_t max_blocks_per_seq, const float* cos_sin,
                         int32_t max_pos, int32_t rotary_dim, int8_t* q_codes, float* q_scales,
                         void* q_rot, void* stream);

/* Options of kvq_attn_decode_int8kv (pass NULL for the defaults). */
typedef struct kvq_decode_opts {
  int32_t split_rows;      /* keys per split in the split route, a multiple of 16; 0 -> sized to
                            * the GPU by kvq_decode_auto_split_rows */
  int32_t route_threshold; /* > 0: max_ctx <= threshold -> single-CTA route ([DOT4] route table
                            * uses 2048); 0 -> automatic: the split route whenever the split size
                            * leaves more than one split of max_ctx, else the single-CTA route */
  int32_t force_route;     /* 0 auto, 1 single CTA per (sequence, KV head), 2 split-K */
  /* Optional profiling hooks: two cudaEvent_t (as void*) recorded on `stream` right before
   * and right after the stage-1 (K/V streaming) kernel launch; NULL to skip. */
  void* stage1_event_begin;
  void* stage1_event_end;
  /* Optional: receives the number of kernels the call launched (1: the single-CTA route; 2: the
   * split route's stage 1 and its merge).  NULL to skip. */
  int32_t* launches;
} kvq_decode_opts;

/* Workspace (bytes) the split route of kvq_attn_decode_int8kv needs; 0 when the call
 * will take the single-CTA route.  With opts->split_rows == 0 it is the bound for the
 * smallest split the automatic rule can choose (64 keys), so it does not depend on the GPU
 * (and with the automatic route it is nonzero whenever max_ctx exceeds that split). */
size_t kvq_decode_workspace_bytes(int32_t batch, int32_t n_q_heads, int32_t max_ctx,
                                  int32_t head_dim, const kvq_decode_opts* opts);

/*
 * kvq_attn_decode_int8kv — one query per sequence over its int8 paged K/V
 * ([DCU] §3.3 decode data flow; [DOT4] route table and split-K stage 1 + stage 2).
 *   out[b][h][:] = sum_t softmax_t(s) * v^[t],   s[t] = softmax_scale * q[b][h] . k^[t],
 *   k^[t] = k_code[t] * k_scale[t] (per token and KV head), same for v^, t < ctx_lens[b],
 *   KV head of query head h = h / (n_q_heads / n_kv_heads) (GQA).
 * The int8 codes are consumed directly; no dequantised copy is written.  Routes: one CTA per
 * (sequence, KV head) walks all keys (single-CTA route), or stage 1 runs one CTA per
 * (split_rows-key split, KV head, sequence) and writes a partial (max, sum, acc[head_dim]) per
 * query head, and stage 2 merges the partials with the log-sum-exp rule (split route).  The
 * default (route_threshold 0) takes the split route whenever the split size leaves more than
 * one split: on a GPU that one CTA per (sequence, KV head) does not fill, splitting even a
 * 1024-key context is faster ([DOT4]'s table switches at 2048 keys for a smaller GPU).
 *   q          : device bf16 [batch][n_q_heads][head_dim]
 *   block_table: device int32 [batch][max_blocks_per_seq]
 *   ctx_lens   : device int32 [batch], each in [0, max_ctx]; ctx 0 gives zeros; a ctx above
 *                max_ctx (or above what the sequence's block-table row maps) is clamped to it on
 *                both routes and sets KVQ_DEV_BAD_POS
 *   max_ctx    : host upper bound of ctx_lens (sizes the grid and the workspace)
 *   out        : device fp32 [batch][n_q_heads][head_dim]
 *   workspace  : device, >= kvq_decode_workspace_bytes(...), 16-byte aligned; its
 *                contents on entry do not matter
 * The GQA group (n_q_heads / n_kv_heads) may be 1..16; a larger one is KVQ_ERR_UNSUPPORTED.
 */
/*
 * kvq_decode_auto_split_rows — the split size the split route uses when opts->split_rows is
 * 0, for a GPU with n_sms SMs (pure host arithmetic).  Stage 1 holds one CTA per SM at head_dim
 * 256 and two at head_dim 128: slots = n_sms * (1 or 2).
 *   units = batch * n_kv_heads, pages = ceil(max_ctx / 16).
 *   If units * ceil(pages / 32) > 2 * slots (at 512-key splits the grid is over two waves),
 *   the split takes clamp(units * pages / (4 * slots), 32, 128) pages: longer splits amortise
 *   each CTA's start-up over more pages.
 *   Otherwise the split takes max(4, ceil(pages / floor(slots / units))) pages: the grid fills
 *   every SM in one wave.
 * Returns keys (pages * 16); 0 if an argument is not positive or head_dim is not 128 / 256.
 * The source pages use a fixed 512 ([DOT4] route table); any split size gives the same result
 * up to fp32 rounding.
 */
int32_t kvq_decode_auto_split_rows(int32_t batch, int32_t n_kv_heads, int32_t head_dim, int32_t max_ctx,
                                   int32_t n_sms);

int kvq_attn_decode_int8kv(const kvq_cache* cache, const void* q, int32_t batch,
                           int32_t n_q_heads, const int32_t* block_table,
                           int32_t max_blocks_per_seq, const int32_t* ctx_lens,
                           int32_t max_ctx, float softmax_scale, float* out,
                           void* workspace, size_t workspace_bytes,
                           const kvq_decode_opts* opts, void* stream);

/*
 * kvq_attn_decode_int8kv_noalloc — kvq_attn_decode_int8kv for callers that cannot allocate
 * device memory.  The source pages have no counterpart of this call; it exists for callers
 * that may not call cudaMalloc where they run decode (a region whose memory plan is fixed in
 * advance, a plugin host that only hands out the tensors it owns, a runtime that reserved all
 * device memory at start-up) and so cannot provide the split route's workspace.
 *   Same arguments and results as kvq_attn_decode_int8kv, without workspace / workspace_bytes:
 *   the split-K partials live in a fixed scratch array of KVQ_NOALLOC_SCRATCH_BYTES bytes
 *   inside the library, which every GPU that loads the library holds until the process exits.
 *   The call allocates nothing.  A problem whose partials, at the split size the call takes
 *   (kvq_decode_auto_split_rows for this GPU unless opts sets split_rows), need more than
 *   KVQ_NOALLOC_SCRATCH_BYTES is rejected with KVQ_ERR_WORKSPACE before any launch.
 *   The first call on a device looks up the scratch array's device address for that device
 *   (a one-time host-side set-up); make that first call before any stream capture.  The
 *   address, like the device status word's, stays valid for the life of the device's context:
 *   after a cudaDeviceReset the library must be unloaded and loaded again.
 *   All calls share the one array: calls that overlap on the GPU (different streams, or
 *   different host threads on one device) race and corrupt each other's results.  The
 *   array keeps the last call's contents; every call writes the partials it reads, so
 *   nothing in it has to start at zero.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u << 20)
int kvq_attn_decode_int8kv_noalloc(const kvq_cache* cache, const void* q, int32_t batch,
                                   int32_t n_q_heads, const int32_t* block_table,
                                   int32_t max_blocks_per_seq, const int32_t* ctx_lens,
                                   int32_t max_ctx, float softmax_scale, float* out,
                                   const kvq_decode_opts* opts, void* stream);

/* Most query rows one (sequence, KV head) of kvq_attn_verify_int8kv can hold:
 * (n_q_heads / n_kv_heads) * n_rows <= KVQ_VERIFY_MAX_ROWS. */
#define KVQ_VERIFY_MAX_ROWS 48

/* Workspace (bytes) the split route of kvq_attn_verify_int8kv needs: the decode workspace of
 * batch * n_rows query rows; 0 when the call takes the single-CTA route or an argument is
 * not positive. */
size_t kvq_verify_workspace_bytes(int32_t batch, int32_t n_rows, int32_t n_q_heads, int32_t max_ctx,
                                  int32_t head_dim, const kvq_decode_opts* opts);

/*
 * kvq_attn_verify_int8kv — decode with n_rows query rows per sequence: the verify step of
 * speculative / multi-token-prediction decoding ([DOT4] "Future Work": MTP verify runs
 * nq = 2-4 query rows per sequence; "ROCm/RDNA4 (gfx1201) vLLM ..." row-shape routing:
 * spec-verify decode with 2-6 rows goes to a multi-row kernel).  The last n_rows tokens of
 * each sequence are the drafted tokens being verified; their K/V must already be in the
 * cache (kvq_quant_write or kvq_rope_quant_write).  With c = ctx_lens[b], row i sits at
 * position c - n_rows + i and attends causally:
 *   out[b][i][h][:] = sum_t softmax_t(s) * v^[t],  s[t] = softmax_scale * q[b][i][h] . k^[t],
 *   over keys t < min(c, c - n_rows + 1 + i); a row with no key gives zeros.
 * n_rows = 1 is kvq_attn_decode_int8kv.  Same routes, options, K/V traffic and precision as
 * kvq_attn_decode_int8kv: every K/V page is read once for all n_rows rows of its sequence.
 *   q          : device bf16 [batch][n_rows][n_q_heads][head_dim]
 *   out        : device fp32 [batch][n_rows][n_q_heads][head_dim]
 *   workspace  : >= kvq_verify_workspace_bytes(...), 16-byte aligned
 *   other arguments as kvq_attn_decode_int8kv.
 * KVQ_ERR_UNSUPPORTED when (n_q_heads / n_kv_heads) * n_rows > KVQ_VERIFY_MAX_ROWS, the GQA
 * group exceeds 16, or batch * n_rows > 65535.
 */
int kvq_attn_verify_int8kv(const kvq_cache* cache, const void* q, int32_t batch, int32_t n_rows,
                           int32_t n_q_heads, const int32_t* block_table, int32_t max_blocks_per_seq,
                           const int32_t* ctx_lens, int32_t max_ctx, float softmax_scale, float* out,
                           void* workspace, size_t workspace_bytes, const kvq_decode_opts* opts,
                           void* stream);

/*
 * kvq_decode_step_int8kv — one decode step in one call: write each sequence's n_new newest
 * tokens into the cache, then attend with their n_new query rows ([DCU] §4.2 times decode
 * together with the producer that writes the new token; §2.2 the producer's quantise-and-
 * write).  With c = ctx_lens[b] (the length including the new tokens), token j of sequence b
 * sits at position c - n_new + j; the call has exactly the effect of
 *   kvq_quant_write(k_new, v_new, seq_idx = b, pos = c - n_new + j)   (the same codes and
 *   scales, bit for bit), then
 *   kvq_attn_verify_int8kv(q, ...)  (kvq_attn_decode_int8kv when n_new = 1),
 * but the write runs inside the attention kernel: the warp that is about to copy a page holding
 * new tokens quantises and stores them first, so the step launches no separate write kernel.
 *   k_new, v_new : device bf16 [batch][n_new][n_kv_heads][head_dim], 16-byte aligned
 *   q            : device bf16 [batch][n_new][n_q_heads][head_dim]
 *   out          : device fp32 [batch][n_new][n_q_heads][head_dim]
 *   workspace    : >= kvq_verify_workspace_bytes(batch, n_new, ...)
 *   other arguments as kvq_attn_verify_int8kv.
 * A sequence with c < n_new or c past what its block-table row maps writes nothing
 * (KVQ_DEV_BAD_POS); a page id outside [0, num_blocks) is skipped (KVQ_DEV_BAD_BLOCK).  The
 * new tokens of different sequences must map to distinct slots.
 */
int kvq_decode_step_int8kv(const kvq_cache* cache, const void* k_new, const void* v_new, const void* q,
                           int32_t batch, int32_t n_new, int32_t n_q_heads, const int32_t* block_table,
                           int32_t max_blocks_per_seq, const int32_t* ctx_lens, int32_t max_ctx,
                           float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                           const kvq_decode_opts* opts, void* stream);

/* Workspace (bytes) of kvq_attn_prefill_int8 for a chunk of n_tokens queries after
 * history_len keys: the int8 Q codes and their fp32 scales, and the K/V codes of every
 * (KV head, 128-key tile) of the history_len + n_tokens keys widened once to fp16 in the
 * attention kernel's shared-memory operand layout (2 * 2 * head_dim bytes per key and KV
 * head), with the tiles' key and value scales.  With history_len >= 128 and at most 16384
 * units of 128 query rows and one query head, also room for the key-range split
 * (kvq_prefill_split_tiles): per unit, 128 rows of head_dim + 2 floats and two counters (more
 * units never split).  0 if an argument is not positive (history_len may be 0). */
size_t kvq_prefill_workspace_bytes(int32_t n_tokens, int32_t n_q_heads, int32_t n_kv_heads,
                                   int32_t history_len, int32_t head_dim);

/*
 * kvq_prefill_split_tiles — the key-range split kvq_attn_prefill_int8 uses at this shape on a
 * GPU with n_sms SMs: 0 (each unit of 128 query rows and one query head is one CTA over all
 * its keys), or r > 0 (each unit runs as two CTAs: a lead segment over key tiles [0, js) and a
 * tail over [js, n_tiles), js = min(n_tiles - r, history_len / 128); the tails fill the SMs
 * that the last wave of lead segments leaves idle, and the segment that finishes second
 * merges the two partial softmax results).  Chosen by simulating the dispatch of the CTAs
 * onto one slot per SM; never > 0 when history_len < 128.  Host only, no device call.
 */
int32_t kvq_prefill_split_tiles(int32_t n_tokens, int32_t n_q_heads, int32_t history_len, int32_t n_sms);

/*
 * kvq_attn_prefill_int8 — a chunk of n_tokens causal queries of one sequence against
 * its history plus the chunk itself, all from the int8 cache, in one online softmax
 * ([DCU] §3.2 non-first prefill chunk; §1.3 and §3.3 INT8 QK / INT8 PV).
 *   Query i sits at position history_len + i and sees keys t <= history_len + i.
 *   Q is quantised per (token, query head) by the kvq_quant_write rule.
 *   S[i][t] = sum_d q_code[i][d] * k_code[t][d]  (exact integer),
 *   score = S * q_scale[i] * k_scale[t] * softmax_scale,
 *   p = exp(score - m) (online max m), l = sum of p (unquantised),
 *   w = p * v_scale[t]; per (query row, KVQ_PV_TILE keys at absolute multiples of 128):
 *   ps = max w / 127, c = rint(w / ps) in [0, 127];
 *   out = (sum over tiles of ps * sum_t c * v_code[t]) / l.
 * The running maximum cancels in w / ps, so the codes are decided in fp32 relative to the
 * tile's own maximum score (exp2 by a fixed polynomial, so that a CPU implementation can
 * reproduce every decision); the running maximum only rescales ps and the tile's sum of p.  Each
 * tile's codes therefore depend on that tile alone, and the call may split a unit's key range
 * between two CTAs (kvq_prefill_split_tiles) without changing any code; the result does not
 * depend on which CTA finishes first, and the workspace's contents on entry do not matter.
 * The integer contractions run on the tensor cores with int8 codes widened to
 * integer-valued fp16 (exact: every partial sum is an integer below 2^24).  The chunk's
 * own K/V must already be in the cache (kvq_quant_write).
 *   q              : device bf16 [n_tokens][n_q_heads][head_dim]
 *   block_table_row: device int32 [n_blocks_row], covering history_len + n_tokens keys
 *   out            : device fp32 [n_tokens][n_q_heads][head_dim]
 *   softmax_scale  : finite and > 0, else KVQ_ERR_INVALID_ARG
 *   workspace      : device, >= kvq_prefill_workspace_bytes(n_tokens, n_q_heads,
 *                    cache->n_kv_heads, history_len, cache->head_dim), 16-byte aligned
 */
int kvq_attn_prefill_int8(const kvq_cache* cache, const void* q, int32_t n_tokens,
                          int32_t n_q_heads, int32_t history_len,
                          const int32_t* block_table_row, int32_t n_blocks_row,
                          float softmax_scale, float* out, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * kvq_attn_prefill_int8_qcodes — kvq_attn_prefill_int8 with Q already quantised (by
 * kvq_rope_quant_write, [DCU] §2.2 "Query quantised once, reused"): the same attention, with
 *   q_codes : device int8 [n_tokens][n_q_heads][head_dim] (16-byte aligned)
 *   q_scales: device fp32 [n_tokens][n_q_heads]
 * in place of bf16 q.  Same workspace.
 */
int kvq_attn_prefill_int8_qcodes(const kvq_cache* cache, const int8_t* q_codes, const float* q_scales,
                                 int32_t n_tokens, int32_t n_q_heads, int32_t history_len,
                                 const int32_t* block_table_row, int32_t n_blocks_row,
                                 float softmax_scale, float* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Workspace (bytes) of kvq_attn_sparse_int8kv: one gather record per (logical page, KV head,
 * slot) of the sequence, 2 * head_dim + 16 bytes each (the token's K codes, V codes, both
 * scales and a page-valid word).  0 if an argument is not positive or head_dim is not 128 / 256. */
size_t kvq_sparse_workspace_bytes(int32_t n_blocks_row, int32_t n_kv_heads, int32_t head_dim);

/*
 * kvq_attn_sparse_int8kv — sparse prompt attention ([QSA] "Problem and result",
 * "Approach"): one CTA per (query, KV head) walks the query's list of selected cells with
 * an online softmax, no scratch in HBM and no merge pass; the GQA group shares each gathered
 * K/V row.  A pre-pass first rewrites the sequence's pages into token-major gather records
 * in the workspace, so that each selected cell is one contiguous copy.
 *   out[i][h] = sum_{t in cells(i)} softmax_t(s) * v^[t], s as in decode.
 *   q           : device bf16 [n_queries][n_q_heads][head_dim]
 *   cell_offsets: device int32 [n_queries + 1]; cells of query i are
 *                 cells[cell_offsets[i] .. cell_offsets[i+1]), logical positions, sorted
 *                 ascending (the order only changes fp32 rounding); an empty list gives zeros
 *   block_table_row: device int32 [n_blocks_row] mapping logical positions to pages
 *   out         : device fp32 [n_queries][n_q_heads][head_dim]
 *   workspace   : device, >= kvq_sparse_workspace_bytes(n_blocks_row, n_kv_heads, head_dim),
 *                 16-byte aligned; its contents on entry do not matter
 * The GQA group (n_q_heads / n_kv_heads) may be 1..16.  A cell outside [0, 16 n_blocks_row)
 * is skipped (KVQ_DEV_BAD_CELL); a cell on a page whose block-table entry is outside
 * [0, num_blocks) is skipped (KVQ_DEV_BAD_BLOCK).
 */
int kvq_attn_sparse_int8kv(const kvq_cache* cache, const void* q, int32_t n_queries,
                           int32_t n_q_heads, const int32_t* cell_offsets,
                           const int32_t* cells, const int32_t* block_table_row,
                           int32_t n_blocks_row, float softmax_scale, float* out,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Workspace (bytes) of kvq_attn_prefill_first_bf16: the fp16 Q rows and their scales, and the
 * chunk's K/V as fp16 operand pieces with their scales (2 * 2 * head_dim bytes per key and KV
 * head).  0 if an argument is not positive or head_dim is not 128 / 256. */
size_t kvq_prefill_first_workspace_bytes(int32_t n_tokens, int32_t n_q_heads, int32_t n_kv_heads,
                                         int32_t head_dim);

/*
 * kvq_attn_prefill_first_bf16 — the first prefill chunk of a sequence ([DCU] §3.1: there is no
 * history to read, so the chunk runs a high-precision attention over its own bf16 Q/K/V while the
 * producer writes its K/V as int8 for the chunks and decode steps that follow; §4.2 measures the
 * int8 path as slower than bf16 for the 0 + 4K chunk).  For tokens t = 0 .. n_tokens - 1:
 *   (1) k_new[t], v_new[t] are quantised by the kvq_quant_write rule into position t of the
 *       sequence (the same codes and scales, bit for bit);
 *   (2) out[t][h] = sum_{s <= t} softmax_s(softmax_scale * q[t][h] . k[s]) * v[s] over the bf16
 *       values themselves (causal, GQA).  The tensor cores see fp16: each row of Q, K and V is
 *       scaled by a power of two into fp16 range (exact for every value within 2^29 of the row's
 *       largest), and the softmax weights of each 128-key tile go in as fp16 w / max w.
 * Later chunks of the sequence use kvq_attn_prefill_int8 (history_len > 0).
 *   q           : device bf16 [n_tokens][n_q_heads][head_dim]
 *   k_new, v_new: device bf16 [n_tokens][n_kv_heads][head_dim]
 *   block_table_row: device int32 [n_blocks_row] of the sequence; n_tokens <= 16 * n_blocks_row
 *   out         : device fp32 [n_tokens][n_q_heads][head_dim]
 *   workspace   : >= kvq_prefill_first_workspace_bytes(...), 16-byte aligned
 *   softmax_scale: finite and > 0
 * A page id outside [0, num_blocks) skips that page's K/V write (KVQ_DEV_BAD_BLOCK); the
 * attention does not read the cache.
 */
int kvq_attn_prefill_first_bf16(const kvq_cache* cache, const void* q, const void* k_new, const void* v_new,
                                int32_t n_tokens, int32_t n_q_heads, const int32_t* block_table_row,
                                int32_t n_blocks_row, float softmax_scale, float* out, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Test entry points of the prefill path (the same device code as kvq_attn_prefill_int8).
 * kvq_debug_prefill_q_codes: the per-(token, query head) Q quantisation step alone.
 *   q: device bf16 [n_tokens][n_q_heads][head_dim]; q_codes: device int8, same shape;
 *   q_scales: device fp32 [n_tokens][n_q_heads].
 * kvq_debug_prefill_qk_int32: kvq_attn_prefill_int8_qcodes (the whole call: the widening pre-pass
 *   and the production attention kernel, writing `out`), compiled with one addition: as its softmax
 *   threads load the integer scores S of the unit (query rows q0 .. q0+127 of query head q_head)
 *   from tensor memory, the ones of keys k0 .. k0+nk-1 are also written, before any masking, to
 *   s_out (device int32 [128][nk]): S[row][key] = sum_d q_code[q0+row][q_head][d] * k_code[key][d]
 *   ([DCU] §1.3, §3.3: Score = MMA_int8(Q, K^T) with an int32 accumulator).  Rows at or past
 *   n_tokens and keys at or past history_len + n_tokens are 0 (their operands are zero).
 *   q0 is a multiple of 128 below n_tokens; k0 and nk are multiples of 128 and the window lies in
 *   the key tiles the unit computes: k0 + nk <= 128 * ((history_len + min(q0 + 127, n_tokens - 1))
 *   / 128 + 1).  split_tiles: -1 for the key-range split the call would choose on this GPU, 0 for
 *   none, r > 0 to force a tail segment of r key tiles (KVQ_ERR_INVALID_ARG when the shape cannot
 *   split: history_len < 128, or r would leave a lead segment empty).  Other arguments and the
 *   workspace as kvq_attn_prefill_int8_qcodes.
 */
int kvq_debug_prefill_q_codes(const void* q, int32_t n_tokens, int32_t n_q_heads,
                              int32_t head_dim, int8_t* q_codes, float* q_scales,
                              void* stream);
int kvq_debug_prefill_qk_int32(const kvq_cache* cache, const int8_t* q_codes, const float* q_scales,
                               int32_t n_tokens, int32_t n_q_heads, int32_t history_len,
                               const int32_t* block_table_row, int32_t n_blocks_row, float softmax_scale,
                               int32_t split_tiles, int32_t q_head, int32_t q0, int32_t k0, int32_t nk,
                               int32_t* s_out, float* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * kvq_debug_stream_floor — measurement entry point: the K/V stream of kvq_attn_decode_int8kv's
 * split route (stage 1) alone.  It launches the same grid (one CTA per (split, KV head, sequence)),
 * the same eight warps with their three-stage shared-memory rings and the same bulk copies of the
 * same pages (K, V and both scale runs of every (page, KV head) below ctx_lens[b]), waits for each
 * copy and computes nothing.  Its duration is the cost of streaming one decode call's K/V by
 * itself on this GPU, launch and ramp-up included: the floor the attention's stage 1 is measured
 * against.  split_rows: 0 for the size kvq_attn_decode_int8kv would choose, else a multiple of 16.
 * Arguments otherwise as kvq_attn_decode_int8kv; writes nothing but the device status word.
 */
int kvq_debug_stream_floor(const kvq_cache* cache, int32_t batch, const int32_t* block_table,
                           int32_t max_blocks_per_seq, const int32_t* ctx_lens, int32_t max_ctx, int32_t split_rows,
                           void* stream);

/*
 * kvq_debug_fault_inject — test entry point of the failure path: every bounded wait of the decode,
 * prefill and sparse kernels launched after this call gives up after wait_budget_cycles SM clock
 * cycles (<= 0: the default, about 2 s), and with mode 1 the first team of decode stage-1 CTA 0
 * does not issue the copy of its second page, with mode 2 the producer of prefill attention CTA 0
 * does not issue its fourth piece, with mode 3 the sparse CTA of (query 0, KV head 0) does not
 * issue the copies of its second chunk (mode 0: no injection).  No copy is left in flight:
 * the consumer's wait runs out, the kernel sets KVQ_DEV_TIMEOUT, waits (bounded) for the copies it
 * did issue, drops that CTA's result (decode single route: zero output rows; split route: an empty
 * partial that the merge skips; prefill: the unit's output rows are not written; sparse: the
 * query's rows are zeros) and returns; the device stays usable.  Process-wide, host only; kvq_debug_fault_inject(0, 0) restores the defaults.
 * KVQ_ERR_INVALID_ARG for an unknown mode.
 */
int kvq_debug_fault_inject(int32_t mode, int64_t wait_budget_cycles);

/* Synchronises `stream`, then returns the device status bits of the current device in
 * *flags_out and clears them.  Returns KVQ_ERR_CUDA if the stream reports an error. */
int kvq_device_status(uint32_t* flags_out, void* stream);

/* Static text for a kvq_status value. */
const char* kvq_status_string(int status);

/* KVQ_ABI_VERSION of the loaded library. */
int kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
