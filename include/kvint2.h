/*
 * kvint2.h -- C ABI of the GB300 2-bit KV-cache hot path (OSCAR-style).
 *
 * The method (gist.science explainer "OSCAR: Offline Spectral Covariance-
 * Aware Rotation for 2-bit KV Cache Quantization", section 2.2 B "Online-
 * Betriebsphase"; yunpan.plus OSCAR write-up, sections "1. 三段式 Token 池"
 * and "2. 在线量化与反量化"):
 *   - each sequence's KV cache has three tiers per KV head: the first 64
 *     tokens (sink) and the last 256 tokens (recent) in BF16, everything in
 *     between (history) in INT2;
 *   - a token leaving the recent window is rotated by a fixed per-head
 *     orthogonal matrix R (x' = x R), clipped per rotated channel, quantized
 *     to asymmetric INT2 with an fp16 scale and zero per token and channel
 *     group, and packed four codes per byte into paged history blocks;
 *   - decode attention dequantizes the history on the fly, attends over all
 *     three tiers with one softmax, and rotates the history value
 *     accumulator back by R^T.
 *
 * Conventions for every entry point
 *   - Pointers named "device" are CUDA device pointers on the pool's device;
 *     host pointers are named "host".  The caller owns every buffer it
 *     passes; the pool owns its own storage.
 *   - The decode calls (kv_decode_attention, _noalloc, _multi) also take q,
 *     the four length arrays, out and lse in mapped page-locked host memory
 *     whose address is valid on the device under unified addressing
 *     (cudaHostAlloc memory; for cudaHostRegister memory pass the pointer
 *     cudaHostGetDevicePointer returns).  The kernel then reads and writes
 *     them across the CPU-GPU link inside the launch, with no staging
 *     copies; results are bit-identical to device buffers.  The host must
 *     not touch them until the stream has passed the call.  The page table,
 *     workspace and every other buffer stay in device memory.
 *   - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream) unless stated otherwise, and validates its arguments on
 *     the host first: on failure it launches nothing and returns
 *     KV_ERR_INVALID_ARG or KV_ERR_UNSUPPORTED.  A failed launch returns
 *     KV_ERR_CUDA.
 *   - The decode calls launch with programmatic dependent launch: their CTAs
 *     may start (and fetch the pool's rotation) while the kernel ahead of them
 *     on `stream` finishes, and read no buffer the caller passes before that
 *     kernel has completed.
 *   - Problems only the GPU can see (a page id outside [0, num_pages), a
 *     length above capacity) are recorded in the pool's device error word and
 *     the offending work is skipped; no kernel traps.  Read it with
 *     kv_pool_get_error().
 *   - Supported: head_dim 128, page_size 16 or 32, group_size 64 or 128,
 *     num_q_heads / num_kv_heads in {1, 2, 4, 8}.
 *   - Calls that touch the same pool layer must be ordered on one stream.
 */
#ifndef KVINT2_H
#define KVINT2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KV_OK = 0,
  KV_ERR_INVALID_ARG = 1,  /* bad pointer, size, index or pool kind          */
  KV_ERR_OOM = 2,          /* device allocation failed                       */
  KV_ERR_CUDA = 3,         /* a CUDA call or launch failed                   */
  KV_ERR_UNSUPPORTED = 4,  /* valid but not implemented (e.g. head_dim 64)   */
  KV_ERR_DEVICE = 5,       /* kv_pool_get_error: the device recorded an error */
  KV_ERR_TIMEOUT = 6,      /* reserved: a bounded device wait gave up        */
  KV_ERR_SCRATCH_LIMIT = 7 /* kv_decode_attention_noalloc: the call needs more
                              scratch than KV_NOALLOC_SCRATCH_BYTES           */
} kv_status_t;

/* Device error codes reported by kv_pool_get_error(). */
enum {
  KV_DEVERR_NONE = 0,
  KV_DEVERR_PAGE_ID = 1,      /* page table entry outside [0, num_pages)     */
  KV_DEVERR_LENGTH = 2,       /* a length above the tier / table capacity    */
  KV_DEVERR_SEQ_RANGE = 3,    /* cu_tokens not monotone or history overflow  */
  KV_DEVERR_TIMEOUT = 4       /* a bounded wait for an asynchronous copy ran
                                 out; the work that needed it was skipped.
                                 The outputs of that call are wrong: discard
                                 them.  A copy that did not arrive within about
                                 a second points to a device problem, and the
                                 library cannot rule out that it lands later;
                                 do not keep using the pool (or the context)
                                 after this code except to tear it down. */
};

typedef enum { KV_POOL_INT2_3TIER = 0, KV_POOL_BF16 = 1 } kv_pool_kind_t;

typedef struct {
  int32_t kind;           /* kv_pool_kind_t                                  */
  int32_t num_layers;
  int32_t num_q_heads;    /* Hq; GQA group G = Hq / Hkv, q head h -> KV head h / G */
  int32_t num_kv_heads;   /* Hkv                                             */
  int32_t head_dim;       /* must be 128                                     */
  int32_t page_size;      /* tokens per page: 16 or 32                       */
  int32_t group_size;     /* INT2 channel group: 64 or 128 (INT2 pool only)  */
  int32_t sink_tokens;    /* 64 for the pages' layout (INT2 pool only)       */
  int32_t recent_tokens;  /* 256 for the pages' layout (INT2 pool only)      */
  int32_t max_seqs;       /* sequence slots of the sink / recent tiers       */
  int64_t num_pages;      /* physical pages per layer                        */
} kv_pool_config_t;

/* Where the pool keeps its data (device pointers and byte strides), so a
 * caller can copy tiers in or out.  For layer `l`:
 *   INT2 history block of (page p, KV head g):
 *       hist + l*hist_layer_stride + p*hist_page_stride + g*hist_head_stride
 *     = page_size/16 tiles of tile_bytes each; a tile is
 *       [K codes 512 B][V codes 512 B][K records 16 * rec_bytes B][V records 16 * rec_bytes B]
 *     rec_bytes = 4 * 128/group_size: per group the (s, z) fp16 pair of the
 *     tensor; record slot 2*(t%8) + t/8 of each block holds token t of the tile
 *     (K and V records in separate 32-byte sectors, so each tensor's writes
 *     cover whole sectors).
 *     Code bit of (m, k, step) with m, k in [0,16), step in [0,8): 16-byte
 *     lane L = 4*(m%8) + (k%8)/2, 32-bit little-endian word step/2, bit
 *     16*(k%2) + 2*(2*(step%2) + m/8 + 4*(k/8)); K: m = token, k = channel%16,
 *     step = channel/16; V: m = channel%16, k = token, step = channel/16.
 *   sink_k / sink_v:   bf16 [max_seqs][Hkv][sink_tokens][128]
 *   recent_k/recent_v: bf16 [max_seqs][Hkv][recent_tokens][128] (ring)
 *   BF16 pool: bf16_k / bf16_v bf16 [num_pages][Hkv][page_size][128]
 * Pointers that do not apply to the pool kind are NULL. */
typedef struct {
  void* hist;
  size_t hist_layer_stride, hist_page_stride, hist_head_stride, tile_bytes;
  void* sink_k;
  void* sink_v;
  void* recent_k;
  void* recent_v;
  size_t tier_layer_stride;      /* bytes between layers of sink_* (and of recent_* below) */
  size_t recent_layer_stride;
  void* bf16_k;
  void* bf16_v;
  size_t bf16_layer_stride;      /* bytes between layers of bf16_k / bf16_v */
} kv_pool_layout_t;

typedef struct kv_pool kv_pool_t;   /* opaque; owns all pool device memory */

/* Create a pool on the current CUDA device.  Allocates and zeroes its
 * storage (synchronously: the call returns when the pool is ready).
 * Rotations default to identity and clips to +inf until set.
 * Returns KV_ERR_OOM if the device allocation fails. */
kv_status_t kv_pool_create(const kv_pool_config_t* cfg, void* stream, kv_pool_t** out);

/* Free the pool's device memory (synchronises the device first). */
kv_status_t kv_pool_destroy(kv_pool_t* pool);

/* Set the fixed rotation and clip thresholds of one layer (gist.science
 * explainer section 2.2 A: R_K = U_Q H P_br, R_V = U_S H P_br, per-layer clip
 * thresholds from rotated calibration data).
 *   R_k, R_v   device fp32 [Hkv][128][128] row-major; x' = x . R (row vector).
 *              Must be orthogonal (R R^T = I); the decode uses R^T as inverse.
 *   clip_k/v   device fp32 [Hkv][128] thresholds c_j > 0 on rotated channels,
 *              y = min(max(x', -c), c); +inf disables clipping.
 * The values are copied into the pool on `stream`, and the call returns once
 * the copy is complete (it synchronises `stream`): decode launches read the
 * rotation while the kernel ahead of them may still run (programmatic
 * dependent launch), so it must be in place before they are issued. */
kv_status_t kv_pool_set_rotation(kv_pool_t* pool, int32_t layer, const float* R_k,
                                 const float* R_v, const float* clip_k, const float* clip_v,
                                 void* stream);

/* Fill `out` with the pool's device pointers and strides for `layer`. */
kv_status_t kv_pool_get_layout(const kv_pool_t* pool, int32_t layer, kv_pool_layout_t* out);

/* Read and clear the device error word (synchronous).  *device_error_code
 * receives a KV_DEVERR_* value; the return is KV_ERR_DEVICE if it was
 * nonzero, KV_OK otherwise. */
kv_status_t kv_pool_get_error(kv_pool_t* pool, int32_t* device_error_code);

/* Write BF16 tokens into the sink (tier 0) or recent ring (tier 1) of an
 * INT2 pool: row i goes to sequence slot seq[i], position slot[i] of that
 * tier, all KV heads.  k, v: device bf16 [n_rows][Hkv][128]; seq, slot:
 * device int32 [n_rows].  Out-of-range seq/slot entries are skipped and
 * flagged (KV_DEVERR_LENGTH). */
kv_status_t kv_store_tier(kv_pool_t* pool, int32_t layer, int32_t tier, int32_t n_rows,
                          const void* k, const void* v, const int32_t* seq,
                          const int32_t* slot, void* stream);

/* Parity entry of the quantizer: clip -> INT2 quantize -> pack for rows that
 * are already rotated (yunpan.plus write-up section 2: "裁剪 -> 量化 -> 打包";
 * four 2-bit codes per byte).
 *   tensor     0 = K (uses clip_k), 1 = V (uses clip_v) of `layer`
 *   x_rot      device fp32 [n_rows][Hkv][128]
 *   codes      device uint8 [n_rows][Hkv][32]: byte b holds channels 4b..4b+3,
 *              channel 4b+j in bits [2j, 2j+2)
 *   scale_zero device fp16 pairs [n_rows][Hkv][128/group_size][2] = (s, z)
 * Quantizer (per row, head, group of group_size contiguous channels, fp32):
 *   s = fp16((max - min) / 3), z = fp16(min), both saturated to +-65504;
 *   code = s == 0 ? 0 : clamp(rint((y - z) / s), 0, 3), ties to even. */
kv_status_t kv_quantize_pack_f32(kv_pool_t* pool, int32_t layer, int32_t tensor,
                                 int64_t n_rows, const float* x_rot, uint8_t* codes,
                                 void* scale_zero, void* stream);

/* Fused append (the eviction step of the yunpan.plus write-up section 2):
 * rotate by R_k / R_v, clip, quantize and pack K and V tokens into the INT2
 * history pages of `layer`.
 *   k, v        device bf16 [T][Hkv][128], T = cu_tokens[n_seqs], 16-byte
 *               aligned (else KV_ERR_INVALID_ARG)
 *   cu_tokens   device int32 [n_seqs+1], prefix sums of tokens per sequence
 *   hist_start  device int32 [n_seqs]: history position of each sequence's
 *               first appended token (its tokens go to consecutive positions)
 *   page_table  device int32 [n_seqs][max_pages_per_seq]: history position p
 *               of sequence i lives in page page_table[i][p / page_size]
 *   max_tokens_per_seq  host bound on tokens of any one sequence (sizes the
 *               grid; sequences above it are flagged and truncated)
 * Tiles partly covered keep the other tokens' bits (appends may continue a
 * partly filled page).  Rotation runs on the tcgen05 tensor cores with R split
 * into two bf16 terms (about 16 significant bits), fp32 accumulation; the
 * codes equal those of kv_append_step for the same token. */
kv_status_t kv_append_quantize(kv_pool_t* pool, int32_t layer, int32_t n_seqs,
                               const void* k, const void* v, const int32_t* cu_tokens,
                               const int32_t* hist_start, const int32_t* page_table,
                               int32_t max_pages_per_seq, int32_t max_tokens_per_seq,
                               void* stream);

/* Several query positions per sequence over the same cache: a chunk of
 * prefill continuing on an INT2 prefix, prefix-cache reuse, or draft tokens
 * being verified (zingnex.cn forum summary of OSCAR, "与其他优化的协同";
 * yunpan.plus write-up, "3. 兼容现有架构").  Each of the T queries of
 * sequence b attends, like kv_decode_attention, over the whole cache of that
 * sequence (sink, INT2 history, recent); there is no masking among the T
 * queries.  The caller attends the chunk's own tokens itself and merges the
 * two by the log-sum-exp rule using `lse`.
 *   T        query positions per sequence; T * (num_q_heads / num_kv_heads)
 *            must be 1, 2, 4 or 8 (else KV_ERR_UNSUPPORTED)
 *   q        device bf16 [B][T][Hq][128]
 *   out      device fp32 [B][T][Hq][128]
 *   lse      device fp32 [B][T][Hq] or NULL: ln sum_t exp(softmax_scale * s_t)
 *            over the cached tokens t (s_t the dot product the attention
 *            uses); -inf when the sequence caches no token
 *   other arguments as for kv_decode_attention; the workspace size comes
 *   from kv_decode_multi_workspace_bytes. */
size_t kv_decode_multi_workspace_bytes(const kv_pool_t* pool, int32_t B, int32_t T,
                                       int32_t max_hist_len);
kv_status_t kv_decode_attention_multi(kv_pool_t* pool, int32_t layer, int32_t B, int32_t T,
                                      const void* q, const int32_t* sink_len,
                                      const int32_t* hist_len, const int32_t* recent_len,
                                      const int32_t* recent_start, const int32_t* page_table,
                                      int32_t max_pages_per_seq, int32_t max_hist_len,
                                      float softmax_scale, float* out, float* lse,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* One decode step's token placement for B sequences (yunpan.plus write-up,
 * "1. 三段式 Token 池" and "2. 在线量化与反量化"): the new token of sequence b
 * (all KV heads) goes to the sink while it holds fewer than sink_tokens
 * tokens (the sequence's first tokens), else to the recent ring while that
 * holds fewer than recent_tokens; when the ring is full its oldest token (at
 * recent_start) is rotated, clipped, quantized and packed into history
 * position hist_len[b] (the same arithmetic, and so the same codes, as
 * kv_append_quantize), the new token takes its ring slot and recent_start
 * advances.  The four length arrays are updated on the device, in stream
 * order, so consecutive steps and decodes need no host round trip.  One
 * launch; calls for the same layer must not overlap on the GPU (they share the
 * layer's completion counters).
 *   k_new, v_new  device bf16 [B][Hkv][128] (8-byte aligned); sequence b
 *                 uses pool slot b
 *   sink_len, hist_len, recent_len, recent_start
 *                 device int32 [B], read and updated in place
 *   page_table    device int32 [B][max_pages_per_seq]: the page of history
 *                 position p is page_table[b][p / page_size]; the caller
 *                 provides it before the step that needs it
 * Errors: KV_ERR_INVALID_ARG for bad arguments (nothing launched).  On the
 * device, lengths out of range set KV_DEVERR_LENGTH and a missing or
 * out-of-range page id for the eviction sets KV_DEVERR_PAGE_ID; that
 * sequence's step is then not applied (no tier or length changes). */
kv_status_t kv_append_step(kv_pool_t* pool, int32_t layer, int32_t B, const void* k_new,
                           const void* v_new, int32_t* sink_len, int32_t* hist_len,
                           int32_t* recent_len, int32_t* recent_start,
                           const int32_t* page_table, int32_t max_pages_per_seq, void* stream);

/* Bytes of device workspace kv_decode_attention / kv_decode_attention_bf16
 * need for a batch of B sequences whose history (INT2 pool) or total length
 * (BF16 pool) is at most max_len tokens.  0 on invalid arguments.  Every
 * decode call takes max_hist_len / max_seq_len <= KV_MAX_DECODE_LEN
 * (else KV_ERR_INVALID_ARG). */
#define KV_MAX_DECODE_LEN 6553600
size_t kv_decode_workspace_bytes(const kv_pool_t* pool, int32_t B, int32_t max_len);

/* One decode step of one layer for B sequences over the three-tier pool
 * (gist.science explainer section 2.2 B): rotate q by R_k, attend over sink,
 * history (INT2, dequantized on the fly in registers) and recent tiers with
 * one split-K online softmax, rotate the history value accumulator back by
 * R_v^T, and merge everything into fp32 outputs.
 *   q            device bf16 [B][Hq][128]; sequence b uses pool slot b
 *   sink_len     device int32 [B] (<= sink_tokens)
 *   hist_len     device int32 [B] (<= max_hist_len and the page table's span;
 *                a longer history sets KV_DEVERR_LENGTH and only its first
 *                min(max_hist_len, span) tokens are attended)
 *   recent_len   device int32 [B] (<= recent_tokens)
 *   recent_start device int32 [B]: ring index of the oldest recent token
 *   page_table   device int32 [B][max_pages_per_seq] (history pages)
 *   max_hist_len host bound on hist_len (sizes the grid)
 *   softmax_scale  tau in exp(tau q.k) (1/sqrt(128) for standard attention)
 *   out          device fp32 [B][Hq][128]
 *   workspace    device, >= kv_decode_workspace_bytes(pool, B, max_hist_len) */
kv_status_t kv_decode_attention(kv_pool_t* pool, int32_t layer, int32_t B, const void* q,
                                const int32_t* sink_len, const int32_t* hist_len,
                                const int32_t* recent_len, const int32_t* recent_start,
                                const int32_t* page_table, int32_t max_pages_per_seq,
                                int32_t max_hist_len, float softmax_scale, float* out,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Append BF16 tokens to an all-BF16 paged pool (the baseline the INT2 path is
 * compared with).  k, v device bf16 [T][Hkv][128]; token i of sequence s goes
 * to position start_pos[s] + i, page page_table[s][pos / page_size]. */
kv_status_t kv_append_bf16(kv_pool_t* pool, int32_t layer, int32_t n_seqs, const void* k,
                           const void* v, const int32_t* cu_tokens, const int32_t* start_pos,
                           const int32_t* page_table, int32_t max_pages_per_seq,
                           int32_t max_tokens_per_seq, void* stream);

/* Decode attention over an all-BF16 paged pool: plain split-K softmax
 * attention of q [B][Hq][128] over seq_len[b] tokens, fp32 out [B][Hq][128].
 * seq_len[b] above max_seq_len (or the page table's span) sets
 * KV_DEVERR_LENGTH and only the covered tokens are attended. */
kv_status_t kv_decode_attention_bf16(kv_pool_t* pool, int32_t layer, int32_t B, const void* q,
                                     const int32_t* seq_len, const int32_t* page_table,
                                     int32_t max_pages_per_seq, int32_t max_seq_len,
                                     float softmax_scale, float* out, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* Size of the fixed device buffer behind kv_decode_attention_noalloc. */
#define KV_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* kv_decode_attention without a caller workspace.  (The pages describe no
 * such call: it exists for users of this library, not for the method.)
 *
 * Some callers cannot allocate device memory at the point where they decode:
 * code running under a memory manager that owns every allocation (a serving
 * engine's arena, a pluggable allocator), or code that must not call
 * cudaMalloc because it may synchronise the device in a latency-critical
 * path.  This entry point takes the same arguments as kv_decode_attention
 * minus the workspace, and keeps the per-split partial results in one
 * file-scope device buffer of KV_NOALLOC_SCRATCH_BYTES (16 MiB) instead.  The
 * buffer is reserved on every GPU that loads the library and is held until
 * the process exits.  The call itself allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine).
 *
 *   - The first call on a device looks up the buffer's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Calls whose workspace need, kv_decode_workspace_bytes(pool, B,
 *     max_hist_len), exceeds KV_NOALLOC_SCRATCH_BYTES return
 *     KV_ERR_SCRATCH_LIMIT and launch nothing.
 *   - Every call on a device shares the one buffer and leaves its own
 *     contents in it; nothing in it has to start at zero (each call writes
 *     every partial it later reads).  Calls that overlap on the GPU (other
 *     streams, other threads, other pools) race on the buffer: order them.
 *   - The current device must be the pool's (the buffer looked up is the
 *     current device's); otherwise KV_ERR_INVALID_ARG, nothing launched.
 * Results equal kv_decode_attention's for the same inputs, bit for bit (same
 * kernel, same split plan, same merge order). */
kv_status_t kv_decode_attention_noalloc(kv_pool_t* pool, int32_t layer, int32_t B, const void* q,
                                        const int32_t* sink_len, const int32_t* hist_len,
                                        const int32_t* recent_len, const int32_t* recent_start,
                                        const int32_t* page_table, int32_t max_pages_per_seq,
                                        int32_t max_hist_len, float softmax_scale, float* out,
                                        void* stream);

/* Test hook for the bounded waits (no counterpart on the pages).  With
 * enable != 0, later decode calls of this pool arm the first ring stage of
 * the first history split for a tile copy that is never issued, so that the
 * warp's bounded wait runs out: the call sets KV_DEVERR_TIMEOUT, waits
 * (bounded) for the copies it did issue, skips that split and returns; and
 * later kv_append_quantize calls never start the x load of the first chunk
 * of the first CTA, so that the wait for it runs out: the call sets
 * KV_DEVERR_TIMEOUT, every warp of that CTA leaves its loop, the CTA waits
 * (bounded) for the loads and products it did start and returns (the
 * history it was to write is left incomplete).  No copy is left in flight,
 * nothing faults and nothing hangs.  max_polls > 0 replaces the default poll
 * limit of those waits (about a second) for the pool's decode and bulk
 * append calls; 0 restores it.  enable = 0 restores normal calls.  Not for
 * production use. */
kv_status_t kv_debug_stall_first_copy(kv_pool_t* pool, int32_t enable, int32_t max_polls);

#ifdef __cplusplus
}
#endif

#endif /* KVINT2_H */
