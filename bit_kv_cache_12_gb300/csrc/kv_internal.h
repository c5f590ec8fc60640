// Internal declarations shared by the translation units of libkvint2.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kvint2.h"

namespace kvint2 {

constexpr int kHeadDim = 128;
constexpr int kTile = 16;           // tokens per INT2 history tile
constexpr int kCodeBlock = 512;     // bytes of K (or V) codes per tile
constexpr int kMaxDecodeLen = 6553600;   // longest history (INT2) or sequence (BF16) one decode covers
constexpr int kMaskWords = 16;      // arrival-mask words per (sequence, KV head): 512 history splits

struct Pool {
  kv_pool_config_t cfg;
  int device = 0;
  int sm_count = 0;
  int G = 1;                        // q heads per KV head

  // INT2 history: [layer][page][head][tiles_per_page][tile_bytes]
  uint8_t* hist = nullptr;
  size_t tile_bytes = 0, page_bytes = 0, hist_layer_stride = 0;
  // BF16 tiers: [layer][seq][head][cap][128]
  uint16_t* sink_k = nullptr;
  uint16_t* sink_v = nullptr;
  uint16_t* rec_k = nullptr;
  uint16_t* rec_v = nullptr;
  size_t sink_layer_stride = 0, rec_layer_stride = 0;   // elements
  // BF16 pool: [layer][page][head][page_size][128]
  uint16_t* bk = nullptr;
  uint16_t* bv = nullptr;
  size_t bf16_layer_stride = 0;     // elements

  // per layer rotation data
  float* Rk = nullptr;              // [layer][Hkv][128][128]  x' = x Rk
  float* RvT = nullptr;             // [layer][Hkv][128][128]  RvT[i][c] = Rv[c][i]
  float* clip = nullptr;            // [layer][2][Hkv][128]
  uint4* rfrag = nullptr;           // [layer][Hkv][kFragBlocks][4096] rotation operands (below)
  unsigned* tickets = nullptr;      // [layer][max_seqs][Hkv] split-merge counters (BF16 decode)
  unsigned* arrive = nullptr;       // [layer][max_seqs][Hkv][kMaskWords] arrival masks (INT2 decode)
  unsigned* step_tickets = nullptr; // [layer][ceil(max_seqs / 128)] per-step placement counters
  int* err = nullptr;               // device error word

  // test hooks (kv_debug_stall_first_copy): 0 in normal use
  int test_stall_first_copy = 0;    // decode: the first tile copy of split 0 is never issued;
                                    // bulk append: the first x load of CTA (0, 0) is never started
  int test_wait_polls = 0;          // decode and bulk append: polls of a bounded wait (0 = the default)
};

// Rotation operands per (layer, KV head), 4096 uint4 (64 KB) each:
//   block 0: mma.sync B operand of q . R_k as fp16 hi/lo pairs (decode q' = q R_k)
//   block 1: tcgen05 B operand of x . R_k: rows n of [R_k^T hi ; R_k^T lo] (256 x 128
//            bf16), K-major, 128-byte swizzle, channels 0-63 then 64-127 (append K)
//   block 2: the same for R_v (append V)
//   block 3: mma.sync B operand of o' . R_v^T, laid out as block 0 (decode back-rotation)
constexpr int kFragBlocks = 4;
inline size_t rfrag_per_head() { return 4096; }   // uint4 per (head, block)

// ---- launchers (return cudaSuccess or the launch error) --------------------
cudaError_t launch_rotation_prep(const Pool& p, int layer, const float* Rk, const float* Rv,
                                 cudaStream_t s);
cudaError_t launch_store_tier(const Pool& p, int layer, int tier, int n_rows, const void* k,
                              const void* v, const int32_t* seq, const int32_t* slot,
                              cudaStream_t s);
cudaError_t launch_quantize_pack(const Pool& p, int layer, int tensor, int64_t n_rows,
                                 const float* x, uint8_t* codes, void* sz, cudaStream_t s);
cudaError_t launch_append(const Pool& p, int layer, int n_seqs, const void* k, const void* v,
                          const int32_t* cu, const int32_t* hist_start, const int32_t* pt,
                          int max_pages, int max_tokens, cudaStream_t s);
cudaError_t launch_append_tc(const Pool& p, int layer, int n_seqs, const void* k, const void* v,
                             const int32_t* cu, const int32_t* hist_start, const int32_t* pt,
                             int max_pages, int max_tokens, cudaStream_t s);
cudaError_t launch_append_step(const Pool& p, int layer, int B, const void* k_new,
                               const void* v_new, int32_t* sink_len, int32_t* hist_len,
                               int32_t* rec_len, int32_t* rec_start, const int32_t* pt,
                               int max_pages, cudaStream_t s);
cudaError_t launch_append_bf16(const Pool& p, int layer, int n_seqs, const void* k,
                               const void* v, const int32_t* cu, const int32_t* start,
                               const int32_t* pt, int max_pages, int max_tokens,
                               cudaStream_t s);

// cuTensorMapEncodeTiled (driver entry point, looked up once; NULL if absent)
void* tensor_map_encode_fn();

struct DecodePlan {
  int n_split = 1;          // history splits per (sequence, KV head)
  int n_tier = 0;           // CTAs for the BF16 sink + recent tiers (INT2 pool)
  int tiles_per_split = 1;  // INT2: 16-token tiles; BF16: tokens
  int max_len = 0;          // history (INT2) or sequence (BF16) tokens the grid covers
  size_t partial_floats = 0;
  size_t bytes = 0;
};
// T query positions per sequence (T * G must be 1, 2, 4 or 8)
DecodePlan plan_decode_int2(const Pool& p, int B, int max_hist_len, int T = 1);
DecodePlan plan_decode_bf16(const Pool& p, int B, int max_len);

cudaError_t launch_decode_int2(const Pool& p, int layer, int B, const void* q,
                               const int32_t* sink_len, const int32_t* hist_len,
                               const int32_t* rec_len, const int32_t* rec_start,
                               const int32_t* pt, int max_pages, const DecodePlan& plan,
                               float scale, float* out, void* ws, cudaStream_t s, int T = 1,
                               float* lse = nullptr);
// Device address and size of the fixed scratch buffer used by
// kv_decode_attention_noalloc on the current device (looked up once per device).
cudaError_t noalloc_scratch(void** ptr, size_t* bytes);

cudaError_t launch_decode_bf16(const Pool& p, int layer, int B, const void* q,
                               const int32_t* seq_len, const int32_t* pt, int max_pages,
                               const DecodePlan& plan, float scale, float* out, void* ws,
                               cudaStream_t s);

}  // namespace kvint2
