// C ABI of libkvint2: argument checks, pool storage, launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <new>

#include "kv_internal.h"

using kvint2::Pool;

struct kv_pool {
  Pool p;
};

namespace {

bool is_pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

kv_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? KV_OK : KV_ERR_CUDA; }

template <class T>
bool dev_alloc(T** ptr, size_t bytes) {
  if (bytes == 0) {
    *ptr = nullptr;
    return true;
  }
  void* v = nullptr;
  if (cudaMalloc(&v, bytes) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  *ptr = static_cast<T*>(v);
  return true;
}

void free_pool(Pool& p) {
  void* ptrs[] = {p.hist, p.sink_k, p.sink_v, p.rec_k,   p.rec_v,        p.bk,  p.bv,  p.Rk,
                  p.RvT,  p.clip,   p.rfrag,  p.tickets, p.step_tickets, p.arrive, p.err};
  for (void* q : ptrs)
    if (q) cudaFree(q);
}

__global__ void init_rotation_kernel(float* Rk, float* RvT, float* clip, size_t n_mat, size_t n_clip) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx < n_mat) {
    const int i = (int)((idx >> 7) & 127), c = (int)(idx & 127);
    const float v = (i == c) ? 1.f : 0.f;
    Rk[idx] = v;
    RvT[idx] = v;
  }
  if (idx < n_clip) clip[idx] = INFINITY;
}

bool valid_layer(const kv_pool_t* pool, int layer) {
  return pool && layer >= 0 && layer < pool->p.cfg.num_layers;
}

}  // namespace

extern "C" {

kv_status_t kv_pool_create(const kv_pool_config_t* cfg, void* stream, kv_pool_t** out) {
  if (!cfg || !out) return KV_ERR_INVALID_ARG;
  *out = nullptr;
  const kv_pool_config_t c = *cfg;
  if (c.kind != KV_POOL_INT2_3TIER && c.kind != KV_POOL_BF16) return KV_ERR_INVALID_ARG;
  if (c.num_layers <= 0 || c.num_kv_heads <= 0 || c.num_q_heads <= 0 || c.max_seqs <= 0 ||
      c.num_pages <= 0 || c.num_pages > (int64_t)INT32_MAX)
    return KV_ERR_INVALID_ARG;
  if (c.num_q_heads % c.num_kv_heads != 0) return KV_ERR_INVALID_ARG;
  if (c.head_dim != 128) return KV_ERR_UNSUPPORTED;
  if (c.page_size != 16 && c.page_size != 32) return KV_ERR_UNSUPPORTED;
  const int G = c.num_q_heads / c.num_kv_heads;
  if (!is_pow2_in(G, 1, 8)) return KV_ERR_UNSUPPORTED;
  if (c.kind == KV_POOL_INT2_3TIER) {
    if (c.group_size != 64 && c.group_size != 128) return KV_ERR_UNSUPPORTED;
    if (c.sink_tokens < 0 || c.recent_tokens <= 0 || c.sink_tokens > 4096 || c.recent_tokens > 4096)
      return KV_ERR_INVALID_ARG;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KV_ERR_CUDA;
  kv_pool_t* pool = new (std::nothrow) kv_pool_t();
  if (!pool) return KV_ERR_OOM;
  Pool& p = pool->p;
  p.cfg = c;
  p.device = dev;
  p.G = G;
  cudaDeviceGetAttribute(&p.sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (p.sm_count <= 0) p.sm_count = 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t L = c.num_layers, H = c.num_kv_heads;
  bool ok = true;
  if (c.kind == KV_POOL_INT2_3TIER) {
    p.tile_bytes = 1024 + kvint2::kTile * 8 * (128 / c.group_size);
    p.page_bytes = H * (c.page_size / kvint2::kTile) * p.tile_bytes;
    p.hist_layer_stride = (size_t)c.num_pages * p.page_bytes;
    p.sink_layer_stride = (size_t)c.max_seqs * H * c.sink_tokens * 128;
    p.rec_layer_stride = (size_t)c.max_seqs * H * c.recent_tokens * 128;
    ok = ok && dev_alloc(&p.hist, L * p.hist_layer_stride);
    ok = ok && dev_alloc(&p.sink_k, L * p.sink_layer_stride * 2);
    ok = ok && dev_alloc(&p.sink_v, L * p.sink_layer_stride * 2);
    ok = ok && dev_alloc(&p.rec_k, L * p.rec_layer_stride * 2);
    ok = ok && dev_alloc(&p.rec_v, L * p.rec_layer_stride * 2);
    ok = ok && dev_alloc(&p.Rk, L * H * 128 * 128 * sizeof(float));
    ok = ok && dev_alloc(&p.RvT, L * H * 128 * 128 * sizeof(float));
    ok = ok && dev_alloc(&p.clip, L * 2 * H * 128 * sizeof(float));
    ok = ok && dev_alloc(&p.rfrag, L * H * kvint2::kFragBlocks * kvint2::rfrag_per_head() * sizeof(uint4));
  } else {
    p.bf16_layer_stride = (size_t)c.num_pages * H * c.page_size * 128;
    ok = ok && dev_alloc(&p.bk, L * p.bf16_layer_stride * 2);
    ok = ok && dev_alloc(&p.bv, L * p.bf16_layer_stride * 2);
  }
  ok = ok && dev_alloc(&p.tickets, L * c.max_seqs * H * sizeof(unsigned));
  ok = ok && dev_alloc(&p.arrive, L * c.max_seqs * H * kvint2::kMaskWords * sizeof(unsigned));
  ok = ok && dev_alloc(&p.step_tickets, L * ((c.max_seqs + 127) / 128) * sizeof(unsigned));
  ok = ok && dev_alloc(&p.err, sizeof(int));
  if (!ok) {
    free_pool(p);
    delete pool;
    return KV_ERR_OOM;
  }
  cudaError_t e = cudaSuccess;
  auto zero = [&](void* ptr, size_t bytes) {
    if (ptr && bytes && e == cudaSuccess) e = cudaMemsetAsync(ptr, 0, bytes, s);
  };
  zero(p.hist, L * p.hist_layer_stride);
  zero(p.sink_k, L * p.sink_layer_stride * 2);
  zero(p.sink_v, L * p.sink_layer_stride * 2);
  zero(p.rec_k, L * p.rec_layer_stride * 2);
  zero(p.rec_v, L * p.rec_layer_stride * 2);
  zero(p.bk, L * p.bf16_layer_stride * 2);
  zero(p.bv, L * p.bf16_layer_stride * 2);
  zero(p.tickets, L * c.max_seqs * H * sizeof(unsigned));
  zero(p.arrive, L * c.max_seqs * H * kvint2::kMaskWords * sizeof(unsigned));
  zero(p.step_tickets, L * ((c.max_seqs + 127) / 128) * sizeof(unsigned));
  zero(p.err, sizeof(int));
  if (e == cudaSuccess && c.kind == KV_POOL_INT2_3TIER) {
    const size_t n_mat = L * H * 128 * 128, n_clip = L * 2 * H * 128;
    init_rotation_kernel<<<(unsigned)((n_mat + 255) / 256), 256, 0, s>>>(p.Rk, p.RvT, p.clip, n_mat, n_clip);
    e = cudaGetLastError();
    for (int l = 0; l < c.num_layers && e == cudaSuccess; ++l) {
      const size_t off = (size_t)l * H * 128 * 128;
      e = kvint2::launch_rotation_prep(p, l, p.Rk + off, p.RvT + off, s);
    }
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    free_pool(p);
    delete pool;
    return KV_ERR_CUDA;
  }
  *out = pool;
  return KV_OK;
}

kv_status_t kv_pool_destroy(kv_pool_t* pool) {
  if (!pool) return KV_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  free_pool(pool->p);
  delete pool;
  return cuda_status(e);
}

kv_status_t kv_pool_set_rotation(kv_pool_t* pool, int32_t layer, const float* R_k,
                                 const float* R_v, const float* clip_k, const float* clip_v,
                                 void* stream) {
  if (!valid_layer(pool, layer) || !R_k || !R_v || !clip_k || !clip_v) return KV_ERR_INVALID_ARG;
  Pool& p = pool->p;
  if (p.cfg.kind != KV_POOL_INT2_3TIER) return KV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t H = p.cfg.num_kv_heads;
  float* cl = p.clip + (size_t)layer * 2 * H * 128;
  cudaError_t e = cudaMemcpyAsync(cl, clip_k, H * 128 * sizeof(float), cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(cl + H * 128, clip_v, H * 128 * sizeof(float), cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = kvint2::launch_rotation_prep(p, layer, R_k, R_v, s);
  // decodes read the rotation before they wait for the kernel ahead of them:
  // the set-up is complete before this call returns
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

kv_status_t kv_pool_get_layout(const kv_pool_t* pool, int32_t layer, kv_pool_layout_t* out) {
  if (!valid_layer(pool, layer) || !out) return KV_ERR_INVALID_ARG;
  const Pool& p = pool->p;
  *out = kv_pool_layout_t{};
  if (p.cfg.kind == KV_POOL_INT2_3TIER) {
    out->hist = p.hist + (size_t)layer * p.hist_layer_stride;
    out->hist_layer_stride = p.hist_layer_stride;
    out->hist_page_stride = p.page_bytes;
    out->hist_head_stride = p.page_bytes / p.cfg.num_kv_heads;
    out->tile_bytes = p.tile_bytes;
    out->sink_k = p.sink_k + (size_t)layer * p.sink_layer_stride;
    out->sink_v = p.sink_v + (size_t)layer * p.sink_layer_stride;
    out->recent_k = p.rec_k + (size_t)layer * p.rec_layer_stride;
    out->recent_v = p.rec_v + (size_t)layer * p.rec_layer_stride;
    out->tier_layer_stride = p.sink_layer_stride * 2;
    out->recent_layer_stride = p.rec_layer_stride * 2;
  } else {
    out->bf16_k = p.bk + (size_t)layer * p.bf16_layer_stride;
    out->bf16_v = p.bv + (size_t)layer * p.bf16_layer_stride;
    out->bf16_layer_stride = p.bf16_layer_stride * 2;
  }
  return KV_OK;
}

kv_status_t kv_pool_get_error(kv_pool_t* pool, int32_t* device_error_code) {
  if (!pool || !device_error_code) return KV_ERR_INVALID_ARG;
  int v = 0;
  cudaError_t e = cudaMemcpy(&v, pool->p.err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(pool->p.err, 0, sizeof(int));
  if (e != cudaSuccess) return KV_ERR_CUDA;
  *device_error_code = v;
  return v ? KV_ERR_DEVICE : KV_OK;
}

kv_status_t kv_store_tier(kv_pool_t* pool, int32_t layer, int32_t tier, int32_t n_rows,
                          const void* k, const void* v, const int32_t* seq, const int32_t* slot,
                          void* stream) {
  if (!valid_layer(pool, layer) || (tier != 0 && tier != 1) || n_rows < 0) return KV_ERR_INVALID_ARG;
  if (pool->p.cfg.kind != KV_POOL_INT2_3TIER) return KV_ERR_INVALID_ARG;
  if (n_rows > 0 && (!k || !v || !seq || !slot)) return KV_ERR_INVALID_ARG;
  return cuda_status(kvint2::launch_store_tier(pool->p, layer, tier, n_rows, k, v, seq, slot,
                                               static_cast<cudaStream_t>(stream)));
}

kv_status_t kv_quantize_pack_f32(kv_pool_t* pool, int32_t layer, int32_t tensor, int64_t n_rows,
                                 const float* x_rot, uint8_t* codes, void* scale_zero,
                                 void* stream) {
  if (!valid_layer(pool, layer) || (tensor != 0 && tensor != 1) || n_rows < 0)
    return KV_ERR_INVALID_ARG;
  if (pool->p.cfg.kind != KV_POOL_INT2_3TIER) return KV_ERR_INVALID_ARG;
  if (n_rows > 0 && (!x_rot || !codes || !scale_zero)) return KV_ERR_INVALID_ARG;
  if (((uintptr_t)x_rot & 15) || ((uintptr_t)scale_zero & 3)) return KV_ERR_INVALID_ARG;
  return cuda_status(kvint2::launch_quantize_pack(pool->p, layer, tensor, n_rows, x_rot, codes,
                                                  scale_zero, static_cast<cudaStream_t>(stream)));
}

kv_status_t kv_append_quantize(kv_pool_t* pool, int32_t layer, int32_t n_seqs, const void* k,
                               const void* v, const int32_t* cu_tokens, const int32_t* hist_start,
                               const int32_t* page_table, int32_t max_pages_per_seq,
                               int32_t max_tokens_per_seq, void* stream) {
  if (!valid_layer(pool, layer) || n_seqs < 0 || max_pages_per_seq <= 0 || max_tokens_per_seq < 0)
    return KV_ERR_INVALID_ARG;
  if (pool->p.cfg.kind != KV_POOL_INT2_3TIER) return KV_ERR_INVALID_ARG;
  if (n_seqs > 0 && (!k || !v || !cu_tokens || !hist_start || !page_table)) return KV_ERR_INVALID_ARG;
  if (((uintptr_t)k & 15) || ((uintptr_t)v & 15)) return KV_ERR_INVALID_ARG;
  return cuda_status(kvint2::launch_append(pool->p, layer, n_seqs, k, v, cu_tokens, hist_start,
                                           page_table, max_pages_per_seq, max_tokens_per_seq,
                                           static_cast<cudaStream_t>(stream)));
}

kv_status_t kv_append_step(kv_pool_t* pool, int32_t layer, int32_t B, const void* k_new,
                           const void* v_new, int32_t* sink_len, int32_t* hist_len,
                           int32_t* recent_len, int32_t* recent_start, const int32_t* page_table,
                           int32_t max_pages_per_seq, void* stream) {
  if (!valid_layer(pool, layer) || B < 0 || max_pages_per_seq <= 0) return KV_ERR_INVALID_ARG;
  const Pool& p = pool->p;
  if (p.cfg.kind != KV_POOL_INT2_3TIER || B > p.cfg.max_seqs) return KV_ERR_INVALID_ARG;
  if (B > 0 && (!k_new || !v_new || !sink_len || !hist_len || !recent_len || !recent_start ||
                !page_table))
    return KV_ERR_INVALID_ARG;
  if (((uintptr_t)k_new & 7) || ((uintptr_t)v_new & 7)) return KV_ERR_INVALID_ARG;
  return cuda_status(kvint2::launch_append_step(p, layer, B, k_new, v_new, sink_len, hist_len,
                                                recent_len, recent_start, page_table,
                                                max_pages_per_seq,
                                                static_cast<cudaStream_t>(stream)));
}

size_t kv_decode_workspace_bytes(const kv_pool_t* pool, int32_t B, int32_t max_len) {
  if (!pool || B <= 0 || max_len < 0 || max_len > kvint2::kMaxDecodeLen || B > pool->p.cfg.max_seqs) return 0;
  const Pool& p = pool->p;
  kvint2::DecodePlan pl = p.cfg.kind == KV_POOL_INT2_3TIER ? kvint2::plan_decode_int2(p, B, max_len)
                                                           : kvint2::plan_decode_bf16(p, B, max_len);
  return pl.bytes;
}

kv_status_t kv_decode_attention(kv_pool_t* pool, int32_t layer, int32_t B, const void* q,
                                const int32_t* sink_len, const int32_t* hist_len,
                                const int32_t* recent_len, const int32_t* recent_start,
                                const int32_t* page_table, int32_t max_pages_per_seq,
                                int32_t max_hist_len, float softmax_scale, float* out,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_layer(pool, layer) || B <= 0 || max_pages_per_seq <= 0 || max_hist_len < 0)
    return KV_ERR_INVALID_ARG;
  const Pool& p = pool->p;
  if (p.cfg.kind != KV_POOL_INT2_3TIER || B > p.cfg.max_seqs) return KV_ERR_INVALID_ARG;
  if (!q || !sink_len || !hist_len || !recent_len || !recent_start || !page_table || !out ||
      !workspace)
    return KV_ERR_INVALID_ARG;
  if ((int64_t)max_hist_len > (int64_t)max_pages_per_seq * p.cfg.page_size || max_hist_len > kvint2::kMaxDecodeLen)
    return KV_ERR_INVALID_ARG;
  if (((uintptr_t)workspace & 15) || ((uintptr_t)q & 1)) return KV_ERR_INVALID_ARG;
  kvint2::DecodePlan pl = kvint2::plan_decode_int2(p, B, max_hist_len);
  if (workspace_bytes < pl.bytes) return KV_ERR_INVALID_ARG;
  return cuda_status(kvint2::launch_decode_int2(p, layer, B, q, sink_len, hist_len, recent_len,
                                                recent_start, page_table, max_pages_per_seq, pl,
                                                softmax_scale, out, workspace,
                                                static_cast<cudaStream_t>(stream)));
}

kv_status_t kv_decode_attention_noalloc(kv_pool_t* pool, int32_t layer, int32_t B, const void* q,
                                        const int32_t* sink_len, const int32_t* hist_len,
                                        const int32_t* recent_len, const int32_t* recent_start,
                                        const int32_t* page_table, int32_t max_pages_per_seq,
                                        int32_t max_hist_len, float softmax_scale, float* out,
                                        void* stream) {
  if (!valid_layer(pool, layer) || B <= 0 || max_pages_per_seq <= 0 || max_hist_len < 0)
    return KV_ERR_INVALID_ARG;
  const Pool& p = pool->p;
  if (p.cfg.kind != KV_POOL_INT2_3TIER || B > p.cfg.max_seqs) return KV_ERR_INVALID_ARG;
  if (!q || !sink_len || !hist_len || !recent_len || !recent_start || !page_table || !out)
    return KV_ERR_INVALID_ARG;
  if ((int64_t)max_hist_len > (int64_t)max_pages_per_seq * p.cfg.page_size || max_hist_len > kvint2::kMaxDecodeLen)
    return KV_ERR_INVALID_ARG;
  if ((uintptr_t)q & 1) return KV_ERR_INVALID_ARG;
  // the scratch buffer looked up below is the current device's: it must be the pool's
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return KV_ERR_CUDA;
  if (cur != p.device) return KV_ERR_INVALID_ARG;
  kvint2::DecodePlan pl = kvint2::plan_decode_int2(p, B, max_hist_len);
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  if (kvint2::noalloc_scratch(&scratch, &scratch_bytes) != cudaSuccess) return KV_ERR_CUDA;
  if (pl.bytes > scratch_bytes) return KV_ERR_SCRATCH_LIMIT;
  return cuda_status(kvint2::launch_decode_int2(p, layer, B, q, sink_len, hist_len, recent_len,
                                                recent_start, page_table, max_pages_per_seq, pl,
                                                softmax_scale, out, scratch,
                                                static_cast<cudaStream_t>(stream)));
}

kv_status_t kv_debug_stall_first_copy(kv_pool_t* pool, int32_t enable, int32_t max_polls) {
  if (!pool || max_polls < 0) return KV_ERR_INVALID_ARG;
  pool->p.test_stall_first_copy = enable ? 1 : 0;
  pool->p.test_wait_polls = max_polls;
  return KV_OK;
}

kv_status_t kv_append_bf16(kv_pool_t* pool, int32_t layer, int32_t n_seqs, const void* k,
                           const void* v, const int32_t* cu_tokens, const int32_t* start_pos,
                           const int32_t* page_table, int32_t max_pages_per_seq,
                           int32_t max_tokens_per_seq, void* stream) {
  if (!valid_layer(pool, layer) || n_seqs < 0 || max_pages_per_seq <= 0 || max_tokens_per_seq < 0)
    return KV_ERR_INVALID_ARG;
  if (pool->p.cfg.kind != KV_POOL_BF16) return KV_ERR_INVALID_ARG;
  if (n_seqs > 0 && (!k || !v || !cu_tokens || !start_pos || !page_table)) return KV_ERR_INVALID_ARG;
  if (((uintptr_t)k & 15) || ((uintptr_t)v & 15)) return KV_ERR_INVALID_ARG;
  return cuda_status(kvint2::launch_append_bf16(pool->p, layer, n_seqs, k, v, cu_tokens, start_pos,
                                                page_table, max_pages_per_seq, max_tokens_per_seq,
                                                static_cast<cudaStream_t>(stream)));
}

size_t kv_decode_multi_workspace_bytes(const kv_pool_t* pool, int32_t B, int32_t T,
                                       int32_t max_hist_len) {
  if (!pool || B <= 0 || T <= 0 || max_hist_len < 0 || B > pool->p.cfg.max_seqs) return 0;
  const Pool& p = pool->p;
  if (p.cfg.kind != KV_POOL_INT2_3TIER || !is_pow2_in((int)std::min<int64_t>((int64_t)T * p.G, 16), 1, 8))
    return 0;
  return kvint2::plan_decode_int2(p, B, max_hist_len, T).bytes;
}

kv_status_t kv_decode_attention_multi(kv_pool_t* pool, int32_t layer, int32_t B, int32_t T,
                                      const void* q, const int32_t* sink_len,
                                      const int32_t* hist_len, const int32_t* recent_len,
                                      const int32_t* recent_start, const int32_t* page_table,
                                      int32_t max_pages_per_seq, int32_t max_hist_len,
                                      float softmax_scale, float* out, float* lse,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_layer(pool, layer) || B <= 0 || T <= 0 || max_pages_per_seq <= 0 || max_hist_len < 0)
    return KV_ERR_INVALID_ARG;
  const Pool& p = pool->p;
  if (p.cfg.kind != KV_POOL_INT2_3TIER || B > p.cfg.max_seqs) return KV_ERR_INVALID_ARG;
  if ((int64_t)T * p.G > 8 || !is_pow2_in(T * p.G, 1, 8)) return KV_ERR_UNSUPPORTED;
  if (!q || !sink_len || !hist_len || !recent_len || !recent_start || !page_table || !out ||
      !workspace)
    return KV_ERR_INVALID_ARG;
  if ((int64_t)max_hist_len > (int64_t)max_pages_per_seq * p.cfg.page_size || max_hist_len > kvint2::kMaxDecodeLen)
    return KV_ERR_INVALID_ARG;
  if (((uintptr_t)workspace & 15) || ((uintptr_t)q & 1) || ((uintptr_t)lse & 3)) return KV_ERR_INVALID_ARG;
  kvint2::DecodePlan pl = kvint2::plan_decode_int2(p, B, max_hist_len, T);
  if (workspace_bytes < pl.bytes) return KV_ERR_INVALID_ARG;
  return cuda_status(kvint2::launch_decode_int2(p, layer, B, q, sink_len, hist_len, recent_len,
                                                recent_start, page_table, max_pages_per_seq, pl,
                                                softmax_scale, out, workspace,
                                                static_cast<cudaStream_t>(stream), T, lse));
}

static_assert(kvint2::kMaxDecodeLen == KV_MAX_DECODE_LEN, "one decode length bound");

kv_status_t kv_decode_attention_bf16(kv_pool_t* pool, int32_t layer, int32_t B, const void* q,
                                     const int32_t* seq_len, const int32_t* page_table,
                                     int32_t max_pages_per_seq, int32_t max_seq_len,
                                     float softmax_scale, float* out, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  if (!valid_layer(pool, layer) || B <= 0 || max_pages_per_seq <= 0 || max_seq_len < 0)
    return KV_ERR_INVALID_ARG;
  const Pool& p = pool->p;
  if (p.cfg.kind != KV_POOL_BF16 || B > p.cfg.max_seqs) return KV_ERR_INVALID_ARG;
  if (!q || !seq_len || !page_table || !out || !workspace) return KV_ERR_INVALID_ARG;
  if ((int64_t)max_seq_len > (int64_t)max_pages_per_seq * p.cfg.page_size || max_seq_len > kvint2::kMaxDecodeLen)
    return KV_ERR_INVALID_ARG;
  if (((uintptr_t)workspace & 15) || ((uintptr_t)q & 1)) return KV_ERR_INVALID_ARG;
  kvint2::DecodePlan pl = kvint2::plan_decode_bf16(p, B, max_seq_len);
  if (workspace_bytes < pl.bytes) return KV_ERR_INVALID_ARG;
  return cuda_status(kvint2::launch_decode_bf16(p, layer, B, q, seq_len, page_table,
                                                max_pages_per_seq, pl, softmax_scale, out,
                                                workspace, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
