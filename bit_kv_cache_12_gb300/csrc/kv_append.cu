// Append-side set-up and the plain stores: the parity entry (clip + quantize +
// canonical pack of already rotated fp32 rows), the rotation set-up (the pool's
// copies of R_k and R_v^T and the tensor-core operands built from them), and
// the BF16 stores (BF16 pool pages, sink and recent tiers).  The INT2 appends
// themselves, bulk and per step, run on tcgen05 (kv_append_tc.cu).
//
// Method: yunpan.plus OSCAR write-up, "2. 在线量化与反量化" (a token leaving
// the recent window goes through rotate, clip, quantize and pack, four 2-bit
// codes per byte, into the INT2 history); gist.science OSCAR explainer,
// section 2.2 B (history is stored after the fixed rotation and the clip).
#include "kv_device.cuh"
#include "kv_internal.h"

namespace kvint2 {

namespace {

// ---------------------------------------------------------------------------
// parity entry: clip + quantize + canonical pack of already rotated fp32 rows
// one warp per (row, head); lane owns channels 4*lane .. 4*lane+3 (one byte)
// ---------------------------------------------------------------------------
template <int GS>
__global__ void quantize_pack_kernel(const float* __restrict__ x, const float* __restrict__ clip,
                                     uint8_t* __restrict__ codes, __half2* __restrict__ sz,
                                     long long n_items, int Hkv) {
  const long long item = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (item >= n_items) return;
  const int lane = threadIdx.x & 31;
  const int head = (int)(item % Hkv);
  const float4 v = *reinterpret_cast<const float4*>(x + item * 128 + 4 * lane);
  const float4 c = *reinterpret_cast<const float4*>(clip + head * 128 + 4 * lane);
  float y[4] = {clip_to(v.x, c.x), clip_to(v.y, c.y), clip_to(v.z, c.z), clip_to(v.w, c.w)};
  float mn = fminf(fminf(y[0], y[1]), fminf(y[2], y[3]));
  float mx = fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3]));
  constexpr int kLanes = GS / 4;   // lanes per group
#pragma unroll
  for (int o = 1; o < kLanes; o <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const ScaleZero q = scale_zero(mn, mx);
  uint32_t byte = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) byte |= quant_code(y[e], q) << (2 * e);
  codes[item * 32 + lane] = (uint8_t)byte;
  if ((lane % kLanes) == 0) sz[item * (128 / GS) + lane / kLanes] = __halves2half2(q.sh, q.zh);
}

// ---------------------------------------------------------------------------
// rotation set-up: pool copies of R_k, R_v^T and the rotation operands
// ---------------------------------------------------------------------------
__global__ void rotation_copy_kernel(const float* __restrict__ Rk, const float* __restrict__ Rv,
                                     float* __restrict__ dRk, float* __restrict__ dRvT, int Hkv) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= Hkv * 128 * 128) return;
  const int h = idx >> 14, i = (idx >> 7) & 127, c = idx & 127;
  dRk[idx] = Rk[idx];
  dRvT[idx] = Rv[((size_t)h * 128 + c) * 128 + i];   // RvT[h][i][c] = Rv[h][c][i]
}

__device__ __forceinline__ void split_bf16(float x, uint16_t& hi, uint16_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(l);
}

__device__ __forceinline__ uint32_t pack2(uint16_t a, uint16_t b) { return (uint32_t)a | ((uint32_t)b << 16); }

// Input channel held by fragment k index kappa at k-step s (the lane j of
// kappa owns input channels 32j .. 32j+31, so rows load as 64-byte runs).
__device__ __forceinline__ int in_ch(int s, int kappa) {
  return 32 * ((kappa & 7) >> 1) + 4 * s + 2 * (kappa >> 3) + (kappa & 1);
}

__global__ void rotation_frag_kernel(const float* __restrict__ Rk, const float* __restrict__ Rv,
                                     uint4* __restrict__ frag, int Hkv) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= Hkv * kFragBlocks * 4096) return;
  const int h = idx / (kFragBlocks * 4096), block = (idx / 4096) % kFragBlocks, f = idx & 4095;
  uint4 out;
  if (block == 1 || block == 2) {
    // tcgen05 B operand of x . R (block 1: R_k, block 2: R_v): row n holds
    // R[k][n % 128] for k = 0..127 as its bf16 hi (n < 128) or lo (n >= 128)
    // term; 128-byte rows, channels 0-63 in the first 32 KB, 64-127 in the
    // second; the 16-byte chunk c of row n sits at chunk position c ^ (n % 8)
    // (the 128-byte swizzle)
    const float* R = (block == 1 ? Rk : Rv) + (size_t)h * 16384;
    const int half = f >> 11, n = (f >> 3) & 255, c = (f & 7) ^ (n & 7);
    const int k0 = 64 * half + 8 * c, col = n & 127;
    uint16_t e[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      uint16_t hi, lo;
      split_bf16(R[(size_t)(k0 + u) * 128 + col], hi, lo);
      e[u] = (n < 128) ? hi : lo;
    }
    out = make_uint4(pack2(e[0], e[1]), pack2(e[2], e[3]), pack2(e[4], e[5]), pack2(e[6], e[7]));
  } else {
    // mma.sync B operand of q . R_k (block 0, decode q' = q R_k) or of
    // o' . R_v^T (block 3, the decode's back-rotation) as fp16 hi / lo pairs:
    // fragment f = (k-step s, n-tile nt, lane); element (kappa, n) =
    // M[in_ch(s, kappa)][8 nt + n] for M = R_k or R_v^T, lane (r, j) holding
    // kappa = 2j, 2j+1, 2j+8, 2j+9 (the decode stages its rows in the same
    // channel order)
    const int lane = f & 31, r = lane >> 2, j = lane & 3;
    const int nt = (f >> 5) & 15, s = f >> 9;
    const int col = 8 * nt + r;
    uint16_t hi[4], lo[4];
    const int ks[4] = {2 * j, 2 * j + 1, 2 * j + 8, 2 * j + 9};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int in = in_ch(s, ks[u]);
      const float m = (block == 0) ? Rk[(size_t)h * 16384 + in * 128 + col]
                                   : Rv[(size_t)h * 16384 + col * 128 + in];   // R_v^T[in][col]
      const __half hh = __float2half_rn(m);
      hi[u] = __half_as_ushort(hh);
      lo[u] = __half_as_ushort(__float2half_rn(m - __half2float(hh)));
    }
    out = make_uint4(pack2(hi[0], hi[1]), pack2(hi[2], hi[3]), pack2(lo[0], lo[1]), pack2(lo[2], lo[3]));
  }
  frag[idx] = out;
}

// ---------------------------------------------------------------------------
// BF16 stores: BF16 pool pages and the sink / recent tiers
// ---------------------------------------------------------------------------
__global__ void append_bf16_kernel(uint16_t* __restrict__ bk, uint16_t* __restrict__ bv,
                                   const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                   const int32_t* __restrict__ cu, const int32_t* __restrict__ start,
                                   const int32_t* __restrict__ pt, int max_pages, int max_tokens,
                                   int n_seqs, int Hkv, int P, long long num_pages, int* err) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long per_tok = (long long)Hkv * 16;
  const long long total = (long long)n_seqs * max_tokens * per_tok;
  if (idx >= total) return;
  const int chunk = (int)(idx % 16);
  const int g = (int)((idx / 16) % Hkv);
  const long long vt = idx / per_tok;
  const int s = (int)(vt / max_tokens), i = (int)(vt % max_tokens);
  const int c0 = cu[s], n = cu[s + 1] - c0;
  if (i >= n) return;
  const int pos = start[s] + i;
  if (pos < 0 || pos >= max_pages * P) {
    flag_error(err, KV_DEVERR_SEQ_RANGE);
    return;
  }
  const int pid = pt[(size_t)s * max_pages + pos / P];
  if (pid < 0 || pid >= num_pages) {
    flag_error(err, KV_DEVERR_PAGE_ID);
    return;
  }
  const size_t dst = (((size_t)pid * Hkv + g) * P + pos % P) * 128 + chunk * 8;
  const size_t src = ((size_t)(c0 + i) * Hkv + g) * 128 + chunk * 8;
  *reinterpret_cast<uint4*>(bk + dst) = *reinterpret_cast<const uint4*>(k + src);
  *reinterpret_cast<uint4*>(bv + dst) = *reinterpret_cast<const uint4*>(v + src);
}

__global__ void store_tier_kernel(uint16_t* __restrict__ tk, uint16_t* __restrict__ tv,
                                  const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                  const int32_t* __restrict__ seq, const int32_t* __restrict__ slot,
                                  int n_rows, int Hkv, int cap, int max_seqs, int* err) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)n_rows * Hkv * 16) return;
  const int chunk = (int)(idx % 16);
  const int g = (int)((idx / 16) % Hkv);
  const int row = (int)(idx / (16 * Hkv));
  const int sq = seq[row], sl = slot[row];
  if (sq < 0 || sq >= max_seqs || sl < 0 || sl >= cap) {
    flag_error(err, KV_DEVERR_LENGTH);
    return;
  }
  const size_t dst = (((size_t)sq * Hkv + g) * cap + sl) * 128 + chunk * 8;
  const size_t src = ((size_t)row * Hkv + g) * 128 + chunk * 8;
  *reinterpret_cast<uint4*>(tk + dst) = *reinterpret_cast<const uint4*>(k + src);
  *reinterpret_cast<uint4*>(tv + dst) = *reinterpret_cast<const uint4*>(v + src);
}

}  // namespace

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_rotation_prep(const Pool& p, int layer, const float* Rk, const float* Rv,
                                 cudaStream_t s) {
  const int H = p.cfg.num_kv_heads;
  const size_t mat = (size_t)H * 128 * 128;
  float* dRk = p.Rk + (size_t)layer * mat;
  float* dRvT = p.RvT + (size_t)layer * mat;
  if (Rk != dRk || Rv != dRvT) {
    rotation_copy_kernel<<<(unsigned)((mat + 255) / 256), 256, 0, s>>>(Rk, Rv, dRk, dRvT, H);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  uint4* frag = p.rfrag + (size_t)layer * H * kFragBlocks * rfrag_per_head();
  const int n = H * kFragBlocks * 4096;
  rotation_frag_kernel<<<(n + 255) / 256, 256, 0, s>>>(Rk, Rv, frag, H);
  return cudaGetLastError();
}

cudaError_t launch_store_tier(const Pool& p, int layer, int tier, int n_rows, const void* k,
                              const void* v, const int32_t* seq, const int32_t* slot,
                              cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int H = p.cfg.num_kv_heads;
  uint16_t* tk = tier == 0 ? p.sink_k + (size_t)layer * p.sink_layer_stride
                           : p.rec_k + (size_t)layer * p.rec_layer_stride;
  uint16_t* tv = tier == 0 ? p.sink_v + (size_t)layer * p.sink_layer_stride
                           : p.rec_v + (size_t)layer * p.rec_layer_stride;
  const int cap = tier == 0 ? p.cfg.sink_tokens : p.cfg.recent_tokens;
  const long long n = (long long)n_rows * H * 16;
  store_tier_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
      tk, tv, static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), seq, slot, n_rows,
      H, cap, p.cfg.max_seqs, p.err);
  return cudaGetLastError();
}

cudaError_t launch_quantize_pack(const Pool& p, int layer, int tensor, int64_t n_rows,
                                 const float* x, uint8_t* codes, void* sz, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int H = p.cfg.num_kv_heads;
  const long long items = (long long)n_rows * H;
  const float* clip = p.clip + ((size_t)layer * 2 + tensor) * H * 128;
  const unsigned blocks = (unsigned)((items + 7) / 8);
  if (p.cfg.group_size == 64)
    quantize_pack_kernel<64><<<blocks, 256, 0, s>>>(x, clip, codes, static_cast<__half2*>(sz), items, H);
  else
    quantize_pack_kernel<128><<<blocks, 256, 0, s>>>(x, clip, codes, static_cast<__half2*>(sz), items, H);
  return cudaGetLastError();
}

cudaError_t launch_append(const Pool& p, int layer, int n_seqs, const void* k, const void* v,
                          const int32_t* cu, const int32_t* hist_start, const int32_t* pt,
                          int max_pages, int max_tokens, cudaStream_t s) {
  if (n_seqs == 0 || max_tokens == 0) return cudaSuccess;
  return launch_append_tc(p, layer, n_seqs, k, v, cu, hist_start, pt, max_pages, max_tokens, s);
}

cudaError_t launch_append_bf16(const Pool& p, int layer, int n_seqs, const void* k,
                               const void* v, const int32_t* cu, const int32_t* start,
                               const int32_t* pt, int max_pages, int max_tokens,
                               cudaStream_t s) {
  if (n_seqs == 0 || max_tokens == 0) return cudaSuccess;
  const int H = p.cfg.num_kv_heads;
  const long long n = (long long)n_seqs * max_tokens * H * 16;
  append_bf16_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
      p.bk + (size_t)layer * p.bf16_layer_stride, p.bv + (size_t)layer * p.bf16_layer_stride,
      static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), cu, start, pt, max_pages,
      max_tokens, n_seqs, H, p.cfg.page_size, p.cfg.num_pages, p.err);
  return cudaGetLastError();
}

}  // namespace kvint2
