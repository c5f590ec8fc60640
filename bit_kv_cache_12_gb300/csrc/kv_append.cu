// Append path: rotate -> clip -> asymmetric INT2 quantize -> pack into pages.
//
// Method: yunpan.plus OSCAR write-up, "2. 在线量化与反量化" (a token leaving
// the recent window goes through rotate, clip, quantize and pack, four 2-bit
// codes per byte, into the INT2 history); gist.science OSCAR explainer,
// section 2.2 B (history is stored after the fixed rotation and the clip).
//
// This file holds the per-step placement (a new token per sequence into the
// sink or the recent ring, the evicted token into INT2 history), the parity
// entry (quantize + canonical pack of rotated fp32 rows), the rotation set-up
// and the BF16 stores; the bulk append runs on tcgen05 (kv_append_tc.cu).
//
// Per-step eviction: a warp owns the one 16-token tile of one KV head and one
// tensor that the evicted token lands in.  The rotation x' = x R runs on the
// tensor cores (mma.sync m16n8k16 bf16): x is exact in bf16 and R is split
// into bf16 hi + lo terms, fp32 accumulate.  The MMA accumulator layout is
// arranged so that each lane ends up owning exactly the 64 codes of its own
// 16-byte slot of the stored tile (K: x R with tokens as rows; V: R^T x^T
// with channels as rows), so packing is lane-local; the bits of the tile's
// other rows are kept.
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
// fused append
// ---------------------------------------------------------------------------
__device__ __forceinline__ void load_row64(const uint16_t* row, bool ok, uint32_t (&w)[16]) {
  if (ok) {
    const uint4* p = reinterpret_cast<const uint4*>(row);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint4 t = __ldg(p + u);
      w[4 * u + 0] = t.x; w[4 * u + 1] = t.y; w[4 * u + 2] = t.z; w[4 * u + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < 16; ++u) w[u] = 0u;
  }
}

__device__ __forceinline__ void store_words(uint8_t* dst, const uint32_t (&w)[4],
                                            const uint32_t (&mask)[4], bool full) {
  uint4* p = reinterpret_cast<uint4*>(dst);
  if (full) {
    *p = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    const uint4 o = *p;
    *p = make_uint4((o.x & ~mask[0]) | (w[0] & mask[0]), (o.y & ~mask[1]) | (w[1] & mask[1]),
                    (o.z & ~mask[2]) | (w[2] & mask[2]), (o.w & ~mask[3]) | (w[3] & mask[3]));
  }
}

// One 16-token tile of one KV head and one tensor (0 = K, 1 = V): the rows
// with row_ok(row) are rotated (frag: the tensor's bf16 hi + lo rotation
// fragments), clipped (clip: the tensor's 128 thresholds), quantized and
// packed into the stored tile at tb; the bits and records of the other rows
// are kept unless `full`.  row_ptr(row) points at channel 32 * (lane % 4) of
// the row's bf16 input.  Each output row depends only on its own input row,
// so a token gets the same codes however many tokens share its tile.
template <int GS, int TENSOR, class RowOk, class RowPtr>
__device__ __forceinline__ void append_tile(const uint4* frag, const float* clip,
                                            uint8_t* tb, bool full, const RowOk& row_ok,
                                            const RowPtr& row_ptr) {
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2, j = lane & 3;
  constexpr int NG = 128 / GS;
  uint32_t xr[16], xr8[16];
  load_row64(row_ptr(r), row_ok(r), xr);
  load_row64(row_ptr(r + 8), row_ok(r + 8), xr8);

  uint32_t word[4] = {0u, 0u, 0u, 0u}, mask[4] = {0u, 0u, 0u, 0u};
  if constexpr (TENSOR == 0) {
    // ---- K: D[token][out channel] = x R_k, tokens as MMA rows ----
    float acc[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[nt][u] = 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const uint4 f = frag[(s * 16 + nt) * 32 + lane];
        mma_bf16(acc[nt], xr[2 * s], xr8[2 * s], xr[2 * s + 1], xr8[2 * s + 1], f.x, f.y);
        mma_bf16(acc[nt], xr[2 * s], xr8[2 * s], xr[2 * s + 1], xr8[2 * s + 1], f.z, f.w);
      }
    }
    // clip; per row (token) and group min / max
    float mn[2][NG], mx[2][NG];
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) { mn[q][grp] = INFINITY; mx[q][grp] = -INFINITY; }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int grp = (GS == 64) ? (nt >> 3) : 0;
      const float cl0 = clip[8 * nt + 2 * j], cl1 = clip[8 * nt + 2 * j + 1];
      acc[nt][0] = clip_to(acc[nt][0], cl0);
      acc[nt][1] = clip_to(acc[nt][1], cl1);
      acc[nt][2] = clip_to(acc[nt][2], cl0);
      acc[nt][3] = clip_to(acc[nt][3], cl1);
      mn[0][grp] = fminf(mn[0][grp], fminf(acc[nt][0], acc[nt][1]));
      mx[0][grp] = fmaxf(mx[0][grp], fmaxf(acc[nt][0], acc[nt][1]));
      mn[1][grp] = fminf(mn[1][grp], fminf(acc[nt][2], acc[nt][3]));
      mx[1][grp] = fmaxf(mx[1][grp], fmaxf(acc[nt][2], acc[nt][3]));
    }
    ScaleZero q[2][NG];
#pragma unroll
    for (int qq = 0; qq < 2; ++qq)
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) {
        float a_ = mn[qq][grp], b_ = mx[qq][grp];
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
          a_ = fminf(a_, __shfl_xor_sync(0xffffffffu, a_, o));
          b_ = fmaxf(b_, __shfl_xor_sync(0xffffffffu, b_, o));
        }
        q[qq][grp] = scale_zero(a_, b_);
      }
    const bool ok0 = row_ok(r), ok1 = row_ok(r + 8);
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int grp = (GS == 64) ? (nt >> 3) : 0;
      const int w = nt >> 2;
      const int pi0 = 2 * ((nt >> 1) & 1) + 4 * (nt & 1);   // row r; row r+8 adds 1
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t ca = quant_code(acc[nt][e], q[0][grp]);
        const uint32_t cb = quant_code(acc[nt][2 + e], q[1][grp]);
        const int bit_a = 16 * e + 2 * pi0, bit_b = 16 * e + 2 * (pi0 + 1);
        word[w] |= (ca << bit_a) | (cb << bit_b);
        mask[w] |= (ok0 ? (3u << bit_a) : 0u) | (ok1 ? (3u << bit_b) : 0u);
      }
    }
    store_words(tb + 16 * lane, word, mask, full);
    if (j == 0) {
      const int rec = 8 * NG;
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        if (!(qq ? ok1 : ok0)) continue;
        const int t = r + 8 * qq;
        __half2* recp = reinterpret_cast<__half2*>(tb + 1024 + (2 * (t & 7) + (t >> 3)) * rec);
#pragma unroll
        for (int grp = 0; grp < NG; ++grp) recp[grp] = __halves2half2(q[qq][grp].sh, q[qq][grp].zh);
      }
    }
  } else {
    // ---- V: D[out channel][token] = R_v^T x^T, channels as MMA rows ----
    float acc[8][2][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[i][nt][u] = 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 fh = frag[((i * 8 + s) * 2 + 0) * 32 + lane];
        const uint4 fl = frag[((i * 8 + s) * 2 + 1) * 32 + lane];
        mma_bf16(acc[i][0], fh.x, fh.y, fh.z, fh.w, xr[2 * s], xr[2 * s + 1]);
        mma_bf16(acc[i][0], fl.x, fl.y, fl.z, fl.w, xr[2 * s], xr[2 * s + 1]);
        mma_bf16(acc[i][1], fh.x, fh.y, fh.z, fh.w, xr8[2 * s], xr8[2 * s + 1]);
        mma_bf16(acc[i][1], fl.x, fl.y, fl.z, fl.w, xr8[2 * s], xr8[2 * s + 1]);
      }
    }
    // lane holds tokens 8*nt + 2j + e for channels 16i + r (+8)
    float mn[2][2][NG], mx[2][2][NG];   // [nt][e][grp]
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int grp = 0; grp < NG; ++grp) { mn[nt][e][grp] = INFINITY; mx[nt][e][grp] = -INFINITY; }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int grp = (GS == 64) ? (i >> 2) : 0;
      const float cl0 = clip[16 * i + r], cl1 = clip[16 * i + r + 8];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          acc[i][nt][e] = clip_to(acc[i][nt][e], cl0);
          acc[i][nt][2 + e] = clip_to(acc[i][nt][2 + e], cl1);
          mn[nt][e][grp] = fminf(mn[nt][e][grp], fminf(acc[i][nt][e], acc[i][nt][2 + e]));
          mx[nt][e][grp] = fmaxf(mx[nt][e][grp], fmaxf(acc[i][nt][e], acc[i][nt][2 + e]));
        }
    }
    ScaleZero q[2][2][NG];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int grp = 0; grp < NG; ++grp) {
          float a_ = mn[nt][e][grp], b_ = mx[nt][e][grp];
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            a_ = fminf(a_, __shfl_xor_sync(0xffffffffu, a_, o));
            b_ = fmaxf(b_, __shfl_xor_sync(0xffffffffu, b_, o));
          }
          q[nt][e][grp] = scale_zero(a_, b_);
        }
    bool tok_ok[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) tok_ok[nt][e] = row_ok(8 * nt + 2 * j + e);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int grp = (GS == 64) ? (i >> 2) : 0;
      const int w = i >> 1;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int pi0 = 2 * (i & 1) + 4 * nt;               // channel 16i+r; +8 adds 1
          const uint32_t ca = quant_code(acc[i][nt][e], q[nt][e][grp]);
          const uint32_t cb = quant_code(acc[i][nt][2 + e], q[nt][e][grp]);
          const int bit_a = 16 * e + 2 * pi0, bit_b = 16 * e + 2 * (pi0 + 1);
          word[w] |= (ca << bit_a) | (cb << bit_b);
          if (tok_ok[nt][e]) mask[w] |= (3u << bit_a) | (3u << bit_b);
        }
    }
    store_words(tb + 512 + 16 * lane, word, mask, full);
    if (r == 0) {
      const int rec = 8 * NG;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (!tok_ok[nt][e]) continue;
          const int t = 8 * nt + 2 * j + e;
          __half2* recp =
              reinterpret_cast<__half2*>(tb + 1024 + (2 * (t & 7) + (t >> 3)) * rec) + NG;
#pragma unroll
          for (int grp = 0; grp < NG; ++grp)
            recp[grp] = __halves2half2(q[nt][e][grp].sh, q[nt][e][grp].zh);
        }
    }
  }
}

// ---------------------------------------------------------------------------
// per-step token placement (yunpan.plus write-up, "2. 在线量化与反量化": a new
// token is written to the recent tier; when that is full its oldest token is
// rotated, clipped, quantized and packed into the INT2 history)
// one CTA per sequence; warps take (KV head, tensor) pairs
// ---------------------------------------------------------------------------
struct StepArgs {
  uint8_t* hist;                  // layer base
  size_t page_bytes, head_block;
  int tile_bytes, P;
  uint16_t* sink_k;               // layer bases [max_seqs][Hkv][cap][128]
  uint16_t* sink_v;
  uint16_t* rec_k;
  uint16_t* rec_v;
  int sink_cap, rec_cap;
  const uint16_t* k_new;          // [B][Hkv][128]
  const uint16_t* v_new;
  int32_t* sink_len;
  int32_t* hist_len;
  int32_t* rec_len;
  int32_t* rec_start;
  const int32_t* pt;
  int max_pages, Hkv;
  long long num_pages;
  const uint4* rfrag;             // layer base [Hkv][kFragBlocks][4096]
  const float* clip;              // layer base [2][Hkv][128]
  int* err;
};

// The placement of sequence b's new token, from its current lengths:
// mode 0: sink slot `slot`; 1: recent ring slot `slot`; 2: evict the ring's
// oldest token (slot `slot`) into history position hist_len, which lands at
// row `pos` of the tile at byte offset `tile` of the layer's history, then
// put the new token in that slot; -1: not applied (error code `err`).
struct StepPlace {
  int mode, slot, pos, err;
  long long tile;
};

__device__ StepPlace step_place(const StepArgs& a, int b) {
  StepPlace s{-1, 0, 0, 0, 0};
  const int sl = a.sink_len[b], hl = a.hist_len[b], rl = a.rec_len[b], rs = a.rec_start[b];
  if (sl < 0 || sl > a.sink_cap || rl < 0 || rl > a.rec_cap || rs < 0 || rs >= a.rec_cap || hl < 0) {
    s.err = KV_DEVERR_LENGTH;
  } else if (sl < a.sink_cap) {                    // one of the sequence's first tokens
    s.mode = 0;
    s.slot = sl;
  } else if (rl < a.rec_cap) {                     // the recent ring has room
    s.mode = 1;
    s.slot = (rs + rl) % a.rec_cap;
  } else {                                         // evict the ring's oldest token
    const int pidx = hl / a.P;
    const int pid = (pidx < a.max_pages) ? a.pt[(size_t)b * a.max_pages + pidx] : -1;
    if (pidx >= a.max_pages) {
      s.err = KV_DEVERR_LENGTH;
    } else if (pid < 0 || pid >= a.num_pages) {
      s.err = KV_DEVERR_PAGE_ID;
    } else {
      s.mode = 2;
      s.slot = rs;
      s.pos = hl % kTile;
      s.tile = (long long)pid * (long long)a.page_bytes + (long long)((hl % a.P) / kTile) * a.tile_bytes;
    }
  }
  return s;
}

// Token movement: CTA (sequence chunk, KV head g, tensor); the tensor's
// rotation fragments and clips of head g go to shared memory once and every
// warp places the tokens of its sequences.  The lengths are read only; the
// next kernel updates them.
constexpr int kStepSeqs = 8;   // sequences per CTA
template <int GS>
__global__ void __launch_bounds__(256, 1) append_step_kernel(StepArgs a, int B) {
  extern __shared__ uint4 sfrag[];                 // 4096 fragments, then clip
  float* sclip = reinterpret_cast<float*>(sfrag + 4096);
  const int g = blockIdx.y, tensor = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint4* src_frag = a.rfrag + ((size_t)g * kFragBlocks + tensor) * 4096;
  for (int i = threadIdx.x; i < 4096; i += blockDim.x) sfrag[i] = __ldg(src_frag + i);
  if (threadIdx.x < 128) sclip[threadIdx.x] = a.clip[((size_t)tensor * a.Hkv + g) * 128 + threadIdx.x];
  __syncthreads();
  const int b0 = blockIdx.x * kStepSeqs;
  for (int b = b0 + warp; b < min(B, b0 + kStepSeqs); b += blockDim.x >> 5) {
    const StepPlace pl = step_place(a, b);
    if (pl.mode < 0) continue;
    const size_t sh = (size_t)b * a.Hkv + g;
    const uint16_t* src = (tensor ? a.v_new : a.k_new) + sh * 128;
    uint16_t* dst = (pl.mode == 0)
                        ? (tensor ? a.sink_v : a.sink_k) + (sh * a.sink_cap + pl.slot) * 128
                        : (tensor ? a.rec_v : a.rec_k) + (sh * a.rec_cap + pl.slot) * 128;
    if (pl.mode == 2) {
      // the slot's current token goes to history position pos of its tile
      uint8_t* tb = a.hist + pl.tile + (size_t)g * a.head_block;
      const uint16_t* old = dst;
      const int pos = pl.pos;
      auto row_ok = [&](int row) { return row == pos; };
      auto row_ptr = [&](int) { return old + 32 * (lane & 3); };
      if (tensor == 0)
        append_tile<GS, 0>(sfrag, sclip, tb, false, row_ok, row_ptr);
      else
        append_tile<GS, 1>(sfrag, sclip, tb, false, row_ok, row_ptr);
      __syncwarp();   // every lane has read the old row before it is overwritten
    }
    *reinterpret_cast<uint2*>(dst + 4 * lane) = *reinterpret_cast<const uint2*>(src + 4 * lane);
  }
}

// Length update after the token movement: one thread per sequence, the same
// placement decision from the same (not yet updated) lengths.
__global__ void append_step_lengths_kernel(StepArgs a, int B) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const StepPlace pl = step_place(a, b);
  if (pl.mode == 0) {
    a.sink_len[b] = pl.slot + 1;
  } else if (pl.mode == 1) {
    a.rec_len[b] += 1;
  } else if (pl.mode == 2) {
    a.hist_len[b] += 1;
    a.rec_start[b] = (pl.slot + 1) % a.rec_cap;
  } else {
    flag_error(a.err, pl.err);
  }
}

// ---------------------------------------------------------------------------
// rotation set-up: pool copies of R_k, R_v^T and the bf16 hi/lo MMA fragments
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
// kappa owns input channels 32j .. 32j+31, so x rows load as 64-byte runs).
__device__ __forceinline__ int in_ch(int s, int kappa) {
  return 32 * ((kappa & 7) >> 1) + 4 * s + 2 * (kappa >> 3) + (kappa & 1);
}

__global__ void rotation_frag_kernel(const float* __restrict__ Rk, const float* __restrict__ Rv,
                                     uint4* __restrict__ frag, int Hkv) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= Hkv * kFragBlocks * 4096) return;
  const int h = idx / (kFragBlocks * 4096), tensor = (idx / 4096) % kFragBlocks, f = idx & 4095;
  const int lane = f & 31;
  const int r = lane >> 2, j = lane & 3;
  uint4 out;
  if (tensor >= 3) {
    // tcgen05 B operand of x . R (R = R_k or R_v): row n holds R[k][n % 128] for
    // k = 0..127 as its bf16 hi (n < 128) or lo (n >= 128) term; 128-byte rows,
    // channels 0-63 in the first 32 KB, 64-127 in the second; the 16-byte chunk c
    // of row n sits at chunk position c ^ (n % 8) (the 128-byte swizzle)
    const float* R = (tensor == 3 ? Rk : Rv) + (size_t)h * 16384;
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
  } else if (tensor != 1) {
    // B operand of x R_k: element (kappa, n) = R_k[in_ch(s, kappa)][8 nt + n];
    // block 0 as bf16 hi/lo (append, x in bf16), block 2 as fp16 hi/lo (decode q')
    const int nt = (f >> 5) & 15, s = f >> 9;
    const int col = 8 * nt + r;
    uint16_t hi[4], lo[4];
    const int ks[4] = {2 * j, 2 * j + 1, 2 * j + 8, 2 * j + 9};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float m = Rk[(size_t)h * 16384 + in_ch(s, ks[u]) * 128 + col];
      if (tensor == 0) {
        split_bf16(m, hi[u], lo[u]);
      } else {
        const __half hh = __float2half_rn(m);
        hi[u] = __half_as_ushort(hh);
        lo[u] = __half_as_ushort(__float2half_rn(m - __half2float(hh)));
      }
    }
    out = make_uint4(pack2(hi[0], hi[1]), pack2(hi[2], hi[3]), pack2(lo[0], lo[1]), pack2(lo[2], lo[3]));
  } else {
    // A operand of R_v^T x^T: element (row m, kappa) = R_v[in_ch(s, kappa)][16 i + m]
    const int hl = (f >> 5) & 1, s = (f >> 6) & 7, i = f >> 9;
    const float* R = Rv + (size_t)h * 16384;
    const int rows[2] = {16 * i + r, 16 * i + r + 8};
    const int ks[2][2] = {{2 * j, 2 * j + 1}, {2 * j + 8, 2 * j + 9}};
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {   // a0 (r, k lo), a1 (r+8, k lo), a2 (r, k hi), a3 (r+8, k hi)
      const int m = rows[q & 1];
      uint16_t h0, l0, h1, l1;
      split_bf16(R[in_ch(s, ks[q >> 1][0]) * 128 + m], h0, l0);
      split_bf16(R[in_ch(s, ks[q >> 1][1]) * 128 + m], h1, l1);
      w[q] = hl ? pack2(l0, l1) : pack2(h0, h1);
    }
    out = make_uint4(w[0], w[1], w[2], w[3]);
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

cudaError_t launch_append_step(const Pool& p, int layer, int B, const void* k_new,
                               const void* v_new, int32_t* sink_len, int32_t* hist_len,
                               int32_t* rec_len, int32_t* rec_start, const int32_t* pt,
                               int max_pages, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  const int H = p.cfg.num_kv_heads;
  StepArgs a{};
  a.hist = p.hist + (size_t)layer * p.hist_layer_stride;
  a.page_bytes = p.page_bytes;
  a.head_block = p.page_bytes / H;
  a.tile_bytes = (int)p.tile_bytes;
  a.P = p.cfg.page_size;
  a.sink_k = p.sink_k + (size_t)layer * p.sink_layer_stride;
  a.sink_v = p.sink_v + (size_t)layer * p.sink_layer_stride;
  a.rec_k = p.rec_k + (size_t)layer * p.rec_layer_stride;
  a.rec_v = p.rec_v + (size_t)layer * p.rec_layer_stride;
  a.sink_cap = p.cfg.sink_tokens;
  a.rec_cap = p.cfg.recent_tokens;
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.sink_len = sink_len;
  a.hist_len = hist_len;
  a.rec_len = rec_len;
  a.rec_start = rec_start;
  a.pt = pt;
  a.max_pages = max_pages;
  a.Hkv = H;
  a.num_pages = p.cfg.num_pages;
  a.rfrag = p.rfrag + (size_t)layer * H * kFragBlocks * rfrag_per_head();
  a.clip = p.clip + (size_t)layer * 2 * H * 128;
  a.err = p.err;
  const size_t smem = 4096 * sizeof(uint4) + 128 * sizeof(float);
  static bool attr64 = false, attr128 = false;
  dim3 grid((unsigned)((B + kStepSeqs - 1) / kStepSeqs), H, 2);
  if (p.cfg.group_size == 64) {
    if (!attr64) {
      cudaError_t e = cudaFuncSetAttribute(append_step_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr64 = true;
    }
    append_step_kernel<64><<<grid, 256, smem, s>>>(a, B);
  } else {
    if (!attr128) {
      cudaError_t e = cudaFuncSetAttribute(append_step_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr128 = true;
    }
    append_step_kernel<128><<<grid, 256, smem, s>>>(a, B);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  append_step_lengths_kernel<<<(B + 127) / 128, 128, 0, s>>>(a, B);
  return cudaGetLastError();
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
