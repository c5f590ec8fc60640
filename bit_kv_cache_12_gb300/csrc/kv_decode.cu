// Decode attention over the three-tier INT2 pool and over an all-BF16 pool.
//
// Method: gist.science explainer "OSCAR: Offline Spectral Covariance-Aware
// Rotation for 2-bit KV Cache Quantization", section 2.2 B: one fused kernel
// unpacks and dequantizes the INT2 history, applies the inverse rotation and
// computes attention, next to the BF16 sink and recent tiers (yunpan.plus
// OSCAR write-up, "1. 三段式 Token 池": 64 sink + INT2 history + 256 recent).
//
// GPU design (one launch per decode step):
//   grid = (history splits + 1, KV heads, sequences), 8 warps per CTA.
//   * history CTAs: q' = q R_k for the CTA's GQA group, then each warp streams
//     16-token tiles straight from HBM into registers (16-byte loads, two
//     tiles in flight), unpacks the 2-bit codes into fp16 MMA fragments with
//     one lop3 + one fma per code pair, and runs QK and PV on the tensor cores
//     (mma.sync m16n8k16).  Dequantization is folded algebraically:
//       q'.deq(k) = s_k (q'.(c_k - 1)) + (z_k + s_k) sum(q')
//       sum_t w_t deq(v_t) = sum_t (w_t s_v)(c_v - 1) + sum_t w_t (z_v + s_v)
//     so the MMA operands are small exact integers and the query / softmax
//     weights enter as fp16 hi + lo pairs (about 22 significant bits).
//     Online softmax per head with warp-shuffle max; per-CTA merge in shared
//     memory; the CTA's value accumulator is rotated back by R_v^T.
//   * one tier CTA: the <= 320 BF16 sink + recent tokens in SIMT fp32.
//   * the last CTA of each (sequence, KV head), found by an atomic ticket (no
//     waiting), merges all partials with the log-sum-exp rule and writes the
//     fp32 output.
#include <math.h>

#include "kv_device.cuh"
#include "kv_internal.h"

namespace kvint2 {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kPart = 132;   // floats per (split, head) partial: m, l, -, -, o[128]
constexpr float kNegInf = -INFINITY;

struct DecodeArgs {
  const uint8_t* hist;      // INT2 layer base
  size_t page_bytes;
  int tile_bytes;
  int tiles_per_page;
  const uint16_t* bk;       // BF16 pool layer base
  const uint16_t* bv;
  const uint16_t* sink_k;   // tier layer bases
  const uint16_t* sink_v;
  const uint16_t* rec_k;
  const uint16_t* rec_v;
  int sink_cap, rec_cap;
  const float* Rk;          // layer base [Hkv][128][128]
  const float* RvT;
  const uint16_t* q;
  const int32_t* sink_len;
  const int32_t* hist_len;
  const int32_t* rec_len;
  const int32_t* rec_start;
  const int32_t* seq_len;
  const int32_t* pt;
  int max_pages;
  int Hq, Hkv, page_size;
  long long num_pages;
  int n_split, per_split;
  float scale_log2;
  float* out;
  float* ws;
  unsigned* tickets;
  int* err;
};

// ---------------------------------------------------------------------------
// shared helpers
// ---------------------------------------------------------------------------

// out[h][c] = sum_i in[h][i] R[i][c], h < NH; 256 threads, i split in halves.
template <int NH>
__device__ void rows_times_R(const float* in, const float* __restrict__ R, float* scratch,
                             float* out) {
  const int c = threadIdx.x & 127, half = threadIdx.x >> 7;
  float acc[NH];
#pragma unroll
  for (int h = 0; h < NH; ++h) acc[h] = 0.f;
  const int i0 = half * 64;
#pragma unroll 8
  for (int i = i0; i < i0 + 64; ++i) {
    const float r = __ldg(R + i * 128 + c);
#pragma unroll
    for (int h = 0; h < NH; ++h) acc[h] = fmaf(in[h * 128 + i], r, acc[h]);
  }
#pragma unroll
  for (int h = 0; h < NH; ++h) scratch[(half * NH + h) * 128 + c] = acc[h];
  __syncthreads();
  for (int idx = threadIdx.x; idx < NH * 128; idx += kThreads)
    out[idx] = scratch[idx] + scratch[NH * 128 + idx];
  __syncthreads();
}

// Merge the 8 warps' (m, l, o) in shared memory into one partial per head.
// merged[h][c] receives o; sm_m / sm_l receive m and l.
template <int G>
__device__ void merge_warps(const float* swo, const float* swm, const float* swl, float* merged,
                            float* sm_m, float* sm_l) {
  for (int idx = threadIdx.x; idx < G * 128; idx += kThreads) {
    const int h = idx >> 7;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, swm[w * G + h]);
    float L = 0.f, O = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = swm[w * G + h];
        const float f = (mw == kNegInf) ? 0.f : exp2f(mw - M);
        L = fmaf(f, swl[w * G + h], L);
        O = fmaf(f, swo[(w * G + h) * 128 + (idx & 127)], O);
      }
    }
    merged[idx] = O;
    if ((idx & 127) == 0) {
      sm_m[h] = M;
      sm_l[h] = L;
    }
  }
  __syncthreads();
}

template <int G>
__device__ void write_partial(float* part, const float* o, const float* sm_m, const float* sm_l) {
  for (int idx = threadIdx.x; idx < G * 128; idx += kThreads) {
    const int h = idx >> 7, c = idx & 127;
    part[h * kPart + 4 + c] = o[idx];
    if (c == 0) {
      part[h * kPart + 0] = sm_m[h];
      part[h * kPart + 1] = sm_l[h];
    }
  }
}

template <int G>
__device__ void write_empty_partial(float* part) {
  for (int idx = threadIdx.x; idx < G * 128; idx += kThreads) {
    const int h = idx >> 7, c = idx & 127;
    part[h * kPart + 4 + c] = 0.f;
    if (c == 0) {
      part[h * kPart + 0] = kNegInf;
      part[h * kPart + 1] = 0.f;
    }
  }
}

// The last CTA to arrive for a (sequence, KV head) returns true.  No waiting.
__device__ bool last_to_arrive(unsigned* ticket, unsigned total) {
  __shared__ unsigned s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(ticket, 1u) == total - 1u) ? 1u : 0u;
  __syncthreads();
  const bool last = s_last != 0u;
  if (last) __threadfence();
  return last;
}

// Log-sum-exp merge of all splits of (b, g) and the final normalisation.
template <int G>
__device__ void final_combine(const DecodeArgs& a, int b, int g, int nparts) {
  const float* base = a.ws + (size_t)(b * a.Hkv + g) * nparts * G * kPart;
  for (int idx = threadIdx.x; idx < G * 128; idx += kThreads) {
    const int h = idx >> 7, c = idx & 127;
    float M = kNegInf;
    for (int s = 0; s < nparts; ++s) M = fmaxf(M, __ldcg(base + (s * G + h) * kPart));
    float L = 0.f, O = 0.f;
    if (M != kNegInf) {
      for (int s = 0; s < nparts; ++s) {
        const float* p = base + (s * G + h) * kPart;
        const float ms = __ldcg(p);
        if (ms == kNegInf) continue;
        const float f = exp2f(ms - M);
        L = fmaf(f, __ldcg(p + 1), L);
        O = fmaf(f, __ldcg(p + 4 + c), O);
      }
    }
    a.out[((size_t)b * a.Hq + g * G + h) * 128 + c] = (L > 0.f) ? O / L : 0.f;
  }
  if (threadIdx.x == 0) a.tickets[b * a.Hkv + g] = 0u;   // ready for the next call
}

// ---------------------------------------------------------------------------
// BF16 rows: warp-cooperative SIMT attention over a token range
// (QK with one token per lane, PV with four channels per lane)
// ---------------------------------------------------------------------------
template <int G>
struct WarpAcc {
  float m[G];      // running max (log2 units), uniform across the warp
  float l[G];      // lane-partial sum of weights
  float o[G][4];   // channels 4*lane .. 4*lane+3
  __device__ void init() {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = kNegInf;
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) o[h][e] = 0.f;
    }
  }
};

// rows(u, &k, &v) gives bf16 row pointers for token u (nullptr = skip token).
template <int G, class RowFn>
__device__ void bf16_rows_attend(const float* sq, float* sp, int u0, int u1, int stride,
                                 const RowFn& rows, float scale_log2, WarpAcc<G>& st) {
  const int lane = threadIdx.x & 31;
  for (int c0 = u0; c0 < u1; c0 += stride) {
    const int u = c0 + lane;
    const uint16_t* krow = nullptr;
    const uint16_t* vrow = nullptr;
    if (u < u1) rows(u, krow, vrow);
    float sc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) sc[h] = 0.f;
    if (krow) {
      const uint4* kr = reinterpret_cast<const uint4*>(krow);
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const uint4 w = __ldg(kr + i);
        const float x[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                            bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 q0 = *reinterpret_cast<const float4*>(sq + h * 128 + 8 * i);
          const float4 q1 = *reinterpret_cast<const float4*>(sq + h * 128 + 8 * i + 4);
          float acc = sc[h];
          acc = fmaf(x[0], q0.x, acc); acc = fmaf(x[1], q0.y, acc);
          acc = fmaf(x[2], q0.z, acc); acc = fmaf(x[3], q0.w, acc);
          acc = fmaf(x[4], q1.x, acc); acc = fmaf(x[5], q1.y, acc);
          acc = fmaf(x[6], q1.z, acc); acc = fmaf(x[7], q1.w, acc);
          sc[h] = acc;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float v = krow ? sc[h] * scale_log2 : kNegInf;
      const float mnew = fmaxf(st.m[h], warp_max_xor(v, 1));
      const float alpha = (st.m[h] == kNegInf) ? 0.f : exp2f(st.m[h] - mnew);
      st.m[h] = mnew;
      st.l[h] *= alpha;
#pragma unroll
      for (int e = 0; e < 4; ++e) st.o[h][e] *= alpha;
      const float p = exp2f(v - ((mnew == kNegInf) ? 0.f : mnew));
      st.l[h] += p;
      sp[lane * G + h] = p;
    }
    __syncwarp();
    const int n = min(32, u1 - c0);
    for (int t = 0; t < n; ++t) {
      const uint16_t* vr = reinterpret_cast<const uint16_t*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(vrow), t));
      if (vr == nullptr) continue;   // uniform across the warp
      const uint2 vv = __ldg(reinterpret_cast<const uint2*>(vr) + lane);
      const float v0 = bf16lo(vv.x), v1 = bf16hi(vv.x), v2 = bf16lo(vv.y), v3 = bf16hi(vv.y);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float p = sp[t * G + h];
        st.o[h][0] = fmaf(p, v0, st.o[h][0]);
        st.o[h][1] = fmaf(p, v1, st.o[h][1]);
        st.o[h][2] = fmaf(p, v2, st.o[h][2]);
        st.o[h][3] = fmaf(p, v3, st.o[h][3]);
      }
    }
    __syncwarp();
  }
}

template <int G>
__device__ void warp_acc_to_smem(WarpAcc<G>& st, float* swo, float* swm, float* swl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float l = warp_sum_xor(st.l[h], 1);
    *reinterpret_cast<float4*>(swo + (warp * G + h) * 128 + 4 * lane) =
        make_float4(st.o[h][0], st.o[h][1], st.o[h][2], st.o[h][3]);
    if (lane == 0) {
      swm[warp * G + h] = st.m[h];
      swl[warp * G + h] = l;
    }
  }
}

template <int G>
__device__ void load_q(const DecodeArgs& a, int b, int g, float* sq, int padded_heads) {
  for (int idx = threadIdx.x; idx < padded_heads * 128; idx += kThreads) {
    const int h = idx >> 7, c = idx & 127;
    float v = 0.f;
    if (h < G) v = __uint_as_float((uint32_t)a.q[((size_t)b * a.Hq + g * G + h) * 128 + c] << 16);
    sq[idx] = v;
  }
  __syncthreads();
}

// Shared-memory carve-up (floats) used by both kernels.
template <int G>
struct Smem {
  static constexpr int HP = (G <= 4) ? 4 : 4 * ((G + 3) / 4);   // padded heads (MMA columns)
  static constexpr int sq = 0;                      // [HP][128]
  static constexpr int sqr = sq + HP * 128;          // [HP][128]
  static constexpr int ssum = sqr + HP * 128;        // [HP][2] (padded to 4)
  static constexpr int swo = ssum + ((2 * HP + 3) / 4) * 4;   // [8][G][128]
  static constexpr int swm = swo + kWarps * G * 128;  // [8][G]
  static constexpr int swl = swm + ((kWarps * G + 3) / 4) * 4;
  static constexpr int sp = swl + ((kWarps * G + 3) / 4) * 4;   // [8][32][G]
  static constexpr int scratch = sp + kWarps * 32 * G;          // [2][HP][128]
  static constexpr int smm = scratch + 2 * HP * 128;            // [G] merged m
  static constexpr int sml = smm + ((G + 3) / 4) * 4;
  static constexpr int total = sml + ((G + 3) / 4) * 4;
};

// ---------------------------------------------------------------------------
// INT2 history split (the hot loop)
// ---------------------------------------------------------------------------
template <int GS>
struct TileRegs {
  uint4 k, v, sz0, sz1;
};

template <int G, int GS>
__device__ void int2_history(const DecodeArgs& a, int b, int g, int split, float* sm,
                             float* part) {
  using S = Smem<G>;
  constexpr int NT = S::HP / 4;      // MMA n-tiles of 8 columns (4 heads x hi/lo)
  constexpr int NG = 128 / GS;       // quantization groups per row
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, j = lane & 3;

  int h = a.hist_len[b];
  const int cap = a.max_pages * a.page_size;
  if (h < 0 || h > cap) {
    if (threadIdx.x == 0) flag_error(a.err, KV_DEVERR_LENGTH);
    h = max(0, min(h, cap));
  }
  const int ntiles = (h + kTile - 1) / kTile;
  const int t_begin = split * a.per_split;
  const int t_end = min(ntiles, t_begin + a.per_split);
  if (t_begin >= t_end) {
    write_empty_partial<G>(part);
    return;
  }

  float* sq = sm + S::sq;
  float* sqr = sm + S::sqr;
  float* ssum = sm + S::ssum;
  load_q<G>(a, b, g, sq, S::HP);
  rows_times_R<S::HP>(sq, a.Rk + (size_t)g * 128 * 128, sm + S::scratch, sqr);

  // per-head sums of q' over each quantization group
  for (int hh = warp; hh < S::HP; hh += kWarps) {
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
      float v = 0.f;
      for (int c = grp * GS + lane; c < (grp + 1) * GS; c += 32) v += sqr[hh * 128 + c];
      v = warp_sum_xor(v, 1);
      if (lane == 0) ssum[hh * 2 + grp] = v;
    }
  }
  __syncthreads();

  // QK B fragments: column n = lane/4 -> local head 4*nt + n/2, part n%2 (hi/lo)
  uint32_t qf[8][NT][2];
  {
    const int hl = r >> 1, e = r & 1;
#pragma unroll
    for (int s = 0; s < 8; ++s)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float* row = sqr + (4 * nt + hl) * 128 + 16 * s + 2 * j;
        float x[4] = {row[0], row[1], row[8], row[9]};
        __half p[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const __half hi = __float2half_rn(x[u]);
          p[u] = e ? __float2half_rn(x[u] - __half2float(hi)) : hi;
        }
        qf[s][nt][0] = h2_as_u32(__halves2half2(p[0], p[1]));
        qf[s][nt][1] = h2_as_u32(__halves2half2(p[2], p[3]));
      }
  }
  float sumq[NT][NG];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) sumq[nt][grp] = ssum[(4 * nt + j) * 2 + grp];

  float m_run[NT], l_run[NT], zs[NT][NG], oacc[8][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = kNegInf;
    l_run[nt] = 0.f;
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) zs[nt][grp] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int u = 0; u < 4; ++u) oacc[i][nt][u] = 0.f;
  }

  const int32_t* ptrow = a.pt + (size_t)b * a.max_pages;
  const uint8_t* head_base = a.hist + (size_t)g * (a.page_bytes / a.Hkv);
  auto page_of = [&](int t) -> int {
    if (t >= t_end) return -1;
    return __ldg(ptrow + t / a.tiles_per_page);
  };
  auto load_tile = [&](int t, int pid, TileRegs<GS>& d) {
    if (t >= t_end || pid < 0 || pid >= a.num_pages) {
      d.k = d.v = d.sz0 = d.sz1 = make_uint4(0, 0, 0, 0);
      return;
    }
    const uint8_t* tb =
        head_base + (size_t)pid * a.page_bytes + (size_t)(t % a.tiles_per_page) * a.tile_bytes;
    d.k = ld_stream_v4(tb + 16 * lane);
    d.v = ld_stream_v4(tb + 512 + 16 * lane);
    if (GS == 128) {
      d.sz0 = ld_stream_v4(tb + 1024 + 16 * r);
      d.sz1 = make_uint4(0, 0, 0, 0);
    } else {
      d.sz0 = ld_stream_v4(tb + 1024 + 32 * r);
      d.sz1 = ld_stream_v4(tb + 1024 + 32 * r + 16);
    }
  };

  int t = t_begin + warp;
  int pid0 = page_of(t), pid1 = page_of(t + kWarps), pid2 = page_of(t + 2 * kWarps);
  TileRegs<GS> cur, nxt;
  load_tile(t, pid0, cur);
  load_tile(t + kWarps, pid1, nxt);
  int pid_cur = pid0, pid_nxt = pid1;

  for (; t < t_end; t += kWarps) {
    // prefetch: page id two tiles ahead of the data prefetch, data one tile ahead
    const int pid3 = page_of(t + 3 * kWarps);
    TileRegs<GS> nn;
    load_tile(t + 2 * kWarps, pid2, nn);

    const bool page_ok = pid_cur >= 0 && pid_cur < a.num_pages;
    if (!page_ok && lane == 0) flag_error(a.err, KV_DEVERR_PAGE_ID);
    const bool v0 = page_ok && (t * kTile + r) < h;
    const bool v1 = page_ok && (t * kTile + r + 8) < h;

    // scale / zero of tokens r and r+8
    float sk[2][NG], zk[2][NG], sv[2][NG], zv[2][NG];
    if (GS == 128) {
      const __half2 a0 = u32_as_h2(cur.sz0.x), a1 = u32_as_h2(cur.sz0.y);
      const __half2 b0 = u32_as_h2(cur.sz0.z), b1 = u32_as_h2(cur.sz0.w);
      sk[0][0] = __low2float(a0); zk[0][0] = __high2float(a0);
      sv[0][0] = __low2float(a1); zv[0][0] = __high2float(a1);
      sk[1][0] = __low2float(b0); zk[1][0] = __high2float(b0);
      sv[1][0] = __low2float(b1); zv[1][0] = __high2float(b1);
    } else {
      const uint4 s0 = cur.sz0, s1 = cur.sz1;
      sk[0][0] = __low2float(u32_as_h2(s0.x)); zk[0][0] = __high2float(u32_as_h2(s0.x));
      sk[0][NG - 1] = __low2float(u32_as_h2(s0.y)); zk[0][NG - 1] = __high2float(u32_as_h2(s0.y));
      sv[0][0] = __low2float(u32_as_h2(s0.z)); zv[0][0] = __high2float(u32_as_h2(s0.z));
      sv[0][NG - 1] = __low2float(u32_as_h2(s0.w)); zv[0][NG - 1] = __high2float(u32_as_h2(s0.w));
      sk[1][0] = __low2float(u32_as_h2(s1.x)); zk[1][0] = __high2float(u32_as_h2(s1.x));
      sk[1][NG - 1] = __low2float(u32_as_h2(s1.y)); zk[1][NG - 1] = __high2float(u32_as_h2(s1.y));
      sv[1][0] = __low2float(u32_as_h2(s1.z)); zv[1][0] = __high2float(u32_as_h2(s1.z));
      sv[1][NG - 1] = __low2float(u32_as_h2(s1.w)); zv[1][NG - 1] = __high2float(u32_as_h2(s1.w));
    }

    // ---- QK: scores[token][column] on the tensor cores ----
    float sacc[NG][NT][4];
#pragma unroll
    for (int grp = 0; grp < NG; ++grp)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u) sacc[grp][nt][u] = 0.f;
    {
      const uint32_t kw[4] = {cur.k.x, cur.k.y, cur.k.z, cur.k.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t fr[8];
        unpack_word(kw[w], fr);
#pragma unroll
        for (int sh = 0; sh < 2; ++sh) {
          const int s = 2 * w + sh;
          const int grp = (GS == 64) ? (s >> 2) : 0;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_f16(sacc[grp][nt], fr[4 * sh + 0], fr[4 * sh + 1], fr[4 * sh + 2], fr[4 * sh + 3],
                    qf[s][nt][0], qf[s][nt][1]);
        }
      }
    }

    // ---- softmax update and PV B fragments ----
    uint32_t bpv[NG][NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float l0 = 0.f, l1 = 0.f;
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) {
        const float d0 = sacc[grp][nt][0] + sacc[grp][nt][1];
        const float d1 = sacc[grp][nt][2] + sacc[grp][nt][3];
        l0 += sk[0][grp] * d0 + (zk[0][grp] + sk[0][grp]) * sumq[nt][grp];
        l1 += sk[1][grp] * d1 + (zk[1][grp] + sk[1][grp]) * sumq[nt][grp];
      }
      l0 = v0 ? l0 * a.scale_log2 : kNegInf;
      l1 = v1 ? l1 * a.scale_log2 : kNegInf;
      float tmax = fmaxf(l0, l1);
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
      const float mnew = fmaxf(m_run[nt], tmax);
      const bool need = mnew > m_run[nt];
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ((m_run[nt] == kNegInf) ? 0.f : exp2f(m_run[nt] - mnew)) : 1.f;
        l_run[nt] *= alpha;
#pragma unroll
        for (int grp = 0; grp < NG; ++grp) zs[nt][grp] *= alpha;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int u = 0; u < 4; ++u) oacc[i][nt][u] *= alpha;
      }
      m_run[nt] = mnew;
      const float base = (mnew == kNegInf) ? 0.f : mnew;
      const float p0 = exp2f(l0 - base), p1 = exp2f(l1 - base);
      l_run[nt] += p0 + p1;
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) {
        const float w0 = v0 ? p0 * sv[0][grp] : 0.f;
        const float w1 = v1 ? p1 * sv[1][grp] : 0.f;
        zs[nt][grp] += (v0 ? p0 * (zv[0][grp] + sv[0][grp]) : 0.f) +
                       (v1 ? p1 * (zv[1][grp] + sv[1][grp]) : 0.f);
        bpv[grp][nt][0] = movmatrix_t(split_hi_lo(w0));
        bpv[grp][nt][1] = movmatrix_t(split_hi_lo(w1));
      }
    }

    // ---- PV: value accumulator [channel][column] on the tensor cores ----
    {
      const uint32_t vw[4] = {cur.v.x, cur.v.y, cur.v.z, cur.v.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t fr[8];
        unpack_word(vw[w], fr);
#pragma unroll
        for (int sh = 0; sh < 2; ++sh) {
          const int i = 2 * w + sh;
          const int grp = (GS == 64) ? (i >> 2) : 0;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_f16(oacc[i][nt], fr[4 * sh + 0], fr[4 * sh + 1], fr[4 * sh + 2], fr[4 * sh + 3],
                    bpv[grp][nt][0], bpv[grp][nt][1]);
        }
      }
    }

    cur = nxt;
    nxt = nn;
    pid_cur = pid_nxt;
    pid_nxt = pid2;
    pid2 = pid3;
  }

  // ---- warp results -> shared memory ----
  float* swo = sm + S::swo;
  float* swm = sm + S::swm;
  float* swl = sm + S::swl;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float l = warp_sum_xor(l_run[nt], 4);
    float z[NG];
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) z[grp] = warp_sum_xor(zs[nt][grp], 4);
    const int hh = 4 * nt + j;
    if (hh < G) {
      float* o = swo + (warp * G + hh) * 128;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float zz = z[(GS == 64) ? (i >> 2) : 0];
        o[16 * i + r] = oacc[i][nt][0] + oacc[i][nt][1] + zz;
        o[16 * i + r + 8] = oacc[i][nt][2] + oacc[i][nt][3] + zz;
      }
      if (r == 0) {
        swm[warp * G + hh] = m_run[nt];
        swl[warp * G + hh] = l;
      }
    }
  }
  __syncthreads();
  float* merged = sm + S::sqr;   // q' no longer needed
  merge_warps<G>(swo, swm, swl, merged, sm + S::smm, sm + S::sml);
  // back to the original basis: o = o' R_v^T
  rows_times_R<G>(merged, a.RvT + (size_t)g * 128 * 128, sm + S::scratch, sm + S::sq);
  write_partial<G>(part, sm + S::sq, sm + S::smm, sm + S::sml);
}

// ---------------------------------------------------------------------------
// BF16 sink + recent tiers of the INT2 pool
// ---------------------------------------------------------------------------
template <int G>
__device__ void bf16_tiers(const DecodeArgs& a, int b, int g, float* sm, float* part) {
  using S = Smem<G>;
  const int warp = threadIdx.x >> 5;
  int ns = a.sink_len[b], nr = a.rec_len[b], rs = a.rec_start[b];
  if (ns < 0 || ns > a.sink_cap || nr < 0 || nr > a.rec_cap || rs < 0 || rs >= a.rec_cap) {
    if (threadIdx.x == 0) flag_error(a.err, KV_DEVERR_LENGTH);
    ns = max(0, min(ns, a.sink_cap));
    nr = max(0, min(nr, a.rec_cap));
    rs = max(0, min(rs, a.rec_cap - 1));
  }
  float* sq = sm + S::sq;
  load_q<G>(a, b, g, sq, G);
  const size_t seq_head = (size_t)b * a.Hkv + g;
  const uint16_t* sk = a.sink_k + seq_head * a.sink_cap * 128;
  const uint16_t* sv = a.sink_v + seq_head * a.sink_cap * 128;
  const uint16_t* rk = a.rec_k + seq_head * a.rec_cap * 128;
  const uint16_t* rv = a.rec_v + seq_head * a.rec_cap * 128;
  const int cap = a.rec_cap;
  auto rows = [&](int u, const uint16_t*& kr, const uint16_t*& vr) {
    if (u < ns) {
      kr = sk + (size_t)u * 128;
      vr = sv + (size_t)u * 128;
    } else {
      int idx = rs + (u - ns);
      idx -= (idx >= cap) ? cap : 0;
      kr = rk + (size_t)idx * 128;
      vr = rv + (size_t)idx * 128;
    }
  };
  WarpAcc<G> st;
  st.init();
  bf16_rows_attend<G>(sq, sm + S::sp + warp * 32 * G, 32 * warp, ns + nr, 32 * kWarps, rows,
                      a.scale_log2, st);
  warp_acc_to_smem<G>(st, sm + S::swo, sm + S::swm, sm + S::swl);
  __syncthreads();
  merge_warps<G>(sm + S::swo, sm + S::swm, sm + S::swl, sm + S::sqr, sm + S::smm, sm + S::sml);
  write_partial<G>(part, sm + S::sqr, sm + S::smm, sm + S::sml);
}

template <int G, int GS>
__global__ void __launch_bounds__(kThreads, (G > 4) ? 1 : 2) decode_int2_kernel(DecodeArgs a) {
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int nparts = a.n_split + 1;
  float* part = a.ws + ((size_t)(b * a.Hkv + g) * nparts + split) * G * kPart;
  if (split < a.n_split)
    int2_history<G, GS>(a, b, g, split, sm, part);
  else
    bf16_tiers<G>(a, b, g, sm, part);
  if (last_to_arrive(a.tickets + b * a.Hkv + g, (unsigned)nparts)) final_combine<G>(a, b, g, nparts);
}

// ---------------------------------------------------------------------------
// All-BF16 paged decode (the baseline)
// ---------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(kThreads, 2) decode_bf16_kernel(DecodeArgs a) {
  using S = Smem<G>;
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int nparts = a.n_split;
  float* part = a.ws + ((size_t)(b * a.Hkv + g) * nparts + split) * G * kPart;
  int n = a.seq_len[b];
  const int cap = a.max_pages * a.page_size;
  if (n < 0 || n > cap) {
    if (threadIdx.x == 0) flag_error(a.err, KV_DEVERR_LENGTH);
    n = max(0, min(n, cap));
  }
  const int u0 = split * a.per_split, u1 = min(n, u0 + a.per_split);
  if (u0 >= u1) {
    write_empty_partial<G>(part);
  } else {
    float* sq = sm + S::sq;
    load_q<G>(a, b, g, sq, G);
    const int32_t* ptrow = a.pt + (size_t)b * a.max_pages;
    const int P = a.page_size;
    auto rows = [&](int u, const uint16_t*& kr, const uint16_t*& vr) {
      const int pid = __ldg(ptrow + u / P);
      if (pid < 0 || pid >= a.num_pages) {
        flag_error(a.err, KV_DEVERR_PAGE_ID);
        kr = vr = nullptr;
        return;
      }
      const size_t off = (((size_t)pid * a.Hkv + g) * P + (u % P)) * 128;
      kr = a.bk + off;
      vr = a.bv + off;
    };
    WarpAcc<G> st;
    st.init();
    bf16_rows_attend<G>(sq, sm + S::sp + warp * 32 * G, u0 + 32 * warp, u1, 32 * kWarps, rows,
                        a.scale_log2, st);
    warp_acc_to_smem<G>(st, sm + S::swo, sm + S::swm, sm + S::swl);
    __syncthreads();
    merge_warps<G>(sm + S::swo, sm + S::swm, sm + S::swl, sm + S::sqr, sm + S::smm, sm + S::sml);
    write_partial<G>(part, sm + S::sqr, sm + S::smm, sm + S::sml);
  }
  if (last_to_arrive(a.tickets + b * a.Hkv + g, (unsigned)nparts)) final_combine<G>(a, b, g, nparts);
}

template <class K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int G, int GS>
cudaError_t launch_int2_t(const DecodeArgs& a, int B, cudaStream_t s) {
  const size_t smem = sizeof(float) * Smem<G>::total;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(decode_int2_kernel<G, GS>, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(a.n_split + 1, a.Hkv, B);
  decode_int2_kernel<G, GS><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_bf16_t(const DecodeArgs& a, int B, cudaStream_t s) {
  const size_t smem = sizeof(float) * Smem<G>::total;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(decode_bf16_kernel<G>, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(a.n_split, a.Hkv, B);
  decode_bf16_kernel<G><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

DecodeArgs base_args(const Pool& p, int layer, const void* q, const int32_t* pt, int max_pages,
                     float scale, float* out, void* ws) {
  DecodeArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.pt = pt;
  a.max_pages = max_pages;
  a.Hq = p.cfg.num_q_heads;
  a.Hkv = p.cfg.num_kv_heads;
  a.page_size = p.cfg.page_size;
  a.num_pages = p.cfg.num_pages;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  a.ws = static_cast<float*>(ws);
  a.tickets = p.tickets + (size_t)layer * p.cfg.max_seqs * p.cfg.num_kv_heads;
  a.err = p.err;
  return a;
}

}  // namespace

// ---------------------------------------------------------------------------
// planning and launch
// ---------------------------------------------------------------------------
static DecodePlan make_plan(const Pool& p, int B, int units, int max_units_per_split, int extra) {
  DecodePlan pl;
  const int pairs = B * p.cfg.num_kv_heads;
  const int slots = 2 * p.sm_count;
  int ns = (slots + pairs - 1) / pairs;
  ns = max(1, min(ns, max(1, units)));
  int per = (max(units, 1) + ns - 1) / ns;
  if (per > max_units_per_split) {
    per = max_units_per_split;
  }
  ns = max(1, (max(units, 1) + per - 1) / per);
  pl.n_split = ns;
  pl.tiles_per_split = per;
  pl.partial_floats = (size_t)pairs * (ns + extra) * p.G * kPart;
  pl.bytes = pl.partial_floats * sizeof(float);
  return pl;
}

DecodePlan plan_decode_int2(const Pool& p, int B, int max_hist_len) {
  const int tiles = (max(max_hist_len, 0) + kTile - 1) / kTile;
  return make_plan(p, B, tiles, 512, 1);
}

DecodePlan plan_decode_bf16(const Pool& p, int B, int max_len) {
  return make_plan(p, B, max(max_len, 0), 8192, 0);
}

cudaError_t launch_decode_int2(const Pool& p, int layer, int B, const void* q,
                               const int32_t* sink_len, const int32_t* hist_len,
                               const int32_t* rec_len, const int32_t* rec_start,
                               const int32_t* pt, int max_pages, const DecodePlan& plan,
                               float scale, float* out, void* ws, cudaStream_t s) {
  DecodeArgs a = base_args(p, layer, q, pt, max_pages, scale, out, ws);
  a.hist = p.hist + (size_t)layer * p.hist_layer_stride;
  a.page_bytes = p.page_bytes;
  a.tile_bytes = (int)p.tile_bytes;
  a.tiles_per_page = p.cfg.page_size / kTile;
  a.sink_k = p.sink_k + (size_t)layer * p.sink_layer_stride;
  a.sink_v = p.sink_v + (size_t)layer * p.sink_layer_stride;
  a.rec_k = p.rec_k + (size_t)layer * p.rec_layer_stride;
  a.rec_v = p.rec_v + (size_t)layer * p.rec_layer_stride;
  a.sink_cap = p.cfg.sink_tokens;
  a.rec_cap = p.cfg.recent_tokens;
  a.Rk = p.Rk + (size_t)layer * p.cfg.num_kv_heads * 128 * 128;
  a.RvT = p.RvT + (size_t)layer * p.cfg.num_kv_heads * 128 * 128;
  a.sink_len = sink_len;
  a.hist_len = hist_len;
  a.rec_len = rec_len;
  a.rec_start = rec_start;
  a.n_split = plan.n_split;
  a.per_split = plan.tiles_per_split;
  const bool g64 = p.cfg.group_size == 64;
  switch (p.G) {
    case 1: return g64 ? launch_int2_t<1, 64>(a, B, s) : launch_int2_t<1, 128>(a, B, s);
    case 2: return g64 ? launch_int2_t<2, 64>(a, B, s) : launch_int2_t<2, 128>(a, B, s);
    case 4: return g64 ? launch_int2_t<4, 64>(a, B, s) : launch_int2_t<4, 128>(a, B, s);
    case 8: return g64 ? launch_int2_t<8, 64>(a, B, s) : launch_int2_t<8, 128>(a, B, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_bf16(const Pool& p, int layer, int B, const void* q,
                               const int32_t* seq_len, const int32_t* pt, int max_pages,
                               const DecodePlan& plan, float scale, float* out, void* ws,
                               cudaStream_t s) {
  DecodeArgs a = base_args(p, layer, q, pt, max_pages, scale, out, ws);
  a.bk = p.bk + (size_t)layer * p.bf16_layer_stride;
  a.bv = p.bv + (size_t)layer * p.bf16_layer_stride;
  a.seq_len = seq_len;
  a.n_split = plan.n_split;
  a.per_split = plan.tiles_per_split;
  switch (p.G) {
    case 1: return launch_bf16_t<1>(a, B, s);
    case 2: return launch_bf16_t<2>(a, B, s);
    case 4: return launch_bf16_t<4>(a, B, s);
    case 8: return launch_bf16_t<8>(a, B, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvint2
