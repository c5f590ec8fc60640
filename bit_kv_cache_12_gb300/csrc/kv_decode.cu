// Decode attention over the three-tier INT2 pool and over an all-BF16 pool.
//
// Method: gist.science explainer "OSCAR: Offline Spectral Covariance-Aware
// Rotation for 2-bit KV Cache Quantization", section 2.2 B: one fused kernel
// unpacks and dequantizes the INT2 history, applies the inverse rotation and
// computes attention, next to the BF16 sink and recent tiers (yunpan.plus
// OSCAR write-up, "1. 三段式 Token 池": 64 sink + INT2 history + 256 recent).
//
// GPU design (one launch per decode step):
//   grid = (history splits + tier CTAs, KV heads, sequences); 16 warps per
//   CTA and one CTA per SM for GQA <= 4 (8 warps for GQA 8), and the split
//   count fills one wave when the batch is small.
//   * history CTAs: one round of loads (page ids of the split, q, length),
//     then each warp streams 16-token tiles from HBM through a 4-stage
//     shared-memory ring, one bulk copy per tile completing on the stage's
//     mbarrier (bounded waits), while q' = q R_k runs on the tensor cores.
//     The 2-bit codes become fp16 MMA fragments by masking alone (exact
//     subnormals, one logic op per code pair) and QK and PV run on the tensor
//     cores (mma.sync m16n8k16).  Dequantization is folded:
//       q'.deq(k) = s_k (q'.c_k) + z_k sum(q')
//       sum_t w_t deq(v_t) = sum_t (w_t s_v) c_v + sum_t w_t z_v
//     so the MMA operands are exact small integers times powers of two and the
//     query / softmax weights enter as fp16 hi + lo pairs.  Against subnormal
//     code operands the tensor cores keep only the upper bits of the lo
//     products (about 16 significant bits overall; measured output error
//     about 2e-5 relative to the fp64 oracle at 100k tokens).  Online softmax per head with warp-shuffle max and a
//     lazily moved exponent reference; per-CTA merge in shared memory; each
//     CTA rotates its partial back by R_v^T (fp32, bulk-copied to shared
//     memory at the start).
//   * tier CTAs: stage their slice of the BF16 sink + recent storage into
//     shared memory in the same first round (valid rows are picked once the
//     lengths arrive; softmax order does not matter) and attend in SIMT fp32.
//   * the last CTA of each (sequence, KV head), found by an atomic ticket (no
//     waiting), merges all partials with the log-sum-exp rule and writes the
//     fp32 output (and, for several queries per sequence, the log-sum-exp).
#include <math.h>

#include <atomic>

#include "kv_device.cuh"
#include "kv_internal.h"

namespace kvint2 {

namespace {

constexpr int kPart = 132;       // floats per (part, head) partial: m, l, -, -, o[128]
constexpr float kNegInf = -INFINITY;
constexpr int kStages = 4;       // tiles in each warp's ring
constexpr int kWaitPolls = 1 << 20;   // bounded mbarrier polls before a copy counts as lost
constexpr int kMaxParts = 400;   // partials per (sequence, KV head) the final merge reads
constexpr int kMaxPids = 1032;   // page ids staged per CTA (a split covers <= 1024 tiles)
constexpr int kTierRows = 320;   // sink + recent storage rows staged per tier CTA
constexpr int kTierRowK = 272;   // staged K row stride (bytes): 256 + 16 keeps lane reads conflict-free
constexpr int kTierRowV = 256;
// The history loop keeps each head's exponent reference kSlack (log2 units)
// above the largest score seen when it was last moved, so weights stay <= 1
// and the accumulators are rescaled only when a score passes the reference.
constexpr float kSlack = 4.0f;
constexpr int kBf16Warps = 8;

__host__ __device__ constexpr int int2_warps(int G) { return G <= 4 ? 16 : 12; }
// a split covers at most 64 tiles per warp, and its page ids (one per tile at
// page 16) are staged in shared memory
static_assert(64 * int2_warps(1) <= kMaxPids && 64 * int2_warps(8) <= kMaxPids,
              "a split's page ids must fit the staging array");
__host__ __device__ constexpr int pad4(int n) { return (n + 3) / 4 * 4; }

struct DecodeArgs {
  const uint8_t* hist;      // INT2 layer base
  size_t page_bytes;
  int tile_bytes;
  int tiles_per_page;
  int tpp_shift;            // log2(tiles_per_page)
  const uint16_t* bk;       // BF16 pool layer base
  const uint16_t* bv;
  const uint16_t* sink_k;   // tier layer bases
  const uint16_t* sink_v;
  const uint16_t* rec_k;
  const uint16_t* rec_v;
  int sink_cap, rec_cap;
  const float* RvT;         // layer base [Hkv][128][128], RvT[i][c] = R_v[c][i]
  const uint4* rfrag;       // layer base [Hkv][kFragBlocks][4096] rotation MMA fragments
  const uint16_t* q;
  const int32_t* sink_len;
  const int32_t* hist_len;
  const int32_t* rec_len;
  const int32_t* rec_start;
  const int32_t* seq_len;
  const int32_t* pt;
  int max_pages;
  int max_len;              // host bound on hist_len (INT2) or seq_len (BF16): longer is an error
  int Hq, Hkv, page_size;
  long long num_pages;
  int n_split, per_split, n_tier;
  int wait_polls;           // polls of a bounded mbarrier wait before it gives up
  int stall_first_copy;     // test hook: the first tile copy of split 0 is never issued
  // T query positions per sequence: the kernel's G "heads" of a KV head are
  // (t, h) pairs, t = head / Gq, h = head % Gq (Gq = Hq / Hkv); q and out are
  // [B][T][Hq][128]; lse (optional) [B][T][Hq]
  int T, Gq;
  float* lse;
  float scale_log2;
  float* out;
  float* ws;
  unsigned* tickets;
  int* err;
};

// Shared-memory carve-up (in floats) for a CTA of NW warps.  A fixed head
// (q, q', page ids, merged m/l; for INT2 also the ring barriers and the
// split's per-tile source addresses) is followed by one region reused by
// phase: the history warps' bulk-copy rings, or a tier CTA's staged rows and
// softmax weights, then the per-warp results; the BF16 decode's final merge
// reuses everything (the INT2 final merge reads only global memory).
template <int G, int GS, int NW, bool kInt2>
struct Lay {
  static constexpr int HP = (G <= 4) ? 4 : 4 * ((G + 3) / 4);   // padded heads (MMA columns)
  static constexpr int TB = 1024 + 16 * 8 * (128 / GS);         // stored tile bytes (one ring stage)
  static constexpr int sq = 0;                                    // [HP][128]
  static constexpr int sqr = sq + HP * 128;                       // [HP][128]
  static constexpr int ssum = sqr + HP * 128;                     // [HP][2]
  static constexpr int smm = ssum + pad4(2 * HP);                 // [G] merged m
  static constexpr int sml = smm + pad4(G);                       // [G] merged l
  static constexpr int spid = sml + pad4(G);                      // [kMaxPids] int
  static constexpr int smbar = spid + kMaxPids;                   // [NW * kStages + 1] mbarriers
  static constexpr int saddr = smbar + (kInt2 ? pad4(2 * (NW * kStages + 1)) : 0);   // [64 * NW] u64
  static constexpr int big = saddr + (kInt2 ? 2 * 64 * NW : 0);
  static constexpr int ring_f = kInt2 ? NW * kStages * TB / 4 : 0;
  static constexpr int res_f = NW * G * 128 + 2 * pad4(NW * G);
  static constexpr int sp_f = NW * 32 * G;
  static constexpr int stage_f = kInt2 ? kTierRows * (kTierRowK + kTierRowV) / 4 : 0;
  static constexpr int swo = big;                                 // [NW][G][128]
  static constexpr int swm = swo + NW * G * 128;                  // [NW][G]
  static constexpr int swl = swm + pad4(NW * G);                  // [NW][G]
  static constexpr int ring = big;
  static constexpr int stage = big;                               // tier rows
  static constexpr int sp = big + (stage_f > res_f ? stage_f : res_f);   // [NW][32][G]
  // history CTAs: R_v^T after the ring, and the back-rotation's row-slice sums
  // inside the ring after the results when they fit, else after R_v^T
  static constexpr int srv = big + ring_f;                        // [128][128] R_v^T
  static constexpr int spr_f = NW * G * 128;                      // [NW][G][128]
  static constexpr int spr = (res_f + spr_f <= ring_f) ? big + res_f : srv + 16384;
  static constexpr int rot_end = kInt2 ? ((spr + spr_f > srv + 16384) ? spr + spr_f : srv + 16384) : 0;
  static constexpr int merge_f = 16 + 2 * NW * 128 + 2 * kMaxParts * G;
  static constexpr int phase_end0 = (big + ring_f > sp + sp_f) ? big + ring_f : sp + sp_f;
  static constexpr int phase_end = (phase_end0 > rot_end) ? phase_end0 : rot_end;
  static constexpr int total = (phase_end > merge_f) ? phase_end : merge_f;
  static_assert(total * 4 <= 227 * 1024, "shared memory of one CTA");
};

// ---------------------------------------------------------------------------
// shared helpers
// ---------------------------------------------------------------------------

// R_k's MMA fragments for rotate_q, held in registers: warp w of NW produces
// q' columns (128/NW)w .., and each lane loads all its fragments at once (one
// memory latency), so the load can be issued early and overlap other loads.
template <int NW>
struct RotFrags {
  static constexpr int NTW = (16 + NW - 1) / NW;   // 8-column n-tiles per warp: warp, warp + NW, ..
  uint4 f[8][NTW];
  __device__ __forceinline__ void load(const uint4* __restrict__ frag) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int s = 0; s < 8; ++s)
#pragma unroll
      for (int u = 0; u < NTW; ++u)
        f[s][u] = (warp + u * NW < 16) ? __ldg(frag + (s * 16 + warp + u * NW) * 32 + lane)
                                       : make_uint4(0u, 0u, 0u, 0u);
  }
};

// q'[h][c] = sum_i q[h][i] R_k[i][c] for the first NROWS rows of X (shared,
// [*][128] fp32 holding bf16 values), on the tensor cores: R_k comes as fp16
// hi + lo B fragments (rotation fragment block 0, loaded by RotFrags), q is
// scaled by 2^-8 (exact) and split into fp16 hi + lo, and the three products
// above 2^-22 relative are accumulated in fp32.  Ends with a barrier.
template <int NROWS, int NW>
__device__ void rotate_q(const float* X, const RotFrags<NW>& fr, float* Y) {
  static_assert(NROWS <= 8, "rows");
  constexpr int NTW = RotFrags<NW>::NTW;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, j = lane & 3;
  const auto& f = fr.f;
  float acc[NTW][4];
#pragma unroll
  for (int u = 0; u < NTW; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
  const bool row_ok = r < NROWS;
  constexpr float kIn = 1.0f / 256.0f;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    // A: row r, k index kappa -> input channel 32*(kappa%8/2) + 4s + 2*(kappa/8) + kappa%2
    float4 x = row_ok ? *reinterpret_cast<const float4*>(X + r * 128 + 32 * j + 4 * s)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    x.x *= kIn; x.y *= kIn; x.z *= kIn; x.w *= kIn;
    const __half2 h01 = __floats2half2_rn(x.x, x.y), h23 = __floats2half2_rn(x.z, x.w);
    const __half2 l01 = __floats2half2_rn(x.x - __low2float(h01), x.y - __high2float(h01));
    const __half2 l23 = __floats2half2_rn(x.z - __low2float(h23), x.w - __high2float(h23));
    const uint32_t a0 = h2_as_u32(h01), a2 = h2_as_u32(h23);
    const uint32_t b0 = h2_as_u32(l01), b2 = h2_as_u32(l23);
#pragma unroll
    for (int u = 0; u < NTW; ++u) {
      mma_f16(acc[u], a0, 0u, a2, 0u, f[s][u].x, f[s][u].y);   // hi * hi
      mma_f16(acc[u], a0, 0u, a2, 0u, f[s][u].z, f[s][u].w);   // hi * lo
      mma_f16(acc[u], b0, 0u, b2, 0u, f[s][u].x, f[s][u].y);   // lo * hi
    }
  }
  if (row_ok) {
#pragma unroll
    for (int u = 0; u < NTW; ++u)
      if (warp + u * NW < 16)
        *reinterpret_cast<float2*>(Y + r * 128 + 8 * (warp + u * NW) + 2 * j) =
            make_float2(acc[u][0] * 256.0f, acc[u][1] * 256.0f);
  }
  __syncthreads();
}

// Merge the NW warps' (m, l, o) in shared memory into one partial per head.
// merged[h][c] receives o; sm_m / sm_l receive m and l.
template <int G, int NW>
__device__ void merge_warps(const float* swo, const float* swm, const float* swl, float* merged,
                            float* sm_m, float* sm_l) {
  for (int idx = threadIdx.x; idx < G * 128; idx += NW * 32) {
    const int h = idx >> 7;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, swm[w * G + h]);
    float L = 0.f, O = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
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

// merge_warps for the history split, writing the merged o transposed for
// rotate_back_to_part: oT[c][hh] (GP = heads padded to 4; padded heads 0).
// The weight of each (warp, head) against the head's maximum is formed once
// (sf: NW * G floats of scratch), then every output element sums over warps.
template <int G, int NW>
__device__ void merge_warps_t(const float* swo, const float* swm, const float* swl, float* oT,
                              float* sm_m, float* sm_l, float* sf) {
  constexpr int GP = (G + 3) & ~3;
  if (threadIdx.x < NW * G) {   // weight of warp w for head h against the head's maximum
    const int w = threadIdx.x / G, h = threadIdx.x % G;
    float M = kNegInf;
#pragma unroll
    for (int v = 0; v < NW; ++v) M = fmaxf(M, swm[v * G + h]);
    const float mw = swm[w * G + h];
    sf[w * G + h] = (mw == kNegInf) ? 0.f : exp2f(mw - M);
    if (w == 0) sm_m[h] = M;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < GP * 128; idx += NW * 32) {
    const int h = idx >> 7, c = idx & 127;
    float O = 0.f;
    if (h < G) {
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = sf[w * G + h];
        L = fmaf(f, swl[w * G + h], L);
        O = fmaf(f, swo[(w * G + h) * 128 + c], O);
      }
      if (c == 0) sm_l[h] = L;
    }
    oT[c * GP + h] = O;
  }
  __syncthreads();
}

template <int G, int NW>
__device__ void write_partial(float* part, const float* o, const float* sm_m, const float* sm_l) {
  for (int idx = threadIdx.x; idx < G * 128; idx += NW * 32) {
    const int h = idx >> 7, c = idx & 127;
    part[h * kPart + 4 + c] = o[idx];
    if (c == 0) {
      part[h * kPart + 0] = sm_m[h];
      part[h * kPart + 1] = sm_l[h];
    }
  }
}

template <int G, int NW>
__device__ void write_empty_partial(float* part) {
  for (int idx = threadIdx.x; idx < G * 128; idx += NW * 32) {
    const int h = idx >> 7, c = idx & 127;
    part[h * kPart + 4 + c] = 0.f;
    if (c == 0) {
      part[h * kPart + 0] = kNegInf;
      part[h * kPart + 1] = 0.f;
    }
  }
}

// The last CTA to arrive for a (sequence, KV head) returns true.  No waiting.
// The barrier orders every thread's partial writes before thread 0's
// acquire-release increment, which publishes them at GPU scope (release is
// cumulative); the CTA that takes the last ticket acquires every other CTA's
// writes, and its second barrier hands them to all of its threads.
__device__ bool last_to_arrive(unsigned* ticket, unsigned total) {
  __shared__ unsigned s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(ticket) : "memory");
    s_last = (old == total - 1u) ? 1u : 0u;
  }
  __syncthreads();
  return s_last != 0u;
}

// Rotate a history split's merged value sums back to the original basis,
// o[h][c] = sum_i o'[h][i] R_v[c][i] = sum_i o'[h][i] R_v^T[i][c], straight
// into the split's partial in global memory (with the merged m and l).  o'
// arrives transposed, oT [128][GP]; each row of R_v^T (shared memory) is read
// once for all heads: warp w takes rows w, w + NW, .., lane c columns
// 4c..4c+3, and the NW row-slice sums (spr) are added while storing.
template <int G, int NW>
__device__ void rotate_back_to_part(const float* oT, const float* sR, float* spr, float* part,
                                    const float* sm_m, const float* sm_l) {
  constexpr int GP = (G + 3) & ~3;
  const int warp = threadIdx.x >> 5, cq = threadIdx.x & 31;
  float acc[GP][4];
#pragma unroll
  for (int hh = 0; hh < GP; ++hh) acc[hh][0] = acc[hh][1] = acc[hh][2] = acc[hh][3] = 0.f;
#pragma unroll 4
  for (int i = warp; i < 128; i += NW) {   // rows of R_v^T: warp, warp + NW, ..
    const float4 r = *reinterpret_cast<const float4*>(sR + i * 128 + 4 * cq);
#pragma unroll
    for (int hq = 0; hq < GP / 4; ++hq) {
      const float4 o = *reinterpret_cast<const float4*>(oT + i * GP + 4 * hq);
      const float ox[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float* d = acc[4 * hq + e];
        d[0] = fmaf(ox[e], r.x, d[0]); d[1] = fmaf(ox[e], r.y, d[1]);
        d[2] = fmaf(ox[e], r.z, d[2]); d[3] = fmaf(ox[e], r.w, d[3]);
      }
    }
  }
#pragma unroll
  for (int hh = 0; hh < G; ++hh)
    *reinterpret_cast<float4*>(spr + (warp * G + hh) * 128 + 4 * cq) =
        make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * 128; idx += NW * 32) {
    const int h = idx >> 7, c = idx & 127;
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) O += spr[w * G * 128 + idx];
    part[h * kPart + 4 + c] = O;
    if (c == 0) {
      part[h * kPart + 0] = sm_m[h];
      part[h * kPart + 1] = sm_l[h];
    }
  }
}

// Log-sum-exp merge of all parts of (b, g) (every part in the original basis)
// and the final normalisation, in one pass with no barrier: thread (h, c)
// merges output element c of head h over the parts itself, a batch of
// kMergeBatch parts per round of loads (m and l of a part are the same for
// all 128 threads of a head and arrive as broadcasts).  Within a batch the
// weights are 2^(m_s - M) against the batch's running maximum M; a later batch
// with a larger maximum rescales what is accumulated so far.
constexpr int kMergeBatch = 20;

template <int G, int NW, bool kMulti>
__device__ void merge_parts(const DecodeArgs& a, int b, int g, int nparts, float* sm) {
  (void)sm;
  const float* base = a.ws + (size_t)(b * a.Hkv + g) * nparts * G * kPart;
  for (int idx = threadIdx.x; idx < G * 128; idx += NW * 32) {
    const int hh = idx >> 7, c = idx & 127;
    const float* ph = base + (size_t)hh * kPart;
    float M = kNegInf, L = 0.f, O = 0.f;
    for (int s0 = 0; s0 < nparts; s0 += kMergeBatch) {
      float mv[kMergeBatch], lv[kMergeBatch], ov[kMergeBatch];
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const int s = s0 + u;
        const float* pp = ph + (size_t)s * G * kPart;
        const float2 ml = (s < nparts) ? __ldcg(reinterpret_cast<const float2*>(pp))
                                       : make_float2(kNegInf, 0.f);
        mv[u] = ml.x;
        lv[u] = ml.y;
        ov[u] = (s < nparts) ? __ldcg(pp + 4 + c) : 0.f;
      }
      float Mb = M;
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) Mb = fmaxf(Mb, mv[u]);
      if (Mb != kNegInf) {
        const float alpha = (M == kNegInf) ? 0.f : exp2f(M - Mb);
        L *= alpha;
        O *= alpha;
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          const float f = (mv[u] == kNegInf) ? 0.f : exp2f(mv[u] - Mb);
          L = fmaf(f, lv[u], L);
          O = fmaf(f, ov[u], O);
        }
        M = Mb;
      }
    }
    if constexpr (kMulti) {
      const size_t row = ((size_t)b * a.T + hh / a.Gq) * a.Hq + g * a.Gq + hh % a.Gq;
      a.out[row * 128 + c] = (L > 0.f) ? O / L : 0.f;
      // ln sum exp(scaled score) = ln 2 * (M + log2 L), the scores being in log2 units
      if (a.lse && c == 0) a.lse[row] = (L > 0.f) ? 0.6931471805599453f * (M + log2f(L)) : kNegInf;
    } else {
      a.out[((size_t)b * a.Hq + g * G + hh) * 128 + c] = (L > 0.f) ? O / L : 0.f;
    }
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

// A zero bf16 row: stands in for tokens a warp must not read (past the end of
// the range or behind an invalid page id); their weight is forced to 0.
__device__ __align__(16) uint16_t g_zero_row[128];
// A zero INT2 tile (largest tile size): copied in place of a tile behind an
// invalid page id, so every ring slot always holds finite data.
__device__ __align__(16) uint8_t g_zero_tile[1280];

template <bool kShared, class T>
__device__ __forceinline__ T load_row(const T* p) {
  if (kShared) return *p;   // rows staged in shared memory (generic load)
  return __ldg(p);
}

// rows(u, k, v) sets bf16 row pointers for token u and returns false if the
// token must be skipped.  All loads of a phase are issued before their use.
template <int G, bool kShared, class RowFn>
__device__ void bf16_rows_attend(const float* sq, float* sp, int u0, int u1, int stride,
                                 const RowFn& rows, float scale_log2, WarpAcc<G>& st) {
  const int lane = threadIdx.x & 31;
  for (int c0 = u0; c0 < u1; c0 += stride) {
    const int u = c0 + lane;
    const uint16_t* krow = g_zero_row;
    const uint16_t* vrow = g_zero_row;
    bool ok = false;
    if (u < u1) ok = rows(u, krow, vrow);
    if (!ok) krow = vrow = g_zero_row;
    float sc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) sc[h] = 0.f;
    const uint4* kr = reinterpret_cast<const uint4*>(krow);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint4 kk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) kk[i] = load_row<kShared>(kr + half * 8 + i);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 w = kk[i];
        const float x[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                            bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
        const int cbase = 8 * (half * 8 + i);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 q0 = *reinterpret_cast<const float4*>(sq + h * 128 + cbase);
          const float4 q1 = *reinterpret_cast<const float4*>(sq + h * 128 + cbase + 4);
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
      const float v = ok ? sc[h] * scale_log2 : kNegInf;
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
    const unsigned long long vbits = reinterpret_cast<unsigned long long>(vrow);
#pragma unroll
    for (int tb = 0; tb < 4; ++tb) {
      uint2 vv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint16_t* vr =
            reinterpret_cast<const uint16_t*>(__shfl_sync(0xffffffffu, vbits, tb * 8 + e));
        vv[e] = load_row<kShared>(reinterpret_cast<const uint2*>(vr) + lane);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int t = tb * 8 + e;
        const float v0 = bf16lo(vv[e].x), v1 = bf16hi(vv[e].x);
        const float v2 = bf16lo(vv[e].y), v3 = bf16hi(vv[e].y);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float p = sp[t * G + h];
          st.o[h][0] = fmaf(p, v0, st.o[h][0]);
          st.o[h][1] = fmaf(p, v1, st.o[h][1]);
          st.o[h][2] = fmaf(p, v2, st.o[h][2]);
          st.o[h][3] = fmaf(p, v3, st.o[h][3]);
        }
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

// q of the GQA group (bf16 -> fp32) into shared memory; padded heads are 0.
// No barrier.
template <int G, int NW, bool kMulti = false>
__device__ void load_q(const DecodeArgs& a, int b, int g, float* sq, int padded_heads) {
  for (int idx = threadIdx.x; idx < padded_heads * 128; idx += NW * 32) {
    const int h = idx >> 7, c = idx & 127;
    float v = 0.f;
    if (h < G) {
      const size_t row = kMulti ? ((size_t)b * a.T + h / a.Gq) * a.Hq + g * a.Gq + h % a.Gq
                                : (size_t)b * a.Hq + g * G + h;
      v = __uint_as_float((uint32_t)a.q[row * 128 + c] << 16);
    }
    sq[idx] = v;
  }
}

// ---------------------------------------------------------------------------
// INT2 history split (the hot loop)
// ---------------------------------------------------------------------------
template <int G, int GS, bool kMulti>
__device__ void int2_history(const DecodeArgs& a, int b, int g, int split, float* sm,
                             float* part) {
  constexpr int NW = int2_warps(G);
  using S = Lay<G, GS, NW, true>;
  constexpr int NT = S::HP / 4;      // MMA n-tiles of 8 columns (4 heads x hi/lo)
  constexpr int NG = 128 / GS;       // quantization groups per row
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, j = lane & 3;

  // ---- barriers, then one round of independent loads: R_k's fragments, the
  // split's page ids, q and the length.  Lane 0 of each warp also reads the
  // page ids of its first tiles itself, so that their copies start as soon as
  // the page table answers, while q' is still being formed. ----
  // A ring stage holds one whole stored tile, brought in by one bulk copy that
  // lane 0 issues and that completes on the stage's mbarrier; R_v^T (for the
  // back-rotation of the partial) comes the same way on its own barrier.
  constexpr uint32_t TB = S::TB;
  uint8_t* ring = reinterpret_cast<uint8_t*>(sm + S::ring) + (size_t)warp * kStages * TB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::smbar);
  uint64_t* wbar = bars + warp * kStages;
  uint64_t* rbar = bars + NW * kStages;
  float* srv = sm + S::srv;
  uint64_t* saddr = reinterpret_cast<uint64_t*>(sm + S::saddr);   // per-tile source addresses
  if (lane < kStages) mbar_init(wbar + lane, 1);
  if (threadIdx.x == 0) mbar_init(rbar, 1);
  mbar_fence_init();

  const int tsh = a.tpp_shift, tmask = a.tiles_per_page - 1;
  const int t_begin = split * a.per_split;
  const int p_begin = t_begin >> tsh;
  const int p_all = min(((t_begin + a.per_split - 1) >> tsh) + 1, a.max_pages) - p_begin;
  const int32_t* ptrow = a.pt + (size_t)b * a.max_pages;
  int pid_first[kStages - 1];
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) {
      const int pg = (t_begin + warp + NW * st) >> tsh;
      pid_first[st] = (pg < a.max_pages) ? __ldg(ptrow + pg) : -1;
    }
  }
  RotFrags<NW> rk;
  rk.load(a.rfrag + ((size_t)g * kFragBlocks + 0) * 4096);
  int* spid = reinterpret_cast<int*>(sm + S::spid);
  for (int i = threadIdx.x; i < p_all; i += NW * 32) spid[i] = __ldg(ptrow + p_begin + i);
  float* sq = sm + S::sq;
  float* sqr = sm + S::sqr;
  float* ssum = sm + S::ssum;
  load_q<G, NW, kMulti>(a, b, g, sq, S::HP);
  int h = __ldg(a.hist_len + b);
  // the grid covers max_len history tokens (and the page table max_pages pages)
  const int cap = min(a.max_pages * a.page_size, a.max_len);
  if (h < 0 || h > cap) {
    if (threadIdx.x == 0) flag_error(a.err, KV_DEVERR_LENGTH);
    h = max(0, min(h, cap));
  }
  const int ntiles = (h + kTile - 1) / kTile;
  const int t_end = min(ntiles, t_begin + a.per_split);
  if (t_begin >= t_end) {   // the same for every thread: no copy was started
    write_empty_partial<G, NW>(part);
    return;
  }

  // ---- start streaming this warp's first tiles into its ring ----
  const uint8_t* head_base = a.hist + (size_t)g * (a.page_bytes / a.Hkv);
  const int lane_sz = (GS == 128) ? 1024 + 16 * r : 1024 + 32 * r;
  auto start_copy = [&](int t, int pid, int stage) {
    const uint8_t* tb = (pid >= 0 && pid < a.num_pages)
                            ? head_base + (size_t)pid * a.page_bytes + (t & tmask) * a.tile_bytes
                            : g_zero_tile;
    mbar_expect_tx(wbar + stage, TB);
    bulk_g2s(ring + stage * TB, tb, TB, wbar + stage);
  };
  auto issue = [&](int t, int stage) {   // tiles k >= kStages - 1, from the address table
    if (lane == 0 && t < t_end) {
      const uint64_t e = saddr[t - t_begin];
      mbar_expect_tx(wbar + stage, TB);
      bulk_g2s(ring + stage * TB, reinterpret_cast<const void*>(e & ~1ull), TB, wbar + stage);
    }
  };
  __syncwarp();   // this warp's barriers are initialised
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) {   // tiles 0..2
      const int t = t_begin + warp + NW * st;
      if (t >= t_end) continue;
      if (st == 0 && a.stall_first_copy && split == 0 && warp == 0)
        mbar_expect_tx(wbar, TB);   // test hook: armed for a copy that is never issued
      else
        start_copy(t, pid_first[st], st);
    }
  }
  if (threadIdx.x == 0) {
    const float* R = a.RvT + (size_t)g * 128 * 128;
    mbar_expect_tx(rbar, 128 * 128 * 4);
#pragma unroll
    for (int c = 0; c < 4; ++c) bulk_g2s(srv + 4096 * c, R + 4096 * c, 16384, rbar);
  }
  __syncthreads();   // q and the page ids are in shared memory

  // ---- the source address of every tile of the split, bit 0 set when its
  // page id is valid (else the copy reads a zero tile and its tokens are
  // masked); bad page ids are reported here, once per tile ----
  for (int i = threadIdx.x; i < t_end - t_begin; i += NW * 32) {
    const int t = t_begin + i;
    const int pid = spid[(t >> tsh) - p_begin];
    if (pid >= 0 && pid < a.num_pages) {
      saddr[i] = reinterpret_cast<uint64_t>(head_base + (size_t)pid * a.page_bytes +
                                            (t & tmask) * a.tile_bytes) | 1ull;
    } else {
      saddr[i] = reinterpret_cast<uint64_t>(g_zero_tile);
      flag_error(a.err, KV_DEVERR_PAGE_ID);
    }
  }

  // ---- q' = q R_k and its per-group sums (overlaps the first copies) ----
  rotate_q<S::HP, NW>(sq, rk, sqr);
  for (int hh = warp; hh < S::HP; hh += NW) {
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
        // group 64: the odd steps' code factor 16 is cancelled here (a power of 2);
        // group 128 removes it from the odd steps' accumulator chain instead
        const float f = (GS == 64 && (s & 1)) ? 0.0625f : 1.0f;
        const float x[4] = {row[0] * f, row[1] * f, row[8] * f, row[9] * f};
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
  // per-group sums of q' in the units of the score accumulator (2^-24)
  float sumq[NT][NG];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) sumq[nt][grp] = ssum[(4 * nt + j) * 2 + grp] * 5.9604644775390625e-8f;
  const float sc24 = a.scale_log2 * 16777216.0f;   // 2^24 back on the scores

  // base: the exponent reference as used (0 while m_run is still -inf)
  float m_run[NT], base[NT], l_run[NT], zs[NT][NG], oacc[8][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = kNegInf;
    base[nt] = 0.f;
    l_run[nt] = 0.f;
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) zs[nt][grp] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int u = 0; u < 4; ++u) oacc[i][nt][u] = 0.f;
  }

  int k = 0;
  bool ok = true;
#pragma unroll 2   // lets one tile's loads, unpack and QK overlap the previous tile's softmax and PV
  for (int t = t_begin + warp; t < t_end; t += NW, ++k) {
    __syncwarp();   // every lane is done with the stage refilled next
    // tile k+3 goes into the stage read in the previous iteration
    issue(t + NW * (kStages - 1), (k + kStages - 1) % kStages);
    const int st = k % kStages;
    if (!__all_sync(0xffffffffu, mbar_wait(wbar + st, (k / kStages) & 1, a.wait_polls))) {
      ok = false;
      break;
    }
    const uint8_t* src = ring + st * TB;
    const uint4 kq4 = *reinterpret_cast<const uint4*>(src + 16 * lane);
    const uint4 vq4 = *reinterpret_cast<const uint4*>(src + 512 + 16 * lane);
    const uint4 sz0 = *reinterpret_cast<const uint4*>(src + lane_sz);
    const uint4 sz1 =
        (GS == 64) ? *reinterpret_cast<const uint4*>(src + lane_sz + 16) : make_uint4(0, 0, 0, 0);
    // tokens of this tile still inside the history (none if its page id is bad)
    const int lim = ((saddr[t - t_begin] & 1ull) != 0) ? h - t * kTile : 0;
    const bool v0 = r < lim;
    const bool v1 = r + 8 < lim;

    // scale / zero of tokens r and r+8
    float sk[2][NG], zk[2][NG], sv[2][NG], zv[2][NG];
    if (GS == 128) {
      const __half2 a0 = u32_as_h2(sz0.x), a1 = u32_as_h2(sz0.y);
      const __half2 b0 = u32_as_h2(sz0.z), b1 = u32_as_h2(sz0.w);
      sk[0][0] = __low2float(a0); zk[0][0] = __high2float(a0);
      sv[0][0] = __low2float(a1); zv[0][0] = __high2float(a1);
      sk[1][0] = __low2float(b0); zk[1][0] = __high2float(b0);
      sv[1][0] = __low2float(b1); zv[1][0] = __high2float(b1);
    } else {
      const uint4 s0 = sz0, s1 = sz1;
      sk[0][0] = __low2float(u32_as_h2(s0.x)); zk[0][0] = __high2float(u32_as_h2(s0.x));
      sk[0][NG - 1] = __low2float(u32_as_h2(s0.y)); zk[0][NG - 1] = __high2float(u32_as_h2(s0.y));
      sv[0][0] = __low2float(u32_as_h2(s0.z)); zv[0][0] = __high2float(u32_as_h2(s0.z));
      sv[0][NG - 1] = __low2float(u32_as_h2(s0.w)); zv[0][NG - 1] = __high2float(u32_as_h2(s0.w));
      sk[1][0] = __low2float(u32_as_h2(s1.x)); zk[1][0] = __high2float(u32_as_h2(s1.x));
      sk[1][NG - 1] = __low2float(u32_as_h2(s1.y)); zk[1][NG - 1] = __high2float(u32_as_h2(s1.y));
      sv[1][0] = __low2float(u32_as_h2(s1.z)); zv[1][0] = __high2float(u32_as_h2(s1.z));
      sv[1][NG - 1] = __low2float(u32_as_h2(s1.w)); zv[1][NG - 1] = __high2float(u32_as_h2(s1.w));
    }
    // token r+8 sits in the score rows with the codes' row factor 4; in PV it
    // is in the upper k half, whose codes arrive as 3 - c: its weight enters
    // negated and its zero point becomes z + 3 s, so that
    //   w (s c + z) = (-w s)(3 - c) + w (z + 3 s)
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
      sk[1][grp] *= 0.25f;
      zv[1][grp] = fmaf(3.0f, sv[1][grp], zv[1][grp]);
      sv[1][grp] = -sv[1][grp];
    }

    // ---- QK: scores[token][column] on the tensor cores ----
    // two independent accumulator chains: the two groups (group 64) or the
    // even / odd k-steps (group 128)
    float sacc[2][NT][4];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u) sacc[ch][nt][u] = 0.f;
    {
      const uint32_t kw[4] = {kq4.x, kq4.y, kq4.z, kq4.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t fr[8];
        unpack_word<false>(kw[w], fr);
#pragma unroll
        for (int sh = 0; sh < 2; ++sh) {
          const int s = 2 * w + sh;
          const int ch = (GS == 64) ? (s >> 2) : (s & 1);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_f16(sacc[ch][nt], fr[2 * sh], fr[2 * sh + 1], fr[4 + 2 * sh], fr[5 + 2 * sh],
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
        float d0, d1;
        if (GS == 64) {
          d0 = sacc[grp][nt][0] + sacc[grp][nt][1];
          d1 = sacc[grp][nt][2] + sacc[grp][nt][3];
        } else {
          // chain 1 holds the odd steps, whose codes carry the factor 16
          d0 = fmaf(sacc[1][nt][0] + sacc[1][nt][1], 0.0625f, sacc[0][nt][0] + sacc[0][nt][1]);
          d1 = fmaf(sacc[1][nt][2] + sacc[1][nt][3], 0.0625f, sacc[0][nt][2] + sacc[0][nt][3]);
        }
        // q'.(s c + z) = s (q'.c) + z sum(q')
        l0 = fmaf(sk[0][grp], d0, fmaf(zk[0][grp], sumq[nt][grp], l0));
        l1 = fmaf(sk[1][grp], d1, fmaf(zk[1][grp], sumq[nt][grp], l1));
      }
      l0 = v0 ? l0 * sc24 : kNegInf;
      l1 = v1 ? l1 * sc24 : kNegInf;
      // m_run is the exponent reference (>= every score seen so far); it only
      // moves when some score of the warp exceeds its head's reference, so the
      // per-head maximum is formed only then
      if (__any_sync(0xffffffffu, fmaxf(l0, l1) > m_run[nt])) {
        float tmax = fmaxf(l0, l1);
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
        const bool need = tmax > m_run[nt];
        const float mnew = need ? tmax + kSlack : m_run[nt];
        const float alpha = need ? ((m_run[nt] == kNegInf) ? 0.f : exp2_neg(m_run[nt] - mnew)) : 1.f;
        m_run[nt] = mnew;
        base[nt] = (mnew == kNegInf) ? 0.f : mnew;
        l_run[nt] *= alpha;
#pragma unroll
        for (int grp = 0; grp < NG; ++grp) zs[nt][grp] *= alpha;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int u = 0; u < 4; ++u) oacc[i][nt][u] *= alpha;
      }
      const float p0 = exp2_neg(l0 - base[nt]), p1 = exp2_neg(l1 - base[nt]);
      l_run[nt] += p0 + p1;
      // masked tokens have p = 0 and finite (stale or zero) records
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) {
        const float w0 = p0 * sv[0][grp];
        const float w1 = p1 * sv[1][grp];
        zs[nt][grp] = fmaf(p0, zv[0][grp], fmaf(p1, zv[1][grp], zs[nt][grp]));
        bpv[grp][nt][0] = movmatrix_t(split_hi_lo(w0));
        bpv[grp][nt][1] = movmatrix_t(split_hi_lo(w1));
      }
    }

    // ---- PV: value accumulator [channel][column] on the tensor cores ----
    {
      const uint32_t vw[4] = {vq4.x, vq4.y, vq4.z, vq4.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t fr[8];
        unpack_word<true>(vw[w], fr);
#pragma unroll
        for (int sh = 0; sh < 2; ++sh) {
          const int i = 2 * w + sh;
          const int grp = (GS == 64) ? (i >> 2) : 0;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_f16(oacc[i][nt], fr[2 * sh], fr[2 * sh + 1], fr[4 + 2 * sh], fr[5 + 2 * sh],
                    bpv[grp][nt][0], bpv[grp][nt][1]);
        }
      }
    }
  }
  if (!ok) {   // a copy did not arrive in time: wait (bounded) for the ones in flight
    // iteration k had already issued tile k + kStages - 1, so the copies that
    // may be in flight are those of tiles k .. k + kStages - 1
    if (lane == 0) flag_error(a.err, KV_DEVERR_TIMEOUT);
    for (int kk = k; kk < k + kStages && t_begin + warp + NW * kk < t_end; ++kk)
      mbar_wait(wbar + kk % kStages, (kk / kStages) & 1, a.wait_polls);
  }
  if (!mbar_wait(rbar, 0, a.wait_polls)) {
    ok = false;
    if (threadIdx.x == 0) flag_error(a.err, KV_DEVERR_TIMEOUT);
  }
  ok = __syncthreads_and(ok);   // every warp is done with its ring before the results reuse it
  if (lane < kStages) mbar_inval(wbar + lane);
  if (threadIdx.x == 0) mbar_inval(rbar);
  if (!ok) {   // the split's result is skipped
    write_empty_partial<G, NW>(part);
    return;
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
        // channel rows carry the codes' 2^-24, row factor 4 for r+8 and step
        // factor 16 for odd i
        const float u = (i & 1) ? 1048576.0f : 16777216.0f;
        o[16 * i + r] = fmaf(oacc[i][nt][0] + oacc[i][nt][1], u, zz);
        o[16 * i + r + 8] = fmaf(oacc[i][nt][2] + oacc[i][nt][3], u * 0.25f, zz);
      }
      if (r == 0) {
        swm[warp * G + hh] = m_run[nt];
        swl[warp * G + hh] = l;
      }
    }
  }
  __syncthreads();
  // merged sums, transposed for the back-rotation, into q's slot (q and q' are
  // no longer needed); then back to the original basis, into the partial
  merge_warps_t<G, NW>(swo, swm, swl, sq, sm + S::smm, sm + S::sml,
                       reinterpret_cast<float*>(spid));   // page ids no longer needed
  rotate_back_to_part<G, NW>(sq, srv, sm + S::spr, part, sm + S::smm, sm + S::sml);
}

// ---------------------------------------------------------------------------
// BF16 sink + recent tiers of the INT2 pool: tier CTA `ti` stages storage
// rows [ti*kTierRows, ...) of [sink slots | recent ring] before it knows the
// lengths, then attends over the rows that hold live tokens.
// ---------------------------------------------------------------------------
template <int G, int GS, bool kMulti>
__device__ void bf16_tiers(const DecodeArgs& a, int b, int g, int ti, float* sm, float* part) {
  constexpr int NW = int2_warps(G);
  using S = Lay<G, GS, NW, true>;
  const int warp = threadIdx.x >> 5;
  const int scap = a.sink_cap, rcap = a.rec_cap;
  const int r0 = min(scap + rcap, ti * kTierRows), r1 = min(scap + rcap, r0 + kTierRows);
  const size_t seq_head = (size_t)b * a.Hkv + g;
  const uint16_t* sk = a.sink_k + seq_head * scap * 128;
  const uint16_t* sv = a.sink_v + seq_head * scap * 128;
  const uint16_t* rk = a.rec_k + seq_head * rcap * 128;
  const uint16_t* rv = a.rec_v + seq_head * rcap * 128;
  uint8_t* stk = reinterpret_cast<uint8_t*>(sm + S::stage);
  uint8_t* stv = stk + (size_t)kTierRows * kTierRowK;
  for (int i = threadIdx.x; i < (r1 - r0) * 32; i += NW * 32) {
    const int t = i >> 5, c = i & 31, key = c < 16, ch = c & 15, row = r0 + t;
    const uint16_t* src = (row < scap) ? (key ? sk : sv) + (size_t)row * 128
                                       : (key ? rk : rv) + (size_t)(row - scap) * 128;
    uint8_t* dst = key ? stk + t * kTierRowK + 16 * ch : stv + t * kTierRowV + 16 * ch;
    cp_async16(dst, reinterpret_cast<const uint8_t*>(src) + 16 * ch);
  }
  cp_async_commit();
  float* sq = sm + S::sq;
  load_q<G, NW, kMulti>(a, b, g, sq, G);
  int ns = __ldg(a.sink_len + b), nr = __ldg(a.rec_len + b), rs = __ldg(a.rec_start + b);
  cp_async_wait<0>();
  __syncthreads();
  if (ns < 0 || ns > scap || nr < 0 || nr > rcap || rs < 0 || rs >= rcap) {
    if (threadIdx.x == 0) flag_error(a.err, KV_DEVERR_LENGTH);
    ns = max(0, min(ns, scap));
    nr = max(0, min(nr, rcap));
    rs = max(0, min(rs, rcap - 1));
  }
  auto rows = [&](int u, const uint16_t*& kr, const uint16_t*& vr) -> bool {
    bool live;
    if (u < scap) {
      live = u < ns;
    } else {
      int d = (u - scap) - rs;
      d += (d < 0) ? rcap : 0;
      live = d < nr;
    }
    kr = reinterpret_cast<const uint16_t*>(stk + (u - r0) * kTierRowK);
    vr = reinterpret_cast<const uint16_t*>(stv + (u - r0) * kTierRowV);
    return live;
  };
  WarpAcc<G> st;
  st.init();
  bf16_rows_attend<G, true>(sq, sm + S::sp + warp * 32 * G, r0 + 32 * warp, r1, 32 * NW, rows,
                            a.scale_log2, st);
  __syncthreads();   // staged rows are dead before the results reuse the region
  warp_acc_to_smem<G>(st, sm + S::swo, sm + S::swm, sm + S::swl);
  __syncthreads();
  merge_warps<G, NW>(sm + S::swo, sm + S::swm, sm + S::swl, sm + S::sqr, sm + S::smm, sm + S::sml);
  write_partial<G, NW>(part, sm + S::sqr, sm + S::smm, sm + S::sml);
}

template <int G, int GS, bool kMulti>
__global__ void __launch_bounds__(int2_warps(G) * 32, 1) decode_int2_kernel(DecodeArgs a) {
  constexpr int NW = int2_warps(G);
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  // launch order: every history split first ((sequence, KV head) pairs in
  // turn, their splits together), then every tier CTA, so that on a grid of
  // several waves the short tier CTAs fill the last wave
  const int nparts = a.n_split + a.n_tier;
  const int lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  const int n_hist = a.n_split * gridDim.y * gridDim.z;
  int split, pair;
  if (lin < n_hist) {
    split = lin % a.n_split;
    pair = lin / a.n_split;
  } else {
    split = a.n_split + (lin - n_hist) % a.n_tier;
    pair = (lin - n_hist) / a.n_tier;
  }
  const int g = pair % a.Hkv, b = pair / a.Hkv;
  float* part = a.ws + ((size_t)(b * a.Hkv + g) * nparts + split) * G * kPart;
  if (split < a.n_split)
    int2_history<G, GS, kMulti>(a, b, g, split, sm, part);
  else
    bf16_tiers<G, GS, kMulti>(a, b, g, split - a.n_split, sm, part);
  if (last_to_arrive(a.tickets + b * a.Hkv + g, (unsigned)nparts))
    merge_parts<G, NW, kMulti>(a, b, g, nparts, sm);
}

// ---------------------------------------------------------------------------
// All-BF16 paged decode (the baseline)
// ---------------------------------------------------------------------------
// Log-sum-exp merge of the BF16 decode's parts (all in the original basis) and
// the final normalisation: part weights in shared memory, then every warp
// accumulates a subset of the parts for one head and the subsets are summed.
template <int G, int NW>
__device__ void final_combine_plain(const DecodeArgs& a, int b, int g, int nparts, float* sm) {
  constexpr int NSUB = NW / G;                     // part subsets per output column quad
  const float* base = a.ws + (size_t)(b * a.Hkv + g) * nparts * G * kPart;
  float* sM = sm;                                  // [8]
  float* sL = sm + 8;                              // [8]
  float* sacc = sm + 16;                           // [NSUB][G][128]
  float* sf = sacc + NSUB * G * 128;               // [nparts * G] m, then weights
  float* sl = sf + nparts * G;                     // [nparts * G]
  for (int i = threadIdx.x; i < nparts * G; i += NW * 32) {
    sf[i] = __ldcg(base + (size_t)i * kPart);
    sl[i] = __ldcg(base + (size_t)i * kPart + 1);
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float M = kNegInf;
    for (int s = 0; s < nparts; ++s) M = fmaxf(M, sf[s * G + threadIdx.x]);
    sM[threadIdx.x] = M;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nparts * G; i += NW * 32) {
    const float m = sf[i], M = sM[i % G];
    sf[i] = (m == kNegInf || M == kNegInf) ? 0.f : exp2f(m - M);
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float L = 0.f;
    for (int s = 0; s < nparts; ++s) L = fmaf(sf[s * G + threadIdx.x], sl[s * G + threadIdx.x], L);
    sL[threadIdx.x] = L;
  }
  {
    const int cq = threadIdx.x & 31, h = (threadIdx.x >> 5) % G, sub = (threadIdx.x >> 5) / G;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int s = sub; s < nparts; s += NSUB) {
      const float f = sf[s * G + h];
      const float4 o =
          __ldcg(reinterpret_cast<const float4*>(base + (size_t)(s * G + h) * kPart + 4) + cq);
      acc.x = fmaf(f, o.x, acc.x);
      acc.y = fmaf(f, o.y, acc.y);
      acc.z = fmaf(f, o.z, acc.z);
      acc.w = fmaf(f, o.w, acc.w);
    }
    *reinterpret_cast<float4*>(sacc + (sub * G + h) * 128 + 4 * cq) = acc;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * 128; idx += NW * 32) {
    const int h = idx >> 7;
    float O = 0.f;
#pragma unroll
    for (int u = 0; u < NSUB; ++u) O += sacc[u * G * 128 + idx];
    const float L = sL[h];
    a.out[((size_t)b * a.Hq + g * G + h) * 128 + (idx & 127)] = (L > 0.f) ? O / L : 0.f;
  }
  if (threadIdx.x == 0) a.tickets[b * a.Hkv + g] = 0u;   // ready for the next call
}

template <int G>
__global__ void __launch_bounds__(kBf16Warps * 32, 2) decode_bf16_kernel(DecodeArgs a) {
  constexpr int NW = kBf16Warps;
  using S = Lay<G, 128, NW, false>;
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int nparts = a.n_split;
  float* part = a.ws + ((size_t)(b * a.Hkv + g) * nparts + split) * G * kPart;
  int n = a.seq_len[b];
  const int cap = min(a.max_pages * a.page_size, a.max_len);
  if (n < 0 || n > cap) {
    if (threadIdx.x == 0) flag_error(a.err, KV_DEVERR_LENGTH);
    n = max(0, min(n, cap));
  }
  const int u0 = split * a.per_split, u1 = min(n, u0 + a.per_split);
  if (u0 >= u1) {
    write_empty_partial<G, NW>(part);
  } else {
    const int P = a.page_size;
    const int p_begin = u0 / P, p_count = (u1 - 1) / P + 1 - p_begin;
    int* spid = reinterpret_cast<int*>(sm + S::spid);
    const int32_t* ptrow = a.pt + (size_t)b * a.max_pages;
    for (int i = threadIdx.x; i < p_count; i += NW * 32) spid[i] = __ldg(ptrow + p_begin + i);
    float* sq = sm + S::sq;
    load_q<G, NW>(a, b, g, sq, G);
    __syncthreads();   // publishes q and the page ids
    auto rows = [&](int u, const uint16_t*& kr, const uint16_t*& vr) -> bool {
      const int pid = spid[u / P - p_begin];
      if (pid < 0 || pid >= a.num_pages) {
        flag_error(a.err, KV_DEVERR_PAGE_ID);
        return false;
      }
      const size_t off = (((size_t)pid * a.Hkv + g) * P + (u % P)) * 128;
      kr = a.bk + off;
      vr = a.bv + off;
      return true;
    };
    WarpAcc<G> st;
    st.init();
    bf16_rows_attend<G, false>(sq, sm + S::sp + warp * 32 * G, u0 + 32 * warp, u1, 32 * NW, rows,
                               a.scale_log2, st);
    warp_acc_to_smem<G>(st, sm + S::swo, sm + S::swm, sm + S::swl);
    __syncthreads();
    merge_warps<G, NW>(sm + S::swo, sm + S::swm, sm + S::swl, sm + S::sqr, sm + S::smm, sm + S::sml);
    write_partial<G, NW>(part, sm + S::sqr, sm + S::smm, sm + S::sml);
  }
  if (last_to_arrive(a.tickets + b * a.Hkv + g, (unsigned)nparts))
    final_combine_plain<G, NW>(a, b, g, nparts, sm);
}

// Sets the dynamic shared-memory limit of a kernel (once) and reports how many
// of its CTAs fit on one SM (-1 on a CUDA error).
template <class K>
int prepare_kernel(K kernel, int threads, size_t smem, bool& done, int& per_sm) {
  if (!done) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return -1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess)
      return -1;
    per_sm = n > 0 ? n : 1;
    done = true;
  }
  return per_sm;
}

template <int G, int GS>
constexpr size_t int2_smem() {
  return sizeof(float) * Lay<G, GS, int2_warps(G), true>::total;
}
template <int G>
constexpr size_t bf16_smem() {
  return sizeof(float) * Lay<G, 128, kBf16Warps, false>::total;
}

template <int G, int GS, bool kMulti>
int int2_blocks_per_sm() {
  static bool done = false;
  static int per_sm = 1;
  return prepare_kernel(decode_int2_kernel<G, GS, kMulti>, int2_warps(G) * 32, int2_smem<G, GS>(), done,
                        per_sm);
}

template <int G>
int bf16_blocks_per_sm() {
  static bool done = false;
  static int per_sm = 1;
  return prepare_kernel(decode_bf16_kernel<G>, kBf16Warps * 32, bf16_smem<G>(), done, per_sm);
}

template <int G, int GS, bool kMulti>
cudaError_t launch_int2_t(const DecodeArgs& a, int B, cudaStream_t s) {
  if (int2_blocks_per_sm<G, GS, kMulti>() < 0) return cudaErrorInvalidConfiguration;
  dim3 grid(a.n_split + a.n_tier, a.Hkv, B);
  decode_int2_kernel<G, GS, kMulti><<<grid, int2_warps(G) * 32, int2_smem<G, GS>(), s>>>(a);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_bf16_t(const DecodeArgs& a, int B, cudaStream_t s) {
  if (bf16_blocks_per_sm<G>() < 0) return cudaErrorInvalidConfiguration;
  dim3 grid(a.n_split, a.Hkv, B);
  decode_bf16_kernel<G><<<grid, kBf16Warps * 32, bf16_smem<G>(), s>>>(a);
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
  a.T = 1;
  a.Gq = p.G;
  a.lse = nullptr;
  a.wait_polls = p.test_wait_polls > 0 ? p.test_wait_polls : kWaitPolls;
  a.stall_first_copy = p.test_stall_first_copy;
  return a;
}

template <bool kMulti>
int int2_occupancy_t(const Pool& p, int G) {
  const bool g64 = p.cfg.group_size == 64;
  switch (G) {
    case 1: return g64 ? int2_blocks_per_sm<1, 64, kMulti>() : int2_blocks_per_sm<1, 128, kMulti>();
    case 2: return g64 ? int2_blocks_per_sm<2, 64, kMulti>() : int2_blocks_per_sm<2, 128, kMulti>();
    case 4: return g64 ? int2_blocks_per_sm<4, 64, kMulti>() : int2_blocks_per_sm<4, 128, kMulti>();
    default: return g64 ? int2_blocks_per_sm<8, 64, kMulti>() : int2_blocks_per_sm<8, 128, kMulti>();
  }
}

int bf16_occupancy(const Pool& p) {
  switch (p.G) {
    case 1: return bf16_blocks_per_sm<1>();
    case 2: return bf16_blocks_per_sm<2>();
    case 4: return bf16_blocks_per_sm<4>();
    default: return bf16_blocks_per_sm<8>();
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// fixed scratch for kv_decode_attention_noalloc
// ---------------------------------------------------------------------------
// Partials of the split-K decode for callers that cannot allocate device
// memory.  Lives for the whole process on every device that loads this code.
// Host code only sees a stand-in for this name: its device address comes from
// cudaGetSymbolAddress below and is what the kernel receives.
static __device__ __align__(256) float g_noalloc_scratch[KV_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {
constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::atomic<int> g_scratch_state[kMaxDevices];   // 0 = unset, 1 = in progress, 2 = ready
}  // namespace

cudaError_t noalloc_scratch(void** ptr, size_t* bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (g_scratch_state[dev].load(std::memory_order_acquire) != 2) {
    int expected = 0;
    if (g_scratch_state[dev].compare_exchange_strong(expected, 1)) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);   // with `dev` current
      if (e != cudaSuccess) {
        g_scratch_state[dev].store(0, std::memory_order_release);
        return e;
      }
      g_scratch_ptr[dev] = p;
      g_scratch_state[dev].store(2, std::memory_order_release);
    } else {
      while (g_scratch_state[dev].load(std::memory_order_acquire) == 1) {
      }
      if (g_scratch_state[dev].load(std::memory_order_acquire) != 2) return cudaErrorNotReady;
    }
  }
  *ptr = g_scratch_ptr[dev];
  *bytes = KV_NOALLOC_SCRATCH_BYTES;
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// planning and launch
// ---------------------------------------------------------------------------

// Splits per (sequence, KV head): fill exactly one wave of resident CTAs when
// the batch is small; cap the work of one split (and the number of parts the
// final merge reads) when it is large.
static DecodePlan make_plan(const Pool& p, int G, int B, int units, int max_per, int n_extra,
                            int per_sm) {
  DecodePlan pl;
  const int pairs = B * p.cfg.num_kv_heads;
  const int slots = max(1, per_sm) * p.sm_count;
  const int u = max(units, 1);
  int ns = slots / pairs - n_extra;
  ns = max(1, min(ns, u));
  int per = (u + ns - 1) / ns;
  per = min(per, max_per);
  per = max(per, (u + kMaxParts - n_extra - 1) / (kMaxParts - n_extra));
  ns = (u + per - 1) / per;
  pl.n_split = ns;
  pl.n_tier = n_extra;
  pl.tiles_per_split = per;
  pl.max_len = 0;
  pl.partial_floats = (size_t)pairs * (ns + n_extra) * G * kPart;
  pl.bytes = pl.partial_floats * sizeof(float);
  return pl;
}

DecodePlan plan_decode_int2(const Pool& p, int B, int max_hist_len, int T) {
  const int G = T * p.G;   // query columns per KV head
  const int tiles = (max(max_hist_len, 0) + kTile - 1) / kTile;
  const int n_tier = max(1, (p.cfg.sink_tokens + p.cfg.recent_tokens + kTierRows - 1) / kTierRows);
  const int per_sm = (T > 1) ? int2_occupancy_t<true>(p, G) : int2_occupancy_t<false>(p, G);
  DecodePlan pl = make_plan(p, G, B, tiles, 64 * int2_warps(G), n_tier, per_sm);
  pl.max_len = max(max_hist_len, 0);
  return pl;
}

DecodePlan plan_decode_bf16(const Pool& p, int B, int max_len) {
  DecodePlan pl = make_plan(p, p.G, B, max(max_len, 0), 8192, 0, bf16_occupancy(p));
  pl.max_len = max(max_len, 0);
  return pl;
}

cudaError_t launch_decode_int2(const Pool& p, int layer, int B, const void* q,
                               const int32_t* sink_len, const int32_t* hist_len,
                               const int32_t* rec_len, const int32_t* rec_start,
                               const int32_t* pt, int max_pages, const DecodePlan& plan,
                               float scale, float* out, void* ws, cudaStream_t s, int T,
                               float* lse) {
  DecodeArgs a = base_args(p, layer, q, pt, max_pages, scale, out, ws);
  a.T = T;
  a.lse = lse;
  a.hist = p.hist + (size_t)layer * p.hist_layer_stride;
  a.page_bytes = p.page_bytes;
  a.tile_bytes = (int)p.tile_bytes;
  a.tiles_per_page = p.cfg.page_size / kTile;
  a.tpp_shift = (a.tiles_per_page == 2) ? 1 : 0;
  a.sink_k = p.sink_k + (size_t)layer * p.sink_layer_stride;
  a.sink_v = p.sink_v + (size_t)layer * p.sink_layer_stride;
  a.rec_k = p.rec_k + (size_t)layer * p.rec_layer_stride;
  a.rec_v = p.rec_v + (size_t)layer * p.rec_layer_stride;
  a.sink_cap = p.cfg.sink_tokens;
  a.rec_cap = p.cfg.recent_tokens;
  a.RvT = p.RvT + (size_t)layer * p.cfg.num_kv_heads * 128 * 128;
  a.rfrag = p.rfrag + (size_t)layer * p.cfg.num_kv_heads * kFragBlocks * rfrag_per_head();
  a.sink_len = sink_len;
  a.hist_len = hist_len;
  a.rec_len = rec_len;
  a.rec_start = rec_start;
  a.n_split = plan.n_split;
  a.per_split = plan.tiles_per_split;
  a.n_tier = plan.n_tier;
  a.max_len = plan.max_len;
  const bool g64 = p.cfg.group_size == 64;
  if (T > 1 || lse) {   // several queries per sequence, or the log-sum-exp wanted
    switch (T * p.G) {
      case 1: return g64 ? launch_int2_t<1, 64, true>(a, B, s) : launch_int2_t<1, 128, true>(a, B, s);
      case 2: return g64 ? launch_int2_t<2, 64, true>(a, B, s) : launch_int2_t<2, 128, true>(a, B, s);
      case 4: return g64 ? launch_int2_t<4, 64, true>(a, B, s) : launch_int2_t<4, 128, true>(a, B, s);
      case 8: return g64 ? launch_int2_t<8, 64, true>(a, B, s) : launch_int2_t<8, 128, true>(a, B, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (p.G) {
    case 1: return g64 ? launch_int2_t<1, 64, false>(a, B, s) : launch_int2_t<1, 128, false>(a, B, s);
    case 2: return g64 ? launch_int2_t<2, 64, false>(a, B, s) : launch_int2_t<2, 128, false>(a, B, s);
    case 4: return g64 ? launch_int2_t<4, 64, false>(a, B, s) : launch_int2_t<4, 128, false>(a, B, s);
    case 8: return g64 ? launch_int2_t<8, 64, false>(a, B, s) : launch_int2_t<8, 128, false>(a, B, s);
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
  a.n_tier = 0;
  a.max_len = plan.max_len;
  switch (p.G) {
    case 1: return launch_bf16_t<1>(a, B, s);
    case 2: return launch_bf16_t<2>(a, B, s);
    case 4: return launch_bf16_t<4>(a, B, s);
    case 8: return launch_bf16_t<8>(a, B, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvint2
