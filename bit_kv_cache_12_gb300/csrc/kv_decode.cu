// Decode attention over the three-tier INT2 pool and over an all-BF16 pool.
//
// Method: gist.science explainer "OSCAR: Offline Spectral Covariance-Aware
// Rotation for 2-bit KV Cache Quantization", section 2.2 B: one fused kernel
// unpacks and dequantizes the INT2 history, applies the inverse rotation and
// computes attention, next to the BF16 sink and recent tiers (yunpan.plus
// OSCAR write-up, "1. 三段式 Token 池": 64 sink + INT2 history + 256 recent).
//
// GPU design (two launches per decode step):
//   * a small pre-pass computes q' = q R_k once per (sequence, KV head) on the
//     tensor cores and writes it as the MMA fragments the history warps use;
//     the decode kernel is its programmatic dependent, so it launches at once
//     and its history CTAs wait for q' only after their first tile copies are
//     in flight.
//   * decode grid = (history splits + 1 tier CTA, KV heads, sequences); 16
//     warps per CTA and one CTA per SM for GQA <= 4 (12 warps for GQA 8), and
//     the split count fills one wave when the batch is small.  Every history
//     split is launched before every tier CTA.
//   * history CTAs: each warp streams 16-token tiles from HBM through a
//     4-stage shared-memory ring, one bulk copy per tile completing on the
//     stage's mbarrier (bounded waits).  The 2-bit codes become fp16 MMA
//     fragments by masking alone (exact subnormals, one logic op per code
//     pair) and QK and PV run on the tensor cores (mma.sync m16n8k16).
//     Dequantization is folded:
//       q'.deq(k) = s_k (q'.c_k) + z_k sum(q')
//       sum_t w_t deq(v_t) = sum_t (w_t s_v) c_v + sum_t w_t z_v
//     so the MMA operands are exact small integers times powers of two and the
//     query / softmax weights enter as fp16 hi + lo pairs.  Against subnormal
//     code operands the tensor cores keep only the upper bits of the lo
//     products (about 16 significant bits overall; measured output error
//     about 2e-5 relative to the fp64 oracle at 100k tokens).  Online softmax
//     per head with warp-shuffle max and a lazily moved exponent reference;
//     each warp puts its result in shared memory as its loop ends, the warps
//     merge there and the split writes its partial (m, l, o') in the rotated
//     basis, then sets its bit in the pair's arrival mask (release).
//   * tier CTA: stages the BF16 sink + recent storage into shared memory
//     before the lengths are known, attends the live rows on the tensor cores
//     (bf16 MMA, the softmax weights as bf16 hi + lo), then
//     merges the history partials in split order as they arrive (acquire),
//     rotates the merged history value sum back by R_v^T once and combines it
//     with its own result into the fp32 output (and, for several queries per
//     sequence, the log-sum-exp).
#include <math.h>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <type_traits>

#include "kv_device.cuh"
#include "kv_internal.h"

namespace kvint2 {

namespace {

constexpr int kPart = 132;       // floats per (part, head) partial: m, l, -, -, o[128]
constexpr float kNegInf = -INFINITY;
constexpr int kStages = 4;       // tiles in each warp's ring
constexpr int kWaitPolls = 1 << 20;   // bounded mbarrier polls before a copy counts as lost
constexpr int kMergePolls = 1 << 21;  // bounded polls of a tier CTA for its history splits
constexpr int kMaxParts = 400;   // partials per (sequence, KV head) a merge reads
constexpr int kMaxTilesPerWarp = 128;   // longest INT2 history split, in tiles per warp
constexpr int kMaxPids = 16 * kMaxTilesPerWarp + 8;   // page ids staged per CTA
constexpr int kTierRows = 320;   // sink + recent storage rows staged per tier CTA
constexpr int kTierRowK = 272;   // staged K row stride (bytes): 256 + 16 keeps lane reads conflict-free
constexpr int kTierRowV = 272;   // staged V row stride: the transposed ldmatrix reads are conflict-free too
// q rows staged for rotate_q: channel c of row h at h * kQStride + c + 4 (c / 32),
// so that the rotation's float4 reads (row r, channels 32 j + 4 s ..) spread over
// all banks; q' rows are kQrStride apart for the same reason in the fragment build.
constexpr int kQStride = 168;
constexpr int kQrStride = 136;
// The history loop keeps each head's exponent reference kSlack (log2 units)
// above the largest score seen when it was last moved, so weights stay <= 1
// and the accumulators are rescaled only when a score passes the reference.
constexpr float kSlack = 4.0f;
constexpr int kBf16Warps = 8;

__host__ __device__ constexpr int int2_warps(int G) { return G <= 4 ? 16 : 12; }
// Longest history split, in tiles per warp, of a grid: grids of several waves
// run fewer CTAs (fewer prologues and ramps) with longer splits; measured on
// the batched workloads, 128 suits up to 4 query columns per KV head (batch 64:
// 244 -> 229 us against 64) and 96 suits 8 (16 x 131k: 472 -> 453 us; 128 gave
// 471).  A split's page ids (one per tile at page 16) are staged in shared memory.
__host__ __device__ constexpr int int2_max_tiles_per_warp(int G) { return G <= 4 ? 128 : 96; }
static_assert((long long)kMaxParts * (kMaxPids - 8) * kTile >= kMaxDecodeLen,
              "a decode of the longest length stages at most kMaxPids - 8 page ids per split");
static_assert(int2_max_tiles_per_warp(1) * int2_warps(1) <= kMaxPids &&
                  int2_max_tiles_per_warp(8) * int2_warps(8) <= kMaxPids &&
                  int2_max_tiles_per_warp(1) <= kMaxTilesPerWarp && int2_max_tiles_per_warp(8) <= kMaxTilesPerWarp,
              "a split's page ids must fit the staging array");
static_assert(kMaxParts <= 32 * kMaskWords, "every split has a bit in the arrival mask");
// Where a history CTA gets q' = q R_k from:
//   kQLocal  it forms q' itself, each warp from its own 4 KB of R_k's
//            fragments held in registers - grids of one wave;
//   kQPre    the batched pre-pass wrote the fragments - grids of several waves.
constexpr int kQLocal = 0, kQPre = 1;

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
  float* ws;                // history partials, then (INT2) the q' fragments
  uint32_t* qfrag;          // INT2: [B][Hkv][32 lanes][qfrag_words] q' fragments in ws
  unsigned* tickets;        // BF16: split-merge counters
  unsigned* arrive;         // INT2: [max_seqs][Hkv][kMaskWords] arrival masks of the splits
  int merge_polls;          // INT2: bounded polls of a tier CTA for its history splits
  int qmode;                // INT2: where a history CTA gets q' from (kQLocal or kQPre)
  int* err;
};

// ---------------------------------------------------------------------------
// shared helpers
// ---------------------------------------------------------------------------

// R_k's MMA fragments held in registers (the q' pre-pass and the history CTAs
// that form q' themselves): warp w of NW produces q' columns 8w.., 8(w + NW)..,
// and each lane loads all its fragments at once (one memory latency).
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
// fp32 holding bf16 values, rows kQStride apart with 4 floats of padding after
// every 32 channels) into Y (rows kQrStride apart), on the tensor cores: R_k
// comes as fp16 hi + lo B fragments (rotation fragment block 0, this warp's in
// registers), q is scaled by 2^-8 (exact) and split into fp16 hi + lo, which
// enter as separate MMA rows (hi in rows 0..7, lo in rows 8..15, or hi in
// rows 0..3 and lo in rows 4..7 for up to 4 rows), so that two products per
// k-step (rows x R_hi, rows x R_lo) give the three terms above 2^-22
// relative, accumulated in fp32 in two chains (even and odd k-steps).  Warp w
// produces columns 8w.., 8(w + NW)...  With kSums, each 8-column n-tile's
// partial row sums go to P[n-tile][row] (for the per-group sums of q').
// Ends with a barrier.
template <int NROWS, int NW, bool kSums = false>
__device__ void rotate_q(const float* X, const RotFrags<NW>& rkf, float* Y, float* P = nullptr,
                         uint32_t* SA = nullptr) {
  static_assert(NROWS <= 8, "rows");
  constexpr int NTW = (16 + NW - 1) / NW;
  constexpr bool kSplitRows = NROWS <= 4;   // hi rows 0..3, lo rows 4..7 (else 0..7 / 8..15)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, j = lane & 3;
  float acc[NTW][4][4];   // [n-tile][R_hi even, R_hi odd, R_lo even, R_lo odd][fragment]
#pragma unroll
  for (int u = 0; u < NTW; ++u)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[u][c][0] = acc[u][c][1] = acc[u][c][2] = acc[u][c][3] = 0.f;
  const int xrow = kSplitRows ? (r & 3) : r;
  const bool row_ok = xrow < NROWS;
  const bool lo_lane = kSplitRows && r >= 4;   // this lane's row holds the lo terms
  constexpr float kIn = 1.0f / 256.0f;
  // the A fragments of k-step s (the same in every warp)
  auto afrag = [&](int s, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
    // A: row r, k index kappa -> input channel 32*(kappa%8/2) + 4s + 2*(kappa/8) + kappa%2
    float4 x = row_ok ? *reinterpret_cast<const float4*>(X + xrow * kQStride + 36 * j + 4 * s)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    x.x *= kIn; x.y *= kIn; x.z *= kIn; x.w *= kIn;
    const __half2 h01 = __floats2half2_rn(x.x, x.y), h23 = __floats2half2_rn(x.z, x.w);
    const __half2 l01 = __floats2half2_rn(x.x - __low2float(h01), x.y - __high2float(h01));
    const __half2 l23 = __floats2half2_rn(x.z - __low2float(h23), x.w - __high2float(h23));
    if (kSplitRows) {
      a0 = lo_lane ? h2_as_u32(l01) : h2_as_u32(h01);
      a2 = lo_lane ? h2_as_u32(l23) : h2_as_u32(h23);
      a1 = a3 = 0u;
    } else {
      a0 = h2_as_u32(h01); a2 = h2_as_u32(h23);
      a1 = h2_as_u32(l01); a3 = h2_as_u32(l23);
    }
  };
  // with SA (8 k-steps x 32 lanes x 4 words of shared memory), warp w < 8
  // builds k-step w for every lane and the others load them
  if (SA) {
    if (warp < 8) {
      uint32_t a0, a1, a2, a3;
      afrag(warp, a0, a1, a2, a3);
      *reinterpret_cast<uint4*>(SA + (warp * 32 + lane) * 4) = make_uint4(a0, a1, a2, a3);
    }
    __syncthreads();
  }
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    uint32_t a0, a1, a2, a3;
    if (SA) {
      const uint4 w = *reinterpret_cast<const uint4*>(SA + (s * 32 + lane) * 4);
      a0 = w.x; a1 = w.y; a2 = w.z; a3 = w.w;
    } else {
      afrag(s, a0, a1, a2, a3);
    }
#pragma unroll
    for (int u = 0; u < NTW; ++u) {
      const uint4 f = rkf.f[s][u];   // zero past the 16 n-tiles
      mma_f16(acc[u][s & 1], a0, a1, a2, a3, f.x, f.y);         // rows x R_hi
      mma_f16(acc[u][2 + (s & 1)], a0, a1, a2, a3, f.z, f.w);   // rows x R_lo
    }
  }
#pragma unroll
  for (int u = 0; u < NTW; ++u) {
    const int nt = warp + u * NW;
    // hi.R_hi + hi.R_lo + lo.R_hi for this lane's hi row
    float y[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float hh = acc[u][0][e] + acc[u][1][e], hl = acc[u][2][e] + acc[u][3][e];
      float lh;
      if (kSplitRows) lh = __shfl_xor_sync(0xffffffffu, hh, 16);   // row r + 4: lo x R_hi
      else lh = acc[u][0][2 + e] + acc[u][1][2 + e];                // row r + 8: lo x R_hi
      y[e] = (hh + hl) + lh;
    }
    const bool out_row = row_ok && !lo_lane && nt < 16;
    if (out_row)
      *reinterpret_cast<float2*>(Y + xrow * kQrStride + 8 * nt + 2 * j) = make_float2(y[0] * 256.0f, y[1] * 256.0f);
    if constexpr (kSums) {   // this n-tile's 8 columns of row xrow, summed over the 4 lanes of the row
      float part = (y[0] + y[1]) * 256.0f;
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      if (out_row && j == 0) P[nt * 8 + xrow] = part;
    }
  }
  __syncthreads();
}

// Merge the NW warps' (m, l, o) in shared memory into one partial per head.
// merged[h][c] receives o; sm_m / sm_l receive m and l.
template <int G, int NW, int WS>
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
        O = fmaf(f, swo[(w * G + h) * WS + (idx & 127)], O);
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

// Partials merged per round of loads.
constexpr int kMergeBatch = 20;

// ---------------------------------------------------------------------------
// shared helpers: the zero tile, ldmatrix
// ---------------------------------------------------------------------------
// A zero INT2 tile (largest tile size): copied in place of a tile behind an
// invalid page id, so every ring slot always holds finite data.
__device__ __align__(16) uint8_t g_zero_tile[1280];

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// one 2D TMA box (x = channel, y = row) of `map` into shared memory, completing on `bar`
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// (hi, lo) bf16 split of an fp32 weight as one bf16x2 register: low half
// bf16(x), high half bf16(x - bf16(x))
__device__ __forceinline__ uint32_t split_hi_lo_bf16(float x) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
  return (uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(lo) << 16);
}

// q of the GQA group (bf16 -> fp32) into shared memory; padded heads are 0.
// No barrier.
template <int G, int NW, bool kMulti = false, bool kPad = false>
__device__ void load_q(const DecodeArgs& a, int b, int g, float* sq, int padded_heads) {
  for (int idx = threadIdx.x; idx < padded_heads * 128; idx += NW * 32) {
    const int h = idx >> 7, c = idx & 127;
    float v = 0.f;
    if (h < G) {
      const size_t row = kMulti ? ((size_t)b * a.T + h / a.Gq) * a.Hq + g * a.Gq + h % a.Gq
                                : (size_t)b * a.Hq + g * G + h;
      v = __uint_as_float((uint32_t)a.q[row * 128 + c] << 16);
    }
    sq[kPad ? h * kQStride + c + 4 * (c >> 5) : idx] = v;
  }
}

// ---------------------------------------------------------------------------
// INT2 decode, step 1: q' = q R_k once per (sequence, KV head)
// ---------------------------------------------------------------------------
// 32-bit words per (sequence, KV head) and lane of a history warp: the QK B
// fragments qf[8 steps][NT][2] (fp16 hi / lo of q'), then the per-group sums
// of q' in the units of the score accumulator (NT * NG <= 4 words).
template <int G>
__host__ __device__ constexpr int qfrag_words() { return 16 * ((G <= 4) ? 1 : 2) + 4; }

// q' = q R_k for every (sequence, KV head) of the batch on the tensor cores:
// q (scaled by 2^-8, exact) split into fp16 hi + lo, R_k as fp16 hi + lo
// fragments (rotation fragment block 0), the three products above 2^-22
// relative accumulated in fp32.  A CTA of eight warps takes one KV head and
// 16 / HP sequences (one 16-row MMA tile of (sequence, head) rows) and writes
// every history warp's fragments of q' and the per-group sums.  It lets the
// decode kernel launch at once (programmatic dependent launch); the decode's
// history CTAs wait for it only when they need q'.
template <int G, int GS, bool kMulti>
__global__ void __launch_bounds__(256) qprep_kernel(DecodeArgs a, int B) {
  constexpr int HP = (G <= 4) ? 4 : 8;   // MMA columns of a KV head (4 heads x hi / lo)
  constexpr int NT = HP / 4;
  constexpr int NG = 128 / GS;
  constexpr int SPB = 16 / HP;           // sequences per CTA
  constexpr int QW = qfrag_words<G>();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ __align__(16) float X[16 * 128];
  __shared__ __align__(16) float Y[16 * 128];
  __shared__ float ssum[16 * 2];
  const int g = blockIdx.x, b0 = blockIdx.y * SPB;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  RotFrags<8> rk;
  rk.load(a.rfrag + (size_t)g * kFragBlocks * 4096);
  for (int idx = threadIdx.x; idx < 16 * 128; idx += 256) {   // row = sequence * HP + head
    const int row = idx >> 7, c = idx & 127, sl = row / HP, hh = row % HP, b = b0 + sl;
    float v = 0.f;
    if (hh < G && b < B) {
      const size_t qrow = kMulti ? ((size_t)b * a.T + hh / a.Gq) * a.Hq + g * a.Gq + hh % a.Gq
                                 : (size_t)b * a.Hq + g * G + hh;
      v = __uint_as_float((uint32_t)a.q[qrow * 128 + c] << 16);
    }
    X[idx] = v;
  }
  __syncthreads();
  {   // rows r and r + 8 of the A fragment; warp w produces q' columns 8w.. and 8(w + 8)..
    const int r = lane >> 2, j = lane & 3;
    float acc[2][6][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int c = 0; c < 6; ++c) acc[u][c][0] = acc[u][c][1] = acc[u][c][2] = acc[u][c][3] = 0.f;
    constexpr float kIn = 1.0f / 256.0f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      // A: row r, k index kappa -> input channel 32*(kappa%8/2) + 4s + 2*(kappa/8) + kappa%2
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float4 x = *reinterpret_cast<const float4*>(X + (r + 8 * half) * 128 + 32 * j + 4 * s);
        x.x *= kIn; x.y *= kIn; x.z *= kIn; x.w *= kIn;
        const __half2 h01 = __floats2half2_rn(x.x, x.y), h23 = __floats2half2_rn(x.z, x.w);
        const __half2 l01 = __floats2half2_rn(x.x - __low2float(h01), x.y - __high2float(h01));
        const __half2 l23 = __floats2half2_rn(x.z - __low2float(h23), x.w - __high2float(h23));
        hi[half] = h2_as_u32(h01); hi[2 + half] = h2_as_u32(h23);
        lo[half] = h2_as_u32(l01); lo[2 + half] = h2_as_u32(l23);
      }
      const int c = 3 * (s & 1);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint4 f = rk.f[s][u];
        mma_f16(acc[u][c], hi[0], hi[1], hi[2], hi[3], f.x, f.y);       // hi * hi
        mma_f16(acc[u][c + 1], hi[0], hi[1], hi[2], hi[3], f.z, f.w);   // hi * lo
        mma_f16(acc[u][c + 2], lo[0], lo[1], lo[2], lo[3], f.x, f.y);   // lo * hi
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float y[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        y[e] = ((acc[u][0][e] + acc[u][3][e]) + ((acc[u][1][e] + acc[u][4][e]) + (acc[u][2][e] + acc[u][5][e])));
      const int col = 8 * (warp + 8 * u) + 2 * j;
      *reinterpret_cast<float2*>(Y + r * 128 + col) = make_float2(y[0] * 256.0f, y[1] * 256.0f);
      *reinterpret_cast<float2*>(Y + (r + 8) * 128 + col) = make_float2(y[2] * 256.0f, y[3] * 256.0f);
    }
  }
  __syncthreads();
  for (int row = warp; row < 16; row += 8) {   // per-group sums of q'
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
      float v = 0.f;
      for (int c = grp * GS + lane; c < (grp + 1) * GS; c += 32) v += Y[row * 128 + c];
      v = warp_sum_xor(v, 1);
      if (lane == 0) ssum[row * 2 + grp] = v;
    }
  }
  __syncthreads();
  // fragments: B column n = lane/4 of n-tile nt -> head 4 nt + n/2, part n%2 (hi / lo)
  for (int idx = threadIdx.x; idx < SPB * 32 * QW; idx += 256) {
    const int sl = idx / (32 * QW), ln = (idx / QW) % 32, w = idx % QW;
    const int b = b0 + sl;
    if (b >= B) continue;
    const int r = ln >> 2, j = ln & 3;
    uint32_t val = 0u;
    if (w < 16 * NT) {
      const int reg = w & 1, nt = (w >> 1) % NT, s = (w >> 1) / NT;
      const float* row = Y + (sl * HP + 4 * nt + (r >> 1)) * 128 + 16 * s + 2 * j + 8 * reg;
      // group 64: the odd steps' code factor 16 is cancelled here (a power of 2);
      // group 128 removes it from the odd steps' accumulator chain instead
      const float f = (GS == 64 && (s & 1)) ? 0.0625f : 1.0f;
      const float x0 = row[0] * f, x1 = row[1] * f;
      const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
      const bool lo_part = r & 1;
      const __half p0 = lo_part ? __float2half_rn(x0 - __half2float(h0)) : h0;
      const __half p1 = lo_part ? __float2half_rn(x1 - __half2float(h1)) : h1;
      val = h2_as_u32(__halves2half2(p0, p1));
    } else if (w - 16 * NT < NT * NG) {
      const int kk = w - 16 * NT, nt = kk / NG, grp = kk % NG;
      val = __float_as_uint(ssum[(sl * HP + 4 * nt + j) * 2 + grp] * 5.9604644775390625e-8f);
    }
    a.qfrag[((size_t)(b * a.Hkv + g) * 32 + ln) * QW + w] = val;
  }
}

// ---------------------------------------------------------------------------
// INT2 decode, step 2: history splits (the hot loop) and the tier CTA that
// attends the BF16 rows and merges everything
// ---------------------------------------------------------------------------
// Shared memory of a history CTA (byte offsets).  The per-warp results reuse
// the ring once the loop is done.
// A ring stage known at compile time (the steady-state loop) or at run time.
template <int V>
struct RingStage {};
template <int V>
__device__ __forceinline__ constexpr int stage_index(RingStage<V>) { return V; }
__device__ __forceinline__ int stage_index(int v) { return v; }

template <int G, int GS>
struct HistLay {
  static constexpr int NW = int2_warps(G);
  static constexpr int TB = 1024 + 16 * 8 * (128 / GS);   // stored tile bytes (one ring stage)
  static constexpr int ring = 0;                          // [NW][kStages][TB]
  static constexpr int bars = ring + NW * kStages * TB;   // [NW][kStages] mbarriers
  static constexpr int saddr = bars + NW * kStages * 8;   // [kMaxTilesPerWarp NW] tile source addresses
  static constexpr int spid = saddr + kMaxTilesPerWarp * NW * 8;   // [kMaxPids] page ids
  static constexpr int HP = (G <= 4) ? 4 : 8;             // padded heads (MMA columns)
  static constexpr int sq = spid + kMaxPids * 4;          // [HP][kQStride] q (q' computed in the CTA)
  static constexpr int sqr = sq + HP * kQStride * 4;      // [HP][kQrStride] q'
  static constexpr int spart = sqr + HP * kQrStride * 4; // [16 n-tiles][8] partial row sums of q'
  static constexpr int sqf = spart + 16 * 8 * 4;         // [8 k-steps][NT][32 lanes][2] QK B fragments
                                                         // (first the A fragments of q: [8][32][4])
  static constexpr int ssum = sqf + 8 * 32 * 4 * 4;      // [NT][NG][4] per-group sums of q'
  // the warps' results, written by each warp as its loop ends (not over the
  // ring, which other warps may still be reading); rows of kWoStride floats
  // put the four heads a lane row writes in different banks
  static constexpr int kWoStride = 136;
  static constexpr int swo = (ssum + 2 * 2 * 4 * 4 + 15) / 16 * 16;   // [NW][G][kWoStride] per-warp o'
  static constexpr int swm = swo + NW * G * kWoStride * 4;             // [NW][G] m
  static constexpr int swl = swm + NW * G * 4;                         // [NW][G] l
  static constexpr int swt = swl + NW * G * 4;                         // [NW][G] the warps' weights
  static constexpr int sM = swt + NW * G * 4;                          // [G] each head's maximum
  static constexpr int total = sM + G * 4;
};

// Shared memory of a tier CTA (byte offsets).  R_v^T, the warp results and the
// merged history o' reuse the staging area once the tier rows are attended.
template <int G>
struct TierLay {
  static constexpr int NW = int2_warps(G);
  static constexpr int sq = 0;                                         // [G][128] q
  static constexpr int stage = sq + G * 128 * 4;                       // staged sink + recent rows
  static constexpr int tier_o = stage + kTierRows * (kTierRowK + kTierRowV);   // [G][128] tier partial o
  static constexpr int tier_m = tier_o + G * 128 * 4;                  // [G]
  static constexpr int tier_l = tier_m + G * 4;                        // [G]
  static constexpr int hist_m = tier_l + G * 4;                        // [G] merged history m
  static constexpr int hist_l = hist_m + G * 4;                        // [G]
  static constexpr int bar = (hist_l + G * 4 + 7) / 8 * 8;             // mbarrier of the R_v^T copy
  static constexpr int ctl = bar + 8;                                  // merge progress
  static constexpr int total = ctl + 16;
  static constexpr int kWoStride = 136;   // warp result rows: 128 + 8 keeps the stores conflict-free
  static constexpr int swo = stage;                                    // [NW][G][kWoStride]
  static constexpr int swm = swo + NW * G * kWoStride * 4;             // [NW][G]
  static constexpr int swl = swm + NW * G * 4;                         // [NW][G]
  static constexpr int rv = (swl + NW * G * 4 + 1023) / 1024 * 1024;   // [128][128] R_v^T
  static constexpr int GP = (G + 3) & ~3;
  static constexpr int oh = rv + 128 * 128 * 4;                        // [128][GP] merged history o', transposed
  static constexpr int spr = swo;                                      // [NW][G][128] row-slice sums
  static_assert(oh + GP * 128 * 4 <= tier_o && spr + NW * G * 128 * 4 <= rv,
                "R_v^T, the row-slice sums and the merge fit in the staging area");
  // the tensor-core back-rotation (more than 4 query columns) instead of rv / oh / spr
  static constexpr int HP = (G <= 4) ? 4 : 8;                          // rows of the back-rotation
  static constexpr int sx = (swl + NW * G * 4 + 15) / 16 * 16;         // [HP][kQStride] scaled o'/L
  static constexpr int sy = sx + HP * kQStride * 4;                    // [HP][kQrStride] rotated
  static constexpr int smax = sy + HP * kQrStride * 4;                 // [HP] max |o'/L| (bits)
  static constexpr int sinv = smax + HP * 4;                           // [HP] 1 / scale
  static_assert(sinv + HP * 4 <= tier_o, "the back-rotation fits in the staging area");
};

template <int G, int GS>
constexpr size_t int2_smem() {
  return (size_t)(HistLay<G, GS>::total > TierLay<G>::total ? HistLay<G, GS>::total : TierLay<G>::total);
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One history split of (sequence b, KV head g): stream its 16-token tiles of
// 2-bit codes and attend them with q' (in the rotated basis), and write the
// split's partial (m, l, o' unnormalised) to `part`.
template <int G, int GS, bool kMulti>
__device__ void int2_history(const DecodeArgs& a, int b, int g, int split, uint8_t* smb, float* part) {
  constexpr int NW = int2_warps(G);
  using S = HistLay<G, GS>;
  constexpr int HP = (G <= 4) ? 4 : 4 * ((G + 3) / 4);
  constexpr int NT = HP / 4;         // MMA n-tiles of 8 columns (4 heads x hi / lo)
  constexpr int NG = 128 / GS;       // quantization groups per row
  constexpr int QW = qfrag_words<G>();
  constexpr uint32_t TB = S::TB;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, j = lane & 3;

  // ---- barriers, then one round of independent loads: the split's page ids
  // and the length; lane 0 of each warp also reads the page ids of its first
  // tiles itself, so that their copies start as soon as the page table answers.
  // A ring stage holds one whole stored tile, brought in by one bulk copy that
  // lane 0 issues and that completes on the stage's mbarrier. ----
  uint8_t* ring = smb + S::ring + (size_t)warp * kStages * TB;
  uint64_t* wbar = reinterpret_cast<uint64_t*>(smb + S::bars) + warp * kStages;
  uint64_t* saddr = reinterpret_cast<uint64_t*>(smb + S::saddr);   // per-tile source addresses
  int* spid = reinterpret_cast<int*>(smb + S::spid);
  if (lane < kStages) mbar_init(wbar + lane, 1);
  mbar_fence_init();
  // q' is formed here (kQLocal) or taken from the pre-pass.  When formed here,
  // each warp loads its own R_k fragments (4 KB, a pool constant) into
  // registers before the wait for the preceding kernel, which this launch may
  // overlap; every buffer the caller passes is read after it
  const bool local = a.qmode == kQLocal;
  RotFrags<NW> rkf;
  if (local) {
    rkf.load(a.rfrag + (size_t)g * kFragBlocks * 4096);
    asm volatile("griddepcontrol.wait;" ::: "memory");
  }

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
  for (int i = threadIdx.x; i < p_all; i += NW * 32) spid[i] = __ldg(ptrow + p_begin + i);
  float* sq = reinterpret_cast<float*>(smb + S::sq);
  if (local) load_q<G, NW, kMulti, true>(a, b, g, sq, S::HP);
  int h = __ldg(a.hist_len + b);
  // the grid covers max_len history tokens (and the page table max_pages pages)
  const int cap = min(a.max_pages * a.page_size, a.max_len);
  if (h < 0 || h > cap) {
    if (threadIdx.x == 0) flag_error(a.err, KV_DEVERR_LENGTH);
    h = max(0, min(h, cap));
  }
  const int ntiles = (h + kTile - 1) / kTile;
  const int t_end = min(ntiles, t_begin + a.per_split);
  if (t_begin >= t_end) {   // the same for every thread: no tile copy was started
    write_empty_partial<G, NW>(part);
    return;
  }

  // ---- start streaming this warp's first tiles into its ring ----
  const uint8_t* head_base = a.hist + (size_t)g * (a.page_bytes / a.Hkv);
  // s/z records of tokens r and r + 8 (record slots 2r, 2r + 1): K block at
  // 1024, V block 16 slots of 4 NG bytes later
  const int lane_szk = 1024 + 8 * NG * r, lane_szv = lane_szk + 64 * NG;
  // the history is read once per step: its lines leave L2 first
  const uint64_t stream_policy = l2_evict_first_policy();
  auto start_copy = [&](int t, int pid, int stage) {
    const uint8_t* tb = (pid >= 0 && pid < a.num_pages)
                            ? head_base + (size_t)pid * a.page_bytes + (t & tmask) * a.tile_bytes
                            : g_zero_tile;
    mbar_expect_tx(wbar + stage, TB);
    bulk_g2s_hint(ring + stage * TB, tb, TB, wbar + stage, stream_policy);
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
  __syncthreads();   // the page ids (and q) are in shared memory

  // ---- the source address of every tile of the split, bit 0 set when its
  // page id is valid (else the copy reads a zero tile and its tokens are
  // masked); bad page ids are reported here, once per tile ----
  int bad = 0;
  for (int i = threadIdx.x; i < t_end - t_begin; i += NW * 32) {
    const int t = t_begin + i;
    const int pid = spid[(t >> tsh) - p_begin];
    if (pid >= 0 && pid < a.num_pages) {
      saddr[i] = reinterpret_cast<uint64_t>(head_base + (size_t)pid * a.page_bytes +
                                            (t & tmask) * a.tile_bytes) | 1ull;
    } else {
      saddr[i] = reinterpret_cast<uint64_t>(g_zero_tile);
      flag_error(a.err, KV_DEVERR_PAGE_ID);
      bad = 1;
    }
  }
  bad = __syncthreads_or(bad);   // the table is complete; any bad page -> every tile masked

  uint32_t qf[8][NT][2];
  float sumq[NT][NG];
  bool ok = true;
  if (local) {   // ---- q' = q R_k here, then its fragments and per-group sums ----
    float* sqr = reinterpret_cast<float*>(smb + S::sqr);
    float* spart = reinterpret_cast<float*>(smb + S::spart);
    rotate_q<S::HP, NW, true>(sq, rkf, sqr, spart, reinterpret_cast<uint32_t*>(smb + S::sqf));   // ends with a barrier
    // The QK B fragments and the per-group sums are the same in every warp:
    // work item p < 8 NT (k-step p / NT, n-tile p % NT) builds one fragment
    // pair for all 32 lanes, item 8 NT the sums; the warps take the items in
    // turn, and every warp then loads its copy from shared memory.
    uint32_t* sqf = reinterpret_cast<uint32_t*>(smb + S::sqf);
    float* ssum = reinterpret_cast<float*>(smb + S::ssum);
    for (int p = warp; p <= 8 * NT; p += NW) {
      if (p < 8 * NT) {
        const int s = p / NT, nt = p % NT;
        // QK B fragments: column n = lane/4 -> local head 4*nt + n/2, part n%2 (hi/lo)
        const int hl = r >> 1, e = r & 1;
        const float* row = sqr + (4 * nt + hl) * kQrStride + 16 * s + 2 * j;
        // group 64: the odd steps' code factor 16 is cancelled here (a power of 2);
        // group 128 removes it from the odd steps' accumulator chain instead
        const float f = (GS == 64 && (s & 1)) ? 0.0625f : 1.0f;
        const float x[4] = {row[0] * f, row[1] * f, row[8] * f, row[9] * f};
        __half hp[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const __half hi = __float2half_rn(x[u]);
          hp[u] = e ? __float2half_rn(x[u] - __half2float(hi)) : hi;
        }
        *reinterpret_cast<uint2*>(sqf + (p * 32 + lane) * 2) =
            make_uint2(h2_as_u32(__halves2half2(hp[0], hp[1])), h2_as_u32(__halves2half2(hp[2], hp[3])));
      } else if (lane < 4 * NT * NG) {
        // per-group sums of q' (over the group's 8-column n-tiles) in the units
        // of the score accumulator (2^-24): lane = (n-tile, group, column pair)
        const int jj = lane & 3, grp = (lane >> 2) % NG, nt = (lane >> 2) / NG;
        float v = 0.f;
        for (int t = grp * (GS / 8); t < (grp + 1) * (GS / 8); ++t) v += spart[t * 8 + 4 * nt + jj];
        ssum[(nt * NG + grp) * 4 + jj] = v * 5.9604644775390625e-8f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int s = 0; s < 8; ++s)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint2 w = *reinterpret_cast<const uint2*>(sqf + ((s * NT + nt) * 32 + lane) * 2);
        qf[s][nt][0] = w.x;
        qf[s][nt][1] = w.y;
      }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) sumq[nt][grp] = ssum[(nt * NG + grp) * 4 + j];
  } else {   // ---- q' fragments and per-group sums from the pre-pass ----
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint4* qp = reinterpret_cast<const uint4*>(a.qfrag + ((size_t)(b * a.Hkv + g) * 32 + lane) * QW);
    uint32_t w[QW];
#pragma unroll
    for (int i = 0; i < QW / 4; ++i) {
      const uint4 v = __ldcg(qp + i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
#pragma unroll
    for (int s = 0; s < 8; ++s)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        qf[s][nt][0] = w[(s * NT + nt) * 2];
        qf[s][nt][1] = w[(s * NT + nt) * 2 + 1];
      }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) sumq[nt][grp] = __uint_as_float(w[16 * NT + nt * NG + grp]);
  }
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

  int k = 0;   // this warp's tile count: ring stage k % kStages, phase k / kStages
  const int n_warp = max(0, (t_end - t_begin - warp + NW - 1) / NW);   // tiles of this warp
  auto issue = [&](int t, int stage) {   // tiles k >= kStages - 1, from the address table
    if (lane == 0 && t < t_end) {
      const uint64_t e = saddr[t - t_begin];
      mbar_expect_tx(wbar + stage, TB);
      bulk_g2s_hint(ring + stage * TB, reinterpret_cast<const void*>(e & ~1ull), TB, wbar + stage, stream_policy);
    }
  };
  // One tile: QK, online softmax and PV.  kMask: the tile may hold tokens past
  // the history or sit behind a bad page id (only the split's last tile, or
  // every tile of a split with a bad page); other tiles need no masks.
  // Returns false if its copy did not arrive in time.
  // st / par: the ring stage and the phase parity of tile k (compile-time
  // stages in the steady-state loop below).
  auto tile = [&](int t, auto mask_tag, auto stage, uint32_t par) -> bool {
    constexpr bool kMask = decltype(mask_tag)::value;
    const int st = stage_index(stage);
    __syncwarp();   // every lane is done with the stage refilled next
    // tile k+3 goes into the stage read in the previous iteration
    issue(t + NW * (kStages - 1), (st + kStages - 1) % kStages);
    {   // one poll first (the copy is usually in); the bounded loop only if it is not
      uint32_t ready;
      asm volatile(
          "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
          : "=r"(ready)
          : "r"(smem_u32(wbar + st)), "r"(par)
          : "memory");
      if (!__all_sync(0xffffffffu, ready != 0u) &&
          !__all_sync(0xffffffffu, mbar_wait(wbar + st, par, a.wait_polls)))
        return false;
    }
    const uint8_t* src = ring + st * TB;
    const uint4 kq4 = *reinterpret_cast<const uint4*>(src + 16 * lane);
    const uint4 vq4 = *reinterpret_cast<const uint4*>(src + 512 + 16 * lane);
    uint4 szk, szv;   // group 128: (x, y) = tokens r, r + 8; group 64: (x, y) token r, (z, w) token r + 8
    if (GS == 128) {
      const uint2 k2 = *reinterpret_cast<const uint2*>(src + lane_szk);
      const uint2 v2 = *reinterpret_cast<const uint2*>(src + lane_szv);
      szk = make_uint4(k2.x, k2.y, 0u, 0u);
      szv = make_uint4(v2.x, v2.y, 0u, 0u);
    } else {
      szk = *reinterpret_cast<const uint4*>(src + lane_szk);
      szv = *reinterpret_cast<const uint4*>(src + lane_szv);
    }
    bool v0 = true, v1 = true;
    if constexpr (kMask) {   // tokens of this tile still inside the history (none if its page id is bad)
      const int lim = ((saddr[t - t_begin] & 1ull) != 0) ? h - t * kTile : 0;
      v0 = r < lim;
      v1 = r + 8 < lim;
    }

    // scale / zero of tokens r and r+8
    float sk[2][NG], zk[2][NG], sv[2][NG], zv[2][NG];
    if (GS == 128) {
      sk[0][0] = __low2float(u32_as_h2(szk.x)); zk[0][0] = __high2float(u32_as_h2(szk.x));
      sk[1][0] = __low2float(u32_as_h2(szk.y)); zk[1][0] = __high2float(u32_as_h2(szk.y));
      sv[0][0] = __low2float(u32_as_h2(szv.x)); zv[0][0] = __high2float(u32_as_h2(szv.x));
      sv[1][0] = __low2float(u32_as_h2(szv.y)); zv[1][0] = __high2float(u32_as_h2(szv.y));
    } else {
      sk[0][0] = __low2float(u32_as_h2(szk.x)); zk[0][0] = __high2float(u32_as_h2(szk.x));
      sk[0][NG - 1] = __low2float(u32_as_h2(szk.y)); zk[0][NG - 1] = __high2float(u32_as_h2(szk.y));
      sk[1][0] = __low2float(u32_as_h2(szk.z)); zk[1][0] = __high2float(u32_as_h2(szk.z));
      sk[1][NG - 1] = __low2float(u32_as_h2(szk.w)); zk[1][NG - 1] = __high2float(u32_as_h2(szk.w));
      sv[0][0] = __low2float(u32_as_h2(szv.x)); zv[0][0] = __high2float(u32_as_h2(szv.x));
      sv[0][NG - 1] = __low2float(u32_as_h2(szv.y)); zv[0][NG - 1] = __high2float(u32_as_h2(szv.y));
      sv[1][0] = __low2float(u32_as_h2(szv.z)); zv[1][0] = __high2float(u32_as_h2(szv.z));
      sv[1][NG - 1] = __low2float(u32_as_h2(szv.w)); zv[1][NG - 1] = __high2float(u32_as_h2(szv.w));
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
      if constexpr (kMask) {
        l0 = v0 ? l0 * sc24 : kNegInf;
        l1 = v1 ? l1 * sc24 : kNegInf;
      } else {
        l0 *= sc24;
        l1 *= sc24;
      }
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
    ++k;
    return true;
  };

  // tiles below t_full are full and behind valid pages: no masks
  const int t_full = bad ? t_begin : min(t_end, h / kTile);
  const bool started = ok;
  int t = ok ? t_begin + warp : t_end;   // a lost R_k copy skips the split
  // steady state: kStages unmasked tiles per pass, one per ring stage, so that
  // stage offsets and barrier addresses are constants (k is a multiple of
  // kStages here); the phase parity flips once per pass
  uint32_t ph = 0;
  for (; ok && t + NW * (kStages - 1) < t_full; t += NW * kStages, ph ^= 1u) {
    ok = tile(t, std::false_type{}, RingStage<0>{}, ph) &&
         tile(t + NW, std::false_type{}, RingStage<1>{}, ph) &&
         tile(t + 2 * NW, std::false_type{}, RingStage<2>{}, ph) &&
         tile(t + 3 * NW, std::false_type{}, RingStage<3>{}, ph);
    if (!ok) t = t_end;   // k counts the tiles done
  }
  static_assert(kStages == 4, "the steady-state pass above takes one tile per stage");
  // the rest (fewer than kStages full tiles, then the tail) through the masked body
  for (; ok && t < t_end; t += NW)
    ok = tile(t, std::true_type{}, k % kStages, (uint32_t)(k / kStages) & 1u);
  if (!ok) {   // a copy did not arrive in time: wait (bounded) for the ones in flight,
    // those of tiles k .. issued - 1 of this warp (tile k issued tile k + kStages - 1
    // before its wait ran out; a split that never started issued the first kStages - 1)
    if (lane == 0) flag_error(a.err, KV_DEVERR_TIMEOUT);
    const int issued = started ? min(k + kStages, n_warp) : min(kStages - 1, n_warp);
    for (int kk = k; kk < issued; ++kk) mbar_wait(wbar + kk % kStages, (kk / kStages) & 1, a.wait_polls);
  }
  if (lane < kStages) mbar_inval(wbar + lane);   // this warp's copies are all in (or given up on)

  // ---- this warp's results -> shared memory, as soon as its loop ends ----
  float* swo = reinterpret_cast<float*>(smb + S::swo);
  float* swm = reinterpret_cast<float*>(smb + S::swm);
  float* swl = reinterpret_cast<float*>(smb + S::swl);
  constexpr int WS = S::kWoStride;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float l = warp_sum_xor(l_run[nt], 4);
    float z[NG];
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) z[grp] = warp_sum_xor(zs[nt][grp], 4);
    const int hh = 4 * nt + j;
    if (hh < G) {
      float* o = swo + (warp * G + hh) * WS;
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
  ok = __syncthreads_and(ok);   // every warp's results are in
  if (!ok) {   // the split's result is skipped
    write_empty_partial<G, NW>(part);
    return;
  }
  // the warps merged with the log-sum-exp rule into the split's partial (rotated
  // basis): for each (warp, head) its head's maximum and the warp's weight
  // exp2(m_w - M), then every output element a sum of NW products
  float* swt = reinterpret_cast<float*>(smb + S::swt);
  float* sM = reinterpret_cast<float*>(smb + S::sM);
  if (threadIdx.x < NW * G) {
    const int hh = threadIdx.x % G;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, swm[w * G + hh]);
    const float mw = swm[threadIdx.x];
    swt[threadIdx.x] = (mw == kNegInf || M == kNegInf) ? 0.f : exp2f(mw - M);
    if (threadIdx.x < G) sM[threadIdx.x] = M;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * 128; idx += NW * 32) {
    const int hh = idx >> 7, c = idx & 127;
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) O = fmaf(swt[w * G + hh], swo[(w * G + hh) * WS + c], O);
    part[hh * kPart + 4 + c] = O;
    if (c == 0) {
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) L = fmaf(swt[w * G + hh], swl[w * G + hh], L);
      part[hh * kPart + 0] = sM[hh];
      part[hh * kPart + 1] = L;
    }
  }
}

// The tier CTA of (sequence b, KV head g), launched after every history
// split: attends the BF16 sink + recent rows (staged in shared memory, on the
// tensor cores), then merges the history splits' partials in split order as they
// arrive (each split sets its bit in the pair's arrival mask with a release
// reduction after writing its partial), rotates the merged history value sum
// back by R_v^T once, combines it with the tier result and writes the output.
template <int G, int GS, bool kMulti>
__device__ void tier_merge(const DecodeArgs& a, int b, int g, uint8_t* smb) {
  constexpr int NW = int2_warps(G);
  using S = TierLay<G>;
  const int warp = threadIdx.x >> 5;
  const int scap = a.sink_cap, rcap = a.rec_cap, rows = scap + rcap;
  const size_t seq_head = (size_t)b * a.Hkv + g;
  const uint16_t* sk = a.sink_k + seq_head * scap * 128;
  const uint16_t* sv = a.sink_v + seq_head * scap * 128;
  const uint16_t* rk = a.rec_k + seq_head * rcap * 128;
  const uint16_t* rv = a.rec_v + seq_head * rcap * 128;
  float* sq = reinterpret_cast<float*>(smb + S::sq);
  uint8_t* stk = smb + S::stage;
  uint8_t* stv = stk + (size_t)kTierRows * kTierRowK;
  // every input of the tier CTA comes from the caller: after the preceding kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");
  auto stage_rows = [&](int r0, int r1) {   // storage rows [r0, r1) of [sink slots | recent ring]
    for (int i = threadIdx.x; i < (r1 - r0) * 32; i += NW * 32) {
      const int t = i >> 5, c = i & 31, key = c < 16, ch = c & 15, row = r0 + t;
      const uint16_t* src = (row < scap) ? (key ? sk : sv) + (size_t)row * 128
                                         : (key ? rk : rv) + (size_t)(row - scap) * 128;
      uint8_t* dst = key ? stk + t * kTierRowK + 16 * ch : stv + t * kTierRowV + 16 * ch;
      cp_async16(dst, reinterpret_cast<const uint8_t*>(src) + 16 * ch);
    }
    cp_async_commit();
  };
  stage_rows(0, min(rows, kTierRows));   // before the lengths are known
  load_q<G, NW, kMulti>(a, b, g, sq, G);
  int ns = __ldg(a.sink_len + b), nr = __ldg(a.rec_len + b), rs = __ldg(a.rec_start + b);
  if (ns < 0 || ns > scap || nr < 0 || nr > rcap || rs < 0 || rs >= rcap) {
    if (threadIdx.x == 0) flag_error(a.err, KV_DEVERR_LENGTH);
    ns = max(0, min(ns, scap));
    nr = max(0, min(nr, rcap));
    rs = max(0, min(rs, rcap - 1));
  }
  // ---- the tier rows on the tensor cores: warp w takes the 16-row tiles w,
  // w + NW, .. of each staged pass; q exact in bf16 as the QK B operand (column
  // 2h: head h, 2h + 1: zero), the softmax weights as bf16 hi + lo for PV, the
  // online softmax with the lazy reference of the history loop ----
  constexpr int NT = (G <= 4) ? 1 : 2;
  const int lane = threadIdx.x & 31, r = lane >> 2, j = lane & 3;
  auto live_row = [&](int u) -> bool {   // storage row u holds a token of the sequence
    if (u < scap) return u < ns;
    int d = (u - scap) - rs;
    d += (d < 0) ? rcap : 0;
    return d < nr;
  };
  uint32_t qf[8][NT][2];
  float m_run[NT], base[NT], l_run[NT], oacc[8][NT][4];
#pragma unroll
  for (int u = 0; u < NT; ++u) {
    m_run[u] = kNegInf;
    base[u] = 0.f;
    l_run[u] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) oacc[i][u][0] = oacc[i][u][1] = oacc[i][u][2] = oacc[i][u][3] = 0.f;
  }
  const uint32_t sk_base = smem_u32(stk), sv_base = smem_u32(stv);
  const int krow = lane & 15, kc = lane >> 4;
  const int vrow = (lane & 7) + 8 * (lane >> 4), vc = (lane >> 3) & 1;
  for (int r0 = 0; r0 < rows; r0 += kTierRows) {
    const int r1 = min(rows, r0 + kTierRows);
    if (r0 > 0) stage_rows(r0, r1);
    cp_async_wait<0>();
    __syncthreads();
    if (r0 == 0) {   // q (in shared memory since the barrier) -> B fragments
      const int hh = r >> 1;
#pragma unroll
      for (int u = 0; u < NT; ++u) {
        const int head = 4 * u + hh;
        const bool on = !(r & 1) && head < G;
        const float* qrow = sq + (on ? head : 0) * 128;
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) {
          const int c = 16 * s2 + 2 * j;
          qf[s2][u][0] = on ? ((__float_as_uint(qrow[c]) >> 16) | (__float_as_uint(qrow[c + 1]) & 0xFFFF0000u)) : 0u;
          qf[s2][u][1] = on ? ((__float_as_uint(qrow[c + 8]) >> 16) | (__float_as_uint(qrow[c + 9]) & 0xFFFF0000u)) : 0u;
        }
      }
    }
    const int nrow = r1 - r0, ntile = (nrow + 15) / 16;
    for (int tt = warp; tt < ntile; tt += NW) {
      const int t0 = 16 * tt;
      // a dead row's V (or a row past the pass) is zeroed, so that its zero
      // weight never meets a stale value
      if (lane < 16 && !(t0 + lane < nrow && live_row(r0 + t0 + lane))) {
        uint4* vz = reinterpret_cast<uint4*>(stv + (size_t)(t0 + lane) * kTierRowV);
#pragma unroll
        for (int c = 0; c < 16; ++c) vz[c] = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
      const bool v0 = t0 + r < nrow && live_row(r0 + t0 + r);
      const bool v1 = t0 + r + 8 < nrow && live_row(r0 + t0 + r + 8);
      float sacc[NT][4];
#pragma unroll
      for (int u = 0; u < NT; ++u) sacc[u][0] = sacc[u][1] = sacc[u][2] = sacc[u][3] = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
        uint32_t fa[4];
        ldmatrix_x4(sk_base + (t0 + krow) * kTierRowK + (2 * s2 + kc) * 16, fa);
#pragma unroll
        for (int u = 0; u < NT; ++u) mma_bf16(sacc[u], fa[0], fa[1], fa[2], fa[3], qf[s2][u][0], qf[s2][u][1]);
      }
      uint32_t bpv[NT][2];
#pragma unroll
      for (int u = 0; u < NT; ++u) {
        const float l0 = v0 ? sacc[u][0] * a.scale_log2 : kNegInf;
        const float l1 = v1 ? sacc[u][2] * a.scale_log2 : kNegInf;
        if (__any_sync(0xffffffffu, fmaxf(l0, l1) > m_run[u])) {
          float tmax = fmaxf(l0, l1);
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
          const bool need = tmax > m_run[u];
          const float mnew = need ? tmax + kSlack : m_run[u];
          const float alpha = need ? ((m_run[u] == kNegInf) ? 0.f : exp2_neg(m_run[u] - mnew)) : 1.f;
          m_run[u] = mnew;
          base[u] = (mnew == kNegInf) ? 0.f : mnew;
          l_run[u] *= alpha;
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[i][u][e] *= alpha;
        }
        const float p0 = exp2_neg(l0 - base[u]), p1 = exp2_neg(l1 - base[u]);
        l_run[u] += p0 + p1;
        bpv[u][0] = movmatrix_t(split_hi_lo_bf16(p0));
        bpv[u][1] = movmatrix_t(split_hi_lo_bf16(p1));
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t fa[4];
        ldmatrix_x4_t(sv_base + (t0 + vrow) * kTierRowV + (2 * i + vc) * 16, fa);
#pragma unroll
        for (int u = 0; u < NT; ++u) mma_bf16(oacc[i][u], fa[0], fa[1], fa[2], fa[3], bpv[u][0], bpv[u][1]);
      }
    }
    __syncthreads();   // the staged rows are dead before they are replaced or reused
  }
  float* swo = reinterpret_cast<float*>(smb + S::swo);
  float* swm = reinterpret_cast<float*>(smb + S::swm);
  float* swl = reinterpret_cast<float*>(smb + S::swl);
  float* tier_o = reinterpret_cast<float*>(smb + S::tier_o);
  float* tier_m = reinterpret_cast<float*>(smb + S::tier_m);
  float* tier_l = reinterpret_cast<float*>(smb + S::tier_l);
#pragma unroll
  for (int u = 0; u < NT; ++u) {   // warp results (hi + lo columns summed) -> shared memory
    const float l = warp_sum_xor(l_run[u], 4);
    const int hh = 4 * u + j;
    if (hh < G) {
      float* o = swo + (warp * G + hh) * S::kWoStride;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        o[16 * i + r] = oacc[i][u][0] + oacc[i][u][1];
        o[16 * i + r + 8] = oacc[i][u][2] + oacc[i][u][3];
      }
      if (r == 0) {
        swm[warp * G + hh] = m_run[u];
        swl[warp * G + hh] = l;
      }
    }
  }
  __syncthreads();
  merge_warps<G, NW, S::kWoStride>(swo, swm, swl, tier_o, tier_m, tier_l);   // ends with a barrier

  // ---- R_v^T for the one back-rotation: up to 4 query columns as fp32 into the
  // staging area, now free (SIMT rotation); more as MMA fragments in registers
  // (tensor-core rotation), both while the history splits finish ----
  uint64_t* rbar = reinterpret_cast<uint64_t*>(smb + S::bar);
  float* srv = reinterpret_cast<float*>(smb + S::rv);
  RotFrags<NW> rvf;
  if constexpr (G > 4) rvf.load(a.rfrag + ((size_t)g * kFragBlocks + 3) * 4096);
  if (G <= 4 && threadIdx.x == 0) {
    mbar_init(rbar, 1);
    mbar_fence_init();
    const float* R = a.RvT + (size_t)g * 128 * 128;
    const uint64_t keep = l2_evict_last_policy();
    mbar_expect_tx(rbar, 128 * 128 * 4);
#pragma unroll
    for (int c = 0; c < 4; ++c) bulk_g2s_hint(srv + 4096 * c, R + 4096 * c, 16384, rbar, keep);
  }

  // ---- merge the history partials, in split order, batch by batch as the
  // splits of a batch arrive (fixed batches: the arithmetic, and so the
  // result, does not depend on arrival order) ----
  constexpr int EPT = (G * 128 + NW * 32 - 1) / (NW * 32);   // output elements per thread
  float M[EPT], L[EPT], O[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    M[e] = kNegInf;
    L[e] = 0.f;
    O[e] = 0.f;
  }
  int* ctl = reinterpret_cast<int*>(smb + S::ctl);
  unsigned* mask = a.arrive + seq_head * kMaskWords;
  const float* pbase = a.ws + seq_head * a.n_split * G * kPart;
  bool merged_all = true;
  if constexpr (G > 4) {
  // 8 query columns: per-head maxima and weights computed once per batch
  // (fewer exponentials than per element, which pays off at this width; with
  // fewer columns the extra barriers cost more than they save); per-head state
  // and the batch's weights in the (dead) tier warp results
  float* sml = reinterpret_cast<float*>(smb + S::swo);   // [kMergeBatch][G] (m, l)
  float* sf = sml + 2 * kMergeBatch * G;                  // [kMergeBatch][G] weights
  float* sMh = sf + kMergeBatch * G;                      // [G] running m
  float* sLh = sMh + G;                                   // [G] running l
  float* sal = sLh + G;                                   // [G] rescale of the running sums
  if (threadIdx.x < G) {
    sMh[threadIdx.x] = kNegInf;
    sLh[threadIdx.x] = 0.f;
  }
  for (int s0 = 0; s0 < a.n_split; s0 += kMergeBatch) {
    const int s1 = min(a.n_split, s0 + kMergeBatch);
    if (threadIdx.x == 0) {   // wait (bounded) until splits s0 .. s1-1 have arrived
      int done = 0;
      for (int it = 0; it < a.merge_polls && !done; ++it) {
        done = 1;
        for (int s = s0; s < s1 && done; s += 32 - (s & 31)) {
          const int n = min(s1 - s, 32 - (s & 31));
          const unsigned want = (n == 32 ? ~0u : ((1u << n) - 1u)) << (s & 31);
          done = (ld_acquire_u32(mask + (s >> 5)) & want) == want;
        }
        if (!done) __nanosleep(16);
      }
      ctl[0] = done;
    }
    __syncthreads();
    const bool arrived = ctl[0] != 0;
    __syncthreads();   // ctl is rewritten for the next batch
    if (!arrived) {
      merged_all = false;
      break;
    }
    // one round of loads: every thread its o values of the batch, the first
    // threads the (m, l) of every (split, head)
    const int nb = s1 - s0;
    float ov[EPT][kMergeBatch];
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int idx = threadIdx.x + e * NW * 32;
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u)
        ov[e][u] = (idx < G * 128 && u < nb)
                       ? __ldcg(pbase + ((size_t)(s0 + u) * G + (idx >> 7)) * kPart + 4 + (idx & 127))
                       : 0.f;
    }
    for (int i = threadIdx.x; i < nb * G; i += NW * 32) {
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(pbase + ((size_t)s0 * G + i) * kPart));
      sml[2 * i] = ml.x;
      sml[2 * i + 1] = ml.y;
    }
    __syncthreads();
    if (threadIdx.x < G) {   // each head's new maximum and the rescale of its running sums
      const int hh = threadIdx.x;
      float Mb = sMh[hh];
      for (int u = 0; u < nb; ++u) Mb = fmaxf(Mb, sml[2 * (u * G + hh)]);
      sal[hh] = (sMh[hh] == kNegInf || Mb == kNegInf) ? 0.f : exp2f(sMh[hh] - Mb);
      sMh[hh] = Mb;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nb * G; i += NW * 32) {   // every (split, head)'s weight
      const float mv = sml[2 * i], Mb = sMh[i % G];
      sf[i] = (mv == kNegInf || Mb == kNegInf) ? 0.f : exp2f(mv - Mb);
    }
    __syncthreads();
    if (threadIdx.x < G) {
      const int hh = threadIdx.x;
      float Le = sLh[hh] * sal[hh];
      for (int u = 0; u < nb; ++u) Le = fmaf(sf[u * G + hh], sml[2 * (u * G + hh) + 1], Le);
      sLh[hh] = Le;
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int idx = threadIdx.x + e * NW * 32;
      if (idx < G * 128) {
        const int hh = idx >> 7;
        float Oe = O[e] * sal[hh];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) Oe = fmaf(u < nb ? sf[u * G + hh] : 0.f, ov[e][u], Oe);
        O[e] = Oe;
      }
    }
    __syncthreads();   // sml / sf / sal are rewritten by the next batch
  }
#pragma unroll
  for (int e = 0; e < EPT; ++e) {   // the per-head m and l of each element's head
    const int idx = threadIdx.x + e * NW * 32;
    if (idx < G * 128) {
      M[e] = sMh[idx >> 7];
      L[e] = sLh[idx >> 7];
    }
  }
  } else {
  for (int s0 = 0; s0 < a.n_split; s0 += kMergeBatch) {
    const int s1 = min(a.n_split, s0 + kMergeBatch);
    if (threadIdx.x == 0) {   // wait (bounded) until splits s0 .. s1-1 have arrived
      int done = 0;
      for (int it = 0; it < a.merge_polls && !done; ++it) {
        done = 1;
        for (int s = s0; s < s1 && done; s += 32 - (s & 31)) {
          const int n = min(s1 - s, 32 - (s & 31));
          const unsigned want = (n == 32 ? ~0u : ((1u << n) - 1u)) << (s & 31);
          done = (ld_acquire_u32(mask + (s >> 5)) & want) == want;
        }
        if (!done) __nanosleep(16);
      }
      ctl[0] = done;
    }
    __syncthreads();
    const bool arrived = ctl[0] != 0;
    __syncthreads();   // ctl is rewritten for the next batch
    if (!arrived) {
      merged_all = false;
      break;
    }
#pragma unroll 1
    for (int e = 0; e < EPT; ++e) {
      const int idx = threadIdx.x + e * NW * 32;
      if (idx >= G * 128) break;
      const int hh = idx >> 7, c = idx & 127;
      const float* ph = pbase + (size_t)hh * kPart;
      float mv[kMergeBatch], lv[kMergeBatch], ov[kMergeBatch];
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const int s = s0 + u;
        const float* pp = ph + (size_t)s * G * kPart;
        const float2 ml = (s < s1) ? __ldcg(reinterpret_cast<const float2*>(pp)) : make_float2(kNegInf, 0.f);
        mv[u] = ml.x;
        lv[u] = ml.y;
        ov[u] = (s < s1) ? __ldcg(pp + 4 + c) : 0.f;
      }
      float Mb = M[e];
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) Mb = fmaxf(Mb, mv[u]);
      if (Mb != kNegInf) {
        const float alpha = (M[e] == kNegInf) ? 0.f : exp2f(M[e] - Mb);
        float Le = L[e] * alpha, Oe = O[e] * alpha;
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          const float f = (mv[u] == kNegInf) ? 0.f : exp2f(mv[u] - Mb);
          Le = fmaf(f, lv[u], Le);
          Oe = fmaf(f, ov[u], Oe);
        }
        M[e] = Mb;
        L[e] = Le;
        O[e] = Oe;
      }
    }
  }
  }
  if (!merged_all && threadIdx.x == 0) flag_error(a.err, KV_DEVERR_TIMEOUT);

  if constexpr (G <= 4) {
  // ---- back to the original basis once: o_hist[h][c] = sum_i o'[h][i] R_v^T[i][c].
  // o' goes to shared memory transposed ([c][GP]); each row of R_v^T is read
  // once for all heads: warp w takes rows w, w + NW, .., lane cq columns
  // 4cq..4cq+3, and the NW row-slice sums are added at the end ----
  constexpr int GP = S::GP;
  float* oT = reinterpret_cast<float*>(smb + S::oh);
  float* spr = reinterpret_cast<float*>(smb + S::spr);
  float* hist_m = reinterpret_cast<float*>(smb + S::hist_m);
  float* hist_l = reinterpret_cast<float*>(smb + S::hist_l);
  for (int idx = threadIdx.x; idx < GP * 128; idx += NW * 32)
    if ((idx >> 7) >= G) oT[(idx & 127) * GP + (idx >> 7)] = 0.f;   // padded heads
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int idx = threadIdx.x + e * NW * 32;
    if (idx < G * 128) {
      oT[(idx & 127) * GP + (idx >> 7)] = O[e];
      if ((idx & 127) == 0) {
        hist_m[idx >> 7] = M[e];
        hist_l[idx >> 7] = L[e];
      }
    }
  }
  if (!mbar_wait(rbar, 0, a.wait_polls) && (threadIdx.x & 31) == 0) flag_error(a.err, KV_DEVERR_TIMEOUT);
  __syncthreads();
  {
    const int cq = threadIdx.x & 31;
    float acc[GP][4];
#pragma unroll
    for (int hh = 0; hh < GP; ++hh) acc[hh][0] = acc[hh][1] = acc[hh][2] = acc[hh][3] = 0.f;
#pragma unroll 4
    for (int i = warp; i < 128; i += NW) {   // rows of R_v^T: warp, warp + NW, ..
      const float4 rr = *reinterpret_cast<const float4*>(srv + i * 128 + 4 * cq);
#pragma unroll
      for (int hq = 0; hq < GP / 4; ++hq) {
        const float4 o = *reinterpret_cast<const float4*>(oT + i * GP + 4 * hq);
        const float ox[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float* d = acc[4 * hq + e];
          d[0] = fmaf(ox[e], rr.x, d[0]); d[1] = fmaf(ox[e], rr.y, d[1]);
          d[2] = fmaf(ox[e], rr.z, d[2]); d[3] = fmaf(ox[e], rr.w, d[3]);
        }
      }
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
      *reinterpret_cast<float4*>(spr + (warp * G + hh) * 128 + 4 * cq) =
          make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * 128; idx += NW * 32) {
    const int hh = idx >> 7, c = idx & 127;
    float oh = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) oh += spr[w * G * 128 + idx];
    const float Mh = hist_m[hh], Lh = hist_l[hh], mt = tier_m[hh], lt = tier_l[hh];
    const float Mx = fmaxf(Mh, mt);
    const float fh = (Mh == kNegInf) ? 0.f : exp2f(Mh - Mx);
    const float ft = (mt == kNegInf) ? 0.f : exp2f(mt - Mx);
    const float Lt = fmaf(Lh, fh, lt * ft);
    const float val = (Lt > 0.f) ? fmaf(oh, fh, tier_o[idx] * ft) / Lt : 0.f;
    if constexpr (kMulti) {
      const size_t row = ((size_t)b * a.T + hh / a.Gq) * a.Hq + g * a.Gq + hh % a.Gq;
      a.out[row * 128 + c] = val;
      // ln sum exp(scaled score) = ln 2 * (M + log2 L), the scores being in log2 units
      if (a.lse && c == 0) a.lse[row] = (Lt > 0.f) ? 0.6931471805599453f * (Mx + log2f(Lt)) : kNegInf;
    } else {
      a.out[((size_t)b * a.Hq + g * G + hh) * 128 + c] = val;
    }
  }
  } else {
  // ---- back to the original basis once, on the tensor cores:
  // o_hist[h][c] = sum_i o'[h][i] R_v^T[i][c].  Each head's merged o' is
  // normalised by its l and scaled by a power of two that puts its largest
  // component near 2^10, so that the fp16 hi + lo terms of rotate_q keep about
  // 22 bits of every component; the scale is taken out afterwards ----
  constexpr int HP = S::HP;
  float* sx = reinterpret_cast<float*>(smb + S::sx);
  float* sy = reinterpret_cast<float*>(smb + S::sy);
  unsigned* smax = reinterpret_cast<unsigned*>(smb + S::smax);
  float* sinv = reinterpret_cast<float*>(smb + S::sinv);
  float* hist_m = reinterpret_cast<float*>(smb + S::hist_m);
  float* hist_l = reinterpret_cast<float*>(smb + S::hist_l);
  if (threadIdx.x < HP) smax[threadIdx.x] = 0u;
  for (int idx = G * 128 + threadIdx.x; idx < HP * 128; idx += NW * 32)   // padded rows
    sx[(idx >> 7) * kQStride + (idx & 127) + 4 * ((idx & 127) >> 5)] = 0.f;
  __syncthreads();
  float ov[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int idx = threadIdx.x + e * NW * 32;
    ov[e] = 0.f;
    if (idx < G * 128) {
      ov[e] = (L[e] > 0.f) ? O[e] / L[e] : 0.f;
      atomicMax(smax + (idx >> 7), __float_as_uint(fabsf(ov[e])));   // order-free: a maximum
      if ((idx & 127) == 0) {
        hist_m[idx >> 7] = M[e];
        hist_l[idx >> 7] = L[e];
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int idx = threadIdx.x + e * NW * 32;
    if (idx < G * 128) {
      const int hh = idx >> 7, c = idx & 127;
      const uint32_t mb = smax[hh];
      // 2^(10 - exponent of the largest component); 1 for an all-zero (or non-finite) row
      const int ex = (int)((mb >> 23) & 0xFFu) - 127;
      const float scale = (mb == 0u || ex > 127) ? 1.0f : ldexpf(1.0f, 10 - max(ex, -100));
      sx[hh * kQStride + c + 4 * (c >> 5)] = ov[e] * scale;
      if (c == 0) sinv[hh] = 1.0f / scale;
    }
  }
  __syncthreads();
  rotate_q<HP, NW>(sx, rvf, sy);   // ends with a barrier
  for (int idx = threadIdx.x; idx < G * 128; idx += NW * 32) {
    const int hh = idx >> 7, c = idx & 127;
    const float Mh = hist_m[hh], Lh = hist_l[hh], mt = tier_m[hh], lt = tier_l[hh];
    const float oh = sy[hh * kQrStride + c] * sinv[hh] * Lh;   // the unnormalised rotated sum
    const float Mx = fmaxf(Mh, mt);
    const float fh = (Mh == kNegInf) ? 0.f : exp2f(Mh - Mx);
    const float ft = (mt == kNegInf) ? 0.f : exp2f(mt - Mx);
    const float Lt = fmaf(Lh, fh, lt * ft);
    const float val = (Lt > 0.f) ? fmaf(oh, fh, tier_o[idx] * ft) / Lt : 0.f;
    if constexpr (kMulti) {
      const size_t row = ((size_t)b * a.T + hh / a.Gq) * a.Hq + g * a.Gq + hh % a.Gq;
      a.out[row * 128 + c] = val;
      // ln sum exp(scaled score) = ln 2 * (M + log2 L), the scores being in log2 units
      if (a.lse && c == 0) a.lse[row] = (Lt > 0.f) ? 0.6931471805599453f * (Mx + log2f(Lt)) : kNegInf;
    } else {
      a.out[((size_t)b * a.Hq + g * G + hh) * 128 + c] = val;
    }
  }
  }
  __syncthreads();
  if (threadIdx.x < kMaskWords) mask[threadIdx.x] = 0u;   // ready for the next call
  if (G <= 4 && threadIdx.x == 0) mbar_inval(rbar);
}

template <int G, int GS, bool kMulti>
__global__ void __launch_bounds__(int2_warps(G) * 32, 1) decode_int2_kernel(DecodeArgs a) {
  extern __shared__ float4 smem4[];
  uint8_t* smb = reinterpret_cast<uint8_t*>(smem4);
  // launch order: every history split first, split-major (every pair's first
  // split, then every pair's second, ..: the longest work goes first on grids
  // of several waves), then the tier CTAs, which wait for the history splits of
  // their pair (earlier in launch order) and merge them
  const int lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  const int n_hist = a.n_split * gridDim.y * gridDim.z;
  // the next kernel may start its own prologue as SMs free up; it waits for
  // this grid before it reads anything this grid writes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (lin < n_hist) {
    const int n_pairs = gridDim.y * gridDim.z;
    const int split = lin / n_pairs, pair = lin % n_pairs;   // split-major: every pair's first split first
    const int g = pair % a.Hkv, b = pair / a.Hkv;
    float* part = a.ws + ((size_t)pair * a.n_split + split) * G * kPart;
    int2_history<G, GS, kMulti>(a, b, g, split, smb, part);
    __syncthreads();   // the partial is written before the release below
    if (threadIdx.x == 0) {
      unsigned* m = a.arrive + (size_t)pair * kMaskWords + (split >> 5);
      asm volatile("red.release.gpu.global.or.b32 [%0], %1;" ::"l"(m), "r"(1u << (split & 31)) : "memory");
    }
  } else {
    const int pair = lin - n_hist;
    tier_merge<G, GS, kMulti>(a, pair / a.Hkv, pair % a.Hkv, smb);
  }
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

// A warp's ring stage holds one 16-token tile of K and of V: four TMA boxes of
// 16 rows x 64 channels (2 KB each, 128-byte swizzle: the 16-byte chunk c of
// row r sits at chunk position c ^ (r % 8), so the ldmatrix reads below are
// conflict-free): [K 0-63][K 64-127][V 0-63][V 64-127].
constexpr int kBfStages = 3;
constexpr int kBfStage = 8192;

template <int G>
struct BfLay {
  static constexpr int NW = kBf16Warps;
  static constexpr int ring = 0;                                  // [NW][kBfStages][kBfStage]
  static constexpr int bars = ring + NW * kBfStages * kBfStage;   // [NW][kBfStages] mbarriers
  static constexpr int spid = bars + NW * kBfStages * 8;          // [kMaxPids] page ids
  static constexpr int total = spid + kMaxPids * 4 + 1024;        // + slack to align the ring to 1 KB
  // after the loop, over the ring: per-warp results, then the final merge
  static constexpr int swo = 0;                                   // [NW][G][128]
  static constexpr int swm = swo + NW * G * 128 * 4;              // [NW][G]
  static constexpr int swl = swm + NW * G * 4;                    // [NW][G]
  static_assert(swl + NW * G * 4 <= bars, "warp results fit in the ring");
  static_assert((16 + 2 * NW * 128 + 2 * kMaxParts * G) * 4 <= bars, "the final merge fits in the ring");
};

// Plain split-K attention over the all-BF16 pool.  Each warp streams its
// 16-token tiles of K and V by TMA through a ring in shared memory; QK runs
// on the tensor cores with q exact in bf16 (B column 2h holds head h, column
// 2h + 1 is zero), PV with the softmax weights as bf16 hi + lo (about 16
// significant bits) in columns 2h and 2h + 1; online softmax per head as in
// the INT2 loop.  The splits merge with the log-sum-exp rule in the CTA that
// takes the last ticket.
template <int G>
__global__ void __launch_bounds__(kBf16Warps * 32, 1)
    decode_bf16_kernel(DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap) {
  constexpr int NW = kBf16Warps;
  constexpr int NT = (G <= 4) ? 1 : 2;   // 8-column n-tiles: 4 heads each
  using S = BfLay<G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smb = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  float* sm = reinterpret_cast<float*>(smb);
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, j = lane & 3;
  const int nparts = a.n_split;
  float* part = a.ws + ((size_t)(b * a.Hkv + g) * nparts + split) * G * kPart;
  // programmatic dependent launch: let the next kernel start its prologue, and
  // wait for the preceding one before reading any input
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int n = a.seq_len[b];
  const int cap = min(a.max_pages * a.page_size, a.max_len);
  if (n < 0 || n > cap) {
    if (threadIdx.x == 0) flag_error(a.err, KV_DEVERR_LENGTH);
    n = max(0, min(n, cap));
  }
  const int ntiles = (n + kTile - 1) / kTile;
  const int t_begin = split * a.per_split, t_end = min(ntiles, t_begin + a.per_split);
  if (t_begin >= t_end) {
    write_empty_partial<G, NW>(part);
  } else {
    uint8_t* ring = smb + S::ring + (size_t)warp * kBfStages * kBfStage;
    uint64_t* wbar = reinterpret_cast<uint64_t*>(smb + S::bars) + warp * kBfStages;
    int* spid = reinterpret_cast<int*>(smb + S::spid);
    if (lane < kBfStages) mbar_init(wbar + lane, 1);
    mbar_fence_init();
    const int tpp = a.page_size / kTile;   // tiles per page
    const int p_begin = t_begin / tpp, p_count = (t_end - 1) / tpp + 1 - p_begin;
    const int32_t* ptrow = a.pt + (size_t)b * a.max_pages;
    for (int i = threadIdx.x; i < p_count; i += NW * 32) spid[i] = __ldg(ptrow + p_begin + i);
    // QK B fragments straight from q (bf16 bits): column n = r of n-tile u is head 4u + r/2 when r is even
    uint32_t qf[8][NT][2];
    {
      const int hh = r >> 1;
#pragma unroll
      for (int u = 0; u < NT; ++u) {
        const int head = 4 * u + hh;
        const bool live = !(r & 1) && head < G;
        const uint32_t* qrow =
            reinterpret_cast<const uint32_t*>(a.q + ((size_t)b * a.Hq + g * G + (live ? head : 0)) * 128);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          qf[s][u][0] = live ? __ldg(qrow + 8 * s + j) : 0u;       // channels 16s + 2j, +1
          qf[s][u][1] = live ? __ldg(qrow + 8 * s + 4 + j) : 0u;   // channels 16s + 2j + 8, +9
        }
      }
    }
    __syncthreads();   // page ids in shared memory, barriers initialised
    // tile t -> its 16 rows of the pool, viewed as [num_pages * Hkv * page_size][128];
    // a bad page id reads page 0 and its tokens are masked
    auto tile_row = [&](int t, bool& valid) -> int {
      const int pid = spid[t / tpp - p_begin];
      valid = pid >= 0 && pid < a.num_pages;
      return (int)(((long long)(valid ? pid : 0) * a.Hkv + g) * a.page_size + (t % tpp) * kTile);
    };
    auto issue = [&](int t, int st) {
      if (t < t_end && lane == 0) {
        bool valid;
        const int row = tile_row(t, valid);
        const uint32_t dst = smem_u32(ring + st * kBfStage);
        mbar_expect_tx(wbar + st, kBfStage);
        tma_load_2d(dst, &kmap, 0, row, wbar + st);
        tma_load_2d(dst + 2048, &kmap, 64, row, wbar + st);
        tma_load_2d(dst + 4096, &vmap, 0, row, wbar + st);
        tma_load_2d(dst + 6144, &vmap, 64, row, wbar + st);
      }
    };
#pragma unroll
    for (int st = 0; st < kBfStages - 1; ++st) issue(t_begin + warp + NW * st, st);
    int issued = min(kBfStages - 1, (t_end - t_begin - warp + NW - 1) / NW);

    float m_run[NT], base[NT], l_run[NT], oacc[8][NT][4];
#pragma unroll
    for (int u = 0; u < NT; ++u) {
      m_run[u] = kNegInf;
      base[u] = 0.f;
      l_run[u] = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) oacc[i][u][0] = oacc[i][u][1] = oacc[i][u][2] = oacc[i][u][3] = 0.f;
    }
    // ldmatrix row / chunk of this lane: K (A of QK): row lane%16, chunk + lane/16;
    // V (A of PV, transposed): row lane%8 + 8 (lane/16), chunk + (lane/8)%2
    const int krow = lane & 15, kc = lane >> 4;
    const int vrow = (lane & 7) + 8 * (lane >> 4), vc = (lane >> 3) & 1;
    int k = 0;
    bool ok = true;
    for (int t = t_begin + warp; t < t_end; t += NW, ++k) {
      __syncwarp();   // every lane is done with the stage refilled next
      issue(t + NW * (kBfStages - 1), (k + kBfStages - 1) % kBfStages);
      if (t + NW * (kBfStages - 1) < t_end) ++issued;
      const int st = k % kBfStages;
      if (!__all_sync(0xffffffffu, mbar_wait(wbar + st, (k / kBfStages) & 1, a.wait_polls))) {
        ok = false;
        break;
      }
      const uint32_t sbase = smem_u32(ring + st * kBfStage);
      bool valid;
      tile_row(t, valid);
      const int lim = valid ? n - t * kTile : 0;
      const bool v0 = r < lim, v1 = r + 8 < lim;
      if (lim < kTile) {
        // V rows past the sequence (or of a bad page) are zeroed, so that a weight of
        // zero never meets a stale non-finite value; the fence orders these writes
        // before the stage's next copy
        for (int idx = lane + 16 * max(lim, 0); idx < 16 * kTile; idx += 32) {
          const int row = idx >> 4, c = idx & 15;
          *reinterpret_cast<uint4*>(ring + st * kBfStage + 4096 + (c >> 3) * 2048 + row * 128 + (c & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      // ---- QK ----
      float sacc[NT][4];
#pragma unroll
      for (int u = 0; u < NT; ++u) sacc[u][0] = sacc[u][1] = sacc[u][2] = sacc[u][3] = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int c = 2 * (s & 3) + kc;
        uint32_t fa[4];
        ldmatrix_x4(sbase + (s >> 2) * 2048 + krow * 128 + ((c ^ (krow & 7)) << 4), fa);
#pragma unroll
        for (int u = 0; u < NT; ++u) mma_bf16(sacc[u], fa[0], fa[1], fa[2], fa[3], qf[s][u][0], qf[s][u][1]);
      }
      // ---- softmax (column 2j: head 4u + j; column 2j + 1 is zero) and PV B fragments ----
      uint32_t bpv[NT][2];
#pragma unroll
      for (int u = 0; u < NT; ++u) {
        const float l0 = v0 ? sacc[u][0] * a.scale_log2 : kNegInf;
        const float l1 = v1 ? sacc[u][2] * a.scale_log2 : kNegInf;
        if (__any_sync(0xffffffffu, fmaxf(l0, l1) > m_run[u])) {
          float tmax = fmaxf(l0, l1);
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
          const bool need = tmax > m_run[u];
          const float mnew = need ? tmax + kSlack : m_run[u];
          const float alpha = need ? ((m_run[u] == kNegInf) ? 0.f : exp2_neg(m_run[u] - mnew)) : 1.f;
          m_run[u] = mnew;
          base[u] = (mnew == kNegInf) ? 0.f : mnew;
          l_run[u] *= alpha;
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[i][u][e] *= alpha;
        }
        const float p0 = exp2_neg(l0 - base[u]), p1 = exp2_neg(l1 - base[u]);
        l_run[u] += p0 + p1;
        bpv[u][0] = movmatrix_t(split_hi_lo_bf16(p0));
        bpv[u][1] = movmatrix_t(split_hi_lo_bf16(p1));
      }
      // ---- PV: value accumulator [channel][column] ----
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = 2 * (i & 3) + vc;
        uint32_t fa[4];
        ldmatrix_x4_t(sbase + 4096 + (i >> 2) * 2048 + vrow * 128 + ((c ^ (vrow & 7)) << 4), fa);
#pragma unroll
        for (int u = 0; u < NT; ++u) mma_bf16(oacc[i][u], fa[0], fa[1], fa[2], fa[3], bpv[u][0], bpv[u][1]);
      }
    }
    if (!ok) {   // a copy did not arrive in time: wait (bounded) for the ones in flight
      if (lane == 0) flag_error(a.err, KV_DEVERR_TIMEOUT);
      for (int kk = k; kk < issued; ++kk) mbar_wait(wbar + kk % kBfStages, (kk / kBfStages) & 1, a.wait_polls);
    }
    ok = __syncthreads_and(ok);   // the ring is free before the results reuse it
    if (lane < kBfStages) mbar_inval(wbar + lane);
    if (!ok) {
      write_empty_partial<G, NW>(part);
    } else {
      float* swo = reinterpret_cast<float*>(smb + S::swo);
      float* swm = reinterpret_cast<float*>(smb + S::swm);
      float* swl = reinterpret_cast<float*>(smb + S::swl);
#pragma unroll
      for (int u = 0; u < NT; ++u) {
        const float l = warp_sum_xor(l_run[u], 4);
        const int hh = 4 * u + j;
        if (hh < G) {
          float* o = swo + (warp * G + hh) * 128;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[16 * i + r] = oacc[i][u][0] + oacc[i][u][1];          // hi + lo columns
            o[16 * i + r + 8] = oacc[i][u][2] + oacc[i][u][3];
          }
          if (r == 0) {
            swm[warp * G + hh] = m_run[u];
            swl[warp * G + hh] = l;
          }
        }
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < G * 128; idx += NW * 32) {
        const int hh = idx >> 7, c = idx & 127;
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, swm[w * G + hh]);
        float L = 0.f, O = 0.f;
        if (M != kNegInf) {
#pragma unroll
          for (int w = 0; w < NW; ++w) {
            const float mw = swm[w * G + hh];
            const float f = (mw == kNegInf) ? 0.f : exp2f(mw - M);
            L = fmaf(f, swl[w * G + hh], L);
            O = fmaf(f, swo[(w * G + hh) * 128 + c], O);
          }
        }
        part[hh * kPart + 4 + c] = O;
        if (c == 0) {
          part[hh * kPart + 0] = M;
          part[hh * kPart + 1] = L;
        }
      }
    }
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

template <int G>
constexpr size_t bf16_smem() {
  return BfLay<G>::total;
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

// A grid of one wave forms q' in every history CTA (one launch); a grid of
// several waves gets q' from the pre-pass, once per (sequence, KV head), and
// the decode kernel is launched as its programmatic dependent.
template <int G, int GS, bool kMulti>
cudaError_t launch_int2_t(DecodeArgs a, int B, int sm_count, cudaStream_t s) {
  const int per_sm = int2_blocks_per_sm<G, GS, kMulti>();
  if (per_sm < 0) return cudaErrorInvalidConfiguration;
  const long long ctas = (long long)(a.n_split + 1) * a.Hkv * B;
  const bool multi_wave = ctas > (long long)per_sm * sm_count;
  a.qmode = multi_wave ? kQPre : kQLocal;
  if (multi_wave) {   // the pre-pass starts after the preceding kernel; the decode overlaps it
    constexpr int SPB = 16 / ((G <= 4) ? 4 : 8);   // sequences per pre-pass CTA
    qprep_kernel<G, GS, kMulti><<<dim3(a.Hkv, (B + SPB - 1) / SPB), 256, 0, s>>>(a, B);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // programmatic dependent launch: the CTAs may start while the preceding
  // kernel finishes; they wait for it (griddepcontrol.wait) before reading
  // any input the caller passes
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_split + 1, a.Hkv, B);
  cfg.blockDim = dim3(int2_warps(G) * 32);
  cfg.dynamicSmemBytes = int2_smem<G, GS>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_int2_kernel<G, GS, kMulti>, a);
}

template <int G>
cudaError_t launch_bf16_t(const DecodeArgs& a, int B, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t s) {
  if (bf16_blocks_per_sm<G>() < 0) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_split, a.Hkv, B);
  cfg.blockDim = dim3(kBf16Warps * 32);
  cfg.dynamicSmemBytes = bf16_smem<G>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_bf16_kernel<G>, a, kmap, vmap);
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
  a.merge_polls = kMergePolls;
  a.arrive = p.arrive + (size_t)layer * p.cfg.max_seqs * p.cfg.num_kv_heads * kMaskWords;
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
                            int per_sm, int min_per = 1) {
  DecodePlan pl;
  const int pairs = B * p.cfg.num_kv_heads;
  const int slots = max(1, per_sm) * p.sm_count;
  const int u = max(units, 1);
  int ns = slots / pairs - n_extra;
  ns = max(1, min(ns, u));
  int per = (u + ns - 1) / ns;
  per = max(per, min_per);   // short histories: fewer, fuller splits (less to merge)
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
  const int per_sm = (T > 1) ? int2_occupancy_t<true>(p, G) : int2_occupancy_t<false>(p, G);
  // one tier CTA per (sequence, KV head) beside the history splits; partials
  // are kept for the history splits only, followed by the q' fragments
  DecodePlan pl = make_plan(p, G, B, tiles, int2_max_tiles_per_warp(G) * int2_warps(G), 1, per_sm, int2_warps(G));
  const size_t pairs = (size_t)B * p.cfg.num_kv_heads;
  pl.partial_floats = pairs * pl.n_split * G * kPart;
  const size_t qwords = pairs * 32 * (G <= 4 ? qfrag_words<4>() : qfrag_words<8>());
  pl.bytes = pl.partial_floats * sizeof(float) + qwords * sizeof(uint32_t);
  pl.max_len = max(max_hist_len, 0);
  return pl;
}

DecodePlan plan_decode_bf16(const Pool& p, int B, int max_len) {
  // splits in 16-token tiles, at most 64 tiles per warp
  const int tiles = (max(max_len, 0) + kTile - 1) / kTile;
  DecodePlan pl = make_plan(p, p.G, B, tiles, 64 * kBf16Warps, 0, bf16_occupancy(p));
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
  a.qfrag = reinterpret_cast<uint32_t*>(a.ws + plan.partial_floats);
  if (plan.tiles_per_split > kMaxPids - 8) return cudaErrorInvalidValue;   // page ids staged per CTA
  const bool g64 = p.cfg.group_size == 64;
  if (T > 1 || lse) {   // several queries per sequence, or the log-sum-exp wanted
    switch (T * p.G) {
      case 1: return g64 ? launch_int2_t<1, 64, true>(a, B, p.sm_count, s) : launch_int2_t<1, 128, true>(a, B, p.sm_count, s);
      case 2: return g64 ? launch_int2_t<2, 64, true>(a, B, p.sm_count, s) : launch_int2_t<2, 128, true>(a, B, p.sm_count, s);
      case 4: return g64 ? launch_int2_t<4, 64, true>(a, B, p.sm_count, s) : launch_int2_t<4, 128, true>(a, B, p.sm_count, s);
      case 8: return g64 ? launch_int2_t<8, 64, true>(a, B, p.sm_count, s) : launch_int2_t<8, 128, true>(a, B, p.sm_count, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (p.G) {
    case 1: return g64 ? launch_int2_t<1, 64, false>(a, B, p.sm_count, s) : launch_int2_t<1, 128, false>(a, B, p.sm_count, s);
    case 2: return g64 ? launch_int2_t<2, 64, false>(a, B, p.sm_count, s) : launch_int2_t<2, 128, false>(a, B, p.sm_count, s);
    case 4: return g64 ? launch_int2_t<4, 64, false>(a, B, p.sm_count, s) : launch_int2_t<4, 128, false>(a, B, p.sm_count, s);
    case 8: return g64 ? launch_int2_t<8, 64, false>(a, B, p.sm_count, s) : launch_int2_t<8, 128, false>(a, B, p.sm_count, s);
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
  if (plan.tiles_per_split > kMaxPids - 8) return cudaErrorInvalidValue;   // page ids staged per CTA
  // K and V of the layer viewed as [num_pages * Hkv * page_size rows][128] bf16,
  // boxes of 16 rows x 64 channels with the 128-byte swizzle
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
  if (!encode) return cudaErrorNotSupported;
  const unsigned long long rows = (unsigned long long)p.cfg.num_pages * p.cfg.num_kv_heads * p.cfg.page_size;
  if (rows >= (1ull << 31)) return cudaErrorInvalidValue;   // row coordinates are 32-bit
  CUtensorMap maps[2];
  const uint16_t* bases[2] = {a.bk, a.bv};
  for (int t = 0; t < 2; ++t) {
    const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {256};
    const cuuint32_t box[2] = {64, (cuuint32_t)kTile};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&maps[t], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(bases[t]), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  switch (p.G) {
    case 1: return launch_bf16_t<1>(a, B, maps[0], maps[1], s);
    case 2: return launch_bf16_t<2>(a, B, maps[0], maps[1], s);
    case 4: return launch_bf16_t<4>(a, B, maps[0], maps[1], s);
    case 8: return launch_bf16_t<8>(a, B, maps[0], maps[1], s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvint2
