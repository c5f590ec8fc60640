// INT2 append on the 5th-generation tensor cores, in bulk (kv_append_quantize)
// and per decode step (kv_append_step): rotate -> clip -> asymmetric INT2
// quantize -> pack into the paged tiles.  Both run the same MMA and the same
// epilogue arithmetic (row_codes), so a token gets the same codes on either
// path.
//
// Method: yunpan.plus OSCAR write-up, "2. 在线量化与反量化" (a token leaving
// the recent window is rotated, clipped, quantized and packed, four 2-bit
// codes per byte, into the INT2 history); gist.science OSCAR explainer,
// section 2.2 B (history is stored after the fixed rotation and the clip).
//
// GPU design: the rotation x' = x R of a chunk of 128 tokens of one KV head
// and one tensor is x [128 x 128] . R_hi + x . R_lo, both terms accumulated
// into one fp32 accumulator (R enters as bf16 hi and lo terms; x is exact in
// bf16).  The bulk append runs one CTA per SM on one (KV head, tensor): two
// teams of eight epilogue warps take the CTA's 128-token chunks in turn, and
// four serving warps feed them:
//   * per team a loader thread walks the tasks and starts each chunk's x load
//     as soon as one of four buffers is free: two TMA tile loads (128-byte
//     swizzle, the K-major operand layout) when the whole chunk lies inside
//     the input, else 16-byte cp.async by the loader's warp with rows outside
//     the append range zero-filled.  R^T hi | lo arrives once per CTA,
//     pre-swizzled in global memory by the rotation set-up, as four bulk
//     copies;
//   * per team an issuer thread starts sixteen tcgen05.mma (kind::f16, M 128,
//     N 128, K 16: per 16-channel step the hi term, then the lo term) into
//     one of four 128-column fp32 accumulators in tensor memory (all 512
//     columns) and commits them to an mbarrier;
//   * every thread of a team owns one token row and one half of the channels
//     of the accumulator (tcgen05.ld; warps w and w + 4 of a team share a
//     lane quarter): clip, per-group min / max (combined across the halves
//     through shared memory for group 128), s and z, the codes (branch-free,
//     with a rare exact fix-up); the codes are packed into the tile's storage
//     order with warp shuffles (partners differ in lane bits 0 and 3) and
//     written as 8-byte word pairs, merging with the bits of rows outside the
//     append range where a tile is only partly written.
// The per-step eviction runs the same product and epilogue on one chunk per
// CTA, two CTAs per SM.
// Every wait is bounded; a wait that runs out sets KV_DEVERR_TIMEOUT, waits
// (bounded) for the work in flight, frees the tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kv_device.cuh"
#include "kv_internal.h"

namespace kvint2 {

namespace {

constexpr int kTcThreads = 256;
constexpr int kChunk = 128;                  // tokens per MMA (the M of one tcgen05.mma)
constexpr int kTilesPerChunk = kChunk / kTile;
constexpr int kTcCols = 128;                 // tensor-memory columns: the fp32 accumulator
constexpr uint32_t kABytes = kChunk * 256;   // x chunk: 128 rows x 128 bf16
constexpr uint32_t kBBytes = 256 * 256;      // R^T hi | lo: 256 rows x 128 bf16
constexpr int kTcPolls = 1 << 20;

// dynamic shared memory carve-up (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kABytes;
constexpr uint32_t kOffClip = kOffB + kBBytes;
constexpr uint32_t kOffStat = kOffClip + 128 * 4;
constexpr uint32_t kOffBar = kOffStat + 2 * 128 * 8;
constexpr uint32_t kOffTmem = kOffBar + 24;

// ---- tcgen05 / descriptor helpers -------------------------------------------
// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzle
// layout: rows of 128 bytes, 8-row atoms of 1024 bytes (stride-dimension byte
// offset 1024; the leading-dimension offset is unused for this layout),
// descriptor version 1, layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// N = 128, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(128 >> 3) << 17) |
                            ((uint32_t)(128 >> 4) << 24);

__device__ __forceinline__ void tc_alloc(uint32_t slot_saddr, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar_saddr) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar_saddr)
               : "memory");
}
// 32 consecutive fp32 columns of this thread's accumulator row
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]),
        "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]),
        "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
// 32 consecutive fp32 columns of this thread's accumulator row, written back
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// generic-proxy shared-memory writes -> visible to the tensor cores
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 16-byte copy global -> shared, zero-filled when !valid (no bytes read)
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

// one TMA tile load (box 64 channels x 1 head x 128 rows, 128-byte swizzle)
// of the x tensor map at (channel c0, head c1, row c2) into shared memory,
// completing on `bar`; rows outside the map read as zero
__device__ __forceinline__ void tma_load_x(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                           uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// 8-byte store of two words of a stored-tile slot, merged with the existing
// bits outside `mask` unless every bit is new
__device__ __forceinline__ void store_merge2(uint8_t* dst, const uint32_t (&w)[2], uint32_t mask) {
  uint2* p = reinterpret_cast<uint2*>(dst);
  if (mask == 0xFFFFFFFFu) {
    *p = make_uint2(w[0], w[1]);
  } else if (mask != 0u) {
    const uint2 o = *p;
    *p = make_uint2((o.x & ~mask) | (w[0] & mask), (o.y & ~mask) | (w[1] & mask));
  }
}

struct TcArgs {
  uint8_t* hist;              // layer base
  size_t page_bytes, head_block;
  int tile_bytes, P;
  const uint16_t* x[2];       // K and V inputs [T][Hkv][128] bf16
  const int32_t* cu;
  const int32_t* hist_start;
  const int32_t* pt;
  int max_pages, n_seqs, max_chunks, Hkv;
  long long num_pages;
  long long map_rows;         // row extent of the x tensor maps (n_seqs * max_tokens)
  const uint4* rfrag;         // layer base [Hkv][kFragBlocks][4096]
  const float* clip;          // layer base [2][Hkv][128]
  int* err;
  int tasks_per_cta;
  int wait_polls;             // bound of the bulk append's waits between its warps
  int stall_first_load;       // test hook: CTA (0, 0) never starts the x load of its first chunk
};

// Chunk of one task: 128 consecutive history positions [P0, P0 + 128) of
// sequence b (P0 a multiple of 16); `live` is false when the task has no work.
struct Chunk {
  int b, c0, nb, h0, first, last, P0;
  bool live;
};

// Walks the tasks [t, t1) of a CTA in order without divisions: the sequence
// index and the chunk index within it advance together, and a sequence's
// range (cu, hist_start) is read once, when the walk enters it.  Errors of a
// sequence (a negative or out-of-range span, more chunks than the grid covers)
// are reported by the thread that walks into its first chunk with `flag` set.
struct TaskCursor {
  int t, t1, b, ci;
  int c0, nb, h0, first, last;
  bool seq_ok;
  __device__ void enter(const TcArgs& a, bool flag) {   // the sequence of task t
    c0 = __ldg(a.cu + b);
    nb = __ldg(a.cu + b + 1) - c0;
    h0 = __ldg(a.hist_start + b);
    seq_ok = false;
    if (nb <= 0) {
      if (flag && nb < 0 && ci == 0) flag_error(a.err, KV_DEVERR_SEQ_RANGE);
      return;
    }
    if (h0 < 0 || (long long)h0 + nb > (long long)a.max_pages * a.P) {
      if (flag && ci == 0) flag_error(a.err, KV_DEVERR_SEQ_RANGE);
      return;
    }
    first = h0 / kTile;
    last = (h0 + nb - 1) / kTile;
    if (flag && ci == 0 && (last - first) / kTilesPerChunk + 1 > a.max_chunks) flag_error(a.err, KV_DEVERR_LENGTH);
    seq_ok = true;
  }
  __device__ void start(const TcArgs& a, int t0, int t_end, bool flag) {
    t = t0;
    t1 = t_end;
    b = t0 / a.max_chunks;
    ci = t0 - b * a.max_chunks;
    if (t < t1) enter(a, flag);
  }
  __device__ bool live() const { return seq_ok && (first + ci * kTilesPerChunk) <= last; }
  __device__ void step(const TcArgs& a, bool flag) {
    ++t;
    if (++ci == a.max_chunks) {
      ci = 0;
      ++b;
      if (t < t1) enter(a, flag);
    }
  }
  __device__ void next_live(const TcArgs& a, bool flag) {   // from the current task on
    while (t < t1 && !live()) step(a, flag);
  }
  __device__ Chunk chunk() const {
    Chunk k;
    k.b = b;
    k.c0 = c0;
    k.nb = nb;
    k.h0 = h0;
    k.first = first;
    k.last = last;
    k.P0 = (first + ci * kTilesPerChunk) * kTile;
    k.live = live();
    return k;
  }
};

// x rows of a chunk -> the swizzled A operand: thread t (0 .. 255) copies half a
// row (row t % 128, channels 64 * (t / 128) ..); rows outside the append range are zero
__device__ __forceinline__ void load_chunk(const TcArgs& a, const uint16_t* X, int g, const Chunk& k,
                                           uint32_t sA, int t) {
  const int row = t & 127, hf = t >> 7;
  const int pos = k.P0 + row;
  const bool ok = pos >= k.h0 && pos < k.h0 + k.nb;
  const uint16_t* src = X + ((size_t)(ok ? k.c0 + (pos - k.h0) : 0) * a.Hkv + g) * 128 + 64 * hf;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    cp_async16_zfill(sA + hf * 16384 + row * 128 + ((c ^ (row & 7)) << 4), src + 8 * c, ok);
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// x' = x . R_hi + x . R_lo for a 128-row chunk on the tensor cores: per
// 16-channel step the hi term, then the lo term, into the 128-column fp32
// accumulator at tmem; completion arrives on `bar`.  One thread issues.
__device__ __forceinline__ void issue_rotation(uint32_t tmem, uint32_t sA, uint32_t sB, uint64_t* bar) {
  tc_fence_after();
  // descriptors of the later steps: the start-address field (address / 16,
  // 14 bits) of the first plus the step's byte offset / 16 (the operands lie
  // below 256 KB, so the field does not carry)
  const uint64_t ad0 = sw128_desc(sA), bd0 = sw128_desc(sB);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t koff = (ks & 3) * 32;   // 16 channels = 32 bytes into the swizzled row
    const uint64_t ad = ad0 + (((ks >> 2) * 16384 + koff) >> 4);
    const uint64_t bd = bd0 + (((ks >> 2) * 32768 + koff) >> 4);   // rows 0-127: hi; 128-255: lo
    tc_mma(tmem, ad, bd, kIdesc, ks > 0 ? 1u : 0u);
    tc_mma(tmem, ad, bd + (16384 >> 4), kIdesc, 1u);
  }
  tc_commit(smem_u32(bar));
}

// Pairs of fp32 values in one 64-bit register for the paired fp32 arithmetic
// of sm_100 and later (add / sub / fma .f32x2: one instruction for two
// values, each rounded exactly as the scalar instruction rounds it).
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// the exact code of one value (the rare fix-up path; kept out of line)
__device__ __noinline__ uint32_t quant_code_exact(float y, ScaleZero q) { return quant_code(y, q); }

// Three-input minimum / maximum (one instruction on sm_100 and later); exact,
// so reductions built from them give the same value in any order (up to the
// sign of a zero, which the quantizer canonicalises).
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// min / max of acc and 32 values: two independent chains of 3-input steps
__device__ __forceinline__ float min_of32(float acc, const float (&v)[32]) {
  float c0 = v[0], c1 = v[1];
#pragma unroll
  for (int i = 2; i < 30; i += 4) {
    c0 = min3f(c0, v[i], v[i + 1]);
    c1 = min3f(c1, v[i + 2], v[i + 3]);
  }
  c0 = min3f(c0, v[30], v[31]);
  return min3f(acc, c0, c1);
}
__device__ __forceinline__ float max_of32(float acc, const float (&v)[32]) {
  float c0 = v[0], c1 = v[1];
#pragma unroll
  for (int i = 2; i < 30; i += 4) {
    c0 = max3f(c0, v[i], v[i + 1]);
    c1 = max3f(c1, v[i + 2], v[i + 3]);
  }
  c0 = max3f(c0, v[30], v[31]);
  return max3f(acc, c0, c1);
}

// The codes of one accumulator row (token row m; channels 64 hf .. 64 hf + 63)
// after clipping, with s and z from the group's range: x' read from tensor
// memory (lanes of this warp's quarter, address trow), the range first and then
// the codes (the accumulator is read again rather than held in registers),
// reductions as trees to keep the dependency chains short.  Codes go into the
// storage words of this channel half (words 2 hf and 2 hf + 1 of each slot; K:
// slot (k % 8) / 2 of the token's four, V: slot c % 8 of the token's eight,
// k = c % 16) at the bit positions of token row 0 of a tile (K) or of tile
// token 0 (V); the caller shifts them to the row's own positions.  Both warps
// of a lane quarter (w and w + 4) call this together: group 128 combines their
// two halves through shared memory behind named barrier `qbar`, of those 64
// threads.
template <int GS, int TENSOR, int NS>
__device__ __forceinline__ ScaleZero row_codes(uint32_t trow, int hf, int m, const float* sclip,
                                               const float* sclipmin, float2* sstat, uint32_t (&wd)[NS][2],
                                               int qbar) {
  // first pass: x' clipped and its range, per block of 32 channels.  The
  // block's range is taken on x' first: when no lane of the warp has a value
  // of magnitude above the block's smallest clip (sclipmin, null: always
  // clip), no value of the block is clipped, x' in tensor memory already is
  // the clipped value and that range is the clipped range; otherwise the
  // block is clipped, written back in place (the second pass reads the
  // clipped values) and its range taken again
  auto rotated32 = [&](int cb, float (&v)[32]) {
    uint32_t u[32];
    tc_ld32(trow + 64 * hf + 32 * cb, u);
    tc_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(u[i]);
  };
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int cb = 0; cb < 2; ++cb) {
    float v[32];
    rotated32(cb, v);
    float bmn = min_of32(INFINITY, v), bmx = max_of32(-INFINITY, v);
    const float cmin = sclipmin ? sclipmin[2 * hf + cb] : -1.0f;
    if (__any_sync(0xffffffffu, !(fmaxf(bmx, -bmn) <= cmin))) {   // warp-uniform: the store is collective
      uint32_t u[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] = clip_to(v[i], sclip[64 * hf + 32 * cb + i]);
        u[i] = __float_as_uint(v[i]);
      }
      tc_st32(trow + 64 * hf + 32 * cb, u);
      bmn = min_of32(INFINITY, v);
      bmx = max_of32(-INFINITY, v);
    }
    mn = fminf(mn, bmn);
    mx = fmaxf(mx, bmx);
  }
  if (GS == 128) {   // the group spans both channel halves: combine with warp w ^ 4
    sstat[hf * 128 + m] = make_float2(mn, mx);
    asm volatile("bar.sync %0, 64;" ::"r"(qbar) : "memory");
    const float2 o = sstat[(hf ^ 1) * 128 + m];
    mn = fminf(mn, o.x);
    mx = fmaxf(mx, o.y);
  }
  const ScaleZero q = scale_zero(mn, mx);   // the group of these 64 channels
  tc_wait_st();                             // any clipped values are in place

  auto clear = [&]() {
#pragma unroll
    for (int u = 0; u < NS; ++u) wd[u][0] = wd[u][1] = 0u;
  };
  // storage word and bit position of channel i of this half
  auto word_of = [&](int i) -> uint32_t& {
    const int kk = i & 15, lw = i >> 5;
    return (TENSOR == 0) ? wd[(kk & 7) >> 1][lw] : wd[kk & 7][lw];
  };
  auto pos_of = [](int i) -> int {
    const int kk = i & 15, s1 = (i >> 4) & 1;
    return (TENSOR == 0) ? 16 * (kk & 1) + 2 * (2 * s1 + 4 * (kk >> 3)) : 2 * (2 * s1 + (kk >> 3));
  };
  // code = rint(clamp(fl(fl(y - z) / s), 0, 3)).  The clamped quotient is
  // 3 u with u = sat(fl(y - z) * fl(fl(1/s) / 3)) (the saturating multiply
  // clamps to [0, 1] for free; 3 u lies within 1e-6 of fl(fl(y - z) / s)
  // clamped); 3 u + 1.5 * 2^23, rounded once, holds rint(3 u) in its low
  // mantissa bits (round to nearest even), unless the quotient lies within
  // 2^-18 of a half-integer, where the IEEE division decides (quant_code).
  // Out of [0, 3] the clamp leaves an integer, so only ties inside the range
  // can need the exact path.
  clear();
  const float rs3 = __fmul_rn(q.rs, 0.3333333432674408f);   // the quotient / 3, saturated to [0, 1]
  const uint64_t zz = f2pack(q.z, q.z), three = f2pack(3.0f, 3.0f), mag = f2pack(12582912.0f, 12582912.0f);
  // channels i and i + 1 as one pair: rr = 3 u + 1.5 * 2^23 rounded once
  // (its bits are 0x4B400000 + code) and e = 3 u - code
  auto fast_pair = [&](float y0, float y1, float& r0, float& r1, float& e0, float& e1) {
    float d0, d1, u0, u1;
    f2unpack(f2sub(f2pack(y0, y1), zz), d0, d1);
    asm("mul.rn.sat.f32 %0, %1, %2;" : "=f"(u0) : "f"(d0), "f"(rs3));
    asm("mul.rn.sat.f32 %0, %1, %2;" : "=f"(u1) : "f"(d1), "f"(rs3));
    const uint64_t up = f2pack(u0, u1);
    const uint64_t rr = f2fma(up, three, mag);
    f2unpack(rr, r0, r1);
    f2unpack(f2fma(up, three, f2sub(mag, rr)), e0, e1);   // the code is exactly 1.5 * 2^23 - rr, negated
  };
  constexpr float kTieBand = 0.499996185302734375f;   // 1/2 - 2^-18
  float emx[2];   // largest distance to the code per 32-channel block
#pragma unroll
  for (int cb = 0; cb < 2; ++cb) {
    float v[32];
    rotated32(cb, v);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float r0, r1, e0, e1;
      fast_pair(v[i], v[i + 1], r0, r1, e0, e1);
      // one integer multiply-add places a code (the constant offsets of a
      // word fold into one; codes do not overlap, so the sum is the OR)
      const int pos0 = pos_of(32 * cb + i), pos1 = pos_of(32 * cb + i + 1);
      word_of(32 * cb + i) += __float_as_uint(r0) * (1u << pos0) - (0x4B400000u << pos0);
      word_of(32 * cb + i + 1) += __float_as_uint(r1) * (1u << pos1) - (0x4B400000u << pos1);
      v[i] = fabsf(e0);
      v[i + 1] = fabsf(e1);
    }
    emx[cb] = max_of32(0.0f, v);
  }
  // a block with a near tie in some lane is read again (a warp-collective
  // tensor-memory load); only the values within the band get the exact code,
  // patched into their 2-bit fields
#pragma unroll
  for (int cb = 0; cb < 2; ++cb) {
    if (!__any_sync(0xffffffffu, emx[cb] >= kTieBand)) continue;
    float v[32];
    rotated32(cb, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float r0, r1, e0, e1;
      if ((i & 1) == 0) fast_pair(v[i], v[i + 1], r0, r1, e0, e1);
      const float r = (i & 1) ? r1 : r0, e = (i & 1) ? e1 : e0;
      if (fabsf(e) >= kTieBand) {
        const uint32_t fast = __float_as_uint(r) - 0x4B400000u;
        word_of(32 * cb + i) ^= ((fast ^ quant_code_exact(v[i], q)) & 3u) << pos_of(32 * cb + i);
      }
    }
  }

  return q;
}

// ---- bulk append: one CTA per SM, warp-specialised ---------------------------
// The CTA's live chunks j = 0, 1, 2, ... alternate between two teams of eight
// epilogue warps (team j % 2).  Chunk j's x lands in buffer j % 4 and its
// product in accumulator j % 4 (tensor-memory columns 128 (j % 4)), so every
// buffer and accumulator belongs to one team.  Four more warps serve the
// teams, one thread each: per team a loader walks the tasks, publishes each
// chunk's record and starts its x load as soon as the buffer is free (product
// j - 4 complete), and an issuer starts product j once its x is in and the
// team has read accumulator j % 4 for chunk j - 4; the product barrier also
// takes the issuer's own arrival after it read the record, so a warp that sees
// the product also sees its record.  A team's end is a record with no chunk,
// signalled on the product barrier the same way once every warp has released
// chunk j - 4 (an earlier signal would complete a phase past one a slow warp
// still waits for).  Nothing waits on a CTA barrier inside the loop: records,
// x, products and accumulators are handed over through mbarriers, and an
// issuer thread that stalls while the tensor cores take its sixteen MMAs holds
// up no epilogue warp.
constexpr int kBkWarps = 20;                 // 16 epilogue + 4 serving warps
constexpr int kBkThreads = 32 * kBkWarps;
constexpr int kBkCols = 512;                 // four 128-column fp32 accumulators
constexpr uint32_t kBkOffB = 0;              // R^T hi | lo
constexpr uint32_t kBkOffA = kBkOffB + kBBytes;             // four x buffers
constexpr uint32_t kBkOffClip = kBkOffA + 4 * kABytes;
constexpr uint32_t kBkOffClipMin = kBkOffClip + 128 * 4;   // [4] smallest clip of each 32-channel block
constexpr uint32_t kBkOffStat = kBkOffClipMin + 16;        // [team][chunk parity][half][128 rows] (min, max)
constexpr uint32_t kBkOffInfo = kBkOffStat + 2 * 2 * 2 * 128 * 8;   // [8] chunk records of 8 ints
// mbarriers: [0] R; [1 + b] x in buffer b; [5 + b] product b done (its commit
// and the issuer's arrival); [9 + b] accumulator b read (eight warps);
// [13 + s] record s published (to the issuer)
constexpr int kBkBars = 21;
constexpr uint32_t kBkOffBar = kBkOffInfo + 8 * 32;
constexpr uint32_t kBkOffMisc = kBkOffBar + kBkBars * 8;     // tensor-memory address, abort flag, last load / product per buffer
constexpr uint32_t kBkSmem = kBkOffMisc + 48 + 1024;        // + alignment slack

// chunk record fields (record j % 8 describes chunk j)
enum { kRecB = 0, kRecC0, kRecNb, kRecH0, kRecLast, kRecP0, kRecState };
enum { kChunkNone = 0, kChunkTma = 1, kChunkCopy = 2 };   // record state: no chunk, x by TMA, x by copies

__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ uint32_t par(int j, int shift) { return (uint32_t)(j >> shift) & 1u; }
// mbar_wait for the serving warps: each poll may suspend the thread until the
// phase completes or about 1 us passes, so that a waiting server takes no
// issue slots from the epilogue warps
__device__ __forceinline__ bool mbar_wait_idle(uint64_t* bar, uint32_t parity, int limit) {
  const uint32_t a = smem_u32(bar);
  for (int it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(a), "r"(parity), "r"(1000u)
        : "memory");
    if (done) return true;
  }
  return false;
}
// whether `p` holds in all 64 threads of named barrier `id` (both warps of a
// lane quarter), so that the two take the same branch before the barrier
// they share in the epilogue of group 128
__device__ __forceinline__ bool pair_and(int id, bool p) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred pi, po;\n"
      "setp.ne.u32 pi, %1, 0;\n"
      "bar.red.and.pred po, %2, 64, pi;\n"
      "selp.u32 %0, 1, 0, po; }"
      : "=r"(r)
      : "r"((uint32_t)p), "r"(id)
      : "memory");
  return r != 0u;
}

template <int GS, int TENSOR>
__device__ __forceinline__ void tc_body(const TcArgs& a, const CUtensorMap* xmap, uint8_t* sm) {
  constexpr int NG = 128 / GS;
  const uint32_t sA0 = smem_u32(sm + kBkOffA), sB = smem_u32(sm + kBkOffB);
  float* sclip = reinterpret_cast<float*>(sm + kBkOffClip);
  float* sclipmin = reinterpret_cast<float*>(sm + kBkOffClipMin);
  int* info = reinterpret_cast<int*>(sm + kBkOffInfo);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBkOffBar);
  uint64_t* xfull = bars + 1;     // x of chunk j in buffer j % 4
  uint64_t* mdone = bars + 5;     // product of chunk j in accumulator j % 4
  uint64_t* accfree = bars + 9;   // accumulator j % 4 read by the team's eight warps
  uint64_t* recready = bars + 13; // record j % 8 published
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kBkOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kBkOffMisc + 4);
  int* last_load = reinterpret_cast<int*>(sm + kBkOffMisc + 8);   // [4] last chunk loaded by TMA per buffer
  int* last_prod = last_load + 4;                                  // [4] last product issued per accumulator
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y;

  if (tid == 0) {
    mbar_init(bars + 0, 1);
    for (int b = 0; b < 4; ++b) {
      mbar_init(xfull + b, 1);
      mbar_init(mdone + b, 2);   // the product's commit and the issuer's arrival
      mbar_init(accfree + b, 8);
      last_load[b] = -1;
      last_prod[b] = -1;
    }
    for (int s2 = 0; s2 < 8; ++s2) mbar_init(recready + s2, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) tc_alloc(smem_u32(tslot), kBkCols);
  if (tid < 128) sclip[tid] = a.clip[((size_t)TENSOR * a.Hkv + g) * 128 + tid];
  if (tid >= 128 && tid < 132) {   // the smallest clip of channels 32 (tid - 128) ..
    const float* c = a.clip + ((size_t)TENSOR * a.Hkv + g) * 128 + 32 * (tid - 128);
    float v = c[0];
    for (int i = 1; i < 32; ++i) v = fminf(v, c[i]);
    sclipmin[tid - 128] = v;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0) {   // R^T hi | lo of this (head, tensor), already in the swizzled operand layout
    const uint4* src = a.rfrag + ((size_t)g * kFragBlocks + 1 + TENSOR) * 4096;
    mbar_expect_tx(bars + 0, kBBytes);
#pragma unroll
    for (int c = 0; c < 4; ++c) bulk_g2s(sm + kBkOffB + 16384 * c, src + 1024 * c, 16384, bars + 0);
  }
  auto fail = [&]() {
    flag_error(a.err, KV_DEVERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp >= 16) {
    // ---- serving warps: 16 + t loads for team t, 18 + t issues its products ----
    const int team = warp & 1;
    if (warp < 18) {
      const uint16_t* X = TENSOR ? a.x[1] : a.x[0];
      const int total = a.n_seqs * a.max_chunks;
      const int t0 = blockIdx.x * a.tasks_per_cta;
      const int t1 = min(total, t0 + a.tasks_per_cta);
      // x of a chunk: two TMA tile loads when all 128 rows lie below the
      // input's row count T and inside the tensor map (rows below 0 read as
      // zero); otherwise, so that nothing past the caller's buffer is read,
      // 16-byte copies by the loader's warp with rows outside the append range
      // zero-filled
      const int row_lim = (int)min((long long)__ldg(a.cu + a.n_seqs), a.map_rows);
      // the walk over the CTA's live chunks, at the team's next chunk (it
      // steps over the other team's); team 0's loader reports the errors of
      // the sequences it walks into
      TaskCursor tc;
      const bool report = team == 0 && lane == 0;
      tc.start(a, t0, t1, report);
      tc.next_live(a, report);
      if (team == 1 && tc.t < t1) {
        tc.step(a, false);
        tc.next_live(a, false);
      }
      for (int J = team;; J += 2) {
        // buffer J % 4 is free once product J - 4 is complete; record J % 8
        // was read by the team before it released accumulator (J - 8) % 4,
        // which came before product J - 4
        if (J >= 4) {
          bool ok = *abort_flag == 0;
          if (ok && lane == 0) ok = mbar_wait_idle(mdone + (J & 3), par(J - 4, 2), a.wait_polls);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) {
            if (lane == 0) fail();
            break;
          }
        }
        int* r = info + 8 * (J & 7);
        const bool have = tc.t < t1;
        Chunk k = tc.chunk();
        const int r0 = k.c0 + (k.P0 - k.h0);
        const bool tma = have && r0 + kChunk <= row_lim;
        // test hook: this chunk's x is never loaded, so its issuer's bounded wait runs out
        const bool withhold = have && a.stall_first_load && J == 0 && blockIdx.x == 0 && blockIdx.y == 0;
        if (lane == 0) {
          r[kRecB] = k.b;
          r[kRecC0] = k.c0;
          r[kRecNb] = k.nb;
          r[kRecH0] = k.h0;
          r[kRecLast] = k.last;
          r[kRecP0] = k.P0;
          r[kRecState] = !have ? kChunkNone : tma ? kChunkTma : kChunkCopy;
          if (tma && !withhold) {
            const uint32_t dst = sA0 + (uint32_t)(J & 3) * kABytes;
            mbar_expect_tx(xfull + (J & 3), kABytes);
            tma_load_x(dst, xmap, 0, g, r0, xfull + (J & 3));
            tma_load_x(dst + 16384, xmap, 64, g, r0, xfull + (J & 3));
            last_load[J & 3] = J;
          }
          mbar_arrive1(recready + (J & 7));   // release: the record is visible to its waiters
        }
        if (!have) break;
        if (!tma && !withhold) {   // the warp's 32 lanes copy the 128 half rows x 2 of the chunk
          for (int i = 0; i < 8; ++i) load_chunk(a, X, g, k, sA0 + (uint32_t)(J & 3) * kABytes, lane + 32 * i);
          asm volatile("cp.async.wait_group 0;" ::: "memory");
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive1(xfull + (J & 3));
        }
        for (int s2 = 0; s2 < 2 && tc.t < t1; ++s2) {   // past the other team's chunk to this team's next
          tc.step(a, report);
          tc.next_live(a, report);
        }
      }
    } else if (lane == 0) {
      bool ok = mbar_wait_idle(bars + 0, 0, a.wait_polls);   // R is needed before the first product
      if (!ok) fail();
      for (int J = team; ok; J += 2) {
        ok = *abort_flag == 0 && mbar_wait_idle(recready + (J & 7), par(J, 3), a.wait_polls);
        if (!ok) {
          fail();
          break;
        }
        if (info[8 * (J & 7) + kRecState] == kChunkNone) {   // the team's end: its warps read the record
          // first every warp has taken product J - 4 from this barrier (and
          // released its accumulator): completing the next phase earlier would
          // hide product J - 4's phase from a warp still waiting for it
          if (J >= 4 && !mbar_wait_idle(accfree + (J & 3), par(J - 4, 2), a.wait_polls)) {
            fail();
            break;
          }
          mbar_arrive1(mdone + (J & 3));
          mbar_arrive1(mdone + (J & 3));
          break;
        }
        // x in, and accumulator J % 4 read by the team for chunk J - 4
        ok = mbar_wait_idle(xfull + (J & 3), par(J, 2), a.wait_polls) &&
             (J < 4 || mbar_wait_idle(accfree + (J & 3), par(J - 4, 2), a.wait_polls));
        if (!ok) {
          fail();
          break;
        }
        issue_rotation(tmem + 128u * (uint32_t)(J & 3), sA0 + (uint32_t)(J & 3) * kABytes, sB, mdone + (J & 3));
        // the second arrival (a release after this thread acquired the record):
        // a warp that sees product J complete also sees record J
        mbar_arrive1(mdone + (J & 3));
        last_prod[J & 3] = J;
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue warps ----
    const int team = warp >> 3, lwarp = warp & 7;
    // warp w of a team reads accumulator rows 32 (w % 4) .. (its tensor-memory
    // lane quarter) and channels 64 (w / 4) .. 64 (w / 4) + 63
    const int quarter = lwarp & 3, hf = lwarp >> 2;
    const int qbar = 1 + 4 * team + quarter;   // the quarter's two warps (group 128)
    const int m = 32 * quarter + lane;         // this thread's token row of a chunk
    const int m16 = m & 15;
    for (int j = team;; j += 2) {
      // product j complete, which also publishes record j (the issuer arrives
      // once it has read the record; at the team's end it arrives twice with
      // no product); at group 128 the two warps of a quarter decide together:
      // they meet at a barrier in the epilogue
      bool ok = __all_sync(0xffffffffu, *abort_flag == 0 && mbar_wait(mdone + (j & 3), par(j, 2), a.wait_polls));
      if (GS == 128) ok = pair_and(qbar, ok);
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      const int* r = info + 8 * (j & 7);
      if (r[kRecState] == kChunkNone) break;
      tc_fence_after();
      Chunk k;
      k.b = r[kRecB];
      k.h0 = r[kRecH0];
      k.nb = r[kRecNb];
      k.last = r[kRecLast];
      k.P0 = r[kRecP0];

      // ---- destination tile of this row (its page id read before the epilogue) ----
      const int pos = k.P0 + m;
      const bool row_ok = pos >= k.h0 && pos < k.h0 + k.nb;
      const int tile = pos / kTile;
      const bool tile_live = tile <= k.last;
      const int pid_raw = __ldg(a.pt + (size_t)k.b * a.max_pages + min((tile * kTile) / a.P, a.max_pages - 1));

      // ---- this thread's row and channel half -> s, z and codes ----
      constexpr int NS = (TENSOR == 0) ? 4 : 8;
      uint32_t wd[NS][2];
      const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16) + 128u * (uint32_t)(j & 3);
      float2* sstat = reinterpret_cast<float2*>(sm + kBkOffStat) + 256 * (2 * team + ((j >> 1) & 1));
      const ScaleZero q = row_codes<GS, TENSOR>(trow, hf, m, sclip, sclipmin, sstat, wd, qbar);
      // the accumulator is read: release it to the team's issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive1(accfree + (j & 3));
      const bool pid_ok = pid_raw >= 0 && pid_raw < a.num_pages;
      if (tile_live && !pid_ok && m16 == 0 && hf == 0) flag_error(a.err, KV_DEVERR_PAGE_ID);
      const bool write = tile_live && pid_ok;
      uint8_t* tb = a.hist + (size_t)(pid_ok ? pid_raw : 0) * a.page_bytes + (size_t)g * a.head_block +
                    (size_t)((tile * kTile) % a.P / kTile) * a.tile_bytes;
      const unsigned okmask = __ballot_sync(0xffffffffu, row_ok && write);

      if constexpr (TENSOR == 0) {
        // K: code (token m16, channel c) -> slot 4*(m16%8) + (k%8)/2, word c/32,
        // bit 16*(k%2) + 2*(2*((c/16)%2) + m16/8 + 4*(k/8)), k = c%16; this half
        // holds words 2 hf and 2 hf + 1 of every slot
        const int mh = m16 >> 3;
        uint32_t out[2][2];
  #pragma unroll
        for (int jj = 0; jj < 2; ++jj)
  #pragma unroll
          for (int w = 0; w < 2; ++w) {
            const uint32_t lo_w = wd[jj][w] << (2 * mh), hi_w = wd[2 + jj][w] << (2 * mh);
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, mh ? lo_w : hi_w, 8);
            out[jj][w] = (mh ? hi_w : lo_w) | recv;
          }
        const bool me = (okmask >> lane) & 1u, other = (okmask >> (lane ^ 8)) & 1u;
        const uint32_t pat_me = mh ? 0xCCCCCCCCu : 0x33333333u;
        const uint32_t mask = (me ? pat_me : 0u) | (other ? ~pat_me : 0u);
        if (write) {
  #pragma unroll
          for (int jj = 0; jj < 2; ++jj)
            store_merge2(tb + 16 * (4 * (m16 & 7) + 2 * mh + jj) + 8 * hf, out[jj], mask);
        }
        if (write && row_ok && (GS == 64 || hf == 0)) {
          __half2* rec = reinterpret_cast<__half2*>(tb + 1024 + (2 * (m16 & 7) + mh) * 4 * NG);
          rec[GS == 64 ? hf : 0] = __halves2half2(q.sh, q.zh);
        }
      } else {
        // V: code (channel c, token m16) -> slot 4*(c%8) + (m16%8)/2, word c/32,
        // bit 16*(m16%2) + 2*(2*((c/16)%2) + (c%16)/8 + 4*(m16/8))
        const int ek = m16 & 1, kh = m16 >> 3;
        const int sh = 16 * ek + 8 * kh;
        uint32_t r1[4][2];   // partner lane ^ 8: keep slots with m8 / 4 == kh
  #pragma unroll
        for (int i = 0; i < 4; ++i)
  #pragma unroll
          for (int w = 0; w < 2; ++w) {
            const uint32_t a0 = wd[i][w] << sh, a1 = wd[4 + i][w] << sh;
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, kh ? a0 : a1, 8);
            r1[i][w] = (kh ? a1 : a0) | recv;
          }
        uint32_t out[2][2];  // partner lane ^ 1: keep m8 % 4 / 2 == ek
  #pragma unroll
        for (int ii = 0; ii < 2; ++ii)
  #pragma unroll
          for (int w = 0; w < 2; ++w) {
            const uint32_t a0 = r1[ii][w], a1 = r1[2 + ii][w];
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, ek ? a0 : a1, 1);
            out[ii][w] = (ek ? a1 : a0) | recv;
          }
        // bits of the four tokens sharing these words: (ek', kh') -> 0x00FF / 0xFF00 in half ek'
        const int base = lane & ~9;
        uint32_t mask = 0u;
  #pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int e2 = t & 1, k2 = t >> 1;
          if ((okmask >> (base | e2 | (k2 << 3))) & 1u) mask |= (k2 ? 0xFF00u : 0x00FFu) << (16 * e2);
        }
        const int jk = (m16 & 7) >> 1;
        if (write) {
  #pragma unroll
          for (int ii = 0; ii < 2; ++ii)
            store_merge2(tb + 512 + 16 * (4 * (4 * kh + 2 * ek + ii) + jk) + 8 * hf, out[ii], mask);
        }
        if (write && row_ok && (GS == 64 || hf == 0)) {
          __half2* rec = reinterpret_cast<__half2*>(tb + 1024 + 64 * NG + (2 * (m16 & 7) + kh) * 4 * NG);
          rec[GS == 64 ? hf : 0] = __halves2half2(q.sh, q.zh);
        }
      }
    }
  }

  // every role is done.  On the normal path every load fed a product and
  // every product was read by its team; after an early exit, wait (bounded)
  // for what may still be in flight: the last TMA load and the last product
  // of each buffer (the phases of a barrier complete in order)
  __syncthreads();
  if (tid == 0 && *abort_flag != 0) {
    mbar_wait(bars + 0, 0, kTcPolls);
    for (int b = 0; b < 4; ++b) {
      if (last_load[b] >= 0) mbar_wait(xfull + b, par(last_load[b], 2), kTcPolls);
      if (last_prod[b] >= 0) mbar_wait(mdone + b, par(last_prod[b], 2), kTcPolls);
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, kBkCols);
  if (tid == 0)
    for (int i = 0; i < kBkBars; ++i) mbar_inval(bars + i);
}

template <int GS, int TENSOR>
__global__ void __launch_bounds__(kBkThreads, 1)
    append_tc_kernel(TcArgs a, const __grid_constant__ CUtensorMap xmap) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned (the swizzled operands), by an offset into the shared
  // array so that the compiler keeps the accesses in the shared space
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // K: the V launch may start as this grid's CTAs leave; V: this grid ends
  // only after the K grid (a later kernel of the stream waits for both)
  if (TENSOR == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc_body<GS, TENSOR>(a, &xmap, sm);
  if (TENSOR == 1 && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
}


// ---------------------------------------------------------------------------
// per-step placement (yunpan.plus write-up, "2. 在线量化与反量化": a new token
// is written to the recent tier; when that is full its oldest token is
// rotated, clipped, quantized and packed into the INT2 history)
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
  unsigned* tickets;              // layer base [ceil(max_seqs / 128)]
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

// One launch per step: CTA (128 sequences, KV head g, tensor).  The evicted
// tokens of the step (the ring's oldest token of every sequence whose ring is
// full) become the rows of one 128-row chunk, rotated and quantized exactly as
// the bulk append does it (same MMA, same row_codes); each row then goes into
// its own tile at its own row, merged with the tile's other rows.  Once a
// thread's copy of the old slot contents has landed it writes the new token's
// half row into the slot (sink or ring).  The CTAs of a chunk count themselves
// on a ticket after reading the lengths; the last one updates the lengths.
constexpr uint32_t kOffRows = kOffTmem + 16;
constexpr uint32_t kEvSmem = kOffRows + 128 * 8 + 2 * 128 * 4 + 16 + 1024;   // + alignment slack

template <int GS, int TENSOR>
__device__ __forceinline__ void evict_body(const StepArgs& a, int B, uint8_t* sm) {
  constexpr int NG = 128 / GS;
  const uint32_t sA = smem_u32(sm + kOffA), sB = smem_u32(sm + kOffB);
  float* sclip = reinterpret_cast<float*>(sm + kOffClip);
  float2* sstat = reinterpret_cast<float2*>(sm + kOffStat);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);   // [0] R copy, [1] MMA done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kOffTmem);
  long long* rtile = reinterpret_cast<long long*>(sm + kOffRows);   // byte offset of the row's tile, -1: none
  int* rpos = reinterpret_cast<int*>(sm + kOffRows + 128 * 8);      // row within the tile
  int* rplace = rpos + 128;                                         // mode | slot << 2 of the placement, -1: none
  unsigned* slast = reinterpret_cast<unsigned*>(rplace + 128);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y;
  const int quarter = warp & 3, hf = warp >> 2;
  const int m = 32 * quarter + lane;

  if (tid == 0) {
    mbar_init(bars + 0, 1);
    mbar_init(bars + 1, 1);
    mbar_fence_init();
  }
  if (warp == 0) tc_alloc(smem_u32(tslot), kTcCols);
  if (tid < 128) sclip[tid] = a.clip[((size_t)TENSOR * a.Hkv + g) * 128 + tid];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0) {
    const uint4* src = a.rfrag + ((size_t)g * kFragBlocks + 1 + TENSOR) * 4096;
    mbar_expect_tx(bars + 0, kBBytes);
#pragma unroll
    for (int c = 0; c < 4; ++c) bulk_g2s(sm + kOffB + 16384 * c, src + 1024 * c, 16384, bars + 0);
  }
  {   // the evicted rows -> the swizzled A operand (thread t: row t % 128, channel half t / 128)
    const int row = tid & 127, hh = tid >> 7;
    const int b = blockIdx.x * kChunk + row;
    StepPlace pl{-1, 0, 0, 0, 0};
    if (b < B) pl = step_place(a, b);
    const bool ev = pl.mode == 2;
    if (hh == 0) {
      rtile[row] = ev ? pl.tile : -1;
      rpos[row] = pl.pos;
    }
    if (hh == 0) rplace[row] = (pl.mode < 0) ? -1 - pl.err : (pl.mode | (pl.slot << 2));
    uint16_t* rec = TENSOR ? a.rec_v : a.rec_k;
    const size_t sh = (size_t)b * a.Hkv + g;
    const uint16_t* src = rec + (ev ? (sh * a.rec_cap + pl.slot) * 128 : 0) + 64 * hh;
#pragma unroll
    for (int c = 0; c < 8; ++c)
      cp_async16_zfill(sA + hh * 16384 + row * 128 + ((c ^ (row & 7)) << 4), src + 8 * c, ev);
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
    // the old contents of this half row are in shared memory: the new token
    // takes the slot (the sequence's next sink slot or its ring slot)
    if (pl.mode >= 0) {
      const uint16_t* nsrc = (TENSOR ? a.v_new : a.k_new) + sh * 128 + 64 * hh;
      uint16_t* dst = (pl.mode == 0) ? (TENSOR ? a.sink_v : a.sink_k) + (sh * a.sink_cap + pl.slot) * 128
                                     : rec + (sh * a.rec_cap + pl.slot) * 128;
#pragma unroll
      for (int c = 0; c < 16; ++c)
        *reinterpret_cast<uint2*>(dst + 64 * hh + 4 * c) = *reinterpret_cast<const uint2*>(nsrc + 4 * c);
    }
  }
  fence_async_smem();
  // every thread has read its rows' lengths: count this CTA on the chunk's
  // ticket; the last CTA of the chunk moves the lengths
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned n = gridDim.y * gridDim.z;
    *slast = (atomicAdd(a.tickets + blockIdx.x, 1u) == n - 1u) ? 1u : 0u;
  }
  __syncthreads();
  if (*slast != 0u && tid < kChunk) {
    __threadfence();
    const int b = blockIdx.x * kChunk + tid;
    const int pc = rplace[tid];
    if (b < B) {
      const int mode = pc & 3, slot = pc >> 2;
      if (pc < 0) {
        flag_error(a.err, -1 - pc);
      } else if (mode == 0) {
        a.sink_len[b] = slot + 1;
      } else if (mode == 1) {
        a.rec_len[b] += 1;
      } else {
        a.hist_len[b] += 1;
        a.rec_start[b] = (slot + 1) % a.rec_cap;
      }
    }
    if (tid == 0) a.tickets[blockIdx.x] = 0u;   // ready for the next step
  }
  bool ok = mbar_wait(bars + 0, 0, kTcPolls);
  if (__syncthreads_and(ok)) {
    if (tid == 0) issue_rotation(tmem, sA, sB, bars + 1);
    ok = mbar_wait(bars + 1, 0, kTcPolls);
    ok = __syncthreads_and(ok);
    if (!ok && tid == 0) {
      flag_error(a.err, KV_DEVERR_TIMEOUT);
      mbar_wait(bars + 1, 0, kTcPolls);   // the MMAs in flight, bounded
    }
  } else if (tid == 0) {
    flag_error(a.err, KV_DEVERR_TIMEOUT);
    mbar_wait(bars + 0, 0, kTcPolls);     // the copies in flight, bounded
  }
  // a lane quarter without an evicted row skips the epilogue (both of its
  // warps see the same rows, so they skip together)
  if (ok && __any_sync(0xffffffffu, rtile[m] >= 0)) {
    tc_fence_after();
    constexpr int NS = (TENSOR == 0) ? 4 : 8;
    uint32_t wd[NS][2];
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    const ScaleZero q = row_codes<GS, TENSOR>(trow, hf, m, sclip, nullptr, sstat, wd, 1 + quarter);
    const long long tof = rtile[m];
    if (tof >= 0) {
      const int pos = rpos[m];
      uint8_t* tb = a.hist + tof + (size_t)g * a.head_block;
      if constexpr (TENSOR == 0) {
        // K: the row's codes at pairs + pos / 8 of its four slots 4 * (pos % 8) + j
        const int mh = pos >> 3;
        const uint32_t mask = mh ? 0xCCCCCCCCu : 0x33333333u;
        // every old word first (one round trip), then the merged words
        uint2* dst[4];
        uint2 old[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          dst[j] = reinterpret_cast<uint2*>(tb + 16 * (4 * (pos & 7) + j) + 8 * hf);
          old[j] = *dst[j];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *dst[j] = make_uint2((old[j].x & ~mask) | ((wd[j][0] << (2 * mh)) & mask),
                               (old[j].y & ~mask) | ((wd[j][1] << (2 * mh)) & mask));
        if (GS == 64 || hf == 0) {
          __half2* rec = reinterpret_cast<__half2*>(tb + 1024 + (2 * (pos & 7) + mh) * 4 * NG);
          rec[GS == 64 ? hf : 0] = __halves2half2(q.sh, q.zh);
        }
      } else {
        // V: the token's codes in byte (pos / 8) of half (pos % 2) of its eight
        // slots 4 * m8 + (pos % 8) / 2
        const int ek = pos & 1, kh = pos >> 3, jk = (pos & 7) >> 1, sh = 16 * ek + 8 * kh;
        const uint32_t mask = (kh ? 0xFF00u : 0x00FFu) << (16 * ek);
        // every old word first (one round trip), then the merged words
        uint2* dst[8];
        uint2 old[8];
#pragma unroll
        for (int m8 = 0; m8 < 8; ++m8) {
          dst[m8] = reinterpret_cast<uint2*>(tb + 512 + 16 * (4 * m8 + jk) + 8 * hf);
          old[m8] = *dst[m8];
        }
#pragma unroll
        for (int m8 = 0; m8 < 8; ++m8)
          *dst[m8] = make_uint2((old[m8].x & ~mask) | ((wd[m8][0] << sh) & mask),
                                (old[m8].y & ~mask) | ((wd[m8][1] << sh) & mask));
        if (GS == 64 || hf == 0) {
          __half2* rec = reinterpret_cast<__half2*>(tb + 1024 + 64 * NG + (2 * (pos & 7) + kh) * 4 * NG);
          rec[GS == 64 ? hf : 0] = __halves2half2(q.sh, q.zh);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, kTcCols);
  if (tid == 0) {
    mbar_inval(bars + 0);
    mbar_inval(bars + 1);
  }
}

template <int GS>
__global__ void __launch_bounds__(kTcThreads, 2) evict_tc_kernel(StepArgs a, int B) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  if (blockIdx.z == 0)
    evict_body<GS, 0>(a, B, sm);
  else
    evict_body<GS, 1>(a, B, sm);
}

}  // namespace

// cuTensorMapEncodeTiled from the driver, looked up once
void* tensor_map_encode_fn() {
  static void* fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return f;
  }();
  return fn;
}

cudaError_t launch_append_tc(const Pool& p, int layer, int n_seqs, const void* k, const void* v,
                             const int32_t* cu, const int32_t* hist_start, const int32_t* pt,
                             int max_pages, int max_tokens, cudaStream_t s) {
  const int H = p.cfg.num_kv_heads;
  TcArgs a;
  a.hist = p.hist + (size_t)layer * p.hist_layer_stride;
  a.page_bytes = p.page_bytes;
  a.head_block = p.page_bytes / H;
  a.tile_bytes = (int)p.tile_bytes;
  a.P = p.cfg.page_size;
  a.x[0] = static_cast<const uint16_t*>(k);
  a.x[1] = static_cast<const uint16_t*>(v);
  a.cu = cu;
  a.hist_start = hist_start;
  a.pt = pt;
  a.max_pages = max_pages;
  a.n_seqs = n_seqs;
  const int max_tiles = (max_tokens + kTile - 1) / kTile + 1;   // +1: an unaligned start spans one more
  a.max_chunks = (max_tiles + kTilesPerChunk - 1) / kTilesPerChunk;
  a.Hkv = H;
  a.num_pages = p.cfg.num_pages;
  a.map_rows = (long long)n_seqs * max_tokens;
  a.wait_polls = p.test_wait_polls > 0 ? p.test_wait_polls : kTcPolls;
  a.stall_first_load = p.test_stall_first_copy;
  a.rfrag = p.rfrag + (size_t)layer * H * kFragBlocks * rfrag_per_head();
  a.clip = p.clip + (size_t)layer * 2 * H * 128;
  a.err = p.err;
  const long long tasks = (long long)n_seqs * a.max_chunks;
  if (tasks >= (1LL << 31)) return cudaErrorInvalidValue;   // task indices are 32-bit
  // x viewed as (128 channels, Hkv heads, rows); the row extent n_seqs * max_tokens
  // bounds the input's row count T, and the kernel uses the map only for boxes below T
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap maps[2];
  for (int t = 0; t < 2; ++t) {
    const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)n_seqs * (cuuint64_t)max_tokens};
    const cuuint64_t strides[2] = {256, (cuuint64_t)H * 256};
    const cuuint32_t box[3] = {64, 1, kChunk};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&maps[t], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(a.x[t]), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // one CTA per SM over the KV heads of one tensor; K, then V
  long long ctas = ((long long)p.sm_count + H - 1) / H;
  ctas = max(1LL, min(ctas, tasks));
  a.tasks_per_cta = (int)((tasks + ctas - 1) / ctas);
  ctas = (tasks + a.tasks_per_cta - 1) / a.tasks_per_cta;
  dim3 grid((unsigned)ctas, H, 1);
  static bool attr[2][2] = {{false, false}, {false, false}};
  auto go = [&](auto kernel, int gi, int t) -> cudaError_t {
    if (!attr[gi][t]) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBkSmem);
      // the whole unified L1 / shared array as shared memory
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return e;
      attr[gi][t] = true;
    }
    // the V launch is the K launch's programmatic dependent: its CTAs take SMs
    // as K's CTAs leave (the two write disjoint bytes of the tiles), and each
    // waits for the K grid before it exits, so that the V grid ends after it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kBkThreads, 1, 1);
    cfg.dynamicSmemBytes = kBkSmem;
    cfg.stream = s;
    cudaLaunchAttribute lattr[1];
    lattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    lattr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = lattr;
    cfg.numAttrs = (t == 1) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, a, maps[t]);
  };
  cudaError_t e;
  if (p.cfg.group_size == 64) {
    e = go(append_tc_kernel<64, 0>, 0, 0);
    if (e == cudaSuccess) e = go(append_tc_kernel<64, 1>, 0, 1);
  } else {
    e = go(append_tc_kernel<128, 0>, 1, 0);
    if (e == cudaSuccess) e = go(append_tc_kernel<128, 1>, 1, 1);
  }
  return e;
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
  a.tickets = p.step_tickets + (size_t)layer * ((p.cfg.max_seqs + kChunk - 1) / kChunk);
  a.err = p.err;
  static bool attr[2] = {false, false};
  auto evict = [&](auto kernel, int gi) -> cudaError_t {
    if (!attr[gi]) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kEvSmem);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return e;
      attr[gi] = true;
    }
    kernel<<<dim3((unsigned)((B + kChunk - 1) / kChunk), H, 2), kTcThreads, kEvSmem, s>>>(a, B);
    return cudaGetLastError();
  };
  return (p.cfg.group_size == 64) ? evict(evict_tc_kernel<64>, 0) : evict(evict_tc_kernel<128>, 1);
}

}  // namespace kvint2
