// Device helpers: error word, number formats, the INT2 quantizer, warp MMA.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace kvint2 {

// ---------------------------------------------------------------------------
// error word: first error wins, nothing traps
// ---------------------------------------------------------------------------
__device__ __forceinline__ void flag_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------
// formats
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp32 -> fp16, round to nearest even, overflow saturated to +-65504.
__device__ __forceinline__ __half f16_sat(float x) {
  __half h = __float2half_rn(x);
  if (__hisinf(h) && isfinite(x))
    h = __ushort_as_half(x > 0.f ? (unsigned short)0x7BFF : (unsigned short)0xFBFF);
  return h;
}

// ---------------------------------------------------------------------------
// The INT2 quantizer (asymmetric, fp16 scale and zero per token per group).
// yunpan.plus OSCAR write-up, "2. 在线量化与反量化": clip -> quantize -> pack.
//   s = fp16((max - min) / 3), z = fp16(min) (saturated, -0 -> +0)
//   code = s == 0 ? 0 : clamp(rint((y - z) / s), 0, 3)
// IEEE fp32 subtraction and division (no contraction, no reciprocal), so the
// codes are reproducible bit for bit.
// ---------------------------------------------------------------------------
struct ScaleZero {
  __half sh, zh;
  float s, z;
  float rs;   // fl(1 / s) for s > 0
};

__device__ __forceinline__ ScaleZero scale_zero(float mn, float mx) {
  ScaleZero r;
  float s32 = __fdiv_rn(__fsub_rn(mx, mn), 3.0f);
  float zf = (mn == 0.0f) ? 0.0f : mn;   // canonical +0
  r.sh = f16_sat(s32);
  r.zh = f16_sat(zf);
  r.s = __half2float(r.sh);
  r.z = __half2float(r.zh);
  r.rs = (r.s > 0.0f) ? __frcp_rn(r.s) : 0.0f;
  return r;
}

// code = clamp(rint(fl(fl(y - z) / s)), 0, 3).  The quotient is formed as
// fl(d * fl(1/s)), which is within 1.5 * 2^-23 * |d / s| of fl(d / s); only a
// half-integer between the two could change rint, and the relevant quotients
// are below 3.5, so outside a 2^-18 band around every half-integer the product
// gives the same code and inside it the IEEE division is taken.
__device__ __forceinline__ uint32_t quant_code(float y, const ScaleZero& q) {
  if (q.s == 0.0f) return 0u;
  const float d = __fsub_rn(y, q.z);
  float t = __fmul_rn(d, q.rs);
  if (fabsf(__fsub_rn(t, floorf(t)) - 0.5f) <= 3.814697265625e-6f) t = __fdiv_rn(d, q.s);
  t = rintf(t);
  t = fminf(fmaxf(t, 0.0f), 3.0f);
  return (uint32_t)t;
}

__device__ __forceinline__ float clip_to(float x, float c) { return fminf(fmaxf(x, -c), c); }

// ---------------------------------------------------------------------------
// memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte global -> shared copy that bypasses L1 (completion per thread).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gsrc) : "memory");
}
// ---- mbarrier + bulk copy (global -> shared through the copy engine) ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// makes initialised barriers visible to the copy engine
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// one arrival that also announces `bytes` of incoming copy traffic
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// bytes (a multiple of 16, both addresses 16-byte aligned) from global to
// shared memory; completion is counted on `bar`
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// L2 eviction priorities for bulk copies: data read once per step (the
// history) leaves L2 first; small data every step reads again (rotation
// fragments, R_v^T) stays behind it.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// bulk_g2s with an L2 cache policy
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// waits for the phase with the given parity to complete, giving up after
// `limit` polls; returns whether it completed
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int limit) {
  const uint32_t a = smem_u32(bar);
  for (int it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Hint that a 128-byte line will be read soon: fetch it into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// warp MMA (m16n8k16, fp32 accumulate) and 8x8 transpose
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// (hi, lo) fp16 split of an fp32 value packed as one f16x2 register:
// low half = fp16(x), high half = fp16(x - fp16(x)).
__device__ __forceinline__ uint32_t split_hi_lo(float x) {
  const float r = x - __half2float(__float2half_rn(x));
  return h2_as_u32(__floats2half2_rn(x, r));   // one packed convert; x rounds to fp16(x) again
}

// All eight f16x2 MMA registers of one 32-bit code word, as exact fp16
// subnormals.  Below 2^-14 an fp16 bit pattern read as an integer is the value
// in units of 2^-24, so masking one 2-bit field of each half is the whole
// conversion.  Register m (0..3) holds the codes at bit pairs m (low half) and
// 8+m (high half), register 4+m those at pairs 4+m and 12+m (taken from the
// word shifted right by 8); both carry the weight 4^m * 2^-24.  The stored
// order puts the A fragment of an even step at pairs {0, 1, 4, 5} and of an
// odd step at {2, 3, 6, 7}, so {a0, a1, a2, a3} weigh {1, 4, 1, 4} x 2^-24,
// times 16 for an odd step: a factor per MMA row half and per step, never
// per k, which the caller removes outside the MMA.  With kFlipHi the upper
// k half (a2, a3: registers 4..7) holds 3 - c instead of c, still one logic
// op (and-not); a caller that negates B's upper k half then accumulates
// sum_lo c w - sum_hi (3 - c) w, whose terms have no common sign.
template <bool kFlipHi>
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t (&r)[8]) {
  const uint32_t w8 = kFlipHi ? ~(w >> 8) : (w >> 8);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    r[m] = w & (0x00030003u << (2 * m));
    r[4 + m] = w8 & (0x00030003u << (2 * m));
  }
}

// 2^x for x <= 0 (softmax weights): the hardware approximation, relative
// error about 2^-22; 2^-inf = +0.
__device__ __forceinline__ float exp2_neg(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max_xor(float v, int from) {
  for (int o = from; o < 32; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum_xor(float v, int from) {
  for (int o = from; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace kvint2
