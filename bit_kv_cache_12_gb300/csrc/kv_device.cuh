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
  __half h = __float2half_rn(x);
  float r = x - __half2float(h);
  return h2_as_u32(__halves2half2(h, __float2half_rn(r)));
}

// lop3 (a & b) | c
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Extract the 2-bit codes at bit pair position pi (0..4) of both 16-bit halves
// of w as (code - 1) in fp16: OR the bits into the mantissa of 1024, then one
// exact fma removes the 1024 bias and the 4^pi weight.
template <int PI>
__device__ __forceinline__ uint32_t codes_m1(uint32_t w) {
  static_assert(PI >= 0 && PI <= 4, "mantissa position");
  constexpr uint32_t mask = 0x00030003u << (2 * PI);
  uint32_t x = and_or(w, mask, 0x64006400u);
  // constants: 4^-PI and -(1024 * 4^-PI + 1), both exact in fp16
  constexpr unsigned short kMul[5] = {0x3C00, 0x3400, 0x2C00, 0x2400, 0x1C00};
  constexpr unsigned short kAdd[5] = {0xE401, 0xDC04, 0xD410, 0xCC40, 0xC500};
  __half2 m = __halves2half2(__ushort_as_half(kMul[PI]), __ushort_as_half(kMul[PI]));
  __half2 a = __halves2half2(__ushort_as_half(kAdd[PI]), __ushort_as_half(kAdd[PI]));
  return h2_as_u32(__hfma2(u32_as_h2(x), m, a));
}

// All eight f16x2 registers of one 32-bit code word: reg pi holds the codes at
// bit pairs pi (low half) and 8+pi (high half), as (code - 1).
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t (&r)[8]) {
  r[0] = codes_m1<0>(w);
  r[1] = codes_m1<1>(w);
  r[2] = codes_m1<2>(w);
  r[3] = codes_m1<3>(w);
  r[4] = codes_m1<4>(w);
  uint32_t w5 = w >> 10;
  r[5] = codes_m1<0>(w5);
  r[6] = codes_m1<1>(w5);
  r[7] = codes_m1<2>(w5);
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
