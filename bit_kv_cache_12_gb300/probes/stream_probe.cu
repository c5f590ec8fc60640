// Streaming-ceiling probe for the INT2 decode's history read: how fast can one
// launch bring the 100k-context history of the Qwen3-4B-shaped decode (57.4 MB:
// 6,230 shuffled pages x 8 KV heads x 1,152-byte tiles) into shared memory when
// nothing is computed?  A measurement tool beside bench.py, not part of the
// library.  Variants:
//   empty        an empty kernel (launch + event overhead)
//   contig       16-byte vector loads over a contiguous 57.4 MB buffer
//   paged Sx hy  the decode's access pattern: 144 CTAs (18 splits x 8 KV-head
//                groups / y) of 16 warps, each warp streaming its tiles through
//                an x-stage ring of bulk copies on mbarriers (lane 0 issues);
//                one copy brings y consecutive KV heads' tiles of a page
//                (1,152 y bytes); "w8": 8 warps per CTA; "linear": pages in order
// Each is timed with CUDA events, after an L2 flush (256 MiB write + read:
// "cold") and without one ("warm": the 57 MB stay in L2).  Every wait is
// bounded; a wait that runs out is counted and reported.
// Build and run: nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o stream_probe stream_probe.cu && ./stream_probe
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <random>
#include <vector>

#define CK(x)                                                                             \
  do {                                                                                    \
    cudaError_t e_ = (x);                                                                 \
    if (e_ != cudaSuccess) {                                                              \
      fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_));          \
      exit(1);                                                                            \
    }                                                                                     \
  } while (0)

constexpr int TB = 1152;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
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

__global__ void empty_kernel(int* p) {
  if (p && threadIdx.x == 1000000) *p = 0;
}

__global__ void contig_kernel(const uint4* __restrict__ src, size_t n16, unsigned* out) {
  unsigned acc = 0;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride), c = __ldcs(src + i + 2 * stride),
          d = __ldcs(src + i + 3 * stride);
    acc ^= a.x ^ b.y ^ c.z ^ d.w;
  }
  for (; i < n16; i += stride) acc ^= __ldcs(src + i).x;
  if (acc == 0x12345678u) out[blockIdx.x] = acc;
}

// grid (n_split, Hkv / HPC); warp w of split s takes tiles s*per + w + NWK*k and
// copies HPC heads' tiles (contiguous in the page) per tile
template <int S, int HPC, int NWK>
__global__ void __launch_bounds__(NWK * 32, 1)
    paged_kernel(const uint8_t* __restrict__ hist, const int* __restrict__ pt, int ntiles, int per_split,
                 int Hkv, unsigned* out, int* err) {
  constexpr int CB = HPC * TB;
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + NWK * S * CB);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t* ring = sm + (size_t)warp * S * CB;
  uint64_t* wbar = bars + warp * S;
  if (lane < S) mbar_init(wbar + lane, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();
  const int g0 = blockIdx.y * HPC;
  const int t_begin = blockIdx.x * per_split;
  const int t_end = min(ntiles, t_begin + per_split);
  const size_t page_bytes = (size_t)Hkv * TB;
  auto issue = [&](int t, int st) {
    if (lane == 0 && t < t_end) {
      const int pid = __ldg(pt + t);
      mbar_expect_tx(wbar + st, CB);
      bulk_g2s(ring + st * CB, hist + (size_t)pid * page_bytes + (size_t)g0 * TB, CB, wbar + st);
    }
  };
#pragma unroll
  for (int st = 0; st < S - 1; ++st) issue(t_begin + warp + NWK * st, st);
  unsigned acc = 0;
  int k = 0;
  bool ok = true;
  for (int t = t_begin + warp; t < t_end; t += NWK, ++k) {
    __syncwarp();
    issue(t + NWK * (S - 1), (k + S - 1) % S);
    const int st = k % S;
    if (!__all_sync(0xffffffffu, mbar_wait(wbar + st, (k / S) & 1, 1 << 20))) {
      ok = false;
      break;
    }
    const uint4 v = *reinterpret_cast<const uint4*>(ring + st * CB + 16 * lane);
    acc ^= v.x ^ v.w;
  }
  if (!ok) {
    if (lane == 0) atomicExch(err, 1);
    for (int kk = k; kk < k + S && t_begin + warp + NWK * kk < t_end; ++kk)
      mbar_wait(wbar + kk % S, (kk / S) & 1, 1 << 20);
  }
  __syncwarp();
  if (lane < S) mbar_inval(wbar + lane);
  if (acc == 0x12345678u) out[blockIdx.x] = acc;
}

struct Timer {
  cudaEvent_t a, b;
  Timer() { CK(cudaEventCreate(&a)); CK(cudaEventCreate(&b)); }
};

int main(int argc, char** argv) {
  const int Hkv = 8, ntiles = 6230, n_split = 18;
  const size_t hist_bytes = (size_t)ntiles * Hkv * TB;
  uint8_t* hist;
  CK(cudaMalloc(&hist, hist_bytes));
  CK(cudaMemset(hist, 1, hist_bytes));
  std::vector<int> perm(ntiles);
  for (int i = 0; i < ntiles; ++i) perm[i] = i;
  std::mt19937 rng(7);
  std::shuffle(perm.begin(), perm.end(), rng);
  int* pt;
  CK(cudaMalloc(&pt, ntiles * sizeof(int)));
  CK(cudaMemcpy(pt, perm.data(), ntiles * sizeof(int), cudaMemcpyHostToDevice));
  unsigned* out;
  int* err;
  CK(cudaMalloc(&out, 4096 * sizeof(unsigned)));
  CK(cudaMalloc(&err, sizeof(int)));
  CK(cudaMemset(err, 0, sizeof(int)));
  const size_t flush_bytes = 256u << 20;
  uint8_t* fl;
  CK(cudaMalloc(&fl, 2 * flush_bytes));
  int nsm = 0;
  CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0));
  auto flush = [&]() {
    CK(cudaMemsetAsync(fl, 0, flush_bytes));
    contig_kernel<<<nsm * 4, 512>>>(reinterpret_cast<const uint4*>(fl + flush_bytes), flush_bytes / 16, out);
  };
  std::vector<cudaEvent_t> ev(2 * 20);
  for (auto& e : ev) CK(cudaEventCreate(&e));
  auto run = [&](const char* name, auto launch, size_t bytes) {
    for (int cold = 1; cold >= 0; --cold) {
      for (int it = 0; it < 3; ++it) { if (cold) flush(); launch(); }
      for (int it = 0; it < 20; ++it) {
        if (cold) flush();
        CK(cudaEventRecord(ev[2 * it]));
        launch();
        CK(cudaEventRecord(ev[2 * it + 1]));
      }
      CK(cudaDeviceSynchronize());
      CK(cudaGetLastError());
      std::vector<float> ts;
      for (int it = 0; it < 20; ++it) {
        float ms;
        CK(cudaEventElapsedTime(&ms, ev[2 * it], ev[2 * it + 1]));
        ts.push_back(ms * 1000.f);
      }
      std::sort(ts.begin(), ts.end());
      const float med = ts[ts.size() / 2], p10 = ts[ts.size() / 10];
      printf("%-16s %-5s median %8.2f us  p10 %8.2f us  %8.1f GB/s (median)\n", name, cold ? "cold" : "warm",
             med, p10, bytes / (med * 1e-6) / 1e9);
      fflush(stdout);
    }
  };
  run("empty", [&]() { empty_kernel<<<nsm, 512>>>(nullptr); }, 0);
  run("contig", [&]() {
    contig_kernel<<<nsm * 2, 512>>>(reinterpret_cast<const uint4*>(hist), hist_bytes / 16, out);
  }, hist_bytes);
  run("contig x4", [&]() {
    contig_kernel<<<nsm * 4, 512>>>(reinterpret_cast<const uint4*>(hist), hist_bytes / 16, out);
  }, hist_bytes);
  int* pt_lin;
  {
    std::vector<int> lin(ntiles);
    for (int i = 0; i < ntiles; ++i) lin[i] = i;
    CK(cudaMalloc(&pt_lin, ntiles * sizeof(int)));
    CK(cudaMemcpy(pt_lin, lin.data(), ntiles * sizeof(int), cudaMemcpyHostToDevice));
  }
  // 144 CTAs in every variant: (n_split x HPC splits) x (Hkv / HPC) head groups
  auto paged = [&](auto kern, int S, int HPC, int NWK, const int* table, const char* name) {
    const size_t smem = (size_t)NWK * S * HPC * TB + NWK * S * 8;
    const int ns = n_split * HPC;
    const int per = (ntiles + ns - 1) / ns;
    CK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    run(name, [&]() { kern<<<dim3(ns, Hkv / HPC), NWK * 32, smem>>>(hist, table, ntiles, per, Hkv, out, err); },
        hist_bytes);
  };
  paged(paged_kernel<4, 1, 16>, 4, 1, 16, pt, "paged S4 h1");
  paged(paged_kernel<8, 1, 16>, 8, 1, 16, pt, "paged S8 h1");
  paged(paged_kernel<4, 1, 16>, 4, 1, 16, pt_lin, "linear S4 h1");
  paged(paged_kernel<4, 2, 16>, 4, 2, 16, pt, "paged S4 h2");
  paged(paged_kernel<3, 4, 16>, 3, 4, 16, pt, "paged S3 h4");
  paged(paged_kernel<3, 8, 8>, 3, 8, 8, pt, "paged S3 h8 w8");
  paged(paged_kernel<2, 8, 8>, 2, 8, 8, pt, "paged S2 h8 w8");
  paged(paged_kernel<8, 1, 8>, 8, 1, 8, pt, "paged S8 h1 w8");
  int h_err = 0;
  CK(cudaMemcpy(&h_err, err, sizeof(int), cudaMemcpyDeviceToHost));
  printf("timeouts: %d\n", h_err);
  return 0;
}
