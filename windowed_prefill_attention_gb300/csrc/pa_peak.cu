// Throughput probe of the tensor-core instructions an int8 attention could use
// on sm_103a, for the roofline the benchmark reports against ("fraction of the
// dense int8 tensor roofline").  sm_103a has no integer tcgen05 MMA, so the
// only true-int8 tensor instruction is the warp-level mma.sync s8 form; its
// fp16 form is timed beside it for comparison.  Built into its own library
// (libpa_peak.so), not into the attention library.
//
// Each warp runs kChains independent accumulator chains of one MMA shape over
// fixed register operands, so the tensor pipe, not a dependency, sets the rate.
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/pa_peak.h"

namespace {

constexpr int kChains = 8;
constexpr int kWarps = 8;

__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// operands from memory (so nothing folds), results summed into one word per thread
__global__ void __launch_bounds__(kWarps * 32) loop_s8(const uint32_t* src, long long iters, uint32_t* sink) {
  const int lane = threadIdx.x & 31;
  uint32_t a[4], b[2];
  for (int i = 0; i < 4; ++i) a[i] = src[(lane + 7 * i) & 63];
  for (int i = 0; i < 2; ++i) b[i] = src[(lane + 11 * i + 3) & 63];
  int d[kChains][4] = {};
  for (long long it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) mma_s8(d[c], a, b);
  }
  uint32_t s = 0;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += (uint32_t)(d[c][0] ^ d[c][1] ^ d[c][2] ^ d[c][3]);
  sink[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void __launch_bounds__(kWarps * 32) loop_f16(const uint32_t* src, long long iters, uint32_t* sink) {
  const int lane = threadIdx.x & 31;
  uint32_t a[4], b[2];
  for (int i = 0; i < 4; ++i) a[i] = src[(lane + 7 * i) & 63] & 0x3bff3bffu;  // finite fp16 pairs below 1
  for (int i = 0; i < 2; ++i) b[i] = src[(lane + 11 * i + 3) & 63] & 0x3bff3bffu;
  float d[kChains][4] = {};
  for (long long it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) mma_f16(d[c], a, b);
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += d[c][0] + d[c][1] + d[c][2] + d[c][3];
  sink[blockIdx.x * blockDim.x + threadIdx.x] = __float_as_uint(s);
}

}  // namespace

extern "C" int pa_peak_mma_sync(int kind, int blocks_per_sm, long long iters, double* tops, double* ms) {
  if ((kind != PA_PEAK_S8 && kind != PA_PEAK_F16) || blocks_per_sm < 1 || blocks_per_sm > 8 || iters < 1 || !tops)
    return -1;
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -3;
  const int blocks = n_sm * blocks_per_sm, threads = kWarps * 32;
  uint32_t *src = nullptr, *sink = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  int rc = -3;
  if (cudaMalloc(&src, 64 * sizeof(uint32_t)) == cudaSuccess &&
      cudaMalloc(&sink, (size_t)blocks * threads * sizeof(uint32_t)) == cudaSuccess &&
      cudaMemset(src, 0x35, 64 * sizeof(uint32_t)) == cudaSuccess && cudaEventCreate(&e0) == cudaSuccess &&
      cudaEventCreate(&e1) == cudaSuccess) {
    auto launch = [&](long long n) {
      if (kind == PA_PEAK_S8) loop_s8<<<blocks, threads>>>(src, n, sink);
      else loop_f16<<<blocks, threads>>>(src, n, sink);
    };
    launch(iters / 16 + 1);  // warm-up (clocks, module load)
    cudaEventRecord(e0);
    launch(iters);
    cudaEventRecord(e1);
    float t = 0.f;
    if (cudaEventSynchronize(e1) == cudaSuccess && cudaGetLastError() == cudaSuccess &&
        cudaEventElapsedTime(&t, e0, e1) == cudaSuccess && t > 0.f) {
      // ops of one MMA: 2 M N K; s8 m16n8k32, f16 m16n8k16
      const double per_mma = kind == PA_PEAK_S8 ? 2.0 * 16 * 8 * 32 : 2.0 * 16 * 8 * 16;
      const double ops = per_mma * kChains * (double)iters * (double)blocks * kWarps;
      *tops = ops / (t * 1e-3) / 1e12;
      if (ms) *ms = t;
      rc = 0;
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (src) cudaFree(src);
  if (sink) cudaFree(sink);
  return rc;
}
