// mufu_rate.cu -- throughput microbenchmark of the MUFU exp2 instruction the
// softmax uses (ex2.approx.ftz.f32), part of the self-test library.
//
// One CTA of 1024 threads per SM; each thread runs 8 independent chains
// x <- -2^x (x stays in (-1, -0.5), so every step is one ex2 whose result feeds
// the next through a sign modifier) for `iters` rounds between two clock64
// reads. 32 warps x 8 chains keep the pipe saturated, so the count per CTA
// divided by its cycle count is the SM's ex2 throughput per clock. Each CTA
// writes its cycle count to cycles[blockIdx.x].
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_b300.h"
#include "ptx.cuh"

namespace {

constexpr int kThreads = 1024;
constexpr int kChains = 8;

__global__ void __launch_bounds__(kThreads, 1)
    ex2_rate_kernel(int iters, unsigned long long* cycles, float* sink) {
  float x[kChains];
#pragma unroll
  for (int k = 0; k < kChains; ++k) x[k] = -0.5f - 0.0001f * static_cast<float>(threadIdx.x % 97 + k);
  __syncthreads();
  const long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < kChains; ++k) x[k] = -attnb3::ex2_approx(x[k]);
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kChains; ++k) s += x[k];
  if (s > 0.f) sink[threadIdx.x] = s;  // never true (every x < 0); keeps the chains live
  if (threadIdx.x == 0) cycles[blockIdx.x] = static_cast<unsigned long long>(t1 - t0);
}

}  // namespace

extern "C" {

// Launches one CTA per SM (num_ctas CTAs) on `stream` and synchronises it.
//   iters   : rounds per thread (each round is 8 ex2 per thread)
//   cycles  : device array of num_ctas entries, written with each CTA's cycles
//   sink    : device array of 1024 floats (never written in practice)
// ex2 per clock on an SM = 1024 * 8 * iters / cycles[i].
// Returns ATTN_OK, ATTN_ERR_INVALID_ARG or ATTN_ERR_CUDA.
int attn_selftest_ex2_rate(int iters, int num_ctas, unsigned long long* cycles, float* sink,
                           attn_stream_t stream) {
  if (iters <= 0 || num_ctas <= 0 || !cycles || !sink) return ATTN_ERR_INVALID_ARG;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ex2_rate_kernel<<<num_ctas, kThreads, 0, st>>>(iters, cycles, sink);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"
