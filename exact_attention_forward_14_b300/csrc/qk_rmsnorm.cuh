// qk_rmsnorm.cuh -- RMSNorm of Q and K across heads, the prologue of the
// attention forward pass.
//
// "QKNorm across heads" (SGLang PR 21503 analysis, secrett2633 blog): each
// token's whole hidden vector (all H heads x d) shares one RMS,
//     y[t, h, c] = x[t, h, c] * rsqrt(eps + mean_{h', c'} x[t, h', c']^2) * w[h d + c],
// with separate weights for Q and K; the page's kernel splits Q and K over
// the second grid dimension so each block holds one tensor's state only.
// Here too blockIdx.y selects Q (0) or K (1).
//
// HBM-bound: 2 bytes read and 2 written per element (the weights stay in
// L1/L2). One 128-thread block per token: each thread loads its 16-byte
// chunks of the row once and keeps them in registers (rows up to 8192
// elements), the block sums the squares in fp32 (warp shuffles, then shared
// memory), and every thread scales its chunks and writes y rounded to nearest
// in the storage type. Longer rows re-read their chunks in the second pass.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace attnb3 {

constexpr int NORM_THREADS = 128;  // one token per block
constexpr int NORM_CACHE = 8;      // 16-byte chunks a thread keeps in registers

template <bool F16>
__device__ __forceinline__ float half_to_float(uint32_t bits16) {
  if constexpr (F16) return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
  else return __uint_as_float(bits16 << 16);
}

// 8 packed 16-bit values -> 8 floats
template <bool F16>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = half_to_float<F16>(w[i] & 0xFFFFu);
    f[2 * i + 1] = half_to_float<F16>(w[i] >> 16);
  }
}

template <bool F16>
__global__ void __launch_bounds__(NORM_THREADS)
    qk_rmsnorm_kernel(const uint16_t* q, const uint16_t* k, const uint16_t* __restrict__ wq,
                      const uint16_t* __restrict__ wk, uint16_t* q_out, uint16_t* k_out,
                      long long tq, long long tk, int nq, int nk, float eps) {
  // q_out may be q and k_out may be k (in place): every thread reads its
  // chunks before the block-wide reduction and writes them after it.
  __shared__ float part[NORM_THREADS / 32];
  const bool is_q = blockIdx.y == 0;
  const long long t = blockIdx.x;
  if (t >= (is_q ? tq : tk)) return;  // uniform over the block
  const int n = is_q ? nq : nk;      // H * d, a multiple of 64
  const int chunks = n / 8;          // 16-byte chunks per token
  const uint4* x = reinterpret_cast<const uint4*>((is_q ? q : k) + t * n);
  const uint4* w = reinterpret_cast<const uint4*>(is_q ? wq : wk);
  uint4* y = reinterpret_cast<uint4*>((is_q ? q_out : k_out) + t * n);
  const int tid = threadIdx.x;

  uint4 keep[NORM_CACHE];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < NORM_CACHE; ++i) {
    const int c = tid + i * NORM_THREADS;
    if (c < chunks) keep[i] = x[c];
  }
#pragma unroll
  for (int i = 0; i < NORM_CACHE; ++i) {
    const int c = tid + i * NORM_THREADS;
    if (c < chunks) {
      float f[8];
      unpack8<F16>(keep[i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
    }
  }
  for (int c = tid + NORM_CACHE * NORM_THREADS; c < chunks; c += NORM_THREADS) {
    float f[8];
    unpack8<F16>(x[c], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((tid & 31) == 0) part[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < NORM_THREADS / 32; ++i) tot += part[i];
  const float r = rsqrtf(eps + tot / static_cast<float>(n));

  auto emit = [&](int c, const uint4& v) {
    float f[8], g[8];
    unpack8<F16>(v, f);
    unpack8<F16>(w[c], g);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = f[2 * i] * r * g[2 * i], b = f[2 * i + 1] * r * g[2 * i + 1];
      o[i] = F16 ? pack_f16x2(a, b) : pack_bf16x2(a, b);
    }
    y[c] = make_uint4(o[0], o[1], o[2], o[3]);
  };
#pragma unroll
  for (int i = 0; i < NORM_CACHE; ++i) {
    const int c = tid + i * NORM_THREADS;
    if (c < chunks) emit(c, keep[i]);
  }
  for (int c = tid + NORM_CACHE * NORM_THREADS; c < chunks; c += NORM_THREADS) emit(c, x[c]);
}

}  // namespace attnb3
