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
// L1/L2). One warp per token; the first pass sums the squares in fp32, the
// second re-reads the row (an L1 hit: the warp read it just before), scales
// it and writes y rounded to nearest in the storage type.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace attnb3 {

constexpr int NORM_THREADS = 256;  // 8 tokens per block
constexpr int NORM_TOKENS_PER_BLOCK = NORM_THREADS / 32;

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
  // q_out may be q and k_out may be k (in place): each lane reads a chunk in
  // both passes before it writes that chunk, and the warp-wide reduction
  // between the passes orders every read of pass 1 before any write.
  const bool is_q = blockIdx.y == 0;
  const long long t = static_cast<long long>(blockIdx.x) * NORM_TOKENS_PER_BLOCK + (threadIdx.x >> 5);
  if (t >= (is_q ? tq : tk)) return;
  const int lane = threadIdx.x & 31;
  const int n = is_q ? nq : nk;  // H * d, a multiple of 64
  const int chunks = n / 8;      // 16-byte chunks per token
  const uint4* x = reinterpret_cast<const uint4*>((is_q ? q : k) + t * n);
  const uint4* w = reinterpret_cast<const uint4*>(is_q ? wq : wk);
  uint4* y = reinterpret_cast<uint4*>((is_q ? q_out : k_out) + t * n);

  float ss = 0.f;
  for (int c = lane; c < chunks; c += 32) {
    float f[8];
    unpack8<F16>(x[c], f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float r = rsqrtf(eps + ss / static_cast<float>(n));

  for (int c = lane; c < chunks; c += 32) {
    float f[8], g[8];
    unpack8<F16>(x[c], f);
    unpack8<F16>(w[c], g);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = f[2 * i] * r * g[2 * i], b = f[2 * i + 1] * r * g[2 * i + 1];
      o[i] = F16 ? pack_f16x2(a, b) : pack_bf16x2(a, b);
    }
    y[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace attnb3
