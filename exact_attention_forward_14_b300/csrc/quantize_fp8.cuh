// quantize_fp8.cuh -- FP8 E4M3 block quantiser (one CTA per scale block).
//
// FlashAttention-3 deep dive (techknowgenie.com/posts/109164421204410442),
// section "FP8 low-precision arithmetic and numerical stability", sub-section
// "block quantisation and dynamic scaling": each small block keeps its own
// scale factor taken from the block's local maximum, so an outlier only
// coarsens its own block. Here a block is 64 consecutive sequence rows of one
// head times all d columns; s = amax / 448 (448 = largest finite E4M3), s = 1
// for an all-zero block; code = round-to-nearest-even, saturating E4M3 of
// x / s with the division done in IEEE fp32.
//
// Memory-bound: reads 4 bytes and writes 1 byte per element (plus one fp32
// scale per block). Each thread keeps its share of the block in registers
// between the max and the encode, so every element is read from HBM once.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace attnb3 {

constexpr int QUANT_THREADS = 256;
constexpr int QUANT_BLOCK_ROWS = 64;

template <int D>
__global__ void __launch_bounds__(QUANT_THREADS)
    quantize_fp8_kernel(const float* __restrict__ x, uint8_t* __restrict__ codes,
                        float* __restrict__ scale, int S, int H, int nblk) {
  constexpr int VPR = D / 4;                                 // float4 per row
  constexpr int VPT = QUANT_BLOCK_ROWS * VPR / QUANT_THREADS;  // float4 per thread
  static_assert(VPT * QUANT_THREADS == QUANT_BLOCK_ROWS * VPR, "whole block per CTA");
  __shared__ float warp_max[QUANT_THREADS / 32];
  const int blk = blockIdx.x % nblk;
  const int bh = blockIdx.x / nblk;
  const int h = bh % H;
  const int b = bh / H;
  const int r0 = blk * QUANT_BLOCK_ROWS;
  const int rows = min(QUANT_BLOCK_ROWS, S - r0);
  const size_t row_stride = static_cast<size_t>(H) * D;
  const size_t base = (static_cast<size_t>(b) * S + r0) * row_stride + static_cast<size_t>(h) * D;

  float4 v[VPT];
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {  // all loads in flight together
    const int i = threadIdx.x + k * QUANT_THREADS;
    const int r = i / VPR, c = (i - r * VPR) * 4;
    v[k] = r < rows ? *reinterpret_cast<const float4*>(x + base + r * row_stride + c)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int k = 0; k < VPT; ++k)
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[k].x), fabsf(v[k].y)),
                             fmaxf(fabsf(v[k].z), fabsf(v[k].w))));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  float m = warp_max[0];
#pragma unroll
  for (int w = 1; w < QUANT_THREADS / 32; ++w) m = fmaxf(m, warp_max[w]);
  const float s = (m == 0.f) ? 1.f : __fdiv_rn(m, 448.f);
  if (threadIdx.x == 0) scale[blockIdx.x] = s;  // [B, H, nblk] == blockIdx order

#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int i = threadIdx.x + k * QUANT_THREADS;
    const int r = i / VPR, c = (i - r * VPR) * 4;
    if (r < rows) {
      const uint32_t q = pack_e4m3x4(__fdiv_rn(v[k].x, s), __fdiv_rn(v[k].y, s),
                                     __fdiv_rn(v[k].z, s), __fdiv_rn(v[k].w, s));
      *reinterpret_cast<uint32_t*>(codes + base + r * row_stride + c) = q;
    }
  }
}

}  // namespace attnb3
