// splitkv_combine.cuh -- merge of split-KV partial attention results.
//
// The online-softmax algebra of the FlashAttention-3 deep dive
// (techknowgenie.com/posts/109164421204410442, sections 2 and 3: running max
// and sum, rescaling when the max changes) applied across key ranges instead
// of across tiles: if key range s gives the normalised output O_s and the
// log-sum-exp LSE_s of its scores, the whole row has
//     LSE = ln sum_s exp(LSE_s),    O = sum_s exp(LSE_s - LSE) * O_s,
// with empty ranges (LSE_s = -inf) contributing nothing; a row whose ranges
// are all empty gets O = 0 and LSE = -inf.
//
// One warp per query row; lane l owns d / 32 consecutive columns. HBM-bound:
// per row it reads nsplit * (d + 1) fp32 and writes d 16-bit values + 1 fp32.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace attnb3 {

constexpr int COMBINE_THREADS = 256;  // 8 rows per block
constexpr float LOG2E_F = 1.4426950408889634f;

template <int D, bool F16>
__global__ void __launch_bounds__(COMBINE_THREADS)
    splitkv_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                           uint16_t* __restrict__ o, float* __restrict__ lse, int B, int Hq,
                           int Sq, int nsplit) {
  constexpr int PER_LANE = D / 32;  // 4 (d = 128) or 2 (d = 64)
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(B) * Hq * Sq;
  const long long r = static_cast<long long>(blockIdx.x) * (COMBINE_THREADS / 32) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const long long stride = rows;  // between splits, in rows

  // LSE over the ranges (in log2 units), lanes striding over the splits
  float m = -INFINITY;
  for (int s = lane; s < nsplit; s += 32) m = fmaxf(m, lse_part[s * stride + r]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float acc[PER_LANE];
#pragma unroll
  for (int c = 0; c < PER_LANE; ++c) acc[c] = 0.f;
  float lse_row = -INFINITY;
  if (m != -INFINITY) {
    const float m2 = m * LOG2E_F;
    float sum = 0.f;
    for (int s = lane; s < nsplit; s += 32) sum += exp2f(lse_part[s * stride + r] * LOG2E_F - m2);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    const float lse2 = m2 + log2f(sum);  // log2 of the row's sum of exponentials
    lse_row = lse2 / LOG2E_F;
    for (int s = 0; s < nsplit; ++s) {
      const float ls = lse_part[s * stride + r];
      if (ls == -INFINITY) continue;
      const float wgt = exp2f(ls * LOG2E_F - lse2);
      const float* src = o_part + (s * stride + r) * D + lane * PER_LANE;
      if constexpr (PER_LANE == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] = fmaf(wgt, x.x, acc[0]);
        acc[1] = fmaf(wgt, x.y, acc[1]);
        acc[2] = fmaf(wgt, x.z, acc[2]);
        acc[3] = fmaf(wgt, x.w, acc[3]);
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(wgt, x.x, acc[0]);
        acc[1] = fmaf(wgt, x.y, acc[1]);
      }
    }
  }
  // r = (b * Hq + hq) * Sq + i; O is [B, Sq, Hq, d]
  const long long i = r % Sq;
  const long long bh = r / Sq;
  const long long hq = bh % Hq, b = bh / Hq;
  uint16_t* dst = o + ((b * Sq + i) * Hq + hq) * D + lane * PER_LANE;
  uint32_t pk[PER_LANE / 2];
#pragma unroll
  for (int c = 0; c < PER_LANE / 2; ++c)
    pk[c] = F16 ? pack_f16x2(acc[2 * c], acc[2 * c + 1]) : pack_bf16x2(acc[2 * c], acc[2 * c + 1]);
  if constexpr (PER_LANE == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
  else *reinterpret_cast<uint32_t*>(dst) = pk[0];
  if (lane == 0) lse[r] = lse_row;
}

}  // namespace attnb3
