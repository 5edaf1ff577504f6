// selftest_umma.cu -- libattn_selftest.so: one-tile checks of the two tensor-
// core contractions the attention kernel issues, through the same helpers
// (tensor maps, shared-memory descriptors, instruction descriptors, TMEM
// layout of P). Used only by the test-suite to localise a layout mistake to a
// single MMA form; the attention library does not depend on it.
//
//   form 0 ("QK"): D[128 x 128] = A[128 x d] * B[128 x d]^T, A and B staged by
//                  TMA K-major (the S = Q K^T step);
//   form 1 ("PV"): D[128 x d]   = A[128 x 128] * B[128 x d], A written to
//                  tensor memory by the threads (the P operand), B staged by
//                  TMA with d contiguous (the O += P V step). For E4M3, A is
//                  fp16 (as the kernel keeps P) and B is staged as E4M3 codes
//                  and widened to fp16 in shared memory first, as the kernel
//                  does.
// d = 128; element type bf16 or E4M3. D is returned as fp32 row-major.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_b300.h"
#include "attn_fwd_kernel.cuh"
#include "tmap.cuh"

namespace {

using namespace attnb3;

constexpr int ST_THREADS = 128;
constexpr unsigned long long ST_LIMIT_NS = 1000000000ull;

__device__ __forceinline__ bool st_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > ST_LIMIT_NS) return false;
  return true;
}

template <bool FP8, int FORM>
__global__ void __launch_bounds__(ST_THREADS, 1)
    umma_selftest_kernel(const __grid_constant__ CUtensorMap tm_a,
                         const __grid_constant__ CUtensorMap tm_b, const uint8_t* a_raw,
                         float* out, int* err) {
  constexpr int D = 128;
  using C = Cfg<D, FP8, false>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t a_smem = sbase;                    // Q-tile sized region
  const uint32_t b_smem = sbase + C::Q_TILE_BYTES;  // K/V-tile sized region
  const uint32_t vf_smem = sbase + 64 * 1024;       // E4M3 PV form: widened V
  const uint32_t bar_load = sbase + 96 * 1024;
  const uint32_t bar_mma = bar_load + 8;
  volatile uint32_t* tmem_holder =
      reinterpret_cast<volatile uint32_t*>(smem + 96 * 1024 + 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_holder)), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);

  if (FORM == 1) {
    // P operand: row = thread, 128 keys packed into tensor-memory columns
    // starting at column 128, exactly as the softmax writes it.
    const int row = threadIdx.x;
    if constexpr (!FP8) {
      const __nv_bfloat16* ar = reinterpret_cast<const __nv_bfloat16*>(a_raw) + row * 128;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c)
          pk[c] = pack_bf16x2(__bfloat162float(ar[64 * i + 2 * c]),
                              __bfloat162float(ar[64 * i + 2 * c + 1]));
        tmem_st32(t_lane + 128 + 32 * i, pk);
      }
    } else {
      // fp16 P (the FP8 path keeps P in fp16): raw bits, packed like bf16
      const uint16_t* ar = reinterpret_cast<const uint16_t*>(a_raw) + row * 128;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c)
          pk[c] = static_cast<uint32_t>(ar[64 * h + 2 * c]) |
                  (static_cast<uint32_t>(ar[64 * h + 2 * c + 1]) << 16);
        tmem_st32(t_lane + 128 + 32 * h, pk);
      }
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();

  bool ok = true;
  if (threadIdx.x == 0) {
    tc_fence_after();
    const uint32_t bytes = (FORM == 0 ? C::Q_TILE_BYTES : 0) + C::KV_TILE_BYTES;
    mbar_arrive_expect_tx(bar_load, bytes);
#pragma unroll
    for (int c = 0; c < C::NCHUNK; ++c) {
      if (FORM == 0)
        tma_load_4d(a_smem + c * C::Q_CHUNK_BYTES, &tm_a, bar_load, c * C::CHUNK_ELEMS, 0, 0, 0);
      tma_load_4d(b_smem + c * C::KV_CHUNK_BYTES, &tm_b, bar_load, c * C::CHUNK_ELEMS, 0, 0, 0);
    }
  }
  // every thread: the staged tiles have landed (FP8 PV form: widen V to fp16)
  const bool landed = st_wait(bar_load, 0);
  if (FP8 && FORM == 1 && landed) {
    widen_v_tile<D>(b_smem, vf_smem, threadIdx.x, ST_THREADS);
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ok = landed;
    if (ok) {
      tc_fence_after();
      if (FORM == 0) issue_qk<D, FP8>(tmem, a_smem, b_smem);
      else issue_pv<D, FP8>(tmem, tmem + 128, FP8 ? vf_smem : b_smem, false);
      tc_commit(bar_mma);
      ok = st_wait(bar_mma, 0);
    }
    if (!ok) atomicExch(err, 1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // D row = thread; 128 fp32 columns
  const int row = threadIdx.x;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t r[32];
    tmem_ld32(t_lane + 32 * i, r);
#pragma unroll
    for (int c = 0; c < 32; ++c) out[row * 128 + 32 * i + c] = __uint_as_float(r[c]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
  (void)lane;
}

template <bool FP8, int FORM>
int run_selftest(const void* a, const void* b, float* out, int* err, cudaStream_t stream) {
  using C = Cfg<128, FP8>;
  CUtensorMap ta, tb;
  // A: 128 rows x 128 columns (FORM 0) -- one [1, 128, 1, 128] tensor
  // B: 128 rows x 128 columns
  if (!encode_bshd(&ta, a, FP8, 1, 128, 1, 128, C::CHUNK_ELEMS, 128) ||
      !encode_bshd(&tb, b, FP8, 1, 128, 1, 128, C::CHUNK_ELEMS, 128))
    return ATTN_ERR_CUDA;
  const int smem = C::SMEM_ALLOC;  // generous: every operand window stays inside
  auto kern = umma_selftest_kernel<FP8, FORM>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return ATTN_ERR_CUDA;
  kern<<<1, ST_THREADS, smem, stream>>>(ta, tb, static_cast<const uint8_t*>(a), out, err);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

// form: 0 = QK form, 1 = PV form; fp8: 0 = bf16, 1 = E4M3. a, b: device,
// 128 x 128 row-major (a: fp16 bits for the E4M3 PV form); out: device
// fp32 128 x 128; err: device int set to 1 if a wait timed out. Returns an
// attn_status_t.
int attn_selftest_umma(int form, int fp8, const void* a, const void* b, float* out, int* err,
                       attn_stream_t stream) {
  int dev = 0, major = 0, minor = 0;
  if (!a || !b || !out || !err) return ATTN_ERR_INVALID_ARG;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;
  if (!get_encoder()) return ATTN_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (form == 0 && !fp8) return run_selftest<false, 0>(a, b, out, err, s);
  if (form == 1 && !fp8) return run_selftest<false, 1>(a, b, out, err, s);
  if (form == 0 && fp8) return run_selftest<true, 0>(a, b, out, err, s);
  if (form == 1 && fp8) return run_selftest<true, 1>(a, b, out, err, s);
  return ATTN_ERR_INVALID_ARG;
}

}  // extern "C"
