// attn_api.cu -- host side of libattn_b300.so: argument validation, TMA
// tensor-map encoding, launch of the fused attention kernels (forward,
// split-KV merge, backward), the QK-RMSNorm prologue and the FP8 block
// quantiser, and the device status word.
//
// The C ABI is declared (with argument meaning, layouts, ownership and error
// behaviour) in include/attn_b300.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_b300.h"
#include "attn_bwd_kernel.cuh"
#include "attn_fwd_d256.cuh"
#include "attn_fwd_kernel.cuh"
#include "quantize_fp8.cuh"
#include "qk_rmsnorm.cuh"
#include "splitkv_combine.cuh"
#include "tmap.cuh"

namespace {

using attnb3::Cfg;
using attnb3::FwdParams;
using attnb3::encode_bshd;
using attnb3::get_encoder;

// Device status word written by the kernels' watchdog (ATTN_ERR_TIMEOUT).
__device__ int g_attn_status = 0;

constexpr int kMaxDevices = 64;
constexpr unsigned long long kWaitLimitDefaultNs = 1000000000ull;  // 1 s per wait
constexpr unsigned long long kWaitLimitMinNs = 1000000ull;            // 1 ms
constexpr unsigned long long kWaitLimitMaxNs = 3600000000000ull;      // 1 h
// Limit of every bounded wait in the kernels, read at each launch.
std::atomic<unsigned long long> g_wait_limit_ns{kWaitLimitDefaultNs};

unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
constexpr int kMaxSplits = 256;  // key ranges per split-KV call
// Backward: share of the SMs given to the dK/dV kernel while the dQ kernel
// runs beside it (the two kernels' times alone on all SMs were 1.51 and
// 1.07 ms on B2 H32 S8192 d128 causal: 0.585 of the sum).
constexpr int kBwdKvShareNum = 585;
constexpr int kBwdKvShareDen = 1000;

struct DeviceInfo {
  std::once_flag once;
  int ok = 0;  // 1 = usable sm_103 device
  int num_sms = 0;
  int* status = nullptr;
  std::atomic<uint32_t> attr_done{0};  // bit per kernel instantiation
  // backward: a second stream for the dQ kernel, forked from and joined back
  // into the caller's stream with two events (created on the first attn_bwd
  // call; side == nullptr if that failed: then both kernels go on the
  // caller's stream one after the other)
  std::once_flag side_once;
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex side_mu;  // one fork / join sequence at a time per device
};
DeviceInfo g_dev[kMaxDevices];

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks on the current device, done once per device.
int current_device(DeviceInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  DeviceInfo& di = g_dev[dev];
  std::call_once(di.once, [&] {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      di.ok = -1;
      return;
    }
    if (major != 10 || minor != 3) {
      di.ok = 0;
      return;
    }
    void* st = nullptr;
    if (cudaGetSymbolAddress(&st, g_attn_status) != cudaSuccess) {
      di.ok = -1;
      return;
    }
    di.status = static_cast<int*>(st);
    di.num_sms = sms;
    di.ok = 1;
  });
  if (di.ok < 0) return ATTN_ERR_CUDA;
  if (di.ok == 0) return ATTN_ERR_UNSUPPORTED;
  *out = &di;
  return ATTN_OK;
}

bool fits_i32(long long a, long long b, long long c, long long d) {
  const long long lim = 0x7fffffffLL;
  long long x = a;
  for (long long f : {b, c, d}) {
    if (x > lim / f) return false;
    x *= f;
  }
  return x <= lim;
}

// Key-range split of one launch: nsplit ranges of kps K/V tiles each (kps = 0:
// all tiles); partial outputs go to o_part / lse_part when those are set.
struct Split {
  int nsplit;
  int kps;
  float* o_part;
  float* lse_part;
};
constexpr Split kNoSplit = {1, 0, nullptr, nullptr};

template <int D, bool FP8, bool F16>
int launch(const void* q, const void* k, const void* v, const float* qs, const float* ks,
           const float* vs, void* o, float* lse, int B, int Hq, int Hkv, int Sq, int Sk,
           int causal, float scale, cudaStream_t stream, DeviceInfo* di, uint32_t attr_bit,
           const Split& sp) {
  using C = Cfg<D, FP8, F16>;
  auto kern = attnb3::attn_fwd_kernel<D, FP8, F16>;
  if (!(di->attr_done.load(std::memory_order_acquire) & attr_bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
    // A kernel that moves registers between its warpgroups (setmaxnreg) must
    // be launched with enough of them for the new split, or the softmax
    // warps' increase would wait forever: refuse to launch instead.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return ATTN_ERR_CUDA;
    if (static_cast<long long>(fa.numRegs) * C::THREADS < C::REGS_NEEDED) return ATTN_ERR_CUDA;
    di->attr_done.fetch_or(attr_bit, std::memory_order_acq_rel);
  }
  CUtensorMap tq, tk, tv;
  if (!encode_bshd(&tq, q, FP8, B, Sq, Hq, D, C::CHUNK_ELEMS, attnb3::BM, F16) ||
      !encode_bshd(&tk, k, FP8, B, Sk, Hkv, D, C::CHUNK_ELEMS, attnb3::BN, F16) ||
      !encode_bshd(&tv, v, FP8, B, Sk, Hkv, D, C::CHUNK_ELEMS, attnb3::BN, F16))
    return ATTN_ERR_CUDA;

  FwdParams P;
  P.o = static_cast<uint16_t*>(o);
  P.lse = lse;
  P.q_scale = qs;
  P.k_scale = ks;
  P.v_scale = vs;
  P.B = B;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.Sq = Sq;
  P.Sk = Sk;
  P.group = Hq / Hkv;
  P.n_qp = (Sq + attnb3::UNIT_ROWS - 1) / attnb3::UNIT_ROWS;
  P.npair = (P.n_qp + 1) / 2;
  P.nkv = (Sk + attnb3::BN - 1) / attnb3::BN;
  P.nsplit = sp.nsplit;
  P.kps = sp.kps > 0 ? sp.kps : P.nkv;
  P.o_part = sp.o_part;
  P.lse_part = sp.lse_part;
  P.num_items = B * Hq * P.npair * P.nsplit;
  P.causal = causal ? 1 : 0;
  P.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  P.timeout_ns = wait_limit_ns();
  P.status = di->status;

  // fewer than 4 whole items per SM leave the last round part-empty: deal
  // single units longest-first instead (see cta_unit in the kernel)
  P.lpt = (P.nsplit == 1 && P.num_items < 4 * di->num_sms) ? 1 : 0;
  const int work = P.lpt ? B * Hq * P.n_qp : P.num_items;
  const int grid = work < di->num_sms ? work : di->num_sms;
  kern<<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, P);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Argument checks shared by both attention entry points (no CUDA calls).
int check_attn_args(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int Hq, int Hkv, int Sq, int Sk, int d, float scale) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!fits_i32(B, Sq, Hq, d) || !fits_i32(B, Sk, Hkv, d)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

// d = 256 forward (bf16 / fp16): one 128-row Q tile per unit, 64-key K/V
// tiles (attn_fwd_d256.cuh).
template <bool F16>
int launch_d256(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                int Hkv, int Sq, int Sk, int causal, float scale, cudaStream_t stream,
                DeviceInfo* di, uint32_t attr_bit) {
  using C = attnb3::WideCfg<F16>;
  auto kern = attnb3::attn_fwd_d256_kernel<F16>;
  if (!(di->attr_done.load(std::memory_order_acquire) & attr_bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
    di->attr_done.fetch_or(attr_bit, std::memory_order_acq_rel);
  }
  CUtensorMap tq, tk, tv;
  if (!encode_bshd(&tq, q, false, B, Sq, Hq, attnb3::WIDE_D, C::CHUNK_ELEMS, attnb3::BM, F16) ||
      !encode_bshd(&tk, k, false, B, Sk, Hkv, attnb3::WIDE_D, C::CHUNK_ELEMS, attnb3::WIDE_BN,
                   F16) ||
      !encode_bshd(&tv, v, false, B, Sk, Hkv, attnb3::WIDE_D, C::CHUNK_ELEMS, attnb3::WIDE_VROWS,
                   F16))
    return ATTN_ERR_CUDA;
  FwdParams P{};
  P.o = static_cast<uint16_t*>(o);
  P.lse = lse;
  P.B = B;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.Sq = Sq;
  P.Sk = Sk;
  P.group = Hq / Hkv;
  P.n_qp = (Sq + attnb3::BM - 1) / attnb3::BM;
  P.npair = (P.n_qp + 1) / 2;
  P.nkv = (Sk + attnb3::WIDE_BN - 1) / attnb3::WIDE_BN;
  P.num_items = B * Hq * P.npair;
  P.causal = causal ? 1 : 0;
  P.nsplit = 1;
  P.kps = P.nkv;
  P.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  P.timeout_ns = wait_limit_ns();
  P.status = di->status;
  const int grid = P.num_items < di->num_sms ? P.num_items : di->num_sms;
  kern<<<grid, attnb3::WIDE_THREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, P);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int run_attn(const void* q, const void* k, const void* v, const float* qs, const float* ks,
             const float* vs, void* o, float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int d,
             int causal, float scale, bool fp8, bool f16, cudaStream_t stream,
             const Split& sp = kNoSplit) {
  DeviceInfo* di = nullptr;
  int rc = current_device(&di);
  if (rc != ATTN_OK) return rc;
  if (!get_encoder()) return ATTN_ERR_CUDA;
  if (d == 256) {  // bf16 / fp16, unsplit only
    if (fp8 || sp.nsplit != 1 || sp.o_part != nullptr) return ATTN_ERR_UNSUPPORTED;
    return f16 ? launch_d256<true>(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, causal, scale, stream,
                                   di, 1024u)
               : launch_d256<false>(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, causal, scale, stream,
                                    di, 2048u);
  }
  if (fp8 && d == 128)
    return launch<128, true, false>(q, k, v, qs, ks, vs, o, lse, B, Hq, Hkv, Sq, Sk, causal,
                                    scale, stream, di, 4u, sp);
  if (fp8 && d == 64)
    return launch<64, true, false>(q, k, v, qs, ks, vs, o, lse, B, Hq, Hkv, Sq, Sk, causal,
                                   scale, stream, di, 8u, sp);
  if (f16 && d == 128)
    return launch<128, false, true>(q, k, v, qs, ks, vs, o, lse, B, Hq, Hkv, Sq, Sk, causal,
                                    scale, stream, di, 16u, sp);
  if (f16 && d == 64)
    return launch<64, false, true>(q, k, v, qs, ks, vs, o, lse, B, Hq, Hkv, Sq, Sk, causal,
                                   scale, stream, di, 32u, sp);
  if (d == 128)
    return launch<128, false, false>(q, k, v, qs, ks, vs, o, lse, B, Hq, Hkv, Sq, Sk, causal,
                                     scale, stream, di, 1u, sp);
  if (d == 64)
    return launch<64, false, false>(q, k, v, qs, ks, vs, o, lse, B, Hq, Hkv, Sq, Sk, causal,
                                    scale, stream, di, 2u, sp);
  return ATTN_ERR_UNSUPPORTED;
}

// K/V tiles per range and the number of non-empty ranges for a requested
// split count.
void split_shape(int Sk, int num_splits, int* kps, int* nsplit) {
  const int nkv = (Sk + attnb3::BN - 1) / attnb3::BN;
  const int want = num_splits < nkv ? num_splits : nkv;
  *kps = (nkv + want - 1) / want;
  *nsplit = (nkv + *kps - 1) / *kps;
}

size_t splitkv_bytes(int B, int Hq, int Sq, int d, int nsplit) {
  const size_t rows = static_cast<size_t>(B) * Hq * Sq;
  return static_cast<size_t>(nsplit) * rows * static_cast<size_t>(d + 1) * sizeof(float);
}

template <int D, bool F16>
int launch_combine(const float* o_part, const float* lse_part, void* o, float* lse, int B, int Hq,
                   int Sq, int nsplit, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * Hq * Sq;
  const long long per_block = attnb3::COMBINE_THREADS / 32;
  const long long blocks = (rows + per_block - 1) / per_block;
  if (blocks > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  attnb3::splitkv_combine_kernel<D, F16>
      <<<static_cast<unsigned>(blocks), attnb3::COMBINE_THREADS, 0, stream>>>(
          o_part, lse_part, static_cast<uint16_t*>(o), lse, B, Hq, Sq, nsplit);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// ---- backward pass ---------------------------------------------------------

size_t bwd_sq_pad(int Sq) {
  return (static_cast<size_t>(Sq) + attnb3::BWD_TILE - 1) / attnb3::BWD_TILE * attnb3::BWD_TILE;
}

size_t bwd_workspace_bytes(int B, int Hq, int Sq) {
  return 2 * static_cast<size_t>(B) * Hq * bwd_sq_pad(Sq) * sizeof(float);
}

template <int D, bool F16>
int launch_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* d_o, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
               int Sk, int causal, float scale, float* ws, cudaStream_t stream, DeviceInfo* di,
               uint32_t attr_bit) {
  using C = attnb3::BwdCfg<D, F16>;
  auto kkv = attnb3::bwd_dkdv_kernel<D, F16>;
  auto kq = attnb3::bwd_dq_kernel<D, F16>;
  if (!(di->attr_done.load(std::memory_order_acquire) & attr_bit)) {
    if (cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) !=
            cudaSuccess)
      return ATTN_ERR_CUDA;
    di->attr_done.fetch_or(attr_bit, std::memory_order_acq_rel);
  }
  CUtensorMap tq, tdo, tk, tv;
  if (!encode_bshd(&tq, q, false, B, Sq, Hq, D, C::CHUNK_ELEMS, attnb3::BWD_TILE, F16) ||
      !encode_bshd(&tdo, d_o, false, B, Sq, Hq, D, C::CHUNK_ELEMS, attnb3::BWD_TILE, F16) ||
      !encode_bshd(&tk, k, false, B, Sk, Hkv, D, C::CHUNK_ELEMS, attnb3::BWD_TILE, F16) ||
      !encode_bshd(&tv, v, false, B, Sk, Hkv, D, C::CHUNK_ELEMS, attnb3::BWD_TILE, F16))
    return ATTN_ERR_CUDA;

  const size_t sq_pad = bwd_sq_pad(Sq);
  const long long rows_pad = static_cast<long long>(B) * Hq * static_cast<long long>(sq_pad);
  attnb3::BwdParams P;
  P.dq = static_cast<uint16_t*>(dq);
  P.dk = static_cast<uint16_t*>(dk);
  P.dv = static_cast<uint16_t*>(dv);
  P.nlse2 = ws;
  P.ndsum = ws + rows_pad;
  P.B = B;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.Sq = Sq;
  P.Sk = Sk;
  P.Sq_pad = static_cast<int>(sq_pad);
  P.group = Hq / Hkv;
  P.causal = causal ? 1 : 0;
  P.nq = static_cast<int>(sq_pad / attnb3::BWD_TILE);
  P.nk = (Sk + attnb3::BWD_TILE - 1) / attnb3::BWD_TILE;
  P.kv_npair = (P.nk + 1) / 2;
  P.kv_items = B * Hkv * P.kv_npair;
  P.q_npair = (P.nq + 1) / 2;
  P.q_items = B * Hq * P.q_npair;
  P.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  P.scale = scale;
  P.timeout_ns = wait_limit_ns();
  P.status = di->status;

  // row statistics: warps over the rows in memory order (D / 8 lanes per row,
  // BWD_PREP_STEPS row groups per warp), then one thread per padded entry
  const long long rows = static_cast<long long>(B) * Sq * Hq;
  const long long rows_per_warp = (32 / (D / 8)) * attnb3::BWD_PREP_STEPS;
  const long long row_warps = (rows + rows_per_warp - 1) / rows_per_warp;
  const long long pad_rows = static_cast<long long>(B) * Hq * (P.Sq_pad - Sq);
  const long long warps = row_warps + (pad_rows + 31) / 32;
  const long long per_block = attnb3::BWD_PREP_THREADS / 32;
  const long long prep_blocks = (warps + per_block - 1) / per_block;
  attnb3::bwd_prep_kernel<D, F16><<<static_cast<unsigned>(prep_blocks),
                                    attnb3::BWD_PREP_THREADS, 0, stream>>>(
      static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(d_o), lse, ws,
      ws + rows_pad, Hq, Sq, P.Sq_pad, rows, row_warps, pad_rows);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;

  // dK/dV and dQ read the same Q, dO, K and V and do not depend on each
  // other. They run side by side on disjoint sets of SMs, sized to their
  // work (dK/dV: four products per (Q tile, key tile) pair, dQ: three, at
  // slightly different efficiencies), and both deal their items head by
  // head in the same order, so the two kernels are on the same few heads at
  // any time and the second read of those heads' tiles comes from L2.
  std::call_once(di->side_once, [&] {
    cudaStream_t s = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) == cudaSuccess &&
        cudaEventCreateWithFlags(&f, cudaEventDisableTiming) == cudaSuccess &&
        cudaEventCreateWithFlags(&j, cudaEventDisableTiming) == cudaSuccess) {
      di->side = s;
      di->fork = f;
      di->join = j;
    } else {  // fall back to one stream; release whatever was created
      if (j != nullptr) cudaEventDestroy(j);
      if (f != nullptr) cudaEventDestroy(f);
      if (s != nullptr) cudaStreamDestroy(s);
      cudaGetLastError();
    }
  });
  const int sms = di->num_sms;
  int share_kv = (sms * kBwdKvShareNum + kBwdKvShareDen / 2) / kBwdKvShareDen;
  share_kv = share_kv < 1 ? 1 : (share_kv > sms - 1 ? sms - 1 : share_kv);
  if (di->side == nullptr || sms < 2) {
    const int gkv = P.kv_items < sms ? P.kv_items : sms;
    kkv<<<gkv, attnb3::BWD_THREADS, C::SMEM_ALLOC, stream>>>(tq, tdo, tk, tv, P);
    const int gq = P.q_items < sms ? P.q_items : sms;
    kq<<<gq, attnb3::BWD_THREADS, C::SMEM_ALLOC, stream>>>(tq, tdo, tk, tv, P);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  const int gkv = P.kv_items < share_kv ? P.kv_items : share_kv;
  const int gq = P.q_items < sms - share_kv ? P.q_items : sms - share_kv;
  std::lock_guard<std::mutex> lock(di->side_mu);
  if (cudaEventRecord(di->fork, stream) != cudaSuccess ||
      cudaStreamWaitEvent(di->side, di->fork, 0) != cudaSuccess)
    return ATTN_ERR_CUDA;
  kkv<<<gkv, attnb3::BWD_THREADS, C::SMEM_ALLOC, stream>>>(tq, tdo, tk, tv, P);
  kq<<<gq, attnb3::BWD_THREADS, C::SMEM_ALLOC, di->side>>>(tq, tdo, tk, tv, P);
  const cudaError_t launched = cudaGetLastError();
  // join even after a failed launch, so that the caller's stream never runs
  // ahead of work already enqueued on the second one
  const bool joined = cudaEventRecord(di->join, di->side) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, di->join, 0) == cudaSuccess;
  return (launched == cudaSuccess && joined) ? ATTN_OK : ATTN_ERR_CUDA;
}

// ---- workspace for attn_fwd_splitkv_noalloc --------------------------------
// A fixed device array in this library, so that callers who may not allocate
// device memory can still use the split-KV path. Every GPU that loads the
// library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(64) << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address, looked up per device (with that device
// current) until a lookup succeeds; in host code the array's name is only a
// stand-in for it. A failed lookup is not cached, so a transient error does
// not disable the entry point for the rest of the process.
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];

int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int Sq, int Sk, int d, int causal, float scale, int dtype,
             attn_stream_t stream) {
  int rc = check_attn_args(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, scale);
  if (rc != ATTN_OK) return rc;
  if (dtype == ATTN_BF16 || dtype == ATTN_F16)
    return run_attn(q, k, v, nullptr, nullptr, nullptr, o, lse, B, Hq, Hkv, Sq, Sk, d, causal,
                    scale, false, dtype == ATTN_F16, reinterpret_cast<cudaStream_t>(stream));
  if (dtype == ATTN_FP8_E4M3 && d == 256) return ATTN_ERR_UNSUPPORTED;
  if (dtype == ATTN_FP8_E4M3)  // null scale pointers: every block scale is 1
    return run_attn(q, k, v, nullptr, nullptr, nullptr, o, lse, B, Hq, Hkv, Sq, Sk, d, causal,
                    scale, true, false, reinterpret_cast<cudaStream_t>(stream));
  return ATTN_ERR_UNSUPPORTED;
}

int attn_fwd_fp8(const void* q, const void* k, const void* v, const float* q_scale,
                 const float* k_scale, const float* v_scale, void* o, float* lse, int B, int Hq,
                 int Hkv, int Sq, int Sk, int d, int causal, float scale, attn_stream_t stream) {
  int rc = check_attn_args(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, scale);
  if (rc != ATTN_OK) return rc;
  if (d == 256) return ATTN_ERR_UNSUPPORTED;
  if (!q_scale || !k_scale || !v_scale) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return ATTN_ERR_MISALIGNED;
  return run_attn(q, k, v, q_scale, k_scale, v_scale, o, lse, B, Hq, Hkv, Sq, Sk, d, causal,
                  scale, true, false, reinterpret_cast<cudaStream_t>(stream));
}

int attn_splitkv_plan(int B, int Hq, int Sq, int Sk, int d, int causal, int num_sms,
                      int* num_splits, size_t* workspace_bytes) {
  if (!num_splits || !workspace_bytes) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Sq <= 0 || Sk <= 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  // Cost model (uniform units): a launch takes ceil(items * s / num_sms) rounds
  // of work items, each ceil(tiles / s) K/V tiles plus ~2 tiles of per-range
  // overhead (pipeline fill, partial write, merge). Under a causal mask a unit
  // sees on average the key tiles minus half the query tiles.
  const long long nkv = (Sk + attnb3::BN - 1) / attnb3::BN;
  const long long nqt = (Sq + attnb3::BM - 1) / attnb3::BM;
  const long long n_qp = (Sq + attnb3::UNIT_ROWS - 1) / attnb3::UNIT_ROWS;
  const long long items = static_cast<long long>(B) * Hq * ((n_qp + 1) / 2);
  long long tiles = causal ? nkv - nqt / 2 : nkv;
  if (tiles < 1) tiles = 1;
  long long smax = nkv / 4 > 1 ? nkv / 4 : 1;  // >= 4 K/V tiles per range
  if (smax > kMaxSplits) smax = kMaxSplits;
  long long best = 1, best_cost = -1;
  for (long long s = 1; s <= smax; ++s) {
    const long long rounds = (items * s + num_sms - 1) / num_sms;
    const long long cost = rounds * ((tiles + s - 1) / s + 2);
    if (best_cost < 0 || cost < best_cost) {
      best = s;
      best_cost = cost;
    }
  }
  int kps = 0, nsplit = 0;
  split_shape(Sk, static_cast<int>(best), &kps, &nsplit);
  *num_splits = nsplit;
  *workspace_bytes = splitkv_bytes(B, Hq, Sq, d, nsplit);
  return ATTN_OK;
}

int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale, int dtype,
                     int num_splits, void* workspace, size_t workspace_bytes,
                     attn_stream_t stream) {
  int rc = check_attn_args(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, scale);
  if (rc != ATTN_OK) return rc;
  if (dtype != ATTN_BF16 && dtype != ATTN_F16) return ATTN_ERR_UNSUPPORTED;
  if (d == 256) return ATTN_ERR_UNSUPPORTED;
  if (num_splits < 1 || num_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  int kps = 0, nsplit = 0;
  split_shape(Sk, num_splits, &kps, &nsplit);
  const size_t need = splitkv_bytes(B, Hq, Sq, d, nsplit);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return ATTN_ERR_MISALIGNED;
  const long long n_qp = (Sq + attnb3::UNIT_ROWS - 1) / attnb3::UNIT_ROWS;
  if (static_cast<long long>(B) * Hq * ((n_qp + 1) / 2) * nsplit > 0x7fffffffLL)
    return ATTN_ERR_INVALID_ARG;
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = o_part + static_cast<size_t>(nsplit) * B * Hq * Sq * d;
  const bool f16 = dtype == ATTN_F16;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  rc = run_attn(q, k, v, nullptr, nullptr, nullptr, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale,
                false, f16, st, Split{nsplit, kps, o_part, lse_part});
  if (rc != ATTN_OK) return rc;
  if (d == 128)
    return f16 ? launch_combine<128, true>(o_part, lse_part, o, lse, B, Hq, Sq, nsplit, st)
               : launch_combine<128, false>(o_part, lse_part, o, lse, B, Hq, Sq, nsplit, st);
  return f16 ? launch_combine<64, true>(o_part, lse_part, o, lse, B, Hq, Sq, nsplit, st)
             : launch_combine<64, false>(o_part, lse_part, o, lse, B, Hq, Sq, nsplit, st);
}

int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int Hq, int Hkv, int Sq, int Sk, int d, int causal,
                             float scale, int dtype, int num_splits, attn_stream_t stream) {
  int rc = check_attn_args(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, scale);
  if (rc != ATTN_OK) return rc;
  // the same type and size checks as attn_fwd_splitkv, in the same order, so
  // both entry points return the same code for the same request
  if (dtype != ATTN_BF16 && dtype != ATTN_F16) return ATTN_ERR_UNSUPPORTED;
  if (d == 256) return ATTN_ERR_UNSUPPORTED;
  if (num_splits < 1 || num_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  int kps = 0, nsplit = 0;
  split_shape(Sk, num_splits, &kps, &nsplit);
  if (splitkv_bytes(B, Hq, Sq, d, nsplit) > kNoAllocScratchBytes) return ATTN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != ATTN_OK) return rc;
  return attn_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, dtype,
                          num_splits, scratch, kNoAllocScratchBytes, stream);
}

int attn_qk_rmsnorm(const void* q, const void* k, const void* q_weight, const void* k_weight,
                    void* q_out, void* k_out, int B, int Sq, int Sk, int Hq, int Hkv, int d,
                    float eps, int dtype, attn_stream_t stream) {
  if (!q || !k || !q_weight || !k_weight || !q_out || !k_out) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Sq <= 0 || Sk <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return ATTN_ERR_INVALID_ARG;
  if (!fits_i32(B, Sq, Hq, d) || !fits_i32(B, Sk, Hkv, d)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_BF16 && dtype != ATTN_F16) return ATTN_ERR_UNSUPPORTED;
  for (const void* p : {q, k, q_weight, k_weight, static_cast<const void*>(q_out),
                        static_cast<const void*>(k_out)})
    if (!aligned(p, 16)) return ATTN_ERR_MISALIGNED;
  DeviceInfo* di = nullptr;
  int rc = current_device(&di);
  if (rc != ATTN_OK) return rc;
  const long long tq = static_cast<long long>(B) * Sq, tk = static_cast<long long>(B) * Sk;
  const long long tmax = tq > tk ? tq : tk;
  const long long blocks = tmax;  // one block per token
  if (blocks > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  const dim3 grid(static_cast<unsigned>(blocks), 2);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  auto* qo = static_cast<uint16_t*>(q_out);
  auto* ko = static_cast<uint16_t*>(k_out);
  auto* qi = static_cast<const uint16_t*>(q);
  auto* ki = static_cast<const uint16_t*>(k);
  auto* wq = static_cast<const uint16_t*>(q_weight);
  auto* wk = static_cast<const uint16_t*>(k_weight);
  if (dtype == ATTN_F16)
    attnb3::qk_rmsnorm_kernel<true><<<grid, attnb3::NORM_THREADS, 0, st>>>(
        qi, ki, wq, wk, qo, ko, tq, tk, Hq * d, Hkv * d, eps);
  else
    attnb3::qk_rmsnorm_kernel<false><<<grid, attnb3::NORM_THREADS, 0, st>>>(
        qi, ki, wq, wk, qo, ko, tq, tk, Hq * d, Hkv * d, eps);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_quantize_fp8_e4m3(const float* x, uint8_t* codes, float* scale, int B, int S, int H,
                           int d, attn_stream_t stream) {
  if (!x || !codes || !scale) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || S <= 0 || H <= 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
  if (!fits_i32(B, S, H, d)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scale, 4)) return ATTN_ERR_MISALIGNED;
  DeviceInfo* di = nullptr;
  int rc = current_device(&di);
  if (rc != ATTN_OK) return rc;
  const int nblk = (S + attnb3::FP8_BLOCK - 1) / attnb3::FP8_BLOCK;
  const long long ctas = static_cast<long long>(B) * H * nblk;
  if (ctas > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (d == 128)
    attnb3::quantize_fp8_kernel<128><<<static_cast<unsigned>(ctas), attnb3::QUANT_THREADS, 0, st>>>(
        x, codes, scale, S, H, nblk);
  else
    attnb3::quantize_fp8_kernel<64><<<static_cast<unsigned>(ctas), attnb3::QUANT_THREADS, 0, st>>>(
        x, codes, scale, S, H, nblk);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_bwd_workspace_size(int B, int Hq, int Sq, size_t* workspace_bytes) {
  if (!workspace_bytes || B <= 0 || Hq <= 0 || Sq <= 0) return ATTN_ERR_INVALID_ARG;
  *workspace_bytes = bwd_workspace_bytes(B, Hq, Sq);
  return ATTN_OK;
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* d_o, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
             int Sk, int d, int causal, float scale, int dtype, void* workspace,
             size_t workspace_bytes, attn_stream_t stream) {
  int rc = check_attn_args(q, k, v, const_cast<void*>(o), const_cast<float*>(lse), B, Hq, Hkv,
                           Sq, Sk, d, scale);
  if (rc != ATTN_OK) return rc;
  if (!d_o || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_F16) return ATTN_ERR_UNSUPPORTED;
  if (d == 256) return ATTN_ERR_UNSUPPORTED;
  // padded row statistics are indexed with 32-bit row counts
  if (static_cast<long long>(B) * Hq * static_cast<long long>(bwd_sq_pad(Sq)) > 0x7fffffffLL)
    return ATTN_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < bwd_workspace_bytes(B, Hq, Sq))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(d_o, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(workspace, 16))
    return ATTN_ERR_MISALIGNED;
  DeviceInfo* di = nullptr;
  rc = current_device(&di);
  if (rc != ATTN_OK) return rc;
  if (!get_encoder()) return ATTN_ERR_CUDA;
  const bool f16 = dtype == ATTN_F16;
  float* ws = static_cast<float*>(workspace);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (d == 128 && !f16)
    return launch_bwd<128, false>(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, Sq, Sk, causal,
                                  scale, ws, st, di, 64u);
  if (d == 64 && !f16)
    return launch_bwd<64, false>(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, Sq, Sk, causal,
                                 scale, ws, st, di, 128u);
  if (d == 128)
    return launch_bwd<128, true>(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, Sq, Sk, causal,
                                 scale, ws, st, di, 256u);
  return launch_bwd<64, true>(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, Sq, Sk, causal,
                              scale, ws, st, di, 512u);
}

int attn_device_status(attn_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_status, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (v != 0 && cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return v;
}

int attn_set_wait_limit_ns(unsigned long long ns) {
  if (ns < kWaitLimitMinNs || ns > kWaitLimitMaxNs) return ATTN_ERR_INVALID_ARG;
  g_wait_limit_ns.store(ns, std::memory_order_relaxed);
  return ATTN_OK;
}

unsigned long long attn_get_wait_limit_ns(void) { return wait_limit_ns(); }

const char* attn_status_string(int code) {
  switch (code) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

}  // extern "C"
