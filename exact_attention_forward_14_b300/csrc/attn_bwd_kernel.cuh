// attn_bwd_kernel.cuh -- exact attention backward pass (dQ, dK, dV) for sm_103a.
//
// The pages describe the forward pass only. The backward pass here is the
// chain rule through the same definition, O = softmax(scale Q K^T + mask) V,
// evaluated tile by tile like the forward of the FlashAttention-3 deep dive
// (techknowgenie.com/posts/109164421204410442, "IO-aware tiling": the score
// and probability matrices never reach HBM):
//   P  = exp(scale Q K^T - LSE)       (recomputed from the forward's LSE)
//   dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D)
//   dQ = scale dS K,  dK = scale dS^T Q
// (GQA: the query heads sharing a KV head sum into its dK and dV.)
//
// Three launches:
//   bwd_prep_kernel  D and LSE * log2(e) per query row, padded to whole
//                    128-row tiles (HBM-bound, one warp per row);
//   bwd_dkdv_kernel  unit = (b, KV head, 128 keys): K and V stay in shared
//                    memory while the Q / dO tiles of every query head of the
//                    group stream past; dK and dV accumulate in tensor memory
//                    and are written once;
//   bwd_dq_kernel    unit = (b, query head, 256 query rows) = two 128-row Q
//                    tiles in ping-pong over 64-key K/V tiles (the forward's
//                    structure), S and dP recomputed, dQ accumulating in
//                    tensor memory.
// Computing dQ apart from dK / dV costs two more matrix products per tile
// pair (7 instead of 5) but keeps every output a plain store: no fp32 dQ
// accumulator round-trips through HBM and the results are deterministic.
//
// Both tensor-core kernels: one persistent CTA per SM, 320 threads --
// warps 0-7 element-wise work in two warpgroups, warp 8 MMA issuer (lane 0)
// and TMEM owner, warp 9 TMA producer (lane 0). P and dS are rounded to the
// input type (bf16 / fp16) and handed to the next MMA from tensor memory.
// Every mbarrier wait is bounded (ATTN_ERR_TIMEOUT, then drain and release),
// as in the forward kernel.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace attnb3 {

constexpr int BWD_THREADS = 320;
constexpr int BWD_WARP_MMA = 8;
constexpr int BWD_WARP_LOAD = 9;
constexpr int BWD_TILE = 128;     // query rows per Q tile; keys per dK/dV unit
constexpr int BWD_HALF = 64;      // query columns per element-wise warpgroup (dK/dV)
constexpr int BWD_KV_ROWS = 64;   // keys per K/V tile of the dQ kernel
constexpr int BWD_UNIT_ROWS = 256;
constexpr int BWD_PREP_THREADS = 256;
constexpr int BWD_STATUS_TIMEOUT = 5;  // ATTN_ERR_TIMEOUT
constexpr float BWD_LOG2E = 1.4426950408889634f;

struct BwdParams {
  uint16_t* dq;         // [B, Sq, Hq, d]
  uint16_t* dk;         // [B, Sk, Hkv, d]
  uint16_t* dv;         // [B, Sk, Hkv, d]
  const float* lse2;    // [B, Hq, Sq_pad]: LSE * log2(e); +inf past Sq and for rows without keys
  const float* dsum;    // [B, Hq, Sq_pad]: D = rowsum(dO * O); 0 past Sq
  int B, Hq, Hkv, Sq, Sk, Sq_pad;
  int group;            // Hq / Hkv
  int causal;
  int nq;               // ceil(Sq / 128) Q tiles
  int nk;               // ceil(Sk / 128) key tiles (dK/dV units per (b, hkv))
  int kv_npair;         // ceil(nk / 2): dK/dV work items per (b, hkv)
  int kv_items;         // B * Hkv * kv_npair
  int n_qp;             // ceil(Sq / 256): dQ units per (b, hq)
  int q_npair;          // ceil(n_qp / 2)
  int q_items;          // B * Hq * q_npair
  int nkv64;            // ceil(Sk / 64) K/V tiles of the dQ kernel
  float scale_log2;     // softmax scale * log2(e)
  float scale;          // softmax scale (dQ and dK carry it)
  unsigned long long timeout_ns;
  int* status;
};

template <int D, bool F16>
struct BwdCfg {
  static constexpr uint32_t FMT = F16 ? 0u : 1u;  // kind::f16 operand format
  static constexpr int CHUNK = 128;               // bytes of a swizzled row chunk (64 elements)
  static constexpr int CHUNK_ELEMS = 64;
  static constexpr int NCHUNK = D / CHUNK_ELEMS;
  static constexpr int TILE128 = 128 * D * 2;     // 128 rows of one head
  static constexpr int CH128 = 128 * CHUNK;       // one 64-column chunk of those rows
  static constexpr int TILE64 = 64 * D * 2;       // 64 rows
  static constexpr int CH64 = 64 * CHUNK;
  static constexpr int KSTEPS_D = D / 16;         // 16 elements (32 bytes) per MMA
  static constexpr uint32_t IDESC_N64 = make_idesc(128, 64, FMT, false);
  static constexpr uint32_t IDESC_ACC = make_idesc(128, D, FMT, true);
  static constexpr int TMEM_COLS = 512;
  static constexpr int SMEM_ALLOC = 227 * 1024;
  // ---- dK/dV kernel: K, V, then NSTAGE stages of (Q, dO, lse2[128], D[128])
  static constexpr int NSTAGE = D == 128 ? 2 : 4;
  static constexpr int STAGE = 2 * TILE128 + 1024;
  static constexpr int KV_OFF_K = 0;
  static constexpr int KV_OFF_V = TILE128;
  static constexpr int KV_OFF_ST = 2 * TILE128;
  static constexpr int KV_OFF_BAR = KV_OFF_ST + NSTAGE * STAGE;
  // kv_full, kv_empty, st_full[NSTAGE], st_empty[NSTAGE], sd_full[2],
  // e_full[2], acc_full, acc_empty, drain
  static constexpr int KV_NBAR = 2 + 2 * NSTAGE + 4 + 3;
  static constexpr int KV_OFF_MISC = KV_OFF_BAR + KV_NBAR * 8;
  static constexpr int KV_SMEM = KV_OFF_MISC + 16 + 1024;
  // TMEM columns: S^T [0,128) (half h at 64 h; P^T packed into its first 32),
  // dP^T [128,256) (dS^T packed likewise), dV, dK
  static constexpr int COL_ST = 0;
  static constexpr int COL_DPT = 128;
  static constexpr int COL_DV = 256;
  static constexpr int COL_DK = 256 + D;
  // ---- dQ kernel: 2 Q tiles, 2 dO tiles, NSLOT 64-key K/V slots
  static constexpr int NSLOT = D == 128 ? 6 : 8;
  static constexpr int Q_OFF_Q = 0;
  static constexpr int Q_OFF_DO = 2 * TILE128;
  static constexpr int Q_OFF_KV = 4 * TILE128;
  static constexpr int Q_OFF_BAR = Q_OFF_KV + NSLOT * TILE64;
  // q_full, q_empty, kv_full[NSLOT], kv_empty[NSLOT], sd_full[2], e_full[2],
  // dq_full[2], drain
  static constexpr int Q_NBAR = 2 + 2 * NSLOT + 6 + 1;
  static constexpr int Q_OFF_MISC = Q_OFF_BAR + Q_NBAR * 8;
  static constexpr int Q_SMEM = Q_OFF_MISC + 16 + 1024;
  // TMEM columns of Q tile t: S [128 t, +64) (dS packed into its first 32),
  // dP [128 t + 64, +64), dQ [256 + t d, +d)
  static constexpr int COL_DQ = 256;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(KV_SMEM <= SMEM_ALLOC && Q_SMEM <= SMEM_ALLOC, "shared memory budget");
  static_assert(COL_DK + D <= TMEM_COLS && COL_DQ + 2 * D <= TMEM_COLS, "TMEM budget");
  static_assert(NSLOT % 2 == 0, "K/V slots alternate");
};

// 1-D bulk copy global -> shared (both 16-byte aligned, bytes a multiple of
// 16), completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

struct BwdCtl {
  uint32_t tmem_base;
  uint32_t abort_flag;
};

// Bounded mbarrier wait (see the forward kernel's wait_bounded).
__device__ __forceinline__ bool bwd_wait(uint32_t bar, uint32_t parity, volatile BwdCtl* ctl,
                                         const BwdParams& P) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (ctl->abort_flag) return false;
    if (global_timer_ns() - t0 > P.timeout_ns) {
      ctl->abort_flag = 1u;
      atomicCAS(P.status, 0, BWD_STATUS_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void bwd_drain_wait(uint32_t bar, uint32_t parity, const BwdParams& P) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > P.timeout_ns) {
      atomicCAS(P.status, 0, BWD_STATUS_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ uint32_t pack16x2(bool f16, float lo, float hi) {
  return f16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}

// ------------------------------------------------------------ MMA helpers --

// D[tmem] = A * B^T with A = 128 rows (K-major, 128-row tile in 64-column
// swizzled chunks) and B = 64 rows starting at row b_row0 of a tile whose
// chunks are b_chunk bytes apart; N = 64, K = d.
template <int D, bool F16>
__device__ __forceinline__ void issue_n64(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem,
                                          uint32_t b_chunk, int b_row0) {
  using C = BwdCfg<D, F16>;
#pragma unroll
  for (int ks = 0; ks < C::KSTEPS_D; ++ks) {
    const uint32_t byte_k = ks * 32;
    const uint32_t chunk = byte_k / C::CHUNK, within = byte_k % C::CHUNK;
    const uint64_t a = make_sdesc(a_smem + chunk * C::CH128 + within, 16, 8 * C::CHUNK, 2u);
    const uint64_t b = make_sdesc(b_smem + chunk * b_chunk + b_row0 * C::CHUNK + within, 16,
                                  8 * C::CHUNK, 2u);
    mma_f16_ss(d_tmem, a, b, C::IDESC_N64, ks > 0 ? 1u : 0u);
  }
}

// D[tmem] (+)= A[tmem] * B with A = 128 lanes x 64 packed 16-bit values (32
// columns) and B = 64 rows (the K dimension) starting at row b_row0 of a tile
// with d contiguous (MN-major), chunks b_chunk bytes apart; N = d.
template <int D, bool F16>
__device__ __forceinline__ void issue_acc64(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem,
                                            uint32_t b_chunk, int b_row0, bool accumulate) {
  using C = BwdCfg<D, F16>;
#pragma unroll
  for (int k = 0; k < 4; ++k) {  // 16 rows of K per instruction
    const uint64_t b =
        make_sdesc(b_smem + (b_row0 + 16 * k) * C::CHUNK, b_chunk, 8 * C::CHUNK, 2u);
    mma_f16_ts(d_tmem, a_tmem + 8 * k, b, C::IDESC_ACC, (accumulate || k > 0) ? 1u : 0u);
  }
}

// ------------------------------------------------------------------ prep --

// D[r] = sum_c dO[r, c] * O[r, c] (fp32) and lse2[r] = LSE[r] * log2(e) for
// every padded row r = (b Hq + hq) Sq_pad + i; rows i >= Sq (and rows whose
// LSE is -inf, i.e. that see no key) get lse2 = +inf, which zeroes their P.
template <int D, bool F16>
__global__ void __launch_bounds__(BWD_PREP_THREADS)
    bwd_prep_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ d_o,
                    const float* __restrict__ lse, float* __restrict__ lse2,
                    float* __restrict__ dsum, int Hq, int Sq, int Sq_pad, long long rows_pad) {
  constexpr int PER = D / 32;  // elements per lane
  const long long r =
      static_cast<long long>(blockIdx.x) * (BWD_PREP_THREADS / 32) + (threadIdx.x >> 5);
  if (r >= rows_pad) return;
  const int lane = threadIdx.x & 31;
  const long long bh = r / Sq_pad;
  const int i = static_cast<int>(r - bh * Sq_pad);
  float acc = 0.f, l2 = INFINITY;
  if (i < Sq) {
    const long long b = bh / Hq, hq = bh - b * Hq;
    const size_t off = ((static_cast<size_t>(b) * Sq + i) * Hq + hq) * D + lane * PER;
    uint32_t ow[PER / 2], gw[PER / 2];
    if constexpr (PER == 4) {
      const uint2 a = *reinterpret_cast<const uint2*>(o + off);
      const uint2 g = *reinterpret_cast<const uint2*>(d_o + off);
      ow[0] = a.x; ow[1] = a.y; gw[0] = g.x; gw[1] = g.y;
    } else {
      ow[0] = *reinterpret_cast<const uint32_t*>(o + off);
      gw[0] = *reinterpret_cast<const uint32_t*>(d_o + off);
    }
#pragma unroll
    for (int e = 0; e < PER / 2; ++e) {
      float a0, a1, g0, g1;
      if constexpr (F16) {
        a0 = __half2float(__ushort_as_half(static_cast<unsigned short>(ow[e] & 0xFFFFu)));
        a1 = __half2float(__ushort_as_half(static_cast<unsigned short>(ow[e] >> 16)));
        g0 = __half2float(__ushort_as_half(static_cast<unsigned short>(gw[e] & 0xFFFFu)));
        g1 = __half2float(__ushort_as_half(static_cast<unsigned short>(gw[e] >> 16)));
      } else {
        a0 = __uint_as_float(ow[e] << 16);
        a1 = __uint_as_float(ow[e] & 0xFFFF0000u);
        g0 = __uint_as_float(gw[e] << 16);
        g1 = __uint_as_float(gw[e] & 0xFFFF0000u);
      }
      acc = fmaf(a0, g0, acc);
      acc = fmaf(a1, g1, acc);
    }
#pragma unroll
    for (int off2 = 16; off2 > 0; off2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off2);
    const float L = lse[bh * Sq + i];
    l2 = (L == -INFINITY) ? INFINITY : L * BWD_LOG2E;
  }
  if (lane == 0) {
    lse2[r] = l2;
    dsum[r] = acc;
  }
}

// ------------------------------------------------------------ dK / dV --

struct KvUnit {
  int b, hkv, key0;
  int i_lo;  // first Q tile that sees a key of the unit
  int nqv;   // Q tiles from i_lo on (per query head)
  int T;     // Q tiles of the unit: group * nqv
};

// The i-th dK/dV unit of this CTA: 0 = none left, 1 = skip, 2 = U filled.
// Work item w = (b, hkv, p) pairs key tile p with key tile nk-1-p, so under a
// causal mask (where key tile j is seen by the Q tiles from about j on)
// every item costs about the same; items are dealt round-robin, KV heads
// outermost, so the CTAs in flight share a few heads' Q and dO in L2.
__device__ __forceinline__ int kv_unit(int i, const BwdParams& P, KvUnit& U) {
  const int w = blockIdx.x + (i >> 1) * gridDim.x;
  if (w >= P.kv_items) return 0;
  const int bh = w / P.kv_npair, p = w - bh * P.kv_npair;
  const int jk = (i & 1) ? P.nk - 1 - p : p;
  if ((i & 1) && jk == p) return 1;  // odd nk: the middle tile
  U.b = bh / P.Hkv;
  U.hkv = bh - U.b * P.Hkv;
  U.key0 = jk * BWD_TILE;
  U.i_lo = 0;
  U.nqv = P.nq;
  if (P.causal) {
    const int qmin = U.key0 - (P.Sk - P.Sq);  // first query that sees key0
    if (qmin >= P.Sq) {
      U.nqv = 0;
    } else if (qmin > 0) {
      U.i_lo = qmin / BWD_TILE;
      U.nqv = P.nq - U.i_lo;
    }
  }
  U.T = U.nqv * P.group;
  return 2;
}

template <int D, bool F16>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const BwdParams P) {
  using C = BwdCfg<D, F16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::KV_OFF_BAR;
  const uint32_t BAR_KV_FULL = bar0;
  const uint32_t BAR_KV_EMPTY = bar0 + 8;
  const uint32_t BAR_ST_FULL = bar0 + 16;                       // + 8 * stage
  const uint32_t BAR_ST_EMPTY = BAR_ST_FULL + 8 * C::NSTAGE;    // + 8 * stage
  const uint32_t BAR_SD_FULL = BAR_ST_EMPTY + 8 * C::NSTAGE;    // + 8 * half
  const uint32_t BAR_E_FULL = BAR_SD_FULL + 16;                 // + 8 * half
  const uint32_t BAR_ACC_FULL = BAR_E_FULL + 16;
  const uint32_t BAR_ACC_EMPTY = BAR_ACC_FULL + 8;
  const uint32_t BAR_DRAIN = BAR_ACC_EMPTY + 8;
  volatile BwdCtl* ctl = reinterpret_cast<volatile BwdCtl*>(smem + C::KV_OFF_MISC);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == BWD_WARP_LOAD && lane == 0) {
    mbar_init(BAR_KV_FULL, 1);
    mbar_init(BAR_KV_EMPTY, 1);
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(BAR_ST_FULL + 8 * s, 1);
      mbar_init(BAR_ST_EMPTY + 8 * s, 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(BAR_SD_FULL + 8 * h, 1);
      mbar_init(BAR_E_FULL + 8 * h, 4);  // one elected arrive per warp of the half
    }
    mbar_init(BAR_ACC_FULL, 1);
    mbar_init(BAR_ACC_EMPTY, 8);  // every element-wise warp, after its epilogue
    mbar_init(BAR_DRAIN, 1);
    ctl->abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == BWD_WARP_MMA) {
    tmem_alloc(sbase + C::KV_OFF_MISC, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  auto stage_smem = [&](uint32_t n) { return sbase + C::KV_OFF_ST + (n % C::NSTAGE) * C::STAGE; };

  if (warp == BWD_WARP_LOAD) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t n = 0, u = 0;  // stage fills, K/V fills
      bool ok = true;
      for (int i = 0; ok; ++i) {
        KvUnit U;
        const int st = kv_unit(i, P, U);
        if (st == 0) break;
        if (st == 1 || U.T == 0) continue;
        if (!bwd_wait(BAR_KV_EMPTY, (u & 1u) ^ 1u, ctl, P)) { ok = false; break; }
        mbar_arrive_expect_tx(BAR_KV_FULL, 2 * C::TILE128);
#pragma unroll
        for (int c = 0; c < C::NCHUNK; ++c) {
          tma_load_4d(sbase + C::KV_OFF_K + c * C::CH128, &tm_k, BAR_KV_FULL,
                      c * C::CHUNK_ELEMS, U.hkv, U.key0, U.b);
          tma_load_4d(sbase + C::KV_OFF_V + c * C::CH128, &tm_v, BAR_KV_FULL,
                      c * C::CHUNK_ELEMS, U.hkv, U.key0, U.b);
        }
        ++u;
        for (int t = 0; t < U.T; ++t) {
          const uint32_t s = n % C::NSTAGE;
          if (!bwd_wait(BAR_ST_EMPTY + 8 * s, ((n / C::NSTAGE) & 1u) ^ 1u, ctl, P)) {
            ok = false;
            break;
          }
          const int g = t / U.nqv, qi = U.i_lo + (t - g * U.nqv);
          const int hq = U.hkv * P.group + g;
          const uint32_t stg = stage_smem(n);
          const uint32_t bar = BAR_ST_FULL + 8 * s;
          mbar_arrive_expect_tx(bar, 2 * C::TILE128 + 1024);
#pragma unroll
          for (int c = 0; c < C::NCHUNK; ++c) {
            tma_load_4d(stg + c * C::CH128, &tm_q, bar, c * C::CHUNK_ELEMS, hq, qi * BWD_TILE,
                        U.b);
            tma_load_4d(stg + C::TILE128 + c * C::CH128, &tm_do, bar, c * C::CHUNK_ELEMS, hq,
                        qi * BWD_TILE, U.b);
          }
          const size_t row = (static_cast<size_t>(U.b) * P.Hq + hq) * P.Sq_pad +
                             static_cast<size_t>(qi) * BWD_TILE;
          bulk_load(stg + 2 * C::TILE128, P.lse2 + row, 512, bar);
          bulk_load(stg + 2 * C::TILE128 + 512, P.dsum + row, 512, bar);
          ++n;
        }
      }
      // Drain: every copy issued lands before the CTA exits.
      if (u > 0) bwd_drain_wait(BAR_KV_FULL, (u - 1) & 1u, P);
      for (uint32_t s = 0; s < static_cast<uint32_t>(C::NSTAGE); ++s)
        if (n > s) bwd_drain_wait(BAR_ST_FULL + 8 * s, ((n - 1 - s) / C::NSTAGE) & 1u, P);
    }
    __syncwarp();
  } else if (warp == BWD_WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // Per Q tile t and half h (64 queries):
    //   S^T_h = K Q_h^T, dP^T_h = V dO_h^T         -> sd_full[h]
    //   (element-wise: P^T_h, dS^T_h into TMEM)    <- e_full[h]
    //   dV += P^T_h dO_h,  dK += dS^T_h Q_h
    // issued as  SD(t,0) SD(t,1) | ACC(t,0) SD(t+1,0) | ACC(t,1) SD(t+1,1) | ...
    // so each half's element-wise work overlaps the other half's MMAs;
    // in-order execution makes SD(t+1,h) wait for ACC(t,h), which reads the
    // same TMEM columns.
    if (lane == 0) {
      uint32_t n = 0, u = 0, e[2] = {0u, 0u};
      bool ok = true;
      const uint32_t k_s = sbase + C::KV_OFF_K, v_s = sbase + C::KV_OFF_V;
      auto issue_sd = [&](uint32_t nn, int h) {
        const uint32_t stg = stage_smem(nn);
        issue_n64<D, F16>(tmem + C::COL_ST + BWD_HALF * h, k_s, stg, C::CH128, BWD_HALF * h);
        issue_n64<D, F16>(tmem + C::COL_DPT + BWD_HALF * h, v_s, stg + C::TILE128, C::CH128,
                          BWD_HALF * h);
        tc_commit(BAR_SD_FULL + 8 * h);
      };
      for (int i = 0; ok; ++i) {
        KvUnit U;
        const int st = kv_unit(i, P, U);
        if (st == 0) break;
        if (st == 1 || U.T == 0) continue;
        if (!bwd_wait(BAR_KV_FULL, u & 1u, ctl, P)) { ok = false; break; }
        if (!bwd_wait(BAR_ST_FULL + 8 * (n % C::NSTAGE), (n / C::NSTAGE) & 1u, ctl, P)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_sd(n, 0);
        issue_sd(n, 1);
        for (int t = 0; ok && t < U.T; ++t) {
          const uint32_t nn = n + t;
          const uint32_t stg = stage_smem(nn);
          for (int h = 0; h < 2; ++h) {
            if (!bwd_wait(BAR_E_FULL + 8 * h, e[h] & 1u, ctl, P)) { ok = false; break; }
            ++e[h];
            // the first products of a unit overwrite dV / dK: the previous
            // unit's epilogue must have read them
            if (t == 0 && h == 0 && !bwd_wait(BAR_ACC_EMPTY, (u & 1u) ^ 1u, ctl, P)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const bool acc = !(t == 0 && h == 0);
            issue_acc64<D, F16>(tmem + C::COL_DV, tmem + C::COL_ST + BWD_HALF * h,
                                stg + C::TILE128, C::CH128, BWD_HALF * h, acc);
            issue_acc64<D, F16>(tmem + C::COL_DK, tmem + C::COL_DPT + BWD_HALF * h, stg,
                                C::CH128, BWD_HALF * h, acc);
            if (h == 1) tc_commit(BAR_ST_EMPTY + 8 * (nn % C::NSTAGE));
            if (t + 1 < U.T) {
              if (h == 0) {
                if (!bwd_wait(BAR_ST_FULL + 8 * ((nn + 1) % C::NSTAGE),
                              ((nn + 1) / C::NSTAGE) & 1u, ctl, P)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              issue_sd(nn + 1, h);
            }
          }
        }
        if (!ok) break;
        tc_commit(BAR_ACC_FULL);
        tc_commit(BAR_KV_EMPTY);
        n += U.T;
        ++u;
      }
      tc_commit(BAR_DRAIN);
      bwd_drain_wait(BAR_DRAIN, 0u, P);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ element-wise
    // Thread = one key row of the unit (TMEM lane); warpgroup h = queries
    // [64 h, 64 h + 64) of each Q tile.
    const int h = warp >> 2;
    const int quad = warp & 3;
    const int rloc = quad * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float cs = P.scale_log2;
    uint32_t n = 0, u = 0, sd = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      KvUnit U;
      const int st = kv_unit(i, P, U);
      if (st == 0) break;
      if (st == 1) continue;
      const int kr = U.key0 + rloc;  // this thread's key
      const bool row_ok = kr < P.Sk;
      uint16_t* out = (h ? P.dk : P.dv) +
                      ((static_cast<size_t>(U.b) * P.Sk + kr) * P.Hkv + U.hkv) *
                          static_cast<size_t>(D);
      if (U.T == 0) {  // no query sees these keys
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
          for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      for (int t = 0; t < U.T; ++t) {
        const uint32_t nn = n + t;
        bool w = bwd_wait(BAR_SD_FULL + 8 * h, sd & 1u, ctl, P);
        ++sd;
        // lse2 / D of this tile were staged by TMA on st_full (already
        // complete: the MMA waited for it before issuing S^T)
        w = w && bwd_wait(BAR_ST_FULL + 8 * (nn % C::NSTAGE), (nn / C::NSTAGE) & 1u, ctl, P);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after();
        const int g = t / U.nqv, qi = U.i_lo + (t - g * U.nqv);
        const int q0 = qi * BWD_TILE + BWD_HALF * h;  // first query of this half
        // key kr is visible to query q iff kr <= q + Sk - Sq: columns c < cmin
        // are masked
        int cmin = 0;
        if (!row_ok) cmin = BWD_HALF;
        else if (P.causal) cmin = kr - (P.Sk - P.Sq) - q0;
        uint32_t sr[64], dr[64];
        {
          uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr);
          uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr + 32);
          uint32_t (&d0)[32] = *reinterpret_cast<uint32_t(*)[32]>(dr);
          uint32_t (&d1)[32] = *reinterpret_cast<uint32_t(*)[32]>(dr + 32);
          tmem_ld32_async(t_lane + C::COL_ST + BWD_HALF * h, s0);
          tmem_ld32_async(t_lane + C::COL_ST + BWD_HALF * h + 32, s1);
          tmem_ld32_async(t_lane + C::COL_DPT + BWD_HALF * h, d0);
          tmem_ld32_async(t_lane + C::COL_DPT + BWD_HALF * h + 32, d1);
          tmem_ld_wait();
          reg_fence(s0);
          reg_fence(s1);
          reg_fence(d0);
          reg_fence(d1);
        }
        const uint32_t lse_s = stage_smem(nn) + 2 * C::TILE128 + 4 * BWD_HALF * h;
        const uint32_t dsum_s = lse_s + 512;
        uint32_t pp[32], pd[32];
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const uint4 l4 = lds128(lse_s + 16 * c4);
          const uint4 d4 = lds128(dsum_s + 16 * c4);
          const float lv[4] = {__uint_as_float(l4.x), __uint_as_float(l4.y),
                               __uint_as_float(l4.z), __uint_as_float(l4.w)};
          const float dv4[4] = {__uint_as_float(d4.x), __uint_as_float(d4.y),
                                __uint_as_float(d4.z), __uint_as_float(d4.w)};
          float p[4], ds[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int c = 4 * c4 + e2;
            float x = ex2_approx(fmaf(__uint_as_float(sr[c]), cs, -lv[e2]));
            x = c < cmin ? 0.f : x;
            p[e2] = x;
            ds[e2] = x * (__uint_as_float(dr[c]) - dv4[e2]);
          }
          pp[2 * c4] = pack16x2(F16, p[0], p[1]);
          pp[2 * c4 + 1] = pack16x2(F16, p[2], p[3]);
          pd[2 * c4] = pack16x2(F16, ds[0], ds[1]);
          pd[2 * c4 + 1] = pack16x2(F16, ds[2], ds[3]);
        }
        tmem_st32(t_lane + C::COL_ST + BWD_HALF * h, pp);
        tmem_st32(t_lane + C::COL_DPT + BWD_HALF * h, pd);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR_E_FULL + 8 * h);
      }
      if (!ok) break;
      // ------------------------------------------------------ epilogue
      // warpgroup 0 writes dV, warpgroup 1 dK (times the softmax scale)
      bool w = bwd_wait(BAR_ACC_FULL, u & 1u, ctl, P);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      tc_fence_after();
      const float mul = h ? P.scale : 1.f;
      const uint32_t col = h ? C::COL_DK : C::COL_DV;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t r[32];
        tmem_ld32(t_lane + col + 32 * q, r);
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = pack16x2(F16, __uint_as_float(r[2 * c]) * mul,
                           __uint_as_float(r[2 * c + 1]) * mul);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(out + 32 * q);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_ACC_EMPTY);
      n += U.T;
      ++u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == BWD_WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ dQ --

struct QUnit {
  int b, hq, hkv, row0;
  int n[2];  // 64-key K/V tiles seen by Q tile 0 / 1 (0 = idle or fully masked)
  int nmax;
};

// The i-th dQ unit of this CTA (the forward's pair order: level n_qp-1-p
// with level p of the same (b, hq), heads innermost): 0 = none left,
// 1 = skip, 2 = U filled.
__device__ __forceinline__ int q_unit(int i, const BwdParams& P, QUnit& U) {
  const int w = blockIdx.x + (i >> 1) * gridDim.x;
  if (w >= P.q_items) return 0;
  const int bh = w / P.q_npair, p = w - bh * P.q_npair;
  const int level = (i & 1) ? p : P.n_qp - 1 - p;
  if ((i & 1) && level == P.n_qp - 1 - p) return 1;
  U.b = bh / P.Hq;
  U.hq = bh - U.b * P.Hq;
  U.hkv = U.hq / P.group;
  U.row0 = level * BWD_UNIT_ROWS;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = U.row0 + t * BWD_TILE;
    int n = 0;
    if (r0 < P.Sq) {
      if (!P.causal) {
        n = P.nkv64;
      } else {
        const int lim = min(r0 + BWD_TILE, P.Sq) - 1 + (P.Sk - P.Sq) + 1;  // keys seen by the last row
        n = lim <= 0 ? 0 : min((lim + BWD_KV_ROWS - 1) / BWD_KV_ROWS, P.nkv64);
      }
    }
    U.n[t] = n;
  }
  U.nmax = max(U.n[0], U.n[1]);
  return 2;
}

template <int D, bool F16>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k64,
                  const __grid_constant__ CUtensorMap tm_v64, const BwdParams P) {
  using C = BwdCfg<D, F16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::Q_OFF_BAR;
  const uint32_t BAR_Q_FULL = bar0;
  const uint32_t BAR_Q_EMPTY = bar0 + 8;
  const uint32_t BAR_KV_FULL = bar0 + 16;                    // + 8 * slot
  const uint32_t BAR_KV_EMPTY = BAR_KV_FULL + 8 * C::NSLOT;  // + 8 * slot
  const uint32_t BAR_SD_FULL = BAR_KV_EMPTY + 8 * C::NSLOT;  // + 8 * t
  const uint32_t BAR_E_FULL = BAR_SD_FULL + 16;              // + 8 * t
  const uint32_t BAR_DQ_FULL = BAR_E_FULL + 16;              // + 8 * t
  const uint32_t BAR_DRAIN = BAR_DQ_FULL + 16;
  volatile BwdCtl* ctl = reinterpret_cast<volatile BwdCtl*>(smem + C::Q_OFF_MISC);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == BWD_WARP_LOAD && lane == 0) {
    mbar_init(BAR_Q_FULL, 1);
    mbar_init(BAR_Q_EMPTY, 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(BAR_KV_FULL + 8 * s, 1);
      mbar_init(BAR_KV_EMPTY + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR_SD_FULL + 8 * t, 1);
      mbar_init(BAR_E_FULL + 8 * t, 4);
      mbar_init(BAR_DQ_FULL + 8 * t, 1);
    }
    mbar_init(BAR_DRAIN, 1);
    ctl->abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k64);
    tma_prefetch_desc(&tm_v64);
  }
  if (warp == BWD_WARP_MMA) {
    tmem_alloc(sbase + C::Q_OFF_MISC, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == BWD_WARP_LOAD) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0, qit = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        QUnit U;
        const int st = q_unit(i, P, U);
        if (st == 0) break;
        if (st == 1 || U.nmax == 0) continue;
        if (!bwd_wait(BAR_Q_EMPTY, (qit & 1u) ^ 1u, ctl, P)) { ok = false; break; }
        const int nqt = (U.n[0] > 0) + (U.n[1] > 0);
        mbar_arrive_expect_tx(BAR_Q_FULL, nqt * 2 * C::TILE128);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (U.n[t] == 0) continue;
#pragma unroll
          for (int c = 0; c < C::NCHUNK; ++c) {
            tma_load_4d(sbase + C::Q_OFF_Q + t * C::TILE128 + c * C::CH128, &tm_q, BAR_Q_FULL,
                        c * C::CHUNK_ELEMS, U.hq, U.row0 + t * BWD_TILE, U.b);
            tma_load_4d(sbase + C::Q_OFF_DO + t * C::TILE128 + c * C::CH128, &tm_do,
                        BAR_Q_FULL, c * C::CHUNK_ELEMS, U.hq, U.row0 + t * BWD_TILE, U.b);
          }
        }
        ++qit;
        for (int j = 0; ok && j < U.nmax; ++j) {
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t slot = it % C::NSLOT;
            if (!bwd_wait(BAR_KV_EMPTY + 8 * slot, ((it / C::NSLOT) & 1u) ^ 1u, ctl, P)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(BAR_KV_FULL + 8 * slot, C::TILE64);
#pragma unroll
            for (int c = 0; c < C::NCHUNK; ++c)
              tma_load_4d(sbase + C::Q_OFF_KV + slot * C::TILE64 + c * C::CH64,
                          kv ? &tm_v64 : &tm_k64, BAR_KV_FULL + 8 * slot, c * C::CHUNK_ELEMS,
                          U.hkv, j * BWD_KV_ROWS, U.b);
            ++it;
          }
        }
      }
      for (uint32_t s = 0; s < static_cast<uint32_t>(C::NSLOT); ++s)
        if (it > s) bwd_drain_wait(BAR_KV_FULL + 8 * s, ((it - 1 - s) / C::NSLOT) & 1u, P);
      if (qit > 0) bwd_drain_wait(BAR_Q_FULL, (qit - 1) & 1u, P);
    }
    __syncwarp();
  } else if (warp == BWD_WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // Per 64-key K/V tile j and Q tile t:
    //   S_t = Q_t K_j^T, dP_t = dO_t V_j^T  -> sd_full[t]
    //   (element-wise: dS_t into TMEM)     <- e_full[t]
    //   dQ_t += dS_t K_j
    // issued as  SD_0(0) SD_1(0) | DQ_0(0) SD_0(1) | DQ_1(0) SD_1(1) | ...
    // K_j is released after both DQ(j), V_j after both SD(j).
    if (lane == 0) {
      uint32_t it = 0, qit = 0, e[2] = {0u, 0u};
      bool ok = true;
      const uint32_t kv_s = sbase + C::Q_OFF_KV;
      auto slot_smem = [&](uint32_t f) { return kv_s + (f % C::NSLOT) * C::TILE64; };
      auto wait_fill = [&](uint32_t f) {
        return bwd_wait(BAR_KV_FULL + 8 * (f % C::NSLOT), (f / C::NSLOT) & 1u, ctl, P);
      };
      auto issue_sd = [&](int t, uint32_t fk) {
        issue_n64<D, F16>(tmem + 128 * t, sbase + C::Q_OFF_Q + t * C::TILE128, slot_smem(fk),
                          C::CH64, 0);
        issue_n64<D, F16>(tmem + 128 * t + 64, sbase + C::Q_OFF_DO + t * C::TILE128,
                          slot_smem(fk + 1), C::CH64, 0);
        tc_commit(BAR_SD_FULL + 8 * t);
      };
      for (int i = 0; ok; ++i) {
        QUnit U;
        const int st = q_unit(i, P, U);
        if (st == 0) break;
        if (st == 1 || U.nmax == 0) continue;
        if (!bwd_wait(BAR_Q_FULL, qit & 1u, ctl, P)) { ok = false; break; }
        if (!wait_fill(it) || !wait_fill(it + 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (U.n[t] > 0) issue_sd(t, it);
        tc_commit(BAR_KV_EMPTY + 8 * ((it + 1) % C::NSLOT));  // V_0
        if (U.nmax == 1) tc_commit(BAR_Q_EMPTY);
        for (int j = 0; j < U.nmax; ++j) {
          const uint32_t fk = it + 2 * j;  // fill of K_j
          const bool more = j + 1 < U.nmax;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (j < U.n[t]) {
              if (!bwd_wait(BAR_E_FULL + 8 * t, e[t] & 1u, ctl, P)) { ok = false; break; }
              ++e[t];
              tc_fence_after();
              issue_acc64<D, F16>(tmem + C::COL_DQ + t * D, tmem + 128 * t, slot_smem(fk),
                                  C::CH64, 0, j > 0);
              if (j == U.n[t] - 1) tc_commit(BAR_DQ_FULL + 8 * t);
            }
            if (t == 0 && more) {
              if (!wait_fill(fk + 2) || !wait_fill(fk + 3)) { ok = false; break; }
              tc_fence_after();
            }
            if (j + 1 < U.n[t]) issue_sd(t, fk + 2);
          }
          if (!ok) break;
          tc_commit(BAR_KV_EMPTY + 8 * (fk % C::NSLOT));  // K_j
          if (more) {
            tc_commit(BAR_KV_EMPTY + 8 * ((fk + 3) % C::NSLOT));  // V_{j+1}
            if (j + 2 == U.nmax) tc_commit(BAR_Q_EMPTY);
          }
        }
        if (!ok) break;
        it += 2 * U.nmax;
        ++qit;
      }
      tc_commit(BAR_DRAIN);
      bwd_drain_wait(BAR_DRAIN, 0u, P);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ element-wise
    // Thread = one query row of Q tile t (TMEM lane).
    const int t = warp >> 2;
    const int quad = warp & 3;
    const int rloc = quad * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t col_s = 128 * t, col_dp = 128 * t + 64, col_dq = C::COL_DQ + t * D;
    const float cs = P.scale_log2;
    uint32_t sd = 0, dqc = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      QUnit U;
      const int st = q_unit(i, P, U);
      if (st == 0) break;
      if (st == 1) continue;
      const int tile_row0 = U.row0 + t * BWD_TILE;
      if (tile_row0 >= P.Sq) continue;
      const int row = tile_row0 + rloc;  // < Sq_pad
      const bool row_ok = row < P.Sq;
      const int n = U.n[t];
      const size_t ridx = (static_cast<size_t>(U.b) * P.Hq + U.hq) * P.Sq_pad + row;
      const float l2 = P.lse2[ridx];
      const float dsr = P.dsum[ridx];
      for (int j = 0; j < n; ++j) {
        const bool w = bwd_wait(BAR_SD_FULL + 8 * t, sd & 1u, ctl, P);
        ++sd;
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[64], dr[64];
        {
          uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr);
          uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr + 32);
          uint32_t (&d0)[32] = *reinterpret_cast<uint32_t(*)[32]>(dr);
          uint32_t (&d1)[32] = *reinterpret_cast<uint32_t(*)[32]>(dr + 32);
          tmem_ld32_async(t_lane + col_s, s0);
          tmem_ld32_async(t_lane + col_s + 32, s1);
          tmem_ld32_async(t_lane + col_dp, d0);
          tmem_ld32_async(t_lane + col_dp + 32, d1);
          tmem_ld_wait();
          reg_fence(s0);
          reg_fence(s1);
          reg_fence(d0);
          reg_fence(d1);
        }
        // keys key0 + c, c >= vis, are masked (past Sk, or after row + Sk - Sq)
        const int key0 = j * BWD_KV_ROWS;
        int vis = P.Sk - key0;
        if (P.causal) vis = min(vis, row + (P.Sk - P.Sq) - key0 + 1);
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float p0 = ex2_approx(fmaf(__uint_as_float(sr[c]), cs, -l2));
          float p1 = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), cs, -l2));
          p0 = c < vis ? p0 : 0.f;
          p1 = c + 1 < vis ? p1 : 0.f;
          pk[c / 2] = pack16x2(F16, p0 * (__uint_as_float(dr[c]) - dsr),
                               p1 * (__uint_as_float(dr[c + 1]) - dsr));
        }
        tmem_st32(t_lane + col_s, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR_E_FULL + 8 * t);
      }
      if (!ok) break;
      // ------------------------------------------------------ epilogue
      uint16_t* out = P.dq + ((static_cast<size_t>(U.b) * P.Sq + row) * P.Hq + U.hq) *
                                 static_cast<size_t>(D);
      if (n > 0) {
        const bool w = bwd_wait(BAR_DQ_FULL + 8 * t, dqc & 1u, ctl, P);
        ++dqc;
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t r[32];
          tmem_ld32(t_lane + col_dq + 32 * q, r);
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[c] = pack16x2(F16, __uint_as_float(r[2 * c]) * P.scale,
                             __uint_as_float(r[2 * c + 1]) * P.scale);
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(out + 32 * q);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      } else if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
        for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == BWD_WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace attnb3
