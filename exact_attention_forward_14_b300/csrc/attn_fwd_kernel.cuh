// attn_fwd_kernel.cuh -- fused exact attention forward for sm_103a (B300).
//
// Method: "FlashAttention-3 deep dive: asynchronous TMA and WGMMA on NVIDIA
// Hopper H100" (techknowgenie.com/posts/109164421204410442), cited as [FA3]:
//   [FA3 intro]  IO-aware tiling + online softmax: the Sq x Sk score matrix
//                stays on chip; work is split over query-row tiles;
//   [FA3 s1]     TMA: one thread issues a bulk tensor copy, completion is
//                tracked by an mbarrier (producer/consumer hand-off);
//   [FA3 s2]     three overlapped stages: TMA load of the next K/V tile,
//                S = Q K^T on the tensor cores, softmax + O += P V for the
//                previous tile; multi-stage K/V buffers;
//   [FA3 s3]     the softmax (exp on the MUFU) is the bottleneck the
//                pipeline must hide; fewer rescales help;
//   [FA3 s4]     FP8: per-block scale factors, FP8 products with fp32
//                accumulation, base-2 exponentials.
// The Hopper specifics there (WGMMA register accumulators, warpgroup-wide
// MMA) are replaced by the Blackwell forms: tcgen05.mma issued by one thread,
// fp32 accumulators in tensor memory (TMEM), P handed to the second MMA
// straight from TMEM.
//
// CTA organisation (one persistent CTA per SM, 320 threads):
//   warps 0-3  softmax for Q tile 0 (thread = one query row = one TMEM lane)
//   warps 4-7  softmax for Q tile 1 (ping-pong partner of tile 0)
//   warp  8    MMA issuer (lane 0) and TMEM owner
//   warp  9    TMA producer (lane 0)
//   warps 10-11 (E4M3 inputs only, 384 threads) widen each staged E4M3 V
//              tile to fp16 in one of two shared-memory buffers: S = Q K^T
//              runs on E4M3 operands, O += P V on fp16 ones, P kept in fp16
//              (both MMA operands must share one element type)
// A work unit is (b, hq, 256 query rows) = two 128-row Q tiles that share one
// stream of 128-key K/V tiles. Per K/V tile j the MMA warp issues, in order,
//   O0 += P0(j) V(j);  S0(j+1) = Q0 K(j+1)^T;  O1 += P1(j) V(j);  S1(j+1) = ...
// so while softmax 0 works on S0(j+1) the tensor cores run tile 1's MMAs and
// vice versa. P(j) overwrites the low columns of S(j) in TMEM (bf16 or fp16
// pairs per 32-bit column); in-order execution of MMAs from one thread
// makes S(j+1) wait for P(j)'s consumer.
//
// TMEM columns (512 allocated): S0 [0,128) S1 [128,256) O0 [256,256+d)
// O1 [256+d, 256+2d).
//
// Online softmax (exact): running max m (log2 units) and sum l per row. The
// max used for the exponent is only raised when the tile max exceeds it by
// more than RESCALE_LOG2 (then O and l are rescaled by 2^(m_old - m_new));
// otherwise p = 2^(s*c - m) <= 2^RESCALE_LOG2. O and l share the stale max,
// so O / l is unchanged.
//
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the CTA
// records ATTN_ERR_TIMEOUT in the device status word, every role leaves its
// loop, outstanding copies and MMAs are drained (again with a limit) and the
// tensor memory is released.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"
#include "widen_v.cuh"

namespace attnb3 {

constexpr int BM = 128;           // query rows per Q tile
constexpr int BN = 128;           // keys per K/V tile
constexpr int UNIT_ROWS = 2 * BM; // query rows per work unit
constexpr int NUM_THREADS = 320;      // bf16 / fp16
constexpr int NUM_THREADS_FP8 = 384;  // + warps 10-11 widening V to fp16
constexpr int WARP_WIDEN = 10;        // first of the two V-widening warps
constexpr int WARP_MMA = 8;
constexpr int WARP_LOAD = 9;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr float LN2 = 0.6931471805599453f;
constexpr int STATUS_TIMEOUT = 5;  // ATTN_ERR_TIMEOUT
constexpr int FP8_BLOCK = 64;      // rows per FP8 scale block

struct FwdParams {
  uint16_t* o;           // bf16 or fp16 bits [B, Sq, Hq, d]
  float* lse;
  const float* q_scale;  // FP8 only: [B, Hq, ceil(Sq/64)]
  const float* k_scale;  // FP8 only: [B, Hkv, ceil(Sk/64)]
  const float* v_scale;  // FP8 only: [B, Hkv, ceil(Sk/64)]
  int B, Hq, Hkv, Sq, Sk;
  int group;      // Hq / Hkv
  int n_qp;       // ceil(Sq / UNIT_ROWS): units (levels) per (b, hq)
  int npair;      // ceil(n_qp / 2): work items per (b, hq)
  int nkv;        // ceil(Sk / BN)
  int num_items;  // B * Hq * npair * nsplit
  int causal;
  // Split-KV (nsplit > 1, or o_part set): the K/V tiles are cut into ranges
  // of kps tiles; a work item covers one range and its epilogue writes the
  // range's normalised O (fp32) and LSE to o_part / lse_part instead of o /
  // lse. nsplit = 1, kps = nkv, o_part = null is the plain forward pass.
  int nsplit;
  int kps;
  int lpt;          // 1: longest-first unit order (see cta_unit)
  float* o_part;    // [nsplit, B, Hq, Sq, d] fp32
  float* lse_part;  // [nsplit, B, Hq, Sq] fp32
  float scale_log2;  // softmax scale * log2(e)
  unsigned long long timeout_ns;
  int* status;       // device status word
};

template <int D, bool FP8, bool F16 = false>
struct Cfg {
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int ROW_BYTES = D * ESZ;
  static constexpr int CHUNK_BYTES = ROW_BYTES < 128 ? ROW_BYTES : 128;  // swizzle span
  static constexpr int CHUNK_ELEMS = CHUNK_BYTES / ESZ;
  static constexpr int NCHUNK = ROW_BYTES / CHUNK_BYTES;
  static constexpr uint32_t SWZ_CODE = CHUNK_BYTES == 128 ? 2u : 4u;
  static constexpr int Q_TILE_BYTES = BM * ROW_BYTES;
  static constexpr int KV_TILE_BYTES = BN * ROW_BYTES;
  static constexpr int Q_CHUNK_BYTES = BM * CHUNK_BYTES;
  static constexpr int KV_CHUNK_BYTES = BN * CHUNK_BYTES;
  static constexpr int NSLOT = KV_TILE_BYTES >= 32768 ? 4 : 8;
  static constexpr int MMA_K = FP8 ? 32 : 16;  // 32 bytes of K per instruction
  static constexpr int KSTEPS_QK = D / MMA_K;
  // O += P V always runs on 16-bit operands: P is bf16 or fp16 (fp16 for
  // FP8 inputs, whose V tiles are widened to fp16 in shared memory first).
  static constexpr int KSTEPS_PV = BN / 16;
  static constexpr int P_COLS = BN * 2 / 4;  // TMEM columns holding P
  static constexpr int P_COLS_PER_KSTEP = 16 * 2 / 4;
  static constexpr int P_PARTS = 1;
  static constexpr float RESCALE = RESCALE_LOG2;  // stale-max threshold, log2 units
  static_assert(P_COLS <= BN, "P must fit in the S columns");
  static constexpr int THREADS = FP8 ? NUM_THREADS_FP8 : NUM_THREADS;
  // E4M3 inputs: warps 8-11 (MMA, TMA, V widening) form a whole warpgroup,
  // which gives up registers at start-up so the softmax warpgroups can use
  // more (the E4M3 softmax, with its per-block scales, does not fit in the
  // 168 a thread the 384-thread launch gets). 256 * REGS_SOFTMAX + 128 *
  // REGS_OTHER must not exceed the registers the block was launched with
  // (384 * 168); the host checks it before launching, since an increase that
  // cannot be met would wait forever.
  static constexpr bool REBALANCE = FP8;
  static constexpr int REGS_SOFTMAX = 192;
  static constexpr int REGS_OTHER = 104;
  static constexpr int REGS_NEEDED = REBALANCE ? 256 * REGS_SOFTMAX + 128 * REGS_OTHER : 0;
  static constexpr int V16_TILE_BYTES = BN * D * 2;  // FP8: a widened V tile
  // operand format: kind::f8f6f4 0 = e4m3; kind::f16 0 = f16, 1 = bf16
  static constexpr uint32_t AB_FMT = (FP8 || F16) ? 0u : 1u;
  static constexpr uint32_t IDESC_S = make_idesc(BM, BN, AB_FMT, false);
  static constexpr uint32_t IDESC_PV = make_idesc(BM, D, (FP8 || F16) ? 0u : 1u, true);
  // the V operand of O += P V (FP8: the widened fp16 tile)
  static constexpr int V_CHUNK_BYTES = 128;            // 128-byte swizzle span
  static constexpr int V_KV_CHUNK_BYTES = BN * V_CHUNK_BYTES;
  static constexpr int COL_S0 = 0;
  static constexpr int COL_O0 = 2 * BN;
  static constexpr int TMEM_COLS = 512;
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = 2 * Q_TILE_BYTES;
  static constexpr int OFF_VF = OFF_KV + NSLOT * KV_TILE_BYTES;  // FP8: 2 widened V tiles
  static constexpr int OFF_BAR = OFF_VF + (FP8 ? 2 * V16_TILE_BYTES : 0);
  // barriers: q_full, q_empty, kv_full[NSLOT], kv_empty[NSLOT], s_full[2],
  // p_full[2 tiles][2 halves], o_full[2], drain, vf_full[2], vf_empty[2]
  static constexpr int NUM_BARS = 2 + 2 * NSLOT + 13;
  // K and V fills alternate, so with an even ring K always lands in even
  // slots and V in odd ones (the FP8 path releases V slots from the widening
  // warps, K slots from the MMA thread)
  static_assert(NSLOT % 2 == 0, "K/V slots alternate");
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  // 16-bit inputs: each softmax warp writes its 32 output rows through a
  // 2 KB staging area (32 rows x 64 bytes, one 32-column quarter of O at a
  // time), so that each global store instruction writes 64 contiguous bytes
  // of 8 rows instead of 16 bytes of 32 rows. (E4M3 inputs: no room left;
  // d = 64: the staging code makes the softmax spill at its register cap.
  // Those rows are stored directly.)
  static constexpr bool STAGE_O = !FP8 && D >= 128;
  static constexpr int OSTAGE_WARP_BYTES = 32 * 64;
  static constexpr int OFF_OSTAGE = (OFF_MISC + 16 + 127) / 128 * 128;
  static constexpr int SMEM_BYTES = OFF_OSTAGE + (STAGE_O ? 8 * OSTAGE_WARP_BYTES : 0) + 1024;
  // Launch with the whole opt-in budget (one CTA per SM either way), so a
  // descriptor stepping past its tile still reads inside this CTA's window.
  static constexpr int SMEM_ALLOC = 227 * 1024;
  static_assert(2 * BN + 2 * D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= SMEM_ALLOC, "shared memory budget");
  static_assert(D % MMA_K == 0 && D % 32 == 0, "head dim");
};

// S = Q K^T for one 128-row Q tile and one 128-key K tile, both staged by TMA
// as K-major rows in 128-byte (or 64-byte) swizzled chunks of CHUNK_BYTES
// columns; each instruction consumes 32 bytes of the head dimension.
template <int D, bool FP8, bool F16 = false>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  using C = Cfg<D, FP8, F16>;
#pragma unroll
  for (int ks = 0; ks < C::KSTEPS_QK; ++ks) {
    const uint32_t byte_k = ks * 32;
    const uint32_t chunk = byte_k / C::CHUNK_BYTES;
    const uint32_t within = byte_k % C::CHUNK_BYTES;
    const uint64_t a = make_sdesc(q_smem + chunk * C::Q_CHUNK_BYTES + within, 16,
                                  8 * C::CHUNK_BYTES, C::SWZ_CODE);
    const uint64_t b = make_sdesc(k_smem + chunk * C::KV_CHUNK_BYTES + within, 16,
                                  8 * C::CHUNK_BYTES, C::SWZ_CODE);
    if constexpr (FP8) mma_f8_ss(d_tmem, a, b, C::IDESC_S, ks > 0);
    else mma_f16_ss(d_tmem, a, b, C::IDESC_S, ks > 0);
  }
}

// O (+)= P V for one half of the K/V tile (keys [64 h, 64 h + 64)): P
// (128 x 128 keys, bf16 or fp16) in tensor memory, packed along the keys; the
// 16-bit V tile (staged by TMA, or for FP8 inputs widened to fp16 in shared
// memory) has d contiguous in 128-byte swizzled chunks (MN-major B operand):
// the leading byte offset steps between d-chunks, the stride byte offset
// between groups of 8 keys; each instruction consumes 16 keys. `accumulate`
// = false starts O afresh.
template <int D, bool FP8, bool F16 = false>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                              int half, bool accumulate) {
  using C = Cfg<D, FP8, F16>;
  constexpr int KS_HALF = C::KSTEPS_PV / 2;
#pragma unroll
  for (int k = 0; k < KS_HALF; ++k) {
    const int ks = half * KS_HALF + k;
    const uint64_t b = make_sdesc(v_smem + ks * 16 * C::V_CHUNK_BYTES, C::V_KV_CHUNK_BYTES,
                                  8 * C::V_CHUNK_BYTES, 2u);
    const uint32_t a = p_tmem + ks * C::P_COLS_PER_KSTEP;
    mma_f16_ts(d_tmem, a, b, C::IDESC_PV, (accumulate || ks > 0) ? 1u : 0u);
  }
}

// Both halves (used by the single-tile self-test).
template <int D, bool FP8, bool F16 = false>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         bool accumulate) {
  issue_pv_half<D, FP8, F16>(d_tmem, p_tmem, v_smem, 0, accumulate);
  issue_pv_half<D, FP8, F16>(d_tmem, p_tmem, v_smem, 1, true);
}

// Warp-collective forms used by the kernel's MMA warp: the whole warp runs
// them with the same operands and one elected lane issues each instruction.
// The operand descriptors are formed once per tile (a_desc, b_desc: the
// tile's first byte); each K step adds a compile-time byte offset to the
// start-address field. Keeping the issue loop to a few uniform instructions
// per MMA matters: the MMA warp shares its SM sub-partition with two softmax
// warps, and an issue path of a dozen scalar instructions per MMA made issue,
// not execution, the pace of the tensor pipe.
template <int D, bool FP8, bool F16 = false>
__device__ __forceinline__ void issue_qk_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
  using C = Cfg<D, FP8, F16>;
#pragma unroll
  for (int ks = 0; ks < C::KSTEPS_QK; ++ks) {
    const uint32_t byte_k = ks * 32;
    const uint32_t chunk = byte_k / C::CHUNK_BYTES;
    const uint32_t within = byte_k % C::CHUNK_BYTES;
    const uint64_t a = sdesc_add(a_desc, chunk * C::Q_CHUNK_BYTES + within);
    const uint64_t b = sdesc_add(b_desc, chunk * C::KV_CHUNK_BYTES + within);
    if constexpr (FP8) mma_f8_ss_w(d_tmem, a, b, C::IDESC_S, ks > 0 ? 1u : 0u);
    else mma_f16_ss_w(d_tmem, a, b, C::IDESC_S, ks > 0 ? 1u : 0u);
  }
}

template <int D, bool FP8, bool F16 = false>
__device__ __forceinline__ void issue_pv_half_w(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                                int half, bool accumulate) {
  using C = Cfg<D, FP8, F16>;
  constexpr int KS_HALF = C::KSTEPS_PV / 2;
#pragma unroll
  for (int k = 0; k < KS_HALF; ++k) {
    const int ks = half * KS_HALF + k;
    const uint64_t b = sdesc_add(v_desc, ks * 16 * C::V_CHUNK_BYTES);
    const uint32_t a = p_tmem + ks * C::P_COLS_PER_KSTEP;
    mma_f16_ts_w(d_tmem, a, b, C::IDESC_PV, (accumulate || ks > 0) ? 1u : 0u);
  }
}

struct Unit {
  int b, hq, hkv, row0;
  int split, j0;  // key range: K/V tiles j0 + [0, n[t])
  int n[2];  // K/V tiles needed by Q tile 0 / 1 (0 = tile idle or fully masked)
  int nmax;
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Work items and units. A unit is (b, hq, 256 query rows); the units of one
// (b, hq) are its n_qp "levels" (level L covers rows [256 L, 256 L + 256)).
//
// Pair order (the default): a work item pairs level n_qp-1-p with level p of
// the same (b, hq), so under a causal mask every item costs the same number
// of K/V tiles (a heavy unit plus its mirror) and a static round-robin over
// items balances the CTAs. Items are numbered (b, hq)-major with hq fastest:
// the CTAs running at the same time cover only a few heads (query heads
// sharing a KV head are adjacent), so those heads' K/V tiles are re-read from
// L2, not HBM. With split-KV, item w covers key range w % nsplit of pair
// w / nsplit.
//
// Single-unit order (lpt != 0; chosen by the host when there are fewer than
// 4 items per CTA, where whole items leave the last round part-empty): single
// units dealt to the CTAs in a snake (round r goes left to right for even r,
// right to left for odd r), which evens out the per-CTA totals. Under a
// causal mask the units are sorted by level, highest (most K/V tiles) first,
// across all heads; without one every unit costs the same and they stay
// head-major, so the few heads in flight keep their K/V in L2.

// Fills U for unit (level, bh, split); the key range is split's K/V tiles.
__device__ __forceinline__ void fill_unit(int level, int bh, int split, const FwdParams& P,
                                          Unit& U) {
  U.split = split;
  U.j0 = split * P.kps;
  const int j1 = min(U.j0 + P.kps, P.nkv);
  U.b = bh / P.Hq;
  U.hq = bh - U.b * P.Hq;
  U.hkv = U.hq / P.group;
  U.row0 = level * UNIT_ROWS;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = U.row0 + t * BM;
    int n = 0;
    if (r0 < P.Sq) {
      if (!P.causal) {
        n = P.nkv;
      } else {
        const int rl = min(r0 + BM, P.Sq) - 1;
        const int lim = rl + (P.Sk - P.Sq) + 1;  // keys visible to the last row
        n = lim <= 0 ? 0 : min(ceil_div(lim, BN), P.nkv);
      }
    }
    U.n[t] = max(0, min(n, j1) - U.j0);
  }
  U.nmax = max(U.n[0], U.n[1]);
}

// The i-th unit of this CTA: 0 = no more units, 1 = nothing at this position
// (skip it), 2 = U filled.
__device__ __forceinline__ int cta_unit(int i, const FwdParams& P, Unit& U) {
  const int G = gridDim.x, c = blockIdx.x;
  if (P.lpt) {
    const int kg = i * G + ((i & 1) ? G - 1 - c : c);
    const int bh_count = P.B * P.Hq;
    if (kg >= bh_count * P.n_qp) return 0;
    if (P.causal)  // costs differ by level: highest level first, all heads
      fill_unit(P.n_qp - 1 - kg / bh_count, kg % bh_count, 0, P, U);
    else           // equal costs: keep heads together (their K/V stay in L2)
      fill_unit(kg % P.n_qp, kg / P.n_qp, 0, P, U);
    return 2;
  }
  int w = c + (i >> 1) * G;
  const int k = i & 1;
  if (w >= P.num_items) return 0;
  const int split = w % P.nsplit;
  w /= P.nsplit;
  const int bh = w / P.npair;
  const int p = w - bh * P.npair;
  const int level = k == 0 ? P.n_qp - 1 - p : p;
  if (k == 1 && level == P.n_qp - 1 - p) return 1;  // odd n_qp: the middle level
  fill_unit(level, bh, split, P, U);
  return 2;
}

struct Ctl {
  uint32_t tmem_base;
  uint32_t abort_flag;
};

// Bounded wait on an mbarrier phase. Returns false when the CTA is aborting
// (another role gave up) or when this wait ran past the limit (it then starts
// the abort and records the timeout).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile Ctl* ctl,
                                             const FwdParams& P) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (ctl->abort_flag) return false;
    if (global_timer_ns() - t0 > P.timeout_ns) {
      ctl->abort_flag = 1u;
      atomicCAS(P.status, 0, STATUS_TIMEOUT);
      return false;
    }
  }
}

// Bounded wait used while draining: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const FwdParams& P) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > P.timeout_ns) {
      atomicCAS(P.status, 0, STATUS_TIMEOUT);
      return;
    }
  }
}

// F16: q, k, v and o are fp16 (P is packed as f16 too); otherwise 16-bit
// data is bf16 and FP8 inputs produce a bf16 O.
template <int D, bool FP8, bool F16>
__global__ void __launch_bounds__(Cfg<D, FP8, F16>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams P) {
  using C = Cfg<D, FP8, F16>;
  static_assert(!(FP8 && F16), "FP8 inputs give a bf16 O");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t BAR_Q_FULL = bar0;
  const uint32_t BAR_Q_EMPTY = bar0 + 8;
  const uint32_t BAR_KV_FULL = bar0 + 16;                     // + 8 * slot
  const uint32_t BAR_KV_EMPTY = BAR_KV_FULL + 8 * C::NSLOT;   // + 8 * slot
  const uint32_t BAR_S_FULL = BAR_KV_EMPTY + 8 * C::NSLOT;    // + 8 * t
  const uint32_t BAR_P_FULL = BAR_S_FULL + 16;                // + 16 * t + 8 * half
  const uint32_t BAR_O_FULL = BAR_P_FULL + 32;                // + 8 * t
  const uint32_t BAR_DRAIN = BAR_O_FULL + 16;
  const uint32_t BAR_VF_FULL = BAR_DRAIN + 8;                 // + 8 * buffer (FP8)
  const uint32_t BAR_VF_EMPTY = BAR_VF_FULL + 16;             // + 8 * buffer (FP8)
  volatile Ctl* ctl = reinterpret_cast<volatile Ctl*>(smem + C::OFF_MISC);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---------------------------------------------------------------- setup
  if (warp == WARP_LOAD && lane == 0) {
    mbar_init(BAR_Q_FULL, 1);
    mbar_init(BAR_Q_EMPTY, 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(BAR_KV_FULL + 8 * s, 1);
      // FP8: V tiles (odd slots) are released by the two widening warps
      mbar_init(BAR_KV_EMPTY + 8 * s, (FP8 && (s & 1)) ? 2 : 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR_S_FULL + 8 * t, 1);
      // one elected arrive per softmax warp; a barrier per P half, so each
      // completes once per K/V tile and its parity cannot run ahead
      mbar_init(BAR_P_FULL + 16 * t, BM / 32);
      mbar_init(BAR_P_FULL + 16 * t + 8, BM / 32);
      mbar_init(BAR_O_FULL + 8 * t, 1);
    }
    mbar_init(BAR_DRAIN, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR_VF_FULL + 8 * b, 2);   // one elected arrive per widening warp
      mbar_init(BAR_VF_EMPTY + 8 * b, 1);  // the MMA thread's commit
    }
    ctl->abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == WARP_MMA) {
    tmem_alloc(sbase + C::OFF_MISC, C::TMEM_COLS);  // writes ctl->tmem_base
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp >= 8) {
  // ===================================== warps 8+ (MMA, TMA, V widening)
  if constexpr (C::REBALANCE) setmaxnreg_dec<C::REGS_OTHER>();
  if (warp == WARP_LOAD) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0, qit = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        Unit U;
        const int st = cta_unit(i, P, U);
        if (st == 0) break;
        if (st == 1 || U.nmax == 0) continue;
        if (!wait_bounded(BAR_Q_EMPTY, (qit & 1u) ^ 1u, ctl, P)) { ok = false; break; }
#ifndef ATTN_TEST_NEVER_ARM_Q
        const int nq = (U.n[0] > 0) + (U.n[1] > 0);
        mbar_arrive_expect_tx(BAR_Q_FULL, nq * C::Q_TILE_BYTES);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (U.n[t] == 0) continue;
#pragma unroll
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_4d(sbase + C::OFF_Q + t * C::Q_TILE_BYTES + c * C::Q_CHUNK_BYTES, &tm_q,
                        BAR_Q_FULL, c * C::CHUNK_ELEMS, U.hq, U.row0 + t * BM, U.b);
        }
        ++qit;
#endif
        // (The watchdog test library is built with ATTN_TEST_NEVER_ARM_Q: Q is
        // never loaded and q_full never completes, so the MMA warp's bounded
        // wait runs out and the launch ends with ATTN_ERR_TIMEOUT.)
        for (int j = 0; ok && j < U.nmax; ++j) {
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t slot = it % C::NSLOT;
            if (!wait_bounded(BAR_KV_EMPTY + 8 * slot, ((it / C::NSLOT) & 1u) ^ 1u, ctl, P)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(BAR_KV_FULL + 8 * slot, C::KV_TILE_BYTES);
#pragma unroll
            for (int c = 0; c < C::NCHUNK; ++c)
              tma_load_4d(sbase + C::OFF_KV + slot * C::KV_TILE_BYTES + c * C::KV_CHUNK_BYTES,
                          kv ? &tm_v : &tm_k, BAR_KV_FULL + 8 * slot, c * C::CHUNK_ELEMS, U.hkv,
                          (U.j0 + j) * BN, U.b);
            ++it;
          }
        }
      }
      // Drain: every copy issued must land before the CTA may exit.
      for (uint32_t s = 0; s < C::NSLOT; ++s) {
        if (it > s) {
          const uint32_t fills = (it - 1 - s) / C::NSLOT + 1;
          drain_wait(BAR_KV_FULL + 8 * s, (fills - 1) & 1u, P);
        }
      }
      if (qit > 0) drain_wait(BAR_Q_FULL, (qit - 1) & 1u, P);
    }
    __syncwarp();
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (warp-uniform control flow, so the loop
    // state and the operand descriptors stay in uniform registers); one
    // elected lane issues every tcgen05.mma and tcgen05.commit.
    uint32_t it = 0, qit = 0;
    uint32_t pc[2] = {0u, 0u};
    bool ok = true;
    // descriptors of Q tile 0 and of K/V slot 0 (K-major, as staged by TMA),
    // and of the V operand of slot 0 or (FP8) of widened buffer 0 (MN-major)
    const uint64_t q_desc = make_sdesc(sbase + C::OFF_Q, 16, 8 * C::CHUNK_BYTES, C::SWZ_CODE);
    const uint64_t k_desc = make_sdesc(sbase + C::OFF_KV, 16, 8 * C::CHUNK_BYTES, C::SWZ_CODE);
    const uint64_t v_desc = make_sdesc(sbase + (FP8 ? C::OFF_VF : C::OFF_KV), C::V_KV_CHUNK_BYTES,
                                       8 * C::V_CHUNK_BYTES, 2u);
    // every lane waits; the warp proceeds only if all of them saw the phase
    auto wait_w = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_bounded(bar, parity, ctl, P));
    };
    auto issue_s = [&](int t, uint32_t slot) {
      issue_qk_w<D, FP8, F16>(tmem + C::COL_S0 + t * BN,
                              sdesc_add(q_desc, t * C::Q_TILE_BYTES),
                              sdesc_add(k_desc, slot * C::KV_TILE_BYTES));
    };
    auto issue_o = [&](int t, uint64_t vd, int half, bool acc) {
      issue_pv_half_w<D, FP8, F16>(tmem + C::COL_O0 + t * D, tmem + C::COL_S0 + t * BN, vd,
                                   half, acc);
    };

    // The next unit is worked out while this one's products run, so that
    // the step from one unit's last P V to the next unit's first S is only
    // waits and issues.
    Unit Un;
    int stn = cta_unit(0, P, Un);
    for (int i = 0; ok; ++i) {
      const Unit U = Un;
      const int st = stn;
      if (st == 0) break;
      if (st == 1 || U.nmax == 0) {
        stn = cta_unit(i + 1, P, Un);
        continue;
      }
      if (!wait_w(BAR_Q_FULL, qit & 1u)) { ok = false; break; }
      tc_fence_after();
      {
        const uint32_t slot = it % C::NSLOT;
        if (!wait_w(BAR_KV_FULL + 8 * slot, (it / C::NSLOT) & 1u)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (U.n[t] > 0) {
            issue_s(t, slot);
            tc_commit_w(BAR_S_FULL + 8 * t);
          }
        tc_commit_w(BAR_KV_EMPTY + 8 * slot);
        if (U.nmax == 1) tc_commit_w(BAR_Q_EMPTY);
      }
      stn = cta_unit(i + 1, P, Un);
      for (int j = 0; j < U.nmax; ++j) {
        const uint32_t itv = it + 2 * j + 1, vslot = itv % C::NSLOT;
        const uint32_t itk = itv + 1, kslot = itk % C::NSLOT;
        const bool more = j + 1 < U.nmax;
        // FP8: the widening warps wait for the staged V tile; this warp
        // waits for their fp16 copy (buffer = V use parity)
        const uint32_t vuse = itv >> 1, vbuf = vuse & 1u;
        const uint64_t vd = FP8 ? sdesc_add(v_desc, vbuf * C::V16_TILE_BYTES)
                                : sdesc_add(v_desc, vslot * C::KV_TILE_BYTES);
        if (FP8) {
          if (!wait_w(BAR_VF_FULL + 8 * vbuf, (vuse >> 1) & 1u)) { ok = false; break; }
        } else {
          if (!wait_w(BAR_KV_FULL + 8 * vslot, (itv / C::NSLOT) & 1u)) { ok = false; break; }
        }
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (j < U.n[t]) {
            // P arrives in two halves of 64 keys, one barrier each
            for (int h = 0; ok && h < 2; ++h) {
              if (!wait_w(BAR_P_FULL + 16 * t + 8 * h, pc[t] & 1u)) { ok = false; break; }
              tc_fence_after();
              issue_o(t, vd, h, j > 0);
            }
            if (!ok) break;
            ++pc[t];
            if (j == U.n[t] - 1) tc_commit_w(BAR_O_FULL + 8 * t);
          }
          if (t == 0 && more) {
            if (!wait_w(BAR_KV_FULL + 8 * kslot, (itk / C::NSLOT) & 1u)) { ok = false; break; }
            tc_fence_after();
          }
          if (j + 1 < U.n[t]) {
            issue_s(t, kslot);
            tc_commit_w(BAR_S_FULL + 8 * t);
          }
        }
        if (!ok) break;
        tc_commit_w(FP8 ? BAR_VF_EMPTY + 8 * vbuf : BAR_KV_EMPTY + 8 * vslot);
        if (more) {
          tc_commit_w(BAR_KV_EMPTY + 8 * kslot);
          if (j + 2 == U.nmax) tc_commit_w(BAR_Q_EMPTY);
        }
      }
      it += 2 * U.nmax;
      ++qit;
    }
    // Drain: all issued MMAs complete before the tensor memory is freed.
    tc_commit_w(BAR_DRAIN);
    drain_wait(BAR_DRAIN, 0u, P);
    __syncwarp();
  } else if (FP8 && warp >= WARP_WIDEN) {
    // ------------------------------------------------ V widening (FP8 only)
    // Each staged E4M3 V tile is copied to fp16 (exactly) in one of two
    // buffers, so that O += P V can keep P in fp16; the staged slot is then
    // released here. Same units and fill order as the producer.
    const int wtid = threadIdx.x - WARP_WIDEN * 32;
    uint32_t it = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      Unit U;
      const int st = cta_unit(i, P, U);
      if (st == 0) break;
      if (st == 1 || U.nmax == 0) continue;
      for (int j = 0; j < U.nmax; ++j) {
        const uint32_t itv = it + 2 * j + 1, vslot = itv % C::NSLOT;
        const uint32_t vuse = itv >> 1, vbuf = vuse & 1u;
        bool w = wait_bounded(BAR_KV_FULL + 8 * vslot, (itv / C::NSLOT) & 1u, ctl, P);
        w = w && wait_bounded(BAR_VF_EMPTY + 8 * vbuf, ((vuse >> 1) & 1u) ^ 1u, ctl, P);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        widen_v_tile<D>(sbase + C::OFF_KV + vslot * C::KV_TILE_BYTES,
                        sbase + C::OFF_VF + vbuf * C::V16_TILE_BYTES, wtid, 64);
        fence_proxy_async_smem();  // the fp16 tile is read by the tensor cores
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(BAR_VF_FULL + 8 * vbuf);
          mbar_arrive(BAR_KV_EMPTY + 8 * vslot);
        }
      }
      it += 2 * U.nmax;
    }
  }
  } else {
    // ========================================= softmax warpgroups 0 and 1
    if constexpr (C::REBALANCE) setmaxnreg_inc<C::REGS_SOFTMAX>();
    const int t = warp >> 2;           // Q tile handled by this warpgroup
    const int quad = warp & 3;         // TMEM lane quadrant of this warp
    const int rloc = quad * 32 + lane; // row within the tile == TMEM lane
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t col_s = C::COL_S0 + t * BN;
    const uint32_t col_o = C::COL_O0 + t * D;
    const float cs = P.scale_log2;
    const int nblk_q = ceil_div(P.Sq, FP8_BLOCK);
    const int nblk_k = ceil_div(P.Sk, FP8_BLOCK);
    uint32_t sc = 0, oc = 0;  // phase counters of s_full[t], o_full[t]
    bool ok = true;

    for (int i = 0; ok; ++i) {
      Unit U;
      const int st = cta_unit(i, P, U);
      if (st == 0) break;
      if (st == 1) continue;
      const int tile_row0 = U.row0 + t * BM;
      if (tile_row0 >= P.Sq) continue;  // idle tile
      const int row = tile_row0 + rloc;
      const bool row_ok = row < P.Sq;
      const int n = t ? U.n[1] : U.n[0];
      float m_run = -INFINITY, l_run = 0.f;
      float cq = cs;         // per-row exponent scale (FP8: times the Q block scale)
      float v_ref = 1.f;     // FP8: largest V block scale of this KV head
      const float* ks_row = nullptr;
      const float* vs_row = nullptr;
      if constexpr (FP8) {
        if (P.q_scale != nullptr) {  // null scales mean all block scales are 1
          const float sq = row_ok ? P.q_scale[(static_cast<size_t>(U.b) * P.Hq + U.hq) * nblk_q +
                                              row / FP8_BLOCK]
                                  : 1.f;
          cq = cs * sq;
          ks_row = P.k_scale + (static_cast<size_t>(U.b) * P.Hkv + U.hkv) * nblk_k;
          vs_row = P.v_scale + (static_cast<size_t>(U.b) * P.Hkv + U.hkv) * nblk_k;
          float vm = 0.f;
          for (int i = 0; i < nblk_k; ++i) vm = fmaxf(vm, vs_row[i]);
          v_ref = vm > 0.f ? vm : 1.f;
        }
      }

      for (int j = 0; j < n; ++j) {
        // per-column-half exponent scales. FP8: the first and second 64 keys
        // of the tile are two scale blocks of K and of V; e_* = log2 of the
        // factor p is multiplied by before it is rounded to fp16 (V block
        // scale / largest V scale of the head, <= 1), inv_* = 1 / that factor.
        // They depend only on the tile, so they are formed before the wait
        // for S, off the path from S to P.
        float c_lo = cq, c_hi = cq;
        float e_lo = 0.f, e_hi = 0.f;
        float inv_lo = 1.f, inv_hi = 1.f;
        if (FP8 && ks_row != nullptr) {
          const int kb0 = 2 * (U.j0 + j), kb1 = kb0 + 1;
          const float vs0 = vs_row[kb0];
          const float vs1 = kb1 < nblk_k ? vs_row[kb1] : v_ref;
          c_lo = cq * ks_row[kb0];
          c_hi = cq * (kb1 < nblk_k ? ks_row[kb1] : 1.f);
          e_lo = __log2f(vs0 / v_ref);
          e_hi = __log2f(vs1 / v_ref);
          inv_lo = v_ref / vs0;
          inv_hi = v_ref / vs1;
        }
        bool w = wait_bounded(BAR_S_FULL + 8 * t, sc & 1u, ctl, P);
        ++sc;
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after();

        // all four 32-column loads in flight, one wait
        float s[BN];
        {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld32_async(t_lane + col_s + 0, r0);
          tmem_ld32_async(t_lane + col_s + 32, r1);
          tmem_ld32_async(t_lane + col_s + 64, r2);
          tmem_ld32_async(t_lane + col_s + 96, r3);
          tmem_ld_wait();
          reg_fence(r0);
          reg_fence(r1);
          reg_fence(r2);
          reg_fence(r3);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            s[c] = __uint_as_float(r0[c]);
            s[32 + c] = __uint_as_float(r1[c]);
            s[64 + c] = __uint_as_float(r2[c]);
            s[96 + c] = __uint_as_float(r3[c]);
          }
        }
        // mask: keys past Sk, and (causal) keys after row + Sk - Sq
        const int key0 = (U.j0 + j) * BN;
        int vis = P.Sk - key0;
        if (P.causal) vis = min(vis, row + (P.Sk - P.Sq) - key0 + 1);
        if (vis < BN) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= vis) s[c] = -INFINITY;
        }
        // row max of each 64-key half (raw scores; the exponent scale of a
        // half is positive, so it commutes with the max)
        float mx[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float* h = s + 64 * i;
          float a0 = h[0], a1 = h[1], a2 = h[2], a3 = h[3];
#pragma unroll
          for (int c = 4; c < 60; c += 8) {
            a0 = max3(a0, h[c], h[c + 1]);
            a1 = max3(a1, h[c + 2], h[c + 3]);
            a2 = max3(a2, h[c + 4], h[c + 5]);
            a3 = max3(a3, h[c + 6], h[c + 7]);
          }
          a0 = max3(a0, h[60], h[61]);
          a1 = max3(a1, h[62], h[63]);
          mx[i] = fmaxf(max3(a0, a1, a2), a3);
        }
        const float m_tile = fmaxf(mx[0] * c_lo, mx[1] * c_hi);
        const float m_new = fmaxf(m_run, m_tile);
        const bool need = (m_new - m_run) > C::RESCALE;  // false when both are -inf
        float factor = 1.f;
        if (need) {
          factor = ex2_approx(m_run - m_new);
          l_run *= factor;
          m_run = m_new;
        }
        const float msafe = (m_run == -INFINITY) ? 0.f : m_run;
        // O_t holds the sum over earlier tiles (S_t(j) completing implies the
        // previous O_t += P V has completed too); it is rescaled before the
        // first half of P is handed over, after that half's registers are free.
        const bool rescale_o = j > 0 && __any_sync(0xffffffffu, need);

        // p = 2^(s * c - m): paired fp32 FMA, one MUFU ex2 per key, paired
        // sums. FP8: p' = p * rr, rr = V block scale / v_ref (log2 rr folded
        // into the offset) so that P V runs on the V codes; each half sums
        // its p' separately and is divided back when added to l. P is kept
        // in fp16 for FP8 and fp16 inputs, bf16 otherwise.
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float cc = i ? c_hi : c_lo;
          const float off = (FP8 ? (i ? e_hi : e_lo) : 0.f) - msafe;
          const uint64_t cc2 = f2_pack(cc, cc), off2 = f2_pack(off, off);
          uint64_t acc0 = 0ull, acc1 = 0ull;  // (+0, +0) pairs
          const float* h = s + 64 * i;
          {
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float x0, x1, x2, x3;
              f2_unpack(f2_fma(f2_pack(h[2 * c], h[2 * c + 1]), cc2, off2), x0, x1);
              f2_unpack(f2_fma(f2_pack(h[2 * c + 2], h[2 * c + 3]), cc2, off2), x2, x3);
              const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
              acc0 = f2_add(acc0, f2_pack(p0, p1));
              acc1 = f2_add(acc1, f2_pack(p2, p3));
              pk[c] = (F16 || FP8) ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
              pk[c + 1] = (F16 || FP8) ? pack_f16x2(p2, p3) : pack_bf16x2(p2, p3);
            }
            tmem_st32(t_lane + col_s + 32 * i, pk);
          }
          float q0, q1, q2, q3;
          f2_unpack(acc0, q0, q1);
          f2_unpack(acc1, q2, q3);
          const float lsum = (q0 + q1) + (q2 + q3);
          if constexpr (FP8) l_run += lsum * (i ? inv_hi : inv_lo);
          else l_run += lsum;
          if (i == 0 && rescale_o) {
#pragma unroll
            for (int k = 0; k < D / 32; ++k) {
              uint32_t r[32];
              tmem_ld32(t_lane + col_o + 32 * k, r);
#pragma unroll
              for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * factor);
              tmem_st32(t_lane + col_o + 32 * k, r);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR_P_FULL + 16 * t + 8 * i);
        }
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      const size_t lse_idx = (static_cast<size_t>(U.b) * P.Hq + U.hq) * P.Sq + row;
      if (P.o_part != nullptr) {
        // split-KV: this key range's O / l (fp32) and LSE, for the combine
        const size_t pidx =
            static_cast<size_t>(U.split) * P.B * P.Hq * P.Sq + lse_idx;
        float* prow = P.o_part + pidx * D;
        float inv = 0.f;
        if (n > 0) {
          bool w = wait_bounded(BAR_O_FULL + 8 * t, oc & 1u, ctl, P);
          ++oc;
          if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
          tc_fence_after();
          inv = l_run > 0.f ? v_ref / l_run : 0.f;
#pragma unroll
          for (int i = 0; i < D / 32; ++i) {
            uint32_t r[32];
            tmem_ld32(t_lane + col_o + 32 * i, r);
            if (row_ok) {
              float4* dst = reinterpret_cast<float4*>(prow + 32 * i);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                     __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
            }
          }
        } else if (row_ok) {
          float4* dst = reinterpret_cast<float4*>(prow);
#pragma unroll
          for (int v = 0; v < D / 4; ++v) dst[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (row_ok)
          P.lse_part[pidx] = (n > 0 && l_run > 0.f) ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
        continue;
      }
      uint16_t* orow =
          P.o + ((static_cast<size_t>(U.b) * P.Sq + row) * P.Hq + U.hq) * static_cast<size_t>(D);
      if (n > 0) {
        bool w = wait_bounded(BAR_O_FULL + 8 * t, oc & 1u, ctl, P);
        ++oc;
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after();
        // FP8: O holds sum p * (V block scale / v_ref) * code
        const float inv = l_run > 0.f ? v_ref / l_run : 0.f;
        if constexpr (C::STAGE_O) {
          // Per 32-column quarter: this thread's 64 bytes of its row go to
          // row `lane` of the warp's staging area (64-byte rows), 16-byte
          // chunk c at position c ^ ((row >> 1) & 3), so that every 8 lanes
          // of a shared-memory access cover all 32 banks; then store k
          // writes rows 8k .. 8k + 7 of the warp, 4 lanes per row, 64
          // contiguous bytes each.
          // (the staging addresses are formed here, not hoisted out of the
          // unit loop, where they would hold registers the softmax needs)
          uint32_t stg = sbase + C::OFF_OSTAGE + warp * C::OSTAGE_WARP_BYTES;
          int ln = lane, sq = P.Sq, hqn = P.Hq;
          asm volatile("" : "+r"(stg), "+r"(ln), "+r"(sq), "+r"(hqn));
          const int c4 = ln & 3;
          const int rr0 = ln >> 2;  // first row this lane stores
          const int rows_left = sq - (tile_row0 + quad * 32 + rr0);
          const size_t ostride = static_cast<size_t>(hqn) * D;  // elements between rows
          uint16_t* odst = P.o + ((static_cast<size_t>(U.b) * sq + tile_row0 + quad * 32 + rr0) * hqn +
                                  U.hq) * static_cast<size_t>(D) + 8 * c4;
#pragma unroll 1
          for (int qq = 0; qq < D / 32; ++qq) {
            uint32_t r[32];
            tmem_ld32(t_lane + col_o + 32 * qq, r);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t pk[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float a = __uint_as_float(r[8 * c + 2 * e]) * inv;
                const float b = __uint_as_float(r[8 * c + 2 * e + 1]) * inv;
                pk[e] = F16 ? pack_f16x2(a, b) : pack_bf16x2(a, b);
              }
              sts128(stg + ln * 64 + ((c ^ ((ln >> 1) & 3)) << 4),
                     make_uint4(pk[0], pk[1], pk[2], pk[3]));
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int rr = 8 * k + rr0;
              const uint4 v = lds128(stg + rr * 64 + ((c4 ^ ((rr >> 1) & 3)) << 4));
              if (8 * k < rows_left)
                *reinterpret_cast<uint4*>(odst + 8 * k * ostride + 32 * qq) = v;
            }
            __syncwarp();  // the next quarter overwrites the staging area
          }
        } else {
#pragma unroll
          for (int i = 0; i < D / 32; ++i) {
            uint32_t r[32];
            tmem_ld32(t_lane + col_o + 32 * i, r);
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
              pk[c] = F16 ? pack_f16x2(__uint_as_float(r[2 * c]) * inv, __uint_as_float(r[2 * c + 1]) * inv)
                          : pack_bf16x2(__uint_as_float(r[2 * c]) * inv, __uint_as_float(r[2 * c + 1]) * inv);
            if (row_ok) {
              uint4* dst = reinterpret_cast<uint4*>(orow + 32 * i);
#pragma unroll
              for (int v = 0; v < 4; ++v)
                dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
          }
        }
        if (row_ok) P.lse[lse_idx] = l_run > 0.f ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
      } else if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
        P.lse[lse_idx] = -INFINITY;
      }
    }
  }

  // --------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace attnb3
