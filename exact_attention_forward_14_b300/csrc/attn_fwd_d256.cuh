// attn_fwd_d256.cuh -- the attention forward pass for head dimension 256.
//
// Same method and numerics as attn_fwd_kernel.cuh (the FlashAttention-3 deep
// dive's tiled forward with an exp2 online softmax and stale-max rescaling,
// techknowgenie.com/posts/109164421204410442, sections 2-3), in a layout that
// fits d = 256: two 128-row Q tiles in ping-pong would need 2 x (128 S +
// 256 O) = 768 TMEM columns against 512. Here a unit is one 128-row Q tile
// (b, hq, 128 rows), and the keys stream past in 128-key steps:
//   TMEM    S in two buffers [0,128) and [128,256), P(j) (packed 16-bit
//           pairs) over the low 64 columns of S(j)'s buffer, O [256,512)
//   smem    Q (64 KB, resident for the unit) and a 5-slot ring of 32 KB
//           chunks: a step's K tile (128 keys x 256) as two chunks of 128
//           columns of d, its V tile as two chunks of 64 keys
//   MMAs    S(j) = Q K_j^T  (M = 128, N = 128, K = 256 in two chunks),
//           issued two steps ahead into buffer j & 1;  O += P(j) V_j
//           (M = 128, N = 256, K = 128 in two chunks, P from TMEM)
//   issue   S(0) S(1) | <-P(0) PV(0) S(2) | <-P(1) PV(1) S(3) | ...
// so the softmax of step j+1 overlaps PV(j) and S(j+2). The ring is filled
// in the order the MMAs read it (K0 K1 V0 K2 V1 K3 ...), so the chunks in
// use and the next ones fit five slots. S(j+2) overwrites the buffer that
// holds P(j) and is issued after PV(j) by the same thread; in-order
// execution keeps it from writing before P(j) has been read.
// The P barrier is per buffer: S(j+1) is already complete when a warp
// finishes P(j), so a fast warp can arrive for step j+1 before a slow one has
// arrived for step j, and with one barrier that early arrival would complete
// step j's phase. A warp cannot run two steps ahead, because S(j+2) waits
// for PV(j). Because the next S is already in flight, "S(j+1) complete" no
// longer implies "PV(j) complete": a softmax step that must rescale O first
// waits for pv_done of PV(j).
//
// 192 threads: warps 0-3 softmax (thread = query row = TMEM lane), warp 4
// MMA issuer and TMEM owner, warp 5 TMA producer. Every wait is bounded
// (wait_bounded / drain_wait of the main kernel).
//
// FwdParams fields as used here: n_qp = ceil(Sq / 128) Q tiles, npair =
// ceil(n_qp / 2) work items per (b, hq) (Q tile n_qp-1-p paired with tile p),
// nkv = ceil(Sk / 128) key steps, num_items = B * Hq * npair.
#pragma once

#include "attn_fwd_kernel.cuh"

namespace attnb3 {

constexpr int WIDE_D = 256;
constexpr int WIDE_BN = 128;        // keys per step (rows of a K tile)
constexpr int WIDE_VROWS = 64;      // keys per V chunk
constexpr int WIDE_THREADS = 192;
constexpr int WIDE_WARP_MMA = 4;
constexpr int WIDE_WARP_LOAD = 5;

template <bool F16>
struct WideCfg {
  static constexpr uint32_t FMT = F16 ? 0u : 1u;
  static constexpr int CHUNK = 128;       // bytes of a swizzled row span (64 elements)
  static constexpr int CHUNK_ELEMS = 64;
  static constexpr int Q_BYTES = BM * WIDE_D * 2;
  static constexpr int Q_CH = BM * CHUNK;                  // one 64-column span of Q
  static constexpr int SLOT_BYTES = 32 * 1024;              // one ring chunk
  static constexpr int K_SUB = WIDE_BN * CHUNK;             // 64-column span of a K chunk
  static constexpr int V_SUB = WIDE_VROWS * CHUNK;          // 64-column span of a V chunk
  static_assert(2 * K_SUB == SLOT_BYTES && 4 * V_SUB == SLOT_BYTES, "chunk sizes");
  static constexpr int NSLOT = 5;
  static constexpr uint32_t IDESC_S = make_idesc(BM, WIDE_BN, FMT, false);
  static constexpr uint32_t IDESC_PV = make_idesc(BM, WIDE_D, FMT, true);
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = Q_BYTES;
  static constexpr int OFF_BAR = OFF_KV + NSLOT * SLOT_BYTES;
  // q_full, q_empty, kv_full[NSLOT], kv_empty[NSLOT], s_full[2], p_full[2],
  // pv_done, o_full, drain
  static constexpr int NBAR = 2 + 2 * NSLOT + 7;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int SMEM_ALLOC = 227 * 1024;
  static constexpr int COL_S0 = 0;
  static constexpr int COL_S1 = WIDE_BN;
  static constexpr int COL_O = 256;
  static constexpr int TMEM_COLS = 512;
  static_assert(SMEM_BYTES <= SMEM_ALLOC, "shared memory budget");
  static_assert(2 * WIDE_BN <= COL_O && COL_O + WIDE_D <= TMEM_COLS, "TMEM budget");
};

struct WideUnit {
  int b, hq, hkv, row0;
  int n;  // 128-key steps seen by the unit's rows (0 = every row fully masked)
};

// The i-th unit of this CTA: 0 = none left, 1 = skip, 2 = U filled. Work
// item w = (b, hq, p) pairs Q tile n_qp-1-p (the most keys under a causal
// mask) with Q tile p; query heads innermost, so the CTAs in flight share a
// few KV heads' K and V in L2.
__device__ __forceinline__ int wide_unit(int i, const FwdParams& P, WideUnit& U) {
  const int w = blockIdx.x + (i >> 1) * gridDim.x;
  if (w >= P.num_items) return 0;
  const int bh = w / P.npair, p = w - bh * P.npair;
  const int qi = (i & 1) ? p : P.n_qp - 1 - p;
  if ((i & 1) && qi == P.n_qp - 1 - p) return 1;  // odd n_qp: the middle tile
  U.b = bh / P.Hq;
  U.hq = bh - U.b * P.Hq;
  U.hkv = U.hq / P.group;
  U.row0 = qi * BM;
  U.n = P.nkv;
  if (P.causal) {
    const int lim = min(U.row0 + BM, P.Sq) + (P.Sk - P.Sq);  // keys seen by the last row
    U.n = lim <= 0 ? 0 : min((lim + WIDE_BN - 1) / WIDE_BN, P.nkv);
  }
  return 2;
}

// Ring fills of a unit with n steps, from its first fill `base`, in the
// order the MMAs read them: K0 K1 V0 K2 V1 K3 ... V(n-2) V(n-1), two chunks
// each (4 n fills in all).
__device__ __forceinline__ uint32_t wide_fill_k(uint32_t base, int j, int c) {
  return base + (j < 2 ? 2 * j : 4 * j - 2) + c;
}
__device__ __forceinline__ uint32_t wide_fill_v(uint32_t base, int n, int j, int c) {
  return base + (n == 1 ? 2 : (j <= n - 2 ? 4 + 4 * j : 4 * n - 2)) + c;
}

// The part of S = Q K^T that one K chunk holds: columns [128 c, 128 c + 128)
// of d, as two 64-column swizzled spans of the chunk; 32 bytes of d per
// instruction. Warp-collective: the MMA warp runs it with descriptors of the
// first bytes of Q and of the chunk, and each K step adds a constant offset.
template <bool F16>
__device__ __forceinline__ void wide_issue_s_chunk(uint32_t d_tmem, uint64_t q_desc,
                                                   uint64_t k_desc, int c) {
  using C = WideCfg<F16>;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t byte_k = ks * 32;
    const uint32_t sub = byte_k / C::CHUNK, within = byte_k % C::CHUNK;
    mma_f16_ss_w(d_tmem, sdesc_add(q_desc, (2 * c + sub) * C::Q_CH + within),
                 sdesc_add(k_desc, sub * C::K_SUB + within), C::IDESC_S,
                 (c > 0 || ks > 0) ? 1u : 0u);
  }
}

// O (+)= P V for the 64 keys of V chunk c: P columns [32 c, 32 c + 32) of
// the S buffer (16-bit pairs), the chunk = 64 keys x 256 (d contiguous,
// MN-major, 64-column spans V_SUB bytes apart); 16 keys per instruction.
template <bool F16>
__device__ __forceinline__ void wide_issue_pv_chunk(uint32_t d_tmem, uint32_t p_tmem,
                                                    uint64_t v_desc, int c, bool accumulate) {
  using C = WideCfg<F16>;
#pragma unroll
  for (int k = 0; k < WIDE_VROWS / 16; ++k)
    mma_f16_ts_w(d_tmem, p_tmem + 32 * c + 8 * k, sdesc_add(v_desc, 16 * k * C::CHUNK),
                 C::IDESC_PV, (accumulate || k > 0) ? 1u : 0u);
}

template <bool F16>
__global__ void __launch_bounds__(WIDE_THREADS, 1)
    attn_fwd_d256_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const FwdParams P) {
  using C = WideCfg<F16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t BAR_Q_FULL = bar0;
  const uint32_t BAR_Q_EMPTY = bar0 + 8;
  const uint32_t BAR_KV_FULL = bar0 + 16;                    // + 8 * slot
  const uint32_t BAR_KV_EMPTY = BAR_KV_FULL + 8 * C::NSLOT;  // + 8 * slot
  const uint32_t BAR_S_FULL = BAR_KV_EMPTY + 8 * C::NSLOT;   // + 8 * S buffer
  const uint32_t BAR_P_FULL = BAR_S_FULL + 16;                // + 8 * S buffer
  const uint32_t BAR_PV_DONE = BAR_P_FULL + 16;
  const uint32_t BAR_O_FULL = BAR_PV_DONE + 8;
  const uint32_t BAR_DRAIN = BAR_O_FULL + 8;
  volatile Ctl* ctl = reinterpret_cast<volatile Ctl*>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == WIDE_WARP_LOAD && lane == 0) {
    mbar_init(BAR_Q_FULL, 1);
    mbar_init(BAR_Q_EMPTY, 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(BAR_KV_FULL + 8 * s, 1);
      mbar_init(BAR_KV_EMPTY + 8 * s, 1);
    }
    mbar_init(BAR_S_FULL, 1);
    mbar_init(BAR_S_FULL + 8, 1);
    mbar_init(BAR_P_FULL, BM / 32);  // one elected arrive per softmax warp
    mbar_init(BAR_P_FULL + 8, BM / 32);
    mbar_init(BAR_PV_DONE, 1);
    mbar_init(BAR_O_FULL, 1);
    mbar_init(BAR_DRAIN, 1);
    ctl->abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == WIDE_WARP_MMA) {
    tmem_alloc(sbase + C::OFF_MISC, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  auto col_sbuf = [](uint32_t j) { return (j & 1u) ? C::COL_S1 : C::COL_S0; };

  if (warp == WIDE_WARP_LOAD) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0, qit = 0;
      bool ok = true;
      // next ring fill: a K chunk (128 keys, columns [128 c, 128 c + 128) of
      // d, two 64-column boxes) or a V chunk (64 keys, all of d, four boxes)
      auto fill = [&](bool is_v, int j, int c, const WideUnit& U) {
        const uint32_t slot = it % C::NSLOT;
        if (!wait_bounded(BAR_KV_EMPTY + 8 * slot, ((it / C::NSLOT) & 1u) ^ 1u, ctl, P))
          return false;
        const uint32_t dst = sbase + C::OFF_KV + slot * C::SLOT_BYTES;
        const uint32_t bar = BAR_KV_FULL + 8 * slot;
        mbar_arrive_expect_tx(bar, C::SLOT_BYTES);
        if (is_v) {
#pragma unroll
          for (int s = 0; s < 4; ++s)
            tma_load_4d(dst + s * C::V_SUB, &tm_v, bar, s * C::CHUNK_ELEMS, U.hkv,
                        j * WIDE_BN + c * WIDE_VROWS, U.b);
        } else {
#pragma unroll
          for (int s = 0; s < 2; ++s)
            tma_load_4d(dst + s * C::K_SUB, &tm_k, bar, (2 * c + s) * C::CHUNK_ELEMS, U.hkv,
                        j * WIDE_BN, U.b);
        }
        ++it;
        return true;
      };
      for (int i = 0; ok; ++i) {
        WideUnit U;
        const int st = wide_unit(i, P, U);
        if (st == 0) break;
        if (st == 1 || U.n == 0) continue;
        if (!wait_bounded(BAR_Q_EMPTY, (qit & 1u) ^ 1u, ctl, P)) { ok = false; break; }
#ifndef ATTN_TEST_NEVER_ARM_Q
        mbar_arrive_expect_tx(BAR_Q_FULL, C::Q_BYTES);
#pragma unroll
        for (int c = 0; c < WIDE_D / C::CHUNK_ELEMS; ++c)
          tma_load_4d(sbase + C::OFF_Q + c * C::Q_CH, &tm_q, BAR_Q_FULL, c * C::CHUNK_ELEMS, U.hq,
                      U.row0, U.b);
        ++qit;
#endif  // (watchdog test library: Q never loaded, q_full never completes)
        // the MMAs' order: K0 K1 V0 K2 V1 K3 ... (wide_fill_k / wide_fill_v)
        const int n = U.n;
        for (int j = 0; ok && j < 2 && j < n; ++j)
          ok = fill(false, j, 0, U) && fill(false, j, 1, U);
        for (int j = 0; ok && j < n; ++j) {
          ok = fill(true, j, 0, U) && fill(true, j, 1, U);
          if (ok && j + 2 < n) ok = fill(false, j + 2, 0, U) && fill(false, j + 2, 1, U);
        }
      }
      for (uint32_t s = 0; s < static_cast<uint32_t>(C::NSLOT); ++s)
        if (it > s) drain_wait(BAR_KV_FULL + 8 * s, ((it - 1 - s) / C::NSLOT) & 1u, P);
      if (qit > 0) drain_wait(BAR_Q_FULL, (qit - 1) & 1u, P);
    }
    __syncwarp();
  } else if (warp == WIDE_WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // Every ring chunk is released as soon as the products that read it are
    // issued (the commit completes when they have run); Q after the unit's
    // last S. The whole warp runs the loop (uniform control flow and
    // descriptors); one elected lane issues each tcgen05 instruction.
    uint32_t it = 0, qit = 0, pc[2] = {0u, 0u};
    bool ok = true;
    const uint64_t q_desc = make_sdesc(sbase + C::OFF_Q, 16, 8 * C::CHUNK, 2u);
    const uint64_t k_desc = make_sdesc(sbase + C::OFF_KV, 16, 8 * C::CHUNK, 2u);
    const uint64_t v_desc = make_sdesc(sbase + C::OFF_KV, C::V_SUB, 8 * C::CHUNK, 2u);
    auto slot_off = [&](uint32_t f) { return (f % C::NSLOT) * C::SLOT_BYTES; };
    auto wait_w = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_bounded(bar, parity, ctl, P));
    };
    auto wait_fill = [&](uint32_t f) {
      return wait_w(BAR_KV_FULL + 8 * (f % C::NSLOT), (f / C::NSLOT) & 1u);
    };
    // S(j) into buffer j & 1, one K chunk at a time
    auto issue_s = [&](int j) {
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        const uint32_t f = wide_fill_k(it, j, c);
        if (!wait_fill(f)) return false;
        tc_fence_after();
        wide_issue_s_chunk<F16>(tmem + col_sbuf(j), q_desc, sdesc_add(k_desc, slot_off(f)), c);
        tc_commit_w(BAR_KV_EMPTY + 8 * (f % C::NSLOT));
      }
      tc_commit_w(BAR_S_FULL + 8 * (j & 1));
      return true;
    };
    for (int i = 0; ok; ++i) {
      WideUnit U;
      const int st = wide_unit(i, P, U);
      if (st == 0) break;
      if (st == 1 || U.n == 0) continue;
      const int n = U.n;
      if (!wait_w(BAR_Q_FULL, qit & 1u)) { ok = false; break; }
      tc_fence_after();
      if (!issue_s(0) || (n > 1 && !issue_s(1))) { ok = false; break; }
      if (n <= 2) tc_commit_w(BAR_Q_EMPTY);
      for (int j = 0; j < n; ++j) {
        if (!wait_w(BAR_P_FULL + 8 * (j & 1), pc[j & 1] & 1u)) { ok = false; break; }
        ++pc[j & 1];
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          const uint32_t f = wide_fill_v(it, n, j, c);
          if (!wait_fill(f)) { ok = false; break; }
          tc_fence_after();
          wide_issue_pv_chunk<F16>(tmem + C::COL_O, tmem + col_sbuf(j),
                                   sdesc_add(v_desc, slot_off(f)), c, j > 0 || c > 0);
          tc_commit_w(BAR_KV_EMPTY + 8 * (f % C::NSLOT));
        }
        if (!ok) break;
        tc_commit_w(BAR_PV_DONE);
        if (j + 2 < n) {
          if (!issue_s(j + 2)) { ok = false; break; }
          if (j + 3 == n) tc_commit_w(BAR_Q_EMPTY);  // S(n-1) was the last reader of Q
        }
      }
      if (!ok) break;
      tc_commit_w(BAR_O_FULL);
      it += 4 * n;
      ++qit;
    }
    tc_commit_w(BAR_DRAIN);
    drain_wait(BAR_DRAIN, 0u, P);
    __syncwarp();
  } else if (warp < BM / 32) {
    // ------------------------------------------------------------- softmax
    const int rloc = warp * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float cs = P.scale_log2;
    const uint64_t cs2 = f2_pack(cs, cs);
    uint32_t sfc[2] = {0u, 0u}, g = 0, oc = 0;  // S buffer phases, P count (global), O phases
    bool ok = true;
    for (int i = 0; ok; ++i) {
      WideUnit U;
      const int st = wide_unit(i, P, U);
      if (st == 0) break;
      if (st == 1) continue;
      const int row = U.row0 + rloc;
      const bool row_ok = row < P.Sq;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < U.n; ++j, ++g) {
        const uint32_t buf = j & 1;
        bool w = wait_bounded(BAR_S_FULL + 8 * buf, sfc[buf] & 1u, ctl, P);
        ++sfc[buf];
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after();
        const uint32_t col_s = col_sbuf(j);
        float s[WIDE_BN];
        {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld32_async(t_lane + col_s, r0);
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
        const int key0 = j * WIDE_BN;
        int vis = P.Sk - key0;
        if (P.causal) vis = min(vis, row + (P.Sk - P.Sq) - key0 + 1);
        if (vis < WIDE_BN) {
#pragma unroll
          for (int c = 0; c < WIDE_BN; ++c)
            if (c >= vis) s[c] = -INFINITY;
        }
        float a0 = s[0], a1 = s[1], a2 = s[2], a3 = s[3];
#pragma unroll
        for (int c = 4; c < 124; c += 8) {
          a0 = max3(a0, s[c], s[c + 1]);
          a1 = max3(a1, s[c + 2], s[c + 3]);
          a2 = max3(a2, s[c + 4], s[c + 5]);
          a3 = max3(a3, s[c + 6], s[c + 7]);
        }
        a0 = max3(a0, s[124], s[125]);
        a1 = max3(a1, s[126], s[127]);
        const float m_tile = fmaxf(max3(a0, a1, a2), a3) * cs;
        const float m_new = fmaxf(m_run, m_tile);
        const bool need = (m_new - m_run) > RESCALE_LOG2;  // false when both are -inf
        float factor = 1.f;
        if (need) {
          factor = ex2_approx(m_run - m_new);
          l_run *= factor;
          m_run = m_new;
        }
        const float msafe = (m_run == -INFINITY) ? 0.f : m_run;
        const uint64_t off2 = f2_pack(-msafe, -msafe);
        // P(j) over the low 64 columns of its S buffer: keys [64 h, 64 h + 64)
        // as 32 columns of 16-bit pairs at column 32 h
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint64_t acc0 = 0ull, acc1 = 0ull;
          uint32_t pk[32];
          const float* sh = s + 64 * h;
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            float x0, x1, x2, x3;
            f2_unpack(f2_fma(f2_pack(sh[c], sh[c + 1]), cs2, off2), x0, x1);
            f2_unpack(f2_fma(f2_pack(sh[c + 2], sh[c + 3]), cs2, off2), x2, x3);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            acc0 = f2_add(acc0, f2_pack(p0, p1));
            acc1 = f2_add(acc1, f2_pack(p2, p3));
            pk[c / 2] = F16 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            pk[c / 2 + 1] = F16 ? pack_f16x2(p2, p3) : pack_bf16x2(p2, p3);
          }
          tmem_st32(t_lane + col_s + 32 * h, pk);
          float q0, q1, q2, q3;
          f2_unpack(acc0, q0, q1);
          f2_unpack(acc1, q2, q3);
          l_run += (q0 + q1) + (q2 + q3);
        }
        // O holds the sum over steps before j once PV(j-1) has completed; it
        // is rescaled only when some row's max grew past the threshold
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          w = wait_bounded(BAR_PV_DONE, (g - 1) & 1u, ctl, P);
          if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int k = 0; k < WIDE_D / 32; ++k) {
            uint32_t r[32];
            tmem_ld32(t_lane + C::COL_O + 32 * k, r);
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * factor);
            tmem_st32(t_lane + C::COL_O + 32 * k, r);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR_P_FULL + 8 * buf);
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      const size_t lse_idx = (static_cast<size_t>(U.b) * P.Hq + U.hq) * P.Sq + row;
      uint16_t* orow = P.o + ((static_cast<size_t>(U.b) * P.Sq + row) * P.Hq + U.hq) *
                                 static_cast<size_t>(WIDE_D);
      if (U.n > 0) {
        const bool w = wait_bounded(BAR_O_FULL, oc & 1u, ctl, P);
        ++oc;
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
        for (int k = 0; k < WIDE_D / 32; ++k) {
          uint32_t r[32];
          tmem_ld32(t_lane + C::COL_O + 32 * k, r);
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[c] = F16 ? pack_f16x2(__uint_as_float(r[2 * c]) * inv,
                                     __uint_as_float(r[2 * c + 1]) * inv)
                        : pack_bf16x2(__uint_as_float(r[2 * c]) * inv,
                                      __uint_as_float(r[2 * c + 1]) * inv);
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(orow + 32 * k);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
        tc_fence_before();
        if (row_ok) P.lse[lse_idx] = l_run > 0.f ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
      } else if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int v = 0; v < WIDE_D / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
        P.lse[lse_idx] = -INFINITY;
      }
    }
  }

  // --------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == WIDE_WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace attnb3
