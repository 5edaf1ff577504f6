// widen_v.cuh -- E4M3 V tile -> fp16 V tile in shared memory, for the FP8
// path's O += P V step (P is kept in fp16; FP8 tensor-core operands must both
// be 8-bit, so V is widened instead; every E4M3 value is exact in fp16).
//
// Layouts, both as a 128-byte-swizzled TMA copy writes them (a row is one
// key; a row's 16-byte units are stored at unit ^ (row % 8) within each
// 1024-byte group of 8 rows):
//   source (E4M3, d bytes per key): d / 128 chunks of [128 keys][128 B];
//   target (fp16, 2 d bytes per key): 2 d / 128 chunks of [128 keys][128 B],
//   chunk c holding elements [64 c, 64 c + 64) of every key.
// One source 16-byte unit (16 codes) becomes two target units.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace attnb3 {

template <int D>
__device__ __forceinline__ void widen_v_tile(uint32_t src, uint32_t dst, int tid, int nthreads) {
  constexpr int KEYS = 128;
  constexpr int SRC_CHUNKS = D / 128 > 0 ? D / 128 : 1;  // d = 64: one 64-byte-row chunk
  constexpr int SRC_ROW = D < 128 ? D : 128;             // bytes per key in a source chunk
  constexpr int UNITS_PER_ROW = SRC_ROW / 16;            // 4 (d = 64) or 8
  constexpr int UNITS = KEYS * SRC_CHUNKS * UNITS_PER_ROW;
  for (int i = tid; i < UNITS; i += nthreads) {
    const int sc = i / (KEYS * UNITS_PER_ROW);         // source chunk
    const int rem = i - sc * KEYS * UNITS_PER_ROW;
    const int row = rem / UNITS_PER_ROW;
    const int u = rem - row * UNITS_PER_ROW;           // logical unit in the row
    // source: 128-byte swizzle for 128-byte rows, 64-byte swizzle for 64-byte
    // rows (unit ^ ((row / 2) % 4) over 512-byte groups)
    const int su = SRC_ROW == 128 ? (u ^ (row & 7)) : (u ^ ((row >> 1) & 3));
    const uint4 v = lds128(src + sc * KEYS * SRC_ROW + row * SRC_ROW + su * 16);
    const int e0 = sc * 128 + u * 16;                  // first element (d index)
    const int tc = e0 / 64;                            // target chunk
    const int tu = (e0 % 64) / 8;                      // first target unit (of 8 elements)
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint4 lo, hi;
    lo.x = e4m3x2_to_f16x2(w[0] & 0xFFFFu);
    lo.y = e4m3x2_to_f16x2(w[0] >> 16);
    lo.z = e4m3x2_to_f16x2(w[1] & 0xFFFFu);
    lo.w = e4m3x2_to_f16x2(w[1] >> 16);
    hi.x = e4m3x2_to_f16x2(w[2] & 0xFFFFu);
    hi.y = e4m3x2_to_f16x2(w[2] >> 16);
    hi.z = e4m3x2_to_f16x2(w[3] & 0xFFFFu);
    hi.w = e4m3x2_to_f16x2(w[3] >> 16);
    const uint32_t base = dst + tc * KEYS * 128 + row * 128;
    sts128(base + ((tu ^ (row & 7)) * 16), lo);
    sts128(base + (((tu + 1) ^ (row & 7)) * 16), hi);
  }
}

}  // namespace attnb3
