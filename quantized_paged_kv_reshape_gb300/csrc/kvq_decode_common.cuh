// Helpers shared by the decode kernels: staged-row geometry of a side,
// cp.async wrappers and the codebook of a side.
#pragma once

#include "kvq_common.cuh"
#include "kvq_launch.h"

namespace kvq {

template <int S, int HD>
struct SideGeom {
  static constexpr int ROW = HD * side_bits(S) / 8;                    // data bytes per row
  static constexpr int SROW = (HD / kGroup) * side_scale_bytes(S);     // scale bytes per row
  static constexpr int CH = (ROW % 16 == 0) ? 16 : (ROW % 8 == 0) ? 8 : 4;  // copy chunk
  static constexpr int SCH = SROW == 0 ? 0 : (SROW >= 16 ? 16 : SROW);
  static constexpr int NCH = ROW / CH;
  static constexpr int NSCH = SCH ? SROW / SCH : 0;
};

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }
// A row of `bytes` in `chunk`-byte pieces (none when bytes is 0): do its
// pieces divide a warp's 32 lanes evenly?
constexpr bool chunks_split_warp(int bytes, int chunk) {
  if (bytes == 0) return true;
  const int n = bytes / chunk;
  return n > 0 && 32 % n == 0;
}

// Virtual slabs that stand for the cost of one unit (a merge, then the first
// copies' round trip) in the decode kernels' work partition.
constexpr int kUnitSlabs = 48;
constexpr int clampi(int x, int lo, int hi) { return x < lo ? lo : x > hi ? hi : x; }

template <int N>
__device__ __forceinline__ void cp_async(void* dst, const void* src, bool valid) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
  const int n = valid ? N : 0;
  if constexpr (N == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(src), "r"(n));
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;\n" ::"r"(s), "l"(src), "n"(N),
                 "r"(n));
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <int S>
__device__ __forceinline__ const float* side_levels(const Codebooks& cb) {
  return S == S_T4 ? cb.lv4 : S == S_T3 ? cb.lv3 : S == S_NVFP4 ? cb.e2m1 : cb.lv2;
}

}  // namespace kvq
