// Split merge and output rotation of the paged decode.
//
// For one (sequence, query head) the split CTAs left partial results
// (m_i, l_i, acc_i) in the exp2 domain.  The merge is the online-softmax
// identity: m = max m_i, l = sum l_i 2^(m_i - m), o = sum acc_i 2^(m_i - m) / l.
// When the V side is stored in the Walsh-Hadamard basis the merged row is
// rotated back once ("spark_runtime/kv_cache.rs", is_wht_rotated: the iWHT(out)
// bookend; the normalised transform is its own inverse).  One warp per row.
#include <math_constants.h>

#include "kvq_common.cuh"
#include "kvq_launch.h"

namespace kvq {

namespace {

template <int HD>
__global__ void __launch_bounds__(128) combine_kernel(const CombineArgs a) {
  constexpr int E = HD / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= (int64_t)a.num_seqs * a.nq) return;
  const float* pp = a.part + row * a.nsplit * (HD + 4);
  float m = -CUDART_INF_F;
  for (int i = 0; i < a.nsplit; ++i) m = fmaxf(m, pp[i * (HD + 4)]);
  float x[E];
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = 0.f;
  float l = 0.f;
  if (m != -CUDART_INF_F) {
    for (int i = 0; i < a.nsplit; ++i) {
      const float* pi = pp + i * (HD + 4);
      const float w = exp2f(pi[0] - m);
      l = fmaf(pi[1], w, l);
#pragma unroll
      for (int e = 0; e < E; ++e) x[e] = fmaf(pi[4 + lane * E + e], w, x[e]);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] *= inv;
  if (a.v_rotated) fwht_warp<E>(x, lane, a.inv_sqrt_hd);
  const int64_t o = row * HD + lane * E;
  if (a.out_bf16) {
    uint16_t* out = reinterpret_cast<uint16_t*>(a.out);
#pragma unroll
    for (int e = 0; e < E; ++e) out[o + e] = bf16_bits_from_float(x[e]);
  } else {
    float* out = reinterpret_cast<float*>(a.out);
#pragma unroll
    for (int e = 0; e < E; ++e) out[o + e] = x[e];
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int head_dim, cudaStream_t st) {
  const int64_t rows = (int64_t)a.num_seqs * a.nq;
  if (rows == 0) return cudaSuccess;
  const int grid = (int)((rows + 3) / 4);
  switch (head_dim) {
    case 64: combine_kernel<64><<<grid, 128, 0, st>>>(a); break;
    case 128: combine_kernel<128><<<grid, 128, 0, st>>>(a); break;
    case 256: combine_kernel<256><<<grid, 128, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace kvq
