// Shared device/host definitions of the quantized paged KV cache kernels.
//
// Side formats and their per-block byte arithmetic follow "spark_runtime/
// kv_cache.rs" (enum KvCacheDtype, KvCacheConfig::block_bytes_dims and the
// turbo*_data_bytes / turbo*_scale_bytes helpers); the block layout
// [num_blocks, block_size, num_kv_heads, head_dim] with a code section
// followed by a scale section follows the module invariants of
// "metrale_model_layers/layers/ops/kv_cache_bf16k_turbov.rs".
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace kvq {

// Side formats use the numbering of the symmetric kvq_format values.
enum Side : int { S_BF16 = 0, S_FP8 = 1, S_NVFP4 = 2, S_T4 = 3, S_T3 = 4, S_T2 = 5, S_T8 = 6 };

constexpr int kGroup = 16;  // one scale per 16 consecutive elements

// Stored bits per element in the code / raw-data section.
__host__ __device__ constexpr int side_bits(int s) {
  return s == S_BF16 ? 16 : s == S_FP8 ? 8 : s == S_T4 ? 4 : s == S_T3 ? 3
       : s == S_T2 ? 2 : s == S_T8 ? 8 : s == S_NVFP4 ? 4 : 0;
}
// Bytes of one group scale (0 = no scale section).
__host__ __device__ constexpr int side_scale_bytes(int s) {
  return (s == S_T4 || s == S_T3 || s == S_T2 || s == S_NVFP4) ? 1 : s == S_T8 ? 2 : 0;
}
__host__ __device__ constexpr bool side_rotated(int s) {
  return s == S_T4 || s == S_T3 || s == S_T2 || s == S_T8;
}
// Sides whose elements are codes into a level table (Turbo2/3/4: Lloyd-Max
// levels; NVFP4: the 16 E2M1 values) times a per-16 E4M3 scale.
__host__ __device__ constexpr bool side_codebook(int s) {
  return s == S_T4 || s == S_T3 || s == S_T2 || s == S_NVFP4;
}
__host__ __device__ constexpr int code_bits(int s) {
  return s == S_T4 || s == S_NVFP4 ? 4 : s == S_T3 ? 3 : s == S_T2 ? 2 : 0;
}

// Lloyd-Max N(0,1) codebooks (fp32 levels ascending, fp32 midpoint
// thresholds) for 4, 3 and 2 bits, and the E2M1 values of the 16 NVFP4 codes
// (code c: sign bit 3, magnitude 0 0.5 1 1.5 2 3 4 6 for c & 7), passed to
// kernels by value.
struct Codebooks {
  float lv4[16], th4[15];
  float lv3[8], th3[7];
  float lv2[4], th2[3];
  float e2m1[16];
};

// E2M1 code of v: round to nearest, ties to the even code, saturating at 6,
// sign bit 3 from the sign bit of v.  The magnitude code counts the midpoints
// below |v|; a midpoint itself goes up only where the code above is even.
__device__ __forceinline__ uint32_t e2m1_from_float(float v) {
  const float m = fabsf(v);
  const uint32_t c = (uint32_t)(m > 0.25f) + (uint32_t)(m >= 0.75f) + (uint32_t)(m > 1.25f) +
                     (uint32_t)(m >= 1.75f) + (uint32_t)(m > 2.5f) + (uint32_t)(m >= 3.5f) +
                     (uint32_t)(m > 5.0f);
  return c | (signbit(v) ? 8u : 0u);
}

// ------------------------------------------------------- number formats

// E4M3 encode: round to nearest even, saturate to +-448 (hardware cvt).
__device__ __forceinline__ uint8_t e4m3_from_float(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float e4m3_to_float(uint8_t b) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
  return __half2float(__half(h));
}
// Two E4M3 bytes (low byte = first) -> two floats.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t b2) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)b2, __NV_E4M3);
  return __half22float2(__half2(h));
}
__device__ __forceinline__ uint16_t bf16_bits_from_float(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// --------------------------------------------------------- rotation

// Normalised Walsh-Hadamard transform of a head_dim row held by one warp,
// E = head_dim / 32 consecutive elements per lane (element lane*E + i).
// Butterfly stages h = 1, 2, 4, ... in that order; each stage maps the pair
// (x[j], x[j+h]) (bit h of j clear) to (x[j] + x[j+h], x[j] - x[j+h]).
// Stages h < E stay in registers, the others pair lane with lane ^ (h/E).
// Finally every element is multiplied once by inv_sqrt_n.  The arithmetic
// per element is identical whatever lane layout runs it.
template <int E>
__device__ __forceinline__ void fwht_warp(float (&x)[E], int lane, float inv_sqrt_n) {
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int j = 0; j < E; ++j) {
      if ((j & h) == 0) {
        float a = x[j], b = x[j + h];
        x[j] = a + b;
        x[j + h] = a - b;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      float other = __shfl_xor_sync(0xffffffffu, x[j], m);
      // lower lane holds a = x[j], partner b; upper lane holds b, partner a
      x[j] = upper ? (other - x[j]) : (x[j] + other);
    }
  }
#pragma unroll
  for (int j = 0; j < E; ++j) x[j] *= inv_sqrt_n;
}

// ---------------------------------------------------- codebook search

// code = number of thresholds <= v (sorted ascending), as a binary search
// whose thresholds are picked by select trees on the bits decided so far.
__device__ __forceinline__ int lm_code4(float v, const float* t) {
  const bool b3 = v >= t[7];
  const bool b2 = v >= (b3 ? t[11] : t[3]);
  const float tb = b3 ? (b2 ? t[13] : t[9]) : (b2 ? t[5] : t[1]);
  const bool b1 = v >= tb;
  const float tc = b3 ? (b2 ? (b1 ? t[14] : t[12]) : (b1 ? t[10] : t[8]))
                      : (b2 ? (b1 ? t[6] : t[4]) : (b1 ? t[2] : t[0]));
  const bool b0 = v >= tc;
  return (b3 << 3) | (b2 << 2) | (b1 << 1) | (int)b0;
}
__device__ __forceinline__ int lm_code3(float v, const float* t) {
  const bool b2 = v >= t[3];
  const bool b1 = v >= (b2 ? t[5] : t[1]);
  const float tc = b2 ? (b1 ? t[6] : t[4]) : (b1 ? t[2] : t[0]);
  const bool b0 = v >= tc;
  return (b2 << 2) | (b1 << 1) | (int)b0;
}
__device__ __forceinline__ int lm_code2(float v, const float* t) {
  const bool b1 = v >= t[1];
  const bool b0 = v >= (b1 ? t[2] : t[0]);
  return (b1 << 1) | (int)b0;
}

}  // namespace kvq
