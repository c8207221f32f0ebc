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

// Normalised Walsh-Hadamard transform of a head_dim row held by LANES
// consecutive lanes of a warp (32, or 16 for a row per half-warp), E =
// head_dim / LANES consecutive elements per lane (element (lane % LANES)*E
// + i).  Butterfly stages h = 1, 2, 4, ... in that order; each stage maps
// the pair (x[j], x[j+h]) (bit h of j clear) to (x[j] + x[j+h], x[j] -
// x[j+h]).  Stages h < E stay in registers, the others pair lane with lane ^
// (h/E).  Finally every element is multiplied once by inv_sqrt_n.  The
// arithmetic per element is identical whatever lane layout runs it.
template <int E, int LANES = 32>
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
  for (int m = 1; m < LANES; m <<= 1) {
    // lower lane holds a = x[j], partner b: a + b; upper lane holds b,
    // partner a: a - b = fma(b, -1, a) (the same single rounding)
    const float sg = (lane & m) ? -1.f : 1.f;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const float other = __shfl_xor_sync(0xffffffffu, x[j], m);
      x[j] = fmaf(x[j], sg, other);
    }
  }
#pragma unroll
  for (int j = 0; j < E; ++j) x[j] *= inv_sqrt_n;
}

// ---------------------------------------------------- codebook search

// 2-bit codes: three thresholds, searched directly (cheaper than a table
// lookup): code = #{i : t[i] <= v}.
__device__ __forceinline__ int lm_code2(float v, const float* t) {
  const bool b1 = v >= t[1];
  const bool b0 = v >= (b1 ? t[2] : t[0]);
  return (b1 << 1) | (int)b0;
}

// x / s rounded to nearest (IEEE), from r = 1/s rounded to nearest: one
// product and one FMA correction (Markstein's correctly rounded quotient;
// s > 0 is an E4M3 value and x / s is normal wherever the rounding can
// decide a code).
__device__ __forceinline__ float div_by_scale(float x, float s, float r) {
  const float q = x * r;
  return fmaf(fmaf(-q, s, x), r, q);
}

}  // namespace kvq
