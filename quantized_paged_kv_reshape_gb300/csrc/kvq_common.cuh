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

// Codebook-search buckets: bucket k of a magnitude m >= 0 with fp32 bits mb
// is clamp(mb >> 20, kBucketLo, kBucketLo + kBuckets - 1) - kBucketLo, i.e.
// the exponent and top 3 mantissa bits; bucket 0 holds [0, 0.140625), the
// last one [4, inf).  Every bucket is narrower than the spacing of the
// positive Lloyd-Max thresholds (>= 0.258), so it holds at most one.
constexpr int kBucketLo = 992;  // bits(0.125f) >> 20
constexpr int kBuckets = 41;    // up to bits(4.0f) >> 20 = 1032

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
  // Bucket tables of the codebook search (see lm_code_bucket), for 4, 3
  // and 2 bits: per bucket (number of positive thresholds below the
  // bucket, bit pattern of the bucket's one positive threshold or
  // 0x7fffffff for none).
  uint32_t bucket[3][kBuckets][2];
};

// E2M1 code of v: round to nearest, ties to the even code, saturating at 6,
// sign bit 3 given by the caller.  The magnitude code counts the midpoints
// below |v|; a midpoint itself goes up only where the code above is even.
// neg: the sign bit to store (that of the unrounded quotient).
__device__ __forceinline__ uint32_t e2m1_from_float(float v, bool neg) {
  const float m = fabsf(v);
  const uint32_t c = (uint32_t)(m > 0.25f) + (uint32_t)(m >= 0.75f) + (uint32_t)(m > 1.25f) +
                     (uint32_t)(m >= 1.75f) + (uint32_t)(m > 2.5f) + (uint32_t)(m >= 3.5f) +
                     (uint32_t)(m > 5.0f);
  return c | (neg ? 8u : 0u);
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

// code = number of thresholds <= v for a symmetric 2^B-level codebook (the
// middle threshold is 0, the others come in pairs +-t), from the bucket
// table of the positive thresholds:
//   v >= 0 (and -0): code = 2^(B-1)     + #{t > 0 : t <= v}
//   v <  0         : code = 2^(B-1) - 1 - #{t > 0 : t <  |v|}
// The count is the bucket's base count plus one compare of |v| with the
// bucket's threshold (on the bit patterns, which order like the values for
// non-negative floats; "<" becomes ">=" against the next pattern).
template <int B>
__device__ __forceinline__ int lm_code_bucket(float v, const uint2* table) {
  const uint32_t vb = __float_as_uint(v + 0.0f);  // -0 becomes +0
  const uint32_t neg = vb >> 31;
  const uint32_t mb = vb & 0x7fffffffu;
  const uint32_t k = min(max(mb >> 20, (uint32_t)kBucketLo), (uint32_t)(kBucketLo + kBuckets - 1)) -
                     (uint32_t)kBucketLo;
  const uint2 e = table[k];
  const int c = (int)e.x + (mb >= e.y + neg ? 1 : 0);
  return neg ? (1 << (B - 1)) - 1 - c : (1 << (B - 1)) + c;
}

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
