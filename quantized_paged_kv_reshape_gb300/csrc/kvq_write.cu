// Cache-write kernel: scatter K/V rows into the paged cache, each side in its
// own storage format, both sides in one launch.
//
// "metrale_model_layers/layers/ops/kv_cache_bf16k_turbov.rs",
// reshape_and_cache_bf16k_turbo{2,3,4}v (arguments: key/value with per-token
// element strides, slot_mapping, k/v block strides in bytes, the V data
// section size); "spark_runtime/kv_cache.rs", KvCacheDtype::Turbo4KTurbo3V
// (one launch forks the K-side and V-side writers) and the Turbo2/3/4/8, Fp8
// and Bf16 storage descriptions.
//
// Work mapping: every lane holds one 16-element scale group of a row
// (head_dim / 16 lanes per row: 4, 8 or 16), so a warp holds 8, 4 or 2 rows
// at once and a group's maximum, scale and code bytes are one lane's own
// work.  The rows of a warp are consecutive (token, kv head) pairs of one
// side, heads fastest, so the input reads and the cache stores of a warp are
// contiguous runs.  The rotation's first four butterfly stages run inside a
// lane's registers, the rest as lane-pair shuffles.
//
// Codebook search, Turbo4/3: the code of a quotient v is  c_lo + (v >= t)
// within each of 256 buckets of width 1/4 in v (every bucket holds at most
// one threshold t, and none lies near a bucket edge); the bucket's byte offset
// in a 2 KB shared-memory table is read off the fp32 bits of one FMA.  NVFP4:
// the code is a step function of v's fp32 bit pattern with at most one step
// among the patterns that share their top 12 bits, read from a 4096-entry
// table.  Both tables are built by each CTA from the codebook.
#include "kvq_common.cuh"
#include "kvq_launch.h"

namespace kvq {

namespace {

constexpr int kKeys = 4096;        // code-table keys: fp32 bits >> 20
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
#ifndef KVQ_WRITE_UNITS
#define KVQ_WRITE_UNITS 2
#endif
constexpr int kUnitsPerWarp = KVQ_WRITE_UNITS;   // units a warp encodes per iteration
#ifndef KVQ_WRITE_CTAS_PER_SM
#define KVQ_WRITE_CTAS_PER_SM 3
#endif
constexpr int kCtasPerSm = KVQ_WRITE_CTAS_PER_SM;

template <int HD>
struct WGeom {
  static constexpr int LANES = HD / kGroup;   // lanes per row
  static constexpr int ROWS = 32 / LANES;     // rows per warp
};

// Bucket tables of the Turbo4/3 search: entry k covers the quotients whose
// fmaf(v, 4, 2^20 + 128.5), rounded to eighths, lies in [2^20 + k, 2^20 + k +
// 1): v in [(k - 128.5) / 4, (k - 127.5) / 4) up to 1/64 at the edges.  The
// fp32 bits of that FMA masked with 0x7f8 are the entry's byte offset (8 B:
// the bucket's threshold, or +inf, and its codes).  Valid for |v| < 31.9;
// the Lloyd-Max thresholds keep more than 0.025 from every edge (checked on
// the host), so the fuzz never moves a code.
constexpr int kLin = 256;
constexpr float kLinMagic = 1048704.5f;   // 2^20 + 128.5

// Sides whose codes come from the 4096-entry key table (NVFP4).
__host__ __device__ __forceinline__ bool side_has_table(int s) { return s == S_NVFP4; }

// Linear-table entry k of Turbo side s: (threshold in the bucket or +inf,
// lo = the number of thresholds below the bucket, as bits).
__device__ float2 lin_entry(int s, int k, const Codebooks& cb) {
  const float* th = s == S_T4 ? cb.th4 : cb.th3;
  const int n = s == S_T4 ? 15 : 7;
  const float lo_v = ((float)k - 128.5f) * 0.25f, hi_v = lo_v + 0.25f;
  uint32_t c = 0;
  float t = __int_as_float(0x7f800000);   // +inf: no threshold in the bucket
  for (int i = 0; i < n; ++i) {
    if (th[i] < lo_v) ++c;
    else if (th[i] < hi_v) t = th[i];
  }
  return make_float2(t, __uint_as_float(c));
}

// NVFP4 key-table entry of key k: every quotient v whose fp32 bits b
// satisfy b >> 20 == k has code  b >= e.x ? hi : lo.  e.y holds the bytes
// (lo, hi, lo << 4, hi << 4), the last two for codes that land in a byte's
// upper nibble.  E2M1 rounds to nearest, ties to the even code, saturating at
// 6: the magnitude code counts the rounding points at or below |v| (a tie
// rounds up where the upper code is even), the sign bit is v's.
__device__ uint2 nvfp4_entry(uint32_t k) {
  const uint32_t neg = k >> 11, mk = k & 0x7ffu;
  // first bit patterns above 0.25, at 0.75, above 1.25, at 1.75, above 2.5,
  // at 3.5, above 5 (ties at 0.25, 1.25, 2.5, 5 stay on the even code)
  constexpr uint32_t kStep[7] = {0x3e800001u, 0x3f400000u, 0x3fa00001u, 0x3fe00000u,
                                 0x40200001u, 0x40600000u, 0x40a00001u};
  const uint32_t b0 = mk << 20, b1 = b0 | 0xfffffu;
  uint32_t c = 0, st = 0xffffffffu;
#pragma unroll
  for (int i = 0; i < 7; ++i) {
    if (kStep[i] <= b0) ++c;
    else if (kStep[i] <= b1) st = kStep[i];
  }
  const uint32_t lo = c | (neg << 3);
  const uint32_t hi = (st != 0xffffffffu ? c + 1 : c) | (neg << 3);
  const uint32_t t = st == 0xffffffffu ? 0xffffffffu : (st | (neg << 31));
  return make_uint2(t, lo | (hi << 8) | (lo << 20) | (hi << 28));
}

// Code byte of quotient bits vb from the key table, placed in byte POS of the
// result (zeros elsewhere); UP = take the nibble-shifted copy.
template <int POS, bool UP>
__device__ __forceinline__ uint32_t pick_code(const uint2* tab, uint32_t vb) {
  const uint2 e = tab[vb >> 20];
  constexpr uint32_t src = UP ? 2u : 0u;
  constexpr uint32_t blank = 0x4444u & ~(0xfu << (4 * POS));
  constexpr uint32_t sel_lo = blank | (src << (4 * POS));
  constexpr uint32_t sel_hi = blank | ((src + 1) << (4 * POS));
  return __byte_perm(e.y, 0u, vb >= e.x ? sel_hi : sel_lo);
}

// n / nkv (n < 2^31) with the host's multiplier and shifts.
__device__ __forceinline__ uint32_t div_nkv(uint32_t n, const WriteArgs& a) {
  const uint32_t h = __umulhi(n, a.nkv_m);
  return (h + ((n - h) >> a.nkv_s1)) >> a.nkv_s2;
}

// One lane's 16 input elements, as loaded: bf16 pairs or fp32.
template <typename InT>
struct Raw;
template <>
struct Raw<__nv_bfloat16> {
  uint32_t w[8];
  __device__ __forceinline__ float at(int i) const {
    return __uint_as_float((i & 1) ? (w[i / 2] & 0xffff0000u) : (w[i / 2] << 16));
  }
};
template <>
struct Raw<float> {
  float f[16];
  __device__ __forceinline__ float at(int i) const { return f[i]; }
};

template <typename InT, bool VEC>
__device__ __forceinline__ void load_raw(const InT* src, Raw<InT>& r) {
  if constexpr (sizeof(InT) == 2) {
    if constexpr (VEC) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(src) + 1);
      r.w[0] = a.x; r.w[1] = a.y; r.w[2] = a.z; r.w[3] = a.w;
      r.w[4] = b.x; r.w[5] = b.y; r.w[6] = b.z; r.w[7] = b.w;
    } else {
      const unsigned short* p = reinterpret_cast<const unsigned short*>(src);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        r.w[i] = (uint32_t)__ldg(p + 2 * i) | ((uint32_t)__ldg(p + 2 * i + 1) << 16);
    }
  } else {
    if constexpr (VEC) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src) + i);
        r.f[4 * i] = v.x; r.f[4 * i + 1] = v.y; r.f[4 * i + 2] = v.z; r.f[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) r.f[i] = __ldg(src + i);
    }
  }
}

__device__ __forceinline__ void st8(uint8_t* p, uint32_t v) { *p = (uint8_t)v; }
__device__ __forceinline__ void st16(uint8_t* p, uint32_t v) {
  *reinterpret_cast<uint16_t*>(p) = (uint16_t)v;
}
__device__ __forceinline__ void st32(uint8_t* p, uint32_t v) { *reinterpret_cast<uint32_t*>(p) = v; }
__device__ __forceinline__ void st64(uint8_t* p, uint32_t a, uint32_t b) {
  *reinterpret_cast<uint2*>(p) = make_uint2(a, b);
}
__device__ __forceinline__ void st128(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}

// Packed fp32 pairs (sm_100+ add/sub/mul/fma .rn.f32x2): each half rounds
// exactly like the scalar instruction, two elements per issue.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2_split(uint64_t d, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(d));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Normalised Walsh-Hadamard transform of a row held by LANES lanes, 16
// consecutive elements per lane, kept as pairs p[k] = (x[k], x[k + 8]).
// Butterfly stages h = 1, 2, 4, 8, 16, ... in that order, each mapping
// (x[j], x[j + h]) to (x[j] + x[j + h], x[j] - x[j + h]): h = 1, 2, 4 pair
// p[k] with p[k + h] (both halves at once), h = 8 works inside each pair,
// the lane stages pair lane with lane ^ (h / 16).  Then every element is
// multiplied by inv_sqrt_n: the roundings of the scalar transform.
template <int LANES>
__device__ __forceinline__ void fwht16_pairs(uint64_t (&p)[8], int rl, float inv_sqrt_n) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if ((k & h) == 0) {
        const uint64_t a = p[k], b = p[k + h];
        p[k] = f2_add(a, b);
        p[k + h] = f2_sub(a, b);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float a, b;
    f2_split(p[k], a, b);
    p[k] = f2(a + b, a - b);
  }
#pragma unroll
  for (int m = 1; m < LANES; m <<= 1) {
    // lower lane holds a, partner b: a + b; upper lane holds b, partner a:
    // a - b = fma(b, -1, a) (the same single rounding)
    const float sg = (rl & m) ? -1.f : 1.f;
    const uint64_t sg2 = f2(sg, sg);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float a, b;
      f2_split(p[k], a, b);
      const float oa = __shfl_xor_sync(0xffffffffu, a, m);
      const float ob = __shfl_xor_sync(0xffffffffu, b, m);
      p[k] = f2_fma(p[k], sg2, f2(oa, ob));
    }
  }
  const uint64_t c2 = f2(inv_sqrt_n, inv_sqrt_n);
#pragma unroll
  for (int k = 0; k < 8; ++k) p[k] = f2_mul(p[k], c2);
}

__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {   // a in the low byte
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Group scale of a lane's 16 values: E4M3(amax / top) (fp32 divide), and
// its value and reciprocal (1/s, 0 for s = 0) from the CTA's table of all
// 256 E4M3 bytes.
__device__ __forceinline__ uint32_t group_scale(const float (&y)[16], float top, uint32_t sr_addr,
                                                float& s, float& r) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(y[i]));
  const uint32_t sbyte = e4m3_from_float(amax / top);
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(s), "=f"(r) : "r"(sr_addr + sbyte * 8));
  return sbyte;
}

// NVFP4: 16 four-bit codes (code i at bits 4i) and the scale byte.  The sign
// bit is x's (also for x = -0, whose quotient loses it); a zero scale gives
// code 0.
__device__ __forceinline__ void encode_nvfp4(const float (&y)[16], const uint2* tab, uint32_t sr,
                                             uint8_t* codes, uint8_t* scale, bool ok) {
  float s, r;
  const uint32_t sbyte = group_scale(y, 6.0f, sr, s, r);
  const uint32_t smask = s != 0.f ? 0x80000000u : 0u;
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t vb = (__float_as_uint(div_by_scale(y[i], s, r)) & 0x7fffffffu) |
                        (__float_as_uint(y[i]) & smask);
    uint32_t c;
    switch (i & 7) {   // byte (i / 2) % 4 of word i / 8, upper nibble for odd i
      case 0: c = pick_code<0, false>(tab, vb); break;
      case 1: c = pick_code<0, true>(tab, vb); break;
      case 2: c = pick_code<1, false>(tab, vb); break;
      case 3: c = pick_code<1, true>(tab, vb); break;
      case 4: c = pick_code<2, false>(tab, vb); break;
      case 5: c = pick_code<2, true>(tab, vb); break;
      case 6: c = pick_code<3, false>(tab, vb); break;
      default: c = pick_code<3, true>(tab, vb); break;
    }
    w[i / 8] |= c;
  }
  if (ok) {
    st64(codes, w[0], w[1]);
    st8(scale, sbyte);
  }
}

// Group scale of a lane's 16 values held as pairs.
__device__ __forceinline__ uint32_t group_scale_pairs(const uint64_t (&p)[8], float top,
                                                      uint32_t sr_addr, float& s, float& r) {
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float a, b;
    f2_split(p[k], a, b);
    amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(b)));
  }
  const uint32_t sbyte = e4m3_from_float(amax / top);
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(s), "=f"(r) : "r"(sr_addr + sbyte * 8));
  return sbyte;
}

// Quotients v = y / s (Markstein's correction of y * (1/s), two elements per
// instruction) and their bucket offsets; CLAMP bounds v to +-31 first
// (groups whose scale saturated at E4M3's 448 have quotients beyond the
// bucket table; elsewhere |v| <= 1.5 x the top level).
template <bool CLAMP>
__device__ __forceinline__ void quot_pairs(const uint64_t (&p)[8], float s, float r,
                                           float (&v)[16], uint32_t (&off)[16]) {
  const uint64_t r2 = f2(r, r), ns2 = f2(-s, -s);
  const uint64_t four = f2(4.0f, 4.0f), magic = f2(kLinMagic, kLinMagic);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint64_t q0 = f2_mul(p[k], r2);
    const uint64_t rem = f2_fma(q0, ns2, p[k]);
    uint64_t q = f2_fma(rem, r2, q0);
    if constexpr (CLAMP) {
      float a, b;
      f2_split(q, a, b);
      q = f2(fminf(fmaxf(a, -31.f), 31.f), fminf(fmaxf(b, -31.f), 31.f));
    }
    float fa, fb;
    f2_split(f2_fma(q, four, magic), fa, fb);
    f2_split(q, v[k], v[k + 8]);
    off[k] = __float_as_uint(fa) & 0x7f8u;
    off[k + 8] = __float_as_uint(fb) & 0x7f8u;
  }
}

// acc * 2^B + code(v): the bucket's lo plus one where v >= its threshold
// (set.ge gives all ones there).  Codes are appended last element first, so
// element 0 ends in the lowest bits.
template <int B>
__device__ __forceinline__ uint32_t lin_step(uint32_t acc, uint32_t lin_addr, uint32_t off,
                                             float v) {
  float t;
  uint32_t lo, ge;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=f"(t), "=r"(lo) : "r"(lin_addr + off));
  asm("set.ge.u32.f32 %0, %1, %2;" : "=r"(ge) : "f"(v), "f"(t));
  return (acc << B) + lo - ge;
}

// Turbo4: 16 four-bit codes (code i at bits 4i) and the scale byte.  A zero
// scale makes every quotient +-0, which takes the middle code.
__device__ __forceinline__ void encode4(const uint64_t (&p)[8], float top, uint32_t lin,
                                        uint32_t sr, uint8_t* codes, uint8_t* scale, bool ok) {
  float s, r;
  const uint32_t sbyte = group_scale_pairs(p, top, sr, s, r);
  float v[16];
  uint32_t off[16];
  if (__any_sync(0xffffffffu, s >= 448.f)) quot_pairs<true>(p, s, r, v, off);
  else quot_pairs<false>(p, s, r, v, off);
  uint32_t w[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t acc = 0u;
#pragma unroll
    for (int j = 7; j >= 0; --j) acc = lin_step<4>(acc, lin, off[8 * h + j], v[8 * h + j]);
    w[h] = acc;
  }
  if (ok) {
    st64(codes, w[0], w[1]);
    st8(scale, sbyte);
  }
}

// Turbo3: 16 three-bit codes (48 bits, code i at bits 3i) and the scale:
// elements 0-9 fill bits 0-29, 11-15 bits 33-47, element 10 straddles bits
// 30-32.  The lane's 6 bytes start 2-byte aligned: 4 + 2 or 2 + 4 bytes.
__device__ __forceinline__ void encode3(const uint64_t (&p)[8], float top, uint32_t lin,
                                        uint32_t sr, uint8_t* codes, uint8_t* scale, int rl,
                                        bool ok) {
  float s, r;
  const uint32_t sbyte = group_scale_pairs(p, top, sr, s, r);
  float v[16];
  uint32_t off[16];
  if (__any_sync(0xffffffffu, s >= 448.f)) quot_pairs<true>(p, s, r, v, off);
  else quot_pairs<false>(p, s, r, v, off);
  uint32_t a = 0u, b = 0u;
#pragma unroll
  for (int j = 9; j >= 0; --j) a = lin_step<3>(a, lin, off[j], v[j]);
#pragma unroll
  for (int j = 15; j >= 11; --j) b = lin_step<3>(b, lin, off[j], v[j]);
  const uint32_t c10 = lin_step<3>(0u, lin, off[10], v[10]);
  const uint32_t lo = a | (c10 << 30), hi = (c10 >> 2) | (b << 1);
  if (ok) {
    if (rl & 1) {
      st16(codes, lo);
      st32(codes + 2, __funnelshift_r(lo, hi, 16));
    } else {
      st32(codes, lo);
      st16(codes + 4, hi);
    }
    st8(scale, sbyte);
  }
}

// Turbo2: 16 two-bit codes from the three thresholds, one 32-bit word; the
// quotients two elements per instruction.
__device__ __forceinline__ void encode2(const uint64_t (&p)[8], const Codebooks& cb, uint32_t sr,
                                        uint8_t* codes, uint8_t* scale, bool ok) {
  float s, r;
  const uint32_t sbyte = group_scale_pairs(p, cb.lv2[3], sr, s, r);
  float th[3];
#pragma unroll
  for (int i = 0; i < 3; ++i) th[i] = cb.th2[i];
  const uint64_t r2 = f2(r, r), ns2 = f2(-s, -s);
  float v[16];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint64_t q0 = f2_mul(p[k], r2);
    const uint64_t rem = f2_fma(q0, ns2, p[k]);
    f2_split(f2_fma(rem, r2, q0), v[k], v[k + 8]);
  }
  uint32_t w = 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) w |= (uint32_t)lm_code2(v[i], th) << (2 * i);
  if (ok) {
    st32(codes, w);
    st8(scale, sbyte);
  }
}

// Turbo8: bf16 scale amax / 448 (fp32 divide, then rounded), codes
// E4M3(y / s) (fp32 divides), a zero scale stores code 0.
__device__ __forceinline__ void encode8(const float (&y)[16], uint8_t* codes, uint8_t* scale,
                                        bool ok) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(y[i]));
  const uint32_t sbits = bf16_bits_from_float(amax / 448.0f);
  const float s = bf16_bits_to_float(sbits);
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const uint32_t p = e4m3x2(y[i] / s, y[i + 1] / s);
    const uint32_t b = s == 0.f ? 0u : p;
    if (i % 4 == 0) w[i / 4] = b;
    else w[i / 4] |= b << 16;
  }
  if (ok) {
    st128(codes, w[0], w[1], w[2], w[3]);
    st16(scale, sbits);
  }
}

// Encode and store one unit: this lane's 16 elements of its row.  Every lane
// of the warp runs it (the rotation's shuffles need them all); ok = false (no
// valid slot) computes but stores nothing.
template <int HD, typename InT>
__device__ __forceinline__ void write_group(const WriteArgs& a, const Codebooks& cb,
                                            const uint2* tab, uint32_t lin, uint32_t sr, int side,
                                            int64_t slot, int h, const Raw<InT>& raw, int rl,
                                            bool ok) {
  if (!ok) slot = 0;
  int64_t blk;
  uint32_t off;
  if (a.bs_shift >= 0) {          // power-of-two block size
    blk = slot >> a.bs_shift;
    off = (uint32_t)slot & (uint32_t)(a.bs - 1);
  } else if (slot < 0xffffffffll) {   // 32-bit division
    const uint32_t s32 = (uint32_t)slot;
    const uint32_t b32 = s32 / (uint32_t)a.bs;
    blk = b32;
    off = s32 - b32 * (uint32_t)a.bs;
  } else {
    blk = slot / a.bs;
    off = (uint32_t)(slot - blk * a.bs);
  }
  const int fmt = side ? a.v_side : a.k_side;
  uint8_t* base = (side ? a.v_cache : a.k_cache) + blk * (side ? a.v_bstride : a.k_bstride);
  uint8_t* ssec = base + (side ? a.v_dsec : a.k_dsec);
  // this lane's group inside the block (a block holds fewer than 2^31 bytes)
  const uint32_t g = (off * (uint32_t)a.nkv + (uint32_t)h) * (HD / kGroup) + (uint32_t)rl;
  if (fmt == S_BF16) {
    uint32_t w[8];
    if constexpr (sizeof(InT) == 2) {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = raw.w[i];   // bf16 in, bf16 out: the input bits
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = (uint32_t)bf16_bits_from_float(raw.at(2 * i)) |
               ((uint32_t)bf16_bits_from_float(raw.at(2 * i + 1)) << 16);
    }
    if (ok) {
      uint8_t* dst = base + (size_t)g * 32;
      st128(dst, w[0], w[1], w[2], w[3]);
      st128(dst + 16, w[4], w[5], w[6], w[7]);
    }
  } else if (fmt == S_FP8) {
    // x / scale (fp32 divide; a product with the exact reciprocal where the
    // scale is a power of two)
    const float sc = side ? a.v_scale : a.k_scale, inv = side ? a.v_inv : a.k_inv;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const float x0 = raw.at(i), x1 = raw.at(i + 1);
      const uint32_t p = inv != 0.f ? e4m3x2(x0 * inv, x1 * inv) : e4m3x2(x0 / sc, x1 / sc);
      if (i % 4 == 0) w[i / 4] = p;
      else w[i / 4] |= p << 16;
    }
    if (ok) st128(base + g * 16, w[0], w[1], w[2], w[3]);
  } else {
    if (fmt == S_NVFP4) {
      float y[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = raw.at(i);
      encode_nvfp4(y, tab, sr, base + g * 8, ssec + g, ok);
      return;
    }
    uint64_t p[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) p[k] = f2(raw.at(k), raw.at(k + 8));
    fwht16_pairs<WGeom<HD>::LANES>(p, rl, a.inv_sqrt_hd);
    if (fmt == S_T4) {
      encode4(p, cb.lv4[15], lin, sr, base + g * 8, ssec + g, ok);
    } else if (fmt == S_T3) {
      encode3(p, cb.lv3[7], lin, sr, base + g * 6, ssec + g, rl, ok);
    } else if (fmt == S_T2) {
      encode2(p, cb, sr, base + g * 4, ssec + g, ok);
    } else {
      float y[16];
#pragma unroll
      for (int k = 0; k < 8; ++k) f2_split(p[k], y[k], y[k + 8]);
      encode8(y, base + g * 16, ssec + g * 2, ok);
    }
  }
}

// One unit's loaded state: the lane's 16 input elements, its row's slot
// (-1: nothing to store) and kv head.
template <typename InT>
struct Unit {
  Raw<InT> raw;
  int64_t slot;
  int head;
};

// Issue the slot and input loads of unit u (units past the end load a valid
// row and get slot -1).
template <int HD, typename InT, bool VEC>
__device__ __forceinline__ void load_unit(const WriteArgs& a, uint32_t u, uint32_t units,
                                          uint32_t nq, int rw, int rl, Unit<InT>& x) {
  constexpr int ROWS = WGeom<HD>::ROWS;
  const int side = (int)(u & 1u);
  uint32_t q = (u >> 1) * ROWS + rw;
  const bool ok = u < units && q < nq;
  if (!ok) q = nq - 1;
  const uint32_t t = div_nkv(q, a);
  x.head = (int)(q - t * (uint32_t)a.nkv);
  x.slot = ok ? a.slots[t] : -1;
  const InT* src = reinterpret_cast<const InT*>(side ? a.value : a.key) +
                   (int64_t)t * (side ? a.value_stride : a.key_stride) + (int64_t)x.head * HD +
                   rl * kGroup;
  load_raw<InT, VEC>(src, x.raw);
}

// Units: (group of ROWS consecutive (token, kv head) pairs, side), side
// fastest.  A warp takes kUnitsPerWarp consecutive units per iteration and
// issues the slot and input loads of all of them before encoding any.
template <int HD, typename InT, bool VEC>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
cache_write_kernel(const WriteArgs a, const Codebooks cb) {
  using G = WGeom<HD>;
  constexpr int LANES = G::LANES, ROWS = G::ROWS, RB = kUnitsPerWarp;
  extern __shared__ uint2 tabs[];
  __shared__ float2 lin[2][kLin];   // Turbo4/3 bucket tables of the K and V sides
  __shared__ float2 sr[256];        // (s, 1/s) of every E4M3 scale byte (1/0 = 0)
  const int lane = threadIdx.x & 31;
  const int rl = lane & (LANES - 1), rw = lane / LANES;   // lane in the row, row of the warp
  const bool tk = side_has_table(a.k_side), tv = side_has_table(a.v_side);
  const bool shared_tab = a.k_side == a.v_side;
  uint2* tab_k = tabs;
  uint2* tab_v = (tk && !shared_tab) ? tabs + kKeys : tabs;
  for (int k = threadIdx.x; k < kKeys; k += kThreads) {
    if (tk) tab_k[k] = nvfp4_entry((uint32_t)k);
    if (tv && !shared_tab) tab_v[k] = nvfp4_entry((uint32_t)k);
  }
  static_assert(kLin == kThreads, "one table entry of each kind per thread");
  if (a.k_side == S_T4 || a.k_side == S_T3) lin[0][threadIdx.x] = lin_entry(a.k_side, threadIdx.x, cb);
  if (a.v_side == S_T4 || a.v_side == S_T3) lin[1][threadIdx.x] = lin_entry(a.v_side, threadIdx.x, cb);
  {
    const float sv = e4m3_to_float((uint8_t)threadIdx.x);
    sr[threadIdx.x] = make_float2(sv, sv == 0.f ? 0.f : 1.f / sv);
  }
  const uint32_t lin_k = (uint32_t)__cvta_generic_to_shared(&lin[0][0]);
  const uint32_t lin_v = (uint32_t)__cvta_generic_to_shared(&lin[1][0]);
  const uint32_t sr_a = (uint32_t)__cvta_generic_to_shared(&sr[0]);
  __syncthreads();
  const uint32_t nq = (uint32_t)a.num_tokens * (uint32_t)a.nkv;   // < 2^31 (host check)
  const uint32_t units = 2u * ((nq + ROWS - 1) / ROWS);
  const uint32_t step = gridDim.x * kWarps * RB;
  for (uint32_t u0 = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * RB; u0 < units; u0 += step) {
    Unit<InT> cur[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) load_unit<HD, InT, VEC>(a, u0 + r, units, nq, rw, rl, cur[r]);
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      int64_t slot = cur[r].slot;
      if (slot >= 0 && a.num_slots > 0 && slot >= a.num_slots) {
        if (rl == 0 && a.err) atomicOr(a.err, 1);
        slot = -1;
      }
      const uint32_t u = u0 + r;
      if (u < units) {   // warp-uniform
        const int side = (int)(u & 1u);
        write_group<HD, InT>(a, cb, side ? tab_v : tab_k, side ? lin_v : lin_k, sr_a, side, slot,
                             cur[r].head, cur[r].raw, rl, slot >= 0);
      }
    }
  }
}

template <int HD, typename InT, bool VEC>
cudaError_t launch_one(const WriteArgs& a, const Codebooks& cb, int sms, cudaStream_t st) {
  auto kern = cache_write_kernel<HD, InT, VEC>;
  const int ntab = (side_has_table(a.k_side) || side_has_table(a.v_side) ? 1 : 0) +
                   (side_has_table(a.k_side) && side_has_table(a.v_side) && a.v_side != a.k_side
                        ? 1 : 0);
  const size_t smem = (size_t)ntab * kKeys * sizeof(uint2);
  static int configured[64] = {0};   // per device: dynamic shared memory limit raised
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               2 * kKeys * (int)sizeof(uint2));
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  constexpr int ROWS = WGeom<HD>::ROWS;
  const int64_t nq = (int64_t)a.num_tokens * a.nkv;
  const int64_t units = 2 * ((nq + ROWS - 1) / ROWS);
  const int64_t want = (units + kWarps * kUnitsPerWarp - 1) / (kWarps * kUnitsPerWarp);
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * kCtasPerSm;
  const int grid = (int)(want < cap ? want : cap);
  kern<<<grid, kThreads, smem, st>>>(a, cb);
  return cudaGetLastError();
}

template <int HD, typename InT>
cudaError_t launch_hd(const WriteArgs& a, const Codebooks& cb, bool vec, int sms,
                      cudaStream_t st) {
  return vec ? launch_one<HD, InT, true>(a, cb, sms, st) : launch_one<HD, InT, false>(a, cb, sms, st);
}

}  // namespace

cudaError_t launch_cache_write(const WriteArgs& a, const Codebooks& cb, int head_dim,
                               bool in_bf16, bool vec, int sms, cudaStream_t st) {
  switch (head_dim) {
    case 64: return in_bf16 ? launch_hd<64, __nv_bfloat16>(a, cb, vec, sms, st)
                            : launch_hd<64, float>(a, cb, vec, sms, st);
    case 128: return in_bf16 ? launch_hd<128, __nv_bfloat16>(a, cb, vec, sms, st)
                             : launch_hd<128, float>(a, cb, vec, sms, st);
    case 256: return in_bf16 ? launch_hd<256, __nv_bfloat16>(a, cb, vec, sms, st)
                             : launch_hd<256, float>(a, cb, vec, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
