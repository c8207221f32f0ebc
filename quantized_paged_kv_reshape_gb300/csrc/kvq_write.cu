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
// Work mapping: a (token, kv head, side) row is held by LANES lanes (16 for
// head_dim 64/128, so a warp encodes two rows at once, 32 for 256); lane l of
// the row holds the E = head_dim/LANES consecutive elements l*E .. l*E+E-1.
// The two rows of a warp are the same (side, kv head) of two consecutive
// tokens, so both halves take the same format path.  The rotation runs in
// registers and shuffles, the 16-element group max in a shuffle reduction
// over the 16/E lanes of the group, the codes are packed per lane and merged
// across the few lanes whose bits complete a byte, then stored.  Units of
// consecutive warps are consecutive kv heads of one token pair, so both the
// strided input reads and the cache stores stay contiguous.
#include "kvq_common.cuh"
#include "kvq_launch.h"

namespace kvq {

namespace {

// Lanes per row and elements per lane of a head_dim.
template <int HD>
struct WGeom {
  static constexpr int LANES = HD == 256 ? 32 : 16;
  static constexpr int HALVES = 32 / LANES;   // rows per warp instruction
  static constexpr int E = HD / LANES;
};

template <int N>
__device__ __forceinline__ void store_bytes(uint8_t* dst, uint32_t lo, uint32_t hi = 0) {
  if constexpr (N == 1) {
    *dst = (uint8_t)lo;
  } else if constexpr (N == 2) {
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)lo;
  } else if constexpr (N == 3) {
    dst[0] = (uint8_t)lo;
    dst[1] = (uint8_t)(lo >> 8);
    dst[2] = (uint8_t)(lo >> 16);
  } else if constexpr (N == 4) {
    *reinterpret_cast<uint32_t*>(dst) = lo;
  } else if constexpr (N == 8) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
  }
}

template <int E, typename InT, bool VEC>
__device__ __forceinline__ void load_row(const InT* src, float (&x)[E]) {
  if constexpr (VEC && sizeof(InT) == 2) {
    // E bf16 = 2E bytes: 4, 8 or 16 byte vector loads
    if constexpr (E == 2) {
      uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(src));
      x[0] = bf16_bits_to_float(w & 0xffffu);
      x[1] = bf16_bits_to_float(w >> 16);
    } else if constexpr (E == 4) {
      uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
      x[0] = bf16_bits_to_float(w.x & 0xffffu); x[1] = bf16_bits_to_float(w.x >> 16);
      x[2] = bf16_bits_to_float(w.y & 0xffffu); x[3] = bf16_bits_to_float(w.y >> 16);
    } else {
      uint4 w = __ldg(reinterpret_cast<const uint4*>(src));
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[2 * i] = bf16_bits_to_float(ws[i] & 0xffffu);
        x[2 * i + 1] = bf16_bits_to_float(ws[i] >> 16);
      }
    }
  } else if constexpr (VEC && sizeof(InT) == 4) {
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      float2 f = __ldg(reinterpret_cast<const float2*>(src) + i / 2);
      x[i] = f.x;
      x[i + 1] = f.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if constexpr (sizeof(InT) == 2)
        x[i] = bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(src) + i));
      else
        x[i] = __ldg(reinterpret_cast<const float*>(src) + i);
    }
  }
}

// Pack E codes of B bits (code i at bits B*i) and store the row's code bytes:
// lanes whose bits do not fill whole bytes are merged into a chunk of C lanes
// first (C*B*E bits, a whole number of bytes <= 4).
template <int B, int E>
__device__ __forceinline__ void store_codes(uint8_t* row_codes, const int (&code)[E], int lane,
                                            bool ok) {
  constexpr int LB = B * E;                       // bits per lane
  constexpr int G = (LB % 8 == 0) ? 8 : (LB % 4 == 0) ? 4 : 2;  // gcd(LB, 8)
  constexpr int C = 8 / G;                        // lanes per whole-byte chunk
  constexpr int CB = C * LB / 8;                  // bytes per chunk
  static_assert(C * LB <= 32, "chunk exceeds 32 bits");
  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < E; ++i) bits |= (uint32_t)code[i] << (B * i);
#pragma unroll
  for (int j = 1; j < C; ++j) {
    uint32_t o = __shfl_down_sync(0xffffffffu, bits, j);
    if ((lane % C) == 0) bits |= o << (j * LB);
  }
  if (ok && (lane % C) == 0) store_bytes<CB>(row_codes + (lane / C) * CB, bits);
}

template <int E>
__device__ __forceinline__ float group_amax(const float (&y)[E]) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) a = fmaxf(a, fabsf(y[i]));
  constexpr int LPG = kGroup / E;  // lanes per group
#pragma unroll
  for (int m = 1; m < LPG; m <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
  return a;
}

template <int E, int B>
__device__ __forceinline__ void write_turbo(float (&y)[E], const float lv_max,
                                            const uint2* bucket, const float* th2,
                                            uint8_t* row_codes, uint8_t* row_scales, int lane,
                                            bool ok) {
  const float amax = group_amax<E>(y);
  const float ratio = amax / lv_max;               // IEEE fp32 divide
  const uint8_t sbyte = e4m3_from_float(ratio);
  const float s = e4m3_to_float(sbyte);
  const float r = s == 0.f ? 0.f : 1.f / s;
  int code[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {  // v = y / s, IEEE-rounded
    const float v = div_by_scale(y[i], s, r);
    code[i] = s == 0.f ? 1 << (B - 1) : B == 2 ? lm_code2(v, th2) : lm_code_bucket<B>(v, bucket);
  }
  store_codes<B, E>(row_codes, code, lane, ok);
  constexpr int LPG = kGroup / E;
  if (ok && (lane % LPG) == 0) row_scales[lane / LPG] = sbyte;
}

// NVFP4: per 16-element group s = E4M3(amax / 6), code = E2M1(x / s) (both
// fp32 divides); a zero scale stores code 0.  No rotation.
template <int E>
__device__ __forceinline__ void write_nvfp4(const float (&x)[E], uint8_t* row_codes,
                                            uint8_t* row_scales, int lane, bool ok) {
  const float amax = group_amax<E>(x);
  const uint8_t sbyte = e4m3_from_float(amax / 6.0f);
  const float s = e4m3_to_float(sbyte);
  const float r = s == 0.f ? 0.f : 1.f / s;
  int code[E];
#pragma unroll
  for (int i = 0; i < E; ++i)   // x / s IEEE-rounded; its sign is that of x
    code[i] = s == 0.f ? 0 : (int)e2m1_from_float(div_by_scale(x[i], s, r), signbit(x[i]));
  store_codes<4, E>(row_codes, code, lane, ok);
  constexpr int LPG = kGroup / E;
  if (ok && (lane % LPG) == 0) row_scales[lane / LPG] = sbyte;
}

// Encode and store one row already loaded into x (this lane's E elements;
// lane = the lane within the row).  Every lane of the warp runs it (the
// shuffles need them all); ok = false (no valid slot) computes but stores
// nothing.
template <int HD>
__device__ __forceinline__ void write_row(const WriteArgs& a, const Codebooks& cb,
                                          const uint2 (*bucket)[kBuckets], int side, int64_t slot,
                                          int h, float (&x)[WGeom<HD>::E], int lane, bool ok) {
  constexpr int E = WGeom<HD>::E, LANES = WGeom<HD>::LANES;
  if (!ok) slot = 0;
  int64_t blk;
  int off;
  if (a.bs_shift >= 0) {          // power-of-two block size
    blk = slot >> a.bs_shift;
    off = (int)(slot & (a.bs - 1));
  } else if (slot < 0xffffffffll) {   // 32-bit division
    const uint32_t s32 = (uint32_t)slot;
    blk = s32 / (uint32_t)a.bs;
    off = (int)(s32 - (uint32_t)blk * (uint32_t)a.bs);
  } else {
    blk = slot / a.bs;
    off = (int)(slot - blk * a.bs);
  }
  const int fmt = side ? a.v_side : a.k_side;
  uint8_t* base = (side ? a.v_cache : a.k_cache) + blk * (side ? a.v_bstride : a.k_bstride);
  const int64_t dsec = side ? a.v_dsec : a.k_dsec;
  const int64_t ridx = (int64_t)off * a.nkv + h;   // row index inside the block
  if (fmt == S_BF16) {
    uint32_t w[(E + 1) / 2];
#pragma unroll
    for (int i = 0; i < E; i += 2)
      w[i / 2] = (uint32_t)bf16_bits_from_float(x[i]) |
                 ((uint32_t)bf16_bits_from_float(x[i + 1]) << 16);
    uint8_t* dst = base + (ridx * HD + lane * E) * 2;
    if (ok) {
      if constexpr (E == 2) store_bytes<4>(dst, w[0]);
      else if constexpr (E == 4) store_bytes<8>(dst, w[0], w[1]);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else if (fmt == S_FP8) {
    const float sc = side ? a.v_scale : a.k_scale;
    uint32_t w[(E + 3) / 4] = {};
#pragma unroll
    for (int i = 0; i < E; ++i) w[i / 4] |= (uint32_t)e4m3_from_float(x[i] / sc) << (8 * (i % 4));
    uint8_t* dst = base + ridx * HD + lane * E;
    if (ok) {
      if constexpr (E == 2) store_bytes<2>(dst, w[0]);
      else if constexpr (E == 4) store_bytes<4>(dst, w[0]);
      else store_bytes<8>(dst, w[0], w[1]);
    }
  } else if (fmt == S_NVFP4) {
    write_nvfp4<E>(x, base + ridx * (HD / 2), base + dsec + ridx * (HD / kGroup), lane, ok);
  } else {
    fwht_warp<E, LANES>(x, lane, a.inv_sqrt_hd);
    if (fmt == S_T8) {
      const float amax = group_amax<E>(x);
      const uint16_t sbits = bf16_bits_from_float(amax / 448.0f);
      const float s = bf16_bits_to_float(sbits);
      uint32_t w[(E + 3) / 4] = {};
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const uint32_t b = s == 0.f ? 0u : (uint32_t)e4m3_from_float(x[i] / s);
        w[i / 4] |= b << (8 * (i % 4));
      }
      uint8_t* dst = base + ridx * HD + lane * E;
      if (ok) {
        if constexpr (E == 2) store_bytes<2>(dst, w[0]);
        else if constexpr (E == 4) store_bytes<4>(dst, w[0]);
        else store_bytes<8>(dst, w[0], w[1]);
      }
      constexpr int LPG = kGroup / E;
      if (ok && (lane % LPG) == 0)
        store_bytes<2>(base + dsec + (ridx * (HD / kGroup) + lane / LPG) * 2, sbits);
    } else if (fmt == S_T4) {
      write_turbo<E, 4>(x, cb.lv4[15], bucket[0], nullptr, base + ridx * (HD / 2),
                        base + dsec + ridx * (HD / kGroup), lane, ok);
    } else if (fmt == S_T3) {
      write_turbo<E, 3>(x, cb.lv3[7], bucket[1], nullptr, base + ridx * (HD * 3 / 8),
                        base + dsec + ridx * (HD / kGroup), lane, ok);
    } else {
      float th[3];
#pragma unroll
      for (int i = 0; i < 3; ++i) th[i] = cb.th2[i];
      write_turbo<E, 2>(x, cb.lv2[3], bucket[2], th, base + ridx * (HD / 4),
                        base + dsec + ridx * (HD / kGroup), lane, ok);
    }
  }
}

// Each warp takes RB consecutive units per iteration (unit = (token pair,
// side, kv head), heads fastest; half h of the warp holds the pair's token
// 2p + h, or the whole warp token p for head_dim 256): the slot and input
// loads of all RB units are issued before any row is encoded, so every warp
// keeps RB units of loads in flight.
template <int HD, typename InT, bool VEC>
__global__ void __launch_bounds__(256, 4)   // <= 64 registers: four CTAs per SM
cache_write_kernel(const WriteArgs a, const Codebooks cb) {
  using G = WGeom<HD>;
  constexpr int E = G::E, LANES = G::LANES, HALVES = G::HALVES;
  constexpr int RB = 2;  // measured on GB300: 2 beats 1 and 4 for every format
  const int lane = threadIdx.x & 31;
  const int rl = lane & (LANES - 1), half = lane / LANES;   // lane in the row, row of the warp
  __shared__ uint2 bucket[3][kBuckets];  // codebook-search buckets (4, 3, 2 bits)
  for (int i = threadIdx.x; i < 3 * kBuckets; i += blockDim.x)
    bucket[i / kBuckets][i % kBuckets] =
        make_uint2(cb.bucket[i / kBuckets][i % kBuckets][0], cb.bucket[i / kBuckets][i % kBuckets][1]);
  __syncthreads();
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  // units fit 32 bits (rows are checked on the host): one division per batch
  const uint32_t upp = 2u * (uint32_t)a.nkv;                  // units per token pair
  const uint32_t pairs = ((uint32_t)a.num_tokens + HALVES - 1) / HALVES;
  const uint32_t units = pairs * upp;
  for (int64_t u00 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RB;
       u00 < units; u00 += warps_total * RB) {
    int64_t slot[RB];
    int side[RB], head[RB];
    float x[RB][E];
    const uint32_t u0 = (uint32_t)u00;
    uint32_t p0 = u0 / upp;
    uint32_t rem0 = u0 - p0 * upp;
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      uint32_t p = p0, rem = rem0 + r;
      while (rem >= upp) { rem -= upp; ++p; }                   // at most RB/upp steps
      const bool unit_ok = u0 + r < units;
      if (!unit_ok) { p = pairs - 1; rem = upp - 1; }           // a valid row, dropped below
      side[r] = (int)rem >= a.nkv;
      head[r] = rem - side[r] * a.nkv;
      uint32_t t = p * HALVES + half;
      const bool tok_ok = unit_ok && t < (uint32_t)a.num_tokens;
      if (t >= (uint32_t)a.num_tokens) t = (uint32_t)a.num_tokens - 1;
      slot[r] = tok_ok ? a.slots[t] : -1;
      const InT* src = reinterpret_cast<const InT*>(side[r] ? a.value : a.key) +
                       (int64_t)t * (side[r] ? a.value_stride : a.key_stride) + (int64_t)head[r] * HD +
                       rl * E;
      load_row<E, InT, VEC>(src, x[r]);
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      if (slot[r] >= 0 && a.num_slots > 0 && slot[r] >= a.num_slots) {
        if (rl == 0 && a.err) atomicOr(a.err, 1);
        slot[r] = -1;
      }
    }
#pragma unroll
    for (int r = 0; r < RB; ++r)
      if (u0 + r < units)   // warp-uniform: both halves encode (their shuffles pair up)
        write_row<HD>(a, cb, bucket, side[r], slot[r], head[r], x[r], rl, slot[r] >= 0);
  }
}

template <int HD, typename InT>
cudaError_t launch_hd(const WriteArgs& a, const Codebooks& cb, bool vec, int grid,
                      cudaStream_t st) {
  if (vec)
    cache_write_kernel<HD, InT, true><<<grid, 256, 0, st>>>(a, cb);
  else
    cache_write_kernel<HD, InT, false><<<grid, 256, 0, st>>>(a, cb);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cache_write(const WriteArgs& a, const Codebooks& cb, int head_dim,
                               bool in_bf16, bool vec, int grid, cudaStream_t st) {
  switch (head_dim) {
    case 64: return in_bf16 ? launch_hd<64, __nv_bfloat16>(a, cb, vec, grid, st)
                            : launch_hd<64, float>(a, cb, vec, grid, st);
    case 128: return in_bf16 ? launch_hd<128, __nv_bfloat16>(a, cb, vec, grid, st)
                             : launch_hd<128, float>(a, cb, vec, grid, st);
    case 256: return in_bf16 ? launch_hd<256, __nv_bfloat16>(a, cb, vec, grid, st)
                             : launch_hd<256, float>(a, cb, vec, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
