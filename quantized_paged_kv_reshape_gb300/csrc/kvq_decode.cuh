// Split-K paged decode attention over the quantized cache (CUDA cores, fp32).
//
// What it computes: "combs_models/kv.rs" attend with one query and
// repeat_kv (query head j reads kv head j / rep), over the pages listed in
// the block tables ("metrale_model_layers/layers/ops/kv_cache_bf16k_turbov.rs",
// paged_decode_attn_*: q, k/v caches, block_tables, seq_lens, inv_sqrt_d,
// q_stride, byte block strides, sliding_window).  For rotated sides
// ("spark_runtime/kv_cache.rs", is_wht_rotated: the WHT(Q) / iWHT(out)
// bookends) q is rotated once in the prologue, K is used as stored, V is
// accumulated in the rotated basis and the combine kernel rotates each
// output row back once.
//
// Work decomposition (flash-decoding): one CTA of 128 threads per
// (split, kv head, sequence).  A split is a run of pages of one sequence;
// the CTA serves all `rep` query heads of its kv head, so each cache byte is
// read from HBM once.  Pages are staged in tiles of 32 tokens through a
// multi-stage cp.async ring in shared memory (zero-filled for positions
// outside the window or the sequence).  Per tile:
//   scores : warp w takes dims [w*hd/4, (w+1)*hd/4), lane t takes token t;
//            the group scale of a 16-dim group multiplies the group's
//            partial dot product once;
//   softmax: warp w owns query heads w, w+4, ...; running max / sum in the
//            exp2 domain; the weights, times each 16-dim V group scale, go
//            to shared memory;
//   P.V    : thread (token group, dim pair) accumulates rep x 2 outputs.
// At the end the CTA writes (m, l, acc[hd]) per query head to the workspace;
// the combine kernel merges the splits.
#pragma once

#include <math_constants.h>

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
constexpr int clampi(int x, int lo, int hi) { return x < lo ? lo : x > hi ? hi : x; }

template <int KS, int VS, int HD, int RMAX>
struct DecodeCfg {
  using KG = SideGeom<KS, HD>;
  using VG = SideGeom<VS, HD>;
  static constexpr int TILE = 32;  // tokens per tile
  // Padded K row stride so that 32 lanes reading 32 rows at one offset spread
  // over the banks (an odd number of 16-byte units).
  static constexpr int KRS = (KG::ROW % 16 == 0 && (KG::ROW / 16) % 2 == 0) ? KG::ROW + 16 : KG::ROW;
  static constexpr int OFF_KS = TILE * KRS;
  static constexpr int OFF_V = OFF_KS + TILE * KG::SROW;
  static constexpr int OFF_VS = OFF_V + TILE * VG::ROW;
  static constexpr int STAGE = align_up(OFF_VS + TILE * VG::SROW, 16);
  static constexpr int NST = clampi(49152 / STAGE, 2, 4);
  static constexpr int GW = side_scale_bytes(VS) ? HD / kGroup : 1;   // V weight groups
  static constexpr int WS_G = TILE * RMAX + 4;                         // floats per weight group
  static constexpr int DP = HD / 2;                                    // dim pairs
  static constexpr int TG = 128 / DP;                                  // token groups in P.V
  static constexpr int OFF_Q = 0;                                      // float [RMAX][HD]
  static constexpr int OFF_LUT = OFF_Q + RMAX * HD * 4;                // float [2][16]
  static constexpr int OFF_SP = OFF_LUT + 128;                         // float [4][RMAX][32]
  static constexpr int OFF_WS = OFF_SP + 4 * RMAX * TILE * 4;          // float [GW][WS_G]
  static constexpr int OFF_AL = OFF_WS + GW * WS_G * 4;                // float [3*RMAX]
  static constexpr int OFF_ST = align_up(OFF_AL + 3 * RMAX * 4, 16);
  static constexpr int RED = TG * RMAX * HD * 4;                       // final reduction
  static constexpr int ST_BYTES = NST * STAGE > RED ? NST * STAGE : RED;
  static constexpr int SMEM = OFF_ST + ST_BYTES + 16;
};

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
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// 16 consecutive stored values (dims d0..d0+15) of a staged row: raw value
// (bf16 / e4m3) or codebook level (group scale not applied).
template <int S>
__device__ __forceinline__ void load16(const uint8_t* row, int d0, const float* lut, float (&v)[16]) {
  if constexpr (S == S_BF16) {
    const uint4 a = *reinterpret_cast<const uint4*>(row + d0 * 2);
    const uint4 b = *reinterpret_cast<const uint4*>(row + d0 * 2 + 16);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else if constexpr (S == S_FP8 || S == S_T8) {
    const uint4 a = *reinterpret_cast<const uint4*>(row + d0);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 lo = e4m3x2_to_float2((uint16_t)(w[i] & 0xffffu));
      const float2 hi = e4m3x2_to_float2((uint16_t)(w[i] >> 16));
      v[4 * i] = lo.x; v[4 * i + 1] = lo.y; v[4 * i + 2] = hi.x; v[4 * i + 3] = hi.y;
    }
  } else if constexpr (S == S_T4) {
    const uint2 a = *reinterpret_cast<const uint2*>(row + d0 / 2);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = lut[(a.x >> (4 * i)) & 15u];
      v[8 + i] = lut[(a.y >> (4 * i)) & 15u];
    }
  } else if constexpr (S == S_T3) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(row + d0 * 3 / 8);
    const uint64_t w = (uint64_t)p[0] | ((uint64_t)p[1] << 16) | ((uint64_t)p[2] << 32);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = lut[(uint32_t)(w >> (3 * i)) & 7u];
  } else if constexpr (S == S_T2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(row + d0 / 4);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = lut[(w >> (2 * i)) & 3u];
  }
}

// Stored values of dims 2*dp, 2*dp+1 of a staged row.
template <int S>
__device__ __forceinline__ float2 load2(const uint8_t* row, int dp, const float* lut) {
  if constexpr (S == S_BF16) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(row + dp * 4);
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  } else if constexpr (S == S_FP8 || S == S_T8) {
    return e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(row + dp * 2));
  } else if constexpr (S == S_T4) {
    const uint32_t b = row[dp];
    return make_float2(lut[b & 15u], lut[b >> 4]);
  } else if constexpr (S == S_T3) {
    const int bit = 6 * dp;
    const uint32_t w = (uint32_t)row[bit >> 3] | ((uint32_t)row[(bit >> 3) + 1] << 8);
    const uint32_t c = w >> (bit & 7);
    return make_float2(lut[c & 7u], lut[(c >> 3) & 7u]);
  } else {  // S_T2
    const uint32_t c = (uint32_t)row[dp >> 1] >> (4 * (dp & 1));
    return make_float2(lut[c & 3u], lut[(c >> 2) & 3u]);
  }
}

// Group scale g of a staged scale row (1 for sides without group scales).
template <int S>
__device__ __forceinline__ float group_scale(const uint8_t* srow, int g) {
  if constexpr (S == S_T4 || S == S_T3 || S == S_T2) {
    return e4m3_to_float(srow[g]);
  } else if constexpr (S == S_T8) {
    return bf16_bits_to_float(*reinterpret_cast<const uint16_t*>(srow + 2 * g));
  } else {
    return 1.0f;
  }
}

template <int S>
__device__ __forceinline__ const float* side_levels(const Codebooks& cb) {
  return S == S_T4 ? cb.lv4 : S == S_T3 ? cb.lv3 : cb.lv2;
}

template <int KS, int VS, int HD, int RMAX>
__global__ void __launch_bounds__(128)
decode_split_kernel(const DecodeArgs a, const Codebooks cb) {
  using C = DecodeCfg<KS, VS, HD, RMAX>;
  using KG = typename C::KG;
  using VG = typename C::VG;
  constexpr int E = HD / 32;
  constexpr int TILE = C::TILE;
  constexpr int RPW = (RMAX + 3) / 4;  // query heads per warp in the softmax

  extern __shared__ __align__(16) uint8_t smem[];
  float* q_s = reinterpret_cast<float*>(smem + C::OFF_Q);
  float* lut_k = reinterpret_cast<float*>(smem + C::OFF_LUT);
  float* lut_v = lut_k + 16;
  float* sp = reinterpret_cast<float*>(smem + C::OFF_SP);
  float* ws = reinterpret_cast<float*>(smem + C::OFF_WS);
  float* al = reinterpret_cast<float*>(smem + C::OFF_AL);
  uint8_t* stage = smem + C::OFF_ST;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int bs = a.bs;
  const int L = a.seq_lens[seq];
  const int lo = a.window > 0 ? max(0, L - a.window) : 0;
  const int first_page = lo / bs;
  int end_page = (L + bs - 1) / bs;
  if (end_page > a.max_blocks) {  // seq_len beyond the table row: clamp and flag
    if (tid == 0 && split == 0 && a.err) atomicOr(a.err, 2);
    end_page = a.max_blocks;
  }
  const int p0 = first_page + split * a.pages_per_split;
  const int p1 = min(p0 + a.pages_per_split, end_page);
  const size_t pstride = (size_t)a.nsplit * (HD + 4);
  float* part = a.part + ((size_t)(seq * a.nq + kvh * a.rep) * a.nsplit + split) * (HD + 4);

  if (p0 >= p1) {  // nothing to attend in this split
    for (int j = warp; j < a.rep; j += 4)
      for (int i = lane; i < HD + 4; i += 32) part[j * pstride + i] = (i == 0) ? -CUDART_INF_F : 0.f;
    return;
  }

  // ---- prologue: codebooks and (rotated) queries
  if constexpr (side_codebook(KS)) {
    if (tid < (1 << code_bits(KS))) lut_k[tid] = side_levels<KS>(cb)[tid];
  }
  if constexpr (side_codebook(VS)) {
    if (tid < (1 << code_bits(VS))) lut_v[tid] = side_levels<VS>(cb)[tid];
  }
  for (int j = warp; j < RMAX; j += 4) {
    float x[E];
    if (j < a.rep) {
      const int64_t qoff = (int64_t)seq * a.q_stride + (int64_t)(kvh * a.rep + j) * HD + lane * E;
#pragma unroll
      for (int i = 0; i < E; ++i)
        x[i] = a.q_bf16 ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(a.q)[qoff + i])
                        : reinterpret_cast<const float*>(a.q)[qoff + i];
      if constexpr (side_rotated(KS)) fwht_warp<E>(x, lane, a.inv_sqrt_hd);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) x[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < E; ++i) q_s[j * HD + lane * E + i] = x[i];
  }

  const int tp = TILE / bs;  // pages per tile
  const int ntiles = (p1 - p0 + tp - 1) / tp;
  const int64_t tab = (int64_t)seq * a.max_blocks;

  // Block id of token j of tile k, or -1 if the position is not attended.
  auto token_block = [&](int k, int j) -> int64_t {
    const int page = p0 + k * tp + j / bs;
    const int pos = page * bs + (j % bs);
    if (page >= p1 || pos < lo || pos >= L) return -1;
    const int64_t b = a.block_tables[tab + page];
    if (b < 0 || (a.num_blocks > 0 && b >= a.num_blocks)) return -2;
    return b;
  };

  auto issue = [&](int k) {
    uint8_t* sb = stage + (k % C::NST) * C::STAGE;
    constexpr int PER = KG::NCH + KG::NSCH + VG::NCH + VG::NSCH;
    for (int it = tid; it < TILE * PER; it += 128) {
      const int j = it / PER;
      int c = it - j * PER;
      const int64_t b = token_block(k, j);
      const bool ok = b >= 0;
      if (b == -2 && c == 0 && a.err) atomicOr(a.err, 2);
      const int64_t ridx = (int64_t)(j % bs) * a.nkv + kvh;
      const int64_t bb = ok ? b : 0;
      if (c < KG::NCH) {
        cp_async<KG::CH>(sb + j * C::KRS + c * KG::CH,
                         a.k_cache + bb * a.k_bstride + ridx * KG::ROW + c * KG::CH, ok);
        continue;
      }
      c -= KG::NCH;
      if constexpr (KG::NSCH > 0) {
        if (c < KG::NSCH) {
          cp_async<KG::SCH>(sb + C::OFF_KS + j * KG::SROW + c * KG::SCH,
                            a.k_cache + bb * a.k_bstride + a.k_dsec + ridx * KG::SROW + c * KG::SCH, ok);
          continue;
        }
        c -= KG::NSCH;
      }
      if (c < VG::NCH) {
        cp_async<VG::CH>(sb + C::OFF_V + j * VG::ROW + c * VG::CH,
                         a.v_cache + bb * a.v_bstride + ridx * VG::ROW + c * VG::CH, ok);
        continue;
      }
      c -= VG::NCH;
      if constexpr (VG::NSCH > 0) {
        cp_async<VG::SCH>(sb + C::OFF_VS + j * VG::SROW + c * VG::SCH,
                          a.v_cache + bb * a.v_bstride + a.v_dsec + ridx * VG::SROW + c * VG::SCH, ok);
      }
    }
  };

#pragma unroll
  for (int k = 0; k < C::NST - 1; ++k) {
    if (k < ntiles) issue(k);
    cp_async_commit();
  }

  float m_run[RPW], l_run[RPW];
#pragma unroll
  for (int i = 0; i < RPW; ++i) { m_run[i] = -CUDART_INF_F; l_run[i] = 0.f; }
  float acc[RMAX][2];
#pragma unroll
  for (int r = 0; r < RMAX; ++r) acc[r][0] = acc[r][1] = 0.f;

  const int dp = tid % C::DP, tg = tid / C::DP;

  for (int k = 0; k < ntiles; ++k) {
    cp_async_wait<C::NST - 2>();
    __syncthreads();
    if (k + C::NST - 1 < ntiles) issue(k + C::NST - 1);
    cp_async_commit();
    const uint8_t* sb = stage + (k % C::NST) * C::STAGE;

    // ---- scores: warp = dims quarter, lane = token
    {
      constexpr int QD = HD / 4;
      const uint8_t* krow = sb + lane * C::KRS;
      const uint8_t* ksrow = sb + C::OFF_KS + lane * KG::SROW;
      float s[RMAX];
#pragma unroll
      for (int r = 0; r < RMAX; ++r) s[r] = 0.f;
#pragma unroll
      for (int gi = 0; gi < QD / kGroup; ++gi) {
        const int d0 = warp * QD + gi * kGroup;
        float kv[16];
        load16<KS>(krow, d0, lut_k, kv);
        const float gs = group_scale<KS>(ksrow, d0 / kGroup);
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          const float4* qp = reinterpret_cast<const float4*>(q_s + r * HD + d0);
          float p = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 qv = qp[i];
            p = fmaf(qv.x, kv[4 * i], p);
            p = fmaf(qv.y, kv[4 * i + 1], p);
            p = fmaf(qv.z, kv[4 * i + 2], p);
            p = fmaf(qv.w, kv[4 * i + 3], p);
          }
          s[r] = fmaf(p, gs, s[r]);
        }
      }
#pragma unroll
      for (int r = 0; r < RMAX; ++r) sp[(warp * RMAX + r) * TILE + lane] = s[r];
    }
    __syncthreads();

    // ---- online softmax: warp w owns query heads w, w+4, ...
    {
      const int64_t b = token_block(k, lane);
      const bool valid = b >= 0;
      const uint8_t* vsrow = sb + C::OFF_VS + lane * VG::SROW;
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        const int r = warp + 4 * i;
        if (r < RMAX) {
          float sc = sp[(0 * RMAX + r) * TILE + lane] + sp[(1 * RMAX + r) * TILE + lane] +
                     sp[(2 * RMAX + r) * TILE + lane] + sp[(3 * RMAX + r) * TILE + lane];
          sc = valid ? sc * a.score_scale : -CUDART_INF_F;
          const float m_new = fmaxf(m_run[i], warp_max(sc));
          float alpha = 1.f, p = 0.f;
          if (m_new != -CUDART_INF_F) {
            alpha = exp2f(m_run[i] - m_new);
            p = exp2f(sc - m_new);
          }
          l_run[i] = l_run[i] * alpha + warp_sum(p);
          m_run[i] = m_new;
          if (a.sparse_thr > 0.f && p <= a.sparse_thr * l_run[i]) p = 0.f;
          if constexpr (C::GW > 1) {
#pragma unroll
            for (int g = 0; g < C::GW; ++g)
              ws[g * C::WS_G + lane * RMAX + r] = p * group_scale<VS>(vsrow, g);
          } else {
            ws[lane * RMAX + r] = p * a.v_mult;
          }
          if (lane == 0) al[r] = alpha;
        }
      }
    }
    __syncthreads();

    // ---- P.V: thread = (token group tg, dim pair dp)
    {
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        const float f = al[r];
        acc[r][0] *= f;
        acc[r][1] *= f;
      }
      const float* wsg = ws + (C::GW > 1 ? (dp * 2 / kGroup) * C::WS_G : 0);
      for (int t = tg; t < TILE; t += C::TG) {
        const float2 v = load2<VS>(sb + C::OFF_V + t * VG::ROW, dp, lut_v);
#pragma unroll
        for (int r = 0; r < RMAX; r += (RMAX >= 4 ? 4 : RMAX)) {
          if constexpr (RMAX >= 4) {
            const float4 w = *reinterpret_cast<const float4*>(wsg + t * RMAX + r);
            acc[r][0] = fmaf(w.x, v.x, acc[r][0]); acc[r][1] = fmaf(w.x, v.y, acc[r][1]);
            acc[r + 1][0] = fmaf(w.y, v.x, acc[r + 1][0]); acc[r + 1][1] = fmaf(w.y, v.y, acc[r + 1][1]);
            acc[r + 2][0] = fmaf(w.z, v.x, acc[r + 2][0]); acc[r + 2][1] = fmaf(w.z, v.y, acc[r + 2][1]);
            acc[r + 3][0] = fmaf(w.w, v.x, acc[r + 3][0]); acc[r + 3][1] = fmaf(w.w, v.y, acc[r + 3][1]);
          } else {
#pragma unroll
            for (int rr = 0; rr < RMAX; ++rr) {
              const float w = wsg[t * RMAX + rr];
              acc[rr][0] = fmaf(w, v.x, acc[rr][0]);
              acc[rr][1] = fmaf(w, v.y, acc[rr][1]);
            }
          }
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- epilogue: merge token groups, write (m, l, acc) per query head
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int r = warp + 4 * i;
    if (r < RMAX && lane == 0) {
      al[RMAX + 2 * r] = m_run[i];
      al[RMAX + 2 * r + 1] = l_run[i];
    }
  }
  float* red = reinterpret_cast<float*>(stage);
  if constexpr (C::TG > 1) {
    if (tg > 0) {
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
        *reinterpret_cast<float2*>(red + ((tg * RMAX) + r) * HD + 2 * dp) =
            make_float2(acc[r][0], acc[r][1]);
    }
  }
  __syncthreads();
  if (tg == 0) {
    if constexpr (C::TG > 1) {
#pragma unroll
      for (int g2 = 1; g2 < C::TG; ++g2)
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          const float2 o = *reinterpret_cast<const float2*>(red + ((g2 * RMAX) + r) * HD + 2 * dp);
          acc[r][0] += o.x;
          acc[r][1] += o.y;
        }
    }
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      if (r < a.rep) {
        float* pp = part + r * pstride;
        *reinterpret_cast<float2*>(pp + 4 + 2 * dp) = make_float2(acc[r][0], acc[r][1]);
        if (dp == 0) {
          pp[0] = al[RMAX + 2 * r];
          pp[1] = al[RMAX + 2 * r + 1];
        }
      }
    }
  }
}

template <int KS, int VS, int HD, int RMAX>
cudaError_t launch_decode_inst(const DecodeArgs& a, const Codebooks& cb, cudaStream_t st) {
  using C = DecodeCfg<KS, VS, HD, RMAX>;
  auto kern = decode_split_kernel<KS, VS, HD, RMAX>;
  if (C::SMEM > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(a.nsplit, a.nkv, a.num_seqs);
  kern<<<grid, 128, C::SMEM, st>>>(a, cb);
  return cudaGetLastError();
}

template <int KS, int VS, int HD>
cudaError_t launch_decode_r(int rmax, const DecodeArgs& a, const Codebooks& cb, cudaStream_t st) {
  switch (rmax) {
    case 1: return launch_decode_inst<KS, VS, HD, 1>(a, cb, st);
    case 2: return launch_decode_inst<KS, VS, HD, 2>(a, cb, st);
    case 4: return launch_decode_inst<KS, VS, HD, 4>(a, cb, st);
    case 8: return launch_decode_inst<KS, VS, HD, 8>(a, cb, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int KS, int VS>
cudaError_t launch_decode_pair(int hd, int rmax, const DecodeArgs& a, const Codebooks& cb,
                               cudaStream_t st) {
  switch (hd) {
    case 64: return launch_decode_r<KS, VS, 64>(rmax, a, cb, st);
    case 128: return launch_decode_r<KS, VS, 128>(rmax, a, cb, st);
    case 256: return launch_decode_r<KS, VS, 256>(rmax, a, cb, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int KS, int VS>
size_t smem_pair(int hd, int rmax) {
#define KVQ_SM(H, R) if (hd == H && rmax == R) return (size_t)DecodeCfg<KS, VS, H, R>::SMEM;
  KVQ_SM(64, 1) KVQ_SM(64, 2) KVQ_SM(64, 4) KVQ_SM(64, 8)
  KVQ_SM(128, 1) KVQ_SM(128, 2) KVQ_SM(128, 4) KVQ_SM(128, 8)
  KVQ_SM(256, 1) KVQ_SM(256, 2) KVQ_SM(256, 4) KVQ_SM(256, 8)
#undef KVQ_SM
  return 0;
}

}  // namespace kvq
