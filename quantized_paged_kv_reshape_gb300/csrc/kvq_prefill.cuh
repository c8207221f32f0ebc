// Chunked-prefill attention over the quantized paged cache, on tensor cores.
//
// "combs_models/kv.rs" attend (scores, causal mask, softmax, P.V) with
// repeat_kv for a chunk of new query tokens per sequence, after the chunk's
// K/V rows were written to the cache; "spark_runtime/kv_cache.rs"
// is_wht_rotated bookends (q rotated forward when K is stored rotated, the
// output rotated back when V is).  Sequence s holds L = seq_lens[s]
// positions; its C = cu_q[s+1] - cu_q[s] queries are the last C positions,
// query i at p = L - C + i attends to [max(0, p + 1 - W), p] (W = window, 0 =
// none).
//
// One CTA per (query tile, kv head, sequence): ROWS = 64 score rows = QT
// query tokens x RP (GQA ratio rounded up to a power of two) heads, 16 rows
// per warp.  Per 16-token KV slab, the raw cache rows are staged by cp.async
// (double buffered) and dequantized once, by all threads, into fp16/bf16
// operand planes in shared memory (level x group scale as hi + lo parts
// where one 16-bit value is not exact), which every warp then reads with
// ldmatrix:
//   S[16 rows x 16 tok] = Q[16 x hd] . K^T      (m16n8k16)
//   causal / window mask, online softmax (exp2 domain, fp32)
//   O[16 x hd] += P[16 x 16 tok] . V[16 tok x hd]
// q and P carry hi + lo 16-bit parts like the decode (products with ~16
// significant bits).  With head_dim 256 two warps share 16 rows and split
// the output dims (both compute S).  At the end each row is normalised,
// rotated back (rotated V) and stored.
#pragma once

#include <math_constants.h>

#include "kvq_decode_common.cuh"
#include "kvq_decode_mma.cuh"
#include "kvq_launch.h"

namespace kvq {

// Operand planes of one side: 1 (the 16-bit value is exact) or 2 (hi + lo).
template <int S>
struct PfSide {
  static constexpr bool BF = S == S_BF16;
  static constexpr int PLANES = (S == S_BF16 || S == S_FP8 || S == S_NVFP4) ? 1 : 2;
};

template <int KS, int VS, int HD>
struct PfCfg {
  static constexpr int DSPLIT = HD / 128 > 1 ? 2 : 1;      // warps sharing 16 rows
  static constexpr int NW = 4 * DSPLIT;
  static constexpr int NT = 32 * NW;
  static constexpr int ROWS = 64;
  static constexpr int PITCH = HD + 8;                       // halves per plane row
  static constexpr int NSUB = 1;  // 16-token sub-slabs per stage (2 measured slower on GB300)
  static constexpr int TOK = 16 * NSUB;                      // tokens per stage
  static constexpr int KROW = SideGeom<KS, HD>::ROW, KSROW = SideGeom<KS, HD>::SROW;
  static constexpr int VROW = SideGeom<VS, HD>::ROW, VSROW = SideGeom<VS, HD>::SROW;
  // raw stage: [TOK][KROW] [TOK][KSROW] [TOK][VROW] [TOK][VSROW], 16-byte aligned parts
  static constexpr int R_KS = align_up(TOK * KROW, 16);
  static constexpr int R_V = R_KS + align_up(TOK * KSROW, 16);
  static constexpr int R_VS = R_V + align_up(TOK * VROW, 16);
  static constexpr int RAW = R_VS + align_up(TOK * VSROW, 16);
  // shared memory map (bytes)
  static constexpr int QPLANE = ROWS * PITCH * 2;
  static constexpr int KPLANE = TOK * PITCH * 2;
  static constexpr int OFF_Q = 0;                                   // q hi, q lo
  static constexpr int OFF_K = OFF_Q + 2 * QPLANE;                  // k planes
  static constexpr int OFF_V = OFF_K + PfSide<KS>::PLANES * KPLANE; // v planes
  static constexpr int OFF_RAW = OFF_V + PfSide<VS>::PLANES * KPLANE;
  static constexpr int OFF_OFFS = OFF_RAW + 2 * RAW;                // int64 [2][64] row offsets
  static constexpr int OFF_LV = OFF_OFFS + 2 * 64 * 8;              // level tables [2][2][16] fp32
  static constexpr int OFF_ML = OFF_LV + 2 * 2 * 16 * 4;            // [NW][16] m, l
  static constexpr int SMEM_MAIN = OFF_ML + NW * 16 * 2 * 4;
  static constexpr int OUTB = ROWS * (HD + 4) * 4;                  // output staging (fp32)
  static constexpr int SMEM = SMEM_MAIN > OUTB ? SMEM_MAIN : OUTB;
};

// Level table entries (hi, lo parts of 7 significant bits; E2M1 values
// exactly) of a codebook side into shared memory.
template <int S>
__device__ __forceinline__ void pf_fill_levels(float* hi, float* lo, const Codebooks& cb, int tid,
                                               int nt) {
  if constexpr (side_codebook(S)) {
    const float* lv = side_levels<S>(cb);
    constexpr int n = 1 << code_bits(S);
    for (int i = tid; i < n; i += nt) {
      const float h = tc::round_sig7(lv[i]);
      hi[i] = h;
      lo[i] = tc::round_sig7(lv[i] - h);
    }
  }
}

// Dequantize EPT consecutive elements (d0 .. d0 + EPT - 1, d0 % 8 == 0) of
// one staged row into 16-bit plane words (pairs, low half = first element).
template <int S, int HD, int EPT>
__device__ __forceinline__ void pf_dequant(const uint8_t* row, const uint8_t* srow, int d0,
                                           const float* lvh, const float* lvl, uint32_t (&hw)[EPT / 2],
                                           uint32_t (&lw)[EPT / 2]) {
  if constexpr (S == S_BF16) {
#pragma unroll
    for (int i = 0; i < EPT / 2; ++i) {
      hw[i] = *reinterpret_cast<const uint32_t*>(row + 2 * d0 + 4 * i);
      lw[i] = 0u;
    }
  } else if constexpr (S == S_FP8) {
#pragma unroll
    for (int i = 0; i < EPT / 2; ++i) {
      hw[i] = tc::e4m3x2_f16x2(*reinterpret_cast<const uint16_t*>(row + d0 + 2 * i));
      lw[i] = 0u;
    }
  } else if constexpr (S == S_T8) {
    // value = E4M3 x BF16 group scale, exact in fp32 (12 significant bits)
#pragma unroll
    for (int i = 0; i < EPT / 2; ++i) {
      const int d = d0 + 2 * i;
      const float sc = bf16_bits_to_float(*reinterpret_cast<const uint16_t*>(srow + 2 * (d / kGroup)));
      const float2 e = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(row + d));
      const float v0 = e.x * sc, v1 = e.y * sc;
      tc::split2<false>(v0, v1, hw[i], lw[i]);
    }
  } else {  // codebook sides: level parts x E4M3 group scale, exact in fp16
    constexpr int B = code_bits(S);
    uint64_t bits = 0;
    constexpr int NB = EPT * B / 8;
    const uint8_t* src = row + d0 * B / 8;
#pragma unroll
    for (int i = 0; i < NB; ++i) bits |= (uint64_t)src[i] << (8 * i);
#pragma unroll
    for (int i = 0; i < EPT / 2; ++i) {
      const int d = d0 + 2 * i;
      const float sc = e4m3_to_float(srow[d / kGroup]);
      const uint32_t c0 = (uint32_t)(bits >> (B * 2 * i)) & ((1u << B) - 1);
      const uint32_t c1 = (uint32_t)(bits >> (B * (2 * i + 1))) & ((1u << B) - 1);
      hw[i] = tc::pack2<false>(lvh[c0] * sc, lvh[c1] * sc);
      lw[i] = PfSide<S>::PLANES == 2 ? tc::pack2<false>(lvl[c0] * sc, lvl[c1] * sc) : 0u;
    }
  }
}

template <int KS, int VS, int HD>
__global__ void __launch_bounds__(PfCfg<KS, VS, HD>::NT)
prefill_tc_kernel(const PrefillArgs a, const Codebooks cb) {
  using C = PfCfg<KS, VS, HD>;
  using KP = PfSide<KS>;
  using VP = PfSide<VS>;
  constexpr int NW = C::NW, NT = C::NT, DS = C::DSPLIT, PITCH = C::PITCH;
  constexpr int E = HD / 32;
  constexpr int EPT = 16 * HD / NT;            // dequantized elements per thread and side
  constexpr int NDT = HD / DS / 8;             // output n-tiles per warp
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* qh_s = reinterpret_cast<uint16_t*>(smem + C::OFF_Q);
  uint16_t* ql_s = qh_s + C::ROWS * PITCH;
  uint16_t* kh_s = reinterpret_cast<uint16_t*>(smem + C::OFF_K);
  uint16_t* kl_s = kh_s + C::TOK * PITCH;     // used when KP::PLANES == 2
  uint16_t* vh_s = reinterpret_cast<uint16_t*>(smem + C::OFF_V);
  uint16_t* vl_s = vh_s + C::TOK * PITCH;     // used when VP::PLANES == 2
  uint8_t* raw = smem + C::OFF_RAW;
  uint8_t* vrow_s = smem + C::OFF_OFFS;        // [2][TOK] row valid flags
  float* lv = reinterpret_cast<float*>(smem + C::OFF_LV);   // [K, V][hi, lo][16]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int tile = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int q0 = a.cu_q[seq];
  const int cq = a.cu_q[seq + 1] - q0;
  const int rp = a.rp, qt = C::ROWS / rp;
  const int t0 = tile * qt;                    // chunk index of the tile's first query
  if (t0 >= cq) return;
  const int nq_tile = min(qt, cq - t0);
  int len = a.seq_lens[seq];
  const int64_t cap = (int64_t)a.max_blocks * a.bs;
  if (len > cap) {
    if (tid == 0 && tile == 0 && kvh == 0 && a.err) atomicOr(a.err, 2);
    len = (int)cap;
  }
  const int pbase = len - cq + t0;             // position of the tile's query 0
  const int p_last = pbase + nq_tile - 1;
  const int lbs = 31 - __clz(a.bs);
  const int64_t tab = (int64_t)seq * a.max_blocks;

  // ---- queries of the tile (rotated when K is), hi/lo planes in K's type
  for (int r = warp; r < C::ROWS; r += NW) {
    const int qi = r / rp, hj = r - qi * rp;
    float x[E];
    if (qi < nq_tile && hj < a.rep) {
      const int64_t off = (int64_t)(q0 + t0 + qi) * a.q_stride + (int64_t)(kvh * a.rep + hj) * HD + lane * E;
#pragma unroll
      for (int i = 0; i < E; ++i)
        x[i] = a.q_bf16 ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(a.q)[off + i])
                        : reinterpret_cast<const float*>(a.q)[off + i];
      if constexpr (side_rotated(KS)) fwht_warp<E>(x, lane, a.inv_sqrt_hd);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) x[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      uint32_t h, l;
      tc::split2<KP::BF>(x[i], x[i + 1], h, l);
      *reinterpret_cast<uint32_t*>(qh_s + r * PITCH + lane * E + i) = h;
      *reinterpret_cast<uint32_t*>(ql_s + r * PITCH + lane * E + i) = l;
    }
  }
  pf_fill_levels<KS>(lv, lv + 16, cb, tid, NT);
  pf_fill_levels<VS>(lv + 32, lv + 48, cb, tid, NT);

  // ---- KV slabs [slab_begin, slab_end) cover every position a query attends
  float o[NDT][4];
#pragma unroll
  for (int i = 0; i < NDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m[2] = {-CUDART_INF_F, -CUDART_INF_F}, l[2] = {0.f, 0.f};
  const int p_first = max(pbase, 0);
  const int lo_first = a.window > 0 ? max(0, p_first + 1 - a.window) : 0;
  const int slab_begin = lo_first / C::TOK;
  const int slab_end = p_last >= 0 ? p_last / C::TOK + 1 : slab_begin;

  // Copy the K/V rows of slab `sl` (positions TOK sl .. TOK sl + TOK - 1) into raw
  // buffer b; rows outside [0, len) or with a bad block id are zero-filled
  // and flagged invalid.
  auto row_src = [&](int pos, int64_t& blk, int64_t& rr) -> bool {
    if (pos < 0 || pos >= len) return false;
    blk = a.block_tables[tab + (pos >> lbs)];
    if (blk < 0 || (a.num_blocks > 0 && blk >= a.num_blocks)) return false;
    rr = (int64_t)(pos & (a.bs - 1)) * a.nkv + kvh;   // row inside the block
    return true;
  };
  auto copy_part = [&](uint8_t* dst, const uint8_t* cache, int64_t stride, int64_t sec, int sl,
                       auto rowbytes_c, auto chunk_c) {
    constexpr int RB = decltype(rowbytes_c)::value, CHB = decltype(chunk_c)::value;
    if constexpr (RB > 0) {
      constexpr int NC = RB / CHB, TOT = C::TOK * NC;
      for (int q = tid; q < TOT; q += NT) {
        const int row = q / NC, ch = q - row * NC;
        int64_t blk = 0, rr = 0;
        const bool ok = row_src(sl * C::TOK + row, blk, rr);
        const int64_t src = ok ? blk * stride + sec + rr * RB : 0;
        cp_async<CHB>(dst + row * RB + ch * CHB, cache + src + ch * CHB, ok);
      }
    }
  };
  auto issue = [&](int sl, int b) {
    uint8_t* rb = raw + b * C::RAW;
    using KG = SideGeom<KS, HD>;
    using VG = SideGeom<VS, HD>;
    copy_part(rb, a.k_cache, a.k_bstride, 0, sl, std::integral_constant<int, KG::ROW>{},
              std::integral_constant<int, KG::CH>{});
    copy_part(rb + C::R_KS, a.k_cache, a.k_bstride, a.k_dsec, sl,
              std::integral_constant<int, KG::SROW>{},
              std::integral_constant<int, (KG::SCH > 0 ? KG::SCH : 1)>{});
    copy_part(rb + C::R_V, a.v_cache, a.v_bstride, 0, sl, std::integral_constant<int, VG::ROW>{},
              std::integral_constant<int, VG::CH>{});
    copy_part(rb + C::R_VS, a.v_cache, a.v_bstride, a.v_dsec, sl,
              std::integral_constant<int, VG::SROW>{},
              std::integral_constant<int, (VG::SCH > 0 ? VG::SCH : 1)>{});
    if (tid < C::TOK) {
      int64_t blk, rr;
      vrow_s[b * C::TOK + tid] = row_src(sl * C::TOK + tid, blk, rr) ? 1 : 0;
    }
  };

  // ---- pipeline over the slabs: copy slab k + 1 while slab k is used
  if (slab_begin < slab_end) issue(slab_begin, 0);
  cp_async_commit();
  const int rw = (warp / DS) * 16;   // this warp's 16 rows
  const int dh = warp % DS;          // its share of the output dims
  const float scale = a.score_scale;
  for (int sl = slab_begin; sl < slab_end; ++sl) {
    const int b = (sl - slab_begin) & 1;
    if (sl + 1 < slab_end) issue(sl + 1, b ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();  // slab sl staged by every thread; the planes are free
#pragma unroll
    for (int u = 0; u < C::NSUB; ++u) {  // dequantize both sides into the operand planes
      const uint8_t* rb = raw + b * C::RAW;
      constexpr int TPR = HD / EPT;  // threads per row
      const int row = u * 16 + tid / TPR, d0 = (tid % TPR) * EPT;
      uint32_t hw[EPT / 2], lw[EPT / 2];
      pf_dequant<KS, HD, EPT>(rb + row * C::KROW, rb + C::R_KS + row * C::KSROW, d0, lv, lv + 16,
                              hw, lw);
#pragma unroll
      for (int i = 0; i < EPT / 2; ++i) {
        *reinterpret_cast<uint32_t*>(kh_s + row * PITCH + d0 + 2 * i) = hw[i];
        if constexpr (KP::PLANES == 2) *reinterpret_cast<uint32_t*>(kl_s + row * PITCH + d0 + 2 * i) = lw[i];
      }
      pf_dequant<VS, HD, EPT>(rb + C::R_V + row * C::VROW, rb + C::R_VS + row * C::VSROW, d0,
                              lv + 32, lv + 48, hw, lw);
#pragma unroll
      for (int i = 0; i < EPT / 2; ++i) {
        *reinterpret_cast<uint32_t*>(vh_s + row * PITCH + d0 + 2 * i) = hw[i];
        if constexpr (VP::PLANES == 2) *reinterpret_cast<uint32_t*>(vl_s + row * PITCH + d0 + 2 * i) = lw[i];
      }
    }
    __syncthreads();

#pragma unroll 1
    for (int u = 0; u < C::NSUB; ++u) {  // 16-token sub-slabs
      // ---- S = Q . K^T for this warp's 16 rows and the slab's 16 positions
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const uint16_t* qa = qh_s + (rw + (lane & 15)) * PITCH + (lane >> 4) * 8;
        const uint16_t* qb = ql_s + (rw + (lane & 15)) * PITCH + (lane >> 4) * 8;
        const int krow = (lane & 7) + ((lane >> 4) << 3), kofs = ((lane >> 3) & 1) * 8;
  #pragma unroll
        for (int j = 0; j < HD / 16; ++j) {
          uint32_t ah[4], al[4], bk[4];
          tc::ldsm_x4(ah, qa + j * 16);
          tc::ldsm_x4(al, qb + j * 16);
          tc::ldsm_x4(bk, kh_s + (u * 16 + krow) * PITCH + j * 16 + kofs);
          tc::mma<KP::BF>(sc[0], ah[0], ah[1], ah[2], ah[3], bk[0], bk[1]);
          tc::mma<KP::BF>(sc[1], ah[0], ah[1], ah[2], ah[3], bk[2], bk[3]);
          tc::mma<KP::BF>(sc[0], al[0], al[1], al[2], al[3], bk[0], bk[1]);
          tc::mma<KP::BF>(sc[1], al[0], al[1], al[2], al[3], bk[2], bk[3]);
          if constexpr (KP::PLANES == 2) {
            uint32_t bl[4];
            tc::ldsm_x4(bl, kl_s + (u * 16 + krow) * PITCH + j * 16 + kofs);
            tc::mma<KP::BF>(sc[0], ah[0], ah[1], ah[2], ah[3], bl[0], bl[1]);
            tc::mma<KP::BF>(sc[1], ah[0], ah[1], ah[2], ah[3], bl[2], bl[3]);
          }
        }
      }
      // ---- mask (causal, window, invalid rows) and online softmax
      const uint8_t* vr = vrow_s + b * C::TOK + u * 16;
      float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
  #pragma unroll
      for (int h = 0; h < 2; ++h) {          // rows g, g + 8
        const int r = rw + g + 8 * h;
        const int qi = r / rp;
        const int p = pbase + qi;
        const bool row_ok = qi < nq_tile && (r - qi * rp) < a.rep;
        const int lo_p = a.window > 0 ? p + 1 - a.window : 0;
  #pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
  #pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int tk = nt * 8 + 2 * c + e;
            const int t = sl * C::TOK + u * 16 + tk;
            const bool ok = row_ok && t <= p && t >= lo_p && vr[tk];
            float& v = sc[nt][2 * h + e];
            v = ok ? v * scale : -CUDART_INF_F;
            mx[h] = fmaxf(mx[h], v);
          }
        }
      }
  #pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      }
      float pr[2][4];
      float al_[2];
  #pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float mn = fmaxf(m[h], mx[h]);
        al_[h] = mn == -CUDART_INF_F ? 1.f : exp2f(m[h] - mn);
  #pragma unroll
        for (int nt = 0; nt < 2; ++nt)
  #pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float v = sc[nt][2 * h + e];
            pr[nt][2 * h + e] = (mn == -CUDART_INF_F || v == -CUDART_INF_F) ? 0.f : exp2f(v - mn);
          }
        l[h] = l[h] * al_[h] + (pr[0][2 * h] + pr[0][2 * h + 1]) + (pr[1][2 * h] + pr[1][2 * h + 1]);
        m[h] = mn;
      }
  #pragma unroll
      for (int i = 0; i < NDT; ++i) {
        o[i][0] *= al_[0]; o[i][1] *= al_[0]; o[i][2] *= al_[1]; o[i][3] *= al_[1];
      }
      // ---- O += P . V (P from the S accumulators: the m16n8 C layout of two
      // n-tiles is the m16k16 A layout)
      uint32_t ph[4], pl[4];
      tc::split2<VP::BF>(pr[0][0], pr[0][1], ph[0], pl[0]);
      tc::split2<VP::BF>(pr[0][2], pr[0][3], ph[1], pl[1]);
      tc::split2<VP::BF>(pr[1][0], pr[1][1], ph[2], pl[2]);
      tc::split2<VP::BF>(pr[1][2], pr[1][3], ph[3], pl[3]);
      {
        const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8, vofs = (lane >> 4) * 8;
  #pragma unroll
        for (int i = 0; i < NDT; i += 2) {
          const int d = dh * (HD / DS) + i * 8;
          uint32_t bv[4];
          tc::ldsm_x4_t(bv, vh_s + (u * 16 + vrow) * PITCH + d + vofs);
          tc::mma<VP::BF>(o[i], ph[0], ph[1], ph[2], ph[3], bv[0], bv[1]);
          tc::mma<VP::BF>(o[i + 1], ph[0], ph[1], ph[2], ph[3], bv[2], bv[3]);
          tc::mma<VP::BF>(o[i], pl[0], pl[1], pl[2], pl[3], bv[0], bv[1]);
          tc::mma<VP::BF>(o[i + 1], pl[0], pl[1], pl[2], pl[3], bv[2], bv[3]);
          if constexpr (VP::PLANES == 2) {
            uint32_t bw[4];
            tc::ldsm_x4_t(bw, vl_s + (u * 16 + vrow) * PITCH + d + vofs);
            tc::mma<VP::BF>(o[i], ph[0], ph[1], ph[2], ph[3], bw[0], bw[1]);
            tc::mma<VP::BF>(o[i + 1], ph[0], ph[1], ph[2], ph[3], bw[2], bw[3]);
          }
        }
      }
    }
  }
  cp_async_wait<0>();

  // ---- normalise, stage the rows in shared memory, rotate back, store
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
  }
  __syncthreads();  // every warp is done with the planes
  float* os = reinterpret_cast<float*>(smem);   // [ROWS][HD + 4]
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float inv = l[h] > 0.f ? a.v_mult / l[h] : 0.f;
    const int r = rw + g + 8 * h;
#pragma unroll
    for (int i = 0; i < NDT; ++i) {
      const int d = dh * (HD / DS) + i * 8 + 2 * c;
      os[r * (HD + 4) + d] = o[i][2 * h] * inv;
      os[r * (HD + 4) + d + 1] = o[i][2 * h + 1] * inv;
    }
  }
  __syncthreads();
  for (int r = warp; r < C::ROWS; r += NW) {
    const int qi = r / rp, hj = r - qi * rp;
    if (qi >= nq_tile || hj >= a.rep) continue;   // warp-uniform
    float x[E];
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] = os[r * (HD + 4) + lane * E + i];
    if constexpr (side_rotated(VS)) fwht_warp<E>(x, lane, a.inv_sqrt_hd);
    const int64_t o_ = ((int64_t)(q0 + t0 + qi) * a.nq + kvh * a.rep + hj) * HD + lane * E;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if (a.out_bf16) reinterpret_cast<uint16_t*>(a.out)[o_ + i] = bf16_bits_from_float(x[i]);
      else reinterpret_cast<float*>(a.out)[o_ + i] = x[i];
    }
  }
}

template <int KS, int VS, int HD>
cudaError_t launch_prefill_inst(const PrefillArgs& a, const Codebooks& cb, int max_chunk,
                                cudaStream_t st) {
  using C = PfCfg<KS, VS, HD>;
  static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
  auto kern = prefill_tc_kernel<KS, VS, HD>;
  if (C::SMEM > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
  }
  const int qt = C::ROWS / a.rp;
  dim3 grid((max_chunk + qt - 1) / qt, a.nkv, a.num_seqs);
  kern<<<grid, C::NT, C::SMEM, st>>>(a, cb);
  return cudaGetLastError();
}

}  // namespace kvq
