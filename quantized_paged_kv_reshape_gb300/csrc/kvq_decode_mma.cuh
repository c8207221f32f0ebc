// Paged decode attention on tensor cores, one kernel launch.
//
// Computes "combs_models/kv.rs" attend (scores, softmax, P.V) with
// repeat_kv for one query per sequence over the pages of its block table,
// with the "spark_runtime/kv_cache.rs" is_wht_rotated bookends: q is rotated
// forward when K is stored rotated and the output back when V is.
//
// Work split.  The (sequence, kv head) rows, laid end to end in 16-token
// slabs, are cut into one equal stretch per persistent CTA (two per SM);
// the NW warps of a CTA take slabs w, w+NW, ... of a stretch, each with a
// private cp.async ring, and are merged through shared memory.  A row cut by
// CTA boundaries leaves one partial (m, l, acc) per CTA in the workspace;
// the last CTA to finish the row merges them (online-softmax identity),
// normalises, rotates back and stores the output.
//
// Per warp and per slab of 16 token positions:
//   S^T[16 tok x 8 cols] = K[16 x hd] . Q^T[hd x 8]      (m16n8k16, hd/16 steps)
//   online softmax on the fp32 accumulators (exp2 domain)
//   O^T[hd x 8] += V^T[hd x 16 tok] . P^T[16 x 8]        (hd/16 m-tiles)
// The query and P operands are split into hi + lo 16-bit parts, so the
// products carry ~16 significant bits: a single 16-bit pass misses the 2e-3
// output bound on outlier-heavy inputs.  With at most 4 query heads per kv
// head the lo parts ride in the otherwise idle columns 4-7 and are added to
// columns 0-3 by one shuffle; with more, they take a second MMA.  P^T's
// operand fragments come from the S accumulators by an in-register 8x8
// transpose (movmatrix).
// Operands by side: BF16 rows through ldmatrix (.trans for V); FP8 E4M3
// converted in registers (K's reduction dimension permuted per thread so
// that each thread converts whole 16-byte chunks, V's bytes of two tokens
// interleaved with prmt); Turbo2/3/4 codes through a shared-memory LUT of
// code pairs whose levels are split into two 7-bit parts, exact in fp16 when
// multiplied by an E4M3 group scale (K: scale applied per 16-dim k-step to
// the fp32 products; V: folded into the operand); Turbo8 E4M3 data with its
// BF16 group scale applied to the products (K) or to P (V).
// Positions outside the attended range or with a bad block id are
// zero-filled and masked to -inf.
#pragma once

#include <math_constants.h>

#include <type_traits>

#include "kvq_decode_common.cuh"

namespace kvq {

namespace tc {

template <bool BF>
__device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                    uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (BF)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(s));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(s));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

// (lo, hi) -> packed 16-bit pair, round to nearest even.
template <bool BF>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (BF)
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
template <bool BF>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  if constexpr (BF) {
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
  } else {
    __half2_raw h;
    h.x = (unsigned short)(v & 0xffffu);
    h.y = (unsigned short)(v >> 16);
    return __half22float2(__half2(h));
  }
}
// x = hi + lo with hi, lo 16-bit: ~16 significant bits in total.
template <bool BF>
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack2<BF>(x0, x1);
  const float2 h = unpack2<BF>(hi);
  lo = pack2<BF>(x0 - h.x, x1 - h.y);
}
// x rounded to 7 significant bits (round to nearest even on the fp32 bits);
// exact in fp16 for the magnitudes used here.
__device__ __forceinline__ float round_sig7(float x) {
  const uint32_t b = __float_as_uint(x);
  const uint32_t r = (b + 0xffffu + ((b >> 17) & 1u)) & ~0x1ffffu;
  return __uint_as_float(r);
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t lo16) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"((unsigned short)lo16));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

}  // namespace tc

// Per-side layout of the staged rows of one slab (16 positions).  Row
// strides are chosen so that the fragment loads of one warp touch distinct
// banks (see the access pattern of each side in decode_tc_kernel).
template <int S, int HD>
struct TcSide {
  static constexpr bool BF = S == S_BF16;                  // bf16 MMA operands (else fp16)
  static constexpr bool CB = side_codebook(S);              // codes through the pair LUT
  static constexpr bool GS = side_scale_bytes(S) > 0;       // per-16 group scales
  static constexpr int BITS = side_bits(S);
  static constexpr int ROW = SideGeom<S, HD>::ROW;          // data bytes per row
  static constexpr int SROW = SideGeom<S, HD>::SROW;        // scale bytes per row
  static constexpr int CH = ROW % 16 == 0 ? 16 : 8;         // copy chunk of data rows
  static constexpr int SCH = SROW == 0 ? 0 : (SROW >= 16 ? 16 : SROW);
  static constexpr int KRS =
      S == S_BF16 ? ROW + 16
      : S == S_FP8 ? (ROW % 128 == 0 ? ROW + 64 : ROW)
      : S == S_T8 || S == S_T4 || S == S_NVFP4 ? ROW + 16
      : S == S_T3 ? (HD == 256 ? ROW + 16 : ROW)
      : /* T2 */ (HD == 64 ? ROW : ROW + 16);
  static constexpr int VRS =
      S == S_BF16 ? ROW + 16
      : S == S_FP8 ? (HD == 64 ? 80 : HD == 128 ? 144 : ROW + 16)
      : S == S_T8 || S == S_T4 || S == S_NVFP4 ? ROW + 16
      : S == S_T3 ? (HD == 256 ? ROW + 16 : ROW)
      : /* T2 */ (HD == 64 ? ROW : ROW + 16);
  static constexpr int LUT_BYTES = CB ? (1 << (2 * code_bits(S))) * 16 * 8 : 0;
};

// Warps per CTA (measured on GB300): 8 for head_dim <= 128 except BF16 K
// (16 warps per SM hide the dependent MMA / LUT chains; one codebook LUT per
// CTA serves more warps), 4 for BF16 K (its 8.5 KB slabs need the shared
// memory for pipeline depth) and for head_dim 256 (accumulators exceed the
// 128-register budget of 16 warps per SM).
#ifndef KVQ_TC_NW_CB
#define KVQ_TC_NW_CB 8
#endif
#ifndef KVQ_TC_NW_RAW
#define KVQ_TC_NW_RAW 8
#endif
#ifndef KVQ_TC_NW_BF16
#define KVQ_TC_NW_BF16 4
#endif
#ifndef KVQ_TC_NST_MAX
#define KVQ_TC_NST_MAX 6
#endif
#ifndef KVQ_TC_CPS_BF16
#define KVQ_TC_CPS_BF16 2
#endif
template <int KS, int VS, int HD>
struct TcWarps {
  static constexpr bool CBS = side_codebook(KS) || side_codebook(VS);
  static constexpr int NW = HD > 128 ? 4 : CBS ? KVQ_TC_NW_CB : (KS == S_BF16 ? KVQ_TC_NW_BF16 : KVQ_TC_NW_RAW);
};

template <int KS, int VS, int HD>
struct TcCfg {
  static constexpr int NW = TcWarps<KS, VS, HD>::NW;
  using K = TcSide<KS, HD>;
  using V = TcSide<VS, HD>;
  static constexpr int NK = HD / 16;
  // token positions per warp iteration: one 16-row MMA tile (32-row
  // iterations measured slower on GB300: fewer pipeline stages fit and the
  // register budget spills)
  static constexpr int SLAB = 16;
  static constexpr int NH = SLAB / 16;
  // stage: [K rows][K scale rows][V rows][V scale rows], SLAB rows each
  static constexpr int OFF_KS = SLAB * K::KRS;
  static constexpr int OFF_V = OFF_KS + SLAB * K::SROW;
  static constexpr int OFF_VS = OFF_V + SLAB * V::VRS;
  static constexpr int STAGE = (OFF_VS + SLAB * V::SROW + 15) / 16 * 16;
  static constexpr bool SHARE_LUT = K::CB && V::CB && KS == VS;
  static constexpr int LUTS = K::LUT_BYTES + (SHARE_LUT ? 0 : V::LUT_BYTES);
  static constexpr int MAXP = 512;                             // pages staged per stretch
  static constexpr int OFF_BLK = 8 * HD * 4;                   // after q_s [8][HD] fp32
  static constexpr int OFF_OFFS = OFF_BLK + MAXP * 4;          // int32 block ids of a stretch
  static constexpr int OFF_SCAN = OFF_OFFS + NW * 128 * 8;     // per-warp row offsets
  static constexpr int OFF_STATE = OFF_SCAN + 16 * 8;          // partition scan / merge scratch
  static constexpr int OFF_LUT = OFF_STATE + 8 * 8;            // CTA loop state
  static constexpr int OFF_RING = OFF_LUT + LUTS;
  // CTAs per SM: BF16 K (light per-slab work, latency bound per warp) runs
  // KVQ_TC_CPS_BF16 CTAs with shallower rings, the others two.
  static constexpr int CPS = (KS == S_BF16 && HD <= 128) ? KVQ_TC_CPS_BF16 : 2;
  static constexpr int BUDGET = (228 - CPS) * 1024 / CPS - OFF_RING;
  static constexpr int NST0 = BUDGET / (NW * STAGE);
  static constexpr int NST = NST0 > KVQ_TC_NST_MAX ? KVQ_TC_NST_MAX : (NST0 < 2 ? 2 : NST0);
  static constexpr int RING = NW * NST * STAGE;
  static constexpr int MERGE = NW * 8 * HD * 4 + NW * 8 * 2 * 4;
  static constexpr int SMEM = OFF_RING + (RING > MERGE ? RING : MERGE);
};

// Dims carried by the B fragment of k-step j for thread c: b0b1 = (d0, d1),
// b2b3 = (d2, d3).  BF16: natural ldmatrix order.  FP8: K's reduction
// dimension permuted so that thread c converts whole 16-byte chunks.
// Group-scaled sides: k-step j is the scale group j, thread c takes its
// dims 4c .. 4c+3.
template <int S, int HD>
__device__ __forceinline__ void k_slot_dims(int j, int c, int (&d)[4]) {
  if constexpr (S == S_BF16) {
    const int b = 16 * j + 2 * c;
    d[0] = b; d[1] = b + 1; d[2] = b + 8; d[3] = b + 9;
  } else if constexpr (S == S_FP8) {
    const int b = 16 * (4 * (j / 4) + c) + 4 * (j % 4);
    d[0] = b; d[1] = b + 1; d[2] = b + 2; d[3] = b + 3;
  } else {
    const int b = 16 * j + 4 * c;
    d[0] = b; d[1] = b + 1; d[2] = b + 2; d[3] = b + 3;
  }
}

// Output dim of accumulator row `row` (0..15) of m-tile i.
template <int S, int HD>
__device__ __forceinline__ int v_row_dim(int i, int row) {
  if constexpr (S == S_BF16) {
    return 16 * i + row;
  } else if constexpr (S == S_FP8) {
    constexpr int DPT = HD / 8;  // dims per thread group g
    return (row & 7) * DPT + 2 * i + (row >> 3);
  } else {  // group-scaled: rows g, g+8 of m-tile i are dims 16i + 2g, 16i + 2g + 1
    return 16 * i + 2 * (row & 7) + (row >> 3);
  }
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t v) {
  __half2_raw h;
  h.x = (unsigned short)(v & 0xffffu);
  h.y = (unsigned short)(v >> 16);
  return __half22float2(__half2(h));
}

// Group scale g of a staged scale row (E4M3 for Turbo2/3/4, BF16 for Turbo8).
template <int S>
__device__ __forceinline__ float tc_group_scale(const uint8_t* srow, int g) {
  if constexpr (S == S_T8)
    return bf16_bits_to_float(*reinterpret_cast<const uint16_t*>(srow + 2 * g));
  else
    return e4m3_to_float(srow[g]);
}

// Code pair (dims 2k, 2k+1 of one token, low code = first dim) starting at
// bit `bit` of a staged code row.
template <int B>
__device__ __forceinline__ uint32_t code_pair(const uint8_t* row, int bit) {
  if constexpr (B == 4) {
    return row[bit >> 3];
  } else if constexpr (B == 2) {
    return ((uint32_t)row[bit >> 3] >> (bit & 7)) & 15u;
  } else {  // 3-bit codes: a 6-bit field that may straddle two bytes
    const uint32_t w = (uint32_t)row[bit >> 3] | ((uint32_t)row[(bit >> 3) + 1] << 8);
    return (w >> (bit & 7)) & 63u;
  }
}

// Pair LUT entry: (hi(c0), hi(c1)) and (lo(c0), lo(c1)) as fp16x2, copy
// lane & 15 so that a half-warp's 8-byte loads fall in distinct banks.
__device__ __forceinline__ uint2 lut_pair(const uint2* lut, uint32_t pair, int lane) {
  return lut[pair * 16 + (lane & 15)];
}

// P^T operand of m16n8k16 from this thread's S^T accumulators (rows g,
// g+8, columns 2c, 2c+1): b[0], b[1] carry the hi parts (k rows 0-7, 8-15)
// and b[2], b[3] the lo parts.  PK: lanes c < 2 (columns 0-3) contribute
// hi parts and lanes c >= 2 (columns 4-7) lo parts, so b[0], b[1] carry
// both and b[2], b[3] are unused.
template <bool BF, bool PK>
__device__ __forceinline__ void p_operand(float p00, float p01, float p10, float p11, int c,
                                          uint32_t (&b)[4]) {
  uint32_t x1h, x1l, x2h, x2l;
  tc::split2<BF>(p00, p01, x1h, x1l);
  tc::split2<BF>(p10, p11, x2h, x2l);
  if constexpr (PK) {
    b[0] = tc::movm_t(c < 2 ? x1h : x1l);
    b[1] = tc::movm_t(c < 2 ? x2h : x2l);
    b[2] = b[3] = 0u;
  } else {
    b[0] = tc::movm_t(x1h);
    b[1] = tc::movm_t(x2h);
    b[2] = tc::movm_t(x1l);
    b[3] = tc::movm_t(x2l);
  }
}

template <int KS, int VS, int HD, bool PK>
__global__ void __launch_bounds__(32 * TcWarps<KS, VS, HD>::NW, 2)
decode_tc_kernel(const DecodeArgs a, const Codebooks cb) {
  using C = TcCfg<KS, VS, HD>;
  constexpr int NW = C::NW;
  constexpr int NT = 32 * NW;
  using KT = typename C::K;
  using VT = typename C::V;
  constexpr int NK = C::NK;
  constexpr int E = HD / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  float* q_s = reinterpret_cast<float*>(smem);
  uint8_t* rings = smem + C::OFF_RING;
  const uint2* lut_k = reinterpret_cast<const uint2*>(smem + C::OFF_LUT);
  const uint2* lut_v = reinterpret_cast<const uint2*>(smem + C::OFF_LUT + (C::SHARE_LUT ? 0 : KT::LUT_BYTES));

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  constexpr int SLAB = C::SLAB;
  const int bs = a.bs;
  const int lbs = 31 - __clz(bs);  // block_size is a power of two
  const int nkv = a.nkv;
  const int64_t cap = (int64_t)a.max_blocks * bs;  // positions the block table covers
  uint8_t* ring = rings + warp * C::NST * C::STAGE;
  int* blk_s = reinterpret_cast<int*>(smem + C::OFF_BLK);
  int64_t* offs = reinterpret_cast<int64_t*>(smem + C::OFF_OFFS) + warp * 128;
  int64_t* scan_s = reinterpret_cast<int64_t*>(smem + C::OFF_SCAN);

  // Attended positions [lo, len) of sequence s and the 16-token slabs
  // [first, first + n) that hold them.
  auto seq_slabs = [&](int s, int& first, int& n, int& lo_, int& len) {
    len = a.seq_lens[s];
    if (len > cap) len = (int)cap;
    if (len <= 0) {
      first = n = lo_ = len = 0;
      return;
    }
    lo_ = a.window > 0 ? max(0, len - a.window) : 0;
    first = lo_ >> 4;
    n = ((len + 15) >> 4) - first;
  };

  // ---- Partition.  Each kv head gets R = gridDim.x / nkv CTAs (the host
  // launches a multiple of nkv).  The sequences' 16-token slabs are laid end
  // to end (S in all); CTA (h, j) takes slabs [j * cpc, (j + 1) * cpc) of
  // kv head h, cpc about ceil(S / R) (see below), so every CTA gets the same
  // amount of work whatever the lengths, and the CTAs of the different kv
  // heads read the same token positions at the same time (their rows share
  // DRAM sectors, the scale rows especially).  A (sequence, kv head) row cut
  // by CTA boundaries leaves one partial per CTA, in slot (j - first j of
  // the row).
  const int N = a.num_seqs;
  const int R = gridDim.x / nkv;
  const int kvh = blockIdx.x / R, jr = blockIdx.x - kvh * R;
  const int chunk = (N + NT - 1) / NT;
  const int s_beg = min(N, tid * chunk), s_end = min(N, s_beg + chunk);
  int64_t mine = 0;
  int longest = 0;
  for (int s = s_beg; s < s_end; ++s) {
    int f, n, l_, e_;
    seq_slabs(s, f, n, l_, e_);
    mine += n;
    longest = max(longest, n);
    if (blockIdx.x == 0 && a.seq_lens[s] > cap && a.err) atomicOr(a.err, 2);
  }
  int64_t incl = mine;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
    longest = max(longest, __shfl_xor_sync(0xffffffffu, longest, d));
  }
  if (lane == 31) scan_s[warp] = incl;
  if (lane == 0) scan_s[8 + warp] = longest;
  __syncthreads();
  int64_t before = 0, total = 0, max_n = 0;
  for (int w2 = 0; w2 < NW; ++w2) {
    const int64_t v = scan_s[w2];
    if (w2 < warp) before += v;
    total += v;
    max_n = max(max_n, scan_s[8 + w2]);
  }
  const int64_t excl = before + incl - mine;  // slabs before this thread's chunk
  // Slabs per CTA: an equal share of a virtual line on which each sequence
  // is preceded by U slabs standing for the cost of a unit (sequence s spans
  // [P_s + U s, P_s + U s + U + n_s), P_s = attended slabs before it), so
  // that a CTA that works on more sequences takes fewer slabs; never so few
  // that a row of max_n slabs spans more than kmax CTAs (the partial slots
  // the host sized): a row of n slabs spans at most floor((n - 1) / cpc) + 2
  // CTAs.  U = kUnitSlabs for the K sides without a code table; a codebook K
  // side's slabs take several times longer here, so a unit costs few of them
  // and U = 0 (measured on GB300, 16 x 8192, head_dim 256: Turbo8 259 ->
  // 255 us with U = 48, Turbo2 288 -> 303 us).
  constexpr int64_t U = side_codebook(KS) ? 0 : kUnitSlabs;
  const int64_t totalv = total + U * N;
  int64_t cpc = (totalv + R - 1) / R;
  if (a.kmax > 1) cpc = max(cpc, (max_n + a.kmax - 2) / (a.kmax - 1));
  if (cpc < 1) cpc = 1;
  const int64_t v0 = (int64_t)jr * cpc, v1 = min(v0 + cpc, totalv);
  __syncthreads();  // scan_s is reused below
  {   // the real slab indices of v0 and v1 (scan_s[2], [3])
    int64_t P = excl;
    for (int s = s_beg; s < s_end; ++s) {
      int f, n, l_, e_;
      seq_slabs(s, f, n, l_, e_);
      const int64_t vp = P + U * s;
      if (v0 >= vp && v0 < vp + U + n) scan_s[2] = P + min(max(v0 - vp - U, (int64_t)0), (int64_t)n);
      if (v1 >= vp && v1 < vp + U + n) scan_s[3] = P + min(max(v1 - vp - U, (int64_t)0), (int64_t)n);
      P += n;
    }
  }
  __syncthreads();
  const int64_t x0 = v0 < totalv ? scan_s[2] : total;
  const int64_t x_end = v1 < totalv ? scan_s[3] : total;
  if (blockIdx.x == 0) {  // sequences with nothing to attend get zero rows
    for (int s = s_beg; s < s_end; ++s) {
      int f, n, l_, e_;
      seq_slabs(s, f, n, l_, e_);
      if (n > 0) continue;
      for (int i = 0; i < a.nq * HD; ++i) {
        const int64_t o_ = (int64_t)s * a.nq * HD + i;
        if (a.out_bf16) reinterpret_cast<uint16_t*>(a.out)[o_] = 0;
        else reinterpret_cast<float*>(a.out)[o_] = 0.f;
      }
    }
  }
  if (kvh < nkv && x0 < total && excl <= x0 && x0 < excl + mine) {  // the chunk holding x0
    int64_t P = excl;
    for (int s = s_beg; s < s_end; ++s) {
      int f, n, l_, e_;
      seq_slabs(s, f, n, l_, e_);
      if (x0 < P + n) {
        scan_s[0] = s;
        scan_s[1] = x0 - P;
        break;
      }
      P += n;
    }
  }
  __syncthreads();
  if (kvh >= nkv || x0 >= total) return;
  int seq = (int)scan_s[0];
  int64_t off = scan_s[1];

  // Pair LUTs of the codebook sides: entry p = (code of dim 2k) | (code of
  // dim 2k+1) << b holds fp16 (hi, hi) and (lo, lo) where hi and lo carry 7
  // significant bits each and level = hi + lo to ~2^-16 relative.  With 7
  // bits, hi and lo times an E4M3 group scale (4 significant bits) are exact
  // in fp16, which lets the V operand absorb its group scale.  Filled once
  // per CTA.
  auto fill_lut = [&](uint2* lut, const float* lv, int bits) {
    const int n = 1 << bits;
    for (int e = tid; e < n * n * 16; e += NT) {
      const int pr = e >> 4;
      const float c0 = lv[pr & (n - 1)], c1 = lv[pr >> bits];
      const float h0 = tc::round_sig7(c0), h1 = tc::round_sig7(c1);
      const float l0 = tc::round_sig7(c0 - h0), l1 = tc::round_sig7(c1 - h1);
      lut[e] = make_uint2(tc::pack2<false>(h0, h1), tc::pack2<false>(l0, l1));
    }
  };
  if constexpr (KT::CB)
    fill_lut(reinterpret_cast<uint2*>(smem + C::OFF_LUT), side_levels<KS>(cb), code_bits(KS));
  if constexpr (VT::CB && !C::SHARE_LUT)
    fill_lut(reinterpret_cast<uint2*>(smem + C::OFF_LUT + KT::LUT_BYTES), side_levels<VS>(cb),
             code_bits(VS));

  // State of the current stretch: attended positions [lo, tok_end), slabs
  // from tok0, block ids of pages p0 .. staged in blk_s.
  int lo = 0, tok_end = 0, tok0 = 0, p0 = 0;
  int64_t tab = 0;

  // Block id of position pos, or -1 if it is not attended / not valid.
  auto pos_block = [&](int pos) -> int {
    if (pos < lo || pos >= tok_end) return -1;
    return blk_s[(pos >> lbs) - p0];
  };

  // Per slab, lanes 0-15 compute the source byte offsets of the K data and
  // K scale rows of position t = lane, lanes 16-31 those of the V rows (-1
  // for positions not attended); then four copy loops move the rows in
  // chunks, consecutive lanes on consecutive chunks of a row.
  auto copy_rows = [&](uint8_t* dst, int dst_stride, const uint8_t* base, const int64_t* tbl,
                       auto rowbytes_c, auto chunk_c) {
    constexpr int RB = decltype(rowbytes_c)::value, CHB = decltype(chunk_c)::value;
    constexpr int NC = RB / CHB, TOT = SLAB * NC;
#pragma unroll
    for (int k = 0; k < (TOT + 31) / 32; ++k) {
      const int q = lane + 32 * k;
      if (TOT % 32 == 0 || q < TOT) {
        const int row = q / NC, ch = q - row * NC;
        const int64_t o_ = tbl[row];
        const bool ok = o_ >= 0;
        cp_async<CHB>(dst + row * dst_stride + ch * CHB, base + (ok ? o_ : 0) + ch * CHB, ok);
      }
    }
  };
  // Fast path of a slab whose 16 positions are all attended and lie in one
  // page (block_size >= 16) or two (block_size 8), both valid: the rows of
  // one (side, kv head) are nkv * row-bytes apart inside a page, so each lane
  // forms its chunks' source addresses directly from the page base.
  auto copy_fast = [&](uint8_t* dst, int dst_stride, const uint8_t* cache, int64_t bstride,
                       int64_t sec, int slab_pos, int ba, int bb, auto rowbytes_c, auto chunk_c) {
    constexpr int RB = decltype(rowbytes_c)::value, CHB = decltype(chunk_c)::value;
    constexpr int NC = RB / CHB, RPI = 32 / NC, PASSES = (SLAB + RPI - 1) / RPI;
    const int r0 = lane / NC, ch = lane - r0 * NC;
    const int64_t rowstep = (int64_t)nkv * RB;
#pragma unroll
    for (int k = 0; k < PASSES; ++k) {
      const int row = r0 + RPI * k;
      if (RPI * PASSES == SLAB || row < SLAB) {
        const int64_t blk = row < 8 ? ba : bb;
        const int64_t src = blk * bstride + sec + (int64_t)((slab_pos + row) & (bs - 1)) * rowstep +
                            (int64_t)kvh * RB + ch * CHB;
        cp_async<CHB>(dst + row * dst_stride + ch * CHB, cache + src, true);
      }
    }
  };
  auto issue = [&](int s) {
    __syncwarp();  // the previous issue's reads of offs are done
    uint8_t* sb = ring + (s % C::NST) * C::STAGE;
    const int slab_pos = tok0 + (warp + NW * s) * SLAB;
    constexpr bool FAST = chunks_split_warp(KT::ROW, KT::CH) && chunks_split_warp(VT::ROW, VT::CH) &&
                          chunks_split_warp(KT::SROW, KT::SCH) && chunks_split_warp(VT::SROW, VT::SCH);
    if constexpr (FAST) {
      if (slab_pos >= lo && slab_pos + SLAB <= tok_end) {
        const int ba = blk_s[(slab_pos >> lbs) - p0], bb = blk_s[((slab_pos + 8) >> lbs) - p0];
        if (ba >= 0 && bb >= 0) {   // warp-uniform
          copy_fast(sb, KT::KRS, a.k_cache, a.k_bstride, 0, slab_pos, ba, bb,
                    std::integral_constant<int, KT::ROW>{}, std::integral_constant<int, KT::CH>{});
          if constexpr (KT::SROW > 0)
            copy_fast(sb + C::OFF_KS, KT::SROW, a.k_cache, a.k_bstride, a.k_dsec, slab_pos, ba, bb,
                      std::integral_constant<int, KT::SROW>{}, std::integral_constant<int, KT::SCH>{});
          copy_fast(sb + C::OFF_V, VT::VRS, a.v_cache, a.v_bstride, 0, slab_pos, ba, bb,
                    std::integral_constant<int, VT::ROW>{}, std::integral_constant<int, VT::CH>{});
          if constexpr (VT::SROW > 0)
            copy_fast(sb + C::OFF_VS, VT::SROW, a.v_cache, a.v_bstride, a.v_dsec, slab_pos, ba, bb,
                      std::integral_constant<int, VT::SROW>{}, std::integral_constant<int, VT::SCH>{});
          return;
        }
      }
    }
    const int b = pos_block(slab_pos + lane);
    const int64_t rr = (int64_t)((slab_pos + lane) & (bs - 1)) * nkv + kvh;   // row in block
    const int64_t bk = (int64_t)b * a.k_bstride, bv = (int64_t)b * a.v_bstride;
    if (lane < SLAB) {
      offs[lane] = b < 0 ? -1 : bk + rr * KT::ROW;
      offs[32 + lane] = b < 0 ? -1 : bv + rr * VT::ROW;
      offs[64 + lane] = b < 0 ? -1 : bk + a.k_dsec + rr * KT::SROW;
      offs[96 + lane] = b < 0 ? -1 : bv + a.v_dsec + rr * VT::SROW;
    }
    __syncwarp();
    copy_rows(sb, KT::KRS, a.k_cache, offs, std::integral_constant<int, KT::ROW>{},
              std::integral_constant<int, KT::CH>{});
    if constexpr (KT::SROW > 0)
      copy_rows(sb + C::OFF_KS, KT::SROW, a.k_cache, offs + 64,
                std::integral_constant<int, KT::SROW>{}, std::integral_constant<int, KT::SCH>{});
    copy_rows(sb + C::OFF_V, VT::VRS, a.v_cache, offs + 32, std::integral_constant<int, VT::ROW>{},
              std::integral_constant<int, VT::CH>{});
    if constexpr (VT::SROW > 0)
      copy_rows(sb + C::OFF_VS, VT::SROW, a.v_cache, offs + 96,
                std::integral_constant<int, VT::SROW>{}, std::integral_constant<int, VT::SCH>{});
  };

  // Q^T operand (B column n = g).  PK: column g carries head g & 3, its hi
  // part for g < 4 and its lo part for g >= 4 (qh only); otherwise column g
  // is head g, with the hi and lo parts in separate operands qh, ql.
  uint32_t qh[NK][2], ql[PK ? 1 : NK][2];
  float o[NK][4];
  float m0, m1, l0, l1;
  const float scale = a.score_scale;

  // S^T of the 16 positions whose K rows start at kbh (scale rows at ksbh).
  auto scores16 = [&](const uint8_t* kbh, const uint8_t* ksbh, float (&sout)[4]) {
    // ---- S^T = K . Q^T for the 16 rows at kbh (K rows) / ksbh (K scale rows)
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      float sacl[4] = {0.f, 0.f, 0.f, 0.f};   // second, independent MMA chain
      if constexpr (KS == S_BF16) {
        const int mi = lane >> 3, rr = lane & 7;
        const uint8_t* base = kbh + ((mi & 1) * 8 + rr) * KT::KRS + (mi >> 1) * 16;
#pragma unroll
        for (int j = 0; j < NK; ++j) {
          uint32_t f[4];
          tc::ldsm_x4(f, base + j * 32);
          if constexpr (PK) {
            tc::mma<true>((j & 1) ? sacl : sacc, f[0], f[1], f[2], f[3], qh[j][0], qh[j][1]);
          } else {
            tc::mma<true>(sacc, f[0], f[1], f[2], f[3], qh[j][0], qh[j][1]);
            tc::mma<true>(sacl, f[0], f[1], f[2], f[3], ql[j][0], ql[j][1]);
          }
        }
      } else if constexpr (KS == S_FP8) {  // thread c converts 16-byte chunks 4jj + c of rows g, g+8
#pragma unroll
        for (int jj = 0; jj < NK / 4; ++jj) {
          const uint4 ra = *reinterpret_cast<const uint4*>(kbh + g * KT::KRS + (4 * jj + c) * 16);
          const uint4 rb = *reinterpret_cast<const uint4*>(kbh + (g + 8) * KT::KRS + (4 * jj + c) * 16);
          const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w};
          const uint32_t wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * jj + e;
            const uint32_t a0 = tc::e4m3x2_f16x2(wa[e] & 0xffffu), a4 = tc::e4m3x2_f16x2(wa[e] >> 16);
            const uint32_t a2 = tc::e4m3x2_f16x2(wb[e] & 0xffffu), a6 = tc::e4m3x2_f16x2(wb[e] >> 16);
            if constexpr (PK) {
              tc::mma<false>((e & 1) ? sacl : sacc, a0, a2, a4, a6, qh[j][0], qh[j][1]);
            } else {
              tc::mma<false>(sacc, a0, a2, a4, a6, qh[j][0], qh[j][1]);
              tc::mma<false>(sacl, a0, a2, a4, a6, ql[j][0], ql[j][1]);
            }
          }
        }
      } else {  // group-scaled sides: k-step j is scale group j
        const uint8_t* ra = kbh + g * KT::KRS;
        const uint8_t* rb = kbh + (g + 8) * KT::KRS;
        const uint8_t* sa = ksbh + g * KT::SROW;
        const uint8_t* sbr = ksbh + (g + 8) * KT::SROW;
#pragma unroll
        for (int j = 0; j < NK; ++j) {
          float cg[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (KS == S_T8) {
            const uint32_t wa = *reinterpret_cast<const uint32_t*>(ra + 16 * j + 4 * c);
            const uint32_t wb = *reinterpret_cast<const uint32_t*>(rb + 16 * j + 4 * c);
            const uint32_t a0 = tc::e4m3x2_f16x2(wa & 0xffffu), a4 = tc::e4m3x2_f16x2(wa >> 16);
            const uint32_t a2 = tc::e4m3x2_f16x2(wb & 0xffffu), a6 = tc::e4m3x2_f16x2(wb >> 16);
            tc::mma<false>(cg, a0, a2, a4, a6, qh[j][0], qh[j][1]);
            if constexpr (!PK) tc::mma<false>(cg, a0, a2, a4, a6, ql[j][0], ql[j][1]);
          } else {
            constexpr int B = code_bits(KS);
            const int bit = B * (16 * j + 4 * c);
            uint32_t pa0, pa1, pb0, pb1;   // code pairs (dims 4c,4c+1) and (4c+2,4c+3)
            if constexpr (B == 4) {
              const uint32_t ua = *reinterpret_cast<const uint16_t*>(ra + (bit >> 3));
              const uint32_t ub = *reinterpret_cast<const uint16_t*>(rb + (bit >> 3));
              pa0 = ua & 0xffu; pa1 = ua >> 8; pb0 = ub & 0xffu; pb1 = ub >> 8;
            } else if constexpr (B == 2) {
              const uint32_t ua = ra[bit >> 3], ub = rb[bit >> 3];
              pa0 = ua & 15u; pa1 = ua >> 4; pb0 = ub & 15u; pb1 = ub >> 4;
            } else {
              const int sh = bit & 7;
              const uint32_t ua = ((uint32_t)ra[bit >> 3] | ((uint32_t)ra[(bit >> 3) + 1] << 8)) >> sh;
              const uint32_t ub = ((uint32_t)rb[bit >> 3] | ((uint32_t)rb[(bit >> 3) + 1] << 8)) >> sh;
              pa0 = ua & 63u; pa1 = (ua >> 6) & 63u; pb0 = ub & 63u; pb1 = (ub >> 6) & 63u;
            }
            const uint2 xa0 = lut_pair(lut_k, pa0, lane);
            const uint2 xa1 = lut_pair(lut_k, pa1, lane);
            const uint2 xb0 = lut_pair(lut_k, pb0, lane);
            const uint2 xb1 = lut_pair(lut_k, pb1, lane);
            // level hi and lo parts times q (PK: the lo x q-lo term comes along)
            tc::mma<false>(cg, xa0.x, xb0.x, xa1.x, xb1.x, qh[j][0], qh[j][1]);
            if constexpr (!PK) tc::mma<false>(cg, xa0.x, xb0.x, xa1.x, xb1.x, ql[j][0], ql[j][1]);
            tc::mma<false>(cg, xa0.y, xb0.y, xa1.y, xb1.y, qh[j][0], qh[j][1]);
          }
          float ga, gb;   // group-j scales of rows g and g+8
          if constexpr (KS == S_T8) {
            ga = tc_group_scale<KS>(sa, j);
            gb = tc_group_scale<KS>(sbr, j);
          } else {
            const float2 gs = unpack_f16x2(tc::e4m3x2_f16x2(
                tc::prmt(*reinterpret_cast<const uint32_t*>(sa + (j & ~3)),
                         *reinterpret_cast<const uint32_t*>(sbr + (j & ~3)),
                         (uint32_t)(j & 3) | ((uint32_t)(4 + (j & 3)) << 4))));
            ga = gs.x;
            gb = gs.y;
          }
          float* acc = (j & 1) ? sacl : sacc;   // two independent accumulators
          acc[0] = fmaf(cg[0], ga, acc[0]);
          acc[1] = fmaf(cg[1], ga, acc[1]);
          acc[2] = fmaf(cg[2], gb, acc[2]);
          acc[3] = fmaf(cg[3], gb, acc[3]);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[e] += sacl[e];
      if constexpr (PK) {  // q-hi columns + q-lo columns (lanes c, c ^ 2)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[e] += __shfl_xor_sync(0xffffffffu, sacc[e], 2);
      }

      sout[0] = sacc[0]; sout[1] = sacc[1]; sout[2] = sacc[2]; sout[3] = sacc[3];
  };
  // O^T += V^T . P^T for the 16 positions whose V rows start at vbh (scale
  // rows at vsbh); p00, p01 (row g) and p10, p11 (row g+8) are this
  // thread's weights in the accumulator layout.
  auto pv16 = [&](const uint8_t* vbh, const uint8_t* vsbh, float p00, float p01, float p10,
                  float p11) {
    // ---- O^T += V^T . P^T
      if constexpr (!VT::GS) {
        // P^T operand (hi + lo) from the accumulator layout
        uint32_t b[4];
        p_operand<VT::BF, PK>(p00, p01, p10, p11, c, b);
        const uint32_t b0h = b[0], b1h = b[1], b0l = b[2], b1l = b[3];
        if constexpr (VS == S_BF16) {
          const int mi = lane >> 3, rr = lane & 7;
          const uint8_t* base = vbh + ((mi >> 1) * 8 + rr) * VT::VRS + (mi & 1) * 16;
#pragma unroll
          for (int i = 0; i < NK; ++i) {
            uint32_t f[4];
            tc::ldsm_x4_t(f, base + i * 32);
            tc::mma<true>(o[i], f[0], f[1], f[2], f[3], b0h, b1h);
            if constexpr (!PK) tc::mma<true>(o[i], f[0], f[1], f[2], f[3], b0l, b1l);
          }
        } else {  // FP8: tokens 2c, 2c+1, 2c+8, 2c+9; dims g*DPT .. g*DPT + DPT - 1
          constexpr int DPT = HD / 8;
          constexpr int W = DPT / 4;  // 32-bit words per token
          uint32_t w[4][W];
          const int toks[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint8_t* src = vbh + toks[t] * VT::VRS + g * DPT;
            if constexpr (W == 2) {
              const uint2 v = *reinterpret_cast<const uint2*>(src);
              w[t][0] = v.x; w[t][1] = v.y;
            } else {
#pragma unroll
              for (int q4 = 0; q4 < W / 4; ++q4) {
                const uint4 v = *reinterpret_cast<const uint4*>(src + q4 * 16);
                w[t][4 * q4] = v.x; w[t][4 * q4 + 1] = v.y; w[t][4 * q4 + 2] = v.z; w[t][4 * q4 + 3] = v.w;
              }
            }
          }
#pragma unroll
          for (int i = 0; i < NK; ++i) {
            const int wi = (2 * i) / 4;
            const uint32_t sel = ((2 * i) % 4 == 0) ? 0x5140u : 0x7362u;
            const uint32_t x01 = tc::prmt(w[0][wi], w[1][wi], sel);   // (t0,t1) @ dims 2i, 2i+1
            const uint32_t x23 = tc::prmt(w[2][wi], w[3][wi], sel);   // (t2,t3)
            const uint32_t a0 = tc::e4m3x2_f16x2(x01 & 0xffffu), a2 = tc::e4m3x2_f16x2(x01 >> 16);
            const uint32_t a4 = tc::e4m3x2_f16x2(x23 & 0xffffu), a6 = tc::e4m3x2_f16x2(x23 >> 16);
            tc::mma<false>(o[i], a0, a2, a4, a6, b0h, b1h);
            if constexpr (!PK) tc::mma<false>(o[i], a0, a2, a4, a6, b0l, b1l);
          }
        }
      } else if constexpr (VT::CB) {
        // Codebook V: m-tile i is scale group i.  The operand is (level hi,
        // level lo) x group scale of its token, exact in fp16 (7-bit level
        // parts, 4-bit scale significand), so P is split once per slab.  Rows
        // g, g+8 of m-tile i are dims 16i + 2g, 16i + 2g + 1; k-slots are
        // tokens 2c, 2c+1, 2c+8, 2c+9.
        uint32_t b[4];
        p_operand<false, PK>(p00, p01, p10, p11, c, b);
        const uint32_t b0h = b[0], b1h = b[1], b0l = b[2], b1l = b[3];
        const uint8_t* r0 = vbh + (2 * c) * VT::VRS;
        const uint8_t* r1 = vbh + (2 * c + 1) * VT::VRS;
        const uint8_t* r2 = vbh + (2 * c + 8) * VT::VRS;
        const uint8_t* r3 = vbh + (2 * c + 9) * VT::VRS;
        const uint8_t* vsc = vsbh;
        constexpr int SW = (VT::SROW + 3) / 4;   // 32-bit words of a scale row
        uint32_t s0[SW], s1[SW], s2[SW], s3[SW];
#pragma unroll
        for (int q4 = 0; q4 < SW; ++q4) {
          s0[q4] = *reinterpret_cast<const uint32_t*>(vsc + (2 * c) * VT::SROW + 4 * q4);
          s1[q4] = *reinterpret_cast<const uint32_t*>(vsc + (2 * c + 1) * VT::SROW + 4 * q4);
          s2[q4] = *reinterpret_cast<const uint32_t*>(vsc + (2 * c + 8) * VT::SROW + 4 * q4);
          s3[q4] = *reinterpret_cast<const uint32_t*>(vsc + (2 * c + 9) * VT::SROW + 4 * q4);
        }
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          constexpr int B = code_bits(VS);
          const int bit = B * (16 * i + 2 * g);
          const uint2 e0 = lut_pair(lut_v, code_pair<B>(r0, bit), lane);
          const uint2 e1 = lut_pair(lut_v, code_pair<B>(r1, bit), lane);
          const uint2 e2 = lut_pair(lut_v, code_pair<B>(r2, bit), lane);
          const uint2 e3 = lut_pair(lut_v, code_pair<B>(r3, bit), lane);
          // group scales of the four tokens as fp16 pairs (t0,t1), (t2,t3)
          const uint32_t bsel = (uint32_t)(i & 3) | ((uint32_t)(4 + (i & 3)) << 4);
          const uint32_t sc01 = tc::e4m3x2_f16x2(tc::prmt(s0[i >> 2], s1[i >> 2], bsel));
          const uint32_t sc23 = tc::e4m3x2_f16x2(tc::prmt(s2[i >> 2], s3[i >> 2], bsel));
          // regroup (dim, dim+1) pairs of one token into (token, token) pairs
          const uint32_t h0 = tc::hmul2(tc::prmt(e0.x, e1.x, 0x5410u), sc01);
          const uint32_t h2 = tc::hmul2(tc::prmt(e0.x, e1.x, 0x7632u), sc01);
          const uint32_t h4 = tc::hmul2(tc::prmt(e2.x, e3.x, 0x5410u), sc23);
          const uint32_t h6 = tc::hmul2(tc::prmt(e2.x, e3.x, 0x7632u), sc23);
          const uint32_t l0_ = tc::hmul2(tc::prmt(e0.y, e1.y, 0x5410u), sc01);
          const uint32_t l2_ = tc::hmul2(tc::prmt(e0.y, e1.y, 0x7632u), sc01);
          const uint32_t l4_ = tc::hmul2(tc::prmt(e2.y, e3.y, 0x5410u), sc23);
          const uint32_t l6_ = tc::hmul2(tc::prmt(e2.y, e3.y, 0x7632u), sc23);
          tc::mma<false>(o[i], h0, h2, h4, h6, b0h, b1h);
          if constexpr (!PK) tc::mma<false>(o[i], h0, h2, h4, h6, b0l, b1l);
          tc::mma<false>(o[i], l0_, l2_, l4_, l6_, b0h, b1h);
        }
      } else {
        // Turbo8 V: m-tile i is scale group i; P is scaled per token by its
        // BF16 group scale before the split (E4M3 x BF16 is not exact in
        // fp16).  Rows g, g+8 of m-tile i are dims 16i + 2g, 16i + 2g + 1;
        // k-slots are tokens 2c, 2c+1, 2c+8, 2c+9.
        const uint8_t* vsa = vsbh + g * VT::SROW;
        const uint8_t* vsb = vsbh + (g + 8) * VT::SROW;
        const uint8_t* r0 = vbh + (2 * c) * VT::VRS;
        const uint8_t* r1 = vbh + (2 * c + 1) * VT::VRS;
        const uint8_t* r2 = vbh + (2 * c + 8) * VT::VRS;
        const uint8_t* r3 = vbh + (2 * c + 9) * VT::VRS;
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          const float ga = tc_group_scale<VS>(vsa, i), gb = tc_group_scale<VS>(vsb, i);
          uint32_t b[4];
          p_operand<false, PK>(p00 * ga, p01 * ga, p10 * gb, p11 * gb, c, b);
          const uint32_t b0h = b[0], b1h = b[1], b0l = b[2], b1l = b[3];
          {
            const int off = 16 * i + 2 * g;
            const uint32_t u0 = *reinterpret_cast<const uint16_t*>(r0 + off);
            const uint32_t u1 = *reinterpret_cast<const uint16_t*>(r1 + off);
            const uint32_t u2 = *reinterpret_cast<const uint16_t*>(r2 + off);
            const uint32_t u3 = *reinterpret_cast<const uint16_t*>(r3 + off);
            const uint32_t x01 = tc::prmt(u0, u1, 0x5140u);   // (t0,t1) @ dims 2g, 2g+1
            const uint32_t x23 = tc::prmt(u2, u3, 0x5140u);
            const uint32_t a0 = tc::e4m3x2_f16x2(x01 & 0xffffu), a2 = tc::e4m3x2_f16x2(x01 >> 16);
            const uint32_t a4 = tc::e4m3x2_f16x2(x23 & 0xffffu), a6 = tc::e4m3x2_f16x2(x23 >> 16);
            tc::mma<false>(o[i], a0, a2, a4, a6, b0h, b1h);
            if constexpr (!PK) tc::mma<false>(o[i], a0, a2, a4, a6, b0l, b1l);
          }
        }
      }
  };


  // ---- the units of this CTA's slab range.  The CTA-uniform loop state
  // lives in shared memory (re-read after each barrier), so that the slab
  // loop keeps only what it uses in registers.
  int64_t* st = reinterpret_cast<int64_t*>(smem + C::OFF_STATE);
  // st: 0 x (next slab of the range), 1 x_end, 2 seq, 4 off (slab of the
  // row at x), 5 next stretch, 6 end of the row's slabs here, 7 cpc
  if (tid == 0) {
    st[0] = x0;
    st[1] = x_end;
    st[2] = seq;
    st[4] = off;
    st[7] = cpc;
  }
  for (;;) {
    __syncthreads();  // loop state visible; the previous unit's merge is done
    {
      const int64_t x = st[0];
      if (x >= st[1]) break;
      int first, n, len;
      seq_slabs((int)st[2], first, n, lo, len);
      if (tid == 0) {
        st[5] = first + st[4];
        st[6] = first + st[4] + min((int64_t)n - st[4], st[1] - x);
      }
    }
#pragma unroll
    for (int i = 0; i < NK; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m0 = m1 = -CUDART_INF_F;
    l0 = l1 = 0.f;
    // Stretches of at most MAXP pages (the staged block ids).
    for (int first_stretch = 1;; first_stretch = 0) {
      __syncthreads();  // blk_s, q_s and the rings are free; st[5] visible
      const int64_t sa = st[5], s_hi = st[6];
      if (sa >= s_hi) break;
      const int sq = (int)st[2];
      int first, n, len;
      seq_slabs(sq, first, n, lo, len);
      const int sub = (C::MAXP - 1) * bs / SLAB;
      const int nsl = (int)min((int64_t)sub, s_hi - sa);
      tok0 = (int)(sa * SLAB);
      tok_end = min(tok0 + nsl * SLAB, len);
      p0 = tok0 >> lbs;
      const int p1 = ((tok_end - 1) >> lbs) + 1;
      tab = (int64_t)sq * a.max_blocks;
      // Block ids of the stretch's pages (-1 = outside the pool).
      for (int i = tid; i < p1 - p0; i += NT) {
        const int64_t b = a.block_tables[tab + p0 + i];
        const bool bad = b < 0 || (a.num_blocks > 0 && b >= a.num_blocks);
        if (bad && a.err) atomicOr(a.err, 2);
        blk_s[i] = bad ? -1 : (int)b;
      }
      __syncthreads();
      if (tid == 0) st[5] = sa + nsl;
      const int my = nsl > warp ? (nsl - 1 - warp) / NW + 1 : 0;
#pragma unroll
      for (int s = 0; s < C::NST - 1; ++s) {
        if (s < my) issue(s);
        cp_async_commit();
      }
      // The unit's queries are staged after its first copies are in flight
      // (those need only the block ids), so their loads overlap the copies.
      if (first_stretch) {
        // ---- queries (rotated when K is stored rotated), rows >= rep are zero
        for (int j = warp; j < 8; j += NW) {
          float xq[E];
          if (j < a.rep) {
            const int64_t qoff = (int64_t)sq * a.q_stride + (int64_t)(kvh * a.rep + j) * HD + lane * E;
#pragma unroll
            for (int i = 0; i < E; ++i)
              xq[i] = a.q_bf16 ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(a.q)[qoff + i])
                               : reinterpret_cast<const float*>(a.q)[qoff + i];
            if constexpr (side_rotated(KS)) fwht_warp<E>(xq, lane, a.inv_sqrt_hd);
          } else {
#pragma unroll
            for (int i = 0; i < E; ++i) xq[i] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < E; ++i) q_s[j * HD + lane * E + i] = xq[i];
        }
        __syncthreads();   // q_s visible
      }
      if (first_stretch) {
#pragma unroll
        for (int j = 0; j < NK; ++j) {
          int d[4];
          k_slot_dims<KS, HD>(j, c, d);
          const float* qr = q_s + (PK ? (g & 3) : g) * HD;
          uint32_t h0, lq0, h1, lq1;
          tc::split2<KT::BF>(qr[d[0]], qr[d[1]], h0, lq0);
          tc::split2<KT::BF>(qr[d[2]], qr[d[3]], h1, lq1);
          if constexpr (PK) {
            qh[j][0] = g < 4 ? h0 : lq0;
            qh[j][1] = g < 4 ? h1 : lq1;
          } else {
            qh[j][0] = h0; ql[j][0] = lq0;
            qh[j][1] = h1; ql[j][1] = lq1;
          }
        }
      }
      for (int s = 0; s < my; ++s) {
        cp_async_wait<C::NST - 2>();
        __syncwarp();
        if (s + C::NST - 1 < my) issue(s + C::NST - 1);
        cp_async_commit();
        const uint8_t* sb = ring + (s % C::NST) * C::STAGE;
        const int slab_pos = tok0 + (warp + NW * s) * SLAB;

        // ---- scores of both row tiles; this thread holds rows g, g+8 of each
        constexpr int NH = C::NH;
        float sv[2][4] = {{-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F},
                          {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F}};
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          float sc4[4];
          scores16(sb + 16 * h * KT::KRS, sb + C::OFF_KS + 16 * h * KT::SROW, sc4);
          const bool va = pos_block(slab_pos + 16 * h + g) >= 0;
          const bool vb_ = pos_block(slab_pos + 16 * h + g + 8) >= 0;
          sv[h][0] = va ? sc4[0] * scale : -CUDART_INF_F;
          sv[h][1] = va ? sc4[1] * scale : -CUDART_INF_F;
          sv[h][2] = vb_ ? sc4[2] * scale : -CUDART_INF_F;
          sv[h][3] = vb_ ? sc4[3] * scale : -CUDART_INF_F;
        }

        // ---- online softmax over the slab's positions (cols 2c, 2c+1)
        float mx0 = fmaxf(fmaxf(sv[0][0], sv[0][2]), fmaxf(sv[1][0], sv[1][2]));
        float mx1 = fmaxf(fmaxf(sv[0][1], sv[0][3]), fmaxf(sv[1][1], sv[1][3]));
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, msk));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, msk));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        float al0 = 1.f, al1 = 1.f;
        float pw[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if (mn0 != -CUDART_INF_F) {
          al0 = exp2f(m0 - mn0);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            pw[h][0] = exp2f(sv[h][0] - mn0);
            pw[h][2] = exp2f(sv[h][2] - mn0);
          }
        }
        if (mn1 != -CUDART_INF_F) {
          al1 = exp2f(m1 - mn1);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            pw[h][1] = exp2f(sv[h][1] - mn1);
            pw[h][3] = exp2f(sv[h][3] - mn1);
          }
        }
        l0 = l0 * al0 + (pw[0][0] + pw[0][2]) + (pw[1][0] + pw[1][2]);
        l1 = l1 * al1 + (pw[0][1] + pw[0][3]) + (pw[1][1] + pw[1][3]);
        m0 = mn0;
        m1 = mn1;
        bool pv_any = true;
        if (a.sparse_thr > 0.f) {  // drop weights <= thr x (this warp's running sum)
          float t0 = l0, t1 = l1;
#pragma unroll
          for (int msk = 4; msk < 32; msk <<= 1) {
            t0 += __shfl_xor_sync(0xffffffffu, t0, msk);
            t1 += __shfl_xor_sync(0xffffffffu, t1, msk);
          }
          bool nz = false;
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            if (pw[h][0] <= a.sparse_thr * t0) pw[h][0] = 0.f;
            if (pw[h][2] <= a.sparse_thr * t0) pw[h][2] = 0.f;
            if (pw[h][1] <= a.sparse_thr * t1) pw[h][1] = 0.f;
            if (pw[h][3] <= a.sparse_thr * t1) pw[h][3] = 0.f;
            nz = nz || pw[h][0] != 0.f || pw[h][1] != 0.f || pw[h][2] != 0.f || pw[h][3] != 0.f;
          }
          // a slab whose weights were all dropped skips its V dequantization
          // and P.V products (the skip the threshold exists for)
          pv_any = __any_sync(0xffffffffu, nz);
        }
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
          for (int i = 0; i < NK; ++i) {
            o[i][0] *= al0; o[i][1] *= al1; o[i][2] *= al0; o[i][3] *= al1;
          }
        }
        if (pv_any) {
#pragma unroll
          for (int h = 0; h < NH; ++h)
            pv16(sb + C::OFF_V + 16 * h * VT::VRS, sb + C::OFF_VS + 16 * h * VT::SROW, pw[h][0],
                 pw[h][1], pw[h][2], pw[h][3]);
        }
      }
      cp_async_wait<0>();
    }

    // ---- merge of the unit's warps; the unit's parameters again from st
    const int64_t x = st[0], off_u = st[4];
    const int seq_u = (int)st[2], kvh_u = kvh;
    int first_u, n_u, len_u, lo_u;
    seq_slabs(seq_u, first_u, n_u, lo_u, len_u);
    const int64_t take = min((int64_t)n_u - off_u, st[1] - x);
    const int64_t ou = x - off_u, cp = st[7];                  // the unit's first slab
    const int64_t vu = ou + U * (int64_t)(seq_u + 1);         // ... on the virtual line
    const int slot = (int)(jr - vu / cp);                      // this CTA's partial
    const int np = (int)((vu + n_u - 1) / cp - vu / cp + 1);   // CTAs on the unit
#pragma unroll
    for (int msk = 4; msk < 32; msk <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, msk);
      l1 += __shfl_xor_sync(0xffffffffu, l1, msk);
    }
    if constexpr (PK) {  // P-hi columns + P-lo columns (lanes c, c ^ 2)
#pragma unroll
      for (int i = 0; i < NK; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[i][e] += __shfl_xor_sync(0xffffffffu, o[i][e], 2);
    }
    const bool writer = !PK || c < 2;
    __syncthreads();  // every warp is done with its ring
    float* mo = reinterpret_cast<float*>(rings);   // [NW warps][8 heads][HD]
    float* ml = mo + NW * 8 * HD;                  // [NW warps][8 heads][m, l]
    if (writer) {
#pragma unroll
      for (int i = 0; i < NK; ++i) {
        const int da = v_row_dim<VS, HD>(i, g), db = v_row_dim<VS, HD>(i, g + 8);
        mo[(warp * 8 + 2 * c) * HD + da] = o[i][0];
        mo[(warp * 8 + 2 * c + 1) * HD + da] = o[i][1];
        mo[(warp * 8 + 2 * c) * HD + db] = o[i][2];
        mo[(warp * 8 + 2 * c + 1) * HD + db] = o[i][3];
      }
    }
    if (g == 0 && writer) {
      ml[(warp * 8 + 2 * c) * 2] = m0;
      ml[(warp * 8 + 2 * c) * 2 + 1] = l0;
      ml[(warp * 8 + 2 * c + 1) * 2] = m1;
      ml[(warp * 8 + 2 * c + 1) * 2 + 1] = l1;
    }
    __syncthreads();
    float* red_s = reinterpret_cast<float*>(scan_s);       // [8 heads][m, l]
    int* last_s = reinterpret_cast<int*>(scan_s + 8);
    for (int idx = tid; idx < a.rep * HD; idx += NT) {
      const int r = idx / HD, d = idx - r * HD;
      float M = -CUDART_INF_F;
#pragma unroll
      for (int w2 = 0; w2 < NW; ++w2) M = fmaxf(M, ml[(w2 * 8 + r) * 2]);
      float acc = 0.f, lsum = 0.f;
      if (M != -CUDART_INF_F) {
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2) {
          const float f = exp2f(ml[(w2 * 8 + r) * 2] - M);
          acc = fmaf(mo[(w2 * 8 + r) * HD + d], f, acc);
          lsum = fmaf(ml[(w2 * 8 + r) * 2 + 1], f, lsum);
        }
      }
      q_s[r * HD + d] = acc * a.v_mult;
      if (d == 0) {
        red_s[2 * r] = M;
        red_s[2 * r + 1] = lsum;
      }
    }
    __syncthreads();
    const int64_t row0 = (int64_t)seq_u * a.nq + kvh_u * a.rep;
    float* part0 = a.part + row0 * a.kmax * (HD + 4);
    // Normalise row r of the unit, rotate it back when V is stored rotated
    // and store it.
    auto finish_row = [&](int r, float (&xr)[E], float lsum) {
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) xr[e] *= inv;
      if constexpr (side_rotated(VS)) fwht_warp<E>(xr, lane, a.inv_sqrt_hd);
      const int64_t o_ = (row0 + r) * HD + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (a.out_bf16) reinterpret_cast<uint16_t*>(a.out)[o_ + e] = bf16_bits_from_float(xr[e]);
        else reinterpret_cast<float*>(a.out)[o_ + e] = xr[e];
      }
    };
    if (np == 1) {  // the whole unit is here
      for (int r = warp; r < a.rep; r += NW) {
        float xr[E];
#pragma unroll
        for (int e = 0; e < E; ++e) xr[e] = q_s[r * HD + lane * E + e];
        finish_row(r, xr, red_s[2 * r + 1]);
      }
    } else {
      // Partial (m, l, acc) to slot `slot`; the last CTA of the unit to
      // arrive merges all np of them (online-softmax identity) and returns
      // the slots and the unit's counter to zero, so that the workspace is
      // all zero between calls whatever their shapes.
      for (int idx = tid; idx < a.rep * (HD + 4); idx += NT) {
        const int r = idx / (HD + 4), d = idx - r * (HD + 4);
        float v = 0.f;
        if (d < 2) v = red_s[2 * r + d];
        else if (d >= 4) v = q_s[r * HD + d - 4];
        part0[((int64_t)r * a.kmax + slot) * (HD + 4) + d] = v;
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        int* ctr = a.counters + (int64_t)seq_u * nkv + kvh_u;
        const int prev = atomicAdd(ctr, 1);
        *last_s = prev == np - 1;
        if (prev == np - 1) *ctr = 0;
      }
      __syncthreads();
      if (*last_s) {
        __threadfence();
        for (int r = warp; r < a.rep; r += NW) {
          const float* pr = part0 + (int64_t)r * a.kmax * (HD + 4);
          float mm = -CUDART_INF_F;
          for (int i = 0; i < np; ++i) mm = fmaxf(mm, __ldcg(pr + i * (HD + 4)));
          float xr[E];
#pragma unroll
          for (int e = 0; e < E; ++e) xr[e] = 0.f;
          float ll = 0.f;
          if (mm != -CUDART_INF_F) {
            for (int i = 0; i < np; ++i) {
              const float* pi = pr + i * (HD + 4);
              const float w = exp2f(__ldcg(pi) - mm);
              ll = fmaf(__ldcg(pi + 1), w, ll);
#pragma unroll
              for (int e = 0; e < E; ++e) xr[e] = fmaf(__ldcg(pi + 4 + lane * E + e), w, xr[e]);
            }
          }
          finish_row(r, xr, ll);
          float* pz = part0 + (int64_t)r * a.kmax * (HD + 4);
          for (int i = lane; i < np * (HD + 4); i += 32) pz[i] = 0.f;
        }
      }
    }

    // next unit
    if (tid == 0) {  // next sequence with positions to attend
      int s2 = seq_u, n2 = 0;
      do {
        ++s2;
        if (s2 >= N) break;
        int f2, l2, e2;
        seq_slabs(s2, f2, n2, l2, e2);
      } while (n2 == 0);
      st[0] = x + take;
      st[2] = s2 < N ? s2 : N - 1;
      st[4] = 0;
      if (s2 >= N) st[1] = st[0];  // nothing left
    }
  }
}

template <int KS, int VS, int HD, bool PK>
cudaError_t launch_tc_kern(const DecodeArgs& a, const Codebooks& cb, cudaStream_t st) {
  using C = TcCfg<KS, VS, HD>;
  static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
  auto kern = decode_tc_kernel<KS, VS, HD, PK>;
  if (C::SMEM > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
  }
  // C::CPS CTAs per SM (one when the stages need more than half of an SM's
  // shared memory); never more CTAs per kv head than the host planned for.
  const int cps = C::SMEM <= (228 - C::CPS) * 1024 / C::CPS ? C::CPS : 1;
  const int ranges = max(1, min(a.max_ranges, cps * a.sms / a.nkv));
  const int grid = ranges * a.nkv;
  kern<<<grid, 32 * C::NW, C::SMEM, st>>>(a, cb);
  return cudaGetLastError();
}

// Up to 4 query heads per KV head leave half of the MMA columns free: they
// carry the lo parts of q and P (packed instances).
template <int KS, int VS, int HD>
cudaError_t launch_tc_inst(const DecodeArgs& a, const Codebooks& cb, cudaStream_t st) {
  return a.rep <= 4 ? launch_tc_kern<KS, VS, HD, true>(a, cb, st)
                    : launch_tc_kern<KS, VS, HD, false>(a, cb, st);
}

template <int KS, int VS>
cudaError_t launch_tc_pair(int hd, const DecodeArgs& a, const Codebooks& cb, cudaStream_t st) {
  switch (hd) {
    case 64: return launch_tc_inst<KS, VS, 64>(a, cb, st);
    case 128: return launch_tc_inst<KS, VS, 128>(a, cb, st);
    case 256: return launch_tc_inst<KS, VS, 256>(a, cb, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
