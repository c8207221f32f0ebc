// Chunked-prefill attention over the quantized paged cache: the pieces the
// tensor-memory kernel (kvq_prefill_tc5.cuh) shares with nothing else of
// the decode: the operand-plane count of a side, its level tables and the
// dequantization of staged rows into 16-bit operand words.
//
// "combs_models/kv.rs" attend (scores, causal mask, softmax, P.V) with
// repeat_kv for a chunk of new query tokens per sequence, after the chunk's
// K/V rows were written to the cache; "spark_runtime/kv_cache.rs"
// is_wht_rotated bookends (q rotated forward when K is stored rotated, the
// output rotated back when V is).  Sequence s holds L = seq_lens[s]
// positions; its C = cu_q[s+1] - cu_q[s] queries are the last C positions,
// query i at p = L - C + i attends to [max(0, p + 1 - W), p] (W = window, 0 =
// none).  Where one 16-bit value is not exact, operands carry hi + lo
// parts (level x group scale), like q and P.
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

}  // namespace kvq
