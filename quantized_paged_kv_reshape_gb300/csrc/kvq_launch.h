// Argument blocks and launchers shared between the C ABI (kvq_api.cpp) and
// the kernel translation units.  Host-validated values only: the kernels
// trust these fields.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace kvq {

struct Codebooks;

struct WriteArgs {
  const void* key;
  const void* value;
  uint8_t* k_cache;
  uint8_t* v_cache;
  const int64_t* slots;
  int32_t num_tokens;
  int64_t num_slots;      // num_blocks * block_size, 0 = unchecked
  int32_t nkv;
  int32_t bs;
  int32_t bs_shift;                     // log2(bs) if bs is a power of two, else -1
  int64_t key_stride, value_stride;     // elements per token
  int64_t k_bstride, v_bstride;         // bytes per block
  int64_t k_dsec, v_dsec;               // scale-section offsets
  float k_scale, v_scale;               // per-tensor FP8 scales
  float k_inv, v_inv;                   // 1/scale where scale is a power of two, else 0
  float inv_sqrt_hd;                    // fp32(1/sqrt(head_dim))
  int k_side, v_side;
  // n / nkv for n < 2^31 as (h + ((n - h) >> nkv_s1)) >> nkv_s2, h =
  // umulhi(n, nkv_m) (Granlund and Montgomery's round-up division)
  uint32_t nkv_m, nkv_s1, nkv_s2;
  int32_t* err;
};

struct DecodeArgs {  // arguments of the paged decode (decode_tc_kernel)
  const void* q;
  int64_t q_stride;       // elements between sequences
  int q_bf16;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;
  int32_t max_blocks;
  const int32_t* seq_lens;
  int32_t num_seqs;
  int64_t num_blocks;     // 0 = unchecked
  int32_t nq, nkv, rep;   // rep = nq / nkv
  int32_t bs;
  int64_t k_bstride, v_bstride, k_dsec, v_dsec;
  float score_scale;      // sm_scale * log2(e) (* k_scale for FP8 K)
  float v_mult;           // v_scale for FP8 V, else 1
  float inv_sqrt_hd;
  int32_t window;
  float sparse_thr;
  int32_t sms;            // SMs of the device
  int32_t max_ranges;     // upper bound of the CTAs per kv head (sizes kmax)
  int32_t kmax;           // partial slots per (sequence, query head)
  float* part;            // [num_seqs][nq][kmax][head_dim + 4] fp32: m, l, -, -, acc[head_dim]
  int32_t* counters;      // [num_seqs][nkv] partials arrived; zero between calls
  void* out;              // [num_seqs][nq][head_dim], fp32 or bf16
  int out_bf16;
  int32_t* err;
};


struct PrefillArgs {  // arguments of the chunked prefill (prefill_tc5_kernel)
  const void* q;
  int64_t q_stride;          // elements between query tokens
  int q_bf16;
  const int32_t* cu_q;       // [num_seqs + 1]
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  void* out;                 // [total_q][nq][hd]
  int out_bf16;
  const int32_t* block_tables;
  int32_t max_blocks;
  const int32_t* seq_lens;
  int32_t num_seqs;
  int64_t num_blocks;        // 0 = unchecked
  int32_t nq, nkv, rep, rp;  // rp = rep rounded up to a power of two
  int32_t bs;
  int64_t k_bstride, v_bstride, k_dsec, v_dsec;
  float score_scale;         // sm_scale * log2(e) (* k_scale for FP8 K)
  float v_mult;              // v_scale for FP8 V, else 1
  float inv_sqrt_hd;
  int32_t window;
  int32_t* err;
};

cudaError_t launch_cache_write(const WriteArgs& a, const Codebooks& cb, int head_dim,
                               bool in_bf16, bool vec, int sms, cudaStream_t st);

// Tensor-core decode (kvq_decode_tc_k_*.cu) for the pairs it supports.
bool decode_tc_supported(int k_side, int v_side);
cudaError_t launch_decode_tc(int k_side, int v_side, int hd, const DecodeArgs& a,
                             const Codebooks& cb, cudaStream_t st);
cudaError_t launch_tc_k_bf16(int v_side, int hd, const DecodeArgs&, const Codebooks&, cudaStream_t);
cudaError_t launch_tc_k_fp8(int v_side, int hd, const DecodeArgs&, const Codebooks&, cudaStream_t);
cudaError_t launch_tc_k_t4(int v_side, int hd, const DecodeArgs&, const Codebooks&, cudaStream_t);
cudaError_t launch_tc_k_t3(int v_side, int hd, const DecodeArgs&, const Codebooks&, cudaStream_t);
cudaError_t launch_tc_k_t2(int v_side, int hd, const DecodeArgs&, const Codebooks&, cudaStream_t);
cudaError_t launch_tc_k_t8(int v_side, int hd, const DecodeArgs&, const Codebooks&, cudaStream_t);
cudaError_t launch_tc_k_nvfp4(int v_side, int hd, const DecodeArgs&, const Codebooks&, cudaStream_t);

// TMA-fed decode (kvq_decode_tma_*.cu) for the sides, head dims and
// shapes it handles; the others run decode_tc_kernel.
struct TmaMaps;
bool decode_tma_supported(int k_side, int v_side, int hd, int nkv, int bs);
cudaError_t launch_decode_tma(int k_side, int v_side, int hd, const DecodeArgs& a,
                              const Codebooks& cb, cudaStream_t st);
cudaError_t launch_tma_k_bf16(int v_side, int hd, const DecodeArgs&, const TmaMaps&, const Codebooks&, cudaStream_t);
cudaError_t launch_tma_k_fp8(int v_side, int hd, const DecodeArgs&, const TmaMaps&, const Codebooks&, cudaStream_t);
cudaError_t launch_tma_k_t4(int v_side, int hd, const DecodeArgs&, const TmaMaps&, const Codebooks&, cudaStream_t);
cudaError_t launch_tma_k_nvfp4(int v_side, int hd, const DecodeArgs&, const TmaMaps&, const Codebooks&, cudaStream_t);

// Chunked prefill (kvq_prefill_k_*.cu), same pairs as the decode.
cudaError_t launch_pf_k_bf16(int v_side, int hd, const PrefillArgs&, const Codebooks&, int, cudaStream_t);
cudaError_t launch_pf_k_fp8(int v_side, int hd, const PrefillArgs&, const Codebooks&, int, cudaStream_t);
cudaError_t launch_pf_k_t4(int v_side, int hd, const PrefillArgs&, const Codebooks&, int, cudaStream_t);
cudaError_t launch_pf_k_t3(int v_side, int hd, const PrefillArgs&, const Codebooks&, int, cudaStream_t);
cudaError_t launch_pf_k_t2(int v_side, int hd, const PrefillArgs&, const Codebooks&, int, cudaStream_t);
cudaError_t launch_pf_k_t8(int v_side, int hd, const PrefillArgs&, const Codebooks&, int, cudaStream_t);
cudaError_t launch_pf_k_nvfp4(int v_side, int hd, const PrefillArgs&, const Codebooks&, int, cudaStream_t);

}  // namespace kvq
