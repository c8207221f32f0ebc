// Tensor-core decode instances whose K side is BF16 (one translation unit
// per K side so the instances compile in parallel).  V sides: the
// catalogue's pairs with this K side ("spark_runtime/kv_cache.rs",
// KvCacheDtype::kv_pair).
#include "kvq_decode_mma.cuh"

namespace kvq {

cudaError_t launch_tc_k_bf16(int v_side, int hd, const DecodeArgs& a, const Codebooks& cb,
                              cudaStream_t st) {
  switch (v_side) {
    case S_BF16: return launch_tc_pair<S_BF16, S_BF16>(hd, a, cb, st);
    case S_T4: return launch_tc_pair<S_BF16, S_T4>(hd, a, cb, st);
    case S_T3: return launch_tc_pair<S_BF16, S_T3>(hd, a, cb, st);
    case S_T2: return launch_tc_pair<S_BF16, S_T2>(hd, a, cb, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq

namespace kvq {

bool decode_tc_supported(int k_side, int v_side) {
  switch (k_side) {
    case S_BF16: case S_FP8: return v_side == k_side || v_side == S_T4 || v_side == S_T3 || v_side == S_T2;
    case S_T4: return v_side == S_T4 || v_side == S_T3 || v_side == S_T8;
    case S_T3: return v_side == S_T3 || v_side == S_T8;
    case S_T2: return v_side == S_T2;
    case S_T8: return v_side == S_T8;
    case S_NVFP4: return v_side == S_NVFP4;
    default: return false;
  }
}

cudaError_t launch_decode_tc(int k_side, int v_side, int hd, const DecodeArgs& a,
                             const Codebooks& cb, cudaStream_t st) {
  switch (k_side) {
    case S_BF16: return launch_tc_k_bf16(v_side, hd, a, cb, st);
    case S_FP8: return launch_tc_k_fp8(v_side, hd, a, cb, st);
    case S_T4: return launch_tc_k_t4(v_side, hd, a, cb, st);
    case S_T3: return launch_tc_k_t3(v_side, hd, a, cb, st);
    case S_T2: return launch_tc_k_t2(v_side, hd, a, cb, st);
    case S_T8: return launch_tc_k_t8(v_side, hd, a, cb, st);
    case S_NVFP4: return launch_tc_k_nvfp4(v_side, hd, a, cb, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
