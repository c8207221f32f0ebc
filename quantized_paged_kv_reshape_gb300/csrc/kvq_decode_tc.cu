// Tensor-core decode instances: (K side, V side) pairs whose stored values
// are exact 16-bit MMA operands.
#include "kvq_decode_mma.cuh"

namespace kvq {

bool decode_tc_supported(int k_side, int v_side) {
  return (k_side == S_BF16 && v_side == S_BF16) || (k_side == S_FP8 && v_side == S_FP8);
}

cudaError_t launch_decode_tc(int k_side, int v_side, int hd, const DecodeArgs& a, cudaStream_t st) {
  if (k_side == S_BF16 && v_side == S_BF16) return launch_tc_pair<S_BF16, S_BF16>(hd, a, st);
  if (k_side == S_FP8 && v_side == S_FP8) return launch_tc_pair<S_FP8, S_FP8>(hd, a, st);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
