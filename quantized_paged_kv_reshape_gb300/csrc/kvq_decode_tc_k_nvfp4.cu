// Tensor-core decode instances whose K side is NVFP4 (one translation unit
// per K side so the instances compile in parallel).  V sides: the
// catalogue's pairs with this K side ("spark_runtime/kv_cache.rs",
// KvCacheDtype::kv_pair: NVFP4 is symmetric only).  NVFP4 runs the codebook
// path with the 16 E2M1 values as its level table and no rotation.
#include "kvq_decode_mma.cuh"

namespace kvq {

cudaError_t launch_tc_k_nvfp4(int v_side, int hd, const DecodeArgs& a, const Codebooks& cb,
                              cudaStream_t st) {
  switch (v_side) {
    case S_NVFP4: return launch_tc_pair<S_NVFP4, S_NVFP4>(hd, a, cb, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
