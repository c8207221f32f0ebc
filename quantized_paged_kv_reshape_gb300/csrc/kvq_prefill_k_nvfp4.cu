// Chunked-prefill instances whose K side is NVFP4 (one translation unit
// per K side so the instances compile in parallel).  V sides: the
// catalogue's pairs with this K side ("spark_runtime/kv_cache.rs",
// KvCacheDtype::kv_pair).
#include "kvq_prefill_tc5.cuh"

namespace kvq {

cudaError_t launch_pf_k_nvfp4(int v_side, int hd, const PrefillArgs& a, const Codebooks& cb,
                            int max_chunk, cudaStream_t st) {
  switch (v_side) {
    case S_NVFP4: return launch_prefill_pair<S_NVFP4, S_NVFP4>(hd, a, cb, max_chunk, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
