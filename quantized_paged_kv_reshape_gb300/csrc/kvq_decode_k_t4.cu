// Decode instances whose K side is T4 (one translation unit per K side
// so the instances compile in parallel).  V sides: the catalogue's pairs
// with this K side ("spark_runtime/kv_cache.rs", KvCacheDtype::kv_pair).
#include "kvq_decode.cuh"

namespace kvq {

cudaError_t launch_decode_k_t4(int v_side, int hd, int rmax, const DecodeArgs& a,
                                 const Codebooks& cb, cudaStream_t st) {
  switch (v_side) {
    case S_T4: return launch_decode_pair<S_T4, S_T4>(hd, rmax, a, cb, st);
    case S_T3: return launch_decode_pair<S_T4, S_T3>(hd, rmax, a, cb, st);
    case S_T8: return launch_decode_pair<S_T4, S_T8>(hd, rmax, a, cb, st);
    default: return cudaErrorInvalidValue;
  }
}

size_t smem_k_t4(int v_side, int hd, int rmax) {
  switch (v_side) {
    case S_T4: return smem_pair<S_T4, S_T4>(hd, rmax);
    case S_T3: return smem_pair<S_T4, S_T3>(hd, rmax);
    case S_T8: return smem_pair<S_T4, S_T8>(hd, rmax);
    default: return 0;
  }
}

}  // namespace kvq
