// TMA-fed decode instances whose K side is NVFP4 (one translation unit per K
// side so the instances compile in parallel).  V sides: the catalogue's
// pairs with this K side ("spark_runtime/kv_cache.rs", KvCacheDtype::kv_pair)
// that the TMA decode handles.
#include "kvq_decode_tma.cuh"

namespace kvq {

cudaError_t launch_tma_k_nvfp4(int v_side, int hd, const DecodeArgs& a, const TmaMaps& maps,
                              const Codebooks& cb, cudaStream_t st) {
  switch (v_side) {
    case S_NVFP4: return hd == 64 ? launch_tma_inst<S_NVFP4, S_NVFP4, 64>(a, maps, cb, st)
                             : launch_tma_inst<S_NVFP4, S_NVFP4, 128>(a, maps, cb, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
