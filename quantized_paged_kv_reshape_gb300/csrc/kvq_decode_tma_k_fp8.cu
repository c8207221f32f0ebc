// TMA-fed decode instances whose K side is FP8 (one translation unit per K
// side so the instances compile in parallel).  V sides: the catalogue's
// pairs with this K side ("spark_runtime/kv_cache.rs", KvCacheDtype::kv_pair)
// that the TMA decode handles.
#include "kvq_decode_tma.cuh"

namespace kvq {

cudaError_t launch_tma_k_fp8(int v_side, int hd, const DecodeArgs& a, const TmaMaps& maps,
                              const Codebooks& cb, cudaStream_t st) {
  switch (v_side) {
    case S_FP8: return hd == 64 ? launch_tma_inst<S_FP8, S_FP8, 64>(a, maps, cb, st)
                             : launch_tma_inst<S_FP8, S_FP8, 128>(a, maps, cb, st);
    case S_T4: return hd == 64 ? launch_tma_inst<S_FP8, S_T4, 64>(a, maps, cb, st)
                             : launch_tma_inst<S_FP8, S_T4, 128>(a, maps, cb, st);
    case S_T3: return hd == 128 ? launch_tma_inst<S_FP8, S_T3, 128>(a, maps, cb, st) : cudaErrorInvalidValue;
    case S_T2: return hd == 64 ? launch_tma_inst<S_FP8, S_T2, 64>(a, maps, cb, st)
                             : launch_tma_inst<S_FP8, S_T2, 128>(a, maps, cb, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
