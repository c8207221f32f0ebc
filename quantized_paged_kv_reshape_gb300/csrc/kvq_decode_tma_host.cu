// Host side of the TMA-fed decode: which calls it serves, the tensor maps of
// the four pool sections, and the dispatch to the per-K-side instances.
//
// A section is described as a tensor over the pool, innermost first:
// (row bytes, kv head, position in the block, block) with the block stride
// the caller's k/v_block_stride_bytes ("metrale_model_layers/layers/ops/
// kv_cache_bf16k_turbov.rs", module invariants: layout [num_blocks,
// block_size, num_kv_heads, head_dim], separate byte strides per pool).
// Scale rows shorter than 16 bytes are described per position instead
// ((num_kv_heads * scale-row bytes), position, block) and copied as the
// 16-byte span that holds the head's row.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kvq_decode_tma.cuh"

namespace kvq {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int row_bytes(int side, int hd) { return hd * side_bits(side) / 8; }
int scale_row_bytes(int side, int hd) { return (hd / kGroup) * side_scale_bytes(side); }

CUtensorMapSwizzle swizzle_of(int boxw) {
  return boxw == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
       : boxw == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
       : boxw == 32  ? CU_TENSOR_MAP_SWIZZLE_32B
                     : CU_TENSOR_MAP_SWIZZLE_NONE;
}

// Rows of `rowb` bytes per (position, kv head), boxes of min(rowb, 128) bytes
// x 1 head x min(bs, 16) positions x 1 block.
bool data_map(CUtensorMap* m, const void* base, int rowb, int nkv, int bs, int64_t nb,
              int64_t bstride, bool swizzle) {
  const int boxw = rowb > 128 ? 128 : rowb;
  const cuuint64_t dim[4] = {(cuuint64_t)rowb, (cuuint64_t)nkv, (cuuint64_t)bs, (cuuint64_t)nb};
  const cuuint64_t str[3] = {(cuuint64_t)rowb, (cuuint64_t)rowb * nkv, (cuuint64_t)bstride};
  const cuuint32_t box[4] = {(cuuint32_t)boxw, 1, (cuuint32_t)(bs < 16 ? bs : 16), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dim, str, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle ? swizzle_of(boxw) : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale rows of `srow` bytes: as data rows when srow >= 16, else per
// position (nkv * srow bytes) with 16-byte boxes.
bool scale_map(CUtensorMap* m, const void* base, int srow, int nkv, int bs, int64_t nb,
               int64_t bstride) {
  if (srow >= 16) return data_map(m, base, srow, nkv, bs, nb, bstride, false);
  const cuuint64_t dim[3] = {(cuuint64_t)nkv * srow, (cuuint64_t)bs, (cuuint64_t)nb};
  const cuuint64_t str[2] = {(cuuint64_t)nkv * srow, (cuuint64_t)bstride};
  const cuuint32_t box[3] = {16, (cuuint32_t)(bs < 16 ? bs : 16), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dim, str, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool side_shape_ok(int side, int hd, int nkv) {
  const int rowb = row_bytes(side, hd);
  if (rowb % 16 != 0) return false;
  const int srow = scale_row_bytes(side, hd);
  if (srow > 0 && srow < 16 && (nkv * srow) % 16 != 0) return false;
  return true;
}

// KVQ_DECODE_KERNEL=mma keeps every call on decode_tc_kernel (the kernel
// choice never changes results beyond rounding order).
bool tma_enabled() {
  const char* e = std::getenv("KVQ_DECODE_KERNEL");
  return !(e && std::strcmp(e, "mma") == 0);
}

// The code tables sit at a fixed shared address that assumes the driver
// reserves 1 KB of shared memory per block ahead of dynamic shared memory.
bool reserved_smem_ok() {
  static int cache[64] = {0};   // 0 unknown, 1 ok, 2 not
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (!cache[dev]) {
    int r = -1;
    cache[dev] = (cudaDeviceGetAttribute(&r, cudaDevAttrReservedSharedMemoryPerBlock, dev) ==
                      cudaSuccess && r == kSmemBase) ? 1 : 2;
  }
  return cache[dev] == 1;
}

}  // namespace

bool decode_tma_supported(int ks, int vs, int hd, int nkv, int bs) {
  if (!tma_enabled() || !encode_fn() || !reserved_smem_ok()) return false;
  if (!tma_k_side(ks) || !tma_v_side(vs)) return false;
  if (hd != 64 && hd != 128) return false;
  if (bs != 8 && bs != 16 && bs != 32) return false;
  if (vs == S_T3 && hd != 128) return false;
  return side_shape_ok(ks, hd, nkv) && side_shape_ok(vs, hd, nkv);
}

cudaError_t launch_decode_tma(int ks, int vs, int hd, const DecodeArgs& a, const Codebooks& cb,
                              cudaStream_t st) {
  TmaMaps maps;
  std::memset(&maps, 0, sizeof maps);
  const int64_t nb = a.num_blocks > 0 ? a.num_blocks : ((int64_t)1 << 31) - 1;
  const int krow = row_bytes(ks, hd), vrow = row_bytes(vs, hd);
  bool ok = data_map(&maps.kd, a.k_cache, krow, a.nkv, a.bs, nb, a.k_bstride, true) &&
            data_map(&maps.vd, a.v_cache, vrow, a.nkv, a.bs, nb, a.v_bstride, true);
  const int ksr = scale_row_bytes(ks, hd), vsr = scale_row_bytes(vs, hd);
  if (ok && ksr > 0) ok = scale_map(&maps.ks, a.k_cache + a.k_dsec, ksr, a.nkv, a.bs, nb, a.k_bstride);
  if (ok && vsr > 0) ok = scale_map(&maps.vs, a.v_cache + a.v_dsec, vsr, a.nkv, a.bs, nb, a.v_bstride);
  if (!ok) return cudaErrorInvalidValue;
  switch (ks) {
    case S_BF16: return launch_tma_k_bf16(vs, hd, a, maps, cb, st);
    case S_FP8: return launch_tma_k_fp8(vs, hd, a, maps, cb, st);
    case S_T4: return launch_tma_k_t4(vs, hd, a, maps, cb, st);
    case S_NVFP4: return launch_tma_k_nvfp4(vs, hd, a, maps, cb, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
