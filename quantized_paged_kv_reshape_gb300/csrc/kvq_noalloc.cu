// Paged decode for callers that cannot allocate device memory.
//
// kvq_paged_decode needs a caller-provided scratch buffer for the partial
// results of rows that several CTAs share and their merge counters.  Some
// callers cannot get one: a runtime that has already handed all device memory
// to its own pool, a plugin host that forbids device allocations by its
// plugins, or a latency-critical loop where cudaMalloc (which may synchronize
// the device) is not acceptable.  This entry point runs the same kernels with
// the scratch taken from a fixed array compiled into the library instead; it
// allocates nothing.
//
// The array lives in every GPU that loads the library, for the life of the
// process.  Host code must not use the array's name as a device address (on
// the host it only names a stand-in).  The device address belongs to the copy
// of the library's device code loaded into the current context, and a new
// context (after cudaDeviceReset, or once the primary context was released
// and created again) loads a new copy, so the address is looked up with
// cudaGetSymbolAddress on every call.  The one exception is a call made
// while its stream is being captured into a graph: it reuses the address that
// the last uncaptured call on the same device looked up (a lookup could load
// the module, which a capture does not allow), and fails if there was none.
// All calls share the one array, so calls whose kernels overlap on the GPU
// race.  The array is zero when its copy is loaded (static storage) and every
// decode leaves it zero, which is the state the next call needs; a call that
// fails after the launch was attempted queues a clear of the part it may have
// touched before it returns.
#include "../../include/kvq.h"

#include <cuda_runtime.h>

#include <mutex>

namespace kvq {
void record_error(const char* msg);
}

namespace {

constexpr size_t kScratchBytes = KVQ_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_last_lookup[kMaxDevices] = {};   // per device: the last uncaptured call's address

kvq_status scratch_address(cudaStream_t stream, void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    kvq::record_error("no usable current CUDA device for the built-in decode scratch");
    return KVQ_ERR_CUDA;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) {
    kvq::record_error("cudaStreamIsCapturing failed on the decode stream");
    return KVQ_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p) {
      g_last_lookup[dev] = nullptr;
      kvq::record_error("cudaGetSymbolAddress of the built-in decode scratch failed");
      return KVQ_ERR_CUDA;
    }
    g_last_lookup[dev] = p;
  } else if (!g_last_lookup[dev]) {
    kvq::record_error(
        "the first decode without a workspace on this device was made during stream capture; "
        "make one uncaptured call first");
    return KVQ_ERR_CUDA;
  }
  *out = g_last_lookup[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_paged_decode_noalloc(
    const void* q, kvq_dtype q_dtype, int64_t q_stride, const void* k_cache, const void* v_cache,
    void* out, kvq_dtype out_dtype, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens, int32_t num_seqs, int64_t num_blocks, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t k_block_stride_bytes,
    int64_t v_block_stride_bytes, float sm_scale, float k_scale, float v_scale,
    int32_t sliding_window, float sparse_v_threshold, kvq_format fmt, int32_t* error_flag,
    void* stream) {
  const size_t need = kvq_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 block_size, max_blocks_per_seq, sliding_window,
                                                 fmt);
  if (need > kScratchBytes) {
    kvq::record_error(
        "decode needs more scratch than the built-in 8 MiB (fewer sequences or heads per call, "
        "or kvq_paged_decode with a caller-provided workspace)");
    return KVQ_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const kvq_status st = scratch_address((cudaStream_t)stream, &scratch);
  if (st != KVQ_OK) return st;
  const kvq_status r = kvq_paged_decode(
      q, q_dtype, q_stride, k_cache, v_cache, out, out_dtype, block_tables, max_blocks_per_seq,
      seq_lens, num_seqs, num_blocks, num_q_heads, num_kv_heads, head_dim, block_size,
      k_block_stride_bytes, v_block_stride_bytes, sm_scale, k_scale, v_scale, sliding_window,
      sparse_v_threshold, scratch, kScratchBytes, fmt, error_flag, stream);
  if (r == KVQ_ERR_CUDA && need > 0) {
    // The launch was attempted: return the part of the array this call may
    // have touched to zero (stream-ordered; kvq_last_error keeps the launch's
    // message).
    cudaMemsetAsync(scratch, 0, need, (cudaStream_t)stream);
  }
  return r;
}
