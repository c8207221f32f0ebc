/*
 * kvq.h - C ABI of the quantized paged KV cache library (libkvq.so).
 *
 * Two operations make up the hot path:
 *
 *   kvq_cache_write   scatter new K/V rows into a paged cache, storing each
 *                     side raw (BF16), as FP8 E4M3 with a per-tensor scale, or
 *                     TurboQuant-style (Walsh-Hadamard rotation, one E4M3
 *                     scale per 16 elements, 2/3/4-bit Lloyd-Max N(0,1)
 *                     codes; Turbo8 stores E4M3 data with BF16 group scales).
 *   kvq_paged_decode  one-query-per-sequence attention over that cache through
 *                     block tables, with grouped-query heads, 1/sqrt(d)
 *                     scaling and an optional sliding window.
 *
 * Sources (web pages, cited by title and section):
 *   [ATLAS]  "spark_runtime/kv_cache.rs": enum KvCacheDtype (formats and their
 *            storage), kv_pair, is_wht_rotated, FromStr spellings,
 *            KvCacheConfig::block_bytes_dims and the turbo*_data_bytes /
 *            turbo*_scale_bytes section helpers, LayerPool (separate K and V
 *            block strides in bytes).
 *   [METRALE] "metrale_model_layers/layers/ops/kv_cache_bf16k_turbov.rs":
 *            module invariants (the [num_blocks, block_size, num_kv_heads,
 *            head_dim] layout, code section then scale section, byte block
 *            strides), reshape_and_cache_* and paged_decode_attn_* launcher
 *            argument lists, the sparse-V threshold.
 *   [BURN]   "combs_models/kv.rs": attend (scores -> softmax -> P.V),
 *            repeat_kv (query head j reads kv head j / (nq/nkv)),
 *            PagedKVCache::attention (slot = page * page_size + offset).
 *
 * Conventions shared by every call:
 *   - All device pointers are plain CUDA device addresses owned by the
 *     caller; the library allocates nothing and keeps no state between
 *     calls except the host-side codebook tables, built once per process,
 *     and the fixed scratch array of kvq_paged_decode_noalloc.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work; none synchronizes the host.
 *   - Errors are returned as kvq_status; arguments are validated on the host
 *     before anything is launched.  kvq_last_error() returns a message for
 *     the last failing call on the calling thread.  Device-side index errors
 *     (a slot or block id outside [0, num_blocks)) never fault: the row is
 *     skipped and, if `error_flag` is non-NULL, KVQ_DEVERR_* bits are OR-ed
 *     into that device word.
 *   - Block layout of one side ([METRALE] invariants, [ATLAS]
 *     block_bytes_dims), E = block_size * num_kv_heads * head_dim:
 *       element e = (offset_in_block * num_kv_heads + kv_head) * head_dim + d
 *       BF16 : 2E bytes, little-endian BF16 at byte 2e
 *       FP8  : E bytes, E4M3 at byte e
 *       TURBO4/3/2: code section of E*b/8 bytes (codes packed LSB-first in a
 *              little-endian bit stream: element e occupies bits [b*e,
 *              b*e+b)), then the scale section: E/16 E4M3 bytes, group
 *              g = e/16 at byte data_section + g
 *       TURBO8: E E4M3 bytes, then E/16 BF16 scales (little-endian) at
 *              data_section + 2g
 *     A side's block stride (bytes) may exceed kvq_block_bytes (padding).
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
    KVQ_OK = 0,
    KVQ_ERR_ARG = 1,        /* null pointer, negative count, bad scale      */
    KVQ_ERR_FORMAT = 2,     /* unknown or unsupported format / dtype        */
    KVQ_ERR_SHAPE = 3,      /* head_dim, GQA ratio or block_size unsupported */
    KVQ_ERR_ALIGN = 4,      /* pointer or stride not 16-byte aligned         */
    KVQ_ERR_WORKSPACE = 5,  /* decode workspace missing or too small         */
    KVQ_ERR_CUDA = 6        /* a CUDA runtime call or launch failed          */
} kvq_status;

/* Device-side error bits written to *error_flag (never a fault). */
#define KVQ_DEVERR_SLOT 1   /* write: slot >= num_blocks * block_size        */
#define KVQ_DEVERR_BLOCK 2  /* decode: block table entry outside the pool    */
#define KVQ_DEVERR_TIMEOUT 4 /* decode: a bounded wait for a page copy gave up */

/* Combined cache formats, in the order of [ATLAS] enum KvCacheDtype.
 * kv_pair: the symmetric formats store the same side format in both pools;
 * the asymmetric ones name (K side, V side). */
typedef enum kvq_format {
    KVQ_FMT_BF16 = 0,
    KVQ_FMT_FP8 = 1,
    KVQ_FMT_NVFP4 = 2,
    KVQ_FMT_TURBO4 = 3,
    KVQ_FMT_TURBO3 = 4,
    KVQ_FMT_TURBO2 = 5,
    KVQ_FMT_TURBO8 = 6,
    KVQ_FMT_TURBO4K_TURBO3V = 7,
    KVQ_FMT_TURBO4K_TURBO8V = 8,
    KVQ_FMT_TURBO3K_TURBO8V = 9,
    KVQ_FMT_BF16K_TURBO4V = 10,
    KVQ_FMT_BF16K_TURBO3V = 11,
    KVQ_FMT_FP8K_TURBO4V = 12,
    KVQ_FMT_FP8K_TURBO3V = 13,
    KVQ_FMT_BF16K_TURBO2V = 14,
    KVQ_FMT_FP8K_TURBO2V = 15,
    KVQ_FMT_COUNT = 16
} kvq_format;

/* Element type of activations (key, value, q, out). */
typedef enum kvq_dtype {
    KVQ_DTYPE_F32 = 0,
    KVQ_DTYPE_BF16 = 1
} kvq_dtype;

/* Which pool of a combined format: [ATLAS] kv_pair().0 / .1 */
#define KVQ_SIDE_K 0
#define KVQ_SIDE_V 1

/* ---------------------------------------------------------------- catalogue */

/* [ATLAS] FromStr: parse a --kv-cache-dtype spelling ("turbo4k_turbo3v",
 * "turbo4k3v", ...). Returns KVQ_ERR_FORMAT for an unknown spelling. */
kvq_status kvq_format_from_string(const char* name, kvq_format* out);

/* Canonical spelling (long form for asymmetric pairs); NULL if out of range. */
const char* kvq_format_name(kvq_format fmt);

/* [ATLAS] kv_pair / is_wht_rotated: the side format stored in pool `side`
 * (as a symmetric kvq_format value), and whether that side is stored in the
 * Walsh-Hadamard basis. Return -1 for an invalid argument. */
int kvq_side_format(kvq_format fmt, int side);
int kvq_side_is_rotated(kvq_format fmt, int side);

/* [ATLAS] block_bytes_dims routed through kv_pair (k_/v_block_bytes_dims):
 * bytes of one block of pool `side`; -1 for invalid arguments. */
int64_t kvq_block_bytes(kvq_format fmt, int side, int32_t block_size,
                        int32_t num_kv_heads, int32_t head_dim);

/* [ATLAS] turbo*_data_bytes / nvfp4_data_bytes: offset of the scale section
 * inside a block (= bytes of the code or raw-data section); -1 if invalid. */
int64_t kvq_data_section_bytes(kvq_format fmt, int side, int32_t block_size,
                               int32_t num_kv_heads, int32_t head_dim);

/* [ATLAS] KvCacheDtype::Turbo4/3/2 (Lloyd-Max N(0,1) codebook): copies the
 * library's fp32 levels (2^bits, ascending) and decision thresholds
 * (2^bits - 1, fp32 midpoints of adjacent fp64 levels) for bits in {2,3,4}.
 * Either pointer may be NULL. Host memory. */
kvq_status kvq_codebook(int bits, float* levels, float* thresholds);

const char* kvq_status_string(kvq_status st);
const char* kvq_last_error(void);

/* ------------------------------------------------------------- cache write */

/* [METRALE] reshape_and_cache_bf16k_turbo{2,3,4}v; [ATLAS] Turbo4KTurbo3V
 * (one launch writes the K side and the V side, each in its own format).
 *
 * For each token t < num_tokens with slot = slot_mapping[t] >= 0, and each
 * kv head h, row (t, h) of `key` (resp. `value`) - the head_dim elements
 * starting at element t*key_stride + h*head_dim - is encoded in the K
 * (resp. V) side format of `fmt` and stored in block
 * slot / block_size at offset slot % block_size of k_cache (resp. v_cache),
 * whose blocks are k_block_stride_bytes (v_...) apart.  Rotated sides apply
 * the normalised Walsh-Hadamard transform in fp32 (butterfly stages
 * h = 1, 2, 4, ..., then one multiply by 1/sqrt(head_dim)), take per group
 * of 16 the scale E4M3(amax / max_level) (Turbo8: BF16(amax / 448)), and
 * store code = #{thresholds <= y / scale}; a zero scale stores code 2^(b-1)
 * (Turbo8: byte 0).  FP8 sides store E4M3(x / k_scale) (v_scale).  NVFP4
 * ([ATLAS] Nvfp4, "E2M1 packed nibbles", Turbo4's layout) is not rotated:
 * scale E4M3(amax / 6) per group of 16, code = E2M1(x / scale) (sign bit 3),
 * a zero scale stores code 0.  All E4M3/BF16/E2M1 encodes round to nearest
 * even and saturate.
 *
 *   key, value       device, in_dtype elements; row (t,h) as above
 *   k_cache, v_cache device, 16-byte aligned pools
 *   slot_mapping     device int64 [num_tokens]; negative = skip the token
 *   num_blocks       blocks in each pool; slots >= num_blocks*block_size
 *                    are skipped and flagged (0 = do not check)
 *   head_dim         64, 128 or 256; block_size >= 1
 *   key_stride, value_stride   elements between consecutive tokens
 *   k_scale, v_scale per-tensor FP8 scales (> 0), used by FP8 sides only
 *   error_flag       optional device int32 (NULL = none)
 * Duplicate slots within one call race (last writer unspecified). */
kvq_status kvq_cache_write(
    const void* key, const void* value, kvq_dtype in_dtype,
    void* k_cache, void* v_cache, const int64_t* slot_mapping,
    int32_t num_tokens, int64_t num_blocks,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    int64_t key_stride, int64_t value_stride,
    int64_t k_block_stride_bytes, int64_t v_block_stride_bytes,
    float k_scale, float v_scale, kvq_format fmt,
    int32_t* error_flag, void* stream);

/* ------------------------------------------------------------ paged decode */

/* Which decode kernel kvq_paged_decode launches on the current device for
 * these arguments: 1 = the kernel that stages cache pages with TMA tensor
 * copies (BF16/FP8/Turbo4/NVFP4 K sides, head_dim 64/128), 0 = the kernel
 * that stages them with cp.async (every other case, and every case when the
 * environment variable KVQ_DECODE_KERNEL is "mma"), -1 = a format, head_dim,
 * num_kv_heads or block_size kvq_paged_decode rejects.  Both compute the
 * same attention ("combs_models/kv.rs", attend; "spark_runtime/kv_cache.rs",
 * is_wht_rotated).  Host only; no device work. */
int32_t kvq_decode_path(kvq_format fmt, int32_t head_dim, int32_t num_kv_heads,
                        int32_t block_size);


/* Bytes of device scratch kvq_paged_decode needs for these arguments: fp32
 * partial results of (sequence, query head) rows that several CTAs share,
 * followed by one int32 merge counter per (sequence, kv head) (the last
 * 16-byte-rounded num_seqs*num_kv_heads*4 bytes).  The size depends on the
 * current device's SM count, so query on the device that will run the
 * decode.  0 on error. */
size_t kvq_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int32_t max_blocks_per_seq,
                                  int32_t sliding_window, kvq_format fmt);

/* [METRALE] paged_decode_attn_bf16k_turbo{2,3,4}v (argument list), [ATLAS]
 * Turbo4KTurbo3V's decode variant and is_wht_rotated ("WHT(Q) / iWHT(out)
 * attention bookends"), [BURN] attend + repeat_kv for one query.
 *
 * For sequence s with L = seq_lens[s] and lo = max(0, L - sliding_window)
 * (lo = 0 when sliding_window == 0), query head j attends to positions
 * p in [lo, L), stored at block block_tables[s*max_blocks_per_seq + p/bs],
 * offset p % bs, kv head j / (num_q_heads/num_kv_heads):
 *   out[s, j, :] = sum_p softmax_p(sm_scale * q[s,j].k_p) v_p
 * with k_p, v_p the dequantized cache rows in the original basis (the
 * kernel rotates q forward when K is rotated and the output back when V is
 * rotated, which is the same result since the transform is orthonormal and
 * its own inverse).  L == 0 gives a zero row.
 *
 *   q            device, q_dtype, row (s, j) at element s*q_stride + j*head_dim
 *   out          device, out_dtype, contiguous [num_seqs, num_q_heads, head_dim]
 *   block_tables device int32; seq_lens device int32 [num_seqs]
 *   num_blocks   pool size for the block-id check (0 = do not check)
 *   head_dim 64/128/256; num_q_heads % num_kv_heads == 0 with ratio <= 8;
 *   block_size 8, 16 or 32
 *   sm_scale     logit scale; 0 selects 1/sqrt(head_dim)
 *   k_scale, v_scale  per-tensor FP8 scales (FP8 sides only)
 *   sparse_v_threshold  0 = exact; > 0 drops the V term of a position whose
 *                weight (normalised by the part of the sequence one warp has
 *                seen so far, which over-estimates the global weight, so it
 *                never drops more) is <= threshold; a 16-position slab whose
 *                weights are all dropped skips its V dequantization and P.V
 *                products.  The denominator keeps every weight.
 *   workspace    device, >= kvq_decode_workspace_bytes(...) bytes, 16-byte
 *                aligned, all zero on entry.  Every call leaves the whole
 *                workspace zero again, so one zeroed once can be reused by
 *                any number of calls, of any shapes, in stream order; calls
 *                that may run at the same time need separate workspaces.
 *   error_flag   optional device int32
 *
 * One kernel launch: persistent CTAs (one or two per SM) each take an equal
 * share of all (sequence, kv head) rows' 16-token slabs, each sequence
 * counted with a fixed extra cost for the unit of work it adds; rows shared
 * by several CTAs are merged by the last of them to finish, or by the CTA
 * holding the row's first slab when the others have finished before it. */
kvq_status kvq_paged_decode(
    const void* q, kvq_dtype q_dtype, int64_t q_stride,
    const void* k_cache, const void* v_cache,
    void* out, kvq_dtype out_dtype,
    const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens, int32_t num_seqs, int64_t num_blocks,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size,
    int64_t k_block_stride_bytes, int64_t v_block_stride_bytes,
    float sm_scale, float k_scale, float v_scale,
    int32_t sliding_window, float sparse_v_threshold,
    void* workspace, size_t workspace_bytes, kvq_format fmt,
    int32_t* error_flag, void* stream);

/* ---------------------------------------------------------- chunked prefill */

/* [BURN] attend with its causal mask for several query rows + repeat_kv;
 * [ATLAS] is_wht_rotated bookends.  Attention of a chunk of new query tokens
 * per sequence over the quantized paged cache, after the chunk's K/V rows
 * were written (kvq_cache_write).  The pages name chunked prefill over the
 * quantized cache as the step after the write; the semantics are read as:
 * sequence s holds L = seq_lens[s] positions, its C = cu_q[s+1] - cu_q[s]
 * queries (rows cu_q[s] .. cu_q[s+1]-1 of q) are the last C positions, and
 * query i at p = L - C + i attends to the positions [lo, p], lo = max(0,
 * p + 1 - sliding_window) (lo = 0 when sliding_window == 0):
 *   out[row, j, :] = sum_t softmax_t(sm_scale * q[row,j].k_t) v_t
 * over those positions, with kv head j / (num_q_heads/num_kv_heads).  A query
 * with p < 0 (C > L) gives a zero row.
 *
 *   q            device, q_dtype, row (r, j) at element r*q_stride + j*head_dim
 *   cu_q         device int32 [num_seqs + 1], cu_q[0] = 0, non-decreasing
 *   max_chunk    host: an upper bound of every C (sizes the launch; queries
 *                beyond it are not computed)
 *   out          device, out_dtype, contiguous [cu_q[num_seqs], num_q_heads, head_dim]
 *   other arguments as kvq_paged_decode (no workspace; no sparse-V skip).
 * One kernel launch: a CTA per (tile of query rows, kv head, sequence); the
 * products run on the tcgen05 tensor cores with accumulators in tensor
 * memory (128-row tiles for head_dim 64/128, 64-row tiles for 256). */
kvq_status kvq_paged_prefill(
    const void* q, kvq_dtype q_dtype, int64_t q_stride,
    const int32_t* cu_q, int32_t max_chunk,
    const void* k_cache, const void* v_cache,
    void* out, kvq_dtype out_dtype,
    const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens, int32_t num_seqs, int64_t num_blocks,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size,
    int64_t k_block_stride_bytes, int64_t v_block_stride_bytes,
    float sm_scale, float k_scale, float v_scale,
    int32_t sliding_window, kvq_format fmt,
    int32_t* error_flag, void* stream);

/* -------------------------------------------- decode without an allocation */

/* Bytes of the scratch array built into the library for
 * kvq_paged_decode_noalloc (per GPU that loads the library, kept until the
 * process exits). */
#define KVQ_NOALLOC_SCRATCH_BYTES (8u << 20)

/* The pages have no counterpart of this call; it exists for callers that
 * cannot allocate device memory - a runtime that has already given all
 * device memory to its own pool, a plugin host that forbids plugins from
 * allocating, or a latency-critical loop where cudaMalloc's possible device
 * synchronization is not acceptable.
 *
 * Same arguments and results as kvq_paged_decode, minus the workspace: the
 * partials and merge counters go to a fixed KVQ_NOALLOC_SCRATCH_BYTES array
 * compiled into the library (zero when the library loads; every call leaves
 * it zero).  Nothing is allocated (no cudaMalloc / cudaFree).
 *   - Returns KVQ_ERR_WORKSPACE if kvq_decode_workspace_bytes(...) for these
 *     arguments exceeds KVQ_NOALLOC_SCRATCH_BYTES.
 *   - The array's device address is looked up (cudaGetSymbolAddress) on
 *     every call, so a new context on the device (after cudaDeviceReset, or
 *     once the primary context was released and created again) is followed.
 *     A call made while its stream is being captured reuses the address that
 *     the last uncaptured call on the same device looked up, and returns
 *     KVQ_ERR_CUDA if there was none: make the first call on a device before
 *     any stream capture.
 *   - Every call shares the one array: calls whose kernels overlap on the GPU
 *     (different streams, or different host threads) race.  Serialize them.
 *   - A call that returns KVQ_ERR_CUDA after its launch was attempted has
 *     queued, on its stream, a clear of the part of the array it may have
 *     touched.  If the context itself has failed, the array is undefined
 *     until the context is created again, which loads a fresh, zero copy. */
kvq_status kvq_paged_decode_noalloc(
    const void* q, kvq_dtype q_dtype, int64_t q_stride,
    const void* k_cache, const void* v_cache,
    void* out, kvq_dtype out_dtype,
    const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens, int32_t num_seqs, int64_t num_blocks,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size,
    int64_t k_block_stride_bytes, int64_t v_block_stride_bytes,
    float sm_scale, float k_scale, float v_scale,
    int32_t sliding_window, float sparse_v_threshold, kvq_format fmt,
    int32_t* error_flag, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
