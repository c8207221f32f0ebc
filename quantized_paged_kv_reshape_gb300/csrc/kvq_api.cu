// C ABI of libkvq: format catalogue, host-side validation and dispatch.
//
// Catalogue: "spark_runtime/kv_cache.rs" (KvCacheDtype, kv_pair,
// is_wht_rotated, FromStr, block_bytes_dims, turbo*_data_bytes).  Launcher
// argument lists: "metrale_model_layers/layers/ops/kv_cache_bf16k_turbov.rs".
// Error convention (status codes, nothing thrown across the ABI, invalid
// arguments rejected before any launch): launchers there return Result<()>,
// FromStr bails on an unknown spelling.
#include "../../include/kvq.h"

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kvq_common.cuh"
#include "kvq_launch.h"

using namespace kvq;

namespace {

thread_local char g_err[512] = "";

kvq_status fail(kvq_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return st;
}

kvq_status ok() {
  g_err[0] = 0;
  return KVQ_OK;
}

struct Entry {
  const char* name;
  const char* alias;
  int k, v;
};

// [ATLAS] enum order; kv_pair gives (k, v).
const Entry kCatalog[KVQ_FMT_COUNT] = {
    {"bf16", nullptr, S_BF16, S_BF16},
    {"fp8", nullptr, S_FP8, S_FP8},
    {"nvfp4", nullptr, S_NVFP4, S_NVFP4},
    {"turbo4", nullptr, S_T4, S_T4},
    {"turbo3", nullptr, S_T3, S_T3},
    {"turbo2", nullptr, S_T2, S_T2},
    {"turbo8", nullptr, S_T8, S_T8},
    {"turbo4k_turbo3v", "turbo4k3v", S_T4, S_T3},
    {"turbo4k_turbo8v", "turbo4k8v", S_T4, S_T8},
    {"turbo3k_turbo8v", "turbo3k8v", S_T3, S_T8},
    {"bf16k_turbo4v", "bf16k4v", S_BF16, S_T4},
    {"bf16k_turbo3v", "bf16k3v", S_BF16, S_T3},
    {"fp8k_turbo4v", "fp8k4v", S_FP8, S_T4},
    {"fp8k_turbo3v", "fp8k3v", S_FP8, S_T3},
    {"bf16k_turbo2v", "bf16k2v", S_BF16, S_T2},
    {"fp8k_turbo2v", "fp8k2v", S_FP8, S_T2},
};

bool fmt_ok(kvq_format f) { return (int)f >= 0 && (int)f < KVQ_FMT_COUNT; }

int side_of(kvq_format f, int side) { return side == KVQ_SIDE_K ? kCatalog[f].k : kCatalog[f].v; }

int64_t data_bytes(int s, int64_t elems) { return elems * side_bits(s) / 8; }
int64_t scale_bytes(int s, int64_t elems) { return elems / kGroup * side_scale_bytes(s); }

// ------------------------------------------------------------ codebooks
//
// Lloyd-Max quantizer of N(0,1) ("spark_runtime/kv_cache.rs", Turbo4/3/2:
// optimal Gaussian codebook with 16/8/4 levels).  Fixed-point iteration of
// the two optimality conditions in double precision: thresholds at the
// midpoints of adjacent levels, each level at the conditional mean of its
// cell, (pdf(a) - pdf(b)) / (cdf(b) - cdf(a)) for the cell (a, b].  Stops
// when no level moves by more than 1e-15; the result is symmetrised.

double npdf(double x) { return std::isinf(x) ? 0.0 : std::exp(-0.5 * x * x) / std::sqrt(2.0 * M_PI); }
double ncdf(double x) {
  if (std::isinf(x)) return x > 0 ? 1.0 : 0.0;
  return 0.5 * std::erfc(-x / std::sqrt(2.0));
}

void lloyd_max(int bits, double* c) {
  const int n = 1 << bits;
  double cn[16], t[15];
  for (int i = 0; i < n; ++i) c[i] = -2.0 + 4.0 * i / (n - 1);
  for (int it = 0; it < 1000000; ++it) {
    for (int i = 0; i + 1 < n; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
    double moved = 0.0;
    for (int i = 0; i < n; ++i) {
      const double a = i == 0 ? -INFINITY : t[i - 1];
      const double b = i == n - 1 ? INFINITY : t[i];
      cn[i] = (npdf(a) - npdf(b)) / (ncdf(b) - ncdf(a));
      moved = std::fmax(moved, std::fabs(cn[i] - c[i]));
    }
    for (int i = 0; i < n; ++i) c[i] = cn[i];
    if (moved < 1e-15) break;
  }
  for (int i = 0; i < n / 2; ++i) {
    const double m = 0.5 * (c[n - 1 - i] - c[i]);
    c[i] = -m;
    c[n - 1 - i] = m;
  }
}

Codebooks g_cb;
std::once_flag g_cb_once;

const Codebooks& codebooks() {
  std::call_once(g_cb_once, [] {
    double c[16];
    auto fill = [&](int bits, float* lv, float* th) {
      lloyd_max(bits, c);
      const int n = 1 << bits;
      for (int i = 0; i < n; ++i) lv[i] = (float)c[i];
      for (int i = 0; i + 1 < n; ++i) th[i] = (float)(0.5 * (c[i] + c[i + 1]));
    };
    fill(4, g_cb.lv4, g_cb.th4);
    fill(3, g_cb.lv3, g_cb.th3);
    fill(2, g_cb.lv2, g_cb.th2);
    // The cache write's Turbo4/3 search buckets quotients by fmaf(v, 4, 2^20 +
    // 128.5) rounded to eighths: edges (k - 128.5) / 4 blur by up to 1/64, so
    // no threshold may lie that close to one.
    auto check_edges = [](const float* th, int n) {
      for (int i = 0; i < n; ++i) {
        const double e = std::floor(4.0 * th[i] + 128.5) - 128.5;
        const double d = std::fmin(std::fabs(th[i] - e / 4.0), std::fabs(th[i] - (e + 1.0) / 4.0));
        if (d < 1.0 / 48) std::abort();   // the blur is 1/64; Turbo4 keeps 0.0257
      }
    };
    check_edges(g_cb.th4, 15);
    check_edges(g_cb.th3, 7);
    static const float e2m1_mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
    for (int c2 = 0; c2 < 16; ++c2) g_cb.e2m1[c2] = (c2 & 8) ? -e2m1_mag[c2 & 7] : e2m1_mag[c2 & 7];
  });
  return g_cb;
}

// ------------------------------------------------------------ devices

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cache[dev] = n;
  return n;
}

// Decode partition.  The decode runs persistent CTAs, two per SM (the
// launcher picks the instance's count, at most four): R per kv head, each
// on an equal share of the sequences' 16-token slabs (measured on GB300: one
// balanced wave of long CTAs beats more, shorter split CTAs, which pay the
// prologue and merge more often and leave a partial last wave).  kmax is the
// number of partial slots per (sequence, query head): a row of n slabs spans
// at most floor((n - 1) / per_cta) + 2 CTAs, and the kernel keeps per_cta >=
// max_n / (kmax - 1) for the longest row max_n.  Here kmax = min(R_max + 1,
// (max_n_bound - 1) / 16 + 2): with at least 16 slabs per CTA for the longest
// possible row, or one slot per CTA of a head.
struct DecodePlan {
  int sms, max_ranges, min_slabs, kmax;
};

// At most 4 CTAs per SM for any instance (the launcher picks its own count).
DecodePlan plan_decode(int nkv, int bs, int max_blocks, int window, int sms) {
  DecodePlan p{};
  p.sms = sms > 0 ? sms : 148;
  p.max_ranges = std::max(1, 4 * p.sms / std::max(1, nkv));
  p.min_slabs = 16;
  int64_t max_n = ((int64_t)max_blocks * bs + 15) / 16;
  if (window > 0) max_n = std::min<int64_t>(max_n, (window + 15) / 16 + 1);
  if (max_n < 1) max_n = 1;
  const int64_t by_len = (max_n - 1) / p.min_slabs + 2;
  p.kmax = (int)std::min<int64_t>(by_len, p.max_ranges + 1);
  return p;
}

// Workspace: partials [num_seqs][nq][kmax][hd + 4] fp32, then the partial
// counts [num_seqs][nkv] int32.
size_t part_bytes(int num_seqs, int nq, int hd, const DecodePlan& p) {
  return (size_t)num_seqs * nq * p.kmax * (hd + 4) * sizeof(float);
}
size_t workspace_need(int num_seqs, int nq, int nkv, int hd, const DecodePlan& p) {
  return part_bytes(num_seqs, nq, hd, p) + ((size_t)num_seqs * nkv * sizeof(int32_t) + 15) / 16 * 16;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// 1/x where x is a power of two whose reciprocal is a normal float (then x *
// (1/x) rounds exactly like a division by x), else 0.
float exact_reciprocal(float x) {
  int e = 0;
  const float m = std::frexp(x, &e);
  if (!(x > 0.f) || !std::isfinite(x) || m != 0.5f) return 0.f;
  const float r = 1.0f / x;
  return (std::isnormal(r) && r * x == 1.0f) ? r : 0.f;
}

// Multiplier and shifts of Granlund and Montgomery's round-up division by d
// ("Division by invariant integers using multiplication", 1994, Figure 4.1):
// with l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1, every 32-bit n
// gives n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0), t = umulhi(m, n).
void set_fast_div(uint32_t d, uint32_t& m, uint32_t& s1, uint32_t& s2) {
  uint32_t l = 0;
  while (l < 32 && ((uint64_t)1 << l) < d) ++l;
  m = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << l) - d)) / d + 1);
  s1 = l < 1 ? l : 1;
  s2 = l > 1 ? l - 1 : 0;
}

int rmax_for(int rep) { return rep <= 1 ? 1 : rep <= 2 ? 2 : rep <= 4 ? 4 : rep <= 8 ? 8 : 0; }

}  // namespace

namespace kvq {
// Lets other translation units of the library report a message through
// kvq_last_error().
void record_error(const char* msg) { snprintf(g_err, sizeof g_err, "%s", msg); }
}  // namespace kvq

extern "C" {

kvq_status kvq_format_from_string(const char* name, kvq_format* out) {
  if (!name || !out) return fail(KVQ_ERR_ARG, "null argument");
  for (int i = 0; i < KVQ_FMT_COUNT; ++i) {
    if (!strcmp(name, kCatalog[i].name) || (kCatalog[i].alias && !strcmp(name, kCatalog[i].alias))) {
      *out = (kvq_format)i;
      return ok();
    }
  }
  return fail(KVQ_ERR_FORMAT, "unsupported kv cache format '%s'", name);
}

const char* kvq_format_name(kvq_format fmt) { return fmt_ok(fmt) ? kCatalog[fmt].name : nullptr; }

int kvq_side_format(kvq_format fmt, int side) {
  if (!fmt_ok(fmt) || (side != KVQ_SIDE_K && side != KVQ_SIDE_V)) return -1;
  return side_of(fmt, side);
}

int kvq_side_is_rotated(kvq_format fmt, int side) {
  const int s = kvq_side_format(fmt, side);
  return s < 0 ? -1 : (side_rotated(s) ? 1 : 0);
}

int64_t kvq_block_bytes(kvq_format fmt, int side, int32_t bs, int32_t nkv, int32_t hd) {
  const int s = kvq_side_format(fmt, side);
  if (s < 0 || bs <= 0 || nkv <= 0 || hd <= 0 || hd % kGroup) return -1;
  const int64_t e = (int64_t)bs * nkv * hd;
  return data_bytes(s, e) + scale_bytes(s, e);
}

int64_t kvq_data_section_bytes(kvq_format fmt, int side, int32_t bs, int32_t nkv, int32_t hd) {
  const int s = kvq_side_format(fmt, side);
  if (s < 0 || bs <= 0 || nkv <= 0 || hd <= 0 || hd % kGroup) return -1;
  return data_bytes(s, (int64_t)bs * nkv * hd);
}

kvq_status kvq_codebook(int bits, float* levels, float* thresholds) {
  const Codebooks& cb = codebooks();
  const float* lv;
  const float* th;
  switch (bits) {
    case 4: lv = cb.lv4; th = cb.th4; break;
    case 3: lv = cb.lv3; th = cb.th3; break;
    case 2: lv = cb.lv2; th = cb.th2; break;
    default: return fail(KVQ_ERR_ARG, "codebook bits must be 2, 3 or 4 (got %d)", bits);
  }
  const int n = 1 << bits;
  if (levels) memcpy(levels, lv, sizeof(float) * n);
  if (thresholds) memcpy(thresholds, th, sizeof(float) * (n - 1));
  return ok();
}

const char* kvq_status_string(kvq_status st) {
  switch (st) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_ARG: return "invalid argument";
    case KVQ_ERR_FORMAT: return "unsupported format";
    case KVQ_ERR_SHAPE: return "unsupported shape";
    case KVQ_ERR_ALIGN: return "misaligned pointer or stride";
    case KVQ_ERR_WORKSPACE: return "workspace too small";
    case KVQ_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char* kvq_last_error(void) { return g_err; }

kvq_status kvq_cache_write(const void* key, const void* value, kvq_dtype in_dtype, void* k_cache,
                           void* v_cache, const int64_t* slot_mapping, int32_t num_tokens,
                           int64_t num_blocks, int32_t nkv, int32_t hd, int32_t bs,
                           int64_t key_stride, int64_t value_stride, int64_t k_bstride,
                           int64_t v_bstride, float k_scale, float v_scale, kvq_format fmt,
                           int32_t* error_flag, void* stream) {
  if (!fmt_ok(fmt)) return fail(KVQ_ERR_FORMAT, "format %d out of range", (int)fmt);
  const int ks = side_of(fmt, 0), vs = side_of(fmt, 1);
  if (in_dtype != KVQ_DTYPE_F32 && in_dtype != KVQ_DTYPE_BF16)
    return fail(KVQ_ERR_FORMAT, "in_dtype must be f32 or bf16");
  if (num_tokens < 0 || num_blocks < 0) return fail(KVQ_ERR_ARG, "negative count");
  if (hd != 64 && hd != 128 && hd != 256) return fail(KVQ_ERR_SHAPE, "head_dim %d not in {64,128,256}", hd);
  if (nkv < 1 || bs < 1) return fail(KVQ_ERR_SHAPE, "num_kv_heads and block_size must be >= 1");
  if (num_tokens == 0) return ok();
  if ((int64_t)num_tokens * nkv * 2 >= (int64_t)1 << 31)
    return fail(KVQ_ERR_SHAPE, "num_tokens * num_kv_heads * 2 must be below 2^31 (split the call)");
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return fail(KVQ_ERR_ARG, "null pointer");
  if (key_stride < (int64_t)nkv * hd || value_stride < (int64_t)nkv * hd)
    return fail(KVQ_ERR_ARG, "key/value stride smaller than num_kv_heads*head_dim");
  const int64_t kb = kvq_block_bytes(fmt, 0, bs, nkv, hd), vb = kvq_block_bytes(fmt, 1, bs, nkv, hd);
  if (k_bstride < kb || v_bstride < vb) return fail(KVQ_ERR_ARG, "block stride below block bytes");
  if (k_bstride % 16 || v_bstride % 16 || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(KVQ_ERR_ALIGN, "cache pointers and block strides must be 16-byte aligned");
  if ((ks == S_FP8 && !(k_scale > 0.f && std::isfinite(k_scale))) ||
      (vs == S_FP8 && !(v_scale > 0.f && std::isfinite(v_scale))))
    return fail(KVQ_ERR_ARG, "FP8 side needs a finite scale > 0");
  const Codebooks& cb = codebooks();
  const bool bf = in_dtype == KVQ_DTYPE_BF16;
  const int el = bf ? 2 : 4;
  // every lane loads 16 consecutive elements (one scale group) as 16-byte
  // vectors: the rows' starts must keep that alignment
  const bool vec = aligned16(key) && aligned16(value) && (key_stride * el) % 16 == 0 &&
                   (value_stride * el) % 16 == 0;
  WriteArgs a{};
  a.key = key;
  a.value = value;
  a.k_cache = (uint8_t*)k_cache;
  a.v_cache = (uint8_t*)v_cache;
  a.slots = slot_mapping;
  a.num_tokens = num_tokens;
  a.num_slots = num_blocks * bs;
  a.nkv = nkv;
  a.bs = bs;
  a.bs_shift = (bs & (bs - 1)) == 0 ? __builtin_ctz((unsigned)bs) : -1;
  a.key_stride = key_stride;
  a.value_stride = value_stride;
  a.k_bstride = k_bstride;
  a.v_bstride = v_bstride;
  a.k_dsec = kvq_data_section_bytes(fmt, 0, bs, nkv, hd);
  a.v_dsec = kvq_data_section_bytes(fmt, 1, bs, nkv, hd);
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.k_inv = exact_reciprocal(k_scale);
  a.v_inv = exact_reciprocal(v_scale);
  a.inv_sqrt_hd = (float)(1.0 / std::sqrt((double)hd));
  a.k_side = ks;
  a.v_side = vs;
  set_fast_div((uint32_t)nkv, a.nkv_m, a.nkv_s1, a.nkv_s2);
  a.err = error_flag;
  cudaError_t e = launch_cache_write(a, cb, hd, bf, vec, sm_count(), (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "cache write launch: %s", cudaGetErrorString(e));
  return ok();
}

int32_t kvq_decode_path(kvq_format fmt, int32_t hd, int32_t nkv, int32_t bs) {
  if (!fmt_ok(fmt) || (hd != 64 && hd != 128 && hd != 256) || nkv < 1 ||
      (bs != 8 && bs != 16 && bs != 32))
    return -1;
  return decode_tma_supported(side_of(fmt, 0), side_of(fmt, 1), hd, nkv, bs) ? 1 : 0;
}

size_t kvq_decode_workspace_bytes(int32_t num_seqs, int32_t nq, int32_t nkv, int32_t hd, int32_t bs,
                                  int32_t max_blocks, int32_t window, kvq_format fmt) {
  if (!fmt_ok(fmt) || num_seqs < 0 || nq < 1 || nkv < 1 || hd < 1 || bs < 1 || max_blocks < 1 ||
      window < 0 || (bs != 8 && bs != 16 && bs != 32))
    return 0;
  return workspace_need(num_seqs, nq, nkv, hd, plan_decode(nkv, bs, max_blocks, window, sm_count()));
}

kvq_status kvq_paged_decode(const void* q, kvq_dtype q_dtype, int64_t q_stride, const void* k_cache,
                            const void* v_cache, void* out, kvq_dtype out_dtype,
                            const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                            int32_t num_seqs, int64_t num_blocks, int32_t nq, int32_t nkv, int32_t hd,
                            int32_t bs, int64_t k_bstride, int64_t v_bstride, float sm_scale,
                            float k_scale, float v_scale, int32_t window, float sparse_v_threshold,
                            void* workspace, size_t workspace_bytes, kvq_format fmt,
                            int32_t* error_flag, void* stream) {
  if (!fmt_ok(fmt)) return fail(KVQ_ERR_FORMAT, "format %d out of range", (int)fmt);
  const int ks = side_of(fmt, 0), vs = side_of(fmt, 1);
  if ((q_dtype != KVQ_DTYPE_F32 && q_dtype != KVQ_DTYPE_BF16) ||
      (out_dtype != KVQ_DTYPE_F32 && out_dtype != KVQ_DTYPE_BF16))
    return fail(KVQ_ERR_FORMAT, "q/out dtype must be f32 or bf16");
  if (hd != 64 && hd != 128 && hd != 256) return fail(KVQ_ERR_SHAPE, "head_dim %d not in {64,128,256}", hd);
  if (bs != 8 && bs != 16 && bs != 32) return fail(KVQ_ERR_SHAPE, "block_size %d not in {8,16,32}", bs);
  if (nkv < 1 || nq < 1 || nq % nkv) return fail(KVQ_ERR_SHAPE, "num_q_heads must be a multiple of num_kv_heads");
  const int rep = nq / nkv;
  const int rmax = rmax_for(rep);
  if (!rmax) return fail(KVQ_ERR_SHAPE, "grouped-query ratio %d above 8", rep);
  if (num_seqs < 0 || num_blocks < 0 || window < 0) return fail(KVQ_ERR_ARG, "negative count");
  if (!(sparse_v_threshold >= 0.f && std::isfinite(sparse_v_threshold)))
    return fail(KVQ_ERR_ARG, "sparse_v_threshold must be finite and >= 0");
  if (!std::isfinite(sm_scale)) return fail(KVQ_ERR_ARG, "sm_scale must be finite");
  if (num_seqs == 0) return ok();
  if (max_blocks < 1) return fail(KVQ_ERR_ARG, "max_blocks_per_seq must be >= 1");
  if (!q || !k_cache || !v_cache || !out || !block_tables || !seq_lens || !workspace)
    return fail(KVQ_ERR_ARG, "null pointer");
  if (q_stride < (int64_t)nq * hd) return fail(KVQ_ERR_ARG, "q_stride smaller than num_q_heads*head_dim");
  const int64_t kb = kvq_block_bytes(fmt, 0, bs, nkv, hd), vb = kvq_block_bytes(fmt, 1, bs, nkv, hd);
  if (k_bstride < kb || v_bstride < vb) return fail(KVQ_ERR_ARG, "block stride below block bytes");
  if (k_bstride % 16 || v_bstride % 16 || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(workspace))
    return fail(KVQ_ERR_ALIGN, "caches, block strides and workspace must be 16-byte aligned");
  if ((ks == S_FP8 && !(k_scale > 0.f && std::isfinite(k_scale))) ||
      (vs == S_FP8 && !(v_scale > 0.f && std::isfinite(v_scale))))
    return fail(KVQ_ERR_ARG, "FP8 side needs a finite scale > 0");
  const DecodePlan p = plan_decode(nkv, bs, max_blocks, window, sm_count());
  const size_t need = workspace_need(num_seqs, nq, nkv, hd, p);
  if (workspace_bytes < need)
    return fail(KVQ_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, need);
  if (!decode_tc_supported(ks, vs)) return fail(KVQ_ERR_FORMAT, "no decode instance for this pair");
  const Codebooks& cb = codebooks();
  const double scale = sm_scale == 0.f ? 1.0 / std::sqrt((double)hd) : (double)sm_scale;
  DecodeArgs a{};
  a.q = q;
  a.q_stride = q_stride;
  a.q_bf16 = q_dtype == KVQ_DTYPE_BF16;
  a.k_cache = (const uint8_t*)k_cache;
  a.v_cache = (const uint8_t*)v_cache;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.num_seqs = num_seqs;
  a.num_blocks = num_blocks;
  a.nq = nq;
  a.nkv = nkv;
  a.rep = rep;
  a.bs = bs;
  a.k_bstride = k_bstride;
  a.v_bstride = v_bstride;
  a.k_dsec = kvq_data_section_bytes(fmt, 0, bs, nkv, hd);
  a.v_dsec = kvq_data_section_bytes(fmt, 1, bs, nkv, hd);
  a.score_scale = (float)(scale * M_LOG2E * (ks == S_FP8 ? (double)k_scale : 1.0));
  a.v_mult = vs == S_FP8 ? v_scale : 1.0f;
  a.inv_sqrt_hd = (float)(1.0 / std::sqrt((double)hd));
  a.window = window;
  a.sparse_thr = sparse_v_threshold;
  a.sms = p.sms;
  a.max_ranges = p.max_ranges;
  a.kmax = p.kmax;
  a.part = (float*)workspace;
  a.counters = (int32_t*)((uint8_t*)workspace + part_bytes(num_seqs, nq, hd, p));
  a.out = out;
  a.out_bf16 = out_dtype == KVQ_DTYPE_BF16;
  a.err = error_flag;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = decode_tma_supported(ks, vs, hd, nkv, bs) ? launch_decode_tma(ks, vs, hd, a, cb, st)
                                                            : launch_decode_tc(ks, vs, hd, a, cb, st);
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return ok();
}

kvq_status kvq_paged_prefill(const void* q, kvq_dtype q_dtype, int64_t q_stride, const int32_t* cu_q,
                             int32_t max_chunk, const void* k_cache, const void* v_cache, void* out,
                             kvq_dtype out_dtype, const int32_t* block_tables, int32_t max_blocks,
                             const int32_t* seq_lens, int32_t num_seqs, int64_t num_blocks, int32_t nq,
                             int32_t nkv, int32_t hd, int32_t bs, int64_t k_bstride, int64_t v_bstride,
                             float sm_scale, float k_scale, float v_scale, int32_t window,
                             kvq_format fmt, int32_t* error_flag, void* stream) {
  if (!fmt_ok(fmt)) return fail(KVQ_ERR_FORMAT, "format %d out of range", (int)fmt);
  const int ks = side_of(fmt, 0), vs = side_of(fmt, 1);
  if ((q_dtype != KVQ_DTYPE_F32 && q_dtype != KVQ_DTYPE_BF16) ||
      (out_dtype != KVQ_DTYPE_F32 && out_dtype != KVQ_DTYPE_BF16))
    return fail(KVQ_ERR_FORMAT, "q/out dtype must be f32 or bf16");
  if (hd != 64 && hd != 128 && hd != 256) return fail(KVQ_ERR_SHAPE, "head_dim %d not in {64,128,256}", hd);
  if (bs != 8 && bs != 16 && bs != 32) return fail(KVQ_ERR_SHAPE, "block_size %d not in {8,16,32}", bs);
  if (nkv < 1 || nq < 1 || nq % nkv) return fail(KVQ_ERR_SHAPE, "num_q_heads must be a multiple of num_kv_heads");
  const int rep = nq / nkv;
  const int rp = rmax_for(rep);
  if (!rp) return fail(KVQ_ERR_SHAPE, "grouped-query ratio %d above 8", rep);
  if (num_seqs < 0 || num_blocks < 0 || window < 0 || max_chunk < 0) return fail(KVQ_ERR_ARG, "negative count");
  if (!std::isfinite(sm_scale)) return fail(KVQ_ERR_ARG, "sm_scale must be finite");
  if (num_seqs == 0 || max_chunk == 0) return ok();
  if (max_blocks < 1) return fail(KVQ_ERR_ARG, "max_blocks_per_seq must be >= 1");
  if (!q || !cu_q || !k_cache || !v_cache || !out || !block_tables || !seq_lens)
    return fail(KVQ_ERR_ARG, "null pointer");
  if (q_stride < (int64_t)nq * hd) return fail(KVQ_ERR_ARG, "q_stride smaller than num_q_heads*head_dim");
  const int64_t kb = kvq_block_bytes(fmt, 0, bs, nkv, hd), vb = kvq_block_bytes(fmt, 1, bs, nkv, hd);
  if (k_bstride < kb || v_bstride < vb) return fail(KVQ_ERR_ARG, "block stride below block bytes");
  if (k_bstride % 16 || v_bstride % 16 || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(KVQ_ERR_ALIGN, "caches and block strides must be 16-byte aligned");
  if ((ks == S_FP8 && !(k_scale > 0.f && std::isfinite(k_scale))) ||
      (vs == S_FP8 && !(v_scale > 0.f && std::isfinite(v_scale))))
    return fail(KVQ_ERR_ARG, "FP8 side needs a finite scale > 0");
  if (!decode_tc_supported(ks, vs)) return fail(KVQ_ERR_FORMAT, "no prefill instance for this pair");
  const Codebooks& cb = codebooks();
  const double scale = sm_scale == 0.f ? 1.0 / std::sqrt((double)hd) : (double)sm_scale;
  PrefillArgs a{};
  a.q = q;
  a.q_stride = q_stride;
  a.q_bf16 = q_dtype == KVQ_DTYPE_BF16;
  a.cu_q = cu_q;
  a.k_cache = (const uint8_t*)k_cache;
  a.v_cache = (const uint8_t*)v_cache;
  a.out = out;
  a.out_bf16 = out_dtype == KVQ_DTYPE_BF16;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.num_seqs = num_seqs;
  a.num_blocks = num_blocks;
  a.nq = nq;
  a.nkv = nkv;
  a.rep = rep;
  a.rp = rp;
  a.bs = bs;
  a.k_bstride = k_bstride;
  a.v_bstride = v_bstride;
  a.k_dsec = kvq_data_section_bytes(fmt, 0, bs, nkv, hd);
  a.v_dsec = kvq_data_section_bytes(fmt, 1, bs, nkv, hd);
  a.score_scale = (float)(scale * M_LOG2E * (ks == S_FP8 ? (double)k_scale : 1.0));
  a.v_mult = vs == S_FP8 ? v_scale : 1.0f;
  a.inv_sqrt_hd = (float)(1.0 / std::sqrt((double)hd));
  a.window = window;
  a.err = error_flag;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e;
  switch (ks) {
    case S_BF16: e = launch_pf_k_bf16(vs, hd, a, cb, max_chunk, st); break;
    case S_FP8: e = launch_pf_k_fp8(vs, hd, a, cb, max_chunk, st); break;
    case S_T4: e = launch_pf_k_t4(vs, hd, a, cb, max_chunk, st); break;
    case S_T3: e = launch_pf_k_t3(vs, hd, a, cb, max_chunk, st); break;
    case S_T2: e = launch_pf_k_t2(vs, hd, a, cb, max_chunk, st); break;
    case S_T8: e = launch_pf_k_t8(vs, hd, a, cb, max_chunk, st); break;
    case S_NVFP4: e = launch_pf_k_nvfp4(vs, hd, a, cb, max_chunk, st); break;
    default: e = cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // extern "C"
