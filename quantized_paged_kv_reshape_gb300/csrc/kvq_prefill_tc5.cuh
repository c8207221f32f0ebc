// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory), head_dim 64, 128 and 256.
//
// "combs_models/kv.rs" attend with the causal / window mask and repeat_kv,
// "spark_runtime/kv_cache.rs" is_wht_rotated bookends: query i of sequence
// s's chunk sits at p = L - C + i and attends to [max(0, p + 1 - W), p].
//
// One CTA (16 warps) per (tile of R score rows = QT query tokens x RP
// heads, kv head, sequence), R = 128 for head_dim 64/128 and R = 64 for
// head_dim 256 (whose planes would not fit a 128-row tile).  With R = 128
// score row r is tensor-memory lane r, held by threads r + 128 i, i = 0..3,
// each with a quarter of its columns; with R = 64 (M = 64 accumulators) row
// r sits in lane 32 floor(r / 16) + r mod 16, so the first 16 lanes of each
// warp hold rows.  Per step of T KV positions (T = 64, or 32 for head_dim
// 256; raw cache rows staged by cp.async two steps ahead):
//   one thread issues S[R x T] = Q . K^T (tcgen05.mma kind::f16, fp32 in
//   tensor memory; K dequantized during the previous step) and commits it
//   to an mbarrier;
//   meanwhile all threads dequantize V into the V^T [hd x T] operand plane
//   (16-bit hi + lo parts where one 16-bit value is not exact);
//   each thread reads its quarter score row (tcgen05.ld), masks it (only on
//   steps that cut a row's range); the quarters' maxima meet in shared
//   memory; it writes its quarter P row (hi + lo) to shared memory; the O
//   accumulator in tensor memory is rescaled only when a row's maximum grew
//   by more than 2^8 since the last rescale (P <= 2^8 otherwise: exact
//   enough in fp32 and in the 16-bit parts);
//   one thread issues O[R x hd] += P . V, and meanwhile all threads
//   dequantize the next step's K into the K [T x hd] plane.
// q (scaled by the score scale) and P carry hi + lo 16-bit parts like the
// decode.  Operands are K-major without swizzle (8 x 16-byte core
// matrices; strides in t5::cm).
#pragma once

#include <math_constants.h>

#include "kvq_prefill.cuh"

namespace kvq {

namespace t5 {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// Shared-memory matrix descriptor: K-major, no swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor of kind::f16: fp32 accumulator, A and B both bf16
// or both fp16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc(bool bf, int M, int N) {
  return (1u << 4) | ((bf ? 1u : 0u) << 7) | ((bf ? 1u : 0u) << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
               : "memory");
}
// Bounded wait for the completion of phase `parity` of an mbarrier.
__device__ __forceinline__ bool wait(uint32_t mbar, uint32_t parity) {
  for (int it = 0; it < (1 << 24); ++it) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
// Generic-proxy shared-memory writes made visible to the tensor cores.
__device__ __forceinline__ void fence_smem_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
      "[%16];\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
        "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                 "=r"(v[7])
               : "r"(taddr));
}
__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]));
}
// 2^x (PTX ex2.approx.ftz: relative error ~2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// Operand planes: K-major core matrices (8 rows x 16 bytes, rows 16 bytes
// apart) placed LBO = 144 bytes apart along K and SBO = (KD / 8) x 144 + 16
// bytes apart along the rows; the 16-byte gaps spread the stores of
// consecutive threads over the shared-memory banks.
constexpr int kLbo = 144;
template <int KD>
constexpr int sbo() { return (KD / 8) * kLbo + 16; }
template <int R, int KD>
constexpr int plane_bytes() { return (R / 8) * sbo<KD>(); }
// Element offset (16-bit units) of (row r, k) in a plane with KD columns.
template <int KD>
__device__ __forceinline__ int cm(int r, int k) {
  return ((r >> 3) * sbo<KD>() + (k >> 3) * kLbo + (r & 7) * 16 + (k & 7) * 2) >> 1;
}

}  // namespace t5

// Codebook sides (Turbo2/3/4, NVFP4): a table of code pairs, entry
// (c0 | c1 << bits) = fp16x2 (hi(c0), hi(c1)) and (lo(c0), lo(c1)) with the
// level split into two parts of 7 significant bits, PCOPY copies
// interleaved against bank conflicts.  A part times an E4M3 group scale (4
// significant bits) is exact in fp16.
constexpr int PCOPY = 4;
template <int S>
constexpr int pair_entries() { return side_codebook(S) ? (1 << (2 * code_bits(S))) * PCOPY : 0; }

template <int S>
__device__ __forceinline__ void t5_fill_pairs(uint2* lut, const Codebooks& cb, int tid, int nt) {
  if constexpr (side_codebook(S)) {
    const float* lv = side_levels<S>(cb);
    constexpr int B = code_bits(S), n = 1 << B;
    for (int e = tid; e < pair_entries<S>(); e += nt) {
      const int pr = e / PCOPY;
      const float c0 = lv[pr & (n - 1)], c1 = lv[pr >> B];
      const float h0 = tc::round_sig7(c0), h1 = tc::round_sig7(c1);
      const float l0 = tc::round_sig7(c0 - h0), l1 = tc::round_sig7(c1 - h1);
      lut[e] = make_uint2(tc::pack2<false>(h0, h1), tc::pack2<false>(l0, l1));
    }
  }
}

// Elements d0 .. d0 + 7 (d0 % 8 == 0, one scale group) of a staged codebook
// row as fp16x2 hi / lo pairs: one table entry per code pair, scaled in fp16.
template <int S>
__device__ __forceinline__ void t5_dequant_pairs(const uint8_t* row, const uint8_t* srow, int d0,
                                                 const uint2* lut, int cpy, uint32_t (&hw)[4],
                                                 uint32_t (&lw)[4]) {
  constexpr int B = code_bits(S);
  uint32_t w;
  if constexpr (B == 4) {
    w = *reinterpret_cast<const uint32_t*>(row + d0 / 2);
  } else if constexpr (B == 2) {
    w = *reinterpret_cast<const uint16_t*>(row + d0 / 4);
  } else {   // 3-bit codes: 24 bits from byte 3 d0 / 8
    const uint8_t* p = row + 3 * (d0 / 8);
    w = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16);
  }
  const uint32_t sb = srow[d0 / kGroup];
  const uint32_t sc2 = tc::e4m3x2_f16x2(sb | (sb << 8));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t pr = (w >> (2 * B * i)) & ((1u << (2 * B)) - 1u);
    const uint2 e = lut[pr * PCOPY + cpy];
    hw[i] = tc::hmul2(e.x, sc2);
    lw[i] = PfSide<S>::PLANES == 2 ? tc::hmul2(e.y, sc2) : 0u;
  }
}

template <int KS, int VS, int HD>
struct T5Cfg {
  static_assert(HD == 64 || HD == 128 || HD == 256, "tensor-memory prefill: head_dim 64, 128 or 256");
  // M of the accumulators (score rows per tile) and KV positions per step;
  // NSPLIT column parts per row (the four warps of a lane quadrant)
  static constexpr int NT = 512, ROWS = HD == 256 ? 64 : 128, TOK = HD == 256 ? 32 : 64, NSPLIT = 4;
  // tokens per V dequantization item: 2, so that every thread has an item
  // (4 per item measured 1-2% slower at head_dim 128 on GB300)
  static constexpr int VTPI = 2;
  static constexpr int KPL = PfSide<KS>::PLANES, VPL = PfSide<VS>::PLANES;
  static constexpr int KROW = SideGeom<KS, HD>::ROW, KSROW = SideGeom<KS, HD>::SROW;
  static constexpr int VROW = SideGeom<VS, HD>::ROW, VSROW = SideGeom<VS, HD>::SROW;
  static constexpr int R_KS = align_up(TOK * KROW, 16);
  static constexpr int R_V = R_KS + align_up(TOK * KSROW, 16);
  static constexpr int R_VS = R_V + align_up(TOK * VROW, 16);
  static constexpr int RAW = R_VS + align_up(TOK * VSROW, 16);
  static constexpr int QB = t5::plane_bytes<ROWS, HD>(), KB = t5::plane_bytes<TOK, HD>();
  static constexpr int VB = t5::plane_bytes<HD, TOK>(), PB = t5::plane_bytes<ROWS, TOK>();
  static constexpr int OFF_Q = 0;                     // q hi, q lo
  static constexpr int OFF_K = OFF_Q + 2 * QB;        // K planes [TOK x HD]
  static constexpr int OFF_V = OFF_K + KPL * KB;      // V^T planes [HD x TOK]
  static constexpr int OFF_P = OFF_V + VPL * VB;      // P hi, lo [ROWS x TOK]
  static constexpr int OFF_RAW = OFF_P + 2 * PB;      // raw rows, two buffers
  static constexpr int OFF_VROW = OFF_RAW + 2 * RAW;  // [2][TOK] row valid flags
  static constexpr int OFF_LV = OFF_VROW + 2 * TOK;   // level tables [2][2][16] fp32
  static constexpr bool SHARE_PAIRS = KS == VS;
  static constexpr int OFF_PK = OFF_LV + 256;          // code-pair tables (K, then V unless shared)
  static constexpr int OFF_PV = OFF_PK + (SHARE_PAIRS ? 0 : pair_entries<KS>() * 8);
  static constexpr int OFF_MX = OFF_PV + pair_entries<VS>() * 8;  // [NSPLIT][ROWS] part-row maxima / sums
  static constexpr int OFF_BAR = OFF_MX + NSPLIT * ROWS * 4;  // 2 mbarriers, tensor-memory address
  // Block ids of the tile's first BLKC pages staged in shared memory at the
  // start (measured on GB300, 8 x 4096 with 512-token chunks: Turbo4 1359 ->
  // 1335 us, head_dim 256 BF16 / Turbo2 / Turbo8 4142 / 5958 / 5668 -> 4047 /
  // 5866 / 5628 us); BF16 and FP8 K at head_dim 64/128 load them at the
  // copies' issue (staged: 896 -> 903 and 893 -> 903 us).
  static constexpr int BLKC = (HD == 256 || side_codebook(KS)) ? 1024 : 0;
  static_assert(BLKC % NT == 0, "block ids per thread");
  static constexpr int OFF_BLKC = OFF_BAR + 32;
  static constexpr int SMEM_MAIN = OFF_BLKC + BLKC * 4;
  static constexpr int OUTB = ROWS * (HD + 4) * 4;    // output staging (fp32), reuses the planes
  static constexpr int SMEM = SMEM_MAIN > OUTB ? SMEM_MAIN : OUTB;
  static constexpr int S_COL = 0, O_COL = TOK;         // tensor-memory columns of S and O
  static constexpr int TCOLS = TOK + HD <= 128 ? 128 : TOK + HD <= 256 ? 256 : 512;
};

template <int KS, int VS, int HD>
__global__ void __launch_bounds__(512, 1)
prefill_tc5_kernel(const PrefillArgs a, const Codebooks cb) {
  using C = T5Cfg<KS, VS, HD>;
  using KP = PfSide<KS>;
  using VP = PfSide<VS>;
  constexpr int NT = C::NT, TOK = C::TOK;
  constexpr int E = HD / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* qh_s = reinterpret_cast<uint16_t*>(smem + C::OFF_Q);
  uint16_t* ql_s = reinterpret_cast<uint16_t*>(smem + C::OFF_Q + C::QB);
  uint16_t* k_s = reinterpret_cast<uint16_t*>(smem + C::OFF_K);   // plane p at + p * KB bytes
  uint16_t* v_s = reinterpret_cast<uint16_t*>(smem + C::OFF_V);   // plane p at + p * VB bytes
  uint16_t* ph_s = reinterpret_cast<uint16_t*>(smem + C::OFF_P);
  uint16_t* pl_s = reinterpret_cast<uint16_t*>(smem + C::OFF_P + C::PB);
  uint8_t* raw = smem + C::OFF_RAW;
  uint8_t* vrow_s = smem + C::OFF_VROW;
  float* lv = reinterpret_cast<float*>(smem + C::OFF_LV);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 16);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int q0 = a.cu_q[seq];
  const int cq = a.cu_q[seq + 1] - q0;
  const int rp = a.rp, qt = C::ROWS / rp;
  const int t0 = tile * qt;
  if (t0 >= cq) return;
  const int nq_tile = min(qt, cq - t0);
  int len = a.seq_lens[seq];
  const int64_t cap = (int64_t)a.max_blocks * a.bs;
  if (len > cap) {
    if (tid == 0 && tile == 0 && kvh == 0 && a.err) atomicOr(a.err, 2);
    len = (int)cap;
  }
  const int pbase = len - cq + t0;
  const int p_last = pbase + nq_tile - 1;
  const int lbs = 31 - __clz(a.bs);
  const int64_t tab = (int64_t)seq * a.max_blocks;
  // steps of the tile's attended positions, and the block ids of its first
  // BLKC pages, requested now (they are staged in shared memory after the
  // queries, before the first copies; -1 where the table holds no valid id)
  const int p_first = max(pbase, 0);
  const int lo_first = a.window > 0 ? max(0, p_first + 1 - a.window) : 0;
  const int st_begin = lo_first / TOK;
  const int st_end = p_last >= 0 ? p_last / TOK + 1 : st_begin;
  const int pg0 = (st_begin * TOK) >> lbs;
  const int npg = st_end > st_begin ? min(((st_end * TOK - 1) >> lbs) + 1 - pg0, C::BLKC) : 0;
  constexpr int BPT = C::BLKC / NT;
  int64_t bq[BPT > 0 ? BPT : 1];
#pragma unroll
  for (int k = 0; k < BPT; ++k) {
    const int i = tid + k * NT, pg = pg0 + i;
    bq[k] = (i < npg && pg < a.max_blocks) ? a.block_tables[tab + pg] : -1;
  }

  // ---- tensor memory and mbarriers
  const uint32_t bar_s = t5::smem_addr(bars), bar_o = t5::smem_addr(bars + 1);
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(bar_s));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(bar_o));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     t5::smem_addr(tslot)),
                 "r"(C::TCOLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }

  // ---- queries of the tile (rotated when K is), hi/lo planes in K's type
  for (int r = warp; r < C::ROWS; r += NT / 32) {
    const int qi = r / rp, hj = r - qi * rp;
    float x[E];
    if (qi < nq_tile && hj < a.rep) {
      const int64_t off = (int64_t)(q0 + t0 + qi) * a.q_stride + (int64_t)(kvh * a.rep + hj) * HD + lane * E;
#pragma unroll
      for (int i = 0; i < E; ++i)
        x[i] = a.q_bf16 ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(a.q)[off + i])
                        : reinterpret_cast<const float*>(a.q)[off + i];
      if constexpr (side_rotated(KS)) fwht_warp<E>(x, lane, a.inv_sqrt_hd);
#pragma unroll
      for (int i = 0; i < E; ++i) x[i] *= a.score_scale;   // scores come out scaled
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) x[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      uint32_t h, l;
      tc::split2<KP::BF>(x[i], x[i + 1], h, l);
      const int o_ = t5::cm<HD>(r, lane * E + i);
      *reinterpret_cast<uint32_t*>(qh_s + o_) = h;
      *reinterpret_cast<uint32_t*>(ql_s + o_) = l;
    }
  }
  pf_fill_levels<KS>(lv, lv + 16, cb, tid, NT);
  pf_fill_levels<VS>(lv + 32, lv + 48, cb, tid, NT);
  const uint2* pk = reinterpret_cast<const uint2*>(smem + C::OFF_PK);
  const uint2* pv = reinterpret_cast<const uint2*>(smem + C::OFF_PV);
  t5_fill_pairs<KS>(reinterpret_cast<uint2*>(smem + C::OFF_PK), cb, tid, NT);
  if constexpr (!C::SHARE_PAIRS) t5_fill_pairs<VS>(reinterpret_cast<uint2*>(smem + C::OFF_PV), cb, tid, NT);

  // ---- raw rows of step st (positions TOK st .. TOK st + TOK - 1) into buffer b
  int* blkc = reinterpret_cast<int*>(smem + C::OFF_BLKC);
#pragma unroll
  for (int k = 0; k < BPT; ++k) {
    const int i = tid + k * NT;
    if (i < npg) blkc[i] = (bq[k] < 0 || bq[k] > 0x7fffffff) ? -1 : (int)bq[k];
  }
  // Block id of this thread's row of step st (-1: no row there).  With the
  // short steps of head_dim 256 it is read at the top of the step that
  // issues the copies.
  auto row_block = [&](int st) -> int64_t {
    const int pos = st * TOK + tid / (NT / TOK);
    if (st >= st_end || pos < 0 || pos >= len) return -1;
    const int i = (pos >> lbs) - pg0;
    if (C::BLKC > 0 && i < C::BLKC) return blkc[i];
    return a.block_tables[tab + (pos >> lbs)];
  };
  // Thread (row t = tid / PARTS, part = tid % PARTS) looks the row's block
  // up once and copies chunks part, part + PARTS, ... of its four rows:
  // consecutive threads write consecutive 16-byte chunks of one row.
  constexpr int PARTS = NT / TOK;
  auto copy_row = [&](uint8_t* dst, const uint8_t* src, const uint8_t* base, bool ok, int part,
                      auto rowbytes_c, auto chunk_c) {
    constexpr int RB = decltype(rowbytes_c)::value, CHB = decltype(chunk_c)::value;
    if constexpr (RB > 0) {
#pragma unroll
      for (int ch = part; ch < RB / CHB; ch += PARTS)
        cp_async<CHB>(dst + ch * CHB, (ok ? src : base) + ch * CHB, ok);
    }
  };
  auto issue = [&](int st, int b, int64_t blk) {
    uint8_t* rb = raw + b * C::RAW;
    using KG = SideGeom<KS, HD>;
    using VG = SideGeom<VS, HD>;
    const int t = tid / PARTS, part = tid % PARTS;
    const bool ok = blk >= 0 && (a.num_blocks <= 0 || blk < a.num_blocks);
    const int64_t rr = (int64_t)((st * TOK + t) & (a.bs - 1)) * a.nkv + kvh;
    if (!ok) blk = 0;
    const uint8_t* kb = a.k_cache + blk * a.k_bstride;
    const uint8_t* vb = a.v_cache + blk * a.v_bstride;
    copy_row(rb + t * KG::ROW, kb + rr * KG::ROW, a.k_cache, ok, part,
             std::integral_constant<int, KG::ROW>{}, std::integral_constant<int, KG::CH>{});
    copy_row(rb + C::R_KS + t * KG::SROW, kb + a.k_dsec + rr * KG::SROW, a.k_cache, ok, part,
             std::integral_constant<int, KG::SROW>{}, std::integral_constant<int, (KG::SCH > 0 ? KG::SCH : 1)>{});
    copy_row(rb + C::R_V + t * VG::ROW, vb + rr * VG::ROW, a.v_cache, ok, part,
             std::integral_constant<int, VG::ROW>{}, std::integral_constant<int, VG::CH>{});
    copy_row(rb + C::R_VS + t * VG::SROW, vb + a.v_dsec + rr * VG::SROW, a.v_cache, ok, part,
             std::integral_constant<int, VG::SROW>{}, std::integral_constant<int, (VG::SCH > 0 ? VG::SCH : 1)>{});
    if (part == 0) vrow_s[b * TOK + t] = ok ? 1 : 0;
  };

  t5::fence_before();
  __syncthreads();   // q planes, level tables, mbarrier init and the tensor-memory address visible
  t5::fence_after();
  const uint32_t tmem = *tslot;
  constexpr int NS = C::NSPLIT, SC = TOK / NS, OC = HD / NS;   // columns per thread of S, of O
  constexpr bool M64 = C::ROWS == 64;
  // score row and column part: lane 32 (warp & 3) + lane of tensor memory
  // holds row 32 (warp & 3) + lane (M = 128), or row 16 (warp & 3) + lane
  // for lanes 0-15 (M = 64; lanes 16-31 hold no row)
  const bool has_row = !M64 || lane < 16;
  const int row = M64 ? 16 * (warp & 3) + (lane & 15) : tid & (C::ROWS - 1);
  const int hf = warp >> 2;
  const uint32_t t_lane = (uint32_t)(32 * (warp & 3)) << 16;   // this warp's lanes (rows)
  const uint32_t s_tm = tmem + C::S_COL + hf * SC, o_tm = tmem + C::O_COL;
  float* mx_s = reinterpret_cast<float*>(smem + C::OFF_MX);    // [NS][ROWS]

  // per-row softmax state (both threads of a row keep the same m_used)
  const int qi_r = row / rp, hj_r = row - qi_r * rp;
  const bool row_ok = has_row && qi_r < nq_tile && hj_r < a.rep;
  const int p_r = pbase + qi_r;
  const int lo_r = a.window > 0 ? p_r + 1 - a.window : 0;
  float m_used = -CUDART_INF_F, l_sum = 0.f;
  bool ok_all = true;
  // positions every row of the tile attends: [all_lo, all_hi]
  const int all_hi = pbase;
  const int all_lo = a.window > 0 ? p_last + 1 - a.window : 0;

  // K of a staged step into the K plane: thread = 8 dims of a token.
  auto dequant_k = [&](int b) {
    const uint8_t* rb = raw + b * C::RAW;
    for (int q = tid; q < TOK * (HD / 8); q += NT) {
      const int t = q / (HD / 8), d0 = (q % (HD / 8)) * 8;
      uint32_t hw[4], lw[4];
      if constexpr (side_codebook(KS))
        t5_dequant_pairs<KS>(rb + t * C::KROW, rb + C::R_KS + t * C::KSROW, d0, pk, tid & (PCOPY - 1), hw, lw);
      else
        pf_dequant<KS, HD, 8>(rb + t * C::KROW, rb + C::R_KS + t * C::KSROW, d0, lv, lv + 16, hw, lw);
      const int o_ = t5::cm<HD>(t, d0);
      *reinterpret_cast<uint4*>(k_s + o_) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      if constexpr (C::KPL == 2)
        *reinterpret_cast<uint4*>(k_s + C::KB / 2 + o_) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  };
  // V of a staged step into the V^T plane: thread = VTPI tokens x 8 dims.
  constexpr int VT = C::VTPI;
  auto dequant_v = [&](int b) {
    const uint8_t* rb = raw + b * C::RAW;
    for (int q = tid; q < (TOK / VT) * (HD / 8); q += NT) {
      const int tb = (q / (HD / 8)) * VT, d0 = (q % (HD / 8)) * 8;
      uint32_t vh[VT][4], vl[VT][4];
#pragma unroll
      for (int t = 0; t < VT; ++t)
        if constexpr (side_codebook(VS))
          t5_dequant_pairs<VS>(rb + C::R_V + (tb + t) * C::VROW, rb + C::R_VS + (tb + t) * C::VSROW, d0, pv,
                               tid & (PCOPY - 1), vh[t], vl[t]);
        else
          pf_dequant<VS, HD, 8>(rb + C::R_V + (tb + t) * C::VROW, rb + C::R_VS + (tb + t) * C::VSROW, d0,
                                lv + 32, lv + 48, vh[t], vl[t]);
      if constexpr (VT == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // dims d0 + 2i, d0 + 2i + 1 over the 2 tokens
          *reinterpret_cast<uint32_t*>(v_s + t5::cm<TOK>(d0 + 2 * i, tb)) = tc::prmt(vh[0][i], vh[1][i], 0x5410u);
          *reinterpret_cast<uint32_t*>(v_s + t5::cm<TOK>(d0 + 2 * i + 1, tb)) = tc::prmt(vh[0][i], vh[1][i], 0x7632u);
          if constexpr (C::VPL == 2) {
            *reinterpret_cast<uint32_t*>(v_s + C::VB / 2 + t5::cm<TOK>(d0 + 2 * i, tb)) =
                tc::prmt(vl[0][i], vl[1][i], 0x5410u);
            *reinterpret_cast<uint32_t*>(v_s + C::VB / 2 + t5::cm<TOK>(d0 + 2 * i + 1, tb)) =
                tc::prmt(vl[0][i], vl[1][i], 0x7632u);
          }
        }
      } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {   // dims d0 + 2i, d0 + 2i + 1 over the 4 tokens
        *reinterpret_cast<uint2*>(v_s + t5::cm<TOK>(d0 + 2 * i, tb)) =
            make_uint2(tc::prmt(vh[0][i], vh[1][i], 0x5410u), tc::prmt(vh[2][i], vh[3][i], 0x5410u));
        *reinterpret_cast<uint2*>(v_s + t5::cm<TOK>(d0 + 2 * i + 1, tb)) =
            make_uint2(tc::prmt(vh[0][i], vh[1][i], 0x7632u), tc::prmt(vh[2][i], vh[3][i], 0x7632u));
        if constexpr (C::VPL == 2) {
          *reinterpret_cast<uint2*>(v_s + C::VB / 2 + t5::cm<TOK>(d0 + 2 * i, tb)) =
              make_uint2(tc::prmt(vl[0][i], vl[1][i], 0x5410u), tc::prmt(vl[2][i], vl[3][i], 0x5410u));
          *reinterpret_cast<uint2*>(v_s + C::VB / 2 + t5::cm<TOK>(d0 + 2 * i + 1, tb)) =
              make_uint2(tc::prmt(vl[0][i], vl[1][i], 0x7632u), tc::prmt(vl[2][i], vl[3][i], 0x7632u));
        }
      }
      }
    }
  };

  // prologue: raw rows of the first two steps in flight, K of the first step
  if (st_begin < st_end) issue(st_begin, 0, row_block(st_begin));
  cp_async_commit();
  if (st_begin + 1 < st_end) issue(st_begin + 1, 1, row_block(st_begin + 1));
  cp_async_commit();
  cp_async_wait<1>();
  __syncthreads();
  if (st_begin < st_end) dequant_k(0);
  t5::fence_smem_async();

  for (int st = st_begin; st < st_end; ++st) {
    const int b = (st - st_begin) & 1;
    const uint32_t par = (uint32_t)((st - st_begin) & 1);
    __syncthreads();   // K of step st in its plane; raw rows of step st visible
    int64_t blk2 = -1;
    if constexpr (HD == 256) blk2 = row_block(st + 2);   // used by the copies issued at the end
    // ---- S = Q . K^T (q hi x K hi, q lo x K hi, q hi x K lo)
    if (tid == 0) {
      t5::fence_after();
      constexpr uint32_t ID = t5::idesc(KP::BF, C::ROWS, TOK);
      constexpr uint32_t SBO = t5::sbo<HD>(), KSTEP = 2 * t5::kLbo;
      const uint32_t qa = t5::smem_addr(qh_s), qb = t5::smem_addr(ql_s), ka = t5::smem_addr(k_s);
#pragma unroll
      for (int j = 0; j < HD / 16; ++j) {
        t5::mma(tmem + C::S_COL, t5::sdesc(qa + KSTEP * j, t5::kLbo, SBO),
                t5::sdesc(ka + KSTEP * j, t5::kLbo, SBO), ID, j > 0);
        t5::mma(tmem + C::S_COL, t5::sdesc(qb + KSTEP * j, t5::kLbo, SBO),
                t5::sdesc(ka + KSTEP * j, t5::kLbo, SBO), ID, 1);
        if constexpr (C::KPL == 2)
          t5::mma(tmem + C::S_COL, t5::sdesc(qa + KSTEP * j, t5::kLbo, SBO),
                  t5::sdesc(ka + C::KB + KSTEP * j, t5::kLbo, SBO), ID, 1);
      }
      t5::commit(bar_s);
    }
    // ---- meanwhile V of this step (its plane is free once O of the previous step is done)
    if (st > st_begin && !t5::wait(bar_o, par ^ 1u)) ok_all = false;
    dequant_v(b);
    t5::fence_smem_async();
    if (!t5::wait(bar_s, par)) ok_all = false;
    t5::fence_after();

    // ---- this part of the score row, masked only where the step cuts a range
    static_assert(SC == 16 || SC == 8, "one tensor-memory load per thread");
    float sv[SC];
    {
      uint32_t v0[SC];
      if constexpr (SC == 16) t5::ld16(s_tm + t_lane, v0);
      else t5::ld8(s_tm + t_lane, v0);
      t5::wait_ld();
#pragma unroll
      for (int j = 0; j < SC; ++j) sv[j] = __uint_as_float(v0[j]);
    }
    const int tbase = st * TOK + hf * SC;
    const uint32_t* vr4 = reinterpret_cast<const uint32_t*>(vrow_s + b * TOK + hf * SC);
    uint32_t vand = 0x01010101u;
#pragma unroll
    for (int w4 = 0; w4 < SC / 4; ++w4) vand &= vr4[w4];
    const bool full = row_ok && st * TOK >= all_lo && st * TOK + TOK - 1 <= all_hi &&
                      vand == 0x01010101u;
    float mx = -CUDART_INF_F;
    if (full) {
#pragma unroll
      for (int j = 0; j < SC; ++j) mx = fmaxf(mx, sv[j]);
    } else {
      const uint8_t* vr = vrow_s + b * TOK + hf * SC;
#pragma unroll
      for (int j = 0; j < SC; ++j) {
        const int t = tbase + j;
        const bool ok = row_ok && t <= p_r && t >= lo_r && vr[j];
        sv[j] = ok ? sv[j] : -CUDART_INF_F;
        mx = fmaxf(mx, sv[j]);
      }
    }
    if (has_row) mx_s[hf * C::ROWS + row] = mx;
    if (!__syncthreads_and(ok_all)) break;   // maxima and the V plane visible
#pragma unroll
    for (int i = 0; i < NS; ++i) mx = fmaxf(mx, mx_s[i * C::ROWS + row]);
    float alpha = 1.f;
    bool resc = false;
    if (mx != -CUDART_INF_F) {
      if (m_used == -CUDART_INF_F) {
        m_used = mx;
      } else if (mx > m_used + 8.f) {
        alpha = t5::ex2(m_used - mx);
        resc = true;
        l_sum *= alpha;
        m_used = mx;
      }
    }
    const bool live = m_used != -CUDART_INF_F;   // else every score so far is masked: P = 0
#pragma unroll
    for (int c8 = 0; c8 < SC; c8 += 8) {
      uint32_t h[4], l[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float x0 = live ? t5::ex2(sv[c8 + 2 * i] - m_used) : 0.f;
        const float x1 = live ? t5::ex2(sv[c8 + 2 * i + 1] - m_used) : 0.f;
        l_sum += x0 + x1;
        tc::split2<VP::BF>(x0, x1, h[i], l[i]);
      }
      const int o_ = t5::cm<TOK>(row, hf * SC + c8);
      if (has_row) {
        *reinterpret_cast<uint4*>(ph_s + o_) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(pl_s + o_) = make_uint4(l[0], l[1], l[2], l[3]);
      }
    }
    // rescale this part of the O rows whose maximum grew (warp-collective accesses)
    if (st > st_begin && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
      for (int c0 = hf * OC; c0 < (hf + 1) * OC; c0 += 16) {
        uint32_t v[16];
        t5::ld16(o_tm + t_lane + c0, v);
        t5::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
        t5::st16(o_tm + t_lane + c0, v);
      }
      t5::wait_st();
    }
    cp_async_wait<0>();   // the next step's raw rows (issued at the end of the previous step)
    t5::fence_smem_async();
    t5::fence_before();
    __syncthreads();   // P plane and the next step's raw rows visible

    // ---- O += P . V (P hi x V hi, P lo x V hi, P hi x V lo)
    if (tid == 0) {
      t5::fence_after();
      constexpr uint32_t ID = t5::idesc(VP::BF, C::ROWS, HD);
      constexpr uint32_t SBO = t5::sbo<TOK>(), KSTEP = 2 * t5::kLbo;
      const uint32_t pa = t5::smem_addr(ph_s), pb = t5::smem_addr(pl_s), va = t5::smem_addr(v_s);
#pragma unroll
      for (int j = 0; j < TOK / 16; ++j) {
        t5::mma(o_tm, t5::sdesc(pa + KSTEP * j, t5::kLbo, SBO), t5::sdesc(va + KSTEP * j, t5::kLbo, SBO), ID,
                (st > st_begin || j > 0) ? 1u : 0u);
        t5::mma(o_tm, t5::sdesc(pb + KSTEP * j, t5::kLbo, SBO), t5::sdesc(va + KSTEP * j, t5::kLbo, SBO), ID, 1);
        if constexpr (C::VPL == 2)
          t5::mma(o_tm, t5::sdesc(pa + KSTEP * j, t5::kLbo, SBO),
                  t5::sdesc(va + C::VB + KSTEP * j, t5::kLbo, SBO), ID, 1);
      }
      t5::commit(bar_o);
    }
    // ---- meanwhile K of the next step (the K plane is free: S of this step is done)
    if (st + 1 < st_end) dequant_k(b ^ 1);
    t5::fence_smem_async();
    // raw rows two steps ahead into this step's buffer (its K and V are in
    // their planes), issued after this step's last proxy fence: a proxy fence
    // also waits for the copies in flight (measured on GB300)
    if (st + 2 < st_end) issue(st + 2, b, HD == 256 ? blk2 : row_block(st + 2));
    cp_async_commit();
  }
  cp_async_wait<0>();
  if (st_end > st_begin && ok_all) {
    if (!t5::wait(bar_o, (uint32_t)((st_end - 1 - st_begin) & 1))) ok_all = false;
  }
  if (!ok_all && tid == 0 && a.err) atomicOr(a.err, 4);
  t5::fence_after();
  if (has_row) mx_s[hf * C::ROWS + row] = l_sum;
  __syncthreads();   // every plane read is done: the output staging reuses them
  l_sum = 0.f;
#pragma unroll
  for (int i = 0; i < NS; ++i) l_sum += mx_s[i * C::ROWS + row];

  // ---- normalise row `row` (this thread's part) from tensor memory, stage,
  // rotate back, store
  float* os = reinterpret_cast<float*>(smem);   // [ROWS][HD + 4]
  {
    const float inv = l_sum > 0.f ? a.v_mult / l_sum : 0.f;
    const bool have_o = st_end > st_begin && ok_all;
#pragma unroll 1
    for (int c0 = hf * OC; c0 < (hf + 1) * OC; c0 += 16) {
      uint32_t v[16];
      if (have_o) {
        t5::ld16(o_tm + t_lane + c0, v);
        t5::wait_ld();
      }
      if (has_row) {
#pragma unroll
        for (int j = 0; j < 16; ++j) os[row * (HD + 4) + c0 + j] = have_o ? __uint_as_float(v[j]) * inv : 0.f;
      }
    }
  }
  t5::fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(C::TCOLS));
  for (int r = warp; r < C::ROWS; r += NT / 32) {
    const int qi = r / rp, hj = r - qi * rp;
    if (qi >= nq_tile || hj >= a.rep) continue;   // warp-uniform
    float x[E];
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] = os[r * (HD + 4) + lane * E + i];
    if constexpr (side_rotated(VS)) fwht_warp<E>(x, lane, a.inv_sqrt_hd);
    const int64_t o_ = ((int64_t)(q0 + t0 + qi) * a.nq + kvh * a.rep + hj) * HD + lane * E;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if (a.out_bf16) reinterpret_cast<uint16_t*>(a.out)[o_ + i] = bf16_bits_from_float(x[i]);
      else reinterpret_cast<float*>(a.out)[o_ + i] = x[i];
    }
  }
}

template <int KS, int VS, int HD>
cudaError_t launch_prefill_tc5(const PrefillArgs& a, const Codebooks& cb, int max_chunk, cudaStream_t st) {
  using C = T5Cfg<KS, VS, HD>;
  static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
  auto kern = prefill_tc5_kernel<KS, VS, HD>;
  if (C::SMEM > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
  }
  const int qt = C::ROWS / a.rp;
  dim3 grid((max_chunk + qt - 1) / qt, a.nkv, a.num_seqs);
  kern<<<grid, C::NT, C::SMEM, st>>>(a, cb);
  return cudaGetLastError();
}

template <int KS, int VS>
cudaError_t launch_prefill_pair(int hd, const PrefillArgs& a, const Codebooks& cb, int max_chunk,
                                cudaStream_t st) {
  switch (hd) {
    case 64: return launch_prefill_tc5<KS, VS, 64>(a, cb, max_chunk, st);
    case 128: return launch_prefill_tc5<KS, VS, 128>(a, cb, max_chunk, st);
    case 256: return launch_prefill_tc5<KS, VS, 256>(a, cb, max_chunk, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
