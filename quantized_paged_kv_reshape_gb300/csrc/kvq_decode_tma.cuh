// Paged decode attention fed by TMA tensor copies, one kernel launch.
//
// The same computation as decode_tc_kernel ("combs_models/kv.rs" attend with
// repeat_kv for one query per sequence, the "spark_runtime/kv_cache.rs"
// is_wht_rotated bookends), organised to spend as few instructions and
// shared-memory wavefronts per cached element as it can:
//
// * Copies.  Each warp streams its own 16-position slabs through a ring of
//   NST stages.  One lane issues, per slab, one cp.async.bulk.tensor copy per
//   section (K rows, K scale rows, V rows, V scale rows) of its kv head,
//   described by tensor maps over the pools ([num_blocks, block_size,
//   num_kv_heads, row bytes]); an mbarrier per stage counts the bytes in.
//   Rows of 32, 64 or 128 bytes land swizzled (16-byte chunk c of row r at
//   c ^ f(r)) so that the fragment loads below touch distinct banks.
// * Codebook K (Turbo4, NVFP4): k-step j is scale group j; thread (g, c)
//   reads code bytes 8j+2c, 8j+2c+1 of tokens g, g+8 (one 32-bit load per
//   token and k-step) and looks each code pair up in a pair table of level
//   parts (fp16 hi, lo with 7 significant bits each).  The table entry of
//   byte b sits at b * 256 + 8 * (lane % 16), so one byte permute of the
//   code word forms its address.  The group scales multiply the fp32
//   products of each k-step.
// * Codebook V (Turbo4, NVFP4, Turbo2, Turbo3): thread g owns HD/8
//   consecutive dims of every token (one scale group for head_dim 128), so
//   m-tile i holds dims g*HD/8 + 2i (row g) and + 1 (row g+8).  For 4-bit
//   and 2-bit codes the table is indexed by the codes of the two tokens a
//   register holds (low nibble: first token), built for four m-tiles at
//   once by two funnel-free logic ops per code word, so the entry is
//   already in operand order; its parts times the tokens' group scales
//   (exact in fp16) are the operands.  Turbo3 looks up (dim, dim+1) pairs of
//   one token and regroups them with byte permutes.
// * Raw sides (BF16 through ldmatrix, FP8 converted in registers) as in
//   decode_tc_kernel, addressed through the swizzle.
// * Online softmax in the exp2 domain with a lazy maximum: the running
//   maximum of a (warp, query head) moves only when a score exceeds it by
//   more than 8 (so weights stay below 2^8), which a warp vote detects;
//   only then are the maxima reduced and the accumulators rescaled.
//
// Partition, partial results and the last-arriver merge are those of
// decode_tc_kernel.
#pragma once

#include <cuda.h>

#include "kvq_decode_mma.cuh"

namespace kvq {

// Tensor maps of the four sections (unused ones zero).
struct TmaMaps {
  CUtensorMap kd, ks, vd, vs;
};

namespace tm {

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void bar_init(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(bar));
}
__device__ __forceinline__ void bar_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Bounded wait for phase `parity` of a stage barrier; false if it gave up.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  for (int it = 0; it < (1 << 22); ++it) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
__device__ __forceinline__ void fence_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tma4(uint32_t dst, const CUtensorMap* m, int x, int y, int z, int w,
                                     uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4, %5}], [%6];\n" ::"r"(dst),
      "l"(m), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma3(uint32_t dst, const CUtensorMap* m, int x, int y, int z,
                                     uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(m), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(a));
  return v;
}
// loads at a + OFF (OFF folded into the instruction)
template <int OFF>
__device__ __forceinline__ uint32_t lds32o(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1+%2];\n" : "=r"(v) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint2 lds64o(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2+%3];\n" : "=r"(v.x), "=r"(v.y) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint4 lds128o(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4+%5];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a), "n"(OFF));
  return v;
}
// 2^x for the softmax weights (x <= 8 or -inf; results below 2^-126 flush
// to zero, far below the fp32 sums they join)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// D = A . B with a zero accumulator (m16n8k16, fp16 operands, fp32 out)
__device__ __forceinline__ void mma_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                      uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];\n" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
template <int OFF>
__device__ __forceinline__ void ldsm_x4o(uint32_t (&r)[4], uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4+%5];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a), "n"(OFF));
}
template <int OFF>
__device__ __forceinline__ void ldsm_x4_to(uint32_t (&r)[4], uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4+%5];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a), "n"(OFF));
}
__device__ __forceinline__ void sts_zero16(uint32_t a) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};\n" ::"r"(a), "r"(0u) : "memory");
}
__device__ __forceinline__ void sts_zero8(uint32_t a) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %1};\n" ::"r"(a), "r"(0u) : "memory");
}
__device__ __forceinline__ void sts_zero4(uint32_t a) {
  asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(a), "r"(0u) : "memory");
}
// (a & m) | (b & ~m)
__device__ __forceinline__ uint32_t bitsel(uint32_t a, uint32_t b, uint32_t m) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xE4;\n" : "=r"(r) : "r"(a), "r"(b), "r"(m));
  return r;
}

}  // namespace tm

// Staged geometry of one side: data rows of ROWB bytes copied as NBOX boxes
// of BOXW bytes (swizzled when BOXW is 32, 64 or 128), scale rows as boxes
// of SBOXW bytes (the 16-byte aligned span holding this head's scales when
// a scale row is shorter than 16 bytes).
template <int S, int HD>
struct TmSide {
  static constexpr int ROWB = HD * side_bits(S) / 8;
  static constexpr int SROW = (HD / kGroup) * side_scale_bytes(S);
  static constexpr int BOXW = ROWB > 128 ? 128 : ROWB;
  static constexpr int NBOX = ROWB / BOXW;
  static constexpr int SWZ = BOXW == 128 ? 3 : BOXW == 64 ? 2 : BOXW == 32 ? 1 : 0;
  static constexpr int TILE = 16 * ROWB;
  static constexpr int SBOXW = SROW == 0 ? 0 : (SROW < 16 ? 16 : SROW);
  static constexpr int STILE = 16 * SBOXW;
  static constexpr bool CB = side_codebook(S);
  static constexpr int BITS = side_bits(S);
  // smem byte offset of byte x of row r inside the side's tile
  __device__ __forceinline__ static uint32_t at(int r, int x) {
    const int b = x / BOXW, xi = x % BOXW;
    int chunk = xi >> 4;
    if constexpr (SWZ > 0) chunk ^= ((r * BOXW) >> 7) & ((1 << SWZ) - 1);
    return (uint32_t)(b * 16 * BOXW + r * BOXW + (chunk << 4) + (xi & 15));
  }
};

// Sides and head dims the TMA decode handles (others use decode_tc_kernel).
__host__ __device__ constexpr bool tma_k_side(int s) {
  return s == S_BF16 || s == S_FP8 || s == S_T4 || s == S_NVFP4;
}
__host__ __device__ constexpr bool tma_v_side(int s) {
  return s == S_BF16 || s == S_FP8 || s == S_T4 || s == S_NVFP4 || s == S_T3 || s == S_T2;
}

// Placement of the stage tiles in dynamic shared memory.  The code tables
// of the codebook sides sit at a shared address that is a multiple of 64 KB
// (dynamic shared memory starts at kSmemBase, after the 1 KB the driver
// reserves per block), so that one byte permute of a code word with a
// per-lane register forms a table entry's whole address: 0x20000 for tables
// of 256 entries (64 KB), 0x30000 for the 64-entry Turbo3 pair table when it
// is the only one, which leaves one larger region below it; the tiles fill
// the space before the tables first, largest section first, then the space
// after them.
constexpr int kSmemBase = 0x400;
constexpr int kSmemLimit = 227 * 1024;

struct TmLayout {
  int kd, vd, ks, vs, merge, end;
  bool ok;
};

template <int KS, int VS, int HD, bool PK>
struct TmCfg {
  using K = TmSide<KS, HD>;
  using V = TmSide<VS, HD>;
  static constexpr int NK = HD / 16;
  static constexpr bool LUT = K::CB || V::CB;
  // pair / quad tables: entry of index b at b * 256; K's in bytes [0, 128)
  // of an entry, V's in [128, 256) unless it is K's table
  static constexpr bool VLUT2 = V::CB && !(K::CB && KS == VS);
  static constexpr int MAXP = 2048;                       // pages staged per stretch
  static constexpr int OFF_Q = 0;                         // q rows [8][HD] fp32
  static constexpr int OFF_BLK = OFF_Q + 8 * HD * 4;      // block ids of a stretch
  static constexpr int OFF_SCAN = OFF_BLK + MAXP * 4;     // partition scan / merge scratch
  static constexpr int OFF_STATE = OFF_SCAN + 48 * 8;     // CTA loop state
  static constexpr int OFF_BAR = OFF_STATE + 8 * 8;       // stage barriers (<= 16 x 4)
  static constexpr int HEAD = align_up(OFF_BAR + 64 * 8, 1024);
  // table entries: 64 Turbo3 pair entries when V's is the only table, else 256
  static constexpr int LUT_ENTRIES = (!K::CB && VS == S_T3) ? 64 : 256;
  static constexpr int LUT_ADDR = LUT_ENTRIES == 64 ? 0x30000 : 0x20000;
  static constexpr int LUT_OFF = LUT ? LUT_ADDR - kSmemBase : 0;   // from the dynamic base
  static constexpr int LUT_END = LUT ? LUT_OFF + LUT_ENTRIES * 256 : 0;
  static constexpr int MERGE_BYTES = 16 * 8 * HD * 4 + 16 * 8 * 2 * 4;   // (for 16 warps)
  // Virtual slabs a unit costs in the partition (measured on GB300 with
  // U = 0 / 24 / 48 / 96: ragged bf16k_turbo3v 264.5 / 254.4 / 244.2 /
  // 250.4 us, fp8k_turbo2v 219.4 / 210.9 / 203.1 / 199.2, llama8b bf16 92.5 /
  // 91.7 / 91.1 / 94.2, turbo4 82.2 / 81.2 / 79.9 / 81.9; fp8k_turbo2v again
  // with U = 48 / 96 / 144: 201.0 / 197.2 / 203.6 us, so it takes 96).
  static constexpr int SWITCH = (KS == S_FP8 && VS == S_T2) ? 2 * kUnitSlabs : kUnitSlabs;

  // CTAs per SM (measured on GB300, llama8b layer): FP8 runs two CTAs of 8
  // warps, whose unit boundaries (merge, next unit's first copies) then
  // overlap each other's streaming (59.9 against 65.5 us with one CTA of 16);
  // BF16 one CTA of 8 warps (94.3 against 98.3 us with two of 4); the sides
  // with code tables one CTA, whose fixed table placement needs the whole of
  // it.
  static constexpr int CPS = (!LUT && KS == S_FP8) ? 2 : 1;
  static constexpr int LIMIT = CPS == 1 ? kSmemLimit : (228 * 1024) / CPS - 1024;
  static constexpr TmLayout layout(int nw, int nst) {
    const int sz[4] = {nw * nst * K::TILE, nw * nst * V::TILE, nw * nst * K::STILE,
                       nw * nst * V::STILE};
    const int al[4] = {1024, 1024, 128, 128};
    int off[4] = {0, 0, 0, 0};
    bool done[4] = {false, false, false, false};
    int a = HEAD, b = LUT ? LUT_END : HEAD;
    for (int n = 0; n < 4; ++n) {
      int best = -1;
      for (int i = 0; i < 4; ++i)
        if (!done[i] && (best < 0 || sz[i] > sz[best])) best = i;
      done[best] = true;
      const int x = align_up(a, al[best]);
      if (LUT && x + sz[best] <= LUT_OFF) {
        off[best] = x;
        a = x + sz[best];
      } else {
        const int y = align_up(b, al[best]);
        off[best] = y;
        b = y + sz[best];
      }
    }
    const int mg = (!LUT || HEAD + MERGE_BYTES <= LUT_OFF) ? HEAD : LUT_END;
    int end = a > b ? a : b;
    if (LUT && end < LUT_END) end = LUT_END;
    if (mg + MERGE_BYTES > end) end = mg + MERGE_BYTES;
    return TmLayout{off[0], off[1], off[2], off[3], mg, end, end <= LIMIT};
  }
  // Warps per CTA: as many as rings of three stages allow (16, 12 or 8),
  // with these exceptions, measured on GB300:
  // - a codebook K side with unpacked queries (q hi and lo in separate
  //   operands: the most live registers) runs 12 warps of up to 168
  //   registers (long-context layer: 315 against 330 us with 16 warps of 128
  //   registers, which spill; with packed queries 16 warps are faster: 82
  //   against 84 us);
  // - with a code table, 12 warps of two stages beat 8 of three (BF16 K
  //   with Turbo4 V 74.0 against 80.2 us, with Turbo2 V 70.0 against 77.8;
  //   without a table, BF16 K and V: 91.2 against 90.6 us).
  static constexpr int pick_nw() {
    if (K::CB && !PK && CPS == 1 && layout(12, 3).ok) return 12;
    if (CPS != 1) return layout(8, 3).ok ? 8 : 4;
    if (layout(16, 3).ok) return 16;
    if (layout(12, 3).ok || (LUT && layout(12, 2).ok)) return 12;
    return 8;
  }
  static constexpr int NW = pick_nw();
  static constexpr int pick_nst() {
    return layout(NW, 4).ok ? 4 : layout(NW, 3).ok ? 3 : 2;
  }
  static constexpr int NST = pick_nst();
  static constexpr TmLayout L = layout(NW, NST);
  static constexpr int R_KD = L.kd, R_VD = L.vd, R_KS = L.ks, R_VS = L.vs, OFF_MERGE = L.merge;
  static constexpr int SMEM = L.end;
  static_assert(L.ok, "shared memory budget");
  // a swizzle pattern repeats every 8 rows of the swizzle span (128 << SWZ bytes)
  static constexpr int KREP = K::SWZ ? (128 << K::SWZ) : 128;
  static constexpr int VREP = V::SWZ ? (128 << V::SWZ) : 128;
  static_assert((16 * K::BOXW) % KREP == 0 && (16 * V::BOXW) % VREP == 0 &&
                    (8 * K::BOXW) % KREP == 0 && (8 * V::BOXW) % VREP == 0,
                "staged tiles (and block-size-8 halves) start at a swizzle repeat");
  static_assert(K::STILE % 128 == 0 && V::STILE % 128 == 0, "scale tiles 128-byte aligned");
  // bytes the copies write per staged position
  static constexpr int ROWBYTES = K::ROWB + K::SBOXW + V::ROWB + V::SBOXW;
};

// Output dim of accumulator row `row` (0..15) of m-tile i.
template <int S, int HD>
__device__ __forceinline__ int tm_v_row_dim(int i, int row) {
  if constexpr (side_codebook(S)) {
    constexpr int DPT = HD / 8;   // dims owned by thread group g
    return (row & 7) * DPT + 2 * i + (row >> 3);
  } else {
    return v_row_dim<S, HD>(i, row);
  }
}

template <int KS, int VS, int HD, bool PK>
__global__ void __launch_bounds__(32 * TmCfg<KS, VS, HD, PK>::NW, TmCfg<KS, VS, HD, PK>::CPS)
decode_tma_kernel(const DecodeArgs a, const __grid_constant__ TmaMaps maps, const Codebooks cb) {
  using C = TmCfg<KS, VS, HD, PK>;
  using KT = typename C::K;
  using VT = typename C::V;
  constexpr int NW = C::NW;
  constexpr int NT = 32 * NW;
  constexpr int NST = C::NST;
  constexpr int NK = C::NK;
  constexpr int E = HD / 32;
  constexpr int SLAB = 16;
  extern __shared__ __align__(1024) uint8_t tma_smem[];   // (its own name: other kernels declare 128-byte alignment)
  uint8_t* const smem = tma_smem;
  const uint32_t sbase = tm::saddr(smem);
  if (C::LUT && sbase != (uint32_t)kSmemBase) {   // the tables' placement assumes it
    if (threadIdx.x == 0 && a.err) atomicOr(a.err, 4);
    return;
  }
  float* q_s = reinterpret_cast<float*>(smem + C::OFF_Q);
  int* blk_s = reinterpret_cast<int*>(smem + C::OFF_BLK);
  int64_t* scan_s = reinterpret_cast<int64_t*>(smem + C::OFF_SCAN);
  const uint32_t lut_k = C::LUT_ADDR;
  const uint32_t lut_v = lut_k + (C::VLUT2 ? 128 : 0);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int bs = a.bs;
  const int lbs = 31 - __clz(bs);
  const int nkv = a.nkv;
  const int64_t cap = (int64_t)a.max_blocks * bs;

  auto seq_slabs = [&](int s, int& first, int& n, int& lo_, int& len) {
    len = a.seq_lens[s];
    if (len > cap) len = (int)cap;
    if (len <= 0) {
      first = n = lo_ = len = 0;
      return;
    }
    lo_ = a.window > 0 ? max(0, len - a.window) : 0;
    first = lo_ >> 4;
    n = ((len + 15) >> 4) - first;
  };

  // ---- Partition (as decode_tc_kernel): R = gridDim.x / nkv CTAs per kv
  // head, each on an equal share of the sequences' 16-position slabs.
  const int N = a.num_seqs;
  const int R = gridDim.x / nkv;
  const int kvh = blockIdx.x / R, jr = blockIdx.x - kvh * R;
  const int chunk = (N + NT - 1) / NT;
  const int s_beg = min(N, tid * chunk), s_end = min(N, s_beg + chunk);
  int64_t mine = 0;
  int longest = 0;
  for (int s = s_beg; s < s_end; ++s) {
    int f, n, l_, e_;
    seq_slabs(s, f, n, l_, e_);
    mine += n;
    longest = max(longest, n);
    if (blockIdx.x == 0 && a.seq_lens[s] > cap && a.err) atomicOr(a.err, 2);
  }
  int64_t incl = mine;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
    longest = max(longest, __shfl_xor_sync(0xffffffffu, longest, d));
  }
  // scan_s: [0, 16) per-warp slab sums, [16, 32) per-warp longest rows,
  // [32] / [33] the first unit's sequence / slab, [34] / [35] the range's
  // first and end slab, [36, 44) merge maxima and sums (float), [44] the
  // last-arriver flag (int)
  if (lane == 31) scan_s[warp] = incl;
  if (lane == 0) scan_s[16 + warp] = longest;
  __syncthreads();
  int64_t before = 0, total = 0, max_n = 0;
  for (int w2 = 0; w2 < NW; ++w2) {
    const int64_t v = scan_s[w2];
    if (w2 < warp) before += v;
    total += v;
    max_n = max(max_n, scan_s[16 + w2]);
  }
  const int64_t excl = before + incl - mine;
  // Sequence s spans [P_s + U s, P_s + U s + U + n_s) of a virtual slab line
  // (P_s = attended slabs before it): its first U positions stand for the
  // cost of a unit (the merge, then the first copies' round trip), and the
  // CTAs split the virtual line evenly, so that a CTA that works on more
  // sequences takes fewer slabs.  Real slab (s, o) sits at P_s + U (s + 1) + o.
  constexpr int64_t U = C::SWITCH;
  const int64_t totalv = total + U * N;
  int64_t cpc = (totalv + R - 1) / R;
  if (a.kmax > 1) cpc = max(cpc, (max_n + a.kmax - 2) / (a.kmax - 1));
  if (cpc < 1) cpc = 1;
  const int64_t v0 = (int64_t)jr * cpc, v1 = min(v0 + cpc, totalv);
  {   // the real slab indices of v0 and v1 (scan_s[34], [35])
    int64_t P = excl;
    for (int s = s_beg; s < s_end; ++s) {
      int f, n, l_, e_;
      seq_slabs(s, f, n, l_, e_);
      const int64_t vp = P + U * s;
      if (v0 >= vp && v0 < vp + U + n) scan_s[34] = P + min(max(v0 - vp - U, (int64_t)0), (int64_t)n);
      if (v1 >= vp && v1 < vp + U + n) scan_s[35] = P + min(max(v1 - vp - U, (int64_t)0), (int64_t)n);
      P += n;
    }
  }
  __syncthreads();
  const int64_t x0 = v0 < totalv ? scan_s[34] : total;
  const int64_t x_end = v1 < totalv ? scan_s[35] : total;
  if (blockIdx.x == 0) {  // sequences with nothing to attend get zero rows
    for (int s = s_beg; s < s_end; ++s) {
      int f, n, l_, e_;
      seq_slabs(s, f, n, l_, e_);
      if (n > 0) continue;
      for (int i = 0; i < a.nq * HD; ++i) {
        const int64_t o_ = (int64_t)s * a.nq * HD + i;
        if (a.out_bf16) reinterpret_cast<uint16_t*>(a.out)[o_] = 0;
        else reinterpret_cast<float*>(a.out)[o_] = 0.f;
      }
    }
  }
  if (kvh < nkv && x0 < total && excl <= x0 && x0 < excl + mine) {
    int64_t P = excl;
    for (int s = s_beg; s < s_end; ++s) {
      int f, n, l_, e_;
      seq_slabs(s, f, n, l_, e_);
      if (x0 < P + n) {
        scan_s[32] = s;
        scan_s[33] = x0 - P;
        break;
      }
      P += n;
    }
  }
  // stage barriers (one arrival per phase: the issuing lane's expect_tx)
  if (tid == 0) {
    for (int i = 0; i < NW * NST; ++i) tm::bar_init(sbase + C::OFF_BAR + 8 * i);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  // Pair / quad tables of the codebook sides.  Index b: 4-bit codes: two
  // codes b & 15 (first) and b >> 4; 2-bit codes: four codes, bits 0-1 and
  // 4-5 the first word's pair, 2-3 and 6-7 the second's; Turbo3: (dim, dim+1)
  // pair b & 7, (b >> 3) & 7.  Levels split into two 7-bit parts (hi, lo),
  // exact in fp16 when multiplied by an E4M3 scale.
  auto fill_lut = [&](uint32_t lut, int side) {
    const float* lv = side == S_T4 ? cb.lv4 : side == S_T3 ? cb.lv3 : side == S_NVFP4 ? cb.e2m1 : cb.lv2;
    if (side == S_T2) {
      for (int e = tid; e < 256 * 8; e += NT) {
        const int b = e >> 3, cp = e & 7;
        float h[4], l[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int code = (b >> (2 * k)) & 3;   // k: bits 2k, 2k+1
          h[k] = tc::round_sig7(lv[code]);
          l[k] = tc::round_sig7(lv[code] - h[k]);
        }
        // words: (code bits 0-1, bits 4-5), (bits 2-3, bits 6-7)
        const uint32_t x0 = tc::pack2<false>(h[0], h[2]), x1 = tc::pack2<false>(h[1], h[3]);
        const uint32_t y0 = tc::pack2<false>(l[0], l[2]), y1 = tc::pack2<false>(l[1], l[3]);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(lut + b * 256 + cp * 16),
                     "r"(x0), "r"(x1), "r"(y0), "r"(y1)
                     : "memory");
      }
    } else {
      const int cbits = side == S_T3 ? 3 : 4;
      for (int e = tid; e < (1 << (2 * cbits)) * 16; e += NT) {   // entries the codes index
        const int b = e >> 4, cp = e & 15;
        const float c0 = lv[b & ((1 << cbits) - 1)];
        const float c1 = lv[(b >> cbits) & ((1 << cbits) - 1)];
        const float h0 = tc::round_sig7(c0), h1 = tc::round_sig7(c1);
        const float l0 = tc::round_sig7(c0 - h0), l1 = tc::round_sig7(c1 - h1);
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};\n" ::"r"(lut + b * 256 + cp * 8),
                     "r"(tc::pack2<false>(h0, h1)), "r"(tc::pack2<false>(l0, l1))
                     : "memory");
      }
    }
  };
  if constexpr (KT::CB) fill_lut(lut_k, KS);
  if constexpr (C::VLUT2) fill_lut(lut_v, VS);
  __syncthreads();
  if (kvh >= nkv || x0 >= total) return;
  int seq = (int)scan_s[32];
  int64_t off = scan_s[33];

  // this warp's stage tiles: section base + stage * tile bytes
  const uint32_t rkd = sbase + C::R_KD + warp * NST * KT::TILE;
  const uint32_t rvd = sbase + C::R_VD + warp * NST * VT::TILE;
  const uint32_t rks = sbase + C::R_KS + warp * NST * KT::STILE;
  const uint32_t rvs = sbase + C::R_VS + warp * NST * VT::STILE;
  const uint32_t bar0 = sbase + C::OFF_BAR + warp * NST * 8;
  int lo = 0, tok_end = 0, tok0 = 0, p0 = 0;
  uint32_t gk = 0;        // slabs this warp has consumed so far (stage/phase clock)
  bool failed = false;

  // Issue the copies of slab s of this warp's share of the stretch into
  // stage (gk + s) % NST (lane 0).  Pieces of 16 rows (block_size >= 16) or
  // two of 8 (block_size 8); a piece outside the attended range or whose
  // block id is invalid is not copied.
  bool dirty = false;     // a stage holds generic-proxy writes the copies must follow
  bool merged = false;    // a unit's merge has run in this CTA (it overlaps the rings)
  auto issue = [&](int s, uint32_t st) {
    // Every lane computes the same operands (all lanes read the same block
    // ids), so that the copies' operands are warp-uniform; lane 0 issues.
    const uint32_t bar = bar0 + st * 8;
    const int slab_pos = tok0 + (warp + NW * s) * SLAB;
    int b0 = -1, b1 = -1;
    if (bs >= 16) {   // one page holds the slab, and the slab meets [lo, tok_end)
      b0 = blk_s[(slab_pos >> lbs) - p0];
    } else {          // two pages of 8 positions; a page outside [lo, tok_end) is skipped
      if (slab_pos + 8 > lo) b0 = blk_s[(slab_pos >> lbs) - p0];
      if (slab_pos + 8 < tok_end) b1 = blk_s[((slab_pos + 8) >> lbs) - p0];
    }
    const int rows = bs < 16 ? 8 : 16;
    const uint32_t bytes = (uint32_t)(((b0 >= 0) + (b1 >= 0)) * rows * C::ROWBYTES);
    const int in_page = slab_pos & (bs - 1);
    if (lane == 0) {
      if (dirty) tm::fence_async();   // generic writes (cleared rows, merge scratch) first
      if (bytes == 0) {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
      } else {
        tm::bar_expect(bar, bytes);
      }
    }
    dirty = false;
    auto piece = [&](int p, int blk, int ip) {
      if (lane != 0 || blk < 0) return;
#pragma unroll
      for (int b = 0; b < KT::NBOX; ++b)
        tm::tma4(rkd + st * KT::TILE + b * 16 * KT::BOXW + p * 8 * KT::BOXW, &maps.kd, b * KT::BOXW,
                 kvh, ip, blk, bar);
#pragma unroll
      for (int b = 0; b < VT::NBOX; ++b)
        tm::tma4(rvd + st * VT::TILE + b * 16 * VT::BOXW + p * 8 * VT::BOXW, &maps.vd, b * VT::BOXW,
                 kvh, ip, blk, bar);
      if constexpr (KT::SROW > 0) {
        const uint32_t d = rks + st * KT::STILE + p * 8 * KT::SBOXW;
        if constexpr (KT::SROW >= 16) tm::tma4(d, &maps.ks, 0, kvh, ip, blk, bar);
        else tm::tma3(d, &maps.ks, (kvh * KT::SROW) & ~15, ip, blk, bar);
      }
      if constexpr (VT::SROW > 0) {
        const uint32_t d = rvs + st * VT::STILE + p * 8 * VT::SBOXW;
        if constexpr (VT::SROW >= 16) tm::tma4(d, &maps.vs, 0, kvh, ip, blk, bar);
        else tm::tma3(d, &maps.vs, (kvh * VT::SROW) & ~15, ip, blk, bar);
      }
    };
    piece(0, b0, in_page);
    if (bs < 16) piece(1, b1, (slab_pos + 8) & (bs - 1));
  };

  // ---- per-thread constants of the fragment loads
  // table-entry address = the code byte in bits 8-15 of one of these (a
  // byte permute): the tables' base (bits 16+), this lane's copy (bits 0-6),
  // V's table half (bit 7)
  const uint32_t laneoff8 = (uint32_t)C::LUT_ADDR | ((uint32_t)(lane & 15) << 3);
  const uint32_t laneoff16 = (uint32_t)C::LUT_ADDR | ((uint32_t)(lane & 7) << 4);
  const uint32_t vlane8 = laneoff8 | (C::VLUT2 ? 0x80u : 0u);
  const uint32_t vlane16 = laneoff16 | (C::VLUT2 ? 0x80u : 0u);
  // K scale span: this head's scale bytes inside a staged scale row
  constexpr int KSO_M = KT::SROW >= 16 ? 0 : 15;
  constexpr int VSO_M = VT::SROW >= 16 ? 0 : 15;
  const int kso = (kvh * KT::SROW) & KSO_M;
  const int vso = (kvh * VT::SROW) & VSO_M;
  // V tokens of this thread in operand order: (first, second) = k-slots
  // (2c, 2c+1) and (+8, +9).  Odd c take them swapped so that the four
  // 8-byte code loads of a warp fall in distinct bank halves; the P
  // operand's halves are swapped to match.
  const int vt0 = 2 * c + (c & 1), vt1 = 2 * c + 1 - (c & 1);
  constexpr int DPT = HD / 8;                    // V dims owned by thread group g
  constexpr int VCB_BYTES = DPT * VT::BITS / 8;  // code bytes of one token's span

  // ---- loop-invariant offsets of this thread's loads inside a stage's tiles
  // K codes: 16-byte chunk k of row g (row g+8 is 8 rows on, same swizzle)
  // plus this thread's word of the chunk
  // K codes (codebook sides): 16-byte chunk k of row g plus this thread's
  // word; FP8 K: this thread's chunk 4jj + c of row g; BF16 K: the ldmatrix
  // row address of this lane for k-steps j with j % 4 == m (k-step j + 4 is
  // the next 128-byte box)
  constexpr int KCH = KT::CB ? KT::ROWB / 16 : KS == S_FP8 ? (NK + 3) / 4 : 4;
  uint32_t kco[KCH];
#pragma unroll
  for (int k = 0; k < KCH; ++k) {
    if constexpr (KT::CB) kco[k] = KT::at(g, 16 * k) + 4 * (c >> 1);
    else if constexpr (KS == S_FP8) kco[k] = KT::at(g, (4 * k + c) * 16);
    else kco[k] = KT::at((lane >> 3 & 1) * 8 + (lane & 7), 32 * k + 16 * (lane >> 4));
  }
  const uint32_t ksoff = g * KT::SBOXW + kso;                // K scales of token g
  // V: codebook sides: the span of tokens (first, second) and (+8, +9);
  // FP8: dims g*DPT.. of tokens 2c, 2c+1, 2c+8, 2c+9; BF16: the ldmatrix
  // (.trans) row address of this lane for m-tiles i with i % 4 == m
  const int vtk[4] = {vt0, vt1, vt0 + 8, vt1 + 8};
  uint32_t vco[4], vso4[4];
  {
    const int gsb = HD == 256 ? 2 * g : (HD == 128 ? g : (g >> 1));   // first group owned
    const int ftk[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if constexpr (VT::CB) vco[t] = VT::at(vtk[t], g * VCB_BYTES);
      else if constexpr (VS == S_FP8) vco[t] = VT::at(ftk[t], g * DPT);
      else vco[t] = VT::at((lane >> 4) * 8 + (lane & 7), 32 * t + 16 * (lane >> 3 & 1));
      vso4[t] = VT::SROW > 0 ? (uint32_t)(vtk[t] * VT::SBOXW + vso + gsb) : 0u;
    }
  }

  uint32_t qh[NK][2], ql[PK ? 1 : NK][2];
  float o[NK][4];
  float m0, m1, l0, l1;
  const float scale = a.score_scale;

  // ---- S^T for the slab staged at stage address sb: this thread's rows
  // g, g+8 x columns 2c, 2c+1 (before the PK column merge).
  auto scores = [&](uint32_t stg, float (&sacc)[4]) {
    const uint32_t sb = rkd + stg * KT::TILE;
    float sacl[4] = {0.f, 0.f, 0.f, 0.f};
    sacc[0] = sacc[1] = sacc[2] = sacc[3] = 0.f;
    if constexpr (KS == S_BF16) {
#pragma unroll
      for (int j = 0; j < NK; ++j) {
        uint32_t f[4];
        if (j < 4) tm::ldsm_x4o<0>(f, sb + kco[j & 3]);
        else tm::ldsm_x4o<16 * KT::BOXW>(f, sb + kco[j & 3]);
        if constexpr (PK) {
          tc::mma<true>((j & 1) ? sacl : sacc, f[0], f[1], f[2], f[3], qh[j][0], qh[j][1]);
        } else {
          tc::mma<true>(sacc, f[0], f[1], f[2], f[3], qh[j][0], qh[j][1]);
          tc::mma<true>(sacl, f[0], f[1], f[2], f[3], ql[j][0], ql[j][1]);
        }
      }
    } else if constexpr (KS == S_FP8) {
#pragma unroll
      for (int jj = 0; jj < NK / 4; ++jj) {
        const uint4 ra = tm::lds128(sb + kco[jj]);
        const uint4 rb = tm::lds128o<8 * KT::BOXW>(sb + kco[jj]);
        const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w};
        const uint32_t wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 4 * jj + e;
          const uint32_t a0 = tc::e4m3x2_f16x2(wa[e] & 0xffffu), a4 = tc::e4m3x2_f16x2(wa[e] >> 16);
          const uint32_t a2 = tc::e4m3x2_f16x2(wb[e] & 0xffffu), a6 = tc::e4m3x2_f16x2(wb[e] >> 16);
          if constexpr (PK) {
            tc::mma<false>((e & 1) ? sacl : sacc, a0, a2, a4, a6, qh[j][0], qh[j][1]);
          } else {
            tc::mma<false>(sacc, a0, a2, a4, a6, qh[j][0], qh[j][1]);
            tc::mma<false>(sacl, a0, a2, a4, a6, ql[j][0], ql[j][1]);
          }
        }
      }
    } else {  // 4-bit codebook K: k-step j is scale group j
      const uint32_t ks = rks + stg * KT::STILE + ksoff;
      // this head's group scales of tokens g and g+8: NK bytes each
      uint32_t sa[(NK + 3) / 4], sbw[(NK + 3) / 4];
      if constexpr (NK == 4) {
        sa[0] = tm::lds32(ks);
        sbw[0] = tm::lds32o<8 * KT::SBOXW>(ks);
      } else if constexpr (NK == 8) {
        const uint2 x = tm::lds64(ks), y = tm::lds64o<8 * KT::SBOXW>(ks);
        sa[0] = x.x; sa[1] = x.y; sbw[0] = y.x; sbw[1] = y.y;
      } else {
        const uint4 x = tm::lds128(ks), y = tm::lds128o<8 * KT::SBOXW>(ks);
        sa[0] = x.x; sa[1] = x.y; sa[2] = x.z; sa[3] = x.w;
        sbw[0] = y.x; sbw[1] = y.y; sbw[2] = y.z; sbw[3] = y.w;
      }
      const uint32_t selb = (uint32_t)(2 * (c & 1));
      const uint32_t sel0 = 0x7604u | (selb << 4), sel1 = 0x7604u | ((selb + 1) << 4);
      if constexpr (PK) {
        // One MMA per token row of the fragment: A's row g holds the token's
        // hi parts, row g + 8 its lo parts, so that each table entry (hi, lo)
        // is an operand register pair as loaded.  Output rows g / g + 8 are
        // the hi / lo dot products, summed after the scaling.
        float sgh[4] = {0.f, 0.f, 0.f, 0.f};   // token g: (hi, lo) rows x columns 2c, 2c+1
        float sbh[4] = {0.f, 0.f, 0.f, 0.f};   // token g + 8
#pragma unroll
        for (int j = 0; j < NK; ++j) {
          const uint32_t ka = sb + kco[j >> 1];
          const uint32_t wa = (j & 1) ? tm::lds32o<8>(ka) : tm::lds32o<0>(ka);
          const uint32_t wb = (j & 1) ? tm::lds32o<8 + 8 * KT::BOXW>(ka) : tm::lds32o<8 * KT::BOXW>(ka);
          const uint2 xa0 = tm::lds64(tc::prmt(wa, laneoff8, sel0));
          const uint2 xa1 = tm::lds64(tc::prmt(wa, laneoff8, sel1));
          const uint2 xb0 = tm::lds64(tc::prmt(wb, laneoff8, sel0));
          const uint2 xb1 = tm::lds64(tc::prmt(wb, laneoff8, sel1));
          float cg[4], cb[4];
          tm::mma_z(cg, xa0.x, xa0.y, xa1.x, xa1.y, qh[j][0], qh[j][1]);
          tm::mma_z(cb, xb0.x, xb0.y, xb1.x, xb1.y, qh[j][0], qh[j][1]);
          const float2 gs = unpack_f16x2(tc::e4m3x2_f16x2(
              tc::prmt(sa[j >> 2], sbw[j >> 2], (uint32_t)(j & 3) | ((uint32_t)(4 + (j & 3)) << 4))));
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sgh[e] = fmaf(cg[e], gs.x, sgh[e]);
            sbh[e] = fmaf(cb[e], gs.y, sbh[e]);
          }
        }
        sacc[0] = sgh[0]; sacc[1] = sgh[1]; sacc[2] = sbh[0]; sacc[3] = sbh[1];
        sacl[0] = sgh[2]; sacl[1] = sgh[3]; sacl[2] = sbh[2]; sacl[3] = sbh[3];
      } else {
        // q hi and lo in separate operands: rows g / g + 8 are tokens g /
        // g + 8, the hi parts against both, the lo parts against q's hi
        // (fewer live registers than the hi / lo rows above)
#pragma unroll
        for (int j = 0; j < NK; ++j) {
          const uint32_t ka = sb + kco[j >> 1];
          const uint32_t wa = (j & 1) ? tm::lds32o<8>(ka) : tm::lds32o<0>(ka);
          const uint32_t wb = (j & 1) ? tm::lds32o<8 + 8 * KT::BOXW>(ka) : tm::lds32o<8 * KT::BOXW>(ka);
          const uint2 xa0 = tm::lds64(tc::prmt(wa, laneoff8, sel0));
          const uint2 xa1 = tm::lds64(tc::prmt(wa, laneoff8, sel1));
          const uint2 xb0 = tm::lds64(tc::prmt(wb, laneoff8, sel0));
          const uint2 xb1 = tm::lds64(tc::prmt(wb, laneoff8, sel1));
          float cg[4];
          tm::mma_z(cg, xa0.x, xb0.x, xa1.x, xb1.x, qh[j][0], qh[j][1]);
          tc::mma<false>(cg, xa0.x, xb0.x, xa1.x, xb1.x, ql[j][0], ql[j][1]);
          tc::mma<false>(cg, xa0.y, xb0.y, xa1.y, xb1.y, qh[j][0], qh[j][1]);
          const float2 gs = unpack_f16x2(tc::e4m3x2_f16x2(
              tc::prmt(sa[j >> 2], sbw[j >> 2], (uint32_t)(j & 3) | ((uint32_t)(4 + (j & 3)) << 4))));
          float* acc = (j & 1) ? sacl : sacc;
          acc[0] = fmaf(cg[0], gs.x, acc[0]);
          acc[1] = fmaf(cg[1], gs.x, acc[1]);
          acc[2] = fmaf(cg[2], gs.y, acc[2]);
          acc[3] = fmaf(cg[3], gs.y, acc[3]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) sacc[e] += sacl[e];
    if constexpr (PK) {
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[e] += __shfl_xor_sync(0xffffffffu, sacc[e], 2);
    }
  };

  // ---- O^T += V^T . P^T for the slab at sb; p00, p01 (token g), p10, p11
  // (token g+8) are this thread's weights in the accumulator layout.
  auto pv = [&](uint32_t stg, float p00, float p01, float p10, float p11) {
    const uint32_t vd = rvd + stg * VT::TILE;
    if constexpr (!VT::CB) {
      uint32_t b[4];
      p_operand<VS == S_BF16, PK>(p00, p01, p10, p11, c, b);
      if constexpr (VS == S_BF16) {
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          uint32_t f[4];
          if (i < 4) tm::ldsm_x4_to<0>(f, vd + vco[i & 3]);
          else tm::ldsm_x4_to<16 * VT::BOXW>(f, vd + vco[i & 3]);
          tc::mma<true>(o[i], f[0], f[1], f[2], f[3], b[0], b[1]);
          if constexpr (!PK) tc::mma<true>(o[i], f[0], f[1], f[2], f[3], b[2], b[3]);
        }
      } else {  // FP8: tokens 2c, 2c+1, 2c+8, 2c+9; dims g*DPT .. g*DPT + DPT - 1
        constexpr int W = DPT / 4;
        uint32_t w[4][W];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if constexpr (W == 2) {
            const uint2 v = tm::lds64(vd + vco[t]);
            w[t][0] = v.x; w[t][1] = v.y;
          } else {
#pragma unroll
            for (int q4 = 0; q4 < W / 4; ++q4) {
              const uint4 v = tm::lds128(vd + vco[t] + 16 * q4);
              w[t][4 * q4] = v.x; w[t][4 * q4 + 1] = v.y; w[t][4 * q4 + 2] = v.z; w[t][4 * q4 + 3] = v.w;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          const int wi = (2 * i) / 4;
          const uint32_t sel = ((2 * i) % 4 == 0) ? 0x5140u : 0x7362u;
          const uint32_t x01 = tc::prmt(w[0][wi], w[1][wi], sel);
          const uint32_t x23 = tc::prmt(w[2][wi], w[3][wi], sel);
          const uint32_t a0 = tc::e4m3x2_f16x2(x01 & 0xffffu), a2 = tc::e4m3x2_f16x2(x01 >> 16);
          const uint32_t a4 = tc::e4m3x2_f16x2(x23 & 0xffffu), a6 = tc::e4m3x2_f16x2(x23 >> 16);
          tc::mma<false>(o[i], a0, a2, a4, a6, b[0], b[1]);
          if constexpr (!PK) tc::mma<false>(o[i], a0, a2, a4, a6, b[2], b[3]);
        }
      }
    } else {
      // Codebook V: operand tokens (first, second) = (vt0, vt1) and
      // (vt0 + 8, vt1 + 8); the P operand's halves follow that order.
      uint32_t b[4];
      p_operand<false, PK>(p00, p01, p10, p11, c, b);
      if (c & 1) {
#pragma unroll
        for (int e = 0; e < (PK ? 2 : 4); ++e) b[e] = tc::prmt(b[e], b[e], 0x1032u);
      }
      const uint32_t vs = rvs + stg * VT::STILE;
      // group scales of the four tokens: fp16 pairs (first, second)
      uint32_t sc01[HD == 256 ? 2 : 1], sc23[HD == 256 ? 2 : 1];
      {
        constexpr int GB = HD == 256 ? 2 : 1;                       // scale bytes per token
        uint32_t s4[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          s4[t] = GB == 2 ? tm::lds_u16(vs + vso4[t]) : tm::lds_u8(vs + vso4[t]);
#pragma unroll
        for (int q = 0; q < GB; ++q) {
          const uint32_t sq = (uint32_t)q | ((uint32_t)(4 + q) << 4);
          sc01[q] = tc::e4m3x2_f16x2(tc::prmt(s4[0], s4[1], sq));
          sc23[q] = tc::e4m3x2_f16x2(tc::prmt(s4[2], s4[3], sq));
        }
      }
      auto vmma = [&](int i, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t l0_,
                      uint32_t l1_, uint32_t l2_, uint32_t l3_) {
        const int q = (HD == 256 && i >= NK / 2) ? 1 : 0;
        const uint32_t h0 = tc::hmul2(a0, sc01[q]), h1 = tc::hmul2(a1, sc01[q]);
        const uint32_t h2 = tc::hmul2(a2, sc23[q]), h3 = tc::hmul2(a3, sc23[q]);
        const uint32_t w0 = tc::hmul2(l0_, sc01[q]), w1 = tc::hmul2(l1_, sc01[q]);
        const uint32_t w2 = tc::hmul2(l2_, sc23[q]), w3 = tc::hmul2(l3_, sc23[q]);
        tc::mma<false>(o[i], h0, h1, h2, h3, b[0], b[1]);
        if constexpr (!PK) tc::mma<false>(o[i], h0, h1, h2, h3, b[2], b[3]);
        tc::mma<false>(o[i], w0, w1, w2, w3, b[0], b[1]);
      };
      if constexpr (VS == S_T3) {
        // (dim, dim+1) pairs of one token: the 6-bit field at bit 6i of the
        // token's span, looked up and regrouped into (first, second) pairs.
        constexpr int NWD = (VCB_BYTES + 3) / 4 + 1;
        uint32_t wd[4][NWD];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t rb = vd + vco[t];
#pragma unroll
          for (int h = 0; h < NWD; ++h) wd[t][h] = 0;
#pragma unroll
          for (int h = 0; h < VCB_BYTES / 2; ++h) {
            const uint32_t u = tm::lds_u16(rb + 2 * h);
            wd[t][h / 2] |= u << (16 * (h & 1));
          }
        }
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          uint2 e[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int bit = 6 * i, wi = bit >> 5, sh = bit & 31;
            uint32_t f;
            if (sh <= 26) f = wd[t][wi] >> sh;
            else f = __funnelshift_r(wd[t][wi], wd[t][wi + 1], sh);
            e[t] = tm::lds64(((f & 63u) << 8) | vlane8);
          }
          vmma(i, tc::prmt(e[0].x, e[1].x, 0x5410u), tc::prmt(e[0].x, e[1].x, 0x7632u),
               tc::prmt(e[2].x, e[3].x, 0x5410u), tc::prmt(e[2].x, e[3].x, 0x7632u),
               tc::prmt(e[0].y, e[1].y, 0x5410u), tc::prmt(e[0].y, e[1].y, 0x7632u),
               tc::prmt(e[2].y, e[3].y, 0x5410u), tc::prmt(e[2].y, e[3].y, 0x7632u));
        }
      } else {
        // 4-bit / 2-bit codes: code words of the four tokens' spans, then
        // the transposed indices: byte k of L = low nibbles of byte k of the
        // first and second token's words, of H = their high nibbles.
        constexpr int NWD = VCB_BYTES >= 4 ? VCB_BYTES / 4 : 1;
        uint32_t wd[4][NWD];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t ad = vd + vco[t];
          if constexpr (VCB_BYTES == 2) {
            wd[t][0] = tm::lds_u16(ad);
          } else if constexpr (VCB_BYTES == 4) {
            wd[t][0] = tm::lds32(ad);
          } else if constexpr (VCB_BYTES == 8) {
            const uint2 v = tm::lds64(ad);
            wd[t][0] = v.x; wd[t][1] = v.y;
          } else {
            const uint4 v = tm::lds128(ad);
            wd[t][0] = v.x; wd[t][1] = v.y; wd[t][2] = v.z; wd[t][3] = v.w;
          }
        }
#pragma unroll
        for (int h = 0; h < NWD; ++h) {
          const uint32_t L01 = tm::bitsel(wd[0][h], wd[1][h] << 4, 0x0f0f0f0fu);
          const uint32_t H01 = tm::bitsel(wd[0][h] >> 4, wd[1][h], 0x0f0f0f0fu);
          const uint32_t L23 = tm::bitsel(wd[2][h], wd[3][h] << 4, 0x0f0f0f0fu);
          const uint32_t H23 = tm::bitsel(wd[2][h] >> 4, wd[3][h], 0x0f0f0f0fu);
          if constexpr (VS == S_T2) {
            // byte k of L: dims of code nibble 2k (m-tile 8h + 2k), of H:
            // nibble 2k+1 (m-tile 8h + 2k + 1); the quad entry holds both
            // dims' (first, second) pairs, hi then lo
            constexpr int KB = VCB_BYTES >= 4 ? 4 : VCB_BYTES;
#pragma unroll
            for (int k = 0; k < KB; ++k) {
              const uint32_t sel = 0x7604u | ((uint32_t)k << 4);
              const uint4 eL = tm::lds128(tc::prmt(L01, vlane16, sel));
              const uint4 eL2 = tm::lds128(tc::prmt(L23, vlane16, sel));
              vmma(8 * h + 2 * k, eL.x, eL.y, eL2.x, eL2.y, eL.z, eL.w, eL2.z, eL2.w);
              const uint4 eH = tm::lds128(tc::prmt(H01, vlane16, sel));
              const uint4 eH2 = tm::lds128(tc::prmt(H23, vlane16, sel));
              vmma(8 * h + 2 * k + 1, eH.x, eH.y, eH2.x, eH2.y, eH.z, eH.w, eH2.z, eH2.w);
            }
          } else {
            // 4-bit: byte k of L is m-tile 4h + k's row-g pair, of H its row-g+8 pair
            constexpr int KB = VCB_BYTES >= 4 ? 4 : VCB_BYTES;
#pragma unroll
            for (int k = 0; k < KB; ++k) {
              const uint32_t sel = 0x7604u | ((uint32_t)k << 4);
              const uint2 e0 = tm::lds64(tc::prmt(L01, vlane8, sel));
              const uint2 e1 = tm::lds64(tc::prmt(H01, vlane8, sel));
              const uint2 e2 = tm::lds64(tc::prmt(L23, vlane8, sel));
              const uint2 e3 = tm::lds64(tc::prmt(H23, vlane8, sel));
              vmma(4 * h + k, e0.x, e1.x, e2.x, e3.x, e0.y, e1.y, e2.y, e3.y);
            }
          }
        }
      }
    }
  };

  // Zero the V rows (data and this head's scales) of the staged positions
  // that are not attended, so that their products with a zero weight stay 0.
  auto clear_rows = [&](uint32_t stg, uint32_t badmask) {
    if (lane < 16 && ((badmask >> lane) & 1u)) {
      const uint32_t vd = rvd + stg * VT::TILE;
#pragma unroll
      for (int x = 0; x < VT::ROWB; x += 16) {
        if constexpr (VT::ROWB % 16 == 0) tm::sts_zero16(vd + VT::at(lane, x));
      }
      if constexpr (VT::SROW > 0) {
        const uint32_t vs = rvs + stg * VT::STILE + lane * VT::SBOXW + vso;
        if constexpr (VT::SROW >= 16) {
#pragma unroll
          for (int x = 0; x < VT::SROW; x += 16) tm::sts_zero16(vs + x);
        } else if constexpr (VT::SROW == 8) {
          tm::sts_zero8(vs);
        } else {
          tm::sts_zero4(vs);
        }
      }
    }
    __syncwarp();
  };

  int64_t* st = reinterpret_cast<int64_t*>(smem + C::OFF_STATE);
  if (tid == 0) {
    st[0] = x0;
    st[1] = x_end;
    st[2] = seq;
    st[4] = off;
    st[7] = cpc;
  }
  constexpr float kLazy = 8.0f;    // the running maximum trails by at most this (log2 units)
  constexpr float kNoMax = -1e30f;  // running maximum before any score (finite: exp2 of
                                    // a masked score minus it is 0, never NaN)
  // state of the open stretch (set by open_stretch)
  int s_sq = 0, s_nsl = 0, s_my = 0;
  bool s_any_bad = false;
  float xq0[E];   // this warp's first query row, requested with the unit's first copies
  // query row j of the unit's sequence (rows >= rep zero)
  auto q_row = [&](int j, float (&xq)[E]) {
#pragma unroll
    for (int i = 0; i < E; ++i) xq[i] = 0.f;
    if (j < a.rep) {
      const int64_t qoff = (int64_t)s_sq * a.q_stride + (int64_t)(kvh * a.rep + j) * HD + lane * E;
#pragma unroll
      for (int i = 0; i < E; ++i)
        xq[i] = a.q_bf16 ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(a.q)[qoff + i])
                         : reinterpret_cast<const float*>(a.q)[qoff + i];
    }
  };
  // Unit bounds from the CTA loop state (st[0] = next slab of the range,
  // st[2] its sequence, st[4] the slab offset in it): st[5], st[6] = the
  // unit's first and end slab.  False when the range is done.
  auto open_unit = [&]() -> bool {
    const int64_t x = st[0];
    if (x >= st[1]) return false;
    int first, n, len;
    seq_slabs((int)st[2], first, n, lo, len);
    if (tid == 0) {
      st[5] = first + st[4];
      st[6] = first + st[4] + min((int64_t)n - st[4], st[1] - x);
    }
    return true;
  };
  // Next stretch of the unit (after a __syncthreads): its block ids into
  // shared memory, then each warp's first copies (the first stretch of a
  // unit also requests the warp's first query row before them: behind them
  // in the memory queues it would wait for their bytes).  False when the
  // unit has no slabs left.  Called by every thread.
  auto open_stretch = [&](bool first_stretch) -> bool {
    const int64_t sa = st[5], s_hi = st[6];
    if (sa >= s_hi) return false;
    s_sq = (int)st[2];
    int first, n, len;
    seq_slabs(s_sq, first, n, lo, len);
    const int sub = (C::MAXP - 1) * bs / SLAB;
    s_nsl = (int)min((int64_t)sub, s_hi - sa);
    tok0 = (int)(sa * SLAB);
    tok_end = min(tok0 + s_nsl * SLAB, len);
    p0 = tok0 >> lbs;
    const int p1 = ((tok_end - 1) >> lbs) + 1;
    const int64_t tab = (int64_t)s_sq * a.max_blocks;
    int bad_ids = 0;
    for (int i = tid; i < p1 - p0; i += NT) {
      const int64_t b = a.block_tables[tab + p0 + i];
      const bool bad = b < 0 || (a.num_blocks > 0 && b >= a.num_blocks);
      if (bad && a.err) atomicOr(a.err, 2);
      bad_ids |= bad;
      blk_s[i] = bad ? -1 : (int)b;
    }
    s_any_bad = __syncthreads_or(bad_ids) != 0;   // in this stretch
    if (tid == 0) st[5] = sa + s_nsl;
    s_my = s_nsl > warp ? (s_nsl - 1 - warp) / NW + 1 : 0;
    if (first_stretch && merged) dirty = true;   // the previous unit's merge wrote over the rings
    if (first_stretch && warp < 8) q_row(warp, xq0);
    for (int s = 0; s < NST && s < s_my; ++s) issue(s, (gk + (uint32_t)s) % NST);
    return true;
  };
  // the next unit's first stretch was opened during this unit's merge
  bool pre_opened = false;
  for (;;) {
    __syncthreads();   // (a pre-opened unit: the previous merge is done with q_s)
    if (!pre_opened && !open_unit()) break;
#pragma unroll
    for (int i = 0; i < NK; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m0 = m1 = kNoMax;
    l0 = l1 = 0.f;
    for (int first_stretch = 1;; first_stretch = 0) {
      if (!(first_stretch && pre_opened)) {
        __syncthreads();
        if (!open_stretch(first_stretch != 0)) break;
      }
      pre_opened = false;
      const int my = s_my;
      const bool any_bad_id = s_any_bad;
      if (first_stretch) {
        // ---- queries (rotated when K is stored rotated), rows >= rep zero
        for (int j = warp; j < 8; j += NW) {
          float xq[E];
          if (j == warp) {
#pragma unroll
            for (int i = 0; i < E; ++i) xq[i] = xq0[i];
          } else {
            q_row(j, xq);
          }
          if constexpr (side_rotated(KS)) fwht_warp<E>(xq, lane, a.inv_sqrt_hd);
#pragma unroll
          for (int i = 0; i < E; ++i) q_s[j * HD + lane * E + i] = xq[i];
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < NK; ++j) {
          int d[4];
          k_slot_dims<KS, HD>(j, c, d);
          const float* qr = q_s + (PK ? (g & 3) : g) * HD;
          uint32_t h0, lq0, h1, lq1;
          tc::split2<KS == S_BF16>(qr[d[0]], qr[d[1]], h0, lq0);
          tc::split2<KS == S_BF16>(qr[d[2]], qr[d[3]], h1, lq1);
          if constexpr (PK) {
            qh[j][0] = g < 4 ? h0 : lq0;
            qh[j][1] = g < 4 ? h1 : lq1;
          } else {
            qh[j][0] = h0; ql[j][0] = lq0;
            qh[j][1] = h1; ql[j][1] = lq1;
          }
        }
      }
      int consumed = 0;
      uint32_t stg = gk % NST, ph = (gk / NST) & 1u;   // stage and phase of slab s
      for (int s = 0; s < my; ++s, stg = stg + 1 == NST ? (ph ^= 1u, 0u) : stg + 1) {
        const int slab_pos = tok0 + (warp + NW * s) * SLAB;
        if (!failed && !tm::bar_wait(bar0 + stg * 8, ph)) {
          failed = true;
          if (lane == 0 && a.err) atomicOr(a.err, 4);   // KVQ_DEVERR_TIMEOUT
        }
        if (failed) continue;
        consumed = s + 1;
        // rows of the slab that are not attended (outside [lo, tok_end) or
        // in a page whose id is invalid): warp-uniform, usually none
        uint32_t bad = 0;
        if (slab_pos < lo || slab_pos + SLAB > tok_end || bs < 16) {
          const int t = lane & 15;
          const int pos = slab_pos + t;
          bool ok = pos >= lo && pos < tok_end;
          if (ok) ok = blk_s[(pos >> lbs) - p0] >= 0;
          bad = __ballot_sync(0xffffffffu, !ok) & 0xffffu;
        } else if (any_bad_id) {
          if (blk_s[(slab_pos >> lbs) - p0] < 0) bad = 0xffffu;
        }
        if (bad == 0xffffu) {   // nothing to attend here
          __syncwarp();
          if (s + NST < my) issue(s + NST, stg);
          continue;
        }
        if (bad) {
          clear_rows(stg, bad);
          dirty = true;
        }

        float sv[4];
        scores(stg, sv);
        sv[0] *= scale; sv[1] *= scale; sv[2] *= scale; sv[3] *= scale;
        if (bad) {
          const bool va = !((bad >> g) & 1u), vb = !((bad >> (g + 8)) & 1u);
          if (!va) sv[0] = sv[1] = -CUDART_INF_F;
          if (!vb) sv[2] = sv[3] = -CUDART_INF_F;
        }
        // ---- lazy online softmax (columns 2c, 2c+1)
        const bool up = fmaxf(sv[0], sv[2]) > m0 + kLazy || fmaxf(sv[1], sv[3]) > m1 + kLazy;
        if (__any_sync(0xffffffffu, up)) {
          float mx0 = fmaxf(sv[0], sv[2]), mx1 = fmaxf(sv[1], sv[3]);
#pragma unroll
          for (int msk = 4; msk < 32; msk <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, msk));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, msk));
          }
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
          const float al0 = tm::ex2(m0 - mn0), al1 = tm::ex2(m1 - mn1);
          l0 *= al0;
          l1 *= al1;
#pragma unroll
          for (int i = 0; i < NK; ++i) {
            o[i][0] *= al0; o[i][1] *= al1; o[i][2] *= al0; o[i][3] *= al1;
          }
          m0 = mn0;
          m1 = mn1;
        }
        float pw[4];
        pw[0] = tm::ex2(sv[0] - m0);
        pw[1] = tm::ex2(sv[1] - m1);
        pw[2] = tm::ex2(sv[2] - m0);
        pw[3] = tm::ex2(sv[3] - m1);
        l0 += pw[0] + pw[2];
        l1 += pw[1] + pw[3];
        bool pv_any = true;
        if (a.sparse_thr > 0.f) {  // drop weights <= thr x (this warp's running sum)
          float t0 = l0, t1 = l1;
#pragma unroll
          for (int msk = 4; msk < 32; msk <<= 1) {
            t0 += __shfl_xor_sync(0xffffffffu, t0, msk);
            t1 += __shfl_xor_sync(0xffffffffu, t1, msk);
          }
          if (pw[0] <= a.sparse_thr * t0) pw[0] = 0.f;
          if (pw[2] <= a.sparse_thr * t0) pw[2] = 0.f;
          if (pw[1] <= a.sparse_thr * t1) pw[1] = 0.f;
          if (pw[3] <= a.sparse_thr * t1) pw[3] = 0.f;
          pv_any = __any_sync(0xffffffffu, pw[0] != 0.f || pw[1] != 0.f || pw[2] != 0.f || pw[3] != 0.f);
        }
        if (pv_any) pv(stg, pw[0], pw[1], pw[2], pw[3]);
        __syncwarp();
        if (s + NST < my) issue(s + NST, stg);
      }
      if (failed) {
        // copies of this stretch still in flight: wait for them (bounded)
        // before the stages are reused or the CTA exits
        const int issued = my < consumed + NST ? my : consumed + NST;
        for (int s = consumed; s < issued; ++s)
          tm::bar_wait(bar0 + ((gk + (uint32_t)s) % NST) * 8, ((gk + (uint32_t)s) / NST) & 1u);
      }
      gk += (uint32_t)my;
    }

    merged = true;
    // ---- merge of the unit's warps (as decode_tc_kernel)
    const int64_t x = st[0], off_u = st[4];
    const int seq_u = (int)st[2], kvh_u = kvh;
    int first_u, n_u, len_u, lo_u;
    seq_slabs(seq_u, first_u, n_u, lo_u, len_u);
    const int64_t take = min((int64_t)n_u - off_u, st[1] - x);
    const int64_t ou = x - off_u, cp = st[7];
    const int64_t vu = ou + C::SWITCH * (int64_t)(seq_u + 1);   // the row's first slab on the virtual line
    const int slot = (int)(jr - vu / cp);
    const int np = (int)((vu + n_u - 1) / cp - vu / cp + 1);
#pragma unroll
    for (int msk = 4; msk < 32; msk <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, msk);
      l1 += __shfl_xor_sync(0xffffffffu, l1, msk);
    }
    if constexpr (PK) {
#pragma unroll
      for (int i = 0; i < NK; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[i][e] += __shfl_xor_sync(0xffffffffu, o[i][e], 2);
    }
    const bool writer = !PK || c < 2;
    __syncthreads();  // every warp is done with its ring
    float* mo = reinterpret_cast<float*>(smem + C::OFF_MERGE);  // [NW][8 heads][HD]
    float* ml = mo + NW * 8 * HD;                                // [NW][8 heads][m, l]
    if (writer) {
#pragma unroll
      for (int i = 0; i < NK; ++i) {
        const int da = tm_v_row_dim<VS, HD>(i, g), db = tm_v_row_dim<VS, HD>(i, g + 8);
        mo[(warp * 8 + 2 * c) * HD + da] = o[i][0];
        mo[(warp * 8 + 2 * c + 1) * HD + da] = o[i][1];
        mo[(warp * 8 + 2 * c) * HD + db] = o[i][2];
        mo[(warp * 8 + 2 * c + 1) * HD + db] = o[i][3];
      }
    }
    if (g == 0 && writer) {
      ml[(warp * 8 + 2 * c) * 2] = m0;
      ml[(warp * 8 + 2 * c) * 2 + 1] = l0;
      ml[(warp * 8 + 2 * c + 1) * 2] = m1;
      ml[(warp * 8 + 2 * c + 1) * 2 + 1] = l1;
    }
    __syncthreads();
    float* red_s = reinterpret_cast<float*>(scan_s + 36);
    int* last_s = reinterpret_cast<int*>(scan_s + 44);
    for (int idx = tid; idx < a.rep * HD; idx += NT) {
      const int r = idx / HD, d = idx - r * HD;
      float M = -CUDART_INF_F;
#pragma unroll
      for (int w2 = 0; w2 < NW; ++w2) M = fmaxf(M, ml[(w2 * 8 + r) * 2]);
      float acc = 0.f, lsum = 0.f;
      if (M != -CUDART_INF_F) {
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2) {
          const float mw = ml[(w2 * 8 + r) * 2];
          const float f = mw == -CUDART_INF_F ? 0.f : exp2f(mw - M);
          acc = fmaf(mo[(w2 * 8 + r) * HD + d], f, acc);
          lsum = fmaf(ml[(w2 * 8 + r) * 2 + 1], f, lsum);
        }
      }
      q_s[r * HD + d] = acc * a.v_mult;
      if (d == 0) {
        red_s[2 * r] = M;
        red_s[2 * r + 1] = lsum;
      }
    }
    // The rings are free again: advance the CTA loop state and open the next
    // unit's first stretch now, so that its first copies are in flight while
    // this unit's partials go out (global stores, the counter's round trip
    // and the last arriver's merge).  Measured on GB300: long-context Turbo4
    // K 315.7 -> 307.8, ragged FP8 K with Turbo2 V 219.3 -> 216.6 us; with
    // BF16 K (the largest burst of copies) the partials waited behind them
    // (llama8b 90.6 -> 91.9 us), and FP8 K and V (two CTAs per SM) measured
    // 57.4 against 56.5 us without it, so those open the unit afterwards.
    if (tid == 0) {
      int s2 = seq_u, n2 = 0;
      do {
        ++s2;
        if (s2 >= N) break;
        int f2, l2, e2;
        seq_slabs(s2, f2, n2, l2, e2);
      } while (n2 == 0);
      st[0] = x + take;
      st[2] = s2 < N ? s2 : N - 1;
      st[4] = 0;
      if (s2 >= N) st[1] = st[0];
    }
    __syncthreads();
    if (KS != S_BF16 && !(KS == S_FP8 && !C::LUT) && open_unit()) {
      __syncthreads();
      pre_opened = open_stretch(true);
    }
    const int64_t row0 = (int64_t)seq_u * a.nq + kvh_u * a.rep;
    float* part0 = a.part + row0 * a.kmax * (HD + 4);
    auto finish_row = [&](int r, float (&xr)[E], float lsum) {
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) xr[e] *= inv;
      if constexpr (side_rotated(VS)) fwht_warp<E>(xr, lane, a.inv_sqrt_hd);
      const int64_t o_ = (row0 + r) * HD + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (a.out_bf16) reinterpret_cast<uint16_t*>(a.out)[o_ + e] = bf16_bits_from_float(xr[e]);
        else reinterpret_cast<float*>(a.out)[o_ + e] = xr[e];
      }
    };
    if (np == 1) {
      for (int r = warp; r < a.rep; r += NW) {
        float xr[E];
#pragma unroll
        for (int e = 0; e < E; ++e) xr[e] = q_s[r * HD + lane * E + e];
        finish_row(r, xr, red_s[2 * r + 1]);
      }
    } else {
      // The CTA of the row's first slab (slot 0) works on the row last in its
      // range, usually after the row's other CTAs, which start their ranges
      // on it, have arrived: it then reads the counter once and merges with
      // its own partial from shared memory (no partial store, fence or
      // atomic round trip).  Otherwise, and for the other slots, the partial
      // goes out and the last of the row's CTAs to arrive merges.  Measured
      // on GB300 (same box): BF16 92.6 -> 91.9, FP8 57.8 -> 57.4, ragged
      // fp8k_turbo2v 202.8 -> 201.0 us; with a codebook K side the extra
      // code cost registers in the slab loop (turbo4 80.1 -> 81.4,
      // long-context 310.9 -> 317.7 us), so those keep the plain path.
      constexpr bool kFastMerge = !KT::CB;
      int* ctr = a.counters + (int64_t)seq_u * nkv + kvh_u;
      if (kFastMerge && slot == 0) {
        if (tid == 0) {
          int arrived;
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(arrived) : "l"(ctr) : "memory");
          *last_s = arrived == np - 1 ? 2 : 0;
          if (arrived == np - 1) *ctr = 0;   // every other CTA of the row is done with it
        }
        __syncthreads();
      }
      const bool own = kFastMerge && slot == 0 && *last_s == 2;   // slot 0's partial stays in shared memory
      if (!own) {
        for (int idx = tid; idx < a.rep * (HD + 4); idx += NT) {
          const int r = idx / (HD + 4), d = idx - r * (HD + 4);
          float v = 0.f;
          if (d < 2) v = red_s[2 * r + d];
          else if (d >= 4) v = q_s[r * HD + d - 4];
          part0[((int64_t)r * a.kmax + slot) * (HD + 4) + d] = v;
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
          const int prev = atomicAdd(ctr, 1);
          *last_s = prev == np - 1;
          if (prev == np - 1) *ctr = 0;
        }
        __syncthreads();
      }
      if (*last_s) {
        __threadfence();
        for (int r = warp; r < a.rep; r += NW) {
          // one pass over the partials, four loaded at a time, with the
          // running maximum rescaling what is summed so far
          const float* pr = part0 + (int64_t)r * a.kmax * (HD + 4);
          float mm = -CUDART_INF_F, ll = 0.f;
          float xr[E];
#pragma unroll
          for (int e = 0; e < E; ++e) xr[e] = 0.f;
          for (int i0 = 0; i0 < np; i0 += 4) {
            float mi[4], li[4], xi[4][E];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float* pi = pr + (i0 + u) * (HD + 4);
              const bool in = i0 + u < np;
              if (own && i0 + u == 0) {   // this CTA's partial, from shared memory
                mi[u] = red_s[2 * r];
                li[u] = red_s[2 * r + 1];
#pragma unroll
                for (int e = 0; e < E; ++e) xi[u][e] = q_s[r * HD + lane * E + e];
                continue;
              }
              mi[u] = in ? __ldcg(pi) : -CUDART_INF_F;
              li[u] = in ? __ldcg(pi + 1) : 0.f;
#pragma unroll
              for (int e = 0; e < E; ++e) xi[u][e] = in ? __ldcg(pi + 4 + lane * E + e) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (mi[u] == -CUDART_INF_F) continue;
              if (mi[u] > mm) {
                const float sc = mm == -CUDART_INF_F ? 0.f : exp2f(mm - mi[u]);
                ll *= sc;
#pragma unroll
                for (int e = 0; e < E; ++e) xr[e] *= sc;
                mm = mi[u];
              }
              const float w = exp2f(mi[u] - mm);
              ll = fmaf(li[u], w, ll);
#pragma unroll
              for (int e = 0; e < E; ++e) xr[e] = fmaf(xi[u][e], w, xr[e]);
            }
          }
          finish_row(r, xr, ll);
          float* pz = part0 + (int64_t)r * a.kmax * (HD + 4);
          for (int i = lane; i < np * (HD + 4); i += 32) pz[i] = 0.f;
        }
      }
    }

  }
}

template <int KS, int VS, int HD, bool PK>
cudaError_t launch_tma_kern(const DecodeArgs& a, const TmaMaps& maps, const Codebooks& cb,
                            cudaStream_t st) {
  using C = TmCfg<KS, VS, HD, PK>;
  static_assert(C::SMEM <= kSmemLimit, "shared memory budget");
  static_assert(C::NST >= 2, "at least two stages per warp");
  auto kern = decode_tma_kernel<KS, VS, HD, PK>;
  static int attr_dev = -1;   // the device whose attribute was set last
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (attr_dev != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_dev = dev;
  }
  const int ranges = max(1, min(a.max_ranges, C::CPS * a.sms / a.nkv));
  kern<<<ranges * a.nkv, 32 * C::NW, C::SMEM, st>>>(a, maps, cb);
  return cudaGetLastError();
}

template <int KS, int VS, int HD>
cudaError_t launch_tma_inst(const DecodeArgs& a, const TmaMaps& maps, const Codebooks& cb,
                            cudaStream_t st) {
  return a.rep <= 4 ? launch_tma_kern<KS, VS, HD, true>(a, maps, cb, st)
                    : launch_tma_kern<KS, VS, HD, false>(a, maps, cb, st);
}

}  // namespace kvq
