// Device pieces shared by the chunked-prefill kernels: the per-sequence
// prologue, the query-tile lookup, the validity checks and the sheared-bias
// loads from a rel box.
#pragma once

#include "relattn_common.cuh"
#include "relattn_internal.h"

namespace relattn {
namespace prefill {

constexpr int kQRows = 128;  // query rows of one tile (the M of every MMA)
// rel boxes: 32 query rows x 100 distances, one per softmax warp.  Row r of a
// box needs the 64 distances P_r - j0 - 63 .. P_r - j0; across 32 rows that is
// 95, plus up to 3 for rounding the box start down to 16 bytes.  Lane l reads
// word 101 l + const - c: 101 is odd, so the 32 lanes hit 32 banks.
constexpr int kRelBoxRows = 32, kRelBoxCols = 100;
constexpr int kRelBoxBytes = kRelBoxRows * kRelBoxCols * 4;  // 12800
constexpr int kRelBoxes = kQRows / kRelBoxRows;              // 4 per tile
// bf16 rel boxes: the box start rounds down to 8 distances (16 bytes), so
// 95 + 7 columns are needed: 104 (208-byte rows).  Rows are read as 8-byte
// pieces (4 distances), whose alignment is the same across a warp.
constexpr int kRelBoxCols16 = 104;
constexpr int kRelBoxBytes16 = kRelBoxRows * kRelBoxCols16 * 2;  // 6656 (52 x 128)
constexpr int kQTileBytes = kQRows * kDqk * 2;                   // 32 KB
constexpr int kKStageBytes = kTileKeys * kDqk * 2;               // 16 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleNat = 5.5451774f;  // move the running max only past e^(8 ln 2)

__device__ __forceinline__ bool seq_ok(int ctx, int n, int max_blocks) {
  return ctx >= 0 && n >= 0 &&
         static_cast<long long>(ctx) + n <= static_cast<long long>(max_blocks) * kBlockSize;
}

// Rows [cu0, cu1) are a valid chunk of the packed [T] token rows.
__device__ __forceinline__ bool rows_ok(int cu0, int cu1, int T) {
  return cu0 >= 0 && cu1 >= cu0 && cu1 <= T;
}

// Per-sequence arrays a CTA keeps in shared memory: first packed row, row
// count (0 for an invalid sequence), cached prefix, and the prefix sum of
// query tiles (B + 1 entries).
struct SeqArrays {
  int* cu0;
  int* n;
  int* ctx;
  int* qpref;
};

// Per-CTA prologue: fills the arrays and returns the number of 128-row query
// tiles over all sequences.  zero_bad: CTA 0 writes zeros to the output rows
// of a sequence whose lengths are invalid (its rows are skipped).
__device__ inline int prologue(const PrefillParams& p, SeqArrays a, bool zero_bad) {
  const int tid = threadIdx.x;
  for (int b = tid; b < p.B; b += blockDim.x) {
    const int c0 = p.cu_seqlens[b], c1 = p.cu_seqlens[b + 1], ctx = p.ctx_lens[b];
    const bool ok = rows_ok(c0, c1, p.T) && seq_ok(ctx, c1 - c0, p.max_blocks);
    a.cu0[b] = c0;
    a.n[b] = ok ? c1 - c0 : 0;
    a.ctx[b] = ctx;
    // query tiles of this sequence, kept in qpref until the scan
    a.qpref[b] = ok ? (c1 - c0 + kQRows - 1) / kQRows : 0;
    if (!ok && zero_bad && blockIdx.x == 0 && rows_ok(c0, c1, p.T)) {
      const int per = p.Hq * p.dv * (p.out_f32 ? 4 : 2) / 4;  // 32-bit words per row
      uint32_t* o = static_cast<uint32_t*>(p.out);
      for (int r = c0; r < c1; ++r)  // a skipped sequence's rows are zero
        for (int i = 0; i < per; ++i) o[static_cast<size_t>(r) * per + i] = 0u;
    }
  }
  __syncthreads();
  if (tid < 32) {
    const int lane = tid;
    const int chunk = (p.B + 31) / 32;
    const int beg = lane * chunk, end = min(p.B, beg + chunk);
    int sum = 0;
    for (int i = beg; i < end; ++i) sum += a.qpref[i];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int i = beg; i < end; ++i) {
      const int cnt = a.qpref[i];
      a.qpref[i] = run;
      run += cnt;
    }
    if (lane == 31) a.qpref[p.B] = incl;
  }
  __syncthreads();
  return a.qpref[p.B];
}

// out[j] = in[(j + rot) & 7] for 8 chunks of 4 words (rot 0 .. 7), by three
// conditional rotations.  A lane that reads or writes a 128-byte-swizzled
// row's chunks starting at chunk lane & 7 spreads the 8 lanes of each
// quarter-warp (rows 4 apart here) over all 8 bank groups; this puts the
// chunks back in order (or into that order).
__device__ __forceinline__ void rotate_chunks(uint32_t (&w)[32], int rot) {
#pragma unroll
  for (int b = 1; b < 8; b <<= 1) {
    const bool on = (rot & b) != 0;
    uint32_t t[32];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) t[4 * j + e] = on ? w[4 * ((j + b) & 7) + e] : w[4 * j + e];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = t[i];
  }
}

// The eight 16-byte chunks of row `row` of a 128-byte-swizzled half tile at
// `base` (rows of 128 bytes), in chunk order, read starting at chunk lane & 7
// (conflict-free when the lanes' rows are 4 apart; see rotate_chunks).
__device__ __forceinline__ void load_row128(const uint8_t* base, int row, int lane,
                                            uint32_t (&w)[32]) {
  const int rot = lane & 7;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint4 v = *reinterpret_cast<const uint4*>(base + sw128(row, (s + rot) & 7));
    w[4 * s] = v.x;
    w[4 * s + 1] = v.y;
    w[4 * s + 2] = v.z;
    w[4 * s + 3] = v.w;
  }
  rotate_chunks(w, (8 - rot) & 7);  // back to chunk order
}

// Query tile qtg (0 .. tiles - 1): its sequence, first packed row, valid rows,
// position of its first row, and its window-aware range of 64-key tiles
// [tf, tf + ntiles): the tiles holding a key that one of its rows sees.
struct QTile {
  int b, r0, rows, P0, tf, ntiles;
};

__device__ __forceinline__ QTile query_tile(int qtg, const PrefillParams& p,
                                            const SeqArrays& a) {
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {  // largest b with qpref[b] <= qtg
    const int mid = (lo + hi + 1) >> 1;
    if (a.qpref[mid] <= qtg)
      lo = mid;
    else
      hi = mid - 1;
  }
  QTile t;
  t.b = lo;
  const int qt = qtg - a.qpref[lo];
  t.r0 = a.cu0[lo] + qt * kQRows;
  t.rows = min(kQRows, a.n[lo] - qt * kQRows);
  t.P0 = a.ctx[lo] + qt * kQRows;
  t.tf = window_lo(t.P0, p.window) / kTileKeys;
  t.ntiles = (t.P0 + t.rows - 1) / kTileKeys - t.tf + 1;
  return t;
}

// Key tile `tile` (64 keys) of a sequence whose block-table row is trow: the
// physical block holding it, whether that id is inside the pool, and the
// tile's first row in the cache's [blocks * 128] token rows.
struct KvTile {
  int id, row;
  bool ok;
};

__device__ __forceinline__ KvTile kv_tile(const int* trow, int tile, int num_blocks) {
  KvTile t;
  t.id = __ldg(trow + (tile >> 1));
  t.ok = t.id >= 0 && t.id < num_blocks;
  t.row = t.id * kBlockSize + (tile & 1) * kTileKeys;
  return t;
}

// x2[i] = (x[2 i], x[2 i + 1]), x[c] = s[c] * scale + rel, for the 64
// columns of one query row, from 17 aligned 16-byte loads.  p4 points A
// floats before the row's lowest needed distance (the one of column 63);
// distances rise towards column 0, so float q of the loads belongs to column
// 63 - q + A.  (Two scalar FMAs per pair: the two distances of a pair sit in
// memory in the opposite order to the pair's columns.)
template <int A>
__device__ __forceinline__ void rel_fma(uint64_t (&x2)[32], const uint32_t (&sr)[64],
                                        const float4* p4, float scale) {
  float rf[68];
#pragma unroll
  for (int w = 0; w < 17; ++w) {
    const float4 v = p4[w];
    rf[4 * w] = v.x;
    rf[4 * w + 1] = v.y;
    rf[4 * w + 2] = v.z;
    rf[4 * w + 3] = v.w;
  }
#pragma unroll
  for (int i = 0; i < 32; ++i)
    x2[i] = f2(fmaf(__uint_as_float(sr[2 * i]), scale, rf[63 - 2 * i + A]),
               fmaf(__uint_as_float(sr[2 * i + 1]), scale, rf[62 - 2 * i + A]));
}

// The same from bf16 rel: 17 aligned 8-byte loads of four distances; bf16 q
// sits in word q / 2, in its high half when q is odd.  Each pair's scores are
// scaled by one paired multiply, and each bias joins its score in a
// mixed-precision add (no widening instruction).
template <int A>
__device__ __forceinline__ void rel_fma16(uint64_t (&x2)[32], const uint32_t (&sr)[64],
                                          const uint2* p2, uint64_t scale2) {
  uint32_t w[34];
#pragma unroll
  for (int k = 0; k < 17; ++k) {
    const uint2 v = p2[k];
    w[2 * k] = v.x;
    w[2 * k + 1] = v.y;
  }
  auto plus_rel = [&](int c, float t) -> float {
    const int q = 63 - c + A;
    return (q & 1) ? add_bf16_f32<true>(w[q >> 1], t) : add_bf16_f32<false>(w[q >> 1], t);
  };
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint64_t t2 = mul_f2(f2u(sr[2 * i], sr[2 * i + 1]), scale2);
    x2[i] = f2(plus_rel(2 * i, f2lo(t2)), plus_rel(2 * i + 1, f2hi(t2)));
  }
}

// The scaled scores plus the sheared bias of one query row for one 64-key
// tile whose rel boxes sit at `slot`, as pairs of columns (x2[i] holds
// columns 2 i and 2 i + 1): row r of the tile (box r / 32, row r % 32 in it),
// P0 the position of the tile's first row.  Every distance of the tile past
// rel_extent: pass has_rel = false (no bias).
template <bool R16>
__device__ __forceinline__ void scores_with_bias(uint64_t (&x2)[32], const uint32_t (&sr)[64],
                                                 const uint8_t* slot, int r, int P0,
                                                 bool has_rel, float scale) {
  const int rbox = r / kRelBoxRows, rrow = r % kRelBoxRows;
  const uint64_t scale2 = f2(scale, scale);
  if (!has_rel) {
#pragma unroll
    for (int i = 0; i < 32; ++i) x2[i] = mul_f2(f2u(sr[2 * i], sr[2 * i + 1]), scale2);
    return;
  }
  if constexpr (R16) {
    // A box starts at distance (P0 + 32 box - j0 - 63) rounded down to 8, so
    // column 63's distance sits rrow + ((P0 + 1) & 7) into this row; it is
    // read from the 4-distance piece below it.
    const int col = rrow + ((P0 + 1) & 7);
    const uint2* p2 = reinterpret_cast<const uint2*>(
        reinterpret_cast<const __nv_bfloat16*>(slot + rbox * kRelBoxBytes16) +
        rrow * kRelBoxCols16 + (col & ~3));
    switch (col & 3) {  // rrow = 4 lane + q4 (mod 32): the same for the warp
      case 0: rel_fma16<0>(x2, sr, p2, scale2); break;
      case 1: rel_fma16<1>(x2, sr, p2, scale2); break;
      case 2: rel_fma16<2>(x2, sr, p2, scale2); break;
      default: rel_fma16<3>(x2, sr, p2, scale2); break;
    }
  } else {
    // A box starts at distance (P0 + 32 box - j0 - 63) rounded down to 4, so
    // column 63's distance sits rrow + ((P0 + 1) & 3) into this row.
    const int col = rrow + ((P0 + 1) & 3);
    const float4* p4 = reinterpret_cast<const float4*>(
        reinterpret_cast<const float*>(slot + rbox * kRelBoxBytes) + rrow * kRelBoxCols +
        (col & ~3));
    switch (col & 3) {  // the same for every lane of the warp
      case 0: rel_fma<0>(x2, sr, p4, scale); break;
      case 1: rel_fma<1>(x2, sr, p4, scale); break;
      case 2: rel_fma<2>(x2, sr, p4, scale); break;
      default: rel_fma<3>(x2, sr, p4, scale); break;
    }
  }
}

// Hidden columns of a row (outside [clo, clo + span)) to -inf, and the row's
// maximum over its pairs of columns (three-input max).
__device__ __forceinline__ float mask_and_max(uint64_t (&x2)[32], bool warp_full, int clo,
                                              int span) {
  if (!warp_full) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float lo = static_cast<unsigned>(2 * i - clo) < static_cast<unsigned>(span)
                           ? f2lo(x2[i]) : kNegInf;
      const float hi = static_cast<unsigned>(2 * i + 1 - clo) < static_cast<unsigned>(span)
                           ? f2hi(x2[i]) : kNegInf;
      x2[i] = f2(lo, hi);
    }
  }
  float mq[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
#pragma unroll
  for (int i = 0; i < 32; ++i) mq[i & 3] = fmax3(mq[i & 3], f2lo(x2[i]), f2hi(x2[i]));
  return fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
}

// P = exp2(x l2f + mb) for a row's 64 columns, packed in pairs (bf16, or f16
// when F16) into pk, and the sum of the 64 values (before packing).
template <bool F16>
__device__ __forceinline__ float exp_pack(const uint64_t (&x2)[32], float l2f, float mb,
                                          uint32_t (&pk)[32]) {
  const uint64_t l2f2 = f2(l2f, l2f), mb2 = f2(mb, mb);
  uint64_t sq[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint64_t a2 = fma_f2(x2[i], l2f2, mb2);
    const float p0 = ex2(f2lo(a2)), p1 = ex2(f2hi(a2));
    sq[i & 1] = add_f2(sq[i & 1], f2(p0, p1));
    pk[i] = F16 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
  }
  const uint64_t sqt = add_f2(sq[0], sq[1]);
  return f2lo(sqt) + f2hi(sqt);
}

// bf16 rel boxes for 128-key tiles: 32 query rows x 200 distances.  A row
// needs the 128 distances P_r - j0 - 127 .. P_r - j0; across 32 rows that is
// 159, plus up to 7 for rounding the box start down to 16 bytes, plus 32 in
// the odd boxes, which start 32 distances lower.  Why: a warp's lanes read
// rows 4 apart from all four boxes (8 rows each); with 100-word rows the 8
// rows of one box fall on 8 distinct even bank pairs, and the 32-distance
// (16-word) shift of the odd boxes moves theirs onto the other 16 banks, so an
// 8-byte load of the warp uses every bank exactly twice (two wavefronts, the
// least for 256 bytes) instead of 16 banks four times.
constexpr int kRelColsW = 200;
constexpr int kRelBoxBytesW = kRelBoxRows * kRelColsW * 2;  // 12800 (100 x 128)
constexpr int kRelOddShift = 32;                            // distances, odd boxes

// The pairs of rel_fma16: x2[i] = (x[2 i], x[2 i + 1]) = s * scale + rel for
// columns 2 i and 2 i + 1, from 17 aligned 8-byte loads of four bf16
// distances; p2 points A distances before the lowest needed one (column
// 63's), distances rise towards column 0.
template <int A>
__device__ __forceinline__ void rel_fma16_x2(uint64_t (&x2)[32], const uint32_t (&sr)[64],
                                             const uint2* p2, uint64_t scale2) {
  uint32_t w[34];
#pragma unroll
  for (int k = 0; k < 17; ++k) {
    const uint2 v = p2[k];
    w[2 * k] = v.x;
    w[2 * k + 1] = v.y;
  }
  // distance u (from the load's start) of column c is 63 - c + A: bf16 u
  // sits in word u / 2, in its high half when u is odd.  The scaled score
  // and the bf16 bias meet in one mixed-precision add.
  auto plus_rel = [&](int c, float t) -> float {
    const int u = 63 - c + A;
    return (u & 1) ? add_bf16_f32<true>(w[u >> 1], t) : add_bf16_f32<false>(w[u >> 1], t);
  };
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint64_t t2 = mul_f2(f2u(sr[2 * i], sr[2 * i + 1]), scale2);
    x2[i] = f2(plus_rel(2 * i, f2lo(t2)), plus_rel(2 * i + 1, f2hi(t2)));
  }
}

// x2[i] = the scaled scores plus the sheared bias of columns 2 i and 2 i + 1 of
// one query row, for half `half` (keys 64 half .. 64 half + 63) of a 128-key
// tile whose rel boxes sit at `slot`: row r of the tile, P0 the position of
// the tile's first row.  With no distance of this half below rel_extent, pass
// has_rel = false (no bias).
__device__ __forceinline__ void scores_with_bias_w2(uint64_t (&x2)[32], const uint32_t (&sr)[64],
                                                    const uint8_t* slot, int r, int P0, int half,
                                                    bool has_rel, float scale) {
  const uint64_t scale2 = f2(scale, scale);
  if (!has_rel) {
    const uint64_t zero2 = f2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 32; ++i) x2[i] = fma_f2(f2u(sr[2 * i], sr[2 * i + 1]), scale2, zero2);
    return;
  }
  const int rbox = r / kRelBoxRows, rrow = r % kRelBoxRows;
  // A box starts at distance (P0 + 32 box - j0 - 127) rounded down to 8 (less
  // kRelOddShift for an odd box), so the distance of this half's column 63
  // sits rrow + ((P0 + 1) & 7) + 64 (1 - half) (+ kRelOddShift) into the row.
  const int col = rrow + ((P0 + 1) & 7) + 64 * (1 - half) + kRelOddShift * (rbox & 1);
  const uint2* p2 = reinterpret_cast<const uint2*>(
      reinterpret_cast<const __nv_bfloat16*>(slot + rbox * kRelBoxBytesW) + rrow * kRelColsW +
      (col & ~3));
  switch (col & 3) {  // the same for the warp
    case 0: rel_fma16_x2<0>(x2, sr, p2, scale2); break;
    case 1: rel_fma16_x2<1>(x2, sr, p2, scale2); break;
    case 2: rel_fma16_x2<2>(x2, sr, p2, scale2); break;
    default: rel_fma16_x2<3>(x2, sr, p2, scale2); break;
  }
}

}  // namespace prefill
}  // namespace relattn
