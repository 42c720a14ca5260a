// Paged split-KV decode for relative-bias GQA attention (sm_103a).
//
// One persistent kernel does the whole decode call:
//  * the window-aware walk: each sequence contributes the 64-key tiles that
//    hold a visible key (at most ceil(W/128)+1 blocks on a local layer --
//    "Inkling-Small on Gaudi 2", section "Decode window");
//  * the work split ("vLLM TML Inkling Support", section "Low-Latency
//    Collectives and Kernels": num_splits chosen from batch size and KV
//    length): the tiles of all (sequence, KV head) segments are laid end to
//    end and cut into gridDim.x equal contiguous ranges, one per CTA.  When
//    no segment is much longer than a CTA's share, the cuts snap to segment
//    boundaries so that no segment is split (no partials, no combine);
//    otherwise segments are cut exactly where the ranges end;
//  * the split kernel: a producer warp streams each piece's query rows, and
//    K, V and the rel slice of every tile, with TMA into shared memory; two
//    groups of four consumer warps take alternate tiles, each warp 16 keys
//    of a tile, with all g query heads of the KV head packed as the 16 rows
//    of an mma.sync tile ("Inkling 2 Small on vLLM", section "vLLM
//    integration and optimisation": the heads of one KV group packed into
//    one tile, KV read once); the bias comes from the stage's rel slice and
//    feeds an online softmax;
//  * multi-token decode (speculative verification: k query tokens per
//    sequence -- "vLLM TML Inkling Support", section "TML Inkling Model
//    Architecture": up to 9 tokens per step): the k tokens are cut into
//    chunks of kpc = min(k, 16 / g), and each chunk's kpc x g (token, head)
//    rows share one tile and one read of their keys.  A chunk is a "virtual
//    sequence": the walk, the split and the combine run over chunks exactly
//    as over sequences for k = 1;
//  * the split-combine: a segment cut by a range boundary leaves one partial
//    (normalised output, base-2 log-sum-exp) per piece in the workspace; the
//    CTA that finishes the segment last (counted with an acq_rel atomic)
//    merges them in a fixed order.
#include <cuda_fp16.h>

#include <type_traits>

#include "relattn_common.cuh"
#include "relattn_internal.h"

namespace relattn {

namespace {

constexpr int kConsumerWarps = 8;  // two groups of four
constexpr int kDecodeThreads = 32 * (1 + kConsumerWarps);
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kWholeSlackTiles = 4;  // tolerated imbalance to avoid a split
constexpr int kQBufBytes = 4096;     // 16 rows x 256 B as two swizzled halves (32 rows: twice)
constexpr int kMiscAbort = 14;       // shared flag word: a consumer warp gave up waiting
// e4m3 cache, f16 query fragments.  One-token kernel: per consumer warp,
// its lanes' B fragments of Q^T for the eight k-steps of d_qk = 128 (8 x 32
// lanes x 8 bytes).  General kernel: one copy for all warps, the lanes' A
// fragments of Q (8 k-steps x 32 lanes x 16 bytes).
constexpr int kPrivQ = 8 * 32 * 8;
constexpr int kPrivQA = 8 * 32 * 16;

constexpr int kSlicePad = 8;         // floats of padding per merge-slice row, at most
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();

// 1 / normaliser of query row qi, whose softmax so far has maximum M (base 2)
// and sum Ls: the optional sink logit joins the normaliser, and the optional
// gate's sigmoid scales the output.
__device__ __forceinline__ float out_scale(const DecodeParams& p, size_t qi, float M, float Ls) {
  float den = Ls;
  if (p.sink) den += ex2(__ldg(p.sink + qi) * kLog2e - M);  // 0 for a sink of -inf
  float s = den > 0.f ? p.v_scale / den : 0.f;               // 0 when den overflows
  if (p.gate) s /= 1.f + ex2(-__ldg(p.gate + qi) * kLog2e);
  return s;
}

__device__ __forceinline__ float rel_f32(float x) { return x; }
__device__ __forceinline__ float rel_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

// Bytes of one token's rel box in a stage (g rows x kRelBoxW floats), padded
// so that every box starts 128-byte aligned.
__host__ __device__ constexpr int rel_token_bytes(int g, int es) {
  return (g * rel_box_w(es) * es + 127) & ~127;
}

// Shared-memory carve-up (byte offsets from a 1024-aligned base); identical
// on host and device.  K/V stages are 1024-aligned for the 128-byte swizzle
// (bf16: two 64-column halves per tile; e4m3: one 128-byte row per key); an
// e4m3 cache adds the consumer warps' f16 query fragments; the rel slices of
// the stages (kpc token boxes each) live in a ring of their own;
// per-sequence lengths take B entries, tile counts and prefixes Bv.
struct DecodeSmem {
  int qbuf, qbytes, stages, stage_bytes, priv, rel, rel_bytes, slices, bars, valid, seqlen, nt,
      pref, m, l, misc, total;
  __host__ __device__ DecodeSmem(int nstages, int B, int Bv, int kpc, int g, int dv, int rel_es,
                                 int kv_es) {
    stage_bytes = kTileKeys * (kDqk + dv) * kv_es;
    rel_bytes = kpc * rel_token_bytes(g, rel_es);
    // chunks of up to 32 rows are split between the two consumer groups
    const int rows = kpc * g;
    const int halves = rows > kMaxDecodeRows ? 2 : 1;
    qbuf = 0;
    qbytes = halves * kQBufBytes;
    stages = qbuf + 2 * qbytes;
    priv = stages + nstages * stage_bytes;
    // the general kernel runs when a tile packs several tokens or g > 8
    const bool multi = kpc > 1 || g > 8;
    rel = priv + (kv_es == 1 ? (multi ? halves * kPrivQA : kConsumerWarps * kPrivQ) : 0);
    slices = rel + nstages * rel_bytes;
    const int wrows = rows < kMaxDecodeRows ? rows : kMaxDecodeRows;  // rows of one warp
    bars = (slices + kConsumerWarps * wrows * (dv + kSlicePad) * 4 + 15) & ~15;
    valid = bars + (2 * nstages + 4) * 8;
    seqlen = valid + nstages * 4;
    nt = seqlen + B * 4;
    pref = nt + Bv * 4;
    m = (pref + (Bv + 1) * 4 + 15) & ~15;
    l = m + kConsumerWarps * 16 * 4;
    misc = l + kConsumerWarps * 16 * 4;
    total = misc + 64;
  }
};

// One virtual sequence: chunk ck of the k query tokens of sequence b (for
// k = 1 the sequence itself).  Its tokens sit at positions pf .. pl; its keys
// are those of [lo, pl], lo the first key visible to the first token.
struct VSeq {
  int b, i0, kc;   // sequence, first token of the chunk, tokens in the chunk
  int pf, pl, lo;  // positions of the first and last token; first visible key
  int tile_first;  // lo / 64
  int ntiles;      // 0 if the sequence's length is invalid
};

// The query-token packing: k tokens per sequence, kpc per chunk, nck chunks.
// The kernel is instantiated twice: with MULTI = false (k = 1, one-token
// decode) these are the constants 1 and the chunk arithmetic folds away.
template <bool MULTI>
struct Tok {
  int k, kpc, nck;
  __device__ __forceinline__ explicit Tok(const DecodeParams& p)
      : k(MULTI ? p.k : 1), kpc(MULTI ? p.kpc : 1), nck(MULTI ? p.nck : 1) {}
  // token of tile row r (rows are token * g + head)
  __device__ __forceinline__ int token_of_row(int r, int g) const { return MULTI ? r / g : 0; }
};

template <bool MULTI>
__device__ __forceinline__ VSeq decode_vseq(int vb, int len, const DecodeParams& p) {
  const Tok<MULTI> t(p);
  VSeq v;
  v.b = vb / t.nck;
  v.i0 = (vb - v.b * t.nck) * t.kpc;
  v.kc = min(t.kpc, t.k - v.i0);
  if (len < t.k || len > p.max_blocks * kBlockSize) {
    v.pf = v.pl = v.lo = v.tile_first = v.ntiles = 0;
    return v;
  }
  v.pf = len - t.k + v.i0;
  v.pl = v.pf + v.kc - 1;
  v.lo = window_lo(v.pf, p.window);
  v.tile_first = v.lo / kTileKeys;
  v.ntiles = v.pl / kTileKeys - v.tile_first + 1;
  return v;
}

// The keys of 64-key tile `tile` that the producer brings for chunk sq:
// [first, first + n).  With HALVES (the one-token kernel over a bf16 cache)
// a tile at an edge of the key range [lo, pl] whose first or last 32 keys all
// lie outside it brings only the other 32; otherwise the whole tile.
struct TileKeys {
  int first, n;
};

template <bool HALVES>
__device__ __forceinline__ TileKeys tile_keys(int tile, const VSeq& sq) {
  constexpr int kHalf = kTileKeys / 2;
  const int key0 = tile * kTileKeys;
  const int h0 = HALVES && key0 + kHalf - 1 < sq.lo ? kHalf : 0;  // first 32 not needed
  const bool half = h0 > 0 || (HALVES && key0 + kHalf > sq.pl);  // or the last 32
  return TileKeys{key0 + h0, half ? kHalf : kTileKeys};
}

// How the CTA ranges are cut.  All tile indices fit in 32 bits (the host
// checks batch * kv heads * tiles per sequence < 2^31), so the cut arithmetic
// is 32-bit: no 64-bit division on the kernel's start-up path.
struct Plan {
  int T;        // tiles of all segments
  int G;        // CTAs with work: min(gridDim.x, T), or the segment count when per_cta
  int whole;    // 1: cuts snap to segment boundaries
  int per_cta;  // 1: whole, and no more segments than CTAs: CTA c takes segment c
  int tq, tr;   // T / G and T % G (exact cuts)
};

// The plan from the tile total, the longest segment and the segment count.
// When whole segments balance (the longest is within kWholeSlackTiles of a
// CTA's share) and there are no more segments than CTAs, the best cut is one
// segment per CTA, and CTA c's segment follows from c alone.
__device__ __forceinline__ Plan make_plan(int T, int mx, int nseg) {
  Plan pl;
  const int grid = static_cast<int>(gridDim.x);
  pl.T = T;
  pl.G = min(grid, T);
  pl.whole = pl.G > 0 && static_cast<long long>(mx) * pl.G <=
                             T + static_cast<long long>(kWholeSlackTiles) * pl.G;
  pl.tq = pl.G > 0 ? T / pl.G : 0;
  pl.tr = pl.G > 0 ? T - pl.tq * pl.G : 0;
  pl.per_cta = pl.whole && nseg <= grid;
  if (pl.per_cta) pl.G = nseg;
  return pl;
}

// The piece of a CTA's range that falls in one (sequence, KV head) segment.
struct Piece {
  int b, kvh, i0, n;
  int seg_start, seg_end;
};

__device__ __forceinline__ int seq_of(int f, const int* s_pref, int B, int Hkv) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (Hkv * s_pref[mid] <= f)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ Piece locate_piece(int f, int a1, const int* s_pref, const int* s_nt,
                                              int B, int Hkv) {
  Piece pc;
  pc.b = seq_of(f, s_pref, B, Hkv);
  const int nt = s_nt[pc.b];
  const int off = f - Hkv * s_pref[pc.b];
  pc.kvh = off / nt;
  pc.i0 = off - pc.kvh * nt;
  pc.seg_start = Hkv * s_pref[pc.b] + pc.kvh * nt;
  pc.seg_end = pc.seg_start + nt;
  pc.n = min(a1, pc.seg_end) - f;
  return pc;
}

// Exact cut c of T tiles into G ranges: floor(c*T/G) = c*(T/G) + floor(c*(T%G)/G),
// where c*(T%G) < G*G fits in 32 bits (the host bounds the grid).
__device__ __forceinline__ int exact_cut(int c, const Plan& pl) {
  return c * pl.tq + (c * pl.tr) / pl.G;
}

// CTA owning flat tile f under exact cuts (split-combine only).
__device__ __forceinline__ int cta_of(int f, const Plan& pl) {
  return static_cast<int>((static_cast<long long>(f + 1) * pl.G - 1) / pl.T);
}

// Start of CTA c's range: the exact cut, snapped to the nearer segment
// boundary in whole-segment mode.
__device__ __forceinline__ int range_cut(int c, const Plan& pl, const int* s_pref,
                                         const int* s_nt, int B, int Hkv) {
  if (pl.per_cta) {  // the start of segment c (c < nseg), else the end
    if (c >= pl.G) return pl.T;
    const int b = c / Hkv;
    return Hkv * s_pref[b] + (c - b * Hkv) * s_nt[b];
  }
  int f = exact_cut(c, pl);
  if (pl.whole && f > 0 && f < pl.T) {
    const int b = seq_of(f, s_pref, B, Hkv);
    const int nt = s_nt[b];
    const int base = Hkv * s_pref[b];
    const int s0 = base + (f - base) / nt * nt;
    const int s1 = s0 + nt;
    f = (f - s0 <= s1 - f) ? s0 : s1;
  }
  return f;
}

__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// Issued first thing in the kernel, so that the prologue's only dependent
// global round trip overlaps the set-up: this thread's seq_lens entry, and L2
// prefetches for the segment the CTA most likely owns (segment c: chunk
// c / Hkv, KV head c % Hkv, which holds when every segment fits one CTA) --
// its block-table row, its query rows and the rel rows its window needs.
// A wrong guess costs only the prefetched bytes.
template <bool MULTI>
__device__ __forceinline__ int decode_early_loads(const DecodeParams& p) {
  const Tok<MULTI> t(p);
  const int tid = threadIdx.x;
  const int len = tid < p.B ? __ldg(p.seq_lens + tid) : 0;
  const int vb = blockIdx.x / p.Hkv, kvh = blockIdx.x - (blockIdx.x / p.Hkv) * p.Hkv;
  if (vb < p.Bv && p.rel != nullptr) {
    const int lane = tid & 31;
    const int b = vb / t.nck, i0 = (vb - b * t.nck) * t.kpc;
    const int rows = min(t.kpc, t.k - i0) * p.g;  // (token, head) rows of the chunk
    // query / rel row of chunk row r: token i0 + r / g, head kvh g + r % g
    auto qrow = [&](int r) {
      const int ti = t.token_of_row(r, p.g);
      return (static_cast<size_t>(b) * t.k + i0 + ti) * p.Hq +
             static_cast<size_t>(kvh) * p.g + (r - ti * p.g);
    };
    if (tid >= 32 && tid < 64) {  // block-table row: 32 lines of 128 bytes at most
      if (lane * 32 < p.max_blocks)
        prefetch_l2(p.block_table + static_cast<size_t>(b) * p.max_blocks + lane * 32);
    } else if (tid >= 64 && tid < 96) {  // query rows: 2 lines each
      if (lane < 2 * rows) prefetch_l2(p.q + qrow(lane / 2) * 128 + (lane & 1) * 64);
    } else if (tid >= 96 && tid < 128) {  // rel rows: distances [0, min(E, W or E))
      const int dist = p.window > 0 ? min(p.rel_extent, p.window) : p.rel_extent;
      const int lines = (dist * p.rel_es + 127) / 128;  // 128-byte lines
      const char* rel = static_cast<const char*>(p.rel);
      for (int i = lane; i < rows * lines && i < 4 * 32; i += 32)
        prefetch_l2(rel + (qrow(i / lines) * p.rel_extent) * p.rel_es + (i % lines) * 128);
    }
  }
  return len;
}

// A CTA's range of flat tiles [a0, a1) and the plan it was cut from;
// first: the piece starting at a0 (valid when has_first).
struct CtaRange {
  Plan pl;
  int a0, a1;
  Piece first;
  bool has_first;
};

// Fast prologue for Bv <= 32, run by warp 0 alone (lane v holds chunk v):
// tile counts, their prefix and the cuts come from shuffles and ballots in
// registers, with no block-wide barrier on the way to the first copy.  The
// results are published in shared memory for the other warps.  Same cut
// arithmetic as range_cut.  len0: seq_lens[lane], already loaded.
//
// The plan is known from two warp reductions (tile total, longest segment)
// before the prefix scan; when it gives CTA c segment c, early(b, kvh, len,
// ids) runs right then, with the segment's chunk, KV head, sequence length
// and first block ids, so that the copies it starts overlap the rest of the
// planning.
template <bool MULTI, typename Early>
__device__ CtaRange decode_plan_warp(const DecodeParams& p, uint8_t* smem, const DecodeSmem& L,
                                     int len0, Early&& early) {
  const Tok<MULTI> t(p);
  int* s_len = reinterpret_cast<int*>(smem + L.seqlen);
  int* s_nt = reinterpret_cast<int*>(smem + L.nt);
  int* s_pref = reinterpret_cast<int*>(smem + L.pref);
  int* s_misc = reinterpret_cast<int*>(smem + L.misc);
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int cb = c / p.Hkv;  // chunk of segment c (one segment per CTA)
  const bool has = lane < p.Bv;
  const int len = MULTI ? __shfl_sync(0xffffffffu, len0, min(lane / t.nck, 31))  // my chunk's
                       : len0;                                                 // sequence
  const int nt = has ? decode_vseq<MULTI>(lane, len, p).ntiles : 0;
  if (has && nt == 0 && blockIdx.x == 0) report(p.status, RELATTN_DEV_BAD_LENGTH);
  // Speculatively, the block ids of segment c's first 32 tiles (lane j:
  // block j from the first), loaded while the plan is reduced: they are the
  // ones needed when the plan gives CTA c segment c.  Indices stay inside the
  // chunk's block-table row.  (With more segments than CTAs the plan never
  // gives one per CTA.)
  const int lenc = __shfl_sync(0xffffffffu, len, cb < p.Bv ? cb : 0);
  int ids = 0;
  if (cb < p.Bv && p.Bv * p.Hkv <= static_cast<int>(gridDim.x)) {
    const VSeq sc = decode_vseq<MULTI>(cb, lenc, p);
    if (sc.ntiles > 0) {
      const int blk0 = sc.tile_first >> 1;
      const int nb = ((sc.tile_first + min(32, sc.ntiles) - 1) >> 1) - blk0 + 1;
      if (lane < nb) ids = __ldg(p.block_table + static_cast<size_t>(sc.b) * p.max_blocks + blk0 + lane);
    }
  }
  const int mx = __reduce_max_sync(0xffffffffu, nt);
  const int total = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(nt)));
  CtaRange cr;
  cr.pl = make_plan(p.Hkv * total, mx, p.Bv * p.Hkv);
  const Plan& pl = cr.pl;
  const bool mine = pl.per_cta && c < pl.G;
  if (mine) early(cb, c - cb * p.Hkv, lenc, ids);
  int incl = nt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int excl = incl - nt;
  if (lane < p.B) s_len[lane] = len0;
  if (has) {
    s_nt[lane] = nt;
    s_pref[lane] = excl;
  }
  if (lane == 0) {
    s_pref[p.Bv] = total;
    s_misc[0] = mx;
  }
  auto cut = [&](int c) -> int {  // range_cut, warp-wide
    int f = c * pl.tq + (c * pl.tr) / pl.G;
    if (pl.whole && f > 0 && f < pl.T) {
      // the last sequence whose prefix is <= f
      const unsigned m = __ballot_sync(0xffffffffu, has && p.Hkv * excl <= f);
      const int b = 31 - __clz(m);
      const int ntb = __shfl_sync(0xffffffffu, nt, b);
      const int base = p.Hkv * __shfl_sync(0xffffffffu, excl, b);
      const int s0 = base + (f - base) / ntb * ntb;
      const int s1 = s0 + ntb;
      f = (f - s0 <= s1 - f) ? s0 : s1;
    }
    return f;
  };
  if (pl.per_cta) {
    // segment c: chunk c / Hkv, KV head c % Hkv, all its tiles
    const int b = mine ? cb : 0;
    const int ntb = __shfl_sync(0xffffffffu, nt, b);
    const int base = p.Hkv * __shfl_sync(0xffffffffu, excl, b);
    Piece& pc = cr.first;
    pc.b = b;
    pc.kvh = c - b * p.Hkv;
    pc.i0 = 0;
    pc.n = ntb;
    pc.seg_start = base + pc.kvh * ntb;
    pc.seg_end = pc.seg_start + ntb;
    cr.a0 = mine ? pc.seg_start : 0;
    cr.a1 = mine ? pc.seg_end : 0;
    cr.has_first = cr.a0 < cr.a1;
  } else {
  cr.a0 = c < pl.G ? cut(c) : 0;
  cr.a1 = c < pl.G ? cut(c + 1) : 0;
  // the first piece, as locate_piece(a0, a1) finds it
  cr.has_first = cr.a0 < cr.a1;
  if (cr.has_first) {
    const unsigned m = __ballot_sync(0xffffffffu, has && p.Hkv * excl <= cr.a0);
    Piece& pc = cr.first;
    pc.b = 31 - __clz(m);
    const int ntb = __shfl_sync(0xffffffffu, nt, pc.b);
    const int base = p.Hkv * __shfl_sync(0xffffffffu, excl, pc.b);
    const int off = cr.a0 - base;
    pc.kvh = off / ntb;
    pc.i0 = off - pc.kvh * ntb;
    pc.seg_start = base + pc.kvh * ntb;
    pc.seg_end = pc.seg_start + ntb;
    pc.n = min(cr.a1, pc.seg_end) - cr.a0;
  }
  }
  if (lane == 0) {
    s_misc[2] = pl.T;
    s_misc[3] = pl.G;
    s_misc[4] = pl.whole;
    s_misc[5] = pl.tq;
    s_misc[6] = pl.tr;
    s_misc[7] = cr.a0;
    s_misc[8] = cr.a1;
    s_misc[9] = pl.per_cta;
  }
  __syncwarp();
  return cr;
}

// The other warps' side of decode_plan_warp, once its results are published.
__device__ __forceinline__ CtaRange decode_plan_read(const uint8_t* smem, const DecodeSmem& L) {
  const int* s_misc = reinterpret_cast<const int*>(smem + L.misc);
  CtaRange cr;
  cr.pl.T = s_misc[2];
  cr.pl.G = s_misc[3];
  cr.pl.whole = s_misc[4];
  cr.pl.tq = s_misc[5];
  cr.pl.tr = s_misc[6];
  cr.a0 = s_misc[7];
  cr.a1 = s_misc[8];
  cr.pl.per_cta = s_misc[9];
  return cr;
}

// Sequences with an invalid length get zeros for all their query tokens
// (CTA 0, the given threads; a sequence's chunks share its length, so its
// first chunk tells).
template <bool MULTI>
__device__ __forceinline__ void decode_zero_bad(const DecodeParams& p, const int* s_nt, int t,
                                                int nthreads) {
  if (blockIdx.x != 0 || p.out == nullptr) return;
  const Tok<MULTI> tk(p);
  const int per = tk.k * p.Hq * p.dv * (p.out_f32 ? 4 : 2) / 4;  // 32-bit words
  for (int b = 0; b < p.B; ++b) {
    if (s_nt[b * tk.nck] != 0) continue;
    uint32_t* o = static_cast<uint32_t*>(p.out) + static_cast<size_t>(b) * per;
    for (int i = t; i < per; i += nthreads) o[i] = 0u;
  }
}

// Per-CTA prologue: each sequence's tile count, their exclusive prefix and
// the cut plan.  len0: seq_lens[threadIdx.x], already loaded.
template <bool MULTI>
__device__ Plan decode_prologue(const DecodeParams& p, uint8_t* smem, const DecodeSmem& L,
                                bool zero_bad, int len0) {
  int* s_len = reinterpret_cast<int*>(smem + L.seqlen);
  int* s_nt = reinterpret_cast<int*>(smem + L.nt);
  int* s_pref = reinterpret_cast<int*>(smem + L.pref);
  int* s_misc = reinterpret_cast<int*>(smem + L.misc);
  const int tid = threadIdx.x;
  for (int b = tid; b < p.B; b += blockDim.x) s_len[b] = b == tid ? len0 : p.seq_lens[b];
  __syncthreads();
  for (int vb = tid; vb < p.Bv; vb += blockDim.x) {
    const int nt = decode_vseq<MULTI>(vb, s_len[vb / Tok<MULTI>(p).nck], p).ntiles;
    s_nt[vb] = nt;
    if (nt == 0 && blockIdx.x == 0) report(p.status, RELATTN_DEV_BAD_LENGTH);
  }
  __syncthreads();
  if (tid < 32) {
    const int lane = tid;
    const int chunk = (p.Bv + 31) / 32;
    const int beg = lane * chunk, end = min(p.Bv, beg + chunk);
    int sum = 0, mx = 0;
    for (int i = beg; i < end; ++i) {
      sum += s_nt[i];
      mx = max(mx, s_nt[i]);
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    int run = incl - sum;
    for (int i = beg; i < end; ++i) {
      s_pref[i] = run;
      run += s_nt[i];
    }
    if (lane == 31) {
      s_pref[p.Bv] = incl;
      s_misc[0] = mx;
    }
  }
  __syncthreads();
  if (zero_bad) decode_zero_bad<MULTI>(p, s_nt, tid, blockDim.x);
  return make_plan(p.Hkv * s_pref[p.Bv], s_misc[0], p.Bv * p.Hkv);
}

// The K and V tensor maps of half-tile boxes, a parameter of the one-token
// kernel over a bf16 cache only (the others keep their smaller parameter
// block).
template <bool H>
struct HalfMaps {
  CUtensorMap k, v;
};
template <>
struct HalfMaps<false> {};

// MULTI: the general kernel (several query tokens per tile, or g > 8), else
// the one-token kernel.  R16: rel is bf16 (else fp32).  KV8: the cache is
// e4m3; the consumer warps widen its bytes to f16 in registers and the MMAs
// take f16 operands.  LS: per-token logit factors are given (general kernel
// only: the one-token kernel reads them whenever they are given, at no cost).
// RS (general kernel only): a chunk of up to 32 rows, both consumer groups
// on every tile, group grp taking rows 16 grp .. 16 grp + 15.
template <int DV, bool MULTI, bool R16, bool KV8, bool LS, bool RS>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_rel,
                  const __grid_constant__ HalfMaps<!MULTI && !KV8> hm,
                  const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const int g = p.g;
  const int ns = p.nstages;
  const RingIndex ri(ns);  // stage n -> slot n % ns, phase (n / ns) & 1
  const Tok<MULTI> tok(p);
  using RelT = typename std::conditional<R16, __nv_bfloat16, float>::type;
  constexpr int RES = R16 ? 2 : 4;                // bytes per rel element
  constexpr int RW = R16 ? kRelBoxW16 : kRelBoxW;  // distances per rel box row
  constexpr int RAL = R16 ? ~7 : ~3;               // box start: 16-byte aligned distance
  constexpr int NB = MULTI ? 2 : 1;                // 8-row blocks of a tile's rows
  constexpr int DB = DV / 16;                      // 16-column blocks of d_v
  // merge-slice row padding: conflict-free writes of O^T columns (NB = 1:
  // rows 2 cq apart by 2 (DV + 4) = 8 banks mod 32) or of O rows (NB = 2)
  constexpr int SP = NB == 1 ? 4 : kSlicePad;
  static_assert(!KV8 || DV == 128, "e4m3 caches: d_v = 128");
  static_assert(!LS || MULTI, "logit factors: a template case of the general kernel only");
  static_assert(!RS || MULTI, "row split: the general kernel only");
  constexpr int QH = RS ? 2 * 2048 : 2048;  // bytes of one 64-column half of a query buffer
  constexpr int QB = 2 * QH;                // bytes of a query buffer (DecodeSmem::qbytes)
  const DecodeSmem L(ns, p.B, p.Bv, tok.kpc, g, DV, RES, KV8 ? 1 : 2);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + ns;
  uint64_t* qfull = empty + ns;
  uint64_t* qempty = qfull + 2;
  int* s_valid = reinterpret_cast<int*>(smem + L.valid);
  const int* s_len = reinterpret_cast<const int*>(smem + L.seqlen);
  const int* s_nt = reinterpret_cast<const int*>(smem + L.nt);
  const int* s_pref = reinterpret_cast<const int*>(smem + L.pref);
  int* s_misc = reinterpret_cast<int*>(smem + L.misc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The next kernel on the stream may start launching now; it waits for this
  // one to finish before it touches global memory, as this one does below.
  grid_dep_launch_dependents();

  // Barriers full[ns], empty[ns], qfull[2], qempty[2], one per lane of
  // warp 0, so that their set-up costs the producer one step.
  if (warp == 0) {
    if (lane < 2 * ns + 4)
      mbar_init(&full[lane], lane < ns ? 1
                             : lane < 2 * ns ? (RS ? kConsumerWarps : kConsumerWarps / 2)
                             : lane < 2 * ns + 2 ? 1 : kConsumerWarps);
    fence_mbar_init();
    if (lane == 0) {
      s_misc[kMiscAbort] = 0;
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_rel);
      if constexpr (!MULTI && !KV8) {  // the half-tile boxes (see issue_tile)
        tma_prefetch_desc(&hm.k);
        tma_prefetch_desc(&hm.v);
      }
    }
    __syncwarp();
  }
  // Everything above touches only shared memory and the kernel parameters;
  // every global access comes after the kernels before this one are done.
  grid_dep_wait();
  const int len0 = decode_early_loads<MULTI>(p);
  // Query rows past a chunk's kc * g are never written or cleared: the MMA
  // rows, the softmax rows and the merge rows are independent, and those
  // rows' results are dropped, whatever the bits there.
  const int q_tx = 2 * tok.kpc * g * 64 * 2;  // kpc tokens x g heads, two halves
  // The query rows of chunk sq, KV head kvh into buffer qb (one lane):
  // rows token * g + head, tokens i0 .. i0 + kpc - 1 (rows past its kc
  // tokens are read but never used).  False on a wait timeout.
  auto issue_q = [&](int qb, int kvh, const VSeq& sq, int parity) -> bool {
    if (!mbar_wait(&qempty[qb], parity)) {
      report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
      return false;
    }
    uint8_t* qs = smem + L.qbuf + qb * QB;
    mbar_arrive_expect_tx(&qfull[qb], q_tx);
    if constexpr (MULTI) {
      tma_load_3d(qs, &tm_q, &qfull[qb], 0, kvh * g, sq.b * tok.k + sq.i0);
      tma_load_3d(qs + QH, &tm_q, &qfull[qb], 64, kvh * g, sq.b * tok.k + sq.i0);
    } else {  // q [B * Hq][128]: the g rows of the group
      tma_load_2d(qs, &tm_q, &qfull[qb], 0, sq.b * p.Hq + kvh * g);
      tma_load_2d(qs + QH, &tm_q, &qfull[qb], 64, sq.b * p.Hq + kvh * g);
    }
    return true;
  };
  const int stage_tx = kTileKeys * (kDqk + DV) * (KV8 ? 1 : 2);
  const int rel_tx = g * RW * RES;                 // one token's rel box
  const int rel_stride = rel_token_bytes(g, RES);  // its place in a stage's rel slice
  // K, V and rel of tile `tile` of chunk sq, KV head kvh, into the stage of
  // CTA tile nn (one lane per tile); 1 on a wait timeout.  One-token kernel
  // over a bf16 cache: a tile at an edge of the key range [lo, p] whose first
  // or last 32 keys all lie outside it brings only the other 32, and the
  // consumer warps of the 32 left out skip the tile (their rows in the stage
  // are never read).  (In the general kernel, at the register cap, and over
  // an e4m3 cache, whose tiles all fit in flight at once, the tests cost more
  // than the bytes saved.)
  auto issue_tile = [&](int nn, int tile, int id, const VSeq& sq, int kvh) -> int {
    const int stage = ri.slot(nn);
    if (!mbar_wait(&empty[stage], ri.phase(nn) ^ 1)) {
      report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
      return 1;
    }
    const bool ok = id >= 0 && id < p.num_blocks;
    s_valid[stage] = ok ? 1 : 0;
    if (ok) {
      const int key0 = tile * kTileKeys;
      // token i's rel box: its g rows from distance dmin_i rounded down to
      // 16 bytes, where dmin_i = (pf + i) - key0 - 63; tokens whose every
      // distance here is past rel_extent need none
      const int dmin0 = sq.pf - key0 - (kTileKeys - 1);
      const int nrel = max(0, min(sq.kc, p.rel_extent - dmin0));
      constexpr bool kHalves = !MULTI && !KV8;
      const TileKeys tk = tile_keys<kHalves>(tile, sq);
      const int h0 = tk.first - key0;
      const bool half = tk.n < kTileKeys;
      mbar_arrive_expect_tx(&full[stage], (half ? stage_tx / 2 : stage_tx) + nrel * rel_tx);
      uint8_t* st = smem + L.stages + stage * L.stage_bytes;
      const int row = id * kBlockSize + (tile & 1) * kTileKeys;
      constexpr int kVOff = KV8 ? kTileKeys * kDqk : 16384;  // V's place in a stage
      if constexpr (KV8) {  // head-major rows: 64 rows x 128 bytes, one box each
        const int hrow = (id * p.Hkv + kvh) * kBlockSize + (tile & 1) * kTileKeys;
        tma_load_2d(st, &tm_k, &full[stage], 0, hrow);
        tma_load_2d(st + kVOff, &tm_v, &full[stage], 0, hrow);
      } else if (!half) {
        tma_load_4d(st, &tm_k, &full[stage], 0, row, 0, kvh);
        tma_load_4d(st + kVOff, &tm_v, &full[stage], 0, row, 0, kvh);
      } else if constexpr (kHalves) {  // one box per 64-column half (8 KB apart)
        tma_load_4d(st + h0 * 128, &hm.k, &full[stage], 0, row + h0, 0, kvh);
        tma_load_4d(st + 8192 + h0 * 128, &hm.k, &full[stage], 0, row + h0, 1, kvh);
#pragma unroll
        for (int hh = 0; hh < DV / 64; ++hh)
          tma_load_4d(st + kVOff + hh * 8192 + h0 * 128, &hm.v, &full[stage], 0, row + h0, hh,
                      kvh);
      }
      for (int i = 0; i < nrel; ++i)
        tma_load_2d(smem + L.rel + stage * L.rel_bytes + i * rel_stride, &tm_rel, &full[stage],
                    (dmin0 + i) & RAL, (sq.b * tok.k + sq.i0 + i) * p.Hq + kvh * g);
    } else {
      report(p.status, RELATTN_DEV_BAD_BLOCK_ID);
      mbar_arrive(&full[stage]);
    }
    return 0;
  };
  // With one segment per CTA the producer knows its first piece as soon as
  // the plan is: it starts the query copy, loads the block ids and sends the
  // first batch of tiles (tile 0 first, so that its data leads) then.
  bool early_q = false;  // warp 0: first piece's query copy and first batch issued
  int early_id = 0;      // warp 0, lane j: block j of the piece's first 32 tiles
  int early_n = 0;       // tiles of that first batch
  int early_bad = 0;     // a wait in it timed out
  auto early = [&](int vb, int kvh, int len, int ids) {
    const VSeq sq = decode_vseq<MULTI>(vb, len, p);
    if (sq.ntiles == 0) return;
    int ok = 1;
    if (lane == 0) ok = issue_q(0, kvh, sq, 1) ? 1 : 0;
    early_q = __shfl_sync(0xffffffffu, ok, 0) != 0;
    if (!early_q) return;
    const int cn = min(32, sq.ntiles);
    const int blk0 = sq.tile_first >> 1;
    early_id = ids;
    const int bn = min(ns, cn);
    const int tile = sq.tile_first + (lane < bn ? lane : 0);
    const int id = __shfl_sync(0xffffffffu, early_id, (tile >> 1) - blk0);
    int bad = 0;
    if (lane == 0) bad = issue_tile(0, tile, id, sq, kvh);
    if (lane > 0 && lane < bn) bad = issue_tile(lane, tile, id, sq, kvh);
    early_n = bn;
    early_bad = __any_sync(0xffffffffu, bad != 0) ? 1 : 0;
  };
  CtaRange cr;
  if (p.Bv <= 32) {
    // warp 0 plans alone and lets the consumers go with a non-blocking arrive
    if (warp == 0) {
      cr = decode_plan_warp<MULTI>(p, smem, L, len0, early);
      named_barrier_arrive(2, kDecodeThreads);
    } else {
      named_barrier(2, kDecodeThreads);
      cr = decode_plan_read(smem, L);
      decode_zero_bad<MULTI>(p, s_nt, tid - 32, kConsumerThreads);
    }
  } else {
    cr.pl = decode_prologue<MULTI>(p, smem, L, true, len0);
    cr.a0 = range_cut(blockIdx.x, cr.pl, s_pref, s_nt, p.Bv, p.Hkv);
    cr.a1 = range_cut(blockIdx.x + 1, cr.pl, s_pref, s_nt, p.Bv, p.Hkv);
    cr.has_first = false;
  }
  const Plan pl = cr.pl;
  if (static_cast<int>(blockIdx.x) >= pl.G) return;
  const int c = blockIdx.x;
  const int a0 = cr.a0, a1 = cr.a1;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int n = 0;     // CTA tile counter
    int k = 0;     // CTA piece counter
    bool abort = early_bad != 0;
    for (int f = a0; f < a1 && !abort; ++k) {
      const Piece pc = (k == 0 && cr.has_first && warp == 0)
                           ? cr.first
                           : locate_piece(f, a1, s_pref, s_nt, p.Bv, p.Hkv);
      const VSeq sq = decode_vseq<MULTI>(pc.b, s_len[pc.b / tok.nck], p);
      const int* trow = p.block_table + static_cast<size_t>(sq.b) * p.max_blocks;
      const bool pre = k == 0 && early_q;  // first piece: its first batch is out
      int bad = 0;
      if (lane == 0 && !pre) bad = issue_q(k & 1, pc.kvh, sq, ((k >> 1) & 1) ^ 1) ? 0 : 1;
      abort = __shfl_sync(0xffffffffu, bad, 0) != 0;
      bad = 0;
      if (pre) n = early_n;
      for (int c0 = 0; c0 < pc.n && !abort; c0 += 32) {
        const int cn = min(32, pc.n - c0);
        const int tile0 = sq.tile_first + pc.i0 + c0;
        const int blk0 = tile0 >> 1;
        const int nb = ((tile0 + cn - 1) >> 1) - blk0 + 1;
        const int myid = pre && c0 == 0 ? early_id : lane < nb ? __ldg(trow + blk0 + lane) : 0;
        // Batches of at most ns tiles, one per lane: their stages are all
        // different, so each lane waits on its own stage one phase ahead at
        // most, and the copies of a batch go out in one pass of the warp.
        for (int jb = pre && c0 == 0 ? early_n : 0; jb < cn && !abort; jb += ns) {
          const int bn = min(ns, cn - jb);
          const int j = jb + (lane < bn ? lane : 0);
          const int tile = tile0 + j;
          const int id = __shfl_sync(0xffffffffu, myid, (tile >> 1) - blk0);
          if (c0 == 0 && jb == 0) {
            // the piece's first tile goes out alone, so that its data leads
            if (lane == 0) bad |= issue_tile(n, tile, id, sq, pc.kvh);
            if (lane > 0 && lane < bn) bad |= issue_tile(n + lane, tile, id, sq, pc.kvh);
          } else if (lane < bn) {
            bad |= issue_tile(n + lane, tile, id, sq, pc.kvh);
          }
          n += bn;
          abort = __any_sync(0xffffffffu, bad != 0);
        }
      }
      f += pc.n;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cwarp = warp - 1;        // 0..7
  const int cw = cwarp & 3;          // keys 16*cw .. 16*cw+15 of a tile
  // Group grp takes the tiles n with n % 2 == grp.  The stage count is even,
  // so every stage belongs to one group and a group never waits on a stage
  // more than one phase ahead of the phase it last consumed there (the
  // parity waits below would alias otherwise).
  const int grp = cwarp >> 2;
  const int ro = RS ? 16 * grp : 0;  // the group's first row of a chunk
  const int ctid = tid - 32;         // 0..255
  const int r0 = lane >> 2, cq = lane & 3;
  float* s_m = reinterpret_cast<float*>(smem + L.m);
  float* s_l = reinterpret_cast<float*>(smem + L.l);
  float* slices = reinterpret_cast<float*>(smem + L.slices);
  int n_base = 0;
  int k = 0;
  bool abort = false;

  int f = a0;
  for (; f < a1 && !abort; ++k) {
    const Piece pc = locate_piece(f, a1, s_pref, s_nt, p.Bv, p.Hkv);
    const VSeq sq = decode_vseq<MULTI>(pc.b, s_len[pc.b / tok.nck], p);
    const int h0 = pc.kvh * g;
    const int nrows = sq.kc * g;  // valid rows of the tile: token * g + head
    // this thread's rows r0 and r0 + 8: validity, query position, first
    // visible key and the offset of their rel row in a stage's slice
    bool rv[2];
    int rP[2], rlo[2], rrel[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = ro + r0 + 8 * rr;
      const int ti = tok.token_of_row(row, g);
      rv[rr] = row < nrows;
      rP[rr] = sq.pf + ti;
      rlo[rr] = window_lo(rP[rr], p.window);
      rrel[rr] = ti * (rel_stride / RES) + (row - ti * g) * RW;
    }
    const int lo_last = window_lo(sq.pl, p.window);
    // The log-position factor f of a row's token scales both terms of its
    // logits.  One-token kernel (all rows one token): f goes into the two
    // logit constants.  General kernel: the logits x stay unscaled and f
    // enters the softmax, exp2(f (x - m)), with m the running max of x
    // (f > 0), and the row's m is reported as f m.
    float fr[2] = {1.f, 1.f};
    if ((LS || !MULTI) && p.logit_scale != nullptr) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int ti = NB == 1 ? 0 : tok.token_of_row(ro + r0 + 8 * rr, g);
        if (NB == 1 || rv[rr])
          fr[rr] = __ldg(p.logit_scale + static_cast<size_t>(sq.b) * p.k + sq.i0 + ti);
      }
    }
    const float sl2 = p.scale_log2 * fr[0], bl2 = kLog2e * fr[0];  // one-token kernel
    const int qb = k & 1;
    bool qok = mbar_wait(&qfull[qb], (k >> 1) & 1);
    if (p.dbg_give_up == k + 1) qok = false;  // test hook (after the wait: no copy in flight)
    if (!qok) report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
    if constexpr (KV8 && MULTI) {
      // e4m3 cache, general kernel: the MMAs run in f16.  The eight warps
      // write the lanes' A fragments of Q (rows r0 and r0 + 8) for the eight
      // k-steps once per piece, in the order of the dimensions of the K
      // fragments (below), and release the query buffer; thread (s, l) writes
      // k-step s of lane l.  Every warp reaches the barrier, also after a
      // failed wait, and then all leave together.
      if (qok) {
        const int fl = ctid & 31, fs = ctid >> 5;
        const int fr = fl >> 2, ft = fl & 3;
        const int d0 = 64 * (ft >> 1) + 16 * (fs >> 1) + 8 * (ft & 1) + 4 * (fs & 1);
        const uint8_t* qsrc = smem + L.qbuf + qb * QB;
        bool q_range = false;  // a valid row's element did not fit f16
        auto pair = [&](int row, int d) {  // bf16 of dimensions d, d + 1 -> f16
          const uint32_t h = bf16x2_to_f16x2(*reinterpret_cast<const uint32_t*>(
              qsrc + (d >> 6) * QH + sw128(row, (d & 63) >> 3) + (d & 7) * 2));
          if (row < nrows && f16x2_nonfinite(h)) q_range = true;
          return h;
        };
#pragma unroll
        for (int h = 0; h < (RS ? 2 : 1); ++h)  // RS: rows 16 h .. 16 h + 15 for group h
          reinterpret_cast<uint4*>(smem + L.priv + h * kPrivQA)[fs * 32 + fl] =
              make_uint4(pair(16 * h + fr, d0), pair(16 * h + fr + 8, d0),
                         pair(16 * h + fr, d0 + 2), pair(16 * h + fr + 8, d0 + 2));
        if (q_range) report(p.status, RELATTN_DEV_Q_RANGE);
      } else if (lane == 0) {
        s_misc[kMiscAbort] = 1;
      }
      named_barrier(1, kConsumerThreads);
      if (s_misc[kMiscAbort]) qok = false;
      else if (lane == 0) mbar_arrive(&qempty[qb]);
    }
    // A failed query wait does not leave the piece loop here: the warp skips
    // the tiles and meets the other warps at the merge barrier, after which
    // they all see the abort flag and leave together (a warp leaving early
    // would strand the others at that barrier).
    if (!qok) abort = true;
    // the query rows stay in their buffer for the whole piece: each tile
    // reads its A fragments from there, one k-step at a time, rather than
    // holding all 32 registers of them next to the 4 x d_v/8 of O
    const uint32_t qbase = smem_u32(smem + L.qbuf + qb * QB);
    // e4m3 cache: the MMAs run in f16.  The lane's B fragments of Q^T (row
    // r0) for the eight k-steps go to the warp's buffer once per piece, in the
    // order of the dimensions of its K fragments (below), after which the
    // shared query buffer is released.  k-step pair u reads dimensions
    // 64 (cq >> 1) + 16 u + 8 (cq & 1) + 0..7: one 16-byte piece of the row.
    uint2* const qfrag = reinterpret_cast<uint2*>(smem + L.priv + cwarp * kPrivQ);
    if (KV8 && !MULTI && qok) {
      bool q_range = false;  // an element of this lane's row r0 did not fit f16
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 v = *reinterpret_cast<const uint4*>(
            smem + L.qbuf + qb * QB + (cq >> 1) * QH + sw128(r0, 2 * u + (cq & 1)));
        const uint2 a = make_uint2(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y));
        const uint2 b = make_uint2(bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
        q_range |= f16x2_nonfinite(a.x) || f16x2_nonfinite(a.y) || f16x2_nonfinite(b.x) ||
                   f16x2_nonfinite(b.y);
        qfrag[(2 * u) * 32 + lane] = a;
        qfrag[(2 * u + 1) * 32 + lane] = b;
      }
      if (q_range && r0 < nrows) report(p.status, RELATTN_DEV_Q_RANGE);
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[qb]);
    }

    float m_[2] = {kNegInf, kNegInf}, l_[2] = {0.f, 0.f};
    // One-token kernel (at most 8 rows, NB = 1): O^T = V^T P^T, 16 columns
    // of d_v by 8 rows per MMA; o[db] holds d_v columns 16 db + lane/4 (+8)
    // of rows 2 cq (+1): half the MMAs of a 16-row P V and half of O's
    // registers.  General kernel (16 rows): O = P V, o[nd] holds rows r0
    // (+8), columns 8 nd + 2 cq (+1).
    float o[DV / 8 / (2 / NB)][4];
#pragma unroll
    for (int i = 0; i < DV / 8 / (2 / NB); ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    for (int t = RS ? 0 : ((n_base + grp) & 1 ? 1 : 0); t < pc.n && !abort; t += RS ? 1 : 2) {
      const int n = n_base + t;
      const int stage = ri.slot(n);
      const int tile = sq.tile_first + pc.i0 + t;
      const int key0 = tile * kTileKeys;
      if (!mbar_wait(&full[stage], ri.phase(n))) {
        report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
        abort = true;
        break;
      }
      // one-token kernel, bf16 cache: a warp whose 16 keys all lie outside
      // [lo, p] has nothing to add (and its rows may not have been loaded)
      const bool idle =
          !MULTI && !KV8 && (key0 + 16 * cw + 15 < sq.lo || key0 + 16 * cw > sq.pl);
      if (s_valid[stage] && !idle) {
        const uint8_t* st = smem + L.stages + stage * L.stage_bytes;
        const uint32_t kbase = smem_u32(st);
        const uint32_t vbase = kbase + 16384;
        const int mi = lane >> 3;
        // logits in log2 units: (q.k/sqrt(d) + rel) * log2(e).  A row's rel
        // box starts at its smallest distance in the tile, P - key0 - 63,
        // rounded down to 16 bytes.
        const RelT* relt = reinterpret_cast<const RelT*>(smem + L.rel + stage * L.rel_bytes);
        const bool edge = key0 < lo_last || key0 + kTileKeys - 1 > sq.pf;  // any mask?
        if constexpr (NB == 1) {
          // ---- one token, at most 8 rows: S^T = K Q^T (16 keys x 8 rows per
          // MMA), softmax down the columns, P^T moved into the B operand of
          // O^T = V^T P^T.  st[0..1]: keys kb (this thread's key), rows
          // 2 cq (+1); st[2..3]: keys kb + 8.
          float sT[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (KV8) {
            // A fragments straight from the e4m3 rows (128 bytes, 128-byte
            // swizzle), widened exactly in registers.  The dot product does
            // not care about the order of the dimensions, so k-step pair u of
            // this lane covers the 8 dimensions its Q fragments hold: one
            // 8-byte read of each of its key rows r0 and r0 + 8 gives columns
            // (2 cq, +1 | 2 cq + 8, +9) of k-steps 2u and 2u + 1.  Lanes with
            // cq < 2 read 16-byte pieces 0-3 of a row, the others 4-7, so
            // each half-warp meets all 32 banks once.
            const uint8_t* kr = st + (16 * cw + r0) * 128 + (cq & 1) * 8;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int off = ((4 * (cq >> 1) + u) ^ r0) * 16;
              const uint2 k0 = *reinterpret_cast<const uint2*>(kr + off);
              const uint2 k8 = *reinterpret_cast<const uint2*>(kr + 1024 + off);
              uint32_t ka[4], kb[4];
              e4m3x4_to_f16x2x2(k0.x, ka[0], ka[2]);
              e4m3x4_to_f16x2x2(k8.x, ka[1], ka[3]);
              e4m3x4_to_f16x2x2(k0.y, kb[0], kb[2]);
              e4m3x4_to_f16x2x2(k8.y, kb[1], kb[3]);
              const uint2 q0 = qfrag[(2 * u) * 32 + lane], q1 = qfrag[(2 * u + 1) * 32 + lane];
              mma_16816_f16(sT, ka, q0.x, q0.y);
              mma_16816_f16(sT, kb, q1.x, q1.y);
            }
          } else {
            // A = the warp's 16 K rows: matrices (keys 0-7 | 8-15) x
            // (dims 0-7 | 8-15); B = Q^T from rows 0-7 of the query buffer
            const int key = 16 * cw + (mi & 1) * 8 + (lane & 7);
            const int qrow = lane & 7, qhalf = (lane >> 3) & 1;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const int chunk = ks * 2 + (mi >> 1);
              uint32_t ka[4];
              ldsm_x4(kbase + (chunk >> 3) * 8192 + sw128(key, chunk & 7), ka[0], ka[1], ka[2],
                      ka[3]);
              const int qchunk = ks * 2 + qhalf;
              uint32_t qb0, qb1;
              ldsm_x2(qbase + (qchunk >> 3) * QH + sw128(qrow, qchunk & 7), qb0, qb1);
              mma_16816(sT, ka, qb0, qb1);
            }
          }
          // one position for all rows: one rel box, present or not for the
          // tile; this thread's keys are kb and kb + 8, kept when their offset
          // (0 or 8) lies in [mlo, mhi]
          const int kb = key0 + 16 * cw + (lane >> 2);
          const int dmin = sq.pf - key0 - (kTileKeys - 1);
          const bool need_rel = dmin < p.rel_extent;
          const int d0 = dmin & RAL;
          const int mlo = edge ? sq.lo - kb : INT_MIN, mhi = edge ? sq.pf - kb : INT_MAX;
          float x[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = 2 * cq + (i & 1);
            const int e = (i >> 1) * 8;
            float bias = 0.f;
            if (need_rel && row < g) bias = rel_f32(relt[row * RW + (sq.pf - kb - e - d0)]);
            const float v = fmaf(sT[i], sl2, bias * bl2);
            x[i] = (e < mlo || e > mhi) ? kNegInf : v;
          }
          // online softmax of rows 2 cq + j over the warp's 16 keys: the 8
          // lanes with this cq hold them (lane bits 2-4)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(x[j], x[2 + j]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_[j], mx);
            const float m_use = m_new == kNegInf ? 0.f : m_new;
            const float alpha = ex2(m_[j] - m_use);
            m_[j] = m_new;
            x[j] = ex2(x[j] - m_use);
            x[2 + j] = ex2(x[2 + j] - m_use);
            l_[j] = l_[j] * alpha + (x[j] + x[2 + j]);  // this thread's two keys
#pragma unroll
            for (int db = 0; db < DB; ++db) {
              o[db][j] *= alpha;
              o[db][2 + j] *= alpha;
            }
          }
          // P^T as the B operand of O^T = V^T P^T: the transposes of this
          // thread's (keys, rows) pairs are its (rows, keys) fragments
          const uint32_t pb0 = movmatrix_t(KV8 ? pack_f16(x[0], x[1]) : pack_bf16(x[0], x[1]));
          const uint32_t pb1 = movmatrix_t(KV8 ? pack_f16(x[2], x[3]) : pack_bf16(x[2], x[3]));
          // V^T as the A operand: transposed 8x8 loads of V's [key][d_v]
          // rows; matrices (keys 0-7 | 8-15) x (columns 16 db + 0-7 | 8-15)
          if constexpr (KV8) {
            // V^T fragments from the e4m3 rows: a 4-byte read gives 4
            // dimensions of one key; two keys' reads interleaved (byte
            // permutes) give f16 pairs (key 2 cq (+8), key + 1) for each of the
            // 4 dimensions.  The output dimensions are permuted to match:
            // O^T row r0 (+8) of block db is d_v column
            // 32 (db >> 1) + 4 r0 + 2 (db & 1) (+1).  Each 4-byte read of the
            // warp meets all 32 banks once.
            const uint8_t* vr = st + kTileKeys * kDqk + (16 * cw + 2 * cq) * 128 + 4 * (r0 & 3);
#pragma unroll
            for (int j = 0; j < DB / 2; ++j) {
              uint32_t va[2][4];
#pragma unroll
              for (int pk = 0; pk < 2; ++pk) {  // keys 2 cq (+1), then 2 cq + 8 (+1)
                const int c = 2 * j + (r0 >> 2);
                const uint32_t xa = *reinterpret_cast<const uint32_t*>(
                    vr + pk * 1024 + ((c ^ (2 * cq)) << 4));
                const uint32_t xb = *reinterpret_cast<const uint32_t*>(
                    vr + pk * 1024 + 128 + ((c ^ (2 * cq + 1)) << 4));
                e4m3x4_to_f16x2x2(__byte_perm(xa, xb, 0x5140), va[0][2 * pk], va[0][2 * pk + 1]);
                e4m3x4_to_f16x2x2(__byte_perm(xa, xb, 0x7362), va[1][2 * pk], va[1][2 * pk + 1]);
              }
              mma_16816_f16(o[2 * j], va[0], pb0, pb1);
              mma_16816_f16(o[2 * j + 1], va[1], pb0, pb1);
            }
          } else {
            const int vkey = 16 * cw + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
            for (int db = 0; db < DB; ++db) {
              const int chunk = 2 * db + (mi & 1);
              uint32_t va[4];
              ldsm_x4_t(vbase + (chunk >> 3) * 8192 + sw128(vkey, chunk & 7), va[0], va[1], va[2],
                        va[3]);
              mma_16816(o[db], va, pb0, pb1);
            }
          }
        } else {
          // ---- several tokens (or g > 8), 16 rows: S = Q K^T, O = P V
          float s[2][4];
#pragma unroll
          for (int i = 0; i < 4; ++i) s[0][i] = s[1][i] = 0.f;
          if constexpr (KV8) {
            // B fragments of K^T straight from the e4m3 rows, as in the
            // one-token kernel: k-step pair u of this lane covers dimensions
            // 64 (cq >> 1) + 16 u + 8 (cq & 1) + 0..7 of key r0 of each
            // 8-key half; the A fragments of Q were written in that order
            const uint4* qf = reinterpret_cast<const uint4*>(smem + L.priv + (RS ? grp * kPrivQA : 0));
            const uint8_t* kr = st + (16 * cw + r0) * 128 + (cq & 1) * 8;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int off = ((4 * (cq >> 1) + u) ^ r0) * 16;
              const uint2 k0 = *reinterpret_cast<const uint2*>(kr + off);
              const uint2 k8 = *reinterpret_cast<const uint2*>(kr + 1024 + off);
#pragma unroll
              for (int v = 0; v < 2; ++v) {  // k-steps 2u, 2u + 1: bytes 0-3, then 4-7
                const uint4 qa = qf[(2 * u + v) * 32 + lane];
                const uint32_t a[4] = {qa.x, qa.y, qa.z, qa.w};
                uint32_t b[2][2];
                e4m3x4_to_f16x2x2(v ? k0.y : k0.x, b[0][0], b[0][1]);
                e4m3x4_to_f16x2x2(v ? k8.y : k8.x, b[1][0], b[1][1]);
                mma_16816_f16(s[0], a, b[0][0], b[0][1]);
                mma_16816_f16(s[1], a, b[1][0], b[1][1]);
              }
            }
          } else {
            const int key = 16 * cw + (mi >> 1) * 8 + (lane & 7);
            const int qrow = ro + (mi & 1) * 8 + (lane & 7);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const int qchunk = ks * 2 + (mi >> 1);
              uint32_t qa[4];
              ldsm_x4(qbase + (qchunk >> 3) * QH + sw128(qrow, qchunk & 7), qa[0], qa[1],
                      qa[2], qa[3]);
              const int chunk = ks * 2 + (mi & 1);
              uint32_t b0, b1, b2, b3;
              ldsm_x4(kbase + (chunk >> 3) * 8192 + sw128(key, chunk & 7), b0, b1, b2, b3);
              mma_16816(s[0], qa, b0, b1);
              mma_16816(s[1], qa, b2, b3);
            }
          }
          // this thread's keys are kb + e, e in {0, 1, 8, 9}; a row keeps the
          // keys with e in [mlo, mhi] (all of them when no key of the tile is
          // masked) -- compares with immediates and selects, no branches.
          // Per row: its token's box, present when the row's smallest
          // distance in the tile is below rel_extent (the box reads 0 past
          // it), and the box entry of key key0 -- the others at -offset
          const int kb = key0 + 16 * cw + cq * 2;
          float x[2][4];
          bool nr[2];
          const RelT* rb[2];
          int mlo[2], mhi[2];
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int dmin = rP[rr] - key0 - (kTileKeys - 1);
            nr[rr] = rv[rr] && dmin < p.rel_extent;
            rb[rr] = relt + rrel[rr] + (rP[rr] - key0 - (dmin & RAL));
            mlo[rr] = edge ? rlo[rr] - kb : INT_MIN;
            mhi[rr] = edge ? rP[rr] - kb : INT_MAX;
          }
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = i >> 1;
              const int e = nt * 8 + (i & 1);
              const int ko = 16 * cw + cq * 2 + e;
              const float bias = nr[rr] ? rel_f32(rb[rr][-ko]) : 0.f;
              const float v = fmaf(s[nt][i], p.scale_log2, bias * kLog2e);
              x[nt][i] = (e < mlo[rr] || e > mhi[rr]) ? kNegInf : v;
            }
          // online softmax, rows r0 (rr=0) and r0+8 (rr=1)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            float mx = fmaxf(fmaxf(x[0][2 * rr], x[0][2 * rr + 1]),
                             fmaxf(x[1][2 * rr], x[1][2 * rr + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_[rr], mx);
            const float m_use = m_new == kNegInf ? 0.f : m_new;
            const float alpha = ex2((m_[rr] - m_use) * fr[rr]);
            const float nmf = -m_use * fr[rr];
            m_[rr] = m_new;
            float sum = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float pv = ex2(fmaf(x[nt][2 * rr + e], fr[rr], nmf));
                x[nt][2 * rr + e] = pv;
                sum += pv;
              }
            l_[rr] = l_[rr] * alpha + sum;
#pragma unroll
            for (int nd = 0; nd < DV / 8; ++nd) {
              o[nd][2 * rr] *= alpha;
              o[nd][2 * rr + 1] *= alpha;
            }
          }
          uint32_t pa[4];
          if constexpr (KV8) {
            pa[0] = pack_f16(x[0][0], x[0][1]);
            pa[1] = pack_f16(x[0][2], x[0][3]);
            pa[2] = pack_f16(x[1][0], x[1][1]);
            pa[3] = pack_f16(x[1][2], x[1][3]);
            // B fragments of V from the e4m3 rows: two keys' 4-byte reads
            // interleaved give f16 pairs (key 2 cq (+8), key + 1) for 4
            // dimensions, one per n-tile: n-tile nd's column r0 is d_v column
            // 32 (nd >> 2) + 4 r0 + (nd & 3) (undone when the slices are
            // written); as in the one-token kernel every read meets all 32
            // banks once
            const uint8_t* vr = st + kTileKeys * kDqk + (16 * cw + 2 * cq) * 128 + 4 * (r0 & 3);
#pragma unroll
            for (int j = 0; j < DV / 32; ++j) {
              uint32_t vb[4][2];
              const int c = 2 * j + (r0 >> 2);
#pragma unroll
              for (int pk = 0; pk < 2; ++pk) {  // keys 2 cq (+1), then 2 cq + 8 (+1)
                const uint32_t xa = *reinterpret_cast<const uint32_t*>(
                    vr + pk * 1024 + ((c ^ (2 * cq)) << 4));
                const uint32_t xb = *reinterpret_cast<const uint32_t*>(
                    vr + pk * 1024 + 128 + ((c ^ (2 * cq + 1)) << 4));
                e4m3x4_to_f16x2x2(__byte_perm(xa, xb, 0x5140), vb[0][pk], vb[1][pk]);
                e4m3x4_to_f16x2x2(__byte_perm(xa, xb, 0x7362), vb[2][pk], vb[3][pk]);
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) mma_16816_f16(o[4 * j + e], pa, vb[e][0], vb[e][1]);
            }
          } else {
            pa[0] = pack_bf16(x[0][0], x[0][1]);
            pa[1] = pack_bf16(x[0][2], x[0][3]);
            pa[2] = pack_bf16(x[1][0], x[1][1]);
            pa[3] = pack_bf16(x[1][2], x[1][3]);
            const int key = 16 * cw + (mi & 1) * 8 + (lane & 7);
#pragma unroll
            for (int nd = 0; nd < DV / 8; nd += 2) {
              const int chunk = nd + (mi >> 1);
              uint32_t b0, b1, b2, b3;
              ldsm_x4_t(vbase + (chunk >> 3) * 8192 + sw128(key, chunk & 7), b0, b1, b2, b3);
              mma_16816(o[nd], pa, b0, b1);
              mma_16816(o[nd + 1], pa, b2, b3);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    __syncwarp();
    if (!KV8 && lane == 0) mbar_arrive(&qempty[qb]);  // the piece's query rows are done
    // A wait that gave up in any consumer warp ends the piece loop of all
    // eight at the same point: each still reaches the next named barrier,
    // and after it they all see the flag.
    if (abort && lane == 0) s_misc[kMiscAbort] = 1;
    n_base += pc.n;

    // ---- merge the eight consumer warps of this piece
    if constexpr (NB == 1) {
      // rows 2 cq + j: m is the same in the 8 lanes of this cq, l sums over
      // their keys
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        l_[j] += __shfl_xor_sync(0xffffffffu, l_[j], 4);
        l_[j] += __shfl_xor_sync(0xffffffffu, l_[j], 8);
        l_[j] += __shfl_xor_sync(0xffffffffu, l_[j], 16);
        if (lane < 4) {
          s_m[cwarp * 16 + 2 * cq + j] = m_[j];
          s_l[cwarp * 16 + 2 * cq + j] = l_[j];
        }
      }
    } else {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        l_[rr] += __shfl_xor_sync(0xffffffffu, l_[rr], 1);
        l_[rr] += __shfl_xor_sync(0xffffffffu, l_[rr], 2);
        if (cq == 0) {
          s_m[cwarp * 16 + r0 + 8 * rr] = m_[rr] * fr[rr];
          s_l[cwarp * 16 + r0 + 8 * rr] = l_[rr];
        }
      }
    }
    // Each warp leaves its unscaled O rows in its slice; after one barrier
    // the threads that write out weigh the eight slices of their row by
    // exp2(m_w - M) themselves, so no second round of scaling is needed.
    const int srows = RS ? kMaxDecodeRows : tok.kpc * g;  // rows of a warp's merge slice
    if constexpr (NB == 1) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int row = 2 * cq + e;  // this thread's O^T column
        if (row >= nrows) continue;
        if constexpr (KV8) {  // permuted d_v columns: see the e4m3 V^T fragments
          float* sl = slices + (cwarp * srows + row) * (DV + SP) + 4 * r0;
#pragma unroll
          for (int j = 0; j < DB / 2; ++j)
            *reinterpret_cast<float4*>(sl + 32 * j) =
                make_float4(o[2 * j][e], o[2 * j][2 + e], o[2 * j + 1][e], o[2 * j + 1][2 + e]);
          continue;
        }
        float* sl = slices + (cwarp * srows + row) * (DV + SP) + (lane >> 2);
#pragma unroll
        for (int db = 0; db < DB; ++db) {
          sl[16 * db] = o[db][e];
          sl[16 * db + 8] = o[db][2 + e];
        }
      }
    } else {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = r0 + 8 * rr;
        if (!rv[rr]) continue;
        if constexpr (KV8) {  // permuted d_v columns: see the e4m3 V fragments
          float* sl = slices + (cwarp * srows + row) * (DV + SP) + 8 * cq;
#pragma unroll
          for (int j = 0; j < DV / 32; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e)
              *reinterpret_cast<float4*>(sl + 32 * j + 4 * e) =
                  make_float4(o[4 * j][2 * rr + e], o[4 * j + 1][2 * rr + e],
                              o[4 * j + 2][2 * rr + e], o[4 * j + 3][2 * rr + e]);
          continue;
        }
        float* sl = slices + (cwarp * srows + row) * (DV + SP) + cq * 2;
#pragma unroll
        for (int nd = 0; nd < DV / 8; ++nd)
          *reinterpret_cast<float2*>(sl + nd * 8) = make_float2(o[nd][2 * rr], o[nd][2 * rr + 1]);
      }
    }
    named_barrier(1, kConsumerThreads);
    if (s_misc[kMiscAbort]) break;

    const bool whole = pc.i0 == 0 && pc.n == s_nt[pc.b];
    const int slot = 2 * c + (a0 < pc.seg_start ? 1 : 0);
    // out row of tile row r: token i0 + r / g of sequence b, head h0 + r % g
    // (out is bf16, or fp32 when p.out_f32: element index, either type)
    // the output row of tile row `row`; its token row / g by a multiply and a
    // shift (this runs per element pair of the store)
    auto orow = [&](int row) -> size_t {
      const int ti = MULTI ? static_cast<int>((static_cast<uint32_t>(row) * p.g_mul) >> 16) : 0;
      return ((static_cast<size_t>(sq.b) * tok.k + sq.i0 + ti) * p.Hq + h0 + (row - ti * g)) * DV;
    };
    for (int idx = ctid; idx < nrows * DV / 2; idx += kConsumerThreads) {
      const int row = idx / (DV / 2), col = 2 * (idx % (DV / 2));
      // the row's (m, l) of every warp that holds it (RS: the four warps of
      // its group, at its row within the group), loaded together, combined
      constexpr int NW = RS ? kConsumerWarps / 2 : kConsumerWarps;
      const int w0 = RS ? NW * (row / kMaxDecodeRows) : 0;
      const int lr = RS ? row % kMaxDecodeRows : row;
      float mw[NW], lw[NW];
      float2 vw[NW];
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        mw[w] = s_m[(w0 + w) * 16 + lr];
        lw[w] = s_l[(w0 + w) * 16 + lr];
        vw[w] = *reinterpret_cast<const float2*>(slices + ((w0 + w) * srows + lr) * (DV + SP) +
                                                 col);
      }
      float M = mw[0];
#pragma unroll
      for (int w = 1; w < NW; ++w) M = fmaxf(M, mw[w]);
      float Ls = 0.f, v0 = 0.f, v1 = 0.f;
      if (M != kNegInf) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float wt = ex2(mw[w] - M);
          Ls += lw[w] * wt;
          v0 += vw[w].x * wt;
          v1 += vw[w].y * wt;
        }
      }
      if (whole) {
        const float inv = out_scale(p, orow(row) / DV, M, Ls);
        if (p.out_f32)
          *reinterpret_cast<float2*>(static_cast<float*>(p.out) + orow(row) + col) =
              make_float2(v0 * inv, v1 * inv);
        else
          *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + orow(row) +
                                             col) = __floats2bfloat162_rn(v0 * inv, v1 * inv);
      } else {  // a partial: normalised over its own keys, no sink or gate yet
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        *reinterpret_cast<float2*>(
            p.part_o + (static_cast<size_t>(slot) * kMaxChunkRows + row) * DV + col) =
            make_float2(v0 * inv, v1 * inv);
        if (col == 0)
          p.part_lse[slot * kMaxChunkRows + row] = Ls > 0.f ? M + lg2(Ls) : kNegInf;
      }
    }
    if (!whole) {
      const int c1 = cta_of(pc.seg_start, pl);
      const int c2 = cta_of(pc.seg_end - 1, pl);
      named_barrier(1, kConsumerThreads);
      if (ctid == 0) {
        const int old = atom_add_acq_rel(&p.counters[pc.b * p.Hkv + pc.kvh], 1);
        s_misc[1] = (old == c2 - c1) ? 1 : 0;
      }
      named_barrier(1, kConsumerThreads);
      if (s_misc[1]) {
        // last piece of this segment to finish: merge all pieces in order
        const int slot1 = 2 * c1 + (exact_cut(c1, pl) < pc.seg_start ? 1 : 0);
        for (int idx = ctid; idx < nrows * DV; idx += kConsumerThreads) {
          const int row = idx / DV, col = idx % DV;
          float M = kNegInf, num = 0.f, den = 0.f;
#pragma unroll 4
          for (int cc = c1; cc <= c2; ++cc) {
            const int sl = cc == c1 ? slot1 : 2 * cc;
            const float lse = __ldcg(p.part_lse + sl * kMaxChunkRows + row);
            const float ov =
                __ldcg(p.part_o + (static_cast<size_t>(sl) * kMaxChunkRows + row) * DV + col);
            if (lse == kNegInf) continue;
            const float M2 = fmaxf(M, lse);
            const float sc = ex2(M - M2);  // 0 while M is -inf
            const float w = ex2(lse - M2);
            num = num * sc + w * ov;
            den = den * sc + w;
            M = M2;
          }
          const float r = num * out_scale(p, orow(row) / DV, M, den);
          if (p.out_f32)
            static_cast<float*>(p.out)[orow(row) + col] = r;
          else
            static_cast<__nv_bfloat16*>(p.out)[orow(row) + col] = __float2bfloat16(r);
        }
        if (ctid == 0) p.counters[pc.b * p.Hkv + pc.kvh] = 0;
      }
    }
    f += pc.n;
  }
  // After a wait gave up (the loop left at the piece starting at f), every
  // split segment that the rest of this CTA's range touches still gets this
  // CTA's partial -- an empty one (lse = -inf, weight 0) -- and its arrival,
  // so each segment's counter completes and returns to zero and the
  // workspace stays ready for the next call.  A segment whose last arrival
  // is this one is left unmerged (the status word reports the timeout).
  for (; f < a1;) {
    const Piece pc = locate_piece(f, a1, s_pref, s_nt, p.Bv, p.Hkv);
    if (!(pc.i0 == 0 && pc.n == s_nt[pc.b])) {
      const int slot = 2 * c + (a0 < pc.seg_start ? 1 : 0);
      if (ctid < kMaxChunkRows) p.part_lse[slot * kMaxChunkRows + ctid] = kNegInf;
      named_barrier(1, kConsumerThreads);
      if (ctid == 0) {
        const int c1 = cta_of(pc.seg_start, pl), c2 = cta_of(pc.seg_end - 1, pl);
        int* cnt = &p.counters[pc.b * p.Hkv + pc.kvh];
        if (atom_add_acq_rel(cnt, 1) == c2 - c1) *cnt = 0;
      }
    }
    f += pc.n;
  }
}

// Replays the producer's walk and split without touching K/V, with the same
// device functions and grid as decode_kernel (MULTI: the general kernel's
// chunks of query tokens; HALVES: the one-token bf16 kernel's half tiles).
// Each tile appends { cta, sequence, kv_head, key_tile, logical_block,
// physical_block }, or with p.dbg_wide { cta, sequence, first_token_of_chunk,
// kv_head, key_tile, physical_block, first_key, keys }.
template <bool MULTI, bool HALVES>
__global__ void __launch_bounds__(128) decode_walk_kernel(const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const Tok<MULTI> tok(p);
  const DecodeSmem L(0, p.B, p.Bv, 1, 1, 64, 4, 2);
  const int* s_len = reinterpret_cast<const int*>(smem + L.seqlen);
  const int* s_nt = reinterpret_cast<const int*>(smem + L.nt);
  const int* s_pref = reinterpret_cast<const int*>(smem + L.pref);
  const int len0 = decode_early_loads<MULTI>(p);
  CtaRange cr;
  if (p.Bv <= 32) {  // the decode kernel's fast prologue, run the same way
    if (threadIdx.x >= 32) return;
    cr = decode_plan_warp<MULTI>(p, smem, L, len0, [](int, int, int, int) {});
  } else {
    cr.pl = decode_prologue<MULTI>(p, smem, L, false, len0);
    cr.a0 = range_cut(blockIdx.x, cr.pl, s_pref, s_nt, p.Bv, p.Hkv);
    cr.a1 = range_cut(blockIdx.x + 1, cr.pl, s_pref, s_nt, p.Bv, p.Hkv);
  }
  const Plan pl = cr.pl;
  if (static_cast<int>(blockIdx.x) >= pl.G || threadIdx.x != 0) return;
  const int c = blockIdx.x;
  const int a0 = cr.a0, a1 = cr.a1;
  for (int f = a0; f < a1;) {
    const Piece pc = locate_piece(f, a1, s_pref, s_nt, p.Bv, p.Hkv);
    const VSeq sq = decode_vseq<MULTI>(pc.b, s_len[pc.b / tok.nck], p);
    const int* trow = p.block_table + static_cast<size_t>(sq.b) * p.max_blocks;
    for (int t = 0; t < pc.n; ++t) {
      const int tile = sq.tile_first + pc.i0 + t;
      const int id = trow[tile >> 1];
      const TileKeys tk = tile_keys<HALVES>(tile, sq);
      const int r = atomicAdd(p.dbg_count, 1);
      if (r < p.dbg_max) {
        if (p.dbg_wide) {
          int32_t* rec = p.dbg_records + 8 * static_cast<size_t>(r);
          rec[0] = c;
          rec[1] = sq.b;
          rec[2] = sq.i0;
          rec[3] = pc.kvh;
          rec[4] = tile;
          rec[5] = id;
          rec[6] = tk.first;
          rec[7] = tk.n;
        } else {
          int32_t* rec = p.dbg_records + 6 * static_cast<size_t>(r);
          rec[0] = c;
          rec[1] = sq.b;
          rec[2] = pc.kvh;
          rec[3] = tile;
          rec[4] = tile >> 1;
          rec[5] = id;
        }
      }
    }
    f += pc.n;
  }
}

}  // namespace

int decode_smem_bytes(int nstages, int B, int Bv, int kpc, int g, int dv, int rel_es, int kv_es) {
  return DecodeSmem(nstages, B, Bv, kpc, g, dv, rel_es, kv_es).total + 1024;
}

template <int DV, bool MULTI, bool R16, bool KV8, bool LS, bool RS>
static cudaError_t launch_decode_rs(const DecodeLaunch& L, int smem, cudaStream_t stream) {
  cudaError_t e = ensure_smem<decode_kernel<DV, MULTI, R16, KV8, LS, RS>>(smem);
  if (e != cudaSuccess) return e;
  // Programmatic stream serialisation: the kernel may begin while the
  // previous kernel on the stream finishes (see grid_dep_wait in the kernel).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  HalfMaps<!MULTI && !KV8> hm;
  if constexpr (!MULTI && !KV8) {
    hm.k = L.tm_kh;
    hm.v = L.tm_vh;
  }
  return cudaLaunchKernelEx(&cfg, decode_kernel<DV, MULTI, R16, KV8, LS, RS>, L.tm_q, L.tm_k,
                            L.tm_v, L.tm_rel, hm, L.p);
}

// The general kernel has a copy for chunks split between the consumer groups.
template <int DV, bool MULTI, bool R16, bool KV8, bool LS = false>
static cudaError_t launch_decode_as(const DecodeLaunch& L, int smem, cudaStream_t stream) {
  if constexpr (MULTI) {
    if (L.p.rs) return launch_decode_rs<DV, MULTI, R16, KV8, LS, true>(L, smem, stream);
  }
  return launch_decode_rs<DV, MULTI, R16, KV8, LS, false>(L, smem, stream);
}

template <int DV, bool MULTI>
static cudaError_t launch_decode_rel(const DecodeLaunch& L, int smem, cudaStream_t stream) {
  // The general kernel has a copy with the logit factors, so that the plain
  // one keeps its registers.
  // (Over an e4m3 cache the general kernel has one copy, which reads the
  // factors whenever they are given: a plain copy measured no fewer spills.)
  const bool ls = MULTI && L.p.logit_scale != nullptr;
  if constexpr (DV == 128) {  // e4m3 caches: d_v = 128
    if (L.p.kv_es == 1)
      return L.p.rel_es == 2 ? launch_decode_as<DV, MULTI, true, true, MULTI>(L, smem, stream)
                             : launch_decode_as<DV, MULTI, false, true, MULTI>(L, smem, stream);
  }
  if (L.p.kv_es != 2) return cudaErrorInvalidValue;  // the host refuses these first
  if constexpr (MULTI) {
    if (ls)
      return L.p.rel_es == 2 ? launch_decode_as<DV, MULTI, true, false, true>(L, smem, stream)
                             : launch_decode_as<DV, MULTI, false, false, true>(L, smem, stream);
  }
  return L.p.rel_es == 2 ? launch_decode_as<DV, MULTI, true, false>(L, smem, stream)
                         : launch_decode_as<DV, MULTI, false, false>(L, smem, stream);
}

cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t stream) {
  const DecodeParams& p = L.p;
  const int smem =
      decode_smem_bytes(p.nstages, p.B, p.Bv, p.kpc, p.g, p.dv, p.rel_es, p.kv_es);
  const bool multi = decode_multi_kernel(p.k, p.g);
  if (p.dv == 128)
    return multi ? launch_decode_rel<128, true>(L, smem, stream)
                 : launch_decode_rel<128, false>(L, smem, stream);
  return multi ? launch_decode_rel<64, true>(L, smem, stream)
               : launch_decode_rel<64, false>(L, smem, stream);
}

cudaError_t launch_decode_walk(const DecodeParams& p, int grid, cudaStream_t stream) {
  const int smem = decode_smem_bytes(0, p.B, p.Bv, 1, 1, 64, 4, 2);
  const bool multi = decode_multi_kernel(p.k, p.g);
  const bool halves = !multi && p.kv_es == 2;
  auto kern = multi ? decode_walk_kernel<true, false>
                    : halves ? decode_walk_kernel<false, true> : decode_walk_kernel<false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace relattn
