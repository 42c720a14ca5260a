// Chunked prefill with a cached prefix for relative-bias GQA attention
// (sm_103a, tcgen05 / TMEM).
//
// Two kernels on the caller's stream:
//  * cache_write scatters each new token's key and value into the paged
//    cache at position ctx_lens[b] + t ("Inkling-Small on Gaudi 2", section
//    "Attention with a relative bias": later chunks and prefix-cache hits
//    prepend the cached context);
//  * prefill_kernel: persistent CTAs take (128-row query tile, query head)
//    work items.  Per item the window-aware walk yields the 64-key tiles of
//    [max(0, P_first - W + 1), P_last]; for each tile
//      S = Q K^T        tcgen05.mma, Q in TMEM, K from TMA (128B swizzle),
//                       S into one of two TMEM buffers
//      bias, masks      one softmax thread per query row adds
//                       rel[row, h, P_row - j] read from a shared-memory box
//                       (the sheared bias: each row reads its own contiguous
//                       distance range; no [Lq, KV] mask is formed), then the
//                       causal and window masks
//      online softmax   the running max only moves when it grows by more
//                       than 2^8, so O is rescaled rarely
//      O += P V         P written back to TMEM as bf16 and used as the A
//                       operand; V from TMA (MN-major, 128B swizzle)
//    ("vLLM TML Inkling Support", section "Low-Latency Collectives and
//    Kernels": the FA4 relative-attention kernel with a sheared bias; "Inkling
//    2 Small on vLLM", section "vLLM integration and optimisation": prefill
//    keeps the sheared-bias path).
//
// Warp roles: 0 = K/V TMA producer, 1 = MMA issuer and TMEM owner, 2-5 =
// softmax (TMEM lane quarters 2, 3, 0, 1), 6 = rel TMA producer.
#include "relattn_common.cuh"
#include "relattn_internal.h"
#include "relattn_prefill.cuh"
#include "relattn_tcgen05.cuh"

namespace relattn {

namespace {

using namespace prefill;

constexpr int kCwTile = 64;                 // cache_write tokens per CTA
constexpr int kPfWarps = 7;  // (an e4m3 cache adds an eighth: the V widener)
constexpr int kKStages = 2, kVStages = 2, kMaxRingStages = 3;
// One ring of shared-memory slots carries, per work item, the query tile,
// then the rel boxes of each key tile, then a scratch slot for storing O.
constexpr int kRingSlotBytes = kRelBoxes * kRelBoxBytes;     // 51200 (50 KB)
static_assert(kRingSlotBytes % 1024 == 0 && kRingSlotBytes >= kQTileBytes, "ring slot");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmQ = 0, kTmS = 64, kTmO = 192;  // S buffer s at kTmS + 64 s
constexpr uint32_t kIdescS = umma_idesc_bf16(128, kTileKeys, 0);

// kRFull / kREmpty: ring slots (producer <-> softmax); kQFull: query tile in
// TMEM (softmax -> MMA).
// kStgK / kStgV: an e4m3 cache's K / V tile in its staging slot (TMA -> the
// warp that widens it into the K / V stage).
enum Bar { kKFull = 0, kKEmpty = 2, kVFull = 4, kVEmpty = 6, kRFull = 8, kREmpty = 11,
           kSFull = 14, kPFull = 16, kOFull = 18, kQFull = 19, kDrain = 20, kStgK = 21,
           kStgV = 23, kNumBars = 25 };
constexpr int kStgBytes = kTileKeys * (kDqk + 128);  // one e4m3 tile: K then V, 16 KB

// Four floats -> four e4m3 codes (low byte first): x / scale rounded to
// nearest even, saturated to +-448 (cvt's satfinite).
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d, float scale) {
  unsigned short lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
      : "=h"(lo)
      : "f"(__fdiv_rn(b, scale)), "f"(__fdiv_rn(a, scale)));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
      : "=h"(hi)
      : "f"(__fdiv_rn(d, scale)), "f"(__fdiv_rn(c, scale)));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Eight bf16 (one uint4) -> eight e4m3 codes (one uint2).
__device__ __forceinline__ uint2 e4m3x8(uint4 x, float scale) {
  auto f = [](uint32_t w, int hi) { return __uint_as_float(hi ? (w & 0xffff0000u) : (w << 16)); };
  return make_uint2(e4m3x4(f(x.x, 0), f(x.x, 1), f(x.y, 0), f(x.y, 1), scale),
                    e4m3x4(f(x.z, 0), f(x.z, 1), f(x.w, 0), f(x.w, 1), scale));
}

// KV8: the cache is e4m3, head-major [NB][Hkv][128][128], and each value is
// quantised with its tensor's scale; a 16-byte piece of the cache holds 16
// codes from 16 bf16 values.  Otherwise a bf16 cache, [NB][128][Hkv][d], where
// a token's Hkv key (or value) rows are contiguous both in k (v) and in its
// cache slot, so they copy as one run of 16-byte pieces.
// One warp per token: its pieces go out lane by lane (coalesced), with no
// division on the way (a division by a run-time value per 16 bytes made the
// copy instruction-bound).
template <bool KV8>
__global__ void __launch_bounds__(256) cache_write_kernel(const PrefillParams p) {
  const int b = blockIdx.y;
  const int r0 = p.cu_seqlens[b];
  const int r1 = p.cu_seqlens[b + 1];
  const int n = r1 - r0;
  const int ctx = p.ctx_lens[b];
  const int t0 = blockIdx.x * kCwTile;
  if (!rows_ok(r0, r1, p.T) || !seq_ok(ctx, n, p.max_blocks)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(p.status, RELATTN_DEV_BAD_LENGTH);
    return;
  }
  if (t0 >= n) return;
  const int nt = min(kCwTile, n - t0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = 256 / 32;
  // 16-byte pieces of one token's keys and values (all KV heads)
  const int kpieces = p.Hkv * (KV8 ? kDqk / 16 : kDqk / 8);
  const int vpieces = p.Hkv * (KV8 ? p.dv / 16 : p.dv / 8);
  const int* trow = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  for (int tt = warp; tt < nt; tt += kWarps) {
    const int pos = ctx + t0 + tt;
    const int phys = __ldg(trow + pos / kBlockSize);
    if (phys < 0 || phys >= p.num_blocks) {  // the same for the whole warp
      if (lane == 0) report(p.status, RELATTN_DEV_BAD_BLOCK_ID);
      continue;
    }
    const size_t row = static_cast<size_t>(r0 + t0 + tt);
    const int in_blk = pos % kBlockSize;
    if constexpr (KV8) {
      // piece c of a token's keys: head c / 8, codes 16 (c % 8) .. of its row
      // (d = 128: 8 pieces per head row), at row (phys * Hkv + head) * 128 +
      // pos % 128 of the head-major cache
#pragma unroll 1
      for (int c = lane; c < kpieces + vpieces; c += 32) {
        const bool isk = c < kpieces;
        const int cc = isk ? c : c - kpieces;
        const int hh = cc >> 3, ch = cc & 7;
        const uint4* src = reinterpret_cast<const uint4*>(
            (isk ? p.k : p.v) + (row * p.Hkv + hh) * kDqk);
        const float sc = isk ? p.k_scale : p.v_scale;
        const uint2 lo = e4m3x8(__ldg(src + 2 * ch), sc), hi = e4m3x8(__ldg(src + 2 * ch + 1), sc);
        const size_t hrow = (static_cast<size_t>(phys) * p.Hkv + hh) * kBlockSize + in_blk;
        uint8_t* dst = reinterpret_cast<uint8_t*>(isk ? p.k_cache : p.v_cache) + hrow * kDqk;
        reinterpret_cast<uint4*>(dst)[ch] = make_uint4(lo.x, lo.y, hi.x, hi.y);
      }
    } else {
      const size_t slot = static_cast<size_t>(phys) * kBlockSize + in_blk;
      const uint4* ks = reinterpret_cast<const uint4*>(p.k + row * p.Hkv * kDqk);
      uint4* kd = reinterpret_cast<uint4*>(p.k_cache + slot * p.Hkv * kDqk);
#pragma unroll 4
      for (int c = lane; c < kpieces; c += 32) kd[c] = __ldg(ks + c);
      const uint4* vs = reinterpret_cast<const uint4*>(p.v + row * p.Hkv * p.dv);
      uint4* vd = reinterpret_cast<uint4*>(p.v_cache + slot * p.Hkv * p.dv);
#pragma unroll 4
      for (int c = lane; c < vpieces; c += 32) vd[c] = __ldg(vs + c);
    }
  }
}

// Shared-memory carve-up (byte offsets from a 1024-aligned base).  An e4m3
// cache adds two staging slots for its tiles.
struct PrefillSmem {
  int k, v, vstage, ring, stg, bars, misc, cu0, nrows, ctx, qpref, total;
  __host__ __device__ PrefillSmem(int B, int dv, int ring_stages, int kv_es) {
    vstage = kTileKeys * dv * 2;
    k = 0;
    v = k + kKStages * kKStageBytes;
    ring = v + kVStages * vstage;  // 1024-aligned: query tiles land 128B-swizzled
    stg = ring + ring_stages * kRingSlotBytes;
    bars = stg + (kv_es == 1 ? 2 * kStgBytes : 0);
    misc = bars + kNumBars * 8;
    cu0 = misc + 16;
    nrows = cu0 + B * 4;
    ctx = nrows + B * 4;
    qpref = ctx + B * 4;
    total = qpref + (B + 1) * 4;
  }
};

struct PItem {
  int b, h, kvh, r0, rows, P0, tf, ntiles;
};

// Work item idx: query tile idx / Hq, head idx % Hq (the heads of one query
// tile run on neighbouring CTAs, so its K/V tiles are shared in L2).
__device__ __forceinline__ void prefill_item(int idx, const PrefillParams& p, const SeqArrays& a,
                                             PItem& it) {
  const int qtg = idx / p.Hq;
  it.h = idx - qtg * p.Hq;
  it.kvh = it.h / p.g;
  const QTile t = query_tile(qtg, p, a);
  it.b = t.b;
  it.r0 = t.r0;
  it.rows = t.rows;
  it.P0 = t.P0;
  it.tf = t.tf;
  it.ntiles = t.ntiles;
}

__device__ __forceinline__ SeqArrays seq_arrays(uint8_t* smem, const PrefillSmem& L) {
  return SeqArrays{reinterpret_cast<int*>(smem + L.cu0), reinterpret_cast<int*>(smem + L.nrows),
                   reinterpret_cast<int*>(smem + L.ctx), reinterpret_cast<int*>(smem + L.qpref)};
}

// One e4m3 tile (64 rows x 128 bytes, 128-byte swizzle) -> its values as
// f16 in the layout the bf16 copies have (two 64-column halves 8 KB apart,
// rows of 128 bytes, 128-byte swizzle).  Lane l takes 16-byte piece j = l & 7
// of rows l / 8 + 4 t, t = 0..15: all 16 loads first, then the conversions
// and stores (the compiler cannot move a load past a store to shared memory).
__device__ __forceinline__ void widen_tile(const uint8_t* src, uint8_t* dst, int lane) {
  const int j = lane & 7, r0 = lane >> 3;
  const int c = 2 * (j & 3);
  uint4 x[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const int r = r0 + 4 * t;
    x[t] = *reinterpret_cast<const uint4*>(src + r * 128 + ((j ^ (r & 7)) << 4));
  }
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const int r = r0 + 4 * t;
    uint32_t h[8];
    e4m3x4_to_f16x2x2(x[t].x, h[0], h[1]);
    e4m3x4_to_f16x2x2(x[t].y, h[2], h[3]);
    e4m3x4_to_f16x2x2(x[t].z, h[4], h[5]);
    e4m3x4_to_f16x2x2(x[t].w, h[6], h[7]);
    uint8_t* row = dst + (j >> 2) * 8192 + r * 128;
    *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(row + (((c + 1) ^ (r & 7)) << 4)) =
        make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// R16: rel is bf16 (else fp32).  O32: out is fp32 (else bf16).  KV8: the
// cache is e4m3 (d_v = 128): warp 0 widens each K tile to f16 and an eighth
// warp each V tile, and every MMA runs in f16 (Q and P are f16 too).
template <int DV, bool R16, bool O32, bool KV8>
__global__ void __launch_bounds__(32 * (kPfWarps + (KV8 ? 1 : 0)), 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_rel, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  static_assert(!KV8 || DV == 128, "e4m3 caches: d_v = 128");
  const int nrs = p.ring_stages;
  const RingIndex ri(p.ring_stages);  // ring entry -> slot, phase
  const PrefillSmem L(p.B, DV, nrs, KV8 ? 1 : 2);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.misc + 4);
  const SeqArrays sa = seq_arrays(smem, L);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars[kKFull + s], 1);
      mbar_init(&bars[kKEmpty + s], 1);
      mbar_init(&bars[kVFull + s], 1);
      mbar_init(&bars[kVEmpty + s], 1);
      mbar_init(&bars[kSFull + s], 1);
      mbar_init(&bars[kPFull + s], 4);
    }
    for (int s = 0; s < nrs; ++s) {
      mbar_init(&bars[kRFull + s], 1);
      mbar_init(&bars[kREmpty + s], 4);
    }
    mbar_init(&bars[kOFull], 1);
    mbar_init(&bars[kQFull], 4);
    mbar_init(&bars[kDrain], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kStgK + s], 1);
      mbar_init(&bars[kStgV + s], 1);
    }
    fence_mbar_init();
    *s_abort = 0;
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_rel);
  }
  // K/V stages start as zeros: a tile whose block id is invalid is never
  // loaded, and its P is zero, so its operands must at least be finite.
  for (int i = tid; i < (L.ring - L.k) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem + L.k)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tc_fence_before();
  }
  const int total = prologue(p, sa, true) * p.Hq;  // contains __syncthreads
  tc_fence_after();
  const uint32_t tbase = *s_tmem;
  const float scale_log2 = p.scale_log2;

  if (KV8 && (warp == 0 || warp == kPfWarps)) {
    // ------------------------- K (warp 0) or V (warp 7) of an e4m3 cache:
    // lane 0 brings tile n into staging slot n & 1 (one 2-D box of 64
    // head-major rows), then the warp widens tile n - 1 into its K or V stage
    // (n - 1) & 1 as f16; the slot tile n lands in was last read when tile
    // n - 2 was widened, before this copy was issued.
    if constexpr (KV8) {
      const bool isv = warp != 0;
      const CUtensorMap* tm = isv ? &tm_v : &tm_k;
      uint64_t* stg_bar = &bars[isv ? kStgV : kStgK];
      uint64_t* full = &bars[isv ? kVFull : kKFull];
      uint64_t* empty = &bars[isv ? kVEmpty : kKEmpty];
      uint8_t* stage0 = smem + (isv ? L.v : L.k);
      const int stage_bytes = isv ? L.vstage : kKStageBytes;
      uint8_t* stg0 = smem + L.stg + (isv ? kTileKeys * kDqk : 0);
      int n = 0;
      bool okp = false;  // tile n - 1 had a valid block id
      auto widen = [&](int m, bool ok) -> bool {
        const int s = m & 1;
        if (!mbar_wait(&empty[s], ((m >> 1) & 1) ^ 1)) return false;
        if (ok) {
          if (!mbar_wait(&stg_bar[s], (m >> 1) & 1)) return false;
          widen_tile(stg0 + s * kStgBytes, stage0 + s * stage_bytes, lane);
          // the MMAs read the stage through the async proxy, and the next
          // copy into this staging slot comes after these reads
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
        return true;
      };
      bool fail = false;
      for (int idx = blockIdx.x; idx < total && !*s_abort && !fail; idx += gridDim.x) {
        PItem it;
        prefill_item(idx, p, sa, it);
        const int* trow = p.block_table + static_cast<size_t>(it.b) * p.max_blocks;
        for (int k = 0; k < it.ntiles; ++k, ++n) {
          const int tile = it.tf + k;
          const int id = __ldg(trow + (tile >> 1));
          const bool ok = id >= 0 && id < p.num_blocks;
          if (lane == 0) {
            if (ok) {
              const int hrow = (id * p.Hkv + it.kvh) * kBlockSize + (tile & 1) * kTileKeys;
              mbar_arrive_expect_tx(&stg_bar[n & 1], kTileKeys * kDqk);
              tma_load_2d(stg0 + (n & 1) * kStgBytes, tm, &stg_bar[n & 1], 0, hrow);
            } else if (!isv) {
              report(p.status, RELATTN_DEV_BAD_BLOCK_ID);
            }
          }
          if (n > 0 && !widen(n - 1, okp)) { fail = true; break; }
          okp = ok;
        }
      }
      if (!fail && n > 0 && !widen(n - 1, okp)) fail = true;
      if (fail && lane == 0) *s_abort = 1;
    }
  } else if (!KV8 && warp == 0 && lane == 0) {
    // ---------------------------------------------------- K/V TMA producer
    int n = 0;
    for (int idx = blockIdx.x; idx < total && !*s_abort; idx += gridDim.x) {
      PItem it;
      prefill_item(idx, p, sa, it);
      const int* trow = p.block_table + static_cast<size_t>(it.b) * p.max_blocks;
      for (int k = 0; k < it.ntiles; ++k, ++n) {
        const int tile = it.tf + k;
        const int id = __ldg(trow + (tile >> 1));
        const bool ok = id >= 0 && id < p.num_blocks;
        const int row = id * kBlockSize + (tile & 1) * kTileKeys;
        const int s = n & 1;
        const uint32_t par = ((n >> 1) & 1) ^ 1;
        if (!mbar_wait(&bars[kKEmpty + s], par)) { *s_abort = 1; break; }
        if (ok) {
          uint8_t* kd = smem + L.k + s * kKStageBytes;
          mbar_arrive_expect_tx(&bars[kKFull + s], kKStageBytes);
          tma_load_3d(kd, &tm_k, &bars[kKFull + s], 0, it.kvh, row);
          tma_load_3d(kd + 8192, &tm_k, &bars[kKFull + s], 64, it.kvh, row);
        } else {
          report(p.status, RELATTN_DEV_BAD_BLOCK_ID);
          mbar_arrive(&bars[kKFull + s]);
        }
        if (!mbar_wait(&bars[kVEmpty + s], par)) { *s_abort = 1; break; }
        if (ok) {
          uint8_t* vd = smem + L.v + s * L.vstage;
          mbar_arrive_expect_tx(&bars[kVFull + s], L.vstage);
          tma_load_3d(vd, &tm_v, &bars[kVFull + s], 0, it.kvh, row);
          if (DV == 128) tma_load_3d(vd + 8192, &tm_v, &bars[kVFull + s], 64, it.kvh, row);
        } else {
          mbar_arrive(&bars[kVFull + s]);
        }
      }
    }
  } else if (warp == 6 && lane == 0) {
    // --------------------------------------------------- ring producer:
    // per item the query tile, the rel boxes of each key tile, and an empty
    // slot the softmax warps use to store O
    int e = 0;
    bool fail = false;
    auto acquire = [&](int entry) -> uint8_t* {
      const int slot = ri.slot(entry);
      if (!mbar_wait(&bars[kREmpty + slot], ri.phase(entry) ^ 1)) return nullptr;
      return smem + L.ring + slot * kRingSlotBytes;
    };
    for (int idx = blockIdx.x; idx < total && !*s_abort && !fail; idx += gridDim.x) {
      PItem it;
      prefill_item(idx, p, sa, it);
      uint8_t* qd = acquire(e);
      if (!qd) { fail = true; break; }
      uint64_t* qbar = &bars[kRFull + ri.slot(e)];
      mbar_arrive_expect_tx(qbar, kQTileBytes);  // rows past T read as zeros
      tma_load_3d(qd, &tm_q, qbar, 0, it.h, it.r0);
      tma_load_3d(qd + kQTileBytes / 2, &tm_q, qbar, 64, it.h, it.r0);
      ++e;
      for (int k = 0; k < it.ntiles; ++k, ++e) {
        const int j0 = (it.tf + k) * kTileKeys;
        uint8_t* rd = acquire(e);
        if (!rd) { fail = true; break; }
        uint64_t* rbar = &bars[kRFull + ri.slot(e)];
        if (it.P0 - j0 - (kTileKeys - 1) < p.rel_extent) {
          constexpr int kBox = R16 ? kRelBoxBytes16 : kRelBoxBytes;
          mbar_arrive_expect_tx(rbar, kRelBoxes * kBox);
          for (int bx = 0; bx < kRelBoxes; ++bx) {
            const int x = (it.P0 + kRelBoxRows * bx - j0 - (kTileKeys - 1)) & (R16 ? ~7 : ~3);
            tma_load_3d(rd + bx * kBox, &tm_rel, rbar, x, it.h, it.r0 + kRelBoxRows * bx);
          }
        } else {
          mbar_arrive(rbar);  // every distance is past rel_extent
        }
      }
      if (fail) break;
      if (!acquire(e)) { fail = true; break; }
      mbar_arrive(&bars[kRFull + ri.slot(e)]);  // the O scratch slot
      ++e;
    }
    if (fail) *s_abort = 1;
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t idesc_pv = KV8 ? umma_idesc_f16(128, DV, 1) : umma_idesc_bf16(128, DV, 1);
    const uint32_t idesc_s = KV8 ? umma_idesc_f16(128, kTileKeys, 0) : kIdescS;
    int n = 0, items = 0;
    auto issue_pv = [&](int m, bool acc) -> bool {
      const int sp = m & 1;
      const uint32_t par = (m >> 1) & 1;
      if (!mbar_wait(&bars[kPFull + sp], par) || !mbar_wait(&bars[kVFull + sp], par)) return false;
      tc_fence_after();
      const uint32_t vb = smem_u32(smem + L.v + sp * L.vstage);
#pragma unroll
      for (int kk = 0; kk < kTileKeys / 16; ++kk)
        umma_tmem_a(tbase + kTmO, tbase + kTmS + 64 * sp + 8 * kk,
                    umma_desc_sw128(vb + kk * 2048, kTileKeys * 128, 1024), idesc_pv,
                    (acc || kk > 0) ? 1 : 0);
      umma_commit(&bars[kOFull]);
      umma_commit(&bars[kVEmpty + sp]);
      return true;
    };
    for (int idx = blockIdx.x; idx < total && !*s_abort; idx += gridDim.x, ++items) {
      PItem it;
      prefill_item(idx, p, sa, it);
      if (!mbar_wait(&bars[kQFull], items & 1)) { *s_abort = 1; break; }
      tc_fence_after();
      bool ok = true;
      for (int k = 0; k < it.ntiles && ok; ++k, ++n) {
        const int s = n & 1;
        if (!mbar_wait(&bars[kKFull + s], (n >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kb = smem_u32(smem + L.k + s * kKStageBytes);
#pragma unroll
        for (int ks = 0; ks < kDqk / 16; ++ks)
          umma_tmem_a(tbase + kTmS + 64 * s, tbase + kTmQ + 8 * ks,
                      umma_desc_sw128(kb + (ks >> 2) * 8192 + (ks & 3) * 32, 0, 1024), idesc_s,
                      ks > 0 ? 1 : 0);
        umma_commit(&bars[kSFull + s]);
        umma_commit(&bars[kKEmpty + s]);
        if (k > 0) ok = issue_pv(n - 1, k > 1);
      }
      if (ok) ok = issue_pv(n - 1, it.ntiles > 1);
      if (!ok) { *s_abort = 1; break; }
    }
    // all MMAs retired before TMEM is released
    umma_commit(&bars[kDrain]);
    if (!mbar_wait(&bars[kDrain], 0)) report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ softmax
    // Thread (q4, lane) owns TMEM lane 32 q4 + lane and puts query row
    // r = 4 lane + q4 there: each warp takes every fourth row, so all its
    // lanes see the same 16-byte alignment of their rows in the rel boxes.
    const int q4 = warp & 3;  // TMEM lane quarter this warp may access
    const int r = 4 * lane + q4;
    const uint32_t tl = tbase + (static_cast<uint32_t>(32 * q4) << 16);
    int n = 0, e = 0, items = 0;  // key tiles and ring entries consumed
    bool fail = false;
    auto slot_wait = [&](int entry) -> uint8_t* {
      const int slot = ri.slot(entry);
      if (!mbar_wait(&bars[kRFull + slot], ri.phase(entry))) return nullptr;
      return smem + L.ring + slot * kRingSlotBytes;
    };
    // This thread's query row, from a ring slot (128-byte swizzled rows) into
    // TMEM, the A operand of S = Q K^T; then the MMA warp may start.  row_valid:
    // the row is one of the item's (an e4m3 cache's f16 query is checked then).
    auto load_q = [&](const uint8_t* qs, int entry, bool row_valid) {
      uint32_t qr[64];
      bool q_range = false;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 v =
              *reinterpret_cast<const uint4*>(qs + c * (kQTileBytes / 2) + sw128(r, j));
          if constexpr (KV8) {  // the f16 MMAs take the query in f16
            qr[(c * 8 + j) * 4] = bf16x2_to_f16x2(v.x);
            qr[(c * 8 + j) * 4 + 1] = bf16x2_to_f16x2(v.y);
            qr[(c * 8 + j) * 4 + 2] = bf16x2_to_f16x2(v.z);
            qr[(c * 8 + j) * 4 + 3] = bf16x2_to_f16x2(v.w);
#pragma unroll
            for (int w = 0; w < 4; ++w) q_range |= f16x2_nonfinite(qr[(c * 8 + j) * 4 + w]);
          } else {
            qr[(c * 8 + j) * 4] = v.x;
            qr[(c * 8 + j) * 4 + 1] = v.y;
            qr[(c * 8 + j) * 4 + 2] = v.z;
            qr[(c * 8 + j) * 4 + 3] = v.w;
          }
        }
      if (KV8 && q_range && row_valid) report(p.status, RELATTN_DEV_Q_RANGE);
      tmem_st32(tl + kTmQ, qr);
      tmem_st32(tl + kTmQ + 32, qr + 32);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kQFull]);
        mbar_arrive(&bars[kREmpty + ri.slot(entry)]);
      }
    };
    for (int idx = blockIdx.x; idx < total && !*s_abort; idx += gridDim.x, ++items) {
      PItem it;
      prefill_item(idx, p, sa, it);
      // A wait that gives up marks the item bad: the warp skips the rest of
      // its work but still meets the other softmax warps at the barrier
      // before the epilogue, after which all four leave together (a warp
      // leaving alone would strand the others at a named barrier).
      bool bad = false;
      if (items == 0) {  // later items' queries are loaded during the previous epilogue
        const uint8_t* qs = slot_wait(e);
        if (!qs) bad = true;
        else load_q(qs, e, r < it.rows);
        ++e;
      }
      const bool row_ok = r < it.rows;
      const int P = it.P0 + r;
      const int* trow = p.block_table + static_cast<size_t>(it.b) * p.max_blocks;

      // Scores in natural-log units: x = q.k / sqrt(d) + rel; exp2 takes
      // log2(e) in its FFMA.  A row's log-position factor f multiplies x:
      // it is folded into that log2(e) (l2f), and the lazy rescale moves the
      // running max of x only past kRescaleNat / f, so f x stays within
      // kRescaleNat of it.
      const float scale = scale_log2 * 0.69314718055994531f;
      float l2f = kLog2e, grow_by = kRescaleNat;
      if (p.logit_scale != nullptr && row_ok) {
        const float f = __ldg(p.logit_scale + it.r0 + r);
        l2f = kLog2e * f;
        grow_by = kRescaleNat / f;
      }
      const int dmax = p.window > 0 ? p.window - 1 : 0x7fffffff;  // visible d in [0, dmax]
      float m_used = kNegInf, l = 0.f;
      bool ok = !bad;
      int next_id = __ldg(trow + (it.tf >> 1));
      for (int k = 0; k < it.ntiles && ok; ++k, ++n, ++e) {
        const int s = n & 1;
        const int j0 = (it.tf + k) * kTileKeys;
        const int id = next_id;
        if (k + 1 < it.ntiles) next_id = __ldg(trow + ((it.tf + k + 1) >> 1));
        // visible columns of this row: c in [clo, clo + span)
        const int dc = P - j0;  // distance of column 0
        const int clo = max(0, dc - dmax);
        int span = min(kTileKeys - 1, dc) - clo + 1;
        if (span < 0 || !row_ok || id < 0 || id >= p.num_blocks) span = 0;
        const bool warp_full = __all_sync(0xffffffffu, clo == 0 && span == kTileKeys);
        if (!mbar_wait(&bars[kSFull + s], (n >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld32(tl + kTmS + 64 * s, sr);
        tmem_ld32(tl + kTmS + 64 * s + 32, sr + 32);
        tmem_wait_ld();
        const uint8_t* slot = slot_wait(e);
        if (!slot) { ok = false; break; }
        uint64_t x2[32];  // the scores of columns (2 i, 2 i + 1)
        scores_with_bias<R16>(x2, sr, slot, r, it.P0,
                              it.P0 - j0 - (kTileKeys - 1) < p.rel_extent, scale);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kREmpty + ri.slot(e)]);
        const float mx = mask_and_max(x2, warp_full, clo, span);
        const bool grow = mx > m_used + grow_by;
        const float m_new = grow ? mx : m_used;
        const float alpha = (grow && m_used != kNegInf) ? ex2((m_used - m_new) * l2f) : 1.f;
        if (k > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O must hold every earlier tile before it is rescaled.  PV of this
          // tile cannot start before P is written below, so O's barrier is at
          // most one phase past the one waited for.
          if (!mbar_wait(&bars[kOFull], (n - 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < DV; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tl + kTmO + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tl + kTmO + c0, o);
          }
          tmem_wait_st();
        }
        l *= alpha;
        m_used = m_new;
        const float mb = m_used == kNegInf ? 0.f : -m_used * l2f;
        uint32_t pk[32];
        l += exp_pack<KV8>(x2, l2f, mb, pk);
        tmem_st32(tl + kTmS + 64 * s, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kPFull + s]);
      }
      // the item's last PV (phase n - 1) completes O, and every S = Q K^T of
      // the item with it
      if (!ok || !mbar_wait(&bars[kOFull], (n - 1) & 1)) bad = true;
      tc_fence_after();
      // The next item's query goes into TMEM first, so its first S = Q K^T
      // runs while this item's O is stored.  Its ring entry follows the
      // O scratch entry.
      const bool has_next = idx + static_cast<int>(gridDim.x) < total;
      if (has_next && !bad) {
        const uint8_t* qs = slot_wait(e + 1);
        PItem nit;
        prefill_item(idx + gridDim.x, p, sa, nit);
        if (!qs) bad = true;
        else load_q(qs, e + 1, r < nit.rows);
      }
      // O / l -> out, through the scratch slot (the tile's 128 rows, 16-byte
      // chunks swizzled by row / 4) so that the global stores are whole rows
      // (16 lanes per 256-byte row).  A bf16 row is DV * 2 bytes; an fp32 row
      // is twice that and goes in two halves of DV / 2 columns, each the size
      // of a bf16 row.
      uint8_t* scr = bad ? nullptr : slot_wait(e);
      if (!scr) bad = true;
      // the four softmax warps, once per item: all leave if any thread gave
      // up a wait or another role raised the abort flag
      if (named_barrier_or(1, 128, bad || *s_abort)) { fail = true; break; }
      // 1 / normaliser; the optional sink logit (not scaled by the factor)
      // joins it, against l's reference f m_used, and the optional gate's
      // sigmoid scales the row
      float inv;
      {
        float den = l;
        const size_t qi = static_cast<size_t>(it.r0 + r) * p.Hq + it.h;
        if (p.sink != nullptr && row_ok)
          den += ex2(__ldg(p.sink + qi) * kLog2e - m_used * l2f);  // 0 for a sink of -inf
        if constexpr (KV8)  // an e4m3 cache's value scale
          inv = den > 0.f ? p.v_scale / den : 0.f;
        else
          inv = den > 0.f ? 1.f / den : 0.f;
        if (p.gate != nullptr && row_ok) inv /= 1.f + ex2(-__ldg(p.gate + qi) * kLog2e);
      }
      constexpr int kCpr = DV / 8;     // 16-byte chunks per scratch row
      constexpr int kRpi = 32 / kCpr;  // rows per store instruction
      constexpr int passes = O32 ? 2 : 1;
#pragma unroll
      for (int half = 0; half < passes; ++half) {
        if (half > 0) named_barrier(1, 128);  // the first half's stores have read the scratch
        constexpr int cw = O32 ? DV / 2 : DV;  // columns of this pass
#pragma unroll 1
        for (int c0 = 0; c0 < cw; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tl + kTmO + half * cw + c0, o);
          tmem_wait_ld();
          if constexpr (O32) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint4 w;
              w.x = __float_as_uint(__uint_as_float(o[4 * i]) * inv);
              w.y = __float_as_uint(__uint_as_float(o[4 * i + 1]) * inv);
              w.z = __float_as_uint(__uint_as_float(o[4 * i + 2]) * inv);
              w.w = __float_as_uint(__uint_as_float(o[4 * i + 3]) * inv);
              const int j = c0 / 4 + i;  // 16-byte chunk of the row
              *reinterpret_cast<uint4*>(scr + r * (DV * 2) + ((j ^ ((r >> 2) & 7)) << 4)) = w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 w;
              w.x = pack_bf16(__uint_as_float(o[8 * i]) * inv, __uint_as_float(o[8 * i + 1]) * inv);
              w.y = pack_bf16(__uint_as_float(o[8 * i + 2]) * inv,
                              __uint_as_float(o[8 * i + 3]) * inv);
              w.z = pack_bf16(__uint_as_float(o[8 * i + 4]) * inv,
                              __uint_as_float(o[8 * i + 5]) * inv);
              w.w = pack_bf16(__uint_as_float(o[8 * i + 6]) * inv,
                              __uint_as_float(o[8 * i + 7]) * inv);
              const int j = c0 / 8 + i;  // 16-byte chunk of the row
              *reinterpret_cast<uint4*>(scr + r * (DV * 2) + ((j ^ ((r >> 2) & 7)) << 4)) = w;
            }
          }
        }
        // O is read before the next item's first PV overwrites it
        if (half == passes - 1) tc_fence_before();
        named_barrier(1, 128);  // the four softmax warps: every row is in the scratch
        // whole-row stores: this warp takes rows [32 q4, 32 q4 + 32)
#pragma unroll
        for (int i = 0; i < kCpr; ++i) {
          const int rr = 32 * q4 + i * kRpi + lane / kCpr;
          const int ch = lane % kCpr;
          const uint4 v =
              *reinterpret_cast<const uint4*>(scr + rr * (DV * 2) + ((ch ^ ((rr >> 2) & 7)) << 4));
          if (rr < it.rows) {
            const size_t orow = (static_cast<size_t>(it.r0 + rr) * p.Hq + it.h) * DV;
            if constexpr (O32)
              *reinterpret_cast<uint4*>(static_cast<float*>(p.out) + orow + half * (DV / 2) +
                                        ch * 4) = v;
            else
              *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow + ch * 8) = v;
          }
        }
      }
      fence_proxy_async_smem();  // these writes come before the slot's next TMA fill
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kREmpty + ri.slot(e)]);
      e += has_next ? 2 : 1;
    }
    if (fail) {
      report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
      *s_abort = 1;
    }
  }
  if (*s_abort && tid == 0) report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
  __syncwarp();  // lanes idle while lane 0 produced/issued rejoin here
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

int prefill_smem_bytes(int B, int dv, int ring_stages, int kv_es) {
  return PrefillSmem(B, dv, ring_stages, kv_es).total + 1024;
}

int prefill_ring_stages(int B, int dv, int kv_es, int smem_optin) {
  for (int nr = kMaxRingStages; nr >= 2; --nr)
    if (prefill_smem_bytes(B, dv, nr, kv_es) <= smem_optin) return nr;
  return 0;
}

// One thread waits on a barrier that nothing completes; the bounded wait
// gives up after its limit and reports it in the status word.
__global__ void wait_timeout_kernel(uint32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!mbar_wait(&bar, 0)) report(status, RELATTN_DEV_WAIT_TIMEOUT);
}

cudaError_t launch_wait_timeout(uint32_t* status, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_cache_write(const PrefillParams& p, cudaStream_t stream) {
  const dim3 grid((p.max_q_len + kCwTile - 1) / kCwTile, p.B);
  if (p.kv_es == 1)
    cache_write_kernel<true><<<grid, 256, 0, stream>>>(p);
  else
    cache_write_kernel<false><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int DV, bool R16, bool O32, bool KV8>
static cudaError_t launch_prefill_as(const PrefillLaunch& L, int grid, int smem,
                                     cudaStream_t stream) {
  cudaError_t e = ensure_smem<prefill_kernel<DV, R16, O32, KV8>>(smem);
  if (e != cudaSuccess) return e;
  prefill_kernel<DV, R16, O32, KV8><<<grid, 32 * (kPfWarps + (KV8 ? 1 : 0)), smem, stream>>>(
      L.tm_q, L.tm_k, L.tm_v, L.tm_rel, L.p);
  return cudaGetLastError();
}

template <int DV, bool R16, bool KV8>
static cudaError_t launch_prefill_out(const PrefillLaunch& L, int grid, int smem,
                                      cudaStream_t stream) {
  return L.p.out_f32 ? launch_prefill_as<DV, R16, true, KV8>(L, grid, smem, stream)
                     : launch_prefill_as<DV, R16, false, KV8>(L, grid, smem, stream);
}

cudaError_t launch_prefill(const PrefillLaunch& L, int grid, cudaStream_t stream) {
  const PrefillParams& p = L.p;
  const int smem = prefill_smem_bytes(p.B, p.dv, p.ring_stages, p.kv_es);
  const bool r16 = p.rel_es == 2;
  if (p.dv == 128) {
    if (p.kv_es == 1)  // e4m3 caches: d_v = 128 only
      return r16 ? launch_prefill_out<128, true, true>(L, grid, smem, stream)
                 : launch_prefill_out<128, false, true>(L, grid, smem, stream);
    return r16 ? launch_prefill_out<128, true, false>(L, grid, smem, stream)
               : launch_prefill_out<128, false, false>(L, grid, smem, stream);
  }
  if (p.kv_es == 1) return cudaErrorInvalidValue;  // the host refuses these first
  return r16 ? launch_prefill_out<64, true, false>(L, grid, smem, stream)
             : launch_prefill_out<64, false, false>(L, grid, smem, stream);
}


}  // namespace relattn
