// Chunked prefill over a bf16 cache with a bf16 rel, one query head per work
// item and 128-key tiles (sm_103a, tcgen05 / TMEM).
//
// A work item is one 128-row query tile of one sequence and one query head;
// a key tile is one whole 128-token cache block.  Per key tile:
//   S = Q K^T         tcgen05.mma, M = N = 128 (the tensor pipe's full rate;
//                     N = 64 runs at about 60%), Q in TMEM, K by TMA
//   bias, masks       the two softmax warpgroups split the tile's columns:
//                     group g takes keys 64 g .. 64 g + 63 of every row, adds
//                     rel[row, h, P_row - j] from the shared-memory rel boxes
//                     (the sheared bias; no [Lq, KV] mask is formed), then the
//                     causal and window masks; the two groups trade their row
//                     maxima through shared memory, so both move the running
//                     max (lazy rescale of O) the same way
//   O += P V          P written back over S in TMEM as bf16
// ("vLLM TML Inkling Support", section "Low-Latency Collectives and Kernels":
// the FA4 relative-attention kernel with a sheared bias; "Inkling 2 Small on
// vLLM": GQA, the heads of a KV group run on neighbouring CTAs so their K/V
// reads meet in L2).  S is double-buffered: the MMA warp computes S of the
// next key tile while the softmax works on this one, so a head's chain
// softmax -> P V -> next S never leaves the softmax waiting on the tensor pipe.
//
// TMEM (512 columns allocated, 448 used): Q [0, 64) (bf16 pairs), S buffers
// [64, 192) and [192, 320), O [320, 448).  Group g writes its P columns over
// the first 32 columns of its own 64-column half of the S buffer.
//
// Shared memory: a ring of three 32 KB K/V stages, used in the order the MMA
// warp needs them (K of tile 0, K of tile 1, V of tile 0, K of tile 2, V of
// tile 1, ...), and a ring of two 50 KB slots carrying, after the first
// item's query tile, per item: the rel boxes of each key tile, the next
// item's query tile, then a scratch slot for storing O (the next query comes
// first: the epilogue loads it before it needs the scratch, and the next
// item's first rel boxes can then be fetched during the epilogue).  Both
// softmax groups consume every ring entry.
//
// Warp roles: 0-3 and 4-7 = the softmax groups (TMEM lane quarters 0-3 each),
// 8 = K/V TMA producer, 9 = MMA issuer and TMEM owner, 10 = ring producer, 11
// idle.  The producer warpgroup hands most of its registers to the softmax.
#include "relattn_common.cuh"
#include "relattn_internal.h"
#include "relattn_prefill.cuh"
#include "relattn_tcgen05.cuh"

namespace relattn {

namespace {

using namespace prefill;

constexpr int kWarps = 12;
constexpr int kThreads = 32 * kWarps;
constexpr int kKvWarp = 8, kMmaWarp = 9, kRingWarp = 10;  // warpgroup 2
// Registers per thread: the launch gives every thread kLaunchRegs (the most
// that 384 threads may hold on one SM; the host checks that the kernel was
// built with exactly that many), then the producer warpgroup drops to
// kProdRegs and the two softmax warpgroups rise to kSoftRegs.
constexpr int kLaunchRegs = 168, kSoftRegs = 208, kProdRegs = 88;
static_assert(2 * 128 * kSoftRegs + 128 * kProdRegs <= kThreads * kLaunchRegs, "register split");
constexpr int kKeys = 128;                        // keys of one tile: one cache block
constexpr int kDv = 128;                          // d_v of this kernel
constexpr int kKvStages = 3;                      // K/V ring depth
constexpr int kKvStageBytes = kKeys * kDqk * 2;   // 32 KB (K, or V with d_v = 128)
constexpr int kRelTileBytes = kRelBoxes * kRelBoxBytesW;  // 51200 = 50 x 1024
constexpr int kSlotBytes = kRelTileBytes;  // also holds a query tile or an O scratch (32 KB)
// ring slots: two 50 KB slots beside the 96 KB of K/V stages (the ring's depth
// is a template parameter, so that entry -> slot and phase are cheap: a
// division by a run-time value costs hundreds of cycles on the softmax's path)
constexpr int kMinSlots = 2, kMaxSlots = 2;
static_assert(kSlotBytes % 1024 == 0 && kSlotBytes >= kQTileBytes, "slot size");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColO = 320;
__host__ __device__ constexpr uint32_t col_s(int b) { return 64u + 128u * b; }
constexpr uint32_t kIdescS = umma_idesc_bf16(128, kKeys, 0);
constexpr uint32_t kIdescPV = umma_idesc_bf16(128, kDv, 1);
constexpr int kXchgBar = 1;  // named barrier of the two softmax groups (256 threads)
// named barriers kPairBar + q4: the two warps (one per group) that hold the
// same 32 query rows, for the per-tile exchange of row maxima (64 threads)
constexpr int kPairBar = 2;

// Barriers.  K/V ring: full (TMA) / empty (MMA commit).  Per S buffer: S full
// (MMA commit), P full (the 8 softmax warps), O full (MMA commit after the
// P V that read this buffer).  Query in TMEM (8 warps).  Ring: full (TMA or
// producer arrive) / empty (the 8 softmax warps).
enum Bar {
  kKvFull = 0, kKvEmpty = kKvFull + kKvStages, kSFull = kKvEmpty + kKvStages,
  kPFull = kSFull + 2, kOFull = kPFull + 2, kQFull = kOFull + 2, kDrain = kQFull + 1,
  kRFull = kDrain + 1, kREmpty = kRFull + kMaxSlots, kNumBars = kREmpty + kMaxSlots
};

// Shared-memory carve-up (byte offsets from a 1024-aligned base).
struct WideSmem {
  int kv, ring, bars, xmax, lsum, misc, cu0, nrows, ctx, qpref, total;
  __host__ __device__ WideSmem(int B, int nslots) {
    kv = 0;
    ring = kv + kKvStages * kKvStageBytes;  // 1024-aligned: query tiles land 128B-swizzled
    bars = ring + nslots * kSlotBytes;
    xmax = bars + kNumBars * 8;  // [2 tiles][2 groups][128 rows] row maxima
    lsum = xmax + 2 * 2 * 128 * 4;  // [2 groups][128 rows] row sums
    misc = lsum + 2 * 128 * 4;
    cu0 = misc + 16;
    nrows = cu0 + B * 4;
    ctx = nrows + B * 4;
    qpref = ctx + B * 4;
    total = qpref + (B + 1) * 4;
  }
};

constexpr int kOutBoxBytes = 128 * 128;  // one 128-byte column box of 128 rows

// Work item idx: query tile idx / Hq, head idx % Hq, so that the heads of one
// query tile run on neighbouring CTAs.  Key tiles are 128-token blocks:
// [tf, tf + ntiles) are the blocks holding a key that a row of the tile sees.
struct WideItem {
  int b, h, kvh, r0, rows, P0, tf, ntiles;
};

__device__ __forceinline__ WideItem wide_item(int idx, const PrefillParams& p,
                                              const SeqArrays& a) {
  const int qtg = idx / p.Hq;
  const QTile t = query_tile(qtg, p, a);
  WideItem it;
  it.h = idx - qtg * p.Hq;
  it.kvh = it.h / p.g;
  it.b = t.b;
  it.r0 = t.r0;
  it.rows = t.rows;
  it.P0 = t.P0;
  it.tf = window_lo(t.P0, p.window) / kKeys;
  it.ntiles = (t.P0 + t.rows - 1) / kKeys - it.tf + 1;
  return it;
}

// The K/V loads of an item with n key tiles, in the order the MMA warp uses
// them: K0, K1, V0, K2, V1, ..., K(n-1), V(n-2), V(n-1).  Load i (0 .. 2n - 1)
// -> (is V, key tile).
__device__ __forceinline__ void kv_op(int i, int n, bool* is_v, int* tile) {
  if (i == 0) { *is_v = false; *tile = 0; return; }
  if (i == 2 * n - 1) { *is_v = true; *tile = n - 1; return; }
  // i = 2k - 1: K of tile k (k >= 1); i = 2k: V of tile k - 1
  *is_v = (i & 1) == 0;
  *tile = *is_v ? (i >> 1) - 1 : (i + 1) >> 1;
}

// O32: out is fp32 (else bf16).  NS: ring slots (kMinSlots .. kMaxSlots).
template <bool O32, int NS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_wide_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_rel,
                        const __grid_constant__ CUtensorMap tm_out, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  constexpr int nslots = NS;
  const WideSmem L(p.B, nslots);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  float* s_xmax = reinterpret_cast<float*>(smem + L.xmax);
  float* s_lsum = reinterpret_cast<float*>(smem + L.lsum);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.misc + 4);
  const SeqArrays sa{reinterpret_cast<int*>(smem + L.cu0), reinterpret_cast<int*>(smem + L.nrows),
                     reinterpret_cast<int*>(smem + L.ctx), reinterpret_cast<int*>(smem + L.qpref)};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(&bars[kKvFull + s], 1);
      mbar_init(&bars[kKvEmpty + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[kSFull + b], 1);
      mbar_init(&bars[kPFull + b], 8);
      mbar_init(&bars[kOFull + b], 1);
    }
    mbar_init(&bars[kQFull], 8);
    mbar_init(&bars[kDrain], 1);
    for (int s = 0; s < nslots; ++s) {
      mbar_init(&bars[kRFull + s], 1);
      mbar_init(&bars[kREmpty + s], 8);
    }
    fence_mbar_init();
    *s_abort = 0;
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_rel);
    tma_prefetch_desc(&tm_out);
  }
  // K/V stages start as zeros: a tile whose block id is invalid is never
  // loaded, and its P is zero, so its operands must at least be finite.
  for (int i = tid; i < (L.ring - L.kv) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem + L.kv)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == kMmaWarp) {
    tmem_alloc(s_tmem, kTmemCols);
    tc_fence_before();
  }
  const int total = prologue(p, sa, true) * p.Hq;  // has __syncthreads
  tc_fence_after();
  const uint32_t tbase = *s_tmem;

  if (warp >= kKvWarp) {
  // Each warpgroup changes its register count inside its own branch, so that
  // the compiler allocates each role's code with that role's count.
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProdRegs));
  if (warp == kKvWarp && lane == 0) {
    // ---------------------------------------------------- K/V TMA producer
    int c = 0;  // loads issued
    for (int idx = blockIdx.x; idx < total && !*s_abort; idx += gridDim.x) {
      const WideItem it = wide_item(idx, p, sa);
      const int* trow = p.block_table + static_cast<size_t>(it.b) * p.max_blocks;
      bool fail = false;
      for (int i = 0; i < 2 * it.ntiles; ++i, ++c) {
        bool is_v;
        int k;
        kv_op(i, it.ntiles, &is_v, &k);
        const int id = __ldg(trow + it.tf + k);
        const int s = c % kKvStages;
        if (!mbar_wait(&bars[kKvEmpty + s], ((c / kKvStages) & 1) ^ 1)) { fail = true; break; }
        uint64_t* full = &bars[kKvFull + s];
        if (id >= 0 && id < p.num_blocks) {
          uint8_t* d = smem + L.kv + s * kKvStageBytes;
          const CUtensorMap* m = is_v ? &tm_v : &tm_k;
          mbar_arrive_expect_tx(full, kKvStageBytes);
          tma_load_3d(d, m, full, 0, it.kvh, id * kKeys);
          tma_load_3d(d + kKvStageBytes / 2, m, full, 64, it.kvh, id * kKeys);
        } else {
          if (!is_v) report(p.status, RELATTN_DEV_BAD_BLOCK_ID);
          mbar_arrive(full);
        }
      }
      if (fail) { *s_abort = 1; break; }
    }
  } else if (warp == kRingWarp && lane == 0) {
    // --------------------------------------------------- ring producer
    int e = 0;
    bool fail = false;
    // A bf16 full tile's O scratch, once the softmax warps have written it and
    // released its slot, leaves through the tensor unit from this thread: when
    // the slot is next acquired, or at the end.  pend_e[slot] is that entry
    // (-1: none), pend_h / pend_r0 its head and first row.
    int pend_e[nslots], pend_h[nslots], pend_r0[nslots];
#pragma unroll
    for (int i = 0; i < nslots; ++i) {
      pend_e[i] = -1;
      pend_h[i] = 0;
      pend_r0[i] = 0;
    }
    auto store_out = [&](int slot) {
      const uint8_t* src = smem + L.ring + slot * kSlotBytes;
      tma_store_3d(&tm_out, src, 0, pend_h[slot], pend_r0[slot]);
      tma_store_3d(&tm_out, src + kOutBoxBytes, 64, pend_h[slot], pend_r0[slot]);
      tma_store_commit();
      tma_store_wait_read();  // the slot may be filled again
      pend_e[slot] = -1;
    };
    auto acquire = [&](int entry) -> uint8_t* {
      const int slot = entry % nslots;
      if (!mbar_wait(&bars[kREmpty + slot], ((entry / nslots) & 1) ^ 1)) return nullptr;
#pragma unroll
      for (int i = 0; i < nslots; ++i)  // (registers: no run-time index)
        if (i == slot && pend_e[i] >= 0) store_out(i);
      return smem + L.ring + slot * kSlotBytes;
    };
    // the query tile of item `qit` into ring entry e; rows past T read as zeros
    auto load_query = [&](const WideItem& qit) -> bool {
      uint8_t* qd = acquire(e);
      if (!qd) return false;
      uint64_t* qbar = &bars[kRFull + e % nslots];
      mbar_arrive_expect_tx(qbar, kQTileBytes);
      tma_load_3d(qd, &tm_q, qbar, 0, qit.h, qit.r0);
      tma_load_3d(qd + kQTileBytes / 2, &tm_q, qbar, 64, qit.h, qit.r0);
      ++e;
      return true;
    };
    if (static_cast<int>(blockIdx.x) < total && !load_query(wide_item(blockIdx.x, p, sa)))
      fail = true;
    for (int idx = blockIdx.x; idx < total && !*s_abort && !fail; idx += gridDim.x) {
      const WideItem it = wide_item(idx, p, sa);
      for (int k = 0; k < it.ntiles; ++k, ++e) {  // the rel boxes of each key tile
        const int j0 = (it.tf + k) * kKeys;
        uint8_t* rd = acquire(e);
        if (!rd) { fail = true; break; }
        uint64_t* rbar = &bars[kRFull + e % nslots];
        if (it.P0 - j0 - (kKeys - 1) < p.rel_extent) {
          mbar_arrive_expect_tx(rbar, kRelTileBytes);
          for (int bx = 0; bx < kRelBoxes; ++bx) {
            const int x = ((it.P0 + kRelBoxRows * bx - j0 - (kKeys - 1)) & ~7) -
                          kRelOddShift * (bx & 1);
            tma_load_3d(rd + bx * kRelBoxBytesW, &tm_rel, rbar, x, it.h,
                        it.r0 + kRelBoxRows * bx);
          }
        } else {
          mbar_arrive(rbar);  // every distance is past rel_extent
        }
      }
      if (fail) break;
      const int nidx = idx + static_cast<int>(gridDim.x);
      if (nidx < total && !load_query(wide_item(nidx, p, sa))) { fail = true; break; }
      if (!acquire(e)) { fail = true; break; }  // the O scratch
      if (!O32 && it.rows == kQRows) {
#pragma unroll
        for (int i = 0; i < nslots; ++i)
          if (i == e % nslots) {
            pend_e[i] = e;
            pend_h[i] = it.h;
            pend_r0[i] = it.r0;
          }
      }
      mbar_arrive(&bars[kRFull + e % nslots]);
      ++e;
    }
    // the scratch tiles not yet stored: once their slot is released
#pragma unroll
    for (int i = 0; i < nslots; ++i) {
      if (pend_e[i] < 0 || fail || *s_abort) continue;
      if (mbar_wait(&bars[kREmpty + i], (pend_e[i] / nslots) & 1))
        store_out(i);
      else
        fail = true;
    }
    tma_store_wait_all();  // the O stores of this thread are done
    if (fail) *s_abort = 1;
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs this loop, so that its counters, addresses and
    // descriptors stay warp-uniform (uniform registers, off the vector pipes
    // that the softmax warps keep busy); lane 0 issues the MMAs and their
    // commits.  A tcgen05.mma costs its issuing thread tens of cycles, so the
    // fewer instructions around each one the better: a k-step's descriptor is
    // the stage's descriptor plus a constant (the address field counts 16-byte
    // units and shared addresses stay below 2^18 bytes, so it cannot carry).
    const bool leader = lane == 0;
    int c = 0;   // K/V loads consumed (the producer's order)
    int ts = 0;  // S tiles issued (buffer ts & 1)
    int tp = 0;  // P tiles consumed by P V (buffer tp & 1)
    int nq = 0;  // query tiles
    const uint32_t kv0 = smem_u32(smem + L.kv);
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity));
    };
    auto kv_ready = [&](uint32_t* addr) -> bool {
      const int s = c % kKvStages;
      if (!wait_all(&bars[kKvFull + s], (c / kKvStages) & 1)) return false;
      tc_fence_after();
      *addr = kv0 + s * kKvStageBytes;
      return true;
    };
    // S = Q K^T of the next key tile into buffer ts & 1
    auto issue_s = [&]() -> bool {
      uint32_t kb;
      if (!kv_ready(&kb)) return false;
      const uint32_t d = tbase + col_s(ts & 1);
      const uint64_t kdesc = umma_desc_sw128(kb, 0, 1024);
      if (leader) {
#pragma unroll
        for (int ks = 0; ks < kDqk / 16; ++ks)
          umma_tmem_a(d, tbase + kColQ + 8 * ks,
                      kdesc + static_cast<uint64_t>(
                                  ((ks >> 2) * (kKvStageBytes / 2) + (ks & 3) * 32) >> 4),
                      kIdescS, ks > 0 ? 1 : 0);
        umma_commit(&bars[kSFull + (ts & 1)]);
        umma_commit(&bars[kKvEmpty + c % kKvStages]);
      }
      __syncwarp();
      ++c;
      ++ts;
      return true;
    };
    // O (+)= P V, P from buffer tp & 1 once the softmax has written it
    auto issue_pv = [&](bool acc) -> bool {
      const int b = tp & 1;
      if (!wait_all(&bars[kPFull + b], (tp >> 1) & 1)) return false;
      uint32_t vb;
      if (!kv_ready(&vb)) return false;
      const uint32_t a = tbase + col_s(b);
      const uint64_t vdesc = umma_desc_sw128(vb, kKeys * 128, 1024);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          umma_tmem_a(tbase + kColO, a + (kk < 4 ? 8 * kk : 64 + 8 * (kk - 4)),
                      vdesc + static_cast<uint64_t>((kk * 2048) >> 4), kIdescPV,
                      (acc || kk > 0) ? 1 : 0);
        umma_commit(&bars[kOFull + b]);
        umma_commit(&bars[kKvEmpty + c % kKvStages]);
      }
      __syncwarp();
      ++c;
      ++tp;
      return true;
    };
    for (int idx = blockIdx.x; idx < total && !*s_abort; idx += gridDim.x) {
      const WideItem it = wide_item(idx, p, sa);
      // the query tile in TMEM before the item's first S (the epilogue of the
      // previous item has read O and every earlier S is complete)
      bool ok = wait_all(&bars[kQFull], nq & 1);
      ++nq;
      tc_fence_after();
      // S of tile k + 1 goes out before P V of tile k, so the softmax finds
      // the next S ready; S of tile k + 2 reuses the buffer of P k, after P V
      // of tile k (the MMAs of one thread run in order)
      for (int k = 0; k < it.ntiles && ok; ++k) {
        ok = issue_s();
        if (ok && k > 0) ok = issue_pv(k > 1);
      }
      if (ok) ok = issue_pv(it.ntiles > 1);
      if (!ok) {
        if (leader) *s_abort = 1;
        break;
      }
    }
    // all MMAs retired before TMEM is released
    if (leader) umma_commit(&bars[kDrain]);
    __syncwarp();
    if (!wait_all(&bars[kDrain], 0) && leader) report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftRegs));
    // ------------------------------------------------------------ softmax
    // Group g takes keys [64 g, 64 g + 64) of every key tile.  Thread (q4,
    // lane) owns TMEM lane 32 q4 + lane and puts query row r = 4 lane + q4
    // there: each warp takes every fourth row, so all its lanes see the same
    // 8-byte alignment of their rows in the rel boxes.  The threads of the
    // two groups with the same (q4, lane) hold the same row.
    // A wait that gives up clears `ok` for its whole warp (the TMEM loads and
    // stores are warp-collective); the next exchange of row maxima, a
    // bar.red.or over the two warps that share its rows, takes both out of the
    // tile loop, and the item's barrier over both groups (after the loop)
    // takes all 256 threads out together (the other warps reach it when
    // their tiles end or their own bounded waits give up).
    const int g = warp >> 2;
    const int q4 = warp & 3;
    const int r = 4 * lane + q4;
    const uint32_t tl = tbase + (static_cast<uint32_t>(32 * q4) << 16);
    auto slot_wait = [&](int entry) -> const uint8_t* {
      const int slot = entry % nslots;
      if (!mbar_wait(&bars[kRFull + slot], (entry / nslots) & 1)) return nullptr;
      return smem + L.ring + slot * kSlotBytes;
    };
    auto slot_free = [&](int entry) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kREmpty + entry % nslots]);
    };
    // This thread's half of its query row (dims 64 g .. 64 g + 63), from the
    // ring slot (128-byte swizzled rows) into TMEM, the A operand of S = Q K^T.
    auto load_q = [&](const uint8_t* qs, int entry) {
      uint32_t qr[32];
      load_row128(qs + g * (kQTileBytes / 2), r, lane, qr);
      tmem_st32(tl + kColQ + 32 * g, qr);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kQFull]);
        mbar_arrive(&bars[kREmpty + entry % nslots]);
      }
    };
    int t = 0;       // S tiles consumed (buffer t & 1)
    int e_base = 1;  // this item's first ring entry (entry 0: the first item's query)
    int idx = blockIdx.x;
    WideItem it{};
    if (idx < total) it = wide_item(idx, p, sa);
    bool q_loaded = false;  // this item's query is in TMEM already
    while (idx < total) {
      const int n = it.ntiles;
      const int nidx = idx + static_cast<int>(gridDim.x);
      const bool has_next = nidx < total;
      const int e_qn = e_base + n;                  // the next item's query (if any)
      const int e_out = e_qn + (has_next ? 1 : 0);  // the item's O scratch
      bool bad = false;
      if (!q_loaded) {
        const uint8_t* qs = slot_wait(0);  // only the first item's query is not preloaded
        bad = !__all_sync(0xffffffffu, qs != nullptr);
        if (!bad) load_q(qs, 0);
      }
      const bool row_ok = r < it.rows;
      const int P = it.P0 + r;
      const int* trow = p.block_table + static_cast<size_t>(it.b) * p.max_blocks;

      // Scores in natural-log units: x = q.k / sqrt(d) + rel; exp2 takes
      // log2(e) in its FFMA.  A row's log-position factor f multiplies x:
      // it is folded into that log2(e) (l2f), and the lazy rescale moves the
      // running max of x only past kRescaleNat / f, so f x stays within
      // kRescaleNat of it.
      const float scale = p.scale_log2 * 0.69314718055994531f;
      float l2f = kLog2e, grow_by = kRescaleNat;
      if (p.logit_scale != nullptr && row_ok) {
        const float f = __ldg(p.logit_scale + it.r0 + r);
        l2f = kLog2e * f;
        grow_by = kRescaleNat / f;
      }
      const int dmax = p.window > 0 ? p.window - 1 : 0x7fffffff;  // visible d in [0, dmax]
      float m_used = kNegInf, l = 0.f;  // l: this group's columns only
      bool ok = !bad;
      int next_id = __ldg(trow + it.tf);
      for (int k = 0; k < n; ++k, ++t) {
        const int jg = (it.tf + k) * kKeys + 64 * g;  // first key of this group's half
        const int id = next_id;
        if (k + 1 < n) next_id = __ldg(trow + it.tf + k + 1);
        // visible columns of this row: c in [clo, clo + span)
        const int dc = P - jg;  // distance of column 0
        const int clo = max(0, dc - dmax);
        int span = min(63, dc) - clo + 1;
        if (span < 0 || !row_ok || id < 0 || id >= p.num_blocks) span = 0;
        const bool warp_full = __all_sync(0xffffffffu, clo == 0 && span == 64);
        const int b = t & 1;
        uint64_t x2[32];  // the scores of columns (2 i, 2 i + 1)
        float mx = kNegInf;
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars[kSFull + b], (t >> 1) & 1));
        if (ok) {
          tc_fence_after();
          uint32_t sr[64];
          tmem_ld32(tl + col_s(b) + 64 * g, sr);
          tmem_ld32(tl + col_s(b) + 64 * g + 32, sr + 32);
          tmem_wait_ld();
          const uint8_t* slot = slot_wait(e_base + k);
          ok = __all_sync(0xffffffffu, slot != nullptr);
          if (ok) {
            scores_with_bias_w2(x2, sr, slot, r, it.P0, g, it.P0 - jg - 63 < p.rel_extent, scale);
            slot_free(e_base + k);
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
            mx = fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
          }
        }
        // the row's max over both halves, traded with the other group's warp
        // that holds the same rows (the buffer alternates with the tile: the
        // pair's next barrier separates these reads from its next writes)
        float* xm = s_xmax + (t & 1) * 256;
        xm[128 * g + r] = mx;
        if (named_barrier_or(kPairBar + q4, 64, !ok)) { ok = false; break; }
        mx = fmaxf(xm[r], xm[128 + r]);
        const bool grow = mx > m_used + grow_by;
        const float m_new = grow ? mx : m_used;
        const float alpha = (grow && m_used != kNegInf) ? ex2((m_used - m_new) * l2f) : 1.f;
        if (k > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O must hold every earlier tile before it is rescaled: P V of the
          // previous tile (its buffer's barrier; the S just read came after
          // the P V before it, so that barrier is at most one phase behind)
          const int tq = t - 1;
          ok = __all_sync(0xffffffffu, mbar_wait(&bars[kOFull + (tq & 1)], (tq >> 1) & 1));
          if (!ok) continue;  // the next exchange (or the epilogue) takes everyone out
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 32) {  // this group's half of O
            uint32_t o[32];
            tmem_ld32(tl + kColO + 64 * g + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tl + kColO + 64 * g + c0, o);
          }
          tmem_wait_st();
        }
        l *= alpha;
        m_used = m_new;
        const float mb = m_used == kNegInf ? 0.f : -m_used * l2f;
        const uint64_t l2f2 = f2(l2f, l2f), mb2 = f2(mb, mb);
        uint32_t pk[32];
        uint64_t sq[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint64_t a2 = fma_f2(x2[i], l2f2, mb2);
          const float p0 = ex2(f2lo(a2)), p1 = ex2(f2hi(a2));
          sq[i & 1] = add_f2(sq[i & 1], f2(p0, p1));
          pk[i] = pack_bf16(p0, p1);
        }
        const uint64_t sqt = add_f2(sq[0], sq[1]);
        l += f2lo(sqt) + f2hi(sqt);
        tmem_st32(tl + col_s(b) + 64 * g, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kPFull + b]);
      }
      if (!ok) bad = true;
      // The next item's query goes into TMEM first: every S = Q K^T of this
      // item is complete (this thread saw the last S), so the next item's
      // first S can run while this item's last P V completes and O is stored.
      // Its ring entry comes before the O scratch, and both are filled
      // without waiting for this epilogue.
      if (has_next && !bad) {
        const uint8_t* qs = slot_wait(e_qn);
        bad = !__all_sync(0xffffffffu, qs != nullptr);
        if (!bad) load_q(qs, e_qn);
      }
      // the item's last P V completes O, and every earlier MMA with it
      if (!bad) {
        const int tq = t - 1;
        bad = !__all_sync(0xffffffffu, mbar_wait(&bars[kOFull + (tq & 1)], (tq >> 1) & 1));
      }
      tc_fence_after();
      uint8_t* scr = bad ? nullptr : const_cast<uint8_t*>(slot_wait(e_out));
      if (!bad) bad = !__all_sync(0xffffffffu, scr != nullptr);
      s_lsum[128 * g + r] = l;
      // both groups, once per item: all leave if any thread gave up a wait or
      // another role raised the abort flag
      if (named_barrier_or(kXchgBar, 256, bad || *s_abort)) break;
      // 1 / normaliser; the optional sink logit (not scaled by the factor)
      // joins it, against l's reference f m_used, and the optional gate's
      // sigmoid scales the row
      float inv;
      {
        float den = s_lsum[r] + s_lsum[128 + r];
        const size_t qi = static_cast<size_t>(it.r0 + r) * p.Hq + it.h;
        if (p.sink != nullptr && row_ok)
          den += ex2(__ldg(p.sink + qi) * kLog2e - m_used * l2f);  // 0 for a sink of -inf
        inv = den > 0.f ? 1.f / den : 0.f;
        if (p.gate != nullptr && row_ok) inv /= 1.f + ex2(-__ldg(p.gate + qi) * kLog2e);
      }
      if (it.rows == kQRows) {
        // A full tile: O / l goes into the scratch slot as 128-byte column
        // boxes of 128 rows (the tensor map's 128-byte swizzle), stored with
        // the tensor unit by the ring producer once the 8 warps released the
        // slot (bf16), or by one softmax thread (fp32).  Group g fills box g (bf16; an
        // fp32 row is twice as long and goes in two passes, box 2 pass + g
        // of each).  Each lane writes its 16-byte chunks starting at chunk
        // lane & 7, so the 8 lanes of a quarter-warp, whose rows are 4
        // apart, hit 8 different bank groups.
        const int rot = lane & 7;
        constexpr int passes = O32 ? 2 : 1;
#pragma unroll
        for (int pass = 0; pass < passes; ++pass) {
          uint32_t w[32];
          if constexpr (O32) {
            tmem_ld32(tl + kColO + 64 * pass + 32 * g, w);
            tmem_wait_ld();
#pragma unroll
            for (int i2 = 0; i2 < 32; ++i2) w[i2] = __float_as_uint(__uint_as_float(w[i2]) * inv);
          } else {
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
              uint32_t o[32];
              tmem_ld32(tl + kColO + 64 * g + c0, o);
              tmem_wait_ld();
#pragma unroll
              for (int i2 = 0; i2 < 16; ++i2)
                w[c0 / 2 + i2] =
                    pack_bf16(__uint_as_float(o[2 * i2]) * inv, __uint_as_float(o[2 * i2 + 1]) * inv);
            }
          }
          if (pass == passes - 1) tc_fence_before();  // O is read before the next item's P V
          rotate_chunks(w, rot);  // chunk (s + rot) & 7 at position s
          uint8_t* box = scr + g * kOutBoxBytes;
#pragma unroll
          for (int s2 = 0; s2 < 8; ++s2)
            *reinterpret_cast<uint4*>(box + sw128(r, (s2 + rot) & 7)) =
                make_uint4(w[4 * s2], w[4 * s2 + 1], w[4 * s2 + 2], w[4 * s2 + 3]);
          fence_proxy_async_smem();  // the boxes are read by the tensor unit
          if constexpr (!O32) {
            // the ring producer stores the tile once all 8 warps released it
            slot_free(e_out);
          } else {
            named_barrier(kXchgBar, 256);
            if (warp == 0 && lane == 0) {
#pragma unroll
              for (int bx = 0; bx < 2; ++bx)
                tma_store_3d(&tm_out, scr + bx * kOutBoxBytes, (2 * pass + bx) * 32, it.h,
                             it.r0);
              tma_store_commit();
              tma_store_wait_read();  // the scratch may be written again
              if (pass == passes - 1) mbar_arrive_n(&bars[kREmpty + e_out % nslots], 8);
            }
            __syncwarp();
            if (pass < passes - 1) named_barrier(kXchgBar, 256);
          }
        }
      } else {
        // O / l -> out, through the scratch slot (the tile's 128 rows of 256
        // bytes, 16-byte chunks swizzled by row / 4) so that the global stores
        // are whole rows (16 lanes per row).  A bf16 row is 256 bytes; an fp32
        // row is twice that and goes in two passes of 64 columns.  Group g
        // fills chunks [8 g, 8 g + 8) of every row of a pass.
        constexpr int passes = O32 ? 2 : 1;
#pragma unroll
        for (int half = 0; half < passes; ++half) {
          if (half > 0) named_barrier(kXchgBar, 256);  // the first pass's stores have read the scratch
          if constexpr (O32) {
            uint32_t o[32];
            tmem_ld32(tl + kColO + 64 * half + 32 * g, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint4 w;
              w.x = __float_as_uint(__uint_as_float(o[4 * i]) * inv);
              w.y = __float_as_uint(__uint_as_float(o[4 * i + 1]) * inv);
              w.z = __float_as_uint(__uint_as_float(o[4 * i + 2]) * inv);
              w.w = __float_as_uint(__uint_as_float(o[4 * i + 3]) * inv);
              const int j = 8 * g + i;
              *reinterpret_cast<uint4*>(scr + r * 256 + ((j ^ ((r >> 2) & 7)) << 4)) = w;
            }
          } else {
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
              uint32_t o[32];
              tmem_ld32(tl + kColO + 64 * g + c0, o);
              tmem_wait_ld();
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
                const int j = 8 * g + c0 / 8 + i;
                *reinterpret_cast<uint4*>(scr + r * 256 + ((j ^ ((r >> 2) & 7)) << 4)) = w;
              }
            }
          }
          // O is read before the next item's first P V overwrites it
          if (half == passes - 1) tc_fence_before();
          named_barrier(kXchgBar, 256);  // every row is in the scratch
          // whole-row stores: warp w takes rows [16 w, 16 w + 16), two per pass
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 16 * warp + 2 * i + (lane >> 4);
            const int ch = lane & 15;
            const uint4 v =
                *reinterpret_cast<const uint4*>(scr + rr * 256 + ((ch ^ ((rr >> 2) & 7)) << 4));
            if (rr < it.rows) {
              const size_t orow = (static_cast<size_t>(it.r0 + rr) * p.Hq + it.h) * kDv;
              if constexpr (O32)
                *reinterpret_cast<uint4*>(static_cast<float*>(p.out) + orow + 64 * half + ch * 4) = v;
              else
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow + ch * 8) = v;
            }
          }
        }
        fence_proxy_async_smem();  // these writes come before the slot's next TMA fill
        slot_free(e_out);
      }
      idx = nidx;
      e_base = e_out + 1;
      if (has_next) it = wide_item(idx, p, sa);
      q_loaded = has_next;
    }
    if (idx < total) {  // left early: a wait gave up here or in another role
      report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
      *s_abort = 1;
    }
  }
  if (tid == 0) tma_store_wait_all();  // the O stores this thread issued are done
  if (*s_abort && tid == 0) report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
  __syncwarp();  // lanes idle while lane 0 produced/issued rejoin here
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, kTmemCols);
}

// Replays the work split and block walk of prefill_wide_kernel with the same
// device functions (prologue, wide_item) and the same grid: each (item, key
// tile) appends { sequence, first row of its query tile within the sequence,
// key tile (a 128-key tile: the logical block), logical block, physical
// block, head }.
__global__ void __launch_bounds__(128) prefill_wide_walk_kernel(const PrefillParams p) {
  extern __shared__ int seq_arrays[];  // 4 B + 1 ints
  const SeqArrays sa{seq_arrays, seq_arrays + p.B, seq_arrays + 2 * p.B, seq_arrays + 3 * p.B};
  const int total = prologue(p, sa, false) * p.Hq;
  if (threadIdx.x != 0) return;
  for (int idx = blockIdx.x; idx < total; idx += gridDim.x) {
    const WideItem it = wide_item(idx, p, sa);
    const int* trow = p.block_table + static_cast<size_t>(it.b) * p.max_blocks;
    for (int k = 0; k < it.ntiles; ++k) {
      const int tile = it.tf + k;
      const int r = atomicAdd(p.dbg_count, 1);
      if (r < p.dbg_max) {
        int32_t* rec = p.dbg_records + 6 * static_cast<size_t>(r);
        rec[0] = it.b;
        rec[1] = it.r0 - sa.cu0[it.b];
        rec[2] = tile;
        rec[3] = tile;
        rec[4] = __ldg(trow + tile);
        rec[5] = it.h;
      }
    }
  }
}

}  // namespace

cudaError_t launch_prefill_wide_walk(const PrefillParams& p, int grid, cudaStream_t stream) {
  const int smem = (4 * p.B + 1) * 4;
  cudaError_t e = ensure_smem<prefill_wide_walk_kernel>(smem);
  if (e != cudaSuccess) return e;
  prefill_wide_walk_kernel<<<grid, 128, smem, stream>>>(p);
  return cudaGetLastError();
}

int prefill_wide_smem_bytes(int B, int nslots) { return WideSmem(B, nslots).total + 1024; }

int prefill_wide_slots(int B, int smem_optin) {
  for (int ns = kMaxSlots; ns >= kMinSlots; --ns)
    if (prefill_wide_smem_bytes(B, ns) <= smem_optin) return ns;
  return 0;
}

template <bool O32, int NS>
static cudaError_t launch_wide_as(const PrefillLaunch& L, int grid, int smem, cudaStream_t stream) {
  // The kernel's register split assumes the launch holds kLaunchRegs per
  // thread; with fewer, the softmax warpgroups' raise could never be met.
  static const int regs = [] {
    cudaFuncAttributes a{};
    return cudaFuncGetAttributes(&a, prefill_wide_kernel<O32, NS>) == cudaSuccess ? a.numRegs
                                                                                  : -1;
  }();
  if (regs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  cudaError_t e = ensure_smem<prefill_wide_kernel<O32, NS>>(smem);
  if (e != cudaSuccess) return e;
  prefill_wide_kernel<O32, NS><<<grid, kThreads, smem, stream>>>(L.tm_q, L.tm_k, L.tm_v,
                                                                 L.tm_rel, L.tm_out, L.p);
  return cudaGetLastError();
}

template <bool O32>
static cudaError_t launch_wide_ns(const PrefillLaunch& L, int grid, int smem,
                                  cudaStream_t stream) {
  static_assert(kMinSlots == 2 && kMaxSlots == 2, "ring depths instantiated here");
  return L.p.ring_stages == 2 ? launch_wide_as<O32, 2>(L, grid, smem, stream)
                              : cudaErrorInvalidValue;
}

cudaError_t launch_prefill_wide(const PrefillLaunch& L, int grid, cudaStream_t stream) {
  const PrefillParams& p = L.p;
  // bf16 caches with d_v = 128 and a bf16 rel only
  if (p.kv_es != 2 || p.rel_es != 2 || p.dv != kDv) return cudaErrorInvalidValue;
  const int smem = prefill_wide_smem_bytes(p.B, p.ring_stages);
  return p.out_f32 ? launch_wide_ns<true>(L, grid, smem, stream)
                   : launch_wide_ns<false>(L, grid, smem, stream);
}

}  // namespace relattn
