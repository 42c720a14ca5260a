// Chunked prefill over a bf16 cache, two query heads of one KV group per work
// item (sm_103a, tcgen05 / TMEM).
//
// A work item is one 128-row query tile of one sequence and a pair of query
// heads that share a KV head (GQA: "Inkling 2 Small on vLLM", section "vLLM
// integration and optimisation": the heads of one KV group share each read of
// their keys and values).  Each 64-key K/V tile is loaded once for both heads.
// For each key tile and head slot i (0, 1):
//   S_i = Q_i K^T     tcgen05.mma, Q_i in TMEM, K from TMA (128B swizzle)
//   bias, masks       softmax warpgroup i adds rel[row, h_i, P_row - j] from
//                     its shared-memory rel boxes (the sheared bias; no
//                     [Lq, KV] mask is formed), then the causal and window
//                     masks, then the online softmax (lazy rescale of O)
//   O_i += P_i V      P_i written back over S_i in TMEM as bf16
// ("vLLM TML Inkling Support", section "Low-Latency Collectives and Kernels":
// the FA4 relative-attention kernel with a sheared bias).  The two softmax
// warpgroups alternate on the tensor pipe: while group 0 turns S_0 into P_0,
// the MMA warp runs O_1 += P_1 V and S_1 of the next key tile, and the other
// way round, so the softmax of one head hides the MMAs of the other.
//
// TMEM (512 columns): Q_0 [0, 64), Q_1 [64, 128) (bf16 pairs), S_0 [128, 192),
// S_1 [192, 256), O_0 and O_1 from 256, d_v columns each.
//
// One ring of shared-memory slots carries, in this order per item: the query
// tile of each head, then for each key tile the rel boxes of each head, then
// a scratch slot per head for storing O.  Each entry is consumed by the
// softmax group of its head; the producer fills entries in order.
//
// Warp roles: 0-3 = softmax of head slot 0, 4-7 = softmax of head slot 1
// (TMEM lane quarters 0-3 each), 8 = K/V TMA producer, 9 = MMA issuer and
// TMEM owner, 10 = ring producer, 11 idle.  The producer warpgroup (8-11)
// hands most of its registers to the two softmax warpgroups.
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
// kProdRegs and the two softmax warpgroups rise to kSoftRegs:
// 2 x 128 x 208 + 128 x 88 = 384 x 168.
constexpr int kLaunchRegs = 168, kSoftRegs = 208, kProdRegs = 88;
static_assert(2 * 128 * kSoftRegs + 128 * kProdRegs <= kThreads * kLaunchRegs, "register split");
constexpr int kMaxSlots = 6;  // ring slots, at most
constexpr int kMinSlots = 3;  // fewer would deadlock the ring (see the epilogue)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescS = umma_idesc_bf16(128, kTileKeys, 0);

__host__ __device__ constexpr uint32_t col_q(int i) { return 64u * i; }
__host__ __device__ constexpr uint32_t col_s(int i) { return 128u + 64u * i; }
__host__ __device__ constexpr uint32_t col_o(int i, int dv) { return 256u + dv * i; }

// Barriers.  K/V stages: full (TMA) / empty (MMA commit).  Per head slot:
// S full (MMA commit), P full (its 4 softmax warps), O full (MMA commit after
// each P V), query in TMEM (4 warps).  Ring: full (TMA or producer arrive) /
// empty (the consuming group's 4 warps).
// A query tile lands on its group's own barrier (kQLoad, once per item of
// that group), not on its slot's full barrier: the second group skips the
// items that have one head only, so its next query entry can be further
// ahead of the producer than a parity wait on the slot can tell apart.
enum Bar {
  kKFull = 0, kKEmpty = 2, kVFull = 4, kVEmpty = 6, kSFull = 8, kPFull = 10, kOFull = 12,
  kQFull = 14, kQLoad = 16, kDrain = 18, kRFull = 19, kREmpty = kRFull + kMaxSlots,
  kNumBars = kREmpty + kMaxSlots
};

// Bytes of one ring slot: the rel boxes of one head and key tile (fp32: 4 x
// 12800; bf16: 4 x 6656), and at least a query tile or an O scratch (32 KB).
__host__ __device__ constexpr int slot_bytes(int rel_es) {
  return rel_es == 2 ? kQTileBytes : kRelBoxes * kRelBoxBytes;
}

// Shared-memory carve-up (byte offsets from a 1024-aligned base).
struct PairSmem {
  int k, v, vstage, ring, slot, bars, misc, cu0, nrows, ctx, qpref, total;
  __host__ __device__ PairSmem(int B, int dv, int rel_es, int nslots) {
    vstage = kTileKeys * dv * 2;
    k = 0;
    v = k + 2 * kKStageBytes;
    ring = v + 2 * vstage;  // 1024-aligned: query tiles land 128B-swizzled
    slot = slot_bytes(rel_es);
    bars = ring + nslots * slot;
    misc = bars + kNumBars * 8;
    cu0 = misc + 16;
    nrows = cu0 + B * 4;
    ctx = nrows + B * 4;
    qpref = ctx + B * 4;
    total = qpref + (B + 1) * 4;
  }
};

// Work item idx: query tile idx / (Hkv * npairs), then KV head, then head
// pair j (heads kvh g + 2 j and, if g allows, kvh g + 2 j + 1).  The items of
// one query tile run on neighbouring CTAs, so its K/V tiles are shared in L2.
struct PairItem {
  int b, kvh, h0, nh, r0, rows, P0, tf, ntiles;
};

__device__ __forceinline__ PairItem pair_item(int idx, const PrefillParams& p,
                                              const SeqArrays& a) {
  const int npairs = (p.g + 1) >> 1;
  const int per_tile = p.Hkv * npairs;
  const int qtg = idx / per_tile;
  const int rem = idx - qtg * per_tile;
  PairItem it;
  it.kvh = rem / npairs;
  const int j = rem - it.kvh * npairs;
  it.h0 = it.kvh * p.g + 2 * j;
  it.nh = min(2, p.g - 2 * j);
  const QTile t = query_tile(qtg, p, a);
  it.b = t.b;
  it.r0 = t.r0;
  it.rows = t.rows;
  it.P0 = t.P0;
  it.tf = t.tf;
  it.ntiles = t.ntiles;
  return it;
}

// Ring entries of one item: a query tile per head, the rel boxes of every
// (key tile, head), an O scratch per head.
__device__ __forceinline__ int item_entries(const PairItem& it) {
  return it.nh * (it.ntiles + 2);
}

// R16: rel is bf16 (else fp32).  O32: out is fp32 (else bf16).
template <int DV, bool R16, bool O32>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_rel, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const int nslots = p.ring_stages;
  const RingIndex ri(p.ring_stages);  // ring entry -> slot, phase
  const PairSmem L(p.B, DV, R16 ? 2 : 4, nslots);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.misc + 4);
  const SeqArrays sa{reinterpret_cast<int*>(smem + L.cu0), reinterpret_cast<int*>(smem + L.nrows),
                     reinterpret_cast<int*>(smem + L.ctx), reinterpret_cast<int*>(smem + L.qpref)};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kKFull + s], 1);
      mbar_init(&bars[kKEmpty + s], 1);
      mbar_init(&bars[kVFull + s], 1);
      mbar_init(&bars[kVEmpty + s], 1);
      mbar_init(&bars[kSFull + s], 1);
      mbar_init(&bars[kPFull + s], 4);
      mbar_init(&bars[kOFull + s], 1);
      mbar_init(&bars[kQFull + s], 4);
      mbar_init(&bars[kQLoad + s], 1);
    }
    for (int s = 0; s < nslots; ++s) {
      mbar_init(&bars[kRFull + s], 1);
      mbar_init(&bars[kREmpty + s], 4);
    }
    mbar_init(&bars[kDrain], 1);
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
  if (warp == kMmaWarp) {
    tmem_alloc(s_tmem, kTmemCols);
    tc_fence_before();
  }
  const int total = prologue(p, sa, true) * p.Hkv * ((p.g + 1) >> 1);  // has __syncthreads
  tc_fence_after();
  const uint32_t tbase = *s_tmem;

  if (warp >= kKvWarp) {
  // Each warpgroup changes its register count inside its own branch, so that
  // the compiler allocates each role's code with that role's count.
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProdRegs));
  if (warp == kKvWarp && lane == 0) {
    // ---------------------------------------------------- K/V TMA producer
    int n = 0;
    for (int idx = blockIdx.x; idx < total && !*s_abort; idx += gridDim.x) {
      const PairItem it = pair_item(idx, p, sa);
      const int* trow = p.block_table + static_cast<size_t>(it.b) * p.max_blocks;
      for (int k = 0; k < it.ntiles; ++k, ++n) {
        const KvTile kt = kv_tile(trow, it.tf + k, p.num_blocks);
        const bool ok = kt.ok;
        const int row = kt.row;
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
  } else if (warp == kRingWarp && lane == 0) {
    // --------------------------------------------------- ring producer
    int e = 0;
    bool fail = false;
    auto acquire = [&](int entry) -> uint8_t* {
      const int slot = ri.slot(entry);
      if (!mbar_wait(&bars[kREmpty + slot], ri.phase(entry) ^ 1)) return nullptr;
      return smem + L.ring + slot * L.slot;
    };
    for (int idx = blockIdx.x; idx < total && !*s_abort && !fail; idx += gridDim.x) {
      const PairItem it = pair_item(idx, p, sa);
      for (int i = 0; i < it.nh; ++i, ++e) {  // the query tile of each head
        uint8_t* qd = acquire(e);
        if (!qd) { fail = true; break; }
        mbar_arrive(&bars[kRFull + ri.slot(e)]);  // the slot's phase; the data lands on kQLoad
        uint64_t* qbar = &bars[kQLoad + i];
        mbar_arrive_expect_tx(qbar, kQTileBytes);  // rows past T read as zeros
        tma_load_3d(qd, &tm_q, qbar, 0, it.h0 + i, it.r0);
        tma_load_3d(qd + kQTileBytes / 2, &tm_q, qbar, 64, it.h0 + i, it.r0);
      }
      for (int k = 0; k < it.ntiles && !fail; ++k) {
        const int j0 = (it.tf + k) * kTileKeys;
        const bool has_rel = it.P0 - j0 - (kTileKeys - 1) < p.rel_extent;
        for (int i = 0; i < it.nh; ++i, ++e) {
          uint8_t* rd = acquire(e);
          if (!rd) { fail = true; break; }
          uint64_t* rbar = &bars[kRFull + ri.slot(e)];
          if (has_rel) {
            constexpr int kBox = R16 ? kRelBoxBytes16 : kRelBoxBytes;
            mbar_arrive_expect_tx(rbar, kRelBoxes * kBox);
            for (int bx = 0; bx < kRelBoxes; ++bx) {
              const int x = (it.P0 + kRelBoxRows * bx - j0 - (kTileKeys - 1)) & (R16 ? ~7 : ~3);
              tma_load_3d(rd + bx * kBox, &tm_rel, rbar, x, it.h0 + i, it.r0 + kRelBoxRows * bx);
            }
          } else {
            mbar_arrive(rbar);  // every distance is past rel_extent
          }
        }
      }
      for (int i = 0; i < it.nh && !fail; ++i, ++e) {  // the O scratch of each head
        if (!acquire(e)) { fail = true; break; }
        mbar_arrive(&bars[kRFull + ri.slot(e)]);
      }
    }
    if (fail) *s_abort = 1;
  } else if (warp == kMmaWarp && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t kIdescPV = umma_idesc_bf16(128, DV, 1);
    int n = 0;               // K/V tiles
    int ts[2] = {0, 0};      // S tiles issued per head slot
    int qi[2] = {0, 0};      // items per head slot
    // O_i += P_i V of K/V tile m, P_i from slot i's last S tile
    auto issue_pv = [&](int i, int m, bool acc) -> bool {
      if (!mbar_wait(&bars[kPFull + i], (ts[i] - 1) & 1) ||
          !mbar_wait(&bars[kVFull + (m & 1)], (m >> 1) & 1))
        return false;
      tc_fence_after();
      const uint32_t vb = smem_u32(smem + L.v + (m & 1) * L.vstage);
#pragma unroll
      for (int kk = 0; kk < kTileKeys / 16; ++kk)
        umma_tmem_a(tbase + col_o(i, DV), tbase + col_s(i) + 8 * kk,
                    umma_desc_sw128(vb + kk * 2048, kTileKeys * 128, 1024), kIdescPV,
                    (acc || kk > 0) ? 1 : 0);
      umma_commit(&bars[kOFull + i]);
      return true;
    };
    for (int idx = blockIdx.x; idx < total && !*s_abort; idx += gridDim.x) {
      const PairItem it = pair_item(idx, p, sa);
      bool ok = true;
      for (int k = 0; k < it.ntiles && ok; ++k, ++n) {
        const int s = n & 1;
        if (!mbar_wait(&bars[kKFull + s], (n >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kb = smem_u32(smem + L.k + s * kKStageBytes);
        for (int i = 0; i < it.nh; ++i) {
          // head i's query tile in TMEM, before its first S
          if (k == 0) {
            if (!mbar_wait(&bars[kQFull + i], qi[i] & 1)) { ok = false; break; }
            ++qi[i];
            tc_fence_after();
          }
          // P_i of the previous key tile goes first: S_i of this one
          // overwrites it in TMEM (the MMAs of one thread run in order)
          if (k > 0 && !issue_pv(i, n - 1, k > 1)) { ok = false; break; }
#pragma unroll
          for (int ks = 0; ks < kDqk / 16; ++ks)
            umma_tmem_a(tbase + col_s(i), tbase + col_q(i) + 8 * ks,
                        umma_desc_sw128(kb + (ks >> 2) * 8192 + (ks & 3) * 32, 0, 1024), kIdescS,
                        ks > 0 ? 1 : 0);
          umma_commit(&bars[kSFull + i]);
          ++ts[i];
        }
        if (!ok) break;
        umma_commit(&bars[kKEmpty + s]);
        if (k > 0) umma_commit(&bars[kVEmpty + ((n - 1) & 1)]);
      }
      for (int i = 0; i < it.nh && ok; ++i) ok = issue_pv(i, n - 1, it.ntiles > 1);
      if (ok) umma_commit(&bars[kVEmpty + ((n - 1) & 1)]);
      if (!ok) { *s_abort = 1; break; }
    }
    // all MMAs retired before TMEM is released
    umma_commit(&bars[kDrain]);
    if (!mbar_wait(&bars[kDrain], 0)) report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftRegs));
    // ------------------------------------------------------------ softmax
    // Group wg = 0, 1 serves head slot wg.  Thread (q4, lane) owns TMEM lane
    // 32 q4 + lane and puts query row r = 4 lane + q4 there: each warp takes
    // every fourth row, so all its lanes see the same 16-byte alignment of
    // their rows in the rel boxes.
    const int wg = warp >> 2;
    const int bar_id = 1 + wg;  // the group's named barrier (128 threads)
    const int q4 = warp & 3;    // TMEM lane quarter this warp may access
    const int r = 4 * lane + q4;
    const uint32_t tl = tbase + (static_cast<uint32_t>(32 * q4) << 16);
    const uint32_t cq = tl + col_q(wg), cs = tl + col_s(wg), co = tl + col_o(wg, DV);
    int t = 0;   // S tiles consumed by this group
    int nq = 0;  // query tiles consumed by this group
    // The query tile of ring entry `entry` (this group's next), once landed.
    auto q_wait = [&](int entry) -> const uint8_t* {
      if (!mbar_wait(&bars[kQLoad + wg], nq & 1)) return nullptr;
      ++nq;
      return smem + L.ring + ri.slot(entry) * L.slot;
    };
    auto slot_wait = [&](int entry) -> uint8_t* {
      const int slot = ri.slot(entry);
      if (!mbar_wait(&bars[kRFull + slot], ri.phase(entry))) return nullptr;
      return smem + L.ring + slot * L.slot;
    };
    // This thread's query row, from a ring slot (128-byte swizzled rows) into
    // TMEM, the A operand of S = Q K^T; then the MMA warp may start.
    auto load_q = [&](const uint8_t* qs, int entry) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t qr[32];
        load_row128(qs + c * (kQTileBytes / 2), r, lane, qr);
        tmem_st32(cq + 32 * c, qr);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kQFull + wg]);
        mbar_arrive(&bars[kREmpty + ri.slot(entry)]);
      }
    };
    // The first item from `idx` on in which this group has a head, with the
    // ring entries of the items before it added to *base.
    auto next_item = [&](int idx, int* base, PairItem* it) -> int {
      for (; idx < total; idx += gridDim.x) {
        *it = pair_item(idx, p, sa);
        if (it->nh > wg) break;
        *base += item_entries(*it);
      }
      return idx;
    };
    int e_base = 0;  // ring entries of all earlier items
    PairItem it;
    int idx = next_item(blockIdx.x, &e_base, &it);
    bool q_loaded = false;  // this item's query is in TMEM already
    while (idx < total) {
      const int nh = it.nh;
      const int e_out = e_base + nh * (it.ntiles + 1) + wg;  // this head's O scratch
      // the next item of this group and its entries
      int nbase = e_base + item_entries(it);
      PairItem nit;
      const int nidx = next_item(idx + gridDim.x, &nbase, &nit);
      // The next item's query is loaded during this epilogue only when that
      // item directly follows this one: its ring entry is then at most three
      // entries past this group's O scratch.  Past an item of the other
      // group alone, the ring could not reach it before this group frees its
      // scratch.
      const bool preload = nidx < total && nidx == idx + static_cast<int>(gridDim.x);
      // A wait that gives up marks the item bad: the warp skips the rest of
      // its work but still meets the other warps of its group at the barrier
      // before the epilogue, after which all four leave together (a warp
      // leaving alone would strand the others at a named barrier).
      bool bad = false;
      if (!q_loaded) {
        const uint8_t* qs = q_wait(e_base + wg);
        if (!qs) bad = true;
        else load_q(qs, e_base + wg);
      }
      const int h = it.h0 + wg;
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
      float m_used = kNegInf, l = 0.f;
      bool ok = !bad;
      int next_id = __ldg(trow + (it.tf >> 1));
      for (int k = 0; k < it.ntiles && ok; ++k, ++t) {
        const int j0 = (it.tf + k) * kTileKeys;
        const int id = next_id;
        if (k + 1 < it.ntiles) next_id = __ldg(trow + ((it.tf + k + 1) >> 1));
        // visible columns of this row: c in [clo, clo + span)
        const int dc = P - j0;  // distance of column 0
        const int clo = max(0, dc - dmax);
        int span = min(kTileKeys - 1, dc) - clo + 1;
        if (span < 0 || !row_ok || id < 0 || id >= p.num_blocks) span = 0;
        const bool warp_full = __all_sync(0xffffffffu, clo == 0 && span == kTileKeys);
        if (!mbar_wait(&bars[kSFull + wg], t & 1)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld32(cs, sr);
        tmem_ld32(cs + 32, sr + 32);
        tmem_wait_ld();
        const int e_rel = e_base + nh * (1 + k) + wg;
        const uint8_t* slot = slot_wait(e_rel);
        if (!slot) { ok = false; break; }
        uint64_t x2[32];  // the scores of columns (2 i, 2 i + 1)
        scores_with_bias<R16>(x2, sr, slot, r, it.P0,
                              it.P0 - j0 - (kTileKeys - 1) < p.rel_extent, scale);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kREmpty + ri.slot(e_rel)]);
        const float mx = mask_and_max(x2, warp_full, clo, span);
        const bool grow = mx > m_used + grow_by;
        const float m_new = grow ? mx : m_used;
        const float alpha = (grow && m_used != kNegInf) ? ex2((m_used - m_new) * l2f) : 1.f;
        if (k > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O must hold every earlier tile before it is rescaled.  P V of this
          // tile cannot start before P is written below, so O's barrier is at
          // most one phase past the one waited for.
          if (!mbar_wait(&bars[kOFull + wg], (t - 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < DV; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(co + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(co + c0, o);
          }
          tmem_wait_st();
        }
        l *= alpha;
        m_used = m_new;
        const float mb = m_used == kNegInf ? 0.f : -m_used * l2f;
        uint32_t pk[32];
        l += exp_pack<false>(x2, l2f, mb, pk);
        tmem_st32(cs, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kPFull + wg]);
      }
      // the item's last P V (phase t - 1) completes O, and every S = Q K^T of
      // this head slot with it
      if (!ok || !mbar_wait(&bars[kOFull + wg], (t - 1) & 1)) bad = true;
      tc_fence_after();
      // The next item's query goes into TMEM first, so its first S = Q K^T
      // runs while this item's O is stored.
      if (preload && !bad) {
        const uint8_t* qs = q_wait(nbase + wg);
        if (!qs) bad = true;
        else load_q(qs, nbase + wg);
      }
      // O / l -> out, through the scratch slot (the tile's 128 rows, 16-byte
      // chunks swizzled by row / 4) so that the global stores are whole rows
      // (16 lanes per 256-byte row).  A bf16 row is DV * 2 bytes; an fp32 row
      // is twice that and goes in two halves of DV / 2 columns, each the size
      // of a bf16 row.
      uint8_t* scr = bad ? nullptr : slot_wait(e_out);
      if (!scr) bad = true;
      // the four warps of the group, once per item: all leave if any thread
      // gave up a wait or another role raised the abort flag
      if (named_barrier_or(bar_id, 128, bad || *s_abort)) break;
      // 1 / normaliser; the optional sink logit (not scaled by the factor)
      // joins it, against l's reference f m_used, and the optional gate's
      // sigmoid scales the row
      float inv;
      {
        float den = l;
        const size_t qi = static_cast<size_t>(it.r0 + r) * p.Hq + h;
        if (p.sink != nullptr && row_ok)
          den += ex2(__ldg(p.sink + qi) * kLog2e - m_used * l2f);  // 0 for a sink of -inf
        inv = den > 0.f ? 1.f / den : 0.f;
        if (p.gate != nullptr && row_ok) inv /= 1.f + ex2(-__ldg(p.gate + qi) * kLog2e);
      }
      constexpr int kCpr = DV / 8;     // 16-byte chunks per scratch row
      constexpr int kRpi = 32 / kCpr;  // rows per store instruction
      constexpr int passes = O32 ? 2 : 1;
#pragma unroll
      for (int half = 0; half < passes; ++half) {
        if (half > 0) named_barrier(bar_id, 128);  // the first half's stores have read the scratch
        constexpr int cw = O32 ? DV / 2 : DV;      // columns of this pass
#pragma unroll 1
        for (int c0 = 0; c0 < cw; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(co + half * cw + c0, o);
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
        // O is read before the next item's first P V overwrites it
        if (half == passes - 1) tc_fence_before();
        named_barrier(bar_id, 128);  // the group's four warps: every row is in the scratch
        // whole-row stores: this warp takes rows [32 q4, 32 q4 + 32)
#pragma unroll
        for (int i = 0; i < kCpr; ++i) {
          const int rr = 32 * q4 + i * kRpi + lane / kCpr;
          const int ch = lane % kCpr;
          const uint4 v =
              *reinterpret_cast<const uint4*>(scr + rr * (DV * 2) + ((ch ^ ((rr >> 2) & 7)) << 4));
          if (rr < it.rows) {
            const size_t orow = (static_cast<size_t>(it.r0 + rr) * p.Hq + h) * DV;
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
      if (lane == 0) mbar_arrive(&bars[kREmpty + ri.slot(e_out)]);
      idx = nidx;
      e_base = nbase;
      it = nit;
      q_loaded = preload;
    }
    if (idx < total) {  // left early: a wait gave up here or in another role
      report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
      *s_abort = 1;
    }
  }
  if (*s_abort && tid == 0) report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
  __syncwarp();  // lanes idle while lane 0 produced/issued rejoin here
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, kTmemCols);
}

// Replays the work split and block walk of prefill_pair_kernel with the same
// device functions (prologue, pair_item, kv_tile) and the same grid: each
// (item, key tile) appends { sequence, first row of its query tile within
// the sequence, key tile, logical block, physical block, first head of the
// item }.
__global__ void __launch_bounds__(128) prefill_walk_kernel(const PrefillParams p) {
  extern __shared__ int seq_arrays[];  // 4 B + 1 ints
  const SeqArrays sa{seq_arrays, seq_arrays + p.B, seq_arrays + 2 * p.B, seq_arrays + 3 * p.B};
  const int total = prologue(p, sa, false) * p.Hkv * ((p.g + 1) >> 1);
  if (threadIdx.x != 0) return;
  for (int idx = blockIdx.x; idx < total; idx += gridDim.x) {
    const PairItem it = pair_item(idx, p, sa);
    const int* trow = p.block_table + static_cast<size_t>(it.b) * p.max_blocks;
    for (int k = 0; k < it.ntiles; ++k) {
      const int tile = it.tf + k;
      const KvTile kt = kv_tile(trow, tile, p.num_blocks);
      const int r = atomicAdd(p.dbg_count, 1);
      if (r < p.dbg_max) {
        int32_t* rec = p.dbg_records + 6 * static_cast<size_t>(r);
        rec[0] = it.b;
        rec[1] = it.r0 - sa.cu0[it.b];
        rec[2] = tile;
        rec[3] = tile >> 1;
        rec[4] = kt.id;
        rec[5] = it.h0;
      }
    }
  }
}

}  // namespace

cudaError_t launch_prefill_walk(const PrefillParams& p, int grid, cudaStream_t stream) {
  const int smem = (4 * p.B + 1) * 4;
  cudaError_t e = ensure_smem<prefill_walk_kernel>(smem);
  if (e != cudaSuccess) return e;
  prefill_walk_kernel<<<grid, 128, smem, stream>>>(p);
  return cudaGetLastError();
}

int prefill_pair_smem_bytes(int B, int dv, int rel_es, int nslots) {
  return PairSmem(B, dv, rel_es, nslots).total + 1024;
}

int prefill_pair_slots(int B, int dv, int rel_es, int smem_optin) {
  for (int ns = kMaxSlots; ns >= kMinSlots; --ns)
    if (prefill_pair_smem_bytes(B, dv, rel_es, ns) <= smem_optin) return ns;
  return 0;
}

template <int DV, bool R16, bool O32>
static cudaError_t launch_pair_as(const PrefillLaunch& L, int grid, int smem, cudaStream_t stream) {
  // The kernel's register split assumes the launch holds kLaunchRegs per
  // thread; with fewer, the softmax warpgroups' raise could never be met.
  static const int regs = [] {
    cudaFuncAttributes a{};
    return cudaFuncGetAttributes(&a, prefill_pair_kernel<DV, R16, O32>) == cudaSuccess
               ? a.numRegs
               : -1;
  }();
  if (regs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  cudaError_t e = ensure_smem<prefill_pair_kernel<DV, R16, O32>>(smem);
  if (e != cudaSuccess) return e;
  prefill_pair_kernel<DV, R16, O32><<<grid, kThreads, smem, stream>>>(L.tm_q, L.tm_k, L.tm_v,
                                                                      L.tm_rel, L.p);
  return cudaGetLastError();
}

template <int DV, bool R16>
static cudaError_t launch_pair_out(const PrefillLaunch& L, int grid, int smem,
                                   cudaStream_t stream) {
  return L.p.out_f32 ? launch_pair_as<DV, R16, true>(L, grid, smem, stream)
                     : launch_pair_as<DV, R16, false>(L, grid, smem, stream);
}

cudaError_t launch_prefill_pair(const PrefillLaunch& L, int grid, cudaStream_t stream) {
  const PrefillParams& p = L.p;
  if (p.kv_es != 2) return cudaErrorInvalidValue;  // bf16 caches only
  const int smem = prefill_pair_smem_bytes(p.B, p.dv, p.rel_es, p.ring_stages);
  const bool r16 = p.rel_es == 2;
  if (p.dv == 128)
    return r16 ? launch_pair_out<128, true>(L, grid, smem, stream)
               : launch_pair_out<128, false>(L, grid, smem, stream);
  return r16 ? launch_pair_out<64, true>(L, grid, smem, stream)
             : launch_pair_out<64, false>(L, grid, smem, stream);
}

}  // namespace relattn
