// Device helpers shared by the relattn kernels: inline PTX for mbarriers,
// TMA, ldmatrix and mma.sync, bounded waits, and the window-aware block walk.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/relattn.h"
#include "relattn_internal.h"

namespace relattn {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// ---------------------------------------------------------------------------
// small utilities
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The dynamic shared-memory array rounded up to 1024 bytes.  The offset is
// added to the array itself, so the compiler still knows the pointer is in
// shared memory (rounding the address as an integer would leave generic
// loads and stores on every access through it).
__device__ __forceinline__ uint8_t* smem_align1024(uint8_t* raw) {
  return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// bf16 pair -> f16 pair (exact for the magnitudes of attention inputs)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const __half2 h = __floats2half2_rn(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Either f16 of a pair is infinite or NaN: a query element narrowed to f16
// that did not fit its range (or was not finite to begin with).
__device__ __forceinline__ bool f16x2_nonfinite(uint32_t h) {
  return (h & 0x7c00u) == 0x7c00u || (h & 0x7c000000u) == 0x7c000000u;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Four e4m3 values (one 32-bit word, low byte first) -> two f16 pairs: bytes
// 0-1 in lo, bytes 2-3 in hi.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(four));
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Arrive at a named barrier without waiting (the producer side of a
// hand-off to warps that wait with named_barrier on the same id and count).
// Named barrier that also ORs a predicate over its threads: every thread
// gets the same answer, so they can all take the same branch after it.
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void named_barrier_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch.  launch_dependents lets the next kernel on
// the stream (launched with programmatic stream serialisation) start once
// every CTA of this grid has issued it; grid_dep_wait blocks until the grids
// this one depends on have completed and their memory is visible.  Both are
// no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void report(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// Entry e of a ring of n slots: slot e mod n and phase (e / n) & 1, by a
// multiply-high with the rounded-up reciprocal of n (exact for 0 <= e <
// 2^32 / n).  A division by a run-time value would put hundreds of cycles on
// a consumer's path at every ring wait.
struct RingIndex {
  uint32_t n, inv;
  __device__ explicit RingIndex(int slots)
      : n(static_cast<uint32_t>(slots)),
        inv(static_cast<uint32_t>((0x100000000ull + slots - 1) / slots)) {}
  __device__ __forceinline__ uint32_t quot(int e) const {
    return __umulhi(static_cast<uint32_t>(e), inv);
  }
  __device__ __forceinline__ int slot(int e) const {
    return static_cast<int>(static_cast<uint32_t>(e) - quot(e) * n);
  }
  __device__ __forceinline__ uint32_t phase(int e) const { return quot(e) & 1u; }
};

// ---- paired fp32 arithmetic (sm_100 family) --------------------------------
// Two fp32 lanes in one 64-bit register pair: one instruction does two FMAs
// or adds, which halves the issue slots of a softmax.  (Scalar FFMA
// streams on other warps slow the tensor pipe's MMAs; the paired form at the
// same FLOP rate does not.)  Each lane rounds exactly as the scalar op does.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ uint64_t f2u(uint32_t lo, uint32_t hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
  return d;
}
__device__ __forceinline__ float f2lo(uint64_t v) {
  return __uint_as_float(static_cast<uint32_t>(v));
}
__device__ __forceinline__ float f2hi(uint64_t v) {
  return __uint_as_float(static_cast<uint32_t>(v >> 32));
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// c + the bf16 in the high (HI) or low half of w, rounded once to fp32 (a
// mixed-precision add: the bf16 operand is read as it is, with no widening
// instruction)
template <bool HI>
__device__ __forceinline__ float add_bf16_f32(uint32_t w, float c) {
  float d;
  if constexpr (HI)
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n add.rn.f32.bf16 %0, h, %2;\n}"
        : "=f"(d) : "r"(w), "f"(c));
  else
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n add.rn.f32.bf16 %0, l, %2;\n}"
        : "=f"(d) : "r"(w), "f"(c));
  return d;
}
// max of three (one instruction)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later TMA
// (async-proxy) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity; false after ~2 s.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---------------------------------------------------------------------------
// TMA (tiled tensor copies, global -> shared, completing on an mbarrier)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m))
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m,
                                            uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// Tensor store shared -> global (bulk async group of the issuing thread):
// the box at `src` goes to the coordinates given; rows past the tensor's
// extent are not written.  commit / wait_read / wait_all as in the PTX
// bulk-group model: wait_read returns once the shared source may be reused,
// wait_all once the global writes are done.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m,
                                            uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1),
      "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m,
                                            uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1),
      "r"(c2), "r"(c3)
      : "memory");
}

// ---------------------------------------------------------------------------
// warp-level tensor core ops (bf16 in, fp32 accumulate)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0,
                                        uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}

// Two 8x8 matrices; lanes 0-15 give the row addresses.
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

// Transpose of an 8x8 matrix of 16-bit elements held as one register per
// lane (lane t: row t/4, columns 2 (t%4) and 2 (t%4) + 1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0,
                                          uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D
// The same with f16 operands.
__device__ __forceinline__ void mma_16816_f16(float* d, const uint32_t* a, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a TMA box
// written with 128-byte swizzling (rows of 128 bytes, 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------------------
// window-aware block walk
// ---------------------------------------------------------------------------

// Keys of a query at position P: [lo, P]; W keys counting its own on a
// sliding-window layer ("Inkling-Small on Gaudi 2", section "Decode window").
__device__ __forceinline__ int window_lo(int P, int window) {
  return window > 0 ? max(0, P - window + 1) : 0;
}

// One decode sequence: its query position and the range of 64-key tiles that
// hold a visible key.  Tiles outside [lo, p] are never fetched, so a local
// layer reads at most ceil(W/128)+1 blocks.
struct DecodeSeq {
  int p;           // query position
  int lo;          // first visible key
  int tile_first;  // lo / 64
  int ntiles;      // 0 if the length is invalid
};

__device__ __forceinline__ DecodeSeq decode_seq(int seq_len, int window,
                                                int max_blocks) {
  DecodeSeq s;
  if (seq_len < 1 || seq_len > max_blocks * kBlockSize) {
    s.p = s.lo = s.tile_first = s.ntiles = 0;
    return s;
  }
  s.p = seq_len - 1;
  s.lo = window_lo(s.p, window);
  s.tile_first = s.lo / kTileKeys;
  s.ntiles = s.p / kTileKeys - s.tile_first + 1;
  return s;
}

}  // namespace relattn
