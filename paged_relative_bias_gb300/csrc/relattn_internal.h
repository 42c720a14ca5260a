// Host <-> kernel interface of the relattn library (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace relattn {

constexpr int kBlockSize = 128;  // tokens per KV block
constexpr int kTileKeys = 64;    // keys per pipeline stage
constexpr int kDqk = 128;
constexpr int kRelBoxW = 68;     // distances per fp32 rel box: 64 keys + 16-byte alignment
constexpr int kRelBoxW16 = 72;   // distances per bf16 rel box: 64 keys + 16-byte alignment

// Distances per decode rel box and its bytes per row, by rel element size.
__host__ __device__ constexpr int rel_box_w(int es) { return es == 2 ? kRelBoxW16 : kRelBoxW; }

struct DecodeParams {
  const __nv_bfloat16* q;      // [B][k][Hq][128]
  const void* rel;             // [B][k][Hq][E], fp32 or bf16 (rel_es bytes)
  const int32_t* block_table;  // [B][max_blocks]
  const int32_t* seq_lens;     // [B]
  void* out;                   // [B][k][Hq][dv], bf16 or fp32 (out_f32)
  const float* sink;           // [B][k][Hq] sink logits, or null
  const float* gate;           // [B][k][Hq] gate logits, or null
  const float* logit_scale;    // [B][k] per-token logit factors, or null
  int rel_es;                  // bytes per rel element: 4 (fp32) or 2 (bf16)
  int out_f32;                 // 1: out is fp32
  int kv_es;                   // bytes per cache element: 2 (bf16) or 1 (e4m3)
  float v_scale;               // e4m3 cache: its value scale (1 for bf16); the key
                               // scale is folded into scale_log2
  uint32_t* status;            // workspace status word
  int32_t* counters;           // [B][Hkv] split-combine arrival counters
  float* part_lse;             // [2*grid][g] base-2 log-sum-exp of a piece
  float* part_o;               // [2*grid][g][dv] normalised output of a piece
  int32_t* dbg_records;        // walk replay only
  int32_t* dbg_count;
  int dbg_max;
  int dbg_wide;                // walk replay: 8-field records (chunk and keys brought)
  int dbg_give_up;             // test hook: > 0 makes the consumer warps of every CTA
                               // treat the query wait of piece dbg_give_up - 1 as given up
  int B, Hq, Hkv, g, dv, max_blocks, num_blocks, window, rel_extent;
  // ceil(2^16 / g): row / g = (row * g_mul) >> 16, exact for the tile rows
  // (row < 32, g <= 16: the error row * (g_mul g - 2^16) / (g 2^16) < 1 / g)
  uint32_t g_mul;
  // query tokens per sequence (k; 1 for plain decode), packed kpc at a time
  // with the g heads into the rows of one tile: nck = ceil(k / kpc) chunks
  // per sequence, Bv = B * nck chunks ("virtual sequences") in all
  int k, kpc, nck, Bv;
  int nstages;  // even unless rows are split: see the consumer groups of decode_kernel
  float scale_log2;  // log2(e) / sqrt(d_qk)
  int rs;            // 1: chunks of up to 32 rows, split between the consumer groups
};

// Raise kernel K's dynamic shared-memory limit to `smem` bytes on the current
// device, calling the runtime only the first time (or for a larger size):
// one attribute call per launch is host time every call would pay.
template <auto K>
cudaError_t ensure_smem(int smem) {
  constexpr int kDevices = 64;
  static std::atomic<int> set[kDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kDevices && set[dev].load(std::memory_order_relaxed) >= smem)
    return cudaSuccess;
  e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && dev >= 0 && dev < kDevices) {
    int cur = set[dev].load(std::memory_order_relaxed);
    while (cur < smem && !set[dev].compare_exchange_weak(cur, smem)) {
    }
  }
  return e;
}

struct DecodeLaunch {
  CUtensorMap tm_q, tm_k, tm_v, tm_rel;
  CUtensorMap tm_kh, tm_vh;  // K and V boxes of half a tile (32 keys)
  DecodeParams p;
  int grid;
};

struct PrefillParams {
  const __nv_bfloat16* q;      // [T][Hq][128]
  const __nv_bfloat16* k;      // [T][Hkv][128]
  const __nv_bfloat16* v;      // [T][Hkv][dv]
  const void* rel;             // [T][Hq][E], fp32 or bf16 (rel_es bytes)
  const int32_t* cu_seqlens;   // [B+1]
  const int32_t* ctx_lens;     // [B]
  const int32_t* block_table;  // [B][max_blocks]
  __nv_bfloat16* k_cache;      // [NB][128][Hkv][128] (e4m3 caches: uint8 [NB][Hkv][128][128])
  __nv_bfloat16* v_cache;      // [NB][128][Hkv][dv]
  void* out;                   // [T][Hq][dv], bf16 or fp32 (out_f32)
  const float* sink;           // [T][Hq] sink logits, or null
  const float* gate;           // [T][Hq] gate logits, or null
  const float* logit_scale;    // [T] per-token logit factors, or null
  int rel_es;                  // bytes per rel element: 4 (fp32) or 2 (bf16)
  int out_f32;                 // 1: out is fp32
  uint32_t* status;
  int32_t* dbg_records;
  int32_t* dbg_count;
  int dbg_max;
  int B, T, Hq, Hkv, g, dv, max_blocks, num_blocks, window, rel_extent, max_q_len;
  int ring_stages;  // depth of the query/rel/scratch ring (2 or 3, as shared memory allows)
  float scale_log2;
  // cache write into an e4m3 cache (kv_es = 1): code = e4m3(x / scale)
  int kv_es;
  float k_scale, v_scale;
};

struct PrefillLaunch {
  CUtensorMap tm_q, tm_k, tm_v, tm_rel;
  CUtensorMap tm_out;  // out as [T][Hq][d_v] boxes of 128 B x 128 rows (the 128-key-tile kernel)
  PrefillParams p;
  int grid;
  int pair;  // 1: the two-heads-per-item kernel (bf16 caches), 0: one head per item
  int wide;  // 1: one head per item over 128-key tiles (bf16 cache and rel, d_v = 128)
};

int decode_smem_bytes(int nstages, int B, int Bv, int kpc, int g, int dv, int rel_es, int kv_es);
constexpr int kMaxDecodeRows = 16;         // rows of one decode tile: g heads x tokens
constexpr int kMaxChunkRows = 32;          // rows of one chunk (two tiles' rows when split)
// The general kernel splits a chunk's rows between its two consumer groups
// when more tokens than one 16-row tile holds share a KV head (g <= 8).
inline bool decode_row_split(int k, int g) { return g <= 8 && k * g > kMaxDecodeRows; }
// The decode kernel has a one-token instantiation for tiles of at most 8 rows
// and a general one (several tokens, or g > 8), which also takes its query
// rows through a 3-D copy.
inline bool decode_multi_kernel(int k, int g) { return k > 1 || g > 8; }
constexpr int kMaxQueryTokens = 16;        // query tokens per sequence in one decode call
cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t stream);
cudaError_t launch_decode_walk(const DecodeParams& p, int grid, cudaStream_t stream);

cudaError_t launch_cache_write(const PrefillParams& p, cudaStream_t stream);
cudaError_t launch_wait_timeout(uint32_t* status, cudaStream_t stream);
constexpr int kCacheWriteMaxGridY = 65535;  // sequences of one cache-write launch
int prefill_smem_bytes(int B, int dv, int ring_stages, int kv_es);
int prefill_ring_stages(int B, int dv, int kv_es, int smem_optin);  // 0 if nothing fits
cudaError_t launch_prefill(const PrefillLaunch& L, int grid, cudaStream_t stream);
// Replay of the bf16-cache prefill's work split and block walk on its grid.
cudaError_t launch_prefill_walk(const PrefillParams& p, int grid, cudaStream_t stream);
// The bf16-cache prefill with two query heads of one KV group per work item:
// its ring slots for these sizes (0 if fewer than it needs fit), its shared
// memory, and its launch (p.ring_stages = the slots).
int prefill_pair_slots(int B, int dv, int rel_es, int smem_optin);
int prefill_pair_smem_bytes(int B, int dv, int rel_es, int nslots);
cudaError_t launch_prefill_pair(const PrefillLaunch& L, int grid, cudaStream_t stream);
// The bf16-cache, bf16-rel prefill (d_v = 128) with one head per work item and
// 128-key tiles: ring slots (0 if fewer than it needs fit), shared memory,
// launch (p.ring_stages = the slots; K/V maps with 128-row boxes, rel boxes of
// 32 rows x 200 distances, the odd boxes starting 32 distances lower).
int prefill_wide_slots(int B, int smem_optin);
int prefill_wide_smem_bytes(int B, int nslots);
cudaError_t launch_prefill_wide(const PrefillLaunch& L, int grid, cudaStream_t stream);
// Replay of that kernel's work split and block walk on its grid.
cudaError_t launch_prefill_wide_walk(const PrefillParams& p, int grid, cudaStream_t stream);

}  // namespace relattn
