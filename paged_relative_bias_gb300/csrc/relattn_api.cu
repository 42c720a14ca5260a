// Host side of the relattn C ABI: argument validation, workspace layout,
// TMA descriptors and kernel launches.  Nothing here reads device memory
// (except relattn_read_status), so every call can be captured in a graph.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/relattn.h"
#include "relattn_internal.h"

namespace relattn {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxStages = 6;       // bf16 cache: 32 KB per stage
constexpr int kMaxStagesE4m3 = 12;  // e4m3 cache: 16 KB per stage
constexpr int kMaxDecodeGrid = 46340;  // grid^2 < 2^31
constexpr size_t kStatusBytes = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_dev[dev].sms == 0) {
    int sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return false;
    if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
      return false;
    g_dev[dev].sms = sms;
    g_dev[dev].smem_optin = smem;
  }
  *out = g_dev[dev];
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

// Tiled map over a row-major tensor; dims/box innermost first.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, void* base,
              const cuuint64_t* dims, const cuuint64_t* strides_bytes,
              const cuuint32_t* box, CUtensorMapSwizzle swz) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, dt, rank, base, dims, strides_bytes, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool cache_maps(const relattn_kv_cache* c, int box_rows, CUtensorMap* tk, CUtensorMap* tv) {
  const cuuint64_t rows = static_cast<cuuint64_t>(c->num_blocks) * c->block_size;
  const cuuint64_t kd[3] = {static_cast<cuuint64_t>(c->d_qk),
                            static_cast<cuuint64_t>(c->num_kv_heads), rows};
  const cuuint64_t ks[2] = {static_cast<cuuint64_t>(c->d_qk) * 2,
                            static_cast<cuuint64_t>(c->num_kv_heads) * c->d_qk * 2};
  const cuuint64_t vd[3] = {static_cast<cuuint64_t>(c->d_v),
                            static_cast<cuuint64_t>(c->num_kv_heads), rows};
  const cuuint64_t vs[2] = {static_cast<cuuint64_t>(c->d_v) * 2,
                            static_cast<cuuint64_t>(c->num_kv_heads) * c->d_v * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  return make_map(tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c->k, kd, ks, box,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c->v, vd, vs, box,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

// Decode's K/V maps: one TMA copy brings a whole 64-key tile of one KV head.
// The 4-D view (64 columns, cache row, 64-column half, head) puts the halves
// outermost in the box, so shared memory receives [half][64 rows][128 B], the
// same 128-byte-swizzled halves as two 3-D copies would.
// box_rows = kTileKeys: a whole tile, both 64-column halves in one box.
// box_rows = kTileKeys / 2: half a tile, one 64-column half per box (so that
// it lands where it would in a whole tile).
bool decode_cache_maps(const relattn_kv_cache* c, int box_rows, CUtensorMap* tk,
                       CUtensorMap* tv) {
  const bool whole = box_rows == kTileKeys;
  const cuuint64_t rows = static_cast<cuuint64_t>(c->num_blocks) * c->block_size;
  const cuuint64_t hkv = static_cast<cuuint64_t>(c->num_kv_heads);
  const cuuint64_t kd[4] = {64, rows, static_cast<cuuint64_t>(c->d_qk / 64), hkv};
  const cuuint64_t ks[3] = {hkv * c->d_qk * 2, 128, static_cast<cuuint64_t>(c->d_qk) * 2};
  const cuuint32_t kb[4] = {64, static_cast<cuuint32_t>(box_rows),
                            whole ? static_cast<cuuint32_t>(c->d_qk / 64) : 1u, 1};
  const cuuint64_t vd[4] = {64, rows, static_cast<cuuint64_t>(c->d_v / 64), hkv};
  const cuuint64_t vs[3] = {hkv * c->d_v * 2, 128, static_cast<cuuint64_t>(c->d_v) * 2};
  const cuuint32_t vb[4] = {64, static_cast<cuuint32_t>(box_rows),
                            whole ? static_cast<cuuint32_t>(c->d_v / 64) : 1u, 1};
  return make_map(tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, c->k, kd, ks, kb,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, c->v, vd, vs, vb,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

// e4m3 caches are head-major, [NB][Hkv][128][d]: a token's head row is only
// 128 bytes, and this keeps a block's 128 rows of one head contiguous.  As a
// 2-D tensor of rows (block * Hkv + head) * 128 + slot, a 64-key tile is one
// 8 KB box, landing as 64 rows x 128 bytes with the 128-byte swizzle (or
// half of one, box_rows = 32).
bool decode_cache_maps_e4m3(const relattn_kv_cache* c, int box_rows, CUtensorMap* tk,
                            CUtensorMap* tv) {
  const cuuint64_t rows =
      static_cast<cuuint64_t>(c->num_blocks) * c->num_kv_heads * c->block_size;
  const cuuint64_t kd[2] = {static_cast<cuuint64_t>(c->d_qk), rows};
  const cuuint64_t ks[1] = {static_cast<cuuint64_t>(c->d_qk)};
  const cuuint32_t kb[2] = {static_cast<cuuint32_t>(c->d_qk), static_cast<cuuint32_t>(box_rows)};
  const cuuint64_t vd[2] = {static_cast<cuuint64_t>(c->d_v), rows};
  const cuuint64_t vs[1] = {static_cast<cuuint64_t>(c->d_v)};
  const cuuint32_t vb[2] = {static_cast<cuuint32_t>(c->d_v), static_cast<cuuint32_t>(box_rows)};
  return make_map(tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c->k, kd, ks, kb,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c->v, vd, vs, vb,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

int check_cache(const relattn_kv_cache* c) {
  if (!c || !c->k || !c->v) return RELATTN_ERR_INVALID_ARG;
  if (!aligned16(c->k) || !aligned16(c->v)) return RELATTN_ERR_INVALID_ARG;
  if (c->num_blocks < 1 || c->num_kv_heads < 1) return RELATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(c->num_blocks) * 128 > 0x7fffffffLL) return RELATTN_ERR_UNSUPPORTED;
  if (c->block_size != 128 || c->d_qk != 128) return RELATTN_ERR_UNSUPPORTED;
  if (c->d_v != 64 && c->d_v != 128) return RELATTN_ERR_UNSUPPORTED;
  return RELATTN_OK;
}

int check_dims(const relattn_dims* d, const relattn_kv_cache* c) {
  if (!d) return RELATTN_ERR_INVALID_ARG;
  if (d->batch < 1 || d->num_q_heads < 1 || d->max_blocks_per_seq < 1 || d->num_ctas < 0)
    return RELATTN_ERR_INVALID_ARG;
  if (d->num_q_heads % c->num_kv_heads != 0) return RELATTN_ERR_INVALID_ARG;
  if (d->num_q_heads / c->num_kv_heads > 16) return RELATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->max_blocks_per_seq) * 128 > 0x7fffffffLL)
    return RELATTN_ERR_UNSUPPORTED;
  return RELATTN_OK;
}

struct WsLayout {
  size_t counters, lse, part, total;
};

// Decode workspace, sized for any query-token count up to kMaxQueryTokens:
// counters per (chunk, KV head) -- at most kMaxQueryTokens chunks per
// sequence -- and two partial slots per CTA of kMaxChunkRows rows each.
WsLayout ws_layout(const relattn_dims* d, const relattn_kv_cache* c, int grid) {
  WsLayout w;
  w.counters = kStatusBytes;
  w.lse = w.counters + round_up(static_cast<size_t>(d->batch) * kMaxQueryTokens *
                                    c->num_kv_heads * 4, 256);
  w.part = w.lse + round_up(static_cast<size_t>(2) * grid * kMaxChunkRows * 4, 256);
  w.total = w.part + static_cast<size_t>(2) * grid * kMaxChunkRows * c->d_v * 4;
  return w;
}

int decode_grid(const relattn_dims* d, const DeviceInfo& di) {
  return d->num_ctas > 0 ? d->num_ctas : di.sms;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? RELATTN_OK : RELATTN_ERR_CUDA; }

}  // namespace
}  // namespace relattn

using namespace relattn;

extern "C" {

int relattn_abi_version(void) { return 100; }

const char* relattn_status_string(int code) {
  switch (code) {
    case RELATTN_OK: return "ok";
    case RELATTN_ERR_INVALID_ARG: return "invalid argument";
    case RELATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case RELATTN_ERR_WORKSPACE: return "workspace too small";
    case RELATTN_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

size_t relattn_workspace_size(const relattn_dims* dims, const relattn_kv_cache* cache) {
  if (check_cache(cache) != RELATTN_OK || check_dims(dims, cache) != RELATTN_OK) return 0;
  DeviceInfo di;
  if (!device_info(&di)) return 0;
  return ws_layout(dims, cache, decode_grid(dims, di)).total;
}

int relattn_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (!workspace || bytes < kStatusBytes) return RELATTN_ERR_INVALID_ARG;
  return to_status(cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)));
}

int relattn_read_status(const void* workspace, uint32_t* status, void* stream) {
  if (!workspace || !status) return RELATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(status, workspace, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return to_status(e);
}

// kq: query tokens per sequence (1 for relattn_decode).
// The call options as the kernels see them.
struct IoTypes {
  int rel_es;         // bytes per rel element: 4 (fp32) or 2 (bf16)
  int out_f32;        // 1: out is fp32, 0: bf16
  const float* sink;  // per (query row, head) sink logits, or null
  const float* gate;  // per (query row, head) gate logits, or null
  int kv_es;          // bytes per cache element: 2 (bf16) or 1 (e4m3)
  float k_scale, v_scale;
  const float* logit_scale;  // per query token logit factors, or null
};
constexpr IoTypes kDefaultIo = {4, 0, nullptr, nullptr, 2, 1.f, 1.f, nullptr};

// From the C ABI's options; false for a value that is not offered (an
// unknown type code, or a sink / gate / logit_scale pointer not 4-byte
// aligned).
static bool io_types(const relattn_options* t, IoTypes* io) {
  if (!t) return false;
  if (t->rel != RELATTN_DTYPE_F32 && t->rel != RELATTN_DTYPE_BF16) return false;
  if (t->out != RELATTN_DTYPE_F32 && t->out != RELATTN_DTYPE_BF16) return false;
  if ((reinterpret_cast<uintptr_t>(t->sink) & 3u) || (reinterpret_cast<uintptr_t>(t->gate) & 3u) ||
      (reinterpret_cast<uintptr_t>(t->logit_scale) & 3u))
    return false;
  io->rel_es = t->rel == RELATTN_DTYPE_BF16 ? 2 : 4;
  io->out_f32 = t->out == RELATTN_DTYPE_F32 ? 1 : 0;
  io->sink = t->sink;
  io->gate = t->gate;
  io->logit_scale = t->logit_scale;
  if (t->kv == 0 || t->kv == RELATTN_DTYPE_BF16) {
    io->kv_es = 2;
    io->k_scale = io->v_scale = 1.f;
  } else if (t->kv == RELATTN_DTYPE_E4M3) {
    const auto ok = [](float x) { return x > 0.f && x < 3.0e38f; };  // finite, positive
    if (!ok(t->k_scale) || !ok(t->v_scale)) return false;
    io->kv_es = 1;
    io->k_scale = t->k_scale;
    io->v_scale = t->v_scale;
  } else {
    return false;
  }
  return true;
}

// rel rows are TMA rows of rel_extent elements: 16-byte multiples, at least
// one 16-byte unit.
static bool rel_extent_ok(int32_t rel_extent, int es) {
  const int unit = 16 / es;
  return rel_extent >= unit && rel_extent % unit == 0;
}

static int prepare_decode(const void* q, const void* rel, IoTypes io,
                          const relattn_kv_cache* cache,
                          const int32_t* block_table, const int32_t* seq_lens, int32_t kq,
                          int32_t window, int32_t rel_extent, const relattn_dims* dims,
                          void* out, void* workspace, size_t ws_bytes, bool walk,
                          DecodeLaunch* L, DeviceInfo* di) {
  int rc = check_cache(cache);
  if (rc != RELATTN_OK) return rc;
  rc = check_dims(dims, cache);
  if (rc != RELATTN_OK) return rc;
  if (!block_table || !seq_lens || !workspace) return RELATTN_ERR_INVALID_ARG;
  if (!walk) {
    if (!q || !rel || !out) return RELATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(rel) || !aligned16(out)) return RELATTN_ERR_INVALID_ARG;
    if (!rel_extent_ok(rel_extent, io.rel_es)) return RELATTN_ERR_UNSUPPORTED;
  }
  if (!aligned16(workspace)) return RELATTN_ERR_INVALID_ARG;
  if (!device_info(di)) return RELATTN_ERR_CUDA;
  const int grid = decode_grid(dims, *di);
  if (kq < 1 || kq > kMaxQueryTokens) return RELATTN_ERR_UNSUPPORTED;
  const int gq = dims->num_q_heads / cache->num_kv_heads;
  // an e4m3 cache: d_v = 128, and 32-bit head-major row coordinates
  if (io.kv_es == 1 && (cache->d_v != 128 ||
                        static_cast<long long>(cache->num_blocks) * cache->num_kv_heads * 128 >
                            0x7fffffffLL))
    return RELATTN_ERR_UNSUPPORTED;
  // tokens per chunk: a 16-row tile's worth, or 32 rows split between the
  // consumer groups when more tokens than that share a KV head
  const bool split = decode_multi_kernel(kq, gq) && decode_row_split(kq, gq);
  const int crow = split ? kMaxChunkRows : kMaxDecodeRows;
  const int kpc = kq < crow / gq ? kq : crow / gq;
  const int nck = (kq + kpc - 1) / kpc;
  // the kernel's work split is 32-bit: all tiles < 2^31, grid^2 < 2^31
  if (static_cast<long long>(dims->batch) * nck * cache->num_kv_heads * 2 *
              dims->max_blocks_per_seq >= (1LL << 31) ||
      grid > kMaxDecodeGrid)
    return RELATTN_ERR_UNSUPPORTED;
  const WsLayout w = ws_layout(dims, cache, grid);
  if (ws_bytes < w.total) return RELATTN_ERR_WORKSPACE;
  const int g = dims->num_q_heads / cache->num_kv_heads;
  std::memset(L, 0, sizeof(*L));
  DecodeParams& p = L->p;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.rel = rel;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.sink = io.sink;
  p.gate = io.gate;
  p.logit_scale = io.logit_scale;
  p.rel_es = io.rel_es;
  p.out_f32 = io.out_f32;
  p.kv_es = io.kv_es;
  p.v_scale = io.v_scale;
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.counters = reinterpret_cast<int32_t*>(ws + w.counters);
  p.part_lse = reinterpret_cast<float*>(ws + w.lse);
  p.part_o = reinterpret_cast<float*>(ws + w.part);
  p.B = dims->batch;
  p.Hq = dims->num_q_heads;
  p.Hkv = cache->num_kv_heads;
  p.g = g;
  p.g_mul = static_cast<uint32_t>((65536 + g - 1) / g);
  p.dv = cache->d_v;
  p.max_blocks = dims->max_blocks_per_seq;
  p.num_blocks = cache->num_blocks;
  p.window = window;
  p.rel_extent = rel_extent;
  p.k = kq;
  p.kpc = kpc;
  p.nck = nck;
  p.Bv = dims->batch * nck;
  // log2(e) / sqrt(d_qk), times the key scale of an e4m3 cache
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(128.0) * io.k_scale);
  L->grid = grid;
  if (walk) {
    p.nstages = 0;
    return RELATTN_OK;
  }
  // An even number of stages: the decode kernel's two consumer groups each
  // own every other stage (any number when they split the rows and both
  // take every stage).
  p.rs = split ? 1 : 0;
  p.nstages = io.kv_es == 1 ? kMaxStagesE4m3 : kMaxStages;
  while (p.nstages >= 2 &&
         decode_smem_bytes(p.nstages, p.B, p.Bv, p.kpc, p.g, p.dv, p.rel_es, p.kv_es) >
             di->smem_optin)
    p.nstages -= split ? 1 : 2;
  if (p.nstages < 2) return RELATTN_ERR_UNSUPPORTED;  // batch too large for shared memory
  // whole tiles, and (one-token kernel, bf16 cache) half tiles for the edges
  // of a sequence's key range
  const bool halves = p.kv_es == 2 && !decode_multi_kernel(kq, gq);
  if (!(p.kv_es == 1 ? decode_cache_maps_e4m3(cache, kTileKeys, &L->tm_k, &L->tm_v)
                     : decode_cache_maps(cache, kTileKeys, &L->tm_k, &L->tm_v)) ||
      (halves && !decode_cache_maps(cache, kTileKeys / 2, &L->tm_kh, &L->tm_vh)))
    return RELATTN_ERR_CUDA;
  // rel [B][k][Hq][E] fp32 or bf16: boxes of one token's g heads x
  // rel_box_w distances
  const cuuint64_t rd[2] = {static_cast<cuuint64_t>(rel_extent),
                            static_cast<cuuint64_t>(dims->batch) * kq * dims->num_q_heads};
  const cuuint64_t rs[1] = {static_cast<cuuint64_t>(rel_extent) * io.rel_es};
  const cuuint32_t rb[2] = {static_cast<cuuint32_t>(rel_box_w(io.rel_es)),
                            static_cast<cuuint32_t>(g)};
  if (!make_map(&L->tm_rel,
                io.rel_es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                2, const_cast<void*>(rel), rd, rs, rb, CU_TENSOR_MAP_SWIZZLE_NONE))
    return RELATTN_ERR_CUDA;
  // query rows of one chunk: q [B*k][Hq][128] bf16 as (column, head, token);
  // a box is one 64-column half of kpc tokens x g heads (rows token * g + head).
  // The one-token kernel (g <= 8): the 2-D view [B*Hq][128] and a box of the
  // group's g rows.
  const cuuint64_t qd[3] = {128, static_cast<cuuint64_t>(dims->num_q_heads),
                            static_cast<cuuint64_t>(dims->batch) * kq};
  const cuuint64_t qs[2] = {256, static_cast<cuuint64_t>(dims->num_q_heads) * 256};
  const cuuint32_t qbx[3] = {64, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(kpc)};
  const cuuint64_t qd1[2] = {128, static_cast<cuuint64_t>(dims->batch) * dims->num_q_heads};
  const bool q3 = decode_multi_kernel(kq, g);
  if (!(q3 ? make_map(&L->tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), qd, qs,
                      qbx, CU_TENSOR_MAP_SWIZZLE_128B)
           : make_map(&L->tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), qd1,
                      qs, qbx, CU_TENSOR_MAP_SWIZZLE_128B)))
    return RELATTN_ERR_CUDA;
  return RELATTN_OK;
}

int relattn_decode(const void* q, const float* rel, const relattn_kv_cache* kv_cache,
                   const int32_t* block_table, const int32_t* seq_lens, int32_t window,
                   int32_t rel_extent, const relattn_dims* dims, void* out, void* workspace,
                   size_t workspace_bytes, void* stream) {
  DecodeLaunch L;
  DeviceInfo di;
  const int rc = prepare_decode(q, rel, kDefaultIo, kv_cache, block_table, seq_lens, 1, window,
                                rel_extent, dims, out, workspace, workspace_bytes, false, &L, &di);
  if (rc != RELATTN_OK) return rc;
  return to_status(launch_decode(L, static_cast<cudaStream_t>(stream)));
}

int relattn_decode_multi(const void* q, const float* rel, const relattn_kv_cache* kv_cache,
                         const int32_t* block_table, const int32_t* seq_lens,
                         int32_t num_query_tokens, int32_t window, int32_t rel_extent,
                         const relattn_dims* dims, void* out, void* workspace,
                         size_t workspace_bytes, void* stream) {
  DecodeLaunch L;
  DeviceInfo di;
  const int rc = prepare_decode(q, rel, kDefaultIo, kv_cache, block_table, seq_lens,
                                num_query_tokens, window, rel_extent, dims, out, workspace,
                                workspace_bytes, false, &L, &di);
  if (rc != RELATTN_OK) return rc;
  return to_status(launch_decode(L, static_cast<cudaStream_t>(stream)));
}

int relattn_decode_ex(const void* q, const void* rel, const relattn_options* options,
                      const relattn_kv_cache* kv_cache, const int32_t* block_table,
                      const int32_t* seq_lens, int32_t num_query_tokens, int32_t window,
                      int32_t rel_extent, const relattn_dims* dims, void* out, void* workspace,
                      size_t workspace_bytes, void* stream) {
  IoTypes io;
  if (!io_types(options, &io)) return RELATTN_ERR_INVALID_ARG;
  DecodeLaunch L;
  DeviceInfo di;
  const int rc = prepare_decode(q, rel, io, kv_cache, block_table, seq_lens, num_query_tokens,
                                window, rel_extent, dims, out, workspace, workspace_bytes, false,
                                &L, &di);
  if (rc != RELATTN_OK) return rc;
  return to_status(launch_decode(L, static_cast<cudaStream_t>(stream)));
}

int relattn_debug_decode_give_up(const void* q, const float* rel,
                                 const relattn_kv_cache* kv_cache, const int32_t* block_table,
                                 const int32_t* seq_lens, int32_t window, int32_t rel_extent,
                                 const relattn_dims* dims, void* out, void* workspace,
                                 size_t workspace_bytes, int32_t piece, void* stream) {
  if (piece < 0) return RELATTN_ERR_INVALID_ARG;
  DecodeLaunch L;
  DeviceInfo di;
  const int rc = prepare_decode(q, rel, kDefaultIo, kv_cache, block_table, seq_lens, 1, window,
                                rel_extent, dims, out, workspace, workspace_bytes, false, &L, &di);
  if (rc != RELATTN_OK) return rc;
  L.p.dbg_give_up = piece + 1;
  return to_status(launch_decode(L, static_cast<cudaStream_t>(stream)));
}

int relattn_debug_walk_decode(const int32_t* block_table, const int32_t* seq_lens,
                              int32_t window, const relattn_kv_cache* cache,
                              const relattn_dims* dims, int32_t* records, int32_t max_records,
                              int32_t* count, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (!records || !count || max_records < 0) return RELATTN_ERR_INVALID_ARG;
  DecodeLaunch L;
  DeviceInfo di;
  const int rc = prepare_decode(nullptr, nullptr, kDefaultIo, cache, block_table, seq_lens, 1,
                                window, 4, dims,
                                nullptr, workspace, workspace_bytes, true, &L, &di);
  if (rc != RELATTN_OK) return rc;
  L.p.dbg_records = records;
  L.p.dbg_count = count;
  L.p.dbg_max = max_records;
  return to_status(launch_decode_walk(L.p, L.grid, static_cast<cudaStream_t>(stream)));
}

int relattn_debug_walk_decode_ex(const int32_t* block_table, const int32_t* seq_lens,
                                 int32_t num_query_tokens, int32_t window,
                                 const relattn_options* options, const relattn_kv_cache* cache,
                                 const relattn_dims* dims, int32_t* records,
                                 int32_t max_records, int32_t* count, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (!records || !count || max_records < 0) return RELATTN_ERR_INVALID_ARG;
  IoTypes io = kDefaultIo;
  if (options && !io_types(options, &io)) return RELATTN_ERR_INVALID_ARG;
  DecodeLaunch L;
  DeviceInfo di;
  const int rc = prepare_decode(nullptr, nullptr, io, cache, block_table, seq_lens,
                                num_query_tokens, window, 4, dims, nullptr, workspace,
                                workspace_bytes, true, &L, &di);
  if (rc != RELATTN_OK) return rc;
  L.p.dbg_records = records;
  L.p.dbg_count = count;
  L.p.dbg_max = max_records;
  L.p.dbg_wide = 1;
  return to_status(launch_decode_walk(L.p, L.grid, static_cast<cudaStream_t>(stream)));
}

// ---- decode with library-owned scratch ----------------------------------
// For callers that may not allocate device memory (their host owns every
// buffer, or cannot pay for an allocation on the decode path): the split
// state that relattn_decode keeps in the caller's workspace lives here, in
// one array that every GPU loading this library holds until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[RELATTN_NOALLOC_SCRATCH_BYTES];
static void* g_noalloc_addr[kMaxDevices];  // device address of the array, per device

// The device address of the scratch array on the current device.  In host
// code the array's name is only a host-side stand-in, so the address is asked
// from the runtime once per device (with that device current) and cached.
static int noalloc_scratch(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RELATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_noalloc_addr[dev]) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess || !a) return RELATTN_ERR_CUDA;
    g_noalloc_addr[dev] = a;
  }
  *addr = g_noalloc_addr[dev];
  return RELATTN_OK;
}

int relattn_decode_noalloc_status(uint32_t* status, void* stream) {
  if (!status) return RELATTN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != RELATTN_OK) return rc;
  return relattn_read_status(scratch, status, stream);  // the array starts with the status word
}

int relattn_decode_noalloc(const void* q, const float* rel, const relattn_kv_cache* kv_cache,
                           const int32_t* block_table, const int32_t* seq_lens, int32_t window,
                           int32_t rel_extent, const relattn_dims* dims, void* out,
                           void* stream) {
  int rc = check_cache(kv_cache);
  if (rc != RELATTN_OK) return rc;
  rc = check_dims(dims, kv_cache);
  if (rc != RELATTN_OK) return rc;
  DeviceInfo di;
  if (!device_info(&di)) return RELATTN_ERR_CUDA;
  const WsLayout w = ws_layout(dims, kv_cache, decode_grid(dims, di));
  if (w.total > RELATTN_NOALLOC_SCRATCH_BYTES) return RELATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != RELATTN_OK) return rc;
  DecodeLaunch L;
  rc = prepare_decode(q, rel, kDefaultIo, kv_cache, block_table, seq_lens, 1, window, rel_extent,
                      dims, out, scratch, RELATTN_NOALLOC_SCRATCH_BYTES, false, &L, &di);
  if (rc != RELATTN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the status word and the
  // split counters must start at zero (the partial results need not).
  cudaError_t e = cudaMemsetAsync(scratch, 0, w.lse, s);
  if (e == cudaSuccess) e = launch_decode(L, s);
  return to_status(e);
}

static int prepare_prefill(const void* q, const void* k, const void* v, const void* rel,
                           IoTypes io, const int32_t* cu_seqlens, const relattn_kv_cache* cache,
                           const int32_t* block_table, const int32_t* ctx_lens,
                           int32_t window, int32_t rel_extent, const relattn_dims* dims,
                           void* out, void* workspace, size_t ws_bytes, bool walk,
                           PrefillLaunch* L) {
  int rc = check_cache(cache);
  if (rc != RELATTN_OK) return rc;
  rc = check_dims(dims, cache);
  if (rc != RELATTN_OK) return rc;
  if (!cu_seqlens || !block_table || !ctx_lens || !workspace) return RELATTN_ERR_INVALID_ARG;
  if (dims->max_q_len < 0 || dims->num_tokens < 0) return RELATTN_ERR_INVALID_ARG;
  if (!walk) {
    if (!q || !k || !v || !rel || !out) return RELATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(rel) || !aligned16(out))
      return RELATTN_ERR_INVALID_ARG;
    if (!rel_extent_ok(rel_extent, io.rel_es)) return RELATTN_ERR_UNSUPPORTED;
  }
  if (!aligned16(workspace) || ws_bytes < kStatusBytes) return RELATTN_ERR_WORKSPACE;
  std::memset(L, 0, sizeof(*L));
  PrefillParams& p = L->p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.rel = rel;
  p.cu_seqlens = cu_seqlens;
  p.ctx_lens = ctx_lens;
  p.block_table = block_table;
  p.k_cache = static_cast<__nv_bfloat16*>(cache->k);
  p.v_cache = static_cast<__nv_bfloat16*>(cache->v);
  p.out = out;
  p.sink = io.sink;
  p.gate = io.gate;
  p.logit_scale = io.logit_scale;
  p.rel_es = io.rel_es;
  p.out_f32 = io.out_f32;
  p.status = static_cast<uint32_t*>(workspace);
  p.B = dims->batch;
  p.T = dims->num_tokens;
  p.Hq = dims->num_q_heads;
  p.Hkv = cache->num_kv_heads;
  p.g = dims->num_q_heads / cache->num_kv_heads;
  p.dv = cache->d_v;
  p.max_blocks = dims->max_blocks_per_seq;
  p.num_blocks = cache->num_blocks;
  p.window = window;
  p.rel_extent = rel_extent;
  p.max_q_len = dims->max_q_len;
  // log2(e) / sqrt(d_qk), times the key scale of an e4m3 cache
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(128.0) * io.k_scale);
  p.kv_es = io.kv_es;
  p.k_scale = io.k_scale;
  p.v_scale = io.v_scale;
  DeviceInfo di;
  if (!device_info(&di)) return RELATTN_ERR_CUDA;
  // bf16 caches: two heads of a KV group per work item when its ring fits;
  // otherwise (e4m3 caches, or very many sequences) one head per item.  A call
  // whose one-head items fit one wave of CTAs is latency-bound, and one head
  // per item spreads it over more SMs; a forced grid (num_ctas > 0) keeps the
  // two-heads kernel.
  const long long one_head_items =
      static_cast<long long>(p.B) * ((p.max_q_len + 127) / 128) * p.Hq;
  const bool one_wave = !walk && dims->num_ctas == 0 && one_head_items <= di.sms;
  // bf16 cache and bf16 rel with d_v = 128: one head per item over 128-key
  // tiles (the tensor pipe at N = 128) when its ring fits
  const int wide_slots = io.kv_es == 2 && io.rel_es == 2 && p.dv == 128 && !one_wave
                             ? prefill_wide_slots(p.B, di.smem_optin)
                             : 0;
  L->wide = wide_slots > 0 ? 1 : 0;
  const int pair_slots = io.kv_es == 2 && !one_wave && !L->wide
                             ? prefill_pair_slots(p.B, p.dv, p.rel_es, di.smem_optin)
                             : 0;
  L->pair = pair_slots > 0 ? 1 : 0;
  p.ring_stages = L->wide   ? wide_slots
                  : L->pair ? pair_slots
                            : prefill_ring_stages(p.B, p.dv, p.kv_es, di.smem_optin);
  if (p.ring_stages == 0) return RELATTN_ERR_UNSUPPORTED;
  const long long heads = L->pair ? static_cast<long long>(p.Hkv) * ((p.g + 1) / 2) : p.Hq;
  const long long items = static_cast<long long>(p.B) * ((p.max_q_len + 127) / 128) * heads;
  const long long want = dims->num_ctas > 0 ? dims->num_ctas : di.sms;
  L->grid = static_cast<int>(items < want ? (items > 0 ? items : 1) : want);
  if (walk) return RELATTN_OK;
  // e4m3 caches: 2-D boxes of 64 head-major rows, landing in staging slots
  if (!(io.kv_es == 1 ? decode_cache_maps_e4m3(cache, kTileKeys, &L->tm_k, &L->tm_v)
                      : cache_maps(cache, L->wide ? 128 : kTileKeys, &L->tm_k, &L->tm_v)))
    return RELATTN_ERR_CUDA;
  // q [T][Hq][128] bf16: one head's 128-token tile as two 64-column boxes
  const cuuint64_t qd[3] = {128, static_cast<cuuint64_t>(dims->num_q_heads),
                            static_cast<cuuint64_t>(dims->num_tokens)};
  const cuuint64_t qs[2] = {256, static_cast<cuuint64_t>(dims->num_q_heads) * 256};
  const cuuint32_t qb[3] = {64, 1, 128};
  if (!make_map(&L->tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), qd, qs, qb,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return RELATTN_ERR_CUDA;
  // rel [T][Hq][E] fp32 or bf16: boxes of 32 tokens x 100 (fp32) or 104
  // (bf16) distances of one head; 200 bf16 distances for 128-key tiles
  const cuuint64_t rd[3] = {static_cast<cuuint64_t>(rel_extent),
                            static_cast<cuuint64_t>(dims->num_q_heads),
                            static_cast<cuuint64_t>(dims->num_tokens)};
  const cuuint64_t rs[2] = {static_cast<cuuint64_t>(rel_extent) * io.rel_es,
                            static_cast<cuuint64_t>(rel_extent) * io.rel_es * dims->num_q_heads};
  const cuuint32_t rb[3] = {L->wide ? 200u : io.rel_es == 2 ? 104u : 100u, 1, 32};
  if (!make_map(&L->tm_rel,
                io.rel_es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                3, const_cast<void*>(rel), rd, rs, rb, CU_TENSOR_MAP_SWIZZLE_NONE))
    return RELATTN_ERR_CUDA;
  if (L->wide) {
    // out [T][Hq][128], bf16 or fp32: a full tile's 128 rows of one head as
    // 128-byte column boxes (64 bf16 or 32 fp32), 128-byte swizzled
    const cuuint64_t oes = io.out_f32 ? 4 : 2;
    const cuuint64_t od[3] = {128, static_cast<cuuint64_t>(dims->num_q_heads),
                              static_cast<cuuint64_t>(dims->num_tokens)};
    const cuuint64_t os[2] = {128 * oes, static_cast<cuuint64_t>(dims->num_q_heads) * 128 * oes};
    const cuuint32_t ob[3] = {static_cast<cuuint32_t>(128 / oes), 1, 128};
    if (!make_map(&L->tm_out,
                  io.out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  3, out, od, os, ob, CU_TENSOR_MAP_SWIZZLE_128B))
      return RELATTN_ERR_CUDA;
  }
  return RELATTN_OK;
}

static int relattn_prefill_io(const void* q, const void* k, const void* v, const void* rel,
                              IoTypes io, const int32_t* cu_seqlens,
                              const relattn_kv_cache* cache, const int32_t* block_table,
                              const int32_t* ctx_lens, int32_t window, int32_t rel_extent,
                              const relattn_dims* dims, void* out, void* workspace,
                              size_t workspace_bytes, void* stream) {
  PrefillLaunch L;
  const int rc = prepare_prefill(q, k, v, rel, io, cu_seqlens, cache, block_table, ctx_lens,
                                 window, rel_extent, dims, out, workspace, workspace_bytes, false,
                                 &L);
  if (rc != RELATTN_OK) return rc;
  if (dims->max_q_len == 0 || dims->num_tokens == 0) return RELATTN_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_cache_write(L.p, s);
  if (e == cudaSuccess)
    e = L.wide   ? launch_prefill_wide(L, L.grid, s)
        : L.pair ? launch_prefill_pair(L, L.grid, s)
                 : launch_prefill(L, L.grid, s);
  return to_status(e);
}

int relattn_prefill(const void* q, const void* k, const void* v, const float* rel,
                    const int32_t* cu_seqlens, const relattn_kv_cache* cache,
                    const int32_t* block_table, const int32_t* ctx_lens, int32_t window,
                    int32_t rel_extent, const relattn_dims* dims, void* out, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return relattn_prefill_io(q, k, v, rel, kDefaultIo, cu_seqlens, cache, block_table, ctx_lens,
                            window, rel_extent, dims, out, workspace, workspace_bytes, stream);
}

int relattn_prefill_ex(const void* q, const void* k, const void* v, const void* rel,
                       const relattn_options* options, const int32_t* cu_seqlens,
                       const relattn_kv_cache* cache, const int32_t* block_table,
                       const int32_t* ctx_lens, int32_t window, int32_t rel_extent,
                       const relattn_dims* dims, void* out, void* workspace,
                       size_t workspace_bytes, void* stream) {
  IoTypes io;
  if (!io_types(options, &io)) return RELATTN_ERR_INVALID_ARG;
  if (io.kv_es == 1 && (!cache || cache->d_v != 128 ||
                        static_cast<long long>(cache->num_blocks) * cache->num_kv_heads * 128 >
                            0x7fffffffLL))
    return RELATTN_ERR_UNSUPPORTED;  // e4m3 caches: d_v = 128, 32-bit row coordinates
  return relattn_prefill_io(q, k, v, rel, io, cu_seqlens, cache, block_table, ctx_lens, window,
                            rel_extent, dims, out, workspace, workspace_bytes, stream);
}

int relattn_cache_write(const void* k, const void* v, const relattn_options* options,
                        const int32_t* cu_seqlens, const relattn_kv_cache* cache,
                        const int32_t* block_table, const int32_t* ctx_lens,
                        const relattn_dims* dims, void* workspace, size_t workspace_bytes,
                        void* stream) {
  IoTypes io = kDefaultIo;
  if (options != nullptr && !io_types(options, &io)) return RELATTN_ERR_INVALID_ARG;
  int rc = check_cache(cache);
  if (rc != RELATTN_OK) return rc;
  if (!dims || !k || !v || !cu_seqlens || !block_table || !ctx_lens || !workspace)
    return RELATTN_ERR_INVALID_ARG;
  if (dims->batch < 0 || dims->max_blocks_per_seq < 1 || dims->num_tokens < 0 ||
      dims->max_q_len < 0)
    return RELATTN_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v)) return RELATTN_ERR_INVALID_ARG;
  if (!aligned16(workspace) || workspace_bytes < kStatusBytes) return RELATTN_ERR_WORKSPACE;
  if (dims->batch > kCacheWriteMaxGridY ||
      static_cast<long long>(dims->max_blocks_per_seq) * 128 > 0x7fffffffLL)
    return RELATTN_ERR_UNSUPPORTED;
  if (io.kv_es == 1 && (cache->d_v != 128 ||
                        static_cast<long long>(cache->num_blocks) * cache->num_kv_heads * 128 >
                            0x7fffffffLL))
    return RELATTN_ERR_UNSUPPORTED;
  PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.cu_seqlens = cu_seqlens;
  p.ctx_lens = ctx_lens;
  p.block_table = block_table;
  p.k_cache = static_cast<__nv_bfloat16*>(cache->k);
  p.v_cache = static_cast<__nv_bfloat16*>(cache->v);
  p.status = static_cast<uint32_t*>(workspace);
  p.B = dims->batch;
  p.T = dims->num_tokens;
  p.Hkv = cache->num_kv_heads;
  p.dv = cache->d_v;
  p.max_blocks = dims->max_blocks_per_seq;
  p.num_blocks = cache->num_blocks;
  p.max_q_len = dims->max_q_len;
  p.kv_es = io.kv_es;
  p.k_scale = io.k_scale;
  p.v_scale = io.v_scale;
  if (p.B == 0 || p.T == 0 || p.max_q_len == 0) return RELATTN_OK;
  return to_status(launch_cache_write(p, static_cast<cudaStream_t>(stream)));
}

int relattn_debug_wait_timeout(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || !aligned16(workspace) || workspace_bytes < kStatusBytes)
    return RELATTN_ERR_WORKSPACE;
  return to_status(
      launch_wait_timeout(static_cast<uint32_t*>(workspace), static_cast<cudaStream_t>(stream)));
}

int relattn_debug_walk_prefill(const int32_t* cu_seqlens, const int32_t* ctx_lens,
                               const int32_t* block_table, int32_t window,
                               const relattn_kv_cache* cache, const relattn_dims* dims,
                               int32_t* records, int32_t max_records, int32_t* count,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (!records || !count || max_records < 0) return RELATTN_ERR_INVALID_ARG;
  PrefillLaunch L;
  const int rc = prepare_prefill(nullptr, nullptr, nullptr, nullptr, kDefaultIo, cu_seqlens,
                                 cache, block_table, ctx_lens, window, 4, dims, nullptr,
                                 workspace, workspace_bytes, true, &L);
  if (rc != RELATTN_OK) return rc;
  if (dims->max_q_len == 0) return RELATTN_OK;
  L.p.dbg_records = records;
  L.p.dbg_count = count;
  L.p.dbg_max = max_records;
  return to_status(launch_prefill_walk(L.p, L.grid, static_cast<cudaStream_t>(stream)));
}

int relattn_debug_walk_prefill_ex(const int32_t* cu_seqlens, const int32_t* ctx_lens,
                                  const int32_t* block_table, int32_t window,
                                  const relattn_options* options, const relattn_kv_cache* cache,
                                  const relattn_dims* dims, int32_t* records,
                                  int32_t max_records, int32_t* count, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (!records || !count || max_records < 0) return RELATTN_ERR_INVALID_ARG;
  IoTypes io = kDefaultIo;
  if (options != nullptr && !io_types(options, &io)) return RELATTN_ERR_INVALID_ARG;
  if (io.kv_es != 2) return RELATTN_ERR_UNSUPPORTED;  // bf16 caches: the kernels with a walk
  PrefillLaunch L;
  const int rc = prepare_prefill(nullptr, nullptr, nullptr, nullptr, io, cu_seqlens, cache,
                                 block_table, ctx_lens, window, 16, dims, nullptr, workspace,
                                 workspace_bytes, true, &L);
  if (rc != RELATTN_OK) return rc;
  if (dims->max_q_len == 0) return RELATTN_OK;
  L.p.dbg_records = records;
  L.p.dbg_count = count;
  L.p.dbg_max = max_records;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return to_status(L.wide ? launch_prefill_wide_walk(L.p, L.grid, s)
                          : launch_prefill_walk(L.p, L.grid, s));
}

}  // extern "C"
