// Chunked prefill with a cached prefix for relative-bias GQA attention.
//
// Two kernels on the caller's stream:
//  * cache_write: scatters each new token's key and value into the paged
//    cache at position ctx_lens[b] + t ("Inkling-Small on Gaudi 2", section
//    "Attention with a relative bias": later chunks and prefix-cache hits
//    prepend the cached context);
//  * prefill: per (64-row query tile, query head), walks the key tiles of the
//    window [max(0, P_first - W + 1), P_last] through the block table, loads
//    K/V tiles with TMA, computes S = QK^T with mma.sync, adds the sheared
//    relative term rel[row, h, P_row - j] in registers (no [Lq, KV] mask is
//    ever formed), applies the causal and window masks and an online
//    softmax, and accumulates O = PV.
#include "relattn_common.cuh"
#include "relattn_internal.h"

namespace relattn {

namespace {

constexpr int kPrefillThreads = 128;  // 4 warps x 16 query rows
constexpr int kQTile = 64;
constexpr int kPrefillStages = 3;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ bool seq_ok(int ctx, int n, int max_blocks) {
  return ctx >= 0 && n >= 0 &&
         static_cast<long long>(ctx) + n <= static_cast<long long>(max_blocks) * kBlockSize;
}

__global__ void __launch_bounds__(256) cache_write_kernel(const PrefillParams p) {
  const int b = blockIdx.y;
  const int r0 = p.cu_seqlens[b];
  const int n = p.cu_seqlens[b + 1] - r0;
  const int ctx = p.ctx_lens[b];
  const int t0 = blockIdx.x * kQTile;
  if (!seq_ok(ctx, n, p.max_blocks)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(p.status, RELATTN_DEV_BAD_LENGTH);
    return;
  }
  if (t0 >= n) return;
  const int nt = min(kQTile, n - t0);
  const int kch = kDqk / 8, vch = p.dv / 8;
  const int per_tok = p.Hkv * (kch + vch);
  const int* trow = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  for (int i = threadIdx.x; i < nt * per_tok; i += blockDim.x) {
    const int tt = i / per_tok;
    const int rem = i - tt * per_tok;
    const int hh = rem / (kch + vch);
    int ch = rem - hh * (kch + vch);
    const int pos = ctx + t0 + tt;
    const int phys = __ldg(trow + pos / kBlockSize);
    if (phys < 0 || phys >= p.num_blocks) {
      report(p.status, RELATTN_DEV_BAD_BLOCK_ID);
      continue;
    }
    const size_t slot = static_cast<size_t>(phys) * kBlockSize + pos % kBlockSize;
    const size_t row = static_cast<size_t>(r0 + t0 + tt);
    if (ch < kch) {
      const uint4 val = __ldg(reinterpret_cast<const uint4*>(
          p.k + (row * p.Hkv + hh) * kDqk) + ch);
      reinterpret_cast<uint4*>(p.k_cache + (slot * p.Hkv + hh) * kDqk)[ch] = val;
    } else {
      ch -= kch;
      const uint4 val = __ldg(reinterpret_cast<const uint4*>(
          p.v + (row * p.Hkv + hh) * p.dv) + ch);
      reinterpret_cast<uint4*>(p.v_cache + (slot * p.Hkv + hh) * p.dv)[ch] = val;
    }
  }
}

template <int DV>
__global__ void __launch_bounds__(kPrefillThreads)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v,
                   const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kStageBytes = 16384 + kTileKeys * DV * 2;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPrefillStages * kStageBytes);
  int* s_valid = reinterpret_cast<int*>(full + kPrefillStages);

  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r_begin = p.cu_seqlens[b];
  const int n = p.cu_seqlens[b + 1] - r_begin;
  const int ctx = p.ctx_lens[b];
  const int t0 = qt * kQTile;
  if (t0 >= n) return;
  const int rows = min(kQTile, n - t0);
  const int r0 = lane >> 2, cq = lane & 3;
  const int rA = warp * 16 + r0, rB = rA + 8;  // tile-local rows of this thread
  __nv_bfloat16* out_base = p.out + (static_cast<size_t>(r_begin + t0) * p.Hq + h) * DV;
  if (!seq_ok(ctx, n, p.max_blocks)) {
    for (int i = tid; i < rows * DV; i += blockDim.x)
      out_base[static_cast<size_t>(i / DV) * p.Hq * DV + i % DV] = __float2bfloat16(0.f);
    return;  // reported by cache_write
  }
  const int kvh = h / p.g;
  const int P0 = ctx + t0;
  const int P1 = P0 + rows - 1;
  const int tf = window_lo(P0, p.window) / kTileKeys;
  const int ntiles = P1 / kTileKeys - tf + 1;
  const int* trow = p.block_table + static_cast<size_t>(b) * p.max_blocks;

  if (tid == 0) {
    for (int s = 0; s < kPrefillStages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  auto issue = [&](int stage, int tile) {
    const int id = __ldg(trow + (tile >> 1));
    const bool ok = id >= 0 && id < p.num_blocks;
    s_valid[stage] = ok ? 1 : 0;
    if (!ok) {
      report(p.status, RELATTN_DEV_BAD_BLOCK_ID);
      mbar_arrive(&full[stage]);
      return;
    }
    uint8_t* st = smem + stage * kStageBytes;
    const int row = id * kBlockSize + (tile & 1) * kTileKeys;
    mbar_arrive_expect_tx(&full[stage], kStageBytes);
    tma_load_3d(st, &tm_k, &full[stage], 0, kvh, row);
    tma_load_3d(st + 8192, &tm_k, &full[stage], 64, kvh, row);
    tma_load_3d(st + 16384, &tm_v, &full[stage], 0, kvh, row);
    if (DV == 128) tma_load_3d(st + 24576, &tm_v, &full[stage], 64, kvh, row);
  };
  if (tid == 0)
    for (int s = 0; s < kPrefillStages && s < ntiles; ++s) issue(s, tf + s);

  // query fragments (rows beyond the chunk are zero)
  uint32_t qa[8][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = (i & 1) ? rB : rA;
      const int col = ks * 16 + cq * 2 + (i >> 1) * 8;
      qa[ks][i] = row < rows
                      ? __ldg(reinterpret_cast<const uint32_t*>(
                            p.q + (static_cast<size_t>(r_begin + t0 + row) * p.Hq + h) * kDqk + col))
                      : 0u;
    }
  const int PA = P0 + rA, PB = P0 + rB;
  const int loA = window_lo(PA, p.window), loB = window_lo(PB, p.window);
  const float* relA = p.rel + (static_cast<size_t>(r_begin + t0 + rA) * p.Hq + h) * p.rel_extent;
  const float* relB = p.rel + (static_cast<size_t>(r_begin + t0 + rB) * p.Hq + h) * p.rel_extent;
  const bool okA = rA < rows, okB = rB < rows;

  float m_[2] = {kNegInf, kNegInf}, l_[2] = {0.f, 0.f};
  float o[DV / 8][4];
#pragma unroll
  for (int i = 0; i < DV / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  bool abort = false;
  for (int k = 0; k < ntiles; ++k) {
    const int stage = k % kPrefillStages;
    const uint32_t parity = (k / kPrefillStages) & 1;
    const int key0 = (tf + k) * kTileKeys;
    // relative term and masks for this thread's 32 elements (issued before
    // the wait so the loads overlap it)
    float x[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool second = i >= 2;
        const int P = second ? PB : PA;
        const int lo = second ? loB : loA;
        const int key = key0 + nt * 8 + cq * 2 + (i & 1);
        const int d = P - key;
        float bias = kNegInf;
        if ((second ? okB : okA) && key >= lo && d >= 0)
          bias = d < p.rel_extent ? __ldg((second ? relB : relA) + d) : 0.f;
        x[nt][i] = bias;
      }
    if (!mbar_wait(&full[stage], parity)) {
      report(p.status, RELATTN_DEV_WAIT_TIMEOUT);
      abort = true;
    }
    if (!abort && s_valid[stage]) {
      const uint32_t kbase = smem_u32(smem + stage * kStageBytes);
      float s[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
      {
        const int mi = lane >> 3;
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int key = np * 16 + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const int chunk = ks * 2 + (mi & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + (chunk >> 3) * 8192 + sw128(key, chunk & 7), b0, b1, b2, b3);
            mma_16816(s[2 * np], qa[ks], b0, b1);
            mma_16816(s[2 * np + 1], qa[ks], b2, b3);
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          x[nt][i] = x[nt][i] == kNegInf ? kNegInf
                                         : fmaf(s[nt][i], p.scale_log2, x[nt][i] * kLog2e);
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        float mx = kNegInf;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) mx = fmaxf(mx, fmaxf(x[nt][2 * rr], x[nt][2 * rr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_[rr], mx);
        const float m_use = m_new == kNegInf ? 0.f : m_new;
        const float alpha = ex2(m_[rr] - m_use);
        m_[rr] = m_new;
        float sum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pv = ex2(x[nt][2 * rr + e] - m_use);
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
      const uint32_t vbase = kbase + 16384;
      const int mi = lane >> 3;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_bf16(x[2 * kk][0], x[2 * kk][1]);
        pa[1] = pack_bf16(x[2 * kk][2], x[2 * kk][3]);
        pa[2] = pack_bf16(x[2 * kk + 1][0], x[2 * kk + 1][1]);
        pa[3] = pack_bf16(x[2 * kk + 1][2], x[2 * kk + 1][3]);
        const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
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
    __syncthreads();
    if (abort) break;
    if (tid == 0 && k + kPrefillStages < ntiles) issue(stage, tf + k + kPrefillStages);
  }

#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l_[rr] += __shfl_xor_sync(0xffffffffu, l_[rr], 1);
    l_[rr] += __shfl_xor_sync(0xffffffffu, l_[rr], 2);
  }
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int row = rr ? rB : rA;
    if (row >= rows) continue;
    const float inv = l_[rr] > 0.f ? 1.f / l_[rr] : 0.f;
    __nv_bfloat16* orow = out_base + static_cast<size_t>(row) * p.Hq * DV;
#pragma unroll
    for (int nd = 0; nd < DV / 8; ++nd)
      *reinterpret_cast<__nv_bfloat162*>(orow + nd * 8 + cq * 2) =
          __floats2bfloat162_rn(o[nd][2 * rr] * inv, o[nd][2 * rr + 1] * inv);
  }
}

__global__ void prefill_walk_kernel(const PrefillParams p) {
  if (threadIdx.x != 0) return;
  const int qt = blockIdx.x, b = blockIdx.y;
  const int n = p.cu_seqlens[b + 1] - p.cu_seqlens[b];
  const int ctx = p.ctx_lens[b];
  const int t0 = qt * kQTile;
  if (t0 >= n || !seq_ok(ctx, n, p.max_blocks)) return;
  const int rows = min(kQTile, n - t0);
  const int P0 = ctx + t0, P1 = P0 + rows - 1;
  const int tf = window_lo(P0, p.window) / kTileKeys;
  const int ntiles = P1 / kTileKeys - tf + 1;
  const int* trow = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  for (int k = 0; k < ntiles; ++k) {
    const int tile = tf + k;
    const int r = atomicAdd(p.dbg_count, 1);
    if (r < p.dbg_max) {
      int32_t* rec = p.dbg_records + 6 * static_cast<size_t>(r);
      rec[0] = b;
      rec[1] = t0;
      rec[2] = tile;
      rec[3] = tile >> 1;
      rec[4] = trow[tile >> 1];
      rec[5] = 0;
    }
  }
}

}  // namespace

cudaError_t launch_cache_write(const PrefillParams& p, cudaStream_t stream) {
  const dim3 grid((p.max_q_len + kQTile - 1) / kQTile, p.B);
  cache_write_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillLaunch& L, cudaStream_t stream) {
  const PrefillParams& p = L.p;
  const dim3 grid((p.max_q_len + kQTile - 1) / kQTile, p.Hq, p.B);
  const int smem = kPrefillStages * (16384 + kTileKeys * p.dv * 2) + 1024 +
                   kPrefillStages * 16 + 64;
  cudaError_t e;
  if (p.dv == 128) {
    e = cudaFuncSetAttribute(prefill_kernel<128>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    prefill_kernel<128><<<grid, kPrefillThreads, smem, stream>>>(L.tm_k, L.tm_v, p);
  } else {
    e = cudaFuncSetAttribute(prefill_kernel<64>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    prefill_kernel<64><<<grid, kPrefillThreads, smem, stream>>>(L.tm_k, L.tm_v, p);
  }
  return cudaGetLastError();
}

cudaError_t launch_prefill_walk(const PrefillParams& p, cudaStream_t stream) {
  const dim3 grid((p.max_q_len + kQTile - 1) / kQTile, p.B);
  prefill_walk_kernel<<<grid, 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace relattn
