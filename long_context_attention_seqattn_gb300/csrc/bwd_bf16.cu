// bwd_bf16.cu -- tensor-core exact backward of one chunk (bf16 in, fp32
// accumulate), with the dK/dV running sums over the prefix.
//
// Operation (StreamBP review page: Eq. (1) -- the gradient is a sum of
// per-chunk terms -- and the running-sum accumulation of the partitioned
// attention gradients named in its "Circularity Check"; major comment 1 of its
// referee report names dK^(:i), dV^(:i) over the prefix).  With the forward's
// row logsumexp L and Delta = rowsum(dO o O):
//   P = exp(scale Q K^T - L), dP = dO V^T, dS = P o (dP - Delta)
//   dV += P^T dO,  dK += scale dS^T Q,  dQ = scale dS K
//
// One CTA owns one 128-key tile of one key/value head: it loops over the G
// query heads of the group and the chunk's 64-row query tiles that can see the
// tile, keeps dK and dV for its 128 keys in TMEM for the whole loop, and
// finally adds them into the float32 accumulators with a plain
// read-modify-write (no other CTA touches those rows in this call, so there is
// no atomic contention across query tiles).  dQ partial products of every key
// tile are summed into the zeroed dq with fp32 reductions.
//   warp 0      TMA producer: K, V once; Q, dO (64 rows) + L, Delta per step
//   warp 1      TMEM owner + MMA issuer (one thread):
//                 S^T = K Q^T, dP^T = V dO^T       (M=128 keys, N=64, K=128)
//                 dV += P^T dO, dK += dS^T Q       (M=128 keys, N=128, K=64)
//                 dQ^T = K^T dS^T                  (M=128 d,    N=64, K=128)
//   warps 2..5  P^T, dS^T from TMEM -> bf16 tiles in shared memory; the
//               final dK/dV read-modify-write
//   warps 6..9  dQ^T from TMEM -> fp32 reductions into dq
// The next step's S^T/dP^T MMAs are issued before this step's dV/dK/dQ MMAs,
// so the tensor pipe works while the compute warps form P and dS.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace seqattn {
namespace {

constexpr int kBK = 128;   // keys per CTA
constexpr int kBQ = 64;    // query rows per step
constexpr int kD = 128;    // head dim
constexpr int kThreads = 320;  // 10 warps

constexpr int kKVTileBytes = kBK * kD * 2;         // 32 KB
constexpr int kKVHalf = kKVTileBytes / 2;          // 16 KB: 128 rows x 128 B
constexpr int kQTileBytes = kBQ * kD * 2;          // 16 KB
constexpr int kQHalf = kQTileBytes / 2;            // 8 KB: 64 rows x 128 B
constexpr int kPTileBytes = kBK * kBQ * 2;         // 16 KB: 128 keys x 64 q

// shared memory carve-up (bytes from the 1024-aligned base)
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKVTileBytes;
constexpr int kOffQ = kOffV + kKVTileBytes;              // 2 stages
constexpr int kOffDO = kOffQ + 2 * kQTileBytes;          // 2 stages
constexpr int kOffP = kOffDO + 2 * kQTileBytes;          // 2 buffers
constexpr int kOffDS = kOffP + 2 * kPTileBytes;          // 2 buffers
constexpr int kOffStat = kOffDS + 2 * kPTileBytes;       // 2 stages x (L[64], Delta[64])
constexpr int kStatBytes = 2 * kBQ * 4;
constexpr int kSmemBytes = kOffStat + 2 * kStatBytes;
constexpr int kSmemAlloc = kSmemBytes + 1024;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColDK = 0;
constexpr uint32_t kColDV = 128;
constexpr uint32_t kColS = 256;
constexpr uint32_t kColDP = 320;
constexpr uint32_t kColDQ = 384;

constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  int B, Hq, Hkv, G;
  int q_len, T;
  int q_start, kv_begin;
  int n_ktiles;
  float scale;
  float scale_log2;
  const float* lse;
  const float* delta;
  float* dq;
  float* dk;
  float* dv;
  unsigned int* err;
};

struct BwdBarriers {
  uint64_t kv_full;
  uint64_t q_full[2], q_empty[2];
  uint64_t sdp_full;
  uint64_t ds_full[2], ds_empty[2];
  uint64_t dq_full, dq_empty;
  uint64_t acc_done;
  uint64_t mma_final;
};

__device__ __forceinline__ bool warp_wait(Watchdog& wd, uint64_t* bar, uint32_t parity) {
  const bool ok = wd.wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// K-major operand whose rows are `rows` long blocks of 128 B (64 bf16 of K):
// K-step ks (16 elements) lies in block ks/4 at byte 32*(ks%4) of each row.
__device__ __forceinline__ uint64_t kmajor(uint32_t base, int block_bytes, int ks) {
  return make_desc_sw128(base + (ks >> 2) * block_bytes + (ks & 3) * 32, 16, 1024);
}
// MN-major operand stored as [K rows][MN] with 128-byte rows: 8 K-rows per
// 1024-byte atom, `mn_block_bytes` between 64-wide MN blocks; K-step ks
// (16 rows) starts 2048 bytes further.
__device__ __forceinline__ uint64_t mnmajor(uint32_t base, int mn_block_bytes, int ks) {
  return make_desc_sw128(base + ks * 2048, mn_block_bytes, 1024);
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_bf16_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                    const BwdParams p) {
  if (error_already_set(p.err)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ BwdBarriers bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  Watchdog wd{&abort_flag, p.err};

  // ---- work item: key tile kt (fastest), kv head g, batch b
  int idx = blockIdx.x;
  const int kt = idx % p.n_ktiles;
  idx /= p.n_ktiles;
  const int g = idx % p.Hkv;
  const int b = idx / p.Hkv;
  const int kb = p.kv_begin + kt * kBK;                  // absolute first key of the tile
  const int n_q64 = p.q_len / kBQ;
  // first query tile that sees any key of this tile; the two tiles covering
  // the diagonal 128 block carry the causal mask
  const int qi_first = kb >= p.q_start ? (kb - p.q_start) / kBQ : 0;
  const bool diag_tile = kb >= p.q_start;
  const int nq = n_q64 - qi_first;
  const int n_steps = p.G * nq;

  const int warp = warp_id();
  const int lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars.kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 1);
      mbar_init(&bars.ds_full[i], 4 * 32);
      mbar_init(&bars.ds_empty[i], 1);
    }
    mbar_init(&bars.sdp_full, 1);
    mbar_init(&bars.dq_full, 1);
    mbar_init(&bars.dq_empty, 4 * 32);
    mbar_init(&bars.acc_done, 1);
    mbar_init(&bars.mma_final, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  const uint32_t sK = smem_u32(smem + kOffK);
  const uint32_t sV = smem_u32(smem + kOffV);
  const uint32_t sQ = smem_u32(smem + kOffQ);
  const uint32_t sDO = smem_u32(smem + kOffDO);
  const uint32_t sP = smem_u32(smem + kOffP);
  const uint32_t sDS = smem_u32(smem + kOffDS);
  float* stat = reinterpret_cast<float*>(smem + kOffStat);  // [stage][L 64 | Delta 64]

  auto step_head = [&](int n) { return g * p.G + n / nq; };
  auto step_qtile = [&](int n) { return qi_first + n % nq; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_do);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      const int krow = b * p.T + kb;
      mbar_arrive_expect_tx(&bars.kv_full, 2 * kKVTileBytes);
      tma_load_3d(smem + kOffK, &map_k, &bars.kv_full, 0, g, krow);
      tma_load_3d(smem + kOffK + kKVHalf, &map_k, &bars.kv_full, 64, g, krow);
      tma_load_3d(smem + kOffV, &map_v, &bars.kv_full, 0, g, krow);
      tma_load_3d(smem + kOffV + kKVHalf, &map_v, &bars.kv_full, 64, g, krow);
      int issued[2] = {0, 0};
      for (int n = 0; n < n_steps; ++n) {
        const int st = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        const int h = step_head(n);
        const int qi = step_qtile(n);
        if (!wd.wait(&bars.q_empty[st], ph ^ 1)) break;
        const int qrow = b * p.q_len + qi * kBQ;
        const int64_t srow = (static_cast<int64_t>(b) * p.Hq + h) * p.q_len + qi * kBQ;
        mbar_arrive_expect_tx(&bars.q_full[st], 2 * kQTileBytes + kStatBytes);
        tma_load_3d(smem + kOffQ + st * kQTileBytes, &map_q, &bars.q_full[st], 0, h, qrow);
        tma_load_3d(smem + kOffQ + st * kQTileBytes + kQHalf, &map_q, &bars.q_full[st], 64, h, qrow);
        tma_load_3d(smem + kOffDO + st * kQTileBytes, &map_do, &bars.q_full[st], 0, h, qrow);
        tma_load_3d(smem + kOffDO + st * kQTileBytes + kQHalf, &map_do, &bars.q_full[st], 64, h, qrow);
        bulk_load(stat + st * 2 * kBQ, p.lse + srow, kBQ * 4, &bars.q_full[st]);
        bulk_load(stat + st * 2 * kBQ + kBQ, p.delta + srow, kBQ * 4, &bars.q_full[st]);
        issued[st] = n + 1;
      }
      if (wd.aborted()) {
        wd.drain(&bars.kv_full, 0, 1000000);
        for (int st = 0; st < 2; ++st)
          if (issued[st] > 0) wd.drain(&bars.q_full[st], ((issued[st] - 1) >> 1) & 1, 1000000);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_sdp = make_idesc_bf16(kBK, kBQ, false, false);  // M128 N64, K-major both
      const uint32_t idesc_kv = make_idesc_bf16(kBK, kD, false, true);     // M128 N128, B MN-major
      const uint32_t idesc_dq = make_idesc_bf16(kD, kBQ, true, true);      // M128 N64, both MN-major
      auto issue_sdp = [&](int n) -> bool {
        const int st = n & 1;
        if (!wd.wait(&bars.q_full[st], (n >> 1) & 1)) return false;
        tc_fence_after_sync();
        const uint32_t qa = sQ + st * kQTileBytes;
        const uint32_t da = sDO + st * kQTileBytes;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks)
          umma_bf16_ss(tmem + kColS, kmajor(sK, kKVHalf, ks), kmajor(qa, kQHalf, ks), idesc_sdp,
                       ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks)
          umma_bf16_ss(tmem + kColDP, kmajor(sV, kKVHalf, ks), kmajor(da, kQHalf, ks), idesc_sdp,
                       ks > 0 ? 1u : 0u);
        umma_commit(&bars.sdp_full);
        return true;
      };
      auto issue_grads = [&](int n) -> bool {
        const int st = n & 1;
        const uint32_t qa = sQ + st * kQTileBytes;
        const uint32_t da = sDO + st * kQTileBytes;
        const uint32_t pa = sP + st * kPTileBytes;
        const uint32_t dsa = sDS + st * kPTileBytes;
        // dV += P^T dO ; dK += dS^T Q   (K = 64 query rows: 4 steps)
#pragma unroll
        for (int ks = 0; ks < kBQ / 16; ++ks)
          umma_bf16_ss(tmem + kColDV, kmajor(pa, kPTileBytes, ks), mnmajor(da, kQHalf, ks), idesc_kv,
                       (n > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < kBQ / 16; ++ks)
          umma_bf16_ss(tmem + kColDK, kmajor(dsa, kPTileBytes, ks), mnmajor(qa, kQHalf, ks), idesc_kv,
                       (n > 0 || ks > 0) ? 1u : 0u);
        // dQ^T = K^T dS^T  (K = 128 keys: 8 steps); the dQ warps must have
        // drained the previous step's dQ^T
        if (n >= 1 && !wd.wait(&bars.dq_empty, (n - 1) & 1)) return false;
        tc_fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks)
          umma_bf16_ss(tmem + kColDQ, mnmajor(sK, kKVHalf, ks), mnmajor(dsa, kPTileBytes, ks), idesc_dq,
                       ks > 0 ? 1u : 0u);
        umma_commit(&bars.dq_full);
        umma_commit(&bars.q_empty[st]);
        umma_commit(&bars.ds_empty[st]);
        return true;
      };
      bool ok = wd.wait(&bars.kv_full, 0);
      if (ok && n_steps > 0) ok = issue_sdp(0);
      for (int n = 0; ok && n < n_steps; ++n) {
        if (!(ok = wd.wait(&bars.ds_full[n & 1], (n >> 1) & 1))) break;
        tc_fence_after_sync();
        if (n + 1 < n_steps && !(ok = issue_sdp(n + 1))) break;
        ok = issue_grads(n);
      }
      umma_commit(&bars.acc_done);
      umma_commit(&bars.mma_final);
      wd.drain(&bars.mma_final, 0, 4000000);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ P / dS
    const int quad = warp & 3;
    const int kr = quad * 32 + lane;                    // key row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int key = kb + kr;
    bool ok = true;
    for (int n = 0; n < n_steps; ++n) {
      const int st = n & 1;
      const int qi = step_qtile(n);
      if (!(ok = warp_wait(wd, &bars.sdp_full, n & 1))) break;
      if (!(ok = warp_wait(wd, &bars.q_full[st], (n >> 1) & 1))) break;
      if (n >= 2 && !(ok = warp_wait(wd, &bars.ds_empty[st], ((n - 2) >> 1) & 1))) break;
      tc_fence_after_sync();
      const float* L = stat + st * 2 * kBQ;
      const float* Dl = L + kBQ;
      const bool masked = diag_tile && (qi - qi_first) < 2;
      const int q_abs0 = p.q_start + qi * kBQ;          // absolute row of query column 0
      uint32_t pk[kBQ / 2];                             // P^T row, packed bf16 pairs
      float pf[kBQ];
#pragma unroll
      for (int c0 = 0; c0 < kBQ; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + kColS + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int c = c0 + j;
          float pv = ex2(fmaf(__uint_as_float(r[j]), p.scale_log2, -L[c] * kLog2e));
          if (masked && key > q_abs0 + c) pv = 0.f;
          pf[c] = pv;
        }
      }
#pragma unroll
      for (int c0 = 0; c0 < kBQ; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + kColDP + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int c = c0 + j;
          pk[c / 2] = pack_bf16x2(pf[c] * (__uint_as_float(r[j]) - Dl[c]),
                                  pf[c + 1] * (__uint_as_float(r[j + 1]) - Dl[c + 1]));
        }
      }
      // rows of 64 bf16 = 128 B, 128-byte swizzle inside 8-row groups
      const uint32_t sw = static_cast<uint32_t>(kr & 7);
      const uint32_t prow = sP + st * kPTileBytes + kr * 128;
      const uint32_t dsrow = sDS + st * kPTileBytes + kr * 128;
#pragma unroll
      for (int ci = 0; ci < 8; ++ci) {
        const int c = ci * 8;
        st_shared_v4(prow + ((ci ^ sw) << 4), pack_bf16x2(pf[c], pf[c + 1]), pack_bf16x2(pf[c + 2], pf[c + 3]),
                     pack_bf16x2(pf[c + 4], pf[c + 5]), pack_bf16x2(pf[c + 6], pf[c + 7]));
        st_shared_v4(dsrow + ((ci ^ sw) << 4), pk[ci * 4], pk[ci * 4 + 1], pk[ci * 4 + 2], pk[ci * 4 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&bars.ds_full[st]);
    }
    // ---- epilogue: dK, dV rows of this tile into the running sums
    if (ok) ok = warp_wait(wd, &bars.acc_done, 0);
    if (ok) {
      tc_fence_after_sync();
      const int64_t row = (static_cast<int64_t>(b) * p.T + key) * p.Hkv + g;
      float4* dkrow = reinterpret_cast<float4*>(p.dk + row * kD);
      float4* dvrow = reinterpret_cast<float4*>(p.dv + row * kD);
#pragma unroll
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + kColDK + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4 a = dkrow[(c0 + j) / 4];
          a.x += p.scale * __uint_as_float(r[j]);
          a.y += p.scale * __uint_as_float(r[j + 1]);
          a.z += p.scale * __uint_as_float(r[j + 2]);
          a.w += p.scale * __uint_as_float(r[j + 3]);
          dkrow[(c0 + j) / 4] = a;
        }
        tmem_ld32(tmem + lane_base + kColDV + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4 a = dvrow[(c0 + j) / 4];
          a.x += __uint_as_float(r[j]);
          a.y += __uint_as_float(r[j + 1]);
          a.z += __uint_as_float(r[j + 2]);
          a.w += __uint_as_float(r[j + 3]);
          dvrow[(c0 + j) / 4] = a;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ
    const int quad = warp & 3;
    const int dcol = quad * 32 + lane;                  // head-dim column (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    for (int n = 0; n < n_steps; ++n) {
      if (!warp_wait(wd, &bars.dq_full, n & 1)) break;
      tc_fence_after_sync();
      uint32_t r0[32], r1[32];
      tmem_ld32(tmem + lane_base + kColDQ, r0);
      tmem_ld32(tmem + lane_base + kColDQ + 32, r1);
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars.dq_empty);
      const int h = step_head(n);
      const int qi = step_qtile(n);
      float* base = p.dq + ((static_cast<int64_t>(b) * p.q_len + qi * kBQ) * p.Hq + h) * kD + dcol;
      const int64_t rstride = static_cast<int64_t>(p.Hq) * kD;
#pragma unroll
      for (int c = 0; c < 32; ++c) atomicAdd(base + c * rstride, p.scale * __uint_as_float(r0[c]));
#pragma unroll
      for (int c = 0; c < 32; ++c) atomicAdd(base + (c + 32) * rstride, p.scale * __uint_as_float(r1[c]));
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_bwd_bf16(const ChunkGeom& g, const Bf16BwdMaps& maps, const float* lse,
                            const float* delta, float* dq, float* dk, float* dv, unsigned int* err,
                            cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(bwd_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemAlloc);
  if (e != cudaSuccess) return e;
  BwdParams p;
  p.B = g.B;
  p.Hq = g.Hq;
  p.Hkv = g.Hkv;
  p.G = g.G;
  p.q_len = static_cast<int>(g.q_len);
  p.T = static_cast<int>(g.T);
  p.q_start = static_cast<int>(g.q_start);
  p.kv_begin = static_cast<int>(g.kv_begin);
  p.n_ktiles = static_cast<int>((g.q_start + g.q_len - g.kv_begin) / kBK);
  p.scale = g.scale;
  p.scale_log2 = g.scale * kLog2e;
  p.lse = lse;
  p.delta = delta;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.err = err;
  const unsigned grid = static_cast<unsigned>(p.n_ktiles) * g.Hkv * g.B;
  bwd_bf16_kernel<<<grid, kThreads, kSmemAlloc, s>>>(maps.q, maps.k, maps.v, maps.d_o, p);
  return cudaGetLastError();
}

}  // namespace seqattn
