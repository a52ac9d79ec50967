// fwd_bf16.cu -- tensor-core forward of one chunk (bf16 in, fp32 accumulate).
//
// Operation: chunk i's queries attend the cached prefix, O^(i) =
// softmax(scale Q^(i) K^(:i)^T, causal) V^(:i), plus the row logsumexp
// (StreamBP review page: Property 3.1 and the partitioned attention of
// Eqs. (12)-(14) named in its "Circularity Check"; the stored row statistic
// M^(i) of the StreamBP verdict page's stored-activation list).
//
// One CTA owns one 128-row query tile of one head and streams the head's
// key/value tiles [kv_begin, q0 + 128) through shared memory:
//   warp 0      TMA producer: Q once, then K/V tiles into 2-stage rings
//   warp 1      TMEM owner + MMA issuer (one thread): S = Q K^T, O += P V
//   warps 2..5  softmax: S row from TMEM -> online max/sum -> P (bf16) into
//               shared memory; rare O rescale in TMEM; epilogue O/l, LSE
// S is double-buffered in TMEM so the next QK^T overlaps this tile's
// softmax.  Only the last (diagonal) key tile carries the causal mask; the
// prefix tiles are unmasked.  The running max is rescaled lazily: O and l
// are only corrected when a row max grows by more than 2^8, which keeps P
// below 256 (exact in fp32/bf16 range) and skips almost every TMEM
// read-modify-write of O.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace seqattn {
namespace {

constexpr int kBM = 128;             // query rows per CTA
constexpr int kBN = 128;             // keys per tile
constexpr int kD = 128;              // head dim
constexpr int kTileBytes = kBM * kD * 2;  // 32 KB: one 128x128 bf16 tile
constexpr int kHalfBytes = kTileBytes / 2;  // one 64-column (128-byte) block
constexpr int kThreads = 192;        // 6 warps

// shared memory carve-up (bytes from the 1024-aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;        // 2 stages
constexpr int kOffV = kOffK + 2 * kTileBytes;    // 2 stages
constexpr int kOffP = kOffV + 2 * kTileBytes;    // 2 buffers
constexpr int kSmemBytes = kOffP + 2 * kTileBytes;
constexpr int kSmemAlloc = kSmemBytes + 1024;    // + alignment slack

// TMEM columns: S buffers at 0 and 128, O at 256.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct FwdParams {
  int B, Hq, Hkv, G;
  int q_len, T;
  int q_start, kv_begin;
  int n_qtiles;
  float scale_log2;
  __nv_bfloat16* o;
  float* lse;
  unsigned int* err;
};

struct FwdBarriers {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t mma_final;
};

// All 32 lanes wait; the warp proceeds only if every lane saw the phase, so
// the warp stays converged for the .sync.aligned tcgen05 instructions.
__device__ __forceinline__ bool warp_wait(Watchdog& wd, uint64_t* bar, uint32_t parity) {
  const bool ok = wd.wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile_addr, int ks) {
  // K-major 128x128 bf16 tile = two 64-column blocks of 128 rows x 128 B.
  // K-step ks (16 elements) -> block ks/4, byte offset 32*(ks%4) in the row.
  return make_desc_sw128(tile_addr + (ks >> 2) * kHalfBytes + (ks & 3) * 32, 16, 1024);
}

__device__ __forceinline__ uint64_t v_mn_desc(uint32_t tile_addr, int ks) {
  // V tile [128 keys][128 d] used as the MN-major B operand (N = d, K = keys):
  // 8-key groups of 1024 B along K, the two 64-wide d blocks 16 KB apart.
  return make_desc_sw128(tile_addr + ks * 2048, kHalfBytes, 1024);
}

__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const FwdParams p) {
  if (error_already_set(p.err)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ FwdBarriers bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  Watchdog wd{&abort_flag, p.err};

  // ---- work item: (b, kv group, head in group, q tile), q tile fastest and
  // heaviest (longest key range) first.
  int idx = blockIdx.x;
  const int qt = p.n_qtiles - 1 - (idx % p.n_qtiles);
  idx /= p.n_qtiles;
  const int h = idx % p.Hq;
  const int b = idx / p.Hq;
  const int g = h / p.G;
  const int q0 = p.q_start + qt * kBM;                 // absolute row of query 0
  const int n_kv = (q0 + kBM - p.kv_begin) / kBN;      // key tiles, last one diagonal

  const int warp = warp_id();
  const int lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars.q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 4 * 32);
      mbar_init(&bars.pv_done[i], 1);
    }
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

  const uint32_t sQ = smem_u32(smem + kOffQ);
  const uint32_t sK = smem_u32(smem + kOffK);
  const uint32_t sV = smem_u32(smem + kOffV);
  const uint32_t sP = smem_u32(smem + kOffP);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      const int qrow = b * p.q_len + qt * kBM;
      mbar_arrive_expect_tx(&bars.q_full, kTileBytes);
      tma_load_3d(smem + kOffQ, &map_q, &bars.q_full, 0, h, qrow);
      tma_load_3d(smem + kOffQ + kHalfBytes, &map_q, &bars.q_full, 64, h, qrow);
      int issued[2] = {0, 0};
      for (int t = 0; t < n_kv; ++t) {
        const int st = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        const int krow = b * p.T + p.kv_begin + t * kBN;
        if (!wd.wait(&bars.k_empty[st], ph ^ 1)) break;
        mbar_arrive_expect_tx(&bars.k_full[st], kTileBytes);
        tma_load_3d(smem + kOffK + st * kTileBytes, &map_k, &bars.k_full[st], 0, g, krow);
        tma_load_3d(smem + kOffK + st * kTileBytes + kHalfBytes, &map_k, &bars.k_full[st], 64, g, krow);
        if (!wd.wait(&bars.v_empty[st], ph ^ 1)) { issued[st] = t + 1; break; }
        mbar_arrive_expect_tx(&bars.v_full[st], kTileBytes);
        tma_load_3d(smem + kOffV + st * kTileBytes, &map_v, &bars.v_full[st], 0, g, krow);
        tma_load_3d(smem + kOffV + st * kTileBytes + kHalfBytes, &map_v, &bars.v_full[st], 64, g, krow);
        issued[st] = t + 1;
      }
      if (wd.aborted()) {
        // let copies already in flight land before the CTA's smem goes away
        wd.drain(&bars.q_full, 0, 1000000);
        for (int st = 0; st < 2; ++st) {
          if (issued[st] > 0) {
            const uint32_t ph = ((issued[st] - 1) >> 1) & 1;
            wd.drain(&bars.k_full[st], ph, 1000000);
            wd.drain(&bars.v_full[st], ph, 1000000);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = make_idesc_bf16(kBM, kBN, false, false);
      const uint32_t idesc_o = make_idesc_bf16(kBM, kD, false, true);
      bool ok = wd.wait(&bars.q_full, 0);
      auto issue_pv = [&](int u) -> bool {
        const int su = u & 1;
        const uint32_t phu = (u >> 1) & 1;
        if (!wd.wait(&bars.v_full[su], phu)) return false;
        if (!wd.wait(&bars.p_full[su], phu)) return false;
        tc_fence_after_sync();
        const uint32_t pa = sP + su * kTileBytes;
        const uint32_t va = sV + su * kTileBytes;
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
          umma_bf16_ss(tmem + kColO, kmajor_desc(pa, ks), v_mn_desc(va, ks), idesc_o,
                       (u > 0 || ks > 0) ? 1u : 0u);
        umma_commit(&bars.pv_done[su]);
        umma_commit(&bars.v_empty[su]);
        return true;
      };
      for (int t = 0; ok && t < n_kv; ++t) {
        const int st = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        if (!(ok = wd.wait(&bars.k_full[st], ph))) break;
        tc_fence_after_sync();
        const uint32_t ka = sK + st * kTileBytes;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks)
          umma_bf16_ss(tmem + kColS + st * kBN, kmajor_desc(sQ, ks), kmajor_desc(ka, ks), idesc_s,
                       ks > 0 ? 1u : 0u);
        umma_commit(&bars.s_full[st]);
        umma_commit(&bars.k_empty[st]);
        if (t >= 1) ok = issue_pv(t - 1);
      }
      if (ok) issue_pv(n_kv - 1);
      // every MMA this thread issued has completed before TMEM is released
      umma_commit(&bars.mma_final);
      wd.drain(&bars.mma_final, 0, 4000000);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;                   // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;            // query row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    float m_run = -INFINITY;                     // running max, log2 units
    float l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < n_kv; ++t) {
      const int st = t & 1;
      const uint32_t ph = (t >> 1) & 1;
      if (!(ok = warp_wait(wd, &bars.s_full[st], ph))) break;
      tc_fence_after_sync();
      float s[kBN];
#pragma unroll
      for (int c0 = 0; c0 < kBN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + kColS + st * kBN + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) s[c0 + j] = __uint_as_float(r[j]) * p.scale_log2;
      }
      if (t == n_kv - 1) {
        // diagonal tile: key c (absolute q0 + c) is visible to row r iff c <= r
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c > row) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < kBN; ++c) mx = fmaxf(mx, s[c]);
      const bool need = mx > m_run + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mx : m_run;
        const float alpha = ex2(m_run - m_new);  // 0 on the first tile, 1 if !need
        l_run *= alpha;
        m_run = m_new;
        if (t > 0) {
          // O holds PV_0..PV_{t-1}: wait for PV_{t-1}, then scale O by alpha
          const int u = t - 1;
          if (!(ok = warp_wait(wd, &bars.pv_done[u & 1], (u >> 1) & 1))) break;
          tc_fence_after_sync();
#pragma unroll
          for (int c0 = 0; c0 < kD; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + kColO + c0, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
            tmem_st32(tmem + lane_base + kColO + c0, r);
          }
          tmem_st_wait();
        }
      }
      // P buffer st was last read by PV_{t-2}
      if (t >= 2) {
        const int u = t - 2;
        if (!(ok = warp_wait(wd, &bars.pv_done[u & 1], (u >> 1) & 1))) break;
      }
      const uint32_t prow = sP + st * kTileBytes + row * 128;
      const uint32_t sw = static_cast<uint32_t>(row & 7);
#pragma unroll
      for (int ci = 0; ci < kBN / 8; ++ci) {
        const int c = ci * 8;
        float e[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          e[j] = ex2(s[c + j] - m_run);
          l_run += e[j];
        }
        const uint32_t addr = prow + (ci >> 3) * kHalfBytes + (((ci & 7) ^ sw) << 4);
        st_shared_v4(addr, pack_bf16x2(e[0], e[1]), pack_bf16x2(e[2], e[3]),
                     pack_bf16x2(e[4], e[5]), pack_bf16x2(e[6], e[7]));
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&bars.p_full[st]);
    }
    if (ok) {
      const int u = n_kv - 1;
      ok = warp_wait(wd, &bars.pv_done[u & 1], (u >> 1) & 1);
    }
    if (ok) {
      tc_fence_after_sync();
      const float inv = 1.f / l_run;
      const int qrow = qt * kBM + row;
      uint4* orow = reinterpret_cast<uint4*>(p.o + ((static_cast<int64_t>(b) * p.q_len + qrow) * p.Hq + h) * kD);
#pragma unroll
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + kColO + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(r[j + 0]) * inv, __uint_as_float(r[j + 1]) * inv);
          v.y = pack_bf16x2(__uint_as_float(r[j + 2]) * inv, __uint_as_float(r[j + 3]) * inv);
          v.z = pack_bf16x2(__uint_as_float(r[j + 4]) * inv, __uint_as_float(r[j + 5]) * inv);
          v.w = pack_bf16x2(__uint_as_float(r[j + 6]) * inv, __uint_as_float(r[j + 7]) * inv);
          orow[(c0 + j) / 8] = v;
        }
      }
      p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.q_len + qrow] = (m_run + __log2f(l_run)) * kLn2;
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

cudaError_t launch_fwd_bf16(const ChunkGeom& g, const Bf16FwdMaps& maps, void* o, float* lse,
                            unsigned int* err, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemAlloc);
  if (e != cudaSuccess) return e;
  FwdParams p;
  p.B = g.B;
  p.Hq = g.Hq;
  p.Hkv = g.Hkv;
  p.G = g.G;
  p.q_len = static_cast<int>(g.q_len);
  p.T = static_cast<int>(g.T);
  p.q_start = static_cast<int>(g.q_start);
  p.kv_begin = static_cast<int>(g.kv_begin);
  p.n_qtiles = static_cast<int>(g.q_len / kBM);
  p.scale_log2 = g.scale * kLog2e;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.err = err;
  const unsigned grid = static_cast<unsigned>(p.n_qtiles) * g.Hq * g.B;
  fwd_bf16_kernel<<<grid, kThreads, kSmemAlloc, s>>>(maps.q, maps.k, maps.v, p);
  return cudaGetLastError();
}

}  // namespace seqattn
