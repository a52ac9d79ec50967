// wgrad_bf16.cu -- projection weight gradient of a chunk's rows on the tensor
// cores, the step after the attention path (SeCO review page, major comment 1
// on Algorithm 2: once chunk i's cache gradient is complete, chunk i's graph
// -- here the Q/K/V projections X = H W -- is backpropagated):
//   dW[d_model, n] += sum over batch entries b and rows r of H[b, r]^T G[b, r]
// with H bf16 (the projections' input) and G float32 (dQ, or the finished
// dK / dV rows), G rounded to bf16 (nearest even) on the way in, float32
// accumulation.
//
// One CTA owns a tile of 128 columns of dW (128 of the n outputs) by 256 rows
// (256 of the d_model inputs) and runs the whole row range through it:
//   D[j, m] = sum_r G[r, j] H[r, m]   (= dW[m, j]),   M = 128 (j), N = 256 (m)
// as tcgen05 MMAs with the A operand (G^T, bf16 pairs) in tensor memory and
// the B operand (H, MN-major) in shared memory.  Both inputs arrive by TMA,
// 64 rows per stage: H (bf16, 128-byte swizzle) and G (fp32, plain rows).  G
// needs rounding, so converter warps read their column of the fp32 stage,
// round it to bf16 pairs and store them into a ring of A slots in TMEM; no
// converted copy of G exists in HBM.
//   warp 0      TMA producer (H and G, 3 stages of 64 KB)
//   warp 1      TMEM owner + MMA issuer (4 MMAs M128 N256 K16 per stage)
//   warps 2..9  converters, one per TMEM lane quadrant and stage parity; then
//               the epilogue: D is written transposed into shared memory (the
//               idle stage ring) as dW's [256 m][128 j] tile, and one thread
//               adds it into dW with TMA reduce-adds, so the read-modify-write
//               of dW runs in L2, overlapped with the next CTAs' work
// TMEM (512 columns): the accumulator D in [0, 256), four A slots of 32
// columns (64 rows as bf16 pairs) in [256, 384).
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace seqattn {
namespace {

constexpr int kBM = 128;               // dW columns (n) per CTA: the MMA's M
constexpr int kBN = 256;               // dW rows (d_model) per CTA: the MMA's N
constexpr int kBK = 64;                // rows (tokens) per stage
constexpr int kStages = 3;             // shared-memory ring of H and G
constexpr int kASlots = 4;             // TMEM ring of converted G
constexpr int kConvWarps = 8;          // two per TMEM lane quadrant
constexpr int kThreads = 32 * (2 + kConvWarps);
constexpr int kBoxBytes = kBK * 128;   // one 64-column block of H: 64 rows x 128 B
constexpr int kHBytes = (kBN / 64) * kBoxBytes;       // 32 KB
constexpr int kGBytes = kBK * kBM * 4;                // 32 KB: 64 rows x 128 fp32
constexpr int kStageBytes = kHBytes + kGBytes;
constexpr int kOutRows = 32;                          // dW rows per TMA reduce box
constexpr int kSmemAlloc = kStages * kStageBytes + 1024;
static_assert(kBN * kBM * 4 <= kStages * kStageBytes, "the dW tile is staged in the ring");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColAcc = 0;
constexpr uint32_t kColA = 256;        // A slot s at kColA + 32 s

struct WgradParams {
  int B;
  int row_begin;
  int rows;             // row_end - row_begin
  int blocks;           // ceil(rows / 64): stages per batch entry
  int d_model, n;
  unsigned int* err;
  long long wait_cycles;
};

struct WgradBarriers {
  uint64_t full[kStages], empty[kStages];
  uint64_t a_full[kASlots], a_empty[kASlots];
  uint64_t acc_full;
  uint64_t mma_final;
};

__device__ __forceinline__ bool warp_wait(Watchdog& wd, uint64_t* bar, uint32_t parity) {
  const bool ok = wd.wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// MN-major B operand (H: 64 rows of K, 256 columns of N in four 64-column
// blocks 8 KB apart): K-step ks (16 rows) starts 2048 bytes further.
__host__ __device__ constexpr uint32_t mnmajor_off(int ks) { return static_cast<uint32_t>((ks * 2048) >> 4); }

__global__ void __launch_bounds__(kThreads, 1)
    wgrad_bf16_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_g,
                      const __grid_constant__ CUtensorMap map_dw, const WgradParams p) {
  if (error_already_set(p.err)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ WgradBarriers bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  Watchdog wd(&abort_flag, p.err, p.wait_cycles);

  // tile: dW columns [n0, n0 + 128), rows [m0, m0 + 256); m fastest, so a
  // wave shares the n-tiles' G rows in L2
  const int m_tiles = (p.d_model + kBN - 1) / kBN;
  const int n0 = (blockIdx.x / m_tiles) * kBM;
  const int m0 = (blockIdx.x % m_tiles) * kBN;
  const int n_st = p.B * p.blocks;       // stages: (batch entry, 64-row block)

  const int warp = warp_id();
  const int lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars.full[i], 1);
      mbar_init(&bars.empty[i], 1);
    }
    for (int i = 0; i < kASlots; ++i) {
      mbar_init(&bars.a_full[i], 4 * 32);    // the four converter warps of the slot's parity
      mbar_init(&bars.a_empty[i], 1);
    }
    mbar_init(&bars.acc_full, 1);
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
  int n_issued = 0;                      // producer: stages issued so far

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&map_h);
      prefetch_tensormap(&map_g);
      prefetch_tensormap(&map_dw);
      for (int s = 0; s < n_st; ++s) {
        const int st = s % kStages;
        if (!wd.wait(&bars.empty[st], ((s / kStages) & 1) ^ 1)) break;
        const int b = s / p.blocks;
        const int r0 = p.row_begin + (s - b * p.blocks) * kBK;
        uint8_t* stage = smem + st * kStageBytes;
        mbar_arrive_expect_tx(&bars.full[st], kStageBytes);
#pragma unroll
        for (int blk = 0; blk < kBN / 64; ++blk)
          tma_load_3d(stage + blk * kBoxBytes, &map_h, &bars.full[st], m0 + 64 * blk, r0, b);
        tma_load_3d(stage + kHBytes, &map_g, &bars.full[st], n0, r0, b);
        n_issued = s + 1;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_bf16(kBM, kBN, false, true);
      const uint64_t b_desc0 = make_desc_sw128(smem_u32(smem), kBoxBytes, 1024);
      bool ok = true;
      for (int s = 0; ok && s < n_st; ++s) {
        const int st = s % kStages;
        const int sl = s % kASlots;
        if (!(ok = wd.wait(&bars.full[st], (s / kStages) & 1))) break;
        if (!(ok = wd.wait(&bars.a_full[sl], (s / kASlots) & 1))) break;
        tc_fence_after_sync();
        const uint64_t bd = b_desc0 + static_cast<uint64_t>(st * (kStageBytes >> 4));
        const uint32_t a = tmem + kColA + 32u * sl;
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks)
          umma_bf16_ts(tmem + kColAcc, a + 8u * ks, bd + mnmajor_off(ks), idesc, (s > 0 || ks > 0) ? 1u : 0u);
        umma_commit(&bars.empty[st]);         // H and G of the stage consumed (G before a_full)
        umma_commit(&bars.a_empty[sl]);
      }
      if (ok) umma_commit(&bars.acc_full);
      umma_commit(&bars.mma_final);
      wd.drain(&bars.mma_final, 0, 4000000);
    }
  } else {
    // ------------------------------------------------------------ converters
    const int quad = warp & 3;
    const int par = (warp - 2) >> 2;                    // stages s with s % 2 == par
    const int jl = quad * 32 + lane;                    // tile column (TMEM lane) of this thread
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = true;
    for (int s = par; s < n_st; s += 2) {
      const int st = s % kStages;
      const int sl = s % kASlots;
      if (!(ok = warp_wait(wd, &bars.a_empty[sl], ((s / kASlots) & 1) ^ 1))) break;
      if (!(ok = warp_wait(wd, &bars.full[st], (s / kStages) & 1))) break;
      const int b = s / p.blocks;
      const int valid = min(kBK, p.rows - (s - b * p.blocks) * kBK);   // rows inside the range
      // this thread's column of the fp32 stage: 64 rows, 128 floats apart
      // (lanes read consecutive words, no bank conflicts); rows past the
      // range become zeros, so whatever H holds there adds nothing
      const float* gs = reinterpret_cast<const float*>(smem + st * kStageBytes + kHBytes) + jl;
      uint32_t pk[32];
      if (valid == kBK) {
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(gs[(2 * c) * kBM], gs[(2 * c + 1) * kBM]);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          pk[c] = pack_bf16x2(2 * c < valid ? gs[(2 * c) * kBM] : 0.f, 2 * c + 1 < valid ? gs[(2 * c + 1) * kBM] : 0.f);
      }
      tmem_st32(tmem + lane_base + kColA + 32u * sl, pk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars.a_full[sl]);
    }
    // ---- epilogue: once every MMA has completed the stage ring is idle (all
    // issued copies were consumed); D goes there transposed, as the dW tile
    // [256 m][128 j] fp32, this warp pair's half of the m rows each
    if (ok) ok = warp_wait(wd, &bars.acc_full, 0);
    if (ok) {
      tc_fence_after_sync();
      float* out = reinterpret_cast<float*>(smem);
#pragma unroll 1
      for (int c0 = par * (kBN / 2); c0 < (par + 1) * (kBN / 2); c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + kColAcc + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) out[(c0 + c) * kBM + jl] = __uint_as_float(r[c]);
      }
      fence_proxy_async_smem();
    }
    named_barrier_sync(1, kConvWarps * 32);
    if (ok && !wd.aborted() && warp == 2 && lane == 0) {
      // dW rows [m0, m0 + 256) x columns [n0, n0 + 128) += the staged tile;
      // the parts past d_model or n are clipped by the tensor map
#pragma unroll 1
      for (int k = 0; k < kBN / kOutRows; ++k)
        tma_reduce_add_3d(&map_dw, smem + k * kOutRows * kBM * 4, n0, m0 + k * kOutRows, 0);
      bulk_commit_group();
      bulk_wait_group_read<0>();            // the tile has been read before the CTA's smem goes away
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (wd.aborted()) {
    // a wait ran out: let the copies already in flight land first
    if (warp == 0 && lane == 0) {
      for (int st = 0; st < kStages && st < n_issued; ++st) {
        const int last = st + kStages * ((n_issued - 1 - st) / kStages);
        wd.drain(&bars.full[st], (last / kStages) & 1, 1000000);
      }
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_wgrad_bf16(const WgradMaps& maps, int32_t batch, int64_t row_begin, int64_t row_end,
                              int32_t d_model, int32_t n, unsigned int* err, long long wait_cycles,
                              cudaStream_t s) {
  WgradParams p;
  p.B = batch;
  p.row_begin = static_cast<int>(row_begin);
  p.rows = static_cast<int>(row_end - row_begin);
  p.blocks = (p.rows + kBK - 1) / kBK;
  p.d_model = d_model;
  p.n = n;
  p.err = err;
  p.wait_cycles = wait_cycles;
  cudaError_t e = cudaFuncSetAttribute(wgrad_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(((n + kBM - 1) / kBM) * ((d_model + kBN - 1) / kBN));
  wgrad_bf16_kernel<<<grid, kThreads, kSmemAlloc, s>>>(maps.h, maps.g, maps.dw, p);
  return cudaGetLastError();
}

}  // namespace seqattn
