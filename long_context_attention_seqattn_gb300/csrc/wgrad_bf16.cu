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
// 64 rows per stage, each in a ring of its own: H (bf16, 128-byte swizzle,
// 32 KB a stage) is held until the stage's MMAs have read it; G (fp32, plain
// rows, 32 KB a stage) only until the converter warps have read it, since
// they round it to bf16 pairs and store those into a ring of A slots in TMEM.
// No converted copy of G exists in HBM.
//   warp 0      TMA producer of H (3 stages)
//   warp 1      TMEM owner + MMA issuer (4 MMAs M128 N256 K16 per stage)
//   warps 2..9  converters: two groups of four (one warp per TMEM lane
//               quadrant); group p converts rows [32p, 32p + 32) of EVERY
//               stage, in order.  (Handing whole stages to the groups in turn
//               would let a group wait on a stage barrier two phases ahead,
//               where the parity of an older phase reads as complete.)  Then
//               the epilogue: D is written transposed into shared memory (the
//               idle rings) as dW's [256 m][128 j] tile, and one thread adds it
//               into dW with TMA reduce-adds, so the read-modify-write of dW
//               runs in L2, overlapped with the next CTAs' work
//   warp 10     TMA producer of G (3 stages)
// TMEM (512 columns): the accumulator D in [0, 256), four A slots of 32
// columns (64 rows as bf16 pairs) in [256, 384).
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace seqattn {
namespace {

constexpr int kBM = 128;               // dW columns (n) per CTA: the MMA's M
constexpr int kBN = 256;               // dW rows (d_model) per CTA: the MMA's N
constexpr int kBK = kWgradStageRows;   // rows (tokens) per stage
constexpr int kHStages = 3;            // shared-memory ring of H
constexpr int kGStages = 3;            // shared-memory ring of G
constexpr int kASlots = 4;             // TMEM ring of converted G
constexpr int kPairs = kBK / 2;        // TMEM columns of one A slot (rows as bf16 pairs)
static_assert(kPairs == 32 || kPairs == 16 || kPairs == 8, "stages of 64, 32 or 16 rows");
constexpr int kConvWarps = 8;          // kConvGroups warps per TMEM lane quadrant
constexpr int kConvGroups = kConvWarps / 4;   // groups of four warps, one per lane quadrant
constexpr int kGroupRows = kBK / kConvGroups; // rows of every stage converted by one group
constexpr int kGroupPairs = kGroupRows / 2;   // their TMEM columns (bf16 pairs)
static_assert(kGroupPairs == 32 || kGroupPairs == 16 || kGroupPairs == 8, "tcgen05.st widths");
constexpr int kGWarp = 2 + kConvWarps;          // producer of G
constexpr int kThreads = 32 * (3 + kConvWarps);
constexpr int kBoxBytes = kBK * 128;   // one 64-column block of H: kBK rows x 128 B
constexpr int kHBytes = (kBN / 64) * kBoxBytes;       // 32 KB
constexpr int kGBytes = kBK * kBM * 4;                // 32 KB: kBK rows x 128 fp32
constexpr int kOffG = kHStages * kHBytes;
constexpr int kOutRows = 32;                          // dW rows per TMA reduce box
constexpr int kSmemAlloc = kOffG + kGStages * kGBytes + 1024;
static_assert(kBN * kBM * 4 <= kOffG + kGStages * kGBytes, "the dW tile is staged in the rings");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColAcc = 0;
constexpr uint32_t kColA = 256;        // A slot s at kColA + kPairs s
static_assert(kColA + kASlots * kPairs <= kTmemCols, "the A slots fit in TMEM");

struct WgradParams {
  int B;
  int row_begin;
  int rows;             // row_end - row_begin
  int blocks;           // ceil(rows / kBK): stages per batch entry
  int d_model, n;
  unsigned int* err;
  long long wait_cycles;
};

struct WgradBarriers {
  uint64_t h_full[kHStages], h_empty[kHStages];
  uint64_t g_full[kGStages], g_empty[kGStages];
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
  const int n_st = p.B * p.blocks;       // stages: (batch entry, kBK-row block)

  const int warp = warp_id();
  const int lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < kHStages; ++i) {
      mbar_init(&bars.h_full[i], 1);
      mbar_init(&bars.h_empty[i], 1);
    }
    for (int i = 0; i < kGStages; ++i) {
      mbar_init(&bars.g_full[i], 1);
      mbar_init(&bars.g_empty[i], kConvWarps * 32);
    }
    for (int i = 0; i < kASlots; ++i) {
      mbar_init(&bars.a_full[i], kConvWarps * 32);   // every converter warp
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
  int n_issued = 0;                      // producers: stages issued so far (each its own)

  if (warp == 0 || warp == kGWarp) {
    // ------------------------------------------------------------ producers
    if (lane == 0) {
      const bool is_h = warp == 0;
      const int ns = is_h ? kHStages : kGStages;
      uint64_t* full = is_h ? bars.h_full : bars.g_full;
      uint64_t* empty = is_h ? bars.h_empty : bars.g_empty;
      prefetch_tensormap(is_h ? &map_h : &map_g);
      if (is_h) prefetch_tensormap(&map_dw);
      for (int s = 0; s < n_st; ++s) {
        const int st = s % ns;
        if (!wd.wait(&empty[st], ((s / ns) & 1) ^ 1)) break;
        const int b = s / p.blocks;
        const int r0 = p.row_begin + (s - b * p.blocks) * kBK;
        if (is_h) {
          uint8_t* stage = smem + st * kHBytes;
          mbar_arrive_expect_tx(&full[st], kHBytes);
#pragma unroll
          for (int blk = 0; blk < kBN / 64; ++blk)
            tma_load_3d(stage + blk * kBoxBytes, &map_h, &full[st], m0 + 64 * blk, r0, b);
        } else {
          mbar_arrive_expect_tx(&full[st], kGBytes);
          tma_load_3d(smem + kOffG + st * kGBytes, &map_g, &full[st], n0, r0, b);
        }
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
        const int st = s % kHStages;
        const int sl = s % kASlots;
        if (!(ok = wd.wait(&bars.h_full[st], (s / kHStages) & 1))) break;
        if (!(ok = wd.wait(&bars.a_full[sl], (s / kASlots) & 1))) break;
        tc_fence_after_sync();
        const uint64_t bd = b_desc0 + static_cast<uint64_t>(st * (kHBytes >> 4));
        const uint32_t a = tmem + kColA + static_cast<uint32_t>(kPairs * sl);
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks)
          umma_bf16_ts(tmem + kColAcc, a + 8u * ks, bd + mnmajor_off(ks), idesc, (s > 0 || ks > 0) ? 1u : 0u);
        umma_commit(&bars.h_empty[st]);       // H of the stage consumed
        umma_commit(&bars.a_empty[sl]);
      }
      if (ok) umma_commit(&bars.acc_full);
      umma_commit(&bars.mma_final);
      wd.drain(&bars.mma_final, 0, 4000000);
    }
  } else {
    // ------------------------------------------------------------ converters
    const int quad = warp & 3;
    const int par = (warp - 2) >> 2;                    // rows [par kGroupRows, +kGroupRows) of each stage
    const int jl = quad * 32 + lane;                    // tile column (TMEM lane) of this thread
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = true;
    // Every converter warp takes every stage, in order, so each of its waits
    // is for the phase right after the one it saw last (a warp that skipped
    // stages could see the parity of an older phase and pass too early).
    for (int s = 0; s < n_st; ++s) {
      const int st = s % kGStages;
      const int sl = s % kASlots;
      if (!(ok = warp_wait(wd, &bars.a_empty[sl], ((s / kASlots) & 1) ^ 1))) break;
      if (!(ok = warp_wait(wd, &bars.g_full[st], (s / kGStages) & 1))) break;
      const int b = s / p.blocks;
      // rows of this group's share that lie inside the range
      const int valid = min(kBK, p.rows - (s - b * p.blocks) * kBK) - par * kGroupRows;
      // this thread's column of the fp32 stage: kBK rows, 128 floats apart
      // (lanes read consecutive words, no bank conflicts); rows past the
      // range become zeros, so whatever H holds there adds nothing
      const float* gs = reinterpret_cast<const float*>(smem + kOffG + st * kGBytes) + par * kGroupRows * kBM + jl;
      uint32_t pk[kGroupPairs];
      if (valid >= kGroupRows) {
#pragma unroll
        for (int c = 0; c < kGroupPairs; ++c) pk[c] = pack_bf16x2(gs[(2 * c) * kBM], gs[(2 * c + 1) * kBM]);
      } else {
#pragma unroll
        for (int c = 0; c < kGroupPairs; ++c)
          pk[c] = pack_bf16x2(2 * c < valid ? gs[(2 * c) * kBM] : 0.f, 2 * c + 1 < valid ? gs[(2 * c + 1) * kBM] : 0.f);
      }
      mbar_arrive(&bars.g_empty[st]);          // this thread's part of the G stage has been read
      const uint32_t slot = tmem + lane_base + kColA + static_cast<uint32_t>(kPairs * sl + kGroupPairs * par);
      if constexpr (kGroupPairs == 32)
        tmem_st32(slot, *reinterpret_cast<const uint32_t(*)[32]>(pk));
      else if constexpr (kGroupPairs == 16)
        tmem_st16(slot, *reinterpret_cast<const uint32_t(*)[16]>(pk));
      else
        tmem_st8(slot, *reinterpret_cast<const uint32_t(*)[8]>(pk));
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars.a_full[sl]);
    }
    // ---- epilogue: once every MMA has completed both rings are idle (every
    // issued copy was consumed); D goes there transposed, as the dW tile
    // [256 m][128 j] fp32, each converter group a 1/kConvGroups share of the m rows
    if (ok) ok = warp_wait(wd, &bars.acc_full, 0);
    if (ok) {
      tc_fence_after_sync();
      float* out = reinterpret_cast<float*>(smem);
#pragma unroll 1
      for (int c0 = par * (kBN / kConvGroups); c0 < (par + 1) * (kBN / kConvGroups); c0 += 32) {
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
    if ((warp == 0 || warp == kGWarp) && lane == 0) {
      const int ns = warp == 0 ? kHStages : kGStages;
      uint64_t* full = warp == 0 ? bars.h_full : bars.g_full;
      for (int st = 0; st < ns && st < n_issued; ++st) {
        const int last = st + ns * ((n_issued - 1 - st) / ns);
        wd.drain(&full[st], (last / ns) & 1, 1000000);
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
