// fwd_bf16.cu -- tensor-core forward of one chunk (bf16 in, fp32 accumulate).
//
// Operation: chunk i's queries attend the cached prefix, O^(i) =
// softmax(scale Q^(i) K^(:i)^T, causal) V^(:i), plus the row logsumexp
// (StreamBP review page: Property 3.1 and the partitioned attention of
// Eqs. (12)-(14) named in its "Circularity Check"; the stored row statistic
// M^(i) of the StreamBP verdict page's stored-activation list).
//
// One CTA owns one 128-row query tile of one head (head dim D = 64 or 128,
// a template parameter) and streams the head's key/value tiles
// [kv_begin, min(q0 + 128, q_end)) through shared memory:
//   warp 0      TMA producer of Q (once) and K tiles (3-stage ring)
//   warp 10     TMA producer of V tiles (its own 3-stage ring, so a K load
//               never queues behind a V slot that frees later)
//   warp 1      TMEM owner + MMA issuer of S = Q K^T (SS)
//   warp 11     MMA issuer of O_h += P_h V_h (A operand P_h read from TMEM);
//               two issuing threads because one thread keeps only about one
//               tcgen05.mma in flight per ~90 cycles
//   warps 2..9  softmax, two warps per TMEM lane quadrant
// Each key tile is split in two 64-key halves; softmax warp half h owns keys
// [64h, 64h + 64) of every tile for its 32 rows, with its own running max and
// sum and its own output accumulator O_h = sum P_h V_h in TMEM.  The two
// halves are merged once, in the epilogue (O = (O_0 2^m0 + O_1 2^m1) /
// (l_0 2^m0 + l_1 2^m1)), so the per-tile softmax needs no exchange between
// warps, and each SM sub-partition runs two softmax warps.  P is written back
// into TMEM (over the S values just read) and never touches shared memory.
// TMEM: S double-buffered (2 x 128 columns), O_0 and O_1 (128 columns each).
// Only key tiles that reach past the tile's first query row carry the causal
// mask (one or two tiles, since chunks may start anywhere).  The running
// maxima are rescaled lazily: O_h and l_h are only corrected when a row max
// grows by more than 2^8 (P stays below 256).  Every wait sleeps in its
// mbarrier (Watchdog::wait_sleep) rather than spinning, so waiting warps
// leave their sub-partition's issue slots to the softmax warps.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace seqattn {
namespace {

constexpr int kBM = 128;                    // query rows per CTA
constexpr int kBN = 128;                    // keys per tile
constexpr int kBlockBytes = kBM * 128;      // one 64-column (128-byte) block of a 128-row tile
constexpr int kSoftmaxWarps = 8;
constexpr int kVWarp = 2 + kSoftmaxWarps;           // V producer warp
constexpr int kPVWarp = kVWarp + 1;                 // second MMA issuer (PV)
constexpr int kThreads = 32 * (kPVWarp + 1);        // 12 warps
constexpr int kStages = 3;                          // K and V ring depth

// Head-dim dependent sizes: a 128-row tile of D bf16 columns is D/64 blocks
// of 128 rows x 128 B, and the shared memory carve-up (bytes from the
// 1024-aligned base).
template <int D>
struct FwdCfg {
  static constexpr int kTileBytes = kBM * D * 2;    // 32 KB (D = 128) or 16 KB (D = 64)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;              // kStages stages
  static constexpr int kOffV = kOffK + kStages * kTileBytes;    // kStages stages
  static constexpr int kSmemBytes = kOffV + kStages * kTileBytes;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;          // + alignment slack
};

// TMEM columns: S buffers at 0 and 128, O_0 at 256, O_1 at 384.  P of key
// half h (bf16 pairs, 32 columns) overwrites columns [64h, 64h + 32) of its S
// buffer once the softmax has read them.
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
  long long wait_cycles;
};

struct FwdBarriers {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t mma_final[2];
};

// All 32 lanes wait; the warp proceeds only if every lane saw the phase, so
// the warp stays converged for the .sync.aligned tcgen05 instructions.
__device__ __forceinline__ bool warp_wait(Watchdog& wd, uint64_t* bar, uint32_t parity) {
  const bool ok = wd.wait_sleep(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// Shared-memory descriptors are built once per tile base; a K-step moves only
// the 14-bit start-address field (16-byte units), so each MMA's operands are
// the base plus a compile-time constant -- building the full descriptor in
// front of every MMA would put a serial integer chain on the issuing thread.
// K-major 128-row bf16 tile = 64-column blocks of 128 rows x 128 B;
// K-step ks (16 elements) -> block ks/4, byte offset 32*(ks%4) in the row.
__host__ __device__ constexpr uint32_t kmajor_off(int ks) {
  return static_cast<uint32_t>(((ks >> 2) * kBlockBytes + (ks & 3) * 32) >> 4);
}
// V tile [128 keys][D] as the MN-major B operand (N = d, K = keys):
// 8-key groups of 1024 B along K, the 64-wide d blocks 16 KB apart.
__host__ __device__ constexpr uint32_t vmn_off(int ks) { return static_cast<uint32_t>((ks * 2048) >> 4); }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int kTileBytes = C::kTileBytes;
  constexpr uint32_t kTileUnits = kTileBytes >> 4;
  if (error_already_set(p.err)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ FwdBarriers bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  Watchdog wd(&abort_flag, p.err, p.wait_cycles);

  // ---- work item: (b, kv group, head in group, q tile), q tile fastest and
  // heaviest (longest key range) first.
  int idx = blockIdx.x;
  const int qt = p.n_qtiles - 1 - (idx % p.n_qtiles);
  idx /= p.n_qtiles;
  const int h = idx % p.Hq;
  const int b = idx / p.Hq;
  const int g = h / p.G;
  const int q0 = p.q_start + qt * kBM;                 // absolute row of query 0
  // keys [kv_begin, min(q0 + 128, q_end)) in 128-key tiles; rows of a partial
  // last query tile past q_end are computed on whatever the copies bring and
  // never stored
  const int q_end = p.q_start + p.q_len;
  const int n_kv = (min(q0 + kBM, q_end) - p.kv_begin + kBN - 1) / kBN;

  const int warp = warp_id();
  const int lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars.q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], kSoftmaxWarps * 32);
      mbar_init(&bars.pv_done[i], 1);
    }
    mbar_init(&bars.mma_final[0], 1);
    mbar_init(&bars.mma_final[1], 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sV = smem_u32(smem + C::kOffV);
  int n_issued = 0;  // producers: tiles issued into their ring so far

  if (warp == 0 || warp == kVWarp) {
    // ------------------------------------------------------------ producers
    // warp 0 streams Q then K, warp kVWarp streams V, each into its own ring,
    // so a K tile never waits behind the slower-to-free V slot.
    if (lane == 0) {
      const bool is_k = (warp == 0);
      const CUtensorMap* map = is_k ? &map_k : &map_v;
      const int off = is_k ? C::kOffK : C::kOffV;
      uint64_t* full = is_k ? bars.k_full : bars.v_full;
      uint64_t* empty = is_k ? bars.k_empty : bars.v_empty;
      prefetch_tensormap(map);
      if (is_k) {
        prefetch_tensormap(&map_q);
        const int qrow = b * p.q_len + qt * kBM;
        mbar_arrive_expect_tx(&bars.q_full, kTileBytes);
#pragma unroll
        for (int blk = 0; blk < D / 64; ++blk)
          tma_load_3d(smem + C::kOffQ + blk * kBlockBytes, &map_q, &bars.q_full, 64 * blk, h, qrow);
      }
      for (int t = 0; t < n_kv; ++t) {
        const int st = t % kStages;
        const uint32_t ph = (t / kStages) & 1;
        const int krow = b * p.T + p.kv_begin + t * kBN;
        if (!wd.wait_sleep(&empty[st], ph ^ 1)) break;
        mbar_arrive_expect_tx(&full[st], kTileBytes);
#pragma unroll
        for (int blk = 0; blk < D / 64; ++blk)
          tma_load_3d(smem + off + st * kTileBytes + blk * kBlockBytes, map, &full[st], 64 * blk, g, krow);
        n_issued = t + 1;
      }
    }
  } else if (warp == 1 || warp == kPVWarp) {
    // ------------------------------------------------------------ MMA issuers
    // warp 1 issues the S = Q K^T products, warp kPVWarp the O_h += P_h V_h
    // products.  Their only shared TMEM columns are the S buffers: S(t)
    // overwrites P(t-2), so S(t) waits for PV(t-2) to complete.
    if (lane == 0) {
      const uint32_t idesc_s = make_idesc_bf16(kBM, kBN, false, false);
      const uint32_t idesc_o = make_idesc_bf16(kBM, D, false, true);
      const uint64_t q_desc = make_desc_sw128(sQ, 16, 1024);
      const uint64_t k_desc0 = make_desc_sw128(sK, 16, 1024);
      const uint64_t v_desc0 = make_desc_sw128(sV, kBlockBytes, 1024);
      const int me = (warp == 1) ? 0 : 1;
      bool ok = true;
      if (me == 0) {
        ok = wd.wait_sleep(&bars.q_full, 0);
        for (int t = 0; ok && t < n_kv; ++t) {
          const int ks_st = t % kStages;
          if (!(ok = wd.wait_sleep(&bars.k_full[ks_st], (t / kStages) & 1))) break;
          if (t >= 2 && !(ok = wd.wait_sleep(&bars.pv_done[t & 1], ((t - 2) >> 1) & 1))) break;
          tc_fence_after_sync();
          const uint64_t kd = k_desc0 + static_cast<uint64_t>(ks_st * kTileUnits);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            umma_bf16_ss(tmem + kColS + (t & 1) * kBN, q_desc + kmajor_off(ks), kd + kmajor_off(ks), idesc_s,
                         ks > 0 ? 1u : 0u);
          umma_commit(&bars.s_full[t & 1]);
          umma_commit(&bars.k_empty[ks_st]);
        }
      } else {
        for (int u = 0; ok && u < n_kv; ++u) {
          const int vs = u % kStages;
          if (!(ok = wd.wait_sleep(&bars.v_full[vs], (u / kStages) & 1))) break;
          if (!(ok = wd.wait_sleep(&bars.p_full[u & 1], (u >> 1) & 1))) break;
          tc_fence_after_sync();
          const uint64_t vd = v_desc0 + static_cast<uint64_t>(vs * kTileUnits);
          const uint32_t pa = tmem + kColS + (u & 1) * kBN;   // P in the S buffer, lane 0
          // O_h += P_h V[64h:64h+64, :] with P_h (bf16 pairs) at columns
          // [64h, 64h+32); the two halves' chains interleaved
#pragma unroll
          for (int j = 0; j < kBN / 16; ++j) {
            const int ks = (j >> 1) + 4 * (j & 1);
            umma_bf16_ts(tmem + kColO + (ks >> 2) * 128, pa + (ks >> 2) * 64 + (ks & 3) * 8,
                         vd + vmn_off(ks), idesc_o, (u > 0 || (ks & 3) > 0) ? 1u : 0u);
          }
          umma_commit(&bars.pv_done[u & 1]);
          umma_commit(&bars.v_empty[vs]);
        }
      }
      // every MMA this thread issued has completed before TMEM is released
      umma_commit(&bars.mma_final[me]);
      wd.drain(&bars.mma_final[me], 0, 4000000);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;                   // TMEM lane quadrant of this warp
    const int half = (warp - 2) >> 2;            // key half of every tile
    const int row = quad * 32 + lane;            // query row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t colO = tmem + lane_base + kColO + half * 128;
    const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
    float m_run = -INFINITY;                     // running max of this half, log2 units
    float l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < n_kv; ++t) {
      const int st = t & 1;
      const uint32_t ph = (t >> 1) & 1;
      if (!(ok = warp_wait(wd, &bars.s_full[st], ph))) break;
      tc_fence_after_sync();
      uint32_t ra[32], rb[32];                   // scores of keys 64h .. 64h+63
      tmem_ld32(tmem + lane_base + kColS + st * kBN + half * 64, ra);
      tmem_ld32(tmem + lane_base + kColS + st * kBN + half * 64 + 32, rb);
      tmem_ld_wait();
      const int key0 = p.kv_begin + t * kBN;              // absolute first key of the tile
      if (key0 + kBN - 1 > q0) {
        // the tile reaches past query row 0: key key0 + c is visible to row r
        // iff key0 + c <= q0 + r, i.e. c <= lim for this thread's keys
        const int lim = q0 + row - key0 - half * 64;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j > lim) ra[j] = __float_as_uint(-INFINITY);
          if (32 + j > lim) rb[j] = __float_as_uint(-INFINITY);
        }
      }
      float mx = fmax3(__uint_as_float(ra[0]), __uint_as_float(ra[1]), __uint_as_float(rb[0]));
#pragma unroll
      for (int j = 1; j < 16; ++j)
        mx = fmax3(mx, __uint_as_float(ra[2 * j]), __uint_as_float(ra[2 * j + 1]));
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (j == 0) mx = fmaxf(mx, __uint_as_float(rb[1]));
        else mx = fmax3(mx, __uint_as_float(rb[2 * j]), __uint_as_float(rb[2 * j + 1]));
      }
      mx *= p.scale_log2;                        // -inf stays -inf: no visible key in this half yet
      const bool need = mx > m_run + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mx : m_run;
        const float alpha = need ? ex2(m_run - m_new) : 1.f;  // 0 on the first visible tile
        l_run *= alpha;
        m_run = m_new;
        if (t > 0) {
          // O_h holds PV_0..PV_{t-1}: wait for PV_{t-1}, then scale O_h by alpha
          const int u = t - 1;
          if (!(ok = warp_wait(wd, &bars.pv_done[u & 1], (u >> 1) & 1))) break;
          tc_fence_after_sync();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {   // 32 columns at a time: the scores stay live
            uint32_t r0[32];
            tmem_ld32(colO + c0, r0);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) r0[j] = __float_as_uint(__uint_as_float(r0[j]) * alpha);
            tmem_st32(colO + c0, r0);
          }
          tmem_st_wait();
        }
      }
      // P = 2^(s * scale * log2e - m) for this row's 64 keys -> bf16 pairs ->
      // TMEM columns [64h, 64h + 32) of the S buffer (already read above)
      // a row with no visible key yet (m_run = -inf) has only -inf scores in
      // this tile: subtracting 0 instead keeps them -inf, and 2^-inf = 0
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      const uint64_t negm = f2_pack(-m_use, -m_use);
      uint64_t lsum = f2_pack(0.f, 0.f);
      uint32_t pw[32];
#pragma unroll
      for (int k2 = 0; k2 < 32; ++k2) {
        const uint32_t* src = k2 < 16 ? &ra[2 * k2] : &rb[2 * (k2 - 16)];
        const uint64_t x = f2_fma(f2_pack(__uint_as_float(src[0]), __uint_as_float(src[1])), scale2, negm);
        float a, c;
        f2_unpack(x, a, c);
        const float ea = ex2(a);
        const float ec = ex2(c);
        lsum = f2_add(lsum, f2_pack(ea, ec));
        pw[k2] = pack_bf16x2(ea, ec);
      }
      {
        float a, c;
        f2_unpack(lsum, a, c);
        l_run += a + c;
      }
      tmem_st32(tmem + lane_base + kColS + st * kBN + half * 64, pw);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars.p_full[st]);
    }
    if (ok) {
      const int u = n_kv - 1;
      ok = warp_wait(wd, &bars.pv_done[u & 1], (u >> 1) & 1);
    }
    // ---- epilogue: merge the two halves of every row.  The exchange uses the
    // K ring, idle once the last PV product has completed.
    float (*merge_m)[kBM] = reinterpret_cast<float (*)[kBM]>(smem + C::kOffK);
    float (*merge_l)[kBM] = reinterpret_cast<float (*)[kBM]>(smem + C::kOffK + 2 * kBM * 4);
    merge_m[half][row] = m_run;
    merge_l[half][row] = l_run;
    named_barrier_sync(1, kSoftmaxWarps * 32);
    const int qrow = qt * kBM + row;                    // chunk-local row
    const bool store = qrow < p.q_len;                  // rows of a partial last tile past q_len are dropped
    if (ok && !wd.aborted()) {                          // warp-uniform: the TMEM loads are .sync.aligned
      tc_fence_after_sync();
      const float m0 = merge_m[0][row], m1 = merge_m[1][row];
      const float M = fmaxf(m0, m1);
      const float a0 = m0 == -INFINITY ? 0.f : ex2(m0 - M);
      const float a1 = m1 == -INFINITY ? 0.f : ex2(m1 - M);
      const float L = merge_l[0][row] * a0 + merge_l[1][row] * a1;
      const float inv = 1.f / L;
      const float f0 = a0 * inv, f1 = a1 * inv;
      // this warp writes head-dim columns [D/2 half, D/2 half + D/2) of the row
      uint4* orow = reinterpret_cast<uint4*>(p.o + ((static_cast<int64_t>(b) * p.q_len + qrow) * p.Hq + h) * D +
                                             half * (D / 2));
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem + lane_base + kColO + half * (D / 2) + c0, r0);
        tmem_ld32(tmem + lane_base + kColO + 128 + half * (D / 2) + c0, r1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          float v[8];
#pragma unroll
          for (int k2 = 0; k2 < 8; ++k2)
            v[k2] = __uint_as_float(r0[j + k2]) * f0 + __uint_as_float(r1[j + k2]) * f1;
          uint4 q;
          q.x = pack_bf16x2(v[0], v[1]);
          q.y = pack_bf16x2(v[2], v[3]);
          q.z = pack_bf16x2(v[4], v[5]);
          q.w = pack_bf16x2(v[6], v[7]);
          if (store) orow[(c0 + j) / 8] = q;
        }
      }
      if (half == 0 && store)
        p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.q_len + qrow] = (M + __log2f(L)) * kLn2;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (wd.aborted()) {
    // A wait ran out.  Every role has left its loop (the MMA issuers after
    // their last MMA completed), but a copy issued before the abort may still
    // be in flight: let it land before the CTA's shared memory goes away.
    if ((warp == 0 || warp == kVWarp) && lane == 0) {
      uint64_t* full = warp == 0 ? bars.k_full : bars.v_full;
      if (warp == 0) wd.drain(&bars.q_full, 0, 1000000);
      for (int st = 0; st < kStages && st < n_issued; ++st) {
        const int last = st + kStages * ((n_issued - 1 - st) / kStages);  // last tile issued into stage st
        wd.drain(&full[st], (last / kStages) & 1, 1000000);
      }
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_fwd_bf16_d(const FwdParams& p, const Bf16FwdMaps& maps, unsigned grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       FwdCfg<D>::kSmemAlloc);
  if (e != cudaSuccess) return e;
  fwd_bf16_kernel<D><<<grid, kThreads, FwdCfg<D>::kSmemAlloc, s>>>(maps.q, maps.k, maps.v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const ChunkGeom& g, const Bf16FwdMaps& maps, void* o, float* lse,
                            unsigned int* err, cudaStream_t s) {
  FwdParams p;
  p.B = g.B;
  p.Hq = g.Hq;
  p.Hkv = g.Hkv;
  p.G = g.G;
  p.q_len = static_cast<int>(g.q_len);
  p.T = static_cast<int>(g.T);
  p.q_start = static_cast<int>(g.q_start);
  p.kv_begin = static_cast<int>(g.kv_begin);
  p.n_qtiles = static_cast<int>((g.q_len + kBM - 1) / kBM);
  p.scale_log2 = g.scale * kLog2e;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.err = err;
  p.wait_cycles = g.wait_cycles;
  const unsigned grid = static_cast<unsigned>(p.n_qtiles) * g.Hq * g.B;
  return g.d == 64 ? launch_fwd_bf16_d<64>(p, maps, grid, s) : launch_fwd_bf16_d<128>(p, maps, grid, s);
}

}  // namespace seqattn
