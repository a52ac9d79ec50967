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
// tile ("steps"), keeps dK and dV for its 128 keys in TMEM for the whole loop,
// and finally stages them in shared memory and adds them into the float32
// accumulators with TMA reduce-adds (bulk fp32 additions carried out in L2,
// atomic per element).  Within one call no other CTA touches those rows, so
// the reductions meet no contention; they need no load of the old sums, and
// backward calls of different chunks may run concurrently on different
// streams.  dQ partial products of every key tile
// are summed into the zeroed dq with fp32 reductions.  Chunks may start
// and end anywhere: a partial last query tile reads padding statistics
// (-inf, 0) that make its extra rows' P exactly 0, and rows past the chunk
// are never stored.
//
// TMEM (512 columns): dK [0,128), dV [128,256) and two step buffers of 128
// columns.  Step n uses buffer n&1: S^T in its first 64 columns, dP^T in the
// last 64.  Compute warp half h reads S^T columns [32h, 32h+32) and writes P^T
// (bf16 pairs) over the first 16 of them and dS^T over the last 16, so the dP^T
// half is free as soon as it has been read and dQ^T can land there.  Two
// buffers let the S^T/dP^T MMAs of step n+1 run while the compute warps form P
// and dS of step n.
//   warp 0       TMA producer: K, V once; Q, dO (64 rows) + the step's row
//                statistics (-L log2 e, Delta) into a 3-stage ring
//   warp 1       TMEM owner + MMA issuer of S^T = K Q^T (M=128 keys, N=64, SS)
//   warp 15      MMA issuer of dP^T = V dO^T (M=128 keys, N=64, SS)
//   warp 14      MMA issuer of dV += P^T dO (as soon as P^T is written),
//                dK += dS^T Q (M=128, N=d, K=64; A from TMEM) and
//                dQ^T = K^T dS^T (M=128 rows of d, zero-padded when d = 64;
//                N=64, K=128; SS)
//   warps 2..9   P^T, then dS^T: two warps per TMEM lane quadrant, 32 query
//                columns each; dS^T also to shared memory for dQ^T; at the
//                end dK (warps 2-5) / dV (6-9) staged for the reduce-adds
//   warps 10..13 dQ^T from TMEM -> fp32 reductions into dq
// Three issuing threads because one thread keeps only about one tcgen05.mma
// in flight per ~90 cycles, whatever its shape; S^T and dP^T, which gate the
// compute warps, each get a thread of their own.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace seqattn {
namespace {

constexpr int kBK = 128;   // keys per CTA
constexpr int kBQ = 64;    // query rows per step
constexpr int kComputeWarps = 8;                      // two per TMEM lane quadrant
constexpr int kDQWarp0 = 2 + kComputeWarps;            // 4 dQ warps
constexpr int kIssuerKV = kDQWarp0 + 4;                // dV, dK, dQ^T issuer
constexpr int kIssuerDP = kIssuerKV + 1;               // dP^T issuer
constexpr int kThreads = 32 * (kIssuerDP + 1);          // 16 warps

constexpr int kDQRows = 128;                       // M of dQ^T = K^T dS^T (d rows, zero-padded when d = 64)
constexpr int kKVHalf = kBK * 128;                 // 16 KB: one 64-column block of 128 rows x 128 B
constexpr int kQHalf = kBQ * 128;                  // 8 KB: one 64-column block of 64 rows x 128 B
constexpr int kPTileBytes = kBK * kBQ * 2;         // 16 KB: 128 keys x 64 q
constexpr int kQStages = 3;                        // Q/dO/statistics ring depth
constexpr int kStatBytes = 2 * kBQ * 4;

// Head-dim dependent sizes and the shared memory carve-up (bytes from the
// 1024-aligned base).  The K tile always holds two 64-column blocks: with
// d = 64 the second is zero, so that dQ^T = K^T dS^T keeps M = 128.
template <int D>
struct BwdCfg {
  static constexpr int kKBytes = 2 * kKVHalf;                 // 32 KB
  static constexpr int kVBytes = kBK * D * 2;                 // 32 KB or 16 KB
  static constexpr int kQTileBytes = kBQ * D * 2;             // 16 KB or 8 KB
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKBytes;
  static constexpr int kOffQ = kOffV + kVBytes;               // kQStages stages
  static constexpr int kOffDO = kOffQ + kQStages * kQTileBytes;   // kQStages stages
  static constexpr int kOffDS = kOffDO + kQStages * kQTileBytes;  // 2 buffers
  static constexpr int kOffStat = kOffDS + 2 * kPTileBytes;   // kQStages x (-L log2 e [64], Delta [64])
  static constexpr int kSmemBytes = kOffStat + kQStages * kStatBytes;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  static_assert(2 * kBK * D * 4 <= kOffStat - kOffQ, "dK and dV are staged in the Q/dO ring and dS buffers");
};

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColDK = 0;
constexpr uint32_t kColDV = 128;
__host__ __device__ constexpr uint32_t col_buf(int b) { return 256u + 128u * static_cast<uint32_t>(b); }
constexpr uint32_t kOffS = 0;    // within a step buffer: S^T, then P^T / dS^T pairs
constexpr uint32_t kOffDP = 64;  // dP^T, then dQ^T (64 cols)

struct BwdParams {
  int B, Hq, Hkv, G;
  int q_len, T;
  int q_start, kv_begin;
  int n_ktiles;
  int n_q64;               // 64-row query tiles of the chunk (the last may be partial)
  int n_pre;               // key tiles wholly before the chunk's first row
  float scale;
  float scale_log2;
  const float* stats;      // [B, Hq, n_q64, 2, 64]: -L log2 e, then Delta, per query tile
  float* dq;
  float* dk;
  float* dv;
  unsigned int* err;
  long long wait_cycles;
  int reverse;             // prefix tiles (and batch entries) in descending order
};

struct BwdBarriers {
  uint64_t kv_full;
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t s_full[2];      // S^T of buffer b computed
  uint64_t dp_full[2];     // dP^T of buffer b computed
  uint64_t p_full[2];      // P^T of buffer b written (compute warps)
  uint64_t ds_full[2];     // dS^T of buffer b written to TMEM and smem (compute warps)
  uint64_t kv_done[2];     // dV, dK of buffer b done: the S^T half is free
  uint64_t ds_empty[2];    // dS^T shared-memory buffer b read by dQ^T
  uint64_t dq_full[2];     // dQ^T in buffer b computed
  uint64_t dq_empty[2];    // dQ^T of buffer b drained (dQ warps)
  uint64_t acc_done;
  uint64_t mma_final[3];
};

__device__ __forceinline__ bool warp_wait(Watchdog& wd, uint64_t* bar, uint32_t parity) {
  const bool ok = wd.wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// Shared-memory descriptors are built once per tile base; a K-step moves only
// the 14-bit start-address field (16-byte units), so each MMA's operands are
// the base plus a compile-time constant.
// K-major operand stored as 128-byte rows in blocks of `block_bytes` (64 bf16
// of K per block): K-step ks (16 elements) lies in block ks/4 at byte
// 32*(ks%4) of each row.
__host__ __device__ constexpr uint32_t kmajor_off(int block_bytes, int ks) {
  return static_cast<uint32_t>(((ks >> 2) * block_bytes + (ks & 3) * 32) >> 4);
}
// MN-major operand stored as [K rows][MN] with 128-byte rows: 8 K-rows per
// 1024-byte atom; K-step ks (16 rows) starts 2048 bytes further.
__host__ __device__ constexpr uint32_t mnmajor_off(int ks) { return static_cast<uint32_t>((ks * 2048) >> 4); }
// Column (relative to a step buffer) of the P^T bf16 pairs of query rows
// [16 ks, 16 ks + 16): compute warp half h packs its 32 rows at [32h, 32h+16);
// the dS^T pairs of the same rows sit 16 columns further.
__host__ __device__ constexpr uint32_t pair_col(int ks) {
  return static_cast<uint32_t>(32 * (ks >> 1) + 8 * (ks & 1));
}
constexpr uint32_t kDSPairs = 16;

// P = 2^x with x = s scale log2(e) - L log2(e) for one thread's 32 scores,
// as fp32 pairs (p2) and packed bf16 pairs (pk).
__device__ __forceinline__ void form_p(const uint32_t (&r)[32], const uint64_t (&nl2)[16], uint64_t scale2,
                                       uint64_t (&p2)[16], uint32_t (&pk)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint64_t x = f2_fma(f2_pack(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), scale2, nl2[j]);
    float x0, x1;
    f2_unpack(x, x0, x1);
    const float p0 = ex2(x0), p1 = ex2(x1);
    p2[j] = f2_pack(p0, p1);
    pk[j] = pack_bf16x2(p0, p1);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_bf16_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                    const __grid_constant__ CUtensorMap map_dk, const __grid_constant__ CUtensorMap map_dv,
                    const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int kDQWarps = D / 32;                   // dQ warps holding live d rows of dQ^T
  if (error_already_set(p.err)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ BwdBarriers bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  Watchdog wd(&abort_flag, p.err, p.wait_cycles);

  // ---- work item: (batch b, kv head g, key tile kt).
  // Per batch entry: first the key tiles that lie wholly before the chunk
  // (all of equal, longest length), key tile fastest within each key/value
  // head so that a wave shares one group's Q, dO and dq in L2 (in ascending
  // or, with p.reverse, descending order of batch entry, head and tile); then
  // the tiles that reach into the chunk (shorter, decreasing), head fastest,
  // so the shortest loops form the last wave.
  const int per_b = p.n_ktiles * p.Hkv;
  const int b0 = blockIdx.x / per_b;
  int idx = blockIdx.x - b0 * per_b;
  const int b = p.reverse ? p.B - 1 - b0 : b0;
  int g, kt;
  if (idx < p.n_pre * p.Hkv) {
    if (p.reverse) idx = p.n_pre * p.Hkv - 1 - idx;
    g = idx / p.n_pre;
    kt = idx - g * p.n_pre;
  } else {
    const int j = idx - p.n_pre * p.Hkv;
    kt = p.n_pre + j / p.Hkv;
    g = j - (j / p.Hkv) * p.Hkv;
  }
  const int kb = p.kv_begin + kt * kBK;                  // absolute first key of the tile
  // first query tile that sees any key of this tile (the one holding row kb)
  const int qi_first = kb > p.q_start ? (kb - p.q_start) / kBQ : 0;
  const int nq = p.n_q64 - qi_first;
  const int n_steps = p.G * nq;

  const int warp = warp_id();
  const int lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars.kv_full, 1);
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 3);   // S^T, dP^T and dV/dK issuers read the stage
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.dp_full[i], 1);
      mbar_init(&bars.p_full[i], kComputeWarps * 32);
      mbar_init(&bars.ds_full[i], kComputeWarps * 32);
      mbar_init(&bars.kv_done[i], 1);
      mbar_init(&bars.ds_empty[i], 1);
      mbar_init(&bars.dq_full[i], 1);
      mbar_init(&bars.dq_empty[i], kDQWarps * 32);
    }
    for (int i = 0; i < 3; ++i) mbar_init(&bars.mma_final[i], 1);
    mbar_init(&bars.acc_done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  if constexpr (D < 128) {
    // second K block: the zero d rows 64..127 of the padded K^T operand of dQ^T
    uint4* z = reinterpret_cast<uint4*>(smem + C::kOffK + kKVHalf);
    for (int i = threadIdx.x; i < kKVHalf / 16; i += kThreads) z[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sV = smem_u32(smem + C::kOffV);
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sDO = smem_u32(smem + C::kOffDO);
  const uint32_t sDS = smem_u32(smem + C::kOffDS);
  float* stat = reinterpret_cast<float*>(smem + C::kOffStat);  // [stage][-L log2 e 64 | Delta 64]

  auto step_head = [&](int n) { return g * p.G + n / nq; };
  auto step_qtile = [&](int n) { return qi_first + n % nq; };
  int n_issued = 0;  // producer: steps issued into the ring so far

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_do);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      const int krow = b * p.T + kb;
      mbar_arrive_expect_tx(&bars.kv_full, 2 * C::kVBytes);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk) {
        tma_load_3d(smem + C::kOffK + blk * kKVHalf, &map_k, &bars.kv_full, 64 * blk, g, krow);
        tma_load_3d(smem + C::kOffV + blk * kKVHalf, &map_v, &bars.kv_full, 64 * blk, g, krow);
      }
      for (int n = 0; n < n_steps; ++n) {
        const int st = n % kQStages;
        const uint32_t ph = (n / kQStages) & 1;
        const int h = step_head(n);
        const int qi = step_qtile(n);
        if (!wd.wait(&bars.q_empty[st], ph ^ 1)) break;
        const int qrow = b * p.q_len + qi * kBQ;
        const int64_t sblk = ((static_cast<int64_t>(b) * p.Hq + h) * p.n_q64 + qi) * (2 * kBQ);
        mbar_arrive_expect_tx(&bars.q_full[st], 2 * C::kQTileBytes + kStatBytes);
#pragma unroll
        for (int blk = 0; blk < D / 64; ++blk) {
          tma_load_3d(smem + C::kOffQ + st * C::kQTileBytes + blk * kQHalf, &map_q, &bars.q_full[st], 64 * blk, h,
                      qrow);
          tma_load_3d(smem + C::kOffDO + st * C::kQTileBytes + blk * kQHalf, &map_do, &bars.q_full[st], 64 * blk,
                      h, qrow);
        }
        bulk_load(stat + st * 2 * kBQ, p.stats + sblk, kStatBytes, &bars.q_full[st]);
        n_issued = n + 1;
      }
    }
  } else if (warp == 1 || warp == kIssuerKV || warp == kIssuerDP) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      const uint32_t idesc_sdp = make_idesc_bf16(kBK, kBQ, false, false);  // M128 N64, K-major both
      const uint32_t idesc_kv = make_idesc_bf16(kBK, D, false, true);      // M128 N=d, B MN-major
      const uint32_t idesc_dq = make_idesc_bf16(kDQRows, kBQ, true, true); // M128 N64, both MN-major
      // role 0: S^T (warp 1), role 1: dV, dK, dQ^T (kIssuerKV), role 2: dP^T
      const int role = warp == 1 ? 0 : (warp == kIssuerKV ? 1 : 2);
      bool ok = wd.wait(&bars.kv_full, 0);
      if (role != 1) {
        // ---- S^T(n) (role 0) or dP^T(n) (role 2) into buffer n&1 as soon as
        // the Q/dO stage has landed and step n-2 has released that half
        const bool is_s = role == 0;
        const uint64_t a_kmaj = make_desc_sw128(is_s ? sK : sV, 16, 1024);
        const uint64_t b_kmaj0 = make_desc_sw128(is_s ? sQ : sDO, 16, 1024);
        uint64_t* full = is_s ? bars.s_full : bars.dp_full;
        uint64_t* release = is_s ? bars.kv_done : bars.dq_empty;
        const uint32_t off = is_s ? kOffS : kOffDP;
        for (int n = 0; ok && n < n_steps; ++n) {
          const int st = n % kQStages;
          const int bb = n & 1;
          if (!(ok = wd.wait(&bars.q_full[st], (n / kQStages) & 1))) break;
          if (n >= 2 && !(ok = wd.wait(&release[bb], ((n - 2) >> 1) & 1))) break;
          tc_fence_after_sync();
          const uint64_t bd = b_kmaj0 + static_cast<uint64_t>(st * (C::kQTileBytes >> 4));
          const uint32_t d = tmem + col_buf(bb) + off;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            umma_bf16_ss(d, a_kmaj + kmajor_off(kKVHalf, ks), bd + kmajor_off(kQHalf, ks), idesc_sdp,
                         ks > 0 ? 1u : 0u);
          umma_commit(&full[bb]);
          umma_commit(&bars.q_empty[st]);
        }
      } else {
        // ---- dV += P^T dO once P^T(n) is written; dK += dS^T Q and
        // dQ^T(n) = K^T dS^T (over the already read dP^T half) once dS^T(n) is
        const uint64_t q_mn0 = make_desc_sw128(sQ, kQHalf, 1024);
        const uint64_t do_mn0 = make_desc_sw128(sDO, kQHalf, 1024);
        const uint64_t k_mn = make_desc_sw128(sK, kKVHalf, 1024);
        const uint64_t ds_mn0 = make_desc_sw128(sDS, kPTileBytes, 1024);
        for (int n = 0; ok && n < n_steps; ++n) {
          const int st = n % kQStages;
          const int bb = n & 1;
          const uint32_t cb = tmem + col_buf(bb);
          if (!(ok = wd.wait(&bars.p_full[bb], (n >> 1) & 1))) break;
          tc_fence_after_sync();
          const uint64_t dm = do_mn0 + static_cast<uint64_t>(st * (C::kQTileBytes >> 4));
#pragma unroll
          for (int ks = 0; ks < kBQ / 16; ++ks)
            umma_bf16_ts(tmem + kColDV, cb + kOffS + pair_col(ks), dm + mnmajor_off(ks), idesc_kv,
                         (n > 0 || ks > 0) ? 1u : 0u);
          if (!(ok = wd.wait(&bars.ds_full[bb], (n >> 1) & 1))) break;
          tc_fence_after_sync();
          const uint64_t qm = q_mn0 + static_cast<uint64_t>(st * (C::kQTileBytes >> 4));
#pragma unroll
          for (int ks = 0; ks < kBQ / 16; ++ks)
            umma_bf16_ts(tmem + kColDK, cb + kOffS + pair_col(ks) + kDSPairs, qm + mnmajor_off(ks), idesc_kv,
                         (n > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&bars.kv_done[bb]);
          umma_commit(&bars.q_empty[st]);
          const uint64_t sm = ds_mn0 + static_cast<uint64_t>(bb * (kPTileBytes >> 4));
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks)
            umma_bf16_ss(cb + kOffDP, k_mn + mnmajor_off(ks), sm + mnmajor_off(ks), idesc_dq, ks > 0 ? 1u : 0u);
          umma_commit(&bars.dq_full[bb]);
          umma_commit(&bars.ds_empty[bb]);
        }
        umma_commit(&bars.acc_done);
      }
      umma_commit(&bars.mma_final[role]);
      wd.drain(&bars.mma_final[role], 0, 4000000);
    }
  } else if (warp < 2 + kComputeWarps) {
    // ------------------------------------------------------------ P / dS
    // Two warps per TMEM lane quadrant: warp half h owns query columns
    // [32h, 32h + 32) of every step, so each thread forms 32 P and 32 dS.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int kr = quad * 32 + lane;                    // key row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int key = kb + kr;
    const int c_off = half * 32;                        // first query column of this warp
    const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
    bool ok = true;
    int st = 0, ph = 0;                                 // ring stage of step n and its phase parity
    int qi = qi_first;                                  // query tile of step n (heads cycle slowest)
    for (int n = 0; n < n_steps; ++n) {
      const int bb = n & 1;
      if (!(ok = warp_wait(wd, &bars.q_full[st], ph))) break;
      if (!(ok = warp_wait(wd, &bars.s_full[bb], (n >> 1) & 1))) break;
      tc_fence_after_sync();
      const uint32_t cb = tmem + lane_base + col_buf(bb);
      uint32_t r[32];
      tmem_ld32(cb + kOffS + c_off, r);
      // -L log2(e) of the step's rows, read while the TMEM load is in flight
      const float4* L4 = reinterpret_cast<const float4*>(stat + st * 2 * kBQ + c_off);
      const float4* D4 = reinterpret_cast<const float4*>(stat + st * 2 * kBQ + kBQ + c_off);
      uint64_t nl2[16];                                 // pairs of query rows
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 l = L4[j];
        nl2[2 * j] = f2_pack(l.x, l.y);
        nl2[2 * j + 1] = f2_pack(l.z, l.w);
      }
      const int q_abs0 = p.q_start + qi * kBQ + c_off;  // absolute row of this warp's column 0
      const bool masked = kb + kBK - 1 > q_abs0;        // some key of the tile follows some row
      tmem_ld_wait();
      // P = 2^(s scale log2(e) - L log2(e)), exactly 0 on padding rows (-inf);
      // kept in fp32 for dS
      uint64_t p2[16];
      uint32_t pk[16];                                  // packed bf16 pairs
      form_p(r, nl2, scale2, p2, pk);
      if (masked) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float p0, p1;
          f2_unpack(p2[j], p0, p1);
          if (key > q_abs0 + 2 * j) p0 = 0.f;
          if (key > q_abs0 + 2 * j + 1) p1 = 0.f;
          p2[j] = f2_pack(p0, p1);
          pk[j] = pack_bf16x2(p0, p1);
        }
      }
      // P^T pairs over the first 16 of this warp's S^T columns: dV can start
      tmem_st16(cb + kOffS + c_off, pk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars.p_full[bb]);
      // dS = P o (dP - Delta)
      if (!(ok = warp_wait(wd, &bars.dp_full[bb], (n >> 1) & 1))) break;
      tc_fence_after_sync();
      tmem_ld32(cb + kOffDP + c_off, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 dd = D4[j];
        const uint64_t a0 = f2_mul(p2[2 * j], f2_sub(f2_pack(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1])),
                                                     f2_pack(dd.x, dd.y)));
        const uint64_t a1 = f2_mul(p2[2 * j + 1],
                                   f2_sub(f2_pack(__uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])),
                                          f2_pack(dd.z, dd.w)));
        float u0, u1, u2, u3;
        f2_unpack(a0, u0, u1);
        f2_unpack(a1, u2, u3);
        pk[2 * j] = pack_bf16x2(u0, u1);
        pk[2 * j + 1] = pack_bf16x2(u2, u3);
      }
      // dS^T pairs over the last 16 of this warp's S^T columns
      tmem_st16(cb + kOffS + c_off + kDSPairs, pk);
      // dS^T row segment to shared memory (B operand of dQ^T) once dQ^T of
      // step n-2 has read that buffer: 128-byte rows, 128-byte swizzle inside
      // 8-row groups; this warp writes 16-byte chunks 4*half .. 4*half+3
      if (n >= 2 && !(ok = warp_wait(wd, &bars.ds_empty[bb], ((n - 2) >> 1) & 1))) break;
      const uint32_t sw = static_cast<uint32_t>(kr & 7);
      const uint32_t dsrow = sDS + bb * kPTileBytes + kr * 128;
#pragma unroll
      for (int ci = 0; ci < 4; ++ci)
        st_shared_v4(dsrow + (((4 * half + ci) ^ sw) << 4), pk[ci * 4], pk[ci * 4 + 1], pk[ci * 4 + 2],
                     pk[ci * 4 + 3]);
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&bars.ds_full[bb]);
      if (++st == kQStages) {
        st = 0;
        ph ^= 1;
      }
      if (++qi == qi_first + nq) qi = qi_first;
    }
    // ---- epilogue: this tile's dK (half 0) and dV (half 1) go to shared
    // memory (the idle Q/dO ring) as 128-row boxes of 32 columns with the
    // 128-byte swizzle, then one thread adds them into the running sums with
    // TMA reduce-adds; rows past the chunk's end are cut by the tensor maps
    if (ok) ok = warp_wait(wd, &bars.acc_done, 0);
    if (ok) {                                           // warp-uniform: the TMEM loads are .sync.aligned
      tc_fence_after_sync();
      const uint32_t col = half == 0 ? kColDK : kColDV;
      const float f = half == 0 ? p.scale : 1.f;
      uint8_t* stage = smem + C::kOffQ + half * (D / 32) * 16384;
      const uint32_t sw = static_cast<uint32_t>(kr & 7);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + col + c0, r);
        tmem_ld_wait();
        const uint32_t rowa = smem_u32(stage + (c0 / 32) * 16384 + kr * 128);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          st_shared_v4(rowa + ((c4 ^ sw) << 4), __float_as_uint(f * __uint_as_float(r[4 * c4])),
                       __float_as_uint(f * __uint_as_float(r[4 * c4 + 1])),
                       __float_as_uint(f * __uint_as_float(r[4 * c4 + 2])),
                       __float_as_uint(f * __uint_as_float(r[4 * c4 + 3])));
      }
      fence_proxy_async_smem();
    }
    named_barrier_sync(2, kComputeWarps * 32);
    if (ok && !wd.aborted() && warp == 2 && lane == 0) {
#pragma unroll 1
      for (int bx = 0; bx < D / 32; ++bx) {
        tma_reduce_add_4d(&map_dk, smem + C::kOffQ + bx * 16384, 32 * bx, g, kb, b);
        tma_reduce_add_4d(&map_dv, smem + C::kOffQ + (D / 32 + bx) * 16384, 32 * bx, g, kb, b);
      }
      bulk_commit_group();
      bulk_wait_group_read<0>();
    }
  } else {
    // ------------------------------------------------------------ dQ
    const int quad = warp & 3;
    const int dcol = quad * 32 + lane;                  // head-dim column (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    // with d = 64 the lanes 64..127 of dQ^T are the zero padding: no work
    for (int n = 0; quad < kDQWarps && n < n_steps; ++n) {
      const int bb = n & 1;
      if (!warp_wait(wd, &bars.dq_full[bb], (n >> 1) & 1)) break;
      tc_fence_after_sync();
      uint32_t r0[32], r1[32];
      tmem_ld32(tmem + lane_base + col_buf(bb) + kOffDP, r0);
      tmem_ld32(tmem + lane_base + col_buf(bb) + kOffDP + 32, r1);
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars.dq_empty[bb]);
      const int h = step_head(n);
      const int qi = step_qtile(n);
      float* base = p.dq + ((static_cast<int64_t>(b) * p.q_len + qi * kBQ) * p.Hq + h) * D + dcol;
      const int64_t rstride = static_cast<int64_t>(p.Hq) * D;
      const int rows = p.q_len - qi * kBQ;              // rows of this query tile inside the chunk
      if (rows >= kBQ) {
        // full tile: 64 back-to-back reductions (a per-row predicate here
        // halved the kernel's speed)
#pragma unroll
        for (int c = 0; c < 32; ++c) atomicAdd(base + c * rstride, p.scale * __uint_as_float(r0[c]));
#pragma unroll
        for (int c = 0; c < 32; ++c) atomicAdd(base + (c + 32) * rstride, p.scale * __uint_as_float(r1[c]));
      } else {
        // partial last tile of a ragged chunk: rows past q_len are dropped
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (c < rows) atomicAdd(base + c * rstride, p.scale * __uint_as_float(r0[c]));
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (c + 32 < rows) atomicAdd(base + (c + 32) * rstride, p.scale * __uint_as_float(r1[c]));
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (wd.aborted()) {
    // A wait ran out.  Every role has left its loop (the MMA issuers after
    // their last MMA completed), but a copy issued before the abort may still
    // be in flight: let it land before the CTA's shared memory goes away.
    if (warp == 0 && lane == 0) {
      wd.drain(&bars.kv_full, 0, 1000000);
      for (int st = 0; st < kQStages && st < n_issued; ++st) {
        const int last = st + kQStages * ((n_issued - 1 - st) / kQStages);  // last step issued into stage st
        wd.drain(&bars.q_full[st], (last / kQStages) & 1, 1000000);
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
cudaError_t launch_bwd_bf16_d(const BwdParams& p, const Bf16BwdMaps& maps, unsigned grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(bwd_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       BwdCfg<D>::kSmemAlloc);
  if (e != cudaSuccess) return e;
  bwd_bf16_kernel<D><<<grid, kThreads, BwdCfg<D>::kSmemAlloc, s>>>(maps.q, maps.k, maps.v, maps.d_o, maps.dk,
                                                                     maps.dv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_bf16(const ChunkGeom& g, const Bf16BwdMaps& maps, const float* stats,
                            float* dq, float* dk, float* dv, unsigned int* err, cudaStream_t s) {
  BwdParams p;
  p.B = g.B;
  p.Hq = g.Hq;
  p.Hkv = g.Hkv;
  p.G = g.G;
  p.q_len = static_cast<int>(g.q_len);
  p.T = static_cast<int>(g.T);
  p.q_start = static_cast<int>(g.q_start);
  p.kv_begin = static_cast<int>(g.kv_begin);
  p.n_ktiles = static_cast<int>((g.q_start + g.q_len - g.kv_begin + kBK - 1) / kBK);
  p.n_q64 = static_cast<int>((g.q_len + kBQ - 1) / kBQ);
  p.n_pre = static_cast<int>((g.q_start - g.kv_begin) / kBK);   // tiles with kb + 127 < q_start
  p.scale = g.scale;
  p.scale_log2 = g.scale * 1.4426950408889634f;
  p.stats = stats;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.err = err;
  p.wait_cycles = g.wait_cycles;
  // Alternate the sweep direction over the prefix from one chunk to the next
  // (by the chunk's index in a uniform partition): the prefix rows a call
  // touched last are then the first the next call touches, while they are
  // still in L2.  Each dK/dV row still receives exactly one addition per call.
  p.reverse = static_cast<int>((g.q_start / (g.q_len > 0 ? g.q_len : 1)) & 1);
  const unsigned grid = static_cast<unsigned>(p.n_ktiles) * g.Hkv * g.B;
  return g.d == 64 ? launch_bwd_bf16_d<64>(p, maps, grid, s) : launch_bwd_bf16_d<128>(p, maps, grid, s);
}

}  // namespace seqattn
