// simt_f32.cu -- the float32 path of the chunk calls (plain FMA arithmetic,
// no tensor cores, so results stay within float32 rounding of the exact
// value), the Delta preprocess of that path, the row-statistics pre-pass of
// the bf16 tensor-core backward, the accumulator zero fill and SpaCO's
// accumulator row scaling.
//
// Operation: the partitioned causal attention of the StreamBP review page
// (Property 3.1 and Eqs. (12)-(14) named in its "Circularity Check"):
// row r of the chunk (absolute position q_start + r) attends keys
// [kv_begin, q_start + r]; backward forms dQ for the chunk and adds the
// chunk's dK/dV contributions into the running sums over the prefix.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace seqattn {
namespace {

constexpr int kRowsPerBlock = 64;  // one query (or key) row per thread
constexpr int kTile = 32;          // rows staged per step for the other operand

__device__ __forceinline__ bool done_early(const unsigned int* err) {
  return error_already_set(err);
}

// ---------------------------------------------------------------------------
// forward: O, LSE for one chunk.  grid (ceil(q_len/64), Hq, B), block 64.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kRowsPerBlock) fwd_f32_kernel(ChunkGeom g, const float* __restrict__ q,
                                                                const float* __restrict__ k,
                                                                const float* __restrict__ v,
                                                                float* __restrict__ o,
                                                                float* __restrict__ lse,
                                                                const unsigned int* err) {
  if (done_early(err)) return;
  extern __shared__ float sm[];
  float* Qs = sm;                              // [64][D+1]
  float* Ks = Qs + kRowsPerBlock * (D + 1);    // [32][D]
  float* Vs = Ks + kTile * D;                  // [32][D]
  const int b = blockIdx.z, h = blockIdx.y, gk = h / g.G;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock;
  const int t = threadIdx.x;
  const int64_t r = r0 + t;
  const bool valid = r < g.q_len;
  const int64_t pos = g.q_start + r;

  for (int i = t; i < kRowsPerBlock * D; i += kRowsPerBlock) {
    const int rr = i / D, e = i % D;
    const int64_t row = r0 + rr;
    Qs[rr * (D + 1) + e] = row < g.q_len ? q[((b * g.q_len + row) * g.Hq + h) * D + e] : 0.f;
  }
  float acc[D];
#pragma unroll
  for (int e = 0; e < D; ++e) acc[e] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int64_t last_pos = g.q_start + min(g.q_len, r0 + kRowsPerBlock) - 1;
  for (int64_t j0 = g.kv_begin; j0 <= last_pos; j0 += kTile) {
    __syncthreads();
    for (int i = t; i < kTile * D; i += kRowsPerBlock) {
      const int jj = i / D, e = i % D;
      const int64_t j = j0 + jj;
      const bool in = j <= last_pos;
      Ks[i] = in ? k[((b * g.T + j) * g.Hkv + gk) * D + e] : 0.f;
      Vs[i] = in ? v[((b * g.T + j) * g.Hkv + gk) * D + e] : 0.f;
    }
    __syncthreads();
    float s[kTile];
    float mt = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < kTile; ++jj) {
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < D; ++e) dot = fmaf(Qs[t * (D + 1) + e], Ks[jj * D + e], dot);
      const bool vis = (j0 + jj) <= pos;
      s[jj] = vis ? dot * g.scale : -INFINITY;
      mt = fmaxf(mt, s[jj]);
    }
    if (!valid || mt == -INFINITY) continue;
    const float m_new = fmaxf(m, mt);
    const float a = expf(m - m_new);
    l *= a;
#pragma unroll
    for (int e = 0; e < D; ++e) acc[e] *= a;
    m = m_new;
#pragma unroll
    for (int jj = 0; jj < kTile; ++jj) {
      const float p = expf(s[jj] - m);
      l += p;
#pragma unroll
      for (int e = 0; e < D; ++e) acc[e] = fmaf(p, Vs[jj * D + e], acc[e]);
    }
  }
  if (!valid) return;
  const float inv = 1.f / l;
  float* orow = o + ((b * g.q_len + r) * g.Hq + h) * D;
#pragma unroll
  for (int e = 0; e < D; ++e) orow[e] = acc[e] * inv;
  lse[(static_cast<int64_t>(b) * g.Hq + h) * g.q_len + r] = m + logf(l);
}

// ---------------------------------------------------------------------------
// backward, dQ: one query row per thread.  grid (ceil(q_len/64), Hq, B).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kRowsPerBlock) bwd_dq_f32_kernel(
    ChunkGeom g, const float* __restrict__ q, const float* __restrict__ k,
    const float* __restrict__ v, const float* __restrict__ lse, const float* __restrict__ d_o,
    const float* __restrict__ delta, float* __restrict__ dq, const unsigned int* err) {
  if (done_early(err)) return;
  extern __shared__ float sm[];
  float* Qs = sm;                              // [64][D+1]
  float* dOs = Qs + kRowsPerBlock * (D + 1);   // [64][D+1]
  float* Ks = dOs + kRowsPerBlock * (D + 1);   // [32][D]
  float* Vs = Ks + kTile * D;                  // [32][D]
  const int b = blockIdx.z, h = blockIdx.y, gk = h / g.G;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock;
  const int t = threadIdx.x;
  const int64_t r = r0 + t;
  const bool valid = r < g.q_len;
  const int64_t pos = g.q_start + r;
  for (int i = t; i < kRowsPerBlock * D; i += kRowsPerBlock) {
    const int rr = i / D, e = i % D;
    const int64_t row = r0 + rr;
    const bool in = row < g.q_len;
    Qs[rr * (D + 1) + e] = in ? q[((b * g.q_len + row) * g.Hq + h) * D + e] : 0.f;
    dOs[rr * (D + 1) + e] = in ? d_o[((b * g.q_len + row) * g.Hq + h) * D + e] : 0.f;
  }
  const int64_t st = (static_cast<int64_t>(b) * g.Hq + h) * g.q_len + r;
  const float lse_r = valid ? lse[st] : 0.f;
  const float delta_r = valid ? delta[st] : 0.f;
  float acc[D];
#pragma unroll
  for (int e = 0; e < D; ++e) acc[e] = 0.f;
  const int64_t last_pos = g.q_start + min(g.q_len, r0 + kRowsPerBlock) - 1;
  for (int64_t j0 = g.kv_begin; j0 <= last_pos; j0 += kTile) {
    __syncthreads();
    for (int i = t; i < kTile * D; i += kRowsPerBlock) {
      const int jj = i / D, e = i % D;
      const int64_t j = j0 + jj;
      const bool in = j <= last_pos;
      Ks[i] = in ? k[((b * g.T + j) * g.Hkv + gk) * D + e] : 0.f;
      Vs[i] = in ? v[((b * g.T + j) * g.Hkv + gk) * D + e] : 0.f;
    }
    __syncthreads();
    if (!valid) continue;
    for (int jj = 0; jj < kTile; ++jj) {
      if (j0 + jj > pos) break;
      float dot = 0.f, dp = 0.f;
#pragma unroll
      for (int e = 0; e < D; ++e) {
        dot = fmaf(Qs[t * (D + 1) + e], Ks[jj * D + e], dot);
        dp = fmaf(dOs[t * (D + 1) + e], Vs[jj * D + e], dp);
      }
      const float p = expf(dot * g.scale - lse_r);
      const float ds = p * (dp - delta_r);
#pragma unroll
      for (int e = 0; e < D; ++e) acc[e] = fmaf(ds, Ks[jj * D + e], acc[e]);
    }
  }
  if (!valid) return;
  float* out = dq + ((b * g.q_len + r) * g.Hq + h) * D;
#pragma unroll
  for (int e = 0; e < D; ++e) out[e] = acc[e] * g.scale;
}

// ---------------------------------------------------------------------------
// backward, dK (kDK) or dV: one key row per thread, looping over the G query
// heads of the key's group and every chunk row that sees the key.  Each key
// row is owned by exactly one thread, so the running-sum update is a plain
// read-modify-write.  grid (ceil(n_keys/64), Hkv, B).
// ---------------------------------------------------------------------------
template <int D, bool kDK>
__global__ void __launch_bounds__(kRowsPerBlock) bwd_kv_f32_kernel(
    ChunkGeom g, const float* __restrict__ q, const float* __restrict__ k,
    const float* __restrict__ v, const float* __restrict__ lse, const float* __restrict__ d_o,
    const float* __restrict__ delta, float* __restrict__ accum, const unsigned int* err) {
  if (done_early(err)) return;
  extern __shared__ float sm[];
  float* Ks = sm;                              // [64][D+1]
  float* Vs = Ks + kRowsPerBlock * (D + 1);    // [64][D+1]
  float* Qs = Vs + kRowsPerBlock * (D + 1);    // [32][D]
  float* dOs = Qs + kTile * D;                 // [32][D]
  float* Ls = dOs + kTile * D;                 // [32]
  float* Ds = Ls + kTile;                      // [32]
  const int b = blockIdx.z, gk = blockIdx.y;
  const int t = threadIdx.x;
  const int64_t kv_end = g.q_start + g.q_len;
  const int64_t jb = g.kv_begin + static_cast<int64_t>(blockIdx.x) * kRowsPerBlock;
  const int64_t j = jb + t;
  const bool valid = j < kv_end;
  for (int i = t; i < kRowsPerBlock * D; i += kRowsPerBlock) {
    const int jj = i / D, e = i % D;
    const int64_t row = jb + jj;
    const bool in = row < kv_end;
    Ks[jj * (D + 1) + e] = in ? k[((b * g.T + row) * g.Hkv + gk) * D + e] : 0.f;
    Vs[jj * (D + 1) + e] = in ? v[((b * g.T + row) * g.Hkv + gk) * D + e] : 0.f;
  }
  float acc[D];
#pragma unroll
  for (int e = 0; e < D; ++e) acc[e] = 0.f;
  // chunk rows that can see any key of this block: absolute position >= jb
  const int64_t r_first = jb > g.q_start ? jb - g.q_start : 0;
  for (int hh = 0; hh < g.G; ++hh) {
    const int h = gk * g.G + hh;
    for (int64_t rt = r_first; rt < g.q_len; rt += kTile) {
      __syncthreads();
      for (int i = t; i < kTile * D; i += kRowsPerBlock) {
        const int rr = i / D, e = i % D;
        const int64_t row = rt + rr;
        const bool in = row < g.q_len;
        Qs[i] = in ? q[((b * g.q_len + row) * g.Hq + h) * D + e] : 0.f;
        dOs[i] = in ? d_o[((b * g.q_len + row) * g.Hq + h) * D + e] : 0.f;
      }
      for (int i = t; i < kTile; i += kRowsPerBlock) {
        const int64_t row = rt + i;
        const bool in = row < g.q_len;
        const int64_t st = (static_cast<int64_t>(b) * g.Hq + h) * g.q_len + row;
        Ls[i] = in ? lse[st] : 0.f;
        Ds[i] = in ? delta[st] : 0.f;
      }
      __syncthreads();
      if (!valid) continue;
      for (int rr = 0; rr < kTile; ++rr) {
        const int64_t row = rt + rr;
        if (row >= g.q_len) break;
        if (g.q_start + row < j) continue;  // causal: key after the query
        float dot = 0.f, dp = 0.f;
#pragma unroll
        for (int e = 0; e < D; ++e) {
          dot = fmaf(Qs[rr * D + e], Ks[t * (D + 1) + e], dot);
          if (kDK) dp = fmaf(dOs[rr * D + e], Vs[t * (D + 1) + e], dp);
        }
        const float p = expf(dot * g.scale - Ls[rr]);
        if (kDK) {
          const float ds = p * (dp - Ds[rr]);
#pragma unroll
          for (int e = 0; e < D; ++e) acc[e] = fmaf(ds, Qs[rr * D + e], acc[e]);
        } else {
#pragma unroll
          for (int e = 0; e < D; ++e) acc[e] = fmaf(p, dOs[rr * D + e], acc[e]);
        }
      }
    }
  }
  if (!valid) return;
  float* out = accum + ((b * g.T + j) * g.Hkv + gk) * D;
  const float f = kDK ? g.scale : 1.f;
#pragma unroll
  for (int e = 0; e < D; ++e) out[e] += acc[e] * f;
}

// ---------------------------------------------------------------------------
// Delta[b, h, r] = sum_e dO[b, r, h, e] * O[b, r, h, e] (float32), one warp per
// (row, head); optionally zero the matching dq row.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p) { return *p; }

template <typename T>
__global__ void __launch_bounds__(256) bwd_prep_kernel(ChunkGeom g, const T* __restrict__ o,
                                                       const T* __restrict__ d_o,
                                                       float* __restrict__ delta,
                                                       float* __restrict__ dq_to_zero) {
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t n_rows = static_cast<int64_t>(g.B) * g.q_len * g.Hq;  // (b, r, h) rows
  if (warp >= n_rows) return;
  const int h = static_cast<int>(warp % g.Hq);
  const int64_t br = warp / g.Hq;  // b * q_len + r
  const int b = static_cast<int>(br / g.q_len);
  const int64_t r = br % g.q_len;
  const T* orow = o + warp * g.d;
  const T* drow = d_o + warp * g.d;
  float s = 0.f;
  for (int e = lane; e < g.d; e += 32) s = fmaf(ld_f(orow + e), ld_f(drow + e), s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) delta[(static_cast<int64_t>(b) * g.Hq + h) * g.q_len + r] = s;
  if (dq_to_zero != nullptr) {
    float* z = dq_to_zero + warp * g.d;
    for (int e = lane; e < g.d; e += 32) z[e] = 0.f;
  }
}

// bf16 tensor-core backward statistics, one warp per (padded row, head):
// stats[((b Hq + h) n64 + r / 64) * 128 + r % 64]      = -L[b, h, r] log2(e)
// stats[((b Hq + h) n64 + r / 64) * 128 + 64 + r % 64] = Delta[b, h, r]
// for r < q_len, and -inf / 0 for the padding rows q_len <= r < 64 n64, so a
// padding row's P = 2^(s scale log2(e) - inf) is exactly 0.  Each 64-row query
// tile's statistics are one contiguous 512-byte block.  Zeroes dq rows too.
__global__ void __launch_bounds__(256) bwd_stats_bf16_kernel(ChunkGeom g, int n64,
                                                             const __nv_bfloat16* __restrict__ o,
                                                             const __nv_bfloat16* __restrict__ d_o,
                                                             const float* __restrict__ lse,
                                                             float* __restrict__ stats,
                                                             float* __restrict__ dq) {
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t q_pad = static_cast<int64_t>(n64) * 64;
  const int64_t n_rows = static_cast<int64_t>(g.B) * q_pad * g.Hq;  // (b, r, h) rows
  if (warp >= n_rows) return;
  const int h = static_cast<int>(warp % g.Hq);
  const int64_t br = warp / g.Hq;
  const int b = static_cast<int>(br / q_pad);
  const int64_t r = br % q_pad;
  float* dst = stats + ((static_cast<int64_t>(b) * g.Hq + h) * n64 + r / 64) * 128 + (r % 64);
  if (r >= g.q_len) {
    if (lane == 0) {
      dst[0] = -INFINITY;
      dst[64] = 0.f;
    }
    return;
  }
  const int64_t row = (static_cast<int64_t>(b) * g.q_len + r) * g.Hq + h;
  const __nv_bfloat16* orow = o + row * g.d;
  const __nv_bfloat16* drow = d_o + row * g.d;
  float s = 0.f;
  for (int e = lane; e < g.d; e += 32) s = fmaf(__bfloat162float(orow[e]), __bfloat162float(drow[e]), s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) {
    dst[0] = -lse[(static_cast<int64_t>(b) * g.Hq + h) * g.q_len + r] * 1.4426950408889634f;
    dst[64] = s;
  }
  float* z = dq + row * g.d;
  for (int e = lane; e < g.d; e += 32) z[e] = 0.f;
}

__global__ void zero2_kernel(float4* __restrict__ a, float4* __restrict__ b, int64_t n4) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    a[i] = z;
    b[i] = z;
  }
}

// rows [r0, r0 + n_rows) of two [B, T, row4] float4 arrays times `scale`
// (0 stores zeros, so NaN or Inf there is cleared too); grid-stride.
__global__ void scale2_rows_kernel(float4* __restrict__ a, float4* __restrict__ b, int64_t T, int64_t r0,
                                   int64_t n_rows, int64_t row4, int64_t n4, float scale) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t per_batch = n_rows * row4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const int64_t bi = i / per_batch;
    const int64_t j = (bi * T + r0) * row4 + (i - bi * per_batch);
    if (scale == 0.f) {
      a[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      b[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      float4 x = a[j], y = b[j];
      x.x *= scale; x.y *= scale; x.z *= scale; x.w *= scale;
      y.x *= scale; y.y *= scale; y.z *= scale; y.w *= scale;
      a[j] = x;
      b[j] = y;
    }
  }
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int D>
cudaError_t fwd_f32_d(const ChunkGeom& g, const float* q, const float* k, const float* v, float* o,
                      float* lse, unsigned int* err, cudaStream_t s) {
  const size_t smem = sizeof(float) * (kRowsPerBlock * (D + 1) + 2 * kTile * D);
  cudaError_t e = cudaFuncSetAttribute(fwd_f32_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((g.q_len + kRowsPerBlock - 1) / kRowsPerBlock), g.Hq, g.B);
  fwd_f32_kernel<D><<<grid, kRowsPerBlock, smem, s>>>(g, q, k, v, o, lse, err);
  return cudaGetLastError();
}

template <int D>
cudaError_t bwd_f32_d(const ChunkGeom& g, const float* q, const float* k, const float* v,
                      const float* lse, const float* d_o, const float* delta, float* dq, float* dk,
                      float* dv, unsigned int* err, cudaStream_t s) {
  const size_t smem_q = sizeof(float) * (2 * kRowsPerBlock * (D + 1) + 2 * kTile * D);
  cudaError_t e = cudaFuncSetAttribute(bwd_dq_f32_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_q);
  if (e != cudaSuccess) return e;
  dim3 grid_q(static_cast<unsigned>((g.q_len + kRowsPerBlock - 1) / kRowsPerBlock), g.Hq, g.B);
  bwd_dq_f32_kernel<D><<<grid_q, kRowsPerBlock, smem_q, s>>>(g, q, k, v, lse, d_o, delta, dq, err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const size_t smem_kv = sizeof(float) * (2 * kRowsPerBlock * (D + 1) + 2 * kTile * D + 2 * kTile);
  const int64_t n_keys = g.q_start + g.q_len - g.kv_begin;
  dim3 grid_kv(static_cast<unsigned>((n_keys + kRowsPerBlock - 1) / kRowsPerBlock), g.Hkv, g.B);
  e = cudaFuncSetAttribute(bwd_kv_f32_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_kv);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_kv_f32_kernel<D, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_kv);
  if (e != cudaSuccess) return e;
  bwd_kv_f32_kernel<D, true><<<grid_kv, kRowsPerBlock, smem_kv, s>>>(g, q, k, v, lse, d_o, delta,
                                                                      dk, err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwd_kv_f32_kernel<D, false><<<grid_kv, kRowsPerBlock, smem_kv, s>>>(g, q, k, v, lse, d_o, delta,
                                                                       dv, err);
  return cudaGetLastError();
}

template <typename T>
cudaError_t prep(const ChunkGeom& g, const T* o, const T* d_o, float* delta, float* dq_to_zero,
                 cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(g.B) * g.q_len * g.Hq;
  const int threads = 256;
  const int64_t blocks = (rows * 32 + threads - 1) / threads;
  bwd_prep_kernel<T><<<static_cast<unsigned>(blocks), threads, 0, s>>>(g, o, d_o, delta, dq_to_zero);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const ChunkGeom& g, const float* q, const float* k, const float* v,
                           float* o, float* lse, unsigned int* err, cudaStream_t s) {
  return g.d == 64 ? fwd_f32_d<64>(g, q, k, v, o, lse, err, s)
                   : fwd_f32_d<128>(g, q, k, v, o, lse, err, s);
}

cudaError_t launch_bwd_f32(const ChunkGeom& g, const float* q, const float* k, const float* v,
                           const float* lse, const float* d_o, const float* delta, float* dq,
                           float* dk, float* dv, unsigned int* err, cudaStream_t s) {
  return g.d == 64 ? bwd_f32_d<64>(g, q, k, v, lse, d_o, delta, dq, dk, dv, err, s)
                   : bwd_f32_d<128>(g, q, k, v, lse, d_o, delta, dq, dk, dv, err, s);
}

cudaError_t launch_bwd_stats_bf16(const ChunkGeom& g, const void* o, const void* d_o,
                                  const float* lse, float* stats, float* dq, cudaStream_t s) {
  const int n64 = static_cast<int>((g.q_len + 63) / 64);
  const int64_t rows = static_cast<int64_t>(g.B) * n64 * 64 * g.Hq;
  const int threads = 256;
  const int64_t blocks = (rows * 32 + threads - 1) / threads;
  bwd_stats_bf16_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
      g, n64, static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(d_o), lse, stats,
      dq);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep_f32(const ChunkGeom& g, const float* o, const float* d_o, float* delta,
                                cudaStream_t s) {
  return prep<float>(g, o, d_o, delta, nullptr, s);
}

cudaError_t launch_scale_rows_f32(float* a, float* b, int B, int64_t T, int64_t r0, int64_t r1,
                                  int64_t row_floats, float scale, cudaStream_t s) {
  const int64_t row4 = row_floats / 4;
  const int64_t n4 = static_cast<int64_t>(B) * (r1 - r0) * row4;
  if (n4 == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (n4 + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  scale2_rows_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
      reinterpret_cast<float4*>(a), reinterpret_cast<float4*>(b), T, r0, r1 - r0, row4, n4, scale);
  return cudaGetLastError();
}

cudaError_t launch_zero_f32(float* a, float* b, int64_t n, cudaStream_t s) {
  const int64_t n4 = n / 4;
  const int threads = 256;
  int64_t blocks = (n4 + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  zero2_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(reinterpret_cast<float4*>(a),
                                                                 reinterpret_cast<float4*>(b), n4);
  return cudaGetLastError();
}

}  // namespace seqattn
