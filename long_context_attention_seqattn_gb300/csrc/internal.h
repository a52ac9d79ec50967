// internal.h -- launch plumbing shared between the C-ABI front end and the
// kernel translation units of libseqattn.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace seqattn {

// Geometry of one chunk call, after validation.
struct ChunkGeom {
  int B, Hq, Hkv, G, d;
  int64_t T;         // cache rows
  int64_t q_start;   // absolute row of the chunk's first query
  int64_t q_len;     // rows in the chunk
  int64_t kv_begin;  // first visible key row (q_start - prefix_len)
  float scale;       // softmax scale
  long long wait_cycles;  // limit of every bounded device wait (SM cycles)
};

// ---- float32 exact path (SIMT FMA) ----------------------------------------
cudaError_t launch_fwd_f32(const ChunkGeom& g, const float* q, const float* k, const float* v,
                           float* o, float* lse, unsigned int* err, cudaStream_t s);
cudaError_t launch_bwd_f32(const ChunkGeom& g, const float* q, const float* k, const float* v,
                           const float* lse, const float* d_o, const float* delta, float* dq,
                           float* dk, float* dv, unsigned int* err, cudaStream_t s);

// ---- Delta = rowsum(dO o O) and the backward row statistics ---------------
// bf16 path: per 64-row query tile, -L log2(e) and Delta side by side in a
// padded [B, Hq, ceil(q_len / 64), 2, 64] float32 array (padding rows -inf, 0);
// also zeroes dq.
cudaError_t launch_bwd_stats_bf16(const ChunkGeom& g, const void* o, const void* d_o,
                                  const float* lse, float* stats, float* dq, cudaStream_t s);
cudaError_t launch_bwd_prep_f32(const ChunkGeom& g, const float* o, const float* d_o,
                                float* delta, cudaStream_t s);

// ---- zero fill of the float32 accumulators ---------------------------------
cudaError_t launch_zero_f32(float* a, float* b, int64_t n, cudaStream_t s);
// rows [r0, r1) of two [B, T, row_floats] float32 arrays times `scale` (0 stores zeros)
cudaError_t launch_scale_rows_f32(float* a, float* b, int B, int64_t T, int64_t r0, int64_t r1,
                                  int64_t row_floats, float scale, cudaStream_t s);

// ---- bf16 tensor-core path (TMA + tcgen05 + TMEM) -------------------------
// Tensor maps are built by the front end (make_map in seqattn_api.cu).
struct Bf16FwdMaps {
  CUtensorMap q, k, v;
};
struct Bf16BwdMaps {
  CUtensorMap q, k, v, d_o;
  CUtensorMap dk, dv;   // fp32 [B][rows < q_end][Hkv][d], box {32, 1, 128, 1}, 128-byte swizzle
};
cudaError_t launch_fwd_bf16(const ChunkGeom& g, const Bf16FwdMaps& maps, void* o, float* lse,
                            unsigned int* err, cudaStream_t s);
// `stats` as written by launch_bwd_stats_bf16.
cudaError_t launch_bwd_bf16(const ChunkGeom& g, const Bf16BwdMaps& maps, const float* stats,
                            float* dq, float* dk, float* dv, unsigned int* err, cudaStream_t s);

// ---- projection weight gradient (tcgen05, G rounded to bf16 in the kernel) -
// Rows (tokens) per pipeline stage: the height of the h and g boxes.
constexpr int kWgradStageRows = 64;
// h: bf16 [B, T, d_model], box {64 columns, kWgradStageRows rows, 1}, 128-byte swizzle;
// g: fp32 [B, T, n], box {128 columns, kWgradStageRows rows, 1}, no swizzle;
// dw: fp32 [1, d_model, n], box {128 columns, 32 rows, 1}, no swizzle (the
// target of the epilogue's reduce-adds).
struct WgradMaps {
  CUtensorMap h, g, dw;
};
cudaError_t launch_wgrad_bf16(const WgradMaps& maps, int32_t batch, int64_t row_begin, int64_t row_end,
                              int32_t d_model, int32_t n, unsigned int* err, long long wait_cycles,
                              cudaStream_t s);

}  // namespace seqattn
