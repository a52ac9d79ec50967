// wgrad.cu -- projection weight gradient of a chunk's rows, the step after
// the attention path (SeCO review page, major comment 1 on Algorithm 2: once
// chunk i's cache gradient is complete, chunk i's graph -- here the Q/K/V
// projections X = H W -- is backpropagated):
//   dW[d_model, n] += sum over batch entries b and rows r of H[b, r]^T G[b, r]
// G (dQ, or the finished dK / dV rows; float32) is rounded to bf16 into the
// caller's workspace by one grid-stride kernel, then a cuBLASLt bf16 GEMM with
// float32 accumulation adds H^T G into dW (one GEMM per batch entry, beta = 1).
#include <cublasLt.h>
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"

namespace seqattn {
namespace {

// rows [r0, r0 + rows) of G [B, T, n] float32 -> dst [B, rows, n] bf16, four
// values per thread and step (n % 4 == 0)
__global__ void rows_to_bf16_kernel(const float4* __restrict__ g, uint2* __restrict__ dst, int64_t T, int64_t r0,
                                    int64_t rows, int64_t n4, int64_t total4) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t per_b = rows * n4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total4; i += stride) {
    const int64_t b = i / per_b;
    const float4 x = g[(b * T + r0) * n4 + (i - b * per_b)];
    __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
    dst[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
}

constexpr int kMaxDevices = 64;
std::mutex g_lt_mu;
cublasLtHandle_t g_lt[kMaxDevices] = {};

cublasStatus_t lt_handle(cublasLtHandle_t* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CUBLAS_STATUS_NOT_INITIALIZED;
  std::lock_guard<std::mutex> lk(g_lt_mu);
  if (g_lt[dev] == nullptr) {
    cublasStatus_t s = cublasLtCreate(&g_lt[dev]);
    if (s != CUBLAS_STATUS_SUCCESS) return s;
  }
  *out = g_lt[dev];
  return CUBLAS_STATUS_SUCCESS;
}

size_t bf16_bytes(int32_t batch, int64_t rows, int32_t n) {
  const size_t b = static_cast<size_t>(batch) * rows * n * 2;
  return (b + 255) & ~static_cast<size_t>(255);
}

}  // namespace

size_t wgrad_workspace_bytes(int32_t batch, int64_t rows, int32_t n) {
  return bf16_bytes(batch, rows, n) + kWgradLtWorkspace;
}

WgradStatus launch_wgrad(int32_t batch, int64_t seq_len, int64_t row_begin, int64_t row_end, int32_t d_model,
                         int32_t n, const void* h, const float* g, float* dw, void* workspace,
                         size_t workspace_bytes, cudaStream_t s) {
  WgradStatus st;
  const int64_t rows = row_end - row_begin;
  const size_t gb = bf16_bytes(batch, rows, n);
  uint2* g16 = static_cast<uint2*>(workspace);
  void* lt_ws = static_cast<uint8_t*>(workspace) + gb;
  const size_t lt_ws_bytes = workspace_bytes - gb;
  // 1. G rows -> bf16
  const int64_t n4 = n / 4;
  const int64_t total4 = static_cast<int64_t>(batch) * rows * n4;
  const int threads = 256;
  int64_t blocks = (total4 + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  rows_to_bf16_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(reinterpret_cast<const float4*>(g), g16,
                                                                         seq_len, row_begin, rows, n4, total4);
  if ((st.cuda = cudaGetLastError()) != cudaSuccess) return st;

  // 2. dW (row-major [d_model][n] = column-major n x d_model) +=
  //    G16 (column-major n x rows) * H^T, H row-major [rows][d_model] being
  //    the column-major d_model x rows matrix taken transposed.
  cublasLtHandle_t lt;
  {
    const cublasStatus_t hs = lt_handle(&lt);
    if (hs != CUBLAS_STATUS_SUCCESS) {
      st.blas = hs;
      return st;
    }
  }
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  const cublasOperation_t tn = CUBLAS_OP_N, tt = CUBLAS_OP_T;
  const float one = 1.f;
  cublasLtMatmulHeuristicResult_t heur = {};
  int found = 0;
  auto done = [&]() {
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (la) cublasLtMatrixLayoutDestroy(la);
    if (lb) cublasLtMatrixLayoutDestroy(lb);
    if (lc) cublasLtMatrixLayoutDestroy(lc);
    if (op) cublasLtMatmulDescDestroy(op);
  };
#define SEQATTN_LT(call)                                   \
  do {                                                     \
    const cublasStatus_t cs_ = (call);                     \
    if (cs_ != CUBLAS_STATUS_SUCCESS) {                    \
      st.blas = cs_;                                       \
      done();                                              \
      return st;                                           \
    }                                                      \
  } while (0)
  SEQATTN_LT(cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F));
  SEQATTN_LT(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &tn, sizeof(tn)));
  SEQATTN_LT(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tt, sizeof(tt)));
  SEQATTN_LT(cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, n, rows, n));
  SEQATTN_LT(cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, d_model, rows, d_model));
  SEQATTN_LT(cublasLtMatrixLayoutCreate(&lc, CUDA_R_32F, n, d_model, n));
  SEQATTN_LT(cublasLtMatmulPreferenceCreate(&pref));
  SEQATTN_LT(cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &lt_ws_bytes,
                                                  sizeof(lt_ws_bytes)));
  SEQATTN_LT(cublasLtMatmulAlgoGetHeuristic(lt, op, la, lb, lc, lc, pref, 1, &heur, &found));
  if (found < 1) {
    st.blas = CUBLAS_STATUS_NOT_SUPPORTED;
    done();
    return st;
  }
  const __nv_bfloat16* hb = static_cast<const __nv_bfloat16*>(h);
  for (int32_t b = 0; b < batch; ++b) {
    const void* a_ptr = reinterpret_cast<const __nv_bfloat16*>(g16) + static_cast<int64_t>(b) * rows * n;
    const void* b_ptr = hb + (static_cast<int64_t>(b) * seq_len + row_begin) * d_model;
    SEQATTN_LT(cublasLtMatmul(lt, op, &one, a_ptr, la, b_ptr, lb, &one, dw, lc, dw, lc, &heur.algo, lt_ws,
                              lt_ws_bytes, s));
  }
#undef SEQATTN_LT
  done();
  return st;
}

}  // namespace seqattn
