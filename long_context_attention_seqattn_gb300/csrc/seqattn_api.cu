// seqattn_api.cu -- the C ABI declared in include/seqattn.h: argument
// validation (before any launch), TMA tensor maps, the per-device error word,
// and dispatch to the float32 and bf16 kernel families, the accumulator row
// scaling and the projection weight gradient kernel.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>

#include "internal.h"
#include "seqattn.h"

namespace seqattn {

// One error word per device (see sm103_ptx.cuh, "device error word").
__device__ unsigned int g_seqattn_error_word = 0u;

namespace {

thread_local std::string t_last_error;

seqattn_status fail(seqattn_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
seqattn_status fail(seqattn_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

seqattn_status ok() {
  t_last_error.clear();
  return SEQATTN_OK;
}

seqattn_status cuda_fail(cudaError_t e, const char* where) {
  return fail(SEQATTN_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_err_ptr[kMaxDevices] = {};

// Limit of every bounded device wait of the kernels launched from now on
// (seqattn_set_wait_limit); the default is about one second.
constexpr long long kDefaultWaitCycles = 2000000000LL;
std::atomic<long long> g_wait_cycles{kDefaultWaitCycles};

// Device address of this device's error word (looked up once per device).
cudaError_t error_word(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_seqattn_error_word);
    if (e != cudaSuccess) return e;
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_err_ptr[dev];
  return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 3-D bf16 tensor map over a [rows, heads, d] row-major tensor: box of
// {64 elements of d, 1 head, box_rows rows}, 128-byte swizzle (one 128-byte
// row of the box per smem row, the layout the MMA descriptors expect).
bool make_map(CUtensorMap* m, const void* base, int d, int heads, int64_t rows, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  memset(m, 0, sizeof(*m));
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(heads) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D tensor map over a row-major [B, T, cols] tensor of bf16 (128-byte
// swizzle, box {64 columns, box_rows rows, 1 batch entry}) or float32 (no
// swizzle, box {box_cols, box_rows, 1}).  Rows past T and columns past
// `cols` read as zero and are never written.
bool make_map_btc(CUtensorMap* m, const void* base, int64_t B, int64_t T, int64_t cols, bool fp32,
                  int box_cols, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  memset(m, 0, sizeof(*m));
  const cuuint64_t es_bytes = fp32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * es_bytes,
                           static_cast<cuuint64_t>(T) * static_cast<cuuint64_t>(cols) * es_bytes};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  fp32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D float32 tensor map over the [B, T, heads, d] accumulator, cut at row
// `rows` of every batch entry (the chunk's end: rows past it are never
// written): box {32 of d, 1 head, 128 rows, 1 batch entry}, 128-byte swizzle.
bool make_map_accum(CUtensorMap* m, const void* base, int d, int heads, int64_t T, int64_t rows, int B) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  memset(m, 0, sizeof(*m));
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(heads) * d * 4,
                           static_cast<cuuint64_t>(T) * heads * d * 4};
  cuuint32_t box[4] = {32, 1, 128, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

seqattn_status check_problem(const seqattn_problem* pb) {
  if (pb == nullptr) return fail(SEQATTN_ERR_INVALID_ARG, "problem is NULL");
  if (pb->batch < 1 || pb->num_q_heads < 1 || pb->num_kv_heads < 1 || pb->seq_capacity < 1)
    return fail(SEQATTN_ERR_INVALID_ARG, "batch, heads and seq_capacity must be >= 1");
  if (pb->num_q_heads % pb->num_kv_heads != 0)
    return fail(SEQATTN_ERR_INVALID_ARG, "num_q_heads (%d) is not a multiple of num_kv_heads (%d)",
                pb->num_q_heads, pb->num_kv_heads);
  if (pb->head_dim != 64 && pb->head_dim != 128)
    return fail(SEQATTN_ERR_INVALID_ARG, "head_dim %d is not 64 or 128", pb->head_dim);
  if (pb->dtype != SEQATTN_BF16 && pb->dtype != SEQATTN_FP32)
    return fail(SEQATTN_ERR_INVALID_ARG, "unknown dtype %d", pb->dtype);
  if (static_cast<int64_t>(pb->batch) * pb->seq_capacity > INT32_MAX)
    return fail(SEQATTN_ERR_INVALID_ARG, "batch * seq_capacity exceeds 2^31 - 1 rows");
  return SEQATTN_OK;
}

seqattn_status check_chunk(const seqattn_problem* pb, int64_t q_start, int64_t q_len,
                           int64_t prefix_len, float scale, ChunkGeom* g) {
  seqattn_status s = check_problem(pb);
  if (s != SEQATTN_OK) return s;
  if (q_len < 0) return fail(SEQATTN_ERR_INVALID_ARG, "q_len %lld < 0", (long long)q_len);
  if (q_start < 0 || prefix_len < 0 || prefix_len > q_start)
    return fail(SEQATTN_ERR_INVALID_ARG, "need 0 <= prefix_len <= q_start (got %lld, %lld)",
                (long long)prefix_len, (long long)q_start);
  if (q_start + q_len > pb->seq_capacity)
    return fail(SEQATTN_ERR_INVALID_ARG, "q_start + q_len = %lld exceeds seq_capacity %lld",
                (long long)(q_start + q_len), (long long)pb->seq_capacity);
  if (!(scale > 0.f) || !isfinite(scale))
    return fail(SEQATTN_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
  if (static_cast<int64_t>(pb->batch) * q_len > INT32_MAX)
    return fail(SEQATTN_ERR_INVALID_ARG, "batch * q_len exceeds 2^31 - 1 rows");
  g->B = pb->batch;
  g->Hq = pb->num_q_heads;
  g->Hkv = pb->num_kv_heads;
  g->G = pb->num_q_heads / pb->num_kv_heads;
  g->d = pb->head_dim;
  g->T = pb->seq_capacity;
  g->q_start = q_start;
  g->q_len = q_len;
  g->kv_begin = q_start - prefix_len;
  g->scale = scale;
  g->wait_cycles = g_wait_cycles.load(std::memory_order_relaxed);
  return SEQATTN_OK;
}

seqattn_status check_ptrs(std::initializer_list<std::pair<const void*, const char*>> ps) {
  for (auto& p : ps) {
    if (p.first == nullptr) return fail(SEQATTN_ERR_INVALID_ARG, "%s is NULL", p.second);
    if (!aligned16(p.first))
      return fail(SEQATTN_ERR_INVALID_ARG, "%s is not 16-byte aligned", p.second);
  }
  return SEQATTN_OK;
}

size_t workspace_bytes(const seqattn_problem* pb, int64_t q_len) {
  // float32: Delta [B, Hq, q_len].  bf16: -L log2(e) and Delta per 64-row
  // query tile, [B, Hq, ceil(q_len / 64), 2, 64].  Rounded up to 256 bytes.
  const size_t rows = pb->dtype == SEQATTN_BF16 ? static_cast<size_t>((q_len + 63) / 64) * 128
                                                : static_cast<size_t>(q_len);
  const size_t bytes = static_cast<size_t>(pb->batch) * pb->num_q_heads * rows * sizeof(float);
  return (bytes + 255) & ~static_cast<size_t>(255);
}

}  // namespace
}  // namespace seqattn

using namespace seqattn;

extern "C" {

seqattn_status seqattn_chunk_fwd(const seqattn_problem* pb, int64_t q_start, int64_t q_len,
                                 int64_t prefix_len, float softmax_scale, const void* q,
                                 const void* k, const void* v, void* o, float* lse,
                                 seqattn_stream_t stream) {
  ChunkGeom g;
  seqattn_status s = check_chunk(pb, q_start, q_len, prefix_len, softmax_scale, &g);
  if (s != SEQATTN_OK) return s;
  if (q_len == 0) return ok();
  s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {o, "o"}, {lse, "lse"}});
  if (s != SEQATTN_OK) return s;
  unsigned int* err = nullptr;
  cudaError_t e = error_word(&err);
  if (e != cudaSuccess) return cuda_fail(e, "error word");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (pb->dtype == SEQATTN_FP32) {
    e = launch_fwd_f32(g, static_cast<const float*>(q), static_cast<const float*>(k),
                       static_cast<const float*>(v), static_cast<float*>(o), lse, err, st);
    return e == cudaSuccess ? ok() : cuda_fail(e, "fwd_f32 launch");
  }
  Bf16FwdMaps maps;
  if (!make_map(&maps.q, q, g.d, g.Hq, static_cast<int64_t>(g.B) * q_len, 128) ||
      !make_map(&maps.k, k, g.d, g.Hkv, static_cast<int64_t>(g.B) * g.T, 128) ||
      !make_map(&maps.v, v, g.d, g.Hkv, static_cast<int64_t>(g.B) * g.T, 128))
    return fail(SEQATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the forward operands");
  e = launch_fwd_bf16(g, maps, o, lse, err, st);
  return e == cudaSuccess ? ok() : cuda_fail(e, "fwd_bf16 launch");
}

seqattn_status seqattn_chunk_bwd(const seqattn_problem* pb, int64_t q_start, int64_t q_len,
                                 int64_t prefix_len, float softmax_scale, const void* q,
                                 const void* k, const void* v, const void* o, const float* lse,
                                 const void* d_o, float* dq, float* dk_accum, float* dv_accum,
                                 void* workspace, size_t workspace_size, seqattn_stream_t stream) {
  ChunkGeom g;
  seqattn_status s = check_chunk(pb, q_start, q_len, prefix_len, softmax_scale, &g);
  if (s != SEQATTN_OK) return s;
  if (q_len == 0) return ok();
  s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {o, "o"}, {lse, "lse"}, {d_o, "d_o"}, {dq, "dq"},
                  {dk_accum, "dk_accum"}, {dv_accum, "dv_accum"}, {workspace, "workspace"}});
  if (s != SEQATTN_OK) return s;
  if (workspace_size < workspace_bytes(pb, q_len))
    return fail(SEQATTN_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_size, workspace_bytes(pb, q_len));
  unsigned int* err = nullptr;
  cudaError_t e = error_word(&err);
  if (e != cudaSuccess) return cuda_fail(e, "error word");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  float* delta = static_cast<float*>(workspace);
  if (pb->dtype == SEQATTN_FP32) {
    e = launch_bwd_prep_f32(g, static_cast<const float*>(o), static_cast<const float*>(d_o), delta,
                            st);
    if (e != cudaSuccess) return cuda_fail(e, "bwd_prep launch");
    e = launch_bwd_f32(g, static_cast<const float*>(q), static_cast<const float*>(k),
                       static_cast<const float*>(v), lse, static_cast<const float*>(d_o), delta,
                       dq, dk_accum, dv_accum, err, st);
    return e == cudaSuccess ? ok() : cuda_fail(e, "bwd_f32 launch");
  }
  Bf16BwdMaps maps;
  if (!make_map(&maps.q, q, g.d, g.Hq, static_cast<int64_t>(g.B) * q_len, 64) ||
      !make_map(&maps.d_o, d_o, g.d, g.Hq, static_cast<int64_t>(g.B) * q_len, 64) ||
      !make_map(&maps.k, k, g.d, g.Hkv, static_cast<int64_t>(g.B) * g.T, 128) ||
      !make_map(&maps.v, v, g.d, g.Hkv, static_cast<int64_t>(g.B) * g.T, 128) ||
      !make_map_accum(&maps.dk, dk_accum, g.d, g.Hkv, g.T, q_start + q_len, g.B) ||
      !make_map_accum(&maps.dv, dv_accum, g.d, g.Hkv, g.T, q_start + q_len, g.B))
    return fail(SEQATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the backward operands");
  e = launch_bwd_stats_bf16(g, o, d_o, lse, delta, dq, st);
  if (e != cudaSuccess) return cuda_fail(e, "bwd_stats launch");
  e = launch_bwd_bf16(g, maps, delta, dq, dk_accum, dv_accum, err, st);
  return e == cudaSuccess ? ok() : cuda_fail(e, "bwd_bf16 launch");
}

seqattn_status seqattn_reset_accum(const seqattn_problem* pb, float* dk_accum, float* dv_accum,
                                   seqattn_stream_t stream) {
  seqattn_status s = check_problem(pb);
  if (s != SEQATTN_OK) return s;
  s = check_ptrs({{dk_accum, "dk_accum"}, {dv_accum, "dv_accum"}});
  if (s != SEQATTN_OK) return s;
  const int64_t n = static_cast<int64_t>(pb->batch) * pb->seq_capacity * pb->num_kv_heads *
                    pb->head_dim;
  cudaError_t e = launch_zero_f32(dk_accum, dv_accum, n, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "reset launch");
}

seqattn_status seqattn_scale_accum_rows(const seqattn_problem* pb, int64_t row_begin,
                                        int64_t row_end, float scale, float* dk_accum,
                                        float* dv_accum, seqattn_stream_t stream) {
  seqattn_status s = check_problem(pb);
  if (s != SEQATTN_OK) return s;
  if (row_begin < 0 || row_end < row_begin || row_end > pb->seq_capacity)
    return fail(SEQATTN_ERR_INVALID_ARG, "need 0 <= row_begin <= row_end <= seq_capacity (got %lld, %lld)",
                (long long)row_begin, (long long)row_end);
  if (!isfinite(scale)) return fail(SEQATTN_ERR_INVALID_ARG, "scale must be finite");
  s = check_ptrs({{dk_accum, "dk_accum"}, {dv_accum, "dv_accum"}});
  if (s != SEQATTN_OK) return s;
  cudaError_t e = launch_scale_rows_f32(dk_accum, dv_accum, pb->batch, pb->seq_capacity, row_begin, row_end,
                                        static_cast<int64_t>(pb->num_kv_heads) * pb->head_dim, scale,
                                        reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "scale launch");
}

seqattn_status seqattn_proj_wgrad(int32_t batch, int64_t seq_len, int64_t row_begin,
                                  int64_t row_end, int32_t d_model, int32_t n, const void* h,
                                  const float* g, float* dw, seqattn_stream_t stream) {
  if (batch < 1 || seq_len < 1) return fail(SEQATTN_ERR_INVALID_ARG, "batch and seq_len must be >= 1");
  if (row_begin < 0 || row_end < row_begin || row_end > seq_len)
    return fail(SEQATTN_ERR_INVALID_ARG, "need 0 <= row_begin <= row_end <= seq_len (got %lld, %lld)",
                (long long)row_begin, (long long)row_end);
  if (d_model < 8 || d_model % 8 || n < 8 || n % 8)
    return fail(SEQATTN_ERR_INVALID_ARG, "d_model (%d) and n (%d) must be positive multiples of 8", d_model, n);
  if (static_cast<int64_t>(batch) * seq_len > INT32_MAX || seq_len * static_cast<int64_t>(n) > INT32_MAX)
    return fail(SEQATTN_ERR_INVALID_ARG, "batch * seq_len or seq_len * n exceeds 2^31 - 1");
  seqattn_status s = check_ptrs({{h, "h"}, {g, "g"}, {dw, "dw"}});
  if (s != SEQATTN_OK) return s;
  if (row_end == row_begin) return ok();
  unsigned int* err = nullptr;
  cudaError_t e = error_word(&err);
  if (e != cudaSuccess) return cuda_fail(e, "error word");
  WgradMaps maps;
  if (!make_map_btc(&maps.h, h, batch, seq_len, d_model, false, 64, kWgradStageRows) ||
      !make_map_btc(&maps.g, g, batch, seq_len, n, true, 128, kWgradStageRows) ||
      !make_map_btc(&maps.dw, dw, 1, d_model, n, true, 128, 32))
    return fail(SEQATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for h, g or dw");
  e = launch_wgrad_bf16(maps, batch, row_begin, row_end, d_model, n, err,
                        g_wait_cycles.load(std::memory_order_relaxed), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "wgrad launch");
}

size_t seqattn_bwd_workspace_size(const seqattn_problem* pb, int64_t q_len) {
  if (check_problem(pb) != SEQATTN_OK || q_len < 0) return 0;
  return workspace_bytes(pb, q_len);
}

seqattn_status seqattn_sync_status(seqattn_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned int* err = nullptr;
  if ((e = error_word(&err)) != cudaSuccess) return cuda_fail(e, "error word");
  unsigned int w = 0;
  if ((e = cudaMemcpy(&w, err, sizeof(w), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read error word");
  if (w != 0) {
    const unsigned int zero = 0;
    if ((e = cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "clear error word");
    return fail(SEQATTN_ERR_TIMEOUT, "a kernel gave up a bounded wait (error word 0x%x)", w);
  }
  return ok();
}

void seqattn_set_wait_limit(int64_t cycles) {
  g_wait_cycles.store(cycles > 0 ? cycles : kDefaultWaitCycles, std::memory_order_relaxed);
}

const char* seqattn_status_string(seqattn_status s) {
  switch (s) {
    case SEQATTN_OK: return "ok";
    case SEQATTN_ERR_INVALID_ARG: return "invalid argument";
    case SEQATTN_ERR_UNSUPPORTED: return "unsupported";
    case SEQATTN_ERR_CUDA: return "CUDA error";
    case SEQATTN_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* seqattn_last_error(void) { return t_last_error.c_str(); }

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward for callers that cannot allocate device memory.
//
// Some callers have no way to provide the backward's scratch buffer: their
// device memory is owned by another allocator (a framework's caching
// allocator or a fixed arena handed out at start-up) and the plugin interface
// they call through passes only the tensors themselves.  For them the Delta
// scratch lives in a fixed array in this file, so the call needs nothing
// beyond its inputs and outputs.
// ---------------------------------------------------------------------------
namespace seqattn {
namespace {

// Row-statistics scratch (what seqattn_bwd_workspace_size asks for, at most
// 4 MiB) on every GPU that loads the library, held until the process exits.
static __device__ __align__(256) float g_noalloc_delta[SEQATTN_NOALLOC_MAX_DELTA];

float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of this device's scratch array.  Host code cannot use the
// array's name as a device pointer, so the address is looked up once per
// device, with that device current, on the first call there.
cudaError_t noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_delta);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace seqattn

extern "C" seqattn_status seqattn_chunk_bwd_noalloc(
    const seqattn_problem* pb, int64_t q_start, int64_t q_len, int64_t prefix_len,
    float softmax_scale, const void* q, const void* k, const void* v, const void* o,
    const float* lse, const void* d_o, float* dq, float* dk_accum, float* dv_accum,
    seqattn_stream_t stream) {
  ChunkGeom g;
  seqattn_status s = check_chunk(pb, q_start, q_len, prefix_len, softmax_scale, &g);
  if (s != SEQATTN_OK) return s;
  if (q_len == 0) return ok();
  s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {o, "o"}, {lse, "lse"}, {d_o, "d_o"}, {dq, "dq"},
                  {dk_accum, "dk_accum"}, {dv_accum, "dv_accum"}});
  if (s != SEQATTN_OK) return s;
  const size_t need = workspace_bytes(pb, q_len);
  if (need > sizeof(float) * static_cast<size_t>(SEQATTN_NOALLOC_MAX_DELTA))
    return fail(SEQATTN_ERR_INVALID_ARG,
                "this chunk needs %zu bytes of row statistics, more than the fixed scratch of %d "
                "floats of seqattn_chunk_bwd_noalloc; use seqattn_chunk_bwd with a workspace",
                need, SEQATTN_NOALLOC_MAX_DELTA);
  float* delta = nullptr;
  cudaError_t e = noalloc_scratch(&delta);
  if (e != cudaSuccess) return cuda_fail(e, "scratch address");
  unsigned int* err = nullptr;
  if ((e = error_word(&err)) != cudaSuccess) return cuda_fail(e, "error word");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (pb->dtype == SEQATTN_FP32) {
    e = launch_bwd_prep_f32(g, static_cast<const float*>(o), static_cast<const float*>(d_o), delta,
                            st);
    if (e != cudaSuccess) return cuda_fail(e, "bwd_prep launch");
    e = launch_bwd_f32(g, static_cast<const float*>(q), static_cast<const float*>(k),
                       static_cast<const float*>(v), lse, static_cast<const float*>(d_o), delta,
                       dq, dk_accum, dv_accum, err, st);
    return e == cudaSuccess ? ok() : cuda_fail(e, "bwd_f32 launch");
  }
  Bf16BwdMaps maps;
  if (!make_map(&maps.q, q, g.d, g.Hq, static_cast<int64_t>(g.B) * q_len, 64) ||
      !make_map(&maps.d_o, d_o, g.d, g.Hq, static_cast<int64_t>(g.B) * q_len, 64) ||
      !make_map(&maps.k, k, g.d, g.Hkv, static_cast<int64_t>(g.B) * g.T, 128) ||
      !make_map(&maps.v, v, g.d, g.Hkv, static_cast<int64_t>(g.B) * g.T, 128) ||
      !make_map_accum(&maps.dk, dk_accum, g.d, g.Hkv, g.T, q_start + q_len, g.B) ||
      !make_map_accum(&maps.dv, dv_accum, g.d, g.Hkv, g.T, q_start + q_len, g.B))
    return fail(SEQATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the backward operands");
  e = launch_bwd_stats_bf16(g, o, d_o, lse, delta, dq, st);
  if (e != cudaSuccess) return cuda_fail(e, "bwd_stats launch");
  e = launch_bwd_bf16(g, maps, delta, dq, dk_accum, dv_accum, err, st);
  return e == cudaSuccess ? ok() : cuda_fail(e, "bwd_bf16 launch");
}
