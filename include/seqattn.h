/*
 * seqattn.h -- C ABI of libseqattn: sequence-partitioned (chunked) causal
 * attention forward and exact backward on one GB300 (sm_103a).
 *
 * The operation is the per-chunk attention of StreamBP ("StreamBP:
 * Memory-Efficient Exact Backpropagation for Long Sequence Training of LLMs",
 * review page): Property 3.1 ("What carries the argument") says chunk i's
 * output needs only Q^(i), K^(:i), V^(:i); Eq. (1) writes the gradient as a
 * sum of per-chunk terms, and the "Circularity Check" names the partitioned
 * attention of Eqs. (12)-(14) and the running sum that accumulates the
 * per-chunk dK/dV over the prefix.  The same chunk-by-chunk backward with
 * key/value caches as checkpoints is SeCO's ("Training Long-Context LLMs
 * Efficiently via Chunk-wise Optimization", review page, "What carries the
 * argument").
 *
 * Notation: B batch, T = seq_capacity (cache rows), Hq query heads, Hkv
 * key/value heads, G = Hq / Hkv, d = head_dim.  Query head h reads key/value
 * head h / G (contiguous groups).  A chunk is q_len query rows at absolute
 * positions [q_start, q_start + q_len); row r attends keys
 * [q_start - prefix_len, q_start + r] (causal inside the chunk).  prefix_len ==
 * q_start is the method's full prefix K^(:i); a smaller prefix_len starts the
 * window later.
 *
 * Tensor layouts (all dense, row-major, element strides implied):
 *   q, o, d_o : [B, q_len, Hq, d]          chunk-local rows
 *   k, v      : [B, T, Hkv, d]             full cache, row 0 = token 0
 *   lse       : [B, Hq, q_len]   float32   natural-log row logsumexp of the
 *                                          scaled scores (the stored M^(i))
 *   dq        : [B, q_len, Hq, d] float32
 *   dk_accum,
 *   dv_accum  : [B, T, Hkv, d]    float32  running sums over chunks
 * Element type of q, k, v, o, d_o: bfloat16 for SEQATTN_BF16, float32 for
 * SEQATTN_FP32.  Every pointer is a DEVICE pointer owned by the caller and
 * must be 16-byte aligned; the library allocates nothing and keeps no state
 * between calls other than a device-side error word (and the fixed scratch
 * array of seqattn_chunk_bwd_noalloc).
 *
 * All work is enqueued asynchronously on `stream` (a cudaStream_t; 0 is the
 * legacy default stream).  Argument errors are detected on the host before
 * anything is launched.  Launch failures return SEQATTN_ERR_CUDA.  Every
 * device-side wait in the kernels is bounded: a wait that runs out sets the
 * device error word and the kernel returns early; that is reported as
 * SEQATTN_ERR_TIMEOUT by the next call of seqattn_sync_status().
 * No function throws, aborts or prints.
 */
#ifndef SEQATTN_H
#define SEQATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* seqattn_stream_t; /* same type as cudaStream_t */

typedef enum {
  SEQATTN_OK = 0,
  SEQATTN_ERR_INVALID_ARG = 1, /* bad pointer, shape, alignment or scale */
  SEQATTN_ERR_UNSUPPORTED = 2, /* valid request this build does not cover */
  SEQATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  SEQATTN_ERR_TIMEOUT = 4      /* a bounded device-side wait ran out */
} seqattn_status;

typedef enum { SEQATTN_BF16 = 0, SEQATTN_FP32 = 1 } seqattn_dtype;

typedef struct {
  int32_t batch;        /* B >= 1 */
  int32_t num_q_heads;  /* Hq >= 1 */
  int32_t num_kv_heads; /* Hkv >= 1, Hq % Hkv == 0 */
  int32_t head_dim;     /* d: 64 or 128 */
  int64_t seq_capacity; /* T: rows of the k/v caches and dk/dv accumulators */
  int32_t dtype;        /* seqattn_dtype */
} seqattn_problem;

/*
 * Forward of one chunk: O^(i) = softmax(scale * Q^(i) K^(:i)^T, causal) V^(:i)
 * and the row logsumexp (StreamBP review page, Property 3.1 and Eqs. (12)-(14)
 * named in the "Circularity Check"; the stored row statistic M^(i) of the
 * verdict page's stored-activation list).
 *   q_start, q_len, prefix_len: chunk rows and key window as described above;
 *     requires 0 <= prefix_len <= q_start and q_start + q_len <= T.
 *     q_len == 0 is a no-op.
 *   softmax_scale: finite, > 0 (usually 1/sqrt(d)).
 *   o (out), lse (out): overwritten.
 * Both dtypes accept any q_start, q_len, prefix_len and d in {64, 128}.
 */
seqattn_status seqattn_chunk_fwd(const seqattn_problem* pb, int64_t q_start, int64_t q_len,
                                 int64_t prefix_len, float softmax_scale, const void* q,
                                 const void* k, const void* v, void* o, float* lse,
                                 seqattn_stream_t stream);

/*
 * Exact backward of one chunk (StreamBP review page, Eq. (1) and the running
 * sum of the "Circularity Check"; major comment 1 of its referee report names
 * dK^(:i), dV^(:i) over the prefix).  With P = exp(scale*QK^T - lse),
 * dP = dO V^T, Delta = rowsum(dO o O), dS = P o (dP - Delta):
 *   dq (out, overwritten)      = scale * dS K
 *   dk_accum rows [q_start - prefix_len, q_start + q_len) += scale * dS^T Q
 *   dv_accum rows [q_start - prefix_len, q_start + q_len) += P^T dO
 * (summed over the G query heads of each key/value head).  o and lse are the
 * forward's outputs for this chunk.  Other accumulator rows are untouched.
 *   workspace: device scratch of at least seqattn_bwd_workspace_size(pb,
 *     q_len) bytes, 256-byte aligned, caller-owned, contents not preserved.
 * Size rules as for seqattn_chunk_fwd.  Calls on one stream accumulate in
 * order.  SEQATTN_BF16: the accumulator updates are fp32 reduce-adds done in
 * L2 (atomic per element), so calls for different chunks may run concurrently
 * on different streams, each with a workspace of its own (the order of the
 * fp32 additions, and so the last bits of the sums, then varies between
 * runs).  SEQATTN_FP32: the updates are
 * plain read-modify-writes; two calls that update the same accumulator rows
 * must not run concurrently.
 */
seqattn_status seqattn_chunk_bwd(const seqattn_problem* pb, int64_t q_start, int64_t q_len,
                                 int64_t prefix_len, float softmax_scale, const void* q,
                                 const void* k, const void* v, const void* o, const float* lse,
                                 const void* d_o, float* dq, float* dk_accum, float* dv_accum,
                                 void* workspace, size_t workspace_bytes,
                                 seqattn_stream_t stream);

/*
 * Backward of one chunk for callers that cannot allocate device memory.  The
 * paper has no counterpart: this is a library convenience.  Some callers own
 * no allocator of their own -- their device memory belongs to another
 * allocator (a framework's caching allocator or a fixed arena) and the
 * interface they call through passes only the tensors -- so they cannot
 * provide the workspace seqattn_chunk_bwd asks for.  This entry point computes
 * exactly what seqattn_chunk_bwd computes, with the same arguments minus the
 * workspace, and calls no allocation routine.
 *
 * Its scratch (the per-row statistics, seqattn_bwd_workspace_size(pb, q_len)
 * bytes) is a fixed device array inside the library of
 * SEQATTN_NOALLOC_MAX_DELTA floats (4 MiB), which every GPU that loads the
 * library holds until the process exits.  Larger requests return
 * SEQATTN_ERR_INVALID_ARG (use seqattn_chunk_bwd instead).  The first
 * call on a device looks up that device's address of the array; make that
 * first call before any stream capture.  Every call shares the one array, so
 * calls that overlap on the GPU (different streams, or different host
 * threads) race on it and must be serialised by the caller.
 */
#define SEQATTN_NOALLOC_MAX_DELTA (1 << 20)
seqattn_status seqattn_chunk_bwd_noalloc(const seqattn_problem* pb, int64_t q_start,
                                         int64_t q_len, int64_t prefix_len, float softmax_scale,
                                         const void* q, const void* k, const void* v,
                                         const void* o, const float* lse, const void* d_o,
                                         float* dq, float* dk_accum, float* dv_accum,
                                         seqattn_stream_t stream);

/* Zero both float32 accumulators ([B, T, Hkv, d] each) before the first chunk
 * of a backward pass (the running sum starts at zero). */
seqattn_status seqattn_reset_accum(const seqattn_problem* pb, float* dk_accum, float* dv_accum,
                                   seqattn_stream_t stream);

/*
 * Multiply rows [row_begin, row_end) of both float32 accumulators by `scale`;
 * scale == 0 stores zeros.  This is the step SpaCO adds to the chunk loop
 * (SeCO review page, "Referee Report": the Summary, where t of the k chunks
 * are backpropagated and the relayed KV-cache gradient is multiplied by k/t,
 * and the major comments on Algorithm 2 and Section 6.4, where the factor
 * is capped at 2).  Before a selected chunk's backward, its own rows --
 * which then hold only what later chunks relayed into them -- are scaled by
 * the compensation factor; the rows of a chunk that is not selected are
 * zeroed, since nothing propagates from them.
 *   0 <= row_begin <= row_end <= seq_capacity; scale finite.  Every batch
 *   entry and every key/value head of those rows is scaled.  dk_accum,
 *   dv_accum: [B, seq_capacity, Hkv, d] float32, 16-byte aligned.
 * Async on `stream`; INVALID_ARG before any launch on a bad argument.
 */
seqattn_status seqattn_scale_accum_rows(const seqattn_problem* pb, int64_t row_begin,
                                        int64_t row_end, float scale, float* dk_accum,
                                        float* dv_accum, seqattn_stream_t stream);

/*
 * Projection weight gradient of rows [row_begin, row_end): the step after the
 * path (SeCO review page, major comment 1 on Algorithm 2 -- once chunk i's
 * cache gradient is complete, chunk i's graph, here the Q/K/V projections
 * X = H W, is backpropagated).  With the last-to-first chunk order the dK/dV
 * rows of chunk i are final right after its backward, so this runs per chunk.
 *   dw[d_model, n] += sum over batch entries b and rows r of h[b, r]^T g[b, r]
 *   h: [batch, seq_len, d_model] bf16 (the projections' input)
 *   g: [batch, seq_len, n] float32 (dQ with n = Hq d, or dK / dV with
 *      n = Hkv d)
 *   dw: [d_model, n] float32, row-major, accumulated (never overwritten)
 * One tensor-core kernel: g is rounded to bf16 (nearest even) as it is read,
 * the products are summed in float32 and each CTA adds its tile into dw with
 * TMA reduce-adds (atomic per element in L2), so calls that update the same
 * dw may run concurrently on different streams (the order of the fp32
 * additions, and so the last bits of dw, then varies between runs).  Rows of
 * h outside [row_begin, row_end) are read only where they meet a zero of g
 * and must be finite.  Requires batch >= 1, 0 <= row_begin <= row_end <= seq_len,
 * d_model and n positive multiples of 8, and 16-byte aligned pointers.  No
 * workspace.  Async on `stream`; INVALID_ARG before any launch on a bad
 * argument; row_begin == row_end is a no-op.
 */
seqattn_status seqattn_proj_wgrad(int32_t batch, int64_t seq_len, int64_t row_begin,
                                  int64_t row_end, int32_t d_model, int32_t n, const void* h,
                                  const float* g, float* dw, seqattn_stream_t stream);

/* Bytes of workspace seqattn_chunk_bwd needs for a chunk of q_len rows
 * (0 for an invalid problem).  Pure host function. */
size_t seqattn_bwd_workspace_size(const seqattn_problem* pb, int64_t q_len);

/* Synchronise `stream`, then read and clear the device error word.  Returns
 * SEQATTN_ERR_TIMEOUT if a kernel gave up a bounded wait since the last
 * check, SEQATTN_ERR_CUDA if the synchronisation failed, else SEQATTN_OK. */
seqattn_status seqattn_sync_status(seqattn_stream_t stream);

/* Limit, in SM clock cycles, of every bounded device-side wait in the kernels
 * launched after this call from any host thread of the process; cycles <= 0
 * restores the default (2e9 cycles, about one second).  This is the knob that
 * lets a caller (or a test) see the timeout path work without a GPU fault: a
 * launch with a limit far below the microseconds its waits normally take has
 * its waits run out, its CTAs let every copy and MMA already issued complete,
 * release their tensor memory and return, and the next seqattn_sync_status()
 * reports SEQATTN_ERR_TIMEOUT; outputs of such a launch are unspecified.
 * Limits below 65536 cycles also make the forward's waits spin instead of
 * sleeping in the barrier.  Pure host function (takes effect at the next
 * launch). */
void seqattn_set_wait_limit(int64_t cycles);

/* Static description of a status code.  Pure host function. */
const char* seqattn_status_string(seqattn_status s);

/* Human-readable reason for the most recent non-OK status returned on the
 * calling host thread ("" if none).  Pure host function. */
const char* seqattn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SEQATTN_H */
