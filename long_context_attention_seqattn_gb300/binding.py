"""ctypes binding of libseqattn (include/seqattn.h).

Every step of the computation runs in the library's CUDA kernels.  The call
wrappers turn torch tensors into device pointers and sizes, pass the torch
CUDA stream, and raise ``SeqattnError`` on a non-OK status.  The layer drivers
below them (``forward_chunks``, ``backward_chunks``, ``layer_forward_backward``,
``LayerGraph``, ``HostLayerPass``) are host logic only: they order the chunk
calls over CUDA streams and events, and do no arithmetic.  If the library has
not been built, the first call raises; there is no other code path.
"""

import ctypes
import os

import torch

from .build import LIB_PATH

SEQATTN_OK = 0
SEQATTN_ERR_INVALID_ARG = 1
SEQATTN_ERR_UNSUPPORTED = 2
SEQATTN_ERR_CUDA = 3
SEQATTN_ERR_TIMEOUT = 4

SEQATTN_BF16 = 0
SEQATTN_FP32 = 1

EXPORTED = (
    "seqattn_chunk_fwd",
    "seqattn_chunk_bwd",
    "seqattn_chunk_bwd_noalloc",
    "seqattn_reset_accum",
    "seqattn_scale_accum_rows",
    "seqattn_proj_wgrad",
    "seqattn_bwd_workspace_size",
    "seqattn_sync_status",
    "seqattn_set_wait_limit",
    "seqattn_status_string",
    "seqattn_last_error",
)


class Problem(ctypes.Structure):
    """Mirror of ``seqattn_problem``."""
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("seq_capacity", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
    ]


class SeqattnError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"seqattn status {status}: {message}")
        self.status = status


_lib = None


def load_library(path=LIB_PATH):
    """Load libseqattn.so (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run long_context_attention_seqattn_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(Problem)
    vp, i64, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.seqattn_chunk_fwd.argtypes = [P, i64, i64, i64, f32, vp, vp, vp, vp, vp, vp]
    lib.seqattn_chunk_fwd.restype = ctypes.c_int
    lib.seqattn_chunk_bwd.argtypes = [P, i64, i64, i64, f32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      vp, sz, vp]
    lib.seqattn_chunk_bwd.restype = ctypes.c_int
    lib.seqattn_chunk_bwd_noalloc.argtypes = [P, i64, i64, i64, f32, vp, vp, vp, vp, vp, vp, vp,
                                              vp, vp, vp]
    lib.seqattn_chunk_bwd_noalloc.restype = ctypes.c_int
    lib.seqattn_reset_accum.argtypes = [P, vp, vp, vp]
    lib.seqattn_reset_accum.restype = ctypes.c_int
    lib.seqattn_scale_accum_rows.argtypes = [P, i64, i64, f32, vp, vp, vp]
    lib.seqattn_scale_accum_rows.restype = ctypes.c_int
    i32 = ctypes.c_int32
    lib.seqattn_proj_wgrad.argtypes = [i32, i64, i64, i64, i32, i32, vp, vp, vp, vp]
    lib.seqattn_proj_wgrad.restype = ctypes.c_int
    lib.seqattn_bwd_workspace_size.argtypes = [P, i64]
    lib.seqattn_bwd_workspace_size.restype = sz
    lib.seqattn_sync_status.argtypes = [vp]
    lib.seqattn_sync_status.restype = ctypes.c_int
    lib.seqattn_set_wait_limit.argtypes = [i64]
    lib.seqattn_set_wait_limit.restype = None
    lib.seqattn_status_string.argtypes = [ctypes.c_int]
    lib.seqattn_status_string.restype = ctypes.c_char_p
    lib.seqattn_last_error.argtypes = []
    lib.seqattn_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status):
    if status != SEQATTN_OK:
        lib = load_library()
        raise SeqattnError(status, lib.seqattn_last_error().decode())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dtype_code(dt):
    if dt == torch.bfloat16:
        return SEQATTN_BF16
    if dt == torch.float32:
        return SEQATTN_FP32
    raise TypeError(f"unsupported element type {dt}")


def problem_for(k, num_q_heads, dtype=None):
    """seqattn_problem for caches ``k`` of shape [B, T, Hkv, d]."""
    B, T, Hkv, d = k.shape
    return Problem(B, num_q_heads, Hkv, d, T, _dtype_code(dtype or k.dtype))


def _need(t, name, dtype, shape=None):
    if not t.is_cuda or not t.is_contiguous() or t.dtype != dtype:
        raise ValueError(f"{name} must be a contiguous CUDA tensor of {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def chunk_fwd(q, k, v, o, lse, q_start, prefix_len=None, scale=None, stream=None):
    """Forward of the chunk whose queries ``q`` [B, c, Hq, d] sit at absolute
    rows [q_start, q_start + c) of the caches ``k``, ``v`` [B, T, Hkv, d].
    Writes ``o`` [B, c, Hq, d] and ``lse`` [B, Hq, c] (float32)."""
    B, c, Hq, d = q.shape
    prefix_len = q_start if prefix_len is None else prefix_len
    scale = d ** -0.5 if scale is None else scale
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _need(t, name, q.dtype)
    _need(lse, "lse", torch.float32, (B, Hq, c))
    pb = problem_for(k, Hq, q.dtype)
    _check(load_library().seqattn_chunk_fwd(ctypes.byref(pb), q_start, c, prefix_len, scale,
                                            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                            _stream(stream)))


def bwd_workspace_size(k, num_q_heads, q_len, dtype=None):
    pb = problem_for(k, num_q_heads, dtype)
    return int(load_library().seqattn_bwd_workspace_size(ctypes.byref(pb), q_len))


def chunk_bwd(q, k, v, o, lse, d_o, dq, dk_accum, dv_accum, q_start, prefix_len=None,
              scale=None, workspace=None, stream=None):
    """Backward of one chunk: overwrites ``dq`` (float32, shape of q) and adds
    into ``dk_accum``/``dv_accum`` (float32, shape of k).  ``workspace`` is a
    uint8 CUDA tensor of at least ``bwd_workspace_size`` bytes (allocated
    here when omitted)."""
    B, c, Hq, d = q.shape
    prefix_len = q_start if prefix_len is None else prefix_len
    scale = d ** -0.5 if scale is None else scale
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("d_o", d_o)):
        _need(t, name, q.dtype)
    _need(lse, "lse", torch.float32, (B, Hq, c))
    _need(dq, "dq", torch.float32, q.shape)
    _need(dk_accum, "dk_accum", torch.float32, k.shape)
    _need(dv_accum, "dv_accum", torch.float32, k.shape)
    pb = problem_for(k, Hq, q.dtype)
    lib = load_library()
    need = int(lib.seqattn_bwd_workspace_size(ctypes.byref(pb), c))
    temp = workspace is None
    if temp:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(lib.seqattn_chunk_bwd(ctypes.byref(pb), q_start, c, prefix_len, scale, _ptr(q), _ptr(k),
                                 _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o), _ptr(dq), _ptr(dk_accum),
                                 _ptr(dv_accum), _ptr(workspace), workspace.numel(),
                                 _stream(stream)))
    if temp and stream is not None:
        # the temporary was allocated on the current stream but is read on
        # `stream`: keep the caching allocator from reusing it before then
        workspace.record_stream(stream)


def reset_accum(dk_accum, dv_accum, num_q_heads=None, stream=None):
    """Zero the float32 running sums (shape [B, T, Hkv, d])."""
    _need(dk_accum, "dk_accum", torch.float32)
    _need(dv_accum, "dv_accum", torch.float32, dk_accum.shape)
    Hkv = dk_accum.shape[2]
    pb = problem_for(dk_accum, num_q_heads or Hkv, torch.float32)
    _check(load_library().seqattn_reset_accum(ctypes.byref(pb), _ptr(dk_accum), _ptr(dv_accum),
                                              _stream(stream)))


def scale_accum_rows(dk_accum, dv_accum, row_begin, row_end, scale, stream=None):
    """Multiply rows [row_begin, row_end) of two float32 [B, T, H, d] arrays
    (the running sums, or any such pair; the same tensor may be passed twice)
    by ``scale`` (0 stores zeros)."""
    _need(dk_accum, "dk_accum", torch.float32)
    _need(dv_accum, "dv_accum", torch.float32, dk_accum.shape)
    B, T, H, d = dk_accum.shape
    pb = Problem(B, H, H, d, T, SEQATTN_FP32)
    _check(load_library().seqattn_scale_accum_rows(ctypes.byref(pb), row_begin, row_end, scale,
                                                   _ptr(dk_accum), _ptr(dv_accum), _stream(stream)))


def proj_wgrad(h, g, dw, row_begin, row_end, stream=None):
    """dw [d_model, n] += sum over batch entries of h[b, r0:r1]^T g[b, r0:r1],
    with h [B, T, d_model] bf16 (hidden states) and g [B, T, ...] float32 (dQ,
    dK or dV; trailing dims flattened to n)."""
    B, T, dm = h.shape
    n = g[0, 0].numel()
    _need(h, "h", torch.bfloat16)
    _need(g, "g", torch.float32)
    _need(dw, "dw", torch.float32, (dm, n))
    if tuple(g.shape[:2]) != (B, T):
        raise ValueError(f"g has leading shape {tuple(g.shape[:2])}, expected {(B, T)}")
    _check(load_library().seqattn_proj_wgrad(B, T, row_begin, row_end, dm, n, _ptr(h), _ptr(g), _ptr(dw),
                                             _stream(stream)))


def sync_status(stream=None):
    """Synchronise the stream and raise if a kernel gave up a bounded wait."""
    _check(load_library().seqattn_sync_status(_stream(stream)))


def set_wait_limit(cycles):
    """Limit (SM cycles) of the kernels' bounded waits for later launches;
    ``cycles <= 0`` restores the default of about one second."""
    load_library().seqattn_set_wait_limit(int(cycles))


def status_string(code):
    return load_library().seqattn_status_string(code).decode()


# ------------------------------------------------------------------ layer driver

class LayerBuffers:
    """Device buffers of one layer pass: outputs and accumulators, allocated
    once and reused across passes."""

    def __init__(self, q, k, chunk):
        B, T, Hq, d = q.shape
        dev = q.device
        self.o = torch.empty_like(q)
        self.dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
        self.dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
        self.dv = torch.empty(k.shape, dtype=torch.float32, device=dev)
        # per-chunk LSE slices must be contiguous [B, Hq, c]: keep one buffer per chunk
        self.chunk = chunk
        self.starts = list(range(0, T, chunk))
        self.lse_chunks = [torch.empty((B, Hq, min(chunk, T - s)), dtype=torch.float32, device=dev)
                           for s in self.starts]
        self.workspace = torch.empty(max(256, bwd_workspace_size(k, Hq, chunk, q.dtype)),
                                     dtype=torch.uint8, device=dev)
        self.workspaces = [self.workspace]

    def workspace_for(self, j):
        """Backward workspace of stream ``j`` (backward calls that may run at
        the same time need one each)."""
        while len(self.workspaces) <= j:
            self.workspaces.append(torch.empty_like(self.workspace))
        return self.workspaces[j]


def _rows(t, s, e):
    """Rows [s, e) of a [B, T, H, d] tensor as a contiguous chunk tensor."""
    v = t[:, s:e]
    return v if v.is_contiguous() else v.contiguous()


def _nvtx(name):
    """An NVTX range around one chunk call (host side; it names the call in a
    profiler's timeline and costs nothing measurable when none is attached)."""
    return torch.cuda.nvtx.range(name)


def _copy_rows(dst, src, s, e):
    """Asynchronous copy of rows [s, e) of [B, T, ...] tensors between host and
    device, one contiguous block per batch entry."""
    for b in range(dst.shape[0]):
        dst[b, s:e].copy_(src[b, s:e], non_blocking=True)


_side_streams = {}


def side_streams(device, n):
    """``n`` long-lived side streams of ``device`` (created once)."""
    key = torch.device(device).index if torch.device(device).index is not None else torch.cuda.current_device()
    have = _side_streams.setdefault(key, [])
    while len(have) < n:
        have.append(torch.cuda.Stream(device=key))
    return have[:n]


def auto_fwd_streams(q, chunk):
    """Streams for the chunk forwards: at least two (one chunk's last wave
    overlaps the next chunk's grid), and enough that the forward grids of the
    chunks in flight together cover the SMs when a chunk's own grid is small
    (128-row query tiles x heads x batch CTAs per chunk); at most eight."""
    B, T, Hq, d = q.shape
    ctas = max(1, -(-min(chunk, T) // 128)) * Hq * B
    sms = torch.cuda.get_device_properties(q.device).multi_processor_count
    return max(2, min(8, -(-sms // ctas)))


def forward_chunks(q, k, v, chunk, bufs, scale=None, stream=None, fwd_streams=None):
    """Forward every chunk into ``bufs``.  The chunk forwards depend only on
    the caches (StreamBP review page, Property 3.1), so chunk i runs on stream
    i % fwd_streams (``stream`` and side streams forked from it): the last,
    partly filled wave of one chunk's grid overlaps the next chunk's, and
    small chunks run side by side.  ``fwd_streams`` defaults to
    ``auto_fwd_streams``.  All streams are joined back into ``stream`` before
    returning."""
    B, T, Hq, d = q.shape
    if fwd_streams is None:
        fwd_streams = auto_fwd_streams(q, chunk)
    main = stream if stream is not None else torch.cuda.current_stream()
    sides = side_streams(q.device, fwd_streams - 1)
    for sd in sides:
        sd.wait_stream(main)
    for i, s in enumerate(bufs.starts):
        e = min(s + chunk, T)
        st = main if i % fwd_streams == 0 else sides[i % fwd_streams - 1]
        # the row gathers of a batched chunk (B > 1) and their temporaries
        # belong to the chunk's own stream
        with torch.cuda.stream(st), _nvtx(f"seqattn fwd chunk {i} rows {s}:{e}"):
            o_c = bufs.o[:, s:e]
            if o_c.is_contiguous():
                chunk_fwd(_rows(q, s, e), k, v, o_c, bufs.lse_chunks[i], s, s, scale, st)
            else:
                tmp = torch.empty_like(o_c.contiguous())
                chunk_fwd(_rows(q, s, e), k, v, tmp, bufs.lse_chunks[i], s, s, scale, st)
                o_c.copy_(tmp)
    for sd in sides:
        main.wait_stream(sd)


def auto_bwd_streams(q, k, chunk):
    """Streams for the chunk backwards.  bf16 backward calls add into the
    accumulators atomically and may overlap, which pays when the chunk grids
    (128-key tiles of the prefix x key/value heads x batch CTAs) are short:
    one chunk's last wave, its statistics pre-pass and the launch boundaries
    then overlap the next chunk's work.  Measured on a 16384-token layer
    (backward TFLOP/s, 1 / 2 / 4 streams): chunk 128: 484 / 567 / 606, 512:
    878 / 974 / 1005, 2048: 1128 / 1160, 4096: 1238 / 1240; on a 32768-token
    layer at chunk 2048 (grids of 7 waves on average) one stream is faster,
    1171 against 1129.  So: one stream when the average chunk grid fills four
    waves of the SMs; otherwise four streams for chunks of at most 512 rows
    (a CTA runs only G ceil(c/64) short steps) and two above.  float32 calls
    update the accumulators with plain read-modify-writes and always take
    one stream."""
    B, T, Hq, d = q.shape
    if q.dtype != torch.bfloat16:
        return 1
    sms = torch.cuda.get_device_properties(q.device).multi_processor_count
    return bwd_streams_for(B, T, k.shape[2], chunk, True, sms)


def bwd_streams_for(batch, seq_len, num_kv_heads, chunk, bf16, sms):
    """The rule of ``auto_bwd_streams`` on plain numbers (host logic only)."""
    if not bf16:
        return 1
    starts = range(0, seq_len, chunk)
    tiles = sum(-(-min(s + chunk, seq_len) // 128) for s in starts) / len(starts)
    if tiles * num_kv_heads * batch >= 4 * sms:
        return 1
    return 4 if chunk <= 512 else 2


def relay_plan(num_chunks, bwd_streams, bwd_order="descending"):
    """Host plan of ``backward_chunks``: for the n-th call in ``bwd_order``,
    ``(i, j, after)`` -- chunk i runs on stream j, and its rows are final once
    the calls at the order positions in ``after`` have completed (the latest
    call on every stream so far, chunk i's own included).  Calls on one
    stream complete in order, so every earlier call is covered."""
    order = list(range(num_chunks))
    if bwd_order == "descending":
        order = order[::-1]
    latest = [None] * bwd_streams
    plan = []
    for n, i in enumerate(order):
        j = n % bwd_streams
        latest[j] = n
        plan.append((i, j, [x for x in latest if x is not None]))
    return plan


def backward_chunks(q, k, v, d_o, chunk, bufs, scale=None, stream=None, bwd_streams=None,
                    bwd_order="descending", on_final=None, before_chunk=None):
    """Backward every chunk of ``bufs`` (after ``forward_chunks``): dQ rows
    overwritten, dK/dV added into the running sums.  The k-th chunk in
    ``bwd_order`` runs on stream k % bwd_streams (``stream`` and side streams
    forked from it), each stream with its own workspace; ``bwd_streams``
    defaults to ``auto_bwd_streams``.

    ``on_final(i, s, e, events)`` (descending order only) is called after
    chunk i's backward is enqueued: once every CUDA event in ``events`` has
    completed, dQ rows [s, e) and the dK/dV rows [s, e) are final -- every
    chunk from i on has added its share (SeCO's relay).
    ``before_chunk(i, st)`` is called before chunk i's backward is enqueued
    on stream ``st`` (to make it wait for that chunk's inputs).  All streams
    are joined back into ``stream`` before returning."""
    B, T, Hq, d = q.shape
    if bwd_streams is None:
        bwd_streams = auto_bwd_streams(q, k, chunk)
    if bwd_streams > 1 and q.dtype != torch.bfloat16:
        raise ValueError("overlapping backward calls need the bf16 path (atomic accumulator updates)")
    if on_final is not None and bwd_order != "descending":
        raise ValueError("rows become final only in the last-to-first relay order")
    main = stream if stream is not None else torch.cuda.current_stream()
    sides = side_streams(q.device, bwd_streams - 1)
    for sd in sides:
        sd.wait_stream(main)
    need_events = on_final is not None or bwd_streams > 1
    events = []                             # event after the call at each order position
    for i, j, after in relay_plan(len(bufs.starts), bwd_streams, bwd_order):
        s = bufs.starts[i]
        e = min(s + chunk, T)
        st = main if j == 0 else sides[j - 1]
        if before_chunk is not None:
            before_chunk(i, st)
        with torch.cuda.stream(st), _nvtx(f"seqattn bwd chunk {i} rows {s}:{e}"):   # as in forward_chunks
            dq_c = bufs.dq[:, s:e]
            tgt = dq_c if dq_c.is_contiguous() else torch.empty_like(dq_c.contiguous())
            chunk_bwd(_rows(q, s, e), k, v, _rows(bufs.o, s, e), bufs.lse_chunks[i], _rows(d_o, s, e),
                      tgt, bufs.dk, bufs.dv, s, s, scale, bufs.workspace_for(j), st)
            if tgt is not dq_c:
                dq_c.copy_(tgt)
        if need_events:
            ev = torch.cuda.Event()
            ev.record(st)
            events.append(ev)
        if on_final is not None:
            on_final(i, s, e, [events[m] for m in after])
    for sd in sides:
        main.wait_stream(sd)


def layer_forward_backward(q, k, v, d_o, chunk, scale=None, bufs=None, stream=None,
                           bwd_order="descending", fwd_streams=None, wgrad=None, bwd_streams=None):
    """One pass of the chunked layer: reset the running sums, forward chunks
    0..D-1 (over ``fwd_streams`` streams, see ``forward_chunks``), backward
    chunks D-1..0 (SeCO's last-to-first relay order; over ``bwd_streams``
    streams, see ``backward_chunks``).  Returns the LayerBuffers holding O,
    per-chunk LSE, dQ, dK, dV.

    ``wgrad = (h, dw_q, dw_k, dw_v)`` also runs the projections' weight
    gradients in the relay: right after chunk i's backward, its dQ rows and
    its dK/dV rows are final (every later chunk has run), so
    dw_x += H^(i)T dX^(i) is added for each of the three (h: [B, T, d_model]
    bf16; dw_q: [d_model, Hq d], dw_k, dw_v: [d_model, Hkv d], float32,
    accumulated).  Needs the descending order.  They run on six relay
    streams (two per projection, alternate chunks) that wait until each
    chunk's rows are final."""
    B, T, Hq, d = q.shape
    if bufs is None:
        bufs = LayerBuffers(q, k, chunk)
    if wgrad is not None and bwd_order != "descending":
        raise ValueError("the projection gradients run in the last-to-first relay order")
    reset_accum(bufs.dk, bufs.dv, Hq, stream)
    forward_chunks(q, k, v, chunk, bufs, scale, stream, fwd_streams)
    if bwd_streams is None:
        bwd_streams = auto_bwd_streams(q, k, chunk)
    main = stream if stream is not None else torch.cuda.current_stream()
    on_final = None
    relays = []
    if wgrad is not None:
        # relay streams after the backward's side streams: two per projection,
        # taken by alternate chunks, so the three weight gradients of a chunk
        # run side by side, beside those of the previous chunk and beside the
        # backwards of the earlier chunks (a dW's reduce-adds are atomic per
        # element, so two chunks may update it at once)
        relays = side_streams(q.device, bwd_streams + 5)[bwd_streams - 1:]
        for r in relays:
            r.wait_stream(main)
        seen = [0]

        def on_final(i, s, e, events):
            h, dw_q, dw_k, dw_v = wgrad
            par = seen[0] % 2
            seen[0] += 1
            for x, (g, dw) in enumerate(((bufs.dq, dw_q), (bufs.dk, dw_k), (bufs.dv, dw_v))):
                r = relays[2 * x + par]
                for ev in events:
                    r.wait_event(ev)
                proj_wgrad(h, g, dw, s, e, r)

    backward_chunks(q, k, v, d_o, chunk, bufs, scale, main, bwd_streams, bwd_order, on_final)
    for r in relays:
        main.wait_stream(r)
    return bufs


def spaco_factor(num_chunks, num_selected, cap=2.0):
    """SpaCO's compensation factor for t = num_selected of k = num_chunks
    chunks: k / t, capped (at 2 in the deployed method)."""
    return min(num_chunks / num_selected, cap)


def spaco_layer_forward_backward(q, k, v, d_o, chunk, selected, factor=None, scale=None, bufs=None,
                                 stream=None):
    """One SpaCO pass of the chunked layer: reset the running sums, forward
    every chunk (the inference pass that builds the caches), then visit the
    chunks last to first.  A selected chunk scales the cache gradient relayed
    into its own rows by ``factor`` and runs its backward; a chunk that is not
    selected has its rows zeroed and no backward.  ``selected`` holds the
    sampled chunk indices (drawn by the caller); ``factor`` defaults to
    ``spaco_factor(D, len(selected))``.  dQ rows of unselected chunks are
    zero.  Returns the LayerBuffers."""
    B, T, Hq, d = q.shape
    if bufs is None:
        bufs = LayerBuffers(q, k, chunk)
    chosen = set(int(i) for i in selected)
    n_chunks = len(bufs.starts)
    if not chosen or min(chosen) < 0 or max(chosen) >= n_chunks:
        raise ValueError(f"selected chunk indices must lie in [0, {n_chunks})")
    if factor is None:
        factor = spaco_factor(n_chunks, len(chosen))
    main = stream if stream is not None else torch.cuda.current_stream()
    reset_accum(bufs.dk, bufs.dv, Hq, main)
    forward_chunks(q, k, v, chunk, bufs, scale, main)
    # one stream: each selected chunk's scaling must follow every later
    # chunk's additions into its rows
    with torch.cuda.stream(main):
        for i, s in reversed(list(enumerate(bufs.starts))):
            e = min(s + chunk, T)
            dq_c = bufs.dq[:, s:e]
            if i not in chosen:
                scale_accum_rows(bufs.dk, bufs.dv, s, e, 0.0, main)
                scale_accum_rows(bufs.dq, bufs.dq, s, e, 0.0, main)   # no dQ for this chunk
                continue
            scale_accum_rows(bufs.dk, bufs.dv, s, e, factor, main)
            tgt = dq_c if dq_c.is_contiguous() else torch.empty_like(dq_c.contiguous())
            chunk_bwd(_rows(q, s, e), k, v, _rows(bufs.o, s, e), bufs.lse_chunks[i], _rows(d_o, s, e),
                      tgt, bufs.dk, bufs.dv, s, s, scale, bufs.workspace, main)
            if tgt is not dq_c:
                dq_c.copy_(tgt)
    return bufs


def gather_lse(bufs):
    """Concatenate the per-chunk LSE buffers into [B, Hq, T]."""
    return torch.cat(bufs.lse_chunks, dim=2)


class LayerGraph:
    """One layer pass (reset, D chunk forwards, D chunk backwards) captured
    into a CUDA graph, so that small chunks are not bound by host launch
    overhead.  ``replay()`` re-runs it on the same input and output buffers
    (update the inputs in place between replays)."""

    def __init__(self, q, k, v, d_o, chunk, scale=None, bufs=None, bwd_order="descending"):
        self.args = (q, k, v, d_o, chunk)
        self.bufs = bufs if bufs is not None else LayerBuffers(q, k, chunk)
        # one eager pass first: loads the kernels and looks up the per-device
        # error word outside the capture
        layer_forward_backward(q, k, v, d_o, chunk, scale, self.bufs, bwd_order=bwd_order)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(self.graph, stream=side):
                layer_forward_backward(q, k, v, d_o, chunk, scale, self.bufs, bwd_order=bwd_order)
        torch.cuda.current_stream().wait_stream(side)

    def replay(self):
        self.graph.replay()
        return self.bufs


class HostLayerPass:
    """A layer pass whose inputs start and whose outputs end in pinned host
    memory, with the transfers overlapped with the chunk calls.

    Forward chunk i needs only query rows of chunk i and key/value rows
    [0, end of chunk i), so inputs are uploaded chunk by chunk ahead of the
    forward calls.  With the last-to-first backward order (the relay order
    of SeCO's Algorithm 2), the dK/dV rows of chunk j receive their last
    contribution from chunk j's backward, so every output chunk (O, LSE, dQ,
    dK, dV rows) is copied back as soon as it is final, while later chunks
    still compute.  Two side streams carry the copies; CUDA events order
    them against the compute stream."""

    def __init__(self, h_q, h_k, h_v, h_do, chunk, device="cuda"):
        B, T, Hq, d = h_q.shape
        self.h_in = (h_q, h_k, h_v, h_do)
        self.chunk = chunk
        self.d_in = tuple(torch.empty(x.shape, dtype=x.dtype, device=device) for x in self.h_in)
        self.bufs = LayerBuffers(self.d_in[0], self.d_in[1], chunk)
        self.h_o = torch.empty(h_q.shape, dtype=h_q.dtype, pin_memory=True)
        self.h_lse = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in self.bufs.lse_chunks]
        self.h_dq = torch.empty(h_q.shape, dtype=torch.float32, pin_memory=True)
        self.h_dk = torch.empty(h_k.shape, dtype=torch.float32, pin_memory=True)
        self.h_dv = torch.empty(h_k.shape, dtype=torch.float32, pin_memory=True)
        self.up = torch.cuda.Stream()
        self.down = torch.cuda.Stream()
        self.bwd_streams = auto_bwd_streams(self.d_in[0], self.d_in[1], chunk)

    def bytes_moved(self):
        h2d = sum(x.numel() * x.element_size() for x in self.h_in)
        d2h = sum(x.numel() * x.element_size() for x in (self.h_o, self.h_dq, self.h_dk, self.h_dv))
        d2h += sum(x.numel() * x.element_size() for x in self.h_lse)
        return h2d, d2h

    def run(self):
        """Enqueue one pass on the current stream (copies on side streams).
        Returns the host output tensors (valid after the stream syncs)."""
        main = torch.cuda.current_stream()
        q, k, v, do = self.d_in
        h_q, h_k, h_v, h_do = self.h_in
        b = self.bufs
        T, c = q.shape[1], self.chunk
        starts = b.starts
        self.up.wait_stream(main)
        self.down.wait_stream(main)
        ev_in = []
        with torch.cuda.stream(self.up):
            for s in starts:
                e = min(s + c, T)
                for dst, src in ((q, h_q), (k, h_k), (v, h_v)):
                    _copy_rows(dst, src, s, e)
                ev = torch.cuda.Event()
                ev.record(self.up)
                ev_in.append(ev)
            # dO in the backward's (last-to-first) order, so that the first
            # backward call waits only for its own chunk
            ev_do = [None] * len(starts)
            for i in range(len(starts) - 1, -1, -1):
                s = starts[i]
                e = min(s + c, T)
                _copy_rows(do, h_do, s, e)
                ev = torch.cuda.Event()
                ev.record(self.up)
                ev_do[i] = ev
        reset_accum(b.dk, b.dv, q.shape[2], main)
        # chunk forwards alternate over two compute streams (see forward_chunks)
        side = side_streams(q.device, 1)[0]
        side.wait_stream(main)
        for i, s in enumerate(starts):
            e = min(s + c, T)
            st = main if i % 2 == 0 else side
            st.wait_event(ev_in[i])
            with torch.cuda.stream(st):      # row gathers of a batched chunk on its own stream
                o_c = b.o[:, s:e]
                tgt = o_c if o_c.is_contiguous() else torch.empty_like(o_c.contiguous())
                chunk_fwd(_rows(q, s, e), k, v, tgt, b.lse_chunks[i], s, s, None, st)
                if tgt is not o_c:
                    o_c.copy_(tgt)
            ev = torch.cuda.Event()
            ev.record(st)
            self.down.wait_event(ev)
            with torch.cuda.stream(self.down):
                _copy_rows(self.h_o, b.o, s, e)
                self.h_lse[i].copy_(b.lse_chunks[i], non_blocking=True)
        main.wait_stream(side)

        def before_chunk(i, st):
            st.wait_event(ev_do[i])

        def on_final(i, s, e, events):
            # rows of chunk i are final: later chunks and this one were the
            # only ones touching them
            for ev in events:
                self.down.wait_event(ev)
            with torch.cuda.stream(self.down):
                for dst, src in ((self.h_dq, b.dq), (self.h_dk, b.dk), (self.h_dv, b.dv)):
                    _copy_rows(dst, src, s, e)

        backward_chunks(q, k, v, do, c, b, None, main, self.bwd_streams, "descending", on_final, before_chunk)
        main.wait_stream(self.down)
        main.wait_stream(self.up)
        return self.h_o, self.h_lse, self.h_dq, self.h_dk, self.h_dv
