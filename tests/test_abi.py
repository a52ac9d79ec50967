"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every entry point include/seqattn.h declares, and rejects bad
arguments with a status code before anything is launched."""

import ctypes
import os
import re

import pytest

from long_context_attention_seqattn_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def _declared():
    text = open(os.path.join(ROOT, "include", "seqattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(seqattn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_surface():
    assert _declared() == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.seqattn_status_string(0) == b"ok"
    assert lib.seqattn_status_string(4) == b"device wait timed out"
    assert lib.seqattn_status_string(99) == b"unknown status"


def _pb(**kw):
    base = dict(batch=1, num_q_heads=4, num_kv_heads=2, head_dim=128, seq_capacity=1024, dtype=0)
    base.update(kw)
    return binding.Problem(**base)


def test_workspace_size(lib):
    # bf16: (-L log2 e, Delta) per 64-row query tile -> B * Hq * ceil(q_len / 64) * 128 floats
    pb = _pb()
    assert lib.seqattn_bwd_workspace_size(ctypes.byref(pb), 512) == 4 * 8 * 128 * 4
    assert lib.seqattn_bwd_workspace_size(ctypes.byref(pb), 500) == 4 * 8 * 128 * 4
    assert lib.seqattn_bwd_workspace_size(ctypes.byref(pb), 1) == 4 * 128 * 4
    # float32: Delta [B, Hq, q_len], rounded up to 256 bytes
    pf = _pb(dtype=1)
    assert lib.seqattn_bwd_workspace_size(ctypes.byref(pf), 512) == 4 * 512 * 4
    assert lib.seqattn_bwd_workspace_size(ctypes.byref(pf), 1) == 256
    assert lib.seqattn_bwd_workspace_size(ctypes.byref(_pb(num_q_heads=3)), 512) == 0
    assert lib.seqattn_bwd_workspace_size(None, 512) == 0


P = ctypes.c_void_p(0x10000)      # aligned fake device address: never dereferenced here
MIS = ctypes.c_void_p(0x10004)    # misaligned
NUL = ctypes.c_void_p(0)


def _fwd(lib, pb, q_start=0, q_len=128, prefix=0, scale=0.088, ptrs=None):
    ptrs = ptrs or [P] * 5
    st = lib.seqattn_chunk_fwd(ctypes.byref(pb) if pb is not None else None, q_start, q_len, prefix,
                               scale, *ptrs, NUL)
    return st, lib.seqattn_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(num_q_heads=3), 1),            # Hq % Hkv != 0
    (dict(head_dim=96), 1),              # unsupported head_dim
    (dict(batch=0), 1),
    (dict(dtype=7), 1),
])
def test_problem_validation(lib, kw, code):
    st, msg = _fwd(lib, _pb(**kw))
    assert st == code and msg


def test_chunk_validation(lib):
    pb = _pb()
    assert _fwd(lib, None)[0] == 1
    assert _fwd(lib, pb, q_len=-1)[0] == 1
    assert _fwd(lib, pb, q_start=128, prefix=256)[0] == 1          # prefix beyond start
    assert _fwd(lib, pb, q_start=1024, q_len=128, prefix=0)[0] == 1  # past the cache
    assert _fwd(lib, pb, scale=0.0)[0] == 1
    assert _fwd(lib, pb, scale=float("nan"))[0] == 1
    assert _fwd(lib, pb, ptrs=[P, NUL, P, P, P])[0] == 1
    st, msg = _fwd(lib, pb, ptrs=[P, P, P, MIS, P])
    assert st == 1 and "aligned" in msg


def test_scale_rows_validation(lib):
    """Argument checks of seqattn_scale_accum_rows, all refused before any launch."""
    pb = _pb()
    f = lib.seqattn_scale_accum_rows
    assert f(ctypes.byref(pb), 0, 1025, 2.0, P, P, NUL) == 1          # past seq_capacity
    assert f(ctypes.byref(pb), 10, 9, 2.0, P, P, NUL) == 1            # row_end < row_begin
    assert f(ctypes.byref(pb), -1, 4, 2.0, P, P, NUL) == 1
    assert f(ctypes.byref(pb), 0, 4, float("nan"), P, P, NUL) == 1
    assert f(ctypes.byref(pb), 0, 4, float("inf"), P, P, NUL) == 1
    assert f(ctypes.byref(pb), 0, 4, 2.0, NUL, P, NUL) == 1
    st = f(ctypes.byref(pb), 0, 4, 2.0, P, MIS, NUL)
    assert st == 1 and b"aligned" in lib.seqattn_last_error()
    assert f(None, 0, 4, 2.0, P, P, NUL) == 1


def test_proj_wgrad_validation(lib):
    """Argument checks of seqattn_proj_wgrad, all refused before any launch."""
    f = lib.seqattn_proj_wgrad
    ok_args = dict(batch=1, seq=64, r0=0, r1=32, dm=64, n=128)

    def call(**kw):
        a = dict(ok_args, **kw)
        ptrs = kw.get("ptrs", [P, P, P])
        return f(a["batch"], a["seq"], a["r0"], a["r1"], a["dm"], a["n"], *ptrs, NUL)

    assert call(batch=0) == 1
    assert call(r1=65) == 1                         # past seq_len
    assert call(r0=10, r1=9) == 1
    assert call(dm=60) == 1                         # not a multiple of 8
    assert call(n=4) == 1
    assert call(ptrs=[P, NUL, P]) == 1
    assert call(ptrs=[P, P, MIS]) == 1
    assert b"aligned" in lib.seqattn_last_error()
    assert call(r0=5, r1=5) == 0                    # empty row range: a no-op, nothing launched


def test_empty_chunk_is_ok_without_touching_memory(lib):
    assert _fwd(lib, _pb(), q_len=0, ptrs=[NUL] * 5)[0] == 0
    st = lib.seqattn_chunk_bwd(ctypes.byref(_pb()), 0, 0, 0, 0.1, *([NUL] * 10), 0, NUL)
    assert st == 0


def test_bwd_validation(lib):
    pb = _pb()
    args = [P] * 10
    st = lib.seqattn_chunk_bwd(ctypes.byref(pb), 0, 128, 0, 0.1, *args, 16, NUL)
    assert st == 1 and b"workspace" in lib.seqattn_last_error()
    args[9] = NUL
    assert lib.seqattn_chunk_bwd(ctypes.byref(pb), 0, 128, 0, 0.1, *args, 1 << 20, NUL) == 1


def test_reset_validation(lib):
    assert lib.seqattn_reset_accum(ctypes.byref(_pb()), NUL, P, NUL) == 1
    assert lib.seqattn_reset_accum(None, P, P, NUL) == 1


# ------------------------------------------------------------------ host logic: backward streams

@pytest.mark.parametrize("B,T,Hkv,chunk,bf16,want", [
    (1, 32768, 8, 2048, True, 1),      # grids of about 7 waves: one stream
    (1, 131072, 8, 4096, True, 1),
    (1, 8192, 8, 512, True, 4),        # short grids, short CTAs
    (1, 16384, 8, 128, True, 4),
    (1, 16384, 8, 512, True, 4),
    (1, 16384, 8, 1024, True, 2),
    (1, 16384, 8, 2048, True, 2),      # 576 CTAs on average, under four waves of 152
    (1, 16384, 8, 4096, True, 1),      # 640 on average
    (1, 16384, 8, 16384, True, 1),
    (1, 512, 2, 128, False, 1),        # float32: plain read-modify-writes, one stream
])
def test_backward_stream_rule(B, T, Hkv, chunk, bf16, want):
    assert binding.bwd_streams_for(B, T, Hkv, chunk, bf16, 152) == want


def test_backward_chunks_guards():
    """Overlapping backward calls need the bf16 path's atomic updates, and
    rows become final only in the last-to-first order; both are refused
    before any launch."""
    import torch
    q32 = torch.zeros((1, 256, 2, 64), dtype=torch.float32)
    with pytest.raises(ValueError, match="bf16"):
        binding.backward_chunks(q32, q32, q32, q32, 128, None, bwd_streams=2)
    q16 = torch.zeros((1, 256, 2, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="relay"):
        binding.backward_chunks(q16, q16, q16, q16, 128, None, bwd_streams=1, bwd_order="ascending",
                                on_final=lambda *a: None)


@pytest.mark.parametrize("D", [1, 2, 5, 16])
@pytest.mark.parametrize("streams", [1, 2, 3, 4])
def test_relay_plan_hands_on_only_final_rows(D, streams):
    """SeCO's relay with overlapping backward calls: the rows of chunk i may
    be handed on (weight gradients, host copy) only after every call that adds
    into them -- chunks i..D-1, all issued before or at chunk i's -- has
    completed.  Each such call must be covered by a waited call on its own
    stream at the same or a later position (calls on a stream complete in
    order)."""
    plan = binding.relay_plan(D, streams)
    stream_of = {}
    for n, (i, j, after) in enumerate(plan):
        assert i == D - 1 - n                  # last to first
        assert j == n % streams                # round robin over the streams
        stream_of[n] = j
        assert n in after
        assert len(after) == min(n + 1, streams)
        for m in range(n + 1):
            assert any(stream_of[w] == stream_of[m] and w >= m for w in after), (n, m)
    asc = binding.relay_plan(D, streams, "ascending")
    assert [i for i, _, _ in asc] == list(range(D))
