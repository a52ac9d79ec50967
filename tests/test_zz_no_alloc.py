"""The workspace-free backward (seqattn_chunk_bwd_noalloc) against the
regular backward (seqattn_chunk_bwd), called through the C ABI.

The no-alloc entry point exists for callers that cannot allocate device
memory: their memory belongs to another allocator and the interface they call
through passes only the tensors, so they cannot hand the regular backward its
workspace.  Its scratch is a fixed array inside the library that every call
shares, so this test also calls it twice in a row and checks that the second
call does not depend on what the first left behind.  The file name sorts last
so that a run stopping at the first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from long_context_attention_seqattn_gb300 import binding, build, inputs

pytestmark = pytest.mark.gpu

BF16_REL = 2e-2
BF16_ABS = 5e-2


def _close(name, got, ref):
    got = got.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    mx = np.abs(got - ref).max()
    assert rel <= BF16_REL and mx <= BF16_ABS, f"{name}: rel-L2 {rel:.3e} max-abs {mx:.3e}"


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("dtype,q_start,c,d", [
    ("bf16", 256, 512, 128),
    ("fp32", 256, 512, 128),
    ("bf16", 200, 300, 64),      # chunk off the tile grid, partial last query tile, head_dim 64
])
def test_noalloc_backward_matches_workspace_backward(dtype, q_start, c, d):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    lib = binding.load_library()
    B, T, Hq, Hkv = 1, 768, 4, 2
    dt = inputs.torch_dtype(dtype)
    q, k, v, do = (inputs.draw(n, 77, B, T, h, d, dt).cuda()
                   for n, h in (("q", Hq), ("k", Hkv), ("v", Hkv), ("do", Hq)))
    qc = q[:, q_start:q_start + c].contiguous()
    doc = do[:, q_start:q_start + c].contiguous()
    o = torch.empty_like(qc)
    lse = torch.empty((B, Hq, c), dtype=torch.float32, device="cuda")
    binding.chunk_fwd(qc, k, v, o, lse, q_start)

    # regular backward, with a caller-provided workspace
    dq_ref = torch.empty(qc.shape, dtype=torch.float32, device="cuda")
    dk_ref = torch.zeros(k.shape, dtype=torch.float32, device="cuda")
    dv_ref = torch.zeros(k.shape, dtype=torch.float32, device="cuda")
    binding.chunk_bwd(qc, k, v, o, lse, doc, dq_ref, dk_ref, dv_ref, q_start)
    binding.sync_status()

    pb = binding.problem_for(k, Hq, dt)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dq = torch.full(qc.shape, float("nan"), dtype=torch.float32, device="cuda")
        dk = torch.zeros(k.shape, dtype=torch.float32, device="cuda")
        dv = torch.zeros(k.shape, dtype=torch.float32, device="cuda")
        st = lib.seqattn_chunk_bwd_noalloc(ctypes.byref(pb), q_start, c, q_start, d ** -0.5,
                                           _p(qc), _p(k), _p(v), _p(o), _p(lse), _p(doc), _p(dq),
                                           _p(dk), _p(dv), stream)
        assert st == 0, lib.seqattn_last_error().decode()
        binding.sync_status()
        _close(f"call {call} dQ", dq, dq_ref)
        _close(f"call {call} dK", dk, dk_ref)
        _close(f"call {call} dV", dv, dv_ref)


def test_noalloc_rejects_requests_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = binding.load_library()
    # B * Hq * q_len = 1 * 64 * 32768 > 2^20 rows of scratch: refused before any launch
    pb = binding.Problem(1, 64, 8, 128, 65536, binding.SEQATTN_BF16)
    fake = ctypes.c_void_p(0x10000)
    st = lib.seqattn_chunk_bwd_noalloc(ctypes.byref(pb), 0, 32768, 0, 0.088, *([fake] * 9),
                                       ctypes.c_void_p(0))
    assert st == binding.SEQATTN_ERR_INVALID_ARG
    assert b"scratch" in lib.seqattn_last_error()
