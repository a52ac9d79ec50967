"""The workspace-free backward (seqattn_chunk_bwd_noalloc) against the
regular backward (seqattn_chunk_bwd), called through the C ABI.

The no-alloc entry point exists for callers that cannot allocate device
memory: their memory belongs to another allocator and the interface they call
through passes only the tensors, so they cannot hand the regular backward its
workspace.  Its scratch is a fixed array inside the library that every call
shares, so this test calls it twice in a row, each time right after a call
for a longer chunk with other inputs has filled more of that array, and
checks that the result does not depend on what was left behind.  The file name sorts last
so that a run stopping at the first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from long_context_attention_seqattn_gb300 import binding, build, inputs

pytestmark = pytest.mark.gpu

# Both backwards run the same kernels on the same inputs: they differ only in
# the order of the fp32 atomic additions into dq, so the bar is tight.
SAME_KERNELS_REL = 1e-5


def _close(name, got, ref):
    got = got.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= SAME_KERNELS_REL, f"{name}: rel-L2 {rel:.3e}"


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

    # a different, longer chunk (the whole sequence, other dO) whose row
    # statistics fill more of the shared scratch than the checked call needs
    o_f = torch.empty_like(q)
    lse_f = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
    binding.chunk_fwd(q, k, v, o_f, lse_f, 0)
    do_f = inputs.draw("do", 78, B, T, Hq, d, dt).cuda()
    filler = [torch.empty(q.shape, dtype=torch.float32, device="cuda"),
              torch.zeros(k.shape, dtype=torch.float32, device="cuda"),
              torch.zeros(k.shape, dtype=torch.float32, device="cuda")]

    pb = binding.problem_for(k, Hq, dt)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        # the scratch keeps what the previous call left; the checked call must
        # rewrite every statistic it reads
        st = lib.seqattn_chunk_bwd_noalloc(ctypes.byref(pb), 0, T, 0, d ** -0.5, _p(q), _p(k), _p(v),
                                           _p(o_f), _p(lse_f), _p(do_f), *(_p(t) for t in filler), stream)
        assert st == 0, lib.seqattn_last_error().decode()
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
