"""The bounded device waits, made to run out on purpose.

Every wait inside the tensor-core kernels gives up after a limit (about one
second by default), sets the device error word, lets the copies and MMAs it
already issued complete, frees its tensor memory and returns; the host reads
the word with seqattn_sync_status(), which reports SEQATTN_ERR_TIMEOUT once
and clears it.  A wait limit of one cycle (seqattn_set_wait_limit) makes every
wait that is not already complete at its first poll run out, so a normal,
valid call (a chunk forward and backward, a projection weight gradient)
exercises that path without any fault.  Afterwards the
default limit is restored and the same calls must succeed and match the
oracle again.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from long_context_attention_seqattn_gb300 import binding, build, inputs

pytestmark = pytest.mark.gpu

BF16_REL = 2e-2
BF16_ABS = 5e-2


def _close(name, got, ref):
    got = got.detach().to("cpu", torch.float64).numpy()
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    mx = float(np.abs(got - ref).max())
    assert rel <= BF16_REL and mx <= BF16_ABS, f"{name}: rel-L2 {rel:.3e} max-abs {mx:.3e}"


@pytest.mark.parametrize("d,B,T,Hq,Hkv", [
    (128, 1, 512, 4, 2),
    (64, 1, 512, 4, 2),
    (128, 2, 2304, 32, 8),   # more backward CTAs than SMs, batch 2
])
def test_waits_run_out_report_timeout_then_recover(d, B, T, Hq, Hkv):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    lib = binding.load_library()
    qs, c = T - 256, 256
    cpu = [inputs.draw(n, 17, B, T, h, d, torch.bfloat16) for n, h in
           (("q", Hq), ("k", Hkv), ("v", Hkv), ("do", Hq))]
    q, k, v, do = (x.cuda() for x in cpu)
    qc, doc = q[:, qs:qs + c].contiguous(), do[:, qs:qs + c].contiguous()
    o = torch.zeros((B, c, Hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, Hq, c), device="cuda")
    dq = torch.zeros((B, c, Hq, d), device="cuda")
    dk = torch.zeros(k.shape, device="cuda")
    dv = torch.zeros(k.shape, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.seqattn_sync_status(stream) == binding.SEQATTN_OK

    try:
        binding.set_wait_limit(1)
        # forward: the launch is accepted, its waits run out on the device
        binding.chunk_fwd(qc, k, v, o, lse, qs)
        assert lib.seqattn_sync_status(stream) == binding.SEQATTN_ERR_TIMEOUT
        assert b"bounded wait" in lib.seqattn_last_error()
        assert lib.seqattn_sync_status(stream) == binding.SEQATTN_OK      # the word was cleared
        # backward (statistics pre-pass, then the tensor-core kernel)
        binding.chunk_bwd(qc, k, v, o, lse, doc, dq, dk, dv, qs)
        assert lib.seqattn_sync_status(stream) == binding.SEQATTN_ERR_TIMEOUT
        assert lib.seqattn_sync_status(stream) == binding.SEQATTN_OK
    finally:
        binding.set_wait_limit(0)

    # default limit again: the same calls complete and match the oracle
    dk.zero_()
    dv.zero_()
    binding.chunk_fwd(qc, k, v, o, lse, qs)
    binding.chunk_bwd(qc, k, v, o, lse, doc, dq, dk, dv, qs)
    assert lib.seqattn_sync_status(stream) == binding.SEQATTN_OK
    qn, kn, vn, don = (x.to(torch.float64).numpy() for x in cpu)
    scale = d ** -0.5
    ro, rl = oracle.chunk_forward(qn[:, qs:qs + c], kn, vn, qs, qs, scale)
    rdk, rdv = np.zeros(kn.shape), np.zeros(vn.shape)
    rdq = oracle.chunk_backward(qn[:, qs:qs + c], kn, vn, ro, rl, don[:, qs:qs + c], qs, qs, scale,
                                rdk, rdv)
    for name, a, r in (("O", o, ro), ("LSE", lse, rl), ("dQ", dq, rdq), ("dK", dk, rdk), ("dV", dv, rdv)):
        _close(name, a, r)


@pytest.mark.parametrize("dm", [256, 512])
def test_weight_gradient_waits_run_out_then_recover(dm):
    """The same for the projection weight-gradient kernel (one and two d_model
    tiles): with a one-cycle limit its waits run out and the status says so
    once; with the default limit it matches the oracle again."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    lib = binding.load_library()
    B, T, n, r0, r1 = 1, 512, 256, 64, 448
    h = inputs.draw("h", 7, B, T, 1, dm, torch.bfloat16)[:, :, 0].contiguous()
    g = inputs.draw("do", 7, B, T, 1, n, torch.float32)[:, :, 0].contiguous()
    hd, gd = h.cuda(), g.cuda()
    dw = torch.zeros((dm, n), device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.seqattn_sync_status(stream) == binding.SEQATTN_OK
    try:
        binding.set_wait_limit(1)
        binding.proj_wgrad(hd, gd, dw, r0, r1)
        assert lib.seqattn_sync_status(stream) == binding.SEQATTN_ERR_TIMEOUT
        assert lib.seqattn_sync_status(stream) == binding.SEQATTN_OK
    finally:
        binding.set_wait_limit(0)
    dw.zero_()
    binding.proj_wgrad(hd, gd, dw, r0, r1)
    assert lib.seqattn_sync_status(stream) == binding.SEQATTN_OK
    ref = oracle.projection_wgrad(h[:, r0:r1].double().numpy(), g[:, r0:r1].double().numpy())
    got = dw.double().cpu().numpy()
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert rel <= BF16_REL, f"dW after the timeout: rel-L2 {rel:.3e}"
