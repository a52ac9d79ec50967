"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs.

Bars: float32 -> rel-L2 <= 1e-5 per output tensor; bf16 -> rel-L2 <= 2e-2 and
max-abs <= 5e-2 per output tensor; D-chunk against D=1 within the bf16 bar.
rel-L2 = ||x - y||_2 / ||y||_2 over the whole tensor, y the reference."""

import numpy as np
import pytest
import torch

import oracle
from long_context_attention_seqattn_gb300 import binding, inputs, workloads

pytestmark = pytest.mark.gpu

F32_REL = 1e-5
BF16_REL = 2e-2
BF16_ABS = 5e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_attention_seqattn_gb300 import build
    build.build()
    binding.load_library()
    yield
    binding.sync_status()


def rel_l2(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300))


def max_abs(x, y):
    return float(np.abs(np.asarray(x, dtype=np.float64) - np.asarray(y, dtype=np.float64)).max())


def assert_bf16(name, got, ref):
    r, a = rel_l2(got, ref), max_abs(got, ref)
    assert r <= BF16_REL and a <= BF16_ABS, f"{name}: rel-L2 {r:.3e} max-abs {a:.3e}"


def assert_f32(name, got, ref):
    r = rel_l2(got, ref)
    assert r <= F32_REL, f"{name}: rel-L2 {r:.3e}"


def cpu64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def run_layer(q, k, v, do, chunk, order="descending"):
    bufs = binding.layer_forward_backward(q, k, v, do, chunk, bwd_order=order)
    binding.sync_status()
    return bufs


def small_inputs(B, T, Hq, Hkv, d, dtype, seed):
    dt = inputs.torch_dtype(dtype)
    return [inputs.draw(n, seed, B, T, h, d, dt) for n, h in (("q", Hq), ("k", Hkv), ("v", Hkv), ("do", Hq))]


# ============================================================== float32 path

def _check_f32_layer(B, T, Hq, Hkv, d, chunk, seed, order="descending"):
    cpu = small_inputs(B, T, Hq, Hkv, d, "fp32", seed)
    q, k, v, do = (x.cuda() for x in cpu)
    bufs = run_layer(q, k, v, do, chunk, order)
    o, lse, dq, dk, dv = oracle.chunked_layer(*(x.numpy() for x in cpu), chunk, d ** -0.5)
    assert_f32("O", cpu64(bufs.o), o)
    assert_f32("LSE", cpu64(binding.gather_lse(bufs)), lse)
    assert_f32("dQ", cpu64(bufs.dq), dq)
    assert_f32("dK", cpu64(bufs.dk), dk)
    assert_f32("dV", cpu64(bufs.dv), dv)


def test_fp32_tiny_exactness_workload():
    w = workloads.WORKLOADS["tiny-fp32-t512-c128"]
    _check_f32_layer(w.batch, w.seq, w.hq, w.hkv, w.head_dim, w.chunk, w.seed)


@pytest.mark.parametrize("B,T,Hq,Hkv,d,chunk", [
    (2, 300, 4, 2, 128, 100),    # ragged chunks, GQA, d=128, batch 2
    (1, 257, 8, 1, 64, 64),      # ragged tail of one row, G=8
    (1, 96, 3, 3, 64, 96),       # single chunk (D=1), MHA
])
def test_fp32_ragged_shapes(B, T, Hq, Hkv, d, chunk):
    _check_f32_layer(B, T, Hq, Hkv, d, chunk, seed=11)


def test_fp32_ascending_order_matches():
    _check_f32_layer(1, 256, 2, 1, 64, 64, seed=5, order="ascending")


def test_fp32_truncated_prefix_single_chunk():
    B, T, Hq, Hkv, d = 1, 200, 2, 1, 64
    cpu = small_inputs(B, T, Hq, Hkv, d, "fp32", 21)
    q, k, v, do = (x.cuda() for x in cpu)
    qs, c, p = 120, 50, 37
    o = torch.empty((B, c, Hq, d), device="cuda")
    lse = torch.empty((B, Hq, c), device="cuda")
    binding.chunk_fwd(q[:, qs:qs + c].contiguous(), k, v, o, lse, qs, p)
    dq = torch.empty((B, c, Hq, d), device="cuda")
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    binding.chunk_bwd(q[:, qs:qs + c].contiguous(), k, v, o, lse, do[:, qs:qs + c].contiguous(),
                      dq, dk, dv, qs, p)
    binding.sync_status()
    qn, kn, vn, don = (x.numpy() for x in cpu)
    ro, rl = oracle.chunk_forward(qn[:, qs:qs + c], kn, vn, qs, p, d ** -0.5)
    rdk, rdv = np.zeros(kn.shape), np.zeros(vn.shape)
    rdq = oracle.chunk_backward(qn[:, qs:qs + c], kn, vn, ro, rl, don[:, qs:qs + c], qs, p,
                                d ** -0.5, rdk, rdv)
    assert_f32("O", cpu64(o), ro)
    assert_f32("LSE", cpu64(lse), rl)
    assert_f32("dQ", cpu64(dq), rdq)
    assert_f32("dK", cpu64(dk), rdk)
    assert_f32("dV", cpu64(dv), rdv)
    # rows outside [q_start - prefix_len, q_start + c) untouched
    assert float(dk[:, :qs - p].abs().max()) == 0.0 and float(dk[:, qs + c:].abs().max()) == 0.0


def test_fp32_guard_bands_untouched():
    """Outputs embedded in larger buffers filled with a canary: the kernels
    write only inside their tensors."""
    B, T, Hq, Hkv, d, c = 1, 256, 2, 2, 64, 128
    cpu = small_inputs(B, T, Hq, Hkv, d, "fp32", 3)
    q, k, v, do = (x.cuda() for x in cpu)
    canary = 12345.0
    pad = 4096
    big_o = torch.full((pad * 2 + B * c * Hq * d,), canary, device="cuda")
    big_l = torch.full((pad * 2 + B * Hq * c,), canary, device="cuda")
    o = big_o[pad:pad + B * c * Hq * d].view(B, c, Hq, d)
    lse = big_l[pad:pad + B * Hq * c].view(B, Hq, c)
    binding.chunk_fwd(q[:, 128:].contiguous(), k, v, o, lse, 128)
    binding.sync_status()
    for big in (big_o, big_l):
        assert float((big[:pad] != canary).sum()) == 0 and float((big[-pad:] != canary).sum()) == 0


def test_empty_chunk_no_op():
    k = torch.zeros((1, 256, 2, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((1, 0, 4, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros((1, 4, 0), device="cuda")
    binding.chunk_fwd(q, k, k, o, lse, 128)
    binding.sync_status()


# ============================================================== bf16 tensor-core path

def _bf16_group_check(w, cpu, bufs, chunk, groups):
    """Full comparison for the given key/value groups (all their query heads),
    against the oracle run on just those heads (groups are independent)."""
    q, k, v, do = cpu
    G = w.hq // w.hkv
    for g in groups:
        hs = slice(g * G, (g + 1) * G)
        args = [x.to(torch.float64).numpy() for x in (q[:, :, hs], k[:, :, g:g + 1], v[:, :, g:g + 1],
                                                       do[:, :, hs])]
        o, lse, dq, dk, dv = oracle.chunked_layer(*args, chunk, w.scale)
        assert_bf16(f"O g{g}", cpu64(bufs.o[:, :, hs]), o)
        assert_bf16(f"LSE g{g}", cpu64(binding.gather_lse(bufs)[:, hs]), lse)
        assert_bf16(f"dQ g{g}", cpu64(bufs.dq[:, :, hs]), dq)
        assert_bf16(f"dK g{g}", cpu64(bufs.dk[:, :, g:g + 1]), dk)
        assert_bf16(f"dV g{g}", cpu64(bufs.dv[:, :, g:g + 1]), dv)


def test_bf16_small_multi_tile():
    """Several q tiles and key tiles, GQA, two chunks plus the D=1 pass."""
    B, T, Hq, Hkv, d = 1, 768, 4, 2, 128
    w = workloads.Workload("small", B, T, Hq, Hkv, d, "bf16", (256,), 40)
    cpu = small_inputs(B, T, Hq, Hkv, d, "bf16", 40)
    dev = [x.cuda() for x in cpu]
    for chunk in (256, 384, 768):
        bufs = run_layer(*dev, chunk)
        _bf16_group_check(w, cpu, bufs, chunk, range(Hkv))


def _check_bf16_layer(B, T, Hq, Hkv, d, chunk, seed):
    w = workloads.Workload("ragged", B, T, Hq, Hkv, d, "bf16", (chunk,), seed)
    cpu = small_inputs(B, T, Hq, Hkv, d, "bf16", seed)
    bufs = run_layer(*[x.cuda() for x in cpu], chunk)
    _bf16_group_check(w, cpu, bufs, chunk, range(Hkv) if Hkv <= 2 else (0, Hkv - 1))


@pytest.mark.parametrize("B,T,Hq,Hkv,d,chunk", [
    (2, 2400, 32, 8, 128, 300),  # 8 key/value heads, G 4, more backward CTAs than SMs, ragged
    (2, 2400, 16, 8, 64, 200),   # the same with head_dim 64, G 2
    (2, 1000, 4, 2, 128, 500),   # the pages' partition size 500, batch 2
    (1, 257, 8, 1, 128, 100),    # ragged 57-row tail, G=8
    (1, 384, 2, 1, 128, 160),    # chunk starts off the 64/128 grid
    (1, 200, 2, 2, 128, 200),    # one chunk (D=1) of 200 rows, MHA
    (1, 70, 2, 1, 128, 1),       # one-row chunks
    (1, 768, 4, 2, 64, 256),     # head_dim 64, on the tile grid
    (2, 300, 4, 1, 64, 100),     # head_dim 64, ragged, G=4, batch 2
])
def test_bf16_ragged_shapes(B, T, Hq, Hkv, d, chunk):
    _check_bf16_layer(B, T, Hq, Hkv, d, chunk, seed=12)


@pytest.mark.parametrize("qs,c,p", [
    (300, 130, 171),   # chunk index q_start / q_len = 2: prefix tiles swept ascending
    (390, 130, 171),   # index 3: swept descending, batch entries in reverse order
])
def test_bf16_truncated_prefix_single_chunk(qs, c, p):
    """prefix_len < q_start: keys [q_start - prefix_len, q_start + r] only,
    with every bound off the tile grid; accumulator rows outside the window
    stay zero."""
    B, T, Hq, Hkv, d = 2, 600, 4, 2, 128
    cpu = small_inputs(B, T, Hq, Hkv, d, "bf16", 23)
    q, k, v, do = (x.cuda() for x in cpu)
    lse = torch.empty((B, Hq, c), device="cuda")
    o_c = torch.empty((B, c, Hq, d), dtype=torch.bfloat16, device="cuda")
    dq_c = torch.empty((B, c, Hq, d), device="cuda")
    binding.chunk_fwd(q[:, qs:qs + c].contiguous(), k, v, o_c, lse, qs, p)
    dk = torch.zeros(k.shape, device="cuda")
    dv = torch.zeros(v.shape, device="cuda")
    binding.chunk_bwd(q[:, qs:qs + c].contiguous(), k, v, o_c, lse, do[:, qs:qs + c].contiguous(),
                      dq_c, dk, dv, qs, p)
    binding.sync_status()
    qn, kn, vn, don = (x.to(torch.float64).numpy() for x in cpu)
    scale = d ** -0.5
    ro, rl = oracle.chunk_forward(qn[:, qs:qs + c], kn, vn, qs, p, scale)
    rdk, rdv = np.zeros(kn.shape), np.zeros(vn.shape)
    rdq = oracle.chunk_backward(qn[:, qs:qs + c], kn, vn, ro, rl, don[:, qs:qs + c], qs, p, scale,
                                rdk, rdv)
    assert_bf16("O", cpu64(o_c), ro)
    assert_bf16("LSE", cpu64(lse), rl)
    assert_bf16("dQ", cpu64(dq_c), rdq)
    assert_bf16("dK", cpu64(dk), rdk)
    assert_bf16("dV", cpu64(dv), rdv)
    assert float(dk[:, :qs - p].abs().max()) == 0.0 and float(dk[:, qs + c:].abs().max()) == 0.0
    assert float(dv[:, :qs - p].abs().max()) == 0.0 and float(dv[:, qs + c:].abs().max()) == 0.0


def test_bf16_ragged_guard_bands_untouched():
    """A chunk of 200 rows (partial last 128-row and 64-row tiles) with its
    outputs embedded in canary-filled buffers: forward and backward write
    only inside their tensors."""
    B, T, Hq, Hkv, d, qs, c = 1, 512, 4, 2, 128, 256, 200
    cpu = small_inputs(B, T, Hq, Hkv, d, "bf16", 31)
    q, k, v, do = (x.cuda() for x in cpu)
    canary = 4096.0                                   # exact in bf16 and fp32
    pad = 8192
    n_o, n_l = B * c * Hq * d, B * Hq * c
    big_o = torch.full((2 * pad + n_o,), canary, dtype=torch.bfloat16, device="cuda")
    big_l = torch.full((2 * pad + n_l,), canary, device="cuda")
    big_dq = torch.full((2 * pad + n_o,), canary, device="cuda")
    n_kv = B * T * Hkv * d
    big_dk = torch.full((2 * pad + n_kv,), canary, device="cuda")
    o = big_o[pad:pad + n_o].view(B, c, Hq, d)
    lse = big_l[pad:pad + n_l].view(B, Hq, c)
    dq = big_dq[pad:pad + n_o].view(B, c, Hq, d)
    dk = big_dk[pad:pad + n_kv].view(B, T, Hkv, d)
    dk.zero_()
    dv = torch.zeros(k.shape, device="cuda")
    binding.chunk_fwd(q[:, qs:qs + c].contiguous(), k, v, o, lse, qs)
    binding.chunk_bwd(q[:, qs:qs + c].contiguous(), k, v, o, lse, do[:, qs:qs + c].contiguous(),
                      dq, dk, dv, qs)
    binding.sync_status()
    for name, big in (("o", big_o), ("lse", big_l), ("dq", big_dq), ("dk", big_dk)):
        assert float((big[:pad].float() != canary).sum()) == 0, name
        assert float((big[-pad:].float() != canary).sum()) == 0, name
    assert float(dk[:, qs + c:].abs().max()) == 0.0 and float(dv[:, qs + c:].abs().max()) == 0.0


@pytest.mark.parametrize("dtype,B,T,Hq,Hkv,d,chunk,selected,factor", [
    ("bf16", 1, 1024, 4, 2, 128, 128, (0, 3, 5, 6), None),    # k/t = 2
    ("bf16", 2, 700, 4, 1, 64, 100, (1, 6), None),            # ragged last chunk, cap at 2
    ("bf16", 1, 512, 2, 2, 128, 128, (0, 1, 2, 3), 1.0),      # every chunk: the exact pass
    ("fp32", 1, 300, 4, 2, 64, 64, (0, 2, 4), 1.5),
])
def test_spaco_pass_matches_oracle(dtype, B, T, Hq, Hkv, d, chunk, selected, factor):
    """SpaCO through the library: forward over every chunk, backward over the
    selected chunks with the relayed rows compensated, other chunks' rows
    zeroed (the float64 oracle's sparse_chunked_layer on the same inputs)."""
    cpu = small_inputs(B, T, Hq, Hkv, d, dtype, 77)
    n_chunks = -(-T // chunk)
    f = binding.spaco_factor(n_chunks, len(selected)) if factor is None else factor
    bufs = binding.spaco_layer_forward_backward(*[x.cuda() for x in cpu], chunk, selected, f)
    binding.sync_status()
    ref = oracle.sparse_chunked_layer(*(x.to(torch.float64).numpy() for x in cpu), chunk, d ** -0.5,
                                      selected, f)
    got = (bufs.o, binding.gather_lse(bufs), bufs.dq, bufs.dk, bufs.dv)
    check = assert_bf16 if dtype == "bf16" else assert_f32
    for name, a, r in zip(("O", "LSE", "dQ", "dK", "dV"), got, ref):
        check(f"SpaCO {name}", cpu64(a), r)
    # rows of chunks that were not selected carry nothing
    for i in set(range(n_chunks)) - set(selected):
        s, e = i * chunk, min((i + 1) * chunk, T)
        for t in (bufs.dq, bufs.dk, bufs.dv):
            assert float(t[:, s:e].abs().max()) == 0.0


def assert_wgrad(name, got, ref):
    """Whole-tensor bars for a weight gradient: every element is a sum over
    many rows, so the element-wise 5e-2 of the attention outputs does not
    apply; rel-L2 <= 2e-2 and max-abs <= 1e-2 of the largest |ref| (G is
    rounded to bf16, relative error <= 2^-8 per term).  Where G is an exact
    input, the test adds the element-wise rounding bound."""
    r, a = rel_l2(got, ref), max_abs(got, ref)
    assert r <= BF16_REL and a <= 1e-2 * float(np.abs(ref).max()), f"{name}: rel-L2 {r:.3e} max-abs {a:.3e}"


@pytest.mark.parametrize("B,T,dm,n,r0,r1", [
    (2, 300, 96, 136, 37, 261),        # partial tiles everywhere: 224 rows, 96 of 256 d_model, 136 of 2 x 128 n
    (1, 4096, 4096, 1024, 2048, 4096),  # a dK/dV-shaped chunk of the 32768-token layer's projections
    (1, 1024, 640, 392, 0, 1000),      # 2.5 d_model tiles, 3 + 1/16 n tiles, ragged last stage
    (2, 700, 512, 200, 13, 650),       # two d_model tiles, a partial n tile, ragged rows, batch 2
])
def test_proj_wgrad_accumulates_h_transpose_g(B, T, dm, n, r0, r1):
    """dw += h^T g over a row range of every batch entry, twice (accumulation
    onto a non-zero dw), against the float64 oracle."""
    h = inputs.draw("h", 5, B, T, 1, dm, torch.bfloat16)[:, :, 0]
    g = inputs.draw("do", 5, B, T, 1, n, torch.float32)[:, :, 0]
    dw = torch.zeros((dm, n), device="cuda")
    hd, gd = h.cuda().contiguous(), g.cuda().contiguous()
    binding.proj_wgrad(hd, gd, dw, r0, r1)
    binding.proj_wgrad(hd, gd, dw, r0, r1)
    binding.sync_status()
    hn, gn = h[:, r0:r1].double().numpy(), g[:, r0:r1].double().numpy()
    ref = 2 * oracle.projection_wgrad(hn, gn)
    got = cpu64(dw)
    assert_wgrad("dW", got, ref)
    # element-wise bound from the arithmetic: H is exact, each G element is
    # rounded once to bf16 (8 significant bits: relative error <= 2^-8) and the
    # products are summed in fp32 (at most ~R 2^-24 <= 2^-12 relative to the
    # sum of magnitudes for R <= 4096 rows), twice; so per element
    # |dW - ref| <= 2 (2^-8 + 2^-12) sum_r |H[r, m]| |G[r, j]|
    bound = 2 * (2.0 ** -8 + 2.0 ** -12) * np.abs(hn.reshape(-1, dm)).T @ np.abs(gn.reshape(-1, n))
    over = np.abs(got - ref) > bound
    assert not over.any(), f"{int(over.sum())} elements beyond the rounding bound"


@pytest.mark.parametrize("B,T,Hq,Hkv,d,dm,chunk,streams", [
    (1, 512, 4, 2, 128, 256, 128, None),
    (1, 512, 4, 2, 128, 256, 128, 1),
    (2, 300, 4, 1, 64, 64, 100, None),  # ragged last chunk, d = 64, batch 2
    (2, 300, 4, 1, 64, 64, 100, 3),
])
def test_layer_pass_with_projection_wgrad(B, T, Hq, Hkv, d, dm, chunk, streams):
    """The relay pass with the projections' weight gradients: after chunk i's
    backward, dW_q, dW_k, dW_v += H^(i)T (dQ, dK, dV rows of chunk i).  The
    sum over chunks equals the oracle's H^T dQ, H^T dK, H^T dV, also with the
    chunk backwards spread over several streams (each chunk's weight
    gradients then wait until every stream has passed every later chunk)."""
    cpu = small_inputs(B, T, Hq, Hkv, d, "bf16", 88)
    h = inputs.draw("h", 88, B, T, 1, dm, torch.bfloat16)[:, :, 0]
    dws = [torch.zeros((dm, n), device="cuda") for n in (Hq * d, Hkv * d, Hkv * d)]
    bufs = binding.layer_forward_backward(*[x.cuda() for x in cpu], chunk,
                                          wgrad=(h.cuda().contiguous(), *dws), bwd_streams=streams)
    binding.sync_status()
    _, _, dq, dk, dv = oracle.chunked_layer(*(x.to(torch.float64).numpy() for x in cpu), chunk, d ** -0.5)
    hn = h.double().numpy()
    for name, got, g in zip(("dW_q", "dW_k", "dW_v"), dws, (dq, dk, dv)):
        assert_wgrad(name, cpu64(got), oracle.projection_wgrad(hn, g))


@pytest.mark.parametrize("streams", [2, 4])
def test_bf16_backward_streams_match_one_stream(streams):
    """Chunk backwards spread over several streams (their dK/dV reductions
    meeting in L2) give the one-stream pass up to the order of the fp32
    additions, and both match the oracle."""
    B, T, Hq, Hkv, d, chunk = 2, 700, 4, 2, 128, 128   # batch 2, ragged last chunk
    cpu = small_inputs(B, T, Hq, Hkv, d, "bf16", 77)
    dev = [x.cuda() for x in cpu]
    one = binding.layer_forward_backward(*dev, chunk, bwd_streams=1)
    ref = [x.clone() for x in (one.dq, one.dk, one.dv)]
    many = binding.layer_forward_backward(*dev, chunk, bwd_streams=streams)
    binding.sync_status()
    for name, a, r in zip(("dQ", "dK", "dV"), (many.dq, many.dk, many.dv), ref):
        a, r = cpu64(a), cpu64(r)
        rel = np.linalg.norm(a - r) / np.linalg.norm(r)
        assert rel <= 1e-5, f"{name}: {streams}-stream vs one-stream rel-L2 {rel:.2e}"
    _, _, dq, dk, dv = oracle.chunked_layer(*(x.to(torch.float64).numpy() for x in cpu), chunk, d ** -0.5)
    for name, a, r in zip(("dQ", "dK", "dV"), (many.dq, many.dk, many.dv), (dq, dk, dv)):
        assert_bf16(f"{streams} streams {name}", cpu64(a), r)


def test_bf16_qwen3_4b_layer_two_groups():
    w = workloads.WORKLOADS["qwen3-4b-layer-t8192-c512"]
    cpu = inputs.layer_inputs(w)
    dev = [x.cuda() for x in cpu]
    bufs = run_layer(*dev, w.chunk)
    _bf16_group_check(w, cpu, bufs, w.chunk, (0, w.hkv - 1))


def _sampled_check(w, bufs, groups, n_tail=256, sample_rows=(0, 1, 127, 128, 2047, 2048)):
    """Sampled rows of a full-size layer against the oracle, computed one by
    one from regenerated inputs (never from the GPU): the last n_tail rows and
    keys of the given groups in full (dK/dV of tail keys only involve tail
    rows), plus O/LSE/dQ of chosen rows anywhere in the sequence."""
    G = w.hq // w.hkv
    dt = inputs.torch_dtype(w.dtype)
    T, d = w.seq, w.head_dim
    lse_all = binding.gather_lse(bufs)
    for g in groups:
        k = inputs.draw_rows("k", w.seed, 0, 0, T, w.hkv, d, dt)[:, g].to(torch.float64).numpy()
        v = inputs.draw_rows("v", w.seed, 0, 0, T, w.hkv, d, dt)[:, g].to(torch.float64).numpy()
        j0 = T - n_tail
        qt = inputs.draw_rows("q", w.seed, 0, j0, T, w.hq, d, dt)[:, g * G:(g + 1) * G]
        dot = inputs.draw_rows("do", w.seed, 0, j0, T, w.hq, d, dt)[:, g * G:(g + 1) * G]
        ref = oracle.tail_block(qt.to(torch.float64).numpy(), k, v, dot.to(torch.float64).numpy(),
                                j0, w.scale)
        hs = slice(g * G, (g + 1) * G)
        assert_bf16(f"tail O g{g}", cpu64(bufs.o[0, j0:, hs]), ref["o"])
        assert_bf16(f"tail LSE g{g}", cpu64(lse_all[0, hs, j0:]), ref["lse"])
        assert_bf16(f"tail dQ g{g}", cpu64(bufs.dq[0, j0:, hs]), ref["dq"])
        assert_bf16(f"tail dK g{g}", cpu64(bufs.dk[0, j0:, g]), ref["dk"])
        assert_bf16(f"tail dV g{g}", cpu64(bufs.dv[0, j0:, g]), ref["dv"])
        got_o, ref_o, got_dq, ref_dq, got_l, ref_l = [], [], [], [], [], []
        for r in sample_rows:
            qr = inputs.draw_rows("q", w.seed, 0, r, r + 1, w.hq, d, dt)[0].to(torch.float64).numpy()
            dr = inputs.draw_rows("do", w.seed, 0, r, r + 1, w.hq, d, dt)[0].to(torch.float64).numpy()
            for h in (g * G, g * G + G - 1):
                o_r, l_r = oracle.row_forward(qr[h], k, v, r, 0, w.scale)
                ref_o.append(o_r)
                ref_l.append(l_r)
                ref_dq.append(oracle.row_dq(qr[h], dr[h], o_r, k, v, r, 0, w.scale))
                got_o.append(cpu64(bufs.o[0, r, h]))
                got_l.append(float(lse_all[0, h, r]))
                got_dq.append(cpu64(bufs.dq[0, r, h]))
        assert_bf16(f"rows O g{g}", np.array(got_o), np.array(ref_o))
        assert_bf16(f"rows LSE g{g}", np.array(got_l), np.array(ref_l))
        assert_bf16(f"rows dQ g{g}", np.array(got_dq), np.array(ref_dq))


def _sum_invariant(w, bufs):
    """sum_j dV[j] = sum over the group's rows of dO (softmax rows sum to one),
    at any size.  The sums run over T*G terms of magnitude ~1, so the
    element-wise absolute bar of the outputs does not apply to them: the check
    is rel-L2 <= 2e-2 and max-abs <= 1e-3 of the largest |sum|.  dO is
    regenerated block by block, so the reference never holds the whole
    tensor in float64."""
    G = w.hq // w.hkv
    dt = inputs.torch_dtype(w.dtype)
    ref = np.zeros((w.batch, w.hkv, w.head_dim))
    for b in range(w.batch):
        for r0 in range(0, w.seq, inputs.BLOCK_ROWS):
            r1 = min(w.seq, r0 + inputs.BLOCK_ROWS)
            blk = inputs.draw_rows("do", w.seed, b, r0, r1, w.hq, w.head_dim, dt).to(torch.float64)
            ref[b] += blk.view(r1 - r0, w.hkv, G, w.head_dim).sum((0, 2)).numpy()
    got = bufs.dv.to(torch.float64).sum(1).cpu().numpy()
    r, a = rel_l2(got, ref), max_abs(got, ref)
    assert r <= BF16_REL and a <= 1e-3 * np.abs(ref).max(), f"sum_j dV: rel-L2 {r:.3e} max-abs {a:.3e}"


def test_bf16_llama3_8b_layer_full_groups():
    """The 32768-token layer in the bench's launch configuration: every O,
    LSE, dQ, dK and dV element of key/value groups 0 and 7 (their four query
    heads each) against the oracle run on just those heads (groups are
    independent), plus sampled rows and the dV column-sum invariant."""
    w = workloads.WORKLOADS["llama3-8b-layer-t32768-c2048"]
    cpu = inputs.layer_inputs(w)
    bufs = run_layer(*[x.cuda() for x in cpu], w.chunk)
    _bf16_group_check(w, cpu, bufs, w.chunk, (0, w.hkv - 1))
    del cpu
    _sampled_check(w, bufs, (0, w.hkv - 1), sample_rows=(0, 1, 2047, 2048, 16383, 30720, 32767))
    _sum_invariant(w, bufs)


def test_bf16_32b_layer_t131072_sampled():
    w = workloads.WORKLOADS["32b-layer-t131072-c4096"]
    dev = inputs.layer_inputs(w, device="cuda")
    bufs = run_layer(*dev, w.chunk)
    _sampled_check(w, bufs, (0,), sample_rows=(0, 4095, 4096, 65536, 131071))
    _sum_invariant(w, bufs)


def test_bf16_partition_sweep_agrees_with_unchunked():
    """Every chunk size of the 16384-token sweep against the unchunked pass
    (the whole layer), and the unchunked pass, the smallest and a middle
    chunk size against the oracle on one key/value group each."""
    w = workloads.WORKLOADS["partition-sweep-t16384"]
    cpu = inputs.layer_inputs(w)
    dev = [x.cuda() for x in cpu]
    ref = run_layer(*dev, 16384)
    ref_t = [x.clone() for x in (ref.o, binding.gather_lse(ref), ref.dq, ref.dk, ref.dv)]
    # D=1 against the oracle on one key/value group
    _bf16_group_check(w, cpu, ref, 16384, (w.hkv - 1,))
    for chunk in w.chunks[:-1]:
        bufs = run_layer(*dev, chunk)
        got = (bufs.o, binding.gather_lse(bufs), bufs.dq, bufs.dk, bufs.dv)
        for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), got, ref_t):
            assert_bf16(f"c={chunk} {name} vs D=1", cpu64(a), cpu64(b))
        if chunk in (128, 512):
            _bf16_group_check(w, cpu, bufs, chunk, (0,))


def test_bf16_run_to_run_spread_qwen3_layer():
    """The 8192-token layer's chunk backwards run on four streams, their dK/dV
    reduce-adds and the dQ reductions meeting in L2 in an order that varies
    between runs.  Two passes on the same inputs differ only in the last bits:
    rel-L2 <= 1e-5 per output."""
    w = workloads.WORKLOADS["qwen3-4b-layer-t8192-c512"]
    dev = inputs.layer_inputs(w, device="cuda")
    assert binding.auto_bwd_streams(dev[0], dev[1], w.chunk) == 4
    first = run_layer(*dev, w.chunk)
    ref = [x.clone() for x in (first.dq, first.dk, first.dv)]
    second = run_layer(*dev, w.chunk)
    for name, a, r in zip(("dQ", "dK", "dV"), (second.dq, second.dk, second.dv), ref):
        rel = rel_l2(cpu64(a), cpu64(r))
        assert rel <= 1e-5, f"{name}: run-to-run rel-L2 {rel:.2e}"


def test_bf16_graph_replay_matches_eager():
    """A layer pass captured into a CUDA graph (for small chunks) computes the
    same as the eager chunk calls, also after the inputs change in place."""
    B, T, Hq, Hkv, d, chunk = 1, 1024, 4, 2, 128, 128
    dev = [x.cuda() for x in small_inputs(B, T, Hq, Hkv, d, "bf16", 55)]
    graph = binding.LayerGraph(*dev, chunk)
    for step in range(2):
        if step == 1:
            dev[0].mul_(0.5)
            dev[3].mul_(-1.0)
        eager = run_layer(*dev, chunk)
        ref = [x.clone() for x in (eager.o, binding.gather_lse(eager), eager.dq, eager.dk, eager.dv)]
        got_b = graph.replay()
        binding.sync_status()
        got = (got_b.o, binding.gather_lse(got_b), got_b.dq, got_b.dk, got_b.dv)
        for name, a, r in zip(("O", "LSE", "dQ", "dK", "dV"), got, ref):
            assert_bf16(f"graph step {step} {name}", cpu64(a), cpu64(r))


@pytest.mark.parametrize("B,T,chunk", [(1, 1024, 256), (2, 700, 256)])
def test_bf16_host_pass_matches_device_pass(B, T, chunk):
    """The host-buffer pass (inputs streamed in chunk by chunk, every output
    chunk copied back as soon as it is final) returns the device pass, also
    for a batch of two with a ragged last chunk."""
    Hq, Hkv, d = 4, 2, 128
    cpu = small_inputs(B, T, Hq, Hkv, d, "bf16", 66)
    pinned = [x.pin_memory() for x in cpu]
    hp = binding.HostLayerPass(*pinned, chunk)
    for _ in range(2):
        h_o, h_lse, h_dq, h_dk, h_dv = hp.run()
        torch.cuda.synchronize()
        binding.sync_status()
        ref = run_layer(*[x.cuda() for x in cpu], chunk)
        assert_bf16("O", h_o.double().numpy(), cpu64(ref.o))
        assert_bf16("LSE", torch.cat(h_lse, dim=2).double().numpy(), cpu64(binding.gather_lse(ref)))
        assert_bf16("dQ", h_dq.double().numpy(), cpu64(ref.dq))
        assert_bf16("dK", h_dk.double().numpy(), cpu64(ref.dk))
        assert_bf16("dV", h_dv.double().numpy(), cpu64(ref.dv))
