"""Pins for the float64 CPU oracle: each check ties the oracle to something
other than itself (a hand-derived example, finite differences, an independent
Jacobian route, torch autograd, closed forms and invariants), on inputs small
enough to run in seconds."""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from long_context_attention_seqattn_gb300 import inputs, workloads


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _layer(T=12, Hq=2, Hkv=1, d=4, B=1, seed=0):
    q = _rand((B, T, Hq, d), seed)
    k = _rand((B, T, Hkv, d), seed + 1)
    v = _rand((B, T, Hkv, d), seed + 2)
    do = _rand((B, T, Hq, d), seed + 3)
    return q, k, v, do


def _read_golden(path):
    vals = {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = line.split("=")
        vals[key.strip()] = np.array([float(x) for x in val.split()])
    return vals


# ---------------------------------------------------------------- hand-derived example

@pytest.mark.parametrize("chunk", [1, 2])
def test_two_token_hand_example(golden_dir, chunk):
    g = _read_golden(os.path.join(golden_dir, "two_token_hand.txt"))
    q = g["q"].reshape(1, 2, 1, 1)
    k = g["k"].reshape(1, 2, 1, 1)
    v = g["v"].reshape(1, 2, 1, 1)
    do = g["do"].reshape(1, 2, 1, 1)
    o, lse, dq, dk, dv = oracle.chunked_layer(q, k, v, do, chunk, float(g["scale"][0]))
    np.testing.assert_allclose(o.ravel(), g["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse.ravel(), g["lse"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dq.ravel(), g["dq"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk.ravel(), g["dk"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv.ravel(), g["dv"], rtol=0, atol=1e-14)


# ---------------------------------------------------------------- finite differences

def _loss(q, k, v, do, scale, chunk):
    o, _, _, _, _ = oracle.chunked_layer(q, k, v, do, chunk, scale)
    return float((o * do).sum())


@pytest.mark.parametrize("chunk", [4, 5])
def test_gradients_match_finite_differences(chunk):
    q, k, v, do = _layer(T=12, Hq=4, Hkv=2, d=4, seed=3)
    scale = 0.7
    _, _, dq, dk, dv = oracle.chunked_layer(q, k, v, do, chunk, scale)
    h = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, do, scale, chunk)
            x[idx] = old - h
            lm = _loss(q, k, v, do, scale, chunk)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(fd - grad).max() / np.abs(grad).max()
        assert err < 1e-7, (name, err)


def test_lse_against_pure_python_sum():
    q, k, v, _ = _layer(T=9, Hq=2, Hkv=1, d=3, seed=11)
    scale = 0.5
    _, lse = oracle.chunk_forward(q[:, 4:9], k, v, 4, 4, scale)
    for h in range(2):
        for r in range(5):
            pos = 4 + r
            terms = [math.exp(scale * sum(q[0, pos, h, e] * k[0, j, 0, e] for e in range(3)))
                     for j in range(pos + 1)]
            assert abs(lse[0, h, r] - math.log(math.fsum(terms))) < 1e-13


# ---------------------------------------------------------------- D-chunk vs dense D=1

@pytest.mark.parametrize("chunk", [1, 3, 4, 7, 16])
def test_chunked_equals_dense_jacobian_route(chunk):
    q, k, v, do = _layer(T=16, Hq=4, Hkv=2, d=8, B=2, seed=21)
    scale = 8 ** -0.5
    o, lse, dq, dk, dv = oracle.chunked_layer(q, k, v, do, chunk, scale)
    o1, lse1, _ = oracle.dense_causal_attention(q, k, v, scale)
    dq1, dk1, dv1 = oracle.dense_causal_attention_grad(q, k, v, do, scale)
    for a, b in ((o, o1), (lse, lse1), (dq, dq1), (dk, dk1), (dv, dv1)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_chunk_sum_invariant_over_partition_sweep():
    """Running sums over D chunks equal the D=1 gradients for every chunk size
    of a partition sweep (StreamBP review page, Eq. (1); Figure 5 varies ps)."""
    q, k, v, do = _layer(T=64, Hq=4, Hkv=1, d=8, seed=5)
    scale = 8 ** -0.5
    ref = oracle.chunked_layer(q, k, v, do, 64, scale)
    for chunk in (4, 8, 16, 32, 64, 20):
        got = oracle.chunked_layer(q, k, v, do, chunk, scale)
        for a, b in zip(got, ref):
            np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_backward_order_is_irrelevant():
    q, k, v, do = _layer(T=24, Hq=2, Hkv=2, d=4, seed=8)
    a = oracle.chunked_layer(q, k, v, do, 6, 0.4, bwd_order="descending")
    b = oracle.chunked_layer(q, k, v, do, 6, 0.4, bwd_order="ascending")
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- torch float64 cross-check

def test_against_torch_autograd_and_sdpa():
    T, Hq, Hkv, d = 20, 6, 2, 8
    q, k, v, do = _layer(T=T, Hq=Hq, Hkv=Hkv, d=d, seed=31)
    scale = 0.3
    o, lse, dq, dk, dv = oracle.chunked_layer(q, k, v, do, 8, scale)

    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    G = Hq // Hkv
    qh = tq[0].permute(1, 0, 2)                               # [Hq, T, d]
    kh = tk[0].permute(1, 0, 2).repeat_interleave(G, dim=0)   # [Hq, T, d]
    vh = tv[0].permute(1, 0, 2).repeat_interleave(G, dim=0)
    s = scale * qh @ kh.transpose(1, 2)
    s = s.masked_fill(~torch.ones(T, T, dtype=torch.bool).tril(), float("-inf"))
    p = torch.softmax(s, dim=-1)
    out = (p @ vh).permute(1, 0, 2).unsqueeze(0)
    (out * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(out.detach().numpy(), o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(torch.logsumexp(s, -1).detach().numpy()[None], lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(tq.grad.numpy(), dq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(tk.grad.numpy(), dk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(tv.grad.numpy(), dv, rtol=0, atol=1e-12)

    sdpa = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q).permute(0, 2, 1, 3), torch.tensor(k).permute(0, 2, 1, 3),
        torch.tensor(v).permute(0, 2, 1, 3), is_causal=True, scale=scale, enable_gqa=True)
    np.testing.assert_allclose(sdpa.permute(0, 2, 1, 3).numpy(), o, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms and invariants

def test_zero_scale_is_prefix_mean():
    q, k, v, do = _layer(T=10, Hq=2, Hkv=1, d=3, seed=2)
    o, lse, dq, dk, dv = oracle.chunked_layer(q, k, v, do, 4, 0.0)
    counts = np.arange(1, 11)
    np.testing.assert_allclose(o[0, :, 0], np.cumsum(v[0, :, 0], axis=0) / counts[:, None], atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], np.log(counts), atol=1e-14)
    assert np.abs(dq).max() == 0 and np.abs(dk).max() == 0


def test_equal_value_rows_give_zero_score_gradients():
    q, k, v, do = _layer(T=10, Hq=2, Hkv=1, d=3, seed=4)
    v[:] = v[:, :1]
    o, lse, dq, dk, dv = oracle.chunked_layer(q, k, v, do, 3, 0.9)
    np.testing.assert_allclose(o, np.broadcast_to(v[:, :1], o.shape), atol=1e-14)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13


def test_first_row_sees_only_itself():
    q, k, v, do = _layer(T=6, Hq=2, Hkv=2, d=5, seed=6)
    o, lse, _, _, _ = oracle.chunked_layer(q, k, v, do, 2, 0.8)
    np.testing.assert_allclose(o[0, 0], v[0, 0], atol=1e-15)
    np.testing.assert_allclose(lse[0, :, 0], 0.8 * (q[0, 0] * k[0, 0]).sum(-1), atol=1e-15)


def test_gradient_sum_invariants():
    """sum_j dV[j] = sum over the group's rows of dO (softmax rows sum to 1);
    sum_j dK[j] = 0 (each row of dS sums to zero because of the Delta term)."""
    Hq, Hkv = 6, 2
    q, k, v, do = _layer(T=15, Hq=Hq, Hkv=Hkv, d=4, seed=9)
    _, _, _, dk, dv = oracle.chunked_layer(q, k, v, do, 4, 0.6)
    G = Hq // Hkv
    for g in range(Hkv):
        np.testing.assert_allclose(dv[0, :, g].sum(0), do[0, :, g * G:(g + 1) * G].sum((0, 1)), atol=1e-12)
        np.testing.assert_allclose(dk[0, :, g].sum(0), 0.0, atol=1e-12)


def test_gqa_equals_duplicated_heads():
    """GQA with group G equals multi-head attention on G-fold duplicated K/V
    heads, with dK/dV summed over the duplicates."""
    Hq, Hkv = 6, 2
    G = Hq // Hkv
    q, k, v, do = _layer(T=11, Hq=Hq, Hkv=Hkv, d=4, seed=12)
    a = oracle.chunked_layer(q, k, v, do, 4, 0.5)
    kk, vv = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    b = oracle.chunked_layer(q, kk, vv, do, 4, 0.5)
    for x, y in zip(a[:3], b[:3]):
        np.testing.assert_allclose(x, y, atol=1e-13)
    np.testing.assert_allclose(a[3], b[3].reshape(1, 11, Hkv, G, 4).sum(3), atol=1e-13)
    np.testing.assert_allclose(a[4], b[4].reshape(1, 11, Hkv, G, 4).sum(3), atol=1e-13)


def test_truncated_prefix_equals_sliced_sequence():
    """prefix_len < q_start: rows attend keys [q_start - prefix_len, row]; the
    same as the full prefix on the sequence cut at q_start - prefix_len."""
    q, k, v, do = _layer(T=20, Hq=2, Hkv=1, d=4, seed=14)
    qs, p, c = 12, 5, 6
    o, lse = oracle.chunk_forward(q[:, qs:qs + c], k, v, qs, p, 0.7)
    o2, lse2 = oracle.chunk_forward(q[:, qs:qs + c], k[:, qs - p:], v[:, qs - p:], p, p, 0.7)
    np.testing.assert_allclose(o, o2, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, atol=1e-14)
    dk, dv = np.zeros_like(k), np.zeros_like(v)
    dk2, dv2 = np.zeros_like(k[:, qs - p:]), np.zeros_like(v[:, qs - p:])
    dq = oracle.chunk_backward(q[:, qs:qs + c], k, v, o, lse, do[:, qs:qs + c], qs, p, 0.7, dk, dv)
    dq2 = oracle.chunk_backward(q[:, qs:qs + c], k[:, qs - p:], v[:, qs - p:], o2, lse2,
                                do[:, qs:qs + c], p, p, 0.7, dk2, dv2)
    np.testing.assert_allclose(dq, dq2, atol=1e-14)
    np.testing.assert_allclose(dk[:, qs - p:], dk2, atol=1e-14)
    assert np.abs(dk[:, :qs - p]).max() == 0 and np.abs(dv[:, :qs - p]).max() == 0


def test_empty_chunk_is_a_no_op():
    q, k, v, do = _layer(T=8, seed=1)
    o, lse = oracle.chunk_forward(q[:, 4:4], k, v, 4, 4, 0.5)
    assert o.shape == (1, 0, 2, 4) and lse.shape == (1, 2, 0)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dq = oracle.chunk_backward(q[:, 4:4], k, v, o, lse, do[:, 4:4], 4, 4, 0.5, dk, dv)
    assert dq.shape == (1, 0, 2, 4) and not dk.any() and not dv.any()


# ---------------------------------------------------------------- sampled-row helpers

def test_row_and_tail_helpers_match_the_layer():
    q, k, v, do = _layer(T=40, Hq=4, Hkv=2, d=6, seed=17)
    scale = 0.45
    o, lse, dq, dk, dv = oracle.chunked_layer(q, k, v, do, 8, scale)
    for r, h in ((0, 0), (17, 3), (39, 1)):
        g = h // 2
        orow, lrow = oracle.row_forward(q[0, r, h], k[0, :, g], v[0, :, g], r, 0, scale)
        np.testing.assert_allclose(orow, o[0, r, h], atol=1e-13)
        assert abs(lrow - lse[0, h, r]) < 1e-13
        dqr = oracle.row_dq(q[0, r, h], do[0, r, h], o[0, r, h], k[0, :, g], v[0, :, g], r, 0, scale)
        np.testing.assert_allclose(dqr, dq[0, r, h], atol=1e-13)
    t = oracle.tail_block(q[0, 29:, 2:4], k[0, :, 1], v[0, :, 1], do[0, 29:, 2:4], 29, scale,
                          row_block=4)
    np.testing.assert_allclose(t["o"], o[0, 29:, 2:4], atol=1e-13)
    np.testing.assert_allclose(t["lse"], lse[0, 2:4, 29:], atol=1e-13)
    np.testing.assert_allclose(t["dq"], dq[0, 29:, 2:4], atol=1e-13)
    np.testing.assert_allclose(t["dk"], dk[0, 29:, 1], atol=1e-13)
    np.testing.assert_allclose(t["dv"], dv[0, 29:, 1], atol=1e-13)


# ---------------------------------------------------------------- planted mistakes

def test_pins_catch_planted_mistakes():
    """Plant plausible mistakes into the oracle's inputs/outputs (on the CPU)
    and check that a pin above fails for each: a dropped Delta term, a dK
    without the scale, and transposed score operands."""
    q, k, v, do = _layer(T=10, Hq=2, Hkv=1, d=3, seed=23)
    scale = 0.8
    o, lse, dq, dk, dv = oracle.chunked_layer(q, k, v, do, 5, scale)
    dq1, dk1, dv1 = oracle.dense_causal_attention_grad(q, k, v, do, scale)
    # dropped Delta: pass O = 0 so that Delta vanishes
    dk_bad, dv_bad = np.zeros_like(k), np.zeros_like(v)
    oracle.chunk_backward(q, k, v, np.zeros_like(o), lse, do, 0, 0, scale, dk_bad, dv_bad)
    assert np.abs(dk_bad - dk1).max() > 1e-3
    assert np.abs(dk_bad[0, :, 0].sum(0)).max() > 1e-3      # sum-invariant fails too
    # missing scale in dK
    assert np.abs(dk / scale - dk1).max() > 1e-3
    # transposed score operands (keys as queries)
    o_t, _, _ = oracle.dense_causal_attention(np.repeat(k, 2, axis=2), q[:, :, :1], v, scale)
    assert np.abs(o_t[:, :, :1] - o[:, :, :1]).max() > 1e-3


# ---------------------------------------------------------------- SpaCO (sampled chunks)

def _spaco_expected(q, k, v, do, chunk, scale, selected, factor):
    """SpaCO's result composed by hand from the dense gradient: the gradient is
    linear in dO, so chunk j's own contribution C_j is the dense gradient with
    dO zeroed outside chunk j.  Rows of a selected chunk i receive
    factor * sum_{selected j > i} C_j + C_i; rows of other chunks are zero;
    dQ rows of a selected chunk come from its own dO only."""
    B, T, Hq, d = q.shape
    starts = list(range(0, T, chunk))
    contrib = []
    for s in starts:
        e = min(s + chunk, T)
        do_j = np.zeros_like(do)
        do_j[:, s:e] = do[:, s:e]
        contrib.append(oracle.dense_causal_attention_grad(q, k, v, do_j, scale))
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for i, s in enumerate(starts):
        e = min(s + chunk, T)
        if i not in selected:
            continue
        dq[:, s:e] = contrib[i][0][:, s:e]
        later = [j for j in selected if j > i]
        dk[:, s:e] = contrib[i][1][:, s:e] + factor * sum((contrib[j][1][:, s:e] for j in later), 0.0)
        dv[:, s:e] = contrib[i][2][:, s:e] + factor * sum((contrib[j][2][:, s:e] for j in later), 0.0)
    return dq, dk, dv


@pytest.mark.parametrize("selected,factor", [((0, 2, 3), 2.0), ((1, 4), 2.0), ((0, 1, 2, 3, 4), 1.25), ((3,), 0.0)])
def test_spaco_matches_the_hand_composition(selected, factor):
    q, k, v, do = _layer(T=20, Hq=4, Hkv=2, d=4, B=2, seed=41)
    scale = 0.6
    o, lse, dq, dk, dv = oracle.sparse_chunked_layer(q, k, v, do, 4, scale, selected, factor)
    edq, edk, edv = _spaco_expected(q, k, v, do, 4, scale, set(selected), factor)
    o1, lse1, _ = oracle.dense_causal_attention(q, k, v, scale)
    for a, b in ((o, o1), (lse, lse1), (dq, edq), (dk, edk), (dv, edv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_spaco_with_every_chunk_and_no_compensation_is_exact():
    """t = k with factor 1 is SeCO: the exact dense gradient."""
    q, k, v, do = _layer(T=15, Hq=2, Hkv=1, d=4, seed=43)
    got = oracle.sparse_chunked_layer(q, k, v, do, 4, 0.5, range(4), 1.0)
    dq1, dk1, dv1 = oracle.dense_causal_attention_grad(q, k, v, do, 0.5)
    for a, b in zip(got[2:], (dq1, dk1, dv1)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_spaco_pin_catches_a_compensated_direct_term():
    """A plausible mistake -- scaling the chunk's own term along with the
    relayed one -- fails the hand composition."""
    q, k, v, do = _layer(T=12, Hq=2, Hkv=1, d=4, seed=47)
    sel, f = (0, 2), 2.0
    _, _, _, dk, _ = oracle.sparse_chunked_layer(q, k, v, do, 4, 0.7, sel, f)
    _, edk, _ = _spaco_expected(q, k, v, do, 4, 0.7, set(sel), f)
    do_0 = np.zeros_like(do)
    do_0[:, 0:4] = do[:, 0:4]
    own_0 = oracle.dense_causal_attention_grad(q, k, v, do_0, 0.7)[1]
    bad = edk.copy()
    bad[:, 0:4] += (f - 1.0) * own_0[:, 0:4]           # chunk 0's own term scaled too
    assert np.abs(bad - dk).max() > 1e-3 and np.abs(edk - dk).max() < 1e-12


# ---------------------------------------------------------------- projection weight gradients

def test_projection_wgrad_matches_autograd_through_the_projections():
    """A tiny float64 model: Q = H W_q, K = H W_k, V = H W_v feed causal GQA
    attention and L = sum dO o O.  torch autograd's dW_q, dW_k, dW_v equal
    H^T dQ, H^T dK, H^T dV with dQ, dK, dV from the chunked oracle."""
    B, T, dm, Hq, Hkv, d = 2, 10, 6, 4, 2, 3
    rng = np.random.default_rng(51)
    h = rng.standard_normal((B, T, dm))
    wq, wk, wv = (rng.standard_normal((dm, n)) for n in (Hq * d, Hkv * d, Hkv * d))
    do = rng.standard_normal((B, T, Hq, d))
    scale = d ** -0.5
    th = torch.tensor(h)
    tw = [torch.tensor(w, requires_grad=True) for w in (wq, wk, wv)]
    q = (th @ tw[0]).view(B, T, Hq, d)
    k = (th @ tw[1]).view(B, T, Hkv, d)
    v = (th @ tw[2]).view(B, T, Hkv, d)
    kk = k.repeat_interleave(Hq // Hkv, dim=2)
    vv = v.repeat_interleave(Hq // Hkv, dim=2)
    s = torch.einsum("bihe,bjhe->bhij", q, kk) * scale
    mask = torch.ones(T, T, dtype=torch.bool).tril()
    p = torch.softmax(s.masked_fill(~mask, float("-inf")), dim=-1)
    o = torch.einsum("bhij,bjhe->bihe", p, vv)
    (o * torch.tensor(do)).sum().backward()
    _, _, dq, dk, dv = oracle.chunked_layer(q.detach().numpy(), k.detach().numpy(), v.detach().numpy(), do, 4,
                                            scale)
    for w, g in zip(tw, (dq, dk, dv)):
        np.testing.assert_allclose(oracle.projection_wgrad(h, g), w.grad.numpy(), rtol=0, atol=1e-11)


def test_projection_wgrad_splits_over_chunks_and_matches_loops():
    """The row sum splits over chunks (the relay order runs it chunk by chunk),
    and equals the element-wise triple loop on a tiny case."""
    rng = np.random.default_rng(53)
    h = rng.standard_normal((2, 7, 3))
    g = rng.standard_normal((2, 7, 4))
    full = oracle.projection_wgrad(h, g)
    parts = sum(oracle.projection_wgrad(h[:, s:s + 3], g[:, s:s + 3]) for s in range(0, 7, 3))
    np.testing.assert_allclose(parts, full, rtol=0, atol=1e-12)
    loops = np.zeros((3, 4))
    for b in range(2):
        for r in range(7):
            for i in range(3):
                for j in range(4):
                    loops[i, j] += h[b, r, i] * g[b, r, j]
    np.testing.assert_allclose(full, loops, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- input generator

def test_inputs_are_seeded_and_block_addressable():
    a = inputs.draw("k", 7, 2, 2500, 3, 8, torch.float32)
    b = inputs.draw("k", 7, 2, 2500, 3, 8, torch.float32)
    assert torch.equal(a, b)
    assert torch.equal(a[1, 1000:2100], inputs.draw_rows("k", 7, 1, 1000, 2100, 3, 8, torch.float32))
    c = inputs.draw("v", 7, 2, 2500, 3, 8, torch.float32)
    assert not torch.equal(a, c)
    assert abs(float(a.mean())) < 0.02 and abs(float(a.std()) - 1) < 0.02
    h = inputs.draw("q", 7, 1, 100, 2, 8, torch.bfloat16)
    assert h.dtype == torch.bfloat16
    assert torch.equal(h, inputs.draw("q", 7, 1, 100, 2, 8, torch.float32).to(torch.bfloat16))


def test_causal_flop_count():
    w = workloads.WORKLOADS["llama3-8b-layer-t32768-c2048"]
    assert w.causal_flops() == 14 * 32 * 128 * 32768 * 32769 // 2
    pairs = sum(workloads.causal_pairs(s, 2048) for s in workloads.chunk_starts(32768, 2048))
    assert pairs == 32768 * 32769 // 2
