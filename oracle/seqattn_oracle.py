"""Float64 CPU oracle for sequence-partitioned causal attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this module:
only the test suite, the package smoke check and the benchmark's CPU-baseline
leg call it.  It shares no code, constants or helpers with the CUDA library.

What it computes
----------------
The method is exact: chunk-wise processing reaches full causal attention and
its exact gradient (StreamBP review page, "What carries the argument", Eq. (1)
and Property 3.1; SeCO review page, "Referee Report", Summary, which reports
element-wise float64 agreement of the chunked and dense gradients).  The oracle
is therefore the textbook definition written out in float64:

  forward, chunk i (queries at absolute rows q_start .. q_start+c-1):
    S[r, j]   = scale * <Q[r], K[j]>        for keys j in [q_start-prefix_len, q_start+r]
    LSE[r]    = ln sum_j exp(S[r, j])        (the stored row statistic M^(i))
    P[r, j]   = exp(S[r, j] - LSE[r])
    O[r]      = sum_j P[r, j] V[j]
  backward, same chunk, given dO:
    dP[r, j]  = <dO[r], V[j]>
    Delta[r]  = <dO[r], O[r]>
    dS[r, j]  = P[r, j] (dP[r, j] - Delta[r])
    dQ[r]     = scale * sum_j dS[r, j] K[j]                 (overwritten)
    dK[j]    += scale * sum_r dS[r, j] Q[r]                 (running sum)
    dV[j]    += sum_r P[r, j] dO[r]                          (running sum)

The partitioned attention of Eqs. (12)-(14) and the running-sum accumulation
of dK/dV over the prefix are named in the StreamBP review page's "Circularity
Check" and in major comment 1 of its "Referee Report".  Readings where the
pages are silent (they print no equations for attention itself):

  * the stored statistic M^(i) is the natural-log row logsumexp of the scaled
    scores (the same symbol also names the mask partition in minor comment 2);
  * K^(:i) includes chunk i's own keys, causal inside the diagonal block;
  * grouped-query attention maps query head h to key/value head h // G with
    G = Hq / Hkv (contiguous groups);
  * the softmax scale multiplies the scores; it therefore appears in dQ and dK
    and not in dV;
  * Delta is formed from the O passed in (the caller's stored O).

Layouts (row-major numpy arrays, any float dtype; upcast to float64 here):
  q, o, do  : [B, c, Hq, d]   chunk-local rows
  k, v      : [B, T, Hkv, d]  full cache, row 0 = token 0
  lse       : [B, Hq, c]
  dk, dv    : [B, T, Hkv, d]  float64 running-sum buffers, updated in place
"""

import numpy as np

__all__ = [
    "chunk_forward",
    "chunk_backward",
    "chunked_layer",
    "sparse_chunked_layer",
    "projection_wgrad",
    "dense_causal_attention",
    "dense_causal_attention_grad",
    "row_forward",
    "row_dq",
    "tail_block",
]


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def _visible(q_start, c, kv_begin, kv_end):
    """Causal mask partition for chunk rows [q_start, q_start+c) against keys
    [kv_begin, kv_end): key j is visible to query row r iff j <= r.

    StreamBP review page, minor comment 2 on Eq. (13) (the mask partition is
    not defined there; this is the causal mask restricted to the chunk's rows
    and the prefix columns)."""
    rows = q_start + np.arange(c)
    cols = np.arange(kv_begin, kv_end)
    return cols[None, :] <= rows[:, None]


def _check(q, k, v, q_start, prefix_len):
    B, c, Hq, d = q.shape
    Bk, T, Hkv, dk = k.shape
    if k.shape != v.shape or Bk != B or dk != d:
        raise ValueError("shape mismatch between q and k/v")
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if not (0 <= prefix_len <= q_start) or q_start + c > T:
        raise ValueError("chunk does not fit the cache")
    return B, c, Hq, d, T, Hkv, Hq // Hkv


def chunk_forward(q, k, v, q_start, prefix_len, scale):
    """Forward pass of one chunk: returns (O^(i), LSE^(i)) in float64.

    StreamBP review page, Property 3.1 ("What carries the argument"): chunk i's
    output needs only Q^(i), K^(:i), V^(:i)."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, c, Hq, d, T, Hkv, G = _check(q, k, v, q_start, prefix_len)
    o = np.zeros((B, c, Hq, d))
    lse = np.zeros((B, Hq, c))
    if c == 0:
        return o, lse
    kv_begin, kv_end = q_start - prefix_len, q_start + c
    vis = _visible(q_start, c, kv_begin, kv_end)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            S = scale * (q[b, :, h, :] @ k[b, kv_begin:kv_end, g, :].T)
            S = np.where(vis, S, -np.inf)
            m = S.max(axis=1)
            l = np.exp(S - m[:, None]).sum(axis=1)
            lse_h = m + np.log(l)
            P = np.exp(S - lse_h[:, None])
            o[b, :, h, :] = P @ v[b, kv_begin:kv_end, g, :]
            lse[b, h, :] = lse_h
    return o, lse


def chunk_backward(q, k, v, o, lse, do, q_start, prefix_len, scale, dk_acc, dv_acc):
    """Backward pass of one chunk.  Returns dQ^(i) (float64, overwritten) and
    adds this chunk's contributions into dk_acc / dv_acc over the prefix rows
    [q_start - prefix_len, q_start + c).

    StreamBP review page: Eq. (1) (gradients are sums of per-chunk terms) and
    "Circularity Check" (the per-chunk dK/dV are accumulated as a running sum);
    major comment 1 names dK^(:i), dV^(:i) over the prefix."""
    q, k, v, o, lse, do = (_as64(x) for x in (q, k, v, o, lse, do))
    B, c, Hq, d, T, Hkv, G = _check(q, k, v, q_start, prefix_len)
    dq = np.zeros((B, c, Hq, d))
    if c == 0:
        return dq
    kv_begin, kv_end = q_start - prefix_len, q_start + c
    vis = _visible(q_start, c, kv_begin, kv_end)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            Qh, dOh, Oh = q[b, :, h, :], do[b, :, h, :], o[b, :, h, :]
            Kg, Vg = k[b, kv_begin:kv_end, g, :], v[b, kv_begin:kv_end, g, :]
            S = scale * (Qh @ Kg.T)
            P = np.where(vis, np.exp(np.where(vis, S, 0.0) - lse[b, h, :, None]), 0.0)
            dP = dOh @ Vg.T
            delta = (dOh * Oh).sum(axis=1)
            dS = P * (dP - delta[:, None])
            dq[b, :, h, :] = scale * (dS @ Kg)
            dk_acc[b, kv_begin:kv_end, g, :] += scale * (dS.T @ Qh)
            dv_acc[b, kv_begin:kv_end, g, :] += P.T @ dOh
    return dq


def chunked_layer(q, k, v, do, chunk, scale, bwd_order="descending"):
    """Whole layer through the chunk calls: forward over chunks 0..D-1, then
    backward chunk by chunk into zeroed running sums.  The SeCO review page's
    major comment 1 (the relayed cache gradient of Algorithm 2) implies the
    last-to-first order; the sum is exact in any order.

    q, do: [B, T, Hq, d]; k, v: [B, T, Hkv, d].  A ragged final chunk is
    allowed.  Returns O, LSE [B, Hq, T], dQ, dK, dV (float64)."""
    q, k, v, do = (_as64(x) for x in (q, k, v, do))
    B, T, Hq, d = q.shape
    starts = list(range(0, T, chunk))
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, T))
    for s in starts:
        e = min(s + chunk, T)
        o[:, s:e], lse[:, :, s:e] = chunk_forward(q[:, s:e], k, v, s, s, scale)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    order = starts[::-1] if bwd_order == "descending" else starts
    for s in order:
        e = min(s + chunk, T)
        dq[:, s:e] = chunk_backward(q[:, s:e], k, v, o[:, s:e], lse[:, :, s:e],
                                    do[:, s:e], s, s, scale, dk, dv)
    return o, lse, dq, dk, dv


def sparse_chunked_layer(q, k, v, do, chunk, scale, selected, factor):
    """SpaCO through the chunk calls (SeCO review page: "Referee Report",
    Summary -- t of the k chunks are chosen for backpropagation and the relayed
    KV-cache gradient is multiplied by k/t -- and its major comments on
    Algorithm 2, whose compensation touches only the relayed cache gradient and
    not a chunk's direct term, and on Section 6.4, which caps the factor at 2).

    The forward (the inference pass that builds every cache) runs over all
    chunks.  The backward visits chunks last to first.  A selected chunk i
    first multiplies the gradient that later selected chunks relayed into its
    own key/value rows by `factor`, then adds its own contributions over its
    whole key range.  A chunk that is not selected is not backpropagated: its
    rows, complete once every later chunk has run, are set to zero, since
    nothing propagates from them.  `selected` (the sampled chunk indices) and
    `factor` (min(k/t, 2) in the deployed method) are inputs.

    Returns O, LSE, dQ (zero rows for chunks not selected), dK, dV (float64)."""
    q, k, v, do = (_as64(x) for x in (q, k, v, do))
    B, T, Hq, d = q.shape
    starts = list(range(0, T, chunk))
    chosen = set(int(i) for i in selected)
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, T))
    for s in starts:
        e = min(s + chunk, T)
        o[:, s:e], lse[:, :, s:e] = chunk_forward(q[:, s:e], k, v, s, s, scale)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for i in reversed(range(len(starts))):
        s = starts[i]
        e = min(s + chunk, T)
        if i in chosen:
            dk[:, s:e] *= factor
            dv[:, s:e] *= factor
            dq[:, s:e] = chunk_backward(q[:, s:e], k, v, o[:, s:e], lse[:, :, s:e],
                                        do[:, s:e], s, s, scale, dk, dv)
        else:
            dk[:, s:e] = 0.0
            dv[:, s:e] = 0.0
    return o, lse, dq, dk, dv


def projection_wgrad(h, g):
    """Weight gradient of a projection X = H W from the gradient G of its
    output: dW = sum over batch entries and rows of H[b, r]^T G[b, r].

    This is the step after the path (SeCO review page, major comment 1 on
    Algorithm 2: once chunk i's cache gradient is complete, chunk i's graph --
    here its Q/K/V projections -- is backpropagated).  With G = dQ it gives
    dW_q; with the finished dK / dV rows it gives dW_k / dW_v.  The sum over
    rows splits over chunks, so chunk-by-chunk accumulation gives the same.

    h: [B, T, d_model]; g: [B, T, n] (any trailing head dims flattened).
    Returns dW [d_model, n] in float64."""
    h = _as64(h)
    g = _as64(g)
    B, T = h.shape[:2]
    h2 = h.reshape(B * T, -1)
    g2 = g.reshape(B * T, -1)
    return h2.T @ g2


def dense_causal_attention(q, k, v, scale):
    """Unchunked (D = 1) causal attention over the whole sequence, built from
    the explicit T x T lower-triangular mask matrix.  Returns O, LSE, P.

    This is the brute-force counterpart that the chunked sum must reproduce
    (StreamBP review page, Eq. (1); SeCO review page, Appendix D check)."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    mask = np.tril(np.ones((T, T), dtype=bool))
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, T))
    P_all = np.zeros((B, Hq, T, T))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            S = scale * np.einsum("re,je->rj", q[b, :, h, :], k[b, :, g, :])
            E = np.where(mask, np.exp(np.where(mask, S, 0.0) - S.max(axis=1, keepdims=True, where=mask, initial=-np.inf)), 0.0)
            Z = E.sum(axis=1, keepdims=True)
            P = E / Z
            lse[b, h] = np.log(Z[:, 0]) + S.max(axis=1, where=mask, initial=-np.inf)
            o[b, :, h, :] = np.einsum("rj,je->re", P, v[b, :, g, :])
            P_all[b, h] = P
    return o, lse, P_all


def dense_causal_attention_grad(q, k, v, do, scale):
    """Gradients of L = sum(dO * O) for the unchunked attention, through the
    explicit softmax Jacobian J_r = diag(p_r) - p_r p_r^T of every row (no
    Delta shortcut), so it is an independent route to the chunked formula.
    Returns dQ, dK, dV (float64)."""
    q, k, v, do = (_as64(x) for x in (q, k, v, do))
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    _, _, P_all = dense_causal_attention(q, k, v, scale)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            P = P_all[b, h]
            dP = np.einsum("re,je->rj", do[b, :, h, :], v[b, :, g, :])
            dS = np.zeros((T, T))
            for r in range(T):
                p = P[r]
                J = np.diag(p) - np.outer(p, p)
                dS[r] = J.T @ dP[r]
            dq[b, :, h, :] = scale * np.einsum("rj,je->re", dS, k[b, :, g, :])
            dk[b, :, g, :] += scale * np.einsum("rj,re->je", dS, q[b, :, h, :])
            dv[b, :, g, :] += np.einsum("rj,re->je", P, do[b, :, h, :])
    return dq, dk, dv


def row_forward(q_row, k_head, v_head, row_pos, kv_begin, scale):
    """O and LSE of ONE query row at absolute position row_pos against keys
    [kv_begin, row_pos] of one key/value head ([T, d] arrays).  Used to check
    sampled rows of outputs too large for the full oracle."""
    q_row, K, V = _as64(q_row), _as64(k_head[kv_begin:row_pos + 1]), _as64(v_head[kv_begin:row_pos + 1])
    s = scale * (K @ q_row)
    m = s.max()
    lse = m + np.log(np.exp(s - m).sum())
    p = np.exp(s - lse)
    return p @ V, lse


def row_dq(q_row, do_row, o_row, k_head, v_head, row_pos, kv_begin, scale):
    """dQ of ONE query row (needs only that row's own softmax row), given the
    O row used for Delta.  Same formulas as chunk_backward."""
    q_row, do_row, o_row = _as64(q_row), _as64(do_row), _as64(o_row)
    K, V = _as64(k_head[kv_begin:row_pos + 1]), _as64(v_head[kv_begin:row_pos + 1])
    s = scale * (K @ q_row)
    m = s.max()
    lse = m + np.log(np.exp(s - m).sum())
    p = np.exp(s - lse)
    dp = V @ do_row
    ds = p * (dp - do_row @ o_row)
    return scale * (ds @ K)


def tail_block(q_tail, k_head, v_head, do_tail, j0, scale, row_block=64):
    """Whole-layer outputs restricted to the sequence tail [j0, T) for ONE
    key/value head and the G query heads of its group, straight from the
    full-sequence definition.  Because of causality, dK[j] and dV[j] for
    j >= j0 receive contributions only from query rows r >= j >= j0, so this
    tail is exact without touching query rows before j0 (StreamBP review page,
    Property 3.1).

    q_tail, do_tail: [T-j0, G, d] (rows j0..T-1 of the group's query heads);
    k_head, v_head: [T, d] (the whole cache of that key/value head).
    Returns a dict with o [T-j0, G, d], lse [G, T-j0], dq [T-j0, G, d],
    dk [T-j0, d], dv [T-j0, d]."""
    K = _as64(k_head)
    V = _as64(v_head)
    T, d = K.shape
    n, G, _ = q_tail.shape
    assert n == T - j0
    out = {"o": np.zeros((n, G, d)), "lse": np.zeros((G, n)), "dq": np.zeros((n, G, d)),
           "dk": np.zeros((n, d)), "dv": np.zeros((n, d))}
    for gi in range(G):
        for r0 in range(j0, T, row_block):
            r1 = min(r0 + row_block, T)
            rows = np.arange(r0, r1)
            Qr = _as64(q_tail[r0 - j0:r1 - j0, gi])
            dOr = _as64(do_tail[r0 - j0:r1 - j0, gi])
            S = scale * (Qr @ K[:r1].T)                      # keys [0, r1)
            vis = np.arange(r1)[None, :] <= rows[:, None]
            S = np.where(vis, S, -np.inf)
            m = S.max(axis=1)
            lse = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
            P = np.exp(S - lse[:, None])
            Or = P @ V[:r1]
            dP = dOr @ V[:r1].T
            dS = P * (dP - (dOr * Or).sum(axis=1)[:, None])
            out["o"][r0 - j0:r1 - j0, gi] = Or
            out["lse"][gi, r0 - j0:r1 - j0] = lse
            out["dq"][r0 - j0:r1 - j0, gi] = scale * (dS @ K[:r1])
            out["dk"][: r1 - j0] += scale * (dS[:, j0:].T @ Qr)
            out["dv"][: r1 - j0] += P[:, j0:].T @ dOr
    return out
