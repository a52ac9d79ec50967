"""Seeded synthetic inputs for chunked causal attention.

This module holds no attention arithmetic: it only draws random tensors.  It
is the one module that both the CUDA-path tests/benchmark and the CPU oracle
checks take their inputs from.

Recipe: Q, K, V and dO (and the hidden states H that feed the projections,
drawn as one head of d_model columns) are iid N(0, 1).  Each tensor is drawn in blocks of
``BLOCK_ROWS`` sequence rows per batch entry; every block has its own
``torch.Generator`` seeded with a 32-bit SplitMix64 hash of (seed, tensor id,
batch entry, block index),
so any block can be regenerated alone (for sampled checks of very long
sequences) and equals the same rows of the whole tensor.  Values are drawn in
float32 and then cast to the workload dtype with round-to-nearest-even.
"""

import torch

BLOCK_ROWS = 1024
TENSOR_IDS = {"q": 0, "k": 1, "v": 2, "do": 3, "h": 4}

_DTYPES = {"bf16": torch.bfloat16, "fp32": torch.float32}


def torch_dtype(name):
    return _DTYPES[name]


def _splitmix64(x):
    x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    return x ^ (x >> 31)


def _block_seed(seed, tensor_id, b, block):
    """32-bit seed of one block (torch's CPU generator keeps only 32 bits)."""
    key = (seed << 48) ^ (tensor_id << 40) ^ (b << 28) ^ block
    return _splitmix64(key) & 0xFFFFFFFF


def draw_rows(name, seed, b, row0, row1, heads, head_dim, dtype):
    """Rows [row0, row1) of tensor ``name`` for batch entry ``b``, shape
    [row1-row0, heads, head_dim], on the CPU in ``dtype``."""
    tid = TENSOR_IDS[name]
    out = torch.empty((max(0, row1 - row0), heads, head_dim), dtype=dtype)
    if row1 <= row0:
        return out
    for blk in range(row0 // BLOCK_ROWS, (row1 - 1) // BLOCK_ROWS + 1):
        g = torch.Generator(device="cpu")
        g.manual_seed(_block_seed(seed, tid, b, blk))
        full = torch.randn((BLOCK_ROWS, heads, head_dim), generator=g, dtype=torch.float32)
        s = max(row0, blk * BLOCK_ROWS)
        e = min(row1, (blk + 1) * BLOCK_ROWS)
        out[s - row0:e - row0] = full[s - blk * BLOCK_ROWS:e - blk * BLOCK_ROWS].to(dtype)
    return out


def draw(name, seed, batch, seq, heads, head_dim, dtype, device="cpu"):
    """Whole tensor ``name``: [batch, seq, heads, head_dim] in ``dtype`` on
    ``device``.  Filled block by block, so the host never holds more than one
    float32 block when ``device`` is a GPU."""
    out = torch.empty((batch, seq, heads, head_dim), dtype=dtype, device=device)
    for b in range(batch):
        for r0 in range(0, seq, BLOCK_ROWS):
            r1 = min(seq, r0 + BLOCK_ROWS)
            out[b, r0:r1].copy_(draw_rows(name, seed, b, r0, r1, heads, head_dim, dtype))
    return out


def layer_inputs(w, device="cpu", seed=None):
    """Q, K, V, dO for a workload ``w`` (see ``workloads``)."""
    seed = w.seed if seed is None else seed
    dt = torch_dtype(w.dtype)
    q = draw("q", seed, w.batch, w.seq, w.hq, w.head_dim, dt, device)
    k = draw("k", seed, w.batch, w.seq, w.hkv, w.head_dim, dt, device)
    v = draw("v", seed, w.batch, w.seq, w.hkv, w.head_dim, dt, device)
    do = draw("do", seed, w.batch, w.seq, w.hq, w.head_dim, dt, device)
    return q, k, v, do


def planted_growth_inputs(batch, seq, hq, hkv, head_dim, seed, dtype=torch.bfloat16, jump_log2=10.0,
                          period=96, levels=3, width=16):
    """Q, K, V, dO whose score row maxima rise along the key axis.

    The iid N(0, 1) tensors of ``draw`` give scores of about N(0, 1) after the
    1/sqrt(d) scale, so a row's maximum hardly moves once the first key tile
    has been seen.  These inputs make it move.  Coordinates [0, width) of key
    row j are overwritten with beta * min(floor(j / period), levels) /
    sqrt(width) (a staircase that rises every ``period`` keys for ``levels``
    steps, then stays flat), and the same coordinates of query row r of head
    h with alpha / sqrt(width) when h % 4 == 0 or (r + h) % 3 != 0, and with 0
    otherwise (every row of heads 0, 4, ...; two rows in three of the others).
    The planted part of a score is then alpha * beta * stair; with the scale
    1/sqrt(head_dim) each stair lifts the score of a planted row by
    ``jump_log2`` in base-2 units (alpha beta = jump_log2 ln(2) sqrt(d)), so its
    maximum grows by that much every ``period`` keys, while the unplanted rows
    in between keep flat scores.  alpha = beta * levels (the geometric middle)
    and the spread over ``width`` coordinates keep every planted entry small,
    which keeps the bf16 rounding of P and dS from being magnified in dQ and
    dK.  V and dO are the plain draws.  Everything else is as in ``draw``."""
    q = draw("q", seed, batch, seq, hq, head_dim, torch.float32)
    k = draw("k", seed, batch, seq, hkv, head_dim, torch.float32)
    v = draw("v", seed, batch, seq, hkv, head_dim, dtype)
    do = draw("do", seed, batch, seq, hq, head_dim, dtype)
    prod = jump_log2 * 0.6931471805599453 * head_dim ** 0.5   # alpha * beta
    alpha = (prod * levels) ** 0.5
    beta = prod / alpha
    spread = width ** -0.5
    stairs = torch.clamp(torch.div(torch.arange(seq), period, rounding_mode="floor"), max=levels)
    k[:, :, :, :width] = (beta * spread * stairs.to(torch.float32))[None, :, None, None]
    rows = torch.arange(seq)[:, None]
    heads = torch.arange(hq)[None, :]
    planted = (heads % 4 == 0) | ((rows + heads) % 3 != 0)
    q[:, :, :, :width] = torch.where(planted, alpha * spread, 0.0)[None, :, :, None]
    return q.to(dtype), k.to(dtype), v, do
