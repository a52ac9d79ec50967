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
