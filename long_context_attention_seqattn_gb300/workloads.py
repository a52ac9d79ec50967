"""Named workloads for chunked causal attention (shapes only, no arithmetic).

Shapes follow the layers the StreamBP and SeCO review pages discuss: a
Qwen3-4B-shaped layer with partition size ~500 (StreamBP verdict,
"skeptic_critique" concrete test), Llama-3-8B and 32B-shaped long-context
layers, and a partition-size sweep in the spirit of the StreamBP review page's
Figure 5 (time and memory against partition size).
"""

import math
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seq: int
    hq: int
    hkv: int
    head_dim: int
    dtype: str            # "bf16" or "fp32"
    chunks: tuple         # chunk lengths to run (one entry = one layer pass)
    seed: int
    note: str = field(default="", compare=False)

    @property
    def chunk(self):
        return self.chunks[0]

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.head_dim)

    def causal_flops(self):
        """Causal fwd+bwd FLOPs credited per layer pass: 14 * B * Hq * d *
        T(T+1)/2 (two contractions forward, five backward, 2 flops per MAC,
        over the T(T+1)/2 visible query/key pairs)."""
        return 14 * self.batch * self.hq * self.head_dim * self.seq * (self.seq + 1) // 2


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny-fp32-t512-c128", 1, 512, 2, 2, 64, "fp32", (128,), 0,
                 "exactness case, fp32"),
        Workload("qwen3-4b-layer-t8192-c512", 1, 8192, 32, 8, 128, "bf16", (512,), 1,
                 "Qwen3-4B-shaped layer, partition 512"),
        Workload("llama3-8b-layer-t32768-c2048", 1, 32768, 32, 8, 128, "bf16", (2048,), 2,
                 "Llama-3-8B-shaped layer, 16 chunks of 2048"),
        Workload("32b-layer-t131072-c4096", 1, 131072, 64, 8, 128, "bf16", (4096,), 3,
                 "32B-shaped long context, 32 chunks of 4096"),
        Workload("partition-sweep-t16384", 1, 16384, 32, 8, 128, "bf16",
                 (128, 256, 512, 1024, 2048, 4096, 16384), 4,
                 "partition-size sweep; 16384 is the unchunked pass"),
    ]
}

BENCH_WORKLOAD = "llama3-8b-layer-t32768-c2048"


def chunk_starts(seq, chunk):
    return list(range(0, seq, chunk))


def causal_pairs(q_start, q_len, kv_begin=0):
    """Number of visible (query, key) pairs of one chunk."""
    # row r (absolute q_start+r) sees keys [kv_begin, q_start+r]
    return q_len * (q_start - kv_begin) + q_len * (q_len + 1) // 2
