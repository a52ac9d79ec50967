"""CPU float64 oracle for sequence-partitioned causal attention.

Test infrastructure: imported only by the tests, the package smoke check and
the benchmark's CPU-baseline leg.  Never by the product path."""
from .seqattn_oracle import *  # noqa: F401,F403
