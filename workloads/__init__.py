"""Seeded synthetic workloads shared by the CUDA path's tests/bench and the oracle."""
from .synth import (Config, Workload, make_workload, pack_bits, centroid_chain, CONFIGS,
                    TINY, LLAMA7B, LLAMA13B, OPT67B, BATCHED7B,
                    SMALL_F16, SMALL_BF16, SMALL_OPT, SMALL_BATCHED)
