"""Seeded synthetic workloads shared by the CUDA path's tests/bench and the CPU oracle."""
from .configs import CONFIGS, SMALL, Config, config
from .gen import (Workload, make_workload, encode, reverse_interleaved, contiguous_table,
                  shuffled_table, fill_stale)

__all__ = ["CONFIGS", "SMALL", "Config", "config", "Workload", "make_workload", "encode",
           "reverse_interleaved", "contiguous_table", "shuffled_table", "fill_stale"]
