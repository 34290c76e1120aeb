"""Workload sizes for the paged sparse-decode step.

Five named workloads, each with the sizes and value structure of one decode
scenario, plus reduced ("small") variants that keep the same structure at
sizes a float64 CPU check finishes in seconds while still spanning several
pages per split, several splits per (request, KV head) and a ragged tail.

Nothing here computes anything of the method; these are plain records.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Optional, Tuple


@dataclass(frozen=True)
class Config:
    cid: int                      # workload id (1..5; 0 for ad-hoc)
    name: str
    B: int                        # requests
    H_q: int                      # query heads
    H_kv: int                     # KV heads (H_q % H_kv == 0)
    D: int                        # head dim
    ps: int                       # page size (tokens per page); 1 = token-level
    dtype: str                    # "bf16" | "fp16"  (K, V, Q, meta, out)
    topk: int = 0                 # pages kept per (request, KV head), tail included
    w_avg: float = 1.0            # weight of the mean-relevance term
    w_peak: float = 0.25          # weight of the envelope (peak) term
    prefill: Optional[Tuple[int, ...]] = None   # per-request prefill lengths
    len_range: Optional[Tuple[int, int]] = None  # ragged prefill, U[lo, hi] integers
    decode_steps: int = 0         # decode steps with append (0 = one step over the prefill)
    num_blocks: Optional[int] = None  # physical blocks (token slots when ps == 1)
    table: str = "reverse"        # "reverse" | "shuffle" | "contiguous"
    structure: str = "iid"        # value recipe, see sa_synth.gen
    # token-level H2O
    budget: int = 0
    n_sink: int = 0
    grace: int = 0
    decay: float = 1.0
    scale: float = 0.0            # softmax scale; <= 0 means head_dim ** -0.5
    stale: str = "normal3"        # contents of unreferenced blocks / unwritten slots
    seed: int = -1                # -1: 1000 + cid

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def rng_seed(self) -> int:
        return self.seed if self.seed >= 0 else 1000 + self.cid

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


# The five workloads (sizes as stated by the scenario list of the step).
CONFIGS = {
    1: Config(cid=1, name="tiny_g4", B=1, H_q=4, H_kv=1, D=64, ps=16, dtype="bf16",
              topk=4, w_avg=1.0, w_peak=0.25, prefill=(256,), decode_steps=0,
              num_blocks=64, table="reverse", structure="page_unit_offset"),
    2: Config(cid=2, name="decode_loop_quest", B=1, H_q=32, H_kv=8, D=128, ps=16,
              dtype="fp16", topk=16, w_avg=0.0, w_peak=1.0, prefill=(1024,),
              decode_steps=64, num_blocks=69, table="reverse",
              structure="page_normal_offset"),
    3: Config(cid=3, name="batched_gqa_ragged", B=16, H_q=32, H_kv=8, D=128, ps=16,
              dtype="bf16", topk=64, w_avg=1.0, w_peak=0.25, len_range=(2048, 32768),
              decode_steps=0, table="shuffle", structure="hot_pages_corr"),
    4: Config(cid=4, name="token_h2o", B=8, H_q=32, H_kv=8, D=128, ps=1, dtype="bf16",
              prefill=(4096,) * 8, decode_steps=256, table="reverse", structure="iid",
              budget=512, n_sink=4, grace=16, decay=0.984375, scale=128 ** -0.5),
    5: Config(cid=5, name="long_context_gqa", B=4, H_q=64, H_kv=8, D=128, ps=16,
              dtype="bf16", topk=256, w_avg=1.0, w_peak=0.25, prefill=(131072,) * 4,
              decode_steps=32, num_blocks=40000, table="reverse",
              structure="hot_pages_qdir"),
}


# Reduced variants: same recipe, CPU-checkable sizes.
SMALL = {
    1: CONFIGS[1],
    2: CONFIGS[2].replace(name="decode_loop_quest_small", H_q=8, H_kv=2, prefill=(200,),
                          decode_steps=12, topk=4, num_blocks=None),
    3: CONFIGS[3].replace(name="batched_gqa_ragged_small", B=3, H_q=8, H_kv=2,
                          len_range=(40, 700), topk=8),
    4: CONFIGS[4].replace(name="token_h2o_small", B=2, H_q=8, H_kv=2, prefill=(300, 300),
                          decode_steps=20, budget=64, n_sink=4, grace=16),
    5: CONFIGS[5].replace(name="long_context_gqa_small", B=2, H_q=16, H_kv=2,
                          prefill=(3000, 3000), decode_steps=5, topk=32, num_blocks=500),
}


def config(cid: int, small: bool = False) -> Config:
    return (SMALL if small else CONFIGS)[cid]
