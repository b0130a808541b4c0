"""Seeded synthetic workloads for the attention hot path.

This module is the one place both sides of a parity check get their inputs from:
the CUDA path (through the C-ABI binding) and the fp64 oracle.  It holds shapes,
seeds and random-number draws only -- none of the attention, RoPE or cache-index
arithmetic lives here.

Every tensor is drawn with a torch CPU ``Generator`` seeded per (workload, tensor),
as float32 ~ N(0, 1) and rounded once to bfloat16 (round-to-nearest-even).  The same
bfloat16 bits go to the GPU and to the oracle.

Shapes follow the workloads the pages describe:
  * PLaMo 3 31B attention: 64 query heads, 8 KV heads, head dim 128, window 2048
    (self + previous 2047), RoPE base 1e4 local / 1e6 global with YaRN on the global
    layers ("PLaMo 3アーキテクチャ徹底解析", §2.1 table, §4.2, §5.1, §6.2-§6.3).
  * Gemma 4: local layers with head dim 256 and window 1024, global layers with head
    dim 512, 2 KV heads and partial (p = 0.25) RoPE (same page §6.4; the qiita.com
    Gemma-4-26B-A4B explainer, Attention block section: 16 query heads).
"""
from .configs import (  # noqa: F401
    PrefillLayer,
    PrefillWorkload,
    DecodeWorkload,
    DecodeModelWorkload,
    RopeSpec,
    WORKLOADS,
    get_workload,
)
from .gen import (  # noqa: F401
    randn_bf16,
    prefill_inputs,
    decode_inputs,
    bf16_bits,
    norm_gains,
)
