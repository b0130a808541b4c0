"""Workload definitions: shapes, masks, RoPE settings and seeds.

Plain data only.  The RoPE settings are the arguments a caller gives the library
(base, YaRN factor and its constants, partial-rotation fraction, amplitude); turning
them into frequencies is the library's and the oracle's job, not this module's.

Readings taken where the workload text is loose (each is listed with its reason in
the design notes):
  * Global-layer YaRN: base 1e6, factor s = 8, L0 = 4096, beta_fast = 32,
    beta_slow = 1 (constants of "PLaMo 3アーキテクチャ徹底解析" §6.3), and the
    "common amplitude factor 1.2 on the logits" taken literally: cos and sin are each
    multiplied by sqrt(1.2), so every logit is multiplied by exactly 1.2.
  * Gemma-4 global layer: partial RoPE, 64 of 256 pairs rotate (same page §6.4),
    base 1e6; scale 1/sqrt(d) because the inputs are raw N(0, 1), not gain-normalised.
  * Decode global caches: lengths S ~ U{8192..65536} inclusive, counted after the new
    token is appended (query position S - 1).  Local rings: capacity W = 2048 holding
    2047 old tokens + the new one, logical positions 0..2047; the number of tokens
    ever appended is drawn so the ring's write slot lands anywhere (wrap-around).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Tuple


@dataclass(frozen=True)
class RopeSpec:
    base: float
    yarn_factor: float = 1.0          # 1.0 = no YaRN
    yarn_L0: float = 4096.0
    beta_fast: float = 32.0
    beta_slow: float = 1.0
    rotate_fraction: float = 1.0      # 1.0 = all pairs rotate; 0.25 = p-RoPE
    amp: float = 1.0                  # multiplies both cos and sin


@dataclass(frozen=True)
class PrefillLayer:
    B: int
    T: int
    S: int
    Hq: int
    Hkv: int
    d: int
    window: int                        # <= 0: full causal
    rope: RopeSpec
    scale: float
    seed: int

    @property
    def label(self) -> str:
        kind = f"W{self.window}" if self.window > 0 else "causal"
        return f"B{self.B}_T{self.T}_S{self.S}_Hq{self.Hq}_Hkv{self.Hkv}_d{self.d}_{kind}"


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    layers: Tuple[PrefillLayer, ...]


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    n_global: int
    n_local: int
    Hq: int
    Hkv: int
    d: int
    global_len_range: Tuple[int, int]  # inclusive, after append
    window: int                        # ring capacity for local sequences
    rope_global: RopeSpec
    rope_local: RopeSpec
    scale: float
    seed: int
    # K and V from one shared projection (Gemma 4 global layers, attention_k_eq_v): the
    # caches hold Zn = N_1(Z) only; keys RoPE(gamma_k Zn), values Zn
    kv_shared: bool = False

    @property
    def nseq(self) -> int:
        return self.n_global + self.n_local


_PLAMO_D = 128
_YARN8 = RopeSpec(base=1e6, yarn_factor=8.0, yarn_L0=4096.0, beta_fast=32.0,
                  beta_slow=1.0, rotate_fraction=1.0, amp=math.sqrt(1.2))
_LOCAL = RopeSpec(base=1e4)

TINY_W64 = PrefillWorkload("tiny_w64", (
    PrefillLayer(B=1, T=256, S=256, Hq=4, Hkv=1, d=128, window=64, rope=_LOCAL,
                 scale=1 / math.sqrt(128), seed=1001),))
TINY_CAUSAL = PrefillWorkload("tiny_causal", (
    PrefillLayer(B=1, T=256, S=256, Hq=4, Hkv=1, d=128, window=0, rope=_LOCAL,
                 scale=1 / math.sqrt(128), seed=1001),))

PLAMO3_LOCAL_PREFILL = PrefillWorkload("plamo3_local_prefill", (
    PrefillLayer(B=2, T=8192, S=8192, Hq=64, Hkv=8, d=_PLAMO_D, window=2048,
                 rope=_LOCAL, scale=1 / math.sqrt(128), seed=2002),))

PLAMO3_GLOBAL_PREFILL = PrefillWorkload("plamo3_global_prefill", (
    PrefillLayer(B=1, T=32768, S=32768, Hq=64, Hkv=8, d=_PLAMO_D, window=0,
                 rope=_YARN8, scale=1 / math.sqrt(128), seed=3003),))

PLAMO3_DECODE = DecodeWorkload(
    "plamo3_decode_batch32", n_global=16, n_local=16, Hq=64, Hkv=8, d=_PLAMO_D,
    global_len_range=(8192, 65536), window=2048, rope_global=_YARN8,
    rope_local=_LOCAL, scale=1 / math.sqrt(128), seed=4004)

_G4_LOCAL = RopeSpec(base=1e4)
_G4_GLOBAL = RopeSpec(base=1e6, rotate_fraction=0.25)
GEMMA4_PERIOD = PrefillWorkload("gemma4_period_6layer", tuple(
    [PrefillLayer(B=1, T=16384, S=16384, Hq=16, Hkv=8, d=256, window=1024,
                  rope=_G4_LOCAL, scale=1 / math.sqrt(256), seed=5005 + i)
     for i in range(5)] +
    [PrefillLayer(B=1, T=16384, S=16384, Hq=16, Hkv=2, d=512, window=0,
                  rope=_G4_GLOBAL, scale=1 / math.sqrt(512), seed=5010)]))

# Gemma-4-shaped decode batches (one head shape per call): the global layer's d = 512,
# 2 KV heads and p-RoPE over linear caches, and the local layers' d = 256, 8 KV heads over
# rings of the 1024-token window.  Lengths as in the PLaMo decode batch.
GEMMA4_DECODE_GLOBAL = DecodeWorkload(
    "gemma4_decode_global", n_global=32, n_local=0, Hq=16, Hkv=2, d=512,
    global_len_range=(8192, 65536), window=1024, rope_global=_G4_GLOBAL,
    rope_local=_G4_LOCAL, scale=1 / math.sqrt(512), seed=6006)
# The global layer as Gemma 4 defines it (attention_k_eq_v, "PLaMo 3アーキテクチャ徹底解析"
# §5.2 and §8): one cache of Zn per sequence for both K and V, scale 1 with the gains
# carrying the logit scale; the same lengths as gemma4_decode_global (same seed).
GEMMA4_DECODE_GLOBAL_KV_SHARED = DecodeWorkload(
    "gemma4_decode_global_kv_shared", n_global=32, n_local=0, Hq=16, Hkv=2, d=512,
    global_len_range=(8192, 65536), window=1024, rope_global=_G4_GLOBAL,
    rope_local=_G4_LOCAL, scale=1.0, seed=6006, kv_shared=True)
GEMMA4_DECODE_LOCAL = DecodeWorkload(
    "gemma4_decode_local", n_global=0, n_local=32, Hq=16, Hkv=8, d=256,
    global_len_range=(1024, 1024), window=1024, rope_global=_G4_GLOBAL,
    rope_local=_G4_LOCAL, scale=1 / math.sqrt(256), seed=7007)

@dataclass(frozen=True)
class DecodeModelWorkload:
    """One decode step through a whole hybrid decoder's attention: `layers` layers in
    periods of `period` (the last layer of each period global with a linear cache of N
    tokens, the others local with a ring of W), `nseq` sequences at context N."""
    name: str
    layers: int
    period: int
    nseq: int
    N: int
    W: int
    Hq: int
    Hkv: int
    d: int
    rope_global: RopeSpec
    rope_local: RopeSpec
    scale: float
    seed: int


# PLaMo 3 31B: 64 layers, 7 sliding-window layers then 1 global in each period of 8, at the
# context N = 4096 of the pages' byte-count table (576 MiB of K/V reads per token).
PLAMO3_DECODE_64LAYER = DecodeModelWorkload(
    "plamo3_decode_64layer", layers=64, period=8, nseq=32, N=4096, W=2048, Hq=64, Hkv=8,
    d=_PLAMO_D, rope_global=_YARN8, rope_local=_LOCAL, scale=1 / math.sqrt(128), seed=8008)

WORKLOADS = {w.name: w for w in (TINY_W64, TINY_CAUSAL, PLAMO3_LOCAL_PREFILL,
                                 PLAMO3_GLOBAL_PREFILL, PLAMO3_DECODE, GEMMA4_PERIOD,
                                 GEMMA4_DECODE_GLOBAL, GEMMA4_DECODE_GLOBAL_KV_SHARED,
                                 GEMMA4_DECODE_LOCAL,
                                 PLAMO3_DECODE_64LAYER)}


def get_workload(name: str):
    try:
        return WORKLOADS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}") from None


def scaled(layer: PrefillLayer, **kw) -> PrefillLayer:
    """A copy of `layer` with some fields replaced (for reduced-size parity cases)."""
    return replace(layer, **kw)
