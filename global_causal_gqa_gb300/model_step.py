"""Decode step over every attention layer of a hybrid local/global decoder.

"PLaMo 3アーキテクチャ徹底解析" §2.3 and §4.4: in a decode step each layer appends the new
token's K and V to its cache and attends over it; local layers keep a ring of the newest
W tokens, global layers a linear cache, in a fixed period (PLaMo 3: 7 local, then 1
global).  `LayerStack` drives that step through the C ABI: per layer one gqa_kv_append
and one gqa_attn_decode on a stream, with every layer's descriptor array in one device
buffer so that a whole step can be replayed from the same cache state (one copy restores
every layer's counts).  The step can be captured once in a CUDA graph and replayed.

Argument marshalling and launch order only: every step of the computation runs in the
library's kernels.  The caller owns the caches, query and new-token tensors, outputs and
RoPE tables.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Sequence

import numpy as np

from . import (KV_DESC_DTYPE, gqa_attn_decode, gqa_decode_workspace_bytes, gqa_kv_append,
               make_kv_descs)


@dataclass
class Layer:
    """One attention layer's caller-owned device tensors for a batch of nseq sequences."""
    k_cache: object        # [nseq, Hkv, cap, d] bf16
    v_cache: object        # [nseq, Hkv, cap, d] bf16
    q: object              # [nseq, Hq, d] bf16, the new query token
    k_new: object          # [nseq, Hkv, d] bf16, the new token's key (before RoPE)
    v_new: object          # [nseq, Hkv, d] bf16
    o: object              # [nseq, Hq, d] bf16, the attention output
    table: object          # RoPE table of the layer type, table_len positions
    table_len: int
    is_ring: bool          # local layer (ring of cap = W) or global (linear)
    count_before: Sequence[int]   # per sequence: tokens held (linear) / ever appended (ring)


class LayerStack:
    """Every layer's descriptors in one device buffer; `step` issues the decode step."""

    def __init__(self, layers: List[Layer], Hq: int, Hkv: int, d: int, scale: float,
                 max_len: int):
        import torch
        self.layers = layers
        self.Hq, self.Hkv, self.d, self.scale, self.max_len = Hq, Hkv, d, scale, max_len
        self.nseq = layers[0].q.shape[0]
        rows = []
        for L in layers:
            nseq, cap = L.k_cache.shape[0], L.k_cache.shape[2]
            a = make_kv_descs([L.k_cache[i] for i in range(nseq)],
                              [L.v_cache[i] for i in range(nseq)], [L.table] * nseq,
                              [cap] * nseq, list(L.count_before), [int(L.is_ring)] * nseq,
                              [L.table_len] * nseq)
            rows.append(torch.from_numpy(a.view(np.uint8).copy()))
        dev = layers[0].q.device
        self.descs0 = torch.stack(rows).to(dev)   # [layers, nseq * sizeof(gqa_kv_desc)]
        self.descs = self.descs0.clone()
        # a ring layer holds at most its capacity; a linear one at most max_len tokens
        self.max_lens = [L.k_cache.shape[2] if L.is_ring else max_len for L in layers]
        self.wsb = max(gqa_decode_workspace_bytes(self.nseq, Hq, Hkv, d, n)
                       for n in set(self.max_lens))
        self.ws = torch.empty(self.wsb, dtype=torch.uint8, device=dev)
        self.graph = None

    def restore(self):
        """Puts every layer's counts back to the state the stack was built with."""
        self.descs.copy_(self.descs0, non_blocking=True)

    def step(self, stream=None, restore: bool = True):
        """One decode step: (restore the counts,) then append + decode per layer."""
        if restore:
            self.restore()
        for l, L in enumerate(self.layers):
            gqa_kv_append(self.descs[l], self.nseq, L.k_new, L.v_new, self.Hkv, self.d, None,
                          stream)
            gqa_attn_decode(L.q, self.descs[l], self.nseq, self.Hq, self.Hkv, self.d,
                            self.scale, self.max_lens[l], L.o, None, self.ws, self.wsb, stream)

    def capture(self):
        """Captures `step` (with the count restore) in a CUDA graph on a side stream."""
        import torch
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                self.step()
        torch.cuda.current_stream().wait_stream(side)
        self.graph = graph
        return graph

    def counts(self, layer: int) -> np.ndarray:
        a = self.descs[layer].cpu().numpy().view(KV_DESC_DTYPE)
        return a["count"].astype(np.int64)
