"""fp64 CPU oracle for causal GQA attention with RoPE -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg
of ``bench.py`` may import this package.  The library path (``global_causal_gqa_gb300``)
never imports it, and the two share no code: the oracle is plain C (``gqa_oracle.c``)
compiled here with gcc, plus a dense numpy twin (``twin.py``) used to cross-check it
on tiny inputs.

What each function follows is cited in the C source, by page and section.  Every
function is pinned by ``tests/test_oracle_*.py`` against values the pages print (the
worked attention example, the YaRN boundaries and amplitude), closed forms, library
routines (torch SDPA, numpy complex rotation) and invariants.  Nothing here is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS = {}


def lib_path(plant: int = 0) -> str:
    name = "libgqa_oracle.so" if plant == 0 else f"libgqa_oracle_plant{plant}.so"
    return os.path.join(_BUILD, name)


def build(plant: int = 0, force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, -O2, IEEE semantics: no -ffast-math)."""
    out = lib_path(plant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    fd, tmp = tempfile.mkstemp(dir=_BUILD, suffix=".so")
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", f"-DORC_PLANT={int(plant)}",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(plant: int = 0) -> ctypes.CDLL:
    with _LOCK:
        if plant in _LIBS:
            return _LIBS[plant]
        lib = ctypes.CDLL(build(plant))
        D, I, L, P = ctypes.c_double, ctypes.c_int, ctypes.c_long, ctypes.c_void_p
        lib.orc_inv_freq.argtypes = [P, I, D, D, D, D, D, D]
        lib.orc_inv_freq.restype = I
        lib.orc_yarn_amp.argtypes = [D]
        lib.orc_yarn_amp.restype = D
        lib.orc_yarn_boundary.argtypes = [I, D, D, D]
        lib.orc_yarn_boundary.restype = D
        lib.orc_rope_rotate.argtypes = [P, I, D, P, D]
        lib.orc_rope_rotate.restype = None
        lib.orc_attention.argtypes = [P, P, P, I, I, I, I, I, I, I, D, P, D, L, P, L,
                                      P, P, P, I]
        lib.orc_attention.restype = I
        lib.orc_append_slot.argtypes = [I, L, L]
        lib.orc_append_slot.restype = L
        lib.orc_retained.argtypes = [I, L, L]
        lib.orc_retained.restype = L
        lib.orc_logical_slot.argtypes = [I, L, L, L]
        lib.orc_logical_slot.restype = L
        lib.orc_decode_step.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, D,
                                        P, P, P, P, I]
        lib.orc_decode_step.restype = I
        lib.orc_attention_kv_shared.argtypes = [P, P, P, P, D, I, I, I, I, I, I, I, D, P, D,
                                                P, L, P, P, I]
        lib.orc_attention_kv_shared.restype = I
        lib.orc_decode_step_kv_shared.argtypes = [P, P, P, P, P, P, P, P, P, P, D, I, I, I, I,
                                                  D, P, P, P, P, I]
        lib.orc_decode_step_kv_shared.restype = I
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_double.restype = D
        lib.orc_allowed_pub.argtypes = [L, L, I]
        lib.orc_allowed_pub.restype = I
        lib.orc_kv_head_pub.argtypes = [I, I, I]
        lib.orc_kv_head_pub.restype = I
        lib.orc_rms_norm.argtypes = [P, L, I, P, D, P]
        lib.orc_rms_norm.restype = None
        lib.orc_plant.restype = I
        _LIBS[plant] = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(x) -> np.ndarray:
    """bfloat16 bits as a C-contiguous uint16 array (torch bf16 tensor or uint16 array)."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Oracle:
    """Thin ctypes front of the C oracle; `plant` selects a planted-mistake build."""

    def __init__(self, plant: int = 0):
        self.lib = _load(plant)
        self.plant = plant

    # -- frequencies ([PL3] §6.1, §6.3, §6.4) ---------------------------------------
    def inv_freq(self, d: int, base: float, yarn_factor: float = 1.0,
                 yarn_L0: float = 4096.0, beta_fast: float = 32.0, beta_slow: float = 1.0,
                 rotate_fraction: float = 1.0) -> np.ndarray:
        w = np.zeros(d // 2, dtype=np.float64)
        rc = self.lib.orc_inv_freq(_ptr(w), d, base, yarn_factor, yarn_L0, beta_fast,
                                   beta_slow, rotate_fraction)
        if rc != 0:
            raise ValueError("orc_inv_freq: bad argument")
        return w

    def inv_freq_spec(self, d: int, rope) -> np.ndarray:
        return self.inv_freq(d, rope.base, rope.yarn_factor, rope.yarn_L0, rope.beta_fast,
                             rope.beta_slow, rope.rotate_fraction)

    def yarn_amp(self, s: float) -> float:
        return self.lib.orc_yarn_amp(s)

    def yarn_boundary(self, d: int, base: float, L0: float, beta: float) -> float:
        return self.lib.orc_yarn_boundary(d, base, L0, beta)

    def rope_rotate(self, x: np.ndarray, pos: float, w: np.ndarray, amp: float) -> np.ndarray:
        y = np.array(x, dtype=np.float64, copy=True)
        w = np.ascontiguousarray(w, dtype=np.float64)
        self.lib.orc_rope_rotate(_ptr(y), y.shape[-1], float(pos), _ptr(w), float(amp))
        return y

    # -- RMSNorm ([PL3] §3.2, §4.3) --------------------------------------------------
    def rms_norm(self, x, gamma, eps: float = 1e-6) -> np.ndarray:
        """RMSNorm over the last axis of bf16 `x` (tensor or uint16 bits) in fp64;
        gamma: effective gain [n] (offset + weight) or None for no gain."""
        xb = _bits(x)
        n = xb.shape[-1]
        rows = xb.size // n
        out = np.zeros(xb.shape, dtype=np.float64)
        g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float64)
        self.lib.orc_rms_norm(_ptr(xb), rows, n, None if g is None else _ptr(g), float(eps),
                              _ptr(out))
        return out

    def allowed(self, qpos: int, kpos: int, window: int) -> bool:
        return bool(self.lib.orc_allowed_pub(qpos, kpos, window))

    def kv_head(self, h: int, Hq: int, Hkv: int) -> int:
        return self.lib.orc_kv_head_pub(h, Hq, Hkv)

    # -- attention ([PL3] §4.4, §4.5, §5.1) -----------------------------------------
    def attention(self, q, k, v, *, window: int, scale: float, w: np.ndarray, amp: float,
                  pos_shift: int = 0, rows: Optional[np.ndarray] = None,
                  want_weights: bool = False, nthreads: int = 0):
        """q [B,Hq,T,d], k/v [B,Hkv,S,d] (bf16).  Returns (o, lse[, weights]).

        With rows=None, o has shape [B,Hq,T,d] and lse [B,Hq,T]; with an int array of
        (b, h, t) triples, o is [n, d] and lse [n]."""
        qb, kb, vb = _bits(q), _bits(k), _bits(v)
        B, Hq, T, d = qb.shape
        _, Hkv, S, _ = kb.shape
        w = np.ascontiguousarray(w, dtype=np.float64)
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
            n = rows.shape[0]
        else:
            n = B * Hq * T
        o = np.zeros((n, d), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        wts = np.zeros((n, S), dtype=np.float64) if want_weights else None
        rc = self.lib.orc_attention(
            _ptr(qb), _ptr(kb), _ptr(vb), B, T, S, Hq, Hkv, d, int(window), float(scale),
            _ptr(w), float(amp), int(pos_shift),
            _ptr(rows) if rows is not None else None, n if rows is not None else 0,
            _ptr(o), _ptr(lse), _ptr(wts) if wts is not None else None, int(nthreads))
        if rc != 0:
            raise ValueError(f"orc_attention failed ({rc})")
        if rows is None:
            o = o.reshape(B, Hq, T, d)
            lse = lse.reshape(B, Hq, T)
            if wts is not None:
                wts = wts.reshape(B, Hq, T, S)
        return (o, lse, wts) if want_weights else (o, lse)

    # -- cache index model ([PL3] §4.4) ---------------------------------------------
    def append_slot(self, is_ring: int, count_before: int, cap: int) -> int:
        return self.lib.orc_append_slot(int(is_ring), int(count_before), int(cap))

    def retained(self, is_ring: int, count_after: int, cap: int) -> int:
        return self.lib.orc_retained(int(is_ring), int(count_after), int(cap))

    def logical_slot(self, is_ring: int, count_after: int, cap: int, t: int) -> int:
        return self.lib.orc_logical_slot(int(is_ring), int(count_after), int(cap), int(t))

    def decode_step(self, q, k_new, v_new, k_cache: Sequence, v_cache: Sequence,
                    cap: Sequence[int], count_before: Sequence[int],
                    is_ring: Sequence[int], w: Sequence[np.ndarray],
                    amp: Sequence[float], scale: float, nthreads: int = 0):
        """One decode step.  Returns (o [nseq,Hq,d], lse [nseq,Hq], slots, counts)."""
        qb, knb, vnb = _bits(q), _bits(k_new), _bits(v_new)
        nseq, Hq, d = qb.shape
        Hkv = knb.shape[1]
        kc = [_bits(t) for t in k_cache]
        vc = [_bits(t) for t in v_cache]
        kp = (ctypes.c_void_p * nseq)(*[c.ctypes.data for c in kc])
        vp = (ctypes.c_void_p * nseq)(*[c.ctypes.data for c in vc])
        ws = [np.ascontiguousarray(x, dtype=np.float64) for x in w]
        wp = (ctypes.c_void_p * nseq)(*[x.ctypes.data for x in ws])
        capa = np.asarray(cap, dtype=np.int64)
        cnt = np.asarray(count_before, dtype=np.int64)
        ring = np.asarray(is_ring, dtype=np.int32)
        ampa = np.asarray(amp, dtype=np.float64)
        o = np.zeros((nseq, Hq, d), dtype=np.float64)
        lse = np.zeros((nseq, Hq), dtype=np.float64)
        slots = np.zeros(nseq, dtype=np.int64)
        after = np.zeros(nseq, dtype=np.int64)
        rc = self.lib.orc_decode_step(
            _ptr(qb), _ptr(knb), _ptr(vnb), ctypes.cast(kp, ctypes.c_void_p),
            ctypes.cast(vp, ctypes.c_void_p), _ptr(capa), _ptr(cnt), _ptr(ring),
            ctypes.cast(wp, ctypes.c_void_p), _ptr(ampa), nseq, Hq, Hkv, d, float(scale),
            _ptr(o), _ptr(lse), _ptr(slots), _ptr(after), int(nthreads))
        if rc != 0:
            raise ValueError(f"orc_decode_step failed ({rc})")
        return o, lse, slots, after


    # -- shared K/V projection (Gemma 4 global layers, [PL3] §5.2 and §8) ----------------
    @staticmethod
    def _gain(g):
        return None if g is None else np.ascontiguousarray(g, dtype=np.float64)

    def attention_kv_shared(self, q, z, *, q_gamma, k_gamma, eps: float, window: int,
                            scale: float, w: np.ndarray, amp: float,
                            rows: Optional[np.ndarray] = None, nthreads: int = 0):
        """attention_k_eq_v: q [B,Hq,T,d] (before its norm) and the shared projection
        output z [B,Hkv,S,d] (bf16).  Q' = RoPE(N_{q_gamma}(q)), K' = RoPE(N_{k_gamma}(z)),
        V = N_1(z).  Gains None mean 1.  Returns (o, lse) shaped as attention()."""
        qb, zb = _bits(q), _bits(z)
        B, Hq, T, d = qb.shape
        _, Hkv, S, _ = zb.shape
        w = np.ascontiguousarray(w, dtype=np.float64)
        gq, gk = self._gain(q_gamma), self._gain(k_gamma)
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
            n = rows.shape[0]
        else:
            n = B * Hq * T
        o = np.zeros((n, d), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        rc = self.lib.orc_attention_kv_shared(
            _ptr(qb), _ptr(zb), None if gq is None else _ptr(gq),
            None if gk is None else _ptr(gk), float(eps), B, T, S, Hq, Hkv, d, int(window),
            float(scale), _ptr(w), float(amp), _ptr(rows) if rows is not None else None,
            n if rows is not None else 0, _ptr(o), _ptr(lse), int(nthreads))
        if rc != 0:
            raise ValueError(f"orc_attention_kv_shared failed ({rc})")
        if rows is None:
            o = o.reshape(B, Hq, T, d)
            lse = lse.reshape(B, Hq, T)
        return o, lse

    def decode_step_kv_shared(self, q, z_new, z_cache: Sequence, cap: Sequence[int],
                              count_before: Sequence[int], is_ring: Sequence[int],
                              w: Sequence[np.ndarray], amp: Sequence[float], *, q_gamma,
                              k_gamma, eps: float, scale: float, nthreads: int = 0):
        """One decode step of a shared-projection layer over caches of projection outputs
        Z.  Returns (o [nseq,Hq,d], lse [nseq,Hq], slots, counts)."""
        qb, znb = _bits(q), _bits(z_new)
        nseq, Hq, d = qb.shape
        Hkv = znb.shape[1]
        zc = [_bits(t) for t in z_cache]
        zp = (ctypes.c_void_p * nseq)(*[c.ctypes.data for c in zc])
        ws = [np.ascontiguousarray(x, dtype=np.float64) for x in w]
        wp = (ctypes.c_void_p * nseq)(*[x.ctypes.data for x in ws])
        capa = np.asarray(cap, dtype=np.int64)
        cnt = np.asarray(count_before, dtype=np.int64)
        ring = np.asarray(is_ring, dtype=np.int32)
        ampa = np.asarray(amp, dtype=np.float64)
        gq, gk = self._gain(q_gamma), self._gain(k_gamma)
        o = np.zeros((nseq, Hq, d), dtype=np.float64)
        lse = np.zeros((nseq, Hq), dtype=np.float64)
        slots = np.zeros(nseq, dtype=np.int64)
        after = np.zeros(nseq, dtype=np.int64)
        rc = self.lib.orc_decode_step_kv_shared(
            _ptr(qb), _ptr(znb), ctypes.cast(zp, ctypes.c_void_p), _ptr(capa), _ptr(cnt),
            _ptr(ring), ctypes.cast(wp, ctypes.c_void_p), _ptr(ampa),
            None if gq is None else _ptr(gq), None if gk is None else _ptr(gk), float(eps),
            nseq, Hq, Hkv, d, float(scale), _ptr(o), _ptr(lse), _ptr(slots), _ptr(after),
            int(nthreads))
        if rc != 0:
            raise ValueError(f"orc_decode_step_kv_shared failed ({rc})")
        return o, lse, slots, after


_DEFAULT = None


def default() -> Oracle:
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle(0)
    return _DEFAULT
