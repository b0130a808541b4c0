"""Python binding of libgqa_attn.so -- causal GQA attention with RoPE for GB300 (sm_103a).

Argument marshalling only: every function here forwards to the C entry point of the same
name declared in ``include/gqa_attn.h`` (tensors become device pointers, streams become
``cudaStream_t`` handles).  All computation happens in the library's CUDA kernels; there
is no fallback.  If the library has not been built, `lib()` raises.  Build it with
``python -m global_causal_gqa_gb300.build`` (or ``__graft_entry__.build()``).

Non-zero status codes raise `GQAError` unless ``check=False`` is passed.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import numpy as np

from .build import LIB as LIB_PATH

__all__ = [
    "GQAError", "lib", "KV_DESC_DTYPE", "make_kv_descs",
    "gqa_rope_inv_freq", "gqa_yarn_amplitude", "gqa_rope_table_bytes", "gqa_rope_table_build",
    "gqa_rope_apply", "gqa_prefill_workspace_bytes", "gqa_attn_prefill", "gqa_kv_append",
    "gqa_decode_workspace_bytes", "gqa_attn_decode", "gqa_attn_decode_static",
    "gqa_qk_norm_rope", "gqa_qk_norm_append", "gqa_prefill_gather", "gqa_kv_append_chunk",
    "gqa_get_device_status", "gqa_get_device_diag", "gqa_watchdog_selftest",
    "gqa_status_string", "gqa_last_error_string", "gqa_device_check",
]

GQA_OK = 0
STATUS_NAMES = {
    0: "GQA_OK", -1: "GQA_ERR_INVALID_ARG", -2: "GQA_ERR_UNSUPPORTED", -3: "GQA_ERR_ALIGNMENT",
    -4: "GQA_ERR_CAPACITY", -5: "GQA_ERR_CUDA", -6: "GQA_ERR_DEVICE_TIMEOUT",
    -7: "GQA_ERR_WORKSPACE", -8: "GQA_ERR_RANGE", -9: "GQA_ERR_DEVICE_BOUNDS",
}


class GQAError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        detail = gqa_status_string(status)
        if status == -5:
            detail += ": " + gqa_last_error_string()
        super().__init__(f"{func}: {STATUS_NAMES.get(status, status)} ({detail})")


# struct gqa_kv_desc { void *k; void *v; const float *rope; int32 cap, count, is_ring, rope_len; }
KV_DESC_DTYPE = np.dtype([("k", "<u8"), ("v", "<u8"), ("rope", "<u8"), ("cap", "<i4"),
                          ("count", "<i4"), ("is_ring", "<i4"), ("rope_len", "<i4")])
assert KV_DESC_DTYPE.itemsize == 40

_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libgqa_attn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -m global_causal_gqa_gb300.build); there is no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        P, I, D, Z, F = (ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_size_t,
                         ctypes.c_float)
        sig = {
            "gqa_rope_inv_freq": ([P, I, D, D, D, D, D, D], I),
            "gqa_yarn_amplitude": ([D], D),
            "gqa_rope_table_bytes": ([I, I], Z),
            "gqa_rope_table_build": ([P, P, I, D, I, P], I),
            "gqa_rope_apply": ([P, P, I, I, I, I, I, P, I, P], I),
            "gqa_prefill_workspace_bytes": ([I, I, I, I], Z),
            "gqa_attn_prefill": ([P, P, P, P, P, I, I, I, I, I, I, I, F, P, I, I, P, Z, P], I),
            "gqa_kv_append": ([P, I, P, P, I, I, P, P], I),
            "gqa_decode_workspace_bytes": ([I, I, I, I, I], Z),
            "gqa_attn_decode": ([P, P, I, I, I, I, F, I, P, P, P, Z, P], I),
            "gqa_attn_decode_static": ([P, P, I, I, I, I, F, I, P, P, P], I),
            "gqa_prefill_gather": ([P, P, P, I, I, I, P, P, I, P, I, P], I),
            "gqa_kv_append_chunk": ([P, I, P, P, I, I, I, P], I),
            "gqa_qk_norm_rope": ([P, P, P, P, P, I, I, I, I, I, I, P, P, F, P, I, P], I),
            "gqa_qk_norm_append": ([P, I, P, P, P, I, I, I, P, P, F, I, P, P, P], I),
            "gqa_qk_norm_rope_kv_shared": ([P, P, P, P, P, I, I, I, I, I, I, P, P, F, P, I, P],
                                           I),
            "gqa_kv_shared_append": ([P, I, P, P, I, I, I, P, F, P, P, P], I),
            "gqa_attn_decode_kv_shared": ([P, P, I, I, I, I, F, P, I, P, P, P, Z, P], I),
            "gqa_get_device_status": ([P], I),
            "gqa_get_device_diag": ([P, P, I], I),
            "gqa_watchdog_selftest": ([ctypes.c_int64, P], I),
            "gqa_status_string": ([I], ctypes.c_char_p),
            "gqa_last_error_string": ([], ctypes.c_char_p),
            "gqa_device_check": ([], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
        return L


def _ptr(x) -> Optional[int]:
    """Device/host address of a tensor or array; None/0 -> NULL; ints pass through."""
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _check(name: str, status: int, check: bool) -> int:
    if check and status != GQA_OK:
        raise GQAError(name, status)
    return status


# ---- RoPE ---------------------------------------------------------------------------------

def gqa_rope_inv_freq(d: int, base: float, yarn_factor: float = 1.0, yarn_L0: float = 4096.0,
                      beta_fast: float = 32.0, beta_slow: float = 1.0,
                      rotate_fraction: float = 1.0) -> np.ndarray:
    out = np.zeros(d // 2 if d > 0 else 0, dtype=np.float64)
    st = lib().gqa_rope_inv_freq(out.ctypes.data if out.size else None, d, base, yarn_factor,
                                 yarn_L0, beta_fast, beta_slow, rotate_fraction)
    _check("gqa_rope_inv_freq", st, True)
    return out


def gqa_yarn_amplitude(s: float) -> float:
    return lib().gqa_yarn_amplitude(s)


def gqa_rope_table_bytes(d: int, max_pos: int) -> int:
    return lib().gqa_rope_table_bytes(d, max_pos)


def gqa_rope_table_build(table, inv_freq: np.ndarray, d: int, amp: float, max_pos: int,
                         stream=None, check: bool = True) -> int:
    w = np.ascontiguousarray(inv_freq, dtype=np.float64)
    st = lib().gqa_rope_table_build(_ptr(table), w.ctypes.data, d, amp, max_pos,
                                    _stream(stream))
    return _check("gqa_rope_table_build", st, check)


def gqa_rope_apply(x, y, B: int, H: int, T: int, d: int, pos0: int, table, table_len: int,
                   stream=None, check: bool = True) -> int:
    st = lib().gqa_rope_apply(_ptr(x), _ptr(y), B, H, T, d, pos0, _ptr(table), table_len,
                              _stream(stream))
    return _check("gqa_rope_apply", st, check)


# ---- prefill ------------------------------------------------------------------------------

def gqa_prefill_workspace_bytes(B: int, Hkv: int, S: int, d: int) -> int:
    return lib().gqa_prefill_workspace_bytes(B, Hkv, S, d)


def gqa_attn_prefill(q, k, v, o, lse, B: int, T: int, S: int, Hq: int, Hkv: int, d: int,
                     window: int, scale: float, table, table_len: int, k_is_rotated: int,
                     workspace, workspace_bytes: int, stream=None, check: bool = True) -> int:
    st = lib().gqa_attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, T, S, Hq,
                                Hkv, d, window, scale, _ptr(table), table_len, k_is_rotated,
                                _ptr(workspace), workspace_bytes, _stream(stream))
    return _check("gqa_attn_prefill", st, check)


# ---- KV cache and decode --------------------------------------------------------------------

def make_kv_descs(k_caches: Sequence, v_caches: Sequence, ropes: Sequence, caps: Sequence[int],
                  counts: Sequence[int], is_ring: Sequence[int],
                  rope_lens: Sequence[int]) -> np.ndarray:
    """Packs per-sequence cache descriptors (struct gqa_kv_desc) into a host array; copy
    its bytes to device memory (e.g. torch.from_numpy(a.view(np.uint8)).cuda())."""
    n = len(k_caches)
    a = np.zeros(n, dtype=KV_DESC_DTYPE)
    for i in range(n):
        a[i] = (_ptr(k_caches[i]), _ptr(v_caches[i]), _ptr(ropes[i]), caps[i], counts[i],
                is_ring[i], rope_lens[i])
    return a


def gqa_kv_append(descs, nseq: int, k_new, v_new, Hkv: int, d: int, slots_out=None,
                  stream=None, check: bool = True) -> int:
    st = lib().gqa_kv_append(_ptr(descs), nseq, _ptr(k_new), _ptr(v_new), Hkv, d,
                             _ptr(slots_out), _stream(stream))
    return _check("gqa_kv_append", st, check)


def gqa_decode_workspace_bytes(nseq: int, Hq: int, Hkv: int, d: int, max_len: int) -> int:
    return lib().gqa_decode_workspace_bytes(nseq, Hq, Hkv, d, max_len)


def gqa_attn_decode(q, descs, nseq: int, Hq: int, Hkv: int, d: int, scale: float,
                    max_len: int, o, lse, workspace, workspace_bytes: int, stream=None,
                    check: bool = True) -> int:
    st = lib().gqa_attn_decode(_ptr(q), _ptr(descs), nseq, Hq, Hkv, d, scale, max_len, _ptr(o),
                               _ptr(lse), _ptr(workspace), workspace_bytes, _stream(stream))
    return _check("gqa_attn_decode", st, check)


def gqa_attn_decode_static(q, descs, nseq: int, Hq: int, Hkv: int, d: int, scale: float,
                           max_len: int, o, lse, stream=None, check: bool = True) -> int:
    """gqa_attn_decode without a workspace argument: for callers that cannot allocate
    device memory; the partials use a fixed 16 MiB array inside the library (shared by all
    calls, so overlapping calls race)."""
    st = lib().gqa_attn_decode_static(_ptr(q), _ptr(descs), nseq, Hq, Hkv, d, scale, max_len,
                                      _ptr(o), _ptr(lse), _stream(stream))
    return _check("gqa_attn_decode_static", st, check)


# ---- chunked prefill over a cache -------------------------------------------------------------

def gqa_prefill_gather(desc, k_new, v_new, T: int, Hkv: int, d: int, k_out, v_out, S: int,
                       table, table_len: int, stream=None, check: bool = True) -> int:
    st = lib().gqa_prefill_gather(_ptr(desc), _ptr(k_new), _ptr(v_new), T, Hkv, d, _ptr(k_out),
                                  _ptr(v_out), S, _ptr(table), table_len, _stream(stream))
    return _check("gqa_prefill_gather", st, check)


def gqa_kv_append_chunk(descs, nseq: int, k_new, v_new, T: int, Hkv: int, d: int, stream=None,
                        check: bool = True) -> int:
    st = lib().gqa_kv_append_chunk(_ptr(descs), nseq, _ptr(k_new), _ptr(v_new), T, Hkv, d,
                                   _stream(stream))
    return _check("gqa_kv_append_chunk", st, check)


# ---- Q/K normalisation ------------------------------------------------------------------------

def gqa_qk_norm_rope(q, k, q_out, k_out, k_rot, B: int, Hq: int, Hkv: int, T: int, d: int,
                     pos0: int, q_gamma, k_gamma, eps: float, table, table_len: int,
                     stream=None, check: bool = True) -> int:
    st = lib().gqa_qk_norm_rope(_ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), _ptr(k_rot), B, Hq,
                                Hkv, T, d, pos0, _ptr(q_gamma), _ptr(k_gamma), eps, _ptr(table),
                                table_len, _stream(stream))
    return _check("gqa_qk_norm_rope", st, check)


def gqa_qk_norm_append(descs, nseq: int, q, k_new, v_new, Hq: int, Hkv: int, d: int, q_gamma,
                       k_gamma, eps: float, v_norm: int, q_out, slots_out=None, stream=None,
                       check: bool = True) -> int:
    st = lib().gqa_qk_norm_append(_ptr(descs), nseq, _ptr(q), _ptr(k_new), _ptr(v_new), Hq, Hkv,
                                  d, _ptr(q_gamma), _ptr(k_gamma), eps, v_norm, _ptr(q_out),
                                  _ptr(slots_out), _stream(stream))
    return _check("gqa_qk_norm_append", st, check)


# ---- shared K/V projection (Gemma 4 global layers) ---------------------------------------

def gqa_qk_norm_rope_kv_shared(q, z, q_out, v_out, k_rot, B: int, Hq: int, Hkv: int, T: int,
                               d: int, pos0: int, q_gamma, k_gamma, eps: float, table,
                               table_len: int, stream=None, check: bool = True) -> int:
    st = lib().gqa_qk_norm_rope_kv_shared(_ptr(q), _ptr(z), _ptr(q_out), _ptr(v_out),
                                          _ptr(k_rot), B, Hq, Hkv, T, d, pos0, _ptr(q_gamma),
                                          _ptr(k_gamma), eps, _ptr(table), table_len,
                                          _stream(stream))
    return _check("gqa_qk_norm_rope_kv_shared", st, check)


def gqa_kv_shared_append(descs, nseq: int, q, z_new, Hq: int, Hkv: int, d: int, q_gamma,
                         eps: float, q_out, slots_out=None, stream=None,
                         check: bool = True) -> int:
    st = lib().gqa_kv_shared_append(_ptr(descs), nseq, _ptr(q), _ptr(z_new), Hq, Hkv, d,
                                    _ptr(q_gamma), eps, _ptr(q_out), _ptr(slots_out),
                                    _stream(stream))
    return _check("gqa_kv_shared_append", st, check)


def gqa_attn_decode_kv_shared(q, descs, nseq: int, Hq: int, Hkv: int, d: int, scale: float,
                              k_gamma, max_len: int, o, lse, workspace, workspace_bytes: int,
                              stream=None, check: bool = True) -> int:
    st = lib().gqa_attn_decode_kv_shared(_ptr(q), _ptr(descs), nseq, Hq, Hkv, d, scale,
                                         _ptr(k_gamma), max_len, _ptr(o), _ptr(lse),
                                         _ptr(workspace), workspace_bytes, _stream(stream))
    return _check("gqa_attn_decode_kv_shared", st, check)


# ---- status ---------------------------------------------------------------------------------

def gqa_get_device_status(stream=None) -> int:
    return lib().gqa_get_device_status(_stream(stream))


def gqa_get_device_diag(stream=None) -> list:
    """Diagnostic codes of the device-side waits that expired (first overall, then the
    first of each kernel role 0-3; 0 where none); cleared by the read."""
    v = (ctypes.c_int32 * 5)()
    _check("gqa_get_device_diag", lib().gqa_get_device_diag(_stream(stream), v, 5), True)
    return list(v)


def gqa_watchdog_selftest(limit_ns: int, stream=None, check: bool = True) -> int:
    """Enqueues a wait that nothing completes, bounded by limit_ns; the device records
    GQA_ERR_DEVICE_TIMEOUT, read back by gqa_get_device_status."""
    st = lib().gqa_watchdog_selftest(int(limit_ns), _stream(stream))
    return _check("gqa_watchdog_selftest", st, check)


def gqa_status_string(status: int) -> str:
    return lib().gqa_status_string(status).decode()


def gqa_last_error_string() -> str:
    return lib().gqa_last_error_string().decode()


def gqa_device_check() -> int:
    return lib().gqa_device_check()
