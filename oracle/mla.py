"""CPU oracle for one decode token of the hybrid's gated attention (MLA) layers.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests and
``__graft_entry__.smoke()`` may import it; the CUDA library and its binding
never do.  The arithmetic lives in ``mla_oracle.c`` (double precision, plain
loops, each function citing the passage it follows); this module only
marshals numpy arrays.

Layouts: q, k_new [N, H, dqk]; v_new, gate, out [N, H, dv];
k_cache [N, H, L_max, dqk]; v_cache [N, H, L_max, dv]; cache_len [N].
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libmla_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False, out_path: str | None = None, src: str | None = None) -> str:
    return _build(force=force, out_path=out_path or _LIB_PATH, src=src or SRC)


def load(path: str | None = None):
    """Load (building if needed) the MLA oracle library and declare its signatures."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        P, I, D, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_long
        lib.mla_oracle_rope.argtypes = [P, L, I, I, P, D]
        lib.mla_oracle_decode_step.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, D, D, I, P]
        lib.mla_oracle_round_bf16.argtypes = [P, L]
        for f in ("mla_oracle_rope", "mla_oracle_decode_step", "mla_oracle_round_bf16"):
            getattr(lib, f).restype = I
        if path is None:
            _lib = lib
        return lib


def _f64(a, shape=None, name="array"):
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and tuple(a.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(a.shape)}")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"MLA oracle {what}: invalid arguments (rc={rc})")


def round_bf16(x, lib=None):
    """Nearest bfloat16 values (ties to even) of x, as float64."""
    lib = lib or load()
    x = _f64(x, name="x").copy()
    _check(lib.mla_oracle_round_bf16(_ptr(x), x.size), "round_bf16")
    return x


def rope(x, pos, rope_dim, theta, lib=None):
    """Rotate-half RoPE of the first rope_dim entries of each row of x [..., d].
    pos: one position per row (broadcast from a scalar)."""
    lib = lib or load()
    x = _f64(x, name="x").copy()
    d = x.shape[-1]
    rows = x.size // d
    p = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.int64), (rows,)).astype(np.int64))
    if ctypes.sizeof(ctypes.c_long) != 8:
        raise RuntimeError("the oracle expects a 64-bit long")
    _check(lib.mla_oracle_rope(_ptr(x), rows, d, int(rope_dim), _ptr(p), float(theta)), "rope")
    return x


def decode_step(q, k_new, v_new, k_cache, v_cache, cache_len, scale, gate=None, rope_dim=0,
                theta=10000.0, cache_bf16=False, lib=None):
    """One decode token.  Returns (out [N, H, dv], k_cache', v_cache', cache_len'): the inputs
    are not modified; the returned caches and lengths are the updated copies."""
    lib = lib or load()
    q = _f64(q, name="q")
    N, H, dqk = q.shape
    k_new = _f64(k_new, (N, H, dqk), "k_new")
    v_new = _f64(v_new, name="v_new")
    dv = v_new.shape[-1]
    if v_new.shape != (N, H, dv):
        raise ValueError("v_new: expected [N, H, dv]")
    kc = _f64(k_cache, name="k_cache").copy()
    L_max = kc.shape[2]
    if kc.shape != (N, H, L_max, dqk):
        raise ValueError("k_cache: expected [N, H, L_max, dqk]")
    vc = _f64(v_cache, (N, H, L_max, dv), "v_cache").copy()
    gate = _f64(gate, (N, H, dv), "gate")
    lens = np.ascontiguousarray(np.asarray(cache_len, dtype=np.int32)).copy()
    if lens.shape != (N,):
        raise ValueError("cache_len: expected [N]")
    out = np.empty((N, H, dv))
    _check(lib.mla_oracle_decode_step(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(gate), _ptr(kc), _ptr(vc),
                                      _ptr(lens), N, H, dqk, dv, L_max, int(rope_dim), float(theta),
                                      float(scale), int(bool(cache_bf16)), _ptr(out)), "decode_step")
    return out, kc, vc, lens
