"""CPU oracle for the KDA mixer (double precision, plain C behind ctypes).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the CUDA library and its
Python binding never do.  The C source (``kda_oracle.c``) cites, for each
function, the passage of the pages it follows; the module here only marshals
numpy arrays.

Every function takes float64 arrays (any input precision is widened first),
checks shapes, and returns new float64 arrays.  Layouts: q, k, g [T, H, dk];
v, gate, o [T, H, dv]; beta [T, H]; states [N, H, dk, dv]; conv weights
[D, W]; conv state [N, W-1, D] with D = 2*H*dk + H*dv for the mixer.

Parity note: the value of the q/k L2-norm eps (named KDA_L2_EPS on the metrale
kimi_k3 page, Constants) is not printed on the pages; ``KDA_L2_EPS`` below is
the reading used (1e-6) and is passed in explicitly -- parity is unpinned at
the eps level.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

KDA_L2_EPS = 1e-6

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False, extra_flags=(), out_path: str | None = None, src: str | None = None) -> str:
    """Compile the oracle with gcc (-O2, OpenMP when available); return the .so path."""
    out = out_path or _LIB_PATH
    src = src or _SRC
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", *extra_flags, src, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(out + ".tmp", out)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle library and declare its signatures."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.kda_oracle_num_threads.restype = I
        lib.kda_oracle_short_conv.argtypes = [P, P, P, P, I, I, I, I, I, P, P]
        lib.kda_oracle_l2norm.argtypes = [P, ctypes.c_long, I, D]
        sig = [P, P, P, P, P, P, P, P, I, I, I, I, I, D, P, P]
        lib.kda_oracle_recurrent.argtypes = sig
        lib.kda_oracle_bruteforce.argtypes = sig
        lib.kda_oracle_chunked.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, D, I, P, P]
        lib.kda_oracle_mixer.argtypes = [P, P, P, P, P, P, P, P, I, P, P, P, I, I, I, I, I, D, I, D, P, P]
        lib.kda_oracle_decode_step.argtypes = [P, P, P, P, P, P, P, I, P, P, I, I, I, I, D, I, D, P]
        lib.kda_oracle_recurrent_backward.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, D, P, P, P, P, P, P]
        for f in ("kda_oracle_short_conv", "kda_oracle_l2norm", "kda_oracle_recurrent",
                  "kda_oracle_bruteforce", "kda_oracle_chunked", "kda_oracle_mixer",
                  "kda_oracle_decode_step"):
            getattr(lib, f).restype = I
        if path is None:
            _lib = lib
        return lib


def num_threads() -> int:
    return int(load().kda_oracle_num_threads())


def _f64(a, shape=None, name="array"):
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and tuple(a.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(a.shape)}")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _cu(cu_seqlens, T):
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int32)
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    return cu, int(cu.shape[0] - 1)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")


def short_conv(x, w, conv_state=None, cu_seqlens=None, apply_silu=True, return_state=False, lib=None):
    """Causal depthwise conv over packed sequences.  x [T, D], w [D, W]."""
    lib = lib or load()
    x = _f64(x, name="x")
    T, D = x.shape
    w = _f64(w, name="w")
    W = w.shape[1]
    cu, N = _cu(cu_seqlens, T)
    cs = _f64(conv_state, (N, W - 1, D), "conv_state")
    y = np.empty_like(x)
    cs_out = np.empty((N, W - 1, D)) if return_state else None
    _check(lib.kda_oracle_short_conv(_ptr(x), _ptr(w), _ptr(cs), _ptr(cu), N, T, D, W,
                                     int(bool(apply_silu)), _ptr(y), _ptr(cs_out)), "short_conv")
    return (y, cs_out) if return_state else y


def l2norm(x, eps=KDA_L2_EPS, lib=None):
    lib = lib or load()
    x = _f64(x, name="x").copy()
    d = x.shape[-1]
    _check(lib.kda_oracle_l2norm(_ptr(x), x.size // d, d, float(eps)), "l2norm")
    return x


def _core(fn, q, k, v, g, beta, S0, gate, cu_seqlens, scale, extra=()):
    q = _f64(q, name="q")
    T, H, dk = q.shape
    k = _f64(k, (T, H, dk), "k")
    v = _f64(v, name="v")
    dv = v.shape[2]
    if v.shape[:2] != (T, H):
        raise ValueError("v: bad shape")
    g = _f64(g, (T, H, dk), "g")
    beta = _f64(beta, (T, H), "beta")
    cu, N = _cu(cu_seqlens, T)
    S0 = _f64(S0, (N, H, dk, dv), "initial_state")
    gate = _f64(gate, (T, H, dv), "gate")
    if scale is None:
        scale = dk ** -0.5
    o = np.empty((T, H, dv))
    Sf = np.empty((N, H, dk, dv))
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(gate), _ptr(cu),
            N, T, H, dk, dv, float(scale)]
    _check(fn(*args, *extra, _ptr(o), _ptr(Sf)), fn.__name__)
    return o, Sf


def recurrent(q, k, v, g, beta, initial_state=None, gate=None, cu_seqlens=None, scale=None, lib=None):
    """Per-token KDA recurrence (the definition). Returns (o [T,H,dv], final_state [N,H,dk,dv])."""
    lib = lib or load()
    return _core(lib.kda_oracle_recurrent, q, k, v, g, beta, initial_state, gate, cu_seqlens, scale)


def recurrent_backward(q, k, v, g, beta, dO, initial_state=None, dS_final=None, cu_seqlens=None, scale=None,
                       lib=None):
    """Gradients of the ungated recurrence (reverse-mode, token by token) for the loss whose
    gradients with respect to o and to the final states are dO [T,H,dv] and dS_final
    [N,H,dk,dv] (optional).  Returns a dict with dq, dk, dv, dg [T,H,*], dbeta [T,H] and
    dS0 [N,H,dk,dv]."""
    lib = lib or load()
    q = _f64(q, name="q")
    T, H, dk = q.shape
    v = _f64(v, name="v")
    dv = v.shape[2]
    k = _f64(k, (T, H, dk), "k")
    g = _f64(g, (T, H, dk), "g")
    beta = _f64(beta, (T, H), "beta")
    dO = _f64(dO, (T, H, dv), "dO")
    cu, N = _cu(cu_seqlens, T)
    S0 = _f64(initial_state, (N, H, dk, dv), "initial_state")
    dSf = _f64(dS_final, (N, H, dk, dv), "dS_final")
    scale = float(dk) ** -0.5 if scale is None else float(scale)
    out = dict(dq=np.zeros((T, H, dk)), dk=np.zeros((T, H, dk)), dv=np.zeros((T, H, dv)), dg=np.zeros((T, H, dk)),
               dbeta=np.zeros((T, H)), dS0=np.zeros((N, H, dk, dv)))
    rc = lib.kda_oracle_recurrent_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(dO),
                                           _ptr(dSf), _ptr(cu), N, T, H, dk, dv, scale, _ptr(out["dq"]),
                                           _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["dbeta"]),
                                           _ptr(out["dS0"]))
    _check(rc, "recurrent_backward")
    return out


def bruteforce(q, k, v, g, beta, initial_state=None, gate=None, cu_seqlens=None, scale=None, lib=None):
    """Dense-transition form S_t = M_t S_{t-1} + beta k v^T (tiny inputs only)."""
    lib = lib or load()
    return _core(lib.kda_oracle_bruteforce, q, k, v, g, beta, initial_state, gate, cu_seqlens, scale)


def chunked(q, k, v, g, beta, initial_state=None, gate=None, cu_seqlens=None, scale=None, chunk=64, lib=None):
    """Chunked (WY/UT) form of the same recurrence, in double precision."""
    lib = lib or load()
    return _core(lib.kda_oracle_chunked, q, k, v, g, beta, initial_state, gate, cu_seqlens, scale,
                 extra=(int(chunk),))


def mixer(q, k, v, g, beta, initial_state=None, gate=None, conv_w=None, conv_state=None,
          cu_seqlens=None, scale=None, use_qk_l2norm=True, eps=KDA_L2_EPS, lib=None):
    """Full mixer: [conv+SiLU on q|k|v] -> [L2 on q,k] -> recurrence -> [sigmoid gate].

    q, k [T, H, dk], v [T, H, dv] pre-conv.  conv_w [2*H*dk + H*dv, W] or None.
    Returns (o, final_state, conv_state_out or None)."""
    lib = lib or load()
    q = _f64(q, name="q")
    T, H, dk = q.shape
    k = _f64(k, (T, H, dk), "k")
    v = _f64(v, name="v")
    dv = v.shape[2]
    g = _f64(g, (T, H, dk), "g")
    beta = _f64(beta, (T, H), "beta")
    cu, N = _cu(cu_seqlens, T)
    S0 = _f64(initial_state, (N, H, dk, dv), "initial_state")
    gate = _f64(gate, (T, H, dv), "gate")
    D = 2 * H * dk + H * dv
    W = 0
    cs_in = cs_out = None
    if conv_w is not None:
        conv_w = _f64(conv_w, name="conv_w")
        if conv_w.shape[0] != D:
            raise ValueError("conv_w: expected [2*H*dk + H*dv, W]")
        W = conv_w.shape[1]
        cs_in = _f64(conv_state, (N, W - 1, D), "conv_state")
        cs_out = np.empty((N, W - 1, D))
    if scale is None:
        scale = dk ** -0.5
    o = np.empty((T, H, dv))
    Sf = np.empty((N, H, dk, dv))
    _check(lib.kda_oracle_mixer(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(gate),
                                _ptr(conv_w), W, _ptr(cs_in), _ptr(cs_out), _ptr(cu), N, T, H, dk, dv,
                                float(scale), int(bool(use_qk_l2norm)), float(eps), _ptr(o), _ptr(Sf)),
           "mixer")
    return o, Sf, cs_out


def decode_step(q, k, v, g, beta, state, gate=None, conv_w=None, conv_state=None, scale=None,
                use_qk_l2norm=True, eps=KDA_L2_EPS, lib=None):
    """One token for each of N sequences.  q, k, g [N, H, dk]; v, gate [N, H, dv];
    beta [N, H]; state [N, H, dk, dv]; conv_state [N, W-1, D].  Returns
    (o [N, H, dv], new_state, new_conv_state or None); inputs are not modified."""
    lib = lib or load()
    q = _f64(q, name="q")
    N, H, dk = q.shape
    k = _f64(k, (N, H, dk), "k")
    v = _f64(v, name="v")
    dv = v.shape[2]
    g = _f64(g, (N, H, dk), "g")
    beta = _f64(beta, (N, H), "beta")
    gate = _f64(gate, (N, H, dv), "gate")
    st = _f64(state, (N, H, dk, dv), "state").copy()
    D = 2 * H * dk + H * dv
    W = 0
    cs = None
    if conv_w is not None:
        conv_w = _f64(conv_w, name="conv_w")
        if conv_w.shape[0] != D:
            raise ValueError("conv_w: expected [2*H*dk + H*dv, W]")
        W = conv_w.shape[1]
        cs = _f64(conv_state, (N, W - 1, D), "conv_state").copy()
    if scale is None:
        scale = dk ** -0.5
    o = np.empty((N, H, dv))
    _check(lib.kda_oracle_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(gate),
                                      _ptr(conv_w), W, _ptr(cs), _ptr(st), N, H, dk, dv, float(scale),
                                      int(bool(use_qk_l2norm)), float(eps), _ptr(o)), "decode_step")
    return o, st, cs


# ---- the FP32 CPU baseline (timed by the benchmark beside the oracle; never a reference) ----

_F32_SRC = os.path.join(_HERE, "cpu_f32.c")
_F32_PATH = os.path.join(_BUILD, "libkda_cpu_f32.so")
_f32_lib = None


def build_cpu_f32(force: bool = False) -> str:
    """Compile the FP32 CPU baseline (cpu_f32.c) like the oracle; return the .so path."""
    return build(force=force, out_path=_F32_PATH, src=_F32_SRC)


def load_cpu_f32():
    global _f32_lib
    with _lock:
        if _f32_lib is None:
            lib = ctypes.CDLL(build_cpu_f32())
            P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            lib.kda_cpu_f32_num_threads.restype = I
            lib.kda_cpu_f32_mixer.argtypes = [P, P, P, P, P, P, P, I, I, I, I, F, F, P, P]
            lib.kda_cpu_f32_mixer.restype = I
            _f32_lib = lib
    return _f32_lib


def cpu_f32_threads() -> int:
    return int(load_cpu_f32().kda_cpu_f32_num_threads())


def cpu_f32_mixer(q, k, v, g, beta, gate=None, conv_w=None, scale=None, eps=KDA_L2_EPS):
    """The mixer of one sequence in FP32 (conv width conv_w.shape[1] + SiLU, q/k L2 norm, the
    per-token recurrence from a zero state, gate): q, k, v, g, gate [T, H, d], beta [T, H],
    conv_w [3 H d, W].  Returns (o [T, H, d], final state [1, H, d, d]), float32."""
    lib = load_cpu_f32()
    f = lambda a: None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    q, k, v, g, beta, gate, conv_w = (f(x) for x in (q, k, v, g, beta, gate, conv_w))
    T, H, d = q.shape
    W = 0 if conv_w is None else conv_w.shape[1]
    o = np.empty((T, H, d), np.float32)
    Sf = np.empty((1, H, d, d), np.float32)
    _check(lib.kda_cpu_f32_mixer(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(gate), _ptr(conv_w), W, T,
                                 H, d, float(d ** -0.5 if scale is None else scale), float(eps), _ptr(o), _ptr(Sf)),
           "cpu_f32_mixer")
    return o, Sf
