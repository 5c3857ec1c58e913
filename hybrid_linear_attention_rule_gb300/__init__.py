"""GB300 (sm_103a) KDA mixer: Python binding of libk3kda.

The functions named ``k3kda_*`` are the C ABI of ``include/k3kda.h``, one for
one, taking torch CUDA tensors (or None) and marshalling their device pointers
and sizes; every step of the computation runs in the library's CUDA kernels.
PyTorch only provides device memory and the current stream.  A nonzero status
raises ``K3KDAError``.  If the CUDA library is missing and cannot be built,
importing the binding's functions raises: there is no CPU fallback.

Layouts (row-major, contiguous): q, k, g [T, H, dk]; v, gate, out [T, H, dv];
beta [T, H]; states [N, H, dk, dv] fp32; cu_seqlens int32 [N+1]; conv weights
[2*H*dk + H*dv, W] fp32; conv state [N, W-1, 2*H*dk + H*dv] fp32.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["K3KDAError", "load_library", "library_path", "F32", "BF16", "L2_EPS",
           "k3kda_version", "k3kda_status_string", "k3kda_launch_count", "k3kda_short_conv",
           "k3kda_prefill_workspace_size", "k3kda_prefill_workspace_min", "k3kda_prefill", "k3kda_prefill_slots",
           "k3kda_decode_step_slots", "k3kda_prefill_noalloc", "k3kda_prefill_noalloc_status",
           "k3kda_decode_status", "k3kda_workspace_status",
           "k3kda_backward_workspace_size", "k3kda_backward", "backward",
           "k3kda_decode_step", "prefill", "decode_step", "short_conv",
           "k3mla_decode_workspace_size", "k3mla_decode_step", "k3mla_decode_step_slots", "mla_decode_step"]

F32, BF16 = 0, 1
L2_EPS = 1e-6
_STATUS = {0: "OK", -1: "INVALID_ARG", -2: "UNSUPPORTED", -3: "ALIGNMENT", -4: "WORKSPACE",
           -5: "CUDA", -6: "TIMEOUT"}

_lib = None
_lock = threading.Lock()


class K3KDAError(RuntimeError):
    def __init__(self, fn, status, detail=""):
        self.status = status
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)} ({status}) {detail}".rstrip())


def library_path() -> str:
    from . import build as _b
    return _b.LIB


def load_library(build_if_missing: bool = True):
    """Load libk3kda.so (building it with nvcc when missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import build as _b
        if build_if_missing and not _b.up_to_date():
            _b.build()
        if not os.path.exists(_b.LIB):
            raise RuntimeError(f"libk3kda.so not found at {_b.LIB}; build it with "
                               "hybrid_linear_attention_rule_gb300.build.build()")
        lib = ctypes.CDLL(_b.LIB)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.k3kda_version.restype = I
        lib.k3kda_status_string.restype = ctypes.c_char_p
        lib.k3kda_status_string.argtypes = [I]
        lib.k3kda_last_error.restype = ctypes.c_char_p
        lib.k3kda_launch_count.restype = ctypes.c_longlong
        lib.k3kda_short_conv.argtypes = [P, I, P, P, P, I, I, I, I, I, P, I, P]
        lib.k3kda_short_conv.restype = I
        lib.k3kda_prefill_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
        lib.k3kda_prefill_workspace_size.restype = Z
        lib.k3kda_prefill_workspace_min.argtypes = [I, I, I, I, I, I, I, I]
        lib.k3kda_prefill_workspace_min.restype = Z
        lib.k3kda_prefill.argtypes = [P, P, P, I, P, P, P, P, P, I, I, I, I, I, I, F, I, P, P, P, I, P,
                                      P, Z, P]
        lib.k3kda_prefill.restype = I
        lib.k3kda_prefill_noalloc.argtypes = [P, P, P, I, P, P, P, P, P, I, I, I, I, I, I, F, I, P, P, P, I, P, P]
        lib.k3kda_prefill_noalloc.restype = I
        lib.k3kda_workspace_status.argtypes = [P, P]
        lib.k3kda_workspace_status.restype = I
        lib.k3kda_prefill_noalloc_status.argtypes = [P]
        lib.k3kda_prefill_noalloc_status.restype = I
        lib.k3kda_decode_status.argtypes = [P]
        lib.k3kda_decode_status.restype = I
        # internal test hook (not in the public header): see k3kda_test_arm_wait_timeout in api.cu
        lib.k3kda_test_arm_wait_timeout.argtypes = [I, ctypes.c_uint]
        lib.k3kda_test_arm_wait_timeout.restype = I
        lib.k3kda_decode_step.argtypes = [P, P, P, I, P, P, P, P, P, P, I, I, I, I, I, F, I, P, I, P]
        lib.k3kda_decode_step.restype = I
        lib.k3kda_prefill_slots.argtypes = [P, P, P, I, P, P, P, P, P, I, P, P, I, I, I, I, I, I, F, I, P, P,
                                            P, I, P, Z, P]
        lib.k3kda_prefill_slots.restype = I
        lib.k3kda_decode_step_slots.argtypes = [P, P, P, I, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, P, I,
                                                P]
        lib.k3kda_decode_step_slots.restype = I
        lib.k3kda_backward_workspace_size.argtypes = [I, I, I, I, I]
        lib.k3kda_backward_workspace_size.restype = ctypes.c_size_t
        lib.k3kda_backward.argtypes = [P, P, P, I, P, P, P, P, P, I, I, I, I, I, F, P, P, P, P, P, P, P, P, P,
                                       ctypes.c_size_t, P]
        lib.k3kda_backward.restype = I
        lib.k3mla_decode_workspace_size.argtypes = [I, I, I, I, I]
        lib.k3mla_decode_workspace_size.restype = Z
        lib.k3mla_decode_step.argtypes = [P, P, P, I, P, P, P, I, P, I, I, I, I, I, I, F, F, P, I, P, Z, P]
        lib.k3mla_decode_step.restype = I
        lib.k3mla_decode_step_slots.argtypes = [P, P, P, I, P, P, P, I, P, P, P, I, I, I, I, I, I, I, F, F, P, I, P,
                                                Z, P]
        lib.k3mla_decode_step_slots.restype = I
        _lib = lib
        return lib


class _ConvArgs(ctypes.Structure):
    _fields_ = [("weight", ctypes.c_void_p), ("conv_state", ctypes.c_void_p), ("W", ctypes.c_int)]


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor or None")
    if not t.is_cuda:
        raise ValueError("k3kda: tensors must live on a CUDA device (no CPU path exists)")
    if not t.is_contiguous():
        raise ValueError("k3kda: tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dtype(t):
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"k3kda: unsupported element type {t.dtype}")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, st):
    if st != 0:
        lib = load_library()
        raise K3KDAError(fn, st, lib.k3kda_last_error().decode() if st == -5 else "")


# ---- the C ABI, one for one ------------------------------------------------

def k3kda_version() -> int:
    return int(load_library().k3kda_version())


def k3kda_launch_count() -> int:
    return int(load_library().k3kda_launch_count())


def k3kda_status_string(status: int) -> str:
    return load_library().k3kda_status_string(int(status)).decode()


def k3kda_short_conv(x, weight, conv_state, cu_seqlens, N, T, D, W, apply_silu, out, stream=None):
    lib = load_library()
    st = lib.k3kda_short_conv(_ptr(x), _dtype(x), _ptr(weight), _ptr(conv_state), _ptr(cu_seqlens),
                              int(N), int(T), int(D), int(W), int(bool(apply_silu)), _ptr(out),
                              _dtype(out), _stream(stream))
    _check("k3kda_short_conv", st)


def k3kda_prefill_workspace_size(N, T, H, dk, dv, chunk, in_dtype, has_conv) -> int:
    return int(load_library().k3kda_prefill_workspace_size(int(N), int(T), int(H), int(dk), int(dv),
                                                           int(chunk), int(in_dtype), int(bool(has_conv))))


def k3kda_prefill_workspace_min(N, T, H, dk, dv, chunk, in_dtype, has_conv) -> int:
    return int(load_library().k3kda_prefill_workspace_min(int(N), int(T), int(H), int(dk), int(dv),
                                                          int(chunk), int(in_dtype), int(bool(has_conv))))


def k3kda_prefill(q, k, v, g, beta, initial_state, cu_seqlens, cu_seqlens_host, N, T, H, dk, dv, chunk,
                  scale, use_qk_l2norm, conv_weight, conv_state, conv_W, gate, out, final_state,
                  workspace, stream=None):
    """cu_seqlens_host: a CPU int32 tensor (or None), passed as the host copy."""
    lib = load_library()
    conv = None
    if conv_weight is not None:
        conv = ctypes.byref(_ConvArgs(_ptr(conv_weight), _ptr(conv_state), int(conv_W)))
    hcu = None
    if cu_seqlens_host is not None:
        if cu_seqlens_host.is_cuda or cu_seqlens_host.dtype != torch.int32 or not cu_seqlens_host.is_contiguous():
            raise ValueError("cu_seqlens_host must be a contiguous CPU int32 tensor")
        hcu = ctypes.c_void_p(cu_seqlens_host.data_ptr())
    st = lib.k3kda_prefill(_ptr(q), _ptr(k), _ptr(v), _dtype(q), _ptr(g), _ptr(beta), _ptr(initial_state),
                           _ptr(cu_seqlens), hcu, int(N), int(T), int(H), int(dk), int(dv), int(chunk),
                           float(scale), int(bool(use_qk_l2norm)), conv, _ptr(gate), _ptr(out), _dtype(out),
                           _ptr(final_state), _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream(stream))
    _check("k3kda_prefill", st)


def _host_i32(t, what):
    if t is None:
        return None
    if t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous CPU int32 tensor")
    return ctypes.c_void_p(t.data_ptr())


def k3kda_prefill_slots(q, k, v, g, beta, state_pool, state_idx, state_idx_host, num_slots, cu_seqlens,
                        cu_seqlens_host, N, T, H, dk, dv, chunk, scale, use_qk_l2norm, conv_weight,
                        conv_state_pool, conv_W, gate, out, workspace, stream=None):
    """k3kda_prefill on slot-indexed state pools: sequence n reads and updates slot state_idx[n]."""
    lib = load_library()
    conv = None
    if conv_weight is not None:
        conv = ctypes.byref(_ConvArgs(_ptr(conv_weight), _ptr(conv_state_pool), int(conv_W)))
    st = lib.k3kda_prefill_slots(_ptr(q), _ptr(k), _ptr(v), _dtype(q), _ptr(g), _ptr(beta), _ptr(state_pool),
                                 _ptr(state_idx), _host_i32(state_idx_host, "state_idx_host"), int(num_slots),
                                 _ptr(cu_seqlens), _host_i32(cu_seqlens_host, "cu_seqlens_host"), int(N), int(T),
                                 int(H), int(dk), int(dv), int(chunk), float(scale), int(bool(use_qk_l2norm)), conv,
                                 _ptr(gate), _ptr(out), _dtype(out), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check("k3kda_prefill_slots", st)


def k3kda_decode_step_slots(q, k, v, g, beta, gate, conv_weight, conv_state_pool, state_pool, state_idx,
                            state_idx_host, num_slots, N, H, dk, dv, W, scale, use_qk_l2norm, out, stream=None):
    """k3kda_decode_step on slot-indexed state pools: sequence n reads and updates slot state_idx[n]."""
    lib = load_library()
    st = lib.k3kda_decode_step_slots(_ptr(q), _ptr(k), _ptr(v), _dtype(q), _ptr(g), _ptr(beta), _ptr(gate),
                                     _ptr(conv_weight), _ptr(conv_state_pool), _ptr(state_pool), _ptr(state_idx),
                                     _host_i32(state_idx_host, "state_idx_host"), int(num_slots), int(N), int(H),
                                     int(dk), int(dv), int(W), float(scale), int(bool(use_qk_l2norm)), _ptr(out),
                                     _dtype(out), _stream(stream))
    _check("k3kda_decode_step_slots", st)


def k3kda_backward_workspace_size(N, T, H, dk, dv):
    return int(load_library().k3kda_backward_workspace_size(int(N), int(T), int(H), int(dk), int(dv)))


def k3kda_backward(q, k, v, g, beta, initial_state, cu_seqlens, cu_seqlens_host, N, T, H, dk, dv, scale, dO,
                   dS_final, dq, dk_out, dv_out, dg, dbeta, dS0, workspace, stream=None):
    """Reverse-mode gradients of the ungated recurrence (see include/k3kda.h)."""
    lib = load_library()
    st = lib.k3kda_backward(_ptr(q), _ptr(k), _ptr(v), _dtype(q), _ptr(g), _ptr(beta), _ptr(initial_state),
                            _ptr(cu_seqlens), _host_i32(cu_seqlens_host, "cu_seqlens_host"), int(N), int(T), int(H),
                            int(dk), int(dv), float(scale), _ptr(dO), _ptr(dS_final), _ptr(dq), _ptr(dk_out),
                            _ptr(dv_out), _ptr(dg), _ptr(dbeta), _ptr(dS0), _ptr(workspace),
                            int(workspace.numel() * workspace.element_size()), _stream(stream))
    _check("k3kda_backward", st)


def backward(q, k, v, g, beta, dO, initial_state=None, dS_final=None, cu_seqlens=None, scale=None, stream=None):
    """Gradients (dict of fp32 tensors dq, dk, dv, dg, dbeta, dS0) of the ungated recurrence for the
    loss gradients dO [T, H, dv] (fp32) and dS_final [N, H, dk, dv] (optional); allocates its outputs
    and workspace with torch."""
    T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        cu_host = torch.tensor([0, T], dtype=torch.int32)
    else:
        cu_host = cu_seqlens.to("cpu", torch.int32)
    N = int(cu_host.numel()) - 1
    cu_dev = cu_host.to(q.device)
    scale = float(dk) ** -0.5 if scale is None else float(scale)
    f32 = dict(dtype=torch.float32, device=q.device)
    out = dict(dq=torch.empty(T, H, dk, **f32), dk=torch.empty(T, H, dk, **f32), dv=torch.empty(T, H, dv, **f32),
               dg=torch.empty(T, H, dk, **f32), dbeta=torch.empty(T, H, **f32), dS0=torch.empty(N, H, dk, dv, **f32))
    ws = torch.empty(k3kda_backward_workspace_size(N, T, H, dk, dv), dtype=torch.uint8, device=q.device)
    k3kda_backward(q, k, v, g, beta, initial_state, cu_dev, cu_host, N, T, H, dk, dv, scale, dO, dS_final,
                   out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta"], out["dS0"], ws, stream)
    return out


def k3kda_prefill_noalloc(q, k, v, g, beta, initial_state, cu_seqlens, cu_seqlens_host, N, T, H, dk, dv,
                          chunk, scale, use_qk_l2norm, conv_weight, conv_state, conv_W, gate, out, final_state,
                          stream=None):
    """k3kda_prefill without a workspace: for callers that cannot allocate device memory where
    they run the mixer.  The scratch is a fixed 16 MiB array the library holds on each GPU; work
    that needs more raises K3KDAError (WORKSPACE).  The first call on a device sets up the array's
    address and should come before any stream capture; calls that overlap on the GPU race on it."""
    lib = load_library()
    conv = None
    if conv_weight is not None:
        conv = ctypes.byref(_ConvArgs(_ptr(conv_weight), _ptr(conv_state), int(conv_W)))
    hcu = None
    if cu_seqlens_host is not None:
        if cu_seqlens_host.is_cuda or cu_seqlens_host.dtype != torch.int32 or not cu_seqlens_host.is_contiguous():
            raise ValueError("cu_seqlens_host must be a contiguous CPU int32 tensor")
        hcu = ctypes.c_void_p(cu_seqlens_host.data_ptr())
    st = lib.k3kda_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _dtype(q), _ptr(g), _ptr(beta), _ptr(initial_state),
                                   _ptr(cu_seqlens), hcu, int(N), int(T), int(H), int(dk), int(dv), int(chunk),
                                   float(scale), int(bool(use_qk_l2norm)), conv, _ptr(gate), _ptr(out), _dtype(out),
                                   _ptr(final_state), _stream(stream))
    _check("k3kda_prefill_noalloc", st)


def k3kda_workspace_status(workspace, stream=None) -> int:
    return int(load_library().k3kda_workspace_status(_ptr(workspace), _stream(stream)))


def k3kda_prefill_noalloc_status(stream=None) -> int:
    return int(load_library().k3kda_prefill_noalloc_status(_stream(stream)))


def k3kda_decode_status(stream=None) -> int:
    return int(load_library().k3kda_decode_status(_stream(stream)))


def k3kda_decode_step(q, k, v, g, beta, gate, conv_weight, conv_state, state, N, H, dk, dv, W, scale,
                      use_qk_l2norm, out, stream=None):
    lib = load_library()
    st = lib.k3kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _dtype(q), _ptr(g), _ptr(beta), _ptr(gate),
                               _ptr(conv_weight), _ptr(conv_state), _ptr(state), int(N), int(H), int(dk),
                               int(dv), int(W), float(scale), int(bool(use_qk_l2norm)), _ptr(out),
                               _dtype(out), _stream(stream))
    _check("k3kda_decode_step", st)


# ---- conveniences: allocate outputs with torch, then call the ABI ----------

def prefill(q, k, v, g, beta, initial_state=None, cu_seqlens=None, chunk=64, scale=None,
            use_qk_l2norm=True, conv_weight=None, conv_state=None, gate=None, out_dtype=None,
            return_final_state=True, workspace=None, min_workspace=False, stream=None):
    """Allocate out / final_state / workspace and run k3kda_prefill.  cu_seqlens may be
    a CPU or CUDA int32 tensor (both copies are passed).  The workspace is the size of
    k3kda_prefill_workspace_size (the fastest path), or of k3kda_prefill_workspace_min
    with min_workspace=True.  Returns (out, final_state)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    dev = q.device
    if cu_seqlens is None:
        cu_h = torch.tensor([0, T], dtype=torch.int32)
    else:
        cu_h = cu_seqlens.to("cpu", torch.int32).contiguous()
    cu_d = cu_h.to(dev)
    N = cu_h.numel() - 1
    out = torch.empty((T, H, dv), dtype=out_dtype or q.dtype, device=dev)
    fs = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev) if return_final_state else None
    W = 0 if conv_weight is None else conv_weight.shape[1]
    if workspace is None:
        size_fn = k3kda_prefill_workspace_min if min_workspace else k3kda_prefill_workspace_size
        nbytes = size_fn(N, T, H, dk, dv, chunk, _dtype(q), conv_weight is not None)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        workspace[:256].zero_()                     # the status word; the rest is written before it is read
    k3kda_prefill(q, k, v, g, beta, initial_state, cu_d, cu_h, N, T, H, dk, dv, chunk,
                  dk ** -0.5 if scale is None else scale, use_qk_l2norm, conv_weight, conv_state, W,
                  gate, out, fs, workspace, stream)
    return out, fs


def decode_step(q, k, v, g, beta, state, gate=None, conv_weight=None, conv_state=None, scale=None,
                use_qk_l2norm=True, out_dtype=None, stream=None):
    """Run k3kda_decode_step; state and conv_state are updated in place.  Returns out."""
    N, H, dk = q.shape
    dv = v.shape[2]
    out = torch.empty((N, H, dv), dtype=out_dtype or q.dtype, device=q.device)
    W = 0 if conv_weight is None else conv_weight.shape[1]
    k3kda_decode_step(q, k, v, g, beta, gate, conv_weight, conv_state, state, N, H, dk, dv, W,
                      dk ** -0.5 if scale is None else scale, use_qk_l2norm, out, stream)
    return out


def short_conv(x, weight, conv_state=None, cu_seqlens=None, apply_silu=True, out_dtype=None, stream=None):
    """Run k3kda_short_conv over x [T, D]; conv_state is updated in place.  Returns out."""
    T, D = x.shape
    W = weight.shape[1]
    cu = None if cu_seqlens is None else cu_seqlens.to(x.device, torch.int32)
    N = 1 if cu is None else cu.numel() - 1
    out = torch.empty((T, D), dtype=out_dtype or x.dtype, device=x.device)
    k3kda_short_conv(x, weight, conv_state, cu, N, T, D, W, apply_silu, out, stream)
    return out


# ---- the gated attention (MLA) layers' decode token ------------------------

def k3mla_decode_workspace_size(N, H, dqk, dv, L_max) -> int:
    return int(load_library().k3mla_decode_workspace_size(int(N), int(H), int(dqk), int(dv), int(L_max)))


def k3mla_decode_step(q, k_new, v_new, gate, k_cache, v_cache, cache_len, N, H, dqk, dv, L_max, rope_dim, rope_theta,
                      scale, out, workspace, stream=None):
    """One decode token of the gated attention layers (see include/k3kda.h): RoPE, append, attention, gate."""
    lib = load_library()
    st = lib.k3mla_decode_step(_ptr(q), _ptr(k_new), _ptr(v_new), _dtype(q), _ptr(gate), _ptr(k_cache),
                               _ptr(v_cache), _dtype(k_cache), _ptr(cache_len), int(N), int(H), int(dqk), int(dv),
                               int(L_max),
                               int(rope_dim), float(rope_theta), float(scale), _ptr(out), _dtype(out),
                               _ptr(workspace), int(workspace.numel() * workspace.element_size()), _stream(stream))
    _check("k3mla_decode_step", st)


def k3mla_decode_step_slots(q, k_new, v_new, gate, k_cache_pool, v_cache_pool, cache_len_pool, cache_idx,
                            cache_idx_host, num_slots, N, H, dqk, dv, L_max, rope_dim, rope_theta, scale, out,
                            workspace, stream=None):
    """One decode token over a slot-indexed cache pool (see include/k3kda.h)."""
    lib = load_library()
    st = lib.k3mla_decode_step_slots(_ptr(q), _ptr(k_new), _ptr(v_new), _dtype(q), _ptr(gate), _ptr(k_cache_pool),
                                     _ptr(v_cache_pool), _dtype(k_cache_pool), _ptr(cache_len_pool), _ptr(cache_idx),
                                     _host_i32(cache_idx_host, "cache_idx_host"), int(num_slots), int(N), int(H),
                                     int(dqk), int(dv), int(L_max), int(rope_dim), float(rope_theta), float(scale),
                                     _ptr(out), _dtype(out), _ptr(workspace),
                                     int(workspace.numel() * workspace.element_size()), _stream(stream))
    _check("k3mla_decode_step_slots", st)


def mla_decode_step(q, k_new, v_new, k_cache, v_cache, cache_len, gate=None, scale=None, rope_dim=0,
                    rope_theta=10000.0, out_dtype=None, workspace=None, stream=None):
    """Decode one token for every sequence: q, k_new [N, H, dqk], v_new [N, H, dv]; caches
    [N, H, L_max, dqk | dv] and cache_len int32 [N] are updated in place.  Returns the output
    [N, H, dv] (allocated with torch, in out_dtype, default q's type)."""
    N, H, dqk = q.shape
    dv = v_new.shape[-1]
    L_max = k_cache.shape[2]
    scale = float(dqk) ** -0.5 if scale is None else float(scale)
    out = torch.empty(N, H, dv, dtype=out_dtype or q.dtype, device=q.device)
    if workspace is None:
        workspace = torch.empty(k3mla_decode_workspace_size(N, H, dqk, dv, L_max), dtype=torch.uint8, device=q.device)
    k3mla_decode_step(q, k_new, v_new, gate, k_cache, v_cache, cache_len, N, H, dqk, dv, L_max, rope_dim, rope_theta,
                      scale, out, workspace, stream)
    return out
