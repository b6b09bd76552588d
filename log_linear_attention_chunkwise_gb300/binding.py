"""Thin ctypes binding of liblla.so: the same entry points, torch tensors in.

Argument marshalling only (shape/dtype/device checks, pointers, the current
stream, workspace allocation through torch's allocator).  Every step of the
operator runs in the library's CUDA kernels; there is no other code path.
If ``liblla.so`` is missing the first call raises, it never falls back.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblla.so")

LLA_F32, LLA_BF16 = 0, 1
STATUS = {0: "LLA_OK", 1: "LLA_ERR_INVALID_ARGUMENT", 2: "LLA_ERR_UNSUPPORTED_SHAPE",
          3: "LLA_ERR_WORKSPACE_TOO_SMALL", 4: "LLA_ERR_CUDA", 5: "LLA_ERR_DEVICE_REPORTED"}

# name -> (restype, argtypes); mirrors include/lla.h
_P, _I, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "lla_status_string": (ctypes.c_char_p, [_I]),
    "lla_version": (_I, []),
    "lla_num_levels": (_I, [_I]),
    "lla_fwd_workspace_bytes": (_Z, [_I] * 6 + [_I]),
    "lla_fwd_launches": (_I, [_I] * 8),
    "lla_fwd": (_I, [_P] * 6 + [_I] * 6 + [_I, _I] + [_P, _Z, _P, _P]),
    "lla_fwd_noalloc_max_scratch_bytes": (_Z, []),
    "lla_fwd_noalloc": (_I, [_P] * 6 + [_I] * 6 + [_I, _I] + [_P, _P]),
    "lla_decode_state_bytes": (_Z, [_I] * 5),
    "lla_decode_step": (_I, [_P] * 9 + [_I] * 5 + [_I, _P, _P]),
    "lla_prefill_workspace_bytes": (_Z, [_I] * 3),
    "lla_prefill_state": (_I, [_P] * 5 + [_I] * 6 + [_I, _P, _Z, _P, _P]),
    "lla_lambda_mlp": (_I, [_P] * 5 + [_I] * 5 + [_I, _P, _P]),
    "lla_bwd_workspace_bytes": (_Z, [_I] * 7),
    "lla_bwd": (_I, [_P] * 11 + [_I] * 7 + [_P, _Z, _P, _P]),
    "lla_gdn_fwd_workspace_bytes": (_Z, [_I] * 5),
    "lla_gdn_fwd": (_I, [_P] * 8 + [_I] * 6 + [_I, _P, _Z, _P]),
    "lla_fwd_host_workspace_bytes": (_Z, [_I] * 9),
    "lla_fwd_host": (_I, [_P] * 6 + [_I] * 6 + [_I, _I, _I, _P, _Z, _P, _P]),
    "lla_gdn_decode_step": (_I, [_P] * 9 + [_I] * 5 + [_I, _P, _P]),
    "lla_device_error_check": (_I, [_P, _P, _P]),
    "lla_fwd_lambda_mlp_workspace_bytes": (_Z, [_I] * 8),
    "lla_fwd_lambda_mlp": (_I, [_P] * 9 + [_I] * 8 + [_I, _P, _Z, _P, _P]),
    "lla_debug_withhold_first_product": (None, [_I]),
}

_lib = None


class LLAError(RuntimeError):
    def __init__(self, name, code):
        super().__init__(f"{name} returned {STATUS.get(code, code)}")
        self.code = code


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load liblla.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"liblla.so not built at {path}: run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LLA_F32
    if t.dtype == torch.bfloat16:
        return LLA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(name, code):
    if code != 0:
        raise LLAError(name, code)


def _err_ptr(device_error):
    if device_error is None:
        return None
    _need(device_error, "device_error", torch.int32, None)
    if device_error.numel() < 1:
        raise ValueError("device_error needs one int32 element")
    return ctypes.c_void_p(device_error.data_ptr())


def device_error_check(device_error, stream=None):
    """lla_device_error_check: synchronise the stream and return the code in
    device_error (0 when no kernel reported anything)."""
    code = ctypes.c_int32(0)
    rc = load().lla_device_error_check(_err_ptr(device_error), ctypes.byref(code), _stream(stream))
    if rc not in (0, 5):
        raise LLAError("lla_device_error_check", rc)
    return int(code.value)


def debug_withhold_first_product(enable: bool):
    """lla_debug_withhold_first_product: the test hook of the reporting path."""
    load().lla_debug_withhold_first_product(1 if enable else 0)


def _need(t, name, dtype=None, ndim=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def num_levels(T: int) -> int:
    return load().lla_num_levels(T)


def fwd_workspace_bytes(B, H, T, dk, dv, chunk, in_dtype) -> int:
    return load().lla_fwd_workspace_bytes(B, H, T, dk, dv, chunk, _dt(torch.empty(0, dtype=in_dtype)))


def fwd(q, k, v, g, lam, chunk: int = 64, out_dtype=torch.float32, out=None, workspace=None,
        device_error=None, stream=None):
    """lla_fwd on torch tensors: q,k [B,H,T,dk], v [B,H,T,dv] (fp32 or bf16),
    g [B,H,T] fp32, lam [B,H,T,L] fp32.  Returns out [B,H,T,dv].
    device_error: optional int32 CUDA tensor of one element (see
    device_error_check)."""
    lib = load()
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need(t, n, q.dtype, 4)
    _need(g, "g", torch.float32, 3)
    _need(lam, "lam", torch.float32, 4)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, H, T) or g.shape != (B, H, T) or \
            lam.shape[:3] != (B, H, T) or lam.shape[3] != max(lib.lla_num_levels(T), 1):
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=out_dtype, device=q.device)
    _need(out, "out", None, 4)
    in_dt = _dt(q)
    need = lib.lla_fwd_workspace_bytes(B, H, T, dk, dv, chunk, in_dt)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    rc = lib.lla_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(lam), _ptr(out), B, H, T, dk, dv,
                     chunk, in_dt, _dt(out), _ptr(workspace), workspace.numel(),
                     _err_ptr(device_error), _stream(stream))
    _check("lla_fwd", rc)
    return out


def fwd_lambda_mlp(q, k, v, g, d, W1, W2, b, chunk: int = 64, out_dtype=torch.float32, out=None,
                   workspace=None, device_error=None, stream=None):
    """lla_fwd_lambda_mlp: the forward with lambda = softplus((d W1) W2 + b)
    computed from d [B,H,T,Dd] (pass d = k for the in-kernel path);
    W1 [Dd,2L], W2 [2L,L], b [L] fp32.  Returns out [B,H,T,dv]."""
    lib = load()
    for n, t in (("q", q), ("k", k), ("v", v), ("d", d)):
        _need(t, n, q.dtype, 4)
    _need(g, "g", torch.float32, 3)
    for n, t in (("W1", W1), ("W2", W2), ("b", b)):
        _need(t, n, torch.float32, None)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    Dd = d.shape[-1]
    L = lib.lla_num_levels(T)
    if k.shape != q.shape or v.shape[:3] != (B, H, T) or g.shape != (B, H, T) or \
            d.shape[:3] != (B, H, T) or W1.shape != (Dd, 2 * L) or W2.shape != (2 * L, L) or \
            b.shape != (L,):
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=out_dtype, device=q.device)
    _need(out, "out", None, 4)
    in_dt = _dt(q)
    need = lib.lla_fwd_lambda_mlp_workspace_bytes(B, H, T, dk, dv, Dd, chunk, in_dt)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    rc = lib.lla_fwd_lambda_mlp(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(d), _ptr(W1), _ptr(W2), _ptr(b),
                                _ptr(out), B, H, T, dk, dv, Dd, chunk, in_dt, _dt(out), _ptr(workspace),
                                workspace.numel(), _err_ptr(device_error), _stream(stream))
    _check("lla_fwd_lambda_mlp", rc)
    return out


def decode_state_bytes(B, H, dk, dv, Ls) -> int:
    return load().lla_decode_state_bytes(B, H, dk, dv, Ls)


def decode_step(state, logdecay, q, k, v, g, lam, pos, out=None, device_error=None, stream=None):
    """lla_decode_step: state [B,H,Ls,dk,dv] fp32 and logdecay [B,H,Ls] fp32
    updated in place; q,k [B,H,dk], v [B,H,dv]; g [B,H]; lam [B,H,Ls+1];
    pos [B] int64 (device).  Returns out [B,H,dv] fp32."""
    lib = load()
    _need(state, "state", torch.float32, 5)
    _need(logdecay, "logdecay", torch.float32, 3)
    _need(q, "q", None, 3)
    _need(k, "k", q.dtype, 3)
    _need(v, "v", q.dtype, 3)
    _need(g, "g", torch.float32, 2)
    _need(lam, "lam", torch.float32, 3)
    _need(pos, "pos", torch.int64, 1)
    B, H, Ls, dk, dv = state.shape
    if q.shape != (B, H, dk) or k.shape != (B, H, dk) or v.shape != (B, H, dv) or \
            g.shape != (B, H) or lam.shape != (B, H, Ls + 1) or pos.shape != (B,) or \
            logdecay.shape != (B, H, Ls):
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((B, H, dv), dtype=torch.float32, device=q.device)
    rc = lib.lla_decode_step(_ptr(state), _ptr(logdecay), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                             _ptr(lam), _ptr(out), _ptr(pos), B, H, dk, dv, Ls, _dt(q),
                             _ptr(device_error), _stream(stream))
    _check("lla_decode_step", rc)
    return out


def prefill_state(k, v, g, Ls: int, state=None, logdecay=None, workspace=None, device_error=None,
                  stream=None):
    """lla_prefill_state: decode state after the prefix k,v [B,H,T,d], g [B,H,T]."""
    lib = load()
    _need(k, "k", None, 4)
    _need(v, "v", k.dtype, 4)
    _need(g, "g", torch.float32, 3)
    B, H, T, dk = k.shape
    dv = v.shape[-1]
    if state is None:
        state = torch.empty((B, H, Ls, dk, dv), dtype=torch.float32, device=k.device)
    if logdecay is None:
        logdecay = torch.empty((B, H, Ls), dtype=torch.float32, device=k.device)
    need = lib.lla_prefill_workspace_bytes(B, H, T)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=k.device)
    rc = lib.lla_prefill_state(_ptr(k), _ptr(v), _ptr(g), _ptr(state), _ptr(logdecay), B, H, T,
                               dk, dv, Ls, _dt(k), _ptr(workspace), workspace.numel(),
                               _err_ptr(device_error), _stream(stream))
    _check("lla_prefill_state", rc)
    return state, logdecay


def lambda_mlp(d, W1, W2, b, out=None, device_error=None, stream=None):
    """lla_lambda_mlp: lambda [B,H,T,L] = softplus((d W1) W2 + b) for
    d [B,H,T,Dd] (fp32 or bf16), W1 [Dd,2L], W2 [2L,L], b [L] fp32."""
    lib = load()
    _need(d, "d", None, 4)
    for n, t in (("W1", W1), ("W2", W2), ("b", b)):
        _need(t, n, torch.float32, None)
    B, H, T, Dd = d.shape
    L = b.shape[0]
    if W1.shape != (Dd, 2 * L) or W2.shape != (2 * L, L):
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((B, H, T, L), dtype=torch.float32, device=d.device)
    rc = lib.lla_lambda_mlp(_ptr(d), _ptr(W1), _ptr(W2), _ptr(b), _ptr(out), B, H, T, Dd, L,
                            _dt(d), _err_ptr(device_error), _stream(stream))
    _check("lla_lambda_mlp", rc)
    return out


def bwd(q, k, v, g, lam, dout, chunk: int = 64, workspace=None, device_error=None, stream=None):
    """lla_bwd: gradients (dq, dk, dv, dg, dlam) of sum(dout * lla_fwd(q, k, v, g, lam))."""
    lib = load()
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need(t, n, q.dtype, 4)
    _need(g, "g", torch.float32, 3)
    _need(lam, "lam", torch.float32, 4)
    _need(dout, "dout", torch.float32, 4)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, H, T) or g.shape != (B, H, T) or \
            dout.shape != v.shape or lam.shape[:3] != (B, H, T) or \
            lam.shape[3] != max(lib.lla_num_levels(T), 1):
        raise ValueError("inconsistent shapes")
    f32 = dict(dtype=torch.float32, device=q.device)
    dq = torch.empty((B, H, T, dk), **f32)
    dkk = torch.empty((B, H, T, dk), **f32)
    dvv = torch.empty((B, H, T, dv), **f32)
    dg = torch.empty((B, H, T), **f32)
    dl = torch.empty(tuple(lam.shape), **f32)
    in_dt = _dt(q)
    need = lib.lla_bwd_workspace_bytes(B, H, T, dk, dv, chunk, in_dt)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    rc = lib.lla_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(lam), _ptr(dout), _ptr(dq), _ptr(dkk),
                     _ptr(dvv), _ptr(dg), _ptr(dl), B, H, T, dk, dv, chunk, in_dt, _ptr(workspace),
                     workspace.numel(), _err_ptr(device_error), _stream(stream))
    _check("lla_bwd", rc)
    return dq, dkk, dvv, dg, dl


def gdn_fwd(q, k, v, g, beta, lam, out=None, state_Ls: int = 0, workspace=None, stream=None):
    """lla_gdn_fwd: Log-Linear Gated DeltaNet over whole sequences.  Returns
    out [B,H,T,dv], or (out, state [B,H,state_Ls,dk,dv]) when state_Ls > 0.
    workspace: a uint8 device tensor of at least
    lla_gdn_fwd_workspace_bytes(B, H, T, dk, dv) bytes (allocated here when None)."""
    lib = load()
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need(t, n, q.dtype, 4)
    _need(g, "g", torch.float32, 3)
    _need(beta, "beta", torch.float32, 3)
    _need(lam, "lam", torch.float32, 4)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, H, T) or g.shape != (B, H, T) or \
            beta.shape != (B, H, T) or lam.shape[:3] != (B, H, T) or \
            lam.shape[3] != max(lib.lla_num_levels(T), 1):
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, 4)
    state = None
    if state_Ls > 0:
        state = torch.empty((B, H, state_Ls, dk, dv), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = lib.lla_gdn_fwd_workspace_bytes(B, H, T, dk, dv)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    rc = lib.lla_gdn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(lam), _ptr(out),
                         _ptr(state) if state is not None else None, B, H, T, dk, dv, state_Ls,
                         _dt(q), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("lla_gdn_fwd", rc)
    return (out, state) if state is not None else out


def gdn_decode_step(state, q, k, v, g, beta, lam, pos, out=None, device_error=None, stream=None):
    """lla_gdn_decode_step: one token per (batch, head) on state [B,H,Ls,dk,dv]
    (updated in place).  Returns out [B,H,dv]."""
    lib = load()
    _need(state, "state", torch.float32, 5)
    B, H, Ls, dk, dv = state.shape
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need(t, n, q.dtype, 3)
    _need(g, "g", torch.float32, 2)
    _need(beta, "beta", torch.float32, 2)
    _need(lam, "lam", torch.float32, 3)
    _need(pos, "pos", torch.int64, 1)
    if q.shape != (B, H, dk) or k.shape != (B, H, dk) or v.shape != (B, H, dv) or \
            lam.shape != (B, H, Ls + 1) or pos.shape != (B,):
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((B, H, dv), dtype=torch.float32, device=q.device)
    rc = lib.lla_gdn_decode_step(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                 _ptr(lam), _ptr(out), _ptr(pos), B, H, dk, dv, Ls, _dt(q),
                                 _ptr(device_error) if device_error is not None else None,
                                 _stream(stream))
    _check("lla_gdn_decode_step", rc)
    return out


def fwd_host(q, k, v, g, lam, out=None, chunk: int = 64, out_dtype=torch.float32, group: int = 0,
             workspace=None, device_error=None, stream=None, device=None):
    """lla_fwd_host: the forward on CPU tensors (pin them for overlap), run on
    `device`; returns the CPU output (valid once `stream` is synchronised)."""
    lib = load()
    for n, t in (("q", q), ("k", k), ("v", v), ("g", g), ("lam", lam)):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CPU tensor")
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=out_dtype, pin_memory=True)
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    need = lib.lla_fwd_host_workspace_bytes(B, H, T, dk, dv, chunk, _dt(q), _dt(out), group)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    with torch.cuda.device(device):
        rc = lib.lla_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(lam), _ptr(out), B, H, T, dk, dv,
                              chunk, _dt(q), _dt(out), group, _ptr(workspace), workspace.numel(),
                              _err_ptr(device_error), _stream(stream))
    _check("lla_fwd_host", rc)
    return out
