"""fp64 CPU oracle for log-linear attention (Log-Linear Mamba-2 form).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  The CUDA library and its Python
binding never import this package, and this package imports nothing from
them.  The arithmetic lives in ``lla_oracle.c`` (plain loops, fp64, OpenMP
over independent (batch, head) pairs); this module only compiles it with gcc
and marshals numpy arrays.

What each function follows (page "Log-Linear Attention", gist.science
2506.04761, technical summary):
  naive              §2.2 output equation, written as the double sum over keys
                     with the Mamba-2 gate of §3 (naive_rows: selected rows);
  fenwick            §2.2 Fenwick buckets + §2.3 recurrent form, per token;
  decode_step        §2.3 recurrent form on a lazily decayed level state;
  state_closed_form  §2.2 bucket states straight from the level definition;
  ssd                the plain gated linear-attention scan (§1 / §3 Mamba-2),
                     which the operator reduces to when every lambda is 1;
  lambda_mlp         page "Adaptive memory decay for Log-Linear Attention",
                     §LambdaMLPSoftplus: lambda = softplus((d W1) W2 + b);
  backward           the derivatives of the §2.2 double sum, term by term
                     (the pages give no backward; see the C source);
  gdn_*              Log-Linear Gated DeltaNet (§3 names it, gives no formula):
                     per-bucket Gated DeltaNet states read out with lambda,
                     in a pair form (gdn_naive), a recurrent form
                     (gdn_fenwick, gdn_decode_step) and the base model
                     (gdn_base).
Every function is pinned by tests in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liblla_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``lla_oracle.c`` into ``liblla_oracle.so`` beside it."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int64
        lib.oracle_naive.argtypes = [P] * 6 + [I] * 6
        lib.oracle_naive_rows.argtypes = [P] * 7 + [I] * 5
        lib.oracle_fenwick.argtypes = [P] * 6 + [I] * 6 + [P]
        lib.oracle_decode_step.argtypes = [P] * 9 + [I] * 5
        lib.oracle_state_closed_form.argtypes = [P] * 6 + [I] * 6
        lib.oracle_ssd.argtypes = [P] * 5 + [I] * 5
        lib.oracle_level.argtypes = [I, I]
        lib.oracle_lambda_mlp.argtypes = [P] * 5 + [I] * 3
        lib.oracle_backward.argtypes = [P] * 11 + [I] * 6
        lib.oracle_backward_rows.argtypes = [P] * 7 + [I, P, I] + [P] * 4 + [I] * 4
        lib.oracle_gdn_naive.argtypes = [P] * 7 + [I] * 6
        lib.oracle_gdn_fenwick.argtypes = [P] * 7 + [I] * 6
        lib.oracle_gdn_base.argtypes = [P] * 6 + [I] * 5
        lib.oracle_gdn_decode_step.argtypes = [P] * 9 + [I] * 5
        for name in ("oracle_naive", "oracle_naive_rows", "oracle_fenwick", "oracle_decode_step",
                     "oracle_state_closed_form", "oracle_ssd", "oracle_level", "oracle_lambda_mlp",
                     "oracle_num_threads", "oracle_backward", "oracle_backward_rows", "oracle_gdn_naive",
                     "oracle_gdn_fenwick", "oracle_gdn_base", "oracle_gdn_decode_step"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # a torch tensor: promote the stored values exactly
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, name: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{name} failed with code {rc}")


def num_threads() -> int:
    return _load().oracle_num_threads()


def num_levels(T: int) -> int:
    """L = 1 + bit_length(T-1): level 0 (the token itself) plus the Fenwick
    levels of the longest prefix [0, T-1)."""
    return 1 + max(T - 1, 0).bit_length()


def level(t: int, s: int) -> int:
    return _load().oracle_level(t, s)


def naive(q, k, v, g, lam) -> np.ndarray:
    q, k, v, g, lam = map(_f64, (q, k, v, g, lam))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    L = lam.shape[-1]
    out = np.zeros((B, H, T, dv), np.float64)
    _check(_load().oracle_naive(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(lam),
                                _ptr(out), B, H, T, dk, dv, L), "oracle_naive")
    return out


def naive_rows(q, k, v, g, lam, rows) -> np.ndarray:
    """Rows ``rows`` of the double sum for ONE (batch, head) slice:
    q,k [T,dk], v [T,dv], g [T], lam [T,L].  Returns [len(rows), dv]."""
    q, k, v, g, lam = map(_f64, (q, k, v, g, lam))
    rows = np.ascontiguousarray(np.asarray(rows), dtype=np.int64)
    T, dk = q.shape
    dv = v.shape[-1]
    L = lam.shape[-1]
    out = np.zeros((len(rows), dv), np.float64)
    _check(_load().oracle_naive_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(lam), _ptr(rows),
                                     _ptr(out), len(rows), T, dk, dv, L), "oracle_naive_rows")
    return out


def fenwick(q, k, v, g, lam, return_live_counts: bool = False):
    q, k, v, g, lam = map(_f64, (q, k, v, g, lam))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    L = lam.shape[-1]
    out = np.zeros((B, H, T, dv), np.float64)
    live = np.zeros((B, H, T), np.int32)
    _check(_load().oracle_fenwick(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(lam),
                                  _ptr(out), B, H, T, dk, dv, L, _ptr(live)),
           "oracle_fenwick")
    return (out, live) if return_live_counts else out


def decode_step(S, d, q, k, v, g, lam, pos):
    """One decode step.  ``S`` [B,H,Ls,dk,dv] and ``d`` [B,H,Ls] are fp64
    arrays updated in place; returns out [B,H,dv]."""
    assert S.dtype == np.float64 and S.flags.c_contiguous
    assert d.dtype == np.float64 and d.flags.c_contiguous
    q, k, v, g, lam = map(_f64, (q, k, v, g, lam))
    pos = np.ascontiguousarray(np.asarray(pos), dtype=np.int64)
    B, H, Ls, dk, dv = S.shape
    out = np.zeros((B, H, dv), np.float64)
    _check(_load().oracle_decode_step(_ptr(S), _ptr(d), _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(g), _ptr(lam), _ptr(out), _ptr(pos),
                                      B, H, dk, dv, Ls), "oracle_decode_step")
    return out


def state_closed_form(k, v, g, pos, Ls: int):
    """Decode state [B,H,Ls,dk,dv] (+ zero log-decay [B,H,Ls]) of the prefixes
    [0, pos[b]) of k [B,H,Tp,dk], v [B,H,Tp,dv], g [B,H,Tp]."""
    k, v, g = map(_f64, (k, v, g))
    pos = np.ascontiguousarray(np.asarray(pos), dtype=np.int64)
    B, H, Tp, dk = k.shape
    dv = v.shape[-1]
    S = np.zeros((B, H, Ls, dk, dv), np.float64)
    d = np.zeros((B, H, Ls), np.float64)
    _check(_load().oracle_state_closed_form(_ptr(k), _ptr(v), _ptr(g), _ptr(pos),
                                            _ptr(S), _ptr(d), B, H, Tp, dk, dv, Ls),
           "oracle_state_closed_form")
    return S, d


def ssd(q, k, v, g) -> np.ndarray:
    q, k, v, g = map(_f64, (q, k, v, g))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, H, T, dv), np.float64)
    _check(_load().oracle_ssd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(out),
                              B, H, T, dk, dv), "oracle_ssd")
    return out


def lambda_mlp(d, W1, W2, b) -> np.ndarray:
    """lambda [..., L] = softplus((d W1) W2 + b) for d [..., Dd], W1 [Dd, 2L],
    W2 [2L, L], b [L]."""
    d, W1, W2, b = map(_f64, (d, W1, W2, b))
    lead = d.shape[:-1]
    Dd = d.shape[-1]
    L = b.shape[0]
    assert W1.shape == (Dd, 2 * L) and W2.shape == (2 * L, L)
    dd = np.ascontiguousarray(d.reshape(-1, Dd))
    out = np.zeros((dd.shape[0], L), np.float64)
    _check(_load().oracle_lambda_mlp(_ptr(dd), _ptr(W1), _ptr(W2), _ptr(b), _ptr(out),
                                     dd.shape[0], Dd, L), "oracle_lambda_mlp")
    return out.reshape(*lead, L)


def backward(q, k, v, g, lam, dout):
    """Gradients (dq, dk, dv, dg, dlam) of sum(dout * naive(q, k, v, g, lam))."""
    q, k, v, g, lam, dout = map(_f64, (q, k, v, g, lam, dout))
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    L = lam.shape[-1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dg = np.zeros_like(g)
    dlam = np.zeros_like(lam)
    _check(_load().oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(lam), _ptr(dout),
                                   _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dlam),
                                   B, H, T, Dk, Dv, L), "oracle_backward")
    return dq, dk, dv, dg, dlam


def gdn_naive(q, k, v, g, beta, lam) -> np.ndarray:
    q, k, v, g, beta, lam = map(_f64, (q, k, v, g, beta, lam))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, H, T, dv), np.float64)
    _check(_load().oracle_gdn_naive(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(lam),
                                    _ptr(out), B, H, T, dk, dv, lam.shape[-1]), "oracle_gdn_naive")
    return out


def gdn_fenwick(q, k, v, g, beta, lam) -> np.ndarray:
    q, k, v, g, beta, lam = map(_f64, (q, k, v, g, beta, lam))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, H, T, dv), np.float64)
    _check(_load().oracle_gdn_fenwick(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(lam),
                                      _ptr(out), B, H, T, dk, dv, lam.shape[-1]), "oracle_gdn_fenwick")
    return out


def gdn_base(q, k, v, g, beta) -> np.ndarray:
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, H, T, dv), np.float64)
    _check(_load().oracle_gdn_base(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(out),
                                   B, H, T, dk, dv), "oracle_gdn_base")
    return out


def gdn_decode_step(S, q, k, v, g, beta, lam, pos) -> np.ndarray:
    """One step on the eager level state S [B,H,Ls,dk,dv] (updated in place);
    returns out [B,H,dv]."""
    assert S.dtype == np.float64 and S.flags.c_contiguous
    q, k, v, g, beta, lam = map(_f64, (q, k, v, g, beta, lam))
    pos = np.ascontiguousarray(np.asarray(pos), dtype=np.int64)
    B, H, Ls, dk, dv = S.shape
    out = np.zeros((B, H, dv), np.float64)
    _check(_load().oracle_gdn_decode_step(_ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                          _ptr(lam), _ptr(out), _ptr(pos), B, H, dk, dv, Ls),
           "oracle_gdn_decode_step")
    return out


def backward_rows(q, k, v, g, lam, dout, query_rows, key_rows):
    """The backward of one (batch, head) slice at selected rows:
    (dq [nq,dk], dlam [nq,L]) at query_rows, (dk [ns,dk], dv [ns,dv]) at key_rows."""
    q, k, v, g, lam, dout = map(_f64, (q, k, v, g, lam, dout))
    T, Dk = q.shape
    Dv = v.shape[-1]
    L = lam.shape[-1]
    tq = np.ascontiguousarray(np.asarray(query_rows), dtype=np.int64)
    ts = np.ascontiguousarray(np.asarray(key_rows), dtype=np.int64)
    dq = np.zeros((len(tq), Dk))
    dl = np.zeros((len(tq), L))
    dk = np.zeros((len(ts), Dk))
    dv = np.zeros((len(ts), Dv))
    _check(_load().oracle_backward_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(lam), _ptr(dout),
                                        _ptr(tq), len(tq), _ptr(ts), len(ts), _ptr(dq), _ptr(dl),
                                        _ptr(dk), _ptr(dv), T, Dk, Dv, L), "oracle_backward_rows")
    return dq, dl, dk, dv
