"""CPU oracle of the mHC site program -- TEST INFRASTRUCTURE.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import
this package.  The CUDA library and its Python binding never do, and this
package imports nothing from them.  It wraps oracle/hc_oracle.c (float64 plain
loops, one token at a time; see that file's header for the formulas and the
pages they follow).  Inputs may be float32 or float64 arrays; they are widened
to float64 before the call, so float32 inputs are used bit-for-bit.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.hco_pre.argtypes = [dp, dp, dp, dp, ctypes.c_long, ctypes.c_int, ctypes.c_long,
                                ctypes.c_int, ctypes.c_double, dp, dp, dp, dp, dp, dp, ctypes.c_int]
        lib.hco_post.argtypes = [dp, dp, dp, dp, dp, ctypes.c_long, ctypes.c_int, ctypes.c_long,
                                 ctypes.c_int]
        lib.hco_expand.argtypes = [dp, dp, ctypes.c_long, ctypes.c_int, ctypes.c_long]
        lib.hco_mean.argtypes = [dp, dp, ctypes.c_long, ctypes.c_int, ctypes.c_long]
        lib.hco_head.argtypes = [dp, dp, dp, dp, ctypes.c_long, ctypes.c_int, ctypes.c_long,
                                 ctypes.c_double, dp, dp, ctypes.c_int]
        lib.hco_rms_norm.argtypes = [dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_double, dp]
        fp = ctypes.POINTER(ctypes.c_float)
        lib.hco_q8_blocks_f32.argtypes = [fp, ctypes.c_long, ctypes.POINTER(ctypes.c_byte), fp]
        for fn in (lib.hco_pre, lib.hco_post, lib.hco_expand, lib.hco_mean, lib.hco_head, lib.hco_rms_norm,
                   lib.hco_q8_blocks_f32):
            fn.restype = ctypes.c_int
        lib.hco_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.float64)


def _p(a: np.ndarray | None):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().hco_max_threads())


def default_threads() -> int:
    return max(1, min(max_threads(), os.cpu_count() or 1))


def pre(x, fn_w, scale, base, iters: int, eps: float, want_mixes: bool = False,
        threads: int | None = None):
    """Pre-chain of one site.  x [T, s, d] -> dict(pre [T,s], post [T,s], comb [T,s,s],
    y [T,d], and with want_mixes also mixes [T,R] (rescaled) and logits [T,R])."""
    x = _f64(x)
    T, s, d = x.shape
    R = (2 + s) * s
    fn_w = _f64(fn_w).reshape(R, s * d)
    scale, base = _f64(scale).reshape(3), _f64(base).reshape(R)
    out = dict(pre=np.empty((T, s)), post=np.empty((T, s)), comb=np.empty((T, s, s)),
               y=np.empty((T, d)))
    mixes = np.empty((T, R)) if want_mixes else None
    logits = np.empty((T, R)) if want_mixes else None
    rc = _load().hco_pre(_p(x), _p(fn_w), _p(scale), _p(base), T, s, d, int(iters), float(eps),
                         _p(out["pre"]), _p(out["post"]), _p(out["comb"]), _p(out["y"]),
                         _p(mixes), _p(logits), threads or default_threads())
    if rc != 0:
        raise ValueError(f"hco_pre failed with code {rc}")
    if want_mixes:
        out["mixes"], out["logits"] = mixes, logits
    return out


def post(x, f, post_gates, comb, threads: int | None = None) -> np.ndarray:
    """hc_post: x [T,s,d], f [T,d], post [T,s], comb [T,s,s] -> x' [T,s,d]."""
    x = _f64(x)
    T, s, d = x.shape
    f, pg, cb = _f64(f).reshape(T, d), _f64(post_gates).reshape(T, s), _f64(comb).reshape(T, s, s)
    out = np.empty((T, s, d))
    rc = _load().hco_post(_p(x), _p(f), _p(pg), _p(cb), _p(out), T, s, d,
                          threads or default_threads())
    if rc != 0:
        raise ValueError(f"hco_post failed with code {rc}")
    return out


def head(x, fn_w, scale, base, eps: float, threads: int | None = None):
    """Gated-head trunk exit: x [T, s, d], fn_w [s, s*d], scale [1], base [s]
    -> dict(gates [T, s], y [T, d])."""
    x = _f64(x)
    T, s, d = x.shape
    fn_w = _f64(fn_w).reshape(s, s * d)
    scale, base = _f64(scale).reshape(1), _f64(base).reshape(s)
    out = dict(gates=np.empty((T, s)), y=np.empty((T, d)))
    rc = _load().hco_head(_p(x), _p(fn_w), _p(scale), _p(base), T, s, d, float(eps),
                          _p(out["gates"]), _p(out["y"]), threads or default_threads())
    if rc != 0:
        raise ValueError(f"hco_head failed with code {rc}")
    return out


def rms_norm(y, norm_w, eps_norm: float) -> np.ndarray:
    """Branch-input norm: y [T, d], norm_w [d] -> z [T, d] (float64)."""
    y = _f64(y)
    T, d = y.shape
    nw = _f64(norm_w).reshape(d)
    z = np.empty((T, d))
    if _load().hco_rms_norm(_p(y), _p(nw), T, d, float(eps_norm), _p(z)) != 0:
        raise ValueError("hco_rms_norm failed")
    return z


def q8_blocks(z32):
    """Q8_0 blocks of 32 along the last axis, decided in float32: z [..., n] float32 ->
    (q int8 [..., n], scale float32 [..., n/32])."""
    z32 = np.ascontiguousarray(np.asarray(z32), dtype=np.float32)
    n = z32.size
    q = np.empty(z32.shape, dtype=np.int8)
    sc = np.empty(z32.shape[:-1] + (z32.shape[-1] // 32,), dtype=np.float32)
    rc = _load().hco_q8_blocks_f32(z32.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), n,
                                   q.ctypes.data_as(ctypes.POINTER(ctypes.c_byte)),
                                   sc.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    if rc != 0:
        raise ValueError("hco_q8_blocks_f32 failed (the last axis must be a multiple of 32)")
    return q, sc


def expand(emb, s: int) -> np.ndarray:
    emb = _f64(emb)
    T, d = emb.shape
    out = np.empty((T, s, d))
    if _load().hco_expand(_p(emb), _p(out), T, s, d) != 0:
        raise ValueError("hco_expand failed")
    return out


def mean(x) -> np.ndarray:
    x = _f64(x)
    T, s, d = x.shape
    out = np.empty((T, d))
    if _load().hco_mean(_p(x), _p(out), T, s, d) != 0:
        raise ValueError("hco_mean failed")
    return out


def site(x, fn_w, scale, base, f, iters: int, eps: float, threads: int | None = None):
    """One whole site: pre-chain, then hc_post with the given branch output f."""
    r = pre(x, fn_w, scale, base, iters, eps, threads=threads)
    r["x_out"] = post(x, f, r["post"], r["comb"], threads=threads)
    return r
