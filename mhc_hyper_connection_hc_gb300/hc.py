"""Thin Python binding of the C ABI in include/hc.h.

Argument marshalling only: each function takes torch CUDA tensors, checks their
dtype, device and contiguity, passes raw device pointers, sizes and the CUDA
stream handle to the C entry point of the same name, and raises HcError on a
non-zero status.  hc_pre_fused, hc_post and hc_post_pre_fused can instead return a
Prepared call (prepare=True) that repeats the same call without re-checking.  Every step of the site program runs in the library's CUDA
kernels; there is no fallback.  If the library has not been built the first
call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmhc_gb300.so")

HC_OK = 0
HC_ERR_NULL, HC_ERR_DIM, HC_ERR_ALIGN, HC_ERR_ALIAS = 1, 2, 3, 4
HC_ERR_WORKSPACE, HC_ERR_CUDA, HC_ERR_DEVICE, HC_ERR_UNSUPPORTED = 5, 6, 7, 8
HC_ERR_TOO_LARGE = 9
HC_PATH_AUTO, HC_PATH_GENERIC, HC_PATH_CLUSTER, HC_PATH_WIDE = 0, 1, 2, 3

EXPORTED = ("hc_status_string", "hc_expand", "hc_pre_workspace_bytes", "hc_workspace_init",
            "hc_workspace_status", "hc_pre_fused", "hc_pre_fused_path", "hc_pre_auto_path", "hc_pre_helper_tokens",
            "hc_post", "hc_mean", "hc_pre_fused_noalloc", "hc_head", "hc_head_path",
            "hc_post_pre_fused", "hc_post_pre_fused_path", "hc_rms_norm_q8", "hc_pre_fused_norm",
            "hc_pre_fused_norm_path")


class HcError(RuntimeError):
    def __init__(self, fn: str, rc: int):
        self.rc = rc
        super().__init__(f"{fn} failed: status {rc} ({status_string(rc)})")


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Open the CUDA library (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.hc_status_string.argtypes, lib.hc_status_string.restype = [i], ctypes.c_char_p
    lib.hc_expand.argtypes = [vp, vp, i, i, i, vp]
    lib.hc_mean.argtypes = [vp, vp, i, i, i, vp]
    lib.hc_post.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp]
    lib.hc_pre_workspace_bytes.argtypes, lib.hc_pre_workspace_bytes.restype = [i, i, i], sz
    lib.hc_workspace_init.argtypes = [vp, sz, vp]
    lib.hc_workspace_status.argtypes = [vp, vp]
    lib.hc_pre_auto_path.argtypes = [i, i, i]
    lib.hc_pre_helper_tokens.argtypes = [i, i, i, i, sz]
    pre_args = [vp, vp, vp, vp, i, i, i, i, f, vp, vp, vp, vp, vp, sz, vp]
    lib.hc_pre_fused.argtypes = pre_args
    lib.hc_pre_fused_path.argtypes = pre_args + [i]
    lib.hc_pre_fused_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, f, vp, vp, vp, vp, vp]
    head_args = [vp, vp, vp, vp, i, i, i, f, vp, vp, vp, sz, vp]
    lib.hc_head.argtypes = head_args
    lib.hc_head_path.argtypes = head_args + [i]
    fused_args = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.hc_post_pre_fused.argtypes = fused_args
    lib.hc_post_pre_fused_path.argtypes = fused_args + [i]
    lib.hc_rms_norm_q8.argtypes = [vp, vp, i, i, f, vp, vp, vp, vp]
    lib.hc_pre_fused_norm.argtypes = [vp, vp, vp, vp, i, i, i, i, f, vp, f, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.hc_pre_fused_norm_path.argtypes = lib.hc_pre_fused_norm.argtypes + [i]
    for name in EXPORTED[1:]:
        if name != "hc_pre_workspace_bytes":
            getattr(lib, name).restype = i
    _lib = lib
    return lib


def status_string(rc: int) -> str:
    return load().hc_status_string(int(rc)).decode()


def _check(fn: str, rc: int) -> None:
    if rc != HC_OK:
        raise HcError(fn, rc)


def _ptr(t: torch.Tensor | None, name: str, dtype=torch.float32):
    """The tensor's device address as an int (None for no tensor or an empty one), after
    checking device, dtype and contiguity; the common case costs four attribute reads."""
    if t is None:
        return None
    if isinstance(t, torch.Tensor) and t.is_cuda and t.dtype is dtype and t.is_contiguous():
        return t.data_ptr() if t.numel() else None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    raise ValueError(f"{name} must be contiguous")


# The current stream's raw handle without building a torch.cuda.Stream object (about 3 us
# per call through torch.cuda.current_stream()); the public call where it is missing.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    """The CUDA stream handle to pass: `stream` (a torch.cuda.Stream or a raw handle), or
    the current device's current stream when it is None."""
    if stream is None:
        if _raw_stream is not None:
            return int(_raw_stream(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


class Prepared:
    """One library call whose arguments were checked and converted once.  Calling it runs
    the C entry point again on the same device pointers, sizes and stream, with none of
    the per-call Python checks: the decode loop's form of a call (the tensors must stay
    alive, at the same addresses and shapes, for as long as it is used; their contents
    may change between calls)."""

    __slots__ = ("_fn", "_name", "_args", "_keep")

    def __init__(self, name: str, args: tuple, keep: tuple):
        self._fn = getattr(load(), name)
        self._name = name
        self._args = args
        self._keep = keep   # the tensors the pointers belong to

    def __call__(self) -> None:
        rc = self._fn(*self._args)
        if rc != HC_OK:
            raise HcError(self._name, rc)


def _run(name: str, args: tuple, prepare: bool, keep: tuple):
    if prepare:
        return Prepared(name, args, keep)
    _check(name, getattr(load(), name)(*args))
    return None


def _shape(x: torch.Tensor):
    shape = x.shape
    if len(shape) != 3:
        raise ValueError("stream state must be [T, s, d]")
    return shape[0], shape[1], shape[2]


def hc_expand(emb: torch.Tensor, x: torch.Tensor, stream=None) -> None:
    T, s, d = _shape(x)
    _check("hc_expand", load().hc_expand(_ptr(emb, "emb"), _ptr(x, "x"), T, s, d, _stream(stream)))


def hc_mean(x: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    T, s, d = _shape(x)
    _check("hc_mean", load().hc_mean(_ptr(x, "x"), _ptr(out, "out"), T, s, d, _stream(stream)))


def hc_post(x, f, post, comb, x_out, stream=None, prepare: bool = False):
    """x_out = post . f + comb^T x.  With prepare=True, returns a Prepared call instead."""
    T, s, d = _shape(x)
    args = (_ptr(x, "x"), _ptr(f, "f"), _ptr(post, "post"), _ptr(comb, "comb"), _ptr(x_out, "x_out"), T, s, d,
            _stream(stream))
    return _run("hc_post", args, prepare, (x, f, post, comb, x_out))


def hc_pre_workspace_bytes(T: int, s: int, d: int) -> int:
    return int(load().hc_pre_workspace_bytes(T, s, d))


def hc_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    _check("hc_workspace_init", load().hc_workspace_init(
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)))


def hc_workspace_status(workspace: torch.Tensor, stream=None) -> int:
    return int(load().hc_workspace_status(_ptr(workspace, "workspace", torch.uint8), _stream(stream)))


def hc_pre_auto_path(T: int, s: int, d: int) -> int:
    return int(load().hc_pre_auto_path(T, s, d))


def hc_pre_helper_tokens(T: int, s: int, d: int, fused: bool, ws_bytes: int) -> int:
    """Tokens the cluster path's helper kernel takes from the end of such a batch (0: none)."""
    return int(load().hc_pre_helper_tokens(T, s, d, int(bool(fused)), int(ws_bytes)))


def hc_pre_fused(x, fn_w, scale, base, iters: int, eps: float, pre, post, comb, y, workspace,
                 stream=None, path: int | None = None, prepare: bool = False):
    """The site's pre-chain.  With prepare=True, returns a Prepared call instead."""
    T, s, d = _shape(x)
    args = (_ptr(x, "x"), _ptr(fn_w, "fn_w"), _ptr(scale, "scale"), _ptr(base, "base"), T, s, d,
            int(iters), float(eps), _ptr(pre, "pre"), _ptr(post, "post"), _ptr(comb, "comb"),
            _ptr(y, "y"), _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
            _stream(stream))
    keep = (x, fn_w, scale, base, pre, post, comb, y, workspace)
    if path is None:
        return _run("hc_pre_fused", args, prepare, keep)
    return _run("hc_pre_fused_path", args + (int(path),), prepare, keep)


def hc_pre_fused_noalloc(x, fn_w, scale, base, iters: int, eps: float, pre, post, comb, y,
                         stream=None) -> None:
    """hc_pre_fused without a workspace, for callers that cannot allocate device memory
    when they run a site (the scratch is a static buffer inside the library; see hc.h)."""
    T, s, d = _shape(x)
    _check("hc_pre_fused_noalloc", load().hc_pre_fused_noalloc(
        _ptr(x, "x"), _ptr(fn_w, "fn_w"), _ptr(scale, "scale"), _ptr(base, "base"), T, s, d,
        int(iters), float(eps), _ptr(pre, "pre"), _ptr(post, "post"), _ptr(comb, "comb"),
        _ptr(y, "y"), _stream(stream)))


def hc_rms_norm_q8(y, norm_w, eps_norm: float, z, q=None, q_scale=None, stream=None) -> None:
    """Branch-input norm z = y * rsqrt(mean(y^2) + eps_norm) * norm_w, and optionally its
    Q8_0 pair q (int8 [T, d]) and q_scale ([T, d/32])."""
    if y.dim() != 2:
        raise ValueError("y must be [T, d]")
    T, d = int(y.shape[0]), int(y.shape[1])
    _check("hc_rms_norm_q8", load().hc_rms_norm_q8(
        _ptr(y, "y"), _ptr(norm_w, "norm_w"), T, d, float(eps_norm), _ptr(z, "z"),
        _ptr(q, "q", torch.int8), _ptr(q_scale, "q_scale"), _stream(stream)))


def hc_pre_fused_norm(x, fn_w, scale, base, iters: int, eps: float, norm_w, eps_norm: float, pre, post,
                      comb, y, z, workspace, q=None, q_scale=None, stream=None, path: int | None = None,
                      prepare: bool = False):
    """The pre-chain and the branch-input norm of its y (z, and the Q8_0 pair q / q_scale
    if given): one launch on the cluster path where the shape allows, else hc_pre_fused
    then hc_rms_norm_q8.  With prepare=True, returns a Prepared call instead."""
    T, s, d = _shape(x)
    args = (_ptr(x, "x"), _ptr(fn_w, "fn_w"), _ptr(scale, "scale"), _ptr(base, "base"), T, s, d, int(iters),
            float(eps), _ptr(norm_w, "norm_w"), float(eps_norm), _ptr(pre, "pre"), _ptr(post, "post"),
            _ptr(comb, "comb"), _ptr(y, "y"), _ptr(z, "z"), _ptr(q, "q", torch.int8), _ptr(q_scale, "q_scale"),
            _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    keep = (x, fn_w, scale, base, norm_w, pre, post, comb, y, z, q, q_scale, workspace)
    if path is None:
        return _run("hc_pre_fused_norm", args, prepare, keep)
    return _run("hc_pre_fused_norm_path", args + (int(path),), prepare, keep)


def hc_post_pre_fused(x_prev, f, post_prev, comb_prev, fn_w, scale, base, iters: int, eps: float,
                      x_new, pre, post, comb, y, workspace, stream=None, path: int | None = None,
                      prepare: bool = False):
    """Site i's hc_post and site i+1's pre-chain in one call: x_new = post_prev . f +
    comb_prev^T x_prev, then pre/post/comb/y of the next site on x_new.  With
    prepare=True, returns a Prepared call instead."""
    T, s, d = _shape(x_prev)
    args = (_ptr(x_prev, "x_prev"), _ptr(f, "f"), _ptr(post_prev, "post_prev"),
            _ptr(comb_prev, "comb_prev"), _ptr(fn_w, "fn_w"), _ptr(scale, "scale"), _ptr(base, "base"),
            T, s, d, int(iters), float(eps), _ptr(x_new, "x_new"), _ptr(pre, "pre"), _ptr(post, "post"),
            _ptr(comb, "comb"), _ptr(y, "y"), _ptr(workspace, "workspace", torch.uint8),
            workspace.numel(), _stream(stream))
    keep = (x_prev, f, post_prev, comb_prev, fn_w, scale, base, x_new, pre, post, comb, y, workspace)
    if path is None:
        return _run("hc_post_pre_fused", args, prepare, keep)
    return _run("hc_post_pre_fused_path", args + (int(path),), prepare, keep)


def hc_head(x, fn_w, scale, base, eps: float, y, workspace, gates=None, stream=None,
            path: int | None = None) -> None:
    """Gated-head trunk exit: x [T, s, d] -> y [T, d] (and gates [T, s] if given)."""
    T, s, d = _shape(x)
    args = (_ptr(x, "x"), _ptr(fn_w, "fn_w"), _ptr(scale, "scale"), _ptr(base, "base"), T, s, d,
            float(eps), _ptr(gates, "gates"), _ptr(y, "y"), _ptr(workspace, "workspace", torch.uint8),
            workspace.numel(), _stream(stream))
    if path is None:
        _check("hc_head", load().hc_head(*args))
    else:
        _check("hc_head_path", load().hc_head_path(*args, int(path)))


# ----------------------------------------------------------------------------- conveniences
# Allocation helpers (PyTorch owns device memory; the library never allocates).


def new_workspace(T: int, s: int, d: int, device="cuda", stream=None) -> torch.Tensor:
    """A zero-initialised workspace of hc_pre_workspace_bytes(T, s, d) bytes."""
    ws = torch.empty(max(256, hc_pre_workspace_bytes(T, s, d)), dtype=torch.uint8, device=device)
    hc_workspace_init(ws, stream)
    return ws


def new_pre_outputs(T: int, s: int, d: int, device="cuda"):
    kw = dict(dtype=torch.float32, device=device)
    return dict(pre=torch.empty(T, s, **kw), post=torch.empty(T, s, **kw),
                comb=torch.empty(T, s, s, **kw), y=torch.empty(T, d, **kw))
