"""CPU-only checks of the C ABI: the library loads, exports every function that
include/hc.h declares, and refuses bad arguments on the host before any CUDA
call (fake pointers are passed; none of these cases reaches a launch).

Fake device addresses must never reach a GPU: if a regression moved a host check
after a launch, a kernel would dereference them.  So in a process that can see a
GPU these tests do not run directly; test_host_checks_in_a_process_without_devices
runs them (and the no-alloc size check) in a child process with no device visible,
where such a regression fails with a CUDA error instead."""

import ctypes
import math
import os
import re
import subprocess
import sys

import pytest

from mhc_hyper_connection_hc_gb300 import hc


def _device_visible() -> bool:
    if os.environ.get("CUDA_VISIBLE_DEVICES") == "":
        return False
    try:
        import torch
        return bool(torch.cuda.is_available())
    except Exception:
        return False


DEVICE_VISIBLE = _device_visible()
fake_addresses = pytest.mark.skipif(
    DEVICE_VISIBLE, reason="fake device addresses: run in a child process without devices")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hc.h")

A = 0x10000000   # fake, 16-byte aligned "device" addresses; never dereferenced
MB = 1 << 20


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hc_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from mhc_hyper_connection_hc_gb300 import build
    build.build()
    return hc.load()


@fake_addresses
def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/hc.h but not exported"
    assert set(names) >= set(hc.EXPORTED)


@fake_addresses
def test_status_strings(lib):
    for rc in range(0, 9):
        assert len(hc.status_string(rc)) >= 2
    assert hc.status_string(99) == "unknown status"


def post_rc(lib, x=A, f=A + 64 * MB, post=A + 96 * MB, comb=A + 97 * MB, out=A + 128 * MB,
            T=2, s=4, d=4096):
    return lib.hc_post(x, f, post, comb, out, T, s, d, None)


@fake_addresses
def test_post_validation(lib):
    assert post_rc(lib, x=0) == hc.HC_ERR_NULL
    assert post_rc(lib, out=0) == hc.HC_ERR_NULL
    assert post_rc(lib, T=-1) == hc.HC_ERR_DIM
    assert post_rc(lib, s=0) == hc.HC_ERR_DIM
    assert post_rc(lib, s=9) == hc.HC_ERR_DIM
    assert post_rc(lib, d=2) == hc.HC_ERR_DIM
    assert post_rc(lib, d=4098) == hc.HC_ERR_ALIGN
    assert post_rc(lib, x=A + 4) == hc.HC_ERR_ALIGN
    assert post_rc(lib, comb=A + 97 * MB + 2) == hc.HC_ERR_ALIGN
    assert post_rc(lib, out=A) == hc.HC_ERR_ALIAS                    # in place
    assert post_rc(lib, out=A + 64 * MB - 16) == hc.HC_ERR_ALIAS     # partial overlap with f
    assert post_rc(lib, T=1 << 20, d=4096) == hc.HC_ERR_DIM          # T*s*d >= 2^31
    assert post_rc(lib, T=0, x=0, f=0, out=0) == hc.HC_OK            # empty batch


@fake_addresses
def test_expand_mean_validation(lib):
    assert lib.hc_expand(A, A, 2, 4, 64, None) == hc.HC_ERR_ALIAS
    assert lib.hc_expand(0, A, 2, 4, 64, None) == hc.HC_ERR_NULL
    assert lib.hc_mean(A, A + 8, 2, 4, 64, None) == hc.HC_ERR_ALIGN
    assert lib.hc_mean(A, A + 1024, 2, 4, 64, None) == hc.HC_ERR_ALIAS
    assert lib.hc_mean(A, A + MB, 0, 4, 64, None) == hc.HC_OK


def pre_rc(lib, T=3, s=4, d=4096, iters=20, eps=1e-6, ws_bytes=None, path=0, **over):
    R = (2 + s) * s
    p = dict(x=A, fn_w=A + 16 * MB, scale=A + 32 * MB, base=A + 32 * MB + 64, pre=A + 33 * MB,
             post=A + 33 * MB + 4096, comb=A + 33 * MB + 8192, y=A + 34 * MB, ws=A + 64 * MB)
    p.update(over)
    if ws_bytes is None:
        ws_bytes = hc.hc_pre_workspace_bytes(max(T, 0), s, d)
    args = [p["x"], p["fn_w"], p["scale"], p["base"], T, s, d, iters, ctypes.c_float(eps),
            p["pre"], p["post"], p["comb"], p["y"], p["ws"], ws_bytes, None, path]
    return lib.hc_pre_fused_path(*args)


@fake_addresses
def test_pre_validation(lib):
    assert pre_rc(lib, iters=0) == hc.HC_ERR_DIM                     # zero iterations refused
    assert pre_rc(lib, eps=0.0) == hc.HC_ERR_DIM                     # eps <= 0 refused
    assert pre_rc(lib, eps=-1e-6) == hc.HC_ERR_DIM
    assert pre_rc(lib, eps=math.inf) == hc.HC_ERR_DIM
    assert pre_rc(lib, eps=math.nan) == hc.HC_ERR_DIM
    assert pre_rc(lib, s=0) == hc.HC_ERR_DIM
    assert pre_rc(lib, path=7) == hc.HC_ERR_DIM
    assert pre_rc(lib, x=0) == hc.HC_ERR_NULL
    assert pre_rc(lib, y=0) == hc.HC_ERR_NULL
    assert pre_rc(lib, x=A + 8) == hc.HC_ERR_ALIGN
    assert pre_rc(lib, d=4094) == hc.HC_ERR_ALIGN
    assert pre_rc(lib, pre=A + 1) == hc.HC_ERR_ALIGN
    assert pre_rc(lib, y=A + 256) == hc.HC_ERR_ALIAS                  # y inside x
    assert pre_rc(lib, post=A + 33 * MB + 4) == hc.HC_ERR_ALIAS       # post overlaps pre
    assert pre_rc(lib, ws=0) == hc.HC_ERR_WORKSPACE
    assert pre_rc(lib, ws_bytes=16) == hc.HC_ERR_WORKSPACE
    assert pre_rc(lib, ws=A + 64 * MB + 8) == hc.HC_ERR_WORKSPACE
    assert pre_rc(lib, ws=A + 34 * MB) == hc.HC_ERR_ALIAS             # workspace over y
    assert pre_rc(lib, T=0, x=0) == hc.HC_OK                          # empty batch


@fake_addresses
def test_workspace_sizes(lib):
    assert hc.hc_pre_workspace_bytes(0, 4, 4096) >= 256
    assert hc.hc_pre_workspace_bytes(1, 9, 4096) == 0
    for T in (1, 8, 37, 512, 4096):
        for s, d in ((4, 4096), (8, 7168), (1, 4), (3, 12)):
            n = hc.hc_pre_workspace_bytes(T, s, d)
            assert n >= 256 and n % 4 == 0
            generic = 256 + 4 * ((2 + s) * s + 1) * T * 304 + 4 * ((2 + s) * s + 1) * 304
            # the wide-stream path (s >= 5): per-tile counters and flags, and 64 slots of
            # per-CTA partials and of tile sums (R dots + squares for 4 tokens, at most 160
            # CTAs)
            ntiles = (T + 3) // 4
            rv = (2 + s) * s + 1
            wide = 256 + 12 * ntiles + 64 * (160 + 1) * 4 * rv * 4 + 3 * 256 if s >= 5 else 0
            assert n <= max(generic, wide)


def test_workspace_holds_the_helper_partials(lib):
    """Shapes the cluster path takes have room in hc_pre_workspace_bytes for the helper
    kernel's partials (after the 256-byte status word: 2 x 16 slices x RV floats a token);
    the helper query refuses bad dimensions and, without a device, reports no helper."""
    for T in (1, 37, 4096, 16390):
        for s, d in ((4, 4096), (3, 3072), (2, 2048), (1, 1024), (4, 1024)):
            rv = ((2 + s) * s + 1 + 3) // 4 * 4
            assert hc.hc_pre_workspace_bytes(T, s, d) >= 256 + T * 32 * rv * 4
    assert hc.hc_pre_helper_tokens(-1, 4, 4096, False, 1 << 30) == -1
    assert hc.hc_pre_helper_tokens(4096, 9, 4096, False, 1 << 30) == -1
    assert hc.hc_pre_helper_tokens(0, 4, 4096, True, 1 << 30) == 0
    if not DEVICE_VISIBLE:
        assert hc.hc_pre_helper_tokens(4096, 4, 4096, False, 1 << 30) == 0


def head_rc(lib, x=A, fn_w=A + 32 * MB, scale=A + 40 * MB, base=A + 40 * MB + 64, gates=A + 41 * MB,
            y=A + 42 * MB, ws=A + 64 * MB, ws_bytes=16 * MB, T=2, s=4, d=4096, eps=1e-6, path=0):
    return lib.hc_head_path(x, fn_w, scale, base, T, s, d, eps, gates, y, ws, ws_bytes, None, path)


@fake_addresses
def test_head_validation(lib):
    assert head_rc(lib, eps=0.0) == hc.HC_ERR_DIM
    assert head_rc(lib, eps=math.nan) == hc.HC_ERR_DIM
    assert head_rc(lib, s=9) == hc.HC_ERR_DIM
    assert head_rc(lib, path=5) == hc.HC_ERR_DIM
    assert head_rc(lib, x=0) == hc.HC_ERR_NULL
    assert head_rc(lib, y=0) == hc.HC_ERR_NULL
    assert head_rc(lib, fn_w=A + 8) == hc.HC_ERR_ALIGN
    assert head_rc(lib, gates=A + 41 * MB + 2) == hc.HC_ERR_ALIGN
    assert head_rc(lib, d=4094) == hc.HC_ERR_ALIGN
    assert head_rc(lib, y=A + 256) == hc.HC_ERR_ALIAS                 # y inside x
    assert head_rc(lib, gates=A + 42 * MB + 4) == hc.HC_ERR_ALIAS     # gates inside y
    assert head_rc(lib, ws=0) == hc.HC_ERR_WORKSPACE
    assert head_rc(lib, ws_bytes=16) == hc.HC_ERR_WORKSPACE
    assert head_rc(lib, ws=A + 42 * MB) == hc.HC_ERR_ALIAS            # workspace over y
    assert head_rc(lib, T=0, x=0) == hc.HC_OK                         # empty batch


def fused_rc(lib, T=2, s=4, d=4096, iters=20, eps=1e-6, path=0, **over):
    p = dict(x_prev=A, f=A + 8 * MB, post_prev=A + 9 * MB, comb_prev=A + 9 * MB + 4096,
             fn_w=A + 10 * MB, scale=A + 12 * MB, base=A + 12 * MB + 64, x_new=A + 13 * MB,
             pre=A + 14 * MB, post=A + 14 * MB + 4096, comb=A + 14 * MB + 8192, y=A + 15 * MB,
             ws=A + 64 * MB)
    p.update(over)
    ws_bytes = p.pop("ws_bytes", 16 * MB)
    return lib.hc_post_pre_fused_path(p["x_prev"], p["f"], p["post_prev"], p["comb_prev"], p["fn_w"],
                                      p["scale"], p["base"], T, s, d, iters, eps, p["x_new"], p["pre"],
                                      p["post"], p["comb"], p["y"], p["ws"], ws_bytes, None, path)


@fake_addresses
def test_post_pre_fused_validation(lib):
    assert fused_rc(lib, iters=0) == hc.HC_ERR_DIM
    assert fused_rc(lib, eps=0.0) == hc.HC_ERR_DIM
    assert fused_rc(lib, path=9) == hc.HC_ERR_DIM
    assert fused_rc(lib, f=0) == hc.HC_ERR_NULL
    assert fused_rc(lib, x_new=0) == hc.HC_ERR_NULL
    assert fused_rc(lib, f=A + 8 * MB + 4) == hc.HC_ERR_ALIGN
    assert fused_rc(lib, comb_prev=A + 9 * MB + 4098) == hc.HC_ERR_ALIGN
    assert fused_rc(lib, x_new=A) == hc.HC_ERR_ALIAS                   # in place refused
    assert fused_rc(lib, y=A + 8 * MB) == hc.HC_ERR_ALIAS              # y over f
    assert fused_rc(lib, pre=A + 13 * MB + 64) == hc.HC_ERR_ALIAS      # pre inside x_new
    assert fused_rc(lib, ws_bytes=16) == hc.HC_ERR_WORKSPACE
    assert fused_rc(lib, ws=A + 13 * MB) == hc.HC_ERR_ALIAS            # workspace over x_new
    assert fused_rc(lib, T=0, x_prev=0) == hc.HC_OK


def norm_rc(lib, y=A, w=A + 8 * MB, z=A + 9 * MB, q=A + 10 * MB, qs=A + 11 * MB, T=2, d=4096, eps=1e-5):
    return lib.hc_rms_norm_q8(y, w, T, d, eps, z, q, qs, None)


@fake_addresses
def test_rms_norm_q8_validation(lib):
    assert norm_rc(lib, T=-1) == hc.HC_ERR_DIM
    assert norm_rc(lib, eps=-1.0) == hc.HC_ERR_DIM
    assert norm_rc(lib, eps=math.inf) == hc.HC_ERR_DIM
    assert norm_rc(lib, y=0) == hc.HC_ERR_NULL
    assert norm_rc(lib, q=0) == hc.HC_ERR_NULL                      # q without its scales
    assert norm_rc(lib, d=4100) == hc.HC_ERR_ALIGN                  # q needs d % 32 == 0
    assert norm_rc(lib, z=A + 9 * MB + 8) == hc.HC_ERR_ALIGN
    assert norm_rc(lib, z=A + 64) == hc.HC_ERR_ALIAS                # z over y
    assert norm_rc(lib, qs=A + 10 * MB + 16) == hc.HC_ERR_ALIAS     # scales over q
    assert norm_rc(lib, T=0, y=0) == hc.HC_OK


@pytest.mark.gpu
def test_host_checks_in_a_process_without_devices():
    """On a machine with a GPU: the fake-address checks of this file and of the no-alloc
    entry point, in a child process that sees no device."""
    if not DEVICE_VISIBLE:
        pytest.skip("no device visible here: the checks run directly in this process")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                        os.path.join(root, "tests", "test_abi_host.py"),
                        os.path.join(root, "tests", "test_zz_no_alloc.py")],
                       capture_output=True, text=True, timeout=600, cwd=root, env=env)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " skipped" not in r.stdout.splitlines()[-1], r.stdout[-2000:]


def test_binding_refuses_bad_tensors_before_any_call():
    """The binding's argument check (hc._ptr): None and empty tensors pass no pointer; a
    non-tensor, a host tensor and (through the slow path's messages) the wrong kind of
    tensor are refused with TypeError / ValueError before the library is called."""
    import torch
    assert hc._ptr(None, "x") is None
    with pytest.raises(TypeError):
        hc._ptr([1.0, 2.0], "x")
    with pytest.raises(ValueError, match="CUDA tensor"):
        hc._ptr(torch.zeros(4), "x")
    with pytest.raises(ValueError, match=r"\[T, s, d\]"):
        hc._shape(torch.zeros(4, 4))
    assert hc._shape(torch.zeros(2, 3, 8)) == (2, 3, 8)


def test_build_variants_are_separate_libraries():
    """The phase-stamp and bounds-checked variants build into their own directories, never over
    the product library, and one call builds one variant."""
    from mhc_hyper_connection_hc_gb300 import build
    libs = {build.LIB, build.STAMPS_LIB, build.BOUNDS_LIB}
    assert len(libs) == 3 and len({os.path.dirname(p) for p in libs}) == 3
    with pytest.raises(ValueError):
        build.build(stamps=True, bounds=True)
