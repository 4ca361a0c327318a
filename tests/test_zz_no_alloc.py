"""hc_pre_fused_noalloc: the pre-chain for callers that cannot allocate device memory
when they run a site (an engine whose memory is all pre-carved into an arena, a plugin
whose host framework owns every allocation, a loop that cannot pay for cudaMalloc /
cudaFree).  It must give the results of the existing entry point with no workspace,
and those of the float64 oracle.

This file is collected last on purpose, so a first failure here comes after every
other test has run.
"""

import ctypes
import os

import numpy as np
import pytest

import oracle
from hc_testutil import TOL, rel_err, to_np
from mhc_hyper_connection_hc_gb300 import hc, synth

A = 0x10000000   # fake, aligned device addresses: the size check happens before any CUDA call
MB = 1 << 20


def _device_visible() -> bool:
    if os.environ.get("CUDA_VISIBLE_DEVICES") == "":
        return False
    try:
        import torch
        return bool(torch.cuda.is_available())
    except Exception:
        return False


@pytest.mark.skipif(_device_visible(), reason="fake device addresses: tests/test_abi_host.py runs this "
                                               "check in a child process without devices")
def test_noalloc_rejects_shapes_beyond_its_static_buffer():
    lib = hc.load()
    T, s, d = 50000, 4, 4096          # needs ~5 MB of split-K scratch, more than the 4 MiB buffer
    assert hc.hc_pre_workspace_bytes(T, s, d) > 4 * MB
    rc = lib.hc_pre_fused_noalloc(A, A + 900 * MB, A + 902 * MB, A + 903 * MB, T, s, d, 20,
                                  ctypes.c_float(1e-6), A + 904 * MB, A + 906 * MB,
                                  A + 908 * MB, A + 910 * MB, None)
    assert rc == hc.HC_ERR_TOO_LARGE
    assert "4 MiB" in hc.status_string(rc)


@pytest.mark.gpu
@pytest.mark.parametrize("T,s,d", [(37, 4, 4096), (5, 8, 7168)])
def test_noalloc_matches_the_existing_entry_point_on_two_calls_in_a_row(T, s, d):
    torch = pytest.importorskip("torch")
    for cid in (201, 202):           # two calls in a row, different inputs each time
        inp = synth.site_inputs(cid, T, s, d)
        dv = {k: torch.from_numpy(v).cuda() for k, v in inp.items()}
        ref = hc.new_pre_outputs(T, s, d)
        ws = hc.new_workspace(T, s, d)
        hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, ref["pre"],
                        ref["post"], ref["comb"], ref["y"], ws)
        got = hc.new_pre_outputs(T, s, d)
        rc = hc.load().hc_pre_fused_noalloc(
            ctypes.c_void_p(dv["x"].data_ptr()), ctypes.c_void_p(dv["fn_w"].data_ptr()),
            ctypes.c_void_p(dv["scale"].data_ptr()), ctypes.c_void_p(dv["base"].data_ptr()),
            T, s, d, 20, ctypes.c_float(1e-6), ctypes.c_void_p(got["pre"].data_ptr()),
            ctypes.c_void_p(got["post"].data_ptr()), ctypes.c_void_p(got["comb"].data_ptr()),
            ctypes.c_void_p(got["y"].data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == hc.HC_OK, hc.status_string(rc)
        torch.cuda.synchronize()
        want = oracle.pre(inp["x"], inp["fn_w"], inp["scale"], inp["base"], 20, float(np.float32(1e-6)))
        for k in ("pre", "post", "comb", "y"):
            err = rel_err(to_np(got[k]), to_np(ref[k]))
            assert err <= TOL, f"call for inputs {cid}: {k} rel err {err:.3e} against hc_pre_fused"
            err = rel_err(to_np(got[k]), want[k])
            assert err <= TOL, f"call for inputs {cid}: {k} rel err {err:.3e} against the oracle"
