"""Prepared calls (hc.py `prepare=True`): the C call repeated on the pointers, sizes and
stream checked once.  Their outputs must be the same bits as the checked calls', on the
cluster and the wide paths and for the fused boundary, and a Prepared call must pick up new
contents of the same tensors (it holds pointers, not values)."""

import numpy as np
import pytest

from mhc_hyper_connection_hc_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _up(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _bits_equal(a, b):
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("T,s,d", [(1, 4, 4096), (8, 4, 4096), (37, 4, 4096), (9, 8, 7168)])
def test_prepared_calls_match_checked_calls(T, s, d):
    from mhc_hyper_connection_hc_gb300 import hc
    inp = synth.site_inputs(930 + T, T, s, d, "normal" if s > 4 else "uniform")
    dv = {k: _up(v) for k, v in inp.items()}
    ws = hc.new_workspace(T, s, d)
    ref, got = hc.new_pre_outputs(T, s, d), hc.new_pre_outputs(T, s, d)
    hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, ref["pre"], ref["post"],
                    ref["comb"], ref["y"], ws)
    pre = hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, got["pre"], got["post"],
                          got["comb"], got["y"], ws, prepare=True)
    assert isinstance(pre, hc.Prepared)
    for _ in range(3):
        pre()
    torch.cuda.synchronize()
    assert hc.hc_workspace_status(ws) == hc.HC_OK
    for k in ref:
        assert _bits_equal(got[k], ref[k]), k

    # hc_post and the fused boundary, prepared
    x_ref, x_got = torch.empty_like(dv["x"]), torch.empty_like(dv["x"])
    hc.hc_post(dv["x"], dv["f"], ref["post"], ref["comb"], x_ref)
    post = hc.hc_post(dv["x"], dv["f"], got["post"], got["comb"], x_got, prepare=True)
    post()
    torch.cuda.synchronize()
    assert _bits_equal(x_got, x_ref)
    fz_ref, fz_got = hc.new_pre_outputs(T, s, d), hc.new_pre_outputs(T, s, d)
    xn_ref, xn_got = torch.empty_like(dv["x"]), torch.empty_like(dv["x"])
    hc.hc_post_pre_fused(dv["x"], dv["f"], ref["post"], ref["comb"], dv["fn_w"], dv["scale"], dv["base"], 20,
                         1e-6, xn_ref, fz_ref["pre"], fz_ref["post"], fz_ref["comb"], fz_ref["y"], ws)
    fz = hc.hc_post_pre_fused(dv["x"], dv["f"], ref["post"], ref["comb"], dv["fn_w"], dv["scale"], dv["base"], 20,
                              1e-6, xn_got, fz_got["pre"], fz_got["post"], fz_got["comb"], fz_got["y"], ws,
                              prepare=True)
    fz()
    torch.cuda.synchronize()
    assert _bits_equal(xn_got, xn_ref)
    for k in fz_ref:
        assert _bits_equal(fz_got[k], fz_ref[k]), "fused " + k

    # new contents of the same input tensor: the prepared call sees them
    x2 = synth.stream_state(931 + T, T, s, d, "normal" if s > 4 else "uniform")
    dv["x"].copy_(_up(x2))
    pre()
    hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, ref["pre"], ref["post"],
                    ref["comb"], ref["y"], ws)
    torch.cuda.synchronize()
    for k in ref:
        assert _bits_equal(got[k], ref[k]), "after new x: " + k


def test_binding_checks_and_stream_handle():
    """The checked binding refuses a float64, a non-contiguous and an int8-for-float tensor;
    an empty tensor passes no pointer; and the stream it passes by default is the current
    stream of the current device, inside a torch.cuda.stream context as well."""
    from mhc_hyper_connection_hc_gb300 import hc
    x = torch.zeros(2, 4, 64, device="cuda")
    assert hc._ptr(x, "x") == x.data_ptr()
    assert hc._ptr(torch.empty(0, device="cuda"), "x") is None
    with pytest.raises(TypeError, match="float32"):
        hc._ptr(x.double(), "x")
    with pytest.raises(TypeError):
        hc._ptr(torch.zeros(8, dtype=torch.int8, device="cuda"), "x")
    with pytest.raises(ValueError, match="contiguous"):
        hc._ptr(x.transpose(1, 2), "x")
    assert hc._ptr(torch.zeros(8, dtype=torch.int8, device="cuda"), "q", torch.int8) is not None
    assert hc._stream(None) == torch.cuda.current_stream().cuda_stream
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert hc._stream(None) == side.cuda_stream
    assert hc._stream(side) == side.cuda_stream
