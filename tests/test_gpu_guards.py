"""Guard bands and the device error word.

Every output of every entry point is placed between two 4 KiB guard bands filled with
a byte pattern; after the call the bands must be intact (no out-of-bounds writes), on
both kernel paths, at ragged shapes.  And the workspace status word: a code written on
the host is reported by hc_workspace_status (HC_ERR_DEVICE), survives further calls
(it is sticky) and is cleared by hc_workspace_init.  The injection uses the generic
path, whose kernels have no device-side waits; a word set before a cluster- or wide-path
call makes that kernel skip its work, leaving every output as it was."""

import numpy as np
import pytest

from mhc_hyper_connection_hc_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side
PATTERN = 0xA5


class Guarded:
    """A float32 (or int8) tensor of the given shape inside a pattern-filled byte buffer."""

    def __init__(self, shape, dtype=torch.float32):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(*shape)
        self.n = n

    def intact(self):
        lo = self.raw[:GUARD].cpu().numpy()
        hi = self.raw[GUARD + self.n:].cpu().numpy()
        return bool(np.all(lo == PATTERN) and np.all(hi == PATTERN))


def _up(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _paths(s, d):
    from mhc_hyper_connection_hc_gb300 import hc
    out = [hc.HC_PATH_GENERIC]
    auto = hc.hc_pre_auto_path(1, s, d)
    if auto in (hc.HC_PATH_CLUSTER, hc.HC_PATH_WIDE):
        out.append(auto)
    return out


@pytest.mark.parametrize("T,s,d", [(37, 4, 4096), (19, 1, 1024), (133, 3, 3072), (17, 3, 4100), (5, 8, 7168),
                                   (130, 8, 2048), (9, 5, 4096), (2050, 4, 1024)])
def test_outputs_stay_inside_their_buffers(T, s, d):
    from mhc_hyper_connection_hc_gb300 import hc
    inp = synth.site_inputs(970 + T, T, s, d)
    dv = {k: _up(v) for k, v in inp.items()}
    ws = hc.new_workspace(T, s, d)
    for path in _paths(s, d):
        g = {k: Guarded(shape) for k, shape in
             (("pre", (T, s)), ("post", (T, s)), ("comb", (T, s, s)), ("y", (T, d)), ("x_out", (T, s, d)))}
        hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, g["pre"].t, g["post"].t,
                        g["comb"].t, g["y"].t, ws, path=path)
        hc.hc_post(dv["x"], dv["f"], g["post"].t, g["comb"].t, g["x_out"].t)
        # the fused site boundary, the head exit and the norm, on the same state
        fz = {k: Guarded(shape) for k, shape in
              (("x_new", (T, s, d)), ("pre", (T, s)), ("post", (T, s)), ("comb", (T, s, s)), ("y", (T, d)))}
        hc.hc_post_pre_fused(dv["x"], dv["f"], g["post"].t, g["comb"].t, dv["fn_w"], dv["scale"], dv["base"],
                             20, 1e-6, fz["x_new"].t, fz["pre"].t, fz["post"].t, fz["comb"].t, fz["y"].t, ws,
                             path=path)
        hw, hs, hb = (_up(a) for a in synth.head_params(970 + T, s, d))
        hd = {"gates": Guarded((T, s)), "y": Guarded((T, d))}
        hpath = hc.HC_PATH_AUTO if path == hc.HC_PATH_WIDE else path   # the head has no wide kernel
        hc.hc_head(dv["x"], hw, hs, hb, 1e-6, hd["y"].t, ws, gates=hd["gates"].t, path=hpath)
        torch.cuda.synchronize()
        assert hc.hc_workspace_status(ws) == 0
        for name, b in list(g.items()) + [("fused " + k, v) for k, v in fz.items()] + \
                [("head " + k, v) for k, v in hd.items()]:
            assert b.intact(), f"{name} guard band overwritten on path {path}"
    if d % 32 == 0:
        nz = {"z": Guarded((T, d)), "q": Guarded((T, d), torch.int8), "qs": Guarded((T, d // 32))}
        hc.hc_rms_norm_q8(g["y"].t, _up(np.ones(d)), 1e-5, nz["z"].t, nz["q"].t, nz["qs"].t)
        torch.cuda.synchronize()
        for name, b in nz.items():
            assert b.intact(), f"norm {name} guard band overwritten"


def test_device_error_word_is_reported_and_sticky():
    from mhc_hyper_connection_hc_gb300 import hc
    T, s, d = 8, 4, 1024
    inp = synth.site_inputs(980, T, s, d)
    dv = {k: _up(v) for k, v in inp.items()}
    ws = hc.new_workspace(T, s, d)
    out = hc.new_pre_outputs(T, s, d)

    def run():
        hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, out["pre"], out["post"],
                        out["comb"], out["y"], ws, path=hc.HC_PATH_GENERIC)

    run()
    assert hc.hc_workspace_status(ws) == hc.HC_OK
    ws[:4] = torch.tensor([7, 0, 0, 0], dtype=torch.uint8, device="cuda")   # inject a device error code
    assert hc.hc_workspace_status(ws) == hc.HC_ERR_DEVICE
    run()                                                                    # still reported after a call
    assert hc.hc_workspace_status(ws) == hc.HC_ERR_DEVICE
    hc.hc_workspace_init(ws)
    assert hc.hc_workspace_status(ws) == hc.HC_OK
    y_before = out["y"].clone()
    run()
    assert hc.hc_workspace_status(ws) == hc.HC_OK
    assert torch.equal(out["y"], y_before)                                   # the context is still usable


@pytest.mark.parametrize("T,s,d", [(37, 4, 4096), (1, 4, 4096), (9, 8, 7168), (2048, 4, 4096)])
def test_nonzero_status_word_makes_waiting_kernels_skip(T, s, d):
    """While the status word is non-zero, the cluster, helper and wide kernels (the ones with
    bounded waits) do nothing: the call returns HC_OK, every output keeps its sentinel
    (NaN), the word is unchanged.  After hc_workspace_init the same call writes them."""
    from mhc_hyper_connection_hc_gb300 import hc
    path = hc.hc_pre_auto_path(T, s, d)
    if path not in (hc.HC_PATH_CLUSTER, hc.HC_PATH_WIDE):
        pytest.skip("shape runs the generic path here")
    inp = synth.site_inputs(990 + T, T, s, d, "normal" if s > 4 else "uniform")
    dv = {k: _up(v) for k, v in inp.items()}
    ws = hc.new_workspace(T, s, d)
    code = torch.tensor([1, 0, 0, 0], dtype=torch.uint8, device="cuda")

    def sentinel_outputs():
        out = hc.new_pre_outputs(T, s, d)
        for v in out.values():
            v.fill_(float("nan"))
        return out

    out = sentinel_outputs()
    ws[:4] = code
    hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, out["pre"], out["post"],
                    out["comb"], out["y"], ws, path=path)
    x_new = torch.full((T, s, d), float("nan"), device="cuda")
    fz = sentinel_outputs()
    post_prev = torch.full((T, s), 0.5, device="cuda")
    comb_prev = torch.eye(s, device="cuda").expand(T, s, s).contiguous()
    hc.hc_post_pre_fused(dv["x"], dv["f"], post_prev, comb_prev, dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6,
                         x_new, fz["pre"], fz["post"], fz["comb"], fz["y"], ws, path=path)
    torch.cuda.synchronize()
    assert hc.hc_workspace_status(ws) == hc.HC_ERR_DEVICE
    assert ws[:4].cpu().tolist() == [1, 0, 0, 0]
    for name, v in list(out.items()) + [("fused " + k, v) for k, v in fz.items()]:
        assert bool(torch.isnan(v).all()), f"{name} was written while the status word was set"
    if path == hc.HC_PATH_CLUSTER:
        assert bool(torch.isnan(x_new).all()), "x_new was written while the status word was set"
    hc.hc_workspace_init(ws)
    hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, out["pre"], out["post"],
                    out["comb"], out["y"], ws, path=path)
    torch.cuda.synchronize()
    assert hc.hc_workspace_status(ws) == hc.HC_OK
    for name, v in out.items():
        assert bool(torch.isfinite(v).all()), f"{name} not written once the word was cleared"
