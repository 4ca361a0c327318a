"""Fused site boundary (hc_post_pre_fused): site i's hc_post and site i+1's pre-chain
in one call.  Checked against the float64 oracle's composition post -> pre, and, on
the cluster path, bit for bit against the two separate calls (hc_post, then
hc_pre_fused on its output), on both kernel paths, small shapes with ragged tails and
every token of a full-size batch."""

import numpy as np
import pytest

import oracle
from hc_testutil import TOL, eps32, rel_err, to_np
from mhc_hyper_connection_hc_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SMALL = [  # (T, s, d)
    (1, 4, 4096), (37, 4, 4096), (200, 4, 4096), (150, 2, 2048), (133, 3, 3072), (19, 1, 1024),
    (17, 3, 4100), (5, 8, 7168), (33, 6, 40), (130, 1, 1024), (300, 4, 2048), (37, 8, 7168), (9, 5, 4096),
]


def _up(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _inputs(cid, T, s, d):
    """Site A's state, branch output and (oracle) gates; site B's trio."""
    dist = "normal" if s == 8 and d == 7168 else "uniform"
    x = synth.stream_state(cid, T, s, d, dist)
    wa, sa, ba = synth.site_params(cid, 0, s, d)
    ga = oracle.pre(x, wa, sa, ba, 20, eps32(1e-6))
    f = synth.branch_output(cid, 0, T, d)
    wb, sb, bb = synth.site_params(cid, 1, s, d)
    return dict(x=x, f=f, post_prev=ga["post"].astype(np.float32), comb_prev=ga["comb"].astype(np.float32),
                fn_w=wb, scale=sb, base=bb)


class Fused:
    def __init__(self, T, s, d):
        from mhc_hyper_connection_hc_gb300 import hc
        self.hc = hc
        self.ws = hc.new_workspace(T, s, d)
        self.out = hc.new_pre_outputs(T, s, d)
        self.x_new = torch.empty(T, s, d, device="cuda")

    def run(self, dv, path=None):
        o = self.out
        self.hc.hc_post_pre_fused(dv["x"], dv["f"], dv["post_prev"], dv["comb_prev"], dv["fn_w"], dv["scale"],
                                  dv["base"], 20, 1e-6, self.x_new, o["pre"], o["post"], o["comb"], o["y"],
                                  self.ws, path=path)
        assert self.hc.hc_workspace_status(self.ws) == 0
        return self.x_new, o


def _paths(s, d):
    from mhc_hyper_connection_hc_gb300 import hc
    out = [hc.HC_PATH_GENERIC]
    auto = hc.hc_pre_auto_path(1, s, d)
    if auto in (hc.HC_PATH_CLUSTER, hc.HC_PATH_WIDE):
        out.append(auto)
    return out


@pytest.mark.parametrize("T,s,d", SMALL)
def test_fused_parity_small(T, s, d):
    from mhc_hyper_connection_hc_gb300 import hc
    inp = _inputs(800 + 3 * s + T, T, s, d)
    x_new_want = oracle.post(inp["x"], inp["f"], inp["post_prev"], inp["comb_prev"])
    want = oracle.pre(x_new_want, inp["fn_w"], inp["scale"], inp["base"], 20, eps32(1e-6))
    dv = {k: _up(v) for k, v in inp.items()}
    fz = Fused(T, s, d)
    for path in _paths(s, d):
        x_new, o = fz.run(dv, path=path)
        assert rel_err(to_np(x_new), x_new_want) <= TOL
        for k in ("pre", "post", "comb", "y"):
            assert rel_err(to_np(o[k]), want[k]) <= TOL, (path, k)
        # the same bits as the two separate calls
        x_sep = torch.empty_like(x_new)
        hc.hc_post(dv["x"], dv["f"], dv["post_prev"], dv["comb_prev"], x_sep)
        assert torch.equal(x_new.view(torch.int32), x_sep.view(torch.int32)), path
        ws = hc.new_workspace(T, s, d)
        sep = hc.new_pre_outputs(T, s, d)
        hc.hc_pre_fused(x_sep, dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, sep["pre"], sep["post"],
                        sep["comb"], sep["y"], ws, path=path)
        for k in ("pre", "post", "comb", "y"):
            assert torch.equal(o[k].view(torch.int32), sep[k].view(torch.int32)), (path, k)


def test_fused_full_size_every_token_and_bit_identical():
    """The bench's step at full size (T = 4096): every token of x_new and of the next
    site's pre/post/comb/y against the oracle's post -> pre composition, each token
    relative to its own scale, then bit-identical reruns."""
    T, s, d = 4096, 4, 4096
    inp = _inputs(3, T, s, d)
    dv = {k: _up(v) for k, v in inp.items()}
    fz = Fused(T, s, d)
    x_new, o = fz.run(dv)
    ref = {k: v.clone() for k, v in o.items()}
    ref["x_new"] = x_new.clone()
    x_new_want = oracle.post(inp["x"], inp["f"], inp["post_prev"], inp["comb_prev"])
    want = oracle.pre(x_new_want, inp["fn_w"], inp["scale"], inp["base"], 20, eps32(1e-6))
    want["x_new"] = x_new_want
    got = {k: to_np(v) for k, v in o.items()}
    got["x_new"] = to_np(x_new)
    for k in ("x_new", "pre", "post", "comb", "y"):
        assert rel_err(got[k], want[k]) <= TOL, k
        g2, w2 = got[k].reshape(T, -1), want[k].reshape(T, -1)
        per_tok = np.max(np.abs(g2 - w2), axis=1) / np.maximum(np.max(np.abs(w2), axis=1), 1e-6)
        assert np.max(per_tok) <= TOL, f"{k}: token {int(np.argmax(per_tok))} rel err {np.max(per_tok):.3e}"
    for _ in range(3):
        x_new, o = fz.run(dv)
        assert torch.equal(x_new.view(torch.int32), ref["x_new"].view(torch.int32))
        for k in ("pre", "post", "comb", "y"):
            assert torch.equal(o[k].view(torch.int32), ref[k].view(torch.int32)), k


def test_fused_largest_state():
    """T*s*d just under 2^31 elements (8 GiB of state in, 8 GiB out): 64-bit offsets and
    tensor-map rows of the fused boundary, on sampled tokens at both ends and the middle."""
    s, d = 4, 4096
    T = (2 ** 31 - 1) // (s * d)
    base_T = 64
    inp = _inputs(43, base_T, s, d)
    reps = (T + base_T - 1) // base_T
    dv = {k: _up(v) for k, v in inp.items()}
    for k in ("x", "f", "post_prev", "comb_prev"):
        t = dv[k]
        dv[k] = t.repeat(reps, *([1] * (t.dim() - 1)))[:T].contiguous()
    fz = Fused(T, s, d)
    x_new, o = fz.run(dv)
    idx = np.array([0, 1, T // 2, T - 2, T - 1])
    src = idx % base_T
    x_new_want = oracle.post(inp["x"][src], inp["f"][src], inp["post_prev"][src], inp["comb_prev"][src])
    want = oracle.pre(x_new_want, inp["fn_w"], inp["scale"], inp["base"], 20, eps32(1e-6))
    assert rel_err(to_np(x_new[idx]), x_new_want) <= TOL
    for k in ("pre", "post", "comb", "y"):
        assert rel_err(to_np(o[k][idx]), want[k]) <= TOL, k
    del dv, x_new
