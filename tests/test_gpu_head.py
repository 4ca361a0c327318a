"""Parity of the gated-head trunk exit (hc_head) against the float64 oracle, through
the C ABI, on both kernel paths: every token of small shapes (several tiles, ragged
tails, stream counts 1..8), every token of a full-size batch, optional gates,
bit-identical reruns and, on the cluster path, independence of a token's bytes from
the batch it is in.  Bar: max relative error <= 1e-4 per output tensor."""

import numpy as np
import pytest

import oracle
from hc_testutil import TOL, eps32, rel_err, to_np
from mhc_hyper_connection_hc_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SMALL = [  # (T, s, d)
    (1, 4, 4096), (37, 4, 4096), (200, 4, 4096), (19, 1, 1024), (150, 2, 2048), (133, 3, 3072),
    (3, 2, 64), (17, 3, 4100), (33, 6, 40), (5, 8, 7168), (1, 8, 4), (130, 1, 1024), (300, 4, 2048),
]


class GpuHead:
    def __init__(self, T, s, d):
        from mhc_hyper_connection_hc_gb300 import hc
        self.hc = hc
        self.ws = hc.new_workspace(T, s, d)
        self.gates = torch.empty(T, s, dtype=torch.float32, device="cuda")
        self.y = torch.empty(T, d, dtype=torch.float32, device="cuda")

    def run(self, x, fn_w, scale, base, eps=1e-6, path=None, gates=True):
        self.hc.hc_head(x, fn_w, scale, base, eps, self.y, self.ws,
                        gates=self.gates if gates else None, path=path)
        assert self.hc.hc_workspace_status(self.ws) == 0
        return self.gates, self.y


def _up(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _inputs(cid, T, s, d):
    dist = "normal" if s == 8 and d == 7168 else "uniform"
    x = synth.stream_state(cid, T, s, d, dist)
    hw, hs, hb = synth.head_params(cid, s, d)
    return x, hw, hs, hb


def _paths(s, d):
    from mhc_hyper_connection_hc_gb300 import hc
    out = [hc.HC_PATH_GENERIC]
    if hc.hc_pre_auto_path(1, s, d) == hc.HC_PATH_CLUSTER:
        out.append(hc.HC_PATH_CLUSTER)
    return out


@pytest.mark.parametrize("T,s,d", SMALL)
def test_head_parity_small(T, s, d):
    x, hw, hs, hb = _inputs(700 + 5 * s + T, T, s, d)
    want = oracle.head(x, hw, hs, hb, eps32(1e-6))
    g = GpuHead(T, s, d)
    dx, dw, ds, db = _up(x), _up(hw), _up(hs), _up(hb)
    for path in _paths(s, d):
        gates, y = g.run(dx, dw, ds, db, path=path)
        assert rel_err(to_np(gates), want["gates"]) <= TOL, path
        assert rel_err(to_np(y), want["y"]) <= TOL, path
        y_with = y.clone()
        _, y2 = g.run(dx, dw, ds, db, path=path, gates=False)   # gates are optional
        assert torch.equal(y2.view(torch.int32), y_with.view(torch.int32))


def test_head_full_size_every_token_and_bit_identical():
    T, s, d = 4096, 4, 4096
    x, hw, hs, hb = _inputs(3, T, s, d)
    g = GpuHead(T, s, d)
    dx, dw, ds, db = _up(x), _up(hw), _up(hs), _up(hb)
    gates, y = g.run(dx, dw, ds, db)
    ref_g, ref_y = gates.clone(), y.clone()
    want = oracle.head(x, hw, hs, hb, eps32(1e-6))
    for k, got in (("gates", to_np(gates)), ("y", to_np(y))):
        assert rel_err(got, want[k]) <= TOL, k
        per_tok = np.max(np.abs(got - want[k]), axis=1) / np.maximum(np.max(np.abs(want[k]), axis=1), 1e-6)
        assert np.max(per_tok) <= TOL, f"{k}: token {int(np.argmax(per_tok))}"
    # properties at any size: gates in (eps, 1 + eps), y finite
    gn = to_np(gates)
    assert np.all(gn > 0) and np.all(gn < 1.0 + 1e-5) and np.all(np.isfinite(to_np(y)))
    for _ in range(5):
        gates, y = g.run(dx, dw, ds, db)
        assert torch.equal(gates.view(torch.int32), ref_g.view(torch.int32))
        assert torch.equal(y.view(torch.int32), ref_y.view(torch.int32))


def test_head_cluster_token_results_do_not_depend_on_the_batch():
    from mhc_hyper_connection_hc_gb300 import hc
    s, d, T = 4, 4096, 300
    if hc.hc_pre_auto_path(1, s, d) != hc.HC_PATH_CLUSTER:
        pytest.skip("fused cluster path not available")
    x, hw, hs, hb = _inputs(62, T, s, d)
    dx, dw, ds, db = _up(x), _up(hw), _up(hs), _up(hb)
    big = GpuHead(T, s, d)
    gates, y = big.run(dx, dw, ds, db, path=hc.HC_PATH_CLUSTER)
    ref = (gates.clone(), y.clone())
    for n in (1, 5, 37):
        small = GpuHead(n, s, d)
        for start in (0, 17, T - n):
            g2, y2 = small.run(dx[start:start + n].contiguous(), dw, ds, db, path=hc.HC_PATH_CLUSTER)
            assert torch.equal(g2.view(torch.int32), ref[0][start:start + n].contiguous().view(torch.int32))
            assert torch.equal(y2.view(torch.int32), ref[1][start:start + n].contiguous().view(torch.int32))


def test_head_empty_batch_and_rejections():
    from mhc_hyper_connection_hc_gb300 import hc
    g = GpuHead(1, 4, 4096)
    x = torch.zeros(0, 4, 4096, device="cuda")
    w = torch.zeros(4, 4 * 4096, device="cuda")
    sc = torch.ones(1, device="cuda")
    b = torch.zeros(4, device="cuda")
    hc.hc_head(x, w, sc, b, 1e-6, torch.zeros(0, 4096, device="cuda"), g.ws)   # empty: no-op
    x1 = torch.zeros(1, 4, 4096, device="cuda")
    with pytest.raises(hc.HcError):
        hc.hc_head(x1, w, sc, b, 0.0, g.y, g.ws)                                # eps <= 0
    with pytest.raises(hc.HcError):
        hc.hc_head(x1, w, sc, b, 1e-6, g.y, g.ws[:16])                          # workspace too small
