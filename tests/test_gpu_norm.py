"""The branch-input norm and its int8 pair (hc_rms_norm_q8, hc_pre_fused_norm) against
the oracle, two ways:

- first-hand: z within 1e-4 of the oracle's float64 norm, and the int8 codes and block
  scales against the oracle's own chain (its float64 z, quantised): block scales within
  1e-4 relative, codes equal except where the oracle's exact value z * 127 / amax lies
  within a stated bound of a half-integer (the rounding decision is then decided by the
  float32 error of z itself), where a difference of one is allowed and counted;
- same-precision: the codes and block scales bit for bit against the float32 quantiser
  applied to the GPU's own z (codes are integers decided in float32 on both sides)."""

import numpy as np
import pytest

import oracle
from hc_testutil import TOL, eps32, rel_err, to_np
from mhc_hyper_connection_hc_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _up(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _norm_w(cid, d):
    return (1.0 + 0.25 * synth.branch_output(cid, 7, 1, d)[0]).astype(np.float32)


def _check_q8_against_oracle_chain(z_gpu, q_gpu, s_gpu, z_ref):
    """Codes and block scales of the GPU against the oracle's float64 z (see the module
    docstring).  The bound: in a block whose GPU z differs from the oracle's by at most
    e * amax, the code's argument z * 127 / amax moves by at most 127 * (2 e + 2^-22)
    (z's own error, the scale's, and one float32 rounding of the product), so the code can
    differ only where the exact argument lies within that of a half-integer."""
    T, d = z_ref.shape
    zb_ref = z_ref.reshape(T, d // 32, 32)
    zb_gpu = np.asarray(z_gpu, dtype=np.float64).reshape(T, d // 32, 32)
    amax = np.max(np.abs(zb_ref), axis=2)
    s_ref = amax / 127.0
    nz = amax > 0
    s_g = np.asarray(s_gpu, dtype=np.float64)
    assert np.all(s_g[~nz] == 0)
    if np.any(nz):
        assert np.max(np.abs(s_g[nz] - s_ref[nz]) / s_ref[nz]) <= 1e-4
    e = np.max(np.abs(zb_gpu - zb_ref), axis=2) / np.where(nz, amax, 1.0)
    bound = 127.0 * (2.0 * e + 2.0 ** -22)
    v = np.where(nz[..., None], zb_ref * (127.0 / np.where(nz, amax, 1.0))[..., None], 0.0)
    q_ref = np.where(v >= 0, np.floor(v + 0.5), -np.floor(-v + 0.5))
    diff = np.asarray(q_gpu, dtype=np.int64).reshape(T, d // 32, 32) - q_ref.astype(np.int64)
    near = np.abs(np.abs(v - np.trunc(v)) - 0.5) <= bound[..., None]
    assert np.all(np.abs(diff) <= 1), "a code differs from the oracle's by more than one"
    bad = (diff != 0) & ~near
    assert not np.any(bad), f"{int(bad.sum())} codes differ away from a rounding tie"
    n_off = int(np.count_nonzero(diff))
    assert n_off <= max(2, q_ref.size // 1000), f"{n_off} codes off by one near ties"
    return n_off


@pytest.mark.parametrize("T,d", [(1, 4096), (37, 4096), (300, 7168), (5, 32), (3, 96)])
def test_norm_q8_parity(T, d):
    from mhc_hyper_connection_hc_gb300 import hc
    y = (2.0 * synth.branch_output(950 + T, 0, T, d)).astype(np.float32)
    y[0, : min(d, 64)] = 0.0                     # a zero block: scale 0, codes 0
    w = _norm_w(950, d)
    z = torch.empty(T, d, device="cuda")
    q = torch.empty(T, d, dtype=torch.int8, device="cuda")
    qs = torch.empty(T, d // 32, device="cuda")
    hc.hc_rms_norm_q8(_up(y), _up(w), 1e-5, z, q, qs)
    torch.cuda.synchronize()
    want = oracle.rms_norm(y, w, eps32(1e-5))
    assert rel_err(to_np(z), want) <= TOL
    _check_q8_against_oracle_chain(z.cpu().numpy(), q.cpu().numpy(), qs.cpu().numpy(), want)
    zq = z.cpu().numpy()
    q_want, s_want = oracle.q8_blocks(zq)
    assert np.array_equal(q.cpu().numpy(), q_want)
    assert np.array_equal(qs.cpu().numpy().view(np.uint32), s_want.view(np.uint32))
    # z alone (no pair), and reruns give the same bits
    z2 = torch.empty_like(z)
    hc.hc_rms_norm_q8(_up(y), _up(w), 1e-5, z2)
    assert torch.equal(z2.view(torch.int32), z.view(torch.int32))


@pytest.mark.parametrize("T,s,d", [(1, 4, 4096), (37, 4, 4096), (200, 4, 4096), (17, 3, 4096), (9, 8, 7168)])
def test_pre_fused_norm_parity(T, s, d):
    from mhc_hyper_connection_hc_gb300 import hc
    inp = synth.site_inputs(960 + T, T, s, d, "normal" if s == 8 else "uniform")
    w = _norm_w(960, d)
    want = oracle.pre(inp["x"], inp["fn_w"], inp["scale"], inp["base"], 20, eps32(1e-6))
    z_want = oracle.rms_norm(want["y"], w, eps32(1e-5))
    ws = hc.new_workspace(T, s, d)
    out = hc.new_pre_outputs(T, s, d)
    z = torch.empty(T, d, device="cuda")
    q = torch.empty(T, d, dtype=torch.int8, device="cuda")
    qs = torch.empty(T, d // 32, device="cuda")
    dv = {k: _up(v) for k, v in inp.items()}
    hc.hc_pre_fused_norm(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, _up(w), 1e-5, out["pre"],
                         out["post"], out["comb"], out["y"], z, ws, q=q, q_scale=qs)
    assert hc.hc_workspace_status(ws) == 0
    for k in ("pre", "post", "comb", "y"):
        assert rel_err(to_np(out[k]), want[k]) <= TOL, k
    assert rel_err(to_np(z), z_want) <= TOL
    _check_q8_against_oracle_chain(z.cpu().numpy(), q.cpu().numpy(), qs.cpu().numpy(), z_want)
    q_want, s_want = oracle.q8_blocks(z.cpu().numpy())
    assert np.array_equal(q.cpu().numpy(), q_want)
    assert np.array_equal(qs.cpu().numpy().view(np.uint32), s_want.view(np.uint32))


def test_norm_rejects_pair_with_ragged_blocks():
    from mhc_hyper_connection_hc_gb300 import hc
    y = torch.zeros(2, 36, device="cuda")
    w = torch.ones(36, device="cuda")
    z = torch.empty(2, 36, device="cuda")
    hc.hc_rms_norm_q8(y, w, 1e-5, z)                                    # z alone: fine
    with pytest.raises(hc.HcError):
        hc.hc_rms_norm_q8(y, w, 1e-5, z, torch.empty(2, 36, dtype=torch.int8, device="cuda"),
                          torch.empty(2, 1, device="cuda"))


@pytest.mark.parametrize("T,s,d", [(1, 4, 4096), (37, 4, 4096), (4096, 4, 4096), (130, 2, 1024), (5, 4, 768)])
def test_pre_fused_norm_one_launch(T, s, d):
    """The cluster path's one-launch pre-chain + norm (where d / 16 is a multiple of 32;
    (5, 4, 768) is a cluster shape whose slices do not hold whole blocks, so it runs the
    cluster pre-chain then the norm kernel): every token against the oracle (T = 4096
    reaches the exchange-slot and stage-ring reuse), pre/post/comb/y the same bits as
    hc_pre_fused on the cluster path, the Q8_0 pair first-hand and bit for bit against the
    float32 quantiser of its own z, z alone equal to z with the pair, reruns bit-identical."""
    from mhc_hyper_connection_hc_gb300 import hc
    if not hc.hc_pre_auto_path(T, s, d) == hc.HC_PATH_CLUSTER:
        pytest.skip("the cluster path does not run this shape here")
    inp = synth.site_inputs(965 + T, T, s, d)
    zt = T // 2 if T >= 3 else None
    if zt is not None:
        inp["x"][zt] = 0.0                         # a zero state: y = 0, z = 0, scales 0
    w = _norm_w(965, d)
    want = oracle.pre(inp["x"], inp["fn_w"], inp["scale"], inp["base"], 20, eps32(1e-6))
    z_want = oracle.rms_norm(want["y"], w, eps32(1e-5))
    dv = {k: _up(v) for k, v in inp.items()}
    wv = _up(w)
    ws = hc.new_workspace(T, s, d)

    def run(with_pair=True):
        out = hc.new_pre_outputs(T, s, d)
        z = torch.empty(T, d, device="cuda")
        q = torch.empty(T, d, dtype=torch.int8, device="cuda") if with_pair else None
        qs = torch.empty(T, d // 32, device="cuda") if with_pair else None
        hc.hc_pre_fused_norm(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, wv, 1e-5, out["pre"],
                             out["post"], out["comb"], out["y"], z, ws, q=q, q_scale=qs, path=hc.HC_PATH_CLUSTER)
        torch.cuda.synchronize()
        assert hc.hc_workspace_status(ws) == 0
        return out, z, q, qs

    out, z, q, qs = run()
    ref = hc.new_pre_outputs(T, s, d)
    hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, ref["pre"], ref["post"], ref["comb"],
                    ref["y"], ws, path=hc.HC_PATH_CLUSTER)
    torch.cuda.synchronize()
    for k in ("pre", "post", "comb", "y"):
        assert torch.equal(out[k].view(torch.int32), ref[k].view(torch.int32)), k
        assert rel_err(to_np(out[k]), want[k]) <= TOL, k
    zn = z.cpu().numpy()
    assert rel_err(zn, z_want) <= TOL
    if zt is not None:
        assert np.all(zn[zt] == 0.0)
    _check_q8_against_oracle_chain(zn, q.cpu().numpy(), qs.cpu().numpy(), z_want)
    q_want, s_want = oracle.q8_blocks(zn)
    assert np.array_equal(q.cpu().numpy(), q_want)
    assert np.array_equal(qs.cpu().numpy().view(np.uint32), s_want.view(np.uint32))
    _, z2, q2, qs2 = run()
    assert torch.equal(z2.view(torch.int32), z.view(torch.int32))
    assert torch.equal(q2, q) and torch.equal(qs2.view(torch.int32), qs.view(torch.int32))
    _, z3, _, _ = run(with_pair=False)
    assert torch.equal(z3.view(torch.int32), z.view(torch.int32))
