"""The cluster path's helper kernel.  At prefill sizes the persistent cluster kernel leaves
SMs free (16-CTA clusters cannot be placed on them) and a second kernel, launched behind it,
takes the batch's last tokens, playing each cluster's 16 CTAs in turn.  Its tokens must be
the same bits as the cluster kernel's: the same batch run with a workspace too small for the
helper's partials runs the cluster kernel alone, and every token of the two runs is compared
bit for bit, for the pre-chain and the fused boundary, at batch sizes with and without a
ragged last tile and with more than one chunk of tokens per helper CTA.  (Agreement with the
float64 oracle at these sizes is checked by the full-size parity tests, which run with the
helper.)"""

import numpy as np
import pytest

from mhc_hyper_connection_hc_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

S, D = 4, 4096


def _up(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _tiled(a, T):
    """Rows of `a` repeated up to T rows (distinct data in every 64-token block's ends is not
    needed here: both runs see the same inputs)."""
    reps = (T + a.shape[0] - 1) // a.shape[0]
    return a.repeat(reps, *([1] * (a.dim() - 1)))[:T].contiguous()


def _inputs(seed, T):
    base_T = 97   # a prime, so tiles and chunks do not line up with the repetition
    inp = synth.site_inputs(seed, base_T, S, D)
    dv = {k: _up(v) for k, v in inp.items()}
    for k in ("x", "f"):
        dv[k] = _tiled(dv[k], T)
    # the previous site's gates for the fused boundary: any valid post / comb
    dv["post_prev"] = _tiled(_up(np.abs(synth.branch_output(seed, 5, base_T, S)) + 0.5), T)
    comb = np.abs(synth.branch_output(seed, 6, base_T, S * S)).reshape(base_T, S, S) + 0.1
    comb /= comb.sum(axis=2, keepdims=True)
    dv["comb_prev"] = _tiled(_up(comb), T)
    return dv


def _small_ws():
    from mhc_hyper_connection_hc_gb300 import hc
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    hc.hc_workspace_init(ws)
    return ws


def _bits(a):
    return a.contiguous().view(torch.int32)


@pytest.mark.parametrize("T", [2048, 4096, 4100, 16390])
def test_helper_tokens_equal_cluster_kernel_tokens_pre_chain(T):
    from mhc_hyper_connection_hc_gb300 import hc
    if hc.hc_pre_auto_path(T, S, D) != hc.HC_PATH_CLUSTER:
        pytest.skip("cluster path not available")
    dv = _inputs(170 + T % 97, T)
    big = hc.new_workspace(T, S, D)
    small = _small_ws()
    n_help = hc.hc_pre_helper_tokens(T, S, D, False, big.numel())
    assert n_help > 0, "the helper should take part at this size"
    assert hc.hc_pre_helper_tokens(T, S, D, False, small.numel()) == 0
    outs = []
    for ws in (big, small):
        o = hc.new_pre_outputs(T, S, D)
        for v in o.values():
            v.fill_(float("nan"))
        hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, o["pre"], o["post"], o["comb"],
                        o["y"], ws)
        torch.cuda.synchronize()
        assert hc.hc_workspace_status(ws) == hc.HC_OK
        outs.append(o)
    for k in ("pre", "post", "comb", "y"):
        a, b = outs[0][k], outs[1][k]
        assert not torch.isnan(a).any(), f"{k}: tokens left unwritten"
        eq = (_bits(a) == _bits(b)).reshape(T, -1).all(dim=1)
        bad = (~eq).nonzero().flatten()
        assert bad.numel() == 0, f"{k}: {bad.numel()} tokens differ, first {int(bad[0])} (helper from {T - n_help})"


@pytest.mark.parametrize("T", [4096, 4100, 16390])
def test_helper_tokens_equal_cluster_kernel_tokens_fused(T):
    from mhc_hyper_connection_hc_gb300 import hc
    if hc.hc_pre_auto_path(T, S, D) != hc.HC_PATH_CLUSTER:
        pytest.skip("cluster path not available")
    dv = _inputs(180 + T % 97, T)
    big = hc.new_workspace(T, S, D)
    small = _small_ws()
    n_help = hc.hc_pre_helper_tokens(T, S, D, True, big.numel())
    assert n_help > 0, "the helper should take part at this size"
    outs = []
    for ws in (big, small):
        o = hc.new_pre_outputs(T, S, D)
        for v in o.values():
            v.fill_(float("nan"))
        x_new = torch.full((T, S, D), float("nan"), device="cuda")
        hc.hc_post_pre_fused(dv["x"], dv["f"], dv["post_prev"], dv["comb_prev"], dv["fn_w"], dv["scale"],
                             dv["base"], 20, 1e-6, x_new, o["pre"], o["post"], o["comb"], o["y"], ws)
        torch.cuda.synchronize()
        assert hc.hc_workspace_status(ws) == hc.HC_OK
        o["x_new"] = x_new
        outs.append(o)
    # x_new is hc_post's output on every token
    x_ref = torch.empty_like(dv["x"])
    hc.hc_post(dv["x"], dv["f"], dv["post_prev"], dv["comb_prev"], x_ref)
    torch.cuda.synchronize()
    assert torch.equal(_bits(outs[0]["x_new"]), _bits(x_ref))
    for k in ("x_new", "pre", "post", "comb", "y"):
        a, b = outs[0][k], outs[1][k]
        assert not torch.isnan(a).any(), f"{k}: tokens left unwritten"
        eq = (_bits(a) == _bits(b)).reshape(T, -1).all(dim=1)
        bad = (~eq).nonzero().flatten()
        assert bad.numel() == 0, f"{k}: {bad.numel()} tokens differ, first {int(bad[0])} (helper from {T - n_help})"


def test_helper_not_used_for_small_batches_or_other_modes():
    """No helper at decode and verify sizes, for the gated head's shape count, or where the
    workspace has no room; and the query refuses bad dimensions."""
    from mhc_hyper_connection_hc_gb300 import hc
    big = hc.hc_pre_workspace_bytes(4096, S, D)
    for T in (1, 8, 37, 112):
        assert hc.hc_pre_helper_tokens(T, S, D, False, big) == 0
        assert hc.hc_pre_helper_tokens(T, S, D, True, big) == 0
    assert hc.hc_pre_helper_tokens(4096, S, D, False, 256) == 0
    assert hc.hc_pre_helper_tokens(4096, 8, 7168, False, big) == 0   # the wide path's shape
    assert hc.hc_pre_helper_tokens(-1, S, D, False, big) == -1


@pytest.mark.parametrize("T,s,d", [(4096, 3, 3072), (3000, 2, 2048), (2600, 1, 1024), (2500, 4, 1024)])
def test_helper_other_shapes_bit_identical_and_against_oracle(T, s, d):
    """The helper's other stream counts and slice widths: every token bit for bit against the
    cluster kernel alone (pre-chain and fused), and sampled tokens from both kernels' ranges
    against the float64 oracle."""
    import oracle
    from hc_testutil import TOL, eps32, rel_err
    from mhc_hyper_connection_hc_gb300 import hc
    if hc.hc_pre_auto_path(T, s, d) != hc.HC_PATH_CLUSTER:
        pytest.skip("cluster path not available")
    inp = synth.site_inputs(190 + s, T, s, d)
    dv = {k: _up(v) for k, v in inp.items()}
    big = hc.new_workspace(T, s, d)
    small = _small_ws()
    n_help = hc.hc_pre_helper_tokens(T, s, d, False, big.numel())
    if n_help == 0:
        pytest.skip("the split model gives the helper nothing at this shape")
    outs = []
    for ws in (big, small):
        o = hc.new_pre_outputs(T, s, d)
        hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, o["pre"], o["post"], o["comb"],
                        o["y"], ws)
        torch.cuda.synchronize()
        assert hc.hc_workspace_status(ws) == hc.HC_OK
        outs.append(o)
    for k in ("pre", "post", "comb", "y"):
        assert torch.equal(_bits(outs[0][k]), _bits(outs[1][k])), k
    toks = np.unique(np.array([0, 1, T - n_help - 1, T - n_help, T - n_help + 7, T - n_help + 8, T // 2, T - 9, T - 1]))
    want = oracle.pre(inp["x"][toks], inp["fn_w"], inp["scale"], inp["base"], 20, eps32(1e-6))
    for k in ("pre", "post", "comb", "y"):
        got = outs[0][k][torch.from_numpy(toks).cuda()].cpu().numpy()
        assert rel_err(got, want[k]) <= TOL, k
    # fused boundary at the same shape, when the cluster kernel takes it
    if hc.hc_pre_helper_tokens(T, s, d, True, big.numel()) == 0:
        return
    post_prev, comb_prev = outs[0]["post"].clone(), outs[0]["comb"].clone()
    res = []
    for ws in (big, small):
        o = hc.new_pre_outputs(T, s, d)
        x_new = torch.empty_like(dv["x"])
        hc.hc_post_pre_fused(dv["x"], dv["f"], post_prev, comb_prev, dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6,
                             x_new, o["pre"], o["post"], o["comb"], o["y"], ws)
        torch.cuda.synchronize()
        assert hc.hc_workspace_status(ws) == hc.HC_OK
        o["x_new"] = x_new
        res.append(o)
    for k in ("x_new", "pre", "post", "comb", "y"):
        assert torch.equal(_bits(res[0][k]), _bits(res[1][k])), "fused " + k


def test_helper_inside_a_cuda_graph():
    """A prefill call whose helper kernel is launched behind the cluster kernel (programmatic
    dependent launch) captures into a CUDA graph; the replays give the eager call's bits, and
    work queued after the graph sees both kernels' outputs (hc_post on the new state)."""
    from mhc_hyper_connection_hc_gb300 import hc
    T = 4096
    if hc.hc_pre_auto_path(T, S, D) != hc.HC_PATH_CLUSTER:
        pytest.skip("cluster path not available")
    dv = _inputs(175, T)
    ws = hc.new_workspace(T, S, D)
    assert hc.hc_pre_helper_tokens(T, S, D, True, ws.numel()) > 0
    ref = hc.new_pre_outputs(T, S, D)
    x_ref = torch.empty(T, S, D, device="cuda")
    hc.hc_post_pre_fused(dv["x"], dv["f"], dv["post_prev"], dv["comb_prev"], dv["fn_w"], dv["scale"], dv["base"],
                         20, 1e-6, x_ref, ref["pre"], ref["post"], ref["comb"], ref["y"], ws)
    torch.cuda.synchronize()
    got = {k: torch.full_like(v, float("nan")) for k, v in ref.items()}
    x_new = torch.full_like(x_ref, float("nan"))
    after = torch.empty_like(x_ref)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            hc.hc_post_pre_fused(dv["x"], dv["f"], dv["post_prev"], dv["comb_prev"], dv["fn_w"], dv["scale"],
                                 dv["base"], 20, 1e-6, x_new, got["pre"], got["post"], got["comb"], got["y"], ws)
            hc.hc_post(x_new, got["y"], got["post"], got["comb"], after)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert hc.hc_workspace_status(ws) == hc.HC_OK
    assert torch.equal(_bits(x_new), _bits(x_ref))
    for k in ref:
        assert torch.equal(_bits(got[k]), _bits(ref[k])), k
    want_after = torch.empty_like(x_ref)
    hc.hc_post(x_ref, ref["y"], ref["post"], ref["comb"], want_after)
    torch.cuda.synchronize()
    assert torch.equal(_bits(after), _bits(want_after))


@pytest.mark.parametrize("fused", [False, True])
def test_helper_runs_repeat_bit_for_bit(fused):
    """In the pre-chain mode the helper's eight warps wait for their tile buffers each on its
    own and the last warp done with a buffer refills it (no barrier between steps); in the
    fused mode one barrier a step orders the in-place transform.  Twenty back-to-back calls of
    each must give the cluster kernel's bits on every token every time."""
    from mhc_hyper_connection_hc_gb300 import hc
    T = 4096
    if hc.hc_pre_auto_path(T, S, D) != hc.HC_PATH_CLUSTER:
        pytest.skip("cluster path not available")
    dv = _inputs(7, T)
    big = hc.new_workspace(T, S, D)
    small = _small_ws()
    assert hc.hc_pre_helper_tokens(T, S, D, fused, big.numel()) > 0

    def run(ws):
        o = hc.new_pre_outputs(T, S, D)
        if fused:
            o["x_new"] = torch.empty(T, S, D, device="cuda")
            hc.hc_post_pre_fused(dv["x"], dv["f"], dv["post_prev"], dv["comb_prev"], dv["fn_w"], dv["scale"],
                                 dv["base"], 20, 1e-6, o["x_new"], o["pre"], o["post"], o["comb"], o["y"], ws)
        else:
            hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, o["pre"], o["post"],
                            o["comb"], o["y"], ws)
        return o

    ref = run(small)
    runs = [run(big) for _ in range(20)]
    torch.cuda.synchronize()
    assert hc.hc_workspace_status(big) == hc.HC_OK
    for i, o in enumerate(runs):
        for k in ref:
            assert torch.equal(_bits(o[k]), _bits(ref[k])), f"call {i}: {k} differs from the cluster kernel's"
