"""Parity of the CUDA path against the float64 oracle, through the C ABI.

Small shapes and the full-size workloads are checked element by element on
every token (several tiles, ragged tails, every stream count 1..8, d not a
multiple of the chunk width), plus properties that hold at any size; only the
2^31-element state is checked on sampled tokens.  Bar: max relative error
<= 1e-4 per output tensor (pre, post, comb, y, x'), float32 GPU math, and
bit-identical reruns.
"""

import numpy as np
import pytest

import oracle
from hc_testutil import TOL, GpuSite, eps32, rel_err, sample_tokens, to_np
from mhc_hyper_connection_hc_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SMALL = [  # (T, s, d)
    (1, 4, 4096), (8, 4, 4096), (37, 4, 4096), (16, 4, 1024), (19, 1, 1024), (3, 2, 64),
    (17, 3, 4100), (2, 5, 12), (33, 6, 40), (4, 7, 8), (1, 8, 4), (5, 8, 7168), (40, 2, 2048),
    (21, 3, 3072), (200, 4, 4096), (150, 2, 2048), (130, 1, 1024), (133, 3, 3072), (300, 4, 2048),
    # wide-stream kernel shapes (s >= 5): several tiles, ragged tails, unequal CTA widths
    (37, 8, 7168), (9, 5, 4096), (33, 6, 4096), (17, 7, 7168), (130, 8, 2048), (1, 8, 7168),
]


def _paths(s, d):
    from mhc_hyper_connection_hc_gb300 import hc
    paths = [hc.HC_PATH_GENERIC]
    auto = hc.hc_pre_auto_path(1, s, d)
    if auto in (hc.HC_PATH_CLUSTER, hc.HC_PATH_WIDE):
        paths.append(auto)
    return paths


def _check_pre(g, want, idx=None, tol=TOL):
    for k in ("pre", "post", "comb", "y"):
        got = to_np(g[k]) if idx is None else to_np(g[k])[idx]
        err = rel_err(got, want[k])
        assert err <= tol, f"{k}: rel err {err:.3e} > {tol:g}"


@pytest.mark.parametrize("T,s,d", SMALL)
def test_site_parity_small(T, s, d):
    cid = 100 + 7 * s + T
    inp = synth.site_inputs(cid, T, s, d)
    eps, iters = eps32(1e-6), 20
    want = oracle.site(inp["x"], inp["fn_w"], inp["scale"], inp["base"], inp["f"], iters, eps)
    gs = GpuSite(T, s, d)
    dev = {k: gs.upload(v) for k, v in inp.items()}
    for path in _paths(s, d):
        g = gs.pre(dev["x"], dev["fn_w"], dev["scale"], dev["base"], iters, 1e-6, path=path)
        _check_pre(g, want)
        # hc_post chained from the GPU's own gates (end to end) ...
        xo = gs.post(dev["x"], dev["f"], g["post"], g["comb"])
        assert rel_err(to_np(xo), want["x_out"]) <= TOL
        assert gs.status() == 0
    # ... and fed the oracle's own gates rounded to float32 (the kernel alone).
    xo = gs.post(dev["x"], dev["f"], gs.upload(want["post"]), gs.upload(want["comb"]))
    want_k = oracle.post(inp["x"], inp["f"], want["post"].astype(np.float32),
                         want["comb"].astype(np.float32))
    assert rel_err(to_np(xo), want_k) <= 1e-6


def test_two_chained_sites_verify_batch():
    """T = 8, s = 4, d = 4096, two sites (attention, FFN) each with its own trio:
    site A's x' is site B's input; every intermediate is checked."""
    w = synth.WORKLOADS[2]
    T, s, d, iters, eps = w.T, w.s, w.d, w.iters, eps32(w.eps)
    x0 = synth.stream_state(w.cid, T, s, d)
    trios = [synth.site_params(w.cid, site, s, d) for site in (0, 1)]
    fs = [synth.branch_output(w.cid, site, T, d) for site in (0, 1)]
    gs = GpuSite(T, s, d)
    x_dev = gs.upload(x0)
    x_ref = x0.astype(np.float64)
    for site in (0, 1):
        fn_w, scale, base = trios[site]
        want = oracle.site(x_ref, fn_w, scale, base, fs[site], iters, eps)
        g = gs.pre(x_dev, gs.upload(fn_w), gs.upload(scale), gs.upload(base), iters, w.eps)
        _check_pre(g, want)
        xo = gs.post(x_dev, gs.upload(fs[site]), g["post"], g["comb"])
        assert rel_err(to_np(xo), want["x_out"]) <= TOL
        x_dev = xo.clone()
        x_ref = want["x_out"]


def _check_every_token(g, want, tol=TOL):
    """Each token's outputs against the oracle's, relative to that token's own scale (a
    stricter bar than the per-tensor measure, which a few corrupted tokens could hide
    under a large tensor-wide maximum)."""
    for k in ("pre", "post", "comb", "y"):
        got = to_np(g[k]).reshape(len(want[k]), -1)
        ref = np.asarray(want[k], dtype=np.float64).reshape(len(want[k]), -1)
        scale = np.maximum(np.max(np.abs(ref), axis=1), 1e-6)
        err = np.max(np.abs(got - ref), axis=1) / scale
        worst = int(np.argmax(err))
        assert err[worst] <= tol, f"{k}: token {worst} rel err {err[worst]:.3e} > {tol:g}"


@pytest.mark.parametrize("cid", [1, 3, 5])
def test_full_size_workloads_every_token(cid):
    """The single-decode, prefill and wide-stream workloads at full size, in the launch
    configuration the bench times: every token against the oracle."""
    w = synth.WORKLOADS[cid]
    inp = synth.workload_inputs(w)
    gs = GpuSite(w.T, w.s, w.d)
    dev = {k: gs.upload(v) for k, v in inp.items()}
    g = gs.pre(dev["x"], dev["fn_w"], dev["scale"], dev["base"], w.iters, w.eps)
    xo = gs.post(dev["x"], dev["f"], g["post"], g["comb"])
    torch.cuda.synchronize()
    assert gs.status() == 0
    want = oracle.site(inp["x"], inp["fn_w"], inp["scale"], inp["base"], inp["f"], w.iters, eps32(w.eps))
    _check_pre(g, want)
    _check_every_token(g, want)
    xo_np = to_np(xo)
    assert rel_err(xo_np, want["x_out"]) <= TOL
    per_tok = np.max(np.abs(xo_np - want["x_out"]).reshape(w.T, -1), axis=1) / \
        np.max(np.abs(want["x_out"]).reshape(w.T, -1), axis=1)
    assert np.max(per_tok) <= TOL, f"x_out: token {int(np.argmax(per_tok))}"
    # properties that hold for every token
    comb = to_np(g["comb"])
    assert np.all(np.isfinite(comb)) and np.all(np.isfinite(xo_np))
    assert np.max(np.abs(comb.sum(axis=1) - 1.0)) < 1e-4          # columns normalised last
    pre = to_np(g["pre"])
    assert np.all(pre > 0) and np.all(pre < 1 + 2e-6)
    post = to_np(g["post"])
    assert np.all(post >= 0) and np.all(post <= 2)


@pytest.mark.parametrize("T", [1, 512])
@pytest.mark.parametrize("iters", [1, 5, 10, 20, 40])
def test_sinkhorn_iteration_sweep(T, iters):
    """Every token of the sweep workload at each iteration count."""
    w = synth.WORKLOADS[4]
    inp = synth.workload_inputs(w, T=T)
    gs = GpuSite(T, w.s, w.d)
    dev = {k: gs.upload(v) for k, v in inp.items()}
    g = gs.pre(dev["x"], dev["fn_w"], dev["scale"], dev["base"], iters, w.eps)
    want = oracle.pre(inp["x"], inp["fn_w"], inp["scale"], inp["base"], iters, eps32(w.eps))
    _check_pre(g, want)
    _check_every_token(g, want)


def test_bit_identical_reruns():
    T, s, d = 300, 4, 4096
    inp = synth.site_inputs(31, T, s, d)
    gs = GpuSite(T, s, d)
    dev = {k: gs.upload(v) for k, v in inp.items()}
    from mhc_hyper_connection_hc_gb300 import hc
    for path in _paths(s, d):
        first = None
        for _ in range(10):
            g = gs.pre(dev["x"], dev["fn_w"], dev["scale"], dev["base"], 20, 1e-6, path=path)
            xo = gs.post(dev["x"], dev["f"], g["post"], g["comb"])
            cur = [t.clone() for t in (g["pre"], g["post"], g["comb"], g["y"], xo)]
            if first is None:
                first = cur
            else:
                for a, b in zip(first, cur):
                    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_largest_state():
    """T*s*d just under 2^31 elements (8 GiB of state): 64-bit offsets everywhere."""
    s, d = 4, 4096
    T = (2 ** 31 - 1) // (s * d)
    base_T = 64
    inp = synth.site_inputs(41, base_T, s, d)
    gs = GpuSite(T, s, d)
    x_small = gs.upload(inp["x"])
    f_small = gs.upload(inp["f"])
    reps = (T + base_T - 1) // base_T
    x = x_small.repeat(reps, 1, 1)[:T].contiguous()
    f = f_small.repeat(reps, 1)[:T].contiguous()
    g = gs.pre(x, gs.upload(inp["fn_w"]), gs.upload(inp["scale"]), gs.upload(inp["base"]), 20, 1e-6)
    xo = gs.post(x, f, g["post"], g["comb"])
    idx = np.array([0, 1, T // 2, T - 2, T - 1])
    src = idx % base_T
    want = oracle.site(inp["x"][src], inp["fn_w"], inp["scale"], inp["base"], inp["f"][src], 20,
                       eps32(1e-6))
    _check_pre(g, want, idx)
    assert rel_err(to_np(xo[idx]), want["x_out"]) <= TOL
    del x, f, xo


@pytest.mark.parametrize("s,d", [(1, 4), (3, 12), (4, 4096), (8, 7168)])
def test_expand_and_mean(s, d):
    from mhc_hyper_connection_hc_gb300 import hc
    T = 9
    e = synth.branch_output(51, 0, T, d)
    x = torch.empty(T, s, d, device="cuda")
    hc.hc_expand(torch.from_numpy(e).cuda(), x)
    want = oracle.expand(e, s)
    assert np.array_equal(to_np(x), want)
    xs = synth.stream_state(52, T, s, d)
    out = torch.empty(T, d, device="cuda")
    hc.hc_mean(torch.from_numpy(xs).cuda(), out)
    assert rel_err(to_np(out), oracle.mean(xs)) <= 1e-6
    m2 = torch.empty(T, d, device="cuda")
    hc.hc_mean(x, m2)
    # a float32 running sum of s equal values is not exact in general (3v rounds)
    assert rel_err(to_np(m2), e) <= 4e-7


def test_empty_batch_and_rejections():
    from mhc_hyper_connection_hc_gb300 import hc
    s, d = 4, 64
    gs = GpuSite(0, s, d)
    z = torch.empty(0, s, d, device="cuda")
    w = torch.zeros((2 + s) * s, s * d, device="cuda")
    sc, b = torch.ones(3, device="cuda"), torch.zeros((2 + s) * s, device="cuda")
    gs.pre(z, w, sc, b, 20, 1e-6)                    # T = 0: nothing to do, no error
    x = torch.zeros(2, s, d, device="cuda")
    f = torch.zeros(2, d, device="cuda")
    p = torch.zeros(2, s, device="cuda")
    c = torch.zeros(2, s, s, device="cuda")
    with pytest.raises(hc.HcError) as e:
        hc.hc_post(x, f, p, c, x)                    # in place is refused
    assert e.value.rc == hc.HC_ERR_ALIAS
    ws = hc.new_workspace(2, s, d)
    o = hc.new_pre_outputs(2, s, d)
    with pytest.raises(hc.HcError) as e:
        hc.hc_pre_fused(x, w, sc, b, 0, 1e-6, o["pre"], o["post"], o["comb"], o["y"], ws)
    assert e.value.rc == hc.HC_ERR_DIM               # zero Sinkhorn iterations refused
    with pytest.raises(hc.HcError) as e:
        hc.hc_pre_fused(x, w, sc, b, 20, 0.0, o["pre"], o["post"], o["comb"], o["y"], ws)
    assert e.value.rc == hc.HC_ERR_DIM               # eps <= 0 refused
    small_ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(hc.HcError) as e:
        hc.hc_pre_fused(x, w, sc, b, 20, 1e-6, o["pre"], o["post"], o["comb"], o["y"], small_ws)
    assert e.value.rc == hc.HC_ERR_WORKSPACE


def test_cluster_path_token_results_do_not_depend_on_the_batch():
    """The fused path sums every dot in one fixed order, so token t's outputs are the
    same bits whether it is alone (T=1), in a one-tile-per-cluster batch, or in a
    persistent multi-tile batch (the pages' pre_exact guarantee, here by construction)."""
    from mhc_hyper_connection_hc_gb300 import hc
    s, d = 4, 4096
    if hc.hc_pre_auto_path(1, s, d) != hc.HC_PATH_CLUSTER:
        pytest.skip("fused cluster path not available")
    T = 300
    inp = synth.site_inputs(61, T, s, d)
    big = GpuSite(T, s, d)
    dev = {k: big.upload(v) for k, v in inp.items()}
    g = big.pre(dev["x"], dev["fn_w"], dev["scale"], dev["base"], 20, 1e-6, path=hc.HC_PATH_CLUSTER)
    ref = {k: g[k].clone() for k in ("pre", "post", "comb", "y")}
    for n in (1, 5, 37):
        small = GpuSite(n, s, d)
        for start in (0, 17, T - n):
            gg = small.pre(dev["x"][start:start + n].contiguous(), dev["fn_w"], dev["scale"],
                           dev["base"], 20, 1e-6, path=hc.HC_PATH_CLUSTER)
            for k in ref:
                a = gg[k].view(torch.int32)
                b = ref[k][start:start + n].contiguous().view(torch.int32)
                assert torch.equal(a, b), f"{k} differs for tokens {start}..{start + n}"


def test_prefill_batch_tokens_equal_single_token_calls():
    """Tokens of the full prefill chunk (T = 4096, the persistent multi-tile launch the
    bench times) carry the same bits as the same tokens run alone (T = 1): the pages'
    pre_exact guarantee at the bench size, on whatever path hc_pre_fused takes there."""
    from mhc_hyper_connection_hc_gb300 import hc
    w = synth.WORKLOADS[3]
    T, s, d = w.T, w.s, w.d
    if hc.hc_pre_auto_path(T, s, d) != hc.HC_PATH_CLUSTER:
        pytest.skip("batch invariance is a property of the fused path")
    inp = synth.workload_inputs(w)
    big = GpuSite(T, s, d)
    dev = {k: big.upload(v) for k, v in inp.items()}
    g = big.pre(dev["x"], dev["fn_w"], dev["scale"], dev["base"], w.iters, w.eps)
    ref = {k: g[k].clone() for k in ("pre", "post", "comb", "y")}
    one = GpuSite(1, s, d)
    for t in sample_tokens(T, n=32):
        gg = one.pre(dev["x"][t:t + 1].contiguous(), dev["fn_w"], dev["scale"], dev["base"], w.iters, w.eps)
        for k in ref:
            assert torch.equal(gg[k].view(torch.int32), ref[k][t:t + 1].contiguous().view(torch.int32)), \
                f"{k} of token {t} differs between T=1 and T={T}"
    assert big.status() == 0 and one.status() == 0


def test_wide_stream_batch_tokens_equal_single_token_calls():
    """Tokens of the full wide-stream workload (T = 2048, s = 8, d = 7168) carry the same
    bits as the same tokens run alone, on the wide-stream kernel (one K split for every
    T, a fixed summation order over CTAs)."""
    from mhc_hyper_connection_hc_gb300 import hc
    w = synth.WORKLOADS[5]
    T, s, d = w.T, w.s, w.d
    if hc.hc_pre_auto_path(T, s, d) != hc.HC_PATH_WIDE:
        pytest.skip("wide-stream kernel not available")
    inp = synth.workload_inputs(w)
    big = GpuSite(T, s, d)
    dev = {k: big.upload(v) for k, v in inp.items()}
    g = big.pre(dev["x"], dev["fn_w"], dev["scale"], dev["base"], w.iters, w.eps)
    ref = {k: g[k].clone() for k in ("pre", "post", "comb", "y")}
    g = big.pre(dev["x"], dev["fn_w"], dev["scale"], dev["base"], w.iters, w.eps)   # a rerun: same bits
    for k in ref:
        assert torch.equal(g[k].view(torch.int32), ref[k].view(torch.int32)), k
    for n in (1, 5):
        small = GpuSite(n, s, d)
        for t in sample_tokens(T - n + 1, n=8):
            gg = small.pre(dev["x"][t:t + n].contiguous(), dev["fn_w"], dev["scale"], dev["base"], w.iters,
                           w.eps)
            for k in ref:
                assert torch.equal(gg[k].view(torch.int32), ref[k][t:t + n].contiguous().view(torch.int32)), \
                    f"{k} of tokens {t}..{t + n} differs between T={n} and T={T}"
        assert small.status() == 0
    assert big.status() == 0


def test_benchmark_shapes_run_their_fused_paths():
    """The workloads' shapes must run the fused kernels on a GB300, not fall back silently:
    the cluster path for s = 4, d = 4096 at T = 1, 8 and 4096, the wide path for the
    wide-stream workload (a layout that outgrew shared memory would otherwise only show
    up as skipped tests and a slower bench)."""
    from mhc_hyper_connection_hc_gb300 import hc
    for T in (1, 8, 512, 4096):
        assert hc.hc_pre_auto_path(T, 4, 4096) == hc.HC_PATH_CLUSTER, T
    assert hc.hc_pre_auto_path(2048, 8, 7168) == hc.HC_PATH_WIDE


@pytest.mark.parametrize("s,d", [(5, 4096), (6, 4096), (7, 7168)])
def test_wide_kernel_other_streams_invariant_and_against_oracle(s, d):
    """The wide kernel at s = 5, 6 and 7 (other row counts R, lane-pair row groups RB and
    split units): a T = 300 batch against the oracle on every token, and tokens of it the
    same bits as the same tokens run alone or in fives."""
    from mhc_hyper_connection_hc_gb300 import hc
    T = 300
    if hc.hc_pre_auto_path(T, s, d) != hc.HC_PATH_WIDE:
        pytest.skip("the wide kernel does not run this shape here")
    inp = synth.site_inputs(940 + s, T, s, d, "normal")
    want = oracle.pre(inp["x"], inp["fn_w"], inp["scale"], inp["base"], 20, eps32(1e-6))
    big = GpuSite(T, s, d)
    dev = {k: big.upload(v) for k, v in inp.items()}
    g = big.pre(dev["x"], dev["fn_w"], dev["scale"], dev["base"], 20, 1e-6, path=hc.HC_PATH_WIDE)
    ref = {k: g[k].clone() for k in ("pre", "post", "comb", "y")}
    for k in ref:
        assert rel_err(to_np(ref[k]), want[k]) <= TOL, k
    for n in (1, 5):
        small = GpuSite(n, s, d)
        for t in sample_tokens(T - n + 1, n=6):
            gg = small.pre(dev["x"][t:t + n].contiguous(), dev["fn_w"], dev["scale"], dev["base"], 20, 1e-6,
                           path=hc.HC_PATH_WIDE)
            for k in ref:
                assert torch.equal(gg[k].view(torch.int32), ref[k][t:t + n].contiguous().view(torch.int32)), \
                    f"{k} of tokens {t}..{t + n} differs between T={n} and T={T}"
        assert small.status() == 0
    assert big.status() == 0


def test_wide_path_shape_rule():
    """HC_PATH_AUTO takes the wide kernel exactly where include/hc.h says it runs: the
    balanced splits of d into widths of the stream count's unit, over at least 32 CTAs."""
    from mhc_hyper_connection_hc_gb300 import hc
    for s, d in ((8, 7168), (8, 4096), (5, 4096), (6, 4096), (7, 4096), (5, 7168), (7, 7168)):
        assert hc.hc_pre_auto_path(64, s, d) == hc.HC_PATH_WIDE, (s, d)
    # 224 units of 32 over 152 CTAs: widths of 64 and 32 columns, balanced to 0.74
    assert hc.hc_pre_auto_path(64, 6, 7168) == hc.HC_PATH_GENERIC
    # 153 units of 8: widths of 16 and 8 columns, balanced to 0.50
    assert hc.hc_pre_auto_path(64, 8, 1224) == hc.HC_PATH_GENERIC
    # fewer than 32 CTAs' worth of units
    assert hc.hc_pre_auto_path(64, 8, 248) == hc.HC_PATH_GENERIC
    assert hc.hc_pre_auto_path(64, 5, 1984) == hc.HC_PATH_GENERIC


def test_wide_kernel_largest_state():
    """The wide kernel at T*s*d just under 2^31 elements (s = 8, d = 7168: T = 37,448, an
    8.6 GB state): tiles, flags and partial slots far past 2^16, 64-bit row offsets.
    Sampled tokens against the oracle, and the same bits as those tokens run alone."""
    from mhc_hyper_connection_hc_gb300 import hc
    s, d = 8, 7168
    T = (2 ** 31 - 1) // (s * d)
    if hc.hc_pre_auto_path(T, s, d) != hc.HC_PATH_WIDE:
        pytest.skip("the wide kernel does not run this shape here")
    base_T = 64
    inp = synth.site_inputs(42, base_T, s, d, "normal")
    gs = GpuSite(T, s, d)
    x_small = gs.upload(inp["x"])
    x = x_small.repeat((T + base_T - 1) // base_T, 1, 1)[:T].contiguous()
    fw, sc, bs = gs.upload(inp["fn_w"]), gs.upload(inp["scale"]), gs.upload(inp["base"])
    g = gs.pre(x, fw, sc, bs, 20, 1e-6, path=hc.HC_PATH_WIDE)
    assert gs.status() == 0
    idx = np.array([0, 1, 3, 4, T // 2, T - 5, T - 2, T - 1])
    src = idx % base_T
    want = oracle.pre(inp["x"][src], inp["fn_w"], inp["scale"], inp["base"], 20, eps32(1e-6))
    sel = torch.from_numpy(idx).cuda()
    _check_pre({k: g[k].index_select(0, sel) for k in ("pre", "post", "comb", "y")}, want)
    one = GpuSite(1, s, d)
    for t in idx:
        gg = one.pre(x[t:t + 1].contiguous(), fw, sc, bs, 20, 1e-6, path=hc.HC_PATH_WIDE)
        for k in ("pre", "post", "comb", "y"):
            assert torch.equal(gg[k].view(torch.int32), g[k][t:t + 1].contiguous().view(torch.int32)), (k, int(t))
    assert one.status() == 0
    del x
