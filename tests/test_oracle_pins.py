"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-derive the oracle's own loop nest: each one checks a value that
a hand derivation, a closed form, an invariant or an independently written
brute-force restatement fixes, and each is chosen so that a plausible slip in
the oracle (a dropped term, a wrong sign, a transposed index, a wrong divisor,
rows and columns normalised in the wrong order) fails it.  The formulas are
those of the memra-engine hyper.rs page, module header "ARITHMETIC CONTRACT".
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import brute_ref
import oracle
from mhc_hyper_connection_hc_gb300 import synth


def _zeros_w(s, d):
    return np.zeros(((2 + s) * s, s * d))


# ----------------------------------------------------------------------------- golden fixtures


def test_golden_split_base_only(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "split_base_only_s2.json")))
    inp = g["inputs"]
    s, d, eps = inp["s"], inp["d"], inp["eps"]
    x = synth.stream_state(900, 1, s, d)
    base = [0.0, math.log(3), -math.log(3), 0.0, 0.0, math.log(2), math.log(3), math.log(4)]
    r = oracle.pre(x, _zeros_w(s, d), inp["scale"], base, inp["iters"], eps)
    tol = g["tolerance_abs"]
    np.testing.assert_allclose(r["pre"][0] - eps, g["expected"]["pre_minus_eps"], atol=tol, rtol=0)
    np.testing.assert_allclose(r["post"][0], g["expected"]["post"], atol=tol, rtol=0)
    want = [[float(Fraction(*fr)) for fr in row] for row in g["expected"]["comb_fractions"]]
    np.testing.assert_allclose(r["comb"][0], want, atol=tol, rtol=0)


@pytest.mark.parametrize("iters", [1, 2, 3])
def test_golden_scalar_recurrence(golden_dir, iters):
    g = json.load(open(os.path.join(golden_dir, "sinkhorn_scalar_recurrence_s1.json")))
    inp = g["inputs"]
    s, d, eps = inp["s"], inp["d"], inp["eps"]
    x = synth.stream_state(901, 1, s, d).astype(np.float64)
    f = synth.branch_output(901, 0, 1, d).astype(np.float64)
    r = oracle.site(x, _zeros_w(s, d), inp["scale"], inp["base"], f, iters, eps)
    tol = g["tolerance_abs"]
    c = float(Fraction(*g["expected"]["comb_by_iters"][str(iters)]))
    assert abs(r["pre"][0, 0] - g["expected"]["pre"]) <= tol
    assert abs(r["post"][0, 0] - g["expected"]["post"]) <= tol
    assert abs(r["comb"][0, 0, 0] - c) <= tol
    np.testing.assert_allclose(r["y"][0], x[0, 0], atol=tol, rtol=0)
    np.testing.assert_allclose(r["x_out"][0, 0], 1.0 * f[0] + c * x[0, 0], atol=tol, rtol=0)


# ----------------------------------------------------------------------------- closed forms


def test_rms_rescale_and_scale_groups_closed_form():
    """Constant x = 1/2 and constant fn_w rows c_r = (r+1)/16 over K = s*d = 16:
    dot_r = c_r * K / 2 = (r+1)/2 and rsqrt(mean(x^2) + eps) = 1/sqrt(1/4 + 1/4) = sqrt(2),
    so mixes_r = (r+1)/sqrt(2); logit_r = mixes_r * scale[group r] + base_r with groups
    (pre, pre, post, post, comb x4).  A divisor of d instead of s*d, a missing sqrt, eps
    outside the sqrt, or a transposed fn_w all change these numbers."""
    s, d, R = 2, 8, 8
    x = np.full((1, s, d), 0.5)
    fn_w = np.repeat(((np.arange(R) + 1) / 16.0)[:, None], s * d, axis=1)
    base = 0.01 * np.arange(R)
    r = oracle.pre(x, fn_w, [1.0, 2.0, 3.0], base, 3, 0.25, want_mixes=True)
    mixes = (np.arange(R) + 1) / math.sqrt(2.0)
    np.testing.assert_allclose(r["mixes"][0], mixes, rtol=1e-14, atol=0)
    group_scale = np.array([1, 1, 2, 2, 3, 3, 3, 3], dtype=np.float64)
    np.testing.assert_allclose(r["logits"][0], mixes * group_scale + base, rtol=1e-14, atol=0)
    # gates from those logits: sigmoid, +eps on pre, x2 on post
    sig = 1.0 / (1.0 + np.exp(-(mixes * group_scale + base)))
    np.testing.assert_allclose(r["pre"][0], sig[:2] + 0.25, rtol=1e-14)
    np.testing.assert_allclose(r["post"][0], 2.0 * sig[2:4], rtol=1e-14)
    # collapse of a constant slab: y = (pre_0 + pre_1) / 2
    np.testing.assert_allclose(r["y"][0], np.full(d, 0.5 * r["pre"][0].sum()), rtol=1e-15)


def test_sinkhorn_2x2_limit_cross_ratio():
    """A positive 2x2 [[a,b],[c,e]] scaled to doubly stochastic is [[p,1-p],[1-p,p]] with
    p/(1-p) = sqrt(ae/(bc)) (the cross ratio survives diagonal scaling)."""
    a, b, c, e = 0.3, 1.7, 2.2, 0.9
    base = [0.0, 0.0, 0.0, 0.0, math.log(a), math.log(b), math.log(c), math.log(e)]
    x = synth.stream_state(902, 1, 2, 8)
    r = oracle.pre(x, _zeros_w(2, 8), [1, 1, 1], base, 2000, 1e-14)
    p = math.sqrt(a * e) / (math.sqrt(a * e) + math.sqrt(b * c))
    np.testing.assert_allclose(r["comb"][0], [[p, 1 - p], [1 - p, p]], atol=1e-10, rtol=0)


def test_sinkhorn_columns_last_and_convergence():
    """Columns are normalised last: column sums equal S/(S+eps) ~ 1 after ANY iteration
    count while row sums are not yet 1 after one; row sums then converge to 1."""
    s, d = 4, 4
    rng_base = synth.normal(903, (2 + s) * s, 0.0, 1.0).astype(np.float64)
    x = synth.stream_state(903, 1, s, d)
    row_err = []
    for iters in (1, 10, 100, 1000):
        r = oracle.pre(x, _zeros_w(s, d), [1, 1, 1], rng_base, iters, 1e-13)
        cm = r["comb"][0]
        assert np.max(np.abs(cm.sum(axis=0) - 1.0)) < 1e-11
        row_err.append(np.max(np.abs(cm.sum(axis=1) - 1.0)))
    assert row_err[0] > 1e-3
    assert all(b <= a * (1 + 1e-9) + 1e-15 for a, b in zip(row_err, row_err[1:]))
    assert row_err[-1] < 1e-10


def test_streams_one_reduces_to_scalar_program():
    """s = 1: y = pre * x with pre = sigmoid(logit_0) + eps, and comb is the scalar map
    c -> c/(c+eps) applied 2*iters times to exp(logit_2)."""
    T, s, d, eps = 5, 1, 64, 1e-3
    inp = synth.site_inputs(904, T, s, d)
    for iters in (1, 4, 20):
        r = oracle.pre(inp["x"], inp["fn_w"], inp["scale"], inp["base"], iters, eps, want_mixes=True)
        for t in range(T):
            lg = r["logits"][t]
            assert abs(r["pre"][t, 0] - (1 / (1 + math.exp(-lg[0])) + eps)) < 1e-15
            assert abs(r["post"][t, 0] - 2 / (1 + math.exp(-lg[1]))) < 1e-15
            c = math.exp(lg[2])
            for _ in range(2 * iters):
                c = c / (c + eps)
            assert abs(r["comb"][t, 0, 0] - c) < 1e-15
            np.testing.assert_allclose(r["y"][t], r["pre"][t, 0] * inp["x"][t, 0].astype(np.float64),
                                       rtol=1e-15, atol=0)


# ----------------------------------------------------------------------------- invariants


def test_scale_invariance():
    """x -> 3.7 x leaves mixes (hence pre/post/comb) unchanged up to O(eps) and scales y."""
    inp = synth.site_inputs(905, 3, 4, 64)
    x = inp["x"].astype(np.float64)
    a = oracle.pre(x, inp["fn_w"], inp["scale"], inp["base"], 20, 1e-14)
    b = oracle.pre(3.7 * x, inp["fn_w"], inp["scale"], inp["base"], 20, 1e-14)
    for k in ("pre", "post", "comb"):
        np.testing.assert_allclose(b[k], a[k], atol=1e-11, rtol=0)
    np.testing.assert_allclose(b["y"], 3.7 * a["y"], rtol=1e-11, atol=1e-13)


def test_stream_permutation_equivariance():
    """Relabel streams by pi (stream c of the new state is stream pi[c] of the old one),
    permuting fn_w's column blocks, the pre/post rows, and the comb block (j,k)->(pi j, pi k)
    to match: pre/post/x' permute, comb permutes on both indices, y is unchanged."""
    T, s, d, iters, eps = 2, 3, 16, 20, 1e-6
    pi = [1, 2, 0]
    inp = synth.site_inputs(906, T, s, d)
    x, w, base = inp["x"].astype(np.float64), inp["fn_w"].astype(np.float64), inp["base"].astype(np.float64)
    R = (2 + s) * s
    row_map = list(pi) + [s + p for p in pi] + [2 * s + pi[j] * s + pi[k] for j in range(s) for k in range(s)]
    xp = x[:, pi, :]
    wp = w[row_map].reshape(R, s, d)[:, pi, :].reshape(R, s * d)
    bp = base[row_map]
    a = oracle.site(x, w, inp["scale"], base, inp["f"], iters, eps)
    b = oracle.site(xp, wp, inp["scale"], bp, inp["f"], iters, eps)
    np.testing.assert_allclose(b["pre"], a["pre"][:, pi], rtol=1e-12)
    np.testing.assert_allclose(b["post"], a["post"][:, pi], rtol=1e-12)
    np.testing.assert_allclose(b["comb"], a["comb"][:, pi][:, :, pi], rtol=1e-11)
    np.testing.assert_allclose(b["y"], a["y"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b["x_out"], a["x_out"][:, pi, :], rtol=1e-11, atol=1e-13)


def test_uniform_and_scaled_streams():
    """Every stream equal to v: y = (sum_c pre_c) v, and with f = 0 every output stream is
    (column sum of comb) * v ~ v.  Streams (c+1) v: y = sum_c pre_c (c+1) v."""
    T, s, d = 3, 4, 32
    inp = synth.site_inputs(907, T, s, d)
    v = inp["x"][:, 0, :].astype(np.float64)
    xu = np.repeat(v[:, None, :], s, axis=1)
    r = oracle.site(xu, inp["fn_w"], inp["scale"], inp["base"], np.zeros((T, d)), 20, 1e-6)
    np.testing.assert_allclose(r["y"], r["pre"].sum(axis=1)[:, None] * v, rtol=1e-13, atol=1e-15)
    colsum = r["comb"].sum(axis=1)                        # [T, k]
    np.testing.assert_allclose(r["x_out"], colsum[:, :, None] * v[:, None, :], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["x_out"], np.repeat(v[:, None, :], s, axis=1), atol=1e-5)
    xs = np.stack([(c + 1) * v for c in range(s)], axis=1)
    r2 = oracle.pre(xs, inp["fn_w"], inp["scale"], inp["base"], 20, 1e-6)
    wsum = (r2["pre"] * (np.arange(s) + 1)).sum(axis=1)
    np.testing.assert_allclose(r2["y"], wsum[:, None] * v, rtol=1e-13, atol=1e-15)


def test_post_special_cases():
    """comb = I, post = 0 -> x' = x; post = 1, comb = 0 -> every stream = f;
    comb = the permutation matrix with comb[j, pi(j)] = 1 routes stream j to stream pi(j),
    which a transposed comb would route backwards."""
    T, s, d = 2, 3, 16
    x = synth.stream_state(908, T, s, d).astype(np.float64)
    f = synth.branch_output(908, 0, T, d).astype(np.float64)
    eye = np.broadcast_to(np.eye(s), (T, s, s))
    np.testing.assert_array_equal(oracle.post(x, f, np.zeros((T, s)), eye), x)
    np.testing.assert_array_equal(oracle.post(x, f, np.ones((T, s)), np.zeros((T, s, s))),
                                  np.repeat(f[:, None, :], s, axis=1))
    pi = [1, 2, 0]
    P = np.zeros((s, s))
    for j in range(s):
        P[j, pi[j]] = 1.0
    out = oracle.post(x, f, np.zeros((T, s)), np.broadcast_to(P, (T, s, s)))
    for j in range(s):
        np.testing.assert_array_equal(out[:, pi[j], :], x[:, j, :])


@pytest.mark.parametrize("s", [1, 2, 3, 4, 8])
def test_expand_then_mean_is_identity(s):
    e = synth.branch_output(909, 0, 3, 40).astype(np.float64)
    x = oracle.expand(e, s)
    for c in range(s):
        np.testing.assert_array_equal(x[:, c, :], e)
    m = oracle.mean(x)
    if s & (s - 1) == 0:
        np.testing.assert_array_equal(m, e)
    else:
        np.testing.assert_allclose(m, e, rtol=4e-16, atol=0)


@pytest.mark.parametrize("s", [1, 2, 3, 4, 8])
def test_mean_of_distinct_streams(s):
    """Stream c holds (c+1) v, so the unweighted mean is ((s+1)/2) v; and stream c holding
    2^c v gives ((2^s - 1)/s) v.  Equal streams (the expand pin) cannot tell a stream-0-only
    mean, a wrong stream stride or a wrong divisor from the right one; these can."""
    T, d = 3, 40
    v = synth.branch_output(912, 0, T, d).astype(np.float64)
    x = np.stack([(c + 1) * v for c in range(s)], axis=1)
    np.testing.assert_allclose(oracle.mean(x), 0.5 * (s + 1) * v, rtol=1e-15, atol=0)
    x2 = np.stack([(2.0 ** c) * v for c in range(s)], axis=1)
    np.testing.assert_allclose(oracle.mean(x2), (2.0 ** s - 1.0) / s * v, rtol=1e-15, atol=0)
    # token-major layout: token t's streams are x[t, :, :], not interleaved across tokens
    x3 = np.stack([(c + 1) * v for c in range(s)], axis=1) + 10.0 * np.arange(T)[:, None, None]
    np.testing.assert_allclose(oracle.mean(x3), 0.5 * (s + 1) * v + 10.0 * np.arange(T)[:, None],
                               rtol=1e-14, atol=1e-13)


# ----------------------------------------------------------------------------- brute force


@pytest.mark.parametrize("s,d,T", [(2, 8, 3), (3, 4, 2), (1, 8, 2)])
@pytest.mark.parametrize("iters", [1, 3, 20])
def test_brute_force_restatement(s, d, T, iters):
    inp = synth.site_inputs(910 + s, T, s, d)
    eps = float(np.float32(1e-6))
    a = oracle.site(inp["x"], inp["fn_w"], inp["scale"], inp["base"], inp["f"], iters, eps)
    b = brute_ref.site(inp["x"].astype(float).tolist(), inp["fn_w"].astype(float).tolist(),
                       inp["scale"].astype(float).tolist(), inp["base"].astype(float).tolist(),
                       inp["f"].astype(float).tolist(), iters, eps)
    for t in range(T):
        for k in ("pre", "post", "comb", "y", "x_out"):
            np.testing.assert_allclose(a[k][t], np.array(b[t][k]), rtol=1e-13, atol=1e-15)


def test_oracle_rejects_bad_arguments():
    x = np.zeros((1, 2, 4))
    with pytest.raises(ValueError):
        oracle.pre(x, np.zeros((8, 8)), [1, 1, 1], np.zeros(8), -1, 1e-6)
    r = oracle.pre(np.zeros((0, 2, 4)), np.zeros((8, 8)), [1, 1, 1], np.zeros(8), 3, 1e-6)
    assert r["y"].shape == (0, 4)


# ----------------------------------------------------------------------------- gated-head exit


def test_head_closed_form_zero_weights():
    """fn_w = 0: every gate is sigmoid(base_c) + eps whatever x is, and y is that weighted
    sum of the streams.  Pins the +eps, the sigmoid and the collapse's stream indexing."""
    s, d, eps = 3, 8, 0.125
    x = synth.stream_state(930, 4, s, d).astype(np.float64)
    base = np.array([-1.0, 0.0, 2.0])
    r = oracle.head(x, np.zeros((s, s * d)), [1.7], base, eps)
    g = 1.0 / (1.0 + np.exp(-base)) + eps
    np.testing.assert_allclose(r["gates"], np.tile(g, (4, 1)), rtol=1e-15)
    np.testing.assert_allclose(r["y"], np.einsum("c,tcd->td", g, x), rtol=1e-14)


def test_head_rescale_and_single_scale_closed_form():
    """Constant x = 1/2, fn_w row c constant (c+1)/16 over K = 16, eps = 1/4:
    mixes_c = (c+1)/sqrt(2) (as in the site test), and the ONE scale multiplies every row."""
    s, d = 2, 8
    x = np.full((1, s, d), 0.5)
    fn_w = np.repeat(((np.arange(s) + 1) / 16.0)[:, None], s * d, axis=1)
    base = np.array([0.01, -0.02])
    r = oracle.head(x, fn_w, [3.0], base, 0.25)
    logit = (np.arange(s) + 1) / math.sqrt(2.0) * 3.0 + base
    np.testing.assert_allclose(r["gates"][0], 1.0 / (1.0 + np.exp(-logit)) + 0.25, rtol=1e-14)
    np.testing.assert_allclose(r["y"][0], np.full(d, 0.5 * r["gates"][0].sum()), rtol=1e-15)


def test_head_equals_site_pre_rows():
    """A site whose pre rows, pre scale and pre bases are the head's computes the same gates
    (its pre) and the same collapse y, whatever its other rows hold."""
    s, d, T = 3, 16, 5
    inp = synth.site_inputs(931, T, s, d)
    hw, hs, hb = synth.head_params(931, s, d)
    fn_w = inp["fn_w"].astype(np.float64).copy()
    fn_w[:s] = hw
    scale = np.array([hs[0], 0.7, 1.3])
    base = inp["base"].astype(np.float64).copy()
    base[:s] = hb
    site = oracle.pre(inp["x"], fn_w, scale, base, 20, 1e-6)
    head = oracle.head(inp["x"], hw, hs, hb, 1e-6)
    np.testing.assert_allclose(head["gates"], site["pre"], rtol=1e-14)
    np.testing.assert_allclose(head["y"], site["y"], rtol=1e-13, atol=1e-15)


def test_head_uniform_streams():
    """Identical streams: y = (sum of gates) * x_0."""
    s, d = 4, 8
    x0 = synth.stream_state(932, 3, 1, d).astype(np.float64)
    x = np.repeat(x0, s, axis=1)
    hw, hs, hb = synth.head_params(932, s, d)
    r = oracle.head(x, hw, hs, hb, 1e-6)
    np.testing.assert_allclose(r["y"], r["gates"].sum(axis=1)[:, None] * x0[:, 0], rtol=1e-13)


@pytest.mark.parametrize("s,d,T", [(2, 8, 3), (3, 4, 2), (1, 8, 2)])
def test_head_brute_force_restatement(s, d, T):
    x = synth.stream_state(933 + s, T, s, d)
    hw, hs, hb = synth.head_params(933 + s, s, d)
    eps = float(np.float32(1e-6))
    a = oracle.head(x, hw, hs, hb, eps)
    b = brute_ref.head(x.astype(float).tolist(), hw.astype(float).tolist(), hs.astype(float).tolist(),
                       hb.astype(float).tolist(), eps)
    for t in range(T):
        np.testing.assert_allclose(a["gates"][t], np.array(b[t]["gates"]), rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(a["y"][t], np.array(b[t]["y"]), rtol=1e-13, atol=1e-15)


def test_head_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.head(np.zeros((1, 2, 4)), np.zeros((2, 8)), [1.0], np.zeros(2), -1.0)
    r = oracle.head(np.zeros((0, 2, 4)), np.zeros((2, 8)), [1.0], np.zeros(2), 1e-6)
    assert r["y"].shape == (0, 4)


# ----------------------------------------------------------------------------- branch-input norm + q8


def test_rms_norm_closed_forms():
    """Row [3, 4]: mean of squares 12.5, so z = [3, 4] / sqrt(12.5 + eps) * w.  A mean over the
    wrong count, a missing sqrt or eps outside it changes these numbers."""
    y = np.array([[3.0, 4.0], [-1.0, 1.0]])
    w = np.array([0.5, 2.0])
    z = oracle.rms_norm(y, w, 0.25)
    np.testing.assert_allclose(z[0], np.array([3.0, 4.0]) / math.sqrt(12.5 + 0.25) * w, rtol=1e-15)
    np.testing.assert_allclose(z[1], np.array([-1.0, 1.0]) / math.sqrt(1.0 + 0.25) * w, rtol=1e-15)


def test_rms_norm_scale_invariance():
    y = synth.branch_output(940, 0, 3, 64).astype(np.float64)
    w = 1.0 + 0.1 * synth.branch_output(941, 0, 1, 64)[0].astype(np.float64)
    np.testing.assert_allclose(oracle.rms_norm(7.5 * y, w, 0.0), oracle.rms_norm(y, w, 0.0), rtol=1e-14)
    # unit mean square after the norm when w = 1 and eps = 0
    z = oracle.rms_norm(y, np.ones(64), 0.0)
    np.testing.assert_allclose((z ** 2).mean(axis=1), 1.0, rtol=1e-14)


def test_q8_hand_computed_block():
    """amax 127 gives scale 1: the codes are z rounded half away from zero."""
    z = np.zeros(32, dtype=np.float32)
    z[:6] = [127.0, -63.5, 0.5, -0.5, 1.5, -2.5]
    q, sc = oracle.q8_blocks(z)
    assert sc[0] == np.float32(1.0)
    assert list(q[:6]) == [127, -64, 1, -1, 2, -3]
    assert np.all(q[6:] == 0)


def test_q8_zero_block_and_extremes():
    z = np.zeros(64, dtype=np.float32)
    z[32:] = synth.branch_output(942, 0, 1, 32)[0]
    q, sc = oracle.q8_blocks(z)
    assert sc[0] == 0 and np.all(q[:32] == 0)
    i = int(np.argmax(np.abs(z[32:])))
    assert abs(int(q[32 + i])) == 127 and np.all(np.abs(q) <= 127)


def _q8_restated(z32):
    """Independent restatement: numpy float32 for the scale and the product, exact float64
    arithmetic for rounding half away from zero."""
    z32 = np.asarray(z32, dtype=np.float32).reshape(-1, 32)
    amax = np.abs(z32).max(axis=1)
    sc = (amax / np.float32(127)).astype(np.float32)
    inv = np.where(sc != 0, np.float32(1) / np.where(sc != 0, sc, np.float32(1)), np.float32(0)).astype(np.float32)
    v = (z32 * inv[:, None]).astype(np.float32).astype(np.float64)
    r = np.where(v >= 0, np.floor(v + 0.5), -np.floor(-v + 0.5))
    return np.clip(r, -127, 127).astype(np.int8).reshape(-1), sc


def test_q8_matches_restatement_and_bounds():
    z = (3.0 * synth.branch_output(943, 0, 1, 4096)[0]).astype(np.float32)
    q, sc = oracle.q8_blocks(z)
    q2, sc2 = _q8_restated(z)
    assert np.array_equal(sc, sc2) and np.array_equal(q, q2)
    err = np.abs(q.astype(np.float64) * np.repeat(sc, 32) - z)
    assert np.all(err <= 0.5 * np.repeat(sc, 32) * (1 + 1e-6) + 1e-12)
