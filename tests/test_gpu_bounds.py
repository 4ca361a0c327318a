"""The bounds-checked build (build.build(bounds=True), -DHC_DEBUG_BOUNDS).  Its cluster, helper
and wide kernels check every plain global store (y, pre, post, comb, the helper's partials)
against the size of the buffer it writes, and report a refused store in the workspace status
word (code 2, the store's site) instead of performing it.  On valid calls the checks never
fire: the outputs are the plain build's bits.  The report itself is exercised without any
out-of-bounds access: that build reads HC_DEBUG_BOUNDS_Y_ROWS and takes y to have that many
rows, so the stores of the last real row are refused although they lie inside the buffer.

Each library runs in its own process (the binding holds one library per process)."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (T, s, d): decode variant, persistent clusters without a helper, clusters with the helper,
# the wide kernel
CASES = [(37, 4, 4096), (1000, 2, 2048), (4100, 4, 4096), (9, 8, 7168)]

_RUNNER = r"""
import hashlib, json, sys
import numpy as np, torch
sys.path.insert(0, ROOT)
from mhc_hyper_connection_hc_gb300 import build, hc, synth
hc.load(build.build(bounds=True) if BOUNDS else build.build())
res = []
for T, s, d in CASES:
    inp = synth.site_inputs(31 + T, T, s, d)
    dv = {k: torch.from_numpy(v).cuda() for k, v in inp.items()}
    ws = hc.new_workspace(T, s, d)
    path = hc.hc_pre_auto_path(T, s, d)
    row = {"T": T, "s": s, "d": d, "path": {hc.HC_PATH_CLUSTER: "cluster", hc.HC_PATH_WIDE: "wide"}.get(path, "other")}
    for mode in ("pre", "fused"):
        out = hc.new_pre_outputs(T, s, d)
        for v in out.values():
            v.fill_(float("nan"))
        if mode == "pre":
            hc.hc_pre_fused(dv["x"], dv["fn_w"], dv["scale"], dv["base"], 20, 1e-6, out["pre"], out["post"],
                            out["comb"], out["y"], ws)
        else:
            post_prev = torch.full((T, s), 0.5, device="cuda")
            comb_prev = torch.full((T, s, s), 1.0 / s, device="cuda")
            out["x_new"] = torch.empty(T, s, d, device="cuda")
            hc.hc_post_pre_fused(dv["x"], dv["f"], post_prev, comb_prev, dv["fn_w"], dv["scale"], dv["base"], 20,
                                 1e-6, out["x_new"], out["pre"], out["post"], out["comb"], out["y"], ws)
        torch.cuda.synchronize()
        word = ws[:12].cpu().numpy().view(np.uint32).tolist()
        y = out["y"]
        row[mode] = {"code": word[0], "where": word[1],
                     "hash": {k: hashlib.sha1(v.cpu().numpy().tobytes()).hexdigest() for k, v in out.items()},
                     "y_rows_written": int(torch.isfinite(y).all(dim=1).sum()),
                     "y_last_row_untouched": bool(torch.isnan(y[-1]).all()),
                     "helper_tokens": hc.hc_pre_helper_tokens(T, s, d, mode == "fused", ws.numel())}
        hc.hc_workspace_init(ws)
    res.append(row)
print(json.dumps(res))
"""


def _run(bounds: bool, y_rows_short: bool = False):
    env = dict(os.environ)
    env.pop("HC_DEBUG_BOUNDS_Y_ROWS", None)
    code = _RUNNER.replace("ROOT", repr(ROOT)).replace("BOUNDS", repr(bounds)).replace("CASES", repr(CASES))
    if y_rows_short:
        results = []
        for case in CASES:   # one process per case: the override is the case's T - 1
            env["HC_DEBUG_BOUNDS_Y_ROWS"] = str(case[0] - 1)
            one = code.replace(repr(CASES), repr([case]))
            r = subprocess.run([sys.executable, "-c", one], capture_output=True, text=True, env=env,
                               timeout=900, cwd=ROOT)
            assert r.returncode == 0, r.stderr[-3000:]
            results += json.loads(r.stdout.strip().splitlines()[-1])
        return results
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_bounds_build_gives_the_plain_build_bits():
    plain, checked = _run(False), _run(True)
    for a, b in zip(plain, checked):
        for mode in ("pre", "fused"):
            assert b[mode]["code"] == 0, f"{a['T']} {mode}: a check fired on a valid call ({b[mode]})"
            assert a[mode]["hash"] == b[mode]["hash"], f"T={a['T']} s={a['s']} {mode}: outputs differ"
            assert b[mode]["y_rows_written"] == a["T"]
    assert any(r["fused"]["helper_tokens"] > 0 for r in checked), "no case ran the helper kernel"
    assert [r["path"] for r in checked] == ["cluster", "cluster", "cluster", "wide"], "cases left their paths"


def test_bounds_build_reports_a_refused_store_and_skips_it():
    for r in _run(True, y_rows_short=True):
        for mode in ("pre", "fused"):
            m = r[mode]
            assert m["code"] == 2 and m["where"] == 100, f"T={r['T']} {mode}: status word {m['code']}, {m['where']}"
            # (once the word is set, the kernels' waits give up, so other rows may be left
            # unwritten too: the status word's usual meaning)
            assert m["y_last_row_untouched"], f"T={r['T']} {mode}: a refused y store was performed"
