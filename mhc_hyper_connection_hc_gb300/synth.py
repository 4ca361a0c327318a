"""Seeded synthetic inputs for the mHC site program.

This module is the one piece shared by the CUDA path, the CPU oracle's callers
(tests, the bench's CPU baseline) and the bench: it turns a seed into float32
arrays with the shapes and value distributions of the workloads, and holds none
of the method's arithmetic.

Generator: splitmix64 over a counter (state_i = seed + (i + 1) * golden gamma,
then the published splitmix64 finaliser), the top 53 bits read as a double in
[0, 1).  U[a, b) is the affine map of that double; N(mu, sigma) is Box-Muller on
two consecutive draws.  Values are rounded to float32 once, so the oracle (which
widens them to float64) and the GPU (which reads them as float32) see the same
bytes.

Seed of a tensor = 0x6D48C000 ^ (config << 16) ^ (site << 8) ^ tensor_id.

The five workloads are the shapes a GLM-5.3-Flash class trunk runs the site
program at (hc_fused_gate.rs header: streams=4, n_embd=4096, 20 Sinkhorn
iterations, eps=1e-6) plus a wide-stream variant (streams=8, hidden=7168).
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

TENSOR_X, TENSOR_FN_W, TENSOR_SCALE, TENSOR_BASE, TENSOR_F = 1, 2, 3, 4, 5
TENSOR_HEAD_FN_W, TENSOR_HEAD_SCALE, TENSOR_HEAD_BASE = 6, 7, 8


def tensor_seed(config: int, site: int, tensor_id: int) -> int:
    return 0x6D48C000 ^ (config << 16) ^ (site << 8) ^ tensor_id


def _u53(seed: int, start: int, n: int) -> np.ndarray:
    """n doubles in [0, 1) from counters start .. start+n-1 of stream `seed`."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def uniform(seed: int, n: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        out[s:s + m] = (lo + (hi - lo) * _u53(seed, s, m)).astype(np.float32)
    return out


def normal(seed: int, n: int, mu: float, sigma: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        u = _u53(seed, 2 * s, 2 * m)
        u1, u2 = u[0::2], u[1::2]
        z = np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * math.pi * u2)
        out[s:s + m] = (mu + sigma * z).astype(np.float32)
    return out


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: T tokens of an s-stream, d-hidden state."""
    cid: int
    name: str
    T: int
    s: int
    d: int
    iters: int = 20
    eps: float = 1e-6
    sites: int = 1
    x_dist: str = "uniform"        # "uniform" = U[-1,1), "normal" = N(0,1)

    @property
    def R(self) -> int:
        return (2 + self.s) * self.s

    @property
    def K(self) -> int:
        return self.s * self.d


WORKLOADS = {
    1: Workload(1, "single decode site", T=1, s=4, d=4096),
    2: Workload(2, "verify batch, 2 chained sites", T=8, s=4, d=4096, sites=2),
    3: Workload(3, "prefill chunk", T=4096, s=4, d=4096),
    4: Workload(4, "Sinkhorn-iteration sweep", T=512, s=4, d=4096),
    5: Workload(5, "wide-stream variant", T=2048, s=8, d=7168, x_dist="normal"),
}


def site_params(cid: int, site: int, s: int, d: int):
    """fn_w [R, s*d] ~ N(0, 1/(s*d)) (variance), scale[3] ~ U[0.5, 1.5), base[R] ~ N(0, 0.1)."""
    R, K = (2 + s) * s, s * d
    fn_w = normal(tensor_seed(cid, site, TENSOR_FN_W), R * K, 0.0, 1.0 / math.sqrt(K)).reshape(R, K)
    scale = uniform(tensor_seed(cid, site, TENSOR_SCALE), 3, 0.5, 1.5)
    base = normal(tensor_seed(cid, site, TENSOR_BASE), R, 0.0, 0.1)
    return fn_w, scale, base


def head_params(cid: int, s: int, d: int):
    """Gated-head exit trio: fn_w [s, s*d] ~ N(0, 1/(s*d)) (variance, as a site's),
    scale [1] ~ U[0.5, 1.5), base [s] ~ N(0, 0.1)."""
    K = s * d
    fn_w = normal(tensor_seed(cid, 0, TENSOR_HEAD_FN_W), s * K, 0.0, 1.0 / math.sqrt(K)).reshape(s, K)
    scale = uniform(tensor_seed(cid, 0, TENSOR_HEAD_SCALE), 1, 0.5, 1.5)
    base = normal(tensor_seed(cid, 0, TENSOR_HEAD_BASE), s, 0.0, 0.1)
    return fn_w, scale, base


def stream_state(cid: int, T: int, s: int, d: int, dist: str = "uniform", site: int = 0) -> np.ndarray:
    n = T * s * d
    seed = tensor_seed(cid, site, TENSOR_X)
    x = normal(seed, n, 0.0, 1.0) if dist == "normal" else uniform(seed, n, -1.0, 1.0)
    return x.reshape(T, s, d)


def branch_output(cid: int, site: int, T: int, d: int) -> np.ndarray:
    """Stand-in for the site's branch output f = branch(rms_norm(y)): U[-1, 1)."""
    return uniform(tensor_seed(cid, site, TENSOR_F), T * d, -1.0, 1.0).reshape(T, d)


def site_inputs(cid: int, T: int, s: int, d: int, dist: str = "uniform", site: int = 0):
    """Everything one site needs: x, fn_w, scale, base, f (all float32, C-contiguous)."""
    x = stream_state(cid, T, s, d, dist, site)
    fn_w, scale, base = site_params(cid, site, s, d)
    f = branch_output(cid, site, T, d)
    return dict(x=x, fn_w=fn_w, scale=scale, base=base, f=f)


def workload_inputs(w: Workload, T: int | None = None):
    return site_inputs(w.cid, w.T if T is None else T, w.s, w.d, w.x_dist)
