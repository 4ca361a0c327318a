"""Shared helpers of the test-suite: the error metric and runners for the CUDA path."""

from __future__ import annotations

import numpy as np

# Tolerance of the GPU float32 path against the float64 oracle, per output tensor.
TOL = 1e-4


def rel_err(got, want) -> float:
    """Worst absolute difference relative to the reference's own scale:
    max|got - want| / max(max|want|, 1e-6) -- the measure of the memra-engine
    glm5_prime_v2_gate.rs page (`relative`)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    if want.size == 0:
        return 0.0
    scale = max(float(np.max(np.abs(want))), 1e-6)
    return float(np.max(np.abs(got - want))) / scale


def eps32(eps: float) -> float:
    """The float32 value the GPU receives, widened (the oracle must use the same number)."""
    return float(np.float32(eps))


def sample_tokens(T: int, n: int = 24, tile: int = 16, seed: int = 7) -> np.ndarray:
    """Tokens to check one by one at full size: first/last, tile edges, and random picks."""
    picks = {0, T - 1, min(T - 1, tile - 1), min(T - 1, tile), T // 2, max(0, T - tile)}
    rng = np.random.default_rng(seed)
    picks.update(int(v) for v in rng.integers(0, T, size=max(0, n - len(picks))))
    return np.array(sorted(p for p in picks if 0 <= p < T), dtype=np.int64)


class GpuSite:
    """Runs the pre-chain and hc_post on the GPU through the C ABI binding."""

    def __init__(self, T, s, d, device="cuda"):
        import torch
        from mhc_hyper_connection_hc_gb300 import hc
        self.torch, self.hc = torch, hc
        self.T, self.s, self.d = T, s, d
        self.ws = hc.new_workspace(T, s, d, device)
        self.out = hc.new_pre_outputs(T, s, d, device)
        self.x_out = torch.empty(T, s, d, dtype=torch.float32, device=device)

    def upload(self, a):
        return self.torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()

    def pre(self, x, fn_w, scale, base, iters, eps, path=None):
        o = self.out
        self.hc.hc_pre_fused(x, fn_w, scale, base, iters, eps, o["pre"], o["post"], o["comb"],
                             o["y"], self.ws, path=path)
        return o

    def post(self, x, f, post, comb):
        self.hc.hc_post(x, f, post, comb, self.x_out)
        return self.x_out

    def status(self):
        return self.hc.hc_workspace_status(self.ws)


def to_np(t):
    return t.detach().cpu().numpy().astype(np.float64)
