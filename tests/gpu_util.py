"""Helpers shared by the GPU parity tests: device copies of the seeded
workloads and the tolerances the comparisons use."""
from __future__ import annotations

import functools

import numpy as np
import pytest
import torch

import oracle
from lossless_speculative_verification_gb300 import api, synth

# Layer-output tolerance for bf16 tensor-core arithmetic against the fp64 oracle.
REL_L2 = 1e-2
MAX_ABS = 2e-2


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from lossless_speculative_verification_gb300 import _build
    _build.build()   # raises (and the test fails) if the library cannot be built
    oracle.build()


def to_dev(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).cuda()


def from_dev_bf16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_f64(u16: np.ndarray) -> np.ndarray:
    return synth.bf16_value(u16).astype(np.float64)


def assert_layer_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    diff = got - ref
    rel = np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300)
    mx = float(np.abs(diff).max()) if diff.size else 0.0
    assert rel <= REL_L2 and mx <= MAX_ABS, "%s rel-L2 %.3e max-abs %.3e" % (what, rel, mx)
    return rel, mx


class DevProblem:
    def __init__(self, prob: synth.MoeProblem):
        self.prob = prob
        d = self.d = prob.dims
        self.x = to_dev(prob.x)
        self.w_router = to_dev(prob.w_router)
        self.w_gate_up = to_dev(prob.w_gate_up)
        self.w_down = to_dev(prob.w_down)
        self.ws_gate_up = to_dev(prob.ws_gate_up) if d.S > 0 else None
        self.ws_down = to_dev(prob.ws_down) if d.S > 0 else None
        self.sh = api.shape(d.T, d.H, d.E, d.k, d.S, d.I)
        self.wts = api.weights(self.w_router, self.w_gate_up, self.w_down, self.ws_gate_up, self.ws_down)
        self.ws = api.workspace(self.sh)
        self._route = None

    def oracle_route(self):
        if self._route is None:
            idx, p, logits = oracle.route(self.prob.x, self.prob.w_router, self.d.k, return_logits=True)
            counts, offsets, perm, inv = oracle.permute(idx, self.d.E)
            self._route = dict(idx=idx, p=p, logits=logits, counts=counts, offsets=offsets, perm=perm, inv=inv)
        return self._route


@functools.lru_cache(maxsize=None)
def dev_problem(name: str, seed: int = 0) -> DevProblem:
    w = synth.WORKLOADS[name]
    return DevProblem(synth.moe_problem(w, seed=seed, row_ok=oracle.gap_ok(w.dims.k)))


def sample_rows(n: int, m: int, seed: int) -> np.ndarray:
    """m row indices of [0, n): the first and last few (ragged tail) plus a seeded spread."""
    if n <= m:
        return np.arange(n)
    rs = np.random.default_rng(seed)
    edge = np.array([0, 1, 2, n - 3, n - 2, n - 1])
    mid = rs.choice(n, size=m - edge.size, replace=False)
    return np.unique(np.concatenate([edge, mid]))
