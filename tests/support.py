"""Shared helpers for the GPU parity tests: build device layers from the
seeded generator, and compare against the oracle."""
from __future__ import annotations

import numpy as np

import synth
from synth import workloads as W


def rms(a) -> float:
    a = np.asarray(a, np.float64)
    return float(np.sqrt(np.mean(a * a)))


def assert_rms_close(got, ref, tol, what=""):
    """max |got - ref| <= tol * RMS(ref)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), what
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    bound = tol * rms(ref)
    assert err <= bound, f"{what}: max err {err:.3e} > {tol} x RMS {rms(ref):.3e}"
    return err / max(rms(ref), 1e-300)


class SynthLayer:
    """One layer of a workload: host generator + oracle expert accessor."""

    def __init__(self, config: int, layer: int = 0, shape: W.LayerShape | None = None,
                 n_experts: int | None = None):
        self.config, self.layer = config, layer
        self.shape = shape or W.WORKLOADS[config].shape
        self.src = W.ExpertSource(config, layer, self.shape)
        self.E = n_experts or self.shape.E
        self._cache = {}

    def expert(self, e: int):
        if e not in self._cache:
            mats = []
            for m in range(3):
                mats.append((self.src.codes(e, m), self.src.codebooks(e, m)))
            self._cache[e] = tuple(mats)
        return self._cache[e]

    def forget(self):
        self._cache.clear()

    def to_gpu(self, k: int | None = None, bias=None, device="cuda"):
        from moe_expert_ffn_router_gb300.layer import MoeLayer
        s = self.shape
        L = MoeLayer(self.E, s.d, s.f, k or s.k, layer=self.layer, device=device)
        for e in range(self.E):
            (gc, gb), (uc, ub), (dc, db) = (
                (self.src.codes(e, m), self.src.codebooks(e, m)) for m in range(3))
            L.load_expert(e, gc, uc, dc, np.stack([gb, ub, db]))
        wr = W.router_weight(self.src.lseed, self.E, s.d)
        L.set_router(wr, bias)
        self.wr = wr
        return L

    def tokens_bf16(self, n: int):
        return W.tokens_bf16(self.src.lseed, n, self.shape.d)


def bf16_bits_to_f64(b) -> np.ndarray:
    return synth.bf16_to_f32(b).astype(np.float64)
