"""The synthetic workloads: shapes, seeds and value distributions.

Every input of every workload is drawn here from counter-based SplitMix64
streams (``synth.gen``), so the CPU oracle and the CUDA path see the same
bytes.  Nothing here computes the method itself.

Recipe
------
* layer seed       ``0x5EED0000 + 1000 * config + 16 * layer``
* matrix seed      ``derive(layer_seed, 1 + 3 * expert + m)``, m = 0 gate, 1 up, 2 down
* codebooks        stage s in {0,1,2}: fp32 N(0, sigma_s^2), sigma = 0.02, 0.01, 0.005,
                   stream ``derive(matrix_seed, 0x100 + s)``, shape [256][8]
* codes            uniform uint8, canonical order [row][chunk][stage], byte stream
                   ``derive(matrix_seed, 0x200)``
* router weight    fp32 N(0, 0.02^2) [E][d], stream ``derive(layer_seed, 0x10000001)``
* activations      N(0, 1) rounded to fp32 then bf16 (round to nearest even),
                   [n][d], stream ``derive(layer_seed, 0x10000002)``; the single-GEMV
                   workload keeps them in fp32
* prefill bias     ``bias_e = -beta * 1.1 * ln(1 + pi(e))`` with pi a seeded permutation
                   of the experts (stream ``derive(layer_seed, 0x10000003)``): a Zipf(1.1)
                   popularity profile over a random expert order
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import bf16_to_f32, bytes_into, derive, f32_to_bf16, normal_f32, permutation

STAGE_SIGMA = (0.02, 0.01, 0.005)
TAG_ROUTER = 0x10000001
TAG_TOKENS = 0x10000002
TAG_ZIPF = 0x10000003
GATE, UP, DOWN = 0, 1, 2


def layer_seed(config: int, layer: int = 0) -> int:
    return 0x5EED0000 + 1000 * config + 16 * layer


def matrix_seed(lseed: int, expert: int, m: int) -> int:
    return derive(lseed, 1 + 3 * expert + m)


def codebooks(mseed: int) -> np.ndarray:
    """fp32 [3][256][8]: one codebook per RVQ stage."""
    out = np.empty((3, 256, 8), np.float32)
    for s in range(3):
        out[s] = normal_f32(derive(mseed, 0x100 + s), 256 * 8, STAGE_SIGMA[s]).reshape(256, 8)
    return out


def codes(mseed: int, rows: int, cols: int, out: np.ndarray | None = None) -> np.ndarray:
    """uint8 [rows][cols/8][3] canonical codes."""
    assert cols % 8 == 0
    if out is None:
        out = np.empty((rows, cols // 8, 3), np.uint8)
    return bytes_into(derive(mseed, 0x200), out)


def router_weight(lseed: int, E: int, d: int) -> np.ndarray:
    return normal_f32(derive(lseed, TAG_ROUTER), E * d, 0.02).reshape(E, d)


def tokens_f32(lseed: int, n: int, d: int) -> np.ndarray:
    return normal_f32(derive(lseed, TAG_TOKENS), n * d, 1.0).reshape(n, d)


def tokens_bf16(lseed: int, n: int, d: int) -> np.ndarray:
    """bf16 bit patterns [n][d]."""
    return f32_to_bf16(tokens_f32(lseed, n, d))


def zipf_bias(lseed: int, E: int, beta: float) -> np.ndarray:
    rank = permutation(derive(lseed, TAG_ZIPF), E)
    return np.array([-beta * 1.1 * math.log(1.0 + float(rank[e])) for e in range(E)],
                    dtype=np.float32)


@dataclass(frozen=True)
class LayerShape:
    d: int
    f: int
    E: int
    k: int


@dataclass(frozen=True)
class Workload:
    config: int
    name: str
    kind: str                       # "gemv" | "layer" | "stack" | "prefill" | "stack_prefill"
    shape: LayerShape | None = None
    rows: int = 0                   # gemv only
    cols: int = 0                   # gemv only
    batches: tuple = (1,)
    layers: int = 1
    zipf_beta: float = 0.0          # prefill only
    notes: str = field(default="", compare=False)

    @property
    def is_prefill(self) -> bool:
        """A prefill chunk: Zipf-biased router, tensor-core experts."""
        return self.kind in ("prefill", "stack_prefill")

    @property
    def n_layers(self) -> int:
        return self.layers if self.kind in ("stack", "stack_prefill") else 1


# Bias strength for the prefill chunk: chosen once so that the 2048 seeded
# tokens, routed top-16 over 256 experts, give at most about 600 tokens to the
# most popular expert (598; the least popular gets about 54).  A CPU test
# re-derives the counts with the oracle router.
PREFILL_ZIPF_BETA = 0.36

WORKLOADS = {
    0: Workload(0, "rvq_gemv_256x512", "gemv", rows=256, cols=512, batches=(1,)),
    1: Workload(1, "decode_layer_d2048_f1024_e64_k8", "layer",
                LayerShape(2048, 1024, 64, 8), batches=(1, 4, 16)),
    2: Workload(2, "k3_decode_layer_d7168_f2048_e256_k16", "layer",
                LayerShape(7168, 2048, 256, 16), batches=(1, 8, 64)),
    3: Workload(3, "k3_stack8_d7168_f2048_e256_k16", "stack",
                LayerShape(7168, 2048, 256, 16), batches=(1, 32), layers=8),
    4: Workload(4, "k3_prefill2048_d7168_f2048_e256_k16_zipf1.1", "prefill",
                LayerShape(7168, 2048, 256, 16), batches=(2048,),
                zipf_beta=PREFILL_ZIPF_BETA),
    # the chunked prefill of the pages (chunks of tokens through the layers)
    # on the 8-layer stack: config 4's chunk, each layer its own seeds and bias
    5: Workload(5, "k3_stack8_prefill2048_d7168_f2048_e256_k16_zipf1.1", "stack_prefill",
                LayerShape(7168, 2048, 256, 16), batches=(2048,), layers=8,
                zipf_beta=PREFILL_ZIPF_BETA),
}


class ExpertSource:
    """Lazily generates one layer's experts (codes + codebooks) on the host."""

    def __init__(self, config: int, layer: int, shape: LayerShape):
        self.config, self.layer, self.shape = config, layer, shape
        self.lseed = layer_seed(config, layer)

    def dims(self, m: int):
        s = self.shape
        return (s.f, s.d) if m in (GATE, UP) else (s.d, s.f)

    def codebooks(self, e: int, m: int) -> np.ndarray:
        return codebooks(matrix_seed(self.lseed, e, m))

    def codes(self, e: int, m: int, out: np.ndarray | None = None) -> np.ndarray:
        rows, cols = self.dims(m)
        return codes(matrix_seed(self.lseed, e, m), rows, cols, out)

    def router_weight(self) -> np.ndarray:
        return router_weight(self.lseed, self.shape.E, self.shape.d)

    def tokens_bf16(self, n: int) -> np.ndarray:
        return tokens_bf16(self.lseed, n, self.shape.d)


__all__ = ["WORKLOADS", "Workload", "LayerShape", "ExpertSource", "layer_seed",
           "matrix_seed", "codebooks", "codes", "router_weight", "tokens_f32",
           "tokens_bf16", "zipf_bias", "bf16_to_f32", "GATE", "UP", "DOWN",
           "PREFILL_ZIPF_BETA"]
