"""The prefill chunk's Zipf-biased routing has the skew its recipe states."""
import numpy as np

import oracle
import synth
from synth import workloads as W


def test_prefill_chunk_tokens_per_expert_range():
    wl = W.WORKLOADS[4]
    s = wl.shape
    lseed = W.layer_seed(4, 0)
    x = synth.bf16_to_f32(W.tokens_bf16(lseed, 2048, s.d)).astype(np.float64)
    wr = W.router_weight(lseed, s.E, s.d)
    bias = W.zipf_bias(lseed, s.E, wl.zipf_beta)
    lg = oracle.router_logits(wr, x, bias).astype(np.float32)
    idx, _, _ = oracle.route(lg, s.k)
    counts = np.bincount(idx.reshape(-1), minlength=s.E)
    assert counts.sum() == 2048 * 16
    assert 560 <= counts.max() <= 640
    assert 10 <= counts.min() <= 100
