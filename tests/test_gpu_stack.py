"""GPU parity for the K3-shaped layer stack (independent seeds per layer,
fp32 residual stream between layers): each layer's routing bit-exact given
the GPU's logits and its outputs within 1e-4 x RMS of the oracle layer fed
with the same input; the stream is chained without copies.  Two of the
eight layers at full size (8.5 GB of codes) keep the test within minutes;
the bench runs all eight."""
import numpy as np
import pytest
import torch

import oracle
from synth import workloads as W
from tests.support import SynthLayer, assert_rms_close, bf16_bits_to_f64

pytestmark = pytest.mark.gpu
rvq = pytest.importorskip("moe_expert_ffn_router_gb300")
DEV = "cuda"


@pytest.mark.parametrize("n,sample", [(1, [0]), (32, [0, 31])])
def test_k3_stack_two_layers(n, sample):
    from moe_expert_ffn_router_gb300.layer import MoeStack
    torch.cuda.empty_cache()
    sls = [SynthLayer(3, layer) for layer in range(2)]
    stack = MoeStack([sl.to_gpu() for sl in sls])
    s = sls[0].shape
    bits = sls[0].tokens_bf16(n)
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    bufs = stack.forward(x)
    torch.cuda.synchronize()
    for L in stack.layers:
        assert L.status(n) == (0, 0)
    h = bf16_bits_to_f64(bits)
    for i, (sl, b) in enumerate(zip(sls, bufs)):
        logits = b["logits"].cpu().numpy()
        idx = b["idx"].cpu().numpy()
        ridx, _, _ = oracle.route(logits, s.k)
        assert np.array_equal(idx, ridx), f"layer {i} routing"
        roff, rpairs = oracle.group(ridx, s.E)
        assert np.array_equal(b["offsets"].cpu().numpy(), roff)
        assert np.array_equal(b["pairs"].cpu().numpy(), rpairs)
        assert_rms_close(logits, oracle.router_logits(sl.wr, h), 1e-5, f"layer {i} logits")
        out = b["out"].cpu().numpy().astype(np.float64)
        for t in sample:
            r = oracle.moe_layer(sl.expert, sl.wr, h[t:t + 1], s.k, s.d, s.f,
                                 route_logits=logits[t:t + 1])
            assert_rms_close(out[t] - h[t], r["out"][0] - h[t], 1e-4, f"layer {i} token {t}")
        h = out  # next layer's input is exactly this layer's fp32 output
        sl.forget()
    del stack, bufs
    torch.cuda.empty_cache()
