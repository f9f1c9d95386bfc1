"""GPU tests of the tiered expert store (moe_layer_forward_streamed): a stack
whose records live in pinned host memory and stream into an HBM cache smaller
than the model gives bit-identical outputs to the resident stack (same kernels
on the same records, only their addresses differ), on the lookup-table and
tensor-core paths, with and without router lookahead; the cache counts add
up; a cache too small for one layer's experts is refused; and each streamed
layer's output matches the oracle layer fed the same normalised input and
residual (lookup tables at 1e-4 x RMS, tensor cores at 2e-2 x RMS)."""
import numpy as np
import pytest
import torch

import oracle
from tests.support import SynthLayer, assert_rms_close, bf16_bits_to_f64

pytestmark = pytest.mark.gpu
rvq = pytest.importorskip("moe_expert_ffn_router_gb300")
DEV = "cuda"


def _layers(n_layers):
    return [SynthLayer(1, layer) for layer in range(n_layers)]


def _resident_outputs(sls, xs, tc_min):
    from moe_expert_ffn_router_gb300.layer import MoeStack
    stack = MoeStack([sl.to_gpu() for sl in sls])
    outs = []
    for x in xs:
        bufs = stack.forward(x, tc_min_tokens=tc_min)
        outs.append([b["out"].clone() for b in bufs])
    torch.cuda.synchronize()
    del stack
    return outs


# (n, tc_min_tokens, lookahead, slots, prefetch expected): at 128 tokens every
# layer routes to all 64 experts, so its own records fill the cache and the
# lookahead has no slot to fill (it is a hint and is skipped)
@pytest.mark.parametrize("n,tc_min,lookahead,slots,prefetch",
                         [(1, 0, 0, 24, False), (4, 0, 3, 48, True), (128, 1, 2, 64, False)])
def test_streamed_stack_matches_resident(n, tc_min, lookahead, slots, prefetch):
    from moe_expert_ffn_router_gb300.layer import MoeStreamedStack
    torch.cuda.empty_cache()
    sls = _layers(3)
    xs = []
    for i in range(3):
        bits = sls[0].tokens_bf16(n * (i + 1))[-n:]
        xs.append(torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16))
    ref = _resident_outputs(sls, xs, tc_min)
    st = MoeStreamedStack([sl.to_gpu() for sl in sls], slots=slots, lookahead=lookahead)
    E = st.E
    assert st.stats()["slots"] == slots < 3 * E  # the cache holds less than the model
    expect_routed = 0
    for x, r in zip(xs, ref):
        bufs = st.forward(x, tc_min_tokens=tc_min)
        torch.cuda.synchronize()
        assert st.status(n) == (0, 0)
        for i, (b, ro) in enumerate(zip(bufs, r)):
            assert torch.equal(b["out"], ro), f"layer {i}"
            expect_routed += int((torch.diff(b["offsets"]) > 0).sum())
    s = st.stats()
    assert s["hits"] + s["misses"] == expect_routed
    assert s["bytes_copied"] == (s["misses"] + s["prefetched"]) * st.host.numel() // (3 * E)
    assert (s["prefetched"] > 0) == prefetch
    assert s["prefetch_used"] <= s["prefetched"]
    st.close()
    torch.cuda.empty_cache()


def test_cache_smaller_than_a_layer_is_refused():
    from moe_expert_ffn_router_gb300.layer import MoeStreamedStack
    sls = _layers(2)
    st = MoeStreamedStack([sl.to_gpu() for sl in sls], slots=4)
    bits = sls[0].tokens_bf16(8)  # 8 tokens x top-8: more than 4 distinct experts
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    with pytest.raises(rvq.RvqError) as ei:
        st.forward(x)
    assert ei.value.status == "RVQ_ENOMEM"
    torch.cuda.synchronize()
    st.close()


# (n, tc_min_tokens, lookahead, slots, sampled tokens, tolerance): the lookup
# tables with router lookahead, and every expert on the tensor cores
@pytest.mark.parametrize("n,tc_min,lookahead,slots,sample,tol",
                         [(4, 0, 3, 48, [0, 3], 1e-4), (128, 1, 2, 64, [0, 77, 127], 2e-2)])
def test_streamed_stack_matches_oracle(n, tc_min, lookahead, slots, sample, tol):
    """The streamed stack (d = 2048, three layers, records from pinned host
    memory through an HBM cache smaller than the model) against the oracle,
    layer by layer: the norm within bf16 rounding, routing and grouping
    bit-exact given the GPU's logits, logits within 1e-5 x RMS, and the
    sampled tokens' outputs (out - residual) within the path's tolerance of
    the oracle layer fed the layer's normalised input."""
    from moe_expert_ffn_router_gb300.layer import MoeStreamedStack
    torch.cuda.empty_cache()
    sls = _layers(3)
    st = MoeStreamedStack([sl.to_gpu() for sl in sls], slots=slots, lookahead=lookahead)
    s = sls[0].shape
    bits = sls[0].tokens_bf16(n)
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    bufs = st.forward(x, tc_min_tokens=tc_min)
    torch.cuda.synchronize()
    assert st.status(n) == (0, 0)
    h = bf16_bits_to_f64(bits)
    for i, (sl, b) in enumerate(zip(sls, bufs)):
        xn = b["xn"].float().cpu().numpy().astype(np.float64)   # exact bf16 values
        ref_xn = oracle.rms_norm(h, eps=st.eps)
        assert np.all(np.abs(xn - ref_xn) <= 2.0 ** -8 * np.abs(ref_xn) + 1e-6), f"layer {i} norm"
        logits = b["logits"].cpu().numpy()
        ridx, _, _ = oracle.route(logits, s.k)
        assert np.array_equal(b["idx"].cpu().numpy(), ridx), f"layer {i} routing"
        roff, rpairs = oracle.group(ridx, s.E)
        assert np.array_equal(b["offsets"].cpu().numpy(), roff), f"layer {i} offsets"
        assert np.array_equal(b["pairs"].cpu().numpy(), rpairs), f"layer {i} pairs"
        assert_rms_close(logits, oracle.router_logits(sl.wr, xn), 1e-5, f"layer {i} logits")
        out = b["out"].cpu().numpy().astype(np.float64)
        for t in sample:
            r = oracle.moe_layer(sl.expert, sl.wr, xn[t:t + 1], s.k, s.d, s.f,
                                 route_logits=logits[t:t + 1])
            delta = r["out"][0] - xn[t]          # sum_slot w * expert(xn)
            assert_rms_close(out[t] - h[t], delta, tol, f"layer {i} token {t}")
        h = out
        sl.forget()
    st.close()
    torch.cuda.empty_cache()
