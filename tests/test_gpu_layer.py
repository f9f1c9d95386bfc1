"""GPU parity for whole MoE layers (router -> top-k -> RVQ SwiGLU expert FFN
-> weighted combine + residual) against the oracle, plus device-side fault
reporting.  Routing is compared bit-exact with the oracle routing the GPU's
own fp32 logits; floats within 1e-4 x RMS."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import workloads as W
from tests.support import SynthLayer, assert_rms_close, bf16_bits_to_f64

pytestmark = pytest.mark.gpu
rvq = pytest.importorskip("moe_expert_ffn_router_gb300")
DEV = "cuda"

_layers = {}


def layer(config, n_experts=None):
    key = (config, n_experts)
    if key not in _layers:
        sl = SynthLayer(config, 0, n_experts=n_experts)
        _layers[key] = (sl, sl.to_gpu())
    return _layers[key]


def drop_layers():
    _layers.clear()
    torch.cuda.empty_cache()


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def check_layer(sl, L, x_bits, tokens=None, steps=False):
    n = x_bits.shape[0]
    x = bf16_dev(x_bits)
    b = L.forward_steps(x) if steps else L.forward(x)
    torch.cuda.synchronize()
    assert L.status(n) == (0, 0)
    logits = b["logits"].cpu().numpy()
    idx, w = b["idx"].cpu().numpy(), b["w"].cpu().numpy()
    off, pairs = b["offsets"].cpu().numpy(), b["pairs"].cpu().numpy()
    out = b["out"].cpu().numpy()
    x64 = bf16_bits_to_f64(x_bits)
    s = sl.shape
    # logits against the oracle's own
    ref_lg = oracle.router_logits(sl.wr, x64)
    assert_rms_close(logits, ref_lg, 1e-5, "logits")
    # routing and grouping bit-exact given the GPU's logits
    ridx, rw, _ = oracle.route(logits, s.k)
    assert np.array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=2e-6, atol=1e-9)
    roff, rpairs = oracle.group(ridx, L.E)
    assert np.array_equal(off, roff) and np.array_equal(pairs, rpairs)
    # expert outputs and combine on a subset of tokens (all by default); the
    # oracle layers run on a thread pool (the C oracle releases the GIL), with
    # the sampled tokens' experts generated first
    tokens = list(range(n) if tokens is None else tokens)
    for t in tokens:
        for e in idx[t]:
            sl.expert(int(e))
    with ThreadPoolExecutor(max_workers=max(1, min(len(tokens), os.cpu_count() or 1))) as ex:
        refs = list(ex.map(lambda t: oracle.moe_layer(sl.expert, sl.wr, x64[t:t + 1], s.k, s.d,
                                                      s.f, route_logits=logits[t:t + 1]),
                           tokens))
    for t, r in zip(tokens, refs):
        assert np.array_equal(r["idx"][0], idx[t])
        delta_ref = r["out"][0] - x64[t]
        assert_rms_close(out[t] - x64[t], delta_ref, 1e-4, f"token {t} out-x")
        assert_rms_close(out[t], r["out"][0], 1e-4, f"token {t} out")
        if steps:
            yp = b["y_pair"].cpu().numpy()[t * s.k:(t + 1) * s.k]
            assert_rms_close(yp, r["y_pair"], 1e-4, f"token {t} y_pair")
    return b


@pytest.mark.parametrize("n", [1, 4, 16])
def test_decode_layer_d2048(n):
    sl, L = layer(1)
    check_layer(sl, L, sl.tokens_bf16(n))


def test_decode_layer_separate_calls():
    sl, L = layer(1)
    check_layer(sl, L, sl.tokens_bf16(5), steps=True)


def test_repeated_tokens_make_large_groups():
    """Seven copies of one token and two others: experts with 7-9 tokens
    (two-token items and an odd remainder) next to single-token experts."""
    sl, L = layer(1)
    base = sl.tokens_bf16(3)
    xb = np.concatenate([np.repeat(base[:1], 7, axis=0), base[1:]])
    b = check_layer(sl, L, xb, tokens=[0, 6, 7, 8])
    counts = np.diff(b["offsets"].cpu().numpy())
    assert counts.max() >= 7


def test_fp32_residual_input():
    """Layer input in fp32 (the residual stream of a stack)."""
    sl, L = layer(1)
    n = 3
    x32 = synth.bf16_to_f32(sl.tokens_bf16(n)) * np.float32(1.37)
    b = L.forward(torch.from_numpy(x32).to(DEV))
    torch.cuda.synchronize()
    assert L.status(n) == (0, 0)
    logits, out = b["logits"].cpu().numpy(), b["out"].cpu().numpy()
    for t in range(n):
        r = oracle.moe_layer(sl.expert, sl.wr, x32[t:t + 1].astype(np.float64), 8, 2048, 1024,
                             route_logits=logits[t:t + 1])
        assert_rms_close(out[t] - x32[t], r["out"][0] - x32[t], 1e-4, "fp32 out-x")


def test_corrupt_record_is_reported_not_used():
    sl, L = layer(1)
    n = 2
    xb = sl.tokens_bf16(n)
    b = L.forward(bf16_dev(xb))
    torch.cuda.synchronize()
    e = int(b["idx"][0, 0])
    rec = L.record(e)
    saved = rec[:4].clone()
    try:
        rec[:4] = 0                                    # break the magic of a selected expert
        with pytest.raises(rvq.RvqError) as ei:
            L.validate()
        assert ei.value.status == "RVQ_ECORRUPT"
        L.forward(bf16_dev(xb))
        rc, bits = L.status(n)
        assert bits & rvq.DEV_ERR_CORRUPT and rc == 4
    finally:
        rec[:4] = saved
    L.validate()
    L.forward(bf16_dev(xb))
    assert L.status(n) == (0, 0)


def test_bad_offsets_are_reported():
    sl, L = layer(1)
    n, k = 2, 8
    x = bf16_dev(sl.tokens_bf16(n))
    b = L.buffers(n)
    off = torch.zeros(L.E + 1, dtype=torch.int32, device=DEV)
    off[-1] = n * k + 5                                # inconsistent total
    pairs = torch.arange(n * k, dtype=torch.int32, device=DEV)
    y = torch.empty((n * k, L.d), dtype=torch.float32, device=DEV)
    rvq.moe_expert_ffn(L.bank, x, n, k, off, pairs, y, b["ws"])
    rc, bits = L.status(n)
    assert bits & rvq.DEV_ERR_INDEX and rc == 5


@pytest.mark.parametrize("n,sample", [(1, [0]), (8, [0, 5]),
                                      (64, [0, 9, 18, 27, 36, 45, 54, 63])])
def test_k3_shaped_layer_full_size(n, sample):
    """d=7168, f=2048, 256 experts, top-16, 4.2 GB bank: all outputs of the
    sampled tokens against the oracle; routing of every token bit-exact.  At
    64 tokens the lookup tables serve two tokens of an expert at a time, and
    an expert with an odd token count gives its last token a one-token item:
    the sample covers pairs of both kinds."""
    drop_layers()
    sl, L = layer(2)
    b = check_layer(sl, L, sl.tokens_bf16(n), tokens=sample)
    if n == 64:
        off, pairs = b["offsets"].cpu().numpy(), b["pairs"].cpu().numpy()
        kinds = set()
        for e in range(L.E):
            seg = pairs[off[e]:off[e + 1]]
            for j, p in enumerate(seg):
                if p // L.k in sample:
                    kinds.add("odd remainder" if len(seg) % 2 and j == len(seg) - 1 else "pair")
        assert kinds == {"odd remainder", "pair"}, kinds
    sl.forget()


@pytest.mark.parametrize("kind", ["pinned", "pageable", "pinned_unaligned"])
def test_host_buffer_layer_call_equals_device_call(kind):
    """moe_layer_forward_host gives bit for bit the device-buffer layer's
    outputs, over several steps on the same buffers.  Pinned buffers (mapped:
    moved by the call's copy kernels), pageable ones and pinned ones off a
    16-byte boundary (both by cudaMemcpyAsync)."""
    sl, L = layer(1)
    n = 3
    pool = sl.tokens_bf16(3 * n)
    x_host = torch.empty((n, L.d), dtype=torch.bfloat16)
    out_host = torch.full((n, L.d), float("nan"), dtype=torch.float32)
    if kind == "pinned":
        x_host, out_host = x_host.pin_memory(), out_host.pin_memory()
    elif kind == "pinned_unaligned":
        # views one element into larger pinned buffers: 2 and 4 bytes off
        x_host = torch.empty(n * L.d + 1, dtype=torch.bfloat16).pin_memory()[1:].view(n, L.d)
        out_host = torch.full((n * L.d + 1,), float("nan"),
                              dtype=torch.float32).pin_memory()[1:].view(n, L.d)
        assert x_host.data_ptr() % 16 and out_host.data_ptr() % 16
    b = L.buffers(n)
    for step in range(3):
        bits = pool[step * n:(step + 1) * n]
        x_host.view(torch.int16).copy_(torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)))
        hb = L.forward_host(x_host, out_host, b)
        torch.cuda.synchronize()
        assert L.status(n) == (0, 0)
        got = out_host.clone()
        ref = L.forward(bf16_dev(bits))
        torch.cuda.synchronize()
        assert torch.equal(got, ref["out"].cpu()), step
        assert torch.equal(hb["x_dev"].cpu().view(torch.int16), x_host.view(torch.int16)), step


def test_layer_graph_replays_the_direct_call():
    """A layer recorded as a CUDA graph (moe_layer_graph_create) and launched
    step after step gives bit for bit what the direct layer call gives on the
    same inputs: routing, pair plan, expert FFN and combine, for lookup-table
    decode batches, through host buffers, and with tensor-core dispatch."""
    sl, L = layer(1)
    pool = sl.tokens_bf16(3 * 40)
    # decode batch on device buffers: new tokens copied into x_dev between launches
    n = 4
    x_dev = torch.empty((n, L.d), dtype=torch.bfloat16, device=DEV)
    b = L.buffers(n)
    g = L.graph(x_dev, b)
    for step in range(3):
        bits = pool[step * n:(step + 1) * n]
        x_dev.copy_(bf16_dev(bits))
        g.launch()
        torch.cuda.synchronize()
        got = b["out"].clone()
        idx = b["idx"].clone()
        ref = L.forward(bf16_dev(bits))
        torch.cuda.synchronize()
        assert torch.equal(got, ref["out"]), step
        assert torch.equal(idx, ref["idx"]), step
    assert L.status(n) == (0, 0)
    g.close()
    # the same batch through pinned host buffers recorded in the graph
    x_host = torch.empty((n, L.d), dtype=torch.bfloat16).pin_memory()
    out_host = torch.full((n, L.d), float("nan"), dtype=torch.float32).pin_memory()
    x2 = torch.empty((n, L.d), dtype=torch.bfloat16, device=DEV)
    b2 = L.buffers(n)
    g2 = L.graph(x2, b2, x_host=x_host, out_host=out_host)
    for step in range(2):
        bits = pool[40 + step * n:40 + (step + 1) * n]
        x_host.view(torch.int16).copy_(torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)))
        g2.launch()
        torch.cuda.synchronize()
        ref = L.forward(bf16_dev(bits))
        torch.cuda.synchronize()
        assert torch.equal(out_host, ref["out"].cpu()), step
    g2.close()
    # a prefill-sized batch with every expert on the tensor cores
    n = 40
    x3 = torch.empty((n, L.d), dtype=torch.bfloat16, device=DEV)
    b3 = L.buffers(n)
    g3 = L.graph(x3, b3, tc_min_tokens=1)
    bits = pool[80:120]
    x3.copy_(bf16_dev(bits))
    g3.launch()
    torch.cuda.synchronize()
    ref = L.forward(bf16_dev(bits), tc_min_tokens=1)
    torch.cuda.synchronize()
    assert torch.equal(b3["out"], ref["out"])
    assert L.status(n) == (0, 0)
    g3.close()
