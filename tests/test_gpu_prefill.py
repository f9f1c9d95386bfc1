"""GPU parity for the prefill (tensor-core) path of the expert FFN: RVQ code
tiles decoded to fp16 and multiplied on tcgen05 with fp16 tokens.  Held to 2e-2 x RMS per pair
output against the double-precision oracle; experts left on the lookup-table
path in a mixed dispatch stay at 1e-4 x RMS.  Routing is the GPU's own (bit-
exactness of routing is covered by test_gpu_router / test_gpu_layer)."""
import os

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
TC_TOL, LUT_TOL = 2e-2, 1e-4

_cache = {}


def layer(config, bias_beta=None):
    key = (config, bias_beta)
    if key not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        sl = SynthLayer(config, 0)
        bias = None
        if bias_beta is not None:
            bias = W.zipf_bias(sl.src.lseed, sl.shape.E, bias_beta)
        L = sl.to_gpu(bias=bias)
        _cache[key] = (sl, L, bias)
    return _cache[key]


def route(L, x, n):
    b = L.buffers(n)
    rvq.moe_router_logits(L.wr, L.bias, x, n, L.E, L.d, b["logits"])
    rvq.moe_route(b["logits"], n, L.E, L.k, b["idx"], b["w"], b["offsets"], b["pairs"], b["ws"])
    return b


def run_ffn(L, x, n, b, tc_min_tokens):
    y = torch.full((n * L.k, L.d), float("nan"), dtype=torch.float32, device=DEV)
    rvq.moe_expert_ffn_ex(L.bank, x, n, L.k, b["offsets"], b["pairs"], y, b["ws"], tc_min_tokens)
    torch.cuda.synchronize()
    assert L.status(n) == (0, 0)
    return y.cpu().numpy()


def check_pairs(sl, x64, idx, y, pairs, tol_of):
    s = sl.shape
    for p in pairs:
        t, slot = divmod(int(p), s.k)
        e = int(idx[t, slot])
        ref = oracle.expert_ffn(*sl.expert(e), s.d, s.f, x64[t])
        assert_rms_close(y[p], ref, tol_of(e), f"pair {p} (token {t}, expert {e})")


def test_tensor_core_path_all_experts_d2048():
    sl, L, _ = layer(1)
    n = 40
    bits = sl.tokens_bf16(n)
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    b = route(L, x, n)
    y = run_ffn(L, x, n, b, tc_min_tokens=1)
    idx = b["idx"].cpu().numpy()
    x64 = bf16_bits_to_f64(bits)
    check_pairs(sl, x64, idx, y, range(0, n * L.k, 3), lambda e: TC_TOL)
    # whole layer through the combine
    out = torch.empty((n, L.d), dtype=torch.float32, device=DEV)
    rvq.moe_combine(torch.from_numpy(y).to(DEV), b["w"], n, L.k, L.d, x, out)
    torch.cuda.synchronize()
    w = b["w"].cpu().numpy()
    for t in (0, n - 1):
        ref_y = np.stack([oracle.expert_ffn(*sl.expert(int(idx[t, q])), sl.shape.d, sl.shape.f,
                                            x64[t]) for q in range(L.k)])
        ref = oracle.combine(ref_y, w[t:t + 1], x64[t:t + 1])[0]
        assert_rms_close(out.cpu().numpy()[t] - x64[t], ref - x64[t], TC_TOL, "out - x")


def test_tensor_core_path_fp32_input():
    """fp32 activations on the tensor-core path: the token conversion reads
    fp32 rows instead of bf16 rows.  The values are bf16-representable, so
    the fp16 conversion is exact and the tolerance applies unchanged."""
    sl, L, _ = layer(1)
    n = 24
    x32 = synth.bf16_to_f32(sl.tokens_bf16(n))
    x = torch.from_numpy(x32).to(DEV)
    b = route(L, x, n)
    y = run_ffn(L, x, n, b, tc_min_tokens=1)
    idx = b["idx"].cpu().numpy()
    check_pairs(sl, x32.astype(np.float64), idx, y, range(0, n * L.k, 2), lambda e: TC_TOL)


def test_mixed_dispatch_by_group_size():
    """Seven copies of each of two tokens plus ten others: their experts get
    groups of >= 7 tokens (tensor cores); the rest stay on lookup tables."""
    sl, L, _ = layer(1)
    base = sl.tokens_bf16(12)
    bits = np.concatenate([np.repeat(base[:2], 7, axis=0), base[2:]])
    n = bits.shape[0]
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    b = route(L, x, n)
    offs = b["offsets"].cpu().numpy()
    counts = np.diff(offs)
    thr = 7
    assert (counts >= thr).any() and ((counts > 0) & (counts < thr)).any()
    y = run_ffn(L, x, n, b, tc_min_tokens=thr)
    idx = b["idx"].cpu().numpy()
    x64 = bf16_bits_to_f64(bits)
    sample = [p for p in range(n * L.k) if p % 5 == 0]
    check_pairs(sl, x64, idx, y, sample,
                lambda e: TC_TOL if counts[e] >= thr else LUT_TOL)


def test_mixed_dispatch_small_batch_fused_swiglu():
    """Four tokens, two of them equal: their experts get groups of two
    (tensor cores at threshold 2) and the rest one token each (lookup
    tables).  Up to 4 tokens the lookup-table down launch reduces its own
    SwiGLU inputs, here with the tensor-core pairs skipped; every pair is
    compared with the oracle."""
    sl, L, _ = layer(1)
    base = sl.tokens_bf16(3)
    bits = np.concatenate([base[:1], base[:1], base[1:]])
    n = bits.shape[0]
    assert n == 4
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    b = route(L, x, n)
    counts = np.diff(b["offsets"].cpu().numpy())
    thr = 2
    assert (counts >= thr).any() and ((counts > 0) & (counts < thr)).any()
    y = run_ffn(L, x, n, b, tc_min_tokens=thr)
    idx = b["idx"].cpu().numpy()
    check_pairs(sl, bf16_bits_to_f64(bits), idx, y, range(n * L.k),
                lambda e: TC_TOL if counts[e] >= thr else LUT_TOL)


def test_prefill_chunk_full_size_zipf():
    """2048 tokens of the K3-shaped layer with the Zipf-skewed router bias
    (tokens per expert ~50-600, several 192-token passes for the largest
    groups); sampled pairs from the largest, a middle and the smallest group."""
    wl = W.WORKLOADS[4]
    sl, L, bias = layer(2, wl.zipf_beta)
    n = 2048
    bits = sl.tokens_bf16(n)
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    b = route(L, x, n)
    y = run_ffn(L, x, n, b, tc_min_tokens=1)
    offs = b["offsets"].cpu().numpy()
    pairs = b["pairs"].cpu().numpy()
    counts = np.diff(offs)
    order = np.argsort(counts)
    picks = []
    for e in [order[-1], order[-1], order[len(order) // 2], order[0]]:
        seg = pairs[offs[e]:offs[e + 1]]
        picks += [int(seg[0]), int(seg[-1])]
    idx = b["idx"].cpu().numpy()
    x64 = bf16_bits_to_f64(bits[sorted(set(p // L.k for p in picks))])
    rows = {t: i for i, t in enumerate(sorted(set(p // L.k for p in picks)))}
    s = sl.shape
    for p in sorted(set(picks)):
        t, slot = divmod(p, s.k)
        e = int(idx[t, slot])
        ref = oracle.expert_ffn(*sl.expert(e), s.d, s.f, x64[rows[t]])
        assert_rms_close(y[p], ref, TC_TOL, f"pair {p} (expert {e}, group {counts[e]})")
    assert np.isfinite(y).all()
    sl.forget()


@pytest.mark.parametrize("n", [2048, 300])
def test_layer_router_on_tensor_cores_k3(n):
    """The layer's router logits for a prefill-sized bf16 batch of the
    K3-shaped layer (Zipf bias) come from the tensor-core GEMM (Wr as three
    bf16 terms): within 1e-5 x RMS of the oracle's logits, routing and
    grouping bit-exact given them.  n = 300 leaves a ragged 44-token tile."""
    wl = W.WORKLOADS[4]
    sl, L, bias = layer(2, wl.zipf_beta)
    bits = sl.tokens_bf16(n)
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    b = L.forward(x, tc_min_tokens=1)
    torch.cuda.synchronize()
    assert L.status(n) == (0, 0)
    x64 = bf16_bits_to_f64(bits)
    logits = b["logits"].cpu().numpy()
    assert_rms_close(logits, oracle.router_logits(sl.wr, x64, bias), 1e-5, "tensor-core logits")
    idx, w = b["idx"].cpu().numpy(), b["w"].cpu().numpy()
    ridx, rw, _ = oracle.route(logits, L.k)
    assert np.array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=2e-6, atol=1e-9)
    roff, rpairs = oracle.group(ridx, L.E)
    assert np.array_equal(b["offsets"].cpu().numpy(), roff)
    assert np.array_equal(b["pairs"].cpu().numpy(), rpairs)
    assert np.isfinite(b["out"].cpu().numpy()).all()


def test_layer_forward_with_dispatch_d2048():
    """Whole layer through moe_layer_forward_ex for 100 tokens (tiled router
    logits, grid-wide selection, tensor-core experts, all-slot combine):
    routing bit-exact given the GPU's logits, sampled outputs within 2e-2."""
    sl, L, _ = layer(1)
    n = 100
    bits = sl.tokens_bf16(n)
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    b = L.forward(x, tc_min_tokens=1)
    torch.cuda.synchronize()
    assert L.status(n) == (0, 0)
    x64 = bf16_bits_to_f64(bits)
    s = sl.shape
    logits = b["logits"].cpu().numpy()
    assert_rms_close(logits, oracle.router_logits(sl.wr, x64), 1e-5, "logits")
    idx, w = b["idx"].cpu().numpy(), b["w"].cpu().numpy()
    ridx, rw, _ = oracle.route(logits, s.k)
    assert np.array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=2e-6, atol=1e-9)
    roff, rpairs = oracle.group(ridx, L.E)
    assert np.array_equal(b["offsets"].cpu().numpy(), roff)
    assert np.array_equal(b["pairs"].cpu().numpy(), rpairs)
    out = b["out"].cpu().numpy()
    for t in (0, 37, n - 1):
        r = oracle.moe_layer(sl.expert, sl.wr, x64[t:t + 1], s.k, s.d, s.f,
                             route_logits=logits[t:t + 1])
        assert_rms_close(out[t] - x64[t], r["out"][0] - x64[t], TC_TOL, f"token {t} out - x")


def test_combine_reduced_outputs_many_tokens():
    """moe_combine with one slot partial per pair and > 64 tokens (the
    all-slots-in-flight kernel), bf16 and fp32 residuals."""
    rng = np.random.default_rng(11)
    n, k, d = 100, 16, 1024
    y = rng.normal(size=(n * k, d)).astype(np.float32)
    w = rng.random(size=(n, k)).astype(np.float32)
    res = rng.normal(size=(n, d)).astype(np.float32)
    res_bits = synth.f32_to_bf16(res)
    cases = [(torch.from_numpy(res).to(DEV), res.astype(np.float64)),
             (torch.from_numpy(res_bits.view(np.int16)).to(DEV).view(torch.bfloat16),
              bf16_bits_to_f64(res_bits))]
    for r, r64 in cases:
        ref = oracle.combine(y.reshape(n, k, d), w, r64)
        out = torch.empty((n, d), dtype=torch.float32, device=DEV)
        rvq.moe_combine(torch.from_numpy(y).to(DEV), torch.from_numpy(w).to(DEV), n, k, d, r, out)
        torch.cuda.synchronize()
        assert_rms_close(out.cpu().numpy(), ref, 1e-5, "combine")


def test_stalled_pipeline_times_out_and_recovers():
    """Failure path of the tensor-core kernel without any fault: its MMA role
    waits for an arrival nothing makes; within a few seconds the kernel gives
    up, reports RVQ_DEV_ERR_TIMEOUT, frees its tensor memory, and the same
    bank and context then compute a correct layer."""
    import time
    sl, L, _ = layer(1)
    ws = L.workspace(1)
    t0 = time.time()
    rvq.rvq_selftest_prefill_timeout(L.bank, ws)
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert dt < 20.0, dt
    rc, bits = rvq.rvq_ws_status(ws)
    assert rc == 6 and bits & rvq.DEV_ERR_TIMEOUT, (rc, bits)   # RVQ_ETIMEOUT
    assert rvq.rvq_ws_status(ws) == (0, 0)                      # the read cleared it
    # the context is healthy: a full tensor-core layer is still correct
    test_tensor_core_path_all_experts_d2048()


def test_tokens_beyond_fp16_range_are_reported():
    """The tensor-core path computes on fp16 operands: a token value beyond
    the fp16 range (65,504) saturates and is reported as RVQ_DEV_ERR_NONFINITE
    in the workspace status, and the context stays usable.  The lookup-table
    path (fp32) takes the same input without a report."""
    sl, L, _ = layer(1)
    n = 8
    bits = sl.tokens_bf16(n).copy()
    bits[3, 17] = 0x47C3                     # bf16 99,840 (1.5234375 x 2^16)
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    b = route(L, x, n)
    y = torch.empty((n * L.k, L.d), dtype=torch.float32, device=DEV)
    rvq.moe_expert_ffn_ex(L.bank, x, n, L.k, b["offsets"], b["pairs"], y, b["ws"], 1)
    torch.cuda.synchronize()
    rc, flags = rvq.rvq_ws_status(b["ws"])
    assert rc == 5 and flags & rvq.DEV_ERR_NONFINITE, (rc, flags)   # RVQ_EDEVICE
    assert rvq.rvq_ws_status(b["ws"]) == (0, 0)                     # the read cleared it
    rvq.moe_expert_ffn_ex(L.bank, x, n, L.k, b["offsets"], b["pairs"], y, b["ws"], 0)
    torch.cuda.synchronize()
    assert rvq.rvq_ws_status(b["ws"]) == (0, 0)
    # the context is healthy: an in-range batch on the tensor cores is correct
    test_tensor_core_path_all_experts_d2048()


def test_prefill_multipass_groups_every_pair_d2048():
    """Groups larger than one pass of the tensor-core kernels (gate/up passes
    of at most 160 tokens, down passes of at most 192): 1024 tokens of the
    d = 2048 layer with a Zipf router bias strong enough (beta 0.5) that the
    three largest groups hold 760, 593 and 487 tokens, i.e. five, four and
    four gate/up passes (four, four and three down passes) with ragged last
    ones.
    Every pair of those three groups (1,840 pairs, first, middle and last
    passes alike) is compared with the oracle expert FFN at 2e-2 x RMS; the
    oracle calls run on a thread pool (the C oracle releases the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    sl, L, bias = layer(1, 0.5)
    n = 1024
    bits = sl.tokens_bf16(n)
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    b = route(L, x, n)
    y = run_ffn(L, x, n, b, tc_min_tokens=1)
    assert np.isfinite(y).all()
    offs = b["offsets"].cpu().numpy()
    pairs = b["pairs"].cpu().numpy()
    idx = b["idx"].cpu().numpy()
    counts = np.diff(offs)
    top3 = np.argsort(counts, kind="stable")[-3:]
    # (the oracle's routing of the same tokens gives 760, 593 and 487)
    assert counts[top3].min() > 2 * 192 and counts[top3].max() > 3 * 192, counts[top3]
    x64 = bf16_bits_to_f64(bits)
    s = sl.shape
    experts = {int(e): sl.expert(int(e)) for e in top3}
    work = [(int(p), int(e)) for e in top3 for p in pairs[offs[e]:offs[e + 1]]]

    def err(item):
        p, e = item
        t, slot = divmod(p, s.k)
        assert int(idx[t, slot]) == e
        ref = oracle.expert_ffn(*experts[e], s.d, s.f, x64[t])
        d = float(np.abs(y[p] - ref).max())
        r = float(np.sqrt(np.mean(ref * ref)))
        return d / r, p, e

    with ThreadPoolExecutor(max_workers=max(1, min(16, (os.cpu_count() or 1)))) as ex:
        res = list(ex.map(err, work))
    assert len(res) == int(counts[top3].sum())
    worst = max(res)
    assert worst[0] <= TC_TOL, f"pair {worst[1]} (expert {worst[2]}): max err {worst[0]:.3e} x RMS"
    sl.forget()
