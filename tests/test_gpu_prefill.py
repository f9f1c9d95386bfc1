"""GPU parity for the prefill (tensor-core) path of the expert FFN: RVQ code
tiles decoded to bf16 and multiplied on tcgen05.  Held to 2e-2 x RMS per pair
output against the double-precision oracle; experts left on the lookup-table
path in a mixed dispatch stay at 1e-4 x RMS.  Routing is the GPU's own (bit-
exactness of routing is covered by test_gpu_router / test_gpu_layer)."""
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


def test_prefill_chunk_full_size_zipf():
    """2048 tokens of the K3-shaped layer with the Zipf-skewed router bias
    (tokens per expert ~50-600, several 256-token passes for the largest
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
