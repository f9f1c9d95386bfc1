"""GPU parity for the router: logits within tolerance, selection, weights and
grouping bit-exact against the oracle given the same fp32 logits."""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import workloads as W
from tests.support import assert_rms_close

pytestmark = pytest.mark.gpu
rvq = pytest.importorskip("moe_expert_ffn_router_gb300")
DEV = "cuda"
rng = np.random.default_rng(11)


def run_route(logits: np.ndarray, k: int):
    n, E = logits.shape
    lg = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).to(DEV)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    pairs = torch.empty(n * k, dtype=torch.int32, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    rvq.moe_route(lg, n, E, k, idx, w, off, pairs, ws)
    rc, bits = rvq.rvq_ws_status(ws)
    return idx.cpu().numpy(), w.cpu().numpy(), off.cpu().numpy(), pairs.cpu().numpy(), rc, bits


def check_route(logits, k):
    idx, w, off, pairs, rc, bits = run_route(logits, k)
    assert (rc, bits) == (0, 0)
    ridx, rw, rrc = oracle.route(logits, k)
    roff, rpairs = oracle.group(ridx, logits.shape[1])
    assert rrc == 0
    assert np.array_equal(idx, ridx)
    assert np.array_equal(off, roff)
    assert np.array_equal(pairs, rpairs)
    np.testing.assert_allclose(w, rw, rtol=2e-6, atol=1e-9)


@pytest.mark.parametrize("n,E,k", [(1, 64, 8), (4, 64, 8), (16, 64, 8), (1, 256, 16),
                                   (8, 256, 16), (64, 256, 16), (333, 256, 16), (2048, 256, 16),
                                   (5, 16, 16), (7, 40, 3), (1, 1, 1)])
def test_route_random(n, E, k):
    check_route(rng.normal(size=(n, E)).astype(np.float32), k)


@pytest.mark.parametrize("E,k", [(256, 16), (64, 8), (16, 16)])
def test_route_at_the_single_launch_token_limit(E, k):
    """The largest batch one routing call takes (its grouping runs in one
    block's shared memory): selection, weights and grouping still bit-exact,
    and the next size up is refused before any launch."""
    n = rvq.moe_route_max_tokens(E)
    check_route(rng.normal(size=(n, E)).astype(np.float32), k)
    with pytest.raises(RuntimeError):
        run_route(np.zeros((n + 1, E), np.float32), k)


def test_route_ties_and_degenerate():
    E, k = 256, 16
    lg = np.round(rng.normal(size=(50, E)) * 2).astype(np.float32)   # many exact ties
    lg[3] = 0.0                                                        # all equal
    lg[4] = -0.0
    lg[5, ::2] = -0.0                                                  # signed zeros tie
    lg[6] = np.float32(1e30)
    check_route(lg, k)
    check_route(lg[:, :64], 1)                                         # k = 1 (argmax)
    check_route(np.tile(lg, (3, 1)), k)                    # > 64 tokens: grid-wide selection


def test_route_skewed_prefill_counts():
    """Zipf-skewed logits: tokens per expert spanning one to hundreds."""
    n, E, k = 2048, 256, 16
    bias = W.zipf_bias(W.layer_seed(4), E, W.PREFILL_ZIPF_BETA)
    lg = (rng.normal(size=(n, E)) * 1.7 + bias).astype(np.float32)
    check_route(lg, k)


def test_route_flags_non_finite():
    lg = rng.normal(size=(4, 64)).astype(np.float32)
    lg[2, 5] = np.nan
    idx, w, off, pairs, rc, bits = run_route(lg, 8)
    assert bits & rvq.DEV_ERR_NONFINITE and rc != 0
    assert ((idx >= 0) & (idx < 64)).all()          # outputs stay in range
    assert off[-1] == 4 * 8
    big = rng.normal(size=(100, 64)).astype(np.float32)
    big[77, 3] = np.inf
    idx, w, off, pairs, rc, bits = run_route(big, 8)
    assert bits & rvq.DEV_ERR_NONFINITE and rc != 0
    assert ((idx >= 0) & (idx < 64)).all() and off[-1] == 100 * 8


@pytest.mark.parametrize("config,n", [(1, 1), (1, 16), (2, 1), (2, 64), (1, 65), (2, 300)])
def test_router_logits_match_oracle(config, n):
    s = W.WORKLOADS[config].shape
    lseed = W.layer_seed(config)
    wr = W.router_weight(lseed, s.E, s.d)
    bits = W.tokens_bf16(lseed, n, s.d)
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    out = torch.empty((n, s.E), dtype=torch.float32, device=DEV)
    rvq.moe_router_logits(torch.from_numpy(wr).to(DEV), None, x, n, s.E, s.d, out)
    ref = oracle.router_logits(wr, synth.bf16_to_f32(bits).astype(np.float64))
    assert_rms_close(out.cpu().numpy(), ref, 1e-5, "logits")


def test_router_logits_prefill_chunk():
    """2048 tokens with the Zipf router bias (the tiled path), bf16 and fp32 x."""
    wl = W.WORKLOADS[4]
    s = wl.shape
    lseed = W.layer_seed(4)
    wr = W.router_weight(lseed, s.E, s.d)
    bias = W.zipf_bias(lseed, s.E, wl.zipf_beta)
    n = 2048
    bits = W.tokens_bf16(lseed, n, s.d)
    x64 = synth.bf16_to_f32(bits).astype(np.float64)
    ref = oracle.router_logits(wr, x64, bias)
    for x in (torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16),
              torch.from_numpy(x64.astype(np.float32)).to(DEV)):
        out = torch.empty((n, s.E), dtype=torch.float32, device=DEV)
        rvq.moe_router_logits(torch.from_numpy(wr).to(DEV), torch.from_numpy(bias).to(DEV), x, n,
                              s.E, s.d, out)
        assert_rms_close(out.cpu().numpy(), ref, 1e-5, "prefill logits")


def test_router_bias():
    E, d, n = 64, 1024, 3
    wr = rng.normal(0, 0.02, size=(E, d)).astype(np.float32)
    b = rng.normal(size=E).astype(np.float32)
    x = rng.normal(size=(n, d)).astype(np.float32)
    out = torch.empty((n, E), dtype=torch.float32, device=DEV)
    rvq.moe_router_logits(torch.from_numpy(wr).to(DEV), torch.from_numpy(b).to(DEV),
                          torch.from_numpy(x).to(DEV), n, E, d, out)
    ref = oracle.router_logits(wr, x.astype(np.float64), b)
    assert_rms_close(out.cpu().numpy(), ref, 1e-5, "biased logits")
