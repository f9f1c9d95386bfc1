"""GPU parity: code packing, the standalone lookup-table build and the RVQ GEMV
against the CPU oracle (through the C ABI)."""
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
rng = np.random.default_rng(7)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def packed_matrix(codes, cb, rows, cols):
    c = to_dev(codes)
    packed = torch.empty(rvq.rvq_code_bytes(rows, cols), dtype=torch.uint8, device=DEV)
    rvq.rvq_pack(c, rows, cols, packed)
    cbp = torch.empty(6144, dtype=torch.float32, device=DEV)
    rvq.rvq_pack_codebooks(to_dev(cb), cbp)
    return packed, cbp


def gemv(codes, cb, rows, cols, x_dev, n):
    packed, cbp = packed_matrix(codes, cb, rows, cols)
    ws = torch.empty(rvq.rvq_gemv_workspace_bytes(rows, cols, n), dtype=torch.uint8, device=DEV)
    rvq.rvq_ws_clear(ws)
    y = torch.empty((n, rows), dtype=torch.float32, device=DEV)
    rvq.rvq_gemv(packed, cbp, rows, cols, x_dev, n, y, ws)
    assert rvq.rvq_ws_status(ws) == (0, 0)
    return y.cpu().numpy()


@pytest.mark.parametrize("rows,cols", [(32, 512), (96, 1024), (2048, 7168)])
def test_pack_roundtrip_and_layout(rows, cols):
    codes = rng.integers(0, 256, size=(rows, cols // 8, 3), dtype=np.uint8)
    c = to_dev(codes)
    packed = torch.empty(rvq.rvq_code_bytes(rows, cols), dtype=torch.uint8, device=DEV)
    rvq.rvq_pack(c, rows, cols, packed)
    back = torch.empty_like(c)
    rvq.rvq_unpack(packed, rows, cols, back)
    assert torch.equal(back, c)
    p = packed.cpu().numpy()
    assert p.size == 3 * rows * cols // 8
    # spot-check the documented layout at random positions
    RB = rows // 32
    for _ in range(200):
        r, j, s = rng.integers(rows), rng.integers(cols // 8), rng.integers(3)
        g, b, l = j // 32, r // 32, r % 32
        t = (j % 32 - l) % 32
        h, i = divmod(t, 16)
        off = (g * RB + b) * 3072 + ((s * 2 + h) * 32 + l) * 16 + i
        assert p[off] == codes[r, j, s]


def test_pack_codebooks_layout():
    cb = rng.normal(size=(3, 256, 8)).astype(np.float32)
    out = torch.empty(6144, dtype=torch.float32, device=DEV)
    rvq.rvq_pack_codebooks(to_dev(cb), out)
    o = out.cpu().numpy()
    for s in range(3):
        for k in (0, 1, 77, 254, 255):
            for i in range(8):
                assert o[((s * 128 + k // 2) * 8 + i) * 2 + (k & 1)] == cb[s, k, i]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_lut_build_matches_oracle(dtype):
    n, cols = 3, 64
    cb = rng.normal(0, 0.02, size=(3, 256, 8)).astype(np.float32)
    xf = rng.normal(size=(n, cols)).astype(np.float32)
    if dtype == "bf16":
        bits = synth.f32_to_bf16(xf)
        x_dev, x64 = bf16_dev(bits), synth.bf16_to_f32(bits).astype(np.float64)
    else:
        x_dev, x64 = to_dev(xf), xf.astype(np.float64)
    lut = torch.empty((n, cols // 8, 3, 256), dtype=torch.float32, device=DEV)
    rvq.rvq_lut_build(to_dev(cb), x_dev, n, cols, lut)
    got = lut.cpu().numpy()
    for t in range(n):
        ref = oracle.rvq_lut_build(cb, x64[t], cols)
        assert_rms_close(got[t], ref, 1e-5, f"lut token {t}")


def test_gemv_single_matrix_workload():
    """The 256 x 512 single-GEMV workload, fp32 x, batch 1."""
    wl = W.WORKLOADS[0]
    lseed = W.layer_seed(0, 0)
    mseed = W.matrix_seed(lseed, 0, 0)
    codes = W.codes(mseed, wl.rows, wl.cols)
    cb = W.codebooks(mseed)
    x = W.tokens_f32(lseed, 1, wl.cols)
    y = gemv(codes, cb, wl.rows, wl.cols, to_dev(x), 1)
    ref = oracle.rvq_gemv(codes, cb, wl.rows, wl.cols, x.astype(np.float64))
    assert_rms_close(y, ref, 1e-4, "cfg0 y")


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gemv_multi_tile(n, dtype):
    """512 x 2048: 16 row tiles, 8 chunk groups; odd n mixes both item kinds."""
    rows, cols = 512, 2048
    codes = rng.integers(0, 256, size=(rows, cols // 8, 3), dtype=np.uint8)
    cb = np.stack([rng.normal(0, s, size=(256, 8)) for s in W.STAGE_SIGMA]).astype(np.float32)
    xf = rng.normal(size=(n, cols)).astype(np.float32)
    if dtype == "bf16":
        bits = synth.f32_to_bf16(xf)
        x_dev, x64 = bf16_dev(bits), synth.bf16_to_f32(bits).astype(np.float64)
    else:
        x_dev, x64 = to_dev(xf), xf.astype(np.float64)
    y = gemv(codes, cb, rows, cols, x_dev, n)
    ref = oracle.rvq_gemv(codes, cb, rows, cols, x64)
    assert_rms_close(y, ref, 1e-4, f"gemv n={n}")


def test_gemv_closed_form_is_exact():
    """One-hot stage-2 codebook, x = 1: y[r] = 8 * #{chunks with code k*} exactly."""
    rows, cols, kstar = 64, 1024, 200
    codes = rng.integers(0, 256, size=(rows, cols // 8, 3), dtype=np.uint8)
    codes[::2, ::3, 1] = kstar
    cb = np.zeros((3, 256, 8), np.float32)
    cb[1, kstar] = 1.0
    y = gemv(codes, cb, rows, cols, to_dev(np.ones((1, cols), np.float32)), 1)[0]
    expect = 8.0 * (codes[:, :, 1] == kstar).sum(axis=1)
    assert np.array_equal(y, expect)
