"""GPU parity for the offline RVQ encoder (residual k-means, 3 x 256 codewords
of 8 dimensions): codes bit-exact and codebooks bit-identical to the oracle
on small matrices (ragged sub-vector counts, N = 256 exactly, an all-zero
matrix, Lloyd rounds 0..4); at the size of one K3 expert matrix
(2048 x 7168), where the oracle takes minutes, properties that hold at any
size: two runs bit-identical, every code a nearest codeword of its stage's
residual, and the encoded matrix closer to w than stage 1 alone.  The
encoder's canonical layout feeds the bank format as it is: packed and run
through the LUT GEMV, the encoded matrix gives the oracle GEMV of the
oracle's codes."""
import numpy as np
import pytest
import torch

import oracle
from tests.support import assert_rms_close

pytestmark = pytest.mark.gpu
rvq = pytest.importorskip("moe_expert_ffn_router_gb300")
DEV = "cuda"


def encode_gpu(w, iters):
    rows, cols = w.shape
    wd = torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(DEV)
    codes = torch.empty((rows, cols // 8, 3), dtype=torch.uint8, device=DEV)
    cb = torch.empty((3, 256, 8), dtype=torch.float32, device=DEV)
    ws = torch.empty(rvq.rvq_encode_workspace_bytes(rows, cols), dtype=torch.uint8, device=DEV)
    rvq.rvq_encode(wd, rows, cols, iters, codes, cb, ws)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), cb.cpu().numpy()


def gaussian(rows, cols, seed, sigma=0.02):
    return np.random.default_rng(seed).normal(0, sigma, size=(rows, cols)).astype(np.float32)


@pytest.mark.parametrize("rows,cols,iters", [
    (256, 512, 0), (256, 512, 4), (37, 72, 3), (1, 2048, 2), (512, 2048, 2)])
def test_encode_bit_exact(rows, cols, iters):
    w = gaussian(rows, cols, seed=rows * 7 + cols + iters)
    got_codes, got_cb = encode_gpu(w, iters)
    ref_codes, ref_cb = oracle.rvq_encode(w, iters)
    assert np.array_equal(got_codes, ref_codes)
    assert np.array_equal(got_cb.view(np.uint32), ref_cb.view(np.uint32))
    if rows % 32 == 0 and cols % 512 == 0:
        n = 2
        x = np.random.default_rng(rows).normal(size=(n, cols)).astype(np.float32)
        packed = torch.empty(rvq.rvq_code_bytes(rows, cols), dtype=torch.uint8, device=DEV)
        rvq.rvq_pack(torch.from_numpy(got_codes).to(DEV), rows, cols, packed)
        cbp = torch.empty(6144, dtype=torch.float32, device=DEV)
        rvq.rvq_pack_codebooks(torch.from_numpy(got_cb).to(DEV), cbp)
        ws = torch.empty(rvq.rvq_gemv_workspace_bytes(rows, cols, n), dtype=torch.uint8, device=DEV)
        rvq.rvq_ws_clear(ws)
        y = torch.empty((n, rows), dtype=torch.float32, device=DEV)
        rvq.rvq_gemv(packed, cbp, rows, cols, torch.from_numpy(x).to(DEV), n, y, ws)
        assert rvq.rvq_ws_status(ws) == (0, 0)
        assert_rms_close(y.cpu().numpy(), oracle.rvq_gemv(ref_codes, ref_cb, rows, cols, x), 1e-4,
                         "gemv of encoded matrix")


def test_encode_heavy_ties_and_zero_matrix():
    """An all-zero matrix (every sub-vector ties with every codeword: code 0
    throughout) and a matrix of four repeated values with wide magnitude
    spread (many members per codeword, negative sums)."""
    z = np.zeros((64, 256), np.float32)
    c, cb = encode_gpu(z, 3)
    assert not c.any() and not cb.any()
    rng = np.random.default_rng(5)
    w = rng.choice(np.float32([-100.0, -1e-3, 2.5e-7, 64.0]), size=(128, 256)).astype(np.float32)
    got = encode_gpu(w, 3)
    ref = oracle.rvq_encode(w, 3)
    assert np.array_equal(got[0], ref[0])
    assert np.array_equal(got[1].view(np.uint32), ref[1].view(np.uint32))


def _residuals(w, codes, cb):
    """Residual before each stage, computed in fp32 as the encoder does."""
    r = w.reshape(-1, 8).astype(np.float32)
    c = codes.reshape(-1, 3)
    out = []
    for s in range(3):
        out.append(r)
        r = (r - cb[s][c[:, s]]).astype(np.float32)
    return out, r


def test_encode_k3_expert_matrix_properties():
    rows, cols, iters = 2048, 7168, 2
    w = gaussian(rows, cols, seed=91)
    c1, cb1 = encode_gpu(w, iters)
    c2, cb2 = encode_gpu(w, iters)
    assert np.array_equal(c1, c2) and np.array_equal(cb1.view(np.uint32), cb2.view(np.uint32))
    rng = np.random.default_rng(0)
    N = rows * cols // 8
    pick = np.sort(rng.choice(N, 4096, replace=False))
    res, last = _residuals(w, c1, cb1)
    cc = c1.reshape(-1, 3)
    for s in range(3):
        r = res[s][pick].astype(np.float64)
        dist = ((r[:, None, :] - cb1[s][None].astype(np.float64)) ** 2).sum(-1)
        got = dist[np.arange(len(pick)), cc[pick, s]]
        assert np.all(got <= dist.min(1) * (1 + 1e-5) + 1e-14), f"stage {s}"
    rms = float(np.sqrt((w.astype(np.float64) ** 2).mean()))
    err3 = float(np.sqrt((last.astype(np.float64) ** 2).mean())) / rms
    err1 = float(np.sqrt((res[1].astype(np.float64) ** 2).mean())) / rms
    assert err3 < err1 < 1.0
    assert err3 < 0.25, err3  # 24 bits per 8 weights on Gaussian data

