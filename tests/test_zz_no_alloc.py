"""rvq_gemv_noalloc: the GEMV entry point for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).  Checked
through the C ABI against rvq_gemv with a caller workspace, on two calls in a
row, so the second call runs on scratch the first one left behind.

This file is collected last on purpose; it needs nothing from other tests.
"""
import numpy as np
import pytest
import torch

import synth
from synth import workloads as W
from tests.support import assert_rms_close

pytestmark = pytest.mark.gpu
rvq = pytest.importorskip("moe_expert_ffn_router_gb300")
DEV = "cuda"


def _matrix(rows, cols, seed):
    mseed = W.matrix_seed(W.layer_seed(7, seed), 0, 0)
    codes = torch.from_numpy(W.codes(mseed, rows, cols)).to(DEV)
    cb = torch.from_numpy(W.codebooks(mseed)).to(DEV)
    packed = torch.empty(rvq.rvq_code_bytes(rows, cols), dtype=torch.uint8, device=DEV)
    rvq.rvq_pack(codes, rows, cols, packed)
    cbp = torch.empty(6144, dtype=torch.float32, device=DEV)
    rvq.rvq_pack_codebooks(cb, cbp)
    return packed, cbp


def _with_workspace(packed, cbp, rows, cols, x, n):
    ws = torch.empty(rvq.rvq_gemv_workspace_bytes(rows, cols, n), dtype=torch.uint8, device=DEV)
    rvq.rvq_ws_clear(ws)
    y = torch.empty((n, rows), dtype=torch.float32, device=DEV)
    rvq.rvq_gemv(packed, cbp, rows, cols, x, n, y, ws)
    return y


def test_noalloc_matches_workspace_gemv_on_two_calls():
    cases = [(256, 512, 1, "f32", 0), (2048, 7168, 3, "bf16", 1)]
    for rows, cols, n, dt, seed in cases:          # two calls in a row, different shapes
        packed, cbp = _matrix(rows, cols, seed)
        xf = synth.normal_f32(1234 + seed, n * cols).reshape(n, cols)
        if dt == "bf16":
            bits = synth.f32_to_bf16(xf)
            x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
        else:
            x = torch.from_numpy(xf).to(DEV)
        y_ref = _with_workspace(packed, cbp, rows, cols, x, n)
        y = torch.full((n, rows), float("nan"), dtype=torch.float32, device=DEV)
        rvq.rvq_gemv_noalloc(packed, cbp, rows, cols, x, n, y)
        # the call's device status, read from the fixed array (waits for the stream)
        assert rvq.rvq_gemv_noalloc_status() == (0, 0)
        assert_rms_close(y.cpu().numpy(), y_ref.cpu().numpy(), 1e-4, f"noalloc {rows}x{cols}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    rows, cols, n = 7168, 2048, 1024
    assert rvq.rvq_gemv_workspace_bytes(rows, cols, n) > rvq.RVQ_NOALLOC_SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.float32, device=DEV)
    with pytest.raises(rvq.RvqError) as ei:
        rvq.rvq_gemv_noalloc(dummy, dummy, rows, cols, dummy, n, dummy)
    assert ei.value.status == "RVQ_ENOMEM"
    assert "scratch" in str(ei.value)


def test_noalloc_rejects_bad_arguments_before_launching():
    """Argument checks run before the status block is cleared or anything is
    queued: a rejected call leaves the last call's output untouched."""
    rows, cols, n = 256, 512, 1
    packed, cbp = _matrix(rows, cols, 3)
    x = torch.from_numpy(synth.normal_f32(77, n * cols).reshape(n, cols)).to(DEV)
    y = torch.empty((n, rows), dtype=torch.float32, device=DEV)
    rvq.rvq_gemv_noalloc(packed, cbp, rows, cols, x, n, y)
    torch.cuda.synchronize()
    before = y.clone()
    xbad = torch.empty(n * cols + 4, dtype=torch.float32, device=DEV)[1:1 + n * cols].view(n, cols)
    with pytest.raises(rvq.RvqError) as ei:
        rvq.rvq_gemv_noalloc(packed, cbp, rows, cols, xbad, n, y)
    assert ei.value.status == "RVQ_EALIGN"
    with pytest.raises(rvq.RvqError) as ei:
        rvq.rvq_gemv_noalloc(packed, cbp, rows + 1, cols, x, n, y)
    assert ei.value.status == "RVQ_EINVAL"
    torch.cuda.synchronize()
    assert torch.equal(y, before)
    assert rvq.rvq_gemv_noalloc_status() == (0, 0)
