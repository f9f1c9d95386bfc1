"""GPU parity for the expert-record checksums (moe_bank_seal / moe_bank_verify):
the device CRC-32 of every record payload equals the oracle's bitwise CRC-32 of
the same bytes (bit-exact), and verification flags exactly the records whose
payload changed after sealing."""
import numpy as np
import pytest
import torch

import oracle
from tests.support import SynthLayer

pytestmark = pytest.mark.gpu
rvq = pytest.importorskip("moe_expert_ffn_router_gb300")
DEV = "cuda"


def _verify(L):
    crc = torch.zeros(L.E, dtype=torch.int32, device=DEV)
    ws = torch.zeros(rvq.RVQ_WS_STATUS_BYTES // 4, dtype=torch.int32, device=DEV)
    rvq.moe_bank_verify(L.bank, crc, ws)
    torch.cuda.synchronize()
    _, bits = rvq.rvq_ws_status(ws)
    return crc.cpu().numpy().view(np.uint32), bits


def _header(rec):
    return int(rec[24:28].view(np.uint32)[0]), int(rec[28:32].view(np.uint32)[0])


@pytest.mark.parametrize("config", [1, 2])
def test_seal_matches_oracle_and_verify_flags_changes(config):
    """config 1: 64 experts of 2.4 MB; config 2: 256 K3-shaped experts of
    16.5 MB (sampled records against the oracle)."""
    sl = SynthLayer(config, 0)
    L = sl.to_gpu()
    rb, E, buf = L.record_bytes, L.E, L.buf
    crc0, bits = _verify(L)  # unsealed: values reported, nothing flagged
    assert bits == 0
    rvq.moe_bank_seal(L.bank)
    crc, bits = _verify(L)
    assert bits == 0
    assert np.array_equal(crc, crc0)
    for e in sorted({0, 1, E // 2, E - 1}):
        rec = buf[e * rb:(e + 1) * rb].cpu().numpy()
        flags, hcrc = _header(rec)
        ref = oracle.crc32(rec[128:])
        assert flags & rvq.RVQ_HDR_FLAG_CRC32
        assert hcrc == ref == int(crc[e]), (e, hex(hcrc), hex(ref), hex(int(crc[e])))
    # one flipped bit in expert 5's payload (a code byte, and separately a
    # codebook byte) is seen, in that record only
    L.validate()
    for off in (rb - 4096, 128 + 17):
        pos = 5 * rb + off
        old = int(buf[pos].item())
        buf[pos] = old ^ 0x10
        crc2, bits = _verify(L)
        assert bits & rvq.DEV_ERR_CORRUPT
        assert int(crc2[5]) != int(crc[5])
        assert np.array_equal(np.delete(crc2, 5), np.delete(crc, 5))
        assert int(crc2[5]) == oracle.crc32(buf[5 * rb + 128:6 * rb].cpu().numpy())
        buf[pos] = old
        crc3, bits = _verify(L)
        assert bits == 0 and np.array_equal(crc3, crc)
    # a rewritten record is no longer sealed, so a change there is not flagged
    e = 3
    (gc, gb), (uc, ub), (dc, db) = ((sl.src.codes(e, m), sl.src.codebooks(e, m)) for m in range(3))
    L.load_expert(e, gc, uc, dc, np.stack([gb, ub, db]))
    flags, _ = _header(buf[e * rb:e * rb + 128].cpu().numpy())
    assert not flags & rvq.RVQ_HDR_FLAG_CRC32
    buf[e * rb + rb - 8] ^= 1
    _, bits = _verify(L)
    assert bits == 0
    del L, buf
    torch.cuda.empty_cache()
