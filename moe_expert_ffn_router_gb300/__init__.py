"""Python binding of librvqmoe (RVQ MoE expert FFN for GB300, sm_103a).

Argument marshalling only: every step runs in the library's CUDA kernels.
Functions carry the C names of include/rvqmoe.h and take torch tensors (device
memory) plus the current CUDA stream.  Importing fails loudly when the
compiled library is missing; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librvqmoe.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "rvqmoe.h")

RVQ_F32, RVQ_BF16 = 0, 1
RVQ_WS_STATUS_BYTES = 256
RVQ_CODEBOOK_BYTES = 24576
RVQ_BANK_MAGIC = 0x31515652
RVQ_HDR_FLAG_CRC32 = 0x1
MOE_LAYER_EVENTS = 8
RVQMOE_PREFILL_MIN_TOKENS = 6
DEV_ERR_INDEX, DEV_ERR_NONFINITE, DEV_ERR_CORRUPT, DEV_ERR_TIMEOUT = 1, 2, 4, 8
STATUS = {0: "RVQ_OK", 1: "RVQ_EINVAL", 2: "RVQ_EALIGN", 3: "RVQ_ENOMEM", 4: "RVQ_ECORRUPT",
          5: "RVQ_EDEVICE", 6: "RVQ_ETIMEOUT", 7: "RVQ_ECUDA", 8: "RVQ_ENOTIMPL"}


class RvqError(RuntimeError):
    def __init__(self, name, code, msg):
        super().__init__(f"{name}: {STATUS.get(code, code)}: {msg}")
        self.code = code
        self.status = STATUS.get(code, str(code))


class RvqMoeBank(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("record_bytes", ctypes.c_uint64),
                ("n_experts", ctypes.c_int32), ("d", ctypes.c_int32),
                ("f", ctypes.c_int32), ("layer", ctypes.c_int32)]


class RvqCacheStats(ctypes.Structure):
    _fields_ = [("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64),
                ("prefetched", ctypes.c_uint64), ("prefetch_used", ctypes.c_uint64),
                ("bytes_copied", ctypes.c_uint64), ("slots", ctypes.c_int32),
                ("pad", ctypes.c_int32)]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; "
                      "g.build()'` (nvcc, sm_103a)")

_vp, _i32, _u32, _u64, _sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32,
                              ctypes.c_uint64, ctypes.c_size_t)
_lib = ctypes.CDLL(LIB_PATH)
_BANKP = ctypes.POINTER(RvqMoeBank)
_SIGS = {
    "rvq_status_string": (ctypes.c_char_p, [_i32]),
    "rvq_last_error": (ctypes.c_char_p, []),
    "rvq_version": (_u32, []),
    "rvq_code_bytes": (_sz, [_i32, _i32]),
    "rvq_pack": (_i32, [_vp, _i32, _i32, _vp, _sz, _vp]),
    "rvq_unpack": (_i32, [_vp, _i32, _i32, _vp, _sz, _vp]),
    "rvq_pack_codebooks": (_i32, [_vp, _vp, _vp]),
    "rvq_lut_build": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp]),
    "rvq_gemv_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "rvq_gemv": (_i32, [_vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _vp, _sz, _vp]),
    "rvq_gemv_noalloc": (_i32, [_vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _vp]),
    "rvq_gemv_noalloc_status": (_i32, [ctypes.POINTER(_u32), _vp]),
    "moe_bank_record_bytes": (_u64, [_i32, _i32]),
    "moe_bank_init": (_i32, [_BANKP, _vp, _u64, _i32, _i32, _i32, _i32]),
    "moe_bank_write_expert": (_i32, [_BANKP, _i32, _vp, _vp, _vp, _vp, _vp]),
    "moe_bank_validate": (_i32, [_BANKP, _vp]),
    "moe_bank_seal": (_i32, [_BANKP, _vp]),
    "rvq_encode_workspace_bytes": (_sz, [_i32, _i32]),
    "rvq_encode": (_i32, [_vp, _i32, _i32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "moe_cache_create": (_i32, [ctypes.POINTER(_vp), _vp, _i32, _i32, _i32, _i32, _vp, _u64,
                                _vp]),
    "moe_cache_destroy": (_i32, [_vp]),
    "moe_cache_stats": (_i32, [_vp, ctypes.POINTER(RvqCacheStats)]),
    "moe_cache_bank": (_i32, [_vp, _i32, _BANKP]),
    "moe_layer_forward_streamed": (_i32, [_vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp,
                                          _vp, _vp, _vp, _vp, _vp, _sz, _vp, _i32, _i32, _vp,
                                          _vp, _i32, _vp, _vp]),
    "moe_bank_verify": (_i32, [_BANKP, _vp, _vp, _sz, _vp]),
    "moe_router_logits": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp]),
    "moe_route_max_tokens": (_i32, [_i32]),
    "moe_route": (_i32, [_vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_workspace_bytes": (_sz, [_BANKP, _i32, _i32]),
    "moe_expert_ffn": (_i32, [_BANKP, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_expert_ffn_ex": (_i32, [_BANKP, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _sz, _i32,
                                 _vp]),
    "moe_combine": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _i32, _vp, _vp]),
    "moe_layer_forward": (_i32, [_BANKP, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp,
                                 _vp, _vp, _vp, _sz, _vp, _vp]),
    "moe_layer_forward_ex": (_i32, [_BANKP, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp,
                                    _vp, _vp, _vp, _vp, _sz, _vp, _i32, _i32, _vp, _vp]),
    "moe_layer_forward_host": (_i32, [_BANKP, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp,
                                      _vp, _vp, _vp, _vp, _vp, _sz, _i32, _vp]),
    "moe_layer_graph_create": (_i32, [_BANKP, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp,
                                      _vp, _vp, _vp, _vp, _vp, _sz, _i32, _vp,
                                      ctypes.POINTER(ctypes.c_void_p)]),
    "moe_layer_graph_launch": (_i32, [_vp, _vp]),
    "moe_layer_graph_destroy": (_i32, [_vp]),
    "moe_layer_forward_prenorm": (_i32, [_BANKP, _vp, _vp, _vp, _i32, _i32, _i32, ctypes.c_float,
                                         _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i32, _vp]),
    "moe_rms_norm": (_i32, [_vp, _i32, _i32, _i32, ctypes.c_float, _vp, _i32, _vp]),
    "rvq_selftest_prefill_timeout": (_i32, [_BANKP, _vp, _sz, _vp]),
    "rvq_ws_clear": (_i32, [_vp, _vp]),
    "rvq_ws_status": (_i32, [_vp, ctypes.POINTER(_u32), _vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def header_functions() -> list[str]:
    """Names of every function declared in include/rvqmoe.h."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(\w+)\s*\([^;{]*\)\s*;", txt)) - {"if", "while"})


def lib_has(name: str) -> bool:
    return hasattr(_lib, name)


# ------------------------------------------------------------------ helpers

def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dt(t) -> int:
    if t.dtype == torch.bfloat16:
        return RVQ_BF16
    if t.dtype == torch.float32:
        return RVQ_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _check(name, rc):
    if rc != 0:
        raise RvqError(name, rc, last_error())


def status_string(code: int) -> str:
    return _lib.rvq_status_string(code).decode()


def last_error() -> str:
    return _lib.rvq_last_error().decode()


def rvq_version() -> int:
    return int(_lib.rvq_version())


# ------------------------------------------------------------------ RVQ calls

def rvq_code_bytes(rows: int, cols: int) -> int:
    return int(_lib.rvq_code_bytes(rows, cols))


def rvq_pack(codes, rows, cols, packed, stream=None):
    _check("rvq_pack", _lib.rvq_pack(_p(codes), rows, cols, _p(packed), _nbytes(packed),
                                     _stream(stream)))


def rvq_unpack(packed, rows, cols, codes, stream=None):
    _check("rvq_unpack", _lib.rvq_unpack(_p(packed), rows, cols, _p(codes), _nbytes(codes),
                                         _stream(stream)))


def rvq_pack_codebooks(cb, cb_packed, stream=None):
    _check("rvq_pack_codebooks", _lib.rvq_pack_codebooks(_p(cb), _p(cb_packed), _stream(stream)))


def rvq_lut_build(codebooks, x, n, cols, lut, stream=None):
    _check("rvq_lut_build", _lib.rvq_lut_build(_p(codebooks), _p(x), _dt(x), n, cols, _p(lut),
                                               _stream(stream)))


def rvq_gemv_workspace_bytes(rows, cols, n) -> int:
    return int(_lib.rvq_gemv_workspace_bytes(rows, cols, n))


def rvq_gemv(packed_codes, packed_cb, rows, cols, x, n, y, ws, stream=None):
    _check("rvq_gemv", _lib.rvq_gemv(_p(packed_codes), _p(packed_cb), rows, cols, _p(x), _dt(x),
                                     n, _p(y), _p(ws), _nbytes(ws), _stream(stream)))


RVQ_NOALLOC_SCRATCH_BYTES = 4 << 20


def rvq_gemv_noalloc(packed_codes, packed_cb, rows, cols, x, n, y, stream=None):
    """rvq_gemv without a workspace, for callers that cannot allocate device
    memory: the scratch is a fixed 4 MiB array inside the library, shared by
    all calls (calls that overlap on the GPU race).  Make the first call on a
    device before any stream capture."""
    _check("rvq_gemv_noalloc",
           _lib.rvq_gemv_noalloc(_p(packed_codes), _p(packed_cb), rows, cols, _p(x), _dt(x), n,
                                 _p(y), _stream(stream)))


def rvq_gemv_noalloc_status(stream=None) -> tuple[int, int]:
    """Device status of the no-allocation GEMV's fixed array: (status code,
    raw bits) after the stream's work; clears the bits."""
    bits = _u32(0)
    rc = _lib.rvq_gemv_noalloc_status(ctypes.byref(bits), _stream(stream))
    return int(rc), int(bits.value)


# ------------------------------------------------------------------ bank

def moe_bank_record_bytes(d: int, f: int) -> int:
    return int(_lib.moe_bank_record_bytes(d, f))


def moe_bank_init(buffer, n_experts, d, f, layer=0) -> RvqMoeBank:
    bank = RvqMoeBank()
    _check("moe_bank_init", _lib.moe_bank_init(ctypes.byref(bank), _p(buffer), _nbytes(buffer),
                                               n_experts, d, f, layer))
    return bank


def moe_bank_write_expert(bank, expert, gate_codes, up_codes, down_codes, codebooks, stream=None):
    _check("moe_bank_write_expert",
           _lib.moe_bank_write_expert(ctypes.byref(bank), expert, _p(gate_codes), _p(up_codes),
                                      _p(down_codes), _p(codebooks), _stream(stream)))


def moe_bank_validate(bank, stream=None):
    _check("moe_bank_validate", _lib.moe_bank_validate(ctypes.byref(bank), _stream(stream)))


def moe_bank_seal(bank, stream=None):
    _check("moe_bank_seal", _lib.moe_bank_seal(ctypes.byref(bank), _stream(stream)))


def rvq_encode_workspace_bytes(rows, cols) -> int:
    return int(_lib.rvq_encode_workspace_bytes(rows, cols))


def rvq_encode(w, rows, cols, iters, codes, codebooks, ws, stream=None):
    _check("rvq_encode", _lib.rvq_encode(_p(w), rows, cols, iters, _p(codes), _p(codebooks),
                                         _p(ws), _nbytes(ws), _stream(stream)))


def moe_cache_create(host_bank, n_layers, n_experts, d, f, slots, slot_map) -> int:
    """host_bank: pinned uint8 tensor of n_layers x n_experts records; slots:
    device uint8 tensor; slot_map: device int32 [n_layers][n_experts].
    Returns the cache handle (an address)."""
    h = _vp()
    _check("moe_cache_create",
           _lib.moe_cache_create(ctypes.byref(h), _p(host_bank), n_layers, n_experts, d, f,
                                 _p(slots), _nbytes(slots), _p(slot_map)))
    return h.value


def moe_cache_destroy(cache):
    _check("moe_cache_destroy", _lib.moe_cache_destroy(cache))


def moe_cache_stats(cache) -> dict:
    st = RvqCacheStats()
    _check("moe_cache_stats", _lib.moe_cache_stats(cache, ctypes.byref(st)))
    return {k: int(getattr(st, k)) for k, _ in RvqCacheStats._fields_ if k != "pad"}


def moe_cache_bank(cache, layer) -> RvqMoeBank:
    bank = RvqMoeBank()
    _check("moe_cache_bank", _lib.moe_cache_bank(cache, layer, ctypes.byref(bank)))
    return bank


def moe_layer_forward_streamed(cache, layer, wr, bias, x, n, k, logits, topk_idx, topk_w,
                               offsets, pairs, out, ws, residual=None, tc_min_tokens=0,
                               next_wr=None, next_bias=None, lookahead=0, next_logits=None,
                               stream=None):
    rdt = _dt(residual) if residual is not None else _dt(x)
    _check("moe_layer_forward_streamed",
           _lib.moe_layer_forward_streamed(
               cache, layer, _p(wr), _p(bias), _p(x), _dt(x), n, k, _p(logits), _p(topk_idx),
               _p(topk_w), _p(offsets), _p(pairs), _p(out), _p(ws), _nbytes(ws), _p(residual),
               rdt, tc_min_tokens, _p(next_wr), _p(next_bias), lookahead, _p(next_logits),
               _stream(stream)))


def moe_bank_verify(bank, crc, ws, stream=None):
    _check("moe_bank_verify", _lib.moe_bank_verify(ctypes.byref(bank), _p(crc), _p(ws),
                                                   _nbytes(ws), _stream(stream)))


# ------------------------------------------------------------------ MoE calls

def moe_router_logits(wr, bias, x, n, E, d, logits, stream=None):
    _check("moe_router_logits",
           _lib.moe_router_logits(_p(wr), _p(bias), _p(x), _dt(x), n, E, d, _p(logits),
                                  _stream(stream)))


def moe_route_max_tokens(E: int) -> int:
    return int(_lib.moe_route_max_tokens(E))


def moe_route(logits, n, E, k, topk_idx, topk_w, offsets, pairs, ws, stream=None):
    _check("moe_route", _lib.moe_route(_p(logits), n, E, k, _p(topk_idx), _p(topk_w),
                                       _p(offsets), _p(pairs), _p(ws), _nbytes(ws),
                                       _stream(stream)))


def moe_workspace_bytes(bank, n, k) -> int:
    return int(_lib.moe_workspace_bytes(ctypes.byref(bank), n, k))


def moe_expert_ffn(bank, x, n, k, offsets, pairs, y_pair, ws, stream=None):
    _check("moe_expert_ffn",
           _lib.moe_expert_ffn(ctypes.byref(bank), _p(x), _dt(x), n, k, _p(offsets), _p(pairs),
                               _p(y_pair), _p(ws), _nbytes(ws), _stream(stream)))


def moe_expert_ffn_ex(bank, x, n, k, offsets, pairs, y_pair, ws, tc_min_tokens, stream=None):
    _check("moe_expert_ffn_ex",
           _lib.moe_expert_ffn_ex(ctypes.byref(bank), _p(x), _dt(x), n, k, _p(offsets), _p(pairs),
                                  _p(y_pair), _p(ws), _nbytes(ws), int(tc_min_tokens),
                                  _stream(stream)))


def moe_combine(y_pair, topk_w, n, k, d, residual, out, stream=None):
    _check("moe_combine", _lib.moe_combine(_p(y_pair), _p(topk_w), n, k, d, _p(residual),
                                           _dt(residual), _p(out), _stream(stream)))


def moe_layer_forward(bank, wr, bias, x, n, k, logits, topk_idx, topk_w, offsets, pairs, out,
                      ws, events=None, stream=None, tc_min_tokens=0, residual=None):
    ev = None
    if events is not None:
        assert len(events) == MOE_LAYER_EVENTS
        ev = (ctypes.c_void_p * MOE_LAYER_EVENTS)(*[e.cuda_event for e in events])
    rdt = _dt(residual) if residual is not None else _dt(x)
    _check("moe_layer_forward",
           _lib.moe_layer_forward_ex(ctypes.byref(bank), _p(wr), _p(bias), _p(x), _dt(x), n, k,
                                     _p(logits), _p(topk_idx), _p(topk_w), _p(offsets),
                                     _p(pairs), _p(out), _p(ws), _nbytes(ws), _p(residual), rdt,
                                     int(tc_min_tokens), ev, _stream(stream)))


def moe_layer_forward_host(bank, wr, bias, x_host, n, k, x_dev, logits, topk_idx, topk_w,
                           offsets, pairs, out, out_host, ws, tc_min_tokens=0, stream=None):
    """The layer with x read from and out written to host tensors (pinned for
    asynchronous copies); x_dev is the device copy of x.  Asynchronous."""
    assert not x_host.is_cuda and not out_host.is_cuda and x_host.dtype == x_dev.dtype
    assert x_host.is_contiguous() and out_host.is_contiguous()
    assert out_host.dtype == torch.float32 and out_host.numel() >= n * out.shape[-1]
    _check("moe_layer_forward_host",
           _lib.moe_layer_forward_host(ctypes.byref(bank), _p(wr), _p(bias),
                                       ctypes.c_void_p(x_host.data_ptr()), _dt(x_dev), n, k,
                                       _p(x_dev), _p(logits), _p(topk_idx), _p(topk_w),
                                       _p(offsets), _p(pairs), _p(out),
                                       ctypes.c_void_p(out_host.data_ptr()), _p(ws), _nbytes(ws),
                                       int(tc_min_tokens), _stream(stream)))


class LayerGraph:
    """A CUDA graph of one layer call (moe_layer_graph_create): launch() runs
    the whole layer as one graph launch; close() frees it.  Holds references
    to the buffers it records, so they outlive it."""

    def __init__(self, handle, keep):
        self._h = handle
        self._keep = keep

    def launch(self, stream=None):
        _check("moe_layer_graph_launch", _lib.moe_layer_graph_launch(self._h, _stream(stream)))

    def close(self):
        if self._h is not None:
            _check("moe_layer_graph_destroy", _lib.moe_layer_graph_destroy(self._h))
            self._h = None
            self._keep = None

    def __del__(self):
        if getattr(self, "_h", None) is not None and _lib is not None:
            _lib.moe_layer_graph_destroy(self._h)


def moe_layer_graph_create(bank, wr, bias, n, k, x_dev, logits, topk_idx, topk_w, offsets, pairs,
                           out, ws, tc_min_tokens=0, x_host=None, out_host=None, stream=None):
    """Records one layer call (optionally with the copies of x_host in and of
    out back to out_host) as a CUDA graph; stream must be capturable (not the
    legacy default stream).  Returns a LayerGraph."""
    if (x_host is None) != (out_host is None):
        raise ValueError("x_host and out_host go together")
    if x_host is not None:
        assert not x_host.is_cuda and not out_host.is_cuda and x_host.dtype == x_dev.dtype
        assert x_host.is_contiguous() and out_host.is_contiguous()
        assert out_host.dtype == torch.float32 and out_host.numel() >= n * out.shape[-1]
    h = ctypes.c_void_p()
    _check("moe_layer_graph_create",
           _lib.moe_layer_graph_create(
               ctypes.byref(bank), _p(wr), _p(bias),
               None if x_host is None else ctypes.c_void_p(x_host.data_ptr()), _dt(x_dev), n, k,
               _p(x_dev), _p(logits), _p(topk_idx), _p(topk_w), _p(offsets), _p(pairs), _p(out),
               None if out_host is None else ctypes.c_void_p(out_host.data_ptr()), _p(ws),
               _nbytes(ws), int(tc_min_tokens), _stream(stream), ctypes.byref(h)))
    return LayerGraph(h, (bank, wr, bias, x_dev, logits, topk_idx, topk_w, offsets, pairs, out,
                          ws, x_host, out_host))


def moe_layer_forward_prenorm(bank, wr, bias, h, n, k, eps, xn, logits, topk_idx, topk_w, offsets,
                              pairs, out, ws, tc_min_tokens=0, stream=None):
    """out = h + MoE(bf16 rms_norm(h)); xn (bf16 [n][d]) receives the normalised rows."""
    _check("moe_layer_forward_prenorm",
           _lib.moe_layer_forward_prenorm(ctypes.byref(bank), _p(wr), _p(bias), _p(h), _dt(h), n, k,
                                          float(eps), _p(xn), _p(logits), _p(topk_idx),
                                          _p(topk_w), _p(offsets), _p(pairs), _p(out), _p(ws),
                                          _nbytes(ws), int(tc_min_tokens), _stream(stream)))


def rvq_selftest_prefill_timeout(bank, ws, stream=None):
    _check("rvq_selftest_prefill_timeout",
           _lib.rvq_selftest_prefill_timeout(ctypes.byref(bank), _p(ws), _nbytes(ws),
                                             _stream(stream)))


def moe_rms_norm(x, n, d, out, eps=1e-6, stream=None):
    _check("moe_rms_norm", _lib.moe_rms_norm(_p(x), _dt(x), n, d, float(eps), _p(out), _dt(out),
                                             _stream(stream)))


def rvq_ws_clear(ws, stream=None):
    _check("rvq_ws_clear", _lib.rvq_ws_clear(_p(ws), _stream(stream)))


def rvq_ws_status(ws, stream=None) -> tuple[int, int]:
    """Returns (status code, raw device bits); clears the bits."""
    bits = _u32(0)
    rc = _lib.rvq_ws_status(_p(ws), ctypes.byref(bits), _stream(stream))
    return int(rc), int(bits.value)
