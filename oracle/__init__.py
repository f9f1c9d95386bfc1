"""CPU oracle for the RVQ MoE expert FFN -- TEST INFRASTRUCTURE.

Only the test suite, the package smoke check and the benchmark's CPU-baseline
and reference legs may import this package.  The product (the CUDA library and
its binding) never loads it, and it never loads the product.

Thin numpy wrappers around ``rvq_oracle.c`` (plain C, double precision).
Parity unpinned: none -- every function here is pinned by ``tests/`` against
closed forms, invariants, brute force and library routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rvq_oracle.c")
_HDR = os.path.join(_HERE, "rvq_oracle.h")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, strict IEEE: no -ffast-math)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i32 = ctypes.c_void_p, ctypes.c_int32
            sig = {
                "oracle_rvq_dequant": (None, [vp, vp, i32, i32, vp]),
                "oracle_rvq_gemv": (None, [vp, vp, i32, i32, vp, i32, vp]),
                "oracle_rvq_lut_build": (None, [vp, vp, i32, vp]),
                "oracle_rvq_lut_gemv": (None, [vp, vp, i32, i32, vp]),
                "oracle_router_logits": (None, [vp, vp, vp, i32, i32, i32, vp]),
                "oracle_route": (i32, [vp, i32, i32, i32, vp, vp]),
                "oracle_group": (None, [vp, i32, i32, i32, vp, vp]),
                "oracle_swiglu": (ctypes.c_double, [ctypes.c_double, ctypes.c_double]),
                "oracle_expert_ffn": (None, [vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, vp]),
                "oracle_combine": (None, [vp, vp, i32, i32, i32, vp, vp]),
                "oracle_rms_norm": (None, [vp, i32, i32, ctypes.c_double, vp]),
                "oracle_moe_layer": (i32, [vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                           vp, vp, vp, vp, vp, vp, vp]),
                "oracle_crc32": (ctypes.c_uint32, [vp, ctypes.c_size_t]),
                "oracle_rvq_encode": (None, [vp, i32, i32, i32, vp, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data


def _check_codes(codes, rows, cols):
    assert cols % 8 == 0
    assert codes.dtype == np.uint8 and codes.size == rows * (cols // 8) * 3


def rvq_dequant(codes, cb, rows, cols):
    codes, cb = _c(codes, np.uint8), _c(cb, np.float32)
    _check_codes(codes, rows, cols)
    w = np.empty((rows, cols), np.float64)
    _load().oracle_rvq_dequant(_p(codes), _p(cb), rows, cols, _p(w))
    return w


def rvq_gemv(codes, cb, rows, cols, x):
    """y[n][rows] = W x for x [n][cols] (W = explicit RVQ decode)."""
    codes, cb = _c(codes, np.uint8), _c(cb, np.float32)
    _check_codes(codes, rows, cols)
    x = _c(np.atleast_2d(x), np.float64)
    assert x.shape[1] == cols
    y = np.empty((x.shape[0], rows), np.float64)
    _load().oracle_rvq_gemv(_p(codes), _p(cb), rows, cols, _p(x), x.shape[0], _p(y))
    return y


def rvq_lut_build(cb, x, cols):
    cb, x = _c(cb, np.float32), _c(x, np.float64)
    assert x.size == cols
    lut = np.empty((cols // 8, 3, 256), np.float64)
    _load().oracle_rvq_lut_build(_p(cb), _p(x), cols, _p(lut))
    return lut


def rvq_lut_gemv(codes, lut, rows, cols):
    codes, lut = _c(codes, np.uint8), _c(lut, np.float64)
    _check_codes(codes, rows, cols)
    y = np.empty(rows, np.float64)
    _load().oracle_rvq_lut_gemv(_p(codes), _p(lut), rows, cols, _p(y))
    return y


def router_logits(wr, x, bias=None):
    wr = _c(wr, np.float32)
    E, d = wr.shape
    x = _c(np.atleast_2d(x), np.float64)
    n = x.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((n, E), np.float64)
    _load().oracle_router_logits(_p(wr), _p(b), _p(x), n, E, d, _p(out))
    return out


def route(logits_f32, k):
    lg = _c(logits_f32, np.float32)
    n, E = lg.shape
    idx = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float32)
    rc = _load().oracle_route(_p(lg), n, E, k, _p(idx), _p(w))
    return idx, w, int(rc)


def group(topk_idx, E):
    idx = _c(topk_idx, np.int32)
    n, k = idx.shape
    offsets = np.empty(E + 1, np.int32)
    pairs = np.empty(n * k, np.int32)
    _load().oracle_group(_p(idx), n, E, k, _p(offsets), _p(pairs))
    return offsets, pairs


def swiglu(g, u):
    return float(_load().oracle_swiglu(float(g), float(u)))


def expert_ffn(gate, up, down, d, f, x, want_h=False):
    """gate/up/down: (codes, codebooks) tuples.  x: [d] float64."""
    gc, gb = _c(gate[0], np.uint8), _c(gate[1], np.float32)
    uc, ub = _c(up[0], np.uint8), _c(up[1], np.float32)
    dc, db = _c(down[0], np.uint8), _c(down[1], np.float32)
    _check_codes(gc, f, d)
    _check_codes(uc, f, d)
    _check_codes(dc, d, f)
    x = _c(x, np.float64).reshape(-1)
    assert x.size == d
    y = np.empty(d, np.float64)
    h = np.empty(f, np.float64) if want_h else None
    _load().oracle_expert_ffn(_p(gc), _p(gb), _p(uc), _p(ub), _p(dc), _p(db), d, f,
                              _p(x), _p(y), _p(h))
    return (y, h) if want_h else y


def combine(y_pair, topk_w, residual):
    w = _c(topk_w, np.float32)
    n, k = w.shape
    res = _c(residual, np.float64)
    d = res.shape[1]
    y = _c(y_pair, np.float64).reshape(n * k, d)
    out = np.empty((n, d), np.float64)
    _load().oracle_combine(_p(y), _p(w), n, k, d, _p(res), _p(out))
    return out


def rms_norm(x, eps=1e-6):
    """Row-wise x / sqrt(mean(x^2) + eps), float64 [n][d] (stack pre-norm)."""
    xx = _c(np.atleast_2d(x), np.float64)
    n, d = xx.shape
    out = np.empty((n, d), np.float64)
    _load().oracle_rms_norm(_p(xx), n, d, float(eps), _p(out))
    return out


def moe_layer(experts, wr, x, k, d, f, bias=None, route_logits=None):
    """One MoE layer.  experts: callable e -> ((gc, gb), (uc, ub), (dc, db)),
    evaluated only for experts the routing selects.  x: [n][d] float64.
    Returns dict(logits, idx, w, y_pair, out, rc)."""
    wr = _c(wr, np.float32)
    E = wr.shape[0]
    x = _c(np.atleast_2d(x), np.float64)
    n = x.shape[0]
    # routing first, so that only the selected experts are materialised
    lg = router_logits(wr, x, bias)
    used = (_c(route_logits, np.float32) if route_logits is not None
            else lg.astype(np.float32))
    idx, _, _ = route(used, k)
    sel = sorted(set(int(e) for e in idx.reshape(-1)))
    keep = []
    code_ptrs = (ctypes.c_void_p * (3 * E))()
    cb_ptrs = (ctypes.c_void_p * (3 * E))()
    for e in sel:
        mats = experts(e)
        for m, (c, b) in enumerate(mats):
            c, b = _c(c, np.uint8), _c(b, np.float32)
            keep += [c, b]
            code_ptrs[3 * e + m] = c.ctypes.data
            cb_ptrs[3 * e + m] = b.ctypes.data
    b = None if bias is None else _c(bias, np.float32)
    logits_used = np.empty((n, E), np.float32)
    topk_idx = np.empty((n, k), np.int32)
    topk_w = np.empty((n, k), np.float32)
    y_pair = np.empty((n * k, d), np.float64)
    out = np.empty((n, d), np.float64)
    rc = _load().oracle_moe_layer(ctypes.addressof(code_ptrs), ctypes.addressof(cb_ptrs),
                                  _p(wr), _p(b), n, E, k, d, f, _p(x), _p(used),
                                  _p(logits_used), _p(topk_idx), _p(topk_w),
                                  _p(y_pair), _p(out))
    del keep
    return dict(logits=lg, logits_used=logits_used, idx=topk_idx, w=topk_w,
                y_pair=y_pair, out=out, rc=int(rc))


def crc32(data) -> int:
    """CRC-32 (ISO-HDLC: reflected 0xEDB88320, preset and final complement)
    of a byte buffer, one bit per step."""
    b = np.ascontiguousarray(np.frombuffer(bytes(data), np.uint8) if isinstance(data, (bytes, bytearray))
                             else np.asarray(data, dtype=np.uint8).reshape(-1))
    return int(_load().oracle_crc32(b.ctypes.data if b.size else None, b.size))


def rvq_encode(w, iters):
    """Residual k-means encoder (3 stages x 256 codewords of 8 dimensions).
    w: fp32 [rows][cols]; returns (codes uint8 [rows][cols/8][3], codebooks
    fp32 [3][256][8])."""
    w = _c(w, np.float32)
    rows, cols = w.shape
    assert cols % 8 == 0 and rows * cols // 8 >= 256
    codes = np.empty((rows, cols // 8, 3), np.uint8)
    cb = np.empty((3, 256, 8), np.float32)
    _load().oracle_rvq_encode(_p(w), rows, cols, int(iters), _p(codes), _p(cb))
    return codes, cb
