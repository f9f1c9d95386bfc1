"""Owning wrapper around one MoE layer's device buffers (expert bank, router,
outputs, workspace).  Marshalling only: every step runs in librvqmoe."""
from __future__ import annotations

import numpy as np
import torch

from . import (RVQ_WS_STATUS_BYTES, moe_bank_init, moe_bank_record_bytes, moe_bank_validate,
               moe_bank_write_expert, moe_cache_bank, moe_cache_create, moe_cache_destroy,
               moe_cache_stats, moe_combine, moe_expert_ffn, moe_layer_forward,
               moe_layer_forward_host, moe_layer_forward_prenorm, moe_layer_forward_streamed,
               moe_layer_graph_create,
               moe_rms_norm, moe_route,
               moe_router_logits,
               moe_workspace_bytes, rvq_ws_clear, rvq_ws_status)


def _dev(a, device, dtype=None):
    if isinstance(a, torch.Tensor):
        return a.to(device=device, dtype=dtype or a.dtype).contiguous()
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device=device, dtype=dtype or t.dtype)


class MoeLayer:
    """Expert bank of `n_experts` RVQ experts (d hidden, f intermediate) plus a
    linear router; top-k routing."""

    def __init__(self, n_experts: int, d: int, f: int, k: int, layer: int = 0,
                 device: str | torch.device = "cuda"):
        self.E, self.d, self.f, self.k, self.layer = n_experts, d, f, k, layer
        self.device = torch.device(device)
        rb = moe_bank_record_bytes(d, f)
        if rb == 0:
            raise ValueError(f"d={d}, f={f} must be multiples of 512")
        self.record_bytes = rb
        self.buf = torch.empty(rb * n_experts, dtype=torch.uint8, device=self.device)
        assert self.buf.data_ptr() % 256 == 0
        self.bank = moe_bank_init(self.buf, n_experts, d, f, layer)
        self.wr = None
        self.bias = None
        self._ws = {}

    # ---------------------------------------------------------------- loading
    def load_expert(self, e: int, gate_codes, up_codes, down_codes, codebooks):
        """Canonical codes uint8 [f][d/8][3], [f][d/8][3], [d][f/8][3] and
        codebooks fp32 [3 matrices][3][256][8] (numpy or tensors)."""
        dev = self.device
        g = _dev(gate_codes, dev, torch.uint8)
        u = _dev(up_codes, dev, torch.uint8)
        dn = _dev(down_codes, dev, torch.uint8)
        cb = _dev(codebooks, dev, torch.float32)
        assert g.numel() == self.f * self.d * 3 // 8 and dn.numel() == self.d * self.f * 3 // 8
        assert cb.numel() == 3 * 3 * 256 * 8
        moe_bank_write_expert(self.bank, e, g, u, dn, cb)

    def set_router(self, wr, bias=None):
        self.wr = _dev(wr, self.device, torch.float32)
        assert self.wr.shape == (self.E, self.d)
        self.bias = None if bias is None else _dev(bias, self.device, torch.float32)

    def validate(self):
        moe_bank_validate(self.bank)

    def record(self, e: int) -> torch.Tensor:
        return self.buf[e * self.record_bytes:(e + 1) * self.record_bytes]

    # ----------------------------------------------------------------- buffers
    def workspace(self, n: int) -> torch.Tensor:
        ws = self._ws.get(n)
        if ws is None:
            nbytes = moe_workspace_bytes(self.bank, n, self.k)
            ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            rvq_ws_clear(ws)
            self._ws[n] = ws
        return ws

    def buffers(self, n: int) -> dict:
        dev, E, k = self.device, self.E, self.k
        return dict(
            logits=torch.empty((n, E), dtype=torch.float32, device=dev),
            idx=torch.empty((n, k), dtype=torch.int32, device=dev),
            w=torch.empty((n, k), dtype=torch.float32, device=dev),
            offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
            pairs=torch.empty(n * k, dtype=torch.int32, device=dev),
            out=torch.empty((n, self.d), dtype=torch.float32, device=dev),
            ws=self.workspace(n))

    # ----------------------------------------------------------------- compute
    def forward(self, x: torch.Tensor, bufs: dict | None = None, events=None,
                tc_min_tokens: int = 0, residual: torch.Tensor | None = None) -> dict:
        """Whole layer: out = residual + sum_slot w * expert(x) (residual
        defaults to x).  Experts with at least tc_min_tokens tokens use the
        tensor-core path (0: none)."""
        n = x.shape[0]
        b = bufs or self.buffers(n)
        moe_layer_forward(self.bank, self.wr, self.bias, x, n, self.k, b["logits"], b["idx"],
                          b["w"], b["offsets"], b["pairs"], b["out"], b["ws"], events=events,
                          tc_min_tokens=tc_min_tokens, residual=residual)
        return b

    def forward_host(self, x_host: torch.Tensor, out_host: torch.Tensor, bufs: dict | None = None,
                     tc_min_tokens: int = 0) -> dict:
        """The layer with its input read from and its output written to host
        tensors (pinned for asynchronous copies), through the library's
        host-buffer call; asynchronous on the current stream."""
        n = x_host.shape[0]
        b = bufs or self.buffers(n)
        xd = b.get("x_dev")
        if xd is None or xd.dtype != x_host.dtype or xd.shape != (n, self.d):
            xd = b["x_dev"] = torch.empty((n, self.d), dtype=x_host.dtype, device=self.device)
        moe_layer_forward_host(self.bank, self.wr, self.bias, x_host, n, self.k, xd, b["logits"],
                               b["idx"], b["w"], b["offsets"], b["pairs"], b["out"], out_host,
                               b["ws"], tc_min_tokens=tc_min_tokens)
        return b

    def graph(self, x_dev: torch.Tensor, bufs: dict, x_host: torch.Tensor | None = None,
              out_host: torch.Tensor | None = None, tc_min_tokens: int = 0):
        """A CUDA graph of this layer on x_dev and bufs (optionally with the
        copy of x_host into x_dev before it and of the output to out_host
        after it), recorded on a side stream; launch() runs it on the current
        stream."""
        side = torch.cuda.Stream(device=self.device)
        side.wait_stream(torch.cuda.current_stream())
        g = moe_layer_graph_create(self.bank, self.wr, self.bias, x_dev.shape[0], self.k, x_dev,
                                   bufs["logits"], bufs["idx"], bufs["w"], bufs["offsets"],
                                   bufs["pairs"], bufs["out"], bufs["ws"],
                                   tc_min_tokens=tc_min_tokens, x_host=x_host, out_host=out_host,
                                   stream=side)
        torch.cuda.current_stream().wait_stream(side)
        return g

    def forward_steps(self, x: torch.Tensor) -> dict:
        """Same layer through the separate calls (router, route, FFN, combine)."""
        n = x.shape[0]
        b = self.buffers(n)
        moe_router_logits(self.wr, self.bias, x, n, self.E, self.d, b["logits"])
        moe_route(b["logits"], n, self.E, self.k, b["idx"], b["w"], b["offsets"], b["pairs"],
                  b["ws"])
        y = torch.empty((n * self.k, self.d), dtype=torch.float32, device=self.device)
        moe_expert_ffn(self.bank, x, n, self.k, b["offsets"], b["pairs"], y, b["ws"])
        moe_combine(y, b["w"], n, self.k, self.d, x, b["out"])
        b["y_pair"] = y
        return b

    def status(self, n: int) -> tuple[int, int]:
        return rvq_ws_status(self.workspace(n))


class MoeStack:
    """Layers applied in order to a residual stream h (the first layer's
    input, then each layer's fp32 output): layer i computes
    out = h + sum_slot w * expert(rms_norm(h)), the normalised stream in
    bf16.  Each layer keeps its own buffers (its "xn" holds the normalised
    input), so the stream is never copied."""

    def __init__(self, layers: list[MoeLayer], eps: float = 1e-6):
        assert layers and all(L.d == layers[0].d for L in layers)
        self.layers = layers
        self.eps = eps
        self._bufs = {}

    def buffers(self, n: int) -> list[dict]:
        b = self._bufs.get(n)
        if b is None:
            # the layers run one after another on one stream, so they share
            # one workspace (24 GB per K3-shaped layer at 2048 tokens)
            ws = self.layers[0].workspace(n)
            for L in self.layers[1:]:
                if moe_workspace_bytes(L.bank, n, L.k) <= ws.numel():
                    L._ws[n] = ws
            b = [L.buffers(n) for L in self.layers]
            for L, bl in zip(self.layers, b):
                bl["xn"] = torch.empty((n, L.d), dtype=torch.bfloat16, device=L.device)
            self._bufs[n] = b
        return b

    def forward(self, x: torch.Tensor, events=None, tc_min_tokens: int = 0) -> list[dict]:
        """Runs every layer; returns the per-layer buffers (the last one's
        "out" is the stack output).  `events`, if given, are layer 0's."""
        n = x.shape[0]
        bufs = self.buffers(n)
        h = x
        for i, L in enumerate(self.layers):
            b = bufs[i]
            if events is not None and i == 0:
                # per-kernel timing marks: the norm and the layer as separate calls
                moe_rms_norm(h, n, L.d, b["xn"], eps=self.eps)
                L.forward(b["xn"], b, events=events, tc_min_tokens=tc_min_tokens, residual=h)
            else:
                moe_layer_forward_prenorm(L.bank, L.wr, L.bias, h, n, L.k, self.eps, b["xn"],
                                          b["logits"], b["idx"], b["w"], b["offsets"], b["pairs"],
                                          b["out"], b["ws"], tc_min_tokens=tc_min_tokens)
            h = b["out"]
        return bufs


class MoeStreamedStack:
    """The same stack with its expert records in pinned host memory and an HBM
    cache of `slots` records (moe_layer_forward_streamed per layer): the
    pages' streaming engine with host memory in place of NVMe.  The layers'
    device banks are copied into one host bank and released.  With
    lookahead > 0 each layer prefetches the next layer's predicted experts."""

    def __init__(self, layers: list[MoeLayer], slots: int, lookahead: int = 0,
                 eps: float = 1e-6):
        assert layers and all(L.d == layers[0].d and L.f == layers[0].f and L.E == layers[0].E
                              for L in layers)
        L0 = layers[0]
        self.n_layers, self.E, self.d, self.f, self.k = len(layers), L0.E, L0.d, L0.f, L0.k
        self.device = L0.device
        self.eps, self.lookahead = eps, lookahead
        rb = L0.record_bytes
        self.host = torch.empty(self.n_layers * self.E * rb, dtype=torch.uint8, pin_memory=True)
        for i, L in enumerate(layers):
            self.host[i * self.E * rb:(i + 1) * self.E * rb].copy_(L.buf)
            L.buf = None  # the device bank is no longer needed
        torch.cuda.synchronize()
        self.wr = [L.wr for L in layers]
        self.bias = [L.bias for L in layers]
        self.slots = torch.empty(slots * rb, dtype=torch.uint8, device=self.device)
        self.slot_map = torch.full((self.n_layers, self.E), -1, dtype=torch.int32,
                                   device=self.device)
        self.cache = moe_cache_create(self.host, self.n_layers, self.E, self.d, self.f,
                                      self.slots, self.slot_map)
        self._bufs = {}

    def buffers(self, n: int) -> list[dict]:
        b = self._bufs.get(n)
        if b is None:
            dev, E, k = self.device, self.E, self.k
            ws = torch.empty(moe_workspace_bytes(moe_cache_bank(self.cache, 0), n, k),
                             dtype=torch.uint8, device=dev)
            rvq_ws_clear(ws)
            b = [dict(logits=torch.empty((n, E), dtype=torch.float32, device=dev),
                      idx=torch.empty((n, k), dtype=torch.int32, device=dev),
                      w=torch.empty((n, k), dtype=torch.float32, device=dev),
                      offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                      pairs=torch.empty(n * k, dtype=torch.int32, device=dev),
                      out=torch.empty((n, self.d), dtype=torch.float32, device=dev),
                      xn=torch.empty((n, self.d), dtype=torch.bfloat16, device=dev),
                      next_logits=torch.empty((n, E), dtype=torch.float32, device=dev),
                      ws=ws) for _ in range(self.n_layers)]
            self._bufs[n] = b
        return b

    def forward(self, x: torch.Tensor, tc_min_tokens: int = 0) -> list[dict]:
        n = x.shape[0]
        bufs = self.buffers(n)
        h = x
        for i in range(self.n_layers):
            bi = bufs[i]
            moe_rms_norm(h, n, self.d, bi["xn"], eps=self.eps)
            nxt = i + 1 < self.n_layers and self.lookahead > 0
            moe_layer_forward_streamed(
                self.cache, i, self.wr[i], self.bias[i], bi["xn"], n, self.k, bi["logits"],
                bi["idx"], bi["w"], bi["offsets"], bi["pairs"], bi["out"], bi["ws"],
                residual=h, tc_min_tokens=tc_min_tokens,
                next_wr=self.wr[i + 1] if nxt else None,
                next_bias=self.bias[i + 1] if nxt else None,
                lookahead=self.lookahead if nxt else 0,
                next_logits=bi["next_logits"] if nxt else None)
            h = bi["out"]
        return bufs

    def stats(self) -> dict:
        return moe_cache_stats(self.cache)

    def status(self, n: int) -> tuple[int, int]:
        return rvq_ws_status(self.buffers(n)[0]["ws"])

    def close(self):
        if self.cache:
            torch.cuda.synchronize()
            moe_cache_destroy(self.cache)
            self.cache = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


__all__ = ["MoeLayer", "MoeStack", "MoeStreamedStack", "RVQ_WS_STATUS_BYTES"]
