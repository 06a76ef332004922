"""The weight-GEMV part of one decode (or speculative-verify) step of a
decoder stack: for every layer, ``kq_layer_step`` (q/k/v in one launch, o,
gate/up in one launch, down), then the LM head with ``kq_gemv``.

The Core AI card for Muse-Glimmer-30B (first table and the sentence under it)
shows decode streams every weight once per token; this object issues exactly
those launches in layer order on one stream, optionally captured into one
CUDA graph so the step costs a single graph launch.  Attention, norms and
activations are not part of it: every projection reads its own activation
buffer (``x``), and every output lands in its own buffer (``y``).
"""
from __future__ import annotations

import torch

from . import (kq_ffn_swiglu, kq_gemv, kq_gemv_multi, kq_layer, kq_layer_io, kq_layer_step,
               make_matrix)

LAYER_NAMES = ("q", "k", "v", "o", "gate", "up", "down")
# the matrices that read the pre-attention hidden state (the attention's
# sigmoid output gate is optional: the pages' own layer has it)
ATTN_NAMES = ("q", "k", "v", "attn_gate")
X_OF = {"q": "x_attn", "k": "x_attn", "v": "x_attn", "attn_gate": "x_attn", "o": "x_o",
        "gate": "x_ffn", "up": "x_ffn", "down": "x_down"}


class DecodeStep:
    """layers: list of {name: (fmt, W_device_uint8, N_out, K)} for the seven
    projections; lm_head: (fmt, W, N_out, K) or None.

    fused_ffn: the feed-forward block of every layer runs as kq_ffn_swiglu --
    the gate/up launch writes h = bf16(silu(gate) * up) (``self.h[l]``) and
    the down projection reads it -- instead of reading its own input
    ``x_down``."""

    def __init__(self, layers, lm_head, n_tok: int, device="cuda", fused_ffn=False):
        self.n_tok = n_tok
        self.layers = layers
        self.lm_head = lm_head
        self.fused_ffn = fused_ffn
        self.x, self.y = [], []
        self._structs = []
        # every activation input of the step is a view into one contiguous
        # bf16 buffer (x_all), so a caller fills all of them with one copy;
        # each view starts on a 16-byte boundary (K is a multiple of 256)
        widths = [L[n][3] for L in layers for n in ("q", "o", "gate", "down")]
        if lm_head is not None:
            widths.append(lm_head[3])
        self.x_all = torch.zeros(n_tok * sum(widths), dtype=torch.bfloat16, device=device)
        views, off = [], 0
        self._xoff = [0]   # x_all elements before layer l (the LM head's input last)
        for i, w in enumerate(widths):
            views.append(self.x_all[off:off + n_tok * w].view(n_tok, w))
            off += n_tok * w
            if i % 4 == 3 or i == len(widths) - 1:
                self._xoff.append(off)
        for li, L in enumerate(layers):
            xs = dict(zip(("x_attn", "x_o", "x_ffn", "x_down"), views[4 * li:4 * li + 4]))
            ys = {n: torch.empty((n_tok, L[n][2]), dtype=torch.float32, device=device)
                  for n in L}
            layer = kq_layer(*[make_matrix(L[n][0], L[n][1], L[n][2], L[n][3]) for n in LAYER_NAMES])
            io = kq_layer_io(*[xs[k].data_ptr() for k in ("x_attn", "x_o", "x_ffn", "x_down")],
                             *[ys[n].data_ptr() for n in LAYER_NAMES])
            self.x.append(xs)
            self.y.append(ys)
            self._structs.append((layer, io))
        self.h = [torch.empty((n_tok, L["gate"][2]), dtype=torch.bfloat16, device=device)
                  for L in layers] if fused_ffn else []
        if lm_head is not None:
            self.x_head = views[-1]
            self.y_head = torch.empty((n_tok, lm_head[2]), dtype=torch.float32, device=device)
        self.graph = None

    def weight_bytes(self) -> int:
        total = sum(L[n][1].numel() for L in self.layers for n in L)
        if self.lm_head is not None:
            total += self.lm_head[1].numel()
        return total

    def launches(self) -> int:
        """Kernel launches per step (one per format-group of a layer step;
        fused_ffn: plus the activation kernel where the gate/up launch does
        not fuse it, i.e. unless one token on Q4_K / Q4_G128 pairs of at
        least 2^25 weights)."""
        per_layer = 0
        for L in self.layers[:1]:
            for group in (ATTN_NAMES, ("o",), ("gate", "up"), ("down",)):
                per_layer += len({L[n][0] for n in group if n in L})
            if self.fused_ffn:
                f, _, N, K = L["gate"]
                if not (self.n_tok == 1 and f in (0, 3) and 2 * N * K >= (1 << 25)):
                    per_layer += 1
        return per_layer * len(self.layers) + (1 if self.lm_head is not None else 0)

    def run(self, stream=None, ready=None):
        """Issue the step's launches on `stream`.  ready: {layer index (the LM
        head's is the number of layers): event} -- that layer's first launch
        waits for the event."""
        s = stream if stream is not None else torch.cuda.current_stream()
        ready = ready or {}
        for li, (layer, io) in enumerate(self._structs):
            L, xs, ys = self.layers[li], self.x[li], self.y[li]
            if li in ready:
                s.wait_event(ready[li])
            if not self.fused_ffn and "attn_gate" not in L:
                kq_layer_step(layer, io, self.n_tok, s)
                continue
            # q, k, v (and the attention's output gate, which reads the same
            # hidden state) in one launch per format; o
            q, o = L["q"], L["o"]
            groups = {}
            for n in ATTN_NAMES:
                if n in L:
                    groups.setdefault(L[n][0], []).append(n)
            for f, names in groups.items():
                kq_gemv_multi(f, [L[n][1] for n in names], [ys[n] for n in names],
                              [L[n][2] for n in names], xs["x_attn"], q[3], self.n_tok, s)
            kq_gemv(o[0], o[1], xs["x_o"], ys["o"], o[2], o[3], self.n_tok, s)
            if self.fused_ffn:
                kq_ffn_swiglu(layer.gate, layer.up, layer.down, xs["x_ffn"], ys["gate"], ys["up"],
                              self.h[li], ys["down"], self.n_tok, s)
            else:
                gt, up, dn = L["gate"], L["up"], L["down"]
                kq_gemv_multi(gt[0], [gt[1], up[1]], [ys["gate"], ys["up"]], [gt[2], up[2]],
                              xs["x_ffn"], gt[3], self.n_tok, s)
                kq_gemv(dn[0], dn[1], xs["x_down"], ys["down"], dn[2], dn[3], self.n_tok, s)
        if self.lm_head is not None:
            if len(self._structs) in ready:
                s.wait_event(ready[len(self._structs)])
            f, W, N, K = self.lm_head
            kq_gemv(f, W, self.x_head, self.y_head, N, K, self.n_tok, s)

    def capture(self, stream=None, host_x=None):
        """Capture one step into a CUDA graph (replay with ``replay``).

        host_x: a pinned host tensor shaped like ``x_all``.  The graph then
        also copies the step's inputs from it on a second stream, in three
        pieces: layer 0's inputs, layers 1..16's, the rest (with the LM
        head's).  Layer 0 waits for the first piece, layer 1 for the second,
        layer 17 for the third, so the copies of later layers overlap the
        earlier layers' work.  (A wait before every layer would cost more than
        it hides: each one also ends the programmatic overlap of that
        layer's first launch with its predecessor's tail.)"""
        s = stream if stream is not None else torch.cuda.Stream()
        self.run(s)                       # warm the launch path outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        if host_x is None:
            with torch.cuda.graph(g, stream=s):
                self.run(s)
        else:
            if host_x.shape != self.x_all.shape or host_x.dtype != self.x_all.dtype:
                raise ValueError("host_x must have the shape and dtype of x_all")
            if not host_x.is_pinned():
                raise ValueError("host_x must be pinned host memory")
            cs = torch.cuda.Stream()
            with torch.cuda.graph(g, stream=s):
                fork = torch.cuda.Event()
                fork.record(s)
                cs.wait_event(fork)
                nl = len(self._structs)
                starts = sorted({0, min(1, nl), min(17, nl)})   # pieces begin at these layers
                ready = {}
                with torch.cuda.stream(cs):
                    for i, li in enumerate(starts):
                        end = starts[i + 1] if i + 1 < len(starts) else len(self._xoff) - 1
                        a, b = self._xoff[li], self._xoff[end]
                        if b > a:
                            self.x_all[a:b].copy_(host_x[a:b], non_blocking=True)
                        ev = torch.cuda.Event()
                        ev.record(cs)
                        ready[li] = ev
                self.run(s, ready)
                s.wait_event(ready[starts[-1]])   # join the copy stream
        self.graph = g
        return g

    def replay(self, stream=None):
        """Replay the captured step on `stream` (default: current stream)."""
        if stream is None:
            self.graph.replay()
        else:
            import torch
            with torch.cuda.stream(stream):
                self.graph.replay()
