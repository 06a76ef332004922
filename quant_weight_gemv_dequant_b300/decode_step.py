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

from . import (kq_gemv, kq_layer, kq_layer_io, kq_layer_step, make_matrix)

LAYER_NAMES = ("q", "k", "v", "o", "gate", "up", "down")
X_OF = {"q": "x_attn", "k": "x_attn", "v": "x_attn", "o": "x_o",
        "gate": "x_ffn", "up": "x_ffn", "down": "x_down"}


class DecodeStep:
    """layers: list of {name: (fmt, W_device_uint8, N_out, K)} for the seven
    projections; lm_head: (fmt, W, N_out, K) or None."""

    def __init__(self, layers, lm_head, n_tok: int, device="cuda"):
        self.n_tok = n_tok
        self.layers = layers
        self.lm_head = lm_head
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
        for w in widths:
            views.append(self.x_all[off:off + n_tok * w].view(n_tok, w))
            off += n_tok * w
        for li, L in enumerate(layers):
            xs = dict(zip(("x_attn", "x_o", "x_ffn", "x_down"), views[4 * li:4 * li + 4]))
            ys = {n: torch.empty((n_tok, L[n][2]), dtype=torch.float32, device=device)
                  for n in LAYER_NAMES}
            layer = kq_layer(*[make_matrix(L[n][0], L[n][1], L[n][2], L[n][3]) for n in LAYER_NAMES])
            io = kq_layer_io(*[xs[k].data_ptr() for k in ("x_attn", "x_o", "x_ffn", "x_down")],
                             *[ys[n].data_ptr() for n in LAYER_NAMES])
            self.x.append(xs)
            self.y.append(ys)
            self._structs.append((layer, io))
        if lm_head is not None:
            self.x_head = views[-1]
            self.y_head = torch.empty((n_tok, lm_head[2]), dtype=torch.float32, device=device)
        self.graph = None

    def weight_bytes(self) -> int:
        total = sum(L[n][1].numel() for L in self.layers for n in LAYER_NAMES)
        if self.lm_head is not None:
            total += self.lm_head[1].numel()
        return total

    def launches(self) -> int:
        """Kernel launches per step (one per format-group of a layer step)."""
        per_layer = 0
        for L in self.layers[:1]:
            for group in (("q", "k", "v"), ("o",), ("gate", "up"), ("down",)):
                per_layer += len({L[n][0] for n in group})
        return per_layer * len(self.layers) + (1 if self.lm_head is not None else 0)

    def run(self, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream()
        for layer, io in self._structs:
            kq_layer_step(layer, io, self.n_tok, s)
        if self.lm_head is not None:
            f, W, N, K = self.lm_head
            kq_gemv(f, W, self.x_head, self.y_head, N, K, self.n_tok, s)

    def capture(self, stream=None):
        """Capture one step into a CUDA graph (replay with ``replay``)."""
        s = stream if stream is not None else torch.cuda.Stream()
        self.run(s)                       # warm the launch path outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self.run(s)
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
