"""Training driver of the small tensor-parallel GPT on one GPU.

Allocates the parameters, their gradients and the AdamW moments as four flat fp32
device buffers (every tensor at a 64-element-aligned offset), points the library's
tp_gpt_weights / tp_gpt_grads structs into them, and sequences one training step as
three library calls: tp_gpt_fwd_bwd (loss and every gradient), tp_train_step_advance
(the device-side step counter and loss history) and tp_adamw_step_device over the whole
flat buffer. No host argument changes from one step to the next, so capture() records a
step once as a CUDA graph and replay() runs it. No arithmetic of the model runs here.

Parameter order (also the flat layout): E, then per layer gamma1, beta1, Wqkv, Wo,
gamma2, beta2, W1, W2, then gammaf, betaf -- the layer and weight shapes of
include/tpmlp.h.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import tpmlp as T

LAYER_KEYS = ("gamma1", "beta1", "Wqkv", "Wo", "gamma2", "beta2", "W1", "W2")
ADAMW = {"lr": 3e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.01}


def param_shapes(vocab, hidden, ffn, layers):
    h, f = hidden, ffn
    shp = {"gamma1": (h,), "beta1": (h,), "Wqkv": (h, 3 * h), "Wo": (h, h), "gamma2": (h,),
           "beta2": (h,), "W1": (h, f), "W2": (f, h)}
    out = [("E", (vocab, h))]
    for li in range(layers):
        out += [(f"L{li}.{k}", shp[k]) for k in LAYER_KEYS]
    return out + [("gammaf", (h,)), ("betaf", (h,))]


class SmallGPT:
    def __init__(self, vocab, hidden, heads, ffn, layers, batch, seq, shards,
                 mode=T.Reduce.BUFFERS, steps=50, device="cuda"):
        import torch
        self.cfg = T.GptConfig(vocab, hidden, heads, ffn, layers, batch, seq, shards)
        self.mode = mode
        self.shapes = param_shapes(vocab, hidden, ffn, layers)
        self.offsets, off = {}, 0
        for name, shp in self.shapes:
            self.offsets[name] = off
            off += -(-int(np.prod(shp)) // 64) * 64
        self.n = off
        z = lambda: torch.zeros(off, dtype=torch.float32, device=device)
        self.p, self.g, self.m, self.v = z(), z(), z(), z()
        self.losses = torch.zeros(max(steps, 1), dtype=torch.float32, device=device)
        self.loss_now = torch.zeros(1, dtype=torch.float32, device=device)
        self.step_dev = torch.zeros(1, dtype=torch.int32, device=device)
        self.graph = None
        wsb = T.tp_gpt_workspace_size(self.cfg, T.DType.F32, mode)
        if wsb == 0:
            raise ValueError("invalid GPT configuration")
        self.ws = torch.empty(wsb, dtype=torch.uint8, device=device)
        self.ids = torch.zeros(batch * seq, dtype=torch.int32, device=device)
        self.targets = torch.zeros(batch * seq, dtype=torch.int32, device=device)
        addr = lambda buf, name: buf.data_ptr() + 4 * self.offsets[name]
        self._lw = (T.LayerWeights * max(layers, 1))()
        self._lg = (T.LayerGrads * max(layers, 1))()
        for li in range(layers):
            for k in LAYER_KEYS:
                setattr(self._lw[li], k, addr(self.p, f"L{li}.{k}"))
                setattr(self._lg[li], "d" + k, addr(self.g, f"L{li}.{k}"))
        self.weights = T.GptWeights(addr(self.p, "E"), addr(self.p, "gammaf"),
                                    addr(self.p, "betaf"), self._lw)
        self.grads = T.GptGrads(addr(self.g, "E"), addr(self.g, "gammaf"),
                                addr(self.g, "betaf"), self._lg)
        self.t = 0

    def view(self, buf, name):
        o = self.offsets[name]
        shp = dict(self.shapes)[name]
        return buf[o:o + int(np.prod(shp))].view(*shp)

    def load(self, params):
        """params: name -> array (float64 / float32) in `param_shapes` order and shapes."""
        import torch
        for name, _ in self.shapes:
            self.view(self.p, name).copy_(torch.from_numpy(np.asarray(params[name], np.float32)))
        self.m.zero_()
        self.v.zero_()
        self.step_dev.zero_()
        self.t = 0

    def set_batch(self, ids, targets):
        import torch
        self.ids.copy_(torch.from_numpy(np.asarray(ids, np.int32).reshape(-1)))
        self.targets.copy_(torch.from_numpy(np.asarray(targets, np.int32).reshape(-1)))

    def fwd_bwd(self, loss_slot=0, stream=None):
        T.tp_gpt_fwd_bwd(self.cfg, self.weights, self.grads, self.ids, self.targets,
                         self.losses[loss_slot:loss_slot + 1], T.DType.F32, self.mode, self.ws,
                         self.ws.numel(), stream)

    def _enqueue_step(self, opt, stream):
        T.tp_gpt_fwd_bwd(self.cfg, self.weights, self.grads, self.ids, self.targets,
                         self.loss_now, T.DType.F32, self.mode, self.ws, self.ws.numel(), stream)
        T.tp_train_step_advance(self.step_dev, self.loss_now, self.losses, self.losses.numel(),
                                stream)
        T.tp_adamw_step_device(self.p, self.g, self.m, self.v, self.n, self.step_dev, opt["lr"],
                               opt["beta1"], opt["beta2"], opt["eps"], opt["weight_decay"], stream)

    def step(self, opt=ADAMW, stream=None):
        """One training step on the loaded batch: loss into losses[t], then AdamW."""
        self._enqueue_step(opt, stream)
        self.t += 1

    def capture(self, opt=ADAMW):
        """Record one training step (the launches of step()) as a CUDA graph. Make at least
        one eager step first: the library sets its kernels' attributes and creates its side
        streams outside a capture."""
        import torch
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._enqueue_step(opt, None)

    def replay(self):
        """One training step from the captured graph (its stream is torch's current one)."""
        self.graph.replay()
        self.t += 1
