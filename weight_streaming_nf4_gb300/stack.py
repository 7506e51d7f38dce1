"""Buffers of one training run of the synthetic stack, allocated with torch.

``StackRun`` owns every device / pinned buffer that ``ws_stack_train_step``
reads or writes (the library allocates nothing): the NF4 block images (a
pinned host image plus a 2-slot HBM window when streamed, one HBM image when
resident), LoRA parameters, gradients, Adam moments, block-boundary
activations, saved activations (resident), the gradient buffer, the
workspace and the loss scalar.  Weights are quantised on the GPU by the
streamed loader (``ws_stack_put_weight``), one tensor at a time, straight
into the block image (device) or through a one-tensor staging buffer into
the pinned image (host).
"""
from __future__ import annotations

import torch

from . import ops


class StackRun:
    def __init__(self, cfg: ops.StackCfg, block_layers: int, streamed: bool, weight_fn,
                 param_fn, device="cuda", image_from: "StackRun" = None, n_micro: int = 1,
                 order: int = ops.GA_MICROBATCH_MAJOR):
        """weight_fn(layer, lin, N, K) -> bf16 [N, K] device tensor (the frozen base);
        param_fn(layer, lin, N, K) -> (A [16, K], B [N, 16]) fp32 device tensors.
        image_from: another run of the same config (resident or streamed) whose
        quantised image is copied instead of quantising again.  n_micro / order: gradient
        accumulation over n_micro micro-batches per step (h0 [n_micro, M*H])."""
        assert cfg.n_layers % block_layers == 0
        self.cfg, self.bl, self.streamed = cfg, block_layers, streamed
        self.n_micro, self.order = n_micro, order
        self.opts = ops.step_opts(n_micro, order)
        self.nb = cfg.n_layers // block_layers
        sz = ops.stack_sizes(cfg, block_layers)
        self.sizes = sz
        bb = sz["block_bytes"]
        dev = torch.device(device)
        M, H = cfg.M, cfg.H
        f32 = dict(dtype=torch.float32, device=dev)
        # ---- frozen NF4 base: the images are zeroed (the bytes between the
        # 256-aligned pieces then compare equal too) and filled one tensor at a
        # time by the streamed loader (ws_stack_put_weight): the GPU holds
        # one bf16 weight and one tensor's NF4 at a time
        if streamed:
            self.host_weights = torch.zeros(self.nb * bb, dtype=torch.uint8, pin_memory=True)
            self.window = torch.empty(2 * bb, dtype=torch.uint8, device=dev)
            self.dev_weights = None
        else:
            self.host_weights = None
            self.window = None
            self.dev_weights = torch.zeros(self.nb * bb, dtype=torch.uint8, device=dev)
        image = self.host_weights if streamed else self.dev_weights
        shapes = cfg.shapes()
        if image_from is not None:
            src = image_from.host_weights if image_from.streamed else image_from.dev_weights
            for b in range(self.nb):
                image[b * bb:(b + 1) * bb].copy_(src[b * bb:(b + 1) * bb])
        else:
            staging = (torch.empty(ops.stack_loader_staging_bytes(cfg), dtype=torch.uint8,
                                   device=dev) if streamed else None)
            for layer in range(cfg.n_layers):
                for lin, (N, K) in enumerate(shapes):
                    W = weight_fn(layer, lin, N, K)
                    ops.stack_put_weight(cfg, block_layers, layer, lin, W, image, staging)
                    del W
            torch.cuda.current_stream(dev).synchronize()
            del staging
        # ---- LoRA parameters, gradients, Adam state
        n = sz["n_params"]
        self.params = torch.zeros(n, **f32)
        for layer in range(cfg.n_layers):
            for lin, (N, K) in enumerate(shapes):
                oA, oB = ops.stack_param_offset(cfg, layer, lin)
                A, B = param_fn(layer, lin, N, K)
                self.params[oA:oA + 16 * K].copy_(A.reshape(-1))
                self.params[oB:oB + 16 * N].copy_(B.reshape(-1))
        self.grads = torch.zeros(n, **f32)
        self.adam_m = torch.zeros(n, **f32)
        self.adam_v = torch.zeros(n, **f32)
        self.boundary = torch.zeros(n_micro * (self.nb + 1) * M * H, **f32)
        self.saved = None if streamed else torch.empty(cfg.n_layers * sz["saved_layer"],
                                                       dtype=torch.uint8, device=dev)
        self.dh = torch.zeros(max(2, n_micro) * M * H, **f32)
        self.workspace = torch.empty(sz["workspace"], dtype=torch.uint8, device=dev)
        self.loss = torch.zeros(1, **f32)
        self.copy_stream = torch.cuda.Stream(device=dev) if streamed else None
        p = lambda t: 0 if t is None else t.data_ptr()
        self.c = ops.StackBuffersC(p(self.host_weights), p(self.dev_weights), p(self.window),
                                   p(self.params), p(self.grads), p(self.adam_m), p(self.adam_v),
                                   p(self.boundary), p(self.saved), p(self.dh), p(self.workspace),
                                   self.workspace.numel(), p(self.loss))

    def step(self, step: int, h0: torch.Tensor, lr: float = 2e-4, stream=None):
        """Enqueue one training step (ws_stack_train_step) on ``stream``."""
        ops.stack_train_step(self.cfg, self.bl, self.streamed, self.c, step, h0, lr, stream=stream,
                             copy_stream=self.copy_stream, opts=self.opts)

    def graph(self, lr: float, stream: torch.cuda.Stream, time_copies: bool = False,
              copy_piece_bytes: int = 0) -> "ops.StepGraph":
        """Capture one training step as a CUDA graph on ``stream`` (a created
        stream, not the default one); ``g.step(step, h0, stream)`` replays it.
        time_copies (streamed runs): time every block copy of a replay;
        copy_piece_bytes: issue each block copy in pieces of that size."""
        opts = ops.step_opts(self.n_micro, self.order, time_copies, copy_piece_bytes)
        return ops.StepGraph(self.cfg, self.bl, self.streamed, self.c, lr, stream, self.copy_stream,
                             opts=opts)

    def param(self, layer: int, lin: int, which: str, t: torch.Tensor = None):
        """View of A [16, K] or B [N, 16] of (layer, lin) inside a parameter-layout array."""
        t = self.params if t is None else t
        N, K = self.cfg.shapes()[lin]
        oA, oB = ops.stack_param_offset(self.cfg, layer, lin)
        if which == "A":
            return t[oA:oA + 16 * K].view(16, K)
        return t[oB:oB + 16 * N].view(N, 16)

    def device_bytes(self) -> int:
        ts = [self.window, self.dev_weights, self.params, self.grads, self.adam_m, self.adam_v,
              self.boundary, self.saved, self.dh, self.workspace, self.loss]
        return sum(t.numel() * t.element_size() for t in ts if t is not None)
