"""User-facing routed MoE expert layer.

``moe_layer(x, W1, W2, topk_idx, topk_weights)`` is the single autograd op of
the pages' design (Primus-Turbo "Mega MoE" README, "Key points": one op that
takes external routing).  Forward calls the routing prologue and the
forward entry point of the C ABI; backward calls the backward entry point.
PyTorch only allocates the buffers and supplies the stream.
"""
from __future__ import annotations

import torch

from . import binding as B


class MoEWorkspace:
    """Caller-owned device buffers of one layer shape (reused across steps).

    The routing tables and the saved activations of a forward live in the
    workspace until its backward reads them.  ``generation`` counts the
    forwards that wrote into it: a backward raises if another forward has
    overwritten the workspace since its own forward (two micro-batches or two
    layers sharing one workspace before their backwards)."""

    def __init__(self, T: int, H: int, I: int, E: int, k: int, device=None, activation_clamp: float = 0.0):
        self.shape = B.shape_of(T, H, I, E, k, activation_clamp=activation_clamp)
        self.layout = B.moe_workspace_layout(self.shape)
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        L = self.layout
        self.route = torch.empty(max(L.route_bytes, 16), dtype=torch.uint8, device=dev)
        self.saved = torch.empty(max(L.saved_bytes, 16), dtype=torch.uint8, device=dev)
        self._bwd = None
        self.device = dev
        self.generation = 0

    @property
    def bwd(self):
        if self._bwd is None:
            self._bwd = torch.empty(max(self.layout.bwd_bytes, 16), dtype=torch.uint8, device=self.device)
        return self._bwd


def _dims(x, W1, W2, topk_idx):
    T, H = x.shape
    E, H1, I2 = W1.shape
    if H1 != H or I2 % 2 or tuple(W2.shape) != (E, I2 // 2, H):
        raise ValueError("expected x [T,H], W1 [E,H,2I], W2 [E,I,H]")
    return T, H, I2 // 2, E, topk_idx.shape[1]


class MoEFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, W1, W2, topk_idx, topk_weights, ws=None, activation_clamp=0.0, main_grad=False):
        T, H, I, E, k = _dims(x, W1, W2, topk_idx)
        if ws is None or (ws.shape.T, ws.shape.H, ws.shape.I, ws.shape.E, ws.shape.k) != (T, H, I, E, k):
            ws = MoEWorkspace(T, H, I, E, k, device=x.device, activation_clamp=activation_clamp)
        elif ws.shape.activation_clamp != activation_clamp:
            ws.shape.activation_clamp = activation_clamp
        idx = topk_idx if topk_idx.dtype == torch.int32 else topk_idx.to(torch.int32)
        idx = idx.contiguous()
        w = topk_weights.to(torch.float32).contiguous()
        x = x.contiguous()
        y = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
        B.moe_route_prologue(ws.shape, idx, ws.route)
        B.moe_forward(ws.shape, x, W1.contiguous(), W2.contiguous(), w, ws.route, ws.saved, y)
        ws.generation += 1
        ctx.save_for_backward(x, W1, W2, w)
        ctx.ws = ws
        ctx.ws_generation = ws.generation
        ctx.w_dtype = topk_weights.dtype
        ctx.main_grad = main_grad
        return y

    @staticmethod
    def backward(ctx, dy):
        x, W1, W2, w = ctx.saved_tensors
        ws = ctx.ws
        if ws.generation != ctx.ws_generation:
            raise RuntimeError(
                "moe_layer backward: its workspace was overwritten by a later forward (this forward wrote "
                f"generation {ctx.ws_generation}, the workspace now holds generation {ws.generation}); give "
                "forwards whose backwards are still pending workspaces of their own")
        s = ws.shape
        dev = x.device
        dx = torch.empty_like(x)
        dw = torch.empty(s.T, s.k, dtype=torch.float32, device=dev)
        if ctx.main_grad:
            # FP32 main gradients: W.main_grad += dW; no bf16 gradient
            B.moe_backward_main_grad(s, dy.to(torch.bfloat16).contiguous(), x, W1.contiguous(), W2.contiguous(), w,
                                     ws.route, ws.saved, ws.bwd, dx, W1.main_grad, W2.main_grad, dw)
            return dx, None, None, None, dw.to(ctx.w_dtype), None, None, None
        dW1 = torch.empty_like(W1)
        dW2 = torch.empty_like(W2)
        B.moe_backward(s, dy.to(torch.bfloat16).contiguous(), x, W1.contiguous(), W2.contiguous(), w, ws.route,
                       ws.saved, ws.bwd, dx, dW1, dW2, dw)
        return dx, dW1, dW2, None, dw.to(ctx.w_dtype), None, None, None


def moe_layer(x, W1, W2, topk_idx, topk_weights, workspace: MoEWorkspace | None = None,
              activation_clamp: float = 0.0, accumulate_main_grad: bool = False):
    """y = sum_j topk_weights[:, j] * SwiGLU-MLP_{topk_idx[:, j]}(x), bf16.

    x bf16 [T,H]; W1 bf16 [E,H,2I] (gate | up); W2 bf16 [E,I,H];
    topk_idx int32/int64 [T,k] (-1 = dropped slot); topk_weights float [T,k].
    Differentiable in x, W1, W2 and topk_weights.  activation_clamp > 0
    clamps both SwiGLU inputs to [-c, c] (gradients pass inside only).
    accumulate_main_grad: W1.main_grad and W2.main_grad (float32 tensors of
    W1's and W2's shapes, set by the caller) get += dW1 / dW2 in FP32 and the
    autograd gradients of W1 and W2 are None."""
    if accumulate_main_grad:
        for n, W in (("W1", W1), ("W2", W2)):
            mg = getattr(W, "main_grad", None)
            if mg is None or mg.dtype != torch.float32 or tuple(mg.shape) != tuple(W.shape):
                raise ValueError(f"accumulate_main_grad needs {n}.main_grad: float32 of {n}'s shape")
    with torch.cuda.device(x.device):
        return MoEFunction.apply(x, W1, W2, topk_idx, topk_weights, workspace, float(activation_clamp),
                                 bool(accumulate_main_grad))


class FP8Experts:
    """The layer's expert weights in FP8 for inference (DeepGEMM Mega-MoE
    article, "Code Example: Fused Overlap Path": the weights are transformed
    once, the activations cast per token before each call).

    Built once from bf16 W1 [E,H,2I] and W2 [E,I,H] (moe_quantize_weights_fp8,
    moe_quantize_w2_fp8); ``forward`` casts x (moe_quantize_fp8), builds the
    routing tables and runs moe_forward_fp8.  Needs H and I multiples of 128.
    Not differentiable."""

    def __init__(self, W1, W2):
        E, H, I2 = W1.shape
        I = I2 // 2
        if I2 % 2 or tuple(W2.shape) != (E, I, H):
            raise ValueError("expected W1 [E,H,2I], W2 [E,I,H]")
        if H % 128 or I % 128:
            raise ValueError("the FP8 path needs H and I to be multiples of 128")
        self.E, self.H, self.I = E, H, I
        dev = W1.device
        s = B.shape_of(1, H, I, E, 1)
        self.W1_fp8 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=dev)
        self.W1_sf = torch.empty(E * 2 * I * H // 32, dtype=torch.uint8, device=dev)
        self.W2_fp8 = torch.empty(E, H, I, dtype=torch.uint8, device=dev)
        self.W2_sf = torch.empty(E * H * I // 32, dtype=torch.uint8, device=dev)
        with torch.cuda.device(dev):
            B.moe_quantize_weights_fp8(s, W1.contiguous(), self.W1_fp8, self.W1_sf)
            B.moe_quantize_w2_fp8(s, W2.contiguous(), self.W2_fp8, self.W2_sf)

    def forward(self, x, topk_idx, topk_weights, workspace: MoEWorkspace | None = None):
        """y bf16 [T,H] of the FP8 layer for x bf16 [T,H] and the routing."""
        T, H = x.shape
        k = topk_idx.shape[1]
        if H != self.H:
            raise ValueError("x's hidden size differs from the weights'")
        ws = workspace
        if ws is None or (ws.shape.T, ws.shape.H, ws.shape.I, ws.shape.E, ws.shape.k) != (T, H, self.I, self.E, k):
            ws = MoEWorkspace(T, H, self.I, self.E, k, device=x.device)
        ws.generation += 1  # the FP8 forward overwrites the saved activations
        idx = (topk_idx if topk_idx.dtype == torch.int32 else topk_idx.to(torch.int32)).contiguous()
        w = topk_weights.to(torch.float32).contiguous()
        xq = torch.empty(T, H, dtype=torch.uint8, device=x.device)
        xsf = torch.empty(T, H // 32, dtype=torch.uint8, device=x.device)
        y = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
        with torch.cuda.device(x.device):
            B.moe_quantize_fp8(ws.shape, x.contiguous(), xq, xsf)
            B.moe_route_prologue(ws.shape, idx, ws.route)
            B.moe_forward_fp8(ws.shape, xq, xsf, self.W1_fp8, self.W1_sf, self.W2_fp8, self.W2_sf, w, ws.route,
                              ws.saved, y)
        return y

    __call__ = forward


def train_step_from_host(x_h, topk_idx_h, topk_w_h, dY_h, W1, W2, ws: MoEWorkspace, outs: dict):
    """One forward+backward of the layer fed from pinned HOST buffers.

    Copies x, topk_idx, topk_weights and dY host->device, runs the routing
    prologue, forward and backward through the C ABI, and copies y, dx and
    d(topk_weights) back to pinned host buffers (outs['y_h'], outs['dx_h'],
    outs['dw_h']).  The weight gradients stay on the device (outs['dW1'],
    outs['dW2']) where an optimizer would consume them.  All on the current
    stream; returns without synchronising."""
    s = ws.shape
    x = outs["x"]
    x.copy_(x_h, non_blocking=True)
    outs["idx"].copy_(topk_idx_h, non_blocking=True)
    outs["w"].copy_(topk_w_h, non_blocking=True)
    outs["dY"].copy_(dY_h, non_blocking=True)
    B.moe_route_prologue(s, outs["idx"], ws.route)
    B.moe_forward(s, x, W1, W2, outs["w"], ws.route, ws.saved, outs["y"])
    B.moe_backward(s, outs["dY"], x, W1, W2, outs["w"], ws.route, ws.saved, ws.bwd, outs["dx"], outs["dW1"],
                   outs["dW2"], outs["dw"])
    outs["y_h"].copy_(outs["y"], non_blocking=True)
    outs["dx_h"].copy_(outs["dx"], non_blocking=True)
    outs["dw_h"].copy_(outs["dw"], non_blocking=True)


class HostPipeline:
    """Forward+backward steps fed from pinned HOST buffers, with the copies
    overlapped with the layer's kernels.

    ``submit(x_h, topk_idx_h, topk_w_h, dY_h, y_h, dx_h, dw_h)`` enqueues one
    step and returns at once: the host->device copies of the step's inputs go
    on an upload stream, the routing prologue, forward and backward on the
    compute stream (the current stream when the pipeline was made), and the
    device->host copies of y (as soon as the forward is done) and of dx and
    d(topk_weights) (after the backward) on a download stream.  Inputs and
    outputs on the device are double-buffered, so step n+1's uploads run
    during step n's kernels and step n's downloads during step n+1's.  The
    weight gradients stay on the device in ``dW1``/``dW2`` (overwritten by
    every step), where an optimizer would consume them.  Host buffers handed
    to ``submit`` must stay untouched until ``synchronize()``."""

    def __init__(self, ws: MoEWorkspace, W1, W2, dW1=None, dW2=None):
        s = ws.shape
        dev = ws.device
        self.ws, self.W1, self.W2 = ws, W1, W2
        self.compute = torch.cuda.current_stream(dev)
        self.up = torch.cuda.Stream(dev)
        self.down = torch.cuda.Stream(dev)
        bf = torch.bfloat16

        def slot():
            return dict(x=torch.empty(s.T, s.H, dtype=bf, device=dev),
                        idx=torch.empty(s.T, s.k, dtype=torch.int32, device=dev),
                        w=torch.empty(s.T, s.k, dtype=torch.float32, device=dev),
                        dY=torch.empty(s.T, s.H, dtype=bf, device=dev),
                        y=torch.empty(s.T, s.H, dtype=bf, device=dev),
                        dx=torch.empty(s.T, s.H, dtype=bf, device=dev),
                        dw=torch.empty(s.T, s.k, dtype=torch.float32, device=dev),
                        uploaded=torch.cuda.Event(), fwd_done=torch.cuda.Event(), bwd_done=torch.cuda.Event(),
                        downloaded=torch.cuda.Event(), used=False)

        self.slots = [slot(), slot()]
        self.dW1 = torch.empty_like(W1) if dW1 is None else dW1
        self.dW2 = torch.empty_like(W2) if dW2 is None else dW2
        self.n = 0

    def submit(self, x_h, topk_idx_h, topk_w_h, dY_h, y_h, dx_h, dw_h):
        sl = self.slots[self.n % 2]
        self.n += 1
        s = self.ws.shape
        if sl["used"]:
            # the slot's previous step must be done with its inputs and
            # outputs before they are overwritten
            self.up.wait_event(sl["bwd_done"])
            self.up.wait_event(sl["downloaded"])
        sl["used"] = True
        with torch.cuda.stream(self.up):
            sl["x"].copy_(x_h, non_blocking=True)
            sl["idx"].copy_(topk_idx_h, non_blocking=True)
            sl["w"].copy_(topk_w_h, non_blocking=True)
            sl["dY"].copy_(dY_h, non_blocking=True)
            sl["uploaded"].record(self.up)
        c = self.compute
        c.wait_event(sl["uploaded"])
        B.moe_route_prologue(s, sl["idx"], self.ws.route, stream=c)
        B.moe_forward(s, sl["x"], self.W1, self.W2, sl["w"], self.ws.route, self.ws.saved, sl["y"], stream=c)
        sl["fwd_done"].record(c)
        B.moe_backward(s, sl["dY"], sl["x"], self.W1, self.W2, sl["w"], self.ws.route, self.ws.saved, self.ws.bwd,
                       sl["dx"], self.dW1, self.dW2, sl["dw"], stream=c)
        sl["bwd_done"].record(c)
        with torch.cuda.stream(self.down):
            self.down.wait_event(sl["fwd_done"])
            y_h.copy_(sl["y"], non_blocking=True)
            self.down.wait_event(sl["bwd_done"])
            dx_h.copy_(sl["dx"], non_blocking=True)
            dw_h.copy_(sl["dw"], non_blocking=True)
            sl["downloaded"].record(self.down)

    def synchronize(self):
        """Makes the compute stream wait for every copy enqueued so far."""
        self.compute.wait_stream(self.up)
        self.compute.wait_stream(self.down)
