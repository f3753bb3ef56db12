"""Thin Python binding of the C ABI in include/moe_layer.h.

Argument marshalling only: every entry point takes torch tensors (device
memory owned by the caller), checks dtype / device / contiguity / size, and
passes raw pointers plus the current CUDA stream to the library.  All work
runs in the library's kernels.  There is no fallback: if the library has not
been built, or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import build as _build

_LOCK = threading.Lock()
_LIB = None

HEADER = os.path.join(_build.INCLUDE, "moe_layer.h")
MOE_OK, MOE_EINVAL, MOE_EUNSUPPORTED, MOE_ECUDA = 0, -1, -2, -3
STATUS_MPAD, STATUS_NUM_TILES, STATUS_N_INVALID, STATUS_FLAGS, STATUS_NUM_PAIRS, STATUS_WORDS = 0, 1, 2, 3, 4, 16
BLOCK_M = 128


class MoeShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "I", "E", "k", "block_m")] + [
        ("activation_clamp", ctypes.c_float)]


class MoeLayout(ctypes.Structure):
    _fields_ = [("rows_cap", ctypes.c_int64), ("tiles_cap", ctypes.c_int64)] + [
        (n, ctypes.c_size_t)
        for n in ("route_bytes", "counts", "offs", "perm", "inv", "tiles", "status", "pair_offs", "pair_owner",
                  "blk_counts", "saved_bytes", "h", "a", "o", "cmask", "bwd_bytes", "dh", "aw", "dxp", "dw_part")
    ] + [("dw_part_cols", ctypes.c_int32), ("route_blocks", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"moe error {code}: {msg}")
        self.code = code


def declared_functions() -> list[str]:
    """Names of the functions include/moe_layer.h declares."""
    text = open(HEADER).read()
    return re.findall(r"^(?:int|const char\*)\s+(moe_\w+)\s*\(", text, flags=re.M)


def lib():
    """The loaded library; raises if it has not been built."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = _build.lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is not built; run routed_grouped_gemm_routing_gb300.build.build()")
            L = ctypes.CDLL(path)
            vp, P = ctypes.c_void_p, ctypes.POINTER
            L.moe_workspace_layout.argtypes = [P(MoeShape), P(MoeLayout)]
            L.moe_route_prologue.argtypes = [P(MoeShape), vp, vp, vp]
            L.moe_router_topk.argtypes = [P(MoeShape)] + [vp] * 5
            L.moe_forward.argtypes = [P(MoeShape)] + [vp] * 8
            L.moe_backward.argtypes = [P(MoeShape)] + [vp] * 13
            L.moe_backward_main_grad.argtypes = [P(MoeShape)] + [vp] * 13
            L.moe_quantize_fp8.argtypes = [P(MoeShape)] + [vp] * 4
            L.moe_dequantize_fp8.argtypes = [P(MoeShape)] + [vp] * 4
            L.moe_forward_fp8.argtypes = [P(MoeShape)] + [vp] * 11
            L.moe_quantize_weights_fp8.argtypes = [P(MoeShape)] + [vp] * 4
            L.moe_quantize_w2_fp8.argtypes = [P(MoeShape)] + [vp] * 4
            L.moe_read_status.argtypes = [P(MoeShape), vp, vp, vp]
            for n in ("moe_workspace_layout", "moe_route_prologue", "moe_router_topk", "moe_forward", "moe_backward", "moe_backward_main_grad",
                      "moe_quantize_fp8", "moe_dequantize_fp8", "moe_forward_fp8", "moe_quantize_weights_fp8",
                      "moe_quantize_w2_fp8", "moe_read_status"):
                getattr(L, n).restype = ctypes.c_int
            L.moe_trace_begin.argtypes = [vp, ctypes.c_int]
            L.moe_trace_begin.restype = ctypes.c_int
            L.moe_trace_end.argtypes = []
            L.moe_trace_end.restype = ctypes.c_int
            L.moe_trace_kernel.argtypes = [ctypes.c_int]
            L.moe_trace_kernel.restype = ctypes.c_char_p
            L.moe_last_error.restype = ctypes.c_char_p
            L.moe_last_error.argtypes = []
            L.moe_version.restype = ctypes.c_char_p
            L.moe_version.argtypes = []
            _LIB = L
    return _LIB


def _check(rc: int):
    if rc != MOE_OK:
        raise MoeError(rc, lib().moe_last_error().decode())


def shape_of(T: int, H: int, I: int, E: int, k: int, block_m: int = BLOCK_M, activation_clamp: float = 0.0) -> MoeShape:
    return MoeShape(T, H, I, E, k, block_m, activation_clamp)


def moe_workspace_layout(shape: MoeShape) -> MoeLayout:
    out = MoeLayout()
    _check(lib().moe_workspace_layout(ctypes.byref(shape), ctypes.byref(out)))
    return out


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t, dtype, numel=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        # the library launches on the current device
        raise ValueError(f"{name} is on {t.device}, the current device is cuda:{torch.cuda.current_device()}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return t.data_ptr()


def moe_router_topk(shape: MoeShape, logits, topk_idx, topk_w, route_ws, stream=None):
    """Router top-k gating (logits f32 [T, E] -> topk_idx int32 [T, k], topk_w
    f32 [T, k]) followed by the routing prologue into route_ws."""
    L = moe_workspace_layout(shape)
    _check(lib().moe_router_topk(
        ctypes.byref(shape), _ptr(logits, torch.float32, shape.T * shape.E, "logits"),
        _ptr(topk_idx, torch.int32, shape.T * shape.k, "topk_idx"),
        _ptr(topk_w, torch.float32, shape.T * shape.k, "topk_w"),
        _ptr(route_ws, torch.uint8, L.route_bytes, "route_ws"), _stream(stream)))


def moe_route_prologue(shape: MoeShape, topk_idx, route_ws, stream=None):
    L = moe_workspace_layout(shape)
    _check(lib().moe_route_prologue(
        ctypes.byref(shape), _ptr(topk_idx, torch.int32, shape.T * shape.k, "topk_idx"),
        _ptr(route_ws, torch.uint8, L.route_bytes, "route_ws"), _stream(stream)))


def moe_forward(shape: MoeShape, x, W1, W2, topk_w, route_ws, saved, y, stream=None):
    L = moe_workspace_layout(shape)
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    bf = torch.bfloat16
    _check(lib().moe_forward(
        ctypes.byref(shape), _ptr(x, bf, T * H, "x"), _ptr(W1, bf, E * H * 2 * I, "W1"), _ptr(W2, bf, E * I * H, "W2"),
        _ptr(topk_w, torch.float32, T * k, "topk_w"), _ptr(route_ws, torch.uint8, L.route_bytes, "route_ws"),
        _ptr(saved, torch.uint8, L.saved_bytes, "saved"), _ptr(y, bf, T * H, "y"), _stream(stream)))


def moe_backward(shape: MoeShape, dY, x, W1, W2, topk_w, route_ws, saved, bwd_ws, dx, dW1, dW2, dtopk_w,
                 stream=None):
    L = moe_workspace_layout(shape)
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    bf = torch.bfloat16
    _check(lib().moe_backward(
        ctypes.byref(shape), _ptr(dY, bf, T * H, "dY"), _ptr(x, bf, T * H, "x"), _ptr(W1, bf, E * H * 2 * I, "W1"),
        _ptr(W2, bf, E * I * H, "W2"), _ptr(topk_w, torch.float32, T * k, "topk_w"),
        _ptr(route_ws, torch.uint8, L.route_bytes, "route_ws"), _ptr(saved, torch.uint8, L.saved_bytes, "saved"),
        _ptr(bwd_ws, torch.uint8, L.bwd_bytes, "bwd_ws"), _ptr(dx, bf, T * H, "dx"),
        _ptr(dW1, bf, E * H * 2 * I, "dW1"), _ptr(dW2, bf, E * I * H, "dW2"),
        _ptr(dtopk_w, torch.float32, T * k, "dtopk_w"), _stream(stream)))


def moe_quantize_fp8(shape: MoeShape, x, x_fp8, x_sf, stream=None):
    """Per-token FP8 quantization: x bf16 [T, H] -> x_fp8 uint8 [T, H] (E4M3
    bytes) and x_sf uint8 [T, H // 32] (UE8M0 scale exponents)."""
    T, H = shape.T, shape.H
    _check(lib().moe_quantize_fp8(ctypes.byref(shape), _ptr(x, torch.bfloat16, T * H, "x"),
                                  _ptr(x_fp8, torch.uint8, T * H, "x_fp8"), _ptr(x_sf, torch.uint8, T * H // 32, "x_sf"),
                                  _stream(stream)))


def moe_dequantize_fp8(shape: MoeShape, x_fp8, x_sf, x_out, stream=None):
    """x_out bf16 [T, H] = decode(x_fp8) * 2^(x_sf - 127) (exact)."""
    T, H = shape.T, shape.H
    _check(lib().moe_dequantize_fp8(ctypes.byref(shape), _ptr(x_fp8, torch.uint8, T * H, "x_fp8"),
                                    _ptr(x_sf, torch.uint8, T * H // 32, "x_sf"),
                                    _ptr(x_out, torch.bfloat16, T * H, "x_out"), _stream(stream)))


def moe_quantize_weights_fp8(shape: MoeShape, W1, W1_fp8, W1_sf, stream=None):
    """W1 bf16 [E, H, 2I] -> W1_fp8 uint8 [E, 2I, H] (E4M3, K-major) and W1_sf
    uint8 [E * 2I * H // 32] (UE8M0 scales in the L1 kernel's atom layout)."""
    H, I, E = shape.H, shape.I, shape.E
    _check(lib().moe_quantize_weights_fp8(
        ctypes.byref(shape), _ptr(W1, torch.bfloat16, E * H * 2 * I, "W1"),
        _ptr(W1_fp8, torch.uint8, E * 2 * I * H, "W1_fp8"), _ptr(W1_sf, torch.uint8, E * 2 * I * H // 32, "W1_sf"),
        _stream(stream)))


def moe_quantize_w2_fp8(shape: MoeShape, W2, W2_fp8, W2_sf, stream=None):
    """W2 bf16 [E, I, H] -> W2_fp8 uint8 [E, H, I] (E4M3, K-major) and W2_sf
    uint8 [E * H * I // 32] (UE8M0 scales in the L2 kernel's atom layout)."""
    H, I, E = shape.H, shape.I, shape.E
    _check(lib().moe_quantize_w2_fp8(
        ctypes.byref(shape), _ptr(W2, torch.bfloat16, E * I * H, "W2"),
        _ptr(W2_fp8, torch.uint8, E * H * I, "W2_fp8"), _ptr(W2_sf, torch.uint8, E * H * I // 32, "W2_sf"),
        _stream(stream)))


def moe_forward_fp8(shape: MoeShape, x_fp8, x_sf, W1_fp8, W1_sf, W2_fp8, W2_sf, topk_w, route_ws, saved, y,
                    stream=None):
    """moe_forward on E4M3 operands (block-scaled MMA in both GEMMs): x_fp8 /
    x_sf from moe_quantize_fp8, W1_fp8 / W1_sf from moe_quantize_weights_fp8,
    W2_fp8 / W2_sf from moe_quantize_w2_fp8; a is quantized between the
    GEMMs (saved's a region then holds its E4M3 rows and scales)."""
    L = moe_workspace_layout(shape)
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    bf = torch.bfloat16
    _check(lib().moe_forward_fp8(
        ctypes.byref(shape), _ptr(x_fp8, torch.uint8, T * H, "x_fp8"), _ptr(x_sf, torch.uint8, T * H // 32, "x_sf"),
        _ptr(W1_fp8, torch.uint8, E * 2 * I * H, "W1_fp8"), _ptr(W1_sf, torch.uint8, E * 2 * I * H // 32, "W1_sf"),
        _ptr(W2_fp8, torch.uint8, E * H * I, "W2_fp8"), _ptr(W2_sf, torch.uint8, E * H * I // 32, "W2_sf"),
        _ptr(topk_w, torch.float32, T * k, "topk_w"),
        _ptr(route_ws, torch.uint8, L.route_bytes, "route_ws"), _ptr(saved, torch.uint8, L.saved_bytes, "saved"),
        _ptr(y, bf, T * H, "y"), _stream(stream)))


def moe_backward_main_grad(shape: MoeShape, dY, x, W1, W2, topk_w, route_ws, saved, bwd_ws, dx, main_grad_W1,
                           main_grad_W2, dtopk_w, stream=None):
    """moe_backward, but main_grad_W1 / main_grad_W2 (float32, same shapes as
    W1 / W2) get += dW1 / dW2 in FP32 instead of bf16 dW being written."""
    L = moe_workspace_layout(shape)
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    bf, f32 = torch.bfloat16, torch.float32
    _check(lib().moe_backward_main_grad(
        ctypes.byref(shape), _ptr(dY, bf, T * H, "dY"), _ptr(x, bf, T * H, "x"), _ptr(W1, bf, E * H * 2 * I, "W1"),
        _ptr(W2, bf, E * I * H, "W2"), _ptr(topk_w, f32, T * k, "topk_w"),
        _ptr(route_ws, torch.uint8, L.route_bytes, "route_ws"), _ptr(saved, torch.uint8, L.saved_bytes, "saved"),
        _ptr(bwd_ws, torch.uint8, L.bwd_bytes, "bwd_ws"), _ptr(dx, bf, T * H, "dx"),
        _ptr(main_grad_W1, f32, E * H * 2 * I, "main_grad_W1"), _ptr(main_grad_W2, f32, E * I * H, "main_grad_W2"),
        _ptr(dtopk_w, f32, T * k, "dtopk_w"), _stream(stream)))


def moe_read_status(shape: MoeShape, route_ws, stream=None) -> list[int]:
    """Status words (synchronises the stream)."""
    L = moe_workspace_layout(shape)
    out = (ctypes.c_int32 * STATUS_WORDS)()
    _check(lib().moe_read_status(ctypes.byref(shape), _ptr(route_ws, torch.uint8, L.route_bytes, "route_ws"),
                                 ctypes.cast(out, ctypes.c_void_p), _stream(stream)))
    return list(out)


def moe_last_error() -> str:
    return lib().moe_last_error().decode()


def moe_version() -> str:
    return lib().moe_version().decode()


def route_tables(shape: MoeShape, route_ws) -> dict:
    """Device views of the routing tables inside route_ws (no copy)."""
    L = moe_workspace_layout(shape)

    def view(off, n):
        return route_ws[off: off + 4 * n].view(torch.int32)

    return dict(counts=view(L.counts, shape.E), offs=view(L.offs, shape.E + 1), perm=view(L.perm, L.rows_cap),
                inv=view(L.inv, shape.T * shape.k), tiles=view(L.tiles, L.tiles_cap),
                status=view(L.status, STATUS_WORDS), pair_offs=view(L.pair_offs, shape.E + 1),
                pair_owner=view(L.pair_owner, L.tiles_cap))


def saved_tensors(shape: MoeShape, saved) -> dict:
    """Device views of h, a, o inside the forward's saved buffer (no copy)."""
    L = moe_workspace_layout(shape)
    R, H, I = L.rows_cap, shape.H, shape.I

    def view(off, rows, cols):
        return saved[off: off + 2 * rows * cols].view(torch.bfloat16).view(rows, cols)

    return dict(h=view(L.h, R, 2 * I), a=view(L.a, R, I), o=view(L.o, R, H))


def backward_tensors(shape: MoeShape, bwd) -> dict:
    """Device views of dh, aw, dxp inside the backward workspace (no copy)."""
    L = moe_workspace_layout(shape)
    R, H, I = L.rows_cap, shape.H, shape.I

    def view(off, rows, cols):
        return bwd[off: off + 2 * rows * cols].view(torch.bfloat16).view(rows, cols)

    return dict(dh=view(L.dh, R, 2 * I), aw=view(L.aw, R, I), dxp=view(L.dxp, R, H))


class KernelTrace:
    """Brackets every kernel the library launches from this thread with a
    pair of CUDA events (moe_trace_begin / moe_trace_end), for per-kernel
    device times.  Events are created here with timing enabled."""

    def __init__(self, max_launches: int):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * max_launches)]
        for ev in self.events:  # force creation of the underlying event
            ev.record()
        self._arr = (ctypes.c_void_p * len(self.events))(*[ev.cuda_event for ev in self.events])
        self.names: list[str] = []
        self.count = 0

    def __enter__(self):
        _check(lib().moe_trace_begin(ctypes.cast(self._arr, ctypes.c_void_p), len(self.events)))
        return self

    def __exit__(self, *exc):
        self.count = lib().moe_trace_end()
        self.names = [lib().moe_trace_kernel(i).decode() for i in range(self.count)]
        return False

    def durations_ms(self) -> list[tuple[str, float]]:
        """(kernel name, device ms) per traced launch; call after synchronising."""
        n = min(self.count, len(self.events) // 2)
        return [(self.names[i], self.events[2 * i].elapsed_time(self.events[2 * i + 1])) for i in range(n)]


def moe_selftest_wait_timeout(shape: MoeShape, route_ws, limit_ns: int, elapsed=None, stream=None):
    """Runs the kernels' bounded-wait give-up path on purpose (diagnostic; see
    include/moe_layer.h): sets bit 0 of route_ws's MOE_STATUS_FLAGS word.
    elapsed: None or an int64 CUDA tensor of 3 elements (ns each waiting warp
    spent before giving up)."""
    L = moe_workspace_layout(shape)
    fn = lib().moe_selftest_wait_timeout
    fn.argtypes = [ctypes.POINTER(MoeShape), ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    _check(fn(ctypes.byref(shape), _ptr(route_ws, torch.uint8, L.route_bytes, "route_ws"), int(limit_ns),
              _ptr(elapsed, torch.int64, 3, "elapsed"), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 32 << 20  # MOE_NOALLOC_SCRATCH_BYTES of include/moe_layer.h


def moe_forward_noalloc(shape: MoeShape, x, W1, W2, topk_idx, topk_w, y, status_out=None, stream=None):
    """Routing prologue + forward with the library's static scratch instead of
    caller workspaces (for callers that cannot allocate device memory; see
    include/moe_layer.h).  Overwrites y; keeps nothing for a backward pass.
    status_out: None or an int32 CUDA tensor of STATUS_WORDS elements that
    receives the call's status words (copied on the stream, no sync)."""
    L = lib()
    fn = L.moe_forward_noalloc
    fn.argtypes = [ctypes.POINTER(MoeShape)] + [ctypes.c_void_p] * 8
    fn.restype = ctypes.c_int
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    bf = torch.bfloat16
    _check(fn(ctypes.byref(shape), _ptr(x, bf, T * H, "x"), _ptr(W1, bf, E * H * 2 * I, "W1"),
              _ptr(W2, bf, E * I * H, "W2"), _ptr(topk_idx, torch.int32, T * k, "topk_idx"),
              _ptr(topk_w, torch.float32, T * k, "topk_w"), _ptr(y, bf, T * H, "y"),
              _ptr(status_out, torch.int32, STATUS_WORDS, "status_out"), _stream(stream)))
