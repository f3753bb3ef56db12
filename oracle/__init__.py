"""CPU oracle for the routed MoE expert layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``routed_grouped_gemm_routing_gb300``) never imports it and shares no code
with it.

The numerical work is plain C (``moe_oracle.c``), built here with gcc and
called through ctypes.  See ``moe_oracle.c`` for the definitions and where
each comes from (Primus-Turbo "Mega MoE" README, "Pipeline" and
"Implementation Map"; DeepGEMM Mega-MoE article, "Block-M Alignment").

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(brute force, closed-form special cases, invariants, finite differences).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIB = None


def lib_path() -> str:
    return os.path.join(_BUILD, f"liboracle_{platform.machine()}.so")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP) into oracle/_build/."""
    out = lib_path()
    src = os.path.join(_HERE, "moe_oracle.c")
    body = os.path.join(_HERE, "moe_oracle_body.h")
    if not force and os.path.exists(out):
        newest = max(os.path.getmtime(src), os.path.getmtime(body))
        if os.path.getmtime(out) >= newest:
            return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = build()
            L = ctypes.CDLL(path)
            i32, i64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
            L.oracle_rows_cap.argtypes = [i32, i32, i32, i32]
            L.oracle_rows_cap.restype = i64
            L.oracle_route.argtypes = [i32, i32, i32, i32] + [vp] * 7
            L.oracle_route.restype = None
            L.oracle_router_topk.argtypes = [i32, i32, i32, vp, vp, vp]
            L.oracle_router_topk.restype = None
            for suf in ("b16", "f64"):
                f64 = ctypes.c_double
                getattr(L, f"oracle_forward_{suf}").argtypes = [i32] * 5 + [f64] + [vp] * 5 + [i32, vp, vp]
                getattr(L, f"oracle_backward_tokens_{suf}").argtypes = [i32] * 5 + [f64] + [vp] * 6 + [i32, vp, vp, vp]
                getattr(L, f"oracle_backward_experts_{suf}").argtypes = [i32] * 5 + [f64] + [vp] * 6 + [i32, vp, vp, vp]
                for n in ("forward", "backward_tokens", "backward_experts"):
                    getattr(L, f"oracle_{n}_{suf}").restype = None
            L.oracle_num_threads.restype = ctypes.c_int
            L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_decode.restype = ctypes.c_double
            L.oracle_e4m3_encode.argtypes = [ctypes.c_double]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_quantize_fp8.argtypes = [i32, i32, i32, vp, vp, vp]
            L.oracle_quantize_fp8.restype = None
            L.oracle_quantize_fp8_f64.argtypes = [i32, i32, i32, vp, vp, vp]
            L.oracle_quantize_fp8_f64.restype = None
            L.oracle_forward_fp8.argtypes = [i32] * 5 + [vp] * 5 + [i32, vp, vp, vp, vp]
            L.oracle_forward_fp8.restype = None
            _LIB = L
    return _LIB


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def num_threads() -> int:
    return int(_lib().oracle_num_threads())


def rows_cap(T: int, E: int, k: int, bm: int) -> int:
    return int(_lib().oracle_rows_cap(T, E, k, bm))


def router_topk(logits: np.ndarray, k: int):
    """Top-k gating of router logits [T, E] (FP32): returns topk_idx int32
    [T, k] (decreasing logit, equal logits in increasing expert id; NaN
    counts as -inf) and topk_w float32 [T, k] (softmax over the k selected
    logits, FP64 then rounded)."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    idx = np.zeros((max(T, 1), k), np.int32)
    w = np.zeros((max(T, 1), k), np.float32)
    _lib().oracle_router_topk(T, E, k, _p(lg), _p(idx), _p(w))
    return idx[:T], w[:T]


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 byte (OCP FP8: bias 7, 3 mantissa bits, no
    infinities, 0x7F / 0xFF NaN)."""
    return float(_lib().oracle_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(v: float) -> int:
    """E4M3 byte of v: round to nearest, ties to even, saturating at +-448."""
    return int(_lib().oracle_e4m3_encode(float(v)))


def quantize_fp8(x_bits: np.ndarray, gran: int = 32):
    """Per-token FP8 quantization with UE8M0 block scales (DeepGEMM Mega-MoE
    article, usage example: per-token cast, granularity 32).  x_bits: bf16
    bit patterns [T, H] (uint16).  Returns q uint8 [T, H] (E4M3 bytes) and
    sf uint8 [T, H // gran] (biased exponents: scale = 2^(sf - 127))."""
    xb = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H = xb.shape
    if H % gran:
        raise ValueError("H must be a multiple of the granularity")
    q = np.zeros((max(T, 1), H), np.uint8)
    sf = np.zeros((max(T, 1), H // gran), np.uint8)
    _lib().oracle_quantize_fp8(T, H, gran, _p(xb), _p(q), _p(sf))
    return q[:T], sf[:T]


def quantize_weights_fp8(W1_bits: np.ndarray, gran: int = 32):
    """FP8 weights for the L1 GEMM (DeepGEMM Mega-MoE article, usage example:
    the weights are transformed once for the low-precision kernel).  W1_bits:
    bf16 bit patterns [E, H, 2I].  Each column W1[e, :, f] is quantized like
    a token of quantize_fp8 (groups of `gran` consecutive h, the contraction
    index of the L1 GEMM).  Returns q uint8 [E, 2I, H] and sf uint8
    [E, 2I, H // gran]."""
    wb = np.ascontiguousarray(W1_bits, dtype=np.uint16)
    E, H, I2 = wb.shape
    q, sf = quantize_fp8(np.ascontiguousarray(wb.transpose(0, 2, 1)).reshape(E * I2, H), gran)
    return q.reshape(E, I2, H), sf.reshape(E, I2, H // gran)


def quantize_fp8_values(v: np.ndarray, gran: int = 32):
    """quantize_fp8's rule on float64 values [T, H] instead of bf16 bit
    patterns (the activations between the FP8 forward's two GEMMs).  Returns
    q uint8 [T, H] and sf uint8 [T, H // gran]."""
    x = np.ascontiguousarray(v, dtype=np.float64)
    T, H = x.shape
    if H % gran:
        raise ValueError("H must be a multiple of the granularity")
    q = np.zeros((max(T, 1), H), np.uint8)
    sf = np.zeros((max(T, 1), H // gran), np.uint8)
    _lib().oracle_quantize_fp8_f64(T, H, gran, _p(x), _p(q), _p(sf))
    return q[:T], sf[:T]


def quantize_w2_fp8(W2_bits: np.ndarray, gran: int = 32):
    """FP8 weights for the L2 GEMM, the counterpart of quantize_weights_fp8:
    W2_bits: bf16 bit patterns [E, I, H]; each column W2[e, :, h] is quantized
    like a token of quantize_fp8 (groups of `gran` consecutive i, the
    contraction index of the L2 GEMM).  Returns q uint8 [E, H, I] and sf
    uint8 [E, H, I // gran]."""
    wb = np.ascontiguousarray(W2_bits, dtype=np.uint16)
    E, I, H = wb.shape
    q, sf = quantize_fp8(np.ascontiguousarray(wb.transpose(0, 2, 1)).reshape(E * H, I), gran)
    return q.reshape(E, H, I), sf.reshape(E, H, I // gran)


def forward_fp8(x, W1, W2, topk_idx, topk_w, tokens=None):
    """FP8 forward for the listed tokens (all by default): x [T, H], W1
    [E, H, 2I], W2 [E, I, H] as the float64 values the E4M3 operands stand
    for; the SwiGLU output of every slot is quantized to E4M3 with UE8M0
    scales per 32 consecutive features before the L2 contraction (see
    oracle_forward_fp8).  Returns y [n, H] float64, aq uint8 [n, k, I] and
    asf uint8 [n, k, I // 32]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    W1 = np.ascontiguousarray(W1, dtype=np.float64)
    W2 = np.ascontiguousarray(W2, dtype=np.float64)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    T, H, I, E, k = _dims(x, W1, W2, idx)
    if I % 32:
        raise ValueError("I must be a multiple of 32")
    toks = np.ascontiguousarray(np.arange(T) if tokens is None else tokens, dtype=np.int32)
    n = len(toks)
    y = np.zeros((max(n, 1), H), np.float64)
    aq = np.zeros((max(n, 1), k, I), np.uint8)
    asf = np.zeros((max(n, 1), k, I // 32), np.uint8)
    _lib().oracle_forward_fp8(T, H, I, E, k, _p(x), _p(W1), _p(W2), _p(idx), _p(w), n, _p(toks), _p(y), _p(aq),
                              _p(asf))
    return y[:n], aq[:n], asf[:n]


def dequantize_fp8(q: np.ndarray, sf: np.ndarray, gran: int = 32) -> np.ndarray:
    """decode(q) * 2^(sf - 127), float64 [T, H]."""
    table = np.array([e4m3_decode(c) for c in range(256)], np.float64)
    scale = np.ldexp(1.0, sf.astype(np.int64) - 127)
    return table[q] * np.repeat(scale, gran, axis=1)


def route(topk_idx: np.ndarray, E: int, bm: int = 128) -> dict:
    """Routing tables from topk_idx [T, k] (int32).  Returns a dict of numpy
    int32 arrays: counts, offs, perm, inv, tiles, and ints mpad, num_tiles,
    n_invalid."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    cap = rows_cap(T, E, k, bm)
    counts = np.zeros(E, np.int32)
    offs = np.zeros(E + 1, np.int32)
    perm = np.zeros(max(cap, 1), np.int32)
    inv = np.zeros(max(T * k, 1), np.int32)
    tiles = np.zeros(max(cap // bm, 1), np.int32)
    scal = np.zeros(3, np.int32)
    _lib().oracle_route(T, E, k, bm, _p(idx), _p(counts), _p(offs), _p(perm), _p(inv), _p(tiles), _p(scal))
    return dict(counts=counts, offs=offs, perm=perm[:cap], inv=inv[: T * k], tiles=tiles[: cap // bm],
                mpad=int(scal[0]), num_tiles=int(scal[1]), n_invalid=int(scal[2]))


def _prep(precision, x, W1, W2, topk_idx, topk_w, dY=None):
    if precision == "b16":
        conv = lambda a: np.ascontiguousarray(a, dtype=np.uint16)  # noqa: E731
        wconv = lambda a: np.ascontiguousarray(a, dtype=np.float32)  # noqa: E731
        rdt = np.float32
    elif precision == "f64":
        conv = wconv = lambda a: np.ascontiguousarray(a, dtype=np.float64)  # noqa: E731
        rdt = np.float64
    else:
        raise ValueError(precision)
    out = [conv(x), conv(W1), conv(W2), np.ascontiguousarray(topk_idx, dtype=np.int32), wconv(topk_w)]
    if dY is not None:
        out.append(conv(dY))
    return out, rdt


def _dims(x, W1, W2, topk_idx):
    T, H = x.shape
    E, H1, I2 = W1.shape
    assert H1 == H and I2 % 2 == 0
    I = I2 // 2
    assert W2.shape == (E, I, H)
    k = topk_idx.shape[1]
    return T, H, I, E, k


def forward(x, W1, W2, topk_idx, topk_w, tokens=None, precision="b16", clamp=0.0):
    """y rows [len(tokens), H] for the listed tokens (all tokens by default).

    precision "b16": x, W1, W2 are bfloat16 bit patterns (uint16 arrays),
    topk_w float32, FP32 arithmetic.  precision "f64": everything float64.
    clamp > 0: SwiGLU inputs clamped to [-clamp, clamp] (0: no clamp)."""
    (x, W1, W2, idx, w), rdt = _prep(precision, x, W1, W2, topk_idx, topk_w)
    T, H, I, E, k = _dims(x, W1, W2, idx)
    toks = np.ascontiguousarray(np.arange(T) if tokens is None else tokens, dtype=np.int32)
    y = np.zeros((len(toks), H), rdt)
    fn = getattr(_lib(), f"oracle_forward_{precision}")
    fn(T, H, I, E, k, float(clamp), _p(x), _p(W1), _p(W2), _p(idx), _p(w), len(toks), _p(toks), _p(y))
    return y


def backward_tokens(x, W1, W2, topk_idx, topk_w, dY, tokens=None, precision="b16", clamp=0.0):
    """(dx [n, H], dtopk_w [n, k]) for the listed tokens."""
    (x, W1, W2, idx, w, dY), rdt = _prep(precision, x, W1, W2, topk_idx, topk_w, dY)
    T, H, I, E, k = _dims(x, W1, W2, idx)
    toks = np.ascontiguousarray(np.arange(T) if tokens is None else tokens, dtype=np.int32)
    dx = np.zeros((len(toks), H), rdt)
    dw = np.zeros((len(toks), k), rdt)
    fn = getattr(_lib(), f"oracle_backward_tokens_{precision}")
    fn(T, H, I, E, k, float(clamp), _p(x), _p(W1), _p(W2), _p(idx), _p(w), _p(dY), len(toks), _p(toks), _p(dx),
       _p(dw))
    return dx, dw


def backward_experts(x, W1, W2, topk_idx, topk_w, dY, experts=None, precision="b16", clamp=0.0):
    """(dW1 [n, H, 2I], dW2 [n, I, H]) for the listed experts."""
    (x, W1, W2, idx, w, dY), rdt = _prep(precision, x, W1, W2, topk_idx, topk_w, dY)
    T, H, I, E, k = _dims(x, W1, W2, idx)
    exps = np.ascontiguousarray(np.arange(E) if experts is None else experts, dtype=np.int32)
    dW1 = np.zeros((len(exps), H, 2 * I), rdt)
    dW2 = np.zeros((len(exps), I, H), rdt)
    fn = getattr(_lib(), f"oracle_backward_experts_{precision}")
    fn(T, H, I, E, k, float(clamp), _p(x), _p(W1), _p(W2), _p(idx), _p(w), _p(dY), len(exps), _p(exps), _p(dW1),
       _p(dW2))
    return dW1, dW2
