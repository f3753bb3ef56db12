"""Pins for the oracle's activation clamp (the DeepGEMM Mega-MoE article's
`activation_clamp` argument, read as: both SwiGLU inputs clamped to [-c, c],
the gradient passing where -c <= z <= c).

Checks from outside the clamp's own code:
  * a clamp above every |pre-activation| is bit-identical to no clamp;
  * when every pre-activation saturates, x gets no gradient and W1 gets none
    (every path through the clamp is cut), and y stops depending on the
    scale of x;
  * FP64 central finite differences of L = sum(y * dY) match every gradient
    with a clamp that cuts a good share of the pre-activations (steps that
    would cross a clamp edge are skipped).
"""
import numpy as np
import pytest

import oracle
from test_oracle_layer import _problem


def _pre_activations(x, W1, idx):
    hs = [x[t] @ W1[e] for t in range(x.shape[0]) for e in idx[t] if e >= 0]
    return np.abs(np.concatenate(hs))


def test_clamp_above_every_preactivation_is_no_clamp():
    x, W1, W2, idx, w, dY = _problem(T=13, H=16, I=8, E=4, k=2, seed=21)
    c = float(_pre_activations(x, W1, idx).max()) * 1.01
    for prec in ("f64", "b16"):
        if prec == "b16":
            args = [np.asarray(a, np.float32).view(np.uint32) >> 16 for a in (x, W1, W2)]
            args = [a.astype(np.uint16) for a in args]
        else:
            args = [x, W1, W2]
        y0 = oracle.forward(*args, idx, w, precision=prec)
        y1 = oracle.forward(*args, idx, w, precision=prec, clamp=c)
        assert np.array_equal(y0, y1)
        d0 = oracle.backward_tokens(*args, idx, w, dY.astype(np.float64) if prec == "f64" else args[0], precision=prec)
        d1 = oracle.backward_tokens(*args, idx, w, dY.astype(np.float64) if prec == "f64" else args[0], precision=prec,
                                    clamp=c)
        assert all(np.array_equal(a, b) for a, b in zip(d0, d1))


def test_full_saturation_cuts_x_and_w1_gradients():
    x, W1, W2, idx, w, dY = _problem(T=9, H=8, I=4, E=3, k=2, seed=22)
    c = 1e-3
    assert _pre_activations(x, W1, idx).min() > c  # every pre-activation saturates
    dx, dw = oracle.backward_tokens(x, W1, W2, idx, w, dY, precision="f64", clamp=c)
    dW1, dW2 = oracle.backward_experts(x, W1, W2, idx, w, dY, precision="f64", clamp=c)
    assert np.all(dx == 0) and np.all(dW1 == 0)
    assert np.any(dW2 != 0) and np.any(dw != 0)  # W2 and the weights still see a (constant) activation
    y1 = oracle.forward(x, W1, W2, idx, w, precision="f64", clamp=c)
    y2 = oracle.forward(3.0 * x, W1, W2, idx, w, precision="f64", clamp=c)
    np.testing.assert_array_equal(y1, y2)


def test_finite_differences_with_clamp_fp64():
    T, H, I, E, k = 5, 8, 4, 4, 2
    x, W1, W2, idx, w, dY = _problem(T, H, I, E, k, seed=23)
    pre = _pre_activations(x, W1, idx)
    c = float(np.median(pre))  # about half of the pre-activations are cut
    assert (pre > c).sum() > 10 and (pre < c).sum() > 10

    def loss(x_, W1_, W2_, w_):
        return float(np.sum(oracle.forward(x_, W1_, W2_, idx, w_, precision="f64", clamp=c) * dY))

    def near_edge(x_, W1_):
        return np.min(np.abs(_pre_activations(x_, W1_, idx) - c)) < 1e-4

    dx, dw = oracle.backward_tokens(x, W1, W2, idx, w, dY, precision="f64", clamp=c)
    dW1, dW2 = oracle.backward_experts(x, W1, W2, idx, w, dY, precision="f64", clamp=c)
    params = dict(x=(x, dx), W1=(W1, dW1), W2=(W2, dW2), w=(w, dw))
    checked = 0
    for name, (val, grad) in params.items():
        flat = val.reshape(-1)
        for q in range(flat.size):
            step = 1e-6 * max(1.0, abs(flat[q]))
            key = {"x": "x_", "W1": "W1_", "W2": "W2_", "w": "w_"}[name]
            plus, minus = val.copy(), val.copy()
            plus.reshape(-1)[q] += step
            minus.reshape(-1)[q] -= step
            args_p = dict(x_=x, W1_=W1, W2_=W2, w_=w)
            args_m = dict(args_p)
            args_p[key], args_m[key] = plus, minus
            if name in ("x", "W1") and (near_edge(args_p["x_"], args_p["W1_"]) or
                                         near_edge(args_m["x_"], args_m["W1_"])):
                continue
            fd = (loss(**args_p) - loss(**args_m)) / (2 * step)
            an = grad.reshape(-1)[q]
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, q, fd, an)
            checked += 1
    assert checked > 0.9 * sum(v.size for v, _ in params.values())
