"""Pins for the oracle's forward and backward (Primus-Turbo Mega MoE README,
"Pipeline": x -> dispatch -> L1 -> SwiGLU -> L2 -> top-k weighted combine,
and the conjugate backward).

Each check reaches the oracle from outside its own code:
  * brute force: every expert run densely on every token with library
    matmuls, then masked by the routing (dense-then-mask);
  * k = 1, weight 1, one expert: a dense SwiGLU MLP computed with torch's
    own silu / matmul / autograd (FP64);
  * E = 1: the dense MLP scaled by the sum of a token's weights;
  * equivariance under a permutation of the tokens;
  * linearity in topk_weights;
  * FP64 central finite differences of L = sum(y * dY) for every input;
  * an expert with no slots has exactly zero weight gradients;
  * the FP32/bfloat16-input instantiation agrees with the FP64 one.
"""
import numpy as np
import pytest
import torch

import oracle


def _problem(T, H, I, E, k, seed, distinct=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    W1 = rng.standard_normal((E, H, 2 * I)) / np.sqrt(H)
    W2 = rng.standard_normal((E, I, H)) / np.sqrt(I)
    if distinct:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    else:
        idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
    w = rng.random((T, k)) + 0.1
    dY = rng.standard_normal((T, H))
    return x, W1, W2, idx, w, dY


def _dense_then_mask(x, W1, W2, idx, w):
    """Every expert on every token (numpy matmul), then the routing mask."""
    T, H = x.shape
    E, _, I2 = W1.shape
    I = I2 // 2
    y = np.zeros((T, H))
    M = np.zeros((T, E))
    for t in range(T):
        for j in range(idx.shape[1]):
            if 0 <= idx[t, j] < E:
                M[t, idx[t, j]] += w[t, j]
    for e in range(E):
        h = x @ W1[e]
        g, u = h[:, :I], h[:, I:]
        a = g / (1.0 + np.exp(-g)) * u
        y += M[:, e: e + 1] * (a @ W2[e])
    return y


@pytest.mark.parametrize("distinct", [True, False])
def test_forward_brute_force(distinct):
    x, W1, W2, idx, w, _ = _problem(T=23, H=16, I=8, E=5, k=3, seed=1, distinct=distinct)
    idx[4, 1] = -1
    idx[9, 0] = 7  # out of range -> dropped
    y = oracle.forward(x, W1, W2, idx, w, precision="f64")
    ref = _dense_then_mask(x, W1, W2, idx, w)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def _torch_dense_mlp(x, W1e, W2e):
    I = W2e.shape[0]
    xt, W1t, W2t = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (x, W1e, W2e))
    h = xt @ W1t
    y = (torch.nn.functional.silu(h[:, :I]) * h[:, I:]) @ W2t
    return y, (xt, W1t, W2t)


def test_top1_weight1_is_dense_swiglu_mlp():
    x, W1, W2, _, _, dY = _problem(T=11, H=12, I=6, E=3, k=1, seed=2)
    idx = np.full((11, 1), 2, np.int32)
    w = np.ones((11, 1))
    y = oracle.forward(x, W1, W2, idx, w, precision="f64")
    yt, (xt, W1t, W2t) = _torch_dense_mlp(x, W1[2], W2[2])
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-12, atol=1e-12)
    # backward against torch autograd of the same dense MLP
    (yt * torch.tensor(dY)).sum().backward()
    dx, dw = oracle.backward_tokens(x, W1, W2, idx, w, dY, precision="f64")
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dw[:, 0], (yt.detach().numpy() * dY).sum(1), rtol=1e-11, atol=1e-12)
    dW1, dW2 = oracle.backward_experts(x, W1, W2, idx, w, dY, precision="f64")
    np.testing.assert_allclose(dW1[2], W1t.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dW2[2], W2t.grad.numpy(), rtol=1e-11, atol=1e-12)
    assert np.all(dW1[:2] == 0) and np.all(dW2[:2] == 0)


def test_single_expert_scales_by_weight_sum():
    x, W1, W2, _, w, _ = _problem(T=9, H=8, I=4, E=1, k=3, seed=3)
    idx = np.zeros((9, 3), np.int32)  # the same expert in every slot
    y = oracle.forward(x, W1, W2, idx, w, precision="f64")
    yt, _ = _torch_dense_mlp(x, W1[0], W2[0])
    np.testing.assert_allclose(y, w.sum(1, keepdims=True) * yt.detach().numpy(), rtol=1e-12, atol=1e-12)


def test_token_permutation_equivariance():
    x, W1, W2, idx, w, dY = _problem(T=17, H=8, I=4, E=6, k=2, seed=4)
    pi = np.random.default_rng(0).permutation(17)
    y = oracle.forward(x, W1, W2, idx, w, precision="f64")
    yp = oracle.forward(x[pi], W1, W2, idx[pi], w[pi], precision="f64")
    np.testing.assert_allclose(yp, y[pi], rtol=1e-13, atol=1e-14)
    dW1, dW2 = oracle.backward_experts(x, W1, W2, idx, w, dY, precision="f64")
    dW1p, dW2p = oracle.backward_experts(x[pi], W1, W2, idx[pi], w[pi], dY[pi], precision="f64")
    np.testing.assert_allclose(dW1p, dW1, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dW2p, dW2, rtol=1e-11, atol=1e-13)


def test_linear_in_topk_weights():
    x, W1, W2, idx, w1, _ = _problem(T=13, H=8, I=4, E=5, k=3, seed=5)
    w2 = np.random.default_rng(1).standard_normal(w1.shape)
    al, be = 0.7, -1.3
    y = oracle.forward(x, W1, W2, idx, al * w1 + be * w2, precision="f64")
    ref = al * oracle.forward(x, W1, W2, idx, w1, precision="f64") + be * oracle.forward(x, W1, W2, idx, w2, precision="f64")
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_dropped_slot_equals_zero_weight():
    x, W1, W2, idx, w, _ = _problem(T=10, H=8, I=4, E=4, k=2, seed=6)
    idx2, w0 = idx.copy(), w.copy()
    idx2[2, 1] = -1
    w0[2, 1] = 0.0
    np.testing.assert_allclose(oracle.forward(x, W1, W2, idx2, w, precision="f64"),
                               oracle.forward(x, W1, W2, idx, w0, precision="f64"), rtol=0, atol=0)


@pytest.mark.parametrize("case", ["distinct", "duplicates_and_empty"])
def test_finite_differences_fp64(case):
    T, H, I, E, k = 5, 8, 4, 4, 2
    x, W1, W2, idx, w, dY = _problem(T, H, I, E, k, seed=7)
    if case == "duplicates_and_empty":
        idx = np.array([[0, 0], [1, 0], [0, 1], [1, 1], [0, -1]], np.int32)  # experts 2, 3 empty

    def loss(x_, W1_, W2_, w_):
        return float(np.sum(oracle.forward(x_, W1_, W2_, idx, w_, precision="f64") * dY))

    dx, dw = oracle.backward_tokens(x, W1, W2, idx, w, dY, precision="f64")
    dW1, dW2 = oracle.backward_experts(x, W1, W2, idx, w, dY, precision="f64")
    params = dict(x=(x, dx), W1=(W1, dW1), W2=(W2, dW2), w=(w, dw))
    for name, (val, grad) in params.items():
        flat = val.reshape(-1)
        for q in range(flat.size):
            step = 1e-6 * max(1.0, abs(flat[q]))
            args = dict(x_=x, W1_=W1, W2_=W2, w_=w)
            key = {"x": "x_", "W1": "W1_", "W2": "W2_", "w": "w_"}[name]
            plus, minus = val.copy(), val.copy()
            plus.reshape(-1)[q] += step
            minus.reshape(-1)[q] -= step
            args[key] = plus
            lp = loss(**args)
            args[key] = minus
            lm = loss(**args)
            fd = (lp - lm) / (2 * step)
            an = grad.reshape(-1)[q]
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, q, fd, an)
    if case == "duplicates_and_empty":
        assert np.all(dW1[2:] == 0) and np.all(dW2[2:] == 0)
        assert dw[4, 1] == 0


def _bf16_round(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16)


def test_fp32_bf16_instantiation_matches_fp64():
    x, W1, W2, idx, w, dY = _problem(T=31, H=64, I=32, E=6, k=2, seed=8)
    xb, W1b, W2b, dYb = (_bf16_round(a) for a in (x, W1, W2, dY))
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    exact = lambda t: t.to(torch.float64).numpy()  # noqa: E731
    w32 = w.astype(np.float32)
    y32 = oracle.forward(bits(xb), bits(W1b), bits(W2b), idx, w32)
    y64 = oracle.forward(exact(xb), exact(W1b), exact(W2b), idx, w32.astype(np.float64), precision="f64")
    assert y32.dtype == np.float32
    np.testing.assert_allclose(y32, y64, rtol=2e-5, atol=2e-5 * np.abs(y64).max())
    dx32, dw32 = oracle.backward_tokens(bits(xb), bits(W1b), bits(W2b), idx, w32, bits(dYb))
    dx64, dw64 = oracle.backward_tokens(exact(xb), exact(W1b), exact(W2b), idx, w32.astype(np.float64),
                                        exact(dYb), precision="f64")
    np.testing.assert_allclose(dx32, dx64, rtol=2e-5, atol=2e-5 * np.abs(dx64).max())
    np.testing.assert_allclose(dw32, dw64, rtol=2e-5, atol=2e-5 * np.abs(dw64).max())
    e_list = np.array([0, 3], np.int32)
    a1, a2 = oracle.backward_experts(bits(xb), bits(W1b), bits(W2b), idx, w32, bits(dYb), experts=e_list)
    b1, b2 = oracle.backward_experts(exact(xb), exact(W1b), exact(W2b), idx, w32.astype(np.float64),
                                     exact(dYb), experts=e_list, precision="f64")
    np.testing.assert_allclose(a1, b1, rtol=2e-5, atol=2e-5 * np.abs(b1).max())
    np.testing.assert_allclose(a2, b2, rtol=2e-5, atol=2e-5 * np.abs(b2).max())


def test_token_and_expert_subsets_match_full():
    x, W1, W2, idx, w, dY = _problem(T=12, H=8, I=4, E=5, k=2, seed=9)
    y = oracle.forward(x, W1, W2, idx, w, precision="f64")
    sub = np.array([7, 2, 11], np.int32)
    np.testing.assert_array_equal(oracle.forward(x, W1, W2, idx, w, tokens=sub, precision="f64"), y[sub])
    dx, dw = oracle.backward_tokens(x, W1, W2, idx, w, dY, precision="f64")
    dxs, dws = oracle.backward_tokens(x, W1, W2, idx, w, dY, tokens=sub, precision="f64")
    np.testing.assert_array_equal(dxs, dx[sub])
    np.testing.assert_array_equal(dws, dw[sub])
    dW1, dW2 = oracle.backward_experts(x, W1, W2, idx, w, dY, precision="f64")
    es = np.array([4, 1], np.int32)
    dW1s, dW2s = oracle.backward_experts(x, W1, W2, idx, w, dY, experts=es, precision="f64")
    np.testing.assert_array_equal(dW1s, dW1[es])
    np.testing.assert_array_equal(dW2s, dW2[es])
