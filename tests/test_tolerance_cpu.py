"""Why the parity bar's max-error term is 2^-7 * max|ref| for bf16 outputs.

The layer's data path (reading c7: intermediates h, a, dh, aw and the outputs
stored in bf16, every product summed in FP32) is emulated here on the CPU
with exact float64 arithmetic and a bf16 rounding at exactly those storage
points, for the weight gradients of one expert with few routed rows (the
case where an output element is made of a few large terms).  Against the
oracle's FP64 weight gradients, the emulation

  * meets the mean-relative bar (5e-3) and the applied max bar
    2e-2 * rms + 1e-3 + 2^-7 * max|ref| in every seeded case, and
  * exceeds the one-rounding bar 2e-2 * rms + 1e-3 + 2^-8 * max|ref| in
    some of them: the output's own half-step is not the only bf16 rounding
    an element carries, so that bar would fail a path that does nothing but
    what the reading prescribes.

The emulation shares nothing with the CUDA library; the reference is the
oracle (FP64 instantiation)."""
import numpy as np
import torch

import oracle
from moe_testlib import compare


def _bf16(a):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def _emulated_weight_grads(x, W1, W2, dY, w):
    """dW1, dW2 of one expert whose rows are x (all routed to it with
    weights w), with bf16 storage of h, a, dh, aw and of the outputs."""
    I = W2.shape[0]
    hb = _bf16(x @ W1)
    g, u = hb[:, :I], hb[:, I:]
    sg = 1.0 / (1.0 + np.exp(-g))
    ab = _bf16(g * sg * u)
    da = w[:, None] * (dY @ W2.T)
    dhb = np.concatenate([_bf16(da * u * sg * (1.0 + g * (1.0 - sg))), _bf16(da * g * sg)], axis=1)
    awb = _bf16(w[:, None] * ab)
    return _bf16(x.T @ dhb), _bf16(awb.T @ dY)


def _bars(got, ref):
    err = np.abs(got - ref)
    rms = np.sqrt(np.mean(ref * ref))
    amax = np.abs(ref).max()
    literal = 2e-2 * rms + 1e-3
    return err.max(), literal + 2.0 ** -8 * amax, literal + 2.0 ** -7 * amax


def test_bf16_data_path_needs_two_half_steps():
    H, I = 1024, 256
    beyond_one_rounding = 0
    for seed in range(16):
        rng = np.random.default_rng(seed)
        rows = (12, 39)[seed % 2]
        x = _bf16(rng.standard_normal((rows, H)))
        W1 = _bf16(rng.standard_normal((1, H, 2 * I)) / np.sqrt(H))
        W2 = _bf16(rng.standard_normal((1, I, H)) / np.sqrt(I))
        dY = _bf16(rng.standard_normal((rows, H)))
        w = rng.uniform(0.05, 0.4, (rows, 1))
        idx = np.zeros((rows, 1), np.int32)
        ref1, ref2 = oracle.backward_experts(x, W1, W2, idx, w, dY, precision="f64")
        got1, got2 = _emulated_weight_grads(x, W1[0], W2[0], dY, w[:, 0])
        for name, got, ref in (("dW1", got1, ref1[0]), ("dW2", got2, ref2[0])):
            compare(f"emulated {name} ({rows} rows, seed {seed})", got, ref)  # the applied bar holds
            emax, one, two = _bars(got, ref)
            assert emax <= two
            beyond_one_rounding += emax > one
    assert beyond_one_rounding > 0, "every case met the one-rounding bar"
