"""Pins of the oracle's per-token FP8 quantization (E4M3 values, UE8M0
power-of-two scales per 32-element group), against things other than the
oracle itself: PyTorch's float8_e4m3fn conversion, a brute-force nearest
search over the 256 codes, and the closed-form properties of the scale."""
import math

import numpy as np
import pytest
import torch

import oracle
from routed_grouped_gemm_routing_gb300.workloads import bf16_bits

pytestmark = pytest.mark.filterwarnings("ignore")


def test_decode_matches_torch_for_every_code():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok].astype(np.float64))


def _values(n=20000, seed=0):
    g = np.random.default_rng(seed)
    v = np.concatenate([
        g.standard_normal(n) * 10.0 ** g.uniform(-4, 2.6, n),
        # exact midpoints between neighbouring codes (ties) and the codes themselves
        np.array([oracle.e4m3_decode(c) for c in range(0x7E)], np.float64),
        np.array([(oracle.e4m3_decode(c) + oracle.e4m3_decode(c + 1)) / 2 for c in range(0x7D)], np.float64),
        np.array([2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -6 - 2.0 ** -10, 447.9, 448.0, 455.9, 0.0]),
    ])
    v = np.concatenate([v, -v])
    return v[np.abs(v) < 464.0]  # beyond, torch's conversion does not saturate


def test_encode_matches_torch_rounding():
    v = _values()
    ref = torch.tensor(v, dtype=torch.float64).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # the oracle takes the float32 value (what the GPU converts)
    got = np.array([oracle.e4m3_encode(float(np.float32(x))) for x in v], np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(v[i], hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_encode_is_the_nearest_code_ties_to_even():
    codes = [c for c in range(256) if not np.isnan(oracle.e4m3_decode(c))]
    vals = np.array([oracle.e4m3_decode(c) for c in codes])
    for x in _values(3000, seed=1):
        d = np.abs(vals - x)
        best = np.nonzero(d == d.min())[0]
        cand = [codes[i] for i in best]
        if len(set(vals[best])) > 1:  # a tie between two values: the even mantissa wins
            cand = [c for c in cand if (c & 1) == 0]
        got = oracle.e4m3_encode(x)
        assert oracle.e4m3_decode(got) == oracle.e4m3_decode(cand[0]), (x, hex(got), [hex(c) for c in cand])


def test_saturation_and_signed_zero():
    assert oracle.e4m3_encode(448.0) == 0x7E and oracle.e4m3_encode(1e6) == 0x7E
    assert oracle.e4m3_encode(-1e6) == 0xFE
    assert oracle.e4m3_encode(-0.0) == 0x80 and oracle.e4m3_encode(0.0) == 0x00


def _bits(a):
    return bf16_bits(torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16))


def test_group_scale_closed_forms():
    # one token, four groups: amax 448 -> e 0; 449 (bf16: 448) ; 450 -> bf16 450 -> e 1; 224 -> e -1; zeros -> e 0
    row = np.zeros((1, 128), np.float32)
    row[0, 5] = 448.0
    row[0, 32 + 7] = -452.0
    row[0, 64 + 1] = 224.0
    q, sf = oracle.quantize_fp8(_bits(row))
    assert list(sf[0]) == [127, 128, 126, 127]
    assert q[0, 5] == 0x7E and q[0, 32 + 7] == 0xF6  # -452 / 2 = -226 -> -224 (f 14, m 6)
    assert q[0, 65] == 0x7E and not q[0, 96:].any()


def test_quantize_properties_random():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(64, 512, generator=g) * torch.logspace(-3, 3, 64).unsqueeze(1)).to(torch.bfloat16)
    xb = bf16_bits(x)
    q, sf = oracle.quantize_fp8(xb)
    xf = x.float().numpy().astype(np.float64)
    deq = oracle.dequantize_fp8(q, sf)
    grp = np.abs(xf).reshape(64, 16, 32).max(axis=2)
    e = sf.astype(np.int64) - 127
    # e is the smallest exponent with amax / 2^e <= 448
    assert np.all(grp <= 448.0 * np.ldexp(1.0, e))
    assert np.all(grp > 224.0 * np.ldexp(1.0, e))
    # dequantized values within half a step of E4M3 (relative 2^-4 for normal codes)
    scale = np.repeat(np.ldexp(1.0, e), 32, axis=1)
    err = np.abs(deq - xf)
    tol = np.maximum(np.abs(xf) * 2.0 ** -4, scale * 2.0 ** -10)
    assert np.all(err <= tol)


def test_weight_quantization_is_the_per_column_rule():
    """quantize_weights_fp8 quantizes each column W1[e, :, f] on its own:
    brute force over the columns of a small W1 with the per-token quantizer
    and the scales' closed form (448 * 2^(sf - 127) >= max|group| > 224 *
    2^(sf - 127) for nonzero groups)."""
    rng = np.random.default_rng(11)
    E, H, I2 = 2, 96, 6
    w = (rng.standard_normal((E, H, I2)) * np.logspace(-3, 2, I2)).astype(np.float32)
    w[0, :32, 1] = 0.0
    bits = bf16_bits(torch.from_numpy(w).to(torch.bfloat16))
    q, sf = oracle.quantize_weights_fp8(bits)
    assert q.shape == (E, I2, H) and sf.shape == (E, I2, H // 32)
    for e in range(E):
        for f in range(I2):
            cq, csf = oracle.quantize_fp8(bits[e, :, f][None, :])
            assert np.array_equal(q[e, f], cq[0]) and np.array_equal(sf[e, f], csf[0])
    vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    for e in range(E):
        for f in range(I2):
            for g in range(H // 32):
                amax = np.abs(vals[e, 32 * g:32 * g + 32, f]).max()
                s = np.ldexp(1.0, int(sf[e, f, g]) - 127)
                if amax == 0:
                    assert sf[e, f, g] == 127
                else:
                    assert 448 * s >= amax > 224 * s


def _nearest_code(x):
    """E4M3 code nearest to x by search over the decoded values (ties: the
    even mantissa), independent of oracle.e4m3_encode."""
    codes = [c for c in range(256) if not np.isnan(oracle.e4m3_decode(c))]
    vals = np.array([oracle.e4m3_decode(c) for c in codes])
    d = np.abs(vals - x)
    best = np.nonzero(d == d.min())[0]
    cand = [codes[i] for i in best]
    if len(set(vals[best])) > 1:
        cand = [c for c in cand if (c & 1) == 0]
    return cand[0]


def _group_exponent(amax):
    """The smallest e with 448 * 2^e >= amax, by search (0 for amax = 0)."""
    if amax == 0:
        return 0
    e = -127
    while 448.0 * 2.0 ** e < amax:
        e += 1
    return e


def test_value_quantization_equals_the_bit_pattern_rule():
    """quantize_fp8_values on bf16-representable float64 values gives the
    bytes quantize_fp8 gives on their bit patterns."""
    g = torch.Generator().manual_seed(21)
    x = (torch.randn(48, 256, generator=g) * torch.logspace(-5, 3, 48).unsqueeze(1)).to(torch.bfloat16)
    x[0, :32] = 0.0
    x[1, 40] = 448.0
    q0, sf0 = oracle.quantize_fp8(bf16_bits(x))
    q1, sf1 = oracle.quantize_fp8_values(x.double().numpy())
    assert np.array_equal(q0, q1) and np.array_equal(sf0, sf1)


def test_value_quantization_brute_force():
    """Values that are not bf16 (the FP8 forward's activations): scale by
    search for the smallest exponent, codes by nearest search."""
    rng = np.random.default_rng(22)
    v = rng.standard_normal((6, 64)) * np.logspace(-6, 4, 6)[:, None]
    v[2, 32:] = 0.0
    v[3, 7] = 448.0 * 2.0 ** 5  # amax on a scale boundary
    q, sf = oracle.quantize_fp8_values(v)
    for t in range(v.shape[0]):
        for g in range(2):
            grp = v[t, 32 * g:32 * g + 32]
            e = _group_exponent(np.abs(grp).max())
            assert sf[t, g] == e + 127, (t, g)
            for i in range(32):
                assert q[t, 32 * g + i] == _nearest_code(grp[i] / 2.0 ** e) or (
                    oracle.e4m3_decode(q[t, 32 * g + i]) == oracle.e4m3_decode(_nearest_code(grp[i] / 2.0 ** e)))


def test_w2_quantization_is_the_per_column_rule():
    """quantize_w2_fp8 quantizes each column W2[e, :, h] (the L2 GEMM's
    contraction index i) like a token."""
    rng = np.random.default_rng(23)
    E, I, H = 2, 64, 5
    w = (rng.standard_normal((E, I, H)) * np.logspace(-2, 3, H)).astype(np.float32)
    bits = bf16_bits(torch.from_numpy(w).to(torch.bfloat16))
    q, sf = oracle.quantize_w2_fp8(bits)
    assert q.shape == (E, H, I) and sf.shape == (E, H, I // 32)
    vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    for e in range(E):
        for h in range(H):
            for g in range(I // 32):
                grp = vals[e, 32 * g:32 * g + 32, h]
                ex = _group_exponent(np.abs(grp).max())
                assert sf[e, h, g] == ex + 127
                got = np.array([oracle.e4m3_decode(c) for c in q[e, h, 32 * g:32 * g + 32]])
                ref = np.array([oracle.e4m3_decode(_nearest_code(x / 2.0 ** ex)) for x in grp])
                assert np.array_equal(got, ref)


def test_forward_fp8_brute_force():
    """oracle.forward_fp8 against the definition written out in Python loops:
    h and SwiGLU per slot, each 32-feature group of the activations scaled
    by a searched exponent and rounded to the nearest code, the L2
    contraction on the dequantized activations, the weighted sum; with an
    invalid slot (-1) and an expert no slot uses."""
    rng = np.random.default_rng(24)
    T, H, I, E, k = 3, 8, 64, 3, 2
    x = rng.standard_normal((T, H))
    W1 = rng.standard_normal((E, H, 2 * I)) * 0.7
    W2 = rng.standard_normal((E, I, H)) * 0.3
    idx = np.array([[0, 2], [2, -1], [0, 0]], np.int32)
    w = np.array([[0.7, 0.3], [1.0, 0.5], [0.25, 0.75]], np.float32)
    y, aq, asf = oracle.forward_fp8(x, W1, W2, idx, w)
    for t in range(T):
        yr = np.zeros(H)
        for j in range(k):
            e = idx[t, j]
            if e < 0:
                assert not aq[t, j].any() and not asf[t, j].any()
                continue
            a = np.zeros(I)
            for i in range(I):
                g = u = 0.0
                for h in range(H):
                    g += x[t, h] * W1[e, h, i]
                    u += x[t, h] * W1[e, h, I + i]
                a[i] = g / (1.0 + math.exp(-g)) * u
            deq = np.zeros(I)
            for gi in range(I // 32):
                grp = a[32 * gi:32 * gi + 32]
                ex = _group_exponent(np.abs(grp).max())
                assert asf[t, j, gi] == ex + 127
                for i in range(32):
                    c = _nearest_code(grp[i] / 2.0 ** ex)
                    assert oracle.e4m3_decode(aq[t, j, 32 * gi + i]) == oracle.e4m3_decode(c)
                    deq[32 * gi + i] = oracle.e4m3_decode(c) * 2.0 ** ex
            o = np.array([sum(deq[i] * W2[e, i, c] for i in range(I)) for c in range(H)])
            yr += float(w[t, j]) * o
        np.testing.assert_allclose(y[t], yr, rtol=1e-12, atol=1e-12)
