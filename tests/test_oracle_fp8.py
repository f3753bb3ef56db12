"""Pins of the oracle's per-token FP8 quantization (E4M3 values, UE8M0
power-of-two scales per 32-element group), against things other than the
oracle itself: PyTorch's float8_e4m3fn conversion, a brute-force nearest
search over the 256 codes, and the closed-form properties of the scale."""
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
