"""CPU-only checks of the C-ABI library: it builds for sm_103a, loads, exports
every function include/moe_layer.h declares, computes the workspace layout on
the host, and rejects bad shapes and pointers without touching a GPU."""
import ctypes

import pytest

import oracle
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.lib()


def test_exports_every_declared_function(lib):
    names = B.declared_functions()
    assert set(names) >= {"moe_workspace_layout", "moe_route_prologue", "moe_forward", "moe_backward",
                          "moe_read_status", "moe_last_error", "moe_version"}
    for n in names:
        assert hasattr(lib, n), f"{n} is declared but not exported"
    assert "sm_103a" in B.moe_version()


@pytest.mark.parametrize("T,H,I,E,k", [(64, 128, 64, 8, 2), (4096, 2048, 1408, 64, 6), (8192, 7168, 2048, 256, 8),
                                       (4096, 7168, 3072, 384, 6), (1, 64, 64, 1024, 3), (0, 64, 64, 4, 2),
                                       (300000, 64, 64, 16, 8)])
def test_layout(lib, T, H, I, E, k):
    L = B.moe_workspace_layout(B.shape_of(T, H, I, E, k))
    assert L.rows_cap == oracle.rows_cap(T, E, k, 128)
    assert L.tiles_cap == L.rows_cap // 128
    assert L.dw_part_cols == (I + 31) // 32
    offs = [L.counts, L.offs, L.perm, L.inv, L.tiles, L.status, L.pair_offs, L.pair_owner]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert L.offs >= L.counts + 4 * E and L.perm >= L.offs + 4 * (E + 1)
    assert L.inv >= L.perm + 4 * L.rows_cap and L.tiles >= L.inv + 4 * T * k
    assert L.status >= L.tiles + 4 * L.tiles_cap and L.pair_offs >= L.status + 64
    assert L.pair_owner >= L.pair_offs + 4 * (E + 1) and L.blk_counts >= L.pair_owner + 4 * L.tiles_cap
    assert L.blk_counts % 256 == 0
    # slot blocks of whole 1024-slot rounds, at most 1024 of them
    tk = T * k
    rounds = -(-tk // 1024)
    per = max(1, -(-rounds // 1024)) * 1024
    assert L.route_blocks == -(-tk // per) and L.route_blocks <= 1024
    assert L.route_bytes >= L.blk_counts + 4 * (L.route_blocks * (E + 1) + 1)
    R = L.rows_cap
    assert L.a >= L.h + 2 * R * 2 * I and L.o >= L.a + 2 * R * I and L.cmask >= L.o + 2 * R * H
    assert L.saved_bytes >= L.cmask + 4 * R * (2 * I // 32)
    assert L.aw >= L.dh + 2 * R * 2 * I and L.dxp >= L.aw + 2 * R * I
    assert L.dw_part >= L.dxp + 2 * R * H and L.bwd_bytes >= L.dw_part + 4 * R * L.dw_part_cols


@pytest.mark.parametrize("bad,code", [((64, 100, 64, 8, 2, 128), B.MOE_EUNSUPPORTED),
                                      ((64, 128, 96, 8, 2, 128), B.MOE_EUNSUPPORTED),
                                      ((64, 128, 64, 8, 9, 128), B.MOE_EINVAL),
                                      ((64, 128, 64, 2000, 2, 128), B.MOE_EINVAL),
                                      ((-1, 128, 64, 8, 2, 128), B.MOE_EINVAL),
                                      ((64, 128, 64, 8, 2, 64), B.MOE_EUNSUPPORTED),
                                      ((64, 0, 64, 8, 2, 128), B.MOE_EINVAL),
                                      ((64, 128, 64, 8, 2, 128, float("nan")), B.MOE_EINVAL),
                                      ((64, 128, 64, 8, 2, 128, float("inf")), B.MOE_EINVAL)])
def test_bad_shapes_rejected_on_host(lib, bad, code):
    s = B.MoeShape(*bad)
    out = B.MoeLayout()
    assert lib.moe_workspace_layout(ctypes.byref(s), ctypes.byref(out)) == code
    assert B.moe_last_error() != ""
    # entry points reject the shape before touching any device
    assert lib.moe_route_prologue(ctypes.byref(s), None, None, None) == code
    assert lib.moe_forward(ctypes.byref(s), *([None] * 8)) == code


def test_null_shape_and_null_pointers(lib):
    assert lib.moe_workspace_layout(None, None) == B.MOE_EINVAL
    s = B.shape_of(64, 128, 64, 8, 2)
    out = B.MoeLayout()
    assert lib.moe_workspace_layout(ctypes.byref(s), None) == B.MOE_EINVAL


def test_null_and_misaligned_pointers_rejected_before_device_use(lib):
    s = B.shape_of(64, 128, 64, 8, 2)
    assert lib.moe_route_prologue(ctypes.byref(s), None, None, None) == B.MOE_EINVAL
    assert lib.moe_forward(ctypes.byref(s), *([None] * 8)) == B.MOE_EINVAL
    assert lib.moe_backward(ctypes.byref(s), *([None] * 13)) == B.MOE_EINVAL
    fake = [4096 * (i + 1) for i in range(13)]
    fake[3] += 4  # misaligned topk_w
    assert lib.moe_backward(ctypes.byref(s), *fake) == B.MOE_EUNSUPPORTED
    assert "aligned" in B.moe_last_error()


def test_variant_entry_points_reject_bad_arguments_before_device_use(lib):
    s = B.shape_of(64, 128, 64, 8, 2)
    # FP32 main-gradient backward: same checks as moe_backward
    assert lib.moe_backward_main_grad(ctypes.byref(s), *([None] * 13)) == B.MOE_EINVAL
    fake = [4096 * (i + 1) for i in range(13)]
    fake[10] += 8  # misaligned main_grad_W2
    assert lib.moe_backward_main_grad(ctypes.byref(s), *fake) == B.MOE_EUNSUPPORTED
    # FP8 entry points
    assert lib.moe_quantize_fp8(ctypes.byref(s), None, None, None, None) == B.MOE_EINVAL
    assert lib.moe_dequantize_fp8(ctypes.byref(s), None, None, None, None) == B.MOE_EINVAL
    assert lib.moe_forward_fp8(ctypes.byref(s), *([None] * 11)) == B.MOE_EINVAL
    assert lib.moe_quantize_weights_fp8(ctypes.byref(s), None, None, None, None) == B.MOE_EINVAL
    assert lib.moe_quantize_w2_fp8(ctypes.byref(s), None, None, None, None) == B.MOE_EINVAL
    # FP8 weights and the FP8 forward need H (W1) and H and I (W2, the
    # forward) multiples of 128: K blocks of 128 E4M3 bytes
    h64 = B.shape_of(64, 192, 128, 8, 2)
    i64 = B.shape_of(64, 256, 192, 8, 2)
    assert lib.moe_quantize_weights_fp8(ctypes.byref(h64), 4096, 8192, 16384, None) == B.MOE_EUNSUPPORTED
    assert lib.moe_quantize_w2_fp8(ctypes.byref(h64), 4096, 8192, 16384, None) == B.MOE_EUNSUPPORTED
    assert lib.moe_quantize_w2_fp8(ctypes.byref(i64), 4096, 8192, 16384, None) == B.MOE_EUNSUPPORTED
    for sh in (h64, i64):
        assert lib.moe_forward_fp8(ctypes.byref(sh), *[4096 * (i + 1) for i in range(10)], None) == B.MOE_EUNSUPPORTED
        assert "128" in B.moe_last_error()
    # no activation clamp in the FP8 forward
    cl = B.MoeShape(64, 256, 128, 8, 2, 128, 10.0)
    assert lib.moe_forward_fp8(ctypes.byref(cl), *[4096 * (i + 1) for i in range(10)], None) == B.MOE_EUNSUPPORTED
    assert "clamp" in B.moe_last_error()
    assert lib.moe_quantize_fp8(ctypes.byref(s), 4096, 8192 + 4, 16384, None) == B.MOE_EUNSUPPORTED
    bad = B.MoeShape(64, 96, 64, 8, 2, 128)  # H not a multiple of 64
    assert lib.moe_quantize_fp8(ctypes.byref(bad), 4096, 8192, 16384, None) == B.MOE_EUNSUPPORTED
    # no tokens: nothing to do, no device touched
    z = B.shape_of(0, 128, 64, 8, 2)
    assert lib.moe_quantize_fp8(ctypes.byref(z), None, None, None, None) == 0
    assert lib.moe_dequantize_fp8(ctypes.byref(z), None, None, None, None) == 0
