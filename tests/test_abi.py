"""The C-ABI library loads on a machine without a GPU, exports every symbol
include/moe.h declares, and rejects bad arguments on the host before
launching anything."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_93_b300 import binding as B
from mixture_experts_layer_93_b300 import build as BUILD

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    BUILD.build()
    return B.lib()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("moe_route", "moe_permute", "moe_token_round", "moe_forward", "moe_expert_up",
                 "moe_expert_down", "moe_combine", "moe_prepare_weights", "moe_workspace_bytes"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    assert sorted(B._SIGNATURES) == declared_symbols()


def test_status_strings(lib):
    for st in range(7):
        assert B.status_string(st) not in ("", "unknown status")
    assert B.status_string(99) == "unknown status"


SHAPES_OK = [(256, 128, 64, 8, 2), (8192, 4096, 14336, 8, 2), (16384, 7168, 2048, 256, 8),
             (32768, 1536, 256, 128, 8), (1, 64, 64, 1, 1), (5, 64, 192, 1024, 32)]
SHAPES_BAD = [(0, 128, 64, 8, 2), (16, 100, 64, 8, 2), (16, 128, 96, 8, 2), (16, 128, 64, 8, 9),
              (16, 128, 64, 2000, 2), (16, 128, 64, 64, 33), (16, 128, 64, 8, 0)]


@pytest.mark.parametrize("T,d,n,E,k", SHAPES_OK)
def test_workspace_bytes_valid(lib, T, d, n, E, k):
    s = B.make_shape(T, d, n, E, k)
    nb = B.moe_workspace_bytes(s)
    cap = B.moe_row_capacity(s)
    assert cap == T * k
    # at least h and ys plus the routing arrays
    assert nb >= cap * (n + d) * 2 + T * E * 4
    lay = B.moe_workspace_layout(s)
    offs = [lay[name] for name in B.WS_SLOTS]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs) and offs[0] >= 256
    assert lay["ys"] + cap * d * 2 <= nb


def test_row_capacity_with_rounding(lib):
    s = B.make_shape(1000, 128, 64, 16, 4, tile=128, round="nearest")
    assert B.moe_row_capacity(s) == 1000 * 4 + 16 * 128
    assert B.moe_workspace_bytes(B.make_shape(10, 128, 64, 4, 2, tile=100, round="up")) == 0


@pytest.mark.parametrize("T,d,n,E,k", SHAPES_BAD)
def test_invalid_shapes_rejected(lib, T, d, n, E, k):
    s = B.make_shape(T, d, n, E, k)
    assert B.moe_workspace_bytes(s) == 0
    assert B.moe_row_capacity(s) == 0
    p = ctypes.c_void_p(4096)
    assert lib.moe_forward(ctypes.byref(s), p, p, None, p, p, p, p, 1 << 40, None) == B.MOE_ERR_INVALID


def test_forward_a_path_policy(lib):
    """moe_forward gathers rows in the up GEMM's operand load (path 2, wide
    tiles) exactly where the up GEMM has two 256-wide n-blocks (n = 256), else
    it stages them (path 0); an invalid shape gets -1."""
    assert B.moe_forward_a_path(B.make_shape(32768, 1536, 256, 128, 8)) == 2
    for n in (64, 128, 384, 1024, 2048, 14336):
        assert B.moe_forward_a_path(B.make_shape(1024, 512, n, 16, 2)) == 0
    assert B.moe_forward_a_path(B.make_shape(1024, 500, 256, 16, 2)) == -1  # d % 64 != 0


def test_null_and_misaligned_pointers_rejected(lib):
    s = B.make_shape(256, 128, 64, 8, 2)
    p = ctypes.c_void_p(4096)
    odd = ctypes.c_void_p(4096 + 8)
    big = 1 << 40
    assert lib.moe_forward(ctypes.byref(s), None, p, None, p, p, p, p, big, None) == B.MOE_ERR_INVALID
    assert lib.moe_forward(ctypes.byref(s), odd, p, None, p, p, p, p, big, None) == B.MOE_ERR_INVALID
    assert lib.moe_permute(ctypes.byref(s), None, None, p, p, p, p, p, None, p, big, None) == B.MOE_ERR_INVALID
    assert lib.moe_combine(ctypes.byref(s), p, None, None, p, None) == B.MOE_ERR_INVALID
    assert lib.moe_forward_bf16(ctypes.byref(s), None, p, None, p, p, p, p, big, None) == B.MOE_ERR_INVALID
    assert lib.moe_forward_bf16(ctypes.byref(s), p, p, None, p, p, odd, p, big, None) == B.MOE_ERR_INVALID
    assert lib.moe_combine_bf16(ctypes.byref(s), p, None, None, p, None) == B.MOE_ERR_INVALID
    assert lib.moe_combine_bf16(ctypes.byref(s), p, None, p, odd, None) == B.MOE_ERR_INVALID
    assert lib.moe_prepare_weights(ctypes.byref(s), p, p, None, p, p, None) == B.MOE_ERR_INVALID
    assert lib.moe_check_device_status(None, None, None) == B.MOE_ERR_INVALID


def test_small_workspace_rejected(lib):
    s = B.make_shape(256, 128, 64, 8, 2)
    need = B.moe_workspace_bytes(s)
    p = ctypes.c_void_p(4096)
    assert lib.moe_forward(ctypes.byref(s), p, p, None, p, p, p, p, need - 1, None) == B.MOE_ERR_WORKSPACE
    assert lib.moe_forward_bf16(ctypes.byref(s), p, p, None, p, p, p, p, need - 1, None) == B.MOE_ERR_WORKSPACE
    assert lib.moe_permute(ctypes.byref(s), p, None, p, p, p, p, p, None, p, need - 256, None) == B.MOE_ERR_WORKSPACE


def test_rounding_mode_needs_valid_tile(lib):
    s = B.make_shape(256, 128, 64, 8, 2, tile=96, round="nearest")
    p = ctypes.c_void_p(4096)
    assert lib.moe_token_round(ctypes.byref(s), p, p, p, p, p, p, p, p, p, 1 << 40, None) == B.MOE_ERR_INVALID
    s_off = B.make_shape(256, 128, 64, 8, 2)
    assert lib.moe_token_round(ctypes.byref(s_off), p, p, p, p, p, p, p, p, p, 1 << 40, None) == B.MOE_ERR_INVALID


def test_product_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    Wr = torch.zeros(64, 4)
    with pytest.raises(ValueError, match="CUDA"):
        B.moe_router_logits(x, Wr, None, None)


def test_output_buffers_are_checked():
    # the kernels write T*d elements of the entry point's output dtype, so a
    # caller's y of another dtype or shape is refused before any launch
    import torch
    with pytest.raises(ValueError, match="bfloat16"):
        B._buf(torch.zeros(4, 64), (4, 64), torch.bfloat16, "cpu", "y")
    with pytest.raises(ValueError, match="float32"):
        B._buf(torch.zeros(4, 64, dtype=torch.bfloat16), (4, 64), torch.float32, "cpu", "y")
    with pytest.raises(ValueError, match="shape"):
        B._buf(torch.zeros(4, 32), (4, 64), torch.float32, "cpu", "y")
    with pytest.raises(ValueError, match="CUDA"):
        B._buf(torch.zeros(4, 64), (4, 64), torch.float32, "cpu", "y")
    assert B._buf(None, (3, 5), torch.float16, "cpu", "ys").shape == (3, 5)
    with pytest.raises(ValueError, match="dW2"):
        B._buf(torch.zeros(8, 64, 64, dtype=torch.bfloat16), (8, 64, 64), torch.float32, "cpu", "dW2")


def test_backward_workspace_and_host_checks(lib):
    p = ctypes.c_void_p(4096)
    odd = ctypes.c_void_p(4096 + 8)
    s = B.make_shape(256, 128, 64, 8, 2)
    need = B.moe_backward_workspace_bytes(s)
    # the forward's arrays plus at least the padded x, dy, pre-activation and w*h rows
    capp = 256 * 2 + 63 * 8
    assert need >= B.moe_workspace_bytes(s) + capp * (2 * 128 + 2 * 128 + 4 * 64 + 2 * 64)
    args = [p, p, None, p, p, p, p, p, p, None, p, p, p, p]
    assert lib.moe_backward(ctypes.byref(s), *args, need - 1, None) == B.MOE_ERR_WORKSPACE
    assert lib.moe_backward(ctypes.byref(s), *([None] + args[1:]), need, None) == B.MOE_ERR_INVALID
    assert lib.moe_backward(ctypes.byref(s), *([odd] + args[1:]), need, None) == B.MOE_ERR_INVALID
    # unsupported: d not a multiple of 128
    bad = B.make_shape(256, 192, 64, 8, 2)
    assert B.moe_backward_workspace_bytes(bad) == 0
    assert lib.moe_backward(ctypes.byref(bad), *args, 1 << 40, None) == B.MOE_ERR_UNSUPPORTED
    # token rounding: rows up to the rounded capacity
    r = B.make_shape(256, 128, 64, 8, 2, tile=128, round="nearest")
    assert B.moe_backward_workspace_bytes(r) >= B.moe_workspace_bytes(r) + B.moe_row_capacity(r) * 2 * 128 * 2
    assert lib.moe_prepare_weights_bwd(ctypes.byref(s), p, None, p, None) == B.MOE_ERR_INVALID
