"""The Python binding's marshalling, on the host: with the compute entry
points replaced by a recorder (the library's host-only queries stay real),
each wrapper allocates its outputs with the shapes and dtypes the C ABI
writes, refuses a caller's buffer of another shape or dtype before calling
the library, and passes the stream and workspace through."""
import ctypes
import types

import pytest
import torch

from mixture_experts_layer_93_b300 import binding as B
from mixture_experts_layer_93_b300 import build as BUILD

HOST_ONLY = {"moe_row_capacity", "moe_workspace_bytes", "moe_workspace_bytes_fp8", "moe_backward_workspace_bytes",
             "moe_forward_a_path", "moe_status_string", "moe_workspace_layout"}


class Recorder:
    """Stands in for libmoe.so: compute entry points record their call and
    return MOE_OK; host-only queries go to the real library."""

    def __init__(self, real):
        self.real = real
        self.calls = []

    def __getattr__(self, name):
        if name in HOST_ONLY:
            return getattr(self.real, name)

        def call(*args):
            self.calls.append((name, args))
            return B.MOE_OK
        return call


@pytest.fixture()
def rec(monkeypatch):
    BUILD.build()
    r = Recorder(B.lib())
    monkeypatch.setattr(B, "lib", lambda: r)
    monkeypatch.setattr(B, "_need_cuda", lambda *ts: None)
    monkeypatch.setattr(B, "_stream", lambda device=None: None)
    return r


def _ws():
    return types.SimpleNamespace(ptr=ctypes.c_void_p(4096), nbytes=1 << 20, buf=torch.empty(1))


SHAPE = dict(T=40, d=128, n=64, E=8, k=2)


def _shape():
    return B.make_shape(SHAPE["T"], SHAPE["d"], SHAPE["n"], SHAPE["E"], SHAPE["k"])


def test_stage_wrappers_allocate_what_the_abi_writes(rec):
    s = _shape()
    T, d, n, k = s.T, s.d, s.n, s.k
    cap = B.moe_row_capacity(s)
    assert cap >= T * k
    x = torch.zeros(T, d, dtype=torch.bfloat16)
    i32 = torch.zeros(8, dtype=torch.int32)
    h = B.moe_expert_up(s, x, x, i32, i32, i32, _ws())
    assert h.shape == (cap, n) and h.dtype == torch.bfloat16
    ys = B.moe_expert_down(s, h, x, i32, i32, torch.zeros(cap), _ws())
    assert ys.shape == (cap, d) and ys.dtype == torch.float16
    y = B.moe_combine(s, ys, None, i32)
    assert y.shape == (T, d) and y.dtype == torch.float32
    y16 = B.moe_combine_bf16(s, ys, None, i32)
    assert y16.shape == (T, d) and y16.dtype == torch.bfloat16
    assert [c[0] for c in rec.calls] == ["moe_expert_up", "moe_expert_down", "moe_combine", "moe_combine_bf16"]


def test_forward_wrappers_allocate_and_check_y(rec):
    s = _shape()
    x = torch.zeros(s.T, s.d, dtype=torch.bfloat16)
    w = torch.zeros(4)
    assert B.moe_forward(s, x, w, None, x, x, _ws()).dtype == torch.float32
    assert B.moe_forward_bf16(s, x, w, None, x, x, _ws()).dtype == torch.bfloat16
    assert B.moe_forward_fp8(s, x, w, None, x, w, x, w, _ws()).shape == (s.T, s.d)
    y_given = torch.empty(s.T, s.d)
    assert B.moe_forward(s, x, w, None, x, x, _ws(), y_given) is y_given
    n_calls = len(rec.calls)
    for fn, bad in [(B.moe_forward, torch.empty(s.T, s.d, dtype=torch.bfloat16)),
                    (B.moe_forward_bf16, torch.empty(s.T, s.d)),
                    (B.moe_forward, torch.empty(s.T + 1, s.d))]:
        with pytest.raises(ValueError, match="y must be"):
            fn(s, x, w, None, x, x, _ws(), bad)
    with pytest.raises(ValueError, match="y must be"):
        B.moe_forward_fp8(s, x, w, None, x, w, x, w, _ws(), torch.empty(s.T, s.d, dtype=torch.bfloat16))
    assert len(rec.calls) == n_calls   # refused before the library was called


def test_stage_wrappers_refuse_wrong_buffers(rec):
    s = _shape()
    cap = B.moe_row_capacity(s)
    x = torch.zeros(s.T, s.d, dtype=torch.bfloat16)
    i32 = torch.zeros(8, dtype=torch.int32)
    with pytest.raises(ValueError, match="h must be"):
        B.moe_expert_up(s, x, x, i32, i32, i32, _ws(), h=torch.empty(cap, s.n, dtype=torch.float16))
    with pytest.raises(ValueError, match="ys must be"):
        B.moe_expert_down(s, x, x, i32, i32, torch.zeros(cap), _ws(), ys=torch.empty(cap, s.d, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="h must be"):
        B.moe_expert_up_fp8(s, x, x, x, i32, i32, i32, _ws(), h=torch.empty(cap - 1, s.n, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="ys must be"):
        B.moe_expert_down_fp8(s, x, x, x, i32, i32, x, _ws(), ys=torch.empty(cap, s.d))
    assert rec.calls == []


def test_backward_outputs_and_dbias(rec):
    s = _shape()
    T, d, n, E = s.T, s.d, s.n, s.E
    x = torch.zeros(T, d, dtype=torch.bfloat16)
    out = B.moe_backward(s, x, x, None, x, x, x, x, _ws())
    want = {"dx": (T, d), "dWr": (d, E), "dbias": (E,), "dW1": (E, d, n), "dW3": (E, d, n), "dW2": (E, n, d)}
    for key, dims in want.items():
        assert out[key].shape == dims and out[key].dtype == torch.float32, key
    assert B.moe_backward(s, x, x, None, x, x, x, x, _ws(), want_dbias=False)["dbias"] is None
    # a caller's dict: its buffers are used as given; None for dbias skips it
    given = {key: torch.empty(dims) for key, dims in want.items()}
    given["dbias"] = None
    got = B.moe_backward(s, x, x, None, x, x, x, x, _ws(), out=given)
    assert got["dbias"] is None and all(got[key] is given[key] for key in want if key != "dbias")
    name, args = rec.calls[-1]
    assert name == "moe_backward" and args[10] is None          # the dbias pointer
    bad = dict(given, dW2=torch.empty(E, d, n))                   # transposed
    n_calls = len(rec.calls)
    with pytest.raises(ValueError, match="dW2 must be"):
        B.moe_backward(s, x, x, None, x, x, x, x, _ws(), out=bad)
    assert len(rec.calls) == n_calls


def test_layer_forward_dtype_choice(rec, monkeypatch):
    # MoELayer without weight packing: only the forward's dispatch is under test
    layer = B.MoELayer.__new__(B.MoELayer)
    layer.E, layer.d, layer.n, layer.k, layer.tile, layer.round, layer.seed = 8, 128, 64, 2, 128, "off", 0
    layer.Wr = layer.bias = layer.W13p = layer.W2p = torch.zeros(4)
    layer._ws = {}
    monkeypatch.setattr(B.MoELayer, "workspace", lambda self, T, device: _ws())
    x = torch.zeros(40, 128, dtype=torch.bfloat16)
    assert layer.forward(x).dtype == torch.float32
    assert layer.forward(x, out_dtype=torch.bfloat16).dtype == torch.bfloat16
    assert [c[0] for c in rec.calls] == ["moe_forward", "moe_forward_bf16"]
    with pytest.raises(ValueError, match="out_dtype"):
        layer.forward(x, out_dtype=torch.float16)
