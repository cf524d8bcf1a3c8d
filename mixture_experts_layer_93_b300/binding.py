"""ctypes binding of libmoe.so (declared in include/moe.h).

Argument marshalling only: torch allocates device memory and supplies the
current stream; every step of the layer runs in the library's CUDA kernels.
There is no CPU fallback: if the library is missing or a call fails, an
exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID = 1
MOE_ERR_CUDA = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_UNSUPPORTED = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_CHECK = 6

ROUND_MODES = {"off": 0, "nearest": 1, "up": 2, "stochastic": 3}

# workspace_layout slots
WS_SLOTS = ["logits", "topk_idx", "topk_w", "counts", "offsets", "src", "dst", "row_token", "row_w",
            "tok_offsets", "tok_rows", "h", "ys"]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str, detail: int | None = None):
        self.status = status
        self.detail = detail
        msg = f"{where}: {status_string(status)} (status {status})"
        if detail is not None:
            msg += f", detail {detail}"
        super().__init__(msg)


class moe_shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("n", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("tile", ctypes.c_int32), ("round", ctypes.c_int32),
                ("seed", ctypes.c_uint32)]


_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_I = ctypes.c_int
_SHP = ctypes.POINTER(moe_shape)

_SIGNATURES = {
    "moe_row_capacity": (ctypes.c_int64, [_SHP]),
    "moe_workspace_bytes": (_SZ, [_SHP]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_check_device_status": (_I, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
    "moe_clear_device_status": (_I, [_P, _P]),
    "moe_prepare_weights": (_I, [_SHP, _P, _P, _P, _P, _P, _P]),
    "moe_router_logits": (_I, [_SHP, _P, _P, _P, _P, _P, _P]),
    "moe_topk_gating": (_I, [_SHP, _P, _P, _P, _P, _P]),
    "moe_route": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_permute": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_route_permute": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_quantize_rows_fp8": (_I, [_P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P]),
    "moe_expert_up_fp8": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_fp8": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_quantize_experts_fp8": (_I, [_P, ctypes.c_int32, ctypes.c_int64, _P, _P, _P]),
    "moe_expert_down_fp8": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_workspace_bytes_fp8": (_SZ, [_SHP]),
    "moe_permute_noalloc": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_token_round": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_up": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _SZ, _P]),
    "moe_expert_down": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_combine": (_I, [_SHP, _P, _P, _P, _P, _P]),
    "moe_combine_bf16": (_I, [_SHP, _P, _P, _P, _P, _P]),
    "moe_forward": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_bf16": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_a_path": (_I, [_SHP]),
    "moe_workspace_layout": (_I, [_SHP, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32]),
    "moe_selftest_timeout": (_I, [_P, ctypes.c_uint64, _P]),
    "moe_backward_workspace_bytes": (_SZ, [_SHP]),
    "moe_prepare_weights_bwd": (_I, [_SHP, _P, _P, _P, _P]),
    "moe_backward": (_I, [_SHP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
}

_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """Load libmoe.so (built in-tree by `python -m mixture_experts_layer_93_b300.build`)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                       "`python -m mixture_experts_layer_93_b300.build`")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in _SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def make_shape(T, d, n, E, k, tile=128, round="off", seed=0) -> moe_shape:
    mode = ROUND_MODES[round] if isinstance(round, str) else int(round)
    return moe_shape(int(T), int(d), int(n), int(E), int(k), int(tile), mode, int(seed) & 0xFFFFFFFF)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(device=None) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoEError(status, where)


def _buf(t, dims, dtype, device, what: str):
    """An output buffer: a new one, or the caller's after checking its shape
    and dtype (the kernels write every element of `dims` in that dtype)."""
    dims = tuple(int(v) for v in dims)
    if t is None:
        return torch.empty(dims, dtype=dtype, device=device)
    if t.dtype != dtype or tuple(t.shape) != dims:
        raise ValueError(f"{what} must be {dtype} of shape {dims}, not {t.dtype} {tuple(t.shape)}")
    _need_cuda(t)
    return t


def _need_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("libmoe works on CUDA tensors only (no CPU fallback)")
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous")


def moe_row_capacity(shape: moe_shape) -> int:
    return int(lib().moe_row_capacity(ctypes.byref(shape)))


def moe_workspace_bytes(shape: moe_shape) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(shape)))


def moe_workspace_layout(shape: moe_shape) -> dict:
    arr = (ctypes.c_int64 * len(WS_SLOTS))()
    _check(lib().moe_workspace_layout(ctypes.byref(shape), arr, len(WS_SLOTS)), "moe_workspace_layout")
    return {name: int(arr[i]) for i, name in enumerate(WS_SLOTS)}


class Workspace:
    """Device workspace for one shape (status block zeroed at creation)."""

    def __init__(self, shape: moe_shape, device="cuda", fp8: bool = False, backward: bool = False):
        if backward:
            nbytes = moe_backward_workspace_bytes(shape)
        else:
            nbytes = moe_workspace_bytes_fp8(shape) if fp8 else moe_workspace_bytes(shape)
        if nbytes == 0:
            raise MoEError(MOE_ERR_INVALID, "moe_workspace_bytes")
        self.shape = shape
        self.nbytes = nbytes
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.buf[:256].zero_()

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    def view(self, slot: str, dtype, numel: int) -> torch.Tensor:
        off = moe_workspace_layout(self.shape)[slot]
        esz = torch.tensor([], dtype=dtype).element_size()
        return self.buf[off:off + numel * esz].view(dtype)


def moe_check_device_status(ws: Workspace, raise_on_error: bool = True) -> int:
    detail = ctypes.c_int32(0)
    st = lib().moe_check_device_status(ws.ptr, ctypes.byref(detail), _stream(ws.buf.device))
    if st != MOE_OK and raise_on_error:
        raise MoEError(st, "device status", detail.value)
    return st


def moe_clear_device_status(ws: Workspace):
    _check(lib().moe_clear_device_status(ws.ptr, _stream(ws.buf.device)), "moe_clear_device_status")


def moe_prepare_weights(W1, W3, W2):
    """Repack W1/W3 [E,d,n] and W2 [E,n,d] into (W13p [E,2n,d], W2p [E,d,n])."""
    _need_cuda(W1, W3, W2)
    E, d, n = W1.shape
    shape = make_shape(1, d, n, E, 1)
    W13p = torch.empty(E, 2 * n, d, dtype=torch.bfloat16, device=W1.device)
    W2p = torch.empty(E, d, n, dtype=torch.bfloat16, device=W1.device)
    _check(lib().moe_prepare_weights(ctypes.byref(shape), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(W13p), _ptr(W2p),
                                     _stream(W1.device)), "moe_prepare_weights")
    return W13p, W2p


def moe_router_logits(x, Wr, bias, ws: Workspace):
    _need_cuda(x, Wr, bias)
    T, d = x.shape
    E = Wr.shape[1]
    shape = make_shape(T, d, 64, E, 1)
    logits = torch.empty(T, E, dtype=torch.float32, device=x.device)
    _check(lib().moe_router_logits(ctypes.byref(shape), _ptr(x), _ptr(Wr), _ptr(bias), _ptr(logits),
                                   ws.ptr, _stream(x.device)), "moe_router_logits")
    return logits


def moe_topk_gating(logits, k: int, ws: Workspace):
    _need_cuda(logits)
    T, E = logits.shape
    shape = make_shape(T, 64, 64, E, k)
    idx = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    _check(lib().moe_topk_gating(ctypes.byref(shape), _ptr(logits), _ptr(idx), _ptr(w), ws.ptr,
                                 _stream(logits.device)), "moe_topk_gating")
    return idx, w


def moe_route(x, Wr, bias, k: int, ws: Workspace):
    _need_cuda(x, Wr, bias)
    T, d = x.shape
    E = Wr.shape[1]
    shape = make_shape(T, d, 64, E, k)
    logits = torch.empty(T, E, dtype=torch.float32, device=x.device)
    idx = torch.empty(T, k, dtype=torch.int32, device=x.device)
    w = torch.empty(T, k, dtype=torch.float32, device=x.device)
    _check(lib().moe_route(ctypes.byref(shape), _ptr(x), _ptr(Wr), _ptr(bias), _ptr(logits), _ptr(idx), _ptr(w),
                           ws.ptr, _stream(x.device)), "moe_route")
    return logits, idx, w


def moe_permute(shape: moe_shape, topk_idx, topk_w, ws: Workspace) -> dict:
    _need_cuda(topk_idx, topk_w)
    dev = topk_idx.device
    A = shape.T * shape.k
    cap = moe_row_capacity(shape)
    out = {
        "counts": torch.empty(shape.E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(shape.E + 1, dtype=torch.int32, device=dev),
        "src": torch.empty(cap, dtype=torch.int32, device=dev),
        "dst": torch.empty(A, dtype=torch.int32, device=dev),
        "row_token": torch.empty(cap, dtype=torch.int32, device=dev),
        "row_w": torch.empty(cap, dtype=torch.float32, device=dev),
    }
    _check(lib().moe_permute(ctypes.byref(shape), _ptr(topk_idx), _ptr(topk_w), _ptr(out["counts"]),
                             _ptr(out["offsets"]), _ptr(out["src"]), _ptr(out["dst"]), _ptr(out["row_token"]),
                             _ptr(out["row_w"]) if topk_w is not None else None, ws.ptr, ws.nbytes,
                             _stream(dev)), "moe_permute")
    return out


def moe_route_permute(shape: moe_shape, x, Wr, bias, ws: Workspace) -> dict:
    """Fused route + permutation: logits, top-k indices and weights, and the
    permutation arrays (as moe_route then moe_permute)."""
    _need_cuda(x, Wr, bias)
    dev = x.device
    T, E, k = shape.T, shape.E, shape.k
    A = T * k
    cap = moe_row_capacity(shape)
    out = {
        "logits": torch.empty(T, E, dtype=torch.float32, device=dev),
        "idx": torch.empty(T, k, dtype=torch.int32, device=dev),
        "w": torch.empty(T, k, dtype=torch.float32, device=dev),
        "counts": torch.empty(E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "src": torch.empty(cap, dtype=torch.int32, device=dev),
        "dst": torch.empty(A, dtype=torch.int32, device=dev),
        "row_token": torch.empty(cap, dtype=torch.int32, device=dev),
        "row_w": torch.empty(cap, dtype=torch.float32, device=dev),
    }
    _check(lib().moe_route_permute(ctypes.byref(shape), _ptr(x), _ptr(Wr), _ptr(bias), _ptr(out["logits"]),
                                   _ptr(out["idx"]), _ptr(out["w"]), _ptr(out["counts"]), _ptr(out["offsets"]),
                                   _ptr(out["src"]), _ptr(out["dst"]), _ptr(out["row_token"]), _ptr(out["row_w"]),
                                   ws.ptr, ws.nbytes, _stream(dev)), "moe_route_permute")
    return out


def moe_quantize_rows_fp8(src):
    """(codes uint8 [rows, K], scales fp32 [rows]) of a bf16 [rows, K] tensor
    (any leading shape is flattened into rows)."""
    _need_cuda(src)
    src = src.contiguous()
    K = src.shape[-1]
    rows = src.numel() // K
    codes = torch.empty(src.shape, dtype=torch.uint8, device=src.device)
    scales = torch.empty(src.shape[:-1], dtype=torch.float32, device=src.device)
    _check(lib().moe_quantize_rows_fp8(_ptr(src), rows, K, _ptr(codes), _ptr(scales), _stream(src.device)),
           "moe_quantize_rows_fp8")
    return codes, scales


def moe_expert_up_fp8(shape: moe_shape, x, W13q, sW13, counts, offsets, tok_rows, ws: Workspace,
                      tok_offsets=None, h=None):
    _need_cuda(x, W13q, sW13, counts, offsets, tok_rows, tok_offsets)
    h = _buf(h, (moe_row_capacity(shape), shape.n), torch.bfloat16, x.device, "h")
    _check(lib().moe_expert_up_fp8(ctypes.byref(shape), _ptr(x), _ptr(W13q), _ptr(sW13), _ptr(counts),
                                   _ptr(offsets), _ptr(tok_offsets), _ptr(tok_rows), _ptr(h), ws.ptr, ws.nbytes,
                                   _stream(x.device)), "moe_expert_up_fp8")
    return h


def moe_quantize_experts_fp8(src):
    """(codes uint8, scales fp32 [E]) of a bf16 [E, ...] tensor with one scale
    per expert (leading dimension)."""
    _need_cuda(src)
    src = src.contiguous()
    E = src.shape[0]
    m = src.numel() // E
    codes = torch.empty(src.shape, dtype=torch.uint8, device=src.device)
    scales = torch.empty(E, dtype=torch.float32, device=src.device)
    _check(lib().moe_quantize_experts_fp8(_ptr(src), E, m, _ptr(codes), _ptr(scales), _stream(src.device)),
           "moe_quantize_experts_fp8")
    return codes, scales


def moe_workspace_bytes_fp8(shape: moe_shape) -> int:
    return int(lib().moe_workspace_bytes_fp8(ctypes.byref(shape)))


def moe_expert_down_fp8(shape: moe_shape, h, W2q, sW2, counts, offsets, row_w, ws: Workspace, ys=None):
    _need_cuda(h, W2q, sW2, counts, offsets, row_w)
    ys = _buf(ys, (moe_row_capacity(shape), shape.d), torch.float16, h.device, "ys")
    _check(lib().moe_expert_down_fp8(ctypes.byref(shape), _ptr(h), _ptr(W2q), _ptr(sW2), _ptr(counts), _ptr(offsets),
                                     _ptr(row_w), _ptr(ys), ws.ptr, ws.nbytes, _stream(h.device)),
           "moe_expert_down_fp8")
    return ys


def moe_forward_fp8(shape: moe_shape, x, Wr, bias, W13q, sW13, W2q, sW2, ws: Workspace, y=None):
    _need_cuda(x, Wr, bias, W13q, sW13, W2q, sW2)
    y = _buf(y, (shape.T, shape.d), torch.float32, x.device, "y")
    _check(lib().moe_forward_fp8(ctypes.byref(shape), _ptr(x), _ptr(Wr), _ptr(bias), _ptr(W13q), _ptr(sW13),
                                 _ptr(W2q), _ptr(sW2), _ptr(y), ws.ptr, ws.nbytes, _stream(x.device)),
           "moe_forward_fp8")
    return y


def moe_token_round(shape: moe_shape, logits, topk_idx, ws: Workspace) -> dict:
    _need_cuda(logits, topk_idx)
    dev = logits.device
    cap = moe_row_capacity(shape)
    out = {
        "counts": torch.empty(shape.E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(shape.E + 1, dtype=torch.int32, device=dev),
        "row_token": torch.empty(cap, dtype=torch.int32, device=dev),
        "row_w": torch.empty(cap, dtype=torch.float32, device=dev),
        "tok_offsets": torch.empty(shape.T + 1, dtype=torch.int32, device=dev),
        "tok_rows": torch.empty(cap, dtype=torch.int32, device=dev),
    }
    _check(lib().moe_token_round(ctypes.byref(shape), _ptr(logits), _ptr(topk_idx), _ptr(out["counts"]),
                                 _ptr(out["offsets"]), _ptr(out["row_token"]), _ptr(out["row_w"]),
                                 _ptr(out["tok_offsets"]), _ptr(out["tok_rows"]), ws.ptr, ws.nbytes,
                                 _stream(dev)), "moe_token_round")
    return out


def moe_expert_up(shape: moe_shape, x, W13p, counts, offsets, row_token, ws: Workspace, gather: int = 2,
                  h=None, tok_offsets=None, tok_rows=None):
    _need_cuda(x, W13p, counts, offsets, row_token, tok_offsets, tok_rows)
    h = _buf(h, (moe_row_capacity(shape), shape.n), torch.bfloat16, x.device, "h")
    _check(lib().moe_expert_up(ctypes.byref(shape), _ptr(x), _ptr(W13p), _ptr(counts), _ptr(offsets),
                               _ptr(row_token), _ptr(tok_offsets), _ptr(tok_rows), _ptr(h), int(gather), ws.ptr,
                               ws.nbytes, _stream(x.device)), "moe_expert_up")
    return h


def moe_expert_down(shape: moe_shape, h, W2p, counts, offsets, row_w, ws: Workspace, ys=None):
    _need_cuda(h, W2p, counts, offsets, row_w)
    ys = _buf(ys, (moe_row_capacity(shape), shape.d), torch.float16, h.device, "ys")
    _check(lib().moe_expert_down(ctypes.byref(shape), _ptr(h), _ptr(W2p), _ptr(counts), _ptr(offsets),
                                 _ptr(row_w), _ptr(ys), ws.ptr, ws.nbytes, _stream(h.device)), "moe_expert_down")
    return ys


def moe_combine(shape: moe_shape, ys, tok_offsets, tok_rows, y=None):
    _need_cuda(ys, tok_offsets, tok_rows)
    y = _buf(y, (shape.T, shape.d), torch.float32, ys.device, "y")
    _check(lib().moe_combine(ctypes.byref(shape), _ptr(ys), _ptr(tok_offsets), _ptr(tok_rows), _ptr(y),
                             _stream(ys.device)), "moe_combine")
    return y


def moe_combine_bf16(shape: moe_shape, ys, tok_offsets, tok_rows, y=None):
    """moe_combine with y bf16: the fp32 sum rounded to nearest-even."""
    _need_cuda(ys, tok_offsets, tok_rows)
    y = _buf(y, (shape.T, shape.d), torch.bfloat16, ys.device, "y")
    _check(lib().moe_combine_bf16(ctypes.byref(shape), _ptr(ys), _ptr(tok_offsets), _ptr(tok_rows), _ptr(y),
                                  _stream(ys.device)), "moe_combine_bf16")
    return y


def moe_forward_a_path(shape: moe_shape) -> int:
    """The A-operand path (moe_expert_up's `gather`) moe_forward uses for the shape."""
    return int(lib().moe_forward_a_path(ctypes.byref(shape)))


def moe_forward(shape: moe_shape, x, Wr, bias, W13p, W2p, ws: Workspace, y=None):
    _need_cuda(x, Wr, bias, W13p, W2p)
    y = _buf(y, (shape.T, shape.d), torch.float32, x.device, "y")
    _check(lib().moe_forward(ctypes.byref(shape), _ptr(x), _ptr(Wr), _ptr(bias), _ptr(W13p), _ptr(W2p), _ptr(y),
                             ws.ptr, ws.nbytes, _stream(x.device)), "moe_forward")
    return y


def moe_forward_bf16(shape: moe_shape, x, Wr, bias, W13p, W2p, ws: Workspace, y=None):
    """moe_forward with y bf16: its fp32 y rounded to nearest-even."""
    _need_cuda(x, Wr, bias, W13p, W2p)
    y = _buf(y, (shape.T, shape.d), torch.bfloat16, x.device, "y")
    _check(lib().moe_forward_bf16(ctypes.byref(shape), _ptr(x), _ptr(Wr), _ptr(bias), _ptr(W13p), _ptr(W2p),
                                  _ptr(y), ws.ptr, ws.nbytes, _stream(x.device)), "moe_forward_bf16")
    return y


def moe_backward_workspace_bytes(shape: moe_shape) -> int:
    return int(lib().moe_backward_workspace_bytes(ctypes.byref(shape)))


def moe_prepare_weights_bwd(W1, W3):
    """W13i [E, d, 2n]: W1 and W3 interleaved along their last dimension."""
    _need_cuda(W1, W3)
    E, d, n = W1.shape
    shape = make_shape(1, d, n, E, 1)
    W13i = torch.empty(E, d, 2 * n, dtype=torch.bfloat16, device=W1.device)
    _check(lib().moe_prepare_weights_bwd(ctypes.byref(shape), _ptr(W1), _ptr(W3), _ptr(W13i), _stream(W1.device)),
           "moe_prepare_weights_bwd")
    return W13i


def moe_backward(shape: moe_shape, x, Wr, bias, W13p, W13i, W2, dy, ws: Workspace, want_dbias: bool = True,
                 out=None) -> dict:
    """Gradients {dx, dWr, dbias, dW1, dW3, dW2} (fp32) of sum <dy, y>; dy bf16 [T, d]."""
    _need_cuda(x, Wr, bias, W13p, W13i, W2, dy)
    dev = x.device
    T, d, n, E = shape.T, shape.d, shape.n, shape.E
    # the caller's buffers (checked), or new ones; dbias is skipped when the
    # caller's dict holds None for it, or has no entry and want_dbias is off
    given = out or {}
    dims = {"dx": (T, d), "dWr": (d, E), "dbias": (E,), "dW1": (E, d, n), "dW3": (E, d, n), "dW2": (E, n, d)}
    skip_dbias = given["dbias"] is None if "dbias" in given else not want_dbias
    out = {key: None if key == "dbias" and skip_dbias else _buf(given.get(key), dims[key], torch.float32, dev, key)
           for key in dims}
    _check(lib().moe_backward(ctypes.byref(shape), _ptr(x), _ptr(Wr), _ptr(bias), _ptr(W13p), _ptr(W13i), _ptr(W2),
                              _ptr(dy), _ptr(out["dx"]), _ptr(out["dWr"]), _ptr(out.get("dbias")), _ptr(out["dW1"]),
                              _ptr(out["dW3"]), _ptr(out["dW2"]), ws.ptr, ws.nbytes, _stream(dev)), "moe_backward")
    return out


def moe_selftest_timeout(ws: Workspace, timeout_ns: int):
    _check(lib().moe_selftest_timeout(ws.ptr, int(timeout_ns), _stream(ws.buf.device)), "moe_selftest_timeout")


class MoELayer:
    """One MoE layer with its weights packed once and a reusable workspace."""

    def __init__(self, Wr, bias, W1, W3, W2, k: int, tile: int = 128, round: str = "off", seed: int = 0):
        self.E, self.d, self.n = W1.shape
        self.k, self.tile, self.round, self.seed = k, tile, round, seed
        self.Wr = Wr.contiguous()
        self.bias = bias.contiguous() if bias is not None else None
        self.W13p, self.W2p = moe_prepare_weights(W1.contiguous(), W3.contiguous(), W2.contiguous())
        self.W13i = None          # backward only: W1/W3 interleaved, built on the first backward
        self._W1, self._W3, self._W2 = W1, W3, W2
        self._ws = {}
        self._bws = {}

    def shape(self, T: int) -> moe_shape:
        return make_shape(T, self.d, self.n, self.E, self.k, self.tile, self.round, self.seed)

    def workspace(self, T: int, device) -> Workspace:
        key = (T, str(device))
        if key not in self._ws:
            self._ws[key] = Workspace(self.shape(T), device)
        return self._ws[key]

    def forward(self, x, y=None, out_dtype=torch.float32):
        """y = the layer applied to x, in fp32 or (out_dtype bf16) rounded to bf16."""
        T = x.shape[0]
        ws = self.workspace(T, x.device)
        if out_dtype == torch.bfloat16:
            return moe_forward_bf16(self.shape(T), x, self.Wr, self.bias, self.W13p, self.W2p, ws, y)
        if out_dtype != torch.float32:
            raise ValueError(f"out_dtype must be torch.float32 or torch.bfloat16, not {out_dtype}")
        return moe_forward(self.shape(T), x, self.Wr, self.bias, self.W13p, self.W2p, ws, y)

    __call__ = forward

    def backward_workspace(self, T: int, device) -> Workspace:
        key = (T, str(device))
        if key not in self._bws:
            self._bws[key] = Workspace(self.shape(T), device, backward=True)
        return self._bws[key]

    def backward(self, x, dy) -> dict:
        """Gradients of sum <dy, forward(x)>: {dx, dWr, dbias, dW1, dW3, dW2}
        (fp32), by recomputation (moe_backward); dy bf16 [T, d]."""
        if self.W13i is None:
            self.W13i = moe_prepare_weights_bwd(self._W1.contiguous(), self._W3.contiguous())
        T = x.shape[0]
        ws = self.backward_workspace(T, x.device)
        return moe_backward(self.shape(T), x, self.Wr, self.bias, self.W13p, self.W13i, self._W2.contiguous(), dy,
                            ws, want_dbias=self.bias is not None)
