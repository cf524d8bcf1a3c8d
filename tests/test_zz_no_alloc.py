"""moe_permute_noalloc: the permutation for callers that may not allocate
device memory (an engine that owns every device byte and forbids cudaMalloc
while it runs).  Its histograms live in a fixed array inside the library; its
results must equal moe_permute's, call after call.

Kept in its own file, collected last, so a failure here cannot stop the rest
of the GPU suite from running first."""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_93_b300 import binding as B
from mixture_experts_layer_93_b300 import inputs as I

pytestmark = pytest.mark.gpu


def _outputs(T, E, k, dev):
    A = T * k
    return {"counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
            "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
            "src": torch.full((A,), -7, dtype=torch.int32, device=dev),
            "dst": torch.full((A,), -7, dtype=torch.int32, device=dev),
            "row_token": torch.full((A,), -7, dtype=torch.int32, device=dev),
            "row_w": torch.full((A,), -7.0, dtype=torch.float32, device=dev)}


def _noalloc(shape, idx, w, out, dev):
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = B.lib().moe_permute_noalloc(ctypes.byref(shape), P(idx), P(w), P(out["counts"]), P(out["offsets"]),
                                     P(out["src"]), P(out["dst"]), P(out["row_token"]), P(out["row_w"]),
                                     ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    assert st == B.MOE_OK, B.status_string(st)
    torch.cuda.synchronize(dev)


@pytest.mark.parametrize("T,E,k,skew", [(4099, 256, 8, 1.5), (777, 8, 2, 0.0)])
def test_noalloc_permute_matches_workspace_permute_twice(cuda_device, T, E, k, skew):
    dev = cuda_device
    s = B.make_shape(T, 64, 64, E, k)
    ws = B.Workspace(s, dev)
    A = T * k
    for call in range(2):
        # a different routing on each call: the second call must not see the
        # first call's histograms
        idx = I.make_topk_idx(T, E, k, seed=100 * call + T, skew=skew).to(dev)
        w = I.make_gate_weights(T, k, seed=call).to(dev)
        ref = B.moe_permute(s, idx, w, ws)
        assert B.moe_check_device_status(ws) == B.MOE_OK
        out = _outputs(T, E, k, dev)
        _noalloc(s, idx, w, out, dev)
        for name in ("counts", "offsets", "dst"):
            assert torch.equal(out[name], ref[name]), (call, name)
        for name in ("src", "row_token"):
            assert torch.equal(out[name], ref[name][:A]), (call, name)
        assert torch.equal(out["row_w"], ref["row_w"][:A]), call


def test_noalloc_rejects_shapes_beyond_its_array(cuda_device):
    # E * ceil(T*k/2048) = 1024 * 257 > 262144
    s = B.make_shape(65793, 64, 64, 1024, 8)
    dummy = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    P = ctypes.c_void_p(dummy.data_ptr())
    st = B.lib().moe_permute_noalloc(ctypes.byref(s), P, None, P, P, P, P, P, None, None)
    assert st == B.MOE_ERR_WORKSPACE


def test_noalloc_accepts_a_shape_exactly_at_its_limit(cuda_device):
    # E * ceil(T*k / 2048) = 128 * 2048 = 262144: the array is filled exactly
    dev = cuda_device
    T, E, k = 2048 * 2048 // 8, 128, 8
    s = B.make_shape(T, 64, 64, E, k)
    ws = B.Workspace(s, dev)
    idx = I.make_topk_idx(T, E, k, device=dev, seed=7)
    w = I.make_gate_weights(T, k, device=dev, seed=7)
    ref = B.moe_permute(s, idx, w, ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    out = _outputs(T, E, k, dev)
    _noalloc(s, idx, w, out, dev)
    A = T * k
    for name in ("counts", "offsets", "dst"):
        assert torch.equal(out[name], ref[name]), name
    for name in ("src", "row_token", "row_w"):
        assert torch.equal(out[name], ref[name][:A]), name


def _check(res, what):
    err = res[0] if isinstance(res, tuple) else res
    assert int(err) == 0, f"{what}: CUresult {int(err)}"
    return res[1] if isinstance(res, tuple) and len(res) == 2 else res


def test_noalloc_from_a_second_context(cuda_device):
    """A caller that runs in a CUDA context of its own (created through the
    driver API, as an engine embedding this library may do) must get the
    scratch array's address in that context, not the primary context's."""
    from cuda.bindings import driver as drv

    dev = cuda_device
    T, E, k = 3001, 64, 4
    A = T * k
    idx = I.make_topk_idx(T, E, k, seed=11, skew=1.2)
    w = I.make_gate_weights(T, k, seed=11)
    # the reference, computed entirely in the primary context (torch's)
    s = B.make_shape(T, 64, 64, E, k)
    ws = B.Workspace(s, dev)
    ref = {kk: v.cpu().numpy() for kk, v in B.moe_permute(s, idx.to(dev), w.to(dev), ws).items()}
    torch.cuda.synchronize(dev)
    idx_h = np.ascontiguousarray(idx.numpy())
    w_h = np.ascontiguousarray(w.numpy())
    sizes = {"counts": E, "offsets": E + 1, "src": A, "dst": A, "row_token": A, "row_w": A}
    got = {name: np.full(n, -7, dtype=np.float32 if name == "row_w" else np.int32) for name, n in sizes.items()}

    # no torch call below until the context is destroyed: while it is
    # current, runtime calls on this thread go to it
    _check(drv.cuInit(0), "cuInit")
    cu_dev = _check(drv.cuDeviceGet(dev.index if dev.index is not None else 0), "cuDeviceGet")
    ctx = _check(drv.cuCtxCreate(None, 0, cu_dev), "cuCtxCreate")
    bufs = {}
    try:
        for name, arr in (("idx", idx_h), ("w", w_h)):
            bufs[name] = _check(drv.cuMemAlloc(arr.nbytes), "cuMemAlloc")
            _check(drv.cuMemcpyHtoD(bufs[name], arr.ctypes.data, arr.nbytes), "cuMemcpyHtoD")
        for name, arr in got.items():
            bufs[name] = _check(drv.cuMemAlloc(arr.nbytes), "cuMemAlloc")
        P = lambda name: ctypes.c_void_p(int(bufs[name]))  # noqa: E731
        for _ in range(2):
            st = B.lib().moe_permute_noalloc(ctypes.byref(s), P("idx"), P("w"), P("counts"), P("offsets"), P("src"),
                                             P("dst"), P("row_token"), P("row_w"), None)
            assert st == B.MOE_OK, B.status_string(st)
            _check(drv.cuCtxSynchronize(), "cuCtxSynchronize")
        for name, arr in got.items():
            _check(drv.cuMemcpyDtoH(arr.ctypes.data, bufs[name], arr.nbytes), "cuMemcpyDtoH")
    finally:
        for b in bufs.values():
            drv.cuMemFree(b)
        drv.cuCtxDestroy(ctx)
    for name in ("counts", "offsets", "dst"):
        assert np.array_equal(got[name], ref[name]), name
    for name in ("src", "row_token", "row_w"):
        assert np.array_equal(got[name], ref[name][:A]), name
