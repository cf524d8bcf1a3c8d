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
