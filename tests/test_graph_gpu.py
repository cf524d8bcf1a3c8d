"""The layer's entry points are CUDA-graph capturable: every launch is
asynchronous on the caller's stream, nothing allocates or synchronises, and a
replayed graph gives the eager results bit for bit (a serving loop can
replay one graph per batch shape)."""
import pytest
import torch

from mixture_experts_layer_93_b300 import binding as B
from mixture_experts_layer_93_b300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,round", [("tiny", "off"), ("tiny", "nearest")])
def test_forward_graph_replay_matches_eager(cuda_device, name, round):
    cfg = I.get_config(name)
    inp = I.make_inputs(cfg, device=cuda_device, seed=1)
    s = B.make_shape(cfg.T, cfg.d, cfg.n, cfg.E, cfg.k, tile=64, round=round)
    W13p, W2p = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    ws = B.Workspace(s, cuda_device)
    x = inp["x"].clone()
    y = torch.empty(cfg.T, cfg.d, dtype=torch.float32, device=cuda_device)
    side = torch.cuda.Stream(cuda_device)
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(side):   # warm-up off the capture (one-time attribute setting)
        B.moe_forward(s, x, inp["Wr"], inp["bias"], W13p, W2p, ws, y)
    torch.cuda.current_stream(cuda_device).wait_stream(side)
    torch.cuda.synchronize()
    eager = y.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.moe_forward(s, x, inp["Wr"], inp["bias"], W13p, W2p, ws, y)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert B.moe_check_device_status(ws) == B.MOE_OK
    assert torch.equal(y, eager)
    # new inputs through the same graph: x is read at replay time
    x.copy_(torch.flip(inp["x"], dims=[0]))
    g.replay()
    torch.cuda.synchronize()
    ref = B.moe_forward(s, x, inp["Wr"], inp["bias"], W13p, W2p, ws)
    assert torch.equal(y, ref)


def test_backward_graph_replay_matches_eager(cuda_device):
    cfg = I.MoEConfig("t", T=300, d=256, n=128, E=6, k=2, bias="normal", bias_scale=0.5)
    inp = I.make_inputs(cfg, device=cuda_device, seed=2)
    dy = torch.randn(cfg.T, cfg.d, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).to(cuda_device)
    s = B.make_shape(cfg.T, cfg.d, cfg.n, cfg.E, cfg.k)
    W13p, _ = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    W13i = B.moe_prepare_weights_bwd(inp["W1"], inp["W3"])
    ws = B.Workspace(s, cuda_device, backward=True)
    out = B.moe_backward(s, inp["x"], inp["Wr"], inp["bias"], W13p, W13i, inp["W2"], dy, ws)
    torch.cuda.synchronize()
    eager = {key: v.clone() for key, v in out.items()}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.moe_backward(s, inp["x"], inp["Wr"], inp["bias"], W13p, W13i, inp["W2"], dy, ws, out=out)
    for v in out.values():
        v.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert B.moe_check_device_status(ws) == B.MOE_OK
    for key, v in out.items():
        assert torch.equal(v, eager[key]), key
