"""bf16 output of the combine and of the whole layer (moe_combine_bf16,
moe_forward_bf16): every element is the fp32 result rounded to nearest-even
bf16, bit for bit.  The fp32 layer meets the layer tolerance against the
oracle; the bf16 one adds that one rounding (up to 2^-8 of |y|), which on
outputs beyond about 5 rms can take it past the max-error bound, so its
oracle check allows the rounding on top of the tolerance."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_93_b300 import binding as B
from mixture_experts_layer_93_b300 import inputs as I
from oracle import moe_oracle as O
from tests.moe_testlib import assert_moe_close, err_stats, robust_tokens, to64

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu()


@pytest.mark.parametrize("T,d,k", [(256, 128, 2), (1001, 512, 8), (3, 4096, 1)])
def test_combine_bf16_fixed_k(cuda_device, T, d, k):
    A = T * k
    g = torch.Generator().manual_seed(T + 7)
    ys = torch.randn(A, d, generator=g).to(torch.float16)
    dst = torch.randperm(A, generator=g).to(torch.int32)
    s = B.make_shape(T, d, 64, max(k, 1), k)
    ys_d, dst_d = ys.to(cuda_device), dst.to(cuda_device)
    y16 = B.moe_combine_bf16(s, ys_d, None, dst_d)
    y32 = B.moe_combine(s, ys_d, None, dst_d)
    assert y16.dtype == torch.bfloat16 and y16.shape == (T, d)
    assert torch.equal(_bits(y16), _bits(y32.to(torch.bfloat16)))
    # against the exact sums: the fp32 bound plus half a bf16 ulp (2^-8 relative)
    parts = to64(ys)[dst.numpy().reshape(T, k)]
    ref = parts.sum(axis=1)
    bound = k * 2.0 ** -24 * np.abs(parts).sum(axis=1) * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(ref)
    assert np.all(np.abs(to64(y16) - ref) <= bound)


def test_combine_bf16_csr_with_empty_tokens(cuda_device):
    T, d, R = 50, 256, 120
    g = torch.Generator().manual_seed(5)
    lens = torch.randint(0, 5, (T,), generator=g)
    lens[:3] = 0
    tok_offsets = torch.cat([torch.zeros(1, dtype=torch.int64), lens.cumsum(0)]).to(torch.int32)
    total = int(tok_offsets[-1])
    ys = torch.randn(max(total, R), d, generator=g).to(torch.float16)
    rows = torch.randperm(total, generator=g).to(torch.int32)
    s = B.make_shape(T, d, 64, 8, 2)
    args = (s, ys.to(cuda_device), tok_offsets.to(cuda_device), rows.to(cuda_device))
    y16 = B.moe_combine_bf16(*args)
    y32 = B.moe_combine(*args)
    assert torch.equal(_bits(y16), _bits(y32.to(torch.bfloat16)))
    assert torch.all(y16[:3] == 0)


def test_combine_bf16_rounds_ties_to_even(cuda_device):
    # one row per token, so the fp32 sum is the fp16 value itself; values
    # halfway between two bf16 neighbours (7 stored mantissa bits) go to the
    # one with an even last bit
    vals = [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2 + 2.0 ** -7, 1 + 2.0 ** -8 + 2.0 ** -10]
    want = [1.0, 1 + 2.0 ** -6, -1.0, 2.0, 1 + 2.0 ** -7]
    T, d = len(vals), 64
    ys = torch.tensor(vals, dtype=torch.float64)[:, None].expand(T, d).to(torch.float16).contiguous()
    assert torch.equal(ys[:, 0].double(), torch.tensor(vals, dtype=torch.float64))   # exact in fp16
    rows = torch.arange(T, dtype=torch.int32)
    s = B.make_shape(T, d, 64, 1, 1)
    y16 = B.moe_combine_bf16(s, ys.to(cuda_device), None, rows.to(cuda_device))
    got = y16.double().cpu()
    assert torch.equal(got, torch.tensor(want, dtype=torch.float64)[:, None].expand(T, d))


# the second shape takes the gather in the up GEMM's operand load (n = 256,
# wide tiles); the third rounds each expert's count to the tile
@pytest.mark.parametrize("T,d,n,E,k,tile,mode", [(256, 128, 64, 8, 2, 128, "off"),
                                                 (1024, 512, 256, 8, 2, 128, "off"),
                                                 (2048, 256, 128, 16, 4, 128, "nearest")])
def test_forward_bf16_is_the_rounded_forward(cuda_device, T, d, n, E, k, tile, mode):
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k, bias="zipf" if mode != "off" else None, bias_scale=1.1)
    inp = I.make_inputs(cfg, device=cuda_device, seed=T + n)
    layer = B.MoELayer(inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=k, tile=tile, round=mode)
    y32 = layer.forward(inp["x"]).clone()
    y16 = layer.forward(inp["x"], out_dtype=torch.bfloat16)
    ws = layer.workspace(T, cuda_device)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    assert y16.dtype == torch.bfloat16 and y16.shape == (T, d)
    assert torch.equal(_bits(y16), _bits(y32.to(torch.bfloat16)))
    if mode == "off":
        # the oracle on the tokens whose top-k fp32 rounding cannot decide
        L64 = O.router_logits(inp["x"], inp["Wr"], inp["bias"])
        keep = np.flatnonzero(robust_tokens(L64, k, 1e-4))
        assert keep.size > 0.9 * T
        y_ref = O.moe_forward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=k, tokens=keep)
        sel = torch.from_numpy(keep).to(cuda_device)
        y32, y16 = y32[sel], y16[sel]
    else:
        # the oracle routed on the GPU's fp32 logits (the rounding path keeps them)
        L = ws.view("logits", torch.float32, T * E).view(T, E).cpu().numpy()
        routing = O.route(None, None, None, k, tile=tile, mode=mode, logits=L)
        y_ref = O.moe_forward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=k, tile=tile,
                              mode=mode, routing=routing)
    stats = assert_moe_close(y32, y_ref)
    # bf16: the fp32 layer's error plus the output rounding
    rms = stats["rms"]
    err16 = np.abs(to64(y16) - y_ref)
    assert np.all(err16 <= 2e-2 * rms + 2.0 ** -8 * np.abs(to64(y32))), float(err16.max() / rms)
    assert err_stats(y16, y_ref)["mean_rel"] <= 5e-3


def test_layer_refuses_other_output_dtypes(cuda_device):
    cfg = I.get_config("tiny")
    inp = I.make_inputs(cfg, device=cuda_device, seed=0)
    layer = B.MoELayer(inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=cfg.k)
    with pytest.raises(ValueError, match="out_dtype"):
        layer.forward(inp["x"], out_dtype=torch.float16)
    with pytest.raises(ValueError, match="bfloat16"):
        layer.forward(inp["x"], y=torch.empty(cfg.T, cfg.d, device=cuda_device), out_dtype=torch.bfloat16)
