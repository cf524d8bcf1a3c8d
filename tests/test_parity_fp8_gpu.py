"""Parity of the e4m3 up-projection path against the oracle.

The quantisation decides integers (the e4m3 codes), so it is compared bit for
bit: codes and fp32 scales equal the oracle's.  Given identical codes, the
up-projection is checked like the bf16 one (h within one bf16 rounding of the
fp64 product of the dequantised operands) and the whole layer against the
oracle's FP8 layer within the layer tolerance.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_93_b300 import binding as B
from mixture_experts_layer_93_b300 import inputs as I
from oracle import moe_oracle as O

from moe_testlib import assert_moe_close, err_stats, robust_tokens, to64, valid_topk

pytestmark = pytest.mark.gpu

LOGIT_MARGIN = 1e-4  # fp64 top-k margin below which fp32 logits may pick another valid set


def decode_e4m3(b) -> np.ndarray:
    """Value of each e4m3 byte from the format definition (sign, 4 exponent
    bits with bias 7, 3 mantissa bits; exponent field 0 subnormal; S.1111.111
    NaN)."""
    b = np.asarray(b, dtype=np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    ef, m = (b >> 3) & 15, b & 7
    v = np.where(ef == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (ef - 7))
    v = np.where((ef == 15) & (m == 7), np.nan, v)
    return sign * v


@pytest.mark.parametrize("rows,K", [(64, 128), (300, 4096), (7, 7168), (1, 16)])
def test_quantize_rows_bit_exact(cuda_device, rows, K):
    g = torch.Generator().manual_seed(rows + K)
    X = torch.randn(rows, K, generator=g) * torch.pow(10.0, torch.empty(rows, 1).uniform_(-3, 3, generator=g))
    X[0, :] = 0.0                       # scale 1, codes 0
    if rows > 2:
        X[1, :] = 0.0
        X[1, K // 2] = -3.0             # one nonzero: code -448
    Xb = X.to(torch.bfloat16)
    codes, scales = B.moe_quantize_rows_fp8(Xb.to(cuda_device))
    q_ref, s_ref = O.quantize_rows_e4m3(Xb.float().numpy())
    assert np.array_equal(decode_e4m3(codes.cpu().numpy()), q_ref)
    assert np.array_equal(scales.cpu().numpy().astype(np.float64), s_ref)


def _routing(T, E, k, seed):
    idx = I.make_topk_idx(T, E, k, seed=seed)
    counts, offsets, src, dst = O.permute(idx.numpy(), E)
    return counts, offsets, src, dst


@pytest.mark.parametrize("T,d,n,E,k", [(700, 256, 256, 6, 2), (1000, 384, 128, 3, 1), (300, 128, 256, 8, 2),
                                       (2500, 512, 384, 5, 4)])
def test_expert_up_fp8(cuda_device, T, d, n, E, k):
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k)
    inp = I.make_inputs(cfg, device=cuda_device, seed=T + d + n)
    counts, offsets, src, dst = _routing(T, E, k, seed=T + 5)
    s = B.make_shape(T, d, n, E, k)
    ws = B.Workspace(s, cuda_device)
    W13p, _ = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    W13q, sW13 = B.moe_quantize_rows_fp8(W13p)
    h = B.moe_expert_up_fp8(s, inp["x"], W13q, sW13, torch.from_numpy(counts.astype(np.int32)).to(cuda_device),
                            torch.from_numpy(offsets.astype(np.int32)).to(cuda_device),
                            torch.from_numpy(dst.astype(np.int32)).to(cuda_device), ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    xh = O.dequantized_rows_e4m3(inp["x"])
    A = T * k
    h_gpu = to64(h[:A])
    h_ref = np.zeros((A, n))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            W1h, W3h = O.quantized_expert_weights(inp["W1"][e], inp["W3"][e])
            h_ref[r0:r1] = O.expert_hidden(xh[src[r0:r1] // k], W1h, W3h)
    rms = float(np.sqrt(np.mean(h_ref ** 2)))
    assert np.all(np.abs(h_gpu - h_ref) <= 2.0 ** -8 * np.abs(h_ref) + 1e-5 * rms), err_stats(h_gpu, h_ref)


def test_expert_up_fp8_rejects_unsupported(cuda_device):
    cfg = I.MoEConfig("t", T=64, d=192, n=128, E=2, k=1)
    s = B.make_shape(64, 192, 128, 2, 1)
    ws = B.Workspace(s, cuda_device)
    dummy = torch.zeros(4096, dtype=torch.int32, device=cuda_device)
    x = torch.zeros(64, 192, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(B.MoEError) as info:
        B.moe_expert_up_fp8(s, x, torch.zeros(2, 256, 192, dtype=torch.uint8, device=cuda_device),
                            torch.ones(512, device=cuda_device), dummy, dummy, dummy, ws)
    assert info.value.status == B.MOE_ERR_UNSUPPORTED
    del cfg


@pytest.mark.parametrize("E,d,n", [(3, 256, 128), (8, 512, 256), (1, 128, 128)])
def test_quantize_experts_bit_exact(cuda_device, E, d, n):
    g = torch.Generator().manual_seed(E + d + n)
    W = (torch.randn(E, d, n, generator=g) * torch.pow(10.0, torch.empty(E, 1, 1).uniform_(-2, 2, generator=g)))
    W = W.to(torch.bfloat16)
    codes, scales = B.moe_quantize_experts_fp8(W.to(cuda_device))
    for e in range(E):
        q_ref, s_ref = O.quantize_rows_e4m3(W[e].float().reshape(1, -1).numpy())
        assert np.array_equal(decode_e4m3(codes[e].cpu().numpy().reshape(1, -1)), q_ref)
        assert float(scales[e]) == float(s_ref[0])


@pytest.mark.parametrize("T,d,n,E,k", [(700, 256, 128, 6, 2), (600, 512, 256, 5, 3), (2000, 256, 384, 3, 2)])
def test_expert_down_fp8(cuda_device, T, d, n, E, k):
    """ys = w * (dequantised h row) @ (dequantised W2) within one fp16 rounding:
    the GPU quantises the same bf16 h, so the codes are the oracle's."""
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k)
    inp = I.make_inputs(cfg, device=cuda_device, seed=d + n)
    counts, offsets, src, dst = _routing(T, E, k, seed=T + 2)
    A = T * k
    g = torch.Generator(device="cpu").manual_seed(9)
    s = B.make_shape(T, d, n, E, k)
    ws = B.Workspace(s, cuda_device, fp8=True)
    cap = B.moe_row_capacity(s)
    hcap = torch.zeros(cap, n, dtype=torch.bfloat16)
    hcap[:A] = torch.randn(A, n, generator=g).to(torch.bfloat16)
    wcap = torch.zeros(cap)
    wcap[:A] = torch.rand(A, generator=g)
    _, W2p = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    W2q, sW2 = B.moe_quantize_rows_fp8(W2p)
    ys = B.moe_expert_down_fp8(s, hcap.to(cuda_device), W2q, sW2,
                               torch.from_numpy(counts.astype(np.int32)).to(cuda_device),
                               torch.from_numpy(offsets.astype(np.int32)).to(cuda_device), wcap.to(cuda_device), ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    hh = O.dequantized_rows_e4m3(hcap[:A].float().numpy())
    ref = np.zeros((A, d))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            ref[r0:r1] = wcap[r0:r1].double().numpy()[:, None] * (hh[r0:r1] @ O.quantized_expert_down_weight(
                inp["W2"][e]))
    got = to64(ys[:A])
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.abs(got - ref) <= 2.0 ** -11 * np.abs(ref) + 1e-5 * rms), err_stats(got, ref)


def test_expert_down_fp8_outlier_channel(cuda_device):
    """W2 with planted outlier output channels (10^4 times the others): with
    one scale per output channel the other channels keep e4m3 precision, and
    ys stays within one fp16 rounding of the oracle's product."""
    T, d, n, E, k = 600, 256, 128, 4, 2
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k)
    inp = I.make_inputs(cfg, device=cuda_device, seed=31)
    W2 = inp["W2"].float()
    W2[:, :, 17] *= 1e4
    W2[2, :, 200] *= 1e4
    W2 = W2.to(torch.bfloat16)
    counts, offsets, src, dst = _routing(T, E, k, seed=5)
    A = T * k
    g = torch.Generator(device="cpu").manual_seed(10)
    s = B.make_shape(T, d, n, E, k)
    ws = B.Workspace(s, cuda_device, fp8=True)
    cap = B.moe_row_capacity(s)
    hcap = torch.zeros(cap, n, dtype=torch.bfloat16)
    hcap[:A] = (torch.randn(A, n, generator=g) * 0.1).to(torch.bfloat16)   # keeps ys in fp16 range
    wcap = torch.zeros(cap)
    wcap[:A] = torch.rand(A, generator=g)
    _, W2p = B.moe_prepare_weights(inp["W1"], inp["W3"], W2)
    W2q, sW2 = B.moe_quantize_rows_fp8(W2p)
    ys = B.moe_expert_down_fp8(s, hcap.to(cuda_device), W2q, sW2,
                               torch.from_numpy(counts.astype(np.int32)).to(cuda_device),
                               torch.from_numpy(offsets.astype(np.int32)).to(cuda_device), wcap.to(cuda_device), ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    hh = O.dequantized_rows_e4m3(hcap[:A].float().numpy())
    ref = np.zeros((A, d))
    exact = np.zeros((A, d))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            wr = wcap[r0:r1].double().numpy()[:, None]
            ref[r0:r1] = wr * (hh[r0:r1] @ O.quantized_expert_down_weight(W2[e]))
            exact[r0:r1] = wr * (hh[r0:r1] @ to64(W2[e]))
    got = to64(ys[:A])
    mag = np.abs(ref)
    assert np.all(np.abs(got - ref) <= 2.0 ** -11 * mag + 1e-5 * np.sqrt(np.mean(ref ** 2, axis=0))[None, :])
    # the ordinary channels stay close to the unquantised weights
    others = np.setdiff1d(np.arange(d), [17, 200])
    rel = np.abs(got[:, others] - exact[:, others]).sum() / np.abs(exact[:, others]).sum()
    assert rel < 0.1, rel


def _forward_fp8_and_check(cfg, dev, seed=0, tokens=None):
    inp = I.make_inputs(cfg, device=dev, seed=seed)
    s = B.make_shape(cfg.T, cfg.d, cfg.n, cfg.E, cfg.k)
    ws = B.Workspace(s, dev, fp8=True)
    W13p, W2p = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    W13q, sW13 = B.moe_quantize_rows_fp8(W13p)
    W2q, sW2 = B.moe_quantize_rows_fp8(W2p)
    del W13p, W2p
    y = B.moe_forward_fp8(s, inp["x"], inp["Wr"], inp["bias"], W13q, sW13, W2q, sW2, ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    T = cfg.T
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    x_s = inp["x"][torch.from_numpy(toks).to(dev)]
    L64 = O.router_logits(x_s, inp["Wr"], inp["bias"])
    gpu_idx = ws.view("topk_idx", torch.int32, T * cfg.k).view(T, cfg.k)[torch.from_numpy(toks).to(dev)]
    gpu_idx = gpu_idx.cpu().numpy()
    robust = robust_tokens(L64, cfg.k, LOGIT_MARGIN)
    for i in np.flatnonzero(~robust):
        assert valid_topk(L64[i], gpu_idx[i], LOGIT_MARGIN), i
    keep = toks[robust]
    y_ref = O.moe_forward_fp8_full(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=cfg.k,
                                   tokens=keep)
    y_gpu = y[torch.from_numpy(keep).to(dev)]
    stats = assert_moe_close(y_gpu, y_ref)
    # and how far the FP8 layer lies from the bf16 one (reported, not a bound)
    y_bf = O.moe_forward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=cfg.k, tokens=keep)
    return stats, err_stats(y_gpu, y_bf), float(robust.mean())


@pytest.mark.parametrize("T,d,n,E,k", [(256, 256, 128, 8, 2), (1000, 256, 256, 16, 4), (777, 512, 128, 5, 5)])
def test_forward_fp8(cuda_device, T, d, n, E, k):
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k)
    stats, vs_bf16, frac = _forward_fp8_and_check(cfg, cuda_device, seed=T + E)
    assert frac > 0.9
    assert vs_bf16["max_err"] < 0.5 * vs_bf16["rms"]   # FP8 stays close to the bf16 layer


@pytest.mark.slow
def test_forward_fp8_full_size_sampled(cuda_device):
    cfg = I.get_config("mixtral")
    rng = np.random.default_rng(2)
    toks = np.sort(rng.choice(cfg.T, size=48, replace=False))
    stats, vs_bf16, frac = _forward_fp8_and_check(cfg, cuda_device, tokens=toks)
    assert frac > 0.9
    torch.cuda.empty_cache()
