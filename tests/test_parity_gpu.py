"""Parity of the CUDA path (through the C ABI) against the fp64 oracle.

Every input comes from the seeded generators; every expected value from the
oracle.  Integer outputs must match exactly; floating-point outputs meet the
bf16 / fp32-accumulation tolerance in moe_testlib."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_93_b300 import binding as B
from mixture_experts_layer_93_b300 import inputs as I
from oracle import moe_oracle as O
from tests.moe_testlib import assert_moe_close, err_stats, robust_tokens, stratified_tokens, to64, valid_topk

pytestmark = pytest.mark.gpu

LOGIT_MARGIN = 1e-4


def ws_for(T, d, n, E, k, dev, tile=128, round="off"):
    s = B.make_shape(T, d, n, E, k, tile, round)
    return s, B.Workspace(s, dev)


# ------------------------------------------------------------------ router
# E <= 16 runs the SIMT router while Wr (fp32) and its x staging fit in
# shared memory (d <= 4160 at E <= 8, d <= 2816 at E <= 16), larger shapes
# the tensor-core one: both sides of both limits, E not a multiple of 8,
# token counts that leave a partial warp task
@pytest.mark.parametrize("T,d,E,bias", [(256, 128, 8, False), (1000, 512, 40, True), (300, 1024, 256, True),
                                        (77, 64, 1, False), (130, 256, 1024, False), (1, 64, 16, True),
                                        (99, 192, 5, True), (517, 1536, 12, True), (258, 2816, 16, False),
                                        (333, 4096, 8, True), (130, 4160, 8, False), (64, 4224, 8, True),
                                        (70, 2880, 16, False), (45, 3200, 3, True)])
def test_router_logits(cuda_device, T, d, E, bias):
    cfg = I.MoEConfig("t", T=T, d=d, n=64, E=E, k=1, bias="normal" if bias else None, bias_scale=0.5)
    inp = I.make_inputs(cfg, device=cuda_device, seed=T + E, weights=False)
    s, ws = ws_for(T, d, 64, E, 1, cuda_device)
    L = B.moe_router_logits(inp["x"], inp["Wr"], inp["bias"], ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    torch.cuda.synchronize()
    _assert_logits_bound(L, inp["x"], inp["Wr"], inp["bias"], d)


def test_router_logits_unaligned_wr(cuda_device):
    """A Wr that does not start on 16 bytes (fp32 alignment only), under the
    same bound."""
    T, d, E = 200, 256, 8
    cfg = I.MoEConfig("t", T=T, d=d, n=64, E=E, k=1, bias="normal", bias_scale=0.5)
    inp = I.make_inputs(cfg, device=cuda_device, seed=5, weights=False)
    buf = torch.empty(d * E + 1, dtype=torch.float32, device=cuda_device)
    Wr = buf[1:].view(d, E)
    Wr.copy_(inp["Wr"])
    assert Wr.data_ptr() % 16 != 0
    s, ws = ws_for(T, d, 64, E, 1, cuda_device)
    L = B.moe_router_logits(inp["x"], Wr, inp["bias"], ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    torch.cuda.synchronize()
    _assert_logits_bound(L, inp["x"], inp["Wr"], inp["bias"], d)


def _assert_logits_bound(L, x, Wr, bias, d):
    L64 = O.router_logits(x, Wr, bias)
    err = np.abs(to64(L) - L64)
    # rigorous bound for an fp32-accumulated dot product of 3d exact terms
    # (the tensor-core router: hi/mid/lo split of Wr, each product exact),
    # rounding toward zero allowed: (3d + 3) * 2^-23 * sum_i |x_i w_ie|, plus
    # the split residue 2^-27.  The SIMT router (d fused multiply-adds in
    # chains of d/32, then a 32-way butterfly) stays far inside it.
    absdot = np.abs(to64(x)) @ np.abs(to64(Wr))
    assert np.all(err <= (3 * d + 3) * 2.0 ** -23 * (absdot + np.abs(L64)) + 1e-30)
    rms = float(np.sqrt(np.mean(L64 ** 2)))
    assert err.max() <= 5e-5 * rms, (err.max(), rms)


# -------------------------------------------------------------------- top-k
@pytest.mark.parametrize("E,k", [(1, 1), (7, 2), (8, 2), (32, 8), (33, 5), (64, 8), (128, 8), (256, 8),
                                 (1024, 32), (20, 20)])
def test_topk_gating_identical_logits(cuda_device, E, k):
    T = 777
    L = I.make_logits(T, E, device="cpu", seed=E * 31 + k, ties=True)
    s, ws = ws_for(T, 64, 64, E, k, cuda_device)
    idx, w = B.moe_topk_gating(L.to(cuda_device), k, ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    ref_idx = O.topk(L.numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    ref_w = O.gate_weights(L.numpy(), ref_idx)
    assert np.abs(to64(w) - ref_w).max() <= 2e-6


def test_topk_nan_is_reported(cuda_device):
    T, E, k = 64, 16, 2
    L = I.make_logits(T, E, seed=5, ties=False)
    L[3, 7] = float("nan")
    s, ws = ws_for(T, 64, 64, E, k, cuda_device)
    idx, _ = B.moe_topk_gating(L.to(cuda_device), k, ws)
    assert B.moe_check_device_status(ws, raise_on_error=False) == B.MOE_ERR_DEVICE_CHECK
    assert 7 not in idx[3].tolist()


# -------------------------------------------------------------- permutation
@pytest.mark.parametrize("T,E,k,skew", [(1, 1, 1, 0.0), (777, 8, 2, 0.0), (3001, 64, 8, 1.2), (5000, 128, 8, 0.0),
                                        (4099, 256, 8, 2.0), (999, 1024, 32, 0.0), (40, 3, 3, 0.0)])
def test_permute_bit_exact(cuda_device, T, E, k, skew):
    idx = I.make_topk_idx(T, E, k, seed=T * 7 + E, skew=skew)
    w = I.make_gate_weights(T, k, seed=T)
    s, ws = ws_for(T, 64, 64, E, k, cuda_device)
    out = B.moe_permute(s, idx.to(cuda_device), w.to(cuda_device), ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    counts, offsets, src, dst = O.permute(idx.numpy(), E)
    A = T * k
    assert np.array_equal(out["counts"].cpu().numpy(), counts)
    assert np.array_equal(out["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(out["src"][:A].cpu().numpy(), src)
    assert np.array_equal(out["dst"].cpu().numpy(), dst)
    assert np.array_equal(out["row_token"][:A].cpu().numpy(), src // k)
    assert torch.equal(out["row_w"][:A].cpu(), w.reshape(-1)[torch.from_numpy(src)])


# ------------------------------------------------------- fused route+permute
@pytest.mark.parametrize("T,d,E,k,bias", [(1, 128, 1, 1, False), (777, 256, 8, 2, True), (1500, 128, 40, 3, False),
                                          (999, 1024, 12, 4, True), (2049, 2816, 16, 8, False),
                                          (513, 4096, 8, 2, True), (301, 4224, 8, 2, False),
                                          (5000, 256, 128, 8, False), (3001, 128, 256, 5, True),
                                          (700, 128, 256, 6, False), (333, 128, 300, 7, True),
                                          (4096, 128, 64, 1, False), (600, 128, 64, 12, False),
                                          (500, 128, 200, 16, True), (777, 256, 16, 12, True),
                                          (500, 128, 12, 10, False), (300, 192, 9, 9, True)])
def test_route_permute_fused_matches_separate(cuda_device, T, d, E, k, bias):
    """moe_route_permute equals moe_route then moe_permute bit for bit (every
    output), matches the oracle's top-k and permutation on the same fp32
    logits, and gives the same bits when called again.  k = 3, 5, 6, 7 put
    tokens across the 2048-assignment chunk boundaries; E = 300 takes the
    unfused path; k = 12 and 16 (k > 8) take the top-k + histogram kernel
    instead of the router epilogue, also behind the SIMT router (E <= 16)."""
    cfg = I.MoEConfig("t", T=T, d=d, n=64, E=E, k=k, bias="normal" if bias else None, bias_scale=0.3)
    inp = I.make_inputs(cfg, device=cuda_device, seed=T + E + k, weights=False)
    s, ws = ws_for(T, d, 64, E, k, cuda_device)
    fused = B.moe_route_permute(s, inp["x"], inp["Wr"], inp["bias"], ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    again = B.moe_route_permute(s, inp["x"], inp["Wr"], inp["bias"], ws)
    logits, idx, w = B.moe_route(inp["x"], inp["Wr"], inp["bias"], k, ws)
    sep = B.moe_permute(s, idx, w, ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    A = T * k
    pairs = [("logits", logits), ("idx", idx), ("w", w)] + [(n, sep[n]) for n in
                                                             ("counts", "offsets", "dst")]
    pairs += [(n, sep[n][:A]) for n in ("src", "row_token", "row_w")]
    for name, ref in pairs:
        got = fused[name] if name in ("logits", "idx", "w", "counts", "offsets", "dst") else fused[name][:A]
        got2 = again[name] if name in ("logits", "idx", "w", "counts", "offsets", "dst") else again[name][:A]
        assert torch.equal(got, ref), name
        assert torch.equal(got2, ref), name
    L = fused["logits"].cpu().numpy()
    ref_idx = O.topk(L, k)
    assert np.array_equal(fused["idx"].cpu().numpy(), ref_idx)
    assert np.abs(to64(fused["w"]) - O.gate_weights(L, ref_idx)).max() <= 2e-6
    counts, offsets, src, dst = O.permute(ref_idx, E)
    assert np.array_equal(fused["counts"].cpu().numpy(), counts)
    assert np.array_equal(fused["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(fused["src"][:A].cpu().numpy(), src)
    assert np.array_equal(fused["dst"].cpu().numpy(), dst)


@pytest.mark.parametrize("E", [16, 64])  # the SIMT router, the tensor-core router's epilogue
def test_route_permute_fused_reports_nan(cuda_device, E):
    T, d, k = 300, 128, 2
    cfg = I.MoEConfig("t", T=T, d=d, n=64, E=E, k=k)
    inp = I.make_inputs(cfg, device=cuda_device, seed=3, weights=False)
    x = inp["x"].clone()
    x[5, 7] = float("nan")
    s, ws = ws_for(T, d, 64, E, k, cuda_device)
    B.moe_clear_device_status(ws)
    out = B.moe_route_permute(s, x, inp["Wr"], inp["bias"], ws)
    assert B.moe_check_device_status(ws, raise_on_error=False) == B.MOE_ERR_DEVICE_CHECK
    assert int(out["offsets"][E]) == T * k
    B.moe_clear_device_status(ws)


def _synthetic_routing(T, E, k, seed, skew=0.0):
    idx = I.make_topk_idx(T, E, k, seed=seed, skew=skew)
    counts, offsets, src, dst = O.permute(idx.numpy(), E)
    return idx, counts, offsets, src, dst


# ---------------------------------------------------------- weight repack
@pytest.mark.parametrize("E,d,n", [(3, 128, 64), (2, 192, 320), (1, 64, 128)])
def test_prepare_weights_layout(cuda_device, E, d, n):
    """W13p row 2j = W1[:, j]^T, row 2j+1 = W3[:, j]^T; W2p = W2^T (bit copies)."""
    g = torch.Generator(device="cpu").manual_seed(E * 1000 + d + n)
    W1 = torch.randn(E, d, n, generator=g).to(torch.bfloat16)
    W3 = torch.randn(E, d, n, generator=g).to(torch.bfloat16)
    W2 = torch.randn(E, n, d, generator=g).to(torch.bfloat16)
    W13p, W2p = B.moe_prepare_weights(W1.to(cuda_device), W3.to(cuda_device), W2.to(cuda_device))
    W13p, W2p = W13p.cpu(), W2p.cpu()
    assert W13p.shape == (E, 2 * n, d) and W2p.shape == (E, d, n)
    assert torch.equal(W13p[:, 0::2, :], W1.transpose(1, 2))
    assert torch.equal(W13p[:, 1::2, :], W3.transpose(1, 2))
    assert torch.equal(W2p, W2.transpose(1, 2))


# ------------------------------------------------------------ up-projection
@pytest.mark.parametrize("gather", [0, 1, 2, "0-token", "0-offsets"])
@pytest.mark.parametrize("T,d,n,E,k,skew", [(700, 256, 192, 6, 2, 0.0), (600, 384, 256, 5, 3, 1.0),
                                            (300, 128, 64, 8, 2, 0.0), (1100, 512, 128, 3, 1, 0.5)])
def test_expert_up_swiglu(cuda_device, gather, T, d, n, E, k, skew):
    """gather "0-token" copies rows in token order from dst; "0-offsets" the
    same through explicit per-token offsets (k rows each)."""
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k)
    inp = I.make_inputs(cfg, device=cuda_device, seed=T + d + n)
    idx, counts, offsets, src, dst = _synthetic_routing(T, E, k, seed=T + 1, skew=skew)
    s, ws = ws_for(T, d, n, E, k, cuda_device)
    W13p, W2p = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    row_token = torch.from_numpy((src // k).astype(np.int32)).to(cuda_device)
    tok_offsets = tok_rows = None
    if isinstance(gather, str):
        tok_rows = torch.from_numpy(dst.astype(np.int32)).to(cuda_device)
        if gather == "0-offsets":
            tok_offsets = torch.arange(0, T * k + 1, k, dtype=torch.int32, device=cuda_device)
        gather = 0
    h = B.moe_expert_up(s, inp["x"], W13p, torch.from_numpy(counts.astype(np.int32)).to(cuda_device),
                        torch.from_numpy(offsets.astype(np.int32)).to(cuda_device), row_token, ws, gather=gather,
                        tok_offsets=tok_offsets, tok_rows=tok_rows)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    A = T * k
    h_gpu = to64(h[:A])
    h_ref = np.zeros((A, n))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            h_ref[r0:r1] = O.expert_hidden(inp["x"][torch.from_numpy(src[r0:r1] // k).to(cuda_device)],
                                           inp["W1"][e], inp["W3"][e])
    # h is a bf16 intermediate: within one bf16 rounding (2^-8 relative) of
    # the exact value, plus fp32 accumulation noise
    rms = float(np.sqrt(np.mean(h_ref ** 2)))
    assert np.all(np.abs(h_gpu - h_ref) <= 2.0 ** -8 * np.abs(h_ref) + 1e-5 * rms), err_stats(h_gpu, h_ref)


# Per-expert counts whose last 128-row block takes sizes across 1..128 rows,
# with odd and even block counts.  Plus 0 (about 200 rows per expert) the SM
# pairs run super tiles and the odd last blocks the separate single-SM launch;
# plus 800 (about 1000 rows per expert) super tiles with the odd last block in
# the last unit; plus 1024 plain pair tiles with odd blocks as half-empty
# pairs.
ODD_COUNTS = [1, 31, 32, 33, 64, 95, 97, 128, 129, 160, 255, 256, 257, 300, 383, 384, 0, 450]


def _routing_with_counts(counts, seed):
    """k = 1 routing whose expert e gets exactly counts[e] tokens (shuffled)."""
    g = np.random.default_rng(seed)
    idx = np.repeat(np.arange(len(counts)), counts)
    g.shuffle(idx)
    idx = torch.from_numpy(idx.astype(np.int32)).reshape(-1, 1)
    c, offsets, src, dst = O.permute(idx.numpy(), len(counts))
    assert list(c) == list(counts)
    return idx, c, offsets, src, dst


@pytest.mark.parametrize("gather", [0, 2])
@pytest.mark.parametrize("extra", [0, 800, 1024])
def test_expert_up_odd_tails(cuda_device, extra, gather):
    """Up GEMM on SM pairs (n % 128 == 0) with odd last blocks of every size:
    h within one bf16 rounding.  gather 2 (rows gathered by cp.async) runs
    wide tiles, both n-blocks of n = 256 against one gathered row block."""
    counts = [c + extra for c in ODD_COUNTS]
    T, d, n, E, k = sum(counts), 256, 256, len(counts), 1
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k)
    inp = I.make_inputs(cfg, device=cuda_device, seed=11)
    idx, c, offsets, src, dst = _routing_with_counts(counts, seed=5)
    s, ws = ws_for(T, d, n, E, k, cuda_device)
    W13p, W2p = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    row_token = torch.from_numpy((src // k).astype(np.int32)).to(cuda_device)
    h = B.moe_expert_up(s, inp["x"], W13p, torch.from_numpy(c.astype(np.int32)).to(cuda_device),
                        torch.from_numpy(offsets.astype(np.int32)).to(cuda_device), row_token, ws, gather=gather,
                        tok_rows=torch.from_numpy(dst.astype(np.int32)).to(cuda_device) if gather == 0 else None)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    h_gpu = to64(h[:T])
    h_ref = np.zeros((T, n))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            h_ref[r0:r1] = O.expert_hidden(inp["x"][torch.from_numpy(src[r0:r1] // k).to(cuda_device)],
                                           inp["W1"][e], inp["W3"][e])
    rms = float(np.sqrt(np.mean(h_ref ** 2)))
    assert np.all(np.abs(h_gpu - h_ref) <= 2.0 ** -8 * np.abs(h_ref) + 1e-5 * rms), err_stats(h_gpu, h_ref)


@pytest.mark.parametrize("extra", [0, 800, 1024])
def test_expert_down_odd_tails(cuda_device, extra):
    """Down GEMM on SM pairs (d % 256 == 0) with odd last blocks of every
    size: ys within one fp16 rounding, gate weight applied per row."""
    counts = [c + extra for c in ODD_COUNTS]
    T, d, n, E, k = sum(counts), 512, 128, len(counts), 1
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k)
    inp = I.make_inputs(cfg, device=cuda_device, seed=12)
    idx, c, offsets, src, dst = _routing_with_counts(counts, seed=6)
    g = torch.Generator(device="cpu").manual_seed(13)
    h = torch.randn(T, n, generator=g).to(torch.bfloat16).to(cuda_device)
    row_w = torch.rand(T, generator=g).to(cuda_device)
    s, ws = ws_for(T, d, n, E, k, cuda_device)
    W13p, W2p = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    cap = B.moe_row_capacity(s)
    hcap = torch.zeros(cap, n, dtype=torch.bfloat16, device=cuda_device)
    hcap[:T] = h
    wcap = torch.zeros(cap, device=cuda_device)
    wcap[:T] = row_w
    ys = B.moe_expert_down(s, hcap, W2p, torch.from_numpy(c.astype(np.int32)).to(cuda_device),
                           torch.from_numpy(offsets.astype(np.int32)).to(cuda_device), wcap, ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    ref = np.zeros((T, d))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            ref[r0:r1] = to64(row_w[r0:r1])[:, None] * O.expert_out(h[r0:r1], inp["W2"][e])
    got = to64(ys[:T])
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.abs(got - ref) <= 2.0 ** -11 * np.abs(ref) + 1e-5 * rms), err_stats(got, ref)


# ---------------------------------------------------------- down-projection
# the last two: more than 1024 rows per expert and K = n over 32 k-blocks
# with two 256-wide n-blocks, which run as wide tiles (odd last blocks in
# the pairs), with a ragged last block
@pytest.mark.parametrize("T,d,n,E,k", [(700, 320, 128, 6, 2), (600, 384, 192, 5, 3), (500, 512, 64, 7, 2),
                                       (256, 128, 64, 8, 2), (3000, 512, 2176, 2, 1), (2601, 512, 2112, 2, 2)])
def test_expert_down_gate_weight(cuda_device, T, d, n, E, k):
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k)
    inp = I.make_inputs(cfg, device=cuda_device, seed=d + n)
    idx, counts, offsets, src, dst = _synthetic_routing(T, E, k, seed=T + 2)
    A = T * k
    g = torch.Generator(device="cpu").manual_seed(9)
    h = torch.randn(A, n, generator=g).to(torch.bfloat16).to(cuda_device)
    row_w = torch.rand(A, generator=g).to(cuda_device)
    s, ws = ws_for(T, d, n, E, k, cuda_device)
    W13p, W2p = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    hcap = torch.zeros(B.moe_row_capacity(s), n, dtype=torch.bfloat16, device=cuda_device)
    hcap[:A] = h
    wcap = torch.zeros(B.moe_row_capacity(s), device=cuda_device)
    wcap[:A] = row_w
    ys = B.moe_expert_down(s, hcap, W2p, torch.from_numpy(counts.astype(np.int32)).to(cuda_device),
                           torch.from_numpy(offsets.astype(np.int32)).to(cuda_device), wcap, ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    ref = np.zeros((A, d))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            ref[r0:r1] = to64(row_w[r0:r1])[:, None] * O.expert_out(h[r0:r1], inp["W2"][e])
    # ys is an fp16 intermediate: within one fp16 rounding (2^-11 relative)
    got = to64(ys[:A])
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.abs(got - ref) <= 2.0 ** -11 * np.abs(ref) + 1e-5 * rms), err_stats(got, ref)


def test_expert_down_fp16_saturation(cuda_device):
    """Rows whose w * (h W2) leaves the fp16 range are stored as +-65504 and
    reported (MOE_ERR_DEVICE_CHECK, detail 16); the other rows are unaffected."""
    T, d, n, E, k = 300, 256, 128, 4, 2
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k)
    inp = I.make_inputs(cfg, device=cuda_device, seed=5)
    idx, counts, offsets, src, dst = _synthetic_routing(T, E, k, seed=3)
    A = T * k
    g = torch.Generator(device="cpu").manual_seed(4)
    h = torch.randn(A, n, generator=g).to(torch.bfloat16).to(cuda_device)
    row_w = torch.rand(A, generator=g) * 0.5 + 0.5
    big = torch.zeros(A, dtype=torch.bool)
    big[::37] = True                       # these rows overflow: |acc| ~ 1 times 1e6
    row_w[big] *= 1e6
    row_w = row_w.to(cuda_device)
    s, ws = ws_for(T, d, n, E, k, cuda_device)
    W13p, W2p = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    cap = B.moe_row_capacity(s)
    hcap = torch.zeros(cap, n, dtype=torch.bfloat16, device=cuda_device)
    hcap[:A] = h
    wcap = torch.zeros(cap, device=cuda_device)
    wcap[:A] = row_w
    B.moe_clear_device_status(ws)
    ys = B.moe_expert_down(s, hcap, W2p, torch.from_numpy(counts.astype(np.int32)).to(cuda_device),
                           torch.from_numpy(offsets.astype(np.int32)).to(cuda_device), wcap, ws)
    with pytest.raises(B.MoEError) as info:
        B.moe_check_device_status(ws)
    assert info.value.status == B.MOE_ERR_DEVICE_CHECK and info.value.detail == 16
    ref = np.zeros((A, d))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            ref[r0:r1] = to64(row_w[r0:r1])[:, None] * O.expert_out(h[r0:r1], inp["W2"][e])
    got = to64(ys[:A])
    over = np.abs(ref) > 65520.0           # rounds past the largest fp16 value
    assert over.any() and big.numpy()[np.nonzero(over)[0]].all()
    assert np.array_equal(got[over], np.sign(ref[over]) * 65504.0)
    inside = np.abs(ref) < 65000.0
    # fp32 accumulation error scales with the row's gate weight: floor per row
    row_rms = np.broadcast_to(np.sqrt(np.mean(ref ** 2, axis=1))[:, None], ref.shape)
    assert np.all(np.abs(got[inside] - ref[inside]) <= 2.0 ** -11 * np.abs(ref[inside]) + 1e-5 * row_rms[inside])
    B.moe_clear_device_status(ws)


# ------------------------------------------------------------------ combine
@pytest.mark.parametrize("T,d,k", [(256, 128, 2), (1001, 512, 8), (3, 4096, 1)])
def test_combine_fixed_k(cuda_device, T, d, k):
    A = T * k
    g = torch.Generator().manual_seed(T)
    ys = torch.randn(A, d, generator=g).to(torch.float16)
    dst = torch.randperm(A, generator=g).to(torch.int32)
    s = B.make_shape(T, d, 64, max(k, 1), k)
    y = B.moe_combine(s, ys.to(cuda_device), None, dst.to(cuda_device))
    parts = to64(ys)[dst.numpy().reshape(T, k)]
    ref = parts.sum(axis=1)
    diff = np.abs(to64(y) - ref)
    # fp32 sum of k terms: k * 2^-24 * sum |terms|
    assert np.all(diff <= k * 2.0 ** -24 * np.abs(parts).sum(axis=1))


def test_combine_csr_with_empty_tokens(cuda_device):
    T, d, R = 50, 256, 120
    g = torch.Generator().manual_seed(1)
    lens = torch.randint(0, 5, (T,), generator=g)
    lens[:3] = 0
    lens[-1] = R - int(lens[:-1].sum()) if int(lens[:-1].sum()) < R else 0
    tok_offsets = torch.cat([torch.zeros(1, dtype=torch.int64), lens.cumsum(0)]).to(torch.int32)
    total = int(tok_offsets[-1])
    ys = torch.randn(max(total, 1), d, generator=g).to(torch.float16)
    rows = torch.randperm(total, generator=g).to(torch.int32)
    s = B.make_shape(T, d, 64, 8, 2)
    y = B.moe_combine(s, ys.to(cuda_device), tok_offsets.to(cuda_device), rows.to(cuda_device))
    y64 = to64(y)
    for t in range(T):
        r = rows[tok_offsets[t]:tok_offsets[t + 1]].numpy()
        ref = to64(ys)[r].sum(axis=0) if r.size else np.zeros(d)
        bound = len(r) * 2.0 ** -24 * np.abs(to64(ys)[r]).sum(axis=0) if r.size else 0.0
        assert np.all(np.abs(y64[t] - ref) <= bound)


# ------------------------------------------------------------ whole layer
def _forward_and_check(cfg, dev, seed=0, tokens=None, layer=None, inp=None):
    if inp is None:
        inp = I.make_inputs(cfg, device=dev, seed=seed)
    if layer is None:
        layer = B.MoELayer(inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=cfg.k)
    y = layer.forward(inp["x"])
    ws = layer.workspace(cfg.T, inp["x"].device)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    T = cfg.T
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    x_s = inp["x"][torch.from_numpy(toks).to(dev)]
    L64 = O.router_logits(x_s, inp["Wr"], inp["bias"])
    gpu_idx = ws.view("topk_idx", torch.int32, T * cfg.k).view(T, cfg.k)[torch.from_numpy(toks).to(dev)]
    gpu_idx = gpu_idx.cpu().numpy()
    robust = robust_tokens(L64, cfg.k, LOGIT_MARGIN)
    # the selection is exact where fp32 rounding cannot decide it ...
    ref_idx = O.topk(O.decision_logits(L64), cfg.k)
    for i in np.flatnonzero(robust):
        assert set(gpu_idx[i].tolist()) == set(ref_idx[i].tolist()), i
    # ... and a valid top-k elsewhere
    for i in np.flatnonzero(~robust):
        assert valid_topk(L64[i], gpu_idx[i], LOGIT_MARGIN), i
    keep = toks[robust]
    y_ref = O.moe_forward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=cfg.k,
                          tokens=keep)
    y_gpu = y[torch.from_numpy(keep).to(dev)]
    stats = assert_moe_close(y_gpu, y_ref)
    return stats, float(robust.mean()), y


def test_forward_tiny_config(cuda_device):
    cfg = I.get_config("tiny")
    stats, frac, _ = _forward_and_check(cfg, cuda_device)
    assert frac > 0.95


# the last shape gives two experts about 3000 rows each: 12 row-pair units,
# which the grouped GEMMs run as a chunk of 8 and a short chunk of 4 over
# every n-block
@pytest.mark.parametrize("T,d,n,E,k,bias", [(1000, 256, 192, 16, 4, True), (333, 128, 128, 9, 9, False),
                                            (2049, 384, 256, 32, 8, True), (1, 64, 64, 4, 2, False),
                                            (130, 64, 64, 1, 1, False), (3001, 512, 384, 2, 2, False)])
def test_forward_ragged_shapes(cuda_device, T, d, n, E, k, bias):
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k, bias="normal" if bias else None, bias_scale=0.3)
    _forward_and_check(cfg, cuda_device, seed=T + E)


def test_forward_deterministic(cuda_device):
    cfg = I.MoEConfig("t", T=1500, d=256, n=128, E=16, k=4)
    inp = I.make_inputs(cfg, device=cuda_device, seed=3)
    layer = B.MoELayer(inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=cfg.k)
    y1 = layer.forward(inp["x"]).clone()
    y2 = layer.forward(inp["x"]).clone()
    assert torch.equal(y1, y2)


def test_device_timeout_is_reported_and_context_survives(cuda_device):
    cfg = I.get_config("tiny")
    s, ws = ws_for(cfg.T, cfg.d, cfg.n, cfg.E, cfg.k, cuda_device)
    B.moe_selftest_timeout(ws, 2_000_000)   # 2 ms wait on a flag nobody sets
    detail = torch.zeros(1)
    st = B.moe_check_device_status(ws, raise_on_error=False)
    assert st == B.MOE_ERR_TIMEOUT
    assert B.moe_check_device_status(ws) == B.MOE_OK   # cleared by the read
    _forward_and_check(cfg, cuda_device)                 # context still usable


# ----------------------------------------------- full-size configurations
def _gpu_routing(ws, T, E, k):
    """The GPU's fp32 logits and permutation arrays, from the workspace."""
    cap = T * k
    L = ws.view("logits", torch.float32, T * E).view(T, E).cpu().numpy()
    idx = ws.view("topk_idx", torch.int32, T * k).view(T, k).cpu().numpy()
    counts = ws.view("counts", torch.int32, E).cpu().numpy()
    offsets = ws.view("offsets", torch.int32, E + 1).cpu().numpy()
    row_token = ws.view("row_token", torch.int32, cap).cpu().numpy()
    dst = ws.view("dst", torch.int32, T * k).cpu().numpy()
    return L, idx, counts, offsets, row_token, dst


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mixtral", "dsv3", "b7", "skew"])
def test_forward_full_size_sampled(cuda_device, name):
    """The full-size layer in the launch configuration the benchmark times.
    Integer work is checked whole: the top-k of the GPU's fp32 logits and the
    permutation of all T*k assignments equal the oracle's on those logits.
    The logits of a token sample meet the fp32 bound against the fp64 gate
    network, and the outputs of an expert-stratified sample (every expert's
    first row, last 128-row block and random rows; all tokens of the least-
    and most-loaded expert; at least 1024 tokens) meet the layer tolerance
    against the oracle routed on the same fp32 logits."""
    cfg = I.get_config(name)
    inp = I.make_inputs(cfg, device=cuda_device, seed=0)
    layer = B.MoELayer(inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=cfg.k)
    y = layer.forward(inp["x"])
    ws = layer.workspace(cfg.T, cuda_device)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    T, E, k = cfg.T, cfg.E, cfg.k
    L, idx, counts, offsets, row_token, dst = _gpu_routing(ws, T, E, k)
    # selection and permutation, every token, bit-exact given the fp32 logits
    assert np.array_equal(idx, O.topk(L, k))
    c_ref, o_ref, src_ref, dst_ref = O.permute(idx, E)
    assert np.array_equal(counts, c_ref) and np.array_equal(offsets, o_ref)
    assert np.array_equal(row_token[:T * k], src_ref // k) and np.array_equal(dst, dst_ref)
    toks = stratified_tokens(offsets, row_token[:T * k], T, seed=1)
    assert len(toks) >= min(1024, T)
    assert set(np.unique(idx[toks])) == set(np.flatnonzero(counts > 0))   # every expert with rows is reached
    # the gate network on a sample of tokens, against fp64
    lt = toks[:: max(1, len(toks) // 256)]
    L64 = O.router_logits(inp["x"][torch.from_numpy(lt).to(cuda_device)], inp["Wr"], inp["bias"])
    absdot = np.abs(to64(inp["x"][torch.from_numpy(lt).to(cuda_device)])) @ np.abs(to64(inp["Wr"]))
    err = np.abs(L[lt].astype(np.float64) - L64)
    assert np.all(err <= (3 * cfg.d + 3) * 2.0 ** -23 * (absdot + np.abs(L64)) + 1e-30)
    # outputs, the oracle routed on the GPU's fp32 logits
    routing = O.route(None, None, None, k, logits=L, tokens=toks)
    y_ref = O.moe_forward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=k,
                          routing=routing)
    assert_moe_close(y[torch.from_numpy(toks).to(cuda_device)], y_ref)
    assert torch.isfinite(y.float()).all()
    y2 = layer.forward(inp["x"])
    assert torch.equal(y, y2)
    del layer, inp
    torch.cuda.empty_cache()


# ----------------------------------------------------------- token rounding
def _expected_rounding(L, idx, tile, mode, seed=0):
    r = O.token_round(L, idx, tile, mode, seed=seed)
    T, E = L.shape
    counts = r["counts"]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    row_token = np.zeros(offsets[-1], dtype=np.int64)
    rowpos = {}
    for e in range(E):
        ts = np.flatnonzero(r["member"][:, e])
        row_token[offsets[e]:offsets[e + 1]] = ts
        for i, t in enumerate(ts):
            rowpos[(int(t), e)] = offsets[e] + i
    sizes = [len(s) for s in r["sets"]]
    tok_offsets = np.concatenate([[0], np.cumsum(sizes)])
    tok_rows = np.array([rowpos[(t, int(e))] for t in range(T) for e in r["sets"][t]], dtype=np.int64)
    row_w = np.zeros(offsets[-1])
    for t in range(T):
        s = r["sets"][t]
        if len(s):
            w = O.softmax(np.asarray(L, np.float64)[t, s])
            for e, we in zip(s, w):
                row_w[rowpos[(t, int(e))]] = we
    return counts, offsets, row_token, tok_offsets, tok_rows, row_w


@pytest.mark.parametrize("T,E,k,tile,mode,zipf", [(1000, 16, 2, 64, "nearest", 0.0), (777, 8, 2, 128, "nearest", 0.0),
                                                 (4099, 64, 4, 128, "nearest", 1.1), (100, 4, 1, 128, "nearest", 0.0),
                                                 (300, 32, 8, 64, "up", 0.0), (2000, 128, 8, 128, "up", 1.1),
                                                 (513, 5, 5, 256, "nearest", 0.0), (3000, 64, 4, 128, "stochastic", 1.1),
                                                 (900, 16, 2, 64, "stochastic", 0.0)])
def test_token_round_bit_exact(cuda_device, T, E, k, tile, mode, zipf):
    seed = 1234 + T
    L = I.make_logits(T, E, seed=T + E + tile, ties=True)
    if zipf:
        L = L - zipf * torch.log(torch.arange(1, E + 1, dtype=torch.float32))[None, :]
        L = (torch.round(L * 4) / 4).contiguous()
    Lnp = L.numpy()
    idx = torch.from_numpy(O.topk(Lnp, k))
    s = B.make_shape(T, 64, 64, E, k, tile, mode, seed)
    ws = B.Workspace(s, cuda_device)
    out = B.moe_token_round(s, L.to(cuda_device), idx.to(cuda_device), ws)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    counts, offsets, row_token, tok_offsets, tok_rows, row_w = _expected_rounding(Lnp, idx.numpy(), tile, mode,
                                                                                  seed)
    R = int(offsets[-1])
    assert np.array_equal(out["counts"].cpu().numpy(), counts)
    assert np.all(counts % tile == 0)
    assert np.array_equal(out["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(out["row_token"][:R].cpu().numpy(), row_token)
    assert np.array_equal(out["tok_offsets"].cpu().numpy(), tok_offsets)
    assert np.array_equal(out["tok_rows"][:R].cpu().numpy(), tok_rows)
    assert np.abs(to64(out["row_w"][:R]) - row_w).max(initial=0.0) <= 2e-6


def _gpu_sets(ws, shape, T):
    cap = B.moe_row_capacity(shape)
    offsets = ws.view("offsets", torch.int32, shape.E + 1).cpu().numpy()
    tok_offsets = ws.view("tok_offsets", torch.int32, T + 1).cpu().numpy()
    tok_rows = ws.view("tok_rows", torch.int32, cap).cpu().numpy()
    sets = []
    for t in range(T):
        rows = tok_rows[tok_offsets[t]:tok_offsets[t + 1]]
        sets.append(np.searchsorted(offsets, rows, side="right") - 1)
    return sets


# the last case rounds to the 256-row SM-pair tile with few rows per expert:
# the super-tile GEMMs, whose odd last blocks rounding leaves none of
@pytest.mark.parametrize("T,d,n,E,k,tile,mode", [(256, 128, 64, 8, 2, 64, "nearest"), (1500, 256, 128, 16, 4, 128, "nearest"),
                                                 (700, 128, 192, 12, 3, 64, "up"),
                                                 (1200, 256, 128, 16, 4, 64, "stochastic"),
                                                 (2048, 256, 256, 64, 8, 256, "nearest")])
def test_forward_token_rounding(cuda_device, T, d, n, E, k, tile, mode):
    """Rounded layer: given the GPU's fp32 logits, every token's final expert
    set equals the oracle's, and the outputs meet the layer tolerance."""
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k, bias="zipf", bias_scale=1.1)
    inp = I.make_inputs(cfg, device=cuda_device, seed=T)
    layer = B.MoELayer(inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=k, tile=tile, round=mode, seed=77)
    y = layer.forward(inp["x"])
    ws = layer.workspace(T, cuda_device)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    gsets = _gpu_sets(ws, layer.shape(T), T)
    counts = ws.view("counts", torch.int32, E).cpu().numpy()
    assert np.all(counts % tile == 0)
    L = ws.view("logits", torch.float32, T * E).view(T, E).cpu().numpy()
    routing = O.route(None, None, None, k, tile=tile, mode=mode, logits=L, seed=77)
    for t in range(T):
        assert np.array_equal(gsets[t], routing[1][t]), t
    y_ref = O.moe_forward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=k, tile=tile,
                          mode=mode, routing=routing)
    assert_moe_close(y, y_ref)
    empty = [t for t in range(T) if len(routing[1][t]) == 0]
    if empty:
        assert torch.all(y[torch.tensor(empty, device=cuda_device)] == 0)


@pytest.mark.slow
@pytest.mark.parametrize("mode", ["nearest", "stochastic"])
def test_forward_full_size_skew_rounding(cuda_device, mode):
    """The skewed-load layer at full size with tile-128 token rounding: every
    rounded count is a tile multiple, the GPU's final expert set of every
    token equals the oracle's rounding of the same fp32 logits, and the
    outputs of an expert-stratified token sample meet the tolerance."""
    cfg = I.get_config("skew")
    inp = I.make_inputs(cfg, device=cuda_device, seed=0)
    layer = B.MoELayer(inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=cfg.k, tile=128, round=mode,
                       seed=5)
    y = layer.forward(inp["x"])
    ws = layer.workspace(cfg.T, cuda_device)
    assert B.moe_check_device_status(ws) == B.MOE_OK
    T, E = cfg.T, cfg.E
    counts = ws.view("counts", torch.int32, E).cpu().numpy()
    assert np.all(counts % 128 == 0)
    gsets = _gpu_sets(ws, layer.shape(T), T)
    L = ws.view("logits", torch.float32, T * E).view(T, E).cpu().numpy()
    full = O.route(None, None, None, cfg.k, tile=128, mode=mode, logits=L, seed=5)
    for t in range(T):
        assert np.array_equal(gsets[t], full[1][t]), t
    cap = B.moe_row_capacity(layer.shape(T))
    offsets = ws.view("offsets", torch.int32, E + 1).cpu().numpy()
    row_token = ws.view("row_token", torch.int32, cap).cpu().numpy()[:offsets[-1]]
    toks = stratified_tokens(offsets, row_token, T, seed=3)
    routing = (toks, [full[1][t] for t in toks], [full[2][t] for t in toks])
    y_ref = O.moe_forward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=cfg.k, tile=128,
                          mode=mode, routing=routing)
    assert_moe_close(y[torch.from_numpy(toks).to(cuda_device)], y_ref)
    del layer, inp
    torch.cuda.empty_cache()
