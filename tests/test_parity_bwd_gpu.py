"""Parity of the backward pass (moe_backward, through the C ABI) against the
oracle's moe_backward.

Both sides select experts from the same fp32 logits (the oracle is handed the
GPU's logits for the selection and the gate weights), so the sets agree
exactly; every gradient must then meet the layer tolerance
  max |g - g_ref| <= 2e-2 rms(g_ref),  sum |g - g_ref| / sum |g_ref| <= 5e-3
where the expert-path gradients (dx, dW1, dW3, dW2), whose bf16 operands carry
one rounding, are held to the elementwise bound |g - g_ref| <= 2^-7 sum|terms|
instead of the max-error term; identities that hold exactly on the device
are checked exactly: a
softmax over one logit passes no gradient (k = 1: dWr = db = 0), an expert
no token selects gets zero weight gradients, and two runs agree bitwise.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_93_b300 import binding as B
from mixture_experts_layer_93_b300 import inputs as I
from oracle import moe_oracle as O

from moe_testlib import assert_grad_close, assert_moe_close, stratified_tokens, to64

pytestmark = pytest.mark.gpu

GRADS = [("dx", "dx"), ("dWr", "dWr"), ("dbias", "db"), ("dW1", "dW1"), ("dW3", "dW3"), ("dW2", "dW2")]


def check_grads(out, ref, skip=()):
    for key, rkey in GRADS:
        if key in skip:
            continue
        if rkey + "_mag" in ref:
            assert_grad_close(out[key], ref[rkey], ref[rkey + "_mag"], what=key)
        else:
            assert_moe_close(out[key], ref[rkey], what=key)


def _setup(cfg, dev, seed, dead_expert=False):
    inp = I.make_inputs(cfg, device=dev, seed=seed)
    if dead_expert:
        bias = torch.zeros(cfg.E, device=dev) if inp["bias"] is None else inp["bias"].clone()
        bias[-1] = -1.0e4  # never selected
        inp["bias"] = bias
    g = torch.Generator(device="cpu").manual_seed(seed + 1)
    dy = torch.randn(cfg.T, cfg.d, generator=g).to(torch.bfloat16).to(dev)
    s = B.make_shape(cfg.T, cfg.d, cfg.n, cfg.E, cfg.k)
    W13p, _ = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    W13i = B.moe_prepare_weights_bwd(inp["W1"], inp["W3"])
    return inp, dy, s, W13p, W13i


def _run(inp, dy, s, W13p, W13i, dev):
    ws = B.Workspace(s, dev, backward=True)
    out = B.moe_backward(s, inp["x"], inp["Wr"], inp["bias"], W13p, W13i, inp["W2"], dy, ws)
    torch.cuda.synchronize()
    assert B.moe_check_device_status(ws) == B.MOE_OK
    logits = ws.view("logits", torch.float32, s.T * s.E).view(s.T, s.E).clone()
    return out, logits


SHAPES = [  # T, d, n, E, k: single-SM and SM-pair tiles, ragged experts, n % 128 != 0
    (256, 128, 64, 8, 2),
    (700, 256, 128, 6, 2),
    (600, 512, 256, 5, 3),
    (300, 384, 192, 4, 2),
    (500, 256, 64, 64, 4),
    (129, 256, 320, 3, 3),
    (200, 128, 64, 300, 3),   # E > 256: the separate top-k and permutation kernels
    (64, 128, 128, 1, 1),     # one expert: a dense FFN, no router gradient
]


@pytest.mark.parametrize("T,d,n,E,k", SHAPES)
def test_backward_matches_oracle(cuda_device, T, d, n, E, k):
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k, bias="normal", bias_scale=0.5)
    inp, dy, s, W13p, W13i = _setup(cfg, cuda_device, seed=T + d + E)
    out, logits = _run(inp, dy, s, W13p, W13i, cuda_device)
    ref = O.moe_backward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], dy, k=k,
                         logits=logits.cpu().numpy(), magnitudes=True)
    check_grads(out, ref)


@pytest.mark.parametrize("T,d,n,E,k,tile,mode", [(700, 256, 128, 6, 2, 64, "nearest"), (900, 256, 192, 8, 3, 128, "up"),
                                                 (1000, 128, 64, 16, 2, 64, "stochastic"),
                                                 (300, 256, 128, 4, 1, 256, "nearest")])
def test_backward_with_token_rounding(cuda_device, T, d, n, E, k, tile, mode):
    """The rounded sets (tokens joining or leaving experts, sets of any size,
    empty ones included) are recomputed and held fixed; gradients against the
    oracle's backward of the rounded layer on the same fp32 logits."""
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=k, bias="normal", bias_scale=0.5)
    inp = I.make_inputs(cfg, device=cuda_device, seed=T + E)
    g = torch.Generator(device="cpu").manual_seed(T)
    dy = torch.randn(T, d, generator=g).to(torch.bfloat16).to(cuda_device)
    s = B.make_shape(T, d, n, E, k, tile=tile, round=mode, seed=7)
    W13p, _ = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    W13i = B.moe_prepare_weights_bwd(inp["W1"], inp["W3"])
    out, logits = _run(inp, dy, s, W13p, W13i, cuda_device)
    ref = O.moe_backward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], dy, k=k, tile=tile,
                         mode=mode, seed=7, logits=logits.cpu().numpy(), magnitudes=True)
    sizes = np.array([len(st) for st in ref["sets"]])
    assert np.any(sizes != k)  # rounding changed some sets
    check_grads(out, ref)


def test_backward_k1_has_no_router_gradient(cuda_device):
    cfg = I.MoEConfig("t", T=300, d=256, n=128, E=5, k=1, bias="normal", bias_scale=0.5)
    inp, dy, s, W13p, W13i = _setup(cfg, cuda_device, seed=3)
    out, logits = _run(inp, dy, s, W13p, W13i, cuda_device)
    assert torch.all(out["dWr"] == 0) and torch.all(out["dbias"] == 0)
    ref = O.moe_backward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], dy, k=1,
                         logits=logits.cpu().numpy(), magnitudes=True)
    check_grads(out, ref, skip=("dWr", "dbias"))


def test_backward_unselected_expert_gets_zero(cuda_device):
    cfg = I.MoEConfig("t", T=400, d=256, n=128, E=6, k=2, bias="normal", bias_scale=0.5)
    inp, dy, s, W13p, W13i = _setup(cfg, cuda_device, seed=4, dead_expert=True)
    ws = B.Workspace(s, cuda_device, backward=True)
    # poison the outputs: every element must be written
    out = {k: torch.full(shape, float("nan"), device=cuda_device) for k, shape in
           [("dx", (400, 256)), ("dWr", (256, 6)), ("dbias", (6,)), ("dW1", (6, 256, 128)), ("dW3", (6, 256, 128)),
            ("dW2", (6, 128, 256))]}
    B.moe_backward(s, inp["x"], inp["Wr"], inp["bias"], W13p, W13i, inp["W2"], dy, ws, out=out)
    torch.cuda.synchronize()
    assert B.moe_check_device_status(ws) == B.MOE_OK
    counts = ws.view("counts", torch.int32, 6).cpu()
    assert counts[-1] == 0
    for key in ("dW1", "dW3", "dW2"):
        assert torch.all(out[key][-1] == 0), key
        assert torch.isfinite(out[key]).all(), key
    assert torch.all(out["dWr"][:, -1] == 0) and out["dbias"][-1] == 0
    logits = ws.view("logits", torch.float32, 400 * 6).view(400, 6).cpu().numpy()
    ref = O.moe_backward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], dy, k=2, logits=logits, magnitudes=True)
    check_grads(out, ref)


def test_backward_is_deterministic(cuda_device):
    cfg = I.MoEConfig("t", T=900, d=256, n=256, E=8, k=2, bias="normal", bias_scale=0.5)
    inp, dy, s, W13p, W13i = _setup(cfg, cuda_device, seed=5)
    a, _ = _run(inp, dy, s, W13p, W13i, cuda_device)
    b, _ = _run(inp, dy, s, W13p, W13i, cuda_device)
    for key, _ in GRADS:
        assert torch.equal(a[key], b[key]), key


def test_backward_tiny_config(cuda_device):
    cfg = I.get_config("tiny")
    inp, dy, s, W13p, W13i = _setup(cfg, cuda_device, seed=0)
    out, logits = _run(inp, dy, s, W13p, W13i, cuda_device)
    ref = O.moe_backward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], dy, k=cfg.k,
                         logits=logits.cpu().numpy(), magnitudes=True)
    check_grads(out, ref)
    # the logit gradient of every token sums to zero, so do dbias and the rows of dWr
    dWr = to64(out["dWr"])
    assert np.all(np.abs(dWr.sum(axis=1)) <= 1e-4 * np.abs(dWr).max() * cfg.E)


def _channel_reference(inp, dy, L, idx, w, e, J):
    """fp64 weight gradients the oracle's formulas give for expert e's
    channels J (dW1[e][:, J], dW3[e][:, J], dW2[e][J, :]) with their
    magnitudes; selection idx and gate weights w from the fp32 logits, as
    moe_backward (oracle) takes them."""
    x64 = to64(inp["x"])
    dy64 = to64(dy)
    rows = np.argwhere(idx == e)               # (t, j) pairs routed to e, in token order
    ts, js = rows[:, 0], rows[:, 1]
    we = w[ts, js]
    W1J, W3J = to64(inp["W1"][e][:, J]), to64(inp["W3"][e][:, J])
    W2J = to64(inp["W2"][e][J, :])
    X = x64[ts]
    g, u = X @ W1J, X @ W3J
    s = O.sigmoid(g)
    a = g * s
    h = a * u
    dh = we[:, None] * (dy64[ts] @ W2J.T)
    dg, du = dh * u * (s * (1 + g * (1 - s))), dh * a
    return {"dW1": X.T @ dg, "dW3": X.T @ du, "dW2": (we[:, None] * h).T @ dy64[ts],
            "dW1_mag": np.abs(X).T @ np.abs(dg), "dW3_mag": np.abs(X).T @ np.abs(du),
            "dW2_mag": np.abs(we[:, None] * h).T @ np.abs(dy64[ts])}


def _dx_reference(inp, dy, idx, w, toks):
    """fp64 dx of the tokens `toks` with magnitudes: every selected expert's
    path in full plus the gate network's term, worked expert by expert so each
    expert's weights are widened once."""
    x64, dy64, Wr = to64(inp["x"]), to64(dy), to64(inp["Wr"])
    k = idx.shape[1]
    sel = idx[toks]                             # [S, k]
    dx = np.zeros((len(toks), x64.shape[1]))
    mag = np.zeros_like(dx)
    dws = np.zeros(sel.shape)
    for e in np.unique(sel):
        ii, jj = np.nonzero(sel == e)
        ts = toks[ii]
        W1e, W3e, W2e = to64(inp["W1"][int(e)]), to64(inp["W3"][int(e)]), to64(inp["W2"][int(e)])
        X = x64[ts]
        g, u = X @ W1e, X @ W3e
        st = O.sigmoid(g)
        a = g * st
        dhu = dy64[ts] @ W2e.T
        dws[ii, jj] = np.sum(dhu * a * u, axis=1)
        wt = w[ts, jj][:, None]
        dg, du = wt * dhu * u * (st * (1 + g * (1 - st))), wt * dhu * a
        np.add.at(dx, ii, dg @ W1e.T + du @ W3e.T)
        np.add.at(mag, ii, np.abs(dg) @ np.abs(W1e).T + np.abs(du) @ np.abs(W3e).T)
    wt = w[toks]
    dl = wt * (dws - np.sum(wt * dws, axis=1, keepdims=True))
    for i in range(len(toks)):
        dx[i] += Wr[:, sel[i]] @ dl[i]
        mag[i] += np.abs(Wr[:, sel[i]]) @ np.abs(dl[i])
    return dx, mag


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mixtral", "dsv3", "b7", "skew"])
def test_backward_full_size_sampled(cuda_device, name):
    """The full-size layers in the bench's launch configuration: dx of an
    expert-stratified token sample (every expert's first row, last 128-row
    block and a random row; all tokens of the least- and most-loaded expert;
    at least 1024 tokens) and the weight-gradient channels of several experts
    (the least- and most-loaded ones among them) against the oracle's
    formulas; dWr and dbias by the zero sum over experts."""
    cfg = I.get_config(name)
    inp, dy, s, W13p, W13i = _setup(cfg, cuda_device, seed=0)
    out, logits = _run(inp, dy, s, W13p, W13i, cuda_device)
    L = logits.cpu().numpy().astype(np.float64)
    idx = O.topk(L, cfg.k)
    w = O.gate_weights(L, idx)
    counts, offsets, src, _ = O.permute(idx, cfg.E)
    toks = stratified_tokens(offsets, src // cfg.k, cfg.T, seed=1, per_expert=1)
    dx_ref, dx_mag = _dx_reference(inp, dy, idx, w, toks)
    assert_grad_close(out["dx"][torch.from_numpy(toks).to(cuda_device)], dx_ref, dx_mag, what="dx")
    rng = np.random.default_rng(1)
    nz = np.flatnonzero(counts > 0)
    experts = {int(nz[np.argmin(counts[nz])]), int(np.argmax(counts))}
    experts.update(int(e) for e in rng.choice(cfg.E, size=min(4, cfg.E), replace=False))
    for e in sorted(experts):
        J = np.sort(rng.choice(cfg.n, size=8, replace=False))
        ref = _channel_reference(inp, dy, L, idx, w, e, J)
        Jt = torch.from_numpy(J).to(cuda_device)
        assert_grad_close(out["dW1"][e][:, Jt], ref["dW1"], ref["dW1_mag"], what=f"dW1[{e}]")
        assert_grad_close(out["dW3"][e][:, Jt], ref["dW3"], ref["dW3_mag"], what=f"dW3[{e}]")
        assert_grad_close(out["dW2"][e][Jt, :], ref["dW2"], ref["dW2_mag"], what=f"dW2[{e}]")
    dWr = to64(out["dWr"])
    assert np.all(np.abs(dWr.sum(axis=1)) <= 1e-4 * np.sqrt(np.mean(dWr ** 2)) * cfg.E)
    db = to64(out["dbias"])
    assert abs(db.sum()) <= 1e-4 * np.sqrt(np.mean(db ** 2)) * cfg.E
    del out
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_backward_full_size_rounded_skew(cuda_device):
    """The skewed layer with nearest rounding to 128 at full size: the rounded
    sets from the device against the oracle's rounding of the same logits,
    then sampled channels of two experts against the formulas on those sets."""
    cfg = I.get_config("skew")
    inp, dy, _, W13p, W13i = _setup(cfg, cuda_device, seed=0)
    s = B.make_shape(cfg.T, cfg.d, cfg.n, cfg.E, cfg.k, tile=128, round="nearest")
    out, logits = _run(inp, dy, s, W13p, W13i, cuda_device)
    logits = logits.cpu().numpy()
    L = logits.astype(np.float64)
    r = O.token_round(L, O.topk(L, cfg.k), 128, O.ROUND_NEAREST)
    member = r["member"]
    rng = np.random.default_rng(3)
    x64, dy64 = to64(inp["x"]), to64(dy)
    for e in rng.choice(cfg.E, size=2, replace=False):
        e = int(e)
        ts = np.flatnonzero(member[:, e])
        assert ts.size % 128 == 0
        we = np.array([O.softmax(L[t, r["sets"][t]])[list(r["sets"][t]).index(e)] for t in ts])
        J = np.sort(rng.choice(cfg.n, size=6, replace=False))
        X = x64[ts]
        W1J, W3J, W2J = to64(inp["W1"][e][:, J]), to64(inp["W3"][e][:, J]), to64(inp["W2"][e][J, :])
        g, u = X @ W1J, X @ W3J
        sg = O.sigmoid(g)
        a = g * sg
        dh = we[:, None] * (dy64[ts] @ W2J.T)
        dg, du = dh * u * (sg * (1 + g * (1 - sg))), dh * a
        Jt = torch.from_numpy(J).to(cuda_device)
        assert_grad_close(out["dW1"][e][:, Jt], X.T @ dg, np.abs(X).T @ np.abs(dg), what=f"dW1[{e}]")
        assert_grad_close(out["dW3"][e][:, Jt], X.T @ du, np.abs(X).T @ np.abs(du), what=f"dW3[{e}]")
        hw = we[:, None] * a * u
        assert_grad_close(out["dW2"][e][Jt, :], hw.T @ dy64[ts], np.abs(hw).T @ np.abs(dy64[ts]), what=f"dW2[{e}]")
    del out
    torch.cuda.empty_cache()
