"""Pins of the oracle's backward pass (CPU).

The backward pass is checked against things other than its own chain rule:
central finite differences of the (separately pinned) forward on tiny
layers, in every parameter, with and without token rounding; the router
gradient's exact zero at k = 1 (a softmax over one logit is constant); the
dense SwiGLU FFN's gradient through torch.autograd at E = 1, k = 1; the zero
sum of each token's logit gradient (softmax is shift-invariant); and
linearity in dy.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O


def _layer(rng, T, d, n, E, scale=1.0):
    return dict(x=rng.normal(size=(T, d)), Wr=rng.normal(size=(d, E)) * scale, bias=rng.normal(size=E) * 0.3,
                W1=rng.normal(size=(E, d, n)) / np.sqrt(d), W3=rng.normal(size=(E, d, n)) / np.sqrt(d),
                W2=rng.normal(size=(E, n, d)) / np.sqrt(n))


def _min_margin(p, k):
    """Smallest gap between the k-th and (k+1)-th fp64 logit of any token."""
    L = np.sort(O.router_logits(p["x"], p["Wr"], p["bias"]), axis=1)[:, ::-1]
    return np.inf if k == L.shape[1] else float(np.min(L[:, k - 1] - L[:, k]))


def _objective(p, dy, k, mode=O.ROUND_OFF, tile=2):
    y = O.moe_forward(p["x"], p["Wr"], p["bias"], p["W1"], p["W3"], p["W2"], k=k, tile=tile, mode=mode)
    return float(np.sum(dy * y))


def _finite_differences(p, dy, k, mode=O.ROUND_OFF, tile=2, h=1e-6):
    out = {}
    for name in ("x", "Wr", "bias", "W1", "W3", "W2"):
        g = np.zeros_like(p[name])
        for i in np.ndindex(p[name].shape):
            q = {kk: v.copy() for kk, v in p.items()}
            q[name][i] += h
            fp = _objective(q, dy, k, mode, tile)
            q[name][i] -= 2 * h
            fm = _objective(q, dy, k, mode, tile)
            g[i] = (fp - fm) / (2 * h)
        out[name] = g
    return out


KEYS = {"x": "dx", "Wr": "dWr", "bias": "db", "W1": "dW1", "W3": "dW3", "W2": "dW2"}


@pytest.mark.parametrize("T,d,n,E,k,seed", [(5, 6, 4, 4, 2, 0), (4, 5, 3, 3, 3, 1), (6, 4, 5, 5, 1, 2),
                                            (3, 7, 2, 6, 4, 3)])
def test_backward_matches_finite_differences(T, d, n, E, k, seed):
    rng = np.random.default_rng(seed)
    p = _layer(rng, T, d, n, E)
    assert _min_margin(p, k) > 1e-3  # the selection does not move under the steps
    dy = rng.normal(size=(T, d))
    g = O.moe_backward(p["x"], p["Wr"], p["bias"], p["W1"], p["W3"], p["W2"], dy, k=k)
    fd = _finite_differences(p, dy, k)
    for name, key in KEYS.items():
        np.testing.assert_allclose(g[key], fd[name], rtol=1e-6, atol=1e-7, err_msg=name)


@pytest.mark.parametrize("mode", [O.ROUND_NEAREST, O.ROUND_UP, O.ROUND_STOCHASTIC])
def test_backward_with_token_rounding_matches_finite_differences(mode):
    """Rounded sets are held fixed as well: tokens that joined an expert get
    its gradient, tokens that left get none (each rounding mode, the
    stochastic one with a fixed seed)."""
    rng = np.random.default_rng(7)
    T, d, n, E, k = 9, 4, 3, 3, 1
    p = _layer(rng, T, d, n, E, scale=2.0)
    dy = rng.normal(size=(T, d))
    L = O.decision_logits(O.router_logits(p["x"], p["Wr"], p["bias"]))
    counts = np.bincount(O.topk(L, k).reshape(-1), minlength=E)
    assert np.any(counts % 2 != 0)  # rounding to tile 2 changes some sets
    # margins of the rounding decisions: every per-expert logit gap > 1e-3
    for e in range(E):
        col = np.sort(L[:, e].astype(np.float64))
        assert np.min(np.diff(col)) > 1e-3
    assert _min_margin(p, k) > 1e-3
    g = O.moe_backward(p["x"], p["Wr"], p["bias"], p["W1"], p["W3"], p["W2"], dy, k=k, tile=2, mode=mode, seed=5)
    sizes = np.array([len(st) for st in g["sets"]])
    assert np.any(sizes != k)  # the rounding changed some token's set
    fd = _finite_differences_seeded(p, dy, k, mode=mode, tile=2, seed=5)
    for name, key in KEYS.items():
        np.testing.assert_allclose(g[key], fd[name], rtol=1e-6, atol=1e-7, err_msg=name)


def _finite_differences_seeded(p, dy, k, mode, tile, seed, h=1e-6):
    def objective(q):
        y = O.moe_forward(q["x"], q["Wr"], q["bias"], q["W1"], q["W3"], q["W2"], k=k, tile=tile, mode=mode,
                          seed=seed)
        return float(np.sum(dy * y))
    out = {}
    for name in ("x", "Wr", "bias", "W1", "W3", "W2"):
        g = np.zeros_like(p[name])
        for i in np.ndindex(p[name].shape):
            q = {kk: v.copy() for kk, v in p.items()}
            q[name][i] += h
            fp = objective(q)
            q[name][i] -= 2 * h
            fm = objective(q)
            g[i] = (fp - fm) / (2 * h)
        out[name] = g
    return out


def test_router_gradient_vanishes_at_k1():
    rng = np.random.default_rng(3)
    p = _layer(rng, 30, 8, 6, 5)
    dy = rng.normal(size=(30, 8))
    g = O.moe_backward(p["x"], p["Wr"], p["bias"], p["W1"], p["W3"], p["W2"], dy, k=1)
    assert np.all(g["dL"] == 0.0) and np.all(g["dWr"] == 0.0) and np.all(g["db"] == 0.0)


def test_logit_gradient_sums_to_zero_per_token():
    rng = np.random.default_rng(4)
    p = _layer(rng, 50, 8, 6, 7)
    dy = rng.normal(size=(50, 8))
    for k in (2, 3, 7):
        g = O.moe_backward(p["x"], p["Wr"], p["bias"], p["W1"], p["W3"], p["W2"], dy, k=k)
        scale = np.abs(g["dL"]).max()
        assert scale > 0
        np.testing.assert_allclose(g["dL"].sum(axis=1), 0.0, atol=1e-13 * scale * 7)
        # unselected experts get nothing
        assert np.count_nonzero(g["dL"]) <= 50 * k


def test_dense_ffn_gradient_via_autograd():
    """E = 1, k = 1 is a dense SwiGLU FFN; torch.autograd differentiates it."""
    rng = np.random.default_rng(5)
    T, d, n = 12, 6, 5
    p = _layer(rng, T, d, n, 1)
    dy = rng.normal(size=(T, d))
    g = O.moe_backward(p["x"], p["Wr"], p["bias"], p["W1"], p["W3"], p["W2"], dy, k=1)
    x = torch.tensor(p["x"], requires_grad=True)
    W1 = torch.tensor(p["W1"][0], requires_grad=True)
    W3 = torch.tensor(p["W3"][0], requires_grad=True)
    W2 = torch.tensor(p["W2"][0], requires_grad=True)
    y = (torch.nn.functional.silu(x @ W1) * (x @ W3)) @ W2
    (y * torch.tensor(dy)).sum().backward()
    np.testing.assert_allclose(g["dx"], x.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dW1"][0], W1.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dW3"][0], W3.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dW2"][0], W2.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_backward_is_linear_in_dy():
    rng = np.random.default_rng(6)
    p = _layer(rng, 20, 6, 4, 4)
    dy1, dy2 = rng.normal(size=(20, 6)), rng.normal(size=(20, 6))
    args = (p["x"], p["Wr"], p["bias"], p["W1"], p["W3"], p["W2"])
    g1 = O.moe_backward(*args, dy1, k=2)
    g2 = O.moe_backward(*args, dy2, k=2)
    g12 = O.moe_backward(*args, dy1 + 2.0 * dy2, k=2)
    for key in KEYS.values():
        np.testing.assert_allclose(g12[key], g1[key] + 2.0 * g2[key], rtol=1e-10, atol=1e-12)


def test_magnitudes_bound_the_gradients():
    """Each magnitude is the sum of |terms| of its element: never below the
    element itself (triangle inequality), equal to it when no terms cancel."""
    rng = np.random.default_rng(8)
    p = _layer(rng, 40, 6, 5, 4)
    dy = rng.normal(size=(40, 6))
    g = O.moe_backward(p["x"], p["Wr"], p["bias"], p["W1"], p["W3"], p["W2"], dy, k=2, magnitudes=True)
    for key in ("dx", "dW1", "dW3", "dW2"):
        assert np.all(np.abs(g[key]) <= g[key + "_mag"] * (1 + 1e-12) + 1e-300), key
    # all-positive operands: nothing cancels in dW2 = sum (w h)^T dy when h, dy > 0
    q = {kk: np.abs(v) for kk, v in p.items()}
    g2 = O.moe_backward(q["x"], q["Wr"], q["bias"], q["W1"], q["W3"], q["W2"], np.abs(dy), k=2, magnitudes=True)
    np.testing.assert_allclose(g2["dW2_mag"], g2["dW2"], rtol=1e-12)
