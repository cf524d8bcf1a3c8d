"""Pins for the fp64 oracle, checked against things other than itself:
brute force on tiny inputs, closed forms, library routines for special cases,
and invariants the pages fix.  CPU only."""
import itertools
import math

import numpy as np
import pytest
import torch
from scipy.special import expit

from oracle import moe_oracle as O
from mixture_experts_layer_93_b300 import inputs as I


def grid_logits(T, E, seed):
    """fp32 logits on a 1/4 grid (exact sums, frequent ties, signed zeros)."""
    return I.make_logits(T, E, seed=seed, ties=True).numpy()


# ---------------------------------------------------------------- top-k
@pytest.mark.parametrize("E,k", [(1, 1), (4, 2), (6, 1), (6, 3), (6, 6), (7, 4)])
def test_topk_brute_force_subsets(E, k):
    L = grid_logits(60, E, seed=E * 10 + k)
    idx = O.topk(L, k)
    for t in range(L.shape[0]):
        # best k-subset: maximal sum of logits; among equal sums, the
        # lexicographically smallest sorted id tuple (lower ids win ties)
        best = None
        for sub in itertools.combinations(range(E), k):
            key = (-sum(float(L[t, e]) for e in sub), sub)
            if best is None or key < best:
                best = key
        assert tuple(sorted(idx[t].tolist())) == best[1]
        vals = L[t, idx[t]]
        for j in range(k - 1):
            assert vals[j] >= vals[j + 1]
            if vals[j] == vals[j + 1]:
                assert idx[t, j] < idx[t, j + 1]


def test_topk_matches_stable_argsort():
    L = torch.randn(500, 37, generator=torch.Generator().manual_seed(3)).numpy()
    L[:, 5] = L[:, 9]            # exact ties
    L[::3, 2] = 0.0
    L[::3, 1] = -0.0             # -0 ties +0, lower id first
    for k in (1, 2, 8, 37):
        ref = np.argsort(-L, axis=1, kind="stable")[:, :k]
        assert np.array_equal(O.topk(L, k), ref)


def test_topk_signed_zero_tie():
    L = np.array([[-0.0, 0.0, -1.0]], dtype=np.float32)
    assert O.topk(L, 1).tolist() == [[0]]
    L = np.array([[0.0, -0.0, -1.0]], dtype=np.float32)
    assert O.topk(L, 2).tolist() == [[0, 1]]


# ---------------------------------------------------------- gate weights
def test_gate_weights_closed_form_k2():
    L = np.random.default_rng(0).normal(size=(200, 9)) * 3
    idx = O.topk(L, 2)
    w = O.gate_weights(L, idx)
    l0 = L[np.arange(200), idx[:, 0]]
    l1 = L[np.arange(200), idx[:, 1]]
    np.testing.assert_allclose(w[:, 0], expit(l0 - l1), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(w[:, 1], expit(l1 - l0), rtol=1e-13, atol=1e-15)


def test_gate_weights_invariants():
    L = grid_logits(300, 16, seed=1).astype(np.float64)
    for k in (1, 3, 16):
        idx = O.topk(L, k)
        w = O.gate_weights(L, idx)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)
        assert np.all(np.diff(w, axis=1) <= 1e-15)       # nonincreasing in slot order
        if k == 1:
            assert np.all(w == 1.0)
    # all-equal logits -> uniform weights
    w = O.gate_weights(np.zeros((3, 5)), O.topk(np.zeros((3, 5)), 4))
    np.testing.assert_allclose(w, 0.25, atol=1e-15)
    # large logits do not overflow (shifted by the max)
    w = O.gate_weights(np.array([[1000.0, 999.0]]), np.array([[0, 1]]))
    np.testing.assert_allclose(w[0, 0], expit(1.0), rtol=1e-13)


# --------------------------------------------------------- permutation
@pytest.mark.parametrize("T,E,k,skew", [(1, 1, 1, 0.0), (100, 8, 2, 0.0), (333, 64, 8, 1.2), (50, 3, 3, 0.0)])
def test_permute_matches_stable_argsort(T, E, k, skew):
    idx = I.make_topk_idx(T, E, k, seed=T + E, skew=skew).numpy()
    counts, offsets, src, dst = O.permute(idx, E)
    flat = idx.reshape(-1)
    assert np.array_equal(src, np.argsort(flat, kind="stable"))
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert counts.sum() == T * k
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(np.sort(src), np.arange(T * k))       # bijection
    assert np.array_equal(dst[src], np.arange(T * k))
    for e in range(E):
        rows = src[offsets[e]:offsets[e + 1]]
        assert np.all(flat[rows] == e)
        assert np.all(np.diff(rows // k) > 0)                    # ascending t


# ------------------------------------------------------------- SwiGLU
def test_silu_values():
    assert O.silu(0.0) == 0.0
    assert math.isclose(float(O.silu(1.0)), 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)
    z = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(O.silu(z), z * expit(z), rtol=1e-13, atol=1e-300)
    assert O.silu(-800.0) == 0.0 or abs(O.silu(-800.0)) < 1e-300


def _one_per_column(rows, cols, rng):
    """A [rows, cols] matrix with one nonzero per column; returns (M, pos, val)."""
    pos = rng.integers(0, rows, size=cols)
    val = rng.normal(size=cols)
    M = np.zeros((rows, cols))
    M[pos, np.arange(cols)] = val
    return M, pos, val


def test_swiglu_index_arithmetic():
    """Weights with one nonzero per column turn each product into a single
    term, so the expected output is written with indices alone (no matmul):
    a transposed or swapped operand changes it."""
    rng = np.random.default_rng(7)
    d, n, T = 5, 3, 11
    x = rng.normal(size=(T, d))
    W1, p1, a = _one_per_column(d, n, rng)
    W3, p3, b = _one_per_column(d, n, rng)
    W2, r, c = _one_per_column(n, d, rng)
    h_ref = np.empty((T, n))
    for t in range(T):
        for j in range(n):
            g = x[t, p1[j]] * a[j]
            h_ref[t, j] = g * expit(g) * (x[t, p3[j]] * b[j])
    y_ref = np.empty((T, d))
    for t in range(T):
        for i in range(d):
            y_ref[t, i] = h_ref[t, r[i]] * c[i]
    np.testing.assert_allclose(O.expert_hidden(x, W1, W3), h_ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(O.expert_out(h_ref, W2), y_ref, rtol=1e-13, atol=1e-15)
    # the full layer with E=1, k=1 (gate weight 1) is the dense FFN
    Wr = rng.normal(size=(d, 1))
    y = O.moe_forward(x, Wr, None, W1[None], W3[None], W2[None], k=1)
    np.testing.assert_allclose(y, y_ref, rtol=1e-13, atol=1e-15)


def _rand_layer(T, d, n, E, seed, bias=False):
    cfg = I.MoEConfig("t", T=T, d=d, n=n, E=E, k=1, bias="normal" if bias else None, bias_scale=0.5)
    return I.make_inputs(cfg, seed=seed)


def test_identical_experts_is_dense_ffn():
    inp = _rand_layer(40, 16, 8, 6, seed=2, bias=True)
    W1 = inp["W1"][:1].repeat(6, 1, 1)
    W3 = inp["W3"][:1].repeat(6, 1, 1)
    W2 = inp["W2"][:1].repeat(6, 1, 1)
    dense = O.dense_swiglu_ffn(inp["x"], W1[0], W3[0], W2[0])
    for k in (1, 2, 6):
        y = O.moe_forward(inp["x"], inp["Wr"], inp["bias"], W1, W3, W2, k=k)
        np.testing.assert_allclose(y, dense, rtol=1e-12, atol=1e-12)


def test_expert_relabelling_invariance():
    inp = _rand_layer(64, 16, 8, 5, seed=3, bias=True)
    perm = torch.tensor([3, 0, 4, 1, 2])
    y = O.moe_forward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=2)
    y2 = O.moe_forward(inp["x"], inp["Wr"][:, perm], inp["bias"][perm], inp["W1"][perm],
                       inp["W3"][perm], inp["W2"][perm], k=2)
    np.testing.assert_allclose(y, y2, rtol=1e-12, atol=1e-12)


def test_zero_down_projection_gives_zero():
    inp = _rand_layer(20, 16, 8, 4, seed=4)
    y = O.moe_forward(inp["x"], inp["Wr"], None, inp["W1"], inp["W3"], torch.zeros_like(inp["W2"]), k=2)
    assert np.all(y == 0.0)


def test_brute_force_loops_tiny_layer():
    """Explicit index loops (no matmul, no sort) on a tiny layer, k=E and k<E."""
    rng = np.random.default_rng(11)
    T, d, n, E = 4, 6, 5, 4
    x = rng.normal(size=(T, d))
    Wr = rng.normal(size=(d, E))
    bias = rng.normal(size=E)
    W1 = rng.normal(size=(E, d, n))
    W3 = rng.normal(size=(E, d, n))
    W2 = rng.normal(size=(E, n, d))
    for k in (2, E):
        y = O.moe_forward(x, Wr, bias, W1, W3, W2, k=k)
        for t in range(T):
            logit = [sum(x[t, i] * Wr[i, e] for i in range(d)) + bias[e] for e in range(E)]
            chosen = []
            for _ in range(k):
                best = None
                for e in range(E):
                    if e not in chosen and (best is None or np.float32(logit[e]) > np.float32(logit[best])):
                        best = e
                chosen.append(best)
            m = max(logit[e] for e in chosen)
            z = [math.exp(logit[e] - m) for e in chosen]
            w = [v / sum(z) for v in z]
            for i in range(d):
                acc = 0.0
                for e, we in zip(chosen, w):
                    o = 0.0
                    for j in range(n):
                        g = sum(x[t, q] * W1[e, q, j] for q in range(d))
                        u = sum(x[t, q] * W3[e, q, j] for q in range(d))
                        o += (g / (1.0 + math.exp(-g))) * u * W2[e, j, i]
                    acc += we * o
                assert math.isclose(y[t, i], acc, rel_tol=1e-11, abs_tol=1e-12)


def test_token_subset_equals_full_rows():
    inp = _rand_layer(50, 16, 8, 6, seed=5, bias=True)
    full = O.moe_forward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=2)
    sub = np.array([0, 7, 13, 49])
    part = O.moe_forward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=2, tokens=sub)
    # BLAS blocking differs with the row count, so only rounding-level noise
    np.testing.assert_allclose(part, full[sub], rtol=1e-13, atol=1e-15)
    _, sets_full, _ = O.route(inp["x"], inp["Wr"], inp["bias"], 2)
    _, sets_sub, _ = O.route(inp["x"], inp["Wr"], inp["bias"], 2, tokens=sub)
    for i, t in enumerate(sub):
        assert np.array_equal(sets_sub[i], sets_full[t])


def test_expert_subset_and_given_routing():
    """moe_forward restricted to a subset of experts keeps exactly the terms of
    those experts (checked by explicit loops), the subsets of a partition add
    up to the full layer, and routing passed in gives the same y as routing
    inside the call."""
    rng = np.random.default_rng(21)
    T, d, n, E, k = 5, 4, 3, 5, 2
    x = rng.normal(size=(T, d))
    Wr = rng.normal(size=(d, E))
    W1 = rng.normal(size=(E, d, n))
    W3 = rng.normal(size=(E, d, n))
    W2 = rng.normal(size=(E, n, d))
    sub = [3, 0]
    y_sub = O.moe_forward(x, Wr, None, W1, W3, W2, k=k, experts=sub)
    for t in range(T):
        logit = [sum(x[t, i] * Wr[i, e] for i in range(d)) for e in range(E)]
        chosen = sorted(range(E), key=lambda e: (-np.float32(logit[e]), e))[:k]
        m = max(logit[e] for e in chosen)
        z = {e: math.exp(logit[e] - m) for e in chosen}
        for i in range(d):
            acc = 0.0
            for e in chosen:
                if e not in sub:
                    continue
                o = 0.0
                for j in range(n):
                    g = sum(x[t, q] * W1[e, q, j] for q in range(d))
                    u = sum(x[t, q] * W3[e, q, j] for q in range(d))
                    o += (g / (1.0 + math.exp(-g))) * u * W2[e, j, i]
                acc += z[e] / sum(z.values()) * o
            assert math.isclose(y_sub[t, i], acc, rel_tol=1e-11, abs_tol=1e-12)
    full = O.moe_forward(x, Wr, None, W1, W3, W2, k=k)
    parts = [O.moe_forward(x, Wr, None, W1, W3, W2, k=k, experts=p) for p in ([0, 3], [1], [2, 4])]
    np.testing.assert_allclose(sum(parts), full, rtol=1e-13, atol=1e-14)
    routing = O.route(x, Wr, None, k)
    np.testing.assert_array_equal(O.moe_forward(x, Wr, None, W1, W3, W2, k=k, routing=routing), full)


# -------------------------------------------------------------- logits
def test_router_logits_one_hot_rows():
    rng = np.random.default_rng(12)
    d, E = 7, 5
    Wr = rng.normal(size=(d, E)).astype(np.float32)
    b = rng.normal(size=E).astype(np.float32)
    x = np.eye(d)[[3, 0, 6, 6]] * np.array([[1.0], [2.0], [-0.5], [0.0]])
    L = O.router_logits(x, Wr, b)
    np.testing.assert_array_equal(L[0], Wr[3].astype(np.float64) + b)
    np.testing.assert_array_equal(L[1], 2.0 * Wr[0].astype(np.float64) + b)
    np.testing.assert_array_equal(L[2], -0.5 * Wr[6].astype(np.float64) + b)
    np.testing.assert_array_equal(L[3], b.astype(np.float64))


# ------------------------------------------------------- token rounding
def _check_rounding(L, idx, tile, mode, seed=0):
    T, E = L.shape
    r = O.token_round(L, idx, tile, mode, seed=seed)
    member0 = np.zeros((T, E), bool)
    member0[np.repeat(np.arange(T), idx.shape[1]), idx.reshape(-1)] = True
    c0 = member0.sum(0)
    cap = tile * (T // tile)
    for e in range(E):
        c, c2 = int(c0[e]), int(r["counts"][e])
        assert c2 % tile == 0
        assert c2 <= cap
        if mode == O.ROUND_NEAREST:
            assert abs(c2 - c) <= (tile // 2 if c <= cap else tile)
        else:
            assert abs(c2 - c) < tile or (c2 - c) == 0
        col0, col = member0[:, e], r["member"][:, e]
        assert np.all(col >= col0) or np.all(col <= col0)      # superset or subset
        add = np.flatnonzero(col & ~col0)
        drop = np.flatnonzero(col0 & ~col)
        rest = np.flatnonzero(~col0 & ~col)
        kept = np.flatnonzero(col0 & col)
        for a in add:           # every added beats every not-added candidate
            for b in rest:
                assert L[a, e] > L[b, e] or (L[a, e] == L[b, e] and a < b)
        for dd in drop:         # every dropped is worse than every kept
            for kk in kept:
                assert L[dd, e] < L[kk, e] or (L[dd, e] == L[kk, e] and dd > kk)
    for t in range(T):
        s = r["sets"][t]
        assert np.array_equal(np.sort(s), np.flatnonzero(r["member"][t]))
        for j in range(len(s) - 1):
            assert L[t, s[j]] > L[t, s[j + 1]] or (L[t, s[j]] == L[t, s[j + 1]] and s[j] < s[j + 1])
    return r


@pytest.mark.parametrize("mode", [O.ROUND_NEAREST, O.ROUND_UP])
@pytest.mark.parametrize("T,E,k,tile,seed", [(40, 5, 2, 8, 0), (64, 6, 3, 8, 1), (37, 4, 2, 4, 2), (30, 3, 1, 16, 3)])
def test_token_rounding_brute_force(mode, T, E, k, tile, seed):
    L = grid_logits(T, E, seed=100 + seed)
    idx = O.topk(L, k)
    _check_rounding(L, idx, tile, mode)


def test_token_rounding_noop_on_multiples():
    T, E, tile = 32, 4, 8
    idx = (np.arange(T) % E).reshape(T, 1).astype(np.int32)    # 8 tokens per expert
    L = grid_logits(T, E, seed=9)
    r = O.token_round(L, idx, tile, O.ROUND_NEAREST)
    assert np.array_equal(r["counts"], np.full(E, 8))
    for t in range(T):
        assert r["sets"][t].tolist() == [idx[t, 0]]


def test_rounded_count_closed_forms():
    tile = 128
    big = 10 ** 6
    # nearest, half up; over one full period the total bias is exactly tile/2
    assert sum(O.rounded_count(c, tile, O.ROUND_NEAREST, big) - c for c in range(tile)) == tile // 2
    assert O.rounded_count(63, tile, O.ROUND_NEAREST, big) == 0
    assert O.rounded_count(64, tile, O.ROUND_NEAREST, big) == 128
    assert O.rounded_count(191, tile, O.ROUND_NEAREST, big) == 128
    assert O.rounded_count(1, tile, O.ROUND_UP, big) == 128
    assert O.rounded_count(128, tile, O.ROUND_UP, big) == 128
    assert O.rounded_count(300, tile, O.ROUND_NEAREST, 330) == 256   # capped at tile*floor(T/tile)
    assert O.rounded_count(77, tile, O.ROUND_OFF, big) == 77


def test_rounded_forward_weights_and_empty_sets():
    """In rounding mode a token may lose all its experts (y_t = 0) or gain
    some; its weights are a softmax over its final set."""
    inp = _rand_layer(24, 16, 8, 3, seed=6)
    toks, sets, ws = O.route(inp["x"], inp["Wr"], None, 1, tile=16, mode=O.ROUND_NEAREST)
    sizes = [len(s) for s in sets]
    for s, w in zip(sets, ws):
        if len(s):
            assert math.isclose(float(np.sum(w)), 1.0, rel_tol=1e-12)
    y = O.moe_forward(inp["x"], inp["Wr"], None, inp["W1"], inp["W3"], inp["W2"], k=1, tile=16,
                      mode=O.ROUND_NEAREST)
    for t, sz in enumerate(sizes):
        if sz == 0:
            assert np.all(y[t] == 0.0)
    assert sum(sizes) % 16 == 0


def test_splitmix64_published_sequence():
    # the first outputs of SplitMix64 started from state 0 (each call adds the
    # golden-ratio increment to the state before mixing)
    expected = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    state = 0
    for want in expected:
        assert O.splitmix64(state) == want
        state = (state + 0x9E3779B97F4A7C15) & O.MASK64


def test_stochastic_rounding_keeps_expected_count():
    tile, big = 128, 10 ** 6
    for c in (0, 1, 37, 64, 127, 128, 300):
        vals = [O.rounded_count(c, tile, O.ROUND_STOCHASTIC, big, e=e, seed=s) for s in range(8) for e in range(512)]
        lo = tile * (c // tile)
        assert set(vals) <= {lo, lo + tile}
        if c % tile == 0:
            assert set(vals) == {c}
        mean = sum(vals) / len(vals)
        # 4096 Bernoulli draws: std of the mean <= tile * 0.5 / 64
        assert abs(mean - c) <= 4 * tile * 0.5 / 64, (c, mean)


@pytest.mark.parametrize("T,E,k,tile,seed", [(40, 5, 2, 8, 0), (64, 6, 3, 8, 7), (200, 9, 2, 16, 3)])
def test_stochastic_token_rounding_brute_force(T, E, k, tile, seed):
    L = grid_logits(T, E, seed=300 + seed)
    idx = O.topk(L, k)
    r = _check_rounding(L, idx, tile, O.ROUND_STOCHASTIC, seed=seed)
    assert np.all(r["counts"] % tile == 0)
    member0 = np.zeros((T, E), bool)
    member0[np.repeat(np.arange(T), k), idx.reshape(-1)] = True
    c0 = member0.sum(0)
    for e in range(E):
        assert abs(int(r["counts"][e]) - int(c0[e])) < tile


# ------------------------------------------------------------------ FP8 e4m3
def _e4m3_brute(v):
    """Nearest value of the format by exhaustive search over all values;
    ties to the even mantissa (even index in the ascending value list, since
    each binade holds 8 mantissas), beyond 448 saturated."""
    vals = O.e4m3_values()
    out = np.empty_like(v)
    for i, x in enumerate(v):
        a = min(abs(x), 448.0)
        d = np.abs(vals - a)
        best = np.flatnonzero(d == d.min())
        j = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        out[i] = np.copysign(vals[j], x)
    return out


def test_e4m3_value_set():
    vals = O.e4m3_values()
    assert len(vals) == 127 and vals[0] == 0.0 and vals[-1] == 448.0
    assert np.all(np.diff(vals) > 0)
    assert vals[1] == 2.0 ** -9 and vals[8] == 2.0 ** -6 and 1.0 in vals


def test_e4m3_round_fixed_points_and_saturation():
    vals = O.e4m3_values()
    assert np.array_equal(O.e4m3_round(vals), vals)
    assert np.array_equal(O.e4m3_round(-vals), -vals)
    assert np.all(O.e4m3_round(np.array([448.5, 470.0, 1e6, -500.0])) == np.array([448, 448, 448, -448]))
    assert np.isnan(O.e4m3_round(np.array([np.nan])))[0]


def test_e4m3_round_matches_brute_force():
    rng = np.random.default_rng(7)
    vals = O.e4m3_values()
    mids = (vals[1:] + vals[:-1]) / 2
    v = np.concatenate([rng.standard_normal(2000) * 10 ** rng.uniform(-4, 2.8, 2000), mids, -mids,
                        mids * (1 + 1e-12), mids * (1 - 1e-12)])
    assert np.array_equal(O.e4m3_round(v), _e4m3_brute(v))


def test_quantize_rows_scale_and_range():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((50, 96)).astype(np.float32)
    X[4] = 0.0
    q, s = O.quantize_rows_e4m3(X)
    assert np.all(np.abs(q) <= 448) and s[4] == 1.0 and np.all(q[4] == 0)
    amax = np.abs(X).max(axis=1)
    assert np.array_equal(s[amax > 0], (amax[amax > 0] / np.float32(448)).astype(np.float32).astype(np.float64))
    assert np.all(np.abs(q[amax > 0]).max(axis=1) == 448.0)
    # the dequantised rows are within half an e4m3 step (2^-4 relative) of x
    Xh = q * s[:, None]
    assert np.all(np.abs(Xh - X) <= 2.0 ** -4 * np.abs(X) + 2.0 ** -10 * s[:, None] + 1e-12)


def test_fp8_forward_on_representable_inputs_equals_plain_forward():
    """Token rows with entries in {0, +-1/2, +-1} and weight columns with
    entries in {0, +-c_j/2, +-c_j} are representable up to the fp32 scale
    (x/s lands on 224 or 448): the FP8 layer equals the plain one to fp32
    rounding of the scales.  Quantising weight rows instead of output columns
    does not (the column maxima c_j in {0.7, 1, 1.1, 1.3} put w/amax off the
    e4m3 grid)."""
    rng = np.random.default_rng(11)
    T, d, n, E, k = 40, 32, 24, 4, 2
    x = rng.choice([0.0, 0.5, -0.5, 1.0, -1.0], size=(T, d))
    x[:, 0] = 1.0
    c = rng.choice([0.7, 1.0, 1.1, 1.3], size=(E, 1, n))
    W1 = rng.choice([0.0, 0.5, -0.5, 1.0, -1.0], size=(E, d, n)) * c
    W3 = rng.choice([0.0, 0.5, -0.5, 1.0, -1.0], size=(E, d, n)) * c[:, :, ::-1]
    W1[:, 0, :] = c[:, 0, :]
    W3[:, 0, :] = c[:, 0, ::-1]
    W2 = rng.standard_normal((E, n, d)) / np.sqrt(n)
    Wr = rng.standard_normal((d, E))
    y = O.moe_forward(x, Wr, None, W1, W3, W2, k)
    y8 = O.moe_forward_fp8(x, Wr, None, W1, W3, W2, k)
    assert np.allclose(y8, y, rtol=1e-5, atol=1e-6 * np.abs(y).max())
    # quantising W rows (over n) instead of columns gives a different layer
    bad = [O.dequantized_rows_e4m3(W1[e]) for e in range(E)]
    assert not all(np.allclose(b, O.quantized_expert_weights(W1[e], W3[e])[0]) for e, b in enumerate(bad))


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(5)
    a = np.concatenate([rng.standard_normal(20000) * 10 ** rng.uniform(-6, 6, 20000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0]])
    ref = torch.from_numpy(a).to(torch.float32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(O.bf16_round(a), ref)


def test_fp8_down_weight_one_scale_per_output_channel():
    """Each output channel (column of W2e [n, d]) has its own scale: its
    largest element codes to exactly 448, and every element is within half
    an e4m3 step of that channel's scale."""
    rng = np.random.default_rng(8)
    W = rng.standard_normal((24, 40)) / 5 * 10.0 ** rng.uniform(-2, 2, size=40)[None, :]
    Wh = O.quantized_expert_down_weight(W)
    s = (np.abs(W).max(axis=0).astype(np.float32) / np.float32(448)).astype(np.float64)
    codes = Wh / s[None, :]
    assert np.all(np.abs(np.abs(codes).max(axis=0) - 448) < 1e-3)
    assert np.all(np.abs(Wh - W) <= 2.0 ** -4 * np.abs(W) + 2.0 ** -9 * s[None, :] + 1e-12)


def test_fp8_down_weight_outlier_channel_stays_local():
    """A planted outlier channel, 10^5 times the others, coarsens only its own
    channel: the other channels keep e4m3's relative precision.  One scale for
    the whole matrix (the failing control) would push them into e4m3's
    subnormal range."""
    rng = np.random.default_rng(9)
    W = rng.standard_normal((64, 32)) / 8
    W[:, 5] *= 1e5
    rel = lambda a, b: np.abs(a - b) / np.abs(b)  # noqa: E731
    per_channel = O.quantized_expert_down_weight(W)
    others = np.delete(np.arange(32), 5)
    assert rel(per_channel[:, others], W[:, others]).max() <= 2.0 ** -4 + 1e-12
    one_scale = O.dequantized_rows_e4m3(W.reshape(1, -1)).reshape(W.shape)
    assert rel(one_scale[:, others], W[:, others]).max() > 0.25


def test_fp8_full_layer_within_quantisation_bound_of_fp8_up_layer():
    """Quantising h per row and W2 per output channel moves each output by at most the
    e4m3 half-step of both factors: |dy| <= sum_e w_e (|h_e| |W2_e|) * 2^-3 (+ tiny)."""
    rng = np.random.default_rng(4)
    T, d, n, E, k = 30, 48, 40, 5, 2
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((d, E)) / np.sqrt(d)
    W1 = rng.standard_normal((E, d, n)) / np.sqrt(d)
    W3 = rng.standard_normal((E, d, n)) / np.sqrt(d)
    W2 = rng.standard_normal((E, n, d)) / np.sqrt(n)
    y8 = O.moe_forward_fp8(x, Wr, None, W1, W3, W2, k)
    y8f = O.moe_forward_fp8_full(x, Wr, None, W1, W3, W2, k)
    _, sets, weights = O.route(x, Wr, None, k)
    xq = O.dequantized_rows_e4m3(x)
    bound = np.zeros((T, d))
    for t in range(T):
        for e, w in zip(sets[t], weights[t]):
            W1h, W3h = O.quantized_expert_weights(W1[e], W3[e])
            h = O.expert_hidden(xq[t:t + 1], W1h, W3h)
            bound[t] += w * (np.abs(h) @ np.abs(W2[e]))[0]
    diff = np.abs(y8f - y8)
    assert np.all(diff <= 2.0 ** -3 * bound + 1e-9)
    assert diff.max() > 0  # the down-projection really is quantised
