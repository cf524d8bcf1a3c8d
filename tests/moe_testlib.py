"""Shared helpers of the parity tests: tolerances and comparisons.

Floating-point outputs are bf16 with fp32 accumulation; the bar is
  max |y - y_ref| <= 2e-2 * rms(y_ref)   and   sum|y - y_ref| / sum|y_ref| <= 5e-3
(y_ref from the fp64 oracle).  Integer outputs (expert ids, counts, offsets,
permutations) must be identical.
"""
import numpy as np
import torch

MAX_ERR_RMS = 2e-2
MEAN_REL = 5e-3


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def err_stats(y, y_ref):
    y, y_ref = to64(y), to64(y_ref)
    diff = np.abs(y - y_ref)
    rms = float(np.sqrt(np.mean(y_ref ** 2))) if y_ref.size else 0.0
    max_err = float(diff.max()) if diff.size else 0.0
    denom = float(np.abs(y_ref).sum())
    mean_rel = float(diff.sum() / denom) if denom > 0 else float(diff.sum())
    return {"max_err": max_err, "rms": rms, "max_over_rms": max_err / rms if rms > 0 else max_err,
            "mean_rel": mean_rel}


def assert_moe_close(y, y_ref, what="y"):
    s = err_stats(y, y_ref)
    assert np.all(np.isfinite(to64(y))), f"{what}: non-finite values"
    assert s["max_err"] <= MAX_ERR_RMS * s["rms"] + 1e-30, f"{what}: {s}"
    assert s["mean_rel"] <= MEAN_REL, f"{what}: {s}"
    return s


def robust_tokens(L64: np.ndarray, k: int, margin: float) -> np.ndarray:
    """Tokens whose top-k set is decided by more than `margin` (the gap between
    the k-th and (k+1)-th largest fp64 logit).  For these the set cannot
    depend on fp32 rounding of the logits."""
    T, E = L64.shape
    if k >= E:
        return np.ones(T, dtype=bool)
    part = -np.sort(-L64, axis=1)
    return (part[:, k - 1] - part[:, k]) > margin


def valid_topk(L64_row: np.ndarray, chosen, margin: float) -> bool:
    """A selected set is a valid top-k under a logit perturbation <= margin."""
    chosen = np.asarray(chosen)
    rest = np.setdiff1d(np.arange(L64_row.size), chosen)
    if rest.size == 0:
        return True
    return float(L64_row[chosen].min()) >= float(L64_row[rest].max()) - 2 * margin


# Gradients of the backward pass: each element is a sum of products whose
# bf16-stored operand (the activation gradient, w h) carries one rounding of
# relative size <= 2^-8, the rest being fp32 arithmetic.  The bar is the
# elementwise bound |g - g_ref| <= 2^-7 * sum|terms| (twice the rounding, for
# the fp32 parts) plus the layer's mean relative error bound.
GRAD_REL = 2.0 ** -7


def assert_grad_close(g, g_ref, mag, what="grad"):
    g64, r64, m64 = to64(g), to64(g_ref), to64(mag)
    assert np.all(np.isfinite(g64)), f"{what}: non-finite values"
    s = err_stats(g64, r64)
    excess = np.abs(g64 - r64) - GRAD_REL * m64
    assert np.all(excess <= 1e-6 * s["rms"] + 1e-30), f"{what}: {s}, worst excess {excess.max():.3e}"
    assert s["mean_rel"] <= MEAN_REL, f"{what}: {s}"
    return s


def stratified_tokens(offsets, row_token, T, seed, minimum=1024, cap_loaded=2048, per_expert=2, block=128):
    """Token sample that reaches every expert's GEMM tiles: for each expert
    with rows, the token of its first row, of its last row and of a random row
    in its last `block`-row block, plus `per_expert` random rows; every token
    of the least- and the most-loaded expert (at most `cap_loaded` of each,
    drawn at random beyond that); then random tokens up to `minimum`.
    offsets [E+1] and row_token [R] are the permutation's arrays (rows of an
    expert contiguous).  Returns sorted unique token ids."""
    rng = np.random.default_rng(seed)
    offsets = np.asarray(offsets, dtype=np.int64)
    row_token = np.asarray(row_token, dtype=np.int64)
    counts = np.diff(offsets)
    toks = set()
    for e in np.flatnonzero(counts > 0):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        last_lo = lo + ((hi - lo - 1) // block) * block
        toks.update(int(row_token[r]) for r in (lo, hi - 1, int(rng.integers(last_lo, hi))))
        toks.update(int(row_token[r]) for r in rng.integers(lo, hi, size=per_expert))
    nz = np.flatnonzero(counts > 0)
    for e in {int(nz[np.argmin(counts[nz])]), int(np.argmax(counts))}:
        rows = row_token[offsets[e]:offsets[e + 1]]
        if rows.size > cap_loaded:
            rows = rng.choice(rows, size=cap_loaded, replace=False)
        toks.update(int(t) for t in rows)
    if len(toks) < min(minimum, T):
        rest = np.setdiff1d(np.arange(T), np.fromiter(toks, dtype=np.int64))
        toks.update(int(t) for t in rng.choice(rest, size=min(minimum, T) - len(toks), replace=False))
    return np.array(sorted(toks), dtype=np.int64)
