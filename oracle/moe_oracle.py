"""fp64 CPU oracle for the single-GPU MoE-layer forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the test suite, `__graft_entry__.smoke()` and the
CPU-baseline / reference arm of `bench.py` use it.  It shares no code with the
CUDA library (no headers, helpers, tables or generators); both sides are fed by
the seeded generators in `mixture_experts_layer_93_b300/inputs.py`, which hold
none of the method's arithmetic.

What it computes is the plain definition of an MoE layer forward, written out
step by step in fp64 with numpy (matmul, lexsort and exp are the only library
primitives used):

  1. gate network: router logits L = x Wr (+ b)
        ("MoE架构的物理瓶颈与扩展限制解析", section 工作原理, moe_forward
        pseudocode, step 1; "硬件加速的考量", section 自定义核与核融合, step 1)
  2. top-k expert selection per token
        (same pseudocode, `top_k(router_logits)`; 自定义核与核融合 step 2)
  3. gather/permutation: rows grouped per expert so each expert's tokens are
     contiguous ("SonicMoE: 加速 MoE 模型的 IO 与 Tile 感知优化", section
     技术细节 / Gather 与加载融合, the "contiguous packed input" mode)
  4. expert SwiGLU FFN (section 关键 Kernel 对比, row "SwiGLU 融合";
     自定义核与核融合 step 4)
  5. gate-score-weighted combine (自定义核与核融合 step 5)
  6. optional token rounding of each expert's token count to a tile multiple
     (SonicMoE page, section "3. Token Rounding 路由算法")
  7. the backward pass of the same layer by recomputation (SonicMoE page,
     "SonicMoE 的三大核心优化" item 1 and section 反向传播优化)

Readings of the pages (where they are silent or at odds):
  * Selection precision: a top-k choice is taken on fp32 logits (the kernel's
    precision); the fp64 logits are rounded to fp32 before ranking.  Gate
    weights are the fp64 softmax over the selected logits.
  * Ties in top-k go to the lower expert id; -0.0 equals +0.0.
  * Gate weights: softmax over the k selected logits (renormalised), which
    is the same function as softmax-over-all-then-top-k-then-renormalise.
  * SwiGLU: h = silu(x W1) * (x W3), silu(z) = z / (1 + exp(-z)); W1 is the
    gated branch, W3 the linear one; o = h W2.
  * Token rounding: the SonicMoE page asks for rounding "up" to a tile
    multiple, for at most one tile of deviation from top-k, and for an
    unchanged expected total.  Always rounding up raises the total, so the
    default mode rounds to the NEAREST multiple (half up); "up" is kept as the
    literal variant, and "stochastic" rounds up with probability
    (c mod tile)/tile (SplitMix64 on the counter seed*2^32+e), which keeps the
    expected total exactly.  Counts are capped at tile*floor(T/tile).  When the
    rounded count c' exceeds c, the c'-c not-yet-routed tokens with the
    highest L[t,e] join (ties: lower t first); when c' < c, the c-c' routed
    tokens with the lowest L[t,e] leave (ties: higher t leaves first).  Each
    expert is rounded from the original top-k sets.  A token's final set is
    ordered by (L desc, id asc) and weighted by softmax over that set; an empty
    set gives y_t = 0.

  * FP8 expert GEMMs (the FP8 quantisation the pages name for MoE compute
    and communication, "硬件加速的考量", section 量化; they fix no recipe):
    e4m3 codes with one fp32 scale per quantised row, scale =
    fp32(amax / 448) and code = e4m3(fp32(x * fp32(448 / amax))), rounded to
    nearest with ties to even and saturated to +-448 (an all-zero row has
    scale 1 and codes 0).  Up-projection: rows are tokens (activations) and
    output channels (a row of the packed W1/W3).  Down-projection (the
    "fp8" layer): rows of the bf16 hidden h (as the up-projection stores it)
    and the output channels of W2 (each column of W2e [n, d], quantised over
    its n elements).  The GEMMs run on the dequantised values code * scale;
    routing and the combine stay as above.
  * Backward: the pages give no formulas, only that the gradients stay
    those of the MoE formula while intermediates are recomputed.  The
    reading is the exact gradient of the forward above for a given dy = dL/dy,
    with the selected sets (and any rounding) held fixed: the selection is
    piecewise constant, so it passes no gradient.  The router gradient goes
    through the renormalised softmax of the selected logits only.

Pins (tests/test_oracle.py): brute-force k-subset top-k; the closed form
w0 = sigmoid(L0 - L1) at k=2; numpy's stable argsort for the permutation;
index-arithmetic SwiGLU on one-nonzero-per-column weights (catches a
transposed operand); E=1,k=1 == dense FFN; identical experts == dense FFN;
relabelling invariance; W2=0 -> 0; token-rounding invariants checked by
brute force on tiny inputs; e4m3 rounding against a brute-force nearest
search over all values of the format; the backward pass against central
finite differences of moe_forward on tiny layers, the zero router gradient
at k=1, the dense-FFN case and the zero sum of each token's logit gradient.
No function here is unpinned.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64

ROUND_OFF = "off"
ROUND_NEAREST = "nearest"
ROUND_UP = "up"
ROUND_STOCHASTIC = "stochastic"

MASK64 = (1 << 64) - 1


def splitmix64(state: int) -> int:
    """One output of SplitMix64 (Steele, Lea, Flood, "Fast splittable
    pseudorandom number generators", OOPSLA 2014) for the given 64-bit state:
    the state is advanced by the golden-ratio increment, then mixed."""
    z = (state + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def stochastic_round_up(c: int, tile: int, seed: int, e: int) -> bool:
    """Whether expert e's count rounds up in the stochastic mode: with
    probability (c mod tile) / tile, decided by the top 32 bits h of
    SplitMix64(seed * 2^32 + e) as h * tile < (c mod tile) * 2^32."""
    h = splitmix64(((seed & 0xFFFFFFFF) << 32) | (e & 0xFFFFFFFF)) >> 32
    return h * tile < (c % tile) << 32


def _f64(a) -> np.ndarray:
    """bf16/fp32 torch tensor or numpy array -> fp64 numpy (exact widening)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            # move in the stored dtype, widen on the host
            return a.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a, dtype=F64)


# --------------------------------------------------------------------------
# 1. gate network
# --------------------------------------------------------------------------
def router_logits(x, Wr, bias=None) -> np.ndarray:
    """L[t, e] = sum_i x[t, i] * Wr[i, e] + bias[e], in fp64.

    Gate network of the moe_forward pseudocode ("MoE架构的物理瓶颈与扩展限制解析",
    section 工作原理, step 1)."""
    L = _f64(x) @ _f64(Wr)
    if bias is not None:
        L = L + _f64(bias)[None, :]
    return L


def decision_logits(L) -> np.ndarray:
    """The logits the selection ranks: fp32, the kernel's precision."""
    return np.asarray(L, dtype=F64).astype(np.float32)


# --------------------------------------------------------------------------
# 2. top-k and gate weights
# --------------------------------------------------------------------------
def topk(L, k: int) -> np.ndarray:
    """idx[t, :k]: the k experts with the largest L[t, e], in descending order
    of L; equal values are ordered by ascending expert id.  int32 [T, k].

    `top_k(router_logits)` of the moe_forward pseudocode (page above, 工作原理)."""
    L = np.asarray(L)
    T, E = L.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    ids = np.broadcast_to(np.arange(E), (T, E))
    # lexsort: last key is primary -> sort by -L ascending, then by id ascending
    order = np.lexsort((ids, -L.astype(F64)), axis=-1)
    return order[:, :k].astype(np.int32)


def softmax(v) -> np.ndarray:
    v = np.asarray(v, dtype=F64)
    if v.size == 0:
        return v.copy()
    z = np.exp(v - v.max())
    return z / z.sum()


def gate_weights(L, idx) -> np.ndarray:
    """w[t, j] = softmax over the selected logits L[t, idx[t, :]] (renormalised
    gating), fp64 [T, k]."""
    L = np.asarray(L, dtype=F64)
    Ls = np.take_along_axis(L, np.asarray(idx, dtype=np.int64), axis=1)
    z = np.exp(Ls - Ls.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


# --------------------------------------------------------------------------
# 3. permutation (stable grouping of assignments by expert)
# --------------------------------------------------------------------------
def permute(idx, E: int):
    """Group the A = T*k assignments a = t*k + j by expert, stably.

    Returns (counts[E], offsets[E+1], src[A], dst[A]) as int64 arrays, with
    src[row] = a (rows of expert e are offsets[e]..offsets[e+1]-1, in ascending
    a) and dst[a] = row."""
    flat = np.asarray(idx).reshape(-1)
    groups = [np.flatnonzero(flat == e) for e in range(E)]
    counts = np.array([g.size for g in groups], dtype=np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    src = np.concatenate(groups).astype(np.int64) if groups else np.zeros(0, np.int64)
    dst = np.empty_like(src)
    dst[src] = np.arange(src.size)
    return counts, offsets, src, dst


# --------------------------------------------------------------------------
# 6. token rounding
# --------------------------------------------------------------------------
def rounded_count(c: int, tile: int, mode: str, T: int, e: int = 0, seed: int = 0) -> int:
    """Per-expert token count after rounding to a multiple of `tile`.  The
    stochastic mode rounds up with probability (c mod tile)/tile, so the
    expected count, and total, is unchanged."""
    if mode == ROUND_OFF:
        return int(c)
    if mode == ROUND_NEAREST:
        c2 = tile * ((c + tile // 2) // tile)
    elif mode == ROUND_UP:
        c2 = tile * (-(-c // tile))
    elif mode == ROUND_STOCHASTIC:
        c2 = tile * (c // tile) + (tile if stochastic_round_up(c, tile, seed, e) else 0)
    else:
        raise ValueError(mode)
    return int(min(c2, tile * (T // tile)))


def token_round(L, idx, tile: int, mode: str, seed: int = 0):
    """Token rounding (SonicMoE page, "3. Token Rounding 路由算法").

    Returns a dict with
      member  [T, E] bool   final membership
      counts  [E]           rounded counts (multiples of tile)
      sets    list of T int arrays: each token's experts, (L desc, id asc)
      added / dropped: per-expert arrays of token ids
    L is the fp32 decision matrix (ranked in fp64, which is exact for fp32)."""
    L = np.asarray(L, dtype=F64)
    T, E = L.shape
    idx = np.asarray(idx)
    member = np.zeros((T, E), dtype=bool)
    member[np.repeat(np.arange(T), idx.shape[1]), idx.reshape(-1)] = True
    final = member.copy()
    counts0 = member.sum(axis=0)
    added, dropped = [], []
    for e in range(E):
        c = int(counts0[e])
        c2 = rounded_count(c, tile, mode, T, e, seed)
        add = np.zeros(0, np.int64)
        drop = np.zeros(0, np.int64)
        if c2 > c:
            cand = np.flatnonzero(~member[:, e])
            order = np.lexsort((cand, -L[cand, e]))      # L desc, then t asc
            add = cand[order[: c2 - c]]
            final[add, e] = True
        elif c2 < c:
            routed = np.flatnonzero(member[:, e])
            order = np.lexsort((routed, -L[routed, e]))  # best first
            drop = routed[order[c2:]]                    # worst c-c2 leave
            final[drop, e] = False
        added.append(add)
        dropped.append(drop)
    sets = []
    for t in range(T):
        es = np.flatnonzero(final[t])
        es = es[np.lexsort((es, -L[t, es]))] if es.size else es
        sets.append(es.astype(np.int64))
    return {"member": final, "counts": final.sum(axis=0).astype(np.int64),
            "sets": sets, "added": added, "dropped": dropped}


# --------------------------------------------------------------------------
# 4. expert SwiGLU FFN
# --------------------------------------------------------------------------
def silu(z) -> np.ndarray:
    z = np.asarray(z, dtype=F64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_hidden(xr, W1e, W3e) -> np.ndarray:
    """h = silu(xr W1e) * (xr W3e), fp64 [m, n]."""
    xr = _f64(xr)
    return silu(xr @ _f64(W1e)) * (xr @ _f64(W3e))


def expert_out(h, W2e) -> np.ndarray:
    """o = h W2e, fp64 [m, d]."""
    return _f64(h) @ _f64(W2e)


# --------------------------------------------------------------------------
# 5. full layer forward
# --------------------------------------------------------------------------
def route(x, Wr, bias, k: int, tile: int = 128, mode: str = ROUND_OFF, tokens=None,
          logits=None, seed: int = 0):
    """Per-token expert sets and gate weights.

    Without rounding only the tokens in `tokens` (all when None) are routed.
    With rounding every token is routed (rounding couples tokens through the
    per-expert counts) and the requested subset is returned.  `logits`, when
    given, replaces the gate network (fp32 decision logits, e.g. synthetic).
    Returns (tokens, sets, weights): lists of int64 / fp64 arrays."""
    x64 = None
    if logits is None:
        x64 = _f64(x)
    T = (x64.shape[0] if logits is None else np.asarray(logits).shape[0])
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    if mode == ROUND_OFF:
        if logits is None:
            L64 = router_logits(x64[tokens], Wr, bias)
        else:
            L64 = np.asarray(logits, dtype=F64)[tokens]
        Ld = decision_logits(L64)
        idx = topk(Ld, k)
        w = gate_weights(L64, idx)
        return tokens, [idx[i].astype(np.int64) for i in range(len(tokens))], [w[i] for i in range(len(tokens))]
    L64 = router_logits(x64, Wr, bias) if logits is None else np.asarray(logits, dtype=F64)
    Ld = decision_logits(L64)
    idx = topk(Ld, k)
    r = token_round(Ld, idx, tile, mode, seed)
    sets = [r["sets"][t] for t in tokens]
    weights = [softmax(L64[t, s]) for t, s in zip(tokens, sets)]
    return tokens, sets, weights


def moe_forward(x, Wr, bias, W1, W3, W2, k: int, tile: int = 128, mode: str = ROUND_OFF,
                tokens=None, return_routing: bool = False, seed: int = 0, routing=None, experts=None):
    """y[t] = sum_{e in S_t} w_te * FFN_e(x[t]) for the requested tokens, fp64.

    Dataflow of the moe_forward pseudocode ("MoE架构的物理瓶颈与扩展限制解析",
    section 工作原理) with both all-to-all steps removed (one GPU), and the
    five steps of the fused kernel ("硬件加速的考量", section 自定义核与核融合).

    `routing`, when given, is the (tokens, sets, weights) that `route` returned
    for these arguments and is used instead of routing again.  `experts`, when
    given, restricts the sum to the experts listed (the terms of the others are
    left out), so y over a partition of the experts adds up to the full y."""
    if routing is None:
        routing = route(x, Wr, bias, k, tile, mode, tokens, seed=seed)
    tokens, sets, weights = routing
    x64 = _f64(x)
    d = x64.shape[1]
    y = np.zeros((len(tokens), d), dtype=F64)
    E = W1.shape[0]
    pos_of = {e: [] for e in range(E)}
    w_of = {e: [] for e in range(E)}
    for p, (s, w) in enumerate(zip(sets, weights)):
        for e, we in zip(s, w):
            pos_of[int(e)].append(p)
            w_of[int(e)].append(we)
    for e in (range(E) if experts is None else sorted({int(v) for v in experts})):
        if not pos_of[e]:
            continue
        pos = np.array(pos_of[e], dtype=np.int64)
        h = expert_hidden(x64[tokens[pos]], W1[e], W3[e])
        o = expert_out(h, W2[e])
        np.add.at(y, pos, np.array(w_of[e])[:, None] * o)
    if return_routing:
        return y, (tokens, sets, weights)
    return y


def dense_swiglu_ffn(x, W1e, W3e, W2e) -> np.ndarray:
    """A dense (one-expert) SwiGLU FFN, the E=1/k=1 special case."""
    return expert_out(expert_hidden(x, W1e, W3e), W2e)


# --------------------------------------------------------------------------
# 7. FP8 (e4m3) up-projection
# --------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_values() -> np.ndarray:
    """Every finite non-negative e4m3 value, from the format's definition:
    1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities; an
    exponent field of 0 is subnormal (m/8 * 2^-6) and the pattern with
    exponent field 15 and mantissa 7 is NaN."""
    vals = []
    for ef in range(16):
        for m in range(8):
            if ef == 15 and m == 7:
                continue
            vals.append(m / 8.0 * 2.0 ** -6 if ef == 0 else (1.0 + m / 8.0) * 2.0 ** (ef - 7))
    return np.array(vals, dtype=F64)


def e4m3_round(v) -> np.ndarray:
    """Nearest e4m3 value, ties to the even mantissa, saturated to +-448
    (NaN stays NaN).  In the binade [2^e, 2^(e+1)), e >= -6, values are
    multiples of 2^(e-3); below 2^-6 of 2^-9.  Division by that power of two is
    exact, and numpy's round() breaks ties to even."""
    v = np.asarray(v, dtype=F64)
    a = np.abs(v)
    _, ex = np.frexp(a)                         # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex.astype(np.int64) - 1, -6)
    q = np.ldexp(1.0, e - 3)
    r = np.minimum(np.round(a / q) * q, E4M3_MAX)
    return np.where(np.isnan(v), np.nan, np.copysign(r, v))


def quantize_rows_e4m3(X):
    """(codes, scales) of each row of X: scale = fp32(amax / 448) and
    code = e4m3(fp32(x * fp32(448 / amax))), every fp32 operation rounded to
    nearest; an all-zero row has scale 1 and codes 0.  Codes are returned as
    their exact fp64 values."""
    X32 = np.asarray(_f64(X), dtype=np.float32)
    amax = np.max(np.abs(X32), axis=1)
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1.0)).astype(np.float32)
    s = np.where(nz, (safe / np.float32(E4M3_MAX)).astype(np.float32), np.float32(1.0)).astype(np.float32)
    inv = (np.float32(E4M3_MAX) / safe).astype(np.float32)
    v = (X32 * inv[:, None]).astype(np.float32)
    q = np.where(nz[:, None], e4m3_round(v.astype(F64)), 0.0)
    return q, s.astype(F64)


def dequantized_rows_e4m3(X) -> np.ndarray:
    """code * scale for each row of X (exact in fp64)."""
    q, s = quantize_rows_e4m3(X)
    return q * s[:, None]


def quantized_expert_weights(W1e, W3e):
    """W1e, W3e [d, n] as the FP8 path uses them: each output column
    quantised over d (a row of the packed weights), dequantised."""
    W1h = dequantized_rows_e4m3(_f64(W1e).T).T
    W3h = dequantized_rows_e4m3(_f64(W3e).T).T
    return W1h, W3h


def moe_forward_fp8(x, Wr, bias, W1, W3, W2, k: int, tokens=None):
    """The layer with the FP8 up-projection: routing on x as in moe_forward,
    the up-projection on the dequantised token rows and weight columns, the
    down-projection and combine as in moe_forward.  fp64 result."""
    tokens, sets, weights = route(x, Wr, bias, k, tokens=tokens)
    x64 = _f64(x)
    xq = dequantized_rows_e4m3(x64[tokens])
    d = x64.shape[1]
    y = np.zeros((len(tokens), d), dtype=F64)
    E = W1.shape[0]
    pos_of = {e: [] for e in range(E)}
    w_of = {e: [] for e in range(E)}
    for p, (st, w) in enumerate(zip(sets, weights)):
        for e, we in zip(st, w):
            pos_of[int(e)].append(p)
            w_of[int(e)].append(we)
    for e in range(E):
        if not pos_of[e]:
            continue
        pos = np.array(pos_of[e], dtype=np.int64)
        W1h, W3h = quantized_expert_weights(W1[e], W3[e])
        h = expert_hidden(xq[pos], W1h, W3h)
        o = expert_out(h, W2[e])
        np.add.at(y, pos, np.array(w_of[e])[:, None] * o)
    return y


def bf16_round(a) -> np.ndarray:
    """Round fp64 values to bf16 (nearest, ties to even) and back: the
    precision the hidden activations are stored in between the GEMMs."""
    a = np.asarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(F64)


def quantized_expert_down_weight(W2e) -> np.ndarray:
    """W2e [n, d] as the FP8 down-projection uses it: each output channel (a
    column, n elements) quantised with its own scale, dequantised."""
    return dequantized_rows_e4m3(_f64(W2e).T).T


def moe_forward_fp8_full(x, Wr, bias, W1, W3, W2, k: int, tokens=None):
    """The layer with both expert GEMMs in e4m3: the up-projection as in
    moe_forward_fp8; h rounded to bf16 (as stored), quantised per row, and
    multiplied by W2 quantised per output channel.  fp64 result."""
    tokens, sets, weights = route(x, Wr, bias, k, tokens=tokens)
    x64 = _f64(x)
    xq = dequantized_rows_e4m3(x64[tokens])
    d = x64.shape[1]
    y = np.zeros((len(tokens), d), dtype=F64)
    E = W1.shape[0]
    pos_of = {e: [] for e in range(E)}
    w_of = {e: [] for e in range(E)}
    for p, (st, w) in enumerate(zip(sets, weights)):
        for e, we in zip(st, w):
            pos_of[int(e)].append(p)
            w_of[int(e)].append(we)
    for e in range(E):
        if not pos_of[e]:
            continue
        pos = np.array(pos_of[e], dtype=np.int64)
        W1h, W3h = quantized_expert_weights(W1[e], W3[e])
        h = dequantized_rows_e4m3(bf16_round(expert_hidden(xq[pos], W1h, W3h)))
        o = expert_out(h, quantized_expert_down_weight(W2[e]))
        np.add.at(y, pos, np.array(w_of[e])[:, None] * o)
    return y



# --------------------------------------------------------------------------
# 8. backward pass
# --------------------------------------------------------------------------
def sigmoid(z) -> np.ndarray:
    z = np.asarray(z, dtype=F64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def moe_backward(x, Wr, bias, W1, W3, W2, dy, k: int, tile: int = 128, mode: str = ROUND_OFF,
                 seed: int = 0, logits=None, magnitudes: bool = False) -> dict:
    """Gradients of the scalar sum_t <dy[t], y[t]> with respect to every input
    of moe_forward, fp64.

    The SonicMoE page ("SonicMoE 的三大核心优化", item 1, and "反向传播优化")
    recomputes the forward's intermediates instead of caching them and keeps
    the gradients mathematically those of the MoE formula; the router
    gradient dS is formed without the expert outputs (the "dS 计算优化" row of
    the 关键 Kernel 对比 table).  Written out by the chain rule:

      per routed pair (t, e) with gate weight w, g = x W1e, u = x W3e,
      s = sigmoid(g), a = g s = silu(g), h = a u, o = h W2e:
        dW2e += h^T (w dy)            dh = w dy W2e^T
        du = dh a                     dg = dh u s (1 + g (1 - s))
        dW1e += x^T dg                dW3e += x^T du
        dx   += dg W1e^T + du W3e^T
        dw   = <dy, o> = <dy W2e^T, h>
      per token, over its selected set S (w = softmax of the logits on S):
        dL[t, i] = w_i (dw_i - sum_{j in S} w_j dw_j) for i in S, 0 elsewhere
      and through the gate network L = x Wr + b:
        dWr = x^T dL,  db = sum_t dL[t],  dx += dL Wr^T.

    The selection itself is piecewise constant in the logits, so no gradient
    flows through it (nor through token rounding's choice of sets).  Returns
    a dict with dx [T, d], dWr [d, E], db [E], dW1, dW3 [E, d, n], dW2 [E, n, d]
    and dL [T, E], dw (per token, the list of its set's dw).  `logits`, as in
    route(), replaces the gate network's output for the selection and the
    gate weights (dWr, db and the router part of dx still follow L = x Wr + b).
    With `magnitudes`, the dict also holds, for dx, dW1, dW3 and dW2, the sum
    of the absolute values of the terms each element adds up (the same
    products with every factor replaced by its magnitude): the scale an
    element's rounding error is measured against."""
    x64 = _f64(x)
    dy64 = _f64(dy)
    T, d = x64.shape
    E, _, n = np.shape(W1)
    tokens, sets, weights = route(x, Wr, bias, k, tile, mode, logits=logits, seed=seed)
    dx = np.zeros((T, d), dtype=F64)
    dW1 = np.zeros((E, d, n), dtype=F64)
    dW3 = np.zeros((E, d, n), dtype=F64)
    dW2 = np.zeros((E, n, d), dtype=F64)
    dw = [np.zeros(len(s), dtype=F64) for s in sets]
    if magnitudes:
        mag = {"dx": np.zeros((T, d)), "dW1": np.zeros((E, d, n)), "dW3": np.zeros((E, d, n)),
               "dW2": np.zeros((E, n, d))}
    for e in range(E):
        pairs = [(t, j) for t, s in enumerate(sets) for j, se in enumerate(s) if int(se) == e]
        if not pairs:
            continue
        ts = np.array([t for t, _ in pairs], dtype=np.int64)
        w = np.array([weights[t][j] for t, j in pairs], dtype=F64)
        W1e, W3e, W2e = _f64(W1[e]), _f64(W3[e]), _f64(W2[e])
        X = x64[ts]
        g, u = X @ W1e, X @ W3e
        s = sigmoid(g)
        a = g * s
        h = a * u
        dh_unweighted = dy64[ts] @ W2e.T          # dy W2e^T
        dW2[e] = h.T @ (w[:, None] * dy64[ts])
        dh = w[:, None] * dh_unweighted
        du = dh * a
        dg = dh * u * (s * (1.0 + g * (1.0 - s)))
        dW1[e] = X.T @ dg
        dW3[e] = X.T @ du
        np.add.at(dx, ts, dg @ W1e.T + du @ W3e.T)
        if magnitudes:
            aX = np.abs(X)
            mag["dW2"][e] = np.abs(h).T @ np.abs(w[:, None] * dy64[ts])
            mag["dW1"][e] = aX.T @ np.abs(dg)
            mag["dW3"][e] = aX.T @ np.abs(du)
            np.add.at(mag["dx"], ts, np.abs(dg) @ np.abs(W1e).T + np.abs(du) @ np.abs(W3e).T)
        dwe = np.sum(dh_unweighted * h, axis=1)   # <dy, h W2e>
        for (t, j), v in zip(pairs, dwe):
            dw[t][j] = v
    dL = np.zeros((T, E), dtype=F64)
    for t, (s, w) in enumerate(zip(sets, weights)):
        if len(s):
            dL[t, np.asarray(s, dtype=np.int64)] = w * (dw[t] - np.dot(w, dw[t]))
    dWr = x64.T @ dL
    db = dL.sum(axis=0)
    dx = dx + dL @ _f64(Wr).T
    out = {"dx": dx, "dWr": dWr, "db": db, "dW1": dW1, "dW3": dW3, "dW2": dW2, "dL": dL, "dw": dw,
           "sets": sets, "weights": weights}
    if magnitudes:
        mag["dx"] += np.abs(dL) @ np.abs(_f64(Wr)).T
        out.update({key + "_mag": v for key, v in mag.items()})
    return out
