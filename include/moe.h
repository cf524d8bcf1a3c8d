/*
 * moe.h — C ABI of libmoe.so: the forward pass of one Mixture-of-Experts
 * layer on one B300 GPU (sm_103a).
 *
 * The layer (dataflow of the moe_forward pseudocode in "MoE架构的物理瓶颈与扩展限制解析",
 * section 工作原理, with both all-to-all steps removed because every expert
 * lives on this GPU; step list of the fused kernel in "硬件加速的考量",
 * section 自定义核与核融合):
 *
 *   L      = x Wr + b                                  router logits      (moe_router_logits)
 *   S_t, w = top-k of L[t], softmax over the selected   gating             (moe_topk_gating)
 *   rows   = assignments grouped by expert (stable)     permutation        (moe_permute)
 *   h[r]   = silu(x[t_r] W1_e) * (x[t_r] W3_e)          up-projection      (moe_expert_up)
 *   ys[r]  = w_r * (h[r] W2_e)                          down-projection    (moe_expert_down)
 *   y[t]   = sum over t's rows of ys[r], fixed order    combine            (moe_combine)
 *
 * Precision: x, the expert weights and h are bf16; every product accumulates
 * in fp32 (tensor memory); ys is stored as fp16 and y is fp32
 * (moe_combine_bf16 / moe_forward_bf16 round it to bf16).
 *
 * Also here: e4m3 variants of the two expert GEMMs (the FP8 block below) and
 * the layer's backward pass by recomputation (moe_backward, at the end).
 *
 * The SwiGLU activation is fused into the up-projection's epilogue and the
 * gate weight into the down-projection's ("SonicMoE: 加速 MoE 模型的 IO 与 Tile
 * 感知优化", the "关键 Kernel 对比" table).  The gather of token rows can also be
 * fused into the up-projection's operand load (same page, "Gather 与加载融合";
 * moe_expert_up with gather = 1 or 2).  moe_forward fuses it (gather = 2,
 * wide tiles) where the up GEMM has two 256-wide n-blocks (n = 256), so each
 * row is gathered once; elsewhere it stages the rows with a token-order copy
 * kernel and loads them with tiled TMA (gather = 0), which measured faster on
 * B300 there (moe_forward_a_path).  The optional token rounding (same page, "3. Token
 * Rounding 路由算法") rounds each expert's row count to a multiple of a tile
 * (moe_token_round).
 *
 * Conventions (every entry point):
 *   - All tensor pointers are DEVICE pointers, 16-byte aligned, row-major and
 *     contiguous.  bf16 tensors are passed as `void*` (IEEE bfloat16 bits).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every launch
 *     goes onto it, in order; no entry point synchronises the stream except
 *     moe_check_device_status.
 *   - The caller allocates and owns every buffer, including the workspace.
 *     The library allocates nothing and frees nothing.
 *   - Arguments are validated on the host before anything is launched; a bad
 *     argument returns MOE_ERR_INVALID (or MOE_ERR_UNSUPPORTED / _WORKSPACE)
 *     and enqueues nothing.
 *   - A launch failure returns MOE_ERR_CUDA.  Problems the kernels detect
 *     (a bounded wait that ran out, an expert id out of range, a NaN logit) are
 *     recorded in a status word at the start of the workspace and read by
 *     moe_check_device_status.
 *   - Results are deterministic: identical inputs give bitwise identical
 *     outputs.  No atomic operation decides an order or a floating-point sum.
 *
 * Shape rules: T >= 1, 1 <= E <= 1024, 1 <= k <= min(E, 32), d % 64 == 0,
 * n % 64 == 0, 64 <= d, n <= 65536; tile in {64, 128, 256} when rounding.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,      /* bad argument: nothing was launched */
  MOE_ERR_CUDA = 2,         /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_WORKSPACE = 3,    /* workspace smaller than moe_workspace_bytes() */
  MOE_ERR_UNSUPPORTED = 4,  /* shape outside what the kernels support */
  MOE_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out */
  MOE_ERR_DEVICE_CHECK = 6  /* a device-side input check failed */
} moe_status;

typedef enum {
  MOE_ROUND_OFF = 0,        /* plain top-k routing */
  MOE_ROUND_NEAREST = 1,    /* each count to the nearest tile multiple, half up */
  MOE_ROUND_UP = 2,         /* each count up to a tile multiple */
  MOE_ROUND_STOCHASTIC = 3  /* down, or up with probability (c mod tile)/tile:
                               the expected count is c.  The draw for expert e
                               is the top 32 bits h of SplitMix64 (Steele, Lea,
                               Flood, OOPSLA 2014) at state seed*2^32 + e; the
                               count rounds up iff h*tile < (c mod tile)*2^32 */
} moe_round_mode;

typedef struct {
  int32_t T;      /* tokens */
  int32_t d;      /* model dim */
  int32_t n;      /* expert intermediate dim */
  int32_t E;      /* experts */
  int32_t k;      /* experts per token */
  int32_t tile;   /* token-rounding tile; ignored when round == MOE_ROUND_OFF */
  int32_t round;  /* moe_round_mode */
  uint32_t seed;  /* MOE_ROUND_STOCHASTIC: seed of the per-expert draws */
} moe_shape;

/* Number of rows the expert GEMMs can see: T*k without rounding, T*k + E*tile
 * with it.  Every per-row buffer (row_token, row_w, h, ys, tok_rows) holds
 * this many rows.  Returns 0 for an invalid shape. */
int64_t moe_row_capacity(const moe_shape* s);

/* Bytes of workspace moe_forward needs (the stage entry points need at most
 * this much).  Returns 0 for an invalid shape. */
size_t moe_workspace_bytes(const moe_shape* s);

/* Static text for a status code. */
const char* moe_status_string(int status);

/* Synchronises `stream`, then reads and clears the device status word at the
 * start of `ws`.  Returns MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_CHECK or
 * MOE_ERR_CUDA.  If `detail` is non-NULL it receives the kernel-specific
 * detail word (which wait, or which bad index). */
int moe_check_device_status(void* ws, int32_t* detail, void* stream);

/* Clears the status word at the start of `ws` (stream-ordered). */
int moe_clear_device_status(void* ws, void* stream);

/* One-time weight repack into the layouts the grouped GEMMs read K-major.
 *   W1, W3   [E, d, n] bf16   (W1 = gated branch, W3 = linear branch)
 *   W2       [E, n, d] bf16
 *   W13p     [E, 2n, d] bf16 out: row 2j holds W1[e][:, j]^T and row 2j+1
 *            holds W3[e][:, j]^T, so every GEMM tile carries matching gate
 *            and linear columns side by side.
 *   W2p      [E, d, n] bf16 out: W2p[e][i][j] = W2[e][j][i]. */
int moe_prepare_weights(const moe_shape* s, const void* W1, const void* W3, const void* W2,
                        void* W13p, void* W2p, void* stream);

/* Router logits (gate network; "MoE架构的物理瓶颈与扩展限制解析", 工作原理 step 1):
 *   logits[T, E] fp32 = float(x[T, d] bf16) @ Wr[d, E] fp32 + bias[E] fp32.
 * bias may be NULL.  The workspace must hold moe_workspace_bytes(s) bytes.
 * With E > 16 (or Wr too large for shared memory) it runs on the tensor
 * cores: Wr is split into three bf16 terms hi + mid + lo (equal to Wr within
 * 2^-27 relative; the split is kept in the workspace), each product with the
 * bf16 x is exact and accumulates in fp32.  With E <= 16 and
 * ((E + 1) & ~1) * d * 4 bytes plus the x staging within an SM's shared
 * memory (d <= 4160 for E <= 8, d <= 2816 for E <= 16) it runs on the SIMT
 * cores: one fp32 fused multiply-add per product, in a fixed order (a copy of
 * Wr laid out by expert pairs is kept in the workspace).  Either way every
 * call gives the same bits for the same inputs, and moe_route_permute and
 * moe_forward use the same router. */
int moe_router_logits(const moe_shape* s, const void* x, const float* Wr, const float* bias,
                      float* logits, void* ws, void* stream);

/* Top-k gating from given fp32 logits (工作原理 step 1, `top_k`):
 *   topk_idx[T, k] int32: the k largest logits of each row in descending
 *     order, equal values ordered by ascending expert id (-0.0 == +0.0);
 *   topk_w[T, k] fp32: softmax over the k selected logits (renormalised).
 * A NaN logit sets MOE_ERR_DEVICE_CHECK in the status word and ranks lowest. */
int moe_topk_gating(const moe_shape* s, const float* logits, int32_t* topk_idx, float* topk_w,
                    void* ws, void* stream);

/* moe_router_logits followed by moe_topk_gating: the same logits, indices
 * and weights, bit for bit.  Where the router can (k <= 8 with E <= 256) it
 * takes the top-k in its own last step, one launch fewer; `ws` must hold
 * moe_workspace_bytes(s) bytes. */
int moe_route(const moe_shape* s, const void* x, const float* Wr, const float* bias,
              float* logits, int32_t* topk_idx, float* topk_w, void* ws, void* stream);

/* Stable grouping of the A = T*k assignments a = t*k + j by expert
 * (bit-exact counting sort; rows of one expert are in ascending a):
 *   counts[E], offsets[E+1] (exclusive prefix, offsets[E] = A)
 *   src[A]       row -> assignment a
 *   dst[A]       assignment a -> row
 *   row_token[A] row -> token a / k
 *   row_w[A]     row -> topk_w[a]
 * topk_w may be NULL (row_w is then not written).  Uses the workspace for
 * per-chunk histograms.  An expert id outside [0, E) sets
 * MOE_ERR_DEVICE_CHECK and that assignment is skipped. */
int moe_permute(const moe_shape* s, const int32_t* topk_idx, const float* topk_w,
                int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dst,
                int32_t* row_token, float* row_w, void* ws, size_t ws_bytes, void* stream);

/* Fused route + permutation (the first three steps of the fused MoE kernel of
 * "硬件加速的考量", section 自定义核与核融合: gate scores, top-k, and the
 * grouping that collects each expert's tokens).  Same outputs, bit for bit, as
 * moe_route followed by moe_permute with topk_w given, in fewer launches:
 * for E <= 256 and k <= 8 the router's last step (the tensor-core GEMM's
 * epilogue, or the SIMT router for E <= 16) takes each token's top-k and gate
 * weights and counts each chunk's assignments per expert (integer atomics);
 * for E <= 256 and larger k one kernel does that from the stored logits; the
 * scan of the counts and the scatter follow.  (E > 256 runs the separate
 * top-k and permutation kernels.)  Arrays as in moe_route and moe_permute;
 * every output pointer is required.  Uses the workspace (router weights,
 * chunk histograms). */
int moe_route_permute(const moe_shape* s, const void* x, const float* Wr, const float* bias,
                      float* logits, int32_t* topk_idx, float* topk_w, int32_t* counts,
                      int32_t* offsets, int32_t* src, int32_t* dst, int32_t* row_token,
                      float* row_w, void* ws, size_t ws_bytes, void* stream);

/* moe_permute without a workspace, for callers that cannot allocate device
 * memory: code running inside a host engine that owns every device byte (a
 * serving runtime with a fixed memory arena, or a plugin loaded into another
 * framework) and is not allowed to call cudaMalloc once it is running, since
 * an allocation there can synchronise the device and bypasses the engine's
 * memory accounting.  The published method has no counterpart of this entry
 * point; it exists for those callers only.
 *
 * Same arguments and results as moe_permute, minus (ws, ws_bytes).  The
 * per-chunk histograms live in a 1 MiB array compiled into the library (a
 * file-scope __device__ array that every GPU loading the library holds until
 * the process exits), so the shape must satisfy E * ceil(T*k / 2048) <=
 * 262144; larger shapes return MOE_ERR_WORKSPACE and launch nothing.  No
 * allocation or free of any kind happens in this call.
 *   - Every call looks up the array's device address (cudaGetSymbolAddress,
 *     which allocates nothing) in the CUDA context current on the calling
 *     thread, and launches into that context.  The address is not cached, so
 *     a caller running in its own driver-API context, or calling again after
 *     cudaDeviceReset, gets the address valid in its context.  The first call
 *     in a context may load the library's kernels into it; make that first
 *     call before any stream capture in that context.
 *   - All calls share the one array: two calls whose kernels overlap on the
 *     GPU (different streams, or different host threads) race and give wrong
 *     results.  Serialise them.
 *   - Every histogram entry a call reads is written earlier in that call, so
 *     what an earlier call left in the array never matters.
 *   - Expert ids outside [0, E) are skipped, as in moe_permute, but are not
 *     reported (there is no status word). */
int moe_permute_noalloc(const moe_shape* s, const int32_t* topk_idx, const float* topk_w,
                        int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dst,
                        int32_t* row_token, float* row_w, void* stream);

/* Token rounding ("SonicMoE: 加速 MoE 模型的 IO 与 Tile 感知优化", 3. Token Rounding 路由算法),
 * mode s->round (NEAREST, UP or STOCHASTIC), tile s->tile.  Each expert's count
 * c becomes c' = a tile multiple (nearest half-up, up, or stochastic with seed
 * s->seed), capped at tile*floor(T/tile).
 * If c' > c the c'-c tokens not routed to e with the highest logits[t, e] join
 * (ties: lower t first); if c' < c the c-c' routed tokens with the lowest
 * logits leave (ties: higher t first); each expert is rounded from the original
 * top-k sets.  Outputs (R = offsets[E] rows, R <= moe_row_capacity):
 *   counts[E], offsets[E+1]; row_token[R], row_w[R] (softmax over the token's
 *   final set), tok_offsets[T+1] and tok_rows[R] (token -> its rows, in the
 *   order logits desc, expert id asc).  logits are the fp32 router logits. */
int moe_token_round(const moe_shape* s, const float* logits, const int32_t* topk_idx,
                    int32_t* counts, int32_t* offsets, int32_t* row_token, float* row_w,
                    int32_t* tok_offsets, int32_t* tok_rows, void* ws, size_t ws_bytes,
                    void* stream);

/* Up-projection grouped GEMM over gathered token rows, with SwiGLU fused into
 * the epilogue:
 *   for each expert e and row r in [offsets[e], offsets[e+1]):
 *     h[r, :] = bf16( silu(x[row_token[r]] W1_e) * (x[row_token[r]] W3_e) )
 *   silu(z) = z / (1 + exp(-z)); fp32 accumulation in tensor memory.
 *   x [T, d] bf16; W13p from moe_prepare_weights; h [moe_row_capacity, n] bf16.
 * gather selects how token rows reach shared memory:
 *   0 = a gather kernel copies the rows into the workspace (ys region), then
 *       tiled TMA loads them.  With tok_rows (token -> its rows, same
 *       convention as moe_combine: tok_rows[tok_offsets[t] ..), or
 *       tok_rows[t*k .. t*k+k) when tok_offsets is NULL, i.e. moe_permute's
 *       dst) the copy runs in token order and reads each x row once; with
 *       tok_rows NULL it runs in row order from row_token;
 *   1 = TMA tile::gather4 (four token rows per copy) straight from x;
 *   2 = per-lane 16-byte cp.async straight from x into the swizzled tile.
 * Any other value returns MOE_ERR_INVALID. */
int moe_expert_up(const moe_shape* s, const void* x, const void* W13p, const int32_t* counts,
                  const int32_t* offsets, const int32_t* row_token, const int32_t* tok_offsets,
                  const int32_t* tok_rows, void* h, int gather, void* ws, size_t ws_bytes,
                  void* stream);

/* Down-projection grouped GEMM with the gate weight in the epilogue:
 *   ys[r, :] = fp16( row_w[r] * (h[r] W2_e) ) for rows of expert e.
 *   h [cap, n] bf16; W2p from moe_prepare_weights; ys [cap, d] fp16.
 * A value beyond the fp16 range (|v| > 65504) is saturated and sets
 * MOE_ERR_DEVICE_CHECK (detail 16) in the status word. */
int moe_expert_down(const moe_shape* s, const void* h, const void* W2p, const int32_t* counts,
                    const int32_t* offsets, const float* row_w, void* ys, void* ws,
                    size_t ws_bytes, void* stream);

/* Deterministic combine back to token order (自定义核与核融合 step 5):
 *   y[t, :] = sum over j of ys[row_j, :]: ys fp16 [cap, d], fp32 sum in list
 *   order, y fp32 [T, d],
 * where t's rows are tok_rows[tok_offsets[t] .. tok_offsets[t+1]) or, when
 * tok_offsets is NULL, tok_rows[t*k .. t*k+k) (the `dst` array of
 * moe_permute).  A token with no rows gets y[t] = 0. */
int moe_combine(const moe_shape* s, const void* ys, const int32_t* tok_offsets,
                const int32_t* tok_rows, void* y, void* stream);

/* The same combine with y bf16 [T, d], the layer's output in a bf16 model:
 * each element is moe_combine's fp32 sum rounded to nearest-even bf16.
 * Arguments, ownership and errors as moe_combine. */
int moe_combine_bf16(const moe_shape* s, const void* ys, const int32_t* tok_offsets,
                     const int32_t* tok_rows, void* y, void* stream);

/* The A-operand path (the `gather` argument of moe_expert_up) that
 * moe_forward uses for this shape: 2 (rows gathered into the operand load by
 * cp.async, with wide tiles that put both 256-wide n-blocks against each
 * gathered row block) where n = 256, else 0 (the token-order staging copy,
 * then tiled TMA).  -1 for an invalid shape. */
int moe_forward_a_path(const moe_shape* s);

/* The whole layer: route, (round), permute, up, down, combine.
 *   x [T, d] bf16, Wr [d, E] fp32, bias [E] fp32 or NULL,
 *   W13p, W2p from moe_prepare_weights, y [T, d] fp32 out.
 * ws must hold moe_workspace_bytes(s) bytes. */
int moe_forward(const moe_shape* s, const void* x, const float* Wr, const float* bias,
                const void* W13p, const void* W2p, void* y, void* ws, size_t ws_bytes,
                void* stream);

/* moe_forward with y bf16 [T, d] out (moe_combine_bf16 as its last step):
 * each element is moe_forward's fp32 y rounded to nearest-even bf16, with
 * half the bytes written and copied out.  That rounding adds up to 2^-8 of
 * |y|: on outputs beyond about 5 rms it can take the error past the layer's
 * max-error tolerance (2e-2 rms), which the fp32 y meets.  Everything else
 * as moe_forward. */
int moe_forward_bf16(const moe_shape* s, const void* x, const float* Wr, const float* bias,
                     const void* W13p, const void* W2p, void* y, void* ws, size_t ws_bytes,
                     void* stream);

/* Byte offsets into the moe_forward workspace of its intermediate arrays, so
 * a caller can inspect them after a forward (all -1 for an invalid shape):
 * [0] logits f32[T*E]  [1] topk_idx i32[T*k]  [2] topk_w f32[T*k]
 * [3] counts i32[E]    [4] offsets i32[E+1]   [5] src i32[cap]  [6] dst i32[T*k]
 * [7] row_token i32[cap] [8] row_w f32[cap]   [9] tok_offsets i32[T+1]
 * [10] tok_rows i32[cap] [11] h bf16[cap*n]   [12] ys fp16[cap*d] */
int moe_workspace_layout(const moe_shape* s, int64_t* offsets_out, int32_t n_out);

/* ---------------------------------------------------------------- FP8 ---
 * e4m3 expert GEMMs.  The pages name FP8 among the precisions MoE compute
 * runs in ("硬件加速的考量", section 量化) without a recipe; reading: one fp32
 * scale per quantised row, scale = fp32(amax / 448), code =
 * e4m3(fp32(x * fp32(448 / amax))) rounded to nearest-even and saturated to
 * +-448; an all-zero row has scale 1 and codes 0.  Rows: tokens and the
 * output channels of the packed gate / linear weights (up-projection), rows
 * of the bf16 hidden h and the output channels of W2, i.e. the rows of the
 * packed W2p (down-projection).  A weight outlier therefore coarsens only its
 * own channel's codes.  Routing and the combine stay as in moe_forward. */

/* Workspace bytes of the FP8 entry points that quantise h
 * (moe_expert_down_fp8, moe_forward_fp8): moe_workspace_bytes plus the e4m3
 * codes of h and one scale per row. */
size_t moe_workspace_bytes_fp8(const moe_shape* s);

/* codes[rows, K] (e4m3 bytes) and scales[rows] fp32 of src[rows, K] bf16.
 * K % 16 == 0; src and codes 16-byte aligned.  For the weights, src is W13p
 * from moe_prepare_weights viewed as [E * 2n, d], or W2p viewed as
 * [E * d, n]. */
int moe_quantize_rows_fp8(const void* src, int64_t rows, int32_t K, void* codes, float* scales,
                          void* stream);

/* Up-projection with e4m3 operands: h[row] = silu(g) * u with
 * g, u = (code_x . code_w) * scale_x * scale_w, fp32 accumulation (kind::f8f6f4
 * on SM pairs), h bf16 as moe_expert_up.  x is quantised per token inside
 * (into the workspace) while it is gathered: tok_rows / tok_offsets as in
 * moe_expert_up's token-order gather (tok_offsets may be NULL: k rows per
 * token).  W13q / sW13 from moe_quantize_rows_fp8 of W13p.  Requires
 * n % 128 == 0 and d % 128 == 0 (else MOE_ERR_UNSUPPORTED). */
int moe_expert_up_fp8(const moe_shape* s, const void* x, const void* W13q, const float* sW13,
                      const int32_t* counts, const int32_t* offsets, const int32_t* tok_offsets,
                      const int32_t* tok_rows, void* h, void* ws, size_t ws_bytes, void* stream);

/* codes[E, m] and scales[E] with one scale per row of m elements (one scale
 * for a whole expert's matrix, e.g. W2p viewed as [E, d * n]).  m % 16 == 0.
 * The FP8 GEMMs do not take these per-expert scales; they are here for
 * callers that store weights that way. */
int moe_quantize_experts_fp8(const void* src, int32_t E, int64_t m, void* codes, float* scales,
                             void* stream);

/* Down-projection with e4m3 operands: h [moe_row_capacity, n] bf16 (as
 * moe_expert_up writes it) is quantised per row into the workspace
 * (moe_workspace_bytes_fp8), then ys[row][c] = w[row] * (code_h . code_W2[c]) *
 * scale_h[row] * scale_W2[e * d + c] in fp32 (kind::f8f6f4 on SM pairs),
 * stored fp16 as moe_expert_down (saturation reported alike).  W2q [E * d, n]
 * / sW2 [E * d] from moe_quantize_rows_fp8 of W2p (one scale per output
 * channel).  Requires n % 128 == 0 and d % 256 == 0 (else
 * MOE_ERR_UNSUPPORTED). */
int moe_expert_down_fp8(const moe_shape* s, const void* h, const void* W2q, const float* sW2,
                        const int32_t* counts, const int32_t* offsets, const float* row_w, void* ys,
                        void* ws, size_t ws_bytes, void* stream);

/* moe_forward with both expert GEMMs in e4m3 (moe_expert_up_fp8,
 * moe_expert_down_fp8).  ws_bytes >= moe_workspace_bytes_fp8(s); n % 128 ==
 * 0 and d % 256 == 0. */
int moe_forward_fp8(const moe_shape* s, const void* x, const float* Wr, const float* bias,
                    const void* W13q, const float* sW13, const void* W2q, const float* sW2,
                    void* y, void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------- backward ---
 * Gradients of sum_t <dy[t], y[t]> for y = moe_forward(x, ...), by
 * recomputation instead of cached activations ("SonicMoE: 加速 MoE 模型的 IO
 * 与 Tile 感知优化", "SonicMoE 的三大核心优化" item 1 and section 反向传播优化):
 * routing, the gathered x rows and the up-projection's pre-activations are
 * recomputed, and the gate weights' gradient is sum_j dh'[j] h[j] per row
 * (dh' = dy W2^T), so no expert output is formed (the 关键 Kernel 对比
 * table's "dS 计算优化").  The selected sets are held fixed (selection passes
 * no gradient); the logits' gradient is that of the softmax over the k
 * selected logits.  bf16 operands, fp32 accumulation; the pre-activations
 * are held in fp32, their gradients and w h in bf16 (the weight-gradient
 * GEMMs' operands), each row's input gradient from the experts in fp16
 * (saturation is reported as for ys);
 * every sum runs in a fixed order, so results are bitwise reproducible.
 * With token rounding (s->round != MOE_ROUND_OFF) the rounded sets of the
 * forward are recomputed and held fixed the same way.  Requires d % 128 == 0
 * (n % 64 == 0 as always), else MOE_ERR_UNSUPPORTED. */

/* Workspace bytes of moe_backward (0 for an invalid or unsupported shape). */
size_t moe_backward_workspace_bytes(const moe_shape* s);

/* W13i [E, d, 2n] bf16 with W13i[e][i][2j] = W1[e][i][j] and
 * W13i[e][i][2j+1] = W3[e][i][j]: the packed up weight transposed, for the
 * input gradient.  One-time, like moe_prepare_weights. */
int moe_prepare_weights_bwd(const moe_shape* s, const void* W1, const void* W3, void* W13i,
                            void* stream);

/* Backward pass of the layer.
 *   in:  x [T, d] bf16, Wr [d, E] fp32, bias [E] fp32 or NULL, W13p from
 *        moe_prepare_weights, W13i from moe_prepare_weights_bwd, W2 [E, n, d]
 *        bf16 (as given to moe_prepare_weights), dy [T, d] bf16;
 *   out: dx [T, d], dWr [d, E], dbias [E] (NULL: not written), dW1 and dW3
 *        [E, d, n], dW2 [E, n, d], all fp32, every element written (an expert
 *        without tokens gets zero weight gradients).
 * x, dy, dx, dW1, dW3, dW2 and ws 16-byte aligned.  ws
 * (moe_backward_workspace_bytes) is caller-owned device memory; its status
 * word reports device-side errors as for moe_forward.
 * Asynchronous on `stream`. */
int moe_backward(const moe_shape* s, const void* x, const float* Wr, const float* bias,
                 const void* W13p, const void* W13i, const void* W2, const void* dy, float* dx,
                 float* dWr, float* dbias, float* dW1, float* dW3, float* dW2, void* ws,
                 size_t ws_bytes, void* stream);

/* Self-test of the bounded-wait machinery: launches one block that waits on a
 * device flag nobody sets, giving up after `timeout_ns` nanoseconds; the
 * kernel then records MOE_ERR_TIMEOUT in the status word of `ws` and returns. */
int moe_selftest_timeout(void* ws, uint64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
