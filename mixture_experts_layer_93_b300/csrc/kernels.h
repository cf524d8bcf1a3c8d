// Host-side launchers of the kernels in libmoe.so (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// route.cu
void launch_topk_gating(const float* logits, int32_t* idx, float* w, int T, int E, int k, int32_t* status,
                        cudaStream_t stream);

// permute.cu
constexpr int kPermChunk = 2048;  // assignments per warp chunk
inline int64_t perm_num_chunks(int64_t A) { return (A + kPermChunk - 1) / kPermChunk; }
// Top-k gating plus the permutation of the assignments; E <= 256 runs the
// fused top-k + histogram kernel (chunk_hist[E * chunks] zero on entry, see
// launch_split_router), then the scan and the scatter.
void launch_topk_permute(const float* logits, int T, int E, int k, int32_t* idx, float* w, int32_t* chunk_hist,
                         int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dst, int32_t* row_token,
                         float* row_w, int32_t* status, cudaStream_t stream);
// The scan and the scatter of launch_topk_permute, for chunk counts already
// made (by the router epilogue).
void launch_perm_scan_scatter(const int32_t* idx, const float* w, int64_t A, int k, int E, int32_t* chunk_hist,
                              int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dst, int32_t* row_token,
                              float* row_w, cudaStream_t stream);
void launch_permute(const int32_t* idx, const float* w, int64_t A, int k, int E, int32_t* chunk_hist,
                    int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dst, int32_t* row_token,
                    float* row_w, int32_t* status, cudaStream_t stream);
// The same sort over a list of `*len` (<= cap, read on the device) assignments
// with explicit tokens: rows of an expert keep list order; dst[a] = row.
void launch_permute_list(const int32_t* expert_of, const float* w, const int32_t* token_of, const int32_t* len,
                         int64_t cap, int E, int32_t* chunk_hist, int32_t* counts, int32_t* offsets, int32_t* dst,
                         int32_t* row_token, float* row_w, int32_t* status, cudaStream_t stream);

// round.cu
size_t round_scratch_bytes(int T, int E, int k, int tile);
void launch_token_round(const float* logits, const int32_t* idx, int T, int E, int k, int tile, int mode,
                        uint32_t seed, int32_t* counts, int32_t* offsets, int32_t* row_token, float* row_w, int32_t* tok_offsets,
                        int32_t* tok_rows, void* scratch, int32_t* status, cudaStream_t stream);

// fp8.cu
void launch_quant_rows(const __nv_bfloat16* src, int64_t rows, int K, uint8_t* codes, float* scales,
                       cudaStream_t stream);
void launch_gather_quant(const __nv_bfloat16* x, const int32_t* tok_rows, const int32_t* tok_offsets, int T, int k,
                         int d, uint8_t* xq, float* row_scale, cudaStream_t stream);
void launch_quant_experts(const __nv_bfloat16* src, int E, int64_t m, uint8_t* codes, float* scales,
                          cudaStream_t stream);
int launch_expert_down_f8(const uint8_t* hq, const float* h_scale, const uint8_t* W2q, const float* sW2,
                          const int32_t* counts, const int32_t* offsets, const float* row_w, __half* ys, int d,
                          int n, int E, int64_t rows_cap, int32_t* status, uint64_t timeout_ns, cudaStream_t stream);

// gemm.cu
int launch_expert_up_f8(const __nv_bfloat16* x, const uint8_t* W13q, const float* sW13, const int32_t* counts,
                        const int32_t* offsets, const int32_t* tok_rows, const int32_t* tok_offsets,
                        __nv_bfloat16* h, int T, int d, int n, int E, int k, int64_t rows_cap, uint8_t* xq_scratch,
                        float* row_scale, int32_t* status, uint64_t timeout_ns, cudaStream_t stream);
int launch_expert_up(const __nv_bfloat16* x, const __nv_bfloat16* W13p, const int32_t* counts,
                     const int32_t* offsets, const int32_t* row_token, const int32_t* tok_rows,
                     const int32_t* tok_offsets, __nv_bfloat16* h, int T, int d, int n, int E, int k,
                     int64_t rows_cap, int gather, __nv_bfloat16* xperm_scratch, int32_t* status,
                     uint64_t timeout_ns, cudaStream_t stream);
int launch_expert_down(const __nv_bfloat16* h, const __nv_bfloat16* W2p, const int32_t* counts,
                       const int32_t* offsets, const float* row_w, __half* ys, int d, int n, int E,
                       int64_t rows_cap, int32_t* status, uint64_t timeout_ns, cudaStream_t stream);
void launch_gather_rows(const __nv_bfloat16* x, const int32_t* row_token, const int32_t* offsets, int E, int d,
                        __nv_bfloat16* out, int64_t rows_cap, cudaStream_t stream);
inline int up_half_block(int n) { return (n % 128 == 0) ? 128 : 64; }
// backward GEMMs (gemm.cu)
inline int bwd_act_block(int n) { return (n % 256 == 0) ? 256 : (n % 128 == 0 ? 128 : 64); }
// partial sums of <dh', h> per row: one per n-block and epilogue column half
inline int bwd_act_parts(int n) { return 2 * (n / bwd_act_block(n)); }
int launch_expert_up_pre(const __nv_bfloat16* xp, const __nv_bfloat16* W13p, const int32_t* counts,
                         const int32_t* offsets, float* gl, int d, int n, int E, int64_t rows_cap,
                         int32_t* status, uint64_t timeout_ns, cudaStream_t stream);
int launch_bwd_act(const __nv_bfloat16* dyp, const __nv_bfloat16* W2, const int32_t* counts, const int32_t* offsets,
                   const float* row_w, const float* gl, __nv_bfloat16* dgl, __nv_bfloat16* hw, float* dw_part, int d,
                   int n, int E, int64_t rows_cap, int32_t* status, uint64_t timeout_ns, cudaStream_t stream);
int launch_expert_dx(const __nv_bfloat16* dgl, const __nv_bfloat16* W13i, const int32_t* counts,
                     const int32_t* offsets, const float* dl_row, const float* WrT, __half* dxr, int d, int n,
                     int E, int64_t rows_cap, int32_t* status, uint64_t timeout_ns, cudaStream_t stream);
int launch_wgrad(const __nv_bfloat16* A, const __nv_bfloat16* B, const int32_t* counts, const int32_t* offsets,
                 int M, int N, int E, int64_t rows_cap, float* out, float* out2, int32_t* status,
                 uint64_t timeout_ns, cudaStream_t stream);
int num_sms();
// router on the tensor cores: Wr split into three bf16 terms (see gemm.cu)
int router_expert_block(int E);
size_t router_split_elems(int d, int E);
// zero[0, zero_count) (nullable): zeroed for launch_topk_permute's fused
// kernel (its chunk counts).
void launch_split_router(const float* Wr, __nv_bfloat16* Wr3, int d, int E, cudaStream_t stream,
                         int32_t* zero = nullptr, int64_t zero_count = 0);
// k > 0 (router_fuses_topk): the epilogue also writes the top-k ids and gate
// weights and counts them into chunk_hist (zero on entry), as the fused
// top-k + histogram kernel does; an SM pair then runs all n-blocks (64
// experts each) of one row block in a row.
constexpr int kFusedTopk = 8;
// Router for few experts on the SIMT cores (route.cu): E <= 16 and Wr (fp32)
// with the kernel's x staging fits in shared memory.  launch_router_small_prep
// lays Wr out for it in Wp (router_small_wp_bytes, 16-byte aligned) and zeroes
// zero[0, zero_count); launch_router_small then computes the logits and, with
// k > 0, the top-k, gate weights and chunk counts (chunk_hist zero on entry),
// as launch_router_tc does.  x must be 16-byte aligned.
constexpr int kRouterSmallSmemMax = 227 * 1024 - 64;  // the per-block limit, less its static barrier
constexpr int kRouterSmallStages = 3;             // x steps per warp in its ring
bool router_is_small(int d, int E);
size_t router_small_wp_bytes(int d, int E);
void launch_router_small_prep(const float* Wr, int d, int E, float* Wp, int32_t* zero, int64_t zero_count,
                              cudaStream_t stream);
int launch_router_small(const __nv_bfloat16* x, const float* Wp, const float* bias, float* logits, int T, int d, int E,
                        int k, int32_t* topk_idx, float* topk_w, int32_t* chunk_hist, int32_t* status,
                        uint64_t timeout_ns, cudaStream_t stream);
inline bool router_fuses_topk(int E, int k) { return E <= 256 && k <= kFusedTopk; }
int launch_router_tc(const __nv_bfloat16* x, const __nv_bfloat16* Wr3, const float* bias, float* logits, int T,
                     int d, int E, int32_t* status, uint64_t timeout_ns, cudaStream_t stream, int k = 0,
                     int32_t* topk_idx = nullptr, float* topk_w = nullptr, int32_t* chunk_hist = nullptr);

// combine.cu
void launch_combine(const __half* ys, const int32_t* tok_offsets, const int32_t* tok_rows, float* y, int T, int d,
                    int k, cudaStream_t stream);
// the same sum rounded to nearest-even bf16
void launch_combine(const __half* ys, const int32_t* tok_offsets, const int32_t* tok_rows, __nv_bfloat16* y, int T,
                    int d, int k, cudaStream_t stream);

// prepare.cu
void launch_prepare_weights(const __nv_bfloat16* W1, const __nv_bfloat16* W3, const __nv_bfloat16* W2,
                            __nv_bfloat16* W13p, __nv_bfloat16* W2p, int E, int d, int n, cudaStream_t stream);

void launch_prepare_weights_bwd(const __nv_bfloat16* W1, const __nv_bfloat16* W3, __nv_bfloat16* W13i, int E, int d,
                                int n, cudaStream_t stream);

// bwd.cu (backward pass around the backward GEMMs; padded row layout)
int bwd_dwr_splits(int E, int d);
void launch_bwd_pad_offsets(const int32_t* counts, int E, int32_t* offsets_p, cudaStream_t stream);
void launch_bwd_rows(const int32_t* idx, const float* w, const int32_t* dst, const int32_t* offsets,
                     const int32_t* offsets_p, int64_t A, int32_t* rowp, float* wp, cudaStream_t stream);
void launch_bwd_zero_pad(const int32_t* counts, const int32_t* offsets_p, int E, int d, int n, __nv_bfloat16* xp,
                         __nv_bfloat16* dyp, __nv_bfloat16* dgl, __nv_bfloat16* hw, cudaStream_t stream);
// rows / tok_offsets: each token's row list (tok_offsets NULL: k entries per token)
void launch_router_bwd(const int32_t* rows, const int32_t* tok_offsets, const float* wp, const float* dw_part,
                       int parts, int T, int k, float* dlp, cudaStream_t stream);
void launch_transpose_router(const float* Wr, int d, int E, float* WrT, cudaStream_t stream);
void launch_bwd_dwr(const __nv_bfloat16* xp, const float* dlp, const int32_t* counts, const int32_t* offsets_p,
                    int E, int d, float* part, float* dbpart, float* dWr, float* db, cudaStream_t stream);
void launch_gather_rows_by_token(const __nv_bfloat16* x, const int32_t* tok_rows, const int32_t* tok_offsets, int T,
                                 int k, int d, __nv_bfloat16* out, cudaStream_t stream);

// selftest
void launch_selftest_timeout(int32_t* status, uint64_t timeout_ns, cudaStream_t stream);

}  // namespace moe
