// C ABI of libmoe.so: argument validation, workspace layout and the stage
// sequence of the MoE-layer forward.  Every declaration is in include/moe.h.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool shape_ok(const moe_shape* s) {
  if (!s) return false;
  if (s->T < 1 || s->E < 1 || s->E > 1024) return false;
  if (s->k < 1 || s->k > s->E || s->k > 32) return false;
  if (s->d < 64 || s->d % 64 != 0 || s->d > 65536) return false;
  if (s->n < 64 || s->n % 64 != 0 || s->n > 65536) return false;
  if (s->round < MOE_ROUND_OFF || s->round > MOE_ROUND_STOCHASTIC) return false;
  if (s->round != MOE_ROUND_OFF && s->tile != 64 && s->tile != 128 && s->tile != 256) return false;
  // row indices and element offsets stay in range of the int32 / int64 math
  const int64_t A = static_cast<int64_t>(s->T) * s->k;
  const int64_t cap = A + (s->round != MOE_ROUND_OFF ? static_cast<int64_t>(s->E) * s->tile : 0);
  if (cap >= (int64_t(1) << 31) - 1) return false;
  return true;
}

inline int64_t row_cap(const moe_shape* s) {
  const int64_t A = static_cast<int64_t>(s->T) * s->k;
  return A + (s->round != MOE_ROUND_OFF ? static_cast<int64_t>(s->E) * s->tile : 0);
}

inline int64_t align256(int64_t v) { return (v + 255) & ~int64_t(255); }

enum Slot {
  kLogits, kTopkIdx, kTopkW, kCounts, kOffsets, kSrc, kDst, kRowToken, kRowW, kTokOffsets, kTokRows, kH, kYs,
  kPermHist, kRoundScratch, kRouterW, kHq, kNumSlots
};

// Byte offsets of each array in the workspace; returns the total size.  The
// last slot (e4m3 codes of h and their row scales) only counts with fp8.
int64_t layout(const moe_shape* s, int64_t* off, bool fp8 = false) {
  const int64_t T = s->T, E = s->E, A = T * s->k, cap = row_cap(s);
  const int64_t sizes[kNumSlots] = {
      T * E * 4,          A * 4,     A * 4,     E * 4,   (E + 1) * 4,       cap * 4,
      A * 4,              cap * 4,   cap * 4,   (T + 1) * 4, cap * 4,       cap * s->n * 2,
      cap * s->d * 2,     E * perm_num_chunks(cap) * 4,
      s->round != MOE_ROUND_OFF ? static_cast<int64_t>(round_scratch_bytes(s->T, s->E, s->k, s->tile)) : 0,
      std::max<int64_t>(static_cast<int64_t>(router_split_elems(s->d, s->E)) * 2,
                        router_is_small(s->d, s->E) ? static_cast<int64_t>(router_small_wp_bytes(s->d, s->E)) : 0),
      fp8 ? align256(cap * s->n) + cap * 4 : 0};
  int64_t pos = static_cast<int64_t>(kStatusBytes);
  for (int i = 0; i < kNumSlots; ++i) {
    off[i] = pos;
    pos = align256(pos + sizes[i]);
  }
  return pos;
}

template <typename T>
inline T* at(void* ws, int64_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline int last_launch() { return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

inline int32_t* status_of(void* ws) { return reinterpret_cast<int32_t*>(ws); }

// A-operand path moe_forward uses for the up-projection (see moe_expert_up):
// rows gathered into the operand load by cp.async (path 2) where the up GEMM
// has exactly two 256-wide n-blocks (n = 256), so that one wide tile covers
// all of N and each row is gathered once; else the token-order staging copy
// and tiled TMA (path 0).  Measured: the 7B-class layer (n = 256) +8 % with
// path 2; the layers with 8 to 112 n-blocks, which would gather each row 4 to
// 56 times, 5-11 % slower.
int forward_gather(const moe_shape* s) { return s->n == 256 ? 2 : 0; }

int check_ws(const moe_shape* s, void* ws, size_t ws_bytes, bool fp8 = false) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID;
  int64_t off[kNumSlots];
  if (static_cast<int64_t>(ws_bytes) < layout(s, off, fp8)) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// Backward workspace: the forward's slots, then the backward's arrays over
// the padded row layout (each expert's rows padded to a multiple of 64).
enum BwdSlot {
  kOffP, kRowP, kWp, kXp, kDyp, kGl, kDgl, kHw, kDwPart, kDxr, kDlp, kWrT, kDwrPart, kDbPart, kNumBwdSlots
};

// rows of the padded layout: the forward's rows plus up to 63 padding rows per expert
inline int64_t padded_cap(const moe_shape* s) { return row_cap(s) + 63 * int64_t(s->E); }

int64_t layout_bwd(const moe_shape* s, int64_t* off_fwd, int64_t* off) {
  const int64_t base = layout(s, off_fwd);
  const int64_t T = s->T, E = s->E, A = T * s->k, capp = padded_cap(s), d = s->d, n = s->n;
  const int64_t S = bwd_dwr_splits(s->E, s->d);
  const int64_t sizes[kNumBwdSlots] = {(E + 1) * 4, A * 4,       capp * 4,
                                       capp * d * 2, capp * d * 2, capp * 2 * n * 4,
                                       capp * 2 * n * 2, capp * n * 2, capp * bwd_act_parts(s->n) * 4, capp * d * 2,
                                       capp * 4,     E * d * 4,
                                       S * E * d * 4, S * E * 4};
  int64_t pos = base;
  for (int i = 0; i < kNumBwdSlots; ++i) {
    off[i] = pos;
    pos = align256(pos + sizes[i]);
  }
  return pos;
}

bool bwd_shape_ok(const moe_shape* s) { return s->d % 128 == 0 && s->n % 64 == 0; }

}  // namespace

extern "C" {

int64_t moe_row_capacity(const moe_shape* s) { return shape_ok(s) ? row_cap(s) : 0; }

size_t moe_workspace_bytes(const moe_shape* s) {
  if (!shape_ok(s)) return 0;
  int64_t off[kNumSlots];
  return static_cast<size_t>(layout(s, off));
}

size_t moe_workspace_bytes_fp8(const moe_shape* s) {
  if (!shape_ok(s)) return 0;
  int64_t off[kNumSlots];
  return static_cast<size_t>(layout(s, off, true));
}

int moe_workspace_layout(const moe_shape* s, int64_t* out, int32_t n_out) {
  if (!out || n_out < 0) return MOE_ERR_INVALID;
  if (!shape_ok(s)) {
    for (int i = 0; i < n_out; ++i) out[i] = -1;
    return MOE_ERR_INVALID;
  }
  int64_t off[kNumSlots];
  layout(s, off);
  for (int i = 0; i < n_out; ++i) out[i] = (i <= kYs) ? off[i] : -1;
  return MOE_OK;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID: return "invalid argument";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or mode";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device-side input check failed";
    default: return "unknown status";
  }
}

int moe_clear_device_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID;
  return cudaMemsetAsync(ws, 0, kStatusBytes, as_stream(stream)) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_check_device_status(void* ws, int32_t* detail, void* stream) {
  if (!ws) return MOE_ERR_INVALID;
  int32_t h[4] = {0, 0, 0, 0};
  cudaStream_t st = as_stream(stream);
  if (cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, kStatusBytes, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (detail) *detail = h[1];
  return h[0];
}

int moe_prepare_weights(const moe_shape* s, const void* W1, const void* W3, const void* W2, void* W13p, void* W2p,
                        void* stream) {
  if (!shape_ok(s) || !W1 || !W3 || !W2 || !W13p || !W2p) return MOE_ERR_INVALID;
  if (!aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(W13p) || !aligned16(W2p))
    return MOE_ERR_INVALID;
  launch_prepare_weights(static_cast<const __nv_bfloat16*>(W1), static_cast<const __nv_bfloat16*>(W3),
                         static_cast<const __nv_bfloat16*>(W2), static_cast<__nv_bfloat16*>(W13p),
                         static_cast<__nv_bfloat16*>(W2p), s->E, s->d, s->n, as_stream(stream));
  return last_launch();
}

int moe_router_logits(const moe_shape* s, const void* x, const float* Wr, const float* bias, float* logits,
                      void* ws, void* stream) {
  if (!shape_ok(s) || !x || !Wr || !logits || !ws || !aligned16(x) || !aligned16(ws)) return MOE_ERR_INVALID;
  int64_t off[kNumSlots];
  layout(s, off);
  if (router_is_small(s->d, s->E)) {  // few experts: SIMT, bound by reading x
    float* Wp = at<float>(ws, off[kRouterW]);
    launch_router_small_prep(Wr, s->d, s->E, Wp, nullptr, 0, as_stream(stream));
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    return launch_router_small(static_cast<const __nv_bfloat16*>(x), Wp, bias, logits, s->T, s->d, s->E, 0, nullptr,
                               nullptr, nullptr, status_of(ws), kDefaultTimeoutNs, as_stream(stream));
  }
  __nv_bfloat16* Wr3 = at<__nv_bfloat16>(ws, off[kRouterW]);
  launch_split_router(Wr, Wr3, s->d, s->E, as_stream(stream));
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  return launch_router_tc(static_cast<const __nv_bfloat16*>(x), Wr3, bias, logits, s->T, s->d, s->E, status_of(ws),
                          kDefaultTimeoutNs, as_stream(stream));
}

int moe_topk_gating(const moe_shape* s, const float* logits, int32_t* topk_idx, float* topk_w, void* ws,
                    void* stream) {
  if (!shape_ok(s) || !logits || !topk_idx || !topk_w || !ws) return MOE_ERR_INVALID;
  launch_topk_gating(logits, topk_idx, topk_w, s->T, s->E, s->k, status_of(ws), as_stream(stream));
  return last_launch();
}

int moe_forward_a_path(const moe_shape* s) { return shape_ok(s) ? forward_gather(s) : -1; }

int moe_route(const moe_shape* s, const void* x, const float* Wr, const float* bias, float* logits,
              int32_t* topk_idx, float* topk_w, void* ws, void* stream) {
  if (!shape_ok(s) || !x || !Wr || !logits || !topk_idx || !topk_w || !ws || !aligned16(x) || !aligned16(ws))
    return MOE_ERR_INVALID;
  // Where the router takes the top-k in its last step (the bits of
  // moe_topk_gating on its logits), one launch fewer.  Its chunk counts go
  // to the permutation's histogram slot, which moe_permute overwrites.
  int64_t off[kNumSlots];
  layout(s, off);
  int32_t* chunk_hist = at<int32_t>(ws, off[kPermHist]);
  const int64_t hist_count = static_cast<int64_t>(s->E) * perm_num_chunks(static_cast<int64_t>(s->T) * s->k);
  if (s->k <= kFusedTopk && router_is_small(s->d, s->E)) {
    float* Wp = at<float>(ws, off[kRouterW]);
    launch_router_small_prep(Wr, s->d, s->E, Wp, chunk_hist, hist_count, as_stream(stream));
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    return launch_router_small(static_cast<const __nv_bfloat16*>(x), Wp, bias, logits, s->T, s->d, s->E, s->k,
                               topk_idx, topk_w, chunk_hist, status_of(ws), kDefaultTimeoutNs, as_stream(stream));
  }
  if (!router_is_small(s->d, s->E) && router_fuses_topk(s->E, s->k)) {
    __nv_bfloat16* Wr3 = at<__nv_bfloat16>(ws, off[kRouterW]);
    launch_split_router(Wr, Wr3, s->d, s->E, as_stream(stream), chunk_hist, hist_count);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    return launch_router_tc(static_cast<const __nv_bfloat16*>(x), Wr3, bias, logits, s->T, s->d, s->E,
                            status_of(ws), kDefaultTimeoutNs, as_stream(stream), s->k, topk_idx, topk_w, chunk_hist);
  }
  int st = moe_router_logits(s, x, Wr, bias, logits, ws, stream);
  if (st != MOE_OK) return st;
  return moe_topk_gating(s, logits, topk_idx, topk_w, ws, stream);
}

int moe_route_permute(const moe_shape* s, const void* x, const float* Wr, const float* bias, float* logits,
                      int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets, int32_t* src,
                      int32_t* dst, int32_t* row_token, float* row_w, void* ws, size_t ws_bytes, void* stream) {
  if (!shape_ok(s) || !x || !Wr || !logits || !topk_idx || !topk_w || !counts || !offsets || !src || !dst ||
      !row_token || !row_w)
    return MOE_ERR_INVALID;
  if (!aligned16(x)) return MOE_ERR_INVALID;
  const int st = check_ws(s, ws, ws_bytes);
  if (st != MOE_OK) return st;
  int64_t off[kNumSlots];
  layout(s, off);
  __nv_bfloat16* Wr3 = at<__nv_bfloat16>(ws, off[kRouterW]);
  int32_t* chunk_hist = at<int32_t>(ws, off[kPermHist]);
  const int64_t hist_count = static_cast<int64_t>(s->E) * perm_num_chunks(static_cast<int64_t>(s->T) * s->k);
  if (router_is_small(s->d, s->E)) {
    // few experts: the weight layout (and zeroed chunk counts), then the SIMT
    // router, which moe_router_logits uses too.  With k <= kFusedTopk it
    // also takes the top-k and the chunk counts, and the scan and the
    // scatter follow (4 launches); with larger k the top-k + histogram
    // kernel reads its logits.
    float* Wp = at<float>(ws, off[kRouterW]);
    launch_router_small_prep(Wr, s->d, s->E, Wp, chunk_hist, hist_count, as_stream(stream));
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    const bool fuse = s->k <= kFusedTopk;
    const int rst = launch_router_small(static_cast<const __nv_bfloat16*>(x), Wp, bias, logits, s->T, s->d, s->E,
                                        fuse ? s->k : 0, fuse ? topk_idx : nullptr, fuse ? topk_w : nullptr,
                                        fuse ? chunk_hist : nullptr, status_of(ws), kDefaultTimeoutNs,
                                        as_stream(stream));
    if (rst != MOE_OK) return rst;
    if (fuse) {
      launch_perm_scan_scatter(topk_idx, topk_w, static_cast<int64_t>(s->T) * s->k, s->k, s->E, chunk_hist, counts,
                               offsets, src, dst, row_token, row_w, as_stream(stream));
      return last_launch();
    }
  } else {
    const bool fused = s->E <= 256;  // the fused top-k + histogram kernel (counts start at zero)
    launch_split_router(Wr, Wr3, s->d, s->E, as_stream(stream), fused ? chunk_hist : nullptr, fused ? hist_count : 0);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    if (router_fuses_topk(s->E, s->k)) {
      // top-k and chunk counts in the router GEMM's epilogue
      const int rst = launch_router_tc(static_cast<const __nv_bfloat16*>(x), Wr3, bias, logits, s->T, s->d, s->E,
                                       status_of(ws), kDefaultTimeoutNs, as_stream(stream), s->k, topk_idx, topk_w,
                                       chunk_hist);
      if (rst != MOE_OK) return rst;
      launch_perm_scan_scatter(topk_idx, topk_w, static_cast<int64_t>(s->T) * s->k, s->k, s->E, chunk_hist, counts,
                               offsets, src, dst, row_token, row_w, as_stream(stream));
      return last_launch();
    }
    const int rst = launch_router_tc(static_cast<const __nv_bfloat16*>(x), Wr3, bias, logits, s->T, s->d, s->E,
                                     status_of(ws), kDefaultTimeoutNs, as_stream(stream));
    if (rst != MOE_OK) return rst;
  }
  launch_topk_permute(logits, s->T, s->E, s->k, topk_idx, topk_w, chunk_hist, counts, offsets, src, dst, row_token,
                      row_w, status_of(ws), as_stream(stream));
  return last_launch();
}

int moe_permute(const moe_shape* s, const int32_t* topk_idx, const float* topk_w, int32_t* counts,
                int32_t* offsets, int32_t* src, int32_t* dst, int32_t* row_token, float* row_w, void* ws,
                size_t ws_bytes, void* stream) {
  if (!shape_ok(s) || !topk_idx || !counts || !offsets || !src || !dst || !row_token) return MOE_ERR_INVALID;
  if (topk_w && !row_w) return MOE_ERR_INVALID;
  const int st = check_ws(s, ws, ws_bytes);
  if (st != MOE_OK) return st;
  int64_t off[kNumSlots];
  layout(s, off);
  const int64_t A = static_cast<int64_t>(s->T) * s->k;
  launch_permute(topk_idx, topk_w, A, s->k, s->E, at<int32_t>(ws, off[kPermHist]), counts, offsets, src, dst,
                 row_token, row_w, status_of(ws), as_stream(stream));
  return last_launch();
}

int moe_token_round(const moe_shape* s, const float* logits, const int32_t* topk_idx, int32_t* counts,
                    int32_t* offsets, int32_t* row_token, float* row_w, int32_t* tok_offsets, int32_t* tok_rows,
                    void* ws, size_t ws_bytes, void* stream) {
  if (!shape_ok(s) || s->round == MOE_ROUND_OFF) return MOE_ERR_INVALID;
  if (!logits || !topk_idx || !counts || !offsets || !row_token || !row_w || !tok_offsets || !tok_rows)
    return MOE_ERR_INVALID;
  const int st = check_ws(s, ws, ws_bytes);
  if (st != MOE_OK) return st;
  int64_t off[kNumSlots];
  layout(s, off);
  launch_token_round(logits, topk_idx, s->T, s->E, s->k, s->tile, s->round, s->seed, counts, offsets, row_token,
                     row_w,
                     tok_offsets, tok_rows, at<void>(ws, off[kRoundScratch]), status_of(ws), as_stream(stream));
  return last_launch();
}

int moe_expert_up(const moe_shape* s, const void* x, const void* W13p, const int32_t* counts, const int32_t* offsets,
                  const int32_t* row_token, const int32_t* tok_offsets, const int32_t* tok_rows, void* h, int gather,
                  void* ws, size_t ws_bytes, void* stream) {
  if (!shape_ok(s) || !x || !W13p || !counts || !offsets || !row_token || !h) return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(W13p) || !aligned16(h)) return MOE_ERR_INVALID;
  if (gather < 0 || gather > 2) return MOE_ERR_INVALID;
  const int st = check_ws(s, ws, ws_bytes);
  if (st != MOE_OK) return st;
  int64_t off[kNumSlots];
  layout(s, off);
  // the non-gather variant stages the gathered rows in the ys region, which
  // the forward only writes after the up-projection
  return launch_expert_up(static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(W13p), counts,
                          offsets, row_token, tok_rows, tok_offsets, static_cast<__nv_bfloat16*>(h), s->T, s->d, s->n,
                          s->E, s->k, row_cap(s), gather, at<__nv_bfloat16>(ws, off[kYs]), status_of(ws),
                          kDefaultTimeoutNs, as_stream(stream));
}

int moe_expert_down(const moe_shape* s, const void* h, const void* W2p, const int32_t* counts,
                    const int32_t* offsets, const float* row_w, void* ys, void* ws, size_t ws_bytes,
                    void* stream) {
  if (!shape_ok(s) || !h || !W2p || !counts || !offsets || !row_w || !ys) return MOE_ERR_INVALID;
  if (!aligned16(h) || !aligned16(W2p) || !aligned16(ys)) return MOE_ERR_INVALID;
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID;
  (void)ws_bytes;
  return launch_expert_down(static_cast<const __nv_bfloat16*>(h), static_cast<const __nv_bfloat16*>(W2p), counts,
                            offsets, row_w, static_cast<__half*>(ys), s->d, s->n, s->E, row_cap(s),
                            status_of(ws), kDefaultTimeoutNs, as_stream(stream));
}

int moe_combine(const moe_shape* s, const void* ys, const int32_t* tok_offsets, const int32_t* tok_rows, void* y,
                void* stream) {
  if (!shape_ok(s) || !ys || !tok_rows || !y || !aligned16(ys) || !aligned16(y)) return MOE_ERR_INVALID;
  launch_combine(static_cast<const __half*>(ys), tok_offsets, tok_rows, static_cast<float*>(y), s->T, s->d, s->k,
                 as_stream(stream));
  return last_launch();
}

int moe_combine_bf16(const moe_shape* s, const void* ys, const int32_t* tok_offsets, const int32_t* tok_rows,
                     void* y, void* stream) {
  if (!shape_ok(s) || !ys || !tok_rows || !y || !aligned16(ys) || !aligned16(y)) return MOE_ERR_INVALID;
  launch_combine(static_cast<const __half*>(ys), tok_offsets, tok_rows, static_cast<__nv_bfloat16*>(y), s->T, s->d,
                 s->k, as_stream(stream));
  return last_launch();
}

namespace {

// The layer with bf16 expert GEMMs: route (+ round) + permute, up, down,
// then the combine into y in fp32 or, with y_bf16, rounded to bf16.
int forward_layer(const moe_shape* s, const void* x, const float* Wr, const float* bias, const void* W13p,
                  const void* W2p, void* y, bool y_bf16, void* ws, size_t ws_bytes, void* stream) {
  if (!shape_ok(s) || !x || !Wr || !W13p || !W2p || !y) return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(W13p) || !aligned16(W2p) || !aligned16(y)) return MOE_ERR_INVALID;
  int st = check_ws(s, ws, ws_bytes);
  if (st != MOE_OK) return st;
  int64_t off[kNumSlots];
  layout(s, off);
  float* logits = at<float>(ws, off[kLogits]);
  int32_t* idx = at<int32_t>(ws, off[kTopkIdx]);
  float* w = at<float>(ws, off[kTopkW]);
  int32_t* counts = at<int32_t>(ws, off[kCounts]);
  int32_t* offsets = at<int32_t>(ws, off[kOffsets]);
  int32_t* src = at<int32_t>(ws, off[kSrc]);
  int32_t* dst = at<int32_t>(ws, off[kDst]);
  int32_t* row_token = at<int32_t>(ws, off[kRowToken]);
  float* row_w = at<float>(ws, off[kRowW]);
  int32_t* tok_offsets = at<int32_t>(ws, off[kTokOffsets]);
  int32_t* tok_rows = at<int32_t>(ws, off[kTokRows]);
  void* h = at<void>(ws, off[kH]);
  void* ys = at<void>(ws, off[kYs]);

  const int32_t* combine_offsets = nullptr;
  const int32_t* combine_rows = dst;
  if (s->round == MOE_ROUND_OFF) {
    if ((st = moe_route_permute(s, x, Wr, bias, logits, idx, w, counts, offsets, src, dst, row_token, row_w, ws,
                                ws_bytes, stream)) != MOE_OK)
      return st;
  } else {
    if ((st = moe_route(s, x, Wr, bias, logits, idx, w, ws, stream)) != MOE_OK) return st;
    if ((st = moe_token_round(s, logits, idx, counts, offsets, row_token, row_w, tok_offsets, tok_rows, ws, ws_bytes,
                              stream)) != MOE_OK)
      return st;
    combine_offsets = tok_offsets;
    combine_rows = tok_rows;
  }
  if ((st = moe_expert_up(s, x, W13p, counts, offsets, row_token, combine_offsets, combine_rows, h,
                          forward_gather(s), ws, ws_bytes, stream)) != MOE_OK)
    return st;
  if ((st = moe_expert_down(s, h, W2p, counts, offsets, row_w, ys, ws, ws_bytes, stream)) != MOE_OK) return st;
  return y_bf16 ? moe_combine_bf16(s, ys, combine_offsets, combine_rows, y, stream)
                : moe_combine(s, ys, combine_offsets, combine_rows, y, stream);
}

}  // namespace

int moe_forward(const moe_shape* s, const void* x, const float* Wr, const float* bias, const void* W13p,
                const void* W2p, void* y, void* ws, size_t ws_bytes, void* stream) {
  return forward_layer(s, x, Wr, bias, W13p, W2p, y, false, ws, ws_bytes, stream);
}

int moe_forward_bf16(const moe_shape* s, const void* x, const float* Wr, const float* bias, const void* W13p,
                     const void* W2p, void* y, void* ws, size_t ws_bytes, void* stream) {
  return forward_layer(s, x, Wr, bias, W13p, W2p, y, true, ws, ws_bytes, stream);
}

int moe_quantize_rows_fp8(const void* src, int64_t rows, int32_t K, void* codes, float* scales, void* stream) {
  if (!src || !codes || !scales || rows < 0 || K <= 0 || K % 16 != 0) return MOE_ERR_INVALID;
  if (!aligned16(src) || !aligned16(codes)) return MOE_ERR_INVALID;
  if (rows == 0) return MOE_OK;
  launch_quant_rows(static_cast<const __nv_bfloat16*>(src), rows, K, static_cast<uint8_t*>(codes), scales,
                    as_stream(stream));
  return last_launch();
}

int moe_expert_up_fp8(const moe_shape* s, const void* x, const void* W13q, const float* sW13, const int32_t* counts,
                      const int32_t* offsets, const int32_t* tok_offsets, const int32_t* tok_rows, void* h,
                      void* ws, size_t ws_bytes, void* stream) {
  if (!shape_ok(s) || !x || !W13q || !sW13 || !counts || !offsets || !tok_rows || !h) return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(W13q) || !aligned16(h)) return MOE_ERR_INVALID;
  if (s->n % 128 != 0 || s->d % 128 != 0) return MOE_ERR_UNSUPPORTED;
  const int st = check_ws(s, ws, ws_bytes);
  if (st != MOE_OK) return st;
  int64_t off[kNumSlots];
  layout(s, off);
  // the codes (cap x d bytes) and row scales (cap floats) fit in the ys
  // region (cap x d x 2 bytes), which the forward writes only afterwards
  const int64_t cap = row_cap(s);
  uint8_t* xq = at<uint8_t>(ws, off[kYs]);
  float* row_scale = reinterpret_cast<float*>(xq + cap * s->d);
  return launch_expert_up_f8(static_cast<const __nv_bfloat16*>(x), static_cast<const uint8_t*>(W13q), sW13, counts,
                             offsets, tok_rows, tok_offsets, static_cast<__nv_bfloat16*>(h), s->T, s->d, s->n, s->E,
                             s->k, cap, xq, row_scale, status_of(ws), kDefaultTimeoutNs, as_stream(stream));
}

int moe_quantize_experts_fp8(const void* src, int32_t E, int64_t m, void* codes, float* scales, void* stream) {
  if (!src || !codes || !scales || E <= 0 || m <= 0 || m % 16 != 0) return MOE_ERR_INVALID;
  if (!aligned16(src) || !aligned16(codes)) return MOE_ERR_INVALID;
  launch_quant_experts(static_cast<const __nv_bfloat16*>(src), E, m, static_cast<uint8_t*>(codes), scales,
                       as_stream(stream));
  return last_launch();
}

int moe_expert_down_fp8(const moe_shape* s, const void* h, const void* W2q, const float* sW2, const int32_t* counts,
                        const int32_t* offsets, const float* row_w, void* ys, void* ws, size_t ws_bytes,
                        void* stream) {
  if (!shape_ok(s) || !h || !W2q || !sW2 || !counts || !offsets || !row_w || !ys) return MOE_ERR_INVALID;
  if (!aligned16(h) || !aligned16(W2q) || !aligned16(ys)) return MOE_ERR_INVALID;
  if (s->n % 128 != 0 || s->d % 256 != 0) return MOE_ERR_UNSUPPORTED;
  const int st = check_ws(s, ws, ws_bytes, true);
  if (st != MOE_OK) return st;
  int64_t off[kNumSlots];
  layout(s, off, true);
  const int64_t cap = row_cap(s);
  uint8_t* hq = at<uint8_t>(ws, off[kHq]);
  float* h_scale = reinterpret_cast<float*>(hq + align256(cap * s->n));
  launch_quant_rows(static_cast<const __nv_bfloat16*>(h), cap, s->n, hq, h_scale, as_stream(stream));
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  return launch_expert_down_f8(hq, h_scale, static_cast<const uint8_t*>(W2q), sW2, counts, offsets, row_w,
                               static_cast<__half*>(ys), s->d, s->n, s->E, cap, status_of(ws), kDefaultTimeoutNs,
                               as_stream(stream));
}

int moe_forward_fp8(const moe_shape* s, const void* x, const float* Wr, const float* bias, const void* W13q,
                    const float* sW13, const void* W2q, const float* sW2, void* y, void* ws, size_t ws_bytes,
                    void* stream) {
  if (!shape_ok(s) || !x || !Wr || !W13q || !sW13 || !W2q || !sW2 || !y) return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(W13q) || !aligned16(W2q) || !aligned16(y)) return MOE_ERR_INVALID;
  if (s->n % 128 != 0 || s->d % 256 != 0) return MOE_ERR_UNSUPPORTED;
  int st = check_ws(s, ws, ws_bytes, true);
  if (st != MOE_OK) return st;
  int64_t off[kNumSlots];
  layout(s, off);
  float* logits = at<float>(ws, off[kLogits]);
  int32_t* idx = at<int32_t>(ws, off[kTopkIdx]);
  float* w = at<float>(ws, off[kTopkW]);
  int32_t* counts = at<int32_t>(ws, off[kCounts]);
  int32_t* offsets = at<int32_t>(ws, off[kOffsets]);
  int32_t* src = at<int32_t>(ws, off[kSrc]);
  int32_t* dst = at<int32_t>(ws, off[kDst]);
  int32_t* row_token = at<int32_t>(ws, off[kRowToken]);
  float* row_w = at<float>(ws, off[kRowW]);
  int32_t* tok_offsets = at<int32_t>(ws, off[kTokOffsets]);
  int32_t* tok_rows = at<int32_t>(ws, off[kTokRows]);
  void* h = at<void>(ws, off[kH]);
  void* ys = at<void>(ws, off[kYs]);
  const int32_t* combine_offsets = nullptr;
  const int32_t* combine_rows = dst;
  if (s->round == MOE_ROUND_OFF) {
    if ((st = moe_route_permute(s, x, Wr, bias, logits, idx, w, counts, offsets, src, dst, row_token, row_w, ws,
                                ws_bytes, stream)) != MOE_OK)
      return st;
  } else {
    if ((st = moe_route(s, x, Wr, bias, logits, idx, w, ws, stream)) != MOE_OK) return st;
    if ((st = moe_token_round(s, logits, idx, counts, offsets, row_token, row_w, tok_offsets, tok_rows, ws, ws_bytes,
                              stream)) != MOE_OK)
      return st;
    combine_offsets = tok_offsets;
    combine_rows = tok_rows;
  }
  if ((st = moe_expert_up_fp8(s, x, W13q, sW13, counts, offsets, combine_offsets, combine_rows, h, ws, ws_bytes,
                              stream)) != MOE_OK)
    return st;
  if ((st = moe_expert_down_fp8(s, h, W2q, sW2, counts, offsets, row_w, ys, ws, ws_bytes, stream)) != MOE_OK)
    return st;
  return moe_combine(s, ys, combine_offsets, combine_rows, y, stream);
}

size_t moe_backward_workspace_bytes(const moe_shape* s) {
  if (!shape_ok(s) || !bwd_shape_ok(s)) return 0;
  int64_t off_f[kNumSlots], off[kNumBwdSlots];
  return static_cast<size_t>(layout_bwd(s, off_f, off));
}

int moe_prepare_weights_bwd(const moe_shape* s, const void* W1, const void* W3, void* W13i, void* stream) {
  if (!shape_ok(s) || !W1 || !W3 || !W13i || !aligned16(W13i)) return MOE_ERR_INVALID;
  launch_prepare_weights_bwd(static_cast<const __nv_bfloat16*>(W1), static_cast<const __nv_bfloat16*>(W3),
                             static_cast<__nv_bfloat16*>(W13i), s->E, s->d, s->n, as_stream(stream));
  return last_launch();
}

int moe_backward(const moe_shape* s, const void* x, const float* Wr, const float* bias, const void* W13p,
                 const void* W13i, const void* W2, const void* dy, float* dx, float* dWr, float* dbias, float* dW1,
                 float* dW3, float* dW2, void* ws, size_t ws_bytes, void* stream) {
  if (!shape_ok(s) || !x || !Wr || !W13p || !W13i || !W2 || !dy || !dx || !dWr || !dW1 || !dW3 || !dW2)
    return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(W13p) || !aligned16(W13i) || !aligned16(W2) || !aligned16(dy) || !aligned16(dx) ||
      !aligned16(dW1) || !aligned16(dW3) || !aligned16(dW2))
    return MOE_ERR_INVALID;
  if (!bwd_shape_ok(s)) return MOE_ERR_UNSUPPORTED;
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID;
  int64_t off_f[kNumSlots], off[kNumBwdSlots];
  if (static_cast<int64_t>(ws_bytes) < layout_bwd(s, off_f, off)) return MOE_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  const int T = s->T, d = s->d, n = s->n, E = s->E, k = s->k;
  const int64_t A = static_cast<int64_t>(T) * k, capp = padded_cap(s);
  float* logits = at<float>(ws, off_f[kLogits]);
  int32_t* idx = at<int32_t>(ws, off_f[kTopkIdx]);
  float* w = at<float>(ws, off_f[kTopkW]);
  int32_t* counts = at<int32_t>(ws, off_f[kCounts]);
  int32_t* offsets = at<int32_t>(ws, off_f[kOffsets]);
  int32_t* src = at<int32_t>(ws, off_f[kSrc]);
  int32_t* dst = at<int32_t>(ws, off_f[kDst]);
  int32_t* row_token = at<int32_t>(ws, off_f[kRowToken]);
  float* row_w = at<float>(ws, off_f[kRowW]);
  int32_t* offsets_p = at<int32_t>(ws, off[kOffP]);
  int32_t* rowp = at<int32_t>(ws, off[kRowP]);
  float* wp = at<float>(ws, off[kWp]);
  int32_t* tok_offsets = at<int32_t>(ws, off_f[kTokOffsets]);
  int32_t* tok_rows = at<int32_t>(ws, off_f[kTokRows]);
  __nv_bfloat16* xp = at<__nv_bfloat16>(ws, off[kXp]);
  __nv_bfloat16* dyp = at<__nv_bfloat16>(ws, off[kDyp]);
  float* gl = at<float>(ws, off[kGl]);
  __nv_bfloat16* dgl = at<__nv_bfloat16>(ws, off[kDgl]);
  __nv_bfloat16* hw = at<__nv_bfloat16>(ws, off[kHw]);
  float* dw_part = at<float>(ws, off[kDwPart]);
  __half* dxr = at<__half>(ws, off[kDxr]);
  float* dlp = at<float>(ws, off[kDlp]);
  float* WrT = at<float>(ws, off[kWrT]);
  int32_t* status = status_of(ws);

  // 1. routing, recomputed: the same kernels and bits as the forward.  Each
  // token's rows form a list (rows, tok_offs) with a weight per row (wrow).
  int rc;
  const int32_t* rows;
  const int32_t* tok_offs;
  const float* wrow;
  if (s->round == MOE_ROUND_OFF) {
    if ((rc = moe_route_permute(s, x, Wr, bias, logits, idx, w, counts, offsets, src, dst, row_token, row_w, ws,
                                ws_bytes, stream)) != MOE_OK)
      return rc;
    launch_bwd_pad_offsets(counts, E, offsets_p, st);
    launch_bwd_rows(idx, w, dst, offsets, offsets_p, A, rowp, wp, st);
    rows = rowp;
    tok_offs = nullptr;
    wrow = wp;
  } else {
    if ((rc = moe_route(s, x, Wr, bias, logits, idx, w, ws, stream)) != MOE_OK) return rc;
    if ((rc = moe_token_round(s, logits, idx, counts, offsets, row_token, row_w, tok_offsets, tok_rows, ws, ws_bytes,
                              stream)) != MOE_OK)
      return rc;
    // rounded counts are multiples of the tile (64, 128 or 256): the padded
    // offsets equal the forward's, so its rows and row weights serve as they are
    launch_bwd_pad_offsets(counts, E, offsets_p, st);
    rows = tok_rows;
    tok_offs = tok_offsets;
    wrow = row_w;
  }
  // 2. zero padding, gathered x and dy
  launch_bwd_zero_pad(counts, offsets_p, E, d, n, xp, dyp, dgl, hw, st);
  launch_gather_rows_by_token(static_cast<const __nv_bfloat16*>(x), rows, tok_offs, T, k, d, xp, st);
  launch_gather_rows_by_token(static_cast<const __nv_bfloat16*>(dy), rows, tok_offs, T, k, d, dyp, st);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  // 3. pre-activations, then the SwiGLU backward fused into dh' = dy W2^T
  if ((rc = launch_expert_up_pre(xp, static_cast<const __nv_bfloat16*>(W13p), counts, offsets_p, gl, d, n, E, capp,
                                 status, kDefaultTimeoutNs, st)) != MOE_OK)
    return rc;
  if ((rc = launch_bwd_act(dyp, static_cast<const __nv_bfloat16*>(W2), counts, offsets_p, wrow, gl, dgl, hw, dw_part, d,
                           n, E, capp, status, kDefaultTimeoutNs, st)) != MOE_OK)
    return rc;
  // 4. gate weights -> logits
  launch_router_bwd(rows, tok_offs, wrow, dw_part, bwd_act_parts(n), T, k, dlp, st);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  // 5. weight gradients: dW2 = (w h)^T dy, dW1 / dW3 = x^T (dg, du)
  if ((rc = launch_wgrad(dyp, hw, counts, offsets_p, d, n, E, capp, dW2, nullptr, status, kDefaultTimeoutNs, st)) !=
      MOE_OK)
    return rc;
  if ((rc = launch_wgrad(dgl, xp, counts, offsets_p, 2 * n, d, E, capp, dW1, dW3, status, kDefaultTimeoutNs, st)) !=
      MOE_OK)
    return rc;
  // 6. dx: per row the expert path [dg du] W13i^T plus the gate network's
  // dL Wr[:, e] (fp16), then each token's rows summed in list order
  launch_transpose_router(Wr, d, E, WrT, st);
  if ((rc = launch_expert_dx(dgl, static_cast<const __nv_bfloat16*>(W13i), counts, offsets_p, dlp, WrT, dxr, d, n, E,
                             capp, status, kDefaultTimeoutNs, st)) != MOE_OK)
    return rc;
  launch_combine(dxr, tok_offs, rows, dx, T, d, k, st);
  // 7. dWr = x^T dL, db = sum dL
  launch_bwd_dwr(xp, dlp, counts, offsets_p, E, d, at<float>(ws, off[kDwrPart]), at<float>(ws, off[kDbPart]), dWr,
                 dbias, st);
  return last_launch();
}

int moe_selftest_timeout(void* ws, uint64_t timeout_ns, void* stream) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID;
  if (cudaMemsetAsync(ws, 0, kStatusBytes, as_stream(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  launch_selftest_timeout(status_of(ws), timeout_ns, as_stream(stream));
  return last_launch();
}

}  // extern "C"
