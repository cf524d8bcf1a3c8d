// Router: top-k gating over the gate-network logits (the logits themselves
// come from the tensor-core GEMM in gemm.cu).
//
// Gate network and top_k of the moe_forward pseudocode
// ("MoE架构的物理瓶颈与扩展限制解析", section 工作原理, step 1) and steps 1-2 of
// the fused MoE kernel ("硬件加速的考量", section 自定义核与核融合).
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Top-k gating: one warp per token.  Lane l holds logits of experts
// l, l+32, ...; k rounds of a warp arg-max pick the experts in descending
// order of logit, equal logits going to the lower expert id.  Gate weights are
// softmax over the selected logits: w_j = exp(L_j - L_max) / sum_j' exp(...).
template <int NV>
__global__ void __launch_bounds__(256) topk_gating_kernel(const float* __restrict__ logits,
                                                          int32_t* __restrict__ topk_idx,
                                                          float* __restrict__ topk_w, int T, int E, int k,
                                                          int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  const float* row = logits + static_cast<size_t>(t) * E;
  float v[NV];
  bool nan_seen = false;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    float val = (e < E) ? row[e] : -INFINITY;
    if (val != val) {  // NaN ranks lowest
      nan_seen = true;
      val = -INFINITY;
    }
    v[i] = val;
  }
  if (__any_sync(0xffffffffu, nan_seen) && lane == 0) report_error(status, MOE_ERR_DEVICE_CHECK, t);
  uint32_t taken = 0;  // bit i: v[i] already selected
  // experts past E are never eligible
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (lane + 32 * i >= E) taken |= 1u << i;

  float my_v = -INFINITY;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bid = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      if (!(taken >> i & 1u) && (v[i] > bv || (v[i] == bv && e < bid))) {
        bv = v[i];
        bid = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oid = __shfl_xor_sync(0xffffffffu, bid, off);
      if (ov > bv || (ov == bv && oid < bid)) {
        bv = ov;
        bid = oid;
      }
    }
    if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
    if (lane == j) {
      my_v = bv;
      my_id = bid;
    }
  }
  const float vmax = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - vmax) : 0.f;
  // sum in slot order j = 0..k-1 (lane 0 walks the lanes)
  float s = 0.f;
  for (int j = 0; j < k; ++j) s += __shfl_sync(0xffffffffu, ex, j);
  if (lane < k) {
    topk_idx[static_cast<size_t>(t) * k + lane] = my_id;
    topk_w[static_cast<size_t>(t) * k + lane] = ex / s;
  }
}

// ---------------------------------------------------------------------------
// The same selection with each lane's candidates pre-sorted (E <= 256), over
// the 64-bit keys of topk.cuh: a round is one warp max over the lanes' heads,
// and the winning lane shifts its list.
template <int NV>
__global__ void __launch_bounds__(256) topk_gating_sorted_kernel(const float* __restrict__ logits,
                                                                 int32_t* __restrict__ topk_idx,
                                                                 float* __restrict__ topk_w, int T, int E, int k,
                                                                 int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  bool nan_seen;
  const uint64_t mine = warp_topk_key<NV>(logits + static_cast<size_t>(t) * E, E, k, lane, nan_seen);
  if (__any_sync(0xffffffffu, nan_seen) && lane == 0) report_error(status, MOE_ERR_DEVICE_CHECK, t);
  const float w = warp_gate_weight(mine, k, lane);
  if (lane < k) {
    topk_idx[static_cast<size_t>(t) * k + lane] = topk_key_expert(mine);
    topk_w[static_cast<size_t>(t) * k + lane] = w;
  }
}

void launch_topk_gating(const float* logits, int32_t* idx, float* w, int T, int E, int k, int32_t* status,
                        cudaStream_t stream) {
  const int blocks = (T + 7) / 8;
  const int nv = (E + 31) / 32;
  if (nv <= 1)
    launch_pdl(topk_gating_sorted_kernel<1>, blocks, 256, 0, stream, 1, logits, idx, w, T, E, k, status);
  else if (nv <= 2)
    launch_pdl(topk_gating_sorted_kernel<2>, blocks, 256, 0, stream, 1, logits, idx, w, T, E, k, status);
  else if (nv <= 4)
    launch_pdl(topk_gating_sorted_kernel<4>, blocks, 256, 0, stream, 1, logits, idx, w, T, E, k, status);
  else if (nv <= 8)
    launch_pdl(topk_gating_sorted_kernel<8>, blocks, 256, 0, stream, 1, logits, idx, w, T, E, k, status);
  else if (nv <= 16)
    launch_pdl(topk_gating_kernel<16>, blocks, 256, 0, stream, 1, logits, idx, w, T, E, k, status);
  else
    launch_pdl(topk_gating_kernel<32>, blocks, 256, 0, stream, 1, logits, idx, w, T, E, k, status);
}

}  // namespace moe
