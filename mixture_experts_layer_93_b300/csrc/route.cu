// Router: gate-network logits and top-k gating.
//
// Gate network and top_k of the moe_forward pseudocode
// ("MoE架构的物理瓶颈与扩展限制解析", section 工作原理, step 1) and steps 1-2 of
// the fused MoE kernel ("硬件加速的考量", section 自定义核与核融合).
#include "common.cuh"
#include "kernels.h"

namespace moe {

// ---------------------------------------------------------------------------
// logits[T, E] = float(x[T, d]) @ Wr[d, E] + bias[E]   (fp32 FMA, K ascending)
//
// Block tile: 64 tokens x BE experts, K step 32.  256 threads; each thread owns
// 4 tokens x (BE/16) experts.  x is converted bf16 -> fp32 (exact) on the way
// into shared memory.
template <int BE>
__global__ void __launch_bounds__(256) router_logits_kernel(const __nv_bfloat16* __restrict__ x,
                                                            const float* __restrict__ Wr,
                                                            const float* __restrict__ bias,
                                                            float* __restrict__ logits, int T, int d, int E) {
  constexpr int BM = 64, BK = 32, RE = BE / 16;
  __shared__ float xs[BK][BM + 4];
  __shared__ float ws[BK][BE];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * BM;
  const int e0 = blockIdx.y * BE;
  const int ty = tid / 16, tx = tid % 16;
  float acc[4][RE];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < RE; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < d; k0 += BK) {
    // x tile: 64 tokens x 32 k = 256 threads x 8 elements (one 16-byte load)
    {
      const int r = tid / 4, c = (tid % 4) * 8;
      const int t = t0 + r;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < T) v = *reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d + k0 + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xs[c + 2 * q][r] = bf16_lo(w[q]);
        xs[c + 2 * q + 1][r] = bf16_hi(w[q]);
      }
    }
    // Wr tile: 32 k x BE experts
    for (int i = tid; i < BK * BE; i += 256) {
      const int kk = i / BE, ee = i % BE;
      const int e = e0 + ee;
      ws[kk][ee] = (e < E) ? Wr[static_cast<size_t>(k0 + kk) * E + e] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[RE];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < RE; ++j) b[j] = ws[kk][tx * RE + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < RE; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < RE; ++j) {
      const int e = e0 + tx * RE + j;
      if (e < E) logits[static_cast<size_t>(t) * E + e] = acc[i][j] + (bias ? bias[e] : 0.f);
    }
  }
}

void launch_router_logits(const __nv_bfloat16* x, const float* Wr, const float* bias, float* logits, int T, int d,
                          int E, cudaStream_t stream) {
  const int gx = (T + 63) / 64;
  if (E <= 16) {
    router_logits_kernel<16><<<dim3(gx, 1), 256, 0, stream>>>(x, Wr, bias, logits, T, d, E);
  } else if (E <= 32) {
    router_logits_kernel<32><<<dim3(gx, 1), 256, 0, stream>>>(x, Wr, bias, logits, T, d, E);
  } else {
    router_logits_kernel<64><<<dim3(gx, (E + 63) / 64), 256, 0, stream>>>(x, Wr, bias, logits, T, d, E);
  }
}

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

void launch_topk_gating(const float* logits, int32_t* idx, float* w, int T, int E, int k, int32_t* status,
                        cudaStream_t stream) {
  const int blocks = (T + 7) / 8;
  const int nv = (E + 31) / 32;
  if (nv <= 1)
    topk_gating_kernel<1><<<blocks, 256, 0, stream>>>(logits, idx, w, T, E, k, status);
  else if (nv <= 2)
    topk_gating_kernel<2><<<blocks, 256, 0, stream>>>(logits, idx, w, T, E, k, status);
  else if (nv <= 4)
    topk_gating_kernel<4><<<blocks, 256, 0, stream>>>(logits, idx, w, T, E, k, status);
  else if (nv <= 8)
    topk_gating_kernel<8><<<blocks, 256, 0, stream>>>(logits, idx, w, T, E, k, status);
  else if (nv <= 16)
    topk_gating_kernel<16><<<blocks, 256, 0, stream>>>(logits, idx, w, T, E, k, status);
  else
    topk_gating_kernel<32><<<blocks, 256, 0, stream>>>(logits, idx, w, T, E, k, status);
}

}  // namespace moe
