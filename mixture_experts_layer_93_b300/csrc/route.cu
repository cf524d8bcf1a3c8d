// Router: top-k gating over the gate-network logits (the logits themselves
// come from the tensor-core GEMM in gemm.cu).
//
// Gate network and top_k of the moe_forward pseudocode
// ("MoE架构的物理瓶颈与扩展限制解析", section 工作原理, step 1) and steps 1-2 of
// the fused MoE kernel ("硬件加速的考量", section 自定义核与核融合).
#include "common.cuh"
#include "kernels.h"

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
// The same selection with each lane's candidates pre-sorted (E <= 256).
//
// Logit L of expert e becomes the 64-bit key (ord(L) << 32) | (2^32-1 - e),
// where ord maps float order onto unsigned order (-0 taken as +0, NaN as
// -inf): a larger key is a larger logit, or an equal logit of a lower expert,
// which is exactly the order the k rounds above pick in.  Lane l sorts its NV
// keys once (Batcher's odd-even merge network); a round is then one warp
// max over the lanes' heads, and the winning lane shifts its list.
__device__ __forceinline__ uint64_t topk_key(float v, int e) {
  if (v != v) v = -INFINITY;
  if (v == 0.f) v = 0.f;  // -0 ranks with +0
  const uint32_t b = __float_as_uint(v);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | (0xffffffffu - static_cast<uint32_t>(e));
}

__device__ __forceinline__ float topk_key_value(uint64_t key) {
  const uint32_t ord = static_cast<uint32_t>(key >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7fffffffu) : ~ord);
}

template <int NV>
__device__ __forceinline__ void sort_desc(uint64_t (&a)[NV]) {
  // Batcher's odd-even merge sort network for NV a power of two
#pragma unroll
  for (int p = 1; p < NV; p <<= 1) {
#pragma unroll
    for (int q = p; q >= 1; q >>= 1) {
#pragma unroll
      for (int j = q % p; j + q < NV; j += 2 * q) {
#pragma unroll
        for (int i = 0; i < q; ++i) {
          if (i + j + q < NV && (i + j) / (2 * p) == (i + j + q) / (2 * p)) {
            const uint64_t x = a[i + j], y = a[i + j + q];
            a[i + j] = x > y ? x : y;
            a[i + j + q] = x > y ? y : x;
          }
        }
      }
    }
  }
}

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
  const float* row = logits + static_cast<size_t>(t) * E;
  uint64_t key[NV];
  bool nan_seen = false;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float val = row[e];
      nan_seen |= (val != val);
      key[i] = topk_key(val, e);
    } else {
      key[i] = 0;  // below every real key: never selected (k <= E)
    }
  }
  if (__any_sync(0xffffffffu, nan_seen) && lane == 0) report_error(status, MOE_ERR_DEVICE_CHECK, t);
  sort_desc<NV>(key);
  uint64_t mine = 0;
  for (int j = 0; j < k; ++j) {
    uint64_t best = key[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, best, off);
      best = o > best ? o : best;
    }
    if (((0xffffffffu - static_cast<uint32_t>(best)) & 31u) == static_cast<uint32_t>(lane)) {
#pragma unroll
      for (int i = 0; i + 1 < NV; ++i) key[i] = key[i + 1];
      key[NV - 1] = 0;
    }
    if (lane == j) mine = best;
  }
  const float my_v = topk_key_value(mine);
  const float vmax = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - vmax) : 0.f;
  float s = 0.f;
  for (int j = 0; j < k; ++j) s += __shfl_sync(0xffffffffu, ex, j);
  if (lane < k) {
    topk_idx[static_cast<size_t>(t) * k + lane] = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(mine));
    topk_w[static_cast<size_t>(t) * k + lane] = ex / s;
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
