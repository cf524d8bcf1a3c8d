// Top-k keys shared by the top-k kernels (route.cu) and the fused
// top-k + histogram + scan kernel (permute.cu).
//
// Logit L of expert e becomes the 64-bit key (ord(L) << 32) | (2^32-1 - e),
// where ord maps float order onto unsigned order (-0 taken as +0, NaN as
// -inf): a larger key is a larger logit, or an equal logit of a lower expert,
// which is the order the top-k of "MoE架构的物理瓶颈与扩展限制解析" (section
// 工作原理, step 1) takes with ties to the lower expert id.
#pragma once

#include "common.cuh"

namespace moe {

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

// Top-k of one token's E <= 32*NV logits by one warp: lane j < k returns
// the key of slot j (descending key order), the other lanes 0.  nan_seen
// tells whether a logit was NaN.
template <int NV>
__device__ __forceinline__ uint64_t warp_topk_key(const float* __restrict__ row, int E, int k, int lane,
                                                  bool& nan_seen) {
  uint64_t key[NV];
  nan_seen = false;
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
  return mine;
}

// Gate weights of the selected slots: softmax over the k selected logits,
// w_j = exp(L_j - L_0) / sum_j' exp(L_j' - L_0) (slot 0 holds the maximum),
// the sum taken in slot order.  Lane j < k returns w_j.
__device__ __forceinline__ float warp_gate_weight(uint64_t mine, int k, int lane) {
  const float my_v = topk_key_value(mine);
  const float vmax = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - vmax) : 0.f;
  float s = 0.f;
  for (int j = 0; j < k; ++j) s += __shfl_sync(0xffffffffu, ex, j);
  return ex / s;
}

__device__ __forceinline__ int32_t topk_key_expert(uint64_t key) {
  return static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(key));
}

}  // namespace moe
