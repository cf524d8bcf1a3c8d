// Combine: expert outputs back to token order, weighted by the gate scores
// (step 5 of the fused kernel in "硬件加速的考量", section 自定义核与核融合;
// the reverse dispatch of the moe_forward pseudocode in
// "MoE架构的物理瓶颈与扩展限制解析", section 工作原理, done in place on one GPU).
//
// The gate weight is already applied by the down-projection epilogue, so
// y[t] = sum_j ys[row_j] (ys fp16, sum in fp32) in the token's list order:
// deterministic, no atomics.  y is the fp32 sum, or that sum rounded to
// nearest-even bf16 (the layer's output in a bf16 model: half the bytes to
// write and to copy out).  Each thread owns 8 columns: one 16-byte load per
// row, two 16-byte stores (fp32) or one (bf16).
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace moe {

template <typename OutT>
__global__ void __launch_bounds__(256) combine_kernel(const __half* __restrict__ ys,
                                                      const int32_t* __restrict__ tok_offsets,
                                                      const int32_t* __restrict__ tok_rows, OutT* __restrict__ y,
                                                      int T, int d, int k) {
  pdl_wait();
  pdl_trigger();
  const int groups = d / 8;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(T) * groups) return;
  const int t = static_cast<int>(i / groups);
  const int g = static_cast<int>(i % groups);
  int r0, r1;
  if (tok_offsets) {
    r0 = tok_offsets[t];
    r1 = tok_offsets[t + 1];
  } else {
    r0 = t * k;
    r1 = r0 + k;
  }
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.f;
  for (int j = r0; j < r1; ++j) {
    const int64_t row = tok_rows[j];
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(ys + row * d) + g);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = unpack_half2(w[q]);
      acc[2 * q] += f.x;
      acc[2 * q + 1] += f.y;
    }
  }
  if constexpr (std::is_same_v<OutT, float>) {
    float4* out = reinterpret_cast<float4*>(y + static_cast<int64_t>(t) * d) + 2 * g;
    out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  } else {
    uint4* out = reinterpret_cast<uint4*>(y + static_cast<int64_t>(t) * d) + g;
    *out = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                      pack_bf16x2(acc[6], acc[7]));
  }
}

namespace {
template <typename OutT>
void launch_combine_as(const __half* ys, const int32_t* tok_offsets, const int32_t* tok_rows, OutT* y, int T, int d,
                       int k, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(T) * (d / 8);
  const int blocks = static_cast<int>((total + 255) / 256);
  launch_pdl(combine_kernel<OutT>, blocks, 256, 0, stream, 1, ys, tok_offsets, tok_rows, y, T, d, k);
}
}  // namespace

void launch_combine(const __half* ys, const int32_t* tok_offsets, const int32_t* tok_rows, float* y, int T, int d,
                    int k, cudaStream_t stream) {
  launch_combine_as(ys, tok_offsets, tok_rows, y, T, d, k, stream);
}

void launch_combine(const __half* ys, const int32_t* tok_offsets, const int32_t* tok_rows, __nv_bfloat16* y, int T,
                    int d, int k, cudaStream_t stream) {
  launch_combine_as(ys, tok_offsets, tok_rows, y, T, d, k, stream);
}

}  // namespace moe
