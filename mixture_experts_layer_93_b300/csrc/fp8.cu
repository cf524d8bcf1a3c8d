// FP8 (e4m3) quantisation for the FP8 up-projection.
//
// The pages name FP8 among the precisions MoE compute runs in
// ("硬件加速的考量", section 量化) and fix no recipe.  Reading: one fp32 scale
// per row (a token's activations, or one output channel of the packed gate /
// linear weights), scale = fp32(amax / 448), code = e4m3(fp32(x * fp32(448 /
// amax))) with round-to-nearest-even and saturation to +-448; an all-zero row
// has scale 1 and codes 0.  Every fp32 operation is IEEE round-to-nearest
// (explicit _rn intrinsics, so no contraction changes a bit).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// amax of a K-element bf16 row (K % 8 == 0, 16-byte aligned) by one warp.
__device__ __forceinline__ float row_amax(const __nv_bfloat16* __restrict__ row, int K, int lane) {
  const uint4* r4 = reinterpret_cast<const uint4*>(row);
  float m = 0.f;
  for (int g = lane; g < K / 8; g += 32) {
    const uint4 v = __ldg(r4 + g);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  return m;
}

// Eight e4m3 codes of the 16-byte group g of a row: x * inv, rounded.
__device__ __forceinline__ uint2 codes8(const __nv_bfloat16* __restrict__ row, int g, float inv) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + g);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint16_t a = cvt_e4m3x2(__fmul_rn(bf16_lo(w[2 * i]), inv), __fmul_rn(bf16_hi(w[2 * i]), inv));
    const uint16_t b = cvt_e4m3x2(__fmul_rn(bf16_lo(w[2 * i + 1]), inv), __fmul_rn(bf16_hi(w[2 * i + 1]), inv));
    c[i] = static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
  }
  return make_uint2(c[0], c[1]);
}

__device__ __forceinline__ void row_scales(float amax, float& scale, float& inv) {
  if (amax > 0.f) {
    scale = __fdiv_rn(amax, 448.f);
    inv = __fdiv_rn(448.f, amax);
  } else {
    scale = 1.f;
    inv = 0.f;  // codes 0
  }
}

// codes[r] / scales[r] of rows [rows, K] bf16, one warp per row.
__global__ void __launch_bounds__(256) quant_rows_kernel(const __nv_bfloat16* __restrict__ src, int64_t rows, int K,
                                                         uint8_t* __restrict__ codes, float* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  if (r >= rows) return;
  const __nv_bfloat16* row = src + r * K;
  float scale, inv;
  row_scales(row_amax(row, K, lane), scale, inv);
  uint2* out = reinterpret_cast<uint2*>(codes + r * K);
  for (int g = lane; g < K / 8; g += 32) out[g] = codes8(row, g, inv);
  if (lane == 0) scales[r] = scale;
}

void launch_quant_rows(const __nv_bfloat16* src, int64_t rows, int K, uint8_t* codes, float* scales,
                       cudaStream_t stream) {
  const int64_t blocks = (rows + 7) / 8;
  launch_pdl(quant_rows_kernel, static_cast<unsigned>(blocks), 256, 0, stream, 1, src, rows, K, codes, scales);
}

// Token-order gather with quantisation: one warp per token quantises x[t]
// once and writes its codes to each of the token's rows (tok_rows[tok_offsets
// [t] ..), or tok_rows[t*k .. t*k+k) without offsets); row_scale[row] gets
// the token's scale.
__global__ void __launch_bounds__(256) gather_quant_kernel(const __nv_bfloat16* __restrict__ x,
                                                           const int32_t* __restrict__ tok_rows,
                                                           const int32_t* __restrict__ tok_offsets, int T, int k,
                                                           int d, uint8_t* __restrict__ xq,
                                                           float* __restrict__ row_scale) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  const int r0 = tok_offsets ? tok_offsets[t] : t * k;
  const int r1 = tok_offsets ? tok_offsets[t + 1] : r0 + k;
  if (r0 == r1) return;
  const __nv_bfloat16* row = x + static_cast<int64_t>(t) * d;
  float scale, inv;
  row_scales(row_amax(row, d, lane), scale, inv);
  for (int g = lane; g < d / 8; g += 32) {
    const uint2 c = codes8(row, g, inv);
    for (int j = r0; j < r1; ++j) reinterpret_cast<uint2*>(xq + static_cast<int64_t>(tok_rows[j]) * d)[g] = c;
  }
  if (lane < r1 - r0) row_scale[tok_rows[r0 + lane]] = scale;
  for (int j = r0 + 32 + lane; j < r1; j += 32) row_scale[tok_rows[j]] = scale;
}

void launch_gather_quant(const __nv_bfloat16* x, const int32_t* tok_rows, const int32_t* tok_offsets, int T, int k,
                         int d, uint8_t* xq, float* row_scale, cudaStream_t stream) {
  launch_pdl(gather_quant_kernel, (T + 7) / 8, 256, 0, stream, 1, x, tok_rows, tok_offsets, T, k, d, xq, row_scale);
}

}  // namespace moe

namespace moe {

// One scale for each of E rows of m elements (a whole expert's W2): the
// maximum |x| over many blocks by atomicMax on the bits of non-negative
// floats (their order is the unsigned order of the bits; the result does not
// depend on the order of the updates), then the codes, then the scales.
__global__ void __launch_bounds__(256) quant_expert_amax_kernel(const __nv_bfloat16* __restrict__ src, int64_t m,
                                                                uint32_t* __restrict__ amax_bits) {
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.y;
  const uint4* r4 = reinterpret_cast<const uint4*>(src + static_cast<int64_t>(e) * m);
  float a = 0.f;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < m / 8;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(r4 + g);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
  if ((threadIdx.x & 31) == 0) atomicMax(&amax_bits[e], __float_as_uint(a));
}

__global__ void __launch_bounds__(256) quant_expert_codes_kernel(const __nv_bfloat16* __restrict__ src, int64_t m,
                                                                 const uint32_t* __restrict__ amax_bits,
                                                                 uint8_t* __restrict__ codes) {
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.y;
  float scale, inv;
  row_scales(__uint_as_float(amax_bits[e]), scale, inv);
  const __nv_bfloat16* row = src + static_cast<int64_t>(e) * m;
  uint2* out = reinterpret_cast<uint2*>(codes + static_cast<int64_t>(e) * m);
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < m / 8;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[g] = codes8(row, static_cast<int>(g), inv);
}

__global__ void quant_expert_scale_kernel(int E, uint32_t* __restrict__ amax_bits_in_scales) {
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float scale, inv;
    row_scales(__uint_as_float(amax_bits_in_scales[e]), scale, inv);
    amax_bits_in_scales[e] = __float_as_uint(scale);
  }
}

// scales doubles as the amax buffer until the last kernel turns it into scales.
void launch_quant_experts(const __nv_bfloat16* src, int E, int64_t m, uint8_t* codes, float* scales,
                          cudaStream_t stream) {
  uint32_t* bits = reinterpret_cast<uint32_t*>(scales);
  cudaMemsetAsync(bits, 0, static_cast<size_t>(E) * sizeof(uint32_t), stream);
  const int64_t groups = m / 8;
  const unsigned bx = static_cast<unsigned>(std::min<int64_t>((groups + 255) / 256, 1024));
  launch_pdl(quant_expert_amax_kernel, dim3(bx, E), 256, 0, stream, 1, src, m, bits);
  launch_pdl(quant_expert_codes_kernel, dim3(bx, E), 256, 0, stream, 1, src, m,
             static_cast<const uint32_t*>(bits), codes);
  launch_pdl(quant_expert_scale_kernel, 1, 256, 0, stream, 1, E, bits);
}

}  // namespace moe
