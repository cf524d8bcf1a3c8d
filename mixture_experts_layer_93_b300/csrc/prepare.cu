// One-time repack of the expert weights into the K-major layouts the grouped
// GEMMs stream with TMA (both operands of a tcgen05 MMA are read K-major).
//
//   W13p[e][2j][i]     = W1[e][i][j]   (gate branch, column j)
//   W13p[e][2j + 1][i] = W3[e][i][j]   (linear branch, column j)
//   W2p[e][i][j]       = W2[e][j][i]
//
// Interleaving gate and linear rows pairwise puts both halves of SwiGLU for
// output column j in adjacent accumulator columns of every tile, whatever its
// width, so the activation runs in the epilogue.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// dst[e][map(c)][r] = src[e][r][c] for a [rows, cols] source per expert.
// mode 0: identity row map (W2 -> W2p); mode 1/2: W1/W3 into W13p.
__global__ void __launch_bounds__(256) transpose_pack_kernel(const __nv_bfloat16* __restrict__ src,
                                                             __nv_bfloat16* __restrict__ dst, int rows, int cols,
                                                             int mode, int64_t dst_expert_stride) {
  __shared__ __nv_bfloat16 tile[32][33];
  const int e = blockIdx.z;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const __nv_bfloat16* s = src + static_cast<int64_t>(e) * rows * cols;
  __nv_bfloat16* dd = dst + static_cast<int64_t>(e) * dst_expert_stride;
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
  for (int i = ty; i < 32; i += 8) {
    const int r = r0 + i, c = c0 + tx;
    if (r < rows && c < cols) tile[i][tx] = s[static_cast<int64_t>(r) * cols + c];
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int c = c0 + i, r = r0 + tx;
    if (r < rows && c < cols) {
      int64_t p = c;
      if (mode != 0) p = 2 * static_cast<int64_t>(c) + (mode == 2 ? 1 : 0);
      dd[p * rows + r] = tile[tx][i];
    }
  }
}

void launch_prepare_weights(const __nv_bfloat16* W1, const __nv_bfloat16* W3, const __nv_bfloat16* W2,
                            __nv_bfloat16* W13p, __nv_bfloat16* W2p, int E, int d, int n, cudaStream_t stream) {
  // W1/W3: [d, n] per expert -> rows of W13p (row length d)
  dim3 g13((n + 31) / 32, (d + 31) / 32, E);
  transpose_pack_kernel<<<g13, 256, 0, stream>>>(W1, W13p, d, n, 1, static_cast<int64_t>(2) * n * d);
  transpose_pack_kernel<<<g13, 256, 0, stream>>>(W3, W13p, d, n, 2, static_cast<int64_t>(2) * n * d);
  // W2: [n, d] per expert -> W2p [d, n]
  dim3 g2((d + 31) / 32, (n + 31) / 32, E);
  transpose_pack_kernel<<<g2, 256, 0, stream>>>(W2, W2p, n, d, 0, static_cast<int64_t>(d) * n);
}

// Backward: W13i[e][i][2j] = W1[e][i][j], W13i[e][i][2j + 1] = W3[e][i][j],
// the packed weight's transpose, so that dx = [dg du] W13i^T reads it K-major
// with the same (g, u) column pairing as the pre-activations.
__global__ void __launch_bounds__(256) interleave_w13_kernel(const __nv_bfloat16* __restrict__ W1,
                                                             const __nv_bfloat16* __restrict__ W3,
                                                             __nv_bfloat16* __restrict__ W13i, int64_t pairs) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < pairs;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    __nv_bfloat162 v;
    v.x = W1[i];
    v.y = W3[i];
    reinterpret_cast<__nv_bfloat162*>(W13i)[i] = v;
  }
}

void launch_prepare_weights_bwd(const __nv_bfloat16* W1, const __nv_bfloat16* W3, __nv_bfloat16* W13i, int E, int d,
                                int n, cudaStream_t stream) {
  const int64_t pairs = static_cast<int64_t>(E) * d * n;
  const int blocks = static_cast<int>(std::min<int64_t>((pairs + 255) / 256, static_cast<int64_t>(num_sms()) * 32));
  interleave_w13_kernel<<<blocks, 256, 0, stream>>>(W1, W3, W13i, pairs);
}

}  // namespace moe
