// Backward pass of the MoE layer: the kernels around the four backward GEMMs
// (gemm.cu).  The forward's intermediates are recomputed, not cached
// ("SonicMoE: 加速 MoE 模型的 IO 与 Tile 感知优化", "SonicMoE 的三大核心优化"
// item 1, and section 反向传播优化), and the gate weights' gradient comes from
// the hidden activations and their gradient rather than the expert outputs
// (the "dS 计算优化" row of the 关键 Kernel 对比 table).
//
// Row layout: the forward's expert-grouped rows, each expert's segment padded
// to a multiple of 64 rows with zero rows, so that the weight-gradient GEMMs
// (K = the expert's rows) read whole 64-row k-blocks.  (Token rounding makes
// every count a multiple of the tile, 64, 128 or 256, so its rows need no
// padding.)  A token's rows are a list: k consecutive entries t*k .. t*k+k-1
// without rounding, or entries tok_offsets[t] .. tok_offsets[t+1]-1 of its
// rounded set.  Every reduction here runs in a fixed order: the results are
// bitwise reproducible.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kPadRows = 64;

// offsets_p[e] = sum over e' < e of counts[e'] rounded up to 64 (one block).
__global__ void __launch_bounds__(1024) bwd_pad_offsets_kernel(const int32_t* __restrict__ counts, int E,
                                                               int32_t* __restrict__ offsets_p) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t warp_sum[32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  const int c = e < E ? (counts[e] + kPadRows - 1) / kPadRows * kPadRows : 0;
  int incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = warp_sum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    warp_sum[lane] = v;  // inclusive sums of the warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sum[warp - 1] : 0) + incl - c;
  if (e < E) offsets_p[e] = before;
  if (e == E - 1) offsets_p[E] = before + c;
}

// rowp[a] = padded row of assignment a; wp[rowp[a]] = its gate weight.
// (The top-k path; with rounding the rows and weights come from the round.)
__global__ void bwd_rows_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w,
                                const int32_t* __restrict__ dst, const int32_t* __restrict__ offsets,
                                const int32_t* __restrict__ offsets_p, int64_t A, int32_t* __restrict__ rowp,
                                float* __restrict__ wp) {
  pdl_wait();
  pdl_trigger();
  for (int64_t a = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; a < A;
       a += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int e = idx[a];
    const int rp = dst[a] - offsets[e] + offsets_p[e];
    rowp[a] = rp;
    wp[rp] = w[a];
  }
}

// Zero the padding rows of the operands the weight-gradient GEMMs read.
// Block (e, i): padding row i of expert e, if it exists.
__global__ void __launch_bounds__(256) bwd_zero_pad_kernel(const int32_t* __restrict__ counts,
                                                           const int32_t* __restrict__ offsets_p, int d, int n,
                                                           __nv_bfloat16* xp, __nv_bfloat16* dyp, __nv_bfloat16* dgl,
                                                           __nv_bfloat16* hw) {
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.x;
  const int64_t row = static_cast<int64_t>(offsets_p[e]) + counts[e] + blockIdx.y;
  if (row >= offsets_p[e + 1]) return;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int g = threadIdx.x; g < d / 8; g += blockDim.x) {
    reinterpret_cast<uint4*>(xp + row * d)[g] = z;
    reinterpret_cast<uint4*>(dyp + row * d)[g] = z;
  }
  for (int g = threadIdx.x; g < n / 4; g += blockDim.x) reinterpret_cast<uint4*>(dgl + row * 2 * n)[g] = z;
  for (int g = threadIdx.x; g < n / 8; g += blockDim.x) reinterpret_cast<uint4*>(hw + row * n)[g] = z;
}

// First and end entry of token t's row list.
__device__ __forceinline__ void token_entries(const int32_t* tok_offsets, int t, int k, int64_t& r0, int64_t& r1) {
  if (tok_offsets) {
    r0 = tok_offsets[t];
    r1 = tok_offsets[t + 1];
  } else {
    r0 = static_cast<int64_t>(t) * k;
    r1 = r0 + k;
  }
}

// Gate-weight and logit gradients, a warp per token; lane l takes the
// entries l, l+32, ... of the token's list:
//   dw_i = sum of the row's partials (in partial order)
//   dL_i = w_i (dw_i - sum_j w_j dw_j)   (softmax over the selected logits)
// written per padded row (dlp).  The sum over j is each lane's entries in
// order, then a fixed butterfly over the lanes.
__global__ void __launch_bounds__(256) router_bwd_kernel(const int32_t* __restrict__ rows,
                                                         const int32_t* __restrict__ tok_offsets,
                                                         const float* __restrict__ wp,
                                                         const float* __restrict__ dw_part, int parts, int T, int k,
                                                         float* __restrict__ dlp) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  int64_t r0, r1;
  token_entries(tok_offsets, t, k, r0, r1);
  auto dw_of = [&](int32_t rp) {
    const float* pp = dw_part + static_cast<int64_t>(rp) * parts;
    float v = 0.f;
    for (int i = 0; i < parts; ++i) v += pp[i];
    return v;
  };
  float dot = 0.f;
  for (int64_t i = r0 + lane; i < r1; i += 32) {
    const int32_t rp = rows[i];
    dot += wp[rp] * dw_of(rp);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  for (int64_t i = r0 + lane; i < r1; i += 32) {
    const int32_t rp = rows[i];
    const float wj = wp[rp];
    dlp[rp] = wj * (dw_of(rp) - dot);
  }
}

// WrT[e][i] = Wr[i][e].
__global__ void transpose_router_kernel(const float* __restrict__ Wr, int d, int E, float* __restrict__ WrT) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < static_cast<int64_t>(d) * E;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int e = static_cast<int>(i / d), c = static_cast<int>(i % d);
    WrT[i] = Wr[static_cast<int64_t>(c) * E + e];
  }
}

// dWr[:, e] = sum over expert e's rows of dL_r x_r, db[e] = sum of dL_r.
// Block (e, 256-column chunk, split s): its 8 warps take the rows
// i = 8 s + w, 8 s + w + 8 S, ... of the expert; lanes own 8 columns; the
// warps' sums are added in warp order, the splits' by the final kernel in
// split order.
__global__ void __launch_bounds__(256) dwr_partial_kernel(const __nv_bfloat16* __restrict__ xp,
                                                          const float* __restrict__ dlp,
                                                          const int32_t* __restrict__ counts,
                                                          const int32_t* __restrict__ offsets_p, int E, int d, int S,
                                                          float* __restrict__ part, float* __restrict__ dbpart) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8][256 + 1];
  const int e = blockIdx.x, chunk = blockIdx.y, split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = chunk * 256 + lane * 8;
  const bool col_ok = c0 < d;
  const int64_t first = offsets_p[e];
  const int count = counts[e];
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.f;
  float dsum = 0.f;
  // rows in order, four loads issued before their FMAs (same sums, more
  // bytes in flight)
  const int stride = 8 * S;
  auto add_row = [&](float l, const uint4& v) {
    dsum += l;
    const uint32_t h[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[2 * q] = fmaf(l, bf16_lo(h[q]), acc[2 * q]);
      acc[2 * q + 1] = fmaf(l, bf16_hi(h[q]), acc[2 * q + 1]);
    }
  };
  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
  int i = split * 8 + warp;
  for (; i + 3 * stride < count; i += 4 * stride) {
    float l[4];
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t r = first + i + u * stride;
      l[u] = dlp[r];
      v[u] = col_ok ? __ldg(reinterpret_cast<const uint4*>(xp + r * d + c0)) : zero4;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) add_row(l[u], v[u]);
  }
  for (; i < count; i += stride) {
    const int64_t r = first + i;
    add_row(dlp[r], col_ok ? __ldg(reinterpret_cast<const uint4*>(xp + r * d + c0)) : zero4);
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) red[warp][lane * 8 + q] = acc[q];
  if (lane == 0) red[warp][256] = dsum;
  __syncthreads();
  const int c = threadIdx.x;  // 0..255: one column of the chunk
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) s += red[w][c];
  const int col = chunk * 256 + c;
  if (col < d) part[(static_cast<int64_t>(split) * E + e) * d + col] = s;
  if (chunk == 0 && threadIdx.x == 0) {
    float b = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) b += red[w][256];
    dbpart[static_cast<int64_t>(split) * E + e] = b;
  }
}

__global__ void dwr_final_kernel(const float* __restrict__ part, const float* __restrict__ dbpart, int S, int E,
                                 int d, float* __restrict__ dWr, float* __restrict__ db) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < static_cast<int64_t>(d) * E;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i / E), e = static_cast<int>(i % E);
    float s = 0.f;
    for (int sp = 0; sp < S; ++sp) s += part[(static_cast<int64_t>(sp) * E + e) * d + c];
    dWr[i] = s;
  }
  if (db && blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      float s = 0.f;
      for (int sp = 0; sp < S; ++sp) s += dbpart[static_cast<int64_t>(sp) * E + e];
      db[e] = s;
    }
  }
}

// ----------------------------------------------------------------- host
int bwd_dwr_splits(int E, int d) {
  const int blocks = E * ((d + 255) / 256);
  return std::max(1, std::min(64, (2 * num_sms() + blocks - 1) / blocks));
}

void launch_bwd_pad_offsets(const int32_t* counts, int E, int32_t* offsets_p, cudaStream_t stream) {
  launch_pdl(bwd_pad_offsets_kernel, 1, 1024, 0, stream, 1, counts, E, offsets_p);
}

void launch_bwd_rows(const int32_t* idx, const float* w, const int32_t* dst, const int32_t* offsets,
                     const int32_t* offsets_p, int64_t A, int32_t* rowp, float* wp, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>(std::min<int64_t>((A + 255) / 256, num_sms() * 8));
  launch_pdl(bwd_rows_kernel, blocks, 256, 0, stream, 1, idx, w, dst, offsets, offsets_p, A, rowp, wp);
}

void launch_bwd_zero_pad(const int32_t* counts, const int32_t* offsets_p, int E, int d, int n, __nv_bfloat16* xp,
                         __nv_bfloat16* dyp, __nv_bfloat16* dgl, __nv_bfloat16* hw, cudaStream_t stream) {
  launch_pdl(bwd_zero_pad_kernel, dim3(E, kPadRows - 1), 256, 0, stream, 1, counts, offsets_p, d, n, xp, dyp, dgl, hw);
}

void launch_router_bwd(const int32_t* rows, const int32_t* tok_offsets, const float* wp, const float* dw_part,
                       int parts, int T, int k, float* dlp, cudaStream_t stream) {
  launch_pdl(router_bwd_kernel, (T + 7) / 8, 256, 0, stream, 1, rows, tok_offsets, wp, dw_part, parts, T, k, dlp);
}

void launch_transpose_router(const float* Wr, int d, int E, float* WrT, cudaStream_t stream) {
  const int64_t wt = static_cast<int64_t>(d) * E;
  launch_pdl(transpose_router_kernel, static_cast<unsigned>(std::min<int64_t>((wt + 255) / 256, num_sms() * 8)), 256,
             0, stream, 1, Wr, d, E, WrT);
}

void launch_bwd_dwr(const __nv_bfloat16* xp, const float* dlp, const int32_t* counts, const int32_t* offsets_p,
                    int E, int d, float* part, float* dbpart, float* dWr, float* db, cudaStream_t stream) {
  const int S = bwd_dwr_splits(E, d);
  launch_pdl(dwr_partial_kernel, dim3(E, (d + 255) / 256, S), 256, 0, stream, 1, xp, dlp, counts, offsets_p, E, d, S,
             part, dbpart);
  const int64_t total = static_cast<int64_t>(d) * E;
  launch_pdl(dwr_final_kernel, static_cast<unsigned>(std::min<int64_t>((total + 255) / 256, num_sms() * 8)), 256, 0,
             stream, 1, static_cast<const float*>(part), static_cast<const float*>(dbpart), S, E, d, dWr, db);
}

}  // namespace moe
