// Router: top-k gating over the gate-network logits (the logits themselves
// come from the tensor-core GEMM in gemm.cu), and the whole router for few
// experts (router_small_kernel).
//
// Gate network and top_k of the moe_forward pseudocode
// ("MoE架构的物理瓶颈与扩展限制解析", section 工作原理, step 1) and steps 1-2 of
// the fused MoE kernel ("硬件加速的考量", section 自定义核与核融合).
#include <algorithm>

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

// ---------------------------------------------------------------------------
// Router for few experts (E <= 16).  The gate network does about E flops per
// byte of x there, so it is bound by reading x, and a tensor-core tile of 256
// token rows would leave most SMs idle (T / 256 SM pairs).  This kernel
// streams x on every SM instead.
//  - Wr, laid out once per call by router_small_prep_kernel (fp32, experts
//    interleaved in pairs), reaches shared memory by 1D bulk copies.
//  - Each warp takes TOK tokens at a time and each lane 16-byte chunks of
//    their rows, staged by cp.async through a per-warp ring of
//    kRouterSmallStages steps; a warp's tasks run as one sequence of steps,
//    so the next task's first chunks are in flight while a task finishes.
//  - L[t][e] = sum_i x[t][i] * Wr[i][e] is accumulated in fp32, one fused
//    multiply-add per product in ascending i; a packed fma.rn.f32x2 does the
//    products of experts 2p and 2p+1 together (each half rounded as a scalar
//    fma).  The lanes' partial sums are added by a butterfly over the warp,
//    so every run gives the same bits.
//  - With topk_k > 0 lane j then takes token j's top-k over the 64-bit keys of
//    topk.cuh, the gate weights (softmax over the selected logits, summed in
//    slot order) and the chunk counts of the permutation, as the router GEMM's
//    epilogue does.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void fma_f32x2(uint64_t& acc, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// Position (in floats) of Wr[i][e] in the pair layout: expert pair p = e / 2
// owns 2d floats; element i = 8c + 4h + 2q + r (chunk c, half h) sits in the
// block of (h, q) at chunk c, as the float pair (Wr[i][2p], Wr[i][2p+1]).  A
// lane's 16-byte read at (p, h, q, c) holds elements 2q and 2q+1 of its
// half-chunk for both experts, and lanes with consecutive chunks read
// consecutive words.
__device__ __forceinline__ int router_small_pos(int i, int e, int d) {
  const int c = i >> 3, h = (i >> 2) & 1, q = (i >> 1) & 1, r = i & 1;
  return (e >> 1) * 2 * d + h * d + q * (d >> 1) + 4 * c + 2 * r + (e & 1);
}

// Wr [d][E] to the pair layout Wp (an odd E's last pair gets zero weights);
// also zeroes zero[0, zero_count) (the permutation's chunk counts).
__global__ void __launch_bounds__(256) router_small_prep_kernel(const float* __restrict__ Wr, int d, int E,
                                                                float* __restrict__ Wp, int32_t* __restrict__ zero,
                                                                int64_t zero_count) {
  pdl_wait();
  pdl_trigger();
  const int E2 = (E + 1) & ~1;
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < d; r += gridDim.x * blockDim.x)
    for (int e = 0; e < E2; ++e) Wp[router_small_pos(r, e, d)] = e < E ? Wr[static_cast<int64_t>(r) * E + e] : 0.f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < zero_count;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    zero[i] = 0;
}

template <int EMAX>
__global__ void __launch_bounds__(256, 1)
    router_small_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ Wp,
                        const float* __restrict__ bias, float* __restrict__ logits, int T, int d, int E, int topk_k,
                        int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ chunk_hist,
                        int nchunks, int32_t* status, uint64_t timeout_ns) {
  static_assert(EMAX == 8 || EMAX == 16, "instantiated for E <= 8 and E <= 16");
  constexpr int TOK = 64 / EMAX;  // tokens per warp task: 64 accumulators per lane
  constexpr int NP = EMAX / 2;    // expert pairs
  constexpr int S = kRouterSmallStages;
  constexpr int STAGE = TOK * 32;  // 16-byte chunks per warp and step: [TOK][32 lanes]
  extern __shared__ float4 wt4[];  // the pair layout, then the warps' x rings
  __shared__ alignas(8) uint64_t wbar;
  __shared__ int wabort;
  const int E2 = (E + 1) & ~1;
  const uint32_t wbytes = static_cast<uint32_t>(E2) * d * 4;
  const uint32_t bar = smem_u32(&wbar);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    wabort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, wbytes);
    for (uint32_t off = 0; off < wbytes; off += 32768u)
      bulk_load_1d(smem_u32(wt4) + off, reinterpret_cast<const char*>(Wp) + off, min(32768u, wbytes - off), bar);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int chunks = d / 8;
  const int nit = (chunks + 31) / 32;  // steps of one 16-byte chunk per lane and token
  const int ntask = (T + TOK - 1) / TOK;
  const int np = E2 >> 1;
  uint4* ring = reinterpret_cast<uint4*>(wt4 + wbytes / 16) + warp * S * STAGE;
  const uint32_t ring_s = smem_u32(ring);
  // tasks first + k * stride of this warp (every SM gets work); step n is
  // chunk step n % nit of its task n / nit
  const int first = warp * gridDim.x + blockIdx.x, stride = gridDim.x * nw;
  const int nsteps = first < ntask ? ((ntask - first + stride - 1) / stride) * nit : 0;
  // a lane copies and reads back only its own chunks; chunk c of token j of
  // the task at t0 is x[t0 + j][8c, 8c + 8), zeros past the rows or chunks
  auto issue = [&](int n) {
    if (n < nsteps) {
      const int kk = n / nit, it = n - kk * nit;
      const int t0 = (first + kk * stride) * TOK;
      const int rows = min(TOK, T - t0);
      const uint4* xt = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t0) * d);
      const int c = lane + 32 * it;
      const uint32_t slot = ring_s + static_cast<uint32_t>((n % S) * STAGE + lane) * 16u;
#pragma unroll
      for (int j = 0; j < TOK; ++j) {
        const bool ok = c < chunks && j < rows;
        cp_async_16_zfill(slot + j * 32 * 16, ok ? static_cast<const void*>(xt + j * chunks + c) : x, ok ? 16u : 0u);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int n = 0; n < S - 1; ++n) issue(n);
  if (!mbar_wait_bounded(bar, 0, &wabort, status, kWaitRouterWeights, timeout_ns)) {
    cp_async_wait_all();
    return;
  }
  uint64_t acc2[TOK][NP];  // (L[t0+j][2p], L[t0+j][2p+1]) partial sums
  for (int n = 0; n < nsteps; ++n) {
    issue(n + S - 1);
    cp_async_wait<S - 1>();  // step n has landed
    const int kk = n / nit, it = n - kk * nit;
    if (it == 0) {
#pragma unroll
      for (int j = 0; j < TOK; ++j)
#pragma unroll
        for (int p = 0; p < NP; ++p) acc2[j][p] = 0ull;
    }
    const int c = lane + 32 * it;
    if (c < chunks) {  // else nothing to read (the slot's later rewrite follows no read)
      uint4 xv[TOK];
#pragma unroll
      for (int j = 0; j < TOK; ++j) xv[j] = ring[(n % S) * STAGE + j * 32 + lane];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          // elements 8c + 4h + 2q and + 1 of every token, as fp32 (bf16 bits
          // in the high half of the word)
          float x0[TOK], x1[TOK];
#pragma unroll
          for (int j = 0; j < TOK; ++j) {
            const uint32_t wd = h == 0 ? (q == 0 ? xv[j].x : xv[j].y) : (q == 0 ? xv[j].z : xv[j].w);
            x0[j] = __uint_as_float(wd << 16);
            x1[j] = __uint_as_float(wd & 0xffff0000u);
          }
          float4 w[NP];
#pragma unroll
          for (int p = 0; p < NP; ++p)
            w[p] = p < np ? wt4[(p * 2 * d + h * d + q * (d >> 1)) / 4 + c] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int j = 0; j < TOK; ++j) {
            const uint64_t xx = pack_f32x2(x0[j], x0[j]);
#pragma unroll
            for (int p = 0; p < NP; ++p) fma_f32x2(acc2[j][p], xx, pack_f32x2(w[p].x, w[p].y));
          }
#pragma unroll
          for (int j = 0; j < TOK; ++j) {
            const uint64_t xx = pack_f32x2(x1[j], x1[j]);
#pragma unroll
            for (int p = 0; p < NP; ++p) fma_f32x2(acc2[j][p], xx, pack_f32x2(w[p].z, w[p].w));
          }
        }
      }
    }
    if (it != nit - 1) continue;
    // the task's last step: sum over the lanes, then lane j has token t0 + j
    const int t0 = (first + kk * stride) * TOK;
    float acc[TOK][EMAX];
#pragma unroll
    for (int j = 0; j < TOK; ++j)
#pragma unroll
      for (int p = 0; p < NP; ++p)
        asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[j][2 * p]), "=f"(acc[j][2 * p + 1]) : "l"(acc2[j][p]));
    // butterfly: every lane ends with every total, bit for bit the same
#pragma unroll
    for (int j = 0; j < TOK; ++j)
#pragma unroll
      for (int e = 0; e < EMAX; ++e)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[j][e] += __shfl_xor_sync(0xffffffffu, acc[j][e], off);
    float v[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) v[e] = acc[0][e];
#pragma unroll
    for (int j = 1; j < TOK; ++j)
      if (lane == j)
#pragma unroll
        for (int e = 0; e < EMAX; ++e) v[e] = acc[j][e];
    const int t = t0 + lane;
    if (lane >= TOK || t >= T) continue;
    bool nan_seen = false;
    uint64_t best[kFusedTopk];
#pragma unroll
    for (int i = 0; i < kFusedTopk; ++i) best[i] = 0;  // below every real key
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      if (e >= E) break;
      const float val = bias ? v[e] + bias[e] : v[e];
      logits[static_cast<int64_t>(t) * E + e] = val;
      if (topk_k > 0) {
        nan_seen |= (val != val);
        uint64_t key = topk_key(val, e);
#pragma unroll
        for (int i = 0; i < kFusedTopk; ++i) {  // insert, carrying the smaller key down
          const uint64_t hi = best[i] > key ? best[i] : key;
          key = best[i] > key ? key : best[i];
          best[i] = hi;
        }
      }
    }
    if (topk_k > 0) {
      if (nan_seen) report_error(status, MOE_ERR_DEVICE_CHECK, t);
      const float vmax = topk_key_value(best[0]);
      float ex[kFusedTopk];
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < kFusedTopk; ++j) {
        ex[j] = j < topk_k ? expf(topk_key_value(best[j]) - vmax) : 0.f;
        if (j < topk_k) sum += ex[j];
      }
#pragma unroll
      for (int j = 0; j < kFusedTopk; ++j) {
        if (j < topk_k) {
          const int64_t a = static_cast<int64_t>(t) * topk_k + j;
          const int32_t e = topk_key_expert(best[j]);
          topk_idx[a] = e;
          topk_w[a] = ex[j] / sum;
          atomicAdd(&chunk_hist[static_cast<int64_t>(e) * nchunks + a / kPermChunk], 1);
        }
      }
    }
  }
  cp_async_wait_all();  // the empty groups committed past the last step
}

// Shared memory of router_small_kernel: Wr by expert pairs, then eight warps'
// x rings (kRouterSmallStages steps of 64 / EMAX tokens x 32 lanes x 16 bytes).
static int64_t router_small_smem(int d, int E) {
  const int emax = E <= 8 ? 8 : 16;
  return static_cast<int64_t>((E + 1) & ~1) * d * 4 + 8LL * kRouterSmallStages * (64 / emax) * 32 * 16;
}

bool router_is_small(int d, int E) {
  return E <= 16 && d % 8 == 0 && router_small_smem(d, E) <= kRouterSmallSmemMax;
}

size_t router_small_wp_bytes(int d, int E) { return static_cast<size_t>((E + 1) & ~1) * d * 4; }

void launch_router_small_prep(const float* Wr, int d, int E, float* Wp, int32_t* zero, int64_t zero_count,
                              cudaStream_t stream) {
  const int64_t work = std::max<int64_t>(d, zero_count);
  const int blocks = static_cast<int>(std::min<int64_t>((work + 255) / 256, 4 * num_sms()));
  launch_pdl(router_small_prep_kernel, blocks, 256, 0, stream, 1, Wr, d, E, Wp, zero, zero_count);
}

int launch_router_small(const __nv_bfloat16* x, const float* Wp, const float* bias, float* logits, int T, int d, int E,
                        int k, int32_t* topk_idx, float* topk_w, int32_t* chunk_hist, int32_t* status,
                        uint64_t timeout_ns, cudaStream_t stream) {
  if (!router_is_small(d, E) || reinterpret_cast<uintptr_t>(x) % 16 != 0 || reinterpret_cast<uintptr_t>(Wp) % 16 != 0)
    return MOE_ERR_UNSUPPORTED;
  if (k > 0 && (k > kFusedTopk || !topk_idx || !topk_w || !chunk_hist)) return MOE_ERR_INVALID;
  const size_t smem = static_cast<size_t>(router_small_smem(d, E));
  auto kern = E <= 8 ? router_small_kernel<8> : router_small_kernel<16>;
  // the shared-memory attribute once per device, so later launches (captured
  // ones included) only launch
  static bool ready[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (!ready[dev]) {
    if (cudaFuncSetAttribute(router_small_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kRouterSmallSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(router_small_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kRouterSmallSmemMax) != cudaSuccess)
      return MOE_ERR_CUDA;
    ready[dev] = true;
  }
  const int nchunks = static_cast<int>(perm_num_chunks(static_cast<int64_t>(T) * (k > 0 ? k : 1)));
  if (launch_pdl(kern, num_sms(), 256, smem, stream, 1, static_cast<const __nv_bfloat16*>(x), Wp, bias, logits, T, d,
                 E, k, topk_idx, topk_w, chunk_hist, nchunks, status, timeout_ns) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
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
