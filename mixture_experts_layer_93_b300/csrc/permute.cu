// Permutation: a stable counting sort of the T*k assignments a = t*k + j by
// expert id, so each expert's rows are contiguous for the grouped GEMM (the
// "contiguous packed input" mode of "SonicMoE: 加速 MoE 模型的 IO 与 Tile 感知优化",
// section "Gather 与加载融合").
//
// Three launches, none of which lets an atomic decide an order:
//   hist    per-chunk expert histograms (a warp per chunk of 2048 assignments)
//   scan    per-expert exclusive prefix over chunks, then over experts
//   scatter each warp walks its chunk in order, 32 assignments at a time;
//           equal experts within a step are ranked by lane (match.any), so
//           rows of an expert come out in ascending a, i.e. ascending t.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"


namespace moe {

// A block of kPermWarps warps owns kPermChunk consecutive assignments; warp w
// owns the sub-chunk [w*kSub, (w+1)*kSub) of it.
constexpr int kPermWarps = 8;
constexpr int kSub = kPermChunk / kPermWarps;  // 256 assignments per warp
constexpr int kPerLane = kSub / 32;            // 8 per lane
static_assert(kPermChunk % (kPermWarps * 32) == 0, "chunk layout");

// A list's length is A, or min(A, *len) when the length lives on the device.
__device__ __forceinline__ int64_t list_length(int64_t A, const int32_t* len) {
  return len ? min(A, static_cast<int64_t>(*len)) : A;
}

// Per-block expert histogram -> chunk_hist[e][block].
__global__ void __launch_bounds__(kPermWarps * 32) perm_hist_kernel(const int32_t* __restrict__ idx, int64_t A,
                                                                  const int32_t* __restrict__ len, int E,
                                                                  int nchunks, int32_t* __restrict__ chunk_hist,
                                                                  int32_t* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int32_t hist_s[];
  const int c = blockIdx.x;
  A = list_length(A, len);
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist_s[e] = 0;
  __syncthreads();
  const int64_t a0 = static_cast<int64_t>(c) * kPermChunk;
  bool bad = false;
  int ev[kPermChunk / (kPermWarps * 32)];
#pragma unroll
  for (int i = 0; i < kPermChunk / (kPermWarps * 32); ++i) {
    const int64_t a = a0 + threadIdx.x + static_cast<int64_t>(i) * blockDim.x;
    ev[i] = (a < A) ? idx[a] : -1;
  }
#pragma unroll
  for (int i = 0; i < kPermChunk / (kPermWarps * 32); ++i) {
    const int64_t a = a0 + threadIdx.x + static_cast<int64_t>(i) * blockDim.x;
    if (a >= A) continue;
    if (ev[i] >= 0 && ev[i] < E)
      atomicAdd(&hist_s[ev[i]], 1);  // counts only: the order of increments does not matter
    else
      bad = true;
  }
  if (bad) report_error(status, MOE_ERR_DEVICE_CHECK, -1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_hist[static_cast<int64_t>(e) * nchunks + c] = hist_s[e];
}

// Run by one block of 1024 threads: warp w scans the chunk counts of experts
// w, w+32, ... (up to 256 chunks per pass, all loads issued first; warp
// shuffles), then the expert totals are scanned and added back as each
// expert's base.  chunk_hist[e][c] becomes the first row of expert e's rows
// from chunk c; counts and offsets are written.  cnt_s: 1024 ints, warp_s: 32
// ints of shared memory.
__device__ void scan_chunk_hist(int32_t* __restrict__ chunk_hist, int E, int nchunks, int32_t* __restrict__ counts,
                                int32_t* __restrict__ offsets, int32_t* cnt_s, int32_t* warp_s) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int e = tid; e < 1024; e += blockDim.x) cnt_s[e] = 0;
  __syncthreads();
  for (int e = wid; e < E; e += 32) {
    int32_t* hrow = chunk_hist + static_cast<int64_t>(e) * nchunks;
    int32_t run = 0;
    // 256 chunk counts per pass, all loads issued before the first scan
    for (int c0 = 0; c0 < nchunks; c0 += 8 * 32) {
      int32_t v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + 32 * i + lane;
        v[i] = (c < nchunks) ? hrow[c] : 0;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (c0 + 32 * i >= nchunks) break;  // warp-uniform
        const int c = c0 + 32 * i + lane;
        int32_t incl = v[i];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += o;
        }
        if (c < nchunks) hrow[c] = run + incl - v[i];
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    if (lane == 0) cnt_s[e] = run;
  }
  __syncthreads();
  // exclusive scan of cnt_s[0..1024) (E <= 1024): one value per thread
  const int32_t v = cnt_s[tid];
  int32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_s[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int32_t s = warp_s[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += o;
    }
    warp_s[lane] = s;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const int32_t excl = incl - v + (wid > 0 ? warp_s[wid - 1] : 0);
  __syncthreads();
  cnt_s[tid] = excl;
  if (tid < E) {
    counts[tid] = v;
    offsets[tid] = excl;
  }
  if (tid == E - 1) offsets[E] = excl + v;
  __syncthreads();
  for (int e = wid; e < E; e += 32) {
    int32_t* hrow = chunk_hist + static_cast<int64_t>(e) * nchunks;
    const int32_t base = cnt_s[e];
    for (int c = lane; c < nchunks; c += 32) hrow[c] += base;
  }
}

__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ chunk_hist, int E, int nchunks,
                                                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t cnt_s[1024];
  __shared__ int32_t warp_s[32];
  scan_chunk_hist(chunk_hist, E, nchunks, counts, offsets, cnt_s, warp_s);
}

// ---------------------------------------------------------------------------
// Fused top-k + chunk histogram (E <= 256): a warp per token runs the top-k
// (topk.cuh: the same code as the top-k kernel, so the same bits), writes the
// indices and weights, and adds each assignment a = t*k + j to the count of
// its expert in chunk a / kPermChunk with an integer atomic (counts only: the
// order of increments does not matter).  The counts are zero on entry: the
// split-weight kernel that precedes this one zeroes them.
template <int NV>
__global__ void __launch_bounds__(256) topk_perm_hist_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                             int32_t* __restrict__ topk_idx,
                                                             float* __restrict__ topk_w, int nchunks,
                                                             int32_t* __restrict__ chunk_hist, int32_t* status) {
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
    const int64_t a = static_cast<int64_t>(t) * k + lane;
    const int32_t e = topk_key_expert(mine);
    topk_idx[a] = e;
    topk_w[a] = w;
    atomicAdd(&chunk_hist[static_cast<int64_t>(e) * nchunks + a / kPermChunk], 1);
  }
}

// token_of == nullptr: the token of assignment a is a / k.  src may be null.
// Warp w of block c places its 256 assignments, in order, after (a) every
// earlier block's rows of the same expert (chunk_base, from the scan) and (b)
// the rows of warps < w of this block; within 32 consecutive assignments,
// equal experts are ranked by lane (match.any).  So rows of an expert come out
// in ascending assignment order.
__global__ void __launch_bounds__(kPermWarps * 32) perm_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ wts, const int32_t* __restrict__ token_of, int64_t A,
    const int32_t* __restrict__ len, int k, int E, int nchunks, const int32_t* __restrict__ chunk_base,
    int32_t* __restrict__ src, int32_t* __restrict__ dst, int32_t* __restrict__ row_token,
    float* __restrict__ row_w) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int32_t wbase[];  // [kPermWarps][E]
  const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = blockIdx.x;
  A = list_length(A, len);
  for (int i = threadIdx.x; i < kPermWarps * E; i += blockDim.x) wbase[i] = 0;
  __syncthreads();
  const int64_t a0 = static_cast<int64_t>(c) * kPermChunk + static_cast<int64_t>(w) * kSub;
  int ev[kPerLane];
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int64_t a = a0 + lane + 32 * i;
    int e = (a < A) ? idx[a] : -1;
    if (e >= E) e = -1;
    ev[i] = e;
  }
  int32_t* mybase = wbase + w * E;
#pragma unroll
  for (int i = 0; i < kPerLane; ++i)
    if (ev[i] >= 0) atomicAdd(&mybase[ev[i]], 1);  // per-warp counts
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = chunk_base[static_cast<int64_t>(e) * nchunks + c];
    for (int ww = 0; ww < kPermWarps; ++ww) {
      const int32_t cnt = wbase[ww * E + e];
      wbase[ww * E + e] = run;
      run += cnt;
    }
  }
  __syncthreads();
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int64_t a = a0 + lane + 32 * i;
    const int e = ev[i];
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    int pos = 0;
    if (e >= 0) pos = mybase[e] + rank;
    __syncwarp();
    if (e >= 0 && rank == 0) mybase[e] += __popc(peers);
    __syncwarp();
    if (e >= 0) {
      if (src) src[pos] = static_cast<int32_t>(a);
      dst[a] = pos;
      row_token[pos] = token_of ? token_of[a] : static_cast<int32_t>(a / k);
      if (wts) row_w[pos] = wts[a];
    }
  }
}

static void permute_impl(const int32_t* idx, const float* w, const int32_t* token_of, int64_t A, const int32_t* len,
                         int k, int E, int32_t* chunk_hist, int32_t* counts, int32_t* offsets, int32_t* src,
                         int32_t* dst, int32_t* row_token, float* row_w, int32_t* status, cudaStream_t stream) {
  const int nchunks = static_cast<int>(perm_num_chunks(A));
  launch_pdl(perm_hist_kernel, nchunks, kPermWarps * 32, static_cast<size_t>(E) * sizeof(int32_t), stream, 1, 
      idx, A, len, E, nchunks, chunk_hist, status);
  launch_pdl(perm_scan_kernel, 1, 1024, 0, stream, 1, chunk_hist, E, nchunks, counts, offsets);
  launch_pdl(perm_scatter_kernel, nchunks, kPermWarps * 32, static_cast<size_t>(kPermWarps) * E * sizeof(int32_t), stream, 1, 
      idx, w, token_of, A, len, k, E, nchunks, chunk_hist, src, dst, row_token, row_w);
}

void launch_permute(const int32_t* idx, const float* w, int64_t A, int k, int E, int32_t* chunk_hist,
                    int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dst, int32_t* row_token,
                    float* row_w, int32_t* status, cudaStream_t stream) {
  permute_impl(idx, w, nullptr, A, nullptr, k, E, chunk_hist, counts, offsets, src, dst, row_token, row_w, status,
               stream);
}

// Top-k gating and the permutation of its assignments.  E <= 256: the fused
// top-k + histogram kernel (chunk_hist zeroed beforehand, by
// launch_split_router or launch_router_small_prep), the scan and the scatter
// (three launches instead of four); larger E: the top-k kernel and the three
// permutation launches.
void launch_topk_permute(const float* logits, int T, int E, int k, int32_t* idx, float* w, int32_t* chunk_hist,
                         int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dst, int32_t* row_token,
                         float* row_w, int32_t* status, cudaStream_t stream) {
  const int64_t A = static_cast<int64_t>(T) * k;
  const int nchunks = static_cast<int>(perm_num_chunks(A));
  const int nv = (E + 31) / 32;
  if (nv > 8) {
    launch_topk_gating(logits, idx, w, T, E, k, status, stream);
    launch_permute(idx, w, A, k, E, chunk_hist, counts, offsets, src, dst, row_token, row_w, status, stream);
    return;
  }
  auto kern = nv <= 1 ? topk_perm_hist_kernel<1>
            : nv <= 2 ? topk_perm_hist_kernel<2>
            : nv <= 4 ? topk_perm_hist_kernel<4>
                      : topk_perm_hist_kernel<8>;
  launch_pdl(kern, (T + 7) / 8, 256, 0, stream, 1, logits, T, E, k, idx, w, nchunks, chunk_hist, status);
  launch_perm_scan_scatter(idx, w, A, k, E, chunk_hist, counts, offsets, src, dst, row_token, row_w, stream);
}

void launch_perm_scan_scatter(const int32_t* idx, const float* w, int64_t A, int k, int E, int32_t* chunk_hist,
                              int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dst, int32_t* row_token,
                              float* row_w, cudaStream_t stream) {
  const int nchunks = static_cast<int>(perm_num_chunks(A));
  launch_pdl(perm_scan_kernel, 1, 1024, 0, stream, 1, chunk_hist, E, nchunks, counts, offsets);
  launch_pdl(perm_scatter_kernel, nchunks, kPermWarps * 32, static_cast<size_t>(kPermWarps) * E * sizeof(int32_t),
             stream, 1, static_cast<const int32_t*>(idx), static_cast<const float*>(w),
             static_cast<const int32_t*>(nullptr), A, static_cast<const int32_t*>(nullptr), k, E, nchunks,
             static_cast<const int32_t*>(chunk_hist), src, dst, row_token, row_w);
}

void launch_permute_list(const int32_t* expert_of, const float* w, const int32_t* token_of, const int32_t* len,
                         int64_t cap, int E, int32_t* chunk_hist, int32_t* counts, int32_t* offsets, int32_t* dst,
                         int32_t* row_token, float* row_w, int32_t* status, cudaStream_t stream) {
  permute_impl(expert_of, w, token_of, cap, len, 1, E, chunk_hist, counts, offsets, nullptr, dst, row_token, row_w,
               status, stream);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free variant of the permutation.
//
// Its chunk histograms live in a file-scope device array instead of a
// caller-provided workspace.  The host cannot pass that array's name to a
// kernel (in host code it is only a stand-in symbol), so its device address is
// looked up with cudaGetSymbolAddress.  The address belongs to the CUDA context
// that is current when it is looked up (each context loads its own copy of the
// module), so it is looked up again on every call rather than cached: a
// caller that runs in its own driver-API context, or calls again after
// cudaDeviceReset, gets the address that is valid in its context.  The lookup
// allocates nothing.
namespace moe {

constexpr int64_t kNoAllocScratchInts = 262144;  // 1 MiB
static __device__ __align__(256) int32_t g_perm_scratch[kNoAllocScratchInts];

// Device address of g_perm_scratch in the current context; nullptr if the
// lookup fails.
static int32_t* noalloc_scratch() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_perm_scratch) != cudaSuccess) return nullptr;
  return static_cast<int32_t*>(ptr);
}

}  // namespace moe

extern "C" int moe_permute_noalloc(const moe_shape* s, const int32_t* topk_idx, const float* topk_w, int32_t* counts,
                                   int32_t* offsets, int32_t* src, int32_t* dst, int32_t* row_token, float* row_w,
                                   void* stream) {
  using namespace moe;
  if (!s || s->T < 1 || s->E < 1 || s->E > 1024 || s->k < 1 || s->k > s->E || s->k > 32) return MOE_ERR_INVALID;
  if (!topk_idx || !counts || !offsets || !src || !dst || !row_token) return MOE_ERR_INVALID;
  if (topk_w && !row_w) return MOE_ERR_INVALID;
  const int64_t A = static_cast<int64_t>(s->T) * s->k;
  if (A >= (int64_t(1) << 31) - 1) return MOE_ERR_INVALID;
  // the histograms need E * ceil(A / 2048) ints of the fixed array
  if (static_cast<int64_t>(s->E) * perm_num_chunks(A) > kNoAllocScratchInts) return MOE_ERR_WORKSPACE;
  int32_t* scratch = noalloc_scratch();
  if (!scratch) return MOE_ERR_CUDA;
  // every histogram entry the scan reads is written by this call's first
  // kernel, so nothing left over from an earlier call is ever read
  launch_permute(topk_idx, topk_w, A, s->k, s->E, scratch, counts, offsets, src, dst, row_token, row_w, nullptr,
                 reinterpret_cast<cudaStream_t>(stream));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
