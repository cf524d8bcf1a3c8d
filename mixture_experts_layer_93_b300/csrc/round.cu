// Token rounding ("SonicMoE: 加速 MoE 模型的 IO 与 Tile 感知优化", section
// "3. Token Rounding 路由算法"): every expert's token count becomes a multiple
// of the GEMM tile, so no tile of the grouped GEMM is padded.
//
// Reading of the page (its three statements cannot all hold for "always
// round up"): the count c of expert e becomes c' = the nearest multiple of
// the tile, half up (mode NEAREST; or the next multiple up, mode UP), capped at
// tile*floor(T/tile).  If c' > c the c'-c tokens not routed to e with the
// highest logit L[t,e] join e (ties: lower t first); if c' < c the c-c' routed
// tokens with the lowest logits leave (ties: higher t leaves first).  Each
// expert is rounded from the original top-k sets.  A token's final set is
// ordered by (logit desc, expert id asc) and weighted by softmax over it.
//
// Launches (all deterministic; the only atomics are bitwise ORs):
//   member   bitmap of the top-k sets, expert-major [E][ceil(T/32)]
//   select   one block per expert: exact selection of the joining / staying
//            tokens by bisection on the (logit, token) order -> final bitmap
//   count    per-token size of the final set
//   scan     exclusive prefix over tokens -> tok_offsets
//   sets     per token (a warp each): its experts in (logit desc, id asc)
//            order and their softmax weights, written in token order
//   permute  the stable counting sort of moe_permute over that list
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kSelectThreads = 1024;

inline int64_t words_per_row(int T) { return (T + 31) / 32; }
inline int64_t align256(int64_t v) { return (v + 255) & ~int64_t(255); }

struct RoundScratch {
  uint32_t* member;     // [E][W]
  uint32_t* final_set;  // [E][W]
  int32_t* tok_count;   // [T + 1]
  int32_t* tok_expert;  // [cap]
  float* tok_w;         // [cap]
  int32_t* tok_token;   // [cap]
  int32_t* new_counts;  // [E]
  int32_t* chunk_hist;  // [E][nchunks(cap)]
  uint32_t* keys;       // [E][T] when a column does not fit in shared memory
};

constexpr int kSmemKeyLimit = 49152;  // tokens whose keys fit in shared memory

RoundScratch carve(void* base, int T, int E, int64_t cap) {
  const int64_t W = words_per_row(T);
  uint8_t* p = static_cast<uint8_t*>(base);
  RoundScratch s;
  int64_t off = 0;
  s.member = reinterpret_cast<uint32_t*>(p + off);
  off = align256(off + E * W * 4);
  s.final_set = reinterpret_cast<uint32_t*>(p + off);
  off = align256(off + E * W * 4);
  s.tok_count = reinterpret_cast<int32_t*>(p + off);
  off = align256(off + (T + 1) * 4);
  s.tok_expert = reinterpret_cast<int32_t*>(p + off);
  off = align256(off + cap * 4);
  s.tok_w = reinterpret_cast<float*>(p + off);
  off = align256(off + cap * 4);
  s.tok_token = reinterpret_cast<int32_t*>(p + off);
  off = align256(off + cap * 4);
  s.new_counts = reinterpret_cast<int32_t*>(p + off);
  off = align256(off + E * 4);
  s.chunk_hist = reinterpret_cast<int32_t*>(p + off);
  off = align256(off + E * perm_num_chunks(cap) * 4);
  s.keys = reinterpret_cast<uint32_t*>(p + off);
  return s;
}

int64_t scratch_size(int T, int E, int64_t cap) {
  const int64_t W = words_per_row(T);
  return align256(E * W * 4) * 2 + align256((T + 1) * 4) + align256(cap * 4) * 3 + align256(E * 4) +
         align256(E * perm_num_chunks(cap) * 4) + (T > kSmemKeyLimit ? align256(int64_t(E) * T * 4) : 0);
}

// Total order key of a logit: larger float -> larger key; -0.0 and +0.0 equal.
__device__ __forceinline__ uint32_t order_key(float f) {
  if (f == 0.0f) return 0x80000000u;
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void member_bitmap_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int64_t W,
                                     uint32_t* __restrict__ member, int32_t* status) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(T) * k) return;
  const int t = static_cast<int>(i / k);
  const int e = idx[i];
  if (e < 0 || e >= E) {
    report_error(status, MOE_ERR_DEVICE_CHECK, -1);
    return;
  }
  atomicOr(&member[static_cast<int64_t>(e) * W + (t >> 5)], 1u << (t & 31));
}

// Block-wide sum of one int per thread (kSelectThreads threads).
__device__ __forceinline__ int block_sum(int v, int* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  int total = 0;
  if (threadIdx.x < 32) {
    total = (lane < kSelectThreads / 32) ? red[lane] : 0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
    if (lane == 0) red[32] = total;
  }
  __syncthreads();
  return red[32];
}

// Keys of the candidates of one expert (0 for non-candidates; every real key
// is > 0), cached in shared memory or, for long columns, in a global row.
__device__ int count_ge(const uint32_t* keys, int T, uint32_t v, int* red) {
  int c = 0;
  for (int t = threadIdx.x; t < T; t += kSelectThreads) c += keys[t] >= v;
  return block_sum(c, red);
}

__device__ int count_eq_upto(const uint32_t* keys, uint32_t v, int tmax, int* red) {
  int c = 0;
  for (int t = threadIdx.x; t <= tmax; t += kSelectThreads) c += keys[t] == v;
  return block_sum(c, red);
}

// One block per expert.  Among the candidates (members when dropping,
// non-members when adding) finds the m best in the order (L desc, t asc):
// v* = the m-th largest key (bisection on the 32-bit key), then among
// candidates with key == v* the lowest t up to t* (bisection on t).  Writes
// the final membership row and the rounded count.
__global__ void __launch_bounds__(kSelectThreads) round_select_kernel(const float* __restrict__ L, int T, int E,
                                                                      int64_t W, int tile, int mode,
                                                                      const uint32_t* __restrict__ member,
                                                                      uint32_t* __restrict__ final_set,
                                                                      int32_t* __restrict__ new_counts,
                                                                      uint32_t* __restrict__ global_keys,
                                                                      int keys_in_smem) {
  extern __shared__ uint32_t smem_keys[];
  __shared__ int red[33];
  const int e = blockIdx.x;
  const uint32_t* mrow = member + static_cast<int64_t>(e) * W;
  uint32_t* frow = final_set + static_cast<int64_t>(e) * W;
  uint32_t* keys = keys_in_smem ? smem_keys : global_keys + static_cast<int64_t>(e) * T;
  int c = 0;
  for (int64_t w = threadIdx.x; w < W; w += kSelectThreads) c += __popc(mrow[w]);
  c = block_sum(c, red);
  int c2;
  if (mode == MOE_ROUND_NEAREST)
    c2 = tile * ((c + tile / 2) / tile);
  else
    c2 = tile * ((c + tile - 1) / tile);
  c2 = min(c2, tile * (T / tile));

  // adding: choose m = c2 - c among non-members; dropping: keep m = c2 members
  const bool adding = c2 > c;
  const uint32_t want = adding ? 0u : 1u;
  const int m = adding ? (c2 - c) : c2;
  const bool select = (c2 != c) && m > 0;
  uint32_t vstar = 0xFFFFFFFFu;
  int tstar = -1;
  if (select) {
    for (int t = threadIdx.x; t < T; t += kSelectThreads) {
      const uint32_t mbit = (mrow[t >> 5] >> (t & 31)) & 1u;
      keys[t] = (mbit == want) ? order_key(L[static_cast<int64_t>(t) * E + e]) : 0u;
    }
    __syncthreads();
    // largest v with count(key >= v) >= m
    uint32_t lo = 1, hi = 0xFFFFFFFFu;
    while (lo < hi) {
      const uint32_t mid = lo + (hi - lo + 1) / 2;
      if (count_ge(keys, T, mid, red) >= m)
        lo = mid;
      else
        hi = mid - 1;
    }
    vstar = lo;
    const int greater = (vstar == 0xFFFFFFFFu) ? 0 : count_ge(keys, T, vstar + 1, red);
    const int need = m - greater;  // ties at v* to take, lowest t first
    int tlo = 0, thi = T - 1;
    while (tlo < thi) {
      const int mid = (tlo + thi) / 2;
      if (count_eq_upto(keys, vstar, mid, red) >= need)
        thi = mid;
      else
        tlo = mid + 1;
    }
    tstar = tlo;
  }
  for (int64_t w = threadIdx.x; w < W; w += kSelectThreads) {
    const uint32_t mw = mrow[w];
    uint32_t out = mw;
    if (c2 != c) {
      uint32_t chosen = 0;
      if (select) {
        for (int b = 0; b < 32; ++b) {
          const int t = static_cast<int>(w * 32 + b);
          if (t >= T) break;
          const uint32_t key = keys[t];
          if (key != 0u && (key > vstar || (key == vstar && t <= tstar))) chosen |= 1u << b;
        }
      }
      out = adding ? (mw | chosen) : chosen;
    }
    frow[w] = out;
  }
  if (threadIdx.x == 0) new_counts[e] = c2;
}

__global__ void token_count_kernel(const uint32_t* __restrict__ final_set, int T, int E, int64_t W,
                                   int32_t* __restrict__ tok_count) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int c = 0;
  for (int e = 0; e < E; ++e) c += (final_set[static_cast<int64_t>(e) * W + (t >> 5)] >> (t & 31)) & 1u;
  tok_count[t] = c;
}

// Exclusive scan of tok_count[0..T) into tok_offsets[0..T]; one block.
__global__ void __launch_bounds__(1024) token_scan_kernel(const int32_t* __restrict__ tok_count, int T,
                                                          int32_t* __restrict__ tok_offsets) {
  __shared__ int32_t warp_s[32];
  __shared__ int32_t carry_s;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < T; base += 1024) {
    const int t = base + tid;
    const int32_t v = (t < T) ? tok_count[t] : 0;
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
      warp_s[lane] = s;
    }
    __syncthreads();
    const int32_t carry = carry_s;
    const int32_t excl = carry + incl - v + (wid > 0 ? warp_s[wid - 1] : 0);
    if (t < T) tok_offsets[t] = excl;
    __syncthreads();
    if (tid == 1023) carry_s = excl + v;
    __syncthreads();
  }
  if (tid == 0) tok_offsets[T] = carry_s;
}

// One warp per token: its final experts in (logit desc, id asc) order, and
// softmax weights over them (fp32, exp of the logit minus the set's max,
// summed in list order).
__global__ void __launch_bounds__(256) token_sets_kernel(const float* __restrict__ L, const uint32_t* __restrict__ final_set,
                                                         int T, int E, int64_t W,
                                                         const int32_t* __restrict__ tok_offsets,
                                                         int32_t* __restrict__ tok_expert, float* __restrict__ tok_w,
                                                         int32_t* __restrict__ tok_token) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  const int off = tok_offsets[t];
  const int cnt = tok_offsets[t + 1] - off;
  if (cnt == 0) return;
  const float* row = L + static_cast<int64_t>(t) * E;
  float vmax = 0.f, sum = 0.f;
  // rounds of a warp arg-max over the experts still eligible; experts are
  // visited lane + 32*i, eligibility re-read from the bitmap each round
  uint32_t taken = 0;  // bit i: expert lane + 32*i already placed
  for (int j = 0; j < cnt; ++j) {
    float bv = -INFINITY;
    int bid = 0x7fffffff;
    for (int i = 0; 32 * i < E; ++i) {
      const int e = lane + 32 * i;
      if (e >= E) break;
      const bool in = ((final_set[static_cast<int64_t>(e) * W + (t >> 5)] >> (t & 31)) & 1u) &&
                      !((taken >> i) & 1u);
      if (!in) continue;
      float v = row[e];
      if (v != v) v = -INFINITY;
      if (v > bv || (v == bv && e < bid)) {
        bv = v;
        bid = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oid = __shfl_xor_sync(0xffffffffu, bid, o);
      if (ov > bv || (ov == bv && oid < bid)) {
        bv = ov;
        bid = oid;
      }
    }
    if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
    if (j == 0) vmax = bv;
    const float ex = expf(bv - vmax);
    sum += ex;
    if (lane == 0) {
      tok_expert[off + j] = bid;
      tok_w[off + j] = ex;
      tok_token[off + j] = t;
    }
  }
  __syncwarp();
  for (int j = lane; j < cnt; j += 32) tok_w[off + j] = tok_w[off + j] / sum;
}

}  // namespace

size_t round_scratch_bytes(int T, int E, int k, int tile) {
  const int64_t cap = static_cast<int64_t>(T) * k + static_cast<int64_t>(E) * tile;
  return static_cast<size_t>(scratch_size(T, E, cap));
}

void launch_token_round(const float* logits, const int32_t* idx, int T, int E, int k, int tile, int mode,
                        int32_t* counts, int32_t* offsets, int32_t* row_token, float* row_w, int32_t* tok_offsets,
                        int32_t* tok_rows, void* scratch, int32_t* status, cudaStream_t stream) {
  const int64_t cap = static_cast<int64_t>(T) * k + static_cast<int64_t>(E) * tile;
  const int64_t W = words_per_row(T);
  RoundScratch s = carve(scratch, T, E, cap);
  cudaMemsetAsync(s.member, 0, static_cast<size_t>(E * W * 4), stream);
  const int64_t A = static_cast<int64_t>(T) * k;
  member_bitmap_kernel<<<static_cast<int>((A + 255) / 256), 256, 0, stream>>>(idx, T, k, E, W, s.member, status);
  const int in_smem = T <= kSmemKeyLimit ? 1 : 0;
  const size_t key_smem = in_smem ? static_cast<size_t>(T) * 4 : 0;
  cudaFuncSetAttribute(round_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(kSmemKeyLimit) * 4);
  round_select_kernel<<<E, kSelectThreads, key_smem, stream>>>(logits, T, E, W, tile, mode, s.member, s.final_set,
                                                              s.new_counts, s.keys, in_smem);
  token_count_kernel<<<(T + 255) / 256, 256, 0, stream>>>(s.final_set, T, E, W, s.tok_count);
  token_scan_kernel<<<1, 1024, 0, stream>>>(s.tok_count, T, tok_offsets);
  token_sets_kernel<<<(T + 7) / 8, 256, 0, stream>>>(logits, s.final_set, T, E, W, tok_offsets, s.tok_expert,
                                                     s.tok_w, s.tok_token);
  // stable grouping by expert of the token-ordered list: rows of an expert
  // come out in ascending t; tok_rows is the list's row map (moe_permute's dst)
  launch_permute_list(s.tok_expert, s.tok_w, s.tok_token, tok_offsets + T, cap, E, s.chunk_hist, counts, offsets,
                      tok_rows, row_token, row_w, status, stream);
}

}  // namespace moe
