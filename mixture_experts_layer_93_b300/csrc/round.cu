// Token rounding ("SonicMoE: 加速 MoE 模型的 IO 与 Tile 感知优化", section
// "3. Token Rounding 路由算法"): every expert's token count becomes a multiple
// of the GEMM tile, so no tile of the grouped GEMM is padded.
//
// Reading of the page (its three statements cannot all hold for "always
// round up"): the count c of expert e becomes c' = the nearest multiple of
// the tile, half up (mode NEAREST; the next multiple up, mode UP; or, mode
// STOCHASTIC, up with probability (c mod tile)/tile so that the expected
// count is exactly c), capped at tile*floor(T/tile).  If c' > c the c'-c tokens not routed to e with the
// highest logit L[t,e] join e (ties: lower t first); if c' < c the c-c' routed
// tokens with the lowest logits leave (ties: higher t leaves first).  Each
// expert is rounded from the original top-k sets.  A token's final set is
// ordered by (logit desc, expert id asc) and weighted by softmax over it.
//
// Launches (all deterministic; the only atomics are bitwise ORs):
//   member   bitmap of the top-k sets, expert-major [E][ceil(T/32)]
//   select   one block per expert: exact selection of the joining / staying
//            tokens by radix select on the (logit, token) order -> final bitmap
//   transpose  the final bitmap to token-major words (warp ballots)
//   offsets  per-token set sizes and their exclusive prefix -> tok_offsets
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
  uint32_t* tok_bits;   // [T][EW] token-major final membership
  int32_t* tok_expert;  // [cap]
  float* tok_w;         // [cap]
  int32_t* tok_token;   // [cap]
  int32_t* new_counts;  // [E]
  int32_t* chunk_hist;  // [E][nchunks(cap)]
  uint32_t* keys;       // [E][T] when a column does not fit in shared memory
  int32_t* block_sums;  // [ceil(T/1024)]
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
  s.tok_bits = reinterpret_cast<uint32_t*>(p + off);
  off = align256(off + static_cast<int64_t>(T) * ((E + 31) / 32) * 4);
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
  s.block_sums = reinterpret_cast<int32_t*>(p + off);
  off = align256(off + ((T + 1023) / 1024) * 4);
  s.keys = reinterpret_cast<uint32_t*>(p + off);
  return s;
}

int64_t scratch_size(int T, int E, int64_t cap) {
  const int64_t W = words_per_row(T);
  return align256(E * W * 4) * 2 + align256(static_cast<int64_t>(T) * ((E + 31) / 32) * 4) + align256(cap * 4) * 3 +
         align256(E * 4) +
         align256(E * perm_num_chunks(cap) * 4) + align256(((T + 1023) / 1024) * 4) +
         (T > kSmemKeyLimit ? align256(int64_t(E) * T * 4) : 0);
}

// SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014): add the golden-ratio increment to the state, then
// two xor-shift-multiply rounds and a final xor-shift.
__device__ __forceinline__ uint64_t splitmix64(uint64_t state) {
  uint64_t z = state + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Total order key of a logit: larger float -> larger key; -0.0 and +0.0 equal.
__device__ __forceinline__ uint32_t order_key(float f) {
  if (f == 0.0f) return 0x80000000u;
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void member_bitmap_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int64_t W,
                                     uint32_t* __restrict__ member, int32_t* status) {
  pdl_wait();
  pdl_trigger();
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

// One block per expert.  Among the candidates (members when dropping,
// non-members when adding) keeps the m best in the order (L desc, t asc):
// a 4-pass radix select (8 bits a pass, from the top) finds v* = the m-th
// largest 32-bit key and how many keys equal to v* to take; one ordered pass
// over t then finds t*, the last tie taken (lowest t first).  Keys of
// non-candidates are 0 (every real key is > 0).  Writes the final membership
// row and the rounded count.
__global__ void __launch_bounds__(kSelectThreads) round_select_kernel(const float* __restrict__ L, int T, int E,
                                                                      int64_t W, int tile, int mode, uint32_t seed,
                                                                      const uint32_t* __restrict__ member,
                                                                      uint32_t* __restrict__ final_set,
                                                                      int32_t* __restrict__ new_counts,
                                                                      uint32_t* __restrict__ global_keys,
                                                                      int keys_in_smem) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t smem_keys[];
  __shared__ int red[33];
  __shared__ int hist[256];
  __shared__ int sel[2];  // chosen digit, remaining rank
  __shared__ int tstar_s;
  const int e = blockIdx.x;
  const uint32_t* mrow = member + static_cast<int64_t>(e) * W;
  uint32_t* frow = final_set + static_cast<int64_t>(e) * W;
  uint32_t* keys = keys_in_smem ? smem_keys : global_keys + static_cast<int64_t>(e) * T;
  int c = 0;
  for (int64_t w = threadIdx.x; w < W; w += kSelectThreads) c += __popc(mrow[w]);
  c = block_sum(c, red);
  int c2;
  if (mode == MOE_ROUND_NEAREST) {
    c2 = tile * ((c + tile / 2) / tile);
  } else if (mode == MOE_ROUND_STOCHASTIC) {
    // up with probability (c mod tile) / tile: exact integer comparison of the
    // draw's top 32 bits against (c mod tile) * 2^32 / tile
    const uint64_t h = splitmix64((static_cast<uint64_t>(seed) << 32) | static_cast<uint32_t>(e)) >> 32;
    const bool up = h * static_cast<uint64_t>(tile) < (static_cast<uint64_t>(c % tile) << 32);
    c2 = tile * (c / tile) + (up ? tile : 0);
  } else {
    c2 = tile * ((c + tile - 1) / tile);
  }
  c2 = min(c2, tile * (T / tile));

  // adding: choose m = c2 - c among non-members; dropping: keep m = c2 members
  const bool adding = c2 > c;
  const uint32_t want = adding ? 0u : 1u;
  const int m = adding ? (c2 - c) : c2;
  const bool select = (c2 != c) && m > 0;
  uint32_t vstar = 0xFFFFFFFFu;
  int tstar = -1;
  if (select) {
    // the column L[:, e] is strided in memory: issue 8 loads before using any
    for (int tb = 0; tb < T; tb += 8 * kSelectThreads) {
      float lv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int t = tb + j * kSelectThreads + threadIdx.x;
        lv[j] = (t < T) ? L[static_cast<int64_t>(t) * E + e] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int t = tb + j * kSelectThreads + threadIdx.x;
        if (t < T) {
          const uint32_t mbit = (mrow[t >> 5] >> (t & 31)) & 1u;
          keys[t] = (mbit == want) ? order_key(lv[j]) : 0u;
        }
      }
    }
    uint32_t prefix = 0, pmask = 0;
    int rem = m;  // rank still to find among keys matching the prefix
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kSelectThreads) hist[i] = 0;
      __syncthreads();
      // counts only: the order of the additions does not matter
      for (int t = threadIdx.x; t < T; t += kSelectThreads) {
        const uint32_t kk = keys[t];
        if (kk != 0u && (kk & pmask) == prefix) atomicAdd(&hist[(kk >> shift) & 255u], 1);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // lane l owns digits 255-8l .. 248-8l (descending)
        const int lane = threadIdx.x;
        int mine = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) mine += hist[255 - 8 * lane - j];
        int incl = mine;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int o = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += o;
        }
        const int before = incl - mine;
        if (before < rem && rem <= incl) {
          int cum = before;
          for (int j = 0; j < 8; ++j) {
            const int dgt = 255 - 8 * lane - j;
            if (cum + hist[dgt] >= rem) {
              sel[0] = dgt;
              sel[1] = rem - cum;
              break;
            }
            cum += hist[dgt];
          }
        }
      }
      __syncthreads();
      prefix |= static_cast<uint32_t>(sel[0]) << shift;
      pmask |= 255u << shift;
      rem = sel[1];
      __syncthreads();
    }
    vstar = prefix;
    // the rem lowest-t keys equal to v* are taken.  Warp w owns the t range
    // [w*R, (w+1)*R) and reads it 32 at a time (coalesced); ballots keep t
    // order; a scan over the warp totals finds the warp holding the rem-th tie.
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    constexpr int kWarps = kSelectThreads / 32;
    const int R = (T + kWarps - 1) / kWarps;
    const int tb = wid * R, te = min(T, tb + R);
    int cnt = 0;
    for (int base = tb; base < te; base += 32) {
      const int t = base + lane;
      cnt += __popc(__ballot_sync(0xffffffffu, t < te && keys[t] == vstar));
    }
    if (threadIdx.x == 0) tstar_s = -1;
    __syncthreads();
    if (lane == 0) red[wid] = cnt;
    __syncthreads();
    int wbefore = 0;
    for (int i = 0; i < wid; ++i) wbefore += red[i];
    if (wbefore < rem && rem <= wbefore + cnt) {
      int running = wbefore;
      for (int base = tb; base < te; base += 32) {
        const int t = base + lane;
        const uint32_t bal = __ballot_sync(0xffffffffu, t < te && keys[t] == vstar);
        const int nb = __popc(bal);
        if (running + nb >= rem) {
          // the (rem - running)-th set bit of bal, counted from bit 0
          int need = rem - running, pos = -1;
          for (int bit = 0; bit < 32; ++bit) {
            if ((bal >> bit) & 1u) {
              if (--need == 0) {
                pos = bit;
                break;
              }
            }
          }
          if (lane == 0) tstar_s = base + pos;
          break;
        }
        running += nb;
      }
    }
    __syncthreads();
    tstar = tstar_s;
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

// Expert-major membership bits [E][W] -> token-major [T][EW] (EW = E/32
// rounded up): one warp per 32 experts x 32 tokens block; lane i holds expert
// 32*eb+i's word, and a ballot over lanes of bit j is token j's 32 experts.
__global__ void bits_transpose_kernel(const uint32_t* __restrict__ final_set, int T, int E, int64_t W, int EW,
                                      uint32_t* __restrict__ tok_bits) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t wg = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nblk = static_cast<int64_t>(EW) * W;
  if (wg >= nblk) return;
  const int eb = static_cast<int>(wg / W);
  const int64_t tw = wg % W;
  const int e = eb * 32 + lane;
  const uint32_t word = (e < E) ? final_set[static_cast<int64_t>(e) * W + tw] : 0u;
  uint32_t mine = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint32_t col = __ballot_sync(0xffffffffu, (word >> j) & 1u);
    if (lane == j) mine = col;
  }
  const int64_t t = tw * 32 + lane;
  if (t < T) tok_bits[t * EW + eb] = mine;
}

// Per-token set sizes and their exclusive prefix, in two launches: block b
// scans the sizes of tokens [1024b, 1024b+1024) (coalesced, warp shuffles)
// into tok_offsets and its total into block_sums[b]; then every block adds
// the sum of the earlier blocks' totals.
__global__ void __launch_bounds__(1024) token_offsets_local_kernel(const uint32_t* __restrict__ tok_bits, int T,
                                                                   int EW, int32_t* __restrict__ tok_offsets,
                                                                   int32_t* __restrict__ block_sums) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t warp_s[32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int t = blockIdx.x * 1024 + tid;
  int32_t v = 0;
  if (t < T)
    for (int w = 0; w < EW; ++w) v += __popc(tok_bits[static_cast<int64_t>(t) * EW + w]);
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
  const int32_t excl = incl - v + (wid > 0 ? warp_s[wid - 1] : 0);
  if (t < T) tok_offsets[t] = excl;
  if (tid == 1023) block_sums[blockIdx.x] = excl + v;
}

__global__ void __launch_bounds__(1024) token_offsets_add_kernel(int T, int32_t* __restrict__ tok_offsets,
                                                                 const int32_t* __restrict__ block_sums) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t base_s;
  const int tid = threadIdx.x;
  if (tid < 32) {
    int32_t s = 0;
    for (int i = tid; i < static_cast<int>(blockIdx.x); i += 32) s += block_sums[i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (tid == 0) base_s = s;
  }
  __syncthreads();
  const int t = blockIdx.x * 1024 + tid;
  if (t < T) tok_offsets[t] += base_s;
  if (t == T - 1) tok_offsets[T] = base_s + block_sums[blockIdx.x];
}

// One warp per token: its final experts in (logit desc, id asc) order and
// softmax weights over them (fp32, exp of the logit minus the set's max,
// summed in list order).  Lane l holds experts l, l+32, ... (membership bit
// and logit in registers), as in the top-k kernel.
template <int NV>
__global__ void __launch_bounds__(256) token_sets_kernel(const float* __restrict__ L,
                                                         const uint32_t* __restrict__ tok_bits, int T, int E, int EW,
                                                         const int32_t* __restrict__ tok_offsets,
                                                         int32_t* __restrict__ tok_expert, float* __restrict__ tok_w,
                                                         int32_t* __restrict__ tok_token) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  const int off = tok_offsets[t];
  const int cnt = tok_offsets[t + 1] - off;
  if (cnt == 0) return;
  const float* row = L + static_cast<int64_t>(t) * E;
  const uint32_t* bits = tok_bits + static_cast<int64_t>(t) * EW;
  float v[NV];
  uint32_t eligible = 0;  // bit i: expert lane + 32*i is in the final set
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    v[i] = -INFINITY;
    if (e < E && i < EW && ((bits[i] >> lane) & 1u)) {
      eligible |= 1u << i;
      const float x = row[e];
      v[i] = (x != x) ? -INFINITY : x;
    }
  }
  float vmax = 0.f, sum = 0.f;
  for (int j = 0; j < cnt; ++j) {
    float bv = -INFINITY;
    int bid = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      if (((eligible >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bid))) {
        bv = v[i];
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
    if ((bid & 31) == lane) eligible &= ~(1u << (bid >> 5));
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

void launch_token_sets(const float* L, const uint32_t* tok_bits, int T, int E, int EW, const int32_t* tok_offsets,
                       int32_t* tok_expert, float* tok_w, int32_t* tok_token, cudaStream_t stream) {
  const int blocks = (T + 7) / 8;
#define MOE_SETS(NV) \
  launch_pdl(token_sets_kernel<NV>, blocks, 256, 0, stream, 1, L, tok_bits, T, E, EW, tok_offsets, tok_expert, tok_w, tok_token)
  if (EW <= 1)
    MOE_SETS(1);
  else if (EW <= 2)
    MOE_SETS(2);
  else if (EW <= 4)
    MOE_SETS(4);
  else if (EW <= 8)
    MOE_SETS(8);
  else if (EW <= 16)
    MOE_SETS(16);
  else
    MOE_SETS(32);
#undef MOE_SETS
}

}  // namespace

size_t round_scratch_bytes(int T, int E, int k, int tile) {
  const int64_t cap = static_cast<int64_t>(T) * k + static_cast<int64_t>(E) * tile;
  return static_cast<size_t>(scratch_size(T, E, cap));
}

void launch_token_round(const float* logits, const int32_t* idx, int T, int E, int k, int tile, int mode,
                        uint32_t seed, int32_t* counts, int32_t* offsets, int32_t* row_token, float* row_w, int32_t* tok_offsets,
                        int32_t* tok_rows, void* scratch, int32_t* status, cudaStream_t stream) {
  const int64_t cap = static_cast<int64_t>(T) * k + static_cast<int64_t>(E) * tile;
  const int64_t W = words_per_row(T);
  RoundScratch s = carve(scratch, T, E, cap);
  cudaMemsetAsync(s.member, 0, static_cast<size_t>(E * W * 4), stream);
  const int64_t A = static_cast<int64_t>(T) * k;
  launch_pdl(member_bitmap_kernel, static_cast<int>((A + 255) / 256), 256, 0, stream, 1, idx, T, k, E, W, s.member, status);
  const int in_smem = T <= kSmemKeyLimit ? 1 : 0;
  const size_t key_smem = in_smem ? static_cast<size_t>(T) * 4 : 0;
  cudaFuncSetAttribute(round_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(kSmemKeyLimit) * 4);
  launch_pdl(round_select_kernel, E, kSelectThreads, key_smem, stream, 1, logits, T, E, W, tile, mode, seed, s.member,
                                                              s.final_set,
                                                              s.new_counts, s.keys, in_smem);
  const int EW = (E + 31) / 32;
  const int64_t tblocks = static_cast<int64_t>(EW) * W;  // warps
  launch_pdl(bits_transpose_kernel, static_cast<int>((tblocks * 32 + 255) / 256), 256, 0, stream, 1, s.final_set, T, E, W, EW,
                                                                                         s.tok_bits);
  const int tb = (T + 1023) / 1024;
  launch_pdl(token_offsets_local_kernel, tb, 1024, 0, stream, 1, s.tok_bits, T, EW, tok_offsets, s.block_sums);
  launch_pdl(token_offsets_add_kernel, tb, 1024, 0, stream, 1, T, tok_offsets, s.block_sums);
  launch_token_sets(logits, s.tok_bits, T, E, EW, tok_offsets, s.tok_expert, s.tok_w, s.tok_token, stream);
  // stable grouping by expert of the token-ordered list: rows of an expert
  // come out in ascending t; tok_rows is the list's row map (moe_permute's dst)
  launch_permute_list(s.tok_expert, s.tok_w, s.tok_token, tok_offsets + T, cap, E, s.chunk_hist, counts, offsets,
                      tok_rows, row_token, row_w, status, stream);
}

}  // namespace moe
