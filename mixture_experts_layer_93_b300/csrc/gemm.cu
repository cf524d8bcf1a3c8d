// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Up-projection:   h[r]  = bf16( silu(x[t_r] W1_e) * (x[t_r] W3_e) )
// Down-projection: ys[r] = fp16( w_r * (h[r] W2_e) )
//
// The row gather is fused into the operand load, the SwiGLU activation and the
// gate weight into the epilogue, and loads overlap the MMAs ("SonicMoE: 加速
// MoE 模型的 IO 与 Tile 感知优化": sections "2. IO 与计算重叠的 GPU Kernel",
// "Gather 与加载融合" and the "关键 Kernel 对比" table, rows "Gather 融合",
// "SwiGLU 融合", "MMA 与 IO 重叠").  The page's kernels use cp.async on
// Hopper; here the same roles map onto Blackwell hardware:
//
//   warp 0      TMA producer.  A rows come either by `tile::gather4` (four
//               arbitrary token rows per copy, 32 lanes x 4 = 128 rows per
//               tile) or by a tiled 2-D copy of contiguous rows; B tiles by a
//               tiled 2-D copy.  128-byte swizzle, a ring of STAGES slots.
//   warp 1      TMEM allocator; lane 0 issues tcgen05.mma (M=128, N=BN,
//               K=16, bf16 -> fp32) and tcgen05.commit to free slots.
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulator (each warp owns
//               32 TMEM lanes = 32 rows), fused SwiGLU or gate scaling, bf16
//               stores.  Two accumulators in TMEM so the epilogue of one tile
//               overlaps the MMAs of the next.
//
// Persistent: one CTA per SM walks tiles tau = blockIdx.x + i*gridDim.x.  The
// tile list is (expert, n-block, m-block) with m fastest, built on the device
// from the per-expert counts, so the host never learns the routing.  Every
// wait is bounded; on a timeout the kernel records MOE_ERR_TIMEOUT, lets its
// copies land, frees its TMEM and returns.
#include "common.cuh"
#include "kernels.h"

#include <mutex>

namespace moe {

struct GemmParams {
  const int32_t* counts;     // [E]
  const int32_t* offsets;    // [E+1]
  const int32_t* row_token;  // [cap] token of each row (gathered A only)
  const float* row_w;        // [cap] gate weight of each row (down only)
  __nv_bfloat16* out;        // up: h [cap, out_ld] bf16
  __half* out_h;             // down: ys [cap, out_ld] fp16
  int64_t out_ld;
  int E;
  int num_kb;                // K / 64
  int n_blocks;              // N tiles per expert
  int b_rows_per_expert;     // rows of packed B per expert
  int gather;                // 1: A rows gathered by token id, 0: contiguous rows
  int32_t* status;
  uint64_t timeout_ns;
};

template <int BN>
struct GemmCfg {
  static constexpr int BM = 128, BK = 64;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int BAR_BYTES = (2 * STAGES + 4) * 8 + 16;
  static constexpr int PREFIX_BYTES = 1025 * 4;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES + PREFIX_BYTES;
};

constexpr int kGemmThreads = 192;

__device__ __forceinline__ void decode_tile(int tau, const int32_t* prefix, int E, int n_blocks, int& e, int& nb,
                                            int& mb) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] * n_blocks <= tau)
      lo = mid;
    else
      hi = mid - 1;
  }
  e = lo;
  const int local = tau - prefix[e] * n_blocks;
  const int me = prefix[e + 1] - prefix[e];
  nb = local / me;
  mb = local - nb * me;
}

template <int BN, int MODE>  // MODE 0: up-projection + SwiGLU, MODE 1: down-projection + gate weight
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmParams p) {
  using C = GemmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::STAGES * C::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::STAGES * C::STAGE_BYTES);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + C::STAGES;
  uint64_t* tfull_bar = bars + 2 * C::STAGES;
  uint64_t* tempty_bar = bars + 2 * C::STAGES + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int32_t* prefix = reinterpret_cast<int32_t*>(base + C::STAGES * C::STAGE_BYTES + C::BAR_BYTES);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull_bar[a]), 1);
      mbar_init(smem_u32(&tempty_bar[a]), 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  } else if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  } else if (warp == 2) {
    // prefix[e] = number of 128-row tiles of experts < e
    int running = 0;
    if (lane == 0) prefix[0] = 0;
    for (int b = 0; b < p.E; b += 32) {
      const int e = b + lane;
      int m = 0;
      if (e < p.E) m = (p.counts[e] + C::BM - 1) / C::BM;
      int incl = m;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (e < p.E) prefix[e + 1] = running + incl;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total_tiles = prefix[p.E] * p.n_blocks;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_a = policy_evict_last();    // A rows are re-read by every n-block
    const uint64_t pol_b = policy_evict_normal();  // B tiles are re-read by the m-blocks of one expert
    int stage = 0;
    uint32_t phase = 0;
    for (int tau = blockIdx.x; tau < total_tiles; tau += gridDim.x) {
      int e, nb, mb;
      decode_tile(tau, prefix, p.E, p.n_blocks, e, nb, mb);
      const int row0 = p.offsets[e] + mb * C::BM;
      const int rows_valid = min(C::BM, p.counts[e] - mb * C::BM);
      int tok[4] = {0, 0, 0, 0};
      if (p.gather) {
#pragma unroll
        for (int q = 0; q < 4; ++q) tok[q] = p.row_token[row0 + min(lane * 4 + q, rows_valid - 1)];
      }
      const int brow = e * p.b_rows_per_expert + nb * BN;
      bool ok = true;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        int w = 1;
        if (lane == 0)
          w = mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag, p.status, kWaitProducerEmpty,
                                p.timeout_ns);
        if (!__shfl_sync(0xffffffffu, w, 0)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&full_bar[stage]);
        if (lane == 0) mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
        __syncwarp();
        const uint32_t a_dst = smem_u32(sA + stage * C::A_BYTES);
        if (p.gather) {
          tma_gather4(a_dst + lane * 512, &tmA, kb * C::BK, tok[0], tok[1], tok[2], tok[3], fb, pol_a);
        } else if (lane == 0) {
          tma_load_2d(a_dst, &tmA, kb * C::BK, row0, fb, pol_a);
        }
        if (lane == 0) tma_load_2d(smem_u32(sB + stage * C::B_BYTES), &tmB, kb * C::BK, brow, fb, pol_b);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(C::BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tau = blockIdx.x; tau < total_tiles && ok; tau += gridDim.x) {
        if (!mbar_wait_bounded(smem_u32(&tempty_bar[acc]), acc_phase ^ 1u, abort_flag, p.status,
                               kWaitMmaTmemEmpty, p.timeout_ns))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full_bar[stage]), phase, abort_flag, p.status, kWaitMmaFull,
                                 p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk) {
            tc_mma_bf16(d_tmem, smem_desc_k128(a0 + kk * 32), smem_desc_k128(b0 + kk * 32), idesc,
                        (kb > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(smem_u32(&empty_bar[stage]));
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tfull_bar[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp & 3;  // TMEM lanes 32*ew .. 32*ew+31
    const int r_in_tile = ew * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tau = blockIdx.x; tau < total_tiles; tau += gridDim.x) {
      int e, nb, mb;
      decode_tile(tau, prefix, p.E, p.n_blocks, e, nb, mb);
      const int row0 = p.offsets[e] + mb * C::BM;
      const int rows_valid = min(C::BM, p.counts[e] - mb * C::BM);
      int w = 1;
      if (lane == 0)
        w = mbar_wait_bounded(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, p.status, kWaitEpiTmemFull,
                              p.timeout_ns);
      if (!__shfl_sync(0xffffffffu, w, 0)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(acc * BN);
      const bool valid = r_in_tile < rows_valid;
      const int64_t row = static_cast<int64_t>(row0) + r_in_tile;
      if constexpr (MODE == 0) {
        constexpr int H = BN / 2;
        __nv_bfloat16* dst = p.out + row * p.out_ld + static_cast<int64_t>(nb) * H;
#pragma unroll 1
        for (int c = 0; c < H; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c, g);
          tmem_ld32(taddr + H + c, u);
          tc_wait_ld();
          uint32_t o[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float g0 = __uint_as_float(g[2 * q]), g1 = __uint_as_float(g[2 * q + 1]);
            const float u0 = __uint_as_float(u[2 * q]), u1 = __uint_as_float(u[2 * q + 1]);
            const float h0 = g0 / (1.0f + __expf(-g0)) * u0;
            const float h1 = g1 / (1.0f + __expf(-g1)) * u1;
            o[q] = pack_bf16x2(h0, h1);
          }
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int q = 0; q < 4; ++q) d4[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          }
        }
      } else {
        // ys = w * acc stored as fp16 (3 more mantissa bits than bf16 at the
        // same traffic); values past the fp16 range saturate and are reported
        const float wr = valid ? p.row_w[row] : 0.f;
        __half* dst = p.out_h + row * p.out_ld + static_cast<int64_t>(nb) * BN;
        bool overflow = false;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          tmem_ld32(taddr + c, v);
          tc_wait_ld();
          uint32_t o[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            float a = wr * __uint_as_float(v[2 * q]), b = wr * __uint_as_float(v[2 * q + 1]);
            overflow |= !(fabsf(a) <= kHalfMax) || !(fabsf(b) <= kHalfMax);
            a = fminf(fmaxf(a, -kHalfMax), kHalfMax);
            b = fminf(fmaxf(b, -kHalfMax), kHalfMax);
            o[q] = pack_half2(a, b);
          }
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int q = 0; q < 4; ++q) d4[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          }
        }
        if (overflow && valid) report_error(p.status, MOE_ERR_DEVICE_CHECK, kYsOverflow);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  __syncthreads();
  if (*abort_flag) {
    // let copies and MMAs already issued land before the memory goes away
    if (threadIdx.x == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) {
      }
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ----------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

// 2-D bf16 tensor [outer, inner] (inner contiguous), box [box_outer, 64], 128-byte swizzle.
static bool make_map_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int num_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

template <int BN, int MODE>
static int launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, cudaStream_t stream) {
  using C = GemmCfg<BN>;
  auto kern = moe_gemm_kernel<BN, MODE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
    return MOE_ERR_CUDA;
  kern<<<num_sms(), kGemmThreads, C::SMEM_BYTES, stream>>>(tmA, tmB, p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ row_token,
                                   const int32_t* __restrict__ offsets, int E, int d,
                                   __nv_bfloat16* __restrict__ out, int64_t rows_cap) {
  const int64_t R = min(static_cast<int64_t>(offsets[E]), rows_cap);
  const int groups = d / 8;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < R * groups;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / groups;
    const int g = static_cast<int>(i % groups);
    const int64_t t = row_token[r];
    reinterpret_cast<uint4*>(out + r * d)[g] = reinterpret_cast<const uint4*>(x + t * d)[g];
  }
}

void launch_gather_rows(const __nv_bfloat16* x, const int32_t* row_token, const int32_t* offsets, int E, int d,
                        __nv_bfloat16* out, int64_t rows_cap, cudaStream_t stream) {
  gather_rows_kernel<<<num_sms() * 8, 256, 0, stream>>>(x, row_token, offsets, E, d, out, rows_cap);
}

int launch_expert_up(const __nv_bfloat16* x, const __nv_bfloat16* W13p, const int32_t* counts,
                     const int32_t* offsets, const int32_t* row_token, __nv_bfloat16* h, int T, int d, int n, int E,
                     int64_t rows_cap, int gather, __nv_bfloat16* xperm_scratch, int32_t* status,
                     uint64_t timeout_ns, cudaStream_t stream) {
  const int H = up_half_block(n);
  const int BN = 2 * H;
  CUtensorMap tmA, tmB;
  if (gather) {
    if (!make_map_bf16(&tmA, x, d, T, 1)) return MOE_ERR_CUDA;
  } else {
    launch_gather_rows(x, row_token, offsets, E, d, xperm_scratch, rows_cap, stream);
    if (!make_map_bf16(&tmA, xperm_scratch, d, rows_cap, 128)) return MOE_ERR_CUDA;
  }
  if (!make_map_bf16(&tmB, W13p, d, static_cast<uint64_t>(E) * 2 * n, BN)) return MOE_ERR_CUDA;
  GemmParams p{};
  p.counts = counts;
  p.offsets = offsets;
  p.row_token = row_token;
  p.row_w = nullptr;
  p.out = h;
  p.out_h = nullptr;
  p.out_ld = n;
  p.E = E;
  p.num_kb = d / 64;
  p.n_blocks = n / H;
  p.b_rows_per_expert = 2 * n;
  p.gather = gather ? 1 : 0;
  p.status = status;
  p.timeout_ns = timeout_ns;
  if (BN == 256) return launch_gemm<256, 0>(tmA, tmB, p, stream);
  return launch_gemm<128, 0>(tmA, tmB, p, stream);
}

int launch_expert_down(const __nv_bfloat16* h, const __nv_bfloat16* W2p, const int32_t* counts,
                       const int32_t* offsets, const float* row_w, __half* ys, int d, int n, int E,
                       int64_t rows_cap, int32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  const int BN = (d % 256 == 0) ? 256 : (d % 128 == 0 ? 128 : 64);
  CUtensorMap tmA, tmB;
  if (!make_map_bf16(&tmA, h, n, rows_cap, 128)) return MOE_ERR_CUDA;
  if (!make_map_bf16(&tmB, W2p, n, static_cast<uint64_t>(E) * d, BN)) return MOE_ERR_CUDA;
  GemmParams p{};
  p.counts = counts;
  p.offsets = offsets;
  p.row_token = nullptr;
  p.row_w = row_w;
  p.out = nullptr;
  p.out_h = ys;
  p.out_ld = d;
  p.E = E;
  p.num_kb = n / 64;
  p.n_blocks = d / BN;
  p.b_rows_per_expert = d;
  p.gather = 0;
  p.status = status;
  p.timeout_ns = timeout_ns;
  if (BN == 256) return launch_gemm<256, 1>(tmA, tmB, p, stream);
  if (BN == 128) return launch_gemm<128, 1>(tmA, tmB, p, stream);
  return launch_gemm<64, 1>(tmA, tmB, p, stream);
}

// ------------------------------------------------------------- selftest
__global__ void selftest_timeout_kernel(int32_t* status, uint64_t timeout_ns) {
  // waits on a flag nothing sets, with the same bounded-wait policy the
  // pipeline uses, then reports the timeout and returns
  volatile int32_t* flag = status + 3;
  const uint64_t t0 = globaltimer_ns();
  while (*flag == 0) {
    if (globaltimer_ns() - t0 > timeout_ns) {
      report_error(status, MOE_ERR_TIMEOUT, kWaitSelftest);
      return;
    }
  }
}

void launch_selftest_timeout(int32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 1, 0, stream>>>(status, timeout_ns);
}

}  // namespace moe
