// Grouped GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Up-projection:   h[r]  = bf16( silu(x[t_r] W1_e) * (x[t_r] W3_e) )
// Down-projection: ys[r] = fp16( w_r * (h[r] W2_e) )
// Router:          L[t]  = x[t] Wr + b, with Wr split exactly into three
//                  bf16 terms (hi, mid, lo) held as three column groups of B;
//                  with at most 64 experts the epilogue also takes the top-k
// e4m3 variants of the up- and down-projection (scaled codes, kind::f8f6f4)
// Backward:        the pre-activations (g, u) in fp32; dh' = dy W2^T with the
//                  SwiGLU backward in its epilogue; the weight gradients, whose
//                  K is each expert's rows, from MN-major operands
//
// The SwiGLU activation and the gate weight are fused into the epilogue, and
// loads overlap the MMAs ("SonicMoE: 加速 MoE 模型的 IO 与 Tile 感知优化":
// sections "2. IO 与计算重叠的 GPU Kernel", "Gather 与加载融合" and the "关键
// Kernel 对比" table, rows "Gather 融合", "SwiGLU 融合", "MMA 与 IO 重叠").  The
// up-projection's A rows come either from a staging buffer the token-order
// copy kernel filled (tiled TMA, `gather` 0, the forward's path) or straight
// from x by a gather fused into the operand load (`gather` 1 and 2).  The
// page's kernels use cp.async on Hopper; here the roles map onto Blackwell
// hardware:
//
//   warps 0..3  producers.  B tiles (and A tiles of contiguous rows) come by
//               tiled TMA, issued by warp 0.  Gathered A rows come either by
//               TMA `tile::gather4` (warp 0, four token rows per copy) or by
//               16-byte cp.async from all four warps, written straight into
//               the 128-byte-swizzled layout, each lane arriving on the stage
//               barrier when its copies land (non-blocking).
//   warp 4      TMEM allocator; lane 0 issues tcgen05.mma (M=128, or 256
//               on an SM pair with cta_group::2; N=BN, K=16 bf16 or 32 e4m3
//               -> fp32 in tensor memory) and tcgen05.commit.
//   warps 5..8  epilogue (5..8 and 10..13 with eight warps, two per lane
//               quadrant): tcgen05.ld of the accumulator (warp w owns TMEM
//               lanes 32*(w%4)..+31 = 32 rows), fused activation / scaling,
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
#include "topk.cuh"

#include <algorithm>

namespace moe {

// F8: e4m3.  UpPre stores the up-projection's pre-activations; BwdAct and
// Wgrad are the backward pass (see their epilogues).
enum GemmMode : int {
  kModeUp = 0, kModeDown = 1, kModeRouter = 2, kModeUpF8 = 3, kModeDownF8 = 4,
  kModeUpPre = 5, kModeBwdAct = 6, kModeWgrad = 7, kModeDxRows = 8
};

struct GemmParams {
  const int32_t* counts;     // [E] rows per group (ignored when single_rows > 0)
  const int32_t* offsets;    // [E+1] first row of each group
  int single_rows;           // > 0: one group of this many rows starting at row 0
  const int32_t* row_token;  // [cap] token of each row (gathered A only)
  const float* row_w;        // [cap] gate weight of each row (down)
  const float* bias;         // [E_out] router bias or nullptr
  __nv_bfloat16* out_bf16;   // up: h [cap, out_ld]
  __half* out_f16;           // down: ys [cap, out_ld]
  float* out_f32;            // router: logits [T, out_ld]
  int64_t out_ld;
  int out_cols;              // router: number of valid output columns (E)
  int E;                     // groups
  int num_kb;                // K / 64
  int n_blocks;              // N tiles per group
  int b_rows_per_expert;     // rows of packed B per group
  int units;                 // tiles per group: 0 every 128-row block, 1 complete pairs of
                             // blocks (PAIR kernels), 2 the odd last block of each group
  int gather;                // A rows: 0 contiguous (tiled TMA), 1 TMA gather4 by token,
                             // 2 16-byte cp.async by token
  const __nv_bfloat16* x;    // gather 2: token rows
  int64_t lda;
  int32_t* status;
  uint64_t timeout_ns;
  const float* row_scale;    // F8: scale of each A row [cap]
  const float* col_scale;    // F8: scale of each B row (output channel) [E * b_rows_per_expert]
  // backward
  const float* pre;          // BwdAct: pre-activations (g, u interleaved) [cap, 2 * out_ld]
  __nv_bfloat16* out2_bf16;  // BwdAct: w * h [cap, out_ld]
  float* out2_f32;           // BwdAct: partial <dh, h> [cap, parts]; Wgrad: odd M rows when interleaved
  int parts;                 // BwdAct: partials per row (n_blocks)
  int m_units;               // Wgrad: M tile units per group
  int64_t out_group_stride;  // Wgrad: elements between the outputs of consecutive groups
  int interleave;            // Wgrad: even M rows go to out_f32, odd ones to out2_f32, at row M / 2
  int m_fast;                // Wgrad: tile order within a group, M units fastest (else N blocks)
  // Router with the top-k fused (topk_k > 0): the tile covers every expert
  int32_t* topk_idx;         // [T * k]
  float* topk_w;             // [T * k]
  int topk_k;                // <= kFusedTopk
  int32_t* chunk_hist;       // [E * nchunks], zero on entry
  int nchunks;
  // DxRows: out = acc + row_add[r] * col_add[group][col] (the gate network's term)
  const float* row_add;      // [cap]
  const float* col_add;      // [E * out_ld]
};

constexpr int kProducerWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kEpiWarp0 = 5;   // epilogue warps 5..8 (and 10..13 with eight)
constexpr int kRelayWarp = 9;  // gather 2: publishes landed rows to the MMA warp
// Epilogue width: four warps (one per TMEM lane quadrant), or eight (two per
// quadrant, each taking half the columns) for short-K tiles whose epilogue is
// on the critical path; eight cost one operand stage of shared memory.
__host__ __device__ constexpr int gemm_threads(int epi_warps) { return (epi_warps == 8 ? 14 : 10) * 32; }

__host__ __device__ constexpr int tmem_cols_for(int n) { return n <= 32 ? 32 : (n <= 64 ? 64 : (n <= 128 ? 128 : (n <= 256 ? 256 : 512))); }

// PAIR: two CTAs of a cluster run one 256-row tile with tcgen05 cta_group::2.
// CTA rank r holds A rows 128r..128r+127 and B rows r*BN/2..r*BN/2+BN/2-1 in
// its own shared memory; the even CTA issues M=256 MMAs that read both CTAs'
// operands; D rows 128r.. land in CTA r's TMEM.  Each SM thus stores and feeds
// half of B: per k-block 32 KB of shared-memory writes and reads instead of
// 48 KB, which is what keeps a 1-CTA M=128 x N=256 MMA from full rate.
// SUP = 1 (super tiles): the pair runs two 256-row tiles of one group against
// the same B tile, so a stage holds two A tiles (one per tile) and one B tile
// and each k-block issues both tiles' MMAs.  Per k-block an SM then stores
// 48 KB and its tensor core reads 64 KB for twice the MMA work: 112 KB of
// shared-memory traffic per 1024 MMA cycles instead of 64 KB per 512, and a
// third less TMA traffic per FLOP.  SUP = 2 (wide tiles): the same along N,
// one A tile against the B tiles of two consecutive n-blocks, so each row
// block reaches shared memory (or is gathered) once per two n-blocks.  Either
// way the two accumulators fill the 512 TMEM columns, so the epilogue of one
// tile does not overlap the next one's MMAs.
template <int BN, bool PAIR, int EPI, int SUP = 0>
struct GemmCfg {
  static constexpr int BM = 128, BK = 64;
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // B rows held per CTA
  static constexpr int A_TILE_BYTES = BM * BK * 2;   // one 128-row A tile
  static constexpr int A_BYTES = A_TILE_BYTES * (SUP == 1 ? 2 : 1);
  static constexpr int B_TILE_BYTES = B_ROWS * BK * 2;  // one n-block's B rows
  static constexpr int B_BYTES = B_TILE_BYTES * (SUP == 2 ? 2 : 1);
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // epilogue staging for TMA stores: per epilogue warp two 32 x 64-byte boxes
  // (one with eight warps on super tiles, which keeps their fourth stage)
  static constexpr int OUT_BOXES = (SUP != 0 && EPI == 8) ? 1 : 2;
  // operand ring: what is left of 227 KB after the staging boxes, barriers,
  // prefix table and token table (at most 8 stages)
  static constexpr int RING_BUDGET =
      232448 - 1024 - EPI * OUT_BOXES * 32 * 64 - (3 * 8 + 4) * 8 - 16 - 1025 * 4 - BM * 4 - 4 - 1024 * 8;
  static constexpr int STAGES = (RING_BUDGET / STAGE_BYTES) > 8 ? 8 : (RING_BUDGET / STAGE_BYTES);
  static constexpr int TMEM_COLS = tmem_cols_for(2 * BN);
  static constexpr int BAR_BYTES = (3 * STAGES + 4) * 8 + 16;
  static constexpr int PREFIX_BYTES = 1025 * 4;
  static constexpr int TOK_BYTES = BM * 4;
  static constexpr int GRP_BYTES = 4 + 1024 * 8;  // alignment pad + (first row, rows) of each group
  static constexpr int STAGE_OUT_BYTES = EPI * OUT_BOXES * 32 * 64;
  static constexpr int SMEM_BYTES =
      1024 + STAGES * STAGE_BYTES + STAGE_OUT_BYTES + BAR_BYTES + PREFIX_BYTES + TOK_BYTES + GRP_BYTES;
  static_assert(B_BYTES % 1024 == 0, "B tile must keep 1024-byte alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(BAR_BYTES % 8 == 0 && STAGE_OUT_BYTES % 8 == 0 && (PREFIX_BYTES + TOK_BYTES + 4) % 8 == 0,
                "group table alignment");
};

// Tile units of one group that run as a chunk (see decode_tile).
constexpr int kMChunk = 8;

// e: on entry the group of a tile at or before tau (each warp visits its tiles
// in increasing order, starting from e = 0); on exit the group of tau.  A few
// linear probes cover the usual step to the same or a nearby group, then a
// binary search over the rest.  prefix[E] * n_blocks > tau bounds both.
// Within a group the m-block runs fastest (N_FAST false): the expert's weight
// slice of one n-block stays in L2 for all its m-blocks.  A group with more
// than kMChunk units runs them in chunks of kMChunk, each over every n-block
// (m fastest within the chunk): its A rows stay in L2 across the n-blocks
// instead of streaming from HBM once per n-block (a heavily loaded expert's
// rows exceed L2).  N_FAST (the router, whose whole B is a few MB) runs the
// n-blocks of one m-block together, so each A row block is read from HBM once.
template <bool N_FAST = false>
__device__ __forceinline__ void decode_tile(int tau, const int32_t* prefix, int E, int n_blocks, int& e, int& nb,
                                            int& mb) {
  for (int probe = 0; prefix[e + 1] * n_blocks <= tau; ++probe) {
    if (probe == 4) {
      int lo = e + 1, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] * n_blocks <= tau)
          lo = mid;
        else
          hi = mid - 1;
      }
      e = lo;
      break;
    }
    ++e;
  }
  const int local = tau - prefix[e] * n_blocks;
  if (N_FAST) {
    mb = local / n_blocks;
    nb = local - mb * n_blocks;
  } else {
    const int me = prefix[e + 1] - prefix[e];
    if (me <= kMChunk) {
      nb = local / me;
      mb = local - nb * me;
    } else {
      const int chunk = local / (kMChunk * n_blocks);
      const int r = local - chunk * (kMChunk * n_blocks);
      const int units = min(kMChunk, me - chunk * kMChunk);  // the last chunk may be short
      nb = r / units;
      mb = chunk * kMChunk + (r - nb * units);
    }
  }
}

// Tile units of a group with mblocks 128-row blocks: 0 every block, 1
// complete pairs, 2 the odd last block, 3 pairs with the odd last block run as
// a half-empty pair; super tiles (two pairs, blocks 4mu..4mu+3): 4 with the
// odd last block in the last unit, 5 over complete pairs only (the odd last
// block runs in the units-2 launch).
__device__ __forceinline__ int tile_units(int units, int mblocks) {
  if (units == 0) return mblocks;
  if (units == 1) return mblocks / 2;
  if (units == 2) return mblocks & 1;
  if (units == 4) return (mblocks + 3) / 4;
  if (units == 5) return (mblocks / 2 + 1) / 2;
  return (mblocks + 1) / 2;
}

// 128-row block of unit mu handled by CTA `rank` (super tiles: its block of
// the unit's first pair; its block of the second pair is 2 more).
__device__ __forceinline__ int unit_block(int units, int mu, int rank, int gcount) {
  if (units == 1 || units == 3) return 2 * mu + rank;
  if (units == 2) return (gcount + 127) / 128 - 1;
  if (units == 4 || units == 5) return 4 * mu + rank;
  return mu;
}

// Blocks of a group that a super-tile kernel runs: all of them (units 4), or
// all but the odd last one (units 5).
__device__ __forceinline__ int super_blocks(int units, int gcount) {
  const int mblocks = (gcount + 127) / 128;
  return units == 5 ? (mblocks & ~1) : mblocks;
}

// First row and row count of group e; grp_s holds (offsets[e], counts[e]),
// copied to shared memory once per CTA.
__device__ __forceinline__ void group_rows(const GemmParams& p, const int2* grp_s, int e, int& row_start,
                                           int& count) {
  if (p.single_rows > 0) {
    row_start = 0;
    count = p.single_rows;
  } else {
    const int2 g = grp_s[e];
    row_start = g.x;
    count = g.y;
  }
}

// Weight-gradient tiles: every group has m_units x n_blocks tiles (empty
// groups too: their gradient is zero).  The tiles that run together share
// one operand block and sweep the other operand of the group, which should
// be the smaller one (it then stays in L2): n fastest sweeps B, m fastest A.
__device__ __forceinline__ void wgrad_tile(int tau, const GemmParams& p, int& e, int& mu, int& nb) {
  const int per = p.m_units * p.n_blocks;
  e = tau / per;
  const int local = tau - e * per;
  if (p.m_fast) {
    nb = local / p.m_units;
    mu = local - nb * p.m_units;
  } else {
    mu = local / p.n_blocks;
    nb = local - mu * p.n_blocks;
  }
}

template <int BN, int MODE, bool PAIR, int EPI, int SUP = 0>
__global__ void __launch_bounds__(gemm_threads(EPI), 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  using C = GemmCfg<BN, PAIR, EPI, SUP>;
  static_assert(SUP == 0 || (PAIR && BN == 256 && (MODE == kModeUp || MODE == kModeDown)),
                "super and wide tiles: up or down GEMM on SM pairs with 256-wide n-blocks");
  static_assert(SUP != 2 || MODE == kModeUp || MODE == kModeDown, "wide tiles: the up or down GEMM");
  constexpr int kPer = PAIR ? 2 : 1;  // CTAs per tile unit
  constexpr bool kF8 = MODE == kModeUpF8 || MODE == kModeDownF8;
  constexpr bool kDown = MODE == kModeDown || MODE == kModeDownF8 || MODE == kModeDxRows;
  constexpr bool kWgrad = MODE == kModeWgrad;
  static_assert(!kF8 || PAIR, "the e4m3 GEMMs run on SM pairs");
  static_assert(!kWgrad || (C::B_ROWS % 64 == 0 && EPI == 4), "weight-gradient tiles: 64-wide B blocks");
  // Wgrad operands are MN-major: [64 K rows][64 elements] boxes, 8 KB each,
  // two for the 128 A columns, B_ROWS / 64 for B
  constexpr uint32_t kMnBlock = 64 * 128;
  // K elements per operand stage: a stage row is 128 bytes (64 bf16 or 128 e4m3)
  constexpr int KB_ELEMS = kF8 ? 128 : C::BK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::STAGES * C::A_BYTES;
  uint8_t* sOut = base + C::STAGES * C::STAGE_BYTES;  // 1024-aligned: STAGE_BYTES is a multiple of 1024
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + C::STAGE_OUT_BYTES);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + C::STAGES;
  uint64_t* tfull_bar = bars + 2 * C::STAGES;
  uint64_t* tempty_bar = bars + 2 * C::STAGES + 2;
  uint64_t* afull_bar = bars + 2 * C::STAGES + 4;  // PAIR + gather 2: this CTA's rows landed
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * C::STAGES + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int32_t* prefix = reinterpret_cast<int32_t*>(sOut + C::STAGE_OUT_BYTES + C::BAR_BYTES);
  int32_t* tok_s = prefix + 1025;  // gather 2: token of each row of the current tile
  // prefix starts 8-byte aligned; one int of padding after tok_s aligns grp_s
  int2* grp_s = reinterpret_cast<int2*>(tok_s + C::BM + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_groups = p.single_rows > 0 ? 1 : p.E;
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = (rank == 0);  // issues the MMAs
  const int unit0 = PAIR ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
  const int unit_stride = PAIR ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);

  if (warp == 0 && lane == 0) {
    // gather 2 (single CTA): one arrival per producer lane (when its copies
    // land) plus warp 0's expect-tx arrival for the B tile.  PAIR: the even
    // CTA's full barrier counts the bytes of both CTAs' TMA copies; with
    // gather 2 it also takes one relay arrival from the odd CTA ("its rows
    // landed"), while each CTA's own rows land on its afull barrier.  The even
    // CTA's tmem-empty barrier takes the four epilogue warps of both CTAs.
    uint32_t full_count = 1;
    if (p.gather == 2) full_count = PAIR ? 3 : 2;  // + one relay arrival per CTA
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), full_count);
      mbar_init(smem_u32(&empty_bar[s]), 1);
      mbar_init(smem_u32(&afull_bar[s]), 32 * kProducerWarps);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull_bar[a]), 1);
      mbar_init(smem_u32(&tempty_bar[a]), EPI * kPer);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (MODE != kModeRouter && MODE != kModeBwdAct && MODE != kModeWgrad) tma_prefetch_desc(&tmC);  // UpPre: fp32 boxes
  } else if (warp == kMmaWarp) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_holder), C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
      tmem_relinquish();
    }
    tc_fence_before();
  } else if (warp == kEpiWarp0) {
    // prefix[e] = number of tile units of groups < e (this warp is free before the pipeline starts)
    pdl_wait();  // counts come from the previous kernel
    if (p.single_rows > 0) {
      if (lane == 0) {
        prefix[0] = 0;
        prefix[1] = tile_units(p.units, (p.single_rows + C::BM - 1) / C::BM);
      }
    } else {
      int running = 0;
      if (lane == 0) prefix[0] = 0;
      for (int b = 0; b < p.E; b += 32) {
        const int e = b + lane;
        int m = 0;
        if (e < p.E) {
          const int c = p.counts[e];
          grp_s[e] = make_int2(p.offsets[e], c);
          m = tile_units(p.units, (c + C::BM - 1) / C::BM);
        }
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
  }
  // barrier init, TMEM allocation and descriptor prefetch above touch no data
  // of earlier kernels; everything below may
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  // the peer's copies, commits and arrivals target our barriers: both CTAs'
  // barriers are initialised before either starts
  if (PAIR) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total_tiles = kWgrad ? p.E * p.m_units * p.n_blocks : prefix[n_groups] * p.n_blocks;
  // The i-th tile of this CTA (pair): unit0 + i * unit_stride.  The router
  // with the top-k fused takes all n-blocks of one m-unit in a row instead,
  // so that a thread has seen every expert of its token before the next one.
  const bool by_unit = MODE == kModeRouter && p.topk_k > 0 && p.n_blocks > 1;
  auto tau_of = [&](int i) -> int {
    if (by_unit) return (unit0 + (i / p.n_blocks) * unit_stride) * p.n_blocks + (i % p.n_blocks);
    return unit0 + i * unit_stride;
  };
  // the tile after tau (the it-th of this CTA): a plain stride step unless by_unit
  auto tau_next = [&](int tau, int it) -> int { return by_unit ? tau_of(it + 1) : tau + unit_stride; };

  if (warp < kProducerWarps) {
    // ------------------------------------------------------------ producers
    const bool issuer = (warp == 0);
    if constexpr (kWgrad) {
      // K runs over the group's rows (padded to 64 with zero rows); A holds
      // this CTA's 128 M columns, B its B_ROWS N columns, both MN-major
      if (issuer) {
        const uint64_t pol = policy_evict_normal();
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tau = unit0; tau < total_tiles && ok; tau += unit_stride) {
          int e, mu, nb;
          wgrad_tile(tau, p, e, mu, nb);
          const int2 g = grp_s[e];
          const int nkb = (g.y + C::BK - 1) / C::BK;
          const int m0 = (mu * kPer + rank) * C::BM;
          const int n0 = nb * BN + rank * C::B_ROWS;
          for (int kb = 0; kb < nkb; ++kb) {
            int w = 1;
            if (lane == 0)
              w = mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag, p.status,
                                    kWaitProducerEmpty, p.timeout_ns);
            if (!__shfl_sync(0xffffffffu, w, 0)) {
              ok = false;
              break;
            }
            if (lane == 0) {
              const uint32_t fb = smem_u32(&full_bar[stage]);
              const uint32_t a_dst = smem_u32(sA + stage * C::A_BYTES);
              const uint32_t b_dst = smem_u32(sB + stage * C::B_BYTES);
              const int krow = g.x + kb * C::BK;
              if (PAIR) {
                const uint32_t fb0 = map_to_cta(fb, 0);
                if (leader) mbar_arrive_expect_tx(fb, 2 * C::STAGE_BYTES);
#pragma unroll
                for (int i = 0; i < C::BM / 64; ++i) tma_load_2d_pair(a_dst + i * kMnBlock, &tmA, m0 + 64 * i, krow, fb0, pol);
#pragma unroll
                for (int i = 0; i < C::B_ROWS / 64; ++i)
                  tma_load_2d_pair(b_dst + i * kMnBlock, &tmB, n0 + 64 * i, krow, fb0, pol);
              } else {
                mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
#pragma unroll
                for (int i = 0; i < C::BM / 64; ++i) tma_load_2d(a_dst + i * kMnBlock, &tmA, m0 + 64 * i, krow, fb, pol);
#pragma unroll
                for (int i = 0; i < C::B_ROWS / 64; ++i)
                  tma_load_2d(b_dst + i * kMnBlock, &tmB, n0 + 64 * i, krow, fb, pol);
              }
            }
            __syncwarp();
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    } else if (issuer || p.gather == 2) {
      // expert GEMMs: A rows are re-read by every n-block, a B slice only by
      // the m-blocks of one group; router: the few-MB B is re-read by every
      // m-block, an A row block only by its n-blocks (run together)
      const uint64_t pol_a = MODE == kModeRouter ? policy_evict_normal() : policy_evict_last();
      const uint64_t pol_b = MODE == kModeRouter ? policy_evict_last() : policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int e = 0;  // group cursor of decode_tile
      for (int it = 0, tau = tau_of(0); tau < total_tiles && ok; tau = tau_next(tau, it), ++it) {
        int nb, mu, gstart, gcount;
        decode_tile<MODE == kModeRouter>(tau, prefix, n_groups, p.n_blocks, e, nb, mu);
        group_rows(p, grp_s, e, gstart, gcount);
        const int mb = unit_block(p.units, mu, rank, gcount);
        const int row0 = gstart + mb * C::BM;
        const int rows_valid = min(C::BM, gcount - mb * C::BM);
        // units 3: the odd CTA's block of the last pair may lie past the group
        const bool partner_empty = PAIR && (2 * mu + 1) * C::BM >= gcount;
        // gathered rows past the group repeat a row of the group
        const int last = max(rows_valid, 1) - 1;
        const int tok_base = rows_valid > 0 ? row0 : gstart;
        int tok[4] = {0, 0, 0, 0};
        if (p.gather == 1) {
#pragma unroll
          for (int q = 0; q < 4; ++q) tok[q] = p.row_token[tok_base + min(lane * 4 + q, last)];
        } else if (p.gather == 2) {
          __syncwarp();
          const int r = warp * 32 + lane;
          tok_s[r] = p.row_token[tok_base + min(r, last)];
          __syncwarp();
        }
        // wide tiles cover n-blocks 2nb and 2nb + 1
        const int brow = e * p.b_rows_per_expert + (SUP == 2 ? 2 * nb : nb) * BN + rank * C::B_ROWS;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          int w = 1;
          if (lane == 0)
            w = mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag, p.status,
                                  kWaitProducerEmpty, p.timeout_ns);
          if (!__shfl_sync(0xffffffffu, w, 0)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full_bar[stage]);
          const uint32_t a_dst = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b_dst = smem_u32(sB + stage * C::B_BYTES);
          if (issuer) {
            if (SUP == 1) {
              // super tile: this CTA's block of each pair (if the kernel runs
              // it) and its half of the B tile; the even CTA's barrier counts
              // every A tile either CTA loads
              const uint32_t fb0 = map_to_cta(fb, 0);
              if (lane == 0) {
                const int lim = super_blocks(p.units, gcount), b0 = 4 * mu;
                if (leader) {
                  const int tiles = (b0 < lim) + (b0 + 1 < lim) + (b0 + 2 < lim) + (b0 + 3 < lim);
                  mbar_arrive_expect_tx(fb, 2 * C::B_BYTES + tiles * C::A_TILE_BYTES);
                }
                if (b0 + rank < lim)
                  tma_load_2d_pair(a_dst, &tmA, kb * KB_ELEMS, gstart + (b0 + rank) * C::BM, fb0, pol_a);
                if (b0 + 2 + rank < lim)
                  tma_load_2d_pair(a_dst + C::A_TILE_BYTES, &tmA, kb * KB_ELEMS, gstart + (b0 + 2 + rank) * C::BM, fb0,
                                   pol_a);
                tma_load_2d_pair(b_dst, &tmB, kb * KB_ELEMS, brow, fb0, pol_b);
              }
            } else if (PAIR) {
              // both CTAs' TMA copies complete on the even CTA's barrier
              const uint32_t fb0 = map_to_cta(fb, 0);
              if (lane == 0) {
                // a half-empty pair tile (the odd CTA's block lies past the
                // group) skips the odd CTA's A rows: its accumulator rows are
                // never stored, so stale operand rows there are harmless
                if (leader)
                  mbar_arrive_expect_tx(fb, p.gather == 2 ? 2 * C::B_BYTES
                                                          : 2 * C::STAGE_BYTES - (partner_empty ? C::A_BYTES : 0));
                if (p.gather == 0 && rows_valid > 0) tma_load_2d_pair(a_dst, &tmA, kb * KB_ELEMS, row0, fb0, pol_a);
                tma_load_2d_pair(b_dst, &tmB, kb * KB_ELEMS, brow, fb0, pol_b);
                // wide tile: the next n-block's B rows beside this one's
                if (SUP == 2)
                  tma_load_2d_pair(b_dst + C::B_TILE_BYTES, &tmB, kb * KB_ELEMS, brow + BN, fb0, pol_b);
              }
            } else {
              if (lane == 0) mbar_arrive_expect_tx(fb, p.gather == 2 ? C::B_BYTES : C::STAGE_BYTES);
              __syncwarp();
              if (p.gather == 1) {
                tma_gather4(a_dst + lane * 512, &tmA, kb * C::BK, tok[0], tok[1], tok[2], tok[3], fb, pol_a);
              } else if (p.gather == 0 && lane == 0) {
                tma_load_2d(a_dst, &tmA, kb * C::BK, row0, fb, pol_a);
              }
              if (lane == 0) tma_load_2d(b_dst, &tmB, kb * C::BK, brow, fb, pol_b);
            }
          }
          if (p.gather == 2) {
            // lane owns 16-byte chunk c of rows r = 32*warp + lane/8 + 4i; the
            // chunk goes to its swizzled slot (c ^ (r mod 8)) of row r
            const int c = lane & 7;
            const __nv_bfloat16* xk = p.x + static_cast<int64_t>(kb) * C::BK + c * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = warp * 32 + (lane >> 3) + 4 * i;
              cp_async_16(a_dst + r * 128 + ((c ^ (r & 7)) << 4), xk + static_cast<int64_t>(tok_s[r]) * p.lda);
            }
            cp_async_arrive_noinc(smem_u32(&afull_bar[stage]));
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (p.gather == 2) cp_async_wait_all();  // nothing of ours in flight at exit
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = kF8       ? idesc_e4m3_f32(kPer * C::BM, BN)
                                 : kWgrad ? idesc_bf16_f32_mn(kPer * C::BM, BN)
                                          : idesc_bf16_f32(kPer * C::BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      [[maybe_unused]] int mma_e = 0;  // SUP: group cursor of decode_tile
      for (int it = 0, tau = tau_of(0); tau < total_tiles && ok; tau = tau_next(tau, it), ++it) {
        if (!mbar_wait_bounded(smem_u32(&tempty_bar[acc]), acc_phase ^ 1u, abort_flag, p.status,
                               kWaitMmaTmemEmpty, p.timeout_ns))
          break;
        tc_fence_after();
        // SUP: one accumulator pair per tile (columns 0..BN-1 and BN..2BN-1);
        // a super tile's second pair's MMAs run only when the kernel runs its
        // blocks, a wide tile's second n-block's always
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(SUP != 0 ? 0 : acc * BN);
        [[maybe_unused]] bool two = SUP == 2;
        if constexpr (SUP == 1) {
          int nb_, mu_, gstart_, gcount_;
          decode_tile<false>(tau, prefix, n_groups, p.n_blocks, mma_e, nb_, mu_);
          group_rows(p, grp_s, mma_e, gstart_, gcount_);
          two = 4 * mu_ + 2 < super_blocks(p.units, gcount_);
        }
        int nkb = p.num_kb;
        if constexpr (kWgrad) {
          // a group without rows issues no MMA: its epilogue writes zeros
          int e, mu, nb;
          wgrad_tile(tau, p, e, mu, nb);
          nkb = (grp_s[e].y + C::BK - 1) / C::BK;
        }
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded<PAIR>(smem_u32(&full_bar[stage]), phase, abort_flag, p.status, kWaitMmaFull,
                                       p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk) {
            // K-major: 16 elements = 32 bytes along a row; MN-major: 16 K rows = 2048 bytes
            const uint64_t ad = kWgrad ? smem_desc_mn128(a0 + kk * 2048, kMnBlock, 1024) : smem_desc_k128(a0 + kk * 32);
            const uint64_t bd = kWgrad ? smem_desc_mn128(b0 + kk * 2048, kMnBlock, 1024) : smem_desc_k128(b0 + kk * 32);
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            if constexpr (kF8)  // 32 e4m3 of K per instruction: the same 32 bytes per row as 16 bf16
              tc_mma_f8_pair(d_tmem, ad, bd, idesc, accum);
            else if (PAIR)
              tc_mma_bf16_pair(d_tmem, ad, bd, idesc, accum);
            else
              tc_mma_bf16(d_tmem, ad, bd, idesc, accum);
          }
          if constexpr (SUP == 1) {
            if (two) {
              const uint32_t a1 = a0 + C::A_TILE_BYTES;
#pragma unroll
              for (int kk = 0; kk < C::BK / 16; ++kk)
                tc_mma_bf16_pair(d_tmem + BN, smem_desc_k128(a1 + kk * 32), smem_desc_k128(b0 + kk * 32), idesc,
                                 (kb > 0 || kk > 0) ? 1u : 0u);
            }
          } else if constexpr (SUP == 2) {
            // wide tile: the same A rows against the next n-block's B rows
            const uint32_t b1 = b0 + C::B_TILE_BYTES;
#pragma unroll
            for (int kk = 0; kk < C::BK / 16; ++kk)
              tc_mma_bf16_pair(d_tmem + BN, smem_desc_k128(a0 + kk * 32), smem_desc_k128(b1 + kk * 32), idesc,
                               (kb > 0 || kk > 0) ? 1u : 0u);
          }
          // the slot is free in both CTAs once these MMAs have read it
          if (PAIR)
            tc_commit_pair_multicast(smem_u32(&empty_bar[stage]), 0x3);
          else
            tc_commit(smem_u32(&empty_bar[stage]));
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (PAIR)
          tc_commit_pair_multicast(smem_u32(&tfull_bar[acc]), 0x3);
        else
          tc_commit(smem_u32(&tfull_bar[acc]));
        if (SUP != 0) {
          acc_phase ^= 1u;  // one accumulator set: every tile waits for the last one's epilogue
        } else {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
    }
  } else if (warp == kRelayWarp) {
    // ------------------------------------------------------------ relay
    // gather 2: once this CTA's gathered rows of a k-block have landed, make
    // them visible to the tensor core's operand reads (generic -> async proxy
    // fence) and arrive on the full barrier the MMA thread waits on (the even
    // CTA's when paired).  The proxy fence stays off the MMA-issuing thread.
    if (p.gather == 2 && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0, tau = tau_of(0); tau < total_tiles && ok; tau = tau_next(tau, it), ++it) {
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&afull_bar[stage]), phase, abort_flag, p.status, kWaitRelay,
                                 p.timeout_ns)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();
          if (PAIR)
            mbar_arrive_cluster(map_to_cta(smem_u32(&full_bar[stage]), 0));
          else
            mbar_arrive(smem_u32(&full_bar[stage]));
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp & 3;  // TMEM lanes 32*ew .. 32*ew+31
    const int epi = warp < kRelayWarp ? warp - kEpiWarp0 : warp - kEpiWarp0 - 1;  // 0..EPI-1
    constexpr int NCH = EPI / 4;  // column slices per TMEM lane quadrant
    const int ch = epi / 4;       // this warp's slice
    const int r_in_tile = ew * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    // 32 rows x 32 columns of 16-bit outputs per chunk go through one of this
    // warp's two staging boxes (64-byte rows, 64-byte swizzle) to a TMA store
    uint8_t* stage_out = sOut + epi * (C::OUT_BOXES * 32 * 64);
    int out_buf = 0;
    auto store_chunk = [&](const uint32_t (&o)[16], int col, int64_t row_w0, int warp_rows, int64_t row,
                           auto* dst_row) {
      if (warp_rows == 32) {
        uint8_t* buf = stage_out + out_buf * (32 * 64);
        if (lane == 0) bulk_wait_read<C::OUT_BOXES - 1>();  // the box to be reused was read
        __syncwarp();
        const int sw = (lane >> 1) & 3;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(buf + lane * 64 + ((q ^ sw) << 4)) =
              make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmC, col, static_cast<int32_t>(row_w0), smem_u32(buf));
          bulk_commit();
        }
        if (C::OUT_BOXES == 2) out_buf ^= 1;
      } else if (lane < warp_rows) {
        uint4* d4 = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
        for (int q = 0; q < 4; ++q) d4[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      }
      (void)row;
    };
    if constexpr (kWgrad) {
      // Lane r_in_tile holds M index m of the tile; TMEM column c is N index
      // nb*BN + c.  Stores run along M (consecutive lanes, consecutive
      // addresses): out[group][N][M], or with interleave the even and odd M
      // rows of out / out2 at M / 2.
      for (int tau = unit0; tau < total_tiles; tau += unit_stride) {
        int e, mu, nb;
        wgrad_tile(tau, p, e, mu, nb);
        const bool empty = grp_s[e].y == 0;
        const int m = (mu * kPer + rank) * C::BM + r_in_tile;
        float* dst = (p.interleave && (m & 1)) ? p.out2_f32 : p.out_f32;
        dst += static_cast<int64_t>(e) * p.out_group_stride + (p.interleave ? (m >> 1) : m);
        int w = 1;
        if (lane == 0)
          w = mbar_wait_bounded(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, p.status, kWaitEpiTmemFull,
                                p.timeout_ns);
        if (!__shfl_sync(0xffffffffu, w, 0)) break;
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          if (!empty) {
            tmem_ld32(taddr + c, v);
            tc_wait_ld();
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = 0u;
          }
          const int64_t n0 = static_cast<int64_t>(nb) * BN + c;
#pragma unroll
          for (int q = 0; q < 32; ++q) dst[(n0 + q) * p.out_ld] = __uint_as_float(v[q]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR)
            mbar_arrive_cluster_relaxed(map_to_cta(smem_u32(&tempty_bar[acc]), 0));
          else
            mbar_arrive(smem_u32(&tempty_bar[acc]));
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
    } else {
      // Tiles are decoded one ahead: the next tile's place (and, down, the
      // gate weight of this thread's row in it) is fetched before this tile's
      // accumulator is waited for, so the load latency hides behind this tile.
      int dec_e = 0;  // group cursor of decode_tile
      int nx_nb = 0, nx_row0 = 0, nx_rows = 0, nx_e = 0;
      float nx_w = 0.f;  // down: gate weight; F8 up: row scale
      // SUP: the tile's second pair (its block of this CTA, rows, gate weight)
      [[maybe_unused]] bool nx_two = false;
      [[maybe_unused]] int nx_row0b = 0, nx_rowsb = 0;
      [[maybe_unused]] float nx_wb = 0.f;
      auto decode_next = [&](int t) {
        int mu, gstart, gcount;
        decode_tile<MODE == kModeRouter>(t, prefix, n_groups, p.n_blocks, dec_e, nx_nb, mu);
        group_rows(p, grp_s, dec_e, gstart, gcount);
        const int mb = unit_block(p.units, mu, rank, gcount);
        nx_row0 = gstart + mb * C::BM;
        nx_rows = min(C::BM, gcount - mb * C::BM);
        nx_e = dec_e;
        if (MODE == kModeDown || MODE == kModeBwdAct || MODE == kModeDxRows)
          nx_w = r_in_tile < nx_rows ? (p.row_w ? p.row_w[nx_row0 + r_in_tile] : 1.f) : 0.f;
        if (MODE == kModeUpF8) nx_w = r_in_tile < nx_rows ? p.row_scale[nx_row0 + r_in_tile] : 0.f;
        // F8 down: the gate weight times the row's scale (the output
        // channels' scales are applied per column)
        if (MODE == kModeDownF8)
          nx_w = r_in_tile < nx_rows ? p.row_w[nx_row0 + r_in_tile] * p.row_scale[nx_row0 + r_in_tile] : 0.f;
        if constexpr (SUP == 1) {
          const int lim = super_blocks(p.units, gcount), mb2 = mb + 2;
          nx_two = 4 * mu + 2 < lim;
          nx_row0b = gstart + mb2 * C::BM;
          nx_rowsb = mb2 < lim ? min(C::BM, gcount - mb2 * C::BM) : 0;
          if (MODE == kModeDown) nx_wb = r_in_tile < nx_rowsb ? (p.row_w ? p.row_w[nx_row0b + r_in_tile] : 1.f) : 0.f;
        }
      };
      if (tau_of(0) < total_tiles) decode_next(tau_of(0));
      // router with the top-k fused: the token's best keys so far (across
      // the n-blocks of one m-unit) and whether a logit was NaN
      uint64_t best[kFusedTopk];
      bool nan_seen = false;
      for (int it = 0, tau = tau_of(0); tau < total_tiles; tau = tau_next(tau, it), ++it) {
        const int nb_t = nx_nb, row0a = nx_row0, rowsa = nx_rows, e_tile = nx_e;
        const float wra = nx_w;
        [[maybe_unused]] const int row0b = nx_row0b, rowsb = nx_rowsb;
        [[maybe_unused]] const float wrb = nx_wb;
        const int n_sub = SUP == 2 ? 2 : ((SUP == 1 && nx_two) ? 2 : 1);
        const int tau_n = tau_next(tau, it);
        if (tau_n < total_tiles) decode_next(tau_n);
        int w = 1;
        if (lane == 0)
          w = mbar_wait_bounded(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, p.status, kWaitEpiTmemFull,
                                p.timeout_ns);
        if (!__shfl_sync(0xffffffffu, w, 0)) break;
        tc_fence_after();
        // SUP: the two accumulators, columns 0.. and BN.. (super tiles: the
        // two pairs' rows; wide tiles: the same rows, n-blocks 2nb and
        // 2nb + 1); else one
#pragma unroll 1
        for (int sp = 0; sp < n_sub; ++sp) {
        const bool rows_b = SUP == 1 && sp;
        const int row0 = rows_b ? row0b : row0a, rows_valid = rows_b ? rowsb : rowsa;
        const float wr = rows_b ? wrb : wra;
        const int nb = SUP == 2 ? 2 * nb_t + sp : nb_t;
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(SUP != 0 ? sp * BN : acc * BN);
        const bool valid = r_in_tile < rows_valid;
        const int64_t row = static_cast<int64_t>(row0) + r_in_tile;
        const int warp_rows = max(0, min(32, rows_valid - ew * 32));
        const int64_t row_w0 = static_cast<int64_t>(row0) + ew * 32;
        if constexpr (MODE == kModeUp || MODE == kModeUpF8) {
          // h columns [ch*H/NCH, (ch+1)*H/NCH) of this tile; accumulator
          // columns 2j and 2j+1 hold the gate and linear branch of h column j.
          // F8: the accumulator is a sum of code products; times the row's and
          // the output channel's scale it is the product of the dequantised
          // operands.  Lane l holds the two channel scales of h column c + l.
          constexpr int H = BN / 2;
          __nv_bfloat16* dst = p.out_bf16 + row * p.out_ld + static_cast<int64_t>(nb) * H;
          const float* cs = kF8 ? p.col_scale + static_cast<int64_t>(e_tile) * p.b_rows_per_expert + nb * BN : nullptr;
#pragma unroll 1
          for (int c = ch * (H / NCH); c < (ch + 1) * (H / NCH); c += 32) {
            uint32_t a[2][32];
            tmem_ld32(taddr + 2 * c, a[0]);
            tmem_ld32(taddr + 2 * c + 32, a[1]);
            float2 sc = make_float2(1.f, 1.f);
            if constexpr (kF8) sc = *reinterpret_cast<const float2*>(cs + 2 * (c + lane));
            tc_wait_ld();
            uint32_t o[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const uint32_t* v = a[q >> 3] + 4 * (q & 7);
              float g0 = __uint_as_float(v[0]), u0 = __uint_as_float(v[1]);
              float g1 = __uint_as_float(v[2]), u1 = __uint_as_float(v[3]);
              if constexpr (kF8) {
                g0 *= wr * __shfl_sync(0xffffffffu, sc.x, 2 * q);
                u0 *= wr * __shfl_sync(0xffffffffu, sc.y, 2 * q);
                g1 *= wr * __shfl_sync(0xffffffffu, sc.x, 2 * q + 1);
                u1 *= wr * __shfl_sync(0xffffffffu, sc.y, 2 * q + 1);
              }
              const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
              const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
              o[q] = pack_bf16x2(h0, h1);
            }
            if (warp_rows > 0) store_chunk(o, nb * H + c, row_w0, warp_rows, row, dst + c);
          }
        } else if constexpr (kDown) {
          // ys = w * acc stored as fp16 (3 more mantissa bits than bf16 at the
          // same traffic); values past the fp16 range saturate and are reported
          // columns [ch*BN/NCH, (ch+1)*BN/NCH), two 32-column TMEM loads per wait.
          // amax = max |acc| over the row (NaN if any is NaN): since rounding is
          // monotonic, some |w * acc| exceeds the fp16 range iff |w| * amax does.
          __half* dst = p.out_f16 + row * p.out_ld + static_cast<int64_t>(nb) * BN;
          float amax = 0.f;
          constexpr int STEP = (BN / NCH) >= 64 ? 64 : 32;
          // DxRows adds l * col_add[e][col] (the same 32 columns for every lane:
          // broadcast loads) and checks the range of the sum
          [[maybe_unused]] float l_row = 0.f;
          [[maybe_unused]] const float* cadd = nullptr;
          if constexpr (MODE == kModeDxRows) {
            l_row = valid ? p.row_add[row] : 0.f;
            cadd = p.col_add + static_cast<int64_t>(e_tile) * p.out_ld + static_cast<int64_t>(nb) * BN;
          }
          // F8: each output column (a row of the packed W2) has its own scale;
          // the same 32 columns for every lane: broadcast loads
          [[maybe_unused]] const float* cscale = nullptr;
          if constexpr (MODE == kModeDownF8)
            cscale = p.col_scale + static_cast<int64_t>(e_tile) * p.b_rows_per_expert + static_cast<int64_t>(nb) * BN;
#pragma unroll 1
          for (int c0 = ch * (BN / NCH); c0 < (ch + 1) * (BN / NCH); c0 += STEP) {
            uint32_t v[2][32];
            tmem_ld32(taddr + c0, v[0]);
            if (STEP == 64) tmem_ld32(taddr + c0 + 32, v[1]);
            tc_wait_ld();
#pragma unroll
            for (int half = 0; half < STEP / 32; ++half) {
              uint32_t o[16];
              if constexpr (MODE == kModeDownF8) {
                const float4* cs4 = reinterpret_cast<const float4*>(cscale + c0 + 32 * half);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                  const float4 sv = __ldg(cs4 + q4);
                  const float a0 = wr * __uint_as_float(v[half][4 * q4]) * sv.x;
                  const float b0 = wr * __uint_as_float(v[half][4 * q4 + 1]) * sv.y;
                  const float a1 = wr * __uint_as_float(v[half][4 * q4 + 2]) * sv.z;
                  const float b1 = wr * __uint_as_float(v[half][4 * q4 + 3]) * sv.w;
                  amax = fmax_nan(amax, fmax_nan(fmax_nan(fabsf(a0), fabsf(b0)), fmax_nan(fabsf(a1), fabsf(b1))));
                  o[2 * q4] = pack_half2_satfinite(a0, b0);
                  o[2 * q4 + 1] = pack_half2_satfinite(a1, b1);
                }
              } else if constexpr (MODE == kModeDxRows) {
                const float4* ca = reinterpret_cast<const float4*>(cadd + c0 + 32 * half);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                  const float4 cv = __ldg(ca + q4);
                  const float a0 = fmaf(l_row, cv.x, wr * __uint_as_float(v[half][4 * q4]));
                  const float b0 = fmaf(l_row, cv.y, wr * __uint_as_float(v[half][4 * q4 + 1]));
                  const float a1 = fmaf(l_row, cv.z, wr * __uint_as_float(v[half][4 * q4 + 2]));
                  const float b1 = fmaf(l_row, cv.w, wr * __uint_as_float(v[half][4 * q4 + 3]));
                  amax = fmax_nan(amax, fmax_nan(fmax_nan(fabsf(a0), fabsf(b0)), fmax_nan(fabsf(a1), fabsf(b1))));
                  o[2 * q4] = pack_half2_satfinite(a0, b0);
                  o[2 * q4 + 1] = pack_half2_satfinite(a1, b1);
                }
              } else {
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                  const float a = __uint_as_float(v[half][2 * q]), b = __uint_as_float(v[half][2 * q + 1]);
                  amax = fmax_nan(amax, fmax_nan(fabsf(a), fabsf(b)));
                  o[q] = pack_half2_satfinite(wr * a, wr * b);
                }
              }
              const int c = c0 + 32 * half;
              if (warp_rows > 0) store_chunk(o, nb * BN + c, row_w0, warp_rows, row, dst + c);
            }
          }
          const float range = (MODE == kModeDxRows || MODE == kModeDownF8) ? amax : fabsf(wr) * amax;
          if (valid && !(range <= kHalfMax)) report_error(p.status, MOE_ERR_DEVICE_CHECK, kYsOverflow);
        } else if constexpr (MODE == kModeUpPre) {
          // the accumulator itself, (g, u) pairs of the packed W1/W3 rows, in
          // fp32, through the TMA-store boxes as 32 rows x 16 columns (64-byte rows)
          float* dst = p.out_f32 + row * p.out_ld + static_cast<int64_t>(nb) * BN;
#pragma unroll 1
          for (int c = ch * (BN / NCH); c < (ch + 1) * (BN / NCH); c += 32) {
            uint32_t v[32];
            tmem_ld32(taddr + c, v);
            tc_wait_ld();
            if (warp_rows > 0) {
              const uint32_t(&lo)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&v[0]);
              const uint32_t(&hi)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&v[16]);
              store_chunk(lo, nb * BN + c, row_w0, warp_rows, row, dst + c);
              store_chunk(hi, nb * BN + c + 16, row_w0, warp_rows, row, dst + c + 16);
            }
          }
        } else if constexpr (MODE == kModeBwdAct) {
          // Accumulator column c is dh'[r, j] = dy[t_r] . W2e[j, :] for channel
          // j = nb*BN + c (no gate weight).  With the stored pre-activations g,
          // u of that channel, s = sigmoid(g), a = g s:
          //   dh = w dh',  du = dh a,  dg = dh u s (1 + g (1 - s)),
          // written as bf16 pairs like (g, u); w h = w a u for the down weight's
          // gradient; and sum_j dh'[r, j] h[r, j], this tile's part of the
          // gate weight's gradient <dy, o> (SonicMoE's dS without the expert
          // outputs), one partial per row and n-block.
          const int64_t ld2 = 2 * p.out_ld;
          float dw_acc = 0.f;
          // 16 channels per step: 16 accumulator columns, 32 fp32
          // pre-activations (128 bytes of this thread's row)
#pragma unroll 1
          for (int c = ch * (BN / NCH); c < (ch + 1) * (BN / NCH); c += 16) {
            const int64_t j0 = static_cast<int64_t>(nb) * BN + c;
            uint32_t v[16];
            tmem_ld16(taddr + c, v);
            float4 pre[8];
            const float4* src = reinterpret_cast<const float4*>(p.pre + row * ld2 + 2 * j0);
            if (valid) {
#pragma unroll
              for (int i = 0; i < 8; ++i) pre[i] = src[i];
            }
            tc_wait_ld();
            if (valid) {
              uint32_t og[16], oh[8];
#pragma unroll
              for (int q = 0; q < 16; ++q) {
                const float g = (&pre[q >> 1].x)[2 * (q & 1)], u = (&pre[q >> 1].x)[2 * (q & 1) + 1];
                const float sg = 1.0f / (1.0f + __expf(-g));
                const float a = g * sg;
                const float h = a * u;
                const float dhu = __uint_as_float(v[q]);
                dw_acc = fmaf(dhu, h, dw_acc);
                const float dh = wr * dhu;
                og[q] = pack_bf16x2(dh * u * (sg * (1.0f + g * (1.0f - sg))), dh * a);
                if (q & 1) {
                  const float hp = __uint_as_float(oh[q >> 1]);
                  oh[q >> 1] = pack_bf16x2(hp, wr * h);
                } else {
                  oh[q >> 1] = __float_as_uint(wr * h);
                }
              }
              uint4* dg = reinterpret_cast<uint4*>(p.out_bf16 + row * ld2 + 2 * j0);
#pragma unroll
              for (int i = 0; i < 4; ++i) dg[i] = make_uint4(og[4 * i], og[4 * i + 1], og[4 * i + 2], og[4 * i + 3]);
              uint4* dhw = reinterpret_cast<uint4*>(p.out2_bf16 + row * p.out_ld + j0);
#pragma unroll
              for (int i = 0; i < 2; ++i) dhw[i] = make_uint4(oh[4 * i], oh[4 * i + 1], oh[4 * i + 2], oh[4 * i + 3]);
            }
          }
          if (valid) p.out2_f32[row * p.parts + nb * NCH + ch] = dw_acc;
        } else if constexpr (MODE == kModeRouter) {
          if (ch == 0) {
            // router (first four epilogue warps only): the three column groups
            // hold x*hi, x*mid, x*lo of the same EB experts; their fp32 sum
            // plus the bias is the logit.  With topk_k > 0 the thread also
            // takes its token's top-k over the n-blocks of its m-unit, which
            // this CTA runs in a row (the 64-bit keys of topk.cuh, kept sorted
            // by insertion), then the gate weights and the chunk histogram,
            // as topk_perm_hist_kernel does from the stored logits.
            constexpr int EB = BN / 3;
            const int e0 = nb * EB;
            float* dst = p.out_f32 + row * p.out_ld;
            if (nb == 0) {
#pragma unroll
              for (int i = 0; i < kFusedTopk; ++i) best[i] = 0;  // below every real key
              nan_seen = false;
            }
#pragma unroll 1
            for (int c = 0; c < EB; c += 16) {
              uint32_t a[16], b[16], q[16];
              tmem_ld16(taddr + c, a);
              tmem_ld16(taddr + EB + c, b);
              tmem_ld16(taddr + 2 * EB + c, q);
              tc_wait_ld();
              if (valid) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  const int ecol = e0 + c + j;
                  if (ecol < p.out_cols) {
                    float v = (__uint_as_float(a[j]) + __uint_as_float(b[j])) + __uint_as_float(q[j]);
                    if (p.bias) v += p.bias[ecol];
                    dst[ecol] = v;
                    if (p.topk_k > 0) {
                      nan_seen |= (v != v);
                      uint64_t key = topk_key(v, ecol);
#pragma unroll
                      for (int i = 0; i < kFusedTopk; ++i) {  // insert, carrying the smaller key down
                        const uint64_t hi = best[i] > key ? best[i] : key;
                        key = best[i] > key ? key : best[i];
                        best[i] = hi;
                      }
                    }
                  }
                }
              }
            }
            if (p.topk_k > 0 && valid && nb == p.n_blocks - 1) {  // the token's last expert block
              if (nan_seen) report_error(p.status, MOE_ERR_DEVICE_CHECK, static_cast<int32_t>(row));
              // softmax over the selected logits, the sum in slot order
              const float vmax = topk_key_value(best[0]);
              float ex[kFusedTopk];
              float sum = 0.f;
#pragma unroll
              for (int j = 0; j < kFusedTopk; ++j) {
                ex[j] = j < p.topk_k ? expf(topk_key_value(best[j]) - vmax) : 0.f;
                if (j < p.topk_k) sum += ex[j];
              }
#pragma unroll
              for (int j = 0; j < kFusedTopk; ++j) {
                if (j < p.topk_k) {
                  const int64_t a_ = row * p.topk_k + j;
                  const int32_t e = topk_key_expert(best[j]);
                  p.topk_idx[a_] = e;
                  p.topk_w[a_] = ex[j] / sum;
                  atomicAdd(&p.chunk_hist[static_cast<int64_t>(e) * p.nchunks + a_ / kPermChunk], 1);
                }
              }
            }
          }
        }
        }  // sub-tiles
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // the TMEM reads are complete (tcgen05.wait::ld) and nothing written
          // here is read by the MMA thread: a relaxed arrival suffices
          if (PAIR)
            mbar_arrive_cluster_relaxed(map_to_cta(smem_u32(&tempty_bar[acc]), 0));  // the even CTA's MMA waits on it
          else
            mbar_arrive(smem_u32(&tempty_bar[acc]));
        }
        if (SUP != 0) {
          acc_phase ^= 1u;
        } else {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // our TMA stores have landed before the CTA exits
    __syncwarp();
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
  // no CTA leaves while its peer may still read its operands or arrive on it
  if (PAIR) cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ----------------------------------------------------------------- host
template <int BN, int MODE, bool PAIR, int EPI, int SUP>
static int launch_gemm_epi(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const GemmParams& p, cudaStream_t stream);

// Eight epilogue warps when the K loop is short enough for the epilogue to be
// on the critical path (measured: 7B-style layer +9 %, long-K layers -2..-3 %
// with eight).
template <int BN, int MODE, bool PAIR, int SUP = 0>
static int launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const GemmParams& p,
                       cudaStream_t stream) {
  const bool wide = ((MODE == kModeUp || MODE == kModeUpF8 || MODE == kModeUpPre) && p.num_kb <= 24) ||
                    ((MODE == kModeDown || MODE == kModeDownF8 || MODE == kModeDxRows) && p.num_kb <= 8);
  if constexpr (MODE == kModeBwdAct) {
    // the SwiGLU backward's epilogue (fp32 pre-activation loads, the
    // activation's derivative) outlasts a tile's MMAs with four warps
    (void)wide;
    return launch_gemm_epi<BN, MODE, PAIR, 8, SUP>(tmA, tmB, tmC, p, stream);
  } else {
    if constexpr (MODE != kModeRouter && MODE != kModeWgrad) {
      // super tiles: eight warps drain their two accumulators before the
      // next tile's MMAs can start
      if (wide || SUP != 0) return launch_gemm_epi<BN, MODE, PAIR, 8, SUP>(tmA, tmB, tmC, p, stream);
    }
    return launch_gemm_epi<BN, MODE, PAIR, 4, SUP>(tmA, tmB, tmC, p, stream);
  }
}

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

// 2-D 16-bit tensor [outer, inner] (inner contiguous).
static bool make_map_16(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand tile: bf16 box [box_outer rows, 64], 128-byte swizzle.
static bool make_map_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  return make_map_16(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, inner, outer, 64, box_outer,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

// Operand tile of e4m3 codes: uint8 box [box_outer rows, 128], 128-byte swizzle.
static bool make_map_u8(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {128, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 output tile for the epilogue's TMA stores: box [32 rows, 16], 64-byte swizzle.
static bool make_map_out32(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {16, 32};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output tile for the epilogue's TMA stores: box [32 rows, 32], 64-byte swizzle.
static bool make_map_out(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer) {
  return make_map_16(m, dt, ptr, inner, outer, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

int num_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

// Per device, the first launch of each kernel variant sets its shared-memory
// size and finds its persistent grid (the SM pairs that can be resident at
// once); later launches, including those captured into a CUDA graph, only
// launch.
constexpr int kMaxGemmDevices = 64;

template <int BN, int MODE, bool PAIR, int EPI, int SUP>
static int launch_gemm_epi(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const GemmParams& p, cudaStream_t stream) {
  using C = GemmCfg<BN, PAIR, EPI, SUP>;
  auto kern = moe_gemm_kernel<BN, MODE, PAIR, EPI, SUP>;
  constexpr int kGemmThreads = gemm_threads(EPI);
  static int grid_of[kMaxGemmDevices] = {0};  // 0: not yet prepared on that device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxGemmDevices) return MOE_ERR_CUDA;
  if (grid_of[dev] == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
      return MOE_ERR_CUDA;
    int grid = num_sms();
    if (PAIR) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.blockDim = dim3(kGemmThreads);
      cfg.dynamicSmemBytes = C::SMEM_BYTES;
      cfg.stream = nullptr;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      // persistent: as many clusters as can be resident at once (SM pairs
      // that share a GPC), so no cluster waits for a second wave
      int clusters = 0;
      cfg.gridDim = dim3(num_sms() & ~1);
      if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
        (void)cudaGetLastError();
        clusters = num_sms() / 2;
      }
      grid = 2 * std::min(clusters, num_sms() / 2);
    }
    grid_of[dev] = grid;
  }
  if (launch_pdl(kern, grid_of[dev], kGemmThreads, C::SMEM_BYTES, stream, PAIR ? 2 : 1, tmA, tmB, tmC, p) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ row_token,
                                   const int32_t* __restrict__ offsets, int E, int d,
                                   __nv_bfloat16* __restrict__ out, int64_t rows_cap) {
  pdl_wait();
  pdl_trigger();
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
  launch_pdl(gather_rows_kernel, num_sms() * 8, 256, 0, stream, 1, x, row_token, offsets, E, d, out, rows_cap);
}

// The same copy in token order: one warp per token reads x[t] once, 4 KB at
// a time into registers, and writes it to each of the token's rows
// (tok_rows[tok_offsets[t] ..), or tok_rows[t*k ..) without offsets).  Every x
// row leaves HBM once instead of once per row it feeds.
__global__ void __launch_bounds__(256) gather_rows_by_token_kernel(const __nv_bfloat16* __restrict__ x,
                                                                   const int32_t* __restrict__ tok_rows,
                                                                   const int32_t* __restrict__ tok_offsets, int T,
                                                                   int k, int d, __nv_bfloat16* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  const int r0 = tok_offsets ? tok_offsets[t] : t * k;
  const int r1 = tok_offsets ? tok_offsets[t + 1] : r0 + k;
  if (r0 == r1) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * d);
  const int groups = d / 8;  // 16-byte groups per row
  for (int g0 = 0; g0 < groups; g0 += 8 * 32) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int g = g0 + i * 32 + lane;
      if (g < groups) v[i] = __ldg(src + g);
    }
    for (int j = r0; j < r1; ++j) {
      uint4* dst = reinterpret_cast<uint4*>(out + static_cast<int64_t>(tok_rows[j]) * d);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int g = g0 + i * 32 + lane;
        if (g < groups) dst[g] = v[i];
      }
    }
  }
}

void launch_gather_rows_by_token(const __nv_bfloat16* x, const int32_t* tok_rows, const int32_t* tok_offsets, int T,
                                 int k, int d, __nv_bfloat16* out, cudaStream_t stream) {
  launch_pdl(gather_rows_by_token_kernel, (T + 7) / 8, 256, 0, stream, 1, x, tok_rows, tok_offsets, T, k, d, out);
}

// How SM-pair GEMMs treat an expert's odd last 128-row block.  Run as a
// half-empty pair inside the main kernel, it costs one pair tile of MMA time
// but reuses the expert's weights from L2; run by a separate single-SM launch,
// it costs half that MMA time but streams those weights from HBM again.  With
// about half the experts odd, odd blocks are ~128*E/rows of all pair tiles:
// measured, half-empty pairs win at 6 % (Mixtral-style +5.5 %, 7B-style
// +1.5 %) and lose at 25 % (DeepSeek-V3-style -3.5 %).
static bool tails_in_pairs(int E, int64_t rows) { return 128.0 * E <= 0.15 * static_cast<double>(rows); }

// 256-wide SM-pair up and down GEMMs over staged rows run super tiles (two
// pairs against one B tile) when super_tiles() says so.  Odd last blocks go
// as with plain pairs: in the last unit (units 4) where they are a small
// share, else to the separate single-SM launch (units 5).  Super tiles pay where a weight slice serves few rows: they halve the
// tiles that stream each slice and cut shared-memory and TMA traffic per
// FLOP, but their epilogue no longer overlaps the next tile's MMAs.
// Measured on the same box (interleaved builds): DeepSeek-V3-style layer
// (512 rows per expert) -6.7 % with eight epilogue warps; Mixtral-style,
// skewed and 7B-class layers (2048 rows per expert) +0 .. +15 %.
static bool super_tiles(int E, int64_t rows) { return static_cast<double>(rows) <= 1024.0 * E; }

static GemmParams base_params(int32_t* status, uint64_t timeout_ns) {
  GemmParams p{};
  p.status = status;
  p.timeout_ns = timeout_ns;
  return p;
}

int launch_expert_up(const __nv_bfloat16* x, const __nv_bfloat16* W13p, const int32_t* counts,
                     const int32_t* offsets, const int32_t* row_token, const int32_t* tok_rows,
                     const int32_t* tok_offsets, __nv_bfloat16* h, int T, int d, int n, int E, int k,
                     int64_t rows_cap, int gather, __nv_bfloat16* xperm_scratch, int32_t* status,
                     uint64_t timeout_ns, cudaStream_t stream) {
  const int H = up_half_block(n);
  const int BN = 2 * H;
  CUtensorMap tmA, tmB;
  if (gather == 1) {
    if (!make_map_bf16(&tmA, x, d, T, 1)) return MOE_ERR_CUDA;
  } else if (gather == 2) {
    if (!make_map_bf16(&tmA, x, d, T, 128)) return MOE_ERR_CUDA;  // not read by the kernel
  } else {
    if (tok_rows)
      launch_gather_rows_by_token(x, tok_rows, tok_offsets, T, k, d, xperm_scratch, stream);
    else
      launch_gather_rows(x, row_token, offsets, E, d, xperm_scratch, rows_cap, stream);
    if (!make_map_bf16(&tmA, xperm_scratch, d, rows_cap, 128)) return MOE_ERR_CUDA;
  }
  const bool pair = (gather == 0 || gather == 2) && BN == 256;
  CUtensorMap tmC;
  if (!make_map_out(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, n, rows_cap)) return MOE_ERR_CUDA;
  if (!make_map_bf16(&tmB, W13p, d, static_cast<uint64_t>(E) * 2 * n, pair ? BN / 2 : BN)) return MOE_ERR_CUDA;
  GemmParams p = base_params(status, timeout_ns);
  p.counts = counts;
  p.offsets = offsets;
  p.row_token = row_token;
  p.out_bf16 = h;
  p.out_ld = n;
  p.E = E;
  p.num_kb = d / 64;
  p.n_blocks = n / H;
  p.b_rows_per_expert = 2 * n;
  p.gather = gather;
  p.x = x;
  p.lda = d;
  if (pair && gather == 0 && BN == 256 && super_tiles(E, rows_cap)) {
    if (tails_in_pairs(E, rows_cap)) {
      p.units = 4;
      return launch_gemm<256, kModeUp, true, 1>(tmA, tmB, tmC, p, stream);
    }
    p.units = 5;
    const int st = launch_gemm<256, kModeUp, true, 1>(tmA, tmB, tmC, p, stream);
    if (st != MOE_OK) return st;
    CUtensorMap tmB1;
    if (!make_map_bf16(&tmB1, W13p, d, static_cast<uint64_t>(E) * 2 * n, BN)) return MOE_ERR_CUDA;
    p.units = 2;
    return launch_gemm<256, kModeUp, false>(tmA, tmB1, tmC, p, stream);
  }
  if (pair && (gather == 0 || gather == 2) && BN == 256 && p.n_blocks % 2 == 0) {
    // wide tiles: each row block serves two n-blocks, so A reaches shared
    // memory once per two n-blocks: half the gather of A path 2, and half
    // the A traffic of staged rows.  Measured over 20 power-capped steps:
    // the 7B-class layer (n = 256, path 2) +8 %; the skewed layer (staged
    // rows) +2-3 %, with rounding +1.8 %; the Mixtral-style layer even.
    // (Super tiles, for few rows per expert, take their own branch above.)
    GemmParams pw = p;
    pw.n_blocks = p.n_blocks / 2;
    if (tails_in_pairs(E, rows_cap)) {
      pw.units = 3;
      return launch_gemm<256, kModeUp, true, 2>(tmA, tmB, tmC, pw, stream);
    }
    pw.units = 1;
    const int st = launch_gemm<256, kModeUp, true, 2>(tmA, tmB, tmC, pw, stream);
    if (st != MOE_OK) return st;
    CUtensorMap tmB1;
    if (!make_map_bf16(&tmB1, W13p, d, static_cast<uint64_t>(E) * 2 * n, BN)) return MOE_ERR_CUDA;
    p.units = 2;
    return launch_gemm<256, kModeUp, false>(tmA, tmB1, tmC, p, stream);
  }
  if (pair && tails_in_pairs(E, rows_cap)) {
    p.units = 3;
    return (BN == 256) ? launch_gemm<256, kModeUp, true>(tmA, tmB, tmC, p, stream)
                       : launch_gemm<128, kModeUp, true>(tmA, tmB, tmC, p, stream);
  }
  if (pair) {
    // complete pairs of 128-row blocks on SM pairs, then each expert's odd
    // last block on single SMs (so no pair runs half empty)
    p.units = 1;
    int st = (BN == 256) ? launch_gemm<256, kModeUp, true>(tmA, tmB, tmC, p, stream)
                         : launch_gemm<128, kModeUp, true>(tmA, tmB, tmC, p, stream);
    if (st != MOE_OK) return st;
    CUtensorMap tmB1;
    if (!make_map_bf16(&tmB1, W13p, d, static_cast<uint64_t>(E) * 2 * n, BN)) return MOE_ERR_CUDA;
    p.units = 2;
    return (BN == 256) ? launch_gemm<256, kModeUp, false>(tmA, tmB1, tmC, p, stream)
                       : launch_gemm<128, kModeUp, false>(tmA, tmB1, tmC, p, stream);
  }
  p.units = 0;
  if (BN == 256) return launch_gemm<256, kModeUp, false>(tmA, tmB, tmC, p, stream);
  return launch_gemm<128, kModeUp, false>(tmA, tmB, tmC, p, stream);
}

// e4m3 up-projection: the token-order gather quantises each x row once
// (codes and a scale per row into the workspace), then the SM-pair GEMM runs
// on the codes with kind::f8f6f4 and applies the row and channel scales in
// the SwiGLU epilogue.  n % 128 == 0 and d % 128 == 0; odd last blocks run as
// half-empty pairs.
int launch_expert_up_f8(const __nv_bfloat16* x, const uint8_t* W13q, const float* sW13, const int32_t* counts,
                        const int32_t* offsets, const int32_t* tok_rows, const int32_t* tok_offsets,
                        __nv_bfloat16* h, int T, int d, int n, int E, int k, int64_t rows_cap, uint8_t* xq_scratch,
                        float* row_scale, int32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  if (n % 128 != 0 || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
  constexpr int BN = 256;
  launch_gather_quant(x, tok_rows, tok_offsets, T, k, d, xq_scratch, row_scale, stream);
  CUtensorMap tmA, tmB, tmC;
  if (!make_map_u8(&tmA, xq_scratch, d, rows_cap, 128)) return MOE_ERR_CUDA;
  if (!make_map_u8(&tmB, W13q, d, static_cast<uint64_t>(E) * 2 * n, BN / 2)) return MOE_ERR_CUDA;
  if (!make_map_out(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, n, rows_cap)) return MOE_ERR_CUDA;
  GemmParams p = base_params(status, timeout_ns);
  p.counts = counts;
  p.offsets = offsets;
  p.out_bf16 = h;
  p.out_ld = n;
  p.E = E;
  p.num_kb = d / 128;
  p.n_blocks = n / (BN / 2);
  p.b_rows_per_expert = 2 * n;
  p.gather = 0;
  p.units = 3;
  p.row_scale = row_scale;
  p.col_scale = sW13;
  return launch_gemm<BN, kModeUpF8, true>(tmA, tmB, tmC, p, stream);
}

// e4m3 down-projection: hq [cap, n] codes with one scale per row, W2q
// [E * d, n] codes with one scale per row (output channel); the epilogue
// multiplies by the gate weight, the row's scale and each column's scale and
// stores fp16 ys as the bf16 path.  n % 128 == 0 and d % 256 == 0; odd last
// blocks run as half-empty pairs.
int launch_expert_down_f8(const uint8_t* hq, const float* h_scale, const uint8_t* W2q, const float* sW2,
                          const int32_t* counts, const int32_t* offsets, const float* row_w, __half* ys, int d,
                          int n, int E, int64_t rows_cap, int32_t* status, uint64_t timeout_ns,
                          cudaStream_t stream) {
  if (n % 128 != 0 || d % 256 != 0) return MOE_ERR_UNSUPPORTED;
  constexpr int BN = 256;
  CUtensorMap tmA, tmB, tmC;
  if (!make_map_u8(&tmA, hq, n, rows_cap, 128)) return MOE_ERR_CUDA;
  if (!make_map_u8(&tmB, W2q, n, static_cast<uint64_t>(E) * d, BN / 2)) return MOE_ERR_CUDA;
  if (!make_map_out(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ys, d, rows_cap)) return MOE_ERR_CUDA;
  GemmParams p = base_params(status, timeout_ns);
  p.counts = counts;
  p.offsets = offsets;
  p.row_w = row_w;
  p.out_f16 = ys;
  p.out_ld = d;
  p.E = E;
  p.num_kb = n / 128;
  p.n_blocks = d / BN;
  p.b_rows_per_expert = d;
  p.gather = 0;
  p.units = 3;
  p.row_scale = h_scale;
  p.col_scale = sW2;
  return launch_gemm<BN, kModeDownF8, true>(tmA, tmB, tmC, p, stream);
}

template <int MODE>
static int launch_down_like(const __nv_bfloat16* h, const __nv_bfloat16* W2p, const int32_t* counts,
                            const int32_t* offsets, const float* row_w, const float* row_add, const float* col_add,
                            __half* ys, int d, int n, int E, int64_t rows_cap, int32_t* status, uint64_t timeout_ns,
                            cudaStream_t stream) {
  const int BN = (d % 256 == 0) ? 256 : (d % 128 == 0 ? 128 : 64);
  CUtensorMap tmA, tmB;
  if (!make_map_bf16(&tmA, h, n, rows_cap, 128)) return MOE_ERR_CUDA;
  if (!make_map_bf16(&tmB, W2p, n, static_cast<uint64_t>(E) * d, BN / 2)) return MOE_ERR_CUDA;
  CUtensorMap tmC;
  if (!make_map_out(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ys, d, rows_cap)) return MOE_ERR_CUDA;
  GemmParams p = base_params(status, timeout_ns);
  p.counts = counts;
  p.offsets = offsets;
  p.row_w = row_w;
  p.row_add = row_add;
  p.col_add = col_add;
  p.out_f16 = ys;
  p.out_ld = d;
  p.E = E;
  p.num_kb = n / 64;
  p.n_blocks = d / BN;
  p.b_rows_per_expert = d;
  p.gather = 0;
  if constexpr (MODE == kModeDown) {
    if (BN == 256 && super_tiles(E, rows_cap)) {
      if (tails_in_pairs(E, rows_cap)) {
        p.units = 4;
        return launch_gemm<256, MODE, true, 1>(tmA, tmB, tmC, p, stream);
      }
      p.units = 5;
      const int st = launch_gemm<256, MODE, true, 1>(tmA, tmB, tmC, p, stream);
      if (st != MOE_OK) return st;
      CUtensorMap tmB1;
      if (!make_map_bf16(&tmB1, W2p, n, static_cast<uint64_t>(E) * d, BN)) return MOE_ERR_CUDA;
      p.units = 2;
      return launch_gemm<256, MODE, false>(tmA, tmB1, tmC, p, stream);
    }
    if (BN == 256 && p.n_blocks % 2 == 0 && p.num_kb > 32) {
      // wide tiles (two n-blocks per row block of h) where K is long enough
      // to cover their epilogue, which cannot overlap the next tile's MMAs:
      // Mixtral-style layer (K = 14336) down GEMM 4-5 % faster, the skewed
      // layer's (K = 1024) 3 % slower
      GemmParams pw = p;
      pw.n_blocks = p.n_blocks / 2;
      if (tails_in_pairs(E, rows_cap)) {
        pw.units = 3;
        return launch_gemm<256, MODE, true, 2>(tmA, tmB, tmC, pw, stream);
      }
      pw.units = 1;
      const int st = launch_gemm<256, MODE, true, 2>(tmA, tmB, tmC, pw, stream);
      if (st != MOE_OK) return st;
      CUtensorMap tmB1;
      if (!make_map_bf16(&tmB1, W2p, n, static_cast<uint64_t>(E) * d, BN)) return MOE_ERR_CUDA;
      p.units = 2;
      return launch_gemm<256, MODE, false>(tmA, tmB1, tmC, p, stream);
    }
  }
  if (tails_in_pairs(E, rows_cap)) {
    p.units = 3;
    return (BN == 256)   ? launch_gemm<256, MODE, true>(tmA, tmB, tmC, p, stream)
           : (BN == 128) ? launch_gemm<128, MODE, true>(tmA, tmB, tmC, p, stream)
                         : launch_gemm<64, MODE, true>(tmA, tmB, tmC, p, stream);
  }
  p.units = 1;
  int st = (BN == 256)   ? launch_gemm<256, MODE, true>(tmA, tmB, tmC, p, stream)
           : (BN == 128) ? launch_gemm<128, MODE, true>(tmA, tmB, tmC, p, stream)
                         : launch_gemm<64, MODE, true>(tmA, tmB, tmC, p, stream);
  if (st != MOE_OK) return st;
  CUtensorMap tmB1;
  if (!make_map_bf16(&tmB1, W2p, n, static_cast<uint64_t>(E) * d, BN)) return MOE_ERR_CUDA;
  p.units = 2;
  return (BN == 256)   ? launch_gemm<256, MODE, false>(tmA, tmB1, tmC, p, stream)
         : (BN == 128) ? launch_gemm<128, MODE, false>(tmA, tmB1, tmC, p, stream)
                       : launch_gemm<64, MODE, false>(tmA, tmB1, tmC, p, stream);
}

int launch_expert_down(const __nv_bfloat16* h, const __nv_bfloat16* W2p, const int32_t* counts,
                       const int32_t* offsets, const float* row_w, __half* ys, int d, int n, int E,
                       int64_t rows_cap, int32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  return launch_down_like<kModeDown>(h, W2p, counts, offsets, row_w, nullptr, nullptr, ys, d, n, E, rows_cap, status,
                                     timeout_ns, stream);
}

// Backward: dxr[r] = dgl[r] W13i_e^T + dL[r] Wr[:, e] (fp16), the expert
// paths' input gradient and the gate network's for each row; K = 2n.
int launch_expert_dx(const __nv_bfloat16* dgl, const __nv_bfloat16* W13i, const int32_t* counts,
                     const int32_t* offsets, const float* dl_row, const float* WrT, __half* dxr, int d, int n,
                     int E, int64_t rows_cap, int32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  return launch_down_like<kModeDxRows>(dgl, W13i, counts, offsets, nullptr, dl_row, WrT, dxr, d, 2 * n, E, rows_cap,
                                       status, timeout_ns, stream);
}

// ------------------------------------------------------------- backward
// The backward GEMMs run on SM pairs with odd last blocks as half-empty pairs
// (M-grouped ones) over the padded row layout: offsets are the padded first
// rows, counts the true row counts.

// gl[r] = xp[r] W13p_e^T: the up-projection's pre-activations (g, u) of each
// channel, interleaved as the packed weight rows, fp32 [rows_cap, 2n].
int launch_expert_up_pre(const __nv_bfloat16* xp, const __nv_bfloat16* W13p, const int32_t* counts,
                         const int32_t* offsets, float* gl, int d, int n, int E, int64_t rows_cap,
                         int32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  const int BN = (n % 128 == 0) ? 256 : 128;
  CUtensorMap tmA, tmB, tmC;
  if (!make_map_bf16(&tmA, xp, d, rows_cap, 128)) return MOE_ERR_CUDA;
  if (!make_map_bf16(&tmB, W13p, d, static_cast<uint64_t>(E) * 2 * n, BN / 2)) return MOE_ERR_CUDA;
  if (!make_map_out32(&tmC, gl, 2 * static_cast<uint64_t>(n), rows_cap)) return MOE_ERR_CUDA;
  GemmParams p = base_params(status, timeout_ns);
  p.counts = counts;
  p.offsets = offsets;
  p.out_f32 = gl;
  p.out_ld = 2 * n;
  p.E = E;
  p.num_kb = d / 64;
  p.n_blocks = 2 * n / BN;
  p.b_rows_per_expert = 2 * n;
  p.units = 3;
  return BN == 256 ? launch_gemm<256, kModeUpPre, true>(tmA, tmB, tmC, p, stream)
                   : launch_gemm<128, kModeUpPre, true>(tmA, tmB, tmC, p, stream);
}

// dh' = dyp W2_e^T (W2 as given, [E * n, d]: rows are the K-major channels),
// then the SwiGLU backward in the epilogue: dgl = (dg, du) pairs (bf16, as
// gl), hw = w h and dw_part[r, nb] = sum over the n-block of dh' h.
int launch_bwd_act(const __nv_bfloat16* dyp, const __nv_bfloat16* W2, const int32_t* counts, const int32_t* offsets,
                   const float* row_w, const float* gl, __nv_bfloat16* dgl, __nv_bfloat16* hw, float* dw_part, int d,
                   int n, int E, int64_t rows_cap, int32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  const int BN = bwd_act_block(n);
  CUtensorMap tmA, tmB;
  if (!make_map_bf16(&tmA, dyp, d, rows_cap, 128)) return MOE_ERR_CUDA;
  if (!make_map_bf16(&tmB, W2, d, static_cast<uint64_t>(E) * n, BN / 2)) return MOE_ERR_CUDA;
  GemmParams p = base_params(status, timeout_ns);
  p.counts = counts;
  p.offsets = offsets;
  p.row_w = row_w;
  p.pre = gl;
  p.out_bf16 = dgl;
  p.out2_bf16 = hw;
  p.out2_f32 = dw_part;
  p.out_ld = n;
  p.parts = bwd_act_parts(n);
  p.E = E;
  p.num_kb = d / 64;
  p.n_blocks = n / BN;
  p.b_rows_per_expert = n;
  p.units = 3;
  const CUtensorMap& tmC = tmA;  // the epilogue stores directly
  return BN == 256   ? launch_gemm<256, kModeBwdAct, true>(tmA, tmB, tmC, p, stream)
         : BN == 128 ? launch_gemm<128, kModeBwdAct, true>(tmA, tmB, tmC, p, stream)
                     : launch_gemm<64, kModeBwdAct, true>(tmA, tmB, tmC, p, stream);
}

// Weight gradient of every group: out[g] = A_g^T B_g over the group's rows,
// A [rows_cap, M] and B [rows_cap, N] row-major (read MN-major), fp32
// out[g][N][M] (or, interleaved, even M to out and odd M to out2 as
// [g][N][M/2]).  Rows past a group's count up to its padded end must be zero.
int launch_wgrad(const __nv_bfloat16* A, const __nv_bfloat16* B, const int32_t* counts, const int32_t* offsets,
                 int M, int N, int E, int64_t rows_cap, float* out, float* out2, int32_t* status,
                 uint64_t timeout_ns, cudaStream_t stream) {
  if (M % 128 != 0 || N % 64 != 0) return MOE_ERR_UNSUPPORTED;
  const bool pair = (M % 256 == 0) && (N % 128 == 0);
  const int BN = (N % 256 == 0) ? 256 : (N % 128 == 0 ? 128 : 64);
  CUtensorMap tmA, tmB;
  if (!make_map_bf16(&tmA, A, M, rows_cap, 64)) return MOE_ERR_CUDA;
  if (!make_map_bf16(&tmB, B, N, rows_cap, 64)) return MOE_ERR_CUDA;
  GemmParams p = base_params(status, timeout_ns);
  p.counts = counts;
  p.offsets = offsets;
  p.out_f32 = out;
  p.out2_f32 = out2;
  p.interleave = out2 != nullptr;
  p.out_ld = p.interleave ? M / 2 : M;
  p.out_group_stride = static_cast<int64_t>(N) * p.out_ld;
  p.E = E;
  p.num_kb = 0;
  p.n_blocks = N / BN;
  p.m_units = M / (pair ? 256 : 128);
  p.m_fast = M < N;  // sweep the narrower operand
  p.units = 0;
  const CUtensorMap& tmC = tmA;
  if (pair)
    return BN == 256 ? launch_gemm<256, kModeWgrad, true>(tmA, tmB, tmC, p, stream)
                     : launch_gemm<128, kModeWgrad, true>(tmA, tmB, tmC, p, stream);
  return BN == 256   ? launch_gemm<256, kModeWgrad, false>(tmA, tmB, tmC, p, stream)
         : BN == 128 ? launch_gemm<128, kModeWgrad, false>(tmA, tmB, tmC, p, stream)
                     : launch_gemm<64, kModeWgrad, false>(tmA, tmB, tmC, p, stream);
}

int router_expert_block(int E) { return E <= 16 ? 16 : (E <= 32 ? 32 : 64); }

int launch_router_tc(const __nv_bfloat16* x, const __nv_bfloat16* Wr3, const float* bias, float* logits, int T,
                     int d, int E, int32_t* status, uint64_t timeout_ns, cudaStream_t stream, int k,
                     int32_t* topk_idx, float* topk_w, int32_t* chunk_hist) {
  const int EB = router_expert_block(E);
  const int BN = 3 * EB;
  const int nblk = (E + EB - 1) / EB;
  // SM pairs: each CTA holds half of the 3*EB split-weight rows, so a k-block
  // moves 28 KB per SM instead of 40 KB through shared memory
  CUtensorMap tmA, tmB;
  if (!make_map_bf16(&tmA, x, d, T, 128)) return MOE_ERR_CUDA;
  if (!make_map_bf16(&tmB, Wr3, d, static_cast<uint64_t>(nblk) * BN, BN / 2)) return MOE_ERR_CUDA;
  const CUtensorMap& tmC = tmA;  // the router epilogue stores fp32 logits directly
  GemmParams p = base_params(status, timeout_ns);
  p.single_rows = T;
  p.bias = bias;
  p.out_f32 = logits;
  p.out_ld = E;
  p.out_cols = E;
  p.E = 1;
  p.num_kb = d / 64;
  p.n_blocks = nblk;
  p.b_rows_per_expert = 0;
  p.gather = 0;
  p.units = 3;  // pairs of 128-row blocks; an odd last block runs as a half-empty pair
  if (k > 0) {
    if (!router_fuses_topk(E, k) || !topk_idx || !topk_w || !chunk_hist) return MOE_ERR_INVALID;
    p.topk_k = k;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.chunk_hist = chunk_hist;
    p.nchunks = static_cast<int>(perm_num_chunks(static_cast<int64_t>(T) * k));
  }
  if (BN == 48) return launch_gemm<48, kModeRouter, true>(tmA, tmB, tmC, p, stream);
  if (BN == 96) return launch_gemm<96, kModeRouter, true>(tmA, tmB, tmC, p, stream);
  return launch_gemm<192, kModeRouter, true>(tmA, tmB, tmC, p, stream);
}

// Wr [d, E] fp32 -> Wr3 [nblk * 3EB, d] bf16: for expert block b, rows
// 3EB*b + g*EB + c hold part g (hi, mid, lo) of column e = EB*b + c, where
// hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid); both differences
// are exact in fp32, so hi + mid + lo equals w to within 2^-27 |w|.  Columns
// past E are zero.
__global__ void split_router_kernel(const float* __restrict__ Wr, __nv_bfloat16* __restrict__ Wr3, int d, int E,
                                    int EB, int nblk, int32_t* zero, int64_t zero_count) {
  pdl_wait();
  pdl_trigger();
  // the counts of the fused top-k + histogram kernel that follows
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < zero_count;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    zero[i] = 0;
  const int64_t total = static_cast<int64_t>(nblk) * EB * d;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int k = static_cast<int>(i % d);
    const int col = static_cast<int>(i / d);  // expert slot 0 .. nblk*EB-1
    const int b = col / EB, c = col % EB;
    const float w = (col < E) ? Wr[static_cast<int64_t>(k) * E + col] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    const int64_t rbase = static_cast<int64_t>(b) * 3 * EB + c;
    Wr3[(rbase + 0 * EB) * d + k] = hi;
    Wr3[(rbase + 1 * EB) * d + k] = mid;
    Wr3[(rbase + 2 * EB) * d + k] = lo;
  }
}

size_t router_split_elems(int d, int E) {
  const int EB = router_expert_block(E);
  const int nblk = (E + EB - 1) / EB;
  return static_cast<size_t>(nblk) * 3 * EB * d;
}

void launch_split_router(const float* Wr, __nv_bfloat16* Wr3, int d, int E, cudaStream_t stream, int32_t* zero,
                         int64_t zero_count) {
  const int EB = router_expert_block(E);
  const int nblk = (E + EB - 1) / EB;
  const int64_t total = static_cast<int64_t>(nblk) * EB * d;
  const int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, num_sms() * 16));
  launch_pdl(split_router_kernel, blocks, 256, 0, stream, 1, Wr, Wr3, d, E, EB, nblk, zero, zero_count);
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
