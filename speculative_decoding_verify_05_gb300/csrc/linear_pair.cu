// Split-K verify GEMM on CTA pairs (tcgen05.mma.cta_group::2) for the verify linears at a few
// hundred rows.
//
// At M = 368 the tensor core of one SM is fed from shared memory: each 128 x 384 x 64 k-step of the
// one-SM kernels moves a 16 KB weight tile and a 48 KB token tile through the TMA into shared
// memory and reads 80 KB back into the MMAs, more than the shared-memory port delivers while the
// MMAs run.  The 2-SM MMA computes a 256-row weight tile on a pair of SMs: each CTA stages its own
// 128 weight rows and HALF of the token rows of every MMA, and the pair's tensor cores exchange the
// token halves, so each SM moves 40 KB in and 56 KB out per k-step.
//
// A thread-block cluster of 2S CTAs holds S pairs; pair p runs the k-steps [p kt / S, (p + 1) kt / S)
// of one 256-row pair tile.  The even CTA of a pair issues the MMAs and commits their completion to
// both CTAs' barriers; both CTAs' TMA loads complete on the even CTA's barrier.  After the main loop
// the S CTAs that hold the same 128 weight rows (one per pair) sum their pieces through distributed
// shared memory in pair order (deterministic) and run the epilogue (bf16 + residual, SwiGLU, RoPE).
#include "internal.h"
#include "linear_tc.cuh"
#include "split_k_exchange.cuh"

namespace spec {
namespace {

constexpr int PR_THREADS = 256;
constexpr int PR_MAX_S = 4;        // pairs per cluster (portable cluster size 8)

template <int BN, int NSUB>
struct PairCfg {
  static constexpr int TN = BN * NSUB;                       // token rows of the tile
  static constexpr int HB = BN / 2;                          // token rows per CTA and MMA
  static constexpr int A_BYTES = 128 * LIN_ROW_BYTES;
  static constexpr int B_BYTES = NSUB * HB * LIN_ROW_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES_FIT = (200 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 12 ? 12 : STAGES_FIT;
  static constexpr int TMEM_COLS = TN <= 32 ? 32 : TN <= 64 ? 64 : TN <= 128 ? 128 : TN <= 256 ? 256 : 512;
  static constexpr int RMS_OFF = STAGES * STAGE_BYTES + 1024;      // row scales of a folded RMSNorm
  static constexpr int SMEM_BYTES = RMS_OFF + TN * 4 + 1024;
};

template <int BN, int NSUB>
__global__ void __launch_bounds__(PR_THREADS, 1)
linear_pair_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                   const LinearArgs args, int S, int cpr) {
  using Cfg = PairCfg<BN, NSUB>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int TN = Cfg::TN;
  constexpr int HB = Cfg::HB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
  float4* slots = reinterpret_cast<float4*>(smem);   // after the main loop: [S][cpr][128] float4
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int half = (int)(rank & 1u), pr = (int)(rank >> 1);
  const uint32_t leader = rank & ~1u, peer = rank ^ 1u;
  // pair tile (256 weight rows x TN tokens): args.dp_tiles is the first pair tile of this launch
  const int tile = (int)args.dp_tiles + blockIdx.x / (2 * S);
  const int kt = args.k_tiles;
  const int k0 = (int)((long long)kt * pr / S), k1 = (int)((long long)kt * (pr + 1) / S);
  const int m_t = tile % args.tiles_m;
  const int n_t = (tile / args.tiles_m) * 2 + half;       // this CTA's 128-row weight tile

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  // the peer's TMA completes on this pair's barriers and the even CTA commits to the odd one's:
  // every barrier of the cluster is initialised first
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs): own 128 weight rows, own half of each MMA's tokens
    if (lane == 0) {
      const uint32_t full_leader = dsmem_map(smem_u32(full), leader);
      for (int k = k0; k < k1; ++k) {
        const int i = k - k0, s = i % STAGES;
        if (i >= STAGES && !mbar_wait(&empty[s], (uint32_t)((i / STAGES - 1) & 1), args.status, 0x171u)) break;
        if (half == 0) mbar_arrive_expect_tx(&full[s], 2 * Cfg::STAGE_BYTES);
        const uint32_t bar = full_leader + (uint32_t)s * 8u;
        tma_load_2d_pair_hint(sA + s * Cfg::A_BYTES, &tm_w, bar, k * LIN_BK, n_t * 128, l2_policy_evict_first());
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub)
          tma_load_2d_pair(sB + s * Cfg::B_BYTES + sub * HB * LIN_ROW_BYTES, &tm_x, bar, k * LIN_BK,
                           m_t * TN + sub * BN + half * HB);
      }
    }
    __syncwarp();
  } else if (warp == 1 && half == 0) {
    // ---------------- MMA issuer (even CTA): M = 256 over the pair, N = BN per MMA
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(256, BN);
      const uint32_t empty_peer = dsmem_map(smem_u32(empty), peer);
      for (int k = k0; k < k1; ++k) {
        const int i = k - k0, s = i % STAGES;
        if (!mbar_wait(&full[s], (uint32_t)((i / STAGES) & 1), args.status, 0x172u)) break;
        tc_fence_after();
        const uint32_t a = smem_u32(sA + s * Cfg::A_BYTES);
        const uint32_t b = smem_u32(sB + s * Cfg::B_BYTES);
#pragma unroll
        for (int kk = 0; kk < LIN_BK / 16; ++kk)
#pragma unroll
          for (int sub = 0; sub < NSUB; ++sub)
            umma_bf16_pair(tmem + sub * BN, umma_desc_lin(a + kk * 32),
                           umma_desc_lin(b + sub * HB * LIN_ROW_BYTES + kk * 32), idesc, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit_pair(smem_u32(&empty[s]));
        umma_commit_pair(empty_peer + (uint32_t)s * 8u);
      }
      umma_commit_pair(smem_u32(acc_full));
      umma_commit_pair(dsmem_map(smem_u32(acc_full), peer));
    }
    __syncwarp();
  } else if (warp >= 2 && args.norm_ssq) {
    // warps 2-7 are idle during the main loop: the row scales of a folded RMSNorm (made visible to
    // the whole CTA by the cluster barriers below)
    fill_row_scales(args, reinterpret_cast<float*>(smem + Cfg::RMS_OFF), split_first_row<TN>(cpr, pr, m_t),
                    split_rows<TN>(cpr, pr), threadIdx.x - 64, PR_THREADS - 64);
  }
  const bool ok = mbar_wait(acc_full, 0u, args.status, 0x173u);
  tc_fence_after();
  if (S == 1 && args.epi == EPI_SWIGLU) {
    // one pair per tile, nothing to sum: the SwiGLU epilogue straight from TMEM, each warp through
    // a transpose block in its CTA's ring (free: the pair's MMAs, the only readers, have completed)
    __syncthreads();   // (the row scales written by warps 2-7)
    if (ok && n_t < args.tiles_n)
      tmem_swiglu_epilogue<TN>(tmem, warp, lane, args, m_t, n_t,
                               args.norm_ssq ? reinterpret_cast<const float*>(smem + Cfg::RMS_OFF) : nullptr,
                               reinterpret_cast<float*>(smem));
    tc_fence_before();
    cluster_sync_all();   // both CTAs done with their TMEM before the pair frees it
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem, Cfg::TMEM_COLS);
    }
    return;
  }
  // every CTA of the cluster is past its main loop: the rings are free
  cluster_sync_all();
  // the S CTAs holding the same weight rows (ranks half, half + 2, ...) exchange their pieces
  push_accumulator<TN>(tmem, warp, lane, k1 > k0 && ok, slots, cpr, pr, 2, half);
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, Cfg::TMEM_COLS);
  }
  if (n_t < args.tiles_n)
    split_sum_epilogue<TN, PR_THREADS>(slots, args, S, cpr, pr, n_t, m_t, reinterpret_cast<float*>(smem + Cfg::RMS_OFF));
}

template <int BN, int NSUB>
struct PairLaunch {
  static bool configure(int dev) {
    static bool configured[64] = {};
    if (dev >= 0 && dev < 64 && configured[dev]) return true;
    if (cudaFuncSetAttribute(linear_pair_kernel<BN, NSUB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PairCfg<BN, NSUB>::SMEM_BYTES) != cudaSuccess)
      return false;
    if (dev >= 0 && dev < 64) configured[dev] = true;
    return true;
  }
  static cudaLaunchConfig_t config(int grid, int cl, cudaStream_t st, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(PR_THREADS);
    cfg.dynamicSmemBytes = PairCfg<BN, NSUB>::SMEM_BYTES;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cfg;
  }
  static int cpr(int S) { return (PairCfg<BN, NSUB>::TN / 4 + S - 1) / S; }
  // CTAs that can be resident at once in clusters of S pairs (0: the slots do not fit, or none)
  static int capacity(int S) {
    using Cfg = PairCfg<BN, NSUB>;
    if ((long long)S * cpr(S) * 128 * 16 > (long long)Cfg::STAGES * Cfg::STAGE_BYTES) return 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configure(dev)) return 0;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = config(2 * S * 32, 2 * S, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)linear_pair_kernel<BN, NSUB>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n * 2 * S;
  }
  static cudaError_t launch(const CUtensorMap& tw, const CUtensorMap& tx, const LinearArgs& a, int S, int pair_tiles,
                            cudaStream_t st) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configure(dev)) return cudaGetLastError();
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = config(pair_tiles * 2 * S, 2 * S, st, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, linear_pair_kernel<BN, NSUB>, tw, tx, a, S, cpr(S));
    return e != cudaSuccess ? e : cudaGetLastError();
  }
};

}  // namespace

// Tile shapes with a pair build (BN = token rows per MMA, NSUB MMAs per k-step).
#define SPEC_PAIR_SHAPES(X) \
  X(1, 64) X(1, 96) X(1, 128) X(1, 160) X(1, 192) X(1, 224) X(1, 256) \
  X(2, 144) X(2, 160) X(2, 176) X(2, 192)

int linear_pair_capacity(int BN, int NSUB, int S) {
  if (S < 1 || S > PR_MAX_S) return 0;
  static int cache[64][3][17][PR_MAX_S + 1];   // [device][NSUB][BN / 16][S]: CTAs + 1, 0 = not asked
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cacheable = dev >= 0 && dev < 64 && NSUB <= 2 && BN % 16 == 0 && BN / 16 <= 16;
  if (cacheable && cache[dev][NSUB][BN / 16][S] != 0) return cache[dev][NSUB][BN / 16][S] - 1;
  int cap = 0;
  switch (NSUB * 1000 + BN) {
#define X(ns, bn) \
  case ns * 1000 + bn: cap = PairLaunch<bn, ns>::capacity(S); break;
    SPEC_PAIR_SHAPES(X)
#undef X
    default: cap = 0;
  }
  if (cacheable) cache[dev][NSUB][BN / 16][S] = cap + 1;
  return cap;
}

cudaError_t launch_linear_pair(int BN, int NSUB, const CUtensorMap& tw, const CUtensorMap& tx, const LinearArgs& a,
                               int S, int pair_tiles, cudaStream_t s) {
  switch (NSUB * 1000 + BN) {
#define X(ns, bn) \
  case ns * 1000 + bn: return PairLaunch<bn, ns>::launch(tw, tx, a, S, pair_tiles, s);
    SPEC_PAIR_SHAPES(X)
#undef X
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spec
