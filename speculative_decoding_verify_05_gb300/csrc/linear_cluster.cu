// Split-K verify GEMM for layers with few weight tiles (cluster variant).
//
// S CTAs of one thread-block cluster share a (128 weight rows x TN tokens) tile:
// CTA rank r runs the k-steps [r kt / S, (r + 1) kt / S) through the same
// TMA -> tcgen05.mma -> TMEM pipeline as the persistent kernel.  Token columns
// are dealt out in groups of 4 ("chunks"), CPR consecutive chunks per rank.
// Once every CTA of the cluster is past its main loop (cluster barrier), each
// CTA pushes every chunk of its fp32 accumulator straight into the owning
// rank's shared-memory ring (idle by then) with 16-byte remote stores, at slot
// [its rank]; after a second barrier each rank sums the S slots of its chunks
// in rank order (deterministic, local reads only), adds the residual and
// stores bf16.
// No partial sum leaves the chip and no second kernel is needed, which is what
// the 4096- and 6144-row projections want: their 32-48 tiles would otherwise be
// cut into 3-5 pieces per tile that travel through L2 twice.
#include "internal.h"
#include "linear_tc.cuh"
#include "split_k_exchange.cuh"

namespace spec {
namespace {

constexpr int MAX_S = 8;
// warps 0 (TMA) and 1 (MMA) run the main loop; after it all 8 warps move the accumulator: warp w
// reads TMEM lane quarter w % 4, half w / 4 of the columns (more warps issue the
// distributed-shared-memory stores faster; the exchange is bound by those stores)
constexpr int CL_THREADS = 256;

template <int BN, int NSUB>
__global__ void __launch_bounds__(CL_THREADS, 1)
linear_cluster_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                      const LinearArgs args, int S, int cpr) {
  using Cfg = LinearCfg<BN, NSUB>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int TN = Cfg::TN;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
  // after the main loop: slots [S][cpr chunks][128 rows] of float4 for this rank's chunks
  float4* slots = reinterpret_cast<float4*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  // a cluster is S consecutive blocks; tiles start at args.dp_tiles (the tiles before it are whole
  // tiles of a persistent launch that ran first)
  const int tile = (int)args.dp_tiles + blockIdx.x / S;
  const int kt = args.k_tiles;
  const int k0 = (int)((long long)kt * rank / S), k1 = (int)((long long)kt * (rank + 1) / S);
  const int m_t = tile % args.tiles_m, n_t = tile / args.tiles_m;

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
  if (warp == 1) tmem_alloc(tmem_slot, Cfg::ACC_COLS < 32 ? 32 : Cfg::ACC_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // shared-memory and TMEM setup above overlaps the previous kernel, and so do the first stages'
  // weight loads when W is not that kernel's output; everything else in global memory only below
  const int n_early = args.w_early ? min(STAGES, k1 - k0) : 0;
  const uint64_t pol = l2_policy_evict_first();
  if (warp == 0 && lane == 0)
    for (int i = 0; i < n_early; ++i) {
      mbar_arrive_expect_tx(&full[i], Cfg::STAGE_BYTES);
      tma_load_2d_hint(sA + i * Cfg::A_BYTES, &tm_w, &full[i], (k0 + i) * LIN_BK, n_t * 128, pol);
    }
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    // ---------------- TMA producer over this rank's k-steps
    if (lane == 0) {
      for (int k = k0; k < k1; ++k) {
        const int i = k - k0, s = i % STAGES;
        if (i >= STAGES && !mbar_wait(&empty[s], (uint32_t)((i / STAGES - 1) & 1), args.status, 0x141u)) break;
        if (i >= n_early) {
          mbar_arrive_expect_tx(&full[s], Cfg::STAGE_BYTES);
          tma_load_2d_hint(sA + s * Cfg::A_BYTES, &tm_w, &full[s], k * LIN_BK, n_t * 128, pol);
        }
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub)
          tma_load_2d(sB + s * Cfg::B_BYTES + sub * BN * LIN_ROW_BYTES, &tm_x, &full[s], k * LIN_BK, m_t * TN + sub * BN);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer: one accumulator for the whole k-range
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(128, BN);
      for (int k = k0; k < k1; ++k) {
        const int i = k - k0, s = i % STAGES;
        if (!mbar_wait(&full[s], (uint32_t)((i / STAGES) & 1), args.status, 0x142u)) break;
        tc_fence_after();
        const uint32_t a = smem_u32(sA + s * Cfg::A_BYTES);
        const uint32_t b = smem_u32(sB + s * Cfg::B_BYTES);
#pragma unroll
        for (int kk = 0; kk < LIN_BK / 16; ++kk)
#pragma unroll
          for (int sub = 0; sub < NSUB; ++sub)
            umma_bf16(tmem + sub * BN, umma_desc_lin(a + kk * 32), umma_desc_lin(b + sub * BN * LIN_ROW_BYTES + kk * 32),
                      idesc, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&empty[s]);
      }
      // completes once every MMA above has (also when the range is empty)
      umma_commit(acc_full);
    }
    __syncwarp();
  } else if (args.norm_ssq) {
    // warps 2-7 are idle during the main loop: the row scales of a folded RMSNorm (made visible to
    // the whole CTA by the cluster barriers below)
    fill_row_scales(args, reinterpret_cast<float*>(smem + Cfg::RMS_OFF), split_first_row<TN>(cpr, (int)rank, m_t),
                    split_rows<TN>(cpr, (int)rank), threadIdx.x - 64, CL_THREADS - 64);
  }
  // every CTA of the cluster is past its main loop: the rings are free
  const bool ok = mbar_wait(acc_full, 0u, args.status, 0x143u);
  tc_fence_after();
  cluster_sync_all();
  push_accumulator<TN>(tmem, warp, lane, k1 > k0 && ok, slots, cpr, (int)rank, 1, 0);
  tc_fence_before();
  // every piece has landed in its owner's slots
  cluster_sync_all();

  split_sum_epilogue<TN, CL_THREADS>(slots, args, S, cpr, (int)rank, n_t, m_t,
                                     reinterpret_cast<float*>(smem + Cfg::RMS_OFF));
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::ACC_COLS < 32 ? 32 : Cfg::ACC_COLS);
  }
}

template <int BN, int NSUB>
struct ClusterLaunch {
  static constexpr int smem() { return LinearCfg<BN, NSUB>::SMEM_BYTES; }
  static bool configure(int dev) {
    static bool configured[64] = {};
    if (dev >= 0 && dev < 64 && configured[dev]) return true;
    if (cudaFuncSetAttribute(linear_cluster_kernel<BN, NSUB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem()) != cudaSuccess)
      return false;
    if (dev >= 0 && dev < 64) configured[dev] = true;
    return true;
  }
  static cudaLaunchConfig_t config(int grid, int S, cudaStream_t st, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(CL_THREADS);
    cfg.dynamicSmemBytes = smem();
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cfg;
  }
  static int capacity(int S) {
    using Cfg = LinearCfg<BN, NSUB>;
    const int cpr = (Cfg::TN / 4 + S - 1) / S;
    if ((long long)S * cpr * 128 * 16 > (long long)Cfg::STAGES * Cfg::STAGE_BYTES) return 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configure(dev)) return 0;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = config(S * 64, S, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)linear_cluster_kernel<BN, NSUB>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n * S;
  }
  static cudaError_t launch(const CUtensorMap& tw, const CUtensorMap& tx, const LinearArgs& a, int S,
                            int tiles, cudaStream_t st) {
    const int cpr = (LinearCfg<BN, NSUB>::TN / 4 + S - 1) / S;
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configure(dev)) return cudaGetLastError();
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = config(tiles * S, S, st, attr);
    return cudaLaunchKernelEx(&cfg, linear_cluster_kernel<BN, NSUB>, tw, tx, a, S, cpr);
  }
};

}  // namespace

// Tile shapes with a cluster build: the accumulator (TN x 128 fp32) must fit in the ring.
#define SPEC_CLUSTER_SHAPES(X) \
  X(1, 16) X(1, 32) X(1, 48) X(1, 64) X(1, 80) X(1, 96) X(1, 112) X(1, 128) X(1, 144) X(1, 160) X(1, 176) \
  X(1, 192) \
  X(1, 208) X(1, 224) X(1, 240) X(1, 256) X(2, 144) X(2, 160) X(2, 176) X(2, 192)

int linear_cluster_capacity(int BN, int NSUB, int S) {
  if (S < 2 || S > MAX_S) return 0;
  static int cache[64][3][17][MAX_S + 1];   // [device][NSUB][BN / 16][S], 0 = not asked yet
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cacheable = dev >= 0 && dev < 64 && NSUB <= 2 && BN % 16 == 0 && BN / 16 <= 16;
  if (cacheable && cache[dev][NSUB][BN / 16][S] != 0) return cache[dev][NSUB][BN / 16][S] - 1;
  int cap = 0;
  switch (NSUB * 1000 + BN) {
#define X(ns, bn) \
  case ns * 1000 + bn: cap = ClusterLaunch<bn, ns>::capacity(S); break;
    SPEC_CLUSTER_SHAPES(X)
#undef X
    default: cap = 0;
  }
  if (cacheable) cache[dev][NSUB][BN / 16][S] = cap + 1;
  return cap;
}

cudaError_t launch_linear_cluster(int BN, int NSUB, const CUtensorMap& tw, const CUtensorMap& tx,
                                  const LinearArgs& a, int S, int tiles, cudaStream_t s) {
  switch (NSUB * 1000 + BN) {
#define X(ns, bn) \
  case ns * 1000 + bn: return ClusterLaunch<bn, ns>::launch(tw, tx, a, S, tiles, s);
    SPEC_CLUSTER_SHAPES(X)
#undef X
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spec
