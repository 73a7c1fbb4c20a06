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

namespace spec {
namespace {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster (release / acquire on shared memory).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t dsmem_map(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void dsmem_st_f4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void smem_st_f4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

constexpr int MAX_S = 8;
// warps 0 (TMA) and 1 (MMA) run the main loop; after it all 8 warps move the accumulator: warp w
// reads TMEM lane quarter w % 4, half w / 4 of the columns (more warps issue the
// distributed-shared-memory stores faster; the exchange is bound by those stores)
constexpr int CL_THREADS = 256;

// Slot row of weight row r: rows are XOR-swizzled inside each group of 8 so that threads
// reading 8 consecutive rows each (rows 8t + i, t = 0..7) hit 8 different bank groups.
__device__ __forceinline__ int slot_row(int r) { return r ^ ((r >> 3) & 7); }

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
  // shared-memory and TMEM setup above overlaps the previous kernel; global memory only below
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    // ---------------- TMA producer over this rank's k-steps
    if (lane == 0) {
      for (int k = k0; k < k1; ++k) {
        const int i = k - k0, s = i % STAGES;
        if (i >= STAGES && !mbar_wait(&empty[s], (uint32_t)((i / STAGES - 1) & 1), args.status, 0x141u)) break;
        mbar_arrive_expect_tx(&full[s], Cfg::STAGE_BYTES);
        tma_load_2d(sA + s * Cfg::A_BYTES, &tm_w, &full[s], k * LIN_BK, n_t * 128);
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
  }
  // every CTA of the cluster is past its main loop: the rings are free
  const int q = warp & 3;
  const int row = q * 32 + lane;
  const bool ok = mbar_wait(acc_full, 0u, args.status, 0x143u);
  tc_fence_after();
  cluster_sync_all();
  {
    // ---------------- every warp (TMEM lane quarter warp % 4, column half warp / 4): push each
    // 4-column chunk to its rank
    const uint32_t t_row = tmem + (uint32_t(q * 32) << 16);
    const uint32_t base = smem_u32(slots);
    constexpr int C_MID = TN / 32 * 16;
    const int c_lo = warp < 4 ? 0 : C_MID, c_hi = warp < 4 ? C_MID : TN;
    // 64 columns per TMEM wait (16, 32 or 48 at the ends: both halves are multiples of 16), then
    // their remote stores back to back
#pragma unroll 1
    for (int c = c_lo; c < c_hi; c += 64) {
      float v[64];
      const int cols = c_hi - c < 64 ? c_hi - c : 64;
      if (k1 > k0 && ok) {
        if (cols == 64) tmem_ld_cols<64>(t_row + c, v);
        else if (cols == 48) tmem_ld_cols<48>(t_row + c, v);
        else if (cols == 32) tmem_ld_cols<32>(t_row + c, v);
        else tmem_ld_cols<16>(t_row + c, v);
      } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        if (4 * e >= cols) break;
        const int chunk = c / 4 + e;
        const int owner = chunk / cpr, kk = chunk - owner * cpr;
        const uint32_t off = (uint32_t)(((rank * cpr + kk) * 128 + slot_row(row)) * 16);
        // (this rank's own chunks take the plain shared-memory store: the cluster path is as slow
        // for a local address as for a peer's)
        if (owner == (int)rank) smem_st_f4(base + off, v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        else dsmem_st_f4(dsmem_map(base + off, (uint32_t)owner), v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
      }
    }
    tc_fence_before();
  }
  // every piece has landed in its owner's slots
  cluster_sync_all();

  // ---------------- this rank's chunks: sum the S slots in rank order, add the residual, store.
  // Item = (chunk, 8 consecutive weight rows): 4 tokens x 8 rows, so the residual and Y move
  // in 16-byte pieces (8 bf16 of one token row).
  const int n_chunks = min(cpr, TN / 4 - (int)rank * cpr);
  if (args.epi == EPI_SWIGLU) {
    // gate and up rows interleaved per 16: item = (chunk, 8 gate rows r8..r8+7 with r8 % 32 < 16);
    // the matching up rows are r8+16..; 8 outputs per token at column n_t 64 + (r8 / 32) 16 + r8 % 32
    const int sitems = (n_chunks > 0 ? n_chunks : 0) * 8;
    for (int it = threadIdx.x; it < sitems; it += CL_THREADS) {
      const int kk = it >> 3, q8 = it & 7, r8 = (q8 >> 1) * 32 + (q8 & 1) * 8;
      float g[8][4], u[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 vg = slots[kk * 128 + slot_row(r8 + i)];
        const float4 vu = slots[kk * 128 + slot_row(r8 + 16 + i)];
        g[i][0] = vg.x; g[i][1] = vg.y; g[i][2] = vg.z; g[i][3] = vg.w;
        u[i][0] = vu.x; u[i][1] = vu.y; u[i][2] = vu.z; u[i][3] = vu.w;
      }
      for (int s2 = 1; s2 < S; ++s2) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 vg = slots[(s2 * cpr + kk) * 128 + slot_row(r8 + i)];
          const float4 vu = slots[(s2 * cpr + kk) * 128 + slot_row(r8 + 16 + i)];
          g[i][0] += vg.x; g[i][1] += vg.y; g[i][2] += vg.z; g[i][3] += vg.w;
          u[i][0] += vu.x; u[i][1] += vu.y; u[i][2] += vu.z; u[i][3] += vu.w;
        }
      }
      const int n = n_t * 64 + (r8 >> 5) * 16 + (r8 & 31);
      const int mb = m_t * TN + ((int)rank * cpr + kk) * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (mb + e >= args.M) break;
        uint32_t o4[4];
#pragma unroll
        for (int h = 0; h < 4; ++h)
          o4[h] = pack_bf16x2(silu(g[2 * h][e]) * u[2 * h][e], silu(g[2 * h + 1][e]) * u[2 * h + 1][e]);
        *reinterpret_cast<uint4*>(args.Y + (size_t)(mb + e) * args.ldy + n) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
    }
  }
  // RoPE heads: item = (chunk, 8 dims r8..r8+7 of the first half); the pair dims r8+64.. rotate
  // with them: (a, b) -> (a c - b s, b c + a s), c, s from row m's table entry for dim r8 + i
  const bool rope = args.epi == EPI_ROPE && n_t < args.rope_tiles;
  if (rope) {
    const int ritems = (n_chunks > 0 ? n_chunks : 0) * 8;
    for (int it = threadIdx.x; it < ritems; it += CL_THREADS) {
      const int kk = it >> 3, r8 = (it & 7) * 8;
      float a[8][4], b[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 va = slots[kk * 128 + slot_row(r8 + i)];
        const float4 vb = slots[kk * 128 + slot_row(r8 + 64 + i)];
        a[i][0] = va.x; a[i][1] = va.y; a[i][2] = va.z; a[i][3] = va.w;
        b[i][0] = vb.x; b[i][1] = vb.y; b[i][2] = vb.z; b[i][3] = vb.w;
      }
      for (int s2 = 1; s2 < S; ++s2) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 va = slots[(s2 * cpr + kk) * 128 + slot_row(r8 + i)];
          const float4 vb = slots[(s2 * cpr + kk) * 128 + slot_row(r8 + 64 + i)];
          a[i][0] += va.x; a[i][1] += va.y; a[i][2] += va.z; a[i][3] += va.w;
          b[i][0] += vb.x; b[i][1] += vb.y; b[i][2] += vb.z; b[i][3] += vb.w;
        }
      }
      const int n = n_t * 128 + r8;
      const int mb = m_t * TN + ((int)rank * cpr + kk) * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = mb + e;
        if (m >= args.M) break;
        const float2* cs = args.rope_cs + (size_t)m * 64 + r8;
        uint32_t x4[4], y4[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 c0 = cs[2 * h], c1 = cs[2 * h + 1];
          const float a0 = a[2 * h][e], a1 = a[2 * h + 1][e], b0 = b[2 * h][e], b1 = b[2 * h + 1][e];
          x4[h] = pack_bf16x2(a0 * c0.x - b0 * c0.y, a1 * c1.x - b1 * c1.y);
          y4[h] = pack_bf16x2(b0 * c0.x + a0 * c0.y, b1 * c1.x + a1 * c1.y);
        }
        *reinterpret_cast<uint4*>(args.Y + (size_t)m * args.ldy + n) = make_uint4(x4[0], x4[1], x4[2], x4[3]);
        *reinterpret_cast<uint4*>(args.Y + (size_t)m * args.ldy + n + 64) = make_uint4(y4[0], y4[1], y4[2], y4[3]);
      }
    }
  }
  const int items = (args.epi == EPI_SWIGLU || rope || n_chunks <= 0) ? 0 : n_chunks * 16;
  for (int it = threadIdx.x; it < items; it += CL_THREADS) {
    const int kk = it >> 4, r8 = (it & 15) * 8;
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = slots[kk * 128 + slot_row(r8 + i)];
      acc[i][0] = v.x; acc[i][1] = v.y; acc[i][2] = v.z; acc[i][3] = v.w;
    }
    for (int s2 = 1; s2 < S; ++s2) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = slots[(s2 * cpr + kk) * 128 + slot_row(r8 + i)];
        acc[i][0] += v.x; acc[i][1] += v.y; acc[i][2] += v.z; acc[i][3] += v.w;
      }
    }
    const int n0 = n_t * 128 + r8;
    const int mb = m_t * TN + ((int)rank * cpr + kk) * 4;
    if (n0 + 8 <= args.N) {
      uint4 res[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        res[e] = (args.residual && mb + e < args.M)
                     ? *reinterpret_cast<const uint4*>(args.residual + (size_t)(mb + e) * args.ldr + n0)
                     : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (mb + e >= args.M) break;
        const uint32_t r4[4] = {res[e].x, res[e].y, res[e].z, res[e].w};
        uint32_t o4[4];
#pragma unroll
        for (int h = 0; h < 4; ++h)
          o4[h] = pack_bf16x2(acc[2 * h][e] + bf16lo(r4[h]), acc[2 * h + 1][e] + bf16hi(r4[h]));
        *reinterpret_cast<uint4*>(args.Y + (size_t)(mb + e) * args.ldy + n0) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
    } else {
      for (int e = 0; e < 4 && mb + e < args.M; ++e)
        for (int i = 0; i < 8 && n0 + i < args.N; ++i) {
          float o = acc[i][e];
          if (args.residual) o += bf16f(args.residual[(size_t)(mb + e) * args.ldr + n0 + i]);
          args.Y[(size_t)(mb + e) * args.ldy + n0 + i] = f2bf(o);
        }
    }
  }
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
