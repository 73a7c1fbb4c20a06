// Weight-streaming chain of verify GEMMs for a handful of rows (M <= 64): one persistent launch
// runs a list of products Y_j = X_j W_j^T (+ residual, or the SwiGLU activation) in order.
//
// At small M the verify pass is a weight stream ("Speculative Decoding Spends Arithmetic You May
// Not Have", "The speedup is borrowed, and there is a lender": one weight read serves every row;
// "How Speculative Decoding Works (and When It Doesn't)", "Prefill and Decode": the pass is bound
// by memory bandwidth, not arithmetic).  One launch per product pays a fill (first TMA stages in
// flight) and a drain (the last tiles' reduction and epilogue) each time; here the weight producer
// of every CTA keeps streaming from the end of one product into the next, because weights never
// depend on activations.  Only the token tiles wait: product j's loads of X_j (and its epilogue's
// residual reads and Y_j writes) wait on device-side flags of the products it depends on, which
// the host derives from the buffers' address ranges.
//
// Work split: every product's (128-row weight tile, 64-wide k-step) units are cut into G equal
// contiguous ranges, one per CTA (stream-K), so every SM streams the same bytes of every product.
// A tile cut between CTAs leaves fp32 pieces: each CTA that does not hold the tile's first k-step
// publishes its piece (one slot per product and CTA) and bumps the tile's arrival counter; the CTA
// that holds k-step 0 (it reaches that part at the end of its range, so the others are usually
// done) waits for the pieces and adds them to its own accumulator in CTA order (deterministic),
// then runs the epilogue and marks the tile stored.
//
// Roles (12 warps): warp 0 streams weight tiles, warp 1 issues tcgen05.mma into a ring of TMEM
// accumulators, warp 2 streams token tiles once their flags allow, warps 4-11 drain the
// accumulators (TMEM lane quarter = warp % 4, one weight row and half of the token columns per
// thread).  Every wait is bounded.
#include "internal.h"
#include "linear_tc.cuh"

namespace spec {
namespace {

constexpr int CH_THREADS = 384;
constexpr int CH_EPI_THREADS = 256;   // warps 4-11: 4 lane quarters x 2 column halves
constexpr int CH_W_BYTES = 128 * LIN_ROW_BYTES;   // one 128 x 64 weight tile

template <int BN>
struct ChainCfg {
  static constexpr int X_BYTES = BN * LIN_ROW_BYTES;
  static constexpr int STAGE_BYTES = CH_W_BYTES + X_BYTES;
  static constexpr int STAGES = (220 * 1024) / STAGE_BYTES > 16 ? 16 : (220 * 1024) / STAGE_BYTES;
  // NACC accumulators of BN columns: the MMA runs up to NACC - 1 segments ahead of the epilogue,
  // which absorbs the latency of a tile owner's wait for its pieces
  static constexpr int NACC = 256 / BN;
  static constexpr int ACC_COLS = BN;
  static constexpr int TMEM_COLS = 256;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 1024;
};

// ------------------------------------------------------------------ global flags
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Bounded spin until *p >= target (false, status set, on timeout).
__device__ __forceinline__ bool spin_geq(const unsigned* p, unsigned target, unsigned* status, unsigned site) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    __nanosleep(64);
    if (ld_acquire(p) >= target) return true;
    if ((it & 63u) == 63u && globaltimer() - t0 > SPEC_WAIT_NS) {
      set_status(status, site);
      return false;
    }
  }
}
// Order this thread's generic-proxy view of global memory with its later async-proxy (TMA)
// accesses, and vice versa.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void bar_chain_epi() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// The same barrier, returning whether `v` held on every epilogue thread (keeps the epilogue's
// control flow uniform after a wait that one thread took and that may have run out).
__device__ __forceinline__ bool bar_chain_epi_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.and.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// N consecutive TMEM columns of this thread's lane (N = 8, 16 or 32: half of a 16-, 32- or
// 64-column accumulator), loaded and waited for.
template <int N>
__device__ __forceinline__ void chain_tmem_ld(uint32_t taddr, float* v) {
  if constexpr (N == 16 || N == 32) {
    tmem_ld_cols<N>(taddr, v);
  } else {
    static_assert(N == 8, "column count");
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8+0];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
  }
}

// ------------------------------------------------------------------ work of one CTA
__device__ __forceinline__ int range_start(int units, int c, int G) {
  return (int)((long long)units * c / G);
}

// Segment = the CTA's units of one (product, tile).
struct CSeg {
  int op, tile, u0, u1;     // units [u0, u1) of product op (unit = tile * k_tiles + k)
  int kind;                 // 0 whole tile, 1 owner (holds k-step 0, not the whole tile), 2 publisher
};

// Walks this CTA's segments over all products in order.
struct SegWalker {
  int op = 0, u = 0, end = 0;
  __device__ __forceinline__ void begin(const ChainParams& p, int c) {
    op = 0;
    u = range_start(p.op[0].units, c, p.grid);
    end = range_start(p.op[0].units, c + 1, p.grid);
    skip_empty(p, c);
  }
  __device__ __forceinline__ void skip_empty(const ChainParams& p, int c) {
    while (op < p.n_ops && u >= end) {
      ++op;
      if (op < p.n_ops) {
        u = range_start(p.op[op].units, c, p.grid);
        end = range_start(p.op[op].units, c + 1, p.grid);
      }
    }
  }
  __device__ __forceinline__ bool done(const ChainParams& p) const { return op >= p.n_ops; }
  __device__ __forceinline__ CSeg next(const ChainParams& p, int c) {
    CSeg s;
    const int kt = p.op[op].k_tiles;
    s.op = op;
    s.tile = u / kt;
    s.u0 = u;
    const int t_end = (s.tile + 1) * kt;
    s.u1 = end < t_end ? end : t_end;
    const bool starts = s.u0 == s.tile * kt, ends = s.u1 == t_end;
    s.kind = starts ? (ends ? 0 : 1) : 2;
    u = s.u1;
    skip_empty(p, c);
    return s;
  }
};

// ------------------------------------------------------------------ dependency waits
// Tiles of product d whose Y columns [c0, c1) a consumer needs: wait until each is stored.
__device__ __forceinline__ bool wait_cols(const ChainParams& p, int d, int c0, int c1, unsigned site) {
  const ChainOp& o = p.op[d];
  int t0 = c0 / o.ycols, t1 = (c1 - 1) / o.ycols;
  if (t1 >= o.tiles_n) t1 = o.tiles_n - 1;
  for (int t = t0; t <= t1; ++t)
    if (!spin_geq(p.done + o.flag_base + t, 1u, p.status, site)) return false;
  return true;
}
__device__ __forceinline__ bool wait_whole(const ChainParams& p, int d, unsigned site) {
  return spin_geq(p.op_done + d, (unsigned)p.op[d].tiles_n, p.status, site);
}

// Token producer: have all the products that X_j reads from finished (one load each)?
__device__ __forceinline__ bool x_deps_complete(const ChainParams& p, int j) {
  const ChainOp& o = p.op[j];
  for (int i = 0; i < o.n_deps; ++i) {
    const ChainDep& dp = o.dep[i];
    if (dp.kind == CH_DEP_X && ld_acquire(p.op_done + dp.op) < (unsigned)p.op[dp.op].tiles_n) return false;
  }
  return true;
}
// Token producer: the X columns [64 k, 64 k + 64) of product j.
__device__ __forceinline__ bool wait_x(const ChainParams& p, int j, int k) {
  const ChainOp& o = p.op[j];
  bool ok = true;
  for (int i = 0; i < o.n_deps && ok; ++i) {
    const ChainDep& dp = o.dep[i];
    if (dp.kind != CH_DEP_X) continue;
    if (dp.shift < 0) ok = wait_whole(p, dp.op, 0x161u);
    else ok = wait_cols(p, dp.op, k * LIN_BK + dp.shift, k * LIN_BK + LIN_BK + dp.shift, 0x162u);
  }
  return ok;
}
// Epilogue of tile t of product j: its residual columns stored and (with `writes`, checked once per
// product and CTA) every earlier reader / writer of its Y region finished.
__device__ __forceinline__ bool wait_epilogue(const ChainParams& p, int j, int t, bool writes) {
  const ChainOp& o = p.op[j];
  bool ok = true;
  for (int i = 0; i < o.n_deps && ok; ++i) {
    const ChainDep& dp = o.dep[i];
    if (dp.kind == CH_DEP_RES) {
      if (dp.shift < 0) ok = wait_whole(p, dp.op, 0x163u);
      else ok = wait_cols(p, dp.op, t * o.ycols + dp.shift, t * o.ycols + o.ycols + dp.shift, 0x164u);
    } else if (dp.kind == CH_DEP_WRITE && writes) {
      ok = wait_whole(p, dp.op, 0x165u);
    }
  }
  return ok;
}

template <int BN>
__global__ void __launch_bounds__(CH_THREADS, 1) linear_chain_kernel(const __grid_constant__ ChainParams p) {
  using Cfg = ChainCfg<BN>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;
  uint8_t* sX = smem + STAGES * CH_W_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + Cfg::NACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + Cfg::NACC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 2);        // one arrival from each producer
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < Cfg::NACC; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], CH_EPI_THREADS);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  if (warp == 0 || warp == 2) {
    // ---------------- producers: the same unit sequence, weights (warp 0) and tokens (warp 2)
    if (lane == 0) {
      const bool tokens = warp == 2;
      SegWalker w;
      w.begin(p, c);
      int i = 0;            // running unit index (ring position)
      int cur_op = -1;
      int sat_op = -1;      // token side: the product whose X dependencies are all met
      bool ok = true;
      while (!w.done(p) && ok) {
        const CSeg g = w.next(p, c);
        const ChainOp& o = p.op[g.op];
        const CUtensorMap* tm = tokens ? &p.tx[g.op] : &p.tw[g.op];
        if (g.op != cur_op) {
          tma_prefetch_desc(tm);
          cur_op = g.op;
        }
        for (int u = g.u0; u < g.u1 && ok; ++u, ++i) {
          const int s = i % STAGES;
          if (i >= STAGES && !mbar_wait(&empty[s], (uint32_t)((i / STAGES - 1) & 1), p.status, 0x151u)) {
            ok = false;
            break;
          }
          const int k = u - g.tile * o.k_tiles;
          if (tokens) {
            // once every product X_j reads from has finished, no further checks for product j;
            // until then, per k-step waits on the tiles it reads.  A proxy fence after each wait
            // orders the other CTAs' stores (seen through the acquire) before this TMA read
            if (g.op != sat_op) {
              if (o.n_deps == 0 || x_deps_complete(p, g.op)) {
                sat_op = g.op;
              } else if (!wait_x(p, g.op, k)) {
                ok = false;
                break;
              }
              fence_proxy_async_global();
            }
            mbar_arrive_expect_tx(&full[s], Cfg::X_BYTES);
            tma_load_2d(sX + s * Cfg::X_BYTES, tm, &full[s], k * LIN_BK, 0);
          } else {
            mbar_arrive_expect_tx(&full[s], CH_W_BYTES);
            tma_load_2d_hint(sW + s * CH_W_BYTES, tm, &full[s], k * LIN_BK, g.tile * 128, l2_policy_evict_first());
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer: one accumulator per segment, NACC in flight
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(128, BN);
      SegWalker w;
      w.begin(p, c);
      int i = 0, seg = 0;
      bool ok = true;
      while (!w.done(p) && ok) {
        const CSeg g = w.next(p, c);
        const int acc = seg % Cfg::NACC, use = seg / Cfg::NACC;
        if (use >= 1 && !mbar_wait(&acc_empty[acc], (uint32_t)((use - 1) & 1), p.status, 0x152u)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * Cfg::ACC_COLS;
        for (int u = g.u0; u < g.u1; ++u, ++i) {
          const int s = i % STAGES;
          if (!mbar_wait(&full[s], (uint32_t)((i / STAGES) & 1), p.status, 0x153u)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a = smem_u32(sW + s * CH_W_BYTES);
          const uint32_t b = smem_u32(sX + s * Cfg::X_BYTES);
#pragma unroll
          for (int kk = 0; kk < LIN_BK / 16; ++kk)
            umma_bf16(d, umma_desc_lin(a + kk * 32), umma_desc_lin(b + kk * 32), idesc, (u > g.u0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&acc_full[acc]);
        ++seg;
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- epilogue: thread r = weight row r of the tile (TMEM lane r), token columns
    // col0 .. col0 + HB - 1 of the accumulator
    constexpr int HB = BN / 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int col0 = ((warp - 4) >> 2) * HB;
    const uint32_t t_lane = (uint32_t(q * 32) << 16) + (uint32_t)col0;
    SegWalker w;
    w.begin(p, c);
    int seg = 0;
    int write_ok_op = -1;
    bool ok = true;
    while (!w.done(p)) {
      const CSeg g = w.next(p, c);
      const ChainOp& o = p.op[g.op];
      const int acc = seg % Cfg::NACC;
      ok = ok && mbar_wait(&acc_full[acc], (uint32_t)((seg / Cfg::NACC) & 1), p.status, 0x154u);
      ok = bar_chain_epi_and(ok);
      tc_fence_after();
      float v[HB];
      if (ok) {
        chain_tmem_ld<HB>(tmem + acc * Cfg::ACC_COLS + t_lane, v);
      } else {
#pragma unroll
        for (int j = 0; j < HB; ++j) v[j] = 0.f;
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[acc]);
      ++seg;
      float* my_piece = p.pieces + ((size_t)g.op * p.grid + c) * (BN * 128);
      if (g.kind == 2) {
        // publisher: the fp32 piece, [column][128 rows] (one 128-byte line per column per warp)
#pragma unroll
        for (int j = 0; j < HB; ++j) __stcg(my_piece + (col0 + j) * 128 + r, v[j]);
        bar_chain_epi();
        if (threadIdx.x == 128) {
          __threadfence();
          atomicAdd(p.arrive + o.flag_base + g.tile, 1u);
        }
        continue;
      }
      if (g.kind == 1) {
        // owner: the other CTAs whose ranges reach into this tile, in CTA order
        const int t_end = (g.tile + 1) * o.k_tiles;
        unsigned n_other = 0;
        for (int c2 = c + 1; c2 < p.grid && range_start(o.units, c2, p.grid) < t_end; ++c2)
          if (range_start(o.units, c2, p.grid) < range_start(o.units, c2 + 1, p.grid)) ++n_other;
        // (thread 128's acquire, then the barrier: the pieces are visible to every epilogue thread)
        if (threadIdx.x == 128) ok = ok && spin_geq(p.arrive + o.flag_base + g.tile, n_other, p.status, 0x155u);
        ok = bar_chain_epi_and(ok);
        // the contributors' pieces, PB CTAs' loads in flight at a time, added in CTA order
        constexpr int PB = HB <= 8 ? 4 : HB <= 16 ? 1 : 2;   // (no register spills at 384 threads)
        int c2 = c + 1;
        while (c2 < p.grid && range_start(o.units, c2, p.grid) < t_end) {
          int cs[PB];
          int nc = 0;
          for (; nc < PB && c2 < p.grid && range_start(o.units, c2, p.grid) < t_end; ++c2)
            if (range_start(o.units, c2, p.grid) < range_start(o.units, c2 + 1, p.grid)) cs[nc++] = c2;
          float pv[PB][HB];
#pragma unroll
          for (int b = 0; b < PB; ++b) {
            if (b >= nc) break;
            const float* pc = p.pieces + ((size_t)g.op * p.grid + cs[b]) * (BN * 128);
#pragma unroll
            for (int j = 0; j < HB; ++j) pv[b][j] = __ldcg(pc + (col0 + j) * 128 + r);
          }
#pragma unroll
          for (int b = 0; b < PB; ++b) {
            if (b >= nc) break;
#pragma unroll
            for (int j = 0; j < HB; ++j) v[j] += pv[b][j];
          }
        }
      }
      // this tile's residual stored and (once per product) every earlier user of Y's region done
      if (threadIdx.x == 128) ok = ok && wait_epilogue(p, g.op, g.tile, g.op != write_ok_op);
      write_ok_op = g.op;
      ok = bar_chain_epi_and(ok);
      const int n = g.tile * 128 + r;
      if (o.epi == EPI_SWIGLU) {
        // rows interleaved per 16: lane l < 16 holds gate row l of the warp's block, lane l + 16
        // the matching up row; output column tile * 64 + q * 16 + l
        const int col = g.tile * 64 + q * 16 + (lane & 15);
#pragma unroll
        for (int j = 0; j < HB; ++j) {
          const float up = __shfl_xor_sync(0xffffffffu, v[j], 16);
          const int m = col0 + j;
          if (lane < 16 && m < p.M) o.Y[(size_t)m * o.ldy + col] = f2bf(silu(v[j]) * up);
        }
      } else if (n < o.N) {
#pragma unroll
        for (int j = 0; j < HB; ++j) {
          const int m = col0 + j;
          if (m >= p.M) break;
          float y = v[j];
          if (o.residual) y += bf16f(o.residual[(size_t)m * o.ldr + n]);
          o.Y[(size_t)m * o.ldy + n] = f2bf(y);
        }
      }
      bar_chain_epi();
      if (threadIdx.x == 128) {
        fence_proxy_async_global();
        __threadfence();
        atomicExch(p.done + o.flag_base + g.tile, 1u);
        atomicAdd(p.op_done + g.op, 1u);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

template <int BN>
cudaError_t launch_chain_bn(const ChainParams& p, cudaStream_t s) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(linear_chain_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         ChainCfg<BN>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  cudaError_t e = launch_k(linear_chain_kernel<BN>, dim3(p.grid), dim3(CH_THREADS), ChainCfg<BN>::SMEM_BYTES, s, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int chain_bn(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= CH_MAX_M ? 64 : -1; }

cudaError_t launch_linear_chain(const ChainParams& p, cudaStream_t s) {
  switch (chain_bn(p.M)) {
    case 16: return launch_chain_bn<16>(p, s);
    case 32: return launch_chain_bn<32>(p, s);
    case 64: return launch_chain_bn<64>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spec
