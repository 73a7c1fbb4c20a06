// CUDA-core weight-streaming GEMM for the tiniest verify passes (M <= 4 rows):
// at ~M FLOP per weight byte this is a pure HBM stream, so no tensor core is
// involved.  Each warp owns 4 weight rows x one K slice: lanes read
// consecutive 16-byte chunks of the rows (coalesced 128-bit loads, all issued
// before any FMA), keep the matching activation chunks in registers, and
// reduce with shuffles.  K is split so that every SM gets several independent
// work items; the warp that finishes a row group last (atomic counter, no
// waiting) sums the fp32 partials in split order and writes bf16.
#include "common.cuh"
#include "internal.h"

namespace spec {
namespace {

constexpr int GEMV_THREADS = 256;
constexpr int ROWS = 4;                 // weight rows per warp item

template <int MT>
struct GemvCfg {
  static constexpr int T = 8 / MT;      // 16-byte chunks per lane per row (T * 256 = K slice)
  static constexpr int KS = T * 256;
};

template <int MT>
__global__ void __launch_bounds__(GEMV_THREADS)
gemv_kernel(const GemvArgs a) {
  pdl_wait();
  pdl_trigger();
  constexpr int T = GemvCfg<MT>::T;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (GEMV_THREADS / 32) + (threadIdx.x >> 5);
  const int TW = gridDim.x * (GEMV_THREADS / 32);
  const int groups = (a.N + ROWS - 1) / ROWS;
  const int items = groups * a.splits;

  uint4 xr[MT][T];
  int cur_split = -1;
  for (int it = gw; it < items; it += TW) {
    const int s = it % a.splits;
    const int g = it / a.splits;
    const int k0 = s * a.k_per_split;
    if (s != cur_split) {
      cur_split = s;
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const int k = k0 + (lane + 32 * t) * 8;
          xr[m][t] = (m < a.M && k < a.K)
                         ? *reinterpret_cast<const uint4*>(a.X + (size_t)m * a.ldx + k)
                         : make_uint4(0, 0, 0, 0);
        }
    }
    uint4 wr[ROWS][T];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const int n = g * ROWS + r;
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const int k = k0 + (lane + 32 * t) * 8;
        wr[r][t] = (n < a.N && k < a.K)
                       ? __ldg(reinterpret_cast<const uint4*>(a.W + (size_t)n * a.ldw + k))
                       : make_uint4(0, 0, 0, 0);
      }
    }
    float acc[ROWS][MT];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;
#pragma unroll
    for (int t = 0; t < T; ++t) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const uint32_t xw[4] = {xr[m][t].x, xr[m][t].y, xr[m][t].z, xr[m][t].w};
        float xf[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          xf[2 * e] = bf16lo(xw[e]);
          xf[2 * e + 1] = bf16hi(xw[e]);
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
          const uint32_t ww[4] = {wr[r][t].x, wr[r][t].y, wr[r][t].z, wr[r][t].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[r][m] = fmaf(bf16lo(ww[e]), xf[2 * e], acc[r][m]);
            acc[r][m] = fmaf(bf16hi(ww[e]), xf[2 * e + 1], acc[r][m]);
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], o);

    if (a.splits == 1) {
      if (lane < ROWS * MT) {
        const int r = lane / MT, m = lane % MT;
        const int n = g * ROWS + r;
        float v = 0.f;
#pragma unroll
        for (int rr = 0; rr < ROWS; ++rr)
#pragma unroll
          for (int mm = 0; mm < MT; ++mm)
            if (rr == r && mm == m) v = acc[rr][mm];
        if (n < a.N && m < a.M) {
          if (a.residual) v += bf16f(a.residual[(size_t)m * a.ldr + n]);
          a.Y[(size_t)m * a.ldy + n] = f2bf(v);
        }
      }
      continue;
    }
    // split-K: publish the partial, then the last warp of this row group reduces
    if (lane < ROWS * MT) {
      const int r = lane / MT, m = lane % MT;
      const int n = g * ROWS + r;
      float v = 0.f;
#pragma unroll
      for (int rr = 0; rr < ROWS; ++rr)
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
          if (rr == r && mm == m) v = acc[rr][mm];
      if (n < a.N && m < a.M) __stcg(&a.partial[((size_t)s * a.M + m) * a.N + n], v);
    }
    __threadfence();
    __syncwarp();
    unsigned prev = 0;
    if (lane == 0) prev = atomicAdd(&a.counters[g], 1u);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    if (prev == (unsigned)(a.splits - 1)) {
      __threadfence();
      if (lane < ROWS * MT) {
        const int r = lane / MT, m = lane % MT;
        const int n = g * ROWS + r;
        if (n < a.N && m < a.M) {
          float v = 0.f;
          for (int ss = 0; ss < a.splits; ++ss) v += __ldcg(&a.partial[((size_t)ss * a.M + m) * a.N + n]);
          if (a.residual) v += bf16f(a.residual[(size_t)m * a.ldr + n]);
          a.Y[(size_t)m * a.ldy + n] = f2bf(v);
        }
      }
      if (lane == 0) a.counters[g] = 0u;
    }
  }
}

}  // namespace

int gemv_k_slice(int M) {
  switch (M) {
    case 1: return GemvCfg<1>::KS;
    case 2: return GemvCfg<2>::KS;
    case 3: return GemvCfg<4>::KS;
    default: return GemvCfg<4>::KS;
  }
}

cudaError_t launch_gemv(const GemvArgs& a, int grid, cudaStream_t s) {
  switch (a.M) {
    case 1: { cudaError_t e = launch_k(gemv_kernel<1>, dim3(grid), dim3(GEMV_THREADS), 0, s, a); if (e != cudaSuccess) return e; break; }
    case 2: { cudaError_t e = launch_k(gemv_kernel<2>, dim3(grid), dim3(GEMV_THREADS), 0, s, a); if (e != cudaSuccess) return e; break; }
    default: { cudaError_t e = launch_k(gemv_kernel<4>, dim3(grid), dim3(GEMV_THREADS), 0, s, a); if (e != cudaSuccess) return e; break; }
  }
  return cudaGetLastError();
}

}  // namespace spec
