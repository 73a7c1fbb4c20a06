// Instantiations of the persistent tcgen05 verify GEMM for the bf16 (+ residual) epilogue.
#include "internal.h"
#include "linear_tc_kernel.cuh"

namespace spec {

int linear_tc_smem_bytes(int BN, int NSUB) {
  switch (NSUB * 1000 + BN) {
    case 1016: return LinearCfg<16, 1>::SMEM_BYTES;
    case 1032: return LinearCfg<32, 1>::SMEM_BYTES;
    case 1048: return LinearCfg<48, 1>::SMEM_BYTES;
    case 1064: return LinearCfg<64, 1>::SMEM_BYTES;
    case 1080: return LinearCfg<80, 1>::SMEM_BYTES;
    case 1096: return LinearCfg<96, 1>::SMEM_BYTES;
    case 1112: return LinearCfg<112, 1>::SMEM_BYTES;
    case 1128: return LinearCfg<128, 1>::SMEM_BYTES;
    case 1144: return LinearCfg<144, 1>::SMEM_BYTES;
    case 1160: return LinearCfg<160, 1>::SMEM_BYTES;
    case 1176: return LinearCfg<176, 1>::SMEM_BYTES;
    case 1192: return LinearCfg<192, 1>::SMEM_BYTES;
    case 1208: return LinearCfg<208, 1>::SMEM_BYTES;
    case 1224: return LinearCfg<224, 1>::SMEM_BYTES;
    case 1240: return LinearCfg<240, 1>::SMEM_BYTES;
    case 1256: return LinearCfg<256, 1>::SMEM_BYTES;
    case 2144: return LinearCfg<144, 2>::SMEM_BYTES;
    case 2160: return LinearCfg<160, 2>::SMEM_BYTES;
    case 2176: return LinearCfg<176, 2>::SMEM_BYTES;
    case 2192: return LinearCfg<192, 2>::SMEM_BYTES;
    case 2208: return LinearCfg<208, 2>::SMEM_BYTES;
    case 2224: return LinearCfg<224, 2>::SMEM_BYTES;
    case 2240: return LinearCfg<240, 2>::SMEM_BYTES;
    case 2256: return LinearCfg<256, 2>::SMEM_BYTES;
    default: return -1;
  }
}

bool linear_tc_supported(int BN, int NSUB) { return linear_tc_smem_bytes(BN, NSUB) > 0; }

cudaError_t launch_linear_tc_bf16(int BN, int NSUB, const CUtensorMap& tw, const CUtensorMap& tx,
                                  const LinearArgs& a, dim3 grid, cudaStream_t s) {
  switch (NSUB * 1000 + BN) {
    case 1016: return launch_linear_tc_one<16, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1032: return launch_linear_tc_one<32, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1048: return launch_linear_tc_one<48, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1064: return launch_linear_tc_one<64, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1080: return launch_linear_tc_one<80, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1096: return launch_linear_tc_one<96, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1112: return launch_linear_tc_one<112, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1128: return launch_linear_tc_one<128, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1144: return launch_linear_tc_one<144, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1160: return launch_linear_tc_one<160, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1176: return launch_linear_tc_one<176, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1192: return launch_linear_tc_one<192, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1208: return launch_linear_tc_one<208, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1224: return launch_linear_tc_one<224, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1240: return launch_linear_tc_one<240, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 1256: return launch_linear_tc_one<256, 1, EPI_BF16>(tw, tx, a, grid, s);
    case 2144: return launch_linear_tc_one<144, 2, EPI_BF16>(tw, tx, a, grid, s);
    case 2160: return launch_linear_tc_one<160, 2, EPI_BF16>(tw, tx, a, grid, s);
    case 2176: return launch_linear_tc_one<176, 2, EPI_BF16>(tw, tx, a, grid, s);
    case 2192: return launch_linear_tc_one<192, 2, EPI_BF16>(tw, tx, a, grid, s);
    case 2208: return launch_linear_tc_one<208, 2, EPI_BF16>(tw, tx, a, grid, s);
    case 2224: return launch_linear_tc_one<224, 2, EPI_BF16>(tw, tx, a, grid, s);
    case 2240: return launch_linear_tc_one<240, 2, EPI_BF16>(tw, tx, a, grid, s);
    case 2256: return launch_linear_tc_one<256, 2, EPI_BF16>(tw, tx, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

// Second pass of a split GEMM.  Every block first tabulates where each work group's stream-K
// range starts (beg[c] = sk_units * c / grid, one 64-bit division per entry; unit u is k-step
// u % kt of work tile dp_tiles + u / kt).  A work tile is split iff a range starts strictly
// inside it; the first such range c names it, and its pieces came from groups c - 1 .. hi (the
// last range starting inside it).  A work group is one CTA, or a CTA pair (a.pair) whose CTA of
// rank r left the piece of 128-row weight tile 2 (t / tiles_m) + r.  Warp item = (c, r, 8 token
// columns); lane l owns weight rows n0 + 4 l .. + 3 (one float4 per column of a piece).
// Pieces are summed in CTA order, two contributors' loads in flight at a time, then the
// residual is added and the sum rounded to bf16.  Launched as one wave (grid-stride over items).
__global__ void __launch_bounds__(256, 2) linear_reduce_kernel(const LinearArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ long long s_beg[];                      // [grid + 1]
  int* s_hi = reinterpret_cast<int*>(s_beg + a.grid + 1);   // [grid] -1: c names no tile
  const int G = a.grid, TN = a.tn;
  const long long kt = a.k_tiles;
  for (int c = threadIdx.x; c <= G; c += blockDim.x) s_beg[c] = a.sk_units * c / G;
  __syncthreads();
  for (int c = threadIdx.x; c < G; c += blockDim.x) {
    int hi = -1;
    if (c > 0) {
      const long long b = s_beg[c], t0 = b / kt * kt;
      if (b != t0 && s_beg[c - 1] <= t0) {
        hi = c;
        while (hi + 1 < G && s_beg[hi + 1] < t0 + kt) ++hi;
      }
    }
    s_hi[c] = hi;
  }
  __syncthreads();
  const int cols8 = (TN + 7) / 8;
  const int R = a.pair ? 2 : 1;
  const long long items = (long long)G * R * cols8;
  const int lane = threadIdx.x & 31;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long it = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items; it += nwarps) {
    const int c = (int)(it / (R * cols8));
    const int hi = s_hi[c];
    if (hi < 0) continue;
    const int rest = (int)(it - (long long)c * R * cols8);
    const int r = rest / cols8;
    const int j0 = (rest - r * cols8) * 8;
    const long long t0 = s_beg[c] / kt * kt;
    const long long ctile = a.dp_tiles + t0 / kt;
    const int n_t = (int)(ctile / a.tiles_m) * R + r;
    if (n_t >= a.tiles_n) continue;   // (the odd half of a pair tile past N)
    const int m0 = (int)(ctile % a.tiles_m) * TN + j0;
    const int n4 = n_t * 128 + lane * 4;
    float4 acc[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) acc[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = c - 1; c0 <= hi; c0 += 2) {
      float4 v[2][8];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int cc = c0 + q;
        // slot 0 holds the piece that opens a CTA's stream-K range: the tile's iff the range starts
        // inside it; a CTA with an empty range (fewer stream-K units than CTAs) left nothing
        const float* base = (cc <= hi && s_beg[cc] < s_beg[cc + 1])
                                ? a.partial + (((size_t)cc * R + r) * 2 + (s_beg[cc] >= t0 ? 0 : 1)) * (TN * 128) + lane * 4
                                : nullptr;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
          v[q][jj] = (base && j0 + jj < TN) ? __ldcg(reinterpret_cast<const float4*>(base + (j0 + jj) * 128))
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          acc[jj].x += v[q][jj].x; acc[jj].y += v[q][jj].y; acc[jj].z += v[q][jj].z; acc[jj].w += v[q][jj].w;
        }
    }
    if (a.epi == EPI_SWIGLU) {
      // gate and up rows interleaved in blocks of 16: lane L holds rows 4L .. 4L + 3, gate rows
      // when L % 8 < 4, and lane L + 4 holds the matching up rows
      const bool gate = (lane & 7) < 4;
      const int n = n_t * 64 + (lane >> 3) * 16 + (lane & 3) * 4;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float u0 = __shfl_down_sync(0xffffffffu, acc[jj].x, 4), u1 = __shfl_down_sync(0xffffffffu, acc[jj].y, 4);
        const float u2 = __shfl_down_sync(0xffffffffu, acc[jj].z, 4), u3 = __shfl_down_sync(0xffffffffu, acc[jj].w, 4);
        const int m = m0 + jj;
        if (!gate || j0 + jj >= TN || m >= a.M) continue;
        const float g[4] = {acc[jj].x, acc[jj].y, acc[jj].z, acc[jj].w}, u[4] = {u0, u1, u2, u3};
        float y[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = silu(g[e]) * u[e];
        *reinterpret_cast<uint2*>(a.Y + (size_t)m * a.ldy + n) = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
      }
      continue;
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int m = m0 + jj;
      if (j0 + jj >= TN || m >= a.M) continue;
      float y[4] = {acc[jj].x, acc[jj].y, acc[jj].z, acc[jj].w};
      if (n4 + 3 < a.N) {
        if (a.residual) {
          const uint2 rr = *reinterpret_cast<const uint2*>(a.residual + (size_t)m * a.ldr + n4);
          y[0] += bf16lo(rr.x); y[1] += bf16hi(rr.x); y[2] += bf16lo(rr.y); y[3] += bf16hi(rr.y);
        }
        *reinterpret_cast<uint2*>(a.Y + (size_t)m * a.ldy + n4) = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
      } else {
        for (int e = 0; e < 4 && n4 + e < a.N; ++e) {
          float v2 = y[e];
          if (a.residual) v2 += bf16f(a.residual[(size_t)m * a.ldr + n4 + e]);
          a.Y[(size_t)m * a.ldy + n4 + e] = f2bf(v2);
        }
      }
    }
  }
}

cudaError_t launch_linear_reduce(const LinearArgs& a, int sms, cudaStream_t s) {
  const size_t smem = (size_t)(a.grid + 1) * 8 + (size_t)a.grid * 4;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    // up to 4096 persistent CTAs: 4097 starts + 4096 ends
    cudaError_t e = cudaFuncSetAttribute(linear_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 4097 * 8 + 4096 * 4);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  // one wave: two 256-thread blocks per SM (register budget), grid-stride over the items
  const long long warps = (long long)a.grid * (a.pair ? 2 : 1) * ((a.tn + 7) / 8);
  long long blocks = (warps + 7) / 8;
  if (blocks > 2LL * sms) blocks = 2LL * sms;
  cudaError_t e = launch_k(linear_reduce_kernel, dim3((unsigned)(blocks > 0 ? blocks : 1)), dim3(256), smem, s, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace spec
