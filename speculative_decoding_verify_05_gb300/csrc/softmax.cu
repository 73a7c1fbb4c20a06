// LM-head normalisation: combine the per-128-token-tile statistics written by
// the GEMM epilogue, then p = exp(z - max) / sum over the whole vocabulary
// (z already divided by the temperature), or a one-hot row at the argmax
// (lowest index on ties) when the temperature is 0.
#include "common.cuh"
#include "internal.h"
#include "lmhead_norm.cuh"

namespace spec {
namespace {

constexpr int NORM_THREADS = 256;
constexpr int NORM_CHUNK = 8192;   // vocabulary entries per CTA

__global__ void __launch_bounds__(NORM_THREADS)
lmhead_normalize_kernel(float* __restrict__ P, long long ldp, const float2* __restrict__ stats, int V,
                        int n_tiles, int greedy) {
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.y;
  const int tid = threadIdx.x;
  const float2* st = stats + (size_t)m * n_tiles;
  __shared__ float s_mx, s_inv;
  __shared__ int s_am;
  float* row = P + (size_t)m * ldp;
  const int x0 = blockIdx.x * NORM_CHUNK;
  const int x1 = min(V, x0 + NORM_CHUNK);

  if (greedy) {
    if (tid < 32) {
      const int am = lm_row_argmax_warp(st, n_tiles);
      if (tid == 0) s_am = am;
    }
    __syncthreads();
    const int bi = s_am;
    for (int x = x0 + tid * 4; x < x1; x += NORM_THREADS * 4) {
      if (x + 3 < x1) {
        float4 v = make_float4(x == bi ? 1.f : 0.f, x + 1 == bi ? 1.f : 0.f,
                               x + 2 == bi ? 1.f : 0.f, x + 3 == bi ? 1.f : 0.f);
        *reinterpret_cast<float4*>(row + x) = v;
      } else {
        for (int k = x; k < x1; ++k) row[k] = (k == bi) ? 1.f : 0.f;
      }
    }
    return;
  }

  // global max, then sum of exp relative to it (the shared per-row normaliser)
  if (tid < 32) {
    float mx, inv;
    lm_row_norm_warp(st, n_tiles, mx, inv);
    if (tid == 0) { s_mx = mx; s_inv = inv; }
  }
  __syncthreads();
  const float mx = s_mx, inv = s_inv;
  for (int x = x0 + tid * 4; x < x1; x += NORM_THREADS * 4) {
    if (x + 3 < x1) {
      float4 v = *reinterpret_cast<float4*>(row + x);
      v.x = exp_sm(v.x - mx) * inv;
      v.y = exp_sm(v.y - mx) * inv;
      v.z = exp_sm(v.z - mx) * inv;
      v.w = exp_sm(v.w - mx) * inv;
      *reinterpret_cast<float4*>(row + x) = v;
    } else {
      for (int k = x; k < x1; ++k) row[k] = exp_sm(row[k] - mx) * inv;
    }
  }
}

}  // namespace

cudaError_t launch_lmhead_normalize(float* P, long long ldp, const float2* stats, int M, int V, int n_tiles,
                                    bool greedy, cudaStream_t s) {
  dim3 grid((V + NORM_CHUNK - 1) / NORM_CHUNK, M);
  cudaError_t e = launch_k(lmhead_normalize_kernel, dim3(grid), dim3(NORM_THREADS), 0, s, P, ldp, stats, V, n_tiles,
                           greedy ? 1 : 0);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace spec
