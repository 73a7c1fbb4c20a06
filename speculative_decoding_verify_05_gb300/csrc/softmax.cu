// LM-head normalisation: combine the per-128-token-tile statistics written by
// the GEMM epilogue, then p = exp(z - max) / sum over the whole vocabulary
// (z already divided by the temperature), or a one-hot row at the argmax
// (lowest index on ties) when the temperature is 0.
#include "common.cuh"
#include "internal.h"

namespace spec {
namespace {

constexpr int NORM_THREADS = 256;
constexpr int NORM_CHUNK = 8192;   // vocabulary entries per CTA

__global__ void __launch_bounds__(NORM_THREADS)
lmhead_normalize_kernel(float* __restrict__ P, const float2* __restrict__ stats, int V,
                        int n_tiles, int greedy) {
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.y;
  const int tid = threadIdx.x;
  const float2* st = stats + (size_t)m * n_tiles;
  __shared__ float s_a[NORM_THREADS / 32];
  __shared__ float s_b[NORM_THREADS / 32];
  __shared__ int s_i[NORM_THREADS / 32];
  const int lane = tid & 31, warp = tid >> 5;
  float* row = P + (size_t)m * V;
  const int x0 = blockIdx.x * NORM_CHUNK;
  const int x1 = min(V, x0 + NORM_CHUNK);

  if (greedy) {
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int t = tid; t < n_tiles; t += NORM_THREADS) {
      const float2 v = st[t];
      const int vi = __float_as_int(v.y);
      if (v.x > best || (v.x == best && vi < bi)) { best = v.x; bi = vi; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
    }
    if (lane == 0) { s_a[warp] = best; s_i[warp] = bi; }
    __syncthreads();
    best = s_a[0]; bi = s_i[0];
    for (int w = 1; w < NORM_THREADS / 32; ++w)
      if (s_a[w] > best || (s_a[w] == best && s_i[w] < bi)) { best = s_a[w]; bi = s_i[w]; }
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

  // global max, then sum of exp relative to it
  float mx = -INFINITY;
  for (int t = tid; t < n_tiles; t += NORM_THREADS) mx = fmaxf(mx, st[t].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) s_a[warp] = mx;
  __syncthreads();
  mx = s_a[0];
  for (int w = 1; w < NORM_THREADS / 32; ++w) mx = fmaxf(mx, s_a[w]);
  float sm = 0.f;
  for (int t = tid; t < n_tiles; t += NORM_THREADS) {
    const float2 v = st[t];
    sm += v.y * expf(v.x - mx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
  if (lane == 0) s_b[warp] = sm;
  __syncthreads();
  sm = 0.f;
  for (int w = 0; w < NORM_THREADS / 32; ++w) sm += s_b[w];
  const float inv = 1.f / sm;
  for (int x = x0 + tid * 4; x < x1; x += NORM_THREADS * 4) {
    if (x + 3 < x1) {
      float4 v = *reinterpret_cast<float4*>(row + x);
      v.x = expf(v.x - mx) * inv;
      v.y = expf(v.y - mx) * inv;
      v.z = expf(v.z - mx) * inv;
      v.w = expf(v.w - mx) * inv;
      *reinterpret_cast<float4*>(row + x) = v;
    } else {
      for (int k = x; k < x1; ++k) row[k] = expf(row[k] - mx) * inv;
    }
  }
}

}  // namespace

cudaError_t launch_lmhead_normalize(float* P, const float2* stats, int M, int V, int n_tiles,
                                    bool greedy, cudaStream_t s) {
  dim3 grid((V + NORM_CHUNK - 1) / NORM_CHUNK, M);
  cudaError_t e = launch_k(lmhead_normalize_kernel, dim3(grid), dim3(NORM_THREADS), 0, s, P, stats, V, n_tiles,
                           greedy ? 1 : 0);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace spec
