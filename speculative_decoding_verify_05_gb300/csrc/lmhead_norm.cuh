// Per-row softmax normaliser of the LM head, from the statistics the GEMM epilogue writes per
// 128-token vocabulary tile: (max_t, sum_t e^(z - max_t)) for sampling, (max_t, argmax_t) for
// greedy rows.  Shared by the normalisation kernel (which materialises p) and the fused
// sampler (which evaluates p only where it needs it), so both see bit-identical probabilities.
// One warp combines one row in a single pass (online maximum: the running sum is rescaled when
// the maximum moves), so a block can normalise as many rows at once as it has warps.
#pragma once

#include "common.cuh"

namespace spec {

// (m, s) <- the combination of two partial (max, sum e^(z - max)) pairs; an empty pair has
// m = -inf, s = 0.
__device__ __forceinline__ void lm_merge(float& m, float& s, float om, float os) {
  const float mm = fmaxf(m, om);
  if (mm == -INFINITY) return;        // both empty
  s = s * exp_sm(m - mm) + os * exp_sm(om - mm);
  m = mm;
}

// Called by all 32 lanes of a warp: max over the row and inv = 1 / sum_x e^(z_x - max), so that
// p_x = exp_sm(z_x - mx) * inv.  Lane l takes tiles l, l + 32, ... in order, then the lanes merge
// in a fixed butterfly order.
__device__ __forceinline__ void lm_row_norm_warp(const float2* __restrict__ st, int n_tiles, float& mx_out,
                                                 float& inv_out) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY, s = 0.f;
  for (int t = lane; t < n_tiles; t += 32) {
    const float2 v = st[t];
    lm_merge(m, s, v.x, v.y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const float os = __shfl_xor_sync(0xffffffffu, s, o);
    lm_merge(m, s, om, os);
  }
  mx_out = m;
  inv_out = 1.f / s;
}

// Greedy rows: the argmax over the row (lowest index on ties) from per-tile (max, index bits);
// called by all 32 lanes of a warp.
__device__ __forceinline__ int lm_row_argmax_warp(const float2* __restrict__ st, int n_tiles) {
  const int lane = threadIdx.x & 31;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int t = lane; t < n_tiles; t += 32) {
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
  return bi;
}

}  // namespace spec
