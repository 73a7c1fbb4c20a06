// Rejection sampler: one CTA per sequence.
//
// Steps (Algorithm 1 on "Speculative Decoding Spends Arithmetic You May Not
// Have", section "What one iteration actually does"):
//   1. warp 0 evaluates all gamma_b acceptance tests at once (lane i: draft
//      i), in fp64 so that u*q is exact; n = first rejection (ballot), else
//      gamma_b;
//   2. the block builds the final weights w(x) = max(0, p - q) at the first
//      rejection (p itself if that is all zero), or w = p_{gamma+1} (bonus);
//   3. inverse CDF in token order: each thread owns a contiguous slice of the
//      vocabulary, slice sums are scanned across the block in fp64, and the
//      thread whose slice crosses u * sum(w) walks it to find the token.
#include "common.cuh"
#include "internal.h"

namespace spec {
namespace {

constexpr int SAMPLER_THREADS = 512;

__device__ __forceinline__ double row_weight(const float* p, const float* q, int x, bool resid,
                                             bool fallback) {
  const double pv = (double)p[x];
  if (!resid || fallback) return pv;
  const double r = pv - (double)q[x];
  return r > 0.0 ? r : 0.0;
}

__global__ void __launch_bounds__(SAMPLER_THREADS)
reject_sample_kernel(const float* __restrict__ P, const float* __restrict__ Q,
                     const int32_t* __restrict__ draft, const float* __restrict__ U,
                     const int32_t* __restrict__ cu_rows, int V, float tie_eps,
                     int32_t* __restrict__ n_acc, int32_t* __restrict__ out_tok,
                     int32_t* __restrict__ near_tie, unsigned* status) {
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int r0 = cu_rows[b];
  const int gamma = cu_rows[b + 1] - r0 - 1;
  const int q0 = r0 - b;
  const double eps = (double)tie_eps;

  __shared__ int s_n;
  __shared__ int s_near;
  __shared__ double s_part[SAMPLER_THREADS / 32];
  __shared__ double s_scan[SAMPLER_THREADS];
  __shared__ int s_pick;
  __shared__ int s_pick_near;

  // ---- 1. acceptance tests (warp 0, 32 drafts per pass)
  if (warp == 0) {
    int n = gamma;
    int near = 0;
    for (int base = 0; base < gamma; base += 32) {
      const int i = base + lane;
      bool reject = false, tie = false;
      if (i < gamma) {
        int x = draft[q0 + i];
        if (x < 0 || x >= V) {           // invalid draft token: flag it, read a valid slot
          set_status(status, 0x3F0u);
          x = x < 0 ? 0 : V - 1;
        }
        const double p = (double)P[(size_t)(r0 + i) * V + x];
        const double q = (double)Q[(size_t)(q0 + i) * V + x];
        const double uq = (double)U[r0 + i] * q;       // exact: 24 x 24 bit product
        reject = !(uq <= p);
        tie = fabs(uq - p) < eps;
      }
      const unsigned rej = __ballot_sync(0xffffffffu, reject);
      const unsigned ties = __ballot_sync(0xffffffffu, tie);
      if (rej) {
        const int first = __ffs(rej) - 1;                 // decisions 0..first were taken
        const unsigned taken = (first == 31) ? 0xffffffffu : ((1u << (first + 1)) - 1u);
        near += __popc(ties & taken);
        n = base + first;
        break;
      }
      near += __popc(ties);
    }
    if (lane == 0) {
      s_n = n;
      s_near = near;
    }
  }
  __syncthreads();
  const int n = s_n;
  const bool resid = n < gamma;
  const float* prow = P + (size_t)(r0 + n) * V;
  const float* qrow = resid ? Q + (size_t)(q0 + n) * V : nullptr;

  // ---- 2. weights: residual total (with fallback to p when it is empty)
  const int per = (V + SAMPLER_THREADS - 1) / SAMPLER_THREADS;
  const int x0 = min(V, tid * per), x1 = min(V, x0 + per);
  double local = 0.0;
  for (int x = x0; x < x1; ++x) local += row_weight(prow, qrow, x, resid, false);
  // block total via warp shuffles + shared partials
  double wsum = local;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  if (lane == 0) s_part[warp] = wsum;
  __syncthreads();
  double total = 0.0;
  for (int w = 0; w < SAMPLER_THREADS / 32; ++w) total += s_part[w];
  const bool fallback = resid && !(total > 0.0);
  if (fallback) {
    __syncthreads();
    local = 0.0;
    for (int x = x0; x < x1; ++x) local += row_weight(prow, qrow, x, resid, true);
    wsum = local;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    if (lane == 0) s_part[warp] = wsum;
    __syncthreads();
    total = 0.0;
    for (int w = 0; w < SAMPLER_THREADS / 32; ++w) total += s_part[w];
  }

  // ---- 3. inclusive scan of slice sums (Hillis-Steele in shared memory)
  s_scan[tid] = local;
  if (tid == 0) {
    s_pick = -1;
    s_pick_near = 0;
  }
  __syncthreads();
  for (int off = 1; off < SAMPLER_THREADS; off <<= 1) {
    const double v = tid >= off ? s_scan[tid - off] : 0.0;
    __syncthreads();
    s_scan[tid] += v;
    __syncthreads();
  }
  const double thr = (double)U[r0 + gamma] * total;
  const double incl = s_scan[tid];
  const double excl = tid > 0 ? s_scan[tid - 1] : 0.0;
  if (excl <= thr && incl > thr) {
    // this slice holds the first token whose CDF exceeds thr
    double cum = excl, lo = excl;
    int pick = -1, last_pos = -1;
    for (int x = x0; x < x1; ++x) {
      const double w = row_weight(prow, qrow, x, resid, fallback);
      lo = cum;
      cum += w;
      if (w > 0.0) last_pos = x;
      if (cum > thr) {
        pick = x;
        break;
      }
    }
    const double band = eps * total;
    if (pick >= 0) {
      s_pick = pick;
      s_pick_near = (fabs(cum - thr) < band || (pick > 0 && fabs(lo - thr) < band)) ? 1 : 0;
    } else if (last_pos >= 0) {
      // the walk's rounding stayed just below thr: the crossing is at the slice end
      s_pick = last_pos;
      s_pick_near = 1;
    }
  }
  __syncthreads();

  if (tid == 0) {
    const int t = s_pick >= 0 ? s_pick : V - 1;   // no positive weight at all: last token
    n_acc[b] = n;
    near_tie[b] = s_near + s_pick_near;
    out_tok[r0 + n] = t;
  }
  for (int k = tid; k <= gamma; k += SAMPLER_THREADS) {
    if (k < n) out_tok[r0 + k] = draft[q0 + k];
    else if (k > n) out_tok[r0 + k] = -1;
  }
}

}  // namespace

cudaError_t launch_reject_sample(const float* P, const float* Q, const int32_t* draft,
                                 const float* U, const int32_t* cu_rows, int B, int V,
                                 float tie_eps, int32_t* n_acc, int32_t* out_tok,
                                 int32_t* near_tie, unsigned* status, cudaStream_t s) {
  reject_sample_kernel<<<B, SAMPLER_THREADS, 0, s>>>(P, Q, draft, U, cu_rows, V, tie_eps, n_acc,
                                                     out_tok, near_tie, status);
  return cudaGetLastError();
}

}  // namespace spec
