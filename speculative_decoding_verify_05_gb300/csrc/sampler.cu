// Rejection sampler: one CTA per sequence.
//
// Steps (Algorithm 1 on "Speculative Decoding Spends Arithmetic You May Not
// Have", section "What one iteration actually does"):
//   1. warp 0 evaluates all gamma_b acceptance tests at once (lane i: draft
//      i), in fp64 so that u*q is exact; n = first rejection (ballot), else
//      gamma_b;
//   2. the block builds the final weights w(x) = max(0, p - q) at the first
//      rejection (p itself if that is all zero), or w = p_{gamma+1} (bonus), in
//      fp32 (exact sign, <= 2^-24 relative rounding per weight), and sums them
//      per 4096-token tile with the tile totals kept in fp64;
//   3. inverse CDF in token order: the fp64 prefix over tile totals finds the
//      tile that crosses u * sum(w); inside it the 8-token slice sums are
//      scanned (fp32 within a warp, fp64 across warps) and the thread whose
//      slice crosses walks it in fp64.  Weights and sums carry ~1e-7 relative
//      rounding, far inside the near-tie band (tie_eps, 1e-5 by default), so a
//      pick differs from an exact fp64 one only where it is counted as a near
//      tie.  (An all-fp64 pass is ~2 fp64 FMA/clock/SM here: 0.3 ms a round.)
//
// The probabilities come either as a materialised p [M x V] (spec_reject_sample) or, for the
// fused LM-head -> sampler path (spec_lmhead_reject_sample), as the LM head's logits z / T and
// per-tile statistics: p_x = exp_sm(z_x - max) * inv with the row's normaliser computed here by
// the same code as the normalisation kernel (bit-identical p; one warp per row, 16 rows at a
// time), or a one-hot row at the argmax when the temperature is 0.  Only the rows the sampler
// reads are ever evaluated.
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "lmhead_norm.cuh"

namespace spec {
namespace {

constexpr int SAMPLER_THREADS = 512;
constexpr int PER_THREAD = 8;                              // consecutive tokens per thread in a tile
constexpr int TILE = SAMPLER_THREADS * PER_THREAD;         // 4096 tokens
constexpr int MAX_TILES = 256;                             // V <= 1,048,576

// Where a row's probabilities come from.
enum { P_GIVEN = 0, P_LOGITS = 1, P_ARGMAX = 2 };
struct RowP {
  const float* v;   // P_GIVEN: the p row; P_LOGITS: the z / T row
  float mx, inv;    // P_LOGITS: p_x = exp_sm(z_x - mx) * inv
  int am;           // P_ARGMAX: p_x = (x == am)
};
template <int MODE>
__device__ __forceinline__ float p_at(const RowP& r, int x) {
  if constexpr (MODE == P_GIVEN) return r.v[x];
  else if constexpr (MODE == P_LOGITS) return exp_sm(r.v[x] - r.mx) * r.inv;
  else return x == r.am ? 1.f : 0.f;
}

// This thread's 8 consecutive weights of a tile: w = max(0, p - q) at a rejection (the sign is
// exact in fp32; the value carries <= 2^-24 relative rounding), p itself for the bonus row or
// when the residual is empty (`use_p`).  Tokens past V weigh 0.
template <int MODE>
__device__ __forceinline__ void load_weights(const RowP& pr, const float* qrow, int x0, int V, bool use_p,
                                             bool vec, float* w) {
  if (vec && x0 + PER_THREAD <= V) {
    if constexpr (MODE == P_ARGMAX) {
#pragma unroll
      for (int e = 0; e < PER_THREAD; ++e) w[e] = (x0 + e == pr.am) ? 1.f : 0.f;
    } else {
      const float4 p0 = __ldcg(reinterpret_cast<const float4*>(pr.v + x0));
      const float4 p1 = __ldcg(reinterpret_cast<const float4*>(pr.v + x0 + 4));
      w[0] = p0.x; w[1] = p0.y; w[2] = p0.z; w[3] = p0.w; w[4] = p1.x; w[5] = p1.y; w[6] = p1.z; w[7] = p1.w;
      if constexpr (MODE == P_LOGITS) {
#pragma unroll
        for (int e = 0; e < PER_THREAD; ++e) w[e] = exp_sm(w[e] - pr.mx) * pr.inv;
      }
    }
    if (!use_p) {
      const float4 q0 = __ldcg(reinterpret_cast<const float4*>(qrow + x0));
      const float4 q1 = __ldcg(reinterpret_cast<const float4*>(qrow + x0 + 4));
      const float q[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
      for (int e = 0; e < PER_THREAD; ++e) w[e] = fmaxf(w[e] - q[e], 0.f);
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < PER_THREAD; ++e) {
    const int x = x0 + e;
    float v = 0.f;
    if (x < V) {
      v = p_at<MODE>(pr, x);
      if (!use_p) v = fmaxf(v - qrow[x], 0.f);
    }
    w[e] = v;
  }
}

// P: p [M x V] (P_GIVEN) or z / T [M x V] (P_LOGITS, unused for P_ARGMAX); stats: the LM head's
// per-tile statistics [M][n_stats] (P_LOGITS, P_ARGMAX).
// TYPICAL: the lossy accept rule instead of step 1 ("How Speculative Decoding Works (and When It
// Doesn't)", "Exactness is a choice"): keep x_i iff p_i(x_i) > max(t_eps, t_delta * e^(-H_i)),
// H_i the entropy of row i, stop at the first failure; the final token is drawn from the target
// row p_{n+1} itself (no residual).  Q is not read.
template <int MODE, bool TYPICAL>
__global__ void __launch_bounds__(SAMPLER_THREADS)
reject_sample_kernel(const float* __restrict__ P, const float2* __restrict__ stats, int n_stats,
                     const float* __restrict__ Q,
                     const int32_t* __restrict__ draft, const float* __restrict__ U,
                     const int32_t* __restrict__ cu_rows, int V, float tie_eps,
                     int32_t* __restrict__ n_acc, int32_t* __restrict__ out_tok,
                     int32_t* __restrict__ near_tie, unsigned* status, int vec, int m_rows,
                     float t_eps, float t_delta, long long ldp) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // cu_rows == nullptr: one row per sequence and no drafts (plain sampling of row b)
  const int r0 = cu_rows ? cu_rows[b] : b;
  const int gamma = cu_rows ? cu_rows[b + 1] - r0 - 1 : 0;
  if (r0 < 0 || gamma < 0 || r0 + gamma + 1 > m_rows) {   // rows outside the verify pass's M rows
    if (tid == 0) {
      set_status(status, 0x3F1u);
      if (n_acc) n_acc[b] = 0;
      if (near_tie) near_tie[b] = 0;
    }
    return;
  }
  const int q0 = r0 - b;
  const double eps = (double)tie_eps;
  const int n_tiles = (V + TILE - 1) / TILE;

  __shared__ int s_n, s_near, s_pick, s_pick_near, s_first;
  __shared__ float s_wp[SAMPLER_THREADS / 32][2];          // per-warp sums (residual, p)
  __shared__ double s_tile_r[MAX_TILES], s_tile_p[MAX_TILES];
  __shared__ float s_part_r[MAX_TILES * (SAMPLER_THREADS / 32)], s_part_p[MAX_TILES * (SAMPLER_THREADS / 32)];
  __shared__ double s_wexcl[SAMPLER_THREADS / 32];
  __shared__ float s_mx[32], s_inv[32];
  __shared__ int s_am[32], s_done;

  // ---- 1. acceptance tests, 32 drafts per pass (warp 0), exact in fp64; rows base .. base + 31
  // (and the final row, which is one of them) get their normaliser first when p is not given
  if (tid == 0) {
    s_n = gamma;
    s_near = 0;
    s_done = 0;
  }
  __syncthreads();
  int base = 0;
  if constexpr (TYPICAL) {
    // one draft row at a time: block-wide entropy pass (fp32 terms, fp64 across warps), then the
    // threshold test by thread 0; the loop ends at the first draft that fails
    for (int i = 0; i < gamma; ++i) {
      const RowP pr{P + (size_t)(r0 + i) * ldp, 0.f, 0.f, 0};
      float h = 0.f;
      for (int x0 = tid * PER_THREAD; x0 < V; x0 += TILE) {
        float w[PER_THREAD];
        load_weights<MODE>(pr, pr.v, x0, V, true, vec, w);
#pragma unroll
        for (int e = 0; e < PER_THREAD; ++e) h -= w[e] > 0.f ? w[e] * logf(w[e]) : 0.f;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) h += __shfl_xor_sync(0xffffffffu, h, o);
      if (lane == 0) s_wp[warp][1] = h;
      __syncthreads();
      if (tid == 0) {
        double H = 0.0;
        for (int k = 0; k < SAMPLER_THREADS / 32; ++k) H += (double)s_wp[k][1];
        const double tau = fmax((double)t_eps, (double)t_delta * exp(-H));
        int x = draft[q0 + i];
        if (x < 0 || x >= V) {           // invalid draft token: flag it, read a valid slot
          set_status(status, 0x3F0u);
          x = x < 0 ? 0 : V - 1;
        }
        const double px = (double)p_at<MODE>(pr, x);
        if (fabs(px - tau) < eps) ++s_near;
        if (!(px > tau)) {
          s_n = i;
          s_done = 1;
        }
      }
      __syncthreads();
      if (s_done) break;
    }
  } else
  for (;; base += 32) {
    const int rows = min(32, gamma + 1 - base);
    // one warp per row: 16 rows at a time
    if constexpr (MODE == P_LOGITS) {
      for (int j = warp; j < rows; j += SAMPLER_THREADS / 32) {
        float mx, inv;
        lm_row_norm_warp(stats + (size_t)(r0 + base + j) * n_stats, n_stats, mx, inv);
        if (lane == 0) { s_mx[j] = mx; s_inv[j] = inv; }
      }
    } else if constexpr (MODE == P_ARGMAX) {
      for (int j = warp; j < rows; j += SAMPLER_THREADS / 32) {
        const int am = lm_row_argmax_warp(stats + (size_t)(r0 + base + j) * n_stats, n_stats);
        if (lane == 0) s_am[j] = am;
      }
    }
    __syncthreads();
    if (warp == 0) {
      const int i = base + lane;
      bool reject = false, tie = false;
      if (i < gamma) {
        int x = draft[q0 + i];
        if (x < 0 || x >= V) {           // invalid draft token: flag it, read a valid slot
          set_status(status, 0x3F0u);
          x = x < 0 ? 0 : V - 1;
        }
        const RowP pr{P + (size_t)(r0 + i) * ldp, s_mx[lane], s_inv[lane], s_am[lane]};
        const double p = (double)p_at<MODE>(pr, x);
        const double q = (double)Q[(size_t)(q0 + i) * V + x];
        const double uq = (double)U[r0 + i] * q;       // exact: 24 x 24 bit product
        reject = !(uq <= p);
        tie = fabs(uq - p) < eps;
      }
      const unsigned rej = __ballot_sync(0xffffffffu, reject);
      const unsigned ties = __ballot_sync(0xffffffffu, tie);
      if (lane == 0) {
        if (rej) {
          const int first = __ffs(rej) - 1;                 // decisions 0..first were taken
          const unsigned taken = (first == 31) ? 0xffffffffu : ((1u << (first + 1)) - 1u);
          s_near += __popc(ties & taken);
          s_n = base + first;
          s_done = 1;
        } else {
          s_near += __popc(ties);
          if (base + 32 > gamma) s_done = 1;             // every draft accepted: n = gamma
        }
      }
    }
    __syncthreads();
    if (s_done) break;
  }
  const int n = s_n;
  const bool resid = !TYPICAL && n < gamma;
  const int ri = (MODE == P_GIVEN) ? 0 : n - base;   // the final row's normaliser slot
  const RowP prow{P + (size_t)(r0 + n) * ldp, s_mx[ri], s_inv[ri], s_am[ri]};
  const float* qrow = resid ? Q + (size_t)(q0 + n) * V : prow.v;

  // ---- 2. per-tile totals of the residual and of p, kept in fp64: each thread reads its 8 tokens of
  // the final row (and of q at a rejection) once per tile, the 16-byte loads of four tiles issued
  // before any of them is used (no block barrier per tile)
  for (int t0 = 0; t0 < n_tiles; t0 += 4) {
    float4 zr[4][2], qr[4][2];
    bool full[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int x0 = (t0 + k) * TILE + tid * PER_THREAD;
      full[k] = vec && t0 + k < n_tiles && x0 + PER_THREAD <= V;
      zr[k][0] = zr[k][1] = qr[k][0] = qr[k][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (full[k]) {
        if constexpr (MODE != P_ARGMAX) {
          zr[k][0] = __ldcg(reinterpret_cast<const float4*>(prow.v + x0));
          zr[k][1] = __ldcg(reinterpret_cast<const float4*>(prow.v + x0 + 4));
        }
        if (resid) {
          qr[k][0] = __ldcg(reinterpret_cast<const float4*>(qrow + x0));
          qr[k][1] = __ldcg(reinterpret_cast<const float4*>(qrow + x0 + 4));
        }
      }
    }
    float sr[4], sp[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      sr[k] = 0.f;
      sp[k] = 0.f;
      const int t = t0 + k;
      if (t >= n_tiles) continue;
      const int x0 = t * TILE + tid * PER_THREAD;
      // p and the residual weights max(0, p - q) of this thread's tokens (tokens past V weigh 0)
      float pv[PER_THREAD], qv[PER_THREAD];
      if (full[k]) {
        const float zz[PER_THREAD] = {zr[k][0].x, zr[k][0].y, zr[k][0].z, zr[k][0].w,
                                      zr[k][1].x, zr[k][1].y, zr[k][1].z, zr[k][1].w};
        const float qq[PER_THREAD] = {qr[k][0].x, qr[k][0].y, qr[k][0].z, qr[k][0].w,
                                      qr[k][1].x, qr[k][1].y, qr[k][1].z, qr[k][1].w};
#pragma unroll
        for (int e = 0; e < PER_THREAD; ++e) {
          if constexpr (MODE == P_ARGMAX) pv[e] = (x0 + e == prow.am) ? 1.f : 0.f;
          else if constexpr (MODE == P_LOGITS) pv[e] = exp_sm(zz[e] - prow.mx) * prow.inv;
          else pv[e] = zz[e];
          qv[e] = qq[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < PER_THREAD; ++e) {
          const int x = x0 + e;
          pv[e] = x < V ? p_at<MODE>(prow, x) : 0.f;
          qv[e] = (resid && x < V) ? qrow[x] : 0.f;
        }
      }
#pragma unroll
      for (int e = 0; e < PER_THREAD; ++e) sp[k] += pv[e];
      if (resid) {
#pragma unroll
        for (int e = 0; e < PER_THREAD; ++e) sr[k] += fmaxf(pv[e] - qv[e], 0.f);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sr[k] += __shfl_xor_sync(0xffffffffu, sr[k], o);
        sp[k] += __shfl_xor_sync(0xffffffffu, sp[k], o);
      }
      if (lane == 0 && t0 + k < n_tiles) {
        s_part_r[(t0 + k) * (SAMPLER_THREADS / 32) + warp] = sr[k];
        s_part_p[(t0 + k) * (SAMPLER_THREADS / 32) + warp] = sp[k];
      }
    }
  }
  __syncthreads();
  for (int t = tid; t < n_tiles; t += SAMPLER_THREADS) {
    double tr = 0.0, tp = 0.0;
    for (int k = 0; k < SAMPLER_THREADS / 32; ++k) {
      tr += (double)s_part_r[t * (SAMPLER_THREADS / 32) + k];
      tp += (double)s_part_p[t * (SAMPLER_THREADS / 32) + k];
    }
    s_tile_r[t] = tr;
    s_tile_p[t] = tp;
  }
  __syncthreads();

  // ---- 3. crossing tile of u * total (fp64 prefix over the tiles); empty residual -> p
  __shared__ double s_thr, s_total, s_tile_excl;
  __shared__ int s_tile, s_use_p;
  if (tid == 0) {
    double tot_r = 0.0, tot_p = 0.0;
    for (int t = 0; t < n_tiles; ++t) {
      tot_r += s_tile_r[t];
      tot_p += s_tile_p[t];
    }
    const bool use_p = !resid || !(tot_r > 0.0);
    const double* tiles = use_p ? s_tile_p : s_tile_r;
    const double total = use_p ? tot_p : tot_r;
    const double thr = (double)U[r0 + gamma] * total;
    double excl = 0.0;
    int tc = -1, last_pos = -1;
    double last_excl = 0.0;
    for (int t = 0; t < n_tiles; ++t) {
      if (tiles[t] > 0.0) { last_pos = t; last_excl = excl; }
      if (tc < 0 && excl + tiles[t] > thr) { tc = t; s_tile_excl = excl; }
      excl += tiles[t];
    }
    if (tc < 0) { tc = last_pos; s_tile_excl = last_excl; }   // rounding left thr at the very end
    s_tile = tc;
    s_use_p = use_p ? 1 : 0;
    s_thr = thr;
    s_total = total;
    s_pick = -1;
    s_pick_near = 0;
    s_first = SAMPLER_THREADS;
  }
  __syncthreads();

  // ---- 4. inside the crossing tile: block scan of the 8-token slice sums, then one thread walks
  const int tc = s_tile;
  if (tc >= 0) {
    const bool use_p = s_use_p != 0;
    const double thr = s_thr;
    const int x0 = tc * TILE + tid * PER_THREAD;
    float w[PER_THREAD];
    load_weights<MODE>(prow, qrow, x0, V, use_p, vec, w);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < PER_THREAD; ++e) s += w[e];
    float incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    float excl_w = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl_w = 0.f;
    if (lane == 31) s_wp[warp][0] = incl;
    __syncthreads();
    if (tid == 0) {
      double acc = s_tile_excl;
      for (int k = 0; k < SAMPLER_THREADS / 32; ++k) {
        s_wexcl[k] = acc;
        acc += (double)s_wp[k][0];
      }
    }
    __syncthreads();
    const double t_excl = s_wexcl[warp] + (double)excl_w;
    const double t_incl = s_wexcl[warp] + (double)incl;
    if (t_incl > thr) atomicMin(&s_first, tid);
    __syncthreads();
    int walker = s_first;
    if (walker == SAMPLER_THREADS) {
      // rounding kept every prefix at or below thr: the last thread with weight walks
      if (s > 0.f) atomicMax(&s_pick, tid);        // s_pick is -1 here: reuse it as "last positive"
      __syncthreads();
      walker = s_pick;
      __syncthreads();
      if (tid == 0) s_pick = -1;
      __syncthreads();
    }
    if (tid == walker) {
      const double band = eps * s_total;
      double cum = t_excl, lo = t_excl;
      int pick = -1, last_pos = -1;
#pragma unroll
      for (int e = 0; e < PER_THREAD; ++e) {
        if (pick >= 0) break;
        lo = cum;
        cum += (double)w[e];
        if (w[e] > 0.f) last_pos = x0 + e;
        if (cum > thr) pick = x0 + e;
      }
      if (pick >= 0) {
        s_pick = pick;
        s_pick_near = (fabs(cum - thr) < band || (pick > 0 && fabs(lo - thr) < band)) ? 1 : 0;
      } else if (last_pos >= 0) {
        // the walk's rounding stayed just below thr: the crossing is at the slice end
        s_pick = last_pos;
        s_pick_near = 1;
      }
    }
  }
  __syncthreads();

  if (tid == 0) {
    const int t = s_pick >= 0 ? s_pick : V - 1;   // no positive weight at all: last token
    if (n_acc) n_acc[b] = n;
    if (near_tie) near_tie[b] = s_near + s_pick_near;
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
  const bool vec = V % 4 == 0 && (reinterpret_cast<uintptr_t>(P) & 15) == 0 && (reinterpret_cast<uintptr_t>(Q) & 15) == 0;
  cudaError_t e = launch_k(reject_sample_kernel<P_GIVEN, false>, dim3(B), dim3(SAMPLER_THREADS), 0, s, P,
                           static_cast<const float2*>(nullptr), 0, Q, draft, U, cu_rows, V, tie_eps, n_acc,
                           out_tok, near_tie, status, vec ? 1 : 0, INT_MAX, 0.f, 0.f, (long long)V);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_reject_sample_logits(const float* Z, const float2* stats, int n_stats, bool greedy,
                                        const float* Q, const int32_t* draft, const float* U,
                                        const int32_t* cu_rows, int B, int M, int V, float tie_eps,
                                        int32_t* n_acc, int32_t* out_tok, int32_t* near_tie, unsigned* status,
                                        cudaStream_t s) {
  const bool vec = V % 4 == 0 && (greedy || (reinterpret_cast<uintptr_t>(Z) & 15) == 0) &&
                   (reinterpret_cast<uintptr_t>(Q) & 15) == 0;
  cudaError_t e = greedy
      ? launch_k(reject_sample_kernel<P_ARGMAX, false>, dim3(B), dim3(SAMPLER_THREADS), 0, s, Z, stats, n_stats, Q,
                 draft, U, cu_rows, V, tie_eps, n_acc, out_tok, near_tie, status, vec ? 1 : 0, M, 0.f, 0.f,
                 (long long)V)
      : launch_k(reject_sample_kernel<P_LOGITS, false>, dim3(B), dim3(SAMPLER_THREADS), 0, s, Z, stats, n_stats, Q,
                 draft, U, cu_rows, V, tie_eps, n_acc, out_tok, near_tie, status, vec ? 1 : 0, M, 0.f, 0.f,
                 (long long)V);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_typical_sample(const float* P, const int32_t* draft, const float* U, const int32_t* cu_rows,
                                  int B, int V, float t_eps, float t_delta, float tie_eps, int32_t* n_acc,
                                  int32_t* out_tok, int32_t* near_tie, unsigned* status, cudaStream_t s) {
  const bool vec = V % 4 == 0 && (reinterpret_cast<uintptr_t>(P) & 15) == 0;
  cudaError_t e = launch_k(reject_sample_kernel<P_GIVEN, true>, dim3(B), dim3(SAMPLER_THREADS), 0, s, P,
                           static_cast<const float2*>(nullptr), 0, static_cast<const float*>(nullptr), draft, U,
                           cu_rows, V, tie_eps, n_acc, out_tok, near_tie, status, vec ? 1 : 0, INT_MAX, t_eps,
                           t_delta, (long long)V);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_sample_rows(const float* P, long long ldp, int M, int V, const float* U, int32_t* out_tok,
                               unsigned* status, cudaStream_t s) {
  const bool vec = V % 4 == 0 && ldp % 4 == 0 && (reinterpret_cast<uintptr_t>(P) & 15) == 0;
  cudaError_t e = launch_k(reject_sample_kernel<P_GIVEN, false>, dim3(M), dim3(SAMPLER_THREADS), 0, s, P,
                           static_cast<const float2*>(nullptr), 0, static_cast<const float*>(nullptr),
                           static_cast<const int32_t*>(nullptr), U, static_cast<const int32_t*>(nullptr), V, 0.f,
                           static_cast<int32_t*>(nullptr), out_tok, static_cast<int32_t*>(nullptr), status,
                           vec ? 1 : 0, M, 0.f, 0.f, ldp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace spec
