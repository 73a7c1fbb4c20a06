// n-gram prompt-lookup drafter: the weightless drafter of "05 · Speculative Decoding" ("Under
// the Hood", N-gram row: it matches the recent context against earlier text and copies what
// followed; "Cheat Sheet": k and the window prompt_lookup_min / prompt_lookup_max).
//
// One CTA per sequence.  The last min(L, n_max) tokens of the history go to shared memory.  For
// n = n_max down to n_min the block scans the starts j of earlier occurrences of the last n
// tokens from the most recent one down (j <= L - 1 - n, so at least one token follows and the
// pattern itself is excluded), 256 starts per step with coalesced reads; the first step that
// holds a match holds the latest one (block OR, then a shared max).  The drafts are the up to k
// tokens after it.  Pure integer work, bounded loops, no waits.
#include "common.cuh"
#include "internal.h"

namespace spec {
namespace {

constexpr int NG_THREADS = 256;

__global__ void __launch_bounds__(NG_THREADS)
ngram_propose_kernel(const int32_t* __restrict__ tokens, const int32_t* __restrict__ cu_len, int k, int n_min,
                     int n_max, int32_t* __restrict__ drafts, int32_t* __restrict__ n_drafts, unsigned* status) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int h0 = cu_len[b];
  const int L = cu_len[b + 1] - h0;
  __shared__ int32_t s_pat[NGRAM_MAX_WINDOW];
  __shared__ int s_best, s_n;
  int32_t* out = drafts + (size_t)b * k;
  if (h0 < 0 || L < 0) {                 // malformed offsets: no drafts, flag it
    if (tid == 0) {
      set_status(status, 0x4F0u);
      n_drafts[b] = 0;
    }
    for (int t = tid; t < k; t += NG_THREADS) out[t] = -1;
    return;
  }
  const int32_t* h = tokens + h0;
  const int m = L < n_max ? L : n_max;   // pattern tokens kept: s_pat[m - n + t] = h[L - n + t]
  for (int t = tid; t < m; t += NG_THREADS) s_pat[t] = h[L - m + t];
  if (tid == 0) {
    s_best = -1;
    s_n = 0;
  }
  __syncthreads();
  for (int n = n_max; n >= n_min; --n) {
    if (L - 1 - n < 0) continue;
    const int32_t* pat = s_pat + (m - n);
    bool done = false;
    for (int top = L - 1 - n; top >= 0; top -= NG_THREADS) {
      const int j = top - tid;
      bool hit = false;
      if (j >= 0) {
        hit = true;
        for (int t = 0; t < n; ++t)
          if (h[j + t] != pat[t]) { hit = false; break; }
      }
      if (__syncthreads_or(hit)) {
        if (hit) atomicMax(&s_best, j);
        if (tid == 0) s_n = n;
        __syncthreads();
        done = true;
        break;
      }
    }
    if (done) break;
  }
  const int j = s_best, n = s_n;
  const int avail = j >= 0 ? L - (j + n) : 0;
  const int cnt = avail < k ? avail : k;
  for (int t = tid; t < k; t += NG_THREADS) out[t] = t < cnt ? h[j + n + t] : -1;
  if (tid == 0) n_drafts[b] = cnt;
}

}  // namespace

cudaError_t launch_ngram_propose(const int32_t* tokens, const int32_t* cu_len, int B, int k, int n_min, int n_max,
                                 int32_t* drafts, int32_t* n_drafts, unsigned* status, cudaStream_t s) {
  cudaError_t e = launch_k(ngram_propose_kernel, dim3(B), dim3(NG_THREADS), 0, s, tokens, cu_len, k, n_min, n_max,
                           drafts, n_drafts, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace spec
