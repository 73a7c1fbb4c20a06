// C ABI of the verify library: argument checks, launch planning (tile widths,
// split-K, key chunks), TMA tensor-map encoding and dispatch to the kernels.
// Nothing here allocates device memory; workspaces come from the caller.
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>
#include <algorithm>

#include "../../include/spec_verify.h"
#include "common.cuh"
#include "internal.h"

using namespace spec;

// Library status word: a bounded device wait that runs out records its site here.
__device__ unsigned g_spec_status;

namespace {

constexpr int kVersion = 1;
thread_local std::string t_err;
thread_local int t_launches = 0;   // kernels the last call on this thread launched

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  t_launches = 0;
  return code;
}
int ok(int launched = 0) {
  t_err.clear();
  t_launches = launched;
  return SPEC_OK;
}
int cuda_fail(cudaError_t e, const char* what) {
  return fail(SPEC_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The current thread's CUDA context (the driver's handle).  Device addresses of the library's
// __device__ variables are cached per context: a device reset (cudaDeviceReset) destroys the
// context and reloads the module, so its next context gets the addresses looked up afresh.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn g_ctx_get = nullptr;
std::once_flag g_ctx_once;

// *ctx = the current context, or NULL when the runtime has not made one current yet.
int current_context(CUcontext* ctx) {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get = reinterpret_cast<CtxGetCurrentFn>(fn);
  });
  if (!g_ctx_get) return fail(SPEC_ECUDA, "cuCtxGetCurrent entry point unavailable");
  *ctx = nullptr;
  if (g_ctx_get(ctx) != CUDA_SUCCESS) return fail(SPEC_ECUDA, "cuCtxGetCurrent failed");
  return SPEC_OK;
}

// Device address of one of the library's __device__ variables in the current context, cached in
// (*cached_ctx, *cached_ptr).  cudaGetSymbolAddress makes the device's primary context current when
// none is yet, so the context is read again after it.
template <typename T>
int symbol_address(const T& symbol, const char* what, CUcontext* cached_ctx, void** cached_ptr) {
  CUcontext ctx = nullptr;
  if (int rc = current_context(&ctx)) return rc;
  if (ctx && ctx == *cached_ctx && *cached_ptr) return SPEC_OK;
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, symbol);
  if (e != cudaSuccess) return cuda_fail(e, what);
  if (int rc = current_context(&ctx)) return rc;
  if (!ctx) return fail(SPEC_ECUDA, "no current CUDA context after %s", what);
  *cached_ctx = ctx;
  *cached_ptr = p;
  return SPEC_OK;
}

struct DevInfo {
  int sms = 0;
  CUcontext ctx = nullptr;     // the context `status` belongs to
  void* status_ptr = nullptr;
  unsigned* status = nullptr;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

int dev_info(DevInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(SPEC_EUNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.sms == 0) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  }
  if (int rc = symbol_address(g_spec_status, "cudaGetSymbolAddress(status)", &d.ctx, &d.status_ptr)) return rc;
  d.status = static_cast<unsigned*>(d.status_ptr);
  *out = &d;
  return SPEC_OK;
}

// sm count for planning without touching the device (workspace queries may
// run before any context exists): falls back to the GB300's 152.
int plan_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_dev[dev].sms > 0) return g_dev[dev].sms;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      return n;
  }
  cudaGetLastError();
  return 152;
}

// --------------------------------------------------------------------------- TMA
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(SPEC_ECUDA, "cuTensorMapEncodeTiled entry point unavailable");
  return SPEC_OK;
}

// bf16 tensor map with 128-byte swizzle; dims/strides innermost first (strides in bytes, rank-1 entries)
constexpr CUtensorMapSwizzle kLinSwizzle = LIN_BK == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
int g_w_promotion = 3;    // tunable: L2 promotion of weight-tile loads (0 none, 1 64 B, 2 128 B, 3 256 B)
int g_kv_promotion = 3;   // tunable: L2 promotion of the attention kernels' K/V tile loads (same scale)

int encode_bf16(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                const cuuint64_t* strides, const cuuint32_t* box, const char* what,
                int promotion = 3, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  if (int rc = get_encoder()) return rc;
  cuuint32_t estr[3] = {1, 1, 1};
  static const CUtensorMapL2promotion kPromo[4] = {
      CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
      CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, kPromo[promotion & 3],
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPEC_ECUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
  return SPEC_OK;
}

// --------------------------------------------------------------------------- workspace layout
// Every workspace starts with a fixed counter region that kernels leave at
// zero; scratch (fp32 partials, statistics) follows.  Because the counters
// always sit at the same place, one zero-filled workspace can serve any
// sequence of calls on one stream, whatever their shapes.
constexpr size_t kCounterBytes = 64 * 1024;
constexpr size_t kMaxCounters = kCounterBytes / 4;

// --------------------------------------------------------------------------- linear plan
int g_gemv_max_m = 0;    // tunable: largest M that takes the CUDA-core path (0: tensor cores for every M)
int g_attn_impl = 1;     // tunable: 0 = mma.sync kernel, 1 = tcgen05 kernel
int g_attn_pair_cost = 12;  // tunable: tcgen05 attention work charged per pair start, quarter tiles
int g_force_grid = 0;    // tunable: CTAs of the persistent kernels, 0 = one per SM
int g_linear_cluster = 1;  // tunable: 0 disables the cluster split-K GEMM
int g_linear_split_rows = 1;  // tunable: 1 lets few-tile products at 257..384 rows take two half-row tiles
int g_weight_prefetch = 1;  // tunable: 1 loads the first weight tiles before the dependency wait
int g_nsub_max = 2;      // tunable: 2 lets one CTA tile cover up to 384 verify rows
int g_lmhead_nsub = 2;   // tunable: the LM head's tiles cover up to 256 (1) or 384 (2) rows
int g_pdl = 1;           // tunable: programmatic dependent launch between the library's kernels
int g_linear_pair = 1;   // tunable: 1 lets the planner run 256-row pair tiles on the 2-SM MMA
int g_linear_pair_few = 0;  // tunable: 1 also for products with fewer tiles than SMs (split-K on pairs)
// tunable: products with more tiles than SMs on the persistent kernel on CTA pairs: 1 = whole pair
// tiles, then stream-K pieces summed by the reduce kernel; 2 = whole pair tiles, then the rest on
// the pair split-K kernel; 0 = off (whole pair tiles, then the rest, each as a launch of the pair
// split-K kernel: measured fastest for gate|up at 368 rows, 63.2 us against 64.8 and 74.5)
int g_linear_pair_persistent = 0;
int g_lmhead_pair = 1;     // tunable: 1 runs the LM head on the persistent kernel on CTA pairs

struct LinPlan {
  bool gemv = false;
  int BN = 16, NSUB = 1, tiles_m = 1, tiles_n = 1, k_tiles = 1, splits = 1;
  int grid = 1;                 // persistent CTAs of the tensor-core path
  int cluster_S = 0;            // > 0: cluster split-K kernel, S CTAs per tile
  int rem_S = 0;                // > 0: whole tiles on the persistent kernel, then the remaining
  long long rem_tiles = 0;      //      rem_tiles on the cluster split-K kernel (S = rem_S)
  int pair_n = 0;               // > 0: launches of the 2-SM pair kernel, launch i covering pair
  int pair_first[2] = {0, 0};   //      tiles pair_first[i] .. + pair_count[i] - 1 with pair_S[i]
  int pair_count[2] = {0, 0};   //      pairs per tile
  int pair_S[2] = {0, 0};
  bool tc_pair = false;          // persistent kernel on CTA pairs: grid counts pairs, dp_tiles and
                                //   sk_units count 256-row pair tiles; pair_n = 1 adds a pair
                                //   split-K launch for the pair tiles after dp_tiles
  // token rows per TMA load: each CTA of a pair stages half of every MMA's token rows
  int x_box_rows() const { return pair_n > 0 || tc_pair ? BN / 2 : BN; }
  bool aligned = false;         // whole tiles only (no stream-K region)
  long long dp_tiles = 0, sk_units = 0;
  long long units = 0;
  int gemv_grid = 1, k_per_split = 0, groups = 0;
  size_t counters_off = 0, partial_off = 0, bytes = 0;
};

// The smallest token-tile width >= BN with a build of the persistent pair kernel (0: none).
int tc_pair_bn(int BN, int NSUB) {
  static const int shapes[][2] = {
#define X(bn, ns) {bn, ns},
      SPEC_TC_PAIR_SHAPES(X)
#undef X
  };
  int best = 0;
  for (const auto& sh : shapes)
    if (sh[1] == NSUB && sh[0] >= BN && (best == 0 || sh[0] < best)) best = sh[0];
  return best;
}

// A cluster split-K plan on one two-MMA tile of 257..384 rows, or two one-MMA tiles of half the
// rows?  After the main loop each CTA of an S-way cluster moves (S - 1) / S of its 128 x TN fp32
// accumulator through distributed shared memory, which is slow (tens of GB/s per SM); half-row
// tiles fill the same SMs with half the split ways, so each CTA moves about a third of the bytes,
// while a k-step keeps its whole 128-row weight tile for half the MMA work.  Model in k-steps of
// the 384-row tile: a k-step of TN rows 0.1 + 0.9 TN / 384, exchange and epilogue 11 (S - 1) / S
// TN / 384 (fitted to the O projection at 368 rows: 21.3 us on 4-way clusters of 384-row tiles,
// 17.9 us on 2-way clusters of 192-row tiles).  The half-row plan must win by 10 %: the down projection
// at 368 rows (K = 12288) models 1 % cheaper and measured within run-to-run noise of its 384-row plan.
void cluster_split_rows(LinPlan& p, int M) {
  auto model = [&](int TN, int S) {
    return double((p.k_tiles + S - 1) / S) * (0.1 + 0.9 * TN / 384.0) + 11.0 * (S - 1) / S * TN / 384.0;
  };
  const int bn1 = std::max(16, ((M + 1) / 2 + 15) / 16 * 16);
  const long long tiles1 = 2LL * p.tiles_n;
  int best = 0;
  double best_cost = 0.9 * model(p.BN * p.NSUB, p.cluster_S);
  for (int S = 2; S <= 8 && S <= p.k_tiles; ++S) {
    const int cap = linear_cluster_capacity(bn1, 1, S);
    if (cap <= 0 || tiles1 * S > cap) continue;
    const double c = model(bn1, S);
    if (c < best_cost) { best = S; best_cost = c; }
  }
  if (best == 0) return;
  p.BN = bn1;
  p.NSUB = 1;
  p.tiles_m = 2;
  p.units = tiles1 * p.k_tiles;
  p.cluster_S = best;
  p.grid = (int)(tiles1 * best);
}

LinPlan plan_linear(int M, int N, int K, bool lmhead, bool swiglu = false, size_t max_bytes = SIZE_MAX) {
  LinPlan p;
  const int sms = plan_sms();
  p.k_tiles = (K + LIN_BK - 1) / LIN_BK;
  if (!lmhead && M <= g_gemv_max_m && M <= 4) {
    p.gemv = true;
    const int ks = gemv_k_slice(M);
    p.k_per_split = ks;
    p.splits = (K + ks - 1) / ks;
    if ((size_t)(N + 3) / 4 > kMaxCounters) p.splits = 1;   // (only for N > 65536)
    p.groups = (N + 3) / 4;
    const long long items = (long long)p.groups * p.splits;
    long long grid = (items + 7) / 8;
    if (grid > (long long)sms * 8) grid = (long long)sms * 8;
    p.gemv_grid = (int)std::max(1LL, grid);
    p.counters_off = 0;
    p.partial_off = kCounterBytes;
    p.bytes = p.splits > 1 ? kCounterBytes + round_up(size_t(p.splits) * M * N * 4, 256) : 0;
    return p;
  }
  // up to 256 rows: one MMA of N = BN per k-substep; more rows: tiles of up to 384 rows as
  // two MMAs of N = BN sharing each weight tile (every weight byte still read once per tile).
  // 384 and not 512: a 512-row tile's 80 KB stage leaves room for two stages only, which
  // measured 32 % of the tensor peak at 512 rows against ~50 % with three 64 KB stages
  if (M <= kMaxBN) {
    p.tiles_m = 1;
    p.NSUB = 1;
    p.BN = std::max(16, (M + 15) / 16 * 16);
  } else if (lmhead ? g_lmhead_nsub == 1 : g_nsub_max == 1) {
    // (one MMA per k-substep; with up to 256 rows two accumulator buffers fit in TMEM, so each
    // tile's epilogue overlaps the next tile's MMAs.  The LM head takes the two-MMA tiles below by
    // default: their one accumulator leaves the epilogue exposed, but at 368 rows they read the
    // weights and tokens once per tile, and the short epilogue costs less than the second read)
    p.tiles_m = (M + kMaxBN - 1) / kMaxBN;
    const int per = (M + p.tiles_m - 1) / p.tiles_m;
    p.NSUB = 1;
    p.BN = std::max(16, (per + 15) / 16 * 16);
  } else {
    p.tiles_m = (M + kMaxTN - 1) / kMaxTN;
    const int per = (M + p.tiles_m - 1) / p.tiles_m;
    p.NSUB = 2;
    p.BN = std::max(144, ((per + 1) / 2 + 15) / 16 * 16);
  }
  const int TN = p.BN * p.NSUB;
  p.tiles_n = (N + 127) / 128;
  const long long tiles = (long long)p.tiles_m * p.tiles_n;
  p.units = tiles * p.k_tiles;
  p.counters_off = 0;
  p.partial_off = kCounterBytes;
  // persistent stream-K: one CTA per SM, each streaming an equal share of (tile, k-step) units;
  // the LM-head epilogue needs whole tiles, so its ranges are tile-aligned
  p.aligned = lmhead || tiles > (long long)kMaxCounters;
  // Many tiles (and the LM head): the persistent kernel on CTA pairs, 256-row pair tiles on the 2-SM
  // MMA, each CTA staging half of the token rows (which halves the shared-memory traffic per MMA
  // that bounds the one-SM kernels at a few hundred rows).  Whole pair tiles go round-robin to the
  // pairs; the pair tiles left over are cut into stream-K pieces (summed by the reduce kernel) or
  // run on the pair split-K kernel.
  // (token tiles round up to the next shape with a pair build; the rows past M are zero-filled)
  const int pbn = tc_pair_bn(p.BN, p.NSUB);
  const bool want_pair = lmhead ? g_lmhead_pair != 0 : (g_linear_pair && g_linear_pair_persistent);
  if (want_pair && g_force_grid == 0 && TN >= 64 && tiles > sms && pbn > 0) {
    const int pairs = linear_tc_pair_capacity(pbn, p.NSUB, lmhead);
    const long long wt = (long long)p.tiles_m * ((p.tiles_n + 1) / 2);
    if (pairs > 0 && wt >= pairs) {
      LinPlan q = p;
      q.BN = pbn;
      q.tc_pair = true;
      q.grid = pairs;
      q.units = wt * p.k_tiles;
      q.aligned = lmhead || wt > (long long)kMaxCounters;
      q.dp_tiles = q.aligned ? wt : wt / pairs * pairs;
      q.sk_units = 0;
      q.bytes = 0;
      bool ok_plan = true;
      if (lmhead) {
        q.bytes = kCounterBytes + round_up(size_t(M) * p.tiles_n * sizeof(float2), 256);
      } else if (q.dp_tiles < wt && g_linear_pair_persistent == 2) {
        // the rest on the pair split-K kernel (S pairs per pair tile, on-chip sums)
        // (the most pairs per pair tile that still fit in one wave)
        int best = 0;
        for (int S = std::min(4, p.k_tiles); S >= 2 && !best; --S)
          if (linear_pair_capacity(p.BN, p.NSUB, S) >= (wt - q.dp_tiles) * 2 * S) best = S;
        ok_plan = best > 0;
        q.pair_n = 1;
        q.pair_first[0] = (int)q.dp_tiles;
        q.pair_count[0] = (int)(wt - q.dp_tiles);
        q.pair_S[0] = best;
      } else if (q.dp_tiles < wt) {
        q.sk_units = (wt - q.dp_tiles) * p.k_tiles;
        bool split = false;
        for (int c = 1; c < pairs && !split; ++c) split = ((q.sk_units * c / pairs) % p.k_tiles) != 0;
        q.bytes = split ? kCounterBytes + round_up(size_t(pairs) * 2 * 2 * pbn * p.NSUB * 128 * 4, 256) : 0;
      }
      if (ok_plan && q.bytes <= max_bytes) return q;
    }
  }
  // 2-SM pair tiles (256 weight rows on a CTA pair; each CTA stages half of the token rows, which
  // halves the shared-memory traffic per MMA that bounds the one-SM kernels at a few hundred rows):
  // few pair tiles -> one cluster split-K launch of S pairs per tile; more -> whole pair tiles on
  // every pair (S = 1), then the rest split
  if (!lmhead && g_linear_pair && g_force_grid == 0 && TN >= 64 && (g_linear_pair_few || tiles > sms)) {
    const long long ptiles = (long long)p.tiles_m * ((p.tiles_n + 1) / 2);
    auto best_S = [&](long long n_pt, long long* cost_out) {
      int best = 0;
      long long best_cost = 0;
      for (int S = 1; S <= 4 && S <= p.k_tiles; ++S) {
        const int cap = linear_pair_capacity(p.BN, p.NSUB, S);
        if (cap <= 0 || n_pt * 2 * S > cap) continue;
        const long long cost = (p.k_tiles + S - 1) / S + (S > 1 ? 6 * 64 / LIN_BK : 2);
        if (best == 0 || cost < best_cost) { best = S; best_cost = cost; }
      }
      *cost_out = best_cost;
      return best;
    };
    long long c1 = 0;
    const int S1 = g_linear_pair_few ? best_S(ptiles, &c1) : 0;
    if (S1 > 0) {
      p.pair_n = 1;
      p.pair_first[0] = 0;
      p.pair_count[0] = (int)ptiles;
      p.pair_S[0] = S1;
      p.bytes = 0;
      return p;
    }
    const int cap1 = linear_pair_capacity(p.BN, p.NSUB, 1);
    const long long whole = cap1 / 2;
    if (whole > 0 && ptiles > whole && ptiles - whole <= whole) {
      long long c2 = 0;
      const int S2 = best_S(ptiles - whole, &c2);
      if (S2 > 0) {
        p.pair_n = 2;
        p.pair_first[0] = 0;
        p.pair_count[0] = (int)whole;
        p.pair_S[0] = 1;
        p.pair_first[1] = (int)whole;
        p.pair_count[1] = (int)(ptiles - whole);
        p.pair_S[1] = S2;
        p.bytes = 0;
        return p;
      }
    }
  }
  // few tiles: S CTAs of a cluster split each tile's k-steps and sum on chip (one wave of
  // tiles * S CTAs).  Cost model in k-steps of one tile on one SM: the cluster kernel takes
  // ceil(kt / S) plus ~6 for its on-chip reduction; stream-K takes ceil(units / SMs) plus
  // ~20 when tiles are split (fp32 pieces through L2 and a second kernel)
  if (!lmhead && g_linear_cluster && g_force_grid == 0 && tiles < sms) {
    int best = 0;
    long long best_cost = 0;
    for (int S = 2; S <= 8 && S <= p.k_tiles; ++S) {
      const int cap = linear_cluster_capacity(p.BN, p.NSUB, S);
      if (cap <= 0 || tiles * S > cap) continue;
      const long long cost = (p.k_tiles + S - 1) / S + 6 * 64 / LIN_BK;
      if (best == 0 || cost < best_cost) { best = S; best_cost = cost; }
    }
    const long long sk_cost = (p.units + sms - 1) / sms + 20 * 64 / LIN_BK;
    if (best >= 2 && best_cost < sk_cost) {
      p.cluster_S = best;
      p.grid = (int)(tiles * best);
      p.bytes = 0;
      if (g_linear_split_rows && p.NSUB == 2 && p.tiles_m == 1) cluster_split_rows(p, M);
      return p;
    }
  }
  const long long ctiles = tiles;
  // many tiles, not a multiple of the SM count: the whole tiles one per CTA (none split) on the
  // persistent kernel, then the remainder on the cluster split-K kernel (on-chip sums: no fp32
  // pieces through L2, no reduce kernel), when that costs fewer k-steps than stream-K
  if (!lmhead && g_linear_cluster && g_force_grid == 0 && tiles > sms && tiles % sms != 0 &&
      !p.aligned) {
    const long long rem = tiles % sms;
    int best = 0;
    long long best_cost = 0;
    for (int S = 2; S <= 8 && S <= p.k_tiles; ++S) {
      const int cap = linear_cluster_capacity(p.BN, p.NSUB, S);
      if (cap <= 0 || rem * S > cap) continue;
      const long long cost = (p.k_tiles + S - 1) / S + 6 * 64 / LIN_BK;
      if (best == 0 || cost < best_cost) { best = S; best_cost = cost; }
    }
    const long long sk_cost = (p.units + sms - 1) / sms + 20 * 64 / LIN_BK;
    if (best >= 2 && (tiles / sms) * p.k_tiles + best_cost < sk_cost) {
      p.rem_S = best;
      p.rem_tiles = rem;
      p.grid = sms;
      p.dp_tiles = tiles - rem;
      p.sk_units = 0;
      p.bytes = 0;
      return p;
    }
  }
  int grid = g_force_grid > 0 ? g_force_grid : sms;
  const long long cap_units = p.aligned ? ctiles : p.units;
  if (grid > cap_units) grid = (int)cap_units;
  p.grid = std::max(1, grid);
  // data-parallel tiles first (every CTA gets as many whole tiles as all can), stream-K
  // for the rest
  if (p.aligned) {
    p.dp_tiles = ctiles;
    p.sk_units = 0;
  } else {
    p.dp_tiles = ctiles / p.grid * p.grid;
    p.sk_units = (ctiles - p.dp_tiles) * p.k_tiles;
  }
  if (lmhead) {
    p.bytes = kCounterBytes + round_up(size_t(M) * p.tiles_n * sizeof(float2), 256);
    return p;
  }
  bool split = false;
  for (int c = 1; c < p.grid && !split && p.sk_units > 0; ++c) split = ((p.sk_units * c / p.grid) % p.k_tiles) != 0;
  p.bytes = split ? kCounterBytes + round_up(size_t(p.grid) * 2 * TN * 128 * 4, 256) : 0;
  return p;
}

// --------------------------------------------------------------------------- attention plan
struct AttnPlan {
  bool tc = false;               // persistent tcgen05 kernel
  int grid = 1;
  int chunk = 256, max_chunks = 1;
  size_t counters_off = 0, partial_off = 0, pfx_off = 0, bytes = 0;
};

AttnPlan plan_attention(int B, int max_rows, int Hq, int Hkv, int cap) {
  AttnPlan p;
  const int sms = plan_sms();
  const int G = Hkv > 0 ? Hq / Hkv : 1;
  p.tc = g_attn_impl == 1 && B <= attention_tc_max_batch() && attention_tc_rows(G, max_rows) > 0;
  p.counters_off = 0;
  p.partial_off = kCounterBytes;
  if (p.tc) {
    p.grid = g_force_grid > 0 ? g_force_grid : sms;
    p.pfx_off = kCounterBytes + round_up(size_t(p.grid) * 2 * 64 * (128 + 2) * 4, 256);
    p.bytes = p.pfx_off + round_up(size_t(p.grid) * (B + 1) * 4, 256);
    return p;
  }
  const double keys = double(B) * Hkv * cap;
  int chunk = 256;
  while (chunk < 4096 && keys / (chunk * 2) >= 8.0 * sms) chunk *= 2;
  p.chunk = chunk;
  p.max_chunks = std::max(1, (cap + chunk - 1) / chunk);
  p.bytes = kCounterBytes + round_up(size_t(B) * Hkv * p.max_chunks * 64 * (128 + 2) * 4, 256);
  return p;
}

}  // namespace

namespace spec {
bool pdl_enabled() { return g_pdl != 0; }
}  // namespace spec

// =========================================================================== C ABI
extern "C" {

const char* spec_last_error(void) { return t_err.c_str(); }
int spec_launches(void) { return t_launches; }
int spec_version(void) { return kVersion; }

int spec_set_option(const char* name, int value) {
  if (!name) return fail(SPEC_EINVAL, "option name is NULL");
  if (!strcmp(name, "gemv_max_m")) {
    if (value < 0 || value > 4) return fail(SPEC_EINVAL, "gemv_max_m must be in [0, 4]");
    g_gemv_max_m = value;
    return ok();
  }
  if (!strcmp(name, "linear_pair")) {
    if (value < 0 || value > 1) return fail(SPEC_EINVAL, "linear_pair must be 0 or 1");
    g_linear_pair = value;
    return ok();
  }
  if (!strcmp(name, "lmhead_pair")) {
    if (value < 0 || value > 1) return fail(SPEC_EINVAL, "lmhead_pair must be 0 or 1");
    g_lmhead_pair = value;
    return ok();
  }
  if (!strcmp(name, "linear_pair_persistent")) {
    if (value < 0 || value > 2) return fail(SPEC_EINVAL, "linear_pair_persistent must be in [0, 2]");
    g_linear_pair_persistent = value;
    return ok();
  }
  if (!strcmp(name, "linear_pair_few")) {
    if (value < 0 || value > 1) return fail(SPEC_EINVAL, "linear_pair_few must be 0 or 1");
    g_linear_pair_few = value;
    return ok();
  }
  if (!strcmp(name, "pdl")) {
    if (value < 0 || value > 1) return fail(SPEC_EINVAL, "pdl must be 0 or 1");
    g_pdl = value;
    return ok();
  }
  if (!strcmp(name, "kv_l2_promotion")) {
    if (value < 0 || value > 3) return fail(SPEC_EINVAL, "kv_l2_promotion must be in [0, 3]");
    g_kv_promotion = value;
    return ok();
  }
  if (!strcmp(name, "weight_l2_promotion")) {
    if (value < 0 || value > 3) return fail(SPEC_EINVAL, "weight_l2_promotion must be in [0, 3]");
    g_w_promotion = value;
    return ok();
  }
  if (!strcmp(name, "lmhead_nsub")) {
    if (value < 1 || value > 2) return fail(SPEC_EINVAL, "lmhead_nsub must be 1 or 2");
    g_lmhead_nsub = value;
    return ok();
  }
  if (!strcmp(name, "linear_cluster")) {
    if (value < 0 || value > 1) return fail(SPEC_EINVAL, "linear_cluster must be 0 or 1");
    g_linear_cluster = value;
    return ok();
  }
  if (!strcmp(name, "weight_prefetch")) {
    if (value < 0 || value > 1) return fail(SPEC_EINVAL, "weight_prefetch must be 0 or 1");
    g_weight_prefetch = value;
    return ok();
  }
  if (!strcmp(name, "linear_split_rows")) {
    if (value < 0 || value > 1) return fail(SPEC_EINVAL, "linear_split_rows must be 0 or 1");
    g_linear_split_rows = value;
    return ok();
  }
  if (!strcmp(name, "attention_pair_cost")) {
    if (value < 0 || value > 64) return fail(SPEC_EINVAL, "attention_pair_cost must be in [0, 64]");
    g_attn_pair_cost = value;
    return ok();
  }
  if (!strcmp(name, "attention_impl")) {
    if (value < 0 || value > 1) return fail(SPEC_EINVAL, "attention_impl must be 0 or 1");
    g_attn_impl = value;
    return ok();
  }
  if (!strcmp(name, "linear_nsub")) {
    if (value < 1 || value > 2) return fail(SPEC_EINVAL, "linear_nsub must be 1 or 2");
    g_nsub_max = value;
    return ok();
  }
  if (!strcmp(name, "persistent_grid")) {
    if (value < 0 || value > 4096) return fail(SPEC_EINVAL, "persistent_grid must be in [0, 4096]");
    g_force_grid = value;
    return ok();
  }
  return fail(SPEC_EINVAL, "unknown option '%s'", name);
}

int spec_device_status(spec_stream stream, int* detail) {
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned v = 0;
  e = cudaMemcpy(&v, d->status, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read status word");
  if (detail) *detail = (int)v;
  if (v) {
    const unsigned zero = 0;
    e = cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear status word");
    if ((v & 0xF0u) == 0xF0u)
      return fail(SPEC_EINVAL, "a kernel rejected device-side input (site 0x%x)", v);
    return fail(SPEC_ETIMEOUT, "a bounded device wait ran out (site 0x%x)", v);
  }
  return ok();
}

int spec_probe_bounded_wait(int limit_us, int arrive, spec_stream stream) {
  if (limit_us < 1 || limit_us > 2000000) return fail(SPEC_EINVAL, "limit_us=%d must be in [1, 2000000]", limit_us);
  if (arrive != 0 && arrive != 1) return fail(SPEC_EINVAL, "arrive must be 0 or 1");
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  cudaError_t e = launch_wait_probe(d->status, SPEC_PROBE_WAIT_SITE, (unsigned long long)limit_us * 1000ull, arrive,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait probe launch");
  return ok(1);
}

// --------------------------------------------------------------------------- linear
size_t spec_linear_workspace_bytes(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return plan_linear(M, N, K, false).bytes;
}

}  // extern "C"

// Host-side checks of a verify-linear call with M >= 1 (everything but the workspace).
static int check_linear_args(const spec_bf16* X, int M, int K, int ldx, const spec_bf16* W, int N, int ldw,
                             const spec_bf16* Y, int ldy, const spec_bf16* residual, int ldr) {
  if (!X || !W || !Y) return fail(SPEC_EINVAL, "X, W and Y must be non-NULL");
  if (K % 8) return fail(SPEC_EINVAL, "K=%d must be a multiple of 8", K);
  if (ldx < K || ldw < K || ldy < N || (residual && ldr < N))
    return fail(SPEC_EINVAL, "leading dimensions too small");
  if (ldx % 8 || ldw % 8 || ldy % 8 || (residual && ldr % 8))
    return fail(SPEC_EINVAL, "leading dimensions must be multiples of 8");
  if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || (residual && !aligned16(residual)))
    return fail(SPEC_EINVAL, "X, W, Y, residual must be 16-byte aligned");
  if (residual && residual != Y) {
    const char* y0 = reinterpret_cast<const char*>(Y);
    const char* y1 = reinterpret_cast<const char*>(Y + (size_t)(M - 1) * ldy + N);
    const char* r0 = reinterpret_cast<const char*>(residual);
    const char* r1 = reinterpret_cast<const char*>(residual + (size_t)(M - 1) * ldr + N);
    if (r0 < y1 && y0 < r1) return fail(SPEC_EINVAL, "residual overlaps Y without being Y");
  }
  if (residual == Y && ldr != ldy) return fail(SPEC_EINVAL, "residual aliases Y with another ldr");
  return SPEC_OK;
}

// The launches of a pair plan (epilogue already set in a).  Returns the number of launches (0 on
// error, *err set).
static int launch_pair_plan(const LinPlan& p, const CUtensorMap& tw, const CUtensorMap& tx, LinearArgs a,
                            cudaStream_t s, cudaError_t* err) {
  for (int i = 0; i < p.pair_n; ++i) {
    a.dp_tiles = p.pair_first[i];
    *err = launch_linear_pair(p.BN, p.NSUB, tw, tx, a, p.pair_S[i], p.pair_count[i], s);
    if (*err != cudaSuccess) return 0;
  }
  return p.pair_n;
}

// The launches of a persistent pair plan (epilogue and args set): the persistent kernel, then
// the pair split-K kernel for the pair tiles after dp_tiles or the reduce kernel for split pieces.
// Returns the number of launches, or a (negative) error from fail().
static int launch_tc_pair_plan(const LinPlan& p, const CUtensorMap& tw, const CUtensorMap& tx, LinearArgs a,
                               cudaStream_t s) {
  a.pair = 1;
  cudaError_t e = launch_linear_tc_pair(p.BN, p.NSUB, a.epi, tw, tx, a, p.grid, s);
  if (e != cudaSuccess) return cuda_fail(e, "pair persistent linear launch");
  if (p.pair_n > 0) {
    a.dp_tiles = p.pair_first[0];
    e = launch_linear_pair(p.BN, p.NSUB, tw, tx, a, p.pair_S[0], p.pair_count[0], s);
    if (e != cudaSuccess) return cuda_fail(e, "pair linear launch (remainder)");
    return 2;
  }
  if (p.bytes == 0) return 1;
  e = launch_linear_reduce(a, plan_sms(), s);
  if (e != cudaSuccess) return cuda_fail(e, "split-K reduce launch");
  return 2;
}

static int verify_linear_plan(const LinPlan& p, const spec_bf16* X, int M, int K, int ldx, const spec_bf16* W, int N,
                              int ldw, spec_bf16* Y, int ldy, const spec_bf16* residual, int ldr,
                              const spec_rownorm* norm, char* ws, DevInfo* d, cudaStream_t s);
static int swiglu_plan(const LinPlan& p, const spec_bf16* X, int M, int K, int ldx, const spec_bf16* Wgu, int ldw,
                       int I, spec_bf16* A, int lda, const spec_rownorm* norm, char* ws, DevInfo* d, cudaStream_t s);

// A folded RMSNorm on a plan: every tensor-core epilogue scales rows by 1 / rms; the split-K
// epilogues (cluster and pair kernels) also sum the squares of what they store.  Otherwise the
// normalised copy of X / a sum-of-squares pass over Y.
static bool plan_fuses_norm_in(const LinPlan& p) { return !p.gemv; }
static bool plan_fuses_norm_out(const LinPlan& p) { return !p.gemv && !p.tc_pair && (p.cluster_S > 0 || p.pair_n > 0); }
// The norm a plan is handed: in_ssq / out_ssq cleared where the caller does that part itself.
static const spec_rownorm* plan_norm(const spec_rownorm* nm, const LinPlan& p, spec_rownorm* tmp) {
  if (!nm) return nullptr;
  *tmp = *nm;
  if (!plan_fuses_norm_in(p)) tmp->in_ssq = nullptr;
  if (!plan_fuses_norm_out(p)) tmp->out_ssq = nullptr;
  return tmp;
}
static bool norm_in(const spec_rownorm* nm) { return nm && nm->in_ssq; }
static bool norm_out(const spec_rownorm* nm) { return nm && nm->out_ssq; }
static int check_norm(const spec_rownorm* nm) {
  if (!nm) return SPEC_OK;
  if (nm->in_ssq && (nm->in_tiles <= 0 || !(nm->eps >= 0.f) || std::isinf(nm->eps)))
    return fail(SPEC_EINVAL, "norm: in_tiles must be >= 1 and eps finite and >= 0");
  return SPEC_OK;
}
// Offset of the normalised copy of X in the workspace: after the plan's own scratch, never inside
// the counter region.
static size_t norm_copy_off(size_t plan_bytes) { return std::max(round_up(plan_bytes, 256), kCounterBytes); }
// (out_ssq only with the plain bf16 epilogue, the one that sums the squares of what it stores)
static void set_norm_args(LinearArgs& a, const spec_rownorm* nm, int K) {
  if (!nm) return;
  if (nm->in_ssq) {
    a.norm_ssq = nm->in_ssq;
    a.norm_tiles = nm->in_tiles;
    a.norm_k = (float)K;
    a.norm_eps = nm->eps;
  }
  if (a.epi == EPI_BF16) a.out_ssq = nm->out_ssq;
}

// (max_bytes: the largest scratch a plan may ask for; plans above it give way to the next choice)
static int verify_linear_impl(const spec_bf16* X, int M, int K, int ldx, const spec_bf16* W, int N, int ldw,
                              spec_bf16* Y, int ldy, const spec_bf16* residual, int ldr, const spec_rownorm* norm,
                              void* workspace, size_t workspace_bytes, spec_stream stream,
                              size_t max_bytes = SIZE_MAX) {
  if (M < 0 || N <= 0 || K <= 0) return fail(SPEC_EINVAL, "bad sizes M=%d N=%d K=%d", M, N, K);
  if (M == 0) return ok();
  if (int rc = check_linear_args(X, M, K, ldx, W, N, ldw, Y, ldy, residual, ldr)) return rc;
  if (int rc = check_norm(norm)) return rc;
  LinPlan p = plan_linear(M, N, K, false, false, max_bytes);
  const bool copy_x = norm_in(norm) && !plan_fuses_norm_in(p);
  const size_t need = copy_x ? norm_copy_off(p.bytes) + round_up(size_t(M) * K * 2, 256) : p.bytes;
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(SPEC_EINVAL, "workspace too small: need %zu bytes", need);
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int extra = 0;
  if (copy_x) {
    // the RMSNorm of X from its sums of squares, into the workspace; the product reads that copy
    spec_bf16* Xn = reinterpret_cast<spec_bf16*>(ws + norm_copy_off(p.bytes));
    cudaError_t e = launch_rownorm_ssq(X, M, K, ldx, norm->in_ssq, norm->in_tiles, norm->eps, Xn, K, s);
    if (e != cudaSuccess) return cuda_fail(e, "row normalisation launch");
    X = Xn;
    ldx = K;
    extra = 1;
  }
  spec_rownorm tmp{};
  const int rc = verify_linear_plan(p, X, M, K, ldx, W, N, ldw, Y, ldy, residual, ldr, plan_norm(norm, p, &tmp),
                                    ws, d, s);
  if (rc) return rc;
  int n = t_launches + extra;
  if (norm_out(norm) && !plan_fuses_norm_out(p)) {
    cudaError_t e = launch_row_ssq(Y, M, N, ldy, norm->out_ssq, s);
    if (e != cudaSuccess) return cuda_fail(e, "sum-of-squares launch");
    ++n;
  }
  return ok(n);
}

extern "C" {

int spec_verify_linear(const spec_bf16* X, int M, int K, int ldx, const spec_bf16* W, int N,
                       int ldw, spec_bf16* Y, int ldy, const spec_bf16* residual, int ldr,
                       void* workspace, size_t workspace_bytes, spec_stream stream) {
  return verify_linear_impl(X, M, K, ldx, W, N, ldw, Y, ldy, residual, ldr, nullptr, workspace, workspace_bytes,
                            stream);
}

int spec_verify_linear_norm(const spec_bf16* X, int M, int K, int ldx, const spec_bf16* W, int N, int ldw,
                            spec_bf16* Y, int ldy, const spec_bf16* residual, int ldr, const spec_rownorm* norm,
                            void* workspace, size_t workspace_bytes, spec_stream stream) {
  return verify_linear_impl(X, M, K, ldx, W, N, ldw, Y, ldy, residual, ldr, norm, workspace, workspace_bytes,
                            stream);
}

size_t spec_linear_norm_workspace_bytes(int M, int N, int K, int swiglu) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  const LinPlan p = plan_linear(M, swiglu ? 2 * N : N, K, false, swiglu != 0);
  const size_t own = swiglu ? spec_swiglu_linear_workspace_bytes(M, N, K) : p.bytes;
  return plan_fuses_norm_in(p) ? own : norm_copy_off(own) + round_up(size_t(M) * K * 2, 256);
}

int spec_row_ssq(const spec_bf16* X, int M, int N, int ldx, float* out, spec_stream stream) {
  if (M < 0 || N <= 0) return fail(SPEC_EINVAL, "bad sizes M=%d N=%d", M, N);
  if (M == 0) return ok();
  if (!X || !out) return fail(SPEC_EINVAL, "NULL argument");
  if (ldx < N) return fail(SPEC_EINVAL, "ldx=%d < N=%d", ldx, N);
  cudaError_t e = launch_row_ssq(X, M, N, ldx, out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sum-of-squares launch");
  return ok(1);
}

}  // extern "C"

// The launches of one linear plan (arguments already checked; the workspace holds p.bytes).
static int verify_linear_plan(const LinPlan& p, const spec_bf16* X, int M, int K, int ldx, const spec_bf16* W, int N,
                              int ldw, spec_bf16* Y, int ldy, const spec_bf16* residual, int ldr,
                              const spec_rownorm* norm, char* ws, DevInfo* d, cudaStream_t s) {
  if (p.gemv) {
    GemvArgs a;
    a.X = X; a.ldx = ldx; a.W = W; a.ldw = ldw; a.Y = Y; a.ldy = ldy;
    a.residual = residual; a.ldr = ldr; a.M = M; a.N = N; a.K = K;
    a.splits = p.splits; a.k_per_split = p.k_per_split;
    a.partial = p.splits > 1 ? reinterpret_cast<float*>(ws + p.partial_off) : nullptr;
    a.counters = p.splits > 1 ? reinterpret_cast<unsigned*>(ws + p.counters_off) : nullptr;
    cudaError_t e = launch_gemv(a, p.gemv_grid, s);
    if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
    return ok(1);
  }
  CUtensorMap tw, tx;
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    cuuint64_t str[1] = {(cuuint64_t)ldw * 2};
    cuuint32_t box[2] = {LIN_BK, 128};
    if (int rc = encode_bf16(&tw, W, 2, dims, str, box, "W", g_w_promotion, kLinSwizzle)) return rc;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t str[1] = {(cuuint64_t)ldx * 2};
    cuuint32_t box[2] = {LIN_BK, (cuuint32_t)p.x_box_rows()};
    if (int rc = encode_bf16(&tx, X, 2, dims, str, box, "X", 3, kLinSwizzle)) return rc;
  }
  LinearArgs a{};
  a.M = M; a.N = N; a.K = K; a.k_tiles = p.k_tiles; a.tiles_m = p.tiles_m; a.tiles_n = p.tiles_n;
  a.units = p.units; a.grid = p.grid; a.dp_tiles = p.dp_tiles; a.sk_units = p.sk_units;
  a.Y = Y; a.ldy = ldy; a.residual = residual; a.ldr = ldr;
  a.partial = p.bytes > 0 ? reinterpret_cast<float*>(ws + p.partial_off) : nullptr;
  a.status = d->status;
  a.w_early = g_weight_prefetch;
  a.tn = p.BN * p.NSUB;
  a.epi = EPI_BF16;
  set_norm_args(a, norm, K);
  if (p.tc_pair) {
    const int n = launch_tc_pair_plan(p, tw, tx, a, s);
    return n > 0 ? ok(n) : n;
  }
  if (p.pair_n > 0) {
    cudaError_t e = cudaSuccess;
    const int n = launch_pair_plan(p, tw, tx, a, s, &e);
    if (!n) return cuda_fail(e, "pair linear launch");
    return ok(n);
  }
  if (p.cluster_S > 0) {
    cudaError_t e = launch_linear_cluster(p.BN, p.NSUB, tw, tx, a, p.cluster_S, p.grid / p.cluster_S, s);
    if (e != cudaSuccess) return cuda_fail(e, "cluster linear launch");
    return ok(1);
  }
  dim3 grid(p.grid);
  cudaError_t e = launch_linear_tc_bf16(p.BN, p.NSUB, tw, tx, a, grid, s);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 linear launch");
  if (p.rem_S > 0) {   // the tiles after a.dp_tiles: cluster split-K
    e = launch_linear_cluster(p.BN, p.NSUB, tw, tx, a, p.rem_S, (int)p.rem_tiles, s);
    if (e != cudaSuccess) return cuda_fail(e, "cluster linear launch (remainder)");
    return ok(2);
  }
  if (p.bytes == 0) return ok(1);
  // some tiles had their k-steps split between CTAs: a second kernel sums their pieces
  e = launch_linear_reduce(a, plan_sms(), s);
  if (e != cudaSuccess) return cuda_fail(e, "split-K reduce launch");
  return ok(2);
}

// --------------------------------------------------------------------------- linear chain (small M)
namespace {

// An [M x cols] bf16 matrix with leading dimension ld, for dependency analysis.
struct Region {
  const char* base = nullptr;
  long long ld = 0, cols = 0;
  bool valid() const { return base != nullptr; }
};

Region region_of(const void* p, int ld, long long cols) {
  Region r;
  r.base = static_cast<const char*>(p);
  r.ld = ld;
  r.cols = cols;
  return r;
}

// Do a and b share an element?  Exact for matrices of the same leading dimension in one row frame,
// a byte-interval test otherwise (conservative).
bool overlaps(const Region& a, const Region& b, int M) {
  if (!a.valid() || !b.valid()) return false;
  if (a.ld == b.ld) {
    const long long d = (a.base - b.base) / 2;
    if ((a.base - b.base) % 2 == 0) {
      if (d >= 0 && d + a.cols <= a.ld) return d < b.cols;              // a's columns [d, d + cols) in b's frame
      if (d < 0 && -d + b.cols <= b.ld) return -d < a.cols;
    }
  }
  const char* a1 = a.base + ((long long)(M - 1) * a.ld + a.cols) * 2;
  const char* b1 = b.base + ((long long)(M - 1) * b.ld + b.cols) * 2;
  return a.base < b1 && b.base < a1;
}

// Is every element of reader r inside writer w, column c of r at column c + shift of w?
bool contains(const Region& w, const Region& r, long long* shift) {
  if (!w.valid() || !r.valid() || w.ld != r.ld || (r.base - w.base) % 2) return false;
  const long long d = (r.base - w.base) / 2;
  if (d < 0 || d + r.cols > w.cols) return false;
  *shift = d;
  return true;
}

struct ChainOpHost {
  Region x, r, y;
  const spec_linear_op* op;
};

// Dependencies of product j on the products [first, j) of its launch (products of earlier launches
// are complete when it starts).  Returns false when they need more than CH_MAX_DEPS entries.
bool chain_deps(const std::vector<ChainOpHost>& h, int first, int j, int M, ChainOp* o) {
  o->n_deps = 0;
  auto add = [&](int op, int kind, long long shift) {
    for (int i = 0; i < o->n_deps; ++i)
      if (o->dep[i].op == op - first && o->dep[i].kind == kind) {
        if (o->dep[i].shift != (int)shift) o->dep[i].shift = -1;
        return true;
      }
    if (o->n_deps >= CH_MAX_DEPS) return false;
    o->dep[o->n_deps++] = ChainDep{op - first, kind, (int)shift};
    return true;
  };
  // read-after-write: the latest writer of each read region; when it covers the region, earlier
  // writers are ordered before it (its own write waited for them)
  for (int kind : {CH_DEP_X, CH_DEP_RES}) {
    const Region& rd = kind == CH_DEP_X ? h[j].x : h[j].r;
    if (!rd.valid()) continue;
    if (kind == CH_DEP_RES && rd.base == h[j].y.base && rd.ld == h[j].y.ld) {
      // in place: the residual is this product's own output region; the writers of that region
      // are found below as well
    }
    for (int i = j - 1; i >= first; --i) {
      if (!overlaps(h[i].y, rd, M)) continue;
      long long shift = -1;
      const bool covered = contains(h[i].y, rd, &shift);
      if (!add(i, kind, covered ? shift : -1)) return false;
      if (covered) break;
    }
  }
  // write-after-read / write-after-write on Y's region: the latest writer (when it covers the
  // region, nothing before it matters) and every reader after it
  int w = first - 1;
  for (int i = j - 1; i >= first; --i) {
    if (!overlaps(h[i].y, h[j].y, M)) continue;
    long long sh;
    if (contains(h[i].y, h[j].y, &sh)) { w = i; break; }
  }
  for (int i = j - 1; i >= first && i >= (w < first ? first : w); --i) {
    const bool reads = overlaps(h[i].x, h[j].y, M) || overlaps(h[i].r, h[j].y, M);
    const bool writes = overlaps(h[i].y, h[j].y, M);
    if (!reads && !writes) continue;
    // in-place residual stream: product i wrote (and read as its own residual) exactly this
    // region, and product j waits for i's tile t before reading its residual tile t; its write of
    // tile t comes after that
    bool per_tile = false;
    for (int d = 0; d < o->n_deps; ++d)
      per_tile = per_tile || (o->dep[d].op == i - first && o->dep[d].kind == CH_DEP_RES && o->dep[d].shift == 0);
    const bool same_y = h[i].y.base == h[j].y.base && h[i].y.ld == h[j].y.ld && h[i].y.cols == h[j].y.cols &&
                        h[i].op->swiglu == h[j].op->swiglu;
    const bool i_in_place = !h[i].r.valid() || (h[i].r.base == h[i].y.base && h[i].r.ld == h[i].y.ld);
    const bool j_in_place = h[j].r.valid() && h[j].r.base == h[j].y.base && h[j].r.ld == h[j].y.ld;
    if (per_tile && same_y && i_in_place && j_in_place && !overlaps(h[i].x, h[j].y, M)) continue;
    if (!add(i, CH_DEP_WRITE, -1)) return false;
  }
  return true;
}

int check_chain_op(const spec_linear_op& op, int M, int k) {
  if (op.N <= 0 || op.K <= 0) return fail(SPEC_EINVAL, "op %d: bad sizes N=%d K=%d", k, op.N, op.K);
  if (op.swiglu) {
    if (op.N % 128) return fail(SPEC_EINVAL, "op %d: SwiGLU needs N = 2I with I a multiple of 64", k);
    if (op.residual) return fail(SPEC_EINVAL, "op %d: SwiGLU takes no residual", k);
    if (!op.X || !op.W || !op.Y) return fail(SPEC_EINVAL, "op %d: X, W and Y must be non-NULL", k);
    if (op.K % 8 || op.ldx < op.K || op.ldw < op.K || op.ldy < op.N / 2 || op.ldx % 8 || op.ldw % 8 || op.ldy % 8)
      return fail(SPEC_EINVAL, "op %d: K and the leading dimensions must be multiples of 8, ld >= width", k);
    if (!aligned16(op.X) || !aligned16(op.W) || !aligned16(op.Y))
      return fail(SPEC_EINVAL, "op %d: X, W, Y must be 16-byte aligned", k);
    return SPEC_OK;
  }
  return check_linear_args(op.X, M, op.K, op.ldx, op.W, op.N, op.ldw, op.Y, op.ldy, op.residual, op.ldr);
}

// Launches of one chain: products [first, last) each (at most CH_MAX_OPS, and a new launch where a
// product's dependencies do not fit).
std::vector<std::pair<int, int>> chain_launches(const std::vector<ChainOpHost>& h, int M) {
  std::vector<std::pair<int, int>> out;
  int first = 0;
  const int n = (int)h.size();
  while (first < n) {
    int last = first + 1;
    ChainOp tmp;
    while (last < n && last - first < CH_MAX_OPS && chain_deps(h, first, last, M, &tmp)) ++last;
    out.emplace_back(first, last);
    first = last;
  }
  return out;
}

size_t chain_flags_bytes(const std::vector<ChainOpHost>& h, int first, int last) {
  long long tiles = 0;
  for (int j = first; j < last; ++j) tiles += (h[j].op->N + 127) / 128;
  return round_up(size_t(2 * tiles + (last - first)) * 4, 256);
}

size_t chain_pieces_bytes(int n_ops, int M) {
  return size_t(n_ops) * plan_sms() * chain_bn(M) * 128 * 4;
}

std::vector<ChainOpHost> chain_host(const spec_linear_op* ops, int n_ops) {
  std::vector<ChainOpHost> h(n_ops);
  for (int j = 0; j < n_ops; ++j) {
    const spec_linear_op& op = ops[j];
    h[j].op = &op;
    h[j].x = region_of(op.X, op.ldx, op.K);
    h[j].y = region_of(op.Y, op.ldy, op.swiglu ? op.N / 2 : op.N);
    if (op.residual) h[j].r = region_of(op.residual, op.ldr, op.N);
  }
  return h;
}

}  // namespace

extern "C" {

size_t spec_linear_chain_workspace_bytes(const spec_linear_op* ops, int n_ops, int M) {
  if (!ops || n_ops <= 0 || M <= 0 || M > CH_MAX_M) return 0;
  const std::vector<ChainOpHost> h = chain_host(ops, n_ops);
  size_t need = 0;
  for (const auto& l : chain_launches(h, M))
    need = std::max(need, kCounterBytes + chain_flags_bytes(h, l.first, l.second) +
                              chain_pieces_bytes(l.second - l.first, M));
  return need;
}

int spec_verify_linear_chain(const spec_linear_op* ops, int n_ops, int M, void* workspace, size_t workspace_bytes,
                             spec_stream stream) {
  if (n_ops < 0 || M < 0) return fail(SPEC_EINVAL, "bad sizes n_ops=%d M=%d", n_ops, M);
  if (n_ops == 0 || M == 0) return ok();
  if (!ops) return fail(SPEC_EINVAL, "ops must be non-NULL");
  if (M > CH_MAX_M) return fail(SPEC_EUNSUPPORTED, "M=%d > %d rows (use spec_verify_linear per product)", M, CH_MAX_M);
  for (int j = 0; j < n_ops; ++j)
    if (int rc = check_chain_op(ops[j], M, j)) return rc;
  const std::vector<ChainOpHost> h = chain_host(ops, n_ops);
  for (int j = 0; j < n_ops; ++j)
    if (overlaps(h[j].x, h[j].y, M)) return fail(SPEC_EINVAL, "op %d: X overlaps its own Y", j);
  const auto launches = chain_launches(h, M);
  size_t need = 0;
  for (const auto& l : launches)
    need = std::max(need, kCounterBytes + chain_flags_bytes(h, l.first, l.second) + chain_pieces_bytes(l.second - l.first, M));
  if (!workspace || workspace_bytes < need) return fail(SPEC_EINVAL, "workspace too small: need %zu bytes", need);
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int BN = chain_bn(M);
  int launched = 0;
  for (const auto& l : launches) {
    static thread_local ChainParams P;   // ~19 KB: kept off the stack
    memset(&P, 0, sizeof(P));
    P.n_ops = l.second - l.first;
    P.M = M;
    P.grid = d->sms;
    const size_t flags = chain_flags_bytes(h, l.first, l.second);
    unsigned* fl = reinterpret_cast<unsigned*>(ws + kCounterBytes);
    long long tiles = 0;
    for (int j = l.first; j < l.second; ++j) tiles += (ops[j].N + 127) / 128;
    P.arrive = fl;
    P.done = fl + tiles;
    P.op_done = fl + 2 * tiles;
    P.pieces = reinterpret_cast<float*>(ws + kCounterBytes + flags);
    P.status = d->status;
    int flag_base = 0;
    for (int j = l.first; j < l.second; ++j) {
      const spec_linear_op& op = ops[j];
      ChainOp& o = P.op[j - l.first];
      o.Y = op.Y;
      o.residual = op.residual;
      o.ldy = op.ldy;
      o.ldr = op.ldr;
      o.N = op.N;
      o.K = op.K;
      o.k_tiles = (op.K + LIN_BK - 1) / LIN_BK;
      o.tiles_n = (op.N + 127) / 128;
      o.units = o.k_tiles * o.tiles_n;
      o.epi = op.swiglu ? EPI_SWIGLU : EPI_BF16;
      o.ycols = op.swiglu ? 64 : 128;
      o.flag_base = flag_base;
      flag_base += o.tiles_n;
      if (!chain_deps(h, l.first, j, M, &o)) return fail(SPEC_ECUDA, "internal: chain dependencies overflow");
      cuuint64_t wd[2] = {(cuuint64_t)op.K, (cuuint64_t)op.N};
      cuuint64_t wst[1] = {(cuuint64_t)op.ldw * 2};
      cuuint32_t wbox[2] = {LIN_BK, 128};
      if (int rc = encode_bf16(&P.tw[j - l.first], op.W, 2, wd, wst, wbox, "W", g_w_promotion, kLinSwizzle)) return rc;
      cuuint64_t xd[2] = {(cuuint64_t)op.K, (cuuint64_t)M};
      cuuint64_t xst[1] = {(cuuint64_t)op.ldx * 2};
      cuuint32_t xbox[2] = {LIN_BK, (cuuint32_t)BN};
      if (int rc = encode_bf16(&P.tx[j - l.first], op.X, 2, xd, xst, xbox, "X", 3, kLinSwizzle)) return rc;
    }
    cudaError_t e = cudaMemsetAsync(fl, 0, flags, s);
    if (e != cudaSuccess) return cuda_fail(e, "clear chain flags");
    e = launch_linear_chain(P, s);
    if (e != cudaSuccess) return cuda_fail(e, "linear chain launch");
    ++launched;
  }
  return ok(launched);
}

}  // extern "C"

extern "C" {

// --------------------------------------------------------------------------- linear + RoPE
int spec_rope_table(const int32_t* cu_rows, const int32_t* ctx_len, int B, int M, int D, float theta, float* cs,
                    spec_stream stream) {
  if (M < 0 || B < 0) return fail(SPEC_EINVAL, "bad sizes M=%d B=%d", M, B);
  if (M == 0) return ok();
  if (B == 0) return fail(SPEC_EINVAL, "rows without sequences");
  if (!cu_rows || !ctx_len || !cs) return fail(SPEC_EINVAL, "NULL argument");
  if (D <= 0 || D % 2 || D > 256) return fail(SPEC_EUNSUPPORTED, "D=%d must be even and <= 256", D);
  if (!(theta > 0.f) || std::isinf(theta)) return fail(SPEC_EINVAL, "theta must be finite and > 0");
  cudaError_t e = launch_rope_table(cu_rows, ctx_len, B, M, D, theta, reinterpret_cast<float2*>(cs),
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rope_table launch");
  return ok(1);
}

}  // extern "C"

static int verify_linear_rope_impl(const spec_bf16* X, int M, int K, int ldx, const spec_bf16* W, int N, int ldw,
                                   spec_bf16* Y, int ldy, const float* cs, int rope_heads, const spec_rownorm* norm,
                                   void* workspace, size_t workspace_bytes, spec_stream stream) {
  constexpr int HD = 128;   // head size: one weight tile of the GEMM is one head
  if (M < 0 || N <= 0 || K <= 0) return fail(SPEC_EINVAL, "bad sizes M=%d N=%d K=%d", M, N, K);
  if (M == 0) return ok();
  if (rope_heads < 0 || (long long)rope_heads * HD > N)
    return fail(SPEC_EINVAL, "rope_heads=%d heads of 128 do not fit in N=%d", rope_heads, N);
  if (rope_heads > 0 && !cs) return fail(SPEC_EINVAL, "cs must be non-NULL");
  if (rope_heads > 0 && !aligned16(cs)) return fail(SPEC_EINVAL, "cs must be 16-byte aligned");
  if (int rc = check_norm(norm)) return rc;
  const LinPlan p = plan_linear(M, N, K, false);
  if (rope_heads > 0 && (p.cluster_S > 0 || p.pair_n > 0) && !p.gemv) {
    // few weight tiles: the cluster (or pair) split-K kernel rotates the q / k heads in its epilogue
    // (and applies a folded RMSNorm's row scales before the rotation)
    if (int rc = check_linear_args(X, M, K, ldx, W, N, ldw, Y, ldy, nullptr, 0)) return rc;
    DevInfo* d = nullptr;
    if (int rc = dev_info(&d)) return rc;
    CUtensorMap tw, tx;
    {
      cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
      cuuint64_t str[1] = {(cuuint64_t)ldw * 2};
      cuuint32_t box[2] = {LIN_BK, 128};
      if (int rc = encode_bf16(&tw, W, 2, dims, str, box, "W", g_w_promotion, kLinSwizzle)) return rc;
    }
    {
      cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
      cuuint64_t str[1] = {(cuuint64_t)ldx * 2};
      cuuint32_t box[2] = {LIN_BK, (cuuint32_t)p.x_box_rows()};
      if (int rc = encode_bf16(&tx, X, 2, dims, str, box, "X", 3, kLinSwizzle)) return rc;
    }
    LinearArgs a{};
    a.M = M; a.N = N; a.K = K; a.k_tiles = p.k_tiles; a.tiles_m = p.tiles_m; a.tiles_n = p.tiles_n;
    a.units = p.units; a.grid = p.grid; a.dp_tiles = p.dp_tiles; a.sk_units = p.sk_units;
    a.Y = Y; a.ldy = ldy; a.residual = nullptr; a.ldr = 0;
    a.status = d->status;
    a.w_early = g_weight_prefetch;
    a.tn = p.BN * p.NSUB;
    a.epi = EPI_ROPE;
    a.rope_cs = reinterpret_cast<const float2*>(cs);
    a.rope_tiles = rope_heads;
    set_norm_args(a, norm, K);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    int n = 1;
    if (p.pair_n > 0) {
      cudaError_t e = cudaSuccess;
      n = launch_pair_plan(p, tw, tx, a, st, &e);
      if (!n) return cuda_fail(e, "pair linear + rope launch");
    } else {
      cudaError_t e = launch_linear_cluster(p.BN, p.NSUB, tw, tx, a, p.cluster_S, p.grid / p.cluster_S, st);
      if (e != cudaSuccess) return cuda_fail(e, "cluster linear + rope launch");
    }
    if (norm_out(norm)) {   // (the rope epilogue does not sum squares)
      cudaError_t e = launch_row_ssq(Y, M, N, ldy, norm->out_ssq, st);
      if (e != cudaSuccess) return cuda_fail(e, "sum-of-squares launch");
      ++n;
    }
    return ok(n);
  }
  // otherwise the plain product, then the rotation from the table
  if (int rc = verify_linear_impl(X, M, K, ldx, W, N, ldw, Y, ldy, nullptr, 0, norm, workspace, workspace_bytes,
                                  stream))
    return rc;
  const int n_lin = t_launches;
  if (rope_heads == 0) return ok(n_lin);
  cudaError_t e = launch_rope_apply(Y, ldy, rope_heads, HD, reinterpret_cast<const float2*>(cs), M,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rope_apply launch");
  if (norm_out(norm)) {   // the rotation changed Y after its sums of squares: take them again
    e = launch_row_ssq(Y, M, N, ldy, norm->out_ssq, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sum-of-squares launch");
    return ok(n_lin + 2);
  }
  return ok(n_lin + 1);
}

extern "C" {

int spec_verify_linear_rope(const spec_bf16* X, int M, int K, int ldx, const spec_bf16* W, int N, int ldw,
                            spec_bf16* Y, int ldy, const float* cs, int rope_heads, void* workspace,
                            size_t workspace_bytes, spec_stream stream) {
  return verify_linear_rope_impl(X, M, K, ldx, W, N, ldw, Y, ldy, cs, rope_heads, nullptr, workspace,
                                 workspace_bytes, stream);
}

int spec_verify_linear_rope_norm(const spec_bf16* X, int M, int K, int ldx, const spec_bf16* W, int N, int ldw,
                                 spec_bf16* Y, int ldy, const float* cs, int rope_heads, const spec_rownorm* norm,
                                 void* workspace, size_t workspace_bytes, spec_stream stream) {
  return verify_linear_rope_impl(X, M, K, ldx, W, N, ldw, Y, ldy, cs, rope_heads, norm, workspace,
                                 workspace_bytes, stream);
}

// --------------------------------------------------------------------------- fused SwiGLU linear
// Scratch for the CUDA-core path: the GEMV writes the interleaved gate|up rows to the workspace,
// after its own split-K scratch and never inside the counter region (which every kernel that
// uses the workspace expects to find zero).
static size_t swiglu_gemv_scratch_off(const LinPlan& p) {
  return p.bytes > 0 ? round_up(p.bytes, 256) : kCounterBytes;
}

size_t spec_swiglu_linear_workspace_bytes(int M, int I, int K) {
  if (M <= 0 || I <= 0 || K <= 0) return 0;
  const LinPlan p = plan_linear(M, 2 * I, K, false, true);
  return p.gemv ? swiglu_gemv_scratch_off(p) + round_up(size_t(M) * 2 * I * 2, 256) : p.bytes;
}

}  // extern "C"

static int verify_linear_swiglu_impl(const spec_bf16* X, int M, int K, int ldx, const spec_bf16* Wgu, int ldw, int I,
                                     spec_bf16* A, int lda, const spec_rownorm* norm, void* workspace,
                                     size_t workspace_bytes, spec_stream stream) {
  if (M < 0 || I <= 0 || K <= 0) return fail(SPEC_EINVAL, "bad sizes M=%d I=%d K=%d", M, I, K);
  if (M == 0) return ok();
  if (!X || !Wgu || !A) return fail(SPEC_EINVAL, "X, Wgu and A must be non-NULL");
  if (I % 64) return fail(SPEC_EINVAL, "I=%d must be a multiple of 64 (whole 128-row weight tiles)", I);
  if (K % 8) return fail(SPEC_EINVAL, "K=%d must be a multiple of 8", K);
  if (ldx < K || ldw < K || lda < I) return fail(SPEC_EINVAL, "leading dimensions too small");
  if (ldx % 8 || ldw % 8 || lda % 8) return fail(SPEC_EINVAL, "leading dimensions must be multiples of 8");
  if (!aligned16(X) || !aligned16(Wgu) || !aligned16(A)) return fail(SPEC_EINVAL, "X, Wgu, A must be 16-byte aligned");
  if (int rc = check_norm(norm)) return rc;
  const int N = 2 * I;
  LinPlan p = plan_linear(M, N, K, false, true);
  const bool copy_x = norm_in(norm) && !plan_fuses_norm_in(p);
  const size_t own = spec_swiglu_linear_workspace_bytes(M, I, K);
  const size_t need = copy_x ? norm_copy_off(own) + round_up(size_t(M) * K * 2, 256) : own;
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(SPEC_EINVAL, "workspace too small: need %zu bytes", need);
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int extra = 0;
  if (copy_x) {
    spec_bf16* Xn = reinterpret_cast<spec_bf16*>(ws + norm_copy_off(own));
    cudaError_t e = launch_rownorm_ssq(X, M, K, ldx, norm->in_ssq, norm->in_tiles, norm->eps, Xn, K, s);
    if (e != cudaSuccess) return cuda_fail(e, "row normalisation launch");
    X = Xn;
    ldx = K;
    extra = 1;
  }
  spec_rownorm tmp{};
  const spec_rownorm* pn = plan_norm(norm, p, &tmp);
  if (pn) tmp.out_ssq = nullptr;   // (the SwiGLU epilogues do not sum squares: the pass below does)
  const int rc = swiglu_plan(p, X, M, K, ldx, Wgu, ldw, I, A, lda, pn, ws, d, s);
  if (rc) return rc;
  int n = t_launches + extra;
  if (norm_out(norm)) {
    cudaError_t e = launch_row_ssq(A, M, I, lda, norm->out_ssq, s);
    if (e != cudaSuccess) return cuda_fail(e, "sum-of-squares launch");
    ++n;
  }
  return ok(n);
}

static int swiglu_plan(const LinPlan& p, const spec_bf16* X, int M, int K, int ldx, const spec_bf16* Wgu, int ldw,
                       int I, spec_bf16* A, int lda, const spec_rownorm* norm, char* ws, DevInfo* d, cudaStream_t s) {
  const int N = 2 * I;
  if (p.gemv) {
    spec_bf16* gu = reinterpret_cast<spec_bf16*>(ws + swiglu_gemv_scratch_off(p));
    GemvArgs g;
    g.X = X; g.ldx = ldx; g.W = Wgu; g.ldw = ldw; g.Y = gu; g.ldy = N;
    g.residual = nullptr; g.ldr = 0; g.M = M; g.N = N; g.K = K;
    g.splits = p.splits; g.k_per_split = p.k_per_split;
    g.partial = p.splits > 1 ? reinterpret_cast<float*>(ws + p.partial_off) : nullptr;
    g.counters = p.splits > 1 ? reinterpret_cast<unsigned*>(ws + p.counters_off) : nullptr;
    cudaError_t e = launch_gemv(g, p.gemv_grid, s);
    if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
    e = launch_swiglu_interleaved(gu, M, I, N, A, lda, s);
    if (e != cudaSuccess) return cuda_fail(e, "swiglu launch");
    return ok(2);
  }
  CUtensorMap tw, tx;
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    cuuint64_t str[1] = {(cuuint64_t)ldw * 2};
    cuuint32_t box[2] = {LIN_BK, 128};
    if (int rc = encode_bf16(&tw, Wgu, 2, dims, str, box, "Wgu", g_w_promotion, kLinSwizzle)) return rc;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t str[1] = {(cuuint64_t)ldx * 2};
    cuuint32_t box[2] = {LIN_BK, (cuuint32_t)p.x_box_rows()};
    if (int rc = encode_bf16(&tx, X, 2, dims, str, box, "X", 3, kLinSwizzle)) return rc;
  }
  LinearArgs a{};
  a.M = M; a.N = N; a.K = K; a.k_tiles = p.k_tiles; a.tiles_m = p.tiles_m; a.tiles_n = p.tiles_n;
  a.units = p.units; a.grid = p.grid; a.dp_tiles = p.dp_tiles; a.sk_units = p.sk_units;
  a.Y = A; a.ldy = lda; a.residual = nullptr; a.ldr = 0;
  a.partial = p.bytes > 0 ? reinterpret_cast<float*>(ws + p.partial_off) : nullptr;
  a.status = d->status;
  a.w_early = g_weight_prefetch;
  a.tn = p.BN * p.NSUB;
  a.epi = EPI_SWIGLU;
  set_norm_args(a, norm, K);
  if (p.tc_pair) {
    const int n = launch_tc_pair_plan(p, tw, tx, a, s);
    return n > 0 ? ok(n) : n;
  }
  if (p.pair_n > 0) {
    cudaError_t e = cudaSuccess;
    const int n = launch_pair_plan(p, tw, tx, a, s, &e);
    if (!n) return cuda_fail(e, "pair swiglu linear launch");
    return ok(n);
  }
  if (p.cluster_S > 0) {
    cudaError_t e = launch_linear_cluster(p.BN, p.NSUB, tw, tx, a, p.cluster_S, p.grid / p.cluster_S, s);
    if (e != cudaSuccess) return cuda_fail(e, "cluster swiglu linear launch");
    return ok(1);
  }
  cudaError_t e = launch_linear_tc_swiglu(p.BN, p.NSUB, tw, tx, a, dim3(p.grid), s);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 swiglu linear launch");
  if (p.rem_S > 0) {
    e = launch_linear_cluster(p.BN, p.NSUB, tw, tx, a, p.rem_S, (int)p.rem_tiles, s);
    if (e != cudaSuccess) return cuda_fail(e, "cluster swiglu linear launch (remainder)");
    return ok(2);
  }
  if (p.bytes == 0) return ok(1);
  e = launch_linear_reduce(a, plan_sms(), s);
  if (e != cudaSuccess) return cuda_fail(e, "split-K reduce launch");
  return ok(2);
}

extern "C" {

int spec_verify_linear_swiglu(const spec_bf16* X, int M, int K, int ldx, const spec_bf16* Wgu, int ldw,
                              int I, spec_bf16* A, int lda, void* workspace, size_t workspace_bytes,
                              spec_stream stream) {
  return verify_linear_swiglu_impl(X, M, K, ldx, Wgu, ldw, I, A, lda, nullptr, workspace, workspace_bytes, stream);
}

int spec_verify_linear_swiglu_norm(const spec_bf16* X, int M, int K, int ldx, const spec_bf16* Wgu, int ldw, int I,
                                   spec_bf16* A, int lda, const spec_rownorm* norm, void* workspace,
                                   size_t workspace_bytes, spec_stream stream) {
  return verify_linear_swiglu_impl(X, M, K, ldx, Wgu, ldw, I, A, lda, norm, workspace, workspace_bytes, stream);
}

// --------------------------------------------------------------------------- LM head
size_t spec_lmhead_workspace_bytes(int M, int K, int V) {
  if (M <= 0 || K <= 0 || V <= 0) return 0;
  return plan_linear(M, V, K, true).bytes;
}

// The LM-head GEMM: z / T of every row into Z (T > 0) and per-128-token-tile statistics (max,
// sum of exp; or max, argmax when T = 0) into the workspace after its counter region.
static int launch_lmhead_gemm(const spec_bf16* H, int M, int K, const spec_bf16* Wlm, int V, float temperature,
                              float* Z, long long ldz, void* workspace, const LinPlan& p, DevInfo* d, cudaStream_t s,
                              float2** stats_out, const spec_rownorm* norm = nullptr) {
  CUtensorMap tw, tx;
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)V};
    cuuint64_t str[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {LIN_BK, 128};
    if (int rc = encode_bf16(&tw, Wlm, 2, dims, str, box, "Wlm", g_w_promotion, kLinSwizzle)) return rc;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t str[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {LIN_BK, (cuuint32_t)p.x_box_rows()};
    if (int rc = encode_bf16(&tx, H, 2, dims, str, box, "H", 3, kLinSwizzle)) return rc;
  }
  const bool greedy = temperature == 0.f;
  LinearArgs a{};
  a.M = M; a.N = V; a.K = K; a.k_tiles = p.k_tiles; a.tiles_m = p.tiles_m; a.tiles_n = p.tiles_n;
  a.units = p.units; a.grid = p.grid; a.dp_tiles = p.dp_tiles; a.sk_units = p.sk_units;
  a.status = d->status;
  a.w_early = g_weight_prefetch;
  a.inv_temp = greedy ? 1.f : 1.f / temperature;
  a.P = Z;
  a.ldp = ldz;
  a.stats = reinterpret_cast<float2*>(static_cast<char*>(workspace) + p.partial_off);
  // a folded final RMSNorm scales each row's logits (the argmax of a row does not change)
  if (norm_in(norm)) {
    a.norm_ssq = norm->in_ssq;
    a.norm_tiles = norm->in_tiles;
    a.norm_k = (float)K;
    a.norm_eps = norm->eps;
  }
  cudaError_t e;
  if (p.tc_pair) {
    a.pair = 1;
    e = launch_linear_tc_pair(p.BN, p.NSUB, greedy ? EPI_ARGMAX : EPI_LOGITS, tw, tx, a, p.grid, s);
  } else {
    e = launch_linear_tc_lmhead(p.BN, p.NSUB, greedy, tw, tx, a, dim3(p.grid), s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "LM-head GEMM launch");
  *stats_out = a.stats;
  return SPEC_OK;
}

static int check_lmhead_args(const spec_bf16* H, int M, int K, const spec_bf16* Wlm, int V, float temperature) {
  if (!H || !Wlm) return fail(SPEC_EINVAL, "H and Wlm must be non-NULL");
  if (K % 8) return fail(SPEC_EINVAL, "K=%d must be a multiple of 8", K);
  if (V % 4) return fail(SPEC_EINVAL, "V=%d must be a multiple of 4", V);
  if (!(temperature >= 0.f) || std::isinf(temperature))
    return fail(SPEC_EINVAL, "temperature must be finite and >= 0");
  if (!aligned16(H) || !aligned16(Wlm)) return fail(SPEC_EINVAL, "H, Wlm must be 16-byte aligned");
  (void)M;
  return SPEC_OK;
}

int spec_lmhead_softmax(const spec_bf16* H, int M, int K, const spec_bf16* Wlm, int V,
                        float temperature, float* P, void* workspace, size_t workspace_bytes,
                        spec_stream stream) {
  return spec_lmhead_softmax_ld(H, M, K, Wlm, V, temperature, P, V, workspace, workspace_bytes, stream);
}

int spec_lmhead_softmax_ld(const spec_bf16* H, int M, int K, const spec_bf16* Wlm, int V, float temperature,
                           float* P, long long ldp, void* workspace, size_t workspace_bytes, spec_stream stream) {
  if (M < 0 || K <= 0 || V <= 0) return fail(SPEC_EINVAL, "bad sizes M=%d K=%d V=%d", M, K, V);
  if (M == 0) return ok();
  if (int rc = check_lmhead_args(H, M, K, Wlm, V, temperature)) return rc;
  if (!P) return fail(SPEC_EINVAL, "P must be non-NULL");
  if (ldp < V || ldp % 4) return fail(SPEC_EINVAL, "ldp=%lld must be >= V and a multiple of 4", ldp);
  if (!aligned16(P)) return fail(SPEC_EINVAL, "P must be 16-byte aligned");
  LinPlan p = plan_linear(M, V, K, true);
  if (!workspace || workspace_bytes < p.bytes)
    return fail(SPEC_EINVAL, "workspace too small: need %zu bytes", p.bytes);
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float2* stats = nullptr;
  if (int rc = launch_lmhead_gemm(H, M, K, Wlm, V, temperature, P, ldp, workspace, p, d, s, &stats)) return rc;
  cudaError_t e = launch_lmhead_normalize(P, ldp, stats, M, V, p.tiles_n, temperature == 0.f, s);
  if (e != cudaSuccess) return cuda_fail(e, "LM-head normalize launch");
  return ok(2);
}

// --------------------------------------------------------------------------- fused LM head -> sampler
// Workspace: counters + per-tile statistics, then (T > 0) the logits z / T [M x V] fp32.
static size_t fused_logits_off(const LinPlan& p) { return round_up(p.bytes, 256); }

size_t spec_lmhead_sample_workspace_bytes(int M, int K, int V, float temperature) {
  if (M <= 0 || K <= 0 || V <= 0) return 0;
  const LinPlan p = plan_linear(M, V, K, true);
  return temperature == 0.f ? p.bytes : fused_logits_off(p) + round_up(size_t(M) * V * 4, 256);
}

}  // extern "C"

static int lmhead_reject_sample_impl(const spec_bf16* H, int M, int K, const spec_bf16* Wlm, int V, float temperature,
                              const float* Q, const int32_t* draft_tok, const float* U, const int32_t* cu_rows,
                              int B, float tie_eps, int32_t* n_acc, int32_t* out_tok, int32_t* near_tie,
                              const spec_rownorm* norm, void* workspace, size_t workspace_bytes, spec_stream stream) {
  if (M < 0 || K <= 0 || V <= 0 || B < 0) return fail(SPEC_EINVAL, "bad sizes M=%d K=%d V=%d B=%d", M, K, V, B);
  if (B == 0) return ok();
  if (M < B) return fail(SPEC_EINVAL, "M=%d verify rows cannot hold B=%d sequences", M, B);
  if (int rc = check_lmhead_args(H, M, K, Wlm, V, temperature)) return rc;
  if (!Q || !draft_tok || !U || !cu_rows || !n_acc || !out_tok || !near_tie)
    return fail(SPEC_EINVAL, "NULL argument");
  if (!(tie_eps >= 0.f)) return fail(SPEC_EINVAL, "tie_eps must be >= 0");
  if (V > (1 << 20)) return fail(SPEC_EUNSUPPORTED, "V=%d > 1048576", V);
  if (int rc = check_norm(norm)) return rc;
  const LinPlan p = plan_linear(M, V, K, true);
  const size_t need = spec_lmhead_sample_workspace_bytes(M, K, V, temperature);
  if (!workspace || workspace_bytes < need) return fail(SPEC_EINVAL, "workspace too small: need %zu bytes", need);
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool greedy = temperature == 0.f;
  float* Z = greedy ? nullptr : reinterpret_cast<float*>(static_cast<char*>(workspace) + fused_logits_off(p));
  float2* stats = nullptr;
  if (int rc = launch_lmhead_gemm(H, M, K, Wlm, V, temperature, Z, V, workspace, p, d, s, &stats, norm)) return rc;
  cudaError_t e = launch_reject_sample_logits(Z, stats, p.tiles_n, greedy, Q, draft_tok, U, cu_rows, B, M, V,
                                              tie_eps, n_acc, out_tok, near_tie, d->status, s);
  if (e != cudaSuccess) return cuda_fail(e, "fused sampler launch");
  return ok(2);
}

extern "C" {

int spec_lmhead_reject_sample(const spec_bf16* H, int M, int K, const spec_bf16* Wlm, int V, float temperature,
                              const float* Q, const int32_t* draft_tok, const float* U, const int32_t* cu_rows,
                              int B, float tie_eps, int32_t* n_acc, int32_t* out_tok, int32_t* near_tie,
                              void* workspace, size_t workspace_bytes, spec_stream stream) {
  return lmhead_reject_sample_impl(H, M, K, Wlm, V, temperature, Q, draft_tok, U, cu_rows, B, tie_eps, n_acc, out_tok,
                                   near_tie, nullptr, workspace, workspace_bytes, stream);
}

int spec_lmhead_reject_sample_norm(const spec_bf16* H, int M, int K, const spec_bf16* Wlm, int V, float temperature,
                                   const float* Q, const int32_t* draft_tok, const float* U, const int32_t* cu_rows,
                                   int B, float tie_eps, int32_t* n_acc, int32_t* out_tok, int32_t* near_tie,
                                   const spec_rownorm* norm, void* workspace, size_t workspace_bytes,
                                   spec_stream stream) {
  return lmhead_reject_sample_impl(H, M, K, Wlm, V, temperature, Q, draft_tok, U, cu_rows, B, tie_eps, n_acc, out_tok,
                                   near_tie, norm, workspace, workspace_bytes, stream);
}

// --------------------------------------------------------------------------- attention
size_t spec_attention_workspace_bytes(int B, int max_rows, int Hq, int Hkv, int D, int cap) {
  if (B <= 0 || max_rows <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || cap <= 0) return 0;
  return plan_attention(B, max_rows, Hq, Hkv, cap).bytes;
}

// Contiguous cache (block_table == nullptr: [B][Hkv][cap][D]) or paged pools ([Hkv][num_pages][128][D],
// key tile t of sequence b in page block_table[b * max_pages + t]; cap = max_pages * 128 keys).
static int verify_attention_impl(const spec_bf16* Q, int ldq, const spec_bf16* Knew, const spec_bf16* Vnew,
                                 int ldkv, const int32_t* cu_rows, const int32_t* ctx_len, int B, int max_rows,
                                 spec_bf16* Kcache, spec_bf16* Vcache, int cap, const int32_t* block_table,
                                 int max_pages, int num_pages, int Hq, int Hkv, int D, float scale, spec_bf16* O,
                                 int ldo, void* workspace, size_t workspace_bytes, spec_stream stream) {
  if (B < 0) return fail(SPEC_EINVAL, "B=%d < 0", B);
  if (B == 0) return ok();
  if (!Q || !Knew || !Vnew || !cu_rows || !ctx_len || !Kcache || !Vcache || !O)
    return fail(SPEC_EINVAL, "NULL tensor argument");
  if (D != 128) return fail(SPEC_EUNSUPPORTED, "head_dim %d: only 128 is implemented", D);
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv) return fail(SPEC_EINVAL, "Hq=%d must be a multiple of Hkv=%d", Hq, Hkv);
  const int G = Hq / Hkv;
  if ((size_t)B * Hkv > kMaxCounters) return fail(SPEC_EUNSUPPORTED, "B*Hkv = %d > %zu", B * Hkv, kMaxCounters);
  if (max_rows <= 0) return fail(SPEC_EINVAL, "max_rows must be >= 1");
  if (G * max_rows > 64)
    return fail(SPEC_EUNSUPPORTED, "(Hq/Hkv)*max_rows = %d > 64 query rows per kv head", G * max_rows);
  if (cap <= 0) return fail(SPEC_EINVAL, "cap must be >= 1");
  if (ldq < Hq * D || ldkv < Hkv * D || ldo < Hq * D || ldq % 8 || ldkv % 8 || ldo % 8)
    return fail(SPEC_EINVAL, "bad leading dimensions");
  if (!aligned16(Q) || !aligned16(Knew) || !aligned16(Vnew) || !aligned16(Kcache) ||
      !aligned16(Vcache) || !aligned16(O))
    return fail(SPEC_EINVAL, "bf16 tensors must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(SPEC_EINVAL, "scale must be finite");
  AttnPlan p = plan_attention(B, max_rows, Hq, Hkv, cap);
  if (block_table && !p.tc)
    return fail(SPEC_EUNSUPPORTED, "the paged cache needs the tcgen05 attention kernel (attention_impl 1)");
  if (!workspace || workspace_bytes < p.bytes)
    return fail(SPEC_EINVAL, "workspace too small: need %zu bytes", p.bytes);
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  CUtensorMap tk, tv;
  const int kt = attention_tc_key_tile();
  const cuuint64_t rows = block_table ? (cuuint64_t)kt : (cuuint64_t)cap;
  const cuuint64_t zs = block_table ? (cuuint64_t)num_pages * Hkv : (cuuint64_t)B * Hkv;
  cuuint64_t dims[3] = {(cuuint64_t)D, rows, zs};
  cuuint64_t str[2] = {(cuuint64_t)D * 2, rows * D * 2};
  cuuint32_t box[3] = {64, p.tc ? (cuuint32_t)kt : 64u, 1};
  if (int rc = encode_bf16(&tk, Kcache, 3, dims, str, box, "Kcache", g_kv_promotion)) return rc;
  if (int rc = encode_bf16(&tv, Vcache, 3, dims, str, box, "Vcache", g_kv_promotion)) return rc;
  char* ws = static_cast<char*>(workspace);
  AttnArgs a{};
  a.Q = Q; a.ldq = ldq; a.Knew = Knew; a.Vnew = Vnew; a.ldkv = ldkv;
  a.cu_rows = cu_rows; a.ctx_len = ctx_len; a.Kc = Kcache; a.Vc = Vcache; a.cap = cap;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.G = G; a.max_rows = max_rows;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.O = O; a.ldo = ldo;
  a.chunk = p.chunk; a.max_chunks = p.max_chunks;
  a.partial = reinterpret_cast<float*>(ws + p.partial_off);
  a.counters = reinterpret_cast<unsigned*>(ws + p.counters_off);
  a.status = d->status;
  a.pair_cost = g_attn_pair_cost;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.pfx = reinterpret_cast<int*>(ws + p.pfx_off);
  cudaError_t e = p.tc ? launch_attention_tc(tk, tv, a, p.grid, static_cast<cudaStream_t>(stream))
                       : launch_attention(tk, tv, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return ok(1);
}

int spec_verify_attention(const spec_bf16* Q, int ldq, const spec_bf16* Knew,
                          const spec_bf16* Vnew, int ldkv, const int32_t* cu_rows,
                          const int32_t* ctx_len, int B, int max_rows, spec_bf16* Kcache,
                          spec_bf16* Vcache, int cap, int Hq, int Hkv, int D, float scale,
                          spec_bf16* O, int ldo, void* workspace, size_t workspace_bytes,
                          spec_stream stream) {
  return verify_attention_impl(Q, ldq, Knew, Vnew, ldkv, cu_rows, ctx_len, B, max_rows, Kcache, Vcache, cap,
                               nullptr, 0, 0, Hq, Hkv, D, scale, O, ldo, workspace, workspace_bytes, stream);
}

size_t spec_attention_paged_workspace_bytes(int B, int max_rows, int Hq, int Hkv, int D, int max_pages) {
  if (max_pages <= 0) return 0;
  return spec_attention_workspace_bytes(B, max_rows, Hq, Hkv, D, max_pages * attention_tc_key_tile());
}

int spec_verify_attention_paged(const spec_bf16* Q, int ldq, const spec_bf16* Knew, const spec_bf16* Vnew,
                                int ldkv, const int32_t* cu_rows, const int32_t* ctx_len, int B, int max_rows,
                                spec_bf16* Kpool, spec_bf16* Vpool, int num_pages, const int32_t* block_table,
                                int max_pages, int Hq, int Hkv, int D, float scale, spec_bf16* O, int ldo,
                                void* workspace, size_t workspace_bytes, spec_stream stream) {
  if (B > 0 && !block_table) return fail(SPEC_EINVAL, "block_table must be non-NULL");
  if (B > 0 && (num_pages <= 0 || max_pages <= 0))
    return fail(SPEC_EINVAL, "num_pages=%d and max_pages=%d must be >= 1", num_pages, max_pages);
  if ((long long)max_pages * attention_tc_key_tile() > INT32_MAX / 2)
    return fail(SPEC_EINVAL, "max_pages=%d too large", max_pages);
  return verify_attention_impl(Q, ldq, Knew, Vnew, ldkv, cu_rows, ctx_len, B, max_rows, Kpool, Vpool,
                               max_pages * attention_tc_key_tile(), block_table, max_pages, num_pages, Hq, Hkv, D,
                               scale, O, ldo, workspace, workspace_bytes, stream);
}

// --------------------------------------------------------------------------- sampler
int spec_reject_sample(const float* P, const float* Q, const int32_t* draft_tok, const float* U,
                       const int32_t* cu_rows, int B, int V, float tie_eps, int32_t* n_acc,
                       int32_t* out_tok, int32_t* near_tie, spec_stream stream) {
  if (B < 0 || V <= 0) return fail(SPEC_EINVAL, "bad sizes B=%d V=%d", B, V);
  if (B == 0) return ok();
  if (!P || !Q || !draft_tok || !U || !cu_rows || !n_acc || !out_tok || !near_tie)
    return fail(SPEC_EINVAL, "NULL argument");
  if (!(tie_eps >= 0.f)) return fail(SPEC_EINVAL, "tie_eps must be >= 0");
  if (V > (1 << 20)) return fail(SPEC_EUNSUPPORTED, "V=%d > 1048576", V);
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  cudaError_t e = launch_reject_sample(P, Q, draft_tok, U, cu_rows, B, V, tie_eps, n_acc, out_tok,
                                       near_tie, d->status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "reject_sample launch");
  return ok(1);
}

int spec_sample_rows(const float* P, long long ldp, int M, int V, const float* U, int32_t* out_tok,
                     spec_stream stream) {
  if (M < 0 || V <= 0) return fail(SPEC_EINVAL, "bad sizes M=%d V=%d", M, V);
  if (M == 0) return ok();
  if (!P || !U || !out_tok) return fail(SPEC_EINVAL, "NULL argument");
  if (ldp < V) return fail(SPEC_EINVAL, "ldp=%lld < V=%d", ldp, V);
  if (V > (1 << 20)) return fail(SPEC_EUNSUPPORTED, "V=%d > 1048576", V);
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  cudaError_t e = launch_sample_rows(P, ldp, M, V, U, out_tok, d->status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sample_rows launch");
  return ok(1);
}

int spec_typical_sample(const float* P, const int32_t* draft_tok, const float* U, const int32_t* cu_rows, int B,
                        int V, float epsilon, float delta, float tie_eps, int32_t* n_acc, int32_t* out_tok,
                        int32_t* near_tie, spec_stream stream) {
  if (B < 0 || V <= 0) return fail(SPEC_EINVAL, "bad sizes B=%d V=%d", B, V);
  if (B == 0) return ok();
  if (!P || !draft_tok || !U || !cu_rows || !n_acc || !out_tok || !near_tie)
    return fail(SPEC_EINVAL, "NULL argument");
  if (!(tie_eps >= 0.f)) return fail(SPEC_EINVAL, "tie_eps must be >= 0");
  if (!(epsilon >= 0.f) || !(delta >= 0.f) || std::isinf(epsilon) || std::isinf(delta))
    return fail(SPEC_EINVAL, "epsilon and delta must be finite and >= 0");
  if (V > (1 << 20)) return fail(SPEC_EUNSUPPORTED, "V=%d > 1048576", V);
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  cudaError_t e = launch_typical_sample(P, draft_tok, U, cu_rows, B, V, epsilon, delta, tie_eps, n_acc, out_tok,
                                        near_tie, d->status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "typical_sample launch");
  return ok(1);
}

// --------------------------------------------------------------------------- n-gram drafter
int spec_ngram_propose(const int32_t* tokens, const int32_t* cu_len, int B, int k, int n_min, int n_max,
                       int32_t* drafts, int32_t* n_drafts, spec_stream stream) {
  if (B < 0) return fail(SPEC_EINVAL, "B=%d < 0", B);
  if (B == 0) return ok();
  if (!tokens || !cu_len || !drafts || !n_drafts) return fail(SPEC_EINVAL, "NULL argument");
  if (k < 1 || k > 4096) return fail(SPEC_EINVAL, "k=%d must be in [1, 4096]", k);
  if (n_min < 1 || n_max < n_min || n_max > NGRAM_MAX_WINDOW)
    return fail(SPEC_EINVAL, "window [%d, %d] must satisfy 1 <= n_min <= n_max <= %d", n_min, n_max,
                NGRAM_MAX_WINDOW);
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  cudaError_t e = launch_ngram_propose(tokens, cu_len, B, k, n_min, n_max, drafts, n_drafts, d->status,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ngram_propose launch");
  return ok(1);
}

// --------------------------------------------------------------------------- glue
int spec_rmsnorm(const spec_bf16* X, int M, int N, int ldx, const spec_bf16* w, float eps,
                 spec_bf16* Y, int ldy, spec_stream stream) {
  if (M < 0 || N <= 0) return fail(SPEC_EINVAL, "bad sizes");
  if (M == 0) return ok();
  if (!X || !w || !Y) return fail(SPEC_EINVAL, "NULL argument");
  if (N % 8 || N > 16384) return fail(SPEC_EUNSUPPORTED, "N=%d must be a multiple of 8 and <= 16384", N);
  if (ldx < N || ldy < N || ldx % 8 || ldy % 8) return fail(SPEC_EINVAL, "bad leading dimensions");
  if (!aligned16(X) || !aligned16(w) || !aligned16(Y)) return fail(SPEC_EINVAL, "16-byte alignment");
  if (!(eps >= 0.f)) return fail(SPEC_EINVAL, "eps must be >= 0");
  cudaError_t e = launch_rmsnorm(X, M, N, ldx, w, eps, Y, ldy, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rmsnorm launch");
  return ok(1);
}

int spec_embed(const int32_t* ids, int M, const spec_bf16* table, int V, int d, int ldt, spec_bf16* X, int ldx,
               spec_stream stream) {
  if (M < 0 || V <= 0 || d <= 0) return fail(SPEC_EINVAL, "bad sizes M=%d V=%d d=%d", M, V, d);
  if (M == 0) return ok();
  if (!ids || !table || !X) return fail(SPEC_EINVAL, "NULL argument");
  if (d % 8 || ldt < d || ldx < d || ldt % 8 || ldx % 8)
    return fail(SPEC_EINVAL, "d, ldt, ldx must be multiples of 8 with ldt, ldx >= d");
  if (!aligned16(table) || !aligned16(X)) return fail(SPEC_EINVAL, "table and X must be 16-byte aligned");
  DevInfo* dv = nullptr;
  if (int rc = dev_info(&dv)) return rc;
  cudaError_t e = launch_embed(ids, M, table, V, d, ldt, X, ldx, dv->status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "embed launch");
  return ok(1);
}

int spec_rope(spec_bf16* Q, int ldq, int Hq, spec_bf16* K, int ldk, int Hkv, int D,
              const int32_t* cu_rows, const int32_t* ctx_len, int B, int M, float theta,
              spec_stream stream) {
  if (M < 0 || B < 0) return fail(SPEC_EINVAL, "bad sizes");
  if (M == 0) return ok();
  if (B == 0) return fail(SPEC_EINVAL, "rows without sequences");
  if (!Q || !K || !cu_rows || !ctx_len) return fail(SPEC_EINVAL, "NULL argument");
  if (D <= 0 || D % 2 || D > 256) return fail(SPEC_EUNSUPPORTED, "D=%d must be even and <= 256", D);
  if (Hq < 0 || Hkv < 0 || ldq < Hq * D || ldk < Hkv * D) return fail(SPEC_EINVAL, "bad heads / strides");
  if (!(theta > 0.f)) return fail(SPEC_EINVAL, "theta must be > 0");
  cudaError_t e = launch_rope(Q, ldq, Hq, K, ldk, Hkv, D, cu_rows, ctx_len, B, M, theta,
                              static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rope launch");
  return ok(1);
}

int spec_silu_mul(const spec_bf16* GU, int M, int I, int ldgu, spec_bf16* A, int lda,
                  spec_stream stream) {
  if (M < 0 || I <= 0) return fail(SPEC_EINVAL, "bad sizes");
  if (M == 0) return ok();
  if (!GU || !A) return fail(SPEC_EINVAL, "NULL argument");
  if (I % 8 || ldgu < 2 * I || lda < I || ldgu % 8 || lda % 8) return fail(SPEC_EINVAL, "bad sizes / strides");
  if (!aligned16(GU) || !aligned16(A)) return fail(SPEC_EINVAL, "16-byte alignment");
  cudaError_t e = launch_silu_mul(GU, M, I, ldgu, A, lda, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "silu_mul launch");
  return ok(1);
}

}  // extern "C"

// =========================================================================== allocation-free linear
// Scratch for spec_verify_linear_noalloc: a file-scope device array (zero at
// module load).  Host code must not pass the symbol itself to a kernel: in
// host code it is only a stand-in, so its device address is looked up once
// per device with that device current and cached here.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

namespace {
struct NoallocSlot {
  CUcontext ctx = nullptr;
  void* ptr = nullptr;
};
NoallocSlot g_noalloc[64];
std::mutex g_noalloc_mu;

int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(SPEC_EUNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoallocSlot& sl = g_noalloc[dev];
  if (int rc = symbol_address(g_noalloc_scratch, "cudaGetSymbolAddress(static scratch)", &sl.ctx, &sl.ptr))
    return rc;
  *out = sl.ptr;
  return SPEC_OK;
}
}  // namespace

extern "C" int spec_verify_linear_noalloc(const spec_bf16* X, int M, int K, int ldx,
                                          const spec_bf16* W, int N, int ldw, spec_bf16* Y,
                                          int ldy, const spec_bf16* residual, int ldr,
                                          spec_stream stream) {
  if (M < 0 || N <= 0 || K <= 0) return fail(SPEC_EINVAL, "bad sizes M=%d N=%d K=%d", M, N, K);
  if (M == 0) return ok();
  // every argument check runs before anything touches the stream or the scratch
  if (int rc = check_linear_args(X, M, K, ldx, W, N, ldw, Y, ldy, residual, ldr)) return rc;
  // (plans are chosen among those whose scratch fits in the static array)
  const size_t need = plan_linear(M, N, K, false, false, SPEC_NOALLOC_SCRATCH_BYTES).bytes;
  if (need > SPEC_NOALLOC_SCRATCH_BYTES)
    return fail(SPEC_EUNSUPPORTED,
                "M=%d N=%d K=%d needs %zu bytes of split-K scratch; the static scratch holds %u "
                "(call spec_verify_linear with a workspace)", M, N, K, need,
                (unsigned)SPEC_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if (int rc = noalloc_scratch(&scratch)) return rc;
  if (need > 0) {
    // the arrival counters must start at zero whatever an earlier call left behind
    const size_t clear = need < kCounterBytes ? need : kCounterBytes;
    cudaError_t e = cudaMemsetAsync(scratch, 0, clear, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "clear static scratch counters");
  }
  return verify_linear_impl(X, M, K, ldx, W, N, ldw, Y, ldy, residual, ldr, nullptr, scratch,
                            SPEC_NOALLOC_SCRATCH_BYTES, stream, SPEC_NOALLOC_SCRATCH_BYTES);
}
