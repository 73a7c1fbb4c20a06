// Verify attention on tcgen05 tensor cores: persistent, stream-K over key tiles.
//
// Work: for every (sequence b, kv head h) the R = G * (gamma_b + 1) query rows
// of the group (padded to RP, a multiple of 16) attend keys 0 .. ctx_b + gamma_b
// under the causal rule "row j sees keys <= ctx_b + j / G".  The keys of all
// (b, h) pairs are cut into 128-key tiles and concatenated (b-major, then h);
// one CTA per SM takes an equal contiguous range of tiles, so every SM streams
// the same number of K/V bytes whatever the context lengths.  A range covers
// whole (b, h) pairs and at most two partial ones; a partial pair's
// unnormalised output (O, running max, running sum) goes to the workspace and
// the CTA that arrives last on the pair's counter merges the pieces in CTA
// order (no waiting anywhere).
//
// Per tile (roles: warps 0-3 softmax + epilogue, warp 4 loads, warp 5 MMA/TMEM):
//   S^T[key, row] = K_tile . Q^T     tcgen05.mma M = 128 keys, N = RP, K = 128 dims
//   softmax (128 threads): scores staged through shared memory, then each query
//   row is owned by TPR threads (row max / exp2 / row sum, P row written bf16)
//   O^T[d, row] += V_tile^T . P^T    tcgen05.mma M = 128 dims (V read MN-major), N = RP
// K and V stream through separate 2-stage TMA rings (K is freed as soon as
// QK^T is done); Q is staged per pair into a double buffer; S^T and O^T are
// double buffered in TMEM so consecutive tiles and pairs overlap.  The newest
// gamma_b + 1 keys come from Knew/Vnew: the producer patches the tail tile
// after its load lands, and the CTA owning a pair's last tile writes the new
// block into the cache once its loads are done.
#include "common.cuh"
#include "internal.h"

namespace spec {
namespace {

constexpr int D = 128;
constexpr int KT = 128;                  // keys per tile = MMA M
constexpr int ST = 2;                    // K and V ring stages
constexpr int KV_HALF = KT * 128;        // 128 keys x 64 dims (128 B rows), 16 KB
constexpr int KV_TILE = 2 * KV_HALF;     // 32 KB
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;      // S^T x2 and O^T x2, 64 columns each
constexpr int MAX_B = 1024;              // sequences per call handled by this kernel

template <int RP>
struct TCfg {
  static constexpr int TPR = RP <= 16 ? 8 : (RP <= 32 ? 4 : 2);   // threads per query row
  static constexpr int KPT = KT / TPR;                            // keys per thread
  static constexpr int Q_HALF = RP * 128;                         // RP rows x 64 elements (bf16)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = ST * KV_TILE;
  static constexpr int OFF_Q = 2 * ST * KV_TILE;                  // 2 buffers x two halves
  static constexpr int OFF_P = OFF_Q + 2 * 2 * Q_HALF;            // P [RP][128 keys], two halves
  static constexpr int OFF_STG = OFF_P + 2 * Q_HALF;              // scores [RP][128 + TPR] fp32
  static constexpr int STG_ROW = KT + TPR;
  static constexpr int OFF_PFX = OFF_STG + ((RP * STG_ROW * 4 + 1023) / 1024) * 1024;
  static constexpr int OFF_BAR = OFF_PFX + (MAX_B + 1) * 4 * 2;   // unit prefix + tiles per seq
  static constexpr int OFF_ROW = OFF_BAR + 256;                    // m[64], l[64], alpha[64], flag
  static constexpr int SMEM = OFF_ROW + 3 * 64 * 4 + 64 + 1024;
};

template <int RP>
__device__ __forceinline__ int stg_idx(int j, int k) {
  using C = TCfg<RP>;
  return j * C::STG_ROW + (k / C::KPT) * (C::KPT + 1) + (k % C::KPT);
}

__device__ __forceinline__ void bar_compute() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// AND of `v` over the 128 softmax threads (named barrier 1): keeps their control flow uniform.
__device__ __forceinline__ bool bar_compute_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.and.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Shared-memory descriptor of an MN-major operand stored as 128-byte swizzled
// rows (8-row atoms 1024 B apart along K; 64-element atom columns `lbo` apart along M/N).
__device__ __forceinline__ uint64_t umma_desc_sw128_mn(uint32_t smem_addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= uint64_t((smem_addr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t(1024 >> 4) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0],"
      " {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// The tile list: unit u -> (b, h, t).  pfx[b] = first unit of sequence b (pfx[B] = total),
// ntl[b] = tiles per (b, h) pair of sequence b.
struct Unit {
  int b, h, t, nt;
  long long pair0;      // first unit of the pair
};
__device__ __forceinline__ Unit unit_at(const int* pfx, const int* ntl, int B, long long u) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pfx[mid] <= u) lo = mid; else hi = mid - 1;
  }
  Unit r;
  r.b = lo;
  r.nt = ntl[lo];
  const int rem = (int)(u - pfx[lo]);
  r.h = rem / r.nt;
  r.t = rem - r.h * r.nt;
  r.pair0 = u - r.t;
  return r;
}
__device__ __forceinline__ long long range_begin(long long total, int grid, int c) {
  return total * c / grid;
}
__device__ __forceinline__ int cta_of(long long total, int grid, long long u) {
  int c = (int)(((u + 1) * grid - 1) / total);
  if (c >= grid) c = grid - 1;
  while (c + 1 < grid && range_begin(total, grid, c + 1) <= u) ++c;
  while (c > 0 && range_begin(total, grid, c) > u) --c;
  return c;
}

template <int RP>
__global__ void __launch_bounds__(THREADS, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const AttnArgs a) {
  using C = TCfg<RP>;
  constexpr int TPR = C::TPR, KPT = C::KPT;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int* pfx = reinterpret_cast<int*>(smem + C::OFF_PFX);
  int* ntl = pfx + (MAX_B + 1);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* k_full = bars;             // [ST]
  uint64_t* v_full = bars + 2;         // [ST]
  uint64_t* k_empty = bars + 4;        // [ST]  QK^T done with the K stage
  uint64_t* v_empty = bars + 6;        // [ST]  PV done with the V stage
  uint64_t* tail_ready = bars + 8;     // [ST]  tail tile (K and V) patched
  uint64_t* s_full = bars + 10;        // [2]   S^T in TMEM
  uint64_t* s_empty = bars + 12;       // [2]   softmax has read S^T
  uint64_t* p_full = bars + 14;        //       P in smem, O rescaled
  uint64_t* pv_done = bars + 15;       //       PV finished
  uint64_t* q_full = bars + 16;        // [2]   Q of a pair staged
  uint64_t* q_empty = bars + 18;       // [2]   last QK^T of a pair done
  uint64_t* o_empty = bars + 20;       // [2]   epilogue has read the O buffer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 22);
  float* stg = reinterpret_cast<float*>(smem + C::OFF_STG);
  float* row_m = reinterpret_cast<float*>(smem + C::OFF_ROW);
  float* row_l = row_m + 64;
  float* row_alpha = row_m + 128;
  unsigned* last_flag = reinterpret_cast<unsigned*>(row_m + 192);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int B = a.B, Hkv = a.Hkv, G = a.G;

  // ---- tile list prefix (warp 0 scans 32 sequences per step); bad rows/contexts are rejected
  if (warp == 0) {
    int carry = 0;
    bool bad = false;
    for (int base = 0; base < B; base += 32) {
      const int b = base + lane;
      int units = 0;
      if (b < B) {
        const int ctx = a.ctx_len[b];
        const int mb = a.cu_rows[b + 1] - a.cu_rows[b];
        bad |= (mb <= 0 || mb > a.max_rows || ctx < 0 || ctx + mb > a.cap || G * mb > RP);
        const int nt = mb > 0 ? (ctx + mb + KT - 1) / KT : 1;
        ntl[b] = nt > 0 ? nt : 1;
        units = ntl[b] * Hkv;
      }
      int incl = units;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (b < B) pfx[b] = carry + incl - units;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      pfx[B] = bad ? 0 : carry;           // nothing to do when the ragged arrays are invalid
      if (bad && blockIdx.x == 0) set_status(a.status, 0x2F1u);
    }
  }
  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&tail_ready[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 128);
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&o_empty[i], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long total = pfx[B];
  const int grid = gridDim.x;
  const long long ub = total > 0 ? range_begin(total, grid, blockIdx.x) : 0;
  const long long ue = total > 0 ? range_begin(total, grid, blockIdx.x + 1) : 0;

  if (warp == 4) {
    // ------------------------------------------------------------ producer: Q staging + K/V TMA
    bool ok = true;
    int piece = -1;
    long long i = 0;
    for (long long u = ub; u < ue && ok; ++u, ++i) {
      const Unit w = unit_at(pfx, ntl, B, u);
      const int ctx = a.ctx_len[w.b];
      const int r0 = a.cu_rows[w.b];
      const int Mb = a.cu_rows[w.b + 1] - r0;
      const int bh = w.b * Hkv + w.h;
      if (u == ub || w.t == 0) {
        // a new pair: stage its Q rows (row j = token row j / G, head j % G), zero-padded to RP
        ++piece;
        const int qb = piece & 1;
        if (piece >= 2) ok = mbar_wait(&q_empty[qb], ((piece >> 1) - 1) & 1, a.status, 0x210u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        uint8_t* qd = smem + C::OFF_Q + qb * 2 * C::Q_HALF;
        const int R = G * Mb;
        for (int idx = lane; idx < RP * 16; idx += 32) {
          const int j = idx >> 4, ch = idx & 15;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (j < R) {
            const int tr = j / G, g = j - tr * G;
            v = *reinterpret_cast<const uint4*>(a.Q + (size_t)(r0 + tr) * a.ldq + (size_t)(w.h * G + g) * D + ch * 8);
          }
          *reinterpret_cast<uint4*>(qd + (ch >> 3) * C::Q_HALF + sw128_off(j, (ch & 7) * 8)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full[qb]);
      }
      const int s = (int)(i % ST);
      const uint32_t ph = (uint32_t)(((i / ST) - 1) & 1);
      const int key0 = w.t * KT;
      uint8_t* kt = smem + C::OFF_K + s * KV_TILE;
      uint8_t* vt = smem + C::OFF_V + s * KV_TILE;
      if (i >= ST) ok = mbar_wait(&k_empty[s], ph, a.status, 0x211u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&k_full[s], KV_TILE);
        tma_load_3d(kt, &tmK, &k_full[s], 0, key0, bh);
        tma_load_3d(kt + KV_HALF, &tmK, &k_full[s], 64, key0, bh);
      }
      if (i >= ST) ok = mbar_wait(&v_empty[s], ph, a.status, 0x212u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&v_full[s], KV_TILE);
        tma_load_3d(vt, &tmV, &v_full[s], 0, key0, bh);
        tma_load_3d(vt + KV_HALF, &tmV, &v_full[s], 64, key0, bh);
      }
      if (key0 + KT > ctx) {
        // tail tile: wait for both loads, then overwrite keys >= ctx (new block, zeros past it)
        ok = mbar_wait(&k_full[s], (uint32_t)((i / ST) & 1), a.status, 0x213u) &&
             mbar_wait(&v_full[s], (uint32_t)((i / ST) & 1), a.status, 0x214u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const int rr0 = ctx > key0 ? ctx - key0 : 0;
        for (int idx = rr0 * 16 + lane; idx < KT * 16; idx += 32) {
          const int rr = idx >> 4, ch = idx & 15;
          const int p = key0 + rr;
          uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
          if (p < ctx + Mb) {
            const size_t off = (size_t)(r0 + p - ctx) * a.ldkv + (size_t)w.h * D + ch * 8;
            kv = *reinterpret_cast<const uint4*>(a.Knew + off);
            vv = *reinterpret_cast<const uint4*>(a.Vnew + off);
          }
          const uint32_t o = (ch >> 3) * KV_HALF + sw128_off(rr, (ch & 7) * 8);
          *reinterpret_cast<uint4*>(kt + o) = kv;
          *reinterpret_cast<uint4*>(vt + o) = vv;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail_ready[s]);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(128, RP);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(128, RP) | (1u << 15);   // A (V^T) MN-major
      const uint32_t p_addr = smem_u32(smem + C::OFF_P);
      const long long n_units = ue - ub;
      int tail_cnt[ST] = {0, 0};
      long long tail_done[ST] = {-1, -1};   // tile whose tail barrier was already consumed
      // wait until tile i can be read from stage i % ST (tail tiles: after the patch)
      auto wait_tile = [&](long long i, int key0, int ctx, uint64_t* full, unsigned site) -> bool {
        const int s = (int)(i % ST);
        if (key0 + KT > ctx) {
          if (tail_done[s] != i) {
            if (!mbar_wait(&tail_ready[s], tail_cnt[s] & 1, a.status, site)) return false;
            tail_cnt[s]++;
            tail_done[s] = i;
          }
          return true;
        }
        return mbar_wait(&full[s], (uint32_t)((i / ST) & 1), a.status, site);
      };
      // S^T(i) = K(i) . Q^T of its pair
      int piece_s = -1;
      auto do_s = [&](long long i) -> bool {
        const long long u = ub + i;
        const Unit w = unit_at(pfx, ntl, B, u);
        if (u == ub || w.t == 0) ++piece_s;
        const bool last = (u + 1 >= ue) || (w.t + 1 == w.nt);
        const int qb = piece_s & 1;
        if ((u == ub || w.t == 0) && !mbar_wait(&q_full[qb], (uint32_t)((piece_s >> 1) & 1), a.status, 0x225u))
          return false;
        if (!wait_tile(i, w.t * KT, a.ctx_len[w.b], k_full, 0x221u)) return false;
        if (i >= 2 && !mbar_wait(&s_empty[i & 1], (uint32_t)(((i >> 1) - 1) & 1), a.status, 0x222u)) return false;
        tc_fence_after();
        const int s = (int)(i % ST);
        const uint32_t k_addr = smem_u32(smem + C::OFF_K + s * KV_TILE);
        const uint32_t q_addr = smem_u32(smem + C::OFF_Q + qb * 2 * C::Q_HALF);
        const uint32_t d_s = tmem + (uint32_t)(i & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t ka = k_addr + (kk >> 2) * KV_HALF + (kk & 3) * 32;
          const uint32_t qa = q_addr + (kk >> 2) * C::Q_HALF + (kk & 3) * 32;
          umma_bf16(d_s, umma_desc_sw128(ka), umma_desc_sw128(qa), idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&k_empty[s]);
        umma_commit(&s_full[i & 1]);
        if (last) umma_commit(&q_empty[qb]);
        return true;
      };
      bool ok = n_units > 0 ? do_s(0) : true;
      int piece_p = -1;
      for (long long i = 0; i < n_units && ok; ++i) {
        if (i + 1 < n_units && !do_s(i + 1)) { ok = false; break; }
        const long long u = ub + i;
        const Unit w = unit_at(pfx, ntl, B, u);
        const bool first = (u == ub || w.t == 0);
        if (first) ++piece_p;
        const int ob = piece_p & 1;
        if (first && piece_p >= 2 &&
            !mbar_wait(&o_empty[ob], (uint32_t)(((piece_p >> 1) - 1) & 1), a.status, 0x226u)) { ok = false; break; }
        if (!mbar_wait(p_full, (uint32_t)(i & 1), a.status, 0x223u) ||
            !wait_tile(i, w.t * KT, a.ctx_len[w.b], v_full, 0x224u)) { ok = false; break; }
        tc_fence_after();
        const int s = (int)(i % ST);
        const uint32_t v_addr = smem_u32(smem + C::OFF_V + s * KV_TILE);
        const uint32_t t_o = tmem + 128 + (uint32_t)ob * 64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t va = v_addr + kk * 16 * 128;                     // 16 keys per step
          const uint32_t pa = p_addr + (kk >> 2) * C::Q_HALF + (kk & 3) * 32;
          umma_bf16(t_o, umma_desc_sw128_mn(va, KV_HALF), umma_desc_sw128(pa), idesc_pv,
                    (!first || kk > 0) ? 1u : 0u);
        }
        umma_commit(&v_empty[s]);
        umma_commit(pv_done);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue warps
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    const int row = tid / TPR, part = tid % TPR;
    const bool owner = row < RP;
    bool ok = true;
    int piece = -1;
    long long i = 0;
    for (long long u = ub; u < ue; ++u, ++i) {
      const Unit w = unit_at(pfx, ntl, B, u);
      const int ctx = a.ctx_len[w.b];
      const int r0 = a.cu_rows[w.b];
      const int Mb = a.cu_rows[w.b + 1] - r0;
      const int R = G * Mb;
      const bool first = (u == ub || w.t == 0);
      const bool last = (u + 1 >= ue) || (w.t + 1 == w.nt);
      if (first) {
        ++piece;
        if (tid < 64) {
          row_m[tid] = -INFINITY;
          row_l[tid] = 0.f;
        }
        bar_compute();
      }
      const int ob = piece & 1;
      const uint32_t t_o = tmem + 128 + (uint32_t)ob * 64 + lane_off;
      const int key0 = w.t * KT;
      const bool tail = key0 + KT > ctx;
      ok = ok && mbar_wait(&s_full[i & 1], (uint32_t)((i >> 1) & 1), a.status, 0x231u);
      ok = bar_compute_and(ok);
      if (!ok) break;
      tc_fence_after();
      {
        float sv[RP];
        tmem_ld_cols<RP>(tmem + (uint32_t)(i & 1) * 64 + lane_off, sv);
        tc_fence_before();
        mbar_arrive(&s_empty[i & 1]);
        const int p = key0 + tid;
#pragma unroll
        for (int j = 0; j < RP; ++j) {
          float v = sv[j] * a.scale_log2;
          if (tail && p > ctx + min(j / G, Mb - 1)) v = -INFINITY;
          stg[stg_idx<RP>(j, tid)] = v;
        }
      }
      bar_compute();
      float pv[KPT];
      bool grew = false;
      if (owner) {
        const float* src = stg + row * C::STG_ROW + part * (KPT + 1);
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < KPT; ++k) {
          pv[k] = src[k];
          mx = fmaxf(mx, pv[k]);
        }
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        // the running max only moves when the tile max exceeds it by more than 2^8: P <= 256
        // stays exact in bf16 and O, l keep using the same (stale) max, so the result is exact
        const float m_old = row_m[row];
        const float m_new = (mx > m_old + 8.f) ? mx : m_old;
        grew = m_new != m_old;
        const float base = m_new == -INFINITY ? 0.f : m_new;
        float sm = 0.f;
#pragma unroll
        for (int k = 0; k < KPT; ++k) {
          pv[k] = exp2f(pv[k] - base);
          sm += pv[k];
        }
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
        __syncwarp();
        if (part == 0) {
          const float alpha = exp2f(m_old - base);
          row_alpha[row] = alpha;
          row_l[row] = row_l[row] * alpha + sm;
          row_m[row] = m_new;
        }
      }
      // PV of the previous tile must be done before P is overwritten and O is rescaled
      if (i >= 1) {
        ok = mbar_wait(pv_done, (uint32_t)((i - 1) & 1), a.status, 0x232u);
        ok = bar_compute_and(ok);
        if (!ok) break;
      }
      if (owner) {
        uint8_t* prow = smem + C::OFF_P;
#pragma unroll
        for (int k = 0; k < KPT; k += 8) {
          const int kk = part * KPT + k;
          const uint4 wv = make_uint4(pack_bf16x2(pv[k], pv[k + 1]), pack_bf16x2(pv[k + 2], pv[k + 3]),
                                      pack_bf16x2(pv[k + 4], pv[k + 5]), pack_bf16x2(pv[k + 6], pv[k + 7]));
          *reinterpret_cast<uint4*>(prow + (kk >> 6) * C::Q_HALF + sw128_off(row, kk & 63)) = wv;
        }
      }
      const bool any_grew = !bar_compute_and(!grew);
      if (!first && any_grew) {
        tc_fence_after();
        float orr[RP];
        tmem_ld_cols<RP>(t_o, orr);
#pragma unroll
        for (int cc = 0; cc < RP; cc += 16) {
          float ov[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) ov[e] = orr[cc + e] * row_alpha[cc + e];
          tmem_st16(t_o + cc, ov);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
      if (!last) continue;

      // ---- piece epilogue: final O^T (lane = dim) once this tile's PV is done
      ok = mbar_wait(pv_done, (uint32_t)(i & 1), a.status, 0x233u);
      ok = bar_compute_and(ok);
      if (!ok) break;
      tc_fence_after();
      float ov[RP];
      tmem_ld_cols<RP>(t_o, ov);
      tc_fence_before();
      mbar_arrive(&o_empty[ob]);
      const int bh = w.b * Hkv + w.h;
      const long long pair_last = w.pair0 + w.nt - 1;
      const bool complete = (w.pair0 >= ub) && (u == pair_last);
      const int d = tid;
      if (complete) {
#pragma unroll
        for (int j = 0; j < RP; ++j) {
          if (j >= R) break;
          const int tr = j / G, g = j - tr * G;
          a.O[(size_t)(r0 + tr) * a.ldo + (size_t)(w.h * G + g) * D + d] = f2bf(ov[j] / row_l[j]);
        }
      } else {
        // slot 0: the piece that opens this CTA's range; slot 1: the piece that closes it
        const int slot = (w.pair0 < ub) ? 0 : 1;
        float* part_buf = a.partial + ((size_t)blockIdx.x * 2 + slot) * (64 * (D + 2));
#pragma unroll
        for (int j = 0; j < RP; ++j) {
          if (j >= R) break;
          __stcg(&part_buf[j * D + d], ov[j]);
        }
        if (tid < R) {
          __stcg(&part_buf[64 * D + tid * 2], row_m[tid]);
          __stcg(&part_buf[64 * D + tid * 2 + 1], row_l[tid]);
        }
      }
      // the owner of a pair's last tile writes the new block into the cache (its loads are done)
      if (u == pair_last) {
        for (int idx = tid; idx < Mb * 16 * 2; idx += 128) {
          const int which = idx / (Mb * 16);
          const int rem = idx - which * Mb * 16;
          const int j = rem >> 4, ch = rem & 15;
          const uint16_t* src = (which ? a.Vnew : a.Knew) + (size_t)(r0 + j) * a.ldkv + (size_t)w.h * D + ch * 8;
          uint16_t* dst = (which ? a.Vc : a.Kc) + ((size_t)bh * a.cap + ctx + j) * D + ch * 8;
          *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
        }
      }
      if (complete) continue;
      // ---- split pair: count this piece's tiles; the last arrival merges in CTA order
      __threadfence();
      bar_compute();
      if (tid == 0) {
        const long long piece_first = w.pair0 > ub ? w.pair0 : ub;
        const unsigned add = (unsigned)(u - piece_first + 1);
        const unsigned prev = atomicAdd(&a.counters[bh], add);
        *last_flag = (prev + add == (unsigned)w.nt) ? 1u : 0u;
      }
      bar_compute();
      const bool merge = *last_flag != 0u;
      bar_compute();
      if (!merge) continue;
      __threadfence();
      const int c_lo = cta_of(total, grid, w.pair0);
      const int c_hi = cta_of(total, grid, pair_last);
      const int n_c = c_hi - c_lo + 1;
      // per contributor and row: weight exp2(m_c - M) / L, staged in the (now idle) score buffer;
      // a pair has at most ceil(cap / 128) <= 128 contributors (the host keeps cap <= 16384 here)
      float* fac = stg;                                      // [n_c][RP]
      const int n_cs = n_c < 128 ? n_c : 128;
      if (tid < R) {
        const int j = tid;
        float M = -INFINITY;
        for (int cc = 0; cc < n_cs; ++cc) {
          const int c2 = c_lo + cc;
          const int sl = (range_begin(total, grid, c2) > w.pair0) ? 0 : 1;
          M = fmaxf(M, __ldcg(a.partial + ((size_t)c2 * 2 + sl) * (64 * (D + 2)) + 64 * D + j * 2));
        }
        const float mb = M == -INFINITY ? 0.f : M;
        float L = 0.f;
        for (int cc = 0; cc < n_cs; ++cc) {
          const int c2 = c_lo + cc;
          const int sl = (range_begin(total, grid, c2) > w.pair0) ? 0 : 1;
          const float* pk = a.partial + ((size_t)c2 * 2 + sl) * (64 * (D + 2));
          const float f = exp2f(__ldcg(&pk[64 * D + j * 2]) - mb);
          fac[cc * RP + j] = f;
          L += __ldcg(&pk[64 * D + j * 2 + 1]) * f;
        }
        const float inv = 1.f / L;
        for (int cc = 0; cc < n_cs; ++cc) fac[cc * RP + j] *= inv;
      }
      bar_compute();
      // O rows: 32 float4 per row; each thread owns up to 16 of the R * 32 items
      constexpr int IT = RP * 32 / 128;
      float4 acc[IT];
#pragma unroll
      for (int q2 = 0; q2 < IT; ++q2) acc[q2] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int cc = 0; cc < n_cs; ++cc) {
        const int c2 = c_lo + cc;
        const int sl = (range_begin(total, grid, c2) > w.pair0) ? 0 : 1;
        const float* pk = a.partial + ((size_t)c2 * 2 + sl) * (64 * (D + 2));
        float4 v[IT];
#pragma unroll
        for (int q2 = 0; q2 < IT; ++q2) {
          const int item = tid + q2 * 128;
          const int j = item >> 5, d4 = (item & 31) * 4;
          v[q2] = (j < R) ? __ldcg(reinterpret_cast<const float4*>(pk + j * D + d4)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q2 = 0; q2 < IT; ++q2) {
          const int j = (tid + q2 * 128) >> 5;
          const float f = j < R ? fac[cc * RP + j] : 0.f;
          acc[q2].x += f * v[q2].x; acc[q2].y += f * v[q2].y; acc[q2].z += f * v[q2].z; acc[q2].w += f * v[q2].w;
        }
      }
#pragma unroll
      for (int q2 = 0; q2 < IT; ++q2) {
        const int item = tid + q2 * 128;
        const int j = item >> 5, d4 = (item & 31) * 4;
        if (j >= R) continue;
        const int tr = j / G, g = j - tr * G;
        *reinterpret_cast<uint2*>(a.O + (size_t)(r0 + tr) * a.ldo + (size_t)(w.h * G + g) * D + d4) =
            make_uint2(pack_bf16x2(acc[q2].x, acc[q2].y), pack_bf16x2(acc[q2].z, acc[q2].w));
      }
      bar_compute();   // the score buffer is reused by the next tile
      if (tid == 0) a.counters[bh] = 0u;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tmem, TMEM_COLS);
}

template <int RP>
cudaError_t launch_rp(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, int grid,
                      cudaStream_t s) {
  constexpr int smem = TCfg<RP>::SMEM;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel<RP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  attention_tc_kernel<RP><<<grid, THREADS, smem, s>>>(tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

int attention_tc_key_tile() { return KT; }
int attention_tc_max_batch() { return MAX_B; }
int attention_tc_rows(int G, int max_rows) {
  const int rows = G * max_rows;
  if (rows > 64) return -1;
  const int rp = rows <= 16 ? 16 : (rows <= 32 ? 32 : (rows <= 48 ? 48 : 64));
  return rp;
}

cudaError_t launch_attention_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, int grid,
                                cudaStream_t s) {
  switch (attention_tc_rows(a.G, a.max_rows)) {
    case 16: return launch_rp<16>(tk, tv, a, grid, s);
    case 32: return launch_rp<32>(tk, tv, a, grid, s);
    case 48: return launch_rp<48>(tk, tv, a, grid, s);
    case 64: return launch_rp<64>(tk, tv, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spec
