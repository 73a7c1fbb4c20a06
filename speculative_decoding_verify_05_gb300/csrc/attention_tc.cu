// Verify attention on tcgen05 tensor cores (TMEM accumulators, TMA K/V stream).
//
// Work split as in the mma.sync kernel: one CTA per (sequence b, kv head h,
// chunk of keys), carrying all R = G * (gamma_b + 1) query rows of the group
// (padded to RP, a multiple of 16) along every 128-key tile.  Per tile:
//
//   S^T[key, row] = K_tile . Q^T     tcgen05.mma M = 128 keys, N = RP, K = 128 dims
//   softmax over keys               128 threads, one key (TMEM lane) each
//   O^T[d, row] += V_tile^T . P^T   tcgen05.mma M = 128 dims (V read MN-major), N = RP, K = 128 keys
//
// Roles (6 warps): warps 0-3 do the softmax, the O rescale and the epilogue
// (thread i owns TMEM lane i); warp 4 streams K/V tiles with TMA and patches
// the tail tile (the newest gamma_b + 1 keys come from Knew/Vnew, keys past
// them are zeroed); warp 5 owns TMEM and issues the MMAs.  S^T is double
// buffered in TMEM so the QK^T of tile t+1 runs while tile t is softmaxed.
// The running max / sum per row live in shared memory; the O accumulator is
// rescaled in TMEM only when some row's max grew.
//
// Split-KV partials and their merge are the same as in the mma.sync kernel.
#include "common.cuh"
#include "internal.h"

namespace spec {
namespace {

constexpr int D = 128;
constexpr int KT = 128;                  // keys per tile = MMA M
constexpr int ST = 2;                    // K/V stages
constexpr int KV_HALF = KT * 128;        // 128 keys x 64 dims (128 B rows), 16 KB
constexpr int KV_TILE = 2 * KV_HALF;     // 32 KB
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;      // S^T x2 (<= 64 cols each) + O^T (<= 64 cols)

template <int RP>
struct TCfg {
  // row-owner softmax: TPR threads per query row, KPT keys each
  static constexpr int TPR = RP <= 16 ? 8 : (RP <= 32 ? 4 : 2);
  static constexpr int KPT = KT / TPR;
  static constexpr int Q_HALF = RP * 128;                   // RP rows x 64 dims (or keys) of bf16
  static constexpr int OFF_K = 0;                           // ST x K tile
  static constexpr int OFF_V = ST * KV_TILE;                // ST x V tile
  static constexpr int OFF_Q = 2 * ST * KV_TILE;            // Q [RP][128 dims], two halves
  static constexpr int OFF_P = OFF_Q + 2 * Q_HALF;           // P [RP][128 keys], two halves
  static constexpr int OFF_STG = OFF_P + 2 * Q_HALF;         // scores staging [RP][128 + TPR] fp32 (skewed)
  static constexpr int STG_ROW = KT + TPR;
  static constexpr int OFF_BAR = OFF_STG + ((RP * STG_ROW * 4 + 1023) / 1024) * 1024;
  static constexpr int OFF_ROW = OFF_BAR + 256;             // m[64], l[64], alpha[64]
  static constexpr int SMEM = OFF_ROW + 3 * 64 * 4 + 1024;
};

// staging index of score (row j, key k): rows skewed by TPR words and key slices by one
// word so that both the key-major writes and the row-owner reads are bank-conflict free
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

template <int RP>
__global__ void __launch_bounds__(THREADS, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const AttnArgs a) {
  using C = TCfg<RP>;
  constexpr int TPR = C::TPR, KPT = C::KPT;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* k_full = bars;             // [ST]  K tile landed
  uint64_t* v_full = bars + 2;         // [ST]  V tile landed
  uint64_t* k_empty = bars + 4;        // [ST]  QK^T done with the K stage
  uint64_t* v_empty = bars + 6;        // [ST]  PV done with the V stage
  uint64_t* tail_ready = bars + 8;     // [ST]  tail tile (K and V) patched
  uint64_t* s_full = bars + 10;        // [2]   S^T in TMEM
  uint64_t* s_empty = bars + 12;       // [2]   softmax has read S^T
  uint64_t* p_full = bars + 14;        // P in smem and O rescaled
  uint64_t* pv_done = bars + 15;       // PV finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  float* stg = reinterpret_cast<float*>(smem + C::OFF_STG);
  float* row_m = reinterpret_cast<float*>(smem + C::OFF_ROW);
  float* row_l = row_m + 64;
  float* row_alpha = row_m + 128;

  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int ctx = a.ctx_len[b];
  const int r0 = a.cu_rows[b];
  const int Mb = a.cu_rows[b + 1] - r0;
  const int R = a.G * Mb;
  const int n_chunks = ctx > 0 ? (ctx + a.chunk - 1) / a.chunk : 1;
  if (c >= n_chunks || Mb <= 0) return;
  if (Mb > a.max_rows || ctx < 0 || ctx + Mb > a.cap || R > RP) {
    if (tid == 0) set_status(a.status, 0x2F1u);
    return;
  }
  const bool last_chunk = (c == n_chunks - 1);
  const int k_begin = c * a.chunk;
  const int k_end = last_chunk ? ctx + Mb : (c + 1) * a.chunk;
  const int nt = (k_end - k_begin + KT - 1) / KT;
  const int bh = b * a.Hkv + h;

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
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(tmem_slot, TMEM_COLS);
  if (warp < 4) {
    // Q rows of the group (row j = token row j / G, head j % G), zero-padded to RP, swizzled halves
    for (int idx = tid; idx < RP * 16; idx += 128) {
      const int j = idx >> 4, ch = idx & 15;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (j < R) {
        const int tr = j / a.G, g = j - tr * a.G;
        v = *reinterpret_cast<const uint4*>(a.Q + (size_t)(r0 + tr) * a.ldq + (size_t)(h * a.G + g) * D + ch * 8);
      }
      *reinterpret_cast<uint4*>(smem + C::OFF_Q + (ch >> 3) * C::Q_HALF + sw128_off(j, (ch & 7) * 8)) = v;
    }
    if (tid < 64) {
      row_m[tid] = -INFINITY;
      row_l[tid] = 0.f;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s0 = tmem, t_s1 = tmem + 64, t_o = tmem + 128;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer (+ tail patch)
    bool ok = true;
    for (int t = 0; t < nt && ok; ++t) {
      const int s = t % ST;
      const uint32_t ph = ((t / ST) - 1) & 1;
      const int key0 = k_begin + t * KT;
      uint8_t* kt = smem + C::OFF_K + s * KV_TILE;
      uint8_t* vt = smem + C::OFF_V + s * KV_TILE;
      if (t >= ST) ok = mbar_wait(&k_empty[s], ph, a.status, 0x211u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&k_full[s], KV_TILE);
        tma_load_3d(kt, &tmK, &k_full[s], 0, key0, bh);
        tma_load_3d(kt + KV_HALF, &tmK, &k_full[s], 64, key0, bh);
      }
      if (t >= ST) ok = mbar_wait(&v_empty[s], ph, a.status, 0x212u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&v_full[s], KV_TILE);
        tma_load_3d(vt, &tmV, &v_full[s], 0, key0, bh);
        tma_load_3d(vt + KV_HALF, &tmV, &v_full[s], 64, key0, bh);
      }
      if (key0 + KT > ctx) {
        // tail tile: wait for both loads, then overwrite keys >= ctx (new block, zeros past it)
        ok = mbar_wait(&k_full[s], (t / ST) & 1, a.status, 0x213u) &&
             mbar_wait(&v_full[s], (t / ST) & 1, a.status, 0x214u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const int rr0 = ctx > key0 ? ctx - key0 : 0;
        for (int idx = rr0 * 16 + lane; idx < KT * 16; idx += 32) {
          const int rr = idx >> 4, ch = idx & 15;
          const int p = key0 + rr;
          uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
          if (p < ctx + Mb) {
            const size_t off = (size_t)(r0 + p - ctx) * a.ldkv + (size_t)h * D + ch * 8;
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
      const uint32_t q_addr = smem_u32(smem + C::OFF_Q);
      const uint32_t p_addr = smem_u32(smem + C::OFF_P);
      int tail_phase[ST] = {0, 0};
      bool tail_seen[ST] = {false, false};
      // the tail tile's loads are complete once tail_ready fired; earlier tiles wait on the TMA barriers
      auto wait_tile = [&](int t, uint64_t* full, unsigned site) -> bool {
        const int s = t % ST;
        if (k_begin + t * KT + KT > ctx) {
          if (!tail_seen[s]) {
            tail_seen[s] = true;
            if (!mbar_wait(&tail_ready[s], tail_phase[s] & 1, a.status, site)) return false;
          }
          return true;
        }
        return mbar_wait(&full[s], (t / ST) & 1, a.status, site);
      };
      auto issue_s = [&](int t) -> bool {
        const int s = t % ST;
        if (!wait_tile(t, k_full, 0x221u)) return false;
        if (t >= 2 && !mbar_wait(&s_empty[t & 1], ((t >> 1) - 1) & 1, a.status, 0x222u)) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + C::OFF_K + s * KV_TILE);
        const uint32_t d_s = (t & 1) ? t_s1 : t_s0;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t ka = k_addr + (kk >> 2) * KV_HALF + (kk & 3) * 32;
          const uint32_t qa = q_addr + (kk >> 2) * C::Q_HALF + (kk & 3) * 32;
          umma_bf16(d_s, umma_desc_sw128(ka), umma_desc_sw128(qa), idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&k_empty[s]);
        umma_commit(&s_full[t & 1]);
        return true;
      };
      bool ok = issue_s(0);
      for (int t = 0; t < nt && ok; ++t) {
        if (t + 1 < nt && !issue_s(t + 1)) { ok = false; break; }
        const int s = t % ST;
        if (!mbar_wait(p_full, t & 1, a.status, 0x223u) || !wait_tile(t, v_full, 0x224u)) { ok = false; break; }
        tc_fence_after();
        const uint32_t v_addr = smem_u32(smem + C::OFF_V + s * KV_TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t va = v_addr + kk * 16 * 128;                     // 16 keys per step
          const uint32_t pa = p_addr + (kk >> 2) * C::Q_HALF + (kk & 3) * 32;
          umma_bf16(t_o, umma_desc_sw128_mn(va, KV_HALF), umma_desc_sw128(pa), idesc_pv,
                    (t > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&v_empty[s]);
        umma_commit(pv_done);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps
    // (a) thread = key lane: TMEM -> scaled, masked scores into the staging buffer
    // (b) thread = (row j, key slice): row max / sum, P row slice, running state
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    const int row = tid / TPR, part = tid % TPR;
    const bool owner = row < RP;
    bool ok = true;
    for (int t = 0; t < nt; ++t) {
      const int key0 = k_begin + t * KT;
      const bool tail = key0 + KT > ctx;
      ok = ok && mbar_wait(&s_full[t & 1], (t >> 1) & 1, a.status, 0x231u);
      ok = bar_compute_and(ok);
      if (!ok) break;
      tc_fence_after();
      {
        float sv[RP];
        tmem_ld_cols<RP>(((t & 1) ? t_s1 : t_s0) + lane_off, sv);
        tc_fence_before();
        mbar_arrive(&s_empty[t & 1]);
        const int p = key0 + tid;
#pragma unroll
        for (int j = 0; j < RP; ++j) {
          float v = sv[j] * a.scale_log2;
          if (tail && p > ctx + min(j / a.G, Mb - 1)) v = -INFINITY;
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
        for (int i = 0; i < KPT; ++i) {
          pv[i] = src[i];
          mx = fmaxf(mx, pv[i]);
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
        for (int i = 0; i < KPT; ++i) {
          pv[i] = exp2f(pv[i] - base);
          sm += pv[i];
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
      // PV(t-1) must be done before P is overwritten and O is rescaled
      if (t >= 1) {
        ok = mbar_wait(pv_done, (t - 1) & 1, a.status, 0x232u);
        ok = bar_compute_and(ok);
        if (!ok) break;
      }
      if (owner) {
        // keys [part*KPT, part*KPT + KPT) of row `row` as bf16, 8 keys (16 B) per store
        uint8_t* prow = smem + C::OFF_P;
#pragma unroll
        for (int i = 0; i < KPT; i += 8) {
          const int k = part * KPT + i;
          const uint4 w = make_uint4(pack_bf16x2(pv[i], pv[i + 1]), pack_bf16x2(pv[i + 2], pv[i + 3]),
                                     pack_bf16x2(pv[i + 4], pv[i + 5]), pack_bf16x2(pv[i + 6], pv[i + 7]));
          *reinterpret_cast<uint4*>(prow + (k >> 6) * C::Q_HALF + sw128_off(row, k & 63)) = w;
        }
      }
      const bool any_grew = !bar_compute_and(!grew);
      if (t >= 1 && any_grew) {
        tc_fence_after();
        const uint32_t to = t_o + lane_off;
        float orr[RP];
        tmem_ld_cols<RP>(to, orr);
#pragma unroll
        for (int cc = 0; cc < RP; cc += 16) {
          float ov[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) ov[e] = orr[cc + e] * row_alpha[cc + e];
          tmem_st16(to + cc, ov);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    // ---- epilogue: wait for the last PV, then O^T (lane = dim) / l per row
    if (ok) ok = mbar_wait(pv_done, (nt - 1) & 1, a.status, 0x233u);
    bar_compute();
    tc_fence_after();
    float ov[RP];
    const uint32_t to = t_o + lane_off;
    tmem_ld_cols<RP>(to, ov);
    const int d = tid;
    const size_t slot = (size_t)bh * a.max_chunks + c;
    float* part_buf = a.partial + slot * (64 * (D + 2));
#pragma unroll
    for (int j = 0; j < RP; ++j) {
      if (j >= R) break;
      if (n_chunks == 1) {
        const int tr = j / a.G, g = j - tr * a.G;
        a.O[(size_t)(r0 + tr) * a.ldo + (size_t)(h * a.G + g) * D + d] = f2bf(ov[j] / row_l[j]);
      } else {
        __stcg(&part_buf[j * D + d], ov[j]);
      }
    }
    if (n_chunks > 1 && tid < R) {
      __stcg(&part_buf[64 * D + tid * 2], row_m[tid]);
      __stcg(&part_buf[64 * D + tid * 2 + 1], row_l[tid]);
    }
    // the last chunk's CTA writes the new block into the cache (all its loads are done)
    if (last_chunk) {
      for (int idx = tid; idx < Mb * 16 * 2; idx += 128) {
        const int which = idx / (Mb * 16);
        const int rem = idx - which * Mb * 16;
        const int j = rem >> 4, ch = rem & 15;
        const uint16_t* src = (which ? a.Vnew : a.Knew) + (size_t)(r0 + j) * a.ldkv + (size_t)h * D + ch * 8;
        uint16_t* dst = (which ? a.Vc : a.Kc) + ((size_t)bh * a.cap + ctx + j) * D + ch * 8;
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tmem, TMEM_COLS);
  if (n_chunks == 1) return;

  // ---- split-KV: the CTA that arrives last merges the chunk partials in chunk order
  __threadfence();
  __syncthreads();
  __shared__ unsigned last_flag;
  if (tid == 0) {
    const unsigned prev = atomicAdd(&a.counters[bh], 1u);
    last_flag = (prev == (unsigned)(n_chunks - 1)) ? 1u : 0u;
  }
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  const float* base_part = a.partial + (size_t)bh * a.max_chunks * (64 * (D + 2));
  for (int idx = tid; idx < R * D; idx += THREADS) {
    const int j = idx / D, d = idx - j * D;
    float M = -INFINITY;
    for (int k = 0; k < n_chunks; ++k) M = fmaxf(M, __ldcg(&base_part[(size_t)k * 64 * (D + 2) + 64 * D + j * 2]));
    const float base = M == -INFINITY ? 0.f : M;
    float L = 0.f, O = 0.f;
    for (int k = 0; k < n_chunks; ++k) {
      const float* pk = base_part + (size_t)k * 64 * (D + 2);
      const float f = exp2f(__ldcg(&pk[64 * D + j * 2]) - base);
      L += __ldcg(&pk[64 * D + j * 2 + 1]) * f;
      O += __ldcg(&pk[j * D + d]) * f;
    }
    const int tr = j / a.G, g = j - tr * a.G;
    a.O[(size_t)(r0 + tr) * a.ldo + (size_t)(h * a.G + g) * D + d] = f2bf(O / L);
  }
  if (tid == 0) a.counters[bh] = 0u;
}

template <int RP>
cudaError_t launch_rp(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, cudaStream_t s) {
  constexpr int smem = TCfg<RP>::SMEM;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel<RP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  dim3 grid(a.max_chunks, a.Hkv, a.B);
  attention_tc_kernel<RP><<<grid, THREADS, smem, s>>>(tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

int attention_tc_key_tile() { return KT; }

cudaError_t launch_attention_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a,
                                cudaStream_t s) {
  const int rows = a.G * a.max_rows;
  if (rows <= 16) return launch_rp<16>(tk, tv, a, s);
  if (rows <= 32) return launch_rp<32>(tk, tv, a, s);
  if (rows <= 48) return launch_rp<48>(tk, tv, a, s);
  return launch_rp<64>(tk, tv, a, s);
}

}  // namespace spec
