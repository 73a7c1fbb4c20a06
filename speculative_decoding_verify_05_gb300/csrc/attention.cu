// Verify attention: gamma_b + 1 causal query rows per sequence attend the
// bf16 KV cache plus their own new block, grouped-query (G query heads share
// one kv head).
//
// One CTA = (sequence b, kv head h, chunk of keys).  All G * (gamma_b + 1)
// query rows of the (b, h) group ride along every K/V tile, so each cache byte
// is read from HBM once for all of them.  K/V tiles of 64 keys x 128 dims are
// streamed by TMA (3D tensor map over [B*Hkv][cap][128], 128-byte swizzle,
// rows past `cap` zero-filled) through a 3-stage ring; QK^T and PV run on
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) with an online softmax kept in
// registers.  The newest gamma_b + 1 keys are taken from Knew/Vnew (and
// written into the cache by the CTA that owns the last chunk once its loads
// are done), so no CTA reads a cache slot that another CTA writes.
//
// Long contexts are split over several CTAs (flash-decoding style); each
// writes an unnormalised partial (O, running max, running sum) and the CTA
// that arrives last on the (b, h) counter merges them in chunk order.
#include "common.cuh"
#include "internal.h"

namespace spec {
namespace {

constexpr int D = 128;
constexpr int KT = 64;                 // keys per tile
constexpr int STAGES = 3;
constexpr int HALF_BYTES = KT * 64 * 2; // 64 keys x 64 dims, 8 KB
constexpr int TILE_BYTES = 2 * HALF_BYTES;
constexpr int Q_BYTES = 64 * D * 2;     // up to 64 query rows
constexpr int SMEM_BYTES = Q_BYTES + STAGES * 2 * TILE_BYTES + 256 + 1024;

// element (row, col) of a [rows][128] tile stored as two 64-column swizzled halves
__device__ __forceinline__ uint32_t tile_off(int row, int col) {
  return uint32_t(col >> 6) * HALF_BYTES + sw128_off(row, col & 63);
}

__device__ __forceinline__ float fast_exp2(float x) { return exp2f(x); }

template <int RTP>
__global__ void __launch_bounds__(128)
attention_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const AttnArgs a) {
  pdl_wait();
  pdl_trigger();
  constexpr int WK = 4 / RTP;         // warps sharing one 16-row m-tile
  constexpr int KPW = KT / WK;        // keys of each tile handled by one warp
  constexpr int NT = KPW / 8;         // 8-key n-tiles per warp per tile

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + Q_BYTES;                 // [stage][K | V] tiles
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Q_BYTES + STAGES * 2 * TILE_BYTES);

  const int c = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int ctx = a.ctx_len[b];
  const int r0 = a.cu_rows[b];
  const int Mb = a.cu_rows[b + 1] - r0;
  const int R = a.G * Mb;
  const int n_chunks = ctx > 0 ? (ctx + a.chunk - 1) / a.chunk : 1;
  if (c >= n_chunks || Mb <= 0) return;
  if (Mb > a.max_rows || ctx < 0 || ctx + Mb > a.cap) {
    // device-side check of the caller's row/context arrays: nothing is read or written
    if (threadIdx.x == 0) set_status(a.status, 0x2F0u);
    return;
  }
  const bool last_chunk = (c == n_chunks - 1);
  const int k_begin = c * a.chunk;
  const int k_end = last_chunk ? ctx + Mb : (c + 1) * a.chunk;
  const int nt = (k_end - k_begin + KT - 1) / KT;
  const int bh = b * a.Hkv + h;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int t = 0; t < nt && t < STAGES; ++t) {
      uint8_t* kd = sKV + t * 2 * TILE_BYTES;
      mbar_arrive_expect_tx(&full[t], 2 * TILE_BYTES);
      const int key = k_begin + t * KT;
      tma_load_3d(kd, &tmK, &full[t], 0, key, bh);
      tma_load_3d(kd + HALF_BYTES, &tmK, &full[t], 64, key, bh);
      tma_load_3d(kd + TILE_BYTES, &tmV, &full[t], 0, key, bh);
      tma_load_3d(kd + TILE_BYTES + HALF_BYTES, &tmV, &full[t], 64, key, bh);
    }
  }
  // Q rows of this group: row r = j * G + g  (token row j, head g within the group)
  for (int idx = threadIdx.x; idx < 64 * 16; idx += 128) {
    const int r = idx >> 4, ch = idx & 15;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < R) {
      const int j = r / a.G, g = r - j * a.G;
      v = *reinterpret_cast<const uint4*>(a.Q + (size_t)(r0 + j) * a.ldq + (size_t)(h * a.G + g) * D + ch * 8);
    }
    *reinterpret_cast<uint4*>(sQ + tile_off(r, ch * 8)) = v;
  }
  __syncthreads();

  const int mt = warp % RTP;            // m-tile of this warp
  const int kpart = warp / RTP;         // key slice of this warp
  const int RT = (R + 15) >> 4;
  const bool active = mt < RT;

  // Q fragments (16 rows x 128 dims) kept in registers
  uint32_t qf[8][4];
  if (active) {
    const uint32_t qbase = smem_u32(sQ);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int row = mt * 16 + (lane & 15);
      const int col = ks * 16 + (lane >> 4) * 8;
      ldsm_x4(qbase + tile_off(row, col), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }
  }
  // causal limit per owned row: visible keys p <= ctx + j
  const int rowA = mt * 16 + (lane >> 2);
  const int rowB = rowA + 8;
  const int jA = min(rowA / a.G, Mb - 1);
  const int jB = min(rowB / a.G, Mb - 1);
  const int limA = ctx + jA;
  const int limB = ctx + jB;

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

  bool ok = true;
  for (int t = 0; t < nt; ++t) {
    const int s = t % STAGES;
    uint8_t* sK = sKV + s * 2 * TILE_BYTES;
    uint8_t* sV = sK + TILE_BYTES;
    const int tile_start = k_begin + t * KT;
    ok = ok && mbar_wait(&full[s], (t / STAGES) & 1, a.status, 0x201u);
    ok = __syncthreads_and(ok);
    if (!ok) break;
    const bool tail = tile_start + KT > ctx;   // holds new keys or keys past the end
    if (tail) {
      // replace rows >= ctx with the new block (or zeros past it)
      for (int idx = threadIdx.x; idx < KT * 16 * 2; idx += 128) {
        const int which = idx / (KT * 16);
        const int rr = (idx >> 4) & (KT - 1), ch = idx & 15;
        const int p = tile_start + rr;
        if (p < ctx) continue;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (p < ctx + Mb) {
          const uint16_t* src = (which ? a.Vnew : a.Knew) + (size_t)(r0 + p - ctx) * a.ldkv + (size_t)h * D + ch * 8;
          v = *reinterpret_cast<const uint4*>(src);
        }
        *reinterpret_cast<uint4*>((which ? sV : sK) + tile_off(rr, ch * 8)) = v;
      }
      __syncthreads();
    }
    if (active) {
      float sc[NT][4];
#pragma unroll
      for (int i = 0; i < NT; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
      const uint32_t kbase = smem_u32(sK);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          const int key = kpart * KPW + np * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int col = ks * 16 + ((lane >> 3) & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + tile_off(key, col), b0, b1, b2, b3);
          mma_bf16_16816(sc[2 * np], qf[ks], b0, b1);
          mma_bf16_16816(sc[2 * np + 1], qf[ks], b2, b3);
        }
      }
      // scale, mask, online softmax
      float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int p = tile_start + kpart * KPW + i * 8 + (lane & 3) * 2 + e;
          float va = sc[i][e] * a.scale_log2;
          float vb = sc[i][2 + e] * a.scale_log2;
          if (tail) {
            if (p > limA) va = -INFINITY;
            if (p > limB) vb = -INFINITY;
          }
          sc[i][e] = va;
          sc[i][2 + e] = vb;
          mxA = fmaxf(mxA, va);
          mxB = fmaxf(mxB, vb);
        }
      }
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
      const float nmA = fmaxf(mA, mxA), nmB = fmaxf(mB, mxB);
      const float baseA = nmA == -INFINITY ? 0.f : nmA;
      const float baseB = nmB == -INFINITY ? 0.f : nmB;
      const float alA = fast_exp2(mA - baseA), alB = fast_exp2(mB - baseB);
      mA = nmA;
      mB = nmB;
      float sA = 0.f, sB = 0.f;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        sc[i][0] = fast_exp2(sc[i][0] - baseA);
        sc[i][1] = fast_exp2(sc[i][1] - baseA);
        sc[i][2] = fast_exp2(sc[i][2] - baseB);
        sc[i][3] = fast_exp2(sc[i][3] - baseB);
        sA += sc[i][0] + sc[i][1];
        sB += sc[i][2] + sc[i][3];
      }
      sA += __shfl_xor_sync(0xffffffffu, sA, 1);
      sA += __shfl_xor_sync(0xffffffffu, sA, 2);
      sB += __shfl_xor_sync(0xffffffffu, sB, 1);
      sB += __shfl_xor_sync(0xffffffffu, sB, 2);
      lA = lA * alA + sA;
      lB = lB * alB + sB;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= alA; o[i][1] *= alA;
        o[i][2] *= alB; o[i][3] *= alB;
      }
      // O += P V
      const uint32_t vbase = smem_u32(sV);
#pragma unroll
      for (int kk = 0; kk < KPW / 16; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_bf16x2(sc[2 * kk][0], sc[2 * kk][1]);
        pa[1] = pack_bf16x2(sc[2 * kk][2], sc[2 * kk][3]);
        pa[2] = pack_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        pa[3] = pack_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
        for (int dn = 0; dn < 8; ++dn) {
          const int key = kpart * KPW + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int col = dn * 16 + (lane >> 4) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vbase + tile_off(key, col), b0, b1, b2, b3);
          mma_bf16_16816(o[2 * dn], pa, b0, b1);
          mma_bf16_16816(o[2 * dn + 1], pa, b2, b3);
        }
      }
    }
    // release the stage: order generic smem accesses before the next TMA write
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0 && t + STAGES < nt) {
      mbar_arrive_expect_tx(&full[s], 2 * TILE_BYTES);
      const int key = k_begin + (t + STAGES) * KT;
      tma_load_3d(sK, &tmK, &full[s], 0, key, bh);
      tma_load_3d(sK + HALF_BYTES, &tmK, &full[s], 64, key, bh);
      tma_load_3d(sV, &tmV, &full[s], 0, key, bh);
      tma_load_3d(sV + HALF_BYTES, &tmV, &full[s], 64, key, bh);
    }
  }

  // ---- merge the warps of each m-tile through shared memory (stage buffers are free now)
  float* so = reinterpret_cast<float*>(sKV);            // [4 warps][16 rows][128]
  float* sml = so + 4 * 16 * D;                         // [4 warps][16 rows][2]
  if (active) {
    const int ra = lane >> 2;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int col = i * 8 + (lane & 3) * 2;
      so[(warp * 16 + ra) * D + col] = o[i][0];
      so[(warp * 16 + ra) * D + col + 1] = o[i][1];
      so[(warp * 16 + ra + 8) * D + col] = o[i][2];
      so[(warp * 16 + ra + 8) * D + col + 1] = o[i][3];
    }
    if ((lane & 3) == 0) {
      sml[(warp * 16 + ra) * 2] = mA;
      sml[(warp * 16 + ra) * 2 + 1] = lA;
      sml[(warp * 16 + ra + 8) * 2] = mB;
      sml[(warp * 16 + ra + 8) * 2 + 1] = lB;
    }
  }
  __syncthreads();

  const size_t slot = (size_t)bh * a.max_chunks + c;
  float* part = a.partial + slot * (64 * (D + 2));
  for (int idx = threadIdx.x; idx < R * D; idx += 128) {
    const int r = idx / D, d = idx - r * D;
    const int m_t = r >> 4, rr = r & 15;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < WK; ++k) M = fmaxf(M, sml[((k * RTP + m_t) * 16 + rr) * 2]);
    const float base = M == -INFINITY ? 0.f : M;
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int k = 0; k < WK; ++k) {
      const int w = k * RTP + m_t;
      const float f = fast_exp2(sml[(w * 16 + rr) * 2] - base);
      L += sml[(w * 16 + rr) * 2 + 1] * f;
      O += so[(w * 16 + rr) * D + d] * f;
    }
    if (n_chunks == 1) {
      const int j = r / a.G, g = r - j * a.G;
      a.O[(size_t)(r0 + j) * a.ldo + (size_t)(h * a.G + g) * D + d] = f2bf(O / L);
    } else {
      __stcg(&part[r * D + d], O);
      if (d == 0) {
        __stcg(&part[64 * D + r * 2], M);
        __stcg(&part[64 * D + r * 2 + 1], L);
      }
    }
  }

  // the last chunk's CTA writes the new block into the cache (all its TMA loads are done)
  if (last_chunk) {
    for (int idx = threadIdx.x; idx < Mb * 16 * 2; idx += 128) {
      const int which = idx / (Mb * 16);
      const int rem = idx - which * Mb * 16;
      const int j = rem >> 4, ch = rem & 15;
      const uint16_t* src = (which ? a.Vnew : a.Knew) + (size_t)(r0 + j) * a.ldkv + (size_t)h * D + ch * 8;
      uint16_t* dst = (which ? a.Vc : a.Kc) + ((size_t)bh * a.cap + ctx + j) * D + ch * 8;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    }
  }

  if (n_chunks == 1) return;
  __threadfence();
  __syncthreads();
  __shared__ unsigned last_flag;
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&a.counters[bh], 1u);
    last_flag = (prev == (unsigned)(n_chunks - 1)) ? 1u : 0u;
  }
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  const float* base_part = a.partial + (size_t)bh * a.max_chunks * (64 * (D + 2));
  for (int idx = threadIdx.x; idx < R * D; idx += 128) {
    const int r = idx / D, d = idx - r * D;
    float M = -INFINITY;
    for (int k = 0; k < n_chunks; ++k) M = fmaxf(M, __ldcg(&base_part[(size_t)k * 64 * (D + 2) + 64 * D + r * 2]));
    const float base = M == -INFINITY ? 0.f : M;
    float L = 0.f, O = 0.f;
    for (int k = 0; k < n_chunks; ++k) {
      const float* pk = base_part + (size_t)k * 64 * (D + 2);
      const float f = fast_exp2(__ldcg(&pk[64 * D + r * 2]) - base);
      L += __ldcg(&pk[64 * D + r * 2 + 1]) * f;
      O += __ldcg(&pk[r * D + d]) * f;
    }
    const int j = r / a.G, g = r - j * a.G;
    a.O[(size_t)(r0 + j) * a.ldo + (size_t)(h * a.G + g) * D + d] = f2bf(O / L);
  }
  if (threadIdx.x == 0) a.counters[bh] = 0u;
}

template <int RTP>
cudaError_t launch_rtp(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a,
                       cudaStream_t s) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attention_kernel<RTP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  dim3 grid(a.max_chunks, a.Hkv, a.B);
  cudaError_t e = launch_k(attention_kernel<RTP>, grid, dim3(128), SMEM_BYTES, s, tk, tv, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a,
                             cudaStream_t s) {
  const int rows = a.G * a.max_rows;
  if (rows <= 16) return launch_rtp<1>(tk, tv, a, s);
  if (rows <= 32) return launch_rtp<2>(tk, tv, a, s);
  return launch_rtp<4>(tk, tv, a, s);
}

}  // namespace spec
