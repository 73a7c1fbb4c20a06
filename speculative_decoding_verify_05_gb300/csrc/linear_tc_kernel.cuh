// Kernel body of the tcgen05 verify GEMM (see linear_tc.cuh for the design).
#pragma once

#include "linear_tc.cuh"

namespace spec {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// (value, index) max with the lowest index winning ties.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
}

template <int BN, int EPI>
__global__ void __launch_bounds__(128, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const LinearArgs args) {
  using Cfg = LinearCfg<BN>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* done = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  float2* red = reinterpret_cast<float2*>(smem + STAGES * Cfg::STAGE_BYTES + 1024);  // [4][BN]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x;
  const int n_tile = blockIdx.y;
  const int split = blockIdx.z;
  const int m0 = m_tile * BN;
  const int n0 = n_tile * 128;
  const int kb = (int)(((long long)split * args.k_tiles) / args.splits);
  const int ke = (int)(((long long)(split + 1) * args.k_tiles) / args.splits);
  const int nk = ke - kb;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_d = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    for (int i = 0; i < nk; ++i) {
      const int s = i % STAGES;
      const int r = i / STAGES;
      if (i >= STAGES && !mbar_wait(&empty[s], (r - 1) & 1, args.status, 0x101u)) break;
      mbar_arrive_expect_tx(&full[s], Cfg::STAGE_BYTES);
      tma_load_2d(sA + s * Cfg::A_BYTES, &tm_w, &full[s], (kb + i) * 64, n0);
      tma_load_2d(sB + s * Cfg::B_BYTES, &tm_x, &full[s], (kb + i) * 64, m0);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc = umma_idesc_bf16(128, BN);
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      const int s = i % STAGES;
      const int r = i / STAGES;
      if (!mbar_wait(&full[s], r & 1, args.status, 0x102u)) { ok = false; break; }
      tc_fence_after();
      const uint32_t a = smem_u32(sA + s * Cfg::A_BYTES);
      const uint32_t b = smem_u32(sB + s * Cfg::B_BYTES);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_bf16(tmem_d, umma_desc_sw128(a + kk * 32), umma_desc_sw128(b + kk * 32), idesc,
                  (i > 0 || kk > 0) ? 1u : 0u);
      umma_commit(&empty[s]);
    }
    if (ok) umma_commit(done);
  }
  __syncwarp();

  // ---------------- epilogue: TMEM -> registers -> global
  bool have = (nk > 0) && mbar_wait(done, 0, args.status, 0x103u);
  have = __all_sync(0xffffffffu, have);
  tc_fence_after();

  const int row = warp * 32 + lane;          // TMEM lane = weight row within the tile
  const int n = n0 + row;
  const uint32_t t_row = tmem_d + (uint32_t(warp * 32) << 16);

  if constexpr (EPI == EPI_BF16) {
    if (args.splits == 1) {
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        float v[16];
        if (have) tmem_ld16(t_row + c, v);
        else {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = m0 + c + j;
          if (m < args.M && n < args.N) {
            float y = v[j];
            if (args.residual) y += bf16f(args.residual[(size_t)m * args.ldr + n]);
            args.Y[(size_t)m * args.ldy + n] = f2bf(y);
          }
        }
      }
    } else {
      const int tile = n_tile * args.tiles_m + m_tile;
      float* part = args.partial + ((size_t)tile * args.splits + split) * (BN * 128);
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        float v[16];
        if (have) tmem_ld16(t_row + c, v);
        else {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) __stcg(&part[(c + j) * 128 + row], v[j]);
      }
      __threadfence();
      __syncthreads();
      __shared__ unsigned last_flag;
      if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(&args.counters[tile], 1u);
        last_flag = (prev == (unsigned)(args.splits - 1)) ? 1u : 0u;
      }
      __syncthreads();
      if (last_flag) {
        // this CTA arrived last: sum the split partials in split order (deterministic),
        // one warp per token column, 4 weight rows per lane, 16-byte loads
        __threadfence();
        const float* base = args.partial + (size_t)tile * args.splits * (BN * 128);
        const int r4 = lane * 4;
        const int n4 = n0 + r4;
#pragma unroll 2
        for (int j = warp; j < BN; j += 4) {
          const int m = m0 + j;
          if (m >= args.M) break;
          float4 acc = __ldcg(reinterpret_cast<const float4*>(base + j * 128 + r4));
          for (int s = 1; s < args.splits; ++s) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(base + (size_t)s * (BN * 128) + j * 128 + r4));
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
          }
          float y[4] = {acc.x, acc.y, acc.z, acc.w};
          if (n4 + 3 < args.N) {
            if (args.residual) {
              const uint2 rr = *reinterpret_cast<const uint2*>(args.residual + (size_t)m * args.ldr + n4);
              y[0] += bf16lo(rr.x); y[1] += bf16hi(rr.x); y[2] += bf16lo(rr.y); y[3] += bf16hi(rr.y);
            }
            *reinterpret_cast<uint2*>(args.Y + (size_t)m * args.ldy + n4) =
                make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
          } else {
            for (int e = 0; e < 4; ++e) {
              if (n4 + e >= args.N) break;
              float v = y[e];
              if (args.residual) v += bf16f(args.residual[(size_t)m * args.ldr + n4 + e]);
              args.Y[(size_t)m * args.ldy + n4 + e] = f2bf(v);
            }
          }
        }
        if (threadIdx.x == 0) args.counters[tile] = 0u;
      }
    }
  } else {
    // LM head epilogues: one split only; per token column j reduce over the 128 rows.
#pragma unroll 1
    for (int c = 0; c < BN; c += 16) {
      float v[16];
      if (have) tmem_ld16(t_row + c, v);
      else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int m = m0 + c + j;
        const bool valid = (n < args.N);
        if constexpr (EPI == EPI_LOGITS) {
          const float z = v[j] * args.inv_temp;
          if (m < args.M && valid) args.P[(size_t)m * args.N + n] = z;
          const float zm = valid ? z : -INFINITY;
          const float mx = warp_max(zm);
          const float e = valid ? expf(z - mx) : 0.f;
          const float sm = warp_sum(e);
          if (lane == 0) red[warp * BN + c + j] = make_float2(mx, sm);
        } else {
          float zv = valid ? v[j] : -INFINITY;
          int idx = valid ? n : 0x7fffffff;
          warp_argmax(zv, idx);
          if (lane == 0) red[warp * BN + c + j] = make_float2(zv, __int_as_float(idx));
        }
      }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < BN; j += blockDim.x) {
      const int m = m0 + j;
      if (m >= args.M) continue;
      float2 acc = red[j];
      for (int w = 1; w < 4; ++w) {
        const float2 o = red[w * BN + j];
        if constexpr (EPI == EPI_LOGITS) {
          const float mx = fmaxf(acc.x, o.x);
          const float s = (acc.x == -INFINITY ? 0.f : acc.y * expf(acc.x - mx)) +
                          (o.x == -INFINITY ? 0.f : o.y * expf(o.x - mx));
          acc = make_float2(mx, s);
        } else {
          const int ai = __float_as_int(acc.y), oi = __float_as_int(o.y);
          if (o.x > acc.x || (o.x == acc.x && oi < ai)) acc = o;
        }
      }
      args.stats[(size_t)m * args.n_tiles + n_tile] = acc;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_d, Cfg::TMEM_COLS);
}

}  // namespace spec
