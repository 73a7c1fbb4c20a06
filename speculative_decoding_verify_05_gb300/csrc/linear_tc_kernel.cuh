// Kernel body of the persistent tcgen05 verify GEMM (see linear_tc.cuh for the design).
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
// Named barrier 2 over the four epilogue warps.
__device__ __forceinline__ void bar_epi() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
__device__ __forceinline__ bool bar_epi_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.and.pred q, 2, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// First work unit of persistent CTA c (c = grid gives the total), and the CTA owning unit u.
__device__ __forceinline__ long long unit_begin(const LinearArgs& a, int c) {
  if (a.aligned) {
    const long long tiles = (long long)a.tiles_m * a.tiles_n;
    return (tiles * c / a.grid) * a.k_tiles;
  }
  return a.units * c / a.grid;
}
__device__ __forceinline__ int cta_of_unit(const LinearArgs& a, long long u) {
  int c = (int)(((u + 1) * a.grid - 1) / a.units);
  if (c >= a.grid) c = a.grid - 1;
  while (c + 1 < a.grid && unit_begin(a, c + 1) <= u) ++c;
  while (c > 0 && unit_begin(a, c) > u) --c;
  return c;
}

template <int BN, int NSUB, int EPI>
__global__ void __launch_bounds__(192, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const LinearArgs args) {
  using Cfg = LinearCfg<BN, NSUB>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int TN = Cfg::TN;
  constexpr int NBUF = Cfg::NBUF;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;   // [NBUF]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  float2* red = reinterpret_cast<float2*>(smem + STAGES * Cfg::STAGE_BYTES + 1024);  // [4][TN]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int kt = args.k_tiles;
  const long long ub = unit_begin(args, cta);
  const long long ue = unit_begin(args, cta + 1);

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 128);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer: one continuous stream over this CTA's units
    if (lane == 0) {
      long long i = 0;
      for (long long u = ub; u < ue; ++u, ++i) {
        const int s = (int)(i % STAGES);
        const long long r = i / STAGES;
        if (i >= STAGES && !mbar_wait(&empty[s], (uint32_t)((r - 1) & 1), args.status, 0x101u)) break;
        const long long tile = u / kt;
        const int k = (int)(u - tile * kt);
        const int m_t = (int)(tile % args.tiles_m);
        const int n_t = (int)(tile / args.tiles_m);
        mbar_arrive_expect_tx(&full[s], Cfg::STAGE_BYTES);
        tma_load_2d(sA + s * Cfg::A_BYTES, &tm_w, &full[s], k * 64, n_t * 128);
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub)
          tma_load_2d(sB + s * Cfg::B_BYTES + sub * BN * 128, &tm_x, &full[s], k * 64, m_t * TN + sub * BN);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer: one TMEM accumulator per tile segment, two in flight
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(128, BN);
      long long i = 0;
      int seg = 0;
      bool ok = true;
      for (long long u = ub; u < ue && ok; ++seg) {
        const long long tile = u / kt;
        const long long seg_end = min(ue, (tile + 1) * kt);
        const int acc = seg % NBUF;
        const int use = seg / NBUF;
        if (use >= 1 && !mbar_wait(&acc_empty[acc], (uint32_t)((use - 1) & 1), args.status, 0x102u)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * Cfg::ACC_COLS;
        for (long long uu = u; uu < seg_end; ++uu, ++i) {
          const int s = (int)(i % STAGES);
          if (!mbar_wait(&full[s], (uint32_t)((i / STAGES) & 1), args.status, 0x103u)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a = smem_u32(sA + s * Cfg::A_BYTES);
          const uint32_t b = smem_u32(sB + s * Cfg::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int sub = 0; sub < NSUB; ++sub)
              umma_bf16(d + sub * BN, umma_desc_sw128(a + kk * 32), umma_desc_sw128(b + sub * BN * 128 + kk * 32),
                        idesc, (uu > u || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&acc_full[acc]);
        u = seg_end;
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps 2..5 drain TMEM lane quarter (warp % 4)
    const int q = warp & 3;
    const int row = q * 32 + lane;            // TMEM lane = weight row within the tile
    const int etid = threadIdx.x - 64;        // 0..127 among the epilogue threads
    const int ewarp = etid >> 5;
    int seg = 0;
    bool ok = true;
    for (long long u = ub; u < ue; ++seg) {
      const long long tile = u / kt;
      const long long seg_end = min(ue, (tile + 1) * kt);
      const bool whole = (u == tile * kt) && (seg_end == (tile + 1) * kt);
      const int acc = seg % NBUF;
      const int m0 = (int)(tile % args.tiles_m) * TN;
      const int n_t = (int)(tile / args.tiles_m);
      const int n0 = n_t * 128;
      const int n = n0 + row;
      ok = ok && mbar_wait(&acc_full[acc], (uint32_t)((seg / NBUF) & 1), args.status, 0x104u);
      ok = bar_epi_and(ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_row = tmem + acc * Cfg::ACC_COLS + (uint32_t(q * 32) << 16);

      if constexpr (EPI == EPI_BF16) {
        if (whole) {
#pragma unroll 1
          for (int c = 0; c < TN; c += 16) {
            float v[16];
            tmem_ld16(t_row + c, v);
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
          tc_fence_before();
          mbar_arrive(&acc_empty[acc]);
        } else {
          // split tile: publish this CTA's fp32 piece (slot 0 = its first segment, 1 = its last);
          // the reduce kernel that follows the GEMM sums the pieces
          const int slot = (u == ub) ? 0 : 1;
          float* part = args.partial + ((size_t)cta * 2 + slot) * (TN * 128);
#pragma unroll 1
          for (int c = 0; c < TN; c += 16) {
            float v[16];
            tmem_ld16(t_row + c, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) __stcg(&part[(c + j) * 128 + row], v[j]);
          }
          tc_fence_before();
          mbar_arrive(&acc_empty[acc]);
        }
      } else {
        // LM-head epilogues (ranges are tile-aligned, so every segment is whole):
        // per token column j reduce over the tile's 128 vocabulary rows
#pragma unroll 1
        for (int c = 0; c < TN; c += 16) {
          float v[16];
          tmem_ld16(t_row + c, v);
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
              if (lane == 0) red[ewarp * TN + c + j] = make_float2(mx, sm);
            } else {
              float zv = valid ? v[j] : -INFINITY;
              int idx = valid ? n : 0x7fffffff;
              warp_argmax(zv, idx);
              if (lane == 0) red[ewarp * TN + c + j] = make_float2(zv, __int_as_float(idx));
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[acc]);
        bar_epi();
        for (int j = etid; j < TN; j += 128) {
          const int m = m0 + j;
          if (m >= args.M) continue;
          float2 accv = red[j];
          for (int w = 1; w < 4; ++w) {
            const float2 o = red[w * TN + j];
            if constexpr (EPI == EPI_LOGITS) {
              const float mx = fmaxf(accv.x, o.x);
              const float s = (accv.x == -INFINITY ? 0.f : accv.y * expf(accv.x - mx)) +
                              (o.x == -INFINITY ? 0.f : o.y * expf(o.x - mx));
              accv = make_float2(mx, s);
            } else {
              const int ai = __float_as_int(accv.y), oi = __float_as_int(o.y);
              if (o.x > accv.x || (o.x == accv.x && oi < ai)) accv = o;
            }
          }
          args.stats[(size_t)m * args.tiles_n + n_t] = accv;
        }
        bar_epi();   // red is reused by the next tile
      }
      u = seg_end;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

}  // namespace spec
