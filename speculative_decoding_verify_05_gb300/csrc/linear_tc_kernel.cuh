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
// Named barrier 2 over the eight epilogue warps.
__device__ __forceinline__ void bar_epi() { asm volatile("bar.sync 2, 256;" ::: "memory"); }
__device__ __forceinline__ bool bar_epi_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.and.pred q, 2, 256, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Work of persistent CTA c: its data-parallel tiles c, c + grid, ... below dp_tiles, then its
// share [sk_begin, sk_end) of the stream-K units (unit u is k-step u % kt of tile dp_tiles + u / kt).
// Tile t covers token tile t % tiles_m and weight tile t / tiles_m.
struct CtaWork {
  int n_dp;
  long long sk_begin, sk_end;
  long long n;          // units in all
};
__device__ __forceinline__ long long sk_start(const LinearArgs& a, int c) { return a.sk_units * c / a.grid; }
__device__ __forceinline__ CtaWork cta_work(const LinearArgs& a, int c) {
  CtaWork w;
  w.n_dp = c < a.dp_tiles ? (int)((a.dp_tiles - 1 - c) / a.grid + 1) : 0;
  w.sk_begin = sk_start(a, c);
  w.sk_end = sk_start(a, c + 1);
  w.n = (long long)w.n_dp * a.k_tiles + (w.sk_end - w.sk_begin);
  return w;
}
// Unit i of a CTA's list: its tile and k-step, the end of the run of units that stay in that tile
// (a segment), whether the segment covers the tile's whole k-range, and whether it opens the CTA's
// stream-K range (its piece then goes to partial slot 0, else slot 1).
struct Seg {
  long long tile, end;
  int k;
  bool whole, first_sk;
};
__device__ __forceinline__ Seg seg_at(const LinearArgs& a, const CtaWork& w, int c, long long i) {
  const int kt = a.k_tiles;
  const long long ndp = (long long)w.n_dp * kt;
  Seg g;
  if (i < ndp) {
    const long long j = i / kt;
    g.tile = c + j * a.grid;
    g.k = (int)(i - j * kt);
    g.end = (j + 1) * kt;
    g.whole = true;
    g.first_sk = false;
  } else {
    const long long u = w.sk_begin + (i - ndp), t = u / kt;
    g.tile = a.dp_tiles + t;
    g.k = (int)(u - t * kt);
    const long long end_u = min(w.sk_end, (t + 1) * kt);
    g.end = ndp + (end_u - w.sk_begin);
    g.whole = g.k == 0 && end_u == (t + 1) * kt;
    g.first_sk = u == w.sk_begin;
  }
  return g;
}

// PAIR: launched in clusters of 2 CTAs; the pair's even CTA issues 2-SM MMAs of 256 weight rows
// (128 in each CTA's TMEM) over the token rows, each CTA loading its own 128 weight rows and half of
// every MMA's token rows with completion counted on the even CTA's barriers; the MMA completions
// are committed to both CTAs' barriers, and both CTAs' epilogues release the accumulator to the
// even CTA.  Every CTA of a pair walks the same work list.
template <int BN, int NSUB, int EPI, bool PAIR = false>
__global__ void __launch_bounds__(320, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const LinearArgs args) {
  using Cfg = LinearCfg<BN, NSUB, PAIR, EPI == EPI_LOGITS || EPI == EPI_ARGMAX>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int TN = Cfg::TN;
  constexpr int HB = Cfg::HB;
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
  float* ebuf_all = reinterpret_cast<float*>(smem + STAGES * Cfg::STAGE_BYTES + 1024 + 4 * TN * 8);
  float* s_rms = reinterpret_cast<float*>(smem + Cfg::RMS_OFF);   // [TN]: folded-RMSNorm row scales

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;                       // partial-sum slots are per CTA
  const int wg = PAIR ? cta >> 1 : cta;             // work group: the CTA or its pair
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int half = (int)(rank & 1u);                // which 128 rows of a pair tile
  const uint32_t leader = rank & ~1u;
  const CtaWork work = cta_work(args, wg);
  // 128-row weight tile of work tile t (token tile t % tiles_m)
  auto n_tile = [&](long long t) { return PAIR ? (int)(t / args.tiles_m) * 2 + half : (int)(t / args.tiles_m); };

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      // (a pair: one arrival from each CTA's epilogue, on the even CTA's barrier)
      mbar_init(&acc_empty[i], PAIR ? 2 : 32 * Cfg::EPI_WARPS);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
    else tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  // a pair's loads complete on, and its MMAs commit to, barriers of both CTAs: all initialised first
  if constexpr (PAIR) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // shared-memory and TMEM setup above overlaps the previous kernel; global memory only below
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    // ---------------- TMA producer: one continuous stream over this CTA's units
    if (lane == 0) {
      const uint32_t full_leader = PAIR ? dsmem_map(smem_u32(full), leader) : 0u;
      for (long long i = 0; i < work.n; ++i) {
        const int s = (int)(i % STAGES);
        const long long r = i / STAGES;
        if (i >= STAGES && !mbar_wait(&empty[s], (uint32_t)((r - 1) & 1), args.status, 0x101u)) break;
        const Seg g = seg_at(args, work, wg, i);
        const int k = g.k;
        const int m_t = (int)(g.tile % args.tiles_m);
        const int n_t = n_tile(g.tile);
        if constexpr (PAIR) {
          // both CTAs' bytes count on the even CTA's barrier (which may see them before its own
          // expect: the transaction count goes negative for a while)
          if (half == 0) mbar_arrive_expect_tx(&full[s], 2 * Cfg::STAGE_BYTES);
          const uint32_t bar = full_leader + (uint32_t)s * 8u;
          tma_load_2d_pair_hint(sA + s * Cfg::A_BYTES, &tm_w, bar, k * LIN_BK, n_t * 128, l2_policy_evict_first());
#pragma unroll
          for (int sub = 0; sub < NSUB; ++sub)
            tma_load_2d_pair(sB + s * Cfg::B_BYTES + sub * HB * LIN_ROW_BYTES, &tm_x, bar, k * LIN_BK,
                             m_t * TN + sub * BN + half * HB);
        } else {
          mbar_arrive_expect_tx(&full[s], Cfg::STAGE_BYTES);
          tma_load_2d_hint(sA + s * Cfg::A_BYTES, &tm_w, &full[s], k * LIN_BK, n_t * 128, l2_policy_evict_first());
#pragma unroll
          for (int sub = 0; sub < NSUB; ++sub)
            tma_load_2d(sB + s * Cfg::B_BYTES + sub * BN * LIN_ROW_BYTES, &tm_x, &full[s], k * LIN_BK,
                        m_t * TN + sub * BN);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (a pair's even CTA): one TMEM accumulator per tile segment, two in
    // flight when they fit
    if (lane == 0 && (!PAIR || half == 0)) {
      constexpr uint32_t idesc = umma_idesc_bf16(PAIR ? 256 : 128, BN);
      const uint32_t peer_empty = PAIR ? dsmem_map(smem_u32(empty), rank ^ 1u) : 0u;
      const uint32_t peer_acc_full = PAIR ? dsmem_map(smem_u32(acc_full), rank ^ 1u) : 0u;
      long long i = 0;
      int seg = 0;
      bool ok = true;
      for (long long u = 0; u < work.n && ok; ++seg) {
        const long long seg_end = seg_at(args, work, wg, u).end;
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
          for (int kk = 0; kk < LIN_BK / 16; ++kk)
#pragma unroll
            for (int sub = 0; sub < NSUB; ++sub) {
              const uint64_t da = umma_desc_lin(a + kk * 32);
              const uint64_t db = umma_desc_lin(b + sub * HB * LIN_ROW_BYTES + kk * 32);
              const uint32_t accum = (uu > u || kk > 0) ? 1u : 0u;
              if constexpr (PAIR) umma_bf16_pair(d + sub * BN, da, db, idesc, accum);
              else umma_bf16(d + sub * BN, da, db, idesc, accum);
            }
          if constexpr (PAIR) {
            umma_commit_pair(smem_u32(&empty[s]));
            umma_commit_pair(peer_empty + (uint32_t)s * 8u);
          } else {
            umma_commit(&empty[s]);
          }
        }
        if (!ok) break;
        if constexpr (PAIR) {
          umma_commit_pair(smem_u32(&acc_full[acc]));
          umma_commit_pair(peer_acc_full + (uint32_t)acc * 8u);
        } else {
          umma_commit(&acc_full[acc]);
        }
        u = seg_end;
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps 2..9: TMEM lane quarter warp % 4, column half (warp - 2) / 4
    const int q = warp & 3;
    const int row = q * 32 + lane;            // TMEM lane = weight row within the tile
    const int etid = threadIdx.x - 64;        // 0..255 among the epilogue threads
    const int ewarp = etid >> 5;
    const int nb = TN / 16, per_half = (nb + 1) / 2;
    const int c_begin = ((warp - 2) >> 2) * per_half * 16;
    const int c_end = min(TN, c_begin + per_half * 16);
    int seg = 0;
    bool ok = true;
    int rms_m0 = -1;       // token tile whose folded-RMSNorm scales s_rms holds
    // hand accumulator `acc` back to the MMA issuer (a pair's: once both CTAs are done with it)
    auto release_acc = [&](int acc) {
      tc_fence_before();
      if constexpr (PAIR) {
        bar_epi();
        if (etid == 0) {
          if (half == 0) mbar_arrive(&acc_empty[acc]);
          else mbar_arrive_cluster(dsmem_map(smem_u32(&acc_empty[acc]), leader));
        }
      } else {
        mbar_arrive(&acc_empty[acc]);
      }
    };
    for (long long u = 0; u < work.n; ++seg) {
      const Seg g = seg_at(args, work, wg, u);
      const long long tile = g.tile;
      const long long seg_end = g.end;
      const bool whole = g.whole;
      const int acc = seg % NBUF;
      const int m0 = (int)(tile % args.tiles_m) * TN;
      const int n_t = n_tile(tile);
      const bool live = n_t < args.tiles_n;   // (the odd half of a pair's last tile may lie past N)
      const int n0 = n_t * 128;
      const int n = n0 + row;
      // folded RMSNorm of X: the scale of every token row of this tile, before waiting for its
      // accumulator (so the first tile's overlaps the main loop); recomputed only when the token
      // tile changes (one token tile up to 384 rows)
      if (args.norm_ssq && m0 != rms_m0) {
        fill_row_scales(args, s_rms, m0, TN, etid, 32 * Cfg::EPI_WARPS);
        bar_epi();
        rms_m0 = m0;
      }
      ok = ok && mbar_wait(&acc_full[acc], (uint32_t)((seg / NBUF) & 1), args.status, 0x104u);
      ok = bar_epi_and(ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_row = tmem + acc * Cfg::ACC_COLS + (uint32_t(q * 32) << 16);

      if constexpr (EPI == EPI_BF16 || EPI == EPI_SWIGLU) {
        // 16 columns at a time: TMEM -> this warp's transpose block -> 16-byte global accesses
        float* ebuf = ebuf_all + ewarp * Cfg::EPI_BUF_FLOATS;
        const int nq = n0 + q * 32;                     // first weight row of this warp
        const int slot = g.first_sk ? 0 : 1;
        float* part = whole ? nullptr : args.partial + ((size_t)cta * 2 + slot) * (TN * 128);
        // TMEM is read 64 columns per wait (16/32/48 at the tail: TN is a multiple of 16); each
        // 16-column block then goes through the transpose buffer
#pragma unroll 1
        for (int c64 = c_begin; c64 < c_end; c64 += 64) {
        const int cols = c_end - c64 < 64 ? c_end - c64 : 64;
        float v64[64];
        if (cols == 64) tmem_ld_cols<64>(t_row + c64, v64);
        else if (cols == 48) tmem_ld_cols<48>(t_row + c64, v64);
        else if (cols == 32) tmem_ld_cols<32>(t_row + c64, v64);
        else tmem_ld_cols<16>(t_row + c64, v64);
        if (args.norm_ssq) {
          // row scales of the folded RMSNorm (linear: a split tile's pieces are scaled alike)
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (k < cols) v64[k] *= s_rms[c64 + k];
        }
        if constexpr (EPI == EPI_SWIGLU) {
          if (whole) {
            if (live) {
              // (columns past `cols` are never stored; give them defined values)
#pragma unroll
              for (int k = 16; k < 64; ++k)
                if (k >= cols) v64[k] = 0.f;
              swiglu_chunk32(v64, cols, ebuf, lane, args, m0 + c64, n_t * 64 + q * 16);
              if (cols > 32)
                swiglu_chunk32(v64 + 32, cols - 32, ebuf, lane, args, m0 + c64 + 32, n_t * 64 + q * 16);
            }
            continue;
          }
        }
#pragma unroll
        for (int c16 = 0; c16 < 64; c16 += 16) {
          if (c16 >= cols) break;
          const int c = c64 + c16;
#pragma unroll
          for (int j = 0; j < 16; ++j) ebuf[j * 33 + lane] = v64[c16 + j];
          __syncwarp();
          if (whole) {
            // item = (token column j, 8 consecutive weight rows): one 16-byte bf16 store
#pragma unroll
            for (int it = 0; it < 2; ++it) {
              const int item = lane + 32 * it, j = item >> 2, r8 = (item & 3) * 8;
              const int m = m0 + c + j, n = nq + r8;
              if (m >= args.M) continue;
              float y[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) y[e] = ebuf[j * 33 + r8 + e];
              if (n + 8 <= args.N) {
                if (args.residual) {
                  const uint4 rr = *reinterpret_cast<const uint4*>(args.residual + (size_t)m * args.ldr + n);
                  const uint32_t r4[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
                  for (int h = 0; h < 4; ++h) {
                    y[2 * h] += bf16lo(r4[h]);
                    y[2 * h + 1] += bf16hi(r4[h]);
                  }
                }
                *reinterpret_cast<uint4*>(args.Y + (size_t)m * args.ldy + n) =
                    make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                               pack_bf16x2(y[6], y[7]));
              } else {
                for (int e = 0; e < 8 && n + e < args.N; ++e) {
                  float o = y[e];
                  if (args.residual) o += bf16f(args.residual[(size_t)m * args.ldr + n + e]);
                  args.Y[(size_t)m * args.ldy + n + e] = f2bf(o);
                }
              }
            }
          } else {
            // split tile: this CTA's fp32 piece, [column][128 rows], float4 along the rows
            // (slot 0 = the piece that opens its stream-K range, 1 = the one that closes it)
#pragma unroll
            for (int it = 0; it < 4; ++it) {
              const int item = lane + 32 * it, j = item >> 3, r4 = (item & 7) * 4;
              const float* src = ebuf + j * 33 + r4;
              __stcg(reinterpret_cast<float4*>(part + (size_t)(c + j) * 128 + q * 32 + r4),
                     make_float4(src[0], src[1], src[2], src[3]));
            }
          }
          __syncwarp();
        }
        }
        release_acc(acc);
      } else {
        // LM-head epilogues (ranges are tile-aligned, so every segment is whole): per token column
        // reduce over the tile's 128 vocabulary rows.  Each 8-column block goes through the warp's
        // transpose block, so lanes 4j .. 4j + 3 scan column j's 32 rows (8 each, reduced as trees)
        // and meet in two shuffles, instead of five shuffles per column per reduction (the butterfly
        // version took 22 us per 192-column tile, 40 us per 384-column tile).
        float* eb = ebuf_all + ewarp * Cfg::EPI_BUF_FLOATS;
        const int jc = lane >> 2, r0 = (lane & 3) * 8;
        const int nr = n0 + q * 32 + r0;        // vocabulary row of this lane's first scanned entry

        // TMEM is read 32 columns per wait (16 at the tail: the halves are multiples of 16)
#pragma unroll 1
        for (int c32 = c_begin; c32 < c_end; c32 += 32) {
          const int cols = c_end - c32 < 32 ? c_end - c32 : 32;
          float v[32];
          if (cols == 32) tmem_ld_cols<32>(t_row + c32, v);
          else tmem_ld_cols<16>(t_row + c32, v);
#pragma unroll
          for (int h = 0; h < 32; h += 8) {
            if (h >= cols) break;
            const int c = c32 + h;
            if constexpr (EPI == EPI_LOGITS) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float z = v[h + j] * (args.norm_ssq ? args.inv_temp * s_rms[c + j] : args.inv_temp);
                const int m = m0 + c + j;
                if (m < args.M && n < args.N) args.P[(size_t)m * args.ldp + n] = z;
                eb[j * 33 + lane] = z;
              }
              __syncwarp();
              float zz[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) zz[i] = nr + i < args.N ? eb[jc * 33 + r0 + i] : -INFINITY;
              float mx = fmaxf(fmaxf(fmaxf(zz[0], zz[1]), fmaxf(zz[2], zz[3])),
                               fmaxf(fmaxf(zz[4], zz[5]), fmaxf(zz[6], zz[7])));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
#pragma unroll
              for (int i = 0; i < 8; ++i) zz[i] = nr + i < args.N ? exp_sm(zz[i] - mx) : 0.f;
              float sm = ((zz[0] + zz[1]) + (zz[2] + zz[3])) + ((zz[4] + zz[5]) + (zz[6] + zz[7]));
              sm += __shfl_xor_sync(0xffffffffu, sm, 1);
              sm += __shfl_xor_sync(0xffffffffu, sm, 2);
              if ((lane & 3) == 0) red[q * TN + c + jc] = make_float2(mx, sm);
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) eb[j * 33 + lane] = v[h + j];
              __syncwarp();
              float zv = -INFINITY;
              int idx = 0x7fffffff;
#pragma unroll
              for (int i = 0; i < 8; ++i) {           // strict > keeps the lowest row on ties
                const float z = eb[jc * 33 + r0 + i];
                if (nr + i < args.N && (z > zv || idx == 0x7fffffff)) { zv = z; idx = nr + i; }
              }
#pragma unroll
              for (int o = 1; o <= 2; o <<= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, zv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
                if (ov > zv || (ov == zv && oi < idx)) { zv = ov; idx = oi; }
              }
              if ((lane & 3) == 0) red[q * TN + c + jc] = make_float2(zv, __int_as_float(idx));
            }
            __syncwarp();                          // eb is rewritten by the next block
          }
        }
        release_acc(acc);
        bar_epi();
        for (int j = etid; j < TN; j += 32 * Cfg::EPI_WARPS) {
          const int m = m0 + j;
          if (m >= args.M || !live) continue;
          float2 accv = red[j];
          for (int w = 1; w < 4; ++w) {
            const float2 o = red[w * TN + j];
            if constexpr (EPI == EPI_LOGITS) {
              const float mx = fmaxf(accv.x, o.x);
              const float s = (accv.x == -INFINITY ? 0.f : accv.y * exp_sm(accv.x - mx)) +
                              (o.x == -INFINITY ? 0.f : o.y * exp_sm(o.x - mx));
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
  if constexpr (PAIR) {
    // the peer may still arrive on this CTA's barriers (or this one on the peer's) until both
    // are here
    cluster_sync_all();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem, Cfg::TMEM_COLS);
    }
  } else {
    if (warp == 1) tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// Host side: one instantiation's launch.
template <int BN, int NSUB, int EPI, bool PAIR = false>
static bool linear_tc_configure() {
  static bool configured[64] = {};   // per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && configured[dev]) return true;
  if (cudaFuncSetAttribute(linear_tc_kernel<BN, NSUB, EPI, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           LinearCfg<BN, NSUB, PAIR, EPI == EPI_LOGITS || EPI == EPI_ARGMAX>::SMEM_BYTES) !=
      cudaSuccess)
    return false;
  if (dev >= 0 && dev < 64) configured[dev] = true;
  return true;
}

template <int BN, int NSUB, int EPI>
static cudaError_t launch_linear_tc_one(const CUtensorMap& tw, const CUtensorMap& tx, const LinearArgs& a,
                                        dim3 grid, cudaStream_t st) {
  using Cfg = LinearCfg<BN, NSUB, false, EPI == EPI_LOGITS || EPI == EPI_ARGMAX>;
  if (!linear_tc_configure<BN, NSUB, EPI>()) return cudaGetLastError();
  cudaError_t e = launch_k(linear_tc_kernel<BN, NSUB, EPI>, grid, dim3(Cfg::THREADS), Cfg::SMEM_BYTES, st,
                           tw, tx, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The pair build: `pairs` clusters of 2 CTAs, and how many pairs can be resident at once.
template <int BN, int NSUB, int EPI>
struct LinearTcPair {
  using Cfg = LinearCfg<BN, NSUB, true, EPI == EPI_LOGITS || EPI == EPI_ARGMAX>;
  static cudaError_t launch(const CUtensorMap& tw, const CUtensorMap& tx, const LinearArgs& a, int pairs,
                            cudaStream_t st) {
    if (!linear_tc_configure<BN, NSUB, EPI, true>()) return cudaGetLastError();
    cudaError_t e = launch_kc(linear_tc_kernel<BN, NSUB, EPI, true>, dim3(2 * pairs), dim3(Cfg::THREADS),
                              Cfg::SMEM_BYTES, st, 2, tw, tx, a);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  static int capacity() {
    if (!linear_tc_configure<BN, NSUB, EPI, true>()) {
      cudaGetLastError();
      return 0;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * 64);
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)linear_tc_kernel<BN, NSUB, EPI, true>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n;
  }
};

}  // namespace spec
