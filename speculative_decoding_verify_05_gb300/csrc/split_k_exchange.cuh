// Split-K exchange on chip: the CTAs of a thread-block cluster that computed pieces of the same
// (weight tile, token tile) sum them through distributed shared memory.  Used by the cluster split-K
// GEMM (one CTA per piece) and its 2-SM variant (one CTA pair per piece, each CTA of a pair holding
// half of the 256 weight rows).  Token columns are dealt out in groups of 4 ("chunks"), cpr
// consecutive chunks per participant; after the main loops each participant pushes every chunk of
// its fp32 accumulator into the owning participant's shared-memory ring (idle by then) at slot [its
// index], and after a cluster barrier each owner sums the S slots of its chunks in participant order
// (deterministic), then runs the epilogue.
#pragma once

#include "linear_tc.cuh"

namespace spec {

__device__ __forceinline__ void dsmem_st_f4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void smem_st_f4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// Slot row of weight row r: rows are XOR-swizzled inside each group of 8 so that threads
// reading 8 consecutive rows each (rows 8t + i, t = 0..7) hit 8 different bank groups.
__device__ __forceinline__ int slot_row(int r) { return r ^ ((r >> 3) & 7); }

// Push this CTA's accumulator (TN token columns of 128 TMEM lanes) to the owners' slots: 8 warps,
// warp w reads lane quarter w % 4 and half w / 4 of the columns.  Participant `me` writes slot
// [me][chunk - owner cpr] of owner `owner`, which lives in cluster rank owner * stride + offset.
// With `have` false the piece is zero (an empty k-range).
template <int TN>
__device__ __forceinline__ void push_accumulator(uint32_t tmem, int warp, int lane, bool have, const void* slots,
                                                 int cpr, int me, int stride, int offset) {
  const int q = warp & 3;
  const int row = q * 32 + lane;
  const uint32_t t_row = tmem + (uint32_t(q * 32) << 16);
  const uint32_t base = smem_u32(slots);
  constexpr int C_MID = TN / 32 * 16;
  const int c_lo = warp < 4 ? 0 : C_MID, c_hi = warp < 4 ? C_MID : TN;
  // 64 columns per TMEM wait (16, 32 or 48 at the ends: both halves are multiples of 16), then
  // their remote stores back to back
#pragma unroll 1
  for (int c = c_lo; c < c_hi; c += 64) {
    float v[64];
    const int cols = c_hi - c < 64 ? c_hi - c : 64;
    if (have) {
      if (cols == 64) tmem_ld_cols<64>(t_row + c, v);
      else if (cols == 48) tmem_ld_cols<48>(t_row + c, v);
      else if (cols == 32) tmem_ld_cols<32>(t_row + c, v);
      else tmem_ld_cols<16>(t_row + c, v);
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) v[j] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      if (4 * e >= cols) break;
      const int chunk = c / 4 + e;
      const int owner = chunk / cpr, kk = chunk - owner * cpr;
      const uint32_t off = (uint32_t)(((me * cpr + kk) * 128 + slot_row(row)) * 16);
      // (a participant's own chunks take the plain shared-memory store: the cluster path is as slow
      // for a local address as for a peer's)
      if (owner == me) smem_st_f4(base + off, v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
      else dsmem_st_f4(dsmem_map(base + off, (uint32_t)(owner * stride + offset)), v[4 * e], v[4 * e + 1],
                       v[4 * e + 2], v[4 * e + 3]);
    }
  }
}

// The token rows participant `me` stores: the first and how many (their row scales of a folded
// RMSNorm go to s_rms before the epilogue, see fill_row_scales).
template <int TN>
__device__ __forceinline__ int split_first_row(int cpr, int me, int m_t) { return m_t * TN + me * cpr * 4; }
template <int TN>
__device__ __forceinline__ int split_rows(int cpr, int me) {
  const int n = min(cpr, TN / 4 - me * cpr);
  return n > 0 ? n * 4 : 0;
}

// Owner `me`'s chunks: sum the S slots in participant order and store them as weight tile n_t,
// token tile m_t of Y with the epilogue args.epi (bf16 + residual, SwiGLU, or RoPE); NT threads.
// With a folded RMSNorm, s_rms holds the scales of the owner's rows (filled and made visible to
// every thread before the call).
template <int TN, int NT>
__device__ __forceinline__ void split_sum_epilogue(const float4* slots, const LinearArgs& args, int S, int cpr,
                                                   int me, int n_t, int m_t, const float* s_rms) {
  // ---------------- this rank's chunks: sum the S slots in rank order, add the residual, store.
  // Item = (chunk, 8 consecutive weight rows): 4 tokens x 8 rows, so the residual and Y move
  // in 16-byte pieces (8 bf16 of one token row).
  const int n_chunks = min(cpr, TN / 4 - me * cpr);
  const bool scale = args.norm_ssq != nullptr;
  if (args.epi == EPI_SWIGLU) {
    // gate and up rows interleaved per 16: item = (chunk, 8 gate rows r8..r8+7 with r8 % 32 < 16);
    // the matching up rows are r8+16..; 8 outputs per token at column n_t 64 + (r8 / 32) 16 + r8 % 32
    const int sitems = (n_chunks > 0 ? n_chunks : 0) * 8;
    for (int it = threadIdx.x; it < sitems; it += NT) {
      const int kk = it >> 3, q8 = it & 7, r8 = (q8 >> 1) * 32 + (q8 & 1) * 8;
      float g[8][4], u[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 vg = slots[kk * 128 + slot_row(r8 + i)];
        const float4 vu = slots[kk * 128 + slot_row(r8 + 16 + i)];
        g[i][0] = vg.x; g[i][1] = vg.y; g[i][2] = vg.z; g[i][3] = vg.w;
        u[i][0] = vu.x; u[i][1] = vu.y; u[i][2] = vu.z; u[i][3] = vu.w;
      }
      for (int s2 = 1; s2 < S; ++s2) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 vg = slots[(s2 * cpr + kk) * 128 + slot_row(r8 + i)];
          const float4 vu = slots[(s2 * cpr + kk) * 128 + slot_row(r8 + 16 + i)];
          g[i][0] += vg.x; g[i][1] += vg.y; g[i][2] += vg.z; g[i][3] += vg.w;
          u[i][0] += vu.x; u[i][1] += vu.y; u[i][2] += vu.z; u[i][3] += vu.w;
        }
      }
      const int n = n_t * 64 + (r8 >> 5) * 16 + (r8 & 31);
      const int mb = m_t * TN + (me * cpr + kk) * 4;
      if (scale) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float rs = s_rms[kk * 4 + e];
#pragma unroll
          for (int i = 0; i < 8; ++i) { g[i][e] *= rs; u[i][e] *= rs; }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (mb + e >= args.M) break;
        uint32_t o4[4];
#pragma unroll
        for (int h = 0; h < 4; ++h)
          o4[h] = pack_bf16x2(silu(g[2 * h][e]) * u[2 * h][e], silu(g[2 * h + 1][e]) * u[2 * h + 1][e]);
        *reinterpret_cast<uint4*>(args.Y + (size_t)(mb + e) * args.ldy + n) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
    }
  }
  // RoPE heads: item = (chunk, 8 dims r8..r8+7 of the first half); the pair dims r8+64.. rotate
  // with them: (a, b) -> (a c - b s, b c + a s), c, s from row m's table entry for dim r8 + i
  const bool rope = args.epi == EPI_ROPE && n_t < args.rope_tiles;
  if (rope) {
    const int ritems = (n_chunks > 0 ? n_chunks : 0) * 8;
    for (int it = threadIdx.x; it < ritems; it += NT) {
      const int kk = it >> 3, r8 = (it & 7) * 8;
      const int mb = m_t * TN + (me * cpr + kk) * 4;
      // this item's table entries first: their global loads overlap the slot sums below
      float2 csr[4][8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = min(mb + e, args.M - 1);
        const float4* cs4 = reinterpret_cast<const float4*>(args.rope_cs + (size_t)m * 64 + r8);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 v = __ldg(cs4 + q);
          csr[e][2 * q] = make_float2(v.x, v.y);
          csr[e][2 * q + 1] = make_float2(v.z, v.w);
        }
      }
      float a[8][4], b[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 va = slots[kk * 128 + slot_row(r8 + i)];
        const float4 vb = slots[kk * 128 + slot_row(r8 + 64 + i)];
        a[i][0] = va.x; a[i][1] = va.y; a[i][2] = va.z; a[i][3] = va.w;
        b[i][0] = vb.x; b[i][1] = vb.y; b[i][2] = vb.z; b[i][3] = vb.w;
      }
      for (int s2 = 1; s2 < S; ++s2) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 va = slots[(s2 * cpr + kk) * 128 + slot_row(r8 + i)];
          const float4 vb = slots[(s2 * cpr + kk) * 128 + slot_row(r8 + 64 + i)];
          a[i][0] += va.x; a[i][1] += va.y; a[i][2] += va.z; a[i][3] += va.w;
          b[i][0] += vb.x; b[i][1] += vb.y; b[i][2] += vb.z; b[i][3] += vb.w;
        }
      }
      const int n = n_t * 128 + r8;
      if (scale) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float rs = s_rms[kk * 4 + e];
#pragma unroll
          for (int i = 0; i < 8; ++i) { a[i][e] *= rs; b[i][e] *= rs; }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = mb + e;
        if (m >= args.M) break;
        uint32_t x4[4], y4[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 c0 = csr[e][2 * h], c1 = csr[e][2 * h + 1];
          const float a0 = a[2 * h][e], a1 = a[2 * h + 1][e], b0 = b[2 * h][e], b1 = b[2 * h + 1][e];
          x4[h] = pack_bf16x2(a0 * c0.x - b0 * c0.y, a1 * c1.x - b1 * c1.y);
          y4[h] = pack_bf16x2(b0 * c0.x + a0 * c0.y, b1 * c1.x + a1 * c1.y);
        }
        *reinterpret_cast<uint4*>(args.Y + (size_t)m * args.ldy + n) = make_uint4(x4[0], x4[1], x4[2], x4[3]);
        *reinterpret_cast<uint4*>(args.Y + (size_t)m * args.ldy + n + 64) = make_uint4(y4[0], y4[1], y4[2], y4[3]);
      }
    }
  }
  const int items = (args.epi == EPI_SWIGLU || rope || n_chunks <= 0) ? 0 : n_chunks * 16;
  // (a chunk's 16 items sit in 16 consecutive lanes: the loop runs whole warps so that they can sum
  // the squares of the chunk's stored values for out_ssq)
  const int items_w = (items + 31) / 32 * 32;
  for (int it = threadIdx.x; it < items_w; it += NT) {
    const bool act = it < items;
    const int kk = act ? it >> 4 : 0, r8 = (it & 15) * 8;
    const int n0 = n_t * 128 + r8;
    const int mb = m_t * TN + (me * cpr + kk) * 4;
    const bool whole = act && n0 + 8 <= args.N;
    // the residual rows first: their global loads overlap the slot sums below
    uint4 res[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      res[e] = (whole && args.residual && mb + e < args.M)
                   ? *reinterpret_cast<const uint4*>(args.residual + (size_t)(mb + e) * args.ldr + n0)
                   : make_uint4(0, 0, 0, 0);
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = slots[kk * 128 + slot_row(r8 + i)];
      acc[i][0] = v.x; acc[i][1] = v.y; acc[i][2] = v.z; acc[i][3] = v.w;
    }
    for (int s2 = 1; s2 < S; ++s2) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = slots[(s2 * cpr + kk) * 128 + slot_row(r8 + i)];
        acc[i][0] += v.x; acc[i][1] += v.y; acc[i][2] += v.z; acc[i][3] += v.w;
      }
    }
    if (scale) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float rs = s_rms[kk * 4 + e];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i][e] *= rs;
      }
    }
    float sq[4] = {0.f, 0.f, 0.f, 0.f};
    if (whole) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (mb + e >= args.M) break;
        const uint32_t r4[4] = {res[e].x, res[e].y, res[e].z, res[e].w};
        uint32_t o4[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          o4[h] = pack_bf16x2(acc[2 * h][e] + bf16lo(r4[h]), acc[2 * h + 1][e] + bf16hi(r4[h]));
          sq[e] += bf16lo(o4[h]) * bf16lo(o4[h]) + bf16hi(o4[h]) * bf16hi(o4[h]);
        }
        *reinterpret_cast<uint4*>(args.Y + (size_t)(mb + e) * args.ldy + n0) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
    } else if (act) {
      for (int e = 0; e < 4 && mb + e < args.M; ++e)
        for (int i = 0; i < 8 && n0 + i < args.N; ++i) {
          float o = acc[i][e];
          if (args.residual) o += bf16f(args.residual[(size_t)(mb + e) * args.ldr + n0 + i]);
          const uint16_t ob = f2bf(o);
          args.Y[(size_t)(mb + e) * args.ldy + n0 + i] = ob;
          sq[e] += bf16f(ob) * bf16f(ob);
        }
    }
    if (args.out_ssq) {
      // the chunk's 16 lanes (128 columns of the tile) in a fixed butterfly
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) sq[e] += __shfl_xor_sync(0xffffffffu, sq[e], o);
      if (act && (it & 15) == 0)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (mb + e < args.M) args.out_ssq[(size_t)(mb + e) * args.tiles_n + n_t] = sq[e];
    }
  }
}

}  // namespace spec
