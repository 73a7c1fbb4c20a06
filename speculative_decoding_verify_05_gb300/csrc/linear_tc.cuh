// Tensor-core (tcgen05 + TMEM + TMA) weight-streaming GEMM for the verify pass.
//
// Orientation: the weight is the MMA's A operand (128 weight rows per tile,
// M_mma = 128) and the verify rows are the B operand (BN tokens, the MMA's
// N), so the accumulator tile D[n, m] = sum_k W[n, k] X[m, k] lives in TMEM
// with one weight row per TMEM lane.  For a handful of verify rows this keeps
// the whole 128-lane tensor core on the weight stream instead of padding the
// token dimension to 128.
//
// Persistent schedule (data-parallel + stream-K): one CTA per SM first takes
// whole tiles round-robin (as many as every CTA can get), then an equal
// contiguous range of the (tile, 64-wide k-step) units of the remaining tiles,
// so every SM streams the same number of weight bytes whatever the matrix shape
// while only the remainder tiles are cut into pieces.  Roles (6 warps): warp 0 issues TMA loads
// of 128x64 weight tiles and BNx64 activation tiles (128-byte swizzle) into a
// STAGES-deep ring without ever draining it; warp 1 issues four
// tcgen05.mma (K = 16) per stage into one of two TMEM accumulators; warps 2-9
// drain the other accumulator meanwhile (two warps per TMEM lane quarter, each
// taking half of the token columns).  A tile whose k-steps are split
// between CTAs leaves one fp32 piece per CTA in the workspace; a second, fully
// parallel kernel sums the pieces in CTA order, adds the residual and rounds
// to bf16 (one SM finishing a whole split tile alone would leave the rest of
// the GPU idle at the end of the GEMM).
#pragma once

#include "common.cuh"

namespace spec {

enum LinearEpilogue : int {
  EPI_BF16 = 0,        // Y = acc (+ residual) -> bf16
  EPI_LOGITS = 1,      // P = acc * inv_temp (fp32) + per-tile (max, sum exp) per token
  EPI_ARGMAX = 2,      // per-tile (max, argmax) per token only
  EPI_SWIGLU = 3,      // weight rows interleaved per 16 (gate block, up block): Y = silu(gate) * up
  EPI_ROPE = 4         // cluster kernel: 128-column heads n_t < rope_tiles rotated (rotate-half) with
                       // the per-row (cos, sin) table rope_cs [M][64] before rounding
};

struct LinearArgs {
  int M, N, K;
  int k_tiles;          // 64-wide k-steps per tile
  int tiles_m, tiles_n;
  long long units;      // work units: cluster tiles * k_tiles
  int grid;             // persistent CTAs
  long long dp_tiles;   // tiles 0 .. dp_tiles - 1 go whole to CTAs c, c + grid, ...
  long long sk_units;   // the k-steps of the other tiles, split evenly between the CTAs (stream-K)
  uint16_t* Y;
  int ldy;
  const uint16_t* residual;
  int ldr;
  float* partial;       // [grid][2][TN][128] fp32 (split tiles only)
  int tn;               // token columns per tile (BN * NSUB)
  int epi;              // the reduce kernel's epilogue: EPI_BF16 (+ residual) or EPI_SWIGLU
  unsigned* status;     // library status word (bounded-wait timeouts)
  const float2* rope_cs;  // EPI_ROPE
  int rope_tiles;
  float inv_temp;       // EPI_LOGITS
  float* P;             // EPI_LOGITS: [M x N] fp32, leading dimension ldp
  long long ldp;
  float2* stats;        // EPI_LOGITS / EPI_ARGMAX: [M][tiles_n] (max, sum) or (max, idx bits)
  // RMSNorm of X folded into the product (its weight folded into W beforehand): row m of the result
  // is scaled by 1 / sqrt(sum_t norm_ssq[m][t] / norm_k + norm_eps) (t in order), the partial sums
  // of squares of X's row m written by the product that stored X (nullptr: no scaling)
  const float* norm_ssq;
  int norm_tiles;
  float norm_k, norm_eps;
  // the partial sums of squares of Y as stored (bf16), per row and 128-column tile: [M][tiles_n]
  // (nullptr: none)
  float* out_ssq;
  // 1: the persistent kernel runs on CTA pairs; its work tiles are 256 weight rows (tile t covers
  // token tile t % tiles_m and the 128-row tiles 2 (t / tiles_m) + 0, 1), grid counts pairs and
  // the CTA of rank r in pair c leaves its split-K pieces in partial slots 2 (2c + r) + 0, 1
  int pair;
  // 1: W is not written by the kernel ahead on the stream, so the first ring stages' weight tiles
  // may be loaded before the programmatic-dependent-launch wait
  int w_early;
};

// 1 / rms of row m from its partial sums of squares (t in order; the loads go out 8 at a time).
__device__ __forceinline__ float row_inv_rms(const LinearArgs& a, int m) {
  const float* p = a.norm_ssq + (size_t)m * a.norm_tiles;
  float s = 0.f;
  int t = 0;
  for (; t + 8 <= a.norm_tiles; t += 8) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldg(p + t + i);
#pragma unroll
    for (int i = 0; i < 8; ++i) s += v[i];
  }
  for (; t < a.norm_tiles; ++t) s += __ldg(p + t);
  return 1.0f / sqrtf(s / a.norm_k + a.norm_eps);
}
// s_rms[j] = 1 / rms of row m_first + j for j < n (1 past M, or without a folded norm), by threads
// tid .. of nthreads: run by warps that are idle during the main loop, so it overlaps the MMAs.
__device__ __forceinline__ void fill_row_scales(const LinearArgs& a, float* s_rms, int m_first, int n, int tid,
                                                int nthreads) {
  for (int j = tid; j < n; j += nthreads) {
    const int m = m_first + j;
    s_rms[j] = (a.norm_ssq && m < a.M) ? row_inv_rms(a, m) : 1.f;
  }
}

// SwiGLU epilogue of 32 token columns of one whole tile held by one warp (v[0..31]; columns
// past `cols` are never stored): gate and up rows are interleaved in blocks of 16, so lane l < 16
// holds gate row l of the warp's block and lane l + 16 the matching up row.  One register
// exchange gives lane l < 16 the up values of columns 0-15 and lane l + 16 the gate values of
// columns 16-31; each lane writes silu(gate) * up for its 16 columns as bf16 into the warp's
// staging buffer ([column][16 rows], column c at slot c ^ (c >> 4) so the two half-warps hit
// different banks), and the warp stores 16-byte runs of 8 outputs along A's rows.
__device__ __forceinline__ void swiglu_chunk32(const float* v, int cols, float* ebuf, int lane,
                                               const LinearArgs& args, int m_first, int n_first) {
  const bool lo = lane < 16;
  uint16_t* eb = reinterpret_cast<uint16_t*>(ebuf);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float send = lo ? v[k + 16] : v[k];
    const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
    const float g = lo ? v[k] : recv;
    const float u = lo ? recv : v[k + 16];
    const int col = lo ? k : k + 16;
    eb[(col ^ (col >> 4)) * 16 + (lane & 15)] = f2bf(silu(g) * u);
  }
  __syncwarp();
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int item = lane + 32 * it, col = item >> 1, h = item & 1;
    const int m = m_first + col;
    if (col < cols && m < args.M)
      *reinterpret_cast<uint4*>(args.Y + (size_t)m * args.ldy + n_first + h * 8) =
          *reinterpret_cast<const uint4*>(eb + (col ^ (col >> 4)) * 16 + h * 8);
  }
  __syncwarp();
}

// SwiGLU epilogue of a whole tile straight from TMEM (no pieces to sum): 8 warps, warp w reads TMEM
// lane quarter w % 4 and half w / 4 of the TN token columns, 64 columns per wait, scales them by a
// folded RMSNorm's row scales (s_rms[column], or nullptr) and stores silu(gate) * up through its
// transpose block eb (16 x 33 floats per warp).
template <int TN>
__device__ __forceinline__ void tmem_swiglu_epilogue(uint32_t tmem, int warp, int lane, const LinearArgs& args,
                                                     int m_t, int n_t, const float* s_rms, float* ebuf) {
  const int q = warp & 3;
  const uint32_t t_row = tmem + (uint32_t(q * 32) << 16);
  constexpr int C_MID = TN / 32 * 16;
  const int c_lo = warp < 4 ? 0 : C_MID, c_hi = warp < 4 ? C_MID : TN;
  float* eb = ebuf + warp * (16 * 33);
#pragma unroll 1
  for (int c64 = c_lo; c64 < c_hi; c64 += 64) {
    const int cols = c_hi - c64 < 64 ? c_hi - c64 : 64;
    float v[64];
    if (cols == 64) tmem_ld_cols<64>(t_row + c64, v);
    else if (cols == 48) tmem_ld_cols<48>(t_row + c64, v);
    else if (cols == 32) tmem_ld_cols<32>(t_row + c64, v);
    else tmem_ld_cols<16>(t_row + c64, v);
#pragma unroll
    for (int k = 0; k < 64; ++k) {
      if (k >= cols) v[k] = 0.f;        // (never stored; defined values)
      else if (s_rms) v[k] *= s_rms[c64 + k];
    }
    swiglu_chunk32(v, cols, eb, lane, args, m_t * TN + c64, n_t * 64 + q * 16);
    if (cols > 32) swiglu_chunk32(v + 32, cols - 32, eb, lane, args, m_t * TN + c64 + 32, n_t * 64 + q * 16);
  }
}

// k-step of the tensor-core GEMMs: LIN_BK bf16 per operand row and stage (one swizzle row of
// LIN_ROW_BYTES): 64 with 128-byte swizzle, or 32 with 64-byte swizzle.  Half-size stages keep
// more of the shared-memory ring in flight while the tensor core works on one of them, but each
// weight row then arrives in 64-byte pieces: measured on GB300 the 32-wide step was 1.3-1.7x
// slower on every verify shape (gate|up 89 -> 115 us, LM head 0.74 -> 1.22 ms), so 64 it is.
constexpr int LIN_BK = 64;
constexpr int LIN_ROW_BYTES = LIN_BK * 2;
__device__ __forceinline__ uint64_t umma_desc_lin(uint32_t smem_addr) {
  return LIN_BK == 64 ? umma_desc_sw128(smem_addr) : umma_desc_sw64(smem_addr);
}

// A CTA tile is 128 weight rows x TN = NSUB * BN verify rows: NSUB MMAs of N = BN per
// k-substep share one weight tile, so with up to 384 verify rows (kMaxTN) every weight byte is
// read from HBM once.  PAIR: the tile of a CTA pair is 256 weight rows (128 per CTA) x TN, and
// each CTA stages half (HB) of every MMA's token rows.
template <int BN, int NSUB, bool PAIR = false, bool STATS = false>
struct LinearCfg {
  static constexpr int TN = BN * NSUB;
  static constexpr int HB = PAIR ? BN / 2 : BN;
  static constexpr int A_BYTES = 128 * LIN_ROW_BYTES;
  static constexpr int B_BYTES = NSUB * HB * LIN_ROW_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // accumulator buffer: power-of-two columns >= TN; two buffers when they fit in TMEM
  static constexpr int ACC_COLS = TN <= 16 ? 16 : (TN <= 32 ? 32 : (TN <= 64 ? 64 : (TN <= 128 ? 128 : (TN <= 256 ? 256 : 512))));
  static constexpr int NBUF = 2 * ACC_COLS <= 512 ? 2 : 1;
  static constexpr int TMEM_COLS = NBUF * ACC_COLS < 32 ? 32 : NBUF * ACC_COLS;
  // producer warp, MMA warp, 8 epilogue warps (two per TMEM lane quarter, each half of the columns)
  static constexpr int THREADS = 320;
  static constexpr int EPI_WARPS = 8;
  // per epilogue warp: a column block x 32 rows of fp32 (row stride 33) to turn TMEM rows into
  // 16-byte stores along the weight rows (16 columns), or to scan the LM head's columns (STATS:
  // 8 columns, which leaves a 2-SM LM head room for a fifth ring stage)
  static constexpr int EPI_COLS = STATS ? 8 : 16;
  static constexpr int EPI_BUF_FLOATS = EPI_COLS * 33;
  // besides the ring: barriers/flags (1 KB) + LM-head reduction scratch (4 warps x TN x float2) +
  // epilogue transpose blocks + row scales of a folded RMSNorm (TN floats) + alignment slack
  static constexpr int EXTRA = 1024 + 4 * TN * 8 + EPI_WARPS * EPI_BUF_FLOATS * 4 + TN * 4 + 1024;
  static constexpr int STAGES_RING = (200 * 1024) / STAGE_BYTES;
  static constexpr int STAGES_SMEM = (227 * 1024 - EXTRA) / STAGE_BYTES;
  static constexpr int STAGES_FIT = STAGES_RING < STAGES_SMEM ? STAGES_RING : STAGES_SMEM;
  static constexpr int STAGES = STAGES_FIT > 24 ? 24 : STAGES_FIT;
  static constexpr int RMS_OFF = STAGES * STAGE_BYTES + 1024 + 4 * TN * 8 + EPI_WARPS * EPI_BUF_FLOATS * 4;
  static constexpr int SMEM_BYTES = RMS_OFF + TN * 4 + 1024;
};

}  // namespace spec
