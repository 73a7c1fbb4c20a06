// Tensor-core (tcgen05 + TMEM + TMA) weight-streaming GEMM for the verify pass.
//
// Orientation: the weight is the MMA's A operand (128 weight rows per CTA
// tile, M_mma = 128) and the verify rows are the B operand (BN tokens, the
// MMA's N), so the accumulator tile D[n, m] = sum_k W[n, k] X[m, k] lives in
// TMEM with one weight row per TMEM lane.  For a handful of verify rows this
// keeps the whole 128-lane tensor core busy on the weight stream instead of
// padding the token dimension to 128.
//
// Pipeline per CTA (128 threads): warp 0 / lane 0 issues TMA loads of
// 128x64 weight tiles and BNx64 activation tiles (128-byte swizzle) into a
// STAGES-deep shared-memory ring; warp 1 / lane 0 issues four
// tcgen05.mma (K = 16 each) per stage and releases the stage with
// tcgen05.commit; all four warps then drain TMEM (tcgen05.ld) in the epilogue.
//
// Split-K: the grid's z dimension splits the K loop.  Each split writes an
// fp32 partial tile to the workspace; the CTA that arrives last on the
// tile's counter (atomicAdd, no waiting) sums the partials in split order,
// adds the residual, rounds to bf16 and resets the counter to zero.
#pragma once

#include "common.cuh"

namespace spec {

enum LinearEpilogue : int {
  EPI_BF16 = 0,        // Y = acc (+ residual) -> bf16
  EPI_LOGITS = 1,      // P = acc * inv_temp (fp32) + per-tile (max, sum exp) per token
  EPI_ARGMAX = 2       // per-tile (max, argmax) per token only
};

struct LinearArgs {
  int M, N, K;
  int k_tiles;          // ceil(K / 64)
  int splits;
  int tiles_m;
  uint16_t* Y;
  int ldy;
  const uint16_t* residual;
  int ldr;
  float* partial;       // [tiles][splits][BN][128] fp32 (split-K only)
  unsigned* counters;   // [tiles] zero-initialised arrival counters (split-K only)
  unsigned* status;     // library status word (bounded-wait timeouts)
  float inv_temp;       // EPI_LOGITS
  float* P;             // EPI_LOGITS: [M x N] fp32
  float2* stats;        // EPI_LOGITS / EPI_ARGMAX: [M][n_tiles] (max, sum) or (max, idx bits)
  int n_tiles;
};

template <int BN>
struct LinearCfg {
  static constexpr int A_BYTES = 128 * 64 * 2;
  static constexpr int B_BYTES = BN * 64 * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES =
      BN <= 64 ? 4 : ((200 * 1024) / STAGE_BYTES > 6 ? 6 : (200 * 1024) / STAGE_BYTES);
  static constexpr int TMEM_COLS = BN <= 32 ? 32 : (BN <= 64 ? 64 : (BN <= 128 ? 128 : 256));
  // ring + barriers + tmem slot + epilogue scratch (4 warps x BN x float2), + 1 KB alignment slack
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 4 * BN * 8 + 1024;
};

}  // namespace spec
