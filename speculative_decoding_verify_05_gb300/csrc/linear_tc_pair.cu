// Instantiations of the persistent tcgen05 verify GEMM on CTA pairs (2-SM MMA, 256-row pair tiles)
// for the bf16 (+ residual) and SwiGLU epilogues, and the resident-pair query.
#include "internal.h"
#include "linear_tc_kernel.cuh"

namespace spec {

int linear_tc_pair_capacity(int BN, int NSUB, bool lmhead) {
  static int cache[64][2][3][17];   // [device][lmhead][NSUB][BN / 16]: pairs + 1, 0 = not asked
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cacheable = dev >= 0 && dev < 64 && NSUB >= 1 && NSUB <= 2 && BN % 16 == 0 && BN / 16 <= 16;
  if (cacheable && cache[dev][lmhead][NSUB][BN / 16] != 0) return cache[dev][lmhead][NSUB][BN / 16] - 1;
  int cap = 0;
  switch (NSUB * 1000 + BN) {
#define X(bn, ns)                                                                                   \
  case ns * 1000 + bn:                                                                              \
    cap = lmhead ? linear_tc_pair_capacity_lmhead(bn, ns) : LinearTcPair<bn, ns, EPI_BF16>::capacity(); \
    break;
    SPEC_TC_PAIR_SHAPES(X)
#undef X
    default: cap = 0;
  }
  if (cacheable) cache[dev][lmhead][NSUB][BN / 16] = cap + 1;
  return cap;
}

static cudaError_t launch_pair_bf16(int BN, int NSUB, bool swiglu, const CUtensorMap& tw, const CUtensorMap& tx,
                                    const LinearArgs& a, int pairs, cudaStream_t s) {
  switch (NSUB * 1000 + BN) {
#define X(bn, ns)                                                                            \
  case ns * 1000 + bn:                                                                       \
    return swiglu ? LinearTcPair<bn, ns, EPI_SWIGLU>::launch(tw, tx, a, pairs, s)            \
                  : LinearTcPair<bn, ns, EPI_BF16>::launch(tw, tx, a, pairs, s);
    SPEC_TC_PAIR_SHAPES(X)
#undef X
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_linear_tc_pair(int BN, int NSUB, int epi, const CUtensorMap& tw, const CUtensorMap& tx,
                                  const LinearArgs& a, int pairs, cudaStream_t s) {
  if (epi == EPI_BF16 || epi == EPI_SWIGLU) return launch_pair_bf16(BN, NSUB, epi == EPI_SWIGLU, tw, tx, a, pairs, s);
  if (epi == EPI_LOGITS || epi == EPI_ARGMAX) return launch_linear_tc_pair_lmhead(BN, NSUB, epi == EPI_ARGMAX, tw, tx, a, pairs, s);
  return cudaErrorInvalidValue;
}

}  // namespace spec
