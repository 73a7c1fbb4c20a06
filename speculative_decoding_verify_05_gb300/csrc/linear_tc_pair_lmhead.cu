// Instantiations of the persistent tcgen05 verify GEMM on CTA pairs for the LM-head epilogues
// (logits + softmax statistics, or argmax).
#include "internal.h"
#include "linear_tc_kernel.cuh"

namespace spec {

int linear_tc_pair_capacity_lmhead(int BN, int NSUB) {
  switch (NSUB * 1000 + BN) {
#define X(bn, ns) \
  case ns * 1000 + bn: return LinearTcPair<bn, ns, EPI_LOGITS>::capacity();
    SPEC_TC_PAIR_SHAPES(X)
#undef X
    default: return 0;
  }
}

cudaError_t launch_linear_tc_pair_lmhead(int BN, int NSUB, bool greedy, const CUtensorMap& tw, const CUtensorMap& tx,
                                         const LinearArgs& a, int pairs, cudaStream_t s) {
  switch (NSUB * 1000 + BN) {
#define X(bn, ns)                                                                   \
  case ns * 1000 + bn:                                                              \
    return greedy ? LinearTcPair<bn, ns, EPI_ARGMAX>::launch(tw, tx, a, pairs, s)   \
                  : LinearTcPair<bn, ns, EPI_LOGITS>::launch(tw, tx, a, pairs, s);
    SPEC_TC_PAIR_SHAPES(X)
#undef X
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spec
