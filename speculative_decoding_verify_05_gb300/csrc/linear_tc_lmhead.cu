// Instantiations of the tcgen05 verify GEMM for the LM-head (logits + softmax statistics, or argmax) epilogue.
#include "internal.h"
#include "linear_tc_kernel.cuh"

namespace spec {

template <int BN, int EPI>
static cudaError_t launch_one(const CUtensorMap& tw, const CUtensorMap& tx, const LinearArgs& a,
                              dim3 grid, cudaStream_t st) {
  constexpr int smem = LinearCfg<BN>::SMEM_BYTES;
  static bool configured[64] = {};   // per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(linear_tc_kernel<BN, EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  linear_tc_kernel<BN, EPI><<<grid, 128, smem, st>>>(tw, tx, a);
  return cudaGetLastError();
}

cudaError_t launch_linear_tc_lmhead(int BN, bool greedy, const CUtensorMap& tw,
                                    const CUtensorMap& tx, const LinearArgs& a, dim3 grid,
                                    cudaStream_t s) {
  if (greedy) {
    switch (BN) {
      case 16: return launch_one<16, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 32: return launch_one<32, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 48: return launch_one<48, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 64: return launch_one<64, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 80: return launch_one<80, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 96: return launch_one<96, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 112: return launch_one<112, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 128: return launch_one<128, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 144: return launch_one<144, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 160: return launch_one<160, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 176: return launch_one<176, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 192: return launch_one<192, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 208: return launch_one<208, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 224: return launch_one<224, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 240: return launch_one<240, EPI_ARGMAX>(tw, tx, a, grid, s);
      case 256: return launch_one<256, EPI_ARGMAX>(tw, tx, a, grid, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (BN) {
    case 16: return launch_one<16, EPI_LOGITS>(tw, tx, a, grid, s);
    case 32: return launch_one<32, EPI_LOGITS>(tw, tx, a, grid, s);
    case 48: return launch_one<48, EPI_LOGITS>(tw, tx, a, grid, s);
    case 64: return launch_one<64, EPI_LOGITS>(tw, tx, a, grid, s);
    case 80: return launch_one<80, EPI_LOGITS>(tw, tx, a, grid, s);
    case 96: return launch_one<96, EPI_LOGITS>(tw, tx, a, grid, s);
    case 112: return launch_one<112, EPI_LOGITS>(tw, tx, a, grid, s);
    case 128: return launch_one<128, EPI_LOGITS>(tw, tx, a, grid, s);
    case 144: return launch_one<144, EPI_LOGITS>(tw, tx, a, grid, s);
    case 160: return launch_one<160, EPI_LOGITS>(tw, tx, a, grid, s);
    case 176: return launch_one<176, EPI_LOGITS>(tw, tx, a, grid, s);
    case 192: return launch_one<192, EPI_LOGITS>(tw, tx, a, grid, s);
    case 208: return launch_one<208, EPI_LOGITS>(tw, tx, a, grid, s);
    case 224: return launch_one<224, EPI_LOGITS>(tw, tx, a, grid, s);
    case 240: return launch_one<240, EPI_LOGITS>(tw, tx, a, grid, s);
    case 256: return launch_one<256, EPI_LOGITS>(tw, tx, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spec
