// Instantiations of the tcgen05 verify GEMM for the bf16 (+ residual) epilogue.
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

int linear_tc_smem_bytes(int BN) {
  switch (BN) {
    case 16: return LinearCfg<16>::SMEM_BYTES;
    case 32: return LinearCfg<32>::SMEM_BYTES;
    case 48: return LinearCfg<48>::SMEM_BYTES;
    case 64: return LinearCfg<64>::SMEM_BYTES;
    case 80: return LinearCfg<80>::SMEM_BYTES;
    case 96: return LinearCfg<96>::SMEM_BYTES;
    case 112: return LinearCfg<112>::SMEM_BYTES;
    case 128: return LinearCfg<128>::SMEM_BYTES;
    case 144: return LinearCfg<144>::SMEM_BYTES;
    case 160: return LinearCfg<160>::SMEM_BYTES;
    case 176: return LinearCfg<176>::SMEM_BYTES;
    case 192: return LinearCfg<192>::SMEM_BYTES;
    case 208: return LinearCfg<208>::SMEM_BYTES;
    case 224: return LinearCfg<224>::SMEM_BYTES;
    case 240: return LinearCfg<240>::SMEM_BYTES;
    case 256: return LinearCfg<256>::SMEM_BYTES;
    default: return -1;
  }
}

int linear_tc_tmem_cols(int BN) {
  switch (BN) {
    case 16: return LinearCfg<16>::TMEM_COLS;
    case 32: return LinearCfg<32>::TMEM_COLS;
    case 48: return LinearCfg<48>::TMEM_COLS;
    case 64: return LinearCfg<64>::TMEM_COLS;
    case 80: return LinearCfg<80>::TMEM_COLS;
    case 96: return LinearCfg<96>::TMEM_COLS;
    case 112: return LinearCfg<112>::TMEM_COLS;
    case 128: return LinearCfg<128>::TMEM_COLS;
    case 144: return LinearCfg<144>::TMEM_COLS;
    case 160: return LinearCfg<160>::TMEM_COLS;
    case 176: return LinearCfg<176>::TMEM_COLS;
    case 192: return LinearCfg<192>::TMEM_COLS;
    case 208: return LinearCfg<208>::TMEM_COLS;
    case 224: return LinearCfg<224>::TMEM_COLS;
    case 240: return LinearCfg<240>::TMEM_COLS;
    case 256: return LinearCfg<256>::TMEM_COLS;
    default: return -1;
  }
}

cudaError_t launch_linear_tc_bf16(int BN, const CUtensorMap& tw, const CUtensorMap& tx,
                                  const LinearArgs& a, dim3 grid, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_one<16, EPI_BF16>(tw, tx, a, grid, s);
    case 32: return launch_one<32, EPI_BF16>(tw, tx, a, grid, s);
    case 48: return launch_one<48, EPI_BF16>(tw, tx, a, grid, s);
    case 64: return launch_one<64, EPI_BF16>(tw, tx, a, grid, s);
    case 80: return launch_one<80, EPI_BF16>(tw, tx, a, grid, s);
    case 96: return launch_one<96, EPI_BF16>(tw, tx, a, grid, s);
    case 112: return launch_one<112, EPI_BF16>(tw, tx, a, grid, s);
    case 128: return launch_one<128, EPI_BF16>(tw, tx, a, grid, s);
    case 144: return launch_one<144, EPI_BF16>(tw, tx, a, grid, s);
    case 160: return launch_one<160, EPI_BF16>(tw, tx, a, grid, s);
    case 176: return launch_one<176, EPI_BF16>(tw, tx, a, grid, s);
    case 192: return launch_one<192, EPI_BF16>(tw, tx, a, grid, s);
    case 208: return launch_one<208, EPI_BF16>(tw, tx, a, grid, s);
    case 224: return launch_one<224, EPI_BF16>(tw, tx, a, grid, s);
    case 240: return launch_one<240, EPI_BF16>(tw, tx, a, grid, s);
    case 256: return launch_one<256, EPI_BF16>(tw, tx, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spec
