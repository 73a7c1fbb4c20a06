// Instantiations of the persistent tcgen05 verify GEMM with the SwiGLU epilogue: the weight
// rows come interleaved per 16 (gate block j, up block j), so every 128-row tile ends in
// silu(gate) * up for 64 output columns, computed on chip.
#include "internal.h"
#include "linear_tc_kernel.cuh"

namespace spec {

cudaError_t launch_linear_tc_swiglu(int BN, int NSUB, const CUtensorMap& tw, const CUtensorMap& tx,
                                  const LinearArgs& a, dim3 grid, cudaStream_t s) {
  switch (NSUB * 1000 + BN) {
    case 1016: return launch_linear_tc_one<16, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1032: return launch_linear_tc_one<32, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1048: return launch_linear_tc_one<48, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1064: return launch_linear_tc_one<64, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1080: return launch_linear_tc_one<80, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1096: return launch_linear_tc_one<96, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1112: return launch_linear_tc_one<112, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1128: return launch_linear_tc_one<128, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1144: return launch_linear_tc_one<144, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1160: return launch_linear_tc_one<160, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1176: return launch_linear_tc_one<176, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1192: return launch_linear_tc_one<192, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1208: return launch_linear_tc_one<208, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1224: return launch_linear_tc_one<224, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1240: return launch_linear_tc_one<240, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 1256: return launch_linear_tc_one<256, 1, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 2144: return launch_linear_tc_one<144, 2, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 2160: return launch_linear_tc_one<160, 2, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 2176: return launch_linear_tc_one<176, 2, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 2192: return launch_linear_tc_one<192, 2, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 2208: return launch_linear_tc_one<208, 2, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 2224: return launch_linear_tc_one<224, 2, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 2240: return launch_linear_tc_one<240, 2, EPI_SWIGLU>(tw, tx, a, grid, s);
    case 2256: return launch_linear_tc_one<256, 2, EPI_SWIGLU>(tw, tx, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spec
