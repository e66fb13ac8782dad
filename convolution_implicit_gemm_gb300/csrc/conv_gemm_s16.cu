// conv_gemm_s16.cu -- the implicit-GEMM kernels whose epilogue holds only
// the 16-bit store path (conv_gemm_kernel.cuh, S16), in a translation unit
// of their own so that the two kernel sets compile in parallel.
#include "conv_gemm_kernel.cuh"

namespace igc {

cudaError_t launch_conv_gemm_s16(const ConvGemmParams& p, int block_n, int grid, cudaStream_t s) {
  return launch_block_n<true>(p, block_n, grid, s);
}

}  // namespace igc
