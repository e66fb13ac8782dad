// conv_gemm_s16.cu -- the implicit-GEMM kernels whose epilogue holds only
// the 16-bit store path (conv_gemm_kernel.cuh, S16) and the halo kernel, in
// a translation unit of their own so that the two kernel sets compile in
// parallel.
#include "conv_gemm_kernel.cuh"

namespace igc {

cudaError_t launch_conv_gemm_s16(const ConvGemmParams& p, int block_n, int grid, cudaStream_t s) {
  return launch_block_n<true>(p, block_n, grid, s);
}

cudaError_t launch_conv_gemm_halo(const ConvGemmParams& p, int grid, cudaStream_t s) {
  auto* k = conv_gemm_halo_kernel<64>;
  cudaError_t e = check_launch_regs(reinterpret_cast<const void*>(k));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, HaloCfg::SMEM);
  if (e != cudaSuccess) return e;
  return launch_hot(k, static_cast<unsigned>(grid), kThreads, static_cast<size_t>(HaloCfg::SMEM),
                    s, 1, p);
}

}  // namespace igc
