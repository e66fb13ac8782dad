// conv_gemm.cu -- launchers of the implicit-GEMM convolution kernel
// (conv_gemm_kernel.cuh): the kernels with every epilogue, the choice of
// epilogue groups and resident filter, and the CTA-pair capacity queries.
// The kernels with the 16-bit-store epilogue are compiled separately, in
// conv_gemm_s16.cu.
#include "conv_gemm_kernel.cuh"

namespace igc {

// Clusters of two that fit on the device at once (each CTA takes a whole SM).
template <int BN>
static int pair_capacity_bn() {
  static int cached = -1;
  if (cached >= 0) return cached;
  const int smem = Cfg<BN, true>::SMEM;
  if (cudaFuncSetAttribute(conv_gemm_kernel<BN, true, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, conv_gemm_kernel<BN, true, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cached = n;
  return n;
}

int conv_gemm_pair_capacity(int block_n) {
  switch (block_n) {
    case 64: return pair_capacity_bn<64>();
    case 128: return pair_capacity_bn<128>();
    case 256: return pair_capacity_bn<256>();
    default: return 0;
  }
}

size_t conv_gemm_smem_bytes(int block_n) {
  switch (block_n) {
    case 64: return Cfg<64>::SMEM;
    case 128: return Cfg<128>::SMEM;
    case 256: return Cfg<256>::SMEM;
    default: return 0;
  }
}

cudaError_t launch_conv_gemm(const ConvGemmParams& p_in, int block_n, int grid, cudaStream_t s) {
  // Two epilogue groups with four TMEM buffers: on 64-wide tiles, whose
  // four buffers of two issuers' accumulators fill the 512 TMEM columns,
  // two tiles' epilogues overlap (measured: strided 112x112 dgrad -13 %,
  // 56x56 64->64 3x3 dgrad -5 %, fprop -1.5 %, dilated dgrad -3 %, the
  // Winograd GEMM -8 %; bit-identical results).  epi_groups: 0 decide here
  // (two groups wherever they fit), 1 never, 2 wherever they fit.
  ConvGemmParams p = p_in;
  const bool fits = block_n == 64 && !p.pair && p.epi != EPI_PARTIAL && 4 * p.num_acc * 64 <= 512;
  p.epi_groups = (fits && p.epi_groups != 1) ? 2 : 1;
  // every unit of a conv plan has blocks unless a sub-problem has none (a
  // residue class no tap reaches)
  p.all_acc = p.epi != EPI_PARTIAL;
  for (int i = 0; i < p.nsub; ++i)
    if (p.sub[i].rcount * p.sub[i].scount * p.cblocks <= 0) p.all_acc = 0;
  // halo and one-issuer plans store 64-column boxes, whole tile rows per
  // warp: two groups always
  if (p.halo || (p.one_issuer && block_n == 64)) p.epi_groups = 2;
  // Resident filter (p.res_b set by the planner when allowed): 64-wide tiles
  // of a single column tile and one sub-problem, whole-tile units, the
  // filter a plain tiled operand, at most kResBlocks blocks per unit.
  const bool res_ok = block_n == 64 && !p.pair && p.nsub == 1 && p.tiles_n == 1 &&
                      p.grp_mul == 0 && p.epi != EPI_PARTIAL && p.a_src == SRC_IM2COL_K &&
                      (p.b_src == SRC_W_K || p.b_src == SRC_W_MN) &&
                      p.sub[0].rcount * p.sub[0].scount * p.cblocks <= kResBlocks;
  p.res_b = p.res_b && res_ok ? 1 : 0;
  // plain 16-bit stores (fprop, dgrad) take the kernels whose epilogue
  // holds only that path, unless the plan asks for the general ones
  const bool vol = p.a_src == SRC_IM2COL_K3 || p.wg_Do > 0;
  if (p.halo) {
    if (block_n != 64 || p.pair || p.epi != EPI_STORE || p.out_f32 || p.int_acc || vol)
      return cudaErrorInvalidValue;
    return launch_conv_gemm_halo(p, grid, s);
  }
  if (p.epi == EPI_STORE && !p.out_f32 && !p.int_acc && !vol && !p.general_epilogue)
    return launch_conv_gemm_s16(p, block_n, grid, s);
  return launch_block_n<false>(p, block_n, grid, s);
}

}  // namespace igc
