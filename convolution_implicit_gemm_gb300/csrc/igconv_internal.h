// igconv_internal.h -- structures shared by the host planner (api.cpp) and
// the kernels (conv_gemm.cu, aux_kernels.cu).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace igc {

// GEMM tiling shared by every pass: 128 rows per CTA tile (one TMEM lane per
// row), 64-element (128-byte) reduction blocks matching the 128-byte swizzle.
constexpr int kBlockM = 128;
constexpr int kBlockK = 64;
constexpr int kBiasCacheBytes = 2048;  // bias vectors up to this size are staged in shared memory
constexpr int kHaloTaps = 9;           // halo plans: filter taps kept resident in shared memory
constexpr int kHaloRows = 320;         // halo plans: pixel rows of 128 bytes per halo stage
constexpr int kMaxSub = 16;      // dgrad stride decomposition: stride_h * stride_w <= 16
constexpr int kThreads = 512;    // warps 0-3 TMA producers, 4-11 epilogue, 12-13 MMA issuers

// Where an operand tile comes from, and its shared-memory major-ness.
enum SrcKind : int {
  SRC_IM2COL_K = 0,   // one im2col load: 128 pixels x 64 channels, K-major
  SRC_W_K = 1,        // one tiled load of the filter, box {64 c, 1, 1, BN k}, K-major
  SRC_W_MN = 2,       // BN/64 tiled loads of the filter, box {64 c, 1, 1, 64 k}, MN-major
  SRC_IM2COL_MN = 3,  // rows/64 im2col loads of 64 pixels x 64 channels, MN-major
  SRC_2D_MN = 4,      // rows/64 tiled loads of a [rows][ld] matrix, box {64, 64}, MN-major
  // few channels (C <= 8, pixels padded to 8 channels): a reduction block is
  // 8 filter taps x 8 channels, stored without swizzle as 8 regions of
  // [rows][16 bytes], one per tap
  SRC_IM2COL_TAPS = 5,  // eight im2col loads of 128 pixels x 8 channels
  SRC_W_TAPS = 6,       // one contiguous copy of the block's filter image (taps_filter)
  // 3D fprop / stride-1 dgrad: one 5D im2col load of 128 output positions
  // x 64 channels (NDHWC, taps (t, r, s)), K-major; the filter is read as
  // [K][T*R][S][C] (SRC_W_K for fprop, SRC_W_MN with flipped taps for dgrad)
  SRC_IM2COL_K3 = 7,
  // few channels in wgrad (C <= 8, pixels padded to 8 channels): a 64-row
  // chunk of the X side is 8 filter taps x 8 channels, eight im2col loads of
  // 64 positions x 16 bytes stored without swizzle, MN-major: tap t of the
  // chunk at 1 KB * t, positions at 16 bytes (8-position groups 128 B apart)
  SRC_IM2COL_TAPS_MN = 8,
};

enum EpiKind : int {
  EPI_STORE = 0,    // 16-bit output: cast(relu?(alpha*acc + beta*Cin + bias))
  EPI_PARTIAL = 1,  // fp32 split-K partial tile into the workspace
  EPI_INT8 = 2,     // int8 output: exact requantisation of the integer accumulator
};

enum DeviceErr : unsigned int {
  DEVERR_NONE = 0,
  DEVERR_PRODUCER_WAIT = 1,
  DEVERR_MMA_FULL_WAIT = 2,
  DEVERR_MMA_TMEM_WAIT = 3,
  DEVERR_EPI_WAIT = 4,
  DEVERR_TEARDOWN_WAIT = 5,
  DEVERR_SELFTEST = 6,
  DEVERR_SMEM_LAYOUT = 7,
};

// One implicit GEMM over a set of output pixels that share a tap list.
// fprop has one; strided dgrad has one per output residue class.
struct SubProblem {
  int M;                  // GEMM rows (output pixels) of this sub-problem
  int tile_begin;         // first work-unit index
  int tiles_m;
  int Hs, Ws;             // traversal grid per image: M = N * Hs * Ws
  int lower_h, lower_w;   // input coordinate of grid index 0 (im2col box lower corner)
  int trav_h, trav_w;     // traversal strides
  int r0, rstep, rcount, offh0, doffh;  // tap j: filter row r0 + j*rstep, im2col offset offh0 + j*doffh
  int s0, sstep, scount, offw0, doffw;
  int out_h0, out_w0, out_sh, out_sw;   // epilogue: output row = out_h0 + out_sh * grid row
  int ws_valid;           // 0: every grid column is an output; else grid columns >= ws_valid
                          // pad the row to Ws (their results are dropped)
  // 3D (Ds > 0): traversal depth, its lower corner and stride.  The r taps
  // run over the merged index jt * rdiv + jr (rcount = depth taps * rdiv):
  // filter row coordinate r0 + jt * tstride + jr * rstep of the [K][T*R]
  // view, depth im2col offset offd0 + jt * doffd; output depth out_d0 +
  // out_sd * grid depth
  int Ds, lower_d, trav_d, rdiv, doffd, tstride, offd0, out_d0, out_sd;
};

struct ConvGemmParams {
  CUtensorMap mapA[kMaxSub];  // operand maps (im2col of X or dY; wgrad: mapA[0] = im2col of X)
  CUtensorMap mapB;           // filter map (fprop/dgrad) or dY 2D map (wgrad)
  CUtensorMap mapY;           // output map for TMA stores (when use_tma_store)
  SubProblem sub[kMaxSub];
  uint32_t mapA_valid;        // bit i: mapA[i] holds an encoded map
  int use_tma_store;          // output tile rows are contiguous: store them with TMA
  int general_epilogue;       // 1: 16-bit store plans run on the kernels with every epilogue
  int halo;                   // 1: halo plan (conv_gemm_halo_kernel): mapA[0] is a tiled map of
                              // the input, box (64 channels, Ws pixels, halo rows, 1); sub[0]
                              // is the stride-1 plan on a grid Ws = 32/64/128 columns wide
  int halo_bytes;             // bytes one halo copy lands (the whole box; wgrad: one channel
                              // plane of it)
  int wh_stage_bytes;         // wgrad halo plans: bytes per pipeline stage (the input planes
                              // and the dY chunks of one block), and the stage count
  int wh_stages;
  int all_acc;                // set by the launcher: every unit has reduction blocks
  int one_issuer;             // halo plans: the two MMA issuers take alternate units whole,
                              // each into the unit's one accumulator (num_acc = 1)
  int store_5d;               // strided dgrad: mapY is dX viewed as (c, w % sw, w / sw, h % sh,
                              // n * H / sh + h / sh), a residue class's grid row is one
                              // (h % sh, row) line and each 32-row box lies inside one
  int store_box64;            // mapY boxes are 64 columns wide (128-byte swizzle)
  int nsub;
  int pair;                   // 1: clusters of two CTAs, 256-row units, cta_group::2 MMAs
  int res_b;                  // 1: the filter may stay resident in shared memory (the launcher
                              // keeps it only where a 64-wide single-column plan allows)
  int raster;                 // tile order of fprop / dgrad units: <= 1 column tiles fastest;
                              // g > 1 runs of g row tiles, rows fastest within a column
  int a_src, b_src;           // SrcKind
  int epi;                    // EpiKind
  int units;                  // work units = tiles (x splits for wgrad)
  int tiles_m_total;          // wgrad: tiles along M
  int tiles_n;
  int splits;                 // wgrad split-K factor (1 otherwise)
  int kblocks_total;          // wgrad: ceil(N*P*Q / 64)
  int cblocks;                // 64-channel blocks per tap (reduction channels; wgrad: X channels)
  int grp_mul, grp_div;       // grouped block-diagonal GEMM (grp_mul != 0, BN = 64): 64-wide
                              // tile n holds whole groups and reduces over the channel
                              // window starting at (n / grp_div) * grp_mul (a multiple of 8)
                              // of the im2col operand (X in fprop and wgrad, dY in dgrad)
                              // and of the dense block-diagonal filter [K][R][S][C]
  int N_gemm;                 // valid GEMM columns
  uint32_t idesc;             // tcgen05 instruction descriptor
  int num_acc;                // TMEM accumulators per tile (issuers x groups)
  int kb_per_acc;             // reduction blocks per accumulator, per issuer
  // wgrad: output-position grid and taps of the X-side im2col operand
  int wg_PQ, wg_Q;
  int wg_lower_h, wg_lower_w, wg_sh, wg_sw;
  int wg_S, wg_RS, wg_dh, wg_dw;
  int wg_K;                   // output channels (extent of the dY side)
  int wg_Do, wg_lower_d, wg_sd, wg_dd, wg_R;  // 3D (wg_Do > 0): depth grid, taps (t, r, s)
  // epilogue
  void* out;
  const void* cin;
  const void* taps_filter;    // SRC_W_TAPS: [block][tile_n][8 taps][BN][8 channels] image
  const void* pf_base;         // filter, fetched into L2 at kernel start (pf_bytes > 0)
  long long pf_bytes;
  const void* bias;
  int bias_cached;        // 1: the kernel copies the bias vector into shared memory
  float alpha, beta;
  int relu;
  int out_bf16;               // 16-bit output: 0 fp16, 1 bf16
  int out_C;                  // elements per output pixel row
  int out_H, out_W;           // output image extent (dgrad); P, Q for fprop
  int out_D;                  // 3D: output depth extent
  long long ws_split_stride;  // wgrad: floats per split in the workspace
  int ws_ld;                  // wgrad: padded N extent
  uint32_t rq_mant;           // int8: multiplier M = rq_mant * 2^rq_exp exactly
  int rq_exp;
  int epi_groups;             // epilogue warp groups: 0 or 2 two groups of four taking
                              // alternate tiles whole (four TMEM buffers) where they fit,
                              // 1 one group of eight warps per tile (two buffers)
  int conv_split;             // 1 with EPI_PARTIAL: split-K over a convolution (fprop or
                              // stride-1 dgrad): conv operand loads, fp32 partial tiles
  int out_f32;                // 1 with EPI_STORE: write alpha * acc as fp32 (no bias, beta
                              // or cast; a later kernel finishes the output)
  int int_acc;                // 1: the accumulators hold exact integers (int8 operands on the
                              // fp16 path); EPI_STORE writes their int32 sum, EPI_PARTIAL
                              // int32 partial sums (int8 dgrad / wgrad)
  unsigned int* status;       // device status word
  unsigned long long timeout_ns;
};

// Launches the persistent implicit-GEMM kernel with tile width block_n.
cudaError_t launch_conv_gemm(const ConvGemmParams& p, int block_n, int grid, cudaStream_t s);
// The same launch on the kernels whose epilogue holds only the 16-bit store
// path (a plan with EPI_STORE, 16-bit outputs and no 3D operands).
cudaError_t launch_conv_gemm_s16(const ConvGemmParams& p, int block_n, int grid, cudaStream_t s);
// The halo kernel (a plan with p.halo set: 64-wide tiles, 16-bit stores).
cudaError_t launch_conv_gemm_halo(const ConvGemmParams& p, int grid, cudaStream_t s);
// The wgrad halo kernel (conv_wgrad_halo.cu): p.splits CTAs, each one unit of
// p.kblocks_total 128-position blocks; partial tiles to p.out (see there).
cudaError_t launch_wgrad_halo(const ConvGemmParams& p, cudaStream_t s);
// Clusters of two CTAs of the kernel with this tile width that fit at once.
int conv_gemm_pair_capacity(int block_n);
size_t conv_gemm_smem_bytes(int block_n);

// Few-channel packing (C <= 8, dilation 1).  X is copied once to a padded
// space-to-depth image Zp[N][Hz][Wz][cz]: packed pixel (i, j) holds the
// fh x fw input pixels (fh*(i + A0) + dy, fw*(j + B0) + dx), channel
// e = (dy * fw + dx) * C + c, zero past fh*fw*C channels and outside the
// input (fh, fw = the strides; cz = 8, 16, 32 or 64).  An im2col map whose
// pixel stride is one packed pixel (cz * 2 bytes) but whose channel box is
// 64 elements then reads ppr = 64 / cz consecutive packed pixels as one
// 128-byte row, so the convolution is a stride-1 one over 64 "channels"
// with R2 x Sv taps, the Sv taps along w ppr packed pixels apart.  Virtual
// channel ev of virtual tap vt = r2 * Sv + sv is packed pixel jp = ev / cz of
// the window, channel ev % cz; few_pack_decode maps it back to the filter
// tap (r * S + s) and channel it multiplies, or reports a zero slot.
struct FewPack {
  int fh, fw;      // space-to-depth factors (the strides)
  int C, R, S;     // the real problem's channels and filter
  int ph, pw;      // its padding
  int cz, ppr;     // channels per packed pixel; packed pixels per 128-byte row
  int A0, B0;      // packed-row / -column offset of virtual tap 0: floor(-pad / f)
  int R2, Sv;      // virtual taps along h and along w
  int Hz, Wz, Wv;  // packed rows, packed columns, window starts along w
};

__host__ __device__ inline bool few_pack_decode(const FewPack& f, int vt, int ev, int* tap,
                                                int* c) {
  const int r2 = vt / f.Sv;
  const int sv = vt - r2 * f.Sv;
  const int jp = ev / f.cz;
  const int e = ev - jp * f.cz;
  const int fwc = f.fw * f.C;
  if (e >= f.fh * fwc) return false;
  const int dy = e / fwc;
  const int rem = e - dy * fwc;
  const int dx = rem / f.C;
  const int r = f.fh * (r2 + f.A0) + dy + f.ph;
  const int s = f.fw * (sv * f.ppr + jp + f.B0) + dx + f.pw;
  if (r < 0 || r >= f.R || s < 0 || s >= f.S) return false;
  *tap = r * f.S + s;
  *c = rem - dx * f.C;
  return true;
}

#ifdef __CUDACC__
// round_half_even(t * M) clamped to int8 without branches, for M = mant *
// 2^-sh and |t| < 2^33.  For 1 <= sh <= 62: with x = t * mant (exact in 64
// bits) and b the lowest bit of floor(x / 2^sh), the quotient
// floor((x + b + 2^(sh-1) - 1) / 2^sh) rounds x / 2^sh to nearest with ties to
// the even neighbour (an arithmetic shift is the floor, also for negative x).
// sh <= 0 means M >= 2^23, so every t != 0 saturates; sh >= 63 means M <
// 2^-39, so |t * M| < 1/2 rounds to 0.  The caller passes sh clamped to
// 1..62 and the mode of the true shift (0 in range, 1 saturate, 2 zero).
__device__ __forceinline__ int requant_rne(long long t, uint32_t mant, int sh,
                                          long long half_m1, int mode) {
  const long long x = t * static_cast<long long>(mant);
  const long long b = (x >> sh) & 1LL;
  long long q = (x + b + half_m1) >> sh;
  if (mode == 1) q = t > 0 ? 127 : (t < 0 ? -128 : 0);
  if (mode == 2) q = 0;
  q = q > 127 ? 127 : q;
  q = q < -128 ? -128 : q;
  return static_cast<int>(q);
}
#endif

// Whether the implicit-GEMM kernels and the split reductions launch with
// programmatic dependent launch (tuning knob IGCONV_TUNE_PDL = 1; off by
// default).  Defined in api.cpp.
bool pdl_enabled();

#ifdef __CUDACC__
// Launches kernel k on stream s in clusters of cluster_x CTAs (1: none).
// With programmatic dependent launch enabled, k may begin launching while
// the kernel before it in the stream finishes; every kernel launched here
// calls pdl_wait() before its first global memory access, so the stream's
// order of memory effects is kept.
template <typename... Params, typename... Args>
cudaError_t launch_hot(void (*k)(Params...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t s, unsigned cluster_x, Args&&... args) {
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, k, static_cast<Args&&>(args)...);
}
#endif

// Auxiliary kernels (aux_kernels.cu).
cudaError_t launch_batched_transpose(const void* src, void* dst, long long batch, long long rows,
                                     long long cols, int elem_bytes, cudaStream_t s);
// rows / columns of the partials are (tap, c) with c < cpad, or, when
// remap is given, few-channel virtual rows (vt * 64 + ev) decoded by
// few_pack_decode
cudaError_t launch_wgrad_reduce(const float* ws, int splits, long long split_stride, int ws_ld,
                                int rows, int cols, int swapped, int K, int RS, int C, int cpad,
                                void* dW, int dw_dtype, const void* cin, float alpha, float beta,
                                cudaStream_t s, const FewPack* remap = nullptr);
// int8 fprop split-K: y[m][k] = requant(relu(sum_s ws[s][m][k] + bias[k]))
// with the int32 partials added modulo 2^32 in split order.
cudaError_t launch_conv_splitk_reduce_i8(const int* ws, int splits, long long split_stride,
                                         int ws_ld, long long rows, int cols, int8_t* out,
                                         const int32_t* bias, uint32_t rq_mant, int rq_exp,
                                         int relu, cudaStream_t s);
cudaError_t launch_conv_splitk_reduce(const float* ws, int splits, long long split_stride,
                                      int ws_ld, long long rows, int cols, void* out,
                                      int out_bf16, const void* cin, const void* bias,
                                      float alpha, float beta, int relu, cudaStream_t s);
cudaError_t launch_unpad_channels(const float* src8, void* dst, long long pixels, int C,
                                  int out_bf16, const void* cin, float beta, cudaStream_t s);
cudaError_t launch_wgrad_reduce_i32(const int* ws, int splits, long long split_stride, int ws_ld,
                                    int rows, int cols, int swapped, int K, int RS, int C,
                                    int cpad, int* dW, cudaStream_t s);
cudaError_t launch_i8_to_f16(const int8_t* src, void* dst, long long count, cudaStream_t s);
cudaError_t launch_pad_pixels8(const void* src, void* dst, long long pixels, int C,
                               cudaStream_t s);
cudaError_t launch_filter_taps8(const void* w, void* dst, int K, int RS, int C, int bn,
                                cudaStream_t s);
cudaError_t launch_few_pack_x(const void* X, void* Zp, const FewPack& f, int N, int H, int W,
                              cudaStream_t s);
cudaError_t launch_few_pack_filter(const void* Wt, void* Wpk, const FewPack& f, int K, int row,
                                   cudaStream_t s);
cudaError_t launch_few_unpack_dx(const float* dz, void* dX, const FewPack& f, int N, int H, int W,
                                 int out_bf16, const void* cin, float beta, cudaStream_t s);
cudaError_t launch_group_filter_dense(const void* w, void* dst, int K, int RS, int C, int cg,
                                      int kg, cudaStream_t s);
cudaError_t launch_group_extract(const float* src, void* dW, int dw_dtype, const void* cin,
                                 float beta, int K, int RS, int cg, int kg, int cpad, int mul,
                                 int div, cudaStream_t s);
cudaError_t launch_wino_input(const void* X, void* V, int N, int H, int W, int C, int TH, int TW,
                              int ph, int pw, int bf16, cudaStream_t s);
cudaError_t launch_wino_filter(const void* Wt, void* U, int K, int C, int bf16, cudaStream_t s);
cudaError_t launch_wino_output(const void* Mx, void* Y, const void* cin, const void* bias, int N,
                               int P, int Q, int K, int TH, int TW, float alpha, float beta,
                               int relu, int bf16, cudaStream_t s);
cudaError_t launch_selftest_wait(unsigned int* status, unsigned long long timeout_ns,
                                 cudaStream_t s);
cudaError_t status_word_address(unsigned int** ptr);

}  // namespace igc
