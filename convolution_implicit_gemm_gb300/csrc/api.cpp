// api.cpp -- the C ABI of libigconv: validation, problem planning (GEMM
// views, tile and split choice, the dgrad residue-class decomposition),
// TMA tensor-map encoding and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <climits>
#include <cstring>
#include <mutex>

#include "igconv.h"
#include "depthwise_internal.h"
#include "igconv_internal.h"

using namespace igc;

namespace {

// ---------------------------------------------------------------------------
// Per-process / per-device state
// ---------------------------------------------------------------------------
typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*PFN_encodeIm2col)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                     const cuuint64_t*, const cuuint64_t*, const int*,
                                     const int*, cuuint32_t, cuuint32_t, const cuuint32_t*,
                                     CUtensorMapInterleave, CUtensorMapSwizzle,
                                     CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;
constexpr unsigned long long kTimeoutNs = 2000000000ull;  // 2 s per pipeline wait

struct DeviceState {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  unsigned int* status = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_encodeTiled g_encode_tiled = nullptr;
PFN_encodeIm2col g_encode_im2col = nullptr;
std::atomic<int> g_tune_splits{0}, g_tune_bn{0}, g_tune_max_ctas{0}, g_tune_no_pairs{0},
    g_tune_epi_groups{0}, g_tune_conv_splits{0}, g_tune_few_channels{0}, g_tune_raster{0},
    g_tune_resident_b{0}, g_tune_dgrad_rows{0}, g_tune_general_epi{0}, g_tune_halo{0},
    g_tune_one_issuer{0}, g_tune_wgrad_halo{0}, g_tune_pdl{0};

// A failed runtime call (a launch, an attribute, a copy) is reported as
// IGCONV_ERR_CUDA, and the runtime's last-error state it set is consumed
// here, so that a later call does not find it and report a second failure
// (a sticky error stays: the runtime keeps those).
igconv_status_t cuda_error() {
  (void)cudaGetLastError();
  return IGCONV_ERR_CUDA;
}

igconv_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? IGCONV_OK : cuda_error(); }

igconv_status_t device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cuda_error();
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cuda_error();
    st.supported = (major == 10 && minor == 3);  // kernels are built for sm_103a only
    if (status_word_address(&st.status) != cudaSuccess) return cuda_error();
    if (!g_encode_tiled || !g_encode_im2col) {
      cudaDriverEntryPointQueryResult q1, q2;
      void* f1 = nullptr;
      void* f2 = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f1, 12000,
                                           cudaEnableDefault, &q1) != cudaSuccess ||
          q1 != cudaDriverEntryPointSuccess ||
          cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &f2, 12000,
                                           cudaEnableDefault, &q2) != cudaSuccess ||
          q2 != cudaDriverEntryPointSuccess)
        return cuda_error();
      g_encode_tiled = reinterpret_cast<PFN_encodeTiled>(f1);
      g_encode_im2col = reinterpret_cast<PFN_encodeIm2col>(f2);
    }
    st.ready = true;
  }
  if (!st.supported) return IGCONV_ERR_UNSUPPORTED;
  *out = &st;
  return IGCONV_OK;
}


bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------
// Validation
// ---------------------------------------------------------------------------
long long out_extent(long long in, long long pad, long long dil, long long k, long long stride) {
  const long long span = in + 2 * pad - dil * (k - 1) - 1;
  if (span < 0) return 0;
  return span / stride + 1;
}

igconv_status_t check_shape(const igconv_problem_t* pb, int* P, int* Q) {
  if (!pb) return IGCONV_ERR_INVALID_ARG;
  if (pb->N < 1 || pb->H < 1 || pb->W < 1 || pb->C < 1 || pb->K < 1 || pb->R < 1 || pb->S < 1)
    return IGCONV_ERR_INVALID_ARG;
  if (pb->pad_h < 0 || pb->pad_w < 0 || pb->stride_h < 1 || pb->stride_w < 1 || pb->dil_h < 1 ||
      pb->dil_w < 1)
    return IGCONV_ERR_INVALID_ARG;
  const long long p = out_extent(pb->H, pb->pad_h, pb->dil_h, pb->R, pb->stride_h);
  const long long q = out_extent(pb->W, pb->pad_w, pb->dil_w, pb->S, pb->stride_w);
  if (p < 1 || q < 1 || p > INT32_MAX || q > INT32_MAX) return IGCONV_ERR_INVALID_ARG;
  if (P) *P = static_cast<int>(p);
  if (Q) *Q = static_cast<int>(q);
  return IGCONV_OK;
}

// Limits of the kernels (valid problems outside them are UNSUPPORTED).
igconv_status_t check_limits(const igconv_problem_t* pb, int P, int Q, int channel_multiple) {
  if (pb->C % channel_multiple != 0 || pb->K % channel_multiple != 0)
    return IGCONV_ERR_UNSUPPORTED;
  if (pb->stride_h > 8 || pb->stride_w > 8) return IGCONV_ERR_UNSUPPORTED;
  if (pb->pad_h > 64 || pb->pad_w > 64 || pb->R > 64 || pb->S > 64) return IGCONV_ERR_UNSUPPORTED;
  if (static_cast<long long>(pb->R - 1) * pb->dil_h > 127 ||
      static_cast<long long>(pb->S - 1) * pb->dil_w > 127)
    return IGCONV_ERR_UNSUPPORTED;
  if (pb->N > 65535) return IGCONV_ERR_UNSUPPORTED;
  const long long in_pix = static_cast<long long>(pb->N) * pb->H * pb->W;
  const long long out_pix = static_cast<long long>(pb->N) * P * Q;
  if (in_pix >= (1LL << 31) || out_pix >= (1LL << 31)) return IGCONV_ERR_UNSUPPORTED;
  if (in_pix * pb->C >= (1LL << 40) || out_pix * pb->K >= (1LL << 40)) return IGCONV_ERR_UNSUPPORTED;
  return IGCONV_OK;
}

// ---------------------------------------------------------------------------
// Tensor maps
// ---------------------------------------------------------------------------
CUtensorMapDataType tma_dtype(int bf16) {
  return bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// im2col map over an NHWC 16-bit tensor [n][h][w][c]: `pixels` output
// positions x 64 channels per load, 128-byte swizzle.  The box corners and
// traversal strides describe the grid of filter-origin positions: the
// traversal visits lower .. (extent - 1 + upper) in steps of trav.
// x_strides (bytes between pixels, rows and images) replaces the dense NHWC
// strides when given: the few-channel packed image is read with a pixel
// stride smaller than the 64-channel box, so consecutive boxes overlap.
bool encode_im2col(CUtensorMap* map, const void* base, int bf16, int n, int h, int w, int c,
                   int lower_h, int lower_w, int upper_h, int upper_w, int trav_h, int trav_w,
                   int pixels, int channels_box = 64,
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
                   const cuuint64_t* x_strides = nullptr) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(c), static_cast<cuuint64_t>(w),
                              static_cast<cuuint64_t>(h), static_cast<cuuint64_t>(n)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(c) * 2, static_cast<cuuint64_t>(c) * 2 * w,
                           static_cast<cuuint64_t>(c) * 2 * w * h};
  if (x_strides) {
    strides[0] = x_strides[0];
    strides[1] = x_strides[1];
    strides[2] = x_strides[2];
  }
  const int lower[2] = {lower_w, lower_h};
  const int upper[2] = {upper_w, upper_h};
  const cuuint32_t estr[4] = {1, static_cast<cuuint32_t>(trav_w), static_cast<cuuint32_t>(trav_h),
                              1};
  const CUresult r = g_encode_im2col(
      map, tma_dtype(bf16), 4, const_cast<void*>(base), dims, strides, lower, upper,
      static_cast<cuuint32_t>(channels_box), static_cast<cuuint32_t>(pixels), estr,
      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tiled map over the KRSC filter viewed as 4D (c, s, r, k), box {64, 1, 1, box_k}.
bool encode_filter(CUtensorMap* map, const void* base, int bf16, int K, int R, int S, int C,
                   int box_k) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(R), static_cast<cuuint64_t>(K)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(C) * 2,
                                 static_cast<cuuint64_t>(C) * 2 * S,
                                 static_cast<cuuint64_t>(C) * 2 * S * R};
  const cuuint32_t box[4] = {64, 1, 1, static_cast<cuuint32_t>(box_k)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode_tiled(map, tma_dtype(bf16), 4, const_cast<void*>(base), dims,
                                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tiled map over a [rows][cols] 16-bit matrix, box {64, 64}.
bool encode_2d(CUtensorMap* map, const void* base, int bf16, long long rows, long long cols) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode_tiled(map, tma_dtype(bf16), 2, const_cast<void*>(base), dims,
                                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tiled map over a row-major [rows][cols] output for TMA stores of 32-row
// boxes of box_cols columns (the epilogue stages them in the given swizzle).
bool encode_out_2d(CUtensorMap* map, void* base, CUtensorMapDataType dt, int esize,
                   long long rows, long long cols, int box_cols, CUtensorMapSwizzle sw) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * esize};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode_tiled(map, dt, 2, base, dims, strides, box, estr,
                                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                                    CU_TENSOR_MAP_L2_PROMOTION_NONE,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 64-wide 16-bit-store plans whose units hold at most four reduction blocks
// (1x1 layers over up to 256 channels, the packed stem, strided dgrad's
// residue classes) are bound by their epilogue: there the two MMA issuers
// take alternate units whole, each into the unit's one accumulator
// (num_acc = 1), so the epilogue reads one accumulator and stores 64-column
// boxes (see run_mma).  Call before the output map is encoded; knob
// IGCONV_TUNE_ONE_ISSUER = 1 keeps two accumulators per unit.
void choose_one_issuer(ConvGemmParams& p, int bn) {
  if (g_tune_one_issuer.load() == 1 || bn != 64 || p.pair || p.halo) return;
  int kb = 0;
  for (int i = 0; i < p.nsub; ++i)
    kb = std::max(kb, p.sub[i].rcount * p.sub[i].scount * p.cblocks);
  if (kb < 1 || kb > 4) return;
  p.one_issuer = 1;
  p.num_acc = 1;
}

// Output map for a 16-bit [rows x cols] output written by TMA stores.  Boxes
// are 32 rows x 32 columns, double-buffered per epilogue warp; a GEMM whose
// reduction is at most two blocks per tile is bound by its epilogue, and
// there boxes of 32 x 64 (128-byte swizzle, one per two chunks) halve the
// store, fence and sync count per tile (measured: 1x1 conv 64 -> 256
// channels 87 -> 80 us), while on longer reductions the single 4 KB staging
// buffer they allow costs a few percent.
void set_out_map_16(ConvGemmParams& p, void* base, long long rows, long long cols, int bf16,
                    int bn, int kblocks_per_tile) {
  // (one accumulator per 64-wide unit: two chunks per 64-column box)
  const bool wide = (bn >= 128 && kblocks_per_tile <= 2) || p.one_issuer;
  p.use_tma_store = encode_out_2d(&p.mapY, base, tma_dtype(bf16), 2, rows, cols, wide ? 64 : 32,
                                  wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B)
                        ? 1
                        : 0;
  p.store_box64 = wide ? p.use_tma_store : 0;
}

// Output map for plans whose grid rows are whole output-row lines: the
// output [N][H][W][C] viewed as (c, w % sw, w / sw, h % sh, n * H/sh + h/sh)
// (H and W multiples of sh and sw), boxes of 32 grid columns of one line,
// the box width and staging swizzle chosen as in set_out_map_16.  Used by the
// strided dgrad's residue classes on one padded grid (padded_class_width)
// and by halo plans (sh = sw = 1).
void set_out_map_lines_5d(ConvGemmParams& p, void* out, int N, int H, int W, int C, int sh,
                          int sw, int bf16, int bn, int kblocks_per_tile) {
  // halo plans store 64-column boxes (one accumulator: two chunks per box)
  const bool wide = (bn >= 128 && kblocks_per_tile <= 2) || p.one_issuer;
  const cuuint64_t px = static_cast<cuuint64_t>(C) * 2;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(sw),
                              static_cast<cuuint64_t>(W / sw), static_cast<cuuint64_t>(sh),
                              static_cast<cuuint64_t>(N) * (H / sh)};
  const cuuint64_t strides[4] = {px, px * sw, px * W, px * W * sh};
  const cuuint32_t box[5] = {wide ? 64u : 32u, 1, 32, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = g_encode_tiled(&p.mapY, tma_dtype(bf16), 5, out, dims, strides, box, estr,
                                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                                    wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                                    CU_TENSOR_MAP_L2_PROMOTION_NONE,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  p.use_tma_store = r == CUDA_SUCCESS ? 1 : 0;
  p.store_box64 = wide ? p.use_tma_store : 0;
  p.store_5d = p.use_tma_store;  // otherwise the padded rows stay valid through the row stores
}

// Halo plan (conv_gemm_kernel.cuh, "Halo tiles") for the stride-1 plan in p
// (fprop over X, or stride-1 dgrad over dY: one sub-problem, 64-wide tiles,
// one column tile, one 64-channel reduction block, 2..kHaloTaps taps with
// non-negative offsets) over the input in [N][Hin][Win][Cin] with an output
// of Hout x Wout pixels.  The grid width Wt is the smallest of 32, 64, 128
// that holds a padded input row (Wout + the largest column offset), so a
// 128-row tile is 128 / Wt whole output rows, and needs Hout to be a multiple
// of that; the halo of HR = 128 / Wt + the largest row offset + 1 rows of Wt
// pixels must fit kHaloRows.  Rewrites p (input map, grid, units) and
// returns true when the plan qualifies and IGCONV_TUNE_HALO allows it.
bool try_halo_plan(ConvGemmParams& p, int bn, const void* in, int N, int Hin, int Win, int Cin,
                   int Hout, int Wout, int bf16) {
  if (g_tune_halo.load() == 1) return false;  // 0 built-in, 1 never
  const SubProblem& sp = p.sub[0];
  if (bn != 64 || p.pair || p.conv_split || p.nsub != 1 || p.tiles_n != 1 || p.cblocks != 1 ||
      p.grp_mul != 0 || p.a_src != SRC_IM2COL_K ||
      (p.b_src != SRC_W_K && p.b_src != SRC_W_MN) || sp.trav_h != 1 || sp.trav_w != 1 ||
      sp.Ds > 0 || sp.tile_begin != 0)
    return false;
  const int taps = sp.rcount * sp.scount;
  if (taps < 2 || taps > kHaloTaps) return false;
  const int oh1 = sp.offh0 + (sp.rcount - 1) * sp.doffh;
  const int ow1 = sp.offw0 + (sp.scount - 1) * sp.doffw;
  if (std::min(sp.offh0, oh1) < 0 || std::min(sp.offw0, ow1) < 0) return false;
  const int max_h = std::max(sp.offh0, oh1), max_w = std::max(sp.offw0, ow1);
  int wt = 32;
  while (wt < Wout + max_w && wt < 256) wt *= 2;
  if (wt > 128 || wt < Wout + max_w) return false;
  const int rows = kBlockM / wt;
  const int hr = rows + max_h + 1;
  if (hr * wt > kHaloRows || hr > 256 || Hout % rows != 0) return false;
  const long long M = static_cast<long long>(N) * Hout * wt;
  if (M > INT_MAX) return false;
  // the input, box (64 channels, wt pixels, hr rows, one image); padding
  // and the columns past the image read as zero
  CUtensorMap map;
  const cuuint64_t px = static_cast<cuuint64_t>(Cin) * 2;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(Cin), static_cast<cuuint64_t>(Win),
                              static_cast<cuuint64_t>(Hin), static_cast<cuuint64_t>(N)};
  const cuuint64_t strides[3] = {px, px * Win, px * Win * Hin};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(wt), static_cast<cuuint32_t>(hr), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  if (g_encode_tiled(&map, tma_dtype(bf16), 4, const_cast<void*>(in), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  p.mapA[0] = map;
  p.mapA_valid = 1u;
  SubProblem& s = p.sub[0];
  s.M = static_cast<int>(M);
  s.tiles_m = static_cast<int>(M / kBlockM);
  s.Ws = wt;
  s.ws_valid = Wout;
  p.units = s.tiles_m;
  p.halo = 1;
  p.halo_bytes = hr * wt * 128;
  p.one_issuer = 1;
  p.num_acc = 1;
  p.res_b = 0;
  return true;
}

// tcgen05 instruction descriptor, kind::f16 with an fp32 accumulator:
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format (0 f16, 1 bf16),
//   15 A MN-major, 16 B MN-major, 17-22 N >> 3, 24-28 M >> 4.
uint32_t make_idesc(int M, int N, int bf16, int a_mn, int b_mn) {
  return (1u << 4) | (static_cast<uint32_t>(bf16) << 7) | (static_cast<uint32_t>(bf16) << 10) |
         (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Relative per-column throughput of a tile width (measured on GB300: a
// 256-wide tile keeps one MMA issuer at full rate, a 128-wide tile with two
// issuers reaches ~80 % of that, a 64-wide tile is bound by shared-memory
// operand reads).
double tile_efficiency(int bn) { return bn == 256 ? 1.0 : (bn == 128 ? 0.8 : 0.55); }

// Tile width along GEMM-N for a GEMM with m_tiles row tiles and n_extent
// columns: the width with the lowest estimated time, counting whole waves
// of persistent CTAs (one per SM) and the padding of the last column tile.
int choose_block_n(int n_extent, long long m_tiles, int sm_count) {
  const int forced = g_tune_bn.load();
  if (forced) return forced;
  const int cands[3] = {256, 128, 64};
  int best = 64;
  double best_cost = 1e300;
  for (int bn : cands) {
    const long long n_tiles = (n_extent + bn - 1) / bn;
    const long long tiles = m_tiles * n_tiles;
    const long long waves = (tiles + sm_count - 1) / sm_count;
    const double cost = static_cast<double>(waves) * bn / tile_efficiency(bn);
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

// MMA issuer threads for a tile width: one thread can issue a tcgen05.mma
// only every ~70 cycles, so tiles narrower than 256 columns use two issuers,
// each with its own TMEM accumulator (the epilogue adds them in order).
int issuers_for(int bn) { return bn == 256 ? 1 : 2; }

// 16-bit passes: one accumulator per issuer.
void set_fp_accumulators(ConvGemmParams& p, int bn) {
  p.num_acc = issuers_for(bn);
  p.kb_per_acc = 1 << 30;
}

int grid_for(int units, const DeviceState* st) {
  int g = units < st->sm_count ? units : st->sm_count;
  const int cap = g_tune_max_ctas.load();
  if (cap > 0 && g > cap) g = cap;
  return g < 1 ? 1 : g;
}

// CTA pairs (clusters of two SMs, 256-row units, cta_group::2 MMAs): one
// issuing thread then drives two SMs' tensor cores and each SM loads half of
// the filter tile, which pays off where the MMA issue rate and the copies
// bound the main loop.  Measured on the ResNet-50 sweep: 128-wide tiles gain
// 13-14 % (28x28 and 14x14 fprop and dgrad), 64-wide ones lose 2 % (their
// epilogue, not the main loop, sets the pace) and 256-wide ones issue fast
// enough alone.  Used when the plan has a single sub-problem and at least
// two row tiles.
bool use_pairs(int bn, int tiles_m, bool mn_major_b) {
  (void)mn_major_b;  // MN-major filter halves are 64 columns wide at bn = 128
  const int mode = g_tune_no_pairs.load();  // 0 built-in, 1 never, 2 also 256-wide tiles
  if (mode == 1) return false;
  if (bn != 128 && !(bn == 256 && mode == 2)) return false;
  if (tiles_m < 2) return false;
  return conv_gemm_pair_capacity(bn) > 0;
}

// Even grid of whole pairs for `units` 256-row units.
int grid_for_pairs(int units, int bn, const DeviceState* st) {
  int pairs = conv_gemm_pair_capacity(bn);
  if (pairs > st->sm_count / 2) pairs = st->sm_count / 2;
  if (units < pairs) pairs = units;
  const int cap = g_tune_max_ctas.load();
  if (cap > 0 && 2 * pairs > cap) pairs = cap / 2;
  return 2 * (pairs < 1 ? 1 : pairs);
}

void init_common(ConvGemmParams& p, const DeviceState* st) {
  std::memset(&p, 0, sizeof(p));
  p.status = st->status;
  p.timeout_ns = kTimeoutNs;
  p.num_acc = 1;
  p.kb_per_acc = 1 << 30;
  p.splits = 1;
  p.epi_groups = g_tune_epi_groups.load();  // 0: the launcher decides
  p.raster = g_tune_raster.load();          // 0: column tiles fastest
  p.res_b = g_tune_resident_b.load() == 1 ? 0 : 1;  // the launcher decides where it applies
  p.general_epilogue = g_tune_general_epi.load();
}

// fprop plan (16-bit, or the int8 path's widened copies) on X [N,H,W,C],
// Wt [K,R,S,C], tile width bn.
igconv_status_t plan_fprop(ConvGemmParams& p, int bn, const igconv_problem_t* pb, int P, int Q,
                           int bf16, const void* X, const void* Wt,
                           const cuuint64_t* x_strides = nullptr) {
  if (bn != 64 && bn != 128 && bn != 256) return IGCONV_ERR_INVALID_ARG;
  const long long M = static_cast<long long>(pb->N) * P * Q;
  SubProblem& sp = p.sub[0];
  sp.M = static_cast<int>(M);
  sp.tile_begin = 0;
  sp.tiles_m = ceil_div(M, kBlockM);
  sp.Hs = P;
  sp.Ws = Q;
  sp.lower_h = -pb->pad_h;
  sp.lower_w = -pb->pad_w;
  sp.trav_h = pb->stride_h;
  sp.trav_w = pb->stride_w;
  sp.r0 = 0; sp.rstep = 1; sp.rcount = pb->R; sp.offh0 = 0; sp.doffh = pb->dil_h;
  sp.s0 = 0; sp.sstep = 1; sp.scount = pb->S; sp.offw0 = 0; sp.doffw = pb->dil_w;
  sp.out_h0 = 0; sp.out_w0 = 0; sp.out_sh = 1; sp.out_sw = 1;
  p.nsub = 1;
  p.a_src = SRC_IM2COL_K;
  p.b_src = SRC_W_K;
  p.cblocks = ceil_div(pb->C, kBlockK);
  p.N_gemm = pb->K;
  p.tiles_n = ceil_div(pb->K, bn);
  p.units = sp.tiles_m * p.tiles_n;
  p.out_C = pb->K;
  p.out_H = P;
  p.out_W = Q;
  p.idesc = make_idesc(kBlockM, bn, bf16, 0, 0);
  set_fp_accumulators(p, bn);
  // box of filter-origin positions: [-pad, H - 1 + pad - dil*(R-1)]
  if (!encode_im2col(&p.mapA[0], X, bf16, pb->N, pb->H, pb->W, pb->C, -pb->pad_h, -pb->pad_w,
                     pb->pad_h - (pb->R - 1) * pb->dil_h, pb->pad_w - (pb->S - 1) * pb->dil_w,
                     pb->stride_h, pb->stride_w, kBlockM, 64, CU_TENSOR_MAP_SWIZZLE_128B,
                     x_strides))
    return IGCONV_ERR_UNSUPPORTED;
  p.mapA_valid = 1u;
  if (!encode_filter(&p.mapB, Wt, bf16, pb->K, pb->R, pb->S, pb->C, bn))
    return IGCONV_ERR_UNSUPPORTED;
  return IGCONV_OK;
}

// Few-channel fprop (C <= 8): the pixels are read as 8-channel, 16-byte rows
// (X itself when C == 8, else a zero-padded copy) and the filter as a
// [R*S][K][8] copy; both copies live in the caller's workspace.
size_t round256(size_t b) { return (b + 255) / 256 * 256; }
struct FewChannelWs {
  size_t x_bytes, w_bytes, total;
};
FewChannelWs few_channel_ws(const igconv_problem_t* pb) {
  FewChannelWs w;
  const size_t pixels = static_cast<size_t>(pb->N) * pb->H * pb->W;
  w.x_bytes = pb->C < 8 ? round256(pixels * 16) : 0;
  // filter image [block][tile_n][8 taps][bn][8]: bn * tiles_n <= K rounded up to 256
  w.w_bytes = round256(static_cast<size_t>(ceil_div(pb->R * pb->S, 8)) *
                       static_cast<size_t>(ceil_div(pb->K, 256)) * 256 * 128);
  w.total = w.x_bytes + w.w_bytes;
  return w;
}

int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Few-channel packing (FewPack, igconv_internal.h) for C <= 8 at dilation 1
// with fh * fw * C <= 64 (fh, fw the strides): the stem's 7x7 stride-2
// filter over 3 channels becomes a stride-1 4x4 one over 2x2x3 (padded to
// 16) channels, four packed pixels per 128-byte row: 4 reduction blocks of
// 64 instead of 7 of the tap-packed path, each one full-width TMA load
// instead of eight 16-byte ones.  Off when IGCONV_TUNE_FEW_CHANNELS is 1.
bool few_pack_plan(const igconv_problem_t* pb, int P, int Q, FewPack* f) {
  if (g_tune_few_channels.load() == 1) return false;
  if (pb->C > 8 || pb->dil_h != 1 || pb->dil_w != 1) return false;
  const int z = pb->stride_h * pb->stride_w * pb->C;
  if (z > 64) return false;
  f->fh = pb->stride_h;
  f->fw = pb->stride_w;
  f->C = pb->C;
  f->R = pb->R;
  f->S = pb->S;
  f->ph = pb->pad_h;
  f->pw = pb->pad_w;
  f->cz = 8;
  while (f->cz < z) f->cz *= 2;
  f->ppr = 64 / f->cz;
  f->A0 = floor_div(-pb->pad_h, f->fh);
  f->B0 = floor_div(-pb->pad_w, f->fw);
  f->R2 = floor_div(pb->R - 1 - pb->pad_h, f->fh) - f->A0 + 1;
  const int S2 = floor_div(pb->S - 1 - pb->pad_w, f->fw) - f->B0 + 1;
  f->Sv = ceil_div(S2, f->ppr);
  f->Hz = P + f->R2 - 1;
  f->Wv = Q + (f->Sv - 1) * f->ppr;
  f->Wz = f->Wv + f->ppr - 1;
  const long long row_bytes = static_cast<long long>(f->Wz) * f->cz * 2;
  return row_bytes * f->Hz * pb->N < (1LL << 40) && f->Hz < (1 << 24) && f->Wz < (1 << 24);
}

// The stride-1 problem the packed image and filter define: 64 channels,
// R2 x Sv taps (Sv along w, ppr packed pixels apart), no padding.
igconv_problem_t few_pack_problem(const igconv_problem_t* pb, const FewPack& f) {
  igconv_problem_t v = *pb;
  v.H = f.Hz;
  v.W = f.Wv;
  v.C = 64;
  v.R = f.R2;
  v.S = f.Sv;
  v.pad_h = v.pad_w = 0;
  v.stride_h = v.stride_w = 1;
  v.dil_h = 1;
  v.dil_w = f.ppr;
  return v;
}

// Few-channel dgrad on the same space-to-depth image but without windows:
// one packed pixel per column (ppr = 1, cz = the used channels rounded up to
// a multiple of 8), so the problem is a stride-1 convolution over cz
// channels with R2 x S2 taps whose data gradient is the gradient of the
// packed image; every X element was copied to exactly one packed element,
// so dX is a gather of it.  Eligibility as few_pack_plan.
bool few_pack_plan_dgrad(const igconv_problem_t* pb, int P, int Q, FewPack* f) {
  if (!few_pack_plan(pb, P, Q, f)) return false;
  const int used = f->fh * f->fw * f->C;
  f->cz = (used + 7) / 8 * 8;
  f->ppr = 1;
  f->Sv = floor_div(pb->S - 1 - pb->pad_w, f->fw) - f->B0 + 1;
  f->Wv = Q + f->Sv - 1;
  f->Wz = f->Wv;
  return true;
}

struct FewDgradPackWs {
  size_t w_bytes, z_bytes, total;
};
FewDgradPackWs few_dgrad_pack_ws(const igconv_problem_t* pb, const FewPack& f) {
  FewDgradPackWs w;
  w.w_bytes = round256(static_cast<size_t>(pb->K) * f.R2 * f.Sv * f.cz * 2);
  w.z_bytes = round256(static_cast<size_t>(pb->N) * f.Hz * f.Wz * f.cz * sizeof(float));
  w.total = w.w_bytes + w.z_bytes;
  return w;
}

struct FewPackWs {
  size_t z_bytes, w_bytes;
  cuuint64_t strides[3];  // pixel, row, image strides of the packed image
};
FewPackWs few_pack_ws(const igconv_problem_t* pb, const FewPack& f) {
  FewPackWs w;
  const cuuint64_t px = static_cast<cuuint64_t>(f.cz) * 2;
  w.strides[0] = px;
  w.strides[1] = px * f.Wz;
  w.strides[2] = px * f.Wz * f.Hz;
  w.z_bytes = round256(static_cast<size_t>(w.strides[2]) * pb->N);
  w.w_bytes = round256(static_cast<size_t>(pb->K) * f.R2 * f.Sv * 128);
  return w;
}

// One reduction block = 8 filter taps x 8 channels (tap = r * S + s), so a
// 7x7 filter takes 7 blocks instead of the 49 (of 64 channels each, 8 of
// them real at most) of the general path.
igconv_status_t plan_fprop_taps(ConvGemmParams& p, int bn, const igconv_problem_t* pb, int P,
                                int Q, int bf16, const void* X8, const void* Wt8) {
  if (bn != 64 && bn != 128 && bn != 256) return IGCONV_ERR_INVALID_ARG;
  const int RS = pb->R * pb->S;
  const long long M = static_cast<long long>(pb->N) * P * Q;
  SubProblem& sp = p.sub[0];
  sp.M = static_cast<int>(M);
  sp.tile_begin = 0;
  sp.tiles_m = ceil_div(M, kBlockM);
  sp.Hs = P;
  sp.Ws = Q;
  sp.lower_h = -pb->pad_h;
  sp.lower_w = -pb->pad_w;
  sp.trav_h = pb->stride_h;
  sp.trav_w = pb->stride_w;
  // blocks per tile: rcount * scount * cblocks
  sp.r0 = 0; sp.rstep = 1; sp.rcount = 1; sp.offh0 = 0; sp.doffh = 0;
  sp.s0 = 0; sp.sstep = 1; sp.scount = ceil_div(RS, 8); sp.offw0 = 0; sp.doffw = 0;
  sp.out_h0 = 0; sp.out_w0 = 0; sp.out_sh = 1; sp.out_sw = 1;
  p.nsub = 1;
  p.a_src = SRC_IM2COL_TAPS;
  p.b_src = SRC_W_TAPS;
  p.cblocks = 1;
  p.wg_S = pb->S;
  p.wg_RS = RS;
  p.wg_dh = pb->dil_h;
  p.wg_dw = pb->dil_w;
  p.N_gemm = pb->K;
  p.tiles_n = ceil_div(pb->K, bn);
  p.units = sp.tiles_m * p.tiles_n;
  p.out_C = pb->K;
  p.out_H = P;
  p.out_W = Q;
  p.idesc = make_idesc(kBlockM, bn, bf16, 0, 0);
  set_fp_accumulators(p, bn);
  if (!encode_im2col(&p.mapA[0], X8, bf16, pb->N, pb->H, pb->W, 8, -pb->pad_h, -pb->pad_w,
                     pb->pad_h - (pb->R - 1) * pb->dil_h, pb->pad_w - (pb->S - 1) * pb->dil_w,
                     pb->stride_h, pb->stride_w, kBlockM, 8, CU_TENSOR_MAP_SWIZZLE_NONE))
    return IGCONV_ERR_UNSUPPORTED;
  p.mapA_valid = 1u;
  p.taps_filter = Wt8;
  return IGCONV_OK;
}

// One spatial dimension of the dgrad residue-class decomposition.
//   Output rows h with (h + pad) % stride == rho are h = h0 + stride * t,
//   t in [0, count).  Filter taps that reach them satisfy
//   r * dil % stride == rho; for such a tap the output-gradient row is
//   p = t + (h0 + pad - r * dil) / stride.  Taps form an arithmetic
//   progression r = r0 + j * rstep.  The im2col base row of t is
//   t + delta_min with per-tap offset (rcount - 1 - j) * rstep * dil / stride.
struct Residue1D {
  int h0, count;          // output rows
  int r0, rstep, rcount;  // taps
  int delta_min;          // base offset
  int off0, doff;         // im2col offsets of tap j
};

int gcd_int(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

Residue1D residue_1d(int rho, int H, int R, int pad, int stride, int dil) {
  Residue1D d{};
  d.h0 = ((rho - pad) % stride + stride) % stride;
  d.count = d.h0 < H ? (H - d.h0 + stride - 1) / stride : 0;
  d.rcount = 0;
  d.r0 = 0;
  for (int r = 0; r < R; ++r) {
    if ((r * dil) % stride == rho) {
      if (d.rcount == 0) d.r0 = r;
      ++d.rcount;
    }
  }
  d.rstep = stride / gcd_int(dil, stride);
  if (d.rcount > 0) {
    const int r_last = d.r0 + (d.rcount - 1) * d.rstep;
    d.delta_min = (d.h0 + pad - r_last * dil) / stride;  // exact division
    d.off0 = (d.rcount - 1) * d.rstep * dil / stride;
    d.doff = -(d.rstep * dil / stride);
  }
  return d;
}

// Strided dgrad with H % stride_h == 0 and W % stride_w == 0: every residue
// class has the same H / stride_h x W / stride_w grid.  Its rows are padded
// to a multiple of 32 grid columns when that adds at most a sixth, so each
// epilogue warp's 32 rows are one residue-class row of dX and go out as one
// TMA store through a 5D view of dX (the padding columns are clipped).
int padded_class_width(const igconv_problem_t* pb) {
  if (pb->stride_h * pb->stride_w < 2 || pb->H % pb->stride_h || pb->W % pb->stride_w) return 0;
  const int ws = pb->W / pb->stride_w;
  const int wsp = ceil_div(ws, 32) * 32;
  return 6 * (wsp - ws) <= ws ? wsp : 0;
}

igconv_status_t plan_dgrad(ConvGemmParams& p, int* block_n, const igconv_problem_t* pb, int P,
                           int Q, int bf16, const void* dY, const void* Wt, int sm_count,
                           int forced_bn = 0, bool pad_rows = false) {
  const int bn = forced_bn ? forced_bn
                           : choose_block_n(pb->C,
                                            ceil_div(static_cast<long long>(pb->N) * pb->H * pb->W,
                                                     kBlockM),
                                            sm_count);
  if (bn != 64 && bn != 128 && bn != 256) return IGCONV_ERR_INVALID_ARG;
  if (pb->stride_h * pb->stride_w > kMaxSub) return IGCONV_ERR_UNSUPPORTED;
  p.tiles_n = ceil_div(pb->C, bn);
  const int wsp = pad_rows && g_tune_dgrad_rows.load() != 1 ? padded_class_width(pb) : 0;
  int nsub = 0, tile_begin = 0;
  for (int rh = 0; rh < pb->stride_h; ++rh) {
    const Residue1D dh = residue_1d(rh, pb->H, pb->R, pb->pad_h, pb->stride_h, pb->dil_h);
    if (dh.count == 0) continue;
    for (int rw = 0; rw < pb->stride_w; ++rw) {
      const Residue1D dw = residue_1d(rw, pb->W, pb->S, pb->pad_w, pb->stride_w, pb->dil_w);
      if (dw.count == 0) continue;
      SubProblem& sp = p.sub[nsub];
      const int ws = wsp > 0 ? wsp : dw.count;  // grid columns per row
      const long long M = static_cast<long long>(pb->N) * dh.count * ws;
      sp.M = static_cast<int>(M);
      sp.tile_begin = tile_begin;
      sp.tiles_m = ceil_div(M, kBlockM);
      sp.Hs = dh.count;
      sp.Ws = ws;
      sp.ws_valid = wsp > 0 ? dw.count : 0;
      sp.lower_h = dh.delta_min;
      sp.lower_w = dw.delta_min;
      sp.trav_h = 1;
      sp.trav_w = 1;
      const bool taps = dh.rcount > 0 && dw.rcount > 0;
      sp.r0 = dh.r0; sp.rstep = dh.rstep; sp.rcount = taps ? dh.rcount : 0;
      sp.offh0 = dh.off0; sp.doffh = dh.doff;
      sp.s0 = dw.r0; sp.sstep = dw.rstep; sp.scount = taps ? dw.rcount : 1;
      sp.offw0 = dw.off0; sp.doffw = dw.doff;
      sp.out_h0 = dh.h0;
      sp.out_w0 = dw.h0;
      sp.out_sh = pb->stride_h;
      sp.out_sw = pb->stride_w;
      if (taps) {
        // base rows of the traversal: [delta_min, delta_min + count - 1] over dY [P][Q]
        // (padded rows: the traversal runs on past the grid, reading zeros;
        // if the map cannot take that corner, plan without the padding)
        if (!encode_im2col(&p.mapA[nsub], dY, bf16, pb->N, P, Q, pb->K, dh.delta_min,
                           dw.delta_min, dh.count - P + dh.delta_min,
                           ws - Q + dw.delta_min, 1, 1, kBlockM)) {
          if (wsp == 0) return IGCONV_ERR_UNSUPPORTED;
          p.mapA_valid = 0;
          return plan_dgrad(p, block_n, pb, P, Q, bf16, dY, Wt, sm_count, forced_bn, false);
        }
        p.mapA_valid |= 1u << nsub;
      }
      tile_begin += sp.tiles_m * p.tiles_n;
      ++nsub;
    }
  }
  p.nsub = nsub;
  p.store_5d = wsp > 0 ? 1 : 0;  // the launcher encodes the 5D view of dX
  p.units = tile_begin;
  p.a_src = SRC_IM2COL_K;
  p.b_src = SRC_W_MN;
  p.cblocks = ceil_div(pb->K, kBlockK);
  p.N_gemm = pb->C;
  p.out_C = pb->C;
  p.out_H = pb->H;
  p.out_W = pb->W;
  p.idesc = make_idesc(kBlockM, bn, bf16, 0, 1);
  set_fp_accumulators(p, bn);
  if (!encode_filter(&p.mapB, Wt, bf16, pb->K, pb->R, pb->S, pb->C, 64))
    return IGCONV_ERR_UNSUPPORTED;
  *block_n = bn;
  return IGCONV_OK;
}

struct WgradPlan {
  int swapped;        // 0: A = X side (M = R*S*cpad), B = dY side (N = K)
  int cblocks, cpad;  // X-channel blocks and padded channels per tap
  int rs;
  int tiles_m, tiles_n, bn;
  int M_pad, N_pad;
  int kblocks, splits;
  size_t ws_bytes;
};

// wgrad plan: the GEMM orientation (which of dY^T and im2col(X) gives the
// rows), the tile width and the split count are chosen together, minimising
// (waves of persistent CTAs) x (columns x reduction blocks per unit) / (tile
// efficiency).  Splits fill at most one wave and keep >= 8 blocks each.
// Orientation, tile width and split count of a wgrad GEMM with an X side of
// `xext` rows (the (tap, c) extent) and the dY side of K rows.
void choose_wgrad_shape(int K, long long xext, int sm_count, WgradPlan* w, int max_bn) {
  const int sms = sm_count > 0 ? sm_count : 148;
  const int forced_splits = g_tune_splits.load();
  const int forced_bn = g_tune_bn.load();
  double best = 1e300;
  for (int swapped = 0; swapped < 2; ++swapped) {
    const long long mext = swapped ? K : xext;
    const long long next = swapped ? xext : K;
    const int cands[3] = {256, 128, 64};
    for (int bn : cands) {
      if (forced_bn && bn != forced_bn) continue;
      if (!forced_bn && bn > max_bn) continue;
      const int tiles_m = ceil_div(mext, kBlockM);
      const int tiles_n = ceil_div(next, bn);
      const long long tiles = static_cast<long long>(tiles_m) * tiles_n;
      int splits = forced_splits;
      if (splits <= 0) {
        splits = static_cast<int>(sms / tiles);
        const int max_by_depth = w->kblocks / 8;
        if (splits > max_by_depth) splits = max_by_depth;
      }
      if (splits > w->kblocks) splits = w->kblocks;
      if (splits < 1) splits = 1;
      const long long units = tiles * splits;
      const long long waves = (units + sms - 1) / sms;
      const double cost = static_cast<double>(waves) * bn * ceil_div(w->kblocks, splits) /
                          tile_efficiency(bn) * (static_cast<double>(tiles_m) * kBlockM / mext);
      if (cost < best * 0.999) {
        best = cost;
        w->swapped = swapped;
        w->bn = bn;
        w->tiles_m = tiles_m;
        w->tiles_n = tiles_n;
        w->splits = splits;
      }
    }
  }
  w->M_pad = w->tiles_m * kBlockM;
  w->N_pad = w->tiles_n * w->bn;
  w->ws_bytes = static_cast<size_t>(w->splits) * w->M_pad * w->N_pad * sizeof(float);
}

void plan_wgrad_shape(const igconv_problem_t* pb, int P, int Q, int sm_count, WgradPlan* w,
                      int max_bn = 256) {
  w->rs = pb->R * pb->S;
  w->cblocks = ceil_div(pb->C, kBlockK);
  w->cpad = w->cblocks * kBlockK;
  const long long npq = static_cast<long long>(pb->N) * P * Q;
  w->kblocks = ceil_div(npq, kBlockK);
  choose_wgrad_shape(pb->K, static_cast<long long>(w->rs) * w->cpad, sm_count, w, max_bn);
}

// Few channels (C < 8, pixels padded to 8): the X side is tap-packed, 8
// taps x 8 channels per 64-row chunk, so row = tap * 8 + c (channel pitch 8)
// and a 7x7 filter needs 7 chunks (448 rows) instead of 49.
void plan_wgrad_taps(const igconv_problem_t* pb, int P, int Q, int sm_count, WgradPlan* w) {
  w->rs = pb->R * pb->S;
  w->cblocks = 1;
  w->cpad = 8;
  const long long npq = static_cast<long long>(pb->N) * P * Q;
  w->kblocks = ceil_div(npq, kBlockK);
  choose_wgrad_shape(pb->K, static_cast<long long>(ceil_div(w->rs, 8)) * kBlockK, sm_count, w, 256);
}

// Channel window of a grouped block-diagonal GEMM whose 64-wide tiles run
// over groups of tile_g channels (K / groups for fprop and wgrad, C / groups
// for dgrad) and reduce over red_g channels per group on the other side:
// every tile holds whole groups, so tile n reduces over the `width` channels
// starting at (n / div) * mul.  False when a tile would split a group or a
// window start is not a multiple of 8 channels (a TMA copy's channel
// coordinate must be 16-byte aligned).
struct GroupWin {
  int mul, div, width, blocks;
};
bool plan_group_window(int tile_g, int red_g, GroupWin* g) {
  if (tile_g < 1 || red_g < 1) return false;
  if (64 % tile_g == 0) {  // 64 / tile_g groups per tile
    g->div = 1;
    g->mul = 64 / tile_g * red_g;
  } else if (tile_g % 64 == 0) {  // tile_g / 64 tiles per group
    g->div = tile_g / 64;
    g->mul = red_g;
  } else {
    return false;
  }
  if (g->mul % 8 != 0) return false;
  g->width = g->mul;
  g->blocks = ceil_div(g->width, kBlockK);
  return true;
}

// Grouped wgrad as a block-diagonal GEMM: rows (tap, c') with c' inside the
// output tile's channel window (win.blocks 64-channel blocks), one 64-wide
// column tile per 64 output channels; the split rule of plan_wgrad_shape.
void plan_wgrad_grouped(const igconv_problem_t* pb, int P, int Q, int sm_count,
                        const GroupWin& win, WgradPlan* w) {
  const int sms = sm_count > 0 ? sm_count : 148;
  w->rs = pb->R * pb->S;
  w->cblocks = win.blocks;
  w->cpad = win.blocks * kBlockK;
  const long long xext = static_cast<long long>(w->rs) * w->cpad;
  const long long npq = static_cast<long long>(pb->N) * P * Q;
  w->kblocks = ceil_div(npq, kBlockK);
  w->swapped = 0;
  w->bn = 64;
  w->tiles_m = ceil_div(xext, kBlockM);
  w->tiles_n = ceil_div(pb->K, 64);
  const long long tiles = static_cast<long long>(w->tiles_m) * w->tiles_n;
  int splits = g_tune_splits.load();
  if (splits <= 0) {
    splits = static_cast<int>(sms / tiles);
    const int max_by_depth = w->kblocks / 8;
    if (splits > max_by_depth) splits = max_by_depth;
  }
  if (splits > w->kblocks) splits = w->kblocks;
  if (splits < 1) splits = 1;
  w->splits = splits;
  w->M_pad = w->tiles_m * kBlockM;
  w->N_pad = w->tiles_n * w->bn;
  w->ws_bytes = static_cast<size_t>(w->splits) * w->M_pad * w->N_pad * sizeof(float);
}

// Workspace of the grouped wgrad GEMM: the split partials, then the fp32
// gradient of the windowed filter [K][R][S][cpad].
size_t grouped_wgrad_gemm_bytes(const WgradPlan& w, const igconv_problem_t* pb) {
  return round256(w.ws_bytes) +
         round256(static_cast<size_t>(pb->K) * w.rs * w.cpad * sizeof(float));
}

// ---------------------------------------------------------------------------
// Depthwise planning (groups == C == K)
// ---------------------------------------------------------------------------
constexpr int kDwHalfRows = 8, kDwChunk = 32;
constexpr int kDwSmemLimit = 227 * 1024 - 128 - 16;

long long round128(long long v) { return (v + 127) / 128 * 128; }

// Tiled map over an NHWC 16-bit tensor [n][h][w][c], box {32 c, box_w, box_h,
// 1 image}, no swizzle; zero fill outside the tensor.
bool encode_nhwc_window(CUtensorMap* map, const void* base, int bf16, int n, int h, int w, int c,
                        int box_w, int box_h) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(c), static_cast<cuuint64_t>(w),
                              static_cast<cuuint64_t>(h), static_cast<cuuint64_t>(n)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(c) * 2,
                                 static_cast<cuuint64_t>(c) * 2 * w,
                                 static_cast<cuuint64_t>(c) * 2 * w * h};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(kDwChunk), static_cast<cuuint32_t>(box_w),
                             static_cast<cuuint32_t>(box_h), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode_tiled(map, tma_dtype(bf16), 4, const_cast<void*>(base), dims,
                                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Common checks of the grouped entry points.  groups == 1 is the dense path
// (*direct = false).  Otherwise the direct kernels cover C == K with a group
// width C/groups of 1 (depthwise), 2, 4, 8, 16 or 32 (*direct = true,
// *cg = C/groups); other group counts (C != K among them) are UNSUPPORTED
// here and run only on the tensor-core path (grouped_gemm_ok).
igconv_status_t check_groups(const igconv_problem_t* prob, int groups, bool* direct, int* cg) {
  if (!prob || groups < 1) return IGCONV_ERR_INVALID_ARG;
  if (prob->C < 1 || prob->K < 1 || prob->C % groups != 0 || prob->K % groups != 0)
    return IGCONV_ERR_INVALID_ARG;
  *direct = groups > 1;
  *cg = prob->C / groups;
  if (groups == 1) return IGCONV_OK;
  if (prob->C != prob->K) return IGCONV_ERR_UNSUPPORTED;
  const int w = *cg;
  if (w != 1 && w != 2 && w != 4 && w != 8 && w != 16 && w != 32) return IGCONV_ERR_UNSUPPORTED;
  return IGCONV_OK;
}

// Shape fields, tile geometry and shared-memory layout of a depthwise launch.
//   mode FWD   (fprop; stride-1 dgrad over dY): window of 8 output rows x
//              tq columns: (7*sh + (R-1)*dh + 1) x ((tq-1)*sw + (S-1)*dw + 1)
//              pixels, plus the column the second half's shift needs
//   mode PHASE (strided dgrad): the dY rows and columns that 8 dX rows x
//              16 column positions of every phase read
//   mode WGRAD the fprop window plus two dY boxes of 8 x (tq + 1) pixels
// `out_h` x `out_w` is the grid the tiles cover.  UNSUPPORTED when a window
// exceeds a TMA box (256) or one ring stage does not fit in shared memory.
igconv_status_t plan_dw(DwParams& p, const DeviceState* dev, const igconv_problem_t* pb,
                        int mode, int bf16, int cg, int out_h, int out_w) {
  std::memset(static_cast<void*>(&p), 0, sizeof(p));
  p.mode = mode;
  p.cg = cg;
  p.bf16 = bf16;
  p.status = dev->status;
  p.timeout_ns = kTimeoutNs;
  p.N = pb->N;
  p.C = pb->C;
  p.R = pb->R;
  p.S = pb->S;
  p.sh = pb->stride_h;
  p.sw = pb->stride_w;
  p.dh = pb->dil_h;
  p.dw = pb->dil_w;
  p.pad_h = pb->pad_h;
  p.pad_w = pb->pad_w;
  p.out_h = out_h;
  p.out_w = out_w;
  p.tq = dw_tile_q(p);
  p.chunks = ceil_div(pb->C, kDwChunk);
  p.rb_per_image = ceil_div(out_h, kDwHalfRows);
  p.row_blocks = static_cast<int>(static_cast<long long>(pb->N) * p.rb_per_image);
  p.tiles_p = ceil_div(p.row_blocks, 2);
  if (mode == DW_MODE_PHASE) {
    p.ih_t = (kDwHalfRows - 1 + (pb->R - 1) * pb->dil_h) / pb->stride_h + 2;
    p.iw_t = (pb->stride_w - 1 + (pb->S - 1) * pb->dil_w) / pb->stride_w + p.tq + 2;
    p.tiles_q = ceil_div(out_w, static_cast<long long>(p.tq) * pb->stride_w);
  } else {
    p.ih_t = (kDwHalfRows - 1) * pb->stride_h + (pb->R - 1) * pb->dil_h + 1;
    p.iw_t = (p.tq - 1) * pb->stride_w + (pb->S - 1) * pb->dil_w + 2;
    p.tiles_q = ceil_div(out_w, p.tq);
  }
  if (p.ih_t > 256 || p.iw_t > 256) return IGCONV_ERR_UNSUPPORTED;
  const long long all_tiles = static_cast<long long>(p.tiles_p) * p.tiles_q * p.chunks;
  if (all_tiles >= (1LL << 30)) return IGCONV_ERR_UNSUPPORTED;  // 32-bit tile indices
  p.div_chunks = make_fast_div(static_cast<uint32_t>(p.chunks));
  p.div_tiles_q = make_fast_div(static_cast<uint32_t>(p.tiles_q));
  p.div_rb = make_fast_div(static_cast<uint32_t>(p.rb_per_image));
  const long long rs = static_cast<long long>(pb->R) * pb->S;
  const long long box = round128(static_cast<long long>(p.ih_t) * p.iw_t * kDwChunk * 2);
  const long long dybox =
      mode == DW_MODE_WGRAD ? round128(static_cast<long long>(kDwHalfRows) * (p.tq + 1) * kDwChunk * 2)
                            : 0;
  const long long stage = 2 * box + 2 * dybox;
  const long long red_bytes = 16 * (cg > 1 ? cg : rs) * 16 * 8;
  if (stage > kDwSmemLimit) return IGCONV_ERR_UNSUPPORTED;
  p.box_bytes = static_cast<int>(box);
  p.dy_box_bytes = static_cast<int>(dybox);
  p.stage_bytes = static_cast<int>(stage);
  for (int stages = 2; stages >= 1; --stages) {
    long long end = stages * stage;
    p.stages = stages;
    p.wts_off = static_cast<int>(end);
    if (mode != DW_MODE_WGRAD) {
      end += rs * cg * 16 * 8 + 16 * 8;
    } else if ((cg > 1 || dw_fast_ks(p) > 0) && red_bytes <= stages * stage) {
      p.red_off = 0;  // scratch over the ring, used after the last tile
    } else {
      p.red_off = static_cast<int>(end < INT32_MAX ? end : 0);
      end += red_bytes;
    }
    end = (end + 15) / 16 * 16;
    if (end <= kDwSmemLimit) {
      p.bar_off = static_cast<int>(end);
      return IGCONV_OK;
    }
  }
  return IGCONV_ERR_UNSUPPORTED;
}

long long floor_div_ll(long long a, long long b) {
  const long long q = a / b;
  return (a % b != 0 && ((a < 0) != (b < 0))) ? q - 1 : q;
}

// Tap tables of the strided dgrad (see DwParams): for each output-row
// residue a (rows rb*8 + w with w % sh == a) the taps r with
// (a + ph - r*dh) divisible by sh, and the window row offset of each, so
// that the row a warp w reads is w / sh + offset; likewise for each column
// phase b.  Left unset (generic loops) unless every entry stays inside the
// window and 8 is a multiple of sh (so that the residue of a row is that of
// its warp).
void build_phase_tables(DwParams& p, const igconv_problem_t* pb) {
  p.use_tables = 0;
  p.col_consecutive = 0;
  const int sh = pb->stride_h, sw = pb->stride_w;
  if (kDwHalfRows % sh != 0 || pb->R > kDwMaxTaps || pb->S > kDwMaxTaps) return;
  const long long h_base = floor_div_ll(pb->pad_h - static_cast<long long>(pb->R - 1) * pb->dil_h, sh);
  const long long w_base = floor_div_ll(pb->pad_w - static_cast<long long>(pb->S - 1) * pb->dil_w, sw);
  for (int a = 0; a < sh; ++a) {
    int n = 0;
    for (int r = 0; r < pb->R; ++r) {
      const long long t = a + pb->pad_h - static_cast<long long>(r) * pb->dil_h;
      if (t - floor_div_ll(t, sh) * sh != 0) continue;
      const long long off = floor_div_ll(t, sh) - h_base;
      if (off < 0 || kDwHalfRows / sh - 1 + off >= p.ih_t) return;
      p.row_r[a][n] = static_cast<int16_t>(r);
      p.row_off[a][n] = static_cast<int16_t>(off);
      ++n;
    }
    p.row_n[a] = static_cast<int8_t>(n);
  }
  for (int b = 0; b < sw; ++b) {
    int n = 0;
    for (int c = 0; c < pb->S; ++c) {
      const long long t = b + pb->pad_w - static_cast<long long>(c) * pb->dil_w;
      if (t - floor_div_ll(t, sw) * sw != 0) continue;
      const long long off = floor_div_ll(t, sw) - w_base;
      if (off < 0 || off + p.tq + 1 > p.iw_t) return;
      p.col_s[b][n] = static_cast<int16_t>(c);
      p.col_off[b][n] = static_cast<int16_t>(off);
      ++n;
    }
    p.col_n[b] = static_cast<int8_t>(n);
  }
  p.use_tables = 1;
  // consecutive column offsets (unit column dilation) let the kernel read
  // each dY word once per filter row
  p.col_consecutive = 1;
  for (int b = 0; b < sw; ++b)
    for (int j = 1; j < p.col_n[b]; ++j)
      if (p.col_off[b][j] != p.col_off[b][j - 1] - 1) p.col_consecutive = 0;
}

// Persistent grid of the fprop / dgrad kernels: as many CTAs as fit at once
// (or the tuning cap), rounded down to a multiple of the channel-chunk count
// so that each CTA keeps one chunk (and stages its filter once).
int dw_grid(const DwParams& p, const DeviceState* dev, cudaError_t* err) {
  int occ = 0;
  *err = dw_occupancy(p, &occ);
  if (*err != cudaSuccess) return 0;
  if (occ < 1) occ = 1;
  long long g = static_cast<long long>(occ) * dev->sm_count;
  const int cap = g_tune_max_ctas.load();
  if (cap > 0 && g > cap) g = cap;
  if (g > p.tiles) g = p.tiles;
  g = g / p.chunks * p.chunks;
  if (g < p.chunks) g = p.chunks;
  return static_cast<int>(g);
}

// Depthwise wgrad plan: the kernel's layout plus the split count.
igconv_status_t plan_dw_wgrad(DwParams& p, const DeviceState* dev, const igconv_problem_t* pb,
                              int P, int Q, int bf16, int cg) {
  igconv_status_t st = plan_dw(p, dev, pb, DW_MODE_WGRAD, bf16, cg, P, Q);
  if (st != IGCONV_OK) return st;
  p.org_h = -pb->pad_h;
  p.org_w = -pb->pad_w;
  p.tiles = static_cast<long long>(p.tiles_p) * p.tiles_q;
  int occ = 0;
  if (dw_occupancy(p, &occ) != cudaSuccess) return cuda_error();
  if (occ < 1) occ = 1;
  // grouped: one CTA per (chunk, filter tap, split)
  const long long per_split = static_cast<long long>(p.chunks) * (cg > 1 ? pb->R * pb->S : 1);
  long long splits = static_cast<long long>(occ) * dev->sm_count / per_split;
  const int tuned = g_tune_splits.load();
  if (tuned > 0) splits = tuned;
  if (splits > p.tiles) splits = p.tiles;
  if (splits < 1) splits = 1;
  p.splits = static_cast<int>(splits);
  return IGCONV_OK;
}

size_t dw_wgrad_ws_bytes(const DwParams& p) {
  return static_cast<size_t>(p.splits) * p.R * p.S * p.C * p.cg * sizeof(float);
}

}  // namespace

namespace igc {
bool pdl_enabled() { return g_tune_pdl.load(std::memory_order_relaxed) == 1; }
}  // namespace igc

// ===========================================================================
// C ABI
// ===========================================================================
namespace {

// int8 dgrad / wgrad planning helpers

int current_sm_count() {
  int sm_count = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      sm_count = v;
  } else {
    cudaGetLastError();  // no device: size for the default SM count
  }
  return sm_count;
}

// Accumulators for a tile whose units have at most max_kb reduction blocks:
// NI issuers, groups of at most 16 blocks per issuer; false when two TMEM
// buffers of them do not fit in the 512 columns.
bool int_accumulators(int bn, int max_kb, int* num_acc, int* kb_per_acc) {
  const int ni = issuers_for(bn);
  const int per_issuer = ceil_div(max_kb > 0 ? max_kb : 1, ni);
  const int groups = ceil_div(per_issuer, 16);
  if (2 * ni * groups * bn > 512) return false;
  *num_acc = ni * groups;
  *kb_per_acc = ceil_div(per_issuer, groups);
  return true;
}

// wgrad plan of the int8 path: the fp16 plan, with the split count raised
// until every split's reduction fits the accumulators of its tile width.
void plan_wgrad_int8(const igconv_problem_t* pb, int P, int Q, int sm_count, WgradPlan* w) {
  // a 256-wide tile has one issuer and room for one accumulator per TMEM
  // buffer (16 blocks per split); 128- and 64-wide tiles have two issuers
  // and room for 32 and 64 blocks, so far fewer splits and partials
  plan_wgrad_shape(pb, P, Q, sm_count, w, 128);
  const int ni = issuers_for(w->bn);
  const int max_groups = 512 / (2 * ni * w->bn);
  const int max_kb = ni * (max_groups < 1 ? 1 : max_groups) * 16;
  const int need = ceil_div(w->kblocks, max_kb);
  if (w->splits < need) w->splits = need;
  if (w->splits > w->kblocks) w->splits = w->kblocks;
  w->ws_bytes = static_cast<size_t>(w->splits) * w->M_pad * w->N_pad * sizeof(int32_t);
}

// Split-K for the forward and stride-1 data passes (single sub-problem,
// single CTAs): each tile's reduction cut into `splits` equal ranges whose
// fp32 partial tiles an ordered reduction adds, applying the epilogue.  It
// runs only when forced by the tuning knob (n >= 2): measured on the
// ResNet-50 layers at batch 128 it loses everywhere, also where whole tiles
// leave most of the last wave empty (7x7 512 -> 512: 98 tiles on 152 SMs,
// 36.5 us unsplit against 38.5 / 42.7 / 42.3 us with 3 / 2 / 4 splits; 14x14
// and 28x28: 1.5-2.7x slower), because the partial tiles' round trip and
// the reduction cost more than the wave they recover.
int conv_split_count(long long units, int kblocks, int sm_count) {
  (void)units;
  (void)sm_count;
  const int forced = g_tune_conv_splits.load();
  if (forced >= 2) return forced < kblocks ? forced : (kblocks < 1 ? 1 : kblocks);
  return 1;
}

// Turns a planned single-CTA conv GEMM (fprop or stride-1 dgrad) into its
// split-K form writing fp32 partials to `ws`; returns the partial bytes.
size_t conv_split_bytes(const ConvGemmParams& p, int bn, int splits) {
  return static_cast<size_t>(splits) * p.sub[0].tiles_m * kBlockM *
         static_cast<size_t>(p.tiles_n) * bn * sizeof(float);
}

bool set_conv_split(ConvGemmParams& p, int bn, int splits, void* ws) {
  const int kb = p.sub[0].rcount * p.sub[0].scount * p.cblocks;
  p.epi = EPI_PARTIAL;
  p.conv_split = 1;
  p.splits = splits;
  p.kblocks_total = kb;
  p.tiles_m_total = p.sub[0].tiles_m;
  p.units = p.sub[0].tiles_m * p.tiles_n * splits;
  const long long m_pad = static_cast<long long>(p.sub[0].tiles_m) * kBlockM;
  const int n_pad = p.tiles_n * bn;
  p.out = ws;
  p.ws_split_stride = m_pad * n_pad;
  p.ws_ld = n_pad;
  p.cin = nullptr;
  p.bias = nullptr;
  p.bias_cached = 0;
  p.use_tma_store = encode_out_2d(&p.mapY, ws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                                  splits * m_pad, n_pad, 16, CU_TENSOR_MAP_SWIZZLE_64B) ? 1 : 0;
  p.store_box64 = 0;
  return true;
}

// Few-channel dgrad (C < 8): the filter padded to 8 channels and the fp32
// result rows of 8 channels, both in the workspace.
struct FewDgradWs {
  size_t w_bytes, x_bytes, total;
};
FewDgradWs few_dgrad_ws(const igconv_problem_t* pb) {
  FewDgradWs w;
  w.w_bytes = round256(static_cast<size_t>(pb->K) * pb->R * pb->S * 16);
  w.x_bytes = round256(static_cast<size_t>(pb->N) * pb->H * pb->W * 8 * sizeof(float));
  w.total = w.w_bytes + w.x_bytes;
  return w;
}

// Few-channel wgrad (C < 8): the pixels copied to 8-channel rows in the
// workspace, then the wgrad GEMM with a tap-packed X side (8 taps x 8
// channels per 64-row chunk, row = tap * 8 + c) and the usual ordered
// split reduction, which writes the C real channels of each tap.
igconv_status_t wgrad_few_channels(const igconv_problem_t* prob, int P, int Q,
                                   igconv_dtype_t dtype, igconv_dtype_t dw_dtype, const void* X,
                                   const void* dY, const void* Cin, void* dW, float alpha,
                                   float beta, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  igconv_problem_t k8 = *prob;
  k8.C = 8;
  igconv_status_t st = check_limits(&k8, P, Q, 8);
  if (st != IGCONV_OK) return st;
  const uintptr_t esz = dw_dtype == IGCONV_F32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(X) & 1) || !aligned16(dY) ||
      (reinterpret_cast<uintptr_t>(dW) & (esz - 1)) ||
      (beta != 0.0f && (reinterpret_cast<uintptr_t>(Cin) & (esz - 1))) ||
      (workspace && !aligned16(workspace)))
    return IGCONV_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  WgradPlan w;
  plan_wgrad_taps(prob, P, Q, dev->sm_count, &w);
  const long long pixels = static_cast<long long>(prob->N) * prob->H * prob->W;
  const size_t x8_bytes = round256(static_cast<size_t>(pixels) * 16);
  if (!workspace || workspace_bytes < x8_bytes + w.ws_bytes) return IGCONV_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* X8 = ws;
  void* part = ws + x8_bytes;
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  const long long xext = static_cast<long long>(ceil_div(w.rs, 8)) * kBlockK;
  ConvGemmParams p;
  init_common(p, dev);
  p.nsub = 1;
  p.a_src = w.swapped ? SRC_2D_MN : SRC_IM2COL_TAPS_MN;
  p.b_src = w.swapped ? SRC_IM2COL_TAPS_MN : SRC_2D_MN;
  p.epi = EPI_PARTIAL;
  p.tiles_m_total = w.tiles_m;
  p.tiles_n = w.tiles_n;
  p.splits = w.splits;
  p.kblocks_total = w.kblocks;
  p.units = w.tiles_m * w.tiles_n * w.splits;
  p.cblocks = 1;
  p.N_gemm = w.N_pad;
  p.idesc = make_idesc(kBlockM, w.bn, bf16, 1, 1);
  set_fp_accumulators(p, w.bn);
  p.wg_PQ = P * Q;
  p.wg_Q = Q;
  p.wg_lower_h = -prob->pad_h;
  p.wg_lower_w = -prob->pad_w;
  p.wg_sh = prob->stride_h;
  p.wg_sw = prob->stride_w;
  p.wg_S = prob->S;
  p.wg_RS = w.rs;
  p.wg_dh = prob->dil_h;
  p.wg_dw = prob->dil_w;
  p.wg_K = prob->K;
  p.out = part;
  p.ws_split_stride = static_cast<long long>(w.M_pad) * w.N_pad;
  p.ws_ld = w.N_pad;
  p.use_tma_store = encode_out_2d(&p.mapY, part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                                  static_cast<long long>(w.splits) * w.M_pad, w.N_pad, 16,
                                  CU_TENSOR_MAP_SWIZZLE_64B) ? 1 : 0;
  // 64 output positions x 8 channels (16 bytes each) per load, no swizzle
  if (!encode_im2col(&p.mapA[0], X8, bf16, prob->N, prob->H, prob->W, 8, -prob->pad_h,
                     -prob->pad_w, prob->pad_h - (prob->R - 1) * prob->dil_h,
                     prob->pad_w - (prob->S - 1) * prob->dil_w, prob->stride_h, prob->stride_w,
                     kBlockK, 8, CU_TENSOR_MAP_SWIZZLE_NONE))
    return IGCONV_ERR_UNSUPPORTED;
  p.mapA_valid = 1u;
  const long long npq = static_cast<long long>(prob->N) * P * Q;
  if (!encode_2d(&p.mapB, dY, bf16, npq, prob->K)) return IGCONV_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_pad_pixels8(X, X8, pixels, prob->C, s) != cudaSuccess) return cuda_error();
  if (launch_conv_gemm(p, w.bn, grid_for(p.units, dev), s) != cudaSuccess) return cuda_error();
  const int dwt = dw_dtype == IGCONV_F32 ? 2 : (dw_dtype == IGCONV_BF16 ? 1 : 0);
  return from_cuda(launch_wgrad_reduce(static_cast<const float*>(part), w.splits,
                                       p.ws_split_stride, w.N_pad,
                                       static_cast<int>(w.swapped ? prob->K : xext),
                                       static_cast<int>(w.swapped ? xext : prob->K), w.swapped,
                                       prob->K, w.rs, prob->C, 8, dW, dwt,
                                       beta != 0.0f ? Cin : nullptr, alpha, beta, s));
}

// Winograd F(2x2, 3x3): output tiles and workspace parts (V [16][T][C],
// U [K][16][C], M [16][T][K], all 16-bit).
struct WinoWs {
  int TH, TW;
  long long T;
  size_t v_bytes, u_bytes, m_bytes, total;
};

bool wino_ws(const igconv_problem_t* pb, int P, int Q, WinoWs* w) {
  w->TH = (P + 1) / 2;
  w->TW = (Q + 1) / 2;
  w->T = static_cast<long long>(pb->N) * w->TH * w->TW;
  if (w->T >= (1LL << 31) || w->T * pb->C >= (1LL << 40) || w->T * pb->K >= (1LL << 40))
    return false;
  w->v_bytes = round256(static_cast<size_t>(16) * w->T * pb->C * 2);
  w->u_bytes = round256(static_cast<size_t>(pb->K) * 16 * pb->C * 2);
  w->m_bytes = round256(static_cast<size_t>(16) * w->T * pb->K * 2);
  w->total = w->v_bytes + w->u_bytes + w->m_bytes;
  return true;
}

bool wino_shape(const igconv_problem_t* pb) {
  return pb->R == 3 && pb->S == 3 && pb->stride_h == 1 && pb->stride_w == 1 && pb->dil_h == 1 &&
         pb->dil_w == 1;
}


// The wgrad GEMM over geometry g (the problem itself, or the few-channel
// packed one, whose X map then has the strides x_strides) into the split
// partials `part`, then the ordered reduction into dW [K][RS][C] of the real
// problem, workspace rows decoded by remap when given.
igconv_status_t run_wgrad(const igconv_problem_t* g, int P, int Q, const WgradPlan& w, int bf16,
                          const void* X, const cuuint64_t* x_strides, const void* dY, void* part,
                          const DeviceState* dev, int RS, int C, const FewPack* remap, void* dW,
                          igconv_dtype_t dw_dtype, const void* Cin, float alpha, float beta,
                          cudaStream_t s) {
  ConvGemmParams p;
  init_common(p, dev);
  p.nsub = 1;
  p.a_src = w.swapped ? SRC_2D_MN : SRC_IM2COL_MN;
  p.b_src = w.swapped ? SRC_IM2COL_MN : SRC_2D_MN;
  p.epi = EPI_PARTIAL;
  p.tiles_m_total = w.tiles_m;
  p.tiles_n = w.tiles_n;
  p.splits = w.splits;
  p.kblocks_total = w.kblocks;
  p.units = w.tiles_m * w.tiles_n * w.splits;
  p.cblocks = w.cblocks;
  p.N_gemm = w.N_pad;
  p.idesc = make_idesc(kBlockM, w.bn, bf16, 1, 1);
  set_fp_accumulators(p, w.bn);
  p.wg_PQ = P * Q;
  p.wg_Q = Q;
  p.wg_lower_h = -g->pad_h;
  p.wg_lower_w = -g->pad_w;
  p.wg_sh = g->stride_h;
  p.wg_sw = g->stride_w;
  p.wg_S = g->S;
  p.wg_RS = w.rs;
  p.wg_dh = g->dil_h;
  p.wg_dw = g->dil_w;
  p.wg_K = g->K;
  p.out = part;
  p.ws_split_stride = static_cast<long long>(w.M_pad) * w.N_pad;
  p.ws_ld = w.N_pad;
  p.use_tma_store = encode_out_2d(&p.mapY, part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                                  static_cast<long long>(w.splits) * w.M_pad, w.N_pad, 16,
                                  CU_TENSOR_MAP_SWIZZLE_64B) ? 1 : 0;
  if (!encode_im2col(&p.mapA[0], X, bf16, g->N, g->H, g->W, g->C, -g->pad_h, -g->pad_w,
                     g->pad_h - (g->R - 1) * g->dil_h, g->pad_w - (g->S - 1) * g->dil_w,
                     g->stride_h, g->stride_w, kBlockK, 64, CU_TENSOR_MAP_SWIZZLE_128B,
                     x_strides))
    return IGCONV_ERR_UNSUPPORTED;
  p.mapA_valid = 1u;
  const long long npq = static_cast<long long>(g->N) * P * Q;
  if (!encode_2d(&p.mapB, dY, bf16, npq, g->K)) return IGCONV_ERR_UNSUPPORTED;
  if (launch_conv_gemm(p, w.bn, grid_for(p.units, dev), s) != cudaSuccess) return cuda_error();
  const int dwt = dw_dtype == IGCONV_F32 ? 2 : (dw_dtype == IGCONV_BF16 ? 1 : 0);
  const int xext = w.rs * w.cpad;
  return from_cuda(launch_wgrad_reduce(static_cast<const float*>(part), w.splits,
                                       p.ws_split_stride, w.N_pad, w.swapped ? g->K : xext,
                                       w.swapped ? xext : g->K, w.swapped, g->K, RS, C, w.cpad,
                                       dW, dwt, beta != 0.0f ? Cin : nullptr, alpha, beta, s,
                                       remap));
}

// wgrad on input halos (conv_wgrad_halo.cu): stride 1, C and K at most 128,
// 2..kHaloTaps taps.  Output positions run on a grid Wt = 32, 64 or 128
// columns wide (the smallest that holds Q + the largest column offset), in
// blocks of 128 positions = 128 / Wt whole output rows, so P must be a
// multiple of 128 / Wt; each block's input halo of HR = 128 / Wt + the
// largest row offset + 1 rows per 64-channel plane and its dY rows per
// 64-channel chunk form one pipeline stage (two or three must fit).  The
// GEMM rows are (tap, plane) entries of 64 rows, two per 128-row M-tile; a
// CTA takes one split of the blocks for a group of M-tiles (as many as fit
// TMEM at N = 64 or 128 columns each, the groups balanced), at most one CTA
// per SM in all; the partial tiles are [split][tiles * 128][N] fp32.
struct WgradHaloPlan {
  int wt, rows, hr, blocks, splits, planes, kchunks, tiles, group_tiles, groups;
  int stage_bytes, stages;
  size_t ws_bytes;
};
bool plan_wgrad_halo(const igconv_problem_t* pb, int P, int Q, int sm_count, WgradHaloPlan* h) {
  if (g_tune_wgrad_halo.load() == 1) return false;
  if (pb->stride_h != 1 || pb->stride_w != 1 || pb->C > 128 || pb->K > 128) return false;
  const int taps = pb->R * pb->S;
  if (taps < 2 || taps > kHaloTaps) return false;
  const int max_h = (pb->R - 1) * pb->dil_h, max_w = (pb->S - 1) * pb->dil_w;
  int wt = 32;
  while (wt < Q + max_w && wt < 256) wt *= 2;
  if (wt > 128 || wt < Q + max_w) return false;
  h->wt = wt;
  h->rows = kBlockM / wt;
  h->hr = h->rows + max_h + 1;
  if (h->hr * wt > kHaloRows || h->hr > 256 || P % h->rows != 0) return false;
  h->planes = ceil_div(pb->C, 64);
  h->kchunks = ceil_div(pb->K, 64);
  h->stage_bytes = h->planes * h->hr * wt * 128 + h->kchunks * kBlockM * 128;
  // stages, epilogue staging (32 KB), barriers and the base alignment in 227 KB
  const int room = 232448 - 32768 - 256 - 1024;
  h->stages = std::min(3, room / h->stage_bytes);
  if (h->stages < 2) return false;
  const long long blocks = static_cast<long long>(pb->N) * (P / h->rows);
  if (blocks < 1 || blocks > INT_MAX) return false;
  h->blocks = static_cast<int>(blocks);
  const int N = 64 * h->kchunks;
  h->tiles = (taps * h->planes + 1) / 2;
  const int max_tiles = std::min(8, 512 / N);
  h->groups = ceil_div(h->tiles, max_tiles);
  h->group_tiles = ceil_div(h->tiles, h->groups);
  const int sms = sm_count > 0 ? sm_count : 148;
  h->splits = std::max(1, std::min(h->blocks, sms / h->groups));
  h->ws_bytes = static_cast<size_t>(h->splits) * h->tiles * kBlockM * N * sizeof(float);
  return true;
}

// Tiled map over an NHWC tensor, box (64 channels, bw pixels, bh rows, 1 image),
// 128-byte swizzle; reads outside the tensor are zero.
bool encode_nhwc_box(CUtensorMap* map, const void* base, int bf16, int N, int H, int W, int C,
                     int bw, int bh) {
  const cuuint64_t px = static_cast<cuuint64_t>(C) * 2;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(W),
                              static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N)};
  const cuuint64_t strides[3] = {px, px * W, px * W * H};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(bw), static_cast<cuuint32_t>(bh), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return g_encode_tiled(map, tma_dtype(bf16), 4, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

igconv_status_t run_wgrad_halo(const igconv_problem_t* g, int P, int Q, const WgradHaloPlan& h,
                               int bf16, const void* X, const void* dY, void* part,
                               const DeviceState* dev, void* dW, igconv_dtype_t dw_dtype,
                               const void* Cin, float alpha, float beta, cudaStream_t s) {
  ConvGemmParams p;
  init_common(p, dev);
  SubProblem& sp = p.sub[0];
  sp.Ws = h.wt;
  sp.Hs = P;
  sp.lower_h = -g->pad_h;
  sp.lower_w = -g->pad_w;
  sp.r0 = 0; sp.rstep = 1; sp.rcount = g->R; sp.offh0 = 0; sp.doffh = g->dil_h;
  sp.s0 = 0; sp.sstep = 1; sp.scount = g->S; sp.offw0 = 0; sp.doffw = g->dil_w;
  const int N = 64 * h.kchunks;
  p.nsub = 1;
  p.epi = EPI_PARTIAL;
  p.splits = h.splits;
  p.kblocks_total = h.blocks;
  p.tiles_m_total = h.tiles;
  p.num_acc = h.group_tiles;
  p.cblocks = h.planes;
  p.tiles_n = h.kchunks;
  p.halo_bytes = h.hr * h.wt * 128;
  p.wh_stage_bytes = h.stage_bytes;
  p.wh_stages = h.stages;
  p.idesc = make_idesc(kBlockM, N, bf16, 1, 1);
  p.out = part;
  if (!encode_nhwc_box(&p.mapA[0], X, bf16, g->N, g->H, g->W, g->C, h.wt, h.hr) ||
      !encode_nhwc_box(&p.mapB, dY, bf16, g->N, P, Q, g->K, h.wt, h.rows) ||
      !encode_out_2d(&p.mapY, part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                     static_cast<long long>(h.splits) * h.tiles * kBlockM, N, 16,
                     CU_TENSOR_MAP_SWIZZLE_64B))
    return IGCONV_ERR_UNSUPPORTED;
  p.mapA_valid = 1u;
  p.use_tma_store = 1;
  if (launch_wgrad_halo(p, s) != cudaSuccess) return cuda_error();
  const int dwt = dw_dtype == IGCONV_F32 ? 2 : (dw_dtype == IGCONV_BF16 ? 1 : 0);
  const int rows = h.tiles * kBlockM;
  return from_cuda(launch_wgrad_reduce(static_cast<const float*>(part), h.splits,
                                       static_cast<long long>(rows) * N, N, rows, N, 0, g->K,
                                       g->R * g->S, g->C, 64 * h.planes, dW, dwt,
                                       beta != 0.0f ? Cin : nullptr, alpha, beta, s, nullptr));
}

}  // namespace

extern "C" {

const char* igconv_status_string(igconv_status_t s) {
  switch (s) {
    case IGCONV_OK: return "IGCONV_OK";
    case IGCONV_ERR_INVALID_ARG: return "IGCONV_ERR_INVALID_ARG";
    case IGCONV_ERR_UNSUPPORTED: return "IGCONV_ERR_UNSUPPORTED";
    case IGCONV_ERR_MISALIGNED: return "IGCONV_ERR_MISALIGNED";
    case IGCONV_ERR_WORKSPACE: return "IGCONV_ERR_WORKSPACE";
    case IGCONV_ERR_CUDA: return "IGCONV_ERR_CUDA";
    case IGCONV_ERR_DEVICE_TIMEOUT: return "IGCONV_ERR_DEVICE_TIMEOUT";
  }
  return "IGCONV_UNKNOWN_STATUS";
}

igconv_status_t conv2d_output_size(const igconv_problem_t* prob, int* P, int* Q) {
  if (!P || !Q) return IGCONV_ERR_INVALID_ARG;
  return check_shape(prob, P, Q);
}

igconv_status_t igconv_set_tuning(igconv_tune_key_t key, int value) {
  switch (key) {
    case IGCONV_TUNE_WGRAD_SPLITS:
      if (value < 0) return IGCONV_ERR_INVALID_ARG;
      g_tune_splits.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_BLOCK_N:
      if (value != 0 && value != 64 && value != 128 && value != 256) return IGCONV_ERR_INVALID_ARG;
      g_tune_bn.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_MAX_CTAS:
      if (value < 0) return IGCONV_ERR_INVALID_ARG;
      g_tune_max_ctas.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_CTA_PAIRS:
      if (value < 0 || value > 2) return IGCONV_ERR_INVALID_ARG;
      g_tune_no_pairs.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_EPI_GROUPS:
      if (value < 0 || value > 2) return IGCONV_ERR_INVALID_ARG;
      g_tune_epi_groups.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_CONV_SPLITS:
      if (value < 0 || value > 16) return IGCONV_ERR_INVALID_ARG;
      g_tune_conv_splits.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_FEW_CHANNELS:
      if (value < 0 || value > 1) return IGCONV_ERR_INVALID_ARG;
      g_tune_few_channels.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_RASTER:
      if (value < 0 || value > 64) return IGCONV_ERR_INVALID_ARG;
      g_tune_raster.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_RESIDENT_FILTER:
      if (value < 0 || value > 1) return IGCONV_ERR_INVALID_ARG;
      g_tune_resident_b.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_DGRAD_ROWS:
      if (value < 0 || value > 1) return IGCONV_ERR_INVALID_ARG;
      g_tune_dgrad_rows.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_EPILOGUE_KERNEL:
      if (value < 0 || value > 1) return IGCONV_ERR_INVALID_ARG;
      g_tune_general_epi.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_HALO:
      if (value < 0 || value > 1) return IGCONV_ERR_INVALID_ARG;
      g_tune_halo.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_ONE_ISSUER:
      if (value < 0 || value > 1) return IGCONV_ERR_INVALID_ARG;
      g_tune_one_issuer.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_WGRAD_HALO:
      if (value < 0 || value > 1) return IGCONV_ERR_INVALID_ARG;
      g_tune_wgrad_halo.store(value);
      return IGCONV_OK;
    case IGCONV_TUNE_PDL:
      if (value < 0 || value > 1) return IGCONV_ERR_INVALID_ARG;
      g_tune_pdl.store(value);
      return IGCONV_OK;
  }
  return IGCONV_ERR_INVALID_ARG;
}

size_t conv2d_fprop_workspace_size(const igconv_problem_t* prob, igconv_dtype_t dtype) {
  int P = 0, Q = 0;
  if (check_shape(prob, &P, &Q) != IGCONV_OK) return 0;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return 0;
  if (prob->C <= 8) {
    FewPack f;
    if (few_pack_plan(prob, P, Q, &f)) {
      const FewPackWs pw = few_pack_ws(prob, f);
      return pw.z_bytes + pw.w_bytes;
    }
    return few_channel_ws(prob).total;
  }
  // split-K partials, when the plan splits (the same decision as conv2d_fprop_ws)
  const int sms = current_sm_count();
  const long long tiles_m = ceil_div(static_cast<long long>(prob->N) * P * Q, kBlockM);
  const int bn = choose_block_n(prob->K, tiles_m, sms);
  if (bn == 128 && g_tune_no_pairs.load() != 1 && g_tune_conv_splits.load() < 2 && tiles_m >= 2)
    return 0;  // CTA pairs, no split
  const int kb = prob->R * prob->S * ceil_div(prob->C, kBlockK);
  const int splits = conv_split_count(tiles_m * ceil_div(prob->K, bn), kb, sms);
  if (splits < 2) return 0;
  return static_cast<size_t>(splits) * tiles_m * kBlockM * static_cast<size_t>(ceil_div(prob->K, bn)) *
         bn * sizeof(float);
}

igconv_status_t conv2d_fprop(const igconv_problem_t* prob, igconv_dtype_t dtype, const void* X,
                             const void* Wt, const void* bias, const void* Cin, void* Y,
                             float alpha, float beta, int relu, void* stream) {
  return conv2d_fprop_ws(prob, dtype, X, Wt, bias, Cin, Y, alpha, beta, relu, nullptr, 0, stream);
}

igconv_status_t conv2d_fprop_ws(const igconv_problem_t* prob, igconv_dtype_t dtype,
                                const void* X, const void* Wt, const void* bias, const void* Cin,
                                void* Y, float alpha, float beta, int relu, void* workspace,
                                size_t workspace_bytes, void* stream) {
  int P = 0, Q = 0;
  igconv_status_t st = check_shape(prob, &P, &Q);
  if (st != IGCONV_OK) return st;
  if (!X || !Wt || !Y || (beta != 0.0f && !Cin)) return IGCONV_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return IGCONV_ERR_INVALID_ARG;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return IGCONV_ERR_UNSUPPORTED;
  // few channels: C < 8 always, C == 8 when a workspace is given; packed
  // (space-to-depth, FewPack) where few_pack_plan allows, else tap-packed
  const bool few = prob->C < 8 || (prob->C == 8 && workspace != nullptr);
  FewPack fpk{};
  const bool packed = few && few_pack_plan(prob, P, Q, &fpk);
  igconv_problem_t vp = packed ? few_pack_problem(prob, fpk) : *prob;
  if (few) {
    igconv_problem_t k8 = *prob;
    k8.C = 8;  // the limits apply to the padded pixels; K must still be a multiple of 8
    if ((st = check_limits(packed ? &vp : &k8, P, Q, 8)) != IGCONV_OK) return st;
    const size_t need = packed ? few_pack_ws(prob, fpk).z_bytes + few_pack_ws(prob, fpk).w_bytes
                               : few_channel_ws(prob).total;
    if (!workspace || workspace_bytes < need) return IGCONV_ERR_WORKSPACE;
    if (!aligned16(workspace) || !aligned16(Y) || (bias && !aligned16(bias)) ||
        (beta != 0.0f && !aligned16(Cin)) || (prob->C == 8 && !aligned16(X)) ||
        (reinterpret_cast<uintptr_t>(X) & 1) || (reinterpret_cast<uintptr_t>(Wt) & 1))
      return IGCONV_ERR_MISALIGNED;
  } else {
    if ((st = check_limits(prob, P, Q, 8)) != IGCONV_OK) return st;
    if (!aligned16(X) || !aligned16(Wt) || !aligned16(Y) || (bias && !aligned16(bias)) ||
        (beta != 0.0f && !aligned16(Cin)))
      return IGCONV_ERR_MISALIGNED;
  }
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  ConvGemmParams p;
  init_common(p, dev);
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  const int bn = choose_block_n(prob->K, ceil_div(static_cast<long long>(prob->N) * P * Q, kBlockM),
                                dev->sm_count);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const void* gW = Wt;  // the filter the GEMM reads
  if (packed) {
    const FewPackWs pw = few_pack_ws(prob, fpk);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* Zp = ws;
    void* Wpk = ws + pw.z_bytes;
    if (launch_few_pack_x(X, Zp, fpk, prob->N, prob->H, prob->W, cs) != cudaSuccess ||
        launch_few_pack_filter(Wt, Wpk, fpk, prob->K, 64, cs) != cudaSuccess)
      return cuda_error();
    if ((st = plan_fprop(p, bn, &vp, P, Q, bf16, Zp, Wpk, pw.strides)) != IGCONV_OK) return st;
    gW = Wpk;
  } else if (few) {
    const FewChannelWs fw = few_channel_ws(prob);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const void* X8 = X;
    if (prob->C < 8) {
      if (launch_pad_pixels8(X, ws, static_cast<long long>(prob->N) * prob->H * prob->W,
                             prob->C, cs) != cudaSuccess)
        return cuda_error();
      X8 = ws;
    }
    void* Wt8 = ws + fw.x_bytes;
    if (launch_filter_taps8(Wt, Wt8, prob->K, prob->R * prob->S, prob->C, bn, cs) != cudaSuccess)
      return cuda_error();
    if ((st = plan_fprop_taps(p, bn, prob, P, Q, bf16, X8, Wt8)) != IGCONV_OK) return st;
  } else if ((st = plan_fprop(p, bn, prob, P, Q, bf16, X, Wt)) != IGCONV_OK) {
    return st;
  }
  int splits = 1;
  if (!few && workspace && !aligned16(workspace)) return IGCONV_ERR_MISALIGNED;
  if (!few && workspace && !(g_tune_conv_splits.load() < 2 && use_pairs(bn, p.sub[0].tiles_m, false))) {
    splits = conv_split_count(static_cast<long long>(p.sub[0].tiles_m) * p.tiles_n,
                              p.sub[0].rcount * p.sub[0].scount * p.cblocks, dev->sm_count);
    if (splits > 1 && workspace_bytes < conv_split_bytes(p, bn, splits)) return IGCONV_ERR_WORKSPACE;
  }
  if ((!few || packed) && splits == 1 && use_pairs(bn, p.sub[0].tiles_m, false)) {
    // 256-row units; each CTA of a pair loads bn/2 filter rows
    p.pair = 1;
    p.units = ceil_div(p.sub[0].tiles_m, 2) * p.tiles_n;
    p.idesc = make_idesc(2 * kBlockM, bn, bf16, 0, 0);
    if (!encode_filter(&p.mapB, gW, bf16, vp.K, vp.R, vp.S, vp.C, bn / 2))
      return IGCONV_ERR_UNSUPPORTED;
  }
  p.epi = EPI_STORE;
  p.out = Y;
  if (!few && splits == 1 && !p.pair && prob->stride_h == 1 && prob->stride_w == 1 &&
      try_halo_plan(p, bn, X, prob->N, prob->H, prob->W, prob->C, P, Q, bf16)) {
    // halo plan: grid rows are whole output rows
    set_out_map_lines_5d(p, Y, prob->N, P, Q, prob->K, 1, 1, bf16, bn,
                         p.sub[0].rcount * p.sub[0].scount * p.cblocks);
  } else {
    // output tile rows are consecutive pixels: store them with TMA
    if (splits == 1) choose_one_issuer(p, bn);
    set_out_map_16(p, Y, static_cast<long long>(prob->N) * P * Q, prob->K, bf16, bn,
                   p.sub[0].rcount * p.sub[0].scount * p.cblocks);
  }
  if (!few) {  // the few-channel filter copy was just written: it is in L2
    p.pf_base = Wt;
    p.pf_bytes = static_cast<long long>(prob->K) * prob->R * prob->S * prob->C * 2;
  }
  p.cin = beta != 0.0f ? Cin : nullptr;
  p.bias = bias;
  p.bias_cached = bias != nullptr && prob->K * 4 <= kBiasCacheBytes ? 1 : 0;
  p.alpha = alpha;
  p.beta = beta;
  p.relu = relu ? 1 : 0;
  p.out_bf16 = bf16;
  if (splits > 1) {
    set_conv_split(p, bn, splits, workspace);
    if (launch_conv_gemm(p, bn, grid_for(p.units, dev), cs) != cudaSuccess) return cuda_error();
    return from_cuda(launch_conv_splitk_reduce(
        static_cast<const float*>(workspace), splits, p.ws_split_stride, p.ws_ld,
        static_cast<long long>(prob->N) * P * Q, prob->K, Y, bf16,
        beta != 0.0f ? Cin : nullptr, bias, alpha, beta, relu ? 1 : 0, cs));
  }
  const int grid = p.pair ? grid_for_pairs(p.units, bn, dev) : grid_for(p.units, dev);
  return from_cuda(launch_conv_gemm(p, bn, grid, cs));
}

// Epilogue settings and launch of a planned dgrad.
static igconv_status_t launch_dgrad_plan(ConvGemmParams& p, int bn, const igconv_problem_t* prob,
                                         void* dX, const void* Cin, float alpha, float beta,
                                         int bf16, const DeviceState* dev, cudaStream_t stream) {
  p.epi = EPI_STORE;
  p.out = dX;
  choose_one_issuer(p, bn);  // whichever way the rows are stored
  if (p.halo) {
    // halo plan: grid rows are whole dX rows
    set_out_map_lines_5d(p, dX, prob->N, prob->H, prob->W, prob->C, 1, 1, bf16, bn,
                         p.sub[0].rcount * p.sub[0].scount * p.cblocks);
  } else if (prob->stride_h == 1 && prob->stride_w == 1) {
    // one sub-problem whose tile rows are consecutive input pixels
    set_out_map_16(p, dX, static_cast<long long>(prob->N) * prob->H * prob->W, prob->C, bf16,
                   bn, p.sub[0].rcount * p.sub[0].scount * p.cblocks);
  } else if (p.store_5d) {
    // residue classes on one padded grid: 32-row boxes through the 5D view
    int kb = 0;
    for (int i = 0; i < p.nsub; ++i)
      kb = std::max(kb, p.sub[i].rcount * p.sub[i].scount * p.cblocks);
    set_out_map_lines_5d(p, dX, prob->N, prob->H, prob->W, prob->C, prob->stride_h,
                         prob->stride_w, bf16, bn, kb);
  }
  p.cin = beta != 0.0f ? Cin : nullptr;
  p.bias = nullptr;
  p.alpha = alpha;
  p.beta = beta;
  p.relu = 0;
  p.out_bf16 = bf16;
  if (p.units == 0) return IGCONV_OK;
  const int grid = p.pair ? grid_for_pairs(p.units, bn, dev) : grid_for(p.units, dev);
  return from_cuda(launch_conv_gemm(p, bn, grid, stream));
}

igconv_status_t conv2d_dgrad(const igconv_problem_t* prob, igconv_dtype_t dtype, const void* dY,
                             const void* Wt, const void* Cin, void* dX, float alpha, float beta,
                             void* stream) {
  return conv2d_dgrad_ws(prob, dtype, dY, Wt, Cin, dX, alpha, beta, nullptr, 0, stream);
}

size_t conv2d_dgrad_workspace_size(const igconv_problem_t* prob, igconv_dtype_t dtype) {
  int P = 0, Q = 0;
  if (check_shape(prob, &P, &Q) != IGCONV_OK) return 0;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return 0;
  if (prob->C < 8) {
    FewPack f;
    if (few_pack_plan_dgrad(prob, P, Q, &f)) return few_dgrad_pack_ws(prob, f).total;
    return few_dgrad_ws(prob).total;
  }
  if (prob->stride_h != 1 || prob->stride_w != 1) return 0;
  const int sms = current_sm_count();
  const long long tiles_m = ceil_div(static_cast<long long>(prob->N) * prob->H * prob->W, kBlockM);
  const int bn = choose_block_n(prob->C, tiles_m, sms);
  if (bn == 128 && g_tune_no_pairs.load() != 1 && g_tune_conv_splits.load() < 2 && tiles_m >= 2)
    return 0;
  const int kb = prob->R * prob->S * ceil_div(prob->K, kBlockK);
  const int splits = conv_split_count(tiles_m * ceil_div(prob->C, bn), kb, sms);
  if (splits < 2) return 0;
  return static_cast<size_t>(splits) * tiles_m * kBlockM * static_cast<size_t>(ceil_div(prob->C, bn)) *
         bn * sizeof(float);
}

igconv_status_t conv2d_dgrad_ws(const igconv_problem_t* prob, igconv_dtype_t dtype,
                                const void* dY, const void* Wt, const void* Cin, void* dX,
                                float alpha, float beta, void* workspace, size_t workspace_bytes,
                                void* stream) {
  int P = 0, Q = 0;
  igconv_status_t st = check_shape(prob, &P, &Q);
  if (st != IGCONV_OK) return st;
  if (!dY || !Wt || !dX || (beta != 0.0f && !Cin)) return IGCONV_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return IGCONV_ERR_INVALID_ARG;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return IGCONV_ERR_UNSUPPORTED;
  FewPack fdp{};
  if (prob->C < 8 && few_pack_plan_dgrad(prob, P, Q, &fdp)) {
    // few input channels at dilation 1: the dgrad of the stride-1 packed
    // problem (filter repacked to [K][R2][S2][cz]) written as alpha * acc in
    // fp32, then each X element's gradient gathered from its packed position
    // and finished with beta * Cin and the cast
    igconv_problem_t vd = *prob;
    vd.H = fdp.Hz;
    vd.W = fdp.Wz;
    vd.C = fdp.cz;
    vd.R = fdp.R2;
    vd.S = fdp.Sv;
    vd.pad_h = vd.pad_w = 0;
    vd.stride_h = vd.stride_w = 1;
    vd.dil_h = vd.dil_w = 1;
    if ((st = check_limits(&vd, P, Q, 8)) != IGCONV_OK) return st;
    if (!aligned16(dY) || (reinterpret_cast<uintptr_t>(Wt) & 1) ||
        (reinterpret_cast<uintptr_t>(dX) & 1) ||
        (beta != 0.0f && (reinterpret_cast<uintptr_t>(Cin) & 1)) ||
        (workspace && !aligned16(workspace)))
      return IGCONV_ERR_MISALIGNED;
    const FewDgradPackWs fw = few_dgrad_pack_ws(prob, fdp);
    if (!workspace || workspace_bytes < fw.total) return IGCONV_ERR_WORKSPACE;
    DeviceState* dev = nullptr;
    if ((st = device_state(&dev)) != IGCONV_OK) return st;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* Wz = ws;
    float* dz = reinterpret_cast<float*>(ws + fw.w_bytes);
    const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (launch_few_pack_filter(Wt, Wz, fdp, prob->K, fdp.cz, cs) != cudaSuccess)
      return cuda_error();
    ConvGemmParams p;
    init_common(p, dev);
    int bn = 0;
    if ((st = plan_dgrad(p, &bn, &vd, P, Q, bf16, dY, Wz, dev->sm_count)) != IGCONV_OK) return st;
    p.epi = EPI_STORE;
    p.out_f32 = 1;
    p.out = dz;
    p.use_tma_store = 0;
    p.alpha = alpha;
    p.out_bf16 = bf16;
    p.pf_base = Wz;
    p.pf_bytes = static_cast<long long>(prob->K) * fdp.R2 * fdp.Sv * fdp.cz * 2;
    if (p.units > 0 && launch_conv_gemm(p, bn, grid_for(p.units, dev), cs) != cudaSuccess)
      return cuda_error();
    return from_cuda(launch_few_unpack_dx(dz, dX, fdp, prob->N, prob->H, prob->W, bf16,
                                          beta != 0.0f ? Cin : nullptr, beta, cs));
  }
  if (prob->C < 8) {
    // few input channels (with dilation, or the tap-packed knob): the dense
    // dgrad over the filter padded to 8 channels, alpha * acc written as fp32
    // rows of 8 channels, then the C real channels finished with beta * Cin
    // and the cast
    igconv_problem_t k8 = *prob;
    k8.C = 8;
    if ((st = check_limits(&k8, P, Q, 8)) != IGCONV_OK) return st;
    if (prob->stride_h * prob->stride_w > kMaxSub) return IGCONV_ERR_UNSUPPORTED;
    if (!aligned16(dY) || (reinterpret_cast<uintptr_t>(Wt) & 1) ||
        (reinterpret_cast<uintptr_t>(dX) & 1) ||
        (beta != 0.0f && (reinterpret_cast<uintptr_t>(Cin) & 1)) ||
        (workspace && !aligned16(workspace)))
      return IGCONV_ERR_MISALIGNED;
    const FewDgradWs fw = few_dgrad_ws(prob);
    if (!workspace || workspace_bytes < fw.total) return IGCONV_ERR_WORKSPACE;
    DeviceState* dev = nullptr;
    if ((st = device_state(&dev)) != IGCONV_OK) return st;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* W8 = ws;
    float* dX8 = reinterpret_cast<float*>(ws + fw.w_bytes);
    const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (launch_pad_pixels8(Wt, W8, static_cast<long long>(prob->K) * prob->R * prob->S, prob->C,
                           cs) != cudaSuccess)
      return cuda_error();
    ConvGemmParams p;
    init_common(p, dev);
    int bn = 0;
    if ((st = plan_dgrad(p, &bn, &k8, P, Q, bf16, dY, W8, dev->sm_count)) != IGCONV_OK) return st;
    p.epi = EPI_STORE;
    p.out_f32 = 1;
    p.out = dX8;
    p.use_tma_store = 0;
    p.alpha = alpha;
    p.out_bf16 = bf16;
    p.pf_base = W8;
    p.pf_bytes = static_cast<long long>(prob->K) * prob->R * prob->S * 16;
    if (p.units > 0 && launch_conv_gemm(p, bn, grid_for(p.units, dev), cs) != cudaSuccess)
      return cuda_error();
    return from_cuda(launch_unpad_channels(dX8, dX,
                                           static_cast<long long>(prob->N) * prob->H * prob->W,
                                           prob->C, bf16, beta != 0.0f ? Cin : nullptr, beta, cs));
  }
  if ((st = check_limits(prob, P, Q, 8)) != IGCONV_OK) return st;
  if (prob->stride_h * prob->stride_w > kMaxSub) return IGCONV_ERR_UNSUPPORTED;
  if (!aligned16(dY) || !aligned16(Wt) || !aligned16(dX) || (beta != 0.0f && !aligned16(Cin)))
    return IGCONV_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  ConvGemmParams p;
  init_common(p, dev);
  int bn = 0;
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  if ((st = plan_dgrad(p, &bn, prob, P, Q, bf16, dY, Wt, dev->sm_count, 0, true)) != IGCONV_OK)
    return st;
  if (workspace && !aligned16(workspace)) return IGCONV_ERR_MISALIGNED;
  const bool unit_stride = prob->stride_h == 1 && prob->stride_w == 1 && p.nsub == 1;
  int splits = 1;
  if (workspace && unit_stride &&
      !(g_tune_conv_splits.load() < 2 && use_pairs(bn, p.sub[0].tiles_m, true))) {
    splits = conv_split_count(static_cast<long long>(p.sub[0].tiles_m) * p.tiles_n,
                              p.sub[0].rcount * p.sub[0].scount * p.cblocks, dev->sm_count);
    if (splits > 1 && workspace_bytes < conv_split_bytes(p, bn, splits)) return IGCONV_ERR_WORKSPACE;
  }
  if (splits > 1) {
    set_conv_split(p, bn, splits, workspace);
    p.alpha = 1.0f;
    p.pf_base = Wt;
    p.pf_bytes = static_cast<long long>(prob->K) * prob->R * prob->S * prob->C * 2;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (launch_conv_gemm(p, bn, grid_for(p.units, dev), cs) != cudaSuccess) return cuda_error();
    return from_cuda(launch_conv_splitk_reduce(
        static_cast<const float*>(workspace), splits, p.ws_split_stride, p.ws_ld,
        static_cast<long long>(prob->N) * prob->H * prob->W, prob->C, dX, bf16,
        beta != 0.0f ? Cin : nullptr, nullptr, alpha, beta, 0, cs));
  }
  if (p.nsub == 1 && p.sub[0].tile_begin == 0 && use_pairs(bn, p.sub[0].tiles_m, true)) {
    // 256-row units; each CTA of a pair loads one 64-column half of the filter tile
    p.pair = 1;
    p.units = ceil_div(p.sub[0].tiles_m, 2) * p.tiles_n;
    p.idesc = make_idesc(2 * kBlockM, bn, bf16, 0, 1);
  } else if (unit_stride) {
    try_halo_plan(p, bn, dY, prob->N, P, Q, prob->K, prob->H, prob->W, bf16);
  }
  p.pf_base = Wt;
  p.pf_bytes = static_cast<long long>(prob->K) * prob->R * prob->S * prob->C * 2;
  return launch_dgrad_plan(p, bn, prob, dX, Cin, alpha, beta, bf16, dev,
                           static_cast<cudaStream_t>(stream));
}

size_t conv2d_wgrad_workspace_size(const igconv_problem_t* prob, igconv_dtype_t dtype,
                                   igconv_dtype_t dw_dtype) {
  int P = 0, Q = 0;
  if (check_shape(prob, &P, &Q) != IGCONV_OK) return 0;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return 0;
  if (dw_dtype != IGCONV_F16 && dw_dtype != IGCONV_BF16 && dw_dtype != IGCONV_F32) return 0;
  int sm_count = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      sm_count = v;
  } else {
    cudaGetLastError();  // no device: size for the default SM count
  }
  WgradPlan w;
  if (prob->C < 8) {
    FewPack f;
    if (few_pack_plan(prob, P, Q, &f)) {  // the packed image, then the partials
      const igconv_problem_t vp = few_pack_problem(prob, f);
      plan_wgrad_shape(&vp, P, Q, sm_count, &w);
      return few_pack_ws(prob, f).z_bytes + w.ws_bytes;
    }
    // the 8-channel pixel copy, then the partials
    plan_wgrad_taps(prob, P, Q, sm_count, &w);
    return round256(static_cast<size_t>(prob->N) * prob->H * prob->W * 16) + w.ws_bytes;
  }
  plan_wgrad_shape(prob, P, Q, sm_count, &w);
  WgradHaloPlan hp;
  if (plan_wgrad_halo(prob, P, Q, sm_count, &hp) && hp.ws_bytes > w.ws_bytes) return hp.ws_bytes;
  return w.ws_bytes;
}

igconv_status_t conv2d_wgrad(const igconv_problem_t* prob, igconv_dtype_t dtype,
                             igconv_dtype_t dw_dtype, const void* X, const void* dY,
                             const void* Cin, void* dW, float alpha, float beta, void* workspace,
                             size_t workspace_bytes, void* stream) {
  int P = 0, Q = 0;
  igconv_status_t st = check_shape(prob, &P, &Q);
  if (st != IGCONV_OK) return st;
  if (!X || !dY || !dW || (beta != 0.0f && !Cin)) return IGCONV_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return IGCONV_ERR_INVALID_ARG;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return IGCONV_ERR_UNSUPPORTED;
  if (dw_dtype != IGCONV_F16 && dw_dtype != IGCONV_BF16 && dw_dtype != IGCONV_F32)
    return IGCONV_ERR_UNSUPPORTED;
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  FewPack fpk{};
  if (prob->C < 8 && few_pack_plan(prob, P, Q, &fpk)) {
    // few channels, packed: the space-to-depth image, then the dense wgrad
    // of the packed problem, its rows decoded back to (tap, c)
    const igconv_problem_t vp = few_pack_problem(prob, fpk);
    if ((st = check_limits(&vp, P, Q, 8)) != IGCONV_OK) return st;
    const uintptr_t esz = dw_dtype == IGCONV_F32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(X) & 1) || !aligned16(dY) ||
        (reinterpret_cast<uintptr_t>(dW) & (esz - 1)) ||
        (beta != 0.0f && (reinterpret_cast<uintptr_t>(Cin) & (esz - 1))) ||
        (workspace && !aligned16(workspace)))
      return IGCONV_ERR_MISALIGNED;
    DeviceState* dev = nullptr;
    if ((st = device_state(&dev)) != IGCONV_OK) return st;
    WgradPlan w;
    plan_wgrad_shape(&vp, P, Q, dev->sm_count, &w);
    const FewPackWs pw = few_pack_ws(prob, fpk);
    if (!workspace || workspace_bytes < pw.z_bytes + w.ws_bytes) return IGCONV_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (launch_few_pack_x(X, ws, fpk, prob->N, prob->H, prob->W, s) != cudaSuccess)
      return cuda_error();
    return run_wgrad(&vp, P, Q, w, bf16, ws, pw.strides, dY, ws + pw.z_bytes, dev,
                     prob->R * prob->S, prob->C, &fpk, dW, dw_dtype, Cin, alpha, beta, s);
  }
  if (prob->C < 8) return wgrad_few_channels(prob, P, Q, dtype, dw_dtype, X, dY, Cin, dW, alpha,
                                             beta, workspace, workspace_bytes, stream);
  if ((st = check_limits(prob, P, Q, 8)) != IGCONV_OK) return st;
  if (!aligned16(X) || !aligned16(dY) || !aligned16(dW) || (beta != 0.0f && !aligned16(Cin)) ||
      (workspace && !aligned16(workspace)))
    return IGCONV_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  WgradHaloPlan hp;
  if (plan_wgrad_halo(prob, P, Q, dev->sm_count, &hp) && workspace &&
      workspace_bytes >= hp.ws_bytes)  // (a smaller workspace takes the plan below)
    return run_wgrad_halo(prob, P, Q, hp, bf16, X, dY, workspace, dev, dW, dw_dtype, Cin, alpha,
                          beta, s);
  WgradPlan w;
  plan_wgrad_shape(prob, P, Q, dev->sm_count, &w);
  if (!workspace || workspace_bytes < w.ws_bytes) return IGCONV_ERR_WORKSPACE;
  return run_wgrad(prob, P, Q, w, bf16, X, nullptr, dY, workspace, dev, w.rs, prob->C, nullptr,
                   dW, dw_dtype, Cin, alpha, beta, s);
}

// ---------------------------------------------------------------------------
// Grouped convolution: groups == 1 is the dense path, groups == C == K the
// depthwise kernels.
// ---------------------------------------------------------------------------
igconv_status_t conv2d_grouped_fprop(const igconv_problem_t* prob, int groups,
                                     igconv_dtype_t dtype, const void* X, const void* Wt,
                                     const void* bias, const void* Cin, void* Y, float alpha,
                                     float beta, int relu, void* stream) {
  bool direct = false;
  int cg = 1;
  igconv_status_t st = check_groups(prob, groups, &direct, &cg);
  if (st != IGCONV_OK) return st;
  if (!direct) return conv2d_fprop(prob, dtype, X, Wt, bias, Cin, Y, alpha, beta, relu, stream);
  int P = 0, Q = 0;
  if ((st = check_shape(prob, &P, &Q)) != IGCONV_OK) return st;
  if (!X || !Wt || !Y || (beta != 0.0f && !Cin)) return IGCONV_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return IGCONV_ERR_INVALID_ARG;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return IGCONV_ERR_UNSUPPORTED;
  if ((st = check_limits(prob, P, Q, 8)) != IGCONV_OK) return st;
  if (!aligned16(X) || !aligned16(Wt) || !aligned16(Y) || (bias && !aligned16(bias)) ||
      (beta != 0.0f && !aligned16(Cin)))
    return IGCONV_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  DwParams p;
  if ((st = plan_dw(p, dev, prob, DW_MODE_FWD, bf16, cg, P, Q)) != IGCONV_OK) return st;
  p.w = Wt;
  p.bias = bias;
  p.cin = beta != 0.0f ? Cin : nullptr;
  p.out = Y;
  p.relu = relu ? 1 : 0;
  p.alpha = alpha;
  p.beta = beta;
  p.org_h = -prob->pad_h;
  p.org_w = -prob->pad_w;
  p.tiles = static_cast<long long>(p.tiles_p) * p.tiles_q * p.chunks;
  if (!encode_nhwc_window(&p.map_in, X, bf16, prob->N, prob->H, prob->W, prob->C, p.iw_t,
                          p.ih_t))
    return IGCONV_ERR_UNSUPPORTED;
  cudaError_t e = cudaSuccess;
  const int grid = dw_grid(p, dev, &e);
  if (e != cudaSuccess) return cuda_error();
  return from_cuda(launch_depthwise(p, grid, static_cast<cudaStream_t>(stream)));
}

// Grouped convolution on the tensor cores: an implicit GEMM with 64-wide
// tiles of whole groups, tile n reducing over its group window of the
// other side's channels (plan_group_window) against a dense block-diagonal
// filter image [K][R][S][C] in the workspace.  Any C / K ratio whose windows
// plan_group_window accepts (multiples of 8 channels); for C == K the
// widths 1 and 2 stay with the direct kernels.  dgrad's tiles run over C,
// fprop's and wgrad's over K.
static bool grouped_gemm_ok(const igconv_problem_t* prob, int groups, bool dgrad,
                            GroupWin* win = nullptr) {
  if (!prob || groups < 2 || prob->C < 1 || prob->K < 1) return false;
  if (prob->C % groups != 0 || prob->K % groups != 0) return false;
  if (prob->C % 8 != 0 || prob->K % 8 != 0) return false;
  const int cg = prob->C / groups, kg = prob->K / groups;
  if (prob->C == prob->K && cg < 4) return false;
  GroupWin w;
  if (!plan_group_window(dgrad ? cg : kg, dgrad ? kg : cg, &w)) return false;
  if (win) *win = w;
  return true;
}

static size_t grouped_filter_bytes(const igconv_problem_t* prob) {
  return round256(static_cast<size_t>(prob->K) * prob->R * prob->S * prob->C * 2);
}

size_t conv2d_grouped_fprop_workspace_size(const igconv_problem_t* prob, int groups,
                                           igconv_dtype_t dtype) {
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return 0;
  if (!prob || groups < 1 || prob->C < 1 || prob->K < 1 || prob->R < 1 || prob->S < 1) return 0;
  if (groups == 1) return conv2d_fprop_workspace_size(prob, dtype);
  if (!grouped_gemm_ok(prob, groups, false)) return 0;
  return grouped_filter_bytes(prob);
}

igconv_status_t conv2d_grouped_fprop_ws(const igconv_problem_t* prob, int groups,
                                        igconv_dtype_t dtype, const void* X, const void* Wt,
                                        const void* bias, const void* Cin, void* Y, float alpha,
                                        float beta, int relu, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (!prob || groups < 1) return IGCONV_ERR_INVALID_ARG;
  if (groups == 1)
    return conv2d_fprop_ws(prob, dtype, X, Wt, bias, Cin, Y, alpha, beta, relu, workspace,
                           workspace_bytes, stream);
  if (prob->C < 1 || prob->K < 1 || prob->C % groups != 0 || prob->K % groups != 0)
    return IGCONV_ERR_INVALID_ARG;
  GroupWin win;
  if (!grouped_gemm_ok(prob, groups, false, &win))  // depthwise, width 2, or uncovered
    return conv2d_grouped_fprop(prob, groups, dtype, X, Wt, bias, Cin, Y, alpha, beta, relu,
                                stream);
  int P = 0, Q = 0;
  igconv_status_t st = check_shape(prob, &P, &Q);
  if (st != IGCONV_OK) return st;
  if (!X || !Wt || !Y || (beta != 0.0f && !Cin)) return IGCONV_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return IGCONV_ERR_INVALID_ARG;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return IGCONV_ERR_UNSUPPORTED;
  if ((st = check_limits(prob, P, Q, 8)) != IGCONV_OK) return st;
  const size_t need = conv2d_grouped_fprop_workspace_size(prob, groups, dtype);
  if (!workspace || workspace_bytes < need) return IGCONV_ERR_WORKSPACE;
  if (!aligned16(X) || !aligned16(Wt) || !aligned16(Y) || !aligned16(workspace) ||
      (bias && !aligned16(bias)) || (beta != 0.0f && !aligned16(Cin)))
    return IGCONV_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (launch_group_filter_dense(Wt, workspace, prob->K, prob->R * prob->S, prob->C,
                                prob->C / groups, prob->K / groups, cs) != cudaSuccess)
    return cuda_error();
  constexpr int bn = 64;
  ConvGemmParams p;
  init_common(p, dev);
  // the dense plan over the block-diagonal filter, with each tile's
  // reduction cut down to its group window
  if ((st = plan_fprop(p, bn, prob, P, Q, bf16, X, workspace)) != IGCONV_OK) return st;
  p.cblocks = win.blocks;
  p.grp_mul = win.mul;
  p.grp_div = win.div;
  p.epi = EPI_STORE;
  p.out = Y;
  set_out_map_16(p, Y, static_cast<long long>(prob->N) * P * Q, prob->K, bf16, bn,
                 p.sub[0].rcount * p.sub[0].scount * p.cblocks);
  p.cin = beta != 0.0f ? Cin : nullptr;
  p.bias = bias;
  p.bias_cached = bias != nullptr && prob->K * 4 <= kBiasCacheBytes ? 1 : 0;
  p.alpha = alpha;
  p.beta = beta;
  p.relu = relu ? 1 : 0;
  p.out_bf16 = bf16;
  return from_cuda(launch_conv_gemm(p, bn, grid_for(p.units, dev), cs));
}

igconv_status_t conv2d_grouped_dgrad(const igconv_problem_t* prob, int groups,
                                     igconv_dtype_t dtype, const void* dY, const void* Wt,
                                     const void* Cin, void* dX, float alpha, float beta,
                                     void* stream) {
  bool direct = false;
  int cg = 1;
  igconv_status_t st = check_groups(prob, groups, &direct, &cg);
  if (st != IGCONV_OK) return st;
  if (!direct) return conv2d_dgrad(prob, dtype, dY, Wt, Cin, dX, alpha, beta, stream);
  int P = 0, Q = 0;
  if ((st = check_shape(prob, &P, &Q)) != IGCONV_OK) return st;
  if (!dY || !Wt || !dX || (beta != 0.0f && !Cin)) return IGCONV_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return IGCONV_ERR_INVALID_ARG;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return IGCONV_ERR_UNSUPPORTED;
  if ((st = check_limits(prob, P, Q, 8)) != IGCONV_OK) return st;
  if (!aligned16(dY) || !aligned16(Wt) || !aligned16(dX) || (beta != 0.0f && !aligned16(Cin)))
    return IGCONV_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  const bool unit = prob->stride_h == 1 && prob->stride_w == 1;
  DwParams p;
  // stride 1: dX[h][w] = sum_{r,s} dY[h + ph - r*dh][w + pw - s*dw] * W[r][s], a
  // forward pass over dY with the filter flipped and origin ph - (R-1)*dh;
  // otherwise the phase kernel
  if ((st = plan_dw(p, dev, prob, unit ? DW_MODE_FWD : DW_MODE_PHASE, bf16, cg, prob->H,
                    prob->W)) != IGCONV_OK)
    return st;
  p.wt_transposed = cg > 1 ? 1 : 0;
  if (unit) {
    p.flip = 1;
    p.org_h = prob->pad_h - (prob->R - 1) * prob->dil_h;
    p.org_w = prob->pad_w - (prob->S - 1) * prob->dil_w;
  } else {
    build_phase_tables(p, prob);
  }
  p.w = Wt;
  p.cin = beta != 0.0f ? Cin : nullptr;
  p.out = dX;
  p.alpha = alpha;
  p.beta = beta;
  p.tiles = static_cast<long long>(p.tiles_p) * p.tiles_q * p.chunks;
  if (!encode_nhwc_window(&p.map_in, dY, bf16, prob->N, P, Q, prob->C, p.iw_t, p.ih_t))
    return IGCONV_ERR_UNSUPPORTED;
  cudaError_t e = cudaSuccess;
  const int grid = dw_grid(p, dev, &e);
  if (e != cudaSuccess) return cuda_error();
  return from_cuda(launch_depthwise(p, grid, static_cast<cudaStream_t>(stream)));
}

size_t conv2d_grouped_dgrad_workspace_size(const igconv_problem_t* prob, int groups,
                                           igconv_dtype_t dtype) {
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return 0;
  if (!prob || groups < 2 || prob->R < 1 || prob->S < 1) return 0;
  if (!grouped_gemm_ok(prob, groups, true)) return 0;
  return grouped_filter_bytes(prob);
}

// Grouped dgrad on the tensor cores: the dgrad implicit GEMM (residue-class
// sub-problems for strides) with 64-wide tiles in which dX channel tile n
// reduces over dY channel block n only, against the same block-diagonal
// filter image as the grouped fprop (read MN-major, rows 64n..).
igconv_status_t conv2d_grouped_dgrad_ws(const igconv_problem_t* prob, int groups,
                                        igconv_dtype_t dtype, const void* dY, const void* Wt,
                                        const void* Cin, void* dX, float alpha, float beta,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  if (!prob || groups < 1) return IGCONV_ERR_INVALID_ARG;
  if (prob->C < 1 || prob->K < 1 || prob->C % groups != 0 || prob->K % groups != 0)
    return IGCONV_ERR_INVALID_ARG;
  GroupWin win;
  if (!grouped_gemm_ok(prob, groups, true, &win))  // dense, depthwise, width 2, or uncovered
    return conv2d_grouped_dgrad(prob, groups, dtype, dY, Wt, Cin, dX, alpha, beta, stream);
  int P = 0, Q = 0;
  igconv_status_t st = check_shape(prob, &P, &Q);
  if (st != IGCONV_OK) return st;
  if (!dY || !Wt || !dX || (beta != 0.0f && !Cin)) return IGCONV_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return IGCONV_ERR_INVALID_ARG;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return IGCONV_ERR_UNSUPPORTED;
  if ((st = check_limits(prob, P, Q, 8)) != IGCONV_OK) return st;
  if (prob->stride_h * prob->stride_w > kMaxSub) return IGCONV_ERR_UNSUPPORTED;
  const size_t need = conv2d_grouped_dgrad_workspace_size(prob, groups, dtype);
  if (!workspace || workspace_bytes < need) return IGCONV_ERR_WORKSPACE;
  if (!aligned16(dY) || !aligned16(Wt) || !aligned16(dX) || !aligned16(workspace) ||
      (beta != 0.0f && !aligned16(Cin)))
    return IGCONV_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (launch_group_filter_dense(Wt, workspace, prob->K, prob->R * prob->S, prob->C,
                                prob->C / groups, prob->K / groups, cs) != cudaSuccess)
    return cuda_error();
  ConvGemmParams p;
  init_common(p, dev);
  int bn = 64;
  // the dense dgrad plan over the block-diagonal filter (read MN-major),
  // each dX channel tile reducing over its window of dY channels
  if ((st = plan_dgrad(p, &bn, prob, P, Q, bf16, dY, workspace, dev->sm_count, 64, true)) !=
      IGCONV_OK)
    return st;
  p.cblocks = win.blocks;
  p.grp_mul = win.mul;
  p.grp_div = win.div;
  p.pf_base = workspace;
  p.pf_bytes = static_cast<long long>(prob->K) * prob->R * prob->S * prob->C * 2;
  return launch_dgrad_plan(p, bn, prob, dX, Cin, alpha, beta, bf16, dev, cs);
}

// Grouped wgrad on the tensor cores: the wgrad GEMM whose rows are (tap,
// X channel of the output tile's group window) and whose 64-wide column
// tiles are output channels, split-K partials reduced in order into the
// gradient of the windowed filter [K][R][S][cpad], whose group entries are
// then copied out (with beta * Cin and the cast).
static igconv_status_t grouped_wgrad_gemm(const igconv_problem_t* prob, int groups, int P, int Q,
                                          int bf16, igconv_dtype_t dw_dtype, const void* X,
                                          const void* dY, const void* Cin, void* dW, float alpha,
                                          float beta, void* workspace, size_t workspace_bytes,
                                          const DeviceState* dev, cudaStream_t s) {
  GroupWin win;
  if (!grouped_gemm_ok(prob, groups, false, &win)) return IGCONV_ERR_UNSUPPORTED;
  WgradPlan w;
  plan_wgrad_grouped(prob, P, Q, dev->sm_count, win, &w);
  if (!workspace || workspace_bytes < grouped_wgrad_gemm_bytes(w, prob))
    return IGCONV_ERR_WORKSPACE;
  ConvGemmParams p;
  init_common(p, dev);
  p.nsub = 1;
  p.a_src = SRC_IM2COL_MN;
  p.b_src = SRC_2D_MN;
  p.epi = EPI_PARTIAL;
  p.tiles_m_total = w.tiles_m;
  p.tiles_n = w.tiles_n;
  p.splits = w.splits;
  p.kblocks_total = w.kblocks;
  p.units = w.tiles_m * w.tiles_n * w.splits;
  p.cblocks = w.cblocks;
  p.grp_mul = win.mul;
  p.grp_div = win.div;
  p.N_gemm = w.N_pad;
  p.idesc = make_idesc(kBlockM, w.bn, bf16, 1, 1);
  set_fp_accumulators(p, w.bn);
  p.wg_PQ = P * Q;
  p.wg_Q = Q;
  p.wg_lower_h = -prob->pad_h;
  p.wg_lower_w = -prob->pad_w;
  p.wg_sh = prob->stride_h;
  p.wg_sw = prob->stride_w;
  p.wg_S = prob->S;
  p.wg_RS = w.rs;
  p.wg_dh = prob->dil_h;
  p.wg_dw = prob->dil_w;
  p.wg_K = prob->K;
  p.out = workspace;
  p.ws_split_stride = static_cast<long long>(w.M_pad) * w.N_pad;
  p.ws_ld = w.N_pad;
  p.use_tma_store = encode_out_2d(&p.mapY, workspace, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                                  static_cast<long long>(w.splits) * w.M_pad, w.N_pad, 16,
                                  CU_TENSOR_MAP_SWIZZLE_64B) ? 1 : 0;
  if (!encode_im2col(&p.mapA[0], X, bf16, prob->N, prob->H, prob->W, prob->C, -prob->pad_h,
                     -prob->pad_w, prob->pad_h - (prob->R - 1) * prob->dil_h,
                     prob->pad_w - (prob->S - 1) * prob->dil_w, prob->stride_h, prob->stride_w,
                     kBlockK))
    return IGCONV_ERR_UNSUPPORTED;
  p.mapA_valid = 1u;
  const long long npq = static_cast<long long>(prob->N) * P * Q;
  if (!encode_2d(&p.mapB, dY, bf16, npq, prob->K)) return IGCONV_ERR_UNSUPPORTED;
  cudaError_t e = launch_conv_gemm(p, w.bn, grid_for(p.units, dev), s);
  if (e != cudaSuccess) return cuda_error();
  float* dwexp = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + round256(w.ws_bytes));
  e = launch_wgrad_reduce(static_cast<const float*>(workspace), w.splits, p.ws_split_stride,
                          w.N_pad, w.rs * w.cpad, prob->K, 0, prob->K, w.rs, w.cpad, w.cpad,
                          dwexp, 2, nullptr, alpha, 0.0f, s);
  if (e != cudaSuccess) return cuda_error();
  const int dwt = dw_dtype == IGCONV_F32 ? 2 : (dw_dtype == IGCONV_BF16 ? 1 : 0);
  return from_cuda(launch_group_extract(dwexp, dW, dwt, beta != 0.0f ? Cin : nullptr, beta,
                                        prob->K, w.rs, prob->C / groups, prob->K / groups,
                                        w.cpad, win.mul, win.div, s));
}

size_t conv2d_grouped_wgrad_workspace_size(const igconv_problem_t* prob, int groups,
                                           igconv_dtype_t dtype, igconv_dtype_t dw_dtype) {
  bool direct = false;
  int cg = 1;
  // widths above 32 and C != K have only the tensor-core path
  if (check_groups(prob, groups, &direct, &cg) != IGCONV_OK &&
      !grouped_gemm_ok(prob, groups, false))
    return 0;
  if (!direct) return conv2d_wgrad_workspace_size(prob, dtype, dw_dtype);
  int P = 0, Q = 0;
  if (check_shape(prob, &P, &Q) != IGCONV_OK) return 0;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return 0;
  DeviceState* dev = nullptr;
  if (device_state(&dev) != IGCONV_OK) return 0;
  GroupWin win;
  if (grouped_gemm_ok(prob, groups, false, &win)) {
    WgradPlan w;
    plan_wgrad_grouped(prob, P, Q, dev->sm_count, win, &w);
    return grouped_wgrad_gemm_bytes(w, prob);
  }
  DwParams p;
  if (plan_dw_wgrad(p, dev, prob, P, Q, dtype == IGCONV_BF16 ? 1 : 0, cg) != IGCONV_OK) return 0;
  return dw_wgrad_ws_bytes(p);
}

igconv_status_t conv2d_grouped_wgrad(const igconv_problem_t* prob, int groups,
                                     igconv_dtype_t dtype, igconv_dtype_t dw_dtype, const void* X,
                                     const void* dY, const void* Cin, void* dW, float alpha,
                                     float beta, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  bool direct = false;
  int cg = 1;
  igconv_status_t st = check_groups(prob, groups, &direct, &cg);
  // widths above 32 and C != K have only the tensor-core path
  if (st != IGCONV_OK && !(st == IGCONV_ERR_UNSUPPORTED && grouped_gemm_ok(prob, groups, false)))
    return st;
  if (!direct)
    return conv2d_wgrad(prob, dtype, dw_dtype, X, dY, Cin, dW, alpha, beta, workspace,
                        workspace_bytes, stream);
  int P = 0, Q = 0;
  if ((st = check_shape(prob, &P, &Q)) != IGCONV_OK) return st;
  if (!X || !dY || !dW || (beta != 0.0f && !Cin)) return IGCONV_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return IGCONV_ERR_INVALID_ARG;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return IGCONV_ERR_UNSUPPORTED;
  if (dw_dtype != IGCONV_F16 && dw_dtype != IGCONV_BF16 && dw_dtype != IGCONV_F32)
    return IGCONV_ERR_UNSUPPORTED;
  if ((st = check_limits(prob, P, Q, 8)) != IGCONV_OK) return st;
  if (!aligned16(X) || !aligned16(dY) || !aligned16(dW) || (beta != 0.0f && !aligned16(Cin)) ||
      (workspace && !aligned16(workspace)))
    return IGCONV_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  if (grouped_gemm_ok(prob, groups, false))
    return grouped_wgrad_gemm(prob, groups, P, Q, bf16, dw_dtype, X, dY, Cin, dW, alpha, beta,
                              workspace, workspace_bytes, dev, static_cast<cudaStream_t>(stream));
  DwParams p;
  if ((st = plan_dw_wgrad(p, dev, prob, P, Q, bf16, cg)) != IGCONV_OK) return st;
  if (!workspace || workspace_bytes < dw_wgrad_ws_bytes(p)) return IGCONV_ERR_WORKSPACE;
  p.ws = static_cast<float*>(workspace);
  if (!encode_nhwc_window(&p.map_in, X, bf16, prob->N, prob->H, prob->W, prob->C, p.iw_t,
                          p.ih_t))
    return IGCONV_ERR_UNSUPPORTED;
  // dY: two boxes of 8 rows x (tq + 1) columns per tile
  if (!encode_nhwc_window(&p.map_dy, dY, bf16, prob->N, P, Q, prob->C, p.tq + 1, kDwHalfRows))
    return IGCONV_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int grid = p.chunks * p.splits * (cg > 1 ? prob->R * prob->S : 1);
  cudaError_t e = launch_depthwise(p, grid, s);
  if (e != cudaSuccess) return cuda_error();
  const int dwt = dw_dtype == IGCONV_F32 ? 2 : (dw_dtype == IGCONV_BF16 ? 1 : 0);
  e = launch_dw_wgrad_reduce(p.ws, p.splits, prob->R * prob->S, prob->C, cg, dW, dwt,
                             beta != 0.0f ? Cin : nullptr, alpha, beta, s);
  return from_cuda(e);
}

// ---------------------------------------------------------------------------
// 3D forward convolution
// ---------------------------------------------------------------------------
// im2col map over an NDHWC 16-bit tensor: `pixels` positions x 64 channels
// per load, 128-byte swizzle; lower / upper corners and traversal strides
// in (w, h, d) order.
static bool encode_im2col_5d(CUtensorMap* map, const void* base, int bf16, int n, int d, int h,
                             int w, int c, const int lower[3], const int upper[3],
                             const int trav[3], int pixels) {
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(c), static_cast<cuuint64_t>(w),
                              static_cast<cuuint64_t>(h), static_cast<cuuint64_t>(d),
                              static_cast<cuuint64_t>(n)};
  const cuuint64_t row = static_cast<cuuint64_t>(c) * 2;
  const cuuint64_t strides[4] = {row, row * w, row * w * h, row * w * h * d};
  const cuuint32_t estr[5] = {1, static_cast<cuuint32_t>(trav[0]), static_cast<cuuint32_t>(trav[1]),
                              static_cast<cuuint32_t>(trav[2]), 1};
  const CUresult r = g_encode_im2col(map, tma_dtype(bf16), 5, const_cast<void*>(base), dims,
                                     strides, lower, upper, static_cast<cuuint32_t>(kBlockK),
                                     static_cast<cuuint32_t>(pixels), estr,
                                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Limits shared by the 3D passes (else UNSUPPORTED): channel multiples of 8,
// strides <= 8, pads and dil*(k-1) <= 15 (the 5D im2col bounding box), N and
// element counts as in 2D.
static igconv_status_t check_limits3d(const igconv_problem3d_t* prob, int Do, int P, int Q) {
  if (prob->C % 8 != 0 || prob->K % 8 != 0) return IGCONV_ERR_UNSUPPORTED;
  const int ks[3] = {prob->T, prob->R, prob->S};
  const int pads[3] = {prob->pad_d, prob->pad_h, prob->pad_w};
  const int strides[3] = {prob->stride_d, prob->stride_h, prob->stride_w};
  const int dils[3] = {prob->dil_d, prob->dil_h, prob->dil_w};
  for (int i = 0; i < 3; ++i) {
    if (strides[i] > 8 || pads[i] > 15) return IGCONV_ERR_UNSUPPORTED;
    if (static_cast<long long>(dils[i]) * (ks[i] - 1) > 15) return IGCONV_ERR_UNSUPPORTED;
  }
  if (prob->N > 65535) return IGCONV_ERR_UNSUPPORTED;
  const long long in_pix = static_cast<long long>(prob->N) * prob->D * prob->H * prob->W;
  const long long out_pix = static_cast<long long>(prob->N) * Do * P * Q;
  if (in_pix >= (1LL << 31) || out_pix >= (1LL << 31)) return IGCONV_ERR_UNSUPPORTED;
  if (in_pix * prob->C >= (1LL << 40) || out_pix * prob->K >= (1LL << 40))
    return IGCONV_ERR_UNSUPPORTED;
  if (static_cast<long long>(prob->T) * prob->R > 65535) return IGCONV_ERR_UNSUPPORTED;
  return IGCONV_OK;
}

static igconv_status_t check_shape3d(const igconv_problem3d_t* pb, int* Do, int* P, int* Q) {
  if (!pb) return IGCONV_ERR_INVALID_ARG;
  if (pb->N < 1 || pb->D < 1 || pb->H < 1 || pb->W < 1 || pb->C < 1 || pb->K < 1 || pb->T < 1 ||
      pb->R < 1 || pb->S < 1)
    return IGCONV_ERR_INVALID_ARG;
  if (pb->pad_d < 0 || pb->pad_h < 0 || pb->pad_w < 0 || pb->stride_d < 1 || pb->stride_h < 1 ||
      pb->stride_w < 1 || pb->dil_d < 1 || pb->dil_h < 1 || pb->dil_w < 1)
    return IGCONV_ERR_INVALID_ARG;
  const long long d = out_extent(pb->D, pb->pad_d, pb->dil_d, pb->T, pb->stride_d);
  const long long p = out_extent(pb->H, pb->pad_h, pb->dil_h, pb->R, pb->stride_h);
  const long long q = out_extent(pb->W, pb->pad_w, pb->dil_w, pb->S, pb->stride_w);
  if (d < 1 || p < 1 || q < 1 || d > INT32_MAX || p > INT32_MAX || q > INT32_MAX)
    return IGCONV_ERR_INVALID_ARG;
  if (Do) *Do = static_cast<int>(d);
  if (P) *P = static_cast<int>(p);
  if (Q) *Q = static_cast<int>(q);
  return IGCONV_OK;
}

igconv_status_t conv3d_output_size(const igconv_problem3d_t* prob, int* Do, int* P, int* Q) {
  if (!Do || !P || !Q) return IGCONV_ERR_INVALID_ARG;
  return check_shape3d(prob, Do, P, Q);
}

igconv_status_t conv3d_fprop(const igconv_problem3d_t* prob, igconv_dtype_t dtype, const void* X,
                             const void* Wt, const void* bias, const void* Cin, void* Y,
                             float alpha, float beta, int relu, void* stream) {
  int Do = 0, P = 0, Q = 0;
  igconv_status_t st = check_shape3d(prob, &Do, &P, &Q);
  if (st != IGCONV_OK) return st;
  if (!X || !Wt || !Y || (beta != 0.0f && !Cin)) return IGCONV_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return IGCONV_ERR_INVALID_ARG;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return IGCONV_ERR_UNSUPPORTED;
  if ((st = check_limits3d(prob, Do, P, Q)) != IGCONV_OK) return st;
  const long long out_pix = static_cast<long long>(prob->N) * Do * P * Q;
  if (!aligned16(X) || !aligned16(Wt) || !aligned16(Y) || (bias && !aligned16(bias)) ||
      (beta != 0.0f && !aligned16(Cin)))
    return IGCONV_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  const int bn = choose_block_n(prob->K, ceil_div(out_pix, kBlockM), dev->sm_count);
  ConvGemmParams p;
  init_common(p, dev);
  SubProblem& sp = p.sub[0];
  sp.M = static_cast<int>(out_pix);
  sp.tile_begin = 0;
  sp.tiles_m = ceil_div(out_pix, kBlockM);
  sp.Hs = P;
  sp.Ws = Q;
  sp.Ds = Do;
  sp.lower_h = -prob->pad_h;
  sp.lower_w = -prob->pad_w;
  sp.lower_d = -prob->pad_d;
  sp.trav_h = prob->stride_h;
  sp.trav_w = prob->stride_w;
  sp.trav_d = prob->stride_d;
  // the r taps run over the merged (t, r) index of the [K][T*R][S][C] filter view
  sp.r0 = 0; sp.rstep = 1; sp.rcount = prob->T * prob->R; sp.offh0 = 0; sp.doffh = prob->dil_h;
  sp.s0 = 0; sp.sstep = 1; sp.scount = prob->S; sp.offw0 = 0; sp.doffw = prob->dil_w;
  sp.rdiv = prob->R;
  sp.doffd = prob->dil_d;
  sp.tstride = prob->R;
  sp.offd0 = 0;
  sp.out_h0 = 0; sp.out_w0 = 0; sp.out_sh = 1; sp.out_sw = 1;
  sp.out_d0 = 0; sp.out_sd = 1;
  p.nsub = 1;
  p.a_src = SRC_IM2COL_K3;
  p.b_src = SRC_W_K;
  p.cblocks = ceil_div(prob->C, kBlockK);
  p.N_gemm = prob->K;
  p.tiles_n = ceil_div(prob->K, bn);
  p.units = sp.tiles_m * p.tiles_n;
  p.out_C = prob->K;
  p.out_D = Do;
  p.out_H = P;
  p.out_W = Q;
  p.idesc = make_idesc(kBlockM, bn, bf16, 0, 0);
  set_fp_accumulators(p, bn);
  {
    const int lower[3] = {-prob->pad_w, -prob->pad_h, -prob->pad_d};
    const int upper[3] = {prob->pad_w - (prob->S - 1) * prob->dil_w,
                          prob->pad_h - (prob->R - 1) * prob->dil_h,
                          prob->pad_d - (prob->T - 1) * prob->dil_d};
    const int trav[3] = {prob->stride_w, prob->stride_h, prob->stride_d};
    if (!encode_im2col_5d(&p.mapA[0], X, bf16, prob->N, prob->D, prob->H, prob->W, prob->C, lower,
                          upper, trav, kBlockM))
      return IGCONV_ERR_UNSUPPORTED;
  }
  p.mapA_valid = 1u;
  if (!encode_filter(&p.mapB, Wt, bf16, prob->K, prob->T * prob->R, prob->S, prob->C, bn))
    return IGCONV_ERR_UNSUPPORTED;
  p.epi = EPI_STORE;
  p.out = Y;
  set_out_map_16(p, Y, out_pix, prob->K, bf16, bn, sp.rcount * sp.scount * p.cblocks);
  p.pf_base = Wt;
  p.pf_bytes = static_cast<long long>(prob->K) * prob->T * prob->R * prob->S * prob->C * 2;
  p.cin = beta != 0.0f ? Cin : nullptr;
  p.bias = bias;
  p.bias_cached = bias != nullptr && prob->K * 4 <= kBiasCacheBytes ? 1 : 0;
  p.alpha = alpha;
  p.beta = beta;
  p.relu = relu ? 1 : 0;
  p.out_bf16 = bf16;
  return from_cuda(launch_conv_gemm(p, bn, grid_for(p.units, dev),
                                    static_cast<cudaStream_t>(stream)));
}

// 3D data gradient: the implicit GEMM over the 5D im2col of dY, one
// sub-problem per output residue class (o mod sd, h mod sh, w mod sw) as in
// the 2D dgrad, each with the taps whose offsets divide by the strides.
igconv_status_t conv3d_dgrad(const igconv_problem3d_t* prob, igconv_dtype_t dtype, const void* dY,
                             const void* Wt, const void* Cin, void* dX, float alpha, float beta,
                             void* stream) {
  int Do = 0, P = 0, Q = 0;
  igconv_status_t st = check_shape3d(prob, &Do, &P, &Q);
  if (st != IGCONV_OK) return st;
  if (!dY || !Wt || !dX || (beta != 0.0f && !Cin)) return IGCONV_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return IGCONV_ERR_INVALID_ARG;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return IGCONV_ERR_UNSUPPORTED;
  if ((st = check_limits3d(prob, Do, P, Q)) != IGCONV_OK) return st;
  if (prob->stride_d * prob->stride_h * prob->stride_w > kMaxSub) return IGCONV_ERR_UNSUPPORTED;
  if (!aligned16(dY) || !aligned16(Wt) || !aligned16(dX) || (beta != 0.0f && !aligned16(Cin)))
    return IGCONV_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  const long long in_pix = static_cast<long long>(prob->N) * prob->D * prob->H * prob->W;
  const int bn = choose_block_n(prob->C, ceil_div(in_pix, kBlockM), dev->sm_count);
  ConvGemmParams p;
  init_common(p, dev);
  p.tiles_n = ceil_div(prob->C, bn);
  int nsub = 0, tile_begin = 0;
  for (int rd = 0; rd < prob->stride_d; ++rd) {
    const Residue1D dd = residue_1d(rd, prob->D, prob->T, prob->pad_d, prob->stride_d,
                                    prob->dil_d);
    if (dd.count == 0) continue;
    for (int rh = 0; rh < prob->stride_h; ++rh) {
      const Residue1D dh = residue_1d(rh, prob->H, prob->R, prob->pad_h, prob->stride_h,
                                      prob->dil_h);
      if (dh.count == 0) continue;
      for (int rw = 0; rw < prob->stride_w; ++rw) {
        const Residue1D dw = residue_1d(rw, prob->W, prob->S, prob->pad_w, prob->stride_w,
                                        prob->dil_w);
        if (dw.count == 0) continue;
        SubProblem& sp = p.sub[nsub];
        const long long M = static_cast<long long>(prob->N) * dd.count * dh.count * dw.count;
        sp.M = static_cast<int>(M);
        sp.tile_begin = tile_begin;
        sp.tiles_m = ceil_div(M, kBlockM);
        sp.Ds = dd.count;
        sp.Hs = dh.count;
        sp.Ws = dw.count;
        sp.lower_d = dd.delta_min;
        sp.lower_h = dh.delta_min;
        sp.lower_w = dw.delta_min;
        sp.trav_d = 1;
        sp.trav_h = 1;
        sp.trav_w = 1;
        const bool taps = dd.rcount > 0 && dh.rcount > 0 && dw.rcount > 0;
        // merged (t, r) taps: filter row (t0 + jt*tstep) * R + r0 + jr*rstep
        sp.rdiv = dh.rcount > 0 ? dh.rcount : 1;
        sp.rcount = taps ? dd.rcount * dh.rcount : 0;
        sp.r0 = dd.r0 * prob->R + dh.r0;
        sp.tstride = dd.rstep * prob->R;
        sp.rstep = dh.rstep;
        sp.offd0 = dd.off0;
        sp.doffd = dd.doff;
        sp.offh0 = dh.off0;
        sp.doffh = dh.doff;
        sp.s0 = dw.r0; sp.sstep = dw.rstep; sp.scount = taps ? dw.rcount : 1;
        sp.offw0 = dw.off0; sp.doffw = dw.doff;
        sp.out_d0 = dd.h0;
        sp.out_h0 = dh.h0;
        sp.out_w0 = dw.h0;
        sp.out_sd = prob->stride_d;
        sp.out_sh = prob->stride_h;
        sp.out_sw = prob->stride_w;
        if (taps) {
          // base positions [delta_min, delta_min + count - 1] over dY [Do][P][Q]
          const int lower[3] = {dw.delta_min, dh.delta_min, dd.delta_min};
          const int upper[3] = {dw.count - Q + dw.delta_min, dh.count - P + dh.delta_min,
                                dd.count - Do + dd.delta_min};
          const int trav[3] = {1, 1, 1};
          if (!encode_im2col_5d(&p.mapA[nsub], dY, bf16, prob->N, Do, P, Q, prob->K, lower,
                                upper, trav, kBlockM))
            return IGCONV_ERR_UNSUPPORTED;
          p.mapA_valid |= 1u << nsub;
        }
        tile_begin += sp.tiles_m * p.tiles_n;
        ++nsub;
      }
    }
  }
  p.nsub = nsub;
  p.units = tile_begin;
  p.a_src = SRC_IM2COL_K3;
  p.b_src = SRC_W_MN;
  p.cblocks = ceil_div(prob->K, kBlockK);
  p.N_gemm = prob->C;
  p.out_C = prob->C;
  p.out_D = prob->D;
  p.out_H = prob->H;
  p.out_W = prob->W;
  p.idesc = make_idesc(kBlockM, bn, bf16, 0, 1);
  set_fp_accumulators(p, bn);
  if (!encode_filter(&p.mapB, Wt, bf16, prob->K, prob->T * prob->R, prob->S, prob->C, 64))
    return IGCONV_ERR_UNSUPPORTED;
  p.epi = EPI_STORE;
  p.out = dX;
  if (prob->stride_d == 1 && prob->stride_h == 1 && prob->stride_w == 1) {
    // one sub-problem whose tile rows are consecutive input positions
    set_out_map_16(p, dX, in_pix, prob->C, bf16, bn,
                   p.sub[0].rcount * p.sub[0].scount * p.cblocks);
  }
  p.pf_base = Wt;
  p.pf_bytes = static_cast<long long>(prob->K) * prob->T * prob->R * prob->S * prob->C * 2;
  p.cin = beta != 0.0f ? Cin : nullptr;
  p.bias = nullptr;
  p.alpha = alpha;
  p.beta = beta;
  p.relu = 0;
  p.out_bf16 = bf16;
  if (p.units == 0) return IGCONV_OK;
  return from_cuda(launch_conv_gemm(p, bn, grid_for(p.units, dev),
                                    static_cast<cudaStream_t>(stream)));
}

// The 3D weight gradient is the 2D wgrad GEMM with the merged tap (t, r)
// and the output positions (n, o, p, q): plan it on the 2D shape with
// R' = T*R and P' = Do*P.
static void plan_wgrad3d(const igconv_problem3d_t* prob, int Do, int P, int Q, int sms,
                         WgradPlan* w) {
  igconv_problem_t f;
  std::memset(&f, 0, sizeof(f));
  f.N = prob->N;
  f.H = prob->H;
  f.W = prob->W;
  f.C = prob->C;
  f.K = prob->K;
  f.R = prob->T * prob->R;
  f.S = prob->S;
  f.stride_h = f.stride_w = f.dil_h = f.dil_w = 1;
  plan_wgrad_shape(&f, Do * P, Q, sms, w);
}

size_t conv3d_wgrad_workspace_size(const igconv_problem3d_t* prob, igconv_dtype_t dtype,
                                   igconv_dtype_t dw_dtype) {
  int Do = 0, P = 0, Q = 0;
  if (check_shape3d(prob, &Do, &P, &Q) != IGCONV_OK) return 0;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return 0;
  if (dw_dtype != IGCONV_F16 && dw_dtype != IGCONV_BF16 && dw_dtype != IGCONV_F32) return 0;
  DeviceState* dev = nullptr;
  if (device_state(&dev) != IGCONV_OK) return 0;
  WgradPlan w;
  plan_wgrad3d(prob, Do, P, Q, dev->sm_count, &w);
  return w.ws_bytes;
}

igconv_status_t conv3d_wgrad(const igconv_problem3d_t* prob, igconv_dtype_t dtype,
                             igconv_dtype_t dw_dtype, const void* X, const void* dY,
                             const void* Cin, void* dW, float alpha, float beta, void* workspace,
                             size_t workspace_bytes, void* stream) {
  int Do = 0, P = 0, Q = 0;
  igconv_status_t st = check_shape3d(prob, &Do, &P, &Q);
  if (st != IGCONV_OK) return st;
  if (!X || !dY || !dW || (beta != 0.0f && !Cin)) return IGCONV_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return IGCONV_ERR_INVALID_ARG;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return IGCONV_ERR_UNSUPPORTED;
  if (dw_dtype != IGCONV_F16 && dw_dtype != IGCONV_BF16 && dw_dtype != IGCONV_F32)
    return IGCONV_ERR_UNSUPPORTED;
  if ((st = check_limits3d(prob, Do, P, Q)) != IGCONV_OK) return st;
  if (!aligned16(X) || !aligned16(dY) || !aligned16(dW) || (beta != 0.0f && !aligned16(Cin)) ||
      (workspace && !aligned16(workspace)))
    return IGCONV_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  WgradPlan w;
  plan_wgrad3d(prob, Do, P, Q, dev->sm_count, &w);
  if (!workspace || workspace_bytes < w.ws_bytes) return IGCONV_ERR_WORKSPACE;
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  ConvGemmParams p;
  init_common(p, dev);
  p.nsub = 1;
  p.a_src = w.swapped ? SRC_2D_MN : SRC_IM2COL_MN;
  p.b_src = w.swapped ? SRC_IM2COL_MN : SRC_2D_MN;
  p.epi = EPI_PARTIAL;
  p.tiles_m_total = w.tiles_m;
  p.tiles_n = w.tiles_n;
  p.splits = w.splits;
  p.kblocks_total = w.kblocks;
  p.units = w.tiles_m * w.tiles_n * w.splits;
  p.cblocks = w.cblocks;
  p.N_gemm = w.N_pad;
  p.idesc = make_idesc(kBlockM, w.bn, bf16, 1, 1);
  set_fp_accumulators(p, w.bn);
  p.wg_PQ = P * Q;
  p.wg_Q = Q;
  p.wg_lower_h = -prob->pad_h;
  p.wg_lower_w = -prob->pad_w;
  p.wg_sh = prob->stride_h;
  p.wg_sw = prob->stride_w;
  p.wg_S = prob->S;
  p.wg_RS = w.rs;
  p.wg_dh = prob->dil_h;
  p.wg_dw = prob->dil_w;
  p.wg_K = prob->K;
  p.wg_Do = Do;
  p.wg_lower_d = -prob->pad_d;
  p.wg_sd = prob->stride_d;
  p.wg_dd = prob->dil_d;
  p.wg_R = prob->R;
  p.out = workspace;
  p.ws_split_stride = static_cast<long long>(w.M_pad) * w.N_pad;
  p.ws_ld = w.N_pad;
  p.use_tma_store = encode_out_2d(&p.mapY, workspace, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                                  static_cast<long long>(w.splits) * w.M_pad, w.N_pad, 16,
                                  CU_TENSOR_MAP_SWIZZLE_64B) ? 1 : 0;
  {
    const int lower[3] = {-prob->pad_w, -prob->pad_h, -prob->pad_d};
    const int upper[3] = {prob->pad_w - (prob->S - 1) * prob->dil_w,
                          prob->pad_h - (prob->R - 1) * prob->dil_h,
                          prob->pad_d - (prob->T - 1) * prob->dil_d};
    const int trav[3] = {prob->stride_w, prob->stride_h, prob->stride_d};
    if (!encode_im2col_5d(&p.mapA[0], X, bf16, prob->N, prob->D, prob->H, prob->W, prob->C, lower,
                          upper, trav, kBlockK))
      return IGCONV_ERR_UNSUPPORTED;
  }
  p.mapA_valid = 1u;
  const long long npq = static_cast<long long>(prob->N) * Do * P * Q;
  if (!encode_2d(&p.mapB, dY, bf16, npq, prob->K)) return IGCONV_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_conv_gemm(p, w.bn, grid_for(p.units, dev), s);
  if (e != cudaSuccess) return cuda_error();
  const int dwt = dw_dtype == IGCONV_F32 ? 2 : (dw_dtype == IGCONV_BF16 ? 1 : 0);
  const int xext = w.rs * w.cpad;
  e = launch_wgrad_reduce(static_cast<const float*>(workspace), w.splits, p.ws_split_stride,
                          w.N_pad, w.swapped ? prob->K : xext, w.swapped ? xext : prob->K,
                          w.swapped, prob->K, w.rs, prob->C, w.cpad, dW, dwt,
                          beta != 0.0f ? Cin : nullptr, alpha, beta, s);
  return from_cuda(e);
}

// Tile width, accumulator groups and split count of the int8 fprop.  Each
// TMEM accumulator sums at most 16 reduction blocks (1024 products of
// magnitude <= 2^14: integers below 2^24, exact in fp32), NI issuers deal
// the blocks round-robin, and two TMEM buffers of NI * groups accumulators
// must fit in the 512 columns.  The tile width shrinks until a tile's whole
// reduction fits; when not even 64-wide tiles hold it (R*S*C above 4096),
// the reduction is cut into equal ranges of at most 64 blocks whose exact
// int32 partial tiles an ordered reduction adds before the requantisation.
struct Int8FpropPlan {
  int bn, groups, splits, kb_unit;  // kb_unit: most blocks one unit reduces
};
Int8FpropPlan plan_int8_fprop(const igconv_problem_t* prob, int P, int Q, int sm_count) {
  Int8FpropPlan ip;
  const int kblocks = prob->R * prob->S * ceil_div(prob->C, kBlockK);
  ip.bn = choose_block_n(prob->K, ceil_div(static_cast<long long>(prob->N) * P * Q, kBlockM),
                         sm_count);
  ip.splits = 1;
  for (;;) {
    const int ni = issuers_for(ip.bn);
    ip.kb_unit = ceil_div(kblocks, ip.splits);
    ip.groups = ceil_div(ceil_div(ip.kb_unit, ni), 16);
    if (2 * ni * ip.groups * ip.bn <= 512) break;
    if (ip.bn > 64) {
      ip.bn >>= 1;
      continue;
    }
    // 64-wide tiles: two issuers x two groups of 16 blocks = 64 blocks a unit
    ip.splits = ceil_div(kblocks, 2 * 2 * 16);
  }
  return ip;
}

size_t int8_fprop_split_bytes(const igconv_problem_t* prob, int P, int Q, const Int8FpropPlan& ip) {
  if (ip.splits < 2) return 0;
  const long long tiles_m = ceil_div(static_cast<long long>(prob->N) * P * Q, kBlockM);
  return round256(static_cast<size_t>(ip.splits) * tiles_m * kBlockM *
                  ceil_div(prob->K, ip.bn) * ip.bn * sizeof(int32_t));
}

size_t conv2d_fprop_int8_workspace_size(const igconv_problem_t* prob) {
  int P = 0, Q = 0;
  if (check_shape(prob, &P, &Q) != IGCONV_OK) return 0;
  const size_t xb = static_cast<size_t>(prob->N) * prob->H * prob->W * prob->C * 2;
  const size_t wb = static_cast<size_t>(prob->K) * prob->R * prob->S * prob->C * 2;
  const Int8FpropPlan ip = plan_int8_fprop(prob, P, Q, current_sm_count());
  return round256(xb) + round256(wb) + int8_fprop_split_bytes(prob, P, Q, ip);
}

igconv_status_t conv2d_fprop_int8(const igconv_problem_t* prob, const int8_t* X, const int8_t* Wt,
                                  const int32_t* bias, int8_t* Y, double act_scale,
                                  double w_scale, double out_scale, int relu, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  int P = 0, Q = 0;
  igconv_status_t st = check_shape(prob, &P, &Q);
  if (st != IGCONV_OK) return st;
  if (!X || !Wt || !Y) return IGCONV_ERR_INVALID_ARG;
  if (!(std::isfinite(act_scale) && act_scale > 0) || !(std::isfinite(w_scale) && w_scale > 0) ||
      !(std::isfinite(out_scale) && out_scale > 0))
    return IGCONV_ERR_INVALID_ARG;
  if ((st = check_limits(prob, P, Q, 16)) != IGCONV_OK) return st;
  const long long kg = static_cast<long long>(prob->R) * prob->S * prob->C;
  if (!aligned16(X) || !aligned16(Wt) || !aligned16(Y) || (bias && !aligned16(bias)) ||
      (workspace && !aligned16(workspace)))
    return IGCONV_ERR_MISALIGNED;
  const size_t need = conv2d_fprop_int8_workspace_size(prob);
  if (!workspace || workspace_bytes < need) return IGCONV_ERR_WORKSPACE;
  const double mq = act_scale * w_scale / out_scale;
  const float M = static_cast<float>(mq);
  if (!(std::isfinite(M) && M > 0.0f)) return IGCONV_ERR_UNSUPPORTED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long xcount = static_cast<long long>(prob->N) * prob->H * prob->W * prob->C;
  const long long wcount = static_cast<long long>(prob->K) * kg;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* Xh = ws;
  void* Wh = ws + ((static_cast<size_t>(xcount) * 2 + 255) / 256) * 256;

  ConvGemmParams p;
  init_common(p, dev);
  // Exactness: each TMEM accumulator sums at most 16 reduction blocks, so
  // every partial sum is an integer of magnitude <= 2^24, exact in fp32
  // (plan_int8_fprop); the accumulators are added as int32.
  const Int8FpropPlan ip = plan_int8_fprop(prob, P, Q, dev->sm_count);
  const int bn = ip.bn;
  if ((st = plan_fprop(p, bn, prob, P, Q, 0, Xh, Wh)) != IGCONV_OK) return st;
  const int ni = issuers_for(bn);
  p.num_acc = ni * ip.groups;
  p.kb_per_acc = ceil_div(ceil_div(ip.kb_unit, ni), ip.groups);
  p.relu = relu ? 1 : 0;
  int ex = 0;
  const float fr = std::frexp(M, &ex);  // M = fr * 2^ex, fr in [0.5, 1)
  p.rq_mant = static_cast<uint32_t>(std::ldexp(fr, 24));
  p.rq_exp = ex - 24;
  int* part = nullptr;
  if (ip.splits > 1) {
    // split reduction: exact int32 partial tiles, then bias, ReLU and the
    // requantisation in the ordered split reduction
    part = reinterpret_cast<int*>(static_cast<uint8_t*>(Wh) +
                                  ((static_cast<size_t>(wcount) * 2 + 255) / 256) * 256);
    set_conv_split(p, bn, ip.splits, part);
    p.int_acc = 1;
  } else {
    p.epi = EPI_INT8;
    p.out = Y;
    p.use_tma_store = encode_out_2d(&p.mapY, Y, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                                    static_cast<long long>(prob->N) * P * Q, prob->K, 32,
                                    CU_TENSOR_MAP_SWIZZLE_32B) ? 1 : 0;
    p.bias = bias;
    p.bias_cached = bias != nullptr && prob->K * 4 <= kBiasCacheBytes ? 1 : 0;
  }

  cudaError_t e = launch_i8_to_f16(X, Xh, xcount, s);
  if (e != cudaSuccess) return cuda_error();
  e = launch_i8_to_f16(Wt, Wh, wcount, s);
  if (e != cudaSuccess) return cuda_error();
  e = launch_conv_gemm(p, bn, grid_for(p.units, dev), s);
  if (e != cudaSuccess || part == nullptr) return from_cuda(e);
  return from_cuda(launch_conv_splitk_reduce_i8(part, ip.splits, p.ws_split_stride, p.ws_ld,
                                                static_cast<long long>(prob->N) * P * Q, prob->K,
                                                Y, bias, p.rq_mant, p.rq_exp, p.relu, s));
}

// ---------------------------------------------------------------------------
// int8 dgrad / wgrad: int8 operands widened to fp16 copies in the workspace
// (exact), the dgrad / wgrad implicit GEMM on the fp16 tensor core with each
// TMEM accumulator summing at most 16 reduction blocks (1024 products of
// magnitude <= 2^14, so every partial sum is an integer below 2^24, exact in
// fp32), and the accumulators added as int32 (modulo 2^32) by the epilogue.
// ---------------------------------------------------------------------------
size_t conv2d_dgrad_int8_workspace_size(const igconv_problem_t* prob) {
  int P = 0, Q = 0;
  if (check_shape(prob, &P, &Q) != IGCONV_OK) return 0;
  return round256(static_cast<size_t>(prob->N) * P * Q * prob->K * 2) +
         round256(static_cast<size_t>(prob->K) * prob->R * prob->S * prob->C * 2);
}

igconv_status_t conv2d_dgrad_int8(const igconv_problem_t* prob, const int8_t* dY,
                                  const int8_t* Wt, int32_t* dX, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  int P = 0, Q = 0;
  igconv_status_t st = check_shape(prob, &P, &Q);
  if (st != IGCONV_OK) return st;
  if (!dY || !Wt || !dX) return IGCONV_ERR_INVALID_ARG;
  if ((st = check_limits(prob, P, Q, 16)) != IGCONV_OK) return st;
  if (prob->stride_h * prob->stride_w > kMaxSub) return IGCONV_ERR_UNSUPPORTED;
  if (!aligned16(dY) || !aligned16(Wt) || !aligned16(dX) || (workspace && !aligned16(workspace)))
    return IGCONV_ERR_MISALIGNED;
  const size_t need = conv2d_dgrad_int8_workspace_size(prob);
  if (!workspace || workspace_bytes < need) return IGCONV_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  const long long ycount = static_cast<long long>(prob->N) * P * Q * prob->K;
  const long long wcount = static_cast<long long>(prob->K) * prob->R * prob->S * prob->C;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* dYh = ws;
  void* Wh = ws + round256(static_cast<size_t>(ycount) * 2);
  ConvGemmParams p;
  int bn = 0, forced = g_tune_bn.load();
  for (;;) {
    init_common(p, dev);
    if ((st = plan_dgrad(p, &bn, prob, P, Q, 0, dYh, Wh, dev->sm_count, forced)) != IGCONV_OK)
      return st;
    int max_kb = 0;
    for (int i = 0; i < p.nsub; ++i) {
      const int kb = p.sub[i].rcount * p.sub[i].scount * p.cblocks;
      if (kb > max_kb) max_kb = kb;
    }
    if (int_accumulators(bn, max_kb, &p.num_acc, &p.kb_per_acc)) break;
    if (bn == 64 || forced) return IGCONV_ERR_UNSUPPORTED;
    forced = bn >> 1;
  }
  p.epi = EPI_STORE;
  p.int_acc = 1;
  p.out = dX;
  p.use_tma_store = 0;
  p.alpha = 1.0f;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_i8_to_f16(dY, dYh, ycount, s);
  if (e != cudaSuccess) return cuda_error();
  e = launch_i8_to_f16(Wt, Wh, wcount, s);
  if (e != cudaSuccess) return cuda_error();
  if (p.units == 0) return IGCONV_OK;
  return from_cuda(launch_conv_gemm(p, bn, grid_for(p.units, dev), s));
}

size_t conv2d_wgrad_int8_workspace_size(const igconv_problem_t* prob) {
  int P = 0, Q = 0;
  if (check_shape(prob, &P, &Q) != IGCONV_OK) return 0;
  WgradPlan w;
  plan_wgrad_int8(prob, P, Q, current_sm_count(), &w);
  return round256(static_cast<size_t>(prob->N) * prob->H * prob->W * prob->C * 2) +
         round256(static_cast<size_t>(prob->N) * P * Q * prob->K * 2) + round256(w.ws_bytes);
}

igconv_status_t conv2d_wgrad_int8(const igconv_problem_t* prob, const int8_t* X, const int8_t* dY,
                                  int32_t* dW, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  int P = 0, Q = 0;
  igconv_status_t st = check_shape(prob, &P, &Q);
  if (st != IGCONV_OK) return st;
  if (!X || !dY || !dW) return IGCONV_ERR_INVALID_ARG;
  if ((st = check_limits(prob, P, Q, 16)) != IGCONV_OK) return st;
  if (!aligned16(X) || !aligned16(dY) || !aligned16(dW) || (workspace && !aligned16(workspace)))
    return IGCONV_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  WgradPlan w;
  plan_wgrad_int8(prob, P, Q, dev->sm_count, &w);
  const long long xcount = static_cast<long long>(prob->N) * prob->H * prob->W * prob->C;
  const long long npq = static_cast<long long>(prob->N) * P * Q;
  const long long ycount = npq * prob->K;
  const size_t xb = round256(static_cast<size_t>(xcount) * 2);
  const size_t yb = round256(static_cast<size_t>(ycount) * 2);
  if (!workspace || workspace_bytes < xb + yb + round256(w.ws_bytes)) return IGCONV_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* Xh = ws;
  void* dYh = ws + xb;
  void* part = ws + xb + yb;
  ConvGemmParams p;
  init_common(p, dev);
  p.nsub = 1;
  p.a_src = w.swapped ? SRC_2D_MN : SRC_IM2COL_MN;
  p.b_src = w.swapped ? SRC_IM2COL_MN : SRC_2D_MN;
  p.epi = EPI_PARTIAL;
  p.int_acc = 1;
  p.tiles_m_total = w.tiles_m;
  p.tiles_n = w.tiles_n;
  p.splits = w.splits;
  p.kblocks_total = w.kblocks;
  p.units = w.tiles_m * w.tiles_n * w.splits;
  p.cblocks = w.cblocks;
  p.N_gemm = w.N_pad;
  p.idesc = make_idesc(kBlockM, w.bn, 0, 1, 1);
  if (!int_accumulators(w.bn, ceil_div(w.kblocks, w.splits), &p.num_acc, &p.kb_per_acc))
    return IGCONV_ERR_UNSUPPORTED;  // not reached: the plan sized the splits for this
  p.wg_PQ = P * Q;
  p.wg_Q = Q;
  p.wg_lower_h = -prob->pad_h;
  p.wg_lower_w = -prob->pad_w;
  p.wg_sh = prob->stride_h;
  p.wg_sw = prob->stride_w;
  p.wg_S = prob->S;
  p.wg_RS = w.rs;
  p.wg_dh = prob->dil_h;
  p.wg_dw = prob->dil_w;
  p.wg_K = prob->K;
  p.out = part;
  p.ws_split_stride = static_cast<long long>(w.M_pad) * w.N_pad;
  p.ws_ld = w.N_pad;
  p.use_tma_store = encode_out_2d(&p.mapY, part, CU_TENSOR_MAP_DATA_TYPE_INT32, 4,
                                  static_cast<long long>(w.splits) * w.M_pad, w.N_pad, 16,
                                  CU_TENSOR_MAP_SWIZZLE_64B) ? 1 : 0;
  if (!encode_im2col(&p.mapA[0], Xh, 0, prob->N, prob->H, prob->W, prob->C, -prob->pad_h,
                     -prob->pad_w, prob->pad_h - (prob->R - 1) * prob->dil_h,
                     prob->pad_w - (prob->S - 1) * prob->dil_w, prob->stride_h, prob->stride_w,
                     kBlockK))
    return IGCONV_ERR_UNSUPPORTED;
  p.mapA_valid = 1u;
  if (!encode_2d(&p.mapB, dYh, 0, npq, prob->K)) return IGCONV_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_i8_to_f16(X, Xh, xcount, s);
  if (e != cudaSuccess) return cuda_error();
  e = launch_i8_to_f16(dY, dYh, ycount, s);
  if (e != cudaSuccess) return cuda_error();
  e = launch_conv_gemm(p, w.bn, grid_for(p.units, dev), s);
  if (e != cudaSuccess) return cuda_error();
  const int xext = w.rs * w.cpad;
  return from_cuda(launch_wgrad_reduce_i32(static_cast<const int*>(part), w.splits,
                                           p.ws_split_stride, w.N_pad,
                                           w.swapped ? prob->K : xext, w.swapped ? xext : prob->K,
                                           w.swapped, prob->K, w.rs, prob->C, w.cpad, dW, s));
}

// ---------------------------------------------------------------------------
// Winograd F(2x2, 3x3) forward pass: input and filter transforms on the CUDA
// cores, the 16 transform-domain GEMMs as one implicit-GEMM launch with one
// sub-problem per transform point xi (a 1x1 GEMM over V[xi] and filter tap xi
// of U viewed as [K][16][1][C], written to rows xi of M viewed as a
// [16][T][K] image), then the output transform with fprop's epilogue.
// ---------------------------------------------------------------------------
size_t conv2d_fprop_winograd_workspace_size(const igconv_problem_t* prob, igconv_dtype_t dtype) {
  int P = 0, Q = 0;
  if (check_shape(prob, &P, &Q) != IGCONV_OK) return 0;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return 0;
  if (!wino_shape(prob)) return 0;
  WinoWs w;
  if (!wino_ws(prob, P, Q, &w)) return 0;
  return w.total;
}

igconv_status_t conv2d_fprop_winograd(const igconv_problem_t* prob, igconv_dtype_t dtype,
                                      const void* X, const void* Wt, const void* bias,
                                      const void* Cin, void* Y, float alpha, float beta, int relu,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  int P = 0, Q = 0;
  igconv_status_t st = check_shape(prob, &P, &Q);
  if (st != IGCONV_OK) return st;
  if (!X || !Wt || !Y || (beta != 0.0f && !Cin)) return IGCONV_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return IGCONV_ERR_INVALID_ARG;
  if (dtype != IGCONV_F16 && dtype != IGCONV_BF16) return IGCONV_ERR_UNSUPPORTED;
  if (!wino_shape(prob)) return IGCONV_ERR_UNSUPPORTED;
  if ((st = check_limits(prob, P, Q, 8)) != IGCONV_OK) return st;
  WinoWs w;
  if (!wino_ws(prob, P, Q, &w)) return IGCONV_ERR_UNSUPPORTED;
  if (!aligned16(X) || !aligned16(Wt) || !aligned16(Y) || (bias && !aligned16(bias)) ||
      (beta != 0.0f && !aligned16(Cin)) || (workspace && !aligned16(workspace)))
    return IGCONV_ERR_MISALIGNED;
  if (!workspace || workspace_bytes < w.total) return IGCONV_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != IGCONV_OK) return st;
  const int bf16 = dtype == IGCONV_BF16 ? 1 : 0;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* V = ws;
  uint8_t* U = ws + w.v_bytes;
  uint8_t* Mx = U + w.u_bytes;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  ConvGemmParams p;
  init_common(p, dev);
  const int tiles_m = ceil_div(w.T, kBlockM);
  const int bn = choose_block_n(prob->K, 16LL * tiles_m, dev->sm_count);
  p.tiles_n = ceil_div(prob->K, bn);
  int tile_begin = 0;
  for (int xi = 0; xi < 16; ++xi) {
    SubProblem& sp = p.sub[xi];
    sp.M = static_cast<int>(w.T);
    sp.tile_begin = tile_begin;
    sp.tiles_m = tiles_m;
    sp.Hs = 1;
    sp.Ws = static_cast<int>(w.T);
    sp.lower_h = 0; sp.lower_w = 0; sp.trav_h = 1; sp.trav_w = 1;
    sp.r0 = xi; sp.rstep = 1; sp.rcount = 1; sp.offh0 = 0; sp.doffh = 0;
    sp.s0 = 0; sp.sstep = 1; sp.scount = 1; sp.offw0 = 0; sp.doffw = 0;
    sp.out_h0 = xi; sp.out_w0 = 0; sp.out_sh = 1; sp.out_sw = 1;
    if (!encode_im2col(&p.mapA[xi], V + static_cast<size_t>(xi) * w.T * prob->C * 2, bf16, 1, 1,
                       static_cast<int>(w.T), prob->C, 0, 0, 0, 0, 1, 1, kBlockM))
      return IGCONV_ERR_UNSUPPORTED;
    p.mapA_valid |= 1u << xi;
    tile_begin += tiles_m * p.tiles_n;
  }
  p.nsub = 16;
  p.units = tile_begin;
  p.a_src = SRC_IM2COL_K;
  p.b_src = SRC_W_K;
  p.cblocks = ceil_div(prob->C, kBlockK);
  p.N_gemm = prob->K;
  p.out_C = prob->K;
  p.out_H = 16;
  p.out_W = static_cast<int>(w.T);
  p.idesc = make_idesc(kBlockM, bn, bf16, 0, 0);
  set_fp_accumulators(p, bn);
  if (!encode_filter(&p.mapB, U, bf16, prob->K, 16, 1, prob->C, bn)) return IGCONV_ERR_UNSUPPORTED;
  p.epi = EPI_STORE;
  p.out = Mx;
  p.use_tma_store = 0;
  p.alpha = 1.0f;
  p.out_bf16 = bf16;
  p.pf_base = U;
  p.pf_bytes = static_cast<long long>(prob->K) * 16 * prob->C * 2;

  cudaError_t e = launch_wino_input(X, V, prob->N, prob->H, prob->W, prob->C, w.TH, w.TW,
                                    prob->pad_h, prob->pad_w, bf16, s);
  if (e != cudaSuccess) return cuda_error();
  e = launch_wino_filter(Wt, U, prob->K, prob->C, bf16, s);
  if (e != cudaSuccess) return cuda_error();
  e = launch_conv_gemm(p, bn, grid_for(p.units, dev), s);
  if (e != cudaSuccess) return cuda_error();
  return from_cuda(launch_wino_output(Mx, Y, beta != 0.0f ? Cin : nullptr, bias, prob->N, P, Q,
                                      prob->K, w.TH, w.TW, alpha, beta, relu ? 1 : 0, bf16, s));
}

igconv_status_t nchw_to_nhwc(const void* src, void* dst, int N, int C, int H, int W,
                             int elem_bytes, void* stream) {
  if (!src || !dst || N < 1 || C < 1 || H < 1 || W < 1) return IGCONV_ERR_INVALID_ARG;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
    return IGCONV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) %
      static_cast<uintptr_t>(elem_bytes))
    return IGCONV_ERR_MISALIGNED;
  if (N > 65535 || (static_cast<long long>(C) + 63) / 64 > 65535) return IGCONV_ERR_UNSUPPORTED;
  DeviceState* dev = nullptr;
  igconv_status_t st = device_state(&dev);
  if (st != IGCONV_OK) return st;
  return from_cuda(launch_batched_transpose(src, dst, N, C, static_cast<long long>(H) * W,
                                            elem_bytes, static_cast<cudaStream_t>(stream)));
}

igconv_status_t nhwc_to_nchw(const void* src, void* dst, int N, int C, int H, int W,
                             int elem_bytes, void* stream) {
  if (!src || !dst || N < 1 || C < 1 || H < 1 || W < 1) return IGCONV_ERR_INVALID_ARG;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
    return IGCONV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) %
      static_cast<uintptr_t>(elem_bytes))
    return IGCONV_ERR_MISALIGNED;
  if (N > 65535 || (static_cast<long long>(H) * W + 63) / 64 > 65535)
    return IGCONV_ERR_UNSUPPORTED;
  DeviceState* dev = nullptr;
  igconv_status_t st = device_state(&dev);
  if (st != IGCONV_OK) return st;
  return from_cuda(launch_batched_transpose(src, dst, N, static_cast<long long>(H) * W, C,
                                            elem_bytes, static_cast<cudaStream_t>(stream)));
}

igconv_status_t igconv_get_device_status(void* stream) {
  DeviceState* dev = nullptr;
  igconv_status_t st = device_state(&dev);
  if (st != IGCONV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int word = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return cuda_error();
  if (cudaMemcpy(&word, dev->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return cuda_error();
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return cuda_error();
    return IGCONV_ERR_DEVICE_TIMEOUT;
  }
  return IGCONV_OK;
}

igconv_status_t igconv_selftest_wait_timeout(int timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 2000000) return IGCONV_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  igconv_status_t st = device_state(&dev);
  if (st != IGCONV_OK) return st;
  return from_cuda(launch_selftest_wait(dev->status,
                                        static_cast<unsigned long long>(timeout_us) * 1000ull,
                                        static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
