// conv_wgrad_halo.cu -- the weight gradient of a stride-1 convolution with
// at most 128 input and 128 output channels and 2..9 filter taps, on input
// halos.
//
// dW[k][tap][c] = sum over output positions (n, p, q) of
//   dY[n][p][q][k] * X[n][p + off_h(tap)][q + off_w(tap)][c]
// (input coordinates relative to the padded origin).  Output positions run
// on a grid Wt columns wide (32, 64 or 128, at least the padded input row),
// in blocks of 128 positions = 128 / Wt whole output rows of one image.  For
// one block every tap's X operand is the same input rows shifted by
// off_h * Wt + off_w grid positions, so one TMA copy of the block's input
// rows per 64-channel plane (the halo, zero outside the image) and one copy
// of its dY rows per 64-channel chunk (zero past the output width, so grid
// padding adds nothing) serve all taps.
//
// The GEMM: rows (tap, c), columns k (64 or 128: N), reduction over the
// positions.  The row entries are (tap, plane) pairs in tap-major order, 64
// rows each; a 128-row MMA tile takes two consecutive entries (with one
// plane: two taps; with two: one tap's two planes).  Its A operand is
// MN-major (64 channels contiguous in each 128-byte pixel row, positions
// along K) and its two halves point at their entries' first rows through the
// descriptor's leading-byte offset.  The 128-byte swizzle follows absolute
// shared-memory addresses, so halves and K steps may start on any pixel row.
// B is the dY block, MN-major, its 64-channel chunks 16 KB apart.
//
// Each CTA takes one split of the blocks for one group of M-tiles (all that
// fit TMEM at N columns each), four issuers taking the group's tiles, and
// writes them as fp32 partial tiles [split][tile * 128 + half * 64 + c][k] --
// row (tap * planes + plane) * 64 + c -- which the ordered split reduction
// adds, scales, casts and scatters to KRSC (launch_wgrad_reduce).
#include "conv_gemm_kernel.cuh"

namespace igc {

namespace {

constexpr int kIssuers = 4;

struct WHaloCfg {
  static constexpr int MAX_STAGES = 3;
  static constexpr int EPI_STAGE = kEpiWarps * kStageWarpBytes;
  static constexpr int BAR_BYTES = 256;
  static constexpr int PIPE_MAX = kSmemLimit - EPI_STAGE - BAR_BYTES;  // stages live here
  static constexpr int SMEM = kSmemLimit;
  static constexpr int MAX_TILES = 8;  // M-tiles per CTA (at 64 columns each)
};

// First row (byte offset within the stage) of row entry e = (tap, plane).
__device__ __forceinline__ uint32_t entry_offset(const SubProblem& sp, int planes,
                                                 uint32_t plane_bytes, int e) {
  const int tap = e / planes;
  const int plane = e - tap * planes;
  const int jr = tap / sp.scount;
  const int js = tap - jr * sp.scount;
  const int row = (sp.offh0 + jr * sp.doffh) * sp.Ws + sp.offw0 + js * sp.doffw;
  return static_cast<uint32_t>(plane) * plane_bytes + static_cast<uint32_t>(row) * 128u;
}

// This CTA's split and group of M-tiles.
struct WUnit {
  int b0, b1;      // blocks [b0, b1)
  int split;
  int t0, nt;      // global M-tiles t0 .. t0 + nt - 1
};
__device__ __forceinline__ WUnit wunit(const ConvGemmParams& p) {
  WUnit u;
  const int S = p.splits;
  const int group = blockIdx.x / S;
  u.split = blockIdx.x - group * S;
  const long long nb = p.kblocks_total;
  u.b0 = static_cast<int>(nb * u.split / S);
  u.b1 = static_cast<int>(nb * (u.split + 1) / S);
  u.t0 = group * p.num_acc;
  u.nt = min(p.num_acc, p.tiles_m_total - u.t0);
  return u;
}

__device__ void whalo_producer(const ConvGemmParams& p, uint8_t* pipe, uint64_t* full,
                               uint64_t* empty, volatile int* abort_flag, int pid, int lane) {
  const SubProblem& sp = p.sub[0];
  const int Wt = sp.Ws;
  const int rows = kBlockM / Wt;
  const int per_img = sp.Hs / rows;  // blocks per image
  const int lower_h = sp.lower_h, lower_w = sp.lower_w;
  const int planes = p.cblocks, kchunks = p.tiles_n;
  const int stages = p.wh_stages;
  const int stage_bytes = p.wh_stage_bytes;
  const uint32_t x_bytes = static_cast<uint32_t>(planes * p.halo_bytes);
  const uint32_t bytes = x_bytes + static_cast<uint32_t>(kchunks) * (kBlockM * 128);
  const unsigned long long timeout = p.timeout_ns;
  const WUnit u = wunit(p);
  uint8_t* stage = pipe + pid * stage_bytes;
  uint32_t phase = 0;
  bool issued = false;
  for (int b = u.b0 + pid; b < u.b1; b += stages) {
    if (!__all_sync(0xffffffffu, mbar_wait(&empty[pid], phase ^ 1u, abort_flag, timeout))) {
      if (lane == 0) report_failure(p, abort_flag, DEVERR_PRODUCER_WAIT);
      break;
    }
    if (elect_one_sync()) {
      const int n = b / per_img;
      const int row0 = (b - n * per_img) * rows;
      mbar_arrive_expect_tx(&full[pid], bytes);
      for (int pl = 0; pl < planes; ++pl)
        tma_load_4d(stage + pl * p.halo_bytes, &p.mapA[0], &full[pid], pl * 64, lower_w,
                    lower_h + row0, n);
      for (int kc = 0; kc < kchunks; ++kc)
        tma_load_4d(stage + x_bytes + kc * (kBlockM * 128), &p.mapB, &full[pid], kc * 64, 0,
                    row0, n);
    }
    __syncwarp();
    issued = true;
    phase ^= 1u;
  }
  if (issued && !mbar_wait(&full[pid], phase ^ 1u, nullptr, timeout) && lane == 0)
    report_failure(p, abort_flag, DEVERR_TEARDOWN_WAIT);
}

// Issuer i (of kIssuers, warps 12..15) takes the group's tiles i, i + 4, ...:
// per block, eight K steps of 16 positions for each of them, issued back to
// back by one lane (a 3x3 filter on one plane: tiles of 2, 1, 1, 1 per
// issuer, so no issuer issues more than 16 MMAs a block).
__device__ void whalo_mma(const ConvGemmParams& p, uint8_t* pipe, uint64_t* full, uint64_t* empty,
                          uint64_t* tfull, uint64_t* done_bar, uint32_t tmem_base,
                          volatile int* abort_flag, int issuer, int lane) {
  using C = WHaloCfg;
  const SubProblem& sp = p.sub[0];
  const int planes = p.cblocks;
  const int entries = sp.rcount * sp.scount * planes;
  const int N = 64 * p.tiles_n;
  const uint32_t plane_bytes = static_cast<uint32_t>(p.halo_bytes);
  const uint32_t x_bytes = static_cast<uint32_t>(planes) * plane_bytes;
  const int stages = p.wh_stages;
  const uint32_t idesc = p.idesc;
  const unsigned long long timeout = p.timeout_ns;
  const uint32_t pipe_addr = smem_u32(pipe);
  const WUnit u = wunit(p);
  // per tile of the group: first half's offset and the distance to the second
  // (an odd last entry reads the row after it as its second half: junk rows)
  uint32_t off0[C::MAX_TILES], dist[C::MAX_TILES];
#pragma unroll
  for (int i = 0; i < C::MAX_TILES; ++i) {
    off0[i] = 0;
    dist[i] = 128;
    if (i < u.nt) {
      const int e0 = 2 * (u.t0 + i);
      off0[i] = entry_offset(sp, planes, plane_bytes, e0);
      if (e0 + 1 < entries) dist[i] = entry_offset(sp, planes, plane_bytes, e0 + 1) - off0[i];
    }
  }
  int st = 0;
  uint32_t ph = 0;
  bool ok = true;
  for (int b = u.b0; b < u.b1; ++b) {
    if (!__all_sync(0xffffffffu, mbar_wait(&full[st], ph, abort_flag, timeout))) {
      if (lane == 0) report_failure(p, abort_flag, DEVERR_MMA_FULL_WAIT);
      ok = false;
      break;
    }
    tc_fence_after_sync();
    if (elect_one_sync()) {
      const uint32_t sbase = pipe_addr + static_cast<uint32_t>(st * p.wh_stage_bytes);
      const uint64_t bd0 = make_smem_desc(sbase + x_bytes, kBlockM * 128, 1024);
      const uint32_t first = b == u.b0 ? 0u : 1u;
#pragma unroll
      for (int i = 0; i < C::MAX_TILES; ++i) {
        if (i >= u.nt || (i % kIssuers) != issuer) continue;
        const uint64_t ad0 = make_smem_desc(sbase + off0[i], dist[i], 1024);
        const uint32_t d = tmem_base + static_cast<uint32_t>(i * N);
#pragma unroll
        for (int k = 0; k < 8; ++k)  // K step: 16 positions = 2048 bytes of both operands
          umma_f16(d, ad0 + static_cast<uint64_t>(k) * (2048 / 16),
                   bd0 + static_cast<uint64_t>(k) * (2048 / 16), idesc, (k > 0) ? 1u : first);
      }
      umma_commit(&empty[st]);
    }
    __syncwarp();
    if (++st == stages) {
      st = 0;
      ph ^= 1u;
    }
  }
  if (ok && elect_one_sync()) umma_commit(tfull);  // this issuer's tiles are complete
  __syncwarp();
  if (elect_one_sync()) umma_commit(done_bar);
  __syncwarp();
  if (!__all_sync(0xffffffffu, mbar_wait(done_bar, 0, nullptr, timeout)) && lane == 0)
    report_failure(p, abort_flag, DEVERR_TEARDOWN_WAIT);
}

// Epilogue warps 4..11: warp w holds TMEM lanes 32 (w % 4).. of every tile
// and the tile's columns half * N / 2 .. + N / 2 - 1 (half = w / 4 - 1), in
// 32-column chunks, each row chunk going out as two 16-column fp32 boxes.
__device__ void whalo_epilogue(const ConvGemmParams& p, uint64_t* tfull, uint32_t tmem_base,
                               volatile int* abort_flag, int warp, uint8_t* stage_buf) {
  const int N = 64 * p.tiles_n;
  const int quarter = warp & 3;
  const int half = (warp - kEpiWarp0) >> 2;
  const int lane = threadIdx.x & 31;
  uint8_t* stage = stage_buf + (warp - kEpiWarp0) * kStageWarpBytes;
  const WUnit u = wunit(p);
  if (u.b1 > u.b0) {
    if (!mbar_wait(tfull, 0u, abort_flag, p.timeout_ns)) {
      report_failure(p, abort_flag, DEVERR_EPI_WAIT);
      return;
    }
    tc_fence_after_sync();
  }
  int flip = 0;
  const int y0 = (u.split * p.tiles_m_total + u.t0) * kBlockM + quarter * 32;
  for (int i = 0; i < u.nt; ++i) {
    for (int ch = 0; ch < N / 64; ++ch) {
      const int col = half * (N / 2) + ch * 32;
      uint32_t v[32];
      if (u.b1 > u.b0) {
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(i * N + col),
                           v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;  // an empty split adds zero
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 o[4] = {
            make_uint4(v[16 * h], v[16 * h + 1], v[16 * h + 2], v[16 * h + 3]),
            make_uint4(v[16 * h + 4], v[16 * h + 5], v[16 * h + 6], v[16 * h + 7]),
            make_uint4(v[16 * h + 8], v[16 * h + 9], v[16 * h + 10], v[16 * h + 11]),
            make_uint4(v[16 * h + 12], v[16 * h + 13], v[16 * h + 14], v[16 * h + 15])};
        warp_tma_store_box(stage, flip, o, 4, &p.mapY, col + h * 16,
                           OutAt{y0 + i * kBlockM, -1, 0, 0, 0}, lane);
      }
    }
  }
  if (lane == 0) bulk_wait_group<0>();
  __syncwarp();
}

__global__ void __launch_bounds__(kThreads, 1)
    conv_wgrad_halo_kernel(const __grid_constant__ ConvGemmParams p) {
  using C = WHaloCfg;
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int pipe_bytes = p.wh_stages * p.wh_stage_bytes;
  if (static_cast<int>(smem - smem_raw) + pipe_bytes + C::EPI_STAGE + C::BAR_BYTES > C::SMEM ||
      p.wh_stages > C::MAX_STAGES) {
    pdl_wait();
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, static_cast<unsigned int>(DEVERR_SMEM_LAYOUT));
    return;
  }
  uint8_t* pipe = smem;
  uint8_t* stage_buf = smem + pipe_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pipe_bytes + C::EPI_STAGE);
  uint64_t* empty = full + C::MAX_STAGES;
  uint64_t* tfull = empty + C::MAX_STAGES;
  uint64_t* done_bar = tfull + 1;  // one per issuer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + kIssuers);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.wh_stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kIssuers);  // every issuer reads every block
    }
    mbar_init(tfull, kIssuers);
    for (int i = 0; i < kIssuers; ++i) mbar_init(&done_bar[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp0) tmem_alloc(tmem_slot, 512);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // nothing above touches global memory: the stream's earlier kernel may
  // still run until here
  pdl_wait();

  if (warp < 4) {
    setmaxnreg_dec<kRegsLow>();
    if (warp < p.wh_stages) {  // producer warp i owns stage i
      if (warp == 0 && lane == 0) {
        tma_prefetch_map(&p.mapA[0]);
        tma_prefetch_map(&p.mapB);
        tma_prefetch_map(&p.mapY);
      }
      __syncwarp();
      whalo_producer(p, pipe, full, empty, abort_flag, warp, lane);
    }
  } else if (warp >= kMmaWarp0) {
    setmaxnreg_dec<kRegsLow>();
    if (warp < kMmaWarp0 + kIssuers)
      whalo_mma(p, pipe, full, empty, tfull, &done_bar[warp - kMmaWarp0], tmem_base, abort_flag,
                warp - kMmaWarp0, lane);
  } else {
    setmaxnreg_inc<kRegsEpi>();
    whalo_epilogue(p, tfull, tmem_base, abort_flag, warp, stage_buf);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace

cudaError_t launch_wgrad_halo(const ConvGemmParams& p, cudaStream_t s) {
  auto* k = conv_wgrad_halo_kernel;
  cudaError_t e = check_launch_regs(reinterpret_cast<const void*>(k));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, WHaloCfg::SMEM);
  if (e != cudaSuccess) return e;
  const int groups = (p.tiles_m_total + p.num_acc - 1) / p.num_acc;
  return launch_hot(k, static_cast<unsigned>(p.splits * groups), kThreads,
                    static_cast<size_t>(WHaloCfg::SMEM), s, 1, p);
}

}  // namespace igc
