// conv_wgrad_halo.cu -- the weight gradient of a stride-1 convolution with
// at most 64 input and 64 output channels and 2..9 filter taps, on input
// halos.
//
// dW[k][tap][c] = sum over output positions (n, p, q) of
//   dY[n][p][q][k] * X[n][p + off_h(tap)][q + off_w(tap)][c]
// (input coordinates relative to the padded origin).  Output positions run
// on a grid Wt columns wide (32, 64 or 128, at least the padded input row),
// in blocks of 128 positions = 128 / Wt whole output rows of one image.  For
// one block every tap's X operand is the same input rows shifted by
// off_h * Wt + off_w grid positions, so one TMA copy of the block's input
// rows (the halo, zero outside the image) and one copy of its dY rows (zero
// past the output width, so grid padding adds nothing) serve all taps.
//
// The GEMM: rows (tap, c), columns k, reduction over the positions.  A 128-
// row tile holds two taps (tap pair m: taps 2m and 2m + 1, 64 channels
// each); its A operand is MN-major (channels contiguous in each 128-byte
// pixel row, positions along K) and the two 64-channel halves point at their
// taps' rows through the descriptor's leading-byte offset (the distance
// between the two taps' first rows).  The 128-byte swizzle follows absolute
// shared-memory addresses, so halves and K steps may start on any pixel row.
// B is the dY block, MN-major (64 channels per position row).
//
// Each CTA takes one unit: a contiguous range of blocks (the split), all
// tap pairs of it in TMEM (up to five 64-column accumulators), and writes
// them as fp32 partial tiles [split][pair * 128 + half * 64 + c][k] -- i.e.
// row tap * 64 + c -- which the ordered split reduction adds, scales, casts
// and scatters to KRSC (launch_wgrad_reduce).
#include "conv_gemm_kernel.cuh"

namespace igc {

namespace {

constexpr int kIssuers = 4;

struct WHaloCfg {
  static constexpr int X_BYTES = kHaloRows * 128;        // the input halo
  static constexpr int Y_BYTES = kBlockM * 128;          // 128 positions x 64 dY channels
  static constexpr int STAGE = X_BYTES + Y_BYTES;
  static constexpr int STAGES = 3;
  static constexpr int PIPE = STAGE * STAGES;
  static constexpr int EPI_STAGE = kEpiWarps * kStageWarpBytes;
  static constexpr int BAR_BYTES = 256;
  static constexpr int USED = PIPE + EPI_STAGE + BAR_BYTES;
  static constexpr int SMEM = kSmemLimit;
  static constexpr int NP = STAGES;  // producer warp i owns stage i
  static constexpr int MAX_PAIRS = (kHaloTaps + 1) / 2;
  static_assert(USED <= kSmemLimit, "exceeds the 227 KB of shared memory a CTA may use");
  static_assert(X_BYTES % 1024 == 0 && STAGE % 1024 == 0, "swizzle atoms need 1024-byte alignment");
};

// Row offset (grid positions) of tap t in the halo.
__device__ __forceinline__ int tap_row(const SubProblem& sp, int t) {
  const int jr = t / sp.scount;
  const int js = t - jr * sp.scount;
  return (sp.offh0 + jr * sp.doffh) * sp.Ws + sp.offw0 + js * sp.doffw;
}

__device__ __forceinline__ void unit_blocks(const ConvGemmParams& p, int* b0, int* b1) {
  const long long nb = p.kblocks_total;
  *b0 = static_cast<int>(nb * blockIdx.x / p.splits);
  *b1 = static_cast<int>(nb * (blockIdx.x + 1) / p.splits);
}

__device__ void whalo_producer(const ConvGemmParams& p, uint8_t* pipe, uint64_t* full,
                               uint64_t* empty, volatile int* abort_flag, int pid, int lane) {
  using C = WHaloCfg;
  const SubProblem& sp = p.sub[0];
  const int Wt = sp.Ws;
  const int rows = kBlockM / Wt;
  const int per_img = sp.Hs / rows;  // blocks per image
  const int lower_h = sp.lower_h, lower_w = sp.lower_w;
  const uint32_t bytes = static_cast<uint32_t>(p.halo_bytes + C::Y_BYTES);
  const unsigned long long timeout = p.timeout_ns;
  int b0, b1;
  unit_blocks(p, &b0, &b1);
  uint8_t* stage = pipe + pid * C::STAGE;
  uint32_t phase = 0;
  bool issued = false;
  for (int b = b0 + pid; b < b1; b += C::NP) {
    if (!__all_sync(0xffffffffu, mbar_wait(&empty[pid], phase ^ 1u, abort_flag, timeout))) {
      if (lane == 0) report_failure(p, abort_flag, DEVERR_PRODUCER_WAIT);
      break;
    }
    if (elect_one_sync()) {
      const int n = b / per_img;
      const int row0 = (b - n * per_img) * rows;
      mbar_arrive_expect_tx(&full[pid], bytes);
      tma_load_4d(stage, &p.mapA[0], &full[pid], 0, lower_w, lower_h + row0, n);
      tma_load_4d(stage + C::X_BYTES, &p.mapB, &full[pid], 0, 0, row0, n);
    }
    __syncwarp();
    issued = true;
    phase ^= 1u;
  }
  if (issued && !mbar_wait(&full[pid], phase ^ 1u, nullptr, timeout) && lane == 0)
    report_failure(p, abort_flag, DEVERR_TEARDOWN_WAIT);
}

// Issuer i (of kIssuers, warps 12..15) takes tap pairs i, i + 4, ...: per
// block, eight K steps of 16 positions for each of its pairs, issued back to
// back by one lane (nine taps: pairs of 2, 1, 1, 1 per issuer, so no issuer
// issues more than 16 MMAs a block).
__device__ void whalo_mma(const ConvGemmParams& p, uint8_t* pipe, uint64_t* full, uint64_t* empty,
                          uint64_t* tfull, uint64_t* done_bar, uint32_t tmem_base,
                          volatile int* abort_flag, int issuer, int lane) {
  using C = WHaloCfg;
  const SubProblem& sp = p.sub[0];
  const int taps = sp.rcount * sp.scount;
  const int pairs = (taps + 1) / 2;
  const uint32_t idesc = p.idesc;
  const unsigned long long timeout = p.timeout_ns;
  const uint32_t pipe_addr = smem_u32(pipe);
  // per pair of this issuer: first row of tap 2m and the distance to tap 2m + 1
  // (a lone last tap reads the row after it as its second half: junk rows)
  int row1[C::MAX_PAIRS], dist[C::MAX_PAIRS];
#pragma unroll
  for (int m = 0; m < C::MAX_PAIRS; ++m) {
    row1[m] = 0;
    dist[m] = 1;
    if (m < pairs) {
      row1[m] = tap_row(sp, 2 * m);
      dist[m] = 2 * m + 1 < taps ? tap_row(sp, 2 * m + 1) - row1[m] : 1;
    }
  }
  int b0, b1;
  unit_blocks(p, &b0, &b1);
  int st = 0;
  uint32_t ph = 0;
  bool ok = true;
  for (int b = b0; b < b1; ++b) {
    if (!__all_sync(0xffffffffu, mbar_wait(&full[st], ph, abort_flag, timeout))) {
      if (lane == 0) report_failure(p, abort_flag, DEVERR_MMA_FULL_WAIT);
      ok = false;
      break;
    }
    tc_fence_after_sync();
    if (elect_one_sync()) {
      const uint32_t sbase = pipe_addr + static_cast<uint32_t>(st * C::STAGE);
      const uint64_t bd0 = make_smem_desc(sbase + C::X_BYTES, 8192, 1024);
      const uint32_t first = b == b0 ? 0u : 1u;
#pragma unroll
      for (int m = 0; m < C::MAX_PAIRS; ++m) {
        if (m >= pairs || (m % kIssuers) != issuer) continue;
        const uint64_t ad0 = make_smem_desc(sbase + static_cast<uint32_t>(row1[m]) * 128u,
                                            static_cast<uint32_t>(dist[m]) * 128u, 1024);
        const uint32_t d = tmem_base + static_cast<uint32_t>(m * 64);
#pragma unroll
        for (int k = 0; k < 8; ++k)  // K step: 16 positions = 2048 bytes of both operands
          umma_f16(d, ad0 + static_cast<uint64_t>(k) * (2048 / 16),
                   bd0 + static_cast<uint64_t>(k) * (2048 / 16), idesc, (k > 0) ? 1u : first);
      }
      umma_commit(&empty[st]);
    }
    __syncwarp();
    if (++st == C::STAGES) {
      st = 0;
      ph ^= 1u;
    }
  }
  if (ok && elect_one_sync()) umma_commit(tfull);  // this issuer's pairs are complete
  __syncwarp();
  if (elect_one_sync()) umma_commit(done_bar);
  __syncwarp();
  if (!__all_sync(0xffffffffu, mbar_wait(done_bar, 0, nullptr, timeout)) && lane == 0)
    report_failure(p, abort_flag, DEVERR_TEARDOWN_WAIT);
}

// Epilogue warps 4..11: warp w holds TMEM lanes 32 (w % 4).. of every pair
// and columns 32 (w / 4 - 1).. + 31; each row chunk goes out as two 16-column
// fp32 boxes.
__device__ void whalo_epilogue(const ConvGemmParams& p, uint64_t* tfull, uint32_t tmem_base,
                               volatile int* abort_flag, int warp, uint8_t* stage_buf) {
  const SubProblem& sp = p.sub[0];
  const int pairs = (sp.rcount * sp.scount + 1) / 2;
  const int quarter = warp & 3;
  const int half = (warp - kEpiWarp0) >> 2;
  const int lane = threadIdx.x & 31;
  uint8_t* stage = stage_buf + (warp - kEpiWarp0) * kStageWarpBytes;
  int b0, b1;
  unit_blocks(p, &b0, &b1);
  if (b1 > b0) {
    if (!mbar_wait(tfull, 0u, abort_flag, p.timeout_ns)) {
      report_failure(p, abort_flag, DEVERR_EPI_WAIT);
      return;
    }
    tc_fence_after_sync();
  }
  int flip = 0;
  const int y0 = blockIdx.x * p.tiles_m_total * kBlockM + quarter * 32;
  for (int m = 0; m < pairs; ++m) {
    uint32_t v[32];
    if (b1 > b0) {
      tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(m * 64 + half * 32),
                         v);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0u;  // an empty split adds zero
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 o[4] = {make_uint4(v[16 * h], v[16 * h + 1], v[16 * h + 2], v[16 * h + 3]),
                          make_uint4(v[16 * h + 4], v[16 * h + 5], v[16 * h + 6], v[16 * h + 7]),
                          make_uint4(v[16 * h + 8], v[16 * h + 9], v[16 * h + 10], v[16 * h + 11]),
                          make_uint4(v[16 * h + 12], v[16 * h + 13], v[16 * h + 14],
                                     v[16 * h + 15])};
      warp_tma_store_box(stage, flip, o, 4, &p.mapY, half * 32 + h * 16,
                         OutAt{y0 + m * kBlockM, -1, 0, 0, 0}, lane);
    }
  }
  if (lane == 0) bulk_wait_group<0>();
  __syncwarp();
}

__global__ void __launch_bounds__(kThreads, 1)
    conv_wgrad_halo_kernel(const __grid_constant__ ConvGemmParams p) {
  using C = WHaloCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  if (static_cast<int>(smem - smem_raw) + C::USED > C::SMEM) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, static_cast<unsigned int>(DEVERR_SMEM_LAYOUT));
    return;
  }
  uint8_t* pipe = smem;
  uint8_t* stage_buf = smem + C::PIPE;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::PIPE + C::EPI_STAGE);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* done_bar = tfull + 1;  // one per issuer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + kIssuers);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
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

  if (warp < 4) {
    setmaxnreg_dec<kRegsLow>();
    if (warp < C::NP) {
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
  k<<<p.splits, kThreads, WHaloCfg::SMEM, s>>>(p);
  return cudaGetLastError();
}

}  // namespace igc
