// conv_gemm_kernel.cuh -- the implicit-GEMM convolution kernel for sm_103a.
//
// One persistent kernel serves every pass; the host planner (api.cpp) fills
// ConvGemmParams to select the operand sources and the epilogue:
//
//   fprop  A = im2col(X)  [pixels x (r,s,c)]   K-major, TMA im2col mode
//          B = W          [k x (r,s,c)]        K-major, TMA tiled
//   dgrad  A = im2col(dY) [pixels x (r,s,k)]   K-major, one sub-problem per
//                                              output residue class
//          B = W          [c x (r,s,k)]        MN-major (c contiguous)
//   wgrad  A/B = im2col(X) [(r,s,c) x npq] and dY^T [k x npq], both MN-major,
//          split-K over npq with fp32 partial tiles in a workspace
//   int8   fprop on fp16 copies of the int8 operands, with the reduction
//          spread over several TMEM accumulators so that every fp32 partial
//          sum stays an exactly representable integer
//
// Roles inside one CTA (512 threads = four warpgroups, one CTA per SM):
//   warps 0-3, lane 0  TMA producers (3 or 4 of them): fill a ring of
//                      shared-memory stages, each issuing every NP-th stage
//   warps 12-13, lane 0 MMA issuers (warp 12 also allocates TMEM; warps 14-15
//                      only take part in the register split).  One
//                      thread can issue a tcgen05.mma only every ~70 cycles,
//                      while an M=128, N=128, K=16 MMA executes in 64, so
//                      tiles narrower than 256 use two issuers that take
//                      alternate reduction blocks into separate accumulators
//                      (summed in a fixed order by the epilogue)
//   warps 4-11         epilogue: warp w reads TMEM lanes 32*(w%4)..+31 for
//                      one half of the tile's columns, applies the fused
//                      math, stages rows in shared memory and writes them
//                      back with coalesced 16-byte stores
// Registers: the CTA launches at 128 per thread (the most 512 threads may
// have), then the producer and MMA warpgroups give back 40 each and the two
// epilogue warpgroups take 168, the count their unrolled TMEM-to-global
// paths need without spilling (at 128, as with 448 threads where some SMSPs
// hold four warps, they spilled ~100 bytes per thread to local memory).
// TMEM holds two accumulator buffers so the epilogue of one tile overlaps
// the main loop of the next.  Every mbarrier wait is bounded; on a timeout
// the CTA records an error code, stops issuing work, waits for its copies
// and MMAs in flight, frees TMEM and exits.
//
// The im2col producer is the hardware form of the explicit im2col gather of
// tensorcore "docs/conv2d.md" ("Strategy": col = im2col(X) then a GEMM) with
// the column buffer removed: rows are loaded straight from NHWC memory, with
// padding supplied as zero fill.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "igconv_internal.h"
#include "ptx.cuh"

namespace igc {

constexpr int kEpiWarps = 8;        // epilogue warps 4..11
constexpr int kEpiWarp0 = 4;
constexpr int kMmaWarp0 = 12;       // MMA issuer warps 12..13 (warp 12 owns TMEM)
constexpr int kLaunchRegs = 65536 / kThreads;  // registers per thread at launch: 128
constexpr int kRegsLow = 88;   // producer and MMA warpgroups after setmaxnreg.dec
constexpr int kRegsEpi = 168;  // each epilogue warpgroup after setmaxnreg.inc
// the four warpgroups' shares must add up to exactly what the CTA launched
// with, or an inc would wait for registers that never come back
static_assert(2 * kRegsLow + 2 * kRegsEpi == 4 * kLaunchRegs, "register split != launch pool");
constexpr int kStagePitch = 80;     // bytes per staged row (coalesced-store path)
constexpr int kStageBufBytes = 2048;               // one 32-row staging buffer (TMA path)
constexpr int kStageWarpBytes = 2 * kStageBufBytes; // double-buffered per epilogue warp
constexpr int kBiasBytes = kBiasCacheBytes;  // bias vector cached in shared memory
constexpr int kSmemLimit = 232448; // 227 KB: the most dynamic shared memory a CTA may use

// RESB: the filter stays resident in shared memory (loaded once per CTA,
// up to kResBlocks reduction blocks of BN x 64), so a stage holds only the
// A tile and the ring keeps all eight stages.  It pays only where the
// per-tile work is short: with room for ten blocks (a 3x3 x 64 filter) the
// ring shrank to six stages and the 64-wide 3x3 layers ran 20 % slower.
constexpr int kResBlocks = 4;

template <int BN, bool PAIR = false, bool RESB = false>
struct Cfg {
  static constexpr int A_BYTES = kBlockM * kBlockK * 2;  // 16 KB
  // a CTA of a pair holds half of the tile's filter rows
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * kBlockK * 2;
  static constexpr int STAGE = A_BYTES + (RESB ? 0 : B_BYTES);
  static constexpr int STAGES =
      RESB ? 8 : (PAIR ? (BN == 256 ? 6 : 8) : (BN == 256 ? 4 : (BN == 128 ? 6 : 8)));
  static constexpr int RES_BYTES = RESB ? kResBlocks * B_BYTES : 0;  // after the stages
  static constexpr int PIPE = STAGE * STAGES + RES_BYTES;
  static constexpr int EPI_STAGE = kEpiWarps * kStageWarpBytes;  // 32 KB
  static constexpr int BAR_BYTES = 256;
  static constexpr int NI = (BN == 256) ? 1 : 2;  // MMA issuer threads
  // Producer warps: one thread needs ~600 cycles per stage (barrier wait,
  // expect-tx and copy issue each take 100-250 cycles), so one lane in each
  // of NP warps issues the copies of every NP-th stage.
  static constexpr int NP = (STAGES % 4 == 0) ? 4 : 3;
  static_assert(STAGES % NP == 0, "producer lanes must tile the stage ring");
  static_assert(NI == 1 || (NI == 2 && STAGES % 2 == 0), "one consumer per stage needs an even ring");
  // Bytes the layout needs past a 1024-byte aligned base; the request is the
  // whole 227 KB, and the kernel checks that the base leaves room for it.
  static constexpr int USED = PIPE + EPI_STAGE + kBiasBytes + BAR_BYTES;
  static constexpr int SMEM = kSmemLimit;
  static_assert(USED <= kSmemLimit, "exceeds the 227 KB of shared memory a CTA may use");
  // full/empty per stage, tfull/tempty per TMEM buffer (up to 4), done per
  // issuer, the resident filter's barrier
  static_assert(2 * STAGES + 11 <= (BAR_BYTES - 8) / 8, "barrier area too small");
};

struct Work {
  int sub, tile_m, tile_n, split, kb0, kb1;
};

// Scalars of the work decomposition, copied once into registers by every
// role (kernel-parameter loads through a reference are slow in hot loops).
struct Sched {
  int epi, units, tiles_m_total, tiles_n, splits, kblocks_total, nsub, cblocks;
  int conv;  // operands are the convolution's (fprop / dgrad), not wgrad's
  int pair;  // CTA pairs: a unit is 256 rows, this CTA takes the half of its rank
  int rank;  // this CTA's rank in its pair (0 without pairs)
  int raster;  // fprop / dgrad tile order (ConvGemmParams::raster)
};

template <bool PAIR>
__device__ __forceinline__ Sched load_sched(const ConvGemmParams& p) {
  Sched s;
  s.epi = p.epi;
  s.conv = p.epi != EPI_PARTIAL || p.conv_split;
  s.units = p.units;
  s.tiles_m_total = p.tiles_m_total;
  s.tiles_n = p.tiles_n;
  s.splits = p.splits;
  s.kblocks_total = p.kblocks_total;
  s.nsub = p.nsub;
  s.cblocks = p.cblocks;
  s.pair = PAIR ? 1 : 0;  // the host sets p.pair for the PAIR kernels only
  s.rank = PAIR ? static_cast<int>(cluster_ctarank() & 1u) : 0;
  s.raster = p.raster;
  return s;
}

// Tile (row um, column tn) of local unit index t in a grid of tm x tn_count
// tiles.  g <= 1: columns fastest (all column tiles of a row tile run at
// about the same time, so its A rows are read from L2 once per wave); g > 1:
// the grid is cut into runs of g row tiles, and within a run the rows are
// walked fastest, column by column, so that a wave of CTAs covers a compact
// block of rows x columns (the swizzled order of CUTLASS's threadblock
// swizzle).
__device__ __forceinline__ void raster_tile(int t, int tm, int tn_count, int g, int* um, int* tn) {
  if (g <= 1) {
    *um = t / tn_count;
    *tn = t - *um * tn_count;
    return;
  }
  const int run = t / (g * tn_count);
  const int r = t - run * g * tn_count;
  const int left = tm - run * g;
  const int rows = left < g ? left : g;
  *tn = r / rows;
  *um = run * g + (r - *tn * rows);
}

// The units of this CTA (pair) are first, first + stride, ...
__device__ __forceinline__ int unit_first(const Sched& sc) {
  return sc.pair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
}
__device__ __forceinline__ int unit_stride(const Sched& sc) {
  return sc.pair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
}

__device__ __forceinline__ Work decode_unit(const ConvGemmParams& p, const Sched& sc, int u) {
  Work w;
  if (sc.epi == EPI_PARTIAL) {
    const int tiles = sc.tiles_m_total * sc.tiles_n;
    w.split = u / tiles;
    const int t = u - w.split * tiles;
    w.tile_m = t / sc.tiles_n;
    w.tile_n = t - w.tile_m * sc.tiles_n;
    w.sub = 0;
    w.kb0 = static_cast<int>(static_cast<long long>(w.split) * sc.kblocks_total / sc.splits);
    w.kb1 = static_cast<int>(static_cast<long long>(w.split + 1) * sc.kblocks_total / sc.splits);
  } else {
    int i = 0;
    while (i + 1 < sc.nsub && u >= p.sub[i + 1].tile_begin) ++i;
    w.sub = i;
    const int local = u - p.sub[i].tile_begin;
    // pairs (one sub-problem only): a unit row is two 128-row tiles
    const int unit_rows = sc.pair ? (p.sub[i].tiles_m + 1) / 2 : p.sub[i].tiles_m;
    raster_tile(local, unit_rows, sc.tiles_n, sc.raster, &w.tile_m, &w.tile_n);
    if (sc.pair) w.tile_m = 2 * w.tile_m + sc.rank;
    w.split = 0;
    w.kb0 = 0;
    w.kb1 = p.sub[i].rcount * p.sub[i].scount * sc.cblocks;
  }
  return w;
}

// Walks this CTA's work units (static stride gridDim.x).  Without a split
// and in the built-in tile order (fprop, dgrad) the walk keeps the unit's
// sub-problem and tile coordinates and advances them by a precomputed
// quotient and remainder, so a step costs no division and no parameter
// loads; only a step into the next sub-problem (the residue classes of a
// strided dgrad) places the walk again from the unit index.
struct UnitWalk {
  int u, stride;
  int tm, tn;    // fast path: tile coordinates of unit u (tm in 128-row tiles)
  int gq, gr;    // stride / tiles_n and stride % tiles_n
  int mstep;     // 128-row tiles per unit row: 2 with pairs
  int nk;        // fast path: reduction blocks per unit of the sub-problem
  int sub;       // fast path: sub-problem of unit u
  int sub_end;   // fast path: first unit past that sub-problem
  bool fast;
};

// Whether walk_begin takes the fast path for these scalars.
__device__ __forceinline__ bool uw_fast_possible(const Sched& sc) {
  return sc.epi != EPI_PARTIAL && sc.raster <= 1;
}

// Places a fast walk at unit it.u (< units).
__device__ __forceinline__ void walk_seek(const ConvGemmParams& p, const Sched& sc,
                                          UnitWalk& it) {
  int i = 0;
  while (i + 1 < sc.nsub && it.u >= p.sub[i + 1].tile_begin) ++i;
  it.sub = i;
  it.sub_end = i + 1 < sc.nsub ? p.sub[i + 1].tile_begin : sc.units;
  const int local = it.u - p.sub[i].tile_begin;
  const int um = local / sc.tiles_n;
  it.tn = local - um * sc.tiles_n;
  it.tm = it.mstep * um + sc.rank;
  it.nk = p.sub[i].rcount * p.sub[i].scount * sc.cblocks;
}

__device__ __forceinline__ void walk_begin(const ConvGemmParams& p, const Sched& sc,
                                           UnitWalk& it) {
  it.u = unit_first(sc);
  it.stride = unit_stride(sc);
  it.fast = uw_fast_possible(sc);
  it.tm = it.tn = it.gq = it.gr = it.nk = it.sub = 0;
  it.sub_end = sc.units;
  it.mstep = sc.pair ? 2 : 1;
  if (it.fast) {
    it.gq = it.stride / sc.tiles_n;
    it.gr = it.stride - it.gq * sc.tiles_n;
    if (it.u < sc.units) walk_seek(p, sc, it);
  }
}

__device__ __forceinline__ Work walk_work(const ConvGemmParams& p, const Sched& sc,
                                          const UnitWalk& it) {
  if (it.fast) {
    Work w;
    w.sub = it.sub;
    w.tile_m = it.tm;
    w.tile_n = it.tn;
    w.split = 0;
    w.kb0 = 0;
    w.kb1 = it.nk;
    return w;
  }
  return decode_unit(p, sc, it.u);
}

__device__ __forceinline__ void walk_next(const ConvGemmParams& p, const Sched& sc,
                                          UnitWalk& it) {
  it.u += it.stride;
  if (it.fast) {
    if (it.u >= it.sub_end) {
      if (it.u < sc.units) walk_seek(p, sc, it);
      return;
    }
    it.tn += it.gr;
    it.tm += it.mstep * it.gq;
    if (it.tn >= sc.tiles_n) {
      it.tn -= sc.tiles_n;
      it.tm += it.mstep;
    }
  }
}

__device__ __forceinline__ void report_failure(const ConvGemmParams& p, volatile int* abort_flag,
                                               unsigned int code) {
  *abort_flag = 1;
  atomicCAS(p.status, 0u, code);
}

// ---------------------------------------------------------------------------
// Producers (lane 0 of warps 0..NP-1).  All reduction blocks of this CTA's
// work units form one sequence; block number q of the sequence uses stage
// q % STAGES.  Producer l handles q = l, l + NP, l + 2*NP, ...
// ---------------------------------------------------------------------------
struct ProdCtx {       // producer scalars, in registers
  Sched sc;
  int a_src, b_src;
  int wg_PQ, wg_Q, wg_lower_h, wg_lower_w, wg_sh, wg_sw, wg_S, wg_RS, wg_dh, wg_dw, wg_K;
  int wg_Do, wg_lower_d, wg_sd, wg_dd, wg_R;
  const CUtensorMap* mapA0;
  const CUtensorMap* mapB;
  const void* taps_filter;
  int grp_mul, grp_div;  // grouped block-diagonal GEMM: channel window of a tile (0: dense)
};

// First channel of the reduction window of 64-wide tile n in a grouped
// block-diagonal GEMM (0 for a dense one).
__device__ __forceinline__ int group_window(const ProdCtx& c, int tile_n) {
  return c.grp_mul ? (tile_n / c.grp_div) * c.grp_mul : 0;
}

struct ProducerPos {
  int u;          // work unit
  int kb;         // reduction block within the unit
  Work w;
  int img, base_h, base_w;  // first pixel of the unit's tile (conv passes)
  int base_d;               // 3D: first depth position
  // tap list of the unit's sub-problem (conv passes)
  int scount, r0, rstep, s0, sstep, offh0, doffh, offw0, doffw;
  int rdiv, doffd;          // 3D: r taps per depth tap, depth offset step
  int tstride, offd0;       // 3D: filter row step per depth tap, first depth offset
  const CUtensorMap* mapA;
  bool active;
};

template <bool VOL>
__device__ __forceinline__ void producer_enter_unit(const ConvGemmParams& p, const ProdCtx& c,
                                                    ProducerPos& s) {
  s.w = decode_unit(p, c.sc, s.u);
  if (c.sc.conv) {
    const SubProblem& sp = p.sub[s.w.sub];
    const int Hs = sp.Hs, Ws = sp.Ws;
    const int m0 = s.w.tile_m * kBlockM;
    const int per_plane = Hs * Ws;
    int rem;
    if (VOL && sp.Ds > 0) {  // 3D: m0 = ((img * Ds + id) * Hs + ih) * Ws + iw
      const int per_img = sp.Ds * per_plane;
      s.img = m0 / per_img;
      const int r3 = m0 - s.img * per_img;
      const int id = r3 / per_plane;
      rem = r3 - id * per_plane;
      s.base_d = sp.lower_d + id * sp.trav_d;
    } else {
      s.img = m0 / per_plane;
      rem = m0 - s.img * per_plane;
      s.base_d = 0;
    }
    const int ih = rem / Ws;
    const int iw = rem - ih * Ws;
    s.base_h = sp.lower_h + ih * sp.trav_h;
    s.base_w = sp.lower_w + iw * sp.trav_w;
    if (VOL) {
      s.rdiv = sp.rdiv;
      s.doffd = sp.doffd;
      s.tstride = sp.tstride;
      s.offd0 = sp.offd0;
    }
    s.scount = sp.scount;
    s.r0 = sp.r0;
    s.rstep = sp.rstep;
    s.s0 = sp.s0;
    s.sstep = sp.sstep;
    s.offh0 = sp.offh0;
    s.doffh = sp.doffh;
    s.offw0 = sp.offw0;
    s.doffw = sp.doffw;
    s.mapA = &p.mapA[s.w.sub];
  }
}

// Moves the position forward by `step` reduction blocks across work units.
template <bool VOL>
__device__ __forceinline__ void producer_advance(const ConvGemmParams& p, const ProdCtx& c,
                                                 ProducerPos& s, int step) {
  s.kb += step;
  while (s.kb >= s.w.kb1) {
    const int over = s.kb - s.w.kb1;
    s.u += unit_stride(c.sc);
    if (s.u >= c.sc.units) {
      s.active = false;
      return;
    }
    producer_enter_unit<VOL>(p, c, s);
    s.kb = s.w.kb0 + over;
  }
}

// VOL: the 3D (volume) paths are compiled in; the 2D kernels carry none of
// their branches.
template <int BN, bool PAIR, bool VOL, bool RESB = false>
__device__ __forceinline__ void issue_stage_loads(const ProdCtx& c, const ProducerPos& s,
                                                  uint8_t* sA, uint8_t* sB, uint64_t* bar) {
  const int kb = s.kb;
  if (c.a_src == SRC_IM2COL_TAPS) {
    // few channels: block kb holds taps 8 kb .. 8 kb + 7 (tap = r * S + s),
    // each 8 channels; taps past R * S only pad the last block, where the
    // filter copy reads as zero (any finite pixels do for A)
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      int t = kb * 8 + i;
      if (t >= c.wg_RS) t = 0;
      const int r = t / c.wg_S;
      const int sc = t - r * c.wg_S;
      tma_load_im2col_4d(sA + i * 2048, s.mapA, bar, 0, s.base_w, s.base_h, s.img,
                         static_cast<uint16_t>(sc * c.wg_dw), static_cast<uint16_t>(r * c.wg_dh));
    }
    bulk_load(sB, static_cast<const uint8_t*>(c.taps_filter) +
                      (static_cast<long long>(kb) * c.sc.tiles_n + s.w.tile_n) * (BN * 128),
              BN * 128, bar);
    return;
  }
  if (VOL && c.a_src == SRC_IM2COL_K3) {
    // 3D fprop: block kb = (merged tap (jt, jr, js), 64-channel block); the
    // filter is [K][T*R][S][C], so its row coordinate is the merged jt*R + jr
    const int tap = kb / c.sc.cblocks;
    const int cb = kb - tap * c.sc.cblocks;
    const int jrt = tap / s.scount;
    const int js = tap - jrt * s.scount;
    const int jt = jrt / s.rdiv;
    const int jr = jrt - jt * s.rdiv;
    tma_load_im2col_5d(sA, s.mapA, bar, cb * kBlockK, s.base_w, s.base_h, s.base_d, s.img,
                       static_cast<uint16_t>(s.offw0 + js * s.doffw),
                       static_cast<uint16_t>(s.offh0 + jr * s.doffh),
                       static_cast<uint16_t>(s.offd0 + jt * s.doffd));
    // filter tap of this block in the [K][T*R][S][C] view (fprop: r0 = 0,
    // tstride = R, steps 1; dgrad: the residue class's taps)
    const int fs = s.s0 + js * s.sstep;
    const int fr = s.r0 + jt * s.tstride + jr * s.rstep;
    if (c.b_src == SRC_W_K) {
      tma_load_4d(sB, c.mapB, bar, cb * kBlockK, fs, fr, s.w.tile_n * BN);
    } else {
#pragma unroll
      for (int i = 0; i < BN / 64; ++i)
        tma_load_4d(sB + i * 8192, c.mapB, bar, s.w.tile_n * BN + 64 * i, fs, fr, cb * kBlockK);
    }
    return;
  }
  if (c.sc.conv) {
    // reduction block kb = (tap, 64-channel block)
    const int tap = kb / c.sc.cblocks;
    const int cb = kb - tap * c.sc.cblocks;
    const int jr = tap / s.scount;
    const int js = tap - jr * s.scount;
    const int r = s.r0 + jr * s.rstep;
    const int sc = s.s0 + js * s.sstep;
    const uint16_t off_h = static_cast<uint16_t>(s.offh0 + jr * s.doffh);
    const uint16_t off_w = static_cast<uint16_t>(s.offw0 + js * s.doffw);
    if (PAIR) {
      // both CTAs' copies count on the even CTA's barrier; this CTA holds
      // filter rows rank * BN/2 .. + BN/2 of the tile
      const uint32_t pbar = mapa_shared(smem_u32(bar), 0);
      const int n0 = s.w.tile_n * BN + c.sc.rank * (BN / 2);
      tma_load_im2col_4d_pair(sA, s.mapA, pbar, cb * kBlockK, s.base_w, s.base_h, s.img, off_w,
                              off_h);
      if (c.b_src == SRC_W_K) {
        tma_load_4d_pair(sB, c.mapB, pbar, cb * kBlockK, sc, r, n0);
      } else {
#pragma unroll
        for (int i = 0; i < BN / 128; ++i)
          tma_load_4d_pair(sB + i * 8192, c.mapB, pbar, n0 + 64 * i, sc, r, cb * kBlockK);
      }
      return;
    }
    // grouped block-diagonal GEMM (BN = 64): tile n reduces over its group
    // window of the im2col operand's channels and the same channels of the
    // dense block-diagonal filter (fprop: filter columns; dgrad: filter rows)
    const int ch = group_window(c, s.w.tile_n) + cb * kBlockK;
    tma_load_im2col_4d(sA, s.mapA, bar, ch, s.base_w, s.base_h, s.img, off_w, off_h);
    if (RESB) {
      // the filter is resident in shared memory
    } else if (c.b_src == SRC_W_K) {
      tma_load_4d(sB, c.mapB, bar, ch, sc, r, s.w.tile_n * BN);
    } else {
#pragma unroll
      for (int i = 0; i < BN / 64; ++i)
        tma_load_4d(sB + i * 8192, c.mapB, bar, s.w.tile_n * BN + 64 * i, sc, r, ch);
    }
  } else {
    // wgrad: reduction block kb = 64 consecutive output positions (n, p, q)
    const int npq0 = kb * kBlockK;
    int n, rem, bd = 0;
    if (VOL && c.wg_Do > 0) {  // 3D: npq0 = ((n * Do + o) * P + p) * Q + q
      const int per = c.wg_Do * c.wg_PQ;
      n = npq0 / per;
      const int r3 = npq0 - n * per;
      const int od = r3 / c.wg_PQ;
      rem = r3 - od * c.wg_PQ;
      bd = c.wg_lower_d + od * c.wg_sd;
    } else {
      n = npq0 / c.wg_PQ;
      rem = npq0 - n * c.wg_PQ;
    }
    const int pp = rem / c.wg_Q;
    const int q = rem - pp * c.wg_Q;
    const int bh = c.wg_lower_h + pp * c.wg_sh;
    const int bw = c.wg_lower_w + q * c.wg_sw;
    const bool x_is_a = (c.a_src == SRC_IM2COL_MN || c.a_src == SRC_IM2COL_TAPS_MN);
    const bool x_taps = (c.a_src == SRC_IM2COL_TAPS_MN || c.b_src == SRC_IM2COL_TAPS_MN);
    uint8_t* x_dst = x_is_a ? sA : sB;
    uint8_t* y_dst = x_is_a ? sB : sA;
    constexpr int XA = 2, XB = BN / 64;  // 64-wide chunks per operand tile
    const int x_chunks = x_is_a ? XA : XB;
    const int y_chunks = x_is_a ? XB : XA;
    const int x_tile = x_is_a ? s.w.tile_m : s.w.tile_n;
    const int y_tile = x_is_a ? s.w.tile_n : s.w.tile_m;
    if (x_taps) {
      // few channels: chunk g holds taps 8g .. 8g + 7 of 8 channels each;
      // taps past R * S only pad the last chunk (their rows are never
      // written back), so any valid tap is loaded there
      for (int i = 0; i < x_chunks; ++i) {
        const int g = x_tile * x_chunks + i;
#pragma unroll 1
        for (int t8 = 0; t8 < 8; ++t8) {
          int tap = g * 8 + t8;
          if (tap >= c.wg_RS) tap = c.wg_RS - 1;
          const int r = tap / c.wg_S;
          const int sc = tap - r * c.wg_S;
          tma_load_im2col_4d(x_dst + i * 8192 + t8 * 1024, c.mapA0, bar, 0, bw, bh, n,
                             static_cast<uint16_t>(sc * c.wg_dw),
                             static_cast<uint16_t>(r * c.wg_dh));
        }
      }
    }
    for (int i = 0; i < (x_taps ? 0 : x_chunks); ++i) {
      const int g = x_tile * x_chunks + i;  // 64-wide chunk of the (tap, c) extent
      int tap = g / c.sc.cblocks;
      const int cb = g - tap * c.sc.cblocks;
      // rows past the last tap only pad the final tile; load any valid
      // tap there, those rows are never written back
      if (tap >= c.wg_RS) tap = c.wg_RS - 1;
      int r = tap / c.wg_S;
      const int sc = tap - r * c.wg_S;
      if (VOL && c.wg_Do > 0) {  // 3D: the merged (t, r) index splits by R
        const int jt = r / c.wg_R;
        r -= jt * c.wg_R;
        tma_load_im2col_5d(x_dst + i * 8192, c.mapA0, bar, cb * kBlockK, bw, bh, bd, n,
                           static_cast<uint16_t>(sc * c.wg_dw), static_cast<uint16_t>(r * c.wg_dh),
                           static_cast<uint16_t>(jt * c.wg_dd));
        continue;
      }
      // grouped block-diagonal wgrad (one 64-wide dY tile): the X channels of
      // output-channel tile n are its group window
      tma_load_im2col_4d(x_dst + i * 8192, c.mapA0, bar, group_window(c, y_tile) + cb * kBlockK, bw,
                         bh, n, static_cast<uint16_t>(sc * c.wg_dw),
                         static_cast<uint16_t>(r * c.wg_dh));
    }
    // dY chunks past the last output channel only pad the tile: load the
    // last valid chunk there instead (those rows/columns are discarded)
    const int last_k0 = ((c.wg_K - 1) / 64) * 64;
    for (int i = 0; i < y_chunks; ++i) {
      int k0 = (y_tile * y_chunks + i) * 64;
      if (k0 > last_k0) k0 = last_k0;
      tma_load_2d(y_dst + i * 8192, c.mapB, bar, k0, npq0);
    }
  }
}

template <int BN, bool PAIR, bool VOL, bool RESB = false>
__device__ __forceinline__ void run_producer(const ConvGemmParams& p, uint8_t* pipe,
                                             uint64_t* full, uint64_t* empty, uint64_t* bfull,
                                             volatile int* abort_flag, int pid, int lane) {
  using C = Cfg<BN, PAIR, RESB>;
  constexpr int NP = C::NP;
  constexpr int OWN = C::STAGES / NP;  // stages this lane owns
  uint32_t last_phase[OWN];
  bool issued[OWN];
#pragma unroll
  for (int s = 0; s < OWN; ++s) {
    issued[s] = false;
    last_phase[s] = 0;
  }
  ProdCtx c;
  c.sc = load_sched<PAIR>(p);
  c.a_src = p.a_src;
  c.b_src = p.b_src;
  c.wg_PQ = p.wg_PQ; c.wg_Q = p.wg_Q; c.wg_lower_h = p.wg_lower_h; c.wg_lower_w = p.wg_lower_w;
  c.wg_sh = p.wg_sh; c.wg_sw = p.wg_sw; c.wg_S = p.wg_S; c.wg_RS = p.wg_RS;
  c.wg_dh = p.wg_dh; c.wg_dw = p.wg_dw; c.wg_K = p.wg_K;
  c.wg_Do = p.wg_Do; c.wg_lower_d = p.wg_lower_d; c.wg_sd = p.wg_sd; c.wg_dd = p.wg_dd;
  c.wg_R = p.wg_R;
  c.mapA0 = &p.mapA[0];
  c.mapB = &p.mapB;
  c.taps_filter = p.taps_filter;
  c.grp_mul = p.grp_mul;
  c.grp_div = p.grp_div > 0 ? p.grp_div : 1;
  const unsigned long long timeout = p.timeout_ns;
  ProducerPos pos;
  pos.u = unit_first(c.sc);
  pos.active = pos.u < c.sc.units;
  if (pos.active) {
    producer_enter_unit<VOL>(p, c, pos);
    pos.kb = pos.w.kb0 - NP;      // so that advancing by NP lands on kb0
    producer_advance<VOL>(p, c, pos, NP + pid);
  }
  // Resident filter: every unit of the launch reduces over the same blocks
  // of the single 64-wide column tile, so producer 0 loads them once, block
  // kb at offset kb * B_BYTES after the stages, on their own barrier.
  bool b_issued = false;
  if (RESB && pid == 0 && pos.active) {
    if (elect_one_sync()) {
      const int nkb = pos.w.kb1 - pos.w.kb0;
      uint8_t* res = pipe + C::STAGE * C::STAGES;
      mbar_arrive_expect_tx(bfull, static_cast<uint32_t>(nkb * C::B_BYTES));
      for (int kb = 0; kb < nkb; ++kb) {
        const int tap = kb / c.sc.cblocks;
        const int cb = kb - tap * c.sc.cblocks;
        const int jr = tap / pos.scount;
        const int js = tap - jr * pos.scount;
        const int r = pos.r0 + jr * pos.rstep;
        const int sc = pos.s0 + js * pos.sstep;
        if (c.b_src == SRC_W_K)
          tma_load_4d(res + kb * C::B_BYTES, c.mapB, bfull, cb * kBlockK, sc, r, 0);
        else
          tma_load_4d(res + kb * C::B_BYTES, c.mapB, bfull, 0, sc, r, cb * kBlockK);
      }
    }
    __syncwarp();
    b_issued = true;
  }
  int stage = pid;                // sequence number q = pid: stage q % STAGES
  uint32_t phase = 0;
  int slot = 0;                   // index of `stage` among this lane's stages
  while (pos.active) {
    if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1u, abort_flag, timeout))) {
      if (lane == 0) report_failure(p, abort_flag, DEVERR_PRODUCER_WAIT);
      break;
    }
    uint8_t* sA = pipe + stage * C::STAGE;
    uint8_t* sB = sA + C::A_BYTES;
    if (elect_one_sync()) {
      // with pairs the even CTA's barrier expects both CTAs' bytes
      if (!PAIR) mbar_arrive_expect_tx(&full[stage], C::STAGE);
      else if (c.sc.rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE);
      issue_stage_loads<BN, PAIR, VOL, RESB>(c, pos, sA, sB, &full[stage]);
    }
    __syncwarp();
    issued[slot] = true;
    last_phase[slot] = phase;
    stage += NP;
    if (++slot == OWN) {
      slot = 0;
      stage -= C::STAGES;
      phase ^= 1u;
    }
    producer_advance<VOL>(p, c, pos, NP);
  }
  // Every copy this producer issued must land before the CTA exits.  With
  // pairs the copies complete on the even CTA's barrier, so each CTA waits
  // instead for its stages to be consumed (which needs them landed).
#pragma unroll
  for (int s = 0; s < OWN; ++s) {
    uint64_t* bar = PAIR ? &empty[pid + s * NP] : &full[pid + s * NP];
    if (issued[s] && !mbar_wait(bar, last_phase[s], nullptr, timeout) && lane == 0)
      report_failure(p, abort_flag, DEVERR_TEARDOWN_WAIT);
  }
  if (b_issued && !mbar_wait(bfull, 0u, nullptr, timeout) && lane == 0)
    report_failure(p, abort_flag, DEVERR_TEARDOWN_WAIT);
}

// Position within its unit of issuer i's first block, the unit's first
// block having CTA-wide sequence number q0 (issuer i takes q = i mod ni).
__device__ __forceinline__ int first_rel(int issuer, int ni, int q0) {
  return ni == 1 ? 0 : (issuer ^ (q0 & 1));
}

// ---------------------------------------------------------------------------
// MMA issuers (one warp each, one elected lane issuing).  All reduction
// blocks of this CTA's units form one sequence (the producers' q); issuer i
// takes the blocks with q % NI == i, and its j-th block of a unit
// accumulates into accumulator i + NI * (j / kb_per_acc).  With an even
// stage count every stage then has a single consumer, which the parity
// waits need: were blocks assigned by their position within the unit, a
// unit with an odd block count would hand each stage to the two issuers in
// turn, and an issuer a full ring ahead of the other could pass its parity
// wait on a fill that is still in flight for the other one.
//
// The issuer is a single thread whose loop is a dependent instruction chain,
// so its per-block cost is what limits the main loop once the copies are in
// flight: everything a block needs is kept incremental (descriptors advance
// by plain adds of the stage offset, the accumulator switch is a countdown),
// leaving a wait, four MMAs and a commit per block.
// ---------------------------------------------------------------------------
template <bool PAIR>
__device__ __forceinline__ void mma_issue(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t acc) {
  if (PAIR)
    umma_f16_pair(d, a, b, idesc, acc);
  else
    umma_f16(d, a, b, idesc, acc);
}
template <bool PAIR>
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  if (PAIR)
    umma_commit_pair(bar);  // the barrier at this offset in both CTAs
  else
    umma_commit(bar);
}

// With pairs only the even CTA runs this; its MMAs (M = 256) read both CTAs'
// stages and write both CTAs' TMEM, and its commits arrive in both CTAs.
template <int BN, bool PAIR, bool RESB = false>
__device__ __forceinline__ void run_mma(const ConvGemmParams& p, uint8_t* pipe, uint64_t* full,
                                        uint64_t* empty, uint64_t* tfull, uint64_t* tempty,
                                        uint64_t* done_bar, uint64_t* bfull, uint32_t tmem_base,
                                        volatile int* abort_flag, int issuer, int lane) {
  using C = Cfg<BN, PAIR, RESB>;
  constexpr int NI = C::NI;
  constexpr int STAGES = C::STAGES;
  const Sched sc = load_sched<PAIR>(p);
  const bool a_mn = (p.a_src == SRC_IM2COL_MN || p.a_src == SRC_2D_MN);
  const bool b_mn = (p.b_src == SRC_W_MN || p.b_src == SRC_IM2COL_MN || p.b_src == SRC_2D_MN);
  // tap-packed few-channel X side of wgrad: no swizzle, MN-major, 8-channel
  // groups (one filter tap each) 1 KB apart along MN, 8-position groups 128 B
  // apart along K; one K = 16 step is 256 bytes.  Without swizzle an MN-major
  // operand takes its MN-direction stride in the stride-byte-offset field and
  // its K-direction stride in the leading-byte-offset field (the reverse of
  // the swizzled MN-major layouts)
  const bool a_tmn = p.a_src == SRC_IM2COL_TAPS_MN;
  const bool b_tmn = p.b_src == SRC_IM2COL_TAPS_MN;
  const uint32_t idesc = p.idesc;
  const int num_acc = p.num_acc;
  const int kb_per_acc = p.kb_per_acc;
  const unsigned long long timeout = p.timeout_ns;
  const uint32_t pipe_addr = smem_u32(pipe);
  // Descriptors of stage 0, K step 0.  The start-address field holds the
  // byte address / 16 in bits 0-13 and every operand lies below 256 KB, so
  // stage s, K step k is the base plus (s * STAGE + k * step) / 16.
  // tap-packed operands (few channels) have no swizzle: a region of
  // [rows][16 bytes] per tap, one K = 16 step is two regions
  const bool taps = p.a_src == SRC_IM2COL_TAPS;
  const uint64_t a0 = taps    ? make_smem_desc_noswizzle(pipe_addr, 2048, 128)
                      : a_tmn ? make_smem_desc_noswizzle(pipe_addr, 128, 1024)
                              : make_smem_desc(pipe_addr, a_mn ? 8192 : 16, 1024);
  // the resident filter (RESB) lies after the stages, one B_BYTES block per
  // reduction block of the unit
  const uint32_t b_base = RESB ? pipe_addr + C::STAGE * C::STAGES : pipe_addr + C::A_BYTES;
  const uint64_t b0 = taps    ? make_smem_desc_noswizzle(pipe_addr + C::A_BYTES, BN * 16, 128)
                      : b_tmn ? make_smem_desc_noswizzle(pipe_addr + C::A_BYTES, 128, 1024)
                              : make_smem_desc(b_base, b_mn ? 8192 : 16, 1024);
  const uint64_t ak = taps ? 4096 / 16 : (a_tmn ? 256 / 16 : (a_mn ? 2048 / 16 : 32 / 16));
  const uint64_t bk = taps ? 2 * BN * 16 / 16 : (b_tmn ? 256 / 16 : (b_mn ? 2048 / 16 : 32 / 16));
  constexpr uint32_t kStageUnits = C::STAGE / 16;
  int stage = 0;        // stage of the first block of the next unit
  uint32_t phase = 0;
  int local = 0;
  // TMEM buffers: two, or four when two epilogue groups take alternate tiles
  const int buf_shift = p.epi_groups == 2 ? 2 : 1;
  const int buf_mask = (1 << buf_shift) - 1;
  bool ok = true;
  if (RESB && unit_first(sc) < sc.units) {  // producer 0 loads it when there is work
    if (!__all_sync(0xffffffffu, mbar_wait(bfull, 0u, abort_flag, timeout))) {
      if (lane == 0) report_failure(p, abort_flag, DEVERR_MMA_FULL_WAIT);
      ok = false;
    }
    tc_fence_after_sync();
  }
  // One issuer per unit (p.one_issuer, 64-wide plans of short reductions): the issuers take alternate units whole, each into the
  // unit's one accumulator.  A stage then serves both issuers over time, so
  // both take part in every stage's release: the issuer that skips a unit
  // waits for each of its fills in order and arrives on the stage's empty
  // barrier (count 2), the other commits there after its MMAs.  The producer
  // cannot refill a stage before both have seen the fill, so neither issuer
  // can fall two phases behind on a stage (where a parity wait would take
  // the phase after next for the one it wants, and never end).
  const bool one = NI == 2 && p.one_issuer != 0;
  const int rstep = one ? 1 : NI;
  UnitWalk uw;
  for (walk_begin(p, sc, uw); ok && uw.u < sc.units; walk_next(p, sc, uw)) {
    const Work w = walk_work(p, sc, uw);
    const int nk = w.kb1 - w.kb0;
    if (nk <= 0) continue;  // no reduction: the epilogue writes beta*Cin alone
    if (one && (local & 1) != issuer) {
      int st = stage;
      uint32_t ph = phase;
      for (int rel = 0; rel < nk; ++rel) {
        if (!__all_sync(0xffffffffu, mbar_wait(&full[st], ph, abort_flag, timeout))) {
          if (lane == 0) report_failure(p, abort_flag, DEVERR_MMA_FULL_WAIT);
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive(&empty[st]);  // this issuer's release of the fill
        __syncwarp();
        if (++st == STAGES) {
          st = 0;
          ph ^= 1u;
        }
      }
      const int adv = stage + nk;
      const int wraps = adv / STAGES;
      stage = adv - wraps * STAGES;
      phase ^= static_cast<uint32_t>(wraps & 1);
      ++local;
      continue;
    }
    const int buf = local & buf_mask;
    const uint32_t tph = static_cast<uint32_t>(local >> buf_shift) & 1u;
    if (!__all_sync(0xffffffffu, mbar_wait(&tempty[buf], tph ^ 1u, abort_flag, timeout))) {
      if (lane == 0) report_failure(p, abort_flag, DEVERR_MMA_TMEM_WAIT);
      break;
    }
    tc_fence_after_sync();
    uint32_t d = tmem_base + static_cast<uint32_t>((buf * num_acc + (one ? 0 : issuer)) * BN);
    const int r0 = one ? 0 : first_rel(issuer, NI, stage);  // stage has the parity of q0
    int st = stage + r0;
    uint32_t ph = phase;
    if (st >= STAGES) {
      st -= STAGES;
      ph ^= 1u;
    }
    int left = kb_per_acc;   // blocks still to add into the current accumulator
    uint32_t acc = 0u;       // 0: the next MMA overwrites the accumulator
    for (int rel = r0; rel < nk; rel += rstep) {
      if (!__all_sync(0xffffffffu, mbar_wait(&full[st], ph, abort_flag, timeout))) {
        if (lane == 0) report_failure(p, abort_flag, DEVERR_MMA_FULL_WAIT);
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint64_t ad = a0 + st * kStageUnits;
      const uint64_t bd =
          RESB ? b0 + static_cast<uint64_t>(rel) * (C::B_BYTES / 16) : b0 + st * kStageUnits;
      if (elect_one_sync()) {
        mma_issue<PAIR>(d, ad, bd, idesc, acc);
        mma_issue<PAIR>(d, ad + ak, bd + bk, idesc, 1u);
        mma_issue<PAIR>(d, ad + 2 * ak, bd + 2 * bk, idesc, 1u);
        mma_issue<PAIR>(d, ad + 3 * ak, bd + 3 * bk, idesc, 1u);
        mma_commit<PAIR>(&empty[st]);  // frees the stage once these MMAs have read it
      }
      __syncwarp();
      acc = 1u;
      if (--left == 0) {        // next accumulator of this issuer
        left = kb_per_acc;
        d += static_cast<uint32_t>(NI * BN);
        acc = 0u;
      }
      st += rstep;
      if (st >= STAGES) {
        st -= STAGES;
        ph ^= 1u;
      }
    }
    if (!ok) break;
    const int adv = stage + nk;
    const int wraps = adv / STAGES;
    stage = adv - wraps * STAGES;
    phase ^= static_cast<uint32_t>(wraps & 1);
    if (elect_one_sync()) mma_commit<PAIR>(&tfull[buf]);  // this issuer's part is ready
    __syncwarp();
    ++local;
  }
  // Every MMA issued must complete before TMEM is released.
  if (elect_one_sync()) mma_commit<PAIR>(done_bar);
  __syncwarp();
  if (!__all_sync(0xffffffffu, mbar_wait(done_bar, 0, nullptr, timeout)) && lane == 0)
    report_failure(p, abort_flag, DEVERR_TEARDOWN_WAIT);
}

// ---------------------------------------------------------------------------
// Epilogue (4 warps; warp w reads TMEM lanes 32*(w%4) .. +31)
// ---------------------------------------------------------------------------
// Two floats to one packed pair (a in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack2(float a, float b, int bf16) {
  if (bf16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8], int bf16) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint16_t lo = static_cast<uint16_t>(w[i] & 0xFFFFu);
    const uint16_t hi = static_cast<uint16_t>(w[i] >> 16);
    if (bf16) {
      f[2 * i] = __bfloat162float(__ushort_as_bfloat16(lo));
      f[2 * i + 1] = __bfloat162float(__ushort_as_bfloat16(hi));
    } else {
      f[2 * i] = __half2float(__ushort_as_half(lo));
      f[2 * i + 1] = __half2float(__ushort_as_half(hi));
    }
  }
}


// Writes 32 staged rows to global memory with coalesced 16-byte stores.
// Each lane first puts its own row's n16 16-byte pieces in the warp's staging
// buffer; then the warp writes row r's piece j to base + off(r) + 16*j, where
// off(r) is lane r's byte offset (negative: the row is outside the output).
__device__ __forceinline__ void warp_store_rows(uint8_t* stage, const uint4* mine, int n16,
                                                long long my_off, uint8_t* base, int lane) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < n16) *reinterpret_cast<uint4*>(stage + lane * kStagePitch + j * 16) = mine[j];
  __syncwarp();
  for (int c = lane; c < 32 * n16; c += 32) {
    const int r = c / n16;
    const int j = c - r * n16;
    const long long off = __shfl_sync(0xffffffffu, my_off, r);
    if (off >= 0)
      *reinterpret_cast<uint4*>(base + off + j * 16) =
          *reinterpret_cast<const uint4*>(stage + r * kStagePitch + j * 16);
  }
  __syncwarp();
}

// Where a warp's 32 output rows go in the output map: row y of a 2D
// [rows][cols] map, or (strided dgrad, b >= 0) the line (b, tw.., a, hrow)
// of the 5D view of dX, the 32 rows being grid columns tw .. tw + 31 of one
// residue-class row (columns past the image are clipped by the map).
struct OutAt {
  int y;
  int b, tw, a, hrow;
};

__device__ __forceinline__ void tma_store_out(const CUtensorMap* map, const void* src, int x,
                                              const OutAt& at) {
  if (at.b >= 0)
    tma_store_5d(map, src, x, at.b, at.tw, at.a, at.hrow);
  else
    tma_store_2d(map, src, x, at.y);
}

// Stages one 32-row box (this lane's row: n16 16-byte pieces, n16 = 2 or 4)
// in the warp's next staging buffer, in the 32-/64-byte TMA swizzle, then
// stores it with one TMA store at column x of the rows `at`.  The buffer is
// reused only after the store that last read it has finished reading.
__device__ __forceinline__ void warp_tma_store_box(uint8_t* stage, int& flip, const uint4* mine,
                                                   int n16, const CUtensorMap* map, int x,
                                                   const OutAt& at, int lane) {
  uint8_t* buf = stage + flip * kStageBufBytes;
  if (lane == 0) bulk_wait_group_read<1>();
  __syncwarp();
  if (n16 == 4) {
    // 64-byte rows, 64-byte swizzle: piece j lands in slot j ^ ((row >> 1) & 3)
    const int x3 = (lane >> 1) & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ x3) << 4)) = mine[j];
  } else {
    // 32-byte rows, 32-byte swizzle: piece j lands in slot j ^ ((row >> 2) & 1)
    const int x1 = (lane >> 2) & 1;
#pragma unroll
    for (int j = 0; j < 2; ++j)
      *reinterpret_cast<uint4*>(buf + lane * 32 + ((j ^ x1) << 4)) = mine[j];
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_out(map, buf, x, at);
    bulk_commit_group();
  }
  flip ^= 1;
}

// alpha * acc (+ beta * Cin) (+ bias) for 32 columns held as 16 pairs, then
// the RNE cast to 16 bits and ReLU: packed fp32x2 arithmetic (each lane
// rounded as its scalar form); ReLU is the conversion's clamp of negative
// results to zero (rounding is monotonic and keeps zero, so clamping the
// rounded value equals rounding the clamped one).
__device__ __forceinline__ void epi_finish(float2 (&f)[16], const uint4 (&craw)[4],
                                           const uint4 (&braw)[4], const uint32_t* bias_s,
                                           bool bias_cached, bool has_bias, int n0, float alpha,
                                           float beta, int relu, int bf16, uint32_t (&pk)[16]) {
  if (alpha != 1.0f) {
    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = __fmul2_rn(a2, f[i]);
  }
  if (beta != 0.0f) {
    const float2 b2 = make_float2(beta, beta);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float c[8];
      unpack8(craw[g], c, bf16);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        f[4 * g + i] = __ffma2_rn(b2, make_float2(c[2 * i], c[2 * i + 1]), f[4 * g + i]);
    }
  }
  if (has_bias) {
    if (bias_cached) {
      const float4* bs = reinterpret_cast<const float4*>(bias_s + n0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 b4 = bs[q];
        f[2 * q] = __fadd2_rn(f[2 * q], make_float2(b4.x, b4.y));
        f[2 * q + 1] = __fadd2_rn(f[2 * q + 1], make_float2(b4.z, b4.w));
      }
    } else {
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float b[8];
        unpack8(braw[g], b, bf16);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          f[4 * g + i] = __fadd2_rn(f[4 * g + i], make_float2(b[2 * i], b[2 * i + 1]));
      }
    }
  }
  // RNE to 16 bits, two values per instruction (x in the low half); with
  // ReLU the conversion's .relu form clamps negative results to +0.
  if (relu) {
    if (bf16) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        asm("cvt.rn.relu.bf16x2.f32 %0, %1, %2;" : "=r"(pk[i]) : "f"(f[i].y), "f"(f[i].x));
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        asm("cvt.rn.relu.f16x2.f32 %0, %1, %2;" : "=r"(pk[i]) : "f"(f[i].y), "f"(f[i].x));
    }
  } else {
    if (bf16) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(pk[i]) : "f"(f[i].y), "f"(f[i].x));
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(pk[i]) : "f"(f[i].y), "f"(f[i].x));
    }
  }
}

// Whether accumulator a (issuer a % ni, group a / ni) received at least one
// reduction block of a unit of nk blocks starting at sequence number q0.
__device__ __forceinline__ bool acc_used(int kb_per_acc, int a, int ni, int nk, int q0) {
  const int grp = a / ni;
  return static_cast<long long>(grp) * kb_per_acc * ni + first_rel(a % ni, ni, q0) < nk;
}

// Integer sum of the used accumulators of 32 columns (chunk at column
// offset col of each accumulator): each holds an exact integer below 2^24 in
// magnitude, converted exactly; the adds wrap modulo 2^32 like an int32
// accumulator.
__device__ __forceinline__ void int_acc_sum(uint32_t t_row, uint32_t col, int num_acc, int bn,
                                            int kb_per_acc, int ni, int nk, int q0,
                                            int (&iacc)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) iacc[i] = 0;
  for (int a = 0; a < num_acc; ++a) {
    if (!acc_used(kb_per_acc, a, ni, nk, q0)) continue;
    uint32_t v[32];
    tmem_ld_32x32b_x32(t_row + a * bn + col, v);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i)
      iacc[i] = static_cast<int>(static_cast<uint32_t>(iacc[i]) +
                                 static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[i]))));
  }
}

// Epilogue scalars, copied into registers once.
struct EpiCtx {
  Sched sc;
  void* out;
  const void* cin;
  const void* bias;
  float alpha, beta;
  int relu, out_bf16, N_gemm, out_C, out_H, out_W, out_D;
  int num_acc, kb_per_acc;
  long long ws_split_stride;
  int ws_ld;
  uint32_t rq_mant;
  int rq_exp;
  unsigned long long timeout;
  int use_tma;
  int store5;           // TMA stores through the 5D strided-dgrad view (see OutAt)
  int one_issuer;       // each unit is issued by one issuer into one accumulator
  int box64;            // 16-bit output boxes of 64 columns (128-byte swizzle)
  int ws_rows_per_split;   // M_pad (wgrad)
  int int_acc;             // accumulators hold exact integers: sum and store them as int32
  int out_f32;             // write alpha * acc as fp32
  const CUtensorMap* mapY;
};

template <int BN, bool PAIR, bool VOL, bool S16>
__device__ __forceinline__ void run_epilogue(const ConvGemmParams& p, uint64_t* tfull,
                                             uint64_t* tempty, uint32_t tmem_base,
                                             volatile int* abort_flag, int warp,
                                             uint8_t* stage_buf, const uint32_t* bias_s) {
  constexpr int NI = Cfg<BN, PAIR>::NI;
  EpiCtx e;
  e.sc = load_sched<PAIR>(p);
  e.out = p.out;
  e.cin = p.cin;
  e.bias = p.bias;
  e.alpha = p.alpha;
  e.beta = p.beta;
  e.relu = p.relu;
  e.out_bf16 = p.out_bf16;
  e.N_gemm = p.N_gemm;
  e.out_C = p.out_C;
  e.out_H = p.out_H;
  e.out_W = p.out_W;
  e.out_D = p.out_D;
  e.num_acc = p.num_acc;
  e.kb_per_acc = p.kb_per_acc;
  e.ws_split_stride = p.ws_split_stride;
  e.ws_ld = p.ws_ld;
  e.rq_mant = p.rq_mant;
  e.rq_exp = p.rq_exp;
  e.timeout = p.timeout_ns;
  e.use_tma = p.use_tma_store;
  e.store5 = p.use_tma_store && p.store_5d && e.sc.epi == EPI_STORE;
  e.one_issuer = p.one_issuer;
  e.box64 = p.use_tma_store && p.store_box64 && e.sc.epi == EPI_STORE;
  e.ws_rows_per_split = p.tiles_m_total * kBlockM;
  e.int_acc = S16 ? 0 : p.int_acc;
  e.out_f32 = S16 ? 0 : p.out_f32;
  e.mapY = &p.mapY;
  // bias_s holds the whole bias vector when it fits in kBiasBytes (fp32 for
  // the 16-bit passes, int32 for int8); every lane reads the same entries,
  // so the reads are shared-memory broadcasts.
  const bool bias_cached = p.bias_cached != 0;
  // int8 multiplier M = rq_mant * 2^-rq_sh (uniform across the launch)
  const int rq_sh_true = -e.rq_exp;
  const int rq_mode = rq_sh_true < 1 ? 1 : (rq_sh_true > 62 ? 2 : 0);
  const int rq_sh = rq_sh_true < 1 ? 1 : (rq_sh_true > 62 ? 62 : rq_sh_true);
  const long long rq_half_m1 = (1LL << (rq_sh - 1)) - 1;

  const int quarter = warp & 3;
  // One group: warps 4-7 take the first half of every tile's columns and
  // warps 8-11 the second.  Two groups: warps 4-7 take the tiles with even
  // accumulator sequence number whole and warps 8-11 the odd ones, each
  // group double-buffered in its own two of four TMEM buffers, so every
  // buffer is only ever waited on by one group, in order.
  const int groups = p.epi_groups == 2 ? 2 : 1;
  const int group = groups == 2 ? (warp - kEpiWarp0) >> 2 : 0;
  const int half = groups == 2 ? 0 : (warp - kEpiWarp0) >> 2;   // which half of the columns
  const int buf_shift = groups == 2 ? 2 : 1;
  const int buf_mask = (1 << buf_shift) - 1;
  const int lane = threadIdx.x & 31;
  const int row = quarter * 32 + lane;
  uint8_t* stage = stage_buf + (warp - kEpiWarp0) * kStageWarpBytes;
  const int j0 = half * (BN / 64);
  const int j1 = groups == 2 ? BN / 32 : j0 + BN / 64;
  int flip = 0;  // staging buffer to use next
  int local = 0;
  int plain = 0;  // units without accumulators seen so far (they alternate between groups)
  int qseq = 0;  // sequence number of the next reduction block (see run_mma)
  const int M0 = p.sub[0].M;  // GEMM rows when there is one sub-problem
  const bool one_sub = e.sc.nsub == 1;
  UnitWalk uw;
  // Every unit has blocks (p.all_acc): tile parity alone names the group, so
  // the other group's units are passed over before any decoding (on the fast
  // walk their block count comes with the walk).
  const bool skip_fast = groups == 2 && p.all_acc && uw_fast_possible(e.sc);
  for (walk_begin(p, e.sc, uw); uw.u < e.sc.units; walk_next(p, e.sc, uw)) {
    if (skip_fast && (local & 1) != group) {
      qseq += uw.nk;
      ++local;
      continue;
    }
    const Work w = walk_work(p, e.sc, uw);
    const int nk = w.kb1 - w.kb0;
    const bool has_acc = nk > 0;
    const int q0 = qseq;
    if (has_acc) qseq += nk;
    // which of the first NI accumulators hold blocks (NI == 2: at least one)
    // (a unit issued by a single issuer has one accumulator, at offset 0)
    const bool use1 = NI >= 2 && !e.one_issuer && acc_used(e.kb_per_acc, 1, NI, nk, q0);
    const uint32_t lone =
        (NI >= 2 && !e.one_issuer && !acc_used(e.kb_per_acc, 0, NI, nk, q0)) ? BN : 0u;
    const int buf = local & buf_mask;
    const uint32_t tph = static_cast<uint32_t>(local >> buf_shift) & 1u;
    if (groups == 2 && ((has_acc ? local : plain) & 1) != group) {
      if (has_acc) ++local; else ++plain;  // the other group's unit
      continue;
    }
    if (has_acc) {
      if (!mbar_wait(&tfull[buf], tph, abort_flag, e.timeout)) {
        report_failure(p, abort_flag, DEVERR_EPI_WAIT);
        break;
      }
      tc_fence_after_sync();
    }
    const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                           static_cast<uint32_t>(buf * e.num_acc * BN);
    if (!S16 && e.sc.epi == EPI_PARTIAL) {
      float* ws = static_cast<float*>(e.out) + static_cast<long long>(w.split) * e.ws_split_stride;
      const long long my_off =
          static_cast<long long>(w.tile_m * kBlockM + row) * e.ws_ld * 4;  // bytes
      // writes 32 fp32 partial sums of this row (chunk j) as two 16-column boxes
      auto store_partial = [&](const float (&acc)[32], int j) {
        uint8_t* base = reinterpret_cast<uint8_t*>(ws + w.tile_n * BN + j * 32);
#pragma unroll
        for (int h = 0; h < 2; ++h) {       // 16 fp32 columns (64 bytes) at a time
          uint4 o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            o[i] = make_uint4(__float_as_uint(acc[16 * h + 4 * i]),
                              __float_as_uint(acc[16 * h + 4 * i + 1]),
                              __float_as_uint(acc[16 * h + 4 * i + 2]),
                              __float_as_uint(acc[16 * h + 4 * i + 3]));
          if (e.use_tma)
            warp_tma_store_box(stage, flip, o, 4, e.mapY, w.tile_n * BN + j * 32 + h * 16,
                               OutAt{w.split * e.ws_rows_per_split + w.tile_m * kBlockM +
                                         quarter * 32,
                                     -1, 0, 0, 0},
                               lane);
          else
            warp_store_rows(stage, o, 4, my_off, base + h * 64, lane);
        }
      };
#pragma unroll 1
      for (int j = j0; j < j1; ++j) {
        if (e.int_acc) {
          // int8 wgrad: the int32 sum of the accumulators, stored as its bits
          int iacc[32];
          int_acc_sum(t_row, static_cast<uint32_t>(j * 32), e.num_acc, BN, e.kb_per_acc, NI, nk,
                      q0, iacc);
          float acc[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = __int_as_float(iacc[i]);
          store_partial(acc, j);
          continue;
        }
        if (NI == 1 && e.num_acc == 1 && j + 1 < j1) {
          // one accumulator: two chunks per TMEM round trip
          uint32_t v[32], u2[32];
          tmem_ld_32x32b_x32(t_row + j * 32, v);
          tmem_ld_32x32b_x32(t_row + (j + 1) * 32, u2);
          tmem_ld_wait();
          float acc[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(v[i]);
          store_partial(acc, j);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(u2[i]);
          store_partial(acc, j + 1);
          ++j;
          continue;
        }
        float acc[32];
        {
          uint32_t v[32];
          if (use1 && lone == 0u) {
            uint32_t u[32];
            tmem_ld_32x32b_x32(t_row + j * 32, v);
            tmem_ld_32x32b_x32(t_row + BN + j * 32, u);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              acc[i] = __fadd_rn(__uint_as_float(v[i]), __uint_as_float(u[i]));
          } else {
            tmem_ld_32x32b_x32(t_row + lone + j * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(v[i]);
          }
        }
        for (int a = 2; a < e.num_acc; ++a) {
          if (!acc_used(e.kb_per_acc, a, NI, nk, q0)) continue;
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_row + a * BN + j * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = __fadd_rn(acc[i], __uint_as_float(v[i]));
        }
        store_partial(acc, j);
      }
    } else {
      const int m = w.tile_m * kBlockM + row;
      bool valid = m < (one_sub ? M0 : p.sub[w.sub].M);
      OutAt at{w.tile_m * kBlockM + quarter * 32, -1, 0, 0, 0};
      if (e.store5) {
        // the warp's 32 rows: one residue-class row of dX (grid width a
        // multiple of 32), written through the 5D view
        const SubProblem& sp = p.sub[w.sub];
        const int per_plane = sp.Hs * sp.Ws;
        const int m0 = at.y;
        const int n = m0 / per_plane;
        const int rem = m0 - n * per_plane;
        const int th = rem / sp.Ws;
        at.b = sp.out_w0;
        at.tw = rem - th * sp.Ws;
        at.a = sp.out_h0;
        at.hrow = n * sp.Hs + th;
      }
      long long row_off = 0;  // elements; only the row-store and Cin paths use it
      if (valid && (!e.use_tma || e.beta != 0.0f)) {
        const SubProblem& sp = p.sub[w.sub];
        const int Hs = sp.Hs, Ws = sp.Ws;
        const int per_plane = Hs * Ws;
        int n, rem;
        long long img_row;  // output image (and depth) index, in output planes
        if (VOL && sp.Ds > 0) {
          const int per_img = sp.Ds * per_plane;
          n = m / per_img;
          const int r3 = m - n * per_img;
          const int td = r3 / per_plane;
          rem = r3 - td * per_plane;
          img_row = static_cast<long long>(n) * e.out_D + sp.out_d0 + sp.out_sd * td;
        } else {
          n = m / per_plane;
          rem = m - n * per_plane;
          img_row = n;
        }
        const int th = rem / Ws;
        const int tw = rem - th * Ws;
        if (sp.ws_valid > 0 && tw >= sp.ws_valid) valid = false;  // row padding
        const int oh = sp.out_h0 + sp.out_sh * th;
        const int ow = sp.out_w0 + sp.out_sw * tw;
        row_off = ((img_row * e.out_H + oh) * e.out_W + ow) * static_cast<long long>(e.out_C);
      }
      // 64-column boxes with one accumulator, no Cin and a staged (or no)
      // bias: chunks go in pairs, one TMEM round trip and one store per pair
      // (with 32-column boxes the pair's extra live registers cost more than
      // the saved round trip).
      const bool pair1 = (NI == 1 || e.one_issuer) && e.box64 && e.num_acc == 1 && has_acc &&
                         e.beta == 0.0f && (e.bias == nullptr || bias_cached);
#pragma unroll 1
      for (int j = j0; j < j1; ++j) {
        const int n0 = w.tile_n * BN + j * 32;
        if (n0 >= e.N_gemm) break;  // warp-uniform
        const int ncols = min(32, e.N_gemm - n0);
        if (e.out_f32) {
          // alpha * (the issuers' accumulators added in the 16-bit path's
          // order), as fp32: 16 columns (64 bytes) per row store, the last
          // one cut to the valid columns (a multiple of 4)
          float v[32];
          if (has_acc) {
            uint32_t a0[32];
            tmem_ld_32x32b_x32(t_row + lone + j * 32, a0);
            if (use1 && lone == 0u) {
              uint32_t a1[32];
              tmem_ld_32x32b_x32(t_row + BN + j * 32, a1);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                v[i] = __fadd_rn(__uint_as_float(a0[i]), __uint_as_float(a1[i]));
            } else {
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(a0[i]);
            }
            for (int a = 2; a < e.num_acc; ++a) {
              if (!acc_used(e.kb_per_acc, a, NI, nk, q0)) continue;
              tmem_ld_32x32b_x32(t_row + a * BN + j * 32, a0);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __fadd_rn(v[i], __uint_as_float(a0[i]));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(e.alpha, v[i]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (16 * h >= ncols) break;  // warp-uniform
            const int n16 = min(4, (ncols - 16 * h) / 4);
            const uint4 o[4] = {
                make_uint4(__float_as_uint(v[16 * h]), __float_as_uint(v[16 * h + 1]),
                           __float_as_uint(v[16 * h + 2]), __float_as_uint(v[16 * h + 3])),
                make_uint4(__float_as_uint(v[16 * h + 4]), __float_as_uint(v[16 * h + 5]),
                           __float_as_uint(v[16 * h + 6]), __float_as_uint(v[16 * h + 7])),
                make_uint4(__float_as_uint(v[16 * h + 8]), __float_as_uint(v[16 * h + 9]),
                           __float_as_uint(v[16 * h + 10]), __float_as_uint(v[16 * h + 11])),
                make_uint4(__float_as_uint(v[16 * h + 12]), __float_as_uint(v[16 * h + 13]),
                           __float_as_uint(v[16 * h + 14]), __float_as_uint(v[16 * h + 15]))};
            warp_store_rows(stage, o, n16, valid ? row_off * 4 : -1LL,
                            static_cast<uint8_t*>(e.out) + static_cast<long long>(n0 + 16 * h) * 4,
                            lane);
          }
          continue;
        }
        if (e.int_acc) {
          // int8 dgrad: the exact int32 sum, written as two 16-column rows
          // of 64 bytes (the column count is a multiple of 16)
          int iacc[32];
          int_acc_sum(t_row, static_cast<uint32_t>(j * 32), e.num_acc, BN, e.kb_per_acc, NI, nk,
                      q0, iacc);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (16 * h >= ncols) break;  // warp-uniform
            const uint4 o[4] = {
                make_uint4(iacc[16 * h], iacc[16 * h + 1], iacc[16 * h + 2], iacc[16 * h + 3]),
                make_uint4(iacc[16 * h + 4], iacc[16 * h + 5], iacc[16 * h + 6], iacc[16 * h + 7]),
                make_uint4(iacc[16 * h + 8], iacc[16 * h + 9], iacc[16 * h + 10], iacc[16 * h + 11]),
                make_uint4(iacc[16 * h + 12], iacc[16 * h + 13], iacc[16 * h + 14],
                           iacc[16 * h + 15])};
            warp_store_rows(stage, o, 4, valid ? row_off * 4 : -1LL,
                            static_cast<uint8_t*>(e.out) + static_cast<long long>(n0 + 16 * h) * 4,
                            lane);
          }
          continue;
        }
        if (!S16 && e.sc.epi == EPI_INT8) {
          int iacc[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) iacc[i] = 0;
          for (int a = 0; a < e.num_acc; ++a) {
            if (!acc_used(e.kb_per_acc, a, NI, nk, q0)) continue;
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_row + a * BN + j * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) iacc[i] += __float2int_rn(__uint_as_float(v[i]));
          }
          int32_t bv[32];
          const int32_t* bias = bias_cached ? reinterpret_cast<const int32_t*>(bias_s)
                                            : static_cast<const int32_t*>(e.bias);
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            int4 b4 = make_int4(0, 0, 0, 0);
            if (bias && 4 * g < ncols) b4 = *reinterpret_cast<const int4*>(bias + n0 + 4 * g);
            bv[4 * g] = b4.x; bv[4 * g + 1] = b4.y; bv[4 * g + 2] = b4.z; bv[4 * g + 3] = b4.w;
          }
          uint32_t packed[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) packed[i] = 0u;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            // |acc| <= 4096 * 2^14 = 2^26, so |t| < 2^32: exact in 64 bits
            long long t = static_cast<long long>(iacc[i]) + bv[i];
            if (e.relu && t < 0) t = 0;
            const int y = requant_rne(t, e.rq_mant, rq_sh, rq_half_m1, rq_mode);
            packed[i >> 2] |= (static_cast<uint32_t>(y) & 0xFFu) << (8 * (i & 3));
          }
          const uint4 o[2] = {make_uint4(packed[0], packed[1], packed[2], packed[3]),
                              make_uint4(packed[4], packed[5], packed[6], packed[7])};
          if (e.use_tma)
            warp_tma_store_box(stage, flip, o, 2, e.mapY, n0, at, lane);
          else
            warp_store_rows(stage, o, ncols / 16, valid ? row_off : -1LL,
                            static_cast<uint8_t*>(e.out) + n0, lane);
        } else {
          uint32_t pk[16];
          const uint4 zero4[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                                  make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
          if (pair1 && j + 1 < j1 && n0 + 32 < e.N_gemm) {
            // One accumulator, 64-column boxes: this chunk and the next come
            // out of TMEM in one round trip and fill one box, stored here.
            uint32_t v[32], u[32];
            tmem_ld_32x32b_x32(t_row + j * 32, v);
            tmem_ld_32x32b_x32(t_row + (j + 1) * 32, u);
            tmem_ld_wait();
            if (lane == 0) bulk_wait_group_read<0>();
            __syncwarp();
            const int x7 = lane & 7;
            float2 f[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              f[i] = make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            epi_finish(f, zero4, zero4, bias_s, true, e.bias != nullptr, n0, e.alpha, 0.0f,
                       e.relu, e.out_bf16, pk);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(stage + lane * 128 + ((q ^ x7) << 4)) =
                  make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              f[i] = make_float2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
            epi_finish(f, zero4, zero4, bias_s, true, e.bias != nullptr, n0 + 32, e.alpha, 0.0f,
                       e.relu, e.out_bf16, pk);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(stage + lane * 128 + (((4 + q) ^ x7) << 4)) =
                  make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_out(e.mapY, stage, n0, at);
              bulk_commit_group();
            }
            ++j;          // the pair's second chunk is done
            continue;
          } else {
            // bias for these 32 columns, loaded before the accumulators so the
            // loads overlap the TMEM reads
            uint4 braw[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                             make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
            if (e.bias && !bias_cached) {
              const uint16_t* bias = static_cast<const uint16_t*>(e.bias);
#pragma unroll
              for (int g = 0; g < 4; ++g)
                if (8 * g < ncols) braw[g] = *reinterpret_cast<const uint4*>(bias + n0 + 8 * g);
            }
            uint4 craw[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                             make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
            if (e.beta != 0.0f && valid) {
              const uint16_t* cin = static_cast<const uint16_t*>(e.cin) + row_off + n0;
#pragma unroll
              for (int g = 0; g < 4; ++g)
                if (8 * g < ncols) craw[g] = *reinterpret_cast<const uint4*>(cin + 8 * g);
            }
            float2 f[16];
            if (has_acc) {
              uint32_t v[32];
              if (use1 && lone == 0u) {
                // both issuers' accumulators in flight together: one TMEM
                // round trip instead of two
                uint32_t u[32];
                tmem_ld_32x32b_x32(t_row + j * 32, v);
                tmem_ld_32x32b_x32(t_row + BN + j * 32, u);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  f[i] = __fadd2_rn(
                      make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                      make_float2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1])));
              } else {
                tmem_ld_32x32b_x32(t_row + lone + j * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  f[i] = make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
              }
              for (int a = 2; a < e.num_acc; ++a) {
                if (!acc_used(e.kb_per_acc, a, NI, nk, q0)) continue;
                tmem_ld_32x32b_x32(t_row + a * BN + j * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  f[i] = __fadd2_rn(f[i], make_float2(__uint_as_float(v[2 * i]),
                                                      __uint_as_float(v[2 * i + 1])));
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) f[i] = make_float2(0.0f, 0.0f);
            }
            epi_finish(f, craw, braw, bias_s, bias_cached, e.bias != nullptr, n0, e.alpha,
                       e.beta, e.relu, e.out_bf16, pk);
          }
          uint4 o[4];
#pragma unroll
          for (int g = 0; g < 4; ++g) o[g] = make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
          if (e.box64) {
            // Two consecutive chunks fill one 32-row x 64-column box (128-byte
            // rows, 128-byte swizzle: piece q of row r in slot q ^ (r & 7)),
            // stored with one TMA store; the warp's whole 4 KB staging area
            // is the box, reused once the previous box has been read.
            const int hh = (j - j0) & 1;
            if (hh == 0) {
              if (lane == 0) bulk_wait_group_read<0>();
              __syncwarp();
            }
            const int x7 = lane & 7;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(stage + lane * 128 + (((4 * hh + q) ^ x7) << 4)) = o[q];
            if (hh == 1 || j + 1 == j1 || n0 + 32 >= e.N_gemm) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_out(e.mapY, stage, n0 - 32 * hh, at);
                bulk_commit_group();
              }
            }
          } else if (e.use_tma)
            warp_tma_store_box(stage, flip, o, 4, e.mapY, n0, at, lane);
          else
            warp_store_rows(stage, o, ncols / 8, valid ? row_off * 2 : -1LL,
                            static_cast<uint8_t*>(e.out) + static_cast<long long>(n0) * 2, lane);
        }
      }
    }
    if (has_acc) {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)  // the even CTA's issuers wait for both CTAs' epilogues
          mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[buf]), 0));
        else
          mbar_arrive(&tempty[buf]);
      }
      ++local;
    } else {
      ++plain;
    }
  }
  // every TMA store this warp issued must complete before the CTA exits
  if (lane == 0) bulk_wait_group<0>();
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Kernel
// ---------------------------------------------------------------------------
__host__ __device__ constexpr uint32_t tmem_cols_for(uint32_t need) {
  uint32_t c = 32;
  while (c < need) c <<= 1;
  return c;
}

// PAIR: launched as clusters of two CTAs (p.pair set), each pair working on
// 256-row units with tcgen05.mma.cta_group::2 issued by the even CTA.
// S16: the epilogue holds only the 16-bit store path (fprop and dgrad with
// 16-bit outputs); the other kernels carry every epilogue.  The smaller
// epilogue runs faster on the layers it bounds (measured: 1x1 64->256 fprop
// -10 %, strided 112x112 dgrad -11 %, the packed stem fprop -7 %, the 3x3
// layers 0-5 %), through fewer instruction fetch stalls.
template <int BN, bool PAIR, bool VOL, bool RESB = false, bool S16 = false>
__global__ void __launch_bounds__(kThreads, 1)
    conv_gemm_kernel(const __grid_constant__ ConvGemmParams p) {
  using C = Cfg<BN, PAIR, RESB>;
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  if (static_cast<int>(smem - smem_raw) + C::USED > C::SMEM) {
    // the dynamic shared memory base leaves too little room after aligning
    // it (never seen: the base is 1024-byte aligned); nothing has started yet
    pdl_wait();
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, static_cast<unsigned int>(DEVERR_SMEM_LAYOUT));
    return;
  }
  uint8_t* pipe = smem;
  uint8_t* stage_buf = smem + C::PIPE;
  uint32_t* bias_s = reinterpret_cast<uint32_t*>(smem + C::PIPE + C::EPI_STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::PIPE + C::EPI_STAGE + kBiasBytes);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 4;
  uint64_t* done_bar = tempty + 4;  // one per issuer
  uint64_t* bfull = done_bar + 2;   // the resident filter (RESB)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nbuf = p.epi_groups == 2 ? 4 : 2;  // TMEM accumulator buffers
  const uint32_t tmem_cols = tmem_cols_for(static_cast<uint32_t>(nbuf * p.num_acc * BN));
  const int rank = PAIR ? static_cast<int>(cluster_ctarank() & 1u) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], p.one_issuer ? 2 : 1);  // one issuer per unit: both release
    }
    // a tile's epilogue is 8 warps (one group) or 4 (two groups); with pairs
    // the even CTA's TMEM-empty barriers count both CTAs' epilogues
    const int epi_warps = p.epi_groups == 2 ? kEpiWarps / 2 : kEpiWarps;
    for (int b = 0; b < 4; ++b) {
      mbar_init(&tfull[b], p.one_issuer ? 1 : C::NI);  // one issuer per unit, or all
      mbar_init(&tempty[b], PAIR ? 2 * epi_warps : epi_warps);
    }
    mbar_init(&done_bar[0], 1);
    mbar_init(&done_bar[1], 1);
    mbar_init(bfull, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // the barriers above are this CTA's own: the stream's earlier kernel may
  // still run until here, not past it (the bias, the inputs, the outputs)
  pdl_wait();
  if (p.bias_cached) {
    for (int i = threadIdx.x; i < p.N_gemm; i += blockDim.x) {
      if (!S16 && p.epi == EPI_INT8) {
        bias_s[i] = static_cast<const uint32_t*>(p.bias)[i];
      } else {
        const uint16_t b = static_cast<const uint16_t*>(p.bias)[i];
        bias_s[i] = __float_as_uint(p.out_bf16 ? __bfloat162float(__ushort_as_bfloat16(b))
                                               : __half2float(__ushort_as_half(b)));
      }
    }
  }
  if (warp == kMmaWarp0) {
    if (PAIR)
      tmem_alloc_pair(tmem_slot, tmem_cols);  // the same columns in both CTAs
    else
      tmem_alloc(tmem_slot, tmem_cols);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // both CTAs' barriers exist before any copy or commit
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  // Each warpgroup resizes its registers first thing in its role branch, so
  // that all of the role's code is compiled under the new limit.
  if (warp < 4) {
    setmaxnreg_dec<kRegsLow>();
    if (warp < C::NP) {
    if (warp == 0 && lane == 0) {
      for (int i = 0; i < p.nsub; ++i)
        if (p.mapA_valid & (1u << i)) tma_prefetch_map(&p.mapA[i]);
      tma_prefetch_map(&p.mapB);
      if (p.use_tma_store) tma_prefetch_map(&p.mapY);
      if (p.pf_bytes > 0) {
        // Every CTA of the first wave reads the same filter blocks at about
        // the same time; on a cold L2 each first touch then stalls them all.
        // The CTAs instead fetch the filter into L2 up front, each its own
        // share in 32 KB pieces (7x7 512->512 fprop after other layers:
        // 40.9 -> 36.8 us).
        long long per = (p.pf_bytes + gridDim.x - 1) / gridDim.x;
        per = (per + 15) & ~15LL;
        const long long o0 = static_cast<long long>(blockIdx.x) * per;
        const long long o1 = o0 + per < p.pf_bytes ? o0 + per : p.pf_bytes;
        for (long long o = o0; o < o1; o += 32768) {
          const long long n = o1 - o < 32768 ? o1 - o : 32768;
          if (n >= 16)
            prefetch_l2(static_cast<const char*>(p.pf_base) + o, static_cast<uint32_t>(n & ~15LL));
        }
      }
    }
    __syncwarp();
    run_producer<BN, PAIR, VOL, RESB>(p, pipe, full, empty, bfull, abort_flag, warp, lane);
    }
  } else if (warp >= kMmaWarp0) {
    setmaxnreg_dec<kRegsLow>();
    if (warp < kMmaWarp0 + C::NI && (!PAIR || rank == 0))
      run_mma<BN, PAIR, RESB>(p, pipe, full, empty, tfull, tempty, &done_bar[warp - kMmaWarp0],
                              bfull, tmem_base, abort_flag, warp - kMmaWarp0, lane);
  } else {
    setmaxnreg_inc<kRegsEpi>();
    run_epilogue<BN, PAIR, VOL, S16>(p, tfull, tempty, tmem_base, abort_flag, warp, stage_buf,
                                     bias_s);
  }

  tc_fence_before_sync();
  __syncthreads();
  // Neither CTA of a pair leaves while the other may still arrive on its
  // barriers (commits, remote TMEM-empty arrivals) or its MMAs run.
  if (PAIR) cluster_sync_all();
  if (warp == kMmaWarp0) {
    tc_fence_after_sync();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, tmem_cols);
    else
      tmem_dealloc(tmem_base, tmem_cols);
  }
}

// ---------------------------------------------------------------------------
// Halo tiles (stride-1 fprop and dgrad, one 64-channel reduction block, one
// 64-wide column tile, at most kHaloTaps filter taps).  Output positions are
// indexed on a grid whose rows are Wt columns wide (Wt = 32, 64 or 128, at
// least the padded input row), so a 128-row tile is 128 / Wt whole output
// rows of one image.  Every filter tap of such a tile reads the same input
// rows shifted by (off_h * Wt + off_w) grid positions, so one TMA copy of
// the tile's input rows -- the halo: HR = 128 / Wt + (R-1) dil_h + 1 rows of
// Wt pixels, zero outside the image -- feeds all its reduction blocks,
// instead of one im2col copy per tap.  The filter stays resident in shared
// memory.  A block's A operand is the 128 halo rows starting at its offset:
// the descriptor's start moves by whole 128-byte pixel rows, also to rows
// that are not on an 8-row (1024-byte) swizzle boundary.  The 128-byte
// swizzle is a function of the absolute shared-memory address (the 16-byte
// chunk index XOR address bits 7-9), for the TMA that writes the halo and
// the MMA that reads it alike, so the base-offset field stays zero (checked
// on the GPU: with the field set to the start's row within the pattern the
// products were wrong, with it zero exact).  The two issuers take alternate
// units whole (p.one_issuer), each into the unit's single accumulator, so
// the epilogue reads one accumulator and stores 64-column boxes; the other
// issuer still waits for each halo and arrives on its empty barrier, so a
// stage is free only once both issuers have seen it (without one_issuer
// both read every halo, each the blocks of its sequence parity).  Junk columns (grid column >= the output width)
// read neighbouring pixels; the epilogue drops them (ws_valid, and the
// output map clips them).
// ---------------------------------------------------------------------------
struct HaloCfg {
  static constexpr int STAGE = 40960;                    // up to 320 rows of 128 bytes
  static constexpr int STAGES = 3;
  static constexpr int B_BYTES = 64 * kBlockK * 2;       // one 64 x 64 filter block
  static constexpr int RES_BYTES = kHaloTaps * B_BYTES;  // after the stages
  static constexpr int PIPE = STAGE * STAGES + RES_BYTES;
  static constexpr int EPI_STAGE = kEpiWarps * kStageWarpBytes;
  static constexpr int BAR_BYTES = 256;
  static constexpr int NI = 2;
  static constexpr int NP = STAGES;  // producer warp i owns stage i
  static constexpr int USED = PIPE + EPI_STAGE + kBiasBytes + BAR_BYTES;
  static constexpr int SMEM = kSmemLimit;
  static_assert(USED <= kSmemLimit, "exceeds the 227 KB of shared memory a CTA may use");
  static_assert(STAGE % 1024 == 0 && PIPE % 1024 == 0, "swizzle atoms need 1024-byte alignment");
  static_assert(2 * STAGES + 11 <= (BAR_BYTES - 8) / 8, "barrier area too small");
};

// Producer warp `pid` (0..2) fills halo stage pid for every third unit of
// this CTA; producer 0 first loads the resident filter.
__device__ __forceinline__ void run_producer_halo(const ConvGemmParams& p, uint8_t* pipe,
                                                  uint64_t* full, uint64_t* empty,
                                                  uint64_t* bfull, volatile int* abort_flag,
                                                  int pid, int lane) {
  using C = HaloCfg;
  const Sched sc = load_sched<false>(p);
  const unsigned long long timeout = p.timeout_ns;
  const int Wt = p.sub[0].Ws;
  const int per_img = p.sub[0].Hs * Wt;
  const int lower_h = p.sub[0].lower_h, lower_w = p.sub[0].lower_w;
  const uint32_t bytes = static_cast<uint32_t>(p.halo_bytes);
  const CUtensorMap* map = &p.mapA[0];
  bool b_issued = false;
  if (pid == 0 && unit_first(sc) < sc.units) {
    if (elect_one_sync()) {
      const SubProblem& sp = p.sub[0];
      const int nkb = sp.rcount * sp.scount;
      uint8_t* res = pipe + C::STAGE * C::STAGES;
      mbar_arrive_expect_tx(bfull, static_cast<uint32_t>(nkb * C::B_BYTES));
      for (int kb = 0; kb < nkb; ++kb) {
        const int jr = kb / sp.scount;
        const int js = kb - jr * sp.scount;
        const int r = sp.r0 + jr * sp.rstep;
        const int sc_ = sp.s0 + js * sp.sstep;
        // K-major (fprop) and MN-major (dgrad) filter maps both start the
        // single column tile and reduction block at coordinate 0
        tma_load_4d(res + kb * C::B_BYTES, &p.mapB, bfull, 0, sc_, r, 0);
      }
    }
    __syncwarp();
    b_issued = true;
  }
  uint8_t* stage = pipe + pid * C::STAGE;
  uint32_t phase = 0;
  bool issued = false;
  int k = 0;  // this CTA's unit count so far
  UnitWalk uw;
  for (walk_begin(p, sc, uw); uw.u < sc.units; walk_next(p, sc, uw), ++k) {
    if (k % C::NP != pid) continue;
    const Work w = walk_work(p, sc, uw);
    if (!__all_sync(0xffffffffu, mbar_wait(&empty[pid], phase ^ 1u, abort_flag, timeout))) {
      if (lane == 0) report_failure(p, abort_flag, DEVERR_PRODUCER_WAIT);
      break;
    }
    if (elect_one_sync()) {
      const int m0 = w.tile_m * kBlockM;
      const int n = m0 / per_img;
      const int row0 = (m0 - n * per_img) / Wt;
      mbar_arrive_expect_tx(&full[pid], bytes);
      tma_load_4d(stage, map, &full[pid], 0, lower_w, lower_h + row0, n);
    }
    __syncwarp();
    issued = true;
    phase ^= 1u;
  }
  // every copy this producer issued must land before the CTA exits
  if (issued && !mbar_wait(&full[pid], phase ^ 1u, nullptr, timeout) && lane == 0)
    report_failure(p, abort_flag, DEVERR_TEARDOWN_WAIT);
  if (b_issued && !mbar_wait(bfull, 0u, nullptr, timeout) && lane == 0)
    report_failure(p, abort_flag, DEVERR_TEARDOWN_WAIT);
}

// MMA issuer `issuer` (0 or 1) of a halo plan: for each unit, the blocks of
// its sequence parity, each four MMAs reading the halo at the block's tap
// offset and the block's resident filter rows; one commit per halo frees
// its share of the stage.
__device__ __forceinline__ void run_mma_halo(const ConvGemmParams& p, uint8_t* pipe,
                                             uint64_t* full, uint64_t* empty, uint64_t* tfull,
                                             uint64_t* tempty, uint64_t* done_bar,
                                             uint64_t* bfull, uint32_t tmem_base,
                                             volatile int* abort_flag, int issuer, int lane) {
  using C = HaloCfg;
  const Sched sc = load_sched<false>(p);
  const unsigned long long timeout = p.timeout_ns;
  const SubProblem& sp = p.sub[0];
  const int Wt = sp.Ws;
  const int scount = sp.scount;
  const int nk = sp.rcount * sp.scount;
  const int offh0 = sp.offh0, doffh = sp.doffh, offw0 = sp.offw0, doffw = sp.doffw;
  const bool b_mn = p.b_src == SRC_W_MN;
  const uint32_t idesc = p.idesc;
  const int num_acc = p.num_acc;
  const uint32_t pipe_addr = smem_u32(pipe);
  const uint64_t a0 = make_smem_desc(pipe_addr, 16, 1024);
  const uint64_t b0 = make_smem_desc(pipe_addr + C::STAGE * C::STAGES, b_mn ? 8192 : 16, 1024);
  const uint64_t ak = 32 / 16;
  const uint64_t bk = b_mn ? 2048 / 16 : 32 / 16;
  const int buf_shift = p.epi_groups == 2 ? 2 : 1;
  const int buf_mask = (1 << buf_shift) - 1;
  bool ok = true;
  if (unit_first(sc) < sc.units) {
    if (!__all_sync(0xffffffffu, mbar_wait(bfull, 0u, abort_flag, timeout))) {
      if (lane == 0) report_failure(p, abort_flag, DEVERR_MMA_FULL_WAIT);
      ok = false;
    }
    tc_fence_after_sync();
  }
  const bool one = p.one_issuer != 0;
  int st = 0;           // halo stage of the next unit
  uint32_t ph = 0;
  int qpar = 0;         // parity of the unit's first block in the CTA-wide sequence
  int local = 0;
  UnitWalk uw;
  for (walk_begin(p, sc, uw); ok && uw.u < sc.units; walk_next(p, sc, uw)) {
    if (one && (local & 1) != issuer) {
      // The other issuer's unit.  With three stages consecutive fills of a
      // stage belong to different issuers, so both take part in every
      // stage's release: this issuer waits for the fill and arrives on the
      // stage's empty barrier (count 2).  The producer cannot refill the stage
      // before both have seen the fill, so neither can fall two phases
      // behind (where its parity wait would take the phase after next).
      if (!__all_sync(0xffffffffu, mbar_wait(&full[st], ph, abort_flag, timeout))) {
        if (lane == 0) report_failure(p, abort_flag, DEVERR_MMA_FULL_WAIT);
        break;
      }
      if (lane == 0) mbar_arrive(&empty[st]);
      __syncwarp();
      if (++st == C::STAGES) {
        st = 0;
        ph ^= 1u;
      }
      ++local;
      continue;
    }
    const int buf = local & buf_mask;
    const uint32_t tph = static_cast<uint32_t>(local >> buf_shift) & 1u;
    if (!__all_sync(0xffffffffu, mbar_wait(&tempty[buf], tph ^ 1u, abort_flag, timeout))) {
      if (lane == 0) report_failure(p, abort_flag, DEVERR_MMA_TMEM_WAIT);
      break;
    }
    tc_fence_after_sync();
    if (!__all_sync(0xffffffffu, mbar_wait(&full[st], ph, abort_flag, timeout))) {
      if (lane == 0) report_failure(p, abort_flag, DEVERR_MMA_FULL_WAIT);
      break;
    }
    tc_fence_after_sync();
    const uint32_t d =
        tmem_base + static_cast<uint32_t>((buf * num_acc + (one ? 0 : issuer)) * 64);
    // The whole halo is in place, so one lane issues all of this issuer's
    // blocks back to back (every block of the unit with one issuer per unit,
    // else those of its sequence parity); the tap position (jr, js) advances
    // without a division.
    if (elect_one_sync()) {
      const int step = one ? 1 : 2;
      int rel = one ? 0 : issuer ^ qpar;
      int jr = 0, js = rel;
      while (js >= scount) {
        js -= scount;
        ++jr;
      }
      uint64_t ad_unit = a0 + (static_cast<uint32_t>(st * C::STAGE) >> 4);
      uint32_t acc = 0u;
      for (; rel < nk; rel += step) {
        const int row = (offh0 + jr * doffh) * Wt + offw0 + js * doffw;
        const uint64_t ad = ad_unit + ((static_cast<uint32_t>(row) * 128u) >> 4);
        const uint64_t bd = b0 + static_cast<uint64_t>(rel) * (C::B_BYTES / 16);
        mma_issue<false>(d, ad, bd, idesc, acc);
        mma_issue<false>(d, ad + ak, bd + bk, idesc, 1u);
        mma_issue<false>(d, ad + 2 * ak, bd + 2 * bk, idesc, 1u);
        mma_issue<false>(d, ad + 3 * ak, bd + 3 * bk, idesc, 1u);
        acc = 1u;
        js += step;
        while (js >= scount) {
          js -= scount;
          ++jr;
        }
      }
      mma_commit<false>(&empty[st]);   // this issuer's reads of the halo
      mma_commit<false>(&tfull[buf]);  // this issuer's accumulator
    }
    __syncwarp();
    qpar ^= nk & 1;
    if (++st == C::STAGES) {
      st = 0;
      ph ^= 1u;
    }
    ++local;
  }
  // Every MMA issued must complete before TMEM is released.
  if (elect_one_sync()) mma_commit<false>(done_bar);
  __syncwarp();
  if (!__all_sync(0xffffffffu, mbar_wait(done_bar, 0, nullptr, timeout)) && lane == 0)
    report_failure(p, abort_flag, DEVERR_TEARDOWN_WAIT);
}

// The halo kernel: the same roles and epilogue (16-bit stores) as
// conv_gemm_kernel<64, false, false, false, true>, with the halo producers
// and issuers above (a template, so that only the translation unit that
// launches it compiles it; BN is 64).
template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    conv_gemm_halo_kernel(const __grid_constant__ ConvGemmParams p) {
  static_assert(BN == 64, "halo plans use 64-wide tiles");
  using C = HaloCfg;
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  if (static_cast<int>(smem - smem_raw) + C::USED > C::SMEM) {
    pdl_wait();
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, static_cast<unsigned int>(DEVERR_SMEM_LAYOUT));
    return;
  }
  uint8_t* pipe = smem;
  uint8_t* stage_buf = smem + C::PIPE;
  uint32_t* bias_s = reinterpret_cast<uint32_t*>(smem + C::PIPE + C::EPI_STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::PIPE + C::EPI_STAGE + kBiasBytes);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 4;
  uint64_t* done_bar = tempty + 4;
  uint64_t* bfull = done_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nbuf = p.epi_groups == 2 ? 4 : 2;
  const uint32_t tmem_cols = tmem_cols_for(static_cast<uint32_t>(nbuf * p.num_acc * 64));

  if (threadIdx.x == 0) {
    // both issuers release every halo (one_issuer: the unit's issuer by its
    // commit, the other by an arrive after seeing the fill); each accumulator
    // has one issuer with one_issuer, else both
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NI);
    }
    const int epi_warps = p.epi_groups == 2 ? kEpiWarps / 2 : kEpiWarps;
    for (int b = 0; b < 4; ++b) {
      mbar_init(&tfull[b], p.one_issuer ? 1 : C::NI);
      mbar_init(&tempty[b], epi_warps);
    }
    mbar_init(&done_bar[0], 1);
    mbar_init(&done_bar[1], 1);
    mbar_init(bfull, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // the barriers above are this CTA's own: the stream's earlier kernel may
  // still run until here, not past it (the bias, the inputs, the outputs)
  pdl_wait();
  if (p.bias_cached) {
    for (int i = threadIdx.x; i < p.N_gemm; i += blockDim.x) {
      const uint16_t b = static_cast<const uint16_t*>(p.bias)[i];
      bias_s[i] = __float_as_uint(p.out_bf16 ? __bfloat162float(__ushort_as_bfloat16(b))
                                             : __half2float(__ushort_as_half(b)));
    }
  }
  if (warp == kMmaWarp0) tmem_alloc(tmem_slot, tmem_cols);
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
        if (p.use_tma_store) tma_prefetch_map(&p.mapY);
      }
      __syncwarp();
      run_producer_halo(p, pipe, full, empty, bfull, abort_flag, warp, lane);
    }
  } else if (warp >= kMmaWarp0) {
    setmaxnreg_dec<kRegsLow>();
    if (warp < kMmaWarp0 + C::NI)
      run_mma_halo(p, pipe, full, empty, tfull, tempty, &done_bar[warp - kMmaWarp0], bfull,
                   tmem_base, abort_flag, warp - kMmaWarp0, lane);
  } else {
    setmaxnreg_inc<kRegsEpi>();
    run_epilogue<BN, false, false, true>(p, tfull, tempty, tmem_base, abort_flag, warp, stage_buf,
                                         bias_s);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

// The register split assumes the kernel was compiled at exactly
// kLaunchRegs per thread (the pool the warpgroups divide); any other count
// is refused before launch instead of risking an inc that cannot complete.
static cudaError_t check_launch_regs(const void* kernel) {
  cudaFuncAttributes fa;
  const cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  return fa.numRegs == kLaunchRegs ? cudaSuccess : cudaErrorInvalidConfiguration;
}

template <int BN, bool PAIR, bool S16>
static cudaError_t launch_bn(const ConvGemmParams& p, int grid, cudaStream_t s) {
  const int smem = Cfg<BN, PAIR>::SMEM;
  if (!PAIR) {
    // 3D problems take the kernel with the volume paths compiled in (never
    // the 16-bit-store kernels, which are 2D only)
    const bool vol = p.a_src == SRC_IM2COL_K3 || p.wg_Do > 0;
    auto* k = conv_gemm_kernel<BN, false, false, false, S16>;
    if constexpr (!S16) {
      if (vol) k = conv_gemm_kernel<BN, false, true>;
    }
    if (BN == 64 && p.res_b && !vol) k = conv_gemm_kernel<64, false, false, true, S16>;
    cudaError_t e = check_launch_regs(reinterpret_cast<const void*>(k));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_hot(k, static_cast<unsigned>(grid), kThreads, static_cast<size_t>(smem), s, 1,
                      p);
  }
  auto* k = conv_gemm_kernel<BN, true, false, false, S16>;
  cudaError_t e = check_launch_regs(reinterpret_cast<const void*>(k));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (grid < 2 || (grid & 1)) return cudaErrorInvalidValue;
  return launch_hot(k, static_cast<unsigned>(grid), kThreads, static_cast<size_t>(smem), s, 2, p);
}

// Launches a plan on the kernel of tile width block_n (64, 128 or 256),
// with (S16) or without the epilogue reduced to 16-bit stores.
template <bool S16>
static cudaError_t launch_block_n(const ConvGemmParams& p, int block_n, int grid, cudaStream_t s) {
  switch (block_n) {
    case 64:
      return p.pair ? launch_bn<64, true, S16>(p, grid, s) : launch_bn<64, false, S16>(p, grid, s);
    case 128:
      return p.pair ? launch_bn<128, true, S16>(p, grid, s) : launch_bn<128, false, S16>(p, grid, s);
    case 256:
      return p.pair ? launch_bn<256, true, S16>(p, grid, s) : launch_bn<256, false, S16>(p, grid, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace igc
