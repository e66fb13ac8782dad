// aux_kernels.cu -- the bandwidth-bound kernels around the implicit GEMM:
//   * batched transpose for the NCHW <-> NHWC permutes
//   * the deterministic split-K reduction of wgrad (fp32, and int32 for int8)
//   * int8 -> fp16 widening of the int8 operands
//   * the per-device status word and the wait-timeout self-test
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "igconv_internal.h"
#include "ptx.cuh"

namespace igc {

// Device status word: set by a kernel whose pipeline wait ran out, read and
// cleared by igconv_get_device_status().
__device__ unsigned int g_igconv_status = 0;

cudaError_t status_word_address(unsigned int** ptr) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_igconv_status);
}

// ---------------------------------------------------------------------------
// Batched transpose: dst[b][j][i] = src[b][i][j], i < rows, j < cols.
//   nchw_to_nhwc: rows = C, cols = H*W;  nhwc_to_nchw: rows = H*W, cols = C.
// General form (any element size, extent or alignment): 64 x 64 element
// tiles staged in shared memory; 16-byte vector loads along j and 16-byte
// vector stores along i whenever row pitches allow.  The common case takes
// the register transpose further down.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) transpose_kernel(const T* __restrict__ src,
                                                        T* __restrict__ dst, long long rows,
                                                        long long cols, int vec_in,
                                                        int vec_out) {
  constexpr int TILE = 64;
  constexpr int V = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte vector
  constexpr int VPR = TILE / V;                          // vectors per tile row
  constexpr int PITCH = TILE + (sizeof(T) >= 4 ? 1 : 4 / static_cast<int>(sizeof(T)));
  __shared__ T tile[TILE][PITCH];

  const long long b = blockIdx.z;
  const long long i0 = static_cast<long long>(blockIdx.y) * TILE;
  const long long j0 = static_cast<long long>(blockIdx.x) * TILE;
  const T* s = src + b * rows * cols;
  T* d = dst + b * rows * cols;

  for (int e = threadIdx.x; e < TILE * VPR; e += blockDim.x) {
    const int ii = e / VPR;
    const int vj = e - ii * VPR;
    const long long i = i0 + ii;
    const long long j = j0 + static_cast<long long>(vj) * V;
    if (i >= rows) continue;
    if (vec_in && j + V <= cols) {
      union {
        uint4 u;
        T t[V];
      } v;
      v.u = *reinterpret_cast<const uint4*>(s + i * cols + j);
#pragma unroll
      for (int t = 0; t < V; ++t) tile[ii][vj * V + t] = v.t[t];
    } else {
      for (int t = 0; t < V; ++t)
        if (j + t < cols) tile[ii][vj * V + t] = s[i * cols + j + t];
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < TILE * VPR; e += blockDim.x) {
    const int jj = e / VPR;
    const int vi = e - jj * VPR;
    const long long j = j0 + jj;
    const long long i = i0 + static_cast<long long>(vi) * V;
    if (j >= cols) continue;
    if (vec_out && i + V <= rows) {
      union {
        uint4 u;
        T t[V];
      } v;
#pragma unroll
      for (int t = 0; t < V; ++t) v.t[t] = tile[vi * V + t][jj];
      *reinterpret_cast<uint4*>(d + j * rows + i) = v.u;
    } else {
      for (int t = 0; t < V; ++t)
        if (i + t < rows) d[j * rows + i + t] = tile[vi * V + t][jj];
    }
  }
}

// ---------------------------------------------------------------------------
// Register transpose for 2- and 4-byte elements when rows and cols are
// multiples of the vector width V = 16 / sizeof(T) and both tensors are
// 16-byte aligned.  Each thread moves one V x V block: V 16-byte loads (rows
// i .. i+V-1, columns j .. j+V-1), a transpose in registers, V 16-byte
// stores (rows j .. j+V-1 of dst, columns i .. i+V-1).  No shared memory and
// no barrier, so a thread keeps all V loads in flight at once.  The lanes of
// a warp form an 8 x 4 grid of blocks (8 along i, 4 along j): every load
// instruction reads eight runs of 4 * 16 = 64 contiguous bytes (two whole
// sectors), every store instruction writes four runs of 8 * 16 = 128 bytes
// (whole lines).  Measured on the 128 x 64 x 56 x 56 bf16 tensor, this
// layout runs at the speed of a plain copy kernel moving the same bytes
// (4.64 TB/s both); the 4 x 8 grid reached 4.38.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void transpose_block(uint4 (&r)[8], uint4 (&o)[8]) {
  // 8 x 8 block of 16-bit elements: r[k] holds row k, o[m] receives column m.
  // Step 1 swaps 16-bit halves between rows 2q and 2q+1, so that word p of
  // t[2q + e] holds rows (2q, 2q+1) of column 2p + e.  Step 2 is then a 4 x 4
  // transpose of 32-bit words for each e (register renaming only).
  uint32_t t[8][4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t a[4] = {r[2 * q].x, r[2 * q].y, r[2 * q].z, r[2 * q].w};
    const uint32_t b[4] = {r[2 * q + 1].x, r[2 * q + 1].y, r[2 * q + 1].z, r[2 * q + 1].w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      t[2 * q][p] = __byte_perm(a[p], b[p], 0x5410);      // low halves: column 2p
      t[2 * q + 1][p] = __byte_perm(a[p], b[p], 0x7632);  // high halves: column 2p + 1
    }
  }
#pragma unroll
  for (int p = 0; p < 4; ++p)
#pragma unroll
    for (int e = 0; e < 2; ++e)
      o[2 * p + e] = make_uint4(t[e][p], t[2 + e][p], t[4 + e][p], t[6 + e][p]);
}

__device__ __forceinline__ void transpose_block(uint4 (&r)[4], uint4 (&o)[4]) {
  // 4 x 4 block of 32-bit elements: word m of row k is element (k, m)
  o[0] = make_uint4(r[0].x, r[1].x, r[2].x, r[3].x);
  o[1] = make_uint4(r[0].y, r[1].y, r[2].y, r[3].y);
  o[2] = make_uint4(r[0].z, r[1].z, r[2].z, r[3].z);
  o[3] = make_uint4(r[0].w, r[1].w, r[2].w, r[3].w);
}

template <int V>
__global__ void __launch_bounds__(256) transpose_reg_kernel(const uint8_t* __restrict__ src,
                                                            uint8_t* __restrict__ dst,
                                                            long long batch, long long rows,
                                                            long long cols, long long tiles_i,
                                                            long long tiles_j) {
  constexpr int EB = 16 / V;  // element bytes
  constexpr int A = 8, B = 4;  // blocks per warp tile along i and j
  const long long warp_tile = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long per_batch = tiles_i * tiles_j;
  if (warp_tile >= batch * per_batch) return;
  const int lane = threadIdx.x & 31;
  const long long bidx = warp_tile / per_batch;
  const long long t = warp_tile - bidx * per_batch;
  const long long ti = t / tiles_j;
  const long long tj = t - ti * tiles_j;
  const long long i = (ti * A + (lane / B)) * V;
  const long long j = (tj * B + (lane % B)) * V;
  if (i >= rows || j >= cols) return;
  const uint8_t* s = src + (bidx * rows * cols + i * cols + j) * EB;
  uint8_t* d = dst + (bidx * rows * cols + j * rows + i) * EB;
  uint4 r[V], o[V];
#pragma unroll
  for (int k = 0; k < V; ++k)
    r[k] = __ldcs(reinterpret_cast<const uint4*>(s + static_cast<long long>(k) * cols * EB));
  transpose_block(r, o);
#pragma unroll
  for (int m = 0; m < V; ++m)
    __stcs(reinterpret_cast<uint4*>(d + static_cast<long long>(m) * rows * EB), o[m]);
}

cudaError_t launch_batched_transpose(const void* src, void* dst, long long batch, long long rows,
                                     long long cols, int elem_bytes, cudaStream_t s) {
  const uintptr_t sa0 = reinterpret_cast<uintptr_t>(src), da0 = reinterpret_cast<uintptr_t>(dst);
  if ((elem_bytes == 2 || elem_bytes == 4) && ((sa0 | da0) & 15) == 0) {
    const int V = 16 / elem_bytes;
    if (rows % V == 0 && cols % V == 0) {
      const long long tiles_i = (rows + 8 * V - 1) / (8 * V);
      const long long tiles_j = (cols + 4 * V - 1) / (4 * V);
      const long long warps = batch * tiles_i * tiles_j;
      const long long blocks = (warps + 7) / 8;
      if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
      if (V == 8)
        transpose_reg_kernel<8><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), batch, rows, cols,
            tiles_i, tiles_j);
      else
        transpose_reg_kernel<4><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), batch, rows, cols,
            tiles_i, tiles_j);
      return cudaGetLastError();
    }
  }
  const dim3 grid(static_cast<unsigned>((cols + 63) / 64), static_cast<unsigned>((rows + 63) / 64),
                  static_cast<unsigned>(batch));
  const uintptr_t sa = reinterpret_cast<uintptr_t>(src), da = reinterpret_cast<uintptr_t>(dst);
  const int vec_in = ((sa & 15) == 0) && ((cols * elem_bytes) % 16 == 0);
  const int vec_out = ((da & 15) == 0) && ((rows * elem_bytes) % 16 == 0);
  switch (elem_bytes) {
    case 1:
      transpose_kernel<uint8_t><<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(src),
                                                     static_cast<uint8_t*>(dst), rows, cols,
                                                     vec_in, vec_out);
      break;
    case 2:
      transpose_kernel<uint16_t><<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(src),
                                                      static_cast<uint16_t*>(dst), rows, cols,
                                                      vec_in, vec_out);
      break;
    case 4:
      transpose_kernel<uint32_t><<<grid, 256, 0, s>>>(static_cast<const uint32_t*>(src),
                                                      static_cast<uint32_t*>(dst), rows, cols,
                                                      vec_in, vec_out);
      break;
    case 8:
      transpose_kernel<unsigned long long><<<grid, 256, 0, s>>>(
          static_cast<const unsigned long long*>(src), static_cast<unsigned long long*>(dst), rows,
          cols, vec_in, vec_out);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// wgrad split-K reduction (the "separate reduction kernel" of parallel
// split-K in the CUTLASS Python example, section "Split-K"):
//   dW[k,r,s,c] = cast(alpha * sum_{split = 0..S-1} ws[split][...] + beta * Cin)
//
// A block owns a tile of 64/G workspace rows x 128 workspace columns.  Its
// eight warps form G split groups (G = 8, 4, 2 or 1 from the split count
// alone, at least two splits per group) x 8/G row warps: each lane holds 4
// consecutive columns (one 16-byte load per row and split) of 8 rows, and
// split group g adds splits g, g + G, ... in index order, two in flight.  The group sums meet in shared
// memory and are added in group order, so the result does not depend on
// scheduling.  The finished values go out with the output's contiguous
// dimension c along the lanes: as vectors of 4 consecutive c when the
// workspace columns are (tap, c), one element per lane when they are k.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float load_any(const void* p, long long i, int dtype) {
  if (dtype == 2) return static_cast<const float*>(p)[i];
  const uint16_t b = static_cast<const uint16_t*>(p)[i];
  return dtype == 1 ? __bfloat162float(__ushort_as_bfloat16(b)) : __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ void store_any(void* p, long long i, int dtype, float v) {
  if (dtype == 2) {
    static_cast<float*>(p)[i] = v;
  } else if (dtype == 1) {
    static_cast<uint16_t*>(p)[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  } else {
    static_cast<uint16_t*>(p)[i] = __half_as_ushort(__float2half_rn(v));
  }
}

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z),
                     __fadd_rn(a.w, b.w));
}

// Four consecutive dW elements starting at dst (dst % 4 == 0).
__device__ __forceinline__ void store4_any(void* p, long long dst, int dtype, float4 v) {
  if (dtype == 2) {
    *reinterpret_cast<float4*>(static_cast<float*>(p) + dst) = v;
  } else {
    uint32_t lo, hi;
    if (dtype == 1) {
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(v.y), "f"(v.x));
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(v.w), "f"(v.z));
    } else {
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(v.y), "f"(v.x));
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(v.w), "f"(v.z));
    }
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p) + dst) = make_uint2(lo, hi);
  }
}

// Target (tap, c) of workspace row / column mx: (mx / cpad, mx % cpad), or
// the few-channel virtual row decode when remap.cz != 0.
__device__ __forceinline__ bool row_target(int mx, int RS, int C, int cpad, const FewPack& remap,
                                           int* tap, int* c) {
  if (remap.cz != 0) return few_pack_decode(remap, mx >> 6, mx & 63, tap, c);
  *tap = mx / cpad;
  *c = mx - *tap * cpad;
  return *tap < RS && *c < C;
}

// Many splits (more than 8): the eight warps of a block are eight split
// groups over the same RPW rows x 64 columns (4-byte loads, lanes along the
// columns); group g adds splits g, g + 8, ... in index order, eight splits'
// loads in flight at a time (then four, then one), and the group sums are
// added in group order.  Eight in flight instead of four took the
// ResNet-50-shaped step from 0.5317 to 0.5308 ms (the 152-split 56x56
// layer has 19 splits per group).
// RPW (8, 4, 2 or 1) is chosen by the launcher so that the small outputs
// these plans have still spread over at least two blocks per SM: with 8 rows
// a 56x56 64->64 3x3 wgrad (576 x 64 outputs, 30 splits) had 72 blocks, ran
// latency-bound at 8 % of the memory throughput and took 7.3 us.
template <int RPW>
__global__ void __launch_bounds__(256) wgrad_reduce_many_kernel(
    const float* __restrict__ ws, int splits, long long split_stride, int ws_ld, int rows,
    int cols, int swapped, int K, int RS, int C, int cpad, void* dW, int dw_dtype,
    const void* cin, float alpha, float beta, FewPack remap) {
  constexpr int G = 8;      // split groups, one per warp
  constexpr int TR = RPW;   // workspace rows per tile
  __shared__ float part[G][TR][65];
  pdl_trigger();
  pdl_wait();  // the partials come from the kernel before this one
  const int g = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_c = (cols + 63) / 64;
  const int tiles = ((rows + TR - 1) / TR) * tiles_c;
  for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int r0 = (t / tiles_c) * TR;
    const int c0 = (t % tiles_c) * 64;
    float acc[RPW][2];
#pragma unroll
    for (int i = 0; i < RPW; ++i) acc[i][0] = acc[i][1] = 0.0f;
    bool rv[RPW], cv[2];
#pragma unroll
    for (int i = 0; i < RPW; ++i) rv[i] = r0 + i < rows;
    cv[0] = c0 + lane < cols;
    cv[1] = c0 + 32 + lane < cols;
    const float* src = ws + static_cast<long long>(r0) * ws_ld + c0 + lane;
    auto load = [&](int sp, float (&v)[RPW][2]) {
      const float* q = src + sp * split_stride;
#pragma unroll
      for (int i = 0; i < RPW; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          v[i][h] = (rv[i] && cv[h]) ? __ldg(q + static_cast<long long>(i) * ws_ld + 32 * h)
                                     : 0.0f;
    };
    auto add = [&](const float (&v)[RPW][2]) {
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        acc[i][0] = __fadd_rn(acc[i][0], v[i][0]);
        acc[i][1] = __fadd_rn(acc[i][1], v[i][1]);
      }
    };
    int sp = g;
    for (; sp + 7 * G < splits; sp += 8 * G) {
      float v[8][RPW][2];
#pragma unroll
      for (int j = 0; j < 8; ++j) load(sp + j * G, v[j]);
#pragma unroll
      for (int j = 0; j < 8; ++j) add(v[j]);
    }
    for (; sp + 3 * G < splits; sp += 4 * G) {
      float v0[RPW][2], v1[RPW][2], v2[RPW][2], v3[RPW][2];
      load(sp, v0);
      load(sp + G, v1);
      load(sp + 2 * G, v2);
      load(sp + 3 * G, v3);
      add(v0);
      add(v1);
      add(v2);
      add(v3);
    }
    for (; sp < splits; sp += G) {
      float v0[RPW][2];
      load(sp, v0);
      add(v0);
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      part[g][i][lane] = acc[i][0];
      part[g][i][lane + 32] = acc[i][1];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < TR * 64; idx += 256) {
      int rr, cc;
      if (swapped) {       // rows k, columns (tap, c): columns across the lanes
        rr = idx >> 6;
        cc = idx & 63;
      } else {             // rows (tap, c), columns k: rows across the lanes
        cc = idx / TR;
        rr = idx - cc * TR;
      }
      const int r = r0 + rr;
      const int col = c0 + cc;
      if (r >= rows || col >= cols) continue;
      float v = part[0][rr][cc];
#pragma unroll
      for (int j = 1; j < G; ++j) v = __fadd_rn(v, part[j][rr][cc]);
      const int k = swapped ? r : col;
      const int mx = swapped ? col : r;
      int tap, c;
      if (k >= K || !row_target(mx, RS, C, cpad, remap, &tap, &c)) continue;
      const long long dst = (static_cast<long long>(k) * RS + tap) * C + c;  // KRSC
      float o = __fmul_rn(alpha, v);
      if (beta != 0.0f) o = __fmaf_rn(beta, load_any(cin, dst, dw_dtype), o);
      store_any(dW, dst, dw_dtype, o);
    }
    __syncthreads();
  }
}

template <int G, bool SWAPPED>
__global__ void __launch_bounds__(256) wgrad_reduce_kernel(
    const float* __restrict__ ws, int splits, long long split_stride, int ws_ld, int rows,
    int cols, int K, int RS, int C, int cpad, void* dW, int dw_dtype, const void* cin,
    float alpha, float beta, FewPack remap) {
  constexpr int RW = 8 / G;   // row warps per split group
  constexpr int RPW = 8;      // rows per warp
  constexpr int TR = RPW * RW;  // workspace rows per tile
  __shared__ float part[G][TR][129];
  pdl_trigger();
  pdl_wait();  // the partials come from the kernel before this one
  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int lane = t & 31;
  const int g = warp % G;
  const int rw = warp / G;
  const int tiles_c = (cols + 127) / 128;
  const int tiles = ((rows + TR - 1) / TR) * tiles_c;
  for (int tt = blockIdx.x; tt < tiles; tt += gridDim.x) {
    const int r0 = (tt / tiles_c) * TR;
    const int c0 = (tt % tiles_c) * 128;
    // Split group g adds splits g, g + G, ... in index order over rows
    // r0 + 8 rw .. + 7, columns c0 + 4 lane .. + 3.  The workspace is
    // [splits][M_pad][ws_ld] with M_pad a multiple of 128, so every row of
    // the tile exists; columns exist below ws_ld (a multiple of 64).
    const int col = c0 + 4 * lane;
    const bool have = col < ws_ld;
    const float* base = ws + static_cast<long long>(r0 + RPW * rw) * ws_ld + col;
    float4 acc[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (have) {
      int sp = g;
      for (; sp + G < splits; sp += 2 * G) {  // two of the group's splits in flight
        const float* q0 = base + sp * split_stride;
        const float* q1 = q0 + G * split_stride;
        float4 v0[RPW], v1[RPW];
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
          v0[i] = __ldg(reinterpret_cast<const float4*>(q0 + static_cast<long long>(i) * ws_ld));
          v1[i] = __ldg(reinterpret_cast<const float4*>(q1 + static_cast<long long>(i) * ws_ld));
        }
#pragma unroll
        for (int i = 0; i < RPW; ++i) acc[i] = add4(add4(acc[i], v0[i]), v1[i]);
      }
      if (sp < splits) {
        const float* q0 = base + sp * split_stride;
#pragma unroll
        for (int i = 0; i < RPW; ++i)
          acc[i] = add4(acc[i], __ldg(reinterpret_cast<const float4*>(
                                    q0 + static_cast<long long>(i) * ws_ld)));
      }
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      float* d = &part[g][RPW * rw + i][4 * lane];
      d[0] = acc[i].x;
      d[1] = acc[i].y;
      d[2] = acc[i].z;
      d[3] = acc[i].w;
    }
    __syncthreads();
    if (SWAPPED && remap.cz != 0) {
      // rows k, few-channel virtual columns: each column decoded on its own
      const int q = lane;
      const int cc = c0 + 4 * q;
      for (int rr = warp; rr < TR; rr += 8) {
        const int k = r0 + rr;
        if (k >= rows || k >= K) break;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int tap, c;
          if (cc + j >= cols || !few_pack_decode(remap, (cc + j) >> 6, (cc + j) & 63, &tap, &c))
            continue;
          float a = part[0][rr][4 * q + j];
#pragma unroll
          for (int h = 1; h < G; ++h) a = __fadd_rn(a, part[h][rr][4 * q + j]);
          float o = __fmul_rn(alpha, a);
          const long long dst = (static_cast<long long>(k) * RS + tap) * C + c;
          if (beta != 0.0f) o = __fmaf_rn(beta, load_any(cin, dst, dw_dtype), o);
          store_any(dW, dst, dw_dtype, o);
        }
      }
    } else if (SWAPPED) {
      // rows k, columns (tap, c): lane q's 4 columns are 4 consecutive c
      const int q = lane;
      const int cc = c0 + 4 * q;
      const int tap = cc / cpad;
      const int c = cc - tap * cpad;
      if (cc < cols && tap < RS && c < C) {
        for (int rr = warp; rr < TR; rr += 8) {
          const int k = r0 + rr;
          if (k >= rows || k >= K) break;
          float v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float a = part[0][rr][4 * q + j];
#pragma unroll
            for (int h = 1; h < G; ++h) a = __fadd_rn(a, part[h][rr][4 * q + j]);
            v[j] = __fmul_rn(alpha, a);
          }
          const long long dst = (static_cast<long long>(k) * RS + tap) * C + c;
          if (c + 3 < C && (dst & 3) == 0) {
            if (beta != 0.0f) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                v[j] = __fmaf_rn(beta, load_any(cin, dst + j, dw_dtype), v[j]);
            }
            store4_any(dW, dst, dw_dtype, make_float4(v[0], v[1], v[2], v[3]));
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (c + j >= C) break;
              float o = v[j];
              if (beta != 0.0f) o = __fmaf_rn(beta, load_any(cin, dst + j, dw_dtype), o);
              store_any(dW, dst + j, dw_dtype, o);
            }
          }
        }
      }
    } else {
      // rows (tap, c), columns k: each thread keeps one row (one c) and walks
      // k, so lanes run along c for the writes
      constexpr int KPT = TR * 128 / 256;  // columns per thread
      const int rr = t % TR;
      const int kq = t / TR;
      const int r = r0 + rr;
      int tap = 0, c = 0;
      if (r < rows && row_target(r, RS, C, cpad, remap, &tap, &c)) {
        const long long kstride = static_cast<long long>(RS) * C;
        long long dst = (static_cast<long long>(c0 + kq * KPT) * RS + tap) * C + c;
        for (int j = 0; j < KPT; ++j, dst += kstride) {
          const int kk = kq * KPT + j;
          const int k = c0 + kk;
          if (k >= cols || k >= K) break;
          float a = part[0][rr][kk];
#pragma unroll
          for (int h = 1; h < G; ++h) a = __fadd_rn(a, part[h][rr][kk]);
          float o = __fmul_rn(alpha, a);
          if (beta != 0.0f) o = __fmaf_rn(beta, load_any(cin, dst, dw_dtype), o);
          store_any(dW, dst, dw_dtype, o);
        }
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_wgrad_reduce(const float* ws, int splits, long long split_stride, int ws_ld,
                                int rows, int cols, int swapped, int K, int RS, int C, int cpad,
                                void* dW, int dw_dtype, const void* cin, float alpha, float beta,
                                cudaStream_t s, const FewPack* remap_in) {
  FewPack remap{};
  if (remap_in) remap = *remap_in;  // remap.cz == 0: plain (tap, c) rows
  if (splits > 8) {
    // rows per tile: the most (of 8, 4, 2, 1) that still gives two blocks per SM
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long tiles_c = (cols + 63) / 64;
    int rpw = 8;
    while (rpw > 1 && ((rows + rpw - 1) / rpw) * tiles_c < 2LL * sms) rpw >>= 1;
    const long long tiles = ((rows + rpw - 1) / rpw) * tiles_c;
    const unsigned grid = static_cast<unsigned>(tiles < 16384 ? (tiles > 0 ? tiles : 1) : 16384);
#define IGC_REDUCE_MANY(R)                                                                     \
  launch_hot(wgrad_reduce_many_kernel<R>, grid, 256, 0, s, 1, ws, splits, split_stride, ws_ld, \
             rows, cols, swapped, K, RS, C, cpad, dW, dw_dtype, cin, alpha, beta, remap)
    switch (rpw) {
      case 8: return IGC_REDUCE_MANY(8);
      case 4: return IGC_REDUCE_MANY(4);
      case 2: return IGC_REDUCE_MANY(2);
      default: return IGC_REDUCE_MANY(1);
    }
#undef IGC_REDUCE_MANY
  }
  // every split group gets at least two splits, so two loads per row are in flight
  const int G = splits >= 8 ? 4 : (splits >= 4 ? 2 : 1);
  const int TR = 64 / G;
  const long long tiles = static_cast<long long>((rows + TR - 1) / TR) * ((cols + 127) / 128);
  const unsigned grid = static_cast<unsigned>(tiles < 16384 ? (tiles > 0 ? tiles : 1) : 16384);
#define IGC_REDUCE(GG)                                                                          \
  (swapped ? launch_hot(wgrad_reduce_kernel<GG, true>, grid, 256, 0, s, 1, ws, splits,          \
                        split_stride, ws_ld, rows, cols, K, RS, C, cpad, dW, dw_dtype, cin,     \
                        alpha, beta, remap)                                                     \
           : launch_hot(wgrad_reduce_kernel<GG, false>, grid, 256, 0, s, 1, ws, splits,         \
                        split_stride, ws_ld, rows, cols, K, RS, C, cpad, dW, dw_dtype, cin,     \
                        alpha, beta, remap))
  switch (G) {
    case 4: return IGC_REDUCE(4);
    case 2: return IGC_REDUCE(2);
    default: return IGC_REDUCE(1);
  }
#undef IGC_REDUCE
}

// ---------------------------------------------------------------------------
// Split-K convolution (fprop, stride-1 dgrad): out[m][n] = cast(relu?(alpha *
// sum_s ws[s][m][n] + beta * cin[m][n] + bias[n])), the splits added in split
// order (deterministic), then fprop's epilogue in the same order as the
// GEMM's own (alpha, beta * Cin, bias, ReLU, round to nearest even).  One
// thread per 8 consecutive columns (16 output bytes); cols % 8 == 0.
// ---------------------------------------------------------------------------
// 8 packed 16-bit values -> fp32, and a pair of fp32 -> packed 16 bits
// (round to nearest even, x in the low half).
__device__ __forceinline__ void unpack_row8(uint4 r, float (&f)[8], int bf16) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = w[i] & 0xFFFFu, hi = w[i] >> 16;
    if (bf16) {
      f[2 * i] = __uint_as_float(lo << 16);
      f[2 * i + 1] = __uint_as_float(hi << 16);
    } else {
      f[2 * i] = __half2float(__ushort_as_half(static_cast<unsigned short>(lo)));
      f[2 * i + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(hi)));
    }
  }
}

__device__ __forceinline__ uint32_t pack_pair16(float a, float b, int bf16) {
  if (bf16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(256) conv_splitk_reduce_kernel(
    const float* __restrict__ ws, int splits, long long split_stride, int ws_ld, long long rows,
    int cols, uint4* __restrict__ out, int out_bf16, const uint4* __restrict__ cin,
    const uint4* __restrict__ bias, float alpha, float beta, int relu) {
  const int c8 = cols / 8;
  const long long total = rows * c8;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long m = e / c8;
    const int n = static_cast<int>(e - m * c8) * 8;
    const float* src = ws + m * ws_ld + n;
    float v[8];
    {
      const float4 a = __ldcs(reinterpret_cast<const float4*>(src));
      const float4 b = __ldcs(reinterpret_cast<const float4*>(src + 4));
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    for (int sp = 1; sp < splits; ++sp) {
      const float* q = src + static_cast<long long>(sp) * split_stride;
      const float4 a = __ldcs(reinterpret_cast<const float4*>(q));
      const float4 b = __ldcs(reinterpret_cast<const float4*>(q + 4));
      v[0] = __fadd_rn(v[0], a.x); v[1] = __fadd_rn(v[1], a.y);
      v[2] = __fadd_rn(v[2], a.z); v[3] = __fadd_rn(v[3], a.w);
      v[4] = __fadd_rn(v[4], b.x); v[5] = __fadd_rn(v[5], b.y);
      v[6] = __fadd_rn(v[6], b.z); v[7] = __fadd_rn(v[7], b.w);
    }
    float cv[8] = {0, 0, 0, 0, 0, 0, 0, 0}, bv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (beta != 0.0f) {
      const uint4 r = cin[e];
      unpack_row8(r, cv, out_bf16);
    }
    if (bias) unpack_row8(bias[n / 8], bv, out_bf16);
    uint32_t pk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float x0 = __fmul_rn(alpha, v[2 * i]), x1 = __fmul_rn(alpha, v[2 * i + 1]);
      if (beta != 0.0f) {
        x0 = __fmaf_rn(beta, cv[2 * i], x0);
        x1 = __fmaf_rn(beta, cv[2 * i + 1], x1);
      }
      x0 = __fadd_rn(x0, bv[2 * i]);
      x1 = __fadd_rn(x1, bv[2 * i + 1]);
      if (relu) {
        x0 = fmaxf(x0, 0.0f);
        x1 = fmaxf(x1, 0.0f);
      }
      pk[i] = pack_pair16(x0, x1, out_bf16);
    }
    out[e] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

// int8 fprop split-K reduction: the splits' exact int32 partial sums of one
// output element added modulo 2^32 in split order (as one int32
// accumulator would), then the bias, ReLU and the exact half-even
// requantisation of the unsplit epilogue (requant_rne).  Four consecutive
// channels per thread.
__global__ void __launch_bounds__(256) conv_splitk_reduce_i8_kernel(
    const int* __restrict__ ws, int splits, long long split_stride, int ws_ld, long long rows,
    int cols, int8_t* __restrict__ out, const int32_t* __restrict__ bias, uint32_t mant, int sh,
    long long half_m1, int mode, int relu) {
  const int cq = cols / 4;
  const long long total = rows * cq;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long m = i / cq;
    const int c = static_cast<int>(i - m * cq) * 4;
    uint32_t a[4] = {0u, 0u, 0u, 0u};
    const int* src = ws + m * ws_ld + c;
    for (int sp = 0; sp < splits; ++sp) {
      const int4 v = *reinterpret_cast<const int4*>(src + sp * split_stride);
      a[0] += static_cast<uint32_t>(v.x);
      a[1] += static_cast<uint32_t>(v.y);
      a[2] += static_cast<uint32_t>(v.z);
      a[3] += static_cast<uint32_t>(v.w);
    }
    uint32_t packed = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      long long t = static_cast<long long>(static_cast<int>(a[j])) + (bias ? bias[c + j] : 0);
      if (relu && t < 0) t = 0;
      const int y = requant_rne(t, mant, sh, half_m1, mode);
      packed |= (static_cast<uint32_t>(y) & 0xFFu) << (8 * j);
    }
    *reinterpret_cast<uint32_t*>(out + m * cols + c) = packed;
  }
}

cudaError_t launch_conv_splitk_reduce_i8(const int* ws, int splits, long long split_stride,
                                         int ws_ld, long long rows, int cols, int8_t* out,
                                         const int32_t* bias, uint32_t rq_mant, int rq_exp,
                                         int relu, cudaStream_t s) {
  if (cols % 4 != 0 || ws_ld % 4 != 0 || split_stride % 4 != 0 || splits < 1)
    return cudaErrorInvalidValue;
  // M = mant * 2^rq_exp: the shift is -rq_exp, clamped as in the epilogue
  const int sh_true = -rq_exp;
  const int mode = sh_true < 1 ? 1 : (sh_true > 62 ? 2 : 0);
  const int sh = sh_true < 1 ? 1 : (sh_true > 62 ? 62 : sh_true);
  const long long half_m1 = (1LL << (sh - 1)) - 1;
  const long long total = rows * (cols / 4);
  long long blocks = (total + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 65536) blocks = 65536;
  conv_splitk_reduce_i8_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      ws, splits, split_stride, ws_ld, rows, cols, out, bias, rq_mant, sh, half_m1, mode, relu);
  return cudaGetLastError();
}

cudaError_t launch_conv_splitk_reduce(const float* ws, int splits, long long split_stride,
                                      int ws_ld, long long rows, int cols, void* out,
                                      int out_bf16, const void* cin, const void* bias,
                                      float alpha, float beta, int relu, cudaStream_t s) {
  const long long total = rows * (cols / 8);
  long long blocks = (total + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 65536) blocks = 65536;
  conv_splitk_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      ws, splits, split_stride, ws_ld, rows, cols, static_cast<uint4*>(out), out_bf16,
      static_cast<const uint4*>(cin), static_cast<const uint4*>(bias), alpha, beta, relu);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// int8 wgrad: dW[k][rs][c] (int32) = the sum of the int32 partial tiles of
// the splits, wrapping modulo 2^32 like the int32 accumulator they stand for
// (exact and order-independent).  One thread per element of the partial matrix, so the reads of
// every split run along its rows; rows past the valid extent are skipped.
//   not swapped: rows (tap, c) over rs * cpad, columns k
//   swapped:     rows k, columns (tap, c)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) wgrad_reduce_i32_kernel(
    const int* __restrict__ ws, int splits, long long split_stride, int ws_ld, int rows, int cols,
    int swapped, int K, int RS, int C, int cpad, int* __restrict__ dW) {
  const long long total = static_cast<long long>(rows) * cols;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(e / cols);
    const int n = static_cast<int>(e - static_cast<long long>(m) * cols);
    const int k = swapped ? m : n;
    const int x = swapped ? n : m;
    const int rs = x / cpad;
    const int c = x - rs * cpad;
    if (k >= K || rs >= RS || c >= C) continue;
    const int* src = ws + static_cast<long long>(m) * ws_ld + n;
    // eight independent loads in flight; integer addition modulo 2^32 is
    // associative, so the grouping changes no bit of the result
    uint32_t acc[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    int sp = 0;
    for (; sp + 8 <= splits; sp += 8) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        acc[i] += static_cast<uint32_t>(__ldcs(src + static_cast<long long>(sp + i) * split_stride));
    }
    for (; sp < splits; ++sp)
      acc[0] += static_cast<uint32_t>(__ldcs(src + static_cast<long long>(sp) * split_stride));
    uint32_t sum = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += acc[i];
    dW[(static_cast<long long>(k) * RS + rs) * C + c] = static_cast<int>(sum);
  }
}

cudaError_t launch_wgrad_reduce_i32(const int* ws, int splits, long long split_stride, int ws_ld,
                                    int rows, int cols, int swapped, int K, int RS, int C,
                                    int cpad, int* dW, cudaStream_t s) {
  const long long total = static_cast<long long>(rows) * cols;
  long long blocks = (total + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 16384) blocks = 16384;
  wgrad_reduce_i32_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      ws, splits, split_stride, ws_ld, rows, cols, swapped, K, RS, C, cpad, dW);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// int8 -> fp16 (exact: every int8 value is an fp16 integer)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) i8_to_f16_kernel(const int8_t* __restrict__ src,
                                                        __half* __restrict__ dst,
                                                        long long count) {
  const long long nvec = count / 16;
  for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec;
       v += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int4 in = reinterpret_cast<const int4*>(src)[v];
    const int w[4] = {in.x, in.y, in.z, in.w};
    uint4 out[2];
    uint32_t* o = reinterpret_cast<uint32_t*>(out);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int8_t a = static_cast<int8_t>((w[i] >> (16 * h)) & 0xFF);
        const int8_t b = static_cast<int8_t>((w[i] >> (16 * h + 8)) & 0xFF);
        const uint32_t lo = __half_as_ushort(__int2half_rn(a));
        const uint32_t hi = __half_as_ushort(__int2half_rn(b));
        o[2 * i + h] = lo | (hi << 16);
      }
    }
    reinterpret_cast<uint4*>(dst)[2 * v] = out[0];
    reinterpret_cast<uint4*>(dst)[2 * v + 1] = out[1];
  }
  // tail (count % 16 elements)
  const long long tail0 = nvec * 16;
  for (long long i = tail0 + static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < count; i += static_cast<long long>(gridDim.x) * blockDim.x)
    dst[i] = __int2half_rn(src[i]);
}

cudaError_t launch_i8_to_f16(const int8_t* src, void* dst, long long count, cudaStream_t s) {
  long long blocks = (count / 16 + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 8192) blocks = 8192;
  i8_to_f16_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(src, static_cast<__half*>(dst),
                                                                 count);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Few-channel operands (C <= 8): the tap-packed producer reads 16-byte pixels
// (8 channels) and the filter as [tap][k][8 channels], so that one reduction
// block holds 8 taps x 8 channels.
//   pad_pixels8:  [pixels][C] -> [pixels][8], channels C..7 zero
//   filter_taps8: W[K][R][S][C] -> the shared-memory image of every
//                 (reduction block, 64..256-wide column tile) pair:
//                 [block][tile_n][8 taps][bn][8 channels], zero past R*S
//                 taps, K output channels and C channels, so that a stage's
//                 filter part is one contiguous copy
// Both are element-wise copies (16-bit elements), one output vector of 8
// channels per thread.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) pad_pixels8_kernel(const uint16_t* __restrict__ src,
                                                          uint4* __restrict__ dst,
                                                          long long pixels, int C) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < pixels;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    uint16_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const uint16_t* p = src + i * C;
    for (int c = 0; c < C; ++c) v[c] = p[c];
    dst[i] = make_uint4(v[0] | (static_cast<uint32_t>(v[1]) << 16),
                        v[2] | (static_cast<uint32_t>(v[3]) << 16),
                        v[4] | (static_cast<uint32_t>(v[5]) << 16),
                        v[6] | (static_cast<uint32_t>(v[7]) << 16));
  }
}

__global__ void __launch_bounds__(256) filter_taps8_kernel(const uint16_t* __restrict__ w,
                                                           uint4* __restrict__ dst, int K, int RS,
                                                           int C, int bn, int tiles_n,
                                                           long long total) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    // i = ((block * tiles_n + tile_n) * 8 + t) * bn + n
    const int n = static_cast<int>(i % bn);
    long long rest = i / bn;
    const int t = static_cast<int>(rest % 8);
    rest /= 8;
    const int tile_n = static_cast<int>(rest % tiles_n);
    const int block = static_cast<int>(rest / tiles_n);
    const int tap = block * 8 + t;
    const int k = tile_n * bn + n;
    uint16_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (tap < RS && k < K) {
      const uint16_t* p = w + (static_cast<long long>(k) * RS + tap) * C;
      for (int c = 0; c < C; ++c) v[c] = p[c];
    }
    dst[i] = make_uint4(v[0] | (static_cast<uint32_t>(v[1]) << 16),
                        v[2] | (static_cast<uint32_t>(v[3]) << 16),
                        v[4] | (static_cast<uint32_t>(v[5]) << 16),
                        v[6] | (static_cast<uint32_t>(v[7]) << 16));
  }
}

// Few-channel dgrad, last step: dst[p][c] = cast(fma(beta, cin[p][c],
// src8[p][c])) for c < C, from fp32 rows of 8 channels (alpha already
// applied); the same operations, in the same order, as the GEMM epilogue.
__global__ void __launch_bounds__(256) unpad_channels_kernel(const float4* __restrict__ src8,
                                                             uint16_t* __restrict__ dst,
                                                             long long pixels, int C,
                                                             int out_bf16,
                                                             const uint16_t* __restrict__ cin,
                                                             float beta) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < pixels;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 a = src8[2 * i], b = src8[2 * i + 1];
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    for (int c = 0; c < C; ++c) {
      float x = v[c];
      if (beta != 0.0f) {
        const uint16_t u = cin[i * C + c];
        const float cv = out_bf16 ? __uint_as_float(static_cast<uint32_t>(u) << 16)
                                  : __half2float(__ushort_as_half(u));
        x = __fmaf_rn(beta, cv, x);
      }
      dst[i * C + c] = out_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x))
                                : __half_as_ushort(__float2half_rn(x));
    }
  }
}

cudaError_t launch_unpad_channels(const float* src8, void* dst, long long pixels, int C,
                                  int out_bf16, const void* cin, float beta, cudaStream_t s) {
  if (C < 1 || C > 8) return cudaErrorInvalidValue;
  long long blocks = (pixels + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 16384) blocks = 16384;
  unpad_channels_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      reinterpret_cast<const float4*>(src8), static_cast<uint16_t*>(dst), pixels, C, out_bf16,
      static_cast<const uint16_t*>(cin), beta);
  return cudaGetLastError();
}

cudaError_t launch_pad_pixels8(const void* src, void* dst, long long pixels, int C,
                               cudaStream_t s) {
  if (C < 1 || C > 8) return cudaErrorInvalidValue;
  long long blocks = (pixels + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 16384) blocks = 16384;
  pad_pixels8_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      static_cast<const uint16_t*>(src), static_cast<uint4*>(dst), pixels, C);
  return cudaGetLastError();
}

cudaError_t launch_filter_taps8(const void* w, void* dst, int K, int RS, int C, int bn,
                                cudaStream_t s) {
  if (C < 1 || C > 8 || bn < 8) return cudaErrorInvalidValue;
  const int tiles_n = (K + bn - 1) / bn;
  const long long total = static_cast<long long>((RS + 7) / 8) * tiles_n * 8 * bn;
  long long blocks = (total + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 16384) blocks = 16384;
  filter_taps8_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      static_cast<const uint16_t*>(w), static_cast<uint4*>(dst), K, RS, C, bn, tiles_n, total);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Few-channel packing (FewPack in igconv_internal.h), 16-bit element copies,
// one 8-element (16-byte) output vector per thread:
//   few_pack_x:      X[N][H][W][C] -> Zp[N][Hz][Wz][cz] (space-to-depth by the
//                    strides, zero padding stored)
//   few_pack_filter: W[K][R][S][C] -> Wpk[K][R2 * Sv][row], each virtual
//                    channel the filter entry few_pack_decode names, or zero
//                    (row = 64 for the windowed fprop; cz for the unwindowed
//                    dgrad problem)
//   few_unpack_dx:   the inverse gather for dgrad: each X element's gradient
//                    is the one packed element it was copied to
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 pack8_u16(const uint16_t v[8]) {
  return make_uint4(v[0] | (static_cast<uint32_t>(v[1]) << 16),
                    v[2] | (static_cast<uint32_t>(v[3]) << 16),
                    v[4] | (static_cast<uint32_t>(v[5]) << 16),
                    v[6] | (static_cast<uint32_t>(v[7]) << 16));
}

__global__ void __launch_bounds__(256) few_pack_x_kernel(const uint16_t* __restrict__ X,
                                                         uint4* __restrict__ Zp, FewPack f, int H,
                                                         int W, long long total) {
  const int vpp = f.cz / 8;  // output vectors per packed pixel
  const int fwc = f.fw * f.C;
  const int used = f.fh * fwc;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    // i = ((n * Hz + zi) * Wz + zj) * vpp + v
    const int v = static_cast<int>(i % vpp);
    long long rest = i / vpp;
    const int zj = static_cast<int>(rest % f.Wz);
    rest /= f.Wz;
    const int zi = static_cast<int>(rest % f.Hz);
    const long long n = rest / f.Hz;
    uint16_t o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int e = v * 8 + t;
      if (e >= used) break;
      const int dy = e / fwc;
      const int rem = e - dy * fwc;
      const int dx = rem / f.C;
      const int c = rem - dx * f.C;
      const int h = f.fh * (zi + f.A0) + dy;
      const int w = f.fw * (zj + f.B0) + dx;
      if (h >= 0 && h < H && w >= 0 && w < W)
        o[t] = X[((n * H + h) * W + w) * f.C + c];
    }
    Zp[i] = pack8_u16(o);
  }
}

__global__ void __launch_bounds__(256) few_pack_filter_kernel(const uint16_t* __restrict__ Wt,
                                                              uint4* __restrict__ Wpk, FewPack f,
                                                              int row, long long total) {
  const int vts = f.R2 * f.Sv;
  const int vpr = row / 8;  // output vectors per virtual tap
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    // i = (k * vts + vt) * vpr + v
    const int v = static_cast<int>(i % vpr);
    const long long rest = i / vpr;
    const int vt = static_cast<int>(rest % vts);
    const long long k = rest / vts;
    uint16_t o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      int tap, c;
      if (few_pack_decode(f, vt, v * 8 + t, &tap, &c))
        o[t] = Wt[(k * f.R * f.S + tap) * f.C + c];
    }
    Wpk[i] = pack8_u16(o);
  }
}

// dX[n][h][w][c] = cast(dz[n][zi][zj][e] + beta * Cin[n][h][w][c]) with
// (zi, zj, e) the packed position X[n][h][w][c] was copied to: zi = h / fh -
// A0, zj = w / fw - B0, e = ((h % fh) * fw + w % fw) * C + c; dz holds alpha
// times the gradient of the packed image as fp32 [N][Hz][Wz][cz] (ppr = 1);
// X elements outside the packed image's extent get 0 + beta * Cin.
__global__ void __launch_bounds__(256) few_unpack_dx_kernel(const float* __restrict__ dz,
                                                            uint16_t* __restrict__ dX, FewPack f,
                                                            int H, int W, long long total,
                                                            int out_bf16,
                                                            const uint16_t* __restrict__ cin,
                                                            float beta) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    // i = ((n * H + h) * W + w) * C + c
    const int c = static_cast<int>(i % f.C);
    long long rest = i / f.C;
    const int w = static_cast<int>(rest % W);
    rest /= W;
    const int h = static_cast<int>(rest % H);
    const long long n = rest / H;
    const int zi = h / f.fh - f.A0, dy = h % f.fh;
    const int zj = w / f.fw - f.B0, dx = w % f.fw;
    const int e = (dy * f.fw + dx) * f.C + c;
    // rows and columns past the packed image are read by no output (stride
    // above the filter extent): their gradient is zero
    float x = (zi < f.Hz && zj < f.Wz) ? dz[((n * f.Hz + zi) * f.Wz + zj) * f.cz + e] : 0.0f;
    if (beta != 0.0f) {
      const uint16_t u = cin[i];
      const float cv = out_bf16 ? __uint_as_float(static_cast<uint32_t>(u) << 16)
                                : __half2float(__ushort_as_half(u));
      x = __fmaf_rn(beta, cv, x);
    }
    dX[i] = out_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x))
                     : __half_as_ushort(__float2half_rn(x));
  }
}

cudaError_t launch_few_pack_x(const void* X, void* Zp, const FewPack& f, int N, int H, int W,
                              cudaStream_t s) {
  if (f.cz < 8 || f.cz > 64 || f.C < 1 || f.C > 8) return cudaErrorInvalidValue;
  const long long total = static_cast<long long>(N) * f.Hz * f.Wz * (f.cz / 8);
  long long blocks = (total + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 65536) blocks = 65536;
  few_pack_x_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      static_cast<const uint16_t*>(X), static_cast<uint4*>(Zp), f, H, W, total);
  return cudaGetLastError();
}

cudaError_t launch_few_pack_filter(const void* Wt, void* Wpk, const FewPack& f, int K, int row,
                                   cudaStream_t s) {
  if (f.cz < 8 || f.cz > 64 || f.C < 1 || f.C > 8 || row % 8 != 0 || row < 8 || row > 64)
    return cudaErrorInvalidValue;
  const long long total = static_cast<long long>(K) * f.R2 * f.Sv * (row / 8);
  long long blocks = (total + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 16384) blocks = 16384;
  few_pack_filter_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      static_cast<const uint16_t*>(Wt), static_cast<uint4*>(Wpk), f, row, total);
  return cudaGetLastError();
}

cudaError_t launch_few_unpack_dx(const float* dz, void* dX, const FewPack& f, int N, int H, int W,
                                 int out_bf16, const void* cin, float beta, cudaStream_t s) {
  if (f.C < 1 || f.C > 8 || f.fh < 1 || f.fw < 1) return cudaErrorInvalidValue;
  const long long total = static_cast<long long>(N) * H * W * f.C;
  long long blocks = (total + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 65536) blocks = 65536;
  few_unpack_dx_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      dz, static_cast<uint16_t*>(dX), f, H, W, total, out_bf16,
      static_cast<const uint16_t*>(cin), beta);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Self-test of the device-side failure path: one thread waits on a barrier
// that nothing completes; the bounded wait gives up and records the code.
// ---------------------------------------------------------------------------
__global__ void selftest_wait_kernel(unsigned int* status, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(&bar, 0u, nullptr, timeout_ns)) atomicCAS(status, 0u, DEVERR_SELFTEST);
  }
}

// Dense block-diagonal filter of a grouped convolution (groups of cg input
// and kg output channels), for the implicit GEMMs over group windows:
// dst[k][tap][c] = w[k][tap][c - g * cg] when c lies in k's group
// g = k / kg, else 0.
__global__ void __launch_bounds__(256) group_filter_dense_kernel(const uint16_t* __restrict__ w,
                                                                 uint16_t* __restrict__ dst,
                                                                 int K, int RS, int C, int cg,
                                                                 int kg) {
  const long long total = static_cast<long long>(K) * RS * C;
  for (long long e = blockIdx.x * 256ll + threadIdx.x; e < total; e += 256ll * gridDim.x) {
    const long long kt = e / C;
    const int c = static_cast<int>(e - kt * C);
    const int k = static_cast<int>(kt / RS);
    const int jj = c - (k / kg) * cg;
    dst[e] = (jj >= 0 && jj < cg) ? w[kt * cg + jj] : 0;
  }
}

// Weight gradient of a grouped convolution from the gradient of the windowed
// filter: src [K][RS][cpad] (fp32, alpha applied) holds, for output channel
// k of 64-wide tile n = k / 64, the gradient against the X channels of n's
// window, which starts at (n / div) * mul; k's own cg channels start at
// g * cg with g = k / kg.  dW[k][tap][j] = cast(src[k][tap][g * cg -
// start + j] + beta * Cin[k][tap][j]), j < cg.
__global__ void __launch_bounds__(256) group_extract_kernel(const float* __restrict__ src,
                                                            void* dW, int dw_dtype,
                                                            const void* cin, float beta, int K,
                                                            int RS, int cg, int kg, int cpad,
                                                            int mul, int div) {
  const long long total = static_cast<long long>(K) * RS * cg;
  for (long long e = blockIdx.x * 256ll + threadIdx.x; e < total; e += 256ll * gridDim.x) {
    const int j = static_cast<int>(e % cg);
    const long long kt = e / cg;
    const int k = static_cast<int>(kt / RS);
    const int off = (k / kg) * cg - ((k >> 6) / div) * mul;
    float v = src[kt * cpad + off + j];
    if (beta != 0.0f) {
      const float ci = dw_dtype == 2   ? static_cast<const float*>(cin)[e]
                       : dw_dtype == 1 ? __bfloat162float(static_cast<const __nv_bfloat16*>(cin)[e])
                                       : __half2float(static_cast<const __half*>(cin)[e]);
      v += beta * ci;
    }
    if (dw_dtype == 2)
      static_cast<float*>(dW)[e] = v;
    else if (dw_dtype == 1)
      static_cast<__nv_bfloat16*>(dW)[e] = __float2bfloat16_rn(v);
    else
      static_cast<__half*>(dW)[e] = __float2half_rn(v);
  }
}

cudaError_t launch_group_extract(const float* src, void* dW, int dw_dtype, const void* cin,
                                 float beta, int K, int RS, int cg, int kg, int cpad, int mul,
                                 int div, cudaStream_t s) {
  if (cg < 1 || kg < 1 || div < 1) return cudaErrorInvalidValue;
  const long long total = static_cast<long long>(K) * RS * cg;
  const long long blocks = (total + 255) / 256;
  const int grid = static_cast<int>(blocks < 8192 ? blocks : 8192);
  group_extract_kernel<<<grid, 256, 0, s>>>(src, dW, dw_dtype, cin, beta, K, RS, cg, kg, cpad,
                                            mul, div);
  return cudaGetLastError();
}

cudaError_t launch_group_filter_dense(const void* w, void* dst, int K, int RS, int C, int cg,
                                      int kg, cudaStream_t s) {
  if (cg < 1 || kg < 1) return cudaErrorInvalidValue;
  const long long total = static_cast<long long>(K) * RS * C;
  const long long blocks = (total + 255) / 256;
  const int grid = static_cast<int>(blocks < 8192 ? blocks : 8192);
  group_filter_dense_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(w),
                                                 static_cast<uint16_t*>(dst), K, RS, C, cg, kg);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(unsigned int* status, unsigned long long timeout_ns,
                                 cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace igc
