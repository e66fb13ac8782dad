// winograd.cu -- the transforms of the Winograd F(2x2, 3x3) forward pass
// (3x3 filters, stride 1, dilation 1), named as future work for 3x3 stride-1
// layers in tensorcore "docs/conv2d.md", "What's not done in v0.1".
//
// Over 4x4 input patches d taken with stride 2 (output tiles of 2x2), and
// the 3x3 filter g of each (k, c), the pass computes
//   V = Bt d B,  U = G g Gt,  M[xi] = sum_c V[xi][c] * U[xi][c],  Y = At M A
// with
//   Bt = [1 0 -1 0; 0 1 1 0; 0 -1 1 0; 0 1 0 -1]
//   G  = [1 0 0; 1/2 1/2 1/2; 1/2 -1/2 1/2; 0 0 1]
//   At = [1 1 1 0; 0 1 -1 -1]
// which gives Y[p][q] = sum_{r,s} d[p+r][q+s] g[r][s] exactly in real
// arithmetic (the correlation that fprop computes).  The 16 products M[xi]
// are 16 independent GEMMs [T x C] x [C x K] (T = output tiles), which run on
// the implicit-GEMM kernel; these kernels are the CUDA-core transforms
// around them:
//   input  X [N][H][W][C]        -> V [16][T][C]   (fp32 arithmetic, rounded
//                                                   to the 16-bit I/O type)
//   filter Wt [K][3][3][C]       -> U [K][16][C]   (the same)
//   output M [16][T][K] (16-bit) -> Y [N][P][Q][K] with alpha, beta * Cin,
//                                   bias, ReLU and the cast, as fprop's
//                                   epilogue
// Each thread takes one pair of adjacent channels (one 32-bit word), so the
// lanes of a warp read and write runs of consecutive words: a 64-channel
// pixel row is one 128-byte run.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "igconv_internal.h"

namespace igc {

namespace {

__device__ __forceinline__ float2 unpack2(uint32_t w, int bf16) {
  if (bf16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
  const __half2 h = *reinterpret_cast<const __half2*>(&w);
  return __half22float2(h);
}

__device__ __forceinline__ uint32_t pack2(float a, float b, int bf16) {
  if (bf16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// V = Bt d B of one 4x4 patch, in place (row-major d[4 * r + s]).
__device__ __forceinline__ void input_transform(float (&d)[16]) {
  float t[16];
#pragma unroll
  for (int s = 0; s < 4; ++s) {  // rows: Bt d
    t[0 + s] = d[0 + s] - d[8 + s];
    t[4 + s] = d[4 + s] + d[8 + s];
    t[8 + s] = d[8 + s] - d[4 + s];
    t[12 + s] = d[4 + s] - d[12 + s];
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // columns: (Bt d) B
    d[4 * i + 0] = t[4 * i + 0] - t[4 * i + 2];
    d[4 * i + 1] = t[4 * i + 1] + t[4 * i + 2];
    d[4 * i + 2] = t[4 * i + 2] - t[4 * i + 1];
    d[4 * i + 3] = t[4 * i + 1] - t[4 * i + 3];
  }
}

}  // namespace

// X [N][H][W][C] -> V [16][T][C]; thread = (tile t, channel pair).
__global__ void __launch_bounds__(256) wino_input_kernel(const uint32_t* __restrict__ X,
                                                         uint32_t* __restrict__ V, int N, int H,
                                                         int W, int C2, int TH, int TW, int ph,
                                                         int pw, int bf16) {
  const long long T = static_cast<long long>(N) * TH * TW;
  const long long total = T * C2;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c2 = static_cast<int>(e % C2);
    const long long t = e / C2;
    const int tj = static_cast<int>(t % TW);
    const long long r = t / TW;
    const int ti = static_cast<int>(r % TH);
    const int n = static_cast<int>(r / TH);
    const int h0 = 2 * ti - ph, w0 = 2 * tj - pw;
    float dx[16], dy[16];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int h = h0 + a, w = w0 + b;
        float2 v = make_float2(0.0f, 0.0f);
        if (h >= 0 && h < H && w >= 0 && w < W)
          v = unpack2(X[((static_cast<long long>(n) * H + h) * W + w) * C2 + c2], bf16);
        dx[4 * a + b] = v.x;
        dy[4 * a + b] = v.y;
      }
    }
    input_transform(dx);
    input_transform(dy);
#pragma unroll
    for (int xi = 0; xi < 16; ++xi)
      V[(static_cast<long long>(xi) * T + t) * C2 + c2] = pack2(dx[xi], dy[xi], bf16);
  }
}

// Wt [K][3][3][C] -> U [K][16][C]; thread = (k, channel pair).
__global__ void __launch_bounds__(256) wino_filter_kernel(const uint32_t* __restrict__ Wt,
                                                          uint32_t* __restrict__ U, int K, int C2,
                                                          int bf16) {
  const long long total = static_cast<long long>(K) * C2;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c2 = static_cast<int>(e % C2);
    const long long k = e / C2;
    float g[2][9];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const float2 v = unpack2(Wt[(k * 9 + i) * C2 + c2], bf16);
      g[0][i] = v.x;
      g[1][i] = v.y;
    }
    float u[2][16];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      float t[12];  // G g: 4 rows x 3 columns
#pragma unroll
      for (int s = 0; s < 3; ++s) {
        const float g0 = g[ch][s], g1 = g[ch][3 + s], g2 = g[ch][6 + s];
        t[0 + s] = g0;
        t[3 + s] = 0.5f * (g0 + g1 + g2);
        t[6 + s] = 0.5f * (g0 - g1 + g2);
        t[9 + s] = g2;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // (G g) Gt
        const float a0 = t[3 * i], a1 = t[3 * i + 1], a2 = t[3 * i + 2];
        u[ch][4 * i + 0] = a0;
        u[ch][4 * i + 1] = 0.5f * (a0 + a1 + a2);
        u[ch][4 * i + 2] = 0.5f * (a0 - a1 + a2);
        u[ch][4 * i + 3] = a2;
      }
    }
#pragma unroll
    for (int xi = 0; xi < 16; ++xi)
      U[(k * 16 + xi) * C2 + c2] = pack2(u[0][xi], u[1][xi], bf16);
  }
}

// M [16][T][K] -> Y [N][P][Q][K] = cast(relu?(alpha * (At M A) + beta * Cin +
// bias)); thread = (tile t, output-channel pair).
__global__ void __launch_bounds__(256) wino_output_kernel(
    const uint32_t* __restrict__ Mx, uint32_t* __restrict__ Y, const uint32_t* __restrict__ cin,
    const uint32_t* __restrict__ bias, int N, int P, int Q, int K2, int TH, int TW, float alpha,
    float beta, int relu, int bf16) {
  const long long T = static_cast<long long>(N) * TH * TW;
  const long long total = T * K2;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int k2 = static_cast<int>(e % K2);
    const long long t = e / K2;
    const int tj = static_cast<int>(t % TW);
    const long long r = t / TW;
    const int ti = static_cast<int>(r % TH);
    const int n = static_cast<int>(r / TH);
    float m[2][16];
#pragma unroll
    for (int xi = 0; xi < 16; ++xi) {
      const float2 v = unpack2(Mx[(static_cast<long long>(xi) * T + t) * K2 + k2], bf16);
      m[0][xi] = v.x;
      m[1][xi] = v.y;
    }
    float y[2][4];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      float a[2][4];  // At M: 2 rows x 4 columns
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        a[0][j] = m[ch][j] + m[ch][4 + j] + m[ch][8 + j];
        a[1][j] = m[ch][4 + j] - m[ch][8 + j] - m[ch][12 + j];
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {  // (At M) A
        y[ch][2 * i + 0] = a[i][0] + a[i][1] + a[i][2];
        y[ch][2 * i + 1] = a[i][1] - a[i][2] - a[i][3];
      }
    }
    float2 b = make_float2(0.0f, 0.0f);
    if (bias) b = unpack2(bias[k2], bf16);
#pragma unroll
    for (int pa = 0; pa < 2; ++pa) {
#pragma unroll
      for (int pb = 0; pb < 2; ++pb) {
        const int p = 2 * ti + pa, q = 2 * tj + pb;
        if (p >= P || q >= Q) continue;
        const long long o = ((static_cast<long long>(n) * P + p) * Q + q) * K2 + k2;
        float v0 = alpha * y[0][2 * pa + pb], v1 = alpha * y[1][2 * pa + pb];
        if (beta != 0.0f) {
          const float2 c = unpack2(cin[o], bf16);
          v0 = fmaf(beta, c.x, v0);
          v1 = fmaf(beta, c.y, v1);
        }
        v0 += b.x;
        v1 += b.y;
        if (relu) {
          v0 = fmaxf(v0, 0.0f);
          v1 = fmaxf(v1, 0.0f);
        }
        Y[o] = pack2(v0, v1, bf16);
      }
    }
  }
}

namespace {
unsigned grid_of(long long total) {
  long long blocks = (total + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 65536) blocks = 65536;
  return static_cast<unsigned>(blocks);
}
}  // namespace

cudaError_t launch_wino_input(const void* X, void* V, int N, int H, int W, int C, int TH, int TW,
                              int ph, int pw, int bf16, cudaStream_t s) {
  const long long total = static_cast<long long>(N) * TH * TW * (C / 2);
  wino_input_kernel<<<grid_of(total), 256, 0, s>>>(static_cast<const uint32_t*>(X),
                                                   static_cast<uint32_t*>(V), N, H, W, C / 2, TH,
                                                   TW, ph, pw, bf16);
  return cudaGetLastError();
}

cudaError_t launch_wino_filter(const void* Wt, void* U, int K, int C, int bf16, cudaStream_t s) {
  const long long total = static_cast<long long>(K) * (C / 2);
  wino_filter_kernel<<<grid_of(total), 256, 0, s>>>(static_cast<const uint32_t*>(Wt),
                                                    static_cast<uint32_t*>(U), K, C / 2, bf16);
  return cudaGetLastError();
}

cudaError_t launch_wino_output(const void* Mx, void* Y, const void* cin, const void* bias, int N,
                               int P, int Q, int K, int TH, int TW, float alpha, float beta,
                               int relu, int bf16, cudaStream_t s) {
  const long long total = static_cast<long long>(N) * TH * TW * (K / 2);
  wino_output_kernel<<<grid_of(total), 256, 0, s>>>(
      static_cast<const uint32_t*>(Mx), static_cast<uint32_t*>(Y),
      static_cast<const uint32_t*>(cin), static_cast<const uint32_t*>(bias), N, P, Q, K / 2, TH,
      TW, alpha, beta, relu, bf16);
  return cudaGetLastError();
}

}  // namespace igc
