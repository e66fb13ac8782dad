/*
 * igconv.h -- C ABI of libigconv: 2D convolution as an implicit GEMM on
 * GB300 (sm_103a), in all three passes, plus an int8 forward pass with
 * requantisation and the NCHW <-> NHWC permutes.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are dense, row-major, innermost dimension last:
 *      X, dX   [N][H][W][C]   activations, NHWC
 *      Wt, dW  [K][R][S][C]   filters, KRSC
 *      Y, dY   [N][P][Q][K]   outputs / output gradients, NHWC
 *    (the channel-last layout of the CUTLASS Python example
 *    "03_basic_conv2d.ipynb", section "General setup", and of the NHWC core
 *    that burn-cubecl "kernel/conv/base.rs" permutes into, `conv_forward`).
 *  - Every data pointer is a DEVICE pointer owned by the caller.  The library
 *    never allocates, frees or copies caller memory, and never synchronises a
 *    stream except in igconv_get_device_status().
 *  - Every data pointer of the convolution calls must be 16-byte aligned,
 *    else IGCONV_ERR_MISALIGNED.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is enqueued on it and the call returns without waiting.
 *  - The returned status covers host-side validation and the kernel launch.
 *    A kernel that detects a failure on the device (a pipeline wait that ran
 *    past its time limit) records it in a per-device status word that
 *    igconv_get_device_status() reads; it never traps.
 *  - Validation happens before any work is enqueued: an invalid argument
 *    returns without touching the stream.
 *  - Output size (CUTLASS "03_basic_conv2d.ipynb", "General setup",
 *    cutlass.Conv2d.output_size; without dilation it is the formula of
 *    tensorcore "docs/conv2d.md", "Output spatial dims"):
 *      P = floor((H + 2*pad_h - dil_h*(R-1) - 1) / stride_h) + 1
 *      Q = floor((W + 2*pad_w - dil_w*(S-1) - 1) / stride_w) + 1
 *  - Preconditions common to the convolution calls: every extent >= 1,
 *    pads >= 0, strides and dilations >= 1, P >= 1 and Q >= 1 (else
 *    IGCONV_ERR_INVALID_ARG); C and K multiples of 8 for 16-bit data and of
 *    16 for int8 (the alignment predicate of apache/tvm PR #10177,
 *    "[CUTLASS] Initial support for conv2d wgrad": every channel count a
 *    multiple of the vector width), strides <= 8, pads <= 64, R and S <= 64,
 *    dil*(R-1) and dil*(S-1) <= 127, N <= 65535 (else
 *    IGCONV_ERR_UNSUPPORTED).  The dense entry points are groups = 1
 *    (burn-cubecl `conv_forward_nhwc` takes the implicit-GEMM path for
 *    groups == 1); grouped and depthwise problems use conv2d_grouped_*.
 *  - Accumulation is fp32 for fp16/bf16 data in every pass (apache/tvm PR
 *    #10177, review of the accumulator dtype: fp32 accumulation for wgrad,
 *    and here for all passes); the output conversion rounds to nearest even.
 *  - beta == 0 means Cin is not read and may be NULL.
 */
#ifndef IGCONV_H
#define IGCONV_H

#include <stddef.h>
#include <stdint.h>

/* Exported from the shared library even when it is built with hidden
 * default visibility. */
#if defined(__GNUC__)
#define IGCONV_API __attribute__((visibility("default")))
#else
#define IGCONV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    IGCONV_OK = 0,
    IGCONV_ERR_INVALID_ARG = 1,    /* a dimension, pointer or scalar is invalid */
    IGCONV_ERR_UNSUPPORTED = 2,    /* valid, but outside what the kernels cover */
    IGCONV_ERR_MISALIGNED = 3,     /* a pointer is not 16-byte aligned */
    IGCONV_ERR_WORKSPACE = 4,      /* workspace missing or smaller than required */
    IGCONV_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed */
    IGCONV_ERR_DEVICE_TIMEOUT = 6  /* a kernel's pipeline wait ran out (device-side) */
} igconv_status_t;

typedef enum {
    IGCONV_F16 = 0,
    IGCONV_BF16 = 1,
    IGCONV_F32 = 2,
    IGCONV_I8 = 3,
    IGCONV_I32 = 4
} igconv_dtype_t;

/* Problem shape.  Field names follow the CUTLASS example's N, H, W, C, K, R,
 * S and its (stride, padding, dilation) tuples; P, Q are derived. */
typedef struct {
    int N, H, W, C, K, R, S;
    int pad_h, pad_w, stride_h, stride_w, dil_h, dil_w;
} igconv_problem_t;

/* P and Q from the formula above.  Host only; no CUDA call.
 * Errors: IGCONV_ERR_INVALID_ARG for NULL pointers, non-positive extents,
 * negative pads, strides or dilations < 1, or P < 1 or Q < 1. */
IGCONV_API igconv_status_t conv2d_output_size(const igconv_problem_t *prob, int *P, int *Q);

/* Forward pass (fprop).
 *   Y[n,p,q,k] = cast( relu?( alpha * sum_{r,s,c} X[n, p*sh - ph + r*dh,
 *                                                    q*sw - pw + s*dw, c] * Wt[k,r,s,c]
 *                              + beta * Cin[n,p,q,k] + bias[k] ) )
 * taps outside the input contribute zero.  Sources: alpha/beta from the
 * CUTLASS example, "Declaring and running a Conv2d Fprop"; the optional
 * per-channel bias from tensorcore "docs/conv2d.md", "Surface" and
 * "Strategy" (bias [OC] or NULL); ReLU after the bias add as in PyTorch's
 * quantized cuDNN Conv.cpp, apply_impl_helper<kReluFused>.
 *   dtype    IGCONV_F16 or IGCONV_BF16: X, Wt, bias, Cin and Y all use it.
 *   X        [N][H][W][C]     Wt [K][R][S][C]      Y [N][P][Q][K] (written)
 *   bias     [K] or NULL      Cin [N][P][Q][K], read only when beta != 0
 *   relu     0 or 1
 * Y must not overlap X, Wt, bias or Cin (Cin == Y is allowed).
 * Fewer than 8 input channels need conv2d_fprop_ws and its workspace; here
 * they give WORKSPACE.
 * Errors: INVALID_ARG (shape, NULL X/Wt/Y, NULL Cin with beta != 0,
 * non-finite alpha/beta), UNSUPPORTED (dtype, limits above), MISALIGNED,
 * WORKSPACE (C < 8), CUDA. */
IGCONV_API igconv_status_t conv2d_fprop(const igconv_problem_t *prob, igconv_dtype_t dtype,
                                        const void *X, const void *Wt, const void *bias,
                                        const void *Cin, void *Y, float alpha, float beta,
                                        int relu, void *stream);

/* Bytes of device workspace conv2d_fprop_ws needs for this problem: for C
 * <= 8 the few-channel copies; for larger C the split-K partial tiles when
 * the plan splits the reduction (see conv2d_fprop_ws), else 0.  0 for an
 * invalid problem or dtype.  Host only; queried on the current device (the
 * split choice depends on its SM count). */
IGCONV_API size_t conv2d_fprop_workspace_size(const igconv_problem_t *prob,
                                              igconv_dtype_t dtype);

/* conv2d_fprop with a caller-owned device workspace, which opens the
 * few-channel path for C <= 8 (the first layer of a CNN: C = 3, 7x7 filter,
 * stride 2).  The same result definition as conv2d_fprop.  The path copies
 * the pixels to 8-channel rows (zero channels C..7; skipped when C == 8) and
 * the filter to a [R*S][K][8] layout in the workspace, and packs 8 filter
 * taps x 8 channels into each 64-deep reduction block.
 * With C > 8 and a workspace, the layer can run split-K when the tuning
 * knob IGCONV_TUNE_CONV_SPLITS asks for it: each tile's reduction cut into
 * equal ranges on separate CTAs, which write fp32 partial tiles to the
 * workspace; a second kernel adds them in split order (deterministic) and
 * applies alpha, beta * Cin, bias, ReLU and the cast.  The sums are then
 * grouped differently from the unsplit path (exact on integer data, within
 * the fp32 accumulation bound otherwise).  The built-in plan never splits
 * (measured slower on every layer tried), so by default the size query
 * returns 0 for C > 8 and the layer runs exactly as conv2d_fprop.
 *   workspace        device memory, 16-byte aligned, at least
 *                    conv2d_fprop_workspace_size(prob, dtype) bytes; it must
 *                    stay untouched until the call's kernels have run
 *   X, Wt            2-byte aligned for C < 8 (16-byte for C == 8); the
 *                    other arguments as in conv2d_fprop
 * Errors: as conv2d_fprop; WORKSPACE if C < 8 and the workspace is NULL or
 * too small (or C == 8 with a non-NULL workspace that is too small, or a
 * split plan with a workspace that is too small). */
IGCONV_API igconv_status_t conv2d_fprop_ws(const igconv_problem_t *prob, igconv_dtype_t dtype,
                                           const void *X, const void *Wt, const void *bias,
                                           const void *Cin, void *Y, float alpha, float beta,
                                           int relu, void *workspace, size_t workspace_bytes,
                                           void *stream);

/* Data gradient (dgrad): the adjoint of fprop in X.
 *   dX[n,h,w,c] = cast( alpha * sum over (k, r, s, p, q) with
 *                 p*sh - ph + r*dh == h and q*sw - pw + s*dw == w of
 *                 dY[n,p,q,k] * Wt[k,r,s,c]  +  beta * Cin[n,h,w,c] )
 * Input positions that no output position reads get beta*Cin (or 0).
 * Source: CUTLASS example, "Declaring and running Conv2d Dgrad and Wgrad"
 * (Conv2dDgrad, checked against torch.nn.grad.conv2d_input); burn-cubecl
 * `conv_data_backward`.  Strided problems are computed as stride_h*stride_w
 * sub-convolutions, one per output residue class, with no atomics.
 *   dtype    IGCONV_F16 or IGCONV_BF16 for dY, Wt, Cin, dX.
 *   dY [N][P][Q][K]   Wt [K][R][S][C]   dX [N][H][W][C] (written, every element)
 *   Cin [N][H][W][C], read only when beta != 0.
 * Errors: as conv2d_fprop; also UNSUPPORTED when stride_h*stride_w > 16;
 * WORKSPACE when C < 8 (that path needs conv2d_dgrad_ws). */
IGCONV_API igconv_status_t conv2d_dgrad(const igconv_problem_t *prob, igconv_dtype_t dtype,
                                        const void *dY, const void *Wt, const void *Cin,
                                        void *dX, float alpha, float beta, void *stream);

/* conv2d_dgrad with a caller-owned device workspace, which lets a unit-
 * stride layer run split-K as conv2d_fprop_ws does (fp32 partials in the
 * workspace, an ordered reduction applying alpha and beta * Cin) when the
 * tuning knob IGCONV_TUNE_CONV_SPLITS asks for it.  The size query returns 0
 * (no workspace needed) for strided problems and unsplit plans, which by
 * default is every plan; it is host-only and queried on the current device.
 * Few input channels (C < 8, the first layer of a CNN): the data gradient
 * runs over the filter copied to 8 channels per tap, writes alpha * acc as
 * fp32 rows of 8 channels, and a second kernel adds beta * Cin to the C real
 * channels and casts.  Both copies live in the workspace, so C < 8 always
 * needs one (round256(K*R*S*16) + round256(N*H*W*32) bytes, from the size
 * query); dY must be 16-byte aligned, Wt, dX and Cin only 2-byte aligned.
 * Arguments, errors and the result definition as conv2d_dgrad; WORKSPACE
 * when a split or few-channel plan's workspace is missing or too small. */
IGCONV_API size_t conv2d_dgrad_workspace_size(const igconv_problem_t *prob,
                                              igconv_dtype_t dtype);
IGCONV_API igconv_status_t conv2d_dgrad_ws(const igconv_problem_t *prob, igconv_dtype_t dtype,
                                           const void *dY, const void *Wt, const void *Cin,
                                           void *dX, float alpha, float beta, void *workspace,
                                           size_t workspace_bytes, void *stream);

/* Bytes of device workspace conv2d_wgrad needs for this problem (fp32
 * split-K partial sums; for C < 8 also the pixels copied to 8-channel rows,
 * round256(N*H*W*16) bytes, ahead of the partials).  The split count depends on the SM count of the
 * current device, which this call queries (no work is enqueued); call it
 * with the same device current as the conv2d_wgrad call.  Returns 0 for an
 * invalid problem. */
IGCONV_API size_t conv2d_wgrad_workspace_size(const igconv_problem_t *prob,
                                              igconv_dtype_t dtype, igconv_dtype_t dw_dtype);

/* Weight gradient (wgrad), split-K over N*P*Q with a deterministic reduction.
 *   dW[k,r,s,c] = cast( alpha * sum_{n,p,q} dY[n,p,q,k] *
 *                 X[n, p*sh - ph + r*dh, q*sw - pw + s*dw, c] + beta * Cin[k,r,s,c] )
 * Source: CUTLASS example, "Declaring and running Conv2d Dgrad and Wgrad"
 * (Conv2dWgrad) and "Split-K" (partials in global memory reduced by a second
 * kernel); apache/tvm PR #10177 (fp32 accumulation; GEMM-K is N*P*Q, so
 * split-K is needed).  The partial sums are added in a fixed order, so the
 * result is bit-identical from run to run.
 * Few input channels (C < 8): the pixels are copied to 8-channel rows in the
 * workspace and each 64-row reduction operand packs 8 filter taps x 8
 * channels, so a 7x7 filter takes 7 operand row blocks instead of 49; the
 * reduction writes the C real channels.  X then needs only 2-byte alignment
 * and dW / Cin only their element size; dY stays 16-byte aligned.
 *   dtype     IGCONV_F16 or IGCONV_BF16 for X and dY.
 *   dw_dtype  IGCONV_F16, IGCONV_BF16 or IGCONV_F32 for dW and Cin.
 *   X [N][H][W][C]   dY [N][P][Q][K]   dW [K][R][S][C] (written)
 *   Cin [K][R][S][C], read only when beta != 0.
 *   workspace  device memory of conv2d_wgrad_workspace_size() bytes (what the
 *              fastest plan for the problem needs), owned by the caller;
 *              contents need not be initialised and are overwritten.  A
 *              smaller workspace that still holds the split-K plan's
 *              partials runs that plan instead of the halo plan (see
 *              IGCONV_TUNE_WGRAD_HALO).  It must not be used by another call
 *              that runs concurrently.
 * Errors: as conv2d_fprop; WORKSPACE if workspace is NULL or smaller than
 * every plan needs. */
IGCONV_API igconv_status_t conv2d_wgrad(const igconv_problem_t *prob, igconv_dtype_t dtype,
                                        igconv_dtype_t dw_dtype, const void *X, const void *dY,
                                        const void *Cin, void *dW, float alpha, float beta,
                                        void *workspace, size_t workspace_bytes, void *stream);

/* Size of the fixed device array that conv2d_wgrad_noalloc uses in place of
 * a workspace (32 MiB). */
#define IGCONV_WGRAD_NOALLOC_SCRATCH_BYTES (32u << 20)

/* Weight gradient without a workspace argument.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory -- code running under a memory manager that owns all device
 * memory and only hands it input and output buffers, or code that must not
 * call cudaMalloc on its hot path (the call can synchronise the device and
 * can fail under memory pressure).
 * It computes exactly what conv2d_wgrad computes (same plan, same kernels,
 * same split count, so the same bits), but keeps the split-K partial sums in
 * a fixed device array of IGCONV_WGRAD_NOALLOC_SCRATCH_BYTES that every GPU
 * loading the library holds until exit.  It allocates nothing and frees
 * nothing.
 *   Arguments: as conv2d_wgrad, without workspace / workspace_bytes.
 *   The first call in a device's context looks up the array's device
 *   address (with that device current) and caches it with the context's ID;
 *   a call from a new context (after cudaDeviceReset) looks it up again.
 *   Make the first call on a device, and the first after a reset, before
 *   any stream capture on that device.
 *   All calls on a device share the array: calls whose kernels can overlap
 *   on the GPU (other streams, other host threads) race and must be
 *   serialised by the caller.  Every partial a call reads was written by the
 *   same call, so nothing needs clearing between calls.
 * Errors: as conv2d_wgrad; IGCONV_ERR_WORKSPACE when no plan's partial sums
 * fit IGCONV_WGRAD_NOALLOC_SCRATCH_BYTES (a problem whose size query exceeds
 * the limit may still run its split-K plan). */
IGCONV_API igconv_status_t conv2d_wgrad_noalloc(const igconv_problem_t *prob,
                                                igconv_dtype_t dtype, igconv_dtype_t dw_dtype,
                                                const void *X, const void *dY, const void *Cin,
                                                void *dW, float alpha, float beta, void *stream);

/* Grouped convolution (all three passes).  `groups` G splits the C input
 * and K output channels into G equal runs: output channel k belongs to group
 * g = k / (K/G) and reads only input channels g*(C/G) .. g*(C/G) + C/G - 1.
 * Filters and filter gradients are [K][R][S][C/G]; activations as above.
 *   Y[n,p,q,k] = cast( relu?( alpha * sum_{r,s,j < C/G}
 *                  X[n, p*sh - ph + r*dh, q*sw - pw + s*dw, g*(C/G) + j]
 *                  * Wt[k,r,s,j] + beta * Cin[n,p,q,k] + bias[k] ) )
 * and dgrad / wgrad are its adjoints in X and Wt, with alpha and beta as in
 * conv2d_dgrad / conv2d_wgrad.
 * Sources: burn-cubecl "kernel/conv/base.rs", conv_forward_nhwc
 * (`options.groups`; grouped problems run a direct kernel instead of the
 * implicit GEMM); tensorcore "docs/conv2d.md", "What's not done in v0.1"
 * (depthwise = groups equal to the input channel count, which wants its own
 * kernel); apache/tvm PR #10177 (depthwise wgrad).  Which channels a group
 * holds is not spelled out there; the contiguous runs above match the
 * [K][R][S][C/G] weight shape.
 * Coverage: G == 1 is exactly conv2d_fprop / conv2d_dgrad / conv2d_wgrad
 * (same kernels, same bits, same errors).  C == K with a group width C/G of
 * 1 (depthwise, filters [C][R][S]), 2, 4, 8, 16 or 32 runs direct CUDA-core
 * kernels in conv2d_grouped_fprop / conv2d_grouped_dgrad: such a layer does
 * R*S*C/G multiply-adds per 4 bytes of traffic.  The tensor cores run
 * grouped layers as block-diagonal implicit GEMMs with 64-wide tiles of
 * whole groups: always in conv2d_grouped_wgrad, and in the _ws variants of
 * fprop and dgrad.  That covers C == K with widths 4 and up, and C != K
 * (channel multipliers, K/G != C/G), whenever the per-group channel count
 * on the tile side (K/G for fprop and wgrad, C/G for dgrad) divides 64 or
 * is a multiple of 64, and the reduction window a tile reads from the
 * other side is a multiple of 8 channels.  The window is 64 / (K/G) * (C/G)
 * channels in the first case and C/G in the second (for dgrad swap C and
 * K).  C and K must be multiples of 8.  Every other G gives UNSUPPORTED,
 * and C != K only runs through the workspace entry points.  Each output accumulates in fp32 over its taps
 * in (r, s) order, group channels innermost (wgrad: over N*P*Q in a fixed
 * per-CTA order, then the CTAs' partial sums in a fixed order), so results
 * are deterministic.
 * Errors: INVALID_ARG (shape, G < 1 or not dividing C and K, NULL pointers,
 * non-finite alpha/beta), UNSUPPORTED (dtype, G outside the coverage, the
 * limits of the dense path, a tile window larger than the kernels' shared
 * memory: roughly (7*stride + (R-1)*dil + 1) x (15*stride + (S-1)*dil + 1)
 * pixels of 128 bytes, twice, within 227 KB), MISALIGNED, WORKSPACE, CUDA. */
IGCONV_API igconv_status_t conv2d_grouped_fprop(const igconv_problem_t *prob, int groups,
                                                igconv_dtype_t dtype, const void *X,
                                                const void *Wt, const void *bias,
                                                const void *Cin, void *Y, float alpha,
                                                float beta, int relu, void *stream);
IGCONV_API igconv_status_t conv2d_grouped_dgrad(const igconv_problem_t *prob, int groups,
                                                igconv_dtype_t dtype, const void *dY,
                                                const void *Wt, const void *Cin, void *dX,
                                                float alpha, float beta, void *stream);

/* Grouped fprop with a caller-owned workspace, which opens the tensor-core
 * path (the coverage above): the convolution runs as an implicit GEMM in
 * which output channels 64n .. 64n + 63 (whole groups) reduce only over the
 * input channels their groups read, against a dense block-diagonal copy of
 * the filter that the call writes into the workspace ([K][R][S][C], zeros
 * outside each output channel's group; K*R*S*C*2 bytes).  Every other G is
 * exactly conv2d_grouped_fprop (the workspace is not used).  Same
 * result definition, arguments and errors as conv2d_grouped_fprop, plus
 *   workspace  device memory of at least
 *              conv2d_grouped_fprop_workspace_size() bytes, caller-owned,
 *              overwritten; not shared with a concurrent call.
 * Errors: as conv2d_grouped_fprop; WORKSPACE if the workspace is NULL or
 * too small on the tensor-core path. */
IGCONV_API size_t conv2d_grouped_fprop_workspace_size(const igconv_problem_t *prob, int groups,
                                                      igconv_dtype_t dtype);
IGCONV_API igconv_status_t conv2d_grouped_fprop_ws(const igconv_problem_t *prob, int groups,
                                                   igconv_dtype_t dtype, const void *X,
                                                   const void *Wt, const void *bias,
                                                   const void *Cin, void *Y, float alpha,
                                                   float beta, int relu, void *workspace,
                                                   size_t workspace_bytes, void *stream);

/* Grouped dgrad with a caller-owned workspace: within the tensor-core
 * coverage above (tiles over C) the dgrad implicit GEMM (with its residue
 * classes for strides) runs with 64-wide tiles in which dX channels
 * 64n .. 64n + 63 (whole groups) reduce only over the dY channels of their
 * groups, against the dense block-diagonal filter image the call writes into
 * the workspace (as in conv2d_grouped_fprop_ws).  Every other G is exactly
 * conv2d_grouped_dgrad.
 * Arguments and errors as conv2d_grouped_dgrad, plus the workspace (at
 * least conv2d_grouped_dgrad_workspace_size() bytes, caller-owned,
 * overwritten, not shared with a concurrent call; WORKSPACE if missing or
 * too small on the tensor-core path). */
IGCONV_API size_t conv2d_grouped_dgrad_workspace_size(const igconv_problem_t *prob, int groups,
                                                      igconv_dtype_t dtype);
IGCONV_API igconv_status_t conv2d_grouped_dgrad_ws(const igconv_problem_t *prob, int groups,
                                                   igconv_dtype_t dtype, const void *dY,
                                                   const void *Wt, const void *Cin, void *dX,
                                                   float alpha, float beta, void *workspace,
                                                   size_t workspace_bytes, void *stream);

/* Workspace bytes conv2d_grouped_wgrad needs (the direct kernels, C == K
 * widths 1 and 2: fp32 partial sums [splits][R*S][C][C/G]; the tensor-core
 * path: the block-diagonal GEMM's split partials and the fp32 gradient of
 * the windowed filter [K][R][S][window rounded up to 64]); the split count follows the current device's SM count
 * and the kernel's occupancy, which this call queries without enqueuing
 * work).  0 for an invalid or uncovered problem. */
IGCONV_API size_t conv2d_grouped_wgrad_workspace_size(const igconv_problem_t *prob, int groups,
                                                      igconv_dtype_t dtype,
                                                      igconv_dtype_t dw_dtype);
/* Workspace: caller-owned device memory of at least the size above,
 * overwritten, not shared with a concurrent call.  dw_dtype F16, BF16 or F32
 * for dW and Cin ([K][R][S][C/G]). */
IGCONV_API igconv_status_t conv2d_grouped_wgrad(const igconv_problem_t *prob, int groups,
                                                igconv_dtype_t dtype, igconv_dtype_t dw_dtype,
                                                const void *X, const void *dY, const void *Cin,
                                                void *dW, float alpha, float beta,
                                                void *workspace, size_t workspace_bytes,
                                                void *stream);

/* 3D convolution (volumes): the same conventions with a depth dimension.
 *   X [N][D][H][W][C]   Wt [K][T][R][S][C]   Y [N][Do][P][Q][K]
 *   Do = floor((D + 2*pad_d - dil_d*(T-1) - 1) / stride_d) + 1 (P, Q as in 2D)
 * Sources: burn-cubecl "kernel/conv/base.rs" (ConvOptions<N>: one stride,
 * padding and dilation per spatial dimension, the convolution generic over
 * the spatial rank); PyTorch quantized cuDNN Conv.cpp (kSpatialDim 2 or 3). */
typedef struct {
    int N, D, H, W, C, K, T, R, S;
    int pad_d, pad_h, pad_w, stride_d, stride_h, stride_w, dil_d, dil_h, dil_w;
} igconv_problem3d_t;

/* Do, P, Q.  Host only.  INVALID_ARG as conv2d_output_size. */
IGCONV_API igconv_status_t conv3d_output_size(const igconv_problem3d_t *prob, int *Do, int *P,
                                              int *Q);

/* 3D forward pass:
 *   Y[n,o,p,q,k] = cast( relu?( alpha * sum_{t,r,s,c}
 *                  X[n, o*sd - pd + t*dd, p*sh - ph + r*dh, q*sw - pw + s*dw, c]
 *                  * Wt[k,t,r,s,c] + beta * Cin[n,o,p,q,k] + bias[k] ) )
 * with taps outside the input contributing zero.  It runs the implicit-GEMM
 * kernel with the input gathered by TMA's 5D im2col mode (one reduction
 * block = one (t, r, s) tap x 64 channels).  dtype, bias, Cin, relu, alpha,
 * beta, aliasing and errors as conv2d_fprop.  Limits (else UNSUPPORTED): C
 * and K multiples of 8, strides <= 8, pads <= 15 and dil*(k-1) <= 15 in
 * every dimension (the 5D im2col bounding box), N <= 65535. */
IGCONV_API igconv_status_t conv3d_fprop(const igconv_problem3d_t *prob, igconv_dtype_t dtype,
                                        const void *X, const void *Wt, const void *bias,
                                        const void *Cin, void *Y, float alpha, float beta,
                                        int relu, void *stream);

/* 3D data gradient (stride_d * stride_h * stride_w <= 16, else UNSUPPORTED):
 *   dX[n,d,h,w,c] = cast( alpha * sum over (k,t,r,s) and the output position
 *                   (o,p,q) that reads (d,h,w) through tap (t,r,s) of
 *                   dY[n,o,p,q,k] * Wt[k,t,r,s,c]  +  beta * Cin[n,d,h,w,c] )
 * computed as the implicit GEMM over the 5D im2col of dY, one sub-problem
 * per output residue class (o mod sd, h mod sh, w mod sw) with the taps that
 * reach it, as conv2d_dgrad does in 2D.  Positions no output reads get
 * beta*Cin (or 0).  dY [N][Do][P][Q][K], dX [N][D][H][W][C]; dtype, Cin,
 * errors and limits as conv3d_fprop. */
IGCONV_API igconv_status_t conv3d_dgrad(const igconv_problem3d_t *prob, igconv_dtype_t dtype,
                                        const void *dY, const void *Wt, const void *Cin,
                                        void *dX, float alpha, float beta, void *stream);

/* 3D weight gradient, split-K over N*Do*P*Q with the deterministic reduction
 * of conv2d_wgrad:
 *   dW[k,t,r,s,c] = cast( alpha * sum_{n,o,p,q} dY[n,o,p,q,k] *
 *                   X[n, o*sd - pd + t*dd, p*sh - ph + r*dh, q*sw - pw + s*dw, c]
 *                   + beta * Cin[k,t,r,s,c] )
 * dW and Cin [K][T][R][S][C] in dw_dtype (F16, BF16 or F32); workspace as
 * conv2d_wgrad (size from conv3d_wgrad_workspace_size, queried on the
 * current device).  Limits as conv3d_fprop. */
IGCONV_API size_t conv3d_wgrad_workspace_size(const igconv_problem3d_t *prob,
                                              igconv_dtype_t dtype, igconv_dtype_t dw_dtype);
IGCONV_API igconv_status_t conv3d_wgrad(const igconv_problem3d_t *prob, igconv_dtype_t dtype,
                                        igconv_dtype_t dw_dtype, const void *X, const void *dY,
                                        const void *Cin, void *dW, float alpha, float beta,
                                        void *workspace, size_t workspace_bytes, void *stream);

/* Forward pass by Winograd's minimal filtering F(2x2, 3x3), for 3x3 filters
 * at stride 1 and dilation 1 (tensorcore "docs/conv2d.md", "What's not done
 * in v0.1", names it for 3x3 stride-1 layers with a 2-2.25x multiply
 * saving).  Over 4x4 input patches d at stride 2 and each 3x3 filter g:
 *   V = Bt d B,  U = G g Gt,  M[xi] = sum_c V[xi][c] U[xi][c],  Y = At M A
 *   Bt = [1 0 -1 0; 0 1 1 0; 0 -1 1 0; 0 1 0 -1]
 *   G  = [1 0 0; 1/2 1/2 1/2; 1/2 -1/2 1/2; 0 0 1],  At = [1 1 1 0; 0 1 -1 -1]
 * which equals conv2d_fprop's sum in real arithmetic; then alpha, beta*Cin,
 * bias, ReLU and the cast exactly as conv2d_fprop.  V, U and M are rounded to
 * the 16-bit I/O type (round to nearest even); the 16 products sum over C in
 * fp32 on the tensor cores (one implicit-GEMM launch, one sub-problem per
 * transform point).  The result is therefore not bit-equal to conv2d_fprop;
 * its error is bounded by the roundings of V, U and M (see the tests).
 *   Arguments as conv2d_fprop, plus workspace (V [16][T][C], U [K][16][C],
 *   M [16][T][K], T = N * ceil(P/2) * ceil(Q/2)) of at least
 *   conv2d_fprop_winograd_workspace_size() bytes, caller-owned, overwritten,
 *   not shared with a concurrent call.
 *   R = S = 3, strides 1, dilations 1, C and K multiples of 8 (else
 *   UNSUPPORTED; the size query returns 0).
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA. */
IGCONV_API size_t conv2d_fprop_winograd_workspace_size(const igconv_problem_t *prob,
                                                       igconv_dtype_t dtype);
IGCONV_API igconv_status_t conv2d_fprop_winograd(const igconv_problem_t *prob,
                                                 igconv_dtype_t dtype, const void *X,
                                                 const void *Wt, const void *bias,
                                                 const void *Cin, void *Y, float alpha,
                                                 float beta, int relu, void *workspace,
                                                 size_t workspace_bytes, void *stream);

/* Bytes of device workspace conv2d_fprop_int8 needs (fp16 copies of X and
 * Wt, which the tensor cores consume, and for R*S*C above 4096 the int32
 * partial tiles of the split reduction).  Host only, queried on the current
 * device; 0 for an invalid problem. */
IGCONV_API size_t conv2d_fprop_int8_workspace_size(const igconv_problem_t *prob);

/* Quantised forward pass.
 *   acc = sum_{r,s,c} X*Wt, exact in integer arithmetic
 *   t   = acc + bias[k]                 (int32 bias in accumulator units)
 *   t   = max(t, 0)  when relu
 *   Y   = clamp(round_half_even(t * M), -128, 127),
 *   M   = (float)((act_scale * w_scale) / out_scale), quotient in double
 * Source: PyTorch quantized cuDNN Conv.cpp, apply_impl_helper<kReluFused>
 * (requantize multiplier act_scale * weight_scale / output_scale from double
 * q_scale() values; conv, then bias add, then ReLU, then the multiply into an
 * int8 output).  The pages do not state the rounding or saturation rule, nor
 * the bias units; the rule above is this library's reading.  The product
 * t * M is evaluated exactly (integer multiply by M's significand and a
 * half-even shift), so Y is unique.  Zero points are 0 (symmetric).
 *   X  [N][H][W][C] int8   Wt [K][R][S][C] int8   bias [K] int32 or NULL
 *   Y  [N][P][Q][K] int8 (written)
 *   scales finite and > 0.  C and K multiples of 16.
 * acc is exact while |acc| < 2^31.  Up to R*S*C = 4096 (64 blocks of 64
 * channels) a tile's whole reduction fits its TMEM accumulators (at most
 * 16 blocks each, so every fp32 partial sum is an exact integer).  Above
 * that the reduction is split into equal ranges of at most 64 blocks whose
 * int32 partial tiles are added in split order (modulo 2^32, as one int32
 * accumulator would) before the bias, ReLU and requantisation.
 *   workspace  >= conv2d_fprop_int8_workspace_size() bytes, caller-owned,
 *              overwritten; not shared with a concurrent call.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA. */
IGCONV_API igconv_status_t conv2d_fprop_int8(const igconv_problem_t *prob, const int8_t *X,
                                             const int8_t *Wt, const int32_t *bias, int8_t *Y,
                                             double act_scale, double w_scale, double out_scale,
                                             int relu, void *workspace, size_t workspace_bytes,
                                             void *stream);

/* int8 data and weight gradients, int32 results (the int8 convolution's
 * INT32 compute type of PyTorch quantized cuDNN Conv.cpp, whose op is generic
 * over the spatial rank, carried to the adjoint passes of conv2d_dgrad and
 * conv2d_wgrad).  The pages define no requantisation for these passes, so
 * the result is the integer sum itself, delivered as int32: the exact sum
 * modulo 2^32 (two's complement), what an int32 accumulator holds.
 *   dX[n,h,w,c] = sum over (k, r, s) and the output position (p, q) that
 *                 reads (h, w) through tap (r, s) of dY[n,p,q,k] * Wt[k,r,s,c]
 *   dW[k,r,s,c] = sum_{n,p,q} dY[n,p,q,k] * X[n, p*sh - ph + r*dh, q*sw - pw + s*dw, c]
 * The operands are widened to fp16 copies in the workspace (exact); the
 * implicit GEMM of the 16-bit pass runs on them with every fp32 accumulator
 * summing at most 1024 products (each partial sum an integer below 2^24, so
 * exact), and the epilogue adds the accumulators as int32.  Input positions
 * no output reads get 0.
 *   dY [N][P][Q][K] int8, X [N][H][W][C] int8, Wt [K][R][S][C] int8,
 *   dX [N][H][W][C] int32 (written), dW [K][R][S][C] int32 (written).
 *   C and K multiples of 16; dgrad: stride_h * stride_w <= 16; dgrad and
 *   the per-split reduction must fit the accumulators (else UNSUPPORTED).
 *   workspace  >= the *_workspace_size() bytes (queried on the current device
 *              for wgrad), caller-owned, overwritten; not shared with a
 *              concurrent call.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA. */
IGCONV_API size_t conv2d_dgrad_int8_workspace_size(const igconv_problem_t *prob);
IGCONV_API igconv_status_t conv2d_dgrad_int8(const igconv_problem_t *prob, const int8_t *dY,
                                             const int8_t *Wt, int32_t *dX, void *workspace,
                                             size_t workspace_bytes, void *stream);
IGCONV_API size_t conv2d_wgrad_int8_workspace_size(const igconv_problem_t *prob);
IGCONV_API igconv_status_t conv2d_wgrad_int8(const igconv_problem_t *prob, const int8_t *X,
                                             const int8_t *dY, int32_t *dW, void *workspace,
                                             size_t workspace_bytes, void *stream);

/* Layout permutes (burn-cubecl "kernel/conv/base.rs": permute_nchw_to_nhwc
 * around the NHWC core in `conv_forward`, permute_nhwc_to_nchw after it).
 *   nchw_to_nhwc: dst[n][h][w][c] = src[n][c][h][w]
 *   nhwc_to_nchw: dst[n][c][h][w] = src[n][h][w][c]
 * elem_bytes is 1, 2, 4 or 8.  src and dst must not overlap.  Pointers need
 * only elem_bytes alignment here (16-byte alignment takes the vector path).
 * Errors: INVALID_ARG (NULL, non-positive extents, bad elem_bytes),
 * MISALIGNED, UNSUPPORTED (N > 65535), CUDA. */
IGCONV_API igconv_status_t nchw_to_nhwc(const void *src, void *dst, int N, int C, int H, int W,
                                        int elem_bytes, void *stream);
IGCONV_API igconv_status_t nhwc_to_nchw(const void *src, void *dst, int N, int C, int H, int W,
                                        int elem_bytes, void *stream);

/* Synchronises `stream`, then returns and clears the current device's
 * status word: IGCONV_OK, or IGCONV_ERR_DEVICE_TIMEOUT if a kernel gave up
 * on a pipeline wait since the last call.  IGCONV_ERR_CUDA if the
 * synchronisation itself failed. */
IGCONV_API igconv_status_t igconv_get_device_status(void *stream);

/* Static, human-readable name of a status code. */
IGCONV_API const char *igconv_status_string(igconv_status_t status);

/* Tuning overrides for tests and sweeps; 0 restores the built-in choice.
 * The grid cap leaves every result bit-identical.  The tile width decides how
 * the fp32 reduction is grouped (widths 64 and 128 add two interleaved
 * partial sums, width 256 keeps one), and the wgrad split count decides where
 * the partial sums are cut; results for different settings agree within
 * rounding (exactly on data whose sums are exact in fp32), and for fixed
 * settings they are deterministic.
 * Not thread-safe: set them before issuing calls from other threads.
 *   IGCONV_TUNE_WGRAD_SPLITS  split-K factor of conv2d_wgrad (clamped to the
 *                             number of 64-deep reduction blocks), and CTAs
 *                             per 64-channel chunk of depthwise wgrad
 *                             (clamped to the number of 8 x 16 dY tiles)
 *   IGCONV_TUNE_BLOCK_N       GEMM tile width: 64, 128 or 256
 *   IGCONV_TUNE_MAX_CTAS      cap on the persistent grid size
 *   IGCONV_TUNE_CTA_PAIRS     0: fprop and stride-1 dgrad with 128-wide
 *                             tiles run on pairs of CTAs (a cluster of two
 *                             SMs sharing 256-row MMAs); 1: never; 2: with
 *                             256-wide tiles as well.
 *                             Results are bit-identical either way.
 *   IGCONV_TUNE_EPI_GROUPS    0 or 2: 64-wide tiles (unpaired, not the
 *                             wgrad partials) run their epilogue as two
 *                             groups of four warps taking alternate tiles,
 *                             with four TMEM buffers; 1: one group of eight
 *                             warps per tile, two buffers (not for halo
 *                             plans, see IGCONV_TUNE_HALO, which always run
 *                             two groups).  Results are bit-identical.
 *   IGCONV_TUNE_CONV_SPLITS   split-K of conv2d_fprop_ws / conv2d_dgrad_ws
 *                             (when given a workspace): 0 or 1 never (the
 *                             built-in choice), n >= 2 always n (at most 16,
 *                             clamped to the reduction blocks; CTA pairs
 *                             are then not used).
 *   IGCONV_TUNE_FEW_CHANNELS  few-channel fprop and wgrad (C <= 8): 0 the
 *                             built-in choice (the space-to-depth packed
 *                             path at dilation 1 when stride_h * stride_w
 *                             * C <= 64, else the tap-packed one); 1 always
 *                             the tap-packed path.  Query workspace sizes
 *                             after setting it.
 *   IGCONV_TUNE_RASTER        order in which the persistent CTAs take the
 *                             fprop / dgrad tiles (the "Swizzling Stride"
 *                             of the CUTLASS example): 0 or 1 column tiles
 *                             fastest (the built-in order); g in 2..64 runs
 *                             of g row tiles, rows fastest within each
 *                             column.  Results are bit-identical.
 *   IGCONV_TUNE_RESIDENT_FILTER  0: fprop / stride-1 dgrad plans with
 *                             64-wide tiles, a single column tile and at
 *                             most 4 reduction blocks per tile keep the
 *                             whole filter in shared memory (loaded once
 *                             per CTA; the pipeline stages then carry only
 *                             the im2col rows); 1: never.  Results are
 *                             bit-identical.
 *   IGCONV_TUNE_DGRAD_ROWS    strided dgrad (stride_h * stride_w > 1) with
 *                             H and W divisible by the strides: 0 pads each
 *                             residue class's rows to a multiple of 32
 *                             grid columns where that adds at most a sixth,
 *                             and writes dX through TMA stores of whole
 *                             class rows (the built-in choice); 1 never:
 *                             every output pixel is stored by its own row
 *                             address.  Results are bit-identical.
 *   IGCONV_TUNE_EPILOGUE_KERNEL  0: 2D fprop / dgrad plans with 16-bit
 *                             outputs run on kernels whose epilogue holds
 *                             only that store path (the built-in choice);
 *                             1: on the kernels that carry every epilogue.
 *                             Results are bit-identical.
 *   IGCONV_TUNE_HALO          stride-1 fprop and dgrad with 64 output
 *                             channels, one 64-channel reduction block and
 *                             2..9 filter taps: 0 reads each tile's input
 *                             rows once (a halo) for all its taps (the
 *                             built-in choice where the output width fits a
 *                             grid of 32, 64 or 128 columns and the output
 *                             height a multiple of 128 / that width); 1 never
 *                             (one im2col copy per tap).  The halo plan adds
 *                             a tile's taps in order into one fp32
 *                             accumulator, the per-tap plan alternates them
 *                             between two, so on non-integer data the two
 *                             round differently (each deterministically).
 *   IGCONV_TUNE_ONE_ISSUER    fprop / dgrad with 64-wide tiles of at most
 *                             four reduction blocks (1x1 layers, the packed
 *                             stem, strided dgrad): 0 each tile is issued by
 *                             one of the two MMA issuers into one
 *                             accumulator (the built-in choice); 1 the
 *                             issuers alternate blocks into two
 *                             accumulators.  The two add the blocks in
 *                             different orders: exact alike on integer data,
 *                             each deterministic otherwise.
 *   IGCONV_TUNE_WGRAD_HALO    conv2d_wgrad with stride 1, C and K at most 128
 *                             and 2..9 filter taps: 0 runs on input halos
 *                             (one copy of a block's input rows for every
 *                             tap, every tap pair of a split in one CTA;
 *                             the built-in choice where the output width
 *                             fits a grid of 32, 64 or 128 columns, P is a
 *                             multiple of 128 / that width and the
 *                             workspace holds its partials); 1 never.  The
 *                             two sum the positions in different orders:
 *                             exact alike on integer data, each
 *                             deterministic otherwise.  Query the workspace
 *                             size after setting it.
 *   IGCONV_TUNE_PDL           0: plain launches (the built-in choice); 1:
 *                             the implicit-GEMM kernels and the wgrad split
 *                             reductions launch with programmatic dependent
 *                             launch: such a kernel may start while the
 *                             kernel before it in the stream finishes, and
 *                             waits for it to complete before it touches
 *                             global memory, so the stream's order holds.
 *                             The results are the same either way; in a
 *                             replayed CUDA graph of back-to-back layers the
 *                             plain launches measured slightly faster.
 * Returns INVALID_ARG for an unknown key or value. */
typedef enum {
    IGCONV_TUNE_WGRAD_SPLITS = 1,
    IGCONV_TUNE_BLOCK_N = 2,
    IGCONV_TUNE_MAX_CTAS = 3,
    IGCONV_TUNE_CTA_PAIRS = 4,
    IGCONV_TUNE_EPI_GROUPS = 5,
    IGCONV_TUNE_CONV_SPLITS = 6,
    IGCONV_TUNE_FEW_CHANNELS = 7,
    IGCONV_TUNE_RASTER = 8,
    IGCONV_TUNE_RESIDENT_FILTER = 9,
    IGCONV_TUNE_DGRAD_ROWS = 10,
    IGCONV_TUNE_EPILOGUE_KERNEL = 11,
    IGCONV_TUNE_HALO = 12,
    IGCONV_TUNE_ONE_ISSUER = 13,
    IGCONV_TUNE_WGRAD_HALO = 14,
    IGCONV_TUNE_PDL = 15
} igconv_tune_key_t;
IGCONV_API igconv_status_t igconv_set_tuning(igconv_tune_key_t key, int value);

/* Self-test of the device-side failure path: launches one small kernel that
 * waits on a barrier nothing will ever complete, with a wait limit of
 * `timeout_us` microseconds (1..2000000).  The kernel records
 * IGCONV_ERR_DEVICE_TIMEOUT in the status word and exits cleanly; the
 * context stays usable.  Read the result with igconv_get_device_status(). */
IGCONV_API igconv_status_t igconv_selftest_wait_timeout(int timeout_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* IGCONV_H */
