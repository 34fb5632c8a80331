/*
 * bitlinear.h -- C ABI of libbitlinear.so, the BitNet b1.58 BitLinear forward
 * pass on NVIDIA B300 (sm_103a).
 *
 * The operation (BitLinear replaces a dense linear layer; its weights take
 * only the values -1, 0, +1, chosen by an absmean quantiser, and its
 * activations are 8-bit integers; anthology note-168 on arXiv 2402.17764,
 * section "What it does"; the yousumm.com transcript of the BitNet b1.58 2B4T
 * video, the paragraph on the warehouse analogy):
 *
 *   gamma  = mean(|W|)                                 one fp32 per matrix
 *   W_q    = clip(round(W / (gamma + eps)), -1, +1)
 *   s[m]   = 127 / max_k |X[m,k]|                      one fp32 per token
 *   x_q    = clip(round(X * s[m]), -128, 127)          int8
 *   acc    = W_q . x_q   (int32; the product only adds and subtracts
 *            activations: anthology note-168, "The part that is a bet rather
 *            than a measurement")
 *   y[m,n] = acc[m,n] * gamma / s[m]                   fp32
 *
 * Numerical contract (every result below is reproduced bit for bit by the
 * library; the test-suite checks it against an independent CPU oracle):
 *   - gamma is the exact real mean of |W| rounded once to fp32 (ties to
 *     even), independent of summation order;
 *   - round() is round-half-to-even; gamma + eps, W / (gamma + eps),
 *     127 / max|x| and X * s are single IEEE fp32 operations;
 *   - max|X[m,:]| is clamped from below at BITLINEAR_ACT_CLAMP_EPS, so an
 *     all-zero token gives x_q = 0 and y = 0;
 *   - y[m,n] = fp32( fp32(acc[m,n]) * fp32(gamma / s[m]) ).
 *
 * Packed weight layout (four ternary weights per byte: yousumm.com
 * transcript, paragraph on running the model on graphics cards): row-major
 * [N, K/4] bytes; weight (n, k) is the 2-bit code W_q + 1 in {0, 1, 2} at
 * bits 2*(k % 4) of byte n*K/4 + k/4.  Code 3 is never written.
 *
 * Conventions for every entry point:
 *   - every array pointer is a DEVICE pointer owned by the caller (e.g. a
 *     torch tensor); the library allocates no device memory in these calls
 *     and keeps no per-call state;
 *   - every call is asynchronous on `stream` (0 = legacy default stream);
 *     arguments are validated on the host before anything is launched, and
 *     on a validation error nothing is launched and no output is touched;
 *   - arrays are dense and row-major; the required alignments are stated per
 *     call (BL_ERR_MISALIGNED otherwise);
 *   - kernels that wait on an on-chip barrier give up after a bounded number
 *     of polls instead of hanging; they then record an error word that
 *     bitlinear_check_device_error() reports as BL_ERR_TIMEOUT.
 */
#ifndef BITLINEAR_H
#define BITLINEAR_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BL_OK = 0,
  BL_ERR_INVALID_ARG = 1,       /* null pointer, size <= 0, bad eps or dtype */
  BL_ERR_UNSUPPORTED_SHAPE = 2, /* a size outside the limits stated per call */
  BL_ERR_MISALIGNED = 3,        /* a pointer without the stated alignment */
  BL_ERR_WORKSPACE = 4,         /* workspace smaller than required */
  BL_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed */
  BL_ERR_TIMEOUT = 6            /* a kernel's bounded wait expired (see above) */
} bl_status;

typedef enum { BL_F32 = 0, BL_BF16 = 1 } bl_dtype;

/* Lower clamp of max|X[m,:]| before s = 127 / max|X[m,:]|. */
#define BITLINEAR_ACT_CLAMP_EPS 1e-5f

/* Largest K accepted by bitlinear_forward: 127 * K stays below 2^24, so every
 * partial sum of the product is an integer that fp32 holds exactly. */
#define BITLINEAR_MAX_K 131072

/* Largest K of the base-3 weight format's forward (bitlinear_forward_tq5). */
#define BITLINEAR_TQ5_MAX_K 40960

/*
 * bitlinear_pack_workspace_bytes -- bytes of device workspace that
 * bitlinear_pack_weights needs for an [N, K] matrix (a small constant).
 */
size_t bitlinear_pack_workspace_bytes(int64_t N, int64_t K);

/*
 * bitlinear_pack_weights -- absmean ternarisation and 2-bit packing of one
 * latent weight matrix (anthology note-168, "What it does": an absmean
 * quantiser maps every weight to -1, 0 or +1; yousumm.com
 * transcript: four weights per byte).
 *
 *   W          in   fp32 [N, K] row-major, 16-byte aligned, finite values
 *   N, K       in   N >= 1, K >= 4, K % 4 == 0, N*K <= 2^32
 *   eps        in   finite, > 0 (the eps of gamma + eps; 1e-5 is usual)
 *   W_packed   out  uint8 [N, K/4], 16-byte aligned (layout above)
 *   gamma      out  one fp32 (device), 4-byte aligned: mean |W|
 *   workspace  tmp  >= bitlinear_pack_workspace_bytes(N, K) bytes, 16-byte
 *                   aligned; clobbered; may be reused once the call's work on
 *                   `stream` is done
 *
 * If W holds an inf or NaN, gamma is NaN and W_packed is unspecified.
 * Launches four kernels on `stream`; touches W twice (read 4*N*K bytes each
 * time) and writes N*K/4 bytes.
 */
bl_status bitlinear_pack_weights(const float* W, int64_t N, int64_t K, float eps, uint8_t* W_packed, float* gamma,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * bitlinear_pack_weights_noalloc -- the same packing as bitlinear_pack_weights
 * (identical W_packed and gamma), for callers that cannot supply device
 * workspace: applications whose device memory belongs to their own pool
 * allocator (an extra cudaMalloc would fail or fragment it), and plug-in
 * hosts that only pass pointers to memory they own.  The BitNet b1.58 pages
 * have no counterpart of this call; it only changes where the workspace
 * lives.
 *
 * The workspace is a fixed 512-byte array inside the library's device image
 * (held by every GPU that loads the library until the process exits), so the
 * call allocates nothing and needs no workspace argument.  Arguments, limits
 * and errors are those of bitlinear_pack_weights; a request needing more
 * workspace than the array holds returns BL_ERR_WORKSPACE (the packing
 * workspace is a constant 272 bytes, so no valid shape does).
 *
 * The first call in a CUDA context (with that context current: normally the
 * device's primary context) looks up the array's device address with
 * cudaGetSymbolAddress and caches it for that context; make that first call
 * before any stream capture.  A device reset, or another context made
 * current, is a new context and gets its own lookup.  Every call in a
 * context shares the one array, whose contents persist between calls and are
 * cleared on `stream` at the start of each call: calls that may overlap on
 * the GPU (different streams without ordering between them) race on it and
 * must be serialised by the caller.
 */
bl_status bitlinear_pack_weights_noalloc(const float* W, int64_t N, int64_t K, float eps, uint8_t* W_packed,
                                         float* gamma, cudaStream_t stream);

/*
 * bitlinear_tq5_row_bytes -- bytes per row of the base-3 weight format:
 * ceil(K / 5) rounded up to a multiple of 16 (0 for K < 1).
 */
int64_t bitlinear_tq5_row_bytes(int64_t K);

/*
 * bitlinear_pack_weights_tq5 -- bitlinear_pack_weights written in the base-3
 * format: five ternary weights per byte, 1.6 bits per weight, close to the
 * log2(3) = 1.58 bits a three-valued weight carries (yousumm.com transcript,
 * the GPU-plumbing paragraph; anthology note-168, "What it does").  Byte j
 * of row n holds sum_{i<5} (W_q[n, 5j+i] + 1) * 3^i, least significant digit
 * first, a value in 0..242; positions at or past K count as W_q = 0, and each
 * row is padded with 121 (five zero codes) to bitlinear_tq5_row_bytes(K)
 * bytes.  gamma and W_q are those of bitlinear_pack_weights bit for bit.
 *
 *   W, N, K, eps, gamma, workspace, workspace_bytes, stream
 *            as for bitlinear_pack_weights (K % 4 == 0, N * K <= 2^32)
 *   W_tq5    out  uint8 [N, bitlinear_tq5_row_bytes(K)], 16-byte aligned
 */
bl_status bitlinear_pack_weights_tq5(const float* W, int64_t N, int64_t K, float eps, uint8_t* W_tq5, float* gamma,
                                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * bitlinear_forward_tq5 -- bitlinear_forward from base-3 packed weights:
 * acc = W_q . x_q exact in int32, y = fp32(fp32(acc) * fp32(gamma / s[m])),
 * bit-identical to bitlinear_forward on the 2-bit packing of the same W_q.
 * Tokens are taken up to four at a time and every pass streams the weights
 * once, so the format serves decode (a few tokens).
 *
 *   W_tq5     in   uint8 [N, bitlinear_tq5_row_bytes(K)], 16-byte aligned
 *   gamma, x_q, s, y, acc   as for bitlinear_forward
 *   M, N, K   in   M >= 1, 1 <= N <= 2048 * (number of SMs), K % 16 == 0,
 *                  16 <= K <= BITLINEAR_TQ5_MAX_K
 *   flags     in   0, BITLINEAR_RELU2, and/or the test hook BITLINEAR_TEST_STALL
 *
 * Errors: BL_ERR_INVALID_ARG (null pointer, size < 1, unknown flag),
 * BL_ERR_UNSUPPORTED_SHAPE, BL_ERR_MISALIGNED, BL_ERR_CUDA.
 */
bl_status bitlinear_forward_tq5(const uint8_t* W_tq5, const float* gamma, const int8_t* x_q, const float* s,
                                int64_t M, int64_t N, int64_t K, float* y, int32_t* acc, unsigned flags,
                                cudaStream_t stream);

/*
 * bitlinear_quant_act -- per-token absmax quantisation of activations to int8
 * (anthology note-168, "What it does": activations at 8 bits; yousumm.com
 * transcript: messages squeezed into "eight-bit numbers").
 *
 *   X      in   [M, K] row-major, dtype BL_BF16 or BL_F32, 16-byte aligned
 *   M, K   in   M >= 1, 1 <= K <= 2^24
 *   x_q    out  int8 [M, K] row-major, 16-byte aligned
 *   s      out  fp32 [M]: s[m] = 127 / max(max_k |X[m,k]|, 1e-5), 4-byte aligned
 *
 * x_q always lies in [-127, 127].  Non-finite X gives unspecified x_q and s.
 */
bl_status bitlinear_quant_act(const void* X, bl_dtype dtype, int64_t M, int64_t K, int8_t* x_q, float* s,
                              cudaStream_t stream);

/*
 * bitlinear_rmsnorm_quant_act -- the normalisation that BitNet b1.58 2B4T adds
 * inside each sub-layer, ahead of a BitLinear (yousumm.com transcript, the
 * paragraph after the poker-chip analogy), followed by the per-token absmax
 * quantisation of the normalised row.  The pages give no formula; this is
 * RMS normalisation with an optional per-channel gain, per token m:
 *
 *   ms   = mean_k X[m,k]^2: the exact real mean of the squares, rounded once
 *          to fp32 (ties to even), so it does not depend on summation order
 *   r    = fp32(sqrt(fp32(ms + eps)))            (IEEE square root)
 *   x_n  = fp32(fp32(X[m,k] * gain[k]) / r)      (one multiply, one division)
 *   x_q, s = bitlinear_quant_act of x_n           (bit for bit)
 *
 * so bitlinear_forward(..., x_q, s, ...) then yields W_q applied to x_n.
 *
 *   X       in   [M, K] row-major, BL_BF16 or BL_F32, element-aligned
 *   M, K    in   M >= 1, 1 <= K <= 2^24
 *   gain    in   fp32 [K] (4-byte aligned) or NULL for all ones
 *   eps     in   finite, > 0
 *   x_q, s  out  as for bitlinear_quant_act (x_q needs no alignment here)
 *
 * Results are unspecified where X holds a non-finite value or X * gain
 * overflows fp32.  A row whose mean square overflows fp32 gives r = inf and
 * x_q = 0.  One CTA per token; rows and gains that are 16-byte aligned take a
 * vectorised path with the same arithmetic; from 1536 tokens with rows of at
 * most 8 KB, one warp per token (same results bit for bit).
 */
bl_status bitlinear_rmsnorm_quant_act(const void* X, bl_dtype dtype, int64_t M, int64_t K, const float* gain,
                                      float eps, int8_t* x_q, float* s, cudaStream_t stream);

/*
 * bitlinear_forward -- y = (W_q . x_q) * gamma / s: the ternary-times-int8
 * product accumulated exactly in int32, rescaled per token by gamma/s[m] in
 * a fused epilogue (anthology note-168, "The part that is a bet rather than a
 * measurement": the product only involves integer addition; yousumm.com
 * transcript, the paragraph on running the model on graphics cards: packed
 * weights are expanded beside the arithmetic units and multiplied with the
 * 8-bit activations).
 *
 *   W_packed  in   uint8 [N, K/4] from bitlinear_pack_weights, 16-byte aligned
 *   gamma     in   one fp32 (device)
 *   x_q, s    in   int8 [M, K] (16-byte aligned) and fp32 [M] from
 *                  bitlinear_quant_act
 *   M, N, K   in   M >= 1, N >= 1, K % 64 == 0, 64 <= K <= BITLINEAR_MAX_K,
 *                  M, N < 2^31
 *   y         out  fp32 [M, N], 16-byte aligned
 *   acc       out  optional (may be NULL): int32 [M, N], 16-byte aligned,
 *                  the exact integer products before the rescale
 *
 * Picks a kernel by M: a streaming GEMV for few tokens and a tensor-core GEMM
 * for many.  Either way the result is the same bit for bit.
 */
bl_status bitlinear_forward(const uint8_t* W_packed, const float* gamma, const int8_t* x_q, const float* s,
                            int64_t M, int64_t N, int64_t K, float* y, int32_t* acc, cudaStream_t stream);

/*
 * bitlinear_forward_lut -- bitlinear_forward computed by table lookup instead
 * of conditional adds: the approach that GPU inference of BitNet b1.58 still
 * relies on (promptinjection.net, "4. GPU Support: The Fragile Boost"), kept
 * as a comparison variant.  For every pair of activations of a token, a
 * 16-entry table holds (c0 - 1) x[2p] + (c1 - 1) x[2p+1] for all 4-bit values
 * c0 + 4 c1 of two packed codes; the product is then one lookup and one
 * integer add per two weights.  acc and y are bit-identical to
 * bitlinear_forward.  The weights are read once per token, so the call suits
 * a few tokens (decode).
 *
 *   W_packed, gamma, x_q, s, y, acc   as for bitlinear_forward (y and acc need
 *                                     only 4-byte alignment here)
 *   M, N, K   in   M >= 1, 1 <= N <= 16384 * (number of SMs), K % 64 == 0,
 *                  64 <= K <= BITLINEAR_MAX_K
 *   flags     in   0 or BITLINEAR_RELU2
 *
 * Errors: BL_ERR_INVALID_ARG (null pointer, size < 1, unknown flag),
 * BL_ERR_UNSUPPORTED_SHAPE, BL_ERR_MISALIGNED, BL_ERR_CUDA.
 */
bl_status bitlinear_forward_lut(const uint8_t* W_packed, const float* gamma, const int8_t* x_q, const float* s,
                                int64_t M, int64_t N, int64_t K, float* y, int32_t* acc, unsigned flags,
                                cudaStream_t stream);

/* Flag of bitlinear_quant_forward: W_packed and gamma are NOT written by any
 * work still pending on `stream` (true once the weights are packed and
 * synchronised, as in serving).  The call may then start streaming weights
 * before the preceding kernel on `stream` has finished (programmatic
 * dependent launch); activations are still read only after it completes. */
#define BITLINEAR_WEIGHTS_RESIDENT 1u

/* Flag of bitlinear_quant_forward(_ws): the epilogue writes the squared ReLU
 * y = fp32(max(y,0) * max(y,0)) of the rescaled product: the FFN activation
 * that BitNet b1.58 2B4T uses in place of a gated one (yousumm.com transcript,
 * the paragraph after the poker-chip analogy).  acc, when requested, still
 * holds the raw integer products. */
#define BITLINEAR_RELU2 2u

/* Test hook, not for production use, of bitlinear_quant_forward(_ws) and
 * bitlinear_forward_tq5: the kernels that wait on copies or on other warps
 * start none of the work those waits depend on, so their bounded waits run
 * out (after about two seconds each); every such kernel then records
 * BL_ERR_TIMEOUT in the device error word, writes no y, and exits cleanly.
 * Lets a test exercise every timeout path without faulting or hanging the
 * GPU.  Which kernels stall:
 *   - M <= 4, K <= 32768: the fused quantise + GEMV kernel;
 *   - bitlinear_quant_forward_ws otherwise: the tensor-core GEMM of the route
 *     (fp8, persistent or stream-K);
 *   - bitlinear_quant_forward otherwise: the GEMM, and the quantisation too
 *     where it is the staged kernel (from 256 tokens), whose x_q and s are
 *     then unspecified;
 *   - bitlinear_forward_tq5: the base-3 GEMV. */
#define BITLINEAR_TEST_STALL 0x80000000u

/*
 * bitlinear_quant_forward -- bitlinear_quant_act followed by
 * bitlinear_forward, as one call: per-token absmax int8 quantisation of X
 * (anthology note-168, "What it does": activations at 8 bits) and the
 * ternary x int8 product with the gamma/s rescale.  For M <= 4 and K <= 16384
 * both run in ONE kernel (each CTA quantises the few token rows it needs; the
 * first CTA writes x_q and s out), which removes a launch and a round trip per
 * layer in decode.  For M <= 4 and longer rows (to K = 32768) the per-token
 * quantisation runs first and the GEMV is launched as its programmatic
 * dependent, so that the weight stream starts while the row is quantised.
 * Otherwise it is the two kernels in sequence.  Results are bit-identical to
 * the two separate calls.
 *
 *   W_packed, gamma     in   as for bitlinear_forward
 *   X, dtype            in   as for bitlinear_quant_act
 *   M, N, K             in   as for bitlinear_forward
 *   y                   out  fp32 [M, N], 16-byte aligned
 *   x_q, s              out  int8 [M, K] (16-byte aligned) and fp32 [M] (4-byte
 *                            aligned): the quantised activations and scales
 *   acc                 out  optional int32 [M, N] (may be NULL)
 *   flags               in   0, or BITLINEAR_WEIGHTS_RESIDENT and/or BITLINEAR_RELU2
 */
bl_status bitlinear_quant_forward(const uint8_t* W_packed, const float* gamma, const void* X, bl_dtype dtype,
                                  int64_t M, int64_t N, int64_t K, float* y, int8_t* x_q, float* s, int32_t* acc,
                                  unsigned flags, cudaStream_t stream);

/*
 * bitlinear_forward_workspace_bytes -- device workspace, in bytes, that
 * bitlinear_forward_ws and bitlinear_quant_forward_ws need for an M x K -> N
 * problem: 0 where the streaming GEMV serves it (M <= 4 and K <= 32768),
 * otherwise 2*M*K (the activations expanded once to fp16).
 */
size_t bitlinear_forward_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * bitlinear_forward_ws -- bitlinear_forward with a caller-owned workspace
 * (same product, identical y and acc bit for bit).  For the tensor-core path
 * the int8 activations are expanded to fp16 once per call into the workspace
 * (in the order the MMA consumes them) instead of once per 128-feature tile
 * inside the GEMM, which removes most of the GEMM's operand-conversion work
 * for many tokens.  The product is that of bitlinear_forward (anthology
 * note-168, "The part that is a bet rather than a measurement"; yousumm.com
 * transcript, the paragraph on running the model on graphics cards: weights
 * expanded beside the arithmetic units).
 *
 *   arguments as bitlinear_forward, plus
 *   workspace        tmp  >= bitlinear_forward_workspace_bytes(M, N, K)
 *                         bytes, 16-byte aligned (may be NULL when that is
 *                         0); clobbered; reusable once the call's work on
 *                         `stream` is done
 *   workspace_bytes  in   its size
 *
 * Errors as bitlinear_forward, plus BL_ERR_WORKSPACE if the workspace is
 * missing or too small and BL_ERR_MISALIGNED if it is not 16-byte aligned.
 */
bl_status bitlinear_forward_ws(const uint8_t* W_packed, const float* gamma, const int8_t* x_q, const float* s,
                               int64_t M, int64_t N, int64_t K, float* y, int32_t* acc, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream);

/*
 * bitlinear_quant_forward_ws -- bitlinear_quant_forward with the workspace of
 * bitlinear_forward_ws (used for more than 4 tokens or K > 32768; the fused
 * GEMV path needs none).  Outputs are bit-identical to bitlinear_quant_forward.
 */
bl_status bitlinear_quant_forward_ws(const uint8_t* W_packed, const float* gamma, const void* X, bl_dtype dtype,
                                     int64_t M, int64_t N, int64_t K, float* y, int8_t* x_q, float* s, int32_t* acc,
                                     unsigned flags, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * bitlinear_quant_forward_requant_ws -- bitlinear_quant_forward_ws whose
 * output is also quantised to int8 for the BitLinear that consumes it: every
 * layer of the model takes 8-bit activations (anthology note-168, "What it
 * does"; yousumm.com transcript, the paragraph on the warehouse analogy), and
 * in the FFN the squared-ReLU output of the first BitLinear feeds the second
 * (yousumm.com transcript, the paragraph on the sub-layer norm and squared
 * ReLU).  After the forward, the per-token quantisation kernel reads y back
 * while it is still resident in L2 and writes
 *
 *   s_y[m]    = 127 / max(max_n |y[m,n]|, BITLINEAR_ACT_CLAMP_EPS)
 *   y_q[m,n]  = clip(round(y[m,n] * s_y[m]), -128, 127)
 *
 * which are, bit for bit, bitlinear_quant_act on y (BL_F32).  y, x_q and s
 * are bit-identical to bitlinear_quant_forward_ws.
 *
 *   arguments as bitlinear_quant_forward_ws, without acc, plus
 *   y_q    out  int8 [M, N], 16-byte aligned
 *   s_y    out  fp32 [M], 4-byte aligned
 *   flags  in   0 or BITLINEAR_RELU2 (the squared ReLU is applied before the
 *               maximum is taken, as the next layer sees it)
 *   K % 64 == 0, K <= BITLINEAR_MAX_K.
 *
 * Errors as for bitlinear_quant_forward_ws.  No path of this call applies the
 * RMS norm: the one-call FFN form is bitlinear_rmsnorm_quant_forward_ws.
 */
bl_status bitlinear_quant_forward_requant_ws(const uint8_t* W_packed, const float* gamma, const void* X, bl_dtype dtype,
                                             int64_t M, int64_t N, int64_t K, float* y, int8_t* x_q, float* s,
                                             int8_t* y_q, float* s_y, unsigned flags, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream);

/*
 * bitlinear_rmsnorm_quant_forward_ws -- the second BitLinear of a BitNet FFN
 * in one call: the sub-layer RMS normalisation and per-token quantisation of
 * bitlinear_rmsnorm_quant_act (same x_q and s, bit for bit), then the forward
 * of bitlinear_forward_ws on them (same y and acc, bit for bit).  For more
 * than 4 tokens (or K > 32768) the normalising kernel also writes the
 * tensor-core GEMM's activation operand into the workspace, so the operand
 * needs no separate expansion pass; for up to 4 tokens it is followed by the
 * GEMV on x_q.
 *
 *   W_packed, gamma, y, acc, workspace, workspace_bytes
 *             as for bitlinear_forward_ws (same workspace size)
 *   X         in   [M, K] row-major, BL_BF16 or BL_F32, 16-byte aligned
 *   gain      in   fp32 [K], 16-byte aligned, or NULL for all ones
 *   eps       in   finite, > 0
 *   x_q, s    out  as for bitlinear_quant_act; x_q 16-byte aligned
 *   flags     in   0 or BITLINEAR_RELU2
 *   K % 64 == 0, K <= BITLINEAR_MAX_K.
 *
 * Errors as for bitlinear_forward_ws; BL_ERR_INVALID_ARG also for a bad eps
 * or flag.
 */
bl_status bitlinear_rmsnorm_quant_forward_ws(const uint8_t* W_packed, const float* gamma, const void* X, bl_dtype dtype,
                                             int64_t M, int64_t N, int64_t K, const float* gain, float eps, float* y,
                                             int8_t* x_q, float* s, int32_t* acc, unsigned flags, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream);

/*
 * bitlinear_check_device_error -- waits for `stream`, then reports and clears
 * the library's device error word: BL_ERR_TIMEOUT if a kernel gave up on a
 * bounded wait since the last check, BL_ERR_CUDA if the stream itself failed,
 * BL_OK otherwise.
 */
bl_status bitlinear_check_device_error(cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* bitlinear_status_string(bl_status status);

#ifdef __cplusplus
}
#endif

#endif /* BITLINEAR_H */
