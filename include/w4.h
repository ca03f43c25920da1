/*
 * w4.h -- C ABI of libw4: group-wise int4 weight-only quantization of a
 * linear layer's bf16 weights, and the mixed bf16 x int4 linear that consumes
 * them, on one NVIDIA B300 (sm_103a).
 *
 * The method, as the pages state it:
 *  - a linear layer's weights are quantized once, ahead of time, to int4 in
 *    groups of 32, 64 or 128 (torchao README, "Quick start": quantize_ with
 *    Int4WeightOnlyConfig(group_size=32); torchao guide, section 3.1 "One
 *    line of code for INT4 quantization"; TorchAO 0.14.0 release notes,
 *    "Deprecations", group_size=128), then the quantized layer is called;
 *  - below 8 bits the projection is group-wise affine with an offset ("zero
 *    point") and the integer mapping is torch.round(), i.e. round half to
 *    even (Optimum Quanto, "Design overview / Tensors");
 *  - groups run along the first axis, the output features (Optimum Quanto,
 *    "Design overview / Modules"), so for W[N,K] a group is g consecutive k
 *    of one output row n;
 *  - bias is not quantized (same section): w4_linear_bias adds it in fp32;
 *  - the matmul result is accumulated at higher precision than its inputs
 *    (Optimum Quanto, "Pitfalls when quantizing activations"); bf16 x int4
 *    matmuls are accelerated on CUDA (Optimum Quanto, feature list).
 *
 * Conventions shared by every call:
 *  - bf16 values travel as uint16_t bit patterns;
 *  - every tensor pointer is a DEVICE pointer owned by the caller, 16-byte
 *    aligned, row-major and densely packed; outputs must not alias inputs;
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *    only enqueues work: it returns before the GPU has run it, keeps no state
 *    between calls, never allocates device or pinned memory and never
 *    synchronizes;
 *  - all argument checks happen on the host before any launch; on an error
 *    nothing is written and no CUDA call is made;
 *  - inputs must be finite.  A group whose range (max - min) overflows fp32
 *    (|w| near the bf16 maximum) gives unspecified but non-faulting output;
 *  - a call with N == 0 (or M == 0 for the linear) succeeds with no launch.
 */
#ifndef W4_H
#define W4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W4_API __attribute__((visibility("default")))
#else
#define W4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Packed layout version: plain row-major codes, two per byte with the code of
 * the even k in the low nibble, qparams [N, K/g] bf16 row-major. */
#define W4_FORMAT_VERSION 1

typedef enum w4_status {
    W4_OK = 0,
    W4_ERR_INVALID_ARG = 1,  /* bad size, K % group_size != 0, NULL pointer, overflow */
    W4_ERR_UNSUPPORTED = 2,  /* group_size not in {32, 64, 128} */
    W4_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned */
    W4_ERR_CUDA = 4,         /* a CUDA call failed; see w4_last_error_detail() */
    W4_ERR_TIMEOUT = 5       /* a kernel gave up a bounded wait (w4_device_fault) */
} w4_status;

/* Kernel choice for w4_linear_ex. */
typedef enum w4_kernel {
    W4_KERNEL_AUTO = 0,            /* M <= 32 with a workspace: stream kernels; without one: the pair kernel
                                      for M == 1, the cluster kernel for M <= 32; GEMM above */
    W4_KERNEL_SKINNY = 1,          /* best memory-bound kernel for M <= 32 (stream, else cluster) */
    W4_KERNEL_GEMM = 2,            /* tcgen05 tensor-core GEMM; any M >= 1 */
    W4_KERNEL_SKINNY_CLUSTER = 3,  /* cluster split-K skinny kernel, M <= 32, no workspace */
    W4_KERNEL_STREAM = 4,          /* persistent stream-K kernels, M <= 32, need the workspace:
                                      per-warp units up to 4 tokens, block-shared X from 5 */
    W4_KERNEL_PAIR = 5,            /* one token on pairs of SMs (clusters of two), no workspace:
                                      M == 1, K <= 16384, K / group_size a multiple of 8 */
    W4_KERNEL_TC_DECODE = 6        /* M <= 32 on the tcgen05 tensor cores: a persistent block per
                                      SM over 128-row x 256-k units; needs the workspace */
} w4_kernel;

/*
 * w4_quantize -- W[N,K] bf16 -> Wq[N,K/2] uint8, scales[N,K/g] bf16,
 * offsets[N,K/g] bf16.
 *
 * For each row n and group j (k in [j*g, (j+1)*g)), with IEEE fp32 arithmetic:
 *   mn, mx = min, max of the group (-0.0 ranks below +0.0)
 *   s32    = (mx - mn) / 15;  s32 = 1e-6 if s32 < 1e-6
 *   s      = bf16(s32) (round to nearest even) -> scales[n, j]
 *   o      = mn (exactly a bf16 value)          -> offsets[n, j]
 *   q      = clamp(round_half_even((w - o) / s), 0, 15)
 *   codes of k = 2p and 2p+1 share byte p of row n; even k in the low nibble.
 * Source: the affine group projection with an offset and torch.round
 * mapping of Optimum Quanto, "Design overview / Tensors"; the formulas are the
 * plainest reading of it (the eps value and coding with the stored bf16 scale
 * are readings).  Results are bit-exact, independent of launch shape, for
 * finite weights (the codes of a group holding an infinity or a NaN are
 * unspecified).
 * Errors: W4_ERR_UNSUPPORTED (group_size), W4_ERR_INVALID_ARG (K <= 0,
 * N < 0, K % group_size, NULL, N*K >= 2^62), W4_ERR_MISALIGNED, W4_ERR_CUDA.
 */
W4_API w4_status w4_quantize(const uint16_t *W, int64_t N, int64_t K, int group_size,
                      uint8_t *Wq, uint16_t *scales, uint16_t *offsets,
                      void *stream);

/*
 * w4_dequantize -- W_out[n,k] = bf16(fp32(q) * s + o): one exact fp32
 * product, one fp32 add, one rounding to bf16 (round to nearest even).
 * Bit-exact.  Source: Optimum Quanto, "Pitfalls when quantizing
 * activations" (the quantized result is brought back to float).
 * Errors as w4_quantize.
 */
W4_API w4_status w4_dequantize(const uint8_t *Wq, const uint16_t *scales,
                        const uint16_t *offsets, int64_t N, int64_t K,
                        int group_size, uint16_t *W_out, void *stream);

/*
 * w4_linear_workspace_bytes -- workspace bytes for this problem: what
 * w4_linear needs to run the persistent stream-K decode kernel (M <= 32 and
 * K/group_size even; without it the call still works on the cluster split-K
 * kernel, usually slower), and what w4_linear_repacked needs (M <= 32).
 * Both need one slot of 16 x M 8-byte words per warp of their grid, at most
 * one warp per 16-row x 256-k unit and at most 4096 warps (8192 with one
 * token, whose warps each stream 32-row units on large problems):
 * min(ceil(N/16) * ceil(K/256), M == 1 ? 8192 : 4096) * 128 * M bytes.
 * With 5 to 32 tokens the stream-K work is done by 4-warp blocks that share
 * one staged slice of X (64-row units); their grid is further capped so that
 * each of its warps still has such a slot.
 * M > 32 (the tcgen05 GEMM): 0, or, when the last round of 128-row x
 * 256-token tiles on this device's SMs is part-empty and splitting it pays,
 * 16 MiB + 128 KB per SM (flags in the first 16 MiB, fp32 partial tiles
 * after; the GEMM splits only with that much room).
 */
W4_API size_t w4_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int group_size);

/*
 * w4_linear -- Y[M,N] bf16 = X[M,K] bf16 . dequant(Wq, scales, offsets)^T,
 * products and sums in fp32, one rounding to bf16 at the end, no bias.
 * Source: the mixed bf16 x int4 matmul of Optimum Quanto (feature list and
 * "Pitfalls when quantizing activations": accumulation in fp32).
 *
 * Kernel choice: M <= 32 with a workspace of w4_linear_workspace_bytes runs
 * the persistent stream-K decode kernels (one 16- or 32-row unit per warp
 * step up to 4 tokens; from 5 tokens 64-row units whose X slice a block
 * stages once for its four warps).  Without a workspace (NULL, 0) one token
 * runs the SM-pair kernel (thread-block clusters of two that split K and add
 * their partial sums in shared memory; K <= 16384 and K / group_size a
 * multiple of 8), other M <= 32 the cluster split-K skinny kernel; larger M
 * the tcgen05 tensor-core GEMM (persistent, one block per SM; with a large
 * enough workspace the last round of tiles is split by k blocks between the
 * blocks, deterministically).  The workspace arguments extend the plain
 * (X, M, K, Wq, scales, offsets, N, group_size, Y, stream) call: passing none
 * gives that call exactly, at a speed cost that is moderate with one token
 * (the 224 one-token Llama-3-8B linears take about 1.29x the time) and larger
 * with 2 to 32 tokens (the cluster kernel: 2 to 5x).  The kernels
 * dequantize each weight as bf16(q * s + o) with a single rounding, which can
 * differ from w4_dequantize's double rounding by one bf16 ulp; the stream
 * kernel with one token does not round the weights at all: it sums
 * (128 + q) x per 32-k slice on the tensor cores and adds
 * s (sum - 128 sum x) + o sum x in fp32.  The summation order is each
 * kernel's own.  Accuracy contract against
 * y_ref = sum_k X[m,k] W'[n,k] in fp64 (W' = w4_dequantize output):
 *   |y - y_ref| <= 4e-3 |y_ref| + 1e-2 rms(y_ref).
 * Every kernel is deterministic bit for bit on a given GPU: the stream
 * kernels add the partial sums of a row tile split between warps (or
 * blocks) in a fixed order (the split depends on the GPU's SM count).
 *
 * workspace: caller-owned device memory of `workspace_bytes` bytes (NULL with
 * 0 is allowed).  It must be zero-filled once before its first use.  Its
 * first 16 MiB hold flags and split-tile slots, and every call returns them to
 * zero, so one workspace serves calls of any shape in sequence.  Past 16 MiB
 * (prefill shapes whose last round of tiles is split, w4_linear_workspace_bytes
 * > 16 MiB) the tensor-core GEMM keeps fp32 partial tiles, which it writes
 * before it reads them and leaves behind.  Without that room the GEMM computes
 * whole tiles only.  Calls that may run at the same time on the GPU must not
 * share a workspace.
 * Kernels of consecutive w4_linear calls on one stream may overlap (the next
 * one starts streaming its weights while the previous one finishes); each
 * still reads X, and touches Y and the workspace, only after everything
 * earlier on the stream has completed, so the weights of a call must not be
 * written by the call just before it.
 * Errors as w4_quantize, plus W4_ERR_INVALID_ARG for M < 0.
 */
W4_API w4_status w4_linear(const uint16_t *X, int64_t M, int64_t K, const uint8_t *Wq,
                           const uint16_t *scales, const uint16_t *offsets, int64_t N,
                           int group_size, uint16_t *Y, void *workspace,
                           size_t workspace_bytes, void *stream);

/* w4_linear with an explicit kernel choice (tests and benchmarks use it to
 * run every kernel on the same problem).  A choice that cannot run the
 * problem (M too large, workspace too small) gives W4_ERR_INVALID_ARG. */
W4_API w4_status w4_linear_ex(const uint16_t *X, int64_t M, int64_t K,
                              const uint8_t *Wq, const uint16_t *scales,
                              const uint16_t *offsets, int64_t N, int group_size,
                              uint16_t *Y, void *workspace, size_t workspace_bytes,
                              w4_kernel kernel, void *stream);

/*
 * w4_linear_bias -- w4_linear with the layer's bias: Y[m,n] = bf16(sum_k
 * X[m,k] w'[n,k] + bias[n]), the bias added to the fp32 sum before the one
 * rounding to bf16.  Source: Optimum Quanto, "Design overview / Modules": a
 * quantized module quantizes its weights, and its bias is not quantized (it
 * stays in float).  bias: [N] bf16 (bit patterns), a device pointer, 2-byte
 * aligned; NULL gives exactly w4_linear.  Kernel choice, workspace rules,
 * accuracy contract (with y_ref = sum_k X[m,k] W'[n,k] + bias[n] in fp64) and
 * errors as w4_linear / w4_linear_ex (W4_ERR_MISALIGNED for an odd bias
 * address).
 */
W4_API w4_status w4_linear_bias(const uint16_t *X, int64_t M, int64_t K, const uint8_t *Wq,
                                const uint16_t *scales, const uint16_t *offsets, int64_t N,
                                int group_size, const uint16_t *bias, uint16_t *Y, void *workspace,
                                size_t workspace_bytes, void *stream);
W4_API w4_status w4_linear_bias_ex(const uint16_t *X, int64_t M, int64_t K, const uint8_t *Wq,
                                   const uint16_t *scales, const uint16_t *offsets, int64_t N,
                                   int group_size, const uint16_t *bias, uint16_t *Y, void *workspace,
                                   size_t workspace_bytes, w4_kernel kernel, void *stream);

/*
 * int8 dynamic activations x int4 weights.  Source: torchao README "Training /
 * QAT" and torchao guide (QAT; edge deployment): Int8DynamicActivationInt4-
 * WeightConfig quantizes a linear's activations to int8 at run time and its
 * weights to int4 in groups; Optimum Quanto, "Design overview / Modules" and
 * "Pitfalls when quantizing activations": activations are quantized
 * symmetrically with one scale per tensor, the integer product is accumulated
 * wider than its inputs and brought back to float, then the float bias added.
 *
 * w4_quantize_activation_i8 -- X [M][K] bf16 -> Xq [M][K] int8 and x_scale (fp32):
 *   a = max |x| over the tensor (per_token = 0: one scale, x_scale[0]) or over
 *   each row (per_token = 1: x_scale[m]);  s = a / 127 (fp32 IEEE division, at
 *   least 1e-6);  Xq = clamp(rne(x / s), -127, 127) (fp32 IEEE division, round
 *   half to even).  Bit-exact against the reference.
 * K: a positive multiple of 32; M >= 0 (0: nothing is launched).  X, Xq: 16-byte
 * aligned; x_scale: 4-byte aligned.  workspace: per tensor with M > 1, at least
 * w4_quantize_activation_workspace_bytes (16-byte aligned, any contents, used
 * as scratch); otherwise it may be NULL.  Errors: W4_ERR_INVALID_ARG,
 * W4_ERR_MISALIGNED, W4_ERR_CUDA.
 */
W4_API size_t w4_quantize_activation_workspace_bytes(int64_t M, int64_t K, int per_token);
W4_API w4_status w4_quantize_activation_i8(const uint16_t *X, int64_t M, int64_t K, int per_token,
                                           int8_t *Xq, float *x_scale, void *workspace,
                                           size_t workspace_bytes, void *stream);

/*
 * w4_linear_i8 -- the linear on int8 activation codes and 4-bit weights (the
 * layout of w4_quantize):
 *   Y[m,n] = bf16( s_x(m) * sum_j (s_j I_j + o_j S_j) + bias[n] ),
 *   I_j = sum_{k in group j} Xq[m,k] q[n,k],  S_j = sum_{k in group j} Xq[m,k],
 * s_x(m) = x_scale[m] (per_token = 1) or x_scale[0] (per_token = 0), bias [N]
 * bf16 or NULL.  The codes are exact in bf16, so the kernels run the bf16
 * tensor-core path on them: with at most 4 tokens they read Xq directly and
 * sum (128 + q) Xq over 16-k slices, exactly in fp32 (every partial sum is an
 * integer below 2^24); with more, the codes are widened to bf16 in the
 * workspace and the weights dequantized to bf16 as in w4_linear.  s_x, the
 * group's scale and offset and the bias are applied in fp32, rounded once.
 * Accuracy: |y - y_ref| <= 4e-3 |y_ref| + 1e-2 rms(y_ref), y_ref the fp64
 * value above.
 * workspace: w4_linear_i8_workspace_bytes(M, N, K, g) bytes, 16-byte aligned,
 * zero-filled once before the first use.  Its first 16 MiB hold the kernels'
 * split-tile slots (as for w4_linear; every call leaves them at zero); calls
 * with more than 4 tokens also write the codes widened to bf16 after them
 * (scratch, 2 M K bytes from 16 MiB on).  So one workspace serves int8 and
 * bf16 calls of any shape in sequence.  Other arguments and errors as
 * w4_linear_bias; x_scale 4-byte aligned.
 */
W4_API size_t w4_linear_i8_workspace_bytes(int64_t M, int64_t N, int64_t K, int group_size);
W4_API w4_status w4_linear_i8(const int8_t *Xq, const float *x_scale, int per_token, int64_t M,
                              int64_t K, const uint8_t *Wq, const uint16_t *scales,
                              const uint16_t *offsets, int64_t N, int group_size,
                              const uint16_t *bias, uint16_t *Y, void *workspace,
                              size_t workspace_bytes, void *stream);

/*
 * w4_linear_i8_dynamic -- w4_quantize_activation_i8 and w4_linear_i8 in one call,
 * on bf16 X [M][K]: Y is bit for bit what the two calls give (the same codes,
 * scales and sums), without the codes leaving the GPU.  With at most 4 tokens
 * one kernel does both: each of its blocks finds X's largest magnitude (of the
 * tensor, or of each token with per_token = 1) while its first weights are on
 * their way, then codes X as it stages it.  With more tokens, or a group count
 * the stream kernel does not take, the two steps run in turn with the codes in
 * the workspace.  workspace: w4_linear_i8_dynamic_workspace_bytes(M, N, K, g)
 * bytes, 16-byte aligned, zero-filled once before the first use (its first
 * 16 MiB as for w4_linear_i8; the rest is scratch).  Other arguments, accuracy
 * and errors as w4_linear_i8 (X 16-byte aligned).
 */
W4_API size_t w4_linear_i8_dynamic_workspace_bytes(int64_t M, int64_t N, int64_t K, int group_size);
W4_API w4_status w4_linear_i8_dynamic(const uint16_t *X, int per_token, int64_t M, int64_t K,
                                      const uint8_t *Wq, const uint16_t *scales, const uint16_t *offsets,
                                      int64_t N, int group_size, const uint16_t *bias, uint16_t *Y,
                                      void *workspace, size_t workspace_bytes, void *stream);

/* Sizes of the packed outputs: N*K/2 bytes of codes, N*(K/g)*2 bytes for each
 * of scales and offsets.  0 for invalid arguments. */
W4_API size_t w4_packed_bytes(int64_t N, int64_t K);
W4_API size_t w4_qparam_bytes(int64_t N, int64_t K, int group_size);

/*
 * w4_device_fault -- synchronizes `stream`, then reports whether any libw4
 * kernel on the current device gave up a bounded wait since the last call
 * (W4_ERR_TIMEOUT), and clears the flag.  Kernels that time out set the flag,
 * release what they hold and return; their outputs are then undefined, and a
 * workspace they used must be zero-filled again before its next use.  W4_OK
 * from w4_linear (or any call) only means the work was enqueued: it does not
 * cover a wait that gives up later, which only this call reports.
 * (include/w4_selftest.h has a hook that makes the waits run out on purpose.)
 */
W4_API w4_status w4_device_fault(void *stream);

/* Human-readable text of a status, and the detail (CUDA error string, failed
 * check) of the last failing call on this host thread. */
W4_API const char *w4_status_string(w4_status s);
W4_API const char *w4_last_error_detail(void);

/* W4_FORMAT_VERSION of the built library. */
W4_API int w4_format_version(void);

/* Bytes of the device array w4_linear_static uses as its workspace. */
#define W4_STATIC_SCRATCH_BYTES (4u << 20)

/*
 * w4_linear_static -- w4_linear for callers that cannot allocate device
 * memory.  The pages have no counterpart: this is an interface convenience,
 * not part of the method.
 *
 * Some callers may not call cudaMalloc or any allocating routine (a plugin
 * inside another framework that owns every device allocation, a service with
 * a fixed device-memory budget reserved up front), yet the persistent
 * stream-K decode kernel needs a workspace.  This entry point runs that kernel
 * with, as workspace, a W4_STATIC_SCRATCH_BYTES (4 MiB) array that libw4 keeps
 * in device memory: every GPU that loads the library holds it until the
 * process exits.  The call itself allocates nothing.  Inputs and outputs are
 * the caller's, as for w4_linear.
 *
 * Limits: M <= 8 and K / group_size even (the workspace such a call needs,
 * at most 4096 * 128 * 8 bytes, always fits the array); other sizes fail with
 * W4_ERR_INVALID_ARG and a message in w4_last_error_detail().
 * Set-up: the first call on each device, with that device current, looks up
 * the array's device address (cudaGetSymbolAddress); make that first call
 * before any stream capture.  With lazy module loading (the CUDA default) the
 * library's device code, and with it the array, is loaded at that first call:
 * the first call on a device is where the 4 MiB are set aside, and it can fail
 * with W4_ERR_CUDA when device memory is short (w4_last_error_detail() has the
 * CUDA error).  Later calls on that device allocate nothing.
 * Every call clears the part of the array it uses (an asynchronous memset on
 * `stream`) and then shares the one array with every other call on the same
 * device: calls that overlap on the GPU (different streams) race and give
 * wrong results; serialize them.
 */
W4_API w4_status w4_linear_static(const uint16_t *X, int64_t M, int64_t K,
                                  const uint8_t *Wq, const uint16_t *scales,
                                  const uint16_t *offsets, int64_t N, int group_size,
                                  uint16_t *Y, void *stream);

/*
 * Decode layout -- an optional second arrangement of the same codes, scales
 * and offsets, for the memory-bound decode linear.  The pages name such
 * arrangements without defining them (torchao README "Quick start":
 * `tile_packed_to_4d`; TorchAO 0.14.0 release notes: Int4PreshuffledTensor,
 * Int4TilePackedTo4dTensor): weights are rearranged once, at load time, into
 * the order the kernel reads them.  The canonical row-major arrays above
 * remain the format of record; this layout holds exactly the same numbers.
 *
 * Layout (byte exact).  Rows are cut into tiles of 16 (tile t = rows
 * 16t..16t+15) and each row into units of 256 k (unit c = k 256c..256c+255);
 * units are stored tile-major: unit (t, c) starts at byte
 * (t * ceil(K/256) + c) * U, U = 2048 + 512 * 32 / group_size
 * (2560, 2304, 2176 for g = 32, 64, 128).  Inside a unit:
 *  - bytes 512j + 16l (j = 0..3, l = 0..31; with r = l / 4, q = l % 4) hold
 *    the 32 codes of row 16t + r + 8(j % 2), k from 256c + 128(j / 2) + 32q,
 *    as four little-endian 32-bit words of 8 codes each (word w: k from
 *    256c + 128(j / 2) + 32q + 8w); inside a word, nibble i (bits 4i..4i+3)
 *    holds the code of k0 + 2i for i < 4 and of k0 + 2(i - 4) + 1 for i >= 4
 *    (k0 the word's first k), so that nibbles i and i + 4 are two
 *    consecutive k;
 *  - bytes 2048 + 16p (p = 0 .. 32*32/group_size - 1) hold the eight bf16
 *    qparams that lanes l with l / (group_size / 32) = p use: with
 *    l0 = p * group_size / 32, r = l0 / 4 and q0 = l0 % 4, for h = 0, 1 the
 *    group j_h = (256c + 128h + 32 q0) / group_size of rows a = 16t + r and
 *    b = a + 8, stored as scale_a(h=0), offset_a(h=0), scale_b(h=0),
 *    offset_b(h=0), then the same four for h = 1.
 * Rows >= N, k >= K and groups >= K/group_size hold zeros.
 */
W4_API size_t w4_repacked_bytes(int64_t N, int64_t K, int group_size);

/*
 * w4_repack -- canonical Wq / scales / offsets -> the decode layout above,
 * in `packed` (w4_repacked_bytes(N, K, group_size) bytes, caller-owned
 * device memory, 16-byte aligned, not overlapping the inputs).  Asynchronous
 * on `stream`, allocates nothing.  Errors as w4_dequantize.
 */
W4_API w4_status w4_repack(const uint8_t *Wq, const uint16_t *scales, const uint16_t *offsets,
                           int64_t N, int64_t K, int group_size, uint8_t *packed, void *stream);

/*
 * w4_linear_repacked -- w4_linear for weights in the decode layout, M <= 32:
 * a persistent stream-K decode kernel that loads each 16-row x 256-k unit
 * with five coalesced warp loads straight into registers and reads X through
 * L1.  Same result contract as w4_linear (the same dequantization and fp32
 * accumulation, deterministic like the stream kernel); the workspace rules
 * of w4_linear apply, with
 * w4_linear_workspace_bytes(M, N, K, group_size) bytes required.  M > 32 or
 * a missing workspace give W4_ERR_INVALID_ARG.
 * Where it pays: with 2 to 8 tokens it matches or beats w4_linear on the
 * canonical layout (each lane reads only its own token's X); with one token
 * w4_linear is faster, and from 16 tokens on it is 1.3 to 1.9 times faster,
 * because this kernel reads each unit's X slice once per 16-row tile through L1.
 * Keep the canonical arrays for callers whose batches exceed 8 tokens.
 */
W4_API w4_status w4_linear_repacked(const uint16_t *X, int64_t M, int64_t K, const uint8_t *packed,
                                    int64_t N, int group_size, uint16_t *Y, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * Other code widths on the same affine path.  Optimum Quanto's feature list
 * names int2, int4 and int8 weights; the torchao README quantizes a
 * diffusion transformer to int8 weight-only in groups of 128.  The pages give
 * the widths, not their formulas; libw4 runs the 4-bit method unchanged with
 * L = 2^bits - 1 levels in place of 15:
 *   s = bf16(max(fp32(max - min) / L, 1e-6)),  o = min,
 *   q = clamp(rne((w - o) / s), 0, L),  w' = bf16(fp32(q * s + o)).
 * (At 8 bits the rounding of the scale to bf16, up to 2^-8 relative, can put
 * a group's maximum above L + 1/2; the clamp then makes its code L.)
 * Packed codes: row n holds K * bits / 8 bytes; byte p of a row holds the
 * 8/bits codes k = (8/bits) p .. (8/bits) p + 8/bits - 1, code k at bits
 * bits * (k mod 8/bits) (the lowest k in the lowest bits; at 4 bits this is
 * the w4_quantize layout).  Scales and offsets as for w4_quantize.
 * bits = 4 calls are exactly w4_quantize / w4_dequantize / w4_linear.
 * bits not in {2, 4, 8} give W4_ERR_UNSUPPORTED; other errors as the 4-bit
 * calls.
 */
W4_API size_t w4_packed_bytes_bits(int64_t N, int64_t K, int bits); /* N * K * bits / 8 */

/* Group-wise quantization to `bits`-bit codes: Wq [N][K*bits/8] bytes,
 * scales / offsets [N][K/group_size] bf16.  Bit-exact. */
W4_API w4_status w4_quantize_bits(const uint16_t *W, int64_t N, int64_t K, int group_size,
                                  int bits, uint8_t *Wq, uint16_t *scales, uint16_t *offsets,
                                  void *stream);

/* W_out[n,k] = bf16(fp32(q) * s + o) for `bits`-bit codes.  Bit-exact. */
W4_API w4_status w4_dequantize_bits(const uint8_t *Wq, const uint16_t *scales,
                                    const uint16_t *offsets, int64_t N, int64_t K,
                                    int group_size, int bits, uint16_t *W_out, void *stream);

/*
 * Y[M,N] bf16 = X[M,K] . dequant(Wq)^T for `bits`-bit codes, fp32 sums, one
 * rounding at the end, same accuracy contract as w4_linear.  M <= 32 with K /
 * group_size even and a workspace of w4_linear_workspace_bytes(M, N, K,
 * group_size) bytes runs the persistent stream-K decode kernel with 64-row
 * units; anything else runs the tcgen05 tensor-core GEMM (any M).  8-bit
 * weights enter the products as bf16(fp32(q s + o)), the w4_dequantize_bits
 * value; 2-bit weights as bf16(q s + o) with one rounding.  The workspace
 * rules of w4_linear apply.  2-bit codes need K % 64 == 0 (their rows are
 * then a whole number of 16-byte pieces); other K give W4_ERR_UNSUPPORTED.
 */
W4_API w4_status w4_linear_bits(const uint16_t *X, int64_t M, int64_t K, const uint8_t *Wq,
                                const uint16_t *scales, const uint16_t *offsets, int64_t N,
                                int group_size, int bits, uint16_t *Y, void *workspace,
                                size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* W4_H */
