/*
 * bitlinear.h -- C ABI of the BitLinear W1.58A8 forward for NVIDIA B300
 * (sm_103a).  libbitlinear.so exports exactly the functions declared here.
 *
 * The operation (BitNet b1.58; citations name the page and its section):
 *   - Weights are ternarised by their absmean: gamma = mean|W| + 1e-5 (one
 *     fp32 scale per weight tensor), Wq = clip(round(W / gamma), -1, +1).
 *     ["20亿参数仅0.4GB…微软开源全球首个2B参数「原生1.58bit」大模型",
 *     blog.csdn.net/soaring_casia, section 2 "BitLinear层", item 1.]
 *   - Activations are quantised per token by their absmax:
 *     s = 127 / max(max|x_t|, 1e-5), xq = clip(round(x * s), -128, 127).
 *     [same page and section, item 2; "微软AI大模型炸场：0.4GB，CPU就能跑",
 *     blog.csdn.net/2401_84494441, section 1 "激活8位量化".]
 *   - y = (Wq @ xq) accumulated in int32, then y = acc * gamma / s in fp32.
 *     ["BitNet b1.58 深度解析", chenxutan.com, section 2.3(2).]
 *   - A subln RMSNorm precedes the quantised projection; no bias anywhere.
 *     [soaring_casia page, section 2, item 3 and "偏置"; 0.4GB page, section 1
 *     "归一化方法" and section 2 "偏置移除".]
 *   - Weights are stored packed, several 2-bit codes per byte, and unpacked
 *     on chip.  [0.4GB page, section 3 "软硬协同", GPU bullet; 深度解析
 *     page, section 2.1: a 2-bit code has four states, one unused.]
 * Rounding is half to even everywhere; every fp32 step is one IEEE op
 * (divisions are true divisions).  The pages fix none of this; it is the
 * reading this library takes, and the CPU oracle in the repository uses the
 * same one.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless marked (host).  The caller owns
 *     and allocates every buffer, including workspaces; the library allocates
 *     no device memory and holds no per-call state.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous: no call synchronises the host.
 *   - Arguments are checked before anything is enqueued.  On any error the
 *     call returns a non-zero bl_status and enqueues nothing (except
 *     BL_ERR_CUDA, returned when a launch itself fails).  Nothing throws.
 *   - Matrices are row-major and dense (row stride = number of columns).
 *   - Limits: 1 <= N, M <= 2^31 - 1; 1 <= K <= 131072 (|acc| <= 127*K stays
 *     below 2^24, so every partial sum is exact on every path).
 *   - Inputs must be finite.  Results for NaN/Inf inputs are unspecified.
 *
 * Packed weight layout ("bl2" layout):
 *   Row n of an [N, K] ternary matrix occupies row_bytes(K) = 16 * ceil(K/64)
 *   bytes starting at n * row_bytes(K) (K is padded to a multiple of 64
 *   weights with code 1 = weight 0).  Code c = Wq + 1 in {0, 1, 2}.  Weight k
 *   lives in the little-endian 32-bit word w = k / 16 of its row at bit
 *   8*j + 2*i, with i = (k % 16) / 4 and j = k % 4; equivalently in byte
 *   4*w + j at bit 2*i.  So (word >> 2*i) & 0x03030303 holds the codes of
 *   k = 16w+4i .. 16w+4i+3 as four bytes, in order.  Packed buffers must be
 *   16-byte aligned.
 */
#ifndef BITLINEAR_H
#define BITLINEAR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BL_API __attribute__((visibility("default")))
#else
#define BL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bl_status {
  BL_OK = 0,
  BL_ERR_NULL = 1,        /* a required pointer is NULL                      */
  BL_ERR_SHAPE = 2,       /* a size is outside the documented limits        */
  BL_ERR_DTYPE = 3,       /* unknown bl_dtype code                           */
  BL_ERR_ALIGN = 4,       /* a pointer violates its alignment requirement    */
  BL_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than required         */
  BL_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed     */
  BL_ERR_UNSUPPORTED = 7, /* current device is not an sm_103 GPU             */
  BL_ERR_DEVICE = 8       /* a kernel gave up a bounded wait (see below)     */
} bl_status;

typedef enum bl_dtype {
  BL_F32 = 0,  /* IEEE binary32                        */
  BL_BF16 = 1  /* bfloat16 (widened to fp32 exactly)   */
} bl_dtype;

/* Activation applied to x before quantisation (bitlinear_forward_ex,
 * bl_chain_call.act). */
enum { BL_ACT_NONE = 0, BL_ACT_RELU2 = 1 };

/* Library version, e.g. 100 for 0.1.0.  Host only; never fails. */
BL_API int bitlinear_version(void);

/* Static English text for a status code (host).  Never returns NULL. */
BL_API const char *bitlinear_status_string(int status);

/* Packed row length in bytes for K weights: 16 * ceil(K / 64).
 * bytes: host pointer.  Errors: BL_ERR_NULL, BL_ERR_SHAPE. */
BL_API bl_status bitlinear_packed_row_bytes(int64_t K, int64_t *bytes);

/* Size of a whole packed [N, K] matrix: N * row_bytes(K).  Host output. */
BL_API bl_status bitlinear_packed_bytes(int64_t N, int64_t K, size_t *bytes);

/* Workspace needed by bitlinear_pack_weights: 8 * N bytes (one fp64 partial
 * sum per row).  Host output. */
BL_API bl_status bitlinear_pack_workspace_bytes(int64_t N, int64_t K, size_t *bytes);

/* Ternarise and pack a weight matrix (offline step, off the hot path).
 * [soaring_casia page, section 2 "BitLinear层", item 1: absmean weights.]
 *   W       [N, K] of `dtype` (BL_F32 or BL_BF16), device.
 *   packed  [N, row_bytes(K)] uint8 out, device, 16-byte aligned.
 *   gamma   1 float out, device: fl32(fl32(S / (N*K)) + 1e-5f) where S is
 *           sum |W| in fp64, added sequentially over k within each row and
 *           then sequentially over the rows (a fixed, reproducible order).
 *   ws      >= bitlinear_pack_workspace_bytes(N, K) bytes, device, 8-aligned.
 * Codes: Wq = clip(rint(fl32(W / gamma)), -1, 1), stored as Wq + 1.
 * Errors: BL_ERR_NULL, BL_ERR_SHAPE, BL_ERR_DTYPE, BL_ERR_ALIGN,
 * BL_ERR_WORKSPACE, BL_ERR_UNSUPPORTED, BL_ERR_CUDA. */
BL_API bl_status bitlinear_pack_weights(const void *W, int dtype, int64_t N, int64_t K,
                                 uint8_t *packed, float *gamma, void *ws,
                                 size_t ws_bytes, void *stream);

/* bitlinear_pack_weights with one scale per group of group_rows consecutive
 * output rows instead of one per tensor: group_rows = 1 gives a scale per
 * output channel, 128 the groups of the trainable BitLinear.  [深度解析 page,
 * section 5.2 (weight viewed as (-1, group_size, in_features), group_size 128)
 * and section 2.2 (a scale per output feature); the absmean-round quantiser
 * of the per-tensor case is kept, the mean runs over the group's rows.]
 *   group_rows  a power of two that divides N.
 *   gamma       [N / group_rows] floats out, device, 4-byte aligned:
 *               gamma_g = fl32(fl32(S_g / (group_rows*K)) + 1e-5f), S_g the
 *               fp64 sum of |W| over the group's rows (sequential over k in
 *               each row, then over the group's rows in order).
 * Codes: Wq[n,k] = clip(rint(fl32(W[n,k] / gamma_{n / group_rows})), -1, 1).
 * Other arguments and workspace as bitlinear_pack_weights.
 * Errors: as bitlinear_pack_weights; BL_ERR_SHAPE for a group_rows that is
 * not a power of two dividing N. */
BL_API bl_status bitlinear_pack_weights_grouped(const void *W, int dtype, int64_t N, int64_t K,
                                                int64_t group_rows, uint8_t *packed, float *gamma,
                                                void *ws, size_t ws_bytes, void *stream);

/* Per-token absmax int8 quantisation of activations.
 * [soaring_casia page, section 2, item 2; 0.4GB page, section 1 "激活8位量化".]
 *   x      [M, K] of `dtype`, device.
 *   xq     [M, K] int8 out, device: clip(rint(fl32(x * s_m)), -128, 127).
 *   scale  [M] float out, device: s_m = fl32(127 / max(max_k |x_mk|, 1e-5f)).
 * Consumers divide by s (s is the multiplicative quantisation scale).
 * Errors: BL_ERR_NULL, BL_ERR_SHAPE, BL_ERR_DTYPE, BL_ERR_UNSUPPORTED,
 * BL_ERR_CUDA. */
BL_API bl_status bitlinear_quant_act(const void *x, int dtype, int64_t M, int64_t K,
                              int8_t *xq, float *scale, void *stream);

/* Fused subln RMSNorm + per-token absmax int8 quantisation.
 * [soaring_casia page, section 2, item 3 (subln); 0.4GB page, section 1
 * "归一化方法"; no bias (section 2 "偏置").]
 *   x      [M, K] of `dtype`, device.
 *   g      [K] float gain, device, or NULL for a gain of 1.
 *   eps    added to mean(x^2) before the square root (e.g. 1e-5).
 *   xq     [M, K] int8 out: the codes of v = x * r_m * g, computed as the
 *          codes of u = fl32(x * g) (absmax codes do not change under the
 *          positive per-token factor r_m).
 *   scale  [M] float out: s_m = fl32(s_u / r_m), the scale of v, where
 *          r_m = 1 / sqrt(fl32(mean_k x^2) + eps) and s_u is u's absmax
 *          scale.  mean(x^2) is summed in compensated fp32 / fp64 on the GPU,
 *          so r_m (hence s_m) may differ from a sequential fp64 sum by an ulp;
 *          xq does not depend on r_m and is exact.
 * Errors: as bitlinear_quant_act, plus BL_ERR_SHAPE for eps < 0. */
BL_API bl_status bitlinear_rmsnorm_quant_act(const void *x, int dtype, const float *g,
                                      float eps, int64_t M, int64_t K,
                                      int8_t *xq, float *scale, void *stream);

/* Squared ReLU fused with the per-token quantisation: the input of a ReLU^2
 * FFN's down projection, from the up projection's output in one pass.
 * [0.4GB page, section "特殊设计", bullet 激活函数: squared ReLU in the FFN
 * instead of SwiGLU; quantisation as bitlinear_quant_act.]
 *   x      [M, K] of `dtype`, device (e.g. the up projection's y).
 *   xq     [M, K] int8 out: the codes of u = fl32(max(x, 0)^2), as
 *          bitlinear_quant_act computes them for u (all >= 0).
 *   scale  [M] float out: the absmax scale of u.
 * Errors: as bitlinear_quant_act. */
BL_API bl_status bitlinear_relu2_quant_act(const void *x, int dtype, int64_t M, int64_t K,
                                           int8_t *xq, float *scale, void *stream);

/* Workspace (device bytes) needed by bitlinear_forward, bitlinear_forward_q
 * and bitlinear_matmul_i32 for these sizes; 0 when the chosen path needs
 * none (small M).  Host output.  Errors: BL_ERR_NULL, BL_ERR_SHAPE (also for
 * sizes whose launch grid would exceed the device's limits, e.g. more than
 * 65535 token tiles: M beyond about 16.7 million). */
BL_API bl_status bitlinear_workspace_bytes(int64_t M, int64_t N, int64_t K,
                                    size_t *bytes);

/* BitLinear forward: y = (Wq @ quant(x)) * gamma / s, with the activation
 * quantisation fused in.  Equal, bit for bit, to bitlinear_quant_act followed
 * by bitlinear_forward_q.
 * [深度解析 page, section 2.3(2): y = (W_quant @ x_quant) * scale.]
 *   packed [N, row_bytes(K)] packed codes, device, 16-byte aligned.
 *   gamma  1 float, device (as written by bitlinear_pack_weights).
 *   x      [M, K] of `dtype`, device.
 *   y      [M, N] float out, device: y = fl32(float(acc) * c_m) with
 *          c_m = fl32(gamma / s_m), acc = sum_k Wq[n,k] * xq[m,k] (exact int32).
 *   ws     >= bitlinear_workspace_bytes(M, N, K) bytes, device, 256-aligned
 *          (may be NULL when that size is 0).  Calls that share a workspace
 *          must be ordered (same stream or synchronised).
 * Errors: BL_ERR_NULL, BL_ERR_SHAPE, BL_ERR_DTYPE, BL_ERR_ALIGN,
 * BL_ERR_WORKSPACE, BL_ERR_UNSUPPORTED, BL_ERR_CUDA. */
BL_API bl_status bitlinear_forward(const uint8_t *packed, const float *gamma, int64_t N,
                            int64_t K, const void *x, int dtype, int64_t M,
                            float *y, void *ws, size_t ws_bytes, void *stream);

/* BitLinear forward of relu2(x) = fl32(max(x, 0)^2): the down projection of a
 * ReLU^2 FFN, with the activation, its quantisation and the contraction in
 * one call (the squared ReLU is applied where the forward quantises x).
 * Equal, bit for bit, to bitlinear_relu2_quant_act followed by
 * bitlinear_forward_q.  [0.4GB page, section "特殊设计", bullet 激活函数.]
 *   Arguments, workspace and errors as bitlinear_forward. */
BL_API bl_status bitlinear_forward_relu2(const uint8_t *packed, const float *gamma, int64_t N,
                                         int64_t K, const void *x, int dtype, int64_t M,
                                         float *y, void *ws, size_t ws_bytes, void *stream);

/* BitLinear forward with the options of a transformer block: an activation
 * on x before quantisation, a bf16 or fp32 output, and a residual added to the
 * output (the residual stream around every projection: 0.4GB page, section 2
 * architecture; the pages leave the output precision open).
 *   x, x_dtype, M, packed, gamma, N, K, ws   as bitlinear_forward.
 *   act        BL_ACT_NONE, or BL_ACT_RELU2: the forward of relu2(x)
 *              (as bitlinear_forward_relu2).
 *   y          [M, N] of y_dtype (BL_F32 or BL_BF16), device, written:
 *              v = fl32(float(acc) * c_m) as in bitlinear_forward, then
 *              v = fl32(v + residual[m, n]) when residual is given, then one
 *              round-to-nearest-even to bf16 for a bf16 y.
 *   residual   [M, N] of y_dtype, device, or NULL; it may be y itself
 *              (in-place residual update).
 * With act = BL_ACT_NONE, y_dtype = BL_F32 and no residual it is
 * bitlinear_forward.  Errors: as bitlinear_forward, plus BL_ERR_DTYPE for
 * y_dtype and BL_ERR_SHAPE for act. */
BL_API bl_status bitlinear_forward_ex(const uint8_t *packed, const float *gamma, int64_t N,
                                      int64_t K, const void *x, int x_dtype, int64_t M, int act,
                                      void *y, int y_dtype, const void *residual, void *ws,
                                      size_t ws_bytes, void *stream);

/* bitlinear_forward_ex for weights packed by bitlinear_pack_weights_grouped:
 * row n is rescaled by its group's scale, y[m,n] = fl32(float(acc) * c) with
 * c = fl32(gamma_{n / group_rows} / s_m) (one division per output element),
 * then the residual and output dtype as bitlinear_forward_ex.
 *   gamma       [N / group_rows] floats, device, 4-byte aligned.
 *   group_rows  the value the weights were packed with (a power of two
 *               dividing N).
 * Other arguments, workspace and errors as bitlinear_forward_ex; BL_ERR_SHAPE
 * for a group_rows that is not a power of two dividing N. */
BL_API bl_status bitlinear_forward_grouped(const uint8_t *packed, const float *gamma, int64_t group_rows,
                                           int64_t N, int64_t K, const void *x, int x_dtype, int64_t M,
                                           int act, void *y, int y_dtype, const void *residual, void *ws,
                                           size_t ws_bytes, void *stream);

/* BitLinear forward on pre-quantised activations.
 *   xq     [M, K] int8 codes, device;  scale [M] float, device (s_m).
 *   Other arguments and the result as bitlinear_forward. */
BL_API bl_status bitlinear_forward_q(const uint8_t *packed, const float *gamma,
                              int64_t N, int64_t K, const int8_t *xq,
                              const float *scale, int64_t M, float *y, void *ws,
                              size_t ws_bytes, void *stream);

/* The bare ternary x int8 contraction: acc[m, n] = sum_k Wq[n,k] * xq[m,k]
 * as exact int32 (no rescale).  Useful to split K across devices: int32
 * partial sums add exactly, so a K-split needs one integer all-reduce before
 * the rescale.  [0.4GB page, section 1: with ternary weights the matrix
 * product reduces to additions.]
 *   acc    [M, N] int32 out, device.  Other arguments as bitlinear_forward_q. */
BL_API bl_status bitlinear_matmul_i32(const uint8_t *packed, int64_t N, int64_t K,
                               const int8_t *xq, int64_t M, int32_t *acc,
                               void *ws, size_t ws_bytes, void *stream);

/* bitlinear_forward without a workspace argument, for callers that cannot
 * allocate device memory when they call it: code that may only use memory
 * it was handed (a serving engine's fixed memory pool, a plugin interface
 * that passes in only its own tensors), or code that must not call
 * cudaMalloc/cudaFree because those can synchronise the device or are not
 * allowed where it runs.  The pages describe no such variant; it is an
 * addition of this library.
 *   Arguments and result as bitlinear_forward.  The call allocates nothing:
 *   the scratch that larger M needs lives in one fixed 8 MiB array inside
 *   the library's device memory, held by every GPU that loads the library
 *   until the process exits.  Sizes whose scratch
 *   (bitlinear_workspace_bytes(M, N, K)) exceeds 8 MiB return
 *   BL_ERR_WORKSPACE before anything is enqueued: use bitlinear_forward with
 *   a workspace for those (e.g. prefill with M in the thousands).
 *   The first call on a device that needs the scratch looks up the array's
 *   device address on that device (current device); make that first call
 *   before any stream capture.  All calls share the one array: calls that can
 *   run at the same time on the GPU (different streams with no ordering,
 *   several host threads) race on it and give wrong results -- order them.
 *   Each call writes everything it later reads from the array (its split-K
 *   accumulators and tickets are zeroed by its own first kernel), so what an
 *   earlier call left there does not matter.
 * Errors: as bitlinear_forward, with BL_ERR_WORKSPACE meaning "larger than
 * the fixed scratch". */
BL_API bl_status bitlinear_forward_noalloc(const uint8_t *packed, const float *gamma,
                                           int64_t N, int64_t K, const void *x, int dtype,
                                           int64_t M, float *y, void *stream);

/* One call of a decode chain (bitlinear_forward_chain).
 *   packed, gamma  as bitlinear_forward (device).
 *   x              [M, K] of x_dtype, device; with M = 1 it may lie inside an
 *                  earlier call's y.
 *   y              [M, N] float out, device, 4-byte aligned; must not overlap
 *                  this call's x, packed or gamma.
 *   N, K           sizes; N <= 2^30, K <= 32768.
 *   M              tokens, 1..16 (0 counts as 1).  A call of more than one
 *                  token must read an x that no earlier call of the chain
 *                  writes (its input is quantised before the chain starts);
 *                  its y is not passed on by output words.
 *   x_dtype        BL_F32 or BL_BF16.
 *   act            BL_ACT_NONE, or BL_ACT_RELU2 for relu2(x) (as
 *                  bitlinear_forward_relu2).
 *   wait_prev      1 forces every earlier call of the chain to finish before
 *                  this one starts.  The library finds the dependencies
 *                  between calls from their buffers and orders them itself,
 *                  so 0 is always safe; 1 only costs a grid-wide barrier. */
typedef struct bl_chain_call {
  const uint8_t *packed;
  const float *gamma;
  const void *x;
  float *y;
  int64_t N, K;
  int x_dtype;
  int act;
  int wait_prev;
  int M;
} bl_chain_call;

/* Workspace (device bytes) that bitlinear_forward_chain needs for these
 * calls, each part rounded up to 256 bytes:
 *   - 256 bytes of control words;
 *   - 88 bytes per call (the call table, rewritten by every launch);
 *   - a record for every call whose input no earlier call writes and that
 *     does not wait (its input is quantised before the chain starts): a
 *     header (128 bytes for one token, 64 + 64 M rounded up to 128 for more),
 *     then M * 64 * P bytes for each of the row's slabs.  A row of
 *     ceil(K / 64) pieces takes the fewest slabs of at most 65 (M = 1), 31
 *     (M = 2..8) or 23 (M = 9..16) pieces, split evenly with an odd piece
 *     count P per slab, so the codes take M * K bytes and a little more;
 *   - 8 * N bytes for every call whose output a later call reads as its x.
 * Host only; the calls' pointers are compared, not dereferenced.  Errors: as
 * bitlinear_forward_chain's argument checks. */
BL_API bl_status bitlinear_chain_workspace_bytes(const bl_chain_call *calls, int n, size_t *bytes);

/* A decode chain: up to 240 BitLinear forwards of 1 to 16 tokens run in order
 * in one persistent launch (one block per SM, all resident), after a short
 * set-up launch on the same stream (the call table into ws, the inputs no
 * earlier call writes quantised) that the persistent launch overlaps.  Each call's
 * result equals, bit for bit, bitlinear_forward (or bitlinear_forward_relu2)
 * of its x as it stands when the call runs in sequence.
 * The packed weights of later calls stream in while earlier calls compute
 * (the "pack-store-load-unpack-compute" weight stream of the 0.4GB page,
 * section 3, carried across calls).  Dependencies are taken from the buffers:
 *   - x inside an earlier call's fp32 y (that call being the last to write
 *     any of x's bytes): the earlier call also writes its outputs as 8-byte
 *     {value, tag} words into ws and this call reads x from them as soon as
 *     they carry the earlier call's tag -- no barrier;
 *   - any other overlap between a call's inputs and an earlier call's output,
 *     or between its output and an earlier call's inputs or output, and
 *     wait_prev = 1: every block first finishes all earlier calls (a
 *     grid-wide barrier).
 *   calls    host array of n descriptors (copied at the call; 1 <= n <= 240).
 *   ws       >= bitlinear_chain_workspace_bytes(calls, n) bytes, device,
 *            256-byte aligned, ZERO-FILLED before its first use; the library
 *            keeps its contents valid from launch to launch (a sequence
 *            number in the control words makes each launch's tags new).
 *            Chains that share ws must be ordered.  If bitlinear_device_error
 *            reports a failure, zero ws again before reusing it.
 * Errors: BL_ERR_NULL, BL_ERR_SHAPE (n, N, K, M or act out of range, a call
 * whose output overlaps its own inputs, or a call of more than one token
 * whose x an earlier call writes), BL_ERR_DTYPE, BL_ERR_ALIGN,
 * BL_ERR_WORKSPACE, BL_ERR_UNSUPPORTED, BL_ERR_CUDA (including a launch the
 * device cannot fit on all its SMs).
 * [The layer structure: 0.4GB page, section 2 (ReLU^2 FFN, no bias);
 * soaring_casia page, section 2 (BitLinear in every projection).] */
BL_API bl_status bitlinear_forward_chain(const bl_chain_call *calls, int n, void *ws,
                                         size_t ws_bytes, void *stream);

/* Launch overlap (programmatic dependent launch) for the forward kernels.
 * Process-wide; host only.  Modes:
 *   0 (default)  ordinary stream order.
 *   1            kernels may start while the previous kernel on the stream is
 *                still running: they prefetch `packed` and `gamma`, then wait
 *                for it before touching anything else.  Precondition:
 *                `packed` and `gamma` are not written by the kernel launched
 *                immediately before on the same stream.
 *   2            as 1, and a call that runs on the GEMV path (M = 1 with
 *                K <= 65536, M = 2 with K <= 32768, or M = 3..4 with
 *                K <= 16384) does not wait at all: for batches of independent
 *                calls.  Precondition: no
 *                buffer of the call (inputs or output) is written or read by
 *                the kernel launched immediately before it on the same
 *                stream.  Calls on the tensor-core paths behave as in 1.
 * Out-of-range values are clamped to 0..2. */
BL_API void bitlinear_set_launch_overlap(int mode);
BL_API int bitlinear_get_launch_overlap(void);

/* Failure detection.  Every wait inside a kernel is bounded (about 2 s);
 * a kernel that gives up sets a device-side flag, releases what it holds and
 * returns early (its outputs are then invalid).  This reads (and, if
 * `clear`, resets) the flag of the current device.  Synchronous: it waits
 * for the device.  flags: host out, 0 = no error; bit 0 = pipeline wait
 * timed out; bit 1 = a kernel received a launch configuration it cannot run
 * (it skipped its work).  Returns BL_ERR_DEVICE when a flag was set, BL_OK otherwise,
 * BL_ERR_CUDA if the device could not be read. */
BL_API bl_status bitlinear_device_error(unsigned int *flags, int clear);

#ifdef __cplusplus
}
#endif

#endif /* BITLINEAR_H */
