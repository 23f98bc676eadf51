/*
 * libkaio_qkv -- GB300 (sm_103a) W4A16 fused QKV projection and dense f16
 * tensor-core matmul behind a plain C ABI.
 *
 * Operations follow two docs.rs source pages of the kaio-candle crate:
 *   "kaio-candle -- src/qkv_project_int4.rs" (qkv_project_int4 and its doc
 *   comment: input contract, validation, output dtype), and
 *   "kaio-candle 0.2.0 -- src/matmul_tc_async.rs" (matmul_tc_async:
 *   f16 x f16 -> f32; MatmulTcAsyncOp::bwd: dA = grad @ B^T, dB = A^T @ grad).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE memory on the current CUDA device, owned
 *     by the caller, dense, row-major, with no offset or stride of their own.
 *     The library never allocates or frees them and never keeps them.
 *   - Every tensor pointer must be 16-byte aligned (TMA and 128-bit loads).
 *   - Calls are asynchronous on `stream` (0 = legacy default stream). The
 *     library does not synchronise the host. Outputs are complete when the
 *     stream reaches that point.
 *   - Return value: KAIO_OK (0) or a kaio_status error code; on error nothing
 *     was launched, and kaio_last_error() returns a message for the calling
 *     thread.
 *   - Empty problems (M == 0 or N == 0) return KAIO_OK without a launch, like
 *     the plan launcher of "baracuda-kernels -- src/quantize/
 *     dequantize_per_group_backward.rs" (run returns early when the element
 *     count is zero). K == 0 is an empty sum: the outputs are set to zero.
 *   - The library is forward-only, like the direct-call bridge it mirrors
 *     (gradient-tracked inputs are rejected there). The matmul backward is a
 *     separate entry point.
 *   - Supported device: compute capability 10.3 (GB300). Anything else gives
 *     KAIO_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef KAIO_QKV_H_
#define KAIO_QKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kaio_stream_t; /* same type as cudaStream_t */

typedef enum {
  KAIO_OK = 0,
  KAIO_ERR_INVALID_VALUE = 1,      /* null pointer, bad dimension, overlap, wrong device */
  KAIO_ERR_MISALIGNED = 2,         /* a tensor pointer is not 16-byte aligned */
  KAIO_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
  KAIO_ERR_CUDA = 4,               /* a CUDA runtime call or kernel launch failed */
  KAIO_ERR_DEVICE_TIMEOUT = 5      /* a kernel's bounded wait gave up (see kaio_device_status) */
} kaio_status;

/*
 * W4A16 fused tri-output QKV projection.
 * ("kaio-candle -- src/qkv_project_int4.rs", doc comment of qkv_project_int4.)
 *
 * For p in {q, k, v}:
 *   out_p[m, n] = f16( sum_{k<K} x[m, k] * Wd_p[k, n] ),
 *   Wd_p[k, n]  = RN_f16( int4(W_p[k, n]) * s_p[k / 128, n] ),
 * accumulated in f32, rounded to f16 (nearest even) inside the kernel.
 *
 *   x          f16  [M, K]      activations, shared by the three projections
 *   wq, wk, wv u32  [K/8, N]    packed INT4 weights: nibble i (bits 4i..4i+3) of
 *                               word [r, n] is the signed two's-complement
 *                               weight of K-row 8r+i, column n (range [-8, 7])
 *   sq, sk, sv f16  [K/128, N]  one scale per group of 128 K-rows and column
 *   q, k, v    f16  [M, N]      outputs; every element is written
 *
 * Errors (KAIO_ERR_INVALID_VALUE unless noted): a null pointer; K not a
 * multiple of 128 (the group size is locked at 128); N not a multiple of 8;
 * an output overlapping an input or another output; a pointer not on the
 * current device; misaligned pointer (KAIO_ERR_MISALIGNED).
 *
 * Path: M <= 16 runs the tcgen05 decode kernel (K split across the CTAs of a
 * thread-block cluster, partial sums reduced in distributed shared memory);
 * M >= 17 runs the tcgen05 tile kernel. Neither allocates device memory.
 */
int kaio_qkv_project_int4(const void* x, const uint32_t* wq, const uint32_t* wk,
                          const uint32_t* wv, const void* sq, const void* sk, const void* sv,
                          void* q, void* k, void* v, uint32_t M, uint32_t N, uint32_t K,
                          kaio_stream_t stream);

/*
 * kaio_qkv_project_int4 for decode-sized M (0..16) without any device memory
 * allocation by the library. The pages have no counterpart of this entry: it
 * exists for callers that cannot allocate device memory themselves or let a
 * library do it -- engines and plugin hosts that own every byte of device
 * memory and forbid cudaMalloc, processes whose memory is fully reserved up
 * front, and latency-critical paths that cannot take an allocation's implicit
 * synchronisation or failure.
 *
 * Same arguments, layouts, results and errors as kaio_qkv_project_int4, with
 * these differences:
 *   - M must be <= 16 (it runs a stream-K decode kernel that spreads the
 *     weight stream evenly over every SM and finishes split column groups
 *     through a global-memory scratch); larger M is rejected with
 *     KAIO_ERR_INVALID_VALUE.
 *   - The kernel's split-K scratch (group counters and partial sums) lives in
 *     one fixed 8 MiB array inside the library; every GPU that loads the
 *     library holds it until the process exits. N is limited to 3*ceil(N/256)
 *     <= 16384 column groups (N <= 1,398,016); larger N is rejected with
 *     KAIO_ERR_INVALID_VALUE.
 *   - All calls share that array. Calls whose kernels overlap on the GPU (for
 *     example on two streams with no ordering between them) race on it and
 *     produce wrong results: issue them in order on one stream. Each call
 *     clears the counters it needs (cudaMemsetAsync on `stream`) before its
 *     kernel.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) and keeps it for the life of the process; make
 *     that first call before any stream capture. A device reset
 *     (cudaDeviceReset, or anything else that destroys the device's primary
 *     context) is not supported: do not call this entry point again in a
 *     process after one.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 */
int kaio_qkv_project_int4_noalloc(const void* x, const uint32_t* wq, const uint32_t* wk,
                                  const uint32_t* wv, const void* sq, const void* sk,
                                  const void* sv, void* q, void* k, void* v, uint32_t M,
                                  uint32_t N, uint32_t K, kaio_stream_t stream);

/*
 * Test entry for the bounded waits of the decode kernel (the failure detection
 * of "baracuda-kernels -- src/quantize/dequantize_per_group_backward.rs",
 * run -> map_status: a failure surfaces as a status, never as a hang).
 *
 * Runs the kernel kaio_qkv_project_int4 runs for M <= 16, with every wait of
 * its pipeline limited to wait_limit_ns instead of 2 s. With a limit shorter
 * than the pipeline's hand-offs (0 makes the first wait that finds its phase
 * incomplete give up), the kernel records a timeout in the device error word,
 * lets the copies and MMAs already in flight finish, frees its tensor memory
 * and returns; the outputs are then undefined. The next kaio_device_status()
 * reports KAIO_ERR_DEVICE_TIMEOUT and clears the word; the context stays
 * usable. Arguments and errors as kaio_qkv_project_int4, with 1 <= M <= 16,
 * K and N positive.
 */
int kaio_debug_decode_wait_limit(const void* x, const uint32_t* wq, const uint32_t* wk,
                                 const uint32_t* wv, const void* sq, const void* sk,
                                 const void* sv, void* q, void* k, void* v, uint32_t M,
                                 uint32_t N, uint32_t K, uint64_t wait_limit_ns,
                                 kaio_stream_t stream);

/*
 * W8A16 fused tri-output QKV projection, the INT8 sibling of
 * kaio_qkv_project_int4. ("kaio-candle -- src/qkv_project_int4.rs", module
 * doc: the INT4 op follows the INT8 op's direct-call pattern but takes seven
 * tensors, three of them group scales; both return f16 converted in-kernel
 * from f32.) The pages show no more of the INT8 op; this entry states its
 * contract as the INT4 layout with 8-bit fields and no group-scale tensors:
 *
 * For p in {q, k, v}:
 *   out_p[m, n] = f16( scale_p * sum_{k<K} x[m, k] * int8(W_p[k, n]) ),
 * products and sum in f32 (exact int8 -> f16 operands on the tensor cores),
 * the scale applied to the f32 sum, rounded to f16 (nearest even) in-kernel.
 *
 *   x          f16  [M, K]      activations, shared by the three projections
 *   wq, wk, wv u32  [K/4, N]    packed INT8 weights: byte i (bits 8i..8i+7) of
 *                               word [r, n] is the signed two's-complement
 *                               weight of K-row 4r+i, column n ([-128, 127])
 *   scale_q, scale_k, scale_v   f32 by value: one scale per projection
 *   q, k, v    f16  [M, N]      outputs; every element is written
 *
 * Errors (KAIO_ERR_INVALID_VALUE unless noted): a null pointer; K not a
 * multiple of 128 (the kernels' K group); N not a multiple of 8; an output
 * overlapping an input or another output; a pointer not on the current
 * device; misaligned pointer (KAIO_ERR_MISALIGNED). Scales are not checked:
 * an infinite or NaN scale gives infinite or NaN outputs.
 *
 * Path: M <= 16 runs the tcgen05 decode kernel (split over K across a
 * thread-block cluster; no workspace, no allocation); larger M runs the
 * tcgen05 tile kernel. Both read the caller's buffers only.
 */
int kaio_qkv_project_int8(const void* x, const uint32_t* wq, const uint32_t* wk, const uint32_t* wv,
                          float scale_q, float scale_k, float scale_v, void* q, void* k, void* v,
                          uint32_t M, uint32_t N, uint32_t K, kaio_stream_t stream);

/*
 * Dense tensor-core matmul C = A @ B.
 * ("kaio-candle 0.2.0 -- src/matmul_tc_async.rs", module doc and
 * MatmulTcAsyncOp::cuda_fwd: f16 x f16 -> f32, inner dimensions must match.)
 *
 *   a  f16 [M, K],  b  f16 [K, N],  c  f32 [M, N] (output, every element written)
 *
 * Errors: null pointer; K or N not a multiple of 8 (16-byte row strides);
 * c overlapping a or b; pointer not on the current device; misalignment.
 */
int kaio_matmul_tc(const void* a, const void* b, float* c, uint32_t M, uint32_t N, uint32_t K,
                   kaio_stream_t stream);

/*
 * Backward of C = A @ B for an upstream gradient G = dL/dC.
 * ("kaio-candle 0.2.0 -- src/matmul_tc_async.rs", MatmulTcAsyncOp::bwd:
 * dA = grad @ B^T, dB = A^T @ grad.)
 *
 *   a  f16 [M, K],  b  f16 [K, N],  g  f16 [M, N]
 *   da f32 [M, K]  = G @ B^T      (output)
 *   db f32 [K, N]  = A^T @ G      (output)
 *
 * The transposes are never materialised: the kernels read B and A in the
 * other major order. The page's bridge casts grad to f16 before and the
 * results to f16 after; here g is f16 on entry and da/db are f32 (cast them
 * if an f16 result is wanted).
 * Errors: as kaio_matmul_tc (K and N multiples of 8), and any output
 * overlapping an input or the other output.
 */
int kaio_matmul_tc_backward(const void* a, const void* b, const void* g, float* da, float* db,
                            uint32_t M, uint32_t N, uint32_t K, kaio_stream_t stream);

/*
 * kaio_matmul_tc with the result rounded to f16 in the kernel's epilogue
 * (round-to-nearest-even of the f32 accumulator): c f16 [M, N]. The page's
 * bridge casts matmul results to f16 afterwards ("kaio-candle 0.2.0 --
 * src/matmul_tc_async.rs", MatmulTcAsyncOp::bwd, the casts of grad_a and
 * grad_b to the input dtype); fusing the cast saves a pass over C.
 * Arguments and errors: as kaio_matmul_tc, with c 16-byte aligned f16.
 */
int kaio_matmul_tc_f16(const void* a, const void* b, void* c, uint32_t M, uint32_t N, uint32_t K,
                       kaio_stream_t stream);

/*
 * kaio_matmul_tc_backward with da f16 [M, K] and db f16 [K, N], each rounded
 * from its f32 accumulator in the kernel (the page casts both to f16 after
 * its matmuls, "kaio-candle 0.2.0 -- src/matmul_tc_async.rs",
 * MatmulTcAsyncOp::bwd). Arguments and errors: as kaio_matmul_tc_backward.
 */
int kaio_matmul_tc_backward_f16(const void* a, const void* b, const void* g, void* da, void* db,
                                uint32_t M, uint32_t N, uint32_t K, kaio_stream_t stream);

/* Element types of the per-group dequantisation entry points. bf16 values are
 * passed as their 16-bit patterns. */
typedef enum {
  KAIO_DTYPE_F32 = 0,
  KAIO_DTYPE_F64 = 1,
  KAIO_DTYPE_F16 = 2,
  KAIO_DTYPE_BF16 = 3,
  KAIO_DTYPE_S8 = 4,
  KAIO_DTYPE_U8 = 5
} kaio_dtype;

/*
 * Straight-through backward of the per-group dequantisation
 * ("baracuda-kernels -- src/quantize/dequantize_per_group_backward.rs",
 * module doc and DequantizePerGroupBackwardPlan):
 *
 *   dx[i, j] = dy[i, j] * scale[i, j / group]
 *
 *   dy, dx  dtype [outer, axis], row-major        dtype: F32, F64, F16 or BF16
 *   scale   dtype [outer, axis / group]            (groups along the last axis)
 *   q_dtype the forward's quantised type, S8 or U8 (checked, as the page's
 *           plan does; it does not change the result)
 * Each product is rounded once to dtype (deterministic, bit-stable). dx may be
 * dy itself (in place); no other overlap is allowed. All pointers are device
 * memory of the current device owned by the caller, aligned to their element
 * size. Asynchronous on `stream`.
 * Errors: KAIO_ERR_INVALID_VALUE for an unsupported dtype or q_dtype, negative
 * outer or axis, group <= 0, axis not a multiple of group, a null pointer,
 * overlap, memory not on the current device; KAIO_ERR_MISALIGNED; an empty
 * problem (outer * axis == 0) returns KAIO_OK without launching.
 */
int kaio_dequantize_per_group_backward(int dtype, int q_dtype, int32_t outer, int32_t axis, int32_t group,
                                       const void* dy, const void* scale, void* dx, kaio_stream_t stream);

/*
 * The per-group dequantisation itself: out[i, j] = dtype(q[i, j]) *
 * scale[i, j / group], q int8 (S8) or uint8 (U8) [outer, axis], no zero point.
 * The page names this plan (DequantizePerGroupPlan, whose backward is above)
 * but does not show it; this is the plainest reading of its backward's
 * straight-through definition. Arguments, layout, rounding and errors as the
 * backward, with q in place of dy (no overlap with out allowed).
 */
int kaio_dequantize_per_group(int q_dtype, int dtype, int32_t outer, int32_t axis, int32_t group,
                              const void* q, const void* scale, void* out, kaio_stream_t stream);

/*
 * Dequantise packed INT4 weights to f16, exactly as the projection kernels do
 * before their multiply: out[k, n] = RN_f16(int4(W[k, n]) * s[k/128, n]).
 * A test entry for bit-exact comparison of the dequant stage.
 *
 *   w  u32 [K/8, N],  s  f16 [K/128, N],  out  f16 [K, N]
 *   variant 0: the K-row-order routine of the tile kernel (M >= 17)
 *   variant 1: the decode kernel's general, paired-nibble routine (M <= 16)
 *   variant 2: the decode kernel's two-instruction routine (one LOP3 and one
 *              f16x2 FMA per pair) wherever the word's scale s lies in
 *              0 < s <= 65504 * 2^-20, the paired-nibble routine elsewhere
 *              (the decode kernel takes it when all three scales of a warp's
 *              32 columns are in range)
 * Errors: as kaio_qkv_project_int4 for K and N; variant not 0, 1 or 2.
 */
int kaio_dequant_int4_debug(const uint32_t* w, const void* s, void* out, uint32_t K, uint32_t N,
                            int variant, kaio_stream_t stream);

/* Which kernel kaio_qkv_project_int4 uses for a given M: 0 = decode
 * (weight-streaming, M <= 16), 1 = tcgen05 tensor-core kernel. */
int kaio_qkv_path(uint32_t M);

/* Message describing the last error returned on the calling thread ("" if
 * none). The pointer stays valid until the thread's next call. */
const char* kaio_last_error(void);

/* Synchronises the current device, then reads and clears the kernels' device
 * error word. Returns KAIO_OK, KAIO_ERR_DEVICE_TIMEOUT if a kernel gave up a
 * bounded wait since the last query, or KAIO_ERR_CUDA if the device reports
 * an error. */
int kaio_device_status(void);

/* Static, human-readable name of a kaio_status value. */
const char* kaio_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* KAIO_QKV_H_ */
