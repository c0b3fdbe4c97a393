/*
 * pq.h -- C ABI of the block-quantized mat-vec library for GB300 (sm_103a).
 *
 * The operation: the decode-step mat-vec y = W x with W kept in
 * block-quantized form and decoded inside the kernel, so that no f32 copy of
 * W is ever made (ember pull request "Project scaffold: modules, CLI, and
 * correctness harness", quant.rs description); the mat-vec is the row-major
 * one that costs the most in a decode step (same page, tensor.rs
 * description).  The block formats are the K-family and Q8_0 formats whose
 * decoding the PESTI README ("What This Is", "Architecture") reports as
 * exact to the byte, plus the per-row symmetric int8 and int4 formats of the
 * ember page.  The inferno README ("Design notes") fixes the boundary
 * style: contiguous row-major buffers in and out.
 *
 * Layouts (all little-endian; the pages print none, these are the public
 * GGUF layouts read as a byte specification):
 *   PQ_Q8_0   34 B per 32 weights: f16 d, int8 q[32].        w = d*q
 *   PQ_Q4_K  144 B per 256 weights: f16 d, f16 dmin, 12 B of packed 6-bit
 *            (scale, min) pairs for 8 sub-blocks of 32, 128 B of 4-bit q.
 *            w = (d*sc)*q - dmin*m
 *   PQ_Q6_K  210 B per 256 weights: 128 B low 4 bits, 64 B high 2 bits,
 *            int8 sc[16] (one per 16 weights), f16 d.   w = (d*sc)*(q-32)
 *   PQ_I8_ROW per-row symmetric int8: int8 q[n_out*k] row-major, then at the
 *            next 16-byte boundary f32 scale[n_out].      w = scale[r]*q
 *   PQ_Q5_K  176 B per 256: f16 d, f16 dmin, 12 B of (scale, min) pairs packed
 *            as in Q4_K, 32 B qh (fifth bits), 128 B of 4-bit q.
 *            w = (d*sc)*q - dmin*m, q in 0..31
 *   PQ_Q3_K  110 B per 256: 32 B hmask (high bits), 64 B of 2-bit q, 12 B of
 *            16 packed signed 6-bit scales, f16 d.  w = (d*sc)*v, v in -4..3
 *   PQ_Q2_K   84 B per 256: 16 B of 4-bit (scale, min) pairs, 64 B of 2-bit
 *            q, f16 d, f16 dmin.                 w = (d*sc)*q - dmin*m
 *   PQ_I4_ROW per-row symmetric int4 (k even): two's-complement 4-bit codes,
 *            weight 2i in the low nibble of byte i of the row, 2i+1 in the
 *            high nibble, rows of k/2 bytes; then at the next 16-byte
 *            boundary f32 scale[n_out].         w = scale[r]*q, q in -8..7
 * (Q5_K, Q3_K and Q2_K are the rest of the K family the PESTI README names;
 * they and PQ_I4_ROW run on the generic kernels.)
 * W is n_out rows; row r holds k/QK consecutive blocks (QK = 32 for Q8_0, 1
 * for PQ_I8_ROW, 2 for PQ_I4_ROW, 256 for the K formats), rows contiguous,
 * no padding.
 *
 * Ownership and threading: the caller allocates and owns every buffer it
 * passes (device memory, e.g. from cudaMalloc or a framework allocator).  The
 * library keeps a per-device record of the device's properties and one
 * library-owned stream-ordered memory pool per device.  pq_gemv draws a small
 * per-call buffer from that pool, allocated and freed on `stream`, for the
 * tensor-core kernel (x image and split-K partial sums, under 8 MB) and
 * for the batch-2 long-row kernel (x image, 4.5 * k bytes); every
 * other path allocates nothing.  The pool keeps freed memory for reuse, so
 * after the first call of a shape no call reaches the device allocator.  Calls
 * are reentrant and may run concurrently on different streams.  Calls are
 * asynchronous on `stream` (NULL = legacy default stream); a fault during
 * execution surfaces at the caller's next synchronization.  All argument
 * checks run on the host before any launch, so a rejected call launches
 * nothing.  pq_gemv_noalloc (below) runs the tensor-core path with no pool.
 */
#ifndef PQ_H
#define PQ_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* == cudaStream_t */

typedef enum {
    PQ_Q8_0 = 0,
    PQ_Q4_K = 1,
    PQ_Q6_K = 2,
    PQ_I8_ROW = 3,
    PQ_Q5_K = 4,
    PQ_Q3_K = 5,
    PQ_Q2_K = 6,
    PQ_I4_ROW = 7
} pq_fmt;

/* Status codes. */
#define PQ_OK 0
#define PQ_ERR_ARG (-1)      /* null pointer, or n_out / k / batch <= 0, or y aliases x or w */
#define PQ_ERR_FMT (-2)      /* unknown format */
#define PQ_ERR_K (-3)        /* k not a multiple of the format's block size QK */
#define PQ_ERR_ALIGN (-4)    /* w_blocks, x or out not 16-byte aligned, or y not 4-byte aligned */
#define PQ_ERR_SIZE (-5)     /* byte or element counts overflow 64-bit arithmetic */
#define PQ_ERR_DEVICE (-6)   /* current device is not compute capability 10.3 (sm_103) */
#define PQ_ERR_LAUNCH (-7)   /* a launch, or the pool allocation before it, failed */
#define PQ_ERR_KERNEL (-8)   /* unknown kernel id passed to pq_gemv_kernel */

/*
 * y[b][r] = sum_i w(r, i) * x[b][i]   for b < batch, r < n_out.
 *
 *   w_blocks  device, pq_weight_bytes(fmt, n_out, k) bytes in the layout above,
 *             16-byte aligned.  Read only.
 *   x         device f32 [batch][k] row-major, 16-byte aligned.  Read only.
 *   y         device f32 [batch][n_out] row-major; fully overwritten (not
 *             accumulated into).  Must not overlap w_blocks or x.
 *   batch     >= 1.  Batches above 32 are processed in chunks of at most 32
 *             (the tensor-core kernel takes up to 32 columns per pass over
 *             W; the CUDA-core kernels up to 4, or one).
 *
 * Accuracy: partial sums are accumulated in f32; the result agrees with the
 * exact dot product of the decoded f32 weights within
 * 2e-3 * RMS(y) + 1e-6 (see the tests).  Range of x: any finite x.  Every
 * kernel scales x per 256 values of each column before narrowing it: the
 * batch 1-4 kernels into two int8 limbs per value, the tensor-core kernel
 * (Q4_K at batch >= 5, and at batch 3-4 for long rows or large matrices; see
 * pq_gemv_choice) by a power of two into an fp16 pair x_hi + x_lo; the
 * generic kernel uses x in f32.  Non-finite x or scale fields give
 * non-finite outputs in the rows they reach.  Deterministic: repeated calls
 * with the same inputs give bit-identical y.  There is no host fallback:
 * every step runs in this library's CUDA kernels.
 */
int pq_gemv(pq_fmt fmt, const void *w_blocks, int n_out, int k,
            const float *x, int batch, float *y, struct CUstream_st *stream);

/*
 * Mat-vec with the bias add fused into the store (the PESTI README,
 * "Conformance", lists a bias on the QKV projections):
 *   y[b][r] = sum_i w(r, i) * x[b][i] + bias[r]
 *   bias  device f32 [n_out], 4-byte aligned, read only; must not overlap y.
 * Other arguments, layouts, errors and the accuracy bar as pq_gemv (the bias
 * is added in f32 to the f32 sum).  The batch-1 kernel (Q4_K, Q6_K) and the
 * tensor-core kernel add it at their final store; the other kernels store y
 * and one small kernel adds the bias after them.
 */
int pq_gemv_bias(pq_fmt fmt, const void *w_blocks, int n_out, int k, const float *x, int batch,
                 const float *bias, float *y, struct CUstream_st *stream);

/*
 * SwiGLU on a fused gate+up matrix (the PESTI README, "Conformance": the MLP
 * multiplies the sigmoid-based silu of the gate projection by the up
 * projection):
 *   h[b][j] = silu(g) * u,  g = sum_i w(j, i) * x[b][i],
 *                           u = sum_i w(n_ff + j, i) * x[b][i],
 *   silu(z) = z / (1 + e^-z)
 *   w_blocks  2 * n_ff rows in the layout above: the n_ff gate rows, then the
 *             n_ff up rows; 16-byte aligned, read only.
 *   h         device f32 [batch][n_ff] row-major, 4-byte aligned, fully
 *             overwritten; must not overlap w_blocks or x.
 * Accuracy: within 2e-3 * RMS(h) + 1e-6 of silu(g) * u on the exact sums.
 * The batch-1 kernel (Q4_K, Q6_K) reduces each gate row and its up row in
 * the same warp and stores only h; the tensor-core kernel pairs gate and up
 * tiles in its finishing kernel; the other kernels write the 2 * n_ff sums to
 * pool memory and one small kernel forms h.  Status codes as pq_gemv.
 */
int pq_gemv_swiglu(pq_fmt fmt, const void *w_blocks, int n_ff, int k, const float *x, int batch,
                   float *h, struct CUstream_st *stream);

/*
 * out[r][i] = w(r, i) as f32, row-major [n_out][k], bit-identical to the
 * layout rules above (one f32 rounding for Q4_K's final subtraction and for
 * PQ_I8_ROW's product; every other step is exact).
 *   out  device, 4 * n_out * k bytes, 16-byte aligned, must not overlap w_blocks.
 */
int pq_dequant(pq_fmt fmt, const void *w_blocks, int n_out, int k,
               float *out, struct CUstream_st *stream);

/* Bytes of a whole W in the given format; 0 when fmt is unknown, n_out or k
 * is <= 0, or k is not a multiple of the block size. */
size_t pq_weight_bytes(pq_fmt fmt, int n_out, int k);

/* Static description of a status code (never NULL). */
const char *pq_strerror(int status);

/*
 * Kernel selection, for tests and tuning.  pq_gemv picks a kernel from
 * (fmt, batch, n_out, k); pq_gemv_kernel runs a named one instead:
 *   PQ_KERNEL_AUTO     the same choice pq_gemv makes
 *   PQ_KERNEL_GENERIC  warp-per-row kernel, any format / shape / batch
 *   PQ_KERNEL_STREAM   bulk-copy ring + integer dot products (Q4_K at
 *                      batch 1-4, Q6_K at batch 1)
 *   PQ_KERNEL_TC       tcgen05 tensor-core kernel (Q4_K, batch 1-32, k a
 *                      multiple of 256 up to 65536; pq_gemv chooses it at
 *                      batch >= 5, and at batch 3-4 for long rows or large
 *                      matrices)
 * A kernel that cannot run the given case returns PQ_ERR_KERNEL without
 * launching anything.
 */
#define PQ_KERNEL_AUTO (-1)
#define PQ_KERNEL_GENERIC 0
#define PQ_KERNEL_STREAM 1
#define PQ_KERNEL_TC 2
int pq_gemv_kernel(pq_fmt fmt, const void *w_blocks, int n_out, int k,
                   const float *x, int batch, float *y, struct CUstream_st *stream,
                   int kernel);

/* The kernel id pq_gemv would choose for this case (>= 0), or a status < 0
 * for arguments it would reject. */
int pq_gemv_choice(pq_fmt fmt, int n_out, int k, int batch);

/*
 * Number of batch slices one pq_gemv call with these arguments runs (slices
 * of up to 32 columns for the tensor-core kernel, up to 4 or 1 otherwise), each
 * with one kernel choice.  A slice is one launch of its kernel, plus, for the
 * tensor-core kernels, and for the two-column kernels at rows longer than
 * 16384 (and the Q6_K kernel at 3-4 columns), one small x-conversion launch
 * before it, and for the tensor-core kernels one split-K finishing launch
 * after it when CTAs share a row tile.
 */
int pq_gemv_launches(pq_fmt fmt, int n_out, int k, int batch);

/*
 * Weight prefetch across kernel boundaries (process-wide, default off).
 * pq_gemv's whole-row kernels (batch 1, the register-operand kernel at batch
 * 2-8 and the two-column kernels) are launched with programmatic dependent
 * launch: each may be scheduled while the preceding kernel on the stream is
 * still finishing, and always waits for that kernel before reading x or
 * writing y.  With prefetch enabled they also start streaming w_blocks
 * before that wait.  Enable it only when no kernel that runs immediately before a
 * pq_gemv on its stream writes that call's w_blocks (the usual case: weights
 * loaded once, then only read).  Copies (cudaMemcpy*) are always waited for.
 * Returns the previous setting.
 */
int pq_set_weight_prefetch(int enable);

/*
 * Number of bounded waits that ran out in this library's kernels on the
 * current device since the last reset (reset != 0 clears the count).  Every
 * barrier wait inside a kernel gives up after 1 s, records the event here
 * and lets the kernel finish instead of hanging; a nonzero count means the
 * affected outputs are invalid.  Synchronous (reads device memory).
 * Returns PQ_ERR_DEVICE if the current device is not sm_103.
 */
int pq_wait_timeouts(int reset);

/*
 * Self-test of that failure detection (no counterpart on the pages: the
 * pages run no GPU kernels of this kind).  Launches one thread on `stream`
 * that waits on a barrier nothing completes, bounded by limit_us
 * microseconds (1 .. 1,000,000); the wait runs out, is counted in
 * pq_wait_timeouts, and the kernel returns normally, leaving the context
 * usable.  Synchronises `stream`.  Returns 1 when the wait ran out as
 * designed, 0 if it completed (never expected), PQ_ERR_ARG for a limit out of
 * range, PQ_ERR_DEVICE, or PQ_ERR_LAUNCH.
 */
int pq_selftest_wait_timeout(unsigned limit_us, struct CUstream_st *stream);

/*
 * Mat-vec that allocates no memory at all (no counterpart on the pages: an
 * addition of this library for callers that cannot allocate).
 *
 * Who needs it: code that may not call cudaMalloc, cudaFree or an
 * allocating pool once it runs -- a serving process whose device memory was
 * carved up ahead of time by another allocator, a runtime with a fixed
 * memory plan checked at start-up, or code recorded into a legacy-stream
 * capture, where allocation calls are not permitted.  pq_gemv's tensor-core
 * path (batch >= 5) takes a small per-call buffer from a stream-ordered pool;
 * this entry runs that same kernel with the buffer in a fixed device array
 * instead (3,743,744 bytes, part of the library image: every GPU that loads
 * the library holds it until the process exits).
 *
 * Same arguments, layouts and accuracy bar as pq_gemv, but it runs the
 * tensor-core kernel at every batch, 1-4 included (where pq_gemv mostly
 * runs other kernels), so its result equals pq_gemv_kernel(...,
 * PQ_KERNEL_TC) bit for bit.  Limits: fmt must be PQ_Q4_K (PQ_ERR_KERNEL
 * otherwise) and k <= 16384 (PQ_ERR_SIZE otherwise); any batch >= 1 (chunks
 * of 16, run one after another on `stream`).
 * Shared state: all calls in the process use the one array per GPU, which
 * keeps the last call's contents; each call writes every byte of it that it
 * later reads, so nothing needs clearing, but calls that overlap on the GPU
 * (different streams, or different threads) race on it and must be ordered
 * by the caller.  The first call on a device looks up the array's device
 * address (a one-time set-up with that device current); make that first call
 * before any stream capture.  The address is looked up once per device
 * ordinal, in the device's primary context (the one the CUDA runtime uses);
 * calls made under another context, or after cudaDeviceReset, are not
 * supported.
 */
int pq_gemv_noalloc(pq_fmt fmt, const void *w_blocks, int n_out, int k,
                    const float *x, int batch, float *y, struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* PQ_H */
