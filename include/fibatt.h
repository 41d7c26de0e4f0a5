/*
 * fibatt.h -- C ABI of libfibatt: Fibottention's per-head sparse
 * self-attention (forward and backward) on NVIDIA GB300 (sm_103a).
 *
 * The operation ("Fibottention: Inceptive Visual Representation Learning
 * with Diverse Attention Across Heads", arXiv 2406.19391, Sec. 3):
 *
 *   head h of H, query j in [0, N) attends exactly the keys k with
 *       |j - k| in Fib(a_h, b_h)  and  |j - k| <= w_h      (support Omega_h)
 *   plus k = j when the main diagonal is included.  Fib(a, b) is the
 *   generalised Fibonacci sequence f_1 = a, f_2 = b, f_{n+2} = f_{n+1} + f_n
 *   (project README, Algorithm 1), and (a_h, b_h) is normally row h of the
 *   Wythoff array (Sec. 3.2).  Scores outside Omega_h are excluded from the
 *   softmax:
 *       s_jk = scale * <Q_j, K_k>                 (j,k) in Omega_h
 *       LSE_j = log sum_{k:(j,k) in Omega_h} exp(s_jk)
 *       O_j  = sum_{k:(j,k) in Omega_h} exp(s_jk - LSE_j) V_k
 *   (README, Algorithm 3: scores, mask, row softmax, weighted sum of V).
 *
 * Conventions shared by every call below:
 *   - Tensors are dense, row-major [B, H, N, D] with D = 64 (one row = 64
 *     contiguous elements), in the I/O dtype fibatt_dtype; LSE is fp32
 *     [B, H, N].  All tensor pointers are DEVICE pointers owned by the
 *     caller, 16-byte aligned (LSE: 4-byte aligned), on the current device.
 *   - Arithmetic is fp32 with fp32 accumulation; bf16 outputs are rounded to
 *     nearest-even once, at the end.  LSE is the natural log.  One exception,
 *     for bf16 I/O in the shared-memory forward kernels: each softmax weight
 *     is rounded to bf16 before its P.V update (products exact, sums fp32),
 *     and O is divided by the sum of those rounded weights, so O stays a
 *     convex combination of value rows; the LSE uses the fp32 weights.
 *   - fwd/bwd are asynchronous on `stream` and never synchronise.  They do not
 *     allocate device memory.
 *   - A support handle is host memory only (its tables travel to the GPU as
 *     kernel arguments), so one handle may be used on any device and from
 *     any stream; it must not be destroyed while a call using it is being
 *     made (kernels already launched do not reference it).
 *   - Every call returns a fibatt_status; on failure, fibatt_last_error()
 *     gives a message for the calling thread.  Nothing is ever trapped on the
 *     device.
 */
#ifndef FIBATT_H_
#define FIBATT_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FIBATT_OK = 0,
    FIBATT_ERR_INVALID_ARG = 1,   /* a size, pointer or parameter is out of its range      */
    FIBATT_ERR_UNSUPPORTED = 2,   /* valid, but outside what this build implements          */
    FIBATT_ERR_CUDA = 3,          /* a CUDA launch or runtime call failed (message attached) */
    FIBATT_ERR_OOM = 4            /* host allocation failed                                 */
} fibatt_status;

typedef enum {
    FIBATT_F32 = 0,               /* float32 I/O                          */
    FIBATT_BF16 = 1               /* bfloat16 I/O, fp32 accumulation      */
} fibatt_dtype;

/* Opaque per-layer support: the signed-offset table of every head. */
typedef struct fibatt_support *fibatt_support_t;

/* Limits of this build (UNSUPPORTED beyond them). */
#define FIBATT_HEAD_DIM 64        /* D                                         */
#define FIBATT_MAX_HEADS 64       /* H                                         */
#define FIBATT_MAX_ENTRIES 1024   /* signed offsets summed over all heads      */

/* ------------------------------------------------------------- helpers --- */

/* Row i (i >= 1) of the Wythoff array (Fibottention Sec. 3.2): writes its
 * first two entries a = floor(floor(i*phi)*phi), b = floor(floor(i*phi)*phi^2),
 * computed in exact integer arithmetic.  Rows are disjoint and together
 * contain every positive integer once.  INVALID_ARG unless 1 <= i <= 1e8. */
fibatt_status fibatt_wythoff_row(int64_t i, int64_t *a, int64_t *b);

/* The "modified" Wythoff row of the project README (Algorithm 2): the two
 * terms that precede row i, (2a - b, b - a).  Same argument rules. */
fibatt_status fibatt_wythoff_row_modified(int64_t i, int64_t *a, int64_t *b);

/* Per-head windows (Fibottention Sec. 3.2):
 *     w[i-1] = w_min + floor((w_max - w_min) * (i - 1) / (h - 1)),  i = 1..h
 * (h = 1 gives w_min).  w has h entries, caller-owned.
 * INVALID_ARG unless h >= 1 and 1 <= w_min <= w_max. */
fibatt_status fibatt_window_schedule(int h, int64_t w_min, int64_t w_max, int64_t *w);

/* ------------------------------------------------------------- support --- */

/* Build the support of H heads over N tokens (Fibottention Sec. 3, support
 * set Omega_w^{Fib(a,b)}; README Algorithm 1 for the sequence).  a, b, w are
 * host arrays of H entries; head h uses Fib(a[h], b[h]) cut at w[h]:
 * the distances kept are the distinct terms f with f <= min(w[h], N - 1), and
 * the head's table is the ascending signed list {-f...} U {0 if include_diag
 * or 0 in Fib} U {+f...}.  A per-layer head permutation is applied by the
 * caller by permuting a, b and w.
 * INVALID_ARG: H < 1, N < 1, a[h] < 0, b[h] < 0, a[h] = b[h] = 0, w[h] < 1 or
 * w[h] > N, out == NULL.  UNSUPPORTED: H > FIBATT_MAX_HEADS or more than
 * FIBATT_MAX_ENTRIES signed entries in total.  *out is owned by the caller
 * and released with fibatt_support_destroy. */
fibatt_status fibatt_support_build(int H, int N, const int64_t *a, const int64_t *b,
                                   const int64_t *w, int include_diag, fibatt_support_t *out);

/* Build a support from explicit unsigned distances (any dilation sequence,
 * Fibottention Sec. 3: constant c*n or exponential dilation, or the full
 * range 0..N-1 for dense attention).  counts[h] distances for head h are
 * concatenated in `distances`; duplicates count once, distances > N - 1 are
 * dropped, 0 means the main diagonal.  INVALID_ARG on a negative count or
 * distance; limits as fibatt_support_build. */
fibatt_status fibatt_support_build_distances(int H, int N, const int32_t *counts,
                                             const int32_t *distances, int include_diag,
                                             fibatt_support_t *out);

/* Make token 0 global in every head of the support, or banded again
 * (enabled = 0): the class token attends every key and every query attends
 * it, on top of the banded Fibonacci support (Fibottention README,
 * Algorithm 2, whose mask keeps row 0 and column 0 all ones).  The signed
 * tables keep describing the banded part; fibatt_support_get's pair counts
 * include the global pairs.  With it enabled, the dense row of token 0 (and
 * for the backward its dense row and the column of key 0) is computed inside
 * the shared-memory-resident kernels when their plan allows it, else by up to
 * three extra small kernels; FIBATT_PATH=generic and fibatt_bwd_noalloc are
 * UNSUPPORTED, and the backward's workspace grows by 2 x N fp32 per (b, h)
 * (used by the extra kernels only).  Not thread-safe against calls using the
 * support. */
fibatt_status fibatt_support_set_global_token(fibatt_support_t s, int enabled);

/* Sizes of a support: heads, tokens, and total signed entries. */
fibatt_status fibatt_support_info(fibatt_support_t s, int *H, int *N, int *total_entries);

/* Copy a support's tables out (host arrays, caller-sized from
 * fibatt_support_info): counts[H] signed entries per head, signed_offsets in
 * CSR order (head 0's ascending list, then head 1's, ...), pairs[H] = |Omega_h|,
 * the number of attended (j,k) pairs of head h.  Any output may be NULL. */
fibatt_status fibatt_support_get(fibatt_support_t s, int32_t *counts, int32_t *signed_offsets,
                                 int64_t *pairs);

void fibatt_support_destroy(fibatt_support_t s);

/* ------------------------------------------------------------ attention --- */

/* Forward pass.  Q, K, V: [B, H, N, D] (dtype); writes O: [B, H, N, D] (dtype)
 * and LSE: [B, H, N] fp32, natural log.  A query row with no support gets
 * O = 0 and LSE = -inf.  scale multiplies every dot product (1/sqrt(D) in
 * ViT; any finite value).  INVALID_ARG: NULL or misaligned pointer, B < 1,
 * B*H > 2^31-1, non-finite scale.  UNSUPPORTED: D != 64, unknown dtype.
 * CUDA: launch failure (the message names the CUDA error). */
fibatt_status fibatt_fwd(fibatt_support_t s, int B, int D, fibatt_dtype dtype,
                         const void *Q, const void *K, const void *V, float scale,
                         void *O, float *LSE, cudaStream_t stream);

/* Device scratch the backward pass may need for B batches of this support,
 * in bytes: the larger of one fp32 per query row (D_j = <dO_j, O_j>, global-
 * memory kernels) and the pair weights P and dS of every attended pair
 * (2 x the largest per-head table x N fp32 per (b, h); kernels for windows
 * too wide for shared memory).  The shared-memory-resident kernels touch
 * none of it. */
size_t fibatt_bwd_workspace_bytes(fibatt_support_t s, int B);

/* Backward pass for the loss whose gradient with respect to O is dO:
 *   P_jk = exp(s_jk - LSE_j),  dP_jk = <dO_j, V_k>,  D_j = <dO_j, O_j>,
 *   dS_jk = P_jk (dP_jk - D_j),
 *   dQ_j = scale sum_k dS_jk K_k,  dK_k = scale sum_j dS_jk Q_j,
 *   dV_k = sum_j P_jk dO_j      (sums over (j,k) in Omega_h)
 * (the exact derivative of the forward pass above; the pages print no
 * backward).  Q, K, V, O, dO: [B, H, N, D] (dtype); LSE from fibatt_fwd;
 * writes dQ, dK, dV: [B, H, N, D] (dtype).  workspace: device memory of at
 * least fibatt_bwd_workspace_bytes(s, B) bytes, 16-byte aligned, caller-owned
 * (contents on entry are ignored); may be NULL when that size is 0.
 * Errors as fibatt_fwd, plus INVALID_ARG when the workspace is too small. */
fibatt_status fibatt_bwd(fibatt_support_t s, int B, int D, fibatt_dtype dtype,
                         const void *Q, const void *K, const void *V, const void *O,
                         const float *LSE, const void *dO, float scale,
                         void *dQ, void *dK, void *dV, void *workspace, size_t ws_bytes,
                         cudaStream_t stream);

/* Scratch rows (fp32 each) built into the library for fibatt_bwd_noalloc. */
#define FIBATT_NOALLOC_MAX_ROWS (1u << 20)

/* Backward pass for callers that cannot allocate device memory (for example
 * code that runs where the allocator is off limits, or a plugin that is
 * handed fixed buffers).  Same arguments, results and errors as fibatt_bwd
 * without the workspace: the scratch (one fp32 per query row) lives in a
 * fixed array of FIBATT_NOALLOC_MAX_ROWS rows that every GPU loading the
 * library holds until the process exits, so this call allocates nothing.
 * INVALID_ARG when B*H*N exceeds FIBATT_NOALLOC_MAX_ROWS.  The first call on
 * a device looks up the array's device address on that device (make it before
 * any stream capture).  All calls on a device share the array: calls that
 * overlap on the GPU race on it.  No counterpart in the paper: this is a
 * library convenience, not part of the method. */
fibatt_status fibatt_bwd_noalloc(fibatt_support_t s, int B, int D, fibatt_dtype dtype,
                                 const void *Q, const void *K, const void *V, const void *O,
                                 const float *LSE, const void *dO, float scale,
                                 void *dQ, void *dK, void *dV, cudaStream_t stream);

/* Message for the last failing call on this thread ("" if none). */
const char *fibatt_last_error(void);

/* Library version string. */
const char *fibatt_version(void);

/* Device-side error word of the current device: bit 0 (1) is set when a
 * kernel gave up waiting for its shared-memory staging copies (a bounded wait
 * of about 2 s; the kernel then returns without writing its outputs); bit 1
 * (2) when a producer left before its last copies had landed (also after
 * about 2 s); bit 2 (4), in the bounds-checked debug build only (built with
 * -DFIBATT_CHECKS), when a kernel's bounds check failed and it skipped the
 * access (the first failing source line is then printed to stderr).  The
 * word is the OR over every kernel file's copy.  This call synchronises with
 * the device.  With clear != 0 the word is reset.  CUDA on a failed copy. */
fibatt_status fibatt_device_error(int clear, unsigned *code);

/* Number of CUDA kernels this library has launched in this process so far
 * (all devices, all threads); for accounting in benchmarks and tests. */
uint64_t fibatt_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FIBATT_H_ */
