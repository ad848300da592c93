/*
 * sgmv.h -- C ABI of libsgmv.so, Punica's SGMV multi-LoRA hot path on one
 * NVIDIA GB300 (sm_103a).
 *
 * SGMV (Segmented Gather Matrix-Vector multiplication) adds each request's
 * LoRA delta to its rows of a batch in which contiguous row segments use
 * different adapters:
 *
 *     Y[row(p), :] += scale * (X[row(p), :] . A[idx[s]]) . B[idx[s]]
 *         for every sorted position p in segment s = [seg_ptr[s], seg_ptr[s+1])
 *
 * Pages this interface follows (cited by title and section):
 *   [Article] "Punica: when LoRA fine-tuned models need multi-tenant serving"
 *             (omica.com.cn):
 *               §2.1 the LoRA part of a layer is x.A.B, A [H1, r], B [r, H2];
 *               §2.2 SGMV = a segmented gather of A_i out of one stack of all
 *                    adapters with v_i = x_i.A_i ("shrink"), then v_i.B_i with
 *                    all B_i stacked the same way ("expand");
 *               §5.1 the batch builder groups requests by LoRA id;
 *               §5.2 a wrong rank or shape shows up as illegal memory access.
 *   [Review]  "Punica: Multi-Tenant LoRA Serving" (nubint.ai review),
 *             "Proposed method": the kernel works on segmented inputs and
 *             outputs so that different LoRA models share one batch.
 *   [Q&A]     "How to deploy several LoRA adapters without reloading the base
 *             model (Punica, S-LoRA)?" (aivaro.ru):
 *               §3.1 each request computes x = x + (x @ A) @ B;
 *               §3.2 adapter weights sit in one contiguous buffer and the
 *                    kernel selects them by index (segmented gather/scatter);
 *                    the kernel accepts any rank r without recompiling.
 *
 * Layouts (all row-major, all tensors in device memory unless stated):
 *   x  [T][H1]    f16 or bf16           batch input rows
 *   A  [L][H1][r] same type as x        stacked adapter "A" matrices
 *   B  [L][r][H2] same type as x        stacked adapter "B" matrices
 *   y  [T][H2]    f16, bf16 or f32      output rows, updated in place
 *   v  [T][r]     f32                   shrink result, by sorted position
 *   perm    int32 [T] or NULL           physical row of sorted position p;
 *                                       NULL means position p is row p
 *   seg_ptr int32 [S+1]                 segment bounds in sorted positions,
 *                                       non-decreasing, inside [0, T]
 *   idx     int32 [S]                   adapter of each segment, in [-1, L);
 *                                       -1 = no adapter (rows left unchanged)
 * Empty segments are allowed; adjacent segments may share an adapter; rows
 * outside [seg_ptr[0], seg_ptr[S]) are neither read nor written.  perm must
 * be one-to-one on the covered positions.
 *
 * Requirements checked on the host (status returned, nothing launched):
 *   pointers non-NULL where used and 16-byte aligned; H1 and H2 multiples of
 *   8 and >= 8; 1 <= r <= 128; T >= 0; L >= 1; dtypes as above.  seg_ptr_host,
 *   when given, is checked for bounds and order.
 * Checked on the device (the bad segment or row is skipped and the sticky
 * device error word is set; read it with sgmv_get_device_error):
 *   idx outside [-1, L) -> SGMV_ERR_BAD_INDEX; a segment outside [0, T] or
 *   with end < start -> SGMV_ERR_BAD_SEGMENTS; perm entry outside [0, T) ->
 *   SGMV_ERR_BAD_INDEX.  No kernel traps or asserts; every wait in a kernel is
 *   bounded and reports SGMV_ERR_TIMEOUT if it runs out.
 *
 * Ownership and execution: the caller owns every buffer; the library never
 * allocates device memory.  Calls are asynchronous on `stream` (a
 * cudaStream_t, NULL = legacy default stream), take no locks and keep no
 * state except the device error word.  The device addresses of the library's
 * own device variables (the error word, the scratch of sgmv_apply_noalloc)
 * are looked up once per device and kept: after cudaDeviceReset, or any other
 * teardown of a device's primary context, the library must not be used again
 * on that device in the same process.  Kernels are launched with
 * programmatic dependent launch: a kernel may start while the previous
 * kernel on the stream finishes, and before it waits for that kernel it
 * reads only A, B, row_adapter and the segment metadata.  So those inputs must
 * not be written by the SGMV kernel launched just before on the same stream
 * (x and y may be: they are read only after the wait).
 */
#ifndef SGMV_H
#define SGMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SGMV_OK = 0,
    SGMV_ERR_INVALID_ARG = 1,   /* NULL pointer, size out of range, bad dtype */
    SGMV_ERR_UNSUPPORTED = 2,   /* valid but outside what the library handles */
    SGMV_ERR_ALIGNMENT = 3,     /* pointer not 16-byte aligned, H1/H2 % 8 != 0 */
    SGMV_ERR_BAD_INDEX = 4,     /* adapter id or perm entry out of range */
    SGMV_ERR_CUDA = 5,          /* a CUDA runtime call failed */
    SGMV_ERR_WORKSPACE = 6,     /* workspace smaller than sgmv_workspace_bytes */
    SGMV_ERR_TIMEOUT = 7,       /* a bounded wait inside a kernel ran out */
    SGMV_ERR_BAD_SEGMENTS = 8   /* seg_ptr out of [0, T] or decreasing */
} sgmv_status;

typedef enum {
    SGMV_F16 = 0,
    SGMV_BF16 = 1,
    SGMV_F32 = 2                /* output y only */
} sgmv_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *sgmv_status_string(int status);

/* Detail of the last SGMV_ERR_CUDA returned on the calling thread (which CUDA
 * call failed and its error string); empty if none.  Thread-local storage
 * owned by the library, valid until the thread's next failing call. */
const char *sgmv_last_error_string(void);

/* Number of kernels the calling thread's last sgmv_shrink / sgmv_expand /
 * sgmv_apply / sgmv_build_segments_device call launched (0 when it returned
 * before launching anything). */
int sgmv_last_launch_count(void);

/* Upper bound on the number of segments that grouping T rows over L adapters
 * (ids -1..L-1) can produce: min(T, L + 1).  Size seg_ptr (bound + 1) and idx
 * (bound) with it for sgmv_build_segments_device. */
int32_t sgmv_max_segments(int32_t T, int32_t L);

/*
 * Group a batch's rows by adapter id, on the host ([Article] §5.1; [Review]
 * "Proposed method").  Stable: ascending id with -1 first, original row order
 * within an id, one segment per id that occurs.
 *   row_adapter  host int32 [T], ids in [-1, L)
 *   perm         host int32 [T]      out: physical row of each sorted position
 *   seg_ptr      host int32 [T + 1]  out: S + 1 entries used
 *   idx          host int32 [T]      out: S entries used
 *   S            host int32 [1]      out: number of segments
 * Returns SGMV_ERR_BAD_INDEX if an id is out of range (outputs undefined).
 */
int sgmv_build_segments(const int32_t *row_adapter, int32_t T, int32_t L,
                        int32_t *perm, int32_t *seg_ptr, int32_t *idx,
                        int32_t *S);

/*
 * The same grouping on the device, one small kernel, no host synchronisation.
 * All pointers are device pointers.  seg_ptr must hold
 * sgmv_max_segments(T, L) + 1 entries and idx sgmv_max_segments(T, L): past
 * the real segment count the kernel writes empty segments (seg_ptr = T,
 * idx = -1), so the arrays can be passed to the SGMV calls with
 * S = sgmv_max_segments(T, L).  *S receives the real count.  An id out of
 * range is grouped as -1 and sets SGMV_ERR_BAD_INDEX in the device error
 * word.  Requires L <= 32767.
 */
int sgmv_build_segments_device(const int32_t *row_adapter, int32_t T, int32_t L,
                               int32_t *perm, int32_t *seg_ptr, int32_t *idx,
                               int32_t *S, void *stream);

/*
 * Bytes of device workspace that lets sgmv_apply use its tensor-core path for
 * long segments: v for T rows as two 16-bit halves, plus 256 bytes for a
 * counter the tensor-core kernels use to share out the last part of the
 * work.  Calls that run at the same time need separate workspaces.
 * sgmv_apply also accepts workspace == NULL with workspace_bytes == 0 and
 * then runs every segment on the CUDA-core path.
 */
size_t sgmv_workspace_bytes(int32_t T, int32_t H1, int32_t H2, int32_t r);

/*
 * Shrink, the first SGMV step ([Article] §2.2):
 *   v[p][k] = sum_h x[row(p)][h] * A[idx[s]][h][k]    (fp32 accumulation)
 * v rows of segments with idx = -1 are set to 0; other rows of v are not
 * written.  seg_ptr_host (host int32 [S+1] copy of seg_ptr, or NULL) lets the
 * host size the launch exactly; without it the launch is sized by a bound.
 */
int sgmv_shrink(float *v, const void *x, const void *A, int in_dtype,
                const int32_t *perm, const int32_t *seg_ptr, const int32_t *idx,
                int32_t S, const int32_t *seg_ptr_host, int32_t T, int32_t L,
                int32_t H1, int32_t r, void *stream);

/*
 * Expand, the second SGMV step ([Article] §2.2), accumulated into y
 * ([Q&A] §3.1):
 *   y[row(p)][j] = round(y[row(p)][j] + scale * sum_k v[p][k] * B[idx[s]][k][j])
 * computed in fp32 and rounded once (to nearest even) to y's type.
 */
int sgmv_expand(void *y, int y_dtype, const float *v, const void *B, int in_dtype,
                float scale, const int32_t *perm, const int32_t *seg_ptr,
                const int32_t *idx, int32_t S, const int32_t *seg_ptr_host,
                int32_t T, int32_t L, int32_t H2, int32_t r, void *stream);

/*
 * Shrink and expand in one call: y += scale * (x . A[idx]) . B[idx] per
 * segment, with v kept on chip (never written to device memory) on the
 * CUDA-core path.  Segments of at least 64 rows use the tensor-core path when
 * a workspace of sgmv_workspace_bytes() is given (it holds v for those rows).
 * Result equals sgmv_shrink followed by sgmv_expand up to fp32 summation
 * order.
 */
int sgmv_apply(void *y, int y_dtype, const void *x, const void *A, const void *B,
               int in_dtype, float scale, const int32_t *perm,
               const int32_t *seg_ptr, const int32_t *idx, int32_t S,
               const int32_t *seg_ptr_host, int32_t T, int32_t L, int32_t H1,
               int32_t H2, int32_t r, void *workspace, size_t workspace_bytes,
               void *stream);

/*
 * Grouping and update in one call, from the batch's row -> adapter ids: the
 * whole hot path (group rows by adapter, gather x, shrink, expand, scatter
 * into y) for a batch whose rows arrive in any order.
 *   row_adapter  device int32 [T], ids in [-1, L) (-1 = no adapter)
 *   perm, seg_ptr, idx, S   device int32 arrays as for
 *                sgmv_build_segments_device, receiving the grouping so later
 *                calls on the same batch (other layers and projections) can
 *                pass it to sgmv_apply; all four NULL or all four set.
 * For T <= 64 rows this is a single kernel: every CTA groups the rows
 * itself, so no metadata is read from device memory (the arrays, if given,
 * are still written).  Otherwise it runs the grouping kernel into the caller's arrays
 * (then required: SGMV_ERR_INVALID_ARG if NULL) followed by sgmv_apply.  An id
 * out of range is treated as -1 and reported as SGMV_ERR_BAD_INDEX in the
 * device error word.
 */
int sgmv_apply_rows(void *y, int y_dtype, const void *x, const void *A, const void *B,
                    int in_dtype, float scale, const int32_t *row_adapter, int32_t T, int32_t L,
                    int32_t H1, int32_t H2, int32_t r, int32_t *perm, int32_t *seg_ptr,
                    int32_t *idx, int32_t *S, void *workspace, size_t workspace_bytes,
                    void *stream);

/*
 * sgmv_apply for callers that cannot allocate device memory: the pages
 * describing SGMV have no counterpart of this call.  It is for code that may
 * not call cudaMalloc where it runs SGMV -- a plugin that only gets the
 * buffers its host engine planned at start-up, a serving loop that forbids
 * allocation after warm-up, or code running while a CUDA graph is captured.
 * Arguments and results are those of sgmv_apply, without the workspace: the
 * scratch for the tensor-core path is a fixed 4 MiB array inside the
 * library's device image, held by every GPU that loads the library until the
 * process exits.  Only problems that can reach the tensor-core path (r = 64
 * or 128 and T >= 64) use it; those whose sgmv_workspace_bytes(T, H1, H2, r)
 * exceeds 4 MiB are refused with SGMV_ERR_WORKSPACE before anything is
 * launched.  Every other problem runs on the CUDA cores without scratch,
 * whatever its size.  The first such call on a device looks the array's
 * device address up (cudaGetSymbolAddress, no allocation); make that first
 * call before any stream capture.  All calls share the one array and it keeps
 * the last call's contents (nothing in it has to start at zero), so calls
 * that overlap on the GPU -- on different streams, or from different threads
 * -- race on it.
 */
int sgmv_apply_noalloc(void *y, int y_dtype, const void *x, const void *A, const void *B,
                       int in_dtype, float scale, const int32_t *perm, const int32_t *seg_ptr,
                       const int32_t *idx, int32_t S, const int32_t *seg_ptr_host, int32_t T,
                       int32_t L, int32_t H1, int32_t H2, int32_t r, void *stream);

/*
 * Bytes of device workspace sgmv_fused_linear_lora needs: v [T][r] fp32, the
 * pair table and the 16-bit v tiles of the adapter terms (at most T tiles of
 * [16][64] elements, two per pair for r > 32), and an fp32 scratch area for
 * the partial sums of tiles split across a cluster (at most 8 x
 * ceil(H2 / 128) x round32(T) x 128 floats); each part 256-byte aligned.
 */
size_t sgmv_fused_workspace_bytes(int32_t T, int32_t H2, int32_t r);

/*
 * The whole LoRA layer in one pass over its weights: the base linear layer and
 * the SGMV update together ([Article] §2.1: a LoRA layer computes
 * y = xW + xAB; [Q&A] §3.2, "Fused Kernel": the LoRA transform is merged into
 * the base model's linear layer so that memory is read fewer times):
 *   y[t][j] = round( sum_h x[t][h] * W[h][j]
 *                    + scale * sum_k v[p][k] * B[idx[s]][k][j] )
 *   with v[p] = x[t] . A[idx[s]], for physical row t = perm[p] of position p
 *   in segment s with idx[s] >= 0; rows in no segment with an adapter get
 *   the base product alone.
 * Every row t in [0, T) of y is overwritten (y is the layer's output; it must
 * not overlap x, W, A or B); the sums are fp32 and y is rounded once.
 *   W  [H1][H2]  device, in_dtype (f16 / bf16), row-major
 *   x, A, B, perm, seg_ptr, idx, S, L, r as for sgmv_apply; y as for
 *   sgmv_apply but written, not updated.
 *   workspace  device, >= sgmv_fused_workspace_bytes(T, H2, r) bytes, 16-byte
 *              aligned (holds v, its tiles and partial sums between the kernels).
 * Decode batches: 1 <= T <= 128 rows and r <= 64 (SGMV_ERR_UNSUPPORTED
 * otherwise).  Three kernels on `stream` (one when S == 0): the CUDA-core
 * shrink writes v; a small kernel lays scale * v out as block-diagonal 16-bit
 * tiles (each value as a high and a low half); a tensor-core kernel streams W
 * and the adapters' B slices once and makes every element of y, base and
 * adapter terms in one fp32 accumulation.  Errors as for sgmv_apply (host checks, device error
 * word).
 */
int sgmv_fused_linear_lora(void *y, int y_dtype, const void *x, const void *W, const void *A,
                           const void *B, int in_dtype, float scale, const int32_t *perm,
                           const int32_t *seg_ptr, const int32_t *idx, int32_t S, int32_t T,
                           int32_t L, int32_t H1, int32_t H2, int32_t r, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * sgmv_apply for P problems at once (1 <= P <= 4) that share the rows, the
 * segments and the shapes but have their own x, A, B and y: the projections
 * of one layer that read the same rows, q / k / v, or gate / up ([Article]
 * §2.1: a LoRA pair A, B sits beside a weight matrix W; §3.2: the pairs are
 * injected into the model's linear layers, e.g. each layer's attention q
 * projection; §2.2 for the operation).  y[k] += scale * (x[k] . A[k][idx]) . B[k][idx], every
 * argument otherwise as for sgmv_apply (host arrays of P device pointers for
 * y, x, A, B; x[k] may all be the same pointer, the y[k] must not overlap
 * one another: the problems' updates run at the same time).  The P problems run as one
 * launch of the streaming CUDA-core kernel when r <= 64, r % 4 == 0 and the
 * batch is large enough for one-CTA clusters (T > 76 on 152 SMs; each CTA
 * walks several (problem, tile) units), with each row's arithmetic exactly
 * that of P separate sgmv_apply calls without a workspace (the same bits);
 * otherwise it makes those P calls.  P = 1 is allowed: a serving loop that
 * sends all its calls here runs a single kernel.
 * No workspace, nothing allocated.  Errors: SGMV_ERR_INVALID_ARG for P out
 * of range or null arrays or pointers, then as sgmv_apply; when the problems
 * run as P calls and call k fails, problems 0 .. k-1 are already queued on
 * `stream` and k .. P-1 are not.
 */
int sgmv_apply_multi(int32_t P, void *const *y, int y_dtype, const void *const *x,
                     const void *const *A, const void *const *B, int in_dtype, float scale,
                     const int32_t *perm, const int32_t *seg_ptr, const int32_t *idx, int32_t S,
                     const int32_t *seg_ptr_host, int32_t T, int32_t L, int32_t H1, int32_t H2,
                     int32_t r, void *stream);

/*
 * Loads one adapter into slot `slot` of the stacked pools: A_src [H1][r] into
 * A_pool[slot] and B_src [r][H2] into B_pool[slot], as two asynchronous copies
 * on `stream`.  Page: [Review] "Punica: Multi-Tenant LoRA Serving" (nubint.ai
 * review), "Proposed method" and findings: LoRA weights are loaded on demand,
 * in milliseconds, instead of keeping every adapter resident.
 *   A_pool  [L][H1][r]  device, in_dtype        stacked "A" matrices
 *   B_pool  [L][r][H2]  device, in_dtype        stacked "B" matrices
 *   A_src, B_src        host or device memory, in_dtype, contiguous; from
 *                       page-locked host memory the copies overlap with
 *                       kernels on other streams and return at once
 * Nothing is allocated.  The caller orders the copies before the SGMV calls
 * that read the slot (an event on `stream`) and must not overwrite a slot that
 * an SGMV call in flight still reads.  Errors: SGMV_ERR_INVALID_ARG for null
 * pointers, slot outside [0, L), non-positive sizes or an input type other
 * than f16 / bf16; SGMV_ERR_CUDA if a copy cannot be enqueued.
 */
int sgmv_load_adapter(void *A_pool, void *B_pool, int in_dtype, int32_t slot, const void *A_src,
                      const void *B_src, int32_t L, int32_t H1, int32_t H2, int32_t r,
                      void *stream);

/*
 * Up to 512 copies dst[i] <- src[i] (bytes[i] bytes each) on `stream`, for
 * loading every piece of an adapter at once (same page and passage as
 * sgmv_load_adapter: one Llama-2-7B adapter is 448 pieces).  Every copy whose
 * source and destination the current device reads directly (its own device
 * memory, or page-locked host memory), both 16-byte aligned, with bytes[i] a
 * multiple of 16, is moved by ONE kernel launch: the SMs read the sources
 * (page-locked host memory over the CPU-GPU link) and write the destinations.
 * Each other copy is enqueued as its own asynchronous copy-engine transfer on
 * `stream`.  All copies are ordered after earlier work on `stream`.
 *   n          number of copies, 0 <= n <= 512 (0: nothing happens)
 *   dst, src   host arrays of n pointers (host or device addresses); the
 *              ranges must not overlap one another
 *   bytes      host array of n sizes; a zero size skips its copy (its
 *              pointers may then be null)
 *   max_ctas   most CTAs of the kernel; 0 = four per SM.  A small cap leaves
 *              SMs to kernels that run at the same time on other streams.
 * The arrays are read before the call returns; the copied memory must stay
 * valid until the copies complete.  Nothing is allocated.  Errors:
 * SGMV_ERR_INVALID_ARG for n outside [0, 512], negative max_ctas, null arrays
 * or a null pointer with a non-zero size; SGMV_ERR_CUDA if a copy or the
 * launch cannot be enqueued (then some copies may have been enqueued).
 * sgmv_last_launch_count() is 1 if the kernel was launched, else 0.
 */
int sgmv_copy_gather(int32_t n, void *const *dst, const void *const *src, const uint64_t *bytes,
                     int32_t max_ctas, void *stream);

/*
 * Diagnostics (no counterpart on the pages).
 *
 * sgmv_read_floor: the floor of a decode-sized SGMV launch on this GPU.  Reads
 * `bytes` (a multiple of 16) of device memory at `src` (16-byte aligned) and
 * nothing else, spread evenly over the grid, cluster size, ring depth and
 * copy size that the streaming kernel gets from sgmv_apply_rows for a batch
 * of T rows over L adapters with these dimensions, types and rank (the
 * one-launch grouped form up to 64 rows; sgmv_apply on the device grouping
 * otherwise).  Pass the batch's algorithmic bytes to time what merely
 * bringing them on chip costs with that launch shape.  *ctas and *cluster
 * (each may be NULL) receive the grid's CTA count and cluster size.
 * SGMV_ERR_UNSUPPORTED when the streaming kernel does not apply (r not a
 * multiple of 4, or above 64).  Asynchronous on `stream`; writes nothing.
 */
int sgmv_read_floor(const void *src, size_t bytes, int32_t T, int32_t L, int32_t H1, int32_t H2,
                    int32_t r, int in_dtype, int y_dtype, int32_t *ctas, int32_t *cluster,
                    void *stream);

/*
 * sgmv_debug_inject_wait_timeout: for tests of the device-side timeout path.
 * While enabled (non-zero) on the calling thread, every streaming-kernel
 * launch it makes takes the timeout path at each compute thread's first wait
 * for a staged chunk, as if that wait had run out: SGMV_ERR_TIMEOUT is set in
 * the device error word, the chunk is then awaited with the full limit (so
 * the kernel still ends normally, with every copy landed) and the thread
 * writes no y.  Other kernels are unaffected.  Returns SGMV_OK.
 */
int sgmv_debug_inject_wait_timeout(int enable);

/*
 * Synchronises `stream`, then reads and clears the current device's sticky
 * error word.  Returns SGMV_OK if no kernel reported an error since the last
 * read, else the first status code reported (SGMV_ERR_BAD_INDEX,
 * SGMV_ERR_BAD_SEGMENTS or SGMV_ERR_TIMEOUT), or SGMV_ERR_CUDA if the
 * synchronisation itself failed.
 */
int sgmv_get_device_error(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SGMV_H */
