/*
 * cr.h - C ABI of the GB300 canonical reduce / scan library (libcr).
 *
 * What is computed: "Canonical Parallel Reduction and Scan" (github README
 * andyD123/canonical-reduce):
 *   P4016R0, Key Design Points - the input is split across L interleaved
 *     lanes by i mod L; each lane is reduced by the iterative pairwise
 *     (shift-reduce) tree; the lane results are combined by the same tree
 *     rule; init is combined once, after the tree, as op(init, R).
 *   P4229R0, Summary and Key Design Points - named expression policies
 *     left_fold, pairwise, iterated_pairwise and block_dyadic<B>; the scan
 *     returns the prefix observations of the named expression.
 * op is IEEE-754 addition in the element type, round to nearest even, no
 * contraction, subnormals kept (the page's FP environment: --fmad=false).
 * Every result is bit-identical to the expression: it does not depend on the
 * GPU, the SM count, the grid or the tile sizes.
 *
 * Conventions for every call:
 *   - Pointers named x, out, ws are DEVICE pointers; init_host points to ONE
 *     element of the call's dtype in HOST memory (read before the call
 *     returns). The caller owns every buffer; libcr allocates nothing and
 *     frees nothing.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream). Calls return without synchronising; results are
 *     valid once the stream reaches that point.
 *   - Sizes and strides are counted in ELEMENTS, not bytes, and are >= 0
 *     (a negative stride is INVALID_ARG). x must be aligned to its element
 *     size.
 *   - ws is a device workspace of at least the size the matching
 *     *_workspace_bytes() call returns, 256-byte aligned. A call may use it
 *     until the stream passes the call; two calls that overlap in time must
 *     not share one workspace.
 *   - Errors: CR_ERR_INVALID_ARG for a bad argument (nothing is enqueued),
 *     CR_ERR_WORKSPACE when ws is NULL, misaligned or too small (nothing is
 *     enqueued), CR_ERR_UNSUPPORTED for a valid request this library version does not
 *     implement, CR_ERR_CUDA when a launch fails. A device-side wait that
 *     gives up after its bounded spin is reported later by cr_sync_status().
 */
#ifndef CR_H_
#define CR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { CR_F32 = 1, CR_F64 = 2 } cr_dtype;

/* Scan expression policies (P4229R0, Summary). */
typedef enum {
  CR_LEFT_FOLD = 0,         /* y[i] = (((x0 op x1) op x2) ... op xi)                */
  CR_PAIRWISE = 1,          /* maximal complete subtrees covering x[0..i], folded   */
                            /* from the left (prefix observation of one tree)       */
  CR_ITERATED_PAIRWISE = 2, /* y[i] = tree(x[0..i]), the P4016 tree with L = 1      */
  CR_BLOCK_DYADIC = 3       /* tree inside blocks of B, blocks chained left to right */
} cr_policy;

typedef enum {
  CR_OK = 0,
  CR_ERR_INVALID_ARG = 1,
  CR_ERR_UNSUPPORTED = 2,
  CR_ERR_WORKSPACE = 3,
  CR_ERR_CUDA = 4,
  CR_ERR_TIMEOUT = 5
} cr_status;

/* ---------------------------------------------------------------- reduce */

/* Workspace bytes for cr_reduce(n, L, dt). Never 0 (the status word lives
 * there). Returns 0 only for invalid arguments. */
size_t cr_reduce_workspace_bytes(int64_t n, int32_t L, cr_dtype dt);

/* Canonical reduction (P4016R0, Key Design Points):
 *   result = op(init, tree(R_0, ..., R_{m-1})),  m = min(n, L),
 *   R_j    = tree(x[j], x[j+L], x[j+2L], ...)   (lane j: i mod L == j),
 *   tree() = the iterative pairwise shift-reduce tree (operands pushed left
 *            to right, the two topmost partial trees combined while they
 *            cover equally many operands, the rest folded from the top down).
 * Empty lanes (n < L) are omitted; n == 0 gives init.
 *   x         device, n contiguous elements of dt
 *   n         >= 0
 *   L         lane count, >= 1 (the sole topology coordinate)
 *   init_host host pointer to one element of dt
 *   out_dev   device pointer to one element of dt, written by the stream
 * Errors: INVALID_ARG if n < 0, L < 1, x/out/init NULL, bad dt. */
cr_status cr_reduce(const void* x, int64_t n, int32_t L, const void* init_host, cr_dtype dt,
                    void* out_dev, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes for cr_reduce_batched with these sizes. */
size_t cr_reduce_batched_workspace_bytes(int64_t batch, int64_t n, int32_t L, cr_dtype dt);

/* A batch of independent canonical reductions with one L and one init:
 * sequence b has elements x[b*batch_stride + i*elem_stride], i < n, and
 * out_dev[b] = reduce(sequence b, n, L, init). Strides are any values >= 0
 * (e.g. rows: elem_stride 1, batch_stride ncols; columns of a level-major
 * array: elem_stride ncols, batch_stride 1; 0 repeats an element or a
 * sequence), but sequences must not alias out_dev. batch >= 0, n >= 0,
 * L >= 1; a negative stride is INVALID_ARG. With two or more sequences
 * laid out densely (rows: elem_stride 1, batch_stride n; or level-major
 * columns: batch_stride 1, elem_stride batch), an out_dev range that meets
 * the input is INVALID_ARG; for other layouts keeping them apart is the
 * caller's duty. */
cr_status cr_reduce_batched(const void* x, void* out_dev, int64_t batch, int64_t n,
                            int64_t elem_stride, int64_t batch_stride, int32_t L,
                            const void* init_host, cr_dtype dt, void* ws, size_t ws_bytes,
                            void* stream);

/* ------------------------------------------------------------------ scan */

/* Workspace bytes for cr_inclusive_scan(n, p, B, dt). */
size_t cr_scan_workspace_bytes(int64_t n, cr_policy p, int64_t B, cr_dtype dt);

/* Inclusive scan: out[i] = the prefix observation at i of the expression
 * named by p (P4229R0, Summary / Key Design Points):
 *   CR_LEFT_FOLD          out[i] = out[i-1] op x[i]
 *   CR_ITERATED_PAIRWISE  out[i] = tree(x[0..i])  (consistent: equals the
 *                         reduce of the prefix under the same expression)
 *   CR_PAIRWISE           the maximal complete subtrees of the one tree over
 *                         x that cover x[0..i], folded from the left (not
 *                         consistent in general)
 *   CR_BLOCK_DYADIC       blocks k = [kB, kB+B): P(i) = tree(x[kB..i]),
 *                         T_k = P(end of block k), C_0 = T_0,
 *                         C_k = C_{k-1} op T_k; out[i] = P(i) in block 0,
 *                         else C_{k-1} op P(i)
 * B is used only by CR_BLOCK_DYADIC and must then be a power of two >= 1.
 * x, out device, n contiguous elements; out == x (in place) is allowed, any
 * other overlap is INVALID_ARG. n == 0 writes nothing. No init: a scan
 * observes the expression itself.
 * Cost: the carry chain of CR_LEFT_FOLD and CR_BLOCK_DYADIC (ceil(n/B)
 * dependent adds) is evaluated exactly in parallel, every step checked
 * exactly against the add it replaces. Binary64 steps are classified against
 * a rigorous error bound; binary32 steps against an estimate of the binary32
 * chain's own rounding with a statistical margin. Where a check fails (in
 * practice: binary32 chains whose rounding is biased for long stretches,
 * such as sums of positive values far below the chain's unit), the chain is
 * recomputed one add at a time on the device (about 3 ns an add on GB300):
 * the result is exact either way. */
cr_status cr_inclusive_scan(const void* x, void* out, int64_t n, cr_policy p, int64_t B,
                            cr_dtype dt, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes for cr_inclusive_scan_batched with these sizes. */
size_t cr_scan_batched_workspace_bytes(int64_t batch, int64_t n, cr_policy p, int64_t B,
                                       cr_dtype dt);

/* A batch of independent inclusive scans with one policy and B: sequence b is
 * x[b*batch_stride + i*elem_stride], i < n, and its result goes to the same
 * positions of out (out uses x's strides). Typical use: columns of a
 * level-major (levels x ncols) array scanned along the levels, elem_stride =
 * ncols, batch_stride = 1. out == x is allowed; sequences must not overlap
 * one another (a zero elem_stride with n >= 2, a zero batch_stride with
 * batch >= 2, or elem_stride == batch_stride with batch >= 2 and n >= 2
 * sends two outputs to one element: INVALID_ARG). With out != x and both
 * laid out densely (rows or level-major columns), an out that meets x is
 * INVALID_ARG; for other layouts keeping them apart is the caller's duty. */
cr_status cr_inclusive_scan_batched(const void* x, void* out, int64_t batch, int64_t n,
                                    int64_t elem_stride, int64_t batch_stride, cr_policy p,
                                    int64_t B, cr_dtype dt, void* ws, size_t ws_bytes,
                                    void* stream);

/* reduce<E>: the root of the named expression whose prefixes
 * cr_inclusive_scan observes (P4229R0, Key Design Points: "reduce observes
 * the root"):
 *   CR_LEFT_FOLD                        ((x0 op x1) op x2) op ...
 *   CR_PAIRWISE, CR_ITERATED_PAIRWISE   tree(x[0..n))  (= cr_reduce with L = 1
 *                                       without init)
 *   CR_BLOCK_DYADIC                     C_{K-1}: C_0 = T_0, C_k = C_{k-1} op T_k
 *                                       over the block trees T_k, K = ceil(n/B)
 * For the policies that are consistent (left_fold, iterated_pairwise,
 * block_dyadic) it equals the inclusive scan's last element; pairwise's last
 * element folds the maximal subtrees from the left instead.
 *   x        device, n >= 1 contiguous elements (an empty expression has no
 *            root: n == 0 is INVALID_ARG)
 *   out_dev  device pointer to one element of dt
 * Workspace from cr_reduce_policy_workspace_bytes (0 for bad arguments). */
size_t cr_reduce_policy_workspace_bytes(int64_t n, cr_policy p, int64_t B, cr_dtype dt);
cr_status cr_reduce_policy(const void* x, int64_t n, cr_policy p, int64_t B, cr_dtype dt,
                           void* out_dev, void* ws, size_t ws_bytes, void* stream);

/* Exclusive scan and the include_initial form (the inclusive/exclusive
 * duality of the page "Vertical scan redesign: research notes", section B.2,
 * with init placed as in P4016R0: combined once, as the left operand, after
 * the named expression). With y the inclusive scan of the same policy:
 *   CR_EXCLUSIVE        m = n outputs:     out[0] = init,
 *                                          out[k] = init op y[k-1], 0 < k < n
 *   CR_INCLUDE_INITIAL  m = n + 1 outputs: out[0] = init,
 *                                          out[k] = init op y[k-1], 0 < k <= n
 * (init = -0.0 gives exactly the inclusive scan moved one place right). */
typedef enum { CR_EXCLUSIVE = 1, CR_INCLUDE_INITIAL = 2 } cr_scan_mode;

/* Workspace bytes for cr_scan_ex(n, p, B, mode, dt); 0 for bad arguments. */
size_t cr_scan_ex_workspace_bytes(int64_t n, cr_policy p, int64_t B, cr_scan_mode mode,
                                  cr_dtype dt);

/* 1-D exclusive / include_initial scan. x: device, n contiguous elements;
 * out: device, m contiguous elements (see above); init_host: host pointer to
 * one element of dt. out == x (in place; for CR_INCLUDE_INITIAL the buffer
 * must hold n + 1 elements) is allowed, any other overlap is INVALID_ARG.
 * n == 0 writes nothing (CR_EXCLUSIVE) or out[0] = init
 * (CR_INCLUDE_INITIAL). Policies and B as for cr_inclusive_scan. */
cr_status cr_scan_ex(const void* x, void* out, int64_t n, cr_policy p, int64_t B,
                     cr_scan_mode mode, const void* init_host, cr_dtype dt, void* ws,
                     size_t ws_bytes, void* stream);

/* Workspace bytes for cr_scan_ex_batched with these sizes. */
size_t cr_scan_ex_batched_workspace_bytes(int64_t batch, int64_t n, cr_policy p, int64_t B,
                                          cr_scan_mode mode, cr_dtype dt);

/* A batch of independent exclusive / include_initial scans: sequence b is
 * x[b*batch_stride + i*elem_stride], i < n; its m outputs go to
 * out[b*out_batch_stride + k*out_elem_stride], k < m. Typical use: the n
 * levels of each column of a level-major array give n + 1 interface values
 * (CR_INCLUDE_INITIAL, out_elem_stride = ncols, out_batch_stride = 1). If
 * out == x the output strides must equal the input strides; otherwise the
 * output must not overlap the input or itself across sequences (a zero
 * out_elem_stride with m >= 2, a zero out_batch_stride with batch >= 2, or
 * out_elem_stride == out_batch_stride with batch >= 2 and m >= 2 is
 * INVALID_ARG, and so is an output that meets the input when both are laid
 * out densely: rows or level-major columns). */
cr_status cr_scan_ex_batched(const void* x, void* out, int64_t batch, int64_t n,
                             int64_t elem_stride, int64_t batch_stride,
                             int64_t out_elem_stride, int64_t out_batch_stride, cr_policy p,
                             int64_t B, cr_scan_mode mode, const void* init_host, cr_dtype dt,
                             void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------- host buffers
 * The same operations with x and out in HOST memory (page-locked memory
 * gives the full host link bandwidth; pageable memory works, slower). The
 * call copies in, computes and copies out, and returns when out is
 * written. For the tiled 1-D scans the copies and the passes are pipelined
 * in chunks over three streams (copy in, compute on `stream`, copy out),
 * so that the transfers overlap the kernels. dev_buf: caller-owned device
 * memory of at least the bytes the query returns (256-byte aligned); it
 * holds the workspace first (its status word at dev_buf itself, so that
 * cr_sync_status(dev_buf, stream) reports on the call), then device copies
 * of x and out. As the call synchronises before it returns, it reports a
 * bounded device-side wait that gave up itself (CR_ERR_TIMEOUT). Errors
 * otherwise as for the device forms. */
size_t cr_inclusive_scan_host_workspace_bytes(int64_t n, cr_policy p, int64_t B, cr_dtype dt);
cr_status cr_inclusive_scan_host(const void* x_host, void* out_host, int64_t n, cr_policy p,
                                 int64_t B, cr_dtype dt, void* dev_buf, size_t dev_bytes,
                                 void* stream);
size_t cr_reduce_host_workspace_bytes(int64_t n, int32_t L, cr_dtype dt);
cr_status cr_reduce_host(const void* x_host, int64_t n, int32_t L, const void* init_host,
                         cr_dtype dt, void* out_host, void* dev_buf, size_t dev_bytes,
                         void* stream);

/* Host-buffer forms of the batched calls: the same operations and strides
 * as cr_reduce_batched and cr_inclusive_scan_batched, with x and out in host
 * memory. The batch is moved in groups of whole sequences (about 16 MB each,
 * at most 16): each group is copied in, computed and copied out on three
 * streams ordered by events, so that transfers overlap kernels; the call
 * returns when out is written. Host layouts: sequences contiguous
 * (elem_stride 1, batch_stride >= n: rows) or element k of every sequence
 * contiguous (batch_stride 1, elem_stride >= batch: columns of a level-major
 * array); any other layout is CR_ERR_UNSUPPORTED. The scan's out uses x's
 * strides; out == x (in place) is allowed, any other overlap of their
 * address ranges is INVALID_ARG (for the reduce, out_host's batch elements
 * must not meet x's range). dev_buf: caller-owned device memory of at least
 * the bytes the query returns (256-byte aligned), laid out and reporting
 * CR_ERR_TIMEOUT as for the 1-D host-buffer forms above. Errors otherwise
 * as for the device forms. */
size_t cr_reduce_batched_host_workspace_bytes(int64_t batch, int64_t n, int32_t L,
                                              cr_dtype dt);
cr_status cr_reduce_batched_host(const void* x_host, void* out_host, int64_t batch, int64_t n,
                                 int64_t elem_stride, int64_t batch_stride, int32_t L,
                                 const void* init_host, cr_dtype dt, void* dev_buf,
                                 size_t dev_bytes, void* stream);
size_t cr_inclusive_scan_batched_host_workspace_bytes(int64_t batch, int64_t n, cr_policy p,
                                                      int64_t B, cr_dtype dt);
cr_status cr_inclusive_scan_batched_host(const void* x_host, void* out_host, int64_t batch,
                                         int64_t n, int64_t elem_stride, int64_t batch_stride,
                                         cr_policy p, int64_t B, cr_dtype dt, void* dev_buf,
                                         size_t dev_bytes, void* stream);

/* Allocation-free canonical reduction. The paper has no counterpart: this
 * serves callers that cannot allocate device memory, such as a plugin whose
 * host framework owns all device memory through its own pool, or a
 * latency-critical path that must not pay cudaMalloc's possible
 * device-wide synchronisation. Same result and arguments as cr_reduce(), but
 * no workspace argument: the scratch is one 16 MiB device array built into
 * libcr, present on every GPU that loads the library until the process
 * exits.
 *   - Calls whose cr_reduce_workspace_bytes(n, L, dt) exceeds 16 MiB return
 *     CR_ERR_WORKSPACE and enqueue nothing (every n <= 2^28 fits for
 *     L <= 4096).
 *   - Each call that is not being captured into a CUDA graph looks up the
 *     array's device address on the current device (so the address stays
 *     right after cudaDeviceReset); a call made during stream capture reuses
 *     the address found by an earlier call on that device, so make the first
 *     call on a device before any stream capture (otherwise
 *     CR_ERR_UNSUPPORTED).
 *   - All calls on a device share the one array, which keeps the previous
 *     call's contents: two calls that may overlap on the GPU (different
 *     streams, no ordering between them) race and give wrong results.
 *     Serialise them, e.g. on one stream.
 *   - It allocates no device memory and frees none. */
cr_status cr_reduce_noalloc(const void* x, int64_t n, int32_t L, const void* init_host,
                            cr_dtype dt, void* out_dev, void* stream);

/* ------------------------------------------------------------- utilities */

/* Synchronises `stream`, then reports the device-side status of the most
 * recent call that used `ws`: CR_ERR_TIMEOUT if one of its bounded
 * cross-block waits gave up (the output is then incomplete), CR_ERR_CUDA if
 * the stream reports an error, else CR_OK. */
cr_status cr_sync_status(void* ws, void* stream);

/* Static text for a status code. */
const char* cr_status_string(cr_status s);

/* Library version as major*10000 + minor*100 + patch. */
int cr_version(void);

/* ----------------------------------------------------------- diagnostics
 * Not part of the pages' operations: launch accounting used by the
 * benchmark and by profiling tools. */

/* Number of kernels libcr has enqueued since it was loaded. */
uint64_t cr_launch_count(void);

/* on != 0: every later launch is bracketed by two CUDA events recorded on its
 * stream (a small per-launch cost); on == 0: stop recording. */
void cr_profile_enable(int on);

/* Restricts the recording of cr_profile_enable to the launches of one kernel
 * (an id as cr_kernel_name() takes), so that a timed sequence of calls
 * carries the events of that kernel only; -1 (or any id out of range)
 * records every kernel again. Process-wide. */
void cr_profile_select(int kernel_id);

/* Waits for the recorded events, writes up to max_records (kernel id, device
 * milliseconds) pairs in launch order, forgets them and returns how many
 * launches were recorded (possibly more than max_records). */
int cr_profile_collect(int* kernel_ids, float* ms, int max_records);

/* Test hook for the bounded waits: while tile >= 0, the single-pass
 * iterated_pairwise scan's tile number `tile` (2048 elements each, counted
 * in start order) does not publish its aggregate, so the tiles that need it
 * give up waiting and the call's cr_sync_status() reports CR_ERR_TIMEOUT
 * (the output is then wrong). -1 turns it off. Process-wide. */
void cr_debug_skip_publish(int64_t tile);

/* Test hook for the block_dyadic scans with 2 <= B <= 2048 whose block
 * carries take the parallel exact chain (inclusive, out != x). For B <= 16
 * the chain's evaluation and the carry fix-up run as one cooperative pass
 * by default; for larger B as separate passes. mode 0: that default; 1: the
 * separate passes for every B; 2: the fused pass for every B, with a
 * validation failure raised once the chain's walk is half-way, so that its
 * recovery (the local pass again, the serial chain, the fix-up again) runs;
 * 3: the fused pass for every B; 4: the fused pass for every B, taken as if
 * the device had refused its cooperative launch, so that the fallback to
 * the separate passes and a plain fix-up runs. Modes 0, 1, 2 and 4 apply to
 * the 1-D left fold too, which runs the fused pass without a fix-up. Every
 * mode gives the same, exact output.
 * Process-wide. */
void cr_debug_fused_fixup(int mode);

/* Static name of a kernel id returned by cr_profile_collect(). */
const char* cr_kernel_name(int id);

/* Device scratch bytes cr_measure_add_peak() needs on the current device
 * (0 if no device is usable). */
size_t cr_measure_add_peak_scratch_bytes(void);

/* Measures, on the current device and `stream`, the throughput of
 * independent round-to-nearest adds of dt (adds per second over all SMs) and
 * the latency of one dependent chain of them (ns per add): the ALU roofline
 * denominators of add-bound kernels. Synchronises the stream. scratch_dev:
 * caller-owned device memory of at least the bytes above. Either output
 * pointer may be NULL. */
cr_status cr_measure_add_peak(cr_dtype dt, void* scratch_dev, size_t scratch_bytes,
                              void* stream, double* adds_per_second,
                              double* dependent_latency_ns);

/* out[i] = a[i] + b[i] (binary64, round to nearest even) computed by libcr's
 * integer-pipe add, written from the IEEE-754 definition of the operation
 * (device pointers, n elements, enqueued on `stream`). A measured
 * alternative to the FP64 pipe that the kernels do not use; exposed so that
 * it can be checked bit for bit against the hardware add. */
cr_status cr_add_pairs_int(const double* a, const double* b, double* out, int64_t n,
                           void* stream);

/* Throughput of that integer-pipe add over all SMs (adds per second; same
 * scratch as cr_measure_add_peak). Synchronises the stream. */
cr_status cr_measure_int_add_rate(void* scratch_dev, size_t scratch_bytes, void* stream,
                                  double* adds_per_second);

#ifdef __cplusplus
}
#endif

#endif /* CR_H_ */
