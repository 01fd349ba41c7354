/*
 * lora_delta.h -- C ABI of the batch-invariant shared LoRA delta operator
 * (GB300 / sm_103a).
 *
 * The operator (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton,
 * both batch-invariant", section "Summary"):
 *
 *   forward    U        = X @ A^T          FP32 accumulate, rounded to BF16
 *              delta_y  = (U @ B^T) * alpha FP32 accumulate, FP32 output
 *   backward   dV = dY * alpha  (rounded to BF16)    dU = dV @ B (rounded to BF16)
 *              dB = dV^T @ U    dX = dU @ A    dA = dU^T @ X   (FP32)
 *
 * No base weight enters either call, so none can be read or given a gradient
 * (same page, "Acceptance criteria", items 2 and 3).
 *
 * Numerics. Every sum is formed from 16-term tensor-core dot products
 * ("leaves": BF16 products, FP32 accumulation, a fresh accumulator each),
 * added in FP32 round-to-nearest by the canonical pairwise tree over the leaf
 * index. The tree depends only on the length of the reduction, never on M,
 * on the tiling or on the device, and no atomics are used: every row of U,
 * delta_y, dU and dX is bitwise independent of the other rows in the batch
 * (batch invariance: same page, "Batch invariance"), and every output is
 * bitwise identical across reruns.
 *
 * Conventions for every entry point:
 *   - Tensors are dense, row-major, contiguous, in device memory (or memory
 *     the device can address), 16-byte aligned. BF16 tensors are passed as
 *     `const void *` (IEEE bfloat16 bit patterns, 2 bytes each).
 *   - Shapes: M >= 0 (batch rows; M = 0 is a no-op returning LORA_OK),
 *     K and N positive multiples of 8, R a multiple of 8 in [8, 64];
 *     M, K, N below 2^31.
 *   - The caller owns every buffer and the stream; the library never
 *     allocates, frees or synchronises. Work is enqueued on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream) of the current device
 *     and the call returns without waiting for it.
 *   - Argument errors are detected on the host before anything is enqueued.
 *   - `workspace` is scratch owned by the caller, at least the size the
 *     matching *_workspace_size() query returns, 256-byte aligned. It starts
 *     with a control block of LORA_DELTA_CONTROL_BYTES, which must be zero
 *     before the first call that uses the workspace (for example, allocate
 *     the workspace zeroed): a 256-byte device status block, then control
 *     words of lora_delta_fwd_fused (work tickets, row-tile counters),
 *     which every call leaves at zero again, also a call whose kernels gave
 *     up on a wait. The rest is scratch that no call reads before writing, so
 *     a workspace serves calls of any shape that fit in it. The status
 *     block's 32-bit words:
 *       word 0  status: a kernel that gives up on an internal wait (every wait
 *               is bounded, 0.1 s by default) writes (site << 8) | 1 there, unless
 *               the word already holds a code (the first failure stays), and
 *               returns; the call's outputs are then undefined. The code stays
 *               until the caller clears the word (read it with
 *               lora_delta_device_status). No kernel of the default schedule
 *               waits for another CTA (those of the cluster schedules wait only
 *               for CTAs of their own cluster, which run together), and nothing
 *               else in the block carries state from call to call, so a call
 *               after a timed-out one needs no reset to run correctly.
 *       word 2  test hook, 0 for normal use: a kernel kind (1 down-projection,
 *               2 up-projection / dX, 3 fused dU + dB pass, 4 weight gradients)
 *               whose producer warp first waits on a barrier that nothing
 *               completes, so that the wait runs out (failure-path tests; the
 *               launch that writes dX and the dA partials for R <= 16 answers
 *               to kinds 2 and 4).
 *       word 3  test hook, 0 for normal use: the wait limit in microseconds.
 *     The library never writes words 2 and 3. A workspace must not be shared
 *     by calls that may run concurrently.
 *   - The library keeps per-device state for the life of the process (kernel
 *     attributes set on first use, the device address of the no-allocation
 *     scratch array). It does not survive cudaDeviceReset or a reset of the
 *     device's primary context: do not call the library after either.
 */
#ifndef LORA_DELTA_H
#define LORA_DELTA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes at the start of every workspace that must be zero before its first use. */
#define LORA_DELTA_CONTROL_BYTES (256 + 65536)

typedef enum lora_status {
  LORA_OK = 0,
  LORA_ERR_NULL = 1,       /* a required pointer is NULL */
  LORA_ERR_SHAPE = 2,      /* M < 0, K or N not a positive multiple of 8, or a size too large */
  LORA_ERR_ALIGN = 3,      /* a tensor or the workspace is not aligned as required */
  LORA_ERR_RANK = 4,       /* R not a multiple of 8 in [8, 64] */
  LORA_ERR_WORKSPACE = 5,  /* workspace smaller than the query returned */
  LORA_ERR_CUDA = 6,       /* a CUDA runtime or driver call failed (incl. kernel launch) */
  LORA_ERR_DEVICE = 7,     /* the current device is not an sm_103 (GB300) GPU */
  LORA_ERR_TIMEOUT = 8     /* a kernel gave up waiting (read from the status block) */
} lora_status;

/*
 * Forward pass.
 *   x        [M][K] bf16   input rows
 *   a        [R][K] bf16   down projection A (used as A^T)
 *   b        [N][R] bf16   up projection B (used as B^T)
 *   alpha                  scale, applied as one FP32 multiply after the FP32 sum
 *   delta_y  [M][N] fp32   out: (U @ B^T) * alpha
 *   u        [M][R] bf16   out: U = bf16(X @ A^T), saved for the backward pass
 *   workspace, workspace_bytes: >= lora_delta_fwd_workspace_size(M, K, N, R)
 * Kernels: down-projection (U partials over K-slices), rows (adds the partials
 * into U and writes u), up-projection (expands u to delta_y).
 */
lora_status lora_delta_fwd(const void *x, const void *a, const void *b, float alpha, int64_t M, int64_t K, int64_t N,
                           int64_t R, float *delta_y, void *u, void *workspace, size_t workspace_bytes, void *stream);

/*
 * The forward pass in a single launch (the fusion of the two GEMMs asked for in
 * the review thread of page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA +
 * Triton, both batch-invariant"; U is still stored). Arguments, outputs, bits,
 * workspace and errors are those of lora_delta_fwd (y_bf16 != 0: a BF16
 * delta_y, as lora_delta_fwd_bf16). Inside the launch the three steps of
 * lora_delta_fwd are ordered by claimed work and counters in the workspace's
 * control block, not by grid barriers: down-projection units are claimed from a
 * ticket counter, a row tile's U rows are formed once all of its slice
 * partials are counted, and an up-projection unit starts once its row tile is
 * flagged ready. No CTA ever waits for work held by a CTA that is not running,
 * so the launch needs no co-residency. Batches of more than 4096 row tiles of
 * 128 rows run the three launches of lora_delta_fwd instead. On a GB300 the
 * three launches of lora_delta_fwd are the faster of the two at every shape
 * measured (the counters and flags cost as much as the launch boundaries they
 * replace); this call exists for callers that want a single launch.
 */
lora_status lora_delta_fwd_fused(const void *x, const void *a, const void *b, float alpha, int64_t M, int64_t K,
                                 int64_t N, int64_t R, void *delta_y, void *u, int y_bf16, void *workspace,
                                 size_t workspace_bytes, void *stream);

/*
 * Forward pass with a BF16 delta_y: the half-size output a reviewer asks for
 * in the review thread of page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA +
 * Triton, both batch-invariant" (the FP32 output doubles the bytes of the
 * widest tensor; casting inside the operator adds one rounding).
 *   delta_y  [M][N] bf16   out: bf16((U @ B^T) * alpha), the FP32 result of
 *                          lora_delta_fwd rounded to nearest even: bit for bit
 *                          that FP32 output converted to BF16
 * Every other argument, the workspace, u and the error behaviour are those of
 * lora_delta_fwd (delta_y must be 16-byte aligned as well).
 */
lora_status lora_delta_fwd_bf16(const void *x, const void *a, const void *b, float alpha, int64_t M, int64_t K,
                                int64_t N, int64_t R, void *delta_y, void *u, void *workspace, size_t workspace_bytes,
                                void *stream);

/*
 * Backward pass with a binary32 dY (the FP32-dY input variant; its BF16-output
 * counterpart is asked for in the review thread of page "[DSv4][P5-3]
 * shared_grouped_lora_delta: CUDA + Triton, both batch-invariant").
 *   dy       [M][N] fp32   upstream gradient; dV = bf16(fp32(dy * alpha))
 * Every other argument, output and error is that of lora_delta_bwd; the
 * workspace (lora_delta_bwd_f32dy_workspace_size) also holds dV, written by a
 * first launch and read by the backward kernels as their dY with alpha = 1.
 * When every dy value is representable in BF16 the outputs are bit for bit
 * those of lora_delta_bwd on that BF16 dY.
 */
size_t lora_delta_bwd_f32dy_workspace_size(int64_t M, int64_t K, int64_t N, int64_t R);
lora_status lora_delta_bwd_f32dy(const float *dy, const void *x, const void *a, const void *b, const void *u,
                                 float alpha, int64_t M, int64_t K, int64_t N, int64_t R, float *dx, float *da,
                                 float *db, void *du, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Grouped calls: up to 4 independent sites (LoRA insertion points, e.g. the
 * fc1 and fc2 adapters of one MLP, page "[DSv4][P5-3] shared_grouped_lora_delta:
 * CUDA + Triton, both batch-invariant", section "Summary": one operator for a
 * group of sites) of the same rank R, each with its own M, K, N, alpha and
 * buffers, in the launches of one single-site call: every kernel deals the
 * work units of all sites out as one space. Each site's results are bit for
 * bit those of the single-site call on the same arguments. Sites with M = 0
 * are skipped; count outside [1, 4] is LORA_ERR_SHAPE; the argument checks and
 * errors are those of the single-site calls, applied to every site.
 */
typedef struct lora_fwd_site {
  const void *x, *a, *b;   /* [M][K], [R][K], [N][R] bf16 */
  float alpha;
  int64_t M, K, N;
  void *delta_y;           /* [M][N] out: fp32, or bf16 when the call's y_bf16 is set */
  void *u;                 /* [M][R] bf16 out */
} lora_fwd_site;

typedef struct lora_bwd_site {
  const void *dy, *x, *a, *b, *u;   /* [M][N], [M][K], [R][K], [N][R], [M][R] bf16 */
  float alpha;
  int64_t M, K, N;
  float *dx, *da, *db;     /* [M][K], [R][K], [N][R] fp32 out */
  void *du;                /* [M][R] bf16 out */
} lora_bwd_site;

/* Workspace bytes of a grouped call (0: invalid count or shape). */
size_t lora_delta_fwd_grouped_workspace_size(const lora_fwd_site *sites, int count, int64_t R);
size_t lora_delta_bwd_grouped_workspace_size(const lora_bwd_site *sites, int count, int64_t R);

/* Forward of every site (three launches: down, rows, up, each over all sites' units); y_bf16:
 * every delta_y is BF16 (as lora_delta_fwd_bf16). */
lora_status lora_delta_fwd_grouped(const lora_fwd_site *sites, int count, int64_t R, int y_bf16, void *workspace,
                                   size_t workspace_bytes, void *stream);
/* Backward of every site (the launches of one lora_delta_bwd). */
lora_status lora_delta_bwd_grouped(const lora_bwd_site *sites, int count, int64_t R, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * Backward pass (no base-weight gradient).
 *   dy       [M][N] bf16   upstream gradient of delta_y
 *   x, a, b               as in the forward pass
 *   u        [M][R] bf16   the U the forward pass returned
 *   alpha                  the forward scale
 *   dx       [M][K] fp32   out: dU @ A
 *   da       [R][K] fp32   out: dU^T @ X
 *   db       [N][R] fp32   out: dV^T @ U
 *   du       [M][R] bf16   out: dU = bf16(dV @ B), dV = bf16(dY * alpha)
 *   workspace, workspace_bytes: >= lora_delta_bwd_workspace_size(M, K, N, R)
 * dA and dB reduce over all M rows in fixed 256-row chunks whose partials are
 * added by the canonical pairwise tree over the chunk index.
 * Kernels: dU and dB partials (one pass over dY for R <= 16), rows (adds the
 * dU partials into dU and writes du; its other blocks add the dB chunk
 * partials into db while they are still in L2), dX, dA partials, combine (dA).
 */
lora_status lora_delta_bwd(const void *dy, const void *x, const void *a, const void *b, const void *u, float alpha,
                           int64_t M, int64_t K, int64_t N, int64_t R, float *dx, float *da, float *db, void *du,
                           void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes the calls need (0 if the shape is invalid). */
size_t lora_delta_fwd_workspace_size(int64_t M, int64_t K, int64_t N, int64_t R);
size_t lora_delta_bwd_workspace_size(int64_t M, int64_t K, int64_t N, int64_t R);
/* The same two queries under the shorter names of the boundary's first
 * description (same results). */
size_t lora_delta_fwd_workspace(int64_t M, int64_t K, int64_t N, int64_t R);
size_t lora_delta_bwd_workspace(int64_t M, int64_t K, int64_t N, int64_t R);

/* Static description of a status code (unknown codes give "unknown status"). */
const char *lora_status_str(lora_status status);

/*
 * Reads the device status block at the start of `workspace` (synchronous:
 * waits for the device). *code receives 0 when no kernel reported a problem,
 * else (site << 8) | 1 for a wait that timed out at internal site `site`.
 * Returns LORA_OK, LORA_ERR_NULL or LORA_ERR_CUDA; LORA_ERR_TIMEOUT when
 * *code is non-zero.
 */
lora_status lora_delta_device_status(const void *workspace, int *code);

/*
 * Profiling hook (process-wide; not thread-safe). When count > 0, later
 * forward and backward calls record events[0] (cudaEvent_t) before their
 * first kernel and events[i] after their i-th kernel, up to count - 1
 * kernels, on the call's stream. count = 0 switches it off. The events stay
 * owned by the caller.
 */
lora_status lora_delta_set_profile_events(void *const *events, int count);

/*
 * Schedule of the passes (process-wide; not thread-safe; no effect on any
 * result bit -- every schedule runs the same leaves, trees and rounding
 * points). The operator's steps can be grouped into launches three ways:
 *   LORA_SCHEDULE_SEPARATE: forward down-projection, rows, up-projection;
 *     backward dU + dB pass, rows (with the dB tree), dX and the dA partials
 *     (one launch for R <= 16, two above), combine.
 *   LORA_SCHEDULE_CLUSTER_REDUCE: the reductions that feed a BF16 row on
 *     thread-block clusters -- a cluster of `cluster_size` CTAs shares each
 *     128-row tile (forward: U partials and the U rows) or 256-row chunk
 *     (backward, R <= 16: the dU + dB pass and the dU rows), the CTAs meeting
 *     at mbarriers in each other's shared memory instead of at a launch
 *     boundary -- then the expansion (forward) or the dX and dA launch
 *     (backward) and one combine launch for dA and dB.
 *   LORA_SCHEDULE_CLUSTER_SINGLE: the forward in one cluster launch (each CTA
 *     also expands its share of the tile's columns of delta_y); the backward
 *     (R <= 16) in one cluster launch (each CTA also writes its share of dX and
 *     the dA chunk partials) and the combine launch.
 *   LORA_SCHEDULE_AUTO (the default): the forward as separate launches; the
 *     single-site backward of R <= 16 as cluster reductions where its 256-row
 *     chunks give at least three quarters of the SMs a CTA (on a GB300, M of
 *     about 7300 rows and more with clusters of 4), else as separate launches --
 *     the faster choice at every shape measured. (Under
 *     LORA_SCHEDULE_CLUSTER_REDUCE, batches with too few chunks for that take
 *     128-row units.)
 * The cluster schedules cover the single-site forward of R <= 32 and the
 * single-site backward of R <= 16 whose per-CTA share of a tile is at most
 * 32 MiB of input; other calls (grouped calls included) run the separate
 * launches. cluster_size is 0 (the default size, 4 CTAs), 2, 4 or 8. Returns
 * LORA_ERR_SHAPE, leaving the setting unchanged, for any other value.
 * lora_delta_schedule returns the current schedule and stores the cluster
 * size setting in *cluster_size (if not NULL).
 */
#define LORA_SCHEDULE_SEPARATE 0
#define LORA_SCHEDULE_CLUSTER_REDUCE 1
#define LORA_SCHEDULE_CLUSTER_SINGLE 2
#define LORA_SCHEDULE_AUTO 3
lora_status lora_delta_set_schedule(int schedule, int cluster_size);
int lora_delta_schedule(int *cluster_size);

/*
 * The launch plan a single-site call of this shape takes on the current device under the
 * current schedule setting (backward != 0: lora_delta_bwd, else lora_delta_fwd): the
 * schedule actually used (LORA_SCHEDULE_SEPARATE, _CLUSTER_REDUCE or _CLUSTER_SINGLE) and the
 * number of kernel launches it enqueues (0 for M = 0). Returns the call's shape errors, or
 * LORA_ERR_DEVICE / LORA_ERR_CUDA when the current device cannot run the operator.
 */
lora_status lora_delta_plan(int backward, int64_t M, int64_t K, int64_t N, int64_t R, int *schedule, int *launches);

/*
 * Writes a NUL-terminated JSON description of the numerics and tiling
 * (provenance) into buf (at most len bytes). Returns the length it needs.
 */
size_t lora_delta_describe(char *buf, size_t len);

/*
 * Forward pass for callers that cannot allocate device memory -- code that
 * must not go around an allocator it does not own (a framework's caching
 * allocator, a server that plans every device byte in advance) or a host
 * program with no allocator of its own where the call is made. The pages have
 * no counterpart to this call: it exists only for such callers.
 *
 * Same arguments, outputs and numerics as lora_delta_fwd, without the
 * workspace: the scratch (status block and FP32 partial sums of U) comes from
 * one fixed 16 MiB array in the library's device image, which every device
 * that loads the library holds until the process exits. Shapes whose
 * lora_delta_fwd_workspace_size exceeds 16 MiB are rejected with
 * LORA_ERR_WORKSPACE before anything is enqueued. The call allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture. Every call clears the status block on `stream` and then shares the
 * same array: calls whose work may overlap on the GPU (other streams, other
 * threads) race on it and must be serialised by the caller.
 */
lora_status lora_delta_fwd_noalloc(const void *x, const void *a, const void *b, float alpha, int64_t M, int64_t K,
                                   int64_t N, int64_t R, float *delta_y, void *u, void *stream);

/*
 * Status block of lora_delta_fwd_noalloc on the current device (the caller has
 * no workspace to pass to lora_delta_device_status). Synchronous: waits for the
 * whole device, then reads the block that the latest lora_delta_fwd_noalloc call
 * on this device used; the next call clears it again. *code and the return value
 * as for lora_delta_device_status (0 and LORA_OK when no kernel gave up, also
 * when no lora_delta_fwd_noalloc call has run on this device yet).
 */
lora_status lora_delta_fwd_noalloc_status(int *code);

/*
 * Exact mode of the weight gradients (page "det-train", sections "Method",
 * "API" and "Correctness": a Kulisch long accumulator per output, partials
 * composed by adding digit arrays, one rounding to FP32 at the end).
 *
 *   dA[r][k] = rn32( sum_m du[m][r] * x[m][k] )
 *   dB[n][r] = rn32( sum_m dv[m][n] * u[m][r] ),  dv = bf16(fp32(dy[m][n] * alpha))
 *
 * where the sums are exact (every BF16 product is exact; the products are
 * added as integers) and rn32 rounds to nearest even once. So dA and dB do not
 * depend on the order of the rows, on the chunking or on how the rows are
 * split between calls: the digit arrays of row shards, added with
 * lora_delta_exact_combine (in any grouping), give the digit arrays of the
 * whole, and lora_delta_exact_finalize rounds those to the same bits. Special
 * values: a NaN product (a NaN factor, or inf * 0), or both an infinite
 * positive and an infinite negative product, gives NaN; otherwise an infinite
 * product gives that infinity; a sum beyond the FP32 range rounds to infinity;
 * an exact zero sum is +0.
 *
 * Digit array: lora_delta_exact_slots() (= 21) int64 per output: 18 digits in
 * radix 2^32, digit i weighing 2^(32 i - 266) (the bottom of the BF16 product
 * range), then the counts of +inf, -inf and NaN products. The library writes
 * them normalised (digits 0..16 in [0, 2^32), digit 17 signed), so equal sums
 * give equal arrays, byte for byte.
 *
 * lora_delta_grads_exact: inputs as in lora_delta_bwd (du is the du output of
 * the backward pass). Outputs, each optional (NULL: not written):
 *   da        [R][K] fp32      da_digits [R][K][21] int64
 *   db        [N][R] fp32      db_digits [N][R][21] int64
 * dA is computed when da or da_digits is given, dB when db or db_digits is;
 * the inputs it reads must then be non-NULL (x, du for dA; dy, u for dB) unless
 * M = 0, which writes zero gradients (+0, and all-zero digit arrays).
 * M < 2^30 (digit headroom); R * K and R * N below 2^31. workspace: at least
 * lora_delta_grads_exact_workspace_size bytes of scratch (no status block: no
 * kernel of this call waits). Kernels: per gradient, the digit kernel (integer
 * accumulation over 64-row units of 16 x 64 output tiles) and the reduce kernel
 * (adds the units' windows and digits, normalises, rounds); with profile events
 * set, events[0] is recorded before dA, events[1] after it, events[2] after dB.
 * The call is much slower than lora_delta_bwd's dA and dB: integer units, not
 * tensor cores.
 */
int lora_delta_exact_slots(void);
size_t lora_delta_grads_exact_workspace_size(int64_t M, int64_t K, int64_t N, int64_t R);
lora_status lora_delta_grads_exact(const void *dy, const void *x, const void *u, const void *du, float alpha,
                                   int64_t M, int64_t K, int64_t N, int64_t R, float *da, float *db,
                                   int64_t *da_digits, int64_t *db_digits, void *workspace, size_t workspace_bytes,
                                   void *stream);

/*
 * The exact mode with a binary32 dY (as lora_delta_bwd_f32dy): dV = bf16(fp32(dy * alpha))
 * is formed by a first launch into the workspace (after the digit kernel's scratch), and
 * the exact pass reads it with alpha = 1. dy [M][N] fp32; everything else as for
 * lora_delta_grads_exact; workspace >= lora_delta_grads_exact_f32dy_workspace_size bytes.
 */
size_t lora_delta_grads_exact_f32dy_workspace_size(int64_t M, int64_t K, int64_t N, int64_t R);
lora_status lora_delta_grads_exact_f32dy(const float *dy, const void *x, const void *u, const void *du, float alpha,
                                         int64_t M, int64_t K, int64_t N, int64_t R, float *da, float *db,
                                         int64_t *da_digits, int64_t *db_digits, void *workspace,
                                         size_t workspace_bytes, void *stream);

/*
 * out_digits = a + b over n digit arrays (n outputs, 21 int64 each), written
 * normalised; out_digits may be a or b (in place). b NULL: out_digits = a,
 * normalised (e.g. after an int64 sum all-reduce of digit arrays across ranks,
 * the det-train page's det_all_reduce). Inputs may be normalised or not, as
 * long as every sum of a digit stays within int64 (digit arrays of fewer than
 * 2^30 rows in all). Returns LORA_ERR_SHAPE for n < 0 or n >= 2^38; n = 0 is a
 * no-op.
 */
lora_status lora_delta_exact_combine(const int64_t *a, const int64_t *b, int64_t n, int64_t *out_digits,
                                     void *stream);

/* out[i] = FP32 value of digit array i (rounded to nearest even, once), i < n;
 * n as for lora_delta_exact_combine. */
lora_status lora_delta_exact_finalize(const int64_t *digits, int64_t n, float *out, void *stream);

/*
 * Measurement aid: the rate at which this device performs the exact mode's
 * product step (one 32-bit by 32-bit multiply-add into a 64-bit sum per
 * product), the ceiling of lora_delta_grads_exact's digit kernel. Enqueues one
 * launch in the digit kernel's shape that performs *products independent such
 * multiply-adds (iters rounds per chain, 1 <= iters < 2^31); time it with CUDA
 * events on `stream`. sink: device scratch of at least
 * lora_delta_exact_rate_probe_sink_bytes() bytes (16-byte aligned; its
 * contents are meaningless), which the launch writes so that no work can be
 * dropped. The sink-size query returns 0 when the current device is unusable.
 */
lora_status lora_delta_exact_rate_probe(int64_t iters, void *sink, size_t sink_bytes, int64_t *products,
                                        void *stream);
size_t lora_delta_exact_rate_probe_sink_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* LORA_DELTA_H */
