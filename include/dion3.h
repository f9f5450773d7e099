/*
 * dion3.h - C ABI of the Dion3 optimizer step on one GB300 (sm_103a).
 *
 * The Dion3 step (source: "Dion3: Full-Stack Orthogonal Updates", the agihunt
 * summary of the paper, paragraphs on the first level - Gram Newton-Schulz -
 * and the third level - fractional row selection) for one n x m matrix:
 *
 *   (a) M <- M + G on every row; S = the k = ceil(f n) rows of M with the
 *       largest l1 norm (ties to the lower row index), ascending;
 *   (b) X = M[S] / (||M[S]||_F + eps) in fp16; Gram Newton-Schulz: R = X X^T,
 *       T iterations of Z = aI + bR + cR^2, Q <- Z Q, R <- Z R Z, a restart
 *       before iteration `restart_iter` (X <- Q X, R = X X^T, Q <- I), and
 *       O = Q X at the end (on X^T when k > m: the Gram matrix is formed on the
 *       short side);
 *   (c) W[S] <- W[S] - (lr / sqrt(f)) O; M[S] <- mu M[S]; other rows of W and
 *       M are not touched (error feedback).
 *
 * Conventions shared by every entry point:
 *   - Memory: every tensor and the workspace is caller-owned DEVICE memory; the
 *     library never allocates device memory (its only CUDA objects are a small
 *     per-device pool of streams and events, made on first use by
 *     dion3_step / dion3_step_lazy with several groups, and the events of the
 *     launch trace).  Arrays of pointers (dion3_group.params, ...) are HOST
 *     arrays read during the call only.
 *   - Layout: matrices are dense row-major with row pitch == cols; each device
 *     pointer must be 16-byte aligned; the workspace 256-byte aligned.
 *   - Ordering: every call only enqueues work on `stream` (or on library
 *     streams forked from it and joined back into it before the call returns)
 *     and returns without synchronising; results are visible to later work on
 *     the same stream.
 *     Calls that share one workspace must not overlap on the device.  Since a
 *     call enqueues kernel launches only (no host synchronisation, no
 *     allocation), it can be captured in a CUDA graph and replayed.  The
 *     tensor-core kernels are launched with programmatic dependent launch
 *     (their set-up may overlap the end of the previous kernel on the stream;
 *     they read nothing before it has completed); the environment variable
 *     DION3_PDL=0 turns that off.
 *   - Errors: arguments are validated on the host before the first launch; an
 *     invalid call returns a status != DION3_OK, enqueues nothing and leaves
 *     every tensor untouched.  A failed launch returns DION3_ERR_CUDA.
 *     dion3_last_error() gives a one-line description (per host thread).
 *   - Device-side waits in the tensor-core kernels are bounded (about one
 *     second); a wait that runs out records DION3_ERR_TIMEOUT in a device
 *     status word that dion3_device_status() reads.
 *   - Exceptions never cross this boundary.
 *   - Per-device state: the library looks up, once per device, the device
 *     addresses of its own static device variables (the status word, the
 *     scratch of dion3_select_rows_noalloc) and keeps them, with its stream
 *     pool, for the life of the process.  After cudaDeviceReset on a device
 *     those addresses are stale, so a process must not call the library on
 *     that device again.
 */
#ifndef DION3_H_
#define DION3_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DION3_ABI_VERSION 1

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* dion3_stream_t;

typedef enum {
  DION3_OK = 0,
  DION3_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad hyperparameter, misalignment */
  DION3_ERR_UNSUPPORTED = 2,  /* valid request that this build does not implement */
  DION3_ERR_WORKSPACE = 3,    /* workspace null or smaller than the *_workspace_size query */
  DION3_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  DION3_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out (see dion3_device_status) */
  DION3_ERR_DEVICE_CHECK = 6  /* a device-side consistency check failed */
} dion3_status;

typedef enum { DION3_F32 = 0, DION3_BF16 = 1, DION3_F16 = 2 } dion3_dtype;

/*
 * Hyperparameters of one step.
 *   f            fraction of rows orthogonalised, 0 < f <= 1; k = ceil(f n)
 *                (third-level paragraph of the summary page).
 *   mu           decay of the selected momentum rows (error feedback).
 *   lr           base learning rate; the applied rate is lr / sqrt(f), computed
 *                in double on the host and passed to the kernels as fp32.
 *   eps          X / (||X||_F + eps) before Newton-Schulz.
 *   ns_steps     T >= 1 Newton-Schulz iterations.
 *   restart_iter 0 for no restart, else 2..T: the 1-based iteration the
 *                restart comes before (the pages restart at iteration 3).
 *   a, b, c      the polynomial Z = aI + bR + cR^2.
 *   ns_dtype     16-bit type of the Gram-NS operands and intermediates (fp32
 *                accumulation): DION3_F16 (the pages' choice) or DION3_BF16.
 *                Other values return DION3_ERR_UNSUPPORTED.
 */
typedef struct {
  float f;
  float mu;
  float lr;
  float eps;
  int32_t ns_steps;
  int32_t restart_iter;
  float a, b, c;
  int32_t ns_dtype;
} dion3_hparams;

/*
 * A shape group ("megabatch"): `batch` matrices of the same rows x cols, all
 * with the same dtypes, stepped by batched launches.
 *   params      host array [batch] of device pointers to W (param_dtype:
 *               DION3_F32 or DION3_BF16), updated in place.
 *   grads       host array [batch] of device pointers to G (grad_dtype:
 *               DION3_F32 or DION3_BF16), read only.
 *   momentum    host array [batch] of device pointers to M (fp32), updated in
 *               place.
 */
typedef struct {
  int32_t rows;
  int32_t cols;
  int32_t batch;
  int32_t param_dtype;
  int32_t grad_dtype;
  void* const* params;
  const void* const* grads;
  float* const* momentum;
} dion3_group;

/* DION3_ABI_VERSION of the loaded library. */
size_t dion3_abi_version(void);

/* Static description of a status code (never NULL). */
const char* dion3_status_string(int status);

/* Description of the last error returned on this host thread ("" if none). */
const char* dion3_last_error(void);

/* Number of selected rows k = ceil(f * rows), clamped to [1, rows]; 0 if the
 * arguments are invalid. */
int32_t dion3_num_selected(float f, int32_t rows);

/*
 * Useful FLOPs of the Gram-NS schedule this library runs on one k x m
 * submatrix with `hp` (a triangle counted as half): with s = min(k, m),
 * L = max(k, m), one SYRK costs s^2 L, a symmetric s^3 product s^3 and a
 * rectangular multiply 2 s^2 L.  T = 5 with a restart gives 6 s^2 L + 14 s^3.
 * Returns a negative value for invalid arguments.
 */
double dion3_useful_flops(int32_t k, int32_t m, const dion3_hparams* hp);

/*
 * Workspace bytes needed by dion3_select_rows for `batch` matrices of
 * rows x cols and k selected rows.
 */
dion3_status dion3_select_workspace_size(int32_t rows, int32_t cols, int32_t batch,
                                         int32_t k, size_t* bytes);

/*
 * Step (a) alone: optional accumulation and l1 top-k selection.
 *   momentum  host array [batch] of device pointers to fp32 rows x cols M.
 *   grads     host array [batch] of device pointers to G (grad_dtype), or NULL:
 *             with grads, M <- M + G (fp32, round-to-nearest, every row) first;
 *             with NULL, M is only read.
 *   k         1 <= k <= rows rows selected per matrix.
 *   idx_out   device int32 [batch][k]: selected row indices, ascending.
 *   fro2_out  device fp32 [batch]: sum of squares of the selected rows of M
 *             (||M[S]||_F^2), or NULL.
 * Ties in l1 go to the lower row index.
 */
dion3_status dion3_select_rows(int32_t rows, int32_t cols, int32_t batch,
                               float* const* momentum, const void* const* grads,
                               int32_t grad_dtype, int32_t k, int32_t* idx_out,
                               float* fro2_out, void* ws, size_t ws_bytes,
                               dion3_stream_t stream);

/* Workspace bytes needed by dion3_gram_ns_batched. */
dion3_status dion3_gram_ns_workspace_size(int32_t k, int32_t m, int32_t batch,
                                          const dion3_hparams* hp, size_t* bytes);

/*
 * Step (b) alone: Gram Newton-Schulz of `batch` k x m matrices.
 *   X  device [batch][k][m] in hp->ns_dtype (fp16 or bf16), read only.
 *   O  device [batch][k][m] in hp->ns_dtype: O = GramNS(X / (||X||_F + hp->eps)).
 * Only hp->eps, ns_steps, restart_iter, a, b, c and ns_dtype are used.
 * Operands are fp16 (or bf16) with fp32 accumulation; R, Z, Q and the
 * products are rounded to that type between steps (first-level paragraph: the
 * method runs in float16).
 */
dion3_status dion3_gram_ns_batched(int32_t k, int32_t m, int32_t batch, const void* X,
                                   void* O, const dion3_hparams* hp, void* ws,
                                   size_t ws_bytes, dion3_stream_t stream);

/*
 * Newton-Schulz variants on the same tensor-core kernels, for the comparison
 * the first-level paragraph of the summary page makes (Gram NS saves 55 % of
 * the FLOPs of standard NS with symmetric GEMMs and 68 % of the common
 * implementation without them):
 *   DION3_NS_GRAM            Gram NS, symmetric products on lower tiles (the
 *                            same computation as dion3_gram_ns_batched);
 *   DION3_NS_GRAM_DENSE      Gram NS with every tile of every product;
 *   DION3_NS_STANDARD        standard NS on X (A = X X^T, B = bA + cA^2,
 *                            X <- aX + BX) with symmetric A and A^2;
 *   DION3_NS_STANDARD_DENSE  standard NS with every tile computed.
 * dion3_ns_batched has the arguments and results of dion3_gram_ns_batched
 * plus the variant; restart_iter applies to the Gram variants only.
 * dion3_ns_useful_flops counts a computed triangle as half, full tiles in
 * full (so the dense variants count every product in full); negative on
 * invalid arguments.
 */
typedef enum {
  DION3_NS_GRAM = 0,
  DION3_NS_GRAM_DENSE = 1,
  DION3_NS_STANDARD = 2,
  DION3_NS_STANDARD_DENSE = 3
} dion3_ns_variant;

double dion3_ns_useful_flops(int32_t variant, int32_t k, int32_t m, const dion3_hparams* hp);
dion3_status dion3_ns_workspace_size(int32_t variant, int32_t k, int32_t m, int32_t batch,
                                     const dion3_hparams* hp, size_t* bytes);
dion3_status dion3_ns_batched(int32_t variant, int32_t k, int32_t m, int32_t batch, const void* X,
                              void* O, const dion3_hparams* hp, void* ws, size_t ws_bytes,
                              dion3_stream_t stream);

typedef enum { DION3_GEMM_RECT = 0, DION3_GEMM_SYM_LOWER = 1 } dion3_gemm_mode;

/*
 * Flags or-ed into the mode of dion3_gemm_f16 for half-stored symmetric
 * matrices.  A half-stored symmetric s x s matrix holds valid values only in
 * the 256 x 256 blocks below the block diagonal and in the full diagonal
 * 256 x 256 blocks (both triangles, mirrored); the rest is never written nor
 * read.  This is the layout of the s x s matrices inside the Gram
 * Newton-Schulz path (dion3_gram_ns_batched / dion3_step).
 *   DION3_GEMM_OUT_HALF: with DION3_GEMM_SYM_LOWER, write D half-stored (the
 *                        mirror is written on the diagonal blocks only).
 *   DION3_GEMM_A_HALF:   A is half-stored (needs M == K); the part of A above
 *                        the diagonal blocks is read from its transpose.
 *   DION3_GEMM_B_HALF:   B is half-stored (needs N == K), likewise.
 * and for operands given as their transpose:
 *   DION3_GEMM_A_TRANS:  A is passed as A^T, stored [batch][K][M] with pitch
 *                        lda >= M (so V = alpha (A^T)^T B^T + ...);
 *   DION3_GEMM_B_TRANS:  B is passed as B^T, stored [batch][K][N], ldb >= N.
 * An operand cannot be both transposed and half-stored.
 */
enum { DION3_GEMM_OUT_HALF = 0x10, DION3_GEMM_A_HALF = 0x20, DION3_GEMM_B_HALF = 0x40,
       DION3_GEMM_A_TRANS = 0x100, DION3_GEMM_B_TRANS = 0x200 };

/*
 * The tensor-core GEMM behind step (b), callable on its own.  Second-level
 * paragraph of the summary page: a symmetric product needs only its lower
 * triangle, which is then copied to the upper one.  Computes
 *     V = alpha A B^T + beta C + gamma I,  rounded to fp16 (fp32 accumulation),
 * with A [batch][M][K] and B [batch][N][K] fp16 (K contiguous, pitches lda /
 * ldb elements, batch strides in elements) and C [batch][M][N] fp16 or NULL
 * (then beta is ignored).
 *   DION3_GEMM_RECT:      every 128 x 128 output tile; V goes to D [batch][M][N]
 *                         (pitch ldd) if D is not NULL, and V^T to DT
 *                         [batch][N][M] (pitch lddt) if DT is not NULL; at least
 *                         one of them.
 *   DION3_GEMM_SYM_LOWER: M == N; only lower-triangle tiles are computed, each
 *                         written in place and mirrored, so D is exactly
 *                         symmetric (DT must be NULL).  Correct whenever
 *                         A B^T is symmetric: A == B, or A and B commuting
 *                         symmetric matrices (then B^T = B).
 *   The mode may carry the DION3_GEMM_*_HALF flags above.
 * Rules: A and B 16-byte aligned; lda, ldb >= K (>= M / N when transposed) and
 * multiples of 8; their batch strides multiples of 8.  D, DT and C may have any pitch >= their row length.
 * An unknown mode or flag, or a flag whose shape rule does not hold, returns
 * DION3_ERR_INVALID_ARG with nothing launched.
 */
dion3_status dion3_gemm_f16(int32_t mode, int32_t M, int32_t N, int32_t K, int32_t batch,
                            const void* A, int32_t lda, int64_t a_bstride,
                            const void* B, int32_t ldb, int64_t b_bstride,
                            const void* C, int32_t ldc, int64_t c_bstride,
                            void* D, int32_t ldd, int64_t d_bstride,
                            void* DT, int32_t lddt, int64_t dt_bstride,
                            float alpha, float beta, float gamma, dion3_stream_t stream);

/* Workspace bytes needed by dion3_step for these groups. */
dion3_status dion3_workspace_size(const dion3_group* groups, int32_t ngroups,
                                  const dion3_hparams* hp, size_t* bytes);

/*
 * The whole Dion3 step (a)-(c) over `ngroups` shape groups.
 *   sel_idx_out  NULL, or a host array [ngroups] of device int32 [batch][k]
 *                buffers (entries may be NULL) that receive each matrix's
 *                selected rows, ascending.
 * With more than one group and the accumulation overlap on (the default, see
 * dion3_set_overlap), the groups run in order on `stream`: each group's
 * momentum accumulation runs inside the previous group's Newton-Schulz
 * launches, and the parameter updates of up to two groups before the last
 * (columns a multiple of 8, at most 128 matrices) inside the last group's;
 * every result is written by the time the
 * call's work on `stream` completes, as without the overlap.  With it off, the
 * groups run concurrently: each on one of up to
 * four streams owned by the library, forked from `stream` (they wait for the
 * work already enqueued on it) and joined back into it before the call
 * returns, so later work on `stream` sees every result, and a graph captured
 * on `stream` holds the forked branches.  No matrix may belong to two groups
 * of one call.  While the launch trace is enabled, or when the environment
 * variable DION3_GROUP_STREAMS=0 is set, the groups run in order on `stream`.
 * The library's streams are created the first time a device needs them, so
 * make the first multi-group call before any stream capture begins.
 */
dion3_status dion3_step(const dion3_group* groups, int32_t ngroups,
                        const dion3_hparams* hp, void* ws, size_t ws_bytes,
                        int32_t* const* sel_idx_out, dion3_stream_t stream);

/*
 * Overlap of the accumulation with Newton-Schulz in dion3_step (and its lazy
 * and NorMuon forms) with more than one shape group: on (the default), the
 * groups run in order on `stream`, the one with the most Newton-Schulz work
 * first; only that group's accumulation (step a's M <- M + G and row norms)
 * runs on its own, and each later group's is handed out row by row to
 * streaming warps inside the previous group's tensor-core GEMM launches, which
 * move it while the tensor cores work, with a memory-bound kernel finishing
 * the rows they did not reach; the last group's launches carry the scatter
 * updates (step c) of up to two groups before it the same way.  Off, each
 * group runs its steps in sequence,
 * the groups on concurrent streams (see dion3_step).  Results are bit-identical
 * either way.  Process-wide; the environment variable DION3_OVERLAP=0 sets the
 * initial value to off.
 */
dion3_status dion3_set_overlap(int32_t on);

/*
 * dion3_select_rows without a workspace, for callers that may not allocate
 * device memory when they step the optimizer (their memory pool belongs to a
 * host framework that must not be bypassed, their device-memory budget is
 * fixed in advance, or they bind the C ABI without an allocator of their own).
 * The paper has no counterpart: this is an interface convenience.
 *
 * Same arguments and results as dion3_select_rows minus ws / ws_bytes.  The
 * row-norm scratch is a static device array inside the library (8 MiB, held by
 * every GPU that loads the library until the process exits), so batch * rows
 * must not exceed 1048576; larger requests return DION3_ERR_INVALID_ARG and
 * enqueue nothing.  No cudaMalloc, cudaFree or other allocating call is made.
 * The first call on each device looks up the array's device address with that
 * device current and keeps it; make that first call before any stream capture
 * begins, and do not call this entry point on a device after cudaDeviceReset
 * (the kept address would be stale).
 * Every call on a device shares the array and leaves its contents behind
 * (nothing in it needs to start at zero); calls whose work overlaps on the GPU
 * race on it, so order them on one stream.
 */
dion3_status dion3_select_rows_noalloc(int32_t rows, int32_t cols, int32_t batch,
                                       float* const* momentum, const void* const* grads,
                                       int32_t grad_dtype, int32_t k, int32_t* idx_out,
                                       float* fro2_out, dion3_stream_t stream);

/*
 * Launch trace (measurement aid).  While enabled, every launch of a
 * memory-bound kernel made by this library, and every chain of tensor-core GEMM
 * launches of one Newton-Schulz run, is bracketed by two CUDA events on its
 * stream and recorded with its algorithmic work: useful FLOPs for the GEMM (a
 * triangle counted as half) and bytes that must cross HBM for the memory-bound
 * kernels.  A chain gets one pair of events so that nothing sits between its
 * GEMMs (each may overlap its set-up with the end of the previous one); with
 * the environment variable DION3_TRACE_DETAIL=1 (or 2) every GEMM launch gets
 * its own pair and is labelled by role (and Gram side).  dion3_trace_enable(1)
 * starts a fresh record, dion3_trace_enable(0) stops and discards it.
 * dion3_trace_collect() waits for the recorded events, aggregates them per
 * kernel into out[0 .. min(*count, capacity)) (launches counts the launches,
 * total_ms the time between each pair of events), sets *count to the number of
 * kernels seen and clears the record (recording goes on if enabled).  Host-side
 * cost: two cudaEventRecord calls per recorded pair.
 */
typedef struct {
  char name[32];
  int64_t launches;
  double total_ms;
  double useful_flops;
  double algo_bytes;
} dion3_trace_entry;

dion3_status dion3_trace_enable(int32_t on);
dion3_status dion3_trace_collect(dion3_trace_entry* out, int32_t capacity, int32_t* count);

/*
 * dion3_step with the momentum decay left pending (lazy error feedback): the
 * selected rows' decay M[S] <- mu M[S] is not written back; instead
 * row_scale[g][b][i] = mu marks it, and the next lazy step applies it while
 * accumulating, M <- fp32(fp32(s M) + G), before resetting the factor to 1.
 * The sequence of selections, parameters and (flushed) momenta is bit-identical
 * to dion3_step's; a step writes k x m x 4 fewer bytes.
 *   row_scale  host array [ngroups] of device fp32 buffers [batch][rows],
 *              caller-owned optimizer state; set every entry to 1 before the
 *              first lazy step.  Between lazy steps the momentum a caller sees
 *              in M is the accumulated, not yet decayed one: the true momentum
 *              of row i is fp32(row_scale[i] M[i]) (dion3_flush_row_scale
 *              writes it back, e.g. before a checkpoint or a switch to
 *              dion3_step).
 * Third-level paragraph of the summary page: error feedback decays only the
 * selected rows; deferring that multiplication to the next accumulation does
 * not change it.
 */
dion3_status dion3_step_lazy(const dion3_group* groups, int32_t ngroups,
                             const dion3_hparams* hp, float* const* row_scale, void* ws,
                             size_t ws_bytes, int32_t* const* sel_idx_out,
                             dion3_stream_t stream);

/*
 * Per-neuron normalisation parameters of dion3_step_normuon.
 *   beta2  decay of the per-row second moment, 0 <= beta2 < 1 (0.95);
 *   eps    added to sqrt(v) before dividing, > 0 (1e-8; 0 is refused, since a
 *          selected row whose orthogonalised values are all zero has v = 0);
 *   rms    RMS of the written update block before the learning rate, > 0 (0.2).
 */
typedef struct {
  float beta2;
  float eps;
  float rms;
} dion3_normuon_params;

/*
 * dion3_step with the per-neuron normalisation that Dion3 inherits from
 * NorMuon ("Dion3 Cuts Muon Optimizer Time by Up to 6x ...", section "Dion3's
 * fastest path is a combined systems stack"; in float32 per the limitations
 * paragraph of "Dion3: Full-Stack Orthogonal Updates").  Neither page defines
 * it; this entry point implements the NorMuon form as a reading.  Between
 * (b) and (c), for each matrix with selected rows S and O (k x m):
 *   v[S_i] <- beta2 v[S_i] + (1 - beta2) mean_j O_ij^2          (fp32)
 *   d_i = 1 / (sqrt(v[S_i]) + eps),   U = g diag(d) O  with g such that
 *   ||U||_F = rms sqrt(k m)  (U = 0 when diag(d) O = 0),
 * and (c) writes W[S] <- W[S] - (lr / sqrt(f)) U.  Rows outside S keep their
 * v, as they keep their momentum.
 *   v   host array [ngroups] of device fp32 [batch][rows] state buffers,
 *       4-byte aligned, zero before the first step; read and written.
 * Same workspace (dion3_workspace_size), ordering and errors as dion3_step;
 * the momentum decay is eager.
 */
dion3_status dion3_step_normuon(const dion3_group* groups, int32_t ngroups,
                                const dion3_hparams* hp, const dion3_normuon_params* nm,
                                float* const* v, void* ws, size_t ws_bytes,
                                int32_t* const* sel_idx_out, dion3_stream_t stream);

/*
 * Applies pending lazy decays of one shape group: M[b][i] <- fp32(s M[b][i])
 * for every row whose factor s = row_scale[b][i] is not 1, then s <- 1.
 *   momentum   host array [batch] of device fp32 rows x cols matrices.
 *   row_scale  device fp32 [batch][rows].
 */
dion3_status dion3_flush_row_scale(int32_t rows, int32_t cols, int32_t batch,
                                   float* const* momentum, float* row_scale,
                                   dion3_stream_t stream);

/*
 * The bounded device-side wait of the tensor-core kernels, run on its own (a
 * diagnostic of the timeout path; the paper has no counterpart).  One thread
 * initialises an mbarrier in shared memory and waits for its first phase with
 * the wait the GEMM uses, giving up after limit_ns nanoseconds of the GPU's
 * global timer.  With arrive != 0 the thread arrives on the barrier first and
 * the wait succeeds at once.  With arrive == 0 nothing completes the phase:
 * the wait runs out, records DION3_ERR_TIMEOUT in the device status word (see
 * dion3_device_status) and the kernel returns.  No copy or MMA is in flight.
 *   limit_ns  1000 <= limit_ns <= 1e9, else DION3_ERR_INVALID_ARG.
 */
dion3_status dion3_wait_probe(int32_t arrive, int64_t limit_ns, dion3_stream_t stream);

/*
 * Synchronises `stream`, reads and clears the device status word written by
 * bounded device-side waits, and returns DION3_OK, DION3_ERR_TIMEOUT or
 * DION3_ERR_DEVICE_CHECK (or DION3_ERR_CUDA if synchronisation fails).
 */
dion3_status dion3_device_status(dion3_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* DION3_H_ */
