/*
 * libprecond: per-layer matrix-preconditioner step of EMA-Gram / KL-Shampoo
 * style optimizers, on one NVIDIA GB300 (sm_103a).
 *
 * For every weight gradient G (m x n, row-major) one step computes
 *
 *   L <- beta L + (1 - beta) G G^T,   R <- beta R + (1 - beta) G^T G
 *   A_hat = L / tr(L) + eps I          (same for R)
 *   X_L = A_hat(L)^power, X_R = A_hat(R)^power,  power in {-1/4, -1/2}
 *   U = X_L G X_R
 *
 * "Sharding EMA-Gram eigensolves" (Marin research note), section Background,
 * defines the step (EMA of G G^T and G^T G, rescale, regularise the
 * eigenvalues, raise to -1/4, reconstruct, shape the update).  The root is
 * computed here without any eigensolver, by the coupled Newton-Schulz
 * iteration of "Online KL Shampoo" (Tilde Research), section 2.2 and the
 * Appendix D algorithm box, generalised to the inverse p-th root
 * (T = alpha_k I - beta_k M, X <- X T, M <- T^p M, X_0 = I, M_0 = A_hat / c,
 * c = 1.01 x the Appendix D upper bound on the largest eigenvalue; the
 * classical step is alpha = (p+1)/p, beta = 1/p, the default is a per-step
 * minimax choice in the spirit of the section 2.3 CANS coefficients), and it
 * stops when ||M - I||_F <= tol * sqrt(d) (M equals X^p A_hat / c in exact
 * arithmetic, so this is the residual of the inverse-root equation that
 * Appendix E calls explicit and measurable).
 *
 * Conventions for every entry point:
 *  - All matrix pointers are DEVICE pointers (cuda_device's memory), owned by
 *    the caller, row-major, densely packed (leading dimension = columns).
 *  - Pointer arrays (grads[], L[], ...) and shape arrays are HOST arrays,
 *    read during the call only.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously on it; the call returns before it completes.
 *  - The library owns a workspace cached in the handle: it grows on demand
 *    (cudaMalloc, synchronising) and is freed by precond_destroy.
 *  - Return value: PRECOND_OK (0) or a negative PRECOND_E* code.  Argument
 *    errors are detected on the host before anything is enqueued.
 *  - Per-root outcomes found on the device (non-convergence, non-finite
 *    input) are reported by precond_get_stats, not by the return value.
 *  - A handle is not thread-safe: use one handle per host thread.
 */
#ifndef LIBPRECOND_PRECOND_H
#define LIBPRECOND_PRECOND_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct precond_ctx* precond_t;

/* status codes */
#define PRECOND_OK          0
#define PRECOND_EINVAL     -1  /* bad argument (null pointer, bad size, bad power/eps/beta, aliasing) */
#define PRECOND_ENOMEM     -2  /* workspace could not be allocated (or exceeds the set limit) */
#define PRECOND_ECUDA      -3  /* a CUDA runtime/driver call failed */
#define PRECOND_ENODEV     -4  /* host-only handle (created with cuda_device = -1): no GPU work possible */
#define PRECOND_ENOTCONV   -5  /* per root: residual above tolerance after the iteration cap; output written */
#define PRECOND_ENONFINITE -6  /* per root: NaN/Inf in the input or the Gram, or a Gram / input whose
                                  trace is not positive (its unit-trace rescaling is undefined, e.g.
                                  an all-zero gradient on zero state); output not written */

/* gradient storage types */
#define PRECOND_F32   0
#define PRECOND_BF16  1

/* option keys for precond_set_option */
#define PRECOND_OPT_TOL            1  /* stop when ||M - I||_F <= tol*sqrt(d); default 1e-4 */
#define PRECOND_OPT_MAX_ITER       2  /* iteration cap; 0 = derived from the scalar model (default) */
#define PRECOND_OPT_MIN_ITER       3  /* stagnation test only after this many iterations; default 4 */
#define PRECOND_OPT_ENGINE         4  /* 0 auto (default), 1 fp64 engine, 2 tcgen05 engine */
#define PRECOND_OPT_SMALL_DIM      5  /* auto engine: max(m,n) <= this -> fp64 engine; default 64.
                                         Tiny Grams go there: with eps = 1e-6 on a unit-trace Gram of a
                                         few rows, a rank-deficient Gram's root is set by eigenvalues
                                         1e-6 below entries of order 1, finer than the tcgen05 engine's
                                         27-bit digits resolve (larger Grams spread that error over
                                         many directions and meet 1e-3) */
#define PRECOND_OPT_WORKSPACE_MAX  6  /* workspace limit in bytes; 0 = unlimited (default) */
#define PRECOND_OPT_TIMING         7  /* 1 = record per-stage CUDA events (read by precond_get_timing) and
                                         events around every iteration-stage GEMM (precond_get_gemm_timing);
                                         2 = per-stage events only (a CUDA graph then holds no event node
                                         between the GEMMs, which costs small steps a third of their time);
                                         0 = none (default) */
#define PRECOND_OPT_USE_GRAPH      8  /* 1 = capture each distinct plan (shapes, options, workspace) once as a
                                         CUDA graph on a handle-owned stream and replay it, ordered after
                                         and before the caller's stream by events; the 4 most recently
                                         used plans stay captured (default 1); 0 = launch every kernel on
                                         the caller's stream */
#define PRECOND_OPT_CLASSICAL      9  /* 1 = classical Newton step (p+1)/p I - M/p at every iteration;
                                         0 = per-step minimax step polynomial (default) */
#define PRECOND_OPT_FOLD          10  /* minimax step: the interval's top may not fall below this
                                         fraction of its bottom's factor, T(1) >= fold T(l); [0, 1), default 0.3 */
#define PRECOND_OPT_BRANCHES      11  /* 1 = when no root class's products fill the GPU (fewer 128 x 128
                                         tiles than SMs), the stages fork onto streams of the handle's own:
                                         the two Gram sides, each root class's start and finish kernels,
                                         and each class's M chain and X chain in the iteration stage, every
                                         stage joined back into the call's stream by events (default 1);
                                         0 = everything on the call's stream.  Results are identical. */
#define PRECOND_OPT_STEP_DEGREE   12  /* degree of the per-step minimax polynomial T_k(M) at p = 4: 2 (default;
                                         T = a I - b M + c M^2, 5 products per iteration, about 7
                                         iterations from l_0 = 1e-6) or 1 (T = a I - b M, 4 products, about
                                         10 iterations).  p = 2 always takes linear steps (both degrees
                                         need 36 products there). */
#define PRECOND_OPT_PACKED_STATE  13  /* 1 = the EMA state L[i], R[i] of precond_step is the upper triangle
                                         only, packed row by row: d(d+1)/2 floats, element (r, c) with
                                         r <= c at offset r d - r (r - 1) / 2 + (c - r) (half the state
                                         memory of the full layout; "Online KL Shampoo", Appendix F).
                                         0 = full d x d row-major state (default).  The full state is
                                         kept exactly symmetric, so both layouts give identical roots
                                         and updates. */
#define PRECOND_OPT_TILE_SPLIT    14  /* most CTAs that share one 128 x 128 tile of a tcgen05 product: 1, 2
                                         or 4 (default 4).  A product with fewer tiles than SMs gives
                                         each tile to the largest of 4, 2, 1 (at most this) CTAs that
                                         still fit one per SM; each computes the whole tile and writes a
                                         share of its outputs.  Results are identical for every value. */

/*
 * Create a handle bound to `cuda_device` (>= 0).  cuda_device = -1 creates a
 * host-only handle that validates arguments and plans workspaces but enqueues
 * nothing (every GPU call then returns PRECOND_ENODEV after validation).
 * Errors: EINVAL (out == NULL or cuda_device < -1), ECUDA (device unusable).
 */
int precond_create(precond_t* out, int cuda_device);

/* Free the workspace and the handle.  NULL is accepted (no-op). */
int precond_destroy(precond_t h);

/*
 * One preconditioner step for `count` (>= 1) weight matrices.
 *   grads[i]     : m_i x n_i gradient, PRECOND_F32 (float*) or PRECOND_BF16
 *                  (16-bit bfloat16 words), per `grad_dtype`.  Read; and, when
 *                  out_f32 == NULL, overwritten with U_i (rounded to bf16 for
 *                  bf16 grads).
 *   shapes       : 2*count int64: m_0, n_0, m_1, n_1, ...  (each >= 1)
 *   L[i], R[i]   : fp32 EMA state, m_i x m_i and n_i x n_i, read and updated
 *                  in place (start from zeros for the first step); with
 *                  PRECOND_OPT_PACKED_STATE, their packed upper triangles
 *                  (m_i (m_i + 1) / 2 and n_i (n_i + 1) / 2 floats).  L[i] and
 *                  R[i] must not alias each other or any other state.
 *   beta         : EMA coefficient in [0, 1)
 *   eps          : regulariser added to the eigenvalues of the unit-trace
 *                  Gram, > 0
 *   power        : -0.25f or -0.5f
 *   out_f32      : NULL (write U in place into grads) or an array of count
 *                  device pointers to fp32 m_i x n_i outputs
 * Roots are numbered 2i (left, L) and 2i+1 (right, R) in precond_get_stats.
 */
int precond_step(precond_t h, int count, void* const grads[], int grad_dtype,
                 const int64_t shapes[], float* const L[], float* const R[],
                 float beta, float eps, float power, float* const out_f32[],
                 void* stream);

/*
 * Inverse root of given SPD matrices (no EMA, no gradient):
 *   X_i = (A_i / tr(A_i) + eps I)^power,  A_i and X_i fp32 d_i x d_i.
 * eps is therefore relative to the trace.  A_i is read only; X_i may not
 * alias A_i.  Roots are numbered i in precond_get_stats.
 */
int precond_inv_root(precond_t h, int count, const float* const A[], const int64_t dims[],
                     float eps, float power, float* const X[], void* stream);

/*
 * Per-root results of the last precond_step / precond_inv_root on this
 * handle.  Synchronises with that call's stream.  `nroots` must equal the
 * number of roots of that call (2*count for a step, count for inv_root).
 * Every output array may be NULL (skipped):
 *   iters[r]  : Newton-Schulz iterations executed
 *   resid[r]  : final ||M - I||_F / sqrt(d)
 *   status[r] : PRECOND_OK, PRECOND_ENOTCONV or PRECOND_ENONFINITE
 *   scale[r]  : c = 1.01 x the largest-eigenvalue bound of A_hat
 */
int precond_get_stats(precond_t h, int nroots, int iters[], float resid[], int status[],
                      float scale[]);

/* Set an option (PRECOND_OPT_*).  EINVAL for an unknown key or a bad value. */
int precond_set_option(precond_t h, int key, double value);

/*
 * Milliseconds spent by stage in the last call when PRECOND_OPT_TIMING is on
 * (synchronises): ms[0] input preparation + Gram EMA, ms[1] bound + start,
 * ms[2] Newton-Schulz iterations, ms[3] finish + apply.  Also the number of
 * GEMM launches of the iteration stage and its algorithmic FLOPs: 2 d^3 per
 * product each root executed (3 or 4 per linear step at p = 2 or 4, 5 per
 * quadratic step, one fewer in the first iteration), summed over roots.
 */
int precond_get_timing(precond_t h, double ms[4], int64_t* ns_gemm_launches, double* ns_flops);

/*
 * With PRECOND_OPT_TIMING on: total milliseconds of the tcgen05 GEMM launches
 * of the last call's iteration stage (CUDA events around each launch on the
 * call's stream; synchronises; -1 in timing mode 2, which records no such
 * events), their number, and the bf16 MMA FLOPs they issued, counted on the
 * device: for every tile actually computed (tiles of converged roots are
 * skipped; a tile spread over several CTAs by PRECOND_OPT_TILE_SPLIT counts
 * once per CTA), 2 x 128 x 128 x 32 per K block and digit product.  Any
 * output pointer may be NULL.
 */
int precond_get_gemm_timing(precond_t h, double* ms_total, int64_t* launches, double* issued_flops);

/*
 * Workspace bytes.  *planned: the plan of the last precond_step /
 * precond_inv_root call on this handle that passed validation, also on a
 * host-only handle (where that call returns PRECOND_ENODEV after planning);
 * 0 before any such call.  *allocated: the device workspace the handle holds
 * now (0 on a host-only handle).  Either pointer may be NULL.  The EMA state,
 * gradients and outputs are the caller's and are not counted.
 */
int precond_get_workspace(precond_t h, int64_t* planned, int64_t* allocated);

/* Kernel launches this handle has issued since creation (every library kernel). */
int64_t precond_launch_count(precond_t h);

/*
 * Read back the fp32 root of root `r` of the last precond_step on this handle
 * (X_L of matrix i for r = 2i, X_R for r = 2i+1) into `dst`, a d x d device
 * buffer owned by the caller.  Enqueued on `stream`.  For tests and
 * diagnostics; the step itself never materialises fp32 roots.  After a
 * precond_inv_root call it reads the root's last iterate instead.
 */
int precond_get_root(precond_t h, int r, float* dst, void* stream);

/*
 * Self-test of the GEMM core (no counterpart in the method: it checks the
 * library's building block).  C = A . B^T with A (M x K), B (N x K), C (M x N)
 * fp32 device buffers, through engine 1 (fp64 planes, double-float products) or 2 (tcgen05: operands as
 * three bf16 digits with a scale per row and 128-column block, exact digit
 * products); `passes` = digits per operand, 3 for engine 2 (ignored by
 * engine 1).  Synchronises `stream`.
 */
int precond_gemm_selftest(precond_t h, int engine, int M, int N, int K, const float* A, const float* B,
                          float* C, int passes, void* stream);

/*
 * Diagnostic read-back (no counterpart in the method) of a work matrix of
 * root `r` of the last call into a d x d fp32 device buffer:
 * which = 0/1 X buffers, 2/3 M buffers, 4 D (the T^2 - a^2 I term), 5 F
 * (the T^4 - a^4 I term, p = 4; with quadratic steps it holds E = T - a I
 * between E's product and F's), 8 the final root (step calls).  Iteration k reads buffers k & 1 and writes
 * (k + 1) & 1.  Enqueued on `stream`.
 */
int precond_debug_plane(precond_t h, int r, int which, float* dst, void* stream);

/*
 * Allocation-free inverse root of ONE matrix (no counterpart in the pages: a
 * deployment variant of precond_inv_root).  For callers that cannot allocate
 * device memory when they need the root -- code inside a pool-allocator
 * hook, a host callback, or a runtime that forbids cudaMalloc after start-up
 * because it would synchronise the device or break a fixed memory budget.
 *
 *   X = (A / tr(A) + eps I)^power,  A and X fp32 d x d device buffers owned by
 *   the caller (X may not alias A), power -0.25f or -0.5f, fp64 engine.
 *
 * All scratch lives in one fixed file-scope device array of 4 MiB that every
 * GPU which loads this library holds until the process exits; no cudaMalloc,
 * cudaFree or other device-memory allocating routine is called, and no
 * stream, event or graph is created (the host side plans in small heap
 * buffers, as any C++ code does).  d above
 * PRECOND_NOALLOC_MAX_D is rejected with PRECOND_EINVAL (and a message on
 * stderr).  The first call on each device looks up the array's device address
 * (with that device current); make that first call before any stream capture.
 * Every call shares the array and overwrites it, so calls whose GPU work
 * overlaps (other streams, other host threads, unsynchronised loops on
 * different streams) race: order them on one stream.  `status` (host, may be
 * NULL): when given, the call synchronises `stream`, stores the root's
 * PRECOND_OK / ENOTCONV / ENONFINITE there and returns PRECOND_ECUDA if the
 * device recorded an error.  When NULL, the call does not synchronise and
 * reports nothing found on the device: a caller who needs to know whether the
 * root converged or the input was finite must pass `status`.
 */
#define PRECOND_NOALLOC_MAX_D 256
int precond_inv_root_noalloc(const float* A, int64_t d, float eps, float power, float* X, void* stream,
                             int* status);

/*
 * The per-step minimax schedule the iteration uses (host only, no device or
 * handle needed): for p in {2, 4}, the interval bottom l0 in (0, 1) of M_0's
 * spectrum, the fold cap in [0, 1) and the polynomial degree (1 or 2), the
 * coefficients of T_k(m) = alpha_k - beta_k m + gamma_k m^2 and the interval
 * bottom lo_k each step starts from, up to max_steps steps (the schedule ends
 * when 1 - lo < 1e-9).  Arrays hold max_steps doubles; *nsteps receives the
 * number written.  Every step maps [lo_k, 1] into [lo_(k+1), 1] with
 * max m T_k(m)^p = 1.  The pages have no counterpart: the step polynomials
 * follow the idea of per-step optimised polynomials (CANS, "Online KL
 * Shampoo" section 2.3) for the coupled iteration.  EINVAL on bad arguments.
 */
int precond_step_schedule(int p, double l0, double fold, int degree, int max_steps, double* alpha, double* beta,
                          double* gamma, double* lo, int* nsteps);

/* Static text for a status code. */
const char* precond_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* LIBPRECOND_PRECOND_H */
