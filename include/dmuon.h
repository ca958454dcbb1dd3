/*
 * dmuon.h -- C ABI of the GB300 owner-rank Muon update library (libdmuon.so).
 *
 * The library runs, on one GPU, the per-parameter Muon update that a DMuon owner rank performs on
 * the matrices it owns: momentum accumulate, fp32 Frobenius normalisation, five-step fp16
 * Newton-Schulz (direct or Gram form) and the weight update.
 *
 * Sources (DMuon documentation and a blog post on distributed Muon):
 *   - "Newton-Schulz 变体" (Newton-Schulz variants) page: sections "直接空间 NS（经典）" (direct
 *     iteration), "Gram 空间 NS（Dao-AILab）" (Gram iteration), "精度流水线" (fp32 normalisation, fp16
 *     iteration), "系数集" (coefficient tables), "重启机制" (restarts), "使用自定义系数集" (the
 *     newton_schulz / NewtonSchulz / Muon calls these entry points stand for).
 *   - DMuon "Core Concepts" page, section "1. Dedicated Ownership": the owner runs Newton-Schulz on
 *     the full matrix with no extra communication.
 *   - pwwt.cn blog on distributed Muon, section "2. Muon执行过程": momentum, then orthogonalise it.
 *
 * Conventions for every entry point:
 *   - Pointers named "device" must be CUDA device (or managed) memory on the current device;
 *     "host" pointers are read during the call only and may be freed when it returns.
 *   - Matrices are dense row-major with the given rows x cols and no padding. Device buffers
 *     passed to the library must be 16-byte aligned.
 *   - The caller owns all tensors. The library owns a cached workspace per device (grown on first
 *     use for a set of shapes, kept until dmuon_release_workspace) and descriptor tables. Calls that
 *     share a device must be serialised by the caller (same stream, or synchronised streams).
 *   - Work is enqueued on `cuda_stream` (a cudaStream_t; NULL = legacy default stream); the call
 *     returns before the GPU finishes. No host synchronisation happens except when a new shape set
 *     needs workspace or new descriptors (first call).
 *   - Every function returns a dmuon_status. Arguments are validated before anything is
 *     launched; on an invalid argument nothing is launched and dmuon_last_error() says why.
 *     Errors the GPU detects while running (a bounded wait that gave up, a non-finite fp16 value)
 *     are recorded in a device status word read by dmuon_check_status().
 */
#ifndef DMUON_H
#define DMUON_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DMUON_API __attribute__((visibility("default")))
#else
#define DMUON_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dmuon_status {
  DMUON_OK = 0,
  DMUON_ERR_INVALID_ARG = 1, /* bad pointer, size, enum, restart list or alignment            */
  DMUON_ERR_UNSUPPORTED = 2, /* no sm_103a device, or a shape beyond the library's limits        */
  DMUON_ERR_OOM = 3,         /* workspace allocation failed or exceeds the set limit           */
  DMUON_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (text in dmuon_last_error)  */
  DMUON_ERR_TIMEOUT = 5,     /* a device-side bounded wait gave up (reported by check_status)  */
  DMUON_ERR_NONFINITE = 6,   /* an fp16 intermediate overflowed or became NaN (check_status)   */
  DMUON_ERR_RANGE = 7        /* checked build only: a device-side range check failed (check_status) */
} dmuon_status;

typedef enum dmuon_ns_backend {
  DMUON_NS_DIRECT = 0, /* X <- a X + b (X X^T) X + c (X X^T)^2 X                                 */
  DMUON_NS_GRAM = 1,   /* R = X X^T, Z = b R + c R^2, Q <- Z Q + a Q, R <- (aI+Z) R (aI+Z), Q X   */
  DMUON_NS_AUTO = 2    /* per matrix, the one with fewer flops: direct when max < 4/3 min
                          (direct 15 m^2 n + 5 m^3 against Gram 6 m^2 n + 17 m^3), else Gram      */
} dmuon_ns_backend;

typedef enum dmuon_dtype { DMUON_F32 = 0, DMUON_BF16 = 1 } dmuon_dtype;

/* Largest number of Newton-Schulz steps accepted (coefficient triples per call). */
#define DMUON_MAX_STEPS 16

/*
 * dmuon_ns -- Newton-Schulz orthogonalisation of one matrix, in place.
 *   ("Newton-Schulz 变体": newton_schulz(G, coefficients=..., restart_iterations=[...]) /
 *    NewtonSchulz(backend, ...); precision pipeline of section "精度流水线".)
 *
 *   x          device fp32, rows m x cols n. Input G; on return O = NS(G / (||G||_F + eps)) in the same
 *              orientation. Internally a matrix with m > n is worked on as its transpose (m x m Gram
 *              matrices stay the small ones) and written back transposed.
 *   coeffs     host, 3 * steps floats (a_0, b_0, c_0, a_1, ...): one odd polynomial per step.
 *   steps      1 .. DMUON_MAX_STEPS.
 *   restarts   host, n_restarts ints, strictly increasing, each in [0, steps - 1]; a restart at k
 *              happens before step k (Gram backend only; ignored by the direct backend). May be NULL
 *              when n_restarts == 0. Index 0 is accepted and has no effect.
 *   backend    DMUON_NS_DIRECT, DMUON_NS_GRAM or DMUON_NS_AUTO.
 *   eps        added to the Frobenius norm (not to its square); must be >= 0.
 * Intermediates are fp16 with fp32 accumulation. A zero matrix gives a zero output.
 */
DMUON_API int dmuon_ns(float* x, int64_t m, int64_t n, const float* coeffs, int steps, const int* restarts,
             int n_restarts, int backend, float eps, void* cuda_stream);

/*
 * dmuon_ns_tp -- dmuon_ns (Gram form) computed the way `shards` tensor-parallel ranks would compute it,
 * emulated on one GPU ("Newton-Schulz 变体", section "Gram 空间 NS": R is a sum of local Gram matrices,
 * so exact TP needs one all-reduce of the (m, m) Gram; DMuon "Core Concepts" §5: O(d^2) instead of O(mn)).
 * The long side of x is split into `shards` column shards (boundaries t * n / shards rounded down to a
 * multiple of 8). The norm is the fixed-order sum of per-shard sums of squares (the one scalar
 * all-reduce); every Gram formation R = X X^T (the initial one and each restart's) is the fixed-order sum
 * of the per-shard products X_t X_t^T, each computed in fp32 (the one m x m all-reduce); the remaining
 * m x m work and Q X_t are what every rank does locally. Same arguments and output as dmuon_ns.
 *   shards     1 .. 64; the long side must be at least 16 * shards.
 * The result equals dmuon_ns up to fp32 summation order and is deterministic run to run.
 */
DMUON_API int dmuon_ns_tp(float* x, int64_t m, int64_t n, int shards, const float* coeffs, int steps,
                          const int* restarts, int n_restarts, float eps, void* cuda_stream);

/*
 * dmuon_muon_step -- one owner-rank Muon update over `count` matrices, batched.
 *   (DMuon "Core Concepts", step "Owner NS update"; Muon(model, lr, ns_backend) on the
 *    "Newton-Schulz 变体" page; momentum-then-orthogonalise of the pwwt.cn post, section 2.)
 *
 * For each matrix i (rows[i] x cols[i], row-major):
 *   M_i <- beta * M_i + G_i                                  (fp32, in place)
 *   X_i  = fp16(M_i / (||M_i||_F + eps)), transposed if rows > cols
 *   O_i  = NS(X_i) with `backend`, `coeffs`, `restarts`       (fp16 operands, fp32 accumulation)
 *   W_i <- W_i - lr * O_i                                     (fp32, in place, original orientation)
 * All matrices advance phase by phase; each phase is one grouped GPU launch over all of them.
 *
 *   count      number of matrices, >= 1.
 *   params     host array of `count` device fp32 pointers W_i.
 *   grads      host array of `count` device pointers G_i, element type `grad_dtype` (fp32 or bf16).
 *   momenta    host array of `count` device fp32 pointers M_i (the momentum state; zero to start).
 *   rows, cols host arrays of `count` sizes, each >= 1.
 *   norms_out  device fp32 array of `count` entries receiving ||M_i||_F after the momentum update,
 *              or NULL.
 *   lr, beta, coeffs, steps, restarts, n_restarts, backend, eps: as above / dmuon_ns.
 * W_i, G_i and M_i must not overlap one another or another matrix's buffers.
 */
DMUON_API int dmuon_muon_step(int count, float* const* params, const void* const* grads, int grad_dtype,
                    float* const* momenta, const int64_t* rows, const int64_t* cols,
                    float* norms_out, float lr, float beta, const float* coeffs, int steps,
                    const int* restarts, int n_restarts, int backend, float eps, void* cuda_stream);

/*
 * dmuon_muon_step_host -- dmuon_muon_step with the step's gradients arriving from host memory, the form a
 * caller whose gradients are produced or staged on the host uses. (The pages transfer gradients between
 * ranks, not from the host; this is the single-GPU form of "gradients in, update out".) Equivalent to
 * copying every grads_host[i] into grads[i] and then calling dmuon_muon_step, with identical results,
 * but the copies overlap the computation: the matrices are taken in `groups` consecutive groups by
 * gradient bytes, their weights rising 1 : 2 : 3 from the start and falling by a factor 0.85 per group
 * towards the end (with a fast host link the first group's copy is what stays exposed, with a slow one
 * the computation still queued after the last copy);
 * group g's copies run on the library's copy stream while earlier groups compute on
 * cuda_stream, and group g's momentum pass waits only for its own copies. Each group runs its row-wise
 * passes and Newton-Schulz phases as grouped launches of its own. With many small matrices (64 or more
 * averaging under 4 MiB of gradient), where one copy per matrix would cost the host more than the
 * transfers, one gather launch on cuda_stream reads every gradient out of host memory instead (the
 * memory must then be device-readable: page-locked, or pageable on devices that read host page tables;
 * otherwise the copies above are used) and the step runs as one group.
 *
 *   grads_host  host array of `count` host pointers to the gradients (rows[i] x cols[i], `grad_dtype`,
 *               row-major, contiguous). For the copies to overlap they must be page-locked
 *               (cudaHostAlloc / cudaHostRegister); pageable memory gives the same results without the
 *               overlap. The caller keeps them unchanged until cuda_stream has passed this call.
 *   grads       host array of `count` device buffers (as in dmuon_muon_step) receiving the gradients;
 *               they are overwritten.
 *   groups      pipeline depth in [1, 64]; <= 0 lets the library choose (one group per ~1 GiB of
 *               gradients, at most 16). More groups than matrices gives one matrix per group.
 *   Other arguments as in dmuon_muon_step.
 * Ordering: the copies start after all work enqueued on cuda_stream before the call and after the
 * previous dmuon_muon_step_host call on this device has read its gradients; all of the call's work,
 * copies included, is complete when cuda_stream reaches the point after it. Not graph-capturable.
 */
DMUON_API int dmuon_muon_step_host(int count, float* const* params, const void* const* grads_host, void* const* grads,
                                   int grad_dtype, float* const* momenta, const int64_t* rows, const int64_t* cols,
                                   float* norms_out, float lr, float beta, const float* coeffs, int steps,
                                   const int* restarts, int n_restarts, int backend, float eps, int groups,
                                   void* cuda_stream);

/*
 * dmuon_momentum_normalize -- the first half of dmuon_muon_step on its own ("精度流水线", stage 1,
 * preceded by the momentum accumulate): for each matrix
 *   M_i <- beta * M_i + G_i (skipped when grads == NULL: M_i is then only read),
 *   norms_out[i] = ||M_i||_F,  X_i = fp16(M_i / (||M_i||_F + eps)) in the m <= n orientation.
 *
 *   x_out      host array of `count` device pointers to caller-owned fp16 buffers of
 *              min(rows,cols) x max(rows,cols) elements, row-major (the oriented X_i).
 *   norms_out  device fp32 array of `count` entries (required here).
 * Other arguments as in dmuon_muon_step.
 */
DMUON_API int dmuon_momentum_normalize(int count, const void* const* grads, int grad_dtype,
                             float* const* momenta, const int64_t* rows, const int64_t* cols,
                             void* const* x_out, float* norms_out, float beta, float eps,
                             void* cuda_stream);

/*
 * dmuon_gemm_f16 -- the tensor-core building block of both iterations, exposed for testing and for
 * callers composing their own schedules. With A (M x K, fp16, row-major, lda), B (fp16, ldb) and
 * an optional E (M x N, fp16, lde):
 *   acc[i][j] = sum_k A[i][k] * Bop[k][j],  Bop = B^T when b_trans != 0 (B is N x K; e.g. X X^T),
 *                                           Bop = B    when b_trans == 0 (B is K x N; e.g. Q X)
 *   v[i][j]   = alpha * acc[i][j] + beta * E[i][j] + (i == j ? gamma : 0)     (fp32)
 *   D[i][j]   = fp16(v[i][j])   (D: M x N fp16, ldd)
 * symmetric != 0 requires M == N and computes only tiles touching the upper triangle, writing
 * D[i][j] and D[j][i] from the upper-triangle value (the SYRK form of X X^T and R^2).
 * E may be NULL (beta is then ignored). Leading dimensions are in elements, >= the row length,
 * and must make every row start 16-byte aligned (multiples of 8). A, B, E and D must not overlap.
 */
DMUON_API int dmuon_gemm_f16(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                   int64_t ldb, int b_trans, const void* E, int64_t lde, void* D, int64_t ldd,
                   float alpha, float beta, float gamma, int symmetric, void* cuda_stream);

/*
 * dmuon_momentum_normalize_noalloc -- dmuon_momentum_normalize for ONE matrix without any device
 * allocation. The pages have no counterpart; this exists for callers that cannot allocate device
 * memory: code whose device memory is owned by someone else (a framework's caching allocator, a fixed
 * memory plan that must account for every byte) and code that cannot afford the device-wide
 * synchronisation cudaMalloc / cudaFree may cause. It calls no cudaMalloc, cudaFree or allocating library
 * routine; its scratch is a fixed array of about 16.5 KB in the library's device image, which every GPU
 * that loads the library holds until the process exits.
 *
 *   grad       device, rows x cols, grad_dtype (fp32 or bf16), or NULL (M is then only read).
 *   momentum   device fp32 rows x cols; M <- beta * M + G in place.
 *   x_out      device fp16, min(rows,cols) x max(rows,cols) row-major: X = fp16(M / (||M||_F + eps)),
 *              transposed when rows > cols.
 *   norm_out   device fp32, one value: ||M||_F after the update.
 *   rows*cols must not exceed DMUON_NOALLOC_MAX_ELEMS (2^28); larger matrices are rejected with
 *   DMUON_ERR_INVALID_ARG before anything is launched.
 * The first call on a device (with that device current) looks up the scratch's device address; make
 * that first call before any stream capture. The address is kept per device together with the CUDA
 * context it belongs to; a call that finds a different context current on the device (for instance
 * after cudaDeviceReset) looks it up again. All calls share the one scratch array and it keeps the
 * last call's contents (nothing in it needs to start at zero), so calls whose work overlaps on the GPU
 * race with each other: order them on one stream or synchronise between them.
 */
#define DMUON_NOALLOC_MAX_ELEMS 268435456
DMUON_API int dmuon_momentum_normalize_noalloc(const void* grad, int grad_dtype, float* momentum, int64_t rows,
                                               int64_t cols, void* x_out, float* norm_out, float beta, float eps,
                                               void* cuda_stream);

/*
 * dmuon_assign_owners -- dedicated ownership: give each of `count` matrices one owner rank out of
 * `nranks`, balancing the work (DMuon "Core Concepts", section "均衡划分" / "Balanced partition":
 * dedicate_params() uses LPT with global balance and same-layer spread; the "Newton-Schulz 变体" page,
 * section "TP 路由", calls it a deterministic LPT inside compute_balanced_assignment).
 *
 * Matrices are taken in decreasing cost (ties: lower index first). Each goes to the rank holding the
 * fewest matrices of its own layer (so a layer's parameters are broadcast from different ranks at
 * once); among those, to the rank with the least load so far (ties: lower rank). Without layer_ids
 * this is plain LPT. Host-only: no device is touched.
 *
 *   rows, cols   host, `count` sizes (>= 1).
 *   layer_ids    host, `count` layer indices (>= 0), or NULL for no layer constraint.
 *   nranks       1 .. 65536.
 *   cost_model   DMUON_COST_ELEMENTS (rows*cols), DMUON_COST_GRAM_FLOPS (6 m^2 n + 17 m^3 with
 *                m = min, n = max: five Gram steps, restart [2]) or DMUON_COST_DIRECT_FLOPS
 *                (15 m^2 n + 5 m^3).
 *   owner_out    host, `count` ints: the owner rank of each matrix.
 *   loads_out    host, `nranks` doubles (the summed cost per rank), or NULL.
 */
#define DMUON_COST_ELEMENTS 0
#define DMUON_COST_GRAM_FLOPS 1
#define DMUON_COST_DIRECT_FLOPS 2
DMUON_API int dmuon_assign_owners(int count, const int64_t* rows, const int64_t* cols, const int* layer_ids,
                                  int nranks, int cost_model, int* owner_out, double* loads_out);

/*
 * dmuon_adamw_step -- AdamW over `count` tensors in one launch, for the parameters that are not Muon
 * targets (DMuon "Core Concepts", section "1. Dedicated Ownership", step 6 of each training step). The
 * pages name the optimizer only; this is AdamW with decoupled weight decay in PyTorch's form. For step t:
 *   p <- p (1 - lr wd);  m <- b1 m + (1 - b1) g;  v <- b2 v + (1 - b2) g^2;
 *   p <- p - lr / (1 - b1^t) * m / (sqrt(v) / sqrt(1 - b2^t) + eps)
 *
 *   params, exp_avg, exp_avg_sq  host arrays of `count` device fp32 pointers (p, m, v; updated in place).
 *   grads        host array of `count` device pointers, element type grad_dtype (fp32 or bf16).
 *   numels       host array of `count` element counts (>= 1); tensors are dense.
 *   step         t >= 1 (the step being taken, counted from 1).
 *   lr, beta1, beta2, eps, weight_decay are doubles: 1 - beta and the bias corrections are formed in
 *   double before the kernel sees them in fp32 (1 - fp32(0.999) would be off by 1.3e-5 relative).
 * The pointer table is cached per device for the same buffers (re-uploaded when they change).
 */
DMUON_API int dmuon_adamw_step(int count, float* const* params, const void* const* grads, int grad_dtype,
                               float* const* exp_avg, float* const* exp_avg_sq, const int64_t* numels, double lr,
                               double beta1, double beta2, double eps, double weight_decay, int step,
                               void* cuda_stream);

/*
 * dmuon_check_status -- synchronise `cuda_stream`, then read and clear the device status word.
 * Returns DMUON_OK, DMUON_ERR_TIMEOUT (a kernel's bounded wait gave up: its results are invalid),
 * DMUON_ERR_RANGE (checked build: an index or tile outside its table or matrix was found and skipped;
 * results are invalid), DMUON_ERR_NONFINITE (an fp16 intermediate overflowed or was NaN) or
 * DMUON_ERR_CUDA (an asynchronous CUDA error surfaced during synchronisation).
 */
DMUON_API int dmuon_check_status(void* cuda_stream);

/*
 * Graph replay of repeated calls (no counterpart on the pages; on by default). dmuon_ns, dmuon_ns_tp,
 * dmuon_muon_step and dmuon_momentum_normalize keep one cached plan per device. When such a call arrives
 * with the same plan and the same arguments (coefficients, lr, beta, eps, norms_out) as the call just before
 * it, the library captures the plan's launches once on a private stream as a CUDA graph and from then on
 * launches that graph on cuda_stream for every such call: the same kernels with the same arguments, so
 * results are identical bit for bit, with the per-launch issue cost of the chain of dependent launches
 * taken off (measured on a single 256 x 1024 Muon step: ~131 -> ~118 us). A call with other arguments, a
 * plan change, dmuon_release_workspace, per-kernel timing (below), or a cuda_stream that the caller is
 * capturing into a graph of its own launches directly (so the caller's graph holds the kernels); a failed
 * capture falls back to direct launches. on = 0 turns replay off (every call launches directly), nonzero back on.
 * Always DMUON_OK. Host-gradient calls (dmuon_muon_step_host) always launch directly.
 */
DMUON_API int dmuon_set_graph_replay(int on);

/*
 * Per-kernel CUDA-event timing (off by default; used by benchmarks). While enabled, the library records
 * a pair of CUDA events on the caller's stream around every kernel it launches. dmuon_timing_read
 * waits for the recorded events, writes per kernel class the summed elapsed milliseconds and the
 * number of launches since the previous read (or enable), and clears the record. Classes:
 *   0 momentum + sum of squares (per-shard sums for dmuon_ns_tp), 1 norm finalisation, 2 normalise +
 *   fp16 cast, 3 tensor-core GEMM (including the fused small-matrix kernel), 4 AdamW, 5 shard Gram
 *   reduction (dmuon_ns_tp).
 * ms_out and launches_out must each hold DMUON_TIMING_CLASSES entries (host memory).
 */
#define DMUON_TIMING_CLASSES 6
DMUON_API int dmuon_timing_enable(int on);
DMUON_API int dmuon_timing_read(double* ms_out, int64_t* launches_out);

/* The same record launch by launch, in launch order: ms_out[i] and class_out[i] for the first
 * min(count, max_launches) launches (host arrays of max_launches entries; may be NULL when
 * max_launches == 0), *count_out = the number recorded. Clears the record like dmuon_timing_read. */
DMUON_API int dmuon_timing_read_launches(int max_launches, double* ms_out, int* class_out, int* count_out);

/*
 * What one run of the device's cached plan (the last dmuon_ns / dmuon_ns_tp / dmuon_muon_step /
 * dmuon_muon_step_host call on this device) issues on the tensor cores: *exec_flops_out = 2 x the
 * multiply-adds of every tile of every GEMM launch (diagonal tiles of symmetric products in full, K
 * rounded up to the 64-wide ring slice), *tiles_out = the tiles, *gemm_launches_out = the GEMM launches.
 * For the fused small-matrix plan exec_flops is -1 (not counted), tiles 0 and launches 1.
 * DMUON_ERR_INVALID_ARG when nothing has been planned on the current device.
 */
DMUON_API int dmuon_plan_info(double* exec_flops_out, int64_t* tiles_out, int* gemm_launches_out);

/*
 * Diagnostic for the library's failure detection (no counterpart on the pages). Every mbarrier wait in
 * the library's kernels is bounded: when one exceeds its limit the kernel records DMUON_ERR_TIMEOUT in the
 * device status word, drains its own copies, frees its tensor memory and returns, leaving the CUDA
 * context usable. This launches one CTA whose wait, through that same bounded wait, is on a phase that
 * nothing completes, with a limit of limit_ns in [1e6, 2e9] nanoseconds; afterwards
 * dmuon_check_status(cuda_stream) returns DMUON_ERR_TIMEOUT (and clears it). Faults and traps are never
 * used.
 */
DMUON_API int dmuon_selftest_bounded_wait(int64_t limit_ns, void* cuda_stream);

/*
 * The checked build. libdmuon_checked.so is built from the same sources with device-side range checks
 * compiled in (the debugging stand-in for a memory checker): every tile's job index and position, every
 * row-wise chunk's matrix, partial-sum slot and cast tile, every AdamW chunk and every small-matrix job's
 * sizes are tested before use; a failed test skips the access and records DMUON_ERR_RANGE for
 * dmuon_check_status. The regular libdmuon.so leaves them out. dmuon_selftest_range_check launches one
 * GEMM whose only tile lies outside its (empty) product, so that in the checked build the next
 * dmuon_check_status returns DMUON_ERR_RANGE; nothing is read or written. In the regular build it returns
 * DMUON_ERR_UNSUPPORTED without launching. No counterpart on the pages.
 */
DMUON_API int dmuon_selftest_range_check(void* cuda_stream);

/* Text of the last error on the calling thread; valid until the next call on that thread. */
DMUON_API const char* dmuon_last_error(void);

/* Library version string, e.g. "dmuon-gb300 0.2.0 (sm_103a)"; the checked build says so. */
DMUON_API const char* dmuon_version(void);

/* Upper bound on workspace bytes per device (0 = no limit). Calls needing more fail with
 * DMUON_ERR_OOM before launching anything. */
DMUON_API int dmuon_set_workspace_limit(size_t bytes);

/* Bytes of workspace the library would need for dmuon_muon_step on these shapes (host query). */
DMUON_API int dmuon_workspace_size(int count, const int64_t* rows, const int64_t* cols, int backend,
                         size_t* bytes_out);

/* Synchronise the current device and free its workspace and cached descriptor tables. */
DMUON_API int dmuon_release_workspace(void);

#ifdef __cplusplus
}
#endif

#endif /* DMUON_H */
