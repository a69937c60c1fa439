/*
 * gemm_f32.h -- C ABI of libgemmf32.so, single-precision dense matrix
 * multiply C = A * B for one NVIDIA GB300 (sm_103a).
 *
 * Operation ("Lecture 12: final project", runguoli.com ECE408 notes l12,
 * section 2, the general M/N/K kernel tiledMatMulKernel, and section 3, the
 * CPU golden reference):
 *
 *     C[i][j] = sum_{k < K} A[i][k] * B[k][j]      0 <= i < M, 0 <= j < N
 *
 * Layout: A is M x K, B is K x N, C is M x N, all packed row-major
 * (leading dimensions K, N and N elements).  There is no alpha, beta or
 * transpose: C is overwritten.  All three are 4-byte floats in DEVICE memory
 * of the current CUDA device; any alignment is accepted (4-byte aligned
 * pointers that are not 16-byte aligned, and row strides that are not a
 * multiple of 16 bytes, are served through an internal padded copy).
 *
 * Accuracy: every algorithm is checked against the double-accumulating CPU
 * reference within |C - C_ref| <= 1e-3 + 1e-3 |C_ref| elementwise (the
 * section 4 atol/rtol of the same page).  Results are run-to-run
 * deterministic for a given (shape, algo, splits) on a given device.
 *
 * Edge semantics (same page, section 7, the early exits of main): a negative
 * dimension is an error; M == 0 or N == 0 returns success and launches
 * nothing; K == 0 writes C = 0.  Elements of memory outside C are never
 * written (out-of-range rows and columns of a boundary tile are skipped, the
 * lecture-5 coarsened kernel's predicated store).
 *
 * Ownership and ordering: the caller owns A, B and C; the library reads A
 * and B, writes C and its own workspace, and keeps no reference to any of
 * them after the call returns.  Every call is asynchronous on `stream`
 * (enqueue and return; no implicit synchronisation).  The library owns a
 * workspace per (device, stream), grown on demand: a call that must grow it
 * synchronises that stream first.  gemm_f32_release() frees all of it.
 * The entry points are thread-safe.
 *
 * CUDA graphs: the calls that take a stream can be captured from it
 * (cudaStreamBeginCapture) and replayed; the graph keeps the pointers,
 * shapes and plan of the capture and reads what the buffers hold at replay.
 * The first call on a device sets it up, and a call may have to grow the
 * stream's workspace (or the host entry's device copies); neither is allowed
 * during a capture, so such a call returns GEMM_F32_ERR_CAPTURE without
 * enqueuing anything.  Issue each captured call once on the same stream
 * before capturing it.  Device memory a captured call uses (the stream's
 * workspace, the host entry's device copies) stays allocated while later
 * calls grow those buffers, until gemm_f32_release(): do not release while
 * a graph that holds such a call may still be replayed.
 *
 * Errors: 0 is success.  Negative values are library errors (GEMM_F32_ERR_*),
 * positive values are the cudaError_t of the failing CUDA runtime call.  No
 * entry point exits or aborts the process.  Nothing runs on the host CPU:
 * there is no CPU fallback, and a device other than sm_103 is rejected.
 */
#ifndef GEMM_F32_H
#define GEMM_F32_H

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define GEMM_F32_SUCCESS                 0
/* negative dimension; NULL pointer with a nonzero extent; unknown algo;
 * splits out of range; C overlapping A or B; a size product that overflows */
#define GEMM_F32_ERR_INVALID_VALUE      (-1)
/* no CUDA device, or the current device is not compute capability 10.3 */
#define GEMM_F32_ERR_UNSUPPORTED_DEVICE (-2)
/* the workspace could not be allocated */
#define GEMM_F32_ERR_WORKSPACE          (-3)
/* a kernel gave up waiting on one of its own pipeline barriers (watchdog) */
#define GEMM_F32_ERR_DEVICE_TIMEOUT     (-4)
/* the driver rejected a tensor-memory-access descriptor */
#define GEMM_F32_ERR_DESCRIPTOR         (-5)
/* the stream is being captured into a CUDA graph and the call would first
 * have to set up this device or allocate device memory (a larger workspace,
 * the host entry's device copies), which capture does not allow: issue the
 * same call once on the stream before capturing it.  Nothing was enqueued. */
#define GEMM_F32_ERR_CAPTURE            (-6)

/* ---- algorithms -------------------------------------------------------- */
/* Choose by shape: the tensor-core 3xTF32 kernels, except the CUDA-core
 * kernel for tiny problems (under 5e7 multiply-adds); among the tensor-core
 * kernels, those that split A and B in shared memory when staging them
 * would cost more than it saves (few flops per operand element). */
#define GEMM_F32_ALGO_AUTO    0
/* CUDA-core FFMA kernel: TMA-fed, swizzled shared-memory tiles, mbarrier
 * pipeline, 8x8 or 8x16 register tile per thread. */
#define GEMM_F32_ALGO_FFMA    1
/* Tensor-core kernel: each operand x split into a TF32 high part trunc(x)
 * (the fp32 word itself, which the tensor core reads truncated) and a TF32
 * low part tf32(x - trunc(x)); three tcgen05 products hi*hi + hi*lo + lo*hi
 * accumulated in tensor memory in fp32, promoted every 128 K into fp32
 * registers.  Non-finite operands: an Inf's low part is Inf - Inf = NaN, so
 * an output that is +-Inf in exact arithmetic may come back NaN; NaN inputs
 * still give NaN, and outputs whose row of op(A) and column of op(B) are
 * finite are unaffected.  The FFMA kernel follows IEEE fp32 there. */
#define GEMM_F32_ALGO_3XTF32  2

/* Largest explicit split-K factor accepted by gemm_f32_algo_splitk. */
#define GEMM_F32_MAX_SPLITS   256

/*
 * gemm_f32 -- C = A * B with the algorithm the library picks for the shape.
 * Same as gemm_f32_algo(A, B, C, M, N, K, GEMM_F32_ALGO_AUTO, stream).
 * A: M*K floats, B: K*N floats, C: M*N floats, device pointers, row-major.
 */
int gemm_f32(const float* A, const float* B, float* C, int M, int N, int K,
             cudaStream_t stream);

/*
 * gemm_f32_algo -- as gemm_f32 with an explicit per-call algorithm
 * (GEMM_F32_ALGO_*).  There is no global state: the choice applies to this
 * call only.  The split-K factor is chosen by the library.
 */
int gemm_f32_algo(const float* A, const float* B, float* C, int M, int N, int K,
                  int algo, cudaStream_t stream);

/*
 * gemm_f32_algo_splitk -- as gemm_f32_algo with an explicit split of the
 * K dimension.  splits == 0 lets the library choose; 1 disables splitting;
 * 2..GEMM_F32_MAX_SPLITS computes that many partial products over disjoint
 * K ranges into the workspace and adds them in a fixed order (split 0 first)
 * in a separate kernel, so the result is deterministic.  A split count
 * larger than the number of K blocks is reduced to it.
 */
int gemm_f32_algo_splitk(const float* A, const float* B, float* C, int M, int N, int K,
                         int algo, int splits, cudaStream_t stream);

/*
 * gemm_f32_ex -- the general row-major form
 *
 *     C = alpha * op(A) * op(B) + beta * C
 *
 * op(A) is M x K: element (i, k) is A[i*lda + k] (transa == 0, A stored
 * M x K, lda >= K) or A[k*lda + i] (transa == 1, A stored K x M, lda >= M).
 * op(B) is K x N: element (k, j) is B[k*ldb + j] (transb == 0, ldb >= N) or
 * B[j*ldb + k] (transb == 1, B stored N x K, ldb >= K).  C[i][j] is
 * C[i*ldc + j], ldc >= N.  Leading dimensions are in elements.  With
 * beta == 0 the old C is not read (NaN or garbage there is harmless); with
 * alpha == 0 or K == 0 A and B are not read and C = beta * C.  algo and
 * splits as for gemm_f32_algo_splitk.  Operands that TMA cannot read in
 * place (transposed for the CUDA-core kernel, or a row stride / base not
 * 16-byte aligned) are first copied into the workspace.  The pages have only
 * the packed alpha = 1, beta = 0 form; this is the same product with the
 * interface a BLAS-style caller expects.  transa or transb other than 0 or
 * 1, or a leading dimension below its minimum, is GEMM_F32_ERR_INVALID_VALUE.
 */
int gemm_f32_ex(int transa, int transb, int M, int N, int K, float alpha, const float* A,
                long long lda, const float* B, long long ldb, float beta, float* C,
                long long ldc, int algo, int splits, cudaStream_t stream);

/*
 * gemm_f32_algo_splitk_ev -- as gemm_f32_algo_splitk, and, for profiling,
 * records `main_begin` on `stream` just before the main GEMM kernel is
 * launched and `main_end` just after it (either may be NULL).  The events
 * must belong to the current device.  Staging copies and the split-K
 * reduction, when a call has them, fall outside the pair.
 */
int gemm_f32_algo_splitk_ev(const float* A, const float* B, float* C, int M, int N, int K,
                            int algo, int splits, cudaStream_t stream,
                            cudaEvent_t main_begin, cudaEvent_t main_end);

/*
 * gemm_f32_host -- C = A * B where A, B and C are HOST pointers (row-major,
 * same shapes as gemm_f32).  The library copies B to the device, then walks
 * row panels of A and C: the copy of panel i+1 of A, the GEMM of panel i
 * and the copy back of panel i-1 of C run at the same time on the call's
 * stream and two internal streams.  For deep K with M <= 4096 it walks K
 * panels instead (each accumulates into C, the first GEMM starts after one
 * panel of A and B has arrived, the last panel returns C by row blocks).  Page-locked host memory is needed for
 * that overlap (pageable memory works, serialised).  Asynchronous on
 * `stream`: the host buffers must stay valid, and C is complete, only when
 * `stream` has reached the end of the call.  Device copies of A, B and C
 * are kept in a library buffer per (device, stream), grown on demand like
 * the workspace; gemm_f32_release() frees them.  Same status codes.
 */
int gemm_f32_host(const float* A, const float* B, float* C, int M, int N, int K, int algo,
                  cudaStream_t stream);

/*
 * gemm_f32_plan_info / gemm_f32_plan -- what a call with these arguments
 * would launch, without launching anything.  Needs a device (it reads the
 * SM count); returns a status code like the compute entry points.
 */
typedef struct gemm_f32_plan_info {
    int algo;            /* resolved GEMM_F32_ALGO_FFMA or _3XTF32 (0 if no launch) */
    int splits;          /* resolved split-K factor (1 = none) */
    int tile_m;          /* output tile rows per CTA */
    int tile_n;          /* output tile columns per CTA */
    int tile_k;          /* K depth of one pipeline stage */
    int stages;          /* pipeline stages in shared memory */
    int ctas;            /* CTAs in the main kernel's grid */
    int stage_a;         /* 1 if A goes through a staging copy */
    int stage_b;         /* 1 if B goes through a staging copy */
    int kernels;         /* kernel launches the call makes */
    long long workspace_bytes; /* workspace the call needs */
    int split_in_kernel; /* 1 if the 3XTF32 TF32 split happens inside the GEMM kernel */
    int cluster_reduce;  /* 1 if split-K partials are added inside thread-block clusters
                            (no workspace, no reduction kernel) */
    int ctas_per_sm;     /* CTAs of the main kernel one SM holds at once (occupancy
                            calculator; 0 if it could not be asked) */
    int threads_per_cta; /* threads of one CTA of the main kernel */
    int b_in_tmem;       /* 1 if the 3XTF32 kernel holds B's split in tensor memory
                            (GEMM_F32_TILE_128x128_TMEM, _256x256_TMEM or
                            _256x128_TMEM) */
    int reduce_in_kernel; /* 1 if that kernel adds its split-K partials itself, in
                             split order (no reduction kernel): from 16 splits,
                             with one unit per CTA (or CTA pair) */
} gemm_f32_plan_info;

int gemm_f32_plan(int M, int N, int K, int algo, int splits,
                  const float* A, const float* B, const float* C,
                  gemm_f32_plan_info* out);

/*
 * gemm_f32_plan_ex -- the plan gemm_f32_ex would run for the same transa,
 * transb, sizes, leading dimensions, algo and splits (alpha and beta do not
 * change it), without running it.  A, B, C are optional (NULL): like the
 * leading dimensions they only decide which operands need a padded or
 * transposed copy.  Returns GEMM_F32_SUCCESS or GEMM_F32_ERR_INVALID_VALUE.
 */
int gemm_f32_plan_ex(int transa, int transb, int M, int N, int K, const float* A, long long lda,
                     const float* B, long long ldb, const float* C, long long ldc, int algo,
                     int splits, gemm_f32_plan_info* out);

/*
 * gemm_f32_config / gemm_f32_configured / gemm_f32_plan_config -- run (or
 * plan) C = A * B with a forced kernel configuration instead of the
 * library's choice: the tool behind design-space sweeps ("Lecture 12: final
 * project", the sweep program: try every configuration, check it, time it,
 * rank it).  Arguments as for gemm_f32; the config fields:
 *   algo    GEMM_F32_ALGO_FFMA or _3XTF32 (AUTO only with tile = AUTO)
 *   tile    GEMM_F32_TILE_* below; 0 lets the library choose
 *   splits  as for gemm_f32_algo_splitk (0 = choose)
 * The 256 x 256 CTA-pair tiles exist for 3XTF32 only: _PAIR reads TF32
 * hi/lo copies of A and B written by staging kernels, _PAIR_SPLIT reads A
 * and B as stored and splits each tile in shared memory (same products, no
 * staging pass).  _128x128_SPLIT is the single-CTA 128 x 128 tile that
 * likewise reads A and B as stored and splits them in shared memory (no
 * staging launch: for small calls, where that launch is a large part of
 * the call).  _128x128_TMEM reads A and B as stored too; it splits A in
 * shared memory and B into tensor memory, where the MMA takes B^T as its
 * operand, and computes each 128 x 128 tile transposed (no staging pass and
 * no transpose in shared memory).  _256x256_TMEM is its CTA-pair form
 * (256 x 256 tiles, N = 256 MMAs), and _256x128_TMEM its wide single-CTA
 * form (256 rows by 128 columns, N = 256 MMAs, 16-deep stages).  AUTO
 * takes one of these for row-major A and B (after padded copies where a
 * row stride or base is not 16-byte aligned; for transposed operands, after
 * transposed copies, once C has at least 3M elements), the one a fitted time
 * model finds shorter (the wide form only for operands read in place).
 * Split-K partials are added in split order: by the 128 x 128 forms (staged,
 * _SPLIT and _TMEM) inside a thread-block cluster when 2..8 splits give
 * every CTA one unit and the clusters all fit at once (cluster_reduce = 1:
 * no workspace for them, no reduction launch); by the _TMEM forms inside the
 * kernel from 16 splits (reduce_in_kernel = 1); otherwise by a reduction
 * kernel over a workspace.
 * Invalid combinations return GEMM_F32_ERR_INVALID_VALUE.
 */
#define GEMM_F32_TILE_AUTO          0
#define GEMM_F32_TILE_128x128       1
#define GEMM_F32_TILE_128x256       2
#define GEMM_F32_TILE_256x256_PAIR  3
#define GEMM_F32_TILE_256x256_PAIR_SPLIT 4
#define GEMM_F32_TILE_128x128_SPLIT 5
#define GEMM_F32_TILE_128x128_TMEM  6
#define GEMM_F32_TILE_256x256_TMEM  7
#define GEMM_F32_TILE_256x128_TMEM  8
typedef struct gemm_f32_config {
    int algo;
    int tile;
    int splits;
} gemm_f32_config;

int gemm_f32_configured(const float* A, const float* B, float* C, int M, int N, int K,
                        const gemm_f32_config* cfg, cudaStream_t stream);
int gemm_f32_plan_config(int M, int N, int K, const gemm_f32_config* cfg, const float* A,
                         const float* B, const float* C, gemm_f32_plan_info* out);

/*
 * gemm_f32_device_status -- read (and with clear != 0, reset) the fault
 * words that kernels set on the current device when a bounded wait on one of
 * their pipeline barriers runs out: the library's own word and, once
 * gemm_f32_noalloc has run on the device, the word at the head of that entry
 * point's fixed array.  Synchronises the current device.  Allocates nothing
 * and sets nothing up (a device no call has used reports 0).  Returns 0, or
 * GEMM_F32_ERR_DEVICE_TIMEOUT if a kernel reported a timeout since the last
 * clear, GEMM_F32_ERR_UNSUPPORTED_DEVICE, or a positive cudaError_t.
 */
int gemm_f32_device_status(int clear);

/*
 * gemm_f32_selftest_watchdog -- launch on `stream` one kernel that waits on
 * a shared-memory barrier that nothing ever completes, with a wait limit of
 * timeout_ns nanoseconds (1e3 .. 1e10), then synchronise the stream and
 * return gemm_f32_device_status(1).  A working watchdog returns
 * GEMM_F32_ERR_DEVICE_TIMEOUT and leaves the context usable.
 */
int gemm_f32_selftest_watchdog(long long timeout_ns, cudaStream_t stream);

/*
 * gemm_f32_noalloc -- C = A * B on the CUDA-core FFMA kernel (with split-K
 * when it helps) without allocating any memory.  The pages have no
 * counterpart: this entry point exists for callers that cannot let a library
 * allocate while they run -- programs that reserve their whole device memory
 * budget up front and hand it out from their own pool, and latency-critical
 * loops that cannot absorb the device-wide synchronisation of cudaFree.
 * A, B, C, M, N, K and the result are exactly as for gemm_f32; `splits` is
 * as for gemm_f32_algo_splitk (0 = choose, limited to what fits).
 *
 * Scratch (split-K partial sums, and padded copies of A or B when a row
 * stride or base address is not 16-byte aligned) comes from one fixed
 * device array of GEMM_F32_NOALLOC_SCRATCH_BYTES, compiled into the library
 * and held by every GPU that loads it until the process exits.  A problem
 * whose padded copies, or whose explicitly requested split partials
 * (splits x M x roundup(N, 4) floats), do not fit returns
 * GEMM_F32_ERR_INVALID_VALUE and launches nothing.  The first call on each
 * device looks up the array's device address and clears its fault word (a
 * kernel-side watchdog flag at the start of the array), waiting on `stream`
 * for the clear; make that first call before any stream capture begins (made
 * on a capturing stream it returns GEMM_F32_ERR_CAPTURE and enqueues
 * nothing).  A kernel of this entry point whose bounded wait runs out sets
 * that word and returns; the call itself has already returned 0, so, as with
 * gemm_f32, the timeout is seen through gemm_f32_device_status, which reads
 * and clears this word too.  Every call uses the same array, so
 * calls whose work overlaps on the GPU (other streams, other host threads)
 * race on it: serialise them.  No cudaMalloc, cudaFree or allocating
 * library routine is called.
 */
#define GEMM_F32_NOALLOC_SCRATCH_BYTES (16u << 20)
int gemm_f32_noalloc(const float* A, const float* B, float* C, int M, int N, int K,
                     int splits, cudaStream_t stream);

/*
 * gemm_f32_noalloc_selftest_watchdog -- the watchdog self-test of
 * gemm_f32_selftest_watchdog, aimed at gemm_f32_noalloc's fault word instead
 * of the library's: one kernel on `stream` waits on a barrier nothing
 * completes, with a limit of timeout_ns nanoseconds (1e3 .. 1e10), and the
 * stream is synchronised.  Returns GEMM_F32_ERR_DEVICE_TIMEOUT when the wait
 * gave up and set the word (the working outcome), 0 if it did not.  The bit
 * is left set, as after a real timeout, for gemm_f32_device_status to report
 * and clear.  Allocates nothing; the pages have no counterpart.
 */
int gemm_f32_noalloc_selftest_watchdog(long long timeout_ns, cudaStream_t stream);

/* Release every workspace (synchronises each device that has one). */
int gemm_f32_release(void);

/* Static text for a status code. */
const char* gemm_f32_status_string(int status);

/*
 * gemm_f32_inject_host_fault -- a testing aid that makes one host-side
 * failure happen on purpose, so that a caller's handling of
 * GEMM_F32_ERR_WORKSPACE and GEMM_F32_ERR_DESCRIPTOR can be exercised
 * without any fault on the GPU.  kind = GEMM_F32_INJECT_WORKSPACE: the next
 * workspace (or host-entry buffer) allocation the library attempts reports
 * failure as if cudaMalloc had failed; GEMM_F32_INJECT_DESCRIPTOR: the next
 * TMA descriptor encoding reports failure; GEMM_F32_INJECT_NONE disarms.
 * One-shot and process-wide; off unless called.  The call that meets it
 * returns the status and launches no GEMM kernel (a descriptor failure may
 * follow staging copies already enqueued into the workspace; C is never
 * written); the next call runs normally.  Returns 0, or
 * GEMM_F32_ERR_INVALID_VALUE for an unknown kind.  The pages' counterpart is
 * the error-check macro of "Lecture 5", which exits the process; here the
 * status codes replace the exit.
 */
#define GEMM_F32_INJECT_NONE 0
#define GEMM_F32_INJECT_WORKSPACE 1
#define GEMM_F32_INJECT_DESCRIPTOR 2
int gemm_f32_inject_host_fault(int kind);

/* Library version, major*10000 + minor*100 + patch. */
int gemm_f32_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F32_H */
