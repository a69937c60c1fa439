// gemm_internal.h -- host-side interfaces between the C-ABI layer and the
// kernel translation units of libgemmf32.so.  Not installed, not exported.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

namespace gemm_f32_impl {

// Default wait limit for every bounded mbarrier wait in the library's kernels.
constexpr long long kDefaultTimeoutNs = 2000000000LL;  // 2 s

// Launch attribute of a kernel that may start before its predecessor in the
// stream ends (programmatic dependent launch); the kernel calls pdl_wait()
// before it touches memory the predecessor writes or reads.
inline cudaLaunchAttribute pdl_attribute() {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

// ---- sgemm_ffma (CUDA-core FFMA kernel) -----------------------------------
struct FfmaConfig {
    int bm, bn, bk, stages, threads, ctas_per_sm;
    int smem_bytes;  // dynamic shared memory per CTA
    int variant;     // 0: 128 x 128 tiles, 8 x 8 per thread; 1: 128 x 256, 8 x 16
};
FfmaConfig ffma_config(int variant);
// Resident CTAs per SM of a variant, from the occupancy calculator.
cudaError_t ffma_ctas_per_sm(int variant, int* ctas_per_sm);

struct FfmaArgs {
    CUtensorMap tmA;  // A as {K, M}, box {bk, bm}, swizzled
    CUtensorMap tmB;  // B as {N, K}, box {bn, bk}, unswizzled
    float* out;             // C, or the split-K partial buffer
    long long ldo;          // row stride of out (elements)
    long long split_stride; // elements between consecutive split partials
    int M, N, K;
    int kb_per_split;       // K blocks (of bk) per split
    int splits;
    int vec_store;          // 1: ldo % 4 == 0 and out 16-byte aligned
    unsigned* fault;
    long long timeout_ns;
    int variant;            // ffma_config variant
    int bn;                 // tile width the B descriptor's box was encoded with
    float alpha, beta;      // output scaling (epilogue.cuh modes)
    int scale_mode;         // 0 plain, 1 alpha, 2 alpha and beta (reads C)
    // 0: split s writes its partial to out + s * split_stride.  2..4 (equal
    // to splits): each tile's splits run as one cluster and add their
    // partials in split order through distributed shared memory; out is C.
    int cluster_splits;
};
cudaError_t launch_sgemm_ffma(const FfmaArgs& a, cudaStream_t s);

// ---- sgemm_3xtf32 (tcgen05 tensor-core kernel) -----------------------------
struct Tf32x3Config {
    int bm, bn, bk, stages, threads;  // bm x bn: output tile of one work unit
    int smem_bytes;
    int pair;    // 1: a two-CTA cluster shares each MMA (M = 256)
    int box_n;   // rows of B^T one CTA loads per stage (TMA box height)
};
// bn = 128 or 256 for one CTA per tile; pair = the 256 x 256 two-CTA kernel
Tf32x3Config tf32x3_config(int bn, bool pair);

struct Tf32x3Args {
    // pre-split operands: A hi / lo as {K, M}, box {bk, bm}, and B^T hi / lo
    // as {K, N}, box {bk, box_n}, all with 128-byte swizzle (A hi may be A
    // itself, with its own row stride: the high part is the fp32 word, which
    // the tensor core truncates to TF32).  split_in_kernel
    // (pair kernel only): tmAhi is A as stored, {K, M}, box {bk, 128}, and
    // tmBhi is B as stored, {N, K}, box {32, bk}; tmAlo and tmBlo are unused.
    CUtensorMap tmAhi, tmAlo;
    CUtensorMap tmBhi, tmBlo;
    int split_in_kernel;
    float* out;
    long long ldo;
    long long split_stride;
    int M, N, K;
    int bn;
    int pair;
    int kb_per_split;
    int splits;
    int vec_store;
    unsigned* fault;
    long long timeout_ns;
    float alpha, beta;      // output scaling (epilogue.cuh modes)
    int scale_mode;
    // pair kernel, splits == 1: the last tail_tiles tiles are cut into
    // tail_splits K shares written to tail_ws (tail_tiles x tail_splits x
    // 256 x 256 floats) and summed into C by a fix-up kernel
    int tail_tiles, tail_splits;
    float* tail_ws;
    // tma_store = 1: the GEMM kernel writes C through shared memory with TMA
    // stores (reading the old C with TMA loads for a beta term), tmC being C
    // as {N, M}, box {16, 32}, 64-byte swizzle (splits == 1 without a
    // cluster split, C 16-byte aligned with N and the row stride multiples
    // of 4, and not the pair kernel that splits in shared memory)
    CUtensorMap tmC;
    int tma_store;
    // single-CTA kernels, 0 or 2..8 (equal to splits, one unit per CTA): each
    // tile's splits run as one cluster and add their partials in split order
    // through distributed shared memory; out is C
    int cluster_splits;
    // the kernel with B's split in tensor memory, splits > 1 with one unit
    // per CTA: out holds the split partials, and the CTAs add them up in
    // split order inside the kernel (counters: 2 x tiles ints, zero between
    // calls) and write c_final (row stride ldc, alpha/beta by c_mode)
    int* counters;
    float* c_final;
    long long ldc;
    int c_mode;
};

// Bytes at the start of every workspace reserved for the in-kernel split-K
// counters: zeroed when the workspace is allocated, and each kernel that
// uses them leaves them zero again.
constexpr size_t kWorkspaceCounterBytes = 4096;
// co-resident two-CTA clusters of the pair kernel on the current device
cudaError_t tf32x3_pair_clusters(int sm_count, int* clusters);
// co-resident clusters of `splits` (1..8) CTAs of the single-CTA kernel with
// 128 x bn tiles on the current device: the SMs do not divide into every
// cluster size (GB300, one CTA per SM: 76 of 2, 46 of 3, 36 of 4, 28 of 5,
// 23 of 6, 15 of 7 or 8)
cudaError_t tf32x3_single_cluster_capacity(int bn, int splits, int* clusters);
// persistent grid: min(units, sm_count) CTAs, or for the pair kernel
// 2 x min(units, co-resident clusters)
cudaError_t launch_sgemm_3xtf32(const Tf32x3Args& a, cudaStream_t s, int sm_count);
// The 128 x 128 kernel with B's split in tensor memory (A and B as stored,
// in tmAhi {K, M} boxes 32 x 128 and tmBhi {N, K} boxes 32 x 32, both with
// 128-byte swizzle); out gets C, or split partials, like the kernels above
// (with cluster_splits, C: the splits of a tile added inside a cluster).
cudaError_t launch_sgemm_3xtf32_tmem(const Tf32x3Args& a, cudaStream_t s, int sm_count);
// clusters of `splits` CTAs of the single-CTA form resident at once
cudaError_t tf32x3_tmem_cluster_capacity(int splits, int* clusters);
Tf32x3Config tf32x3_tmem_config(bool pair);
cudaError_t tf32x3_tmem_ctas_per_sm(int* ctas_per_sm);
// Its wide single-CTA form: 256 x 128 tiles (256 rows m, 128 columns n) with
// N = 256 MMAs and 16-deep stages (A {K, M} boxes 16 x 256 with 64-byte
// swizzle, B {N, K} boxes 32 x 16 with 128-byte swizzle).
cudaError_t launch_sgemm_3xtf32_tmem_wide(const Tf32x3Args& a, cudaStream_t s, int sm_count);
Tf32x3Config tf32x3_tmem_wide_config();
// Its CTA-pair form: 256 x 256 tiles (pair = 1; A {K, M} boxes 32 x 128, B
// {N, K} boxes 32 x 32); co-resident clusters of two on the current device.
cudaError_t launch_sgemm_3xtf32_tmem_pair(const Tf32x3Args& a, cudaStream_t s, int sm_count);
// Adds the tail shares of a pair kernel's K-split last round (tail_ws) into
// C (out, ldo) in share order, with alpha/beta.
cudaError_t launch_pair_tail_fixup(const Tf32x3Args& a, cudaStream_t s);
cudaError_t tf32x3_tmem_pair_clusters(int sm_count, int* clusters);

// ---- TF32 hi/lo staging (tf32_split.cu) --------------------------------------
// hi = x as stored (read by the tensor core as trunc(x)), lo = tf32(x - trunc(x)).
// hi/lo[r*ldd + c] from src[r*lds + c] (same orientation); hi may be null
// (lo only)
cudaError_t launch_split_rows(const float* src, long long lds, long long rows, long long cols,
                              float* hi, float* lo, long long ldd, cudaStream_t s);
// hi/lo[n*ldt + k] from src[k*lds + n] (K x N -> N x K)
cudaError_t launch_split_transpose(const float* src, long long lds, int K, int N, float* hi,
                                   float* lo, long long ldt, cudaStream_t s);
// both of the above in one launch: A (M x K, row stride lda) -> a_hi/a_lo
// (row stride ldd; a_hi may be null) and B (K x N, row stride ldb) ->
// b_hi/b_lo (N x K, ldt)
cudaError_t launch_split_operands(const float* a, long long lda, int M, int K, float* a_hi,
                                  float* a_lo, long long ldd, const float* b, long long ldb, int N,
                                  float* b_hi, float* b_lo, long long ldt, cudaStream_t s);

// ---- helper kernels (gemm_aux.cu) ------------------------------------------
// dst[r*ldd + c] = src[r*lds + c] for r < rows, c < cols
cudaError_t launch_pad_copy(const float* src, long long lds, long long rows, long long cols,
                            float* dst, long long ldd, cudaStream_t s);
// v = sum_{s < splits} ws[s*split_stride + i*ldw + j], s ascending; then
// C[i*ldc + j] = v, alpha v or alpha v + beta C (scale_mode 0, 1, 2)
cudaError_t launch_splitk_reduce(const float* ws, long long split_stride, long long ldw,
                                 int splits, float* C, long long ldc, int M, int N,
                                 float alpha, float beta, int scale_mode, cudaStream_t s);
// dst[c*ldd + r] = src[r*lds + c] for r < rows, c < cols (a transposed copy)
cudaError_t launch_transpose_pad(const float* src, long long lds, long long rows, long long cols,
                                 float* dst, long long ldd, cudaStream_t s);
// C[i*ldc + j] = beta C (or 0 when beta == 0) for i < M, j < N: the K = 0 case
cudaError_t launch_scale_c(float* C, long long ldc, int M, int N, float beta, cudaStream_t s);
// C[0 .. count) = 0
cudaError_t launch_fill_zero(float* C, long long count, cudaStream_t s);
// watchdog self-test: waits on a never-completed barrier for timeout_ns
cudaError_t launch_watchdog_selftest(unsigned* fault, long long timeout_ns, cudaStream_t s);

// gemm_f32_noalloc's fault word on device `dev` (0 if that entry point has
// not set the device up); blocking read, zeroed afterwards when `clear`.
int noalloc_fault_word(int dev, int clear, unsigned* word);

}  // namespace gemm_f32_impl
