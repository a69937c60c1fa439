// tf32_split.cu -- operand staging for the 3xTF32 tensor-core kernel.
//
// Each fp32 value x is written as two TF32 numbers (fp32 bit patterns whose
// low 13 mantissa bits are zero):
//     hi = tf32(x)          round to nearest, ties to even
//     lo = tf32(x - hi)     x - hi is exact in fp32
// so that x = hi + lo up to the rounding of lo (relative 2^-22 of x).  The
// product A*B is then taken as Ahi*Bhi + Ahi*Blo + Alo*Bhi, dropping the
// Alo*Blo term (relative 2^-22): the "split-precision tensor-core correction"
// published by Ootomo and Yokota (2022) and used as "3xTF32" in NVIDIA's
// CUTLASS; the code here is written from that description.
//
// A (M x K, K-contiguous) keeps its layout.  B (K x N, N-contiguous) is
// transposed on the way to N x K so that both tensor-core operands are
// K-major.  Output rows are padded to a multiple of 4 floats (16 bytes) for
// the TMA descriptors.  Both kernels are memory-bound copies.
#include <cstdint>

#include "device_sync.cuh"
#include "gemm_internal.h"

namespace gemm_f32_impl {
namespace {

using gemm_f32_dev::pdl_trigger;

__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rn.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

constexpr int kThreads = 256;

// The kernels' bodies take their block coordinates and grid extent as
// arguments, so that the fused launch below can run A's and B's staging as
// two ranges of one grid.

__device__ __forceinline__ void split_rows_body(const float* __restrict__ src, long long lds,
                                                long long rows, long long cols,
                                                float* __restrict__ hi, float* __restrict__ lo,
                                                long long ldd, unsigned bx, unsigned by,
                                                unsigned gx, unsigned gy) {
    for (long long r = by; r < rows; r += gy) {
        const float* s = src + r * lds;
        for (long long c = static_cast<long long>(bx) * kThreads + threadIdx.x; c < cols;
             c += static_cast<long long>(gx) * kThreads) {
            const float x = s[c];
            const float h = to_tf32(x);
            hi[r * ldd + c] = h;
            lo[r * ldd + c] = to_tf32(x - h);
        }
    }
}

// Vector form: 4 consecutive elements per thread (cols, lds, ldd multiples of
// 4 and both bases 16-byte aligned); one block covers 1024 columns of a row.
__device__ __forceinline__ void split_rows4_body(const float4* __restrict__ src, long long lds4,
                                                 long long rows, long long cols4,
                                                 float4* __restrict__ hi, float4* __restrict__ lo,
                                                 long long ldd4, unsigned bx, unsigned by,
                                                 unsigned gx, unsigned gy) {
    for (long long r = by; r < rows; r += gy) {
        for (long long c = static_cast<long long>(bx) * kThreads + threadIdx.x; c < cols4;
             c += static_cast<long long>(gx) * kThreads) {
            const float4 x = src[r * lds4 + c];
            float4 h, l;
            h.x = to_tf32(x.x);
            h.y = to_tf32(x.y);
            h.z = to_tf32(x.z);
            h.w = to_tf32(x.w);
            l.x = to_tf32(x.x - h.x);
            l.y = to_tf32(x.y - h.y);
            l.z = to_tf32(x.z - h.z);
            l.w = to_tf32(x.w - h.w);
            hi[r * ldd4 + c] = h;
            lo[r * ldd4 + c] = l;
        }
    }
}

// 32 x 32 tiles through shared memory (row pitch 33 floats: the transposed
// read of a column hits 32 different banks).  src is K x N with row stride
// lds; hi/lo are N x K with row stride ldt.  256 threads as 32 x 8.
__device__ __forceinline__ void split_transpose_body(const float* __restrict__ src, long long lds,
                                                     int K, int N, float* __restrict__ hi,
                                                     float* __restrict__ lo, long long ldt,
                                                     unsigned bx, unsigned by, unsigned gy,
                                                     float (*tile)[33]) {
    const int tx = threadIdx.x & 31;
    const int ty = threadIdx.x >> 5;
    const int kblocks = (K + 31) / 32;
    const int n0 = static_cast<int>(bx) * 32;
    for (int kb = static_cast<int>(by); kb < kblocks; kb += static_cast<int>(gy)) {
        const int k0 = kb * 32;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = k0 + ty + 8 * i;
            const int n = n0 + tx;
            tile[ty + 8 * i][tx] = (k < K && n < N) ? src[static_cast<long long>(k) * lds + n] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int n = n0 + ty + 8 * i;
            const int k = k0 + tx;
            if (n < N && k < K) {
                const float x = tile[tx][ty + 8 * i];
                const float h = to_tf32(x);
                hi[static_cast<long long>(n) * ldt + k] = h;
                lo[static_cast<long long>(n) * ldt + k] = to_tf32(x - h);
            }
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kThreads)
split_rows_kernel(const float* __restrict__ src, long long lds, long long rows, long long cols,
                  float* __restrict__ hi, float* __restrict__ lo, long long ldd) {
    pdl_trigger();  // the GEMM may launch; it waits for this grid to finish
    split_rows_body(src, lds, rows, cols, hi, lo, ldd, blockIdx.x, blockIdx.y, gridDim.x,
                    gridDim.y);
}

__global__ void __launch_bounds__(kThreads)
split_rows4_kernel(const float4* __restrict__ src, long long lds4, long long rows, long long cols4,
                   float4* __restrict__ hi, float4* __restrict__ lo, long long ldd4) {
    pdl_trigger();  // the GEMM may launch; it waits for this grid to finish
    split_rows4_body(src, lds4, rows, cols4, hi, lo, ldd4, blockIdx.x, blockIdx.y, gridDim.x,
                     gridDim.y);
}

__global__ void __launch_bounds__(kThreads)
split_transpose_kernel(const float* __restrict__ src, long long lds, int K, int N,
                       float* __restrict__ hi, float* __restrict__ lo, long long ldt) {
    pdl_trigger();  // the GEMM may launch; it waits for this grid to finish
    __shared__ float tile[32][33];
    split_transpose_body(src, lds, K, N, hi, lo, ldt, blockIdx.x, blockIdx.y, gridDim.y, tile);
}

// One launch for both operands of a call: blocks [0, ga_x * ga_y) split the
// rows of A (vector form when a_vec), the rest split and transpose B.
__global__ void __launch_bounds__(kThreads)
split_operands_kernel(const float* __restrict__ a, long long lda, long long a_rows,
                      long long a_cols, float* __restrict__ a_hi, float* __restrict__ a_lo,
                      long long ldd, int a_vec, unsigned ga_x, unsigned ga_y,
                      const float* __restrict__ b, long long ldb, int K, int N,
                      float* __restrict__ b_hi, float* __restrict__ b_lo, long long ldt,
                      unsigned gb_x, unsigned gb_y) {
    pdl_trigger();  // the GEMM may launch; it waits for this grid to finish
    __shared__ float tile[32][33];
    const unsigned na = ga_x * ga_y;
    if (blockIdx.x < na) {
        const unsigned bx = blockIdx.x % ga_x, by = blockIdx.x / ga_x;
        if (a_vec)
            split_rows4_body(reinterpret_cast<const float4*>(a), lda / 4, a_rows, a_cols / 4,
                             reinterpret_cast<float4*>(a_hi), reinterpret_cast<float4*>(a_lo),
                             ldd / 4, bx, by, ga_x, ga_y);
        else
            split_rows_body(a, lda, a_rows, a_cols, a_hi, a_lo, ldd, bx, by, ga_x, ga_y);
    } else {
        const unsigned i = blockIdx.x - na;
        split_transpose_body(b, ldb, K, N, b_hi, b_lo, ldt, i % gb_x, i / gb_x, gb_y, tile);
    }
}

struct RowsGrid {
    bool vec;
    unsigned gx, gy;
};
RowsGrid rows_grid(const float* src, long long lds, long long rows, long long cols,
                   const float* hi, const float* lo, long long ldd) {
    RowsGrid g;
    g.vec = (cols % 4 == 0) && (lds % 4 == 0) && (ldd % 4 == 0) &&
            ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(hi) |
              reinterpret_cast<uintptr_t>(lo)) % 16 == 0);
    long long gx = ((g.vec ? cols / 4 : cols) + kThreads - 1) / kThreads;
    if (gx > 64) gx = 64;
    g.gx = static_cast<unsigned>(gx);
    g.gy = static_cast<unsigned>(rows < 65535 ? rows : 65535);
    return g;
}

}  // namespace

cudaError_t launch_split_rows(const float* src, long long lds, long long rows, long long cols,
                              float* hi, float* lo, long long ldd, cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const RowsGrid g = rows_grid(src, lds, rows, cols, hi, lo, ldd);
    if (g.vec)
        split_rows4_kernel<<<dim3(g.gx, g.gy), kThreads, 0, s>>>(
            reinterpret_cast<const float4*>(src), lds / 4, rows, cols / 4,
            reinterpret_cast<float4*>(hi), reinterpret_cast<float4*>(lo), ldd / 4);
    else
        split_rows_kernel<<<dim3(g.gx, g.gy), kThreads, 0, s>>>(src, lds, rows, cols, hi, lo, ldd);
    return cudaGetLastError();
}

cudaError_t launch_split_transpose(const float* src, long long lds, int K, int N, float* hi,
                                   float* lo, long long ldt, cudaStream_t s) {
    if (K <= 0 || N <= 0) return cudaSuccess;
    const long long kblocks = (static_cast<long long>(K) + 31) / 32;
    dim3 grid(static_cast<unsigned>((N + 31) / 32),
              static_cast<unsigned>(kblocks < 65535 ? kblocks : 65535));
    split_transpose_kernel<<<grid, kThreads, 0, s>>>(src, lds, K, N, hi, lo, ldt);
    return cudaGetLastError();
}

cudaError_t launch_split_operands(const float* a, long long lda, int M, int K, float* a_hi,
                                  float* a_lo, long long ldd, const float* b, long long ldb, int N,
                                  float* b_hi, float* b_lo, long long ldt, cudaStream_t s) {
    if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
    const RowsGrid ga = rows_grid(a, lda, M, K, a_hi, a_lo, ldd);
    const long long kblocks = (static_cast<long long>(K) + 31) / 32;
    const unsigned gb_x = static_cast<unsigned>((N + 31) / 32);
    const unsigned gb_y = static_cast<unsigned>(kblocks < 65535 ? kblocks : 65535);
    const unsigned long long blocks =
        static_cast<unsigned long long>(ga.gx) * ga.gy + static_cast<unsigned long long>(gb_x) * gb_y;
    if (blocks > 0x7FFFFFFFull) {
        // too many blocks for one 1-D grid: two launches
        cudaError_t e = launch_split_rows(a, lda, M, K, a_hi, a_lo, ldd, s);
        if (e != cudaSuccess) return e;
        return launch_split_transpose(b, ldb, K, N, b_hi, b_lo, ldt, s);
    }
    split_operands_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
        a, lda, M, K, a_hi, a_lo, ldd, ga.vec ? 1 : 0, ga.gx, ga.gy, b, ldb, K, N, b_hi, b_lo,
        ldt, gb_x, gb_y);
    return cudaGetLastError();
}

}  // namespace gemm_f32_impl
