// tf32_split.cu -- operand staging for the 3xTF32 tensor-core kernel.
//
// Each fp32 value x is written as two TF32 numbers (fp32 bit patterns whose
// low 13 mantissa bits are zero):
//     hi = tf32(x)          round to nearest, ties away from zero
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

#include "gemm_internal.h"

namespace gemm_f32_impl {
namespace {

__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
split_rows_kernel(const float* __restrict__ src, long long lds, long long rows, long long cols,
                  float* __restrict__ hi, float* __restrict__ lo, long long ldd) {
    for (long long r = blockIdx.y; r < rows; r += gridDim.y) {
        const float* s = src + r * lds;
        for (long long c = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; c < cols;
             c += static_cast<long long>(gridDim.x) * kThreads) {
            const float x = s[c];
            const float h = to_tf32(x);
            hi[r * ldd + c] = h;
            lo[r * ldd + c] = to_tf32(x - h);
        }
    }
}

// Vector form: 4 consecutive elements per thread (cols, lds, ldd multiples of
// 4 and both bases 16-byte aligned); one block covers 1024 columns of a row.
__global__ void __launch_bounds__(kThreads)
split_rows4_kernel(const float4* __restrict__ src, long long lds4, long long rows, long long cols4,
                   float4* __restrict__ hi, float4* __restrict__ lo, long long ldd4) {
    for (long long r = blockIdx.y; r < rows; r += gridDim.y) {
        for (long long c = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; c < cols4;
             c += static_cast<long long>(gridDim.x) * kThreads) {
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
// lds; hi/lo are N x K with row stride ldt.
__global__ void __launch_bounds__(256)
split_transpose_kernel(const float* __restrict__ src, long long lds, int K, int N,
                       float* __restrict__ hi, float* __restrict__ lo, long long ldt) {
    __shared__ float tile[32][33];
    const int tx = threadIdx.x;  // 0..31
    const int ty = threadIdx.y;  // 0..7
    const int kblocks = (K + 31) / 32;
    const int n0 = blockIdx.x * 32;
    for (int kb = blockIdx.y; kb < kblocks; kb += gridDim.y) {
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

}  // namespace

cudaError_t launch_split_rows(const float* src, long long lds, long long rows, long long cols,
                              float* hi, float* lo, long long ldd, cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const unsigned gy = static_cast<unsigned>(rows < 65535 ? rows : 65535);
    const bool vec = (cols % 4 == 0) && (lds % 4 == 0) && (ldd % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(hi) |
                       reinterpret_cast<uintptr_t>(lo)) % 16 == 0);
    if (vec) {
        long long gx = (cols / 4 + kThreads - 1) / kThreads;
        if (gx > 64) gx = 64;
        split_rows4_kernel<<<dim3(static_cast<unsigned>(gx), gy), kThreads, 0, s>>>(
            reinterpret_cast<const float4*>(src), lds / 4, rows, cols / 4,
            reinterpret_cast<float4*>(hi), reinterpret_cast<float4*>(lo), ldd / 4);
    } else {
        long long gx = (cols + kThreads - 1) / kThreads;
        if (gx > 64) gx = 64;
        split_rows_kernel<<<dim3(static_cast<unsigned>(gx), gy), kThreads, 0, s>>>(
            src, lds, rows, cols, hi, lo, ldd);
    }
    return cudaGetLastError();
}

cudaError_t launch_split_transpose(const float* src, long long lds, int K, int N, float* hi,
                                   float* lo, long long ldt, cudaStream_t s) {
    if (K <= 0 || N <= 0) return cudaSuccess;
    const long long kblocks = (static_cast<long long>(K) + 31) / 32;
    dim3 grid(static_cast<unsigned>((N + 31) / 32),
              static_cast<unsigned>(kblocks < 65535 ? kblocks : 65535));
    split_transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(src, lds, K, N, hi, lo, ldt);
    return cudaGetLastError();
}

}  // namespace gemm_f32_impl
