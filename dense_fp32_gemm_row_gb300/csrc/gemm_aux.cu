// gemm_aux.cu -- the memory-bound helper kernels of the GEMM path:
//
//  * pad_copy:       copies a row-major operand into a buffer whose row
//                    stride is a multiple of 16 bytes and whose base is
//                    256-byte aligned, the form a TMA descriptor requires
//                    (16-byte stores of four columns a thread).
//  * splitk_reduce:  C = sum of the split-K partial products, added in split
//                    order 0, 1, ..., S-1 so that the result is deterministic;
//                    the partials are loaded several at a time (independent
//                    loads in flight), and few outputs with many partials
//                    get one thread per output over a flat grid.
//  * fill_zero:      C = 0 for K == 0 (the empty sum of the lecture-12
//                    golden reference); scale_c: C = beta C for K == 0.
//  * transpose_pad:  a transposed copy, for operands stored the other way
//                    round from what a kernel reads.
//  * watchdog:       a self-test that waits on a barrier nothing completes.
//
// All are grid-stride loops with coalesced accesses along rows; they are
// bounded by HBM (or L2) bandwidth or, for a reduction of few outputs, by the
// latency of each thread's loads, never by arithmetic.
#include <cstdint>

#include "device_sync.cuh"
#include "epilogue.cuh"
#include "gemm_internal.h"

namespace gemm_f32_impl {
namespace {

using namespace gemm_f32_dev;

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
pad_copy_kernel(const float* __restrict__ src, long long lds, long long rows, long long cols,
                float* __restrict__ dst, long long ldd) {
    pdl_trigger();
    for (long long r = blockIdx.y; r < rows; r += gridDim.y) {
        const float* s = src + r * lds;
        float* d = dst + r * ldd;
        for (long long c = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; c < cols;
             c += static_cast<long long>(gridDim.x) * kThreads)
            d[c] = s[c];
    }
}

// Vector form: the destination rows 16-byte aligned (ldd a multiple of 4,
// 16-byte base).  A thread copies four adjacent columns: four scalar loads
// of the source (coalesced across the warp whatever its alignment) and one
// 16-byte store, so that each thread has four loads in flight; a bounded
// grid of blocks steps over the rows (one 256-column block a row moved 1 KB
// a block and left the copies of deep-K operands at a fraction of HBM
// bandwidth).
__global__ void __launch_bounds__(kThreads)
pad_copy4_kernel(const float* __restrict__ src, long long lds, long long rows, long long cols,
                 float* __restrict__ dst, long long ldd) {
    pdl_trigger();
    const long long quads = (cols + 3) / 4;
    for (long long r = blockIdx.y; r < rows; r += gridDim.y) {
        const float* s = src + r * lds;
        float* d = dst + r * ldd;
        for (long long q = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; q < quads;
             q += static_cast<long long>(gridDim.x) * kThreads) {
            const long long c = 4 * q;
            if (c + 3 < cols) {
                *reinterpret_cast<float4*>(d + c) = make_float4(s[c], s[c + 1], s[c + 2], s[c + 3]);
            } else {
                for (long long i = c; i < cols; ++i) d[i] = s[i];
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads)
splitk_reduce_kernel(const float* __restrict__ ws, long long split_stride, long long ldw,
                     int splits, float* __restrict__ C, long long ldc, int M, int N, float alpha,
                     float beta, int mode) {
    pdl_wait();  // the partials of the GEMM kernel before it
    for (long long r = blockIdx.y; r < M; r += gridDim.y) {
        const float* w = ws + r * ldw;
        float* c = C + r * ldc;
        for (long long j = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; j < N;
             j += static_cast<long long>(gridDim.x) * kThreads) {
            float sum = w[j];
            for (int s = 1; s < splits; ++s) sum += w[s * split_stride + j];
            c[j] = scale1(sum, c + j, alpha, beta, mode);
        }
    }
}

// Vector form: the partials are read as float4 (ldw and the split stride
// multiples of 4, ldw at least N rounded up to 4, the workspace 16-byte
// aligned: the padding columns are read and dropped), kVecBatch at a time
// (independent loads in flight), and added in split order, as above.  C is
// written as float4 where its rows allow (cvec: ldc a multiple of 4 and C
// 16-byte aligned) and element by element otherwise, so that an odd N keeps
// the vector loads.
constexpr int kVecBatch = 4;
__global__ void __launch_bounds__(kThreads)
splitk_reduce4_kernel(const float4* __restrict__ ws, long long split_stride4, long long ldw4,
                      int splits, float* __restrict__ C, long long ldc, int M, int N, bool cvec,
                      float alpha, float beta, int mode) {
    pdl_wait();  // the partials of the GEMM kernel before it
    const long long N4 = (static_cast<long long>(N) + 3) / 4;
    for (long long r = blockIdx.y; r < M; r += gridDim.y) {
        const float4* w = ws + r * ldw4;
        float* c = C + r * ldc;
        for (long long j = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; j < N4;
             j += static_cast<long long>(gridDim.x) * kThreads) {
            float4 sum = w[j];
            for (int s0 = 1; s0 < splits; s0 += kVecBatch) {
                float4 v[kVecBatch];
#pragma unroll
                for (int b = 0; b < kVecBatch; ++b)
                    if (s0 + b < splits) v[b] = w[(s0 + b) * split_stride4 + j];
#pragma unroll
                for (int b = 0; b < kVecBatch; ++b) {
                    if (s0 + b < splits) {
                        sum.x += v[b].x;
                        sum.y += v[b].y;
                        sum.z += v[b].z;
                        sum.w += v[b].w;
                    }
                }
            }
            store4(c, static_cast<int>(4 * j), N, sum, cvec, alpha, beta, mode);
        }
    }
}

// Few outputs, many partials (256 x 256 x 65536: 65536 outputs, 76 partials
// each): one output per thread over a flat index, so that every SM takes
// part, with kDeepBatch partials loaded at once; each thread's chain of
// round trips to L2 is what bounds the kernel.  Same split order.
constexpr int kDeepBatch = 40;
__global__ void __launch_bounds__(kThreads)
splitk_reduce_deep_kernel(const float* __restrict__ ws, long long split_stride, long long ldw,
                          int splits, float* __restrict__ C, long long ldc, int M, int N,
                          float alpha, float beta, int mode) {
    pdl_wait();  // the partials of the GEMM kernel before it
    const long long total = static_cast<long long>(M) * N;
    for (long long idx = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * kThreads) {
        const long long r = idx / N;
        const long long j = idx - r * N;
        const float* w = ws + r * ldw + j;
        float sum = w[0];
        for (int s0 = 1; s0 < splits; s0 += kDeepBatch) {
            float v[kDeepBatch];
#pragma unroll
            for (int b = 0; b < kDeepBatch; ++b)
                if (s0 + b < splits) v[b] = w[static_cast<long long>(s0 + b) * split_stride];
#pragma unroll
            for (int b = 0; b < kDeepBatch; ++b)
                if (s0 + b < splits) sum += v[b];
        }
        float* c = C + r * ldc + j;
        *c = scale1(sum, c, alpha, beta, mode);
    }
}

// 32 x 32 tiles through shared memory, row pitch 33 (conflict-free columns).
__global__ void __launch_bounds__(256)
transpose_pad_kernel(const float* __restrict__ src, long long lds, long long rows, long long cols,
                     float* __restrict__ dst, long long ldd) {
    pdl_trigger();
    __shared__ float tile[32][33];
    const int tx = threadIdx.x;
    const int ty = threadIdx.y;
    const long long c0 = static_cast<long long>(blockIdx.x) * 32;
    const long long rblocks = (rows + 31) / 32;
    for (long long rb = blockIdx.y; rb < rblocks; rb += gridDim.y) {
        const long long r0 = rb * 32;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const long long r = r0 + ty + 8 * i, c = c0 + tx;
            tile[ty + 8 * i][tx] = (r < rows && c < cols) ? src[r * lds + c] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const long long c = c0 + ty + 8 * i, r = r0 + tx;
            if (c < cols && r < rows) dst[c * ldd + r] = tile[tx][ty + 8 * i];
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kThreads)
scale_c_kernel(float* __restrict__ C, long long ldc, int M, int N, float beta) {
    for (long long r = blockIdx.y; r < M; r += gridDim.y)
        for (long long j = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; j < N;
             j += static_cast<long long>(gridDim.x) * kThreads)
            C[r * ldc + j] = beta == 0.0f ? 0.0f : beta * C[r * ldc + j];
}

__global__ void __launch_bounds__(kThreads) fill_zero_kernel(float* __restrict__ C, long long n) {
    for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kThreads)
        C[i] = 0.0f;
}

__global__ void watchdog_selftest_kernel(unsigned* fault, long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // Nothing arrives on the barrier, so its first phase never completes and
    // the bounded wait must give up after timeout_ns and flag the fault word.
    mbar_wait(b, 0, timeout_ns, threadIdx.x == 0 ? fault : nullptr, kFaultSelfTest);
}

unsigned grid_1d(long long work, long long per_block, unsigned cap) {
    long long g = (work + per_block - 1) / per_block;
    if (g < 1) g = 1;
    return static_cast<unsigned>(g < cap ? g : cap);
}

}  // namespace

cudaError_t launch_pad_copy(const float* src, long long lds, long long rows, long long cols,
                            float* dst, long long ldd, cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    if (ldd % 4 == 0 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
        // about 2048 blocks in all: a few per SM, each over many rows
        const unsigned gx = grid_1d((cols + 3) / 4, kThreads, 64);
        const long long gy_cap = (2048 + gx - 1) / gx;
        const unsigned gy = static_cast<unsigned>(rows < gy_cap ? rows : gy_cap);
        pad_copy4_kernel<<<dim3(gx, gy), kThreads, 0, s>>>(src, lds, rows, cols, dst, ldd);
        return cudaGetLastError();
    }
    dim3 grid(grid_1d(cols, kThreads, 64), static_cast<unsigned>(rows < 65535 ? rows : 65535));
    pad_copy_kernel<<<grid, kThreads, 0, s>>>(src, lds, rows, cols, dst, ldd);
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const float* ws, long long split_stride, long long ldw,
                                 int splits, float* C, long long ldc, int M, int N, float alpha,
                                 float beta, int scale_mode, cudaStream_t s) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    const unsigned gy = static_cast<unsigned>(M < 65535 ? M : 65535);
    const bool vec = (ldw % 4 == 0) && (ldw >= (static_cast<long long>(N) + 3) / 4 * 4) &&
                     (split_stride % 4 == 0) && (reinterpret_cast<uintptr_t>(ws) % 16 == 0);
    const bool cvec = (ldc % 4 == 0) && (reinterpret_cast<uintptr_t>(C) % 16 == 0);
    // launched programmatically after the GEMM kernel (pdl_wait in the kernel)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (splits >= 8 && static_cast<long long>(M) * N <= (1LL << 20)) {
        // latency-bound: a flat grid of one output per thread
        const long long total = static_cast<long long>(M) * N;
        const long long blocks = (total + kThreads - 1) / kThreads;
        cfg.gridDim = dim3(static_cast<unsigned>(blocks < 65535 ? blocks : 65535));
        e = cudaLaunchKernelEx(&cfg, splitk_reduce_deep_kernel, ws, split_stride, ldw, splits, C,
                               ldc, M, N, alpha, beta, scale_mode);
    } else if (vec) {
        cfg.gridDim = dim3(grid_1d((N + 3) / 4, kThreads, 64), gy);
        e = cudaLaunchKernelEx(&cfg, splitk_reduce4_kernel, reinterpret_cast<const float4*>(ws),
                               split_stride / 4, ldw / 4, splits, C, ldc, M, N, cvec, alpha, beta,
                               scale_mode);
    } else {
        cfg.gridDim = dim3(grid_1d(N, kThreads, 64), gy);
        e = cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, ws, split_stride, ldw, splits, C, ldc,
                               M, N, alpha, beta, scale_mode);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_transpose_pad(const float* src, long long lds, long long rows, long long cols,
                                 float* dst, long long ldd, cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const long long rblocks = (rows + 31) / 32;
    dim3 grid(static_cast<unsigned>((cols + 31) / 32),
              static_cast<unsigned>(rblocks < 65535 ? rblocks : 65535));
    transpose_pad_kernel<<<grid, dim3(32, 8), 0, s>>>(src, lds, rows, cols, dst, ldd);
    return cudaGetLastError();
}

cudaError_t launch_scale_c(float* C, long long ldc, int M, int N, float beta, cudaStream_t s) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    dim3 grid(grid_1d(N, kThreads, 64), static_cast<unsigned>(M < 65535 ? M : 65535));
    scale_c_kernel<<<grid, kThreads, 0, s>>>(C, ldc, M, N, beta);
    return cudaGetLastError();
}

cudaError_t launch_fill_zero(float* C, long long count, cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    fill_zero_kernel<<<grid_1d(count, kThreads, 4096), kThreads, 0, s>>>(C, count);
    return cudaGetLastError();
}

cudaError_t launch_watchdog_selftest(unsigned* fault, long long timeout_ns, cudaStream_t s) {
    watchdog_selftest_kernel<<<1, 32, 0, s>>>(fault, timeout_ns);
    return cudaGetLastError();
}

}  // namespace gemm_f32_impl
