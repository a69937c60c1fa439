// tf32_split.cu -- operand staging for the 3xTF32 tensor-core kernel.
//
// Each fp32 value x is taken as the sum of two TF32 numbers:
//     hi = trunc(x)         x with its low 13 mantissa bits cleared
//     lo = tf32(x - hi)     x - hi is exact in fp32; rounded to nearest even
// so that x = hi + lo up to the rounding of lo (relative 2^-21 of x).  The
// product A*B is then taken as Ahi*Bhi + Ahi*Blo + Alo*Bhi, dropping the
// Alo*Blo term (relative 2^-20): the "split-precision tensor-core correction"
// published by Ootomo and Yokota (2022) and used as "3xTF32" in NVIDIA's
// CUTLASS; the code here is written from that description.
//
// The tensor core reads an fp32 word given to a kind::tf32 MMA as its TF32
// truncation (measured on this part: 8192 probe values, ties and near-ties
// of both parities and signs, all read as trunc(x)).  So the high part needs
// no conversion: the hi plane holds the fp32 words as they are, and when A
// can be read in place no hi plane of A is written at all.
//
// A (M x K, K-contiguous) keeps its layout.  B (K x N, N-contiguous) is
// transposed on the way to N x K so that both tensor-core operands are
// K-major.  Output rows are padded to a multiple of 4 floats (16 bytes) for
// the TMA descriptors.  Both kernels are memory-bound copies (8 bytes of HBM
// traffic per element of A read in place, 12 otherwise); each thread keeps
// 64 bytes of loads in flight, and the transpose goes through a
// bank-conflict-free swizzled 64 x 64 tile with 16-byte accesses on both
// sides where the strides and bases allow.
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

// The low part of the split: tf32(x - trunc(x)).
__device__ __forceinline__ float lo_part(float x) {
    return to_tf32(x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u));
}
__device__ __forceinline__ float4 lo_part4(float4 x) {
    return make_float4(lo_part(x.x), lo_part(x.y), lo_part(x.z), lo_part(x.w));
}

constexpr int kThreads = 256;
// Vector elements (float4) each thread of the row kernel moves per pass: the
// loads are all issued before the first conversion, so that 64 bytes per
// thread are in flight (one float4 per thread left HBM a third idle).
constexpr int kRowUnroll = 4;
// Edge of the square transpose tile (elements).
constexpr int kT = 64;

// The kernels' bodies take their block coordinates and grid extent as
// arguments, so that the fused launch below can run A's and B's staging as
// two ranges of one grid.

__device__ __forceinline__ void split_rows_body(const float* __restrict__ src, long long lds,
                                                long long rows, long long cols,
                                                float* __restrict__ hi, float* __restrict__ lo,
                                                long long ldd, unsigned bx, unsigned by,
                                                unsigned gx, unsigned gy) {
    const long long step = static_cast<long long>(gx) * kThreads;
    for (long long r = by; r < rows; r += gy) {
        const float* s = src + r * lds;
        for (long long c = static_cast<long long>(bx) * kThreads + threadIdx.x; c < cols;
             c += kRowUnroll * step) {
            float x[kRowUnroll];
#pragma unroll
            for (int u = 0; u < kRowUnroll; ++u) x[u] = c + u * step < cols ? s[c + u * step] : 0.0f;
#pragma unroll
            for (int u = 0; u < kRowUnroll; ++u) {
                const long long cu = c + u * step;
                if (cu < cols) {
                    if (hi) hi[r * ldd + cu] = x[u];
                    lo[r * ldd + cu] = lo_part(x[u]);
                }
            }
        }
    }
}

// Vector form: 4 consecutive elements per thread and load (cols, lds, ldd
// multiples of 4 and all bases 16-byte aligned).  In both forms a null hi
// writes the lo plane only (A read in place as its own high part).
__device__ __forceinline__ void split_rows4_body(const float4* __restrict__ src, long long lds4,
                                                 long long rows, long long cols4,
                                                 float4* __restrict__ hi, float4* __restrict__ lo,
                                                 long long ldd4, unsigned bx, unsigned by,
                                                 unsigned gx, unsigned gy) {
    const long long step = static_cast<long long>(gx) * kThreads;
    for (long long r = by; r < rows; r += gy) {
        for (long long c = static_cast<long long>(bx) * kThreads + threadIdx.x; c < cols4;
             c += kRowUnroll * step) {
            float4 x[kRowUnroll];
#pragma unroll
            for (int u = 0; u < kRowUnroll; ++u)
                x[u] = c + u * step < cols4 ? src[r * lds4 + c + u * step]
                                            : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int u = 0; u < kRowUnroll; ++u) {
                const long long cu = c + u * step;
                if (cu < cols4) {
                    if (hi) hi[r * ldd4 + cu] = x[u];
                    lo[r * ldd4 + cu] = lo_part4(x[u]);
                }
            }
        }
    }
}

// Shared-tile index of element (k, n) of a kT x kT tile held k-major (row k
// = 64 consecutive n): the n index is XORed with 4 * ((k / 4) % 8).  The XOR
// leaves n's low two bits alone, so four consecutive n stay one aligned
// 16-byte word (the loads store whole float4); and the transposed reads (32
// lanes taking 8 groups of four k x 4 consecutive n) fall in 32 distinct
// banks, since n ^ 4 * q covers the 32 residues as q runs over 0..7.
__device__ __forceinline__ int tile_index(int k, int n) {
    return k * kT + (n ^ (((k >> 2) & 7) << 2));
}

// One kT x kT tile: src (K x N, row stride lds) rows k0.., columns n0.. to
// hi/lo (N x K, row stride ldt) rows n0.., columns k0...  vec_in: src and lds
// allow float4 loads; vec_out: hi, lo and ldt allow float4 stores and ldt >=
// K, so a store may run into columns K .. ldt - 1 (written as zeros there).
// Elements outside K x N are read as zeros and not written.
__device__ __forceinline__ void split_transpose_tile(const float* __restrict__ src, long long lds,
                                                     int K, int N, float* __restrict__ hi,
                                                     float* __restrict__ lo, long long ldt,
                                                     bool vec_in, bool vec_out, int k0, int n0,
                                                     float* __restrict__ tile) {
    constexpr int SLOTS = kT * kT / 4 / kThreads;  // float4 per thread and phase
    const int t = static_cast<int>(threadIdx.x);
    float4 v[SLOTS];
    // load: slot s is float4 (s % 16) of tile row s / 16 (one warp: two rows)
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) {
        const int s = t + kThreads * i;
        const int k = k0 + (s >> 4);
        const int n = n0 + 4 * (s & 15);
        const float* p = src + static_cast<long long>(k) * lds + n;
        if (vec_in && k < K && n + 3 < N) {
            v[i] = *reinterpret_cast<const float4*>(p);
        } else {
            const bool kin = k < K;
            v[i].x = kin && n < N ? p[0] : 0.0f;
            v[i].y = kin && n + 1 < N ? p[1] : 0.0f;
            v[i].z = kin && n + 2 < N ? p[2] : 0.0f;
            v[i].w = kin && n + 3 < N ? p[3] : 0.0f;
        }
    }
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) {
        const int s = t + kThreads * i;
        *reinterpret_cast<float4*>(tile + tile_index(s >> 4, 4 * (s & 15))) = v[i];
    }
    __syncthreads();
    // store: slot s is k = 32 (s / 512) + 4 (s % 8) .. + 3 of n = (s / 8) % 64;
    // eight lanes write one 128-byte run of an output row
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) {
        const int s = t + kThreads * i;
        const int kl = 32 * (s >> 9) + 4 * (s & 7);
        const int nl = (s >> 3) & (kT - 1);
        const int n = n0 + nl, k = k0 + kl;
        if (n < N && k < K) {
            const float h[4] = {tile[tile_index(kl, nl)], tile[tile_index(kl + 1, nl)],
                                tile[tile_index(kl + 2, nl)], tile[tile_index(kl + 3, nl)]};
            float l[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) l[e] = lo_part(h[e]);
            float* ph = hi + static_cast<long long>(n) * ldt + k;
            float* pl = lo + static_cast<long long>(n) * ldt + k;
            if (vec_out) {
                *reinterpret_cast<float4*>(ph) = make_float4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<float4*>(pl) = make_float4(l[0], l[1], l[2], l[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (k + e < K) {
                        ph[e] = h[e];
                        pl[e] = l[e];
                    }
                }
            }
        }
    }
    __syncthreads();  // the tile is free for the next one
}

// Tiles (bx, by), (bx, by + gy), ... of the transpose (bx: n tile, by: k tile).
__device__ __forceinline__ void split_transpose_body(const float* __restrict__ src, long long lds,
                                                     int K, int N, float* __restrict__ hi,
                                                     float* __restrict__ lo, long long ldt,
                                                     int vec, unsigned bx, unsigned by,
                                                     unsigned gy, float* __restrict__ tile) {
    const int ktiles = (K + kT - 1) / kT;
    const int n0 = static_cast<int>(bx) * kT;
    for (int kb = static_cast<int>(by); kb < ktiles; kb += static_cast<int>(gy))
        split_transpose_tile(src, lds, K, N, hi, lo, ldt, (vec & 1) != 0, (vec & 2) != 0,
                             kb * kT, n0, tile);
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
                       float* __restrict__ hi, float* __restrict__ lo, long long ldt, int vec) {
    pdl_trigger();  // the GEMM may launch; it waits for this grid to finish
    __shared__ __align__(16) float tile[kT * kT];
    split_transpose_body(src, lds, K, N, hi, lo, ldt, vec, blockIdx.x, blockIdx.y, gridDim.y,
                         tile);
}

// One launch for both operands of a call: blocks [0, gb_x * gb_y) split and
// transpose B, the rest split the rows of A (vector form when a_vec).  The
// transpose blocks, which take longer, are dispatched first.
__global__ void __launch_bounds__(kThreads)
split_operands_kernel(const float* __restrict__ a, long long lda, long long a_rows,
                      long long a_cols, float* __restrict__ a_hi, float* __restrict__ a_lo,
                      long long ldd, int a_vec, unsigned ga_x, unsigned ga_y,
                      const float* __restrict__ b, long long ldb, int K, int N,
                      float* __restrict__ b_hi, float* __restrict__ b_lo, long long ldt,
                      int b_vec, unsigned gb_x, unsigned gb_y) {
    pdl_trigger();  // the GEMM may launch; it waits for this grid to finish
    __shared__ __align__(16) float tile[kT * kT];
    const unsigned nb = gb_x * gb_y;
    if (blockIdx.x >= nb) {
        const unsigned ia = blockIdx.x - nb;
        const unsigned bx = ia % ga_x, by = ia / ga_x;
        if (a_vec)
            split_rows4_body(reinterpret_cast<const float4*>(a), lda / 4, a_rows, a_cols / 4,
                             reinterpret_cast<float4*>(a_hi), reinterpret_cast<float4*>(a_lo),
                             ldd / 4, bx, by, ga_x, ga_y);
        else
            split_rows_body(a, lda, a_rows, a_cols, a_hi, a_lo, ldd, bx, by, ga_x, ga_y);
    } else {
        const unsigned i = blockIdx.x;
        split_transpose_body(b, ldb, K, N, b_hi, b_lo, ldt, b_vec, i % gb_x, i / gb_x, gb_y, tile);
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
    const long long per_block = static_cast<long long>(kThreads) * kRowUnroll;
    long long gx = ((g.vec ? cols / 4 : cols) + per_block - 1) / per_block;
    if (gx > 64) gx = 64;
    g.gx = static_cast<unsigned>(gx);
    g.gy = static_cast<unsigned>(rows < 65535 ? rows : 65535);
    return g;
}

struct TransposeGrid {
    int vec;  // bit 0: float4 loads of src; bit 1: float4 stores of hi and lo
    unsigned gx, gy;
};
TransposeGrid transpose_grid(const float* src, long long lds, int K, int N, const float* hi,
                             const float* lo, long long ldt) {
    TransposeGrid g;
    const bool vin = lds % 4 == 0 && reinterpret_cast<uintptr_t>(src) % 16 == 0;
    const bool vout = ldt % 4 == 0 && ldt >= K &&
                      (reinterpret_cast<uintptr_t>(hi) | reinterpret_cast<uintptr_t>(lo)) % 16 == 0;
    g.vec = (vin ? 1 : 0) | (vout ? 2 : 0);
    const long long ktiles = (static_cast<long long>(K) + kT - 1) / kT;
    g.gx = static_cast<unsigned>((static_cast<long long>(N) + kT - 1) / kT);
    g.gy = static_cast<unsigned>(ktiles < 65535 ? ktiles : 65535);
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
    const TransposeGrid g = transpose_grid(src, lds, K, N, hi, lo, ldt);
    split_transpose_kernel<<<dim3(g.gx, g.gy), kThreads, 0, s>>>(src, lds, K, N, hi, lo, ldt,
                                                                 g.vec);
    return cudaGetLastError();
}

cudaError_t launch_split_operands(const float* a, long long lda, int M, int K, float* a_hi,
                                  float* a_lo, long long ldd, const float* b, long long ldb, int N,
                                  float* b_hi, float* b_lo, long long ldt, cudaStream_t s) {
    if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
    const RowsGrid ga = rows_grid(a, lda, M, K, a_hi, a_lo, ldd);
    const TransposeGrid gb = transpose_grid(b, ldb, K, N, b_hi, b_lo, ldt);
    const unsigned long long blocks =
        static_cast<unsigned long long>(ga.gx) * ga.gy + static_cast<unsigned long long>(gb.gx) * gb.gy;
    if (blocks > 0x7FFFFFFFull) {
        // too many blocks for one 1-D grid: two launches
        cudaError_t e = launch_split_rows(a, lda, M, K, a_hi, a_lo, ldd, s);
        if (e != cudaSuccess) return e;
        return launch_split_transpose(b, ldb, K, N, b_hi, b_lo, ldt, s);
    }
    split_operands_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
        a, lda, M, K, a_hi, a_lo, ldd, ga.vec ? 1 : 0, ga.gx, ga.gy, b, ldb, K, N, b_hi, b_lo,
        ldt, gb.vec, gb.gx, gb.gy);
    return cudaGetLastError();
}

}  // namespace gemm_f32_impl
