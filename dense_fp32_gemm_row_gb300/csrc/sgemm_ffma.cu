// sgemm_ffma.cu -- the CUDA-core single-precision GEMM kernel for sm_103a.
//
// Computes one 128 x 128 tile of C = A * B (row-major, arbitrary M/N/K) per
// CTA, or one split-K partial of it.  The general-M/N/K tiled kernel of
// "Lecture 12: final project" (section 2, tiledMatMulKernel: zero-filled
// out-of-range operand loads, guarded stores, C overwritten) and the
// register-tiled, double-buffered, asynchronous-copy kernels of the
// "cuda-gemm" README's optimisation table (steps 4-7) are the prior art; the
// design here is Blackwell's:
//
//  * Operand tiles are moved global -> shared by the tensor memory accelerator
//    (cp.async.bulk.tensor), one elected thread issuing two box loads per
//    stage.  Out-of-range rows/columns of a box are zero-filled by the
//    hardware, which is exactly the page's zero-fill boundary rule, so the
//    inner loop carries no bounds checks.
//  * A STAGES-deep ring of shared-memory stages, each with a "full"
//    mbarrier (transaction-count completion of the TMA bytes) and an "empty"
//    mbarrier (one arrival per consumer warp).  The refill of a stage is
//    issued as soon as every warp has released it, STAGES-1 stages ahead of
//    the consumer; no __syncthreads in the main loop.
//  * A (K-contiguous) lands 128-byte swizzled: row m's 16-byte chunk c sits at
//    chunk c ^ (m & 7).  Each thread reads 4 consecutive k of one A row with a
//    single 128-bit shared load; the four rows a warp touches at once have
//    distinct (m & 7), so the read is conflict-free without the lecture-5
//    "+1 padding" (which TMA cannot produce).
//  * B (N-contiguous) lands unswizzled; eight lanes read eight consecutive
//    float4 of one k row, a conflict-free 128-byte wavefront.
//  * 8 x 8 outputs per thread (rows tm + 4r, columns two float4 groups 32
//    apart): per 4-deep k step a thread does 256 FFMA for 16 shared loads.
//  * Every accumulator sums its products in ascending k, so the result is
//    run-to-run deterministic; split-K partials are summed in split order by
//    a separate kernel.
//  * The epilogue stores float4 when the row stride allows it and falls back
//    to predicated scalar stores on ragged edges; nothing outside C is
//    written.
#include <cstdint>

#include "device_sync.cuh"
#include "gemm_internal.h"

namespace gemm_f32_impl {
namespace {

using namespace gemm_f32_dev;

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 32;       // 32 floats = one 128-byte swizzle row of A
constexpr int STAGES = 3;
constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int CTAS_PER_SM = 2;
constexpr int A_BYTES = BM * BK * 4;
constexpr int B_BYTES = BK * BN * 4;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 2 * STAGES * 8 + 1024;  // + barriers + align slack
constexpr int GROUP_M = 8;   // tile rows per raster group (L2 reuse of B panels)

static_assert(BK == 32, "A-tile read addressing assumes the 128-byte swizzle of a 32-float row");
static_assert(THREADS == 256 && BM == 128 && BN == 128, "warp layout is 4 x 2 warps of 32 x 64");

__global__ void __launch_bounds__(THREADS, CTAS_PER_SM)
sgemm_ffma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  float* __restrict__ out, long long ldo, long long split_stride, int M, int N,
                  int K, int kb_per_split, int vec_store, unsigned* fault, long long timeout_ns) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t smem_base = smem_addr(smem);
    const uint32_t full0 = smem_base + STAGES * STAGE_BYTES;  // full[s]  at full0 + 8 s
    const uint32_t empty0 = full0 + 8 * STAGES;               // empty[s] at empty0 + 8 s

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int wm = warp >> 1;  // 32-row slab of the tile
    const int wn = warp & 1;   // 64-column slab of the tile
    const int tm = lane >> 3;  // 0..3
    const int tn = lane & 7;   // 0..7

    // grouped raster: GROUP_M tile rows walk the tile columns together
    const int tiles_m = (M + BM - 1) / BM;
    const int tiles_n = (N + BN - 1) / BN;
    const int per_group = GROUP_M * tiles_n;
    const int group = blockIdx.x / per_group;
    const int first_m = group * GROUP_M;
    const int rows_in_group = min(tiles_m - first_m, GROUP_M);
    const int within = blockIdx.x - group * per_group;
    const int m0 = (first_m + within % rows_in_group) * BM;
    const int n0 = (within / rows_in_group) * BN;

    const int kb_total = (K + BK - 1) / BK;
    const int kb_begin = blockIdx.y * kb_per_split;
    const int nkb = max(0, min(kb_total, kb_begin + kb_per_split) - kb_begin);

    if (tid == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, WARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();

    int issued = 0;  // k blocks whose loads thread 0 has issued
    if (tid == 0) {
        const int pre = min(STAGES, nkb);
        for (; issued < pre; ++issued) {
            const int s = issued % STAGES;
            const uint32_t dst = smem_base + s * STAGE_BYTES;
            const int k0 = (kb_begin + issued) * BK;
            mbar_arrive_expect_tx(full0 + 8 * s, STAGE_BYTES);
            tma_load_2d(dst, &tmA, full0 + 8 * s, k0, m0);
            tma_load_2d(dst + A_BYTES, &tmB, full0 + 8 * s, n0, k0);
        }
    }

    float acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[r][j] = 0.0f;

    const float* smemf = reinterpret_cast<const float*>(smem);
    const int a_off = (wm * 32 + tm) * BK;  // row wm*32+tm; row r of the thread is +4r
    const int b_off = wn * 64 + tn * 4;     // first column group; second is +32

    bool ok = true;
    int kb = 0;
    for (; kb < nkb; ++kb) {
        const int s = kb % STAGES;
        bool prod_ok = true;
        // refill the stage released in the previous iteration, STAGES-1 ahead
        if (tid == 0 && kb >= 1) {
            const int done = kb - 1;
            const int next = done + STAGES;
            if (next < nkb) {
                const int sd = done % STAGES;
                prod_ok = mbar_wait(empty0 + 8 * sd, (done / STAGES) & 1, timeout_ns, fault,
                                    kFaultEmptyBarrier);
                if (prod_ok) {
                    const uint32_t dst = smem_base + sd * STAGE_BYTES;
                    const int k0 = (kb_begin + next) * BK;
                    mbar_arrive_expect_tx(full0 + 8 * sd, STAGE_BYTES);
                    tma_load_2d(dst, &tmA, full0 + 8 * sd, k0, m0);
                    tma_load_2d(dst + A_BYTES, &tmB, full0 + 8 * sd, n0, k0);
                    issued = next + 1;
                }
            }
        }
        const bool full_ok =
            mbar_wait(full0 + 8 * s, (kb / STAGES) & 1, timeout_ns, fault, kFaultFullBarrier);
        if (!__all_sync(0xffffffffu, prod_ok && full_ok)) {
            ok = false;
            break;
        }

        const float* As = smemf + s * (STAGE_BYTES / 4);
        const float* Bs = As + A_BYTES / 4;
#pragma unroll
        for (int c = 0; c < BK / 4; ++c) {
            float4 b0[4], b1[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                b0[q] = *reinterpret_cast<const float4*>(Bs + (c * 4 + q) * BN + b_off);
                b1[q] = *reinterpret_cast<const float4*>(Bs + (c * 4 + q) * BN + b_off + 32);
            }
            // rows with even r have (m & 7) == tm, odd r have tm + 4
            const int xe = (c ^ tm) << 2;
            const int xo = (c ^ (tm + 4)) << 2;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float4 a = *reinterpret_cast<const float4*>(As + a_off + r * 4 * BK +
                                                                  ((r & 1) ? xo : xe));
                const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[r][0] = fmaf(av[q], b0[q].x, acc[r][0]);
                    acc[r][1] = fmaf(av[q], b0[q].y, acc[r][1]);
                    acc[r][2] = fmaf(av[q], b0[q].z, acc[r][2]);
                    acc[r][3] = fmaf(av[q], b0[q].w, acc[r][3]);
                    acc[r][4] = fmaf(av[q], b1[q].x, acc[r][4]);
                    acc[r][5] = fmaf(av[q], b1[q].y, acc[r][5]);
                    acc[r][6] = fmaf(av[q], b1[q].z, acc[r][6]);
                    acc[r][7] = fmaf(av[q], b1[q].w, acc[r][7]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }

    if (!ok) {
        // wind down: let every copy this CTA issued land before the CTA exits
        if (tid == 0) {
            for (int j = kb; j < issued; ++j)
                mbar_wait(full0 + 8 * (j % STAGES), (j / STAGES) & 1, timeout_ns / 4 + 1000, fault,
                          kFaultDrain);
        }
        return;
    }

    float* outp = out + static_cast<long long>(blockIdx.y) * split_stride;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int m = m0 + wm * 32 + tm + 4 * r;
        if (m >= M) continue;
        float* row = outp + static_cast<long long>(m) * ldo;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int n = n0 + b_off + 32 * g;
            const float* v = &acc[r][4 * g];
            if (vec_store && n + 3 < N) {
                *reinterpret_cast<float4*>(row + n) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (n + e < N) row[n + e] = v[e];
            }
        }
    }
}

}  // namespace

FfmaConfig ffma_config() { return {BM, BN, BK, STAGES, THREADS, CTAS_PER_SM, SMEM_BYTES}; }

cudaError_t launch_sgemm_ffma(const FfmaArgs& a, cudaStream_t s) {
    static thread_local int attr_done_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (attr_done_dev != dev) {
        e = cudaFuncSetAttribute(sgemm_ffma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done_dev = dev;
    }
    const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
    dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(a.splits));
    sgemm_ffma_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(a.tmA, a.tmB, a.out, a.ldo, a.split_stride,
                                                         a.M, a.N, a.K, a.kb_per_split,
                                                         a.vec_store, a.fault, a.timeout_ns);
    return cudaGetLastError();
}

}  // namespace gemm_f32_impl
