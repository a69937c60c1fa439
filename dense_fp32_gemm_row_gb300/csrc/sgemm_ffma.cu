// sgemm_ffma.cu -- the CUDA-core single-precision GEMM kernel for sm_103a.
//
// Computes one 128 x BN tile of C = A * B (row-major, arbitrary M/N/K) per
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
//    mbarrier (one arrival per consumer warp).  A stage released LAG
//    iterations ago is refilled STAGES - LAG blocks ahead of the consumer; no
//    __syncthreads in the main loop.
//  * A (K-contiguous) lands 128-byte swizzled: row m's 16-byte chunk c sits at
//    chunk c ^ (m & 7).  Each thread reads 4 consecutive k of one A row with a
//    single 128-bit shared load; the four rows a warp touches at once have
//    distinct (m & 7), so the read is conflict-free without the lecture-5
//    "+1 padding" (which TMA cannot produce).
//  * B (N-contiguous) lands unswizzled; eight lanes read eight consecutive
//    float4 of one k row, a conflict-free 128-byte wavefront.
//  * 8 x 4G outputs per thread (rows tm + 4r, columns G float4 groups 32
//    apart).  A 128-bit shared load moves 4 floats to each of 32 threads in
//    four 128-byte wavefronts, so a thread tile of TM x TN costs
//    (TM + TN) / (TM TN) wavefronts per FFMA instruction: 0.25 for 8 x 8,
//    which would need the whole 128-byte/clock shared-memory pipe at full
//    FFMA rate, and 0.1875 for 8 x 16 (G = 4), which leaves a quarter of it.
//  * Every accumulator sums its products in ascending k, so the result is
//    run-to-run deterministic.  Split-K partials are summed in split order,
//    either by a separate kernel over a workspace or, for 2..4 splits, inside
//    a thread-block cluster: the S CTAs computing one tile's K splits form a
//    cluster, each parks its partial tile in its own shared memory, and after
//    a cluster barrier CTA r adds up rows r/S .. (r+1)/S of the tile over
//    distributed shared memory, split 0 first (the workspace kernel's order,
//    so both give the same bits), and writes them to C.
//  * The epilogue stores float4 when the row stride allows it and falls back
//    to predicated scalar stores on ragged edges; nothing outside C is
//    written.
#include <cstdint>

#include "device_sync.cuh"
#include "epilogue.cuh"
#include "gemm_internal.h"

namespace gemm_f32_impl {
namespace {

using namespace gemm_f32_dev;

// Packed two-lane fp32 FMA of sm_100-family GPUs: d.x = a.x b.x + d.x and
// d.y = a.y b.y + d.y, each lane an IEEE fma like fmaf (same bits), one
// instruction for two multiply-adds.
__device__ __forceinline__ void ffma2(uint64_t& d, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
__device__ __forceinline__ uint64_t pack2(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& x, float& y) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ void lds_v2_b64(uint32_t addr, uint64_t& x, uint64_t& y) {
    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(x), "=l"(y) : "r"(addr));
}

__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t cluster_addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

constexpr int BM = 128;
constexpr int BK = 32;       // 32 floats = one 128-byte swizzle row of A
// splits added inside a cluster: at 512^3 (a latency-bound call) 2 and 4
// splits ran faster in a cluster than through the workspace (33.5 / 23.2
// against 35.5 / 24.6 us) but 8 ran slower (23.2 against 19.1 us)
constexpr int MAX_CLUSTER_SPLITS = 4;
constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int A_BYTES = BM * BK * 4;
constexpr int GROUP_M = 8;   // tile rows per raster group (L2 reuse of B panels)

// G: float4 column groups per thread (thread tile 8 x 4G, CTA tile 128 x 64G)
template <int G, int STAGES, int LAG, int MIN_BLOCKS>
struct FfmaVariant {
    static constexpr int BN = 64 * G;
    static constexpr int B_BYTES = BK * BN * 4;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 2 * STAGES * 8 + 1024;
    static_assert(LAG >= 1 && LAG < STAGES, "refill lag");
    static_assert(BN <= 256, "TMA box");
    static_assert(BM * BN * 4 <= STAGES * STAGE_BYTES, "a partial tile fits in the stages");
};

// Accumulators are held as column pairs and updated by packed two-lane FMAs,
// the A value duplicated into both lanes.
template <int G, int STAGES, int LAG, int MIN_BLOCKS>
__global__ void __launch_bounds__(THREADS, MIN_BLOCKS)
sgemm_ffma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  float* __restrict__ out, long long ldo, long long split_stride, int M, int N,
                  int K, int kb_per_split, int vec_store, unsigned* fault, long long timeout_ns,
                  float alpha, float beta, int scale_mode, int cluster_splits) {
    using V = FfmaVariant<G, STAGES, LAG, MIN_BLOCKS>;
    constexpr int BN = V::BN;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t smem_base = smem_addr(smem);
    const uint32_t full0 = smem_base + STAGES * V::STAGE_BYTES;  // full[s]  at full0 + 8 s
    const uint32_t empty0 = full0 + 8 * STAGES;                  // empty[s] at empty0 + 8 s

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int wm = warp >> 1;  // 32-row slab of the tile
    const int wn = warp & 1;   // (BN/2)-column slab of the tile
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
    // launched programmatically: operands (possibly padded by the kernel
    // before) are read only after this
    pdl_wait();
    pdl_trigger();

    int issued = 0;  // k blocks whose loads thread 0 has issued
    if (tid == 0) {
        const int pre = min(STAGES, nkb);
        for (; issued < pre; ++issued) {
            const int s = issued % STAGES;
            const uint32_t dst = smem_base + s * V::STAGE_BYTES;
            const int k0 = (kb_begin + issued) * BK;
            mbar_arrive_expect_tx(full0 + 8 * s, V::STAGE_BYTES);
            tma_load_2d(dst, &tmA, full0 + 8 * s, k0, m0);
            tma_load_2d(dst + A_BYTES, &tmB, full0 + 8 * s, n0, k0);
        }
    }

    uint64_t acc2[8][2 * G];  // column pairs (2p, 2p+1) of each of the 8 rows
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int j = 0; j < 2 * G; ++j) acc2[r][j] = 0ull;

    const float* smemf = reinterpret_cast<const float*>(smem);
    const int a_off = (wm * 32 + tm) * BK;      // row wm*32+tm; row r of the thread is +4r
    const int b_off = wn * (BN / 2) + tn * 4;   // first column group; group g is +32 g

    bool ok = true;
    int kb = 0;
    for (; kb < nkb; ++kb) {
        const int s = kb % STAGES;
        bool prod_ok = true;
        // refill the stage released LAG iterations ago, STAGES - LAG blocks ahead
        if (tid == 0 && kb >= LAG) {
            const int done = kb - LAG;
            const int next = done + STAGES;
            if (next < nkb) {
                const int sd = done % STAGES;
                prod_ok = mbar_wait(empty0 + 8 * sd, (done / STAGES) & 1, timeout_ns, fault,
                                    kFaultEmptyBarrier);
                if (prod_ok) {
                    const uint32_t dst = smem_base + sd * V::STAGE_BYTES;
                    const int k0 = (kb_begin + next) * BK;
                    mbar_arrive_expect_tx(full0 + 8 * sd, V::STAGE_BYTES);
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

        const float* As = smemf + s * (V::STAGE_BYTES / 4);
        const float* Bs = As + A_BYTES / 4;
#pragma unroll
        for (int c = 0; c < BK / 4; ++c) {
            // rows with even r have (m & 7) == tm, odd r have tm + 4
            const int xe = (c ^ tm) << 2;
            const int xo = (c ^ (tm + 4)) << 2;
            float4 a[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
                a[r] = *reinterpret_cast<const float4*>(As + a_off + r * 4 * BK +
                                                        ((r & 1) ? xo : xe));
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint64_t bp[2 * G];
#pragma unroll
                for (int g = 0; g < G; ++g)
                    lds_v2_b64(smem_addr(Bs + (c * 4 + q) * BN + b_off + 32 * g), bp[2 * g],
                               bp[2 * g + 1]);
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const float av = q == 0 ? a[r].x : q == 1 ? a[r].y : q == 2 ? a[r].z : a[r].w;
                    const uint64_t ad = pack2(av, av);
#pragma unroll
                    for (int p = 0; p < 2 * G; ++p) ffma2(acc2[r][p], ad, bp[p]);
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
        // a cluster member still takes both cluster barriers below, so that
        // its partners are not left waiting (the result is void: the fault
        // word reports the timeout)
        if (cluster_splits < 2) return;
    }

    float acc[8][4 * G];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int p = 0; p < 2 * G; ++p) unpack2(acc2[r][p], acc[r][2 * p], acc[r][2 * p + 1]);

    if (cluster_splits >= 2) {
        // ---- split-K reduction inside the cluster (blockIdx.y = split = rank) ----
        __syncthreads();  // every warp is done with the stages
        // this CTA's partial tile, BM x BN row-major, over the first stages
        if (ok) {
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int g = 0; g < G; ++g)
                    sts128(smem_base + 4u * static_cast<uint32_t>((wm * 32 + tm + 4 * r) * BN +
                                                                  b_off + 32 * g),
                           make_float4(acc[r][4 * g], acc[r][4 * g + 1], acc[r][4 * g + 2],
                                       acc[r][4 * g + 3]));
        }
        cluster_sync();  // all partials written and visible across the cluster
        const int S = cluster_splits;
        const int rank = blockIdx.y;
        const int rows = (BM + S - 1) / S;
        const int r0 = rank * rows;
        const int r1 = min(BM, r0 + rows);
        constexpr int Q = BN / 4;  // float4 per tile row
        uint32_t peer[MAX_CLUSTER_SPLITS];
#pragma unroll
        for (int q = 0; q < MAX_CLUSTER_SPLITS; ++q)
            peer[q] = q < S ? map_to_cta(smem_base, static_cast<uint32_t>(q)) : 0u;
        if (ok) {
            for (int idx = tid; idx < (r1 - r0) * Q; idx += THREADS) {
                const int i = r0 + idx / Q;
                const int j4 = idx - (idx / Q) * Q;
                const int m = m0 + i;
                if (m >= M) continue;
                const uint32_t off = 4u * static_cast<uint32_t>(i * BN + 4 * j4);
                float4 sum = ld_dsmem_v4(peer[0] + off);
#pragma unroll
                for (int q = 1; q < MAX_CLUSTER_SPLITS; ++q) {
                    if (q < S) {
                        const float4 v = ld_dsmem_v4(peer[q] + off);
                        sum.x += v.x;
                        sum.y += v.y;
                        sum.z += v.z;
                        sum.w += v.w;
                    }
                }
                store4(out + static_cast<long long>(m) * ldo, n0 + 4 * j4, N, sum, vec_store != 0,
                       alpha, beta, scale_mode);
            }
        }
        cluster_sync();  // no CTA leaves while a partner may still read its partial
        return;
    }

    float* outp = out + static_cast<long long>(blockIdx.y) * split_stride;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int m = m0 + wm * 32 + tm + 4 * r;
        if (m >= M) continue;
        float* row = outp + static_cast<long long>(m) * ldo;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float* v = &acc[r][4 * g];
            store4(row, n0 + b_off + 32 * g, N, make_float4(v[0], v[1], v[2], v[3]),
                   vec_store != 0, alpha, beta, scale_mode);
        }
    }
}

// the two variants the planner chooses between
using Narrow = FfmaVariant<2, 3, 1, 2>;  // 128 x 128 tiles, 2 CTAs / SM
using Wide = FfmaVariant<4, 4, 2, 1>;    // 128 x 256 tiles, 1 CTA / SM

template <int G, int STAGES, int LAG, int MIN_BLOCKS>
cudaError_t launch_variant(const FfmaArgs& a, cudaStream_t s) {
    using V = FfmaVariant<G, STAGES, LAG, MIN_BLOCKS>;
    auto kern = sgemm_ffma_kernel<G, STAGES, LAG, MIN_BLOCKS>;
    // the kernel's stage layout and transaction count assume this box width
    if (a.bn != V::BN) return cudaErrorInvalidValue;
    static thread_local int attr_done_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (attr_done_dev != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, V::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done_dev = dev;
    }
    const int tiles = ((a.M + BM - 1) / BM) * ((a.N + V::BN - 1) / V::BN);
    dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(a.splits));
    if (a.cluster_splits) {
        // the splits of one tile form a cluster along y
        if (a.cluster_splits != a.splits || a.splits < 2 || a.splits > MAX_CLUSTER_SPLITS)
            return cudaErrorInvalidValue;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = static_cast<unsigned>(a.splits);
        attr[0].val.clusterDim.z = 1;
        attr[1] = pdl_attribute();
        cfg.gridDim = grid;
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = V::SMEM_BYTES;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, kern, a.tmA, a.tmB, a.out, a.ldo, a.split_stride, a.M, a.N,
                               a.K, a.kb_per_split, a.vec_store, a.fault, a.timeout_ns, a.alpha,
                               a.beta, a.scale_mode, a.cluster_splits);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = V::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a.tmA, a.tmB, a.out, a.ldo, a.split_stride, a.M, a.N, a.K,
                           a.kb_per_split, a.vec_store, a.fault, a.timeout_ns, a.alpha, a.beta,
                           a.scale_mode, 0);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

FfmaConfig ffma_config(int variant) {
    if (variant == 1)
        return {BM, Wide::BN, BK, 4, THREADS, 1, Wide::SMEM_BYTES, 1};
    return {BM, Narrow::BN, BK, 3, THREADS, 2, Narrow::SMEM_BYTES, 0};
}

namespace {
template <int G, int STAGES, int LAG, int MIN_BLOCKS>
cudaError_t occupancy(int* ctas_per_sm) {
    using V = FfmaVariant<G, STAGES, LAG, MIN_BLOCKS>;
    auto kern = sgemm_ffma_kernel<G, STAGES, LAG, MIN_BLOCKS>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, V::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, kern, THREADS,
                                                         V::SMEM_BYTES);
}
}  // namespace

cudaError_t ffma_ctas_per_sm(int variant, int* ctas_per_sm) {
    return variant == 1 ? occupancy<4, 4, 2, 1>(ctas_per_sm) : occupancy<2, 3, 1, 2>(ctas_per_sm);
}

cudaError_t launch_sgemm_ffma(const FfmaArgs& a, cudaStream_t s) {
    if (a.variant == 1) return launch_variant<4, 4, 2, 1>(a, s);
    return launch_variant<2, 3, 1, 2>(a, s);
}

}  // namespace gemm_f32_impl
