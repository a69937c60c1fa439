// sgemm_3xtf32_tmem.cu -- the 3xTF32 GEMM with B's split held in tensor
// memory, for operands read as stored (no staging pass).
//
// The tensor core reads a kind::tf32 operand from shared memory only K-major
// (with the B-major bit of the instruction descriptor set, kind::tf32 MMAs
// wrote zeros on this part; the same descriptors with bf16 operands were
// exact).  A row-major K x N matrix B is N-contiguous, so the kernels that
// split in shared memory transpose B there, and that transpose, with the
// hi and lo planes it writes, is what bounds them.  An MMA can instead take
// its A operand from tensor memory, one operand row per lane; and a thread
// that writes tensor memory writes its own lane.  So here each CTA computes
// the transposed tile:
//
//     D[n][m] (+)= sum_k B[k][n] * A[m][k]      (tensor memory: lane n, column m)
//
// with B^T as the MMA's A operand in tensor memory and A as its B operand in
// shared memory (K-major as stored).  Thread n of the B splitter warpgroup
// reads column n of the stage's B box (32 k values, one 128-byte row per k:
// conflict-free), splits each value into hi = trunc(x) (x with its low 13
// mantissa bits cleared: the TF32 value the tensor core reads from the word)
// and lo = tf32(x - hi), rounded to nearest even, and stores both as 32
// columns of its lane: the transpose costs nothing.  Per K step of 8 the MMA
// lane issues  Bhi*Alo + Blo*Ahi + Bhi*Ahi  (the products of the other
// 3xTF32 kernels, small terms first, Blo*Alo dropped), with the chunked
// promotion of those kernels.  The epilogue thread of lane n holds column n
// of the tile's C for 128 rows m, so each warp store writes 32 consecutive
// columns of one row of C: 128 contiguous bytes.  A measured microbenchmark
// put MMAs with A in tensor memory ahead of shared-memory operands (M128 N256:
// 1130 against 912 TFLOP/s tf32; M128 N128: 841 against 729).
//
// One 128 x 128 tile per work unit; a persistent grid of one CTA per SM;
// 384 threads:
//   warp 0       one lane issues the TMA loads of a stage: a 128 x 32 box of
//                A ({K, M}, 128-byte swizzle) and four 32 x 32 boxes of B
//                ({N, K}, N-contiguous), into a 4-deep ring of 48 KB stages
//                (A, A lo, B), with an L2 prefetch two K blocks ahead;
//   warp 1       allocates all 512 tensor-memory columns (two 128-column
//                accumulators, then four 64-column B operand stages: hi in
//                the first 32, lo in the next 32) and one lane issues the
//                MMAs (M = 128 lanes of n, N = 128 of m, K = 8) and commits;
//   warps 2-3    split A in shared memory, half of every stage fill each:
//                x stays as its own high part, lo = tf32(x - trunc(x)) goes
//                16 KB further on;
//   warps 4-7    split B into tensor memory (warp 4 + q owns lanes 32q ..
//                32q + 31, the lane quarter its index gives it); all six
//                splitter warps arrive on one barrier per stage, the MMA
//                lane's one wait per fill;
//   warps 8-11   the epilogue: per chunk, load the accumulator lanes of the
//                warp's quarter (128 columns), hand the buffer back and add
//                them into 128 registers in chunk order; at the end of a
//                unit store them to C (or to the split-K partials).
// With 2..8 K splits and one unit per CTA the splits of a tile can run as
// one thread-block cluster (cluster_splits): each CTA parks its partial in
// its drained stage memory, and after a cluster barrier every CTA sums a
// band of the tile's rows over the S partials through distributed shared
// memory, in split order, and writes C; no workspace, no reduction launch.
// Every wait is bounded; a timeout sets the device fault word and a shared
// abort flag that ends the other roles' waits, and the CTA winds down (its
// in-flight copies and MMAs waited for, bounded) before freeing its tensor
// memory.  The kernel is launched as a programmatic dependent.
#include <cstdint>

#include "device_sync.cuh"
#include "epilogue.cuh"
#include "gemm_internal.h"
#include "tcgen05.cuh"
#include "tf32x3_common.cuh"

namespace gemm_f32_impl {
namespace {

using namespace gemm_f32_dev;

struct TmemCfg {
    static constexpr int BN = 128;                 // tile columns n: tensor-memory lanes
    static constexpr int STAGES = 4;
    static constexpr int A_BYTES = BM * BK * 4;    // A as stored: its own high part
    static constexpr int B_BYTES = BN * BK * 4;    // B as stored: four 32 x 32 boxes
    static constexpr int B_BOX_BYTES = 32 * BK * 4;
    static constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;  // A, A lo, B
    static constexpr int NSPLIT_A = 2;             // A splitter warps, half of every fill each
    // full barriers: one per (fill mod STAGES * NSPLIT_A)
    static constexpr int NFULL = STAGES * NSPLIT_A;
    static constexpr int THREADS = 384;
    static constexpr int TMEM_COLS = 512;
    static constexpr int D_COLS = BM;              // accumulator columns: m
    static constexpr int OP_COL0 = 2 * D_COLS;     // B operand stage s at OP_COL0 + 64 s
    static constexpr int OP_COLS = 2 * BK;         // hi (32 columns), lo (32 columns)
    // full (NFULL), empty, A converted, B converted (per stage),
    // acc_full x2, acc_empty x2, drain
    static constexpr int NBARS = NFULL + 2 * STAGES + 5;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + NBARS * 8 + 16 + 1024;
    // MMA M = the tile's 128 columns n (lanes), N = its 128 rows m
    static constexpr uint32_t IDESC = idesc_tf32_f32(BN, BM);
    static_assert(OP_COL0 + STAGES * OP_COLS <= TMEM_COLS, "tensor-memory columns");
    static_assert(A_BYTES == 16384, "split_a_stage's map: a 16 KB A slot, lo 16 KB further on");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

__device__ __forceinline__ float lds32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void sts32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// 16 bytes of another CTA's shared memory (a shared::cluster address)
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t cluster_addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

// split-K partials of the single-CTA form added inside a (portable) cluster
constexpr int kMaxTmemClusterSplits = 8;

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Hardware barrier `id` for the `count` threads (whole warps) that execute
// it; id 0 with the whole CTA is __syncthreads.
__device__ __forceinline__ void bar_sync_named(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Sum the S partials of float4 groups [tid, ngroups) step nthreads of a
// band (group i: row row0 + i / (TN_ / 4), columns n0 + 4 (i % (TN_ / 4))
// .. + 3) in split order, and write them to C.  G groups a pass, CHUNK
// partials of each loaded before any is added.
template <int G, int CHUNK, int TN_>
__device__ __forceinline__ void reduce_band(const float* __restrict__ parts, long long ldw,
                                            long long split_stride, int row0, int n0,
                                            int ngroups, int S, int tid, int nthreads,
                                            float* __restrict__ C, long long ldc, int M, int N,
                                            float alpha, float beta, int mode) {
    constexpr int TN4 = TN_ / 4;
    const long long stride4 = split_stride / 4;
    for (int base = tid; base < ngroups; base += G * nthreads) {
        const float4* src[G];
        float4 sum[G];
        bool live[G];
        int m[G], n[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int idx = base + g * nthreads;
            m[g] = row0 + idx / TN4;
            n[g] = n0 + 4 * (idx % TN4);
            live[g] = idx < ngroups && m[g] < M && n[g] < N;
            src[g] = reinterpret_cast<const float4*>(
                parts + (live[g] ? static_cast<long long>(m[g]) * ldw + n[g] : 0));
            if (live[g]) sum[g] = __ldcg(src[g]);
        }
        for (int s0 = 1; s0 < S; s0 += CHUNK) {
            float4 v[G][CHUNK];
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int j = 0; j < CHUNK; ++j)
                    if (live[g] && s0 + j < S)
                        v[g][j] = __ldcg(src[g] + static_cast<long long>(s0 + j) * stride4);
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int j = 0; j < CHUNK; ++j)
                    if (live[g] && s0 + j < S) {
                        sum[g].x += v[g][j].x;
                        sum[g].y += v[g][j].y;
                        sum[g].z += v[g][j].z;
                        sum[g].w += v[g][j].w;
                    }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (!live[g]) continue;
            float* dst = C + static_cast<long long>(m[g]) * ldc + n[g];
            const float r[4] = {sum[g].x, sum[g].y, sum[g].z, sum[g].w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (n[g] + i < N) dst[i] = scale1(r[i], dst + i, alpha, beta, mode);
        }
    }
}

// The split-K partials of a tile added inside the kernel.  Every CTA holds
// exactly one unit (one K split of one tile) and all CTAs are co-resident,
// the launch being cooperative.  The tile's `parts` contributors (S CTAs,
// or 2 S for the CTA pair, which writes its partial in two halves) each
// announce their partial on the tile's arrival counter, wait (bounded) until
// all have arrived, then each sums a band of ceil(TM_ / parts) tile rows
// over the S partials in split order (the order of the separate reduction
// kernel) and writes C; the last contributor to finish resets both counters
// for the next call.  `nthreads` threads (tid 0 .. nthreads - 1) call this
// together; `bar_id` is their named barrier (0 for the whole CTA).  LOADS:
// partials of one output group a thread keeps in flight (20 on the
// 128 x 128 form's registers; 25 on the epilogue warpgroups' 200, the most
// that stays unspilled: 76 partials in three round trips instead of four).
template <int TM_, int TN_, int LOADS = 20>
__device__ __forceinline__ void reduce_tile_in_kernel(
    const float* __restrict__ parts, long long ldw, long long split_stride, int* counters,
    int tiles, int t, int m0, int n0, int S, int nparts, int part, int tid, int nthreads,
    int bar_id, float* __restrict__ C, long long ldc, int M, int N, float alpha, float beta,
    int mode, unsigned* fault, long long timeout_ns, uint32_t abort_flag) {
    __shared__ int go;
    if (tid == 0) {
        // the threads that stored the partial fenced their stores before the
        // barrier that precedes this call
        atomicAdd(counters + t, 1);
        int ok = 1;
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(counters + t) < nparts) {
            if (globaltimer_ns() - t0 > static_cast<uint64_t>(timeout_ns)) {
                if (fault) atomicOr(fault, kFaultAccumBarrier);
                ok = 0;
                break;
            }
        }
        go = ok && ld_shared_volatile(abort_flag) == 0u;
    }
    bar_sync_named(bar_id, nthreads);
    if (go) {
        const int rows = (TM_ + nparts - 1) / nparts;
        const int r0 = part * rows;
        const int r1 = min(TM_, r0 + rows);
        // four adjacent outputs (a float4 group: the workspace rows are
        // padded to a multiple of 4 floats, its bases 256-byte aligned) at a
        // time; a thread's chain of L2 round trips bounds the band, so its
        // loads go out in batches: with one group a thread, LOADS partials
        // of it at once; with several (few splits, wide bands), 5 partials
        // of each of 4 groups
        const int ngroups = (r1 - r0) * (TN_ / 4);
        if (ngroups <= nthreads)
            reduce_band<1, LOADS, TN_>(parts, ldw, split_stride, m0 + r0, n0, ngroups, S, tid,
                                    nthreads, C, ldc, M, N, alpha, beta, mode);
        else
            reduce_band<4, 5, TN_>(parts, ldw, split_stride, m0 + r0, n0, ngroups, S, tid,
                                   nthreads, C, ldc, M, N, alpha, beta, mode);
    }
    bar_sync_named(bar_id, nthreads);
    if (tid == 0 && atomicAdd(counters + tiles + t, 1) == nparts - 1) {
        // every contributor of the tile has passed its wait: reset for the
        // next call
        counters[t] = 0;
        counters[tiles + t] = 0;
    }
}

__global__ void __launch_bounds__(TmemCfg::THREADS, 1)
sgemm_3xtf32_tmem_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, float* __restrict__ out,
                         long long ldo, long long split_stride, int M, int N, int K,
                         int kb_per_split, int splits, unsigned* fault, long long timeout_ns,
                         float alpha, float beta, int scale_mode, int* counters,
                         float* __restrict__ c_final, long long ldc, int c_mode,
                         int cluster_splits, int vec_store) {
    using C = TmemCfg;
    constexpr int STAGES = C::STAGES;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t full0 = sbase + STAGES * C::STAGE_BYTES;  // full[f]: + 8 f
    const uint32_t empty0 = full0 + 8 * C::NFULL;            // empty[s]: + 8 s
    const uint32_t aconv0 = empty0 + 8 * STAGES;             // A lo written, B in TMEM[s]
    const uint32_t accf0 = aconv0 + 8 * STAGES;              // acc_full[b]
    const uint32_t acce0 = accf0 + 16;                       // acc_empty[b]
    const uint32_t drain = acce0 + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + STAGES * C::STAGE_BYTES + C::NBARS * 8);
    const uint32_t abort_flag = smem_addr(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles_m = (M + BM - 1) / BM;
    const int tiles_n = (N + C::BN - 1) / C::BN;
    const int units = tiles_m * tiles_n * splits;
    const int kb_total = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        for (int f = 0; f < C::NFULL; ++f) mbar_init(full0 + 8 * f, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(empty0 + 8 * s, 1);
            // every arrival the MMA lane needs for a fill: A's two splitter
            // warps and B's four
            mbar_init(aconv0 + 8 * s, C::NSPLIT_A + 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, 4);
        }
        mbar_init(drain, 1);
        st_shared_volatile(abort_flag, 0u);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // launched programmatically: the set-up above overlapped the kernel
    // before this one; its outputs are read only after this
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------ TMA producer ------------------------------
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, C::BN, BM,
                                      cluster_splits);
                for (int kb = 0; kb < w.nkb; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (it >= STAGES &&
                        !role_wait(empty0 + 8 * s, ((it / STAGES) & 1) ^ 1, timeout_ns, fault,
                                   kFaultEmptyBarrier, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sbase + s * C::STAGE_BYTES;
                    const int k0 = (w.kb_begin + kb) * BK;
                    const uint32_t fb = full0 + 8 * (it % C::NFULL);
                    mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_BYTES);
                    tma_load_2d(st, &tmA, fb, k0, w.m0);
#pragma unroll
                    for (int j = 0; j < C::BN / 32; ++j)
                        tma_load_2d(st + 2 * C::A_BYTES + j * C::B_BOX_BYTES, &tmB, fb,
                                    w.n0 + 32 * j, k0);
                    if (kb + kPrefetchAhead < w.nkb) {
                        const int kp = k0 + kPrefetchAhead * BK;
                        tma_prefetch_2d(&tmA, kp, w.m0);
#pragma unroll
                        for (int j = 0; j < C::BN / 32; ++j)
                            tma_prefetch_2d(&tmB, w.n0 + 32 * j, kp);
                    }
                }
            }
            // wind down: every issued copy has landed and every stage has been
            // released by the MMA commits before the CTA may exit
            const long long tail = ok ? timeout_ns : timeout_ns / 8 + 1000;
            for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j) {
                mbar_wait(full0 + 8 * (j % C::NFULL), (j / C::NFULL) & 1, tail, fault,
                          kFaultDrain);
                mbar_wait(empty0 + 8 * (j % STAGES), (j / STAGES) & 1, tail, fault, kFaultDrain);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------ MMA issuer --------------------------------
            int it = 0;  // K blocks consumed (ring position)
            int g = 0;   // chunks issued (accumulator buffer g & 1)
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, C::BN, BM,
                                      cluster_splits);
                for (int c0 = 0; c0 < w.nkb && ok; c0 += CH, ++g) {
                    const int buf = g & 1;
                    if (g >= 2 && !role_wait(acce0 + 8 * buf, ((g >> 1) & 1) ^ 1, timeout_ns, fault,
                                             kFaultAccumBarrier, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + static_cast<uint32_t>(buf * C::D_COLS);
                    const int c1 = min(w.nkb, c0 + CH);
                    for (int kb = c0; kb < c1; ++kb, ++it) {
                        const int s = it % STAGES;
                        const uint32_t par = (it / STAGES) & 1;
                        // A's and B's splitters, on one barrier
                        if (!role_wait(aconv0 + 8 * s, par, timeout_ns, fault, kFaultFullBarrier,
                                       abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t st = sbase + s * C::STAGE_BYTES;
                        const uint64_t a_hi = smem_desc_sw128_kmajor(st);
                        const uint64_t a_lo = smem_desc_sw128_kmajor(st + C::A_BYTES);
                        const uint32_t b_hi =
                            tmem_base + static_cast<uint32_t>(C::OP_COL0 + C::OP_COLS * s);
                        const uint32_t b_lo = b_hi + BK;
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            // shared-memory start address + k * 32 bytes (encoded >> 4);
                            // tensor-memory operand columns + k * 8
                            const uint64_t off = static_cast<uint64_t>(k * UMMA_K * 4) >> 4;
                            const uint32_t kc = static_cast<uint32_t>(k * UMMA_K);
                            const uint32_t acc = (kb > c0 || k > 0) ? 1u : 0u;
                            mma_tf32_tmem_a(d, b_hi + kc, a_lo + off, C::IDESC, acc);
                            mma_tf32_tmem_a(d, b_lo + kc, a_hi + off, C::IDESC, 1u);
                            mma_tf32_tmem_a(d, b_hi + kc, a_hi + off, C::IDESC, 1u);
                        }
                        mma_commit(empty0 + 8 * s);
                    }
                    if (!ok) break;
                    mma_commit(accf0 + 8 * buf);
                }
            }
            // all issued MMAs complete before tensor memory is released
            mma_commit(drain);
            mbar_wait(drain, 0, ok ? timeout_ns : timeout_ns / 8 + 1000, fault, kFaultDrain);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------ A splitters (warps 2-3) -------------------
        // each warp half of every stage fill (whole fills taken in turn left
        // a fill's split as long as one warp's ~0.8 us)
        int it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, C::BN, BM,
                                  cluster_splits);
            for (int kb = 0; kb < w.nkb; ++kb, ++it) {
                const int s = it % STAGES;
                const bool got = role_wait(full0 + 8 * (it % C::NFULL), (it / C::NFULL) & 1,
                                           timeout_ns, fault, kFaultFullBarrier, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const uint32_t st = sbase + s * C::STAGE_BYTES;
                split_a_stage(st, lane + 32 * (warp - 2));  // this warp's half
                // the tensor core reads these words through the async proxy
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(aconv0 + 8 * s);
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------ B splitters (warps 4-7) -------------------
        // Lane quarter q = warp - 4: tile columns n = 32 q + lane, i.e. box q
        // of the stage's B.  Column n of k-row r of a box sits in 16-byte
        // chunk (n / 4) ^ (r % 8) of that 128-byte row (the TMA's swizzle),
        // word n % 4: for each r the warp reads one whole row.
        const int q = warp & 3;
        const uint32_t chunk = static_cast<uint32_t>(lane >> 2);
        const uint32_t word = static_cast<uint32_t>(lane & 3) * 4u;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
        int it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, C::BN, BM,
                                  cluster_splits);
            for (int kb = 0; kb < w.nkb; ++kb, ++it) {
                const int s = it % STAGES;
                const bool got = role_wait(full0 + 8 * (it % C::NFULL), (it / C::NFULL) & 1,
                                           timeout_ns, fault, kFaultFullBarrier, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                // the MMAs that last read operand stage s completed before its
                // smem stage was refilled (the producer waited on empty[s]),
                // so its tensor-memory columns are free
                const uint32_t box =
                    sbase + s * C::STAGE_BYTES + 2 * C::A_BYTES + q * C::B_BOX_BYTES;
                const uint32_t col = lane_base + static_cast<uint32_t>(C::OP_COL0 + C::OP_COLS * s);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint32_t r = static_cast<uint32_t>(16 * h + i);
                        const float x = lds32(box + r * 128u + ((chunk ^ (r & 7u)) << 4) + word);
                        hi[i] = __float_as_uint(x) & 0xFFFFE000u;
                        lo[i] = __float_as_uint(to_tf32(x - __uint_as_float(hi[i])));
                    }
                    tmem_st_32x32b_x16(col + 16u * h, hi);
                    tmem_st_32x32b_x16(col + BK + 16u * h, lo);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(aconv0 + 8 * s);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------ epilogue (warps 8-11) ---------------------
        const int q = warp & 3;              // tensor-memory lanes 32q .. 32q + 31
        const int nl = 32 * q + lane;        // this thread's tile column
        float acc[EPI_COLS];
        static_assert(EPI_COLS == BM, "one thread holds its column of the whole tile");
        int g = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, C::BN, BM,
                                  cluster_splits);
            for (int c0 = 0; c0 < w.nkb; c0 += CH, ++g) {
                const int buf = g & 1;
                const bool got = role_wait(accf0 + 8 * buf, (g >> 1) & 1, timeout_ns, fault,
                                           kFaultAccumBarrier, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                       static_cast<uint32_t>(buf * C::D_COLS);
#pragma unroll
                for (int j = 0; j < EPI_COLS / 16; ++j) {
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(tbase + 16 * j, r);
                    tmem_ld_wait(r);
                    if (c0 == 0) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[16 * j + i] = __uint_as_float(r[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[16 * j + i] += __uint_as_float(r[i]);
                    }
                }
                // the chunk is in registers: give the buffer back to the MMA lane
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce0 + 8 * buf);
            }
            if (!ok) break;
            if (cluster_splits) {
                // this CTA's only unit: its raw partial goes into the stage
                // memory, row-major 128 x 128 (every MMA of the unit, and so
                // every read of a stage, has completed); a warp writes 32
                // consecutive words of a row
                const uint32_t pcol = sbase + 4u * static_cast<uint32_t>(nl);
#pragma unroll
                for (int j = 0; j < EPI_COLS; ++j)
                    sts32(pcol + 4u * static_cast<uint32_t>(C::BN * j), acc[j]);
                continue;
            }
            const int n = w.n0 + nl;
            if (n < N) {
                float* p = out + static_cast<long long>(w.split) * split_stride +
                           static_cast<long long>(w.m0) * ldo + n;
                const int rows = M - w.m0;
#pragma unroll
                for (int j = 0; j < EPI_COLS; ++j, p += ldo)
                    if (j < rows) *p = scale1(acc[j], p, alpha, beta, scale_mode);
            }
        }
        // the partial must be visible to the other CTAs of the tile before
        // this CTA announces it
        if (counters) __threadfence();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    if (cluster_splits) {
        // ---- split-K inside the cluster: CTA rank q of the cluster holds
        // split q of one tile.  Each CTA sums a 1/S band of the tile's rows
        // over the S partials through distributed shared memory, in split
        // order, and writes C (alpha and beta applied there).  Every thread
        // takes both cluster barriers, whatever its role did. ----
        cluster_sync();  // every partial parked and visible across the cluster
        const int S = cluster_splits;
        const Unit w = decode(static_cast<int>(blockIdx.x), tiles_m, tiles_n, kb_per_split,
                              kb_total, C::BN, BM, S);
        const int rows = (BM + S - 1) / S;
        const int r0 = static_cast<int>(cluster_ctarank()) * rows;
        const int r1 = min(BM, r0 + rows);
        constexpr int Q = C::BN / 4;  // 16-byte words per tile row
        // G float4 groups a thread, each partial's G loads issued together
        constexpr int G = 6;
        const int ngroups = (r1 - r0) * Q;
        if (ld_shared_volatile(abort_flag) == 0u) {
            for (int base = threadIdx.x; base < ngroups; base += G * C::THREADS) {
                uint32_t off[G];
                bool live[G];
                float4 sum[G];
                const uint32_t p0 = map_to_cta(sbase, 0u);
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    const int idx = base + j * C::THREADS;
                    const int i = r0 + idx / Q;
                    const int c4 = idx - (idx / Q) * Q;
                    live[j] = idx < ngroups && w.m0 + i < M && w.n0 + 4 * c4 < N;
                    off[j] = 16u * static_cast<uint32_t>(i * Q + c4);
                    if (live[j]) sum[j] = ld_dsmem_v4(p0 + off[j]);
                }
                for (int q = 1; q < S; ++q) {
                    const uint32_t pq = map_to_cta(sbase, static_cast<uint32_t>(q));
                    float4 v[G];
#pragma unroll
                    for (int j = 0; j < G; ++j)
                        if (live[j]) v[j] = ld_dsmem_v4(pq + off[j]);
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        if (live[j]) {
                            sum[j].x += v[j].x;
                            sum[j].y += v[j].y;
                            sum[j].z += v[j].z;
                            sum[j].w += v[j].w;
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    if (!live[j]) continue;
                    const int idx = base + j * C::THREADS;
                    const int i = r0 + idx / Q;
                    const int c4 = idx - (idx / Q) * Q;
                    store4(out + static_cast<long long>(w.m0 + i) * ldo, w.n0 + 4 * c4, N, sum[j],
                           vec_store != 0, alpha, beta, scale_mode);
                }
            }
        }
        cluster_sync();  // no CTA leaves while a partner may still read its partial
    }
    if (counters) {
        const int tiles = tiles_m * tiles_n;
        const int u = blockIdx.x;  // this CTA's only unit
        const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, C::BN, BM);
        reduce_tile_in_kernel<BM, C::BN>(out, ldo, split_stride, counters, tiles,
                                         u - w.split * tiles, w.m0, w.n0, splits, splits,
                                         w.split, threadIdx.x, blockDim.x, 0, c_final, ldc, M, N,
                                         alpha, beta, c_mode, fault, timeout_ns, abort_flag);
    }
}

// ============================================================================
// The CTA-pair form: a cluster of two CTAs computes a 256 x 256 tile with
// tcgen05.mma.cta_group::2 (M = 256 tile columns n across the pair, N = 256
// tile rows m, K = 8), B^T in tensor memory, A in shared memory.  CTA rank r
// holds tile columns n0 + 128 r .. in its tensor-memory lanes and tile rows
// m0 + 128 r .. of A in its shared memory; each MMA reads half of its
// shared-memory operand from each SM.  N = 256 MMAs run at the tensor
// core's full rate (a microbenchmark: 1215 TFLOP/s tf32 with A in tensor
// memory, against 841 for the N = 128 MMAs of the single-CTA form), but the
// 256-column accumulator then fits only once beside four 64-column operand
// stages: it is single-buffered, and the MMA lane waits at the start of each
// chunk until both epilogues have drained the previous one (measured: 5 %
// of the MMA rate at 128-deep chunks).
//
// 512 threads per CTA, four warpgroups, registers rebalanced at start
// (launched at 128 per thread): warpgroups 0-1 down to 56, the two epilogue
// warpgroups up to 200 (2 x 128 x 56 + 2 x 128 x 200 = 65536), so that an
// epilogue thread can hold 64 loaded values beside its 128 sums:
//   warp 0      one lane: TMA loads of the stage (A {32 k, 128 m}, four B
//               boxes {32 n, 32 k}) onto this CTA's own full barrier;
//   warp 1      tensor-memory allocation for the pair; in the leader, one
//               lane issues the MMAs and multicasts the commits;
//   warps 2-3   split A in shared memory (half of every fill each);
//   warps 4-7   split B into this CTA's tensor memory (warp 4 + q: lanes
//               32 q ..); in the leader all six arrive on its stage-ready
//               barrier, which the MMA lane waits on; in the peer they
//               arrive on its own A- and B-converted barriers and one lane
//               of warp 1 relays both to the leader's stage-ready barrier
//               (one cluster-scope arrival per stage fill; the MMA lane's
//               three waits a fill on separate barriers cost ~1 %);
//   warps 8-15  the epilogue: warp 8 + e drains lanes 32 (e % 4) .., columns
//               128 (e / 4) .. of the accumulator and arrives on the
//               leader's acc-empty barrier.
// ============================================================================
struct TmemPairCfg {
    static constexpr int TN = 256;                 // tile columns n (lanes across the pair)
    static constexpr int TM = 256;                 // tile rows m (MMA N)
    static constexpr int HALF = 128;               // per CTA
    static constexpr int STAGES = 4;
    static constexpr int A_BYTES = HALF * BK * 4;
    static constexpr int B_BYTES = HALF * BK * 4;
    static constexpr int B_BOX_BYTES = 32 * BK * 4;
    static constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;  // A, A lo, B
    // A splitter warps, each splitting half of every fill: a fill's split
    // then takes half as long (alternating whole fills between the two
    // warps, ~0.84 us each, left the four-stage ring short of ready stages
    // at the MMA rate)
    static constexpr int NSPLIT_A = 2;
    static constexpr int NFULL = STAGES * NSPLIT_A;
    static constexpr int THREADS = 512;
    static constexpr int TMEM_COLS = 512;
    static constexpr int D_COLS = TM;              // one accumulator: m
    static constexpr int OP_COL0 = D_COLS;         // operand stage s at OP_COL0 + 64 s
    static constexpr int OP_COLS = 2 * BK;
    static constexpr int EPI_WARPS = 8;
    // full (NFULL), empty, A converted, B converted, peer ready (per
    // stage), acc_full, acc_empty, drain
    static constexpr int NBARS = NFULL + 4 * STAGES + 3;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + NBARS * 8 + 16 + 1024;
    static constexpr uint32_t IDESC = idesc_tf32_f32(TN, TM);
    static constexpr int REGS_LOW = 56, REGS_HIGH = 200;
    static constexpr int DRAIN_BATCH = 4;  // 16-column loads in flight per wait
    // K blocks per promotion chunk: the single accumulator stalls the MMAs
    // for each drain, so the chunks are twice as deep as the other kernels'
    static constexpr int CHUNK = 2 * CH;
    static_assert(2 * 128 * REGS_LOW + 2 * 128 * REGS_HIGH == 65536, "register shares");
    static_assert(OP_COL0 + STAGES * OP_COLS <= TMEM_COLS, "tensor-memory columns");
    static_assert(A_BYTES == 16384, "split_a_stage's map");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

__global__ void __launch_bounds__(TmemPairCfg::THREADS, 1)
sgemm_3xtf32_tmem_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                              const __grid_constant__ CUtensorMap tmB, float* __restrict__ out,
                              long long ldo, long long split_stride, int M, int N, int K,
                              int kb_per_split, int splits, unsigned* fault,
                              long long timeout_ns, float alpha, float beta, int scale_mode,
                              int tail_tiles, int tail_splits, float* __restrict__ tail_ws,
                              int* counters, float* __restrict__ c_final, long long ldc,
                              int c_mode) {
    using C = TmemPairCfg;
    constexpr int STAGES = C::STAGES;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t full0 = sbase + STAGES * C::STAGE_BYTES;  // own: + 8 f
    const uint32_t empty0 = full0 + 8 * C::NFULL;            // own, multicast commit: + 8 s
    const uint32_t aconv0 = empty0 + 8 * STAGES;             // own: the A splitter warp
    const uint32_t bconv0 = aconv0 + 8 * STAGES;             // own: 4 B splitter warps
    const uint32_t peer0 = bconv0 + 8 * STAGES;              // leader: the peer's relay
    const uint32_t accf = peer0 + 8 * STAGES;                // own, multicast commit
    const uint32_t acce = accf + 8;                          // leader: 8 warps x 2 CTAs
    const uint32_t drain = acce + 8;
    uint32_t* tmem_slot =
        reinterpret_cast<uint32_t*>(smem + STAGES * C::STAGE_BYTES + C::NBARS * 8);
    const uint32_t abort_flag = smem_addr(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x >> 1;
    const int nclusters = gridDim.x >> 1;
    const int tiles_m = (M + C::TM - 1) / C::TM;
    const int tiles_n = (N + C::TN - 1) / C::TN;
    const int units = tail_tiles ? tiles_m * tiles_n - tail_tiles + tail_tiles * tail_splits
                                 : tiles_m * tiles_n * splits;
    const int kb_total = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        for (int f = 0; f < C::NFULL; ++f) mbar_init(full0 + 8 * f, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(empty0 + 8 * s, 1);
            // the leader's A-converted barrier takes every arrival the MMA
            // lane needs: its A and B splitters and the peer's relay
            mbar_init(aconv0 + 8 * s, rank == 0 ? C::NSPLIT_A + 4 + 1 : C::NSPLIT_A);
            mbar_init(bconv0 + 8 * s, 4);
            mbar_init(peer0 + 8 * s, 1);
        }
        mbar_init(accf, 1);
        mbar_init(acce, 2 * C::EPI_WARPS);
        mbar_init(drain, 1);
        st_shared_volatile(abort_flag, 0u);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(tmem_slot), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();
    pdl_trigger();

    if (warp < 8) {
        // warpgroups 0-1 give registers to the epilogue warpgroups
        regs_dec<C::REGS_LOW>();
    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------ TMA producer (both CTAs) ------------------
            int it = 0;
            bool ok = true;
            for (int u = cluster; u < units && ok; u += nclusters) {
                const Unit w = decode_pair(u, tiles_m, tiles_n, kb_per_split, kb_total, C::TN, tail_tiles, tail_splits);
                const int ma = w.m0 + static_cast<int>(rank) * C::HALF;
                const int nb = w.n0 + static_cast<int>(rank) * C::HALF;
                for (int kb = 0; kb < w.nkb; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (it >= STAGES &&
                        !role_wait(empty0 + 8 * s, ((it / STAGES) & 1) ^ 1, timeout_ns, fault,
                                   kFaultEmptyBarrier, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sbase + s * C::STAGE_BYTES;
                    const int k0 = (w.kb_begin + kb) * BK;
                    const uint32_t fb = full0 + 8 * (it % C::NFULL);
                    mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_BYTES);
                    tma_load_2d(st, &tmA, fb, k0, ma);
#pragma unroll
                    for (int j = 0; j < C::HALF / 32; ++j)
                        tma_load_2d(st + 2 * C::A_BYTES + j * C::B_BOX_BYTES, &tmB, fb,
                                    nb + 32 * j, k0);
                    if (kb + kPrefetchAhead < w.nkb) {
                        const int kp = k0 + kPrefetchAhead * BK;
                        tma_prefetch_2d(&tmA, kp, ma);
#pragma unroll
                        for (int j = 0; j < C::HALF / 32; ++j)
                            tma_prefetch_2d(&tmB, nb + 32 * j, kp);
                    }
                }
            }
            // wind down: this CTA's copies have landed and its stages have been
            // released by the MMAs
            const long long tail = ok ? timeout_ns : timeout_ns / 8 + 1000;
            for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j) {
                mbar_wait(full0 + 8 * (j % C::NFULL), (j / C::NFULL) & 1, tail, fault,
                          kFaultDrain);
                mbar_wait(empty0 + 8 * (j % STAGES), (j / STAGES) & 1, tail, fault, kFaultDrain);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------ MMA issuer (leader) -----------------------
            int it = 0;
            int g = 0;  // chunks issued
            bool ok = true;
            for (int u = cluster; u < units && ok; u += nclusters) {
                const Unit w = decode_pair(u, tiles_m, tiles_n, kb_per_split, kb_total, C::TN, tail_tiles, tail_splits);
                for (int c0 = 0; c0 < w.nkb && ok; c0 += C::CHUNK, ++g) {
                    // the single accumulator: both epilogues have drained chunk g - 1
                    if (g >= 1 && !role_wait(acce, (g - 1) & 1, timeout_ns, fault,
                                             kFaultAccumBarrier, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int c1 = min(w.nkb, c0 + C::CHUNK);
                    for (int kb = c0; kb < c1; ++kb, ++it) {
                        const int s = it % STAGES;
                        const uint32_t par = (it / STAGES) & 1;
                        // this CTA's splitters (CTA scope) and the peer's,
                        // relayed by one lane there (cluster scope), all on
                        // one barrier
                        if (!role_wait(aconv0 + 8 * s, par, timeout_ns, fault, kFaultFullBarrier,
                                       abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t st = sbase + s * C::STAGE_BYTES;
                        const uint64_t a_hi = smem_desc_sw128_kmajor(st);
                        const uint64_t a_lo = smem_desc_sw128_kmajor(st + C::A_BYTES);
                        const uint32_t b_hi =
                            tmem_base + static_cast<uint32_t>(C::OP_COL0 + C::OP_COLS * s);
                        const uint32_t b_lo = b_hi + BK;
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            const uint64_t off = static_cast<uint64_t>(k * UMMA_K * 4) >> 4;
                            const uint32_t kc = static_cast<uint32_t>(k * UMMA_K);
                            const uint32_t acc = (kb > c0 || k > 0) ? 1u : 0u;
                            mma_tf32_pair_tmem_a(tmem_base, b_hi + kc, a_lo + off, C::IDESC, acc);
                            mma_tf32_pair_tmem_a(tmem_base, b_lo + kc, a_hi + off, C::IDESC, 1u);
                            mma_tf32_pair_tmem_a(tmem_base, b_hi + kc, a_hi + off, C::IDESC, 1u);
                        }
                        mma_commit_pair_multicast(empty0 + 8 * s, 0x3);
                    }
                    if (!ok) break;
                    mma_commit_pair_multicast(accf, 0x3);
                }
            }
            mma_commit_pair(drain);
            mbar_wait(drain, 0, ok ? timeout_ns : timeout_ns / 8 + 1000, fault, kFaultDrain);
        } else if (lane == 0) {
            // ------------------------------ relay (peer CTA) --------------------------
            // One cluster-scope arrival per stage fill on the leader, once this
            // CTA's splitters have arrived on its own barriers (a release at
            // cluster scope by every splitter warp stalled them on memory
            // barriers: 1.25 us a fill against 0.79 us of MMA work, 4096^3).
            const uint32_t peer_leader = map_to_cta(aconv0, 0);
            int it = 0;
            bool ok = true;
            for (int u = cluster; u < units && ok; u += nclusters) {
                const Unit w = decode_pair(u, tiles_m, tiles_n, kb_per_split, kb_total, C::TN, tail_tiles, tail_splits);
                for (int kb = 0; kb < w.nkb; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t par = (it / STAGES) & 1;
                    if (!role_wait(aconv0 + 8 * s, par, timeout_ns, fault, kFaultFullBarrier,
                                   abort_flag) ||
                        !role_wait(bconv0 + 8 * s, par, timeout_ns, fault, kFaultFullBarrier,
                                   abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_cluster(peer_leader + 8 * s);
                }
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------ A splitters (warps 2-3, both CTAs) --------
        int it = 0;
        bool ok = true;
        for (int u = cluster; u < units && ok; u += nclusters) {
            const Unit w = decode_pair(u, tiles_m, tiles_n, kb_per_split, kb_total, C::TN, tail_tiles, tail_splits);
            for (int kb = 0; kb < w.nkb; ++kb, ++it) {
                const int s = it % STAGES;
                const bool got = role_wait(full0 + 8 * (it % C::NFULL), (it / C::NFULL) & 1,
                                           timeout_ns, fault, kFaultFullBarrier, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const uint32_t st = sbase + s * C::STAGE_BYTES;
                split_a_stage(st, lane + 32 * (warp - 2));  // this warp's half
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(aconv0 + 8 * s);
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------ B splitters (warps 4-7, both CTAs) --------
        const int q = warp & 3;
        const uint32_t chunk = static_cast<uint32_t>(lane >> 2);
        const uint32_t word = static_cast<uint32_t>(lane & 3) * 4u;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
        int it = 0;
        bool ok = true;
        for (int u = cluster; u < units && ok; u += nclusters) {
            const Unit w = decode_pair(u, tiles_m, tiles_n, kb_per_split, kb_total, C::TN, tail_tiles, tail_splits);
            for (int kb = 0; kb < w.nkb; ++kb, ++it) {
                const int s = it % STAGES;
                const bool got = role_wait(full0 + 8 * (it % C::NFULL), (it / C::NFULL) & 1,
                                           timeout_ns, fault, kFaultFullBarrier, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const uint32_t box =
                    sbase + s * C::STAGE_BYTES + 2 * C::A_BYTES + q * C::B_BOX_BYTES;
                const uint32_t col =
                    lane_base + static_cast<uint32_t>(C::OP_COL0 + C::OP_COLS * s);
                // eight k at a time: this warpgroup runs on 56 registers
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t r = static_cast<uint32_t>(8 * h + i);
                        const float x = lds32(box + r * 128u + ((chunk ^ (r & 7u)) << 4) + word);
                        hi[i] = __float_as_uint(x) & 0xFFFFE000u;
                        lo[i] = __float_as_uint(to_tf32(x - __uint_as_float(hi[i])));
                    }
                    tmem_st_32x32b_x8(col + 8u * h, hi);
                    tmem_st_32x32b_x8(col + BK + 8u * h, lo);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive((rank == 0 ? aconv0 : bconv0) + 8 * s);
            }
        }
        __syncwarp();
    }
    } else {
        // ------------------------------ epilogue (warps 8-15, both CTAs) ----------
        regs_inc<C::REGS_HIGH>();
        const int e = warp - 8;
        const int q = warp & 3;                 // lanes 32 q .. 32 q + 31
        const int col0 = (e >> 2) * EPI_COLS;   // accumulator columns (tile rows m)
        const int nl = static_cast<int>(rank) * C::HALF + 32 * q + lane;  // tile column
        const uint32_t acce_leader = map_to_cta(acce, 0);
        float acc[EPI_COLS];
        int g = 0;
        bool ok = true;
        for (int u = cluster; u < units && ok; u += nclusters) {
            const Unit w = decode_pair(u, tiles_m, tiles_n, kb_per_split, kb_total, C::TN, tail_tiles, tail_splits);
            for (int c0 = 0; c0 < w.nkb; c0 += C::CHUNK, ++g) {
                const bool got = role_wait(accf, g & 1, timeout_ns, fault, kFaultAccumBarrier,
                                           abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                       static_cast<uint32_t>(col0);
                // the MMA lane waits for this drain (one accumulator): keep
                // DRAIN_BATCH loads in flight per wait (one at a time, the
                // eight round trips took ~1.07 us a chunk)
#pragma unroll
                for (int j0 = 0; j0 < EPI_COLS / 16; j0 += C::DRAIN_BATCH) {
                    uint32_t r[C::DRAIN_BATCH][16];
#pragma unroll
                    for (int b = 0; b < C::DRAIN_BATCH; ++b)
                        tmem_ld_32x32b_x16(tbase + 16 * (j0 + b), r[b]);
#pragma unroll
                    for (int b = 0; b < C::DRAIN_BATCH; ++b) tmem_ld_wait(r[b]);
#pragma unroll
                    for (int b = 0; b < C::DRAIN_BATCH; ++b) {
                        const int j = j0 + b;
                        if (c0 == 0) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[16 * j + i] = __uint_as_float(r[b][i]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[16 * j + i] += __uint_as_float(r[b][i]);
                        }
                    }
                }
                // the loads have completed: the arrival hands the accumulator
                // back and orders no writes, so CTA-scope release suffices
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(acce_leader);
            }
            if (!ok) break;
            if (w.slot >= 0) {
                // a K share of a tail tile: the raw 256 x 256 sum, tile-local
                float* p = tail_ws + static_cast<long long>(w.slot) * (C::TM * C::TN) +
                           static_cast<long long>(col0) * C::TN + nl;
#pragma unroll
                for (int j = 0; j < EPI_COLS; ++j) p[static_cast<long long>(j) * C::TN] = acc[j];
                continue;
            }
            const int n = w.n0 + nl;
            if (n < N) {
                float* p = out + static_cast<long long>(w.split) * split_stride +
                           static_cast<long long>(w.m0 + col0) * ldo + n;
                const int rows = M - (w.m0 + col0);
#pragma unroll
                for (int j = 0; j < EPI_COLS; ++j, p += ldo)
                    if (j < rows) *p = scale1(acc[j], p, alpha, beta, scale_mode);
            }
        }
        if (counters) {
            // the in-kernel reduction, here on the epilogue's register share:
            // the partial must be visible to the other CTAs of the tile
            // before this CTA announces it; then each CTA of each split sums
            // its band of the tile's rows
            __threadfence();
            bar_sync_named(1, 32 * C::EPI_WARPS);
            const int tiles = tiles_m * tiles_n;
            const Unit w =
                decode_pair(cluster, tiles_m, tiles_n, kb_per_split, kb_total, C::TN, 0, 0);
            reduce_tile_in_kernel<C::TM, C::TN, 25>(
                out, ldo, split_stride, counters, tiles, cluster - w.split * tiles, w.m0, w.n0,
                splits, 2 * splits, 2 * w.split + static_cast<int>(rank), 32 * e + lane,
                32 * C::EPI_WARPS, 1, c_final, ldc, M, N, alpha, beta, c_mode, fault, timeout_ns,
                abort_flag);
        }
        __syncwarp();
    }

    // neither CTA may leave while its partner can still reach its shared or
    // tensor memory
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}


// ============================================================================
// The wide single-CTA form: one CTA computes a 256 x 128 tile (256 rows m of
// C by 128 columns n) with tcgen05.mma.cta_group::1 M128 N256 K8 (M = the
// tile's columns n in tensor-memory lanes, N = its rows m), B^T in tensor
// memory, A in shared memory.  N = 256 MMAs run at ~1130 TFLOP/s tf32 with A
// in tensor memory (a microbenchmark) against 841 for the N = 128 MMAs of
// the 128 x 128 form, without the CTA pair's cluster; the price is shared
// memory: a 32-deep stage would hold 256 rows of A and of A lo (64 KB) beside
// B, so the stages are 16 deep (A as {16 k, 256 m} boxes with 64-byte
// swizzle, 40 KB a stage, five stages), and, as in the pair form, the
// 256-column accumulator is single-buffered with 256-deep promotion chunks.
//
// 512 threads in four warpgroups, registers rebalanced as in the pair form
// (56 for warpgroups 0-1, 200 for the epilogue warpgroups):
//   warp 0      one lane: TMA loads of the stage (A {16 k, 256 m}, four B
//               boxes {32 n, 16 k});
//   warp 1      tensor-memory allocation; one lane issues the MMAs;
//   warps 2-3   split A in shared memory, half of every fill each;
//   warps 4-7   split B into tensor memory (warp 4 + q: lanes 32 q ..);
//               all six splitter warps arrive on one barrier per stage;
//   warps 8-15  the epilogue: warp 8 + e drains lanes 32 (e % 4) .., columns
//               128 (e / 4) .. of the accumulator.
// ============================================================================
struct TmemWideCfg {
    static constexpr int TN = 128;                   // tile columns n (lanes)
    static constexpr int TM = 256;                   // tile rows m (MMA N)
    static constexpr int KB = 16;                    // K per stage
    static constexpr int STAGES = 5;
    static constexpr int A_BYTES = TM * KB * 4;
    static constexpr int B_BYTES = TN * KB * 4;
    static constexpr int B_BOX_BYTES = 32 * KB * 4;
    static constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;  // A, A lo, B
    static constexpr int NSPLIT_A = 2;
    static constexpr int NFULL = STAGES * NSPLIT_A;
    static constexpr int THREADS = 512;
    static constexpr int TMEM_COLS = 512;
    static constexpr int D_COLS = TM;                // one accumulator: m
    static constexpr int OP_COL0 = D_COLS;           // operand stage s at OP_COL0 + 32 s
    static constexpr int OP_COLS = 2 * KB;           // hi, then lo
    static constexpr int EPI_WARPS = 8;
    // full (NFULL), empty, stage ready (per stage), acc_full, acc_empty, drain
    static constexpr int NBARS = NFULL + 2 * STAGES + 3;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + NBARS * 8 + 16 + 1024;
    static constexpr uint32_t IDESC = idesc_tf32_f32(TN, TM);
    static constexpr int REGS_LOW = 56, REGS_HIGH = 200;
    static constexpr int DRAIN_BATCH = 4;
    static constexpr int CHUNK = 256 / KB;           // K blocks a promotion chunk (256 deep)
    static_assert(2 * 128 * REGS_LOW + 2 * 128 * REGS_HIGH == 65536, "register shares");
    static_assert(OP_COL0 + STAGES * OP_COLS <= TMEM_COLS, "tensor-memory columns");
    static_assert(A_BYTES == 16384, "split_a_stage's map");
    static_assert(STAGE_BYTES % 1024 == 0, "stage bases 1024-byte aligned");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

__global__ void __launch_bounds__(TmemWideCfg::THREADS, 1)
sgemm_3xtf32_tmem_wide_kernel(const __grid_constant__ CUtensorMap tmA,
                              const __grid_constant__ CUtensorMap tmB, float* __restrict__ out,
                              long long ldo, long long split_stride, int M, int N, int K,
                              int kb_per_split, int splits, unsigned* fault,
                              long long timeout_ns, float alpha, float beta, int scale_mode,
                              int* counters, float* __restrict__ c_final, long long ldc,
                              int c_mode) {
    using C = TmemWideCfg;
    constexpr int STAGES = C::STAGES;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t full0 = sbase + STAGES * C::STAGE_BYTES;  // + 8 f
    const uint32_t empty0 = full0 + 8 * C::NFULL;            // + 8 s
    const uint32_t ready0 = empty0 + 8 * STAGES;             // + 8 s: A and B split
    const uint32_t accf = ready0 + 8 * STAGES;
    const uint32_t acce = accf + 8;
    const uint32_t drain = acce + 8;
    uint32_t* tmem_slot =
        reinterpret_cast<uint32_t*>(smem + STAGES * C::STAGE_BYTES + C::NBARS * 8);
    const uint32_t abort_flag = smem_addr(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles_m = (M + C::TM - 1) / C::TM;
    const int tiles_n = (N + C::TN - 1) / C::TN;
    const int units = tiles_m * tiles_n * splits;
    const int kb_total = (K + C::KB - 1) / C::KB;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        for (int f = 0; f < C::NFULL; ++f) mbar_init(full0 + 8 * f, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(empty0 + 8 * s, 1);
            mbar_init(ready0 + 8 * s, C::NSPLIT_A + 4);
        }
        mbar_init(accf, 1);
        mbar_init(acce, C::EPI_WARPS);
        mbar_init(drain, 1);
        st_shared_volatile(abort_flag, 0u);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();
    pdl_trigger();

    if (warp < 8) {
        // warpgroups 0-1 give registers to the epilogue warpgroups
        regs_dec<C::REGS_LOW>();
    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------ TMA producer ------------------------------
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, C::TN, C::TM);
                for (int kb = 0; kb < w.nkb; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (it >= STAGES &&
                        !role_wait(empty0 + 8 * s, ((it / STAGES) & 1) ^ 1, timeout_ns, fault,
                                   kFaultEmptyBarrier, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sbase + s * C::STAGE_BYTES;
                    const int k0 = (w.kb_begin + kb) * C::KB;
                    const uint32_t fb = full0 + 8 * (it % C::NFULL);
                    mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_BYTES);
                    tma_load_2d(st, &tmA, fb, k0, w.m0);
#pragma unroll
                    for (int j = 0; j < C::TN / 32; ++j)
                        tma_load_2d(st + 2 * C::A_BYTES + j * C::B_BOX_BYTES, &tmB, fb,
                                    w.n0 + 32 * j, k0);
                    // the same distance ahead in K as the 32-deep kernels
                    if (kb + 2 * kPrefetchAhead < w.nkb) {
                        const int kp = k0 + 2 * kPrefetchAhead * C::KB;
                        tma_prefetch_2d(&tmA, kp, w.m0);
#pragma unroll
                        for (int j = 0; j < C::TN / 32; ++j)
                            tma_prefetch_2d(&tmB, w.n0 + 32 * j, kp);
                    }
                }
            }
            // wind down: every issued copy has landed and every stage has been
            // released by the MMA commits before the CTA may exit
            const long long tail = ok ? timeout_ns : timeout_ns / 8 + 1000;
            for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j) {
                mbar_wait(full0 + 8 * (j % C::NFULL), (j / C::NFULL) & 1, tail, fault,
                          kFaultDrain);
                mbar_wait(empty0 + 8 * (j % STAGES), (j / STAGES) & 1, tail, fault, kFaultDrain);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------ MMA issuer --------------------------------
            int it = 0;
            int g = 0;  // chunks issued
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, C::TN, C::TM);
                for (int c0 = 0; c0 < w.nkb && ok; c0 += C::CHUNK, ++g) {
                    // the single accumulator: the epilogue has drained chunk g - 1
                    if (g >= 1 && !role_wait(acce, (g - 1) & 1, timeout_ns, fault,
                                             kFaultAccumBarrier, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int c1 = min(w.nkb, c0 + C::CHUNK);
                    for (int kb = c0; kb < c1; ++kb, ++it) {
                        const int s = it % STAGES;
                        const uint32_t par = (it / STAGES) & 1;
                        if (!role_wait(ready0 + 8 * s, par, timeout_ns, fault, kFaultFullBarrier,
                                       abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t st = sbase + s * C::STAGE_BYTES;
                        const uint64_t a_hi = smem_desc_sw64_kmajor(st);
                        const uint64_t a_lo = smem_desc_sw64_kmajor(st + C::A_BYTES);
                        const uint32_t b_hi =
                            tmem_base + static_cast<uint32_t>(C::OP_COL0 + C::OP_COLS * s);
                        const uint32_t b_lo = b_hi + C::KB;
#pragma unroll
                        for (int k = 0; k < C::KB / UMMA_K; ++k) {
                            // start address + k * 32 bytes (encoded >> 4)
                            const uint64_t off = static_cast<uint64_t>(k * UMMA_K * 4) >> 4;
                            const uint32_t kc = static_cast<uint32_t>(k * UMMA_K);
                            const uint32_t acc = (kb > c0 || k > 0) ? 1u : 0u;
                            mma_tf32_tmem_a(tmem_base, b_hi + kc, a_lo + off, C::IDESC, acc);
                            mma_tf32_tmem_a(tmem_base, b_lo + kc, a_hi + off, C::IDESC, 1u);
                            mma_tf32_tmem_a(tmem_base, b_hi + kc, a_hi + off, C::IDESC, 1u);
                        }
                        mma_commit(empty0 + 8 * s);
                    }
                    if (!ok) break;
                    mma_commit(accf);
                }
            }
            // all issued MMAs complete before tensor memory is released
            mma_commit(drain);
            mbar_wait(drain, 0, ok ? timeout_ns : timeout_ns / 8 + 1000, fault, kFaultDrain);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------ A splitters (warps 2-3) -------------------
        int it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, C::TN, C::TM);
            for (int kb = 0; kb < w.nkb; ++kb, ++it) {
                const int s = it % STAGES;
                const bool got = role_wait(full0 + 8 * (it % C::NFULL), (it / C::NFULL) & 1,
                                           timeout_ns, fault, kFaultFullBarrier, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                split_a_stage(sbase + s * C::STAGE_BYTES, lane + 32 * (warp - 2));
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(ready0 + 8 * s);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------ B splitters (warps 4-7) -------------------
        const int q = warp & 3;
        const uint32_t chunk = static_cast<uint32_t>(lane >> 2);
        const uint32_t word = static_cast<uint32_t>(lane & 3) * 4u;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
        int it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, C::TN, C::TM);
            for (int kb = 0; kb < w.nkb; ++kb, ++it) {
                const int s = it % STAGES;
                const bool got = role_wait(full0 + 8 * (it % C::NFULL), (it / C::NFULL) & 1,
                                           timeout_ns, fault, kFaultFullBarrier, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const uint32_t box =
                    sbase + s * C::STAGE_BYTES + 2 * C::A_BYTES + q * C::B_BOX_BYTES;
                const uint32_t col =
                    lane_base + static_cast<uint32_t>(C::OP_COL0 + C::OP_COLS * s);
                // eight k at a time: this warpgroup runs on 56 registers
#pragma unroll
                for (int h = 0; h < C::KB / 8; ++h) {
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t r = static_cast<uint32_t>(8 * h + i);
                        const float x = lds32(box + r * 128u + ((chunk ^ (r & 7u)) << 4) + word);
                        hi[i] = __float_as_uint(x) & 0xFFFFE000u;
                        lo[i] = __float_as_uint(to_tf32(x - __uint_as_float(hi[i])));
                    }
                    tmem_st_32x32b_x8(col + 8u * h, hi);
                    tmem_st_32x32b_x8(col + C::KB + 8u * h, lo);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ready0 + 8 * s);
            }
        }
        __syncwarp();
    }
    } else {
        // ------------------------------ epilogue (warps 8-15) ---------------------
        regs_inc<C::REGS_HIGH>();
        const int e = warp - 8;
        const int q = warp & 3;                 // lanes 32 q .. 32 q + 31
        const int col0 = (e >> 2) * EPI_COLS;   // accumulator columns (tile rows m)
        const int nl = 32 * q + lane;           // tile column
        float acc[EPI_COLS];
        int g = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, C::TN, C::TM);
            for (int c0 = 0; c0 < w.nkb; c0 += C::CHUNK, ++g) {
                const bool got = role_wait(accf, g & 1, timeout_ns, fault, kFaultAccumBarrier,
                                           abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                       static_cast<uint32_t>(col0);
#pragma unroll
                for (int j0 = 0; j0 < EPI_COLS / 16; j0 += C::DRAIN_BATCH) {
                    uint32_t r[C::DRAIN_BATCH][16];
#pragma unroll
                    for (int b = 0; b < C::DRAIN_BATCH; ++b)
                        tmem_ld_32x32b_x16(tbase + 16 * (j0 + b), r[b]);
#pragma unroll
                    for (int b = 0; b < C::DRAIN_BATCH; ++b) tmem_ld_wait(r[b]);
#pragma unroll
                    for (int b = 0; b < C::DRAIN_BATCH; ++b) {
                        const int j = j0 + b;
                        if (c0 == 0) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[16 * j + i] = __uint_as_float(r[b][i]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[16 * j + i] += __uint_as_float(r[b][i]);
                        }
                    }
                }
                // the chunk is in registers: hand the accumulator back
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce);
            }
            if (!ok) break;
            const int n = w.n0 + nl;
            if (n < N) {
                float* p = out + static_cast<long long>(w.split) * split_stride +
                           static_cast<long long>(w.m0 + col0) * ldo + n;
                const int rows = M - (w.m0 + col0);
#pragma unroll
                for (int j = 0; j < EPI_COLS; ++j, p += ldo)
                    if (j < rows) *p = scale1(acc[j], p, alpha, beta, scale_mode);
            }
        }
        if (counters) {
            // the in-kernel reduction, on the epilogue's register share: the
            // partial is made visible before this CTA announces it, then each
            // CTA of the tile sums its band of the tile's rows
            __threadfence();
            bar_sync_named(1, 32 * C::EPI_WARPS);
            const int tiles = tiles_m * tiles_n;
            const Unit w = decode(blockIdx.x, tiles_m, tiles_n, kb_per_split, kb_total, C::TN,
                                  C::TM);
            reduce_tile_in_kernel<C::TM, C::TN, 25>(
                out, ldo, split_stride, counters, tiles, static_cast<int>(blockIdx.x) - w.split * tiles,
                w.m0, w.n0, splits, splits, w.split, 32 * e + lane, 32 * C::EPI_WARPS, 1,
                c_final, ldc, M, N, alpha, beta, c_mode, fault, timeout_ns, abort_flag);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_sgemm_3xtf32_tmem(const Tf32x3Args& a, cudaStream_t s, int sm_count) {
    using C = TmemCfg;
    constexpr auto kern = sgemm_3xtf32_tmem_kernel;
    static thread_local int attr_done_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (attr_done_dev != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done_dev = dev;
    }
    if (a.bn != C::BN || a.pair || a.tail_tiles) return cudaErrorInvalidValue;
    // split-K in a cluster: one unit per CTA, the S splits of a tile as one
    // cluster of S CTAs, C written by the kernel (no workspace)
    if (a.cluster_splits && (a.cluster_splits != a.splits || a.splits < 2 ||
                             a.splits > kMaxTmemClusterSplits || a.counters))
        return cudaErrorInvalidValue;
    const int units = ((a.M + BM - 1) / BM) * ((a.N + C::BN - 1) / C::BN) * a.splits;
    int grid = units < sm_count ? units : sm_count;
    // the in-kernel reduction: one unit per CTA, every CTA resident at once
    if (a.counters && (a.splits < 2 || units > sm_count)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0] = pdl_attribute();
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.numAttrs = a.counters ? 2 : 1;
    if (a.cluster_splits) {
        grid = units;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(a.splits);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    e = cudaLaunchKernelEx(&cfg, kern, a.tmAhi, a.tmBhi, a.out, a.ldo, a.split_stride, a.M, a.N,
                           a.K, a.kb_per_split, a.splits, a.fault, a.timeout_ns, a.alpha, a.beta,
                           a.scale_mode, a.counters, a.c_final, a.ldc, a.c_mode,
                           a.cluster_splits, a.vec_store);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// How many clusters of `splits` CTAs of the single-CTA form can be resident
// at once (one CTA per SM; clusters are placed within a GPC, so this is
// below sm_count / splits for most sizes).
cudaError_t tf32x3_tmem_cluster_capacity(int splits, int* clusters) {
    using C = TmemCfg;
    constexpr auto kern = sgemm_3xtf32_tmem_kernel;
    if (splits < 1 || splits > kMaxTmemClusterSplits) return cudaErrorInvalidValue;
    static thread_local int cached_dev = -1;
    static thread_local int cap[kMaxTmemClusterSplits + 1] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (cached_dev != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        for (int sz = 1; sz <= kMaxTmemClusterSplits; ++sz) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = static_cast<unsigned>(sz);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(sz));
            cfg.blockDim = dim3(C::THREADS);
            cfg.dynamicSmemBytes = C::SMEM_BYTES;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
            if (e != cudaSuccess) return e;
            cap[sz] = n;
        }
        cached_dev = dev;
    }
    *clusters = cap[splits];
    return cudaSuccess;
}

cudaError_t launch_sgemm_3xtf32_tmem_wide(const Tf32x3Args& a, cudaStream_t s, int sm_count) {
    using C = TmemWideCfg;
    constexpr auto kern = sgemm_3xtf32_tmem_wide_kernel;
    static thread_local int attr_done_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (attr_done_dev != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done_dev = dev;
    }
    if (a.pair || a.cluster_splits || a.tail_tiles) return cudaErrorInvalidValue;
    const int units = ((a.M + C::TM - 1) / C::TM) * ((a.N + C::TN - 1) / C::TN) * a.splits;
    const int grid = units < sm_count ? units : sm_count;
    // the in-kernel reduction: one unit per CTA, every CTA resident at once
    if (a.counters && (a.splits < 2 || units > sm_count)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0] = pdl_attribute();
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = a.counters ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, a.tmAhi, a.tmBhi, a.out, a.ldo, a.split_stride, a.M, a.N,
                           a.K, a.kb_per_split, a.splits, a.fault, a.timeout_ns, a.alpha, a.beta,
                           a.scale_mode, a.counters, a.c_final, a.ldc, a.c_mode);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

Tf32x3Config tf32x3_tmem_wide_config() {
    using C = TmemWideCfg;
    return {C::TM, C::TN, C::KB, C::STAGES, C::THREADS, C::SMEM_BYTES, 0, 32};
}

Tf32x3Config tf32x3_tmem_config(bool pair) {
    if (pair) {
        using P = TmemPairCfg;
        return {P::TM, P::TN, BK, P::STAGES, P::THREADS, P::SMEM_BYTES, 1, 32};
    }
    using C = TmemCfg;
    return {BM, C::BN, BK, C::STAGES, C::THREADS, C::SMEM_BYTES, 0, 32};
}

cudaError_t tf32x3_tmem_ctas_per_sm(int* ctas_per_sm) {
    using C = TmemCfg;
    cudaError_t e = cudaFuncSetAttribute(sgemm_3xtf32_tmem_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, sgemm_3xtf32_tmem_kernel,
                                                         C::THREADS, C::SMEM_BYTES);
}


// Co-resident clusters of the pair form on this device (cached per device).
cudaError_t tf32x3_tmem_pair_clusters(int sm_count, int* out) {
    using C = TmemPairCfg;
    static thread_local int done_dev = -1;
    static thread_local int clusters = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (done_dev != dev) {
        e = cudaFuncSetAttribute(sgemm_3xtf32_tmem_pair_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * (sm_count / 2));
        cfg.blockDim = dim3(C::THREADS);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, sgemm_3xtf32_tmem_pair_kernel, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        clusters = n;
        done_dev = dev;
    }
    *out = clusters;
    return cudaSuccess;
}

cudaError_t launch_sgemm_3xtf32_tmem_pair(const Tf32x3Args& a, cudaStream_t s, int sm_count) {
    using C = TmemPairCfg;
    if (!a.pair || a.cluster_splits) return cudaErrorInvalidValue;
    int max_clusters = 0;
    cudaError_t e = tf32x3_tmem_pair_clusters(sm_count, &max_clusters);
    if (e != cudaSuccess) return e;
    const int tiles = ((a.M + C::TM - 1) / C::TM) * ((a.N + C::TN - 1) / C::TN);
    const int units = a.tail_tiles ? tiles - a.tail_tiles + a.tail_tiles * a.tail_splits
                                   : tiles * a.splits;
    const int clusters = units < max_clusters ? units : max_clusters;
    // the in-kernel reduction: one unit per cluster, every cluster resident
    // at once, no tail split
    if (a.counters && (a.splits < 2 || units > max_clusters || a.tail_tiles))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[3];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    attr[2].id = cudaLaunchAttributeCooperative;
    attr[2].val.cooperative = 1;
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = a.counters ? 3 : 2;
    e = cudaLaunchKernelEx(&cfg, sgemm_3xtf32_tmem_pair_kernel, a.tmAhi, a.tmBhi, a.out, a.ldo,
                           a.split_stride, a.M, a.N, a.K, a.kb_per_split, a.splits, a.fault,
                           a.timeout_ns, a.alpha, a.beta, a.scale_mode, a.tail_tiles,
                           a.tail_splits, a.tail_ws, a.counters, a.c_final, a.ldc, a.c_mode);
    if (e != cudaSuccess) return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.tail_tiles) e = launch_pair_tail_fixup(a, s);
    return e;
}

}  // namespace gemm_f32_impl
