// sgemm_3xtf32.cu -- single-precision GEMM on the sm_103a tensor cores.
//
// C = A * B with FP32-level accuracy from TF32 tensor-core products: the
// operands arrive pre-split into high and low parts (tf32_split.cu; the high
// part is the fp32 word itself, which the tensor core reads truncated), and
// every K step issues three tcgen05.mma kind::tf32 products into one fp32
// accumulator in tensor memory:  Alo*Bhi + Ahi*Blo + Ahi*Bhi  (small terms
// first, Alo*Blo dropped).  See "Lecture 12: final project" (section 2,
// tiledMatMulKernel) for the operation and its boundary rules; the pages have
// no tensor-core kernel, so the structure below is this library's own.
//
// The tensor core adds products into its fp32 accumulator with truncation
// (measured here: over an 8192-deep chain the error grows to several times
// the 1e-3 tolerance near zero crossings).  So the accumulation is split:
// each CHUNK of K (CH blocks of 32) is summed by the tensor core into a fresh
// tensor-memory accumulator, and the epilogue warps add the chunk results,
// in chunk order, into fp32 registers with round-to-nearest adds.
//
// Persistent, warp-specialised CTA (one per SM), 128 + 32 * EPI_WARPS threads:
//   warp 0      one lane issues TMA box loads of Ahi, Alo (BM x 32) and Bhi,
//               Blo (BN x 32, from the transposed copy) per K block into a
//               STAGES-deep ring of 128-byte-swizzled shared-memory stages;
//   warp 1      allocates 2*BN tensor-memory columns (two chunk accumulators),
//               and one lane issues the MMAs (128 x BN x 8 each) and the
//               commits that release a stage / publish a chunk;
//   warps 2-3   idle, or the splitters below (the epilogue starts on a
//               warpgroup boundary, as the tensor-memory lane quarters
//               follow the warp index modulo 4);
//   warps 4..   the epilogue: warp e owns tensor-memory lanes 32*(e % 4) ..
//               +31 (rows) and 128 of the BN columns; per chunk it reads them
//               with tcgen05.ld, hands the chunk buffer back at once, and adds
//               the values into its 128 register accumulators; at the end of
//               a tile it writes them to C while the MMAs of the next tile
//               already run: through two 2 KB shared-memory slabs and TMA
//               stores of 32 x 16 boxes, a beta term reading the old box
//               with a TMA load (one K split, C rows a whole number of
//               16-byte units), else with its own loads and stores
//               (float4 where the row stride allows, predicated on ragged
//               edges).  One thread storing a whole row puts 32 rows in each
//               warp store; on 8192 x 8192 x 1024 that left the tensor pipe
//               waiting ~7 us per tile, which the TMA stores remove.
// Work units are (tile, split) pairs in a grouped raster order, strided by
// the grid size.  Every mbarrier wait is bounded; a timeout sets the device
// fault word and a shared abort flag, and the CTA winds down (waits, bounded,
// for its in-flight copies and MMAs, then frees its tensor memory).
//
// SPLIT_IN_KERNEL (128 x 128 tiles only): A and B arrive as stored, a 128 x
// 32 box of A and four 32 x 32 boxes of B per stage, and warps 2-3 split
// them in shared memory exactly as in the pair kernel further down (whose
// header describes the split); the MMA lane then waits on the stage's
// converted barrier instead of its full barrier.
//
// Split K without a workspace (cluster_splits = S, 2..8): the grid is one
// unit per CTA and the S K splits of a tile are the S CTAs of one cluster.
// Each parks its partial tile in its own (drained) stage memory; after a
// cluster barrier every CTA sums a 1/S band of rows over the S partials
// through distributed shared memory, in split order, and stores it.
//
// Both kernels of this file are launched as programmatic dependents: their
// set-up (barriers, tensor memory, descriptor prefetch) overlaps the tail of
// the kernel before them on the stream, and they wait for it (griddepcontrol)
// before the first operand load.
//
// The CTA-pair kernel further down (cta_group::2, 256 x 256 tiles) shares the
// chunked promotion, the bounded waits and the tail handling; its header
// describes its roles and its in-shared-memory split of raw operands.
#include <cstdint>

#include "device_sync.cuh"
#include "epilogue.cuh"
#include "gemm_internal.h"
#include "tcgen05.cuh"
#include "tf32x3_common.cuh"

namespace gemm_f32_impl {
namespace {

using namespace gemm_f32_dev;

constexpr int kMaxClusterSplits = 8;  // split-K partials added inside a (portable) cluster

__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t cluster_addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

// Output slabs of the TMA-store epilogue: two per epilogue warp, each 32 rows
// x 16 columns of C with 64-byte swizzle, after the pipeline stages.
constexpr int EPI_SLAB_COLS = 16;
constexpr int EPI_SLAB_BYTES = 32 * EPI_SLAB_COLS * 4;

template <int BN, int STAGES>
struct Cfg {
    static constexpr int EPI_WARPS = 4 * (BN / EPI_COLS);
    // warpgroup 0: producer, MMA issuer, two idle warps; then the epilogue
    static constexpr int THREADS = 128 + 32 * EPI_WARPS;
    static constexpr int A_BYTES = BM * BK * 4;
    static constexpr int B_BYTES = BN * BK * 4;
    static constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    // Barriers: full (one per stage; in the variant that splits A and B in
    // shared memory one per stage fill mod 2 STAGES, each waited on by one
    // of the two splitter warps), empty, converted (that variant), acc_full
    // x2, acc_empty x2, drain, old-C load per epilogue warp.  Both variants
    // reserve the larger set: one shared-memory size, one occupancy.
    static constexpr int NSPLIT = 2;
    static constexpr int NBARS = STAGES * NSPLIT + 2 * STAGES + 5 + EPI_WARPS;
    static constexpr int EPI_BYTES = EPI_WARPS * 2 * EPI_SLAB_BYTES;  // output slabs
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + NBARS * 8 + 16 + 1024;
    static constexpr uint32_t IDESC = idesc_tf32_f32(BM, BN);
    static_assert(BN % EPI_COLS == 0 && BN <= 256, "MMA N for M = 128, whole epilogue blocks");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512 || TMEM_COLS == 128, "power-of-two TMEM");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// One warp's 32 rows x EPI_COLS columns of C (lane = row y + lane, columns x0
// ..) through its two shared-memory slabs and TMA stores.  A 16-column piece
// goes to a slab (the 16-byte chunk c of row r at chunk c ^ ((r >> 1) & 3),
// the 64-byte swizzle, so the lanes' float4 writes hit distinct banks) and out
// with one TMA store: whole lines, and the warp moves on while the store
// drains.  Ragged edges are clipped by the tensor map's extent; pieces wholly
// outside C are skipped, and the slabs alternate by stores issued (`stores`,
// the warp's running count), so that the store that last read a slab is
// always the one before the latest.  With a beta term the old box of C is
// first loaded into the slab (TMA, completion on the warp's barrier `cbar`,
// `loads` counting its phases; a bounded wait) and each lane replaces its row
// of it by alpha v + beta C.  Returns false if that wait gave up.
__device__ __forceinline__ bool store_rows_tma(const float (&acc)[EPI_COLS], uint32_t slabs,
                                               int& stores, int& loads, uint32_t cbar, int lane,
                                               const CUtensorMap* tmC, int x0, int y, int M,
                                               int N, float alpha, float beta, int scale_mode,
                                               long long timeout_ns, unsigned* fault,
                                               uint32_t abort_flag) {
    if (y >= M) return true;  // the same for the whole warp
    const uint32_t sw = static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll
    for (int pc = 0; pc < EPI_COLS / EPI_SLAB_COLS; ++pc) {
        const int x = x0 + pc * EPI_SLAB_COLS;
        if (x >= N) continue;
        const uint32_t slab = slabs + (stores & 1) * EPI_SLAB_BYTES;
        ++stores;
        // the store issued from this slab two stores ago has read it
        if (lane == 0) {
            bulk_wait_read<1>();
            if (scale_mode == kStoreAlphaBeta) {
                mbar_arrive_expect_tx(cbar, EPI_SLAB_BYTES);
                tma_load_2d(slab, tmC, cbar, x, y);
            }
        }
        __syncwarp();
        if (scale_mode == kStoreAlphaBeta) {
            const uint32_t parity = static_cast<uint32_t>(loads & 1);
            const bool got =
                role_wait(cbar, parity, timeout_ns, fault, kFaultOutputLoad, abort_flag);
            ++loads;
            if (!__all_sync(0xffffffffu, got)) {
                // giving up (another role aborted, or this wait timed out):
                // the load may still be landing in the slab, so wait for it,
                // bounded, before the CTA can leave
                mbar_wait(cbar, parity, timeout_ns / 8 + 1000, fault, kFaultDrain);
                return false;
            }
        }
#pragma unroll
        for (int c = 0; c < EPI_SLAB_COLS / 4; ++c) {
            const int j = pc * EPI_SLAB_COLS + 4 * c;
            const uint32_t a = slab + lane * 64 + ((static_cast<uint32_t>(c) ^ sw) << 4);
            float4 v = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
            if (scale_mode != kStorePlain) {
                v.x *= alpha;
                v.y *= alpha;
                v.z *= alpha;
                v.w *= alpha;
            }
            if (scale_mode == kStoreAlphaBeta) {
                const float4 o = lds128(a);
                v.x = fmaf(beta, o.x, v.x);
                v.y = fmaf(beta, o.y, v.y);
                v.z = fmaf(beta, o.z, v.z);
                v.w = fmaf(beta, o.w, v.w);
            }
            sts128(a, v);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmC, slab, x, y);
            bulk_commit();
        }
    }
    return true;
}

// With a beta term: bring the warp's boxes of the old C into L2 when its tile
// starts, so that the loads of store_rows_tma find them there (lane 0).
__device__ __forceinline__ void prefetch_rows_tma(const CUtensorMap* tmC, int x0, int y, int M,
                                                  int N) {
    if (y >= M) return;
#pragma unroll
    for (int pc = 0; pc < EPI_COLS / EPI_SLAB_COLS; ++pc)
        if (x0 + pc * EPI_SLAB_COLS < N) tma_prefetch_2d(tmC, x0 + pc * EPI_SLAB_COLS, y);
}


// B slot (16 KB at sb): on entry four TMA boxes of 32 k-rows x 32 columns
// (128-byte rows, box j holding columns 32 j .. 32 j + 31; 16-byte chunk c
// of row k sits at chunk c ^ (k & 7)).  On exit the K-major hi plane in its
// place (row n = 128 bytes of k = 0..31, chunk q at q ^ (n & 7): the layout
// TMA gives a box of the transposed copy) and the lo plane 16 KB further on.
// Call w (0, 1) does boxes 2w and 2w + 1, i.e. bytes [8192 w, 8192 w +
// 8192) of both layouts, so the in-place transpose of one call needs only
// its own warp; one warp makes both calls for a stage.
// Lane l takes the 4 x 4 blocks (n = 32 j + 4 c .. + 3, k = 4 kq .. + 3)
// with c = l % 8, kq = l / 8 and l / 8 + 4, j = 2w, 2w + 1: it loads all of
// them (eight lanes read one 128-byte row: conflict-free), the warp syncs,
// then it stores each n's four k values as one 16-byte word.  The store
// order over a block's four n is rotated by c / 2 so that the eight lanes
// of a quarter-warp write eight different n % 8, i.e. eight different
// 16-byte bank groups.
__device__ __forceinline__ void split_b_stage(uint32_t sb, int w, int lane) {
    const int c = lane & 7;
    const int rot = (c >> 1) & 3;
    float4 v[2][2][4];  // [box j - 2w][kq half][k - 4 kq], lanes over n - 32 j - 4 c
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int k = 4 * ((lane >> 3) + 4 * h) + kk;
                v[jj][h][kk] = rotate4(
                    lds128(sb + (2 * w + jj) * 4096 + k * 128 + ((c ^ (k & 7)) << 4)), rot);
            }
    __syncwarp();  // every raw word of this warp's half is in registers
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int kq = (lane >> 3) + 4 * h;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int n = 32 * (2 * w + jj) + 4 * c + ((e + rot) & 3);
                // lane e of the rotated words is column n; k = 4 kq + 0..3
                const float4 x = make_float4(lane_of(v[jj][h][0], e), lane_of(v[jj][h][1], e),
                                             lane_of(v[jj][h][2], e), lane_of(v[jj][h][3], e));
                const uint32_t a = sb + n * 128 + ((kq ^ (n & 7)) << 4);
                sts128(a, x);
                sts128(a + 16384, lo4(x));
            }
        }
}

template <int BN, int STAGES, bool SPLIT_IN_KERNEL = false>
__global__ void __launch_bounds__(Cfg<BN, STAGES>::THREADS, 1)
sgemm_3xtf32_kernel(const __grid_constant__ CUtensorMap tmAhi,
                    const __grid_constant__ CUtensorMap tmAlo,
                    const __grid_constant__ CUtensorMap tmBhi,
                    const __grid_constant__ CUtensorMap tmBlo, float* __restrict__ out,
                    long long ldo, long long split_stride, int M, int N, int K, int kb_per_split,
                    int splits, int vec_store, unsigned* fault, long long timeout_ns,
                    float alpha, float beta, int scale_mode, int cluster_splits,
                    const __grid_constant__ CUtensorMap tmC, int tma_store) {
    using C = Cfg<BN, STAGES>;
    static_assert(!SPLIT_IN_KERNEL || BN == 128, "the splitter's maps: 128 x 32 A and B slots");
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t epi0 = sbase + STAGES * C::STAGE_BYTES;  // output slabs
    const uint32_t bar0 = epi0 + C::EPI_BYTES;
    // full[f]: f = stage, or (split in kernel) f = stage fill mod NFULL
    constexpr int NFULL = SPLIT_IN_KERNEL ? STAGES * C::NSPLIT : STAGES;
    const uint32_t full0 = bar0;
    const uint32_t empty0 = full0 + 8 * STAGES * C::NSPLIT;  // empty[s]     = empty0 + 8 s
    const uint32_t conv0 = empty0 + 8 * STAGES;              // converted[s] = conv0 + 8 s
    const uint32_t accf0 = conv0 + 8 * STAGES;               // acc_full[b]  = accf0 + 8 b
    const uint32_t acce0 = accf0 + 16;                       // acc_empty[b] = acce0 + 8 b
    const uint32_t drain = acce0 + 16;
    const uint32_t cload0 = drain + 8;                // old-C load of epilogue warp e: + 8 e
    uint32_t* tmem_slot =
        reinterpret_cast<uint32_t*>(smem + STAGES * C::STAGE_BYTES + C::EPI_BYTES + C::NBARS * 8);
    const uint32_t abort_flag = smem_addr(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles_m = (M + BM - 1) / BM;
    const int tiles_n = (N + BN - 1) / BN;
    const int units = tiles_m * tiles_n * splits;
    const int kb_total = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmAhi);
        prefetch_tmap(&tmBhi);
        if (!SPLIT_IN_KERNEL) {
            prefetch_tmap(&tmAlo);
            prefetch_tmap(&tmBlo);
        }
        if (tma_store) prefetch_tmap(&tmC);
        for (int f = 0; f < NFULL; ++f) mbar_init(full0 + 8 * f, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(empty0 + 8 * s, 1);
            mbar_init(conv0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, C::EPI_WARPS);
        }
        mbar_init(drain, 1);
        for (int w = 0; w < C::EPI_WARPS; ++w) mbar_init(cload0 + 8 * w, 1);
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
    // launched programmatically: the set-up above overlapped the staging
    // kernel; its operands are read only after this
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------ TMA producer ------------------------------
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, BN, BM,
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
                    if (SPLIT_IN_KERNEL) {
                        // A and B as stored, into the hi slots: a 128 x 32
                        // box of A (K-major already) and four 32 x 32 boxes
                        // of B (N-contiguous), for a splitter warp to split
                        const uint32_t fb = full0 + 8 * (it % NFULL);
                        mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_BYTES);
                        tma_load_2d(st, &tmAhi, fb, k0, w.m0);
#pragma unroll
                        for (int j = 0; j < BN / 32; ++j)
                            tma_load_2d(st + 2 * C::A_BYTES + j * 4096, &tmBhi, fb, w.n0 + 32 * j,
                                        k0);
                        if (kb + kPrefetchAhead < w.nkb) {
                            const int kp = k0 + kPrefetchAhead * BK;
                            tma_prefetch_2d(&tmAhi, kp, w.m0);
#pragma unroll
                            for (int j = 0; j < BN / 32; ++j)
                                tma_prefetch_2d(&tmBhi, w.n0 + 32 * j, kp);
                        }
                    } else {
                        const uint32_t fb = full0 + 8 * s;
                        mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                        tma_load_2d(st, &tmAhi, fb, k0, w.m0);
                        tma_load_2d(st + C::A_BYTES, &tmAlo, fb, k0, w.m0);
                        tma_load_2d(st + 2 * C::A_BYTES, &tmBhi, fb, k0, w.n0);
                        tma_load_2d(st + 2 * C::A_BYTES + C::B_BYTES, &tmBlo, fb, k0, w.n0);
                    }

                }
            }
            // wind down: every issued copy has landed and every stage has been
            // released by the MMA commits before the CTA may exit
            const long long tail = ok ? timeout_ns : timeout_ns / 8 + 1000;
            for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j) {
                mbar_wait(full0 + 8 * (j % NFULL), (j / NFULL) & 1, tail, fault, kFaultDrain);
                mbar_wait(empty0 + 8 * (j % STAGES), (j / STAGES) & 1, tail, fault, kFaultDrain);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------ MMA issuer --------------------------------
            int it = 0;  // K blocks consumed (smem ring position)
            int g = 0;   // chunks issued (tensor-memory buffer g & 1)
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, BN, BM,
                                      cluster_splits);
                for (int c0 = 0; c0 < w.nkb && ok; c0 += CH, ++g) {
                    const int buf = g & 1;
                    if (g >= 2 && !role_wait(acce0 + 8 * buf, ((g >> 1) & 1) ^ 1, timeout_ns, fault,
                                             kFaultAccumBarrier, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
                    const int c1 = min(w.nkb, c0 + CH);
                    for (int kb = c0; kb < c1; ++kb, ++it) {
                        const int s = it % STAGES;
                        // split in kernel: the stage's converted barrier
                        if (!role_wait((SPLIT_IN_KERNEL ? conv0 : full0) + 8 * s,
                                       (it / STAGES) & 1, timeout_ns, fault, kFaultFullBarrier,
                                       abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t st = sbase + s * C::STAGE_BYTES;
                        const uint64_t a_hi = smem_desc_sw128_kmajor(st);
                        const uint64_t a_lo = smem_desc_sw128_kmajor(st + C::A_BYTES);
                        const uint64_t b_hi = smem_desc_sw128_kmajor(st + 2 * C::A_BYTES);
                        const uint64_t b_lo =
                            smem_desc_sw128_kmajor(st + 2 * C::A_BYTES + C::B_BYTES);
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            // advance the start address by k * 32 bytes (encoded >> 4)
                            const uint64_t off = static_cast<uint64_t>(k * UMMA_K * 4) >> 4;
                            const uint32_t acc = (kb > c0 || k > 0) ? 1u : 0u;
                            mma_tf32(d, a_lo + off, b_hi + off, C::IDESC, acc);
                            mma_tf32(d, a_hi + off, b_lo + off, C::IDESC, 1u);
                            mma_tf32(d, a_hi + off, b_hi + off, C::IDESC, 1u);
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
        if (SPLIT_IN_KERNEL) {
            // ------------------------------ splitter (warps 2-3) ----------------------
            // as in the pair kernel: warp 2 splits the even-numbered stage
            // fills, warp 3 the odd ones, each a whole stage, so that one
            // warp's store drain overlaps the other's conversions
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, BN, BM,
                                      cluster_splits);
                for (int kb = 0; kb < w.nkb; ++kb, ++it) {
                    if (it % C::NSPLIT != warp - 2) continue;  // the other splitter's turn
                    const int s = it % STAGES;
                    const bool got = role_wait(full0 + 8 * (it % NFULL), (it / NFULL) & 1,
                                               timeout_ns, fault, kFaultFullBarrier, abort_flag);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sbase + s * C::STAGE_BYTES;
                    split_a_stage(st, lane);
                    split_a_stage(st, lane + 32);
                    split_b_stage(st + 2 * C::A_BYTES, 0, lane);
                    split_b_stage(st + 2 * C::A_BYTES, 1, lane);
                    // the tensor core reads these words through the async proxy
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(conv0 + 8 * s);
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------ epilogue ----------------------------------
        const int e = warp - 4;
        const int q = warp & 3;             // tensor-memory lanes 32q .. 32q+31
        const int col0 = (e >> 2) * EPI_COLS;  // this warp's 128 accumulator columns
        const int row = 32 * q + lane;
        float acc[EPI_COLS];
        int g = 0;
        int stores = 0;  // TMA stores this warp has issued
        int loads = 0;   // old-C boxes this warp has loaded
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const Unit w = decode(u, tiles_m, tiles_n, kb_per_split, kb_total, BN, BM,
                                  cluster_splits);
            if (tma_store && scale_mode == kStoreAlphaBeta && lane == 0)
                prefetch_rows_tma(&tmC, w.n0 + col0, w.m0 + 32 * q, M, N);
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
                                       static_cast<uint32_t>(buf * BN + col0);
                // 16 columns at a time: load, wait, add (keeps 16 + 128 registers live)
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
                // the chunk is in registers: give the buffer back to the MMA warp
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce0 + 8 * buf);
            }
            if (!ok) break;
            if (cluster_splits) {
                // this CTA's only unit: its partial tile goes into the stage
                // memory (every MMA, and so every operand read, has completed),
                // row-major 128 x BN with 16-byte word c of row r at c ^ (r & 7)
#pragma unroll
                for (int j = 0; j < EPI_COLS; j += 4) {
                    const int c4 = (col0 + j) >> 2;
                    sts128(sbase + 16u * static_cast<uint32_t>(row * (BN / 4) + (c4 ^ (row & 7))),
                           make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]));
                }
                continue;
            }
            if (tma_store) {
                ok = store_rows_tma(acc, epi0 + static_cast<uint32_t>(e) * 2 * EPI_SLAB_BYTES,
                                    stores, loads, cload0 + 8 * e, lane, &tmC, w.n0 + col0,
                                    w.m0 + 32 * q, M, N, alpha, beta, scale_mode, timeout_ns,
                                    fault, abort_flag);
                continue;
            }
            const int m = w.m0 + row;
            if (m < M) {
                float* orow = out + static_cast<long long>(w.split) * split_stride +
                              static_cast<long long>(m) * ldo;
                const int nb = w.n0 + col0;
#pragma unroll
                for (int j = 0; j < EPI_COLS; j += 4)
                    store4(orow, nb + j, N, make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]),
                           vec_store != 0, alpha, beta, scale_mode);
            }
        }
        // the output stores have completed (and no longer read the slabs)
        if (tma_store && lane == 0) bulk_wait_all();
        __syncwarp();
    }

    if (cluster_splits) {
        // ---- split-K reduction inside the cluster: the S CTAs of the cluster
        // hold the S K splits of one tile (each its only unit).  Every thread
        // of every CTA takes both barriers, whatever its role did. ----
        cluster_sync();  // all partials parked and visible across the cluster
        const int S = cluster_splits;
        const uint32_t rank = cluster_ctarank();
        const Unit w = decode(static_cast<int>(blockIdx.x), tiles_m, tiles_n, kb_per_split,
                              kb_total, BN, BM, S);
        const int rows = (BM + S - 1) / S;
        const int r0 = static_cast<int>(rank) * rows;
        const int r1 = min(BM, r0 + rows);
        constexpr int Q = BN / 4;  // 16-byte words per tile row
        uint32_t peer[kMaxClusterSplits];
#pragma unroll
        for (int q = 0; q < kMaxClusterSplits; ++q)
            peer[q] = q < S ? map_to_cta(sbase, static_cast<uint32_t>(q)) : 0u;
        if (ld_shared_volatile(abort_flag) == 0u) {
            for (int idx = threadIdx.x; idx < (r1 - r0) * Q; idx += C::THREADS) {
                const int i = r0 + idx / Q;
                const int c4 = idx - (idx / Q) * Q;
                const int m = w.m0 + i;
                if (m >= M) continue;
                const uint32_t off = 16u * static_cast<uint32_t>(i * Q + (c4 ^ (i & 7)));
                float4 sum = ld_dsmem_v4(peer[0] + off);
#pragma unroll
                for (int q = 1; q < kMaxClusterSplits; ++q) {
                    if (q < S) {
                        const float4 v = ld_dsmem_v4(peer[q] + off);
                        sum.x += v.x;
                        sum.y += v.y;
                        sum.z += v.z;
                        sum.w += v.w;
                    }
                }
                store4(out + static_cast<long long>(m) * ldo, w.n0 + 4 * c4, N, sum,
                       vec_store != 0, alpha, beta, scale_mode);
            }
        }
        cluster_sync();  // no CTA leaves while a partner may still read its partial
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int BN, int STAGES, bool SPLIT_IN_KERNEL = false>
cudaError_t launch_impl(const Tf32x3Args& a, cudaStream_t s, int sm_count) {
    using C = Cfg<BN, STAGES>;
    constexpr auto kern = sgemm_3xtf32_kernel<BN, STAGES, SPLIT_IN_KERNEL>;
    static thread_local int attr_done_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (attr_done_dev != dev) {
        e = cudaFuncSetAttribute(kern,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done_dev = dev;
    }
    const int units = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN) * a.splits;
    if (a.cluster_splits) {
        // one unit per CTA, the splits of a tile as one cluster
        if (a.cluster_splits != a.splits || a.splits < 2 || a.splits > kMaxClusterSplits)
            return cudaErrorInvalidValue;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(a.splits);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1] = pdl_attribute();
        cfg.gridDim = dim3(static_cast<unsigned>(units));
        cfg.blockDim = dim3(C::THREADS);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, kern, a.tmAhi, a.tmAlo, a.tmBhi,
                               a.tmBlo, a.out, a.ldo, a.split_stride, a.M, a.N, a.K,
                               a.kb_per_split, a.splits, a.vec_store, a.fault, a.timeout_ns,
                               a.alpha, a.beta, a.scale_mode, a.cluster_splits, a.tmC, 0);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    const int grid = units < sm_count ? units : sm_count;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a.tmAhi, a.tmAlo, a.tmBhi,
                           a.tmBlo, a.out, a.ldo, a.split_stride, a.M, a.N, a.K, a.kb_per_split,
                           a.splits, a.vec_store, a.fault, a.timeout_ns, a.alpha, a.beta,
                           a.scale_mode, 0, a.tmC, a.tma_store);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}


// ============================================================================
// CTA-pair variant: a cluster of two CTAs on two SMs computes a 256 x 256
// tile with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 8).  CTA rank r
// holds rows m0 + 128 r of A and columns n0 + 128 r of B in its own shared
// memory, so every SM reads 8 KB of operands per MMA instead of the 12 KB of
// the single-CTA 128 x 256 MMA; that is what lets the tensor pipe outrun
// shared-memory bandwidth.  Each CTA's tensor memory holds its 128 rows x 256
// columns; its epilogue warps promote and store them.
//
// Two ways to feed it, chosen by SPLIT_IN_KERNEL:
//   false  the operands arrive pre-split (Ahi, Alo and the transposed Bhi,
//          Blo planes of tf32_split.cu), all K-major.  Both producers arrive
//          (with their own transaction bytes) on the leader's full barrier
//          and point their TMA completions at it.
//   true   each CTA's producer loads the operands as stored into the hi
//          slots, signalling its own full barrier: a 128 x 32 box of A
//          (K-major already) and four 32 x 32 boxes of B (N-contiguous).
//          Warp 2 or 3 of each CTA (taking turns by stage fill) then
//          splits the stage in shared memory:
//          A elementwise (x stays in the hi slot as its own high part, lo =
//          tf32(x - trunc(x)) goes to the lo slot); B by 4 x 4 blocks read
//          into registers, transposed and written back K-major as hi (the
//          words themselves) and lo.  These are the
//          values and the layout the staging kernels would have produced,
//          so the MMAs are the same.  The splitters fence their writes for
//          the tensor core and arrive on the leader's converted barrier.
//          (The tensor core is not given B N-major: with the B-major bit of
//          the instruction descriptor set, kind::tf32 MMAs of this kernel
//          wrote zeros on this part.)
// In both, the leader's MMA lane multicasts each commit to the same barrier
// offset in both CTAs (stage free / chunk ready), and both epilogues release
// a chunk buffer by arriving on the leader's acc_empty barrier.
// ============================================================================
template <int STAGES, bool SPLIT_IN_KERNEL = false>
struct PairCfg {
    static constexpr int BN = 256;       // MMA N, shared by the pair
    static constexpr int HALF_N = 128;   // columns of B held by each CTA
    static constexpr int A_BYTES = BM * BK * 4;
    static constexpr int B_BYTES = HALF_N * BK * 4;
    static constexpr int B_BOX_N = 32;   // N-contiguous B box width: one 128-byte swizzle row
    static constexpr int B_BOX_BYTES = B_BOX_N * BK * 4;
    static constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int EPI_WARPS = BN / EPI_COLS * 4;
    static constexpr int THREADS = 128 + 32 * EPI_WARPS;
    // splitter warps 2-3: each splits whole stages, the two taking turns
    static constexpr int NSPLIT = 2;
    // Full barriers.  Pre-split operands: one per stage.  Split in kernel:
    // one per (stage fill mod STAGES * NSPLIT), so that every full barrier
    // is waited on by one splitter warp, phase after phase.  (With one
    // barrier per stage, a warp that takes every other fill of a stage would
    // skip a phase, and a parity wait cannot tell phase k from phase k + 2.)
    static constexpr int NFULL = SPLIT_IN_KERNEL ? STAGES * NSPLIT : STAGES;
    // full (NFULL), empty, converted (per stage), acc_full x2, acc_empty x2, drain
    // ... and an old-C load barrier per epilogue warp
    static constexpr int NBARS = NFULL + 2 * STAGES + 5 + EPI_WARPS;
    static constexpr int EPI_BYTES = EPI_WARPS * 2 * EPI_SLAB_BYTES;  // output slabs
    // both variants reserve room for the split variant's barriers, so that
    // they have the same shared-memory size (and occupancy)
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES +
                                      (STAGES * NSPLIT + 2 * STAGES + 5 + EPI_WARPS) * 8 + 16 +
                                      1024;
    static constexpr uint32_t IDESC = idesc_tf32_f32(2 * BM, BN);
    static_assert(A_BYTES == B_BYTES && B_BYTES == 16384,
                  "the splitter's thread-to-element maps below");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

template <int STAGES, bool SPLIT_IN_KERNEL>
__global__ void __launch_bounds__(PairCfg<STAGES, SPLIT_IN_KERNEL>::THREADS, 1)
sgemm_3xtf32_pair_kernel(const __grid_constant__ CUtensorMap tmAhi,
                         const __grid_constant__ CUtensorMap tmAlo,
                         const __grid_constant__ CUtensorMap tmBhi,
                         const __grid_constant__ CUtensorMap tmBlo, float* __restrict__ out,
                         long long ldo, long long split_stride, int M, int N, int K,
                         int kb_per_split, int splits, int vec_store, unsigned* fault,
                         long long timeout_ns, float alpha, float beta, int scale_mode,
                         int tail_tiles, int tail_splits, float* __restrict__ tail_ws,
                         const __grid_constant__ CUtensorMap tmC, int tma_store) {
    using C = PairCfg<STAGES, SPLIT_IN_KERNEL>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t epi0 = sbase + STAGES * C::STAGE_BYTES;  // output slabs
    const uint32_t bar0 = epi0 + C::EPI_BYTES;
    // full[f]: pre-split operands: f = stage, the leader's, count 2 (both
    //          producers); split in kernel: f = fill mod NFULL, each CTA's
    //          own, count 1
    const uint32_t full0 = bar0;
    const uint32_t empty0 = full0 + 8 * C::NFULL;  // empty[s]: both CTAs, one multicast commit
    const uint32_t conv0 = empty0 + 8 * STAGES;    // converted[s]: leader, 1 warp x 2 CTAs
    const uint32_t accf0 = conv0 + 8 * STAGES;     // acc_full[b]: both CTAs, one multicast commit
    const uint32_t acce0 = accf0 + 16;            // acc_empty[b]: leader, both epilogues
    const uint32_t drain = acce0 + 16;
    const uint32_t cload0 = drain + 8;             // old-C load of epilogue warp e: + 8 e
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + STAGES * C::STAGE_BYTES +
                                                      C::EPI_BYTES + C::NBARS * 8);
    const uint32_t abort_flag = smem_addr(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x >> 1;
    const int nclusters = gridDim.x >> 1;
    const int tiles_m = (M + 2 * BM - 1) / (2 * BM);
    const int tiles_n = (N + C::BN - 1) / C::BN;
    const int units = tail_tiles ? tiles_m * tiles_n - tail_tiles + tail_tiles * tail_splits
                                 : tiles_m * tiles_n * splits;
    const int kb_total = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmAhi);
        prefetch_tmap(&tmBhi);
        if (!SPLIT_IN_KERNEL) {
            prefetch_tmap(&tmAlo);
            prefetch_tmap(&tmBlo);
        }
        if (!SPLIT_IN_KERNEL && tma_store) prefetch_tmap(&tmC);
        for (int f = 0; f < C::NFULL; ++f) mbar_init(full0 + 8 * f, SPLIT_IN_KERNEL ? 1 : 2);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(empty0 + 8 * s, 1);
            mbar_init(conv0 + 8 * s, 2);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, 2 * C::EPI_WARPS);
        }
        mbar_init(drain, 1);
        for (int w = 0; w < C::EPI_WARPS; ++w) mbar_init(cload0 + 8 * w, 1);
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
    pdl_wait();  // as in the single-CTA kernel
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------ TMA producer (both CTAs) ------------------
            int it = 0;
            bool ok = true;
            for (int u = cluster; u < units && ok; u += nclusters) {
                const Unit w = decode_pair(u, tiles_m, tiles_n, kb_per_split, kb_total, C::BN, tail_tiles, tail_splits);
                const int ma = w.m0 + static_cast<int>(rank) * BM;
                const int nb = w.n0 + static_cast<int>(rank) * C::HALF_N;
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
                    if (SPLIT_IN_KERNEL) {
                        const uint32_t fb = full0 + 8 * (it % C::NFULL);
                        mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_BYTES);
                        tma_load_2d(st, &tmAhi, fb, k0, ma);
#pragma unroll
                        for (int j = 0; j < C::HALF_N / C::B_BOX_N; ++j)
                            tma_load_2d(st + 2 * C::A_BYTES + j * C::B_BOX_BYTES, &tmBhi, fb,
                                        nb + j * C::B_BOX_N, k0);
                        if (kb + kPrefetchAhead < w.nkb) {
                            const int kp = k0 + kPrefetchAhead * BK;
                            tma_prefetch_2d(&tmAhi, kp, ma);
#pragma unroll
                            for (int j = 0; j < C::HALF_N / C::B_BOX_N; ++j)
                                tma_prefetch_2d(&tmBhi, nb + j * C::B_BOX_N, kp);
                        }
                    } else {
                        const uint32_t fb = map_to_cta(full0 + 8 * s, 0);
                        mbar_arrive_expect_tx_cluster(fb, C::STAGE_BYTES);
                        tma_load_2d_pair(st, &tmAhi, fb, k0, ma);
                        tma_load_2d_pair(st + C::A_BYTES, &tmAlo, fb, k0, ma);
                        tma_load_2d_pair(st + 2 * C::A_BYTES, &tmBhi, fb, k0, nb);
                        tma_load_2d_pair(st + 2 * C::A_BYTES + C::B_BYTES, &tmBlo, fb, k0, nb);
                    }
                }
            }
            // wind down: every stage this CTA filled has landed (own full
            // barrier, split in kernel) and been consumed and released
            const long long tail = ok ? timeout_ns : timeout_ns / 8 + 1000;
            for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j) {
                if (SPLIT_IN_KERNEL)
                    mbar_wait(full0 + 8 * (j % C::NFULL), (j / C::NFULL) & 1, tail, fault,
                              kFaultDrain);
                mbar_wait(empty0 + 8 * (j % STAGES), (j / STAGES) & 1, tail, fault, kFaultDrain);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------ MMA issuer (leader CTA) ------------------
            int it = 0;
            int g = 0;
            bool ok = true;
            for (int u = cluster; u < units && ok; u += nclusters) {
                const Unit w = decode_pair(u, tiles_m, tiles_n, kb_per_split, kb_total, C::BN, tail_tiles, tail_splits);
                for (int c0 = 0; c0 < w.nkb && ok; c0 += CH, ++g) {
                    const int buf = g & 1;
                    if (g >= 2 && !role_wait(acce0 + 8 * buf, ((g >> 1) & 1) ^ 1, timeout_ns, fault,
                                             kFaultAccumBarrier, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + static_cast<uint32_t>(buf * C::BN);
                    const int c1 = min(w.nkb, c0 + CH);
                    for (int kb = c0; kb < c1; ++kb, ++it) {
                        const int s = it % STAGES;
                        const bool got =
                            SPLIT_IN_KERNEL
                                ? role_wait<true>(conv0 + 8 * s, (it / STAGES) & 1, timeout_ns,
                                                  fault, kFaultFullBarrier, abort_flag)
                                : role_wait(full0 + 8 * s, (it / STAGES) & 1, timeout_ns, fault,
                                            kFaultFullBarrier, abort_flag);
                        if (!got) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t st = sbase + s * C::STAGE_BYTES;
                        const uint64_t a_hi = smem_desc_sw128_kmajor(st);
                        const uint64_t a_lo = smem_desc_sw128_kmajor(st + C::A_BYTES);
                        const uint64_t b_hi = smem_desc_sw128_kmajor(st + 2 * C::A_BYTES);
                        const uint64_t b_lo =
                            smem_desc_sw128_kmajor(st + 2 * C::A_BYTES + C::B_BYTES);
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            const uint64_t off = static_cast<uint64_t>(k * UMMA_K * 4) >> 4;
                            const uint32_t acc = (kb > c0 || k > 0) ? 1u : 0u;
                            mma_tf32_pair(d, a_lo + off, b_hi + off, C::IDESC, acc);
                            mma_tf32_pair(d, a_hi + off, b_lo + off, C::IDESC, 1u);
                            mma_tf32_pair(d, a_hi + off, b_hi + off, C::IDESC, 1u);
                        }
                        mma_commit_pair_multicast(empty0 + 8 * s, 0x3);
                    }
                    if (!ok) break;
                    mma_commit_pair_multicast(accf0 + 8 * buf, 0x3);
                }
            }
            mma_commit_pair(drain);
            mbar_wait(drain, 0, ok ? timeout_ns : timeout_ns / 8 + 1000, fault, kFaultDrain);
        }
        __syncwarp();
    } else if (warp < 4) {
        if (SPLIT_IN_KERNEL) {
            // ------------------------------ splitter (warps 2-3, both CTAs) -----------
            // Warp 2 splits the even-numbered stage fills, warp 3 the odd
            // ones, each a whole stage: one warp's wait for its stores to
            // drain (the fence before the arrive) overlaps the other's
            // conversions.  Splitting every stage by both warps, half each,
            // was slower by 7-13 % (8192^3 on this kernel: 4.94 against 4.28
            // ms; 256 x 256 x 65536: 71.3 against 66.2 us).
            const uint32_t conv_leader = map_to_cta(conv0, 0);
            int it = 0;
            bool ok = true;
            for (int u = cluster; u < units && ok; u += nclusters) {
                const Unit w = decode_pair(u, tiles_m, tiles_n, kb_per_split, kb_total, C::BN,
                                           tail_tiles, tail_splits);
                for (int kb = 0; kb < w.nkb; ++kb, ++it) {
                    if (it % C::NSPLIT != warp - 2) continue;  // the other splitter's turn
                    const int s = it % STAGES;
                    const bool got = role_wait(full0 + 8 * (it % C::NFULL), (it / C::NFULL) & 1,
                                               timeout_ns, fault, kFaultFullBarrier, abort_flag);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sbase + s * C::STAGE_BYTES;
                    split_a_stage(st, lane);
                    split_a_stage(st, lane + 32);
                    split_b_stage(st + 2 * C::A_BYTES, 0, lane);
                    split_b_stage(st + 2 * C::A_BYTES, 1, lane);
                    // the tensor core reads these words through the async proxy
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(conv_leader + 8 * s);
                }
            }
        }
    } else {
        // ------------------------------ epilogue (both CTAs) ----------------------
        const int e = warp - 4;
        const int q = warp & 3;
        const int col0 = (e >> 2) * EPI_COLS;
        const int row = 32 * q + lane;
        float acc[EPI_COLS];
        int g = 0;
        int stores = 0;  // TMA stores this warp has issued
        int loads = 0;   // old-C boxes this warp has loaded
        bool ok = true;
        for (int u = cluster; u < units && ok; u += nclusters) {
            const Unit w = decode_pair(u, tiles_m, tiles_n, kb_per_split, kb_total, C::BN, tail_tiles, tail_splits);
            if (!SPLIT_IN_KERNEL && tma_store && scale_mode == kStoreAlphaBeta && w.slot < 0 &&
                lane == 0)
                prefetch_rows_tma(&tmC, w.n0 + col0, w.m0 + static_cast<int>(rank) * BM + 32 * q, M,
                                  N);
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
                                       static_cast<uint32_t>(buf * C::BN + col0);
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
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(map_to_cta(acce0 + 8 * buf, 0));
            }
            if (!ok) break;
            if (w.slot >= 0) {
                // a K share of a tail tile: the raw 256 x 256 sum, tile-local rows
                float* trow = tail_ws + static_cast<long long>(w.slot) * (2 * BM * C::BN) +
                              static_cast<long long>(static_cast<int>(rank) * BM + row) * C::BN;
#pragma unroll
                for (int j = 0; j < EPI_COLS; j += 4)
                    store4(trow, col0 + j, C::BN,
                           make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]), true, 1.0f,
                           0.0f, kStorePlain);
                continue;
            }
            // The variant that splits in shared memory keeps the per-thread
            // stores: its splitter warps are short of registers, and with the
            // TMA path compiled in it ran 5-10 % slower on deep K (2048 x
            // 512 x 8192: 0.111 against 0.101 ms) though few of its tiles
            // reach the epilogue.
            if (!SPLIT_IN_KERNEL && tma_store) {
                ok = store_rows_tma(acc, epi0 + static_cast<uint32_t>(e) * 2 * EPI_SLAB_BYTES,
                                    stores, loads, cload0 + 8 * e, lane, &tmC, w.n0 + col0,
                                    w.m0 + static_cast<int>(rank) * BM + 32 * q, M, N, alpha,
                                    beta, scale_mode, timeout_ns, fault, abort_flag);
                continue;
            }
            const int m = w.m0 + static_cast<int>(rank) * BM + row;
            if (m < M) {
                float* orow = out + static_cast<long long>(w.split) * split_stride +
                              static_cast<long long>(m) * ldo;
                const int nb = w.n0 + col0;
#pragma unroll
                for (int j = 0; j < EPI_COLS; j += 4)
                    store4(orow, nb + j, N, make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]),
                           vec_store != 0, alpha, beta, scale_mode);
            }
        }
        // the output stores have completed (and no longer read the slabs)
        if (!SPLIT_IN_KERNEL && tma_store && lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // neither CTA may leave while its partner can still reach its shared memory
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

// Tail fix-up: C = sum of the tail_splits K shares of each tail tile, added
// in share order (deterministic), then scaled like any other output.
// One block per (tile, row), one thread per column.
__global__ void __launch_bounds__(256)
pair_tail_fixup_kernel(const float* __restrict__ tail_ws, int tiles_m, int tiles_n,
                       int tail_tiles, int tail_splits, float* __restrict__ C, long long ldc, int M,
                       int N, float alpha, float beta, int mode) {
    pdl_wait();  // the shares written by the GEMM kernel before it
    constexpr int TM = 2 * BM, TN = PairCfg<3>::BN;
    const int t = blockIdx.x;
    const int i = blockIdx.y;
    const int j = threadIdx.x;
    const Unit w = decode(tiles_m * tiles_n - tail_tiles + t, tiles_m, tiles_n, 1, 1, TN, TM);
    const int m = w.m0 + i, n = w.n0 + j;
    if (m >= M || n >= N) return;
    const float* src = tail_ws + static_cast<long long>(t) * tail_splits * TM * TN +
                       static_cast<long long>(i) * TN + j;
    float sum = src[0];
    for (int p = 1; p < tail_splits; ++p) sum += src[static_cast<long long>(p) * TM * TN];
    float* dst = C + static_cast<long long>(m) * ldc + n;
    *dst = scale1(sum, dst, alpha, beta, mode);
}

// Co-resident clusters of the pair kernel on this device (cached per device).
cudaError_t pair_clusters(int sm_count, int* out) {
    using C = PairCfg<3>;
    static thread_local int done_dev = -1;
    static thread_local int clusters = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (done_dev != dev) {
        auto kern = sgemm_3xtf32_pair_kernel<3, false>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
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
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        clusters = n;
        done_dev = dev;
    }
    *out = clusters;
    return cudaSuccess;
}

template <int STAGES, bool SPLIT_IN_KERNEL>
cudaError_t launch_pair(const Tf32x3Args& a, cudaStream_t s, int sm_count) {
    using C = PairCfg<STAGES, SPLIT_IN_KERNEL>;
    static_assert(C::SMEM_BYTES == PairCfg<3>::SMEM_BYTES && C::THREADS == PairCfg<3>::THREADS,
                  "both pair kernels have the occupancy pair_clusters measures");
    auto kern = sgemm_3xtf32_pair_kernel<STAGES, SPLIT_IN_KERNEL>;
    int max_clusters = 0;
    cudaError_t e = pair_clusters(sm_count, &max_clusters);
    if (e != cudaSuccess) return e;
    static thread_local int attr_done_dev = -1;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (attr_done_dev != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done_dev = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const int tiles_m = (a.M + 2 * BM - 1) / (2 * BM);
    const int tiles_n = (a.N + C::BN - 1) / C::BN;
    const int units = a.tail_tiles
                          ? tiles_m * tiles_n - a.tail_tiles + a.tail_tiles * a.tail_splits
                          : tiles_m * tiles_n * a.splits;
    const int clusters = units < max_clusters ? units : max_clusters;
    cfg.gridDim = dim3(2 * clusters);
    e = cudaLaunchKernelEx(&cfg, kern, a.tmAhi, a.tmAlo, a.tmBhi, a.tmBlo, a.out, a.ldo,
                           a.split_stride, a.M, a.N, a.K, a.kb_per_split, a.splits, a.vec_store,
                           a.fault, a.timeout_ns, a.alpha, a.beta, a.scale_mode, a.tail_tiles,
                           a.tail_splits, a.tail_ws, a.tmC, a.tma_store);
    if (e != cudaSuccess) return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.tail_tiles) e = launch_pair_tail_fixup(a, s);
    return e;
}

}  // namespace

// The tail fix-up of a 256 x 256 pair kernel's K-split last round (either
// pair kernel: both write the shares as tile-local 256 x 256 raw sums).
cudaError_t launch_pair_tail_fixup(const Tf32x3Args& a, cudaStream_t s) {
    constexpr int TM = 2 * BM, TN = PairCfg<3>::BN;
    const int tiles_m = (a.M + TM - 1) / TM;
    const int tiles_n = (a.N + TN - 1) / TN;
    cudaLaunchConfig_t fc = {};
    cudaLaunchAttribute fattr[1] = {pdl_attribute()};
    fc.gridDim = dim3(static_cast<unsigned>(a.tail_tiles), TM);
    fc.blockDim = dim3(TN);
    fc.stream = s;
    fc.attrs = fattr;
    fc.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&fc, pair_tail_fixup_kernel,
                                       static_cast<const float*>(a.tail_ws), tiles_m, tiles_n,
                                       a.tail_tiles, a.tail_splits, a.out, a.ldo, a.M, a.N,
                                       a.alpha, a.beta, a.scale_mode);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t tf32x3_pair_clusters(int sm_count, int* clusters) {
    return pair_clusters(sm_count, clusters);
}

Tf32x3Config tf32x3_config(int bn, bool pair) {
    if (pair) return {2 * BM, 256, BK, 3, PairCfg<3>::THREADS, PairCfg<3>::SMEM_BYTES, 1, 128};
    if (bn == 128) return {BM, 128, BK, 3, Cfg<128, 3>::THREADS, Cfg<128, 3>::SMEM_BYTES, 0, 128};
    return {BM, 256, BK, 2, Cfg<256, 2>::THREADS, Cfg<256, 2>::SMEM_BYTES, 0, 256};
}

namespace {
// Co-resident clusters of `splits` CTAs of the single-CTA kernel (one CTA per
// SM by its shared memory), from the occupancy calculator, cached per device.
template <int BN, int STAGES>
cudaError_t single_cluster_capacity(int splits, int* clusters) {
    using C = Cfg<BN, STAGES>;
    static thread_local int cached_dev = -1;
    static thread_local int cap[kMaxClusterSplits + 1] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (cached_dev != dev) {
        auto kern = sgemm_3xtf32_kernel<BN, STAGES>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        for (int sz = 1; sz <= kMaxClusterSplits; ++sz) {
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
}  // namespace

cudaError_t tf32x3_single_cluster_capacity(int bn, int splits, int* clusters) {
    if (splits < 1 || splits > kMaxClusterSplits) return cudaErrorInvalidValue;
    return bn == 128 ? single_cluster_capacity<128, 3>(splits, clusters)
                     : single_cluster_capacity<256, 2>(splits, clusters);
}

cudaError_t launch_sgemm_3xtf32(const Tf32x3Args& a, cudaStream_t s, int sm_count) {
    if (a.pair)
        return a.split_in_kernel ? launch_pair<3, true>(a, s, sm_count)
                                 : launch_pair<3, false>(a, s, sm_count);
    if (a.bn == 128)
        return a.split_in_kernel ? launch_impl<128, 3, true>(a, s, sm_count)
                                 : launch_impl<128, 3>(a, s, sm_count);
    return launch_impl<256, 2>(a, s, sm_count);
}

}  // namespace gemm_f32_impl
