// tf32x3_common.cuh -- pieces shared by the 3xTF32 tensor-core kernels:
// tile and pipeline constants, the persistent work-unit order, the bounded
// role waits with a CTA-wide abort flag, and the TF32 split of fp32 values
// (the high part is the fp32 word itself, which the tensor core reads
// truncated; the low part is tf32(x - trunc(x)), rounded to nearest even).
#pragma once

#include <cstdint>

#include "device_sync.cuh"

namespace gemm_f32_impl {
namespace {

using namespace gemm_f32_dev;

constexpr int BM = 128;
constexpr int BK = 32;      // one 128-byte swizzle row of tf32
constexpr int UMMA_K = 8;   // K of one kind::tf32 MMA
constexpr int CH = 4;       // K blocks per tensor-core chunk (128-deep K)
constexpr int EPI_COLS = 128;  // accumulator columns per epilogue thread
constexpr int GROUP_M = 8;
// K blocks between an L2 prefetch and the load of the same boxes, in the
// pair kernel that splits in shared memory: its stages wait on DRAM (it reads
// each operand once), and prefetching two blocks ahead took 256 x 256 x 65536
// from 88.7 to 84.5 us.  The kernels on pre-split operands run slower with
// prefetching (8192^3: 3.85 against 4.42 ms), so they do not prefetch.
constexpr int kPrefetchAhead = 2;

struct Unit {
    int m0, n0, split, kb_begin, nkb;
    int slot;  // >= 0: a K share of a tail tile, written raw to the tail workspace
};

// Work unit u: split u / tiles of tile u % tiles (split-major), or, when the
// splits of a tile form one cluster (cluster_splits = S > 0), split u % S of
// tile u / S (tile-major, so that a cluster's CTAs share a tile).
__device__ __forceinline__ Unit decode(int u, int tiles_m, int tiles_n, int kb_per_split,
                                       int kb_total, int bn, int bm = BM, int cluster_splits = 0) {
    const int tiles = tiles_m * tiles_n;
    Unit w;
    w.split = cluster_splits ? u % cluster_splits : u / tiles;
    const int t = cluster_splits ? u / cluster_splits : u - w.split * tiles;
    const int per_group = GROUP_M * tiles_n;
    const int group = t / per_group;
    const int first_m = group * GROUP_M;
    const int rows_in_group = min(tiles_m - first_m, GROUP_M);
    const int within = t - group * per_group;
    w.m0 = (first_m + within % rows_in_group) * bm;
    w.n0 = (within / rows_in_group) * bn;
    w.kb_begin = w.split * kb_per_split;
    w.nkb = max(0, min(kb_total, w.kb_begin + kb_per_split) - w.kb_begin);
    w.slot = -1;
    return w;
}


__device__ __forceinline__ uint32_t ld_shared_volatile(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_volatile(uint32_t addr, uint32_t v) {
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Bounded wait that also gives up when another role has aborted (the abort
// word is a shared-memory flag any role sets when one of its waits times out).
// CLUSTER: acquire at cluster scope (the other CTA of the pair arrives after
// writing shared memory that this CTA's MMAs read).
template <bool CLUSTER>
__device__ __forceinline__ bool try_wait_scoped(uint32_t bar, uint32_t parity) {
    return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
}
template <bool CLUSTER>
__device__ __forceinline__ bool role_wait_slow(uint32_t bar, uint32_t parity, long long timeout_ns,
                                            unsigned* fault, unsigned bit, uint32_t abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (try_wait_scoped<CLUSTER>(bar, parity)) return true;
        if (ld_shared_volatile(abort_flag)) return false;
        if (globaltimer_ns() - t0 > static_cast<uint64_t>(timeout_ns)) {
            if (fault) atomicOr(fault, bit);
            st_shared_volatile(abort_flag, 1u);
            return false;
        }
    }
}
template <bool CLUSTER = false>
__device__ __forceinline__ bool role_wait(uint32_t bar, uint32_t parity, long long timeout_ns,
                                          unsigned* fault, unsigned bit, uint32_t abort_flag) {
    if (try_wait_scoped<CLUSTER>(bar, parity)) return true;
    return role_wait_slow<CLUSTER>(bar, parity, timeout_ns, fault, bit, abort_flag);
}

// Round to TF32 (nearest, ties to even), for the low part of the split.  The
// ties-to-even form is a single native conversion; the ties-away form
// (cvt.rna) made the in-kernel split a fifth slower (4096^3: 0.996 against
// 0.799 ms) and gives no better split.
__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rn.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

__device__ __forceinline__ float4 tf32x4(float4 x) {
    return make_float4(to_tf32(x.x), to_tf32(x.y), to_tf32(x.z), to_tf32(x.w));
}

__device__ __forceinline__ float4 sub4(float4 a, float4 b) {
    return make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w);
}

// x with the low 13 mantissa bits of each lane cleared: the TF32 value the
// tensor core reads from the fp32 word x (it truncates; measured on this
// part for ties and near-ties of both parities and signs).
__device__ __forceinline__ float4 trunc4(float4 x) {
    return make_float4(__uint_as_float(__float_as_uint(x.x) & 0xFFFFE000u),
                       __uint_as_float(__float_as_uint(x.y) & 0xFFFFE000u),
                       __uint_as_float(__float_as_uint(x.z) & 0xFFFFE000u),
                       __uint_as_float(__float_as_uint(x.w) & 0xFFFFE000u));
}

// The low part of the TF32 split of four values, lo = tf32(x - trunc(x));
// the high part is the word x itself (the split of tf32_split.cu).
__device__ __forceinline__ float4 lo4(float4 x) { return tf32x4(sub4(x, trunc4(x))); }

__device__ __forceinline__ float lane_of(float4 v, int e) {
    return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// Rotate the four lanes of v left by r (0..3): result.x = v[r], .y = v[r + 1], ...
__device__ __forceinline__ float4 rotate4(float4 v, int r) {
    const float4 a = (r & 1) ? make_float4(v.y, v.z, v.w, v.x) : v;
    return (r & 2) ? make_float4(a.z, a.w, a.x, a.y) : a;
}

// A slot (16 KB at sa, K-major, 128-byte swizzled as the TMA wrote it): each
// value x stays where it is as its own high part, and lo = tf32(x -
// trunc(x)) goes 16 KB further on.  The map is elementwise, so the layout
// carries over.  Call t takes 16-byte words t, t + 64, ... (t = 0..63: two
// calls by the 32 lanes of one warp, t = lane and lane + 32; conflict-free).
__device__ __forceinline__ void split_a_stage(uint32_t sa, int t) {
#pragma unroll 1
    for (int i0 = 0; i0 < 16; i0 += 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = lds128(sa + 16 * t + 1024 * (i0 + j));
#pragma unroll
        for (int j = 0; j < 8; ++j)
            sts128(sa + 16 * t + 1024 * (i0 + j) + 16384, lo4(v[j]));
    }
}

// Work units of the pair kernel.  Without a tail (tail_tiles == 0) they are
// (tile, split) pairs as above.  With one, the last tail_tiles tiles of the
// raster (what would otherwise be a partly idle last round of the persistent
// grid) are each cut into tail_splits K ranges: unit full + t is share
// t % tail_splits of tile full + t / tail_splits, and its raw sum goes to
// slot t of the tail workspace, to be added up by the fix-up kernel.
__device__ __forceinline__ Unit decode_pair(int u, int tiles_m, int tiles_n, int kb_per_split,
                                            int kb_total, int bn, int tail_tiles,
                                            int tail_splits) {
    const int full = tiles_m * tiles_n - tail_tiles;
    if (tail_tiles == 0 || u < full) return decode(u, tiles_m, tiles_n, kb_per_split, kb_total, bn, 2 * BM);
    const int t = u - full;
    Unit w = decode(full + t / tail_splits, tiles_m, tiles_n, kb_total, kb_total, bn, 2 * BM);
    const int per = (kb_total + tail_splits - 1) / tail_splits;
    w.kb_begin = (t % tail_splits) * per;
    w.nkb = max(0, min(kb_total, w.kb_begin + per) - w.kb_begin);
    w.slot = t;
    return w;
}

}  // namespace
}  // namespace gemm_f32_impl
