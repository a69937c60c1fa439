// gemm_f32_api.cu -- the C ABI of libgemmf32.so: argument validation, the
// edge rules, algorithm and split-K planning, operand staging, TMA
// descriptor encoding, workspace management and kernel dispatch.
//
// Edge rules follow "Lecture 12: final project" (section 7, the early exits
// of main): negative sizes are an error, M == 0 or N == 0 is a successful
// no-op, and K == 0 yields C = 0.  Unlike the page's CUDA_CHECK, nothing here
// exits the process: every failure is a status code.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "gemm_f32.h"
#include "gemm_internal.h"

using namespace gemm_f32_impl;

namespace {

constexpr int kMaxDevices = 64;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    unsigned* fault = nullptr;  // device fault word (256-byte allocation)
};

struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
    // a call captured into a CUDA graph used ptr: the graph keeps the
    // pointer, so a grown workspace retires the old buffer (freed by
    // gemm_f32_release) instead of freeing it
    bool captured = false;
    std::vector<void*> retired;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
EncodeTiledFn g_encode = nullptr;

// A host-side failure armed by gemm_f32_inject_host_fault (0: none), taken
// by the first site of its kind that runs.
std::atomic<int> g_inject{GEMM_F32_INJECT_NONE};

bool injected(int kind) {
    int want = kind;
    return g_inject.load(std::memory_order_relaxed) == kind &&
           g_inject.compare_exchange_strong(want, GEMM_F32_INJECT_NONE);
}

long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

bool misaligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes) {
    if (!a || !b || abytes == 0 || bbytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// Device lookup; g_mutex must be held.
// True if `stream` is being captured into a CUDA graph (or cannot be asked).
bool stream_capturing(cudaStream_t stream) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return cs != cudaStreamCaptureStatusNone;
}

// The device's state, set up on first use.  `capture_stream`: the stream of
// the call, which must not be capturing a graph while the set-up (allocation
// and zeroing of the fault word) runs.
int device_state(DeviceState** out, int* dev_out, const cudaStream_t* capture_stream = nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        if (capture_stream && stream_capturing(*capture_stream)) return GEMM_F32_ERR_CAPTURE;
        if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess) {
            cudaGetLastError();
            return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
        }
        if (d.cc_major != 10 || d.cc_minor != 3) return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
        void* f = nullptr;
        cudaError_t e = cudaMalloc(&f, 256);
        if (e != cudaSuccess) return GEMM_F32_ERR_WORKSPACE;
        e = cudaMemset(f, 0, 256);
        if (e != cudaSuccess) return static_cast<int>(e);
        d.fault = static_cast<unsigned*>(f);
        d.ready = true;
    }
    *out = &d;
    *dev_out = dev;
    return GEMM_F32_SUCCESS;
}

int get_encoder() {
    if (g_encode) return GEMM_F32_SUCCESS;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return GEMM_F32_ERR_DESCRIPTOR;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    return GEMM_F32_SUCCESS;
}

// 2-D fp32 tensor map over a row-major matrix: dim0 (contiguous) x dim1 rows
// with a row stride of ld elements.
int encode_2d(CUtensorMap* map, const float* base, long long dim0, long long dim1, long long ld,
              int box0, int box1, CUtensorMapSwizzle swizzle) {
    if (injected(GEMM_F32_INJECT_DESCRIPTOR)) return GEMM_F32_ERR_DESCRIPTOR;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(dim0), static_cast<cuuint64_t>(dim1)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4u};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box0), static_cast<cuuint32_t>(box1)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_F32_SUCCESS : GEMM_F32_ERR_DESCRIPTOR;
}

// Workspace of at least `bytes` for (dev, stream); g_mutex must be held.
int workspace(int dev, cudaStream_t stream, size_t bytes, void** out) {
    Workspace& w = g_ws[std::make_pair(dev, stream)];
    const bool capturing = stream_capturing(stream);
    if (w.bytes < bytes) {
        // growing synchronises the stream and allocates: not while capturing
        if (capturing) return GEMM_F32_ERR_CAPTURE;
        if (w.ptr) {
            // earlier calls on this stream may still read the old buffer
            cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return static_cast<int>(e);
            if (w.captured)
                w.retired.push_back(w.ptr);
            else
                cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
            w.captured = false;
        }
        const size_t grow = static_cast<size_t>(round_up(static_cast<long long>(bytes), 1 << 20));
        if (injected(GEMM_F32_INJECT_WORKSPACE) || cudaMalloc(&w.ptr, grow) != cudaSuccess) {
            cudaGetLastError();
            w.ptr = nullptr;
            return GEMM_F32_ERR_WORKSPACE;
        }
        // the in-kernel split-K counters start at zero
        cudaError_t e = cudaMemsetAsync(w.ptr, 0, kWorkspaceCounterBytes, stream);
        if (e != cudaSuccess) {
            cudaFree(w.ptr);
            w.ptr = nullptr;
            return static_cast<int>(e);
        }
        w.bytes = grow;
    }
    if (capturing) w.captured = true;
    *out = w.ptr;
    return GEMM_F32_SUCCESS;
}

struct Plan {
    int algo = 0;
    int variant = 0;  // FFMA tile variant
    int bn = 0;
    int pair = 0;     // 3xTF32: two-CTA kernel
    int split_in_kernel = 0;  // 3xTF32 pair kernel: TF32 split done in shared memory
    int tmem_b = 0;           // 3xTF32: the 128 x 128 kernel with B's split in tensor memory
    int tmem_wide = 0;        // ... in its wide single-CTA form (256 x 128 tiles, N = 256 MMAs)
    int reduce_in_kernel = 0; // that kernel adds its split-K partials itself (one unit per CTA)
    int cluster_splits = 0;   // split-K partials added inside a cluster (FFMA 2..4, the
                              // single-CTA tensor-core kernels 2..8)
    int fused_staging = 0;    // 3xTF32 staged: A and B split by one launch
    int box_n = 0;    // 3xTF32: B^T rows per TMA box
    int tail_tiles = 0, tail_splits = 0;  // pair kernel: K-split last partial round
    int tail_m = 0, tail_n = 0;           // the output extent the tail split was planned for
    size_t off_t = 0;
    int splits = 1;
    int kb_per_split = 0;
    int stage_a = 0, stage_b = 0;
    long long lda = 0, ldb = 0;   // row strides of the operands the kernel reads (elements)
    // 3xTF32 staged: A is its own high part (read in place, row stride
    // lda_hi); only its low plane is written
    int a_in_place = 0;
    long long lda_hi = 0;
    long long ldw = 0;            // split-K partial row stride
    size_t off_a = 0, off_a2 = 0, off_b = 0, off_b2 = 0, off_w = 0, ws_bytes = 0;
    int tile_m = 0, tile_n = 0, tile_k = 0, stages = 0, ctas = 0, kernels = 0;
};

// One call's operands in the general row-major form C = alpha op(A) op(B) +
// beta C.  op(A) is M x K: A[i*lda + k], or A[k*lda + i] when ta; op(B) is
// K x N: B[k*ldb + j], or B[j*ldb + k] when tb; C[i*ldc + j].
struct Problem {
    int M = 0, N = 0, K = 0;
    const float* A = nullptr;
    long long lda = 0;
    int ta = 0;
    const float* B = nullptr;
    long long ldb = 0;
    int tb = 0;
    float* C = nullptr;
    long long ldc = 0;
    float alpha = 1.0f, beta = 0.0f;
};

Problem packed(const float* A, const float* B, float* C, int M, int N, int K) {
    Problem q;
    q.M = M;
    q.N = N;
    q.K = K;
    // packed strides; an empty dimension still has a stride of at least 1
    q.A = A;
    q.lda = K > 1 ? K : 1;
    q.B = B;
    q.ldb = N > 1 ? N : 1;
    q.C = C;
    q.ldc = N > 1 ? N : 1;
    return q;
}

// epilogue mode: plain store, alpha scale, or alpha and beta (reads C)
int scale_mode(const Problem& q) {
    if (q.beta != 0.0f) return 2;
    return q.alpha == 1.0f ? 0 : 1;
}

int validate(const Problem& q, int algo, int splits, bool need_ptrs = true) {
    const int M = q.M, N = q.N, K = q.K;
    if (M < 0 || N < 0 || K < 0) return GEMM_F32_ERR_INVALID_VALUE;
    if (algo < GEMM_F32_ALGO_AUTO || algo > GEMM_F32_ALGO_3XTF32) return GEMM_F32_ERR_INVALID_VALUE;
    if (splits < 0 || splits > GEMM_F32_MAX_SPLITS) return GEMM_F32_ERR_INVALID_VALUE;
    if ((q.ta != 0 && q.ta != 1) || (q.tb != 0 && q.tb != 1)) return GEMM_F32_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return GEMM_F32_SUCCESS;  // empty output: nothing is looked at
    // stored shapes: A is (ta ? K x M : M x K), B is (tb ? N x K : K x N)
    const long long a_rows = q.ta ? K : M, a_cols = q.ta ? M : K;
    const long long b_rows = q.tb ? N : K, b_cols = q.tb ? K : N;
    if (q.lda < (a_cols > 1 ? a_cols : 1) || q.ldb < (b_cols > 1 ? b_cols : 1) ||
        q.ldc < (N > 1 ? N : 1))
        return GEMM_F32_ERR_INVALID_VALUE;
    const size_t a_bytes = (a_rows && a_cols) ? static_cast<size_t>((a_rows - 1) * q.lda + a_cols) * 4u : 0;
    const size_t b_bytes = (b_rows && b_cols) ? static_cast<size_t>((b_rows - 1) * q.ldb + b_cols) * 4u : 0;
    const size_t c_bytes = (M && N) ? static_cast<size_t>((static_cast<long long>(M) - 1) * q.ldc + N) * 4u : 0;
    if (M > 0 && N > 0) {
        if (need_ptrs && !q.C) return GEMM_F32_ERR_INVALID_VALUE;
        if (need_ptrs && K > 0 && (!q.A || !q.B)) return GEMM_F32_ERR_INVALID_VALUE;
        if (overlaps(q.C, c_bytes, q.A, a_bytes) || overlaps(q.C, c_bytes, q.B, b_bytes))
            return GEMM_F32_ERR_INVALID_VALUE;
        if ((reinterpret_cast<uintptr_t>(q.C) & 3u) ||
            (q.A && (reinterpret_cast<uintptr_t>(q.A) & 3u)) ||
            (q.B && (reinterpret_cast<uintptr_t>(q.B) & 3u)))
            return GEMM_F32_ERR_INVALID_VALUE;
    }
    return GEMM_F32_SUCCESS;
}

// Split-K factor: spread a grid that would fill less than half of the
// concurrent CTA slots over disjoint K ranges, keeping >= 4 K blocks each.
int choose_splits(int requested, int tiles, int kb_total, int slots, int min_kb = 4) {
    int s = requested;
    if (s == 0) {
        s = 1;
        if (tiles * 2 <= slots) {
            s = slots / tiles;
            const int max_by_depth = kb_total / min_kb;
            if (s > max_by_depth) s = max_by_depth;
            if (s > GEMM_F32_MAX_SPLITS) s = GEMM_F32_MAX_SPLITS;
            if (s < 1) s = 1;
        }
    }
    if (s > kb_total) s = kb_total;
    if (s < 1) s = 1;
    return s;
}

// The split-K factor the single-CTA tensor-core kernel gets for tiles of
// 128 x bn (see make_plan): choose_splits, capped at 4 (K <= 1024) or 8
// (K <= 4096) splits when the library chooses.  A factor of 2..8 with one
// unit per CTA adds its partials inside clusters, all of which must be
// co-resident: a library-chosen factor is lowered until the tiles' clusters
// fit on the device at once (101 x 5159 x 61036: 21 tiles of 128 x 256 in
// clusters of 7 ran in two waves, only 15 such clusters fitting).
int single_cta_splits(int sm_count, int tiles, int K, int splits, int bn) {
    const int kb_total = (K + 31) / 32;
    int s = choose_splits(splits, tiles, kb_total, sm_count, 4);
    if (splits == 0 && K <= 4096) {
        const int cap = K <= 1024 ? 4 : 8;
        if (s > cap) s = cap;
    }
    if (splits == 0) {
        while (s >= 2 && s <= 8 && static_cast<long long>(tiles) * s <= sm_count) {
            int fit = 0;
            if (tf32x3_single_cluster_capacity(bn, s, &fit) != cudaSuccess) {
                cudaGetLastError();
                break;
            }
            if (tiles <= fit) break;
            --s;
        }
    }
    return s;
}

// The fraction of the SMs' round capacity that 128 x bn tiles with their
// split-K factor keep busy, divided by the padding of N to whole tiles.
double single_cta_fill(int sm_count, int M, int N, int K, int bn, int splits) {
    const int tiles_n = (N + bn - 1) / bn;
    const int tiles = ((M + 127) / 128) * tiles_n;
    const long long units =
        static_cast<long long>(tiles) * single_cta_splits(sm_count, tiles, K, splits, bn);
    const long long rounds = (units + sm_count - 1) / sm_count;
    const double busy = static_cast<double>(units) / (static_cast<double>(rounds) * sm_count);
    return busy * N / (static_cast<double>(tiles_n) * bn);
}

// Whether cutting the R tiles of the pair kernels' last round into T K
// shares pays: the round's time falls by (1 - 1/T) of a unit (~0.029 us a
// unit of K for a 256 x 256 tile), the fix-up kernel costs a ~4 us launch
// plus reading the T shares and writing the R tiles ((T + 1) R 256^2 floats
// at ~3 TB/s).
bool tail_split_pays(int K, int r, int t) {
    const double saving = (1.0 - 1.0 / t) * K * 0.029;
    const double cost = 4.0 + (t + 1.0) * r * 256.0 * 256.0 * 4.0 / 3.0e6;
    return saving > cost;
}

// Modelled time of the kernels with B's split in tensor memory: rounds of
// the persistent grid (slots: CTAs, or clusters of the pair form) x K blocks
// per unit x the time of one K block, plus a fixed cost (launch, pipeline
// fill, last epilogue) and, for S > 1, the partials' cost: ~3 us and their
// traffic, S M N floats written and read back and M N written, at ~5 TB/s
// (1536^2 x 4096 with 2 pair splits: 76 us; 1024^2 x 8192 with 4: 76 us,
// with 9 in two rounds: 85).  Fitted on the boundary sweep: one K block of
// a 128 x 128 unit ~0.57 us, fixed ~12 us (4096 x 512 x 8192: one round of
// 256 blocks, 154.3 us; 1536^2 x 4096: one round of 128, 84.6 us); of a
// 256 x 256 pair unit ~0.92 us, fixed ~12 us (2048^2 x 8192: 242 us;
// 8192^3: 13.5 rounds of 256, 3.14 ms).  The
// pair form's tail split counts, with its fix-up: 2048 x 8192 x 8192 (256
// tiles on 76 clusters) keeps S = 1, 3.5 rounds of 256 blocks, rather than
// S = 2 and a reduction.  Returns the modelled us and the S that minimises
// it (1280^2 x 8192 on 128 x 128 tiles: 100 tiles, S = 3, two rounds of 86
// blocks, over S = 1, one round of 256 with 52 SMs idle; 256 x 256 x 65536:
// 4 tiles, S = 38).
struct TmemModel {
    double us_per_block;
    double fixed_us;
    bool tail_split;        // the pair form's K-split last round
    double reduce_wait_us;  // extra per split for a reduction inside the kernel
    bool one_round;         // only plans whose units all run at once
};
// The pair's in-kernel reduction (16 splits or more, one unit per cluster)
// measured ~70 ns a split above the model: 256 x 256 x 65536 with 76 splits
// 52-54 us against 48 modelled (the single-CTA form with 38: 50 against
// 50), 512^2 x 16384 with 19 splits 47.8 against 48
constexpr TmemModel kTmemSingle = {0.57, 12.0, false, 0.0, false};
constexpr TmemModel kTmemPair = {0.92, 12.0, true, 0.07, false};
// The wide single-CTA form: a 16-deep K block of a 256 x 128 unit ~0.455 us
// (2048^3: one round of 128 blocks, 70.3 us), as fast per SM as the pair in
// one round of its grid (and ~4 % faster with 16 or more splits added in
// the kernel: 256 x 256 x 65536, 512^2 x 16384).  Over several rounds, and
// on padded copies of the operands, it ran 10-25 % behind the pair (4096^3
// 490 against 431 us, 2560^3 136 against 124, 961 x 6697 x 8131 810
// against 650): a unit loads 1.5 times the pair's operand bytes per output,
// so AUTO takes it only for operands read in place and one round of units.
constexpr TmemModel kTmemWide = {0.455, 12.0, false, 0.0, true};

double tmem_estimate(int slots, int tiles, int kb_total, int M, int N, const TmemModel& mdl,
                     int forced_splits, int* splits_out) {
    constexpr double kReduceLaunchUs = 3.0, kReduceBytesPerUs = 5.0e6;
    int best = 1;
    double best_us = 0.0;
    bool found = false;
    const int s_max = std::min(GEMM_F32_MAX_SPLITS, std::max(1, kb_total / 4));
    const int s_lo = forced_splits > 0 ? std::min(forced_splits, std::max(kb_total, 1)) : 1;
    const int s_hi = forced_splits > 0 ? s_lo : s_max;
    for (int s = s_lo; s <= s_hi; ++s) {
        const int per = (kb_total + s - 1) / s;
        const int eff = (kb_total + per - 1) / per;  // splits that get work
        if (eff != s && forced_splits <= 0) continue;
        const long long units = static_cast<long long>(tiles) * s;
        if (mdl.one_round && units > slots) continue;
        double rounds = static_cast<double>((units + slots - 1) / slots);
        // without split-K the pair form cuts a partly idle last round into
        // T K shares (see make_plan): that round then takes 1 / T
        const int r = tiles % slots;
        const int t = r ? std::min(slots / r, 4) : 0;
        const bool tail = s == 1 && mdl.tail_split && tiles > slots && t >= 2 &&
                          kb_total >= 2 * t && tail_split_pays(kb_total * 32, r, t);
        if (tail) rounds = static_cast<double>(tiles / slots) + 1.0 / t;
        double us = rounds * per * mdl.us_per_block + mdl.fixed_us;
        if (tail) us += 4.0 + (t + 1.0) * r * 256.0 * 256.0 * 4.0 / 3.0e6;
        if (s > 1)
            us += kReduceLaunchUs +
                  (2.0 * s + 1.0) * M * static_cast<double>(N) * 4.0 / kReduceBytesPerUs;
        if (s >= 16 && units <= slots) us += mdl.reduce_wait_us * s;
        if (!found || us < best_us) {
            best = s;
            best_us = us;
            found = true;
        }
    }
    if (splits_out) *splits_out = best;
    return found ? best_us : 1e30;
}

size_t carve(size_t* off, long long bytes) {
    const size_t at = *off;
    *off += static_cast<size_t>(round_up(bytes, 256));
    return at;
}

void make_plan(const DeviceState& d, const Problem& q, int algo, int splits, Plan* p,
               int tile = GEMM_F32_TILE_AUTO) {
    const int M = q.M, N = q.N, K = q.K;
    // AUTO: the tensor-core kernel, except for tiny problems (under 5e7
    // multiply-adds, e.g. 256^3: 17.1 against 25.2 us), where the CUDA-core
    // kernel's single launch beats the staging launch plus GEMM of the
    // tensor-core path.  From 512^3 on the tensor-core path is ahead (512^3:
    // 18.0 us with 4 splits added in a cluster, against 19.1 us)
    const double macs = static_cast<double>(M) * N * K;
    p->algo = algo != GEMM_F32_ALGO_AUTO ? algo
              : macs < 5e7               ? GEMM_F32_ALGO_FFMA
                                         : GEMM_F32_ALGO_3XTF32;
    int bm, bn, bk, slots;
    if (p->algo == GEMM_F32_ALGO_3XTF32) {
        // the two-CTA 256 x 256 kernel when its tiles fill at least four
        // fifths of the SM pairs (it keeps the tensor pipe busier than one
        // CTA per tile: 2048^2 x 8192, 64 pair tiles on 76 pairs, 309 against
        // 330 us for 128 x 256; 2048^3 even) and K is at least 1024 (with a
        // few K blocks per tile the fill and the 256 x 256 epilogue of each
        // tile dominate: 2378 x 4792 x 286, 74 against 49 us for 128 x 128);
        // otherwise one CTA per 128 x 256 tile when those fill at least three
        // quarters of the SMs, else 128 x 128 tiles with split-K
        const int units_pair = ((M + 255) / 256) * ((N + 255) / 256);
        const int tiles256 = ((M + 127) / 128) * ((N + 255) / 256);
        p->pair = (5 * units_pair >= 4 * (d.sm_count / 2) && K >= 1024) ? 1 : 0;
        if (!p->pair && K >= 1024) {
            // ... or when its tiles, net of padding, keep at least as much of
            // the machine busy as 128 x 128 tiles with their split-K factor
            // (1792^2 x 4096: 49 pair tiles and 196 single tiles both fill 64
            // %; 162.5 against 172.7 us)
            const int pairs = d.sm_count / 2;
            const int rounds = (units_pair + pairs - 1) / pairs;
            const double pad = static_cast<double>(M) * N /
                               (static_cast<double>(round_up(M, 256)) * round_up(N, 256));
            const double pair_fill = static_cast<double>(units_pair) / (rounds * pairs) * pad;
            if (pair_fill >= single_cta_fill(d.sm_count, M, N, K, 128, splits)) p->pair = 1;
        }
        p->bn = (p->pair || (4 * tiles256 >= 3 * d.sm_count && N > 128)) ? 256 : 128;
        if (!p->pair) {
            // ... unless the other single-CTA width keeps clearly more of the
            // SMs busy (its tiles x K splits per round, net of padding in N):
            // 5170 x 151 x 5906, 82 tiles of 128 x 128 leave 46 % of the SMs
            // idle where 41 of 128 x 256 in 3 in-cluster splits fill 81 %
            // (162 against 214 us).  The 128 x 256 kernel's 2-stage ring runs
            // a unit of given work ~15 % slower than the 3-stage 128 x 128
            // one, so its fill counts 0.85 (896^2 x 4096: 5 splits of 128 x
            // 256, 87 us, against 3 of 128 x 128, 75 us)
            const double u128 = single_cta_fill(d.sm_count, M, N, K, 128, splits);
            const double u256 = 0.85 * single_cta_fill(d.sm_count, M, N, K, 256, splits);
            // With deep K (>= 8192, and each 128 x 256 unit at least 2048 of
            // it) the 128 x 256 kernel, whose tiles read less shared memory
            // per flop, unless 128 x 128 tiles keep 3 % more of the SMs busy
            // (unweighted fills): 177 x 4459 x 16098 361 against 397 us,
            // 1500 x 2079 x 21955 1087 against 1272 us, 272 x 6979 x 37601
            // 2139 against 2396 us.  Shorter units pay the 2-stage ring's
            // fill too often: 640^2 x 8192, 10 splits of 819, 73 against 61
            // us for 128 x 128 tiles.
            const int tiles_256 = ((M + 127) / 128) * ((N + 255) / 256);
            const int s256 = single_cta_splits(d.sm_count, tiles_256, K, splits, 256);
            if (K >= 8192 && K / s256 >= 2048)
                p->bn = (u128 > 1.03 * (u256 / 0.85)) ? 128 : 256;
            else if (u256 > 1.1 * u128) p->bn = 256;
            else if (u128 > 1.1 * u256) p->bn = 128;
        }
        // A and B read as stored (K-contiguous A and N-contiguous B rows,
        // 16-byte row strides and bases): the kernels with B's split in
        // tensor memory, which need no staging pass and no transpose in
        // shared memory.  They beat the staged kernels on every such shape
        // of the boundary sweep (256 x 256 x 65536 51.9 against 66.2 us,
        // 896^2 x 4096 39.6 against 58.0, 2048^3 76 against 89, 8192^3 3.18
        // against 3.53 ms), and the kernels that split A and B in shared
        // memory (now forced configurations only) on every shape those were
        // chosen for (89 x 1216 x 24336 47.7 against 74.4 us).  Row-major
        // operands that need padded copies (a row stride or base off 16
        // bytes) take them too: with the copies at HBM rate the pair or
        // single-CTA form after them beat the staged kernels on 24 of the 29
        // such random shapes and trailed by at most 10 % on the others, all
        // calls of ~20 us (5170 x 151 x 5906 126 against 166 us, 1184 x 988
        // x 30671 321 against 490, 301 x 1874 x 563 25 against 23).
        // Transposed operands do once C has 3M elements (their transposed
        // copy against the staged kernels' split-and-transpose pass).  The
        // CTA-pair form (256 x 256 tiles, N = 256 MMAs) or the single-CTA
        // one, whichever the model times shorter with its own split-K
        // factor: 1536^2 x 8192 pair with 2 splits 136 against 164.5 us for
        // one round of 128 x 128 tiles; 512^2 x 4096 single with 9 splits
        // 25 against 27 us.
        const bool in_place = !q.ta && !q.tb && q.lda % 4 == 0 && q.ldb % 4 == 0 &&
                              !misaligned16(q.A) && !misaligned16(q.B);
        if (in_place || (!q.ta && !q.tb) || static_cast<double>(M) * N >= 3.0e6) {
            int clusters = 0;
            const bool have_pair =
                tf32x3_tmem_pair_clusters(d.sm_count, &clusters) == cudaSuccess && clusters > 0;
            cudaGetLastError();
            const int kb = (K + tf32x3_tmem_config(false).bk - 1) / tf32x3_tmem_config(false).bk;
            const int kbw = (K + tf32x3_tmem_wide_config().bk - 1) / tf32x3_tmem_wide_config().bk;
            const int t128 = ((M + 127) / 128) * ((N + 127) / 128);
            const int t256 = ((M + 255) / 256) * ((N + 255) / 256);
            const int twide = ((M + 255) / 256) * ((N + 127) / 128);
            const double us1 = tmem_estimate(d.sm_count, t128, kb, M, N, kTmemSingle, splits,
                                             nullptr);
            const double us2 =
                have_pair ? tmem_estimate(clusters, t256, kb, M, N, kTmemPair, splits, nullptr)
                          : us1 + 1.0;
            const double us3 =
                in_place ? tmem_estimate(d.sm_count, twide, kbw, M, N, kTmemWide, splits, nullptr)
                         : 1e30;
            p->tmem_b = 1;
            p->pair = us2 < us1 && us2 <= us3 ? 1 : 0;
            p->tmem_wide = !p->pair && us3 < us1 ? 1 : 0;
            p->split_in_kernel = 1;
            p->bn = p->pair ? 256 : 128;
        }
        if (tile != GEMM_F32_TILE_AUTO) {
            p->pair = tile == GEMM_F32_TILE_256x256_PAIR ||
                      tile == GEMM_F32_TILE_256x256_PAIR_SPLIT || tile == GEMM_F32_TILE_256x256_TMEM;
            p->tmem_b = tile == GEMM_F32_TILE_128x128_TMEM || tile == GEMM_F32_TILE_256x256_TMEM ||
                        tile == GEMM_F32_TILE_256x128_TMEM;
            p->tmem_wide = tile == GEMM_F32_TILE_256x128_TMEM;
            p->split_in_kernel = tile == GEMM_F32_TILE_256x256_PAIR_SPLIT ||
                                 tile == GEMM_F32_TILE_128x128_SPLIT || p->tmem_b;
            p->bn = (tile == GEMM_F32_TILE_128x128 || tile == GEMM_F32_TILE_128x128_SPLIT ||
                     tile == GEMM_F32_TILE_128x128_TMEM || tile == GEMM_F32_TILE_256x128_TMEM)
                        ? 128
                        : 256;
        }
        const Tf32x3Config tc = p->tmem_wide ? tf32x3_tmem_wide_config()
                                : p->tmem_b  ? tf32x3_tmem_config(p->pair != 0)
                                          : tf32x3_config(p->bn, p->pair != 0);
        bm = tc.bm;
        bn = tc.bn;
        bk = tc.bk;
        p->stages = tc.stages;
        p->box_n = tc.box_n;
        slots = p->pair ? d.sm_count / 2 : d.sm_count;
    } else {
        // wide tiles (8 x 16 per thread) once they fill four fifths of the
        // SMs, else 128 x 128 (2048^3: 128 wide tiles on 152 SMs 0.330 ms,
        // 256 narrow ones at two CTAs an SM 0.371 ms)
        const int tiles_wide = ((M + 127) / 128) * ((N + 255) / 256);
        p->variant = 5 * tiles_wide >= 4 * d.sm_count ? 1 : 0;
        if (tile != GEMM_F32_TILE_AUTO) p->variant = tile == GEMM_F32_TILE_128x256 ? 1 : 0;
        const FfmaConfig fc = ffma_config(p->variant);
        bm = fc.bm;
        bn = fc.bn;
        bk = fc.bk;
        p->bn = bn;
        p->stages = fc.stages;
        slots = d.sm_count * fc.ctas_per_sm;
    }
    p->tile_m = bm;
    p->tile_n = bn;
    p->tile_k = bk;
    const int tiles = ((M + bm - 1) / bm) * ((N + bn - 1) / bn);
    const int kb_total = (K + bk - 1) / bk;
    // the CUDA-core kernel keeps >= 2 K blocks a split (512^3: 8 splits,
    // 19.1 us, against 25.2 us with 4) unless K is at most 8 blocks (128^3:
    // 4 splits of one block, 13.0 us, against 17.1 us with 2; 256^3: 8
    // splits, 15.0 us, against 17.0 us with 4); the tensor-core kernels >= 4
    int s = choose_splits(splits, tiles, kb_total, slots,
                          p->algo == GEMM_F32_ALGO_FFMA ? (kb_total <= 8 ? 1 : 2) : 4);
    // The single-CTA tensor-core kernel adds up to 8 splits inside a cluster
    // (no reduction launch, ~6 us saved); for K <= 4096 that beats the extra
    // splits' shorter main loops (300 x 260 x 3000: 8 splits in a cluster
    // 25.8 us, 16 through the workspace 28.3 us), and for K <= 1024 four
    // splits beat eight (400 x 400 x 1024: 21.1 against 25.2 us); its
    // clusters must all fit on the device at once (single_cta_splits)
    if (p->algo == GEMM_F32_ALGO_3XTF32 && !p->pair && !p->tmem_b)
        s = single_cta_splits(d.sm_count, tiles, K, splits, p->bn);
    if (p->tmem_b && splits == 0) {
        int clusters = 0;
        if (p->pair && tf32x3_tmem_pair_clusters(d.sm_count, &clusters) == cudaSuccess &&
            clusters > 0)
            slots = clusters;
        cudaGetLastError();
        tmem_estimate(slots, tiles, kb_total, M, N,
                      p->pair ? kTmemPair : p->tmem_wide ? kTmemWide : kTmemSingle, 0, &s);
    }
    p->kb_per_split = (kb_total + s - 1) / s;
    p->splits = (kb_total + p->kb_per_split - 1) / p->kb_per_split;
    const int units = tiles * p->splits;
    p->ldw = round_up(N, 4);

    size_t off = kWorkspaceCounterBytes;  // the counters of in-kernel split-K reductions
    if (p->algo == GEMM_F32_ALGO_3XTF32 && !p->split_in_kernel) {
        // A -> Alo (M x K), and Ahi unless TMA can read A in place as its own
        // high part; B -> B^T hi, lo (N x K); rows padded to 16 bytes
        p->stage_a = 1;
        p->stage_b = 1;
        p->lda = round_up(K, 4);
        p->ldb = round_up(K, 4);
        p->a_in_place = !q.ta && q.lda % 4 == 0 && !misaligned16(q.A);
        p->lda_hi = p->a_in_place ? q.lda : p->lda;
        if (!p->a_in_place) p->off_a = carve(&off, static_cast<long long>(M) * p->lda * 4);
        p->off_a2 = carve(&off, static_cast<long long>(M) * p->lda * 4);
        p->off_b = carve(&off, static_cast<long long>(N) * p->ldb * 4);
        p->off_b2 = carve(&off, static_cast<long long>(N) * p->ldb * 4);
        p->ctas = units < slots ? units : slots;
        if (p->pair) p->ctas *= 2;
    } else {
        // FFMA, and 3xTF32 splitting in the kernel: read in place when TMA
        // can describe the operand as stored: K- (A) or N-contiguous (B)
        // rows, 16-byte row stride and base
        p->stage_a = q.ta || (q.lda % 4 != 0) || misaligned16(q.A);
        p->stage_b = q.tb || (q.ldb % 4 != 0) || misaligned16(q.B);
        p->lda = p->stage_a ? round_up(K, 4) : q.lda;
        p->ldb = p->stage_b ? round_up(N, 4) : q.ldb;
        if (p->stage_a) p->off_a = carve(&off, static_cast<long long>(M) * p->lda * 4);
        if (p->stage_b) p->off_b = carve(&off, static_cast<long long>(K) * p->ldb * 4);
        p->ctas = units;
        if (p->pair) p->ctas = 2 * (units < slots ? units : slots);
    }
    // FFMA with 2..4 splits: each tile's splits run as one thread-block
    // cluster and add their partials through distributed shared memory (no
    // workspace, no reduction kernel); more splits use the workspace, which
    // measured faster from 8 splits on (512^3: 19.1 against 23.2 us)
    if (p->algo == GEMM_F32_ALGO_FFMA && p->splits >= 2 && p->splits <= 4)
        p->cluster_splits = p->splits;
    // The single-CTA tensor-core kernel likewise, when every CTA gets exactly
    // one unit (its stage memory then holds the partial after the main loop)
    if (p->algo == GEMM_F32_ALGO_3XTF32 && !p->pair && !p->tmem_b && p->splits >= 2 &&
        p->splits <= 8 && units <= d.sm_count) {
        // ... whose clusters all fit on the device at once (else, with a
        // caller's split factor, the workspace reduction)
        int fit = 0;
        if (tf32x3_single_cluster_capacity(p->bn, p->splits, &fit) == cudaSuccess &&
            tiles <= fit)
            p->cluster_splits = p->splits;
        cudaGetLastError();
    }
    // The single-CTA form with B's split in tensor memory likewise (its stage
    // memory holds the 128 x 128 partial after the main loop): no workspace
    // and no reduction launch (1025 x 1023 x 1000, 2 splits: 72 clusters of
    // 2 of the 76 that fit, 37.2 -> 34.6 us a call).  Clusters of 3 or more
    // keep a tenth of the capacity free: with the device filled to the last
    // cluster they were not always placed at once (301 x 1874 x 563, 45
    // clusters of 3 of 46: 35.5 us against 27.3 through the workspace).
    // From 16 splits the kernel adds them itself through the workspace
    // (below).
    if (p->tmem_b && !p->pair && !p->tmem_wide && p->splits >= 2 && p->splits <= 8 &&
        units <= d.sm_count) {
        int fit = 0;
        if (tf32x3_tmem_cluster_capacity(p->splits, &fit) == cudaSuccess && tiles <= fit &&
            (p->splits == 2 || 10 * tiles <= 9 * fit))
            p->cluster_splits = p->splits;
        cudaGetLastError();
    }
    if (p->splits > 1 && !p->cluster_splits)
        p->off_w = carve(&off, static_cast<long long>(p->splits) * M * p->ldw * 4);
    // The pair kernel's last round of tiles is usually only partly full
    // (e.g. 1024 tiles over 76 clusters leave 36 for the 14th round).  Cut
    // those tiles into T K shares (T * tail <= clusters) so that the last
    // round takes 1/T of the time; a fix-up kernel adds the shares.  Only
    // where the time saved beats the fix-up's (tail_split_pays): 8192^3
    // saves ~119 us for ~13 us, 2378 x 4792 x 286 would save ~4 us for ~14.
    int clusters = 0;
    if (p->pair && p->splits == 1 && splits == 0 &&
        (p->tmem_b ? tf32x3_tmem_pair_clusters(d.sm_count, &clusters)
                   : tf32x3_pair_clusters(d.sm_count, &clusters)) == cudaSuccess &&
        tiles > clusters) {
        const int r = tiles % clusters;
        int t = r ? clusters / r : 0;
        if (t > 4) t = 4;
        if (r && t >= 2 && kb_total >= 2 * t && tail_split_pays(K, r, t)) {
            p->tail_tiles = r;
            p->tail_splits = t;
            p->tail_m = M;
            p->tail_n = N;
            p->off_t = carve(&off, static_cast<long long>(r) * t * 256 * 256 * 4);
            p->ctas = 2 * clusters;
        }
    }
    cudaGetLastError();
    // The kernel with B's split in tensor memory adds its partials itself when
    // every CTA has exactly one unit (all co-resident, a cooperative launch)
    // and there are at least 16 of them: the CTAs of a tile wait for each
    // other's partials and each sums a band of the tile's rows in split
    // order.  No reduction launch (256 x 256 x 65536, 38 splits: one launch
    // of ~52 us against ~51-56 us for the kernel and a separate reduction);
    // with few splits the cooperative launch costs more than the reduction
    // launch it saves (512^3, 4 splits: ~25 against ~17 us).
    // The CTA pair likewise, with one unit per cluster (and no tail split):
    // its two CTAs each sum a band of the tile's rows.  There the reduction
    // launch it saves is no dearer than the wait for the tile's slowest
    // split (1536^2 x 8192, 2 splits: 139.9 against 135.8 us with the
    // reduction kernel; 256 x 256 x 65536, 76 splits: 53.9 either way), so
    // it too starts at 16 splits, for the single launch.
    const bool counters_fit = 2 * tiles * static_cast<long long>(sizeof(int)) <=
                              static_cast<long long>(kWorkspaceCounterBytes);
    if (p->tmem_b && !p->pair && p->splits >= 16 && units <= d.sm_count && counters_fit)
        p->reduce_in_kernel = 1;
    if (p->tmem_b && p->pair && p->splits >= 16 && !p->tail_tiles && counters_fit &&
        tf32x3_tmem_pair_clusters(d.sm_count, &clusters) == cudaSuccess && units <= clusters)
        p->reduce_in_kernel = 1;
    cudaGetLastError();
    p->ws_bytes = off > kWorkspaceCounterBytes ? off : 0;
    // pre-split operands as stored (A row-major, B not transposed): one
    // staging launch for both
    p->fused_staging = p->algo == GEMM_F32_ALGO_3XTF32 && !p->split_in_kernel && !q.ta && !q.tb;
    p->kernels = 1 + p->stage_a + p->stage_b - p->fused_staging +
                 (p->splits > 1 && !p->cluster_splits && !p->reduce_in_kernel ? 1 : 0) +
                 (p->tail_tiles ? 1 : 0);
}

// Device operands the GEMM kernel reads, after staging.
struct Operands {
    const float* a = nullptr;  // FFMA: A (padded copy when its layout needs one)
    const float* b = nullptr;  // FFMA: B (padded copy when its layout needs one)
    const float* a_hi = nullptr;
    const float* a_lo = nullptr;  // 3xTF32: split A, rows padded to lda
    const float* b_hi = nullptr;
    const float* b_lo = nullptr;  // 3xTF32: split B^T (N x K), rows padded to ldb
};

// Stage B once per call: K-major TF32 hi/lo (3xTF32), or an N-contiguous
// padded copy (FFMA) when B cannot be read in place.
int stage_b(const Plan& p, const Problem& q, unsigned char* ws, Operands* o, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    const int K = q.K, N = q.N;
    if (p.algo == GEMM_F32_ALGO_3XTF32 && !p.split_in_kernel) {
        float* hi = reinterpret_cast<float*>(ws + p.off_b);
        float* lo = reinterpret_cast<float*>(ws + p.off_b2);
        e = q.tb ? launch_split_rows(q.B, q.ldb, N, K, hi, lo, p.ldb, stream)        // N x K already
                 : launch_split_transpose(q.B, q.ldb, K, N, hi, lo, p.ldb, stream);  // K x N -> N x K
        if (e != cudaSuccess) return static_cast<int>(e);
        o->b_hi = hi;
        o->b_lo = lo;
    } else if (p.stage_b) {
        float* dst = reinterpret_cast<float*>(ws + p.off_b);
        e = q.tb ? launch_transpose_pad(q.B, q.ldb, N, K, dst, p.ldb, stream)
                 : launch_pad_copy(q.B, q.ldb, K, N, dst, p.ldb, stream);
        if (e != cudaSuccess) return static_cast<int>(e);
        o->b = dst;
    } else {
        o->b = q.B;
    }
    return GEMM_F32_SUCCESS;
}

// Stage op(A) rows [r0, r0 + M) (r0 > 0 only for untransposed A): TF32 hi/lo
// (3xTF32), or a K-contiguous padded copy (FFMA) when A cannot be read in place.
int stage_a(const Plan& p, const Problem& q, long long r0, int M, unsigned char* ws, Operands* o,
            cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    const int K = q.K;
    const float* a = q.ta ? q.A + r0 : q.A + r0 * q.lda;
    if (p.algo == GEMM_F32_ALGO_3XTF32 && !p.split_in_kernel) {
        float* hi = p.a_in_place ? nullptr : reinterpret_cast<float*>(ws + p.off_a);
        float* lo = reinterpret_cast<float*>(ws + p.off_a2);
        e = q.ta ? launch_split_transpose(a, q.lda, K, M, hi, lo, p.lda, stream)  // K x M -> M x K
                 : launch_split_rows(a, q.lda, M, K, hi, lo, p.lda, stream);
        if (e != cudaSuccess) return static_cast<int>(e);
        o->a_hi = p.a_in_place ? a : hi;
        o->a_lo = lo;
    } else if (p.stage_a) {
        float* dst = reinterpret_cast<float*>(ws + p.off_a);
        e = q.ta ? launch_transpose_pad(a, q.lda, K, M, dst, p.lda, stream)
                 : launch_pad_copy(a, q.lda, M, K, dst, p.lda, stream);
        if (e != cudaSuccess) return static_cast<int>(e);
        o->a = dst;
    } else {
        o->a = a;
    }
    return GEMM_F32_SUCCESS;
}

// The GEMM kernel on staged operands: M rows of C starting at C (row stride
// ldc), then the split-K reduction.  alpha/beta are applied where C is written.
int launch_gemm(const Plan& p, const DeviceState& d, const Operands& o, float* C, long long ldc,
                int M, int N, int K, float alpha, float beta, int mode, unsigned char* ws,
                cudaStream_t stream, cudaEvent_t ev_begin, cudaEvent_t ev_end) {
    float* out = C;
    long long ldo = ldc, split_stride = 0;
    int kmode = mode;
    if (p.splits > 1 && !p.cluster_splits) {
        out = reinterpret_cast<float*>(ws + p.off_w);
        ldo = p.ldw;
        split_stride = static_cast<long long>(M) * p.ldw;
        kmode = 0;  // partials are raw sums; the reduction scales
    }
    const int vec_store = (ldo % 4 == 0) && !misaligned16(out);
    cudaError_t e = cudaSuccess;
    int st = GEMM_F32_SUCCESS;
    if (p.algo == GEMM_F32_ALGO_3XTF32) {
        Tf32x3Args ta;
        std::memset(&ta, 0, sizeof(ta));
        if (p.tmem_b) {
            // the operands as stored: A {K, M} in 128 x 32 boxes, B {N, K}
            // in 32 x 32 boxes (one 128-byte swizzle row wide); the wide form
            // A in 256 x 16 boxes (64-byte swizzle), B in 32 x 16
            if ((st = encode_2d(&ta.tmAhi, o.a, K, M, p.lda, p.tile_k, p.tmem_wide ? 256 : 128,
                                p.tmem_wide ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM_F32_SUCCESS ||
                (st = encode_2d(&ta.tmBhi, o.b, N, K, p.ldb, 32, p.tile_k,
                                CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM_F32_SUCCESS)
                return st;
            ta.out = out;
            ta.ldo = ldo;
            ta.split_stride = split_stride;
            ta.M = M;
            ta.N = N;
            ta.K = K;
            ta.bn = p.bn;
            ta.kb_per_split = p.kb_per_split;
            ta.splits = p.splits;
            ta.fault = d.fault;
            ta.timeout_ns = kDefaultTimeoutNs;
            ta.alpha = alpha;
            ta.beta = beta;
            ta.scale_mode = kmode;
            ta.cluster_splits = p.cluster_splits;
            ta.vec_store = vec_store;
            if (p.reduce_in_kernel) {
                ta.counters = reinterpret_cast<int*>(ws);
                ta.c_final = C;
                ta.ldc = ldc;
                ta.c_mode = mode;
            }
            if (ev_begin && (e = cudaEventRecord(ev_begin, stream)) != cudaSuccess)
                return static_cast<int>(e);
            ta.pair = p.pair;
            // the tail split names tiles of the extent it was planned for
            const bool tail = p.tail_tiles && M == p.tail_m && N == p.tail_n;
            ta.tail_tiles = tail ? p.tail_tiles : 0;
            ta.tail_splits = tail ? p.tail_splits : 0;
            ta.tail_ws = tail ? reinterpret_cast<float*>(ws + p.off_t) : nullptr;
            if ((e = p.pair        ? launch_sgemm_3xtf32_tmem_pair(ta, stream, d.sm_count)
                     : p.tmem_wide ? launch_sgemm_3xtf32_tmem_wide(ta, stream, d.sm_count)
                                   : launch_sgemm_3xtf32_tmem(ta, stream, d.sm_count)) != cudaSuccess)
                return static_cast<int>(e);
            if (ev_end && (e = cudaEventRecord(ev_end, stream)) != cudaSuccess)
                return static_cast<int>(e);
            if (p.splits > 1 && !p.cluster_splits && !p.reduce_in_kernel) {
                e = launch_splitk_reduce(out, split_stride, p.ldw, p.splits, C, ldc, M, N, alpha,
                                         beta, mode, stream);
                if (e != cudaSuccess) return static_cast<int>(e);
            }
            return GEMM_F32_SUCCESS;
        }
        if (p.split_in_kernel) {
            // the operands as stored: A {K, M} in 128 x 32 boxes, B {N, K}
            // in 32 x 32 boxes (one 128-byte swizzle row wide)
            if ((st = encode_2d(&ta.tmAhi, o.a, K, M, p.lda, p.tile_k, 128,
                                CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM_F32_SUCCESS ||
                (st = encode_2d(&ta.tmBhi, o.b, N, K, p.ldb, 32, p.tile_k,
                                CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM_F32_SUCCESS)
                return st;
            ta.tmAlo = ta.tmAhi;
            ta.tmBlo = ta.tmBhi;
            ta.split_in_kernel = 1;
        } else if ((st = encode_2d(&ta.tmAhi, o.a_hi, K, M, p.lda_hi, p.tile_k, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM_F32_SUCCESS ||
            (st = encode_2d(&ta.tmAlo, o.a_lo, K, M, p.lda, p.tile_k, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM_F32_SUCCESS ||
            (st = encode_2d(&ta.tmBhi, o.b_hi, K, N, p.ldb, p.tile_k, p.box_n,
                            CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM_F32_SUCCESS ||
            (st = encode_2d(&ta.tmBlo, o.b_lo, K, N, p.ldb, p.tile_k, p.box_n,
                            CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM_F32_SUCCESS)
            return st;
        ta.out = out;
        ta.ldo = ldo;
        ta.split_stride = split_stride;
        ta.M = M;
        ta.N = N;
        ta.K = K;
        ta.bn = p.bn;
        ta.pair = p.pair;
        ta.kb_per_split = p.kb_per_split;
        ta.splits = p.splits;
        ta.vec_store = vec_store;
        ta.fault = d.fault;
        ta.timeout_ns = kDefaultTimeoutNs;
        ta.alpha = alpha;
        ta.beta = beta;
        ta.scale_mode = kmode;
        // the tail split names tiles of the extent it was planned for; a
        // launch on another extent (a shorter last row panel, a column
        // block) runs without it
        const bool tail = p.tail_tiles && M == p.tail_m && N == p.tail_n;
        ta.tail_tiles = tail ? p.tail_tiles : 0;
        ta.tail_splits = tail ? p.tail_splits : 0;
        ta.tail_ws = tail ? reinterpret_cast<float*>(ws + p.off_t) : nullptr;
        ta.cluster_splits = p.cluster_splits;
        // C through TMA stores (and, with a beta term, TMA loads of the old
        // C): one K split, and not the pair kernel that splits in shared
        // memory.
        // TMA stores clip a box at C's extent in 16-byte pieces: the row
        // length must be a whole number of them, or a ragged last piece
        // would be written in full, past column N.
        if (vec_store && N % 4 == 0 && p.splits == 1 && !(p.split_in_kernel && p.pair)) {
            if ((st = encode_2d(&ta.tmC, out, N, M, ldo, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B)) !=
                GEMM_F32_SUCCESS)
                return st;
            ta.tma_store = 1;
        }
        if (ev_begin && (e = cudaEventRecord(ev_begin, stream)) != cudaSuccess)
            return static_cast<int>(e);
        if ((e = launch_sgemm_3xtf32(ta, stream, d.sm_count)) != cudaSuccess)
            return static_cast<int>(e);
        if (ev_end && (e = cudaEventRecord(ev_end, stream)) != cudaSuccess)
            return static_cast<int>(e);
    } else {
        FfmaArgs fa;
        std::memset(&fa, 0, sizeof(fa));
        if ((st = encode_2d(&fa.tmA, o.a, K, M, p.lda, p.tile_k, p.tile_m,
                            CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM_F32_SUCCESS ||
            (st = encode_2d(&fa.tmB, o.b, N, K, p.ldb, p.tile_n, p.tile_k,
                            CU_TENSOR_MAP_SWIZZLE_NONE)) != GEMM_F32_SUCCESS)
            return st;
        fa.out = out;
        fa.ldo = ldo;
        fa.split_stride = split_stride;
        fa.M = M;
        fa.N = N;
        fa.K = K;
        fa.kb_per_split = p.kb_per_split;
        fa.splits = p.splits;
        fa.vec_store = vec_store;
        fa.fault = d.fault;
        fa.timeout_ns = kDefaultTimeoutNs;
        fa.variant = p.variant;
        fa.bn = p.tile_n;
        fa.alpha = alpha;
        fa.beta = beta;
        fa.scale_mode = kmode;
        fa.cluster_splits = p.cluster_splits;
        if (ev_begin && (e = cudaEventRecord(ev_begin, stream)) != cudaSuccess)
            return static_cast<int>(e);
        if ((e = launch_sgemm_ffma(fa, stream)) != cudaSuccess) return static_cast<int>(e);
        if (ev_end && (e = cudaEventRecord(ev_end, stream)) != cudaSuccess)
            return static_cast<int>(e);
    }
    if (p.splits > 1 && !p.cluster_splits) {
        e = launch_splitk_reduce(out, split_stride, p.ldw, p.splits, C, ldc, M, N, alpha, beta,
                                 mode, stream);
        if (e != cudaSuccess) return static_cast<int>(e);
    }
    return GEMM_F32_SUCCESS;
}

// Enqueue one GEMM on `stream` (validated problem, g_mutex held, device known).
int enqueue(const Problem& q, int algo, int splits, DeviceState* d, int dev, cudaStream_t stream,
            cudaEvent_t ev_begin, cudaEvent_t ev_end, int tile) {
    if (q.M == 0 || q.N == 0) return GEMM_F32_SUCCESS;
    if (q.K == 0 || q.alpha == 0.0f) {
        // empty sum (or a zero multiplier): C = beta C, A and B not read
        cudaError_t e = launch_scale_c(q.C, q.ldc, q.M, q.N, q.beta, stream);
        return e == cudaSuccess ? GEMM_F32_SUCCESS : static_cast<int>(e);
    }
    int st = get_encoder();
    if (st != GEMM_F32_SUCCESS) return st;

    Plan p;
    make_plan(*d, q, algo, splits, &p, tile);

    unsigned char* ws = nullptr;
    if (p.ws_bytes) {
        void* w = nullptr;
        st = workspace(dev, stream, p.ws_bytes, &w);
        if (st != GEMM_F32_SUCCESS) return st;
        ws = static_cast<unsigned char*>(w);
    }
    Operands o;
    if (p.fused_staging) {
        float* a_hi = p.a_in_place ? nullptr : reinterpret_cast<float*>(ws + p.off_a);
        float* a_lo = reinterpret_cast<float*>(ws + p.off_a2);
        float* b_hi = reinterpret_cast<float*>(ws + p.off_b);
        float* b_lo = reinterpret_cast<float*>(ws + p.off_b2);
        const cudaError_t e = launch_split_operands(q.A, q.lda, q.M, q.K, a_hi, a_lo, p.lda, q.B,
                                                    q.ldb, q.N, b_hi, b_lo, p.ldb, stream);
        if (e != cudaSuccess) return static_cast<int>(e);
        o.a_hi = p.a_in_place ? q.A : a_hi;
        o.a_lo = a_lo;
        o.b_hi = b_hi;
        o.b_lo = b_lo;
    } else {
        if ((st = stage_a(p, q, 0, q.M, ws, &o, stream)) != GEMM_F32_SUCCESS) return st;
        if ((st = stage_b(p, q, ws, &o, stream)) != GEMM_F32_SUCCESS) return st;
    }
    return launch_gemm(p, *d, o, q.C, q.ldc, q.M, q.N, q.K, q.alpha, q.beta, scale_mode(q), ws,
                       stream, ev_begin, ev_end);
}

int run(const Problem& q, int algo, int splits, cudaStream_t stream,
        cudaEvent_t ev_begin = nullptr, cudaEvent_t ev_end = nullptr,
        int tile = GEMM_F32_TILE_AUTO) {
    int st = validate(q, algo, splits);
    if (st != GEMM_F32_SUCCESS) return st;
    if (q.M == 0 || q.N == 0) return GEMM_F32_SUCCESS;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* d = nullptr;
    int dev = 0;
    st = device_state(&d, &dev, &stream);
    if (st != GEMM_F32_SUCCESS) return st;
    return enqueue(q, algo, splits, d, dev, stream, ev_begin, ev_end, tile);
}

// ---- host-buffer entry: copies overlapped with the GEMM, by row panels ----
constexpr int kMaxPanels = 16;
constexpr int kMaxColBlocks = 4;  // column blocks of the first and last row panel

struct HostPipe {
    bool ready = false;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_b = nullptr, ev_done = nullptr;
    cudaEvent_t ev_a[kMaxPanels] = {}, ev_c[kMaxPanels] = {};
    cudaEvent_t ev_bblk[kMaxColBlocks] = {}, ev_cblk[kMaxColBlocks] = {};
    void* dev_buf = nullptr;  // device copies of A, B and C
    size_t dev_bytes = 0;
    bool captured = false;          // as for Workspace
    std::vector<void*> retired;
};
std::map<std::pair<int, cudaStream_t>, HostPipe> g_pipes;

// Side streams, events and the device copies for (dev, stream); g_mutex held.
int host_pipe(int dev, cudaStream_t stream, size_t bytes, HostPipe** out) {
    HostPipe& hp = g_pipes[std::make_pair(dev, stream)];
    cudaError_t e = cudaSuccess;
    const bool capturing = stream_capturing(stream);
    if ((!hp.ready || hp.dev_bytes < bytes) && capturing) return GEMM_F32_ERR_CAPTURE;
    if (capturing) hp.captured = true;
    if (!hp.ready) {
        const unsigned fl = cudaEventDisableTiming;
        if ((e = cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&hp.ev_start, fl)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&hp.ev_b, fl)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&hp.ev_done, fl)) != cudaSuccess)
            return static_cast<int>(e);
        for (int i = 0; i < kMaxPanels; ++i)
            if ((e = cudaEventCreateWithFlags(&hp.ev_a[i], fl)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&hp.ev_c[i], fl)) != cudaSuccess)
                return static_cast<int>(e);
        for (int i = 0; i < kMaxColBlocks; ++i)
            if ((e = cudaEventCreateWithFlags(&hp.ev_bblk[i], fl)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&hp.ev_cblk[i], fl)) != cudaSuccess)
                return static_cast<int>(e);
        hp.ready = true;
    }
    if (hp.dev_bytes < bytes) {
        if (hp.dev_buf) {
            if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return static_cast<int>(e);
            if (hp.captured)
                hp.retired.push_back(hp.dev_buf);
            else
                cudaFree(hp.dev_buf);
            hp.dev_buf = nullptr;
            hp.dev_bytes = 0;
            hp.captured = false;
        }
        if (injected(GEMM_F32_INJECT_WORKSPACE) || cudaMalloc(&hp.dev_buf, bytes) != cudaSuccess) {
            cudaGetLastError();
            hp.dev_buf = nullptr;
            return GEMM_F32_ERR_WORKSPACE;
        }
        hp.dev_bytes = bytes;
    }
    *out = &hp;
    return GEMM_F32_SUCCESS;
}

// Deep K: K panels.  Panel k of A (M x Kp, a strided 2-D copy from the host)
// and of B (Kp x N rows) arrive on the copy-in stream while the GEMM of panel
// k-1 runs; panel k accumulates into C (beta = 1 after the first).  The last
// panel's GEMM is cut into row blocks so that finished rows of C go back to
// the host on the copy-out stream while the rest is still computing.  Only
// the first panel's copy and the last row block's copy are not overlapped.
int run_host_kpanels(const float* A, const float* B, float* C, int M, int N, int K, int algo,
                     DeviceState* d, int dev, HostPipe* hp, float* dA, float* dB, float* dC,
                     int kp, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    int st = GEMM_F32_SUCCESS;
    const int panels = (K + kp - 1) / kp;
    for (int i = 0; i < panels; ++i) {
        const int k0 = i * kp;
        const int kw = (K - k0) < kp ? (K - k0) : kp;
        float* a_i = dA + static_cast<size_t>(i) * M * kp;  // panel i, row stride kp
        float* b_i = dB + static_cast<size_t>(k0) * N;      // rows k0 .. k0+kw of B
        if ((e = cudaMemcpy2DAsync(a_i, static_cast<size_t>(kp) * 4, A + k0,
                                   static_cast<size_t>(K) * 4, static_cast<size_t>(kw) * 4, M,
                                   cudaMemcpyHostToDevice, hp->s_in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(b_i, B + static_cast<size_t>(k0) * N,
                                 static_cast<size_t>(kw) * N * 4, cudaMemcpyHostToDevice,
                                 hp->s_in)) != cudaSuccess ||
            (e = cudaEventRecord(hp->ev_a[i], hp->s_in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(stream, hp->ev_a[i], 0)) != cudaSuccess)
            return static_cast<int>(e);
        Problem q = packed(a_i, b_i, dC, M, N, kw);
        q.lda = kp;
        q.beta = i ? 1.0f : 0.0f;
        if (i + 1 < panels) {
            if ((st = enqueue(q, algo, 0, d, dev, stream, nullptr, nullptr, GEMM_F32_TILE_AUTO)) !=
                GEMM_F32_SUCCESS)
                return st;
            continue;
        }
        // last panel: row blocks, each copied back as soon as it is final
        const int blocks = M >= 4096 ? 8 : (M >= 1024 ? 4 : 1);
        const int rows = ((M + blocks - 1) / blocks + 255) / 256 * 256;
        for (int r0 = 0, j = 0; r0 < M; r0 += rows, ++j) {
            const int mr = (M - r0) < rows ? (M - r0) : rows;
            Problem qr = q;
            qr.M = mr;
            qr.A = a_i + static_cast<size_t>(r0) * kp;
            qr.C = dC + static_cast<size_t>(r0) * N;
            if ((st = enqueue(qr, algo, 0, d, dev, stream, nullptr, nullptr, GEMM_F32_TILE_AUTO)) !=
                GEMM_F32_SUCCESS)
                return st;
            if ((e = cudaEventRecord(hp->ev_c[j], stream)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(hp->s_out, hp->ev_c[j], 0)) != cudaSuccess ||
                (e = cudaMemcpyAsync(C + static_cast<size_t>(r0) * N,
                                     dC + static_cast<size_t>(r0) * N,
                                     static_cast<size_t>(mr) * N * 4, cudaMemcpyDeviceToHost,
                                     hp->s_out)) != cudaSuccess)
                return static_cast<int>(e);
        }
    }
    if ((e = cudaEventRecord(hp->ev_done, hp->s_out)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, hp->ev_done, 0)) != cudaSuccess)
        return static_cast<int>(e);
    return GEMM_F32_SUCCESS;
}

int run_host(const float* A, const float* B, float* C, int M, int N, int K, int algo,
             cudaStream_t stream) {
    int st = validate(packed(A, B, C, M, N, K), algo, 0);
    if (st != GEMM_F32_SUCCESS) return st;
    if (M == 0 || N == 0) return GEMM_F32_SUCCESS;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* d = nullptr;
    int dev = 0;
    if ((st = device_state(&d, &dev, &stream)) != GEMM_F32_SUCCESS) return st;
    if ((st = get_encoder()) != GEMM_F32_SUCCESS) return st;

    // Row panels need all of B before the first GEMM: with B arriving at
    // ~210 GB/s and the GEMM at ~300 TFLOP/s that wait is about 2900/M of the
    // compute time.  For M <= 4096 with deep K the K-panel schedule (panels of
    // >= 1024, first GEMM after one panel) wins; at 8192^3 row panels were
    // measured faster (185.6 vs 174.3 TFLOPS end to end: K panels re-read C).
    const bool kpanels =
        K >= 2048 && M <= 4096 && static_cast<long long>(M) * N >= (1LL << 22);
    const int kp = !kpanels ? K
                   : (K + kMaxPanels - 1) / kMaxPanels > 1024
                       ? static_cast<int>(round_up((K + kMaxPanels - 1) / kMaxPanels, 32))
                       : 1024;
    const long long a_cols = kpanels ? static_cast<long long>((K + kp - 1) / kp) * kp : K;
    // device copies: A (M x K, or its K panels), B (K x N), C (M x N), 256-byte aligned
    const size_t bytes_a =
        static_cast<size_t>(round_up(static_cast<long long>(M) * a_cols * 4, 256));
    const size_t bytes_b = static_cast<size_t>(round_up(static_cast<long long>(K) * N * 4, 256));
    const size_t bytes_c = static_cast<size_t>(round_up(static_cast<long long>(M) * N * 4, 256));
    HostPipe* hp = nullptr;
    if ((st = host_pipe(dev, stream, bytes_a + bytes_b + bytes_c, &hp)) != GEMM_F32_SUCCESS)
        return st;
    float* dA = static_cast<float*>(hp->dev_buf);
    float* dB = reinterpret_cast<float*>(static_cast<unsigned char*>(hp->dev_buf) + bytes_a);
    float* dC = reinterpret_cast<float*>(static_cast<unsigned char*>(hp->dev_buf) + bytes_a +
                                         bytes_b);

    if (kpanels) {
        cudaError_t e0 = cudaEventRecord(hp->ev_start, stream);
        if (e0 == cudaSuccess) e0 = cudaStreamWaitEvent(hp->s_in, hp->ev_start, 0);
        if (e0 == cudaSuccess) e0 = cudaStreamWaitEvent(hp->s_out, hp->ev_start, 0);
        if (e0 != cudaSuccess) return static_cast<int>(e0);
        return run_host_kpanels(A, B, C, M, N, K, algo, d, dev, hp, dA, dB, dC, kp, stream);
    }

    // row panels: a quarter of M (at least 512 rows, at most kMaxPanels of
    // them); big enough for a panel's tiles to fill several rounds of the
    // persistent grid
    long long rows = (M + 3) / 4;
    rows = round_up(rows < 512 ? 512 : rows, 256);
    if ((M + rows - 1) / rows > kMaxPanels) rows = round_up((M + kMaxPanels - 1) / kMaxPanels, 128);
    const int P = static_cast<int>(rows < M ? rows : M);
    const int panels = (M + P - 1) / P;

    cudaError_t e = cudaSuccess;
#define GEMM_F32_TRY(x)                                      \
    do {                                                     \
        if ((e = (x)) != cudaSuccess) return static_cast<int>(e); \
    } while (0)
    // the side streams start after everything already queued on `stream`
    GEMM_F32_TRY(cudaEventRecord(hp->ev_start, stream));
    GEMM_F32_TRY(cudaStreamWaitEvent(hp->s_in, hp->ev_start, 0));
    GEMM_F32_TRY(cudaStreamWaitEvent(hp->s_out, hp->ev_start, 0));

    if (K == 0) {
        GEMM_F32_TRY(launch_fill_zero(dC, static_cast<long long>(M) * N, stream));
        GEMM_F32_TRY(cudaMemcpyAsync(C, dC, static_cast<size_t>(M) * N * 4,
                                     cudaMemcpyDeviceToHost, stream));
        return GEMM_F32_SUCCESS;
    }

    // device-side problem: the device copies, one panel of P rows at a time
    Problem q = packed(dA, dB, dC, M, N, K);
    Problem qp = q;
    qp.M = P;
    Plan p;
    make_plan(*d, qp, algo, 0, &p);

    // Column blocks.  With row panels alone the first GEMM waits for all of
    // B (8192^3: 1.25 ms of copying).  On staged tensor-core operands the
    // first and the last row panel are instead computed by column blocks of
    // B: the first block's GEMM starts once panel 0 of A and that block of B
    // are on the device (B's blocks are staged into the full B^T planes, so
    // the middle panels reuse them), and the last panel's blocks go back to
    // the host one by one, so only the last block's copy is not overlapped.
    // With B's split in tensor memory there is nothing to stage: a block's
    // GEMM reads its columns of B where they landed (row stride N), which
    // TMA can do only when that stride (and A's, K) is a multiple of 16
    // bytes; otherwise the row panels run on the padded copies.
    const int nc = static_cast<int>(round_up((N + 3) / 4, 256));
    const int nblk = (N + nc - 1) / nc;
    Plan pc;
    const bool tmem_blocks = p.algo == GEMM_F32_ALGO_3XTF32 && p.tmem_b && p.splits == 1 &&
                             !p.stage_a && !p.stage_b && panels >= 2 && N >= 1024 &&
                             nblk >= 2 && nblk <= kMaxColBlocks;
    bool col_blocks = p.algo == GEMM_F32_ALGO_3XTF32 && !p.split_in_kernel && p.splits == 1 &&
                      panels >= 2 && N >= 1024 && nblk >= 2 && nblk <= kMaxColBlocks;
    if (tmem_blocks) {
        Problem qc = qp;
        qc.N = nc;
        qc.ldb = N;
        qc.ldc = N;
        make_plan(*d, qc, GEMM_F32_ALGO_3XTF32, 0, &pc);
        col_blocks = pc.tmem_b && pc.splits == 1 && !pc.stage_a && !pc.stage_b;
        pc.off_w += p.ws_bytes;
        pc.off_t += p.ws_bytes;
    } else if (col_blocks) {
        Problem qc = qp;
        qc.N = nc;
        // the two-CTA kernel for a block (2048 x 2048: 64 pair tiles in one
        // round), faster there than the single-CTA 128 x 256 kernel AUTO picks
        make_plan(*d, qc, GEMM_F32_ALGO_3XTF32, 0, &pc,
                  nc >= 1024 ? GEMM_F32_TILE_256x256_PAIR : GEMM_F32_TILE_AUTO);
        // the block GEMMs read the panel plan's staged operands; only their
        // split-K partials or tail shares need space, after the panel plan's
        col_blocks = pc.algo == GEMM_F32_ALGO_3XTF32 && !pc.split_in_kernel &&
                     pc.lda == p.lda && pc.lda_hi == p.lda_hi && pc.ldb == p.ldb &&
                     pc.tile_k == p.tile_k;
        pc.off_w += p.ws_bytes;
        pc.off_t += p.ws_bytes;
    }
    const size_t ws_total = p.ws_bytes + (col_blocks ? pc.ws_bytes : 0);
    unsigned char* ws = nullptr;
    if (ws_total) {
        void* w = nullptr;
        if ((st = workspace(dev, stream, ws_total, &w)) != GEMM_F32_SUCCESS) return st;
        ws = static_cast<unsigned char*>(w);
    }

    if (!col_blocks) {
        GEMM_F32_TRY(cudaMemcpyAsync(dB, B, static_cast<size_t>(K) * N * 4,
                                     cudaMemcpyHostToDevice, hp->s_in));
        GEMM_F32_TRY(cudaEventRecord(hp->ev_b, hp->s_in));
        GEMM_F32_TRY(cudaStreamWaitEvent(stream, hp->ev_b, 0));
        Operands o;
        if ((st = stage_b(p, q, ws, &o, stream)) != GEMM_F32_SUCCESS) return st;

        for (int i = 0; i < panels; ++i) {
            const int r0 = i * P;
            const int mp = (M - r0) < P ? (M - r0) : P;
            const size_t off_a = static_cast<size_t>(r0) * K, off_c = static_cast<size_t>(r0) * N;
            GEMM_F32_TRY(cudaMemcpyAsync(dA + off_a, A + off_a, static_cast<size_t>(mp) * K * 4,
                                         cudaMemcpyHostToDevice, hp->s_in));
            GEMM_F32_TRY(cudaEventRecord(hp->ev_a[i], hp->s_in));
            GEMM_F32_TRY(cudaStreamWaitEvent(stream, hp->ev_a[i], 0));
            if ((st = stage_a(p, q, r0, mp, ws, &o, stream)) != GEMM_F32_SUCCESS) return st;
            if ((st = launch_gemm(p, *d, o, dC + off_c, N, mp, N, K, 1.0f, 0.0f, 0, ws, stream,
                                  nullptr, nullptr)) != GEMM_F32_SUCCESS)
                return st;
            GEMM_F32_TRY(cudaEventRecord(hp->ev_c[i], stream));
            GEMM_F32_TRY(cudaStreamWaitEvent(hp->s_out, hp->ev_c[i], 0));
            GEMM_F32_TRY(cudaMemcpyAsync(C + off_c, dC + off_c, static_cast<size_t>(mp) * N * 4,
                                         cudaMemcpyDeviceToHost, hp->s_out));
        }
    } else {
        // copies in: A panel 0, the column blocks of B, then the other A panels
        GEMM_F32_TRY(cudaMemcpyAsync(dA, A, static_cast<size_t>(P) * K * 4, cudaMemcpyHostToDevice,
                                     hp->s_in));
        GEMM_F32_TRY(cudaEventRecord(hp->ev_a[0], hp->s_in));
        for (int c = 0; c < nblk; ++c) {
            const int c0 = c * nc, w = (N - c0) < nc ? (N - c0) : nc;
            GEMM_F32_TRY(cudaMemcpy2DAsync(dB + c0, static_cast<size_t>(N) * 4, B + c0,
                                           static_cast<size_t>(N) * 4, static_cast<size_t>(w) * 4,
                                           K, cudaMemcpyHostToDevice, hp->s_in));
            GEMM_F32_TRY(cudaEventRecord(hp->ev_bblk[c], hp->s_in));
        }
        for (int i = 1; i < panels; ++i) {
            const int r0 = i * P;
            const int mp = (M - r0) < P ? (M - r0) : P;
            const size_t off_a = static_cast<size_t>(r0) * K;
            GEMM_F32_TRY(cudaMemcpyAsync(dA + off_a, A + off_a, static_cast<size_t>(mp) * K * 4,
                                         cudaMemcpyHostToDevice, hp->s_in));
            GEMM_F32_TRY(cudaEventRecord(hp->ev_a[i], hp->s_in));
        }
        Operands o;
        float* bt_hi = tmem_blocks ? nullptr : reinterpret_cast<float*>(ws + p.off_b);
        float* bt_lo = tmem_blocks ? nullptr : reinterpret_cast<float*>(ws + p.off_b2);
        o.b_hi = bt_hi;
        o.b_lo = bt_lo;
        o.b = dB;
        for (int i = 0; i < panels; ++i) {
            const int r0 = i * P;
            const int mp = (M - r0) < P ? (M - r0) : P;
            const size_t off_c = static_cast<size_t>(r0) * N;
            GEMM_F32_TRY(cudaStreamWaitEvent(stream, hp->ev_a[i], 0));
            if ((st = stage_a(p, q, r0, mp, ws, &o, stream)) != GEMM_F32_SUCCESS) return st;
            if (i == 0 || i == panels - 1) {
                for (int c = 0; c < nblk; ++c) {
                    const int c0 = c * nc, w = (N - c0) < nc ? (N - c0) : nc;
                    if (i == 0) {
                        GEMM_F32_TRY(cudaStreamWaitEvent(stream, hp->ev_bblk[c], 0));
                        // staged operands: this block of B into rows c0.. of
                        // the B^T planes
                        if (!tmem_blocks)
                            GEMM_F32_TRY(launch_split_transpose(
                                dB + c0, N, K, w, bt_hi + static_cast<size_t>(c0) * p.ldb,
                                bt_lo + static_cast<size_t>(c0) * p.ldb, p.ldb, stream));
                    }
                    Operands ob = o;
                    if (tmem_blocks) {
                        ob.b = dB + c0;
                    } else {
                        ob.b_hi = bt_hi + static_cast<size_t>(c0) * p.ldb;
                        ob.b_lo = bt_lo + static_cast<size_t>(c0) * p.ldb;
                    }
                    if ((st = launch_gemm(pc, *d, ob, dC + off_c + c0, N, mp, w, K, 1.0f, 0.0f, 0,
                                          ws, stream, nullptr, nullptr)) != GEMM_F32_SUCCESS)
                        return st;
                    if (i == panels - 1) {
                        // this block of the last panel is final: back to the host
                        GEMM_F32_TRY(cudaEventRecord(hp->ev_cblk[c], stream));
                        GEMM_F32_TRY(cudaStreamWaitEvent(hp->s_out, hp->ev_cblk[c], 0));
                        GEMM_F32_TRY(cudaMemcpy2DAsync(
                            C + off_c + c0, static_cast<size_t>(N) * 4, dC + off_c + c0,
                            static_cast<size_t>(N) * 4, static_cast<size_t>(w) * 4, mp,
                            cudaMemcpyDeviceToHost, hp->s_out));
                    }
                }
                if (i == panels - 1) continue;
            } else {
                if ((st = launch_gemm(p, *d, o, dC + off_c, N, mp, N, K, 1.0f, 0.0f, 0, ws, stream,
                                      nullptr, nullptr)) != GEMM_F32_SUCCESS)
                    return st;
            }
            GEMM_F32_TRY(cudaEventRecord(hp->ev_c[i], stream));
            GEMM_F32_TRY(cudaStreamWaitEvent(hp->s_out, hp->ev_c[i], 0));
            GEMM_F32_TRY(cudaMemcpyAsync(C + off_c, dC + off_c, static_cast<size_t>(mp) * N * 4,
                                         cudaMemcpyDeviceToHost, hp->s_out));
        }
    }
    // the call is complete on `stream` once the last panel of C is on the host
    GEMM_F32_TRY(cudaEventRecord(hp->ev_done, hp->s_out));
    GEMM_F32_TRY(cudaStreamWaitEvent(stream, hp->ev_done, 0));
#undef GEMM_F32_TRY
    return GEMM_F32_SUCCESS;
}

// A forced configuration: tile id within range and valid for the algorithm.
int check_config(const gemm_f32_config* cfg) {
    if (!cfg) return GEMM_F32_ERR_INVALID_VALUE;
    if (cfg->tile < GEMM_F32_TILE_AUTO || cfg->tile > GEMM_F32_TILE_256x128_TMEM)
        return GEMM_F32_ERR_INVALID_VALUE;
    if ((cfg->tile == GEMM_F32_TILE_256x256_PAIR || cfg->tile == GEMM_F32_TILE_256x256_PAIR_SPLIT ||
         cfg->tile == GEMM_F32_TILE_128x128_SPLIT || cfg->tile == GEMM_F32_TILE_128x128_TMEM ||
         cfg->tile == GEMM_F32_TILE_256x256_TMEM || cfg->tile == GEMM_F32_TILE_256x128_TMEM) &&
        cfg->algo == GEMM_F32_ALGO_FFMA)
        return GEMM_F32_ERR_INVALID_VALUE;
    if (cfg->tile != GEMM_F32_TILE_AUTO && cfg->algo == GEMM_F32_ALGO_AUTO)
        return GEMM_F32_ERR_INVALID_VALUE;  // a tile names one algorithm's kernels
    return GEMM_F32_SUCCESS;
}

// The plan a call of problem q with configuration cfg would run, without
// running it (plan_info out): the body of the gemm_f32_plan entry points.
int plan_problem(const Problem& q, const gemm_f32_config* cfg, gemm_f32_plan_info* out) {
    if (!out) return GEMM_F32_ERR_INVALID_VALUE;
    std::memset(out, 0, sizeof(*out));
    int st = check_config(cfg);
    if (st != GEMM_F32_SUCCESS) return st;
    const int M = q.M, N = q.N, K = q.K;
    st = validate(q, cfg->algo, cfg->splits, false);
    if (st != GEMM_F32_SUCCESS) return st;
    out->splits = 1;
    if (M == 0 || N == 0) return GEMM_F32_SUCCESS;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* d = nullptr;
    int dev = 0;
    st = device_state(&d, &dev);
    if (st != GEMM_F32_SUCCESS) return st;
    if (K == 0) {
        out->kernels = 1;
        return GEMM_F32_SUCCESS;
    }
    Plan p;
    make_plan(*d, q, cfg->algo, cfg->splits, &p, cfg->tile);
    out->algo = p.algo;
    out->splits = p.splits;
    out->tile_m = p.tile_m;
    out->tile_n = p.tile_n;
    out->tile_k = p.tile_k;
    out->stages = p.stages;
    out->ctas = p.ctas;
    out->stage_a = p.stage_a;
    out->stage_b = p.stage_b;
    out->kernels = p.kernels;
    out->workspace_bytes = static_cast<long long>(p.ws_bytes);
    out->split_in_kernel = p.split_in_kernel;
    out->cluster_reduce = p.cluster_splits ? 1 : 0;
    out->reduce_in_kernel = p.reduce_in_kernel;
    // residency of the main kernel, from the occupancy calculator
    int per_sm = 0;
    cudaError_t e = cudaSuccess;
    if (p.algo == GEMM_F32_ALGO_FFMA) {
        e = ffma_ctas_per_sm(p.variant, &per_sm);
        out->threads_per_cta = ffma_config(p.variant).threads;
    } else if (p.tmem_b && p.pair) {
        int clusters = 0;
        e = tf32x3_tmem_pair_clusters(d->sm_count, &clusters);
        per_sm = d->sm_count ? (2 * clusters + d->sm_count - 1) / d->sm_count : 0;
        out->threads_per_cta = tf32x3_tmem_config(true).threads;
    } else if (p.tmem_wide) {
        per_sm = 1;  // the whole tensor memory and 201 KB of shared memory
        out->threads_per_cta = tf32x3_tmem_wide_config().threads;
    } else if (p.tmem_b) {
        e = tf32x3_tmem_ctas_per_sm(&per_sm);
        out->threads_per_cta = tf32x3_tmem_config(false).threads;
    } else if (p.pair) {
        int clusters = 0;
        e = tf32x3_pair_clusters(d->sm_count, &clusters);
        per_sm = d->sm_count ? (2 * clusters + d->sm_count - 1) / d->sm_count : 0;
        out->threads_per_cta = tf32x3_config(256, true).threads;
    } else {
        int ctas = 0;
        e = tf32x3_single_cluster_capacity(p.bn, 1, &ctas);
        per_sm = d->sm_count ? (ctas + d->sm_count - 1) / d->sm_count : 0;
        out->threads_per_cta = tf32x3_config(p.bn, false).threads;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        per_sm = 0;
    }
    out->ctas_per_sm = per_sm;
    out->b_in_tmem = p.tmem_b;
    return GEMM_F32_SUCCESS;
}

}  // namespace

extern "C" {

int gemm_f32(const float* A, const float* B, float* C, int M, int N, int K, cudaStream_t stream) {
    return run(packed(A, B, C, M, N, K), GEMM_F32_ALGO_AUTO, 0, stream);
}

int gemm_f32_algo(const float* A, const float* B, float* C, int M, int N, int K, int algo,
                  cudaStream_t stream) {
    return run(packed(A, B, C, M, N, K), algo, 0, stream);
}

int gemm_f32_algo_splitk(const float* A, const float* B, float* C, int M, int N, int K, int algo,
                         int splits, cudaStream_t stream) {
    return run(packed(A, B, C, M, N, K), algo, splits, stream);
}

int gemm_f32_ex(int transa, int transb, int M, int N, int K, float alpha, const float* A,
                long long lda, const float* B, long long ldb, float beta, float* C, long long ldc,
                int algo, int splits, cudaStream_t stream) {
    Problem q;
    q.M = M;
    q.N = N;
    q.K = K;
    q.A = A;
    q.lda = lda;
    q.ta = transa;
    q.B = B;
    q.ldb = ldb;
    q.tb = transb;
    q.C = C;
    q.ldc = ldc;
    q.alpha = alpha;
    q.beta = beta;
    return run(q, algo, splits, stream);
}

int gemm_f32_algo_splitk_ev(const float* A, const float* B, float* C, int M, int N, int K,
                            int algo, int splits, cudaStream_t stream, cudaEvent_t main_begin,
                            cudaEvent_t main_end) {
    return run(packed(A, B, C, M, N, K), algo, splits, stream, main_begin, main_end);
}

int gemm_f32_configured(const float* A, const float* B, float* C, int M, int N, int K,
                        const gemm_f32_config* cfg, cudaStream_t stream) {
    const int st = check_config(cfg);
    if (st != GEMM_F32_SUCCESS) return st;
    return run(packed(A, B, C, M, N, K), cfg->algo, cfg->splits, stream, nullptr, nullptr,
               cfg->tile);
}

int gemm_f32_host(const float* A, const float* B, float* C, int M, int N, int K, int algo,
                  cudaStream_t stream) {
    return run_host(A, B, C, M, N, K, algo, stream);
}

int gemm_f32_plan_config(int M, int N, int K, const gemm_f32_config* cfg, const float* A,
                         const float* B, const float* C, gemm_f32_plan_info* out) {
    // pointers are optional here: they only decide the alignment staging
    return plan_problem(packed(A, B, const_cast<float*>(C), M, N, K), cfg, out);
}

int gemm_f32_plan_ex(int transa, int transb, int M, int N, int K, const float* A, long long lda,
                     const float* B, long long ldb, const float* C, long long ldc, int algo,
                     int splits, gemm_f32_plan_info* out) {
    Problem q;
    q.M = M;
    q.N = N;
    q.K = K;
    q.A = A;
    q.lda = lda;
    q.ta = transa;
    q.B = B;
    q.ldb = ldb;
    q.tb = transb;
    q.C = const_cast<float*>(C);
    q.ldc = ldc;
    gemm_f32_config cfg;
    cfg.algo = algo;
    cfg.tile = GEMM_F32_TILE_AUTO;
    cfg.splits = splits;
    return plan_problem(q, &cfg, out);
}


int gemm_f32_plan(int M, int N, int K, int algo, int splits, const float* A, const float* B,
                  const float* C, gemm_f32_plan_info* out) {
    gemm_f32_config cfg;
    cfg.algo = algo;
    cfg.tile = GEMM_F32_TILE_AUTO;
    cfg.splits = splits;
    return gemm_f32_plan_config(M, N, K, &cfg, A, B, C, out);
}

int gemm_f32_device_status(int clear) {
    std::lock_guard<std::mutex> lock(g_mutex);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
        }
        if (major != 10 || minor != 3) return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
    }
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return static_cast<int>(e);
    // the library's own word, if its set-up has run on this device (a status
    // query never sets the device up, so it allocates nothing)
    unsigned word = 0;
    if (d.ready) {
        e = cudaMemcpy(&word, d.fault, sizeof(word), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return static_cast<int>(e);
        if (clear && word) {
            e = cudaMemset(d.fault, 0, sizeof(unsigned));
            if (e != cudaSuccess) return static_cast<int>(e);
        }
    }
    // and gemm_f32_noalloc's word, which lives in that entry point's array
    unsigned noalloc_word = 0;
    int st = noalloc_fault_word(dev, clear, &noalloc_word);
    if (st != GEMM_F32_SUCCESS) return st;
    return (word | noalloc_word) ? GEMM_F32_ERR_DEVICE_TIMEOUT : GEMM_F32_SUCCESS;
}

int gemm_f32_selftest_watchdog(long long timeout_ns, cudaStream_t stream) {
    if (timeout_ns < 1000 || timeout_ns > 10000000000LL) return GEMM_F32_ERR_INVALID_VALUE;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        DeviceState* d = nullptr;
        int dev = 0;
        int st = device_state(&d, &dev);
        if (st != GEMM_F32_SUCCESS) return st;
        cudaError_t e = launch_watchdog_selftest(d->fault, timeout_ns, stream);
        if (e != cudaSuccess) return static_cast<int>(e);
        e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return static_cast<int>(e);
    }
    return gemm_f32_device_status(1);
}

int gemm_f32_release(void) {
    std::lock_guard<std::mutex> lock(g_mutex);
    int prev = 0;
    cudaGetDevice(&prev);
    int status = GEMM_F32_SUCCESS;
    for (auto& kv : g_ws) {
        if (!kv.second.ptr) continue;
        cudaSetDevice(kv.first.first);
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess && status == GEMM_F32_SUCCESS) status = static_cast<int>(e);
        cudaFree(kv.second.ptr);
    }
    for (auto& kv : g_ws) {
        cudaSetDevice(kv.first.first);
        for (void* p : kv.second.retired) cudaFree(p);
    }
    g_ws.clear();
    for (auto& kv : g_pipes) {
        HostPipe& hp = kv.second;
        cudaSetDevice(kv.first.first);
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess && status == GEMM_F32_SUCCESS) status = static_cast<int>(e);
        if (hp.dev_buf) cudaFree(hp.dev_buf);
        for (void* p : hp.retired) cudaFree(p);
        if (hp.ready) {
            cudaStreamDestroy(hp.s_in);
            cudaStreamDestroy(hp.s_out);
            cudaEventDestroy(hp.ev_start);
            cudaEventDestroy(hp.ev_b);
            cudaEventDestroy(hp.ev_done);
            for (int i = 0; i < kMaxPanels; ++i) {
                cudaEventDestroy(hp.ev_a[i]);
                cudaEventDestroy(hp.ev_c[i]);
            }
            for (int i = 0; i < kMaxColBlocks; ++i) {
                cudaEventDestroy(hp.ev_bblk[i]);
                cudaEventDestroy(hp.ev_cblk[i]);
            }
        }
    }
    g_pipes.clear();
    cudaSetDevice(prev);
    return status;
}

const char* gemm_f32_status_string(int status) {
    switch (status) {
        case GEMM_F32_SUCCESS: return "success";
        case GEMM_F32_ERR_INVALID_VALUE: return "invalid value";
        case GEMM_F32_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
        case GEMM_F32_ERR_WORKSPACE: return "workspace allocation failed";
        case GEMM_F32_ERR_DEVICE_TIMEOUT: return "device barrier wait timed out";
        case GEMM_F32_ERR_DESCRIPTOR: return "tensor map encoding failed";
        case GEMM_F32_ERR_CAPTURE:
            return "set-up or allocation needed while the stream is captured (call once before capturing)";
        default: break;
    }
    if (status > 0) return cudaGetErrorString(static_cast<cudaError_t>(status));
    return "unknown status";
}

int gemm_f32_inject_host_fault(int kind) {
    if (kind != GEMM_F32_INJECT_NONE && kind != GEMM_F32_INJECT_WORKSPACE &&
        kind != GEMM_F32_INJECT_DESCRIPTOR)
        return GEMM_F32_ERR_INVALID_VALUE;
    g_inject.store(kind);
    return GEMM_F32_SUCCESS;
}

int gemm_f32_version(void) { return 100; }

}  // extern "C"
