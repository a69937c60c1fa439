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

#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/gemm_f32.h"
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
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
EncodeTiledFn g_encode = nullptr;

long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

bool misaligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes) {
    if (!a || !b || abytes == 0 || bbytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// Device lookup; g_mutex must be held.
int device_state(DeviceState** out, int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
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
    if (w.bytes < bytes) {
        if (w.ptr) {
            // earlier calls on this stream may still read the old buffer
            cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return static_cast<int>(e);
            cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
        }
        const size_t grow = static_cast<size_t>(round_up(static_cast<long long>(bytes), 1 << 20));
        if (cudaMalloc(&w.ptr, grow) != cudaSuccess) {
            cudaGetLastError();
            w.ptr = nullptr;
            return GEMM_F32_ERR_WORKSPACE;
        }
        w.bytes = grow;
    }
    *out = w.ptr;
    return GEMM_F32_SUCCESS;
}

struct Plan {
    int algo = 0;
    int splits = 1;
    int kb_per_split = 0;
    int stage_a = 0, stage_b = 0;
    long long lda = 0, ldb = 0;   // row strides the kernel reads (elements)
    long long ldw = 0;            // split-K partial row stride
    size_t off_a = 0, off_b = 0, off_w = 0, ws_bytes = 0;
    int tile_m = 0, tile_n = 0, tile_k = 0, stages = 0, ctas = 0, kernels = 0;
};

int validate(const float* A, const float* B, const float* C, int M, int N, int K, int algo,
             int splits, bool need_ptrs = true) {
    if (M < 0 || N < 0 || K < 0) return GEMM_F32_ERR_INVALID_VALUE;
    if (algo < GEMM_F32_ALGO_AUTO || algo > GEMM_F32_ALGO_3XTF32) return GEMM_F32_ERR_INVALID_VALUE;
    if (splits < 0 || splits > GEMM_F32_MAX_SPLITS) return GEMM_F32_ERR_INVALID_VALUE;
    const size_t a_bytes = static_cast<size_t>(M) * static_cast<size_t>(K) * 4u;
    const size_t b_bytes = static_cast<size_t>(K) * static_cast<size_t>(N) * 4u;
    const size_t c_bytes = static_cast<size_t>(M) * static_cast<size_t>(N) * 4u;
    if (M > 0 && N > 0) {
        if (need_ptrs && !C) return GEMM_F32_ERR_INVALID_VALUE;
        if (need_ptrs && K > 0 && (!A || !B)) return GEMM_F32_ERR_INVALID_VALUE;
        if (overlaps(C, c_bytes, A, a_bytes) || overlaps(C, c_bytes, B, b_bytes))
            return GEMM_F32_ERR_INVALID_VALUE;
        if ((reinterpret_cast<uintptr_t>(C) & 3u) || (A && (reinterpret_cast<uintptr_t>(A) & 3u)) ||
            (B && (reinterpret_cast<uintptr_t>(B) & 3u)))
            return GEMM_F32_ERR_INVALID_VALUE;
    }
    return GEMM_F32_SUCCESS;
}

void make_plan(const DeviceState& d, const float* A, const float* B, int M, int N, int K, int algo,
               int splits, Plan* p) {
    const FfmaConfig fc = ffma_config();
    p->algo = (algo == GEMM_F32_ALGO_AUTO) ? GEMM_F32_ALGO_FFMA : algo;
    p->tile_m = fc.bm;
    p->tile_n = fc.bn;
    p->tile_k = fc.bk;
    p->stages = fc.stages;
    const int tiles = ((M + fc.bm - 1) / fc.bm) * ((N + fc.bn - 1) / fc.bn);
    const int kb_total = (K + fc.bk - 1) / fc.bk;
    int s = splits;
    if (s == 0) {
        const int slots = d.sm_count * fc.ctas_per_sm;
        s = 1;
        if (tiles * 2 <= slots) {
            s = slots / tiles;
            const int max_by_depth = kb_total / 4;  // keep >= 4 K blocks per split
            if (s > max_by_depth) s = max_by_depth;
            if (s > GEMM_F32_MAX_SPLITS) s = GEMM_F32_MAX_SPLITS;
            if (s < 1) s = 1;
        }
    }
    if (s > kb_total) s = kb_total;
    if (s < 1) s = 1;
    p->kb_per_split = (kb_total + s - 1) / s;
    p->splits = (kb_total + p->kb_per_split - 1) / p->kb_per_split;
    p->ctas = tiles * p->splits;

    p->stage_a = (K % 4 != 0) || misaligned16(A);
    p->stage_b = (N % 4 != 0) || misaligned16(B);
    p->lda = p->stage_a ? round_up(K, 4) : K;
    p->ldb = p->stage_b ? round_up(N, 4) : N;
    p->ldw = round_up(N, 4);
    size_t off = 0;
    if (p->stage_a) {
        p->off_a = off;
        off += static_cast<size_t>(round_up(static_cast<long long>(M) * p->lda * 4, 256));
    }
    if (p->stage_b) {
        p->off_b = off;
        off += static_cast<size_t>(round_up(static_cast<long long>(K) * p->ldb * 4, 256));
    }
    if (p->splits > 1) {
        p->off_w = off;
        off += static_cast<size_t>(
            round_up(static_cast<long long>(p->splits) * M * p->ldw * 4, 256));
    }
    p->ws_bytes = off;
    p->kernels = 1 + p->stage_a + p->stage_b + (p->splits > 1 ? 1 : 0);
}

int run(const float* A, const float* B, float* C, int M, int N, int K, int algo, int splits,
        cudaStream_t stream, cudaEvent_t ev_begin = nullptr, cudaEvent_t ev_end = nullptr) {
    int st = validate(A, B, C, M, N, K, algo, splits);
    if (st != GEMM_F32_SUCCESS) return st;
    if (algo == GEMM_F32_ALGO_3XTF32) return GEMM_F32_ERR_INVALID_VALUE;  // not built yet
    if (M == 0 || N == 0) return GEMM_F32_SUCCESS;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* d = nullptr;
    int dev = 0;
    st = device_state(&d, &dev);
    if (st != GEMM_F32_SUCCESS) return st;

    if (K == 0) {
        cudaError_t e = launch_fill_zero(C, static_cast<long long>(M) * N, stream);
        return e == cudaSuccess ? GEMM_F32_SUCCESS : static_cast<int>(e);
    }

    st = get_encoder();
    if (st != GEMM_F32_SUCCESS) return st;

    Plan p;
    make_plan(*d, A, B, M, N, K, algo, splits, &p);

    unsigned char* ws = nullptr;
    if (p.ws_bytes) {
        void* w = nullptr;
        st = workspace(dev, stream, p.ws_bytes, &w);
        if (st != GEMM_F32_SUCCESS) return st;
        ws = static_cast<unsigned char*>(w);
    }

    const float* a_src = A;
    const float* b_src = B;
    cudaError_t e = cudaSuccess;
    if (p.stage_a) {
        float* dst = reinterpret_cast<float*>(ws + p.off_a);
        e = launch_pad_copy(A, K, M, K, dst, p.lda, stream);
        if (e != cudaSuccess) return static_cast<int>(e);
        a_src = dst;
    }
    if (p.stage_b) {
        float* dst = reinterpret_cast<float*>(ws + p.off_b);
        e = launch_pad_copy(B, N, K, N, dst, p.ldb, stream);
        if (e != cudaSuccess) return static_cast<int>(e);
        b_src = dst;
    }

    const FfmaConfig fc = ffma_config();
    FfmaArgs fa;
    std::memset(&fa, 0, sizeof(fa));
    st = encode_2d(&fa.tmA, a_src, K, M, p.lda, fc.bk, fc.bm, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != GEMM_F32_SUCCESS) return st;
    st = encode_2d(&fa.tmB, b_src, N, K, p.ldb, fc.bn, fc.bk, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != GEMM_F32_SUCCESS) return st;
    fa.M = M;
    fa.N = N;
    fa.K = K;
    fa.kb_per_split = p.kb_per_split;
    fa.splits = p.splits;
    fa.fault = d->fault;
    fa.timeout_ns = kDefaultTimeoutNs;
    if (p.splits > 1) {
        fa.out = reinterpret_cast<float*>(ws + p.off_w);
        fa.ldo = p.ldw;
        fa.split_stride = static_cast<long long>(M) * p.ldw;
    } else {
        fa.out = C;
        fa.ldo = N;
        fa.split_stride = 0;
    }
    fa.vec_store = (fa.ldo % 4 == 0) && !misaligned16(fa.out);
    if (ev_begin && (e = cudaEventRecord(ev_begin, stream)) != cudaSuccess) return static_cast<int>(e);
    e = launch_sgemm_ffma(fa, stream);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (ev_end && (e = cudaEventRecord(ev_end, stream)) != cudaSuccess) return static_cast<int>(e);
    if (p.splits > 1) {
        e = launch_splitk_reduce(fa.out, fa.split_stride, p.ldw, p.splits, C, N, M, N, stream);
        if (e != cudaSuccess) return static_cast<int>(e);
    }
    return GEMM_F32_SUCCESS;
}

}  // namespace

extern "C" {

int gemm_f32(const float* A, const float* B, float* C, int M, int N, int K, cudaStream_t stream) {
    return run(A, B, C, M, N, K, GEMM_F32_ALGO_AUTO, 0, stream);
}

int gemm_f32_algo(const float* A, const float* B, float* C, int M, int N, int K, int algo,
                  cudaStream_t stream) {
    return run(A, B, C, M, N, K, algo, 0, stream);
}

int gemm_f32_algo_splitk(const float* A, const float* B, float* C, int M, int N, int K, int algo,
                         int splits, cudaStream_t stream) {
    return run(A, B, C, M, N, K, algo, splits, stream);
}

int gemm_f32_algo_splitk_ev(const float* A, const float* B, float* C, int M, int N, int K,
                            int algo, int splits, cudaStream_t stream, cudaEvent_t main_begin,
                            cudaEvent_t main_end) {
    return run(A, B, C, M, N, K, algo, splits, stream, main_begin, main_end);
}

int gemm_f32_plan(int M, int N, int K, int algo, int splits, const float* A, const float* B,
                  const float* C, gemm_f32_plan_info* out) {
    if (!out) return GEMM_F32_ERR_INVALID_VALUE;
    std::memset(out, 0, sizeof(*out));
    // pointers are optional here: they only decide the alignment staging
    int st = validate(A, B, C, M, N, K, algo, splits, false);
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
    make_plan(*d, A, B, M, N, K, algo, splits, &p);
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
    return GEMM_F32_SUCCESS;
}

int gemm_f32_device_status(int clear) {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* d = nullptr;
    int dev = 0;
    int st = device_state(&d, &dev);
    if (st != GEMM_F32_SUCCESS) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return static_cast<int>(e);
    unsigned word = 0;
    e = cudaMemcpy(&word, d->fault, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (clear && word) {
        e = cudaMemset(d->fault, 0, sizeof(unsigned));
        if (e != cudaSuccess) return static_cast<int>(e);
    }
    return word ? GEMM_F32_ERR_DEVICE_TIMEOUT : GEMM_F32_SUCCESS;
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
    g_ws.clear();
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
        default: break;
    }
    if (status > 0) return cudaGetErrorString(static_cast<cudaError_t>(status));
    return "unknown status";
}

int gemm_f32_version(void) { return 100; }

}  // extern "C"
