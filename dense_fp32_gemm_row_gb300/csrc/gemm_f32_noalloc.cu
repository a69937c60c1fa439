// gemm_f32_noalloc.cu -- gemm_f32_noalloc(): the CUDA-core split-K GEMM
// with its scratch memory in a fixed, file-scope device array instead of
// the library's lazily grown workspace.
//
// Who needs it: some programs cannot let a library call cudaMalloc or
// cudaFree while they run.  An application that reserves its whole device
// memory budget up front and hands it out from its own pool cannot have a
// library grow a private workspace behind its back, and a latency-critical
// loop cannot afford the device-wide synchronisation that cudaFree (and the
// workspace growth that needs it) implies.  For them this entry point
// allocates nothing: its scratch (split-K partial sums, and padded copies of
// operands whose row stride TMA cannot describe) lives in g_noalloc_scratch,
// a static device array of GEMM_F32_NOALLOC_SCRATCH_BYTES that every GPU
// using the library holds until the process exits.
//
// The array's name in host code is only a host-side stand-in for the device
// symbol, so its device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) on the first call made on
// that device, and passed to the kernels.  That first call therefore does
// host-side set-up work and should be made before any stream capture
// begins.  All calls share the one array: calls whose executions overlap on
// the GPU (different streams, or several host threads) race on it and must
// be serialised by the caller.  Its first 256 bytes hold the kernels' fault
// word, cleared (and the clear waited for) at set-up; the rest is scratch
// that every call writes before it reads, so nothing else needs clearing
// between calls.  A kernel whose bounded wait gave up sets a bit in that
// word; gemm_f32_device_status() reads it (and clears it on request) beside
// the library's own word, and allocates nothing to do so.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "gemm_f32.h"
#include "gemm_internal.h"

using namespace gemm_f32_impl;

namespace {

constexpr size_t kHeaderBytes = 256;  // fault word + padding
constexpr size_t kScratchBytes = static_cast<size_t>(GEMM_F32_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kHeaderBytes + kScratchBytes];

struct NoallocDevice {
    bool ready = false;
    int sm_count = 0;
    unsigned char* base = nullptr;  // device address of g_noalloc_scratch
};

std::mutex g_noalloc_mutex;
NoallocDevice g_noalloc_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_noalloc_encode = nullptr;

long long up(long long x, long long m) { return (x + m - 1) / m * m; }

int noalloc_encode(CUtensorMap* map, const float* base, long long dim0, long long dim1,
                   long long ld, int box0, int box1, CUtensorMapSwizzle swizzle) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(dim0), static_cast<cuuint64_t>(dim1)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4u};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box0), static_cast<cuuint32_t>(box1)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_noalloc_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base),
                                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_F32_SUCCESS : GEMM_F32_ERR_DESCRIPTOR;
}

// One-time set-up for the current device; g_noalloc_mutex must be held.
// The set-up waits for work on `stream`, so it is refused while that stream
// is being captured into a graph.
int noalloc_setup(NoallocDevice** out, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
    }
    NoallocDevice& d = g_noalloc_dev[dev];
    if (!d.ready) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_F32_ERR_CAPTURE;
        }
        if (cs != cudaStreamCaptureStatusNone) return GEMM_F32_ERR_CAPTURE;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess) {
            cudaGetLastError();
            return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
        }
        if (major != 10 || minor != 3) return GEMM_F32_ERR_UNSUPPORTED_DEVICE;
        if (!g_noalloc_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn) {
                cudaGetLastError();
                return GEMM_F32_ERR_DESCRIPTOR;
            }
            g_noalloc_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return static_cast<int>(e);
        // the fault word must start at zero before any call (on any stream)
        // can use it: clear it and wait for the clear here
        e = cudaMemsetAsync(p, 0, kHeaderBytes, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return static_cast<int>(e);
        d.base = static_cast<unsigned char*>(p);
        d.ready = true;
    }
    *out = &d;
    return GEMM_F32_SUCCESS;
}

}  // namespace

namespace gemm_f32_impl {

// The no-allocation entry point's fault word on device `dev`: 0 when that
// device has not been set up by it.  Reading synchronises with the device
// (a blocking copy); `clear` zeroes a nonzero word afterwards.
int noalloc_fault_word(int dev, int clear, unsigned* word) {
    *word = 0;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (dev < 0 || dev >= kMaxDevices || !g_noalloc_dev[dev].ready) return GEMM_F32_SUCCESS;
    unsigned* fault = reinterpret_cast<unsigned*>(g_noalloc_dev[dev].base);
    cudaError_t e = cudaMemcpy(word, fault, sizeof(unsigned), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (clear && *word) {
        e = cudaMemset(fault, 0, sizeof(unsigned));
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return static_cast<int>(e);
    }
    return GEMM_F32_SUCCESS;
}

}  // namespace gemm_f32_impl

extern "C" int gemm_f32_noalloc_selftest_watchdog(long long timeout_ns, cudaStream_t stream) {
    if (timeout_ns < 1000 || timeout_ns > 10000000000LL) return GEMM_F32_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoallocDevice* d = nullptr;
    int st = noalloc_setup(&d, stream);
    if (st != GEMM_F32_SUCCESS) return st;
    unsigned* fault = reinterpret_cast<unsigned*>(d->base);
    cudaError_t e = launch_watchdog_selftest(fault, timeout_ns, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return static_cast<int>(e);
    unsigned word = 0;
    e = cudaMemcpy(&word, fault, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return static_cast<int>(e);
    // the bit stays set, as after a real timeout, until a status call clears it
    return word ? GEMM_F32_ERR_DEVICE_TIMEOUT : GEMM_F32_SUCCESS;
}

extern "C" int gemm_f32_noalloc(const float* A, const float* B, float* C, int M, int N, int K,
                                int splits, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0 || splits < 0 || splits > GEMM_F32_MAX_SPLITS)
        return GEMM_F32_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return GEMM_F32_SUCCESS;
    const size_t a_bytes = static_cast<size_t>(M) * K * 4, b_bytes = static_cast<size_t>(K) * N * 4;
    const size_t c_bytes = static_cast<size_t>(M) * N * 4;
    if (!C || (K > 0 && (!A || !B))) return GEMM_F32_ERR_INVALID_VALUE;
    auto overlap = [](const void* x, size_t xb, const void* y, size_t yb) {
        const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), y0 = reinterpret_cast<uintptr_t>(y);
        return x && y && xb && yb && x0 < y0 + yb && y0 < x0 + xb;
    };
    if (overlap(C, c_bytes, A, a_bytes) || overlap(C, c_bytes, B, b_bytes))
        return GEMM_F32_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(C) | reinterpret_cast<uintptr_t>(A) |
         reinterpret_cast<uintptr_t>(B)) & 3u)
        return GEMM_F32_ERR_INVALID_VALUE;

    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoallocDevice* d = nullptr;
    int st = noalloc_setup(&d, stream);
    if (st != GEMM_F32_SUCCESS) return st;
    if (K == 0) {
        cudaError_t e = launch_fill_zero(C, static_cast<long long>(M) * N, stream);
        return e == cudaSuccess ? GEMM_F32_SUCCESS : static_cast<int>(e);
    }

    // scratch layout after the header: [padded A][padded B][split partials]
    const FfmaConfig fc = ffma_config(0);
    const bool stage_a = (K % 4 != 0) || (reinterpret_cast<uintptr_t>(A) & 15u);
    const bool stage_b = (N % 4 != 0) || (reinterpret_cast<uintptr_t>(B) & 15u);
    const long long lda = stage_a ? up(K, 4) : K;
    const long long ldb = stage_b ? up(N, 4) : N;
    const long long ldw = up(N, 4);
    const long long bytes_a = stage_a ? up(static_cast<long long>(M) * lda * 4, 256) : 0;
    const long long bytes_b = stage_b ? up(static_cast<long long>(K) * ldb * 4, 256) : 0;
    const long long room = static_cast<long long>(kScratchBytes) - bytes_a - bytes_b;
    if (room < 0) return GEMM_F32_ERR_INVALID_VALUE;  // operand copies exceed the scratch
    const long long part_bytes = static_cast<long long>(M) * ldw * 4;

    const int tiles = ((M + fc.bm - 1) / fc.bm) * ((N + fc.bn - 1) / fc.bn);
    const int kb_total = (K + fc.bk - 1) / fc.bk;
    int s = splits;
    if (s == 0) {
        const int slots = d->sm_count * fc.ctas_per_sm;
        s = 1;
        if (tiles * 2 <= slots) {
            s = slots / tiles;
            if (s > kb_total / 4) s = kb_total / 4;
            if (s > GEMM_F32_MAX_SPLITS) s = GEMM_F32_MAX_SPLITS;
        }
        // automatic choice: as many splits as the scratch holds
        const long long fit = part_bytes > 0 ? room / part_bytes : 1;
        if (s > fit) s = static_cast<int>(fit);
        if (s < 1) s = 1;
    }
    if (s > kb_total) s = kb_total;
    const int kb_per_split = (kb_total + s - 1) / s;
    s = (kb_total + kb_per_split - 1) / kb_per_split;
    if (s > 1 && static_cast<long long>(s) * part_bytes > room)
        return GEMM_F32_ERR_INVALID_VALUE;  // requested splits exceed the scratch

    unsigned char* scratch = d->base + kHeaderBytes;
    unsigned* fault = reinterpret_cast<unsigned*>(d->base);
    const float* a_src = A;
    const float* b_src = B;
    cudaError_t e;
    if (stage_a) {
        float* dst = reinterpret_cast<float*>(scratch);
        if ((e = launch_pad_copy(A, K, M, K, dst, lda, stream)) != cudaSuccess)
            return static_cast<int>(e);
        a_src = dst;
    }
    if (stage_b) {
        float* dst = reinterpret_cast<float*>(scratch + bytes_a);
        if ((e = launch_pad_copy(B, N, K, N, dst, ldb, stream)) != cudaSuccess)
            return static_cast<int>(e);
        b_src = dst;
    }
    FfmaArgs fa;
    std::memset(&fa, 0, sizeof(fa));
    if ((st = noalloc_encode(&fa.tmA, a_src, K, M, lda, fc.bk, fc.bm,
                             CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM_F32_SUCCESS ||
        (st = noalloc_encode(&fa.tmB, b_src, N, K, ldb, fc.bn, fc.bk,
                             CU_TENSOR_MAP_SWIZZLE_NONE)) != GEMM_F32_SUCCESS)
        return st;
    float* parts = reinterpret_cast<float*>(scratch + bytes_a + bytes_b);
    fa.M = M;
    fa.N = N;
    fa.K = K;
    fa.kb_per_split = kb_per_split;
    fa.splits = s;
    fa.fault = fault;
    fa.timeout_ns = kDefaultTimeoutNs;
    fa.variant = 0;
    fa.bn = fc.bn;
    if (s > 1) {
        fa.out = parts;
        fa.ldo = ldw;
        fa.split_stride = static_cast<long long>(M) * ldw;
    } else {
        fa.out = C;
        fa.ldo = N;
        fa.split_stride = 0;
    }
    fa.vec_store = (fa.ldo % 4 == 0) && !(reinterpret_cast<uintptr_t>(fa.out) & 15u);
    if ((e = launch_sgemm_ffma(fa, stream)) != cudaSuccess) return static_cast<int>(e);
    if (s > 1 &&
        (e = launch_splitk_reduce(parts, fa.split_stride, ldw, s, C, N, M, N, 1.0f, 0.0f, 0,
                                  stream)) != cudaSuccess)
        return static_cast<int>(e);
    return GEMM_F32_SUCCESS;
}
