// epilogue.cuh -- the output step shared by the GEMM kernels and the split-K
// reduction: C = v (mode 0), C = alpha v (mode 1) or C = alpha v + beta C
// (mode 2; only this mode reads C), for four consecutive columns, as one
// 16-byte store when the row allows it and predicated scalar stores on a
// ragged edge.  Nothing outside the first `N` columns is touched.
#pragma once

namespace gemm_f32_dev {

constexpr int kStorePlain = 0;
constexpr int kStoreAlpha = 1;
constexpr int kStoreAlphaBeta = 2;

__device__ __forceinline__ float scale1(float v, const float* old, float alpha, float beta,
                                        int mode) {
    if (mode == kStorePlain) return v;
    const float a = alpha * v;
    return mode == kStoreAlphaBeta ? fmaf(beta, *old, a) : a;
}

// row points at column 0 of the output row; columns n .. n+3 of v.
__device__ __forceinline__ void store4(float* row, int n, int N, float4 v, bool vec, float alpha,
                                       float beta, int mode) {
    if (vec && n + 3 < N) {
        float4* p = reinterpret_cast<float4*>(row + n);
        if (mode != kStorePlain) {
            v.x *= alpha;
            v.y *= alpha;
            v.z *= alpha;
            v.w *= alpha;
            if (mode == kStoreAlphaBeta) {
                const float4 o = *p;
                v.x = fmaf(beta, o.x, v.x);
                v.y = fmaf(beta, o.y, v.y);
                v.z = fmaf(beta, o.z, v.z);
                v.w = fmaf(beta, o.w, v.w);
            }
        }
        *p = v;
    } else {
        const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (n + i < N) row[n + i] = scale1(e[i], row + n + i, alpha, beta, mode);
    }
}

}  // namespace gemm_f32_dev
