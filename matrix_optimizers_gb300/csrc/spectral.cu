// Spectral-scale normalisation for the Newton-Schulz step.
//
// With spectral scaling the iteration starts from X0 = F / sigma_hat, F =
// X/||X||_F, where sigma_hat is estimated by q power iterations on the Gram
// matrix A = F F^T that the first Gram phase has just written (bf16, m x m):
//   v0 = ones/sqrt(m);  repeat q times: y = A v, v = y/||y||;  lambda = v^T A v.
// Nothing is rescaled in memory: with lambda = sigma_hat^2 the first step's
// polynomial uses b/lambda and c/lambda^2, and its apply scales by
// 1/sqrt(lambda), which the epilogues read from the per-matrix scales
// (scales[2..4]; 1 under Frobenius scaling).
//
//   power_init       v = 1/sqrt(m) for every matrix
//   power_matvec     y = A v, one warp per row over the rows of all matrices
//   power_normalize  one CTA per matrix: v = y/||y||, or on the last call
//                    lambda = v.y and the folded scales
// All reductions run in a fixed order, so the estimate is deterministic.
#include <cuda_bf16.h>

#include "internal.h"

namespace mo {

using bf16 = __nv_bfloat16;

namespace {

__device__ __forceinline__ int find_by_row(const MatDesc* mats, int nmats, int64_t row) {
    int lo = 0, hi = nmats - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (mats[mid].row_begin <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(256) power_init_kernel(const MatDesc* mats) {
    const MatDesc& md = mats[blockIdx.x];
    const float v0 = rsqrtf(static_cast<float>(md.m));
    for (int i = threadIdx.x; i < md.m; i += blockDim.x) md.pv[i] = v0;
}

__global__ void __launch_bounds__(256) power_matvec_kernel(const MatDesc* mats, int nmats, int64_t total_rows) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t row = warp; row < total_rows; row += nwarps) {
        const MatDesc& md = mats[find_by_row(mats, nmats, row)];
        const int i = static_cast<int>(row - md.row_begin), m = md.m;
        const bf16* a = static_cast<const bf16*>(md.gram) + static_cast<int64_t>(i) * md.lda;
        float acc = 0.f;
        for (int k = lane * 8; k < m; k += 256) {
            if (k + 8 <= m) {
                const uint4 u = *reinterpret_cast<const uint4*>(a + k);
                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
                const float4 v0 = *reinterpret_cast<const float4*>(md.pv + k);
                const float4 v1 = *reinterpret_cast<const float4*>(md.pv + k + 4);
                acc = fmaf(__low2float(h[0]), v0.x, acc);
                acc = fmaf(__high2float(h[0]), v0.y, acc);
                acc = fmaf(__low2float(h[1]), v0.z, acc);
                acc = fmaf(__high2float(h[1]), v0.w, acc);
                acc = fmaf(__low2float(h[2]), v1.x, acc);
                acc = fmaf(__high2float(h[2]), v1.y, acc);
                acc = fmaf(__low2float(h[3]), v1.z, acc);
                acc = fmaf(__high2float(h[3]), v1.w, acc);
            } else {
                for (int q = k; q < m; ++q) acc = fmaf(__bfloat162float(a[q]), md.pv[q], acc);
            }
        }
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) md.py[i] = acc;
    }
}

__device__ __forceinline__ float block_sum(float v, float* red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) s += red[w];
    __syncthreads();
    return s;
}

__global__ void __launch_bounds__(256) power_normalize_kernel(const MatDesc* mats, int final_call) {
    __shared__ float red[8];
    const MatDesc& md = mats[blockIdx.x];
    float ss = 0.f, vy = 0.f;
    for (int i = threadIdx.x; i < md.m; i += blockDim.x) {
        const float y = md.py[i];
        ss = fmaf(y, y, ss);
        vy = fmaf(md.pv[i], y, vy);
    }
    ss = block_sum(ss, red);
    vy = block_sum(vy, red);
    if (!final_call) {
        const float inv = ss > 0.f ? 1.f / sqrtf(ss) : 0.f;
        for (int i = threadIdx.x; i < md.m; i += blockDim.x) md.pv[i] = md.py[i] * inv;
    } else if (threadIdx.x == 0) {
        // lambda = v^T A v with ||v|| = 1 estimates sigma_max(F)^2
        const float lam = vy;
        if (lam > 0.f) {
            md.scales[2] = 1.f / lam;
            md.scales[3] = 1.f / (lam * lam);
            md.scales[4] = 1.f / sqrtf(lam);
        }
    }
}

}  // namespace

cudaError_t launch_spectral_estimate(const MatDesc* mats, int nmats, int64_t total_rows, int iters, int sm_count,
                                     cudaStream_t s) {
    if (nmats == 0 || iters <= 0) return cudaSuccess;
    power_init_kernel<<<nmats, 256, 0, s>>>(mats);
    int64_t blocks = (total_rows + 7) / 8;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    for (int t = 0; t <= iters; ++t) {
        power_matvec_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(mats, nmats, total_rows);
        power_normalize_kernel<<<nmats, 256, 0, s>>>(mats, t == iters ? 1 : 0);
    }
    return cudaGetLastError();
}

}  // namespace mo
