// fp32 Newton-Schulz phases on CUDA cores, for the reference-accuracy mode.
//
// One 64 x 64 output tile per CTA, 256 threads each owning a 4 x 4 block, K
// staged through shared memory 16 at a time.  Operands of each phase, for
// D(i, j) = sum_k P(i, k) Q(k, j):
//   kGram   P = X (m x n), Q(k, j) = X(j, k)      K = n
//   kPoly   P = A,         Q = A                  K = m
//   kApply  P = B,         Q = X                  K = m
// The epilogues match the tensor-core path; in this mode the operand buffer
// is the fp32 iterate itself (x_op[step & 1]; x_op[0] holds M unscaled).
#include <cuda_bf16.h>

#include "internal.h"

namespace mo {

using bf16 = __nv_bfloat16;

namespace {

__device__ __forceinline__ float uload(const void* p, int dt, int64_t off) {
    return dt == MO_F32 ? static_cast<const float*>(p)[off] : __bfloat162float(static_cast<const bf16*>(p)[off]);
}
__device__ __forceinline__ void ustore(void* p, int dt, int64_t off, float v) {
    if (dt == MO_F32)
        static_cast<float*>(p)[off] = v;
    else
        static_cast<bf16*>(p)[off] = __float2bfloat16_rn(v);
}

}  // namespace

__global__ void __launch_bounds__(256) ns_fp32_kernel(const __grid_constant__ NsLaunch p) {
    __shared__ float Ps[kFpBK][kFpBM + 4];
    __shared__ float Qs[kFpBK][kFpBN + 4];
    const TileDesc td = p.tiles[blockIdx.x];
    const MatDesc& md = p.mats[td.mat];
    const int m = md.m, n = md.n;
    const int i0 = td.ti * kFpBM, j0 = td.tj * kFpBN;
    const float* X = static_cast<const float*>(md.x_op[p.step & 1]);
    const float* A = static_cast<const float*>(md.gram);
    const float* B = static_cast<const float*>(md.poly);

    const float* P;
    const float* Q;
    int64_t ldp, ldq;
    int K, jlim;
    bool q_k_contig;   // Q(k, j) stored with k contiguous (Q(k, j) = base[j*ld + k])
    if (p.phase == kGram) {
        P = X; ldp = md.ldx; Q = X; ldq = md.ldx; K = n; jlim = m; q_k_contig = true;
    } else if (p.phase == kPoly) {
        P = A; ldp = md.lda; Q = A; ldq = md.lda; K = m; jlim = m; q_k_contig = false;
    } else {
        P = B; ldp = md.lda; Q = X; ldq = md.ldx; K = m; jlim = n; q_k_contig = false;
    }

    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;

    for (int k0 = 0; k0 < K; k0 += kFpBK) {
        // P tile: rows i0..i0+63, k0..k0+15, k contiguous in memory
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = threadIdx.x + 256 * q;
            const int ii = e >> 4, kk = e & 15;
            const int i = i0 + ii, k = k0 + kk;
            Ps[kk][ii] = (i < m && k < K) ? P[static_cast<int64_t>(i) * ldp + k] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = threadIdx.x + 256 * q;
            if (q_k_contig) {
                const int jj = e >> 4, kk = e & 15;
                const int j = j0 + jj, k = k0 + kk;
                Qs[kk][jj] = (j < jlim && k < K) ? Q[static_cast<int64_t>(j) * ldq + k] : 0.f;
            } else {
                const int kk = e >> 6, jj = e & 63;
                const int j = j0 + jj, k = k0 + kk;
                Qs[kk][jj] = (j < jlim && k < K) ? Q[static_cast<int64_t>(k) * ldq + j] : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kFpBK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) a[r] = Ps[kk][ty * 4 + r];
#pragma unroll
            for (int c = 0; c < 4; ++c) b[c] = Qs[kk][tx * 4 + c];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
        }
        __syncthreads();
    }

    const bool last = p.step + 1 >= p.steps;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = i0 + ty * 4 + r;
        if (i >= m) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int j = j0 + tx * 4 + c;
            if (j >= jlim) continue;
            const float v = acc[r][c];
            if (p.phase == kGram) {
                float* G = static_cast<float*>(md.gram);
                G[static_cast<int64_t>(i) * md.lda + j] = v * (p.step == 0 ? md.scales[1] : 1.f);
            } else if (p.phase == kPoly) {
                float* Bw = static_cast<float*>(md.poly);
                const int64_t o = static_cast<int64_t>(i) * md.lda + j;
                Bw[o] = fmaf(p.c, v, p.b * A[o]);
            } else {
                const int64_t o = static_cast<int64_t>(i) * md.ldx + j;
                float x = X[o];
                x = p.step == 0 ? md.scales[0] * fmaf(p.a, x, v) : fmaf(p.a, x, v);
                if (!last) {
                    static_cast<float*>(md.x_op[(p.step + 1) & 1])[o] = x;
                } else {
                    const int64_t uo = md.transposed ? static_cast<int64_t>(j) * md.ld + i
                                                     : static_cast<int64_t>(i) * md.ld + j;
                    if (p.apply_update) {
                        if (md.W != nullptr) {
                            const float w = uload(md.W, md.w_dtype, uo);
                            ustore(md.W, md.w_dtype, uo, fmaf(-p.alpha, x, w - p.decay * w));
                        }
                    } else if (md.out != nullptr) {
                        ustore(md.out, md.out_dtype, uo, x);
                    }
                }
            }
        }
    }
}

cudaError_t launch_ns_fp32_phase(const NsLaunch& p, int grid, cudaStream_t s) {
    if (grid <= 0) return cudaSuccess;
    ns_fp32_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mo
