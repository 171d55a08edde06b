// HBM-bound kernels of the Muon owner step:
//   momentum_norm  M <- mu*M + G, per-tile sum of squares, NS operand written
//                  in the oriented (m <= n) frame;
//   norm_finalize  per-matrix 1/||X||_F and 1/||X||_F^2 from the tile sums;
//   ns_k0          O = X/||X||_F applied directly when the step count is 0;
//   sign_pack      sign -> 1 bit per element -> uint32 words (warp ballot);
//   vote_update    popcount majority over M packed buffers fused with W -= lr*vote;
//   adamw          vectorised AdamW on the flat float32 tail.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "internal.h"
#include "ptx.cuh"

namespace mo {

namespace {
// Resident blocks per SM of `kernel` at `threads` threads (queried once per
// kernel and device); 1 if the query fails.  Grids of the one-pass
// streaming kernels are sized to a single resident wave.
template <typename K>
int resident_blocks_per_sm(K kernel, int threads) {
    // keyed by the kernel itself: kernels of one signature share a pointer type
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const auto key = std::make_tuple(reinterpret_cast<const void*>(kernel), dev, threads);
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = n;
    return n;
}
}  // namespace

using bf16 = __nv_bfloat16;

__device__ __forceinline__ float load_elem(const void* p, int dt, int64_t i) {
    return dt == MO_F32 ? static_cast<const float*>(p)[i]
                        : __bfloat162float(static_cast<const bf16*>(p)[i]);
}
__device__ __forceinline__ void store_elem(void* p, int dt, int64_t i, float v) {
    if (dt == MO_F32)
        static_cast<float*>(p)[i] = v;
    else
        static_cast<bf16*>(p)[i] = __float2bfloat16_rn(v);
}
// Loads up to 4 consecutive elements; a full group uses one vector access
// (16-byte for f32, 8-byte for bf16; callers keep offsets 4-aligned).
__device__ __forceinline__ void load4(const void* p, int dt, int64_t off, int nvalid, float v[4]) {
    if (nvalid == 4) {
        if (dt == MO_F32) {
            float4 x = *reinterpret_cast<const float4*>(static_cast<const float*>(p) + off);
            v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
        } else {
            uint2 x = *reinterpret_cast<const uint2*>(static_cast<const bf16*>(p) + off);
            __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162*>(&x.x);
            __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162*>(&x.y);
            v[0] = __low2float(lo); v[1] = __high2float(lo);
            v[2] = __low2float(hi); v[3] = __high2float(hi);
        }
    } else {
        for (int k = 0; k < 4; ++k) v[k] = k < nvalid ? load_elem(p, dt, off + k) : 0.f;
    }
}
__device__ __forceinline__ void store4(void* p, int dt, int64_t off, int nvalid, const float v[4]) {
    if (nvalid == 4) {
        if (dt == MO_F32) {
            *reinterpret_cast<float4*>(static_cast<float*>(p) + off) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
            __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
            uint2 x;
            x.x = *reinterpret_cast<uint32_t*>(&lo);
            x.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(static_cast<bf16*>(p) + off) = x;
        }
    } else {
        for (int k = 0; k < nvalid; ++k) store_elem(p, dt, off + k, v[k]);
    }
}

__device__ __forceinline__ int find_matrix(const MatDesc* mats, int nmats, int64_t t) {
    int lo = 0, hi = nmats - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (mats[mid].mom_tile_begin <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ float block_sum_256(float v, float* red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.f;
    if (threadIdx.x == 0)
        for (int w = 0; w < 8; ++w) s += red[w];
    __syncthreads();
    return s;
}

// Element (i, j) of the NS operand: fp32 row-major (leading dimension ldx),
// or bf16 in 8-column blocks of xrows rows.
__device__ __forceinline__ int64_t xop_offset(const MatDesc& md, bool fp32, int i, int j) {
    return fp32 ? static_cast<int64_t>(i) * md.ldx + j
                : (static_cast<int64_t>(j >> 3) * md.xrows + i) * 8 + (j & 7);
}

// ------------------------------------------------------------ momentum_norm
// Tile of 64 x 64 user elements per iteration, 256 threads: thread t owns
// columns 4*(t%16)..+3 of rows t/16 + 16q, q = 0..3.
__global__ void __launch_bounds__(256, 8) momentum_norm_kernel(MomLaunch p) {
    __shared__ float tileT[kMomTile][kMomTile + 1];
    __shared__ float red[8];
    const int col4 = threadIdx.x & 15, rsub = threadIdx.x >> 4;
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const MatDesc& md = p.mats[find_matrix(p.mats, p.nmats, t)];
        const int64_t local = t - md.mom_tile_begin;
        const int r0 = static_cast<int>(local / md.mom_tiles_c) * kMomTile;
        const int c0 = static_cast<int>(local % md.mom_tiles_c) * kMomTile;
        const int c = c0 + 4 * col4;
        const int nvalid = max(0, min(4, md.cols - c));
        const int op_dt = p.fp32_operand ? MO_F32 : MO_BF16;
        float ss = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int rl = rsub + 16 * q, r = r0 + rl;
            float x[4] = {0.f, 0.f, 0.f, 0.f};
            if (r < md.rows && nvalid > 0) {
                const int64_t off = static_cast<int64_t>(r) * md.ld + c;
                float s[4];
                load4(md.src, md.src_dtype, off, nvalid, s);
                if (md.has_momentum) {
                    float g[4];
                    load4(md.grad, md.g_dtype, off, nvalid, g);
#pragma unroll
                    for (int k = 0; k < 4; ++k) x[k] = fmaf(p.mu, s[k], g[k]);
                    if (md.src_dtype == MO_BF16) {   // stored momentum is the bf16 value
#pragma unroll
                        for (int k = 0; k < 4; ++k) x[k] = __bfloat162float(__float2bfloat16_rn(x[k]));
                    }
                    store4(md.src, md.src_dtype, off, nvalid, x);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) x[k] = s[k];
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) ss = fmaf(x[k], x[k], ss);
                if (!md.transposed)
                    store4(md.x_op[0], op_dt, xop_offset(md, p.fp32_operand, r, c), nvalid, x);
            }
            if (md.transposed) {
#pragma unroll
                for (int k = 0; k < 4; ++k) tileT[4 * col4 + k][rl] = x[k];
            }
        }
        if (md.transposed) {
            __syncthreads();
            // through the tile transpose: oriented row xr = user column
            // c0 + xr, oriented columns = user rows r0 + seg .. +15
            void* dst = md.x_op[0];
            const int dt = op_dt;
            const int xr = threadIdx.x >> 2, seg = (threadIdx.x & 3) * 16;
            const int orow = c0 + xr;
            if (orow < md.cols && !p.fp32_operand) {
                // bf16 operand in 8-column blocks: each thread writes whole
                // 16-byte runs (8 consecutive oriented columns of one row), so
                // a warp stores four full 128-byte lines per instruction
#pragma unroll
                for (int g8 = 0; g8 < 2; ++g8) {
                    const int ocol = r0 + seg + 8 * g8;
                    const int nv = max(0, min(8, md.rows - ocol));
                    if (nv > 0) {
                        bf16* d = static_cast<bf16*>(dst) + xop_offset(md, false, orow, ocol);
                        const float* v = &tileT[xr][seg + 8 * g8];
                        if (nv == 8) {
                            uint4 u;
                            uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
                                w[q] = *reinterpret_cast<uint32_t*>(&h);
                            }
                            *reinterpret_cast<uint4*>(d) = u;
                        } else {
                            for (int k = 0; k < nv; ++k) d[k] = __float2bfloat16_rn(v[k]);
                        }
                    }
                }
            } else if (orow < md.cols) {
#pragma unroll
                for (int g4 = 0; g4 < 4; ++g4) {
                    const int ocol = r0 + seg + 4 * g4;
                    const int nv = max(0, min(4, md.rows - ocol));
                    if (nv > 0) {
                        float v[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) v[k] = tileT[xr][seg + 4 * g4 + k];
                        store4(dst, dt, xop_offset(md, p.fp32_operand, orow, ocol), nv, v);
                    }
                }
            }
        }
        const float total = block_sum_256(ss, red);   // also orders tileT reuse
        if (threadIdx.x == 0) p.partials[t] = total;
    }
}

// Momentum stored in bf16 with an fp32 gradient, untransposed, bf16 operand
// (the Sign-Muon workers): 8 consecutive columns per thread, so each of its
// accesses is one 16-byte run (the momentum, the operand's 8-column block
// row) or two (the gradient), where the general kernel's 4 columns of bf16
// give 8-byte momentum accesses.  The host picks this kernel only when every
// matrix of the call qualifies: bf16 momentum, fp32 gradient, rows <= cols,
// ld a multiple of 8 and 16-byte aligned momentum and gradient.
// Tile of 64 x 64 as above; thread t owns columns 8*(t%8)..+7 of rows
// t/8 + 32q, q = 0, 1.  The tile's sum of squares runs in this fixed order.
__global__ void __launch_bounds__(256, 6) momentum_norm_bf16m_kernel(MomLaunch p) {
    __shared__ float red[8];
    const int col8 = threadIdx.x & 7, rsub = threadIdx.x >> 3;
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const MatDesc& md = p.mats[find_matrix(p.mats, p.nmats, t)];
        const int64_t local = t - md.mom_tile_begin;
        const int r0 = static_cast<int>(local / md.mom_tiles_c) * kMomTile;
        const int c0 = static_cast<int>(local % md.mom_tiles_c) * kMomTile;
        const int c = c0 + 8 * col8;
        const int nvalid = max(0, min(8, md.cols - c));
        float ss = 0.f;
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
            const int r = r0 + rsub + 32 * q;
            if (r >= md.rows || nvalid <= 0) continue;
            const int64_t off = static_cast<int64_t>(r) * md.ld + c;
            float x[8];
            if (nvalid == 8) {
                const uint4 mv = *reinterpret_cast<const uint4*>(static_cast<const bf16*>(md.src) + off);
                const float4 g0 = *reinterpret_cast<const float4*>(static_cast<const float*>(md.grad) + off);
                const float4 g1 = *reinterpret_cast<const float4*>(static_cast<const float*>(md.grad) + off + 4);
                const __nv_bfloat162* mh = reinterpret_cast<const __nv_bfloat162*>(&mv);
                const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                uint4 xv;
                uint32_t* xw = reinterpret_cast<uint32_t*>(&xv);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(fmaf(p.mu, __low2float(mh[q]), g[2 * q]),
                                                                   fmaf(p.mu, __high2float(mh[q]), g[2 * q + 1]));
                    xw[q] = *reinterpret_cast<const uint32_t*>(&h);
                    x[2 * q] = __low2float(h);
                    x[2 * q + 1] = __high2float(h);
                }
                *reinterpret_cast<uint4*>(static_cast<bf16*>(md.src) + off) = xv;
                *reinterpret_cast<uint4*>(static_cast<bf16*>(md.x_op[0]) + xop_offset(md, false, r, c)) = xv;
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    x[k] = 0.f;
                    if (k < nvalid) {
                        const float m = load_elem(md.src, MO_BF16, off + k);
                        const float g = load_elem(md.grad, MO_F32, off + k);
                        x[k] = __bfloat162float(__float2bfloat16_rn(fmaf(p.mu, m, g)));
                        store_elem(md.src, MO_BF16, off + k, x[k]);
                        store_elem(md.x_op[0], MO_BF16, xop_offset(md, false, r, c + k), x[k]);
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) ss = fmaf(x[k], x[k], ss);
        }
        const float total = block_sum_256(ss, red);
        if (threadIdx.x == 0) p.partials[t] = total;
    }
}

cudaError_t launch_momentum_norm_bf16m(const MomLaunch& p, int grid, cudaStream_t s) {
    if (p.ntiles == 0) return cudaSuccess;
    momentum_norm_bf16m_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_momentum_norm(const MomLaunch& p, int grid, cudaStream_t s) {
    if (p.ntiles == 0) return cudaSuccess;
    momentum_norm_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

// ------------------------------------------------------------ norm_finalize
// One block of 256 threads per matrix sums its tile partials in a fixed order
// (float64): thread k takes partials k, k + 256, ... in turn, then a fixed
// pairwise tree combines the 256 sums.  One warp per matrix would wait on
// 32 rounds of L2 loads for a 2048 x 2048 matrix (1024 partials) and 344 for
// a 4096 x 11008 one.
constexpr int kFinThreads = 256;
__global__ void __launch_bounds__(kFinThreads) norm_finalize_kernel(const MatDesc* mats, const float* partials) {
    __shared__ double red[kFinThreads];
    const MatDesc& md = mats[blockIdx.x];
    const int k = threadIdx.x;
    const int64_t nt = static_cast<int64_t>(md.mom_tiles_r) * md.mom_tiles_c;
    const float* part = partials + md.mom_tile_begin;
    double s = 0.0;
#pragma unroll 4
    for (int64_t i = k; i < nt; i += kFinThreads) s += static_cast<double>(part[i]);
    red[k] = s;
    __syncthreads();
    for (int w = kFinThreads / 2; w > 0; w >>= 1) {
        if (k < w) red[k] += red[k + w];
        __syncthreads();
    }
    if (k == 0) {
        const double t = red[0];
        float inv_s = 0.f, inv_s2 = 0.f;
        if (t > 0.0) {
            inv_s = static_cast<float>(1.0 / sqrt(t));
            inv_s2 = static_cast<float>(1.0 / t);
        }
        md.scales[0] = inv_s;
        md.scales[1] = inv_s2;
        md.scales[2] = 1.f;     // spectral folding factors: identity under Frobenius scaling
        md.scales[3] = 1.f;
        md.scales[4] = 1.f;
    }
}

cudaError_t launch_norm_finalize(const MatDesc* mats, int nmats, const float* partials, cudaStream_t s) {
    if (nmats == 0) return cudaSuccess;
    norm_finalize_kernel<<<nmats, kFinThreads, 0, s>>>(mats, partials);
    return cudaGetLastError();
}

// ------------------------------------------------------------------- ns_k0
// Zero Newton-Schulz steps: O = X / ||X||_F, elementwise in the user layout.
struct K0Args {
    MomLaunch p;
    float alpha, decay;
    int apply_update;
};
__global__ void __launch_bounds__(256) ns_k0_kernel(K0Args a) {
    const MomLaunch& p = a.p;
    const int col4 = threadIdx.x & 15, rsub = threadIdx.x >> 4;
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const MatDesc& md = p.mats[find_matrix(p.mats, p.nmats, t)];
        const int64_t local = t - md.mom_tile_begin;
        const int r0 = static_cast<int>(local / md.mom_tiles_c) * kMomTile;
        const int c0 = static_cast<int>(local % md.mom_tiles_c) * kMomTile;
        const int c = c0 + 4 * col4;
        const int nvalid = max(0, min(4, md.cols - c));
        const float inv_s = md.scales[0];
        for (int q = 0; q < 4; ++q) {
            const int r = r0 + rsub + 16 * q;
            if (r >= md.rows || nvalid <= 0) continue;
            const int64_t off = static_cast<int64_t>(r) * md.ld + c;
            float x[4];
            load4(md.src, md.src_dtype, off, nvalid, x);
            for (int k = 0; k < 4; ++k) x[k] *= inv_s;
            if (a.apply_update) {
                float w[4];
                load4(md.W, md.w_dtype, off, nvalid, w);
                for (int k = 0; k < 4; ++k) w[k] = fmaf(-a.alpha, x[k], w[k] - a.decay * w[k]);
                store4(md.W, md.w_dtype, off, nvalid, w);
            } else {
                store4(md.out, md.out_dtype, off, nvalid, x);
            }
        }
    }
}

cudaError_t launch_ns_k0(const MomLaunch& p, float alpha, float decay, int apply_update, int grid,
                         cudaStream_t s) {
    if (p.ntiles == 0) return cudaSuccess;
    K0Args a{p, alpha, decay, apply_update};
    ns_k0_kernel<<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

// --------------------------------------------------------------- sign_pack
// One warp packs 16 consecutive words per iteration: lane l reads element
// 32w + l of each word w and __ballot_sync assembles the word (bit l = lane l).
constexpr int kPackWords = 16;

template <typename T>
__device__ __forceinline__ float to_float(T x);
template <> __device__ __forceinline__ float to_float<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_float<bf16>(bf16 x) { return __bfloat162float(x); }

template <typename T>
__global__ void __launch_bounds__(256) sign_pack_kernel(const T* __restrict__ U, int64_t rows, int64_t cols,
                                                        int64_t ld, uint32_t* __restrict__ words,
                                                        int64_t nwords) {
    const int lane = threadIdx.x & 31;
    const int64_t numel = rows * cols;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t w0 = warp * kPackWords; w0 < nwords; w0 += nwarps * kPackWords) {
        int64_t e = w0 * 32 + lane;
        int64_t r = e / cols, c = e - r * cols;
        float v[kPackWords];
#pragma unroll
        for (int q = 0; q < kPackWords; ++q) {
            v[q] = 0.f;
            if (e + 32 * q < numel) v[q] = to_float<T>(U[r * ld + c]);
            c += 32;
            while (c >= cols) { c -= cols; ++r; }
        }
        uint32_t mine = 0;
#pragma unroll
        for (int q = 0; q < kPackWords; ++q) {
            const bool valid = (e + 32 * q) < numel;
            const uint32_t word = __ballot_sync(0xffffffffu, valid && !(v[q] < 0.f));
            if (lane == q) mine = word;
        }
        if (lane < kPackWords && w0 + lane < nwords) words[w0 + lane] = mine;
    }
}

// Fast path when every run of 8 elements lies in one row and starts 16-byte
// aligned (cols % 8 == 0, ld % 8 == 0, U 16-byte aligned): lane l loads 8
// consecutive elements with 16-byte loads, forms their 8 sign bits, and 4
// neighbouring lanes OR their bytes into one word.  A warp packs 32 words
// (1024 elements) per iteration.
__device__ __forceinline__ uint32_t sign_byte(const float (&x)[8]) {
    uint32_t b = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) b |= (x[k] < 0.f ? 0u : 1u) << k;
    return b;
}
__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void load8(const bf16* p, float (&x)[8]) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        x[2 * q] = __low2float(h[q]);
        x[2 * q + 1] = __high2float(h[q]);
    }
}

__device__ __forceinline__ void unpack_bf16x8_pack(const uint4& u, float (&x)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        x[2 * q] = __low2float(h[q]);
        x[2 * q + 1] = __high2float(h[q]);
    }
}

constexpr int kMaxPackBatch = 128;
struct PackPtrs {
    const void* U[kMaxPackBatch];
    uint32_t* words[kMaxPackBatch];
};

// blockIdx.y selects the matrix of a batch (all of one shape).
template <typename T>
__global__ void __launch_bounds__(256) sign_pack_vec_kernel(const __grid_constant__ PackPtrs pp, int64_t rows,
                                                            int64_t cols, int64_t ld, int64_t nwords) {
    constexpr int kSub = 4;                       // 4 x 256 elements per warp iteration
    const T* __restrict__ U = static_cast<const T*>(pp.U[blockIdx.y]);
    uint32_t* __restrict__ words = pp.words[blockIdx.y];
    const int lane = threadIdx.x & 31;
    const int64_t noct = rows * cols / 8;         // runs of 8 elements
    const int64_t opr = cols / 8;                 // runs per row
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t o0 = warp * 32 * kSub; o0 < noct; o0 += nwarps * 32 * kSub) {
        int64_t o = o0 + lane;
        int64_t r = o / opr, c8 = o - r * opr;
        float x[kSub][8];
#pragma unroll
        for (int u = 0; u < kSub; ++u) {
            if (o + 32 * u < noct) {
                load8(U + r * ld + c8 * 8, x[u]);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) x[u][k] = -1.f;     // beyond the matrix: bit 0
            }
            c8 += 32;
            while (c8 >= opr) { c8 -= opr; ++r; }
        }
#pragma unroll
        for (int u = 0; u < kSub; ++u) {
            uint32_t v = sign_byte(x[u]) << (8 * (lane & 3));
            v |= __shfl_xor_sync(0xffffffffu, v, 1);
            v |= __shfl_xor_sync(0xffffffffu, v, 2);
            const int64_t w = (o0 + 32 * u) / 4 + (lane >> 2);
            if ((lane & 3) == 0 && w < nwords) words[w] = v;
        }
    }
}

// Bounded wait on an mbarrier phase (about 2 s of SM clock); false on timeout.
__device__ __forceinline__ bool wait_phase_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

// Bulk path for contiguous bf16 matrices whose element count is a multiple of
// kPackChunk: each block streams chunks of kPackChunk elements (of any
// matrix of the batch) through a kPackStages-deep ring in shared memory, one
// bulk copy per chunk; warps then read consecutive 16-byte pieces (8
// elements -> one sign byte), and four lanes combine their bytes into a word.
// Two 32 KB stages (three blocks per SM) measured faster than three 16 KB
// ones (four per SM) at 2048^2 and at 8192^2 elements per matrix.
constexpr int kPackChunk = 16384;
constexpr int kPackStages = 2;

__global__ void __launch_bounds__(256) sign_pack_bulk_kernel(const __grid_constant__ PackPtrs pp,
                                                             int64_t chunks_per_matrix, int64_t nchunks) {
    extern __shared__ __align__(128) uint8_t psm[];
    __shared__ __align__(8) uint64_t full[kPackStages];
    constexpr uint32_t kBytes = kPackChunk * 2;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    if (t == 0) {
        for (int s2 = 0; s2 < kPackStages; ++s2) mbar_init(smem_u32(&full[s2]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int64_t q, int st) {                 // thread 0
        const int64_t m = q / chunks_per_matrix, c = q - m * chunks_per_matrix;
        const uint32_t bar = smem_u32(&full[st]);
        mbar_arrive_expect_tx(bar, kBytes);
        bulk_load(smem_u32(psm + st * kBytes), static_cast<const bf16*>(pp.U[m]) + c * kPackChunk, kBytes, bar);
    };
    if (t == 0)
        for (int s2 = 0; s2 < kPackStages; ++s2)
            if (blockIdx.x + s2 * static_cast<int64_t>(gridDim.x) < nchunks) issue(blockIdx.x + s2 * gridDim.x, s2);
    int k = 0;
    bool ok = true;
    for (int64_t q = blockIdx.x; q < nchunks; q += gridDim.x, ++k) {
        const int st = k % kPackStages;
        ok = wait_phase_bounded(smem_u32(&full[st]), (k / kPackStages) & 1);
        if (!__syncthreads_and(ok)) break;                 // never expected: a bounded give-up
        const int64_t m = q / chunks_per_matrix, c = q - m * chunks_per_matrix;
        const uint4* src = reinterpret_cast<const uint4*>(psm + st * kBytes);
        uint32_t* dst = pp.words[m] + c * (kPackChunk / 32);
#pragma unroll
        for (int it = 0; it < kPackChunk / 8 / 256; ++it) {
            const int piece = it * 256 + warp * 32 + lane;           // 8 elements each
            float x[8];
            unpack_bf16x8_pack(src[piece], x);
            uint32_t v = sign_byte(x) << (8 * (lane & 3));
            v |= __shfl_xor_sync(0xffffffffu, v, 1);
            v |= __shfl_xor_sync(0xffffffffu, v, 2);
            if ((lane & 3) == 0) dst[piece >> 2] = v;
        }
        __syncthreads();                                   // the stage is read
        if (t == 0) {
            const int64_t qn = q + kPackStages * static_cast<int64_t>(gridDim.x);
            if (qn < nchunks) issue(qn, st);
        }
    }
    if (t == 0 && !ok) {
        // let copies still landing in this block's shared memory finish
        for (int s2 = 0; s2 < kPackStages; ++s2) (void)wait_phase_bounded(smem_u32(&full[s2]), (k / kPackStages) & 1);
    }
}

cudaError_t launch_sign_pack_batched(const void* const* U, uint32_t* const* words, int M, int dtype, int64_t rows,
                                     int64_t cols, int64_t ld, cudaStream_t s) {
    const int64_t nwords = (rows * cols + 31) / 32;
    if (nwords == 0 || M <= 0) return cudaSuccess;
    bool vec = cols % 8 == 0 && ld % 8 == 0;
    for (int m = 0; m < M; ++m) vec = vec && (reinterpret_cast<uintptr_t>(U[m]) & 15u) == 0;
    const bool bulk = vec && dtype == MO_BF16 && ld == cols && (rows * cols) % kPackChunk == 0;
    if (bulk) {
        PackPtrs pp{};
        for (int m = 0; m < M; ++m) {
            pp.U[m] = U[m];
            pp.words[m] = words[m];
        }
        const int smem = kPackStages * kPackChunk * 2;
        static std::atomic<uint64_t> attr_set{0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const uint64_t bit = uint64_t(1) << (dev & 63);
        if (!(attr_set.load() & bit)) {
            e = cudaFuncSetAttribute(sign_pack_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            attr_set.fetch_or(bit);
        }
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sign_pack_bulk_kernel, 256, smem);
        if (e != cudaSuccess || per_sm < 1) per_sm = 1;
        const int64_t cpm = rows * cols / kPackChunk, nchunks = cpm * M;
        const int64_t g = std::min<int64_t>(nchunks, static_cast<int64_t>(device_sm_count()) * per_sm);
        sign_pack_bulk_kernel<<<static_cast<int>(g), 256, smem, s>>>(pp, cpm, nchunks);
        return cudaGetLastError();
    }
    if (vec) {
        PackPtrs pp{};
        for (int m = 0; m < M; ++m) {
            pp.U[m] = U[m];
            pp.words[m] = words[m];
        }
        const int64_t warps_needed = (rows * cols / 8 + 127) / 128;
        const int64_t blocks = (warps_needed + 7) / 8;
        const int per_sm = dtype == MO_F32 ? resident_blocks_per_sm(sign_pack_vec_kernel<float>, 256)
                                           : resident_blocks_per_sm(sign_pack_vec_kernel<bf16>, 256);
        int64_t cap = static_cast<int64_t>(device_sm_count()) * per_sm / M;     // one resident wave
        if (cap < 1) cap = 1;
        const dim3 grid(static_cast<unsigned>(blocks < cap ? blocks : cap), static_cast<unsigned>(M));
        if (dtype == MO_F32)
            sign_pack_vec_kernel<float><<<grid, 256, 0, s>>>(pp, rows, cols, ld, nwords);
        else
            sign_pack_vec_kernel<bf16><<<grid, 256, 0, s>>>(pp, rows, cols, ld, nwords);
        return cudaGetLastError();
    }
    for (int m = 0; m < M; ++m) {
        cudaError_t e = launch_sign_pack(U[m], dtype, rows, cols, ld, words[m], s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_sign_pack(const void* U, int dtype, int64_t rows, int64_t cols, int64_t ld,
                             uint32_t* words, cudaStream_t s) {
    const int64_t nwords = (rows * cols + 31) / 32;
    if (nwords == 0) return cudaSuccess;
    const bool vec = cols % 8 == 0 && ld % 8 == 0 && (reinterpret_cast<uintptr_t>(U) & 15u) == 0;
    if (vec) return launch_sign_pack_batched(&U, &words, 1, dtype, rows, cols, ld, s);
    const int64_t warps_needed = (nwords + kPackWords - 1) / kPackWords;
    const int64_t blocks = (warps_needed + 7) / 8;
    const int grid = static_cast<int>(blocks < device_sm_count() * 16LL ? blocks : device_sm_count() * 16LL);
    if (dtype == MO_F32)
        sign_pack_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(U), rows, cols, ld, words, nwords);
    else
        sign_pack_kernel<bf16><<<grid, 256, 0, s>>>(static_cast<const bf16*>(U), rows, cols, ld, words, nwords);
    return cudaGetLastError();
}

// ------------------------------------------------------------- vote_update
// A warp takes 32 consecutive words: lane l reads word (base + l) of all M
// buffers (coalesced), counts +1 votes per bit position with a bit-sliced
// ripple counter, compares the count with ceil(M/2) bit-sliced, then the warp
// updates the 1024 covered elements, 32 at a time (coalesced along W).
constexpr int kMaxVoters = 128;
struct VotePtrs {
    const uint32_t* w[kMaxVoters];
};

template <typename T>
__global__ void __launch_bounds__(256) vote_update_kernel(const __grid_constant__ VotePtrs ptrs, int M, int nbits, uint32_t thr,
                                                          int64_t rows, int64_t cols, int64_t ld,
                                                          T* __restrict__ W, float lr, int64_t nwords) {
    const int lane = threadIdx.x & 31;
    const int64_t numel = rows * cols;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t base = warp * 32; base < nwords; base += nwarps * 32) {
        const int64_t w = base + lane;
        uint32_t cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (w < nwords) {
            for (int m = 0; m < M; ++m) {
                uint32_t x = __ldg(ptrs.w[m] + w);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j < nbits) {
                        const uint32_t carry = cnt[j] & x;
                        cnt[j] ^= x;
                        x = carry;
                    }
                }
            }
        }
        uint32_t gt = 0u, eq = 0xffffffffu;
#pragma unroll
        for (int j = 7; j >= 0; --j) {
            if (j < nbits) {
                if ((thr >> j) & 1u) {
                    eq &= cnt[j];
                } else {
                    gt |= eq & cnt[j];
                    eq &= ~cnt[j];
                }
            }
        }
        const uint32_t plus = gt | eq;   // bit set: count >= ceil(M/2), i.e. vote +1
        int64_t e = base * 32 + lane;
        int64_t r = e / cols, c = e - r * cols;
        for (int q = 0; q < 32; ++q) {
            const uint32_t vw = __shfl_sync(0xffffffffu, plus, q);
            if (e < numel) {
                const int64_t idx = r * ld + c;
                const float wv = to_float<T>(W[idx]);
                const float nv = ((vw >> lane) & 1u) ? (wv - lr) : (wv + lr);
                if constexpr (sizeof(T) == 4)
                    W[idx] = nv;
                else
                    W[idx] = __float2bfloat16_rn(nv);
            }
            e += 32;
            c += 32;
            while (c >= cols) { c -= cols; ++r; }
        }
    }
}

// Bit-sliced count of +1 votes of 32 elements over the M buffers, compared
// with ceil(M/2): bit k of the result is 1 when element k votes +1.
__device__ __forceinline__ uint32_t vote_word(const VotePtrs& ptrs, int M, int nbits, uint32_t thr, int64_t w) {
    uint32_t cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll 8
    for (int m = 0; m < M; ++m) {
        uint32_t x = __ldcs(ptrs.w[m] + w);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < nbits) {
                const uint32_t carry = cnt[j] & x;
                cnt[j] ^= x;
                x = carry;
            }
        }
    }
    uint32_t gt = 0u, eq = 0xffffffffu;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
        if (j < nbits) {
            if ((thr >> j) & 1u) {
                eq &= cnt[j];
            } else {
                gt |= eq & cnt[j];
                eq &= ~cnt[j];
            }
        }
    }
    return gt | eq;
}

template <typename T> struct Vec4;
template <> struct Vec4<float> {
    using type = float4;
    static __device__ __forceinline__ void unpack(const float4& v, float (&x)[4]) { x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w; }
    static __device__ __forceinline__ float4 pack(const float (&x)[4]) { return make_float4(x[0], x[1], x[2], x[3]); }
};
template <> struct Vec4<bf16> {
    using type = uint2;
    static __device__ __forceinline__ void unpack(const uint2& v, float (&x)[4]) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
        x[0] = __low2float(h[0]); x[1] = __high2float(h[0]); x[2] = __low2float(h[1]); x[3] = __high2float(h[1]);
    }
    static __device__ __forceinline__ uint2 pack(const float (&x)[4]) {
        __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
        uint2 v;
        v.x = *reinterpret_cast<uint32_t*>(&a);
        v.y = *reinterpret_cast<uint32_t*>(&b);
        return v;
    }
};

// Fast path when runs of 4 elements lie in one row and are vector-aligned
// (cols % 4 == 0, ld % 4 == 0, W aligned to 4 elements): a warp takes 32
// words; lane l updates elements 128q + 4l .. +3 (q = 0..7) with 4-element
// vector accesses, all loads issued before the stores.
template <typename T>
__global__ void __launch_bounds__(256) vote_update_vec_kernel(const __grid_constant__ VotePtrs ptrs, int M, int nbits,
                                                              uint32_t thr, int64_t rows, int64_t cols, int64_t ld,
                                                              T* __restrict__ W, float lr, int64_t nwords) {
    using V = typename Vec4<T>::type;
    const int lane = threadIdx.x & 31;
    const int64_t numel = rows * cols;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t base = warp * 32; base < nwords; base += nwarps * 32) {
        // W loads first, so they are in flight with the word loads below; the
        // store pass walks the same positions again rather than keeping them
        const int64_t e = base * 32 + 4 * lane;
        const int64_t r0 = e / cols, c0 = e - r0 * cols;
        V val[8];
        {
            int64_t r = r0, c = c0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (e + 128 * q < numel) val[q] = *reinterpret_cast<const V*>(W + r * ld + c);
                c += 128;
                while (c >= cols) { c -= cols; ++r; }
            }
        }
        const uint32_t plus = base + lane < nwords ? vote_word(ptrs, M, nbits, thr, base + lane) : 0u;
        int64_t r = r0, c = c0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t vw = __shfl_sync(0xffffffffu, plus, 4 * q + (lane >> 3));
            const uint32_t bits = vw >> (4 * (lane & 7));
            if (e + 128 * q < numel) {
                float x[4];
                Vec4<T>::unpack(val[q], x);
#pragma unroll
                for (int k = 0; k < 4; ++k) x[k] = ((bits >> k) & 1u) ? (x[k] - lr) : (x[k] + lr);
                *reinterpret_cast<V*>(W + r * ld + c) = Vec4<T>::pack(x);
            }
            c += 128;
            while (c >= cols) { c -= cols; ++r; }
        }
    }
}

// ------------------------------------------------- vote + update, bulk path
// For a contiguous W (ld == cols) whose element count is a multiple of
// kVoteChunk, with up to kBulkVoters workers: each block streams chunks of
// kVoteChunk elements through shared memory, two chunks in flight.  A chunk's
// W and its kVoteChunk/32 words of every worker arrive by bulk copies on one
// mbarrier; the first kVoteChunkWords threads count one word each, then all
// 256 update the chunk in registers and store it back with consecutive
// threads on consecutive elements.  Same arithmetic as vote_update_vec_kernel.
// 4096-element chunks keep the per-SM share even on small matrices: a 2048^2 W
// is 1024 chunks over one resident wave of 5 blocks per SM (6 or 7 chunks per
// SM), where 8192-element chunks left 3 or 4 per SM.
constexpr int kVoteChunk = 4096;
constexpr int kVoteChunkWords = kVoteChunk / 32;
constexpr int kBulkVoters = 16;

template <typename T>
__global__ void __launch_bounds__(256) vote_update_bulk_kernel(const __grid_constant__ VotePtrs ptrs, int M,
                                                               int nbits, uint32_t thr, T* __restrict__ W, float lr,
                                                               int64_t nchunks) {
    extern __shared__ __align__(128) uint8_t vsm[];
    __shared__ __align__(8) uint64_t full[2];
    __shared__ uint32_t vote[kVoteChunkWords];
    constexpr uint32_t kWBytes = kVoteChunk * sizeof(T);
    const uint32_t stage_bytes = kWBytes + static_cast<uint32_t>(M) * kVoteChunkWords * 4;
    const int t = threadIdx.x;
    if (t == 0) {
        mbar_init(smem_u32(&full[0]), 1);
        mbar_init(smem_u32(&full[1]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int64_t c, int st) {                 // thread 0
        uint8_t* base = vsm + st * stage_bytes;
        const uint32_t bar = smem_u32(&full[st]);
        mbar_arrive_expect_tx(bar, stage_bytes);
        bulk_load(smem_u32(base), W + c * kVoteChunk, kWBytes, bar);
        for (int m = 0; m < M; ++m)
            bulk_load(smem_u32(base + kWBytes + m * kVoteChunkWords * 4), ptrs.w[m] + c * kVoteChunkWords,
                      kVoteChunkWords * 4, bar);
    };
    const int64_t c0 = blockIdx.x;
    if (t == 0) {
        if (c0 < nchunks) issue(c0, 0);
        if (c0 + gridDim.x < nchunks) issue(c0 + gridDim.x, 1);
    }
    int k = 0;
    bool ok = true;
    for (int64_t c = c0; c < nchunks; c += gridDim.x, ++k) {
        const int st = k & 1;
        ok = wait_phase_bounded(smem_u32(&full[st]), (k >> 1) & 1);
        if (!__syncthreads_and(ok)) break;                 // never expected: a bounded give-up
        uint8_t* base = vsm + st * stage_bytes;
        const uint32_t* wd = reinterpret_cast<const uint32_t*>(base + kWBytes);
        // bit-sliced count of +1 votes of word t over the M workers
        if (t < kVoteChunkWords) {
            uint32_t cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int m = 0; m < M; ++m) {
                uint32_t x = wd[m * kVoteChunkWords + t];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j < nbits) {
                        const uint32_t carry = cnt[j] & x;
                        cnt[j] ^= x;
                        x = carry;
                    }
                }
            }
            uint32_t gt = 0u, eq = 0xffffffffu;
#pragma unroll
            for (int j = 7; j >= 0; --j) {
                if (j < nbits) {
                    if ((thr >> j) & 1u) {
                        eq &= cnt[j];
                    } else {
                        gt |= eq & cnt[j];
                        eq &= ~cnt[j];
                    }
                }
            }
            vote[t] = gt | eq;
        }
        __syncthreads();
        const T* w = reinterpret_cast<const T*>(base);
        T* wg = W + c * kVoteChunk;
#pragma unroll 8
        for (int j = 0; j < kVoteChunk / 256; ++j) {
            const int e = t + 256 * j;                     // a warp stores 32 consecutive elements
            const float x = static_cast<float>(w[e]);
            wg[e] = static_cast<T>(((vote[e >> 5] >> (e & 31)) & 1u) ? (x - lr) : (x + lr));
        }
        __syncthreads();                                   // the stage is read
        if (t == 0) {
            const int64_t cn = c + 2 * static_cast<int64_t>(gridDim.x);
            if (cn < nchunks) issue(cn, st);
        }
    }
    if (t == 0) {
        if (!ok) {
            // let copies still landing in this block's shared memory finish
            for (int s2 = 0; s2 < 2; ++s2) (void)wait_phase_bounded(smem_u32(&full[s2]), (k >> 1) & 1);
        }
    }
}

cudaError_t launch_sign_vote_update(const uint32_t* const* words, int M, int64_t rows, int64_t cols,
                                    void* W, int w_dtype, int64_t ld, float lr, cudaStream_t s) {
    const int64_t nwords = (rows * cols + 31) / 32;
    if (nwords == 0) return cudaSuccess;
    VotePtrs ptrs{};
    for (int m = 0; m < M; ++m) ptrs.w[m] = words[m];
    int nbits = 0;
    while ((1 << nbits) <= M) ++nbits;
    const uint32_t thr = static_cast<uint32_t>((M + 1) / 2);
    const int64_t warps_needed = (nwords + 31) / 32;
    const int64_t blocks = (warps_needed + 7) / 8;
    int grid = static_cast<int>(blocks < device_sm_count() * 16LL ? blocks : device_sm_count() * 16LL);
    const size_t vbytes = w_dtype == MO_F32 ? 16 : 8;
    const bool vec = cols % 4 == 0 && ld % 4 == 0 && (reinterpret_cast<uintptr_t>(W) % vbytes) == 0;
    const int64_t numel = rows * cols;
    bool bulk = ld == cols && numel % kVoteChunk == 0 && M <= kBulkVoters && (reinterpret_cast<uintptr_t>(W) & 15u) == 0;
    for (int m = 0; m < M && bulk; ++m) bulk = (reinterpret_cast<uintptr_t>(words[m]) & 15u) == 0;
    if (bulk) {
        const int esz = w_dtype == MO_F32 ? 4 : 2;
        const int smem = 2 * (kVoteChunk * esz + M * kVoteChunkWords * 4);
        static std::atomic<uint64_t> attr_set{0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const uint64_t bit = uint64_t(1) << (dev & 63);
        if (!(attr_set.load() & bit)) {
            const int max_smem = 2 * (kVoteChunk * 4 + kBulkVoters * kVoteChunkWords * 4);
            e = cudaFuncSetAttribute(vote_update_bulk_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     max_smem);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(vote_update_bulk_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     max_smem);
            if (e != cudaSuccess) return e;
            attr_set.fetch_or(bit);
        }
        const int64_t nchunks = numel / kVoteChunk;
        int per_sm = 0;
        if (w_dtype == MO_F32)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vote_update_bulk_kernel<float>, 256, smem);
        else
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vote_update_bulk_kernel<bf16>, 256, smem);
        if (e != cudaSuccess || per_sm < 1) per_sm = 1;
        const int64_t g = std::min<int64_t>(nchunks, static_cast<int64_t>(device_sm_count()) * per_sm);
        if (w_dtype == MO_F32)
            vote_update_bulk_kernel<float><<<static_cast<int>(g), 256, smem, s>>>(ptrs, M, nbits, thr,
                                                                               static_cast<float*>(W), lr, nchunks);
        else
            vote_update_bulk_kernel<bf16><<<static_cast<int>(g), 256, smem, s>>>(ptrs, M, nbits, thr,
                                                                              static_cast<bf16*>(W), lr, nchunks);
        return cudaGetLastError();
    }
    if (vec) {
        const int per_sm = w_dtype == MO_F32 ? resident_blocks_per_sm(vote_update_vec_kernel<float>, 256)
                                             : resident_blocks_per_sm(vote_update_vec_kernel<bf16>, 256);
        const int64_t wave = static_cast<int64_t>(device_sm_count()) * per_sm;   // one resident wave
        if (grid > wave) grid = static_cast<int>(wave);
        if (w_dtype == MO_F32)
            vote_update_vec_kernel<float><<<grid, 256, 0, s>>>(ptrs, M, nbits, thr, rows, cols, ld,
                                                               static_cast<float*>(W), lr, nwords);
        else
            vote_update_vec_kernel<bf16><<<grid, 256, 0, s>>>(ptrs, M, nbits, thr, rows, cols, ld,
                                                              static_cast<bf16*>(W), lr, nwords);
        return cudaGetLastError();
    }
    if (w_dtype == MO_F32)
        vote_update_kernel<float><<<grid, 256, 0, s>>>(ptrs, M, nbits, thr, rows, cols, ld,
                                                       static_cast<float*>(W), lr, nwords);
    else
        vote_update_kernel<bf16><<<grid, 256, 0, s>>>(ptrs, M, nbits, thr, rows, cols, ld,
                                                      static_cast<bf16*>(W), lr, nwords);
    return cudaGetLastError();
}

// ------------------------------------------------------------ vote_matrix
// The voted sign matrix itself, S_bar = +1 / -1 as bf16, written in a
// rows x cols layout with leading dimension ld (input of the optional local
// polar step).  Element-wise over words, coalesced along the flattening.
__global__ void __launch_bounds__(256) vote_matrix_kernel(const __grid_constant__ VotePtrs ptrs, int M, int nbits,
                                                          uint32_t thr, int64_t rows, int64_t cols, int64_t ld,
                                                          bf16* __restrict__ S, int64_t nwords) {
    const int lane = threadIdx.x & 31;
    const int64_t numel = rows * cols;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const bf16 plus1 = __float2bfloat16_rn(1.f), minus1 = __float2bfloat16_rn(-1.f);
    for (int64_t base = warp * 32; base < nwords; base += nwarps * 32) {
        const uint32_t plus = base + lane < nwords ? vote_word(ptrs, M, nbits, thr, base + lane) : 0u;
        int64_t e = base * 32 + lane;
        int64_t r = e / cols, c = e - r * cols;
        for (int q = 0; q < 32; ++q) {
            const uint32_t vw = __shfl_sync(0xffffffffu, plus, q);
            if (e < numel) S[r * ld + c] = ((vw >> lane) & 1u) ? plus1 : minus1;
            e += 32;
            c += 32;
            while (c >= cols) { c -= cols; ++r; }
        }
    }
}

cudaError_t launch_vote_matrix(const uint32_t* const* words, int M, int64_t rows, int64_t cols, void* S, int64_t ld,
                               cudaStream_t s) {
    const int64_t nwords = (rows * cols + 31) / 32;
    if (nwords == 0) return cudaSuccess;
    VotePtrs ptrs{};
    for (int m = 0; m < M; ++m) ptrs.w[m] = words[m];
    int nbits = 0;
    while ((1 << nbits) <= M) ++nbits;
    const uint32_t thr = static_cast<uint32_t>((M + 1) / 2);
    const int64_t blocks = ((nwords + 31) / 32 + 7) / 8;
    const int grid = static_cast<int>(blocks < device_sm_count() * 16LL ? blocks : device_sm_count() * 16LL);
    vote_matrix_kernel<<<grid, 256, 0, s>>>(ptrs, M, nbits, thr, rows, cols, ld, static_cast<bf16*>(S), nwords);
    return cudaGetLastError();
}

// ------------------------------------------------ int8 all-reduce variant
// sign_int8: out[j] = -1 if U_j < 0 else +1 over the row-major flattening
// (dense, no padding).  vote_int8: per element, the integer sum of the M
// workers' int8 signs, vote = +1 iff sum >= 0, W -= lr * vote (one fp32
// rounding).  Vector paths take 8 (sign) or 16 (vote) elements per thread
// when such runs lie in one row and are aligned; others go element-wise.
template <typename T>
__global__ void __launch_bounds__(256) sign_int8_kernel(const T* __restrict__ U, int64_t rows, int64_t cols,
                                                        int64_t ld, int8_t* __restrict__ out, int vec) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (vec) {
        const int64_t noct = rows * cols / 8, opr = cols / 8;
        for (int64_t o = first; o < noct; o += stride) {
            const int64_t r = o / opr, c = (o - r * opr) * 8;
            float x[8];
            load8(U + r * ld + c, x);
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                lo |= (x[k] < 0.f ? 0xFFu : 0x01u) << (8 * k);
                hi |= (x[k + 4] < 0.f ? 0xFFu : 0x01u) << (8 * k);
            }
            reinterpret_cast<uint2*>(out)[o] = make_uint2(lo, hi);
        }
    } else {
        const int64_t numel = rows * cols;
        for (int64_t e = first; e < numel; e += stride) {
            const int64_t r = e / cols, c = e - r * cols;
            out[e] = to_float<T>(U[r * ld + c]) < 0.f ? int8_t(-1) : int8_t(1);
        }
    }
}

struct Int8Ptrs {
    const int8_t* s[kMaxVoters];
};

template <typename T>
__global__ void __launch_bounds__(256) vote_int8_kernel(const __grid_constant__ Int8Ptrs p, int M, int64_t rows,
                                                        int64_t cols, int64_t ld, T* __restrict__ W, float lr,
                                                        int vec) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (vec) {
        using V = typename Vec4<T>::type;
        const int64_t ngrp = rows * cols / 16, gpr = cols / 16;
        for (int64_t g = first; g < ngrp; g += stride) {
            uint32_t acc[4] = {0, 0, 0, 0};        // 16 signed byte sums (|sum| <= M <= 127)
            for (int m = 0; m < M; ++m) {
                const uint4 v = __ldcs(reinterpret_cast<const uint4*>(p.s[m]) + g);
                acc[0] = __vadd4(acc[0], v.x);
                acc[1] = __vadd4(acc[1], v.y);
                acc[2] = __vadd4(acc[2], v.z);
                acc[3] = __vadd4(acc[3], v.w);
            }
            const int64_t r = g / gpr, c = (g - r * gpr) * 16;
            T* row = W + r * ld + c;
            V val[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) val[q] = reinterpret_cast<const V*>(row)[q];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float x[4];
                Vec4<T>::unpack(val[q], x);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const bool neg = (acc[q] >> (8 * k + 7)) & 1u;     // byte sum < 0
                    x[k] = neg ? (x[k] + lr) : (x[k] - lr);
                }
                reinterpret_cast<V*>(row)[q] = Vec4<T>::pack(x);
            }
        }
    } else {
        const int64_t numel = rows * cols;
        for (int64_t e = first; e < numel; e += stride) {
            int sum = 0;
            for (int m = 0; m < M; ++m) sum += p.s[m][e];
            const int64_t r = e / cols, c = e - r * cols;
            const float w = to_float<T>(W[r * ld + c]);
            const float nv = sum >= 0 ? (w - lr) : (w + lr);
            if constexpr (sizeof(T) == 4)
                W[r * ld + c] = nv;
            else
                W[r * ld + c] = __float2bfloat16_rn(nv);
        }
    }
}

cudaError_t launch_sign_int8(const void* U, int dtype, int64_t rows, int64_t cols, int64_t ld, int8_t* out,
                             cudaStream_t s) {
    const int64_t numel = rows * cols;
    if (numel == 0) return cudaSuccess;
    const int vec = cols % 8 == 0 && ld % 8 == 0 && (reinterpret_cast<uintptr_t>(U) & 15u) == 0 &&
                    (reinterpret_cast<uintptr_t>(out) & 7u) == 0;
    const int64_t items = vec ? numel / 8 : numel;
    int64_t blocks = (items + 255) / 256;
    const int64_t cap = device_sm_count() * 8LL;
    if (blocks > cap) blocks = cap;
    if (dtype == MO_F32)
        sign_int8_kernel<float><<<static_cast<int>(blocks), 256, 0, s>>>(static_cast<const float*>(U), rows, cols,
                                                                         ld, out, vec);
    else
        sign_int8_kernel<bf16><<<static_cast<int>(blocks), 256, 0, s>>>(static_cast<const bf16*>(U), rows, cols, ld,
                                                                        out, vec);
    return cudaGetLastError();
}

cudaError_t launch_vote_int8(const int8_t* const* signs, int M, int64_t rows, int64_t cols, void* W, int w_dtype,
                             int64_t ld, float lr, cudaStream_t s) {
    const int64_t numel = rows * cols;
    if (numel == 0) return cudaSuccess;
    Int8Ptrs p{};
    bool aligned = true;
    for (int m = 0; m < M; ++m) {
        p.s[m] = signs[m];
        aligned = aligned && (reinterpret_cast<uintptr_t>(signs[m]) & 15u) == 0;
    }
    const size_t vbytes = w_dtype == MO_F32 ? 16 : 8;
    const int vec = aligned && cols % 16 == 0 && ld % 4 == 0 && (reinterpret_cast<uintptr_t>(W) % vbytes) == 0;
    const int64_t items = vec ? numel / 16 : numel;
    int64_t blocks = (items + 255) / 256;
    const int64_t cap = device_sm_count() * 8LL;
    if (blocks > cap) blocks = cap;
    if (w_dtype == MO_F32)
        vote_int8_kernel<float><<<static_cast<int>(blocks), 256, 0, s>>>(p, M, rows, cols, ld, static_cast<float*>(W),
                                                                         lr, vec);
    else
        vote_int8_kernel<bf16><<<static_cast<int>(blocks), 256, 0, s>>>(p, M, rows, cols, ld, static_cast<bf16*>(W),
                                                                        lr, vec);
    return cudaGetLastError();
}

// ------------------------------------------------------------------- adamw
struct AdamArgs {
    float* W; const float* g; float* m; float* v;
    int64_t numel;
    float beta1, beta2, eps, step_size, inv_bc2, decay;
};

__device__ __forceinline__ void adam_one(const AdamArgs& a, float& w, float g, float& m, float& v) {
    m = fmaf(a.beta1, m, (1.f - a.beta1) * g);
    v = fmaf(a.beta2, v, (1.f - a.beta2) * g * g);
    const float denom = sqrtf(v * a.inv_bc2) + a.eps;
    w = w - a.decay * w - a.step_size * (m / denom);
}

__global__ void __launch_bounds__(256) adamw_kernel(AdamArgs a) {
    const int64_t n4 = a.numel >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 w = reinterpret_cast<float4*>(a.W)[i];
        const float4 g = __ldcs(reinterpret_cast<const float4*>(a.g) + i);
        float4 m = reinterpret_cast<float4*>(a.m)[i];
        float4 v = reinterpret_cast<float4*>(a.v)[i];
        adam_one(a, w.x, g.x, m.x, v.x);
        adam_one(a, w.y, g.y, m.y, v.y);
        adam_one(a, w.z, g.z, m.z, v.z);
        adam_one(a, w.w, g.w, m.w, v.w);
        reinterpret_cast<float4*>(a.W)[i] = w;
        reinterpret_cast<float4*>(a.m)[i] = m;
        reinterpret_cast<float4*>(a.v)[i] = v;
    }
    // scalar tail (numel % 4), handled by the first threads of block 0
    if (blockIdx.x == 0 && threadIdx.x < (a.numel & 3)) {
        const int64_t i = (n4 << 2) + threadIdx.x;
        float w = a.W[i], m = a.m[i], v = a.v[i];
        adam_one(a, w, a.g[i], m, v);
        a.W[i] = w; a.m[i] = m; a.v[i] = v;
    }
}

cudaError_t launch_adamw(const mo_adamw_tail& t, cudaStream_t s) {
    if (t.numel == 0) return cudaSuccess;
    AdamArgs a;
    a.W = t.W; a.g = t.g; a.m = t.m; a.v = t.v; a.numel = t.numel;
    a.beta1 = t.beta1; a.beta2 = t.beta2; a.eps = t.eps;
    const double bc1 = 1.0 - pow(static_cast<double>(t.beta1), static_cast<double>(t.step));
    const double bc2 = 1.0 - pow(static_cast<double>(t.beta2), static_cast<double>(t.step));
    a.step_size = static_cast<float>(static_cast<double>(t.lr) / bc1);
    a.inv_bc2 = static_cast<float>(1.0 / bc2);
    a.decay = static_cast<float>(static_cast<double>(t.lr) * t.weight_decay);
    const int64_t n4 = t.numel >> 2;
    int64_t blocks = (n4 + 255) / 256;
    const int64_t cap = device_sm_count() * 8LL;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    adamw_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace mo
