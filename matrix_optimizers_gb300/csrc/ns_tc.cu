// Grouped tensor-core GEMM for the quintic Newton-Schulz step on sm_103a.
//
// One persistent launch per phase covers every matrix of the batch:
//   kGram   A = s * X X^T          (X: m x n bf16, K = n; s = 1/||M||_F^2 at step 0)
//   kPoly   B = b*A + c * A A      (K = m; A is symmetric so A A = A A^T)
//   kApply  X' = a*X + B X         (K = m; step 0: X' = (a*M + B Xb)/||M||_F)
//           the last step writes W <- W - lr*wd*W - lr*scale*X' (or the output)
// kGram and kPoly compute only the 128 x 256 tiles that meet the upper
// triangle (j >= i) and store each upper element at (i, j) and (j, i).
//
// Roles per CTA (320 threads, one CTA per SM):
//   warps 0-7  epilogue: tcgen05.ld of the fp32 accumulator, fused math,
//              global stores; warp w reads TMEM lanes 32*(w%4).. and column
//              half w/4 of the 256-column accumulator;
//   warp 8     TMA producer: 64 x 64 bf16 boxes (128-byte swizzle) into a
//              4-stage shared-memory ring (48 KB per stage);
//   warp 9     TMEM allocator and single-thread tcgen05.mma issuer
//              (M = 128, N = 256, K = 16 per instruction) into a double-
//              buffered accumulator (2 x 256 TMEM columns), so the epilogue
//              of one tile overlaps the main loop of the next.
// Every barrier wait is bounded (see ptx.cuh); a timeout raises the CTA's
// abort flag, records an error code and unwinds after draining copies.
#include <cuda_bf16.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace mo {

using bf16 = __nv_bfloat16;

namespace {

constexpr int kStages = 4;
constexpr int kBox = 64;                                   // TMA box edge (elements)
constexpr int kBoxBytes = kBox * kBox * 2;                 // 8 KB
constexpr int kABytes = kTcBM * kTcBK * 2;                 // 16 KB
constexpr int kBBytes = kTcBN * kTcBK * 2;                 // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 32 * (kEpiWarps + 2);
constexpr uint32_t kTmemCols = 512;
constexpr int kCtlBytes = 1024;                            // barriers, TMEM address, abort flag
constexpr int kEpiBufBytesAll = kEpiWarps * 32 * 33 * 4;   // per-warp 32 x 33 fp32 transpose blocks
// ring + control + epilogue blocks + worst-case 1 KB alignment slack = 227 KB
constexpr int kSmemBytes = kStages * kStageBytes + kCtlBytes + kEpiBufBytesAll + 1024;
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB of dynamic shared memory per CTA");

struct Ctl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block overflows its shared-memory slot");

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ float load1(const void* p, int dt, int64_t off) {
    return dt == MO_F32 ? static_cast<const float*>(p)[off] : __bfloat162float(static_cast<const bf16*>(p)[off]);
}
__device__ __forceinline__ void store1(void* p, int dt, int64_t off, float v) {
    if (dt == MO_F32)
        static_cast<float*>(p)[off] = v;
    else
        static_cast<bf16*>(p)[off] = __float2bfloat16_rn(v);
}

// ------------------------------------------------------------- epilogues
// The accumulator arrives in "row layout": lane l of a warp holds row
// rowbase + l, columns j0 .. j0+31.  Global accesses along a row are
// coalesced in "column layout" (lane l holds column j0 + l of rows
// rowbase .. rowbase+31), reached by a 32 x 32 transpose through the warp's
// shared-memory block (33-float rows: conflict-free both ways).  Accesses
// that run down a column of the user matrix (mirror stores, transposed
// matrices) stay in row layout, where consecutive lanes touch consecutive
// addresses.  Both epilogues are called by all 32 lanes (warp-uniform).
constexpr int kEpiPitch = 33;
constexpr int kEpiBufBytes = 32 * kEpiPitch * 4;

__device__ __forceinline__ void transpose32(float* buf, const float (&in)[32], float (&out)[32]) {
    const int lane = threadIdx.x & 31;
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 32; ++k) buf[lane * kEpiPitch + k] = in[k];
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 32; ++r) out[r] = buf[r * kEpiPitch + lane];
}

// Symmetric phases: keep elements with j >= i, store at (i, j) and (j, i).
__device__ __forceinline__ void epi_symmetric(const NsLaunch& p, const MatDesc& md, int rowbase, int j0,
                                              float (&v)[32], float* buf) {
    const int m = md.m, lane = threadIdx.x & 31;
    if (j0 + 31 < rowbase || j0 >= m || rowbase >= m) return;     // block wholly below the diagonal / outside
    bf16* dst = static_cast<bf16*>(p.phase == kGram ? md.gram : md.poly);
    const int jc = j0 + lane;                                        // column-layout column
    float c[32];
    if (p.phase == kGram) {
        const float sc = p.step == 0 ? md.scales[1] : 1.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] *= sc;
        transpose32(buf, v, c);
    } else {
        transpose32(buf, v, c);
        const bf16* A = static_cast<const bf16*>(md.gram);
        float a[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int i = rowbase + r;
            a[r] = (i < m && jc < m) ? __bfloat162float(A[static_cast<int64_t>(i) * md.lda + jc]) : 0.f;
        }
#pragma unroll
        for (int r = 0; r < 32; ++r) c[r] = fmaf(p.c, c[r], p.b * a[r]);
        transpose32(buf, c, v);                                      // back to row layout for the mirror
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) {                                   // (i, j), j >= i: along rows
        const int i = rowbase + r;
        if (i < m && jc < m && jc >= i) dst[static_cast<int64_t>(i) * md.lda + jc] = __float2bfloat16_rn(c[r]);
    }
    const int ir = rowbase + lane;
#pragma unroll
    for (int k = 0; k < 32; ++k) {                                   // (j, i), j > i: down columns
        const int j = j0 + k;
        if (ir < m && j < m && j > ir) dst[static_cast<int64_t>(j) * md.lda + ir] = __float2bfloat16_rn(v[k]);
    }
}

__device__ __forceinline__ void epi_apply(const NsLaunch& p, const MatDesc& md, int rowbase, int j0,
                                          float (&v)[32], float* buf) {
    const int m = md.m, n = md.n, lane = threadIdx.x & 31;
    if (j0 >= n || rowbase >= m) return;
    const int jc = j0 + lane;
    const bool col_ok = jc < n;
    const int ir = rowbase + lane;
    float x[32];                                                     // column layout
    if (p.step == 0 && md.transposed) {
        // X(i, j) = M(j, i): read M down its columns in row layout
        float s[32];
#pragma unroll
        for (int k = 0; k < 32; ++k)
            s[k] = (ir < m && j0 + k < n) ? load1(md.src, md.src_dtype, static_cast<int64_t>(j0 + k) * md.ld + ir)
                                          : 0.f;
        const float inv_s = md.scales[0];
#pragma unroll
        for (int k = 0; k < 32; ++k) s[k] = inv_s * fmaf(p.a, s[k], v[k]);
        transpose32(buf, s, x);
    } else {
        transpose32(buf, v, x);
        float s[32];
        if (p.step == 0) {
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const int i = rowbase + r;
                s[r] = (i < m && col_ok) ? load1(md.src, md.src_dtype, static_cast<int64_t>(i) * md.ld + jc) : 0.f;
            }
            const float inv_s = md.scales[0];
#pragma unroll
            for (int r = 0; r < 32; ++r) x[r] = inv_s * fmaf(p.a, s[r], x[r]);
        } else {
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const int i = rowbase + r;
                s[r] = (i < m && col_ok) ? __ldcs(md.x_master + static_cast<int64_t>(i) * md.ldx + jc) : 0.f;
            }
#pragma unroll
            for (int r = 0; r < 32; ++r) x[r] = fmaf(p.a, s[r], x[r]);
        }
    }
    if (p.step + 1 < p.steps) {
        bf16* xb = static_cast<bf16*>(md.x_op[(p.step + 1) & 1]);
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int i = rowbase + r;
            if (i < m && col_ok) {
                const int64_t o = static_cast<int64_t>(i) * md.ldx + jc;
                __stcs(md.x_master + o, x[r]);
                xb[o] = __float2bfloat16_rn(x[r]);
            }
        }
        return;
    }
    void* dst = p.apply_update ? md.W : md.out;
    if (dst == nullptr) return;
    const int dt = p.apply_update ? md.w_dtype : md.out_dtype;
    if (!md.transposed) {
        float w[32];
        if (p.apply_update) {
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const int i = rowbase + r;
                w[r] = (i < m && col_ok) ? load1(dst, dt, static_cast<int64_t>(i) * md.ld + jc) : 0.f;
            }
#pragma unroll
            for (int r = 0; r < 32; ++r) x[r] = fmaf(-p.alpha, x[r], w[r] - p.decay * w[r]);
        }
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int i = rowbase + r;
            if (i < m && col_ok) store1(dst, dt, static_cast<int64_t>(i) * md.ld + jc, x[r]);
        }
    } else {
        float xr[32];                                                // row layout: X(ir, j0 + k) = U(j0 + k, ir)
        transpose32(buf, x, xr);
        if (p.apply_update) {
            float w[32];
#pragma unroll
            for (int k = 0; k < 32; ++k)
                w[k] = (ir < m && j0 + k < n) ? load1(dst, dt, static_cast<int64_t>(j0 + k) * md.ld + ir) : 0.f;
#pragma unroll
            for (int k = 0; k < 32; ++k) xr[k] = fmaf(-p.alpha, xr[k], w[k] - p.decay * w[k]);
        }
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (ir < m && j0 + k < n) store1(dst, dt, static_cast<int64_t>(j0 + k) * md.ld + ir, xr[k]);
    }
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) ns_tc_kernel(const __grid_constant__ NsLaunch p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + kStages * kStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&ctl->tfull[a]), 1);
            mbar_init(smem_u32(&ctl->tempty[a]), kEpiWarps);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int* abort_flag = &ctl->abort_flag;
    const int2 range = p.cta_range[blockIdx.x];
    const bool mn_b = p.phase == kApply;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed[kStages] = {0, 0, 0, 0};
            bool ok = true;
            for (int t = 0; t < range.y && ok; ++t) {
                const TileDesc td = p.tiles[range.x + t];
                const MatDesc& md = p.mats[td.mat];
                const int i0 = td.ti * kTcBM, j0 = td.tj * kTcBN;
                const CUtensorMap* tma;
                const CUtensorMap* tmb;
                if (p.phase == kGram) {
                    tma = tmb = md.tm_x[p.step & 1];
                } else if (p.phase == kPoly) {
                    tma = tmb = md.tm_gram;
                } else {
                    tma = md.tm_poly;
                    tmb = md.tm_x[p.step & 1];
                }
                for (int kb = 0; kb < td.nkb; ++kb) {
                    const uint32_t empty = smem_u32(&ctl->empty[stage]);
                    const uint32_t full = smem_u32(&ctl->full[stage]);
                    if (!mbar_wait_bounded(empty, phase ^ 1u, abort_flag, p.err, 0x101)) { ok = false; break; }
                    mbar_arrive_expect_tx(full, kStageBytes);
                    ++armed[stage];
                    const uint32_t sa = smem_u32(smem + stage * kStageBytes);
                    const uint32_t sb = sa + kABytes;
                    const int k0 = kb * kTcBK;
                    tma_load_2d(sa, tma, full, k0, i0);
                    tma_load_2d(sa + kBoxBytes, tma, full, k0, i0 + kBox);
                    if (!mn_b) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) tma_load_2d(sb + q * kBoxBytes, tmb, full, k0, j0 + q * kBox);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q) tma_load_2d(sb + q * kBoxBytes, tmb, full, j0 + q * kBox, k0);
                    }
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // let every armed copy land before the CTA exits
                for (int s = 0; s < kStages; ++s) {
                    if (armed[s] == 0) continue;
                    const uint32_t full = smem_u32(&ctl->full[s]);
                    const uint32_t par = (armed[s] - 1u) & 1u;
                    long long t0 = clock64();
                    while (!mbar_try_wait(full, par) && clock64() - t0 < kWaitCycles) {}
                }
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = 0; t < range.y && ok; ++t) {
                const TileDesc td = p.tiles[range.x + t];
                const int acc = t & 1;
                const uint32_t acc_phase = (t >> 1) & 1;
                if (!mbar_wait_bounded(smem_u32(&ctl->tempty[acc]), acc_phase ^ 1u, abort_flag, p.err, 0x102)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * kTcBN);
                for (int kb = 0; kb < td.nkb; ++kb) {
                    if (!mbar_wait_bounded(smem_u32(&ctl->full[stage]), phase, abort_flag, p.err, 0x103)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * kStageBytes);
                    const uint32_t sb = sa + kABytes;
#pragma unroll
                    for (int k = 0; k < kTcBK / 16; ++k) {
                        const uint64_t ad = sdesc_sw128(sa + k * 32, 16, 1024);
                        const uint64_t bd = mn_b ? sdesc_sw128(sb + k * 16 * 128, p.mn_lbo, p.mn_sbo)
                                                 : sdesc_sw128(sb + k * 32, 16, 1024);
                        umma_bf16(d, ad, bd, p.idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    umma_commit(smem_u32(&ctl->empty[stage]));
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(smem_u32(&ctl->tfull[acc]));
            }
            // all issued MMAs complete before TMEM is released
            umma_commit(smem_u32(&ctl->drain));
            long long t0 = clock64();
            while (!mbar_try_wait(smem_u32(&ctl->drain), 0) && clock64() - t0 < kWaitCycles) {}
        }
    } else {
        const int quarter = warp & 3, half = warp >> 2;
        float* buf = reinterpret_cast<float*>(smem + kStages * kStageBytes + kCtlBytes + warp * kEpiBufBytes);
        for (int t = 0; t < range.y; ++t) {
            const TileDesc td = p.tiles[range.x + t];
            const MatDesc& md = p.mats[td.mat];
            const int acc = t & 1;
            const uint32_t acc_phase = (t >> 1) & 1;
            const bool ok = mbar_wait_bounded(smem_u32(&ctl->tfull[acc]), acc_phase, abort_flag, p.err, 0x104);
            if (!__all_sync(0xffffffffu, ok)) break;                     // warp-uniform exit
            tc_fence_after();
            const int rowbase = td.ti * kTcBM + quarter * 32;
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                const int col = half * 128 + ch * 32;
                uint32_t r[32];
                __syncwarp();
                tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(acc * kTcBN + col),
                                   r);
                tmem_wait_ld();
                float v[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
                const int j0 = td.tj * kTcBN + col;
                if (p.phase == kApply)
                    epi_apply(p, md, rowbase, j0, v, buf);
                else
                    epi_symmetric(p, md, rowbase, j0, v, buf);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

int tc_smem_bytes() { return kSmemBytes; }

cudaError_t launch_ns_tc_phase(const NsLaunch& p, int grid, cudaStream_t s) {
    if (grid <= 0) return cudaSuccess;
    static std::atomic<uint64_t> attr_set{0};   // one bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = uint64_t(1) << (dev & 63);
    if (!(attr_set.load() & bit)) {
        e = cudaFuncSetAttribute(ns_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(bit);
    }
    ns_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mo
