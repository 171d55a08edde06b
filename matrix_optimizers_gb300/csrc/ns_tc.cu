// Grouped tensor-core GEMM for the quintic Newton-Schulz step on sm_103a.
//
// Three phases per iteration, each a grouped GEMM over every matrix of the batch:
//   kGram   A = s * X X^T          (X: m x n bf16, K = n; s = 1/||M||_F^2 at step 0)
//   kPoly   B = a*I + b*A + c * A A   (K = m; A is symmetric so A A = A A^T)
//   kApply  X' = B X               (K = m; step 0: X' = B Xb / ||M||_F, Xb = bf16(M))
//           + d_i X(i, j), d_i = B_ii - bf16(B_ii): the bf16 rounding of B's
//           diagonal (values near a = 3.44) is the largest error of the step,
//           so the polynomial epilogue keeps its fp32 residual per row
//           the last step writes W <- W - lr*wd*W - lr*scale*X' (or the output)
// kGram and kPoly compute only the 128 x 256 tiles that meet the upper
// triangle (j >= i) and store each upper element at (i, j) and (j, i).
//
// A launch runs a range of (step, phase) levels.  With one level per launch
// the kernel boundary orders the phases.  A fused launch runs all levels in
// one cooperative persistent grid: each CTA walks its scheduled tiles level by
// level, and a tile waits (its loads, through the dependency warp) on per-matrix
// completion counters that the epilogue warps release, so one matrix's next
// phase starts as soon as its own inputs are complete.
//
// Roles per CTA (608 threads, one CTA per SM):
//   warps 0-15 epilogue: tcgen05.ld of the fp32 accumulator, fused math,
//              stores (the symmetric phases' through a 2 KB shared-memory
//              block per warp and TMA); two groups of 8 warps take alternate
//              tiles (accumulator 0 and 1), so one group's stores drain while
//              the other works; warp w reads TMEM lanes 32*(w%4).. and the
//              128-column slice (w/4)%2 of its group's accumulator;
//   warp 16    TMA producer: 64 x 64 bf16 boxes (128-byte swizzle) into a
//              4-stage shared-memory ring (48 KB per stage);
//   warp 17    TMEM allocator and single-thread tcgen05.mma issuer
//              (M = 128, N = 256, K = 16 per instruction) into a double-
//              buffered accumulator (2 x 256 TMEM columns), so the epilogue
//              of one tile overlaps the main loop of the next;
//   warp 18    dependency waits: runs ahead along the producer's tile list,
//              acquires the completion counters a tile needs and hands the
//              producer and epilogue a shared-memory count of cleared tiles.
// Every barrier wait is bounded (see ptx.cuh); a timeout raises the CTA's
// abort flag, records an error code and unwinds after draining copies.
#include <cuda_bf16.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace mo {

using bf16 = __nv_bfloat16;

namespace {

constexpr int kBox = 64;                                   // TMA box edge (elements)
constexpr int kBoxBytes = kBox * kBox * 2;                 // 8 KB
constexpr int kABytes = kTcBM * kTcBK * 2;                 // 16 KB: 128 rows of A per CTA
constexpr int kEpiWarps = kTcEpiWarps;                     // two groups of 8 that alternate tiles
constexpr int kEpiGroupWarps = kTcEpiGroupWarps;           // 4 lane quarters x 2 column slices
constexpr int kEpiSliceCols = kTcBN / (kEpiGroupWarps / 4);  // 128 accumulator columns per epilogue warp
constexpr int kProducerWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr int kDepWarp = kEpiWarps + 2;
constexpr int kThreads = 32 * (kEpiWarps + 3);
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxStages = 6;
constexpr int kEpiStageBytes = 32 * 32 * 2;                // one epilogue warp's 32 x 32 bf16 store block

// Tile geometry.  Single CTA (cta_group::1): a 128 x 256 tile per CTA, the
// stage holding 128 rows of A and all 256 columns of B.  CTA pair
// (cta_group::2, cluster of 2): a 256 x 256 tile per pair; each CTA holds 128
// rows of A, 128 columns of B and its own 128 x 256 accumulator, so a stage
// is 32 KB and the ring is six deep.
template <bool kPair>
struct Geo {
    static constexpr int kStages = kPair ? 6 : 4;
    static constexpr int kBBoxes = kPair ? 2 : 4;            // 64-wide B boxes per CTA and stage
    static constexpr int kStageBytes = kABytes + kBBoxes * kBoxBytes;
    static constexpr int kTileRows = kPair ? 2 * kTcBM : kTcBM;
    // ring, control block (1 KB), the epilogue warps' store staging, alignment slack
    static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + kEpiWarps * kEpiStageBytes + 1024;
    static constexpr int kTxBytes = (kPair ? 2 : 1) * kStageBytes;   // counted on the leader's full barrier
    static constexpr uint32_t kTemptyCount = (kPair ? 2 : 1) * kEpiGroupWarps;
};
static_assert(Geo<true>::kStages <= kMaxStages && Geo<false>::kStages <= kMaxStages, "ring depth");
static_assert(Geo<true>::kSmemBytes <= 232448 && Geo<false>::kSmemBytes <= 232448, "shared memory");

struct Ctl {                   // 1 KB after the ring; the store staging follows
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint64_t wbar[kEpiWarps];  // per epilogue warp: a TMA load into its staging block has landed
    uint32_t tmem_base;
    int abort_flag;
    int dep_ready;             // tiles of this CTA's list whose inputs the dependency warp has acquired
    int prod_seq;              // tiles of this CTA's list the producer has started loading
};
static_assert(sizeof(Ctl) <= 1024, "control block");

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* v) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        v[2 * q] = __low2float(h[q]);
        v[2 * q + 1] = __high2float(h[q]);
    }
}
__device__ __forceinline__ uint4 pack_bf16x8(const float* v) {
    uint4 u;
    uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
        w[q] = *reinterpret_cast<uint32_t*>(&h);
    }
    return u;
}

// 256-bit global accesses (sm_100 and later): one whole 32-byte sector per
// lane and instruction.  `p` must be 32-byte aligned.
__device__ __forceinline__ void ld_v8(const void* p, uint32_t (&w)[8]) {
    asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}
__device__ __forceinline__ void ld_v8_cs(const void* p, uint32_t (&w)[8]) {     // evict-first
    asm volatile("ld.global.cs.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}
__device__ __forceinline__ void ld_v8_cg(const void* p, uint32_t (&w)[8]) {     // at L2
    asm volatile("ld.global.cg.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}
__device__ __forceinline__ void st_v8(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
__device__ __forceinline__ void st_v8_cs(void* p, const uint32_t (&w)[8]) {     // evict-first
    asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
__device__ __forceinline__ bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31) == 0; }

__device__ __forceinline__ void unpack_bf16x16(const uint32_t (&w)[8], float* v) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        v[2 * q] = __uint_as_float(w[q] << 16);
        v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ void pack_bf16x16(const float* v, uint32_t (&w)[8]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
        w[q] = *reinterpret_cast<uint32_t*>(&h);
    }
}

// 32 consecutive elements starting at p[off]; `nv` of them valid.  A full
// group moves as 32-byte accesses where the row segment is 32-byte aligned
// (16-byte vectors otherwise; offsets are 32-element aligned and leading
// dimensions 16-byte multiples).
__device__ __forceinline__ void load32(const void* p, int dt, int64_t off, int nv, float (&v)[32]) {
    if (nv == 32) {
        if (dt == MO_F32) {
            const float* s = static_cast<const float*>(p) + off;
            if (aligned32(s)) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[8];
                    ld_v8(s + 8 * q, w);
#pragma unroll
                    for (int k = 0; k < 8; ++k) v[8 * q + k] = __uint_as_float(w[k]);
                }
            } else {
                const float4* s4 = reinterpret_cast<const float4*>(s);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 x = s4[q];
                    v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
                }
            }
        } else {
            const bf16* s = static_cast<const bf16*>(p) + off;
            if (aligned32(s)) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t w[8];
                    ld_v8(s + 16 * q, w);
                    unpack_bf16x16(w, &v[16 * q]);
                }
            } else {
                const uint4* s4 = reinterpret_cast<const uint4*>(s);
#pragma unroll
                for (int q = 0; q < 4; ++q) unpack_bf16x8(s4[q], &v[8 * q]);
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            float x = 0.f;
            if (k < nv)
                x = dt == MO_F32 ? static_cast<const float*>(p)[off + k]
                                 : __bfloat162float(static_cast<const bf16*>(p)[off + k]);
            v[k] = x;
        }
    }
}
__device__ __forceinline__ void store32(void* p, int dt, int64_t off, int nv, const float (&v)[32]) {
    if (nv == 32) {
        if (dt == MO_F32) {
            float* d = static_cast<float*>(p) + off;
            if (aligned32(d)) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(v[8 * q + k]);
                    st_v8(d + 8 * q, w);
                }
            } else {
                float4* d4 = reinterpret_cast<float4*>(d);
#pragma unroll
                for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        } else {
            bf16* d = static_cast<bf16*>(p) + off;
            if (aligned32(d)) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t w[8];
                    pack_bf16x16(&v[16 * q], w);
                    st_v8(d + 16 * q, w);
                }
            } else {
                uint4* d4 = reinterpret_cast<uint4*>(d);
#pragma unroll
                for (int q = 0; q < 4; ++q) d4[q] = pack_bf16x8(&v[8 * q]);
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            if (k < nv) {
                if (dt == MO_F32)
                    static_cast<float*>(p)[off + k] = v[k];
                else
                    static_cast<bf16*>(p)[off + k] = __float2bfloat16_rn(v[k]);
            }
        }
    }
}
// bf16 Gram entries written by other CTAs of the same launch: read at L2
// (ld.global.cg), never from a non-coherent cache.
__device__ __forceinline__ void load32_bf16_l2(const bf16* p, int64_t off, int nv, float (&v)[32]) {
    if (nv == 32) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint32_t w[8];
            ld_v8_cg(p + off + 16 * q, w);        // lda is a multiple of 64: 32-byte aligned
            unpack_bf16x16(w, &v[16 * q]);
        }
    } else {
        const unsigned short* h = reinterpret_cast<const unsigned short*>(p + off);
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = k < nv ? __uint_as_float(static_cast<uint32_t>(__ldcg(h + k)) << 16) : 0.f;
    }
}
__device__ __forceinline__ float load1(const void* p, int dt, int64_t off) {
    return dt == MO_F32 ? static_cast<const float*>(p)[off] : __bfloat162float(static_cast<const bf16*>(p)[off]);
}
__device__ __forceinline__ void store1(void* p, int dt, int64_t off, float v) {
    if (dt == MO_F32)
        static_cast<float*>(p)[off] = v;
    else
        static_cast<bf16*>(p)[off] = __float2bfloat16_rn(v);
}

// Oriented access to a user matrix: X(i, j) = U(i, j), or U(j, i) when the
// matrix was transposed to reach m <= n.  Transposed accesses are per
// element; across a warp (consecutive i) they are contiguous.
__device__ __forceinline__ void user_load32(const MatDesc& md, const void* p, int dt, int i, int j0, int nv,
                                            float (&v)[32]) {
    if (!md.transposed) {
        load32(p, dt, static_cast<int64_t>(i) * md.ld + j0, nv, v);
    } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = k < nv ? load1(p, dt, static_cast<int64_t>(j0 + k) * md.ld + i) : 0.f;
    }
}
__device__ __forceinline__ void user_store32(const MatDesc& md, void* p, int dt, int i, int j0, int nv,
                                             const float (&v)[32]) {
    if (!md.transposed) {
        store32(p, dt, static_cast<int64_t>(i) * md.ld + j0, nv, v);
    } else {
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (k < nv) store1(p, dt, static_cast<int64_t>(j0 + k) * md.ld + i, v[k]);
    }
}

// ------------------------------------------------------------- epilogues
// Symmetric phases.  The warp holds the 32 x 32 block of rows i0 + lane
// and columns j0 .. j0 + 31 (one row per lane).  Blocks below the diagonal
// are dropped; a block above it is stored at (i0, j0) and, transposed, at
// (j0, i0); a diagonal block (j0 == i0) is stored once, holding the upper
// values in both triangles, so each element of the symmetric result comes
// from the one upper-triangle accumulator entry.  The blocks go out through
// the warp's 2 KB shared-memory block and TMA stores (a warp's scattered
// 32- and 64-byte row pieces measured several times slower).  The staging
// uses the 64-byte swizzle of the store view: 16-byte chunk c of row r sits
// at chunk c ^ ((r >> 1) & 3), which spreads a warp's writes over all banks.
__device__ __forceinline__ uint32_t stage_off(int r, int c16) {
    return static_cast<uint32_t>(r * 64 + ((c16 ^ ((r >> 1) & 3)) << 4));
}
__device__ __forceinline__ void st_shared_v4(uint32_t a, const uint4& v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_shared_b16(uint32_t a, bf16 v) {
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(*reinterpret_cast<unsigned short*>(&v)) : "memory");
}

// Called by all 32 lanes of the warp; lane 0 issues the copies.  `sbuf` is
// the warp's staging block (shared-memory address), `wbar` its barrier and
// `wuse` / `wpend` its use count and in-flight flag (see epi_update_tma).
// The polynomial phase's A block, read for bA, comes into the staging block by
// a TMA load (each lane's 32-byte pieces, 32 rows per instruction, are many
// small requests).  Returns false when that wait gave up.
__device__ __forceinline__ bool epi_symmetric(const NsLaunch& p, const MatDesc& md, int phase, int step, int i0,
                                              int j0, float (&v)[32], uint32_t sbuf, uint32_t wbar, uint32_t& wuse,
                                              bool& wpend, volatile int* abort_flag) {
    const int lane = threadIdx.x & 31;
    const int m = md.m;
    if (j0 < i0 || j0 >= m || i0 >= m) return true;             // warp-uniform
    const int i = i0 + lane;
    const bool row_ok = i < m;
    const int nv = min(32, m - j0);
    if (phase == kGram) {
        const float sc = step == 0 ? md.scales[1] : 1.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] *= sc;
    } else {
        if (lane == 0) {
            bulk_wait_read_all();                    // the last store has read the block
            if (p.deps) fence_proxy_async_global();  // A was released by other CTAs
            mbar_arrive_expect_tx(wbar, kEpiStageBytes);
            tma_load_2d(sbuf, md.tm_gram_st, wbar, j0, i0);
        }
        wpend = true;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(wbar, wuse & 1u, abort_flag, p.err, 0x107))) return false;
        wpend = false;
        ++wuse;
        float a[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint4 u;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                         : "r"(sbuf + stage_off(lane, c))
                         : "memory");
            unpack_bf16x8(u, &a[8 * c]);
        }
        __syncwarp();                                // the block is read: the stores may reuse it
        // step 0 folds the spectral scale into the coefficients (1 otherwise);
        // the diagonal also takes a: B = bA + cA^2 + aI, so that the apply
        // phase is the plain product X' = B X
        const float bs = step == 0 ? p.b * md.scales[2] : p.b;
        const float cs = step == 0 ? p.c * md.scales[3] : p.c;
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = fmaf(cs, v[k], bs * a[k]) + (j0 + k == i ? p.a : 0.f);
        if (row_ok && i >= j0 && i < j0 + nv) {
            // the diagonal lies near a = 3.44, where the bf16 spacing is 2^-6:
            // keep its rounding residual (exact in fp32) for the apply epilogue
            float dv = 0.f;
#pragma unroll
            for (int k = 0; k < 32; ++k)
                if (j0 + k == i) dv = v[k];
            md.dlo[i] = dv - __bfloat162float(__float2bfloat16_rn(dv));
        }
    }
    const CUtensorMap* tm = phase == kGram ? md.tm_gram_st : md.tm_poly_st;
    if (lane == 0) bulk_wait_read_all();             // the last store has read the block
    __syncwarp();
    if (j0 != i0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) st_shared_v4(sbuf + stage_off(lane, c), pack_bf16x8(&v[8 * c]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tm, sbuf, j0, i0);
            bulk_commit();
            bulk_wait_read_all();
        }
        __syncwarp();
        // the transpose: row k of the block at (j0, i0) is column k of this one
#pragma unroll
        for (int k = 0; k < 32; ++k)
            st_shared_b16(sbuf + stage_off(k, lane >> 3) + (lane & 7) * 2, __float2bfloat16_rn(v[k]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tm, sbuf, i0, j0);
            bulk_commit();
        }
    } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const bf16 h = __float2bfloat16_rn(v[k]);
            if (k >= lane) st_shared_b16(sbuf + stage_off(lane, k >> 3) + (k & 7) * 2, h);
            if (k > lane) st_shared_b16(sbuf + stage_off(k, lane >> 3) + (lane & 7) * 2, h);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tm, sbuf, j0, i0);
            bulk_commit();
        }
    }
    return true;
}

// Fused Sign-Muon sign + 1-bit pack of the last step's output: bit = 1
// unless the output, as stored in out_dtype, is below zero; bits follow the
// row-major flattening of the user matrix, whose column count is a multiple
// of 32, so every word is written whole by one warp.
__device__ __forceinline__ bool sign_bit(float v, int out_dtype) {
    if (out_dtype == MO_BF16) v = __bfloat162float(__float2bfloat16_rn(v));
    return !(v < 0.f);
}

__device__ __forceinline__ void epi_sign_pack(const MatDesc& md, int i, bool row_ok, int j0, int nv,
                                              const float (&x)[32]) {
    const int lane = threadIdx.x & 31;
    if (!md.transposed) {
        // the lane's 32 columns are one word of its row
        if (!row_ok) return;
        uint32_t w = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (k < nv && sign_bit(x[k], md.out_dtype)) w |= 1u << k;
        md.sign_words[(static_cast<int64_t>(i) * md.cols + j0) >> 5] = w;
    } else {
        // lanes are 32 consecutive user columns: one ballot per user row j0 + k
        uint32_t mine = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const uint32_t w = __ballot_sync(0xffffffffu, row_ok && k < nv && sign_bit(x[k], md.out_dtype));
            if (lane == k) mine = w;
        }
        const int rowbase = i - lane;
        if (rowbase < md.m && lane < nv)
            md.sign_words[(static_cast<int64_t>(j0 + lane) * md.cols + rowbase) >> 5] = mine;
    }
}

// The apply epilogue's share of the diagonal correction: the lane's 32
// operand elements X(i, j0 .. j0+31) (4 x 8-column blocks) and the residual
// d_i of B's diagonal.  Both were written by other CTAs of the launch: read
// at L2.
__device__ __forceinline__ void load_diag_fix(const MatDesc& md, int step, int i, bool row_ok, int j0, uint4 (&xr)[4],
                                              float& di) {
    di = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) xr[q] = make_uint4(0, 0, 0, 0);
    if (!row_ok || j0 >= md.n) return;
    di = __ldcg(md.dlo + i);
    const uint4* src = static_cast<const uint4*>(md.x_op[step & 1]) + static_cast<int64_t>(j0 >> 3) * md.xrows + i;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (j0 + 8 * q < md.n) xr[q] = __ldcg(src + static_cast<int64_t>(q) * md.xrows);
}

// Last-step weight update W <- W - decay W - alpha X' of the warp's 32 x 32
// block through its staging block: a TMA load of W's box (32 rows x 64 B:
// 16 fp32 or 32 bf16 columns, so an fp32 block takes two), the update in
// shared memory, a TMA store back.  Each lane's own 32-byte row pieces of W,
// 32 rows per warp instruction, took about twice as long.  In the transposed
// frame the box's rows are W's rows j0 .. j0 + 31 and a lane reads a column
// of it.  `wuse` counts the warp's loads into its staging block (the parity
// of its barrier); `wpend` is set while one may still be landing (a wait
// that gave up), for the drain before the CTA exits.  Called by all 32 lanes.
__device__ __forceinline__ bool epi_update_tma(const NsLaunch& p, const MatDesc& md, int i0, int j0,
                                               const float (&x)[32], uint32_t sbuf, uint32_t wbar, uint32_t& wuse,
                                               bool& wpend, volatile int* abort_flag) {
    const int lane = threadIdx.x & 31;
    const bool f32 = md.w_dtype == MO_F32;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (h == 1 && !f32) break;
        const int off = f32 ? 16 * h : 0;
        const int bx = md.transposed ? i0 + off : j0 + off;
        const int by = md.transposed ? j0 : i0;
        if (lane == 0) {
            bulk_wait_read_all();                    // the last store has read the block
            mbar_arrive_expect_tx(wbar, kEpiStageBytes);
            tma_load_2d(sbuf, md.tm_w, wbar, bx, by);
        }
        wpend = true;
        const bool ok = mbar_wait_bounded(wbar, wuse & 1u, abort_flag, p.err, 0x106);
        if (!__all_sync(0xffffffffu, ok)) return false;
        wpend = false;
        ++wuse;
        if (!md.transposed) {
            // lane = row: 4 chunks of 16 bytes
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t a = sbuf + stage_off(lane, c);
                uint4 u;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                             : "r"(a)
                             : "memory");
                if (f32) {
                    float w[4] = {__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                  __uint_as_float(u.w)};
#pragma unroll
                    for (int e = 0; e < 4; ++e) w[e] = fmaf(-p.alpha, x[off + 4 * c + e], w[e] - p.decay * w[e]);
                    u = make_uint4(__float_as_uint(w[0]), __float_as_uint(w[1]), __float_as_uint(w[2]),
                                   __float_as_uint(w[3]));
                } else {
                    float w[8];
                    unpack_bf16x8(u, w);
#pragma unroll
                    for (int e = 0; e < 8; ++e) w[e] = fmaf(-p.alpha, x[8 * c + e], w[e] - p.decay * w[e]);
                    u = pack_bf16x8(w);
                }
                st_shared_v4(a, u);
            }
        } else if (f32) {
            // lanes 16h .. 16h + 15 own the box's columns (their rows of X')
            if ((lane >> 4) == h) {
                const int col = lane & 15;
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const uint32_t a = sbuf + stage_off(k, col >> 2) + (col & 3) * 4;
                    float w;
                    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(w) : "r"(a) : "memory");
                    w = fmaf(-p.alpha, x[k], w - p.decay * w);
                    asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(w) : "memory");
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const uint32_t a = sbuf + stage_off(k, lane >> 3) + (lane & 7) * 2;
                unsigned short hb;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(hb) : "r"(a) : "memory");
                float w = __uint_as_float(static_cast<uint32_t>(hb) << 16);
                w = fmaf(-p.alpha, x[k], w - p.decay * w);
                st_shared_b16(a, __float2bfloat16_rn(w));
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(md.tm_w, sbuf, bx, by);
            bulk_commit();
        }
    }
    return true;
}

// Called by all 32 lanes of a warp (the fused pack takes warp ballots);
// lanes whose row lies beyond the matrix touch no memory.
// Returns false when a wait of the weight update gave up.
__device__ __forceinline__ bool epi_apply(const NsLaunch& p, const MatDesc& md, int step, int i, bool row_ok,
                                          int j0, float (&v)[32], uint32_t sbuf, uint32_t wbar, uint32_t& wuse,
                                          bool& wpend, volatile int* abort_flag) {
    const int n = md.n;
    if (j0 >= n) return true;
    const int nv = row_ok ? min(32, n - j0) : 0;
    uint4 xr[4];
    float di;
    load_diag_fix(md, step, i, row_ok, j0, xr, di);
    float (&x)[32] = v;
    // X' = (aI + bA + cA^2) X is the accumulator (the polynomial phase put a
    // on B's diagonal), plus d_i X(i, j) for the diagonal's bf16 residual;
    // step 0 multiplied the unscaled bf16(M), so it scales.
    const float scale = step == 0 ? md.scales[0] * md.scales[4] : 1.f;   // 1/||M||_F (x 1/sigma_hat)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float xo[8];
        unpack_bf16x8(xr[q], xo);
#pragma unroll
        for (int r = 0; r < 8; ++r) x[8 * q + r] = scale * fmaf(di, xo[r], v[8 * q + r]);
    }
    if (step + 1 < p.steps) {
        // the next operand, in 8-column blocks: the warp's 32 rows of one block
        // are 512 contiguous bytes (columns past n hold the accumulator's zeros)
        if (!row_ok) return true;
        uint4* dst = static_cast<uint4*>(md.x_op[(step + 1) & 1]) + static_cast<int64_t>(j0 >> 3) * md.xrows + i;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (j0 + 8 * q < n) dst[static_cast<int64_t>(q) * md.xrows] = pack_bf16x8(&x[8 * q]);
        return true;
    }
    if (md.sign_words != nullptr) {
        epi_sign_pack(md, i, row_ok, j0, min(32, n - j0), x);
        return true;
    }
    if (p.apply_update && md.W != nullptr && md.tm_w != nullptr)
        return epi_update_tma(p, md, i - (threadIdx.x & 31), j0, x, sbuf, wbar, wuse, wpend, abort_flag);
    if (!row_ok) return true;
    if (p.apply_update) {
        if (md.W == nullptr) return true;
        float w[32];
        user_load32(md, md.W, md.w_dtype, i, j0, nv, w);
#pragma unroll
        for (int k = 0; k < 32; ++k) w[k] = fmaf(-p.alpha, x[k], w[k] - p.decay * w[k]);
        user_store32(md, md.W, md.w_dtype, i, j0, nv, w);
    } else if (md.out != nullptr) {
        user_store32(md, md.out, md.out_dtype, i, j0, nv, x);
    }
    return true;
}

// Last NS step with the weight update: while the epilogue waits for the
// current tile, pull this lane's W lines of the CTA's next apply tile into L2,
// so that the update's loads find them there instead of waiting on DRAM.
// Only for short K (= m): a long tile hides the update's latency anyway, and
// over its longer period the operand stream evicts part of the prefetched
// lines, which are then read twice.
// The lane's row (row_off within the tile) and the slice column col0 follow
// the epilogue's own mapping; each 32-column chunk the update reads is one
// line per lane (W row i, or in the transposed frame W row j0 + lane).
constexpr int kPrefetchUpdateMaxK = 2048;
__device__ __noinline__ void prefetch_update_tile(const NsLaunch& p, int tile, int tile_rows, int row_off,
                                                  int col0, int lane) {
    const TileDesc td = p.tc_tiles[kApply][tile];
    const MatDesc& md = p.mats[td.mat];
    const int i = td.ti * tile_rows + row_off;
    if (md.W == nullptr || md.sign_words != nullptr || md.m > kPrefetchUpdateMaxK) return;
    const char* w = static_cast<const char*>(md.W);
    const int esz = md.w_dtype == MO_F32 ? 4 : 2;
#pragma unroll
    for (int ch = 0; ch < kEpiSliceCols / 32; ++ch) {
        const int j0 = td.tj * kTcBN + col0 + ch * 32;
        if (!md.transposed) {
            if (i < md.m && j0 < md.n) prefetch_l2(w + (static_cast<int64_t>(i) * md.ld + j0) * esz);
        } else {
            const int r0 = i - lane;
            if (r0 < md.m && j0 + lane < md.n) prefetch_l2(w + (static_cast<int64_t>(j0 + lane) * md.ld + r0) * esz);
        }
    }
}

// ------------------------------------------------- fused-launch dependencies
// A fused launch runs several (step, phase) levels; a tile of level (t, ph)
// of matrix md may start once, within this launch, every tile it reads or
// overwrites the inputs of has finished:
//   Gram(t)  reads X_t from Apply(t-1) and overwrites A, read by Poly(t-1);
//   Poly(t)  reads A_t from Gram(t) and overwrites B, read by Apply(t-1);
//   Apply(t) reads B_t from Poly(t), X_t from Apply(t-1), and overwrites the
//            other X operand, read by Gram(t-1) and Apply(t-1).
// Each warp of the epilogue group that finished a tile releases one count (8
// per CTA, so 8 or 16 per tile), so phase ph of step s is complete when its counter reaches
// (its tiles x releases per tile) times
// the number of its steps up to s that this launch runs.  The counters are
// per matrix (mode 1), or one set over all matrices (mode 2: each level then
// waits for the whole previous level, a grid-wide barrier per phase).
struct Deps {
    int* cnt;                 // [3] completion counters
    int nt_sym, nt_apply;     // tiles they count per symmetric / apply level
};
__device__ __forceinline__ Deps deps_of(const NsLaunch& p, const MatDesc& md) {
    return p.deps == 2 ? Deps{p.level_deps, p.tot_sym, p.tot_apply} : Deps{md.deps, md.nt_sym, md.nt_apply};
}

__device__ __forceinline__ int dep_need(const NsLaunch& p, const Deps& d, int ph, int upto) {
    const int first = (p.lv_begin - ph + 2) / 3;      // first step of phase ph in this launch
    const int cnt = upto - first + 1;
    return cnt <= 0 ? 0 : cnt * (ph == kApply ? d.nt_apply : d.nt_sym) * p.rel_per_tile;
}

// Returns 1 when the dependencies were already met, 2 after spinning, 0 on
// timeout / abort; *waited_ns accumulates the time spent spinning.
__device__ __noinline__ int wait_deps(const NsLaunch& p, const Deps& d, int ph, int step, bool stall,
                                      volatile int* abort_flag, unsigned long long* waited_ns) {
    // a stalled matrix needs far more releases than a launch can give
    const int need_g = dep_need(p, d, kGram, ph == kGram ? step - 1 : step) + (stall ? (1 << 30) : 0);
    const int need_p = dep_need(p, d, kPoly, ph == kApply ? step : step - 1);
    const int need_a = dep_need(p, d, kApply, step - 1);
    long long t0 = 0;
    unsigned long long g0 = 0;
    for (uint32_t it = 0;; ++it) {
        const bool ready = (need_g == 0 || ld_acquire_gpu(d.cnt + kGram) >= need_g) &&
                           (need_p == 0 || ld_acquire_gpu(d.cnt + kPoly) >= need_p) &&
                           (need_a == 0 || ld_acquire_gpu(d.cnt + kApply) >= need_a);
        if (ready) {
            if (it == 0) return 1;
            *waited_ns += globaltimer_ns() - g0;
            return 2;
        }
        if (it == 0) {
            t0 = clock64();
            g0 = globaltimer_ns();
        }
        if (*abort_flag || *static_cast<volatile int*>(p.err) != 0) {
            *abort_flag = 1;
            return 0;
        }
        if (clock64() - t0 > p.dep_wait_cycles) {
            *abort_flag = 1;
            atomicCAS(p.err, 0, 0x105);
            return 0;
        }
        __nanosleep(100);
    }
}

// A symmetric-phase tile whose first 128 columns lie wholly below the
// diagonal (row block 2J + 1 of column block J) computes only its last 128
// columns: an N = 128 MMA over half of B, into the accumulator's upper 128
// columns.  Its epilogue skips the first 128 columns as it does any block
// below the diagonal.  Single-CTA tiles only.
template <bool kPair>
__device__ __forceinline__ bool half_tile(int ph, const TileDesc& td) {
    return !kPair && ph != kApply && td.tj * kTcBN + kTcBN / 2 <= td.ti * kTcBM;
}

// Gram tiles with at least this many K blocks alternate their K direction.
constexpr int kReverseMinKBlocks = 64;

// The producer's wait for the dependency warp to clear tile `seq` of the
// CTA's list: a CTA-scope acquire of its count.  The dependency warp either
// advances the count or raises the abort flag within its own bound, so this
// wait's bound (that one plus the barrier bound) only guards against a bug.
__device__ __forceinline__ bool wait_dep_ready(Ctl* ctl, int seq, volatile int* abort_flag, int* err,
                                               long long limit) {
    if (ld_acquire_cta_smem(&ctl->dep_ready) > seq) return true;
    const long long t0 = clock64();
    for (;;) {
        __nanosleep(32);   // a tight spin would take issue slots from the epilogue warps beside it
        if (ld_acquire_cta_smem(&ctl->dep_ready) > seq) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            atomicCAS(err, 0, 0x108);
            return false;
        }
    }
}

// The dependency warp starts a tile's wait only once the producer has started
// the tile this many places before it: early enough to take the acquire off
// the producer's path, late enough that 152 CTAs do not poll a grid-wide
// counter for a whole level (those polls crowd the L2 slice that serves it).
constexpr int kDepLead = 2;

__device__ __forceinline__ bool wait_producer_near(const Ctl* ctl, int seq, volatile int* abort_flag, int* err) {
    const volatile int* ps = &ctl->prod_seq;
    if (*ps + kDepLead >= seq) return true;
    const long long t0 = clock64();
    for (;;) {
        __nanosleep(128);
        if (*ps + kDepLead >= seq) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitCycles) {
            *abort_flag = 1;
            atomicCAS(err, 0, 0x109);
            return false;
        }
    }
}

// TMA loads of one box, the pair form counting on the leader's barrier.
template <bool kPair>
__device__ __forceinline__ void load2(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y) {
    if constexpr (kPair)
        tma_load_2d_pair(dst, m, bar, x, y);
    else
        tma_load_2d(dst, m, bar, x, y);
}
// blocked operand (3D view): box origin at row group y, column block z
template <bool kPair>
__device__ __forceinline__ void load3(uint32_t dst, const CUtensorMap* m, uint32_t bar, int y, int z) {
    if constexpr (kPair)
        tma_load_3d_pair(dst, m, bar, 0, y, z);
    else
        tma_load_3d(dst, m, bar, 0, y, z);
}

// Tiles of phase ph scheduled on schedule unit `unit` (a CTA, or a CTA pair).
__device__ __forceinline__ int2 unit_tiles(const NsLaunch& p, int ph, int unit) {
    return unit < p.tc_ctas[ph] ? p.tc_ranges[ph][unit] : make_int2(0, 0);
}

}  // namespace


// 608 threads are 19 warps, so three of the SM's four sub-partitions hold 5
// of them: 16 K registers per sub-partition cap a thread at 96 (a larger per-kernel cap
// leaves the block unlaunchable).
template <bool kPair>
__global__ void __launch_bounds__(kThreads, 1) ns_tc_kernel(const __grid_constant__ NsLaunch p) {
    using G = Geo<kPair>;
    constexpr int kBRows = G::kBBoxes * kBox;                 // B-operand rows (Gram) one CTA holds
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + G::kStages * G::kStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;      // rank 0 leads the pair
    const bool leader = rank == 0;
    const int unit = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < G::kStages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&ctl->tfull[a]), 1);
            mbar_init(smem_u32(&ctl->tempty[a]), G::kTemptyCount);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        for (int w = 0; w < kEpiWarps; ++w) mbar_init(smem_u32(&ctl->wbar[w]), 1);
        ctl->abort_flag = 0;
        ctl->dep_ready = 0;
        ctl->prod_seq = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        if constexpr (kPair) {
            tmem_alloc_pair(smem_u32(&ctl->tmem_base), kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync();          // both CTAs' barriers exist before any remote signal
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int* abort_flag = &ctl->abort_flag;
    if (p.stamps != nullptr && threadIdx.x == 0) p.stamps[4 * blockIdx.x] = globaltimer_ns();

    if (warp == kProducerWarp) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t narmed = 0;                     // stages armed so far, in ring order
            bool ok = true;
            int seq = 0;                             // tiles so far in this CTA's list
            for (int lv = p.lv_begin; lv < p.lv_end && ok; ++lv) {
                const int ph = lv % 3, step = lv / 3;
                const int2 range = unit_tiles(p, ph, unit);
                int dep_key = -1;                    // counter set last seen met at this level
                for (int t = 0; t < range.y && ok; ++t, ++seq) {
                    const TileDesc td = p.tc_tiles[ph][range.x + t];
                    const MatDesc& md = p.mats[td.mat];
                    const int key = p.deps == 2 ? 0 : td.mat;
                    if (p.deps) *static_cast<volatile int*>(&ctl->prod_seq) = seq;
                    if (p.deps && key != dep_key) {
                        // the dependency warp, running ahead along the same list, has
                        // acquired the inputs of this tile and of the tiles after it
                        // up to the next change of counter set
                        if (!wait_dep_ready(ctl, seq, abort_flag, p.err, p.dep_wait_cycles + kWaitCycles)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_global();
                        dep_key = key;
                    }
                    // this CTA's rows of A and columns of B
                    const int i0 = td.ti * G::kTileRows + static_cast<int>(rank) * kTcBM;
                    const int j0 = td.tj * kTcBN + (kPair ? static_cast<int>(rank) * (kTcBN / 2) : 0);
                    const CUtensorMap* tma;
                    const CUtensorMap* tmb;
                    if (ph == kGram) {                 // both from the blocked operand
                        tma = md.tm_xa[step & 1];
                        tmb = md.tm_xb[step & 1];
                    } else if (ph == kPoly) {          // both from A (128-byte swizzle)
                        tma = md.tm_gram;
                        tmb = md.tm_gram_b;
                    } else {                           // B (swizzled), then the blocked operand
                        tma = md.tm_poly;
                        tmb = md.tm_xn[step & 1];
                    }
                    // one K loop per phase, chosen once per tile: the copies differ by
                    // phase, and any branch among them inside the loop measured ~20%
                    // slower in every phase (the producer's issue rate is on the
                    // critical path).  In the Gram phase with a long K, every other
                    // tile of the CTA's list walks K backwards: the CTAs of one wave
                    // stream the X panels' K slices together, so the next wave starts
                    // on the slices the last one read most recently, still in L2
                    // (walking one way each wave re-reads from DRAM what the wave
                    // before evicted)
                    const bool rev = ph == kGram && td.nkb >= kReverseMinKBlocks && (t & 1);
                    const int k_last = rev ? td.nkb - 1 : 0;
                    const int k_inc = rev ? -1 : 1;
                    const bool half = half_tile<kPair>(ph, td);
                    const uint32_t tx = half ? static_cast<uint32_t>(2 * kABytes) : static_cast<uint32_t>(G::kTxBytes);
                    auto k_loop = [&](auto&& load) {
                        for (int kb = 0, kk = k_last; kb < td.nkb; ++kb, kk += k_inc) {
                            const uint32_t empty = smem_u32(&ctl->empty[stage]);
                            const uint32_t full = smem_u32(&ctl->full[stage]);
                            if (!mbar_wait_bounded(empty, phase ^ 1u, abort_flag, p.err, 0x101)) {
                                ok = false;
                                return;
                            }
                            if (leader) mbar_arrive_expect_tx(full, tx);
                            ++narmed;
                            const uint32_t sa = smem_u32(smem + stage * G::kStageBytes);
                            const uint32_t bar = kPair ? mapa_shared(full, 0) : full;   // the leader's barrier
                            load(sa, sa + kABytes, bar, kk * kTcBK);
                            if (++stage == G::kStages) { stage = 0; phase ^= 1u; }
                        }
                    };
                    if (ph == kGram && half) {
                        // B: the tile's last 128 rows, through the 128-row view
                        k_loop([&](uint32_t sa, uint32_t sb, uint32_t bar, int k0) {
                            load3<kPair>(sa, tma, bar, i0 >> 3, k0 >> 3);
                            load3<kPair>(sb, tma, bar, (j0 + kTcBN / 2) >> 3, k0 >> 3);
                        });
                    } else if (ph == kGram) {
                        k_loop([&](uint32_t sa, uint32_t sb, uint32_t bar, int k0) {
                            load3<kPair>(sa, tma, bar, i0 >> 3, k0 >> 3);
                            load3<kPair>(sb, tmb, bar, j0 >> 3, k0 >> 3);
                        });
                    } else if (ph == kPoly && half) {
                        k_loop([&](uint32_t sa, uint32_t sb, uint32_t bar, int k0) {
                            load2<kPair>(sa, tma, bar, k0, i0);
                            load2<kPair>(sb, tma, bar, k0, j0 + kTcBN / 2);
                        });
                    } else if (ph == kPoly) {
                        k_loop([&](uint32_t sa, uint32_t sb, uint32_t bar, int k0) {
                            // 128 rows of A and all B rows of the stage, one copy each
                            load2<kPair>(sa, tma, bar, k0, i0);
                            load2<kPair>(sb, tmb, bar, k0, j0);
                        });
                    } else {
                        k_loop([&](uint32_t sa, uint32_t sb, uint32_t bar, int k0) {
                            load2<kPair>(sa, tma, bar, k0, i0);
                            load3<kPair>(sb, tmb, bar, k0 >> 3, j0 >> 3);
                        });
                    }
                }
            }
            if (leader) {
                // every armed copy lands before the CTA exits, also when the MMA
                // warp gave up before consuming them (a no-op when it consumed
                // them all); in a pair the leader's barriers also count the
                // peer's copies of the stages it armed
                for (int s = 0; s < G::kStages; ++s) {
                    // stage s was armed by the arms s, s + kStages, ...
                    if (narmed <= static_cast<uint32_t>(s)) continue;
                    const uint32_t times = (narmed - 1u - static_cast<uint32_t>(s)) / G::kStages + 1u;
                    const uint32_t full = smem_u32(&ctl->full[s]);
                    const uint32_t par = (times - 1u) & 1u;
                    long long t0 = clock64();
                    while (!mbar_try_wait(full, par) && clock64() - t0 < kWaitCycles) {}
                }
            } else if (!ok) {
                // the peer cannot wait on the leader's barriers, which its copies
                // complete on: give those in flight time to land (~2 ms, far
                // above a copy's latency); the closing cluster barrier keeps
                // this CTA's shared memory alive until the leader has drained
                long long t0 = clock64();
                while (clock64() - t0 < (1LL << 22)) {}
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int q = 0;                                // tiles so far: accumulator ping-pong
            for (int lv = p.lv_begin; lv < p.lv_end && ok; ++lv) {
                const int ph = lv % 3;
                const int2 range = unit_tiles(p, ph, unit);
                const bool mn_b = ph == kApply;
                const uint32_t idesc = mn_b ? p.idesc_apply : p.idesc_sym;
                // Descriptors with a zero address field, and the per-16-wide-K-step
                // address increments (16-byte units), by phase: Gram reads both
                // operands blocked (no swizzle, K-major: 8-column blocks rows x 16 B
                // apart, 8-row groups 128 B apart); poly reads A swizzled twice;
                // apply reads B swizzled and the blocked operand MN-major (8-row K
                // groups 128 B apart, 8-column blocks 1 KB apart; 16 K rows = 256 B)
                uint64_t adesc0, bdesc0;
                uint32_t a_step, b_step;
                if (ph == kGram) {
                    adesc0 = sdesc_noswz(0, kTcBM * 16, 128);
                    bdesc0 = sdesc_noswz(0, kBRows * 16, 128);
                    a_step = (2 * kTcBM * 16) >> 4;
                    b_step = (2 * kBRows * 16) >> 4;
                } else if (ph == kPoly) {
                    adesc0 = bdesc0 = sdesc_sw128(0, 16, 1024);
                    a_step = b_step = 32 >> 4;
                } else {
                    adesc0 = sdesc_sw128(0, 16, 1024);
                    bdesc0 = sdesc_noswz(0, p.mn_lbo, p.mn_sbo);
                    a_step = 32 >> 4;
                    b_step = 256 >> 4;
                }
                for (int t = 0; t < range.y && ok; ++t, ++q) {
                    const TileDesc td = p.tc_tiles[ph][range.x + t];
                    const int acc = q & 1;
                    const uint32_t acc_phase = (q >> 1) & 1;
                    if (!mbar_wait_bounded(smem_u32(&ctl->tempty[acc]), acc_phase ^ 1u, abort_flag, p.err, 0x102)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // a half tile: N = 128 into the accumulator's last 128 columns; the
                    // Gram phase's 128-row B block has half the column-block stride
                    const bool half = half_tile<kPair>(ph, td);
                    const uint32_t idesc_t = half ? idesc_bf16_f32(kTcBM, kTcBN / 2, 0u) : idesc;
                    const uint64_t bdesc_t = half && ph == kGram ? sdesc_noswz(0, (kBRows / 2) * 16, 128) : bdesc0;
                    const uint32_t b_step_t = half && ph == kGram ? (2 * (kBRows / 2) * 16) >> 4 : b_step;
                    const uint32_t d = tmem + static_cast<uint32_t>(acc * kTcBN + (half ? kTcBN / 2 : 0));
                    for (int kb = 0; kb < td.nkb; ++kb) {
                        if (!mbar_wait_bounded(smem_u32(&ctl->full[stage]), phase, abort_flag, p.err, 0x103)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = smem_u32(smem + stage * G::kStageBytes);
                        const uint32_t sb = sa + kABytes;
#pragma unroll
                        for (int k = 0; k < kTcBK / 16; ++k) {
                            // shared addresses stay below 256 KB: the 14-bit field never carries
                            const uint64_t ad = adesc0 + ((sa >> 4) + k * a_step);
                            const uint64_t bd = bdesc_t + ((sb >> 4) + k * b_step_t);
                            if constexpr (kPair)
                                umma_bf16_pair(d, ad, bd, idesc_t, (kb | k) != 0 ? 1u : 0u);
                            else
                                umma_bf16(d, ad, bd, idesc_t, (kb | k) != 0 ? 1u : 0u);
                        }
                        if constexpr (kPair)
                            umma_commit_pair(smem_u32(&ctl->empty[stage]), 0x3);
                        else
                            umma_commit(smem_u32(&ctl->empty[stage]));
                        if (++stage == G::kStages) { stage = 0; phase ^= 1u; }
                    }
                    if (!ok) break;
                    if constexpr (kPair)
                        umma_commit_pair(smem_u32(&ctl->tfull[acc]), 0x3);
                    else
                        umma_commit(smem_u32(&ctl->tfull[acc]));
                }
            }
            // all issued MMAs complete before TMEM is released (in both CTAs of a pair)
            if constexpr (kPair)
                umma_commit_pair(smem_u32(&ctl->drain), 0x3);
            else
                umma_commit(smem_u32(&ctl->drain));
            long long t0 = clock64();
            while (!mbar_try_wait(smem_u32(&ctl->drain), 0) && clock64() - t0 < kWaitCycles) {}
        } else if (kPair && lane == 0) {
            // the peer's accumulators are written by the leader's MMAs
            long long t0 = clock64();
            while (!mbar_try_wait(smem_u32(&ctl->drain), 0) && clock64() - t0 < kWaitCycles) {}
        }
    } else if (warp == kDepWarp) {
        // Dependency warp: walks the CTA's tile list in the producer's order and,
        // for each tile that starts a new matrix (per-matrix counters) or a new
        // level (grid-wide counters), waits (bounded) until the tiles whose
        // results it reads and whose inputs it overwrites have released their
        // counters; then publishes the count of tiles so cleared.  Its gpu-scope
        // acquires are off the producer's path, which reads the count with a
        // CTA-scope acquire.
        if (lane == 0 && p.deps) {
            unsigned long long dep_wait_ns = 0, dep_spins = 0;
            int seq = 0;
            bool ok = true;
            for (int lv = p.lv_begin; lv < p.lv_end && ok; ++lv) {
                const int ph = lv % 3, step = lv / 3;
                const int2 range = unit_tiles(p, ph, unit);
                int dep_key = -1;
                for (int t = 0; t < range.y; ++t) {
                    const TileDesc td = p.tc_tiles[ph][range.x + t];
                    const int key = p.deps == 2 ? 0 : td.mat;
                    if (key != dep_key) {
                        if (!wait_producer_near(ctl, seq, abort_flag, p.err)) { ok = false; break; }
                        // (grid-wide counters serve every matrix: there every wait stalls)
                        const bool stall = p.stall_mat >= 0 && (td.mat == p.stall_mat || p.deps == 2);
                        const int w = wait_deps(p, deps_of(p, p.mats[td.mat]), ph, step, stall, abort_flag,
                                                &dep_wait_ns);
                        if (w == 0) { ok = false; break; }
                        dep_spins += w == 2;
                        dep_key = key;
                    }
                    st_release_cta_smem(&ctl->dep_ready, ++seq);
                }
            }
            if (p.stamps != nullptr) {
                p.stamps[4 * blockIdx.x + 2] = dep_wait_ns;
                p.stamps[4 * blockIdx.x + 3] = dep_spins;
            }
        }
    } else {
        // group g = warp / 8 takes the tiles of accumulator g (every other
        // tile of the CTA's list), so one group's stores drain while the
        // other works through the next tile
        const int quarter = warp & 3, slice = (warp >> 2) & 1, group = warp >> 3;
        const uint32_t tempty_leader[2] = {kPair ? mapa_shared(smem_u32(&ctl->tempty[0]), 0) : 0u,
                                           kPair ? mapa_shared(smem_u32(&ctl->tempty[1]), 0) : 0u};
        bool ok = true;
        int q = 0;
        uint32_t wuse = 0;                        // TMA loads into this warp's staging block (its barrier's parity)
        bool wpend = false;                       // a load may still be landing after a wait gave up
        for (int lv = p.lv_begin; lv < p.lv_end && ok; ++lv) {
            const int ph = lv % 3, step = lv / 3;
            const int2 range = unit_tiles(p, ph, unit);
            const bool prefetch_w = ph == kApply && step + 1 == p.steps && p.apply_update;
            for (int t = 0; t < range.y; ++t, ++q) {
                if ((q & 1) != group) continue;           // the other group's tile
                const TileDesc td = p.tc_tiles[ph][range.x + t];
                const MatDesc& md = p.mats[td.mat];
                const int acc = group;
                const uint32_t acc_phase = (q >> 1) & 1;
                if (prefetch_w && t + 2 < range.y)        // this group's next tile
                    prefetch_update_tile(p, range.x + t + 2, G::kTileRows,
                                         static_cast<int>(rank) * kTcBM + quarter * 32 + lane, slice * kEpiSliceCols,
                                         lane);
                ok = mbar_wait_bounded(smem_u32(&ctl->tfull[acc]), acc_phase, abort_flag, p.err, 0x104);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }          // warp-uniform exit
                tc_fence_after();
                if (p.deps && ph != kGram) {
                    // the Gram entries (poly), or the operand and B's diagonal
                    // residual (apply), read below were released by other CTAs and
                    // acquired by the dependency warp before this tile was loaded
                    if (lane == 0) (void)ld_acquire_cta_smem(&ctl->dep_ready);
                    __syncwarp();
                }
                const int i = td.ti * G::kTileRows + static_cast<int>(rank) * kTcBM + quarter * 32 + lane;
                const bool row_ok = i < md.m;
#pragma unroll 1
                for (int ch = 0; ch < kEpiSliceCols / 32; ++ch) {
                    const int col = slice * kEpiSliceCols + ch * 32;
                    const int j0 = td.tj * kTcBN + col;
                    uint32_t r[32];
                    __syncwarp();
                    tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                           static_cast<uint32_t>(acc * kTcBN + col),
                                       r);
                    tmem_wait_ld();
                    float v[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
                    if (ph == kApply) {
                        if (!epi_apply(p, md, step, i, row_ok, j0, v,
                                       smem_u32(smem + G::kStages * G::kStageBytes + 1024 + warp * kEpiStageBytes),
                                       smem_u32(&ctl->wbar[warp]), wuse, wpend, abort_flag)) {
                            ok = false;
                            break;
                        }
                    } else if (!epi_symmetric(p, md, ph, step, i - lane, j0, v,
                                              smem_u32(smem + G::kStages * G::kStageBytes + 1024 + warp * kEpiStageBytes),
                                              smem_u32(&ctl->wbar[warp]), wuse, wpend, abort_flag)) {
                        ok = false;
                        break;
                    }
                }
                // the accumulator is in registers by now: hand it back to the
                // MMA warp before waiting for this tile's stores to drain
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (leader)
                        mbar_arrive(smem_u32(&ctl->tempty[acc]));
                    else
                        mbar_arrive_cluster(tempty_leader[acc]);
                }
                if (p.deps) {
                    if (lane == 0 && ph != kApply) bulk_wait_all();   // the tile's TMA stores have landed
                    fence_proxy_async_global();   // the stores above feed later TMA loads
                    __syncwarp();
                    if (lane == 0) red_release_gpu_add(deps_of(p, md).cnt + ph, 1);
                }
            }
        }
        if (lane == 0) {
            bulk_wait_all();                      // no store still reads this CTA's shared memory
            if (wpend) {                          // nor does a load land in it after the CTA left
                const long long t0 = clock64();
                while (!mbar_try_wait(smem_u32(&ctl->wbar[warp]), wuse & 1u) && clock64() - t0 < kWaitCycles) {}
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (p.stamps != nullptr && threadIdx.x == 0) p.stamps[4 * blockIdx.x + 1] = globaltimer_ns();
    if constexpr (kPair) cluster_sync();          // neither CTA leaves while the other may signal it
    if (warp == kMmaWarp) {
        tc_fence_after();
        if constexpr (kPair)
            tmem_dealloc_pair(tmem, kTmemCols);
        else
            tmem_dealloc(tmem, kTmemCols);
    }
}

int tc_smem_bytes(bool pair) { return pair ? Geo<true>::kSmemBytes : Geo<false>::kSmemBytes; }

namespace {
// Sets the kernels' shared-memory limit once per device ordinal.
cudaError_t prepare_kernels() {
    static std::atomic<uint64_t> attr_set{0};   // one bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = uint64_t(1) << (dev & 63);
    if (!(attr_set.load() & bit)) {
        e = cudaFuncSetAttribute(ns_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Geo<false>::kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(ns_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Geo<true>::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(bit);
    }
    return cudaSuccess;
}

cudaLaunchConfig_t launch_config(bool pair, int grid, cudaStream_t s, cudaLaunchAttribute* attr, bool cooperative) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = tc_smem_bytes(pair);
    cfg.stream = s;
    int n = 0;
    if (pair) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cfg;
}
}  // namespace

int tc_max_coresident_ctas(bool pair) {
    if (prepare_kernels() != cudaSuccess) return 0;
    if (!pair) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ns_tc_kernel<false>, kThreads,
                                                          Geo<false>::kSmemBytes) != cudaSuccess)
            return 0;
        return per_sm * device_sm_count();
    }
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config(true, 2 * device_sm_count(), nullptr, attr, false);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, ns_tc_kernel<true>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return 2 * clusters;
}

// A launch with dependency waits is cooperative: the runtime then guarantees
// that every CTA is resident at once (or refuses the launch), which the
// cross-CTA waits rely on to make progress.  A pair launch is a cluster
// launch of 2-CTA clusters (grid even).
cudaError_t launch_ns_tc(const NsLaunch& p, int grid, bool cooperative, bool pair, cudaStream_t s) {
    if (grid <= 0) return cudaSuccess;
    if (pair && (grid & 1)) return cudaErrorInvalidConfiguration;
    cudaError_t e = prepare_kernels();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    const cudaLaunchConfig_t cfg = launch_config(pair, grid, s, attr, cooperative);
    return pair ? cudaLaunchKernelEx(&cfg, ns_tc_kernel<true>, p) : cudaLaunchKernelEx(&cfg, ns_tc_kernel<false>, p);
}

}  // namespace mo
