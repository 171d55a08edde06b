// Structures shared by the host orchestration and the kernels.  Plain
// old data only: they are staged on the host and copied into the workspace.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/matrixopt.h"

namespace mo {

// Tile geometry of the tensor-core Newton-Schulz GEMM.
constexpr int kTcBM = 128;   // rows of D per tile (TMEM lanes)
constexpr int kTcBN = 256;   // columns of D per tile (TMEM columns per accumulator)
constexpr int kTcBK = 64;    // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int kTcEpiWarps = 16;   // epilogue warps per CTA of the tensor-core kernel
constexpr int kTcEpiGroupWarps = 8;   // of which one group finishes a tile (the groups alternate tiles)
// Tile geometry of the CUDA-core fp32 GEMM.
constexpr int kFpBM = 64, kFpBN = 64, kFpBK = 16;
// Momentum / normalisation kernel tile.
constexpr int kMomTile = 64;
// SM cycles a fused launch's dependency wait spins before it gives up (about
// 2 s at 2 GHz, as the kernels' other bounded waits).
constexpr long long kDepWaitCycles = 4000000000LL;
// The most workers a vote counts over (8-bit bit-sliced counts).
constexpr int kMaxVoteWorkers = 128;

enum NsPhase : int32_t { kGram = 0, kPoly = 1, kApply = 2 };

// tcgen05 instruction descriptor of kind::f16: bf16 x bf16 -> f32, A K-major,
// B K-major (b_mn = 0) or MN-major (b_mn = 1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t b_mn) {
    return (1u << 4)            // D format f32
           | (1u << 7)          // A format bf16
           | (1u << 10)         // B format bf16
           | (b_mn << 16)       // B major
           | ((N >> 3) << 17)   // N / 8
           | ((M >> 4) << 24);  // M / 16
}

// One matrix of the Newton-Schulz path, in the oriented frame: the NS
// iterate X is m x n with m <= n; element (i, j) of X is element (i, j) of
// the user matrix, or (j, i) when `transposed`.
struct MatDesc {
    int32_t m, n;              // oriented sizes
    int32_t ldx, lda;          // workspace leading dims (elements) of X and of m x m buffers
    int64_t ld;                // user leading dim (elements) of src / W / out / M / G
    int32_t rows, cols;        // user sizes
    int32_t transposed;
    int32_t src_dtype;         // momentum / input dtype
    int32_t g_dtype;           // gradient dtype (momentum kernel)
    int32_t w_dtype;
    int32_t out_dtype;
    int32_t has_momentum;      // 1: src = M updated from G; 0: src = input X read only
    void* src;                 // M (muon) or X (pure NS), user layout
    const void* grad;          // G (muon) or null
    void* W;                   // update target or null
    void* out;                 // NS output target or null
    uint32_t* sign_words;      // fused sign + 1-bit pack target of the output, or null
    void* x_op[2];             // NS operand ping-pong: fp32 m x ldx row-major (fp32 mode), or bf16 in
                               // 8-column blocks: element (i, j) at ((j / 8) * xrows + i) * 8 + j % 8
    int32_t xrows;             // rows of one 8-column block of the bf16 operand (m rounded up to 8)
    void* gram;                // m x lda  (A = X X^T)
    void* poly;                // m x lda  (B = b A + c A^2)
    // bf16 operand views (3D: 64 elements = 8 rows x 8 columns of a block, row groups, column blocks)
    const CUtensorMap* tm_xa[2];   // box 128 rows x 64 columns: A operand of the Gram phase
    const CUtensorMap* tm_xb[2];   // box (256 or 128) rows x 64 columns: B operand of the Gram phase
    const CUtensorMap* tm_xn[2];   // box 64 rows x (256 or 128) columns: B operand of the apply phase
    const CUtensorMap* tm_gram;    // box 64 columns x 128 rows (A operand of the polynomial phase)
    const CUtensorMap* tm_gram_b;  // box 64 columns x (256 or 128) rows (its B operand)
    const CUtensorMap* tm_poly;    // box 64 columns x 128 rows (A operand of the apply phase)
    const CUtensorMap* tm_gram_st; // box 32 x 32, 64-byte swizzle: the Gram epilogue's stores of A
    const CUtensorMap* tm_poly_st; // box 32 x 32, 64-byte swizzle: the polynomial epilogue's stores of B
    const CUtensorMap* tm_w;       // user W, 64-byte rows x 32 rows, 64-byte swizzle: the last step's
                                   // update (null: W unaligned for TMA, updated by plain accesses)
    float* scales;             // [0] = 1/||X||_F, [1] = 1/||X||_F^2 (0 for a zero matrix),
                               // [2..4] = 1/lambda, 1/lambda^2, 1/sqrt(lambda) of the spectral
                               // estimate (1 under Frobenius scaling); kScaleStride floats
    float* pv;                 // power-iteration vectors (m floats each)
    float* py;
    float* dlo;                // m floats: B_ii - bf16(B_ii), the rounding residual of the polynomial
                               // matrix's diagonal, added back by the apply epilogue
    int64_t row_begin;         // first global row of this matrix (power iteration)
    int64_t mom_tile_begin;    // first global index of this matrix's momentum tiles
    int32_t mom_tiles_r, mom_tiles_c;
    int32_t nt_sym, nt_apply;  // tensor-core tiles of one Gram / polynomial phase, of one apply phase
    int* deps;                 // [3] epilogue-warp tile completions per phase within one fused launch
};
constexpr int kScaleStride = 8;

// One tile of a grouped GEMM phase.
struct TileDesc {
    int32_t mat;       // matrix index
    int32_t ti, tj;    // tile row / column index
    int32_t nkb;       // K blocks
};

struct NsLaunch {
    const MatDesc* mats;
    const TileDesc* tiles;     // CUDA-core path: one tile per block of phase `phase`
    int* err;
    int32_t phase, step, steps;
    int32_t apply_update;
    float a, b, c;
    float alpha;               // lr * update_scale
    float decay;               // lr * weight_decay
    int32_t ntiles;
    // tensor-core path: the launch runs levels [lv_begin, lv_end), level = 3 * step + phase,
    // each CTA walking its scheduled tiles of every level in order
    const TileDesc* tc_tiles[3];
    const int2* tc_ranges[3];  // per CTA {first tile, tile count} of each phase
    int32_t tc_ctas[3];        // CTAs that hold tiles of each phase
    int32_t lv_begin, lv_end;
    int32_t deps;              // 0: none (one level); 1: per-matrix counters; 2: one grid-wide
                               // counter set (every tile of a level waits for the whole previous level)
    int* level_deps;           // [3] the grid-wide counters of mode 2
    int32_t tot_sym, tot_apply;  // tiles of one symmetric / apply level over all matrices
    int32_t rel_per_tile;      // counter releases per finished tile (one group of 8 epilogue warps per CTA)
    uint32_t idesc_sym, idesc_apply;
    uint32_t mn_lbo, mn_sbo;   // descriptor strides of the MN-major operand
    unsigned long long* stamps;  // null, or [4 * gridDim.x]: per CTA start / end %globaltimer (ns),
                                 // ns spent waiting on dependencies, number of waits that spun
    long long dep_wait_cycles;   // SM cycles a dependency wait spins before it gives up
    int32_t stall_mat;           // -1; else the dependency waits of this matrix's tiles can never be met
                                 // (failure-path test: the wait runs out and reports MO_ERR_TIMEOUT)
};

struct MomLaunch {
    const MatDesc* mats;
    int32_t nmats;
    int64_t ntiles;
    float mu;
    int32_t fp32_operand;      // write the fp32 operand (fp32 NS) instead of bf16
    float* partials;           // one fp32 sum of squares per momentum tile
};

// ------------------------------------------------------------------ launchers
cudaError_t launch_momentum_norm(const MomLaunch& p, int grid, cudaStream_t s);
// bf16 momentum, fp32 gradient, rows <= cols, ld % 8 == 0, 16-byte aligned M and G (6 blocks per SM)
cudaError_t launch_momentum_norm_bf16m(const MomLaunch& p, int grid, cudaStream_t s);
cudaError_t launch_norm_finalize(const MatDesc* mats, int nmats, const float* partials,
                                 cudaStream_t s);
cudaError_t launch_ns_k0(const MomLaunch& p, float alpha, float decay, int apply_update, int grid,
                         cudaStream_t s);
// pair: the 2-CTA (cta_group::2) form, grid = 2 x CTA pairs
cudaError_t launch_ns_tc(const NsLaunch& p, int grid, bool cooperative, bool pair, cudaStream_t s);
int tc_max_coresident_ctas(bool pair);   // CTAs of that form that fit on the device at once
cudaError_t launch_ns_fp32_phase(const NsLaunch& p, int grid, cudaStream_t s);
cudaError_t launch_sign_pack(const void* U, int dtype, int64_t rows, int64_t cols, int64_t ld,
                             uint32_t* words, cudaStream_t s);
cudaError_t launch_sign_vote_update(const uint32_t* const* words, int M, int64_t rows,
                                    int64_t cols, void* W, int w_dtype, int64_t ld, float lr,
                                    cudaStream_t s);
cudaError_t launch_adamw(const mo_adamw_tail& t, cudaStream_t s);
cudaError_t launch_sign_pack_batched(const void* const* U, uint32_t* const* words, int M, int dtype, int64_t rows,
                                     int64_t cols, int64_t ld, cudaStream_t s);
cudaError_t launch_spectral_estimate(const MatDesc* mats, int nmats, int64_t total_rows, int iters, int sm_count,
                                     cudaStream_t s);
cudaError_t launch_vote_matrix(const uint32_t* const* words, int M, int64_t rows, int64_t cols, void* S, int64_t ld,
                               cudaStream_t s);
cudaError_t launch_sign_int8(const void* U, int dtype, int64_t rows, int64_t cols, int64_t ld, int8_t* out,
                             cudaStream_t s);
cudaError_t launch_vote_int8(const int8_t* const* signs, int M, int64_t rows, int64_t cols, void* W, int w_dtype,
                             int64_t ld, float lr, cudaStream_t s);

int tc_smem_bytes(bool pair);
int device_sm_count();

}  // namespace mo
