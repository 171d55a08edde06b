/*
 * matrixopt.h -- C ABI of a GB300 (sm_103a) library for the optimizer step one
 * owner GPU executes for full 2D weight matrices: Muon (momentum, quintic
 * Newton-Schulz orthogonalisation, scaled update), the Sign-Muon sign / 1-bit
 * pack / majority-vote update, AdamW on the 1D tail, and the owner planner.
 *
 * Sources of the operations (web pages on matrix optimizers):
 *   "Riassunto Tecnico: MatrixFSDP" (gist.science/it/paper/2607.05895)
 *     §Metodologia 1 -- every 2D matrix has one owner rank holding it whole;
 *       Newton-Schulz runs there with no matrix communication; 1D tensors go
 *       to a separate "tail" owner that keeps AdamW.
 *     §Metodologia 2 "Metadati MatrixShard & Global Planner" -- a planner
 *       assigns owners balancing resident bytes and optimizer work.
 *   "Riepilogo Tecnico: SignMuon" (gist.science/it/paper/2605.16311)
 *     §2 "Meccanismo Principale" / "Flusso Algoritmico" -- per-worker momentum
 *       and NS polar direction U, S = sign(U), 1-bit packing for the
 *       all-gather variant, majority vote sign(sum S), W <- W - eta * vote.
 *
 * Conventions (every call):
 *   - Returns MO_OK (0) or a negative MO_ERR_* code; nothing aborts and no
 *     exception crosses the boundary.  mo_status_string() names a code.
 *   - Device buffers and the stream belong to the caller.  The library never
 *     allocates device memory: calls that need scratch take a caller-provided
 *     workspace whose size the matching *_workspace_bytes() call reports.
 *   - Device calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  plan_owners and the *_workspace_bytes calls
 *     are host-only.
 *   - Matrices are row-major with a leading dimension `ld` in ELEMENTS
 *     (ld >= cols).  Device base pointers must be 16-byte aligned and
 *     ld * element_size must be a multiple of 16 bytes, else MO_ERR_ALIGNMENT.
 *   - A matrix with rows == 0 or cols == 0 is skipped; n == 0 is a no-op.
 *   - Calls with distinct workspaces may run concurrently from any threads;
 *     two in-flight calls must not share a workspace.
 */
#ifndef MATRIXOPT_H
#define MATRIXOPT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mo_stream_t;      /* same type as cudaStream_t */

/* status codes */
#define MO_OK               0
#define MO_ERR_INVALID_ARG (-1)   /* null pointer, negative size, ld < cols, M <= 0, ... */
#define MO_ERR_ALIGNMENT   (-2)   /* base not 16-byte aligned or ld*elem % 16 != 0 */
#define MO_ERR_WORKSPACE   (-3)   /* workspace null, misaligned (256 B) or too small */
#define MO_ERR_CUDA        (-4)   /* a CUDA runtime/driver call failed */
#define MO_ERR_TIMEOUT     (-5)   /* a device-side bounded wait gave up (see mo_check_device_status) */
#define MO_ERR_UNSUPPORTED (-6)   /* valid request outside what this build implements */

/* element types */
#define MO_F32  0
#define MO_BF16 1

/* Newton-Schulz arithmetic */
#define MO_NS_BF16 0   /* bf16 tensor-core operands (tcgen05), fp32 accumulate and epilogue */
#define MO_NS_FP32 1   /* fp32 throughout (CUDA cores), for reference-grade accuracy */

/* One 2D parameter owned by this GPU.  W, M and G share rows, cols and ld.
 * W: weights (updated in place), M: momentum state (updated in place),
 * G: gradient (read only).  dtypes are MO_F32 or MO_BF16 each. */
typedef struct {
    int64_t rows, cols, ld;
    int32_t w_dtype, m_dtype, g_dtype, reserved;
    void*       W;
    void*       M;
    const void* G;
} mo_matrix;

/* Muon hyper-parameters.  The step is
 *   M <- mu*M + G                          (heavy-ball momentum)
 *   X <- orient(M): M^T when rows > cols   (so m <= n)
 *   X <- X / ||X||_F  (0 stays 0); with spectral_iters = q > 0 instead
 *        X <- X / (||X||_F * sigma_hat), sigma_hat^2 = v^T A v after q power
 *        iterations v <- A v / ||A v|| from v = ones/sqrt(m) on the Gram
 *        matrix A of X/||X||_F (the spectral scale; SignMuon §4 compares it
 *        with the Frobenius scale).  bf16 NS and ns_steps >= 1 only.
 *   repeat ns_steps: A = X X^T; B = b*A + c*A*A; X <- a*X + B*X
 *   O <- orient back(X)
 *   apply_update != 0:  W <- W - lr*weight_decay*W - lr*update_scale*O
 *   apply_update == 0:  out[i] <- O (dtype out_dtype, layout of matrix i)  */
typedef struct {
    float   mu, lr, update_scale, weight_decay;
    int32_t ns_steps;              /* k >= 0 */
    float   a, b, c;               /* quintic coefficients */
    int32_t ns_precision;          /* MO_NS_BF16 or MO_NS_FP32 */
    int32_t apply_update;
    int32_t out_dtype;             /* MO_F32 / MO_BF16, used when apply_update == 0 */
    int32_t spectral_iters;        /* 0: Frobenius scale; q in 1..64: spectral scale */
} mo_muon_cfg;

/* The flat float32 tail updated by decoupled AdamW at step number `step`
 * (>= 1, the caller counts):
 *   m <- beta1*m + (1-beta1)*g ; v <- beta2*v + (1-beta2)*g^2
 *   W <- W - lr*weight_decay*W - lr*(m/(1-beta1^t)) / (sqrt(v/(1-beta2^t)) + eps) */
typedef struct {
    int64_t      numel;
    float*       W;
    const float* g;
    float*       m;
    float*       v;
    float        lr, beta1, beta2, eps, weight_decay;
    int32_t      reserved;
    int64_t      step;
} mo_adamw_tail;

/* Workspace size (bytes) muon_step_batched needs for these matrices and cfg.
 * Host only.  MO_ERR_INVALID_ARG for bad shapes / cfg. */
int mo_workspace_bytes(const mo_matrix* mats, int n, const mo_muon_cfg* cfg,
                       size_t* bytes_out);

/* One Muon step over n matrices owned by this GPU, plus optionally the AdamW
 * tail (tail may be NULL).  out may be NULL when cfg->apply_update != 0; else
 * it is a host array of n device pointers, output i laid out like matrix i
 * (rows x cols, leading dimension ld).  ws must be 256-byte aligned and at
 * least mo_workspace_bytes() long.  Runs the fused momentum + norm kernel,
 * then the Newton-Schulz phases grouped over all n matrices, the update fused
 * into the last phase, then the tail.  Asynchronous on `stream`. */
int muon_step_batched(const mo_matrix* mats, int n, const mo_muon_cfg* cfg,
                      const mo_adamw_tail* tail, void* const* out,
                      void* ws, size_t ws_bytes, mo_stream_t stream);

/* A Sign-Muon worker's step with the sign extraction and 1-bit packing
 * fused into the last Newton-Schulz epilogue (SignMuon §2 "Flusso
 * Algoritmico" steps 1-3): momentum and NS as muon_step_batched, no weight
 * update, and instead of the direction U the packed words of sign(U) are
 * written to words[i] (host array of n device pointers, ceil(rows*cols/32)
 * uint32 each, sign_pack's layout and tie rule).  The sign is taken of U as
 * stored in cfg->out_dtype, so the words equal sign_pack of the output
 * muon_step_batched would write.  bf16 NS only, ns_steps >= 1, and every
 * matrix's cols a multiple of 32 (else MO_ERR_UNSUPPORTED); ws sized by
 * mo_workspace_bytes. */
int muon_step_sign_packed(const mo_matrix* mats, int n, const mo_muon_cfg* cfg,
                          uint32_t* const* words, void* ws, size_t ws_bytes, mo_stream_t stream);

/* The whole Sign-Muon step of one GPU that holds the M workers (SignMuon §2
 * "Flusso Algoritmico" steps 1-4, "Meccanismo Principale" 3): each worker's
 * momentum, NS and fused sign + 1-bit pack as muon_step_sign_packed (mats[i]
 * is worker i, words[i] receives its packed signs), then the majority vote
 * over the M = n packed buffers and W <- W - lr*vote as sign_vote_update.
 * Every worker has the same rows x cols (cols a multiple of 32); W is
 * rows x cols with leading dimension ld (>= cols), MO_F32 or MO_BF16, element
 * alignment; 1 <= M <= 128 non-empty workers (else MO_ERR_INVALID_ARG or
 * MO_ERR_UNSUPPORTED).  Two launches on `stream`: the NS with the fused pack,
 * then the vote.  W and the words equal those of muon_step_sign_packed +
 * sign_vote_update.  ws sized by mo_workspace_bytes. */
int muon_step_sign_vote(const mo_matrix* mats, int n, const mo_muon_cfg* cfg, uint32_t* const* words,
                        void* W, int w_dtype, int64_t ld, float lr, void* ws, size_t ws_bytes,
                        mo_stream_t stream);

/* Workspace size for ns_orthogonalize on these shapes (host only). */
int ns_workspace_bytes(const int64_t* rows, const int64_t* cols, int n,
                       int precision, size_t* bytes_out);

/* Pure Newton-Schulz on n matrices: out[i] = orient back(NS_k(X_i/||X_i||_F)).
 * X, out: host arrays of n device pointers (X[i] of dtype in_dtype, out[i] of
 * out_dtype), both rows[i] x cols[i] with leading dimension ld[i].
 * steps >= 0; precision MO_NS_BF16 or MO_NS_FP32.  X is not modified;
 * out may not alias X. */
int ns_orthogonalize(const void* const* X, void* const* out,
                     const int64_t* rows, const int64_t* cols, const int64_t* ld,
                     int n, int in_dtype, int out_dtype, int steps,
                     float a, float b, float c, int precision,
                     void* ws, size_t ws_bytes, mo_stream_t stream);

/* ns_orthogonalize for ONE matrix (bf16 tensor-core mode) that allocates
 * nothing and takes no workspace.  The pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory, such as a
 * plugin handed only its input and output buffers by a host framework that
 * owns and accounts for every byte of device memory, or a latency-critical
 * loop where a cudaMalloc would synchronise the device.
 *   - Scratch: a fixed array of MO_NOALLOC_SCRATCH_BYTES (32 MiB) compiled
 *     into the library in device global memory; every GPU that loads the
 *     library holds it until the process exits.
 *   - Size limit: ns_workspace_bytes() for this shape must not exceed
 *     MO_NOALLOC_SCRATCH_BYTES, else MO_ERR_UNSUPPORTED (for example
 *     768 x 3072 and 1024 x 2048 fit, 2048 x 2048 does not).
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.
 *   - Every call shares the one array per device and it keeps the last
 *     call's contents; calls whose work overlaps on the GPU (other streams,
 *     other threads) race and corrupt each other's results.
 *   - No cudaMalloc, cudaFree or other allocating routine is called.
 *   - A run whose bounded device waits expire (about 2 s) leaves `out`
 *     unspecified and still returns MO_OK (the wait happens on the GPU after
 *     the call returned); ns_orthogonalize_noalloc_status reports it.
 *   - The call's small control block is copied from ordinary (pageable)
 *     host memory with cudaMemcpyAsync, so the call may return only once
 *     that copy has been staged: it is not fully asynchronous to the host.
 *   - The looked-up device address is kept for the life of the process;
 *     calls after a cudaDeviceReset on that device are not supported.
 * Arguments as ns_orthogonalize with n = 1 (X, out device pointers). */
#define MO_NOALLOC_SCRATCH_BYTES (32u << 20)
int ns_orthogonalize_noalloc(const void* X, void* out, int64_t rows, int64_t cols, int64_t ld,
                             int in_dtype, int out_dtype, int steps, float a, float b, float c,
                             mo_stream_t stream);

/* Status of the allocation-free runs on the current device: waits for
 * `stream`, then returns MO_ERR_TIMEOUT if a run's bounded device wait gave
 * up since the last check (and clears that record), else MO_OK; MO_ERR_CUDA
 * if the device cannot be queried.  As mo_check_device_status, applied to the
 * fixed scratch; it allocates nothing. */
int ns_orthogonalize_noalloc_status(mo_stream_t stream);

/* Sign extraction and 1-bit packing (SignMuon §2 step 2 and the all-gather
 * variant of step 3).  Element j of the row-major flattening of U (rows x
 * cols, leading dimension ld, dtype MO_F32/MO_BF16) goes to bit (j % 32) of
 * words[j / 32]; the bit is 1 unless U_j < 0 (so +0, -0 and NaN give 1, the
 * sign(0) = +1 rule).  words has ceil(rows*cols/32) uint32 entries; unused
 * bits of the last word are written 0.  No workspace.  Only element alignment
 * is required of U (4 or 2 bytes) and of words (4 bytes), and any ld >= cols. */
int sign_pack(const void* U, int dtype, int64_t rows, int64_t cols, int64_t ld,
              uint32_t* words, mo_stream_t stream);

/* sign_pack for M same-shaped matrices in one launch (the M workers of a
 * Sign-Muon step): U and words are host arrays of M device pointers, each
 * pair laid out as for sign_pack.  1 <= M <= 128. */
int sign_pack_batched(const void* const* U, int M, int dtype, int64_t rows, int64_t cols,
                      int64_t ld, uint32_t* const* words, mo_stream_t stream);

/* Majority vote over M packed sign buffers and the voted update (SignMuon §2
 * "Meccanismo Principale" item 3 and step 4).  words: host array of M device
 * pointers, each ceil(rows*cols/32) words in sign_pack's layout.  For each
 * element, with c of the M workers voting +1, vote = +1 if 2c >= M (ties go
 * to +1) else -1, and W <- W - lr*vote in float32 (one rounding; a bf16 W is
 * rounded to bf16 once).  1 <= M <= 128 (MO_ERR_INVALID_ARG for M <= 0,
 * MO_ERR_UNSUPPORTED above 128).  W needs element alignment only, any
 * ld >= cols; word buffers need 4-byte alignment. */
int sign_vote_update(const uint32_t* const* words, int M, int64_t rows, int64_t cols,
                     void* W, int w_dtype, int64_t ld, float lr, mo_stream_t stream);

/* The optional local polar step on the vote (SignMuon §2 "Flusso
 * Algoritmico" step 5): the voted sign matrix S_bar (+1/-1, majority of the M
 * packed buffers, ties +1) is orthogonalised locally with the quintic
 * Newton-Schulz iteration (bf16 tensor cores, k = steps, X0 = S_bar/||S_bar||_F)
 * and W <- W - lr * NS(S_bar).  W follows the 16-byte rules of
 * muon_step_batched; ws (256-byte aligned) holds S_bar and the NS buffers,
 * sized by sign_vote_polar_workspace_bytes (host only).  1 <= M <= 128. */
int sign_vote_polar_workspace_bytes(int64_t rows, int64_t cols, int64_t ld, size_t* bytes_out);
int sign_vote_polar_update(const uint32_t* const* words, int M, int64_t rows, int64_t cols,
                           void* W, int w_dtype, int64_t ld, float lr, int steps,
                           float a, float b, float c, void* ws, size_t ws_bytes, mo_stream_t stream);

/* The int8 all-reduce variant of the vote (SignMuon §2 step 3 "Variante
 * All-Reduce": an integer-sum all-reduce of the signs, then the local
 * threshold; 8 bits per element, §2 "Efficienza di Comunicazione").
 * sign_int8 writes out[j] = -1 if U_j < 0 else +1 (int8) over the row-major
 * flattening of U (dense, rows*cols bytes; U element-aligned, any ld >= cols).
 * sign_vote_update_int8 takes a host array of M device pointers to such
 * buffers (the pre-reduction payloads of M workers), forms each element's
 * integer sum and applies W <- W - lr*vote with vote = +1 iff sum >= 0 (ties
 * +1), one fp32 rounding, as sign_vote_update.  1 <= M <= 127 (the int8 sum
 * range): MO_ERR_INVALID_ARG for M <= 0, MO_ERR_UNSUPPORTED above. */
int sign_int8(const void* U, int dtype, int64_t rows, int64_t cols, int64_t ld,
              int8_t* out, mo_stream_t stream);
int sign_vote_update_int8(const int8_t* const* signs, int M, int64_t rows, int64_t cols,
                          void* W, int w_dtype, int64_t ld, float lr, mo_stream_t stream);

/* Owner planner (MatrixFSDP §Metodologia 2), host only.  For matrix i,
 *   bytes_i = rows_i*cols_i*2, flops_i = ns_steps*(4 m^2 n + 2 m^3) (m<=n),
 *   cost_i  = w_bytes*bytes_i/sum(bytes) + w_flops*flops_i/sum(flops);
 * matrices in decreasing cost (ties: lower index first) each go to the rank
 * with the least accumulated cost (ties: lower rank).  Sums run in index
 * order in double, so the plan is reproducible bit for bit.
 * owner_out[n] receives ranks; load_out[world] (nullable) the per-rank cost.
 * world <= 0 or a negative size gives MO_ERR_INVALID_ARG. */
int plan_owners(const int64_t* rows, const int64_t* cols, int n, int world, int ns_steps,
                double w_bytes, double w_flops, int32_t* owner_out, double* load_out);

/* Synchronises `stream`, reads the device error word in workspace `ws`
 * (written by bounded waits inside the kernels), clears it, and returns
 * MO_OK, MO_ERR_TIMEOUT or MO_ERR_CUDA. */
int mo_check_device_status(void* ws, mo_stream_t stream);

/* Static string naming a status code. */
const char* mo_status_string(int status);

/* Library version, e.g. 0x000100 for 0.1.0. */
int mo_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MATRIXOPT_H */
