/*
 * matrixopt_debug.h -- introspection entry points for tests.  They expose
 * where the Newton-Schulz intermediates live inside a workspace so that a
 * test can check each phase (the Gram matrix X X^T, the polynomial
 * b*A + c*A^2, the applied X) separately.  The pages have no counterpart;
 * these calls compute nothing.
 */
#ifndef MATRIXOPT_DEBUG_H
#define MATRIXOPT_DEBUG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Placement of matrix `index`'s Newton-Schulz buffers in the workspace that
 * ns_orthogonalize / muon_step_batched use for these shapes (offsets are in
 * bytes from the workspace base).  Orientation: m = min(rows, cols),
 * n = max(rows, cols), transposed = rows > cols.
 *   bf16 mode: x_op[0], x_op[1] = bf16 m x n operand ping-pong in 8-column
 *              blocks: element (i, j) at byte ((j/8)*ldx + i)*16 + (j%8)*2,
 *              where ldx = m rounded up to 8 (X is kept in bf16 between
 *              steps); gram = bf16 m x m row-major (lda), poly = bf16 m x m
 *              (lda); diag_res = m fp32 values, B_ii - bf16(B_ii) of the
 *              polynomial matrix's diagonal, which the apply phase adds back
 *              as a row scale of X.
 *   fp32 mode: x_op[0], x_op[1] = fp32 m x n ping-pong, gram, poly = fp32
 *              m x m; diag_res = 0 (unused).
 * After a call with steps = 1 the gram buffer holds X0 X0^T, the poly buffer
 * aI + b*A + c*A*A of that step (bf16) and diag_res its diagonal's residual.
 * deps: three int32 completion counters (Gram, polynomial, apply) of a fused
 * bf16 launch with per-matrix ordering; after such a call each holds
 * releases_per_tile x (that phase's tiles of this matrix: tiles_sym for Gram
 * and polynomial, tiles_apply for apply) x (the steps of that phase the fused
 * launch ran); all three stay 0 after a call with one launch per phase.  The
 * tile counts and releases_per_tile are those of the tile geometry the
 * library uses on the current device (128 x 256 tiles per CTA, 8 releases;
 * or 256 x 256 tiles per CTA pair, 16 releases). */
typedef struct {
    int64_t m, n, ldx, lda;
    int32_t transposed, precision;
    int64_t x_op[2], diag_res, gram, poly;
    int64_t deps;
    int32_t tiles_sym, tiles_apply;
    int32_t releases_per_tile, reserved;
} mo_ns_view;

int mo_debug_ns_view(const int64_t* rows, const int64_t* cols, int n, int precision,
                     int index, mo_ns_view* view);

/* Number of SMs the grouped kernels size their grids for on the current
 * device (0 if no device). */
int mo_debug_sm_count(void);

/* Chooses the tile geometry of the bf16 tensor-core Newton-Schulz kernel:
 * on = 1 runs 256 x 256 tiles on CTA pairs (clusters of 2, tcgen05
 * cta_group::2: each CTA loads 128 rows of A and 128 columns of B) when the
 * device can co-schedule such clusters; on = 0 (the default) runs 128 x 256
 * tiles on single CTAs.  The two geometries walk K in different orders on
 * some tiles, so they agree to fp32 accumulation noise, not bit for bit.
 * Returns the previous setting, or
 * MO_ERR_INVALID_ARG for a value other than 0 / 1.  Process-wide. */
int mo_debug_set_ns_pair(int on);

/* Chooses how the bf16 tensor-core Newton-Schulz iterations are launched:
 *   1: every (step, phase) of a call in one cooperative persistent launch,
 *      each tile waiting on per-matrix completion counters for the tiles
 *      whose results it reads or whose inputs it overwrites;
 *   2: the same launch with one grid-wide counter set, so each phase waits
 *      for the whole previous phase of every matrix;
 *   3 (the default): 1 when a symmetric phase has fewer than 16 tiles per
 *      CTA, else 2;
 *   0: one launch per (step, phase).
 * The fused modes fall back to 0 when the grid cannot be co-resident.  All
 * modes compute identical results.  Returns the previous setting, or
 * MO_ERR_INVALID_ARG for a value outside 0..3.  Process-wide; affects calls
 * issued after it. */
int mo_debug_set_ns_fused(int on);

/* Failure-path test hook.  With matrix >= 0, every fused bf16 Newton-Schulz
 * launch issued after the call makes the dependency waits of that matrix's
 * tiles (index into the call's non-empty matrices; with grid-wide counters,
 * every dependency wait of the launch) impossible to meet, and
 * those launches' dependency waits give up after wait_cycles SM cycles
 * (1000 .. 4e9; e.g. 2e6, about 1 ms) instead of about 2 s.  The wait then
 * runs out, the launch unwinds (armed copies drained, issued MMAs drained,
 * TMEM freed) and records MO_ERR_TIMEOUT for mo_check_device_status; the
 * outputs of that call are unspecified.  matrix = -1 (the default) turns the
 * hook off.  Per-phase launches have no dependency waits and are unaffected.
 * Process-wide.  Returns MO_ERR_INVALID_ARG for matrix < -1 or a budget out
 * of range. */
int mo_debug_inject_dep_stall(int matrix, int64_t wait_cycles);

/* SM load-balance record.  With a device buffer `buf` of
 * 4 * capacity * max_ctas uint64 values, each of the calling thread's next
 * `capacity` tensor-core Newton-Schulz launches (grid <= max_ctas) has CTA c
 * write, at buf[4*(k*max_ctas + c)] onwards (k counting launches from 0):
 * its start and end %globaltimer (ns), the ns its TMA producer spent waiting
 * on fused-launch dependencies, and the number of those waits that had to
 * spin (both 0 for a per-phase launch).  *recorded (nullable) receives the
 * number of launches recorded since the previous call.  buf = NULL stops
 * recording.  Measurement only: no effect on results. */
int mo_debug_cta_stamps(uint64_t* buf, int capacity, int max_ctas, int* recorded);

/* Launch tracing, for measurement.  mo_trace_enable(capacity) makes every
 * later kernel launch of the calling thread (any entry point) record a CUDA
 * event before and after it on the call's stream, for up to `capacity`
 * launches (events are created once and reused; no device memory).
 * capacity 0 disables tracing.  mo_trace_read() synchronises on the last
 * recorded event, writes up to `cap` entries (kind, milliseconds) of the
 * launches recorded since the previous read, sets *count, and starts a new
 * record.  Kinds: */
#define MO_K_MOMENTUM 1   /* fused momentum + norm partials (+ NS operand) */
#define MO_K_FINALIZE 2   /* per-matrix norm finalisation */
#define MO_K_GRAM     3   /* NS A = X X^T   (tensor cores, or CUDA cores in fp32 mode) */
#define MO_K_POLY     4   /* NS B = aI + bA + cA^2 (a on the diagonal) */
#define MO_K_APPLY    5   /* NS X = BX (+ fused update on the last step) */
#define MO_K_NS0      6   /* zero-step normalise/update */
#define MO_K_ADAMW    7
#define MO_K_PACK     8
#define MO_K_VOTE     9
#define MO_K_SPECTRAL 10  /* power-iteration spectral estimate (all of its launches) */
#define MO_K_NS_FUSED 11  /* all NS levels of a call in one launch (Gram, polynomial, apply) */
int mo_trace_enable(int capacity);
int mo_trace_read(int32_t* kinds, float* ms, int cap, int* count);

#ifdef __cplusplus
}
#endif

#endif /* MATRIXOPT_DEBUG_H */
