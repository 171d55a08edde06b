// Host side of the C ABI: argument validation, workspace layout, tensor-map
// encoding, tile scheduling across SMs, launch sequencing, the owner planner.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>
#include <queue>
#include <vector>

#include "../../include/matrixopt.h"
#include "../../include/matrixopt_debug.h"
#include "internal.h"

namespace mo {

namespace {

constexpr int64_t kMaxMinDim = 32768;        // m = min(rows, cols): the m x m buffers
constexpr int64_t kMaxDim = 1 << 20;
constexpr size_t kWsAlign = 256;
constexpr size_t kBufAlign = 1024;
constexpr size_t kHeaderBytes = 256;         // int error word + reserved

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t elem_size(int dt) { return dt == MO_F32 ? 4 : 2; }
inline bool valid_dtype(int dt) { return dt == MO_F32 || dt == MO_BF16; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int map_cuda(cudaError_t e) { return e == cudaSuccess ? MO_OK : MO_ERR_CUDA; }

// ------------------------------------------------------------ device info
int g_sm_count_cache[64];
std::once_flag g_sm_once[64];

}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    std::call_once(g_sm_once[dev], [dev] {
        int c = 0;
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) c = 1;
        g_sm_count_cache[dev] = c;
    });
    return g_sm_count_cache[dev];
}

namespace {

// ------------------------------------------------------- tensor-map encode
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// bf16 rows x cols (leading dim ld elements), box 64 columns x box_rows rows,
// 128-byte swizzle: the box lands as box_rows contiguous 128-byte rows, the
// same layout as box_rows / 64 stacked 64-row boxes, in one copy.
bool encode_bf16_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Store view of an m x m bf16 buffer for the symmetric epilogues: 32 x 32
// boxes (64-byte rows) with the 64-byte swizzle their shared-memory staging uses.
bool encode_bf16_store_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The user's W for the last step's update: boxes of 32 rows x 64 bytes (16
// fp32 or 32 bf16 columns), 64-byte swizzle.  False when W's address or row
// pitch is not 16-byte aligned (TMA's rule); the update then uses plain accesses.
bool encode_w_map(CUtensorMap* map, const void* W, int dtype, int64_t rows, int64_t cols, int64_t ld) {
    const int64_t esz = dtype == MO_F32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(W) & 15) != 0 || (ld * esz) % 16 != 0) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * esz)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(64 / esz), 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dtype == MO_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(W), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Descriptor strides of the apply phase's MN-major B operand (no swizzle:
// 8-row K groups 128 B apart, 8-column MN blocks 1 KB apart), as (lbo, sbo).
constexpr uint32_t kMnLbo = 128, kMnSbo = 1024;
// How the tensor-core iterations are launched: 1 one fused cooperative launch
// (when the grid fits on the device at once) ordered by per-matrix counters;
// 2 the same launch ordered by one grid-wide counter set; 3 (default) 1 when a
// symmetric level holds few tiles per CTA, else 2; 0 one launch per (step, phase).
std::atomic<int> g_ns_fused{3};
// Below this many symmetric-phase tiles per CTA the barrier tail of each level
// is a large share of it, and per-matrix ordering (which lets one matrix's
// next phase fill the tail) wins; above it the grid-wide ordering keeps every
// CTA on the same few matrices, which measured faster through L2 reuse.
constexpr int64_t kPerMatrixDepsMaxSymTilesPerCta = 16;
// 1: the tensor-core kernel runs 256 x 256 tiles on CTA pairs (cta_group::2)
// when the device can co-schedule 2-CTA clusters; 0 (default): 128 x 256
// tiles per CTA.  The two measured within about 1% of each other on every
// workload; the single-CTA form is the default because its fused
// (cooperative) launch can also be captured by the profiler.
std::atomic<int> g_ns_pair{0};
// Failure-path test hook: -1, or the matrix whose fused-launch dependency
// waits can never be met, with the wait budget those launches then use.
std::atomic<int> g_stall_mat{-1};
std::atomic<long long> g_stall_wait_cycles{0};

// Co-resident CTAs of the tensor-core kernel per device ordinal, queried once.
std::mutex g_cap_mu;
int g_cap[64][2];
bool g_cap_known[64][2];
int tc_capacity(bool pair) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lk(g_cap_mu);
    if (!g_cap_known[dev & 63][pair]) {
        g_cap[dev & 63][pair] = tc_max_coresident_ctas(pair);
        g_cap_known[dev & 63][pair] = true;
    }
    return g_cap[dev & 63][pair];
}

// ------------------------------------------------------------- the request
struct Job {
    int64_t rows, cols, ld;
    int src_dtype, g_dtype, w_dtype, out_dtype;
    int has_momentum;
    void* src;
    const void* grad;
    void* W;
    void* out;
    uint32_t* words = nullptr;   // fused sign + pack target (muon_step_sign_packed)
};

struct Shape {
    int64_t m, n, ldx, lda;
    int64_t xrows, xblocks;        // bf16 operand: rows of an 8-column block (m rounded to 8), blocks
    int transposed;
};

Shape oriented(int64_t rows, int64_t cols) {
    Shape s;
    s.transposed = rows > cols;
    s.m = s.transposed ? cols : rows;
    s.n = s.transposed ? rows : cols;
    s.ldx = static_cast<int64_t>(align_up(static_cast<size_t>(s.n), 64));
    s.lda = static_cast<int64_t>(align_up(static_cast<size_t>(s.m), 64));
    s.xrows = static_cast<int64_t>(align_up(static_cast<size_t>(s.m), 8));
    s.xblocks = ceil_div(s.n, 8);
    return s;
}

// The bf16 operand X in 8-column blocks, viewed by TMA as 3D: 64 elements
// (8 rows x 8 columns of one block, 128 contiguous bytes), row groups of 8,
// column blocks.  A box of `rows` x `cols` of X lands in shared memory as
// [column block][row][8 elements], the no-swizzle canonical layout.
constexpr int kMapsPerMatrix = 12;   // 3 views of each operand buffer, 2 of the Gram matrix, polynomial, 2 store views, W
bool encode_xop_map(CUtensorMap* map, const void* base, const Shape& s, int rows, int cols) {
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(s.xrows / 8), static_cast<cuuint64_t>(s.xblocks)};
    cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(s.xrows * 16)};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows / 8), static_cast<cuuint32_t>(cols / 8)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


struct MatBufs {
    size_t x_op[2], gram, poly;
};

// Counts of tiles per phase for one matrix.
// Rows of one tensor-core output tile: 128 for a single CTA, 256 for a CTA pair.
int64_t tile_rows(bool pair) { return pair ? 2 * kTcBM : kTcBM; }

// Tiles of one symmetric phase (those that meet the upper triangle) and of
// one apply phase of an m x n iterate.
int64_t sym_tiles(int64_t m, bool pair = false) {
    int64_t cnt = 0;
    const int64_t bm = tile_rows(pair);
    const int64_t tr = ceil_div(m, bm), tc = ceil_div(m, kTcBN);
    for (int64_t I = 0; I < tr; ++I)
        for (int64_t J = 0; J < tc; ++J)
            if (std::min(J * kTcBN + kTcBN - 1, m - 1) >= I * bm) ++cnt;
    return cnt;
}
int64_t apply_tiles(int64_t m, int64_t n, bool pair = false) {
    return ceil_div(m, tile_rows(pair)) * ceil_div(n, kTcBN);
}

struct Layout {
    int precision;
    size_t mats, tmaps, tiles[3], ranges[3], deps, partials, scales, power, bufs_begin, total;
    int64_t total_rows;            // sum of m (power-iteration rows)
    std::vector<size_t> pv;        // per matrix: offset of its two power-iteration vectors and its
                                   // diagonal residual vector (3 x lda floats)
    size_t ctl_bytes;              // [0, ctl_bytes) is uploaded every call
    int64_t ntiles[3];
    int64_t mom_tiles;
    std::vector<MatBufs> buf;
    std::vector<Shape> shape;
};

Layout make_layout(const std::vector<std::pair<int64_t, int64_t>>& dims, int precision) {
    Layout L;
    L.precision = precision;
    const size_t n = dims.size();
    L.shape.resize(n);
    L.buf.resize(n);
    L.ntiles[0] = L.ntiles[1] = L.ntiles[2] = 0;
    L.mom_tiles = 0;
    for (size_t i = 0; i < n; ++i) {
        const Shape s = oriented(dims[i].first, dims[i].second);
        L.shape[i] = s;
        L.mom_tiles += ceil_div(dims[i].first, kMomTile) * ceil_div(dims[i].second, kMomTile);
        if (precision == MO_NS_BF16) {
            const int64_t st = sym_tiles(s.m);
            L.ntiles[0] += st;
            L.ntiles[1] += st;
            L.ntiles[2] += apply_tiles(s.m, s.n);   // single-CTA counts bound the pair ones
        } else {
            const int64_t t = ceil_div(s.m, kFpBM);
            L.ntiles[0] += t * t;
            L.ntiles[1] += t * t;
            L.ntiles[2] += t * ceil_div(s.n, kFpBN);
        }
    }
    size_t off = kHeaderBytes;
    L.mats = off;
    off = align_up(off + n * sizeof(MatDesc), 128);
    L.tmaps = off;
    if (precision == MO_NS_BF16) off = align_up(off + n * kMapsPerMatrix * sizeof(CUtensorMap), 128);
    for (int ph = 0; ph < 3; ++ph) {
        L.tiles[ph] = off;
        off = align_up(off + static_cast<size_t>(L.ntiles[ph]) * sizeof(TileDesc), 128);
        L.ranges[ph] = off;
        off = align_up(off + static_cast<size_t>(L.ntiles[ph]) * sizeof(int2), 128);
    }
    L.deps = off;                  // per matrix 4 ints (3 used), then the grid-wide set; zeroed by every upload
    off = align_up(off + (n + 1) * 4 * sizeof(int), 128);
    L.ctl_bytes = off;
    L.partials = off;
    off = align_up(off + static_cast<size_t>(L.mom_tiles) * sizeof(float), 128);
    L.scales = off;
    off = align_up(off + n * kScaleStride * sizeof(float), 128);
    L.power = off;
    L.pv.resize(n);
    L.total_rows = 0;
    for (size_t i = 0; i < n; ++i) {
        L.pv[i] = off;
        off = align_up(off + 3 * static_cast<size_t>(L.shape[i].lda) * sizeof(float), 128);
        L.total_rows += L.shape[i].m;
    }
    off = align_up(off, kBufAlign);
    L.bufs_begin = off;
    const size_t xe = precision == MO_NS_BF16 ? 2 : 4;
    for (size_t i = 0; i < n; ++i) {
        const Shape& s = L.shape[i];
        const size_t xbytes = precision == MO_NS_BF16 ? static_cast<size_t>(s.xblocks) * s.xrows * 16
                                                      : static_cast<size_t>(s.m) * s.ldx * xe;
        const size_t abytes = static_cast<size_t>(s.m) * s.lda * xe;
        MatBufs& b = L.buf[i];
        b.x_op[0] = off; off = align_up(off + xbytes, kBufAlign);
        b.x_op[1] = off; off = align_up(off + xbytes, kBufAlign);
        b.gram = off; off = align_up(off + abytes, kBufAlign);
        b.poly = off; off = align_up(off + abytes, kBufAlign);
    }
    L.total = off;
    return L;
}

// LPT assignment of tiles to CTAs: tiles sorted by cost (descending, then
// matrix / row / column), each to the least-loaded CTA (ties: lower index).
// The symmetric phases' tiles whose first 128 columns lie below the diagonal
// issue half their MMAs but keep a full epilogue; costed at half their K
// blocks they took more tiles per CTA and measured slower (GPT-small +10%),
// so every tile is costed by its K blocks.
void schedule(std::vector<TileDesc>& tiles, int ctas, int epi_cost, std::vector<TileDesc>& out,
              std::vector<int2>& ranges) {
    std::stable_sort(tiles.begin(), tiles.end(), [](const TileDesc& a, const TileDesc& b) {
        return a.nkb > b.nkb;
    });
    using Item = std::pair<int64_t, int>;
    std::priority_queue<Item, std::vector<Item>, std::greater<Item>> heap;
    for (int c = 0; c < ctas; ++c) heap.push({0, c});
    std::vector<std::vector<int>> per(ctas);
    for (size_t t = 0; t < tiles.size(); ++t) {
        Item it = heap.top();
        heap.pop();
        per[it.second].push_back(static_cast<int>(t));
        it.first += tiles[t].nkb + epi_cost;
        heap.push(it);
    }
    out.clear();
    ranges.assign(ctas, make_int2(0, 0));
    for (int c = 0; c < ctas; ++c) {
        ranges[c].x = static_cast<int>(out.size());
        ranges[c].y = static_cast<int>(per[c].size());
        for (int t : per[c]) out.push_back(tiles[t]);
    }
}

int validate_ws(void* ws, size_t ws_bytes, size_t need) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % kWsAlign) != 0) return MO_ERR_WORKSPACE;
    if (ws_bytes < need) return MO_ERR_WORKSPACE;
    return MO_OK;
}

int validate_dims(int64_t rows, int64_t cols, int64_t ld) {
    if (rows < 0 || cols < 0 || ld < 0) return MO_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return MO_OK;
    if (ld < cols) return MO_ERR_INVALID_ARG;
    if (std::min(rows, cols) > kMaxMinDim || std::max(rows, cols) > kMaxDim) return MO_ERR_UNSUPPORTED;
    return MO_OK;
}

int validate_buffer(const void* p, int dt, int64_t ld) {
    if (!valid_dtype(dt)) return MO_ERR_INVALID_ARG;
    if (p == nullptr) return MO_ERR_INVALID_ARG;
    if (!aligned16(p) || (static_cast<size_t>(ld) * elem_size(dt)) % 16 != 0) return MO_ERR_ALIGNMENT;
    return MO_OK;
}

int validate_tail(const mo_adamw_tail* t) {
    if (t == nullptr) return MO_OK;
    if (t->numel < 0) return MO_ERR_INVALID_ARG;
    if (t->numel == 0) return MO_OK;
    if (t->step < 1) return MO_ERR_INVALID_ARG;
    if (!t->W || !t->g || !t->m || !t->v) return MO_ERR_INVALID_ARG;
    if (!aligned16(t->W) || !aligned16(t->g) || !aligned16(t->m) || !aligned16(t->v)) return MO_ERR_ALIGNMENT;
    return MO_OK;
}

struct NsOpts {
    int precision, steps, apply_update;
    float mu, a, b, c, alpha, decay;
    int spectral_iters = 0;        // > 0: spectral-scale normalisation with this many power iterations
    // Sign-Muon vote after the NS (muon_step_sign_vote): W <- W - lr * vote of
    // the jobs' packed signs, a launch of its own after the NS
    void* vote_W = nullptr;
    int vote_w_dtype = MO_F32;
    int64_t vote_ld = 0;
    float vote_lr = 0.f;
};

// ------------------------------------------------------------ launch trace
// Optional per-thread record of a CUDA event pair around each kernel launch
// (enabled by mo_trace_enable), read back by mo_trace_read.
struct Trace {
    int capacity = 0;
    int count = 0;
    std::vector<cudaEvent_t> begin, end;
    std::vector<int32_t> kind;
};
thread_local Trace t_trace;

// Optional per-CTA stamps of the tensor-core NS launches (mo_debug_cta_stamps):
// launch k of the record writes 4 * max_ctas values at buf + 4 * k * max_ctas.
struct Stamps {
    unsigned long long* buf = nullptr;
    int capacity = 0, max_ctas = 0, count = 0;
};
thread_local Stamps t_stamps;

template <typename F>
cudaError_t traced(int kind, cudaStream_t s, F&& launch) {
    Trace& t = t_trace;
    const bool on = t.capacity > 0 && t.count < t.capacity;
    if (on && cudaEventRecord(t.begin[t.count], s) != cudaSuccess) return cudaErrorUnknown;
    cudaError_t e = launch();
    if (on && e == cudaSuccess) {
        if (cudaEventRecord(t.end[t.count], s) != cudaSuccess) return cudaErrorUnknown;
        t.kind[t.count] = kind;
        ++t.count;
    }
    return e;
}

// A built control block (descriptor table, tensor maps, scheduled tile
// lists) for one request placed in one workspace.  The staged bytes are
// uploaded on every call; building them (tensor-map encoding, LPT
// scheduling) is cached by everything that shapes their content.
struct Plan {
    std::vector<int64_t> key;
    Layout L;
    std::vector<uint8_t> stage;
    bool pair = false;             // tensor-core tiles for CTA pairs (cta_group::2)
    int grids[3] = {0, 0, 0};      // schedule units (CTAs, or CTA pairs) holding tiles, per phase
    int64_t ntiles[3] = {0, 0, 0}; // tiles per phase in this geometry
};

std::mutex g_plan_mu;
std::vector<std::shared_ptr<const Plan>> g_plans;   // most recently used first
constexpr size_t kPlanCacheSize = 16;

std::vector<int64_t> plan_key(const std::vector<Job>& jobs, int precision, const void* ws, bool pair, int units) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    std::vector<int64_t> k;
    k.reserve(6 + jobs.size() * 13);
    k.push_back(dev);
    k.push_back(precision);
    k.push_back(pair ? 1 : 0);
    k.push_back(units);
    k.push_back(static_cast<int64_t>(reinterpret_cast<uintptr_t>(ws)));
    k.push_back(device_sm_count());
    for (const Job& j : jobs) {
        const int64_t f[12] = {j.rows, j.cols, j.ld, j.src_dtype, j.g_dtype, j.w_dtype, j.out_dtype, j.has_momentum,
                               static_cast<int64_t>(reinterpret_cast<uintptr_t>(j.src)),
                               static_cast<int64_t>(reinterpret_cast<uintptr_t>(j.grad)),
                               static_cast<int64_t>(reinterpret_cast<uintptr_t>(j.W)),
                               static_cast<int64_t>(reinterpret_cast<uintptr_t>(j.out))};
        k.insert(k.end(), f, f + 12);
        k.push_back(static_cast<int64_t>(reinterpret_cast<uintptr_t>(j.words)));
    }
    return k;
}

// `units`: schedule units of the tensor-core path (CTAs, or CTA pairs when `pair`).
int build_plan(const std::vector<Job>& jobs, int precision, void* ws, bool pair, int units,
               std::shared_ptr<Plan>& out) {
    std::vector<std::pair<int64_t, int64_t>> dims;
    dims.reserve(jobs.size());
    for (const Job& j : jobs) dims.push_back({j.rows, j.cols});
    auto plan = std::make_shared<Plan>();
    plan->L = make_layout(dims, precision);
    const Layout& L = plan->L;
    if (precision == MO_NS_BF16 && !get_encode()) return MO_ERR_CUDA;

    uint8_t* base = static_cast<uint8_t*>(ws);
    plan->pair = pair;
    plan->stage.assign(L.ctl_bytes, 0);
    uint8_t* h = plan->stage.data();
    const NsOpts o{precision, 0, 0, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0};
    MatDesc* hm = reinterpret_cast<MatDesc*>(h + L.mats);
    CUtensorMap* htm = reinterpret_cast<CUtensorMap*>(h + L.tmaps);
    const CUtensorMap* dtm = reinterpret_cast<const CUtensorMap*>(base + L.tmaps);

    int64_t mom_begin = 0, row_begin = 0;
    for (size_t i = 0; i < jobs.size(); ++i) {
        const Job& j = jobs[i];
        const Shape& s = L.shape[i];
        const MatBufs& b = L.buf[i];
        MatDesc& d = hm[i];
        d.m = static_cast<int32_t>(s.m);
        d.n = static_cast<int32_t>(s.n);
        d.ldx = static_cast<int32_t>(s.ldx);
        d.xrows = static_cast<int32_t>(s.xrows);
        d.lda = static_cast<int32_t>(s.lda);
        d.ld = j.ld;
        d.rows = static_cast<int32_t>(j.rows);
        d.cols = static_cast<int32_t>(j.cols);
        d.transposed = s.transposed;
        d.src_dtype = j.src_dtype;
        d.g_dtype = j.g_dtype;
        d.w_dtype = j.w_dtype;
        d.out_dtype = j.out_dtype;
        d.has_momentum = j.has_momentum;
        d.src = j.src;
        d.grad = j.grad;
        d.W = j.W;
        d.out = j.out;
        d.sign_words = j.words;
        d.x_op[0] = base + b.x_op[0];
        d.x_op[1] = base + b.x_op[1];
        d.gram = base + b.gram;
        d.poly = base + b.poly;
        d.scales = reinterpret_cast<float*>(base + L.scales) + kScaleStride * i;
        d.pv = reinterpret_cast<float*>(base + L.pv[i]);
        d.py = d.pv + s.lda;
        d.dlo = d.pv + 2 * s.lda;
        d.row_begin = row_begin;
        row_begin += s.m;
        d.mom_tile_begin = mom_begin;
        d.mom_tiles_r = static_cast<int32_t>(ceil_div(j.rows, kMomTile));
        d.mom_tiles_c = static_cast<int32_t>(ceil_div(j.cols, kMomTile));
        mom_begin += static_cast<int64_t>(d.mom_tiles_r) * d.mom_tiles_c;
        d.nt_sym = static_cast<int32_t>(sym_tiles(s.m, pair));
        d.nt_apply = static_cast<int32_t>(apply_tiles(s.m, s.n, pair));
        d.deps = reinterpret_cast<int*>(base + L.deps) + 4 * i;
        if (o.precision == MO_NS_BF16) {
            const int bn = pair ? kTcBN / 2 : kTcBN;     // B-operand columns one CTA loads
            CUtensorMap* hm0 = htm + kMapsPerMatrix * i;
            const CUtensorMap* dm0 = dtm + kMapsPerMatrix * i;
            for (int q = 0; q < 2; ++q) {
                if (!encode_xop_map(&hm0[3 * q + 0], d.x_op[q], s, kTcBM, kTcBK) ||
                    !encode_xop_map(&hm0[3 * q + 1], d.x_op[q], s, bn, kTcBK) ||
                    !encode_xop_map(&hm0[3 * q + 2], d.x_op[q], s, kTcBK, bn))
                    return MO_ERR_CUDA;
                d.tm_xa[q] = dm0 + 3 * q + 0;
                d.tm_xb[q] = dm0 + 3 * q + 1;
                d.tm_xn[q] = dm0 + 3 * q + 2;
            }
            if (!encode_bf16_map(&hm0[6], d.gram, s.m, s.m, s.lda, kTcBM)) return MO_ERR_CUDA;
            if (!encode_bf16_map(&hm0[7], d.gram, s.m, s.m, s.lda, bn)) return MO_ERR_CUDA;
            if (!encode_bf16_map(&hm0[8], d.poly, s.m, s.m, s.lda, kTcBM)) return MO_ERR_CUDA;
            if (!encode_bf16_store_map(&hm0[9], d.gram, s.m, s.m, s.lda)) return MO_ERR_CUDA;
            if (!encode_bf16_store_map(&hm0[10], d.poly, s.m, s.m, s.lda)) return MO_ERR_CUDA;
            d.tm_gram = dm0 + 6;
            d.tm_gram_b = dm0 + 7;
            d.tm_poly = dm0 + 8;
            d.tm_gram_st = dm0 + 9;
            d.tm_poly_st = dm0 + 10;
            d.tm_w = j.W != nullptr && encode_w_map(&hm0[11], j.W, j.w_dtype, j.rows, j.cols, j.ld) ? dm0 + 11 : nullptr;
        } else {
            for (int q = 0; q < 2; ++q) d.tm_xa[q] = d.tm_xb[q] = d.tm_xn[q] = nullptr;
            d.tm_gram = d.tm_gram_b = d.tm_poly = d.tm_gram_st = d.tm_poly_st = d.tm_w = nullptr;
        }
    }

    // tile lists per phase
    int* grids = plan->grids;
    for (int ph = 0; ph < 3; ++ph) {
        std::vector<TileDesc> tiles;
        tiles.reserve(static_cast<size_t>(L.ntiles[ph]));
        for (size_t i = 0; i < jobs.size(); ++i) {
            const Shape& s = L.shape[i];
            if (o.precision == MO_NS_BF16) {
                const int nkb = static_cast<int>(ceil_div(ph == kGram ? s.n : s.m, kTcBK));
                const int64_t bm = tile_rows(pair);
                const int64_t tr = ceil_div(s.m, bm);
                const int64_t tc = ceil_div(ph == kApply ? s.n : s.m, kTcBN);
                if (ph == kApply) {
                    // column-block-major: the CTAs of one wave share a few
                    // 256-column panels of X while B (m x m) stays in L2
                    for (int64_t J = 0; J < tc; ++J)
                        for (int64_t I = 0; I < tr; ++I)
                            tiles.push_back(TileDesc{static_cast<int32_t>(i), static_cast<int32_t>(I),
                                                     static_cast<int32_t>(J), nkb});
                } else {
                    for (int64_t I = 0; I < tr; ++I)
                        for (int64_t J = 0; J < tc; ++J) {
                            if (std::min(J * kTcBN + kTcBN - 1, s.m - 1) < I * bm) continue;
                            tiles.push_back(TileDesc{static_cast<int32_t>(i), static_cast<int32_t>(I),
                                                     static_cast<int32_t>(J), nkb});
                        }
                }
            } else {
                const int nkb = static_cast<int>(ceil_div(ph == kGram ? s.n : s.m, kFpBK));
                const int64_t tr = ceil_div(s.m, kFpBM);
                const int64_t tc = ceil_div(ph == kApply ? s.n : s.m, kFpBN);
                for (int64_t I = 0; I < tr; ++I)
                    for (int64_t J = 0; J < tc; ++J)
                        tiles.push_back(TileDesc{static_cast<int32_t>(i), static_cast<int32_t>(I),
                                                 static_cast<int32_t>(J), nkb});
            }
        }
        TileDesc* ht = reinterpret_cast<TileDesc*>(h + L.tiles[ph]);
        plan->ntiles[ph] = static_cast<int64_t>(tiles.size());
        if (o.precision == MO_NS_BF16) {
            const int ctas = static_cast<int>(std::min<int64_t>(units, static_cast<int64_t>(tiles.size())));
            std::vector<TileDesc> sorted;
            std::vector<int2> ranges;
            schedule(tiles, ctas, ph == kApply ? 6 : 4, sorted, ranges);
            std::memcpy(ht, sorted.data(), sorted.size() * sizeof(TileDesc));
            std::memcpy(h + L.ranges[ph], ranges.data(), ranges.size() * sizeof(int2));
            grids[ph] = ctas;
        } else {
            std::memcpy(ht, tiles.data(), tiles.size() * sizeof(TileDesc));
            grids[ph] = static_cast<int>(tiles.size());
        }
    }
    out = plan;
    return MO_OK;
}

int get_plan(const std::vector<Job>& jobs, int precision, void* ws, bool pair, int units,
             std::shared_ptr<const Plan>& out) {
    std::vector<int64_t> key = plan_key(jobs, precision, ws, pair, units);
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        for (size_t i = 0; i < g_plans.size(); ++i) {
            if (g_plans[i]->key == key) {
                out = g_plans[i];
                std::rotate(g_plans.begin(), g_plans.begin() + i, g_plans.begin() + i + 1);
                return MO_OK;
            }
        }
    }
    std::shared_ptr<Plan> p;
    int st = build_plan(jobs, precision, ws, pair, units, p);
    if (st != MO_OK) return st;
    p->key = std::move(key);
    std::lock_guard<std::mutex> lk(g_plan_mu);
    g_plans.insert(g_plans.begin(), p);
    if (g_plans.size() > kPlanCacheSize) g_plans.pop_back();
    out = p;
    return MO_OK;
}

// Uploads the (cached) control block for `jobs` into `ws` and launches the
// whole path on `stream`.
// Launch errors that mean the launch was refused before anything ran.
bool launch_refused(cudaError_t e) {
    return e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorLaunchOutOfResources ||
           e == cudaErrorInvalidConfiguration || e == cudaErrorNotSupported || e == cudaErrorInvalidClusterSize;
}

int run_ns(const std::vector<Job>& jobs, const NsOpts& o, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (jobs.empty()) return MO_OK;
    int st = validate_ws(ws, ws_bytes, 0);
    if (st != MO_OK) return st;
    const bool tc = o.precision == MO_NS_BF16;
    const int nsm = device_sm_count();
    const bool pair = tc && g_ns_pair.load() != 0 && tc_capacity(true) >= 2;
    const int units = pair ? std::min(nsm / 2, tc_capacity(true) / 2) : nsm;
    const int cta_per_unit = pair ? 2 : 1;
    std::shared_ptr<const Plan> plan;
    if ((st = get_plan(jobs, o.precision, ws, pair, units, plan)) != MO_OK) return st;
    const Layout& L = plan->L;
    if ((st = validate_ws(ws, ws_bytes, L.total)) != MO_OK) return st;
    const int* grids = plan->grids;
    uint8_t* base = static_cast<uint8_t*>(ws);

    cudaError_t e = cudaMemcpyAsync(base, plan->stage.data(), L.ctl_bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return MO_ERR_CUDA;
    if (tc) {
        // The bf16 operand's padding is read by the tensor cores (inside whole
        // 128-byte TMA lines) and must hold zeros: the rows from m up to a
        // multiple of 8 in every block of both buffers, and the columns of the
        // last block from n on (bf16(M) is written over the rest of that block).
        for (size_t i = 0; i < jobs.size(); ++i) {
            const Shape& sh = L.shape[i];
            const MatBufs& b = L.buf[i];
            if (sh.xrows > sh.m)
                for (int q = 0; q < 2; ++q) {
                    e = cudaMemset2DAsync(base + b.x_op[q] + sh.m * 16, static_cast<size_t>(sh.xrows) * 16, 0,
                                          static_cast<size_t>(sh.xrows - sh.m) * 16, static_cast<size_t>(sh.xblocks),
                                          stream);
                    if (e != cudaSuccess) return MO_ERR_CUDA;
                }
            if (sh.n % 8 != 0) {
                e = cudaMemsetAsync(base + b.x_op[0] + static_cast<size_t>(sh.xblocks - 1) * sh.xrows * 16, 0,
                                    static_cast<size_t>(sh.xrows) * 16, stream);
                if (e != cudaSuccess) return MO_ERR_CUDA;
            }
        }
    }

    const MatDesc* dmats = reinterpret_cast<const MatDesc*>(base + L.mats);
    MomLaunch mp;
    mp.mats = dmats;
    mp.nmats = static_cast<int32_t>(jobs.size());
    mp.ntiles = L.mom_tiles;
    mp.mu = o.mu;
    mp.fp32_operand = o.precision == MO_NS_FP32;
    mp.partials = reinterpret_cast<float*>(base + L.partials);
    const int mom_grid = static_cast<int>(std::min<int64_t>(L.mom_tiles, static_cast<int64_t>(nsm) * 8));
    // bf16 momentum with an fp32 gradient, untransposed and 16-byte aligned
    // throughout: the kernel with 16-byte momentum accesses
    bool bf16m = o.precision == MO_NS_BF16;
    for (const Job& j : jobs)
        bf16m = bf16m && j.has_momentum && j.src_dtype == MO_BF16 && j.g_dtype == MO_F32 && j.rows <= j.cols &&
                j.ld % 8 == 0 && reinterpret_cast<uintptr_t>(j.src) % 16 == 0 &&
                reinterpret_cast<uintptr_t>(j.grad) % 16 == 0;
    if (bf16m) {
        const int grid6 = static_cast<int>(std::min<int64_t>(L.mom_tiles, static_cast<int64_t>(nsm) * 6));
        e = traced(MO_K_MOMENTUM, stream, [&] { return launch_momentum_norm_bf16m(mp, grid6, stream); });
    } else {
        e = traced(MO_K_MOMENTUM, stream, [&] { return launch_momentum_norm(mp, mom_grid, stream); });
    }
    if (e != cudaSuccess) return MO_ERR_CUDA;
    e = traced(MO_K_FINALIZE, stream, [&] { return launch_norm_finalize(dmats, mp.nmats, mp.partials, stream); });
    if (e != cudaSuccess) return MO_ERR_CUDA;

    if (o.steps == 0) {
        e = traced(MO_K_NS0, stream,
                   [&] { return launch_ns_k0(mp, o.alpha, o.decay, o.apply_update, mom_grid, stream); });
        return map_cuda(e);
    }
    NsLaunch np{};
    np.mats = dmats;
    np.err = reinterpret_cast<int*>(base);
    np.steps = o.steps;
    np.apply_update = o.apply_update;
    np.a = o.a;
    np.b = o.b;
    np.c = o.c;
    np.alpha = o.alpha;
    np.decay = o.decay;
    np.mn_lbo = kMnLbo;
    np.mn_sbo = kMnSbo;
    np.stall_mat = g_stall_mat.load();
    np.dep_wait_cycles = np.stall_mat >= 0 ? g_stall_wait_cycles.load() : kDepWaitCycles;
    np.level_deps = reinterpret_cast<int*>(base + L.deps) + 4 * jobs.size();
    np.tot_sym = static_cast<int32_t>(plan->ntiles[kGram]);
    np.tot_apply = static_cast<int32_t>(plan->ntiles[kApply]);
    np.rel_per_tile = kTcEpiGroupWarps * cta_per_unit;
    const uint32_t mma_m = static_cast<uint32_t>(kTcBM * cta_per_unit);
    np.idesc_sym = idesc_bf16_f32(mma_m, kTcBN, 0u);
    np.idesc_apply = idesc_bf16_f32(mma_m, kTcBN, 1u);
    for (int ph = 0; ph < 3; ++ph) {
        np.tc_tiles[ph] = reinterpret_cast<const TileDesc*>(base + L.tiles[ph]);
        np.tc_ranges[ph] = reinterpret_cast<const int2*>(base + L.ranges[ph]);
        np.tc_ctas[ph] = grids[ph];
    }
    const int levels = 3 * o.steps;
    const int units_fused = std::max(grids[0], std::max(grids[1], grids[2]));
    int mode = g_ns_fused.load();             // 0 per-phase, 1 / 2 fused (counter granularity)
    if (mode == 3) mode = plan->ntiles[kGram] < kPerMatrixDepsMaxSymTilesPerCta * units_fused ? 1 : 2;

    // one launch of levels [lv0, lv1): the per-phase form, or the fused one
    auto launch_levels = [&](int lv0, int lv1) -> cudaError_t {
        const bool fused = lv1 - lv0 > 1;
        np.lv_begin = lv0;
        np.lv_end = lv1;
        np.deps = fused ? mode : 0;
        np.phase = lv0 % 3;
        np.step = lv0 / 3;
        np.tiles = reinterpret_cast<const TileDesc*>(base + L.tiles[np.phase]);
        np.ntiles = static_cast<int32_t>(L.ntiles[np.phase]);
        const int grid = (fused ? units_fused : grids[np.phase]) * (tc ? cta_per_unit : 1);
        np.stamps = nullptr;
        Stamps& sp = t_stamps;
        if (tc && sp.buf != nullptr && sp.count < sp.capacity && grid <= sp.max_ctas)
            np.stamps = sp.buf + 4 * static_cast<int64_t>(sp.count++) * sp.max_ctas;
        return traced(fused ? MO_K_NS_FUSED : MO_K_GRAM + np.phase, stream, [&] {
            return tc ? launch_ns_tc(np, grid, fused, pair, stream) : launch_ns_fp32_phase(np, grid, stream);
        });
    };

    // the spectral estimate runs between the first Gram phase and the rest
    const int lv_fuse = o.spectral_iters > 0 ? 1 : 0;
    const bool fuse = tc && mode != 0 && levels - lv_fuse > 1 && units_fused * cta_per_unit <= tc_capacity(pair);
    for (int lv = 0; lv < levels;) {
        const int lv1 = fuse && lv >= lv_fuse ? levels : lv + 1;
        e = launch_levels(lv, lv1);
        if (e != cudaSuccess && lv1 - lv > 1 && launch_refused(e)) {
            // the runtime refused the cooperative launch (another client holding
            // SMs, a profiler, ...): nothing ran, so run the levels one by one
            (void)cudaGetLastError();
            for (int l = lv; l < lv1 && (e = launch_levels(l, l + 1)) == cudaSuccess; ++l) {}
        }
        if (e != cudaSuccess) return MO_ERR_CUDA;
        if (lv == 0 && o.spectral_iters > 0) {
            // spectral scale: power iteration on the first Gram matrix, folded
            // into the first polynomial and apply through the per-matrix scales
            e = traced(MO_K_SPECTRAL, stream, [&] {
                return launch_spectral_estimate(dmats, static_cast<int>(jobs.size()), L.total_rows,
                                                o.spectral_iters, nsm, stream);
            });
            if (e != cudaSuccess) return MO_ERR_CUDA;
        }
        lv = lv1;
    }
    if (o.vote_W != nullptr) {
        // the Sign-Muon vote over the packed signs the last epilogue wrote
        std::vector<const uint32_t*> wp;
        for (const Job& j : jobs) wp.push_back(j.words);
        e = traced(MO_K_VOTE, stream, [&] {
            return launch_sign_vote_update(wp.data(), static_cast<int>(wp.size()), jobs[0].rows, jobs[0].cols,
                                           o.vote_W, o.vote_w_dtype, o.vote_ld, o.vote_lr, stream);
        });
        if (e != cudaSuccess) return MO_ERR_CUDA;
    }
    return MO_OK;
}

int ns_workspace_for(const std::vector<std::pair<int64_t, int64_t>>& dims, int precision, size_t* out) {
    if (out == nullptr) return MO_ERR_INVALID_ARG;
    *out = make_layout(dims, precision).total;
    return MO_OK;
}

int gather_muon_jobs(const mo_matrix* mats, int n, const mo_muon_cfg* cfg, void* const* out,
                     bool check_ptrs, std::vector<Job>& jobs, std::vector<int>* index_map) {
    if (n < 0 || cfg == nullptr || (n > 0 && mats == nullptr)) return MO_ERR_INVALID_ARG;
    if (cfg->ns_steps < 0 || (cfg->ns_precision != MO_NS_BF16 && cfg->ns_precision != MO_NS_FP32))
        return MO_ERR_INVALID_ARG;
    if (cfg->spectral_iters < 0) return MO_ERR_INVALID_ARG;
    if (cfg->spectral_iters > 0 && (cfg->ns_precision != MO_NS_BF16 || cfg->ns_steps < 1 || cfg->spectral_iters > 64))
        return MO_ERR_UNSUPPORTED;
    if (!cfg->apply_update && !valid_dtype(cfg->out_dtype)) return MO_ERR_INVALID_ARG;
    if (check_ptrs && !cfg->apply_update && n > 0 && out == nullptr) return MO_ERR_INVALID_ARG;
    jobs.clear();
    for (int i = 0; i < n; ++i) {
        const mo_matrix& mt = mats[i];
        int st = validate_dims(mt.rows, mt.cols, mt.ld);
        if (st != MO_OK) return st;
        if (!valid_dtype(mt.w_dtype) || !valid_dtype(mt.m_dtype) || !valid_dtype(mt.g_dtype))
            return MO_ERR_INVALID_ARG;
        if (mt.rows == 0 || mt.cols == 0) continue;
        if (check_ptrs) {
            if ((st = validate_buffer(mt.M, mt.m_dtype, mt.ld)) != MO_OK) return st;
            if ((st = validate_buffer(mt.G, mt.g_dtype, mt.ld)) != MO_OK) return st;
            if (cfg->apply_update) {
                if ((st = validate_buffer(mt.W, mt.w_dtype, mt.ld)) != MO_OK) return st;
            } else {
                if ((st = validate_buffer(out[i], cfg->out_dtype, mt.ld)) != MO_OK) return st;
            }
        }
        Job j;
        j.rows = mt.rows;
        j.cols = mt.cols;
        j.ld = mt.ld;
        j.src_dtype = mt.m_dtype;
        j.g_dtype = mt.g_dtype;
        j.w_dtype = mt.w_dtype;
        j.out_dtype = cfg->out_dtype;
        j.has_momentum = 1;
        j.src = mt.M;
        j.grad = mt.G;
        j.W = cfg->apply_update ? mt.W : nullptr;
        j.out = (!cfg->apply_update && out) ? out[i] : nullptr;
        jobs.push_back(j);
        if (index_map) index_map->push_back(i);
    }
    return MO_OK;
}

}  // namespace
}  // namespace mo

using namespace mo;

extern "C" {

int mo_version(void) { return 0x000100; }

const char* mo_status_string(int s) {
    switch (s) {
        case MO_OK: return "MO_OK";
        case MO_ERR_INVALID_ARG: return "MO_ERR_INVALID_ARG: invalid argument";
        case MO_ERR_ALIGNMENT: return "MO_ERR_ALIGNMENT: pointer or leading dimension not 16-byte aligned";
        case MO_ERR_WORKSPACE: return "MO_ERR_WORKSPACE: workspace null, misaligned or too small";
        case MO_ERR_CUDA: return "MO_ERR_CUDA: a CUDA call failed";
        case MO_ERR_TIMEOUT: return "MO_ERR_TIMEOUT: a device-side wait gave up";
        case MO_ERR_UNSUPPORTED: return "MO_ERR_UNSUPPORTED: outside what this build implements";
        default: return "unknown status";
    }
}

int mo_workspace_bytes(const mo_matrix* mats, int n, const mo_muon_cfg* cfg, size_t* bytes_out) {
    if (bytes_out == nullptr) return MO_ERR_INVALID_ARG;
    std::vector<Job> jobs;
    int st = gather_muon_jobs(mats, n, cfg, nullptr, false, jobs, nullptr);
    if (st != MO_OK) return st;
    std::vector<std::pair<int64_t, int64_t>> dims;
    for (const Job& j : jobs) dims.push_back({j.rows, j.cols});
    return ns_workspace_for(dims, cfg->ns_precision, bytes_out);
}

int muon_step_batched(const mo_matrix* mats, int n, const mo_muon_cfg* cfg, const mo_adamw_tail* tail,
                      void* const* out, void* ws, size_t ws_bytes, mo_stream_t stream) {
    std::vector<Job> jobs;
    int st = gather_muon_jobs(mats, n, cfg, out, true, jobs, nullptr);
    if (st != MO_OK) return st;
    if ((st = validate_tail(tail)) != MO_OK) return st;
    if (!jobs.empty()) {
        std::vector<std::pair<int64_t, int64_t>> dims;
        for (const Job& j : jobs) dims.push_back({j.rows, j.cols});
        size_t need = 0;
        ns_workspace_for(dims, cfg->ns_precision, &need);
        if ((st = validate_ws(ws, ws_bytes, need)) != MO_OK) return st;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (tail != nullptr && tail->numel > 0) {
        if (traced(MO_K_ADAMW, s, [&] { return launch_adamw(*tail, s); }) != cudaSuccess) return MO_ERR_CUDA;
    }
    NsOpts o;
    o.precision = cfg->ns_precision;
    o.steps = cfg->ns_steps;
    o.apply_update = cfg->apply_update;
    o.mu = cfg->mu;
    o.a = cfg->a;
    o.b = cfg->b;
    o.c = cfg->c;
    o.alpha = cfg->lr * cfg->update_scale;
    o.decay = cfg->lr * cfg->weight_decay;
    o.spectral_iters = cfg->spectral_iters;
    return run_ns(jobs, o, ws, ws_bytes, s);
}

}  // extern "C"

namespace mo {
namespace {
// The jobs of a Sign-Muon step with the sign + 1-bit pack fused into the last
// NS epilogue: momentum and gradient buffers validated, packed-word targets
// attached, no W update or output.
int gather_sign_jobs(const mo_matrix* mats, int n, const mo_muon_cfg* cfg, uint32_t* const* words,
                     std::vector<Job>& jobs) {
    if (cfg == nullptr) return MO_ERR_INVALID_ARG;
    if (cfg->ns_precision != MO_NS_BF16 || cfg->ns_steps < 1) return MO_ERR_UNSUPPORTED;
    mo_muon_cfg c2 = *cfg;
    c2.apply_update = 0;
    std::vector<int> idx;
    int st = gather_muon_jobs(mats, n, &c2, nullptr, false, jobs, &idx);
    if (st != MO_OK) return st;
    if (!jobs.empty() && words == nullptr) return MO_ERR_INVALID_ARG;
    for (size_t k = 0; k < jobs.size(); ++k) {
        const mo_matrix& mt = mats[idx[k]];
        if ((st = validate_buffer(mt.M, mt.m_dtype, mt.ld)) != MO_OK) return st;
        if ((st = validate_buffer(mt.G, mt.g_dtype, mt.ld)) != MO_OK) return st;
        uint32_t* w = words[idx[k]];
        if (w == nullptr) return MO_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(w) & 3u) != 0) return MO_ERR_ALIGNMENT;
        if (mt.cols % 32 != 0) return MO_ERR_UNSUPPORTED;    // rows must start on word boundaries
        jobs[k].words = w;
        jobs[k].W = nullptr;
        jobs[k].out = nullptr;
    }
    return MO_OK;
}
}  // namespace
}  // namespace mo

extern "C" {

int muon_step_sign_packed(const mo_matrix* mats, int n, const mo_muon_cfg* cfg, uint32_t* const* words, void* ws,
                          size_t ws_bytes, mo_stream_t stream) {
    std::vector<Job> jobs;
    int st = gather_sign_jobs(mats, n, cfg, words, jobs);
    if (st != MO_OK) return st;
    NsOpts o;
    o.precision = MO_NS_BF16;
    o.steps = cfg->ns_steps;
    o.apply_update = 0;
    o.mu = cfg->mu;
    o.a = cfg->a;
    o.b = cfg->b;
    o.c = cfg->c;
    o.alpha = 0.f;
    o.decay = 0.f;
    o.spectral_iters = cfg->spectral_iters;
    return run_ns(jobs, o, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int muon_step_sign_vote(const mo_matrix* mats, int n, const mo_muon_cfg* cfg, uint32_t* const* words, void* W,
                        int w_dtype, int64_t ld, float lr, void* ws, size_t ws_bytes, mo_stream_t stream) {
    std::vector<Job> jobs;
    int st = gather_sign_jobs(mats, n, cfg, words, jobs);
    if (st != MO_OK) return st;
    if (jobs.empty()) return MO_OK;
    if (static_cast<int>(jobs.size()) > kMaxVoteWorkers) return MO_ERR_UNSUPPORTED;
    for (const Job& j : jobs)
        if (j.rows != jobs[0].rows || j.cols != jobs[0].cols) return MO_ERR_INVALID_ARG;
    if (W == nullptr || !valid_dtype(w_dtype) || ld < jobs[0].cols) return MO_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) % elem_size(w_dtype)) != 0) return MO_ERR_ALIGNMENT;
    NsOpts o;
    o.precision = MO_NS_BF16;
    o.steps = cfg->ns_steps;
    o.apply_update = 0;
    o.mu = cfg->mu;
    o.a = cfg->a;
    o.b = cfg->b;
    o.c = cfg->c;
    o.alpha = 0.f;
    o.decay = 0.f;
    o.spectral_iters = cfg->spectral_iters;
    o.vote_W = W;
    o.vote_w_dtype = w_dtype;
    o.vote_ld = ld;
    o.vote_lr = lr;
    return run_ns(jobs, o, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int ns_workspace_bytes(const int64_t* rows, const int64_t* cols, int n, int precision, size_t* bytes_out) {
    if (bytes_out == nullptr || n < 0 || (n > 0 && (rows == nullptr || cols == nullptr))) return MO_ERR_INVALID_ARG;
    if (precision != MO_NS_BF16 && precision != MO_NS_FP32) return MO_ERR_INVALID_ARG;
    std::vector<std::pair<int64_t, int64_t>> dims;
    for (int i = 0; i < n; ++i) {
        int st = validate_dims(rows[i], cols[i], cols[i]);
        if (st != MO_OK) return st;
        if (rows[i] > 0 && cols[i] > 0) dims.push_back({rows[i], cols[i]});
    }
    return ns_workspace_for(dims, precision, bytes_out);
}

int ns_orthogonalize(const void* const* X, void* const* out, const int64_t* rows, const int64_t* cols,
                     const int64_t* ld, int n, int in_dtype, int out_dtype, int steps, float a, float b, float c,
                     int precision, void* ws, size_t ws_bytes, mo_stream_t stream) {
    if (n < 0 || steps < 0) return MO_ERR_INVALID_ARG;
    if (precision != MO_NS_BF16 && precision != MO_NS_FP32) return MO_ERR_INVALID_ARG;
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return MO_ERR_INVALID_ARG;
    if (n > 0 && (!X || !out || !rows || !cols || !ld)) return MO_ERR_INVALID_ARG;
    std::vector<Job> jobs;
    for (int i = 0; i < n; ++i) {
        int st = validate_dims(rows[i], cols[i], ld[i]);
        if (st != MO_OK) return st;
        if (rows[i] == 0 || cols[i] == 0) continue;
        if ((st = validate_buffer(X[i], in_dtype, ld[i])) != MO_OK) return st;
        if ((st = validate_buffer(out[i], out_dtype, ld[i])) != MO_OK) return st;
        Job j;
        j.rows = rows[i];
        j.cols = cols[i];
        j.ld = ld[i];
        j.src_dtype = in_dtype;
        j.g_dtype = in_dtype;
        j.w_dtype = out_dtype;
        j.out_dtype = out_dtype;
        j.has_momentum = 0;
        j.src = const_cast<void*>(X[i]);
        j.grad = nullptr;
        j.W = nullptr;
        j.out = out[i];
        jobs.push_back(j);
    }
    NsOpts o;
    o.precision = precision;
    o.steps = steps;
    o.apply_update = 0;
    o.mu = 0.f;
    o.a = a;
    o.b = b;
    o.c = c;
    o.alpha = 0.f;
    o.decay = 0.f;
    return run_ns(jobs, o, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int sign_pack(const void* U, int dtype, int64_t rows, int64_t cols, int64_t ld, uint32_t* words,
              mo_stream_t stream) {
    if (!valid_dtype(dtype) || rows < 0 || cols < 0) return MO_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return MO_OK;
    if (ld < cols || U == nullptr || words == nullptr) return MO_ERR_INVALID_ARG;
    // element accesses only: element alignment suffices
    if ((reinterpret_cast<uintptr_t>(U) % elem_size(dtype)) != 0 || (reinterpret_cast<uintptr_t>(words) & 3u) != 0)
        return MO_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return map_cuda(traced(MO_K_PACK, s, [&] { return launch_sign_pack(U, dtype, rows, cols, ld, words, s); }));
}

int sign_vote_update(const uint32_t* const* words, int M, int64_t rows, int64_t cols, void* W, int w_dtype,
                     int64_t ld, float lr, mo_stream_t stream) {
    if (M <= 0 || !valid_dtype(w_dtype) || rows < 0 || cols < 0) return MO_ERR_INVALID_ARG;
    if (M > 128) return MO_ERR_UNSUPPORTED;
    if (rows == 0 || cols == 0) return MO_OK;
    if (words == nullptr || W == nullptr || ld < cols) return MO_ERR_INVALID_ARG;
    for (int m = 0; m < M; ++m) {
        if (words[m] == nullptr) return MO_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(words[m]) & 3u) != 0) return MO_ERR_ALIGNMENT;
    }
    if ((reinterpret_cast<uintptr_t>(W) % elem_size(w_dtype)) != 0) return MO_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return map_cuda(traced(MO_K_VOTE, s, [&] {
        return launch_sign_vote_update(words, M, rows, cols, W, w_dtype, ld, lr, s);
    }));
}

int sign_pack_batched(const void* const* U, int M, int dtype, int64_t rows, int64_t cols, int64_t ld,
                      uint32_t* const* words, mo_stream_t stream) {
    if (M <= 0 || !valid_dtype(dtype) || rows < 0 || cols < 0) return MO_ERR_INVALID_ARG;
    if (M > 128) return MO_ERR_UNSUPPORTED;
    if (rows == 0 || cols == 0) return MO_OK;
    if (ld < cols || U == nullptr || words == nullptr) return MO_ERR_INVALID_ARG;
    for (int m = 0; m < M; ++m) {
        if (U[m] == nullptr || words[m] == nullptr) return MO_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(U[m]) % elem_size(dtype)) != 0 ||
            (reinterpret_cast<uintptr_t>(words[m]) & 3u) != 0)
            return MO_ERR_ALIGNMENT;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return map_cuda(traced(MO_K_PACK, s, [&] {
        return launch_sign_pack_batched(U, words, M, dtype, rows, cols, ld, s);
    }));
}

int sign_vote_polar_workspace_bytes(int64_t rows, int64_t cols, int64_t ld, size_t* bytes_out) {
    if (bytes_out == nullptr) return MO_ERR_INVALID_ARG;
    int st = validate_dims(rows, cols, ld);
    if (st != MO_OK) return st;
    if (rows == 0 || cols == 0) {
        *bytes_out = 0;
        return MO_OK;
    }
    const size_t sbytes = align_up(static_cast<size_t>(rows) * ld * 2, kBufAlign);
    *bytes_out = sbytes + make_layout({{rows, cols}}, MO_NS_BF16).total;
    return MO_OK;
}

int sign_vote_polar_update(const uint32_t* const* words, int M, int64_t rows, int64_t cols, void* W, int w_dtype,
                           int64_t ld, float lr, int steps, float a, float b, float c, void* ws, size_t ws_bytes,
                           mo_stream_t stream) {
    if (M <= 0 || !valid_dtype(w_dtype) || steps < 0) return MO_ERR_INVALID_ARG;
    if (M > 128) return MO_ERR_UNSUPPORTED;
    int st = validate_dims(rows, cols, ld);
    if (st != MO_OK) return st;
    if (rows == 0 || cols == 0) return MO_OK;
    if (words == nullptr) return MO_ERR_INVALID_ARG;
    for (int m = 0; m < M; ++m) {
        if (words[m] == nullptr) return MO_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(words[m]) & 3u) != 0) return MO_ERR_ALIGNMENT;
    }
    if ((st = validate_buffer(W, w_dtype, ld)) != MO_OK) return st;
    size_t need = 0;
    sign_vote_polar_workspace_bytes(rows, cols, ld, &need);
    if ((st = validate_ws(ws, ws_bytes, need)) != MO_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // S_bar (bf16, W's layout) at the start of the workspace, the NS workspace after it
    void* S = ws;
    const size_t sbytes = align_up(static_cast<size_t>(rows) * ld * 2, kBufAlign);
    cudaError_t e = traced(MO_K_VOTE, s, [&] { return launch_vote_matrix(words, M, rows, cols, S, ld, s); });
    if (e != cudaSuccess) return MO_ERR_CUDA;
    Job j;
    j.rows = rows;
    j.cols = cols;
    j.ld = ld;
    j.src_dtype = MO_BF16;
    j.g_dtype = MO_BF16;
    j.w_dtype = w_dtype;
    j.out_dtype = w_dtype;
    j.has_momentum = 0;
    j.src = S;
    j.grad = nullptr;
    j.W = W;
    j.out = nullptr;
    NsOpts o;
    o.precision = MO_NS_BF16;
    o.steps = steps;
    o.apply_update = 1;
    o.mu = 0.f;
    o.a = a;
    o.b = b;
    o.c = c;
    o.alpha = lr;
    o.decay = 0.f;
    return run_ns({j}, o, static_cast<uint8_t*>(ws) + sbytes, ws_bytes - sbytes, s);
}

int sign_int8(const void* U, int dtype, int64_t rows, int64_t cols, int64_t ld, int8_t* out, mo_stream_t stream) {
    if (!valid_dtype(dtype) || rows < 0 || cols < 0) return MO_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return MO_OK;
    if (ld < cols || U == nullptr || out == nullptr) return MO_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(U) % elem_size(dtype)) != 0) return MO_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return map_cuda(traced(MO_K_PACK, s, [&] { return launch_sign_int8(U, dtype, rows, cols, ld, out, s); }));
}

int sign_vote_update_int8(const int8_t* const* signs, int M, int64_t rows, int64_t cols, void* W, int w_dtype,
                          int64_t ld, float lr, mo_stream_t stream) {
    if (M <= 0 || !valid_dtype(w_dtype) || rows < 0 || cols < 0) return MO_ERR_INVALID_ARG;
    if (M > 127) return MO_ERR_UNSUPPORTED;
    if (rows == 0 || cols == 0) return MO_OK;
    if (signs == nullptr || W == nullptr || ld < cols) return MO_ERR_INVALID_ARG;
    for (int m = 0; m < M; ++m)
        if (signs[m] == nullptr) return MO_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) % elem_size(w_dtype)) != 0) return MO_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return map_cuda(traced(MO_K_VOTE, s, [&] {
        return launch_vote_int8(signs, M, rows, cols, W, w_dtype, ld, lr, s);
    }));
}

int plan_owners(const int64_t* rows, const int64_t* cols, int n, int world, int ns_steps, double w_bytes,
                double w_flops, int32_t* owner_out, double* load_out) {
    if (world <= 0 || n < 0 || ns_steps < 0) return MO_ERR_INVALID_ARG;
    if (n > 0 && (rows == nullptr || cols == nullptr || owner_out == nullptr)) return MO_ERR_INVALID_ARG;
    std::vector<double> bytes(n), flops(n), cost(n);
    for (int i = 0; i < n; ++i) {
        if (rows[i] < 0 || cols[i] < 0) return MO_ERR_INVALID_ARG;
        const double r = static_cast<double>(rows[i]), c = static_cast<double>(cols[i]);
        bytes[i] = r * c * 2.0;
        const double m = rows[i] <= cols[i] ? r : c;
        const double nn = rows[i] <= cols[i] ? c : r;
        flops[i] = static_cast<double>(ns_steps) * (4.0 * m * m * nn + 2.0 * m * m * m);
    }
    double sb = 0.0, sf = 0.0;
    for (int i = 0; i < n; ++i) sb += bytes[i];
    for (int i = 0; i < n; ++i) sf += flops[i];
    for (int i = 0; i < n; ++i) {
        const double cb = sb > 0.0 ? bytes[i] / sb : 0.0;
        const double cf = sf > 0.0 ? flops[i] / sf : 0.0;
        const double tb = w_bytes * cb;
        const double tf = w_flops * cf;
        cost[i] = tb + tf;
    }
    std::vector<int> order(n);
    for (int i = 0; i < n; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
        if (cost[x] != cost[y]) return cost[x] > cost[y];
        return x < y;
    });
    std::vector<double> load(world, 0.0);
    for (int i : order) {
        int best = 0;
        for (int r = 1; r < world; ++r)
            if (load[r] < load[best]) best = r;
        owner_out[i] = best;
        load[best] += cost[i];
    }
    if (load_out != nullptr)
        for (int r = 0; r < world; ++r) load_out[r] = load[r];
    return MO_OK;
}

int mo_check_device_status(void* ws, mo_stream_t stream) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % kWsAlign) != 0) return MO_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int err = 0;
    if (cudaMemcpyAsync(&err, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MO_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MO_ERR_CUDA;
    if (err != 0) {
        const int zero = 0;
        if (cudaMemcpyAsync(ws, &zero, sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess) return MO_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return MO_ERR_CUDA;
        return MO_ERR_TIMEOUT;
    }
    return MO_OK;
}

int mo_debug_ns_view(const int64_t* rows, const int64_t* cols, int n, int precision, int index,
                     mo_ns_view* view) {
    if (view == nullptr || n < 0 || index < 0 || index >= n || rows == nullptr || cols == nullptr)
        return MO_ERR_INVALID_ARG;
    if (precision != MO_NS_BF16 && precision != MO_NS_FP32) return MO_ERR_INVALID_ARG;
    if (rows[index] <= 0 || cols[index] <= 0) return MO_ERR_INVALID_ARG;
    std::vector<std::pair<int64_t, int64_t>> dims;
    int active = -1;
    for (int i = 0; i < n; ++i) {
        if (rows[i] > 0 && cols[i] > 0) {
            if (i == index) active = static_cast<int>(dims.size());
            dims.push_back({rows[i], cols[i]});
        }
    }
    const Layout L = make_layout(dims, precision);
    const Shape& s = L.shape[active];
    const MatBufs& b = L.buf[active];
    view->m = s.m;
    view->n = s.n;
    view->ldx = precision == MO_NS_BF16 ? s.xrows : s.ldx;   // bf16: rows of an 8-column block
    view->lda = s.lda;
    view->transposed = s.transposed;
    view->precision = precision;
    view->x_op[0] = static_cast<int64_t>(b.x_op[0]);
    view->x_op[1] = static_cast<int64_t>(b.x_op[1]);
    view->diag_res = precision == MO_NS_BF16
                         ? static_cast<int64_t>(L.pv[active] + 2 * static_cast<size_t>(s.lda) * sizeof(float))
                         : 0;
    view->gram = static_cast<int64_t>(b.gram);
    view->poly = static_cast<int64_t>(b.poly);
    view->deps = static_cast<int64_t>(L.deps + 4 * sizeof(int) * static_cast<size_t>(active));
    const bool pair = precision == MO_NS_BF16 && g_ns_pair.load() != 0 && tc_capacity(true) >= 2;
    view->tiles_sym = static_cast<int32_t>(sym_tiles(s.m, pair));
    view->tiles_apply = static_cast<int32_t>(apply_tiles(s.m, s.n, pair));
    view->releases_per_tile = kTcEpiGroupWarps * (pair ? 2 : 1);
    view->reserved = 0;
    return MO_OK;
}

int mo_debug_sm_count(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return c;
}

int mo_debug_cta_stamps(uint64_t* buf, int capacity, int max_ctas, int* recorded) {
    Stamps& sp = t_stamps;
    if (recorded != nullptr) *recorded = sp.count;
    if (buf == nullptr) {
        sp = Stamps{};
        return MO_OK;
    }
    if (capacity <= 0 || max_ctas <= 0 || (reinterpret_cast<uintptr_t>(buf) & 7u) != 0) return MO_ERR_INVALID_ARG;
    sp.buf = reinterpret_cast<unsigned long long*>(buf);
    sp.capacity = capacity;
    sp.max_ctas = max_ctas;
    sp.count = 0;
    return MO_OK;
}

int mo_trace_enable(int capacity) {
    Trace& t = t_trace;
    if (capacity < 0) return MO_ERR_INVALID_ARG;
    for (int i = static_cast<int>(t.begin.size()); i < capacity; ++i) {
        cudaEvent_t b, e;
        if (cudaEventCreate(&b) != cudaSuccess) return MO_ERR_CUDA;
        if (cudaEventCreate(&e) != cudaSuccess) return MO_ERR_CUDA;
        t.begin.push_back(b);
        t.end.push_back(e);
        t.kind.push_back(0);
    }
    t.capacity = capacity;
    t.count = 0;
    return MO_OK;
}

int mo_trace_read(int32_t* kinds, float* ms, int cap, int* count) {
    Trace& t = t_trace;
    if (count == nullptr || cap < 0 || (cap > 0 && (kinds == nullptr || ms == nullptr))) return MO_ERR_INVALID_ARG;
    const int n = std::min(cap, t.count);
    if (t.count > 0 && cudaEventSynchronize(t.end[t.count - 1]) != cudaSuccess) return MO_ERR_CUDA;
    for (int i = 0; i < n; ++i) {
        kinds[i] = t.kind[i];
        if (cudaEventElapsedTime(&ms[i], t.begin[i], t.end[i]) != cudaSuccess) return MO_ERR_CUDA;
    }
    *count = t.count;
    t.count = 0;
    return MO_OK;
}

int mo_debug_set_ns_pair(int on) {
    if (on != 0 && on != 1) return MO_ERR_INVALID_ARG;
    return g_ns_pair.exchange(on);
}

int mo_debug_inject_dep_stall(int matrix, int64_t wait_cycles) {
    if (matrix < -1) return MO_ERR_INVALID_ARG;
    if (matrix >= 0 && (wait_cycles < 1000 || wait_cycles > kDepWaitCycles)) return MO_ERR_INVALID_ARG;
    g_stall_wait_cycles.store(matrix >= 0 ? wait_cycles : 0);
    g_stall_mat.store(matrix);
    return MO_OK;
}

int mo_debug_set_ns_fused(int on) {
    if (on < 0 || on > 3) return MO_ERR_INVALID_ARG;
    return g_ns_fused.exchange(on);
}

}  // extern "C"
