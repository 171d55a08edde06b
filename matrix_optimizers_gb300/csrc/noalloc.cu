// ns_orthogonalize_noalloc: Newton-Schulz on one matrix with no caller
// workspace and no allocation.  Its scratch is a fixed array in device global
// memory, compiled into the library, of MO_NOALLOC_SCRATCH_BYTES; every GPU
// that loads the library holds it until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/matrixopt.h"

namespace {

// The scratch.  In host code this name is only a host-side stand-in for the
// device array: its address must come from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MO_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) on the first call that runs there.
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MO_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MO_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MO_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MO_OK;
}

}  // namespace

extern "C" int ns_orthogonalize_noalloc(const void* X, void* out, int64_t rows, int64_t cols, int64_t ld,
                                        int in_dtype, int out_dtype, int steps, float a, float b, float c,
                                        mo_stream_t stream) {
    if (rows < 0 || cols < 0 || steps < 0) return MO_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return MO_OK;
    size_t need = 0;
    int st = ns_workspace_bytes(&rows, &cols, 1, MO_NS_BF16, &need);
    if (st != MO_OK) return st;
    if (need > MO_NOALLOC_SCRATCH_BYTES) return MO_ERR_UNSUPPORTED;   // matrix too large for the fixed scratch
    void* ws = nullptr;
    if ((st = scratch_address(&ws)) != MO_OK) return st;
    // Everything the run reads from the scratch is written earlier in the
    // same run (the control block and the zeroed error word are uploaded
    // first), so stale contents of a previous call need no clearing.
    return ns_orthogonalize(&X, &out, &rows, &cols, &ld, 1, in_dtype, out_dtype, steps, a, b, c, MO_NS_BF16, ws,
                            MO_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" int ns_orthogonalize_noalloc_status(mo_stream_t stream) {
    void* ws = nullptr;
    const int st = scratch_address(&ws);
    if (st != MO_OK) return st;
    return mo_check_device_status(ws, stream);
}
