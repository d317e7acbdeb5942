// txl_relattn_fwd_noalloc: the relative-position attention forward for callers
// that cannot allocate device memory when they run it.
//
// Some callers may not call cudaMalloc at that point: plugins of inference
// engines whose execute step must not allocate, and runtimes whose device
// memory budget is fixed once at start-up.  txl_relattn_fwd needs a caller
// workspace when it splits a head's key range over several blocks; this entry
// point instead uses a scratch array that is part of the library itself, so it
// needs nothing from the caller and allocates nothing.
//
// The scratch is one file-scope __device__ array of TXL_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  All calls
// share it and each call overwrites what the previous one left; the partial
// results written there are complete before they are read, so nothing needs
// clearing.  Two calls that can run at the same time on the GPU (different
// streams, or different host threads without ordering) race on it.
#include <mutex>

#include "txl.h"

namespace {

// Partial outputs and log-sum-exps of split key ranges.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TXL_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of the scratch array on the current device.  Host code may
// not use the array's name as an address (it is a host-side stand-in), so it is
// looked up once per device, with that device current, and cached.
void *scratch_address(int *status)
{
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = TXL_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            *status = TXL_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
    }
    *status = TXL_OK;
    return addr[dev];
}

} // namespace

extern "C" int txl_relattn_fwd_noalloc(const void *q, const void *k, const void *v,
                                       const void *r, int r_rows, const void *u,
                                       const void *v_bias, void *out, float *lse, int B, int H,
                                       int M, int L, int dh, float scale, int dtype,
                                       int n_splits, void *stream)
{
    // txl_relattn_fwd sizes the split it will actually run (decode key ranges
    // merged inside a thread-block cluster need no scratch; requests above the
    // key-tile count are capped) against the scratch and refuses, before
    // anything is launched, a split whose partial results do not fit.
    int status = TXL_OK;
    void *scratch = scratch_address(&status);
    if (!scratch) return status;
    return txl_relattn_fwd(q, k, v, r, r_rows, u, v_bias, out, lse, B, H, M, L, dh, scale,
                           dtype, n_splits, scratch, (size_t)TXL_NOALLOC_SCRATCH_BYTES, stream);
}
