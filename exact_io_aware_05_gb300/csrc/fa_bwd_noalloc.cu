// fa_bwd_noalloc.cu -- fa_bwd for callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers and may not
// call cudaMalloc: plug-ins whose host framework owns every byte of device
// memory and exposes no allocator to them, and latency-critical code that
// cannot afford cudaMalloc's implicit device synchronisation.  fa_bwd needs a
// scratch workspace (the log2-domain lse, the row terms D and the fp32 dQ
// accumulator); this entry point takes it from a fixed array that the library
// itself places in device memory, so the caller passes no workspace.
//
// The array is a file-scope __device__ variable of FA_BWD_NOALLOC_SCRATCH_BYTES.
// Each device on which the library's code for this file is loaded holds it
// until the process exits (with CUDA's default lazy module loading, that is
// from the first call of fa_bwd_noalloc on that device).  In host code the
// array's name is only a host-side stand-in, so its device address is looked
// up once per device with cudaGetSymbolAddress, with that device current,
// and cached.
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_noalloc_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device; looked up on the
// first call for that device.
int scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_noalloc_scratch) != cudaSuccess || p == nullptr)
            return FA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const float *lse,
                              const void *dO, void *dq, void *dk, void *dv, int B, int H, int Tq, int Tk, int d,
                              int causal, float scale, fa_stream_t stream)
{
    const size_t need = fa_bwd_workspace_bytes(B, H, Tq, Tk, d);
    if (need > (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES)
        return FA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != FA_OK)
        return st;
    return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, Tq, Tk, d, causal, scale, scratch,
                  (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES, stream);
}
