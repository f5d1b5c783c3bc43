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
// up with cudaGetSymbolAddress, with the device current, and cached per device
// together with the CUDA context it belongs to: a call under another context
// (after cudaDeviceReset, or a context the caller made current) looks it up
// again instead of using an address of a context that no longer holds it.
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_noalloc_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
    CUcontext ctx;
    void *addr;
};
Cached g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

CtxGetCurrentFn ctx_get_current()
{
    static std::once_flag once;
    static CtxGetCurrentFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// Device address of the scratch array in the current device's current context;
// looked up on the first call for that (device, context).
int scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return FA_ERR_UNSUPPORTED;
    CtxGetCurrentFn get = ctx_get_current();
    if (!get)
        return FA_ERR_CUDA;
    // With no context current yet, cudaGetSymbolAddress below makes the device's primary
    // context current; the context is read again after it.
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS)
        return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch[dev].addr || !ctx || g_scratch[dev].ctx != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_noalloc_scratch) != cudaSuccess || p == nullptr)
            return FA_ERR_CUDA;
        if (get(&ctx) != CUDA_SUCCESS || !ctx)
            return FA_ERR_CUDA;
        g_scratch[dev] = Cached{ctx, p};
    }
    *out = g_scratch[dev].addr;
    return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const float *lse,
                              const void *dO, void *dq, void *dk, void *dv, int B, int H, int Tq, int Tk, int d,
                              int causal, float scale, fa_stream_t stream)
{
    // fa_bwd's own argument errors first (no CUDA call), then the scratch limit
    if (causal != 0 && causal != 1)
        return FA_ERR_INVALID_ARG;
    const int st = fa::bwd_check_args(q, k, v, o, lse, dO, dq, dk, dv, B, H, Tq, Tk, d, fa::causal_spec(causal),
                                      scale);
    if (st != FA_OK)
        return st;
    const size_t need = fa_bwd_workspace_bytes(B, H, Tq, Tk, d);
    if (need > (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES)
        return FA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const int sa = scratch_address(&scratch);
    if (sa != FA_OK)
        return sa;
    return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, Tq, Tk, d, causal, scale, scratch,
                  (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES, stream);
}
