// fa_bwd_sm103.cu -- backward pass (placeholder until the tcgen05 kernels land).
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {

__device__ int g_bwd_status;

int bwd_launch(const void *, const void *, const void *, const void *, const float *, const void *, void *, void *,
               void *, int, int, int, int, int, float, const BwdWorkspace &, cudaStream_t)
{
    return ERR_UNSUPPORTED;
}

int bwd_status_fetch_clear(cudaStream_t s, int *host_word)
{
    int zero = 0;
    if (cudaMemcpyFromSymbolAsync(host_word, g_bwd_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_bwd_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return ERR_CUDA;
    return OK;
}

}  // namespace fa
