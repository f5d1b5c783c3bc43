// fa_fwd_f32.cu -- fp32 forward pass with plain FFMA arithmetic (no tensor cores).
//
// The same tiled algorithm as the tensor-core path (zerotofrontier.app
// "FlashAttention", 12.3, "The forward pass"): a query block stays in shared
// memory while key/value blocks stream past it; per row a running maximum m,
// a running sum l and an unnormalised output O~ are corrected by e^(m - m_new)
// whenever the maximum grows, and O = O~ / l, lse = m + log l are written once.
// It exists for fp32 inputs and for results within ~1e-5 of exact attention,
// which tf32/bf16 tensor cores cannot give.  Block sizes are small and fixed
// (32 x 32); this kernel is a precision reference, not a throughput path.
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int FBR = 32, FBC = 32, FTHREADS = 256;

template <int D>
__global__ void __launch_bounds__(FTHREADS) fwd_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                                                           const float *__restrict__ v, float *__restrict__ o,
                                                           float *__restrict__ lse, int Tq, int Tk, int causal,
                                                           float scale, int nqb)
{
    extern __shared__ float sm[];
    float *Qs = sm;                    // [FBR][D]
    float *Ks = Qs + FBR * D;          // [FBC][D]
    float *Vs = Ks + FBC * D;          // [FBC][D]
    float *Os = Vs + FBC * D;          // [FBR][D]
    float *Ss = Os + FBR * D;          // [FBR][FBC + 1]
    float *ms = Ss + FBR * (FBC + 1);  // [FBR]
    float *ls = ms + FBR;              // [FBR]
    float *as = ls + FBR;              // [FBR]

    const int bh = blockIdx.x / nqb;
    const int row0 = (blockIdx.x % nqb) * FBR;
    const float *qh = q + (size_t)bh * Tq * D;
    const float *kh = k + (size_t)bh * Tk * D;
    const float *vh = v + (size_t)bh * Tk * D;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int i = tid; i < FBR * D; i += FTHREADS) {
        const int r = row0 + i / D;
        Qs[i] = r < Tq ? qh[(size_t)r * D + i % D] : 0.f;
        Os[i] = 0.f;
    }
    if (tid < FBR) {
        ms[tid] = -INFINITY;
        ls[tid] = 0.f;
    }
    const int r_last = min(row0 + FBR, Tq) - 1;
    int nkv = (Tk + FBC - 1) / FBC;
    if (causal) {
        const long lim = (long)r_last + Tk - Tq;          // last key any row of the block may see
        nkv = lim < 0 ? 0 : min(nkv, (int)(lim / FBC) + 1);
    }
    for (int j = 0; j < nkv; ++j) {
        __syncthreads();
        const int kv0 = j * FBC;
        for (int i = tid; i < FBC * D; i += FTHREADS) {
            const int l = kv0 + i / D;
            Ks[i] = l < Tk ? kh[(size_t)l * D + i % D] : 0.f;
            Vs[i] = l < Tk ? vh[(size_t)l * D + i % D] : 0.f;
        }
        __syncthreads();
        // scores of the tile, masked entries -inf
        for (int e = tid; e < FBR * FBC; e += FTHREADS) {
            const int rr = e / FBC, cc = e % FBC;
            const int r = row0 + rr, l = kv0 + cc;
            float acc = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c)
                acc = fmaf(Qs[rr * D + c], Ks[cc * D + c], acc);
            const bool ok = l < Tk && (!causal || (long)l <= (long)r + Tk - Tq);
            Ss[rr * (FBC + 1) + cc] = ok ? acc * scale : -INFINITY;
        }
        __syncthreads();
        // online softmax: one warp per row, lane = key within the tile
        for (int rr = warp; rr < FBR; rr += FTHREADS / 32) {
            const float s = Ss[rr * (FBC + 1) + lane];
            float mx = s;
            for (int off = 16; off > 0; off >>= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_old = ms[rr];
            const float m_new = fmaxf(m_old, mx);
            const float ref = m_new == -INFINITY ? 0.f : m_new;
            const float p = s == -INFINITY ? 0.f : expf(s - ref);
            float sum = p;
            for (int off = 16; off > 0; off >>= 1)
                sum += __shfl_xor_sync(0xffffffffu, sum, off);
            const float alpha = m_old == -INFINITY ? 0.f : expf(m_old - ref);
            Ss[rr * (FBC + 1) + lane] = p;
            __syncwarp();
            if (lane == 0) {
                ls[rr] = alpha * ls[rr] + sum;
                ms[rr] = m_new;
                as[rr] = alpha;
            }
        }
        __syncthreads();
        for (int e = tid; e < FBR * D; e += FTHREADS) {
            const int rr = e / D, c = e % D;
            float acc = as[rr] * Os[e];
#pragma unroll 8
            for (int l = 0; l < FBC; ++l)
                acc = fmaf(Ss[rr * (FBC + 1) + l], Vs[l * D + c], acc);
            Os[e] = acc;
        }
    }
    __syncthreads();
    for (int e = tid; e < FBR * D; e += FTHREADS) {
        const int rr = e / D, r = row0 + rr;
        if (r < Tq) {
            const float l = ls[rr];
            o[((size_t)bh * Tq + r) * D + e % D] = l > 0.f ? Os[e] / l : 0.f;
        }
    }
    if (tid < FBR && row0 + tid < Tq) {
        const float l = ls[tid];
        lse[(size_t)bh * Tq + row0 + tid] = l > 0.f ? ms[tid] + logf(l) : -INFINITY;
    }
}

template <int D>
int launch_f32(const float *q, const float *k, const float *v, float *o, float *lse, int BH, int Tq, int Tk,
               int causal, float scale, cudaStream_t s)
{
    const size_t smem = sizeof(float) * (size_t)(4 * FBR * D + FBR * (FBC + 1) + 3 * FBR);
    if (cudaFuncSetAttribute(fwd_f32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return ERR_CUDA;
    const int nqb = (Tq + FBR - 1) / FBR;
    fwd_f32_kernel<D><<<nqb * BH, FTHREADS, smem, s>>>(q, k, v, o, lse, Tq, Tk, causal, scale, nqb);
    return cudaGetLastError() == cudaSuccess ? OK : ERR_CUDA;
}

}  // namespace

int fwd_f32_launch(const float *q, const float *k, const float *v, float *o, float *lse, int BH, int Tq, int Tk,
                   int d, int causal, float scale, cudaStream_t s)
{
    switch (d) {
    case 64:
        return launch_f32<64>(q, k, v, o, lse, BH, Tq, Tk, causal, scale, s);
    case 128:
        return launch_f32<128>(q, k, v, o, lse, BH, Tq, Tk, causal, scale, s);
    case 256:
        return launch_f32<256>(q, k, v, o, lse, BH, Tq, Tk, causal, scale, s);
    default:
        return ERR_UNSUPPORTED;
    }
}

}  // namespace fa
