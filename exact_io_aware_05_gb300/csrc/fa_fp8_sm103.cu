// fa_fp8_sm103.cu -- the FP8 forward's quantization pass on sm_103a.
//
// atlas.blal.pro "FlashAttention -- IO-Aware Exact Attention", "The version ladder:
// FA1 -> FA2 -> FA3" (the FA3 entry): the FP8 forward quantizes its operands in
// blocks, one scale per block, after an "incoherent processing" step, a random
// rotation of Q and K that spreads outlier features over all channels and leaves
// Q K^T unchanged.  Here:
//   * rotation: x -> x diag(s) H, s a vector of d signs given by the caller and H
//     the Sylvester Hadamard matrix, computed as the unnormalised fast transform
//     (butterflies with h = 1, 2, 4, ... in fp32); the 1/sqrt(d) that makes it
//     orthonormal goes into the block's descale;
//   * Q and K: one scale per 128 rows (the forward's tile height), the block's
//     largest |value| maps to 448, the largest e4m3 value; codes are decided in fp32
//     (448 / amax, then x * (448 / amax), then round to nearest even e4m3, saturating);
//   * V: one scale per feature channel over all keys of a head (it factors out of
//     P V), written transposed, [channel][key], so that the P V product reads V with
//     the keys, its reduction dimension, contiguous.
// The pass is bound by HBM: it reads the bf16 operands (V twice) and writes one byte
// per element.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {

namespace {

constexpr int QB = 128;          // rows per scale block
constexpr int QWARPS = 16;       // warps per row block: 8 rows each
constexpr float kE4M3Max = 448.f;

template <int E>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16 *p, float (&x)[E])
{
    if constexpr (E == 2) {
        const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(p);
        x[0] = __bfloat162float(h.x);
        x[1] = __bfloat162float(h.y);
    } else if constexpr (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            x[2 * i] = __bfloat162float(h[i].x);
            x[2 * i + 1] = __bfloat162float(h[i].y);
        }
    } else {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __bfloat162float(h[i].x);
            x[2 * i + 1] = __bfloat162float(h[i].y);
        }
    }
}

// Unnormalised Walsh-Hadamard transform of one row held by a warp, lane L holding
// elements [L*E, L*E + E): butterflies for h = 1, 2, ..., D/2 in that order, each pair
// (i, i + h) -> (a + b, a - b) rounded to fp32; h < E inside the thread, h >= E
// across lanes (the lane with bit h/E set holds the upper element).
template <int E>
__device__ __forceinline__ void fwht_row(float (&x)[E], uint32_t lane)
{
#pragma unroll
    for (int h = 1; h < E; h <<= 1) {
#pragma unroll
        for (int i = 0; i < E; ++i)
            if ((i & h) == 0) {
                const float a = x[i], b = x[i + h];
                x[i] = __fadd_rn(a, b);
                x[i + h] = __fsub_rn(a, b);
            }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & (uint32_t)m) != 0;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const float p = __shfl_xor_sync(0xffffffffu, x[i], m);
            x[i] = upper ? __fsub_rn(p, x[i]) : __fadd_rn(x[i], p);
        }
    }
}

// Q or K: block (blockIdx.x) of 128 rows of head blockIdx.y; blockIdx.z picks the tensor.
struct RowQuantArgs {
    const __nv_bfloat16 *x[2];
    uint8_t *codes[2];
    float *descale[2];
    int T[2];
    const float *signs;      // d signs, or null: no rotation
    int BH;
};

template <int D>
__global__ void __launch_bounds__(QWARPS * 32) fp8_rows_kernel(const RowQuantArgs a)
{
    constexpr int E = D / 32;
    constexpr int RPW = QB / QWARPS;          // rows per warp
    const int z = blockIdx.z;
    const int T = a.T[z];
    const int nb = (T + QB - 1) / QB;
    if ((int)blockIdx.x >= nb)
        return;
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const size_t bh = blockIdx.y;
    const int r0 = blockIdx.x * QB + (int)warp * RPW;
    float sg[E];
#pragma unroll
    for (int i = 0; i < E; ++i)
        sg[i] = a.signs ? a.signs[lane * E + i] : 1.f;
    float x[RPW][E];
    float amax = 0.f;
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int r = r0 + rr;
        if (r < T) {
            load_bf16<E>(a.x[z] + (bh * T + r) * D + lane * E, x[rr]);
        } else {
#pragma unroll
            for (int i = 0; i < E; ++i)
                x[rr][i] = 0.f;
        }
        if (a.signs) {
#pragma unroll
            for (int i = 0; i < E; ++i)
                x[rr][i] *= sg[i];
            fwht_row<E>(x[rr], lane);
        }
#pragma unroll
        for (int i = 0; i < E; ++i)
            amax = fmaxf(amax, fabsf(x[rr][i]));
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    __shared__ float wmax[QWARPS];
    if (lane == 0)
        wmax[warp] = amax;
    __syncthreads();
    amax = 0.f;
#pragma unroll
    for (int w = 0; w < QWARPS; ++w)
        amax = fmaxf(amax, wmax[w]);
    const float inv = amax > 0.f ? __fdiv_rn(kE4M3Max, amax) : 0.f;
    if (threadIdx.x == 0) {
        const float norm = a.signs ? __frsqrt_rn((float)D) : 1.f;
        a.descale[z][bh * nb + blockIdx.x] = amax / kE4M3Max * norm;
    }
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int r = r0 + rr;
        if (r >= T)
            continue;
        uint8_t *dst = a.codes[z] + (bh * T + r) * D + lane * E;
        if constexpr (E == 2) {
            const uint32_t c = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(x[rr][0], inv), __fmul_rn(x[rr][1], inv)),
                                                        __NV_SATFINITE, __NV_E4M3);
            *reinterpret_cast<uint16_t *>(dst) = (uint16_t)c;
        } else {
            uint32_t w[E / 4];
#pragma unroll
            for (int i = 0; i < E / 4; ++i)
                w[i] = pack_e4m3x4(__fmul_rn(x[rr][4 * i], inv), __fmul_rn(x[rr][4 * i + 1], inv),
                              __fmul_rn(x[rr][4 * i + 2], inv), __fmul_rn(x[rr][4 * i + 3], inv));
            if constexpr (E == 4)
                *reinterpret_cast<uint32_t *>(dst) = w[0];
            else
                *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
        }
    }
}

// V, pass 1: per-channel max |v| of 128 keys, merged into amax[bh][c] (float bits; the
// values are >= 0, so their bit patterns order like the values).
template <int D>
__global__ void __launch_bounds__(256) fp8_vmax_kernel(const __nv_bfloat16 *__restrict__ v, unsigned *amax, int Tk)
{
    constexpr int E = D / 32;
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const size_t bh = blockIdx.y;
    float m[E];
#pragma unroll
    for (int i = 0; i < E; ++i)
        m[i] = 0.f;
    for (int rr = (int)warp; rr < QB; rr += 8) {
        const int l = blockIdx.x * QB + rr;
        if (l >= Tk)
            break;
        float x[E];
        load_bf16<E>(v + (bh * Tk + l) * D + lane * E, x);
#pragma unroll
        for (int i = 0; i < E; ++i)
            m[i] = fmaxf(m[i], fabsf(x[i]));
    }
    __shared__ float sm[8][D];
#pragma unroll
    for (int i = 0; i < E; ++i)
        sm[warp][lane * E + i] = m[i];
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        float r = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w)
            r = fmaxf(r, sm[w][c]);
        atomicMax(amax + bh * D + c, __float_as_uint(r));
    }
}

// V, pass 2: codes of 128 keys x D channels, transposed into vt[bh][c][l] (row stride ld).
template <int D>
__global__ void __launch_bounds__(256) fp8_vquant_kernel(const __nv_bfloat16 *__restrict__ v,
                                                         const unsigned *__restrict__ amax, uint8_t *vt, int Tk,
                                                         size_t ld)
{
    constexpr int E = D / 32;
    constexpr int LDS = QB + 4;                 // padded [channel][key] rows in shared memory
    __shared__ __align__(16) uint8_t tile[D * LDS];
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const size_t bh = blockIdx.y;
    const int l0 = blockIdx.x * QB;
    float inv[E];
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const float am = __uint_as_float(amax[bh * D + lane * E + i]);
        inv[i] = am > 0.f ? __fdiv_rn(kE4M3Max, am) : 0.f;
    }
    for (int rr = (int)warp; rr < QB; rr += 8) {
        const int l = l0 + rr;
        float x[E];
        if (l < Tk) {
            load_bf16<E>(v + (bh * Tk + l) * D + lane * E, x);
        } else {
#pragma unroll
            for (int i = 0; i < E; ++i)
                x[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < E; i += 2) {
            const uint32_t c = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(x[i], inv[i]), __fmul_rn(x[i + 1], inv[i + 1])),
                                                        __NV_SATFINITE, __NV_E4M3);
            tile[(lane * E + i) * LDS + rr] = (uint8_t)(c & 0xffu);
            tile[(lane * E + i + 1) * LDS + rr] = (uint8_t)(c >> 8);
        }
    }
    __syncthreads();
    // rows of the transposed tile: keys [l0, min(l0 + 128, Tk)) of each channel, 4 bytes a thread
    const int nk = min(QB, Tk - l0);
    for (int idx = threadIdx.x; idx < D * (QB / 4); idx += blockDim.x) {
        const int c = idx / (QB / 4), w4 = idx - c * (QB / 4);
        const int k4 = w4 * 4;
        if (k4 >= nk)
            continue;
        const uint32_t word = *reinterpret_cast<const uint32_t *>(tile + c * LDS + k4);
        uint8_t *dst = vt + (bh * D + c) * ld + l0 + k4;
        if (k4 + 4 <= nk) {
            *reinterpret_cast<uint32_t *>(dst) = word;   // ld and l0 are multiples of 16
        } else {
            for (int e = 0; e < nk - k4; ++e)
                dst[e] = (uint8_t)(word >> (8 * e));
        }
    }
}

__global__ void fp8_vdescale_kernel(float *vd, size_t n)
{
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        vd[i] = vd[i] / kE4M3Max;   // the buffer held the channel's max |v| (float bits)
}

template <int D>
int quantize(const void *q, const void *k, const void *v, const float *signs, int BH, int Tq, int Tk, void *q8,
             void *k8, void *vt8, float *qd, float *kd, float *vd, cudaStream_t s)
{
    RowQuantArgs a;
    a.x[0] = static_cast<const __nv_bfloat16 *>(q);
    a.x[1] = static_cast<const __nv_bfloat16 *>(k);
    a.codes[0] = static_cast<uint8_t *>(q8);
    a.codes[1] = static_cast<uint8_t *>(k8);
    a.descale[0] = qd;
    a.descale[1] = kd;
    a.T[0] = Tq;
    a.T[1] = Tk;
    a.signs = signs;
    a.BH = BH;
    const int nb = ((Tq > Tk ? Tq : Tk) + QB - 1) / QB;
    fp8_rows_kernel<D><<<dim3(nb, BH, Tk > 0 ? 2 : 1), QWARPS * 32, 0, s>>>(a);
    if (Tk > 0) {
        unsigned *amax = reinterpret_cast<unsigned *>(vd);
        if (cudaMemsetAsync(amax, 0, (size_t)BH * D * sizeof(float), s) != cudaSuccess)
            return ERR_CUDA;
        const dim3 grid((Tk + QB - 1) / QB, BH);
        fp8_vmax_kernel<D><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(v), amax, Tk);
        fp8_vquant_kernel<D><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(v), amax,
                                                  static_cast<uint8_t *>(vt8), Tk, fp8_vt_stride(Tk));
        fp8_vdescale_kernel<<<(BH * D + 255) / 256, 256, 0, s>>>(vd, (size_t)BH * D);
    }
    return cudaGetLastError() == cudaSuccess ? OK : ERR_CUDA;
}

}  // namespace

size_t fp8_vt_stride(int Tk) { return ((size_t)Tk + 15) / 16 * 16; }

int fp8_quantize_launch(const void *q, const void *k, const void *v, const float *signs, int BH, int Tq, int Tk,
                        int d, void *q8, void *k8, void *vt8, float *qd, float *kd, float *vd, cudaStream_t s)
{
    switch (d) {
    case 64:
        return quantize<64>(q, k, v, signs, BH, Tq, Tk, q8, k8, vt8, qd, kd, vd, s);
    case 128:
        return quantize<128>(q, k, v, signs, BH, Tq, Tk, q8, k8, vt8, qd, kd, vd, s);
    case 256:
        return quantize<256>(q, k, v, signs, BH, Tq, Tk, q8, k8, vt8, qd, kd, vd, s);
    default:
        return ERR_UNSUPPORTED;
    }
}

}  // namespace fa
