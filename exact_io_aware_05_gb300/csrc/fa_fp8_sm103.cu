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

// Eight consecutive bf16 values (one 16-byte load) as floats.
__device__ __forceinline__ void unpack8(const uint4 &u, float (&x)[8])
{
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __bfloat162float(h[i].x);
        x[2 * i + 1] = __bfloat162float(h[i].y);
    }
}

// Unnormalised Walsh-Hadamard transform of one row held by TPR consecutive lanes, lane j
// of the group holding elements [8j, 8j + 8): butterflies for h = 1, 2, 4 inside the
// thread, then h = 8, 16, ... across lanes (the lane with bit h/8 set holds the upper
// element), each pair (i, i + h) -> (a + b, a - b) rounded to fp32, h increasing.
template <int TPR>
__device__ __forceinline__ void fwht_row8(float (&x)[8], uint32_t lane)
{
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if ((i & h) == 0) {
                const float a = x[i], b = x[i + h];
                x[i] = __fadd_rn(a, b);
                x[i + h] = __fsub_rn(a, b);
            }
    }
#pragma unroll
    for (int m = 1; m < TPR; m <<= 1) {
        const bool upper = (lane & (uint32_t)m) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
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

// 16 warps x 8 rows; a row is held by D/8 lanes, 8 elements (16 bytes) each.
template <int D>
__global__ void __launch_bounds__(QWARPS * 32) fp8_rows_kernel(const RowQuantArgs a)
{
    constexpr int TPR = D / 8;                // lanes per row
    constexpr int RPS = 32 / TPR;             // rows per warp step
    constexpr int STEPS = (QB / QWARPS) / RPS;
    const bool z = blockIdx.z != 0;   // selects, not run-time array indexing (keeps the args in registers)
    const int T = z ? a.T[1] : a.T[0];
    const __nv_bfloat16 *src = z ? a.x[1] : a.x[0];
    uint8_t *codes = z ? a.codes[1] : a.codes[0];
    float *descale = z ? a.descale[1] : a.descale[0];
    const int nb = (T + QB - 1) / QB;
    if ((int)blockIdx.x >= nb)
        return;
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const size_t bh = blockIdx.y;
    const int col = (int)(lane % TPR) * 8;
    const int rbase = blockIdx.x * QB + (int)warp * (QB / QWARPS) + (int)(lane / TPR);
    uint4 raw[STEPS];
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
        const int r = rbase + st * RPS;
        raw[st] = r < T ? *reinterpret_cast<const uint4 *>(src + (bh * T + r) * D + col) : make_uint4(0, 0, 0, 0);
    }
    float sg[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        sg[i] = a.signs ? a.signs[col + i] : 1.f;
    float x[STEPS][8];
    float amax = 0.f;
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
        unpack8(raw[st], x[st]);
        if (a.signs) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[st][i] *= sg[i];
            fwht_row8<TPR>(x[st], lane);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            amax = fmaxf(amax, fabsf(x[st][i]));
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
        descale[bh * nb + blockIdx.x] = amax / kE4M3Max * norm;
    }
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
        const int r = rbase + st * RPS;
        if (r >= T)
            continue;
        uint32_t w[2];
#pragma unroll
        for (int i = 0; i < 2; ++i)
            w[i] = pack_e4m3x4(__fmul_rn(x[st][4 * i], inv), __fmul_rn(x[st][4 * i + 1], inv),
                               __fmul_rn(x[st][4 * i + 2], inv), __fmul_rn(x[st][4 * i + 3], inv));
        *reinterpret_cast<uint2 *>(codes + (bh * T + r) * D + col) = make_uint2(w[0], w[1]);
    }
}

// A 128-key tile of V for 256 threads: D/8 threads per key row, 8 channels (16 bytes)
// each; thread t holds channels [8 (t % TPR), +8) of RPT consecutive keys.
template <int D>
struct VTile {
    static constexpr int TPR = D / 8, RG = 256 / TPR, RPT = QB / RG;
};

template <int D>
__device__ __forceinline__ void load_vtile(const __nv_bfloat16 *__restrict__ v, size_t bh, int l0, int Tk,
                                           uint4 (&raw)[VTile<D>::RPT])
{
    using V = VTile<D>;
    const int cg = (int)threadIdx.x % V::TPR, rg = (int)threadIdx.x / V::TPR;
#pragma unroll
    for (int w = 0; w < V::RPT; ++w) {
        const int l = l0 + rg * V::RPT + w;
        raw[w] = l < Tk ? *reinterpret_cast<const uint4 *>(v + (bh * Tk + l) * D + cg * 8) : make_uint4(0, 0, 0, 0);
    }
}

// V, pass 1: per-channel max |v| of 128 keys, merged into amax[bh][c] (float bits; the
// values are >= 0, so their bit patterns order like the values).
template <int D>
__global__ void __launch_bounds__(256) fp8_vmax_kernel(const __nv_bfloat16 *__restrict__ v, unsigned *amax, int Tk)
{
    using V = VTile<D>;
    const size_t bh = blockIdx.y;
    uint4 raw[V::RPT];
    load_vtile<D>(v, bh, blockIdx.x * QB, Tk, raw);
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        m[i] = 0.f;
#pragma unroll
    for (int w = 0; w < V::RPT; ++w) {
        float x[8];
        unpack8(raw[w], x);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            m[i] = fmaxf(m[i], fabsf(x[i]));
    }
    __shared__ float sm[V::RG][D];
    const int cg = (int)threadIdx.x % V::TPR, rg = (int)threadIdx.x / V::TPR;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        sm[rg][cg * 8 + i] = m[i];
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        float r = 0.f;
#pragma unroll
        for (int g = 0; g < V::RG; ++g)
            r = fmaxf(r, sm[g][c]);
        atomicMax(amax + bh * D + c, __float_as_uint(r));
    }
}

// V, pass 2: codes of 128 keys x D channels, transposed into vt[bh][c][l] (row stride ld,
// a multiple of 16): through shared memory, then 16-byte stores along the keys.  Codes
// of keys past Tk inside the last 16-byte chunk are 0.
template <int D>
__global__ void __launch_bounds__(256) fp8_vquant_kernel(const __nv_bfloat16 *__restrict__ v,
                                                         const unsigned *__restrict__ amax, uint8_t *vt, int Tk,
                                                         size_t ld)
{
    using V = VTile<D>;
    constexpr int LDS = QB + 4;                 // bytes per [channel] row of the tile
    __shared__ __align__(16) uint8_t tile[D * LDS];
    const size_t bh = blockIdx.y;
    const int l0 = blockIdx.x * QB;
    const int cg = (int)threadIdx.x % V::TPR, rg = (int)threadIdx.x / V::TPR;
    uint4 raw[V::RPT];
    load_vtile<D>(v, bh, l0, Tk, raw);
    float inv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float am = __uint_as_float(amax[bh * D + cg * 8 + i]);
        inv[i] = am > 0.f ? __fdiv_rn(kE4M3Max, am) : 0.f;
    }
    // codes of channel cg*8 + i for keys rg*RPT .. +RPT, four keys per word
    uint32_t cw[8][V::RPT / 4];
#pragma unroll
    for (int w4 = 0; w4 < V::RPT / 4; ++w4) {
        float x[4][8];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            unpack8(raw[4 * w4 + e], x[e]);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            cw[i][w4] = pack_e4m3x4(__fmul_rn(x[0][i], inv[i]), __fmul_rn(x[1][i], inv[i]),
                                    __fmul_rn(x[2][i], inv[i]), __fmul_rn(x[3][i], inv[i]));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int w4 = 0; w4 < V::RPT / 4; ++w4)
            *reinterpret_cast<uint32_t *>(tile + (cg * 8 + i) * LDS + rg * V::RPT + 4 * w4) = cw[i][w4];
    __syncthreads();
    for (int idx = threadIdx.x; idx < D * (QB / 16); idx += blockDim.x) {
        const int c = idx / (QB / 16), k16 = (idx % (QB / 16)) * 16;
        if (l0 + k16 >= Tk)
            continue;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(tile + c * LDS + k16);
        *reinterpret_cast<uint4 *>(vt + (bh * D + c) * ld + l0 + k16) = make_uint4(src[0], src[1], src[2], src[3]);
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
