// fa_decode_sm103.cu -- split-KV attention for a few query rows per head
// (decode), on sm_103a.
//
// What it computes: the same O and lse as the forward pass (zerotofrontier.app
// "FlashAttention", "The forward pass"), for Tq <= 16 query rows per head.
// Such rows are too few to fill 128-row tiles, which is why decode kernels
// parallelise over the key/value sequence instead (atlas.blal.pro
// "FlashAttention -- IO-Aware Exact Attention", "Honest caveats & open
// questions": FlashDecoding).  Each CTA runs the online softmax over one chunk
// of the keys of one head and writes a partial state (m, l, O~) per row; a
// second kernel merges the chunks with the online-softmax rescale of the
// pages' section ("The forward pass" step 2.5; llmdeepdive.com lesson 7.7, the
// worked [1, 3] then [5] example): with m = max m_s,
//     l = sum_s e^{c (m_s - m)} l_s,   O = sum_s e^{c (m_s - m)} O~_s / l,
//     lse = c m + ln l.
//
// GB300 design: the work is HBM-bound (about 1 flop per byte of K and V at
// one query row), so it runs on the CUDA cores, not the tensor cores, and is
// built to stream K/V at full bandwidth:
//   * one warp per CTA, several CTAs per SM; 32-key K and V tiles come in
//     through a ring of 2-3 stages by TMA with 128-byte swizzle (conflict-free row
//     reads); the kernel is compiled per bucket of query rows (1, 2, 4, 8, 16);
//   * lane = key for the scores (each lane a full dot product per row), lane =
//     features for P V; scores, P and O~ in fp32 (P is not rounded);
//   * the chunking depends on the sizes only (not on the device), so results
//     are the same on every GB300;
//   * every wait is bounded; a timeout leaves a status word, never a trap.
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {

__device__ int g_dec_status;   // device status word of the decode kernels

namespace {

constexpr int DBK = 32;    // keys per tile (one per lane)

// Row bucket TQ: the kernel is compiled for 1, 2, 4, 8 or 16 query rows, the
// smallest bucket that holds Tq, so that the usual one-row case carries no
// per-row guards and little code.
template <int D, int TQ = (D == 256 ? 8 : 16)>
struct DecCfg {
    static constexpr int TQM = TQ;                  // query rows this instance handles, at most
    // ring stages: one row streams fastest with three tiles in flight; more rows do more
    // arithmetic per tile and gain more from the extra CTAs per SM that two stages allow
    static constexpr int DNS = TQ == 1 ? 3 : 2;
    static constexpr int FPL = D / 32;              // features per lane in P V
    static constexpr int KCH = D / 64;              // 128-byte chunks per row
    static constexpr int CHUNK = DBK * 128;         // one 64-column chunk of a tile
    static constexpr int TILE = KCH * CHUNK;        // K or V tile
    static constexpr int STAGE = 2 * TILE;          // K then V
    static constexpr int OFF_ST = 0;                // 1024-aligned stages first
    static constexpr int OFF_Q = DNS * STAGE;       // q rows, fp32 [TQM][D]
    static constexpr int OFF_BAR = OFF_Q + TQM * D * 4;
    static constexpr int OFF_MISC = OFF_BAR + DNS * 8;   // abort flag
    static constexpr int SMEM = OFF_MISC + 16 + 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

enum DecSite : int { SITE_DEC_FULL = 1 };

struct DecArgs {
    const __nv_bfloat16 *q;
    float *part;        // [BH][nsplit][Tq][D + 2]: O~ (D floats), m, l
    int BH, Tq, Tk, causal;
    float scale_log2;
    int nsplit, tps;    // chunks per head, tiles per chunk
    uint64_t timeout_ns;
};

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float &lo, float &hi)
{
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
}

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// One CTA (one warp) = one chunk of key tiles of one head: online softmax over
// the chunk for every query row, partial (O~, m, l) to the workspace.
template <int D, int TQ>
__global__ void __launch_bounds__(32) decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                    const __grid_constant__ CUtensorMap tm_v, const DecArgs a)
{
    using C = DecCfg<D, TQ>;
    constexpr int TQM = C::TQM, FPL = C::FPL;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const uint32_t bar0 = sbase + C::OFF_BAR;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC);
    const int lane = (int)threadIdx.x;
    const int bh = (int)blockIdx.x / a.nsplit, sp = (int)blockIdx.x - bh * a.nsplit;
    const int ntiles = (a.Tk + DBK - 1) / DBK;
    const int t0 = sp * a.tps, t1 = min(ntiles, t0 + a.tps);
    const int nt = t1 - t0;
    const WaitCtx ctx{abort_flag, &g_dec_status, a.timeout_ns};

    if (lane == 0) {
        for (int s = 0; s < C::DNS; ++s)
            mbar_init(bar0 + 8u * s, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    __syncwarp();
    auto issue = [&](int k) {   // tile t0 + k (K then V) into stage k mod C::DNS
        const uint32_t st = sbase + C::OFF_ST + (uint32_t)(k % C::DNS) * C::STAGE;
        const uint32_t b = bar0 + 8u * (uint32_t)(k % C::DNS);
        mbar_arrive_expect_tx(b, C::STAGE);
        for (int c = 0; c < C::KCH; ++c) {
            tma_load_3d(st + c * C::CHUNK, &tm_k, b, c * 64, (t0 + k) * DBK, bh);
            tma_load_3d(st + C::TILE + c * C::CHUNK, &tm_v, b, c * 64, (t0 + k) * DBK, bh);
        }
    };
    if (lane == 0)
        for (int k = 0; k < C::DNS && k < nt; ++k)
            issue(k);
    // the query rows, as fp32
    float *qs = reinterpret_cast<float *>(smem + C::OFF_Q);
    const __nv_bfloat16 *qg = a.q + (size_t)bh * a.Tq * D;
    for (int e = lane; e < a.Tq * D; e += 32)
        qs[e] = __bfloat162float(qg[e]);
    __syncwarp();

    float m[TQM], l[TQM], o[TQM][FPL];
#pragma unroll
    for (int r = 0; r < TQM; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < FPL; ++e)
            o[r][e] = 0.f;
    }
    const float sl2 = a.scale_log2;
    // P V: this lane's features f0 .. f0 + FPL - 1 of a V row: chunk, byte offset in it
    const int f0 = lane * FPL, vch = f0 / 64, vbyte = (f0 % 64) * 2;
    int k = 0;
    bool ok = true;
    for (; k < nt; ++k) {
        if (!mbar_wait_warp(bar0 + 8u * (uint32_t)(k % C::DNS), (uint32_t)(k / C::DNS) & 1u, ctx, SITE_DEC_FULL)) {
            ok = false;
            break;
        }
        const uint8_t *st = smem + C::OFF_ST + (k % C::DNS) * C::STAGE;
        const int key = (t0 + k) * DBK + lane;
        // scores: lane = key, a full dot product per row (K row read with the swizzle)
        float s[TQM], s2[TQM];
#pragma unroll
        for (int r = 0; r < TQM; ++r)
            s[r] = s2[r] = 0.f;
        const uint8_t *krow = st + lane * 128;
#pragma unroll
        for (int c = 0; c < C::KCH; ++c) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint4 kw = *reinterpret_cast<const uint4 *>(krow + c * C::CHUNK + ((u ^ (lane & 7)) << 4));
                float kf[8];
                bf16x2_to_f32(kw.x, kf[0], kf[1]);
                bf16x2_to_f32(kw.y, kf[2], kf[3]);
                bf16x2_to_f32(kw.z, kf[4], kf[5]);
                bf16x2_to_f32(kw.w, kf[6], kf[7]);
#pragma unroll
                for (int r = 0; r < TQM; ++r) {
                    if (TQ == 1 || r < a.Tq) {
                        const float4 *qr = reinterpret_cast<const float4 *>(qs + r * D + c * 64 + u * 8);
                        const float4 qa = qr[0], qb = qr[1];
                        // packed fp32x2 FMAs on (even, odd) features: the pair (s, s2) is summed
                        // after the row
                        ffma2(s[r], s2[r], qa.x, qa.y, kf[0], kf[1], s[r], s2[r]);
                        ffma2(s[r], s2[r], qa.z, qa.w, kf[2], kf[3], s[r], s2[r]);
                        ffma2(s[r], s2[r], qb.x, qb.y, kf[4], kf[5], s[r], s2[r]);
                        ffma2(s[r], s2[r], qb.z, qb.w, kf[6], kf[7], s[r], s2[r]);
                    }
                }
            }
        }
        // online softmax over the tile's 32 keys, per row; s[r] becomes this lane's P
#pragma unroll
        for (int r = 0; r < TQM; ++r) {
            if (TQ == 1 || r < a.Tq) {
                s[r] += s2[r];
                const bool valid = key < a.Tk && (!a.causal || key <= r + a.Tk - a.Tq);
                const float sv = valid ? s[r] : -INFINITY;
                const float mn = fmaxf(m[r], warp_max(sv));
                // m = -inf: nothing seen yet, l and O~ are 0 (and stay so if mn is -inf too)
                const float alpha = (m[r] == mn) ? 1.f : ex2_approx((m[r] - mn) * sl2);
                const float p = valid ? ex2_approx((sv - mn) * sl2) : 0.f;
                l[r] = l[r] * alpha + p;
#pragma unroll
                for (int e = 0; e < FPL; ++e)
                    o[r][e] *= alpha;
                m[r] = mn;
                s[r] = p;
            }
        }
        // P V: lane = features; V row j read with the swizzle
#pragma unroll 4
        for (int j = 0; j < DBK; ++j) {
            const uint8_t *vp = st + C::TILE + vch * C::CHUNK + j * 128 +
                                ((((vbyte >> 4) ^ (j & 7)) << 4) | (vbyte & 15));
            float vf[FPL];
            if constexpr (FPL == 2) {
                bf16x2_to_f32(*reinterpret_cast<const uint32_t *>(vp), vf[0], vf[1]);
            } else if constexpr (FPL == 4) {
                const uint2 w = *reinterpret_cast<const uint2 *>(vp);
                bf16x2_to_f32(w.x, vf[0], vf[1]);
                bf16x2_to_f32(w.y, vf[2], vf[3]);
            } else {
                const uint4 w = *reinterpret_cast<const uint4 *>(vp);
                bf16x2_to_f32(w.x, vf[0], vf[1]);
                bf16x2_to_f32(w.y, vf[2], vf[3]);
                bf16x2_to_f32(w.z, vf[4], vf[5]);
                bf16x2_to_f32(w.w, vf[6], vf[7]);
            }
#pragma unroll
            for (int r = 0; r < TQM; ++r) {
                if (TQ == 1 || r < a.Tq) {
                    const float pj = __shfl_sync(0xffffffffu, s[r], j);
#pragma unroll
                    for (int e = 0; e < FPL; e += 2)
                        ffma2(o[r][e], o[r][e + 1], pj, pj, vf[e], vf[e + 1], o[r][e], o[r][e + 1]);
                }
            }
        }
        __syncwarp();   // every lane is done with this stage before it is refilled
        if (lane == 0 && k + C::DNS < nt)
            issue(k + C::DNS);
    }
    if (!ok) {
        // copies already issued land before the CTA exits
        if (lane == 0)
            for (int kk = k; kk < nt && kk < k + C::DNS; ++kk)
                mbar_wait_drain(bar0 + 8u * (uint32_t)(kk % C::DNS), (uint32_t)(kk / C::DNS) & 1u);
        return;
    }
#pragma unroll
    for (int r = 0; r < TQM; ++r) {
        if (TQ == 1 || r < a.Tq) {
            const float lsum = warp_sum(l[r]);
            float *pr = a.part + (((size_t)bh * a.nsplit + sp) * a.Tq + r) * (D + 2);
#pragma unroll
            for (int e = 0; e < FPL; ++e)
                pr[f0 + e] = o[r][e];
            if (lane == 0) {
                pr[D] = m[r];
                pr[D + 1] = lsum;
            }
        }
    }
}

}  // namespace

// Chunks per head for these sizes: about 2048 CTAs in all, at least 8 tiles a
// chunk where the keys allow it, and no empty chunk.
void decode_split(int BH, int Tk, int *nsplit, int *tps)
{
    const int ntiles = (Tk + DBK - 1) / DBK;
    if (ntiles == 0 || BH == 0) {
        *nsplit = 0;
        *tps = 0;
        return;
    }
    int ns = (2048 + BH - 1) / BH;
    const int cap = ntiles / 8 > 1 ? ntiles / 8 : 1;
    ns = ns < cap ? ns : cap;
    const int t = (ntiles + ns - 1) / ns;
    *tps = t;
    *nsplit = (ntiles + t - 1) / t;
}

size_t decode_workspace_bytes(int BH, int Tq, int Tk, int d)
{
    int ns, t;
    decode_split(BH, Tk, &ns, &t);
    return ((size_t)BH * ns * Tq * (d + 2) * sizeof(float) + 255) / 256 * 256;
}

int decode_max_rows(int d) { return d == 256 ? DecCfg<256>::TQM : DecCfg<128>::TQM; }

namespace {

// Merge of the chunk states of one query row (one warp per row): with m the
// largest chunk maximum, l = sum_s 2^{c log2e (m_s - m)} l_s and
// O = sum_s 2^{c log2e (m_s - m)} O~_s / l; lse = c m + ln l.  A row that saw
// no key (every m_s = -inf) gets O = 0 and lse = -inf.
template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const float *__restrict__ part, __nv_bfloat16 *__restrict__ o,
                                                           float *__restrict__ lse, int BH, int Tq, int nsplit,
                                                           float scale_log2)
{
    constexpr int FPL = D / 32;
    const int lane = threadIdx.x & 31;
    const size_t rows = (size_t)BH * Tq;
    for (size_t gr = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5; gr < rows;
         gr += ((size_t)gridDim.x * blockDim.x) >> 5) {
        const size_t bh = gr / Tq;
        const int r = (int)(gr - bh * Tq);
        const size_t stride = (size_t)Tq * (D + 2);   // between the chunks of one row
        const float *p0 = part + (bh * nsplit * Tq + r) * (size_t)(D + 2);
        float mx = -INFINITY;
        for (int s = lane; s < nsplit; s += 32)
            mx = fmaxf(mx, p0[s * stride + D]);
        mx = warp_max(mx);
        float acc[FPL];
#pragma unroll
        for (int e = 0; e < FPL; ++e)
            acc[e] = 0.f;
        float lsum = 0.f;
        if (mx != -INFINITY) {
            for (int s = 0; s < nsplit; ++s) {
                const float *ps = p0 + s * stride;
                const float ms = ps[D];
                if (ms == -INFINITY)
                    continue;
                const float w = ex2_approx((ms - mx) * scale_log2);
                lsum = fmaf(w, ps[D + 1], lsum);
#pragma unroll
                for (int e = 0; e < FPL; ++e)
                    acc[e] = fmaf(w, ps[lane * FPL + e], acc[e]);
            }
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        __nv_bfloat16 *dst = o + gr * D + lane * FPL;
#pragma unroll
        for (int e = 0; e < FPL; e += 2)
            *reinterpret_cast<uint32_t *>(dst + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
        if (lane == 0)
            lse[gr] = lsum > 0.f ? (mx * scale_log2 + log2f(lsum)) * 0.69314718055994530942f : -INFINITY;
    }
}

template <int D, int TQ>
int launch_decode_split(const CUtensorMap &tk, const CUtensorMap &tv, const DecArgs &a, int grid, cudaStream_t s)
{
    using C = DecCfg<D, TQ>;
    if (cudaFuncSetAttribute(decode_kernel<D, TQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
        return ERR_CUDA;
    decode_kernel<D, TQ><<<grid, 32, C::SMEM, s>>>(tk, tv, a);
    return cudaGetLastError() == cudaSuccess ? OK : ERR_CUDA;
}

template <int D>
int launch_decode(const void *q, const void *k, const void *v, void *o, float *lse, int BH, int Tq, int Tk,
                  int causal, float scale, void *workspace, cudaStream_t s)
{
    using C = DecCfg<D>;
    if (Tq > C::TQM)
        return ERR_UNSUPPORTED;
    int ns, tps;
    decode_split(BH, Tk, &ns, &tps);
    float *part = static_cast<float *>(workspace);
    const float sl2 = scale * 1.4426950408889634f;
    if (ns > 0) {
        CUtensorMap tk, tv;
        int st = encode_tmap_3d(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Tk, BH, 64, DBK);
        if (st == OK)
            st = encode_tmap_3d(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Tk, BH, 64, DBK);
        if (st != OK)
            return st;
        DecArgs a;
        a.q = static_cast<const __nv_bfloat16 *>(q);
        a.part = part;
        a.BH = BH;
        a.Tq = Tq;
        a.Tk = Tk;
        a.causal = causal;
        a.scale_log2 = sl2;
        a.nsplit = ns;
        a.tps = tps;
        a.timeout_ns = wait_timeout_ns();
        const int grid = BH * ns;
        if (Tq == 1)
            st = launch_decode_split<D, 1>(tk, tv, a, grid, s);
        else if (Tq == 2)
            st = launch_decode_split<D, 2>(tk, tv, a, grid, s);
        else if (Tq <= 4)
            st = launch_decode_split<D, 4>(tk, tv, a, grid, s);
        else if (Tq <= 8 || D == 256)
            st = launch_decode_split<D, 8>(tk, tv, a, grid, s);
        else
            st = launch_decode_split<D, (D == 256 ? 8 : 16)>(tk, tv, a, grid, s);
        if (st != OK)
            return st;
    }
    const size_t rows = (size_t)BH * Tq;
    const size_t blocks = (rows + 7) / 8;
    const int sms = device_sm_count();
    const int grid = (int)(blocks < (size_t)sms * 16 ? blocks : (size_t)sms * 16);
    decode_merge_kernel<D><<<grid, 256, 0, s>>>(part, static_cast<__nv_bfloat16 *>(o), lse, BH, Tq, ns, sl2);
    if (cudaGetLastError() != cudaSuccess)
        return ERR_CUDA;
    return OK;
}

}  // namespace

int decode_launch(const void *q, const void *k, const void *v, void *o, float *lse, int BH, int Tq, int Tk, int d,
                  int causal, float scale, void *workspace, cudaStream_t s)
{
    switch (d) {
    case 64:
        return launch_decode<64>(q, k, v, o, lse, BH, Tq, Tk, causal, scale, workspace, s);
    case 128:
        return launch_decode<128>(q, k, v, o, lse, BH, Tq, Tk, causal, scale, workspace, s);
    case 256:
        return launch_decode<256>(q, k, v, o, lse, BH, Tq, Tk, causal, scale, workspace, s);
    default:
        return ERR_UNSUPPORTED;
    }
}

int dec_status_fetch_clear(cudaStream_t s, int *host_word)
{
    int zero = 0;
    if (cudaMemcpyFromSymbolAsync(host_word, g_dec_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_dec_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return ERR_CUDA;
    return OK;
}

}  // namespace fa
