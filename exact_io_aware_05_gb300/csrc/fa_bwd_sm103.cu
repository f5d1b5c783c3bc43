// fa_bwd_sm103.cu -- backward pass of IO-aware exact attention on sm_103a.
//
// What it computes (zerotofrontier.app "FlashAttention", Efficient attention
// 12.3, section "The backward pass, derived"), with c the softmax scale:
//   preprocess   D_r = dO_r . O_r                       (observation 2)
//   per tile     P_ij = exp(c S_ij - lse_i)             (observation 1, S_ij = Q_i K_j^T)
//                dV_j += P_ij^T dO_i,  dP_ij = dO_i V_j^T,  dS_ij = P_ij o (dP_ij - D_i)
//                dK_j += c dS_ij^T Q_i,  dQ_i += c dS_ij K_j      (observation 3)
// with the key blocks outside: dK_j and dV_j accumulate on chip and are
// written once, dQ_i is accumulated in HBM by fp32 reduce-additions ("Which
// loop goes outside?").  Causal tiles wholly above the diagonal are skipped,
// exactly as in the forward pass.  Five tile products per tile ("The price of
// recomputation").
//
// GB300 design:
//   * three kernels on one stream: bwd_pre (-D, -lse in log2 units, dQ
//     accumulator zeroed), bwd_main (the tile loop below), bwd_dq (scale and
//     round dQ);
//   * bwd_main is persistent; a unit is one 128-key block of one head; units are
//     ordered longest-first within groups of heads and dealt to the CTAs in snake
//     order (passes alternate direction); query blocks are 128 rows, so every
//     product is a full M128 x N128 (d = 128) tensor-core instruction;
//   * warp 0 streams K_j, V_j once per unit and Q_i, dO_i per query block
//     through a ring of stages (TMA); warp 1 issues all tcgen05.mma; warp 2
//     stages each block's lse and D (bulk copies); two softmax warpgroups each
//     rebuild half of a block's P^T and dS^T from S^T and dP^T in tensor
//     memory; a fourth warpgroup drains dQ from tensor memory into the fp32
//     accumulator through shared memory with bulk reduce-adds (TMA) and
//     writes dK, dV at the end of the unit;
//   * tensor memory (512 columns): S^T, dP^T (128 keys x 128 queries) and the
//     dV, dK accumulators.  For d = 128 dQ is formed transposed
//     (dQ^T = K_j^T dS^T, M = d) in the dP^T columns once the softmax has
//     read dP^T from them; for d = 64, dQ = dS K_j has two buffers of its own;
//   * every MMA that overwrites a tensor-memory region waits for the MMA (or
//     the drain) that last read it, and every wait is bounded.
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {

__device__ int g_bwd_status;   // device status word of the backward kernels

namespace {

constexpr int BK = 128;   // keys per unit (= MMA M for S^T, dP^T, dV, dK)
constexpr int BQ = 128;   // queries per block (= N of S^T, dP^T; K of dV, dK)

template <int D>
struct BwdLayout {
    // d = 128: dQ^T = K_j^T dS^T (M = d) takes the dP^T columns of tensor memory once the
    // softmax has read dP^T, so that S^T, dP^T, dV and dK (4 x 128 columns) fit;
    // d = 64: dQ = dS K_j has two buffers of its own.
    static constexpr bool DQ_ALIAS = (D == 128);
    static constexpr int KCH = D / 64;
    static constexpr int KV_CHUNK = BK * 128;            // one 64-column chunk of K_j or V_j
    static constexpr int KV_TILE = KCH * KV_CHUNK;
    static constexpr int Q_CHUNK = BQ * 128;
    static constexpr int Q_TILE = KCH * Q_CHUNK;
    // d = 128: dQ^T leaves through shared memory as bulk reduce-adds (TMA), staged in two
    // 16 KB buffers; to make room, dO has one buffer of its own and only Q is staged
    // ahead.  d = 64: Q and dO share each stage; each drain warp stages its own dQ rows.
    static constexpr bool BULK = DQ_ALIAS;
    static constexpr int NST = D == 128 ? 2 : 3;          // Q (and dO) stages
    static constexpr int ST_Q = 0, ST_DO = BULK ? 0 : Q_TILE, ST_BYTES = BULK ? Q_TILE : 2 * Q_TILE;
    static constexpr int DS_CHUNK = BK * 128;            // dS^T: 128 keys x 64 queries bf16
    static constexpr int DS_TILE = (BQ / 64) * DS_CHUNK;
    static constexpr int NDS = DQ_ALIAS ? 1 : 2;         // dS^T buffers in shared memory
    static constexpr int OFF_K = 0, OFF_V = KV_TILE, OFF_ST = 2 * KV_TILE;
    static constexpr int OFF_DO = OFF_ST + NST * ST_BYTES;   // BULK: the dO buffer
    static constexpr int OFF_DS = OFF_DO + (BULK ? Q_TILE : 0);
    // dQ of 32 queries (fp32) per staging buffer: d = 128, two buffers the drain warpgroup
    // shares; d = 64, one per drain warp (a warp's TMEM lanes are 32 queries)
    static constexpr int STG_BYTES = 32 * D * 4;
    static constexpr int NSTG = BULK ? 2 : 4;
    static constexpr int OFF_STG = OFF_DS + NDS * DS_TILE;
    static constexpr int OFF_LSE = OFF_STG + NSTG * STG_BYTES;   // -lse log2(e) of the current block
    static constexpr int OFF_DEL = OFF_LSE + BQ * 4;          // -D of the current block
    static constexpr int OFF_BAR = OFF_DEL + BQ * 4;
    enum : int {
        B_KVFULL = 0, B_KVEMPTY, B_STFULL, B_STEMPTY = B_STFULL + NST, B_SFULL = B_STEMPTY + NST,
        B_DPFULL, B_PFULL, B_DSFULL, B_DVDONE, B_DQFULL, B_DQEMPTY = B_DQFULL + 2, B_DKVFULL = B_DQEMPTY + 2,
        B_DKVEMPTY, B_LFULL, B_DFULL, B_DRAIN, B_DOFULL, B_DOEMPTY, NBAR
    };
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    // tensor memory columns
    static constexpr int T_S = 0, T_DP = BQ, T_DV = 2 * BQ, T_DK = 2 * BQ + D;
    static constexpr int T_DQ = DQ_ALIAS ? T_DP : T_DK + D;
    static constexpr int DQ_COLS = DQ_ALIAS ? BQ : D;
    static constexpr int TMEM_COLS = 512;
    static_assert(T_DK + D <= TMEM_COLS && T_DQ + (DQ_ALIAS ? 1 : 2) * DQ_COLS <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static constexpr int NTHREADS = 512;
    static constexpr uint32_t ID_SDP = idesc_bf16_f32(128, BQ, false, false);   // K_j Q_i^T, V_j dO_i^T
    static constexpr uint32_t ID_DKV = idesc_bf16_f32(128, D, false, true);     // P^T dO_i, dS^T Q_i
    static constexpr uint32_t ID_DQ = DQ_ALIAS ? idesc_bf16_f32(128, BQ, true, true)   // K_j^T dS^T
                                               : idesc_bf16_f32(128, D, true, true);   // dS K_j
};

enum WaitSite : int {
    SITE_P_KVEMPTY = 1, SITE_P_STEMPTY, SITE_M_KVFULL, SITE_M_STFULL, SITE_M_DVDONE, SITE_M_DSFULL,
    SITE_M_DPDV, SITE_M_DQEMPTY, SITE_S_SFULL, SITE_S_DPFULL, SITE_D_DQFULL, SITE_D_DKVFULL, SITE_L_PFULL,
    SITE_L_DSFULL, SITE_S_LFULL, SITE_S_DFULL
};

struct BwdArgs {
    const float *nlse2, *ndelta;   // -lse * log2(e) and -D per (padded) query row
    float *dq_acc;
    __nv_bfloat16 *dk, *dv;
    int BH, Tq, Tk, Tq_pad, causal;
    float scale, scale_log2;
    int nkb, units, group;
    uint64_t timeout_ns;
    int withhold;           // test-only build: the arrive this launch leaves out (else 0, unused)
    const int *det_bound;   // deterministic mode: per 128-row query block, bound on |dq_acc| (else null)
    // masked instance: allowed keys of row r are r + Tk - Tq - left .. r + Tk - Tq + right
    // (-1: unbounded side), in 128 x 128 blocks marked by bmask ([heads][nqbm][nkbm] or null)
    int left, right;
    const uint8_t *bmask;
    int bm_per_head, nqbm, nkbm;
};

// Deterministic mode.  dQ_i is a sum over key blocks whose terms arrive in any
// order; held as int32 fixed point their sum is the same in every order.  The
// fixed point of query block i is 2^(30 - e) with 2^e above a bound on every
// partial sum: |sum_l dS_rl K_lc| <= max_l |K_lc| sum_l P_rl |dP_rl - D_r|
// <= 2 |dO_r|_2 max_l |V_l|_2 max_lc |K_lc|, since the P_rl sum to 1 and
// |dP_rl|, |D_r| <= |dO_r|_2 max_l |V_l|_2.  The bound's factor-2 headroom
// below 2^31 absorbs the rounding of each term.
__device__ __forceinline__ float det_block_scale(int bound_bits)
{
    const float B = __int_as_float(bound_bits);
    if (!(B <= 3.0e38f))
        return 0.f;                       // non-finite inputs: no meaningful fixed point
    int e;
    frexpf(B, &e);                        // B < 2^e (e = 0 for B = 0)
    return ldexpf(1.f, 30 - max(e, -96));
}

struct Unit {
    int bh, j;     // head, key block
    int i0, nq;    // first query block, number of query blocks visited
    int i1;        // last query block visited
    const uint8_t *bm;   // masked instance: the key block's mask column (stride nkbm), or null
};

// The first query block at or after i that unit x visits (i1 + 1 if none).
__device__ __forceinline__ int unit_next(const Unit &x, int i, int nkbm)
{
    while (i <= x.i1 && x.bm && !x.bm[(size_t)i * nkbm])
        ++i;
    return i;
}

// MASKED = false: causal or not, every unit visits a contiguous run of query blocks.
template <bool MASKED>
__device__ __forceinline__ Unit make_unit(int u, const BwdArgs &a)
{
    const int per_group = a.group * a.nkb;
    const int g = u / per_group;
    const int w = u - g * per_group;
    const int heads_here = min(a.group, a.BH - g * a.group);
    const int lvl = w / heads_here;            // key block: smaller blocks see more queries (causal)
    Unit x;
    x.bh = g * a.group + (w - lvl * heads_here);
    x.j = lvl;
    const int nqb = (a.Tq + BQ - 1) / BQ;
    int first_row = 0;
    if (a.causal) {
        const long r = (long)x.j * BK - (a.Tk - a.Tq);   // first query that sees key j*BK
        first_row = r < 0 ? 0 : (int)min(r, (long)a.Tq);
    }
    x.i0 = first_row / BQ;
    x.nq = nqb - x.i0;
    if (x.nq < 0)
        x.nq = 0;
    x.i1 = x.i0 + x.nq - 1;
    x.bm = nullptr;
    if constexpr (MASKED) {
        // rows that see some key of the block: r >= first key - off - right (right bound),
        // r <= last key - off + left (left bound); then the block mask's column
        const long off = (long)a.Tk - a.Tq;
        const long kf = (long)x.j * BK, kl = min((long)a.Tk - 1, kf + BK - 1);
        const long rlo = a.right >= 0 ? max(0L, kf - off - a.right) : 0L;
        const long rhi = a.left >= 0 ? min((long)a.Tq - 1, kl - off + a.left) : (long)a.Tq - 1;
        if (rlo > rhi) {
            x.nq = 0;
            x.i1 = x.i0 - 1;
            return x;
        }
        x.i0 = (int)(rlo / BQ);
        x.i1 = (int)(rhi / BQ);
        if (a.bmask) {
            x.bm = a.bmask + (size_t)(a.bm_per_head ? x.bh : 0) * a.nqbm * a.nkbm + x.j;
            // count with i1 still the window's last block; then narrow it to the last marked one
            int n = 0, last = x.i0 - 1;
            x.i0 = unit_next(x, x.i0, a.nkbm);
            for (int i = x.i0; i <= x.i1; i = unit_next(x, i + 1, a.nkbm)) {
                ++n;
                last = i;
            }
            x.nq = n;
            x.i1 = last;
        } else {
            x.nq = x.i1 - x.i0 + 1;
        }
    }
    return x;
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most one bulk group of this thread still reading shared memory
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// no bulk group of this thread still reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every bulk group of this thread complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// A-operand column (P^T, bf16 pairs) of K-step kk: each softmax warpgroup packs its 64
// query columns at the start of its own 64-column half of the S^T region.
__device__ __forceinline__ uint32_t half_packed_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

// P = exp2(c log2(e) S - lse log2(e)) for 32 query columns of one key row, in place.
template <bool MASK>
__device__ __forceinline__ void softmax_p32(uint32_t (&sv)[32], const float4 *nl4, float sl2, int q0, int qmin,
                                            int qmax)
{
#pragma unroll
    for (int e4 = 0; e4 < 8; ++e4) {
        const float4 lz = nl4[e4];
        float p0, p1, p2, p3;
        ffma2(p0, p1, __uint_as_float(sv[4 * e4]), __uint_as_float(sv[4 * e4 + 1]), sl2, sl2, lz.x, lz.y);
        ffma2(p2, p3, __uint_as_float(sv[4 * e4 + 2]), __uint_as_float(sv[4 * e4 + 3]), sl2, sl2, lz.z, lz.w);
        p0 = ex2_approx(p0);
        p1 = ex2_approx(p1);
        p2 = ex2_approx(p2);
        p3 = ex2_approx(p3);
        if (MASK) {
            const int q = q0 + 4 * e4;
            p0 = (q >= qmin && q < qmax) ? p0 : 0.f;
            p1 = (q + 1 >= qmin && q + 1 < qmax) ? p1 : 0.f;
            p2 = (q + 2 >= qmin && q + 2 < qmax) ? p2 : 0.f;
            p3 = (q + 3 >= qmin && q + 3 < qmax) ? p3 : 0.f;
        }
        sv[4 * e4] = __float_as_uint(p0);
        sv[4 * e4 + 1] = __float_as_uint(p1);
        sv[4 * e4 + 2] = __float_as_uint(p2);
        sv[4 * e4 + 3] = __float_as_uint(p3);
    }
}

template <int D, bool MASKED>
__global__ void __launch_bounds__(512, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const __grid_constant__ CUtensorMap tm_acc, const BwdArgs a)
{
    using L = BwdLayout<D>;
    constexpr int NST = L::NST;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const uint32_t bar0 = sbase + L::OFF_BAR;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);
    const uint32_t warp = warp_id(), lane = lane_id();

    if (threadIdx.x == 0) {
        mbar_init(bar(L::B_KVFULL), 1);
        mbar_init(bar(L::B_KVEMPTY), 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar(L::B_STFULL + s), 1);
            mbar_init(bar(L::B_STEMPTY + s), 1);
        }
        mbar_init(bar(L::B_SFULL), 1);
        mbar_init(bar(L::B_DPFULL), 1);
        mbar_init(bar(L::B_PFULL), 256);
        mbar_init(bar(L::B_DSFULL), 256);
        mbar_init(bar(L::B_DVDONE), 1);
        mbar_init(bar(L::B_DOFULL), 1);
        mbar_init(bar(L::B_DOEMPTY), 1);   // dP and dV of the block have read dO
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::B_DQFULL + b), 1);
            mbar_init(bar(L::B_DQEMPTY + b), 128);
        }
        mbar_init(bar(L::B_DKVFULL), 1);
        mbar_init(bar(L::B_DKVEMPTY), 128);
        mbar_init(bar(L::B_LFULL), 1);
        mbar_init(bar(L::B_DFULL), 1);
        mbar_init(bar(L::B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_dk);
        tma_prefetch_desc(&tm_dv);
        tma_prefetch_desc(&tm_acc);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx ctx{abort_flag, &g_bwd_status, a.timeout_ns};

    // Register split (launch: 512 threads x 128): the producer/MMA/loader warpgroup gives
    // 32 per thread to the drain warpgroup, which holds a whole dQ^T tile (128 values per
    // thread) so that it can return the tensor-memory columns before it adds them.
    // 96 + 128 + 128 + 160 = 4 x 128.
    if (warp < 4) {
        regs_dealloc<96>();
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------------- producer
            const uint64_t pol_keep = policy_evict_last();
            uint32_t n_kv = 0, n_st = 0, n_do = 0;   // K/V, stage (Q, and dO unless BULK) and BULK dO loads issued
            bool ok = true;
            for (int pass = 0, u = snake_unit<!MASKED>(0); u < a.units && ok; u = snake_unit<!MASKED>(++pass)) {
                const Unit x = make_unit<MASKED>(u, a);
                if (x.nq == 0)
                    continue;
                if (n_kv > 0 && !mbar_wait<true>(bar(L::B_KVEMPTY), (n_kv - 1) & 1, ctx, SITE_P_KVEMPTY))
                    break;
                mbar_arrive_expect_tx(bar(L::B_KVFULL), 2 * L::KV_TILE);
                for (int c = 0; c < L::KCH; ++c) {
                    tma_load_3d(sbase + L::OFF_K + c * L::KV_CHUNK, &tm_k, bar(L::B_KVFULL), c * 64, x.j * BK, x.bh);
                    tma_load_3d(sbase + L::OFF_V + c * L::KV_CHUNK, &tm_v, bar(L::B_KVFULL), c * 64, x.j * BK, x.bh);
                }
                ++n_kv;
                for (int k = 0, i = x.i0; k < x.nq; ++k, i = MASKED ? unit_next(x, i + 1, a.nkbm) : i + 1) {
                    const uint32_t s = n_st % NST;
                    if (n_st >= NST && !mbar_wait<true>(bar(L::B_STEMPTY + s), ((n_st / NST) - 1) & 1, ctx, SITE_P_STEMPTY)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sbase + L::OFF_ST + s * L::ST_BYTES;
                    mbar_arrive_expect_tx(bar(L::B_STFULL + s), (L::BULK ? 1 : 2) * L::Q_TILE);
                    for (int c = 0; c < L::KCH; ++c) {
                        tma_load_3d_hint(st + L::ST_Q + c * L::Q_CHUNK, &tm_q, bar(L::B_STFULL + s), c * 64, i * BQ,
                                         x.bh, pol_keep);
                        if constexpr (!L::BULK)
                            tma_load_3d_hint(st + L::ST_DO + c * L::Q_CHUNK, &tm_do, bar(L::B_STFULL + s), c * 64,
                                             i * BQ, x.bh, pol_keep);
                    }
                    ++n_st;   // counted as soon as issued: the drain below waits for every issued copy
                    if constexpr (L::BULK) {
                        // dO of this block: its one buffer is free once dP and dV of the previous
                        // block, its readers, have completed
                        if (n_do > 0 && !mbar_wait<true>(bar(L::B_DOEMPTY), (n_do - 1) & 1, ctx, SITE_P_STEMPTY)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar(L::B_DOFULL), L::Q_TILE);
                        for (int c = 0; c < L::KCH; ++c)
                            tma_load_3d_hint(sbase + L::OFF_DO + c * L::Q_CHUNK, &tm_do, bar(L::B_DOFULL), c * 64,
                                             i * BQ, x.bh, pol_keep);
                        ++n_do;
                    }
                }
            }
            // drain copies in flight
            const uint32_t lo = n_st > (uint32_t)NST ? n_st - NST : 0;
            for (uint32_t i = lo; i < n_st; ++i)
                mbar_wait_drain(bar(L::B_STFULL + i % NST), (i / NST) & 1);
            if (L::BULK && n_do > 0)
                mbar_wait_drain(bar(L::B_DOFULL), (n_do - 1) & 1);
            if (n_kv > 0)
                mbar_wait_drain(bar(L::B_KVFULL), (n_kv - 1) & 1);
        } else if (warp == 1) {
            // -------------------------------------------------------- MMA issuer
        // Per block g the tensor core runs dP(g) dV(g) S(g+1) dQ(g) dK(g): dP first (its inputs
        // are ready earliest), dV once the softmax's P phase is done, S of the next block as
        // soon as dV(g) frees its columns so that the next softmax starts early, and dQ right
        // after the softmax's dS phase so that its drain starts early.  dS(g) in shared memory
        // is rewritten by the softmax of a later block only after dP of that block has
        // completed, and dP is issued after dK(g) and dQ(g), so the softmax's wait on dP also
        // covers that hazard.
        // The whole warp runs this loop, which keeps the descriptor arithmetic warp-uniform and
        // measured faster than one thread alone; lane 0 issues each group of MMAs and its
        // commit (a commit tracks the MMAs of its own thread).  Every lane waits on its own:
        // outcomes differ only when a wait gives up, no warp-collective operation runs in the
        // loop, and lanes that leave it at different points meet at the __syncwarp below.
            uint32_t g = 0, nu = 0;   // global query-block and unit counters of this CTA
            bool ok = true;
            const uint32_t k_s = sbase + L::OFF_K, v_s = sbase + L::OFF_V;
            const uint64_t kd_k = sdesc_sw128(k_s, 16, 1024), vd_k = sdesc_sw128(v_s, 16, 1024);
            const uint64_t kd_mn = sdesc_sw128(k_s, L::KV_CHUNK, 1024);
            auto stage_addr = [&](uint32_t gq) { return sbase + L::OFF_ST + (gq % NST) * L::ST_BYTES; };
            auto ds_addr = [&](uint32_t gq) { return sbase + L::OFF_DS + (L::NDS == 1 ? 0u : (gq & 1u)) * L::DS_TILE; };
            auto wait = [&](uint32_t b, uint32_t parity, int site) { return mbar_wait<true>(b, parity, ctx, site); };
            // S^T(gq) = K_j Q^T: waits for its stage and for dV(gq-1), the last reader of P^T
            auto issue_s = [&](uint32_t gq) -> bool {
                if (!wait(bar(L::B_STFULL + gq % NST), (gq / NST) & 1, SITE_M_STFULL))
                    return false;
                if (gq > 0 && !wait(bar(L::B_DVDONE), (gq - 1) & 1, SITE_M_DVDONE))
                    return false;
                tc_fence_after();
                const uint64_t qd_k = sdesc_sw128(stage_addr(gq) + L::ST_Q, 16, 1024);
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t ka = (uint64_t)(((kk >> 2) * L::KV_CHUNK + (kk & 3) * 32) >> 4);
                        const uint64_t qa = (uint64_t)(((kk >> 2) * L::Q_CHUNK + (kk & 3) * 32) >> 4);
                        mma_ss(tmem + L::T_S, kd_k + ka, qd_k + qa, L::ID_SDP, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar(L::B_SFULL));
                }
                return true;
            };
            for (int pass = 0, u = snake_unit<!MASKED>(0); u < a.units && ok; u = snake_unit<!MASKED>(++pass)) {
                const Unit x = make_unit<MASKED>(u, a);
                if (x.nq == 0)
                    continue;
                if (!wait(bar(L::B_KVFULL), nu & 1, SITE_M_KVFULL) || !issue_s(g))
                    break;
                for (int i = 0; i < x.nq; ++i, ++g) {
                    const uint32_t st = stage_addr(g);
                    const uint32_t dos = L::BULK ? sbase + L::OFF_DO : st + L::ST_DO;   // dO(g)
                    const uint64_t dod_k = sdesc_sw128(dos, 16, 1024);
                    const uint64_t qd_mn = sdesc_sw128(st + L::ST_Q, L::Q_CHUNK, 1024);
                    const uint64_t dod_mn = sdesc_sw128(dos, L::Q_CHUNK, 1024);
                    // dP^T(g) = V_j dO^T, once dO(g) has landed (BULK: its own buffer) and, for
                    // d = 128, into the columns of dQ^T(g-1) after its drain has read them
                    if ((L::BULK && !wait(bar(L::B_DOFULL), g & 1, SITE_M_DPDV)) ||
                        (L::DQ_ALIAS && g > 0 && !wait(bar(L::B_DQEMPTY), (g - 1) & 1, SITE_M_DQEMPTY))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t ka = (uint64_t)(((kk >> 2) * L::KV_CHUNK + (kk & 3) * 32) >> 4);
                            const uint64_t qa = (uint64_t)(((kk >> 2) * L::Q_CHUNK + (kk & 3) * 32) >> 4);
                            mma_ss(tmem + L::T_DP, vd_k + ka, dod_k + qa, L::ID_SDP, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(bar(L::B_DPFULL));
                    }
                    // dV_j += P^T dO after the softmax's P phase; the first block of a unit
                    // overwrites the accumulator, after the previous unit's epilogue has read it
                    if (!wait(bar(L::B_PFULL), g & 1, SITE_M_DPDV) ||
                        (i == 0 && nu > 0 && !wait(bar(L::B_DKVEMPTY), (nu - 1) & 1, SITE_M_DPDV))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
#pragma unroll
                        for (int kk = 0; kk < BQ / 16; ++kk) {
                            const uint64_t step = (uint64_t)((kk * 2048) >> 4);
                            mma_ts(tmem + L::T_DV, tmem + L::T_S + half_packed_col(kk), dod_mn + step, L::ID_DKV,
                                   (i > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc_commit(bar(L::B_DVDONE));
                        if constexpr (L::BULK)
                            tc_commit(bar(L::B_DOEMPTY));   // dO(g) free: dP(g) and dV(g) complete
                    }
                    // S of the next block as soon as dV(g) has read P^T from its columns, so that
                    // the next P phase can follow this dS phase; then, once dS(g) is in shared
                    // memory, dQ and dK
                    if (i + 1 < x.nq && !issue_s(g + 1)) {
                        ok = false;
                        break;
                    }
                    if (!wait(bar(L::B_DSFULL), g & 1, SITE_M_DSFULL)) {
                        ok = false;
                        break;
                    }
                    const uint32_t b = L::DQ_ALIAS ? 0u : (g & 1u);
                    if (!L::DQ_ALIAS && g >= 2 && !wait(bar(L::B_DQEMPTY + b), ((g - 2) >> 1) & 1, SITE_M_DQEMPTY)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ds = ds_addr(g);
                    const uint64_t dsd_mn = sdesc_sw128(ds, L::DS_CHUNK, 1024);
                    const uint64_t dsd_k = sdesc_sw128(ds, 16, 1024);
                    if (lane == 0) {
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint64_t step = (uint64_t)((kk * 2048) >> 4);
                            if constexpr (L::DQ_ALIAS)
                                mma_ss(tmem + L::T_DQ, kd_mn + step, dsd_mn + step, L::ID_DQ, kk > 0 ? 1u : 0u);
                            else
                                mma_ss(tmem + L::T_DQ + b * L::DQ_COLS, dsd_mn + step, kd_mn + step, L::ID_DQ,
                                       kk > 0 ? 1u : 0u);
                        }
                        tc_commit(bar(L::B_DQFULL + b));
                        // dK_j += dS^T Q  (dS^T from shared memory, K-major; Q MN-major)
#pragma unroll
                        for (int kk = 0; kk < BQ / 16; ++kk) {
                            const uint64_t da = (uint64_t)(((kk >> 2) * L::DS_CHUNK + (kk & 3) * 32) >> 4);
                            const uint64_t step = (uint64_t)((kk * 2048) >> 4);
                            mma_ss(tmem + L::T_DK, dsd_k + da, qd_mn + step, L::ID_DKV, (i > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc_commit(bar(L::B_STEMPTY + g % NST));
                        if (i == x.nq - 1) {
#if FA_TEST_WITHHOLD
                            const bool hold = a.withhold == WITHHOLD_BWD_DKV && blockIdx.x == 0 && nu == 0;
#else
                            constexpr bool hold = false;
#endif
                            if (!hold)
                                tc_commit(bar(L::B_DKVFULL));
                            tc_commit(bar(L::B_KVEMPTY));
                        }
                    }
                }
                ++nu;
            }
            if (lane == 0)
                tc_commit(bar(L::B_DRAIN));
            mbar_wait_drain(bar(L::B_DRAIN), 0);
        } else if (warp == 2 && lane == 0) {
            // -------------------------------------------------------- lse / D loader
            // One buffer each: -lse of block g is loaded once the P phase of block g-1 is
            // done, -D of block g once its dS phase is done.
            uint32_t g = 0;
            bool ok = true;
            for (int pass = 0, u = snake_unit<!MASKED>(0); u < a.units && ok; u = snake_unit<!MASKED>(++pass)) {
                const Unit x = make_unit<MASKED>(u, a);
                for (int i = 0, qi = x.i0; i < x.nq; ++i, ++g, qi = MASKED ? unit_next(x, qi + 1, a.nkbm) : qi + 1) {
                    const size_t roff = (size_t)x.bh * a.Tq_pad + (size_t)qi * BQ;
                    if (g > 0 && !mbar_wait<true>(bar(L::B_PFULL), (g - 1) & 1, ctx, SITE_L_PFULL)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(L::B_LFULL), BQ * 4);
                    bulk_load(sbase + L::OFF_LSE, a.nlse2 + roff, BQ * 4, bar(L::B_LFULL));
                    if (g > 0 && !mbar_wait<true>(bar(L::B_DSFULL), (g - 1) & 1, ctx, SITE_L_DSFULL)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(L::B_DFULL), BQ * 4);
                    bulk_load(sbase + L::OFF_DEL, a.ndelta + roff, BQ * 4, bar(L::B_DFULL));
                }
            }
            // copies in flight: the last phase of each buffer that was started
            if (g > 0) {
                mbar_wait_drain(bar(L::B_LFULL), (g - 1) & 1);
                mbar_wait_drain(bar(L::B_DFULL), (g - 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp < 12) {
        // ------------------------------------------------------------ softmax (two warpgroups)
        const int half = (int)(warp - 4) >> 2;          // query columns [64*half, 64*half + 64)
        const uint32_t quarter = warp & 3u;
        const int key_in_blk = (int)(quarter * 32 + lane);
        const uint32_t lane_base = tmem + ((quarter * 32u) << 16);
        const float sl2 = a.scale_log2;
        uint32_t g = 0;
        bool ok = true;
        for (int pass = 0, u = snake_unit<!MASKED>(0); u < a.units && ok; u = snake_unit<!MASKED>(++pass)) {
            const Unit x = make_unit<MASKED>(u, a);
            const int l = x.j * BK + key_in_blk;         // this thread's key
            for (int i = 0, qi = x.i0; i < x.nq; ++i, ++g, qi = MASKED ? unit_next(x, qi + 1, a.nkbm) : qi + 1) {
                const int qb = qi * BQ + half * 64;   // first query row of this half
                // column q is allowed iff the key exists and (causal) qb + q >= l - (Tk - Tq)
                int qmin = l < a.Tk ? 0 : 64, qmax = 64;   // allowed query columns [qmin, qmax)
                if (a.causal && l < a.Tk) {
                    const long lim = (long)l - (a.Tk - a.Tq) - qb;
                    qmin = (int)max(0L, min(64L, lim));
                }
                if (MASKED && l < a.Tk) {
                    const long off = (long)a.Tk - a.Tq;
                    if (a.right >= 0)
                        qmin = (int)max(0L, min(64L, (long)l - off - a.right - qb));
                    if (a.left >= 0)
                        qmax = (int)max(0L, min(64L, (long)l - off + a.left - qb + 1));
                }
                const bool mask = __any_sync(0xffffffffu, qmin > 0 || qmax < 64);
                if (!mbar_wait_warp(bar(L::B_SFULL), g & 1, ctx, SITE_S_SFULL) ||
                    !mbar_wait_warp(bar(L::B_LFULL), g & 1, ctx, SITE_S_LFULL)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // P phase: P^T (bf16) over the first half of this warpgroup's own S^T columns
                uint32_t p0[32], p1[32];
                tmem_ld_x32_nowait(lane_base + L::T_S + half * 64, p0);
                tmem_ld_x32_nowait(lane_base + L::T_S + half * 64 + 32, p1);
                tmem_wait_ld_x32(p0);
                tmem_wait_ld_x32(p1);
                const float4 *nl4 = reinterpret_cast<const float4 *>(smem + L::OFF_LSE) + half * 16;
                if (mask) {
                    softmax_p32<true>(p0, nl4, sl2, 0, qmin, qmax);
                    softmax_p32<true>(p1, nl4 + 8, sl2, 32, qmin, qmax);
                } else {
                    softmax_p32<false>(p0, nl4, sl2, 0, 0, 64);
                    softmax_p32<false>(p1, nl4 + 8, sl2, 32, 0, 64);
                }
                {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(p0[2 * e]), __uint_as_float(p0[2 * e + 1]));
                    tmem_st_x16(lane_base + L::T_S + half * 64, pk);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(p1[2 * e]), __uint_as_float(p1[2 * e + 1]));
                    tmem_st_x16(lane_base + L::T_S + half * 64 + 16, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(L::B_PFULL));
                // dS phase: dS = P o (dP - D) into shared memory ([key][query], 128-byte
                // swizzle, 64 queries per 128-byte row)
                if (!mbar_wait_warp(bar(L::B_DPFULL), g & 1, ctx, SITE_S_DPFULL) ||
                    !mbar_wait_warp(bar(L::B_DFULL), g & 1, ctx, SITE_S_DFULL)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint8_t *ds_row = smem + L::OFF_DS + (L::NDS == 1 ? 0u : (g & 1)) * L::DS_TILE + half * L::DS_CHUNK +
                                  key_in_blk * 128;
                const float4 *nd4 = reinterpret_cast<const float4 *>(smem + L::OFF_DEL) + half * 16;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t dv[32];
                    tmem_ld_x32(lane_base + L::T_DP + half * 64 + c * 32, dv);
                    const uint32_t(&pc_)[32] = c == 0 ? p0 : p1;
                    uint32_t dk[16];
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 dz = nd4[c * 8 + e4];
                        float t0, t1, t2, t3;
                        fadd2(t0, t1, __uint_as_float(dv[4 * e4]), __uint_as_float(dv[4 * e4 + 1]), dz.x, dz.y);
                        fadd2(t2, t3, __uint_as_float(dv[4 * e4 + 2]), __uint_as_float(dv[4 * e4 + 3]), dz.z, dz.w);
                        fmul2(t0, t1, t0, t1, __uint_as_float(pc_[4 * e4]), __uint_as_float(pc_[4 * e4 + 1]));
                        fmul2(t2, t3, t2, t3, __uint_as_float(pc_[4 * e4 + 2]), __uint_as_float(pc_[4 * e4 + 3]));
                        dk[2 * e4] = pack_bf16x2(t0, t1);
                        dk[2 * e4 + 1] = pack_bf16x2(t2, t3);
                    }
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        const int sw = (c * 4 + v4) ^ (key_in_blk & 7);
                        *reinterpret_cast<uint4 *>(ds_row + sw * 16) =
                            make_uint4(dk[4 * v4], dk[4 * v4 + 1], dk[4 * v4 + 2], dk[4 * v4 + 3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(L::B_DSFULL));
            }
        }
    } else {
        // ------------------------------------------------------------ dQ drain + dK/dV epilogue
        regs_alloc<160>();
        const uint32_t quarter = warp & 3u;
        const int row = (int)(quarter * 32 + lane);      // TMEM lane
        const uint32_t lane_base = tmem + ((quarter * 32u) << 16);
        uint32_t g = 0, nu = 0;
        uint32_t stg_n = 0;                          // dQ boxes this warp has staged (d = 128)
        bool ok = true;
        for (int pass = 0, u = snake_unit<!MASKED>(0); u < a.units && ok; u = snake_unit<!MASKED>(++pass)) {
            const Unit x = make_unit<MASKED>(u, a);
            const int l = x.j * BK + row;
            const size_t krow = (size_t)x.bh * a.Tk + l;
            if (x.nq == 0) {
                if (l < a.Tk) {
                    uint4 *pk_ = reinterpret_cast<uint4 *>(a.dk + krow * D);
                    uint4 *pv_ = reinterpret_cast<uint4 *>(a.dv + krow * D);
                    for (int e = 0; e < D / 8; ++e) {
                        pk_[e] = make_uint4(0, 0, 0, 0);
                        pv_[e] = make_uint4(0, 0, 0, 0);
                    }
                }
                continue;
            }
            for (int i = 0, qi = x.i0; i < x.nq; ++i, ++g, qi = MASKED ? unit_next(x, qi + 1, a.nkbm) : qi + 1) {
                const uint32_t b = L::DQ_ALIAS ? 0u : (g & 1u);
                const uint32_t ph = L::DQ_ALIAS ? (g & 1u) : ((g >> 1) & 1u);
                // one decision for the warp (tensor-memory loads follow)
                const bool got = __all_sync(0xffffffffu, mbar_wait<true>(bar(L::B_DQFULL + b), ph, ctx, SITE_D_DQFULL));
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int qb = qi * BQ;
                const float dsc = a.det_bound ? det_block_scale(a.det_bound[((size_t)x.bh * a.Tq_pad + qb) / BQ]) : 0.f;
                if constexpr (L::DQ_ALIAS) {
                    // lane = feature, column = query.  The whole tile is read into registers
                    // first, so the columns go back to the MMA at once; then four chunks of 32
                    // queries go through shared memory ([query][feature], the accumulator's own
                    // layout: a warp writes 32 consecutive words per query) and the TMA engine
                    // adds each 16 KB chunk into the accumulator, off the load/store path.
                    uint32_t va[32], vb[32], vc[32], vd[32];
                    tmem_ld_x32_nowait(lane_base + L::T_DQ, va);
                    tmem_ld_x32_nowait(lane_base + L::T_DQ + 32, vb);
                    tmem_ld_x32_nowait(lane_base + L::T_DQ + 64, vc);
                    tmem_ld_x32_nowait(lane_base + L::T_DQ + 96, vd);
                    tmem_wait_ld_x32(va);
                    tmem_wait_ld_x32(vb);
                    tmem_wait_ld_x32(vc);
                    tmem_wait_ld_x32(vd);
                    tc_fence_before();
                    mbar_arrive(bar(L::B_DQEMPTY));
                    // Each warp stages its 32 features of a chunk of 32 queries as a 4 KB box
                    // ([query][feature], 128-byte rows: a warp writes one row per instruction) in its
                    // own two buffers and its lane 0 hands the box to the TMA engine as a tensor
                    // reduce-add; the four warps never wait for one another.
                    auto stage_chunk = [&](const uint32_t(&v)[32], int c) {
                        const uint32_t sb = stg_n & 1u;
                        const uint32_t boff = L::OFF_STG + quarter * 8192u + sb * 4096u;
                        if (lane == 0 && stg_n >= 2)
                            bulk_wait_read_1();   // the box two back, in this buffer, has been read
                        __syncwarp();
                        uint32_t *dst = reinterpret_cast<uint32_t *>(smem + boff) + lane;
                        if (a.det_bound) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                dst[e * 32] = (uint32_t)__float2int_rn(__uint_as_float(v[e]) * dsc);
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                dst[e * 32] = v[e];
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_reduce_add_3d(&tm_acc, sbase + boff, (int)quarter * 32, qb + c * 32, x.bh);
                            bulk_commit();
                        }
                        ++stg_n;
                    };
                    stage_chunk(va, 0);
                    stage_chunk(vb, 1);
                    stage_chunk(vc, 2);
                    stage_chunk(vd, 3);
                } else {
                    // lane = query, column = feature: each drain warp holds the 32 queries of its
                    // TMEM lanes and writes them into its own staging buffer as two boxes of 32
                    // queries x 32 features with the 128-byte swizzle (16-byte unit u of row r at
                    // unit u ^ (r mod 8)), so that the 32 lanes' stores of one unit fall in distinct
                    // banks; its lane 0 hands each box to the TMA engine as a tensor reduce-add.
                    // The buffer's previous reduce-adds (one block earlier) have long finished
                    // reading it; lane 0 confirms before the warp writes.
                    uint32_t v[L::DQ_COLS / 32][32];
#pragma unroll
                    for (int c = 0; c < L::DQ_COLS / 32; ++c)
                        tmem_ld_x32_nowait(lane_base + L::T_DQ + b * L::DQ_COLS + c * 32, v[c]);
#pragma unroll
                    for (int c = 0; c < L::DQ_COLS / 32; ++c)
                        tmem_wait_ld_x32(v[c]);
                    tc_fence_before();
                    mbar_arrive(bar(L::B_DQEMPTY + b));
                    if (lane == 0)
                        bulk_wait_read_all();
                    __syncwarp();
                    static_assert(L::DQ_COLS / 32 * 4096 == L::STG_BYTES, "two 4 KB boxes per drain warp");
                    const uint32_t wbox = L::OFF_STG + quarter * L::STG_BYTES;   // 1024-byte aligned
                    uint8_t *srow = smem + wbox + lane * 128;
#pragma unroll
                    for (int c = 0; c < L::DQ_COLS / 32; ++c) {
                        uint32_t w[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            w[e] = a.det_bound ? (uint32_t)__float2int_rn(__uint_as_float(v[c][e]) * dsc) : v[c][e];
#pragma unroll
                        for (int u4 = 0; u4 < 8; ++u4)
                            *reinterpret_cast<uint4 *>(srow + c * 4096 + ((u4 ^ (lane & 7)) << 4)) =
                                make_uint4(w[4 * u4], w[4 * u4 + 1], w[4 * u4 + 2], w[4 * u4 + 3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
#pragma unroll
                        for (int c = 0; c < L::DQ_COLS / 32; ++c)
                            tma_reduce_add_3d(&tm_acc, sbase + wbox + c * 4096, c * 32, qb + (int)quarter * 32, x.bh);
                        bulk_commit();
                    }
                }
            }
            if (!ok)
                break;
            const bool kv_ok = __all_sync(0xffffffffu, mbar_wait<true>(bar(L::B_DKVFULL), nu & 1, ctx, SITE_D_DKVFULL));
            if (!kv_ok)
                break;
            tc_fence_after();
            // dV, then dK (x c): each warp packs its 32 key rows (the TMEM lanes it reads) to bf16
            // into its own 8 KB of shared memory (d = 128: a quarter of the two staging buffers,
            // free once the last dQ chunk has been read; d = 64: the warp's own buffer) as boxes of
            // 32 rows x 64 columns with the 128-byte swizzle, and its lane 0 hands them to the TMA
            // engine as tensor stores (rows past Tk are not written).  This keeps the 64 KB per
            // unit off the load/store path that the softmax of the next unit is using.  Both
            // accumulators are read out of tensor memory first (at d = 128 dK waits in registers
            // while dV is stored), so the next unit's dV and dK may overwrite them at once.
            if (lane == 0)
                bulk_wait_read_all();   // this warp's dQ chunks have been read
            __syncwarp();
            {
                const uint32_t wbuf = sbase + L::OFF_STG + quarter * 8192u;
                uint8_t *wrow = smem + L::OFF_STG + quarter * 8192u + lane * 128;
                // 32 columns (16 bf16 pairs) of this row at column 32c of a 64-column box grid
                auto put = [&](uint8_t *boxes, const uint32_t *w, int c) {
                    uint8_t *box = boxes + (c >> 1) * 4096;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int unit = (c & 1) * 4 + e;
                        *reinterpret_cast<uint4 *>(box + ((unit ^ (lane & 7)) << 4)) =
                            make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                    }
                };
                uint32_t dkp[L::BULK ? D / 2 : 1];   // d = 128: dK of this row, packed
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32], w[16];
                    tmem_ld_x32(lane_base + L::T_DV + c * 32, v);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                    put(wrow, w, c);
                }
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_x32(lane_base + L::T_DK + c * 32, v);
                    if constexpr (L::BULK) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            dkp[c * 16 + e] =
                                pack_bf16x2(__uint_as_float(v[2 * e]) * a.scale, __uint_as_float(v[2 * e + 1]) * a.scale);
                    } else {   // d = 64: dK's box right after dV's
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * a.scale, __uint_as_float(v[2 * e + 1]) * a.scale);
                        put(wrow + 4096, w, c);
                    }
                }
                tc_fence_before();
                mbar_arrive(bar(L::B_DKVEMPTY));   // dV and dK are out of tensor memory
                // a box whose first row is past Tk has nothing to write and is not issued
                const bool rows_here = x.j * BK + (int)quarter * 32 < a.Tk;
                const int y0 = x.j * BK + (int)quarter * 32;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && rows_here) {
                    if constexpr (L::BULK) {
                        tma_store_3d(&tm_dv, wbuf, 0, y0, x.bh);
                        tma_store_3d(&tm_dv, wbuf + 4096, 64, y0, x.bh);
                    } else {
                        tma_store_3d(&tm_dv, wbuf, 0, y0, x.bh);
                        tma_store_3d(&tm_dk, wbuf + 4096, 0, y0, x.bh);
                    }
                    bulk_commit();
                }
                if constexpr (L::BULK) {
                    if (lane == 0)
                        bulk_wait_read_all();   // dV has left the buffer
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c)
                        put(wrow, dkp + c * 16, c);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && rows_here) {
                        tma_store_3d(&tm_dk, wbuf, 0, y0, x.bh);
                        tma_store_3d(&tm_dk, wbuf + 4096, 64, y0, x.bh);
                        bulk_commit();
                    }
                }
                if (lane == 0)
                    bulk_wait_read_all();   // the buffer is free again for the next unit's dQ
                __syncwarp();
            }
            ++nu;
        }
        if (lane == 0)
            bulk_wait_all();   // every reduce-add and store of this warp has completed
    }
    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// Deterministic mode, first: per head the largest |V_l|_2 and |K_lc| (float bits,
// maxima of non-negative values in any order).  One warp per key row.
template <int D>
__global__ void __launch_bounds__(256) bwd_kvmax_kernel(const __nv_bfloat16 *__restrict__ k,
                                                        const __nv_bfloat16 *__restrict__ v, float *__restrict__ kvmax,
                                                        int BH, int Tk)
{
    const size_t rows = (size_t)BH * Tk;
    const int lane = threadIdx.x & 31;
    constexpr int PER = D / 32;
    for (size_t gr = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5; gr < rows;
         gr += ((size_t)gridDim.x * blockDim.x) >> 5) {
        float ss = 0.f, km = 0.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const float vv = __bfloat162float(v[gr * D + lane * PER + e]);
            const float kv = __bfloat162float(k[gr * D + lane * PER + e]);
            ss = fmaf(vv, vv, ss);
            km = fmaxf(km, fabsf(kv));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            ss += __shfl_xor_sync(0xffffffffu, ss, off);
            km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, off));
        }
        if (lane == 0) {
            const size_t bh = gr / Tk;
            atomicMax(reinterpret_cast<int *>(kvmax) + 2 * bh, __float_as_int(sqrtf(ss)));
            atomicMax(reinterpret_cast<int *>(kvmax) + 2 * bh + 1, __float_as_int(km));
        }
    }
}

// -D_r = -(dO_r . O_r) and -lse_r in log2 units (-inf where no key is allowed or
// past Tq), stored negated so that the tile loop adds them; the fp32 dQ
// accumulator zeroed; deterministic mode: the fixed-point bound of each query
// block, max over its rows of 2 |dO_r|_2 max|V|_2 max|K|.  A group of D/8 lanes
// takes a (padded) row, 16 bytes of O and of dO per lane, and every group keeps
// two rows in flight so that enough loads are outstanding to stream HBM.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16 *__restrict__ o,
                                                      const __nv_bfloat16 *__restrict__ dO,
                                                      const float *__restrict__ lse, float *__restrict__ lse2,
                                                      float *__restrict__ delta, float *__restrict__ dq_acc,
                                                      const float *__restrict__ kvmax, int *__restrict__ bound, int BH,
                                                      int Tq, int Tq_pad)
{
    constexpr int G = D / 8;        // lanes per row
    constexpr int RPW = 32 / G;     // rows per warp and pass
    constexpr int U = 2;            // passes in flight
    const size_t rows = (size_t)BH * Tq_pad;
    const int lane = threadIdx.x & 31, gi = lane / G, sub = lane % G;
    const size_t warp = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5;
    const size_t nwarps = ((size_t)gridDim.x * blockDim.x) >> 5;
    // the loop is warp-uniform (whole warps take U * RPW rows), so the shuffles see all lanes
    for (size_t wb = warp * (RPW * U); wb < rows; wb += nwarps * (RPW * U)) {
        uint4 ov[U], gv[U];
        size_t gr[U], bh[U];
        int r[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            gr[k] = wb + (size_t)k * RPW + gi;
            bh[k] = gr[k] / Tq_pad;
            r[k] = (int)(gr[k] - bh[k] * Tq_pad);
            ov[k] = gv[k] = make_uint4(0u, 0u, 0u, 0u);
            if (gr[k] < rows && r[k] < Tq) {
                const size_t src = (bh[k] * Tq + r[k]) * D + sub * 8;
                ov[k] = *reinterpret_cast<const uint4 *>(o + src);
                gv[k] = *reinterpret_cast<const uint4 *>(dO + src);
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            float dsum = 0.f, ss = 0.f;
            const __nv_bfloat162 *o2 = reinterpret_cast<const __nv_bfloat162 *>(&ov[k]);
            const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&gv[k]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 a2 = __bfloat1622float2(o2[e]), b2 = __bfloat1622float2(g2[e]);
                dsum = fmaf(a2.x, b2.x, dsum);
                dsum = fmaf(a2.y, b2.y, dsum);
                ss = fmaf(b2.x, b2.x, ss);
                ss = fmaf(b2.y, b2.y, ss);
            }
#pragma unroll
            for (int off = G / 2; off > 0; off >>= 1) {
                dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
                ss += __shfl_xor_sync(0xffffffffu, ss, off);
            }
            if (gr[k] >= rows)
                continue;
            if (sub == 0) {
                float l2 = -INFINITY;
                if (r[k] < Tq) {
                    const float lv = lse[bh[k] * Tq + r[k]];
                    l2 = (lv == -INFINITY) ? -INFINITY : -lv * 1.4426950408889634f;
                }
                lse2[gr[k]] = l2;
                delta[gr[k]] = r[k] < Tq ? -dsum : 0.f;
                if (bound && r[k] < Tq) {
                    const float bnd = 2.f * sqrtf(ss) * kvmax[2 * bh[k]] * kvmax[2 * bh[k] + 1];
                    atomicMax(bound + (gr[k] >> 7), __float_as_int(bnd));
                }
            }
            float4 *z = reinterpret_cast<float4 *>(dq_acc + gr[k] * D) + sub * 2;
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

// dQ = scale * dq_acc, rounded to bf16.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float *__restrict__ dq_acc, __nv_bfloat16 *__restrict__ dq,
                                                     const int *__restrict__ bound, int BH, int Tq, int Tq_pad,
                                                     float scale)
{
    const size_t n8 = (size_t)BH * Tq * (D / 8);
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
        const size_t row = i / (D / 8);
        const int c8 = (int)(i - row * (D / 8));
        const size_t bh = row / Tq;
        const int r = (int)(row - bh * Tq);
        const float4 *src = reinterpret_cast<const float4 *>(dq_acc + (bh * Tq_pad + r) * D + c8 * 8);
        float4 x0 = src[0], x1 = src[1];
        if (bound) {   // int32 fixed point of the row's query block -> float
            const float sc = det_block_scale(bound[(bh * Tq_pad + r) >> 7]);
            const float inv = sc > 0.f ? 1.f / sc : 0.f;   // a power of two: exact
            const int4 *isrc = reinterpret_cast<const int4 *>(src);
            const int4 i0 = isrc[0], i1 = isrc[1];
            x0 = make_float4((float)i0.x * inv, (float)i0.y * inv, (float)i0.z * inv, (float)i0.w * inv);
            x1 = make_float4((float)i1.x * inv, (float)i1.y * inv, (float)i1.z * inv, (float)i1.w * inv);
        }
        uint4 w;
        w.x = pack_bf16x2(x0.x * scale, x0.y * scale);
        w.y = pack_bf16x2(x0.z * scale, x0.w * scale);
        w.z = pack_bf16x2(x1.x * scale, x1.y * scale);
        w.w = pack_bf16x2(x1.z * scale, x1.w * scale);
        reinterpret_cast<uint4 *>(dq)[i] = w;
    }
}

template <int D>
int launch_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO,
               void *dq, void *dk, void *dv, int BH, int Tq, int Tk, const MaskSpec &mask, float scale,
               const BwdWorkspace &ws, int stages, cudaStream_t s)
{
    const int causal = mask.right == 0 ? 1 : 0;
    const bool masked = mask.left >= 0 || mask.right > 0 || mask.block;
    using L = BwdLayout<D>;
    const int Tq_pad = (int)bwd_row_stride(Tq);
    const int sms = device_sm_count();
    const bool det = (stages & kBwdDeterministic) != 0;
    // 1. preprocess (deterministic mode: the K/V maxima first, for the fixed-point bounds)
    if ((stages & 1) && Tq > 0) {
        const size_t rows = (size_t)BH * Tq_pad;
        if (det) {
            const size_t det_bytes = (size_t)BH * 2 * sizeof(float) + rows / 128 * sizeof(int);
            if (cudaMemsetAsync(ws.kvmax, 0, det_bytes, s) != cudaSuccess)
                return ERR_CUDA;
            if (Tk > 0) {
                const size_t kblocks = ((size_t)BH * Tk + 7) / 8;
                const int kgrid = (int)(kblocks < (size_t)sms * 16 ? kblocks : (size_t)sms * 16);
                bwd_kvmax_kernel<D><<<kgrid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(k),
                                                          static_cast<const __nv_bfloat16 *>(v), ws.kvmax, BH, Tk);
                if (cudaGetLastError() != cudaSuccess)
                    return ERR_CUDA;
            }
        }
        const size_t rows_per_block = 8 * (32 / (D / 8)) * 2;   // 8 warps x rows per warp x passes in flight
        const size_t blocks = (rows + rows_per_block - 1) / rows_per_block;
        const int grid = (int)(blocks < (size_t)sms * 8 ? blocks : (size_t)sms * 8);
        bwd_pre_kernel<D><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(o),
                                               static_cast<const __nv_bfloat16 *>(dO), lse, ws.lse2, ws.delta,
                                               ws.dq_acc, ws.kvmax, det ? ws.bound : nullptr, BH, Tq, Tq_pad);
        if (cudaGetLastError() != cudaSuccess)
            return ERR_CUDA;
    }
    // 2. tile loop
    if ((stages & 2) && Tk > 0) {
        CUtensorMap tq, tk, tv, tdo;
        const int tq_rows = Tq > 0 ? Tq : 1;
        int st = encode_tmap_3d(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Tk, BH, 64, BK);
        if (st == OK)
            st = encode_tmap_3d(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Tk, BH, 64, BK);
        if (st == OK)
            st = encode_tmap_3d(&tq, Tq > 0 ? q : k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, tq_rows, BH, 64, BQ);
        if (st == OK)
            st = encode_tmap_3d(&tdo, Tq > 0 ? dO : k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, tq_rows, BH, 64, BQ);
        // dQ accumulator ([BH][Tq_pad][D], fp32 or, deterministic, int32): each drain warp adds
        // boxes of 32 features x 32 queries, staged plain (d = 128: a warp writes one query's 32
        // features per instruction) or with the 128-byte swizzle (d = 64: a thread writes its
        // query's row)
        CUtensorMap tacc;
        if (st == OK) {
            const CUtensorMapDataType at = det ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
            const uint64_t arows = (uint64_t)(Tq_pad > 0 ? Tq_pad : 1);   // unused when Tq = 0
            st = L::DQ_ALIAS ? encode_tmap_3d_plain(&tacc, ws.dq_acc, at, 4, D, arows, BH, 32, 32)
                             : encode_tmap_3d(&tacc, ws.dq_acc, at, 4, D, arows, BH, 32, 32);
        }
        // dK, dV leave as TMA stores: each drain warp stores its 32 key rows, 64 columns per box
        CUtensorMap tdk, tdv;
        if (st == OK)
            st = encode_tmap_3d(&tdk, dk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Tk, BH, 64, 32);
        if (st == OK)
            st = encode_tmap_3d(&tdv, dv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Tk, BH, 64, 32);
        if (st != OK)
            return st;
        BwdArgs a;
        a.nlse2 = ws.lse2;
        a.ndelta = ws.delta;
        a.dq_acc = ws.dq_acc;
        a.dk = static_cast<__nv_bfloat16 *>(dk);
        a.dv = static_cast<__nv_bfloat16 *>(dv);
        a.BH = BH;
        a.Tq = Tq;
        a.Tk = Tk;
        a.Tq_pad = Tq_pad;
        a.causal = causal;
        a.scale = scale;
        a.scale_log2 = scale * 1.4426950408889634f;
        a.nkb = (Tk + BK - 1) / BK;
        a.units = BH * a.nkb;
        // heads per group: Q, dO, K, V of the group within ~80 MB of L2, a whole number of
        // passes where possible (B8 H32 N4096 d128: 19 heads; measured faster than 12).  The
        // masked instance keeps ~48 MB groups and same-direction passes (measured faster
        // there: its units' lengths do not follow the order).
        const double bytes_head = 2.0 * (Tq + Tk) * D * 2.0;
        int gsz = (int)((masked ? 48.0 : 80.0) * 1024 * 1024 / (bytes_head > 1 ? bytes_head : 1));
        gsz = gsz < 1 ? 1 : (gsz > BH ? BH : gsz);
        a.group = masked ? gsz : grid_aligned_group(gsz, a.nkb, a.units < sms ? a.units : sms);
        a.timeout_ns = wait_timeout_ns();
        a.withhold = WITHHOLD_NONE;
#if FA_TEST_WITHHOLD
        a.withhold = test_withhold_take(WITHHOLD_BWD_DKV, WITHHOLD_BWD_DKV);
#endif
        a.det_bound = det ? ws.bound : nullptr;
        a.left = mask.left;
        a.right = mask.right;
        a.bmask = mask.block;
        a.bm_per_head = mask.per_head;
        a.nqbm = (Tq + 127) / 128;
        a.nkbm = (Tk + 127) / 128;
        auto kernel = masked ? bwd_main_kernel<D, true> : bwd_main_kernel<D, false>;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES) != cudaSuccess)
            return ERR_CUDA;
        const int grid = a.units < sms ? a.units : sms;
        kernel<<<grid, L::NTHREADS, L::SMEM_BYTES, s>>>(tq, tk, tv, tdo, tdk, tdv, tacc, a);
        if (cudaGetLastError() != cudaSuccess)
            return ERR_CUDA;
    }
    // 3. dQ
    if ((stages & 4) && Tq > 0) {
        const size_t n8 = (size_t)BH * Tq * (D / 8);
        const size_t blocks = (n8 + 255) / 256;
        const int grid = (int)(blocks < (size_t)sms * 8 ? blocks : (size_t)sms * 8);
        bwd_dq_kernel<D><<<grid, 256, 0, s>>>(ws.dq_acc, static_cast<__nv_bfloat16 *>(dq), det ? ws.bound : nullptr,
                                              BH, Tq, Tq_pad, scale);
        if (cudaGetLastError() != cudaSuccess)
            return ERR_CUDA;
    }
    return OK;
}

}  // namespace

int bwd_launch(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO, void *dq,
               void *dk, void *dv, int BH, int Tq, int Tk, int d, const MaskSpec &mask, float scale,
               const BwdWorkspace &ws, int stages, cudaStream_t s)
{
    switch (d) {
    case 64:
        return launch_bwd<64>(q, k, v, o, lse, dO, dq, dk, dv, BH, Tq, Tk, mask, scale, ws, stages, s);
    case 128:
        return launch_bwd<128>(q, k, v, o, lse, dO, dq, dk, dv, BH, Tq, Tk, mask, scale, ws, stages, s);
    default:
        return ERR_UNSUPPORTED;
    }
}

int bwd_status_fetch_clear(cudaStream_t s, int *host_word)
{
    int zero = 0;
    if (cudaMemcpyFromSymbolAsync(host_word, g_bwd_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_bwd_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return ERR_CUDA;
    return OK;
}

}  // namespace fa
