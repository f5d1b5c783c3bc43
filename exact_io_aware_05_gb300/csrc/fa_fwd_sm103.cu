// fa_fwd_sm103.cu -- forward pass of IO-aware exact attention on sm_103a.
//
// What it computes (zerotofrontier.app "FlashAttention", Efficient attention
// 12.3, section "The forward pass"): for every query block Q_i of 128 rows,
// stream the key/value blocks K_j, V_j through shared memory and keep per
// row a running maximum m, a running sum l and an unnormalised output O~:
//     S_ij = Q_i K_j^T                    (tcgen05.mma, fp32 in tensor memory)
//     m_new = max(m, rowmax(S_ij))
//     P~ = exp(c S_ij - c m_new)          (exp2 with c*log2(e) folded in)
//     l <- e^{c(m - m_new)} l + rowsum(P~),  O~ <- e^{c(m - m_new)} O~ + P~ V_j
// then write O_i = O~ / l and lse_i = c m + log l once.  Causal tiles wholly
// above the diagonal are never loaded or computed; the skip test compares the
// first key of the block with the last query of the block ("The causal mask,
// and the tiles you never visit").  The N x N matrices S and P never reach
// HBM: S lives in tensor memory; P (bf16) goes to shared memory with two query
// tiles per CTA, or back over S in tensor memory with one, and feeds the second MMA.
//
// GB300 design (differs from the pages' A100/H100 kernels):
//   * persistent CTAs, one per SM, each owning a 256-row unit (two 128-row
//     query tiles, d = 64/128) or a 128-row unit (d = 256); units are ordered
//     longest-first within groups of heads sized so their K/V stay in L2, and
//     dealt to the CTAs in snake order (passes alternate direction);
//   * warp 0: TMA producer (Q once per unit, K/V tiles through an NSLOT-deep
//     ring with full/empty mbarriers);
//   * warps 1 and 2 (two tiles): one thread each issues the tcgen05.mma and
//     commits of its tile, S of key block k+1 ahead of P V of block k (P lives
//     in shared memory, so S may be overwritten once the softmax has read it);
//     with one tile, warp 1 issues the S products and warp 2 the P V products,
//     and the K/V ring holds 16 KB chunks that each product consumes in order;
//   * one 128-thread softmax warpgroup per query tile (thread = query row =
//     tensor-memory lane) doing the online softmax and the epilogue; the two
//     warpgroups run independently;
//   * the running maximum that P~, l and O~ refer to moves only when a row's
//     maximum has grown by more than 2^8 in the exp2 domain (the rescale of
//     O~ in tensor memory is skipped for a warp when none of its 32 rows needs
//     it); O~ / l and lse are the same quantities for any reference maximum,
//     P~ <= 2^8 keeps every sum far from fp32 overflow, and with scores of
//     unit scale the rescale all but disappears after the first key block.
//   * every wait is bounded (see fa_common.cuh); on a timeout the CTA drains
//     its in-flight copies and MMAs, frees tensor memory and returns.
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {

__device__ int g_fwd_status;   // device status word of the forward kernels

namespace {

constexpr int BR = 128;                 // query rows per tile (= MMA M = TMEM lanes)
// O~ and l are rescaled to a new row maximum only once it exceeds the one they refer to
// by more than 2^kRescaleLog2 in the exp2 domain; until then P~ <= 2^kRescaleLog2.
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct FwdCfg;
template <>
struct FwdCfg<64> {
    static constexpr int BC = 128, NQ = 2;
};
template <>
struct FwdCfg<128> {
    static constexpr int BC = 128, NQ = 2;
};
template <>
struct FwdCfg<256> {
    static constexpr int BC = 128, NQ = 1;
};

// F8: e4m3 operands (Q, K row-major; V transposed, [channel][key]), d = 128 only.
//
// Two query tiles (NQ = 2): P goes to shared memory (the A operand of P V), so that
// S of the next key block can overwrite S in tensor memory as soon as the softmax has
// read it, while P V of this block still runs.  One tile (d = 256): P is written
// back over S in tensor memory and read from there by P V.
template <int D, bool F8 = false>
struct FwdLayout {
    using C = FwdCfg<D>;
    static constexpr int BC = C::BC, NQ = C::NQ;
    static constexpr bool PSM = NQ == 2;               // P in shared memory
    static constexpr int ESZ = F8 ? 1 : 2;             // bytes per operand element
    static constexpr int KCH = D * ESZ / 128;          // 128-byte chunks per row
    static constexpr int CH_ELEMS = 128 / ESZ;         // elements per chunk
    static constexpr int KSTEPS_S = D * ESZ / 32;      // S = Q K^T: 32 bytes of K per instruction
    static constexpr int KSTEPS_PV = BC * ESZ / 32;    // O += P V: 32 bytes of keys per instruction
    static constexpr float RESCALE = F8 ? 4.f : kRescaleLog2;
    static_assert(!F8 || (D == 128 && BC == 128 && NQ == 2), "FP8 layout: d = 128");
    static constexpr int Q_CHUNK = BR * 128;
    static constexpr int Q_TILE = KCH * Q_CHUNK;
    static constexpr int KV_CHUNK = BC * 128;
    static constexpr int KV_TILE = KCH * KV_CHUNK;
    static constexpr int P_CHUNK = BR * 128;           // P of a tile: BR rows x BC keys, K-major,
    static constexpr int PCH = BC * ESZ / 128;         // in 128-byte chunks of keys
    static constexpr int P_TILE = PSM ? PCH * P_CHUNK : 0;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_P = NQ * Q_TILE;
    static constexpr int OFF_SLOT = OFF_P + NQ * P_TILE;
    // K/V ring.  Two tiles: a slot holds a whole K_j or V_j tile.  One tile (d = 256): a slot
    // holds a 16 KB chunk, so that a 64 KB tile streams through the ring and each chunk is
    // released as soon as its products have read it: K_j in KCH chunks of 64 channels (S
    // consumes them in order along its contraction), V_j in VCH chunks of 32 keys, each
    // [KCH][32 keys][128 bytes] (P V consumes them in order along its contraction).
    static constexpr int VCH = BC / 32;
    static_assert(NQ != 1 || (VCH == KCH && VCH * 32 * 128 * KCH == KCH * KV_CHUNK), "one tile: equal chunks");
    static constexpr int SLOT_BYTES = NQ == 1 ? KV_CHUNK : KV_TILE;
    // as many slots as the remaining shared memory holds, at most 8 (one tile: 12 chunks)
    static constexpr int NSLOT_FIT = (227 * 1024 - 1024 - 512 - OFF_SLOT) / SLOT_BYTES;
    static constexpr int NSLOT = PSM ? (NSLOT_FIT < 8 ? NSLOT_FIT : 8)
                                     : (F8 ? 8 : (NSLOT_FIT < 12 ? NSLOT_FIT : 12));
    static_assert(NSLOT >= 3 && (NQ != 1 || NSLOT >= 2 * KCH + 1), "K/V ring depth");
    static constexpr int OFF_BAR = OFF_SLOT + NSLOT * SLOT_BYTES;
    // S buffers in tensor memory: one per tile with two tiles; with one tile two that the
    // key blocks take in turn (P goes back over S there, so S of block k + 2 waits for P V
    // of block k)
    static constexpr int NSB = 2;
    // barrier indices
    static constexpr int B_FULL = 0, B_EMPTY = NSLOT, B_QFULL = 2 * NSLOT, B_QEMPTY = 2 * NSLOT + 1,
                         B_SFULL = 2 * NSLOT + 2, B_PFULL = B_SFULL + NSB, B_ODONE = B_PFULL + NSB,
                         B_OEMPTY = B_ODONE + 2, B_DRAIN = B_OEMPTY + 2, B_PREAD = B_DRAIN + 1,
                         B_OFINAL = B_PREAD + NSB, B_DRAIN1 = B_OFINAL + 2, B_SFREE = B_DRAIN1 + 1,
                         NBAR = B_SFREE + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // tmem base (u32), abort flag (int)
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1024-byte alignment
    static constexpr int S_COL = 0;                  // S buffer b at columns [b*BC, (b+1)*BC)
    static constexpr int O_COL = NSB * BC;           // O~ of tile t at [O_COL + t*D, +D)
    static constexpr int TMEM_COLS = 512;
    static constexpr int NTHREADS = 128 + NQ * 128;
    static_assert(O_COL + NQ * D <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static constexpr uint32_t IDESC_S =
        F8 ? idesc_e4m3_f32(128, BC) : idesc_bf16_f32(128, BC, false, false);   // Q K^T, both K-major
    // P V: P K-major (shared or tensor memory); bf16 V is MN-major ([key][channel]), the
    // e4m3 V is stored transposed, K-major
    static constexpr uint32_t IDESC_PV = F8 ? idesc_e4m3_f32(128, D) : idesc_bf16_f32(128, D, false, true);
};

enum WaitSite : int {
    SITE_P_EMPTY = 1, SITE_P_QEMPTY, SITE_M_QFULL, SITE_M_FULL, SITE_M_PFULL, SITE_M_OEMPTY,
    SITE_S_SFULL, SITE_S_ODONE, SITE_S_EPI, SITE_M_PREAD
};

struct FwdArgs {
    __nv_bfloat16 *o;
    float *lse;
    int BH, Tq, Tk;
    // allowed keys of row r: r + Tk - Tq - left <= l <= r + Tk - Tq + right (-1: that side
    // unbounded; causal is left = -1, right = 0), in 128 x 128 blocks marked by bmask
    int left, right;
    const uint8_t *bmask;   // null, or [heads][nqbm][nkbm], nonzero = visit
    int bm_per_head;        // one mask per head (else one for all heads)
    int nqbm, nkbm;         // ceil(Tq / 128), ceil(Tk / 128)
    int masked;             // a left bound or a block mask: the MASKED instance runs
    float scale_log2;    // scale * log2(e)
    // FP8: dequantization factors of the e4m3 operands: Q per 128-row block, K per
    // 128-key block, V per channel ([heads][nqd], [heads][nkd], [heads][D])
    const float *qd, *kd, *vd;
    int nqd, nkd;
    int nqb;             // units per head
    int units;           // BH * nqb
    int group;           // heads per L2 group
    uint64_t timeout_ns;
    int withhold;        // test-only build: the arrive this launch leaves out (else 0, unused)
};

// One unit = NQ consecutive 128-row query tiles of one (b, h).  Tile t visits the KV
// blocks j in [lo, hi] (its rows' window) whose 128-key block its mask row marks.
struct TileRange {
    int lo, hi;              // KV block range (lo > hi: none)
    const uint8_t *bm;       // mask row of the tile's 128 rows, or null
    int n;                   // KV blocks the tile visits (0: none)
    int first, last;         // first and last of them
    int rows;                // the tile has at least one query row
};

struct Plan {
    int bh, row0;
    TileRange tr0, tr1;      // tiles 0 and 1
    int J;                   // jobs (one S and one PV MMA each) in the unit
    int js, je;              // first and last KV block any tile visits
};

// Tile t's range, chosen with a select (no run-time array indexing).
__device__ __forceinline__ TileRange tile_of(const Plan &p, int t) { return t ? p.tr1 : p.tr0; }

template <int BC>
__device__ __forceinline__ bool tile_active(const TileRange &r, int j)
{
    if (!r.rows || j < r.lo || j > r.hi)
        return false;
    return !r.bm || r.bm[(j * BC) >> 7] != 0;
}

// The first KV block at or after j that the tile visits (hi + 1 if none).
template <int BC>
__device__ __forceinline__ int next_active(const TileRange &r, int j)
{
    while (j <= r.hi && !tile_active<BC>(r, j))
        ++j;
    return j;
}

// MASKED = false: no left bound and no block mask, so every tile visits a prefix
// 0 .. n-1 of the KV blocks (causal, non-causal, right-bounded windows).
template <int D, bool MASKED>
__device__ __forceinline__ Plan make_plan(int u, const FwdArgs &a)
{
    using L = FwdLayout<D>;
    const int per_group = a.group * a.nqb;
    const int g = u / per_group;
    const int w = u - g * per_group;
    const int heads_here = min(a.group, a.BH - g * a.group);
    const int lvl = w / heads_here;                // 0 = longest units first
    Plan p;
    p.bh = g * a.group + (w - lvl * heads_here);
    const int qb = a.nqb - 1 - lvl;
    p.row0 = qb * L::NQ * BR;
    const long off = (long)a.Tk - a.Tq;
    p.J = 0;
    p.js = 1 << 30;
    p.je = -1;
    if constexpr (!MASKED) {
        const int nkv = (a.Tk + L::BC - 1) / L::BC;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            TileRange tr;
            const int r_first = p.row0 + t * BR;
            tr.rows = (t < L::NQ) && (r_first < a.Tq);
            int n = 0;
            if (tr.rows) {
                if (a.right < 0) {
                    n = nkv;
                } else {
                    const long lim = (long)min(r_first + BR - 1, a.Tq - 1) + off + a.right;   // last row's last key
                    n = lim < 0 ? 0 : min(nkv, (int)(lim / L::BC) + 1);
                }
            }
            tr.lo = tr.first = 0;
            tr.hi = tr.last = n - 1;
            tr.bm = nullptr;
            tr.n = n;
            p.J += n;
            if (t == 0)
                p.tr0 = tr;
            else
                p.tr1 = tr;
        }
        p.js = 0;
        p.je = max(p.tr0.n, p.tr1.n) - 1;
        return p;
    } else {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            TileRange tr;
            const int r_first = p.row0 + t * BR;
            tr.rows = (t < L::NQ) && (r_first < a.Tq);
            tr.lo = 0;
            tr.hi = -1;
            tr.bm = nullptr;
            if (tr.rows) {
                const int r_last = min(r_first + BR - 1, a.Tq - 1);
                // keys any row of the tile may see: from the first row's lowest to the last row's highest
                const long klo = a.left >= 0 ? max(0L, (long)r_first + off - a.left) : 0L;
                const long khi = a.right >= 0 ? min((long)a.Tk - 1, (long)r_last + off + a.right) : (long)a.Tk - 1;
                if (klo <= khi) {
                    tr.lo = (int)(klo / L::BC);
                    tr.hi = (int)(khi / L::BC);
                }
                if (a.bmask)
                    tr.bm = a.bmask + ((size_t)(a.bm_per_head ? p.bh : 0) * a.nqbm + (r_first >> 7)) * a.nkbm;
            }
            int n = 0;
            if (!tr.bm) {
                n = tr.hi - tr.lo + 1;
                tr.first = tr.lo;
                tr.last = tr.hi;
            } else {
                tr.first = tr.hi + 1;
                tr.last = tr.lo - 1;
                for (int j = tr.lo; j <= tr.hi; ++j)
                    if (tile_active<L::BC>(tr, j)) {
                        tr.first = min(tr.first, j);
                        tr.last = j;
                        ++n;
                    }
            }
            tr.n = n > 0 ? n : 0;
            if (n > 0) {
                p.js = min(p.js, tr.first);
                p.je = max(p.je, tr.last);
            }
            p.J += tr.n;
            if (t == 0)
                p.tr0 = tr;
            else
                p.tr1 = tr;
        }
        return p;
    }
}

// Two tiles: the K/V blocks either tile of the unit visits (both walk them, each
// skipping the blocks that are not its own).  union_next gives the first such block at
// or after j (je + 1 if none), union_count their number.
template <int BC, bool MASKED>
__device__ __forceinline__ int union_next(const Plan &p, int j)
{
    if constexpr (MASKED)
        while (j <= p.je && !tile_active<BC>(p.tr0, j) && !tile_active<BC>(p.tr1, j))
            ++j;
    return j;
}

template <int BC, bool MASKED>
__device__ __forceinline__ int union_count(const Plan &p)
{
    if constexpr (!MASKED)
        return p.je - p.js + 1;
    int n = 0;
    for (int j = union_next<BC, MASKED>(p, p.js); j <= p.je; j = union_next<BC, MASKED>(p, j + 1))
        ++n;
    return n;
}

// Generic-proxy writes to shared memory (P) made visible to the tensor core's reads.
__device__ __forceinline__ void fence_smem_to_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// The MMA order of a unit: S(0), S(1), then PV(k) followed by S(k+2).  The
// producer walks the same order to load tiles in first-use order.
template <typename FS, typename FPV>
__device__ __forceinline__ bool walk_ops(int J, FS &&fs, FPV &&fpv)
{
    if (!fs(0))
        return false;
    if (J > 1 && !fs(1))
        return false;
    for (int k = 0; k < J; ++k) {
        if (!fpv(k))
            return false;
        if (k + 2 < J && !fs(k + 2))
            return false;
    }
    return true;
}

template <int D, bool MASKED, bool F8 = false>
__global__ void __launch_bounds__(FwdLayout<D, F8>::NTHREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdArgs a)
{
    using L = FwdLayout<D, F8>;
    static_assert(!(F8 && MASKED), "the FP8 forward takes no window or block mask");
    constexpr int BC = L::BC, NQ = L::NQ, NSLOT = L::NSLOT;
    constexpr bool INL = NQ == 2;   // register split below: bounded waits inlined (no calls)
    constexpr bool L1 = NQ == 1;    // softmax waits: lane 0 polls for the warp (see mbar_wait_warp)
    constexpr uint32_t HN = NQ == 1 ? 4000u : 0u;   // one tile: waits suspend up to 4 us per poll
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
        // with two query tiles, each tile's MMA warp releases every K/V slot and the Q tiles
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(bar(L::B_FULL + s), 1);
            mbar_init(bar(L::B_EMPTY + s), NQ);
        }
        mbar_init(bar(L::B_QFULL), 1);
        mbar_init(bar(L::B_QEMPTY), NQ);
        for (int b = 0; b < L::NSB; ++b) {
            mbar_init(bar(L::B_SFULL + b), 1);
            mbar_init(bar(L::B_PFULL + b), 128);
            mbar_init(bar(L::B_PREAD + b), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::B_ODONE + b), 1);
            mbar_init(bar(L::B_OEMPTY + b), 128);
        }
        mbar_init(bar(L::B_OFINAL), 1);
        mbar_init(bar(L::B_OFINAL + 1), 1);
        mbar_init(bar(L::B_DRAIN), 1);
        mbar_init(bar(L::B_DRAIN1), 1);
        mbar_init(bar(L::B_SFREE), 128);       // softmax of tile 0 has read S_0 (P in shared memory)
        mbar_init(bar(L::B_SFREE + 1), 128);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx ctx{abort_flag, &g_fwd_status, a.timeout_ns};

    uint32_t n_loads = 0, n_q = 0;   // producer counters, kept for the drain

    // Register split with two query tiles (launch: 384 threads x 168): the producer/MMA
    // warpgroup keeps 104 per thread, the softmax warpgroups take 200; 104 + 2 x 200 <=
    // 3 x 168, with no spills in the unmasked instances.
    if (warp < 4) {
        if constexpr (INL)
            regs_dealloc<104>();
        if (warp == 0) {
            // ------------------------------------------------ TMA producer
            if (lane == 0) {
                const uint64_t pol_kv = policy_evict_last();
                const uint64_t pol_q = policy_evict_first();
                for (int pass = 0, u = snake_unit<!MASKED>(0); u < a.units; u = snake_unit<!MASKED>(++pass)) {
                    const Plan p = make_plan<D, MASKED>(u, a);
                    if (p.J == 0)
                        continue;
                    if (n_q > 0 && !mbar_wait<INL, HN>(bar(L::B_QEMPTY), (n_q - 1) & 1, ctx, SITE_P_QEMPTY))
                        break;
                    uint32_t qbytes = 0;
                    for (int t = 0; t < NQ; ++t)
                        qbytes += tile_of(p, t).n > 0 ? L::Q_TILE : 0;
                    mbar_arrive_expect_tx(bar(L::B_QFULL), qbytes);
                    for (int t = 0; t < NQ; ++t)
                        if (tile_of(p, t).n > 0)
                            for (int c = 0; c < L::KCH; ++c)
                                tma_load_3d_hint(sbase + L::OFF_Q + t * L::Q_TILE + c * L::Q_CHUNK, &tm_q,
                                                 bar(L::B_QFULL), c * L::CH_ELEMS, p.row0 + t * BR, p.bh, pol_q);
                    ++n_q;
                    auto load = [&](const CUtensorMap *map, int j) -> bool {
                        const uint32_t slot = n_loads % NSLOT;
                        if (n_loads >= NSLOT &&
                            !mbar_wait<INL, HN>(bar(L::B_EMPTY + slot), ((n_loads / NSLOT) - 1) & 1, ctx, SITE_P_EMPTY))
                            return false;
                        mbar_arrive_expect_tx(bar(L::B_FULL + slot), L::KV_TILE);
                        const uint32_t dst = sbase + L::OFF_SLOT + slot * L::KV_TILE;
                        if (F8 && map == &tm_v)   // V^T: one box of BC keys x D channels
                            tma_load_3d_hint(dst, map, bar(L::B_FULL + slot), j * BC, 0, p.bh, pol_kv);
                        else
                            for (int c = 0; c < L::KCH; ++c)
                                tma_load_3d_hint(dst + c * L::KV_CHUNK, map, bar(L::B_FULL + slot), c * L::CH_ELEMS,
                                                 j * BC, p.bh, pol_kv);
                        ++n_loads;
                        return true;
                    };
                    // one tile: K_j or V_j as KCH chunk slots (see FwdLayout)
                    auto load_chunks = [&](bool is_k, int j) -> bool {
                        for (int c = 0; c < L::KCH; ++c) {
                            const uint32_t slot = n_loads % NSLOT;
                            if (n_loads >= NSLOT &&
                                !mbar_wait<INL, HN>(bar(L::B_EMPTY + slot), ((n_loads / NSLOT) - 1) & 1, ctx, SITE_P_EMPTY))
                                return false;
                            mbar_arrive_expect_tx(bar(L::B_FULL + slot), L::SLOT_BYTES);
                            const uint32_t dst = sbase + L::OFF_SLOT + slot * L::SLOT_BYTES;
                            if (is_k)   // channels [64c, 64c + 64) of the block's BC keys
                                tma_load_3d_hint(dst, &tm_k, bar(L::B_FULL + slot), c * L::CH_ELEMS, j * BC, p.bh, pol_kv);
                            else        // keys [32c, 32c + 32), all channels, 64 at a time
                                for (int dc = 0; dc < L::KCH; ++dc)
                                    tma_load_3d_hint(dst + dc * 32 * 128, &tm_v, bar(L::B_FULL + slot), dc * L::CH_ELEMS,
                                                     j * BC + 32 * c, p.bh, pol_kv);
                            ++n_loads;
                        }
                        return true;
                    };
                    bool ok = true;
                    if constexpr (NQ == 2) {
                        // each tile's MMA warp consumes K_j, V_j of every block either tile visits,
                        // in the order S(0), S(1), PV(0), S(2), PV(1), ...
                        int kj = union_next<BC, MASKED>(p, p.js), vj = kj;
                        ok = walk_ops(
                            union_count<BC, MASKED>(p),
                            [&](int) {
                                const bool r = load(&tm_k, kj);
                                kj = union_next<BC, MASKED>(p, kj + 1);
                                return r;
                            },
                            [&](int) {
                                const bool r = load(&tm_v, vj);
                                vj = union_next<BC, MASKED>(p, vj + 1);
                                return r;
                            });
                    } else {
                        // one tile: its visited blocks in the MMA order S(0), S(1), PV(0), S(2), ...
                        int kj = p.tr0.first, vj = p.tr0.first;
                        ok = walk_ops(
                            p.J,
                            [&](int) {
                                const bool r = load_chunks(true, kj);
                                kj = next_active<BC>(p.tr0, kj + 1);
                                return r;
                            },
                            [&](int) {
                                const bool r = load_chunks(false, vj);
                                vj = next_active<BC>(p.tr0, vj + 1);
                                return r;
                            });
                    }
                    if (!ok)
                        break;
                }
                // drain: every copy still in flight lands before the CTA exits
                const uint32_t lo = n_loads > (uint32_t)NSLOT ? n_loads - NSLOT : 0;
                for (uint32_t i = lo; i < n_loads; ++i)
                    mbar_wait_drain(bar(L::B_FULL + i % NSLOT), (i / NSLOT) & 1);
                if (n_q > 0)
                    mbar_wait_drain(bar(L::B_QFULL), (n_q - 1) & 1);
            }
            __syncwarp();
        } else if (NQ == 2 && (warp == 1 || warp == 2)) {
            // ------------------------------------------------ MMA issuer of query tile t
            // One issuing thread per tile.  Both walk the K/V blocks either tile visits in the
            // producer's order S(0), S(1), PV(0), S(2), PV(1), ...: with P in shared memory, S of
            // block k+1 only waits for the softmax to have read S of block k, and runs while
            // P V of block k waits for its P.
            if (lane == 0) {
                const int t = (int)warp - 1;
                const uint32_t s_col = L::S_COL + t * BC, o_col = L::O_COL + t * D;
                const uint64_t qd = sdesc_sw128(sbase + L::OFF_Q + t * L::Q_TILE, 16, 1024);
                const uint64_t pd = sdesc_sw128(sbase + L::OFF_P + t * L::P_TILE, 16, 1024);
                const uint32_t drain_bar = bar(t == 0 ? L::B_DRAIN : L::B_DRAIN1);
                uint32_t ld = 0, q_seen = 0, sn = 0, pvn = 0, epi = 0;
                bool ok = true;
                for (int pass = 0, u = snake_unit<!MASKED>(0); u < a.units && ok; u = snake_unit<!MASKED>(++pass)) {
                    const Plan p = make_plan<D, MASKED>(u, a);
                    if (p.J == 0)
                        continue;
                    if (!mbar_wait<INL, HN>(bar(L::B_QFULL), q_seen & 1, ctx, SITE_M_QFULL))
                        break;
                    ++q_seen;
                    const TileRange me = tile_of(p, t);
                    if (me.n == 0)
                        mbar_arrive(bar(L::B_QEMPTY));      // this tile reads no Q in this unit
                    auto mine = [&](int j) { return MASKED ? tile_active<BC>(me, j) : j < me.n; };
                    auto acquire = [&](uint32_t &slot) -> bool {
                        slot = ld % NSLOT;
                        const bool r = mbar_wait<INL, HN>(bar(L::B_FULL + slot), (ld / NSLOT) & 1, ctx, SITE_M_FULL);
                        ++ld;
                        return r;
                    };
                    int kj = union_next<BC, MASKED>(p, p.js), vj = kj;
                    ok = walk_ops(
                        union_count<BC, MASKED>(p),
                        [&](int) -> bool {
                            // K_j: S_t = Q_t K_j^T
                            uint32_t ks;
                            if (!acquire(ks))
                                return false;
                            const int j = kj;
                            kj = union_next<BC, MASKED>(p, kj + 1);
                            if (!mine(j)) {
                                mbar_arrive(bar(L::B_EMPTY + ks));   // K_j is only for the other tile
                                return true;
                            }
                            // S_t is overwritten once the softmax has read the previous S_t
                            if (sn > 0 && !mbar_wait<INL, HN>(bar(L::B_SFREE + t), (sn - 1) & 1, ctx, SITE_M_PREAD))
                                return false;
                            tc_fence_after();
                            // descriptors: bases once, then compile-time offsets (address field in
                            // 16-byte units), so that the issuing thread spends no time between MMAs
                            const uint64_t kd = sdesc_sw128(sbase + L::OFF_SLOT + ks * L::KV_TILE, 16, 1024);
#pragma unroll
                            for (int kk = 0; kk < L::KSTEPS_S; ++kk) {
                                const uint32_t off = ((kk >> 2) * L::Q_CHUNK + (kk & 3) * 32) >> 4;
                                const uint32_t offk = ((kk >> 2) * L::KV_CHUNK + (kk & 3) * 32) >> 4;
                                if constexpr (F8)
                                    mma_ss_f8(tmem + s_col, qd + off, kd + offk, L::IDESC_S, kk > 0 ? 1u : 0u);
                                else
                                    mma_ss(tmem + s_col, qd + off, kd + offk, L::IDESC_S, kk > 0 ? 1u : 0u);
                            }
                            tc_commit(bar(L::B_SFULL + t));
#if FA_TEST_WITHHOLD
                            const bool hold = a.withhold == WITHHOLD_FWD_KV && blockIdx.x == 0 && t == 0 && sn == 0;
#else
                            constexpr bool hold = false;
#endif
                            if (!hold)
                                tc_commit(bar(L::B_EMPTY + ks));
                            if (j == me.last)
                                tc_commit(bar(L::B_QEMPTY));
                            ++sn;
                            return true;
                        },
                        [&](int) -> bool {
                            // V_j: O_t += P_t V_j, P_t from shared memory
                            uint32_t vs;
                            if (!acquire(vs))
                                return false;
                            const int j = vj;
                            vj = union_next<BC, MASKED>(p, vj + 1);
                            if (!mine(j)) {
                                mbar_arrive(bar(L::B_EMPTY + vs));
                                return true;
                            }
                            if (!mbar_wait<INL, HN>(bar(L::B_PFULL + t), pvn & 1, ctx, SITE_M_PFULL))
                                return false;
                            const bool first = j == (MASKED ? me.first : 0);
                            if (first && epi > 0 &&
                                !mbar_wait<INL, HN>(bar(L::B_OEMPTY + t), (epi - 1) & 1, ctx, SITE_M_OEMPTY))
                                return false;
                            tc_fence_after();
                            // P: K-major, 32 bytes of keys per step; V^T (FP8) K-major likewise, bf16 V
                            // MN-major: 16 keys = 16 rows of 128 bytes
                            const uint32_t va = sbase + L::OFF_SLOT + vs * L::KV_TILE;
                            const uint64_t vd = F8 ? sdesc_sw128(va, 16, 1024) : sdesc_sw128(va, L::KV_CHUNK, 1024);
#pragma unroll
                            for (int kk = 0; kk < L::KSTEPS_PV; ++kk) {
                                const uint32_t offp = ((kk >> 2) * L::P_CHUNK + (kk & 3) * 32) >> 4;
                                const uint32_t offv = (F8 ? kk * 32 : kk * 16 * 128) >> 4;
                                const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
                                if constexpr (F8)
                                    mma_ss_f8(tmem + o_col, pd + offp, vd + offv, L::IDESC_PV, acc);
                                else
                                    mma_ss(tmem + o_col, pd + offp, vd + offv, L::IDESC_PV, acc);
                            }
                            tc_commit(bar(L::B_ODONE + t));   // O~ current and P read: one signal
                            tc_commit(bar(L::B_EMPTY + vs));
                            ++pvn;
                            if (j == me.last) {
#if FA_TEST_WITHHOLD
                                const bool hold = a.withhold == WITHHOLD_FWD_EPI && blockIdx.x == 0 && t == 0 && epi == 0;
#else
                                constexpr bool hold = false;
#endif
                                if (!hold)
                                    tc_commit(bar(L::B_OFINAL + t));
                                ++epi;
                            }
                            return true;
                        });
                }
                tc_commit(drain_bar);
                mbar_wait_drain(drain_bar, 0);
            }
            __syncwarp();
        } else if (NQ == 1 && (warp == 1 || warp == 2)) {
            // ------------------------------------------------ MMA issuers (one query tile)
            // Warp 1 issues the S products and warp 2 the P V products, so that neither waits
            // behind the other's barriers: S(k+2) goes out as soon as P V(k) has read P(k) from
            // the S buffer that it overwrites, and P V(k) as soon as the softmax has written
            // P(k).  A tcgen05.mma blocks its issuing thread while the tensor core's queue is
            // full, so with one issuer every wait of one product stalled the other's issue.
            // Both warps locate their chunks in the K/V ring by the producer's load order of the
            // unit, S(0), S(1), PV(0), S(2), PV(1), ..., KCH chunks each: S(k) is op k ? 2k - 1 : 0
            // and P V(k) is op min(J, k + 2) + k.  Each chunk is released as soon as the
            // products that read it have completed.
            if (lane == 0) {
                const bool s_side = warp == 1;
                uint32_t base = 0, kg = 0, q_seen = 0, epi = 0;
                bool ok = true;
                const uint64_t qd = sdesc_sw128(sbase + L::OFF_Q, 16, 1024);
                for (int pass = 0, u = snake_unit<!MASKED>(0); u < a.units && ok; u = snake_unit<!MASKED>(++pass)) {
                    const Plan p = make_plan<D, MASKED>(u, a);
                    const int J = p.J;
                    if (J == 0)
                        continue;
                    if (s_side) {
                        if (!mbar_wait<INL, HN>(bar(L::B_QFULL), q_seen & 1, ctx, SITE_M_QFULL))
                            break;
                        ++q_seen;
                    }
                    for (int k = 0; k < J && ok; ++k) {
                        const uint32_t g = kg + k, b = g % L::NSB;
                        const uint32_t op = (uint32_t)(s_side ? (k ? 2 * k - 1 : 0) : min(J, k + 2) + k);
                        const uint32_t n0 = base + op * L::KCH;   // first chunk of this product
                        if (s_side) {
                            // S(g) overwrites the columns that held P(g - NSB): P V(g - NSB) must
                            // have finished reading them
                            if (g >= (uint32_t)L::NSB &&
                                !mbar_wait<INL, HN>(bar(L::B_PREAD + b), (g / L::NSB - 1) & 1, ctx, SITE_M_PREAD)) {
                                ok = false;
                                break;
                            }
                            // K_j chunk c: channels [64c, 64c + 64), four K steps of 16
#pragma unroll
                            for (int c = 0; c < L::KCH; ++c) {
                                const uint32_t n = n0 + c, slot = n % NSLOT;
                                if (!mbar_wait<INL, HN>(bar(L::B_FULL + slot), (n / NSLOT) & 1, ctx, SITE_M_FULL)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                const uint64_t kd = sdesc_sw128(sbase + L::OFF_SLOT + slot * L::SLOT_BYTES, 16, 1024);
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {   // 16 bf16 = 32 bytes along K
                                    const uint32_t off = (c * L::Q_CHUNK + kk * 32) >> 4;
                                    mma_ss(tmem + L::S_COL + b * BC, qd + off, kd + ((kk * 32) >> 4), L::IDESC_S,
                                           (c > 0 || kk > 0) ? 1u : 0u);
                                }
                                tc_commit(bar(L::B_EMPTY + slot));
                            }
                            if (!ok)
                                break;
                            tc_commit(bar(L::B_SFULL + b));
                            if (k == J - 1)
                                tc_commit(bar(L::B_QEMPTY));
                        } else {
                            if (!mbar_wait<INL, HN>(bar(L::B_PFULL + b), (g / L::NSB) & 1, ctx, SITE_M_PFULL)) {
                                ok = false;
                                break;
                            }
                            if (k == 0 && epi > 0 &&
                                !mbar_wait<INL, HN>(bar(L::B_OEMPTY), (epi - 1) & 1, ctx, SITE_M_OEMPTY)) {
                                ok = false;
                                break;
                            }
                            // V_j chunk c: keys [32c, 32c + 32) as [KCH][32 keys][128 bytes], two K
                            // steps of 16 keys; P from tensor memory (16 keys = 8 packed columns)
#pragma unroll
                            for (int c = 0; c < L::VCH; ++c) {
                                const uint32_t n = n0 + c, slot = n % NSLOT;
                                if (!mbar_wait<INL, HN>(bar(L::B_FULL + slot), (n / NSLOT) & 1, ctx, SITE_M_FULL)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                const uint64_t vd = sdesc_sw128(sbase + L::OFF_SLOT + slot * L::SLOT_BYTES, 32 * 128, 1024);
#pragma unroll
                                for (int kk = 0; kk < 2; ++kk)
                                    mma_ts(tmem + L::O_COL, tmem + L::S_COL + b * BC + (2 * c + kk) * 8,
                                           vd + ((kk * 16 * 128) >> 4), L::IDESC_PV, (k > 0 || c > 0 || kk > 0) ? 1u : 0u);
                                tc_commit(bar(L::B_EMPTY + slot));
                            }
                            if (!ok)
                                break;
                            // O~ holds P V(g): the softmax may be up to NSB jobs ahead, so the
                            // signal alternates between two barriers to stay within one phase
                            tc_commit(bar(L::B_ODONE + (g & 1)));
                            tc_commit(bar(L::B_PREAD + b));
                            if (k == J - 1) {   // last P V of the unit
                                tc_commit(bar(L::B_OFINAL));
                                ++epi;
                            }
                        }
                    }
                    base += 2u * (uint32_t)L::KCH * (uint32_t)J;
                    kg += (uint32_t)J;
                }
                // drain: all MMAs this thread issued complete before tensor memory is released
                const uint32_t drain_bar = bar(s_side ? L::B_DRAIN : L::B_DRAIN1);
                tc_commit(drain_bar);
                mbar_wait_drain(drain_bar, 0);
            }
            __syncwarp();
        }
    } else {
        if constexpr (INL)
            regs_alloc<200>();
        // ------------------------------------------------ softmax + epilogue
        const int t = (int)(warp - 4) >> 2;            // query tile of this warpgroup
        const uint32_t quarter = warp & 3u;            // TMEM lanes [32*quarter, +32)
        const int rit = (int)(quarter * 32 + lane);    // row within the tile
        const float sl2 = a.scale_log2;
        const uint32_t lane_base = tmem + ((quarter * 32u) << 16);
        uint32_t pv = 0, ep = 0;   // jobs and epilogues of this tile so far
        // The two softmax warpgroups run unsynchronised: each follows its own tile's S.
        for (int pass = 0, u = snake_unit<!MASKED>(0); u < a.units; u = snake_unit<!MASKED>(++pass)) {
            const Plan p = make_plan<D, MASKED>(u, a);
            const int r = p.row0 + t * BR + rit;
            const TileRange me = tile_of(p, t);
            const bool row_ok = r < a.Tq;
            const size_t grow = (size_t)p.bh * a.Tq + r;
            if (!me.rows)
                continue;
            if (me.n == 0) {   // no key is allowed for any row of this tile
                if (row_ok) {
                    uint4 *dst = reinterpret_cast<uint4 *>(a.o + grow * D);
                    for (int i = 0; i < D / 8; ++i)
                        dst[i] = make_uint4(0, 0, 0, 0);
                    a.lse[grow] = -INFINITY;
                }
                continue;
            }
            // FP8: c log2(e) times the tile's Q dequantization factor; per key block the K
            // factor joins it.  m is then kept in the exp2 domain (scores times c log2 e).
            float sq = 1.f;
            if constexpr (F8)
                sq = a.scale_log2 * __ldg(a.qd + (size_t)p.bh * a.nqd + ((p.row0 + t * BR) >> 7));
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            // jj: job index of this tile; j: the KV block it visits
            for (int jj = 0, j = MASKED ? me.first : 0; jj < me.n && ok;
                 ++jj, j = MASKED ? next_active<BC>(me, j + 1) : jj) {
                // two tiles: S buffer t, one phase per job of this tile; one tile: the NSB
                // S buffers take consecutive jobs in turn
                const uint32_t b = NQ == 2 ? (uint32_t)t : (pv % L::NSB);
                const uint32_t ph = NQ == 2 ? (pv & 1) : ((pv / L::NSB) & 1);
                if (!mbar_wait_warp<INL, L1, HN>(bar(L::B_SFULL + b), ph, ctx, SITE_S_SFULL)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // S row: all column chunks in flight, one wait
                uint32_t sv[BC / 32][32];
#pragma unroll
                for (int c = 0; c < BC / 32; ++c)
                    tmem_ld_x32_nowait(lane_base + L::S_COL + b * BC + c * 32, sv[c]);
#pragma unroll
                for (int c = 0; c < BC / 32; ++c)
                    tmem_wait_ld_x32(sv[c]);
                if constexpr (L::PSM) {   // S_t is in registers: the next S may overwrite it
                    tc_fence_before();
                    mbar_arrive(bar(L::B_SFREE + t));
                }
                float s[BC];
#pragma unroll
                for (int c = 0; c < BC / 32; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        s[c * 32 + i] = __uint_as_float(sv[c][i]);
                // mask: tail keys beyond Tk, and keys outside the row's window (causal: after
                // its diagonal key), only where the block is not wholly inside every row's window
                const int kv0 = j * BC;
                const int first_row = p.row0 + t * BR;
                const int last_row = min(first_row + BR - 1, a.Tq - 1);
                const long off = (long)a.Tk - a.Tq;
                const bool need_mask = (kv0 + BC > a.Tk) ||
                                       (a.right >= 0 && (long)kv0 + BC - 1 > (long)first_row + off + a.right) ||
                                       (MASKED && a.left >= 0 && (long)kv0 < (long)last_row + off - a.left);
                if (need_mask) {
                    long hi = a.Tk;   // allowed keys of row r: [lo, hi)
                    if (a.right >= 0)
                        hi = min(hi, (long)r + off + a.right + 1);
                    const long lo = (MASKED && a.left >= 0) ? (long)r + off - a.left : 0L;
                    const int ch = (int)max(0L, min((long)BC, hi - kv0));
                    const int cl = MASKED ? (int)max(0L, min((long)BC, lo - kv0)) : 0;
#pragma unroll
                    for (int i = 0; i < BC; ++i)
                        if (i < cl || i >= ch)
                            s[i] = -INFINITY;
                }
                // row max: four independent chains of three-input max
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
                static_assert(BC % 8 == 0, "row max covers BC in steps of 8");
#pragma unroll
                for (int i = 0; i < BC; i += 8) {
                    mx0 = fmax3(mx0, s[i], s[i + 1]);
                    mx1 = fmax3(mx1, s[i + 2], s[i + 3]);
                    mx2 = fmax3(mx2, s[i + 4], s[i + 5]);
                    mx3 = fmax3(mx3, s[i + 6], s[i + 7]);
                }
                const float rowmax = fmax3(mx0, mx1, fmax3(mx2, mx3, -INFINITY));
                bool resc;
                float alpha = 1.f, mref, sl2t = sl2;
                if constexpr (F8) {
                    // scores scale per tile: compare in the exp2 domain.  A zero factor (an
                    // all-zero block, whose raw scores are exactly 0) is kept positive so
                    // that masked -inf scores stay -inf.
                    sl2t = fmaxf(sq * __ldg(a.kd + (size_t)p.bh * a.nkd + ((j * BC) >> 7)), 1e-30f);
                    const float m_new = fmaxf(m, rowmax * sl2t);
                    resc = (m != -INFINITY) && (m_new - m > L::RESCALE);
                    if (m == -INFINITY) {
                        m = m_new;
                    } else if (resc) {
                        alpha = ex2_approx(m - m_new);
                        l *= alpha;
                        m = m_new;
                    }
                    // P~ carries a factor 2^4 (P~ <= 2^8 <= 448, small values stay normal in
                    // e4m3); l carries the same factor, so O~ / l does not see it
                    mref = (m == -INFINITY) ? 0.f : m - 4.f;
                } else {
                    const float m_new = fmaxf(m, rowmax);
                    resc = (m != -INFINITY) && ((m_new - m) * sl2 > L::RESCALE);
                    if (m == -INFINITY) {
                        m = m_new;                     // O~ and l of this row are still exactly 0
                    } else if (resc) {
                        alpha = ex2_approx((m - m_new) * sl2);
                        l *= alpha;
                        m = m_new;
                    }
                    mref = (m == -INFINITY) ? 0.f : m * sl2;
                }
                // P~ = exp2(c log2e (s - m)), 32 keys at a time, packed to bf16 pairs (e4m3
                // quadruples).  Two tiles: all of the row's P stays in registers until the
                // previous P V of the tile has finished reading the tile's P buffer in shared
                // memory, so that the wait overlaps the exponentials; then it is stored (128-byte
                // rows of keys, 16-byte units swizzled by the row, as the P V product reads
                // them).  One tile: P goes over the first columns of this S buffer.
                uint8_t *prow = smem + L::OFF_P + t * L::P_TILE + rit * 128;
                if constexpr (F8) {   // measured faster with the wait ahead of the exponentials
                    if (pv > 0 && !mbar_wait_warp<INL, false, HN>(bar(L::B_ODONE + t), (pv - 1) & 1, ctx, SITE_S_ODONE)) {
                        ok = false;
                        break;
                    }
                }
                float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
                uint32_t pw[F8 ? BC / 4 : 1];                   // e4m3 quadruples
                uint32_t pb[(!F8 && L::PSM) ? BC / 2 : 1];     // bf16 pairs (two tiles)
#pragma unroll
                for (int c = 0; c < BC / 32; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        const int e = c * 32 + 2 * i;
                        float x0, x1, x2, x3;
                        ffma2(x0, x1, s[e], s[e + 1], sl2t, sl2t, -mref, -mref);
                        ffma2(x2, x3, s[e + 2], s[e + 3], sl2t, sl2t, -mref, -mref);
                        x0 = ex2_approx(x0);
                        x1 = ex2_approx(x1);
                        x2 = ex2_approx(x2);
                        x3 = ex2_approx(x3);
                        fadd2(l0, l1, l0, l1, x0, x1);
                        fadd2(l2, l3, l2, l3, x2, x3);
                        if constexpr (F8) {
                            pw[c * 8 + i / 2] = pack_e4m3x4(x0, x1, x2, x3);
                        } else if constexpr (L::PSM) {
                            pb[c * 16 + i] = pack_bf16x2(x0, x1);
                            pb[c * 16 + i + 1] = pack_bf16x2(x2, x3);
                        } else {
                            pk[i] = pack_bf16x2(x0, x1);
                            pk[i + 1] = pack_bf16x2(x2, x3);
                        }
                    }
                    if constexpr (!F8 && !L::PSM)
                        tmem_st_x16(lane_base + L::S_COL + b * BC + c * 16, pk);
                }
                if constexpr (L::PSM) {
                    if (!F8 && pv > 0 && !mbar_wait_warp<INL, false, HN>(bar(L::B_ODONE + t), (pv - 1) & 1, ctx, SITE_S_ODONE)) {
                        ok = false;
                        break;
                    }
                    if constexpr (F8) {   // 128 keys: one 128-byte row, units of 16 keys
#pragma unroll
                        for (int unit = 0; unit < 8; ++unit)
                            *reinterpret_cast<uint4 *>(prow + ((unit ^ (rit & 7)) << 4)) =
                                make_uint4(pw[4 * unit], pw[4 * unit + 1], pw[4 * unit + 2], pw[4 * unit + 3]);
                    } else {              // keys [64h, 64h + 64): chunk h, units of 8 keys
#pragma unroll
                        for (int h = 0; h < BC / 64; ++h)
#pragma unroll
                            for (int unit = 0; unit < 8; ++unit)
                                *reinterpret_cast<uint4 *>(prow + h * L::P_CHUNK + ((unit ^ (rit & 7)) << 4)) =
                                    make_uint4(pb[h * 32 + 4 * unit], pb[h * 32 + 4 * unit + 1],
                                               pb[h * 32 + 4 * unit + 2], pb[h * 32 + 4 * unit + 3]);
                    }
                }
                l0 += l2;
                l1 += l3;
                l += l0 + l1;
                if (__any_sync(0xffffffffu, resc)) {
                    // O~ must hold the previous PV of this tile before it is rescaled (two tiles:
                    // waited for above)
                    if (!L::PSM &&
                        !mbar_wait_warp<INL, L1, HN>(bar(L::B_ODONE + ((pv - 1) & 1)), ((pv - 1) >> 1) & 1, ctx, SITE_S_ODONE)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // whole O~ row in flight at once (the S registers are free by now)
                    constexpr int OCH = D / 32 < 4 ? D / 32 : 4;   // chunks per batch
#pragma unroll
                    for (int c0 = 0; c0 < D / 32; c0 += OCH) {
                        uint32_t ov[OCH][32];
#pragma unroll
                        for (int c = 0; c < OCH; ++c)
                            tmem_ld_x32_nowait(lane_base + L::O_COL + t * D + (c0 + c) * 32, ov[c]);
#pragma unroll
                        for (int c = 0; c < OCH; ++c)
                            tmem_wait_ld_x32(ov[c]);
#pragma unroll
                        for (int c = 0; c < OCH; ++c) {
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                float y0, y1;
                                fmul2(y0, y1, __uint_as_float(ov[c][i]), __uint_as_float(ov[c][i + 1]), alpha, alpha);
                                ov[c][i] = __float_as_uint(y0);
                                ov[c][i + 1] = __float_as_uint(y1);
                            }
                            tmem_st_x32(lane_base + L::O_COL + t * D + (c0 + c) * 32, ov[c]);
                        }
                    }
                }
                if constexpr (L::PSM)
                    fence_smem_to_async();
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(L::B_PFULL + b));
                ++pv;
            }
            if (!ok)
                break;
            // epilogue: O = O~ / l, lse = c m + ln l.  With one tile the softmax can be up
            // to two PVs ahead of the tensor core here, too far for a parity wait on the
            // per-PV barrier; the per-unit barrier completes exactly once per epilogue.
            if (!mbar_wait_warp<INL, L1, HN>(bar(L::B_OFINAL + t), ep & 1, ctx, SITE_S_EPI))
                break;
            ++ep;
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld_x32(lane_base + L::O_COL + t * D + c * 32, v);
                if constexpr (F8) {   // the V dequantization factor of each channel
                    const float4 *vd4 = reinterpret_cast<const float4 *>(a.vd + (size_t)p.bh * D + c * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 f = __ldg(vd4 + i);
                        v[4 * i] = __float_as_uint(__uint_as_float(v[4 * i]) * f.x);
                        v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) * f.y);
                        v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) * f.z);
                        v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) * f.w);
                    }
                }
                if (row_ok) {
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
                    uint4 *dst = reinterpret_cast<uint4 *>(a.o + grow * D + c * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                }
            }
            if (row_ok) {
                const float m2 = F8 ? m - 4.f : m * sl2;   // exp2-domain reference of P~ and l
                a.lse[grow] = l > 0.f ? (m2 + log2f(l)) * 0.69314718055994530942f : -INFINITY;
            }
            tc_fence_before();
            mbar_arrive(bar(L::B_OEMPTY + t));
        }
    }
    // ---------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

template <int D>
int launch(const void *q, const void *k, const void *v, void *o, float *lse, int BH, int Tq, int Tk,
           const MaskSpec &mask, float scale, cudaStream_t s)
{
    using L = FwdLayout<D>;
    CUtensorMap tq, tk, tv;
    int st = encode_tmap_3d(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Tq, BH, 64, BR);
    if (st == OK)
        st = encode_tmap_3d(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Tk, BH, 64, L::BC);
    if (st == OK)
        st = encode_tmap_3d(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Tk, BH, 64, L::NQ == 1 ? 32 : L::BC);
    if (st != OK)
        return st;
    FwdArgs a;
    a.o = static_cast<__nv_bfloat16 *>(o);
    a.lse = lse;
    a.BH = BH;
    a.Tq = Tq;
    a.Tk = Tk;
    a.left = mask.left;
    a.right = mask.right;
    a.bmask = mask.block;
    a.bm_per_head = mask.per_head;
    a.nqbm = (Tq + 127) / 128;
    a.nkbm = (Tk + 127) / 128;
    a.masked = (mask.left >= 0 || mask.block) ? 1 : 0;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.qd = a.kd = a.vd = nullptr;
    a.nqd = a.nkd = 0;
    a.nqb = (Tq + L::NQ * BR - 1) / (L::NQ * BR);
    a.units = BH * a.nqb;
    // heads per group: keep the group's K and V within ~80 MB of L2, a whole number of
    // passes where possible (B8 H32 N4096 d128: 38 heads; measured faster than 24).  The
    // masked instance keeps ~48 MB groups and same-direction passes: its units' lengths
    // do not follow the order, and there the smaller groups measured faster.
    const double kv_head = 2.0 * Tk * D * 2.0;
    const int grid = a.units < device_sm_count() ? a.units : device_sm_count();
    int g = (int)((a.masked ? 48.0 : 80.0) * 1024 * 1024 / (kv_head > 1 ? kv_head : 1));
    g = g < 1 ? 1 : (g > BH ? BH : g);
    a.group = a.masked ? g : grid_aligned_group(g, a.nqb, grid);
    a.timeout_ns = wait_timeout_ns();
    a.withhold = WITHHOLD_NONE;
#if FA_TEST_WITHHOLD
    if (L::NQ == 2)
        a.withhold = test_withhold_take(WITHHOLD_FWD_KV, WITHHOLD_FWD_EPI);
#endif
    auto kernel = a.masked ? fwd_kernel<D, true> : fwd_kernel<D, false>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES) != cudaSuccess)
        return ERR_CUDA;
    kernel<<<grid, L::NTHREADS, L::SMEM_BYTES, s>>>(tq, tk, tv, a);
    return cudaGetLastError() == cudaSuccess ? OK : ERR_CUDA;
}

// The FP8 forward at d = 128: e4m3 Q, K ([heads][rows][128]) and V^T ([heads][128][ld],
// ld = fp8_vt_stride(Tk)), causal or not.
int launch_f8(const void *q8, const void *k8, const void *vt8, const float *qd, const float *kd, const float *vd,
              void *o, float *lse, int BH, int Tq, int Tk, int causal, float scale, cudaStream_t s)
{
    constexpr int D = 128;
    using L = FwdLayout<D, true>;
    CUtensorMap tq, tk, tv;
    int st = encode_tmap_3d(&tq, q8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, D, Tq, BH, 128, BR);
    if (st == OK)
        st = encode_tmap_3d(&tk, k8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, D, Tk, BH, 128, L::BC);
    if (st == OK)
        st = encode_tmap_3d_strided(&tv, vt8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Tk, D, BH, fp8_vt_stride(Tk), L::BC,
                                    D);
    if (st != OK)
        return st;
    FwdArgs a;
    a.o = static_cast<__nv_bfloat16 *>(o);
    a.lse = lse;
    a.BH = BH;
    a.Tq = Tq;
    a.Tk = Tk;
    a.left = -1;
    a.right = causal ? 0 : -1;
    a.bmask = nullptr;
    a.bm_per_head = 0;
    a.nqbm = (Tq + 127) / 128;
    a.nkbm = (Tk + 127) / 128;
    a.masked = 0;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.qd = qd;
    a.kd = kd;
    a.vd = vd;
    a.nqd = (Tq + 127) / 128;
    a.nkd = (Tk + 127) / 128;
    a.nqb = (Tq + L::NQ * BR - 1) / (L::NQ * BR);
    a.units = BH * a.nqb;
    // heads per group: K and V (e4m3) within ~48 MB of L2, which measured faster than 80 MB here
    const double kv_head = 2.0 * Tk * D;
    int g = (int)(48.0 * 1024 * 1024 / (kv_head > 1 ? kv_head : 1));
    const int grid = a.units < device_sm_count() ? a.units : device_sm_count();
    a.group = grid_aligned_group(g < 1 ? 1 : (g > BH ? BH : g), a.nqb, grid);
    a.timeout_ns = wait_timeout_ns();
    a.withhold = WITHHOLD_NONE;
    auto kernel = fwd_kernel<D, false, true>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES) != cudaSuccess)
        return ERR_CUDA;
    kernel<<<grid, L::NTHREADS, L::SMEM_BYTES, s>>>(tq, tk, tv, a);
    return cudaGetLastError() == cudaSuccess ? OK : ERR_CUDA;
}

}  // namespace

int fwd_fp8_launch(const void *q8, const void *k8, const void *vt8, const float *qd, const float *kd,
                   const float *vd, void *o, float *lse, int BH, int Tq, int Tk, int d, int causal, float scale,
                   cudaStream_t s)
{
    if (d != 128)
        return ERR_UNSUPPORTED;
    return launch_f8(q8, k8, vt8, qd, kd, vd, o, lse, BH, Tq, Tk, causal, scale, s);
}

int fwd_bf16_launch(const void *q, const void *k, const void *v, void *o, float *lse, int BH, int Tq,
                    int Tk, int d, const MaskSpec &mask, float scale, cudaStream_t s)
{
    switch (d) {
    case 64:
        return launch<64>(q, k, v, o, lse, BH, Tq, Tk, mask, scale, s);
    case 128:
        return launch<128>(q, k, v, o, lse, BH, Tq, Tk, mask, scale, s);
    case 256:
        return launch<256>(q, k, v, o, lse, BH, Tq, Tk, mask, scale, s);
    default:
        return ERR_UNSUPPORTED;
    }
}

int fwd_status_fetch_clear(cudaStream_t s, int *host_word)
{
    int zero = 0;
    if (cudaMemcpyFromSymbolAsync(host_word, g_fwd_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_fwd_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return ERR_CUDA;
    return OK;
}

}  // namespace fa
