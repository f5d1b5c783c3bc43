// fa_common.cuh -- sm_103a building blocks shared by the attention kernels:
// mbarrier handoff with bounded waits, TMA tensor loads, tcgen05 MMA issue,
// tensor-memory allocation and load/store, and the UMMA descriptors.
//
// Everything here is inline PTX written for sm_103a (Blackwell Ultra):
//   * mbarrier.*                      -- producer/consumer phase handoff in shared memory
//   * cp.async.bulk.tensor (TMA)      -- HBM/L2 -> shared-memory tile copies, 128B swizzle
//   * tcgen05.mma / commit            -- 5th-generation tensor-core MMA into tensor memory
//   * tcgen05.alloc / ld / st / fence -- tensor memory (TMEM) management and access
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// ------------------------------------------------------------------ status
// Kernel-side failure codes written to a per-translation-unit device status
// word; the host reads them back in fa_sync_status().  Low byte: fa_status,
// next byte: the wait site that gave up.
constexpr int kStatusTimeout = 4;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }
__device__ __forceinline__ uint32_t warp_id() { return threadIdx.x >> 5; }

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// kHintNs > 0: the thread may stay suspended in the instruction up to about that many
// nanoseconds while the phase is incomplete (it resumes as soon as the phase completes),
// instead of the hardware's own limit; fewer polls of the barrier word.
template <uint32_t kHintNs = 0>
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    if constexpr (kHintNs == 0) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "r"(kHintNs)
            : "memory");
    }
    return ok;
}

// Unit of pass k of this CTA in a persistent loop over units.  SNAKE: passes
// alternate direction, so that with units sorted longest-first inside a group
// each CTA takes long and short units alike; otherwise every pass runs the same
// way.  The sequence increases with k, so a loop ends at the first unit past the
// end.
template <bool SNAKE>
__device__ __forceinline__ int snake_unit(int k)
{
    const int c = (SNAKE && (k & 1)) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
    return k * (int)gridDim.x + c;
}

// Per-CTA context of the bounded waits: a shared abort flag that every role
// polls, the kernel's device status word and the time limit.
struct WaitCtx {
    volatile int *abort;    // shared memory
    int *status;            // global memory (device status word)
    uint64_t timeout_ns;
};

// Waits for the phase of `bar` with parity `parity` to complete.  Gives up
// (returns false) when another role of the CTA has aborted, or after
// ctx.timeout_ns, in which case it raises the abort flag and records
// (site << 8 | FA_ERR_TIMEOUT) in the status word.  Never traps.
template <uint32_t kHintNs = 0>
__device__ __forceinline__ bool mbar_wait_loop(uint32_t bar, uint32_t parity, const WaitCtx &ctx, int site)
{
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait<kHintNs>(bar, parity))
            return true;
        if (*ctx.abort)
            return false;
        if ((it & 31u) == 0u && globaltimer_ns() - t0 > ctx.timeout_ns) {
            *ctx.abort = 1;
            atomicCAS(ctx.status, 0, (site << 8) | kStatusTimeout);
            __threadfence();
            return false;
        }
    }
}

template <uint32_t kHintNs>
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, const WaitCtx &ctx, int site)
{
    return mbar_wait_loop<kHintNs>(bar, parity, ctx, site);
}

// kInline: the slow path inlined instead of called.  Code that runs under a
// setmaxnreg register count cannot call out-of-line functions.  kHintNs: see
// mbar_try_wait.
template <bool kInline = false, uint32_t kHintNs = 0>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtx &ctx, int site)
{
    if (mbar_try_wait<kHintNs>(bar, parity))
        return true;
    if constexpr (kInline)
        return mbar_wait_loop<kHintNs>(bar, parity, ctx, site);
    else
        return mbar_wait_slow<kHintNs>(bar, parity, ctx, site);
}

// The same wait for roles whose warps run warp-collective instructions (tensor-memory
// loads, shuffles, votes) after it: the lanes vote, so the whole warp goes on only when
// every lane saw the phase complete, and leaves together otherwise.  Lanes of one warp
// can see different outcomes when a wait gives up: one lane may see the phase complete
// while another, polling a moment earlier, has seen the abort flag.  Every lane of the
// warp must call it.
//
// kLane0: lane 0 alone polls, its outcome goes to every lane, and the warp barrier that
// follows orders the other lanes' reads after lane 0's observation of the phase.  Where
// the tensor core's operand reads keep shared memory busy (the one-tile forward), 32
// lanes polling one barrier word take wavefronts from them; elsewhere the vote measured
// faster.
template <bool kInline = false, bool kLane0 = false, uint32_t kHintNs = 0>
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const WaitCtx &ctx, int site)
{
    if constexpr (kLane0) {
        uint32_t ok = 0;
        if ((threadIdx.x & 31u) == 0)
            ok = mbar_wait<kInline, kHintNs>(bar, parity, ctx, site) ? 1u : 0u;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        return ok != 0;
    } else {
        return __all_sync(0xffffffffu, mbar_wait<kInline, kHintNs>(bar, parity, ctx, site));
    }
}

// Limit of the teardown waits below, fixed and independent of the main waits' limit
// (which a caller may shorten): copies and MMAs already issued complete in
// microseconds, whatever the other roles of the CTA do.
constexpr uint64_t kDrainTimeoutNs = 4000000000ull;

// Teardown variant: bounded by time only (ignores the abort flag), used to
// drain copies and MMAs still in flight before the CTA releases its memory.
static __device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 31u) == 0u && globaltimer_ns() - t0 > kDrainTimeoutNs)
            return false;
    }
}

// Warpgroup register reallocation.  The sum over warpgroups must stay within
// the registers the block was launched with (threads x registers per thread).
template <uint32_t N>
__device__ __forceinline__ void regs_dealloc()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_alloc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load (x = element within a row, y = row, z = batch*head) into
// shared memory, completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y, int z)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// Same with an L2 cache-policy hint (createpolicy result).
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int x, int y, int z, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

// 3-D tiled reduce-add of a shared-memory box into global memory (fp32 or 32-bit integer
// add, after the map's data type), in the executing thread's current bulk group.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap *map, uint32_t src, int x, int y, int z)
{
    asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// 3-D tiled store of a shared-memory box (the map's box, same swizzle as the loads) to
// global memory, in the executing thread's current bulk group; rows past the tensor's
// extent are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrives once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same two products with e4m3 A and B (kind::f8f6f4: 32 elements of K per instruction).
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

#include "tmem_ldst.inc"

// TMEM address of (lane, column): lane in bits 31..16, column in bits 15..0.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col)
{
    return base + (lane << 16) + col;
}

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor for a 128-byte-swizzled operand (the layout
// TMA writes with CU_TENSOR_MAP_SWIZZLE_128B): rows of 128 bytes, 8-row
// (1024-byte) swizzle atoms.
//   K-major operand  : sbo = byte stride between 8-row groups, lbo unused.
//   MN-major operand : lbo = byte stride between 64-element column chunks,
//                      sbo = byte stride between 8-row groups along K.
// Bits: [0,14) addr>>4, [16,30) lbo>>4, [32,46) sbo>>4, [46,48) version 1,
// [61,64) layout 2 = SWIZZLE_128B.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma.kind::f16 with bf16 A and B and an
// fp32 accumulator.  a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn)
{
    return (1u << 4)                                // D format: f32
           | (1u << 7)                              // A format: bf16
           | (1u << 10)                             // B format: bf16
           | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor of tcgen05.mma.kind::f8f6f4 with e4m3 A and B (format code 0),
// both K-major, and an fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N)
{
    return (1u << 4)                                // D format: f32
           | (0u << 7) | (0u << 10)                 // A, B format: e4m3
           | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------ math
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (f32x2): two lanes of work per instruction.
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b0, float b1, float c0, float c1)
{
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ void fadd2(float &d0, float &d1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void fmul2(float &d0, float &d1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// max of three (one instruction on sm_100+)
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Four floats to e4m3 (round to nearest even, saturating at +-448); byte i = value i.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d)
{
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x = lo (low 16 bits), .y = hi
    return *reinterpret_cast<uint32_t *>(&h);
}

}  // namespace fa
