// fa_internal.h -- host-side glue between the C-ABI layer (fa_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fa {

// Status codes, identical to fa_status in include/fa.h.
enum : int { OK = 0, ERR_INVALID_ARG = 1, ERR_UNSUPPORTED = 2, ERR_CUDA = 3, ERR_TIMEOUT = 4 };

// Encodes a 3-D tiled TMA map over a contiguous [planes][rows][inner] tensor
// with 128-byte swizzle; the box is [1][box_rows][box_inner].  Returns OK or
// ERR_CUDA (driver entry point missing, or the driver rejected the map).
int encode_tmap_3d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                   uint64_t inner, uint64_t rows, uint64_t planes, uint32_t box_inner,
                   uint32_t box_rows);

int device_sm_count();          // SMs of the current device (cached per device)
uint64_t wait_timeout_ns();     // bounded-wait limit for device spin waits

// Test-only build of the library (compiled with FA_TEST_WITHHOLD=1 into a separate
// shared object; the product library is built without it and has none of this): one
// launch may leave out one mbarrier arrive, so that a bounded wait of one CTA runs out
// and the timeout path (abort flag, drains, status word) runs.  The case is armed from
// the host, once, and taken by the next launch of the matching kernel:
//   WITHHOLD_FWD_KV   forward, CTA 0: query tile 0's release of its first K/V slot;
//                     the producer waits for that slot again (the MMA issuers and the
//                     softmax then wait for copies that never come)
//   WITHHOLD_FWD_EPI  forward, CTA 0: the "O~ final" signal of query tile 0 in the first
//                     unit; only that tile's softmax waits for it (epilogue)
//   WITHHOLD_BWD_DKV  backward tile loop, CTA 0: the "dK, dV complete" signal of its
//                     first unit; only the drain warpgroup waits for it
#ifndef FA_TEST_WITHHOLD
#define FA_TEST_WITHHOLD 0
#endif
enum : int { WITHHOLD_NONE = 0, WITHHOLD_FWD_KV = 1, WITHHOLD_FWD_EPI = 2, WITHHOLD_BWD_DKV = 3 };
#if FA_TEST_WITHHOLD
int test_withhold_take(int lo, int hi);   // the armed case if in [lo, hi] (then disarmed), else 0
#endif
// Heads per group of a persistent kernel's unit order.  gmax keeps the group's
// tensors within the L2 budget; where a group size in [gmax/2, gmax] makes a group
// a whole number of passes over the grid (levels units per head), the snake order
// of the passes balances the CTAs, so that size is taken.
inline int grid_aligned_group(int gmax, int levels, int grid)
{
    if (gmax < 1)
        gmax = 1;
    for (int g = gmax; g >= 1 && 2 * g >= gmax; --g)
        if (grid > 0 && ((long long)g * levels) % grid == 0)
            return g;
    return gmax;
}

// Allowed (row, key) pairs: key l is allowed for row r iff
//   r + Tk - Tq - left <= l <= r + Tk - Tq + right   (left, right = -1: that side unbounded)
// and, with a block mask, block[(r / 128) * nkbm + l / 128] != 0 for the head's mask
// ([heads][ceil(Tq / 128)][ceil(Tk / 128)] bytes in device memory, one mask per head when
// per_head, else one for all heads).  Causal is left = -1, right = 0.
struct MaskSpec {
    int left, right;
    const uint8_t *block;
    int per_head;
};
inline MaskSpec causal_spec(int causal) { return MaskSpec{-1, causal ? 0 : -1, nullptr, 0}; }

// Kernel launchers (arguments already validated by the ABI layer).
int fwd_bf16_launch(const void *q, const void *k, const void *v, void *o, float *lse, int BH,
                    int Tq, int Tk, int d, const MaskSpec &mask, float scale, cudaStream_t s);
int fwd_f32_launch(const float *q, const float *k, const float *v, float *o, float *lse, int BH,
                   int Tq, int Tk, int d, int causal, float scale, cudaStream_t s);
int fill_empty_launch(void *o, float *lse, size_t rows, int d, int elem_bytes, cudaStream_t s);

// FP8 forward (fa_fp8_sm103.cu, fa_fwd_sm103.cu): row stride in bytes of the
// transposed V codes, the quantization pass, and the forward over its output.
size_t fp8_vt_stride(int Tk);
int fp8_quantize_launch(const void *q, const void *k, const void *v, const float *signs, int BH, int Tq, int Tk,
                        int d, void *q8, void *k8, void *vt8, float *qd, float *kd, float *vd, cudaStream_t s);
int fwd_fp8_launch(const void *q8, const void *k8, const void *vt8, const float *qd, const float *kd,
                   const float *vd, void *o, float *lse, int BH, int Tq, int Tk, int d, int causal, float scale,
                   cudaStream_t s);
// encode_tmap_3d without swizzle (the box is plain row-major in shared memory)
int encode_tmap_3d_plain(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                         uint64_t inner, uint64_t rows, uint64_t planes, uint32_t box_inner, uint32_t box_rows);
// encode_tmap_3d with an explicit row stride in bytes (a multiple of 16)
int encode_tmap_3d_strided(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                           uint64_t inner, uint64_t rows, uint64_t planes, uint64_t row_stride,
                           uint32_t box_inner, uint32_t box_rows);

// Backward workspace; rows of every head are padded to Tq_pad = roundup(Tq, 128).
struct BwdWorkspace {
    float *lse2;     // [BH][Tq_pad]    -lse * log2(e); -inf for padding rows and rows without keys
    float *delta;    // [BH][Tq_pad]    -D_r = -(dO_r . O_r) (0 for padding rows)
    float *dq_acc;   // [BH][Tq_pad][d] fp32 dQ accumulator (unscaled)
    // deterministic mode: dq_acc holds int32 fixed point; per head the largest |V_l|_2
    // and |K_lc| (float bits), and per 128-row query block a bound on |dq_acc| (float bits)
    float *kvmax;    // [BH][2]
    int *bound;      // [BH][Tq_pad / 128]
};
size_t bwd_row_stride(int Tq);
size_t bwd_workspace_bytes(size_t BH, int Tq, int d);
BwdWorkspace bwd_workspace_carve(void *ws, int BH, int Tq, int d);
// stages: bit 0 = preprocess (D, lse2, zero dQ accumulator; fixed-point bounds),
// bit 1 = tile loop (dK, dV, dQ accumulation), bit 2 = dQ scale-and-round;
// kBwdDeterministic: dQ is accumulated as int32 fixed point (order-independent sums).
constexpr int kBwdDeterministic = 8;
// Every check of fa_bwd's arguments except the workspace's and the device's (no CUDA call).
int bwd_check_args(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO,
                   const void *dq, const void *dk, const void *dv, int B, int H, int Tq, int Tk, int d,
                   const MaskSpec &mask, float scale);
int bwd_launch(const void *q, const void *k, const void *v, const void *o, const float *lse,
               const void *dO, void *dq, void *dk, void *dv, int BH, int Tq, int Tk, int d,
               const MaskSpec &mask, float scale, const BwdWorkspace &ws, int stages, cudaStream_t s);

// Split-KV decode (fa_decode_sm103.cu): chunks per head and key tiles per
// chunk for these sizes, partial-state workspace bytes, query rows allowed per
// head at head width d, and the launch (split kernel + merge kernel).
void decode_split(int BH, int Tk, int *nsplit, int *tps);
size_t decode_workspace_bytes(int BH, int Tq, int Tk, int d);
int decode_max_rows(int d);
int decode_launch(const void *q, const void *k, const void *v, void *o, float *lse, int BH, int Tq, int Tk, int d,
                  int causal, float scale, void *workspace, cudaStream_t s);

// Device status words of the kernel translation units: read, add into *acc
// the first nonzero value, and clear.  Stream-ordered; the caller syncs.
int fwd_status_fetch_clear(cudaStream_t s, int *host_word);
int bwd_status_fetch_clear(cudaStream_t s, int *host_word);
int dec_status_fetch_clear(cudaStream_t s, int *host_word);

}  // namespace fa
