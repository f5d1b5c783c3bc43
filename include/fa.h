/*
 * fa.h -- C ABI of libfa.so: IO-aware exact attention for GB300 (sm_103a).
 *
 * Every tensor is a plain device pointer to a contiguous row-major array:
 *   q, o, dO, dq : [B][H][Tq][d]      k, v, dk, dv : [B][H][Tk][d]
 *   lse          : [B][H][Tq] float32 (natural-log log-sum-exp of the scaled scores)
 * "bf16" tensors hold IEEE bfloat16 values; "f32" tensors hold float32.
 * Every base pointer must be 16-byte aligned.
 *
 * Semantics.  S = scale * Q K^T per (b, h); P = softmax(S) row-wise over the
 * allowed keys; O = P V; lse_r = log sum_l exp(S_rl).  With causal != 0 key l
 * is allowed for query r iff l <= r + (Tk - Tq) (bottom-right alignment; for
 * Tq == Tk this is "query r sees keys l <= r").  A query row with no allowed
 * key gets O = 0, lse = -inf and zero gradients.  scale must be finite and
 * > 0 (the usual value is 1/sqrt(d)); there is no implicit default.
 *
 * Sources (page titles and sections):
 *   zerotofrontier.app "FlashAttention" (Efficient attention 12.3):
 *     "The forward pass" -- O_i = diag(l)^-1 O~ and lse_i = m + log l written once;
 *     "The causal mask, and the tiles you never visit" -- the three tile kinds;
 *     "What the forward pass leaves behind" -- O plus one lse per row is all
 *       the backward pass needs;
 *     "The backward pass, derived" -- D_r = dO_r . O_r, dS = P o (dP - D),
 *       key blocks outside, dQ accumulated by atomic additions.
 *   atlas.blal.pro "FlashAttention -- IO-Aware Exact Attention":
 *     "Online softmax" and "Recomputation in the backward pass".
 *
 * Ownership.  The caller allocates and owns every buffer, including the
 * backward workspace.  The library keeps no per-call state; tensor maps are
 * built on the host per call and passed by value.  Calls are thread-safe.
 *
 * Errors.  Calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 * legacy default stream).  The return value reports argument validation and
 * launch errors only.  A device-side failure (a bounded wait that timed out)
 * is recorded in a per-device status word and returned by fa_sync_status().
 * On any nonzero return, no kernel was launched and outputs are untouched,
 * except FA_ERR_CUDA from a failed launch.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, aliasing outputs, bad scale */
    FA_ERR_UNSUPPORTED = 2,   /* head width not supported, or the device is not sm_103 */
    FA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
    FA_ERR_TIMEOUT = 4        /* a device-side bounded wait ran out (from fa_sync_status) */
} fa_status;

typedef struct CUstream_st *fa_stream_t;   /* identical to cudaStream_t */

/*
 * Forward pass, bf16 in / bf16 O / f32 lse, fp32 accumulation on tcgen05
 * tensor cores.  d in {64, 128, 256}.  B, H, Tq, Tk >= 0; a call with
 * B*H*Tq == 0 is a no-op; Tk == 0 writes O = 0 and lse = -inf.
 * o and lse must not overlap q, k, v or each other.
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int H, int Tq, int Tk, int d, int causal, float scale,
           fa_stream_t stream);

/*
 * Forward pass with f32 tensors and plain fp32 FFMA arithmetic (no tensor
 * cores): the debug/reference-precision build of the same tiled online
 * softmax.  Same shapes, rules and errors as fa_fwd.
 */
int fa_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse,
               int B, int H, int Tq, int Tk, int d, int causal, float scale,
               fa_stream_t stream);

/*
 * fa_fwd under a sliding window and/or a block mask (zerotofrontier.app
 * "FlashAttention", "Dropout, block-sparsity, and other real-kernel
 * details": windows are functions of (r, l) computed inside the tile, and
 * tiles a block mask marks empty are skipped exactly as causal tiles are).
 * Key l is allowed for query row r iff
 *     r + Tk - Tq - window_left <= l <= r + Tk - Tq + window_right
 * (-1 leaves that side unbounded: (-1, 0) is fa_fwd's causal mask, (-1, -1)
 * no mask) and, when block_mask is not NULL, its byte for the 128 x 128 block
 * (r / 128, l / 128) is nonzero.  block_mask is device memory, row-major
 * [mask_per_head ? B*H : 1][ceil(Tq / 128)][ceil(Tk / 128)], read-only,
 * owned by the caller, not overlapping o or lse.  Rows with no allowed key
 * get O = 0 and lse = -inf.  Other arguments and errors as fa_fwd; a window
 * side below -1 or mask_per_head outside {0, 1} is FA_ERR_INVALID_ARG.
 */
int fa_fwd_masked(const void *q, const void *k, const void *v, void *o, float *lse,
                  int B, int H, int Tq, int Tk, int d, int window_left, int window_right,
                  const unsigned char *block_mask, int mask_per_head, float scale,
                  fa_stream_t stream);

/*
 * FP8 forward (atlas.blal.pro "FlashAttention -- IO-Aware Exact Attention",
 * "The version ladder: FA1 -> FA2 -> FA3", the FA3 entry: e4m3 tensor-core
 * products with block quantization and incoherent processing; "Honest caveats &
 * open questions": a precision trade-off).  Two calls: fa_fp8_quantize turns the
 * bf16 q, k, v of fa_fwd into e4m3 codes and fp32 dequantization factors, and
 * fa_fwd_fp8 runs the forward over them.
 *
 * fa_fp8_quantize: q [B][H][Tq][d], k, v [B][H][Tk][d] bf16 as in fa_fwd.
 * signs: d fp32 values of +-1.0 in device memory (the random rotation), or NULL
 * for none.  With signs, each row x of q and k becomes x diag(signs) H (H the
 * Sylvester Hadamard matrix, unnormalised, in fp32), which leaves q k^T unchanged
 * up to the factor d folded into the descales.  Then, per 128-row block of q and of
 * k, the block's largest |value| a maps to 448: code = e4m3(x * (448 / a)), both
 * steps rounded to fp32, the last to nearest even with saturation; descale =
 * a / 448 (/ sqrt(d) with signs).  v gets one scale per channel over all Tk keys
 * and is stored transposed.  Outputs (device memory, caller-owned, 16-byte
 * aligned, overlapping nothing else):
 *   q8 [B][H][Tq][d], k8 [B][H][Tk][d]   e4m3 codes (one byte each);
 *   vt8 [B][H][d][fa_fp8_vt_stride(Tk)]  e4m3 codes of v transposed; the bytes of a
 *                                        row past Tk are zero;
 *   q_descale [B][H][ceil(Tq/128)], k_descale [B][H][ceil(Tk/128)],
 *   v_descale [B][H][d]                  fp32.
 * d in {64, 128, 256}; other errors as fa_fwd.
 *
 * fa_fwd_fp8: O and lse of attention over q^ = q8 * q_descale (per row block),
 * k^ = k8 * k_descale, v^ = vt8^T * v_descale (per channel):
 *     O = softmax(scale q^ k^T) v^,  lse = log sum exp(scale q^ k^T)
 * with fa_fwd's causal convention, output layouts and empty-row rules.  The
 * probabilities enter the P V product as e4m3 (relative rounding error at most
 * 2^-4 each); scores and the row sums stay fp32.  d = 128 only, else
 * FA_ERR_UNSUPPORTED.  Arguments as produced by fa_fp8_quantize with the same
 * sizes (every buffer 16-byte aligned); o and lse must not overlap them.  With
 * no elements (Tq = 0, or Tk = 0 for the key side) a buffer may be NULL.
 */
size_t fa_fp8_vt_stride(int Tk);          /* bytes per row of vt8: Tk rounded up to 16 */
int fa_fp8_quantize(const void *q, const void *k, const void *v, const float *signs,
                    int B, int H, int Tq, int Tk, int d, void *q8, void *k8, void *vt8,
                    float *q_descale, float *k_descale, float *v_descale, fa_stream_t stream);
int fa_fwd_fp8(const void *q8, const void *k8, const void *vt8, const float *q_descale,
               const float *k_descale, const float *v_descale, void *o, float *lse,
               int B, int H, int Tq, int Tk, int d, int causal, float scale, fa_stream_t stream);

/*
 * Split-KV attention for decoding: the O and lse of fa_fwd for a few query
 * rows per head against a long key/value sequence (atlas.blal.pro
 * "FlashAttention -- IO-Aware Exact Attention", "Honest caveats & open
 * questions": one query row leaves the tiled kernel idle; FlashDecoding
 * splits the keys instead).  Each chunk of 32-key tiles of a head is reduced
 * to a partial (m, l, O~) per row by the online softmax, and the chunks are
 * merged by its rescale (zerotofrontier.app "FlashAttention", "The forward
 * pass", step 2.5).  Same layouts, causal convention (bottom-right), scale
 * and edge cases as fa_fwd; scores and P stay fp32.  Tq must be at most 16
 * (d = 64, 128) or 8 (d = 256), else FA_ERR_UNSUPPORTED: use fa_fwd for more
 * rows.  workspace: at least fa_decode_workspace_bytes(...) bytes, 256-byte
 * aligned, not overlapping any argument; contents on entry ignored.  The
 * chunking depends on the sizes only, so results do not depend on the device.
 */
size_t fa_decode_workspace_bytes(int B, int H, int Tq, int Tk, int d);   /* 0: invalid or unsupported sizes */
int fa_decode(const void *q, const void *k, const void *v, void *o, float *lse,
              int B, int H, int Tq, int Tk, int d, int causal, float scale,
              void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd and fa_bwd_deterministic need for these
 * sizes: a log2-domain copy of lse and the row terms D (each [B][H][Tq_pad]
 * f32), the dQ accumulator [B][H][Tq_pad][d] (f32, or int32 fixed point in
 * fa_bwd_deterministic), two f32 per head and one int32 per 128-row query
 * block (the fixed-point bounds), where Tq_pad rounds Tq up to a multiple of
 * 128; each region is 256-byte aligned.  Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int Tq, int Tk, int d);

/*
 * Backward pass, bf16 q, k, v, o, dO, dq, dk, dv; f32 lse.  o and lse must be
 * what fa_fwd returned for the same q, k, v, causal and scale.  d in {64, 128}
 * (d = 256 returns FA_ERR_UNSUPPORTED).  workspace must hold at least
 * fa_bwd_workspace_bytes(...) bytes, 256-byte aligned; its contents on entry
 * are ignored.  dq, dk, dv must not overlap any input, the workspace or each
 * other.  dQ is accumulated with fp32 atomic additions, so its last bits may
 * differ from run to run.
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dO, void *dq, void *dk, void *dv,
           int B, int H, int Tq, int Tk, int d, int causal, float scale,
           void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_bwd with dq bitwise the same on every run with the same inputs
 * (zerotofrontier.app "FlashAttention", "The backward pass, derived", "Which
 * loop goes outside?": dQ_i is a sum over key blocks added by different
 * thread blocks, and floating-point additions in arrival order make its last
 * bits vary between runs).  Here the contributions are added as int32 fixed
 * point, whose sums do not depend on the order: query block i (128 rows) uses
 * the grid 2^(e-30) where 2^e exceeds the bound 2 |dO_r|_2 max_l |V_l|_2
 * max |K| of every partial sum of its rows (the rows of P sum to one), so
 * nothing overflows and each term is rounded to about 1e-9 of that bound.
 * dk and dv are computed as by fa_bwd.  It costs one more pass over K and V
 * (the per-head maxima) and the conversions.  Non-finite inputs give no
 * meaningful dq.  Arguments, workspace, validation and errors are those of
 * fa_bwd.
 */
int fa_bwd_deterministic(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, const void *dO, void *dq, void *dk, void *dv,
                         int B, int H, int Tq, int Tk, int d, int causal, float scale,
                         void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Backward of fa_fwd_masked: the gradients under the same window and block
 * mask (see fa_fwd_masked for their meaning, layout and ownership; o and lse
 * must come from fa_fwd_masked with the same mask).  Each 128-key block
 * visits only the query blocks that its window and mask admit.
 * deterministic = 1 selects fa_bwd_deterministic's order-independent dQ.
 * Other arguments, workspace and errors as fa_bwd; window sides below -1,
 * mask_per_head or deterministic outside {0, 1} are FA_ERR_INVALID_ARG.
 */
int fa_bwd_masked(const void *q, const void *k, const void *v, const void *o,
                  const float *lse, const void *dO, void *dq, void *dk, void *dv,
                  int B, int H, int Tq, int Tk, int d, int window_left, int window_right,
                  const unsigned char *block_mask, int mask_per_head, int deterministic,
                  float scale, void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * One stage of fa_bwd, for callers that schedule or time the three kernels
 * separately: stage 1 computes D_r = dO_r . O_r and the log2-domain lse into
 * the workspace and zeroes the dQ accumulator; stage 2 runs the tile loop
 * (recomputes P from lse, writes dK and dV, adds dQ into the accumulator);
 * stage 3 scales the accumulator by `scale` and writes dq.  Running stages
 * 1, 2, 3 in that order on one stream with the same arguments and workspace
 * is exactly fa_bwd.  Arguments, validation and errors are those of fa_bwd;
 * stage outside 1..3 returns FA_ERR_INVALID_ARG.
 */
int fa_bwd_stage(int stage, const void *q, const void *k, const void *v, const void *o,
                 const float *lse, const void *dO, void *dq, void *dk, void *dv,
                 int B, int H, int Tq, int Tk, int d, int causal, float scale,
                 void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Size of the fixed device scratch array behind fa_bwd_noalloc (64 MiB).  It
 * holds fa_bwd_workspace_bytes(B, H, Tq, Tk, d) bytes, about 520 bytes per
 * padded query row at d = 128 and 264 at d = 64, when B*H*Tq_pad is at most
 * about 129,000 rows at d = 128 (B8 H8 T1920, B1 H32 T3840; not B8 H8 T2048)
 * or 254,000 rows at d = 64 (B8 H16 T1920), where Tq_pad rounds Tq up to 128.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * fa_bwd for callers that cannot allocate device memory.  The pages have no
 * counterpart: this serves callers that are handed only their input and
 * output buffers and may not call cudaMalloc -- plug-ins whose host framework
 * owns all device memory and offers them no allocator, or latency-critical
 * code that cannot take cudaMalloc's implicit device synchronisation.
 * Arguments, results and errors are those of fa_bwd without the workspace:
 * the scratch comes from a fixed array of FA_BWD_NOALLOC_SCRATCH_BYTES that
 * the library keeps in device memory (each device holds it until the process
 * exits).  The call allocates nothing.
 *   - Arguments are checked as fa_bwd checks them (FA_ERR_INVALID_ARG,
 *     FA_ERR_UNSUPPORTED for d = 256) before anything else.  Then sizes whose
 *     fa_bwd_workspace_bytes(...) exceeds FA_BWD_NOALLOC_SCRATCH_BYTES return
 *     FA_ERR_UNSUPPORTED, still before any CUDA call; use fa_bwd with a
 *     caller-owned workspace for those.
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress, with that device current) and caches it with the
 *     current CUDA context; make that first call before any stream capture.
 *     A call under a different context (after cudaDeviceReset, for one) looks
 *     the address up again, so make the first call after a reset before any
 *     capture too.
 *   - Every call on a device shares the one array.  Each call rewrites all of
 *     the scratch it uses before reading it (the dQ accumulator is zeroed),
 *     so nothing carries over between calls, but calls that overlap on the
 *     GPU (different streams or threads on one device) race and corrupt each
 *     other's results: order them, e.g. on one stream.
 */
int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dO, void *dq, void *dk, void *dv,
                   int B, int H, int Tq, int Tk, int d, int causal, float scale,
                   fa_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device: FA_OK, FA_ERR_TIMEOUT (a kernel's bounded wait ran out;
 * its outputs are invalid) or FA_ERR_CUDA (the synchronise failed).
 */
int fa_sync_status(fa_stream_t stream);

/* Static, never-NULL description of a status code. */
const char *fa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
