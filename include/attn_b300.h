/*
 * attn_b300.h -- C ABI of the B300 (sm_103a) exact attention library
 * (libattn_b300.so): forward pass, its split-KV and FP8 forms, the QK-RMSNorm
 * prologue and the backward pass.
 *
 * The operation (FlashAttention-3 deep dive, techknowgenie.com/posts/
 * 109164421204410442, introduction and section "3-stage asynchronous software
 * pipelining"): exact softmax attention, computed tile by tile with an online
 * softmax so the Sq x Sk score matrix never reaches device memory:
 *
 *     O[b,i,hq,:] = sum_j softmax_j( scale * Q[b,i,hq,:] . K[b,j,hkv,:] ) V[b,j,hkv,:]
 *     LSE[b,hq,i] = ln sum_j exp( scale * Q[b,i,hq,:] . K[b,j,hkv,:] )
 *
 * with j restricted to the visible keys. The pages do not define the causal
 * alignment, grouped-query heads or the LSE output; this library reads them as:
 *   - causal: key j is visible to query i iff j <= i + Sk - Sq (bottom-right);
 *   - GQA: hkv = hq / (Hq / Hkv), i.e. consecutive query heads share a KV head;
 *   - LSE is the natural logarithm; a row with no visible key gets O = 0 and
 *     LSE = -inf.
 *
 * Layouts (all dense, row-major, no padding):
 *   q, o : [B, Sq, Hq, d]     k, v : [B, Sk, Hkv, d]     lse : [B, Hq, Sq] fp32
 * O has the inputs' 16-bit type (bf16 or fp16); for E4M3 inputs it is bf16.
 *
 * Ownership and execution: every pointer is a DEVICE pointer owned by the
 * caller. The library allocates no device memory, holds no per-call workspace
 * and keeps no state between calls except a cached driver entry point, the
 * per-device kernel attributes, one device status word (below) and, once
 * attn_bwd has run on a device, one stream and two events of its own there
 * (see attn_bwd). Work is enqueued on `stream` (0 = legacy default stream)
 * and the call returns without synchronising; device-side failures surface
 * through attn_device_status(). All entry points are thread-safe.
 *
 * Error behaviour: argument checks run on the host before anything is
 * enqueued; a failed check returns its code and launches nothing.
 */
#ifndef ATTN_B300_H
#define ATTN_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* attn_stream_t; /* same type as cudaStream_t */

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, Hq % Hkv != 0,
                                 scale not finite and > 0, an index that does
                                 not fit in 32 bits */
    ATTN_ERR_UNSUPPORTED = 2, /* d not in {64, 128} (or 256 outside attn_fwd's
                                 bf16 / fp16 path), unknown dtype, device is
                                 not compute capability 10.3 (B300) */
    ATTN_ERR_MISALIGNED = 3,  /* a pointer not 16-byte aligned (TMA rule) */
    ATTN_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed */
    ATTN_ERR_TIMEOUT = 5      /* a kernel-internal wait gave up (watchdog, see
                                 attn_set_wait_limit_ns); reported by
                                 attn_device_status() only */
} attn_status_t;

typedef enum {
    ATTN_BF16 = 0,     /* q, k, v and o are bf16 */
    ATTN_FP8_E4M3 = 1, /* q, k, v are OCP E4M3 codes with unit scales; o is bf16 */
    ATTN_F16 = 2       /* q, k, v and o are IEEE fp16 (P is kept in fp16 too) */
} attn_dtype_t;

/* Rows of one FP8 scale block (per batch, head and block of consecutive
 * sequence rows; all d columns share the scale). */
#define ATTN_FP8_BLOCK_ROWS 64

/*
 * attn_fwd -- fused attention forward.
 *   q, k, v : device inputs in the layouts above, element type `dtype`
 *   o       : device output [B, Sq, Hq, d]: fp16 for ATTN_F16, else bf16
 *   lse     : device output, fp32 [B, Hq, Sq]
 *   B, Hq, Hkv, Sq, Sk, d : sizes; Hq % Hkv == 0; d in {64, 128}, or 256
 *             for ATTN_BF16 / ATTN_F16 (a kernel with one 128-row Q tile per
 *             unit and 64-key K/V tiles, since two d = 256 O accumulators do
 *             not fit the tensor memory beside the scores)
 *   causal  : 0 or non-zero (bottom-right causal mask)
 *   scale   : softmax scale applied to Q.K (finite, > 0; usually 1/sqrt(d))
 *   dtype   : attn_dtype_t; ATTN_FP8_E4M3 behaves as attn_fwd_fp8 with all
 *             block scales equal to 1
 * Every element count (B*S*H*d per tensor) must be below 2^31.
 * Returns an attn_status_t.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int Hq, int Hkv, int Sq, int Sk, int d,
             int causal, float scale, int dtype, attn_stream_t stream);

/*
 * attn_fwd_fp8 -- attention forward on E4M3 inputs with per-block scales
 * (FlashAttention-3 deep dive, section "FP8 low-precision arithmetic and
 * numerical stability": block quantisation with one scale per tile block,
 * FP8 products with fp32 accumulation, base-2 exponentials).
 *   q, k, v    : E4M3 codes, layouts as above
 *   q_scale    : fp32 [B, Hq,  ceil(Sq / 64)]
 *   k_scale,
 *   v_scale    : fp32 [B, Hkv, ceil(Sk / 64)]
 * The value of an element is code * scale of its (b, h, row / 64) block.
 * Scales must be finite and > 0. Other arguments as attn_fwd, with d in {64, 128}.
 */
int attn_fwd_fp8(const void* q, const void* k, const void* v,
                 const float* q_scale, const float* k_scale, const float* v_scale,
                 void* o, float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int d,
                 int causal, float scale, attn_stream_t stream);

/*
 * attn_splitkv_plan -- split count and workspace size for attn_fwd_splitkv.
 * Chooses the number of key ranges s (1..256, at least 4 K/V tiles of 128
 * keys per range) that minimises a simple cost model: rounds of work items,
 * ceil(items * s / num_sms), times the K/V tiles per range plus two tiles of
 * per-range overhead. 1 when the query side alone already fills the GPU in
 * whole rounds.
 *   causal          : as attn_fwd (a causal unit sees about half the tiles)
 *   num_sms         : SMs to fill; <= 0 queries the current device
 *   num_splits      : out, number of key ranges (>= 1)
 *   workspace_bytes : out, bytes of device workspace attn_fwd_splitkv needs
 *                     for that split count
 * Pure arithmetic unless num_sms <= 0. Returns an attn_status_t.
 */
int attn_splitkv_plan(int B, int Hq, int Sq, int Sk, int d, int causal, int num_sms,
                      int* num_splits, size_t* workspace_bytes);

/*
 * attn_fwd_splitkv -- the same forward pass with the keys cut into ranges
 * processed by separate work items, merged by a second kernel (the online-
 * softmax rescaling of the FlashAttention-3 deep dive, sections 2-3, applied
 * across key ranges: LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s).
 * Arguments as attn_fwd (dtype ATTN_BF16 or ATTN_F16, d in {64, 128}), plus:
 *   num_splits      : requested ranges, 1..256 (ranges of ceil(Sk/128/n) K/V
 *                     tiles; fewer if some would be empty)
 *   workspace       : device buffer owned by the caller, 16-byte aligned, at
 *                     least num_splits * B * Hq * Sq * (d + 1) * 4 bytes (what
 *                     attn_splitkv_plan reports); holds the per-range O (fp32)
 *                     and LSE between the two kernels; contents on entry are
 *                     ignored, on return undefined
 *   workspace_bytes : its size
 * Two kernels are enqueued on `stream`; calls that share a workspace must not
 * overlap. Errors: as attn_fwd; ATTN_ERR_INVALID_ARG for a bad split count or a
 * missing / too small workspace, ATTN_ERR_MISALIGNED for a misaligned one,
 * ATTN_ERR_UNSUPPORTED for ATTN_FP8_E4M3.
 */
int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                     int dtype, int num_splits, void* workspace, size_t workspace_bytes,
                     attn_stream_t stream);

/*
 * attn_fwd_splitkv_noalloc -- attn_fwd_splitkv for callers that may not
 * allocate device memory themselves: for example a plugin inside a host
 * application that owns every device buffer, or a latency-critical loop that
 * must not call cudaMalloc / cudaFree (which can synchronise the device) or
 * that runs under a fixed device-memory budget. It takes no workspace
 * argument: the per-range partial results go to a 64 MiB array built into
 * this library, which every GPU that loads the library holds until the
 * process exits. Nothing here allocates memory.
 *   Arguments as attn_fwd_splitkv without workspace / workspace_bytes.
 *   The workspace the call needs, num_splits' * B * Hq * Sq * (d + 1) * 4
 *   bytes (num_splits' = the non-empty ranges), must not exceed 64 MiB;
 *   larger requests return ATTN_ERR_INVALID_ARG without launching anything.
 *   The first successful call on a device (with that device current) looks
 *   up the array's device address; make that first call before any stream
 *   capture. A failed lookup is not cached: the next call tries again.
 *   Every call on a device shares the one array and it keeps the last call's
 *   contents; nothing in it needs clearing (each call writes every entry it
 *   reads), but calls whose kernels overlap on the GPU (other streams, other
 *   host threads) race on it: serialise them.
 * There is no counterpart on the source pages: this entry point exists only
 * for callers that cannot allocate. Returns an attn_status_t.
 */
int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int Hq, int Hkv, int Sq, int Sk, int d, int causal,
                             float scale, int dtype, int num_splits, attn_stream_t stream);

/*
 * attn_qk_rmsnorm -- the attention prologue "QKNorm across heads" (SGLang PR
 * 21503 analysis on the secrett2633 blog): RMSNorm of Q and of K in which each
 * token's whole hidden vector (all heads x d) shares one RMS:
 *     y[b, s, h, c] = x[b, s, h, c] * w[h * d + c]
 *                     / sqrt(eps + mean over (h', c') of x[b, s, h', c']^2)
 *   q, k       : device inputs [B, Sq, Hq, d] and [B, Sk, Hkv, d]
 *   q_weight,
 *   k_weight   : device weights [Hq * d] and [Hkv * d]
 *   q_out,
 *   k_out      : device outputs, same shapes as q and k; may be q and k
 *                themselves (in place), must not otherwise overlap them
 *   eps        : finite, >= 0
 *   dtype      : ATTN_BF16 or ATTN_F16, for every tensor here
 * Arithmetic in fp32, y rounded to nearest in the storage type. All pointers
 * 16-byte aligned; d in {64, 128}. One kernel on `stream`. Returns an
 * attn_status_t (ATTN_ERR_UNSUPPORTED for other dtypes or d).
 */
int attn_qk_rmsnorm(const void* q, const void* k, const void* q_weight, const void* k_weight,
                    void* q_out, void* k_out, int B, int Sq, int Sk, int Hq, int Hkv, int d,
                    float eps, int dtype, attn_stream_t stream);

/*
 * attn_quantize_fp8_e4m3 -- block quantiser producing attn_fwd_fp8 inputs
 * (same section of the FlashAttention-3 deep dive: per-block scale from the
 * block's local maximum).
 *   x     : device fp32 [B, S, H, d]
 *   codes : device uint8 [B, S, H, d] (E4M3)
 *   scale : device fp32 [B, H, ceil(S / 64)]
 * Per block of 64 rows of one head: s = amax / 448 (fp32 division), or 1 when
 * amax == 0; code = round-to-nearest-even, saturating E4M3 of x / s (fp32
 * IEEE division). A ragged last block uses its own rows only.
 * Sizes as attn_fwd (d in {64, 128}). Returns an attn_status_t.
 */
int attn_quantize_fp8_e4m3(const float* x, uint8_t* codes, float* scale,
                           int B, int S, int H, int d, attn_stream_t stream);

/*
 * attn_bwd_workspace_size -- bytes of device workspace attn_bwd needs:
 * 2 * B * Hq * Sq_pad * 4 with Sq_pad = Sq rounded up to a multiple of 128
 * (one fp32 per padded query row for D = rowsum(dO * O) and one for
 * LSE * log2(e)). Pure arithmetic. Returns an attn_status_t
 * (ATTN_ERR_INVALID_ARG for a null output or non-positive sizes).
 */
int attn_bwd_workspace_size(int B, int Hq, int Sq, size_t* workspace_bytes);

/*
 * attn_bwd -- exact attention backward pass: the gradients of
 * L = sum(d_o * O) for O = attn_fwd(q, k, v) with the same mask and scale.
 * The pages define the forward pass only; these are its derivatives by the
 * chain rule (no approximation), with P = exp(scale Q K^T - LSE):
 *     dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D),
 *     dQ = scale dS K,  dK = scale dS^T Q,
 * the query heads sharing a KV head summing into its dK and dV, and rows with
 * no visible key contributing nothing.
 *   q, k, v    : the forward's inputs (layouts as attn_fwd)
 *   o, lse     : the forward's outputs for them (lse in natural-log units)
 *   d_o        : device input dL/dO, [B, Sq, Hq, d], q's element type
 *   dq         : device output [B, Sq, Hq, d]
 *   dk, dv     : device outputs [B, Sk, Hkv, d]
 *   dtype      : ATTN_BF16 or ATTN_F16, for every 16-bit tensor here
 *   workspace  : device buffer owned by the caller, 16-byte aligned, at least
 *                attn_bwd_workspace_size bytes; contents on entry ignored, on
 *                return undefined
 * Other arguments as attn_fwd, with d in {64, 128}. P and dS are rounded to dtype before they
 * enter the tensor cores (fp32 accumulation); the gradients are rounded to
 * nearest in dtype. Three kernels run: row statistics on `stream`, then
 * dK/dV on `stream` and dQ on a second stream of the library's, side by side
 * on disjoint SMs (that stream waits for `stream` through an event before dQ,
 * and `stream` waits for it after; work later on `stream` sees all three
 * gradients, and the sequence can be captured into a CUDA graph). The first
 * call on a device creates that stream and its two events: make it before
 * any stream capture. If creating them fails, both kernels go on `stream`
 * one after the other. Every output element is written exactly once, so
 * results are deterministic and the same either way. Calls that share a
 * workspace must not overlap. Errors as
 * attn_fwd; ATTN_ERR_INVALID_ARG for a missing or too small workspace or for
 * B * Hq * Sq_pad >= 2^31, ATTN_ERR_MISALIGNED for a workspace or gradient
 * pointer not 16-byte aligned, ATTN_ERR_UNSUPPORTED for d = 256 or E4M3.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* d_o, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
             int Sk, int d, int causal, float scale, int dtype, void* workspace,
             size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_device_status -- synchronises `stream`, then returns and clears the
 * device status word: ATTN_OK, ATTN_ERR_TIMEOUT if a kernel's bounded wait
 * gave up since the last call (the kernel then abandoned its work and its
 * outputs are undefined), or ATTN_ERR_CUDA if the synchronisation failed.
 * The word is shared by every launch on the current device.
 */
int attn_device_status(attn_stream_t stream);

/*
 * attn_set_wait_limit_ns -- wall-clock limit of every bounded wait inside the
 * tensor-core kernels (a wait on a shared-memory barrier for a copy, a matrix
 * product or another warp). Default 1,000,000,000 (1 s). The limit is read
 * when a kernel is launched, so it applies to calls enqueued after this one
 * returns; it is process-wide (all devices, all threads).
 * The waits measure wall time (the GPU's global timer), not the time the
 * kernel actually ran: on a GPU shared with other contexts (time slicing,
 * preemption, a debugger) a healthy launch can be descheduled for longer
 * than the limit, and it then ends early with ATTN_ERR_TIMEOUT and undefined
 * outputs. Callers on such GPUs should raise the limit.
 *   ns : new limit, 1,000,000 (1 ms) .. 3,600,000,000,000 (1 h)
 * Returns ATTN_OK, or ATTN_ERR_INVALID_ARG (limit unchanged) outside that range.
 */
int attn_set_wait_limit_ns(unsigned long long ns);

/* attn_get_wait_limit_ns -- the limit currently in force, in nanoseconds. */
unsigned long long attn_get_wait_limit_ns(void);

/* attn_status_string -- static, human-readable name of a status code. */
const char* attn_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_B300_H */
