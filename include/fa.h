/*
 * fa.h -- C ABI of the GB300 (sm_103a) FlashAttention-2 backward library.
 *
 * Operation (FlashAttention-2 backward as described by boostr 0.1.0,
 * src/ops/cuda/attention/flash_bwd.rs, doc comment of
 * flash_attention_bwd_impl, "Two-step process"):
 *   step 1 (preprocess)  D_i   = sum_c dO_ic * O_ic              (fp32)
 *   step 2 (main)        P_ij  = exp(scale * <Q_i, K_j> - LSE_i)  (masked -> 0)
 *                        dV_j  = sum_i P_ij dO_i
 *                        dS_ij = P_ij * (<dO_i, V_j> - D_i)
 *                        dK_j  = scale * sum_i dS_ij Q_i
 *                        dQ_i  = scale * sum_j dS_ij K_j
 * dK and dV of a key/value head are summed over the H / H_kv query heads
 * that share it; query head h uses key/value head h / (H / H_kv).
 * Query i sits at key position p_i = i + (S_k - S_q) (bottom-right alignment).
 * Causal masking keeps key j for query i iff j <= p_i.  A sliding window of
 * size w > 0 (fa_bwd_ex / fa_fwd_ex; boostr autograd_attention.rs carries
 * window_size through FlashAttentionConfig into both passes, 0 = none) also
 * drops keys with p_i - j >= w and, when not causal, keys with j - p_i >= w:
 * a causal query sees its w most recent keys, itself included.
 *
 * Layouts (shape checks of flash_attention_bwd_impl in flash_bwd.rs and of
 * flash_attention_backward in rustytorch rtx-flash-metal-attention
 * backward.rs): every tensor is dense row-major,
 *   Q, O, dO, dQ : [B, H,    S_q, d]   element type `dtype`
 *   K, V, dK, dV : [B, H_kv, S_k, d]   element type `dtype`
 *   LSE, D       : [B, H,    S_q]      float32, natural-log log-sum-exp of
 *                                      the scaled scores (-inf for a row
 *                                      that sees no key)
 *
 * Pointers are DEVICE pointers unless an entry point says otherwise.  The
 * caller owns every buffer it passes; the library owns an internal workspace
 * (fp32 dQ accumulator, D and a padded copy of LSE) cached per
 * (device, stream) and released by fa_shutdown().  All calls are
 * asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream):
 * they return after enqueueing, results are valid in stream order, inputs
 * are never modified and outputs are fully overwritten.
 *
 * Errors: every entry point returns an fa_status.  Argument errors are
 * detected on the host before anything is enqueued (FA_ERR_INVALID_ARG /
 * FA_ERR_UNSUPPORTED) and fa_last_error() then names the argument and the
 * reason, like the InvalidArgument { arg, reason } errors of flash_bwd.rs.
 * CUDA launch failures give FA_ERR_CUDA.  Device-side waits are bounded: a
 * kernel whose wait runs out records it in the workspace error word and
 * returns; fa_check_device(stream) reports it as FA_ERR_TIMEOUT.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FA_F32 = 0, FA_F16 = 1, FA_BF16 = 2 } fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* bad pointer, shape, dtype, scale or alignment */
    FA_ERR_UNSUPPORTED = 2, /* valid but not implemented (head dim not 32/64/96/128/256) */
    FA_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed */
    FA_ERR_TIMEOUT = 4,     /* a device-side bounded wait ran out */
    FA_ERR_NOMEM = 5        /* workspace allocation failed */
} fa_status;

/*
 * fa_bwd -- full FlashAttention-2 backward: preprocess D, then dQ, dK, dV.
 *   dO, Q, O      : [B, H, S_q, d]  dtype, 16-byte aligned
 *   K, V          : [B, H_kv, S_k, d] dtype, 16-byte aligned
 *   LSE           : [B, H, S_q] float32, 4-byte aligned
 *   dQ            : [B, H, S_q, d]  dtype, written
 *   dK, dV        : [B, H_kv, S_k, d] dtype, written (rows no query sees get 0)
 *   B, H, H_kv, S_q, S_k > 0, H % H_kv == 0, d in {32, 64, 96, 128, 256}
 *   scale         : finite, > 0 (usually 1/sqrt(d))
 *   causal        : 0 or 1
 *   dtype         : fa_dtype (F32, F16, BF16); accumulation is fp32
 *   stream        : cudaStream_t
 * F16/BF16 run tcgen05 tensor-core kernels: one for d <= 128 (d = 32 and 96
 * on the d = 64 and 128 instances, the missing columns read as zeros), one
 * for d = 256 (64-key tiles, dK and dV accumulated transposed); F32 runs an
 * FFMA kernel.
 * dQ is reduced across key tiles with fp32 atomics, so dQ may differ in the
 * last bits between runs (flash_bwd.rs, "dQ must be zeroed -- backward uses
 * atomicAdd"); dK and dV are deterministic.  fa_bwd_ex(..., deterministic = 1)
 * makes dQ reproducible too.
 */
int fa_bwd(const void* dO, const void* Q, const void* K, const void* V, const void* O,
           const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int H_kv, int S_q,
           int S_k, int d, float scale, int causal, int dtype, void* stream);

/*
 * fa_bwd_preprocess -- step 1 alone (flash_bwd.rs, "Step 1: Preprocessing --
 * compute D = rowsum(dO (.) O) per query position"):
 *   D[b, h, i] = sum_c dO[b, h, i, c] * O[b, h, i, c], accumulated in fp32.
 *   dO, O : [B, H, S_q, d] dtype, 16-byte aligned;  D : [B, H, S_q] float32.
 */
int fa_bwd_preprocess(const void* dO, const void* O, float* D, int B, int H, int S_q, int d,
                      int dtype, void* stream);

/*
 * fa_fwd -- attention forward helper producing the O and LSE the backward
 * consumes (boostr autograd_attention.rs, var_flash_attention saves
 * q, k, v, output, lse):  O_i = sum_j softmax_j(scale <Q_i, K_j>) V_j and
 * LSE_i = log sum_j exp(scale <Q_i, K_j>) over the visible keys.
 *   Q : [B, H, S_q, d], K, V : [B, H_kv, S_k, d], O : [B, H, S_q, d] dtype;
 *   LSE : [B, H, S_q] float32.  Rows that see no key get O = 0, LSE = -inf.
 * F16/BF16 run a tcgen05 tensor-core kernel (fp32 accumulation, online
 * softmax over 128-key tiles, 64-key tiles at d = 256); F32 runs an FFMA
 * kernel.
 */
int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
           int H_kv, int S_q, int S_k, int d, float scale, int causal, int dtype, void* stream);

/*
 * fa_bwd_ex / fa_fwd_ex -- fa_bwd / fa_fwd with the remaining arguments of the
 * pages' flash_attention_bwd / flash_attention_fwd calls (boostr
 * autograd_attention.rs, FlashAttentionBackward::backward and
 * var_flash_attention):
 *   window_size   : >= 0; 0 = no window, else the band described at the top.
 *                   Key tiles outside the band are skipped, not just masked.
 *                   A negative value gives FA_ERR_INVALID_ARG.
 *   deterministic : 0 = dQ reduced with fp32 atomics (as fa_bwd; the pages'
 *                   atomicAdd accumulation), bits may vary between runs;
 *                   1 = bitwise reproducible dQ: F16/BF16 add each 128x128
 *                   dQ tile's per-key-tile contributions in key-tile order
 *                   (the CTAs pass a turn counter in the workspace along; each
 *                   CTA takes its tile from a ticket counter in the order the
 *                   CTAs start and only ever waits for CTAs that started
 *                   before it, and every wait is bounded); F32 computes
 *                   dQ in its own kernel, each row summed over keys in index
 *                   order.  Other values give FA_ERR_INVALID_ARG.
 * dK and dV are bitwise reproducible in both modes.  Every other argument,
 * layout and result is that of fa_bwd / fa_fwd, which are these calls with
 * window_size = 0 and deterministic = 0.  The pages' backward rejects
 * window_size != 0; this library implements it.
 */
int fa_bwd_ex(const void* dO, const void* Q, const void* K, const void* V, const void* O,
              const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int H_kv, int S_q,
              int S_k, int d, float scale, int causal, int window_size, int deterministic, int dtype,
              void* stream);
int fa_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
              int H_kv, int S_q, int S_k, int d, float scale, int causal, int window_size, int dtype,
              void* stream);

/*
 * fa_bwd_host -- fa_bwd on HOST buffers (same arguments and layouts, every
 * pointer a host pointer; pinned memory gives full copy bandwidth and lets
 * copies overlap compute).  Copies the inputs to device buffers cached per
 * (device, stream), runs the backward on `stream`, copies dQ, dK, dV back and
 * returns once they are in the host buffers.  Problems with more than 32 MiB
 * of input are split into up to 4 chunks of whole (batch, kv head) units:
 * chunk c's inputs are copied on a library-owned stream while chunk c-1
 * computes on `stream` and chunk c-2's results are copied back on a second
 * library-owned stream.  Results are those of fa_bwd (dQ up to the order of
 * its fp32 reduction).
 */
int fa_bwd_host(const void* dO, const void* Q, const void* K, const void* V, const void* O,
                const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int H_kv, int S_q,
                int S_k, int d, float scale, int causal, int dtype, void* stream);

/*
 * fa_bwd_noalloc -- fa_bwd for callers that cannot allocate device memory
 * (an allocator or memory pool that owns the GPU's memory, a host that must
 * not see the implicit synchronization of cudaMalloc / cudaFree, a runtime
 * that forbids libraries from allocating).  The pages have no counterpart of
 * this entry point.  Same arguments, layouts and results as fa_bwd; the
 * caller still passes every input and output buffer, and the library's
 * scratch comes from one fixed 32 MiB array compiled into the library, which
 * every GPU that loads the library holds until the process exits.
 *   * A shape needs 256 + 8*B*H*ceil(S_q/128)*128 + 4*B*H*S_q*d bytes of
 *     scratch (parts rounded up to 256 bytes); beyond 32 MiB the call returns
 *     FA_ERR_INVALID_ARG ("scratch: ...") and launches nothing.
 *   * The first call on a device looks the array's device address up and
 *     enqueues the clearing of its error words on `stream`: make that first
 *     call before any stream capture.
 *   * Every call shares the array (it keeps the last call's contents; each
 *     call re-zeroes what must start at zero).  Calls whose GPU work overlaps,
 *     e.g. on different streams, race: keep them in one stream's order.
 *   * The main kernel is the one fa_bwd would run for the same arguments.
 *   * Bounded-wait timeouts of this variant are recorded in the array and
 *     reported (then cleared) by fa_check_device(stream), as for fa_bwd.
 */
int fa_bwd_noalloc(const void* dO, const void* Q, const void* K, const void* V, const void* O,
                   const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int H_kv,
                   int S_q, int S_k, int d, float scale, int causal, int dtype, void* stream);

/* Workspace bytes fa_bwd / fa_bwd_ex need for a shape (informational; the
 * library allocates and caches it itself): error words, padded LSE and D
 * copies, the fp32 dQ accumulator and the deterministic mode's turn counters. */
size_t fa_bwd_workspace_bytes(int B, int H, int S_q, int d);

/* Synchronizes `stream`, then returns FA_ERR_TIMEOUT if a kernel of this
 * library on that stream, or an fa_bwd_noalloc call on this device, recorded
 * a bounded-wait timeout since the last check (clearing the record), else
 * FA_OK (or FA_ERR_CUDA). */
int fa_check_device(void* stream);

/*
 * Per-kernel timing of fa_bwd calls (CUDA events recorded on the caller's
 * stream around each of the three launches: preprocess, main, dQ finalise).
 * fa_profile(1) clears the record and starts collecting, fa_profile(0)
 * stops.  fa_profile_read synchronizes on the recorded events and returns
 * the summed milliseconds per kernel in ms[0..2] and the number of fa_bwd
 * calls recorded.  Recording adds event records to the stream, nothing else.
 */
int fa_profile(int enable);
int fa_profile_read(float* ms, int* calls);

/*
 * fa_selftest_timeout -- failure-detection self-test (not needed in normal
 * use): launches on `stream` one CTA that waits, through the same bounded wait
 * the backward kernel uses, on a barrier nothing ever completes, with a limit
 * of `limit_ns` nanoseconds (0 < limit_ns <= 1e9).  The wait runs out and the
 * kernel records a timeout in the stream's workspace error word and returns;
 * fa_check_device(stream) then reports FA_ERR_TIMEOUT and the CUDA context
 * stays usable.  The bounded waits of the backward are the device side of the
 * pages' KernelError reporting (boostr flash_bwd.rs launch errors).
 */
int fa_selftest_timeout(unsigned long long limit_ns, void* stream);

/* Thread-local text of the last error ("arg: reason"); "" if none. */
const char* fa_last_error(void);

/* Frees every cached workspace of the calling process (all devices).  Must
 * not race with calls in flight. */
void fa_shutdown(void);

/* Library version string. */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
