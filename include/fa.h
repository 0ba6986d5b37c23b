/*
 * fa.h -- C ABI of libfa: exact softmax attention on NVIDIA B300 (sm_103a).
 *
 * The operation (per batch b and head h, matrices row-major, head dim innermost):
 *
 *     S = scale * Q K^T,  masked entries -> -inf,
 *     O = softmax_rows(S) V,   lse_i = ln sum_j exp(S_ij),
 *     a row with no visible key gives O_i = 0 and lse_i = -inf.
 *
 * Sources: "Foundations -- Flash attention and efficient attention", sections 4
 * (the N x N score matrix Q K^T), 7-8 (softmax with the max subtracted) and 9 (the
 * 1/sqrt(d_k) score scale); "The Flash Attention" page, online recurrence panel
 * (the tiled one-pass algorithm the kernels use); "Flash attention and efficient
 * attention: Worked examples", Cell D (causal: query i sees keys j <= i) and Cell
 * D2 (l = 0: return the zero vector).  Key padding (keys j >= kv_len[b] masked)
 * is an extension the pages do not describe; it uses the same -inf mask.
 *
 * Conventions for every entry point below:
 *   - Tensors are dense, contiguous [B, H, N, d] (d innermost); lse is [B, H, N]
 *     float32.  All tensor pointers are DEVICE pointers owned by the caller; the
 *     library never allocates, frees or retains them.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream).  A returned FA_OK means the work was validated
 *     and enqueued; kernel-side failures are reported by fa_check_device_error.
 *   - The library never aborts the process, never calls exit and never traps.
 *     Invalid arguments return FA_ERR_INVALID or FA_ERR_UNSUPPORTED before any
 *     work is enqueued; fa_last_error_string() then describes the problem.
 *   - scale must be finite and > 0 (the pages' scale is 1/sqrt(d_k)).
 *   - Every kernel waits on its pipeline with a time limit; a wait that runs out
 *     ends the kernel early with garbage outputs and records FA_ERR_TIMEOUT, so
 *     a broken pipeline cannot hang the GPU.
 *   - Per device, the library keeps the device addresses of its own variables
 *     and the kernels' shared-memory limits.  It sets them up on the first call
 *     in each CUDA context and again whenever the current context has changed
 *     (for instance after the caller ran cudaDeviceReset), so such a reset is
 *     safe between calls; it is not safe while the library's work is in flight.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID = 1,     /* bad pointer, size, alignment or scale */
  FA_ERR_UNSUPPORTED = 2, /* valid but not served (head dim, device) */
  FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  FA_ERR_TIMEOUT = 4      /* a kernel's bounded pipeline wait ran out */
} fa_status;

typedef enum { FA_BF16 = 0, FA_FP32 = 1 } fa_dtype;

/*
 * fa_fwd -- attention forward, bfloat16 inputs and output, float32 lse.
 *   q, k, v : const bf16*, [B, H, N, d], 16-byte aligned.
 *   o       : bf16*, [B, H, N, d], 16-byte aligned; written.
 *   lse     : float*, [B, H, N] or NULL (then not written); natural-log
 *             log-sum-exp of each row's scaled, masked scores.
 *   d       : 64 or 128 (else FA_ERR_UNSUPPORTED).
 *   causal  : 0 -> no mask; 1 -> query i attends to keys j <= i ("Flash
 *             attention and efficient attention: Worked examples", Cell D);
 *             2 -> keys j < i only, the strictly causal setup of Cell D2, where
 *             query 0 sees no key (O = 0, lse = -inf).  Other values return
 *             FA_ERR_INVALID.  The same codes apply to every call below.
 * Runs on the tensor cores (tcgen05.mma, accumulators in tensor memory,
 * operands staged by TMA); the N x N scores never reach device memory.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, void* stream);

/*
 * fa_fwd_ex -- as fa_fwd, with the element type and key padding explicit.
 *   dtype  : FA_BF16 (tensor cores; d in {64, 128}) or FA_FP32 (float32 in and
 *            out on the CUDA cores; 1 <= d <= 128; q, k, v, o 4-byte aligned).
 *   kv_len : NULL, or a DEVICE pointer to B int32 values; keys j >= kv_len[b]
 *            are masked for every query of batch b.  Values are clamped to
 *            [0, N]; kv_len[b] = 0 gives O = 0 and lse = -inf for batch b.
 */
fa_status fa_fwd_ex(int dtype, const void* q, const void* k, const void* v, void* o, float* lse,
                    const int32_t* kv_len, int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * fa_fwd_qk -- as fa_fwd_ex, with Nq queries and Nk keys per (batch, head):
 * q, o are [B, H, Nq, d], lse is [B, H, Nq], k, v are [B, H, Nk, d].  The
 * queries are taken to be the last Nq positions of the key sequence (query i
 * at position i + Nk - Nq), so under causal = 1 query i sees keys
 * j <= i + Nk - Nq and the last query sees every key; causal = 2 excludes the
 * query's own position; a query that sees no key gets O = 0, lse = -inf.  With
 * Nq = Nk this is exactly fa_fwd_ex.  kv_len values are clamped to [0, Nk].
 * (The source pages treat Nq = Nk; this placement is the reading used for
 * decoding and chunked prefill.)
 */
fa_status fa_fwd_qk(int dtype, const void* q, const void* k, const void* v, void* o, float* lse,
                    const int32_t* kv_len, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                    void* stream);

/*
 * fa_bwd_workspace_size -- bytes of device workspace fa_bwd / fa_bwd_ex /
 * fa_bwd_qk need for this problem (N = the number of query rows): two float32
 * arrays of B*H*Np entries, Np = N rounded up to a multiple of 128 (per query row: -lse * log2(e), and -scale * D with
 * D = rowsum(dO * O)).  The content is private to the call.  Returns 0 for
 * non-positive sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * fa_bwd -- attention backward by recomputation, bfloat16 inputs, float32
 * gradients.  The probabilities are rebuilt from q, k and the forward's lse
 * instead of being read from a stored N x N matrix ("Question bank -- Flash
 * attention and efficient attention", the recomputation items); the gradient is
 * that of L = sum(O * dO) for the forward above:
 *     dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,  dS = P * (dP - D),
 *     dQ = scale dS K,  dK = scale dS^T Q.
 *   q, k, v, o, dO : const bf16*, [B, H, N, d], 16-byte aligned; o and lse are
 *                    the outputs of fa_fwd for the same q, k, v, scale, causal.
 *   lse            : const float*, [B, H, N] (required).
 *   dq, dk, dv     : float*, [B, H, N, d], 16-byte aligned; every element is
 *                    written once (contents on entry do not matter).  Each row
 *                    is summed in a fixed order, so repeated calls agree bit
 *                    for bit.  Three kernels: a row preprocess, one kernel per
 *                    128-key tile for dK and dV, one per 128-query tile for dQ.
 *   workspace      : device memory of at least fa_bwd_workspace_size(B, H, N, d)
 *                    bytes, 16-byte aligned, owned by the caller; its contents
 *                    on entry do not matter and are overwritten.
 *   d              : 128 (else FA_ERR_UNSUPPORTED).
 * Asynchronous on `stream` like every call here; the library allocates nothing.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 float* dq, float* dk, float* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                 float scale, int causal, void* stream);

/*
 * fa_bwd_ex -- as fa_bwd, with the key-padding lengths of fa_fwd_ex: kv_len is
 * NULL or a DEVICE pointer to B int32 values (clamped to [0, N]); keys
 * j >= kv_len[b] get zero probability, so their dK and dV rows are zero.
 */
fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                    const int32_t* kv_len, float* dq, float* dk, float* dv, void* workspace, size_t workspace_bytes,
                    int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * fa_bwd_qk -- as fa_bwd_ex, for the forward fa_fwd_qk: Nq queries and Nk keys
 * per head, the queries read as the last Nq positions of the key sequence, so a
 * causal mask is aligned bottom-right (query i sees keys j <= i + Nk - Nq, or
 * j < i + Nk - Nq when strict).  The pages treat Nq = Nk only; this is the
 * reading fa_fwd_qk documents.
 *   q, o, dO       : [B, H, Nq, d];  lse : [B, H, Nq];  dq : [B, H, Nq, d]
 *   k, v           : [B, H, Nk, d];  dk, dv : [B, H, Nk, d]
 *   kv_len         : NULL or a device pointer to B int32 values, clamped to [0, Nk]
 *   workspace      : at least fa_bwd_workspace_size(B, H, Nq, d) bytes
 * Query rows that see no key get dq = 0; keys no query sees get dk = dv = 0.
 * Errors as fa_bwd_ex; Nk < 1 is FA_ERR_INVALID.
 */
fa_status fa_bwd_qk(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                    const int32_t* kv_len, float* dq, float* dk, float* dv, void* workspace, size_t workspace_bytes,
                    int B, int H, int Nq, int Nk, int d, float scale, int causal, void* stream);

/*
 * fa_merge -- combine partial attention results computed over disjoint key
 * sets (split-key attention).  Part p gives, for every query row, an output O_p
 * already divided by its own normaliser and that normaliser's natural log lse_p
 * (what fa_fwd returns for the keys it was given).  The merge is the generic
 * rule of "Exercises -- Flash attention and efficient attention" (two- and
 * three-block merges), applied to the states (m = lse_p, l = 1, O~ = O_p):
 *     m = max_p lse_p,  f_p = e^(lse_p - m),  O = sum_p f_p O_p / sum_p f_p,
 *     lse = m + ln sum_p f_p.
 * A part with lse_p = -inf carries no weight; if all are -inf, O = 0 and
 * lse = -inf.
 *   dtype     : FA_BF16 or FA_FP32, the element type of o_parts and o.
 *   o_parts   : DEVICE, [n_parts][B][H][N][d], contiguous, element-aligned.
 *   lse_parts : DEVICE float*, [n_parts][B][H][N].
 *   o         : DEVICE, [B][H][N][d], written.
 *   lse       : DEVICE float*, [B][H][N], or NULL (not written).
 *   1 <= n_parts <= 4096; 1 <= d <= 256 (else FA_ERR_UNSUPPORTED).
 */
fa_status fa_merge(int dtype, const void* o_parts, const float* lse_parts, int n_parts, void* o, float* lse, int B,
                   int H, int N, int d, void* stream);

/*
 * fa_bwd_noalloc -- fa_bwd for callers that cannot allocate device memory.
 * The source pages have no counterpart: it exists only because of how some
 * callers manage memory.  A caller that cannot call cudaMalloc when it needs a
 * gradient cannot hand fa_bwd a workspace.  That includes code running inside
 * an allocator's own hooks, runtimes whose device pool is fixed and fully
 * handed out at start-up, and hosts whose policy forbids allocation after
 * initialisation.  This call instead uses a fixed device array inside the
 * library (2 * FA_BWD_NOALLOC_MAX_ROWS floats, 4 MiB).  Every GPU that loads
 * the library holds that array until the process exits.
 *   Arguments are those of fa_bwd without the workspace; q, k, v, o, dO, lse,
 *   dq, dk, dv are still the caller's device memory.  The library allocates
 *   nothing, through the CUDA runtime or otherwise.
 *   Limit: B * H * Np <= FA_BWD_NOALLOC_MAX_ROWS, where Np is N rounded up to
 *   a multiple of 128.  Larger problems return FA_ERR_UNSUPPORTED with a message
 *   naming the limit; use fa_bwd with a workspace for them.
 *   The first call on each device (and the first after the CUDA context has
 *   changed, e.g. after a cudaDeviceReset) looks up the array's device address
 *   with cudaGetSymbolAddress, so make that first call before any stream
 *   capture.
 *   All calls share the one array.  Calls whose work overlaps on the GPU (say,
 *   on two streams without ordering) corrupt each other's gradients; order
 *   them.  Stale contents left by an earlier call are harmless: every part of
 *   the array a call reads is first written by that call.
 */
#define FA_BWD_NOALLOC_MAX_ROWS 524288
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, float* dq, float* dk, float* dv, int B, int H, int N, int d, float scale,
                         int causal, void* stream);

/*
 * fa_std_fwd -- standard attention, the comparator the tiled method is measured
 * against ("Foundations -- Flash attention and efficient attention", section 10;
 * "Exercises", the memory-size and HBM-traffic exercises): the N x N score
 * matrix S = scale * Q K^T is written to device memory in full (float32), then
 * P = softmax_rows(S) (bf16, masked entries 0), then O = P V and lse.  Same
 * inputs, outputs, masks (causal 0 / 1 / 2, kv_len) and conventions as
 * fa_fwd_ex with FA_BF16; d = 64 or 128.  Not the fast path: it exists to
 * measure what keeping S and P on chip saves.
 *   workspace : device memory of at least fa_std_workspace_size(B, H, N) bytes,
 *               16-byte aligned, owned by the caller (S and P live there).
 * The products run on the tensor cores (tcgen05), the softmax on the CUDA cores.
 */
size_t fa_std_workspace_size(int B, int H, int N);
fa_status fa_std_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* kv_len,
                     void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                     void* stream);

/* Human-readable name of a status code (static storage). */
const char* fa_status_string(int status);

/* Detail of the last error returned on the calling thread (thread-local; ""
 * when none). */
const char* fa_last_error_string(void);

/*
 * fa_check_device_error -- synchronise `stream`, then take the library's device
 * status word on the current device (read and cleared in one atomic exchange,
 * enqueued on `stream`, so a bit set meanwhile by a kernel on another stream is
 * reported by a later call, never lost).  Returns FA_ERR_TIMEOUT if any kernel
 * since the last check gave up on a pipeline wait, FA_ERR_CUDA if the stream
 * reported an error or a kernel found its shared memory misaligned (it then did
 * nothing), else FA_OK.
 */
fa_status fa_check_device_error(void* stream);

/*
 * fa_set_wait_timeout_ms -- time limit for every pipeline wait inside the
 * kernels (default 1000 ms; values < 1 are raised to 1).  Process-wide.
 */
void fa_set_wait_timeout_ms(int ms);

/*
 * fa_debug_inject -- test hook.  code 1 makes the next fa_fwd bf16 launches'
 * producers stop feeding K/V tiles after the first one; code 2 makes the next
 * fa_bwd launches' dK/dV producers stop feeding Q/dO tiles after the first one;
 * code 3 makes their dQ producers stop feeding K/V tiles after the first one.
 * Every way the consumers' bounded waits run out, each CTA drains the copies
 * and tensor-core work it has in flight, frees its tensor memory and exits, and
 * fa_check_device_error reports FA_ERR_TIMEOUT.  code 0 (the default) turns it
 * off.  Nothing faults, traps or hangs either way.
 */
void fa_debug_inject(int code);

/* Library version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
