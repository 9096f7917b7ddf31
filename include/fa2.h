/*
 * fa2.h - C ABI of the GB300 (sm_103a) FlashAttention-2 forward library.
 *
 * The operation. Exact scaled-dot-product attention, forward pass only, as
 * defined for FlashAttention-2 in "A Case Study in CUDA Kernel Fusion:
 * Implementing FlashAttention-2 on NVIDIA Hopper Architecture using the
 * CUTLASS Library" (abstract: online softmax fused with two back-to-back
 * GEMMs), restricted to the slice listed under "Kernel Specification" in
 * "FlashAttention-2 from scratch on Ampere, Part 1" (lubitschian.com/flash/
 * Part-1): non-causal, equal query/key/value sequence lengths, sequence
 * lengths divisible by the block size, 16-bit (bf16 or fp16) inputs and
 * outputs, softmax in fp32. For every batch b, query head h and query row i:
 *
 *     S[j]   = scale * <Q[b,h,i,:], K[b,g(h),j,:]>        j = 0 .. N-1
 *     O[b,h,i,:] = sum_j softmax(S)[j] * V[b,g(h),j,:]
 *     LSE[b,h,i] = ln sum_j exp(S[j])                     (natural log)
 *
 * with g(h) = h / (Hq / Hkv). Grouped KV heads (Hq > Hkv) use the query-head
 * packing named in "FlashAttention-3 for Inference: INT8 Quantization and
 * Query Head Packing for MQA/GQA" (Colfax Research author page): the Hq/Hkv
 * query heads that share a KV head are consecutive, so their rows form one
 * contiguous block of Hq/Hkv * N query rows that is processed against a
 * single stream of K/V tiles. The N x N score matrix never reaches memory.
 *
 * Data layout. All tensors are dense, row-major, caller-owned device memory:
 *     q, o : [B, Hq,  N, d]   16-bit elements (bf16 or fp16, same for all)
 *     k, v : [B, Hkv, N, d]   16-bit elements
 *     lse  : [B, Hq,  N]      fp32
 * Every pointer must be 16-byte aligned. Outputs are fully overwritten.
 *
 * Execution. Calls are asynchronous on `stream` (0 = legacy default stream);
 * each forward call launches exactly one kernel, fa2_bwd three (in stream
 * order). The library allocates no memory per call;
 * it owns one status word per device (a __device__ variable), which the
 * kernel sets if one of its bounded waits gives up.
 *
 * Errors. Argument errors (FA2_ERR_INVALID_ARG) and unsupported sizes or
 * devices (FA2_ERR_UNSUPPORTED) are detected on the host before anything is
 * launched. FA2_ERR_CUDA means a CUDA call of the library failed; each launch
 * is judged by its own return code, so an error the caller left pending does
 * not turn a successful call into a failure, and a failed call leaves none
 * of its own (non-sticky) errors pending. No entry point exits the process
 * or throws.
 */
#ifndef FA2_H_
#define FA2_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA2_BF16 = 0,
    FA2_FP16 = 1
} fa2_dtype;

typedef enum {
    FA2_OK = 0,
    FA2_ERR_INVALID_ARG = 1,  /* NULL/misaligned pointer, non-positive size,
                                 Hq % Hkv != 0, scale not finite and > 0 */
    FA2_ERR_UNSUPPORTED = 2,  /* d not in {64, 128}, N % 128 != 0, sizes past
                                 32-bit coordinates, or a device that is not
                                 compute capability 10.3 */
    FA2_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
    FA2_ERR_TIMEOUT = 4,      /* the kernel's watchdog gave up on a wait */
    FA2_ERR_BOUNDS = 5        /* debug builds only (libfa2_debug.so, compiled
                                 with FA2_DEBUG): a device-side bounds check
                                 failed and the access was skipped */
} fa2_status;

/*
 * Multi-head attention forward (Hq == Hkv == H).
 *   q, k, v : [B, H, N, d] 16-bit, device, 16-byte aligned (inputs, read only)
 *   o       : [B, H, N, d] 16-bit, device (output)
 *   lse     : [B, H, N] fp32, device (output, natural-log logsumexp of the
 *             scaled scores)
 *   B, H, N : positive; N a multiple of 128
 *   d       : 64 or 128
 *   scale   : finite, > 0 (usually 1/sqrt(d))
 *   dtype   : element type of q, k, v and o
 *   stream  : CUDA stream the kernel is queued on
 * Returns FA2_OK once the kernel is queued; FA2_ERR_* otherwise, and then
 * nothing was launched.
 */
fa2_status fa2_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int N, int d, float scale, fa2_dtype dtype,
                   cudaStream_t stream);

/*
 * Grouped-KV (GQA/MQA) attention forward. Same contract as fa2_fwd, with
 * q, o : [B, H_q, N, d], k, v : [B, H_kv, N, d], lse : [B, H_q, N] and
 * H_q a multiple of H_kv; query head h reads KV head h / (H_q / H_kv).
 * fa2_fwd(..., H, ...) is fa2_fwd_gqa(..., H, H, ...).
 */
fa2_status fa2_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int H_q, int H_kv, int N, int d, float scale,
                       fa2_dtype dtype, cudaStream_t stream);

/*
 * General attention forward: query and key lengths may differ and need not be
 * multiples of 128, with an optional causal mask. This goes beyond the
 * "Kernel Specification" of "FlashAttention-2 from scratch on Ampere,
 * Part 1" (equal lengths, non-causal, lengths divisible by the block size),
 * which excludes these variants; they are built here as extensions.
 *   q, o : [B, H_q, N_q, d]; k, v : [B, H_kv, N_k, d]; lse : [B, H_q, N_q]
 *   N_q, N_k : positive, any value
 *   causal   : 0 or 1. With 1, query row i attends key j iff
 *              j < min(N_k, i + 1 + N_k - N_q) (the mask aligned to the end of
 *              the key sequence; j <= i when N_q == N_k). A row with no
 *              allowed key gets O = 0 and LSE = -inf.
 * Other arguments, layouts and errors as fa2_fwd_gqa (causal not in {0, 1}
 * is FA2_ERR_INVALID_ARG; no N % 128 restriction). The non-causal
 * equal-length case with N % 128 == 0 runs the same kernel as fa2_fwd_gqa.
 */
fa2_status fa2_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int H_q, int H_kv, int N_q, int N_k, int d, float scale,
                      int causal, fa2_dtype dtype, cudaStream_t stream);

/*
 * FP8 attention forward with in-kernel scaling: the inference variant named
 * by "FlashAttention-3 for Inference: INT8 Quantization and Query Head
 * Packing for MQA/GQA" (Colfax Research author page: quantised inputs,
 * in-kernel pre-processing by specialised warps, query-head packing). The
 * pages give no more than that; the form here:
 *   q       : [B, H_q, N, d] e4m3 codes (OCP FP8 E4M3, one byte each), device
 *   k, v    : [B, H_kv, N, d] e4m3 codes, device
 *   q_descale, k_descale, v_descale : [B * H_kv] fp32, device; the value of
 *             a code of (batch b, KV head g) -- for q, of the query heads
 *             that share KV head g -- is code * descale[b * H_kv + g];
 *             each finite and >= 0 (negative descales: results undefined)
 *   o       : [B, H_q, N, d] bf16, device (output)
 *   lse     : [B, H_q, N] fp32, device (output, natural-log logsumexp of the
 *             scaled scores of the dequantised inputs)
 *   d       : 128 (other values: FA2_ERR_UNSUPPORTED)
 *   B, H_q, H_kv, N, scale, stream : as fa2_fwd_gqa (N % 128 == 0)
 * Both products run on e4m3 tensor-core operands: S = Q K^T exactly in fp32
 * (then scaled by scale * dq * dk), and the softmax weights are scaled by
 * 2^8 and rounded to e4m3 before P V; l sums the unrounded weights. So O
 * differs from attention on the dequantised inputs by at most
 * 2^-4 sum_j p_j |v_j| / l + 2^-18 sum_j |v_j| / l per element (plus the
 * bf16 rounding of O); the LSE carries no rounding of P.
 * Alignment: q, k, v, o, lse 16-byte aligned; descales 4-byte aligned.
 * Errors as fa2_fwd_gqa. Nothing is allocated; all buffers are the caller's.
 */
fa2_status fa2_fwd_fp8(const void* q, const void* k, const void* v, const float* q_descale,
                       const float* k_descale, const float* v_descale, void* o, float* lse,
                       int B, int H_q, int H_kv, int N, int d, float scale, cudaStream_t stream);

/*
 * fa2_fwd_fp8 generalised as fa2_fwd_ex generalises fa2_fwd_gqa: separate
 * query and key lengths, any N_q, N_k >= 1, and the optional bottom-right
 * causal mask (query row i attends keys j < min(N_k, i + 1 + N_k - N_q),
 * "FlashAttention-2 from scratch on Ampere, Part 1", Kernel Specification,
 * lists both as left out of its kernel; the reading is that of fa2_fwd_ex).
 *   q       : [B, H_q, N_q, d] e4m3 codes; o : [B, H_q, N_q, d] bf16;
 *   lse     : [B, H_q, N_q] fp32 (a row with no allowed key: o = 0,
 *             lse = -inf)
 *   k, v    : [B, H_kv, N_k, d] e4m3 codes
 *   descales, d, alignment, numerics: as fa2_fwd_fp8. Key tiles of 128
 *             start at key 0, so a masked row rounds its weights exactly as
 *             the unmasked method on its visible keys.
 *   causal  : 0 or 1 (other values FA2_ERR_INVALID_ARG)
 * Non-causal calls with N_q == N_k and N_q % 128 == 0 run fa2_fwd_fp8.
 * More than 2^31 - 1 query or key rows: FA2_ERR_UNSUPPORTED. Errors
 * otherwise as fa2_fwd_fp8. Nothing is allocated.
 */
fa2_status fa2_fwd_fp8_ex(const void* q, const void* k, const void* v, const float* q_descale,
                          const float* k_descale, const float* v_descale, void* o, float* lse,
                          int B, int H_q, int H_kv, int N_q, int N_k, int d, float scale, int causal,
                          cudaStream_t stream);

/*
 * Attention backward (gradients of the forward with optional causal mask and
 * equal query/key lengths N; any N >= 1, like fa2_fwd_ex). The forward pages exclude the
 * backward pass ("FlashAttention-2 from scratch on Ampere, Part 1", Kernel
 * Specification: forward pass only); it is built here as an extension and
 * recomputes P = exp(scale*S - LSE) from the forward's logsumexp:
 *     D = rowsum(dO o O), dP = dO V^T, dS = P o (dP - D),
 *     dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO
 * (grouped KV heads: dK, dV summed over the query heads that share them).
 *   q, o, dout, dq : [B, H_q, N, d] 16-bit (q, o, dout read; dq written)
 *   k, v, dk, dv   : [B, H_kv, N, d] 16-bit (k, v read; dk, dv written)
 *   lse            : [B, H_q, N] fp32, the forward's logsumexp (read)
 *   delta          : [B, H_q, N] fp32, caller-owned workspace; the call
 *                    writes D into it and then reads it back
 *   causal         : 0 or 1 (same mask as the forward with N_q == N_k)
 * All pointers device memory, 16-byte aligned. Launches three kernels on
 * `stream` (D, then dK/dV, then dQ); allocates nothing. Errors as
 * fa2_fwd_gqa except that N need not be a multiple of 128; B*H_q > 65535
 * is FA2_ERR_UNSUPPORTED. If one of the three launches fails
 * (FA2_ERR_CUDA), the kernels before it may already be queued and the
 * gradients are undefined.
 */
fa2_status fa2_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, float* delta,
                   int B, int H_q, int H_kv, int N, int d, float scale, int causal,
                   fa2_dtype dtype, cudaStream_t stream);

/*
 * fa2_bwd without the `delta` workspace, for callers that cannot allocate
 * device memory: a plugin handed only its input and output tensors by a host
 * framework that owns every device allocation, or code running where a
 * device allocation is not allowed or its implicit synchronisation cannot be
 * afforded. (The source pages have no counterpart; this is an interface
 * convenience of this library.)
 *
 * Same arguments and results as fa2_bwd minus `delta`. D = rowsum(dO o O)
 * lives instead in a fixed device array inside this library, sized for
 * B * H_q * N <= 1048576 query rows (4 MiB of fp32, held on every GPU that
 * loads the library until the process exits). Errors: first those of
 * fa2_bwd for the same arguments (so a NULL pointer is FA2_ERR_INVALID_ARG
 * whatever the size, and a device that is not compute capability 10.3 is
 * FA2_ERR_UNSUPPORTED), then more than 1048576 query rows is
 * FA2_ERR_UNSUPPORTED; nothing is launched in those cases. Nothing is
 * allocated by the call.
 * Each call looks up the array's device address in the current device's
 * context (cudaGetSymbolAddress, a host-side lookup), so the address stays
 * right after cudaDeviceReset or under another context. The first call on a
 * device may load this library's device code on it; make that first call
 * before any stream capture. Every call uses the same array: calls that may
 * overlap on the GPU (other streams, other host threads) race on it and
 * must be ordered by the caller. The array keeps the last call's D; each
 * call rewrites the rows it uses before reading them.
 */
fa2_status fa2_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                           const void* dout, void* dq, void* dk, void* dv,
                           int B, int H_q, int H_kv, int N, int d, float scale, int causal,
                           fa2_dtype dtype, cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the status word of the device
 * that `stream` belongs to (the current device is switched to it for the
 * read and restored afterwards). Returns FA2_ERR_TIMEOUT if a kernel since
 * the last check abandoned a wait (its outputs are then undefined),
 * FA2_ERR_BOUNDS if (debug builds only) a device-side bounds check failed,
 * FA2_ERR_CUDA if the stream reported an error, FA2_OK otherwise.
 * There is one status word per device, shared by every stream and host
 * thread that uses the device: a timeout of a kernel on another stream is
 * reported to whichever caller checks first (and then cleared), and a kernel
 * still running on another stream may set the word after this call read it.
 * Callers that need per-stream attribution check after synchronising all
 * streams that ran the library's kernels.
 */
fa2_status fa2_check_status(cudaStream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* fa2_status_string(fa2_status status);

/*
 * Watchdog limit for each in-kernel wait, in nanoseconds, for kernels
 * launched after the call on any device of this process (default 2e9, i.e.
 * two seconds; values <= 0 restore the default). Returns the previous value.
 */
int64_t fa2_set_wait_limit_ns(int64_t limit_ns);

/*
 * Test hook for the watchdog. With flags = 1 the next 16-bit forward kernels
 * and the backward's dK/dV kernel skip the load of their query tiles, so
 * their waits run out and the status word reports
 * FA2_ERR_TIMEOUT; the kernel still frees its tensor memory, waits for its
 * own copies and returns normally. 0 (the default) restores normal
 * operation. Returns the previous flags.
 */
int fa2_set_debug_flags(int flags);

/*
 * The planner's kernel choice where two kernels compute the same result
 * (process-wide, for calls made after it returns). Bit 0 (value 1): d = 64
 * with equal lengths runs the 16-bit kernel's d = 64 path (P written over S,
 * one MMA-issuing warp) instead of the default d = 64 kernel (P in TMEM
 * columns of its own, separate warps for Q K^T and P V), which measured
 * faster. Results differ only by rounding order and are within the same
 * tolerance. The first call to the library reads the initial value from the
 * environment: FA2_TILE_CFG=d64=shared sets bit 0, anything else or no
 * variable gives 0. Returns the previous value, or -1 (nothing changed) if
 * config is negative or has a bit other than bit 0 set.
 */
int fa2_set_tile_config(int config);

/* Library version string, e.g. "fa2-sm103a 0.3.0" ("... debug" for the
 * FA2_DEBUG build, libfa2_debug.so). */
const char* fa2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA2_H_ */
