/*
 * fa.h — C ABI of the GB300 (sm_103a) exact attention forward library, libfa.so.
 *
 * The operation, for every batch b and head h of contiguous [B, H, T, d] tensors:
 *
 *     S    = scale · Q Kᵀ                       (T × T, never written to memory)
 *     S_ij = −∞ for j > i                       (only when causal != 0)
 *     O    = softmax_rows(S) · V                (bf16 output, fp32 accumulation)
 *     LSE_i = ln Σ_j exp(S_ij)                  (fp32, natural log of the scaled scores)
 *
 * This is the naive form written out in step ① of "手写 FlashAttention:拆开 SDPA 这个黑盒"
 * (Hand-written FlashAttention, learn-llm.fim.ai ch. 19), computed exactly as its steps
 * ② and ③ describe: Q is cut into row blocks, each block scans the K/V blocks while keeping
 * a running row max m, a running sum l and an accumulator that are rescaled by
 * exp(m_old − m_new) whenever the max rises, followed by a single division by l at the
 * end; fully masked causal blocks are skipped. The per-row logsumexp is what step ④ says
 * the forward pass keeps for a backward pass.
 *
 * Conventions for every call:
 *   - Pointers q, k, v, o, lse are DEVICE pointers owned by the caller. The library
 *     allocates nothing and keeps no state between calls (it caches, once per process,
 *     a driver entry point and per-device kernel attributes).
 *   - Layout: q, k, v, o are bf16, contiguous [B][H][T][d] (strides H·T·d, T·d, d, 1);
 *     lse is fp32, contiguous [B][H][T].
 *   - Every pointer must be 16-byte aligned (a requirement of the tensor-memory-access
 *     copy engine), and o must not overlap q, k or v.
 *   - Supported: d ∈ {64, 128}; 1 ≤ T; B·H ≥ 1; B·H·T·d < 2^62; device of compute
 *     capability 10.3 (GB300, sm_103a).
 *   - The call is asynchronous on `stream` (a cudaStream_t; NULL means the legacy
 *     default stream). It returns after the launch is enqueued; errors that happen
 *     while the kernel runs surface at the caller's next synchronisation.
 *   - Argument errors are detected on the host and returned before anything is
 *     launched; nothing is written to o or lse in that case.
 *   - Thread safety: calls from several host threads are safe.
 */
#ifndef FA_GB300_FA_H_
#define FA_GB300_FA_H_

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,        /* null pointer, bad size, d not 64/128, non-finite scale, o aliasing q/k/v */
  FA_ERR_MISALIGNED = 2,         /* a pointer is not 16-byte aligned */
  FA_ERR_UNSUPPORTED_DEVICE = 3, /* no CUDA device, or its compute capability is not 10.3 */
  FA_ERR_LAUNCH = 4,             /* the CUDA runtime refused the launch or a driver entry point is missing */
  FA_ERR_TIMEOUT = 5             /* (device status only) an internal wait gave up; outputs are NaN */
} fa_status;

/*
 * fa_fwd — exact attention forward (see the top of this file).
 *
 *   q, k, v : const bf16*, [B, H, T, d], device memory
 *   o       : bf16*, [B, H, T, d], device memory, written
 *   lse     : float*, [B, H, T], device memory, written (natural-log logsumexp of the
 *             scaled scores of each query row)
 *   causal  : nonzero → key j is visible to query i only when j ≤ i
 *   scale   : multiplies Q Kᵀ (1/√d for standard attention); must be finite and > 0
 *   stream  : cudaStream_t or NULL
 *
 * Returns FA_OK or an fa_status code; see the conventions above.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int T,
           int d, int causal, float scale, void* stream);

/*
 * fa_fwd_ex — fa_fwd with the kernel's fault-reporting controls exposed.
 *
 *   status     : optional DEVICE int (NULL allowed). If any internal wait of the kernel
 *                times out, the kernel stores FA_ERR_TIMEOUT there (it never clears it;
 *                the caller zeroes it before the call) and writes NaN to the o and lse
 *                rows of the work it abandoned. A timeout means a bug, never an input
 *                property.
 *   timeout_ns : limit for every internal wait, in nanoseconds; 0 selects 2 s.
 *   flags      : 0 for normal use. Bit 0 (FA_FLAG_TEST_STARVE_Q) makes the kernel omit
 *                the query-tile loads so that every dependent wait runs out; it exists
 *                only to test the timeout path and produces NaN outputs.
 *
 * Everything else as fa_fwd.
 */
#define FA_FLAG_TEST_STARVE_Q 1u
int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int T, int d, int causal, float scale, int* status, unsigned long long timeout_ns,
              unsigned int flags, void* stream);

/* Static text for a status code (never NULL). */
const char* fa_strerror(int status);

/* Static version string of the library, e.g. "fa-gb300 0.1.0 sm_103a". */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H_ */
