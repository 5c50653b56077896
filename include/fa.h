/*
 * fa.h — C ABI of the GB300 (sm_103a) exact attention library, libfa.so: the forward
 * pass (fa_fwd) and its gradient (fa_bwd, further down).
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
 *   - Kernels are launched as programmatic dependents of the kernel before them on the
 *     stream (cudaLaunchKernelEx with programmatic stream serialisation): their set-up
 *     overlaps that kernel's tail, and they read and write global memory only after it
 *     has completed, so stream order is kept. Earlier work of any other kind (copies,
 *     event waits) is waited for as usual.
 *   - Argument errors are detected on the host and returned before anything is
 *     launched; nothing is written to o or lse in that case.
 *   - Thread safety: calls from several host threads are safe.
 */
#ifndef FA_GB300_FA_H_
#define FA_GB300_FA_H_

#include <stddef.h>

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
 *   scale   : multiplies Q Kᵀ (1/√d for standard attention); any finite value: 0 weighs
 *             every visible key equally, a negative value favours the lowest scores
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
 *                the query-tile loads so that every dependent wait runs out; bit 1
 *                (FA_FLAG_TEST_STARVE_LATER_Q) omits them from each CTA's second work
 *                unit on, so that the waits run out after a first unit has finished.
 *                Both exist only to test the timeout path and produce NaN outputs.
 *                Bit 2 (FA_FLAG_CTA_PAIR), d = 64 and bf16 only, runs the forward on CTA
 *                pairs: two CTAs of a cluster share every tensor-core product (256 rows,
 *                each CTA loading half of every K and V tile). Same results; on GB300 it
 *                measures slower than the default single-CTA kernel (B4 H12 T16384
 *                causal: 908 against 1017 TFLOP/s), so it is not the default. Not combined
 *                with the test bits (FA_ERR_INVALID_ARG).
 *
 * Everything else as fa_fwd.
 */
#define FA_FLAG_TEST_STARVE_Q 1u
#define FA_FLAG_TEST_STARVE_LATER_Q 2u
#define FA_FLAG_CTA_PAIR 4u
int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int T, int d, int causal, float scale, int* status, unsigned long long timeout_ns,
              unsigned int flags, void* stream);

/*
 * ---------------------------------------------------------------------------------------
 * General forms of the forward.
 *
 * Both compute, for every b, h, the attention of Tq query rows over Tk key rows with a
 * visibility mask, in the same tiled online-softmax way as fa_fwd:
 *
 *   query i sees key j  iff  (causal == 0 or j ≤ i + Tk − Tq)        [bottom-right causal]
 *                        and (no block mask or mask[i/128][j/128] ≠ 0)
 *
 * A row that sees no key at all gets O = 0 and LSE = −∞. Layouts, alignment, ownership,
 * asynchrony and error behaviour are those of fa_fwd (q, o: [B, H, Tq, d]; k, v:
 * [B, H, Tk, d]; lse: [B, H, Tq]); d ∈ {64, 128}.
 * ---------------------------------------------------------------------------------------
 */

/*
 * fa_fwd_kv — Tq queries against Tk keys, e.g. new tokens (or one decoded token,
 * Tq = 1) against the K/V of every earlier token, which generation keeps ("手写
 * FlashAttention" step ①). causal requires Tq ≤ Tk. One or two query rows run on the CUDA
 * cores (a dot product and a scaled add per cached row, which a 128-row tensor tile would
 * mostly pad); more run on the tensor cores. When the CTAs of either leave SMs idle, the
 * key range is split into n_splits ranges processed by different CTAs; each writes a partial result (normalised O, LSE) to the workspace and a second
 * kernel merges them with weights exp(LSE_s − max LSE) — the merge over K/V blocks that
 * step ③ of the same page attributes to the first FlashAttention's outer loop.
 *
 *   n_splits  : key ranges; 0 picks a number from the SM count of the current device
 *               (ranges count keys for Tq ≤ 2 and 128-key tiles above)
 *   workspace : device memory, 256-byte aligned, at least fa_fwd_kv_workspace_size(...)
 *               bytes, owned by the caller; unused (may be NULL) when one range is used.
 *               Must not overlap any argument or be used by a concurrent call.
 */
size_t fa_fwd_kv_workspace_size(int B, int H, int Tq, int Tk, int d, int n_splits);
int fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Tq, int Tk, int d, int causal, float scale, int n_splits, void* workspace,
              size_t workspace_bytes, void* stream);
/* fa_fwd_kv_workspace_size returns the bytes needed for these sizes and n_splits (0: the
 * automatic choice on the current device), 1 when no workspace is needed, and 0 for
 * unsupported sizes or (automatic choice) no usable device. */

/*
 * fa_fwd_block_sparse — self-attention (Tq = Tk = T) in which whole 128×128 blocks of the
 * score matrix are switched off by a block mask and never computed: the generalisation of
 * skipping fully masked causal blocks ("内核案例研究：Flash Attention", "块稀疏注意力 V2 和
 * V3": a block whose mask is all zero is skipped).
 *
 *   block_mask : DEVICE uint8 array [mask_heads][ceil(T/128)][ceil(T/128)], row-major,
 *                nonzero = compute the block; owned by the caller, not modified
 *   mask_heads : 1 (one mask for every head) or B·H (one per (b, h), in b-major order)
 *   causal     : combined with the block mask (element-wise within kept blocks)
 */
int fa_fwd_block_sparse(const void* q, const void* k, const void* v, void* o, float* lse,
                        const unsigned char* block_mask, int mask_heads, int B, int H, int T,
                        int d, int causal, float scale, void* stream);

/*
 * ---------------------------------------------------------------------------------------
 * Backward pass.
 *
 * The gradients of the forward above for an upstream gradient dO = ∂L/∂O:
 *
 *     P     = exp(S − LSE)            (recomputed from q, k and the forward's lse)
 *     dV    = Pᵀ dO
 *     dP    = dO Vᵀ,   D_i = Σ_c dO_ic O_ic
 *     dS    = P ∘ (dP − D)
 *     dQ    = scale · dS K,   dK = scale · dSᵀ Q
 *
 * Step ④ of "手写 FlashAttention" (Hand-written FlashAttention) explains why the forward
 * keeps the row logsumexp: so that the backward can rebuild S and P block by block
 * instead of storing them; §2.2 of "FlashAttention 核心思路解析" (FlashAttention core
 * ideas, ijyty.com) adds that the per-block query gradients are summed into the global
 * gradient with atomic adds. Neither page writes out the derivative; the formulas above
 * are the chain rule applied to the forward's definition.
 * ---------------------------------------------------------------------------------------
 */

/*
 * fa_bwd_workspace_size — bytes of device workspace that fa_bwd needs for these sizes
 * (fp32 row statistics and an fp32 dQ accumulator: about B·H·T·(d + 2)·4 bytes).
 * Returns 0 when the sizes are not supported by fa_bwd (d must be 64 or 128).
 */
size_t fa_bwd_workspace_size(int B, int H, int T, int d);

/*
 * fa_bwd — exact attention backward.
 *
 *   q, k, v   : const bf16*, [B, H, T, d], device memory: the forward's inputs
 *   o         : const bf16*, [B, H, T, d]: the forward's output
 *   dout      : const bf16*, [B, H, T, d]: the upstream gradient dO
 *   lse       : const float*, [B, H, T]: the forward's lse
 *   dq, dk, dv: bf16*, [B, H, T, d], device memory, written
 *   workspace : device memory owned by the caller, at least fa_bwd_workspace_size(...)
 *               bytes, 256-byte aligned; its contents on entry do not matter (the call
 *               initialises what it uses). It must not be used by another call that may
 *               run at the same time.
 *   causal, scale, stream : as for fa_fwd, and equal to the values of the forward call.
 *
 * Supported: d ∈ {64, 128}; otherwise as fa_fwd. dq, dk, dv and the workspace must not overlap
 * any input or one another. The call enqueues three kernels on `stream` and returns; the
 * library allocates nothing. Returns FA_OK or an fa_status code (host-side validation
 * as for fa_fwd; nothing is launched on failure).
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, void* workspace,
           size_t workspace_bytes, int B, int H, int T, int d, int causal, float scale,
           void* stream);

/*
 * fa_bwd_ex — fa_bwd with the fault-reporting controls of fa_fwd_ex: a timed-out internal
 * wait stores FA_ERR_TIMEOUT in *status and leaves NaN in the dq, dk, dv rows of the
 * abandoned work; flag FA_FLAG_TEST_STARVE_Q omits the query-tile and dO loads (test only).
 */
int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout,
              const float* lse, void* dq, void* dk, void* dv, void* workspace,
              size_t workspace_bytes, int B, int H, int T, int d, int causal, float scale,
              int* status, unsigned long long timeout_ns, unsigned int flags, void* stream);

/*
 * fa_bwd_noalloc — fa_bwd without a caller-provided workspace. The pages describe no
 * such call; it exists for callers that cannot give the library a device buffer (their
 * memory is already committed to their own pools, or they call from a path where a
 * device allocation is not acceptable).
 *
 * The workspace is a fixed reservation of FA_BWD_NOALLOC_SCRATCH_BYTES (32 MiB) of device
 * memory inside the library, made when the library's device code is loaded onto a
 * device. The call allocates nothing. Its contents need not start at zero: every call
 * initialises what it uses.
 *
 *   - Sizes whose workspace (fa_bwd_workspace_size) exceeds the reservation are rejected
 *     with FA_ERR_INVALID_ARG before anything is launched; with d = 64 that is
 *     B·H·ceil(T/128)·128·66·4 bytes > 32 MiB, e.g. B·H = 12 allows T ≤ 10496.
 *   - The first call on each device looks up the reservation's device address (which
 *     may load the library's device code); FA_ERR_LAUNCH if that fails. Make that first
 *     call before any stream capture on the device. The address is kept per device
 *     together with the id of the context it was found in; after a device reset (a new
 *     context) the next call looks it up again, so make that call before any capture too.
 *   - There is one reservation per device: calls that may overlap in time on the same
 *     device (different streams, or several host threads) race on it and give wrong
 *     results. Order them on one stream, or with events.
 *   - Everything else (arguments, layout, validation, asynchrony) as fa_bwd.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES 33554432
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int T, int d,
                   int causal, float scale, void* stream);

/*
 * fa_fwd_fp8 — the forward with Q and K given as FP8 (e4m3) codes with per-tensor scales:
 * the query and key values are q8·q_scale and k8·k_scale, and S = scale·Q·Kᵀ is computed
 * from the codes on the tensor cores' 8-bit path (exact products, fp32 sums) with
 * q_scale·k_scale folded into the softmax's exponent factor. V stays bf16 and P is rounded
 * to bf16 as in fa_fwd, so the output carries the bf16 path's error on the quantised
 * inputs. Low-precision modes are the direction the section on versions V2 and V3 of
 * "内核案例研究：Flash Attention" ("块稀疏注意力 V2 和 V3") points to.
 *
 *   q8, k8           : const uint8*, [B, H, T, d] e4m3 codes, device memory, 16-byte aligned
 *   q_scale, k_scale : finite and > 0
 *   v, o, lse, B, H, T, d, causal, scale, stream : as for fa_fwd (d ∈ {64, 128})
 */
int fa_fwd_fp8(const void* q8, const void* k8, const void* v, void* o, float* lse, float q_scale,
               float k_scale, int B, int H, int T, int d, int causal, float scale, void* stream);

/*
 * fa_fwd_host — the forward of fa_fwd on tensors that live in HOST memory. The B·H heads are
 * taken in chunks of `heads_per_chunk` (0: the library picks enough heads to give every SM
 * two work units); each chunk is copied into a device staging buffer, attended with fa_fwd's
 * kernel and copied back. Copies in, computation and copies out run on three streams with
 * three staging buffers, so a chunk's transfers overlap its neighbours' computation. The
 * kernels run on `stream`; the copies on two streams the library creates once per device.
 * Everything is enqueued behind the work already on `stream`, and `stream` is made to wait
 * for the last copy out: o and lse may be read once `stream` has been synchronised, and the
 * workspace may then be reused. Results are bit-identical to fa_fwd on the same values.
 *
 *   q, k, v   : const bf16*, [B, H, T, d] contiguous, host memory (page-locked memory lets
 *               the copies run asynchronously; pageable memory works, without the overlap)
 *   o, lse    : bf16* [B, H, T, d] and float* [B, H, T], host memory, written asynchronously
 *   workspace : device memory of at least fa_fwd_host_workspace_size(B, H, T, d,
 *               heads_per_chunk) bytes, 256-byte aligned, owned by the caller
 *   B, H, T, d, causal, scale : as for fa_fwd
 *
 * Errors: the argument checks of fa_fwd (applied to the host tensors), plus a null,
 * misaligned or too small workspace and heads_per_chunk < 0, are returned before anything
 * is enqueued. A CUDA error while enqueuing returns FA_ERR_LAUNCH; chunks enqueued before it
 * still run.
 */
size_t fa_fwd_host_workspace_size(int B, int H, int T, int d, int heads_per_chunk);
int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int T, int d, int causal, float scale, int heads_per_chunk, void* workspace,
                size_t workspace_bytes, void* stream);

/* Static text for a status code (never NULL). */
const char* fa_strerror(int status);

/* Static version string of the library, e.g. "fa-gb300 0.1.0 sm_103a". */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H_ */
