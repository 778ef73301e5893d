/*
 * kda.h -- C ABI of the GB300 (sm_103a) recurrent KDA training forward/backward.
 *
 * The method: Kimi Delta Attention, a gated delta rule with a per-key-dimension
 * decay and a value-first FP32 state S[V, K] per (sequence, value head),
 * K = V = 128. Per token (flashinfer.kda_backward.recurrent_kda_backward,
 * description; flashinfer.kda.recurrent_kda, parameter lower_bound):
 *   q^ = q / sqrt(|q|^2 + 1e-6),   k^ = k / sqrt(|k|^2 + 1e-6)
 *   d  = exp(lower_bound * sigmoid(exp(A_log[h]) * (g + dt_bias[h])))   (per key dim)
 *   beta = sigmoid(beta_logit)
 *   S' = S diag(d);  u = v - S' k^;  S = S' + beta u k^T;  o = scale S q^
 * The pages give the gate, norm, beta, scale and shape contracts; the order of
 * the update (decay, delta correction, rank-1 write, output from the updated
 * state) is the plain reading this library adopts.
 *
 * Two entry points form one training pair (flashinfer.kda_training, module
 * description): kda_fwd returns the output, the final state and a saved
 * context; kda_bwd consumes that context (it never reruns the forward) and
 * returns the eight gradients in the documented order
 * (dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dinitial_state).
 *
 * Conventions shared by every entry point:
 *  - Tensor pointers are DEVICE pointers to contiguous row-major storage, owned
 *    by the caller, on the current CUDA device. The only host pointer is the
 *    trusted cu_seqlens mirror (flashinfer.kda_training.recurrent_kda_training_forward,
 *    parameter cu_seqlens_cpu).
 *  - BF16 tensors are passed as kda_bf16 (raw bfloat16 bits).
 *  - `stream` is a cudaStream_t (struct CUstream_st*); NULL is the legacy
 *    default stream. All work is enqueued asynchronously on it.
 *  - Argument errors are detected on the host before any launch; nothing is
 *    enqueued and the call returns a non-zero kda_status. A message describing
 *    the last failure on the calling thread is available from
 *    kda_last_error_message().
 *  - Outputs are overwritten, never accumulated into.
 *  - Thread safety: distinct contexts may be used from different threads;
 *    calls sharing one context must be serialised by the caller.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef uint16_t kda_bf16;

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARGUMENT = 1,    /* null pointer, bad shape, bad cu_seqlens, empty sequence */
  KDA_ERR_UNSUPPORTED = 2,         /* head dim != 128, scale != 1/sqrt(128), lower_bound != -5,
                                      device not compute capability 10.3 */
  KDA_ERR_ALIASING = 3,            /* an output overlaps an input, another output or the context */
  KDA_ERR_CONTEXT = 4,             /* context shape/device/stream mismatch, or context busy */
  KDA_ERR_CUDA = 5,                /* a CUDA runtime call failed */
  KDA_ERR_DEVICE_TIMEOUT = 6,      /* a bounded device-side wait gave up (see kda_ctx_status) */
  KDA_ERR_WORKSPACE_TOO_SMALL = 7  /* ctx_bytes below kda_ctx_workspace_bytes() */
} kda_status;

/* Opaque saved-forward context: host metadata (shapes, the launch plan), the
 * borrowed input pointers and offsets into the caller's workspace, which holds
 * the state checkpoints and the backward's scratch. */
typedef struct kda_ctx kda_ctx;

/*
 * Bytes of device workspace one context needs for this problem.
 *   Fixed layout  (flashinfer.kda_training, module description): cu_seqlens_host = NULL,
 *                 num_seqs ignored; B >= 1 sequences of T >= 1 tokens each.
 *   Packed layout: B == 1, cu_seqlens_host[num_seqs + 1] with cu[0] = 0,
 *                 cu[num_seqs] = T and every sequence non-empty.
 * Writes the size to *bytes. Returns KDA_ERR_INVALID_ARGUMENT on a bad shape.
 */
kda_status kda_ctx_workspace_bytes(int64_t B, int64_t T, int64_t Hqk, int64_t Hv,
                                   const int64_t* cu_seqlens_host, int64_t num_seqs,
                                   size_t* bytes);

/*
 * Training forward (flashinfer.kda_training.recurrent_kda_training_forward).
 * Inputs (device, contiguous):
 *   q, k     BF16 [B, T, Hqk, 128]      v, g  BF16 [B, T, Hv, 128]
 *   beta     BF16 [B, T, Hv]  raw logits       A_log FP32 [Hv]   dt_bias FP32 [Hv, 128]
 *   h0       FP32 [N, Hv, 128, 128] value-first initial state (N = B fixed, num_seqs packed)
 *   cu_seqlens_dev  INT64 [num_seqs + 1] for packed input, NULL for fixed input
 *   cu_seqlens_host its trusted host mirror (NULL for fixed input); the launch plan
 *                   (longest sequence first) is built from it and must match the device copy
 *   head_dim must be 128; Hv % Hqk == 0 (value head h reads query/key head h / (Hv/Hqk)).
 *   scale: NaN selects 1/sqrt(128); any other value must equal it.
 *   lower_bound must be -5.
 * Outputs (device, caller-owned, must not overlap any input, each other or the workspace):
 *   o    BF16 [B, T, Hv, 128]         h_T  FP32 [N, Hv, 128, 128]
 * Context:
 *   ctx_workspace / ctx_bytes: device memory of at least kda_ctx_workspace_bytes(),
 *   256-byte aligned, owned by the caller and bound to the context until it is
 *   destroyed. *ctx == NULL creates a context; a non-NULL *ctx is reused, which
 *   requires identical shapes, device, stream and workspace, and overwrites its
 *   saved checkpoints. The inputs are borrowed by the context: they must stay
 *   allocated and unmodified until kda_bwd has been enqueued.
 * CUDA graphs: creating a context copies the launch plan from host memory, so
 *   create it outside any capture; a call that reuses it (and kda_bwd) only
 *   launches kernels on `stream` and may be captured into a CUDA graph. A replay
 *   reads whatever the captured input buffers hold at that time.
 */
kda_status kda_fwd(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                   const kda_bf16* beta, const float* A_log, const float* dt_bias,
                   const float* h0, const int64_t* cu_seqlens_dev,
                   const int64_t* cu_seqlens_host, int64_t num_seqs, int64_t B, int64_t T,
                   int64_t Hqk, int64_t Hv, int64_t head_dim, float scale, float lower_bound,
                   kda_bf16* o, float* h_T, void* ctx_workspace, size_t ctx_bytes,
                   kda_ctx** ctx, struct CUstream_st* stream);

/*
 * Training backward (flashinfer.kda_training, recurrent_kda_training_backward;
 * gradient list of flashinfer.kda_backward.recurrent_kda_backward).
 * Inputs: the context of the last kda_fwd, the output adjoint d_o BF16 [B, T, Hv, 128]
 * and the final-state adjoint d_hT FP32 [N, Hv, 128, 128].
 * Outputs (device, caller-owned, all written, none may overlap an input, the
 * context workspace or each other):
 *   dq, dk BF16 [B, T, Hqk, 128]   dv, dg BF16 [B, T, Hv, 128]   dbeta BF16 [B, T, Hv]
 *   dA_log FP32 [Hv]   ddt_bias FP32 [Hv, 128]   dh0 FP32 [N, Hv, 128, 128]
 * dg and dbeta are gradients with respect to the raw gate and raw beta logits.
 * dA_log and ddt_bias are summed over all sequences and tokens in a fixed order
 * (bitwise reproducible). Must be called on the stream and device that created
 * the context.
 */
kda_status kda_bwd(kda_ctx* ctx, const kda_bf16* d_o, const float* d_hT, kda_bf16* dq,
                   kda_bf16* dk, kda_bf16* dv, kda_bf16* dg, kda_bf16* dbeta, float* dA_log,
                   float* ddt_bias, float* dh0, struct CUstream_st* stream);

/* Synchronises the context's stream and reports the first device-side error
 * (KDA_ERR_DEVICE_TIMEOUT if a bounded wait gave up, KDA_ERR_CUDA on a CUDA
 * error), else KDA_OK. The timeout word lives in the workspace and is cleared
 * only when a context is created: once set, it stays set for this context and
 * the outputs of every call made with it since are not to be trusted. */
kda_status kda_ctx_status(kda_ctx* ctx);

/* Frees the host-side context. The workspace stays owned by the caller. Safe on NULL. */
void kda_ctx_destroy(kda_ctx* ctx);

/* Static description of a status code. */
const char* kda_status_string(kda_status status);

/* Message of the last failed call on this thread ("" if none). */
const char* kda_last_error_message(void);

/*
 * Standalone backward with a caller-owned workspace
 * (flashinfer.kda_backward.recurrent_kda_backward: signature, description and
 * the parameters workspace and out). From the forward's inputs, the initial
 * state and the two adjoints it returns the eight gradients of kda_bwd, in the
 * same order, into caller-owned buffers: it runs the training forward into the
 * workspace (the checkpoints, and the output and final state, which it does
 * not return) and then the backward.
 * Bytes: kda_bwd_standalone_workspace_bytes() (same shape arguments and errors
 * as kda_ctx_workspace_bytes): a context workspace followed by room for o and
 * the final state.
 * Inputs: those of kda_fwd (same layouts, rules and head mapping) and of
 *   kda_bwd (d_o BF16 [B, T, Hv, 128], d_hT FP32 [N, Hv, 128, 128]).
 * Outputs: dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dh0 as for kda_bwd.
 * workspace / workspace_bytes: device memory, 256-byte aligned, owned by the
 *   caller; no input or output may overlap it.
 * ws_ctx: a host handle bound to the workspace, like kda_fwd's ctx. Pass a
 *   pointer to NULL on the first call (it uploads the launch plan, built from
 *   cu_seqlens_host, into the workspace: the "eager warm-up" of the page);
 *   later calls with the same handle, shapes, workspace, device and stream only
 *   launch kernels and may be captured into a CUDA graph (a replay reads the
 *   buffers the captured pointers name). Free it with kda_ctx_destroy.
 * Errors: those of kda_fwd and kda_bwd; KDA_ERR_WORKSPACE_TOO_SMALL;
 *   KDA_ERR_ALIASING when an adjoint or gradient overlaps the workspace.
 *   Device-side timeouts are reported by kda_ctx_status(*ws_ctx).
 * Nothing is allocated on the device.
 */
kda_status kda_bwd_standalone_workspace_bytes(int64_t B, int64_t T, int64_t Hqk, int64_t Hv,
                                              const int64_t* cu_seqlens_host, int64_t num_seqs,
                                              size_t* bytes);
kda_status kda_bwd_standalone(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                              const kda_bf16* beta, const float* A_log, const float* dt_bias, const float* h0,
                              const int64_t* cu_seqlens_dev, const int64_t* cu_seqlens_host, int64_t num_seqs,
                              int64_t B, int64_t T, int64_t Hqk, int64_t Hv, int64_t head_dim, float scale,
                              float lower_bound, const kda_bf16* d_o, const float* d_hT, kda_bf16* dq,
                              kda_bf16* dk, kda_bf16* dv, kda_bf16* dg, kda_bf16* dbeta, float* dA_log,
                              float* ddt_bias, float* dh0, void* workspace, size_t workspace_bytes,
                              kda_ctx** ws_ctx, struct CUstream_st* stream);

/*
 * Standalone backward that allocates nothing. The documentation pages have no
 * counterpart for this entry point; it exists for callers that cannot call
 * cudaMalloc: code running while another component owns all device memory
 * through its own pool (a framework caching allocator, a server that carves
 * the GPU up front), hosts that forbid allocation inside a plug-in call, and
 * loops that cannot afford the device-wide synchronisation cudaMalloc/cudaFree
 * may imply. Such callers own their inputs and outputs but cannot provide the
 * context workspace kda_fwd/kda_bwd need.
 *
 * Inputs and outputs are those of kda_fwd (inputs, same layouts and rules) plus
 * those of kda_bwd (d_o, d_hT and the eight gradients); the function recomputes
 * the forward's checkpoints itself and returns the same eight gradients.
 * Scratch: one fixed array of KDA_NOALLOC_SCRATCH_BYTES compiled into the
 * library (a static __device__ array), resident on every GPU where the library's
 * module is loaded until the process exits. A problem whose checkpoints and
 * intermediates exceed it is rejected with KDA_ERR_WORKSPACE_TOO_SMALL (use
 * kda_fwd + kda_bwd for it). With a checkpoint every kda_checkpoint_tokens()
 * = 16 tokens about 4.9 KiB per token-head (5.9 KiB when Hv > Hqk) plus 65 KiB
 * per (sequence, head) are needed: e.g. 1024 tokens x 12 heads with Hv = Hqk fit.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture. Every call shares the one array and leaves its contents
 * behind; the only part that must start at zero, a status word at the start of
 * the array, is cleared by each call before its first launch. Calls whose work
 * overlaps on the GPU (different streams, or several host threads) race on the
 * array: serialise them. Units run in index order; the per-sequence plan is
 * built on the device from cu_seqlens_dev and checked against what the host
 * mirror implies (start 0, end T, non-empty sequences, the same checkpoint
 * totals), so a device copy that disagrees never sends a kernel outside its
 * buffers: it is reported by kda_noalloc_status instead. Nothing is allocated:
 * no cudaMalloc, cudaFree or allocating library routine is called.
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
kda_status kda_bwd_noalloc(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                           const kda_bf16* g, const kda_bf16* beta, const float* A_log,
                           const float* dt_bias, const float* h0, const int64_t* cu_seqlens_dev,
                           const int64_t* cu_seqlens_host, int64_t num_seqs, int64_t B, int64_t T,
                           int64_t Hqk, int64_t Hv, int64_t head_dim, float scale,
                           float lower_bound, const kda_bf16* d_o, const float* d_hT,
                           kda_bf16* dq, kda_bf16* dk, kda_bf16* dv, kda_bf16* dg,
                           kda_bf16* dbeta, float* dA_log, float* ddt_bias, float* dh0,
                           struct CUstream_st* stream);

/* Reads back the status word of the last kda_bwd_noalloc call on the current
 * device, after synchronising `stream` (the stream that call used). Returns
 * KDA_OK; KDA_ERR_INVALID_ARGUMENT when the device cu_seqlens disagreed with
 * its host mirror (the gradients are then not meaningful); KDA_ERR_DEVICE_TIMEOUT
 * when a bounded device wait gave up (some gradients were not written);
 * KDA_ERR_CUDA on a CUDA error. Allocates nothing. */
kda_status kda_noalloc_status(struct CUstream_st* stream);

/* State element types for kda_decode. */
enum { KDA_STATE_BF16 = 0, KDA_STATE_FP32 = 1 };

/* Device bytes of the arena kda_step_host needs for this problem: the device
 * copies of its eleven inputs and ten outputs (each 256-byte aligned) followed
 * by one context workspace (kda_ctx_workspace_bytes). Same shape arguments and
 * errors as kda_ctx_workspace_bytes. */
kda_status kda_step_arena_bytes(int64_t B, int64_t T, int64_t Hqk, int64_t Hv,
                                const int64_t* cu_seqlens_host, int64_t num_seqs, size_t* bytes);

/* One training step from and to host memory (flashinfer.kda_training forward
 * and backward; gradient list of flashinfer.kda_backward.recurrent_kda_backward):
 * enqueues on `stream` the host-to-device copies of q, k, v, g, beta, A_log,
 * dt_bias, initial_state h0, cu_seqlens (packed layout only), d_o and d_hT
 * into `arena`, then kda_fwd and kda_bwd on those copies, then the
 * device-to-host copies of o, h_T and the eight gradients, and returns without
 * waiting. Every tensor argument is a HOST pointer with the layout and dtype
 * of kda_fwd / kda_bwd; cu_seqlens_host (NULL for the fixed layout) is read
 * during the call. Host buffers should be page-locked (cudaHostAlloc or
 * cudaHostRegister): then the copies are asynchronous and run on the copy
 * engines; pageable buffers work but their copies are staged by the host.
 * The host buffers must stay valid and untouched until the stream reaches the
 * end of the step. `arena`: caller-owned device memory of at least
 * kda_step_arena_bytes(), 256-byte aligned, not used by anything else until
 * the step completes. `ctx`: as for kda_fwd (NULL on the first call; reused
 * afterwards with the same arena, shapes and stream; freed with
 * kda_ctx_destroy). The kernels run on `stream`; the input copies on
 * `h2d_stream` and the output copies on `d2h_stream` (each NULL for `stream`).
 * The context orders them with three events of its own: the kernels wait for
 * this step's input copies and for the previous step's output copies from
 * the same arena, the input copies wait for the previous step's kernels on
 * the same arena, the output copies wait for this step's kernels. A caller that
 * alternates two arenas (two contexts) on shared copy and compute streams gets
 * step i+1's inputs copied in while step i computes, and step i's outputs
 * copied out while step i+1 computes. To wait for a step, synchronise
 * `d2h_stream` (or the device).
 * Errors: those of kda_fwd and kda_bwd; KDA_ERR_WORKSPACE_TOO_SMALL for a small
 * arena; KDA_ERR_INVALID_ARGUMENT for a NULL pointer, a misaligned arena or a
 * device pointer where a host buffer is expected. Nothing is allocated. */
kda_status kda_step_host(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                         const kda_bf16* beta, const float* A_log, const float* dt_bias, const float* h0,
                         const int64_t* cu_seqlens_host, int64_t num_seqs, int64_t B, int64_t T,
                         int64_t Hqk, int64_t Hv, int64_t head_dim, float scale, float lower_bound,
                         const kda_bf16* d_o, const float* d_hT, kda_bf16* o, float* h_T, kda_bf16* dq,
                         kda_bf16* dk, kda_bf16* dv, kda_bf16* dg, kda_bf16* dbeta, float* dA_log,
                         float* ddt_bias, float* dh0, void* arena, size_t arena_bytes, kda_ctx** ctx,
                         struct CUstream_st* stream, struct CUstream_st* h2d_stream,
                         struct CUstream_st* d2h_stream);

/* Gate modes of kda_decode and kda_prefill (flashinfer.kda.recurrent_kda,
 * parameters g, beta, A_log, use_gate_in_kernel, lower_bound and
 * beta_is_logit):
 *   use_gate_in_kernel = 1: the decay is computed in the kernel,
 *       d = exp(lower_bound * sigmoid(exp(A_log[h]) * (g + dt_bias[h]))),
 *       with lower_bound -5 (the sigmoid-bounded formula; the softplus gate
 *       the page names without a formula is not offered: KDA_ERR_UNSUPPORTED
 *       for any other lower_bound);
 *   use_gate_in_kernel = 0: g is already the log decay, d = exp(g); A_log and
 *       dt_bias may be NULL and lower_bound is ignored;
 *   beta_is_logit = 1: the learning rate is sigmoid(beta);
 *   beta_is_logit = 0: beta is the learning rate itself (already sigmoided).
 * The training entry points kda_fwd / kda_bwd always use the in-kernel gate
 * and beta logits. */

/* One decode step, T = 1 (flashinfer.kda.recurrent_kda, description and the
 * parameters q ("T=1 selects decode"), initial_state ("Updated in-place") and
 * ssm_state_indices): for every sequence n and value head h, with the state S
 * of pool slot state_indices[n] (slot n when state_indices is NULL),
 *   S' = S diag(d),  u = v - S' k^,  S <- S' + beta u k^^T,  o = scale S q^
 * with q^, k^ L2-normalised in the kernel (eps 1e-6) and d and beta as the
 * gate modes above say. Arithmetic is FP32; a BF16 state is read, updated
 * in FP32 and written back rounded to nearest even.
 *   q, k            BF16 [N, 1, Hqk, 128]
 *   v, g            BF16 [N, 1, Hv, 128]; beta BF16 [N, 1, Hv]
 *   A_log           FP32 [Hv]; dt_bias FP32 [Hv, 128] (may be NULL when
 *                   use_gate_in_kernel is 0)
 *   state           [num_slots, Hv, 128, 128] value-first, KDA_STATE_BF16 or
 *                   KDA_STATE_FP32 per state_dtype; read and written in place
 *   state_indices   device int32 [N] and its trusted host mirror
 *                   state_indices_host (both NULL, or both set); every index in
 *                   [0, num_slots) and no slot used twice. The call checks the
 *                   mirror; the kernel reads the device copy and checks its
 *                   range again: a device index outside [0, num_slots) (one
 *                   that no longer matches the mirror, as in a replayed CUDA
 *                   graph whose indices were rewritten) leaves the pool alone
 *                   and sets that sequence's o to NaN. Distinct slots on the
 *                   device stay the caller's duty there.
 *   o               BF16 [N, 1, Hv, 128], overwritten
 * Hv must be a multiple of Hqk (value head h reads query/key head h / (Hv/Hqk));
 * head_dim 128; scale NaN or 1/sqrt(128); lower_bound -5. Device pointers are
 * caller-owned, 16-byte aligned for the token and state tensors; the state,
 * o and the inputs must not overlap. Validation errors return before any
 * launch (KDA_ERR_INVALID_ARGUMENT, KDA_ERR_UNSUPPORTED, KDA_ERR_ALIASING);
 * otherwise the step is enqueued on `stream` and KDA_OK returned (KDA_ERR_CUDA
 * on a launch error). Nothing is allocated. */
kda_status kda_decode(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                      const kda_bf16* beta, const float* A_log, const float* dt_bias, void* state,
                      int32_t state_dtype, const int32_t* state_indices,
                      const int32_t* state_indices_host, int64_t num_slots, int64_t N, int64_t Hqk,
                      int64_t Hv, int64_t head_dim, float scale, float lower_bound,
                      int32_t use_gate_in_kernel, int32_t beta_is_logit, kda_bf16* o,
                      struct CUstream_st* stream);

/* Inference prefill over whole sequences from a state pool (flashinfer.kda.
 * recurrent_kda, parameters initial_state "Updated in-place",
 * ssm_state_indices, state_checkpoints, checkpoint_cu_starts and
 * checkpoint_every_n_tokens): the forward recurrence of kda_fwd for every
 * sequence n and value head h, starting from the state of pool slot
 * state_indices[n] (slot n when NULL) and writing the final state back to it,
 * with the output o, and nothing saved for a backward. Same layouts, head
 * mapping and scale rules as kda_fwd (fixed layout with cu_seqlens NULL;
 * packed with B = 1, device cu_seqlens and its trusted host mirror); d and
 * beta as the gate modes above say. With use_gate_in_kernel = 1 and
 * beta_is_logit = 1 the arithmetic is that of kda_fwd, bit for bit. A BF16 pool
 * is read, carried in FP32 and written back rounded to nearest even.
 * With use_gate_in_kernel = 0, every g must lie in [-5, 0], the range of the
 * in-kernel gate: the chunked evaluation scales keys by the inverse of the
 * decay accumulated over up to 16 tokens, which leaves FP32 range below about
 * -5.4 per token. The kernel checks this; a value outside the range (or NaN)
 * sets bit 1 (value 2) of device_status and o and the pool are then unspecified.
 *   state            [num_slots, Hv, 128, 128] value-first, state_dtype
 *                    KDA_STATE_BF16 or KDA_STATE_FP32, read and written in place
 *   state_indices    device int32 [N] and its host mirror (both NULL, or both
 *                    set); in range, no slot used twice. The kernel checks the
 *                    range of the device copy again: an index outside
 *                    [0, num_slots) sets bit 2 (value 4) of device_status and
 *                    leaves that sequence's slot alone (its o unspecified).
 *   o                BF16 [B, T, Hv, 128]
 *   checkpoints      optional BF16 [num_checkpoints, Hv, 128, 128] value-first:
 *                    for each sequence, rows checkpoint_cu_starts[n] + j hold
 *                    the state before token j * checkpoint_every_n_tokens
 *                    (row 0 is the initial state), j < ceil(len_n / N); the
 *                    device checkpoint_cu_starts [N + 1] and its host mirror must
 *                    hold those cumulative counts, ending at num_checkpoints.
 *                    checkpoint_every_n_tokens: a positive multiple of 16 (0
 *                    with checkpoints NULL).
 *   device_status    optional device int32: bit 0 (value 1) is set if a
 *                    bounded device wait gave up (then o and the pool are
 *                    incomplete), bits 1 and 2 (values 2, 4) as said above; bits are only
 *                    ever set, never cleared. NULL uses a word inside the library.
 * Units run in index order. Validation errors return before any launch;
 * otherwise the work is enqueued on `stream`. Nothing is allocated. */
kda_status kda_prefill(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                       const kda_bf16* beta, const float* A_log, const float* dt_bias,
                       const int64_t* cu_seqlens, const int64_t* cu_seqlens_host, int64_t num_seqs,
                       int64_t B, int64_t T, int64_t Hqk, int64_t Hv, int64_t head_dim, float scale,
                       float lower_bound, int32_t use_gate_in_kernel, int32_t beta_is_logit,
                       void* state, int32_t state_dtype, const int32_t* state_indices,
                       const int32_t* state_indices_host, int64_t num_slots, kda_bf16* o,
                       kda_bf16* checkpoints, int64_t num_checkpoints, const int64_t* checkpoint_cu_starts,
                       const int64_t* checkpoint_cu_starts_host, int64_t checkpoint_every_n_tokens,
                       int32_t* device_status, struct CUstream_st* stream);

/* Self-test of the device-side timeout path (no counterpart on the pages: the
 * kernels' own failure handling). Launches one CTA of 32 threads on `stream`
 * whose mbarrier wait can never complete, because nothing arrives on the
 * barrier. The wait is the same bounded wait the kernels use, with a limit of
 * 2^21 SM clock cycles (about 1 ms), after which the CTA writes a device status
 * word and exits; the call synchronises the stream and reads the word.
 * Returns KDA_ERR_DEVICE_TIMEOUT when the wait gave up (the expected outcome),
 * KDA_OK if it did not, KDA_ERR_UNSUPPORTED on a device that is not sm_103,
 * KDA_ERR_CUDA on a launch or copy error. Nothing faults, traps or hangs, and
 * the device and any contexts stay usable. Not for use inside stream capture. */
kda_status kda_selftest_device_timeout(struct CUstream_st* stream);

/* Internal tiling, for tooling and tests: sub-chunk length in tokens and the
 * checkpoint interval in tokens. */
int32_t kda_chunk_tokens(void);
int32_t kda_checkpoint_tokens(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
