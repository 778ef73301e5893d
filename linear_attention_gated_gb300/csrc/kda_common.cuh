// kda_common.cuh -- constants, launch parameters and small device helpers
// shared by the KDA forward and backward kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

struct kda_ctx;  // the saved-forward context of the C ABI (kda_api.cu)

namespace kda {

constexpr int kDim = 128;      // K = V = 128 (flashinfer.kda_training, module description)
constexpr int kChunk = 16;     // tokens per sub-chunk of the chunked (WY / UT) form
constexpr int kCkTokens = 16;  // tokens between saved state checkpoints (multiple of kChunk)
constexpr int kLds = 132;      // padded shared-memory row stride (floats) of 128-wide tiles
constexpr float kNormEps = 1e-6f;  // L2-norm epsilon (recurrent_kda_backward, description)

// One (sequence, value head) pair is a "unit"; it owns one 128x128 state.
struct SeqInfo {
  int64_t t0;       // first token of the sequence on the packed token axis
  int64_t len;      // tokens in the sequence (>= 1)
  int64_t ck_base;  // first checkpoint slot of the sequence
  int64_t ch_base;  // first sub-chunk slot of the sequence (sub-chunk tapes)
};

struct Problem {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* g;
  const __nv_bfloat16* beta;
  const float* A_log;
  const float* dt_bias;
  const float* h0;
  const int32_t* order;   // launch slot -> unit id (n * Hv + h), longest sequence first
  const SeqInfo* seq;     // [N]
  float* ckpt;            // [n_ck, Hv, 128 x 128] state at the start of every checkpoint interval,
                          // element (v, k) at ckpt_index(v, k) (see below)
  float* utape;           // [Ttot, Hv, 128]: u_t = v_t - S'_t k^_t of every token (forward -> backward)
  float* abtape;          // [n_sub_chunks, Hv, 2, 16, 16]: the FP32 A (strictly lower) and B (lower)
                          // matrices of every sub-chunk (forward -> backward)
  int32_t* status;        // device status word: bit 0 when a bounded device wait gave up, bit 1
                          // when a prefill log-space gate value is outside [-5, 0]
  int64_t N, Hqk, Hv;
  int32_t r;              // Hv / Hqk
  float scale, lb;
};

struct FwdOut {
  __nv_bfloat16* o;
  float* hT;
};

// Inference prefill (the forward without tapes or training checkpoints): the
// initial state comes from a state-pool slot and the final state goes back to
// it; optional BF16 state checkpoints every ck_every_chunks sub-chunks.
struct PrefillArgs {
  const int64_t* cu;           // device cu_seqlens [N + 1], or null for B sequences of T tokens
  int64_t T;                   // tokens per sequence in the fixed layout
  const int32_t* slots;        // pool slot per sequence, or null (slot n)
  int64_t num_slots;           // slots in the pool
  void* pool;                  // [num_slots, Hv, 128, 128] value-first, BF16 or FP32, in place
  int pool_bf16;               // 1: BF16 pool, 0: FP32 pool
  __nv_bfloat16* ck;           // [C, Hv, 128, 128] BF16 value-first, or null
  const int64_t* ck_starts;    // [N + 1] first checkpoint row of each sequence
  int ck_every_chunks;         // checkpoint interval in sub-chunks
  int gate_in_kernel;          // 1: d = exp(lb sigmoid(exp(A_log)(g + dt_bias))); 0: g is log d, in [-5, 0]
  int beta_logit;              // 1: beta = sigmoid(input); 0: the input is beta
};

struct BwdArgs {
  const __nv_bfloat16* d_o;
  const float* d_hT;
  __nv_bfloat16* dq;     // written directly when r == 1
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  __nv_bfloat16* dg;
  __nv_bfloat16* dbeta;
  float* dh0;
  float* dqk_part;       // r > 1: [Ttot, Hv, 2, 128] per-value-head d(q^), d(k^)
  float* par_part;       // [N * Hv, kParStride]: per-unit ddt_bias (128) and dA_log (1)
};

constexpr int kParStride = 132;

// Position of state element (v, k) inside one saved checkpoint: value quads
// are outermost, then the key, then the 4 values of the quad. Copied unchanged
// to shared memory these bytes are S^T as a K-major tensor-core operand (rows
// k, K = v: 8-row groups 128 bytes apart, K-adjacent 4-element core matrices
// 2048 bytes apart), and a thread per key reads 16-byte runs of its own row
// with the warp covering 512 contiguous bytes.
__host__ __device__ __forceinline__ int ckpt_index(int v, int k) { return ((v >> 2) * 128 + k) * 4 + (v & 3); }

// Element maths of the prologue and epilogue. Divisions use __fdividef (at most
// 2 ulp off for divisors in [2^-126, 2^126], 0 for an infinite divisor), the
// sigmoids __expf (its error grows with |x|, but where e^-x is not negligible
// next to 1, |x| < 20, it stays near 1e-6 relative) and the norm factor rsqrtf:
// none has a special-case branch, so the eight independent per-thread chains
// interleave. Forward and backward call the same
// functions, so they see bit-identical decays and normalised vectors.
__device__ __forceinline__ float sigmoid_of(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
__device__ __forceinline__ float log_decay_of(float lb, float z) { return __fdividef(lb, 1.0f + __expf(-z)); }
__device__ __forceinline__ float inv_norm_of(float sumsq) { return rsqrtf(sumsq + kNormEps); }

__device__ __forceinline__ void unpack_bf16x8(const uint4 raw, float* out) {
  const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h2[i]);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ void load_bf16x8(const __nv_bfloat16* p, float* out) {
  uint4 raw = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h2[i]);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ void store_bf16x8(__nv_bfloat16* p, const float* in) {
  uint4 raw;
  __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) h2[i] = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = raw;
}

// acc += a * b elementwise: four independent FMA chains for long dot products
// (one running sum would make every FMA wait for the previous one).
__device__ __forceinline__ void fma4(float4& acc, float4 a, float4 b) {
  acc.x = fmaf(a.x, b.x, acc.x);
  acc.y = fmaf(a.y, b.y, acc.y);
  acc.z = fmaf(a.z, b.z, acc.z);
  acc.w = fmaf(a.w, b.w, acc.w);
}
__device__ __forceinline__ float hsum4(float4 a) { return (a.x + a.y) + (a.z + a.w); }

// Sum over the 16 lanes that share a token row (lanes 0-15 or 16-31 of a warp).
__device__ __forceinline__ float row16_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 8);
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x;
}

// Sets the message kda_last_error_message() returns on this thread (kda_api.cu).
void set_last_error(const char* msg);

// The three events kda_step_host orders its streams with, owned by the context
// and created on first use (kda_api.cu): [0] inputs copied in, [1] forward and
// backward done, [2] outputs copied out.
cudaError_t step_events(::kda_ctx* c, cudaEvent_t ev[3]);

// Launchers (defined in kda_fwd.cu / kda_bwd.cu).
cudaError_t launch_forward(const Problem& P, const FwdOut& out, int64_t units, cudaStream_t s);
cudaError_t launch_prefill(const Problem& P, const FwdOut& out, const PrefillArgs& pf, int64_t units,
                           cudaStream_t s);
cudaError_t launch_backward(const Problem& P, const BwdArgs& a, int64_t units, int64_t Ttot,
                            float* dA_log, float* ddt_bias, cudaStream_t s);

}  // namespace kda
