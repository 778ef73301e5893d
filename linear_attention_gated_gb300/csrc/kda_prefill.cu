// kda_prefill.cu -- host side of kda_prefill: inference prefill over whole
// sequences from a state pool (flashinfer.kda.recurrent_kda, parameters
// initial_state "Updated in-place", ssm_state_indices, state_checkpoints,
// checkpoint_cu_starts and checkpoint_every_n_tokens). The recurrence runs in
// the training forward kernel's prefill instantiation (kda_fwd.cu): the same
// chunked arithmetic, without the backward's tapes and checkpoints, with the
// initial state read from and the final state written back to the pool slot,
// optional BF16 state checkpoints, and the page's gate modes (g precomputed in
// log space, beta already sigmoided).
#include "../../include/kda.h"
#include "kda_common.cuh"
#include "kda_host.h"

#include <cmath>
#include <unordered_set>
#include <vector>

namespace {

__device__ int32_t g_prefill_status;

kda_status pfail(kda_status st, const char* msg) {
  kda::set_last_error(msg);
  return st;
}

struct Span {
  const void* p;
  size_t bytes;
};

bool overlap(const Span& a, const Span& b) {
  const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
  return a.p && b.p && a.bytes && b.bytes && a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

}  // namespace

extern "C" kda_status kda_prefill(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                                  const kda_bf16* beta, const float* A_log, const float* dt_bias,
                                  const int64_t* cu_seqlens, const int64_t* cu_seqlens_host, int64_t num_seqs,
                                  int64_t B, int64_t T, int64_t Hqk, int64_t Hv, int64_t head_dim, float scale,
                                  float lower_bound, int32_t use_gate_in_kernel, int32_t beta_is_logit,
                                  void* state, int32_t state_dtype,
                                  const int32_t* state_indices, const int32_t* state_indices_host,
                                  int64_t num_slots, kda_bf16* o, kda_bf16* checkpoints,
                                  int64_t num_checkpoints, const int64_t* checkpoint_cu_starts,
                                  const int64_t* checkpoint_cu_starts_host, int64_t checkpoint_every_n_tokens,
                                  int32_t* device_status, struct CUstream_st* stream) {
  return kda::guarded([&]() -> kda_status {
    // ---- shapes and layout
    if (B < 1 || T < 1) return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: B and T must be >= 1");
    if (Hqk < 1 || Hv < 1 || Hv % Hqk != 0)
      return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: Hv must be a positive multiple of Hqk");
    if (head_dim != kda::kDim) return pfail(KDA_ERR_UNSUPPORTED, "prefill: head_dim must be 128");
    if (kda::size_limit_violation(B, T, Hv, cu_seqlens_host ? num_seqs : 0))
      return pfail(KDA_ERR_UNSUPPORTED, "prefill: problem too large (over 2^40 tokens or token-heads, "
                                        "2^20 heads, or more sequences than tokens)");
    if (num_slots > (int64_t(1) << 31) || num_checkpoints > (int64_t(1) << 31))
      return pfail(KDA_ERR_UNSUPPORTED, "prefill: more than 2^31 pool slots or checkpoints");
    const float s_def = 1.0f / std::sqrt((float)kda::kDim);
    if (!std::isnan(scale) && scale != s_def)
      return pfail(KDA_ERR_UNSUPPORTED, "prefill: scale must be 1/sqrt(128) (NaN selects it)");
    if ((use_gate_in_kernel != 0 && use_gate_in_kernel != 1) || (beta_is_logit != 0 && beta_is_logit != 1))
      return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: use_gate_in_kernel and beta_is_logit must be 0 or 1");
    if (use_gate_in_kernel && lower_bound != -5.0f)
      return pfail(KDA_ERR_UNSUPPORTED, "prefill: lower_bound must be -5 with the gate computed in the kernel");
    if (state_dtype != KDA_STATE_BF16 && state_dtype != KDA_STATE_FP32)
      return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: state_dtype must be KDA_STATE_BF16 or KDA_STATE_FP32");
    if (!q || !k || !v || !g || !beta || !state || !o || (use_gate_in_kernel && (!A_log || !dt_bias)))
      return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: null tensor pointer");
    if ((cu_seqlens == nullptr) != (cu_seqlens_host == nullptr))
      return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: cu_seqlens needs its host mirror (and the reverse)");
    std::vector<int64_t> cu;
    int64_t N;
    if (cu_seqlens_host == nullptr) {
      N = B;
      for (int64_t i = 0; i <= B; ++i) cu.push_back(i * T);
    } else {
      if (B != 1) return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: packed input needs a physical batch of one");
      if (num_seqs < 1) return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: packed input needs num_seqs >= 1");
      N = num_seqs;
      cu.assign(cu_seqlens_host, cu_seqlens_host + N + 1);
      if (cu[0] != 0 || cu[N] != T) return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: cu_seqlens must run from 0 to T");
      for (int64_t i = 0; i < N; ++i)
        if (cu[i + 1] <= cu[i])
          return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: a sequence is empty or cu_seqlens decreases");
    }
    if (N * Hv > INT32_MAX) return pfail(KDA_ERR_UNSUPPORTED, "prefill: too many (sequence, head) units");
    const int64_t Ttot = B * T;
    // ---- state pool slots
    if ((state_indices == nullptr) != (state_indices_host == nullptr))
      return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: state_indices needs its host mirror (and the reverse)");
    if (state_indices_host) {
      std::unordered_set<int32_t> seen;
      for (int64_t i = 0; i < N; ++i) {
        const int32_t sl = state_indices_host[i];
        if (sl < 0 || sl >= num_slots) return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: state index out of range");
        if (!seen.insert(sl).second) return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: two sequences share a state slot");
      }
    } else if (num_slots < N) {
      return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: without state_indices the pool needs a slot per sequence");
    }
    // ---- checkpoints: ceil(len / N) rows per sequence, counted by checkpoint_cu_starts
    if (checkpoints) {
      if (checkpoint_every_n_tokens <= 0 || checkpoint_every_n_tokens % kda::kChunk != 0)
        return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: checkpoint_every_n_tokens must be a positive multiple of 16");
      if (!checkpoint_cu_starts || !checkpoint_cu_starts_host)
        return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: checkpoints need checkpoint_cu_starts and its host mirror");
      if (checkpoint_cu_starts_host[0] != 0) return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: checkpoint_cu_starts must start at 0");
      for (int64_t i = 0; i < N; ++i) {
        const int64_t want = (cu[i + 1] - cu[i] + checkpoint_every_n_tokens - 1) / checkpoint_every_n_tokens;
        if (checkpoint_cu_starts_host[i + 1] - checkpoint_cu_starts_host[i] != want)
          return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: checkpoint counts must be ceil(len / checkpoint_every_n_tokens)");
      }
      if (checkpoint_cu_starts_host[N] != num_checkpoints)
        return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: checkpoint_cu_starts must end at num_checkpoints");
    } else if (checkpoint_every_n_tokens != 0) {
      return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: checkpoint_every_n_tokens without a checkpoint buffer");
    }
    // ---- alignment and aliasing
    const void* ptrs[] = {q, k, v, g, state, o, checkpoints};
    for (const void* p : ptrs)
      if ((uintptr_t)p & 15u) return pfail(KDA_ERR_INVALID_ARGUMENT, "prefill: token and state tensors must be 16-byte aligned");
    const size_t esz = state_dtype == KDA_STATE_BF16 ? 2 : 4;
    const size_t st_elems = (size_t)kda::kDim * kda::kDim;
    const Span outs[] = {{state, esz * (size_t)num_slots * Hv * st_elems},
                         {o, 2 * (size_t)Ttot * Hv * kda::kDim},
                         {checkpoints, 2 * (size_t)num_checkpoints * Hv * st_elems},
                         {device_status, device_status ? sizeof(int32_t) : 0}};
    const Span ins[] = {{q, 2 * (size_t)Ttot * Hqk * kda::kDim}, {k, 2 * (size_t)Ttot * Hqk * kda::kDim},
                        {v, 2 * (size_t)Ttot * Hv * kda::kDim},  {g, 2 * (size_t)Ttot * Hv * kda::kDim},
                        {beta, 2 * (size_t)Ttot * Hv},
                        {A_log, use_gate_in_kernel ? 4 * (size_t)Hv : 0},
                        {dt_bias, use_gate_in_kernel ? 4 * (size_t)Hv * kda::kDim : 0},
                        {cu_seqlens, cu_seqlens ? 8 * (size_t)(N + 1) : 0},
                        {state_indices, state_indices ? 4 * (size_t)N : 0},
                        {checkpoint_cu_starts, checkpoint_cu_starts ? 8 * (size_t)(N + 1) : 0}};
    for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
      for (const Span& in : ins)
        if (overlap(in, outs[i])) return pfail(KDA_ERR_ALIASING, "prefill: an input overlaps an output");
      for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
        if (overlap(outs[i], outs[j])) return pfail(KDA_ERR_ALIASING, "prefill: two outputs overlap");
    }
    // ---- device
    int dev = -1, major = 0, minor = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return pfail(KDA_ERR_CUDA, cudaGetErrorString(e));
    if (major != 10 || minor != 3) return pfail(KDA_ERR_UNSUPPORTED, "prefill: kernels are built for sm_103a");
    int32_t* status = device_status;
    if (!status && (e = cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_prefill_status)) != cudaSuccess)
      return pfail(KDA_ERR_CUDA, cudaGetErrorString(e));

    kda::Problem P{};
    P.q = reinterpret_cast<const __nv_bfloat16*>(q);
    P.k = reinterpret_cast<const __nv_bfloat16*>(k);
    P.v = reinterpret_cast<const __nv_bfloat16*>(v);
    P.g = reinterpret_cast<const __nv_bfloat16*>(g);
    P.beta = reinterpret_cast<const __nv_bfloat16*>(beta);
    P.A_log = A_log;
    P.dt_bias = dt_bias;
    P.status = status;
    P.N = N;
    P.Hqk = Hqk;
    P.Hv = Hv;
    P.r = (int32_t)(Hv / Hqk);
    P.scale = s_def;
    P.lb = lower_bound;
    kda::FwdOut fo{reinterpret_cast<__nv_bfloat16*>(o), nullptr};
    kda::PrefillArgs pf{};
    pf.cu = cu_seqlens;
    pf.T = T;
    pf.slots = state_indices;
    pf.num_slots = num_slots;
    pf.pool = state;
    pf.pool_bf16 = state_dtype == KDA_STATE_BF16 ? 1 : 0;
    pf.ck = reinterpret_cast<__nv_bfloat16*>(checkpoints);
    pf.ck_starts = checkpoint_cu_starts;
    pf.ck_every_chunks = checkpoints ? (int)(checkpoint_every_n_tokens / kda::kChunk) : 1;
    pf.gate_in_kernel = use_gate_in_kernel;
    pf.beta_logit = beta_is_logit;
    if ((e = kda::launch_prefill(P, fo, pf, N * Hv, stream)) != cudaSuccess)
      return pfail(KDA_ERR_CUDA, cudaGetErrorString(e));
    return KDA_OK;
  });
}
