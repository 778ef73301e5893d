// kda_step.cu -- one training step (forward + backward) from and to host memory:
// the inputs are copied into a caller-owned device arena, kda_fwd and kda_bwd
// run on the arena's copies, and the output and the eight gradients are copied
// back, all enqueued on one stream (flashinfer.kda_training: the forward's
// o / final_state and the backward's gradient list of
// flashinfer.kda_backward.recurrent_kda_backward).
//
// The call returns once the work is enqueued. With page-locked host buffers
// the copies run on the copy engines. The copies in, the kernels and the
// copies out may go to three streams, ordered by three events the context
// owns; with two arenas taken in turn, step i+1's inputs travel while step i
// computes and step i's outputs travel while step i+1 computes.
#include "../../include/kda.h"
#include "kda_common.cuh"

#include <cstdint>

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

kda_status sfail(kda_status st, const char* msg) {
  kda::set_last_error(msg);
  return st;
}

// Device copies in the arena, in this order, each 256-byte aligned; the
// context workspace comes last.
struct StepLayout {
  size_t q, k, v, g, beta, A_log, dt_bias, h0, cu, d_o, d_hT;  // inputs
  size_t o, h_T, dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dh0;  // outputs
  size_t ctx, ctx_bytes, total;
  // byte sizes
  size_t tok_qk, tok_v, beta_b, state_b, cu_b;
};

kda_status step_layout(int64_t B, int64_t T, int64_t Hqk, int64_t Hv, const int64_t* cu_host, int64_t num_seqs,
                       StepLayout* L) {
  size_t ctx_bytes = 0;
  kda_status st = kda_ctx_workspace_bytes(B, T, Hqk, Hv, cu_host, num_seqs, &ctx_bytes);
  if (st != KDA_OK) return st;
  const int64_t N = cu_host ? num_seqs : B;
  const size_t ttot = (size_t)B * T;
  L->tok_qk = 2 * ttot * Hqk * 128;
  L->tok_v = 2 * ttot * Hv * 128;
  L->beta_b = 2 * ttot * Hv;
  L->state_b = 4 * (size_t)N * Hv * 128 * 128;
  L->cu_b = cu_host ? 8 * (size_t)(N + 1) : 0;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t at = off; off = align_up(off + bytes); return at; };
  L->q = take(L->tok_qk);
  L->k = take(L->tok_qk);
  L->v = take(L->tok_v);
  L->g = take(L->tok_v);
  L->beta = take(L->beta_b);
  L->A_log = take(4 * (size_t)Hv);
  L->dt_bias = take(4 * (size_t)Hv * 128);
  L->h0 = take(L->state_b);
  L->cu = take(L->cu_b);
  L->d_o = take(L->tok_v);
  L->d_hT = take(L->state_b);
  L->o = take(L->tok_v);
  L->h_T = take(L->state_b);
  L->dq = take(L->tok_qk);
  L->dk = take(L->tok_qk);
  L->dv = take(L->tok_v);
  L->dg = take(L->tok_v);
  L->dbeta = take(L->beta_b);
  L->dA_log = take(4 * (size_t)Hv);
  L->ddt_bias = take(4 * (size_t)Hv * 128);
  L->dh0 = take(L->state_b);
  L->ctx = take(ctx_bytes);
  L->ctx_bytes = ctx_bytes;
  L->total = off;
  return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_step_arena_bytes(int64_t B, int64_t T, int64_t Hqk, int64_t Hv,
                                           const int64_t* cu_seqlens_host, int64_t num_seqs, size_t* bytes) {
  if (!bytes) return sfail(KDA_ERR_INVALID_ARGUMENT, "bytes is NULL");
  StepLayout L;
  const kda_status st = step_layout(B, T, Hqk, Hv, cu_seqlens_host, num_seqs, &L);
  if (st != KDA_OK) return st;
  *bytes = L.total;
  return KDA_OK;
}

extern "C" kda_status kda_step_host(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                                    const kda_bf16* beta, const float* A_log, const float* dt_bias,
                                    const float* h0, const int64_t* cu_seqlens_host, int64_t num_seqs, int64_t B,
                                    int64_t T, int64_t Hqk, int64_t Hv, int64_t head_dim, float scale,
                                    float lower_bound, const kda_bf16* d_o, const float* d_hT, kda_bf16* o,
                                    float* h_T, kda_bf16* dq, kda_bf16* dk, kda_bf16* dv, kda_bf16* dg,
                                    kda_bf16* dbeta, float* dA_log, float* ddt_bias, float* dh0, void* arena,
                                    size_t arena_bytes, kda_ctx** ctx, struct CUstream_st* stream_,
                                    struct CUstream_st* h2d_stream_, struct CUstream_st* d2h_stream_) {
  if (!ctx) return sfail(KDA_ERR_INVALID_ARGUMENT, "step: ctx is NULL");
  if (!q || !k || !v || !g || !beta || !A_log || !dt_bias || !h0 || !d_o || !d_hT || !o || !h_T || !dq || !dk ||
      !dv || !dg || !dbeta || !dA_log || !ddt_bias || !dh0 || !arena)
    return sfail(KDA_ERR_INVALID_ARGUMENT, "step: a required pointer is NULL");
  if (head_dim != 128) return sfail(KDA_ERR_UNSUPPORTED, "step: head dimension must be 128");
  StepLayout L;
  kda_status st = step_layout(B, T, Hqk, Hv, cu_seqlens_host, num_seqs, &L);
  if (st != KDA_OK) return st;
  if (arena_bytes < L.total) return sfail(KDA_ERR_WORKSPACE_TOO_SMALL, "step: arena smaller than kda_step_arena_bytes()");
  if ((uintptr_t)arena % kAlign != 0) return sfail(KDA_ERR_INVALID_ARGUMENT, "step: arena must be 256-byte aligned");
  // every host pointer must be host memory (page-locked for the copies to be asynchronous)
  const void* host_ptrs[] = {q, k, v, g, beta, A_log, dt_bias, h0, d_o, d_hT,
                             o, h_T, dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dh0};
  for (const void* p : host_ptrs) {
    cudaPointerAttributes at{};
    const cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return sfail(KDA_ERR_CUDA, "step: cudaPointerGetAttributes failed on a host buffer");
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged)
      return sfail(KDA_ERR_INVALID_ARGUMENT, "step: inputs and outputs must be host buffers (device memory given)");
  }
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  cudaStream_t h2d = h2d_stream_ ? reinterpret_cast<cudaStream_t>(h2d_stream_) : stream;
  cudaStream_t d2h = d2h_stream_ ? reinterpret_cast<cudaStream_t>(d2h_stream_) : stream;
  // events of this arena's previous step (a context lives with one arena): its
  // kernels must be done reading the inputs before new ones are copied in, and
  // its outputs copied out before the kernels overwrite them
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  cudaError_t e;
  if (*ctx && (e = kda::step_events(*ctx, ev)) != cudaSuccess) return sfail(KDA_ERR_CUDA, cudaGetErrorString(e));
  if (ev[1] && (e = cudaStreamWaitEvent(h2d, ev[1], 0)) != cudaSuccess)
    return sfail(KDA_ERR_CUDA, cudaGetErrorString(e));
  char* a = static_cast<char*>(arena);
  const struct {
    size_t off;
    const void* src;
    size_t bytes;
  } ins[] = {{L.q, q, L.tok_qk},          {L.k, k, L.tok_qk},          {L.v, v, L.tok_v},
             {L.g, g, L.tok_v},           {L.beta, beta, L.beta_b},    {L.A_log, A_log, 4 * (size_t)Hv},
             {L.dt_bias, dt_bias, 4 * (size_t)Hv * 128}, {L.h0, h0, L.state_b}, {L.cu, cu_seqlens_host, L.cu_b},
             {L.d_o, d_o, L.tok_v},       {L.d_hT, d_hT, L.state_b}};
  for (const auto& c : ins) {
    if (c.bytes == 0) continue;
    if ((e = cudaMemcpyAsync(a + c.off, c.src, c.bytes, cudaMemcpyHostToDevice, h2d)) != cudaSuccess)
      return sfail(KDA_ERR_CUDA, cudaGetErrorString(e));
  }
  cudaEvent_t in_done = nullptr;
  if (*ctx) {
    in_done = ev[0];
    if ((e = cudaEventRecord(in_done, h2d)) != cudaSuccess || (e = cudaStreamWaitEvent(stream, in_done, 0)) != cudaSuccess ||
        (ev[2] && (e = cudaStreamWaitEvent(stream, ev[2], 0)) != cudaSuccess))
      return sfail(KDA_ERR_CUDA, cudaGetErrorString(e));
  } else if (h2d != stream) {
    // first step of this arena: no context (and no events) yet; order through a temporary event
    if ((e = cudaEventCreateWithFlags(&in_done, cudaEventDisableTiming)) != cudaSuccess)
      return sfail(KDA_ERR_CUDA, cudaGetErrorString(e));
    e = cudaEventRecord(in_done, h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, in_done, 0);
    cudaEventDestroy(in_done);
    if (e != cudaSuccess) return sfail(KDA_ERR_CUDA, cudaGetErrorString(e));
  }
  auto bf = [&](size_t off) { return reinterpret_cast<kda_bf16*>(a + off); };
  auto f32 = [&](size_t off) { return reinterpret_cast<float*>(a + off); };
  st = kda_fwd(bf(L.q), bf(L.k), bf(L.v), bf(L.g), bf(L.beta), f32(L.A_log), f32(L.dt_bias), f32(L.h0),
               cu_seqlens_host ? reinterpret_cast<const int64_t*>(a + L.cu) : nullptr, cu_seqlens_host, num_seqs, B, T,
               Hqk, Hv, head_dim, scale, lower_bound, bf(L.o), f32(L.h_T), a + L.ctx, L.ctx_bytes, ctx, stream_);
  if (st != KDA_OK) return st;
  st = kda_bwd(*ctx, bf(L.d_o), f32(L.d_hT), bf(L.dq), bf(L.dk), bf(L.dv), bf(L.dg), bf(L.dbeta), f32(L.dA_log),
               f32(L.ddt_bias), f32(L.dh0), stream_);
  if (st != KDA_OK) return st;
  if ((e = kda::step_events(*ctx, ev)) != cudaSuccess || (e = cudaEventRecord(ev[1], stream)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(d2h, ev[1], 0)) != cudaSuccess)
    return sfail(KDA_ERR_CUDA, cudaGetErrorString(e));
  const struct {
    void* dst;
    size_t off;
    size_t bytes;
  } outs[] = {{o, L.o, L.tok_v},          {h_T, L.h_T, L.state_b},   {dq, L.dq, L.tok_qk},
              {dk, L.dk, L.tok_qk},       {dv, L.dv, L.tok_v},       {dg, L.dg, L.tok_v},
              {dbeta, L.dbeta, L.beta_b}, {dA_log, L.dA_log, 4 * (size_t)Hv},
              {ddt_bias, L.ddt_bias, 4 * (size_t)Hv * 128}, {dh0, L.dh0, L.state_b}};
  for (const auto& c : outs) {
    if ((e = cudaMemcpyAsync(c.dst, a + c.off, c.bytes, cudaMemcpyDeviceToHost, d2h)) != cudaSuccess)
      return sfail(KDA_ERR_CUDA, cudaGetErrorString(e));
  }
  if ((e = cudaEventRecord(ev[2], d2h)) != cudaSuccess) return sfail(KDA_ERR_CUDA, cudaGetErrorString(e));
  return KDA_OK;
}
