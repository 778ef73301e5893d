// kda_noalloc.cu -- kda_bwd_noalloc: the standalone backward for callers that
// cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: code that runs while another
// component owns every byte of device memory through its own pool (a framework
// caching allocator, an inference server that carves the GPU up front), hosts
// that forbid allocation inside a plug-in call, and latency-critical loops that
// cannot afford the device-wide synchronisation cudaMalloc / cudaFree may imply.
// They still own their inputs and outputs, but cannot provide the context
// workspace that kda_fwd / kda_bwd need. This entry point uses instead one
// fixed scratch array compiled into the library (kNoAllocScratchBytes below),
// resident on every GPU that loads the library until the process exits.
//
// It runs the same forward kernel (to rebuild the state checkpoints; its output
// and final state land in the scratch and are discarded) and the same backward
// and reduction kernels as kda_fwd + kda_bwd, with every intermediate buffer
// carved out of the scratch array in the context layout kda_fwd uses. Units run
// in index order (no host-side plan upload: a one-thread kernel writes the plan
// into the scratch). The first 256 bytes of the array hold the status word that
// kda_noalloc_status reads; each call clears it before its first launch.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "../../include/kda.h"
#include "kda_common.cuh"
#include "kda_host.h"
#include "kda_layout.h"

namespace {

constexpr size_t kNoAllocScratchBytes = KDA_NOALLOC_SCRATCH_BYTES;  // 64 MiB
constexpr size_t kStatusBytes = kda::kCtxAlign;                     // status word, then the context
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

kda_status nfail(kda_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  kda::set_last_error(buf);  // reported by kda_last_error_message()
  return st;
}

size_t up(size_t x) { return kda::ctx_align_up(x); }

// Device address of the scratch array on the current device, looked up once
// per device (the host-side symbol is only a stand-in for it).
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

kda_status scratch_for_device(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return nfail(KDA_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess)
      return nfail(KDA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KDA_OK;
}

kda_status current_sm103(int* dev_out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return nfail(KDA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  int major = 0, minor = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
    return nfail(KDA_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  if (major != 10 || minor != 3)
    return nfail(KDA_ERR_UNSUPPORTED, "kernels are built for sm_103a; device %d is compute capability %d.%d", dev,
                 major, minor);
  *dev_out = dev;
  return KDA_OK;
}

// Plan written on the device: identity unit order and per-sequence offsets, from
// the device cu_seqlens (null: B sequences of T tokens). The scratch was sized
// from the host mirror, so the device copy is checked against what that sizing
// relied on: it starts at 0, every sequence is non-empty, it ends at B * T and
// it gives the same checkpoint and sub-chunk totals. Then every token, checkpoint
// and sub-chunk index the kernels form stays inside its buffer. A copy that
// fails the check sets bit 2 (value 4) of the status word, and every sequence
// becomes the first token with base 0, which keeps all accesses in bounds (the
// gradients are then meaningless; kda_noalloc_status reports the error).
__global__ void kda_noalloc_plan_kernel(const int64_t* cu, int64_t B, int64_t T, int64_t N, int64_t Hv,
                                        int64_t n_ck, int64_t n_ch, int32_t* order, kda::SeqInfo* seq,
                                        int32_t* status) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    bool ok = cu == nullptr || cu[0] == 0;
    int64_t ck = 0, chn = 0;
    for (int64_t n = 0; n < N && ok; ++n) {
      const int64_t t0 = cu ? cu[n] : n * T;
      const int64_t len = (cu ? cu[n + 1] : (n + 1) * T) - t0;
      ok = len >= 1 && len <= B * T;
      seq[n].t0 = t0;
      seq[n].len = len;
      seq[n].ck_base = ck;
      seq[n].ch_base = chn;
      ck += kda::checkpoints_of(len);
      chn += kda::subchunks_of(len);
    }
    ok = ok && (cu == nullptr || cu[N] == B * T) && ck == n_ck && chn == n_ch;
    if (!ok) {
      for (int64_t n = 0; n < N; ++n) {
        seq[n].t0 = 0;
        seq[n].len = 1;
        seq[n].ck_base = 0;
        seq[n].ch_base = 0;
      }
      atomicOr(status, 4);
    }
  }
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < N * Hv;
       u += (int64_t)gridDim.x * blockDim.x)
    order[u] = (int32_t)u;
}

struct Range {
  const void* p;
  size_t bytes;
  const char* name;
};

bool overlap(const Range& a, const Range& b) {
  if (!a.p || !b.p || !a.bytes || !b.bytes) return false;
  const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

}  // namespace

extern "C" kda_status kda_bwd_noalloc(
    const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const kda_bf16* g, const kda_bf16* beta,
    const float* A_log, const float* dt_bias, const float* h0, const int64_t* cu_seqlens_dev,
    const int64_t* cu_seqlens_host, int64_t num_seqs, int64_t B, int64_t T, int64_t Hqk, int64_t Hv,
    int64_t head_dim, float scale, float lower_bound, const kda_bf16* d_o, const float* d_hT,
    kda_bf16* dq, kda_bf16* dk, kda_bf16* dv, kda_bf16* dg, kda_bf16* dbeta, float* dA_log,
    float* ddt_bias, float* dh0, struct CUstream_st* stream_) {
  return kda::guarded([&]() -> kda_status {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    kda::set_last_error("");
    if (!q || !k || !v || !g || !beta || !A_log || !dt_bias || !h0 || !d_o || !d_hT || !dq || !dk || !dv ||
        !dg || !dbeta || !dA_log || !ddt_bias || !dh0)
      return nfail(KDA_ERR_INVALID_ARGUMENT, "a required tensor pointer is NULL");
    if ((cu_seqlens_dev == nullptr) != (cu_seqlens_host == nullptr))
      return nfail(KDA_ERR_INVALID_ARGUMENT, "packed input needs both cu_seqlens and its host mirror");
    if (head_dim != kda::kDim) return nfail(KDA_ERR_UNSUPPORTED, "head dimension must be 128");
    const float s_req = (float)(1.0 / std::sqrt(128.0));
    if (std::isnan(scale)) scale = s_req;
    if (std::fabs(scale - s_req) > 1e-6f * s_req) return nfail(KDA_ERR_UNSUPPORTED, "scale must be 1/sqrt(128)");
    if (lower_bound != -5.0f) return nfail(KDA_ERR_UNSUPPORTED, "lower_bound must be -5");
    if (B < 1 || T < 1 || Hqk < 1 || Hv < 1 || Hv % Hqk != 0)
      return nfail(KDA_ERR_INVALID_ARGUMENT, "need B, T >= 1 and Hv a positive multiple of Hqk");
    if (const char* why = kda::size_limit_violation(B, T, Hv, cu_seqlens_host ? num_seqs : 0))
      return nfail(KDA_ERR_UNSUPPORTED, "problem too large: %s", why);
    int64_t N = B;
    int64_t n_ck = 0, n_ch = 0;
    if (cu_seqlens_host) {
      if (B != 1 || num_seqs < 1) return nfail(KDA_ERR_INVALID_ARGUMENT, "packed input needs B == 1, num_seqs >= 1");
      N = num_seqs;
      if (cu_seqlens_host[0] != 0 || cu_seqlens_host[N] != T)
        return nfail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must run from 0 to T");
      for (int64_t i = 0; i < N; ++i) {
        const int64_t len = cu_seqlens_host[i + 1] - cu_seqlens_host[i];
        if (len < 1) return nfail(KDA_ERR_INVALID_ARGUMENT, "sequence %lld is empty", (long long)i);
        n_ck += kda::checkpoints_of(len);
        n_ch += kda::subchunks_of(len);
      }
    } else {
      n_ck = B * kda::checkpoints_of(T);
      n_ch = B * kda::subchunks_of(T);
    }
    const void* vec_ptrs[] = {q, k, v, g, h0, d_o, d_hT, dq, dk, dv, dg, dh0};
    for (const void* p : vec_ptrs)
      if ((uintptr_t)p & 15u) return nfail(KDA_ERR_INVALID_ARGUMENT, "token and state tensors must be 16-byte aligned");

    const int64_t Ttot = B * T, units = N * Hv, r = Hv / Hqk;
    const size_t D = kda::kDim;
    // scratch layout: the status word, the context of kda_fwd, the forward's o and final state
    kda::CtxCounts cc;
    cc.N = N; cc.Ttot = Ttot; cc.Hqk = Hqk; cc.Hv = Hv; cc.n_ck = n_ck; cc.n_ch = n_ch;
    const kda::CtxLayout L = kda::context_layout(cc);
    size_t off = kStatusBytes;
    const size_t o_ctx = off;   off = up(off + L.total);
    const size_t o_o = off;     off = up(off + sizeof(kda_bf16) * (size_t)Ttot * Hv * D);
    const size_t o_hT = off;    off = up(off + sizeof(float) * (size_t)N * Hv * D * D);
    if (off > kNoAllocScratchBytes)
      return nfail(KDA_ERR_WORKSPACE_TOO_SMALL,
                   "problem needs %zu bytes of scratch; kda_bwd_noalloc has %zu (use kda_fwd + kda_bwd)",
                   off, kNoAllocScratchBytes);

    const size_t tok_qk = sizeof(kda_bf16) * (size_t)Ttot * Hqk * D, tok_v = sizeof(kda_bf16) * (size_t)Ttot * Hv * D;
    const size_t state = sizeof(float) * (size_t)N * Hv * D * D;
    const Range ins[] = {{q, tok_qk, "q"}, {k, tok_qk, "k"}, {v, tok_v, "v"}, {g, tok_v, "g"},
                         {beta, sizeof(kda_bf16) * (size_t)Ttot * Hv, "beta"}, {A_log, sizeof(float) * Hv, "A_log"},
                         {dt_bias, sizeof(float) * Hv * D, "dt_bias"}, {h0, state, "initial_state"},
                         {cu_seqlens_dev, cu_seqlens_dev ? sizeof(int64_t) * (N + 1) : 0, "cu_seqlens"},
                         {d_o, tok_v, "do"}, {d_hT, state, "dfinal_state"}};
    const Range outs[] = {{dq, tok_qk, "dq"}, {dk, tok_qk, "dk"}, {dv, tok_v, "dv"}, {dg, tok_v, "dg"},
                          {dbeta, sizeof(kda_bf16) * (size_t)Ttot * Hv, "dbeta"}, {dA_log, sizeof(float) * Hv, "dA_log"},
                          {ddt_bias, sizeof(float) * Hv * D, "ddt_bias"}, {dh0, state, "dinitial_state"}};
    for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
      for (const Range& in : ins)
        if (overlap(outs[i], in)) return nfail(KDA_ERR_ALIASING, "output %s overlaps %s", outs[i].name, in.name);
      for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
        if (overlap(outs[i], outs[j])) return nfail(KDA_ERR_ALIASING, "output %s overlaps %s", outs[i].name, outs[j].name);
    }

    int dev = -1;
    kda_status st = current_sm103(&dev);
    if (st != KDA_OK) return st;
    void* base = nullptr;
    st = scratch_for_device(dev, &base);
    if (st != KDA_OK) return st;
    char* sc = static_cast<char*>(base);
    char* cx = sc + o_ctx;
    int32_t* status = reinterpret_cast<int32_t*>(sc);

    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return nfail(KDA_ERR_CUDA, "status reset: %s", cudaGetErrorString(e));
    kda_noalloc_plan_kernel<<<(unsigned)((units + 255) / 256), 256, 0, stream>>>(
        cu_seqlens_dev, B, T, N, Hv, n_ck, n_ch, reinterpret_cast<int32_t*>(cx + L.order),
        reinterpret_cast<kda::SeqInfo*>(cx + L.seq), status);
    if ((e = cudaGetLastError()) != cudaSuccess) return nfail(KDA_ERR_CUDA, "plan launch: %s", cudaGetErrorString(e));

    kda::Problem P{};
    P.q = reinterpret_cast<const __nv_bfloat16*>(q);
    P.k = reinterpret_cast<const __nv_bfloat16*>(k);
    P.v = reinterpret_cast<const __nv_bfloat16*>(v);
    P.g = reinterpret_cast<const __nv_bfloat16*>(g);
    P.beta = reinterpret_cast<const __nv_bfloat16*>(beta);
    P.A_log = A_log;
    P.dt_bias = dt_bias;
    P.h0 = h0;
    P.order = reinterpret_cast<const int32_t*>(cx + L.order);
    P.seq = reinterpret_cast<const kda::SeqInfo*>(cx + L.seq);
    P.ckpt = reinterpret_cast<float*>(cx + L.ckpt);
    P.status = status;
    P.utape = reinterpret_cast<float*>(cx + L.utape);
    P.abtape = reinterpret_cast<float*>(cx + L.abtape);
    P.N = N;
    P.Hqk = Hqk;
    P.Hv = Hv;
    P.r = (int32_t)r;
    P.scale = scale;
    P.lb = lower_bound;
    kda::FwdOut fo{reinterpret_cast<__nv_bfloat16*>(sc + o_o), reinterpret_cast<float*>(sc + o_hT)};
    if ((e = kda::launch_forward(P, fo, units, stream)) != cudaSuccess)
      return nfail(KDA_ERR_CUDA, "forward launch: %s", cudaGetErrorString(e));
    kda::BwdArgs a{};
    a.d_o = reinterpret_cast<const __nv_bfloat16*>(d_o);
    a.d_hT = d_hT;
    a.dq = reinterpret_cast<__nv_bfloat16*>(dq);
    a.dk = reinterpret_cast<__nv_bfloat16*>(dk);
    a.dv = reinterpret_cast<__nv_bfloat16*>(dv);
    a.dg = reinterpret_cast<__nv_bfloat16*>(dg);
    a.dbeta = reinterpret_cast<__nv_bfloat16*>(dbeta);
    a.dh0 = dh0;
    a.dqk_part = reinterpret_cast<float*>(cx + L.dqk);
    a.par_part = reinterpret_cast<float*>(cx + L.par);
    if ((e = kda::launch_backward(P, a, units, Ttot, dA_log, ddt_bias, stream)) != cudaSuccess)
      return nfail(KDA_ERR_CUDA, "backward launch: %s", cudaGetErrorString(e));
    return KDA_OK;
  });
}

extern "C" kda_status kda_noalloc_status(struct CUstream_st* stream_) {
  return kda::guarded([&]() -> kda_status {
    kda::set_last_error("");
    int dev = -1;
    kda_status st = current_sm103(&dev);
    if (st != KDA_OK) return st;
    void* base = nullptr;
    if ((st = scratch_for_device(dev, &base)) != KDA_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return nfail(KDA_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
    int32_t word = 0;
    e = cudaMemcpy(&word, base, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return nfail(KDA_ERR_CUDA, "status readback: %s", cudaGetErrorString(e));
    if (word & 4)
      return nfail(KDA_ERR_INVALID_ARGUMENT, "the device cu_seqlens disagreed with its host mirror (status %d)", word);
    if (word & 1) return nfail(KDA_ERR_DEVICE_TIMEOUT, "a bounded device wait gave up (status %d)", word);
    if (word != 0) return nfail(KDA_ERR_CUDA, "unexpected device status %d", word);
    return KDA_OK;
  });
}
