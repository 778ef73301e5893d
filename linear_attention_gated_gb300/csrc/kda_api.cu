// kda_api.cu -- host side of the C ABI declared in include/kda.h: argument
// validation, the longest-sequence-first launch plan, the context workspace
// layout, and the kernel launches. No allocation happens here: the caller owns
// every device buffer, including the context workspace.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/kda.h"
#include "kda_common.cuh"
#include "kda_host.h"
#include "kda_layout.h"
#include "tc.cuh"

using kda::SeqInfo;

namespace {

thread_local std::string g_last_error;

kda_status fail(kda_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

kda_status cuda_fail(cudaError_t e, const char* where) {
  return fail(KDA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

constexpr size_t kAlign = kda::kCtxAlign;

struct Shape {
  int64_t B = 0, T = 0, Hqk = 0, Hv = 0, N = 0, Ttot = 0, units = 0, n_ck = 0, n_ch = 0;
  bool packed = false;
  std::vector<int64_t> cu;  // N + 1 token offsets
  bool operator==(const Shape& o) const {
    return B == o.B && T == o.T && Hqk == o.Hqk && Hv == o.Hv && packed == o.packed && cu == o.cu;
  }
};

using Layout = kda::CtxLayout;

Layout make_layout(const Shape& s) {
  kda::CtxCounts c;
  c.N = s.N; c.Ttot = s.Ttot; c.Hqk = s.Hqk; c.Hv = s.Hv; c.n_ck = s.n_ck; c.n_ch = s.n_ch;
  return kda::context_layout(c);
}

// Validates sizes and the host cu_seqlens mirror; fills the Shape.
kda_status make_shape(int64_t B, int64_t T, int64_t Hqk, int64_t Hv, const int64_t* cu_host,
                      int64_t num_seqs, Shape* out) {
  Shape s;
  if (B < 1 || T < 1) return fail(KDA_ERR_INVALID_ARGUMENT, "B and T must be >= 1 (got B=%lld T=%lld)",
                                  (long long)B, (long long)T);
  if (Hqk < 1 || Hv < 1 || Hv % Hqk != 0)
    return fail(KDA_ERR_INVALID_ARGUMENT, "Hv must be a positive multiple of Hqk (Hqk=%lld Hv=%lld)",
                (long long)Hqk, (long long)Hv);
  if (Hv / Hqk > 1024) return fail(KDA_ERR_UNSUPPORTED, "Hv / Hqk above 1024 is not supported");
  if (const char* why = kda::size_limit_violation(B, T, Hv, cu_host ? num_seqs : 0))
    return fail(KDA_ERR_UNSUPPORTED, "problem too large: %s", why);
  s.B = B; s.T = T; s.Hqk = Hqk; s.Hv = Hv;
  if (cu_host == nullptr) {
    s.packed = false;
    s.N = B;
    s.cu.resize(B + 1);
    for (int64_t i = 0; i <= B; ++i) s.cu[i] = i * T;
  } else {
    if (B != 1) return fail(KDA_ERR_INVALID_ARGUMENT, "packed input needs a physical batch of one (B=%lld)", (long long)B);
    if (num_seqs < 1) return fail(KDA_ERR_INVALID_ARGUMENT, "packed input needs num_seqs >= 1");
    s.packed = true;
    s.N = num_seqs;
    s.cu.assign(cu_host, cu_host + num_seqs + 1);
    if (s.cu[0] != 0) return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must start at 0");
    if (s.cu[num_seqs] != T)
      return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must end at the token count %lld (got %lld)",
                  (long long)T, (long long)s.cu[num_seqs]);
    for (int64_t i = 0; i < num_seqs; ++i)
      if (s.cu[i + 1] <= s.cu[i])
        return fail(KDA_ERR_INVALID_ARGUMENT, "sequence %lld is empty or cu_seqlens decreases", (long long)i);
  }
  s.Ttot = B * T;
  if (s.N * Hv > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "too many (sequence, head) units");
  s.units = s.N * Hv;
  s.n_ck = 0;
  s.n_ch = 0;
  for (int64_t i = 0; i < s.N; ++i) {
    s.n_ck += kda::checkpoints_of(s.cu[i + 1] - s.cu[i]);
    s.n_ch += kda::subchunks_of(s.cu[i + 1] - s.cu[i]);
  }
  *out = std::move(s);
  return KDA_OK;
}

struct Range {
  const void* p;
  size_t bytes;
  const char* name;
};

bool overlaps(const Range& a, const Range& b) {
  if (!a.p || !b.p || !a.bytes || !b.bytes) return false;
  const uintptr_t a0 = (uintptr_t)a.p, a1 = a0 + a.bytes;
  const uintptr_t b0 = (uintptr_t)b.p, b1 = b0 + b.bytes;
  return a0 < b1 && b0 < a1;
}

// Every output must be disjoint from every input and from every other output.
kda_status check_aliasing(const std::vector<Range>& inputs, const std::vector<Range>& outputs) {
  for (size_t i = 0; i < outputs.size(); ++i) {
    for (const Range& in : inputs)
      if (overlaps(outputs[i], in))
        return fail(KDA_ERR_ALIASING, "output %s overlaps %s", outputs[i].name, in.name);
    for (size_t j = i + 1; j < outputs.size(); ++j)
      if (overlaps(outputs[i], outputs[j]))
        return fail(KDA_ERR_ALIASING, "output %s overlaps output %s", outputs[i].name, outputs[j].name);
  }
  return KDA_OK;
}

kda_status check_device(int* dev_out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3)
    return fail(KDA_ERR_UNSUPPORTED, "kernels are built for sm_103a; device %d is compute capability %d.%d",
                dev, major, minor);
  *dev_out = dev;
  return KDA_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

void kda::set_last_error(const char* msg) { g_last_error = msg; }

namespace {

__device__ int32_t g_selftest_status;

// One CTA waits on an mbarrier that nothing arrives at; the bounded wait must
// give up after `limit` cycles and the CTA records that in the status word.
__global__ void kda_selftest_timeout_kernel(long long limit) {
  __shared__ unsigned long long mbar;
  if (threadIdx.x == 0) kda::tc::mbar_init(kda::tc::smem_u32(&mbar), 1);
  __syncthreads();
  const bool completed = kda::tc::mbar_wait(kda::tc::smem_u32(&mbar), 0, limit);
  if (threadIdx.x == 0) g_selftest_status = completed ? 0 : 1;
}

}  // namespace

struct kda_ctx {
  Shape shape;
  Layout layout;
  int device = -1;
  cudaStream_t stream = nullptr;
  char* ws = nullptr;
  size_t ws_bytes = 0;
  std::vector<int32_t> order;
  std::vector<SeqInfo> seq;
  bool forward_done = false;
  kda::Problem prob{};
  std::vector<Range> inputs;  // borrowed forward inputs, for the backward's aliasing checks
  cudaEvent_t step_ev[3] = {nullptr, nullptr, nullptr};  // kda_step_host stream ordering
  ~kda_ctx() {
    for (cudaEvent_t e : step_ev)
      if (e) cudaEventDestroy(e);
  }
};

cudaError_t kda::step_events(kda_ctx* c, cudaEvent_t ev[3]) {
  for (int i = 0; i < 3; ++i) {
    if (!c->step_ev[i]) {
      const cudaError_t e = cudaEventCreateWithFlags(&c->step_ev[i], cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
    }
    ev[i] = c->step_ev[i];
  }
  return cudaSuccess;
}

extern "C" {

const char* kda_status_string(kda_status st) {
  switch (st) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported configuration";
    case KDA_ERR_ALIASING: return "output overlaps an input, another output or the context";
    case KDA_ERR_CONTEXT: return "context mismatch or misuse";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case KDA_ERR_WORKSPACE_TOO_SMALL: return "context workspace too small";
  }
  return "unknown status";
}

const char* kda_last_error_message(void) { return g_last_error.c_str(); }

kda_status kda_selftest_device_timeout(struct CUstream_st* stream) {
  int dev = -1;
  kda_status st = check_device(&dev);
  if (st != KDA_OK) return st;
  const int32_t unset = -1;
  cudaError_t e = cudaMemcpyToSymbolAsync(g_selftest_status, &unset, sizeof(unset), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return cuda_fail(e, "self-test status reset");
  kda_selftest_timeout_kernel<<<1, 32, 0, stream>>>(1ll << 21);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "self-test launch");
  int32_t status = -1;
  e = cudaMemcpyFromSymbolAsync(&status, g_selftest_status, sizeof(status), 0, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return cuda_fail(e, "self-test status read");
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "self-test synchronise");
  if (status == 1) return fail(KDA_ERR_DEVICE_TIMEOUT, "self-test: the device-side wait gave up as designed");
  if (status == 0) return KDA_OK;
  return fail(KDA_ERR_CUDA, "self-test: status word not written");
}

int32_t kda_chunk_tokens(void) { return kda::kChunk; }
int32_t kda_checkpoint_tokens(void) { return kda::kCkTokens; }

kda_status kda_ctx_workspace_bytes(int64_t B, int64_t T, int64_t Hqk, int64_t Hv,
                                   const int64_t* cu_seqlens_host, int64_t num_seqs, size_t* bytes) {
  return kda::guarded([&]() -> kda_status {
    if (!bytes) return fail(KDA_ERR_INVALID_ARGUMENT, "bytes is NULL");
    Shape s;
    kda_status st = make_shape(B, T, Hqk, Hv, cu_seqlens_host, num_seqs, &s);
    if (st != KDA_OK) return st;
    *bytes = make_layout(s).total;
    return KDA_OK;
  });
}

kda_status kda_fwd(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                   const kda_bf16* beta, const float* A_log, const float* dt_bias, const float* h0,
                   const int64_t* cu_seqlens_dev, const int64_t* cu_seqlens_host, int64_t num_seqs,
                   int64_t B, int64_t T, int64_t Hqk, int64_t Hv, int64_t head_dim, float scale,
                   float lower_bound, kda_bf16* o, float* h_T, void* ctx_workspace, size_t ctx_bytes,
                   kda_ctx** ctx, struct CUstream_st* stream_) {
  return kda::guarded([&]() -> kda_status {
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (!ctx) return fail(KDA_ERR_INVALID_ARGUMENT, "ctx is NULL");
    if (!q || !k || !v || !g || !beta || !A_log || !dt_bias || !h0 || !o || !h_T || !ctx_workspace)
      return fail(KDA_ERR_INVALID_ARGUMENT, "a required tensor pointer is NULL");
    if ((cu_seqlens_dev == nullptr) != (cu_seqlens_host == nullptr))
      return fail(KDA_ERR_INVALID_ARGUMENT, "packed input needs both cu_seqlens and its host mirror");
    if (head_dim != kda::kDim)
      return fail(KDA_ERR_UNSUPPORTED, "head dimension must be 128 (got %lld)", (long long)head_dim);
    const float s_req = (float)(1.0 / std::sqrt(128.0));
    if (std::isnan(scale)) scale = s_req;
    if (std::fabs(scale - s_req) > 1e-6f * s_req)
      return fail(KDA_ERR_UNSUPPORTED, "scale must be 1/sqrt(128) (got %g)", (double)scale);
    if (lower_bound != -5.0f)
      return fail(KDA_ERR_UNSUPPORTED, "lower_bound must be -5 (got %g)", (double)lower_bound);
    Shape s;
    kda_status st = make_shape(B, T, Hqk, Hv, cu_seqlens_host, num_seqs, &s);
    if (st != KDA_OK) return st;
    const Layout L = make_layout(s);
    if (ctx_bytes < L.total)
      return fail(KDA_ERR_WORKSPACE_TOO_SMALL, "context workspace needs %zu bytes, got %zu", L.total, ctx_bytes);
    if (((uintptr_t)ctx_workspace % kAlign) != 0)
      return fail(KDA_ERR_INVALID_ARGUMENT, "context workspace must be 256-byte aligned");
    const void* vec_ptrs[] = {q, k, v, g, o, h_T, h0};
    for (const void* p : vec_ptrs)
      if (!aligned16(p)) return fail(KDA_ERR_INVALID_ARGUMENT, "token and state tensors must be 16-byte aligned");
    const size_t tok_qk = sizeof(kda_bf16) * (size_t)s.Ttot * Hqk * kda::kDim;
    const size_t tok_v = sizeof(kda_bf16) * (size_t)s.Ttot * Hv * kda::kDim;
    const size_t state = sizeof(float) * (size_t)s.N * Hv * kda::kDim * kda::kDim;
    std::vector<Range> inputs = {
        {q, tok_qk, "q"}, {k, tok_qk, "k"}, {v, tok_v, "v"}, {g, tok_v, "g"},
        {beta, sizeof(kda_bf16) * (size_t)s.Ttot * Hv, "beta"}, {A_log, sizeof(float) * (size_t)Hv, "A_log"},
        {dt_bias, sizeof(float) * (size_t)Hv * kda::kDim, "dt_bias"}, {h0, state, "initial_state"},
        {cu_seqlens_dev, cu_seqlens_dev ? sizeof(int64_t) * (size_t)(s.N + 1) : 0, "cu_seqlens"}};
    std::vector<Range> outputs = {{o, tok_v, "o"}, {h_T, state, "final_state"},
                                  {ctx_workspace, ctx_bytes, "context workspace"}};
    if ((st = check_aliasing(inputs, outputs)) != KDA_OK) return st;
    int dev = -1;
    if ((st = check_device(&dev)) != KDA_OK) return st;

    kda_ctx* c = *ctx;
    bool fresh = false;
    if (c == nullptr) {
      c = new (std::nothrow) kda_ctx();
      if (!c) return fail(KDA_ERR_INVALID_ARGUMENT, "out of host memory");
      fresh = true;
      c->shape = s;
      c->layout = L;
      c->device = dev;
      c->stream = stream;
      c->ws = static_cast<char*>(ctx_workspace);
      c->ws_bytes = ctx_bytes;
      // longest sequence first; ties by (sequence, head)
      c->order.resize(s.units);
      for (int64_t u = 0; u < s.units; ++u) c->order[u] = (int32_t)u;
      std::stable_sort(c->order.begin(), c->order.end(), [&](int32_t a, int32_t b) {
        const int64_t la = s.cu[a / Hv + 1] - s.cu[a / Hv], lb = s.cu[b / Hv + 1] - s.cu[b / Hv];
        return la > lb;
      });
      c->seq.resize(s.N);
      int64_t ck = 0, chn = 0;
      for (int64_t i = 0; i < s.N; ++i) {
        c->seq[i].t0 = s.cu[i];
        c->seq[i].len = s.cu[i + 1] - s.cu[i];
        c->seq[i].ck_base = ck;
        c->seq[i].ch_base = chn;
        ck += kda::checkpoints_of(c->seq[i].len);
        chn += kda::subchunks_of(c->seq[i].len);
      }
    } else {
      if (!(c->shape == s)) return fail(KDA_ERR_CONTEXT, "context was created for a different shape");
      if (c->device != dev) return fail(KDA_ERR_CONTEXT, "context belongs to device %d", c->device);
      if (c->stream != stream) return fail(KDA_ERR_CONTEXT, "context must be reused on the stream that created it");
      if (c->ws != ctx_workspace || c->ws_bytes != ctx_bytes)
        return fail(KDA_ERR_CONTEXT, "context must be reused with the workspace it was created with");
    }
    cudaError_t e;
    if (fresh) {
      if ((e = cudaMemcpyAsync(c->ws + L.order, c->order.data(), sizeof(int32_t) * s.units,
                               cudaMemcpyHostToDevice, stream)) != cudaSuccess ||
          (e = cudaMemcpyAsync(c->ws + L.seq, c->seq.data(), sizeof(SeqInfo) * s.N,
                               cudaMemcpyHostToDevice, stream)) != cudaSuccess ||
          (e = cudaMemsetAsync(c->ws + L.status, 0, 16, stream)) != cudaSuccess) {
        delete c;
        return cuda_fail(e, "plan upload");
      }
    }
    kda::Problem& P = c->prob;
    P.q = reinterpret_cast<const __nv_bfloat16*>(q);
    P.k = reinterpret_cast<const __nv_bfloat16*>(k);
    P.v = reinterpret_cast<const __nv_bfloat16*>(v);
    P.g = reinterpret_cast<const __nv_bfloat16*>(g);
    P.beta = reinterpret_cast<const __nv_bfloat16*>(beta);
    P.A_log = A_log;
    P.dt_bias = dt_bias;
    P.h0 = h0;
    P.order = reinterpret_cast<const int32_t*>(c->ws + L.order);
    P.seq = reinterpret_cast<const SeqInfo*>(c->ws + L.seq);
    P.ckpt = reinterpret_cast<float*>(c->ws + L.ckpt);
    P.status = reinterpret_cast<int32_t*>(c->ws + L.status);
    P.utape = reinterpret_cast<float*>(c->ws + L.utape);
    P.abtape = reinterpret_cast<float*>(c->ws + L.abtape);
    P.N = s.N;
    P.Hqk = Hqk;
    P.Hv = Hv;
    P.r = (int32_t)(Hv / Hqk);
    P.scale = scale;
    P.lb = lower_bound;
    kda::FwdOut out{reinterpret_cast<__nv_bfloat16*>(o), h_T};
    c->forward_done = false;
    if ((e = kda::launch_forward(P, out, s.units, stream)) != cudaSuccess) {
      if (fresh) delete c;
      return cuda_fail(e, "forward launch");
    }
    c->inputs = inputs;
    c->forward_done = true;
    *ctx = c;
    return KDA_OK;
  });
}

kda_status kda_bwd(kda_ctx* c, const kda_bf16* d_o, const float* d_hT, kda_bf16* dq, kda_bf16* dk,
                   kda_bf16* dv, kda_bf16* dg, kda_bf16* dbeta, float* dA_log, float* ddt_bias,
                   float* dh0, struct CUstream_st* stream_) {
  return kda::guarded([&]() -> kda_status {
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (!c) return fail(KDA_ERR_INVALID_ARGUMENT, "ctx is NULL");
    if (!c->forward_done) return fail(KDA_ERR_CONTEXT, "context holds no completed forward");
    if (!d_o || !d_hT || !dq || !dk || !dv || !dg || !dbeta || !dA_log || !ddt_bias || !dh0)
      return fail(KDA_ERR_INVALID_ARGUMENT, "a required tensor pointer is NULL");
    if (stream != c->stream) return fail(KDA_ERR_CONTEXT, "backward must run on the context's stream");
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != c->device)
      return fail(KDA_ERR_CONTEXT, "backward must run on the context's device (%d)", c->device);
    const void* vec_ptrs[] = {d_o, d_hT, dq, dk, dv, dg, dh0};
    for (const void* p : vec_ptrs)
      if (!aligned16(p)) return fail(KDA_ERR_INVALID_ARGUMENT, "token and state tensors must be 16-byte aligned");
    const Shape& s = c->shape;
    const size_t tok_qk = sizeof(kda_bf16) * (size_t)s.Ttot * s.Hqk * kda::kDim;
    const size_t tok_v = sizeof(kda_bf16) * (size_t)s.Ttot * s.Hv * kda::kDim;
    const size_t state = sizeof(float) * (size_t)s.N * s.Hv * kda::kDim * kda::kDim;
    std::vector<Range> inputs = c->inputs;
    inputs.push_back({d_o, tok_v, "do"});
    inputs.push_back({d_hT, state, "dfinal_state"});
    inputs.push_back({c->ws, c->ws_bytes, "context workspace"});
    std::vector<Range> outputs = {
        {dq, tok_qk, "dq"}, {dk, tok_qk, "dk"}, {dv, tok_v, "dv"}, {dg, tok_v, "dg"},
        {dbeta, sizeof(kda_bf16) * (size_t)s.Ttot * s.Hv, "dbeta"},
        {dA_log, sizeof(float) * (size_t)s.Hv, "dA_log"},
        {ddt_bias, sizeof(float) * (size_t)s.Hv * kda::kDim, "ddt_bias"},
        {dh0, state, "dinitial_state"}};
    kda_status st = check_aliasing(inputs, outputs);
    if (st != KDA_OK) return st;
    kda::BwdArgs a;
    a.d_o = reinterpret_cast<const __nv_bfloat16*>(d_o);
    a.d_hT = d_hT;
    a.dq = reinterpret_cast<__nv_bfloat16*>(dq);
    a.dk = reinterpret_cast<__nv_bfloat16*>(dk);
    a.dv = reinterpret_cast<__nv_bfloat16*>(dv);
    a.dg = reinterpret_cast<__nv_bfloat16*>(dg);
    a.dbeta = reinterpret_cast<__nv_bfloat16*>(dbeta);
    a.dh0 = dh0;
    a.dqk_part = reinterpret_cast<float*>(c->ws + c->layout.dqk);
    a.par_part = reinterpret_cast<float*>(c->ws + c->layout.par);
    cudaError_t e = kda::launch_backward(c->prob, a, s.units, s.Ttot, dA_log, ddt_bias, stream);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return KDA_OK;
  });
}

kda_status kda_ctx_status(kda_ctx* c) {
  if (!c) return fail(KDA_ERR_INVALID_ARGUMENT, "ctx is NULL");
  cudaError_t e = cudaStreamSynchronize(c->stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int32_t word = 0;
  e = cudaMemcpy(&word, c->ws + c->layout.status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status readback");
  if (word != 0) return fail(KDA_ERR_DEVICE_TIMEOUT, "device wait gave up (code %d)", word);
  return KDA_OK;
}

void kda_ctx_destroy(kda_ctx* c) { delete c; }

namespace {

// kda_bwd_standalone's workspace: the context workspace of kda_fwd, then the
// forward's output o and final state, which the backward does not return.
struct StandaloneLayout {
  size_t ctx_bytes = 0, o = 0, h_T = 0, total = 0;
};

kda_status standalone_layout(int64_t B, int64_t T, int64_t Hqk, int64_t Hv, const int64_t* cu_host,
                             int64_t num_seqs, StandaloneLayout* L) {
  Shape s;
  kda_status st = make_shape(B, T, Hqk, Hv, cu_host, num_seqs, &s);
  if (st != KDA_OK) return st;
  L->ctx_bytes = make_layout(s).total;
  L->o = L->ctx_bytes;
  L->h_T = kda::ctx_align_up(L->o + sizeof(kda_bf16) * (size_t)s.Ttot * Hv * kda::kDim);
  L->total = kda::ctx_align_up(L->h_T + sizeof(float) * (size_t)s.N * Hv * kda::kDim * kda::kDim);
  return KDA_OK;
}

}  // namespace

kda_status kda_bwd_standalone_workspace_bytes(int64_t B, int64_t T, int64_t Hqk, int64_t Hv,
                                              const int64_t* cu_seqlens_host, int64_t num_seqs,
                                              size_t* bytes) {
  return kda::guarded([&]() -> kda_status {
    g_last_error.clear();
    if (!bytes) return fail(KDA_ERR_INVALID_ARGUMENT, "bytes is NULL");
    StandaloneLayout L;
    kda_status st = standalone_layout(B, T, Hqk, Hv, cu_seqlens_host, num_seqs, &L);
    if (st != KDA_OK) return st;
    *bytes = L.total;
    return KDA_OK;
  });
}

kda_status kda_bwd_standalone(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                              const kda_bf16* beta, const float* A_log, const float* dt_bias, const float* h0,
                              const int64_t* cu_seqlens_dev, const int64_t* cu_seqlens_host, int64_t num_seqs,
                              int64_t B, int64_t T, int64_t Hqk, int64_t Hv, int64_t head_dim, float scale,
                              float lower_bound, const kda_bf16* d_o, const float* d_hT, kda_bf16* dq,
                              kda_bf16* dk, kda_bf16* dv, kda_bf16* dg, kda_bf16* dbeta, float* dA_log,
                              float* ddt_bias, float* dh0, void* workspace, size_t workspace_bytes,
                              kda_ctx** ws_ctx, struct CUstream_st* stream) {
  return kda::guarded([&]() -> kda_status {
    g_last_error.clear();
    if (!ws_ctx) return fail(KDA_ERR_INVALID_ARGUMENT, "ws_ctx is NULL");
    if (!workspace) return fail(KDA_ERR_INVALID_ARGUMENT, "workspace is NULL");
    if (!d_o || !d_hT || !dq || !dk || !dv || !dg || !dbeta || !dA_log || !ddt_bias || !dh0)
      return fail(KDA_ERR_INVALID_ARGUMENT, "a required tensor pointer is NULL");
    if (head_dim != kda::kDim)
      return fail(KDA_ERR_UNSUPPORTED, "head dimension must be 128 (got %lld)", (long long)head_dim);
    StandaloneLayout L;
    kda_status st = standalone_layout(B, T, Hqk, Hv, cu_seqlens_host, num_seqs, &L);
    if (st != KDA_OK) return st;
    if (workspace_bytes < L.total)
      return fail(KDA_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes, got %zu", L.total, workspace_bytes);
    if (((uintptr_t)workspace % kAlign) != 0)
      return fail(KDA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
    // The forward writes the workspace before the backward reads the adjoints, and the
    // backward writes the gradients while it reads the workspace: none may overlap it.
    const int64_t N = cu_seqlens_host ? num_seqs : B;
    const size_t Ttot = (size_t)B * T;
    const size_t tok_qk = sizeof(kda_bf16) * Ttot * Hqk * kda::kDim, tok_v = sizeof(kda_bf16) * Ttot * Hv * kda::kDim;
    const size_t state = sizeof(float) * (size_t)N * Hv * kda::kDim * kda::kDim;
    const Range ws{workspace, workspace_bytes, "workspace"};
    const Range others[] = {{d_o, tok_v, "do"}, {d_hT, state, "dfinal_state"}, {dq, tok_qk, "dq"},
                            {dk, tok_qk, "dk"}, {dv, tok_v, "dv"}, {dg, tok_v, "dg"},
                            {dbeta, sizeof(kda_bf16) * Ttot * Hv, "dbeta"}, {dA_log, sizeof(float) * Hv, "dA_log"},
                            {ddt_bias, sizeof(float) * Hv * kda::kDim, "ddt_bias"}, {dh0, state, "dinitial_state"}};
    for (const Range& r : others)
      if (overlaps(ws, r)) return fail(KDA_ERR_ALIASING, "%s overlaps the workspace", r.name);
    char* base = static_cast<char*>(workspace);
    st = kda_fwd(q, k, v, g, beta, A_log, dt_bias, h0, cu_seqlens_dev, cu_seqlens_host, num_seqs, B, T, Hqk, Hv,
                 head_dim, scale, lower_bound, reinterpret_cast<kda_bf16*>(base + L.o),
                 reinterpret_cast<float*>(base + L.h_T), base, L.ctx_bytes, ws_ctx, stream);
    if (st != KDA_OK) return st;
    return kda_bwd(*ws_ctx, d_o, d_hT, dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dh0, stream);
  });
}

}  // extern "C"
