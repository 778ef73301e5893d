// kda_decode.cu -- one decode step (T = 1) of the recurrent KDA recurrence
// (flashinfer.kda.recurrent_kda, description and parameters: "T=1 selects
// decode"; the state is updated in place, optionally through state-cache slot
// indices).
//
// For every (sequence n, value head h) the 128x128 state S (value-first, the
// slot state_indices[n] of the state pool) is read once, decayed per key
// column, delta-corrected and written back, and the output token produced:
//   S' = S diag(d),  u = v - S' k^,  S <- S' + beta u k^^T,  o = s S q^
// with q^, k^ L2-normalised, d = exp(lb sigmoid(exp(A_log) (g + dt_bias)))
// (or d = exp(g) with the gate precomputed in log space) and beta = sigmoid(
// logit) (or beta as given, already sigmoided). Since S q^ = S' q^ + beta u (k^ . q^), each state
// row needs two dot products with the decayed row and one rank-1 update.
//
// The step moves the state through HBM once in each direction and does 8 flops
// per state element, so it is bandwidth-bound. One CTA of 256 threads per unit
// starts the state's loads first: a BF16 state (32 KiB) is staged into shared
// memory with cp.async, an FP32 state (64 KiB) is loaded into registers, eight
// rows' slices per thread; meanwhile it computes the token's vectors. Then a
// half-warp updates one state row at a time (8 keys per lane) and writes it
// straight back.
#include "../../include/kda.h"
#include "kda_common.cuh"
#include "kda_host.h"
#include "tc.cuh"

#include <cmath>
#include <unordered_set>

namespace kda {
namespace {

constexpr int kDecThreads = 256;
constexpr int kRowsPerPass = kDecThreads / 16;     // 16 rows: two per warp
constexpr int kPasses = kDim / kRowsPerPass;       // 8

struct DecodeArgs {
  const __nv_bfloat16* q;     // [N, Hqk, 128]
  const __nv_bfloat16* k;     // [N, Hqk, 128]
  const __nv_bfloat16* v;     // [N, Hv, 128]
  const __nv_bfloat16* g;     // [N, Hv, 128]
  const __nv_bfloat16* beta;  // [N, Hv] (logits when beta_logit)
  const float* A_log;         // [Hv]
  const float* dt_bias;       // [Hv, 128]
  void* state;                // [num_slots, Hv, 128, 128], BF16 or FP32
  const int32_t* idx;         // [N] slot per sequence, or null (slot n)
  int64_t num_slots;          // slots in the pool
  __nv_bfloat16* o;           // [N, Hv, 128]
  int64_t Hqk, Hv, r;
  float scale, lb;
  int gate_in_kernel;         // 1: d = exp(lb sigmoid(exp(A_log)(g + dt_bias))); 0: d = exp(g)
  int beta_logit;             // 1: beta = sigmoid(input); 0: the input is beta
};

// 8 consecutive state elements of one row <-> FP32 registers
template <typename T>
struct Row8;
template <>
struct Row8<__nv_bfloat16> {
  using Raw = uint4;
  static __device__ __forceinline__ Raw load(const void* p) { return *reinterpret_cast<const uint4*>(p); }
  static __device__ __forceinline__ void unpack(const Raw& r, float* x) { unpack_bf16x8(r, x); }
  static __device__ __forceinline__ void store(void* p, const float* x) {
    store_bf16x8(reinterpret_cast<__nv_bfloat16*>(p), x);
  }
};
template <>
struct Row8<float> {
  struct Raw {
    float4 a, b;
  };
  static __device__ __forceinline__ Raw load(const void* p) {
    const float4* f = reinterpret_cast<const float4*>(p);
    return Raw{f[0], f[1]};
  }
  static __device__ __forceinline__ void unpack(const Raw& r, float* x) {
    x[0] = r.a.x; x[1] = r.a.y; x[2] = r.a.z; x[3] = r.a.w;
    x[4] = r.b.x; x[5] = r.b.y; x[6] = r.b.z; x[7] = r.b.w;
  }
  static __device__ __forceinline__ void store(void* p, const float* x) {
    float4* f = reinterpret_cast<float4*>(p);
    f[0] = make_float4(x[0], x[1], x[2], x[3]);
    f[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
};

// A BF16 state is staged through shared memory (bytes in flight bounded by
// shared memory, four CTAs per SM); an FP32 state, twice the bytes per row, is
// loaded straight into registers, all eight rows of a thread at once.
template <typename StateT>
constexpr bool kStaged = sizeof(StateT) == 2;
template <typename StateT>
constexpr int kDecMinBlocks = kStaged<StateT> ? 4 : 2;

template <typename StateT>
__global__ void __launch_bounds__(kDecThreads, kDecMinBlocks<StateT>) kda_decode_kernel(const DecodeArgs a) {
  const int64_t unit = blockIdx.x;
  const int64_t n = unit / a.Hv, h = unit % a.Hv, qh = h / a.r;
  const int64_t slot = a.idx ? a.idx[n] : n;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (slot < 0 || slot >= a.num_slots) {
    // a device index outside the pool (it no longer matches the host mirror the call was checked
    // against, e.g. in a replayed graph): the state is not touched and this row of o reads NaN
    if (tid < kDim / 8) {
      float nan8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) nan8[e] = __int_as_float(0x7fc00000);
      store_bf16x8(a.o + (n * a.Hv + h) * kDim + 8 * tid, nan8);
    }
    return;
  }
  const int hl = lane & 15, half = lane >> 4;  // keys 8 hl .. 8 hl + 7 of row 2 warp + half (+16 per pass)
  StateT* S = reinterpret_cast<StateT*>(a.state) + ((slot * a.Hv + h) * kDim) * kDim;
  extern __shared__ __align__(16) unsigned char st_smem[];
  StateT* Ss = reinterpret_cast<StateT*>(st_smem);

  // the state first: it is the bandwidth
  typename Row8<StateT>::Raw raw[kStaged<StateT> ? 1 : kPasses];
  if constexpr (kStaged<StateT>) {
    constexpr int kPieces = kDim * kDim * (int)sizeof(StateT) / 16;
#pragma unroll 4
    for (int i = tid; i < kPieces; i += kDecThreads)
      tc::cp_async16(st_smem + 16 * i, reinterpret_cast<const unsigned char*>(S) + 16 * i, 16u);
    tc::cp_async_commit();
  } else {
#pragma unroll
    for (int p = 0; p < kPasses; ++p)
      raw[p] = Row8<StateT>::load(S + (kRowsPerPass * p + 2 * warp + half) * kDim + 8 * hl);
  }

  // the token's vectors (every half-warp holds all 128 keys)
  float qv[8], kv[8], gv[8];
  load_bf16x8(a.q + (n * a.Hqk + qh) * kDim + 8 * hl, qv);
  load_bf16x8(a.k + (n * a.Hqk + qh) * kDim + 8 * hl, kv);
  load_bf16x8(a.g + (n * a.Hv + h) * kDim + 8 * hl, gv);
  float sq = 0.f, sk = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) { sq += qv[e] * qv[e]; sk += kv[e] * kv[e]; }
  sq = row16_sum(sq);
  sk = row16_sum(sk);
  const float rq = inv_norm_of(sq), rk = inv_norm_of(sk);
  const float ea = a.gate_in_kernel ? expf(a.A_log[h]) : 0.f;
  float d[8], kq = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    qv[e] *= rq;
    kv[e] *= rk;
    kq += kv[e] * qv[e];
    d[e] = a.gate_in_kernel ? expf(log_decay_of(a.lb, ea * (gv[e] + a.dt_bias[h * kDim + 8 * hl + e])))
                            : expf(gv[e]);
  }
  kq = row16_sum(kq);
  const float braw = __bfloat162float(a.beta[n * a.Hv + h]);
  const float bt = a.beta_logit ? sigmoid_of(braw) : braw;
  const __nv_bfloat16* vrow = a.v + (n * a.Hv + h) * kDim;
  __nv_bfloat16* orow = a.o + (n * a.Hv + h) * kDim;
  if constexpr (kStaged<StateT>) {
    tc::cp_async_wait_all();
    __syncthreads();
  }

#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int row = kRowsPerPass * p + 2 * warp + half;
    float s[8];
    if constexpr (kStaged<StateT>) Row8<StateT>::unpack(Row8<StateT>::load(Ss + row * kDim + 8 * hl), s);
    else Row8<StateT>::unpack(raw[p], s);
    float pk = 0.f, pq = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      s[e] *= d[e];
      pk = fmaf(s[e], kv[e], pk);
      pq = fmaf(s[e], qv[e], pq);
    }
    pk = row16_sum(pk);
    pq = row16_sum(pq);
    const float u = __bfloat162float(vrow[row]) - pk;
    const float bu = bt * u;
#pragma unroll
    for (int e = 0; e < 8; ++e) s[e] = fmaf(bu, kv[e], s[e]);
    Row8<StateT>::store(S + row * kDim + 8 * hl, s);
    if (hl == 0) orow[row] = __float2bfloat16_rn(a.scale * (pq + bu * kq));
  }
}

}  // namespace
}  // namespace kda

namespace {

kda_status dfail(kda_status st, const char* msg) {
  kda::set_last_error(msg);
  return st;
}

struct Span {
  const void* p;
  size_t bytes;
};

bool overlap(const Span& a, const Span& b) {
  const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
  return a.bytes && b.bytes && a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

}  // namespace

extern "C" kda_status kda_decode(const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                                 const kda_bf16* beta, const float* A_log, const float* dt_bias, void* state,
                                 int32_t state_dtype, const int32_t* state_indices,
                                 const int32_t* state_indices_host, int64_t num_slots, int64_t N, int64_t Hqk,
                                 int64_t Hv, int64_t head_dim, float scale, float lower_bound,
                                 int32_t use_gate_in_kernel, int32_t beta_is_logit, kda_bf16* o,
                                 struct CUstream_st* stream) {
  return kda::guarded([&]() -> kda_status {
    if (N < 1 || Hqk < 1 || Hv < 1) return dfail(KDA_ERR_INVALID_ARGUMENT, "decode: N, Hqk and Hv must be positive");
    if (Hv % Hqk != 0) return dfail(KDA_ERR_INVALID_ARGUMENT, "decode: Hv must be a multiple of Hqk");
    if (kda::size_limit_violation(N, 1, Hv, 0) || N > INT32_MAX / Hv)
      return dfail(KDA_ERR_UNSUPPORTED, "decode: too many (sequence, head) units");
    if (num_slots > (int64_t(1) << 31)) return dfail(KDA_ERR_UNSUPPORTED, "decode: more than 2^31 pool slots");
    if (head_dim != kda::kDim) return dfail(KDA_ERR_UNSUPPORTED, "decode: head_dim must be 128");
    const float s_def = 1.0f / std::sqrt((float)kda::kDim);
    if (!std::isnan(scale) && scale != s_def)
      return dfail(KDA_ERR_UNSUPPORTED, "decode: scale must be 1/sqrt(128) (NaN selects it)");
    if ((use_gate_in_kernel != 0 && use_gate_in_kernel != 1) || (beta_is_logit != 0 && beta_is_logit != 1))
      return dfail(KDA_ERR_INVALID_ARGUMENT, "decode: use_gate_in_kernel and beta_is_logit must be 0 or 1");
    if (use_gate_in_kernel && lower_bound != -5.0f)
      return dfail(KDA_ERR_UNSUPPORTED, "decode: lower_bound must be -5 with the gate computed in the kernel");
    if (state_dtype != KDA_STATE_BF16 && state_dtype != KDA_STATE_FP32)
      return dfail(KDA_ERR_INVALID_ARGUMENT, "decode: state_dtype must be KDA_STATE_BF16 or KDA_STATE_FP32");
    if (!q || !k || !v || !g || !beta || !state || !o || (use_gate_in_kernel && (!A_log || !dt_bias)))
      return dfail(KDA_ERR_INVALID_ARGUMENT, "decode: null tensor pointer");
    if ((state_indices == nullptr) != (state_indices_host == nullptr))
      return dfail(KDA_ERR_INVALID_ARGUMENT, "decode: state_indices needs its host mirror (and the reverse)");
    if (state_indices_host) {
      std::unordered_set<int32_t> seen;
      for (int64_t i = 0; i < N; ++i) {
        const int32_t s = state_indices_host[i];
        if (s < 0 || s >= num_slots) return dfail(KDA_ERR_INVALID_ARGUMENT, "decode: state index out of range");
        if (!seen.insert(s).second)
          return dfail(KDA_ERR_INVALID_ARGUMENT, "decode: two sequences share a state slot");
      }
    } else if (num_slots < N) {
      return dfail(KDA_ERR_INVALID_ARGUMENT, "decode: without state_indices the pool needs a slot per sequence");
    }
    const void* ptrs[] = {q, k, v, g, state, o};
    for (const void* p : ptrs)
      if ((uintptr_t)p & 15u) return dfail(KDA_ERR_INVALID_ARGUMENT, "decode: token and state tensors must be 16-byte aligned");
    const size_t esz = state_dtype == KDA_STATE_BF16 ? 2 : 4;
    const Span st{state, esz * (size_t)num_slots * Hv * kda::kDim * kda::kDim};
    const Span out{o, 2 * (size_t)N * Hv * kda::kDim};
    const Span ins[] = {{q, 2 * (size_t)N * Hqk * kda::kDim}, {k, 2 * (size_t)N * Hqk * kda::kDim},
                        {v, 2 * (size_t)N * Hv * kda::kDim},  {g, 2 * (size_t)N * Hv * kda::kDim},
                        {beta, 2 * (size_t)N * Hv},
                        {A_log, use_gate_in_kernel ? 4 * (size_t)Hv : 0},
                        {dt_bias, use_gate_in_kernel ? 4 * (size_t)Hv * kda::kDim : 0}};
    for (const Span& in : ins)
      if (overlap(in, st) || overlap(in, out)) return dfail(KDA_ERR_ALIASING, "decode: an input overlaps the state or o");
    if (overlap(st, out)) return dfail(KDA_ERR_ALIASING, "decode: o overlaps the state");
    if (state_indices && overlap(Span{state_indices, 4 * (size_t)N}, st))
      return dfail(KDA_ERR_ALIASING, "decode: state_indices overlaps the state");

    int dev = -1, major = 0, minor = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return dfail(KDA_ERR_CUDA, cudaGetErrorString(e));
    if (major != 10 || minor != 3) return dfail(KDA_ERR_UNSUPPORTED, "decode: kernels are built for sm_103a");

    kda::DecodeArgs a{};
    a.q = reinterpret_cast<const __nv_bfloat16*>(q);
    a.k = reinterpret_cast<const __nv_bfloat16*>(k);
    a.v = reinterpret_cast<const __nv_bfloat16*>(v);
    a.g = reinterpret_cast<const __nv_bfloat16*>(g);
    a.beta = reinterpret_cast<const __nv_bfloat16*>(beta);
    a.A_log = A_log;
    a.dt_bias = dt_bias;
    a.state = state;
    a.idx = state_indices;
    a.num_slots = num_slots;
    a.o = reinterpret_cast<__nv_bfloat16*>(o);
    a.Hqk = Hqk;
    a.Hv = Hv;
    a.r = Hv / Hqk;
    a.scale = s_def;
    a.lb = lower_bound;
    a.gate_in_kernel = use_gate_in_kernel;
    a.beta_logit = beta_is_logit;
    const unsigned grid = (unsigned)(N * Hv);
    const size_t smem = state_dtype == KDA_STATE_BF16 ? esz * kda::kDim * kda::kDim : 0;
    if (state_dtype == KDA_STATE_BF16) {
      e = cudaFuncSetAttribute(kda::kda_decode_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) kda::kda_decode_kernel<__nv_bfloat16><<<grid, kda::kDecThreads, smem, stream>>>(a);
    } else {
      e = cudaFuncSetAttribute(kda::kda_decode_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) kda::kda_decode_kernel<float><<<grid, kda::kDecThreads, smem, stream>>>(a);
    }
    if (e != cudaSuccess) return dfail(KDA_ERR_CUDA, cudaGetErrorString(e));
    e = cudaGetLastError();
    if (e != cudaSuccess) return dfail(KDA_ERR_CUDA, cudaGetErrorString(e));
    return KDA_OK;
  });
}
