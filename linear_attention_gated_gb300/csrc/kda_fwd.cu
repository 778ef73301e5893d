// kda_fwd.cu -- chunked forward of the recurrent KDA training recurrence.
//
// One CTA owns one (sequence, value head) unit and walks its tokens in
// sub-chunks of kChunk = 16, keeping the 128x128 FP32 value-first state on
// chip. Within a sub-chunk starting from state S0, with Gam_i the cumulative
// log-decay of tokens 1..i (per key dim) and gamma_i = exp(Gam_i):
//   A_ij = k^_i . (k^_j * gamma_i / gamma_j)   (j < i)
//   B_ij = q^_i . (k^_j * gamma_i / gamma_j)   (j <= i)
//   T    = (I + diag(beta) A)^-1
//   Y    = V - (k^ * gamma) S0^T,   W = T diag(beta) Y      (rows: beta_i u_i)
//   O    = scale ((q^ * gamma) S0^T + B W)
//   S_C  = S0 diag(gamma_C) + W^T (k^ * gamma_C / gamma)
// which equals the token-by-token rule S' = S diag(d); u = v - S' k^;
// S = S' + beta u k^T; o = scale S q^ (flashinfer.kda_backward.recurrent_kda_backward,
// description: gate, norm and sigmoid contracts). The gate, L2 norm and sigmoid
// of each token are computed on chip (the fused prologue). The state at the
// start of every checkpoint interval is stored for the backward.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = kChunk * kLds;
constexpr int kSq = kChunk * (kChunk + 1);

struct FwdSmem {
  float Qt[kTile];   // q^ * gamma
  float Kt[kTile];   // k^ * gamma
  float Ki[kTile];   // k^ / gamma
  float Kb[kTile];   // k^ * gamma_C / gamma
  float Vs[kTile];   // v
  float Am[kSq];
  float Bm[kSq];
  float Tm[kSq];
  float bs[kChunk];  // beta = sigmoid(logit)
  float gC[kDim];    // gamma at the end of the sub-chunk
};

__global__ void __launch_bounds__(kThreads, 1)
kda_fwd_kernel(const Problem P, const FwdOut out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int unit = P.order[blockIdx.x];
  const int64_t n = unit / P.Hv;
  const int64_t h = unit % P.Hv;
  const int64_t qh = h / P.r;
  const SeqInfo si = P.seq[n];

  // state ownership: row sv, key quads kq(m) = m*8 + half*4, m = 0..15
  const int sv = tid >> 1;
  const int half = tid & 1;
  float S[64];
  {
    const float* src = P.h0 + ((n * P.Hv + h) * kDim + sv) * kDim;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float4 x = *reinterpret_cast<const float4*>(src + m * 8 + half * 4);
      S[4 * m] = x.x; S[4 * m + 1] = x.y; S[4 * m + 2] = x.z; S[4 * m + 3] = x.w;
    }
  }
  // tile mapping: token row ti, 8 columns from c8
  const int ti = tid >> 4;
  const int c8 = (tid & 15) * 8;
  const float ea = expf(P.A_log[h]);
  float dtb[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) dtb[e] = P.dt_bias[h * kDim + c8 + e];

  const int64_t nchunks = (si.len + kChunk - 1) / kChunk;
  const int ck_every = kCkTokens / kChunk;
  for (int64_t c = 0; c < nchunks; ++c) {
    const int64_t tc0 = si.t0 + c * kChunk;
    const int nt = (int)((si.len - c * kChunk) < kChunk ? (si.len - c * kChunk) : kChunk);
    if (c % ck_every == 0) {
      float* dst = P.ckpt + (((si.ck_base + c / ck_every) * P.Hv + h) * kDim + sv) * kDim;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        *reinterpret_cast<float4*>(dst + m * 8 + half * 4) =
            make_float4(S[4 * m], S[4 * m + 1], S[4 * m + 2], S[4 * m + 3]);
    }
    // ---- load the sub-chunk and run the prologue (L2 norm, gate, sigmoid beta)
    {
      float qv[8], kv[8], gv[8], vv[8];
      const bool valid = ti < nt;
      if (valid) {
        const int64_t t = tc0 + ti;
        load_bf16x8(P.q + (t * P.Hqk + qh) * kDim + c8, qv);
        load_bf16x8(P.k + (t * P.Hqk + qh) * kDim + c8, kv);
        load_bf16x8(P.g + (t * P.Hv + h) * kDim + c8, gv);
        load_bf16x8(P.v + (t * P.Hv + h) * kDim + c8, vv);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[e] = kv[e] = gv[e] = vv[e] = 0.f;
      }
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) { sq += qv[e] * qv[e]; sk += kv[e] * kv[e]; }
      sq = row16_sum(sq);
      sk = row16_sum(sk);
      const float rq = valid ? 1.0f / sqrtf(sq + kNormEps) : 0.f;
      const float rk = valid ? 1.0f / sqrtf(sk + kNormEps) : 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float z = ea * (gv[e] + dtb[e]);
        const float a = valid ? P.lb / (1.0f + expf(-z)) : 0.f;  // log decay
        sm.Qt[ti * kLds + c8 + e] = qv[e] * rq;
        sm.Kt[ti * kLds + c8 + e] = kv[e] * rk;
        sm.Ki[ti * kLds + c8 + e] = a;
        sm.Vs[ti * kLds + c8 + e] = vv[e];
      }
      if (tid < kChunk)
        sm.bs[tid] = (tid < nt) ? 1.0f / (1.0f + expf(-__bfloat162float(P.beta[(tc0 + tid) * P.Hv + h])))
                                : 0.f;
    }
    __syncthreads();
    // ---- cumulative decay along the sub-chunk (one key column per thread)
    if (tid < kDim) {
      const int kc = tid;
      float G = 0.f;
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        G += sm.Ki[i * kLds + kc];
        sm.Ki[i * kLds + kc] = G;  // keep Gam_i for the second pass
      }
      const float GC = G;
      sm.gC[kc] = expf(GC);
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        const float Gi = sm.Ki[i * kLds + kc];
        const float kh = sm.Kt[i * kLds + kc];
        const float gam = expf(Gi);
        sm.Qt[i * kLds + kc] *= gam;
        sm.Kt[i * kLds + kc] = kh * gam;
        sm.Ki[i * kLds + kc] = kh * expf(-Gi);
        sm.Kb[i * kLds + kc] = kh * expf(GC - Gi);
      }
    }
    __syncthreads();
    // ---- A (strictly lower) and B (lower with diagonal)
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
      const int e = tid + rep * kThreads;
      const int mat = e >> 8, i = (e >> 4) & 15, j = e & 15;
      const float* X = mat ? sm.Qt : sm.Kt;
      float acc = 0.f;
      if (j < i || (mat && j == i)) {
#pragma unroll 8
        for (int kk = 0; kk < kDim; kk += 4)
          acc += dot4(*reinterpret_cast<const float4*>(X + i * kLds + kk),
                      *reinterpret_cast<const float4*>(sm.Ki + j * kLds + kk));
      }
      (mat ? sm.Bm : sm.Am)[i * (kChunk + 1) + j] = acc;
    }
    __syncthreads();
    // ---- T = (I + diag(beta) A)^-1 by forward substitution, one column per lane
    if (tid < kChunk) {
      const int j = tid;
      float tc[kChunk];
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < i; ++m)
          if (m >= j) acc += sm.Am[i * (kChunk + 1) + m] * tc[m];
        tc[i] = (i < j) ? 0.f : (i == j ? 1.f : -sm.bs[i] * acc);
        sm.Tm[i * (kChunk + 1) + j] = tc[i];
      }
    }
    __syncthreads();
    // ---- state products for row sv of the state
    float y[kChunk], oa[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) { y[i] = 0.f; oa[i] = 0.f; }
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const int kk = m * 8 + half * 4;
      const float4 s4 = make_float4(S[4 * m], S[4 * m + 1], S[4 * m + 2], S[4 * m + 3]);
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        y[i] += dot4(*reinterpret_cast<const float4*>(sm.Kt + i * kLds + kk), s4);
        oa[i] += dot4(*reinterpret_cast<const float4*>(sm.Qt + i * kLds + kk), s4);
      }
    }
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      y[i] += __shfl_xor_sync(0xffffffffu, y[i], 1);
      oa[i] += __shfl_xor_sync(0xffffffffu, oa[i], 1);
      y[i] = sm.bs[i] * (sm.Vs[i * kLds + sv] - y[i]);  // beta_i (v_i - S0 k~_i)
    }
    float w[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j <= i; ++j) acc += sm.Tm[i * (kChunk + 1) + j] * y[j];
      w[i] = acc;
    }
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      float acc = oa[i];
#pragma unroll
      for (int j = 0; j <= i; ++j) acc += sm.Bm[i * (kChunk + 1) + j] * w[j];
      if ((i & 1) == half && i < nt)
        out.o[((tc0 + i) * P.Hv + h) * kDim + sv] = __float2bfloat16_rn(P.scale * acc);
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const int kk = m * 8 + half * 4;
      const float4 g4 = *reinterpret_cast<const float4*>(sm.gC + kk);
      float s0 = S[4 * m] * g4.x, s1 = S[4 * m + 1] * g4.y, s2 = S[4 * m + 2] * g4.z,
            s3 = S[4 * m + 3] * g4.w;
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        const float4 kb = *reinterpret_cast<const float4*>(sm.Kb + i * kLds + kk);
        s0 += w[i] * kb.x; s1 += w[i] * kb.y; s2 += w[i] * kb.z; s3 += w[i] * kb.w;
      }
      S[4 * m] = s0; S[4 * m + 1] = s1; S[4 * m + 2] = s2; S[4 * m + 3] = s3;
    }
    __syncthreads();
  }
  float* dst = out.hT + ((n * P.Hv + h) * kDim + sv) * kDim;
#pragma unroll
  for (int m = 0; m < 16; ++m)
    *reinterpret_cast<float4*>(dst + m * 8 + half * 4) =
        make_float4(S[4 * m], S[4 * m + 1], S[4 * m + 2], S[4 * m + 3]);
}

}  // namespace

cudaError_t launch_forward(const Problem& P, const FwdOut& out, int64_t units, cudaStream_t s) {
  const size_t smem = sizeof(FwdSmem);
  cudaError_t e = cudaFuncSetAttribute(kda_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  kda_fwd_kernel<<<(unsigned)units, kThreads, smem, s>>>(P, out);
  return cudaGetLastError();
}

}  // namespace kda
