// kda_bwd.cu -- reverse-time chunked backward of the recurrent KDA recurrence.
//
// One CTA owns one (sequence, value head) unit. It walks the unit's sub-chunks
// from last to first, carrying the state adjoint G = dL/dS (value-first,
// 128x128 FP32, on chip).
// Per sub-chunk it reloads the chunk-start state S0 saved by the forward and
// recomputes the chunk's WY quantities (never the whole forward):
//   Y  = V - (k^ gamma) S0^T,     W = T diag(beta) Y,     U = Y - A W  (u_i)
//   dW = (k^ gamma_C/gamma) G^T + scale B^T dO,   E = T^T dW,   dV = diag(beta) E
//   dbeta_i = E_i . U_i  (before the sigmoid derivative)
//   dq^ = scale gamma * (dO S0 + tril(dO W^T) (k^/gamma))
//   dk^ = -gamma * (dV S0 + stril(dV W^T) (k^/gamma))                 (read key)
//       + (1/gamma) * (gamma_C * (W G) + triu(scale W dO^T) (q^ gamma)
//                      - striu(W dV^T) (k^ gamma))                     (write key)
//   G  <- G diag(gamma_C) + (scale dO)^T (q^ gamma) - dV^T (k^ gamma)
// The decay gradient uses the gauge identity of the per-key-dim decay: scaling
// the decay of token t in key dim j by e^eps equals scaling, for every later
// token, the query and the read key by e^eps and the written key by e^-eps, and
// the final state's column j by e^eps. Applied at the end of each sub-chunk,
// where scaling column j of the state S_C has the direct effect
// sum_v G[v,j] S_C[v,j], it gives for the tokens t of the sub-chunk
//   da_t = sum_{s >= t in chunk} (q^ dq^ + k^ (dk^_read - dk^_write))_s + rho,
//   rho  = gamma_C * sum_v (G * S0) + sum_i (k^ gamma_C/gamma)_i * (W G)_i,
// so no per-token elementwise state product is needed and no sum runs across
// sub-chunks (a running sum over the whole sequence drifts in FP32).
// The gate, sigmoid and L2-norm backward are applied in the epilogue
// (flashinfer.kda_backward.recurrent_kda_backward, description: gradients with
// respect to the raw gate and raw beta logits, Q/K normalised with eps 1e-6).
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = kChunk * kLds;
constexpr int kSq = kChunk * (kChunk + 1);
constexpr int kState = kDim * kLds;

struct BwdSmem {
  float S0[kState];  // chunk-start state; later reused for dq^, dk^, da tiles
  float G[kState];   // adjoint of the state at the end of the current sub-chunk
  float Qt[kTile];   // q^ gamma
  float Kt[kTile];   // k^ gamma
  float Ki[kTile];   // k^ / gamma
  float Kb[kTile];   // k^ gamma_C / gamma
  float Gm[kTile];   // gamma
  float Vs[kTile];   // v, then Y, then E*U
  float Ws[kTile];   // W
  float dO[kTile];   // do
  float DU[kTile];   // dW (k-part), then dV = beta E
  float Am[kSq];
  float Bm[kSq];
  float Tm[kSq];
  float M1[kSq];     // dO W^T
  float M2[kSq];     // dV W^T
  float bs[kChunk];
  float dba[kChunk]; // dbeta before the sigmoid derivative
  float gC[kDim];
  float rho[3][kDim]; // sum_v G*S0, and the two halves of sum_i Kb (W G)
};

__global__ void __launch_bounds__(kThreads, 1)
kda_bwd_kernel(const Problem P, const BwdArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int unit = P.order[blockIdx.x];
  const int64_t n = unit / P.Hv;
  const int64_t h = unit % P.Hv;
  const int64_t qh = h / P.r;
  const SeqInfo si = P.seq[n];
  const float s = P.scale;

  // G <- dfinal_state
  {
    const float* src = a.d_hT + (n * P.Hv + h) * kDim * kDim;
    for (int f = tid; f < kDim * kDim / 4; f += kThreads) {
      const int row = f >> 5, c4 = (f & 31) * 4;
      *reinterpret_cast<float4*>(sm.G + row * kLds + c4) =
          *reinterpret_cast<const float4*>(src + row * kDim + c4);
    }
  }
  const int ti = tid >> 4;
  const int c8 = (tid & 15) * 8;
  const float ea = expf(P.A_log[h]);
  float dtb[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) dtb[e] = P.dt_bias[h * kDim + c8 + e];
  float ddt_acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) ddt_acc[e] = 0.f;
  float dA_acc = 0.f;

  const int64_t nchunks = (si.len + kChunk - 1) / kChunk;
  const int ck_every = kCkTokens / kChunk;
  for (int64_t c = nchunks - 1; c >= 0; --c) {
    const int64_t tc0 = si.t0 + c * kChunk;
    const int nt = (int)((si.len - c * kChunk) < kChunk ? (si.len - c * kChunk) : kChunk);
    // ---- P0: chunk-start state, token tiles and prologue
    {
      const float* src = P.ckpt + ((si.ck_base + c / ck_every) * P.Hv + h) * kDim * kDim;
      for (int f = tid; f < kDim * kDim / 4; f += kThreads) {
        const int row = f >> 5, c4 = (f & 31) * 4;
        *reinterpret_cast<float4*>(sm.S0 + row * kLds + c4) =
            *reinterpret_cast<const float4*>(src + row * kDim + c4);
      }
    }
    float qhat[8], khat[8], zz[8], rq, rk;
    {
      float qv[8], kv[8], gv[8], vv[8], dv8[8];
      const bool valid = ti < nt;
      const int64_t t = tc0 + ti;
      if (valid) {
        load_bf16x8(P.q + (t * P.Hqk + qh) * kDim + c8, qv);
        load_bf16x8(P.k + (t * P.Hqk + qh) * kDim + c8, kv);
        load_bf16x8(P.g + (t * P.Hv + h) * kDim + c8, gv);
        load_bf16x8(P.v + (t * P.Hv + h) * kDim + c8, vv);
        load_bf16x8(a.d_o + (t * P.Hv + h) * kDim + c8, dv8);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[e] = kv[e] = gv[e] = vv[e] = dv8[e] = 0.f;
      }
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) { sq += qv[e] * qv[e]; sk += kv[e] * kv[e]; }
      sq = row16_sum(sq);
      sk = row16_sum(sk);
      rq = valid ? 1.0f / sqrtf(sq + kNormEps) : 0.f;
      rk = valid ? 1.0f / sqrtf(sk + kNormEps) : 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        qhat[e] = qv[e] * rq;
        khat[e] = kv[e] * rk;
        zz[e] = ea * (gv[e] + dtb[e]);
        const float la = valid ? P.lb / (1.0f + expf(-zz[e])) : 0.f;
        sm.Qt[ti * kLds + c8 + e] = qhat[e];
        sm.Kt[ti * kLds + c8 + e] = khat[e];
        sm.Ki[ti * kLds + c8 + e] = la;
        sm.Vs[ti * kLds + c8 + e] = vv[e];
        sm.dO[ti * kLds + c8 + e] = dv8[e];
      }
      if (tid < kChunk)
        sm.bs[tid] = (tid < nt) ? 1.0f / (1.0f + expf(-__bfloat162float(P.beta[(tc0 + tid) * P.Hv + h])))
                                : 0.f;
    }
    __syncthreads();
    // ---- P1: cumulative decay (one key column per thread)
    if (tid < kDim) {
      const int kc = tid;
      float Gc = 0.f;
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        Gc += sm.Ki[i * kLds + kc];
        sm.Ki[i * kLds + kc] = Gc;
      }
      const float GC = Gc;
      sm.gC[kc] = expf(GC);
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        const float Gi = sm.Ki[i * kLds + kc];
        const float kh = sm.Kt[i * kLds + kc];
        const float gam = expf(Gi);
        sm.Gm[i * kLds + kc] = gam;
        sm.Qt[i * kLds + kc] *= gam;
        sm.Kt[i * kLds + kc] = kh * gam;
        sm.Ki[i * kLds + kc] = kh * expf(-Gi);
        sm.Kb[i * kLds + kc] = kh * expf(GC - Gi);
      }
    }
    __syncthreads();
    // ---- P2: A, B; Y = V - Kt S0^T and dWk = Kb G^T (reductions over k)
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
    {
      const int vv = tid & 127, i0 = (tid >> 7) * 8;
      float y[8], dw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) { y[i] = 0.f; dw[i] = 0.f; }
#pragma unroll 4
      for (int kk = 0; kk < kDim; kk += 4) {
        const float4 s4 = *reinterpret_cast<const float4*>(sm.S0 + vv * kLds + kk);
        const float4 g4 = *reinterpret_cast<const float4*>(sm.G + vv * kLds + kk);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          y[i] += dot4(*reinterpret_cast<const float4*>(sm.Kt + (i0 + i) * kLds + kk), s4);
          dw[i] += dot4(*reinterpret_cast<const float4*>(sm.Kb + (i0 + i) * kLds + kk), g4);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        sm.Vs[(i0 + i) * kLds + vv] -= y[i];
        sm.DU[(i0 + i) * kLds + vv] = dw[i];
      }
    }
    __syncthreads();
    // ---- P3: T = (I + diag(beta) A)^-1
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
    // ---- P4: per value column: W, U, dW, E, dV, E*U
    if (tid < kDim) {
      const int vv = tid;
      float y[kChunk], w[kChunk], dw[kChunk];
#pragma unroll
      for (int i = 0; i < kChunk; ++i) y[i] = sm.Vs[i * kLds + vv];
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j <= i; ++j) acc += sm.Tm[i * (kChunk + 1) + j] * sm.bs[j] * y[j];
        w[i] = acc;
      }
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        float acc = sm.DU[i * kLds + vv];
#pragma unroll
        for (int j = i; j < kChunk; ++j) acc += s * sm.Bm[j * (kChunk + 1) + i] * sm.dO[j * kLds + vv];
        dw[i] = acc;
      }
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        float e = 0.f;
#pragma unroll
        for (int j = i; j < kChunk; ++j) e += sm.Tm[j * (kChunk + 1) + i] * dw[j];
        float u = y[i];
#pragma unroll
        for (int j = 0; j < i; ++j) u -= sm.Am[i * (kChunk + 1) + j] * w[j];
        sm.Ws[i * kLds + vv] = w[i];
        sm.DU[i * kLds + vv] = sm.bs[i] * e;
        sm.Vs[i * kLds + vv] = e * u;
      }
    }
    __syncthreads();
    // ---- P5: reductions over v: dO S0, dV S0, W G, sum G*S0; dO W^T, dV W^T; dbeta rows
    float accq[8], accr[8], accw[8];
    const int kc = tid & 127, i0 = (tid >> 7) * 8;
    {
      float gs = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) { accq[i] = 0.f; accr[i] = 0.f; accw[i] = 0.f; }
#pragma unroll 2
      for (int vv = 0; vv < kDim; vv += 4) {
        float s0[4], g0[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          s0[x] = sm.S0[(vv + x) * kLds + kc];
          g0[x] = sm.G[(vv + x) * kLds + kc];
          gs += s0[x] * g0[x];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 o4 = *reinterpret_cast<const float4*>(sm.dO + (i0 + i) * kLds + vv);
          const float4 u4 = *reinterpret_cast<const float4*>(sm.DU + (i0 + i) * kLds + vv);
          const float4 w4 = *reinterpret_cast<const float4*>(sm.Ws + (i0 + i) * kLds + vv);
          accq[i] += o4.x * s0[0] + o4.y * s0[1] + o4.z * s0[2] + o4.w * s0[3];
          accr[i] += u4.x * s0[0] + u4.y * s0[1] + u4.z * s0[2] + u4.w * s0[3];
          accw[i] += w4.x * g0[0] + w4.y * g0[1] + w4.z * g0[2] + w4.w * g0[3];
        }
      }
      if (tid < kDim) sm.rho[0][kc] = gs;
#pragma unroll
      for (int rep = 0; rep < 2; ++rep) {
        const int e = tid + rep * kThreads;
        const int mat = e >> 8, i = (e >> 4) & 15, j = e & 15;
        const float* X = mat ? sm.DU : sm.dO;
        float acc = 0.f;
#pragma unroll 8
        for (int vv = 0; vv < kDim; vv += 4)
          acc += dot4(*reinterpret_cast<const float4*>(X + i * kLds + vv),
                      *reinterpret_cast<const float4*>(sm.Ws + j * kLds + vv));
        (mat ? sm.M2 : sm.M1)[i * (kChunk + 1) + j] = acc;
      }
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int i = warp * 2 + rr;
        const float4 x = *reinterpret_cast<const float4*>(sm.Vs + i * kLds + lane * 4);
        float acc = x.x + x.y + x.z + x.w;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) sm.dba[i] = acc;
      }
    }
    __syncthreads();
    // ---- P6: assemble dq^, dk^ and the gauge term; update G
    {
      float* dQh = sm.S0;              // tiles reuse the (no longer needed) S0 storage
      float* dKh = sm.S0 + kTile;
      float* tv = sm.S0 + 2 * kTile;
      const float gck = sm.gC[kc];
      float rp = 0.f;
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        const int i = i0 + ii;
        rp += sm.Kb[i * kLds + kc] * accw[ii];
        const float gam = sm.Gm[i * kLds + kc];
        const float inv = 1.0f / gam;
        float pq = accq[ii], pr = accr[ii], pw = gck * accw[ii];
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
          const float kij = sm.Ki[j * kLds + kc];
          if (j <= i) pq += sm.M1[i * (kChunk + 1) + j] * kij;
          if (j < i) pr += sm.M2[i * (kChunk + 1) + j] * kij;
          if (j >= i) pw += s * sm.M1[j * (kChunk + 1) + i] * sm.Qt[j * kLds + kc];
          if (j > i) pw -= sm.M2[j * (kChunk + 1) + i] * sm.Kt[j * kLds + kc];
        }
        const float dq_ = s * gam * pq;
        const float dkr = -gam * pr;
        const float dkw = inv * pw;
        const float qh_ = sm.Qt[i * kLds + kc] * inv;
        const float kh_ = sm.Kt[i * kLds + kc] * inv;
        dQh[i * kLds + kc] = dq_;
        dKh[i * kLds + kc] = dkr + dkw;
        tv[i * kLds + kc] = qh_ * dq_ + kh_ * (dkr - dkw);
      }
      sm.rho[1 + (tid >> 7)][kc] = rp;
      // G <- G diag(gC) + (scale dO)^T Qt - dV^T Kt
      const int gv = tid >> 1, half = tid & 1;
#pragma unroll 4
      for (int m = 0; m < 16; ++m) {
        const int kk = m * 8 + half * 4;
        float4 g4 = *reinterpret_cast<const float4*>(sm.G + gv * kLds + kk);
        const float4 c4 = *reinterpret_cast<const float4*>(sm.gC + kk);
        g4.x *= c4.x; g4.y *= c4.y; g4.z *= c4.z; g4.w *= c4.w;
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
          const float od = s * sm.dO[i * kLds + gv];
          const float ud = sm.DU[i * kLds + gv];
          const float4 q4 = *reinterpret_cast<const float4*>(sm.Qt + i * kLds + kk);
          const float4 k4 = *reinterpret_cast<const float4*>(sm.Kt + i * kLds + kk);
          g4.x += od * q4.x - ud * k4.x;
          g4.y += od * q4.y - ud * k4.y;
          g4.z += od * q4.z - ud * k4.z;
          g4.w += od * q4.w - ud * k4.w;
        }
        *reinterpret_cast<float4*>(sm.G + gv * kLds + kk) = g4;
      }
    }
    __syncthreads();
    // ---- P7: da = rho + reverse cumulative sum of the gauge term within the sub-chunk
    if (tid < kDim) {
      float* tv = sm.S0 + 2 * kTile;
      float run = sm.gC[tid] * sm.rho[0][tid] + sm.rho[1][tid] + sm.rho[2][tid];
#pragma unroll
      for (int i = kChunk - 1; i >= 0; --i) {
        run += tv[i * kLds + tid];
        tv[i * kLds + tid] = run;
      }
    }
    __syncthreads();
    // ---- P8: epilogue: gate / sigmoid / L2-norm backward and stores
    {
      const float* dQh = sm.S0;
      const float* dKh = sm.S0 + kTile;
      const float* da = sm.S0 + 2 * kTile;
      const bool valid = ti < nt;
      const int64_t t = tc0 + ti;
      float dg8[8], dq8[8], dk8[8], dv8[8];
      float pq = 0.f, pk = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        // sigmoid'(z) = sigmoid(z) sigmoid(-z), both evaluated directly (no 1 - s cancellation)
        const float sg = 1.0f / (1.0f + expf(-zz[e]));
        const float sn = 1.0f / (1.0f + expf(zz[e]));
        const float dz = valid ? da[ti * kLds + c8 + e] * P.lb * sg * sn : 0.f;
        dg8[e] = dz * ea;
        ddt_acc[e] += dg8[e];
        dA_acc += dz * zz[e];
        dq8[e] = dQh[ti * kLds + c8 + e];
        dk8[e] = dKh[ti * kLds + c8 + e];
        dv8[e] = sm.DU[ti * kLds + c8 + e];
        pq += qhat[e] * dq8[e];
        pk += khat[e] * dk8[e];
      }
      if (P.r == 1) {
        pq = row16_sum(pq);
        pk = row16_sum(pk);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          dq8[e] = rq * (dq8[e] - qhat[e] * pq);
          dk8[e] = rk * (dk8[e] - khat[e] * pk);
        }
      }
      if (valid) {
        store_bf16x8(a.dg + (t * P.Hv + h) * kDim + c8, dg8);
        store_bf16x8(a.dv + (t * P.Hv + h) * kDim + c8, dv8);
        if (P.r == 1) {
          store_bf16x8(a.dq + (t * P.Hqk + qh) * kDim + c8, dq8);
          store_bf16x8(a.dk + (t * P.Hqk + qh) * kDim + c8, dk8);
        } else {
          float* dst = a.dqk_part + ((t * P.Hv + h) * 2) * kDim + c8;
          *reinterpret_cast<float4*>(dst) = make_float4(dq8[0], dq8[1], dq8[2], dq8[3]);
          *reinterpret_cast<float4*>(dst + 4) = make_float4(dq8[4], dq8[5], dq8[6], dq8[7]);
          *reinterpret_cast<float4*>(dst + kDim) = make_float4(dk8[0], dk8[1], dk8[2], dk8[3]);
          *reinterpret_cast<float4*>(dst + kDim + 4) = make_float4(dk8[4], dk8[5], dk8[6], dk8[7]);
        }
      }
      if (tid < nt) {
        const float bl = __bfloat162float(P.beta[(tc0 + tid) * P.Hv + h]);
        const float bn = 1.0f / (1.0f + expf(bl));  // sigmoid(-logit)
        a.dbeta[(tc0 + tid) * P.Hv + h] = __float2bfloat16_rn(sm.dba[tid] * sm.bs[tid] * bn);
      }
    }
    __syncthreads();
  }
  // dinitial_state = G
  {
    float* dst = a.dh0 + (n * P.Hv + h) * kDim * kDim;
    for (int f = tid; f < kDim * kDim / 4; f += kThreads) {
      const int row = f >> 5, c4 = (f & 31) * 4;
      *reinterpret_cast<float4*>(dst + row * kDim + c4) =
          *reinterpret_cast<const float4*>(sm.G + row * kLds + c4);
    }
  }
  // per-unit parameter-gradient partials, reduced in a fixed order
  {
    float* red = sm.S0;  // [16 rows][128] + [256]
#pragma unroll
    for (int e = 0; e < 8; ++e) red[ti * kDim + c8 + e] = ddt_acc[e];
    red[kChunk * kDim + tid] = dA_acc;
    __syncthreads();
    float* dst = a.par_part + (int64_t)unit * kParStride;
    if (tid < kDim) {
      float acc = 0.f;
      for (int i = 0; i < kChunk; ++i) acc += red[i * kDim + tid];
      dst[tid] = acc;
    }
    if (tid == 0) {
      float acc = 0.f;
      for (int i = 0; i < kThreads; ++i) acc += red[kChunk * kDim + i];
      dst[kDim] = acc;
    }
  }
}

// dA_log[h] and ddt_bias[h, :] summed over sequences in index order.
__global__ void kda_param_reduce_kernel(const float* __restrict__ par_part, int64_t N, int64_t Hv,
                                        float* __restrict__ dA_log, float* __restrict__ ddt_bias) {
  const int64_t h = blockIdx.x;
  const int k = threadIdx.x;
  float acc = 0.f;
  for (int64_t n = 0; n < N; ++n) acc += par_part[(n * Hv + h) * kParStride + k];
  if (k < kDim) ddt_bias[h * kDim + k] = acc;
  else dA_log[h] = acc;
}

// GQA: sum d(q^), d(k^) over the value heads of each query/key head (fixed
// order), then the L2-norm backward  dx = r (dx^ - x^ (x^ . dx^)).
__global__ void kda_gqa_reduce_kernel(const Problem P, const float* __restrict__ part, int64_t Ttot,
                                      __nv_bfloat16* __restrict__ dq, __nv_bfloat16* __restrict__ dk) {
  const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= Ttot * P.Hqk) return;
  const int64_t t = gw / P.Hqk, qh = gw % P.Hqk;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int hh = 0; hh < P.r; ++hh) {
      const int64_t h = qh * P.r + hh;
      const float4 x = *reinterpret_cast<const float4*>(part + ((t * P.Hv + h) * 2 + which) * kDim + lane * 4);
      acc[0] += x.x; acc[1] += x.y; acc[2] += x.z; acc[3] += x.w;
    }
    const __nv_bfloat16* src = (which == 0 ? P.q : P.k) + (t * P.Hqk + qh) * kDim + lane * 4;
    float xv[4];
    {
      const uint2 raw = *reinterpret_cast<const uint2*>(src);
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
      const float2 f0 = __bfloat1622float2(h2[0]), f1 = __bfloat1622float2(h2[1]);
      xv[0] = f0.x; xv[1] = f0.y; xv[2] = f1.x; xv[3] = f1.y;
    }
    float ss = xv[0] * xv[0] + xv[1] * xv[1] + xv[2] * xv[2] + xv[3] * xv[3];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float r = 1.0f / sqrtf(ss + kNormEps);
    float pd = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) { xv[e] *= r; pd += xv[e] * acc[e]; }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) pd += __shfl_xor_sync(0xffffffffu, pd, off);
    uint2 outraw;
    __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&outraw);
    o2[0] = __floats2bfloat162_rn(r * (acc[0] - xv[0] * pd), r * (acc[1] - xv[1] * pd));
    o2[1] = __floats2bfloat162_rn(r * (acc[2] - xv[2] * pd), r * (acc[3] - xv[3] * pd));
    *reinterpret_cast<uint2*>((which == 0 ? dq : dk) + (t * P.Hqk + qh) * kDim + lane * 4) = outraw;
  }
}

}  // namespace

cudaError_t launch_backward(const Problem& P, const BwdArgs& a, int64_t units, int64_t Ttot,
                            float* dA_log, float* ddt_bias, cudaStream_t s) {
  const size_t smem = sizeof(BwdSmem);
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  kda_bwd_kernel<<<(unsigned)units, kThreads, smem, s>>>(P, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  kda_param_reduce_kernel<<<(unsigned)P.Hv, kDim + 1, 0, s>>>(a.par_part, P.N, P.Hv, dA_log, ddt_bias);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (P.r > 1) {
    const int64_t warps = Ttot * P.Hqk;
    const int per_block = 8;
    kda_gqa_reduce_kernel<<<(unsigned)((warps + per_block - 1) / per_block), per_block * 32, 0, s>>>(
        P, a.dqk_part, Ttot, a.dq, a.dk);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kda
