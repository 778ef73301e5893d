// kda_fwd.cu -- chunked forward of the recurrent KDA training recurrence on
// sm_103a tensor cores.
//
// One CTA owns one (sequence, value head) unit and walks its tokens in
// sub-chunks of kChunk = 16, keeping the 128x128 FP32 value-first state in
// tensor memory (one value row per lane), where it is also the accumulator of
// the state update; two CTAs fit on one SM. Within a sub-chunk starting from
// state S0, with Gam_i the cumulative log-decay of tokens 1..i (per key dim)
// and gamma_i = exp(Gam_i):
//   A_ij = k^_i . (k^_j gamma_i / gamma_j)   (j < i)      B_ij likewise with q^_i (j <= i)
//   Y    = V - (k^ gamma) S0^T
//   W    solves (I + diag(beta) A) W = diag(beta) Y      (rows: beta_i u_i)
//   O    = scale ((q^ gamma) S0^T + B W)
//   S_C  = S0 diag(gamma_C) + W^T (k^ gamma_C / gamma)
// which equals the token-by-token rule S' = S diag(d); u = v - S' k^;
// S = S' + beta u k^T; o = scale S q^ (flashinfer.kda_backward.recurrent_kda_backward,
// description: gate, norm and sigmoid contracts; the update order is the plain
// reading the library adopts).
//
// Tensor cores (tcgen05.mma kind::tf32, FP32 accumulators in TMEM) compute the
// two state-sized contractions S0 [k^ gamma; q^ gamma]^T (128x32, the state as
// the tensor-memory A operand) and W^T (k^ gamma_C/gamma) (128x128, added into
// the state, W^T written by the solving threads into tensor memory as its A
// operand), as well as the 16x16 A and B (an M = 64 product next to the first
// contraction) and the output's B W term (next to the second); the next
// sub-chunk's prologue runs while the second group is in flight. Token tiles
// are prefetched into registers one sub-chunk ahead. Between the two groups,
// the two independent passes run side by side on the two warp halves: warps
// 0-3 solve for W (one state row per thread) and then build the (k^ gamma_C /
// gamma)^T operand of the second group (needed by no earlier step) while warps
// 4-7 store the state checkpoint and decay the state. The 16x16 A and B are read
// out of TMEM before the solve by warps 0, 1 (columns 0-7) and 4, 5 (columns
// 8-15, the same lane quarters; prefill: warps 0, 1 alone). Value rows are placed in TMEM
// lanes so that a 16-lane (.16x128b) load gives a thread four consecutive
// value rows of a key column, which is one 16-byte group of the transposed
// checkpoint: the checkpoint needs no exchange between lanes.
// Operands written to shared memory are rounded to TF32; the state read as the
// A operand is truncated to TF32 by the tensor core (it only feeds the
// sub-chunk's Y and O); the state update uses split TF32 (x = hi + lo, three
// products) so that the carried FP32 state keeps FP32-level accuracy.
// Accumulation, the triangular solve, the output and the state stay FP32.
// Each token's u = v - S' k^ and each sub-chunk's A and B are saved for the
// backward. The gate, L2 norm and sigmoid of each token are computed on chip
// (the fused prologue). The state at the start of every checkpoint interval is
// stored for the backward (transposed, in the layout the backward's
// tensor-core products read).
#include <type_traits>

#include "kda_common.cuh"
#include "tc.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kTileF = kChunk * kLds;
constexpr uint32_t kTmemCols = 256;  // two CTAs per SM share the 512 columns
constexpr uint32_t kColS = 0;        // FP32 state S (one value row per lane, see sv below; column = key k)
constexpr uint32_t kColYO = 128;     // S0 [k^g; q^g]^T : 32 columns; the last 16 then also take + W^T B^T
constexpr uint32_t kColAB = 160;     // [k^g; q^g] (k^/g)^T (M = 64): A in lanes 0..15, B in lanes 32..47, 16 columns
constexpr uint32_t kColW = 176;      // W^T (value rows as in S, column = token): TF32 hi in 16 columns, lo in the next 16
constexpr uint32_t kColU = 208;      // u (value rows as in S, column = token), for the tape

struct FwdSmem {
  // rows 0..15 k^ gamma, rows 16..31 q^ gamma (K-major, K = 128). As the A operand of the A/B
  // product (M = 64) it is read as 64 rows: rows 32..63 fall on the tile below and only fill TMEM
  // lanes that are never read. Once the first group has completed it holds, until the next tile
  // build, the sub-chunk's B^T in FP32 (16 x 16, after 16 x kLds floats) for the tape.
  unsigned char KQ[32 * kDim * 4];
  unsigned char KiT[kChunk * kDim * 4];    // k^ / gamma rows t, TF32 (K-major, K = 128)
  unsigned char Bt[kChunk * kChunk * 4];   // B rows t, TF32 (K-major, K = 16): O += W^T B^T
  unsigned char KbT[2][kDim * kChunk * 4]; // (k^ gamma_C / gamma)^T, rows k, TF32 hi / lo (K = 16)
  float Pq[kTileF];                        // q^
  float Pk[kTileF];                        // k^
  float Kif[kTileF];                       // k^ / gamma (FP32), from the tile build
  float Pa[kTileF];                        // log decay, then gamma
  float Vs[kTileF];                        // v
  float AsT[kChunk][kChunk];               // A transposed: AsT[j][t] = A[t][j]
  float bs[kChunk];
  float gC[kDim];
  unsigned long long mbar;
  uint32_t tmem_base;
};

// kPf = false: the training forward (tapes and checkpoints for the backward,
// h0 in, h_T out). kPf = true: inference prefill (PrefillArgs; units in index
// order, sequence offsets from the device cu_seqlens, no tapes).
template <bool kPf>
__global__ void __launch_bounds__(kThreads, 2)
kda_fwd_kernel(const Problem P, const FwdOut out, const PrefillArgs pf) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int unit = kPf ? (int)blockIdx.x : P.order[blockIdx.x];
  const int64_t n = unit / P.Hv;
  const int64_t h = unit % P.Hv;
  const int64_t qh = h / P.r;
  SeqInfo si;
  if constexpr (kPf) {
    si.t0 = pf.cu ? pf.cu[n] : n * pf.T;
    si.len = pf.cu ? pf.cu[n + 1] - si.t0 : pf.T;
    si.ck_base = 0;
    si.ch_base = 0;
  } else {
    si = P.seq[n];
  }
  const int64_t slot = kPf ? (pf.slots ? pf.slots[n] : n) : 0;
  if constexpr (kPf) {
    if (slot < 0 || slot >= pf.num_slots) {
      // a device index outside the pool (it no longer matches the host mirror the call was
      // checked against, e.g. in a replayed graph): flagged, and the pool is not touched
      if (threadIdx.x == 0) atomicOr(P.status, 4);
      return;
    }
  }

  const int sv = 32 * (warp & 3) + 4 * (lane & 7) + (lane >> 3);  // state row held in this thread's TMEM lane
  const int ch = warp >> 2;               // column half [64 ch, 64 ch + 64)
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&sm.tmem_base), kTmemCols);
  if (tid == 0) tc::mbar_init(tc::smem_u32(&sm.mbar), 1);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = sm.tmem_base;
  const uint32_t tl = tbase + ((uint32_t)(32 * (warp & 3)) << 16);
  const uint32_t mbar = tc::smem_u32(&sm.mbar);
  uint32_t parity = 0;
  bool ok = true;
  bool aborted = false;

  // S <- h0 (prefill: the pool slot)
  {
    const int64_t row = ((kPf ? slot : n) * P.Hv + h) * kDim + sv;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      float x[16];
      if (kPf && pf.pool_bf16) {
        const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(pf.pool) + row * kDim + 64 * ch + 16 * q;
        load_bf16x8(src, x);
        load_bf16x8(src + 8, x + 8);
      } else {
        const float* src = (kPf ? reinterpret_cast<const float*>(pf.pool) : P.h0) + row * kDim + 64 * ch + 16 * q;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 y = *reinterpret_cast<const float4*>(src + 4 * m);
          x[4 * m] = y.x; x[4 * m + 1] = y.y; x[4 * m + 2] = y.z; x[4 * m + 3] = y.w;
        }
      }
      tc::tmem_st16(tl + kColS + 64 * ch + 16 * q, x);
    }
    tc::tmem_wait_st();
  }

  const int ti = tid >> 4;
  const int c8 = (tid & 15) * 8;
  // prefill gate modes: g already in log space (A_log and dt_bias unused), beta already sigmoided
  const bool log_g = kPf && !pf.gate_in_kernel;
  const bool beta_logit = !kPf || pf.beta_logit;
  bool g_range_bad = false;
  const float ea = log_g ? 0.f : expf(P.A_log[h]);
  float dtb[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) dtb[e] = log_g ? 0.f : P.dt_bias[h * kDim + c8 + e];

  const int64_t nchunks = (si.len + kChunk - 1) / kChunk;
  const int ck_every = kCkTokens / kChunk;
  // raw BF16 tiles of the next sub-chunk (token row ti, columns c8..c8+7)
  uint4 nq = make_uint4(0u, 0u, 0u, 0u), nk = nq, ng = nq, nv = nq;
  __nv_bfloat16 nb = __float2bfloat16_rn(0.f);
  auto prefetch = [&](int64_t cc) {
    const int64_t t = si.t0 + cc * kChunk + ti;
    const bool ok_row = cc < nchunks && (cc * kChunk + ti) < si.len;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    nq = ok_row ? *reinterpret_cast<const uint4*>(P.q + (t * P.Hqk + qh) * kDim + c8) : z;
    nk = ok_row ? *reinterpret_cast<const uint4*>(P.k + (t * P.Hqk + qh) * kDim + c8) : z;
    ng = ok_row ? *reinterpret_cast<const uint4*>(P.g + (t * P.Hv + h) * kDim + c8) : z;
    nv = ok_row ? *reinterpret_cast<const uint4*>(P.v + (t * P.Hv + h) * kDim + c8) : z;
    if (tid < kChunk) {
      const int64_t tb = si.t0 + cc * kChunk + tid;
      nb = (cc < nchunks && (cc * kChunk + tid) < si.len) ? P.beta[tb * P.Hv + h] : __float2bfloat16_rn(0.f);
    }
  };
  // prologue and cumulative decay of sub-chunk cc (token tiles already prefetched)
  auto prologue = [&](int64_t cc) {
    const int ntc = (int)((si.len - cc * kChunk) < kChunk ? (si.len - cc * kChunk) : kChunk);
    {
      float qv[8], kv[8], gv[8], vv[8];
      const bool valid = ti < ntc;
      unpack_bf16x8(nq, qv);
      unpack_bf16x8(nk, kv);
      unpack_bf16x8(ng, gv);
      unpack_bf16x8(nv, vv);
      const float braw = __bfloat162float(nb);
      prefetch(cc + 1);
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) { sq += qv[e] * qv[e]; sk += kv[e] * kv[e]; }
      sq = row16_sum(sq);
      sk = row16_sum(sk);
      const float rq = valid ? inv_norm_of(sq) : 0.f;
      const float rk = valid ? inv_norm_of(sk) : 0.f;
      float la[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float z = ea * (gv[e] + dtb[e]);
        qv[e] *= rq;
        kv[e] *= rk;
        if (log_g) {
          g_range_bad |= valid && !(gv[e] >= -5.f && gv[e] <= 0.f);
          la[e] = valid ? gv[e] : 0.f;
        } else {
          la[e] = valid ? log_decay_of(P.lb, z) : 0.f;
        }
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int o = 4 * hh, col = ti * kLds + c8 + o;
        *reinterpret_cast<float4*>(sm.Pq + col) = make_float4(qv[o], qv[o + 1], qv[o + 2], qv[o + 3]);
        *reinterpret_cast<float4*>(sm.Pk + col) = make_float4(kv[o], kv[o + 1], kv[o + 2], kv[o + 3]);
        *reinterpret_cast<float4*>(sm.Pa + col) = make_float4(la[o], la[o + 1], la[o + 2], la[o + 3]);
        *reinterpret_cast<float4*>(sm.Vs + col) = make_float4(vv[o], vv[o + 1], vv[o + 2], vv[o + 3]);
      }
      if (tid < kChunk) sm.bs[tid] = (tid < ntc) ? (beta_logit ? sigmoid_of(braw) : braw) : 0.f;
    }
    __syncthreads();
    if (tid < kDim) {
      float av[kChunk];
#pragma unroll
      for (int i = 0; i < kChunk; ++i) av[i] = sm.Pa[i * kLds + tid];
      float G = 0.f;
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        G += av[i];
        av[i] = expf(G);
      }
#pragma unroll
      for (int i = 0; i < kChunk; ++i) sm.Pa[i * kLds + tid] = av[i];
      sm.gC[tid] = av[kChunk - 1];
    }
  };

  prefetch(0);
  prologue(0);
  __syncthreads();  // the first prologue is complete; later ones end at the loop's last barrier
  for (int64_t c = 0; c < nchunks; ++c) {
    const int64_t tc0 = si.t0 + c * kChunk;
    const int nt = (int)((si.len - c * kChunk) < kChunk ? (si.len - c * kChunk) : kChunk);
    // ---- operand tiles: token t, key quads q4 and q4 + 16
    {
      const int t = tid & 15;
#pragma unroll
      for (int rep = 0; rep < 2; ++rep) {
        const int k0 = 4 * ((tid >> 4) + 16 * rep);
        const float4 qh4 = *reinterpret_cast<const float4*>(sm.Pq + t * kLds + k0);
        const float4 kh4 = *reinterpret_cast<const float4*>(sm.Pk + t * kLds + k0);
        const float4 g4 = *reinterpret_cast<const float4*>(sm.Pa + t * kLds + k0);
        const float qa[4] = {qh4.x, qh4.y, qh4.z, qh4.w}, ka[4] = {kh4.x, kh4.y, kh4.z, kh4.w};
        const float ga[4] = {g4.x, g4.y, g4.z, g4.w};
        float kt[4], qt[4], ki[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float inv = __fdividef(1.0f, ga[e]);  // gamma is in [e^-80, 1]
          kt[e] = ka[e] * ga[e];
          qt[e] = qa[e] * ga[e];
          ki[e] = ka[e] * inv;
        }
        *reinterpret_cast<float4*>(sm.KQ + tc::kmaj(t, k0, kDim)) =
            make_float4(tc::round_tf32(kt[0]), tc::round_tf32(kt[1]), tc::round_tf32(kt[2]), tc::round_tf32(kt[3]));
        *reinterpret_cast<float4*>(sm.KQ + tc::kmaj(16 + t, k0, kDim)) =
            make_float4(tc::round_tf32(qt[0]), tc::round_tf32(qt[1]), tc::round_tf32(qt[2]), tc::round_tf32(qt[3]));
        *reinterpret_cast<float4*>(sm.KiT + tc::kmaj(t, k0, kDim)) =
            make_float4(tc::round_tf32(ki[0]), tc::round_tf32(ki[1]), tc::round_tf32(ki[2]), tc::round_tf32(ki[3]));
        *reinterpret_cast<float4*>(sm.Kif + t * kLds + k0) = make_float4(ki[0], ki[1], ki[2], ki[3]);
      }
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    // ---- tensor cores: S0 [k^g; q^g]^T with the state read from tensor memory, and the 16x16
    // A_ij = (k^g)_i . (k^/g)_j, B_ij = (q^g)_i . (k^/g)_j (TF32 operands, FP32 accumulation)
    if (warp == 0) {
      if (tc::elect_one()) {
        tc::fence_after();
        // K-step st of a tile adds 16 * st to its descriptor's address field
        const uint64_t dkq = tc::kdesc(tc::smem_u32(sm.KQ), 0, kDim), dkit = tc::kdesc(tc::smem_u32(sm.KiT), 0, kDim);
#pragma unroll
        for (int st = 0; st < kDim / 8; ++st)
          tc::mma_ts(tbase + kColYO, tbase + kColS + 8 * st, dkq + 16u * st, tc::idesc_tf32(128, 32), st > 0);
#pragma unroll
        for (int st = 0; st < kDim / 8; ++st)
          tc::mma_ss(tbase + kColAB, dkq + 16u * st, dkit + 16u * st, tc::idesc_tf32(64, 16), st > 0);
        tc::mma_commit(mbar);
      }
      __syncwarp();
    }
    if (ok) ok = tc::mbar_wait_warp(mbar, parity);
    parity ^= 1;
    tc::fence_after();
    // A (D rows 0..15: lanes 0..15 of lane quarter 0, strictly lower) and B (D rows 16..31: lanes
    // 0..15 of quarter 1, lower) from tensor memory (an M = 64 product places rows 16 w .. 16 w + 15
    // in lanes 32 w .. 32 w + 15). Training: warps 0 / 1 take columns 0..7 and warps 4 / 5 columns
    // 8..15 (warps 4-7 reach this point well ahead of their own pass's end); prefill: warps 0 / 1
    // take all 16 (measured faster there, with no tape copy to make). The backward's tape, written
    // by all threads after the second group, holds A row-major (from AsT) and B transposed (its
    // columns are read there; from the FP32 copy left in the KQ tile)
    constexpr int kRb = kPf ? 16 : 8;  // columns per readback thread
    if ((warp & 3) < 2 && (!kPf || warp < 4)) {
      const int j0 = 8 * (warp >> 2);
      float d8[kRb];
      if constexpr (kRb == 16) tc::tmem_ld16(tl + kColAB, d8);
      else tc::tmem_ld8(tl + kColAB + j0, d8);
      if (lane < kChunk) {
        const int i = lane;
        if ((warp & 3) == 0) {
#pragma unroll
          for (int jj = 0; jj < kRb; ++jj) sm.AsT[j0 + jj][i] = j0 + jj < i ? d8[jj] : 0.f;
        } else {
#pragma unroll
          for (int jj = 0; jj < kRb; ++jj) {
            d8[jj] = j0 + jj <= i ? d8[jj] : 0.f;
            if constexpr (!kPf) reinterpret_cast<float*>(sm.KQ)[kChunk * kLds + (j0 + jj) * 16 + i] = d8[jj];  // B^T
          }
#pragma unroll
          for (int q4 = 0; q4 < kRb / 4; ++q4) {
            *reinterpret_cast<float4*>(sm.Bt + tc::kmaj(i, j0 + 4 * q4, kChunk)) =
                make_float4(tc::round_tf32(d8[4 * q4]), tc::round_tf32(d8[4 * q4 + 1]), tc::round_tf32(d8[4 * q4 + 2]),
                            tc::round_tf32(d8[4 * q4 + 3]));
          }
        }
      }
      if (warp >= 4) asm volatile("bar.arrive 2, 192;" ::: "memory");  // warps 0-3 wait on it below
    }
    if (warp < 4) {
      // ---- warps 0-3: once A and B are in shared memory (warps 0, 1, 4, 5 above), W by forward
      // substitution for state row sv; u of all 16 tokens into tensor memory; W's two TF32 parts;
      // then the second group's (k^ gamma_C / gamma)^T operand
      asm volatile("bar.sync 2, %0;" ::"n"(kPf ? 128 : 192) : "memory");  // warps 0-3 (and 4, 5 in training)
      float yp[16];
      tc::tmem_ld16(tl + kColYO, yp);
      float w[kChunk], acc[kChunk];
#pragma unroll
      for (int t = 0; t < kChunk; ++t) acc[t] = sm.Vs[t * kLds + sv] - yp[t];
#pragma unroll
      for (int j = 0; j < kChunk; ++j) {
        w[j] = sm.bs[j] * acc[j];  // acc[j] is final here: u_j
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          if (4 * q4 + 3 <= j) continue;
          const float4 x = *reinterpret_cast<const float4*>(&sm.AsT[j][4 * q4]);
          const float ar[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (4 * q4 + e > j) acc[4 * q4 + e] = fmaf(-ar[e], w[j], acc[4 * q4 + e]);
        }
      }
      if constexpr (!kPf) tc::tmem_st16(tl + kColU, acc);  // u_t for the backward's tape
      float xh[kChunk], xl[kChunk];
#pragma unroll
      for (int t = 0; t < kChunk; ++t) {
        xh[t] = tc::round_tf32(w[t]);
        xl[t] = tc::round_tf32(w[t] - xh[t]);
      }
      tc::tmem_st16(tl + kColW, xh);  // the tensor-memory A operand of the update
      tc::tmem_st16(tl + kColW + 16, xl);
      {  // (k^ gamma_C / gamma)^T as rows k (K = token) in TF32 hi + lo, for the second group: key k,
         // all 16 tokens, each float4 store covering 4 tokens
        const int k = tid;
        const float gck = sm.gC[k];
#pragma unroll 2
        for (int t4 = 0; t4 < kChunk; t4 += 4) {
          float hi[4], lo[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int t = t4 + j;
            const float kb = sm.Kif[t * kLds + k] * gck;
            hi[j] = tc::round_tf32(kb);
            lo[j] = tc::round_tf32(kb - hi[j]);
          }
          *reinterpret_cast<float4*>(sm.KbT[0] + tc::kmaj(k, t4, kChunk)) = make_float4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<float4*>(sm.KbT[1] + tc::kmaj(k, t4, kChunk)) = make_float4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
    } else {
      // ---- warps 4-7: state checkpoint and decay S <- S0 diag(gamma_C), all columns
      if constexpr (!kPf) {
        // TMEM lanes 32 w + 8 j + a hold value rows 32 w + 4 a + j (j = 0..3), so the two .16x128b
        // loads of a 16-column slice give this thread value rows 32 w + 4 (lane / 4) + 0..3 of the
        // four key columns 4 i + lane % 4: one 16-byte group of the checkpoint layout each
        float* dst = P.ckpt + ((si.ck_base + c / ck_every) * P.Hv + h) * kDim * kDim +
                     ckpt_index(32 * (warp & 3) + 4 * (lane >> 2), lane & 3);
        const bool ck = (c % ck_every) == 0;
#pragma unroll 1
        for (int q = 0; q < 8; ++q) {
          const int col = 16 * q;
          float x0[8], x1[8];
          tc::tmem_ld16x128_nowait(tl + kColS + col, x0);
          tc::tmem_ld16x128_nowait(tl + (16u << 16) + kColS + col, x1);
          tc::tmem_wait_ld8x2(x0, x1);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (ck)
              *reinterpret_cast<float4*>(dst + 4 * (col + 4 * i)) = make_float4(x0[2 * i], x0[2 * i + 1], x1[2 * i], x1[2 * i + 1]);
            const float gk = sm.gC[col + 4 * i + (lane & 3)];
            x0[2 * i] *= gk; x0[2 * i + 1] *= gk; x1[2 * i] *= gk; x1[2 * i + 1] *= gk;
          }
          tc::tmem_st16x128(tl + kColS + col, x0);
          tc::tmem_st16x128(tl + (16u << 16) + kColS + col, x1);
        }
      } else {
        const bool pck = pf.ck != nullptr && (c % pf.ck_every_chunks) == 0;
        __nv_bfloat16* pdst = pck ? pf.ck + ((pf.ck_starts[n] + c / pf.ck_every_chunks) * P.Hv + h) * kDim * kDim +
                                        (int64_t)sv * kDim
                                  : nullptr;
#pragma unroll 1
        for (int q = 0; q < 8; ++q) {
          const int col = 16 * q;
          float x[16];
          tc::tmem_ld16(tl + kColS + col, x);
          if (pck) {
            store_bf16x8(pdst + 16 * q, x);
            store_bf16x8(pdst + 16 * q + 8, x + 8);
          }
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float4 g4 = *reinterpret_cast<const float4*>(sm.gC + col + 4 * m);
            x[4 * m] *= g4.x; x[4 * m + 1] *= g4.y; x[4 * m + 2] *= g4.z; x[4 * m + 3] *= g4.w;
          }
          tc::tmem_st16(tl + kColS + col, x);
        }
      }
    }
    tc::tmem_wait_st();
    tc::fence_async_smem();
    tc::fence_before();
    if (__syncthreads_or(!ok)) { aborted = true; break; }
    // ---- tensor cores: S += W^T (k^ gamma_C / gamma) in split TF32 (hi hi + lo hi + hi lo), and
    // the output's W^T B^T added to S0 (q^ gamma)^T (W split, B in TF32)
    if (warp == 0) {
      if (tc::elect_one()) {
        tc::fence_after();
        // base descriptors made opaque here, so each K-step's descriptor is one add next to its MMA
        // rather than a register held across the sub-chunk loop
        uint64_t dkb0 = tc::kdesc(tc::smem_u32(sm.KbT[0]), 0, kChunk), dkb1 = tc::kdesc(tc::smem_u32(sm.KbT[1]), 0, kChunk);
        uint64_t dbt = tc::kdesc(tc::smem_u32(sm.Bt), 0, kChunk);
        asm volatile("" : "+l"(dkb0), "+l"(dkb1), "+l"(dbt));
        const int pa[3] = {0, 16, 0};
        const uint64_t pb[3] = {dkb0, dkb0, dkb1};
#pragma unroll
        for (int p = 0; p < 3; ++p)
#pragma unroll
          for (int st = 0; st < kChunk / 8; ++st)
            tc::mma_ts(tbase + kColS, tbase + kColW + pa[p] + 8 * st, pb[p] + 16u * st, tc::idesc_tf32(128, 128), 1);
#pragma unroll
        for (int p = 0; p < 2; ++p)
#pragma unroll
          for (int st = 0; st < kChunk / 8; ++st)
            tc::mma_ts(tbase + kColYO + 16, tbase + kColW + 16 * p + 8 * st, dbt + 16u * st, tc::idesc_tf32(128, 16), 1);
        tc::mma_commit(mbar);
      }
      __syncwarp();
    }
    // ---- meanwhile, the next sub-chunk's prologue (it touches no tensor-core operand)
    prologue(c + 1);  // also past the last sub-chunk (all rows invalid, unused): no branch before the output
    if (ok) ok = tc::mbar_wait_warp(mbar, parity);
    parity ^= 1;
    tc::fence_after();
    {  // the output of this warp's half of the tokens: o = scale (S0 (q^ gamma)^T + W^T B^T); two
       // 16-lane loads give this thread value rows 32 w + 4 (lane / 4) + 0..3 of tokens
       // 8 ch + 4 i + lane % 4 (i = 0, 1): one 8-byte store per token
      float x0[4], x1[4];
      tc::tmem_ld16x128x2_nowait(tl + kColYO + 16 + 8 * ch, x0);
      tc::tmem_ld16x128x2_nowait(tl + (16u << 16) + kColYO + 16 + 8 * ch, x1);
      tc::tmem_wait_ld4x2(x0, x1);
      const int v0 = 32 * (warp & 3) + 4 * (lane >> 2);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t = 8 * ch + 4 * i + (lane & 3);
        if (t < nt) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(P.scale * x0[2 * i], P.scale * x0[2 * i + 1]);
          __nv_bfloat162 hi = __floats2bfloat162_rn(P.scale * x1[2 * i], P.scale * x1[2 * i + 1]);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t*>(&lo);
          pk.y = *reinterpret_cast<uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(out.o + ((tc0 + t) * P.Hv + h) * kDim + v0) = pk;
        }
      }
    }
    if constexpr (!kPf) {  // the A/B tape: A row-major (from AsT), B transposed
      float* tape = P.abtape + ((si.ch_base + c) * P.Hv + h) * 512;
      tape[tid] = sm.AsT[tid & 15][tid >> 4];
      tape[256 + tid] = reinterpret_cast<const float*>(sm.KQ)[kChunk * kLds + tid];
    }
    if constexpr (!kPf) {  // the u tape: value rows 32 w + 4 (lane / 4) + 0..3 of tokens 8 ch + 4 i + lane % 4
      float u0[4], u1[4];
      tc::tmem_ld16x128x2_nowait(tl + kColU + 8 * ch, u0);
      tc::tmem_ld16x128x2_nowait(tl + (16u << 16) + kColU + 8 * ch, u1);
      tc::tmem_wait_ld4x2(u0, u1);
      const int v0 = 32 * (warp & 3) + 4 * (lane >> 2);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t = 8 * ch + 4 * i + (lane & 3);
        if (t < nt)
          *reinterpret_cast<float4*>(P.utape + ((tc0 + t) * P.Hv + h) * kDim + v0) =
              make_float4(u0[2 * i], u0[2 * i + 1], u1[2 * i], u1[2 * i + 1]);
      }
    }
    if (__syncthreads_or(!ok)) { aborted = true; break; }
  }
  if (!aborted) {
    const int64_t row = ((kPf ? slot : n) * P.Hv + h) * kDim + sv;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      float x[16];
      tc::tmem_ld16(tl + kColS + 64 * ch + 16 * q, x);
      if (kPf && pf.pool_bf16) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(pf.pool) + row * kDim + 64 * ch + 16 * q;
        store_bf16x8(dst, x);
        store_bf16x8(dst + 8, x + 8);
      } else {
        float* dst = (kPf ? reinterpret_cast<float*>(pf.pool) : out.hT) + row * kDim + 64 * ch + 16 * q;
#pragma unroll
        for (int m = 0; m < 4; ++m)
          *reinterpret_cast<float4*>(dst + 4 * m) = make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
      }
    }
  } else if (tid == 0) {
    atomicOr(P.status, 1);
  }
  if (g_range_bad) atomicOr(P.status, 2);
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_forward(const Problem& P, const FwdOut& out, int64_t units, cudaStream_t s) {
  const size_t smem = sizeof(FwdSmem);
  cudaError_t e = cudaFuncSetAttribute(kda_fwd_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kda_fwd_kernel<false><<<(unsigned)units, kThreads, smem, s>>>(P, out, PrefillArgs{});
  return cudaGetLastError();
}

cudaError_t launch_prefill(const Problem& P, const FwdOut& out, const PrefillArgs& pf, int64_t units,
                           cudaStream_t s) {
  const size_t smem = sizeof(FwdSmem);
  cudaError_t e = cudaFuncSetAttribute(kda_fwd_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kda_fwd_kernel<true><<<(unsigned)units, kThreads, smem, s>>>(P, out, pf);
  return cudaGetLastError();
}

}  // namespace kda
