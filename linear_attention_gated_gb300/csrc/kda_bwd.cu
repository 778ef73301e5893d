// kda_bwd.cu -- reverse-time chunked backward of the recurrent KDA recurrence
// on sm_103a tensor cores.
//
// One CTA owns one (sequence, value head) unit. It walks the unit's sub-chunks
// from last to first, carrying the state adjoint G = dL/dS as an FP32
// accumulator in tensor memory twice, as G (lane = value dim v) and as G^T
// (lane = key dim k): both receive the same rank-32 update, and each is the
// tensor-memory A operand of the products that contract over its columns.
// Per sub-chunk it reads the chunk-start state S0 saved by the
// forward and the forward's per-token u = v - S' k^ (so W = diag(beta) U is
// never recomputed), and with Gd = G diag(gamma_C) (the adjoint moved to the
// decayed end state):
//   dW = (k^/gamma) Gd^T + scale B^T dO,   E = T^T dW,   dV = diag(beta) E
//   dbeta_i = E_i . U_i  (before the sigmoid derivative)
//   dq^ = scale gamma * (dO S0 + tril(dO W^T) (k^/gamma))
//   dk^ = -gamma * (dV S0 + stril(dV W^T) (k^/gamma))                  (read key)
//       + (1/gamma) * (W Gd + triu(scale W dO^T) (q^ gamma)
//                      - striu(W dV^T) (k^ gamma))                      (write key)
//   G  <- Gd + (scale dO)^T (q^ gamma) - dV^T (k^ gamma)
// with T = (I + diag(beta) A)^-1 applied by substitution. The decay gradient
// uses the gauge identity of the per-key-dim decay: scaling the decay of token
// t in key dim j by e^eps equals scaling, for every later token, the query and
// the read key by e^eps and the written key by e^-eps, and the final state's
// column j by e^eps. Applied at the end of each sub-chunk, where scaling column
// j of the state S_C has the direct effect sum_v G[v,j] S_C[v,j], it gives for
// the tokens t of the sub-chunk
//   da_t = sum_{s >= t in chunk} (q^ dq^ + k^ (dk^_read - dk^_write))_s + rho,
//   rho  = sum_v (Gd * S0) + sum_i (k^/gamma)_i * (W Gd)_i,
// so no per-token elementwise state product is needed and no sum runs across
// sub-chunks (a running sum over the whole sequence drifts in FP32).
//
// Each sub-chunk first decays both copies of the adjoint to Gd = G diag(gamma_C)
// on CUDA cores. Tensor cores (tcgen05.mma kind::tf32, FP32 accumulators in
// TMEM) then compute the state-sized contractions dW = Gd (k^/g)^T + scale dO^T B
// (B split into TF32 hi + lo), S0^T [dO; dV]^T,
// Gd^T W^T (W split into TF32 hi + lo) and the rank-32 adjoint update (dV split
// into hi + lo; dO is exact in TF32). The forward saves S0 transposed, so the
// staged checkpoint is itself the shared-memory A operand S0^T; it is rounded
// to TF32 in place after sum_v Gd * S0 has been taken from it in FP32. Gd is
// read by the tensor core at TF32 (truncated); Gd^T W^T adds the product of
// Gd^T's truncated-away low part, so it is split TF32 on both sides. dO W^T
// (dO exact in TF32, W split) also runs on the tensor core. The first group
// (dW first, then Gd^T W^T and dO W^T) runs while warps 0-3 solve for E; the
// dO half of the adjoint update follows it once warps 4-7 have stored the
// (scale q^ gamma, -k^ gamma) tile; the second group, once dV is in place, is
// S0^T [dO; dV]^T as one N = 32 product (the staged checkpoint is read once)
// and the dV half of the update. The forward's FP32 A and B of each sub-chunk
// are reused. The next sub-chunk's
// token tiles, u and A/B are prefetched with cp.async into buffers freed
// earlier in the current sub-chunk; its state checkpoint (64 KiB, contiguous)
// arrives by four bulk copies that the MMA warp issues once the second group
// has finished reading S0. Operand tiles whose K dimension is the token are
// stored key-major (one float4 per 4 tokens of a row), so that a warp's
// stores fill whole core matrices without bank conflicts. The 16x16 intra-chunk
// products, the substitutions and the combination run in FP32 on CUDA cores:
// the decay gradient is a difference of nearly equal terms and needs them at
// full single precision. The gate, sigmoid and L2-norm backward are applied in
// the epilogue (flashinfer.kda_backward.recurrent_kda_backward, description:
// gradients with respect to the raw gate and raw beta logits, Q/K normalised
// with eps 1e-6).
#include <type_traits>

#include "kda_common.cuh"
#include "tc.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;             // compute threads
constexpr int kBlock = kThreads + 32;      // plus the MMA-issuing warp
constexpr int kTileF = kChunk * kLds;
constexpr int kDopLd = kDim + 8;          // padded row (BF16 elements) of the staged dO tile: a token
                                          // per lane then falls on different banks
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColG = 0;     // G, FP32 accumulator (lanes v, columns k)
constexpr uint32_t kColGT = 128;  // G^T, the same adjoint transposed (lanes k, columns v)
constexpr uint32_t kColGL = 256;  // Gd^T minus its TF32 truncation (the part the tensor core drops)
constexpr uint32_t kColDW = 384;  // Gd (k^ / gamma)^T : lanes v, 16 columns
constexpr uint32_t kColQ = 400;   // S0^T dO^T : lanes k, 16 columns
constexpr uint32_t kColR = 416;   // S0^T dV^T : lanes k, 16 columns (right after Q: one N = 32 product)
constexpr uint32_t kColWG = 432;  // Gd^T [W_hi; W_lo]^T : lanes k, 32 columns
constexpr uint32_t kColM1 = 464;  // dO [W_hi; W_lo]^T : lanes 0..15 (token i), 32 columns

struct BwdSmem {
  // chunk-start state as saved (ckpt_index layout, cp.async staging): S0^T,
  // the K-major A operand (rows k, K = v) of S0^T dO^T and S0^T dV^T once
  // rounded to TF32 in place
  unsigned char S0s[kDim * kDim * 4];
  unsigned char Ki[kChunk * kDim * 4];    // k^ / gamma rows t                  (K-major, K = 128)
  // Wt and dOU are contiguous: after the second MMA group they hold the
  // combination tiles (d q^, d k^, gauge term).
  unsigned char Wt[2][kChunk * kDim * 4]; // W rows t, TF32 hi then lo (one N = 32 operand)
  unsigned char dOU[32 * kDim * 4];       // rows 0..15 dO, 16..31 dV           (K-major, K = 128)
  unsigned char dOUv[kDim * 32 * 4];      // rows v: cols 0..15 dO, 16..31 dV (hi) (K-major, K = 32)
  unsigned char dUlo[kDim * kChunk * 4];  // rows v: dV lo part                 (K-major, K = 16)
  unsigned char QKT[kDim * 32 * 4];       // rows k: cols 0..15 scale q^g, 16..31 -k^g (K-major, K = 32)
  unsigned char Bsc[2][kChunk * kChunk * 4]; // scale B^T rows t (K = token j), TF32 hi / lo  (K = 16)
  float Pa[kTileF];                       // log decay, then gamma
  float Qtp[kTileF];                      // q^, then q^ gamma (FP32)
  float Ktp[kTileF];                      // k^, then k^ gamma (FP32)
  float Kip[kTileF];                      // k^ / gamma (FP32)
  float Up[kTileF];                       // u from the forward (cp.async staging)
  float DUp[kTileF];                      // E (dV = diag(beta) E)
  __nv_bfloat16 Sq[kChunk * kDim];        // q, k, g, do of the sub-chunk (cp.async staging)
  __nv_bfloat16 Sk[kChunk * kDim];
  __nv_bfloat16 Sg[kChunk * kDim];
  __nv_bfloat16 dOp[kChunk * kDopLd];
  float As[kChunk][kChunk];               // A and B^T of the sub-chunk, from the forward (cp.async
  float BsT[kChunk][kChunk];              // staging); As and BsT must stay contiguous
  float M1[kChunk][kChunk];               // dO W^T (W = diag(beta) U)
  float M2[kChunk][kChunk];               // dV W^T
  float M1T[kChunk][kChunk];
  float M2T[kChunk][kChunk];
  float bs[kChunk];
  float braw[kChunk];
  float dba[kChunk];                      // dbeta before the sigmoid derivative
  float gC[kDim];
  float rho0[2][kDim];                    // halves of sum_v Gd * S0
  float rho2[2][kDim];                    // halves of sum_i (k^/g)_i (W Gd)_i
  unsigned long long mbar[7];
  const float* ck_next[2];                // checkpoint of sub-chunk c - 1, for the MMA warp (slot (c - 1) & 1)
  uint32_t tmem_base;
};

// Barrier among the compute warps only (the MMA-issuing warp does not take part).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }
__device__ __forceinline__ bool csync_or(bool p) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, 1, %2, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)p), "n"(kThreads)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(kBlock, 1)
kda_bwd_kernel(const Problem P, const BwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int unit = P.order[blockIdx.x];
  const int64_t n = unit / P.Hv;
  const int64_t h = unit % P.Hv;
  const int64_t qh = h / P.r;
  const SeqInfo si = P.seq[n];
  const float s = P.scale;

  const int kl = 32 * (warp & 3) + lane;  // TMEM lane of this thread (key dim k, or value dim v)
  const int hv = warp >> 2;               // column half handled by this thread
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&sm.tmem_base), kTmemCols);
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 7; ++i) tc::mbar_init(tc::smem_u32(&sm.mbar[i]), i == 3 || i == 4 ? kThreads : i == 6 ? 128 : 1);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = sm.tmem_base;
  const uint32_t tl = tbase + lane_off;
  const uint32_t mbD = tc::smem_u32(&sm.mbar[0]), mb1 = tc::smem_u32(&sm.mbar[1]);
  const uint32_t mb2 = tc::smem_u32(&sm.mbar[2]);
  // compute -> MMA warp: each of the 256 compute threads arrives once its operand tiles are stored
  const uint32_t rdy1 = tc::smem_u32(&sm.mbar[3]), rdy2 = tc::smem_u32(&sm.mbar[4]);
  const uint32_t mbS = tc::smem_u32(&sm.mbar[5]);  // a sub-chunk's checkpoint has landed in S0s
  const uint32_t rdyQ = tc::smem_u32(&sm.mbar[6]);  // warps 4-7 -> MMA warp: the QKT tile is stored
  uint32_t ph = 0;  // every barrier completes once per sub-chunk
  bool ok = true;
  bool aborted = false;

  const int64_t nchunks = (si.len + kChunk - 1) / kChunk;
  const int ck_every = kCkTokens / kChunk;
  // staging mapping: row tid / 16, 8 consecutive columns
  const int srow = tid >> 4, scol = (tid & 15) * 8;
  __nv_bfloat16 nb = __float2bfloat16_rn(0.f);
  auto rows_of = [&](int64_t cc) { return (int)((si.len - cc * kChunk) < kChunk ? (si.len - cc * kChunk) : kChunk); };
  auto prefetch_qkg = [&](int64_t cc) {
    const int ntc = rows_of(cc);
    const bool okr = srow < ntc;
    const int64_t t = si.t0 + cc * kChunk + srow;
    tc::cp_async16(sm.Sq + srow * kDim + scol, okr ? P.q + (t * P.Hqk + qh) * kDim + scol : P.q, okr ? 16u : 0u);
    tc::cp_async16(sm.Sk + srow * kDim + scol, okr ? P.k + (t * P.Hqk + qh) * kDim + scol : P.k, okr ? 16u : 0u);
    tc::cp_async16(sm.Sg + srow * kDim + scol, okr ? P.g + (t * P.Hv + h) * kDim + scol : P.g, okr ? 16u : 0u);
    tc::cp_async_commit();
    if (tid < kChunk)
      nb = (tid < ntc) ? P.beta[(si.t0 + cc * kChunk + tid) * P.Hv + h] : __float2bfloat16_rn(0.f);
  };
  auto prefetch_late = [&](int64_t cc) {
    const int ntc = rows_of(cc);
    const bool okr = srow < ntc;
    const int64_t t = si.t0 + cc * kChunk + srow;
    tc::cp_async16(sm.dOp + srow * kDopLd + scol, okr ? a.d_o + (t * P.Hv + h) * kDim + scol : a.d_o, okr ? 16u : 0u);
    const float* us = okr ? P.utape + (t * P.Hv + h) * kDim + scol : P.utape;
    tc::cp_async16(sm.Up + srow * kLds + scol, us, okr ? 16u : 0u);
    tc::cp_async16(sm.Up + srow * kLds + scol + 4, okr ? us + 4 : us, okr ? 16u : 0u);
    if (tid < 128)
      tc::cp_async16(&sm.As[0][0] + tid * 4, P.abtape + ((si.ch_base + cc) * P.Hv + h) * 512 + tid * 4, 16u);
    tc::cp_async_commit();
  };
  // The checkpoint (64 KiB, contiguous) is staged by the copy engine: four bulk copies issued by
  // one thread, counted in transaction bytes on mbS.
  auto stage_state = [&](int64_t cc) {
    const float* src = P.ckpt + ((si.ck_base + cc / ck_every) * P.Hv + h) * kDim * kDim;
    tc::mbar_arrive_expect_tx(mbS, (uint32_t)(kDim * kDim * 4));
#pragma unroll
    for (int i = 0; i < 4; ++i) tc::bulk_g2s(tc::smem_u32(sm.S0s + i * 16384), src + i * 4096, 16384u, mbS);
  };

  if (warp == kThreads / 32) {
    // The MMA-issuing warp: one elected lane issues both groups of every
    // sub-chunk once the compute warps signal that the operands are in place,
    // so no compute warp is held by the tensor pipe's queue.
    if (tc::elect_one()) {
      uint32_t mph = 0;
      // Base descriptors of the operand tiles; K-step st of a tile adds 16 * st (256 bytes) to the
      // address field, and step st of the S0^T tile 256 * st. They are made opaque once per
      // sub-chunk, so that ptxas forms each step's descriptor with one add next to its MMA
      // instead of hoisting every (tile, step) descriptor out of the loop into registers.
      const uint64_t kKi = tc::kdesc(tc::smem_u32(sm.Ki), 0, kDim), kS0 = tc::sdesc(tc::smem_u32(sm.S0s), 2048u, 128u);
      const uint64_t kDou = tc::kdesc(tc::smem_u32(sm.dOU), 0, kDim);
      const uint64_t kWt = tc::kdesc(tc::smem_u32(sm.Wt[0]), 0, kDim), kDouv = tc::kdesc(tc::smem_u32(sm.dOUv), 0, 32);
      const uint64_t kBs0 = tc::kdesc(tc::smem_u32(sm.Bsc[0]), 0, kChunk), kBs1 = tc::kdesc(tc::smem_u32(sm.Bsc[1]), 0, kChunk);
      const uint64_t kQkt = tc::kdesc(tc::smem_u32(sm.QKT), 0, 32), kDul = tc::kdesc(tc::smem_u32(sm.dUlo), 0, kChunk);
      for (int64_t c = nchunks - 1; c >= 0; --c) {
        if (!tc::mbar_wait(rdy1, mph)) break;
        tc::fence_after();
        uint64_t dKi = kKi, dS0 = kS0, dDou = kDou, dWt = kWt, dDouv = kDouv, dBs0 = kBs0, dBs1 = kBs1,
                 dQkt = kQkt, dDul = kDul;
        asm volatile("" : "+l"(dKi), "+l"(dS0), "+l"(dDou), "+l"(dWt));
        asm volatile("" : "+l"(dDouv), "+l"(dBs0), "+l"(dBs1), "+l"(dQkt), "+l"(dDul));
        {
          const uint32_t i16 = tc::idesc_tf32(128, 16), i32 = tc::idesc_tf32(128, 32);
#pragma unroll
          for (int st = 0; st < kDim / 8; ++st)
            tc::mma_ts(tbase + kColDW, tbase + kColG + 8 * st, dKi + 16u * st, i16, st > 0);
#pragma unroll
          for (int st = 0; st < 2; ++st)  // dO (rows v, exact in TF32) with scale B^T hi and lo
            tc::mma_ss(tbase + kColDW, dDouv + 16u * st, dBs0 + 16u * st, i16, 1);
#pragma unroll
          for (int st = 0; st < 2; ++st)
            tc::mma_ss(tbase + kColDW, dDouv + 16u * st, dBs1 + 16u * st, i16, 1);
          tc::mma_commit(mbD);
#pragma unroll
          for (int st = 0; st < kDim / 8; ++st)
            tc::mma_ts(tbase + kColWG, tbase + kColGT + 8 * st, dWt + 16u * st, i32, st > 0);
#pragma unroll
          for (int st = 0; st < kDim / 8; ++st)  // the low part of Gd^T with [W_hi; W_lo]
            tc::mma_ts(tbase + kColWG, tbase + kColGL + 8 * st, dWt + 16u * st, i32, 1);
          // dO W^T with M = 64: the A tile is read as 64 rows from dOU on, of which rows 0..15
          // are dO and land in TMEM lanes 0..15 (M = 64 puts rows 16 w .. 16 w + 15 in lanes
          // 32 w .. 32 w + 15); the other rows only fill lanes that are never read
#pragma unroll
          for (int st = 0; st < kDim / 8; ++st)
            tc::mma_ss(tbase + kColM1, dDou + 16u * st, dWt + 16u * st, tc::idesc_tf32(64, 32), st > 0);
          tc::mma_commit(mb1);
        }
        // the dO half of the adjoint update, once QKT is stored and the first group (which reads G
        // and G^T) has completed; the second group's commit covers it
        if (!tc::mbar_wait(rdyQ, mph) || !tc::mbar_wait(mb1, mph)) break;
        tc::fence_after();
        {
          const uint32_t i128 = tc::idesc_tf32(128, 128);
#pragma unroll
          for (int st = 0; st < 2; ++st) {
            tc::mma_ss(tbase + kColGT, dQkt + 16u * st, dDouv + 16u * st, i128, 1);
            tc::mma_ss(tbase + kColG, dDouv + 16u * st, dQkt + 16u * st, i128, 1);
          }
        }
        if (!tc::mbar_wait(rdy2, mph)) break;
        tc::fence_after();
        {
          const uint32_t i32 = tc::idesc_tf32(128, 32), i128 = tc::idesc_tf32(128, 128);
#pragma unroll
          for (int st = 0; st < kDim / 8; ++st)  // S0^T [dO; dV]^T (dOU rows 0..31) into the Q and R columns
            tc::mma_ss(tbase + kColQ, dS0 + 256u * st, dDou + 16u * st, i32, st > 0);
#pragma unroll
          for (int st = 2; st < 4; ++st) {  // the dV half (the dO half was issued after the first group)
            tc::mma_ss(tbase + kColGT, dQkt + 16u * st, dDouv + 16u * st, i128, 1);
            tc::mma_ss(tbase + kColG, dDouv + 16u * st, dQkt + 16u * st, i128, 1);
          }
#pragma unroll
          for (int st = 0; st < 2; ++st)  // -k^g (columns 16..31 of QKT) with the dV lo part, for G^T only:
            // G (lanes v) is only ever read truncated to TF32, as the A operand of Gd (k^/g)^T
            tc::mma_ss(tbase + kColGT, dQkt + 16u * (2 + st), dDul + 16u * st, i128, 1);
          tc::mma_commit(mb2);
        }
        // once this group has completed, S0s is free: stage the next (earlier) sub-chunk's
        // checkpoint, whose address the compute warps left in shared memory
        if (c > 0) {
          if (!tc::mbar_wait(mb2, mph)) break;
          const float* src;
          asm volatile("ld.volatile.shared.u64 %0, [%1];" : "=l"(src) : "r"(tc::smem_u32(&sm.ck_next[(c - 1) & 1])));
          tc::mbar_arrive_expect_tx(mbS, (uint32_t)(kDim * kDim * 4));
#pragma unroll
          for (int i = 0; i < 4; ++i) tc::bulk_g2s(tc::smem_u32(sm.S0s + i * 16384), src + i * 4096, 16384u, mbS);
        }
        mph ^= 1;
      }
    }
    __syncwarp();
  } else {
    // G <- dfinal_state (lanes v) and G^T (lanes k)
    {
      const float* src = a.d_hT + (n * P.Hv + h) * kDim * kDim;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        const int c0 = 64 * hv + 16 * q;
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = src[(c0 + j) * kDim + kl];
        tc::tmem_st16(tl + kColGT + c0, x);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 y = *reinterpret_cast<const float4*>(src + kl * kDim + c0 + 4 * m);
          x[4 * m] = y.x; x[4 * m + 1] = y.y; x[4 * m + 2] = y.z; x[4 * m + 3] = y.w;
        }
        tc::tmem_st16(tl + kColG + c0, x);
      }
      tc::tmem_wait_st();
    }
    prefetch_qkg(nchunks - 1);
    prefetch_late(nchunks - 1);
    if (tid == 0) stage_state(nchunks - 1);
    int64_t staged = 1;  // checkpoint bulk copies issued; each completes one phase of mbS

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
    float* cmb = reinterpret_cast<float*>(sm.Wt[0]);  // d q^, d k^, gauge / da tiles (after the MMAs)
    const int ot = tid & 15, oq = tid >> 4;           // operand-tile mapping: token ot, quads oq, oq + 16

    // P0, the prologue of sub-chunk cc (token row ti, columns c8..c8+7): L2 norm, gate,
    // sigmoid beta. It runs in the same barrier interval as the previous (later) sub-chunk's
    // epilogue, with which it shares no data, so the two latency chains interleave.
    float qhat[8], khat[8], zz[8], rq = 0.f, rk = 0.f;
    auto prologue = [&](int64_t cc) {
      const int ntc = rows_of(cc);
        {
          float qv[8], kv[8], gv[8];
          const bool valid = ti < ntc;
          unpack_bf16x8(*reinterpret_cast<const uint4*>(sm.Sq + ti * kDim + c8), qv);
          unpack_bf16x8(*reinterpret_cast<const uint4*>(sm.Sk + ti * kDim + c8), kv);
          unpack_bf16x8(*reinterpret_cast<const uint4*>(sm.Sg + ti * kDim + c8), gv);
          float sq = 0.f, sk = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) { sq += qv[e] * qv[e]; sk += kv[e] * kv[e]; }
          sq = row16_sum(sq);
          sk = row16_sum(sk);
          rq = valid ? inv_norm_of(sq) : 0.f;
          rk = valid ? inv_norm_of(sk) : 0.f;
          float la[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            qhat[e] = qv[e] * rq;
            khat[e] = kv[e] * rk;
            zz[e] = ea * (gv[e] + dtb[e]);
            la[e] = valid ? log_decay_of(P.lb, zz[e]) : 0.f;
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int o = 4 * hh;
            *reinterpret_cast<float4*>(sm.Qtp + ti * kLds + c8 + o) = make_float4(qhat[o], qhat[o + 1], qhat[o + 2], qhat[o + 3]);
            *reinterpret_cast<float4*>(sm.Ktp + ti * kLds + c8 + o) = make_float4(khat[o], khat[o + 1], khat[o + 2], khat[o + 3]);
            *reinterpret_cast<float4*>(sm.Pa + ti * kLds + c8 + o) = make_float4(la[o], la[o + 1], la[o + 2], la[o + 3]);
          }
          if (tid < kChunk) {
            const float bl = __bfloat162float(nb);
            sm.braw[tid] = bl;
            sm.bs[tid] = (tid < ntc) ? sigmoid_of(bl) : 0.f;
          }
        }
    };
    tc::cp_async_wait<1>();  // q, k, g of the first sub-chunk (dO/u/A/B may be in flight)
    csync();
    prologue(nchunks - 1);
    for (int64_t c = nchunks - 1; c >= 0; --c) {
      const int64_t tc0 = si.t0 + c * kChunk;
      const int nt = rows_of(c);
      csync();  // the prologue of this sub-chunk is in place
      // ---- P1: cumulative decay (one key column per thread); the next q, k, g are fetched meanwhile
      if (c > 0) {
        prefetch_qkg(c - 1);
        // two slots: the MMA warp reads this one after the group-2 completion of sub-chunk c, and it
        // is written again two sub-chunks later, after that warp has issued sub-chunk c - 1's work
        if (tid == 0) sm.ck_next[(c - 1) & 1] = P.ckpt + ((si.ck_base + (c - 1) / ck_every) * P.Hv + h) * kDim * kDim;
      }
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
      if (c > 0) tc::cp_async_wait<1>();  // dO, u and A/B of this sub-chunk (the next q, k, g may be in flight)
      else tc::cp_async_wait_all();
      ok = ok && tc::mbar_wait(mbS, ph);  // and its checkpoint
      csync();
      // ---- P2: decay of the adjoint, G <- G diag(gamma_C) (lanes v) and G^T <- diag(gamma_C) G^T
      // (lanes k), with sum_v Gd * S0 from the FP32 checkpoint, the low part of Gd^T for the
      // split Gd^T W^T, and S0 rounded to TF32 in place for the tensor core; then the operand tiles
      {
        const float gck = sm.gC[kl];
        float4 racc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
        for (int q = 0; q < 4; ++q) {
          const int c0 = 64 * hv + 16 * q;
          float g16[16], x16[16];
          tc::tmem_ld16_nowait(tl + kColGT + c0, g16);
          tc::tmem_ld16_nowait(tl + kColG + c0, x16);
          float4 s4[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) s4[b] = *reinterpret_cast<const float4*>(sm.S0s + ckpt_index(c0 + 4 * b, kl) * 4);
          tc::tmem_wait_ld2(g16, x16);
          float lo16[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            g16[j] *= gck;
            lo16[j] = g16[j] - __uint_as_float(__float_as_uint(g16[j]) & 0xFFFFE000u);
          }
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float4 y = *reinterpret_cast<const float4*>(sm.gC + c0 + 4 * m);
            x16[4 * m] *= y.x; x16[4 * m + 1] *= y.y; x16[4 * m + 2] *= y.z; x16[4 * m + 3] *= y.w;
          }
          tc::tmem_st16(tl + kColGT + c0, g16);
          tc::tmem_st16(tl + kColGL + c0, lo16);
          tc::tmem_st16(tl + kColG + c0, x16);
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            fma4(racc, make_float4(g16[4 * b], g16[4 * b + 1], g16[4 * b + 2], g16[4 * b + 3]), s4[b]);
            *reinterpret_cast<float4*>(sm.S0s + ckpt_index(c0 + 4 * b, kl) * 4) =
                make_float4(tc::round_tf32(s4[b].x), tc::round_tf32(s4[b].y), tc::round_tf32(s4[b].z),
                            tc::round_tf32(s4[b].w));
          }
        }
        sm.rho0[hv][kl] = hsum4(racc);
      }
#pragma unroll
      for (int rep = 0; rep < 2; ++rep) {
        const int k0 = 4 * (oq + 16 * rep);
        const float4 qh4 = *reinterpret_cast<const float4*>(sm.Qtp + ot * kLds + k0);
        const float4 kh4 = *reinterpret_cast<const float4*>(sm.Ktp + ot * kLds + k0);
        const float4 g4 = *reinterpret_cast<const float4*>(sm.Pa + ot * kLds + k0);
        const float4 u4 = *reinterpret_cast<const float4*>(sm.Up + ot * kLds + k0);
        const float qa[4] = {qh4.x, qh4.y, qh4.z, qh4.w}, ka[4] = {kh4.x, kh4.y, kh4.z, kh4.w};
        const float ga[4] = {g4.x, g4.y, g4.z, g4.w}, ua[4] = {u4.x, u4.y, u4.z, u4.w};
        const float bt = sm.bs[ot];
        float kt[4], qt[4], ki[4], whi[4], wlo[4], dof[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float inv = __fdividef(1.0f, ga[e]);  // gamma is in [e^-80, 1]
          kt[e] = ka[e] * ga[e];
          qt[e] = qa[e] * ga[e];
          ki[e] = ka[e] * inv;
          const float w = bt * ua[e];
          whi[e] = tc::round_tf32(w);
          wlo[e] = tc::round_tf32(w - whi[e]);
          dof[e] = __bfloat162float(sm.dOp[ot * kDopLd + k0 + e]);
        }
        *reinterpret_cast<float4*>(sm.Ktp + ot * kLds + k0) = make_float4(kt[0], kt[1], kt[2], kt[3]);
        *reinterpret_cast<float4*>(sm.Qtp + ot * kLds + k0) = make_float4(qt[0], qt[1], qt[2], qt[3]);
        *reinterpret_cast<float4*>(sm.Kip + ot * kLds + k0) = make_float4(ki[0], ki[1], ki[2], ki[3]);
        *reinterpret_cast<float4*>(sm.Ki + tc::kmaj(ot, k0, kDim)) =
            make_float4(tc::round_tf32(ki[0]), tc::round_tf32(ki[1]), tc::round_tf32(ki[2]), tc::round_tf32(ki[3]));
        *reinterpret_cast<float4*>(sm.Wt[0] + tc::kmaj(ot, k0, kDim)) = make_float4(whi[0], whi[1], whi[2], whi[3]);
        *reinterpret_cast<float4*>(sm.Wt[1] + tc::kmaj(ot, k0, kDim)) = make_float4(wlo[0], wlo[1], wlo[2], wlo[3]);
        *reinterpret_cast<float4*>(sm.dOU + tc::kmaj(ot, k0, kDim)) = make_float4(dof[0], dof[1], dof[2], dof[3]);
      }
      {  // dO as rows v (K = token) for dO^T B and the adjoint updates: value dim v, 8 tokens, so that
         // each float4 store covers 4 tokens and a warp's stores cover whole 8 x 4 core matrices
        const int v = tid & (kDim - 1), t0 = 8 * (tid >> 7);
        float d8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) d8[j] = __bfloat162float(sm.dOp[(t0 + j) * kDopLd + v]);
        *reinterpret_cast<float4*>(sm.dOUv + tc::kmaj(v, t0, 32)) = make_float4(d8[0], d8[1], d8[2], d8[3]);
        *reinterpret_cast<float4*>(sm.dOUv + tc::kmaj(v, t0 + 4, 32)) = make_float4(d8[4], d8[5], d8[6], d8[7]);
      }
      {  // scale B^T as rows t, K = j (B[j][t] is BsT[t][j]), split into TF32 hi + lo
        const int t = tid >> 4, j = tid & 15;
        const float x = s * sm.BsT[t][j];
        const float hi = tc::round_tf32(x);
        *reinterpret_cast<float*>(sm.Bsc[0] + tc::kmaj(t, j, kChunk)) = hi;
        *reinterpret_cast<float*>(sm.Bsc[1] + tc::kmaj(t, j, kChunk)) = tc::round_tf32(x - hi);
      }
      tc::tmem_wait_st();
      tc::fence_async_smem();
      tc::fence_before();
      // ---- MMA group 1 (issued by the MMA warp): dW = Gd (k^/g)^T + scale dO^T B first (the dV
      // chain needs it), then Gd^T W^T and dO W^T; every compute thread arrives once its own operand
      // tiles are written (no CTA barrier)
      tc::mbar_arrive(rdy1);
      if (warp >= 4) {
        ok = ok && tc::mbar_wait(rdy1, ph);  // QKT below reads every thread's q^g and k^g rows
        {  // QKT, rows k: columns 0..15 scale q^g, 16..31 -k^g (the adjoint updates); once it is stored,
           // the MMA warp issues the dO half of the update after the first group
          const int k = tid - 128;
#pragma unroll
          for (int t4 = 0; t4 < kChunk; t4 += 4) {
            float qv[4], kv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              qv[j] = tc::round_tf32(s * sm.Qtp[(t4 + j) * kLds + k]);
              kv[j] = tc::round_tf32(-sm.Ktp[(t4 + j) * kLds + k]);
            }
            *reinterpret_cast<float4*>(sm.QKT + tc::kmaj(k, t4, 32)) = make_float4(qv[0], qv[1], qv[2], qv[3]);
            *reinterpret_cast<float4*>(sm.QKT + tc::kmaj(k, 16 + t4, 32)) = make_float4(kv[0], kv[1], kv[2], kv[3]);
          }
          tc::fence_async_smem();
          tc::fence_before();
          tc::mbar_arrive(rdyQ);
        }
        // dO W^T = dO (W_hi + W_lo)^T from tensor memory (dO is exact in TF32)
        ok = ok && tc::mbar_wait(mb1, ph);
        tc::fence_after();
        if (warp == 4) {
          float hi16[16], lo16[16];
          tc::tmem_ld16_nowait(tl + kColM1, hi16);
          tc::tmem_ld16_nowait(tl + kColM1 + 16, lo16);
          tc::tmem_wait_ld2(hi16, lo16);
          if (lane < kChunk) {
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
              const float m = hi16[j] + lo16[j];
              sm.M1T[j][lane] = m;
              hi16[j] = m;
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              *reinterpret_cast<float4*>(&sm.M1[lane][4 * q4]) =
                  make_float4(hi16[4 * q4], hi16[4 * q4 + 1], hi16[4 * q4 + 2], hi16[4 * q4 + 3]);
          }
        }
      } else {
        ok = ok && tc::mbar_wait(mbD, ph);
        tc::fence_after();
        // ---- P5: per value column (warps 0-3): dW, E, dV
        const int vv = kl;
        float acc[kChunk], ev[kChunk];
        tc::tmem_ld16(tl + kColDW, acc);  // dW (rows v)
        // E solves (I + A^T diag(beta)) E = dW, last row first (right-looking)
        float bsv[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) bsv[i] = sm.bs[i];
#pragma unroll
        for (int i = kChunk - 1; i >= 0; --i) {
          const float ei = acc[i];
          ev[i] = ei;
          const float du = bsv[i] * ei;
          acc[i] = du;  // keep dV in place
          float arow[kChunk];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const float4 x = *reinterpret_cast<const float4*>(&sm.As[i][4 * q4]);
            arow[4 * q4] = x.x; arow[4 * q4 + 1] = x.y; arow[4 * q4 + 2] = x.z; arow[4 * q4 + 3] = x.w;
          }
#pragma unroll
          for (int m = 0; m < i; ++m) acc[m] = fmaf(-arow[m], du, acc[m]);
        }
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
          sm.DUp[i * kLds + vv] = ev[i];  // E; dV = diag(beta) E
        }
#pragma unroll
        for (int t4 = 0; t4 < kChunk; t4 += 4) {  // dv: lane (quad base + j) writes token t4 + j
          float y[4] = {acc[t4], acc[t4 + 1], acc[t4 + 2], acc[t4 + 3]};
          tc::quad_transpose(y, lane);
          const int t = t4 + (lane & 3);
          if (t < nt) {
            __nv_bfloat162 p0 = __floats2bfloat162_rn(y[0], y[1]), p1 = __floats2bfloat162_rn(y[2], y[3]);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&p0);
            pk.y = *reinterpret_cast<uint32_t*>(&p1);
            *reinterpret_cast<uint2*>(a.dv + ((tc0 + t) * P.Hv + h) * kDim + (vv & ~3)) = pk;
          }
        }
#pragma unroll
        for (int a4 = 0; a4 < 4; ++a4) {
          float hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi[e] = tc::round_tf32(acc[4 * a4 + e]);
            lo[e] = tc::round_tf32(acc[4 * a4 + e] - hi[e]);
          }
          *reinterpret_cast<float4*>(sm.dOUv + tc::kmaj(vv, 16 + 4 * a4, 32)) = make_float4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<float4*>(sm.dUlo + tc::kmaj(vv, 4 * a4, kChunk)) = make_float4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      tc::fence_before();
      csync();
      // dV rows (beta E) of the S0^T dV^T operand (token ot, quads oq and oq + 16)
#pragma unroll
      for (int rep = 0; rep < 2; ++rep) {
        const int k0 = 4 * (oq + 16 * rep);
        const float4 d4 = *reinterpret_cast<const float4*>(sm.DUp + ot * kLds + k0);
        const float bt = sm.bs[ot];
        *reinterpret_cast<float4*>(sm.dOU + tc::kmaj(16 + ot, k0, kDim)) =
            make_float4(tc::round_tf32(bt * d4.x), tc::round_tf32(bt * d4.y), tc::round_tf32(bt * d4.z),
                        tc::round_tf32(bt * d4.w));
      }
      tc::fence_async_smem();
      tc::fence_before();
      // ---- MMA group 2 (issued by the MMA warp): S0^T [dO; dV]^T and the dV half of the adjoint
      // update of G and G^T; every compute thread arrives once its own operand tiles are written (no
      // CTA barrier)
      tc::mbar_arrive(rdy2);
      {  // dV W^T in FP32 as diag(beta) (E U^T) diag(beta): a warp takes a 4 (i) x 8 (j) block of
         // entries, a lane a 2 x 4 block over an eighth o of the value columns (float4 groups
         // 4 o + 32 m), so that each 16-byte load feeds 16 or 32 FMAs instead of 4 (the loop is bound
         // by shared-memory wavefronts); an 8-lane phase reads 128 contiguous bytes of one row. A
         // reduce-scatter over the eight lanes of a block (three shuffle rounds) leaves entry o in
         // lane o; the diagonal of E U^T is dbeta. Only the strict lower triangle of M2 is read
         // (by the combination), so 12 of the 32 blocks, wholly above the diagonal, load nothing
        constexpr int BI = 2, BJ = 4, KS = BI * BJ;
        const int o = lane % KS, g = lane / KS;
        const int i0 = 4 * (warp >> 1) + BI * (g / (8 / BJ)), j0 = 8 * (warp & 1) + BJ * (g % (8 / BJ));
        const float* e0 = sm.DUp + i0 * kLds + 4 * o;
        const float* u0 = sm.Up + j0 * kLds + 4 * o;
        float ac[KS];
#pragma unroll
        for (int e = 0; e < KS; ++e) ac[e] = 0.f;
        // blocks wholly above the diagonal (i0 + 1 < j0) are not needed: their lanes keep zeros
        const int mend = i0 + BI - 1 >= j0 ? 32 / KS : 0;
#pragma unroll 2
        for (int m = 0; m < mend; ++m) {
          float4 a[BI], x[BJ];
#pragma unroll
          for (int ii = 0; ii < BI; ++ii) a[ii] = *reinterpret_cast<const float4*>(e0 + ii * kLds + 4 * KS * m);
#pragma unroll
          for (int jj = 0; jj < BJ; ++jj) x[jj] = *reinterpret_cast<const float4*>(u0 + jj * kLds + 4 * KS * m);
#pragma unroll
          for (int ii = 0; ii < BI; ++ii)
#pragma unroll
            for (int jj = 0; jj < BJ; ++jj) {
              float& r = ac[BJ * ii + jj];
              r = fmaf(a[ii].w, x[jj].w, fmaf(a[ii].z, x[jj].z, fmaf(a[ii].y, x[jj].y, fmaf(a[ii].x, x[jj].x, r))));
            }
        }
#pragma unroll
        for (int w = KS / 2; w >= 1; w >>= 1) {
          const bool up = o & w;
#pragma unroll
          for (int r = 0; r < w; ++r) {
            const float mine = up ? ac[w + r] : ac[r], oth = up ? ac[r] : ac[w + r];
            ac[r] = mine + __shfl_xor_sync(0xffffffffu, oth, w);
          }
        }
        const float acc = ac[0];  // sum_v E_i U_j
        const int i = i0 + o / BJ, j = j0 + o % BJ;
        if (i == j) sm.dba[i] = acc;  // dbeta_i = E_i . U_i (before the sigmoid derivative)
        const float m2 = acc * sm.bs[i] * sm.bs[j];
        sm.M2[i][j] = m2;
        sm.M2T[j][i] = m2;
      }
      ok = ok && tc::mbar_wait(mb1, ph);
      ok = ok && tc::mbar_wait(mb2, ph);
      tc::fence_after();
      if (csync_or(!ok)) { aborted = true; break; }
      if (c > 0) {  // dO, u, A/B and S0 of this sub-chunk are no longer read
        prefetch_late(c - 1);
        ++staged;  // the MMA warp stages the checkpoint of c - 1
      }
      // ---- P7: assemble d q^, d k^ and the gauge term (lane k, rows i0 .. i0 + 7 with
      // i0 = 8 hv a compile-time constant, so the triangular masks drop whole terms)
      {
        auto combine = [&](auto i0c) {
          constexpr int i0 = decltype(i0c)::value;
          float* dQh = cmb;
          float* dKh = cmb + kTileF;
          float* tv = cmb + 2 * kTileF;
          float qd[8], rd[8], wh[8], wl[8];
          tc::tmem_ld8(tl + kColQ + i0, qd);
          tc::tmem_ld8(tl + kColR + i0, rd);
          tc::tmem_ld8(tl + kColWG + i0, wh);
          tc::tmem_ld8(tl + kColWG + 16 + i0, wl);
          const int k = kl;
          float kic[kChunk], qtc[kChunk], ktc[kChunk];
#pragma unroll
          for (int j = 0; j < kChunk; ++j) {
            kic[j] = sm.Kip[j * kLds + k];
            qtc[j] = sm.Qtp[j * kLds + k];
            ktc[j] = sm.Ktp[j * kLds + k];
          }
          float rp = 0.f;
#pragma unroll
          for (int ii = 0; ii < 8; ++ii) {
            const int i = i0 + ii;
            const float gam = sm.Pa[i * kLds + k];
            const float inv = __fdividef(1.0f, gam);
            const float wg = wh[ii] + wl[ii];
            float pq = qd[ii], pr = rd[ii], pw = wg;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              if (4 * q4 <= i) {  // tril(M1) and stril(M2) rows
                const float4 a4 = *reinterpret_cast<const float4*>(&sm.M1[i][4 * q4]);
                const float4 b4 = *reinterpret_cast<const float4*>(&sm.M2[i][4 * q4]);
                const float m1r[4] = {a4.x, a4.y, a4.z, a4.w}, m2r[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int j = 4 * q4 + e;
                  if (j <= i) pq = fmaf(m1r[e], kic[j], pq);
                  if (j < i) pr = fmaf(m2r[e], kic[j], pr);
                }
              }
              if (4 * q4 + 3 >= i) {  // triu(M1^T) and striu(M2^T) rows
                const float4 c4 = *reinterpret_cast<const float4*>(&sm.M1T[i][4 * q4]);
                const float4 d4 = *reinterpret_cast<const float4*>(&sm.M2T[i][4 * q4]);
                const float m1c[4] = {c4.x, c4.y, c4.z, c4.w}, m2c[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int j = 4 * q4 + e;
                  if (j >= i) pw = fmaf(s * m1c[e], qtc[j], pw);
                  if (j > i) pw = fmaf(-m2c[e], ktc[j], pw);
                }
              }
            }
            rp = fmaf(kic[i], wg, rp);
            const float dq_ = s * gam * pq;
            const float dkr = -gam * pr;
            const float dkw = inv * pw;
            dQh[i * kLds + k] = dq_;
            dKh[i * kLds + k] = dkr + dkw;
            tv[i * kLds + k] = qtc[i] * inv * dq_ + ktc[i] * inv * (dkr - dkw);
          }
          sm.rho2[i0 / 8][k] = rp;
        };
        if (hv == 0) combine(std::integral_constant<int, 0>{});
        else combine(std::integral_constant<int, 8>{});
      }
      csync();
      // ---- P8: da = rho + reverse cumulative sum of the gauge term within the sub-chunk
      if (tid < kDim) {
        float* tv = cmb + 2 * kTileF;
        float run = sm.rho0[0][tid] + sm.rho0[1][tid] + sm.rho2[0][tid] + sm.rho2[1][tid];
#pragma unroll
        for (int i = kChunk - 1; i >= 0; --i) {
          run += tv[i * kLds + tid];
          tv[i * kLds + tid] = run;
        }
      }
      if (c > 0) tc::cp_async_wait<1>();  // q, k, g of the next sub-chunk, for its prologue below
      csync();
      // ---- P9: epilogue: gate / sigmoid / L2-norm backward and stores
      {
        const float* dQh = cmb;
        const float* dKh = cmb + kTileF;
        const float* da = cmb + 2 * kTileF;
        const bool valid = ti < nt;
        const int64_t t = tc0 + ti;
        float dg8[8], dq8[8], dk8[8], da8[8];
        float pq = 0.f, pk = 0.f;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int o = ti * kLds + c8 + 4 * hh;
          const float4 x = *reinterpret_cast<const float4*>(da + o);
          const float4 y = *reinterpret_cast<const float4*>(dQh + o);
          const float4 z = *reinterpret_cast<const float4*>(dKh + o);
          da8[4 * hh] = x.x; da8[4 * hh + 1] = x.y; da8[4 * hh + 2] = x.z; da8[4 * hh + 3] = x.w;
          dq8[4 * hh] = y.x; dq8[4 * hh + 1] = y.y; dq8[4 * hh + 2] = y.z; dq8[4 * hh + 3] = y.w;
          dk8[4 * hh] = z.x; dk8[4 * hh + 1] = z.y; dk8[4 * hh + 2] = z.z; dk8[4 * hh + 3] = z.w;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          // sigmoid'(z) = sigmoid(z) sigmoid(-z) = e / (1 + e)^2 with e = exp(-|z|) (no cancellation)
          const float ex = __expf(-fabsf(zz[e]));
          const float den = __fdividef(1.0f, 1.0f + ex);
          const float dz = valid ? da8[e] * P.lb * ex * den * den : 0.f;
          dg8[e] = dz * ea;
          ddt_acc[e] += dg8[e];
          dA_acc += dz * zz[e];
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
          const float bn = sigmoid_of(-sm.braw[tid]);
          a.dbeta[(tc0 + tid) * P.Hv + h] = __float2bfloat16_rn(sm.dba[tid] * sm.bs[tid] * bn);
        }
      }
      prologue(c - 1);  // also after the last sub-chunk (harmless, unused): no branch between it and the epilogue
      ph ^= 1;
      tc::fence_before();
    }
    tc::cp_async_wait_all();
    // no bulk copy may still be landing when the block exits (normally every one has been waited for)
    if (tid == 0) tc::mbar_wait(mbS, (uint32_t)((staged - 1) & 1));
    csync();
    if (!aborted) {
      // dinitial_state = G (from its transposed copy, for coalesced stores)
      float* dst = a.dh0 + (n * P.Hv + h) * kDim * kDim;
      tc::fence_after();
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        const int v0 = 64 * hv + 16 * q;
        float x[16];
        tc::tmem_ld16(tl + kColGT + v0, x);
#pragma unroll
        for (int j = 0; j < 16; ++j) dst[(v0 + j) * kDim + kl] = x[j];
      }
      // per-unit parameter-gradient partials, reduced in a fixed order
      float* red = sm.Qtp;  // [16 rows][128] + [256]: spans Qtp and Ktp
#pragma unroll
      for (int e = 0; e < 8; ++e) red[ti * kDim + c8 + e] = ddt_acc[e];
      red[kChunk * kDim + tid] = dA_acc;
      csync();
      float* pp = a.par_part + (int64_t)unit * kParStride;
      if (tid < kDim) {
        float acc = 0.f;
        for (int i = 0; i < kChunk; ++i) acc += red[i * kDim + tid];
        pp[tid] = acc;
      }
      if (tid == 0) {
        float acc = 0.f;
        for (int i = 0; i < kThreads; ++i) acc += red[kChunk * kDim + i];
        pp[kDim] = acc;
      }
    } else if (tid == 0) {
      atomicOr(P.status, 1);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::tmem_dealloc(tbase, kTmemCols);
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
    const float r = inv_norm_of(ss);
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
  kda_bwd_kernel<<<(unsigned)units, kBlock, smem, s>>>(P, a);
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
