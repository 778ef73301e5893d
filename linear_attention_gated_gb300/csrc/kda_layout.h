// kda_layout.h -- byte layout of the saved-forward context (host side). One
// definition serves every entry point that carves it out of device memory:
// kda_fwd / kda_bwd and kda_bwd_standalone (a caller-owned workspace) and
// kda_bwd_noalloc (the library's fixed scratch array).
#pragma once

#include <cstddef>
#include <cstdint>

#include "kda_common.cuh"

namespace kda {

constexpr size_t kCtxAlign = 256;
inline size_t ctx_align_up(size_t x) { return (x + kCtxAlign - 1) / kCtxAlign * kCtxAlign; }

// State checkpoints and sub-chunks of one sequence of `len` tokens.
__host__ __device__ inline int64_t checkpoints_of(int64_t len) { return (len + kCkTokens - 1) / kCkTokens; }
__host__ __device__ inline int64_t subchunks_of(int64_t len) { return (len + kChunk - 1) / kChunk; }

struct CtxCounts {
  int64_t N = 0, Ttot = 0, Hqk = 0, Hv = 0, n_ck = 0, n_ch = 0;
};

// Offsets (bytes, each 256-byte aligned) of the context's regions.
struct CtxLayout {
  size_t order = 0, seq = 0, ckpt = 0, utape = 0, abtape = 0, dqk = 0, par = 0, status = 0, total = 0;
};

inline CtxLayout context_layout(const CtxCounts& c) {
  CtxLayout L;
  const int64_t units = c.N * c.Hv;
  size_t off = 0;
  L.order = off; off = ctx_align_up(off + sizeof(int32_t) * (size_t)units);
  L.seq = off;   off = ctx_align_up(off + sizeof(SeqInfo) * (size_t)c.N);
  L.ckpt = off;  off = ctx_align_up(off + sizeof(float) * (size_t)c.n_ck * c.Hv * kDim * kDim);
  L.utape = off; off = ctx_align_up(off + sizeof(float) * (size_t)c.Ttot * c.Hv * kDim);
  L.abtape = off; off = ctx_align_up(off + sizeof(float) * (size_t)c.n_ch * c.Hv * 2 * kChunk * kChunk);
  L.dqk = off;
  if (c.Hv != c.Hqk) off = ctx_align_up(off + sizeof(float) * (size_t)c.Ttot * c.Hv * 2 * kDim);
  L.par = off;   off = ctx_align_up(off + sizeof(float) * (size_t)units * kParStride);
  L.status = off; off = ctx_align_up(off + 16);
  L.total = off;
  return L;
}

}  // namespace kda
