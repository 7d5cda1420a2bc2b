// bwd_common.cuh -- index helpers shared by the backward kernels
// (attn_bwd.cu, attn_bwd128.cu): sequence bounds, tensor row offsets and
// workspace rows, and the plain bulk copy global -> shared memory.
#pragma once

#include "kernels.h"
#include "sm103.cuh"

namespace gqa {
namespace bwd {

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Workspace row of (sequence s, head h, position p).  Dense: s is the batch
// index and every head owns T_pad rows.  Packed: every head owns total_pad
// rows and sequence s starts at a 4-aligned base, 132 rows further apart than
// the tokens before it, so a 128-row tile never reaches the next sequence.
__device__ __forceinline__ long ws_row(const BwdArgs& a, int s, int tok0, int h, int p) {
  if (a.varlen) return (long)h * a.total_pad + (long)(((tok0 + 3) & ~3) + 132 * s) + p;
  return ((long)s * a.Hq + h) * a.T_pad + p;
}

__device__ __forceinline__ bool seq_bounds(const BwdArgs& a, int s, int& tok0, int& L) {
  if (!a.varlen) {
    tok0 = 0;
    L = a.T;
    return true;
  }
  tok0 = a.cu_seqlens[s];
  const int tok1 = a.cu_seqlens[s + 1];
  L = tok1 - tok0;
  return tok0 >= 0 && L >= 0 && tok1 <= a.total;
}

// Element offset of row p of head h (of a tensor with H heads) in sequence s.
__device__ __forceinline__ long row_off(const BwdArgs& a, int s, int tok0, int h, int H, int p, int D) {
  if (a.varlen) return ((long)(tok0 + p) * H + h) * D;
  return (((long)s * H + h) * a.T + p) * D;
}


// Bounds used by the debug build's checks: elements of a [.., H, .., D]
// tensor, and whether a tile's start coordinates (c1, c2) lie inside its
// tensor map (dense (D, T, num_seqs*H); packed (D, H, total)).
__device__ __forceinline__ long elems(const BwdArgs& a, int H) {
  return a.varlen ? (long)a.total * H * a.D : (long)a.num_seqs * H * a.T * a.D;
}
__device__ __forceinline__ bool tile_ok(const BwdArgs& a, int H, int c1, int c2) {
  return a.varlen ? (c1 >= 0 && c1 < H && c2 >= 0 && c2 < a.total)
                  : (c1 >= 0 && c1 < a.T && c2 >= 0 && c2 < a.num_seqs * H);
}

}  // namespace bwd
}  // namespace gqa
