// rope.h -- rotary (RoPE) prefill: declarations shared by api.cu and attn_fwd.cu.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace gqa {

// Rows of a rotary pass: q rows then k rows, and how a row finds its
// position.  Dense ([N, T, D], cu == nullptr): row r is position r % T.
// Packed ([total, H, D]): row r is token r / H at its offset in the sequence
// cu_seqlens[num_seqs + 1] puts it in.  Positions outside [0, n_table) are
// reported on `status` (ATTN_ERR_SEQLENS) and their rows written as zeros.
struct RopeRows {
  long rows_q, rows_k;
  int T;                 // dense
  int Hq, Hkv;           // packed
  const int* cu;         // packed: device cu_seqlens, or nullptr (dense)
  int num_seqs;          // packed
  int n_table;           // rows of the cos/sin table
  int* status;           // device status word
};

// One pass over bf16 q and k rows (D features each) into f16 copies rotated
// at their positions: x'_i = x_i c_i - x_{i+D/2} s_i,
// x'_{i+D/2} = x_{i+D/2} c_i + x_i s_i with c, s from row p of cos_sin
// [n_table, D] (cos for i < D/2, then sin); in f32, rounded once to f16.
// All pointers 16-byte aligned.
cudaError_t launch_rope_qk_f16(const void* q, const void* k, void* q_out, void* k_out, const RopeRows& rr, int D,
                               const float* cos_sin, cudaStream_t stream);

// The forward of launch_attn_fwd with f16 Q and K (the rotated copies): the
// score MMA takes f16 operands, P V stays bf16.
cudaError_t launch_attn_fwd_f16qk(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                  const FwdArgs& a, int D, int grid, cudaStream_t stream);

}  // namespace gqa
