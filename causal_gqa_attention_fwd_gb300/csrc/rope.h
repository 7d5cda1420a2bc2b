// rope.h -- rotary (RoPE) prefill: declarations shared by api.cu and attn_fwd.cu.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace gqa {

// One pass over dense bf16 q [rows_q, D] and k [rows_k, D] (row r is position
// r % T of its head) into f16 copies rotated at their positions:
// x'_i = x_i c_i - x_{i+D/2} s_i, x'_{i+D/2} = x_{i+D/2} c_i + x_i s_i with
// c, s from row p of cos_sin [>= T, D] (cos for i < D/2, then sin); in f32,
// rounded once to f16.  All pointers 16-byte aligned.
cudaError_t launch_rope_qk_f16(const void* q, const void* k, void* q_out, void* k_out, long rows_q, long rows_k,
                               int T, int D, const float* cos_sin, cudaStream_t stream);

// The forward of launch_attn_fwd with f16 Q and K (the rotated copies): the
// score MMA takes f16 operands, P V stays bf16.
cudaError_t launch_attn_fwd_f16qk(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                  const FwdArgs& a, int D, int grid, cudaStream_t stream);

}  // namespace gqa
