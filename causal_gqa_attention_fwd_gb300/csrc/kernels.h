// kernels.h -- internal launch interface between the C-ABI layer (api.cu) and
// the kernel translation units.  Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace gqa {

// Forward.  Dense layout: Q,O [B,Hq,T,D], K,V [B,Hkv,T,D], LSE [B,Hq,T]
// (num_seqs = B).  Packed layout (varlen = 1): Q,O [total,Hq,D],
// K,V [total,Hkv,D], LSE [Hq,total], sequences [cu[s], cu[s+1]).
struct FwdArgs {
  __nv_bfloat16* o;
  float* lse;
  const int* cu_seqlens;  // device, varlen only
  int* status;            // device status word
  int num_seqs;           // B for the dense layout
  int T;                  // dense sequence length (unused for varlen)
  int total;              // varlen total tokens
  int Hq, Hkv, G;
  int causal;
  int varlen;
  int pair_heads;         // 1: a CTA's two tiles are heads 2p, 2p+1; 0: row blocks 2m, 2m+1
  int pairs_per_seq;      // head pairs (pair_heads) or heads
  int m_items;            // row-block items per sequence
  float scale_log2;       // scale * log2(e)
  // failure-path test only (attn_test_inject_timeout): when inject_step >= 0,
  // CTA 0's producer stops before the load of that step and every wait of
  // the launch gives up after wait_ns
  int inject_step;
  uint64_t wait_ns;
  int* dbg_line;          // debug builds: source line of the first failed bounds check
};

cudaError_t launch_attn_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const FwdArgs& a,
                            int D, int grid, cudaStream_t stream);

// Backward.  Same layouts; the workspace holds -Delta and -LSE*log2(e) per
// query row (row-padded to whole 128-row tiles).
struct BwdArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* delta;           // workspace: -Delta, [B,Hq,T_pad] or [Hq,total_pad]
  float* lse_log2;        // workspace: -LSE * log2(e), same layout as delta
  int* tile_counter;      // workspace: the dQ kernel's next tile (zeroed by the preprocess)
  const int* cu_seqlens;
  int* status;
  int num_seqs;
  int T;                  // dense sequence length; varlen: the longest sequence
  int T_pad;              // dense rows per head in the f32 workspaces
  int total;
  int total_pad;          // varlen rows per head in the f32 workspaces
  int Hq, Hkv, G;
  int D;
  int causal;
  int varlen;
  int n_items;            // key-block items per sequence (max)
  float scale;
  float scale_log2;
  // rotary backward (f16 Q/K copies): [positions, D] cos/sin table; dK and
  // dQ rows get the transposed rotation at their positions
  const float* rope_cs;
  // failure-path test only (attn_test_inject_timeout): in the kernel named by
  // inject_kernel (1 dK/dV, 2 dQ), the producer of CTA 0 (dK/dV) or of the
  // CTA that takes the first tile (dQ) stops before the load of step
  // inject_step, and every wait gives up after wait_ns
  int inject_kernel;
  int inject_step;
  uint64_t wait_ns;
  long ws_rows;           // rows of each workspace section (bounds of the debug build)
  int n_table;            // rows of rope_cs
  int* dbg_line;          // debug builds: source line of the first failed bounds check
};

// The preprocess, then the dK/dV and dQ kernels.  f16qk: q and k are the f16
// rotated copies (the rotary backward).
cudaError_t launch_attn_bwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dout, const BwdArgs& a, cudaStream_t stream, bool f16qk = false);

// After the preprocess: the key/value-stationary dK/dV kernel and the
// query-stationary dQ kernel (attn_bwd_split.cu).  f16qk: q and k are the
// f16 rotated copies (the rotary backward).
cudaError_t launch_attn_bwd_split(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                  const CUtensorMap& dout, const BwdArgs& a, bool f16qk, cudaStream_t stream);


// Cached (decode) attention.  Q, O [B,Hq,Tq,D]; K/V cache [B,Hkv,S,D];
// LSE [B,Hq,Tq]; cache_lens [B].  The R = G*Tq query rows of a (row, K/V
// head) pair are processed in nrb blocks of 16; a (row, K/V head, block) is
// a unit, u = (b*Hkv + hkv)*nrb + block.  The ctas CTAs share the stream of
// the units' 128-key chunks evenly; a unit cut between CTAs leaves one
// partial per piece in ws_o / ws_ml ([unit][slot][rows_ws]) and a merge
// kernel produces its O and LSE.
constexpr int kDecodeMaxSlots = 160;  // pieces per unit the workspace holds (>= CTAs launched)

struct DecodeArgs {
  const __nv_bfloat16* q;
  const int* cache_lens;  // device
  __nv_bfloat16* o;
  float* lse;
  float* ws_o;            // [units * slots * rows_ws, D] f32 (slots > 1)
  float2* ws_ml;          // [units * slots * rows_ws] (max in log2 units, sum)
  int* status;
  int B, Hq, Hkv, G, Tq, S, D, R;
  int nrb;                // row blocks per (row, K/V head)
  int slots;              // workspace slots per unit: min(chunks at capacity S, kDecodeMaxSlots)
  int rows_ws;            // rows per slot: min(R, 16)
  int ctas;               // CTAs of the partial kernel
  float scale_log2;
  // paged caches (k, v maps over [num_pages * Hkv, page_size, D]): key
  // position j of row b is row j % page_size of page block_table[b * max_pages + j / page_size]
  const int* block_table; // device, nullptr for contiguous caches
  int page_size, max_pages, num_pages;
  // rotary queries: rope_cs [positions, D] f32 (cos half, then sin half), nullptr = none
  const float* rope_cs;
  // FP8 (E4M3) caches: the k, v maps are 8-bit ([.., D] rows, 128-key
  // boxes, no swizzle); K's scale is folded into scale_log2, V's applied to O
  int fp8;
  float v_scale;          // 1 for 16-bit caches
};

// k, v: dense maps over the caches ([B*Hkv, S, D], 64 x 128 boxes) or, paged,
// over the pages ([num_pages*Hkv, page_size, D], 64 x min(page_size, 128)
// boxes); q: 2-D map over the query rows ([B*Hq*Tq, D], 64 x 16 boxes).
cudaError_t launch_attn_decode(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q, const DecodeArgs& a,
                               int grid, cudaStream_t stream);

// Kernel-level timing (opt-in instrumentation, api.cu): event pairs recorded
// on the launch stream around each kernel.
enum ProfKind {
  kProfFwd = 0,
  kProfBwdPre = 1,
  kProfBwdDkdv = 2,
  kProfUnused3 = 3,
  kProfDecode = 4,
  kProfDecodeMerge = 5,
  kProfBwdDq = 6,
  kProfKinds = 7
};
// Launch with programmatic stream serialization (see griddep_wait in
// sm103.cuh): the kernel's CTAs may be scheduled, and run their set-up, while
// the previous kernel in the stream drains.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

void prof_begin(int kind, cudaStream_t s);
void prof_end(cudaStream_t s);

}  // namespace gqa
