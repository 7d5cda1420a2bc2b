// attn_bwd.cu -- causal grouped-query attention backward for sm_103a: the
// preprocess and the launch sequence.
//
// For L = sum(dO * O) with O = softmax(scale QK^T + mask) V (the causal GQA
// backward of the microLLM-rocm README, section "Why this project exists"),
// with P recomputed from the forward's LSE instead of stored:
//   P  = exp(scale S - LSE),  dV = P^T dO,  dP = dO V^T,
//   Delta_i = sum_d dO_id O_id,  dS = P * (dP - Delta),
//   dQ = scale dS K,  dK = scale dS^T Q  (dK, dV summed over the G heads of a group).
// Three kernels:
//   1. bwd_pre   -Delta and -LSE*log2(e) per query row into the workspace
//                (negated so the main kernels form P and dS with single
//                paired ops); HBM-bound.
//   2. bwd_dkdv  key/value-stationary dK, dV          (attn_bwd_split.cu)
//   3. bwd_dq    query-stationary dQ                  (attn_bwd_split.cu)
#include "sm103.cuh"
#include "kernels.h"
#include "bwd_common.cuh"

namespace gqa {

using namespace bwd;

// ================================================================ preprocess
// grid: (row blocks of 128, num_seqs * Hq); 256 threads.  A row is handled by
// D/8 lanes (16 bytes of O and of dO each); a warp covers 32/(D/8) rows per
// pass.  Two forms:
//   SWEEP = false  four passes per sweep, each used as it lands (about 31
//                  registers, eight CTAs per SM): grids of several waves;
//   SWEEP = true   (D = 128) one sweep of the CTA's 128 rows whose eight
//                  passes are all issued before any is used (256 bytes in
//                  flight per thread): a grid of one wave at two CTAs per SM,
//                  whose few CTAs must each keep many bytes in flight.
template <int D, bool SWEEP>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdArgs a) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerPass = 32 / kLanesPerRow;            // per warp
  constexpr int P = SWEEP ? 128 / (8 * kRowsPerPass) : 4;    // passes per sweep
  static_assert(128 % (8 * kRowsPerPass * P) == 0, "sweeps tile the row block");
  griddep_wait();      // O (and dO) may come from the previous grid
  griddep_launch();
  // the dQ kernel's tile counter (the previous call's dQ grid has completed:
  // it preceded this grid in the stream)
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *a.tile_counter = 0;
  const int s = blockIdx.y / a.Hq, h = blockIdx.y % a.Hq;
  int tok0, L;
  if (!seq_bounds(a, s, tok0, L)) {
    if (threadIdx.x == 0) atomicCAS(a.status, 0, kDevBadSeqlens);
    return;
  }
  const int Lr = (L + 127) & ~127;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow, part = lane % kLanesPerRow;
  // Delta of row p from its 16-byte pieces of O and dO (this lane's part),
  // reduced over the row's lanes; written with -LSE*log2(e) by lane part 0
  auto finish = [&](float acc, int p) {
#pragma unroll
    for (int m = kLanesPerRow / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (p >= Lr) return;
    const long w = ws_row(a, s, tok0, h, p);
    if (part == 0 && GQA_CHECK(w >= 0 && w < a.ws_rows, a.status, a.dbg_line)) {
      float dl = 0.f, l2 = -INFINITY;       // stored negated: -Delta, -LSE*log2(e)
      const long li = a.varlen ? (long)h * a.total + tok0 + p : ((long)s * a.Hq + h) * a.T + p;
      if (p < L && GQA_CHECK(li >= 0 && li < elems(a, a.Hq) / a.D, a.status, a.dbg_line)) {
        dl = -acc;
        l2 = -a.lse[li] * 1.4426950408889634f;
      }
      a.delta[w] = dl;
      a.lse_log2[w] = l2;
    }
  };
  auto dot8 = [](const uint4& ov, const uint4& gv) {
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 of = __bfloat1622float2(o2[e]), gf = __bfloat1622float2(g2[e]);
      acc = fmaf(of.x, gf.x, acc);
      acc = fmaf(of.y, gf.y, acc);
    }
    return acc;
  };
  for (int base = warp * kRowsPerPass * P; base < 128; base += 8 * kRowsPerPass * P) {
    if constexpr (SWEEP) {
      uint4 ov[P], gv[P];
#pragma unroll
      for (int u = 0; u < P; ++u) {
        const int p = blockIdx.x * 128 + base + u * kRowsPerPass + sub;
        ov[u] = make_uint4(0, 0, 0, 0);
        gv[u] = make_uint4(0, 0, 0, 0);
        const long off = row_off(a, s, tok0, h, a.Hq, p, D) + part * 8;
        if (p < L && GQA_CHECK(off >= 0 && off + 8 <= elems(a, a.Hq), a.status, a.dbg_line)) {
          ov[u] = *reinterpret_cast<const uint4*>(a.o + off);
          gv[u] = *reinterpret_cast<const uint4*>(a.dout + off);
        }
      }
#pragma unroll
      for (int u = 0; u < P; ++u) finish(dot8(ov[u], gv[u]), blockIdx.x * 128 + base + u * kRowsPerPass + sub);
    } else {
      float acc[P];
#pragma unroll
      for (int u = 0; u < P; ++u) {
        const int p = blockIdx.x * 128 + base + u * kRowsPerPass + sub;
        acc[u] = 0.f;
        const long off = row_off(a, s, tok0, h, a.Hq, p, D) + part * 8;
        if (p < L && GQA_CHECK(off >= 0 && off + 8 <= elems(a, a.Hq), a.status, a.dbg_line))
          acc[u] = dot8(*reinterpret_cast<const uint4*>(a.o + off), *reinterpret_cast<const uint4*>(a.dout + off));
      }
#pragma unroll
      for (int u = 0; u < P; ++u) finish(acc[u], blockIdx.x * 128 + base + u * kRowsPerPass + sub);
    }
  }
}

template <int D>
static cudaError_t launch_pre(const BwdArgs& a, cudaStream_t stream) {
  static int sms[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return cudaErrorUnknown;
    sms[dev] = n;
  }
  const int n_sm = dev < 64 ? sms[dev] : 148;
  const int rblocks = (a.T + 127) / 128;   // T: dense length, or the longest sequence
  dim3 gpre(rblocks, a.num_seqs * a.Hq);
  const bool one_wave = (long)rblocks * a.num_seqs * a.Hq <= 2L * n_sm;
  prof_begin(kProfBwdPre, stream);
  cudaError_t e;
  if constexpr (D == 128)
    e = one_wave ? launch_programmatic(bwd_pre_kernel<D, true>, gpre, dim3(256), 0, stream, a)
                 : launch_programmatic(bwd_pre_kernel<D, false>, gpre, dim3(256), 0, stream, a);
  else
    e = launch_programmatic(bwd_pre_kernel<D, false>, gpre, dim3(256), 0, stream, a);
  prof_end(stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dout, const BwdArgs& a, cudaStream_t stream, bool f16qk) {
  cudaError_t e = a.D == 128 ? launch_pre<128>(a, stream) : launch_pre<64>(a, stream);
  if (e != cudaSuccess) return e;
  return launch_attn_bwd_split(q, k, v, dout, a, f16qk, stream);
}

}  // namespace gqa
