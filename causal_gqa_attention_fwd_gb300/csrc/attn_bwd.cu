// attn_bwd.cu -- causal grouped-query attention backward for sm_103a.
//
// For L = sum(dO * O) with O = softmax(scale QK^T + mask) V (the causal GQA
// backward of the microLLM-rocm README, section "Why this project exists"),
// with P recomputed from the forward's LSE instead of stored:
//   P  = exp(scale S - LSE),  dV = P^T dO,  dP = dO V^T,
//   Delta_i = sum_d dO_id O_id,  dS = P * (dP - Delta),
//   dQ = scale dS K,  dK = scale dS^T Q  (dK, dV summed over the G heads of a group).
// Three kernels:
//   1. bwd_pre   -Delta, -LSE*log2(e) into workspace rows (negated so the
//                main kernel forms P and dS with single paired ops); zero the
//                f32 dQ accumulator (HBM-bound).
//   2. bwd_main  key/value-stationary: one CTA per (sequence, K/V head, block
//                of 128 keys) keeps K, V in shared memory and dK, dV in TMEM,
//                and walks the G query heads of the group and every query
//                block that sees its keys.  Per step, five tcgen05 MMAs:
//                  S^T = K Q^T,  dP^T = V dO^T          (TMEM)
//                  dV += P^T dO, dK += dS^T Q           (TMEM accumulators)
//                  dQ partial = dS K                    (TMEM -> smem -> bulk
//                                                        reduce-add into f32)
//                dK and dV leave the CTA once, complete (no atomics).
//   3. bwd_post  dQ = bf16(scale * accumulator).
// Roles in bwd_main (512 threads): warp 0 TMA producer, warp 1 MMA issuer
// (warp-uniform, one elected lane issues; TMEM owner), warps 4-11 two warpgroups that form P and dS (thread = key
// row, each warpgroup half of the step's query columns), warps 12-15 drain dQ
// partials and write dK, dV.
#include "sm103.cuh"
#include "kernels.h"
#include "bwd_common.cuh"

namespace gqa {

using namespace bwd;

namespace {

constexpr int kBN = 128;  // keys per CTA
constexpr int kComputeWGs = 2;                          // warpgroups forming P and dS
constexpr int kBwdThreads = 128 * (2 + kComputeWGs);    // + control warpgroup + drain warpgroup

// dst tensor (f32) += 128-byte-swizzled smem box at coordinates (x, y).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}

}  // namespace

// =========================================================== 1. preprocess
// grid: (row blocks of 128, num_seqs * Hq); 256 threads.  A row is handled by
// D/8 lanes (16 bytes of O and of dO each); a warp covers 32/(D/8) rows per
// pass and keeps four passes of loads in flight.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdArgs a) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerPass = 32 / kLanesPerRow;            // per warp
  constexpr int kPasses = 4;
  const int s = blockIdx.y / a.Hq, h = blockIdx.y % a.Hq;
  int tok0, L;
  if (!seq_bounds(a, s, tok0, L)) {
    if (threadIdx.x == 0) atomicCAS(a.status, 0, kDevBadSeqlens);
    return;
  }
  const int Lr = (L + 127) & ~127;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow, part = lane % kLanesPerRow;
  for (int base = warp * kRowsPerPass * kPasses; base < 128; base += 8 * kRowsPerPass * kPasses) {
    float acc[kPasses];
    int prow[kPasses];
#pragma unroll
    for (int u = 0; u < kPasses; ++u) {
      const int p = blockIdx.x * 128 + base + u * kRowsPerPass + sub;
      prow[u] = p;
      acc[u] = 0.f;
      if (p < L) {
        const long off = row_off(a, s, tok0, h, a.Hq, p, D) + part * 8;
        const uint4 ov = *reinterpret_cast<const uint4*>(a.o + off);
        const uint4 gv = *reinterpret_cast<const uint4*>(a.dout + off);
        const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
        const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 of = __bfloat1622float2(o2[e]), gf = __bfloat1622float2(g2[e]);
          acc[u] = fmaf(of.x, gf.x, acc[u]);
          acc[u] = fmaf(of.y, gf.y, acc[u]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kPasses; ++u) {
#pragma unroll
      for (int m = kLanesPerRow / 2; m > 0; m >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], m);
      const int p = prow[u];
      if (p >= Lr) continue;
      const long w = ws_row(a, s, tok0, h, p);
      if (part == 0) {
        float dl = 0.f, l2 = -INFINITY;       // stored negated: -Delta, -LSE*log2(e)
        if (p < L) {
          const long li = a.varlen ? (long)h * a.total + tok0 + p : ((long)s * a.Hq + h) * a.T + p;
          dl = -acc[u];
          l2 = -a.lse[li] * 1.4426950408889634f;
        }
        a.delta[w] = dl;
        a.lse_log2[w] = l2;
      }
      // zero this row of the f32 dQ accumulator (D floats: 2 x 16 bytes per
      // lane), where the dQ products are summed in one (D = 64)
      if (a.dq_accum) {
        float4* z = reinterpret_cast<float4*>(a.dq_accum + w * D) + part * 2;
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// ============================================================ 3. postprocess
template <int D>
__global__ void __launch_bounds__(256) bwd_post_kernel(const BwdArgs a) {
  const int s = blockIdx.y / a.Hq, h = blockIdx.y % a.Hq;
  int tok0, L;
  if (!seq_bounds(a, s, tok0, L)) return;
  constexpr int kChunks = D / 8;
  for (int idx = threadIdx.x; idx < 128 * kChunks; idx += 256) {
    const int p = blockIdx.x * 128 + idx / kChunks, c = idx % kChunks;
    if (p >= L) continue;
    const float* src = a.dq_accum + ws_row(a, s, tok0, h, p) * D + c * 8;
    const float4 x0 = *reinterpret_cast<const float4*>(src);
    const float4 x1 = *reinterpret_cast<const float4*>(src + 4);
    uint4 out;
    out.x = pack_bf16x2(x0.x * a.scale, x0.y * a.scale);
    out.y = pack_bf16x2(x0.z * a.scale, x0.w * a.scale);
    out.z = pack_bf16x2(x1.x * a.scale, x1.y * a.scale);
    out.w = pack_bf16x2(x1.z * a.scale, x1.w * a.scale);
    *reinterpret_cast<uint4*>(a.dq + row_off(a, s, tok0, h, a.Hq, p, D) + c * 8) = out;
  }
}

// ============================================================== 2. main
namespace {

template <int D>
struct BwdCfg {
  static constexpr int kBM = D == 128 ? 64 : 128;     // queries per step
  static constexpr int kStages = 2;
  static constexpr int kKVBytes = kBN * D * 2;         // K or V tile
  static constexpr int kQBytes = kBM * D * 2;          // Q or dO tile
  static constexpr int kQBoxBytes = kBM * 128;         // one 64-column box of a Q tile
  static constexpr int kStatBytes = kBM * 4;
  static constexpr int kStageBytes = 2 * kQBytes + 1024;   // Q, dO, -LSE2 and -Delta (padded)
  static constexpr int kPBytes = kBN * kBM * 2;        // dS^T tile (for the dQ MMA)
  static constexpr int kStgBytes = kBM * D * 4;        // f32 dQ staging
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKVBytes;
  static constexpr int kOffStage = kOffV + kKVBytes;
  static constexpr int kOffDS = kOffStage + kStages * kStageBytes;
  static constexpr int kOffStg = kOffDS + kPBytes;
  static constexpr int kSmemBytes = kOffStg + kStgBytes + 1024;
  // TMEM columns.  P^T (bf16) is written over S^T and dS^T over dP^T: each
  // compute warpgroup packs its own kCols query columns into the first half
  // of the same kCols columns it read them from.
  static constexpr int kCols = kBM / kComputeWGs;
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = kBM;
  static constexpr uint32_t kColDQ = 2 * kBM;
  static constexpr uint32_t kColK = 2 * kBM + 64;      // K tile as a TMEM A operand (D/2 columns)
  static constexpr uint32_t kColDK = D == 128 ? 256 : 352;
  static constexpr uint32_t kColDV = kColDK + D;
  static_assert(kColK + D / 2 <= kColDK && kColDV + D <= 512, "TMEM budget");
  static constexpr uint32_t kIdescS = idesc_bf16(kBN, kBM, false, false);    // S^T, dP^T
  static constexpr uint32_t kIdescKV = idesc_bf16(kBN, D, false, true);      // dV, dK
  static constexpr uint32_t kIdescQ = idesc_bf16(128, 64, true, true);       // dQ^T (D=128) / dQ (D=64)
  // TMEM column of the packed bf16 operand for the 16 queries of K-step kk
  __device__ static constexpr uint32_t packed_col(uint32_t base, int kk) {
    return base + (uint32_t)((16 * kk) / kCols * kCols + ((16 * kk) % kCols) / 2);
  }
};

struct __align__(8) BwdBarriers {
  uint64_t kv_full, k_tmem;
  uint64_t st_full[2];
  uint64_t st_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full;
  uint64_t dq_full, dq_empty;
  uint64_t stg_full, stg_free;
  uint64_t dkdv_done;
  uint64_t teardown[2];
  uint32_t tmem_base;
  int abort;
};

}  // namespace

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dqacc, const BwdArgs a) {
  using C = BwdCfg<D>;
  constexpr int BM = C::kBM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ BwdBarriers bars;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Guard guard{&bars.abort, a.status};

  // ------------------------------------------------------------- decode
  int item = blockIdx.x;
  const int hkv = item % a.Hkv;
  item /= a.Hkv;
  const int s = item % a.num_seqs;
  const int nb = item / a.num_seqs;                    // key block; heaviest (0) first
  int tok0, L;
  if (!seq_bounds(a, s, tok0, L)) {
    if (threadIdx.x == 0) atomicCAS(a.status, 0, kDevBadSeqlens);
    return;
  }
  const int k0 = nb * kBN;
  if (k0 >= L) return;
  const int n_mb = (L + BM - 1) / BM;
  const int mb0 = a.causal ? k0 / BM : 0;
  const int per_head = n_mb - mb0;
  const int n_it = a.G * per_head;

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.kv_full, 1);
    mbar_init(&bars.k_tmem, 4);                 // barriers fed by whole warps count warps
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.st_full[i], 1);
      mbar_init(&bars.st_empty[i], 2);      // one commit from each MMA issuer
      mbar_init(&bars.teardown[i], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.p_full, 4 * kComputeWGs);
    mbar_init(&bars.ds_full, 4 * kComputeWGs);
    mbar_init(&bars.dq_full, 1);
    mbar_init(&bars.dq_empty, 4);
    mbar_init(&bars.stg_full, 4);
    mbar_init(&bars.stg_free, 1);
    mbar_init(&bars.dkdv_done, 2);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sDS = smem + C::kOffDS;
  uint8_t* sStg = smem + C::kOffStg;
  auto stage_q = [&](int st) { return smem + C::kOffStage + st * C::kStageBytes; };
  auto stage_do = [&](int st) { return smem + C::kOffStage + st * C::kStageBytes + C::kQBytes; };
  auto stage_lse = [&](int st) {
    return reinterpret_cast<float*>(smem + C::kOffStage + st * C::kStageBytes + 2 * C::kQBytes);
  };
  auto stage_delta = [&](int st) {
    return reinterpret_cast<float*>(smem + C::kOffStage + st * C::kStageBytes + 2 * C::kQBytes + 512);
  };
  // iteration -> (query head, query block)
  auto it_head = [&](int i) { return hkv * a.G + i / per_head; };
  auto it_mb = [&](int i) { return mb0 + i % per_head; };

  if (warp == 0) {
    // ======================================================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      int c1, c2;
      if (a.varlen) { c1 = hkv; c2 = tok0 + k0; } else { c1 = k0; c2 = s * a.Hkv + hkv; }
      mbar_expect_tx(&bars.kv_full, 2 * C::kKVBytes);
      for (int b = 0; b < D / 64; ++b) {
        tma_load_3d(sK + b * 16384, &tm_k, &bars.kv_full, b * 64, c1, c2);
        tma_load_3d(sV + b * 16384, &tm_v, &bars.kv_full, b * 64, c1, c2);
      }
      int last_phase[2] = {-1, -1};
      for (int i = 0; i < n_it; ++i) {
        const int st = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!mbar_wait(&bars.st_empty[st], ph ^ 1, guard)) break;
        const int h = it_head(i), mb = it_mb(i);
        if (a.varlen) { c1 = h; c2 = tok0 + mb * BM; } else { c1 = mb * BM; c2 = s * a.Hq + h; }
        mbar_expect_tx(&bars.st_full[st], 2 * C::kQBytes + 2 * C::kStatBytes);
        for (int b = 0; b < D / 64; ++b) {
          tma_load_3d(stage_q(st) + b * C::kQBoxBytes, &tm_q, &bars.st_full[st], b * 64, c1, c2);
          tma_load_3d(stage_do(st) + b * C::kQBoxBytes, &tm_do, &bars.st_full[st], b * 64, c1, c2);
        }
        const long w = ws_row(a, s, tok0, h, mb * BM);
        bulk_load(stage_lse(st), a.lse_log2 + w, C::kStatBytes, &bars.st_full[st]);
        bulk_load(stage_delta(st), a.delta + w, C::kStatBytes, &bars.st_full[st]);
        last_phase[st] = (int)ph;
      }
      mbar_wait_drain(&bars.kv_full, 0);
      for (int st = 0; st < 2; ++st)
        if (last_phase[st] >= 0) mbar_wait_drain(&bars.st_full[st], (uint32_t)last_phase[st]);
    }
  } else if (warp == 1) {
    // ===================================== MMA issuer A: S^T = K Q^T, dV += P^T dO
    // (whole warp, warp-uniform operands, one elected lane issues)
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars.kv_full, 0, guard));
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars.k_tmem, 0, guard));
    auto mma_s = [&](int st) {             // A = K (TMEM), B = Q stage tile (K-major)
      const uint32_t qb = smem_u32(stage_q(st));
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ts_warp(tmem + C::kColS, tmem + C::kColK + kk * 8,
                    sdesc_sw128(qb + (kk >> 2) * C::kQBoxBytes + (kk & 3) * 32, 16, 1024), C::kIdescS, kk > 0);
    };
    if (ok && n_it > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.st_full[0], 0, guard));
      if (ok) {
        tc_fence_after();
        mma_s(0);
        tc_commit_warp(&bars.s_full);
      }
    }
    for (int i = 0; i < n_it && ok; ++i) {
      const int st = i & 1;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.p_full, i & 1, guard)))) break;
      tc_fence_after();
      const uint32_t dob = smem_u32(stage_do(st));      // dO as [N = D x K = queries], MN-major
#pragma unroll
      for (int kk = 0; kk < BM / 16; ++kk)
        mma_ts_warp(tmem + C::kColDV, tmem + C::packed_col(C::kColS, kk),
                    sdesc_sw128(dob + kk * 2048, C::kQBoxBytes, 1024), C::kIdescKV, (i > 0 || kk > 0) ? 1u : 0u);
      tc_commit_warp(&bars.st_empty[st]);
      if (i + 1 < n_it) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.st_full[(i + 1) & 1], ((i + 1) >> 1) & 1, guard))))
          break;
        tc_fence_after();
        mma_s((i + 1) & 1);
        tc_commit_warp(&bars.s_full);
      }
    }
    if (ok) tc_commit_warp(&bars.dkdv_done);
    tc_commit_warp(&bars.teardown[0]);
    mbar_wait_drain(&bars.teardown[0], 0);
  } else if (warp == 2) {
    // =========== MMA issuer B: dP^T = V dO^T, dK += dS^T Q, dQ partial (dS K)
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars.kv_full, 0, guard));
    const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aDS = smem_u32(sDS);
    auto mma_dp = [&](int st) {            // A = V (smem, K-major), B = dO stage tile (K-major)
      const uint32_t db = smem_u32(stage_do(st));
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss_warp(tmem + C::kColDP, sdesc_sw128(aV + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                    sdesc_sw128(db + (kk >> 2) * C::kQBoxBytes + (kk & 3) * 32, 16, 1024), C::kIdescS, kk > 0);
    };
    if (ok && n_it > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.st_full[0], 0, guard));
      if (ok) {
        tc_fence_after();
        mma_dp(0);
        tc_commit_warp(&bars.dp_full);
      }
    }
    for (int i = 0; i < n_it && ok; ++i) {
      const int st = i & 1;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.ds_full, i & 1, guard)))) break;
      tc_fence_after();
      const uint32_t qb = smem_u32(stage_q(st));        // Q as [N = D x K = queries], MN-major
#pragma unroll
      for (int kk = 0; kk < BM / 16; ++kk)
        mma_ts_warp(tmem + C::kColDK, tmem + C::packed_col(C::kColDP, kk),
                    sdesc_sw128(qb + kk * 2048, C::kQBoxBytes, 1024), C::kIdescKV, (i > 0 || kk > 0) ? 1u : 0u);
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.dq_empty, (i & 1) ^ 1, guard)))) break;
      tc_fence_after();
      {
        // dQ^T = K^T dS^T (D = 128) or dQ = dS K (D = 64): both operands
        // MN-major in smem, contraction over the 128 keys.
        const uint32_t qa = D == 128 ? aK : aDS, qbb = D == 128 ? aDS : aK;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ss_warp(tmem + C::kColDQ, sdesc_sw128(qa + kk * 2048, 16384, 1024),
                      sdesc_sw128(qbb + kk * 2048, 16384, 1024), C::kIdescQ, kk > 0);
      }
      tc_commit_warp(&bars.dq_full);
      tc_commit_warp(&bars.st_empty[st]);
      if (i + 1 < n_it) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.st_full[(i + 1) & 1], ((i + 1) >> 1) & 1, guard))))
          break;
        tc_fence_after();
        mma_dp((i + 1) & 1);
        tc_commit_warp(&bars.dp_full);
      }
    }
    if (ok) tc_commit_warp(&bars.dkdv_done);
    tc_commit_warp(&bars.teardown[1]);
    mbar_wait_drain(&bars.teardown[1], 0);
  } else if (warp >= 4 && warp < 4 + 4 * kComputeWGs) {
    // ================================================ compute P^T and dS^T
    // kComputeWGs warpgroups split each step's query columns; thread = key row.
    constexpr int kCols = C::kCols;
    const int c0 = ((warp - 4) >> 2) * kCols;          // first query column of this warpgroup
    const int r = threadIdx.x & 127;                  // key row
    const int key = k0 + r;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float c = a.scale_log2;
    const uint32_t rowDS = smem_u32(sDS) + r * 128;
    bool ok = true;
    if (c0 == 0) {
      // K tile -> TMEM (A operand of S^T = K Q^T): row r = key r, D/2 packed columns
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.kv_full, 0, guard));
      if (ok) {
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          uint32_t kr[32];
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 x = ld_shared_v4(smem_u32(sK) + h * 16384 + r * 128 + ((ch ^ (r & 7)) << 4));
            kr[4 * ch] = x.x;
            kr[4 * ch + 1] = x.y;
            kr[4 * ch + 2] = x.z;
            kr[4 * ch + 3] = x.w;
          }
          tmem_st_x32(tmem + lane_base + C::kColK + h * 32, kr);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&bars.k_tmem);
      }
    }
    for (int i = 0; i < n_it && ok; ++i) {
      const int st = i & 1;
      const uint32_t par = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars.st_full[st], (i >> 1) & 1, guard))) break;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars.s_full, par, guard))) break;
      tc_fence_after();
      const float* nlse2 = stage_lse(st) + c0;     // -LSE*log2(e) per query column
      const float* ndl = stage_delta(st) + c0;      // -Delta per query column
      const int q0 = it_mb(i) * BM + c0;
      const bool need_mask = (a.causal && q0 <= k0 + kBN - 1) || (k0 + kBN > L) || (q0 + kCols > L);
      // visible iff key < L, query < L and (not causal or key <= query)
      const int qmin = a.causal ? key : 0;     // smallest visible query index
      uint32_t pv[kCols];                       // S^T row, then P^T row (f32 bits)
#pragma unroll
      for (int q = 0; q < kCols / 32; ++q) tmem_ld_x32(tmem + lane_base + C::kColS + c0 + q * 32, pv + q * 32);
      tmem_ld_wait();
      reg_fence<kCols>(pv);
      float* p = reinterpret_cast<float*>(pv);
      const uint64_t c2 = f2(c, c);
#pragma unroll
      for (int j = 0; j < kCols; j += 2) {
        const uint64_t nl = *reinterpret_cast<const uint64_t*>(nlse2 + j);
        f2_split(fma2(f2(p[j], p[j + 1]), c2, nl), p[j], p[j + 1]);
        p[j] = ex2_approx(p[j]);
        p[j + 1] = ex2_approx(p[j + 1]);
      }
      if (need_mask) {
        const bool krow_ok = key < L;
#pragma unroll
        for (int j = 0; j < kCols; ++j) {
          const int qi = q0 + j;
          if (!krow_ok || qi >= L || qi < qmin) p[j] = 0.f;
        }
      }
      // P^T row segment -> bf16 pairs -> TMEM over this warpgroup's S^T columns
#pragma unroll
      for (int q = 0; q < kCols / 32; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(p[32 * q + 2 * e], p[32 * q + 2 * e + 1]);
        tmem_st_x16(tmem + lane_base + C::kColS + c0 + q * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars.p_full);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars.dp_full, par, guard))) break;
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < kCols / 32; ++q) {
        uint32_t dv[32];
        tmem_ld_x32(tmem + lane_base + C::kColDP + c0 + q * 32, dv);
        tmem_ld_wait();
        reg_fence<32>(dv);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int j = q * 32 + 2 * e;
          const uint64_t nd = *reinterpret_cast<const uint64_t*>(ndl + j);
          float d0, d1;
          f2_split(mul2(f2(p[j], p[j + 1]), add2(f2(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])), nd)),
                   d0, d1);                                  // P (dP - Delta)
          w[e] = pack_bf16x2(d0, d1);
        }
        // dS^T: into TMEM over this warpgroup's dP^T columns (A of dK += dS^T Q)
        // and into smem (operand of the dQ MMA), 128-byte swizzled K-major rows
        tmem_st_x16(tmem + lane_base + C::kColDP + c0 + q * 16, w);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int ch = (c0 + q * 32) / 8 + cc;
          st_shared_v4(rowDS + (ch >> 3) * 16384 + (((ch & 7) ^ (r & 7)) << 4), w[4 * cc], w[4 * cc + 1],
                       w[4 * cc + 2], w[4 * cc + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive_warp(&bars.ds_full);
    }
  } else if (warp >= 4 + 4 * kComputeWGs) {
    // ===================================== drain dQ partials; dK, dV epilogue
    const int r = threadIdx.x & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const bool leader = (r == 0);
    const uint32_t stg = smem_u32(sStg);
    bool ok = true;
    for (int i = 0; i < n_it; ++i) {
      const uint32_t par = i & 1;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.dq_full, par, guard)))) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld_x32(tmem + lane_base + C::kColDQ, v);
      tmem_ld_x32(tmem + lane_base + C::kColDQ + 32, v + 32);
      tmem_ld_wait();
      reg_fence<64>(v);
      tc_fence_before();
      mbar_arrive_warp(&bars.dq_empty);
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.stg_free, par ^ 1, guard)))) break;
      if (D == 128) {
        // lane = feature d, columns = 64 queries: staging [q][d]
#pragma unroll
        for (int q = 0; q < 64; ++q)
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(stg + (q * 128 + r) * 4), "r"(v[q]) : "memory");
      } else {
        // lane = query, columns = 64 features: two 128-byte-swizzled boxes of
        // [128 queries][32 features] (the layout the tensor reduce reads)
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            st_shared_v4(stg + b * 16384 + r * 128 + ((ch ^ (r & 7)) << 4), v[32 * b + 4 * ch],
                         v[32 * b + 4 * ch + 1], v[32 * b + 4 * ch + 2], v[32 * b + 4 * ch + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive_warp(&bars.stg_full);
      if (leader) {
        if (!mbar_wait(&bars.stg_full, par, guard)) { ok = false; }
        if (ok) {
          const long w = ws_row(a, s, tok0, it_head(i), it_mb(i) * BM);
          if (D == 128) {
            bulk_reduce_add_f32(a.dq_accum + w * D, sStg, C::kStgBytes);
          } else {
            tma_reduce_add_2d(&tm_dqacc, sStg, 0, (int)w);
            tma_reduce_add_2d(&tm_dqacc, sStg + 16384, 32, (int)w);
          }
          bulk_commit();
          bulk_wait_read0();
        }
        mbar_arrive(&bars.stg_free);
      }
      if (!__all_sync(0xffffffffu, ok)) break;
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars.dkdv_done, 0, guard));
    if (ok) {
      tc_fence_after();
      // dK (scaled) into sK, dV into sV (both dead now: every MMA is done): row r,
      // swizzled 16-byte chunks
      for (int t = 0; t < 2; ++t) {
        const uint32_t col = t == 0 ? C::kColDK : C::kColDV;
        const float mul = t == 0 ? a.scale : 1.f;
        const uint32_t srow = smem_u32(t == 0 ? sK : sV) + r * (D * 2);
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t x[32];
          tmem_ld_x32(tmem + lane_base + col + q * 32, x);
          tmem_ld_wait();
          reg_fence<32>(x);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int ch = q * 4 + cc;
            st_shared_v4(srow + ((ch ^ (r & 7)) << 4),
                         pack_bf16x2(__uint_as_float(x[8 * cc]) * mul, __uint_as_float(x[8 * cc + 1]) * mul),
                         pack_bf16x2(__uint_as_float(x[8 * cc + 2]) * mul, __uint_as_float(x[8 * cc + 3]) * mul),
                         pack_bf16x2(__uint_as_float(x[8 * cc + 4]) * mul, __uint_as_float(x[8 * cc + 5]) * mul),
                         pack_bf16x2(__uint_as_float(x[8 * cc + 6]) * mul, __uint_as_float(x[8 * cc + 7]) * mul));
          }
        }
      }
      __syncwarp();
      constexpr int kChunks = D * 2 / 16;
      const int rows_valid = min(kBN, L - k0);
      const int row0 = (warp & 3) * 32;
      for (int t = 0; t < 2; ++t) {
        __nv_bfloat16* dst = t == 0 ? a.dk : a.dv;
        const uint32_t sb = smem_u32(t == 0 ? sK : sV);
        for (int idx = lane; idx < 32 * kChunks; idx += 32) {
          const int row = row0 + idx / kChunks, cch = idx % kChunks;
          if (row < rows_valid) {
            const uint4 val = ld_shared_v4(sb + row * (D * 2) + ((cch ^ (row & 7)) << 4));
            *reinterpret_cast<uint4*>(dst + row_off(a, s, tok0, hkv, a.Hkv, k0 + row, D) + cch * 8) = val;
          }
        }
      }
    }
    if (leader) bulk_wait0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int D>
static cudaError_t launch_pre(const BwdArgs& a, cudaStream_t stream) {
  const int rblocks = (a.T + 127) / 128;   // T: dense length, or the longest sequence
  dim3 gpre(rblocks, a.num_seqs * a.Hq);
  prof_begin(kProfBwdPre, stream);
  bwd_pre_kernel<D><<<gpre, 256, 0, stream>>>(a);
  prof_end(stream);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const BwdArgs& a, cudaStream_t stream) {
  return a.D == 128 ? launch_pre<128>(a, stream) : launch_pre<64>(a, stream);
}

cudaError_t launch_attn_bwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dout, const CUtensorMap& dqacc, const BwdArgs& a,
                            cudaStream_t stream) {
  cudaError_t e = launch_bwd_pre(a, stream);
  if (e != cudaSuccess) return e;
  if (a.D == 128) return launch_attn_bwd128(q, k, v, dout, a, false, stream);
  // D = 64: key/value-stationary kernel with dQ partials reduced into f32
  using C = BwdCfg<64>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(bwd_main_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long grid = (long)a.n_items * a.num_seqs * a.Hkv;
  prof_begin(kProfBwdMain, stream);
  bwd_main_kernel<64><<<(unsigned)grid, kBwdThreads, C::kSmemBytes, stream>>>(q, k, v, dout, dqacc, a);
  prof_end(stream);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 gpost((a.T + 127) / 128, a.num_seqs * a.Hq);
  prof_begin(kProfBwdPost, stream);
  bwd_post_kernel<64><<<gpost, 256, 0, stream>>>(a);
  prof_end(stream);
  return cudaGetLastError();
}

int bwd_query_block(int D) { return D == 128 ? 128 : BwdCfg<64>::kBM; }

}  // namespace gqa
