// attn_bwd_split.cu -- causal grouped-query attention backward for sm_103a,
// head dimension 64 or 128.
//
// The gradients of L = sum(dO * O) (the causal GQA backward of the
// microLLM-rocm README, section "Why this project exists"), with P recomputed
// from the forward's LSE:  P = exp(scale S - LSE), dP = dO V^T,
// dS = P * (dP - Delta);  dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K.
// After the preprocess (Delta and -LSE*log2(e) per row, attn_bwd.cu), two
// kernels, each keeping its accumulators in TMEM for its whole walk, so no
// partial sum ever leaves the chip:
//
//  bwd_dkdv     key/value-stationary: one CTA per (sequence, K/V head, 128
//     keys) walks the G query heads of the group and the 128-query blocks
//     that see its keys.  Per step four MMAs (128 x 128 x D, 128 x D x 128):
//       S^T = K Q^T, dP^T = V dO^T (recomputed), dV += P^T dO, dK += dS^T Q.
//     Issue order dV(i), S^T(i+1), dK(i), dP^T(i+1): the compute warpgroups
//     form P^T(i+1) while dK(i) runs and dS^T(i+1) while dV(i+1) runs.
//  bwd_dq       query-stationary (the separate dQ pass): one CTA per
//     (sequence, query head, 128 queries) walks the key blocks its queries
//     see.  Per step three MMAs:  S = Q K^T, dP = dO V^T (both recomputed),
//     dQ += dS K.  S is double-buffered in TMEM, so S(j+2) and dP(j+1) run
//     while the compute warpgroups form dS(j); dP is issued by a second warp,
//     so its stream fills the tensor pipe while the S / dQ issuer waits.
//
// dQ is therefore written once, complete and bit-reproducible, with no f32
// accumulator in memory and no conversion pass; the price is recomputing S
// and dP once more (7 matrix products per (query block, key block) instead
// of 5).  FLOPs are still counted by the 5 products the method needs.
//
// Roles in both kernels (384 threads): warp 0 TMA producer, warp 1 MMA issuer
// (warp-uniform operands, one elected lane issues; TMEM owner) -- in
// bwd_dq warp 2 issues the dP stream beside it --, warps 4-11 two compute
// warpgroups (thread = TMEM lane = key row in bwd_dkdv, query
// row in bwd_dq; warpgroup w takes the step's columns [64w, 64w+64)).
//
// F16: Q and K are f16 (the rotated copies of the rotary backward), so every
// product with Q or K takes f16 operands and dS is packed as f16; the
// products with V, dO and P stay bf16.
#include "bwd_common.cuh"
#include "kernels.h"
#include "rope.h"
#include "sm103.cuh"

namespace gqa {

using namespace bwd;

namespace {

constexpr int kBox = 128 * 128;        // one 64-feature box: 128 rows x 128 bytes
template <int D>
constexpr int kTileOf = 128 * D * 2;   // one 128-row tile: D / 64 boxes
constexpr int kStatBytes = 128 * 4;
constexpr int kThreads = 384;
constexpr int kCols = 64;              // columns per compute warpgroup

// TMEM column of the packed 16-bit operand for the 16 columns of K-step kk
// (each warpgroup packs its 64 columns into the first 32 it read them from).
__device__ constexpr uint32_t packed_col(uint32_t base, int kk) {
  return base + (uint32_t)((16 * kk) / kCols * kCols + ((16 * kk) % kCols) / 2);
}

// --------------------------------------------------------------- dK, dV
template <int D>
struct KvCfg {
  static constexpr int kTile = kTileOf<D>;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTile;
  static constexpr int kOffQ = 2 * kTile;       // two stages
  static constexpr int kOffDO = 4 * kTile;      // two stages
  static constexpr int kOffStats = 6 * kTile;   // per stage: -LSE*log2(e) [128], then -Delta [128]
  static constexpr int kOffBars = kOffStats + 2 * 2 * kStatBytes;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDK = 256, kColDV = 256 + D;
};

struct __align__(8) KvBars {
  uint64_t kv_full;
  uint64_t q_full[2], q_empty[2], do_full[2], do_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full;
  uint64_t dkdv_done, teardown;
  uint32_t tmem_base;
  int abort;
};
template <int D>
constexpr int kKvSmem = KvCfg<D>::kOffBars + (int)sizeof(KvBars);

// ------------------------------------------------------------------ dQ
template <int D>
struct QCfg {
  static constexpr int kTile = kTileOf<D>;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kTile;
  static constexpr int kOffK = 2 * kTile;       // three K slots
  static constexpr int kOffV = 5 * kTile;       // two V slots
  static constexpr int kOffBars = 7 * kTile;
  static constexpr uint32_t kColS = 0;          // two S buffers: [0,128), [128,256)
  static constexpr uint32_t kColDP = 256, kColDQ = 384;
};

struct __align__(8) QBars {
  uint64_t q_full, q_empty, do_full, do_empty;
  uint64_t k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t s_full[2], dp_full, dp_read, ds_full;
  uint64_t dq_done, dq_free, teardown;
  uint64_t tile_full[2], tile_empty[2];   // the mailbox of claimed tiles
  int tile[2];
  uint32_t tmem_base;
  int abort;
};
template <int D>
constexpr int kQSmem = QCfg<D>::kOffBars + (int)sizeof(QBars);
static_assert(kKvSmem<128> <= 232448 && kQSmem<128> <= 232448, "shared memory budget");
// TMEM layouts fit the 512 columns the kernels allocate
static_assert(KvCfg<128>::kColDV + 128 <= 512 && KvCfg<64>::kColDV + 64 <= 512, "dK/dV TMEM layout");
static_assert(QCfg<128>::kColDQ + 128 <= 512 && QCfg<64>::kColDQ + 64 <= 512, "dQ TMEM layout");
static_assert(KvCfg<128>::kColDP + 128 <= KvCfg<128>::kColDK && QCfg<128>::kColS + 256 <= QCfg<128>::kColDP,
              "TMEM regions do not overlap");
// shared-memory tiles stay 1024-byte aligned (the 128-byte swizzle is address-based)
static_assert(kTileOf<64> % 1024 == 0 && kBox % 1024 == 0 && KvCfg<128>::kOffStats % 1024 == 0, "tile alignment");

// Rotary transpose for the gradient of a rotated row at position pos (the
// rotation took x to x'_i = x_i c - x_{i+D/2} s, x'_{i+D/2} = x_{i+D/2} c + x_i s):
// g_i = g'_i c + g'_{i+D/2} s,  g_{i+D/2} = g'_{i+D/2} c - g'_i s, for the NP
// pairs i = i0 .. i0+NP-1 of one thread (lo = columns i, hi = columns i + D/2).
template <int D, int NP>
__device__ __forceinline__ void rope_grad_transpose(float* lo, float* hi, const float* cos_sin, int pos, int i0) {
  const float* cs = cos_sin + (long)pos * D;
#pragma unroll
  for (int e = 0; e < NP; e += 4) {
    const float4 c4 = *reinterpret_cast<const float4*>(cs + i0 + e);
    const float4 s4 = *reinterpret_cast<const float4*>(cs + D / 2 + i0 + e);
    const float c[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float a = lo[e + u], b = hi[e + u];
      lo[e + u] = fmaf(a, c[u], b * sn[u]);
      hi[e + u] = fmaf(b, c[u], -a * sn[u]);
    }
  }
}

// N TMEM columns (16 or 32) of this thread's lane into registers.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
  if constexpr (N == 32) tmem_ld_x32(taddr, r);
  else tmem_ld_x16(taddr, r);
}

}  // namespace

// ====================================================================== dK, dV
template <int D, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdArgs a) {
  using C = KvCfg<D>;
  constexpr int BM = 128;
  constexpr int kTile = C::kTile;
  constexpr int NB = D / 64;                   // 64-feature boxes per tile
  constexpr uint32_t kIdS = F16 ? idesc_f16(128, 128, false, false) : idesc_bf16(128, 128, false, false);
  constexpr uint32_t kIdDP = idesc_bf16(128, 128, false, false);
  constexpr uint32_t kIdDV = idesc_bf16(128, D, false, true);
  constexpr uint32_t kIdDK = F16 ? idesc_f16(128, D, false, true) : idesc_bf16(128, D, false, true);
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // A packed batch's decode reads cu_seqlens: wait for the preprocess grid
  // first.  A dense one reads no memory before the set-up below.
  if (a.varlen) griddep_wait();

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
  const int k0 = nb * 128;
  if (k0 >= L) return;
  if (smem_u32(smem) & 1023u) {      // the swizzled tiles need a 1024-byte-aligned base
    if (threadIdx.x == 0) atomicCAS(a.status, 0, kDevInternal);
    return;
  }
  const int n_mb = (L + BM - 1) / BM;
  const int mb0 = a.causal ? nb : 0;
  const int per_head = n_mb - mb0;
  const int n_it = a.G * per_head;

  KvBars& bars = *reinterpret_cast<KvBars*>(smem + C::kOffBars);
  Guard guard{&bars.abort, a.status, a.inject_kernel == 1 ? a.wait_ns : kWaitLimitNs};
  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 1);
      mbar_init(&bars.do_full[i], 1);
      mbar_init(&bars.do_empty[i], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.p_full, 8);                  // one arrive per compute warp
    mbar_init(&bars.ds_full, 8);
    mbar_init(&bars.dkdv_done, 1);
    mbar_init(&bars.teardown, 1);
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
  float* stats = reinterpret_cast<float*>(smem + C::kOffStats);   // [stage][2][BM]
  // The preprocess grid's rows are complete and visible past this wait.
  if (!a.varlen) griddep_wait();
  // The dQ kernel (launched next, programmatic dependent launch) reads
  // nothing this grid writes, only the preprocess's rows, which are complete
  // once every CTA of this grid has passed the wait above (or exited without
  // reading anything): let its CTAs take SMs as this grid's finish.
  griddep_launch();
  auto it_head = [&](int i) { return hkv * a.G + i / per_head; };
  auto it_mb = [&](int i) { return mb0 + i % per_head; };

  if (warp == 0) {
    // ======================================================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      int c1, c2;
      if (a.varlen) { c1 = hkv; c2 = tok0 + k0; } else { c1 = k0; c2 = s * a.Hkv + hkv; }
      mbar_expect_tx(&bars.kv_full, 2 * kTile);
      if (GQA_CHECK(tile_ok(a, a.Hkv, c1, c2), a.status, a.dbg_line))
        for (int b = 0; b < NB; ++b) {
          tma_load_3d(smem + C::kOffK + b * kBox, &tm_k, &bars.kv_full, b * 64, c1, c2);
          tma_load_3d(smem + C::kOffV + b * kBox, &tm_v, &bars.kv_full, b * 64, c1, c2);
        }
      int lastq[2] = {-1, -1}, lastd[2] = {-1, -1};
      for (int i = 0; i < n_it; ++i) {
        if (a.inject_kernel == 1 && blockIdx.x == 0 && i == a.inject_step) break;   // failure-path test
        const int st = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        const int h = it_head(i), mb = it_mb(i);
        if (a.varlen) { c1 = h; c2 = tok0 + mb * BM; } else { c1 = mb * BM; c2 = s * a.Hq + h; }
        if (!mbar_wait(&bars.q_empty[st], ph ^ 1, guard)) break;
        mbar_expect_tx(&bars.q_full[st], kTile + 2 * kStatBytes);
        const long w = ws_row(a, s, tok0, h, mb * BM);
        if (GQA_CHECK(tile_ok(a, a.Hq, c1, c2) && w >= 0 && w + BM <= a.ws_rows, a.status, a.dbg_line)) {
          for (int b = 0; b < NB; ++b)
            tma_load_3d(smem + C::kOffQ + st * kTile + b * kBox, &tm_q, &bars.q_full[st], b * 64, c1, c2);
          bulk_load(stats + st * 2 * BM, a.lse_log2 + w, kStatBytes, &bars.q_full[st]);
          bulk_load(stats + st * 2 * BM + BM, a.delta + w, kStatBytes, &bars.q_full[st]);
        }
        lastq[st] = (int)ph;
        if (!mbar_wait(&bars.do_empty[st], ph ^ 1, guard)) break;
        mbar_expect_tx(&bars.do_full[st], kTile);
        for (int b = 0; b < NB; ++b)
          tma_load_3d(smem + C::kOffDO + st * kTile + b * kBox, &tm_do, &bars.do_full[st], b * 64, c1, c2);
        lastd[st] = (int)ph;
      }
      // never leave the CTA with copies in flight
      mbar_wait_drain(&bars.kv_full, 0);
      for (int st = 0; st < 2; ++st) {
        if (lastq[st] >= 0) mbar_wait_drain(&bars.q_full[st], (uint32_t)lastq[st]);
        if (lastd[st] >= 0) mbar_wait_drain(&bars.do_full[st], (uint32_t)lastd[st]);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer (whole warp, one elected lane issues)
    // Issue order dV(i), S^T(i+1), dK(i), dP^T(i+1).  (Two issuers, one per
    // path, measured slower here: their interleaving delays S^T(i+1) and so
    // the compute warpgroups' P^T(i+1).)
    // K-major operand descriptors (contraction over features, 64 per box) and
    // MN-major ones (contraction over the 128 rows, 16 per step), per stage
    const uint64_t dK = sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dV = sdesc_sw128(smem_u32(smem + C::kOffV), 16, 1024);
    const uint64_t dQk = sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
    const uint64_t dDOk = sdesc_sw128(smem_u32(smem + C::kOffDO), 16, 1024);
    const uint64_t dQm = sdesc_sw128(smem_u32(smem + C::kOffQ), kBox, 1024);
    const uint64_t dDOm = sdesc_sw128(smem_u32(smem + C::kOffDO), kBox, 1024);
    // S^T = K Q^T: A = K, B = Q, both K-major, contraction over the D features
    auto mma_s = [&](int st) {
      const uint64_t q = sdesc_add(dQk, st * kTile);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          mma_ss(tmem + C::kColS, sdesc_add(dK, off), sdesc_add(q, off), kIdS, kk > 0);
        }
      }
      __syncwarp();
    };
    // dP^T = V dO^T
    auto mma_dp = [&](int st) {
      const uint64_t g = sdesc_add(dDOk, st * kTile);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          mma_ss(tmem + C::kColDP, sdesc_add(dV, off), sdesc_add(g, off), kIdDP, kk > 0);
        }
      }
      __syncwarp();
    };
    // dV += P^T dO: A = P^T from TMEM, B = dO [queries x features], MN-major
    auto mma_dv = [&](int st, bool acc) {
      const uint64_t g = sdesc_add(dDOm, st * kTile);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + C::kColDV, tmem + packed_col(C::kColS, kk), sdesc_add(g, kk * 2048), kIdDV,
                      (acc || kk > 0) ? 1u : 0u);
      }
      __syncwarp();
    };
    // dK += dS^T Q
    auto mma_dk = [&](int st, bool acc) {
      const uint64_t q = sdesc_add(dQm, st * kTile);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + C::kColDK, tmem + packed_col(C::kColDP, kk), sdesc_add(q, kk * 2048), kIdDK,
                      (acc || kk > 0) ? 1u : 0u);
      }
      __syncwarp();
    };
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars.kv_full, 0, guard));
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars.q_full[0], 0, guard));
    if (ok) {
      tc_fence_after();
      mma_s(0);
      tc_commit_warp(&bars.s_full);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.do_full[0], 0, guard));
    }
    if (ok) {
      tc_fence_after();
      mma_dp(0);
      tc_commit_warp(&bars.dp_full);
    }
    for (int i = 0; i < n_it && ok; ++i) {
      const int st = i & 1, st1 = (i + 1) & 1;
      const uint32_t ph1 = ((i + 1) >> 1) & 1;
      const bool more = i + 1 < n_it;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.p_full, i & 1, guard)))) break;
      tc_fence_after();
      mma_dv(st, i > 0);
      tc_commit_warp(&bars.do_empty[st]);
      if (more) {   // the S^T columns are free once dV(i) has read P^T(i): in-order issue
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.q_full[st1], ph1, guard)))) break;
        tc_fence_after();
        mma_s(st1);
        tc_commit_warp(&bars.s_full);
      }
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.ds_full, i & 1, guard)))) break;
      tc_fence_after();
      mma_dk(st, i > 0);
      tc_commit_warp(&bars.q_empty[st]);
      if (more) {   // the dP^T columns are free once dK(i) has read dS^T(i)
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.do_full[st1], ph1, guard)))) break;
        tc_fence_after();
        mma_dp(st1);
        tc_commit_warp(&bars.dp_full);
      }
    }
    if (ok) tc_commit_warp(&bars.dkdv_done);
    tc_commit_warp(&bars.teardown);
    mbar_wait_drain(&bars.teardown, 0);
  } else if (warp >= 4) {
    // ============================================ compute warpgroups
    const int wg = (warp - 4) >> 2;
    const int c0 = wg * kCols;                          // first query column of this warpgroup
    const int r = threadIdx.x & 127;                    // key row = TMEM lane
    const int key = k0 + r;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float c = a.scale_log2;
    bool ok = true;
    float p[kCols];                                     // P^T row segment of the current step
    for (int i = 0; i < n_it; ++i) {
      const int st = i & 1;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.q_full[st], (i >> 1) & 1, guard)))) break;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full, i & 1, guard)))) break;
      tc_fence_after();
      const float* nlse2 = stats + st * 2 * BM + c0;       // -LSE*log2(e) per query column
      const float* ndl = stats + st * 2 * BM + BM + c0;     // -Delta per query column
      const int q0 = it_mb(i) * BM + c0;
      const bool need_mask = (a.causal && q0 <= k0 + 127) || (k0 + 128 > L) || (q0 + kCols > L);
      const int qmin = a.causal ? key : 0;               // smallest visible query index
      {
        uint32_t* pv = reinterpret_cast<uint32_t*>(p);
        tmem_ld_x32(tmem + lane_base + C::kColS + c0, pv);
        tmem_ld_x32(tmem + lane_base + C::kColS + c0 + 32, pv + 32);
        tmem_ld_wait();
        reg_fence<kCols>(pv);
      }
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
      // P^T (bf16) over this warpgroup's first 32 S^T columns: A of dV += P^T dO
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(p[32 * q + 2 * e], p[32 * q + 2 * e + 1]);
        tmem_st_x16(tmem + lane_base + C::kColS + c0 + q * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars.p_full);
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.dp_full, i & 1, guard)))) break;
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < 2; ++q) {
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
          w[e] = F16 ? pack_f16x2(d0, d1) : pack_bf16x2(d0, d1);
        }
        // dS^T over this warpgroup's dP^T columns: A of dK += dS^T Q
        tmem_st_x16(tmem + lane_base + C::kColDP + c0 + q * 16, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars.ds_full);
    }
    // ------------------------------------------------ dK (wg 0), dV (wg 1)
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars.dkdv_done, 0, guard));
    if (ok) {
      tc_fence_after();
      const uint32_t col = wg == 0 ? C::kColDK : C::kColDV;
      uint8_t* tile = smem + (wg == 0 ? C::kOffK : C::kOffV);   // dead: every MMA has completed
      const uint32_t srow = smem_u32(tile) + r * (2 * D);
      // Each half-row pair (features i, i + D/2) together, so the rotary
      // backward can undo the key rotation of dK at the key's position.
#pragma unroll 1
      for (int q = 0; q < D / 64; ++q) {
        float lo[32], hi[32];
        tmem_ld_x32(tmem + lane_base + col + q * 32, reinterpret_cast<uint32_t*>(lo));
        tmem_ld_x32(tmem + lane_base + col + D / 2 + q * 32, reinterpret_cast<uint32_t*>(hi));
        tmem_ld_wait();
        reg_fence<32>(reinterpret_cast<uint32_t*>(lo));
        reg_fence<32>(reinterpret_cast<uint32_t*>(hi));
        if (wg == 0) {
          if (F16 && key < L && GQA_CHECK(key < a.n_table, a.status, a.dbg_line))
            rope_grad_transpose<D, 32>(lo, hi, a.rope_cs, key, q * 32);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            lo[e] *= a.scale;
            hi[e] *= a.scale;
          }
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const float* x = half == 0 ? lo : hi;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int ch = half * (D / 16) + q * 4 + cc;
            st_shared_v4(srow + ((ch ^ (r & 7)) << 4), pack_bf16x2(x[8 * cc], x[8 * cc + 1]),
                         pack_bf16x2(x[8 * cc + 2], x[8 * cc + 3]), pack_bf16x2(x[8 * cc + 4], x[8 * cc + 5]),
                         pack_bf16x2(x[8 * cc + 6], x[8 * cc + 7]));
          }
        }
      }
      __syncwarp();
      // this warp's 32 rows, coalesced 16-byte stores (rows inside the sequence)
      constexpr int kChunks = D / 8;                 // 16-byte chunks per row
      const int rows_valid = min(128, L - k0);
      const int row0 = (warp & 3) * 32;
      __nv_bfloat16* dst = wg == 0 ? a.dk : a.dv;
      const uint32_t sb = smem_u32(tile);
      for (int idx = lane; idx < 32 * kChunks; idx += 32) {
        const int row = row0 + idx / kChunks, cch = idx % kChunks;
        const long off = row_off(a, s, tok0, hkv, a.Hkv, k0 + row, D) + cch * 8;
        if (row < rows_valid && GQA_CHECK(off >= 0 && off + 8 <= elems(a, a.Hkv), a.status, a.dbg_line)) {
          const uint4 val = ld_shared_v4(sb + row * (2 * D) + ((cch ^ (row & 7)) << 4));
          *reinterpret_cast<uint4*>(dst + off) = val;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ========================================================================= dQ
// Persistent: one CTA per SM takes (query head, sequence, 128-query block)
// tiles, heaviest first, until none is left: CTA c starts with tile c, and
// every later tile comes from a counter in the workspace (zeroed by the
// preprocess).  Warp 3 claims the tiles and loads each tile's
// Q and dO; the other roles read the claimed tile from a two-slot mailbox.
// The K/V rings, the S buffers and every barrier run on across tiles (step
// counters continue), so a tile's first loads and its first S MMAs overlap
// the previous tile's last steps: Q(e+1) is loaded once the last S of tile e
// is done (q_empty), dO(e+1) once tile e's epilogue has read its staging
// area, the dO tile (do_empty), and the first dQ MMA of tile e+1 waits until
// tile e's accumulator has been read out (dq_free).
template <int D, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdArgs a) {
  using C = QCfg<D>;
  constexpr int BM = 128;
  constexpr int kTile = C::kTile;
  constexpr int NB = D / 64;                   // 64-feature boxes per tile
  constexpr uint32_t kIdS = F16 ? idesc_f16(128, 128, false, false) : idesc_bf16(128, 128, false, false);
  constexpr uint32_t kIdDP = idesc_bf16(128, 128, false, false);
  constexpr uint32_t kIdDQ = F16 ? idesc_f16(128, D, false, true) : idesc_bf16(128, D, false, true);
  constexpr int kReaders = 11;                 // mailbox readers: warps 0, 1, 2 and the 8 compute warps
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicCAS(a.status, 0, kDevInternal);
    return;
  }
  const int n_tiles = a.n_items * a.num_seqs * a.Hq;

  QBars& bars = *reinterpret_cast<QBars*>(smem + C::kOffBars);
  Guard guard{&bars.abort, a.status, a.inject_kernel == 2 ? a.wait_ns : kWaitLimitNs};
  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 1);
    mbar_init(&bars.do_full, 1);
    mbar_init(&bars.do_empty, 8);                // one arrive per compute warp, after its epilogue
    for (int i = 0; i < 3; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.tile_full[i], 1);
      mbar_init(&bars.tile_empty[i], kReaders);
    }
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.dp_read, 8);
    mbar_init(&bars.ds_full, 8);
    mbar_init(&bars.dq_done, 1);
    mbar_init(&bars.dq_free, 8);
    mbar_init(&bars.teardown, 2);                // one commit from each issuer
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

  // A tile's coordinates; empty when its queries lie past its sequence (or
  // the sequence's bounds are invalid, which the fetcher reports).
  struct Tile {
    int h, s, mb, tok0, L, q0, n_kb;
    bool empty;
  };
  auto decode = [&](int t, bool report) {
    Tile x;
    x.h = t % a.Hq;
    t /= a.Hq;
    x.s = t % a.num_seqs;
    x.mb = a.n_items - 1 - t / a.num_seqs;
    x.empty = !seq_bounds(a, x.s, x.tok0, x.L);
    if (x.empty && report) atomicCAS(a.status, 0, kDevBadSeqlens);
    x.q0 = x.mb * BM;
    x.empty = x.empty || x.q0 >= x.L;
    x.n_kb = a.causal ? x.mb + 1 : (x.L + 127) / 128;   // key blocks these queries see
    return x;
  };
  // The k-th claimed tile (-1: none left), read from the mailbox by every
  // role except the fetcher; false if the wait gave up.
  auto read_tile = [&](int k, int& t) {
    if (!__all_sync(0xffffffffu, mbar_wait(&bars.tile_full[k & 1], (k >> 1) & 1, guard))) return false;
    t = *reinterpret_cast<volatile int*>(&bars.tile[k & 1]);
    mbar_arrive_warp(&bars.tile_empty[k & 1]);
    return true;
  };

  if (warp == 3) {
    // ================================= tile fetcher and Q / dO loads
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      int e = 0;                                 // non-empty tiles loaded
      for (int k = 0;; ++k) {
        const int slot = k & 1;
        if (k >= 2 && !mbar_wait(&bars.tile_empty[slot], ((k >> 1) - 1) & 1, guard)) break;
        // the first tile of each CTA is its own index (the grid is no larger
        // than the tile count), so its loads start without a round trip to
        // the counter; later tiles come from the counter, after the first
        // gridDim.x
        int t = k == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(a.tile_counter, 1);
        if (t >= n_tiles) t = -1;
        bars.tile[slot] = t;
        mbar_arrive(&bars.tile_full[slot]);
        if (t < 0) break;
        const Tile x = decode(t, true);
        if (x.empty) continue;
        int c1, c2;
        if (a.varlen) { c1 = x.h; c2 = x.tok0 + x.q0; } else { c1 = x.q0; c2 = x.s * a.Hq + x.h; }
        const bool ok_tile = GQA_CHECK(tile_ok(a, a.Hq, c1, c2), a.status, a.dbg_line);
        if (e >= 1 && !mbar_wait(&bars.q_empty, (e - 1) & 1, guard)) break;
        mbar_expect_tx(&bars.q_full, kTile);
        if (ok_tile)
          for (int b = 0; b < NB; ++b) tma_load_3d(smem + C::kOffQ + b * kBox, &tm_q, &bars.q_full, b * 64, c1, c2);
        if (e >= 1 && !mbar_wait(&bars.do_empty, (e - 1) & 1, guard)) {
          ++e;                                   // Q(e) was issued: drain it below
          break;
        }
        mbar_expect_tx(&bars.do_full, kTile);
        if (ok_tile)
          for (int b = 0; b < NB; ++b)
            tma_load_3d(smem + C::kOffDO + b * kBox, &tm_do, &bars.do_full, b * 64, c1, c2);
        ++e;
      }
      // never leave the CTA with copies in flight
      if (e >= 1) {
        mbar_wait_drain(&bars.q_full, (uint32_t)(e - 1) & 1);
        mbar_wait_drain(&bars.do_full, (uint32_t)(e - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 0) {
    // ================================================ K / V TMA producer
    int lastk[3] = {-1, -1, -1}, lastv[2] = {-1, -1};
    int g = 0;                                   // steps of the tiles before this one
    bool stop = false;
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    for (int k = 0; !stop; ++k) {
      int t;
      if (!read_tile(k, t) || t < 0) break;
      const Tile x = decode(t, false);
      if (x.empty) continue;
      const int hkv = x.h / a.G;
      if (lane == 0) {
        for (int j = 0; j < x.n_kb; ++j) {
          const int gs = g + j;
          if (a.inject_kernel == 2 && t == 0 && j == a.inject_step) {   // failure-path test: the first tile
            stop = true;
            break;
          }
          int c1, c2;
          if (a.varlen) { c1 = hkv; c2 = x.tok0 + j * 128; } else { c1 = j * 128; c2 = x.s * a.Hkv + hkv; }
          const int ks = gs % 3, vs = gs & 1;
          const uint32_t kph = (gs / 3) & 1, vph = (gs >> 1) & 1;
          if (!mbar_wait(&bars.k_empty[ks], kph ^ 1, guard)) { stop = true; break; }
          mbar_expect_tx(&bars.k_full[ks], kTile);
          const bool kv_ok = GQA_CHECK(tile_ok(a, a.Hkv, c1, c2), a.status, a.dbg_line);
          if (kv_ok)
            for (int b = 0; b < NB; ++b)
              tma_load_3d(smem + C::kOffK + ks * kTile + b * kBox, &tm_k, &bars.k_full[ks], b * 64, c1, c2);
          lastk[ks] = (int)kph;
          if (!mbar_wait(&bars.v_empty[vs], vph ^ 1, guard)) { stop = true; break; }
          mbar_expect_tx(&bars.v_full[vs], kTile);
          if (kv_ok)
            for (int b = 0; b < NB; ++b)
              tma_load_3d(smem + C::kOffV + vs * kTile + b * kBox, &tm_v, &bars.v_full[vs], b * 64, c1, c2);
          lastv[vs] = (int)vph;
        }
      }
      stop = __shfl_sync(0xffffffffu, stop, 0);
      g += x.n_kb;
    }
    if (lane == 0) {
      for (int i = 0; i < 3; ++i)
        if (lastk[i] >= 0) mbar_wait_drain(&bars.k_full[i], (uint32_t)lastk[i]);
      for (int i = 0; i < 2; ++i)
        if (lastv[i] >= 0) mbar_wait_drain(&bars.v_full[i], (uint32_t)lastv[i]);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ============ two MMA issuers (whole warps, one elected lane issues):
    // warp 1 S(j) and dQ += dS(j) K_j, warp 2 dP(j); disjoint TMEM columns.
    const uint64_t dQ = sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
    const uint64_t dDO = sdesc_sw128(smem_u32(smem + C::kOffDO), 16, 1024);
    const uint64_t dKk = sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dKm = sdesc_sw128(smem_u32(smem + C::kOffK), kBox, 1024);
    const uint64_t dV = sdesc_sw128(smem_u32(smem + C::kOffV), 16, 1024);
    bool ok = true;
    int g = 0, e = 0;                            // steps and non-empty tiles before this one
    if (warp == 1) {
      auto wait_k = [&](int gs) {
        return __all_sync(0xffffffffu, mbar_wait(&bars.k_full[gs % 3], (gs / 3) & 1, guard));
      };
      // S(gs) = Q K^T into S buffer gs & 1: A = Q, B = K, both K-major
      auto mma_s = [&](int gs) {
        const uint64_t kd = sdesc_add(dKk, (gs % 3) * kTile);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
            mma_ss(tmem + C::kColS + (gs & 1) * 128, sdesc_add(dQ, off), sdesc_add(kd, off), kIdS, kk > 0);
          }
        }
        __syncwarp();
      };
      // dQ += dS(gs) K: A = dS from TMEM (packed over S buffer gs & 1), B = K [keys x features], MN-major
      auto mma_dq = [&](int gs, bool first) {
        const uint64_t kd = sdesc_add(dKm, (gs % 3) * kTile);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::kColDQ, tmem + packed_col(C::kColS + (gs & 1) * 128, kk), sdesc_add(kd, kk * 2048),
                        kIdDQ, (!first || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
      };
      for (int k = 0; ok; ++k) {
        int t;
        if (!(ok = read_tile(k, t)) || t < 0) break;
        const Tile x = decode(t, false);
        if (x.empty) continue;
        const int n = x.n_kb;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.q_full, e & 1, guard)))) break;
        for (int j = 0; j < 2 && j < n && ok; ++j) {
          if (!(ok = wait_k(g + j))) break;
          tc_fence_after();
          mma_s(g + j);
          tc_commit_warp(&bars.s_full[(g + j) & 1]);
          if (j == n - 1) tc_commit_warp(&bars.q_empty);   // the tile's last S: Q may be replaced
        }
        for (int j = 0; j < n && ok; ++j) {
          const int gs = g + j;
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.ds_full, gs & 1, guard)))) break;
          if (j == 0 && e >= 1 && !(ok = __all_sync(0xffffffffu, mbar_wait(&bars.dq_free, (e - 1) & 1, guard))))
            break;                               // the previous tile's dQ has left TMEM
          tc_fence_after();
          mma_dq(gs, j == 0);
          tc_commit_warp(&bars.k_empty[gs % 3]);
          if (j + 2 < n) {   // S buffer gs & 1 is free once dQ(gs) has read dS(gs): in-order issue
            if (!(ok = wait_k(gs + 2))) break;
            tc_fence_after();
            mma_s(gs + 2);
            tc_commit_warp(&bars.s_full[gs & 1]);
            if (j + 2 == n - 1) tc_commit_warp(&bars.q_empty);
          }
        }
        if (ok) tc_commit_warp(&bars.dq_done);
        g += n;
        ++e;
      }
    } else {
      // dP(gs) = dO V^T; the dP columns are free once the compute warps have read dP(gs-1)
      for (int k = 0; ok; ++k) {
        int t;
        if (!(ok = read_tile(k, t)) || t < 0) break;
        const Tile x = decode(t, false);
        if (x.empty) continue;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.do_full, e & 1, guard)))) break;
        for (int j = 0; j < x.n_kb && ok; ++j) {
          const int gs = g + j;
          if (gs > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(&bars.dp_read, (gs - 1) & 1, guard)))) break;
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.v_full[gs & 1], (gs >> 1) & 1, guard)))) break;
          tc_fence_after();
          const uint64_t vd = sdesc_add(dV, (gs & 1) * kTile);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
              mma_ss(tmem + C::kColDP, sdesc_add(dDO, off), sdesc_add(vd, off), kIdDP, kk > 0);
            }
          }
          __syncwarp();
          tc_commit_warp(&bars.dp_full);
          tc_commit_warp(&bars.v_empty[gs & 1]);
        }
        g += x.n_kb;
        ++e;
      }
    }
    tc_commit_warp(&bars.teardown);
    mbar_wait_drain(&bars.teardown, 0);
  } else if (warp >= 4) {
    // ============================================ compute warpgroups
    const int wg = (warp - 4) >> 2;
    const int c0 = wg * kCols;                          // first key column of this warpgroup
    const int r = threadIdx.x & 127;                    // query row = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float c = a.scale_log2;
    bool ok = true;
    int g = 0, e = 0;                                   // steps and non-empty tiles before this one
    for (int k = 0; ok; ++k) {
      int t;
      if (!(ok = read_tile(k, t)) || t < 0) break;
      const Tile x = decode(t, false);
      if (x.empty) continue;
      const int qi = x.q0 + r;
      const long wrow = ws_row(a, x.s, x.tok0, x.h, qi);
      const bool wrow_ok = GQA_CHECK(wrow >= 0 && wrow < a.ws_rows, a.status, a.dbg_line);
      const float nlse2 = wrow_ok ? a.lse_log2[wrow] : -INFINITY;   // -LSE*log2(e) (-inf past the sequence)
      const float ndl = wrow_ok ? a.delta[wrow] : 0.f;              // -Delta
      const uint64_t c2 = f2(c, c), nl2 = f2(nlse2, nlse2), nd2 = f2(ndl, ndl);
      for (int j = 0; j < x.n_kb; ++j) {
        const int gs = g + j;
        const uint32_t sb = C::kColS + (gs & 1) * 128;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[gs & 1], (gs >> 1) & 1, guard)))) break;
        tc_fence_after();
        float p[kCols];
        {
          uint32_t* pv = reinterpret_cast<uint32_t*>(p);
          tmem_ld_x32(tmem + lane_base + sb + c0, pv);
          tmem_ld_x32(tmem + lane_base + sb + c0 + 32, pv + 32);
          tmem_ld_wait();
          reg_fence<kCols>(pv);
        }
#pragma unroll
        for (int e2 = 0; e2 < kCols; e2 += 2) {
          f2_split(fma2(f2(p[e2], p[e2 + 1]), c2, nl2), p[e2], p[e2 + 1]);
          p[e2] = ex2_approx(p[e2]);
          p[e2 + 1] = ex2_approx(p[e2 + 1]);
        }
        const int kbase = j * 128 + c0;                   // key index of this warpgroup's column 0
        if ((a.causal && j == x.mb) || kbase + kCols > x.L || x.q0 + 128 > x.L) {
          const int lim = a.causal ? min(qi + 1, x.L) : x.L;   // visible keys: k < lim (none past the sequence)
#pragma unroll
          for (int e2 = 0; e2 < kCols; ++e2)
            if (kbase + e2 >= lim || qi >= x.L) p[e2] = 0.f;
        }
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.dp_full, gs & 1, guard)))) break;
        tc_fence_after();
        uint32_t dv[kCols];
        tmem_ld_x32(tmem + lane_base + C::kColDP + c0, dv);
        tmem_ld_x32(tmem + lane_base + C::kColDP + c0 + 32, dv + 32);
        tmem_ld_wait();
        reg_fence<kCols>(dv);
        tc_fence_before();
        mbar_arrive_warp(&bars.dp_read);                  // dP(gs+1) may overwrite the dP columns
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t w[16];
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            const int xx = q * 32 + 2 * e2;
            float d0, d1;
            f2_split(mul2(f2(p[xx], p[xx + 1]), add2(f2(__uint_as_float(dv[xx]), __uint_as_float(dv[xx + 1])), nd2)),
                     d0, d1);                               // P (dP - Delta)
            w[e2] = F16 ? pack_f16x2(d0, d1) : pack_bf16x2(d0, d1);
          }
          // dS over this warpgroup's first 32 columns of S buffer gs & 1: A of dQ += dS K
          tmem_st_x16(tmem + lane_base + sb + c0 + q * 16, w);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&bars.ds_full);
      }
      if (!ok) break;
      // ----------------------------------------------------- dQ epilogue
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars.dq_done, e & 1, guard)))) break;
      tc_fence_after();
      // warpgroup wg: feature pairs (i, i + D/2) for i in [NP wg, NP wg + NP)
      constexpr int NP = D / 4;
      float lo[NP], hi[NP];
      tmem_ld_cols<NP>(tmem + lane_base + C::kColDQ + NP * wg, reinterpret_cast<uint32_t*>(lo));
      tmem_ld_cols<NP>(tmem + lane_base + C::kColDQ + D / 2 + NP * wg, reinterpret_cast<uint32_t*>(hi));
      tmem_ld_wait();
      reg_fence<NP>(reinterpret_cast<uint32_t*>(lo));
      reg_fence<NP>(reinterpret_cast<uint32_t*>(hi));
      tc_fence_before();
      mbar_arrive_warp(&bars.dq_free);                  // the next tile's dQ may overwrite the accumulator
      if (F16 && qi < x.L && GQA_CHECK(qi < a.n_table, a.status, a.dbg_line))
        rope_grad_transpose<D, NP>(lo, hi, a.rope_cs, qi, NP * wg);
      // staged through the dO tile: every dP of this tile has completed (its
      // dS came before dq_done), and the next dO waits for do_empty
      const uint32_t srow = smem_u32(smem + C::kOffDO) + r * (2 * D);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float* xv = half == 0 ? lo : hi;
#pragma unroll
        for (int cc = 0; cc < NP / 8; ++cc) {
          const int ch = half * (D / 16) + wg * (NP / 8) + cc;
          st_shared_v4(srow + ((ch ^ (r & 7)) << 4), pack_bf16x2(xv[8 * cc] * a.scale, xv[8 * cc + 1] * a.scale),
                       pack_bf16x2(xv[8 * cc + 2] * a.scale, xv[8 * cc + 3] * a.scale),
                       pack_bf16x2(xv[8 * cc + 4] * a.scale, xv[8 * cc + 5] * a.scale),
                       pack_bf16x2(xv[8 * cc + 6] * a.scale, xv[8 * cc + 7] * a.scale));
        }
      }
      __syncwarp();
      // this warp's 32 rows, the 2 NP / 8 chunks this warpgroup wrote in each
      constexpr int kMine = 2 * (NP / 8);
      const int rows_valid = min(128, x.L - x.q0);
      const int row0 = (warp & 3) * 32;
      const uint32_t sbase = smem_u32(smem + C::kOffDO);
      for (int idx = lane; idx < 32 * kMine; idx += 32) {
        const int row = row0 + idx / kMine, k8 = idx % kMine;
        const int cch = (k8 / (NP / 8)) * (D / 16) + wg * (NP / 8) + k8 % (NP / 8);
        const long off = row_off(a, x.s, x.tok0, x.h, a.Hq, x.q0 + row, D) + cch * 8;
        if (row < rows_valid && GQA_CHECK(off >= 0 && off + 8 <= elems(a, a.Hq), a.status, a.dbg_line)) {
          const uint4 val = ld_shared_v4(sbase + row * (2 * D) + ((cch ^ (row & 7)) << 4));
          *reinterpret_cast<uint4*>(a.dq + off) = val;
        }
      }
      mbar_arrive_warp(&bars.do_empty);                 // the staging area may take the next dO
      g += x.n_kb;
      ++e;
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ==================================================================== launch
template <int D, bool F16>
static cudaError_t launch_split(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& dout, const BwdArgs& a, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(bwd_dkdv_kernel<D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kKvSmem<D>);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_dq_kernel<D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem<D>);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long kv_grid = (long)a.n_items * a.num_seqs * a.Hkv;
  prof_begin(kProfBwdDkdv, stream);
  cudaError_t e = launch_programmatic(bwd_dkdv_kernel<D, F16>, dim3((unsigned)kv_grid), dim3(kThreads), kKvSmem<D>,
                                      stream, q, k, v, dout, a);
  prof_end(stream);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // dQ kernel: programmatic dependent launch.  It reads only the inputs and
  // the preprocess's rows (complete once every dK/dV CTA has passed its
  // griddep_wait, which is when that grid lets this one start) and writes
  // only dQ, so it never waits on the dK/dV grid: its CTAs fill the SMs that
  // grid leaves idle (its tail; all of a small grid's spare SMs).
  // persistent: at most one CTA per SM, each taking tiles until none is left
  static int sms[64] = {};
  if (dev < 64 && sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return cudaErrorUnknown;
    sms[dev] = n;
  }
  const long n_sm = dev < 64 ? sms[dev] : 148;
  const long q_tiles = (long)a.n_items * a.num_seqs * a.Hq;
  const long q_grid = q_tiles < n_sm ? q_tiles : n_sm;
  prof_begin(kProfBwdDq, stream);
  e = launch_programmatic(bwd_dq_kernel<D, F16>, dim3((unsigned)q_grid), dim3(kThreads), kQSmem<D>, stream, q, k, v,
                          dout, a);
  prof_end(stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_split(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                  const CUtensorMap& dout, const BwdArgs& a, bool f16qk, cudaStream_t stream) {
  if (a.D == 128)
    return f16qk ? launch_split<128, true>(q, k, v, dout, a, stream) : launch_split<128, false>(q, k, v, dout, a, stream);
  return f16qk ? launch_split<64, true>(q, k, v, dout, a, stream) : launch_split<64, false>(q, k, v, dout, a, stream);
}

}  // namespace gqa
