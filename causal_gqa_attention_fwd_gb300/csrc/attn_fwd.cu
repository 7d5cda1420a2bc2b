// attn_fwd.cu -- causal grouped-query attention forward for sm_103a.
//
// Computes, per query head h (key/value head h / G), O = softmax(scale*QK^T +
// causal mask) V and the natural-log row log-sum-exp LSE, keeping the softmax
// statistics block by block (running max and running sum) instead of
// materialising the score matrix -- the blockwise scheme named in "Project
// Overview" (llm-from-scratch), section "Performance Layer: kernel/ and
// parallel/"; the operation itself is the ScaledDotProductAttention of its
// llm/transformer.py list and the "Decoder-only MHA/GQA ... causal attention"
// of the microLLM-rocm README, section "Why this project exists".
//
// One CTA owns two 128-row query tiles that read the same key/value blocks:
// two query heads of one GQA group at the same rows (G even), or two
// consecutive row blocks of one head (G odd).  Roles (384 threads):
//   warp 0      TMA producer: Q tiles once, then K_j, V_j through a ring.
//   warp 1      MMA issuer (warp-uniform, one elected lane issues): S = Q K^T
//               into TMEM (SS form), then O += P V with P read from TMEM (TS
//               form); allocates TMEM.
//   warps 4-7   softmax for tile A, warps 8-11 for tile B; thread = row.
// TMEM columns: S_A [0,128), S_B [128,256), O_A, O_B (D columns each).
// D = 128: P (bf16) overwrites the first 64 columns of its S block, so a
// tile's next S = Q K^T waits for its P V.  D = 64: P_A [384,448) and P_B
// [448,512) have their own columns, so the next S is issued as soon as the
// softmax has read the current one into registers (s_free) and is computed
// while that softmax runs; the softmax waits for the previous P V (pv_done)
// before it writes P or rescales O.
// Tiles of key blocks past the diagonal are never visited; only the diagonal
// block and a ragged last block are masked.
//
// Rotary prefill (RoPE of MultiHeadAttentionWithRoPE, llm-from-scratch
// "Project Overview"; positions-aware RoPE of the microLLM-rocm README):
// rope_qk_f16_kernel rotates Q and K at their positions into f16 copies in
// one bandwidth-bound pass, and the same kernel (F16QK) takes them as f16
// operands of the score MMA.  f16 keeps 11 significant bits of the rotated
// values; rounding them to bf16 would alone put the LSE about 3e-3 off.
#include <cuda_fp16.h>

#include "sm103.cuh"
#include "kernels.h"
#include "rope.h"

namespace gqa {

namespace {

constexpr int kBM = 128;       // query rows per tile
constexpr int kBN = 128;       // keys per block
constexpr float kRescaleThreshold = 8.0f;  // log2 units: lazy O rescale

template <int D, bool F16QK = false>
struct FwdCfg {
  static constexpr int kTileBytes = kBM * D * 2;        // one Q / K / V tile
  static constexpr int kBoxes = D / 64;                  // 64-element TMA boxes
  static constexpr int kBoxBytes = kBM * 128;            // 16 KB
  static constexpr int kStages = D == 128 ? 4 : 8;       // K/V ring depth
  static constexpr int kSmemQ = 2 * kTileBytes;
  static constexpr int kSmemRing = kStages * kTileBytes;
  static constexpr int kSmemBytes = kSmemQ + kSmemRing + 1024;  // + alignment slack
  // D = 64 leaves TMEM room for P columns of its own (see the layout above)
  static constexpr bool kSepP = D == 64;
  __device__ static constexpr uint32_t col_s(int x) { return (uint32_t)x * 128u; }
  __device__ static constexpr uint32_t col_o(int x) { return 256u + (uint32_t)x * D; }
  __device__ static constexpr uint32_t col_p(int x) { return kSepP ? 384u + (uint32_t)x * 64u : col_s(x); }
  // score MMA: bf16 Q and K, or f16 (rotated copies; A/B format code 0 = f16)
  static constexpr uint32_t kIdescQK =
      F16QK ? (idesc_bf16(kBM, kBN, false, false) & ~((7u << 7) | (7u << 10))) : idesc_bf16(kBM, kBN, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16(kBM, D, false, true);
};

// TMEM layout (S_A, S_B, O_A, O_B; at D = 64 also P_A, P_B) fits the 512
// columns the kernel allocates
static_assert(256 + 2 * 128 <= 512, "forward TMEM layout");
static_assert(256 + 2 * 64 + 2 * 64 <= 512, "forward TMEM layout with P columns (D = 64)");

struct __align__(8) FwdBarriers {
  uint64_t q_full[2];
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t p_half[2];    // D = 128: keys 0-63 of P are in TMEM (p_full: all of P)
  uint64_t o_done[2];
  uint64_t s_free[2];    // D = 64: the softmax has read S into registers
  uint64_t pv_done[2];   // D = 64: a tile's P V has completed
  uint64_t teardown;
  uint32_t tmem_base;
  int abort;
};

struct TileInfo {
  int valid;
  int hq;        // query head
  int mb;        // row block within the sequence
  int nkv;       // key blocks to visit
};

}  // namespace

template <int D, bool F16QK>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdArgs args) {
  using C = FwdCfg<D, F16QK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                      // 2 tiles
  uint8_t* sRing = smem + C::kSmemQ;       // kStages tiles
  __shared__ FwdBarriers bars;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  Guard guard{&bars.abort, args.status, args.inject_step >= 0 ? args.wait_ns : kWaitLimitNs};

  // A packed batch's decode reads cu_seqlens: wait for the previous grid
  // first.  A dense one reads no memory before the set-up below.
  if (args.varlen) griddep_wait();

  // ---------------------------------------------------------- work decode
  // blockIdx.x -> (row-block item, sequence/batch, head pair); heaviest
  // (largest row block) first.
  int item = blockIdx.x;
  const int pairs = args.pairs_per_seq;
  const int pair = item % pairs;
  item /= pairs;
  const int seq = item % args.num_seqs;
  const int mitem = args.m_items - 1 - item / args.num_seqs;

  int tok0 = 0, L = args.T;
  if (args.varlen) {
    tok0 = args.cu_seqlens[seq];
    const int tok1 = args.cu_seqlens[seq + 1];
    L = tok1 - tok0;
    if (L < 0 || tok0 < 0 || tok1 > args.total) {
      if (threadIdx.x == 0) atomicCAS(args.status, 0, kDevBadSeqlens);
      return;
    }
  }
  const int nkv_all = (L + kBN - 1) / kBN;
  TileInfo ti[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    if (args.pair_heads) {           // two heads of one group, same rows
      ti[x].hq = 2 * pair + x;
      ti[x].mb = mitem;
    } else {                         // one head, two consecutive row blocks
      ti[x].hq = pair;
      ti[x].mb = 2 * mitem + x;
    }
    ti[x].valid = ti[x].mb * kBM < L;
    ti[x].nkv = !ti[x].valid ? 0 : (args.causal ? min(ti[x].mb + 1, nkv_all) : nkv_all);
  }
  if (!ti[0].valid && !ti[1].valid) return;
  const int hkv = ti[0].valid ? ti[0].hq / args.G : ti[1].hq / args.G;
  const int nkv = max(ti[0].nkv, ti[1].nkv);

  // ------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    bars.abort = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], kBM / 32);      // one arrive per softmax warp
      mbar_init(&bars.p_half[i], kBM / 32);
      mbar_init(&bars.o_done[i], 1);
      mbar_init(&bars.s_free[i], kBM / 32);
      mbar_init(&bars.pv_done[i], 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
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
  if (!args.varlen) griddep_wait();   // the inputs may come from the previous grid
  griddep_launch();
  // Register split (launched 384 x 168 = 64512), set at the top of each
  // role: the control warpgroup (warps 0-3) keeps 64, the two softmax
  // warpgroups take 216 each, so a softmax thread holds its whole 128-column
  // score row without spilling: 128*64 + 256*216 = 63488 <= 64512, and per
  // sub-partition (warps w, w+4, w+8) 32*(64 + 216 + 216) = 15872 <= 16384.

  // Coordinates of a 128-row tile in a Q / K / V tensor map.
  auto coords = [&](int head, int nheads_b, int row0, int& c1, int& c2) {
    if (args.varlen) {
      c1 = head;
      c2 = tok0 + row0;
    } else {
      c1 = row0;
      c2 = seq * nheads_b + head;
    }
  };
  // debug builds: a tile's start lies inside its tensor map
  auto tile_ok = [&](int nheads_b, int c1, int c2) {
    return args.varlen ? (c1 >= 0 && c1 < nheads_b && c2 >= 0 && c2 < args.total)
                       : (c1 >= 0 && c1 < args.T && c2 >= 0 && c2 < args.num_seqs * nheads_b);
  };
  (void)tile_ok;

  if (warp == 0) {
    // ======================================================== TMA producer
    regs_dec<64>();
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      for (int x = 0; x < 2; ++x) {
        if (!ti[x].valid) continue;
        int c1, c2;
        coords(ti[x].hq, args.Hq, ti[x].mb * kBM, c1, c2);
        mbar_expect_tx(&bars.q_full[x], C::kTileBytes);
        if (GQA_CHECK(tile_ok(args.Hq, c1, c2), args.status, args.dbg_line))
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(sQ + x * C::kTileBytes + b * C::kBoxBytes, &tm_q, &bars.q_full[x], b * 64, c1, c2);
      }
      int last_phase[8];
      for (int s = 0; s < 8; ++s) last_phase[s] = -1;
      int idx = 0;
      bool ok = true;
      for (int j = 0; j < nkv && ok; ++j) {
        if (blockIdx.x == 0 && j == args.inject_step) break;   // failure-path test: a load never issued
        for (int kv = 0; kv < 2 && ok; ++kv, ++idx) {
          const int st = idx % C::kStages;
          const uint32_t ph = (idx / C::kStages) & 1;
          if (!mbar_wait(&bars.kv_empty[st], ph ^ 1, guard)) { ok = false; break; }
          int c1, c2;
          coords(hkv, args.Hkv, j * kBN, c1, c2);
          uint8_t* dst = sRing + st * C::kTileBytes;
          mbar_expect_tx(&bars.kv_full[st], C::kTileBytes);
          const CUtensorMap* tm = kv == 0 ? &tm_k : &tm_v;
          if (GQA_CHECK(tile_ok(args.Hkv, c1, c2), args.status, args.dbg_line))
            for (int b = 0; b < C::kBoxes; ++b)
              tma_load_3d(dst + b * C::kBoxBytes, tm, &bars.kv_full[st], b * 64, c1, c2);
          last_phase[st] = (int)ph;
        }
      }
      // Never leave the CTA with copies in flight.
      for (int x = 0; x < 2; ++x)
        if (ti[x].valid) mbar_wait_drain(&bars.q_full[x], 0);
      for (int s = 0; s < C::kStages; ++s)
        if (last_phase[s] >= 0) mbar_wait_drain(&bars.kv_full[s], (uint32_t)last_phase[s]);
    }
  } else if (warp == 1) {
    // ============================================ MMA issuer (whole warp, one lane issues)
    regs_dec<64>();
    {
      bool ok = true;
      for (int x = 0; x < 2 && ok; ++x)
        if (ti[x].valid) ok = __all_sync(0xffffffffu, mbar_wait(&bars.q_full[x], 0, guard));
      const uint32_t sq_addr = smem_u32(sQ);
      const uint32_t ring_addr = smem_u32(sRing);
      auto issue_qk = [&](int x, int st) {
        const uint32_t qa = sq_addr + x * C::kTileBytes;
        const uint32_t ka = ring_addr + st * C::kTileBytes;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
            mma_ss(tmem + C::col_s(x), sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                   C::kIdescQK, kk > 0);
          }
        }
        __syncwarp();
      };
      // P V over the keys [16 kk0, 16 kk1) of the block (P packed in TMEM)
      auto issue_pv_part = [&](int x, int st, int acc, int kk0, int kk1) {
        const uint32_t va = ring_addr + st * C::kTileBytes;
        if (elect_one()) {
#pragma unroll
          for (int kk = kk0; kk < kk1; ++kk) {
            mma_ts(tmem + C::col_o(x), tmem + C::col_p(x) + kk * 8, sdesc_sw128(va + kk * 2048, C::kBoxBytes, 1024),
                   C::kIdescPV, (acc || kk > 0) ? 1u : 0u);
          }
        }
        __syncwarp();
      };
      auto issue_pv = [&](int x, int st, int acc) { issue_pv_part(x, st, acc, 0, kBN / 16); };
      // K_j sits at ring index 2j, V_j at 2j + 1.
      auto stage_of = [&](int idx) { return idx % C::kStages; };
      auto phase_of = [&](int idx) { return (uint32_t)((idx / C::kStages) & 1); };
      if (ok && nkv > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.kv_full[stage_of(0)], phase_of(0), guard));
        if (ok) {
          tc_fence_after();
          for (int x = 0; x < 2; ++x)
            if (ti[x].nkv > 0) {
              issue_qk(x, stage_of(0));
              tc_commit_warp(&bars.s_full[x]);
            }
          tc_commit_warp(&bars.kv_empty[stage_of(0)]);
        }
      }
      if constexpr (C::kSepP) {
        // Per step j: the next scores of each tile as soon as its softmax has
        // read S_j (K_{j+1}), then each tile's P_j V_j once P_j is written.
        for (int j = 0; j < nkv && ok; ++j) {
          const int vi = 2 * j + 1, ki = 2 * j + 2;
          if (j + 1 < nkv) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.kv_full[stage_of(ki)], phase_of(ki), guard));
            for (int x = 0; x < 2 && ok; ++x) {
              if (j + 1 >= ti[x].nkv) continue;
              ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_free[x], j & 1, guard));
              if (!ok) break;
              tc_fence_after();
              issue_qk(x, stage_of(ki));
              tc_commit_warp(&bars.s_full[x]);
            }
            if (!ok) break;
            tc_commit_warp(&bars.kv_empty[stage_of(ki)]);
          }
          ok = __all_sync(0xffffffffu, mbar_wait(&bars.kv_full[stage_of(vi)], phase_of(vi), guard));
          for (int x = 0; x < 2 && ok; ++x) {
            if (j >= ti[x].nkv) continue;
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.p_full[x], j & 1, guard));
            if (!ok) break;
            tc_fence_after();
            issue_pv(x, stage_of(vi), j > 0);
            tc_commit_warp(&bars.pv_done[x]);
            if (j + 1 == ti[x].nkv) tc_commit_warp(&bars.o_done[x]);
          }
          if (!ok) break;
          tc_commit_warp(&bars.kv_empty[stage_of(vi)]);
        }
      }
      for (int j = 0; j < nkv && ok && !C::kSepP; ++j) {
        const int vi = 2 * j + 1, ki = 2 * j + 2;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.kv_full[stage_of(vi)], phase_of(vi), guard));
        if (ok && j + 1 < nkv) ok = __all_sync(0xffffffffu, mbar_wait(&bars.kv_full[stage_of(ki)], phase_of(ki), guard));
        if (!ok) break;
        tc_fence_after();
        for (int x = 0; x < 2 && ok; ++x) {
          if (j >= ti[x].nkv) continue;
          // P_j arrives in two halves (keys 0-63, then 64-127): the first
          // half's P V runs while the softmax forms the second half
          ok = __all_sync(0xffffffffu, mbar_wait(&bars.p_half[x], j & 1, guard));
          if (!ok) break;
          tc_fence_after();
          issue_pv_part(x, stage_of(vi), j > 0, 0, kBN / 32);
          ok = __all_sync(0xffffffffu, mbar_wait(&bars.p_full[x], j & 1, guard));
          if (!ok) break;
          tc_fence_after();
          issue_pv_part(x, stage_of(vi), 1, kBN / 32, kBN / 16);
          if (j + 1 < ti[x].nkv) {
            issue_qk(x, stage_of(ki));
            tc_commit_warp(&bars.s_full[x]);
          } else {
            tc_commit_warp(&bars.o_done[x]);
          }
        }
        if (!ok) break;
        tc_commit_warp(&bars.kv_empty[stage_of(vi)]);
        if (j + 1 < nkv) tc_commit_warp(&bars.kv_empty[stage_of(ki)]);
      }
      // Let every issued MMA finish before TMEM is released.
      tc_commit_warp(&bars.teardown);
      mbar_wait_drain(&bars.teardown, 0);
    }
  } else if (warp < 4) {
    regs_dec<64>();                         // idle: registers go to the softmax warpgroups
  } else {
    // ============================================================ softmax
    regs_inc<216>();
    const int x = (warp - 4) >> 2;          // tile
    const int r = threadIdx.x & 127;        // row within the tile
    const TileInfo t = ti[x];
    if (t.valid) {
      const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t tS = tmem + lane_base + C::col_s(x);
      const uint32_t tP = tmem + lane_base + C::col_p(x);
      const uint32_t tO = tmem + lane_base + C::col_o(x);
      const float c = args.scale_log2;
      const int qi = t.mb * kBM + r;        // query index within the sequence
      float m_run = -INFINITY;              // running max, log2 units (scale folded in)
      float l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < t.nkv; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[x], j & 1, guard));
        if (!ok) break;
        tc_fence_after();
        uint32_t s[kBN];
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q) tmem_ld_x32(tS + q * 32, s + q * 32);
        tmem_ld_wait();
        reg_fence<kBN>(s);
        if constexpr (C::kSepP) {
          tc_fence_before();
          mbar_arrive_warp(&bars.s_free[x]);   // S_j is in registers: the next S may overwrite it
        }
        float* sf = reinterpret_cast<float*>(s);
        const int k0 = j * kBN;
        const bool need_mask = (args.causal && j == t.mb) || (k0 + kBN > L);
        if (need_mask) {
          const int lim = args.causal ? min(qi + 1, L) : L;   // visible keys: k < lim
#pragma unroll
          for (int i = 0; i < kBN; ++i)
            if (k0 + i >= lim) sf[i] = -INFINITY;
        }
        // row max: eight independent chains of three-input max
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = fmaxf(sf[e], sf[e + 8]);
#pragma unroll
        for (int i = 16; i < kBN; i += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e) m8[e] = max3f(m8[e], sf[i + e], sf[i + 8 + e]);
        const float mx = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        const float m_new = fmaxf(m_run, mx * c);
        float alpha = 1.f;
        bool resc = false;
        if (j == 0) {
          m_run = m_new;
        } else if (m_new > m_run + kRescaleThreshold) {
          alpha = ex2_approx(m_run - m_new);
          m_run = m_new;
          resc = true;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        if constexpr (C::kSepP) {
          // P_{j-1} V_{j-1} has read the P columns and finished adding into O
          if (j > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.pv_done[x], (j - 1) & 1, guard));
            if (!ok) break;
            tc_fence_after();
          }
        }
        // Split P (D = 128): O is rescaled first (P_{j-1} V_{j-1} has
        // completed: the commit of S_j covered it), then P goes out in two
        // halves, signalled on p_half and p_full (each completes once per
        // step), so the first half's P V overlaps the second half's
        // exponentials.
        constexpr bool kSplitP = !C::kSepP;
        if (kSplitP && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            tmem_ld_x32(tO + q * 32, o);
            tmem_ld_wait();
            reg_fence<32>(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st_x32(tO + q * 32, o);
          }
        }
        // p = 2^(s c - m): exponent arguments and the row sum in paired f32
        const uint64_t c2 = f2(c, c), nm2 = f2(-m_use, -m_use);
        uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float t0, t1;
            f2_split(fma2(f2(sf[q * 32 + 2 * i], sf[q * 32 + 2 * i + 1]), c2, nm2), t0, t1);
            const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
            acc[i & 3] = add2(acc[i & 3], f2(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st_x16(tP + q * 16, pk);
          if (kSplitP && q == kBN / 64 - 1) {
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(&bars.p_half[x]);   // keys 0-63 of P_j are in TMEM
          }
        }
        float rs0, rs1;
        f2_split(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])), rs0, rs1);
        const float rs = rs0 + rs1;
        l_run = l_run * alpha + rs;
        if (!kSplitP && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            tmem_ld_x32(tO + q * 32, o);
            tmem_ld_wait();
            reg_fence<32>(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st_x32(tO + q * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&bars.p_full[x]);
      }
      // ------------------------------------------------------- epilogue
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars.o_done[x], 0, guard));
      if (ok) {
        tc_fence_after();
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
        uint8_t* stage = sQ + x * C::kTileBytes;           // Q tile is dead now
        const uint32_t srow = smem_u32(stage) + r * (D * 2);
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld_x32(tO + q * 32, o);
          tmem_ld_wait();
          reg_fence<32>(o);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
#pragma unroll
          for (int cch = 0; cch < 4; ++cch) {
            const int chunk = q * 4 + cch;                   // 16-byte chunk in the row
            st_shared_v4(srow + ((chunk ^ (r & 7)) << 4), pk[4 * cch], pk[4 * cch + 1], pk[4 * cch + 2],
                         pk[4 * cch + 3]);
          }
        }
        const int rows_valid = min(kBM, L - t.mb * kBM);
        if (r < rows_valid) {
          const float lse = (m_run + __log2f(l_run)) * 0.69314718055994531f;
          const long li = args.varlen ? (long)t.hq * args.total + tok0 + qi
                                      : ((long)seq * args.Hq + t.hq) * args.T + qi;
          const long n_lse = args.varlen ? (long)args.Hq * args.total : (long)args.num_seqs * args.Hq * args.T;
          if (GQA_CHECK(li >= 0 && li < n_lse, args.status, args.dbg_line)) args.lse[li] = lse;
        }
        __syncwarp();
        // coalesced copy of this warp's 32 rows (those inside the sequence)
        constexpr int kChunks = D * 2 / 16;
        __nv_bfloat16* obase;
        long ors;
        if (args.varlen) {
          obase = args.o + ((long)(tok0 + t.mb * kBM) * args.Hq + t.hq) * D;
          ors = (long)args.Hq * D;
        } else {
          obase = args.o + (((long)seq * args.Hq + t.hq) * args.T + t.mb * kBM) * D;
          ors = D;
        }
        const uint32_t sbase = smem_u32(stage);
        const int row0 = (warp & 3) * 32;
#pragma unroll 4
        for (int idx = lane; idx < 32 * kChunks; idx += 32) {
          const int row = row0 + idx / kChunks, cch = idx % kChunks;
          const long n_o = (args.varlen ? (long)args.total : (long)args.num_seqs * args.T) * args.Hq * D;
          if (row < rows_valid &&
              GQA_CHECK(obase + row * ors + cch * 8 >= args.o && obase + row * ors + cch * 8 + 8 <= args.o + n_o,
                        args.status, args.dbg_line)) {
            const uint4 v = ld_shared_v4(sbase + row * (D * 2) + ((cch ^ (row & 7)) << 4));
            *reinterpret_cast<uint4*>(obase + row * ors + cch * 8) = v;
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int D, bool F16QK>
static cudaError_t launch_fwd_d(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const FwdArgs& a, int grid, cudaStream_t stream) {
  using C = FwdCfg<D, F16QK>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, F16QK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  prof_begin(kProfFwd, stream);
  cudaError_t e = launch_programmatic(attn_fwd_kernel<D, F16QK>, dim3(grid), dim3(384), C::kSmemBytes, stream, q, k,
                                      v, a);
  prof_end(stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const FwdArgs& a,
                            int D, int grid, cudaStream_t stream) {
  if (D == 128) return launch_fwd_d<128, false>(q, k, v, a, grid, stream);
  return launch_fwd_d<64, false>(q, k, v, a, grid, stream);
}

cudaError_t launch_attn_fwd_f16qk(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                  const FwdArgs& a, int D, int grid, cudaStream_t stream) {
  if (D == 128) return launch_fwd_d<128, true>(q, k, v, a, grid, stream);
  return launch_fwd_d<64, true>(q, k, v, a, grid, stream);
}

namespace {

// Eight rotated pairs per thread: features i0..i0+7 of the low half with
// i0+D/2.. of the high half; D/16 threads per row, rows of q then of k.
// Dense rows ([N, T, D]) are at position row % T.  Packed rows
// ([total, H, D]: token row / H) are at the token's offset in its sequence,
// found by a binary search of cu_seqlens; tokens in no sequence get zero
// rows; a position outside the table (a malformed cu_seqlens) is reported
// as ATTN_ERR_SEQLENS and the row written as zeros, the table never read
// out of bounds.
template <int D, bool PACKED>
__global__ void __launch_bounds__(256) rope_qk_f16_kernel(const __nv_bfloat16* __restrict__ q,
                                                          const __nv_bfloat16* __restrict__ k, __half* __restrict__ qo,
                                                          __half* __restrict__ ko, RopeRows rr,
                                                          const float* __restrict__ cos_sin) {
  constexpr int H = D / 2, kPer = 8, kThr = H / kPer;
  const long gid = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const long row = gid / kThr;
  if (row >= rr.rows_q + rr.rows_k) return;
  const int i0 = (int)(gid % kThr) * kPer;
  const bool is_q = row < rr.rows_q;
  const long r = is_q ? row : row - rr.rows_q;
  const __nv_bfloat16* x = (is_q ? q : k) + r * D;
  __half* y = (is_q ? qo : ko) + r * D;
  long pos;
  if constexpr (PACKED) {
    const long tok = r / (is_q ? rr.Hq : rr.Hkv);
    if (tok < rr.cu[0] || tok >= rr.cu[rr.num_seqs]) {  // in no sequence: never read by the attention
      *reinterpret_cast<uint4*>(y + i0) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(y + H + i0) = make_uint4(0, 0, 0, 0);
      return;
    }
    int lo = 0, hi = rr.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (rr.cu[mid] <= tok) lo = mid;
      else hi = mid - 1;
    }
    pos = tok - rr.cu[lo];
  } else {
    pos = r % rr.T;
  }
  if (pos < 0 || pos >= rr.n_table) {
    if (i0 == 0) atomicCAS(rr.status, 0, kDevBadSeqlens);
    *reinterpret_cast<uint4*>(y + i0) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(y + H + i0) = make_uint4(0, 0, 0, 0);
    return;
  }
  const float* cs = cos_sin + pos * D;
  const uint4 lo = *reinterpret_cast<const uint4*>(x + i0), hi = *reinterpret_cast<const uint4*>(x + H + i0);
  const float4 c0 = *reinterpret_cast<const float4*>(cs + i0), c1 = *reinterpret_cast<const float4*>(cs + i0 + 4);
  const float4 s0 = *reinterpret_cast<const float4*>(cs + H + i0);
  const float4 s1 = *reinterpret_cast<const float4*>(cs + H + i0 + 4);
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  const uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w}, wh[4] = {hi.x, hi.y, hi.z, hi.w};
  uint32_t ol[4], oh[4];
  // f16 holds magnitudes below 65520 (larger ones round to infinity): a
  // value outside that, or not finite, is reported (ATTN_ERR_RANGE) and
  // written as f16 rounds it
  bool fits = true;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wl[e]));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wh[e]));
    const float l0 = fmaf(a.x, c[2 * e], -b.x * sn[2 * e]), l1 = fmaf(a.y, c[2 * e + 1], -b.y * sn[2 * e + 1]);
    const float h0 = fmaf(b.x, c[2 * e], a.x * sn[2 * e]), h1 = fmaf(b.y, c[2 * e + 1], a.y * sn[2 * e + 1]);
    fits = fits && fabsf(l0) < 65520.f && fabsf(l1) < 65520.f && fabsf(h0) < 65520.f && fabsf(h1) < 65520.f;
    const __half2 yl = __floats2half2_rn(l0, l1);
    const __half2 yh = __floats2half2_rn(h0, h1);
    ol[e] = *reinterpret_cast<const uint32_t*>(&yl);
    oh[e] = *reinterpret_cast<const uint32_t*>(&yh);
  }
  if (!fits) atomicCAS(rr.status, 0, kDevRange);
  *reinterpret_cast<uint4*>(y + i0) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
  *reinterpret_cast<uint4*>(y + H + i0) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
}

}  // namespace

cudaError_t launch_rope_qk_f16(const void* q, const void* k, void* q_out, void* k_out, const RopeRows& rr, int D,
                               const float* cos_sin, cudaStream_t stream) {
  const long threads = (rr.rows_q + rr.rows_k) * (D / 16);
  const long blocks = (threads + 255) / 256;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffL) return cudaErrorInvalidValue;
  auto qi = static_cast<const __nv_bfloat16*>(q);
  auto ki = static_cast<const __nv_bfloat16*>(k);
  auto qo = static_cast<__half*>(q_out);
  auto ko = static_cast<__half*>(k_out);
  const unsigned g = (unsigned)blocks;
  const bool packed = rr.cu != nullptr;
  if (D == 128) {
    if (packed) rope_qk_f16_kernel<128, true><<<g, 256, 0, stream>>>(qi, ki, qo, ko, rr, cos_sin);
    else rope_qk_f16_kernel<128, false><<<g, 256, 0, stream>>>(qi, ki, qo, ko, rr, cos_sin);
  } else {
    if (packed) rope_qk_f16_kernel<64, true><<<g, 256, 0, stream>>>(qi, ki, qo, ko, rr, cos_sin);
    else rope_qk_f16_kernel<64, false><<<g, 256, 0, stream>>>(qi, ki, qo, ko, rr, cos_sin);
  }
  return cudaGetLastError();
}

}  // namespace gqa
