// attn_decode.cu -- cached (decode) grouped-query attention for sm_103a.
//
// The newest Tq positions of each batch row attend to that row's KV cache:
// query t of row b sits at position cache_lens[b] - Tq + t and sees the
// cached keys j <= cache_lens[b] - Tq + t (the causal mask aligned to the end
// of the cache).  This is the cached GQA / per-row-prefix cached attention of
// the microLLM-rocm README, section "Why this project exists" (KV-cache
// decode for batch rows B1/2/4/8).  A few query rows meet a long stream of
// keys, so the work is bound by reading the cache from HBM; it runs on the
// CUDA cores, and the design is about keeping that stream full:
//
//   decode_partial  persistent, one CTA per SM.  Work items are (batch row,
//     K/V head, block of <= 16 query rows, split of the key range); a CTA
//     takes items blockIdx.x, blockIdx.x + gridDim.x, ...  Warp 8 is the
//     producer: it TMA-loads 128-key K/V chunks (128-byte swizzled boxes)
//     into a ring of stages, running ahead across item boundaries, and
//     stages each item's query rows in shared memory as f32.  Warps 0-7 are
//     consumers in two groups that take alternate chunks; inside a group,
//     warp w owns keys [32w, 32w+32) of the chunk.  Per chunk a warp scores
//     its keys (lane = key) against every query row of the block, updates
//     its own running max / sum (log2 units), writes the probabilities to a
//     warp-private buffer and accumulates P V with each lane owning 2 (or 4)
//     output features.  At the end of an item the eight warps' states are
//     combined in the stage that held the item's last chunk and written
//     out: the final O / LSE when the key range is not split, else an
//     unnormalised partial with its max and sum.
//   decode_merge  combines a row's splits with the usual rescaling.
#include "sm103.cuh"
#include "kernels.h"

namespace gqa {

namespace {

constexpr int kCK = 128;          // keys per chunk (rows of one TMA box)
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kBoxBytes = kCK * 128;  // one 64-feature x 128-key bf16 box

template <int D, int RB>
struct DecCfg {
  static constexpr int kChunkBytes = 2 * (D / 64) * kBoxBytes;  // K then V
  static constexpr int kStages = D == 128 ? 3 : 6;
  static constexpr int kOffQ = kStages * kChunkBytes;          // f32 [2][RB][D]
  static constexpr int kOffP = kOffQ + 2 * RB * D * 4;          // f32 [8 warps][32][RB]
  static constexpr int kOffML = kOffP + kConsumerWarps * 32 * RB * 4;  // float2 [8][RB]
  static constexpr int kSmemBytes = kOffML + kConsumerWarps * RB * 8 + 1024;  // + alignment slack
  static_assert(kConsumerWarps * RB * D * 4 <= kChunkBytes, "item combine must fit in one stage");
  static_assert(kSmemBytes + 256 <= 232448, "shared memory");
};

struct __align__(8) DecBarriers {
  uint64_t full[6];
  uint64_t empty[6];
  uint64_t qfull[2];
  uint64_t qempty[2];
  int abort;
};

// One work item, decoded identically by the producer and every consumer.
struct Item {
  int bh, b, hkv, rb, split;
  int r0, rows;       // query rows [r0, r0 + rows) of the group's R rows
  int len;            // keys in the row's cache
  int kbeg, nch;      // first key of the split, chunks in it (0: nothing to do)
};

__device__ __forceinline__ Item decode_item(const DecodeArgs& a, int item, int RBmax) {
  Item it;
  it.bh = item % (a.B * a.Hkv);
  const int rest = item / (a.B * a.Hkv);
  it.rb = rest % a.nrb;
  it.split = rest / a.nrb;
  it.b = it.bh / a.Hkv;
  it.hkv = it.bh % a.Hkv;
  it.r0 = it.rb * RBmax;
  it.rows = min(RBmax, a.R - it.r0);
  it.len = a.cache_lens[it.b];
  it.kbeg = it.split * a.cps * kCK;
  it.nch = 0;
  if (it.len >= a.Tq && it.len <= a.S && it.kbeg < it.len) {
    const int kend = min(it.len, it.kbeg + a.cps * kCK);
    it.nch = (kend - it.kbeg + kCK - 1) / kCK;
  }
  return it;
}

__device__ __forceinline__ float warp_max(float x) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// bf16 pair (low half = first element) -> two f32 in one 64-bit register pair
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t x) {
  return f2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

}  // namespace

template <int D, int RB>
__global__ void __launch_bounds__(kThreads, 1)
    decode_partial_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const DecodeArgs a) {
  using C = DecCfg<D, RB>;
  constexpr int S = C::kStages;
  constexpr int NB = D / 64;  // boxes (64 features each) per K or V chunk
  constexpr int kSU = RB <= 8 ? D / 8 : 2;  // score loop unroll (16-byte K pieces)
  constexpr int kPU = RB <= 8 ? 4 : 2;      // keys per P V step
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* sQ = reinterpret_cast<float*>(smem + C::kOffQ);
  float* sPall = reinterpret_cast<float*>(smem + C::kOffP);
  float2* sML = reinterpret_cast<float2*>(smem + C::kOffML);
  __shared__ DecBarriers bars;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Guard guard{&bars.abort, a.status};
  if (threadIdx.x == 0) {
    bars.abort = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(&bars.full[i], 1);
      mbar_init(&bars.empty[i], 4);              // the four warps of the consuming group
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.qfull[i], 1);
      mbar_init(&bars.qempty[i], kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    int cs = 0, uses = 0;
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
      const Item it = decode_item(a, item, RB);
      if (it.len < a.Tq || it.len > a.S) {
        if (lane == 0 && it.rb == 0 && it.split == 0 && it.hkv == 0) atomicCAS(a.status, 0, kDevBadSeqlens);
      }
      if (it.nch == 0) continue;
      // query rows of the block -> f32 shared memory (rows past `rows` are zero)
      const int slot = uses & 1;
      if (uses >= 2) mbar_wait(&bars.qempty[slot], ((uses >> 1) - 1) & 1, guard);
      const __nv_bfloat16* qg = a.q + (((long)it.b * a.Hq + (long)it.hkv * a.G) * a.Tq + it.r0) * D;
      float* sq = sQ + slot * RB * D;
      for (int idx = lane; idx < RB * D / 8; idx += 32) {
        const int r = idx / (D / 8);
        uint4 x = make_uint4(0, 0, 0, 0);
        if (r < it.rows) x = *reinterpret_cast<const uint4*>(qg + (long)idx * 8);
        float4 lo, hi;
        lo.x = __uint_as_float(x.x << 16); lo.y = __uint_as_float(x.x & 0xffff0000u);
        lo.z = __uint_as_float(x.y << 16); lo.w = __uint_as_float(x.y & 0xffff0000u);
        hi.x = __uint_as_float(x.z << 16); hi.y = __uint_as_float(x.z & 0xffff0000u);
        hi.z = __uint_as_float(x.w << 16); hi.w = __uint_as_float(x.w & 0xffff0000u);
        reinterpret_cast<float4*>(sq)[2 * idx] = lo;
        reinterpret_cast<float4*>(sq)[2 * idx + 1] = hi;
      }
      mbar_arrive_warp(&bars.qfull[slot]);
      ++uses;
      // K/V chunks of the item
      for (int c = 0; c < it.nch; ++c, ++cs) {
        const int stage = cs % S, fill = cs / S;
        if (fill >= 1) mbar_wait(&bars.empty[stage], (fill - 1) & 1, guard);
        if (lane == 0) {
          uint8_t* dst = smem + stage * C::kChunkBytes;
          uint64_t* bar = &bars.full[stage];
          if (guard.aborted()) {
            mbar_arrive(bar);  // nothing loaded; consumers run on without data and write nothing
          } else {
            mbar_expect_tx(bar, C::kChunkBytes);
            const int y = it.kbeg + c * kCK;
#pragma unroll
            for (int x = 0; x < NB; ++x) {
              tma_load_3d(dst + x * kBoxBytes, &tm_k, bar, x * 64, y, it.bh);
              tma_load_3d(dst + (NB + x) * kBoxBytes, &tm_v, bar, x * 64, y, it.bh);
            }
          }
        }
        __syncwarp();
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int group = warp >> 2, wg = warp & 3;
  float* sP = sPall + warp * 32 * RB;
  const int j = 32 * wg + lane;  // this lane's key within a chunk (score phase)
  int cs = 0, uses = 0;
  for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
    const Item it = decode_item(a, item, RB);
    if (it.nch == 0) continue;
    const int slot = uses & 1;
    mbar_wait(&bars.qfull[slot], (uses >> 1) & 1, guard);
    const float* sq = sQ + slot * RB * D;
    float m[RB], l[RB];
    uint64_t o[RB][NB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      m[r] = -INFINITY;
      l[r] = 0.f;
#pragma unroll
      for (int x = 0; x < NB; ++x) o[r][x] = 0;
    }
    const int last_vis0 = it.len - a.Tq;  // last visible key of a row with t = 0

    for (int c = 0; c < it.nch; ++c) {
      const int csc = cs + c;
      if ((csc & 1) != group) continue;
      const int stage = csc % S;
      mbar_wait(&bars.full[stage], (csc / S) & 1, guard);
      const uint8_t* sK = smem + stage * C::kChunkBytes;
      const uint8_t* sV = sK + NB * kBoxBytes;
      const int k0 = it.kbeg + c * kCK;
      const int nvis = min(kCK, it.len - k0);  // keys of the chunk inside the cache

      // scores: lane = key j, all RB rows, f32x2 accumulation
      uint64_t acc[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) acc[r] = 0;
#pragma unroll kSU
      for (int cc = 0; cc < D / 8; ++cc) {
        const int box = cc >> 3, ch = cc & 7;
        const uint4 kx = *reinterpret_cast<const uint4*>(sK + box * kBoxBytes + j * 128 + ((ch ^ (j & 7)) << 4));
        const uint64_t k01 = bf2_to_f2(kx.x), k23 = bf2_to_f2(kx.y), k45 = bf2_to_f2(kx.z),
                       k67 = bf2_to_f2(kx.w);
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(sq + r * D + cc * 8);
          const ulonglong2 qb = *reinterpret_cast<const ulonglong2*>(sq + r * D + cc * 8 + 4);
          uint64_t t = acc[r];
          t = fma2(qa.x, k01, t);
          t = fma2(qa.y, k23, t);
          t = fma2(qb.x, k45, t);
          t = fma2(qb.y, k67, t);
          acc[r] = t;
        }
      }
      // online softmax per row over this warp's 32 keys
      const int kpos = k0 + j;
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        float lo, hi;
        f2_split(acc[r], lo, hi);
        const int t = (it.r0 + r) % a.Tq;
        const float s = (j < nvis && kpos <= last_vis0 + t) ? (lo + hi) * a.scale_log2 : -INFINITY;
        const float m_new = fmaxf(m[r], warp_max(s));
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = ex2_approx(m[r] - m_use);
        const float p = ex2_approx(s - m_use);
        l[r] = fmaf(l[r], alpha, p);
        m[r] = m_new;
        const uint64_t al = f2(alpha, alpha);
#pragma unroll
        for (int x = 0; x < NB; ++x) o[r][x] = mul2(o[r][x], al);
        sP[lane * RB + r] = p;
      }
      __syncwarp();
      // O += P V over this warp's keys; lane owns features (2*lane, 2*lane+1) of each box.
      // kPU keys per step: their shared-memory loads are issued before the FMAs.
      const int nk = min(32, nvis - 32 * wg);
      int jj = 0;
      for (; jj + kPU <= nk; jj += kPU) {
        uint64_t v2[kPU][NB];
        float4 p4[kPU][RB / 4];
#pragma unroll
        for (int u = 0; u < kPU; ++u) {
          const int row = 32 * wg + jj + u;
          const int voff = row * 128 + (((lane >> 2) ^ (row & 7)) << 4) + 4 * (lane & 3);
#pragma unroll
          for (int x = 0; x < NB; ++x)
            v2[u][x] = bf2_to_f2(*reinterpret_cast<const uint32_t*>(sV + x * kBoxBytes + voff));
#pragma unroll
          for (int r4 = 0; r4 < RB / 4; ++r4) p4[u][r4] = *reinterpret_cast<const float4*>(sP + (jj + u) * RB + 4 * r4);
        }
#pragma unroll
        for (int u = 0; u < kPU; ++u)
#pragma unroll
          for (int r4 = 0; r4 < RB / 4; ++r4) {
            const float pv[4] = {p4[u][r4].x, p4[u][r4].y, p4[u][r4].z, p4[u][r4].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint64_t pp = f2(pv[e], pv[e]);
#pragma unroll
              for (int x = 0; x < NB; ++x) o[4 * r4 + e][x] = fma2(pp, v2[u][x], o[4 * r4 + e][x]);
            }
          }
      }
      for (; jj < nk; ++jj) {
        const int row = 32 * wg + jj;
        const int voff = row * 128 + (((lane >> 2) ^ (row & 7)) << 4) + 4 * (lane & 3);
        uint64_t v2[NB];
#pragma unroll
        for (int x = 0; x < NB; ++x)
          v2[x] = bf2_to_f2(*reinterpret_cast<const uint32_t*>(sV + x * kBoxBytes + voff));
#pragma unroll
        for (int r4 = 0; r4 < RB; r4 += 4) {
          const float4 p4 = *reinterpret_cast<const float4*>(sP + jj * RB + r4);
          const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint64_t pp = f2(pv[e], pv[e]);
#pragma unroll
            for (int x = 0; x < NB; ++x) o[r4 + e][x] = fma2(pp, v2[x], o[r4 + e][x]);
          }
        }
      }
      __syncwarp();
      if (c != it.nch - 1) mbar_arrive_warp(&bars.empty[stage]);
    }

    // ------------------------------------------------ combine the 8 warps
    const int cs_last = cs + it.nch - 1;
    float* scratch = reinterpret_cast<float*>(smem + (cs_last % S) * C::kChunkBytes);  // [8][RB][D]
    named_bar_sync(1, kConsumerWarps * 32);  // every warp is done with the item's chunks
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const float lw = warp_sum(l[r]);
      if (lane == 0) sML[warp * RB + r] = make_float2(m[r], lw);
#pragma unroll
      for (int x = 0; x < NB; ++x)
        *reinterpret_cast<uint64_t*>(scratch + (warp * RB + r) * D + x * 64 + 2 * lane) = o[r][x];
    }
    named_bar_sync(1, kConsumerWarps * 32);
    const bool single = a.n_splits == 1;
    for (int e = threadIdx.x; e < it.rows * D; e += kConsumerWarps * 32) {
      const int r = e / D, d = e % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sML[w * RB + r].x);
      const float Mu = M == -INFINITY ? 0.f : M;
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float2 ml = sML[w * RB + r];
        const float wgt = ex2_approx(ml.x - Mu);
        L = fmaf(ml.y, wgt, L);
        O = fmaf(scratch[(w * RB + r) * D + d], wgt, O);
      }
      if (guard.aborted()) continue;
      const int rg = it.r0 + r;  // row within the group: query head (rg / Tq), position t (rg % Tq)
      if (single) {
        const long orow = ((long)it.b * a.Hq + (long)it.hkv * a.G) * a.Tq + rg;
        a.o[orow * D + d] = __float2bfloat16_rn(O / L);
        if (d == 0) a.lse[orow] = (M + __log2f(L)) * 0.69314718055994531f;
      } else {
        const long prow = ((long)it.bh * a.n_splits + it.split) * a.R + rg;
        a.ws_o[prow * D + d] = O;
        if (d == 0) a.ws_ml[prow] = make_float2(M, L);
      }
    }
    fence_proxy_async_smem();  // generic accesses to the stage before the next TMA write into it
    named_bar_sync(1, kConsumerWarps * 32);
    if ((cs_last & 1) == group) mbar_arrive_warp(&bars.empty[cs_last % S]);
    mbar_arrive_warp(&bars.qempty[slot]);
    cs += it.nch;
    ++uses;
  }
}

// One CTA per output row (b, h, t).  Warp 0 turns the splits' (max, sum)
// pairs into weights 2^(m_s - M) / L in shared memory; then every thread
// (= feature) sums its weighted partials with independent loads.  Splits
// that hold no key visible to the row (max = -inf) get weight 0.
constexpr int kMergeMaxSplits = 1024;

__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeArgs a) {
  __shared__ float s_w[kMergeMaxSplits];
  __shared__ float s_lse;
  const int row = blockIdx.x;  // (b * Hq + h) * Tq + t
  const int t = row % a.Tq, bq = row / a.Tq;
  const int h = bq % a.Hq, b = bq / a.Hq;
  const int len = a.cache_lens[b];
  if (len < a.Tq || len > a.S) return;
  const int bh = b * a.Hkv + h / a.G;
  const int rg = (h % a.G) * a.Tq + t;
  const int n_act = min(((len + kCK - 1) / kCK + a.cps - 1) / a.cps, kMergeMaxSplits);
  const float2* ml = a.ws_ml + (long)bh * a.n_splits * a.R + rg;
  const float* wo = a.ws_o + ((long)bh * a.n_splits * a.R + rg) * a.D;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float M = -INFINITY;
    for (int s = lane; s < n_act; s += 32) M = fmaxf(M, ml[(long)s * a.R].x);
    M = warp_max(M);
    float L = 0.f;
    for (int s = lane; s < n_act; s += 32) {
      const float2 v = ml[(long)s * a.R];
      const float w = v.x == -INFINITY ? 0.f : ex2_approx(v.x - M);
      s_w[s] = w;
      L = fmaf(v.y, w, L);
    }
    L = warp_sum(L);
    const float inv = 1.f / L;
    for (int s = lane; s < n_act; s += 32) s_w[s] *= inv;
    if (lane == 0) s_lse = (M + __log2f(L)) * 0.69314718055994531f;
  }
  __syncthreads();
  for (int d = threadIdx.x; d < a.D; d += blockDim.x) {
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    int s = 0;
    for (; s + 4 <= n_act; s += 4) {
      const float x0 = wo[(long)s * a.R * a.D + d], x1 = wo[(long)(s + 1) * a.R * a.D + d];
      const float x2 = wo[(long)(s + 2) * a.R * a.D + d], x3 = wo[(long)(s + 3) * a.R * a.D + d];
      acc0 = fmaf(x0, s_w[s], acc0);
      acc1 = fmaf(x1, s_w[s + 1], acc1);
      acc2 = fmaf(x2, s_w[s + 2], acc2);
      acc3 = fmaf(x3, s_w[s + 3], acc3);
    }
    for (; s < n_act; ++s) acc0 = fmaf(wo[(long)s * a.R * a.D + d], s_w[s], acc0);
    a.o[(long)row * a.D + d] = __float2bfloat16_rn((acc0 + acc1) + (acc2 + acc3));
  }
  if (threadIdx.x == 0) a.lse[row] = s_lse;
}

template <int D, int RB>
static cudaError_t launch_decode_rb(const CUtensorMap& k, const CUtensorMap& v, const DecodeArgs& a, int grid,
                                    cudaStream_t stream) {
  using C = DecCfg<D, RB>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<D, RB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  prof_begin(kProfDecode, stream);
  decode_partial_kernel<D, RB><<<grid, kThreads, C::kSmemBytes, stream>>>(k, v, a);
  prof_end(stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.n_splits == 1) return e;
  prof_begin(kProfDecodeMerge, stream);
  decode_merge_kernel<<<a.B * a.Hq * a.Tq, D, 0, stream>>>(a);
  prof_end(stream);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_decode_d(const CUtensorMap& k, const CUtensorMap& v, const DecodeArgs& a, int grid,
                                   cudaStream_t stream) {
  if (a.rb_rows == 4) return launch_decode_rb<D, 4>(k, v, a, grid, stream);
  if (a.rb_rows == 8) return launch_decode_rb<D, 8>(k, v, a, grid, stream);
  return launch_decode_rb<D, 16>(k, v, a, grid, stream);
}

cudaError_t launch_attn_decode(const CUtensorMap& k, const CUtensorMap& v, const DecodeArgs& a, int grid,
                               cudaStream_t stream) {
  if (a.D == 128) return launch_decode_d<128>(k, v, a, grid, stream);
  return launch_decode_d<64>(k, v, a, grid, stream);
}

}  // namespace gqa
