// attn_decode.cu -- cached (decode) grouped-query attention for sm_103a.
//
// The newest Tq positions of each batch row attend to that row's KV cache:
// query t of row b sits at position cache_lens[b] - Tq + t and sees the
// cached keys j <= cache_lens[b] - Tq + t (the causal mask aligned to the end
// of the cache).  This is the cached GQA / per-row-prefix cached attention of
// the microLLM-rocm README, section "Why this project exists" (KV-cache
// decode for batch rows B1/2/4/8).  A few query rows meet a long stream of
// keys: the kernel has to keep the HBM stream full, and with G query heads
// per K/V head it does G flops per cache byte, more than the CUDA cores
// sustain next to that stream -- so both contractions run on tcgen05 with
// the long side (128 keys, or the D features) as M and the query rows as N:
//
//   S^T[key][row]  = sum_d K[key][d] Q[row][d]          (M = 128 keys, N = 16)
//   O^T[d][row]   += sum_key V[key][d] P[row][key]       (M = 128 features, N = 16)
//
// decode_partial  persistent, one CTA per SM.  The work is a stream of
//   128-key chunks: unit by unit (batch row, K/V head, block of 16 query
//   rows), each unit's chunks in key order.  CTA c takes the contiguous
//   share [c*C/G, (c+1)*C/G) of the C chunks, so every CTA streams the same
//   number of chunks whatever the rows' lengths.  A share cuts units into
//   pieces; a unit processed as one piece writes O / LSE, the pieces of a
//   cut unit write partials that decode_merge combines.
//   Roles (256 threads; 384 for E4M3 caches, below):
//   warp 0     producer: TMA-loads the share's 128-key K chunks (128-byte
//              swizzled boxes) into the K ring, running ahead across pieces
//              (paged caches: one box per page, the pages looked up in the
//              block table by the warp's lanes before the slot wait).
//   warp 6     producer of the V ring.  K and V have rings of their own: a
//              K chunk is released as soon as its score MMA is done, a V
//              chunk only after P V, so K refills run further ahead.
//   warp 1     score MMA issuer (S^T into a double buffer, so the softmax of
//              one chunk overlaps the score MMA of the next); TMEM owner;
//              TMA-loads each piece's 16 query rows one piece ahead (a
//              K-major swizzled tile); with a rotary table it first rotates
//              them in place at their positions (positions-aware RoPE),
//              keeping the rounding remainder in a second bf16 tile that a
//              second set of score MMAs adds in.
//   warp 7     P V MMA issuer: O^T += V^T P^T as soon as a chunk's P and V
//              are ready, independently of the score issuer.
//   warps 2-5  softmax: thread = key for S^T (and = feature for O^T); row
//              maxima cross the four warps through shared memory; P (bf16)
//              goes to a K-major swizzled tile; O^T is rescaled lazily, only
//              when a row's maximum grows by more than 2^8; at the end of an
//              item they write O / LSE (unsplit key range) or an unnormalised
//              partial with its max and sum.
// TMEM: S^T buffers at columns 0 and 16, O^T buffers at 32 and 48.
//
// E4M3 (FP8) caches, one scale per cache: K and V arrive as 8-bit codes,
//   half the bytes of bf16.  The score MMA reads the K codes as they land
//   (kind::f8f6f4, E4M3 x E4M3): the score issuer splits each piece's query
//   rows into three E4M3 parts with a scale per row, q = s_r (h0 + h1 + h2)
//   to about 2^-12, and all three accumulate into the same S^T, which the
//   softmax multiplies by s_r.  V lands in a staging ring; four converter
//   warps (8-11, 384 threads in all, one per SM sub-partition beside its
//   softmax warp) convert each landed chunk to f16 (exact) into an operand
//   tile, one key row per thread, so the P V MMA stays kind::f16 with an
//   f16 P.  k_scale is folded into the score scale, v_scale into the output.
//
// decode_merge  combines the pieces of a cut unit with the usual rescaling;
//   it is launched as a programmatic dependent of decode_partial, so its
//   launch overlaps the partial kernel's tail.
#include <cuda_fp16.h>

#include "sm103.cuh"
#include "kernels.h"

namespace gqa {

namespace {

constexpr int kCK = 128;                  // keys per chunk (rows of one TMA box; M of the score MMA)
constexpr int kRows = 16;                 // query rows per piece (N of both MMAs)
constexpr int kBoxBytes = kCK * 128;      // 64 features x 128 keys, bf16
constexpr int kRowBoxBytes = kRows * 128; // 64 features (or keys) x 16 rows, bf16
constexpr int kThreads = 256;             // 16-bit caches: 8 warps
constexpr int kThreads8 = 384;            // E4M3 caches: 8 warps + 4 V converter warps
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// kind::f16 instruction descriptor with f32 accumulation and bf16 (f16 = false)
// or f16 (f16 = true) A and B.
__host__ __device__ constexpr uint32_t idesc_16(int M, int N, bool a_mn, bool b_mn, bool f16) {
  return f16 ? (idesc_bf16(M, N, a_mn, b_mn) & ~((7u << 7) | (7u << 10))) : idesc_bf16(M, N, a_mn, b_mn);
}

// TMEM columns (lane = key of the chunk for S^T, feature for O^T): two S^T
// buffers, then two O^T buffers of kRows columns.  A score MMA stacks the
// query operand's parts along N -- the three E4M3 part tiles, or a rotary
// query's bf16 value and remainder rows -- so the S^T buffers are 3 (2)
// kRows wide and the softmax adds the column groups.
template <bool FP8>
constexpr int kSCols = (FP8 ? 3 : 2) * kRows;
template <bool FP8>
constexpr uint32_t kTmemCols = FP8 ? 128 : 64;
template <bool FP8>
__device__ __forceinline__ uint32_t col_s(int b) { return (uint32_t)(b * kSCols<FP8>); }
template <bool FP8>
__device__ __forceinline__ uint32_t col_o(int b) { return (uint32_t)(2 * kSCols<FP8> + b * kRows); }

template <int D, bool FP8>
struct DecCfg {
  static constexpr int NB = D / 64;                       // 64-feature boxes per K or V chunk
  static constexpr int kTileBytes = NB * kBoxBytes;       // one K or V chunk as a 16-bit MMA operand
  static constexpr int kTile8 = kCK * D;                  // one chunk of 8-bit codes, rows of D bytes
  // bf16 caches: a K ring and a V ring of kSlotsK operand tiles each.
  // FP8 caches: a K ring of kSlotsK 8-bit tiles (the score MMA reads the
  // codes as they land), a V staging ring of kSlotsV 8-bit tiles, and kVop
  // f16 V operand tiles (chunk i is converted into tile i % kVop).  Loads
  // take microseconds to land under full load, so the shared memory goes to
  // 8-bit slots in flight rather than to a second operand tile.
  static constexpr int kSlotsK = FP8 ? (D == 128 ? 6 : 8) : (D == 128 ? 3 : 6);
  static constexpr int kSlotsV = FP8 ? (D == 128 ? 4 : 8) : kSlotsK;
  static constexpr int kVop = FP8 ? (D == 128 ? 1 : 2) : 0;
  static constexpr int kTileK = FP8 ? kTile8 : kTileBytes;          // bytes per K ring slot
  static constexpr int kOffV = kSlotsK * kTileK;                    // V ring / FP8 V operand tiles
  static constexpr int kOffStage = kOffV + (FP8 ? kVop : kSlotsV) * kTileBytes;  // FP8 V staging ring
  static constexpr int kOffQ = kOffStage + (FP8 ? kSlotsV * kTile8 : 0);
  static constexpr int kQBytes = NB * kRowBoxBytes;       // 16 query rows, bf16, K-major
  // query slots (one per piece, two pieces): bf16 caches, per 64-feature box
  // the 16 value rows then the 16 remainder rows (rotary queries), so that
  // one 32-row K-major operand covers both; FP8 [bf16 tile] followed by
  // [three E4M3 part tiles] per slot
  static constexpr int kQBoxStride = (FP8 ? 1 : 2) * kRowBoxBytes;
  static constexpr int kQSlot = NB * kQBoxStride;
  static constexpr int kQ8Bytes = kRows * D;              // one E4M3 part: 16 rows of D bytes, K-major
  static constexpr int kOffQ8 = kOffQ + 2 * kQSlot;
  static constexpr int kPBytes = 2 * kRowBoxBytes;        // 16 rows x 128 keys, K-major
  static constexpr int kOffP = kOffQ8 + (FP8 ? 2 * 3 * kQ8Bytes : 0);
  static constexpr int kOffMax = kOffP + 2 * kPBytes;           // f32 [2][16 rows][4 warps]
  static constexpr int kOffSum = kOffMax + 2 * kRows * 4 * 4;   // f32 [16 rows][4 warps]
  static constexpr int kOffFin = kOffSum + kRows * 4 * 4;       // float2 [2 pieces][16 rows]: (max, sum)
  static constexpr int kOffQs = kOffFin + 2 * kRows * 8;        // f32 [2 slots][16 rows]: FP8 query row scales
  static constexpr int kSmemBytes = kOffQs + 2 * kRows * 4 + 1024;  // + alignment slack
  // score MMA: bf16 x bf16 (kind::f16), or E4M3 K codes x E4M3 query parts
  // (kind::f8f6f4, format code 0 for both); P V MMA: bf16, or f16 V and P
  static constexpr uint32_t kIdescS = idesc_16(kCK, kSCols<FP8>, false, false, FP8);
  static constexpr uint32_t kIdescS1 = idesc_16(kCK, kRows, false, false, FP8);   // bf16, plain queries
  static constexpr uint32_t kIdescO = idesc_16(128, kRows, true, false, FP8);
  // V^T as an MN-major A operand of 128 rows: the second 64-feature atom is
  // the second box (D = 128) or the first one again (D = 64; rows 64-127 of
  // O^T are then a copy and are never read).
  static constexpr uint32_t kLboV = D == 128 ? kBoxBytes : 0;
  static constexpr int kMaxSlots = kSlotsK > kSlotsV ? kSlotsK : kSlotsV;
  static_assert(kMaxSlots <= 8, "barrier arrays");
  static_assert(kSmemBytes + 2048 <= 232448, "shared memory (dynamic + static: barriers, lengths)");
};

// One piece: a run of a unit's chunks inside one CTA's share.
struct Piece {
  int u, b, hkv, bh;
  int r0, rows;       // query rows [r0, r0 + rows) of the group's R rows
  int len;            // keys in the row's cache
  int kbeg, nch;      // first key of the piece, chunks in it
  int slot, npieces;  // piece index within its unit, pieces of the unit
};

struct __align__(8) DecBarriers {
  uint64_t k_full[8], k_empty[8];
  uint64_t v_full[8], v_empty[8];  // FP8: the V staging ring (emptied by the converter warps)
  uint64_t vo_full[2];             // FP8: an f16 V operand tile is ready (per tile)
  uint64_t q_full[2], q_empty[2];
  uint64_t qs_full[2], qs_empty[2];  // FP8: a piece's query parts and row scales are ready / read
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], p_empty[2];
  uint64_t o_full[2], o_empty[2];
  uint64_t teardown[2];
  uint32_t tmem_base;
  int abort;
};

constexpr int kDevBadPages = 11;  // device status: a block-table entry names no page (ATTN_ERR_PAGES)

constexpr int kLenCache = 256;  // batch rows whose lengths are kept in shared memory (larger batches read them from global memory)

// Chunks of batch row b's cache: ceil(len / 128), 0 for an invalid length.
// `lens` is the shared-memory copy of cache_lens (B <= kLenCache) or cache_lens itself.
__device__ __forceinline__ int row_chunks(const DecodeArgs& a, const int* lens, int b, int& len) {
  len = lens[b];
  return (len >= a.Tq && len <= a.S) ? (len + kCK - 1) / kCK : 0;
}

// The CTA's share of the chunk stream.  The stream holds the chunks of every
// unit in order (units u = 0, 1, ..., each unit's chunks in key order); of
// its C chunks, CTA c < G takes [c*C/G, (c+1)*C/G), G = min(CTAs, C) so
// that no share is empty.
struct Share {
  long C;
  int G;
  long g0, g1;    // this CTA's share
  int b0;         // batch row holding chunk g0
  long P0;        // stream index of row b0's first chunk
};

// The CTA whose share holds stream chunk g.
__device__ __forceinline__ int owner_of(long g, long C, int G) { return (int)(((g + 1) * G - 1) / C); }

// Position in the CTA's stream of (piece, chunk) pairs; every role walks it.
struct Cursor {
  Piece it;
  int c;      // chunk within the piece
  int cs;     // chunk index in the CTA's stream
  int uses;   // pieces before this one
  bool valid;
  long g, g1; // stream index of the piece's first chunk; end of the share
  int b, nb;  // batch row of the piece, chunks per unit of that row
  long Pb;    // stream index of row b's first chunk
};

__device__ __forceinline__ void cursor_piece(const DecodeArgs& a, const Share& sh, Cursor& cur) {
  const int upb = a.Hkv * a.nrb;  // units per batch row
  const long off = cur.g - cur.Pb;
  const int k = (int)(off / cur.nb), cu = (int)(off % cur.nb);
  Piece& p = cur.it;
  p.b = cur.b;
  p.u = cur.b * upb + k;
  p.hkv = k / a.nrb;
  p.bh = cur.b * a.Hkv + p.hkv;
  p.r0 = (k % a.nrb) * kRows;
  p.rows = min(kRows, a.R - p.r0);
  p.kbeg = cu * kCK;
  p.nch = (int)min((long)(cur.nb - cu), cur.g1 - cur.g);
  const long Pu = cur.Pb + (long)k * cur.nb;
  const int first = owner_of(Pu, sh.C, sh.G);
  p.slot = (int)blockIdx.x - first;
  p.npieces = owner_of(Pu + cur.nb - 1, sh.C, sh.G) - first + 1;
  cur.valid = true;
}

__device__ __forceinline__ Cursor cursor_begin(const DecodeArgs& a, const Share& sh, const int* lens) {
  Cursor cur;
  cur.c = 0;
  cur.cs = 0;
  cur.uses = 0;
  cur.valid = false;
  cur.g = sh.g0;
  cur.g1 = sh.g1;
  if (sh.g0 >= sh.g1) return cur;
  cur.b = sh.b0;
  cur.Pb = sh.P0;
  cur.nb = row_chunks(a, lens, cur.b, cur.it.len);
  cursor_piece(a, sh, cur);
  return cur;
}

__device__ __forceinline__ void cursor_next(const DecodeArgs& a, const Share& sh, const int* lens, Cursor& cur) {
  ++cur.cs;
  if (++cur.c < cur.it.nch) return;
  cur.c = 0;
  ++cur.uses;
  cur.g += cur.it.nch;
  if (cur.g >= cur.g1) {
    cur.valid = false;
    return;
  }
  const long upb = (long)a.Hkv * a.nrb;
  while (cur.g >= cur.Pb + upb * cur.nb) {  // past row b: next row with chunks
    cur.Pb += upb * cur.nb;
    ++cur.b;
    cur.nb = row_chunks(a, lens, cur.b, cur.it.len);
  }
  cursor_piece(a, sh, cur);
}

// The share of CTA `cta` among G = min(ctas, C): one warp, lengths read
// through `lens`.  Used by the partial kernel (its own share) and by the
// merge kernel (to find how many pieces a unit was cut into).
__device__ Share find_share(const DecodeArgs& a, const int* lens, int cta, int ctas) {
  const int lane = threadIdx.x & 31;
  const long upb = (long)a.Hkv * a.nrb;
  long C = 0;
  for (int b0 = 0; b0 < a.B; b0 += 32) {
    int len = 0, n = 0;
    if (b0 + lane < a.B) n = row_chunks(a, lens, b0 + lane, len);
    C += upb * (long)__reduce_add_sync(0xffffffffu, (unsigned)n);
  }
  Share sh;
  sh.C = C;
  sh.G = (int)min((long)ctas, C);
  sh.g0 = cta < sh.G ? (long)cta * C / sh.G : 0;
  sh.g1 = cta < sh.G ? (long)(cta + 1) * C / sh.G : 0;
  sh.b0 = 0;
  sh.P0 = 0;
  if (sh.g0 < sh.g1) {
    long P = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
      int len = 0, n = 0;
      if (b0 + lane < a.B) n = row_chunks(a, lens, b0 + lane, len);
      long incl = upb * n;  // inclusive prefix over the 32 rows
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, P + incl > sh.g0);
      if (hit) {
        const int l = __ffs(hit) - 1;
        sh.b0 = b0 + l;
        sh.P0 = P + __shfl_sync(0xffffffffu, incl - upb * n, l);
        break;
      }
      P += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  return sh;
}

__device__ __forceinline__ float warp_max(float x) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}

// Named barrier over `n` threads that also ORs a predicate across them.
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %3, 0;\n\tbar.red.or.pred p, %1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(n), "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

}  // namespace

// D(tmem) (+)= A(smem) * B(smem)^T   (8-bit A and B, f32 accumulate; 32 K-elements per MMA)
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Shared-memory matrix descriptor for a 64-byte-swizzled K-major operand: rows of 64 bytes, 8-row
// groups `sbo` (512) bytes apart, 512-byte-aligned tile base.
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)4 << 61;  // 64-byte swizzle
  return d;
}

// Two E4M3 codes (low byte = first) as two f16 (low half = first): the
// hardware conversion, exact (every E4M3 value, NaN included, is an f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(codes));
  return d;
}

// Two f32 as E4M3 codes (low byte = lo), rounded to nearest even and
// saturated to +-448.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t codes) {
  const uint32_t h = e4m3x2_to_f16x2(codes);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Byte offset of 16-byte piece `c` of row r in an 8-bit K-major tile of
// D-byte rows as the TMA writes it and the MMA reads it: 128-byte swizzle
// (D = 128: piece c ^ (r % 8)) or 64-byte swizzle (D = 64: c ^ ((r / 2) % 4)).
template <int D>
__device__ __forceinline__ int swz8(int r, int c) {
  return r * D + ((D == 128 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3))) << 4);
}

// Key row j of a landed E4M3 V chunk (staging tile `st`, rows swizzled as
// swz8) into row j of the f16 operand tile `vo` (K-major, 128-byte swizzled
// boxes of 64 features), exact: one thread per row.  A row past the row's
// length (vis false: its codes may be anything, NaN included) is written as
// zeros so that 0 * V stays 0 in the P V MMA.
template <int D>
__device__ __forceinline__ void convert_v_row(const uint8_t* __restrict__ st, uint8_t* __restrict__ vo, int j,
                                              bool vis) {
  constexpr int kC = D / 16;  // 16-code pieces per row
#pragma unroll
  for (int c0 = 0; c0 < kC; c0 += 4) {
    uint4 x[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      x[k] = vis ? *reinterpret_cast<const uint4*>(st + swz8<D>(j, c0 + k)) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
      uint32_t h[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h[2 * e] = e4m3x2_to_f16x2((uint16_t)(w[e] & 0xffffu));
        h[2 * e + 1] = e4m3x2_to_f16x2((uint16_t)(w[e] >> 16));
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int f = 16 * (c0 + k) + 8 * half;  // first feature of this 16-byte operand piece
        *reinterpret_cast<uint4*>(vo + (f >> 6) * kBoxBytes + j * 128 + ((((f & 63) >> 3) ^ (j & 7)) << 4)) =
            make_uint4(h[4 * half], h[4 * half + 1], h[4 * half + 2], h[4 * half + 3]);
      }
    }
  }
}

// A piece's 16 query rows (bf16 tile as loaded: K-major, 128-byte swizzled
// boxes of 64 features) as three E4M3 part tiles and a scale per row, for
// the 8-bit score MMA against E4M3 K codes: with s_r = amax_r / 448 and
// x = q / s_r, h0 = e4m3(x), h1 = e4m3(x - h0), h2 = e4m3(x - h0 - h1), so
// that q = s_r (h0 + h1 + h2) to about 2^-12 of each element (or 2^-19 of
// the row's largest, for elements below E4M3's normal range).  All three
// parts accumulate into the same scores, which the softmax multiplies by
// s_r.  Rotary queries are rotated first, in f32, at the row's position
// (pairs i, i + D/2).  One warp, out of line: lane 2r + h makes the features
// [h D/2, (h + 1) D/2) of row r.
template <int D>
__device__ __noinline__ void q_tile_to_e4m3_parts(const uint8_t* qt, uint8_t* parts, float* qscale, const Piece& it,
                                                  const DecodeArgs& a, int lane) {
  constexpr int H = D / 2;
  const int r = lane >> 1, hh = lane & 1;
  auto ld8 = [&](int d) {  // bf16 features d .. d + 7 of row r
    return *reinterpret_cast<const uint4*>(qt + (d >> 6) * kRowBoxBytes + r * 128 + ((((d & 63) >> 3) ^ (r & 7)) << 4));
  };
  auto unpack = [](uint4 v, float* y) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      y[2 * e] = f.x;
      y[2 * e + 1] = f.y;
    }
  };
  const bool rope = a.rope_cs != nullptr && r < it.rows;
  const float* cs = rope ? a.rope_cs + (long)(it.len - a.Tq + (it.r0 + r) % a.Tq) * D : nullptr;
  // y = the 16 features 16 g .. 16 g + 15 of this lane's half
  auto load_y = [&](int g, float* y) {
    const int i0 = 16 * g;  // pair index (feature of the low half)
    if (!rope) {
      unpack(ld8(hh * H + i0), y);
      unpack(ld8(hh * H + i0 + 8), y + 8);
      return;
    }
    float lo[16], hi[16], c[16], sn[16];
    unpack(ld8(i0), lo);
    unpack(ld8(i0 + 8), lo + 8);
    unpack(ld8(H + i0), hi);
    unpack(ld8(H + i0 + 8), hi + 8);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float4 cv = *reinterpret_cast<const float4*>(cs + i0 + 4 * e);
      const float4 sv = *reinterpret_cast<const float4*>(cs + H + i0 + 4 * e);
      c[4 * e] = cv.x, c[4 * e + 1] = cv.y, c[4 * e + 2] = cv.z, c[4 * e + 3] = cv.w;
      sn[4 * e] = sv.x, sn[4 * e + 1] = sv.y, sn[4 * e + 2] = sv.z, sn[4 * e + 3] = sv.w;
    }
#pragma unroll
    for (int e = 0; e < 16; ++e)
      y[e] = hh == 0 ? fmaf(lo[e], c[e], -hi[e] * sn[e]) : fmaf(hi[e], c[e], lo[e] * sn[e]);
  };
  float amax = 0.f;
  for (int g = 0; g < H / 16; ++g) {
    float y[16];
    load_y(g, y);
#pragma unroll
    for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(y[e]));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  const float inv = amax > 0.f ? 448.f / amax : 1.f;
  for (int g = 0; g < H / 16; ++g) {
    float y[16];
    load_y(g, y);
    uint32_t p[3][4];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float x0 = y[2 * e] * inv, x1 = y[2 * e + 1] * inv;
      uint32_t code[3];
#pragma unroll
      for (int t = 0; t < 3; ++t) {
        const uint16_t cc = f32x2_to_e4m3x2(x0, x1);
        code[t] = cc;
        if (t < 2) {
          const float2 v = e4m3x2_to_float2(cc);
          x0 -= v.x;
          x1 -= v.y;
        }
      }
#pragma unroll
      for (int t = 0; t < 3; ++t) {
        if (e & 1) p[t][e >> 1] |= code[t] << 16;
        else p[t][e >> 1] = code[t];
      }
    }
    const int off = swz8<D>(r, (hh * H + 16 * g) >> 4);
#pragma unroll
    for (int t = 0; t < 3; ++t)
      *reinterpret_cast<uint4*>(parts + t * kRows * D + off) = make_uint4(p[t][0], p[t][1], p[t][2], p[t][3]);
  }
  if (hh == 0) qscale[r] = amax > 0.f ? amax * (1.f / 448.f) : 1.f;
}

// Rotary embedding of a piece's query rows (one warp, out of line), written
// back as bf16 value (over the loaded rows) plus bf16 remainder (the 16 rows
// under them in the same box): row r is query position t = (r0 + r) % Tq of
// its head, at position len - Tq + t of the row; feature i pairs with
// i + D/2 (rotate-half), x'_i = x_i c - x_{i+D/2} s,
// x'_{i+D/2} = x_{i+D/2} c + x_i s with c, s from the table row of that
// position.  The slot is K-major, 128-byte swizzled, one 4 KB box per 64
// features (value rows 0-15, remainder rows 16-31): feature d of row r sits
// in box d / 64, row r (value) or 16 + r (remainder), 16-byte chunk
// ((d % 64) / 8) ^ (r % 8).
template <int D>
__device__ __noinline__ void rope_rotate_tile(uint8_t* qs, const Piece& it, const DecodeArgs& a, int lane) {
  constexpr int H = D / 2;
  constexpr int kChunks = H / 8;  // 8-feature chunks of the low half
  auto off = [&](int r, int d) {
    return (d >> 6) * (2 * kRowBoxBytes) + r * 128 + ((((d & 63) >> 3) ^ (r & 7)) << 4);
  };
  auto at = [&](int r, int d) -> uint4* { return reinterpret_cast<uint4*>(qs + off(r, d)); };
  auto rem = [&](int r, int d) -> uint4* { return reinterpret_cast<uint4*>(qs + kRowBoxBytes + off(r, d)); };
  for (int idx = lane; idx < kRows * kChunks; idx += 32) {
    const int r = idx / kChunks, d0 = (idx % kChunks) * 8;
    if (r >= it.rows) {  // unused rows: no remainder
      *rem(r, d0) = make_uint4(0, 0, 0, 0);
      *rem(r, d0 + H) = make_uint4(0, 0, 0, 0);
      continue;
    }
    const int pos = it.len - a.Tq + (it.r0 + r) % a.Tq;
    const float* cs = a.rope_cs + (long)pos * D;
    const float4 c0 = *reinterpret_cast<const float4*>(cs + d0), c1 = *reinterpret_cast<const float4*>(cs + d0 + 4);
    const float4 s0 = *reinterpret_cast<const float4*>(cs + H + d0);
    const float4 s1 = *reinterpret_cast<const float4*>(cs + H + d0 + 4);
    const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    uint4 lo = *at(r, d0), hi = *at(r, d0 + H), rlo, rhi;
    uint32_t* l32 = reinterpret_cast<uint32_t*>(&lo);
    uint32_t* h32 = reinterpret_cast<uint32_t*>(&hi);
    uint32_t* rl32 = reinterpret_cast<uint32_t*>(&rlo);
    uint32_t* rh32 = reinterpret_cast<uint32_t*>(&rhi);
    // value = bf16(y), remainder = bf16(y - value): the pair carries y to
    // about 16 significant bits
    auto split = [](float y0, float y1, uint32_t& v, uint32_t& rm) {
      v = pack_bf16x2(y0, y1);
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
      rm = pack_bf16x2(y0 - b.x, y1 - b.y);
    };
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 xl = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&l32[e]));
      const float2 xh = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&h32[e]));
      const float yl0 = fmaf(xl.x, c[2 * e], -xh.x * sn[2 * e]), yh0 = fmaf(xh.x, c[2 * e], xl.x * sn[2 * e]);
      const float yl1 = fmaf(xl.y, c[2 * e + 1], -xh.y * sn[2 * e + 1]);
      const float yh1 = fmaf(xh.y, c[2 * e + 1], xl.y * sn[2 * e + 1]);
      split(yl0, yl1, l32[e], rl32[e]);
      split(yh0, yh1, h32[e], rh32[e]);
    }
    *at(r, d0) = lo;
    *at(r, d0 + H) = hi;
    *rem(r, d0) = rlo;
    *rem(r, d0 + H) = rhi;
  }
}

// A piece's output (softmax warps, once per piece, out of line): wait for
// its O^T, read this thread's feature row of it, release the buffer and
// write O / LSE (one-split unit) or the unnormalised partial and its
// (max, sum) -- the row statistics wait in shared memory (s_fin).
template <int D, bool FP8>
__device__ __noinline__ void decode_write_out(const DecodeArgs& a, const Piece& it, int uses, uint32_t tmem_lane,
                                              uint64_t* o_full, uint64_t* o_empty, const float2* s_fin, int j,
                                              const Guard& guard) {
  const int ob = uses & 1;
  mbar_wait(&o_full[ob], (uses >> 1) & 1, guard);
  tc_fence_after();
  uint32_t ov[kRows];
  tmem_ld_x16(tmem_lane + col_o<FP8>(ob), ov);
  tmem_ld_wait();
  reg_fence<kRows>(ov);
  tc_fence_before();
  mbar_arrive_warp(&o_empty[ob]);
  if (guard.aborted() || j >= D) return;
  const bool whole = it.npieces == 1;
  const long pbase = ((long)it.u * a.slots + it.slot) * a.rows_ws;
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    if (r >= it.rows) break;
    const int rg = it.r0 + r;  // row within the group: query head rg / Tq, position rg % Tq
    const float O = __uint_as_float(ov[r]) * a.v_scale;
    const float2 ml = s_fin[ob * kRows + r];
    if (whole) {
      const long orow = ((long)it.b * a.Hq + (long)it.hkv * a.G) * a.Tq + rg;
      a.o[orow * D + j] = __float2bfloat16_rn(O / ml.y);
      if (j == 0) a.lse[orow] = (ml.x + __log2f(ml.y)) * 0.69314718055994531f;
    } else {
      a.ws_o[(pbase + r) * D + j] = O;
      if (j == 0) a.ws_ml[pbase + r] = ml;
    }
  }
}

template <int D, bool PAGED, bool FP8>
__global__ void __launch_bounds__(FP8 ? kThreads8 : kThreads, 1)
    decode_partial_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_q, const DecodeArgs a) {
  using C = DecCfg<D, FP8>;
  constexpr int SK = C::kSlotsK, SV = C::kSlotsV;
  constexpr int NB = C::NB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DecBarriers bars;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Guard guard{&bars.abort, a.status};
  __shared__ int s_len[kLenCache];
  const int* lens = a.B <= kLenCache ? s_len : a.cache_lens;
  __shared__ Share share;
  if (warp == 0) {
    // the rows' lengths, kept in shared memory (invalid ones reported once),
    // then this CTA's share of the chunk stream
    bool bad = false;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
      if (b0 + lane < a.B) {
        const int len = a.cache_lens[b0 + lane];
        if (a.B <= kLenCache) s_len[b0 + lane] = len;
        bad |= len < a.Tq || len > a.S;
      }
    }
    if (__any_sync(0xffffffffu, bad) && blockIdx.x == 0 && lane == 0) atomicCAS(a.status, 0, kDevBadSeqlens);
    __syncwarp();
    const Share sh0 = find_share(a, lens, blockIdx.x, gridDim.x);
    if (lane == 0) share = sh0;
  }
  if (threadIdx.x == 0) {
    bars.abort = 0;
    for (int i = 0; i < SK; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
    }
    for (int i = 0; i < SV; ++i) {
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], FP8 ? 4 : 1);  // FP8: one arrive per converter warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 1);
      mbar_init(&bars.qs_full[i], 1);
      mbar_init(&bars.qs_empty[i], 4);
      mbar_init(&bars.vo_full[i], 4);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.s_empty[i], 4);   // one arrive per softmax warp
      mbar_init(&bars.p_full[i], 4);
      mbar_init(&bars.p_empty[i], 1);
      mbar_init(&bars.o_full[i], 1);
      mbar_init(&bars.o_empty[i], 4);
    }
    mbar_init(&bars.teardown[0], 1);
    mbar_init(&bars.teardown[1], 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars.tmem_base, kTmemCols<FP8>);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const uint32_t sbase = smem_u32(smem);
  // let the merge kernel's CTAs be scheduled; they wait for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const Share sh = share;
  auto begin = [&]() { return cursor_begin(a, sh, lens); };
  auto next = [&](Cursor& cur) { cursor_next(a, sh, lens, cur); };

  if (warp == 0 || warp == 6) {
    // ============================== producers: warp 0 K chunks, warp 6 V chunks
    // into rings of operand tiles (bf16), or of 8-bit tiles (FP8: the K ring
    // feeds the score MMA, the V ring the softmax warps' conversion)
    const bool is_k = warp == 0;
    const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
    uint64_t* full = is_k ? bars.k_full : bars.v_full;
    uint64_t* empty = is_k ? bars.k_empty : bars.v_empty;
    uint8_t* ring = smem + (is_k ? 0 : (FP8 ? C::kOffStage : C::kOffV));
    const int ns = is_k ? SK : SV;
    const int tile = FP8 ? C::kTile8 : C::kTileBytes;
    if (lane == 0) tma_prefetch_desc(tm);
    int last_fill[C::kMaxSlots];
#pragma unroll
    for (int i = 0; i < C::kMaxSlots; ++i) last_fill[i] = -1;
    // TMA of stream chunk (piece it, chunk c of it) into `dst`, completing on
    // `bar`.  Paged: lane i looks up the chunk's i-th page (before the slot
    // wait, so the lookup's latency overlaps it); pages that hold none of the
    // row's keys, and invalid entries (reported), get a coordinate past the
    // tensor, which the TMA fills with zeros.
    auto load_chunk = [&](const Piece& it, int c, uint8_t* dst, uint64_t* bar, uint64_t* wait_bar, int wait_parity,
                          int* fill_rec, int fill) {
      const int k0 = it.kbeg + c * kCK;
      int pages[kCK / 16];
      int npc = 1;
      if constexpr (PAGED) {
        const int psz = a.page_size;
        npc = psz >= kCK ? 1 : kCK / psz;
        const int idx = k0 / psz + lane;
        const int used = (it.len + psz - 1) / psz;
        int pg = -1;
        bool bad = false;
        if (lane < npc && idx < used) {
          const int e = a.block_table[(long)it.b * a.max_pages + idx];
          if (e >= 0 && e < a.num_pages) pg = e;
          else bad = true;
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicCAS(a.status, 0, kDevBadPages);
#pragma unroll
        for (int i = 0; i < kCK / 16; ++i) pages[i] = __shfl_sync(0xffffffffu, pg, i);
      }
      if (wait_bar != nullptr) mbar_wait(wait_bar, wait_parity, guard);
      if (lane == 0) {
        if (guard.aborted()) {
          mbar_arrive(bar);  // nothing loaded; the other roles are on their way out
        } else {
          constexpr int kRowBytes = FP8 ? D : 128;      // bytes per key row of one TMA box
          constexpr int kBoxes = FP8 ? 1 : NB;          // boxes per key row
          mbar_expect_tx(bar, FP8 ? C::kTile8 : C::kTileBytes);
          if constexpr (PAGED) {
            const int psz = a.page_size;
            const int row = psz >= kCK ? k0 % psz : 0;  // first row of the chunk inside its page
            for (int i = 0; i < npc; ++i) {
              const int z = pages[i] >= 0 ? pages[i] * a.Hkv + it.hkv : a.num_pages * a.Hkv;
#pragma unroll
              for (int x = 0; x < kBoxes; ++x)
                tma_load_3d(dst + x * kBoxBytes + i * psz * kRowBytes, tm, bar, x * 64, row, z);
            }
          } else {
#pragma unroll
            for (int x = 0; x < kBoxes; ++x) tma_load_3d(dst + x * kBoxBytes, tm, bar, x * 64, k0, it.bh);
          }
          *fill_rec = fill;
        }
      }
      __syncwarp();
    };
    int slot = 0, fill = 0;
    for (Cursor cur = begin(); cur.valid; next(cur)) {
      load_chunk(cur.it, cur.c, ring + slot * tile, &full[slot], fill >= 1 ? &empty[slot] : nullptr, (fill - 1) & 1,
                 &last_fill[slot], fill);
      if (++slot == ns) {
        slot = 0;
        ++fill;
      }
    }
    // never leave the CTA with copies in flight
    if (lane == 0)
      for (int i = 0; i < ns; ++i)
        if (last_fill[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)last_fill[i] & 1);
    __syncwarp();
  } else if (warp == 1) {
    // ===================== score MMA issuer (warp-uniform, one elected lane issues)
    // The query rows of each piece: TMA one piece ahead (the piece's 16 rows,
    // K-major, 128-byte swizzled, as the bf16 score MMA reads them; rows past
    // it.rows belong to other heads or lie past the tensor and only fill
    // unused columns of S^T).
    if (lane == 0) tma_prefetch_desc(&tm_q);
    Cursor qc = begin();
    int last_q[2] = {-1, -1};
    auto load_q = [&]() {
      if (!qc.valid) return;
      const int u = qc.uses, qslot = u & 1;
      if (u >= 2) mbar_wait(&bars.q_empty[qslot], ((u >> 1) - 1) & 1, guard);
      if (lane == 0) {
        if (guard.aborted()) {
          mbar_arrive(&bars.q_full[qslot]);
        } else {
          const int row0 = (qc.it.b * a.Hq + qc.it.hkv * a.G) * a.Tq + qc.it.r0;
          mbar_expect_tx(&bars.q_full[qslot], C::kQBytes);
#pragma unroll
          for (int x = 0; x < NB; ++x)
            tma_load_2d(smem + C::kOffQ + qslot * C::kQSlot + x * C::kQBoxStride, &tm_q, &bars.q_full[qslot],
                        x * 64, row0);
          last_q[qslot] = (u >> 1) & 1;
        }
      }
      __syncwarp();
      const int n = qc.it.nch;
      for (int c = 0; c < n; ++c) next(qc);
    };
    load_q();
    int slot = 0, fill = 0;  // K ring position of the current chunk
    for (Cursor cur = begin(); cur.valid; next(cur)) {
      const int qslot = cur.uses & 1, sb = cur.cs & 1;
      if (cur.c == 0) {
        load_q();  // the next piece's rows
        mbar_wait(&bars.q_full[qslot], (cur.uses >> 1) & 1, guard);
        uint8_t* qt = smem + C::kOffQ + qslot * C::kQSlot;
        if constexpr (FP8) {
          // the piece's rows as E4M3 parts with row scales (read by the
          // softmax warps once the previous use of this slot is done)
          if (cur.uses >= 2) mbar_wait(&bars.qs_empty[qslot], ((cur.uses >> 1) - 1) & 1, guard);
          q_tile_to_e4m3_parts<D>(qt, smem + C::kOffQ8 + qslot * 3 * C::kQ8Bytes,
                                  reinterpret_cast<float*>(smem + C::kOffQs) + qslot * kRows, cur.it, a, lane);
          fence_proxy_async_smem();  // the part tiles are read by the MMAs below
          mbar_arrive_warp(&bars.qs_full[qslot]);
        } else if (a.rope_cs != nullptr) {
          rope_rotate_tile<D>(qt, cur.it, a, lane);
          fence_proxy_async_smem();  // the rewritten tiles are read by the MMAs below
          __syncwarp();
        }
      }
      mbar_wait(&bars.k_full[slot], fill & 1, guard);
      if (cur.cs >= 2) mbar_wait(&bars.s_empty[sb], ((cur.cs >> 1) - 1) & 1, guard);
      tc_fence_after();
      if (!guard.aborted()) {
        const uint32_t ka = sbase + slot * C::kTileK;
        if constexpr (FP8) {
          // E4M3 K codes x the three E4M3 query parts, 32 features per MMA:
          // the part tiles lie back to back (row 16 t + r of a 48-row K-major
          // operand is row r of part t), so one N = 48 MMA covers all three
          const uint32_t qa = sbase + C::kOffQ8 + qslot * 3 * C::kQ8Bytes;
          auto desc8 = [](uint32_t addr) { return D == 128 ? sdesc_sw128(addr, 16, 1024) : sdesc_sw64(addr, 16, 512); };
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk)
              mma_ss_f8(tmem + col_s<FP8>(sb), desc8(ka + kk * 32), desc8(qa + kk * 32), C::kIdescS,
                             kk > 0 ? 1u : 0u);
          }
          __syncwarp();
        } else {
          const uint32_t qa = sbase + C::kOffQ + qslot * C::kQSlot;
          // rotary queries: the value rows and the remainder rows under them,
          // one N = 32 operand (columns [0, 16) and [16, 32) of S^T)
          const uint32_t idesc = a.rope_cs != nullptr ? C::kIdescS : C::kIdescS1;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ss(tmem + col_s<FP8>(sb), sdesc_sw128(ka + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024),
                          sdesc_sw128(qa + (kk >> 2) * C::kQBoxStride + (kk & 3) * 32, 16, 1024), idesc,
                          kk > 0 ? 1u : 0u);
          }
          __syncwarp();
        }
      }
      tc_commit_warp(&bars.s_full[sb]);
      tc_commit_warp(&bars.k_empty[slot]);
      if (cur.c == cur.it.nch - 1) tc_commit_warp(&bars.q_empty[qslot]);
      if (++slot == SK) {
        slot = 0;
        ++fill;
      }
    }
    // every issued MMA finishes, and no copy is in flight, before TMEM and
    // shared memory are released
    tc_commit_warp(&bars.teardown[0]);
    mbar_wait_drain(&bars.teardown[0], 0);
    if (lane == 0)
      for (int i = 0; i < 2; ++i)
        if (last_q[i] >= 0) mbar_wait_drain(&bars.q_full[i], (uint32_t)last_q[i]);
    __syncwarp();
  } else if (warp == 7) {
    // ===================== P V MMA issuer: independent of the score issuer, so
    // that a V chunk is released as soon as its own P is ready.  FP8: chunk
    // i's f16 V is operand tile i % kVop (vo_full, from the converter
    // warps), released when the P V MMA is done (p_empty).
    int slot = 0, fill = 0;  // V ring position (bf16)
    for (Cursor cur = begin(); cur.valid; next(cur)) {
      const int ob = cur.uses & 1, pb = cur.cs & 1;
      if (cur.c == 0 && cur.uses >= 2) mbar_wait(&bars.o_empty[ob], ((cur.uses >> 1) - 1) & 1, guard);
      if constexpr (FP8) mbar_wait(&bars.vo_full[cur.cs % C::kVop], (cur.cs / C::kVop) & 1, guard);
      else mbar_wait(&bars.v_full[slot], fill & 1, guard);
      mbar_wait(&bars.p_full[pb], (cur.cs >> 1) & 1, guard);
      tc_fence_after();
      if (!guard.aborted()) {
        const uint32_t va = sbase + C::kOffV + (FP8 ? cur.cs % C::kVop : slot) * C::kTileBytes;
        const uint32_t pa = sbase + C::kOffP + pb * C::kPBytes;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kCK / 16; ++kk)
            mma_ss(tmem + col_o<FP8>(ob), sdesc_sw128(va + kk * 2048, C::kLboV, 1024),
                        sdesc_sw128(pa + (kk >> 2) * kRowBoxBytes + (kk & 3) * 32, 16, 1024), C::kIdescO,
                        (cur.c > 0 || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
      }
      tc_commit_warp(&bars.p_empty[pb]);
      if constexpr (!FP8) tc_commit_warp(&bars.v_empty[slot]);
      if (cur.c == cur.it.nch - 1) tc_commit_warp(&bars.o_full[ob]);
      if (++slot == SV) {
        slot = 0;
        ++fill;
      }
    }
    tc_commit_warp(&bars.teardown[1]);
    mbar_wait_drain(&bars.teardown[1], 0);
  } else if (warp >= 2 && warp <= 5) {
    // ============================================================ softmax
    const int wq = warp & 3;                  // TMEM lane quarter of this warp
    const int j = 32 * wq + lane;             // key of the chunk (S^T row) / feature (O^T row)
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    float* s_max = reinterpret_cast<float*>(smem + C::kOffMax);
    float* s_sum = reinterpret_cast<float*>(smem + C::kOffSum);
    const float sc_log2 = a.scale_log2;
    float m_used[kRows], lpart[kRows];
    float sc_row[FP8 ? kRows : 1];  // FP8: score scale times the row's query scale
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      m_used[r] = -INFINITY;
      lpart[r] = 0.f;
    }
    float2* s_fin = reinterpret_cast<float2*>(smem + C::kOffFin);
    bool pend = false;  // a piece whose O / partial is still to be written
    Piece pend_it;
    int pend_uses = 0;
    auto write_out = [&]() {
      pend = false;
      decode_write_out<D, FP8>(a, pend_it, pend_uses, tmem + lane_off, bars.o_full, bars.o_empty, s_fin, j, guard);
    };
    for (Cursor cur = begin(); cur.valid; next(cur)) {
      const Piece& it = cur.it;
      const int i = cur.cs, sb = i & 1;
      if (cur.c == 0) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          m_used[r] = -INFINITY;
          lpart[r] = 0.f;
        }
        if constexpr (FP8) {
          const int qslot = cur.uses & 1;
          mbar_wait(&bars.qs_full[qslot], (cur.uses >> 1) & 1, guard);
          const float* qs = reinterpret_cast<const float*>(smem + C::kOffQs) + qslot * kRows;
#pragma unroll
          for (int r = 0; r < kRows; ++r) sc_row[r] = qs[r] * sc_log2;
          mbar_arrive_warp(&bars.qs_empty[qslot]);
        }
      }
      mbar_wait(&bars.s_full[sb], (i >> 1) & 1, guard);
      tc_fence_after();
      uint32_t sr[kRows];
      if constexpr (FP8) {
        // the three query parts' scores, summed in order
        uint32_t s1[kRows], s2[kRows];
        tmem_ld_x16(tmem + lane_off + col_s<FP8>(sb), sr);
        tmem_ld_x16(tmem + lane_off + col_s<FP8>(sb) + kRows, s1);
        tmem_ld_x16(tmem + lane_off + col_s<FP8>(sb) + 2 * kRows, s2);
        tmem_ld_wait();
        reg_fence<kRows>(sr);
        reg_fence<kRows>(s1);
        reg_fence<kRows>(s2);
#pragma unroll
        for (int r = 0; r < kRows; ++r)
          sr[r] = __float_as_uint((__uint_as_float(sr[r]) + __uint_as_float(s1[r])) + __uint_as_float(s2[r]));
      } else if (a.rope_cs != nullptr) {
        // a rotary query's value and remainder scores
        uint32_t s1[kRows];
        tmem_ld_x16(tmem + lane_off + col_s<FP8>(sb), sr);
        tmem_ld_x16(tmem + lane_off + col_s<FP8>(sb) + kRows, s1);
        tmem_ld_wait();
        reg_fence<kRows>(sr);
        reg_fence<kRows>(s1);
#pragma unroll
        for (int r = 0; r < kRows; ++r) sr[r] = __float_as_uint(__uint_as_float(sr[r]) + __uint_as_float(s1[r]));
      } else {
        tmem_ld_x16(tmem + lane_off + col_s<FP8>(sb), sr);
        tmem_ld_wait();
        reg_fence<kRows>(sr);
      }
      tc_fence_before();
      mbar_arrive_warp(&bars.s_empty[sb]);

      // mask: key j (position k0 + j) is visible to the row of position t iff
      // k0 + j <= len - Tq + t; keys at or past len never are.  A chunk that
      // every row sees whole (all but a piece's last one or two) skips it.
      const int k0 = it.kbeg + cur.c * kCK;
      const int lim0 = it.len - a.Tq - k0;
      float s[kRows];
      if (lim0 >= kCK - 1) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) s[r] = __uint_as_float(sr[r]) * (FP8 ? sc_row[FP8 ? r : 0] : sc_log2);
      } else {
        int t = it.r0 % a.Tq;  // query position of row r, stepped along the rows
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          s[r] = j <= lim0 + t ? __uint_as_float(sr[r]) * (FP8 ? sc_row[FP8 ? r : 0] : sc_log2) : -INFINITY;
          t = t + 1 == a.Tq ? 0 : t + 1;
        }
      }
      // The maximum in use moves only when a score exceeds it by more than
      // 2^8 (or at a piece's first chunk): one barrier-reduction tells
      // whether any of the 128 threads needs that; only then are the chunk's
      // row maxima exchanged across the four warps.
      bool over = false;
#pragma unroll
      for (int r = 0; r < kRows; ++r) over |= s[r] > m_used[r] + kRescaleThreshold;
      float alpha[kRows];
      bool resc = false;
#pragma unroll
      for (int r = 0; r < kRows; ++r) alpha[r] = 1.f;
      if (bar_red_or(1, 128, over)) {
        float mine = -INFINITY;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          const float mr = warp_max(s[r]);
          if (lane == r) mine = mr;
        }
        float* mxb = s_max + sb * kRows * 4;
        if (lane < kRows) mxb[lane * 4 + wq] = mine;
        named_bar_sync(1, 128);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          const float4 v = *reinterpret_cast<const float4*>(mxb + r * 4);
          const float mc = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
          if (mc > m_used[r] + kRescaleThreshold) {  // also when m_used is -inf and mc is finite
            alpha[r] = ex2_approx(m_used[r] - mc);
            m_used[r] = mc;
            resc = true;
          }
        }
      }
      // cache rows at or past len are outside the cache and may hold
      // anything: zero their V (once it has landed) so that 0 * V stays 0
      // in the MMA (FP8: the converter warps write them as zeros)
      const int nvis = it.len - k0;
      if (!FP8 && nvis < kCK) {
        mbar_wait(&bars.v_full[i % SV], (i / SV) & 1, guard);
        uint8_t* vs = smem + C::kOffV + (i % SV) * C::kTileBytes;
        if (j >= nvis) {
#pragma unroll
          for (int x = 0; x < NB; ++x)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<uint4*>(vs + x * kBoxBytes + j * 128 + q * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      // P = 2^(s - m) as bf16 into the K-major swizzled P tile; partial row sums
      const int pb = i & 1;
      if (i >= 2) mbar_wait(&bars.p_empty[pb], ((i >> 1) - 1) & 1, guard);
      uint8_t* pt = smem + C::kOffP + pb * C::kPBytes + (j >> 6) * kRowBoxBytes + (j & 7) * 2;
      const int pch = (j & 63) >> 3;
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const float mu = m_used[r] == -INFINITY ? 0.f : m_used[r];
        const float pr = ex2_approx(s[r] - mu);
        lpart[r] = fmaf(lpart[r], alpha[r], pr);
        if constexpr (FP8)
          *reinterpret_cast<__half*>(pt + r * 128 + ((pch ^ (r & 7)) << 4)) = __float2half_rn(pr);
        else
          *reinterpret_cast<__nv_bfloat16*>(pt + r * 128 + ((pch ^ (r & 7)) << 4)) = __float2bfloat16_rn(pr);
      }
      fence_proxy_async_smem();
      if (resc && cur.c > 0) {
        // rows whose maximum moved: scale their O^T columns once the previous P V is done
        const int pp = (i - 1) & 1;
        mbar_wait(&bars.p_empty[pp], ((i - 1) >> 1) & 1, guard);
        tc_fence_after();
        const uint32_t to = tmem + lane_off + col_o<FP8>(cur.uses & 1);
        uint32_t ov[kRows];
        tmem_ld_x16(to, ov);
        tmem_ld_wait();
        reg_fence<kRows>(ov);
#pragma unroll
        for (int r = 0; r < kRows; ++r) ov[r] = __float_as_uint(__uint_as_float(ov[r]) * alpha[r]);
        tmem_st_x16(to, ov);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive_warp(&bars.p_full[pb]);

      if (cur.c == it.nch - 1) {
        // ---------------------------------------------------- piece end
        // row sums over the 128 threads' keys; with the maxima in use they go
        // to shared memory until the piece's O^T is read (write_out)
        // (recursive halving: 16 shuffles leave lane l with the warp's sum of
        // row (l >> 1) & 15)
        float w8[8], w4[4], w2[2];
        const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4, h2 = lane & 2;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          w8[k] = (h16 ? lpart[k + 8] : lpart[k]) + __shfl_xor_sync(0xffffffffu, h16 ? lpart[k] : lpart[k + 8], 16);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          w4[k] = (h8 ? w8[k + 4] : w8[k]) + __shfl_xor_sync(0xffffffffu, h8 ? w8[k] : w8[k + 4], 8);
#pragma unroll
        for (int k = 0; k < 2; ++k)
          w2[k] = (h4 ? w4[k + 2] : w4[k]) + __shfl_xor_sync(0xffffffffu, h4 ? w4[k] : w4[k + 2], 4);
        float wsum = (h2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, h2 ? w2[0] : w2[1], 2);
        wsum += __shfl_xor_sync(0xffffffffu, wsum, 1);
        if ((lane & 1) == 0) s_sum[((lane >> 1) & 15) * 4 + wq] = wsum;
        named_bar_sync(1, 128);
        if (j < kRows) {
          const float4 v = *reinterpret_cast<const float4*>(s_sum + j * 4);
          float mj = m_used[0];
#pragma unroll
          for (int r = 1; r < kRows; ++r) mj = j == r ? m_used[r] : mj;
          s_fin[(cur.uses & 1) * kRows + j] = make_float2(mj, (v.x + v.y) + (v.z + v.w));
        }
        named_bar_sync(1, 128);  // s_sum is read (and s_fin written) before anyone goes on
        // the previous piece's output, deferred to here (a whole piece after
        // its last P V was issued, so its O^T is ready); its O^T buffer is
        // needed again only by the next piece
        if (pend) write_out();
        pend = true;
        pend_it = it;
        pend_uses = cur.uses;
      }
    }
    if (pend) write_out();
  }

  if constexpr (FP8) {
    if (warp >= 8) {
      // ================= V converters (FP8): warp 8 + q converts key rows
      // 32 q .. 32 q + 31 of each landed chunk, one row per thread, into f16
      // operand tile i % kVop once the P V MMA of chunk i - kVop (its
      // previous reader; p_empty of that chunk) is done; one converter warp
      // per SM sub-partition, beside the softmax warp there
      constexpr int NV = C::kVop;
      const int j = 32 * (warp - 8) + lane;
      for (Cursor cur = begin(); cur.valid; next(cur)) {
        const int i = cur.cs, ot = i % NV;
        mbar_wait(&bars.v_full[i % SV], (i / SV) & 1, guard);
        if (i >= NV) mbar_wait(&bars.p_empty[(i - NV) & 1], ((i - NV) >> 1) & 1, guard);
        const int nvis = cur.it.len - (cur.it.kbeg + cur.c * kCK);
        convert_v_row<D>(smem + C::kOffStage + (i % SV) * C::kTile8, smem + C::kOffV + ot * C::kTileBytes, j,
                         j < nvis);
        fence_proxy_async_smem();  // operand writes and staging reads before async-proxy use
        mbar_arrive_warp(&bars.v_empty[i % SV]);
        mbar_arrive_warp(&bars.vo_full[ot]);
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols<FP8>);
}

// One CTA per output row (b, h, t) of a cut unit (rows of units processed
// whole were written by decode_partial).  Warp 0 finds how many pieces the
// unit was cut into (the partial kernel's share arithmetic, from the
// lengths) and turns their (max, sum) pairs into weights 2^(m_s - M) / L in
// shared memory; then every thread (= feature) sums its weighted partials
// with independent loads.  Pieces that hold no key visible to the row
// (max = -inf) get weight 0.
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeArgs a) {
  __shared__ float s_w[kDecodeMaxSlots];
  __shared__ float s_lse;
  __shared__ int s_np;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // decode_partial has finished and its writes are visible
  const int row = blockIdx.x;  // (b * Hq + h) * Tq + t
  const int t = row % a.Tq, bq = row / a.Tq;
  const int h = bq % a.Hq, b = bq / a.Hq;
  const int len = a.cache_lens[b];
  if (len < a.Tq || len > a.S) return;
  const int rg = (h % a.G) * a.Tq + t;
  const int k = (h / a.G) * a.nrb + rg / kRows;  // unit within the batch row
  const int u = b * a.Hkv * a.nrb + k;
  const long base = (long)u * a.slots * a.rows_ws + rg % kRows;  // (max, sum) of piece s: base + s * rows_ws
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const long upb = (long)a.Hkv * a.nrb;
    long C = 0, Pb = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
      int n = 0, lb = 0;
      if (b0 + lane < a.B) n = row_chunks(a, a.cache_lens, b0 + lane, lb);
      C += upb * (long)__reduce_add_sync(0xffffffffu, (unsigned)n);
      Pb += upb * (long)__reduce_add_sync(0xffffffffu, (unsigned)(b0 + lane < b ? n : 0));
    }
    const int nb = (len + kCK - 1) / kCK;
    const long Pu = Pb + (long)k * nb;
    const int G = (int)min((long)a.ctas, C);
    const int np = owner_of(Pu + nb - 1, C, G) - owner_of(Pu, C, G) + 1;
    if (np > 1 && np <= a.slots) {
      float M = -INFINITY;
      for (int s = lane; s < np; s += 32) M = fmaxf(M, a.ws_ml[base + (long)s * a.rows_ws].x);
      M = warp_max(M);
      float L = 0.f;
      for (int s = lane; s < np; s += 32) {
        const float2 v = a.ws_ml[base + (long)s * a.rows_ws];
        const float w = v.x == -INFINITY ? 0.f : ex2_approx(v.x - M);
        s_w[s] = w;
        L = fmaf(v.y, w, L);
      }
      L = warp_sum(L);
      const float inv = 1.f / L;
      for (int s = lane; s < np; s += 32) s_w[s] *= inv;
      if (lane == 0) s_lse = (M + __log2f(L)) * 0.69314718055994531f;
    }
    if (lane == 0) s_np = np;
  }
  __syncthreads();
  const int np = s_np;
  if (np <= 1 || np > a.slots) return;  // one piece: decode_partial wrote the row
  const long step = (long)a.rows_ws * a.D;
  for (int d = threadIdx.x; d < a.D; d += blockDim.x) {
    const float* wo = a.ws_o + base * a.D + d;
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    int s = 0;
    for (; s + 4 <= np; s += 4) {
      const float x0 = wo[s * step], x1 = wo[(s + 1) * step], x2 = wo[(s + 2) * step], x3 = wo[(s + 3) * step];
      acc0 = fmaf(x0, s_w[s], acc0);
      acc1 = fmaf(x1, s_w[s + 1], acc1);
      acc2 = fmaf(x2, s_w[s + 2], acc2);
      acc3 = fmaf(x3, s_w[s + 3], acc3);
    }
    for (; s < np; ++s) acc0 = fmaf(wo[s * step], s_w[s], acc0);
    a.o[(long)row * a.D + d] = __float2bfloat16_rn((acc0 + acc1) + (acc2 + acc3));
  }
  if (threadIdx.x == 0) a.lse[row] = s_lse;
}

template <int D, bool PAGED, bool FP8>
static cudaError_t launch_decode_dp(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q,
                                    const DecodeArgs& a, int grid, cudaStream_t stream) {
  using C = DecCfg<D, FP8>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<D, PAGED, FP8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  prof_begin(kProfDecode, stream);
  decode_partial_kernel<D, PAGED, FP8><<<grid, FP8 ? kThreads8 : kThreads, C::kSmemBytes, stream>>>(k, v, q, a);
  prof_end(stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.slots <= 1) return e;  // no unit can be cut
  // programmatic dependent launch: the merge grid may start while the
  // partial grid drains; it waits (griddepcontrol.wait) before reading
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B * a.Hq * a.Tq));
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_begin(kProfDecodeMerge, stream);
  e = cudaLaunchKernelEx(&cfg, decode_merge_kernel, a);
  prof_end(stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_decode_d(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q,
                                   const DecodeArgs& a, int grid, cudaStream_t stream) {
  if (a.fp8) {
    if (a.block_table != nullptr) return launch_decode_dp<D, true, true>(k, v, q, a, grid, stream);
    return launch_decode_dp<D, false, true>(k, v, q, a, grid, stream);
  }
  if (a.block_table != nullptr) return launch_decode_dp<D, true, false>(k, v, q, a, grid, stream);
  return launch_decode_dp<D, false, false>(k, v, q, a, grid, stream);
}

cudaError_t launch_attn_decode(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q, const DecodeArgs& a,
                               int grid, cudaStream_t stream) {
  if (a.D == 128) return launch_decode_d<128>(k, v, q, a, grid, stream);
  return launch_decode_d<64>(k, v, q, a, grid, stream);
}

}  // namespace gqa
