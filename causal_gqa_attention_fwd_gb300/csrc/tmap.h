// tmap.h -- host-side construction of TMA tensor maps (cuTensorMapEncodeTiled,
// fetched through the runtime's driver entry-point query so the library does
// not link libcuda directly).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gqa {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Everything a tiled map is encoded from.  Two equal keys encode to the same
// 128-byte map, so an encoded map can be reused for as long as the caller
// passes the same address and geometry.
struct TmapKey {
  const void* base;
  uint64_t dims[5];
  uint64_t strides[4];
  uint32_t box[5];
  int32_t dtype, rank, swizzle, pad;
};

// Per-thread cache of recently encoded maps (round-robin replacement): a
// training or serving loop calls with the same buffers every step, and the
// lookup (a few dozen compares) costs less than re-encoding.
constexpr int kTmapCacheSize = 32;
struct TmapCache {
  TmapKey key[kTmapCacheSize];
  CUtensorMap map[kTmapCacheSize];
  int used = 0, next = 0;
};

inline bool same_key(const TmapKey& a, const TmapKey& b) {
  if (a.base != b.base || a.dtype != b.dtype || a.rank != b.rank || a.swizzle != b.swizzle) return false;
  for (int i = 0; i < a.rank; ++i)
    if (a.dims[i] != b.dims[i] || a.box[i] != b.box[i]) return false;
  for (int i = 0; i + 1 < a.rank; ++i)
    if (a.strides[i] != b.strides[i]) return false;
  return true;
}

// Tiled map of rank 2..5.  dims[0] is the contiguous dimension; strides_bytes
// has rank-1 entries (for dims 1..rank-1).  Out-of-range elements load as 0.
inline bool make_tmap(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int rank,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle) {
  if (rank < 1 || rank > 5) return false;
  TmapKey k{};
  k.base = base;
  k.dtype = (int32_t)dtype;
  k.rank = rank;
  k.swizzle = (int32_t)swizzle;
  for (int i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) k.strides[i] = strides_bytes[i];
  static thread_local TmapCache cache;
  for (int i = 0; i < cache.used; ++i)
    if (same_key(cache.key[i], k)) {
      *map = cache.map[i];
      return true;
    }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
  CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  const int slot = cache.next;
  cache.key[slot] = k;
  cache.map[slot] = *map;
  cache.next = (slot + 1) % kTmapCacheSize;
  if (cache.used < kTmapCacheSize) ++cache.used;
  return true;
}

}  // namespace gqa
