// api.cu -- the C ABI declared in include/gqa_attn.h: argument validation,
// TMA tensor-map construction, workspace carving and kernel launches.
// Every host-detectable error is returned before anything is launched.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <vector>

#include "gqa_attn.h"
#include "kernels.h"
#include "rope.h"
#include "sm103.cuh"
#include "tmap.h"

namespace {

using gqa::BwdArgs;
using gqa::FwdArgs;

// Per-device status word (first device-detected error since last cleared),
// and, in debug builds, the source line of the first failed bounds check.
__device__ int g_attn_status;
__device__ int g_attn_check_line;

constexpr int kMaxDevices = 64;

int* status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  static int* cache[kMaxDevices] = {};
  if (dev < kMaxDevices && cache[dev]) return cache[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_attn_status) != cudaSuccess) return nullptr;
  if (dev < kMaxDevices) cache[dev] = static_cast<int*>(p);
  return static_cast<int*>(p);
}

int* check_line_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  static int* cache[kMaxDevices] = {};
  if (dev < kMaxDevices && cache[dev]) return cache[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_attn_check_line) != cudaSuccess) return nullptr;
  if (dev < kMaxDevices) cache[dev] = static_cast<int*>(p);
  return static_cast<int*>(p);
}

attn_status check_arch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  static signed char known[kMaxDevices] = {};  // 0 unknown, 1 ok, -1 wrong arch
  if (dev < kMaxDevices && known[dev]) return known[dev] > 0 ? ATTN_OK : ATTN_ERR_ARCH;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const bool ok = major == 10 && minor == 3;
  if (dev < kMaxDevices) known[dev] = ok ? 1 : -1;
  return ok ? ATTN_OK : ATTN_ERR_ARCH;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the current device (looked up once per device; 0 on error).
int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cache[kMaxDevices] = {};
  if (dev < kMaxDevices && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < kMaxDevices) cache[dev] = n;
  return n;
}

attn_status check_heads(int Hq, int Hkv, int D) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_SHAPE;
  if (Hq > 65535 || Hkv > 65535) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_HEADDIM;
  return ATTN_OK;
}

// Dense [N, T, D] 16-bit tensor (bf16, or f16 for the rotated copies) seen as
// 3-D (D, T, N); box_rows x 64-element boxes.
bool map_dense(CUtensorMap* m, const void* base, int D, int T, long nheads, int box_rows = 128,
               CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const uint64_t dims[3] = {(uint64_t)D, (uint64_t)T, (uint64_t)nheads};
  const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)T * D * 2};
  const uint32_t box[3] = {64, (uint32_t)box_rows, 1};
  return gqa::make_tmap(m, base, dtype, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Packed [total, H, D] 16-bit tensor (bf16, or f16 for the rotated copies)
// seen as 3-D (D, H, total); boxes of 128 tokens.
bool map_packed(CUtensorMap* m, const void* base, int D, int H, int total, int box_rows,
                CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const uint64_t dims[3] = {(uint64_t)D, (uint64_t)H, (uint64_t)total};
  const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)H * D * 2};
  const uint32_t box[3] = {64, 1, (uint32_t)box_rows};
  return gqa::make_tmap(m, base, dtype, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

attn_status launch_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// Failure-path test (attn_test_inject_timeout): one armed injection, consumed
// by the next launch of the named kernel (1 forward, 2 backward dK/dV,
// 3 backward dQ); 0 = none.
struct Inject {
  int kernel = 0;
  uint64_t wait_ns = 0;
};
Inject g_inject;

size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

// Backward workspace: Delta [rows], LSE*log2(e) [rows], each section
// 256-byte aligned (dQ comes from a query-stationary kernel and needs no
// accumulator).  Dense rows: B*Hq*round_up(T, 128).  Packed rows: Hq * total_pad (every
// sequence gets a 4-aligned base and at least 128 rows of slack before the
// next one).
long varlen_total_pad(int num_seqs, int total) { return (long)round_up((size_t)total + 132L * num_seqs + 256, 128); }

size_t ws_bytes(long rows, int D) {
  (void)D;
  return round_up((size_t)rows * 4, 256) * 2 + 256;   // -Delta, -LSE*log2(e), the dQ kernel's tile counter
}

attn_status bwd_common(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, void* ws, const int* cu, int num_seqs,
                       int T, int total, int max_seqlen, int Hq, int Hkv, int D, int causal, float scale,
                       void* stream, bool varlen, const float* rope_cs = nullptr, int n_table = 0) {
  // rope_cs: q and k are the f16 copies rotated at their positions by the
  // rotary table rope_cs; dQ and dK are taken back through the rotation
  const bool f16qk = rope_cs != nullptr;
  const CUtensorMapDataType qk_type = f16qk ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  BwdArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.o = static_cast<const __nv_bfloat16*>(o);
  a.dout = static_cast<const __nv_bfloat16*>(dout);
  a.lse = lse;
  a.dq = static_cast<__nv_bfloat16*>(dq);
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.cu_seqlens = cu;
  a.status = status;
  a.num_seqs = num_seqs;
  a.T = varlen ? max_seqlen : T;
  a.T_pad = varlen ? 0 : (int)round_up((size_t)T, 128);
  a.total = total;
  a.total_pad = varlen ? (int)varlen_total_pad(num_seqs, total) : 0;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.D = D;
  a.causal = causal ? 1 : 0;
  a.varlen = varlen ? 1 : 0;
  a.n_items = (a.T + 127) / 128;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  const long rows = varlen ? (long)Hq * a.total_pad : (long)num_seqs * Hq * a.T_pad;
  a.ws_rows = rows;
  char* w = static_cast<char*>(ws);
  a.delta = reinterpret_cast<float*>(w);
  a.lse_log2 = reinterpret_cast<float*>(w + round_up((size_t)rows * 4, 256));
  a.tile_counter = reinterpret_cast<int*>(w + 2 * round_up((size_t)rows * 4, 256));
  a.rope_cs = rope_cs;
  a.n_table = n_table;
  a.dbg_line = check_line_word();
  a.inject_kernel = 0;
  a.inject_step = -1;
  if (g_inject.kernel == 2 || g_inject.kernel == 3) {
    a.inject_kernel = g_inject.kernel - 1;   // 1 dK/dV, 2 dQ
    a.inject_step = 1;
    a.wait_ns = g_inject.wait_ns;
    g_inject.kernel = 0;
  }
  const long grid = (long)a.n_items * num_seqs * Hkv;
  if (grid > 0x7fffffffL || rows > 0x7fffffffL || (long)a.num_seqs * Hq > 65535L * 65535L) return ATTN_ERR_SHAPE;
  const int bm = 128;   // query rows per step of both backward kernels
  CUtensorMap tq, tk, tv, tdo;
  bool ok;
  if (varlen)
    ok = map_packed(&tq, q, D, Hq, total, bm, qk_type) && map_packed(&tdo, dout, D, Hq, total, bm) &&
         map_packed(&tk, k, D, Hkv, total, 128, qk_type) && map_packed(&tv, v, D, Hkv, total, 128);
  else
    ok = map_dense(&tq, q, D, T, (long)num_seqs * Hq, bm, qk_type) &&
         map_dense(&tdo, dout, D, T, (long)num_seqs * Hq, bm) &&
         map_dense(&tk, k, D, T, (long)num_seqs * Hkv, 128, qk_type) && map_dense(&tv, v, D, T, (long)num_seqs * Hkv);
  if (!ok) return ATTN_ERR_CUDA;
  return launch_status(gqa::launch_attn_bwd(tq, tk, tv, tdo, a, static_cast<cudaStream_t>(stream), f16qk));
}

attn_status fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu,
                       int num_seqs, int T, int total, int max_seqlen, int Hq, int Hkv, int D, int causal,
                       float scale, void* stream, bool varlen, bool f16qk = false) {
  const int rows = varlen ? max_seqlen : T;
  int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  FwdArgs a{};
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.cu_seqlens = cu;
  a.status = status;
  a.num_seqs = num_seqs;
  a.T = T;
  a.total = total;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.causal = causal ? 1 : 0;
  a.varlen = varlen ? 1 : 0;
  a.pair_heads = (a.G % 2 == 0) ? 1 : 0;
  a.pairs_per_seq = a.pair_heads ? Hq / 2 : Hq;
  const int mblocks = (rows + 127) / 128;
  a.m_items = a.pair_heads ? mblocks : (mblocks + 1) / 2;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.dbg_line = check_line_word();
  a.inject_step = -1;
  if (g_inject.kernel == 1) {
    a.inject_step = 1;
    a.wait_ns = g_inject.wait_ns;
    g_inject.kernel = 0;
  }
  const long grid = (long)a.m_items * num_seqs * a.pairs_per_seq;
  if (grid <= 0) return ATTN_OK;
  if (grid > 0x7fffffffL) return ATTN_ERR_SHAPE;
  CUtensorMap tq, tk, tv;
  bool ok;
  const CUtensorMapDataType qk_type = f16qk ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (varlen)
    ok = map_packed(&tq, q, D, Hq, total, 128, qk_type) && map_packed(&tk, k, D, Hkv, total, 128, qk_type) &&
         map_packed(&tv, v, D, Hkv, total, 128);
  else {
    ok = map_dense(&tq, q, D, T, (long)num_seqs * Hq, 128, qk_type) &&
         map_dense(&tk, k, D, T, (long)num_seqs * Hkv, 128, qk_type) && map_dense(&tv, v, D, T, (long)num_seqs * Hkv);
  }
  if (!ok) return ATTN_ERR_CUDA;
  if (f16qk)
    return launch_status(
        gqa::launch_attn_fwd_f16qk(tq, tk, tv, a, D, (int)grid, static_cast<cudaStream_t>(stream)));
  return launch_status(gqa::launch_attn_fwd(tq, tk, tv, a, D, (int)grid, static_cast<cudaStream_t>(stream)));
}

// Waits, through the same bounded mbarrier wait every pipeline uses, on a
// barrier phase that nothing completes; the wait expires after limit_ns,
// records the timeout in the status word and the kernel returns.
__global__ void selftest_wait_timeout_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    gqa::mbar_init(&bar, 1);
    gqa::fence_barrier_init();
  }
  __syncthreads();
  gqa::Guard g{&abort_flag, status};
  (void)gqa::mbar_wait(&bar, 0, g, limit_ns);
}

}  // namespace

// ------------------------------------------------------- kernel timing
namespace gqa {
namespace {
struct ProfRec {
  int kind;
  cudaEvent_t start, stop;
};
std::vector<ProfRec> g_prof;       // event pool; [0, g_prof_used) hold records
size_t g_prof_used = 0;
bool g_prof_on = false;
bool g_prof_open = false;
constexpr size_t kProfMax = 1u << 16;
}  // namespace

void prof_begin(int kind, cudaStream_t s) {
  g_prof_open = false;
  if (!g_prof_on || g_prof_used >= kProfMax) return;
  if (g_prof_used == g_prof.size()) {
    ProfRec r{};
    if (cudaEventCreate(&r.start) != cudaSuccess) return;
    if (cudaEventCreate(&r.stop) != cudaSuccess) {
      cudaEventDestroy(r.start);
      return;
    }
    g_prof.push_back(r);
  }
  g_prof[g_prof_used].kind = kind;
  if (cudaEventRecord(g_prof[g_prof_used].start, s) == cudaSuccess) g_prof_open = true;
}

void prof_end(cudaStream_t s) {
  if (!g_prof_open) return;
  g_prof_open = false;
  if (cudaEventRecord(g_prof[g_prof_used].stop, s) == cudaSuccess) ++g_prof_used;
}
}  // namespace gqa

extern "C" {

attn_status attn_profile_enable(int enable) {
  gqa::g_prof_on = enable != 0;
  return ATTN_OK;
}

attn_status attn_profile_reset(void) {
  gqa::g_prof_used = 0;
  return ATTN_OK;
}

attn_status attn_profile_read(int kind, int* launches, double* total_ms) {
  if (!launches || !total_ms) return ATTN_ERR_NULL;
  if (kind < 0 || kind >= gqa::kProfKinds) return ATTN_ERR_SHAPE;
  int n = 0;
  double ms = 0.0;
  for (size_t i = 0; i < gqa::g_prof_used; ++i) {
    const gqa::ProfRec& r = gqa::g_prof[i];
    if (r.kind != kind) continue;
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      return ATTN_ERR_CUDA;
    ++n;
    ms += t;
  }
  *launches = n;
  *total_ms = ms;
  return ATTN_OK;
}


attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int T, int D, int causal, float scale, void* stream) {
  if (B < 0 || T < 0) return ATTN_ERR_SHAPE;
  attn_status st = check_heads(Hq, Hkv, D);
  if (st != ATTN_OK) return st;
  if (B == 0 || T == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_ALIGN;
  if ((long)B * Hq > 0x7fffffffL || !isfinite(scale)) return ATTN_ERR_SHAPE;
  if ((st = check_arch()) != ATTN_OK) return st;
  return fwd_common(q, k, v, o, lse, nullptr, B, T, 0, 0, Hq, Hkv, D, causal, scale, stream, false);
}

size_t attn_fwd_rope_workspace_size(int B, int Hq, int Hkv, int T, int D) {
  if (B < 0 || T < 0 || check_heads(Hq, Hkv, D) != ATTN_OK) return 0;
  return round_up((size_t)B * Hq * T * D * 2, 256) + (size_t)B * Hkv * T * D * 2;
}

attn_status attn_fwd_rope(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                          size_t workspace_bytes, int B, int Hq, int Hkv, int T, int D, int causal, float scale,
                          const float* rope_cos_sin, int rope_positions, void* stream) {
  if (B < 0 || T < 0 || rope_positions < 0) return ATTN_ERR_SHAPE;
  attn_status st = check_heads(Hq, Hkv, D);
  if (st != ATTN_OK) return st;
  if (B == 0 || T == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse || !rope_cos_sin) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(rope_cos_sin))
    return ATTN_ERR_ALIGN;
  if ((long)B * Hq > 0x7fffffffL || !isfinite(scale) || rope_positions < T) return ATTN_ERR_SHAPE;
  const size_t need = attn_fwd_rope_workspace_size(B, Hq, Hkv, T, D);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_ALIGN;
  if ((st = check_arch()) != ATTN_OK) return st;
  // rotated f16 copies of q and k in the workspace, then the forward on them
  int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  uint8_t* wq = static_cast<uint8_t*>(workspace);
  uint8_t* wk = wq + round_up((size_t)B * Hq * T * D * 2, 256);
  gqa::RopeRows rr{};
  rr.rows_q = (long)B * Hq * T;
  rr.rows_k = (long)B * Hkv * T;
  rr.T = T;
  rr.n_table = rope_positions;
  rr.status = status;
  const cudaError_t e =
      gqa::launch_rope_qk_f16(q, k, wq, wk, rr, D, rope_cos_sin, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return fwd_common(wq, wk, v, o, lse, nullptr, B, T, 0, 0, Hq, Hkv, D, causal, scale, stream, false, true);
}

size_t attn_varlen_fwd_rope_workspace_size(int total_tokens, int Hq, int Hkv, int D) {
  if (total_tokens < 0 || check_heads(Hq, Hkv, D) != ATTN_OK) return 0;
  return round_up((size_t)total_tokens * Hq * D * 2, 256) + (size_t)total_tokens * Hkv * D * 2;
}

attn_status attn_varlen_fwd_rope(const void* q, const void* k, const void* v, void* o, float* lse,
                                 const int* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen, int Hq,
                                 int Hkv, int D, int causal, float scale, const float* rope_cos_sin,
                                 int rope_positions, void* workspace, size_t workspace_bytes, void* stream) {
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || rope_positions < 0) return ATTN_ERR_SHAPE;
  attn_status st = check_heads(Hq, Hkv, D);
  if (st != ATTN_OK) return st;
  if (num_seqs == 0 || total_tokens == 0 || max_seqlen == 0) return ATTN_OK;
  if (max_seqlen > total_tokens || !isfinite(scale) || rope_positions < max_seqlen) return ATTN_ERR_SHAPE;
  if (!q || !k || !v || !o || !lse || !cu_seqlens || !rope_cos_sin) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(rope_cos_sin))
    return ATTN_ERR_ALIGN;
  const size_t need = attn_varlen_fwd_rope_workspace_size(total_tokens, Hq, Hkv, D);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_ALIGN;
  if ((st = check_arch()) != ATTN_OK) return st;
  int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  uint8_t* wq = static_cast<uint8_t*>(workspace);
  uint8_t* wk = wq + round_up((size_t)total_tokens * Hq * D * 2, 256);
  gqa::RopeRows rr{};
  rr.rows_q = (long)total_tokens * Hq;
  rr.rows_k = (long)total_tokens * Hkv;
  rr.Hq = Hq;
  rr.Hkv = Hkv;
  rr.cu = cu_seqlens;
  rr.num_seqs = num_seqs;
  rr.n_table = rope_positions;
  rr.status = status;
  const cudaError_t e =
      gqa::launch_rope_qk_f16(q, k, wq, wk, rr, D, rope_cos_sin, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return fwd_common(wq, wk, v, o, lse, cu_seqlens, num_seqs, 0, total_tokens, max_seqlen, Hq, Hkv, D, causal,
                    scale, stream, true, true);
}

attn_status attn_varlen_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen, int Hq,
                            int Hkv, int D, int causal, float scale, void* stream) {
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0) return ATTN_ERR_SHAPE;
  attn_status st = check_heads(Hq, Hkv, D);
  if (st != ATTN_OK) return st;
  if (num_seqs == 0 || total_tokens == 0 || max_seqlen == 0) return ATTN_OK;
  if (max_seqlen > total_tokens || !isfinite(scale)) return ATTN_ERR_SHAPE;
  if (!q || !k || !v || !o || !lse || !cu_seqlens) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_ALIGN;
  if ((st = check_arch()) != ATTN_OK) return st;
  return fwd_common(q, k, v, o, lse, cu_seqlens, num_seqs, 0, total_tokens, max_seqlen, Hq, Hkv, D, causal,
                    scale, stream, true);
}

size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int T, int D) {
  if (B < 0 || T < 0 || check_heads(Hq, Hkv, D) != ATTN_OK) return 0;
  return ws_bytes((long)B * Hq * (long)round_up((size_t)T, 128), D);
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                     int T, int D, int causal, float scale, void* stream) {
  if (B < 0 || T < 0) return ATTN_ERR_SHAPE;
  attn_status st = check_heads(Hq, Hkv, D);
  if (st != ATTN_OK) return st;
  if (B == 0 || T == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_ALIGN;
  if (!isfinite(scale)) return ATTN_ERR_SHAPE;
  if (!workspace || workspace_bytes < attn_bwd_workspace_size(B, Hq, Hkv, T, D) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_WORKSPACE;
  if ((st = check_arch()) != ATTN_OK) return st;
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, nullptr, B, T, 0, 0, Hq, Hkv, D, causal, scale,
                    stream, false);
}

size_t attn_varlen_bwd_workspace_size(int num_seqs, int total_tokens, int Hq, int Hkv, int D) {
  if (num_seqs < 0 || total_tokens < 0 || check_heads(Hq, Hkv, D) != ATTN_OK) return 0;
  return ws_bytes((long)Hq * varlen_total_pad(num_seqs, total_tokens), D);
}

attn_status attn_varlen_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                            const int* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen, int Hq, int Hkv,
                            int D, int causal, float scale, void* stream) {
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0) return ATTN_ERR_SHAPE;
  attn_status st = check_heads(Hq, Hkv, D);
  if (st != ATTN_OK) return st;
  if (num_seqs == 0 || total_tokens == 0 || max_seqlen == 0) return ATTN_OK;
  if (max_seqlen > total_tokens || !isfinite(scale)) return ATTN_ERR_SHAPE;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !cu_seqlens) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_ALIGN;
  if (!workspace || workspace_bytes < attn_varlen_bwd_workspace_size(num_seqs, total_tokens, Hq, Hkv, D) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_WORKSPACE;
  if ((st = check_arch()) != ATTN_OK) return st;
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, cu_seqlens, num_seqs, 0, total_tokens,
                    max_seqlen, Hq, Hkv, D, causal, scale, stream, true);
}

size_t attn_bwd_rope_workspace_size(int B, int Hq, int Hkv, int T, int D) {
  if (B < 0 || T < 0 || check_heads(Hq, Hkv, D) != ATTN_OK) return 0;
  return round_up(attn_fwd_rope_workspace_size(B, Hq, Hkv, T, D), 256) + attn_bwd_workspace_size(B, Hq, Hkv, T, D);
}

attn_status attn_bwd_rope(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                          int B, int Hq, int Hkv, int T, int D, int causal, float scale, const float* rope_cos_sin,
                          int rope_positions, void* stream) {
  if (B < 0 || T < 0 || rope_positions < 0) return ATTN_ERR_SHAPE;
  attn_status st = check_heads(Hq, Hkv, D);
  if (st != ATTN_OK) return st;
  if (B == 0 || T == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !rope_cos_sin) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(rope_cos_sin))
    return ATTN_ERR_ALIGN;
  if ((long)B * Hq > 0x7fffffffL || !isfinite(scale) || rope_positions < T) return ATTN_ERR_SHAPE;
  if (!workspace || workspace_bytes < attn_bwd_rope_workspace_size(B, Hq, Hkv, T, D) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_WORKSPACE;
  if ((st = check_arch()) != ATTN_OK) return st;
  int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  // rotated f16 copies of q and k, then the backward on them
  uint8_t* wq = static_cast<uint8_t*>(workspace);
  uint8_t* wk = wq + round_up((size_t)B * Hq * T * D * 2, 256);
  uint8_t* wb = wq + round_up(attn_fwd_rope_workspace_size(B, Hq, Hkv, T, D), 256);
  gqa::RopeRows rr{};
  rr.rows_q = (long)B * Hq * T;
  rr.rows_k = (long)B * Hkv * T;
  rr.T = T;
  rr.n_table = rope_positions;
  rr.status = status;
  if (gqa::launch_rope_qk_f16(q, k, wq, wk, rr, D, rope_cos_sin, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return bwd_common(wq, wk, v, o, lse, dout, dq, dk, dv, wb, nullptr, B, T, 0, 0, Hq, Hkv, D, causal, scale, stream,
                    false, rope_cos_sin, rope_positions);
}

size_t attn_varlen_bwd_rope_workspace_size(int num_seqs, int total_tokens, int Hq, int Hkv, int D) {
  if (num_seqs < 0 || total_tokens < 0 || check_heads(Hq, Hkv, D) != ATTN_OK) return 0;
  return round_up(attn_varlen_fwd_rope_workspace_size(total_tokens, Hq, Hkv, D), 256) +
         attn_varlen_bwd_workspace_size(num_seqs, total_tokens, Hq, Hkv, D);
}

attn_status attn_varlen_bwd_rope(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                 const void* dout, void* dq, void* dk, void* dv, void* workspace,
                                 size_t workspace_bytes, const int* cu_seqlens, int num_seqs, int total_tokens,
                                 int max_seqlen, int Hq, int Hkv, int D, int causal, float scale,
                                 const float* rope_cos_sin, int rope_positions, void* stream) {
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || rope_positions < 0) return ATTN_ERR_SHAPE;
  attn_status st = check_heads(Hq, Hkv, D);
  if (st != ATTN_OK) return st;
  if (num_seqs == 0 || total_tokens == 0 || max_seqlen == 0) return ATTN_OK;
  if (max_seqlen > total_tokens || !isfinite(scale) || rope_positions < max_seqlen) return ATTN_ERR_SHAPE;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !cu_seqlens || !rope_cos_sin)
    return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(rope_cos_sin))
    return ATTN_ERR_ALIGN;
  if (!workspace ||
      workspace_bytes < attn_varlen_bwd_rope_workspace_size(num_seqs, total_tokens, Hq, Hkv, D) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_WORKSPACE;
  if ((st = check_arch()) != ATTN_OK) return st;
  int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  uint8_t* wq = static_cast<uint8_t*>(workspace);
  uint8_t* wk = wq + round_up((size_t)total_tokens * Hq * D * 2, 256);
  uint8_t* wb = wq + round_up(attn_varlen_fwd_rope_workspace_size(total_tokens, Hq, Hkv, D), 256);
  gqa::RopeRows rr{};
  rr.rows_q = (long)total_tokens * Hq;
  rr.rows_k = (long)total_tokens * Hkv;
  rr.Hq = Hq;
  rr.Hkv = Hkv;
  rr.cu = cu_seqlens;
  rr.num_seqs = num_seqs;
  rr.n_table = rope_positions;
  rr.status = status;
  if (gqa::launch_rope_qk_f16(q, k, wq, wk, rr, D, rope_cos_sin, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return bwd_common(wq, wk, v, o, lse, dout, dq, dk, dv, wb, cu_seqlens, num_seqs, 0, total_tokens, max_seqlen, Hq,
                    Hkv, D, causal, scale, stream, true, rope_cos_sin, rope_positions);
}

}  // extern "C"

// ------------------------------------------------------ cached (decode) attention
namespace {

// Work layout of the decode kernels; a pure function of the sizes, so the
// workspace size never depends on the device.  Query rows go in blocks of
// 16 (the N of the kernel's MMAs); a (batch row, K/V head, row block) is a
// unit.  The kernel's CTAs (at most gqa::kDecodeMaxSlots) share the units'
// 128-key chunks evenly, so a unit of n chunks is cut into at most
// min(n, CTAs) pieces: the workspace holds that many partials per unit.
struct DecodePlan {
  int R, nrb, slots, rows_ws;
  long units;
};

constexpr int kDecodeChunk = 128;
constexpr int kDecodeRows = 16;

DecodePlan decode_plan(int B, int Hq, int Hkv, int Tq, int S) {
  DecodePlan p{};
  p.R = (Hq / Hkv) * Tq;
  p.nrb = (p.R + kDecodeRows - 1) / kDecodeRows;
  p.rows_ws = p.R < kDecodeRows ? p.R : kDecodeRows;
  p.units = (long)B * Hkv * p.nrb;
  const long chunks = ((long)S + kDecodeChunk - 1) / kDecodeChunk;
  p.slots = (int)(chunks < gqa::kDecodeMaxSlots ? chunks : gqa::kDecodeMaxSlots);
  return p;
}

// Workspace: f32 partial O [units][slots][rows_ws][D] and (max, sum) pairs
// [units][slots][rows_ws], 256-byte aligned; none when no unit can be cut.
size_t decode_ws_bytes(const DecodePlan& p, int D) {
  if (p.slots <= 1) return 0;
  const size_t rows = (size_t)p.units * p.slots * p.rows_ws;
  return round_up(rows * D * 4, 256) + rows * 8;
}

attn_status decode_check(int B, int Hq, int Hkv, int Tq, int S, int D) {
  if (B < 0 || Tq < 0 || S < 0) return ATTN_ERR_SHAPE;
  attn_status st = check_heads(Hq, Hkv, D);
  if (st != ATTN_OK) return st;
  if (B == 0 || Tq == 0) return ATTN_OK;
  if (Tq > S) return ATTN_ERR_SHAPE;
  if ((long)B * Hq * Tq > 0x7fffffffL || (long)B * Hkv > 0x7fffffffL) return ATTN_ERR_SHAPE;
  const DecodePlan p = decode_plan(B, Hq, Hkv, Tq, S);
  if (p.units * ((S + 127L) / 128) > 0x7fffffffL) return ATTN_ERR_SHAPE;  // chunk stream indices
  return ATTN_OK;
}

}  // namespace

namespace {

// Shared part of the contiguous and paged decode entry points: everything
// after the layout-specific checks (capacity S = keys per row at most).
attn_status decode_common(const void* q, const CUtensorMap& tk, const CUtensorMap& tv, const int* cache_lens,
                          void* o, float* lse, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                          int Tq, int S, int D, float scale, const int* block_table, int page_size, int max_pages,
                          int num_pages, const float* rope_cos_sin, bool fp8, float k_scale, float v_scale,
                          void* stream) {
  const DecodePlan p = decode_plan(B, Hq, Hkv, Tq, S);
  const size_t need = decode_ws_bytes(p, D);  // checked by the caller
  (void)workspace_bytes;
  attn_status st = check_arch();
  if (st != ATTN_OK) return st;
  int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  const int sms = sm_count();
  if (sms < 1) return ATTN_ERR_CUDA;
  gqa::DecodeArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.cache_lens = cache_lens;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  if (need > 0) {
    const size_t rows = (size_t)p.units * p.slots * p.rows_ws;
    a.ws_o = static_cast<float*>(workspace);
    a.ws_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) + round_up(rows * D * 4, 256));
  }
  a.status = status;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.Tq = Tq;
  a.S = S;
  a.D = D;
  a.R = p.R;
  a.nrb = p.nrb;
  a.slots = p.slots;
  a.rows_ws = p.rows_ws;
  // one CTA per SM (the kernel holds most of an SM's shared memory), never
  // more than the workspace has slots for
  a.ctas = sms < gqa::kDecodeMaxSlots ? sms : gqa::kDecodeMaxSlots;
  a.scale_log2 = scale * (fp8 ? k_scale : 1.f) * 1.4426950408889634f;
  a.fp8 = fp8 ? 1 : 0;
  a.v_scale = fp8 ? v_scale : 1.f;
  a.block_table = block_table;
  a.page_size = page_size;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.rope_cs = rope_cos_sin;
  CUtensorMap tq;
  const uint64_t qdims[2] = {(uint64_t)D, (uint64_t)B * Hq * Tq};
  const uint64_t qstrides[1] = {(uint64_t)D * 2};
  const uint32_t qbox[2] = {64, (uint32_t)kDecodeRows};
  if (!gqa::make_tmap(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, qdims, qstrides, qbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return ATTN_ERR_CUDA;
  return launch_status(gqa::launch_attn_decode(tk, tv, tq, a, a.ctas, static_cast<cudaStream_t>(stream)));
}

attn_status decode_check_workspace(int B, int Hq, int Hkv, int Tq, int S, int D, const void* workspace,
                                   size_t workspace_bytes) {
  const size_t need = decode_ws_bytes(decode_plan(B, Hq, Hkv, Tq, S), D);
  if (need > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

// Rotary table: none, or [rope_positions, D] f32, 16-byte aligned, covering
// every position a query can take (< S).
attn_status decode_check_rope(const float* rope_cos_sin, int rope_positions, int S) {
  if (!rope_cos_sin) return ATTN_OK;
  if ((reinterpret_cast<uintptr_t>(rope_cos_sin) & 15u)) return ATTN_ERR_ALIGN;
  if (rope_positions < S) return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

// 8-bit cache [N, T, D] seen as 3-D (D, T, N): boxes of whole D-byte rows,
// box_rows rows, swizzled as the 8-bit K-major MMA operand reads them
// (128-byte swizzle for D = 128, 64-byte for D = 64).
bool map_bytes(CUtensorMap* m, const void* base, int D, int T, long n, int box_rows) {
  const uint64_t dims[3] = {(uint64_t)D, (uint64_t)T, (uint64_t)n};
  const uint64_t strides[2] = {(uint64_t)D, (uint64_t)T * D};
  const uint32_t box[3] = {(uint32_t)D, (uint32_t)box_rows, 1};
  return gqa::make_tmap(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, dims, strides, box,
                        D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

bool decode_page_size_ok(int page_size) {
  return page_size == 16 || page_size == 32 || page_size == 64 || (page_size > 0 && page_size % 128 == 0);
}

}  // namespace

extern "C" {

size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Tq, int S, int D) {
  if (decode_check(B, Hq, Hkv, Tq, S, D) != ATTN_OK || B == 0 || Tq == 0) return 0;
  return decode_ws_bytes(decode_plan(B, Hq, Hkv, Tq, S), D);
}

attn_status attn_decode_fwd(const void* q, const void* k_cache, const void* v_cache, const int* cache_lens,
                            void* o, float* lse, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                            int Tq, int S, int D, float scale, const float* rope_cos_sin, int rope_positions,
                            void* stream) {
  attn_status st = decode_check(B, Hq, Hkv, Tq, S, D);
  if (st != ATTN_OK) return st;
  if (B == 0 || Tq == 0) return ATTN_OK;
  if (!isfinite(scale)) return ATTN_ERR_SHAPE;
  if (!q || !k_cache || !v_cache || !cache_lens || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(lse) ||
      (reinterpret_cast<uintptr_t>(cache_lens) & 3u))
    return ATTN_ERR_ALIGN;
  if ((st = decode_check_rope(rope_cos_sin, rope_positions, S)) != ATTN_OK) return st;
  if ((st = decode_check_workspace(B, Hq, Hkv, Tq, S, D, workspace, workspace_bytes)) != ATTN_OK) return st;
  CUtensorMap tk, tv;
  if (!map_dense(&tk, k_cache, D, S, (long)B * Hkv) || !map_dense(&tv, v_cache, D, S, (long)B * Hkv))
    return ATTN_ERR_CUDA;
  return decode_common(q, tk, tv, cache_lens, o, lse, workspace, workspace_bytes, B, Hq, Hkv, Tq, S, D, scale,
                       nullptr, 0, 0, 0, rope_cos_sin, false, 1.f, 1.f, stream);
}

attn_status attn_decode_paged_fwd(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                                  const int* cache_lens, void* o, float* lse, void* workspace,
                                  size_t workspace_bytes, int B, int Hq, int Hkv, int Tq, int page_size,
                                  int num_pages, int max_pages, int D, float scale, const float* rope_cos_sin,
                                  int rope_positions, void* stream) {
  if (page_size < 0 || num_pages < 0 || max_pages < 0) return ATTN_ERR_SHAPE;
  const long S = (long)page_size * max_pages;
  if (S > 0x7fffffffL) return ATTN_ERR_SHAPE;
  attn_status st = decode_check(B, Hq, Hkv, Tq, (int)S, D);
  if (st != ATTN_OK) return st;
  if (B == 0 || Tq == 0) return ATTN_OK;
  if (!decode_page_size_ok(page_size) || num_pages < 1 || (long)num_pages * Hkv > 0x7fffffffL ||
      (long)B * max_pages > 0x7fffffffL || !isfinite(scale))
    return ATTN_ERR_SHAPE;
  if (!q || !k_pages || !v_pages || !block_table || !cache_lens || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) || !aligned16(lse) ||
      (reinterpret_cast<uintptr_t>(cache_lens) & 3u) || (reinterpret_cast<uintptr_t>(block_table) & 3u))
    return ATTN_ERR_ALIGN;
  if ((st = decode_check_rope(rope_cos_sin, rope_positions, (int)S)) != ATTN_OK) return st;
  if ((st = decode_check_workspace(B, Hq, Hkv, Tq, (int)S, D, workspace, workspace_bytes)) != ATTN_OK) return st;
  const int box = page_size < 128 ? page_size : 128;
  CUtensorMap tk, tv;
  if (!map_dense(&tk, k_pages, D, page_size, (long)num_pages * Hkv, box) ||
      !map_dense(&tv, v_pages, D, page_size, (long)num_pages * Hkv, box))
    return ATTN_ERR_CUDA;
  return decode_common(q, tk, tv, cache_lens, o, lse, workspace, workspace_bytes, B, Hq, Hkv, Tq, (int)S, D, scale,
                       block_table, page_size, max_pages, num_pages, rope_cos_sin, false, 1.f, 1.f, stream);
}

attn_status attn_decode_fp8_fwd(const void* q, const void* k8, const void* v8, float k_scale, float v_scale,
                                const int* cache_lens, void* o, float* lse, void* workspace, size_t workspace_bytes,
                                int B, int Hq, int Hkv, int Tq, int S, int D, float scale, const float* rope_cos_sin,
                                int rope_positions, void* stream) {
  attn_status st = decode_check(B, Hq, Hkv, Tq, S, D);
  if (st != ATTN_OK) return st;
  if (B == 0 || Tq == 0) return ATTN_OK;
  if (!isfinite(scale) || !isfinite(k_scale) || !isfinite(v_scale)) return ATTN_ERR_SHAPE;
  if (!q || !k8 || !v8 || !cache_lens || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k8) || !aligned16(v8) || !aligned16(o) || !aligned16(lse) ||
      (reinterpret_cast<uintptr_t>(cache_lens) & 3u))
    return ATTN_ERR_ALIGN;
  if ((st = decode_check_rope(rope_cos_sin, rope_positions, S)) != ATTN_OK) return st;
  if ((st = decode_check_workspace(B, Hq, Hkv, Tq, S, D, workspace, workspace_bytes)) != ATTN_OK) return st;
  CUtensorMap tk, tv;
  if (!map_bytes(&tk, k8, D, S, (long)B * Hkv, 128) || !map_bytes(&tv, v8, D, S, (long)B * Hkv, 128))
    return ATTN_ERR_CUDA;
  return decode_common(q, tk, tv, cache_lens, o, lse, workspace, workspace_bytes, B, Hq, Hkv, Tq, S, D, scale,
                       nullptr, 0, 0, 0, rope_cos_sin, true, k_scale, v_scale, stream);
}

attn_status attn_decode_paged_fp8_fwd(const void* q, const void* k8_pages, const void* v8_pages, float k_scale,
                                      float v_scale, const int* block_table, const int* cache_lens, void* o,
                                      float* lse, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                                      int Tq, int page_size, int num_pages, int max_pages, int D, float scale,
                                      const float* rope_cos_sin, int rope_positions, void* stream) {
  if (page_size < 0 || num_pages < 0 || max_pages < 0) return ATTN_ERR_SHAPE;
  const long S = (long)page_size * max_pages;
  if (S > 0x7fffffffL) return ATTN_ERR_SHAPE;
  attn_status st = decode_check(B, Hq, Hkv, Tq, (int)S, D);
  if (st != ATTN_OK) return st;
  if (B == 0 || Tq == 0) return ATTN_OK;
  if (!decode_page_size_ok(page_size) || num_pages < 1 || (long)num_pages * Hkv > 0x7fffffffL ||
      (long)B * max_pages > 0x7fffffffL || !isfinite(scale) || !isfinite(k_scale) || !isfinite(v_scale))
    return ATTN_ERR_SHAPE;
  if (!q || !k8_pages || !v8_pages || !block_table || !cache_lens || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k8_pages) || !aligned16(v8_pages) || !aligned16(o) || !aligned16(lse) ||
      (reinterpret_cast<uintptr_t>(cache_lens) & 3u) || (reinterpret_cast<uintptr_t>(block_table) & 3u))
    return ATTN_ERR_ALIGN;
  if ((st = decode_check_rope(rope_cos_sin, rope_positions, (int)S)) != ATTN_OK) return st;
  if ((st = decode_check_workspace(B, Hq, Hkv, Tq, (int)S, D, workspace, workspace_bytes)) != ATTN_OK) return st;
  const int box = page_size < 128 ? page_size : 128;
  CUtensorMap tk, tv;
  if (!map_bytes(&tk, k8_pages, D, page_size, (long)num_pages * Hkv, box) ||
      !map_bytes(&tv, v8_pages, D, page_size, (long)num_pages * Hkv, box))
    return ATTN_ERR_CUDA;
  return decode_common(q, tk, tv, cache_lens, o, lse, workspace, workspace_bytes, B, Hq, Hkv, Tq, (int)S, D, scale,
                       block_table, page_size, max_pages, num_pages, rope_cos_sin, true, k_scale, v_scale, stream);
}

// ------------------------------------------------- allocation-free backward
// Scratch for attn_bwd_noalloc: a file-scope device array, so the library
// never has to allocate device memory for it.  Every device that loads the
// library holds these bytes until the process exits.
#define GQA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
static __device__ __align__(256) unsigned char g_bwd_scratch[GQA_NOALLOC_SCRATCH_BYTES];

// Device address of g_bwd_scratch on the current device.  The name is only a
// host-side stand-in in host code, so the address is looked up once per
// device (with that device current) and cached.
static void* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  static void* cache[kMaxDevices] = {};
  if (dev < kMaxDevices && cache[dev]) return cache[dev];
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess) return nullptr;
  if (dev < kMaxDevices) cache[dev] = ptr;
  return ptr;
}

size_t attn_bwd_noalloc_scratch_bytes(void) { return GQA_NOALLOC_SCRATCH_BYTES; }

attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int T, int D,
                             int causal, float scale, void* stream) {
  if (B < 0 || T < 0) return ATTN_ERR_SHAPE;
  attn_status st = check_heads(Hq, Hkv, D);
  if (st != ATTN_OK) return st;
  if (B == 0 || T == 0) return ATTN_OK;
  if (attn_bwd_workspace_size(B, Hq, Hkv, T, D) > GQA_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_SCRATCH_LIMIT;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return ATTN_ERR_NULL;
  if ((st = check_arch()) != ATTN_OK) return st;
  void* scratch = noalloc_scratch();
  if (!scratch) return ATTN_ERR_CUDA;
  return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, scratch, GQA_NOALLOC_SCRATCH_BYTES, B, Hq, Hkv, T, D, causal,
                  scale, stream);
}

attn_status attn_test_inject_timeout(int kernel, int limit_ms) {
  if (kernel < 0 || kernel > 3 || limit_ms < 1 || limit_ms > 5000) return ATTN_ERR_SHAPE;
  g_inject.kernel = kernel;
  g_inject.wait_ns = (uint64_t)limit_ms * 1000000ull;
  return ATTN_OK;
}

attn_status attn_selftest_wait_timeout(int limit_ms, void* stream) {
  if (limit_ms < 1 || limit_ms > 5000) return ATTN_ERR_SHAPE;
  attn_status st = check_arch();
  if (st != ATTN_OK) return st;
  int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  selftest_wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status,
                                                                                 (uint64_t)limit_ms * 1000000ull);
  return launch_status(cudaGetLastError());
}

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "invalid sizes (negative, Hq % Hkv != 0, or too large)";
    case ATTN_ERR_HEADDIM: return "head dimension must be 64 or 128";
    case ATTN_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case ATTN_ERR_SEQLENS: return "cu_seqlens or cache_lens is invalid";
    case ATTN_ERR_WORKSPACE: return "workspace is NULL or too small";
    case ATTN_ERR_ARCH: return "the current device is not compute capability 10.3 (sm_103a)";
    case ATTN_ERR_CUDA: return "a CUDA runtime call failed";
    case ATTN_ERR_TIMEOUT: return "a bounded in-kernel wait expired";
    case ATTN_ERR_SCRATCH_LIMIT:
      return "the problem needs more backward scratch than attn_bwd_noalloc's built-in array holds";
    case ATTN_ERR_PAGES: return "a block-table entry names no page of the pool";
    case ATTN_ERR_CHECK: return "a bounds check of the debug build failed (attn_get_check_line gives its line)";
    case ATTN_ERR_RANGE: return "a rotated q or k value is not finite or does not fit f16 (|x| >= 65520)";
  }
  return "unknown status";
}

attn_status attn_get_check_line(void* stream, int* out, int clear) {
  if (!out) return ATTN_ERR_NULL;
  int* w = check_line_word();
  if (!w) return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  *out = v;
  return ATTN_OK;
}

int attn_is_debug_build(void) {
#ifdef GQA_DEBUG
  return 1;
#else
  return 0;
#endif
}

attn_status attn_get_device_status(void* stream, int* out, int clear) {
  if (!out) return ATTN_ERR_NULL;
  int* w = status_word();
  if (!w) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  *out = v;
  return ATTN_OK;
}

}  // extern "C"
