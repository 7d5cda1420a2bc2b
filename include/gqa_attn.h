/*
 * gqa_attn.h -- C ABI of libgqa_attn.so: causal grouped-query scaled-dot-
 * product attention, forward and backward, for bf16 tensors on an sm_103a GPU.
 *
 * The operation is the ScaledDotProductAttention / MultiHeadAttention of the
 * "Project Overview" page of llm-from-scratch (section "Core Stack: llm/",
 * llm/transformer.py) with the grouped-query heads and causal mask of the
 * microLLM-rocm README (section "Why this project exists": "Decoder-only
 * MHA/GQA ... causal attention" and the causal GQA backward), computed
 * blockwise with running softmax statistics as in the Flash Attention kernel
 * of "Project Overview", section "Performance Layer: kernel/ and parallel/":
 *
 *   S = scale * Q K^T,  key j visible to query i iff j <= i (causal != 0),
 *   LSE_i = ln sum_j exp(S_ij) over visible j,   P = exp(S - LSE),  O = P V,
 *   and for the loss L = sum(dO * O):
 *   dP = dO V^T, Delta_i = sum_d dO_id O_id, dS = P * (dP - Delta),
 *   dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO,
 *   dK and dV summed over the G = Hq / Hkv query heads that share a K/V head
 *   (query head h reads K/V head h / G).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers, 16-byte aligned, densely
 *     packed (no strides).  bf16 = IEEE bfloat16 stored as uint16.
 *   - Dense layout:  Q, O, dO, dQ  [B, Hq, T, D];  K, V, dK, dV  [B, Hkv, T, D];
 *                    LSE  [B, Hq, T] float32 (natural log).
 *   - Packed (varlen) layout, sequences s = 0..num_seqs-1 occupying token rows
 *     [cu_seqlens[s], cu_seqlens[s+1]):  Q, O, dO, dQ  [total, Hq, D];
 *     K, V, dK, dV  [total, Hkv, D];  LSE  [Hq, total] float32.  cu_seqlens
 *     is a DEVICE int32 array of num_seqs + 1 entries, cu_seqlens[0] = 0,
 *     non-decreasing, cu_seqlens[num_seqs] = total_tokens.  The mask is causal
 *     within each sequence; sequences never see each other.
 *   - D (head dim) is 64 or 128; Hq % Hkv == 0.
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls are asynchronous on that stream; errors found on the host are
 *     returned before anything is launched; errors found on the device (a
 *     bounded wait that timed out, invalid cu_seqlens contents) are recorded
 *     in a per-device status word read by attn_get_device_status().
 *   - Ownership: the caller allocates every buffer; the library allocates no
 *     device memory and never frees caller memory.  Outputs are fully
 *     overwritten (no zero-initialisation needed).  Inputs are read-only.
 *   - Sizes of zero (B, T, num_seqs or total_tokens) are no-ops returning
 *     ATTN_OK.
 */
#ifndef GQA_ATTN_H_
#define GQA_ATTN_H_

#include <stddef.h>

#if defined(__GNUC__)
#define GQA_ATTN_API __attribute__((visibility("default")))
#else
#define GQA_ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = 1,       /* a required pointer is NULL */
    ATTN_ERR_SHAPE = 2,      /* negative size, Hq % Hkv != 0, Hq/Hkv < 1, size too large */
    ATTN_ERR_HEADDIM = 3,    /* D not 64 or 128 */
    ATTN_ERR_ALIGN = 4,      /* a pointer is not 16-byte aligned */
    ATTN_ERR_SEQLENS = 5,    /* cu_seqlens / cache_lens invalid (device-detected: status word) */
    ATTN_ERR_WORKSPACE = 6,  /* workspace NULL or smaller than the *_workspace_size() value */
    ATTN_ERR_ARCH = 7,       /* current device is not compute capability 10.3 */
    ATTN_ERR_CUDA = 8,       /* a CUDA runtime call failed (launch, tensor map, attribute) */
    ATTN_ERR_TIMEOUT = 9,    /* device-detected: a bounded in-kernel wait expired */
    ATTN_ERR_SCRATCH_LIMIT = 10, /* attn_bwd_noalloc: sizes need more than its built-in scratch */
    ATTN_ERR_PAGES = 11,     /* device-detected: a block-table entry names no page of the pool */
    ATTN_ERR_CHECK = 12,     /* device-detected, debug build only: a bounds check of a computed index failed */
    ATTN_ERR_RANGE = 13      /* device-detected: a rotated q or k value is not finite or does not fit f16 */
} attn_status;

/* Forward, dense layout.  Writes O (bf16) and LSE (float32). */
GQA_ATTN_API attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int T, int D, int causal, float scale, void* stream);

/* Bytes of device workspace attn_bwd needs for these sizes (0 if invalid). */
GQA_ATTN_API size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int T, int D);

/* Backward, dense layout.  Reads Q, K, V, the forward's O and LSE, and dO;
 * writes dQ, dK, dV (bf16).  workspace: device memory of at least
 * attn_bwd_workspace_size() bytes, 256-byte aligned, owned by the caller; it
 * holds Delta and LSE*log2(e) per query row and the dQ kernel's tile counter,
 * and needs no initialisation (the call writes all of it first); two calls
 * in flight at once need two workspaces.  dK and dV come from a
 * key/value-stationary kernel, dQ from a persistent query-stationary one
 * that takes its tiles from that counter; each tile's gradient is summed in
 * a fixed order inside one CTA, so the results are bit-reproducible. */
GQA_ATTN_API attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                     int B, int Hq, int Hkv, int T, int D, int causal, float scale, void* stream);

/* Backward, dense layout, without a caller-provided workspace and without
 * allocating anything.  (No counterpart in the pages: an operational
 * variant of attn_bwd.)  It is for callers that cannot hand the library
 * device memory or let it allocate: code running where allocation is not
 * allowed or not available -- e.g. a host framework that has reserved every
 * byte of the device for its own pool, a plugin that only ever receives the
 * tensors it must read and write, or a stream that is being captured into a
 * CUDA graph, during which cudaMalloc is not permitted.
 * The scratch is a static device array of attn_bwd_noalloc_scratch_bytes()
 * bytes (16 MiB: 8 bytes per query row, so up to 2^21 rows B*Hq*T, T rounded
 * up to 128) inside the library; every GPU that loads the library holds it
 * until the process exits.  Sizes whose attn_bwd_workspace_size() exceeds
 * it return ATTN_ERR_SCRATCH_LIMIT before anything is launched.  The first
 * call on a device looks up the array's device address (once per device,
 * with that device current), so make that first call before any stream
 * capture.  All calls share the one array and the kernels re-initialise
 * everything they read from it, but calls whose work overlaps on the GPU
 * (other streams, other host threads) race on it: serialise them.
 * The looked-up address (like the device status word's) stays cached for the
 * life of the process: after cudaDeviceReset() or anything else that
 * destroys the device's primary context, do not call this library on that
 * device again in the same process.
 * Otherwise identical to attn_bwd (same arguments minus the workspace, same
 * results bit for bit). */
GQA_ATTN_API attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                          const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                          int B, int Hq, int Hkv, int T, int D, int causal, float scale,
                                          void* stream);

/* Size in bytes of attn_bwd_noalloc's built-in scratch array. */
GQA_ATTN_API size_t attn_bwd_noalloc_scratch_bytes(void);

/* Forward, packed variable-length layout.  max_seqlen must be >= every
 * sequence's length (it sizes the launch grid). */
GQA_ATTN_API attn_status attn_varlen_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
                            int Hq, int Hkv, int D, int causal, float scale, void* stream);

GQA_ATTN_API size_t attn_varlen_bwd_workspace_size(int num_seqs, int total_tokens, int Hq, int Hkv, int D);

/* Forward with rotary queries and keys (RoPE of MultiHeadAttentionWithRoPE,
 * llm-from-scratch "Project Overview"; positions-aware RoPE of the
 * microLLM-rocm README, section "Why this project exists"): the dense layout
 * of attn_fwd; q and k of every row are rotated at their positions
 * 0..T-1 before the attention, with the rotary table of attn_decode_fwd
 * (rope_cos_sin: DEVICE float32 [rope_positions, D], 16-byte aligned,
 * rope_positions >= T; row p holds cos(p*theta_i) for i < D/2, then
 * sin(p*theta_i); feature i pairs with feature i + D/2).  The rotated q and
 * k are written as f16 (11 significant bits) into the workspace and the
 * score MMA takes them as f16; P V and everything else is as attn_fwd.
 * A rotated value that is not finite or has |value| >= 65520 (beyond f16;
 * it becomes infinite there) is recorded in the device status word as
 * ATTN_ERR_RANGE; the call still completes, and its outputs for the rows
 * that meet that value are then not meaningful.  The rotary backward
 * (attn_bwd_rope, attn_varlen_bwd_rope) reports the same way.
 * workspace: DEVICE, 256-byte aligned, >= attn_fwd_rope_workspace_size()
 * bytes (the two rotated copies), no initialisation; errors as attn_fwd,
 * plus ATTN_ERR_WORKSPACE. */
GQA_ATTN_API size_t attn_fwd_rope_workspace_size(int B, int Hq, int Hkv, int T, int D);
GQA_ATTN_API attn_status attn_fwd_rope(const void* q, const void* k, const void* v, void* o, float* lse,
                                       void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int T,
                                       int D, int causal, float scale, const float* rope_cos_sin,
                                       int rope_positions, void* stream);

/* attn_fwd_rope for the packed variable-length layout of attn_varlen_fwd:
 * every sequence's tokens are at positions 0..len-1 (the offset from
 * cu_seqlens[s]); rope_positions >= max_seqlen.  A cu_seqlens whose
 * positions fall outside the table is reported through the device status
 * word (ATTN_ERR_SEQLENS), as attn_varlen_fwd reports it.
 * workspace: DEVICE, 256-byte aligned, >= attn_varlen_fwd_rope_workspace_size()
 * bytes. */
GQA_ATTN_API size_t attn_varlen_fwd_rope_workspace_size(int total_tokens, int Hq, int Hkv, int D);
GQA_ATTN_API attn_status attn_varlen_fwd_rope(const void* q, const void* k, const void* v, void* o, float* lse,
                                              const int* cu_seqlens, int num_seqs, int total_tokens,
                                              int max_seqlen, int Hq, int Hkv, int D, int causal, float scale,
                                              const float* rope_cos_sin, int rope_positions, void* workspace,
                                              size_t workspace_bytes, void* stream);

/* Backward of attn_fwd_rope (rotary queries and keys; RoPE of
 * MultiHeadAttentionWithRoPE, llm-from-scratch "Project Overview";
 * positions-aware RoPE of the microLLM-rocm README, section "Why this project
 * exists"): the gradients of L = sum(dO * O) with respect to the UNROTATED
 * q and k (and v).  Arguments as attn_bwd, plus the rotary table of
 * attn_fwd_rope (rope_cos_sin DEVICE float32 [rope_positions, D], 16-byte
 * aligned, rope_positions >= T); o and lse are attn_fwd_rope's outputs.
 * The kernels rotate q and k at positions 0..T-1 into f16 copies (as the
 * forward does), run the backward with f16 Q/K operands and an f16 dS, and
 * take dQ and dK back through the rotation (x -> R^T x at each row's
 * position) before rounding them to bf16.
 * workspace: DEVICE, 256-byte aligned, >= attn_bwd_rope_workspace_size()
 * bytes (the rotated copies and attn_bwd's workspace), no initialisation. */
GQA_ATTN_API size_t attn_bwd_rope_workspace_size(int B, int Hq, int Hkv, int T, int D);
GQA_ATTN_API attn_status attn_bwd_rope(const void* q, const void* k, const void* v, const void* o,
                                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                       void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int T,
                                       int D, int causal, float scale, const float* rope_cos_sin,
                                       int rope_positions, void* stream);

/* attn_bwd_rope for the packed variable-length layout (attn_varlen_bwd's
 * arguments plus the table; positions 0..len-1 in every sequence,
 * rope_positions >= max_seqlen).  workspace >=
 * attn_varlen_bwd_rope_workspace_size() bytes. */
GQA_ATTN_API size_t attn_varlen_bwd_rope_workspace_size(int num_seqs, int total_tokens, int Hq, int Hkv, int D);
GQA_ATTN_API attn_status attn_varlen_bwd_rope(const void* q, const void* k, const void* v, const void* o,
                                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                              void* workspace, size_t workspace_bytes, const int* cu_seqlens,
                                              int num_seqs, int total_tokens, int max_seqlen, int Hq, int Hkv, int D,
                                              int causal, float scale, const float* rope_cos_sin,
                                              int rope_positions, void* stream);

/* Backward, packed variable-length layout (arguments as attn_bwd plus the
 * sequence description of attn_varlen_fwd). */
GQA_ATTN_API attn_status attn_varlen_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, void* workspace,
                            size_t workspace_bytes, const int* cu_seqlens, int num_seqs, int total_tokens,
                            int max_seqlen, int Hq, int Hkv, int D, int causal, float scale, void* stream);

/* Cached (decode) attention: the newest Tq positions of each batch row
 * attend to that row's KV cache -- the cached GQA / per-row-prefix cached
 * attention and KV-cache decode of the microLLM-rocm README (section "Why
 * this project exists"), with the forward's mathematics above restricted to
 * Tq query rows per sequence:
 *
 *   row b holds n_b = cache_lens[b] keys (the Tq new ones included); query
 *   t (0 <= t < Tq) of row b is position n_b - Tq + t and sees the keys
 *   j <= n_b - Tq + t of its own row (the causal mask aligned to the end of
 *   the cache); query head h reads K/V head h / (Hq / Hkv).
 *
 * Layouts (device pointers, 16-byte aligned, densely packed):
 *   q, o      bf16 [B, Hq, Tq, D]     (the new queries, the output)
 *   k_cache,
 *   v_cache   bf16 [B, Hkv, S, D]     (S = cache capacity; rows past n_b are
 *                                      never used and may hold anything)
 *   lse       float32 [B, Hq, Tq]     (natural log)
 *   cache_lens DEVICE int32 [B], Tq <= cache_lens[b] <= S.  A row outside
 *             that range is reported through the device status word
 *             (ATTN_ERR_SEQLENS) and its outputs are left unwritten.
 * workspace: attn_decode_workspace_size() bytes, 256-byte aligned, no
 * initialisation needed; the size is 0 (workspace may be NULL) when the
 * key range is not split.  Limits: Tq <= S; B*Hq*Tq < 2^31. */
GQA_ATTN_API size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Tq, int S, int D);

/* Rotary queries (positions-aware RoPE of the microLLM-rocm README, section
 * "Why this project exists"; RoPE / MultiHeadAttentionWithRoPE of the
 * llm-from-scratch "Project Overview"), for both decode entry points:
 * rope_cos_sin NULL = none; otherwise a DEVICE float32 table
 * [rope_positions, D], 16-byte aligned, rope_positions >= the cache capacity
 * (S, or max_pages * page_size): row p holds cos(p*theta_i) for i < D/2, then
 * sin(p*theta_i).  Each query t of row b is rotated at its position
 * p = cache_lens[b] - Tq + t before the scores: feature i pairs with feature
 * i + D/2, x'_i = x_i cos - x_{i+D/2} sin, x'_{i+D/2} = x_{i+D/2} cos + x_i sin,
 * computed in f32 and carried into the score MMA to about 2^-16 of each
 * element (a bf16 value plus a bf16 remainder; E4M3 caches: the three E4M3
 * parts below).  The cache must hold keys already rotated at their
 * positions (as appending them rotated leaves them). */
GQA_ATTN_API attn_status attn_decode_fwd(const void* q, const void* k_cache, const void* v_cache,
                                         const int* cache_lens, void* o, float* lse, void* workspace,
                                         size_t workspace_bytes, int B, int Hq, int Hkv, int Tq, int S, int D,
                                         float scale, const float* rope_cos_sin, int rope_positions, void* stream);

/* Cached attention over a PAGED KV cache (the paged KV-cache management of
 * the RoseLLM README, section "Inference and serving").  Same queries, mask
 * and outputs as attn_decode_fwd; the cache is a pool of pages:
 *   k_pages, v_pages  bf16 [num_pages, Hkv, page_size, D]: a page holds
 *                     page_size consecutive positions of one batch row,
 *                     every K/V head (each (page, head) block contiguous)
 *   block_table       DEVICE int32 [B, max_pages]: key position j of row b
 *                     is row j % page_size of page block_table[b*max_pages + j/page_size];
 *                     only the entries of pages that hold one of the row's
 *                     cache_lens[b] keys are read
 *   cache_lens        DEVICE int32 [B], Tq <= cache_lens[b] <= max_pages * page_size
 * page_size: 16, 32, 64 or a multiple of 128.  workspace: as attn_decode_fwd
 * with S = max_pages * page_size (attn_decode_workspace_size).  An entry
 * outside [0, num_pages) is reported through the device status word
 * (ATTN_ERR_PAGES) and the page is read as zeros (the row's result is then
 * meaningless, no memory outside the pool is touched). */
GQA_ATTN_API attn_status attn_decode_paged_fwd(const void* q, const void* k_pages, const void* v_pages,
                                               const int* block_table, const int* cache_lens, void* o, float* lse,
                                               void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                                               int Tq, int page_size, int num_pages, int max_pages, int D,
                                               float scale, const float* rope_cos_sin, int rope_positions,
                                               void* stream);

/* Cached attention over FP8 K/V caches (the FP8 E4M3 quantize/dequantize
 * and KV-cache decode of the microLLM-rocm README, section "Why this project
 * exists"): same queries, mask and outputs as attn_decode_fwd /
 * attn_decode_paged_fwd, with the caches stored as E4M3 codes (1 byte each:
 * sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities) and one
 * scale per cache: K = e4m3(k8) * k_scale, V = e4m3(v8) * v_scale.
 *   k8, v8           uint8 [B, Hkv, S, D]  (contiguous), or
 *   k8_pages, v8_pages uint8 [num_pages, Hkv, page_size, D]  (paged, as
 *                    attn_decode_paged_fwd)
 * The scores are taken on the K codes as stored: each query row q (after
 * rotation, if any) is split into three E4M3 parts with one f32 scale per
 * row, q = s (h0 + h1 + h2), s = max|q| / 448, which holds q to about 2^-12
 * of each element (2^-19 of the row's largest for elements below E4M3's
 * normal range); the products accumulate in f32.  V is widened exactly to
 * f16 and P is rounded to f16 for the P V product (f32 accumulation).  NaN
 * codes at visible keys give NaN where the definition does; codes past
 * cache_lens[b] are never used.  Workspace, rotary table and errors as
 * attn_decode_fwd. */
GQA_ATTN_API attn_status attn_decode_fp8_fwd(const void* q, const void* k8, const void* v8, float k_scale,
                                             float v_scale, const int* cache_lens, void* o, float* lse,
                                             void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Tq,
                                             int S, int D, float scale, const float* rope_cos_sin,
                                             int rope_positions, void* stream);

GQA_ATTN_API attn_status attn_decode_paged_fp8_fwd(const void* q, const void* k8_pages, const void* v8_pages,
                                                   float k_scale, float v_scale, const int* block_table,
                                                   const int* cache_lens, void* o, float* lse, void* workspace,
                                                   size_t workspace_bytes, int B, int Hq, int Hkv, int Tq,
                                                   int page_size, int num_pages, int max_pages, int D, float scale,
                                                   const float* rope_cos_sin, int rope_positions, void* stream);

/* Static description of a status code. */
GQA_ATTN_API const char* attn_status_string(attn_status status);

/* Synchronises `stream`, then reads the current device's status word into
 * *out (ATTN_OK or the first device-detected error since it was last
 * cleared); clears it when clear != 0.  Returns ATTN_ERR_CUDA if the copy
 * fails (e.g. a sticky CUDA error), else ATTN_OK. */
GQA_ATTN_API attn_status attn_get_device_status(void* stream, int* out, int clear);

/* Debug build (libgqa_attn_debug.so, compiled with -DGQA_DEBUG; no
 * counterpart in the pages): the kernels check every computed tensor-map
 * coordinate, global row offset, workspace row and rotary-table row against
 * its bounds before the access; a failed check skips the access, records
 * ATTN_ERR_CHECK in the status word and its source line in a second word.
 * attn_get_check_line synchronises `stream` and reads (and clears when
 * clear != 0) that line: 0 when no check failed, always 0 in the release
 * build.  attn_is_debug_build returns 1 in the debug build, 0 otherwise. */
GQA_ATTN_API attn_status attn_get_check_line(void* stream, int* out, int clear);
GQA_ATTN_API int attn_is_debug_build(void);

/* Failure-path self-test (no counterpart in the pages).  Launches one small
 * kernel that waits, through the library's bounded in-kernel wait, on a
 * barrier that nothing ever completes, with a limit of limit_ms milliseconds
 * (1..5000).  The wait expires, ATTN_ERR_TIMEOUT is recorded in the device
 * status word and the kernel returns normally: the GPU is neither hung nor
 * faulted, and attn_get_device_status() then reports the timeout. */
GQA_ATTN_API attn_status attn_selftest_wait_timeout(int limit_ms, void* stream);

/* Failure-path test of the production kernels (no counterpart in the pages;
 * not thread-safe).  Arms one injected failure for the next launch of one
 * kernel: 1 the forward (attn_fwd and attn_fwd_rope), 2 the backward's dK/dV
 * kernel, 3 the backward's dQ kernel (attn_bwd and its variants); 0 disarms.
 * In that launch every bounded wait gives up after limit_ms (1..5000) instead
 * of the usual 2 s, and one CTA's TMA producer stops before the loads of
 * its second step (the forward's and the dK/dV kernel's first CTA; for the
 * persistent dQ kernel, the CTA that takes its first tile), so one of that
 * CTA's waits expires.  The kernel then
 * records ATTN_ERR_TIMEOUT in the device status word, its other roles see
 * the CTA's abort flag and stop, the issued copies and MMAs are drained,
 * TMEM is freed and the kernel returns: the GPU is neither hung nor faulted
 * and the next call runs normally.  The failing CTA's outputs are left
 * unwritten or partial; every other CTA completes.  The injection is
 * consumed by the launch that takes it. */
GQA_ATTN_API attn_status attn_test_inject_timeout(int kernel, int limit_ms);

/* Kernel timing (instrumentation; not thread-safe).  While enabled, every
 * kernel launch is bracketed by a CUDA event pair recorded on the caller's
 * stream.  attn_profile_read synchronises those events and returns, for one
 * kernel kind (0 forward, 1 backward preprocess, 2 backward dK/dV kernel,
 * 3 unused, 4 decode partial, 5 decode split merge, 6 backward dQ kernel),
 * the
 * number of launches and their summed device
 * time in milliseconds since the last attn_profile_reset.  At most 65536
 * launches are recorded between resets.  Off by default. */
GQA_ATTN_API attn_status attn_profile_enable(int enable);
GQA_ATTN_API attn_status attn_profile_reset(void);
GQA_ATTN_API attn_status attn_profile_read(int kind, int* launches, double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H_ */
