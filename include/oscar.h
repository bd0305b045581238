/*
 * oscar.h -- C ABI of the GB300 (sm_103a) OSCAR INT2 rotated KV-cache library.
 *
 * OSCAR keeps a mixed-precision paged KV cache: the first 64 tokens (attention
 * sinks) and the last 256 tokens before the current position stay BF16, and
 * everything in between is stored as 2-bit codes after a fixed per-layer
 * rotation R = U * H_Had * P_br and per-layer clipping.
 *   - ainsights.it "OSCAR: Come Together AI Comprime la KV Cache a 2-bit per
 *     LLM", sections "I tre fattori della rotazione" and "Architettura del
 *     Sistema di Serving e Layout di Memoria";
 *   - edge.aivizor.me "Together AI выпустила исходники OSCAR — INT2-квантование
 *     KV-кэша для долгих контекстов LLM", composition and deployment paragraphs;
 *   - gist.science "Resumen Técnico: OSCAR - Rotación Consciente de la
 *     Covarianza Espectral Offline para Cuantización de Cache KV de 2 bits",
 *     §2.2 A (rotations, clip thresholds) and §2.2 B (paged cache, fused kernel).
 *
 * Conventions for every call
 *   - All pointers named "device" point to memory on the context's CUDA
 *     device; the caller allocates and frees them.  "host" pointers are read
 *     before the call returns.  The library allocates device memory only in
 *     oscar_create (a 4-byte error word) and oscar_load_rotation (rotation
 *     constants); append and decode never allocate.
 *   - Work is queued asynchronously on the given stream (a cudaStream_t passed
 *     as void*; NULL is the legacy default stream).
 *   - Host-side argument checks return a status and launch nothing.
 *   - Index checks that need device data (page ids, slots, lengths) are made
 *     by the kernels: a bad index sets a bit in the context's device error
 *     word and the offending work item is skipped (never a trap).  Read and
 *     clear the word with oscar_check_device_error.
 *   - Nothing throws across the ABI.  The library is not thread-safe per
 *     context; distinct contexts are independent.
 *
 * Fixed shape: head_dim 128, page 64 tokens, sink 64, recent window 256,
 * quantisation group 64 channels (one fp16 scale per token per group).
 */
#ifndef OSCAR_H
#define OSCAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OSCAR_HEAD_DIM 128
#define OSCAR_PAGE_TOKENS 64
#define OSCAR_SINK_TOKENS 64
#define OSCAR_RECENT_TOKENS 256
#define OSCAR_GROUP 64
#define OSCAR_MAX_GQA 8

/*
 * Packed INT2 block: one page (64 positions) of one KV head, 4608 bytes.
 *   [   0, 2048)  K codes      [2048, 2304)  K scales fp16 [64 tokens][2 groups]
 *   [2304, 4352)  V codes      [4352, 4608)  V scales fp16 [64 tokens][2 groups]
 * Codes come in 16-token tiles of 512 bytes (tile T = t / 16 at byte 512*T of
 * the code area).  With u = t % 16, the 2-bit code of rotated channel j is at
 *   K: lane = 4*(u%8) + (j/4)%4,   word = 2*(u/8) + j/64,
 *      bit  = 8*(j%4) + 2*(2*((j/32)%2) + (j/16)%2)
 *   V: lane = 4*(j%8) + (u%8)/2,   word = 2*(u/8) + (j%16)/8,
 *      bit  = 16*(u%2) + 2*(j/16)
 *   byte = 512*T + 16*lane + 4*word + bit/8, bit-in-byte = bit%8
 * (little-endian 32-bit words).  A code c stands for the level (c - 1.5) * s.
 * The layout lets one warp load a 16-token tile with one 16-byte load per
 * lane and hand the unpacked codes straight to the tensor cores.
 */
#define OSCAR_BLOCK_BYTES 4608
#define OSCAR_BLOCK_K_CODES 0
#define OSCAR_BLOCK_K_SCALES 2048
#define OSCAR_BLOCK_V_CODES 2304
#define OSCAR_BLOCK_V_SCALES 4352

typedef enum {
  OSCAR_OK = 0,
  OSCAR_ERR_INVALID_ARG = 1,   /* null pointer, bad size or index, unsupported shape */
  OSCAR_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement */
  OSCAR_ERR_NOT_LOADED = 3,    /* the layer's rotation was never loaded */
  OSCAR_ERR_CUDA = 4,          /* a CUDA runtime call failed */
  OSCAR_ERR_DEVICE_CHECK = 5,  /* a kernel found a bad index (see oscar_check_device_error) */
  OSCAR_ERR_WORKSPACE = 6      /* workspace missing or too small */
} oscar_status;

/* Device error word bits (oscar_check_device_error). */
#define OSCAR_DEVERR_PAGE 1u       /* page-table entry outside [0, num_pages) */
#define OSCAR_DEVERR_SINK 2u       /* sink page index outside [0, num_sink_pages) */
#define OSCAR_DEVERR_RING 4u       /* ring slot outside [0, num_ring_slots) */
#define OSCAR_DEVERR_LENGTH 8u     /* a length or position beyond the table's capacity */
#define OSCAR_DEVERR_TOKENS 16u    /* cu_seqlens inconsistent with n_tokens */
#define OSCAR_DEVERR_TIMEOUT 32u   /* a kernel's bounded wait on an asynchronous copy or a
                                      shared-memory barrier gave up (the copy never landed);
                                      the kernel skipped the rest of that work item, waited
                                      (bounded) for its copies in flight and returned, so the
                                      context stays usable but that call's outputs are invalid */

typedef struct oscar_ctx oscar_ctx;

typedef struct {
  int32_t num_layers;
  int32_t num_q_heads;
  int32_t num_kv_heads;   /* num_q_heads % num_kv_heads == 0, ratio <= 8 */
  int32_t head_dim;       /* must be 128 */
  int32_t page_size;      /* must be 64 */
  int32_t sink;           /* must be 64 */
  int32_t recent;         /* must be 256 */
  int32_t group;          /* must be 64 */
  int32_t device;         /* CUDA device ordinal */
} oscar_config;

/*
 * One layer's cache, all device memory owned by the caller; every pool
 * 16-byte aligned.
 *   int2_pages  [num_pages][num_kv_heads][OSCAR_BLOCK_BYTES] bytes.
 *   k_sink, v_sink  bf16 [num_sink_pages][num_kv_heads][64][128]: positions 0..63.
 *   k_ring, v_ring  bf16 [num_ring_slots][num_kv_heads][256][128]: position p >= 64
 *               of a request lives in row (p - 64) % 256 of its ring slot.
 *               With a recent_page_table they are instead a pool of
 *               num_ring_slots BF16 pages [num_kv_heads][64][128].
 *   page_table  int32 [batch][max_pages_per_req]: entry i (i >= 1) is the
 *               physical INT2 page of positions [64 i, 64 i + 64); entry 0 is
 *               unused.  Entries may alias (shared prefixes); the caller
 *               allocates pages, including the page an upcoming eviction
 *               writes, and never lets an append write a shared page.
 *   sink_page   int32 [batch]: physical sink page of each request (may alias).
 *   ring_slot   int32 [batch]: ring slot of each request (must not alias).
 * The same view describes every layer when the caller keeps per-layer pools;
 * only the pool pointers differ between layers.
 */
typedef struct {
  void* int2_pages;
  int64_t num_pages;
  void* k_sink;
  void* v_sink;
  int64_t num_sink_pages;
  void* k_ring;
  void* v_ring;
  int64_t num_ring_slots;
  const int32_t* page_table;
  int32_t max_pages_per_req;
  const int32_t* sink_page;
  const int32_t* ring_slot;
  int32_t batch;
  /*
   * Optional paged recent window (NULL: the ring).  int32 [batch][max_pages_per_req]:
   * entry i names the BF16 page (in k_ring / v_ring) holding the recent rows of
   * positions [64 i, 64 i + 64), row p % 64 for position p.  The window is still
   * the last 256 positions ([IT] "Architettura ...": the 256 most recent tokens
   * stay BF16); the entries of the logical pages it touches (at most five, and
   * the one an append writes) must be valid, the others are not read.  Pages of
   * positions shared by several requests may alias; as with page_table, the
   * caller never lets an append write a shared page.  ring_slot may be NULL.
   */
  const int32_t* recent_page_table;
} oscar_cache_view;

/* Append flags. */
#define OSCAR_APPEND_FRESH_RING 1u  /* positions before pos[] are already sink/history
                                       (e.g. an aliased prefix): evict nothing.  The
                                       ring then holds only new tokens, so each request
                                       must append >= 256 tokens unless pos <= 64
                                       (else OSCAR_DEVERR_LENGTH, nothing written). */

/*
 * New tokens.  k, v: device bf16 [n_tokens][num_kv_heads][128], 16-byte aligned.
 *   pos         device int32 [batch]: position of each request's first new token
 *               (its context length before this append).
 *   cu_seqlens  device int32 [batch + 1]: request b owns tokens
 *               [cu_seqlens[b], cu_seqlens[b+1]); NULL means exactly one token
 *               per request (decode) and n_tokens == batch.
 *   max_tokens_per_req  host upper bound of cu_seqlens[b+1] - cu_seqlens[b].
 */
typedef struct {
  const void* k;
  const void* v;
  const int32_t* pos;
  const int32_t* cu_seqlens;
  int32_t n_tokens;
  int32_t max_tokens_per_req;
  uint32_t flags;
} oscar_append_args;

/*
 * Decode queries: one new query per request, attending over its whole context
 * (the just-appended token included; no mask is needed for the last query).
 *   q        device bf16 [batch][num_q_heads][128], original (unrotated) basis.
 *   out      device fp32 [batch][num_q_heads][128].  Query head h reads KV
 *            head h / (num_q_heads / num_kv_heads).  A request with
 *            ctx_len 0 gets zeros.
 *   ctx_len  device int32 [batch]: context length after the append.
 *   max_ctx_len  host upper bound of ctx_len (sizes the launch grid).
 *   sm_scale softmax scale; <= 0 selects 1/sqrt(128).
 */
typedef struct {
  const void* q;
  float* out;
  const int32_t* ctx_len;
  int32_t max_ctx_len;
  float sm_scale;
} oscar_decode_args;

/* BF16-cache comparator: every position BF16 in 64-token pages.
 *   k_pages, v_pages  bf16 [num_pages][num_kv_heads][64][128]
 *   page_table        int32 [batch][max_pages_per_req]: entry i holds positions
 *                     [64 i, 64 i + 64) (entry 0 included). */
typedef struct {
  const void* k_pages;
  const void* v_pages;
  int64_t num_pages;
  const int32_t* page_table;
  int32_t max_pages_per_req;
  int32_t batch;
} oscar_bf16_cache_view;

/* Rotation flags for oscar_load_rotation: which factors of R = U H P to use.
 * OSCAR_ROT_ALL is the method; dropping factors gives the pages' baselines
 * (naive INT2: none; Hadamard-only: H|P). */
#define OSCAR_ROT_U 1u
#define OSCAR_ROT_H 2u
#define OSCAR_ROT_P 4u
#define OSCAR_ROT_ALL 7u

/* Create a context for one model shape on config->device.  Fails with
 * OSCAR_ERR_INVALID_ARG for any shape other than the fixed one above. */
oscar_status oscar_create(const oscar_config* config, oscar_ctx** out);

/* Free the context and its device constants.  NULL is a no-op. */
void oscar_destroy(oscar_ctx* ctx);

/*
 * Upload one layer's rotation: R_K = U_K H P and R_V = U_V H P ([ES] §2.2 A.3;
 * [RU] composition paragraph) and the clip thresholds tau_k, tau_v
 * ([ES] §2.2 A.4).  U_K, U_V: host fp32 [128][128] row-major, columns are
 * the eigenvectors (a token row x is rotated as x' = x R).  They must be
 * orthogonal; the library does not check.  tau > 0, finite or +inf, and
 * tau / 1.5 must fit fp16 (tau <= 98256).  The library forms the composite
 * R = U H P of the enabled factors (flags) in double precision and keeps R_K,
 * R_V and R_V^T in fp32 on the device; every kernel applies the rotation as
 * one dense product with R.  Synchronous (copies before return).
 */
oscar_status oscar_load_rotation(oscar_ctx* ctx, int32_t layer, const float* U_K, const float* U_V,
                                 float tau_k, float tau_v, uint32_t flags);

/*
 * Append new K/V tokens to one layer's cache ([IT] "Architettura ...": each
 * token is rotated, clipped and quantised when it enters the INT2 history).
 * Phase 1 (unless OSCAR_APPEND_FRESH_RING) moves ring tokens that fall out of
 * the 256-token window into their INT2 rows; phase 2 writes each new token:
 * positions < 64 to the sink page, positions >= L - 256 (L = final length) to
 * the ring, the rest straight into INT2 rows.  Rotation: x' = x R in fp32
 * with the layer's composite R, clip a = min(max|x'|, tau) per group of 64,
 * s = fp16(a / 1.5), code = [x' >= -s] + [x' >= 0] + [x' >= s].
 */
oscar_status oscar_kv_append(oscar_ctx* ctx, int32_t layer, const oscar_cache_view* view,
                             const oscar_append_args* args, void* stream);

/* Workspace bytes oscar_decode_attention needs for up to max_batch requests
 * of up to max_ctx_len tokens. */
size_t oscar_decode_workspace_bytes(const oscar_ctx* ctx, int32_t max_batch, int32_t max_ctx_len);

/*
 * Fused decode attention over one layer's mixed cache ([ES] §2.2 B: one
 * kernel unpacks, de-quantises, undoes the rotation and computes attention;
 * [IT] "Architettura ...": no extra memory traffic).  q is rotated into the
 * K basis (q' = q R_K), the INT2 history is unpacked in registers and
 * consumed by split-K flash-decoding on the tensor cores, the BF16 sink and
 * recent tokens are attended in the original basis, and the rotated-basis
 * part of the output is rotated back (acc R_V^T) when the splits are merged.
 * No dequantised cache is materialised.  workspace: device, at least
 * oscar_decode_workspace_bytes(ctx, batch, max_ctx_len) bytes, 256-byte
 * aligned, owned by the caller; its contents need no initialisation for
 * this call and are scratch between calls (oscar_decode_step wants them
 * zero before its first use).  Calls that share a workspace must not
 * overlap on the GPU.
 */
oscar_status oscar_decode_attention(oscar_ctx* ctx, int32_t layer, const oscar_cache_view* view,
                                    const oscar_decode_args* args, void* workspace, size_t workspace_bytes,
                                    void* stream);

/*
 * Extend (chunk) attention over one layer's mixed cache (the second workload
 * on the same layout: a chunk of new queries reading the cached prefix --
 * [IT] "Architettura ...": SGLang serves prefix-cache hits and chunked
 * prefill from the same paged INT2 cache; [ES] §2.2 B).  Query b attends,
 * through the cache of its table row b, the positions p < min(limit[b],
 * ctx_len[b]) of the cache as it stands: ctx_len[b] is the cache length
 * (the chunk appended first with oscar_kv_append), and the sink / INT2
 * history / BF16 recent split follows ctx_len[b]; limit[b] (device int32
 * [batch], e.g. P + i + 1 for the i-th token of a chunk appended at P) is
 * the causal bound.  The queries of one chunk are batch rows whose table
 * entries alias the same pages, sink page and ring slot.  Each query runs
 * the split-K decode over the shared pages (the unpack is not shared across
 * the queries of a chunk).  Same arguments, workspace, errors and output as
 * oscar_decode_attention.
 */
oscar_status oscar_extend_attention(oscar_ctx* ctx, int32_t layer, const oscar_cache_view* view,
                                    const oscar_decode_args* args, const int32_t* limit, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * Extend attention for equal-size chunks, with the work shared across each
 * chunk's queries (the prefill / extend workload of [ES] §2.2 B and [IT]
 * "Architettura ...").  Request b of the view (its own table row) has
 * ctx_len[b] cached positions, the chunk at pos0[b] .. pos0[b] + chunk - 1
 * among them (appended first); query i of request b attends positions
 * p < min(pos0[b] + i + 1, ctx_len[b]), as oscar_extend_attention would.
 * q: device bf16 [batch][chunk][H_q][128]; out: device fp32, same shape.
 * One block serves 128 / g queries of one (request, KV head), g = H_q / H_kv:
 * each INT2 page is copied once and unpacked once into fp16 tiles in shared
 * memory, and the group's 128 (query, head) rows run its Q.K and P.V as
 * tensor-core MMAs with the scores and outputs in tensor memory.  Needs
 * g <= 4 (else OSCAR_ERR_UNSUPPORTED;
 * oscar_extend_attention serves any GQA ratio) and batch * chunk <= 65535.
 * workspace: device, 256-byte aligned, at least
 * oscar_extend_workspace_bytes(ctx, batch, chunk, max_ctx_len) bytes; zero
 * before its first use (as for oscar_decode_step).  max_ctx_len: the largest
 * ctx_len[b] of the call.  Errors: as oscar_decode_attention.
 */
size_t oscar_extend_workspace_bytes(const oscar_ctx* ctx, int32_t batch, int32_t chunk, int32_t max_ctx_len);
oscar_status oscar_extend_chunk(oscar_ctx* ctx, int32_t layer, const oscar_cache_view* view, const void* q,
                                float* out, const int32_t* ctx_len, const int32_t* pos0, int32_t chunk,
                                int32_t max_ctx_len, float sm_scale, void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * One decode step of one layer: oscar_kv_append of one new token per
 * request, then oscar_decode_attention, in one kernel launch instead of
 * three ([IT] "Architettura ...": the decode path is append, evict/quantise,
 * attend).  Every block of the split-K decode rotates its request's queries
 * into the K basis itself; the block whose history pages hold the row the
 * new token evicts writes the new K/V token (evicting and quantising the
 * ring row it replaces) and attends that row from its own copy; the BF16
 * tiles take the new token's row from the input.  The kernel is launched
 * with programmatic dependent launch, so it may start its prologue (loads of
 * the layer's constants and L2 prefetches) while the kernel before it on the
 * stream drains; it reads nothing that kernel writes until it has completed.
 * append: cu_seqlens NULL, n_tokens == batch, flags 0 or
 * OSCAR_APPEND_FRESH_RING (same meaning as for oscar_kv_append); decode: as
 * oscar_decode_attention, with ctx_len[b] normally pos[b] + 1 so that the
 * token just written is attended.  Results equal oscar_kv_append followed by
 * oscar_decode_attention on the same arguments.  workspace: as for
 * oscar_decode_attention, except that it must hold zeros before its first
 * use by this call (every decode call leaves the counters it uses at zero).
 * Errors: as the two calls; nothing is launched when either argument set is
 * rejected.
 */
oscar_status oscar_decode_step(oscar_ctx* ctx, int32_t layer, const oscar_cache_view* view,
                               const oscar_append_args* append, const oscar_decode_args* decode,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * Allocation-free variant of oscar_decode_attention (the pages have no
 * counterpart: this is a service of this library).  Some callers cannot
 * allocate device memory: a plugin inside an inference engine whose memory
 * planner owns every device allocation and hands out no workspace, or a
 * latency-critical serving loop that must not call cudaMalloc (it can
 * synchronise the device) once it is running.  This entry point takes the
 * decode scratch from a static device array of OSCAR_NOALLOC_SCRATCH_BYTES
 * (16 MiB) built into the library; every GPU that loads the library holds it
 * until the process exits.  Same arguments and results as
 * oscar_decode_attention minus the workspace; the caller still owns q, out,
 * the cache and the lengths.  A call whose scratch need
 * (oscar_decode_workspace_bytes for its batch and max_ctx_len) exceeds the
 * array returns OSCAR_ERR_WORKSPACE and launches nothing.  The first call on
 * a device looks up the array's device address with that device current, so
 * make that first call before any stream capture.  All calls share the one
 * array, which keeps the last call's contents (the kernels re-initialise what
 * they need): calls that overlap on the GPU, from any stream or thread, race
 * and must be serialised by the caller.  Allocates nothing.
 */
#define OSCAR_NOALLOC_SCRATCH_BYTES (16u << 20)
oscar_status oscar_decode_attention_noalloc(oscar_ctx* ctx, int32_t layer, const oscar_cache_view* view,
                                            const oscar_decode_args* args, void* stream);

/* Comparator: the same decode over a plain BF16 paged cache (the baseline
 * the pages' decode speed-ups are quoted against).  Same workspace rules. */
oscar_status oscar_decode_attention_bf16(oscar_ctx* ctx, const oscar_bf16_cache_view* view,
                                         const oscar_decode_args* args, void* workspace,
                                         size_t workspace_bytes, void* stream);

/*
 * Offline calibration on the GPU ([RU] "Техническая идея": the keys' basis
 * from C_Q = (1/N) sum_n q_n^T q_n, the values' basis from the score-weighted
 * C_S = (1/N) V^T S^T S V; [ES] §2.2 A steps 1-4: both covariances on a
 * small calibration set, a spectral decomposition, per-layer clip
 * thresholds from the rotated calibration activations).  The
 * eigendecomposition (U = eigenvectors of C_Q or C_S by descending
 * eigenvalue) is left to the caller, on the host; its U then goes to
 * oscar_calib_clip_threshold and oscar_load_rotation.
 *
 * Workspace: device, 256-byte aligned, at least
 * oscar_calib_workspace_bytes(n_queries, n_keys, n_kv_heads, n_clip_rows)
 * bytes (0: arguments out of range), owned by the caller, scratch between
 * calls.  Row counts are at most OSCAR_CALIB_MAX_ROWS.
 */
#define OSCAR_CALIB_MAX_ROWS (1 << 20)
size_t oscar_calib_workspace_bytes(int64_t n_queries, int64_t n_keys, int32_t n_kv_heads, int64_t n_clip_rows);

/*
 * C_Q and C_S of one layer.  q: device fp32 [n_q][128] calibration queries;
 * k, v: device fp32 [n_kv_heads][n_k][128] calibration keys and values per
 * KV head.  S = softmax(q k_h^T sm_scale) row-wise over the n_k keys of head
 * h (no causal mask); C_S averages (1/n_q) (S_h v_h)^T (S_h v_h) over the
 * heads.  Outputs: device fp64 [128][128] c_q and c_s (row-major).  Products
 * in fp32 within 32-row stages, sums across stages in fp64; the attention in
 * fp32 with an online softmax.  Asynchronous on the stream.  Errors:
 * OSCAR_ERR_INVALID_ARG (null pointers, counts out of range, sm_scale not
 * positive and finite), OSCAR_ERR_WORKSPACE, OSCAR_ERR_CUDA.
 */
oscar_status oscar_calib_covariances(oscar_ctx* ctx, const float* q, int64_t n_q, const float* k, const float* v,
                                     int64_t n_k, int32_t n_kv_heads, float sm_scale, double* c_q, double* c_s,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Clip threshold: the given percentile (0..100) of |x R| over all n_rows x
 * 128 entries, with numpy's linear interpolation between the order
 * statistics around percentile / 100 (n - 1).  x: device fp32 [n_rows][128]
 * (e.g. every calibration K row of a layer, all heads); U: host fp32
 * [128][128] with the flags of oscar_load_rotation, R = U H P formed in fp64
 * as there.  |x R| is sorted on the device (an exact bitonic sort of the
 * float bits).  Synchronises the stream and writes the threshold to the host
 * double *tau.  Errors: OSCAR_ERR_INVALID_ARG (null pointers, counts or
 * percentile out of range, unknown flags, non-finite U), OSCAR_ERR_WORKSPACE,
 * OSCAR_ERR_CUDA.
 */
oscar_status oscar_calib_clip_threshold(oscar_ctx* ctx, const float* x, int64_t n_rows, const float* U,
                                        uint32_t flags, double percentile, double* tau, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Synchronise the stream, return and clear the device error word in *bits
 * (may be NULL).  Returns OSCAR_ERR_DEVICE_CHECK when any bit was set. */
oscar_status oscar_check_device_error(oscar_ctx* ctx, void* stream, uint32_t* bits);

/*
 * Self-test of the failure path (no page passage: a library service).  One
 * block runs both bounded waits the kernels use on their copies and barriers,
 * each on a shared-memory barrier that nothing completes: the polled wait
 * gives up after `polls` polls (1 .. 2^18, the kernels' own limit: about a
 * second), the timed wait (the chunk-extend kernel's) after polls x 4 us on
 * the global timer.  When both have given up it sets OSCAR_DEVERR_TIMEOUT in
 * the context's device error word and returns, leaving nothing in flight.
 * The context stays usable.  Asynchronous on `stream`; read the result with
 * oscar_check_device_error.  Errors: OSCAR_ERR_INVALID_ARG (null context,
 * polls out of range), OSCAR_ERR_CUDA.
 */
oscar_status oscar_selftest_bounded_wait(oscar_ctx* ctx, uint32_t polls, void* stream);

/* Number of SMs of the context's device (used to size launch grids). */
int32_t oscar_device_sm_count(const oscar_ctx* ctx);

/* Static description of a status code. */
const char* oscar_status_string(oscar_status status);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H */
