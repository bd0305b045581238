// Internal launch interface between the C-ABI layer (oscar_api.cu) and the
// kernels (oscar_append.cu, oscar_decode.cu).  Not part of the public ABI.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace oscar {

// Raise a kernel's dynamic shared-memory limit once per device.  `done`
// holds one bit per device ordinal (0..63) whose attribute is set; it is an
// atomic, so concurrent first launches from several host threads are safe
// (both may set the attribute, which is idempotent).
inline cudaError_t smem_attr_once(const void* kernel, size_t bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// One layer's rotation constants on the device: R = U H P (the factors the
// layer enables) as dense matrices, formed in double precision on the host
// and rounded to fp32.
struct LayerRotation {
  const float* R_K = nullptr;   // [128][128] row-major: a K row x is rotated as x R_K
  const float* R_V = nullptr;   // [128][128] row-major
  const float* R_VT = nullptr;  // [128][128] = R_V transposed (inverse rotation of outputs)
  // bf16 bit patterns [2 (K, V)][3][128 n][128 k]: R[k][n] = sum of the three
  // terms up to ~2^-24 relative (the bulk append's tensor-core operand)
  const uint16_t* RT_split = nullptr;
  float tau_k = 0.f, tau_v = 0.f;
  // the factors R is made of (kRotU | kRotH | kRotP).  Without a calibrated U
  // the one-token writes, the q rotation and the decode's inverse rotation
  // apply H as an in-register Walsh-Hadamard butterfly and P as an index map
  // instead of the dense product; the bulk append and the chunk kernel keep
  // the dense R (its tensor-core product costs the same either way).
  uint32_t flags = 7u;
};
constexpr uint32_t kRotU = 1u, kRotH = 2u, kRotP = 4u;

struct CacheRefs {
  uint8_t* pages = nullptr;
  int64_t num_pages = 0;
  uint16_t* k_sink = nullptr;
  uint16_t* v_sink = nullptr;
  int64_t num_sink = 0;
  uint16_t* k_ring = nullptr;
  uint16_t* v_ring = nullptr;
  int64_t num_ring = 0;
  const int32_t* page_table = nullptr;
  int32_t max_pages = 0;
  const int32_t* sink_page = nullptr;
  const int32_t* ring_slot = nullptr;
  int32_t batch = 0;
  int32_t num_kv_heads = 0;
  const int32_t* recent_table = nullptr;  // [batch][max_pages] BF16 recent pages (null: the ring)
};

struct AppendLaunch {
  CacheRefs c;
  LayerRotation rot;
  const uint16_t* k = nullptr;  // bf16 [n_tokens][Hkv][128]
  const uint16_t* v = nullptr;
  const int32_t* pos = nullptr;
  const int32_t* cu_seqlens = nullptr;  // nullptr: one token per request
  int32_t n_tokens = 0;
  int32_t max_tokens_per_req = 0;
  unsigned flags = 0;
  unsigned* err = nullptr;
};

cudaError_t launch_append(const AppendLaunch& a, cudaStream_t stream);

// One block's bounded wait on a barrier nothing completes: sets the timeout bit in *err.
cudaError_t launch_selftest_wait(unsigned* err, unsigned polls, cudaStream_t stream);

// A launch that may start once the kernel before it in the stream has let its
// dependents go (griddepcontrol.launch_dependents) or has finished; the kernel
// waits (griddepcontrol.wait) before it touches what that kernel writes.
inline cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// decode workspace layout (bytes, all offsets 256-aligned)
struct DecodePlan {
  int32_t batch = 0, Hq = 0, Hkv = 0, g = 0;
  int32_t chunk_pages = 0;   // pages per work item
  int32_t n_chunks = 0;      // paged work items per (request, KV head)
  int32_t n_items = 0;       // all work items per (request, KV head)
  int32_t tiles_per_item = 0;  // mixed cache: BF16 sink/recent tiles per item (items 0, 1, ... take them)
  int32_t rec_floats = 0;      // floats per partial record
  int32_t prep_rows = 1;       // rows (requests) per block of the q rotation kernel
  size_t off_counters = 0, off_qfrag = 0, off_qplain = 0, off_qconst = 0, off_partials = 0, total = 0;
};

// a warp state in shared memory: m[8], l[8], acc[8][kStateStride] (a head's
// 128 channels, padded so that the packed state stores hit distinct banks)
constexpr int kStateStride = 128 + 8;
constexpr int kPartialFloats = 16 + 8 * kStateStride;
// a partial record in the workspace: m[8], l[8], acc[g][128]
constexpr int partial_record_floats(int g) { return 16 + 128 * g; }
constexpr int kQConstFloats = 32;
constexpr int kQFragWords = 32 * 32;   // q fragments per (request, KV head): [lane][32]

DecodePlan plan_decode(int mode, int batch, int Hq, int Hkv, int max_ctx_len, int num_sms);

struct DecodeLaunch {
  int mode = 0;   // 0: mixed INT2 + BF16 cache, 1: plain BF16 paged cache
  CacheRefs c;
  const uint16_t* kb_pages = nullptr;   // mode 1
  const uint16_t* vb_pages = nullptr;
  LayerRotation rot;                    // mode 0
  const uint16_t* q = nullptr;
  float* out = nullptr;
  const int32_t* ctx_len = nullptr;
  float sm_scale = 0.f;
  DecodePlan plan;
  uint8_t* workspace = nullptr;
  unsigned* err = nullptr;
  const int32_t* limit = nullptr;  // mode 0: per-request causal limit (extend attention), or none
};

cudaError_t launch_decode(const DecodeLaunch& d, cudaStream_t stream);

// fused: decode append (one token per request) + q rotation, then the decode kernel
cudaError_t launch_decode_step(const AppendLaunch& ap, const DecodeLaunch& d, cudaStream_t stream);

// extend (chunk) attention: a chunk of queries per request reading its cached pages
struct ExtendPlan {
  int32_t batch = 0, chunk = 0, Hq = 0, Hkv = 0, g = 0;
  int32_t ngpr = 0;            // query groups per request
  int32_t qpg = 0;             // queries per group: 128 / g (the group's (query, head) rows fill one MMA)
  int32_t chunk_pages = 0, n_items = 0, tiles_per_item = 0;
  int32_t prep_rows = 1;       // rows (queries) per block of the q rotation kernel
  size_t off_counters = 0, off_qfrag = 0, off_qplain = 0, off_qconst = 0, off_partials = 0, total = 0;
};
ExtendPlan plan_extend(int batch, int chunk, int Hq, int Hkv, int max_ctx_len, int num_sms);

struct ExtendLaunch {
  CacheRefs c;
  LayerRotation rot;
  const uint16_t* q = nullptr;        // bf16 [batch][chunk][Hq][128]
  float* out = nullptr;               // fp32 [batch][chunk][Hq][128]
  const int32_t* ctx_len = nullptr;   // [batch] cache lengths
  const int32_t* pos0 = nullptr;      // [batch] chunk start positions
  float sm_scale = 0.f;
  ExtendPlan plan;
  uint8_t* workspace = nullptr;
  unsigned* err = nullptr;
};
cudaError_t launch_extend(const ExtendLaunch& e, cudaStream_t stream);

// offline calibration (oscar_calib.cu)
int gram_parts(int64_t n_rows);  // fp64 partial tiles a Gram matrix of n_rows rows needs (x 128 x 128)
// C = scale X^T X (or C += ...) for X [n_rows][128] fp32; partial: gram_parts(n_rows) x 128 x 128 doubles
cudaError_t launch_gram(const float* X, int64_t n_rows, double scale, double* C, bool accumulate, double* partial,
                        cudaStream_t stream);
// O[h] = softmax(Q K[h]^T sm_scale) V[h] for every head h; Q [n_q][128], K, V [heads][n_k][128], O [heads][n_q][128]
cudaError_t launch_calib_attention(const float* Q, int64_t n_q, const float* K, const float* V, int64_t n_k,
                                   int n_heads, float sm_scale, float* O, cudaStream_t stream);
int64_t sort_size(int64_t n);  // keys the sort of n values needs (a power of two >= 2048)
// keys[0 .. n_rows 128) = |X R| ascending (as float bits), then +inf up to sort_size
cudaError_t launch_sorted_abs_rotated(const float* X, int64_t n_rows, const float* R, uint32_t* keys,
                                      cudaStream_t stream);

}  // namespace oscar
