// C ABI of the OSCAR library: argument checks, rotation constants, launches.
// See include/oscar.h for the contract of every entry point.

#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/oscar.h"
#include "oscar_device.cuh"
#include "oscar_internal.h"

using namespace oscar;

struct oscar_ctx {
  oscar_config cfg;
  int num_sms = 0;
  unsigned* d_err = nullptr;
  // per layer: R_K | R_V | R_V^T (3 * 128 * 128 floats), then the bf16
  // three-term splits of R_K^T and R_V^T (6 * 128 * 128 bf16)
  std::vector<float*> d_rot;
  std::vector<float> tau_k, tau_v;
  std::vector<uint32_t> rot_flags;
  std::vector<bool> loaded;
};

namespace {

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

bool valid_view(const oscar_ctx* ctx, const oscar_cache_view* v) {
  if (v == nullptr || v->batch < 0) return false;
  if (v->batch == 0) return true;
  // the BF16 pools move in 16-byte pieces
  for (const void* pool : {v->k_sink, v->v_sink, v->k_ring, v->v_ring})
    if ((reinterpret_cast<uintptr_t>(pool) & 15u) != 0) return false;
  return v->int2_pages && v->k_sink && v->v_sink && v->k_ring && v->v_ring && v->page_table && v->sink_page &&
         (v->ring_slot || v->recent_page_table) && v->num_pages > 0 && v->num_sink_pages > 0 && v->num_ring_slots > 0 &&
         v->max_pages_per_req > 0 && v->num_pages <= INT32_MAX && v->num_sink_pages <= INT32_MAX &&
         v->num_ring_slots <= INT32_MAX && ctx != nullptr;
}

CacheRefs refs_of(const oscar_ctx* ctx, const oscar_cache_view* v) {
  CacheRefs c;
  c.pages = static_cast<uint8_t*>(v->int2_pages);
  c.num_pages = v->num_pages;
  c.k_sink = static_cast<uint16_t*>(v->k_sink);
  c.v_sink = static_cast<uint16_t*>(v->v_sink);
  c.num_sink = v->num_sink_pages;
  c.k_ring = static_cast<uint16_t*>(v->k_ring);
  c.v_ring = static_cast<uint16_t*>(v->v_ring);
  c.num_ring = v->num_ring_slots;
  c.page_table = v->page_table;
  c.max_pages = v->max_pages_per_req;
  c.sink_page = v->sink_page;
  c.ring_slot = v->ring_slot;
  c.batch = v->batch;
  c.num_kv_heads = ctx->cfg.num_kv_heads;
  c.recent_table = v->recent_page_table;
  return c;
}

LayerRotation rotation_of(const oscar_ctx* ctx, int layer) {
  LayerRotation r;
  const float* base = ctx->d_rot[layer];
  r.R_K = base;
  r.R_V = base + 128 * 128;
  r.R_VT = base + 2 * 128 * 128;
  r.RT_split = reinterpret_cast<const uint16_t*>(base + 3 * 128 * 128);
  r.tau_k = ctx->tau_k[layer];
  r.tau_v = ctx->tau_v[layer];
  r.flags = ctx->rot_flags[layer];
  return r;
}

// Round to bf16 (nearest even) through fp32; returns the bit pattern.
uint16_t bf16_bits(double x) {
  const float f = (float)x;
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

double bf16_value(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// R = U H P in double precision (gist.science "Resumen Técnico: OSCAR ...",
// §2.2 A.3): U the calibrated basis (identity without OSCAR_ROT_U), H the
// 128-point Sylvester Hadamard matrix scaled by 1/sqrt(128), P the 7-bit
// bit-reversal permutation, so that (y P)_j = y_{rev(j)}.
void composite_rotation(const float* U, uint32_t flags, double* R) {
  const int n = 128;
  std::vector<double> M(n * n), T(n * n);
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) M[i * n + j] = (flags & OSCAR_ROT_U) ? (double)U[i * n + j] : (i == j ? 1.0 : 0.0);
  if (flags & OSCAR_ROT_H) {
    const double c = 1.0 / std::sqrt((double)n);
    for (int i = 0; i < n; ++i)
      for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int k = 0; k < n; ++k) acc += (__builtin_popcount(k & j) & 1) ? -M[i * n + k] : M[i * n + k];
        T[i * n + j] = acc * c;
      }
    M.swap(T);
  }
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) {
      int r = 0;
      for (int b = 0; b < 7; ++b) r |= ((j >> b) & 1) << (6 - b);
      R[i * n + j] = (flags & OSCAR_ROT_P) ? M[i * n + r] : M[i * n + j];
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

const char* oscar_status_string(oscar_status s) {
  switch (s) {
    case OSCAR_OK: return "ok";
    case OSCAR_ERR_INVALID_ARG: return "invalid argument";
    case OSCAR_ERR_UNSUPPORTED: return "unsupported";
    case OSCAR_ERR_NOT_LOADED: return "rotation not loaded for this layer";
    case OSCAR_ERR_CUDA: return "CUDA error";
    case OSCAR_ERR_DEVICE_CHECK: return "device-side index check failed";
    case OSCAR_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

oscar_status oscar_create(const oscar_config* cfg, oscar_ctx** out) {
  if (cfg == nullptr || out == nullptr) return OSCAR_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg->head_dim != OSCAR_HEAD_DIM || cfg->page_size != OSCAR_PAGE_TOKENS || cfg->sink != OSCAR_SINK_TOKENS ||
      cfg->recent != OSCAR_RECENT_TOKENS || cfg->group != OSCAR_GROUP)
    return OSCAR_ERR_INVALID_ARG;
  if (cfg->num_layers <= 0 || cfg->num_kv_heads <= 0 || cfg->num_q_heads <= 0 ||
      cfg->num_q_heads % cfg->num_kv_heads != 0 || cfg->num_q_heads / cfg->num_kv_heads > OSCAR_MAX_GQA ||
      cfg->num_layers > 4096 || cfg->num_kv_heads > 1024)
    return OSCAR_ERR_INVALID_ARG;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (cfg->device < 0 || cfg->device >= ndev) return OSCAR_ERR_INVALID_ARG;
  DeviceGuard guard(cfg->device);
  oscar_ctx* ctx = new (std::nothrow) oscar_ctx();
  if (ctx == nullptr) return OSCAR_ERR_CUDA;
  ctx->cfg = *cfg;
  if (cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, cfg->device) != cudaSuccess ||
      cudaMalloc(&ctx->d_err, sizeof(unsigned)) != cudaSuccess || cudaMemset(ctx->d_err, 0, sizeof(unsigned)) != cudaSuccess) {
    if (ctx->d_err) cudaFree(ctx->d_err);
    delete ctx;
    return OSCAR_ERR_CUDA;
  }
  ctx->d_rot.assign(cfg->num_layers, nullptr);
  ctx->tau_k.assign(cfg->num_layers, 0.f);
  ctx->rot_flags.assign(cfg->num_layers, OSCAR_ROT_ALL);
  ctx->tau_v.assign(cfg->num_layers, 0.f);
  ctx->loaded.assign(cfg->num_layers, false);
  *out = ctx;
  return OSCAR_OK;
}

void oscar_destroy(oscar_ctx* ctx) {
  if (ctx == nullptr) return;
  DeviceGuard guard(ctx->cfg.device);
  for (float* p : ctx->d_rot)
    if (p) cudaFree(p);
  if (ctx->d_err) cudaFree(ctx->d_err);
  delete ctx;
}

int32_t oscar_device_sm_count(const oscar_ctx* ctx) { return ctx ? ctx->num_sms : 0; }

oscar_status oscar_load_rotation(oscar_ctx* ctx, int32_t layer, const float* U_K, const float* U_V, float tau_k,
                                 float tau_v, uint32_t flags) {
  if (ctx == nullptr || U_K == nullptr || U_V == nullptr) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if ((flags & ~OSCAR_ROT_ALL) != 0) return OSCAR_ERR_INVALID_ARG;
  const float tmax = 65504.0f * 1.5f;
  if (!(tau_k > 0.f) || !(tau_v > 0.f) || std::isnan(tau_k) || std::isnan(tau_v)) return OSCAR_ERR_INVALID_ARG;
  if ((std::isfinite(tau_k) && tau_k > tmax) || (std::isfinite(tau_v) && tau_v > tmax)) return OSCAR_ERR_INVALID_ARG;
  const int n = 128 * 128;
  for (int i = 0; i < n; ++i)
    if ((flags & OSCAR_ROT_U) && (!std::isfinite(U_K[i]) || !std::isfinite(U_V[i]))) return OSCAR_ERR_INVALID_ARG;
  std::vector<double> rk(n), rv(n);
  composite_rotation(U_K, flags, rk.data());
  composite_rotation(U_V, flags, rv.data());
  std::vector<float> host(3 * n);
  for (int i = 0; i < 128; ++i)
    for (int j = 0; j < 128; ++j) {
      host[i * 128 + j] = (float)rk[i * 128 + j];
      host[n + i * 128 + j] = (float)rv[i * 128 + j];
      host[2 * n + j * 128 + i] = (float)rv[i * 128 + j];
    }
  // three bf16 terms of R^T per matrix: t0 = bf16(R), t1 = bf16(R - t0), t2 = bf16(R - t0 - t1)
  std::vector<uint16_t> split(6 * n);
  for (int m = 0; m < 2; ++m) {
    const std::vector<double>& R = m == 0 ? rk : rv;
    for (int kk = 0; kk < 128; ++kk)
      for (int nn = 0; nn < 128; ++nn) {
        double r = R[kk * 128 + nn];
        for (int t = 0; t < 3; ++t) {
          const uint16_t b = bf16_bits(r);
          split[((size_t)(m * 3 + t) * 128 + nn) * 128 + kk] = b;
          r -= bf16_value(b);
        }
      }
  }
  const size_t bytes = sizeof(float) * 3 * n + sizeof(uint16_t) * 6 * n;
  DeviceGuard guard(ctx->cfg.device);
  if (ctx->d_rot[layer] == nullptr) {
    if (cudaMalloc(&ctx->d_rot[layer], bytes) != cudaSuccess) {
      ctx->d_rot[layer] = nullptr;
      return OSCAR_ERR_CUDA;
    }
  }
  if (cudaMemcpy(ctx->d_rot[layer], host.data(), sizeof(float) * 3 * n, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(ctx->d_rot[layer] + 3 * n, split.data(), sizeof(uint16_t) * 6 * n, cudaMemcpyHostToDevice) !=
          cudaSuccess)
    return OSCAR_ERR_CUDA;
  ctx->tau_k[layer] = tau_k;
  ctx->tau_v[layer] = tau_v;
  ctx->rot_flags[layer] = flags;
  ctx->loaded[layer] = true;
  return OSCAR_OK;
}

oscar_status oscar_kv_append(oscar_ctx* ctx, int32_t layer, const oscar_cache_view* view,
                             const oscar_append_args* args, void* stream) {
  if (ctx == nullptr || view == nullptr || args == nullptr) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if (!ctx->loaded[layer]) return OSCAR_ERR_NOT_LOADED;
  if (!valid_view(ctx, view)) return OSCAR_ERR_INVALID_ARG;
  if (view->batch == 0) return OSCAR_OK;
  if (args->k == nullptr || args->v == nullptr || args->pos == nullptr || args->n_tokens < 0) return OSCAR_ERR_INVALID_ARG;
  if ((args->flags & ~OSCAR_APPEND_FRESH_RING) != 0) return OSCAR_ERR_INVALID_ARG;
  if (args->cu_seqlens == nullptr) {
    if (args->n_tokens != view->batch) return OSCAR_ERR_INVALID_ARG;
  } else if (args->max_tokens_per_req <= 0 || args->max_tokens_per_req > (1 << 28)) {
    return OSCAR_ERR_INVALID_ARG;
  }
  if (!aligned16(view->int2_pages) || !aligned16(args->k) || !aligned16(args->v)) return OSCAR_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->cfg.device);
  AppendLaunch a;
  a.c = refs_of(ctx, view);
  a.rot = rotation_of(ctx, layer);
  a.k = static_cast<const uint16_t*>(args->k);
  a.v = static_cast<const uint16_t*>(args->v);
  a.pos = args->pos;
  a.cu_seqlens = args->cu_seqlens;
  a.n_tokens = args->n_tokens;
  a.max_tokens_per_req = args->max_tokens_per_req;
  a.flags = args->flags;
  a.err = ctx->d_err;
  return launch_append(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

size_t oscar_decode_workspace_bytes(const oscar_ctx* ctx, int32_t max_batch, int32_t max_ctx_len) {
  if (ctx == nullptr || max_batch < 0 || max_ctx_len < 0) return 0;
  size_t best = 0;
  // the plan depends on the batch actually passed; take the largest over 1..max_batch
  for (int b = 1; b <= max_batch; ++b) {
    for (int mode = 0; mode < 2; ++mode) {
      const DecodePlan p = plan_decode(mode, b, ctx->cfg.num_q_heads, ctx->cfg.num_kv_heads, max_ctx_len, ctx->num_sms);
      if (p.total > best) best = p.total;
    }
  }
  return best;
}

static oscar_status check_decode_args(const oscar_ctx* ctx, const oscar_decode_args* args, int batch, void* ws,
                                      size_t ws_bytes, int mode, DecodePlan* plan) {
  if (args == nullptr || args->q == nullptr || args->out == nullptr || args->ctx_len == nullptr) return OSCAR_ERR_INVALID_ARG;
  if (args->max_ctx_len < 0 || std::isnan(args->sm_scale)) return OSCAR_ERR_INVALID_ARG;
  *plan = plan_decode(mode, batch, ctx->cfg.num_q_heads, ctx->cfg.num_kv_heads, args->max_ctx_len, ctx->num_sms);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < plan->total) return OSCAR_ERR_WORKSPACE;
  if (plan->n_items > 65535 * 16) return OSCAR_ERR_UNSUPPORTED;
  return OSCAR_OK;
}

oscar_status oscar_decode_attention(oscar_ctx* ctx, int32_t layer, const oscar_cache_view* view,
                                    const oscar_decode_args* args, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  if (ctx == nullptr || view == nullptr) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if (!ctx->loaded[layer]) return OSCAR_ERR_NOT_LOADED;
  if (!valid_view(ctx, view)) return OSCAR_ERR_INVALID_ARG;
  if (view->batch == 0) return OSCAR_OK;
  if (view->batch > 65535) return OSCAR_ERR_UNSUPPORTED;
  DecodePlan plan;
  const oscar_status st = check_decode_args(ctx, args, view->batch, workspace, workspace_bytes, 0, &plan);
  if (st != OSCAR_OK) return st;
  if (!aligned16(view->int2_pages)) return OSCAR_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->cfg.device);
  DecodeLaunch d;
  d.mode = 0;
  d.c = refs_of(ctx, view);
  d.rot = rotation_of(ctx, layer);
  d.q = static_cast<const uint16_t*>(args->q);
  d.out = args->out;
  d.ctx_len = args->ctx_len;
  d.sm_scale = args->sm_scale > 0.f ? args->sm_scale : 1.0f / std::sqrt(128.0f);
  d.plan = plan;
  d.workspace = static_cast<uint8_t*>(workspace);
  d.err = ctx->d_err;
  return launch_decode(d, static_cast<cudaStream_t>(stream)) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

oscar_status oscar_extend_attention(oscar_ctx* ctx, int32_t layer, const oscar_cache_view* view,
                                    const oscar_decode_args* args, const int32_t* limit, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  if (ctx == nullptr || view == nullptr || limit == nullptr) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if (!ctx->loaded[layer]) return OSCAR_ERR_NOT_LOADED;
  if (!valid_view(ctx, view)) return OSCAR_ERR_INVALID_ARG;
  if (view->batch == 0) return OSCAR_OK;
  if (view->batch > 65535) return OSCAR_ERR_UNSUPPORTED;
  DecodePlan plan;
  const oscar_status st = check_decode_args(ctx, args, view->batch, workspace, workspace_bytes, 0, &plan);
  if (st != OSCAR_OK) return st;
  if (!aligned16(view->int2_pages)) return OSCAR_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->cfg.device);
  DecodeLaunch d;
  d.mode = 0;
  d.c = refs_of(ctx, view);
  d.rot = rotation_of(ctx, layer);
  d.q = static_cast<const uint16_t*>(args->q);
  d.out = args->out;
  d.ctx_len = args->ctx_len;
  d.sm_scale = args->sm_scale > 0.f ? args->sm_scale : 1.0f / std::sqrt(128.0f);
  d.plan = plan;
  d.workspace = static_cast<uint8_t*>(workspace);
  d.err = ctx->d_err;
  d.limit = limit;
  return launch_decode(d, static_cast<cudaStream_t>(stream)) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

size_t oscar_extend_workspace_bytes(const oscar_ctx* ctx, int32_t batch, int32_t chunk, int32_t max_ctx_len) {
  if (ctx == nullptr || batch < 1 || chunk < 1 || max_ctx_len < 0 || (int64_t)batch * chunk > 65535) return 0;
  return plan_extend(batch, chunk, ctx->cfg.num_q_heads, ctx->cfg.num_kv_heads, max_ctx_len, ctx->num_sms).total;
}

oscar_status oscar_extend_chunk(oscar_ctx* ctx, int32_t layer, const oscar_cache_view* view, const void* q,
                                float* out, const int32_t* ctx_len, const int32_t* pos0, int32_t chunk,
                                int32_t max_ctx_len, float sm_scale, void* workspace, size_t workspace_bytes,
                                void* stream) {
  if (ctx == nullptr || view == nullptr || q == nullptr || out == nullptr || ctx_len == nullptr || pos0 == nullptr)
    return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if (!ctx->loaded[layer]) return OSCAR_ERR_NOT_LOADED;
  if (!valid_view(ctx, view)) return OSCAR_ERR_INVALID_ARG;
  if (chunk < 1 || max_ctx_len < 0) return OSCAR_ERR_INVALID_ARG;
  if (view->batch == 0) return OSCAR_OK;
  if ((int64_t)view->batch * chunk > 65535) return OSCAR_ERR_UNSUPPORTED;
  if (ctx->cfg.num_q_heads / ctx->cfg.num_kv_heads > 4) return OSCAR_ERR_UNSUPPORTED;
  if (!aligned16(view->int2_pages)) return OSCAR_ERR_INVALID_ARG;
  const ExtendPlan plan = plan_extend(view->batch, chunk, ctx->cfg.num_q_heads, ctx->cfg.num_kv_heads, max_ctx_len,
                                      ctx->num_sms);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < plan.total)
    return OSCAR_ERR_WORKSPACE;
  DeviceGuard guard(ctx->cfg.device);
  ExtendLaunch e;
  e.c = refs_of(ctx, view);
  e.rot = rotation_of(ctx, layer);
  e.q = static_cast<const uint16_t*>(q);
  e.out = out;
  e.ctx_len = ctx_len;
  e.pos0 = pos0;
  e.sm_scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(128.0f);
  e.plan = plan;
  e.workspace = static_cast<uint8_t*>(workspace);
  e.err = ctx->d_err;
  return launch_extend(e, static_cast<cudaStream_t>(stream)) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

oscar_status oscar_decode_step(oscar_ctx* ctx, int32_t layer, const oscar_cache_view* view,
                               const oscar_append_args* append, const oscar_decode_args* decode, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (ctx == nullptr || view == nullptr || append == nullptr) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if (!ctx->loaded[layer]) return OSCAR_ERR_NOT_LOADED;
  if (!valid_view(ctx, view)) return OSCAR_ERR_INVALID_ARG;
  if (view->batch == 0) return OSCAR_OK;
  if (view->batch > 65535) return OSCAR_ERR_UNSUPPORTED;
  if (append->k == nullptr || append->v == nullptr || append->pos == nullptr) return OSCAR_ERR_INVALID_ARG;
  if (append->cu_seqlens != nullptr || append->n_tokens != view->batch) return OSCAR_ERR_INVALID_ARG;
  if ((append->flags & ~OSCAR_APPEND_FRESH_RING) != 0) return OSCAR_ERR_INVALID_ARG;
  DecodePlan plan;
  const oscar_status st = check_decode_args(ctx, decode, view->batch, workspace, workspace_bytes, 0, &plan);
  if (st != OSCAR_OK) return st;
  if (!aligned16(view->int2_pages)) return OSCAR_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->cfg.device);
  AppendLaunch a;
  a.c = refs_of(ctx, view);
  a.rot = rotation_of(ctx, layer);
  a.k = static_cast<const uint16_t*>(append->k);
  a.v = static_cast<const uint16_t*>(append->v);
  a.pos = append->pos;
  a.cu_seqlens = nullptr;
  a.n_tokens = append->n_tokens;
  a.max_tokens_per_req = 1;
  a.flags = append->flags;
  a.err = ctx->d_err;
  DecodeLaunch d;
  d.mode = 0;
  d.c = a.c;
  d.rot = a.rot;
  d.q = static_cast<const uint16_t*>(decode->q);
  d.out = decode->out;
  d.ctx_len = decode->ctx_len;
  d.sm_scale = decode->sm_scale > 0.f ? decode->sm_scale : 1.0f / std::sqrt(128.0f);
  d.plan = plan;
  d.workspace = static_cast<uint8_t*>(workspace);
  d.err = ctx->d_err;
  return launch_decode_step(a, d, static_cast<cudaStream_t>(stream)) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

oscar_status oscar_decode_attention_bf16(oscar_ctx* ctx, const oscar_bf16_cache_view* view,
                                         const oscar_decode_args* args, void* workspace, size_t workspace_bytes,
                                         void* stream) {
  if (ctx == nullptr || view == nullptr || view->batch < 0) return OSCAR_ERR_INVALID_ARG;
  if (view->batch == 0) return OSCAR_OK;
  if (view->batch > 65535) return OSCAR_ERR_UNSUPPORTED;
  if (view->k_pages == nullptr || view->v_pages == nullptr || view->page_table == nullptr || view->num_pages <= 0 ||
      view->num_pages > INT32_MAX || view->max_pages_per_req <= 0)
    return OSCAR_ERR_INVALID_ARG;
  DecodePlan plan;
  const oscar_status st = check_decode_args(ctx, args, view->batch, workspace, workspace_bytes, 1, &plan);
  if (st != OSCAR_OK) return st;
  DeviceGuard guard(ctx->cfg.device);
  DecodeLaunch d;
  d.mode = 1;
  d.c.page_table = view->page_table;
  d.c.max_pages = view->max_pages_per_req;
  d.c.num_pages = view->num_pages;
  d.c.batch = view->batch;
  d.c.num_kv_heads = ctx->cfg.num_kv_heads;
  d.kb_pages = static_cast<const uint16_t*>(view->k_pages);
  d.vb_pages = static_cast<const uint16_t*>(view->v_pages);
  d.q = static_cast<const uint16_t*>(args->q);
  d.out = args->out;
  d.ctx_len = args->ctx_len;
  d.sm_scale = args->sm_scale > 0.f ? args->sm_scale : 1.0f / std::sqrt(128.0f);
  d.plan = plan;
  d.workspace = static_cast<uint8_t*>(workspace);
  d.err = ctx->d_err;
  // the prep kernel needs a rotation matrix; the plain path only uses the unrotated q
  for (size_t l = 0; l < ctx->d_rot.size(); ++l)
    if (ctx->loaded[l]) {
      d.rot = rotation_of(ctx, (int)l);
      break;
    }
  if (d.rot.R_K == nullptr) return OSCAR_ERR_NOT_LOADED;
  return launch_decode(d, static_cast<cudaStream_t>(stream)) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

// ---------------------------------------------------------------- offline calibration
namespace {

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

size_t calib_cov_bytes(int64_t n_q, int64_t n_k, int32_t heads) {
  (void)n_k;
  const int64_t rows = n_q * heads;
  const int parts = oscar::gram_parts(rows > n_q ? rows : n_q);
  return align_up((size_t)parts * 128 * 128 * sizeof(double)) + align_up((size_t)rows * 128 * sizeof(float));
}

size_t calib_clip_bytes(int64_t n_rows) {
  return align_up(128 * 128 * sizeof(float)) + align_up((size_t)oscar::sort_size(n_rows * 128) * sizeof(uint32_t));
}

}  // namespace

size_t oscar_calib_workspace_bytes(int64_t n_queries, int64_t n_keys, int32_t n_kv_heads, int64_t n_clip_rows) {
  if (n_queries < 1 || n_keys < 1 || n_kv_heads < 1 || n_clip_rows < 1 || n_clip_rows > OSCAR_CALIB_MAX_ROWS ||
      n_queries > OSCAR_CALIB_MAX_ROWS || n_keys > OSCAR_CALIB_MAX_ROWS || n_kv_heads > 256)
    return 0;
  const size_t a = calib_cov_bytes(n_queries, n_keys, n_kv_heads), b = calib_clip_bytes(n_clip_rows);
  return a > b ? a : b;
}

oscar_status oscar_calib_covariances(oscar_ctx* ctx, const float* q, int64_t n_q, const float* k, const float* v,
                                     int64_t n_k, int32_t n_kv_heads, float sm_scale, double* c_q, double* c_s,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  if (ctx == nullptr || q == nullptr || k == nullptr || v == nullptr || c_q == nullptr || c_s == nullptr)
    return OSCAR_ERR_INVALID_ARG;
  if (n_q < 1 || n_k < 1 || n_kv_heads < 1 || n_q > OSCAR_CALIB_MAX_ROWS || n_k > OSCAR_CALIB_MAX_ROWS ||
      n_kv_heads > 256 || !(sm_scale > 0.f) || !std::isfinite(sm_scale))
    return OSCAR_ERR_INVALID_ARG;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < calib_cov_bytes(n_q, n_k, n_kv_heads))
    return OSCAR_ERR_WORKSPACE;
  DeviceGuard guard(ctx->cfg.device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int64_t rows = n_q * n_kv_heads;
  double* partial = reinterpret_cast<double*>(ws);
  float* O = reinterpret_cast<float*>(
      ws + align_up((size_t)oscar::gram_parts(rows > n_q ? rows : n_q) * 128 * 128 * sizeof(double)));
  if (oscar::launch_gram(q, n_q, 1.0 / (double)n_q, c_q, false, partial, st) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (oscar::launch_calib_attention(q, n_q, k, v, n_k, n_kv_heads, sm_scale, O, st) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  // C_S = (1 / heads) sum_h (1 / N) O_h^T O_h = (1 / (N heads)) over the rows of every O_h
  if (oscar::launch_gram(O, rows, 1.0 / (double)rows, c_s, false, partial, st) != cudaSuccess) return OSCAR_ERR_CUDA;
  return OSCAR_OK;
}

oscar_status oscar_calib_clip_threshold(oscar_ctx* ctx, const float* x, int64_t n_rows, const float* U,
                                        uint32_t flags, double percentile, double* tau, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (ctx == nullptr || x == nullptr || U == nullptr || tau == nullptr) return OSCAR_ERR_INVALID_ARG;
  if (n_rows < 1 || n_rows > OSCAR_CALIB_MAX_ROWS || (flags & ~OSCAR_ROT_ALL) != 0) return OSCAR_ERR_INVALID_ARG;
  if (!(percentile >= 0.0 && percentile <= 100.0)) return OSCAR_ERR_INVALID_ARG;
  for (int i = 0; i < 128 * 128; ++i)
    if ((flags & OSCAR_ROT_U) && !std::isfinite(U[i])) return OSCAR_ERR_INVALID_ARG;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < calib_clip_bytes(n_rows))
    return OSCAR_ERR_WORKSPACE;
  DeviceGuard guard(ctx->cfg.device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the composite R = U H P, formed in fp64 exactly as for oscar_load_rotation
  std::vector<double> r(128 * 128);
  composite_rotation(U, flags, r.data());
  std::vector<float> rf(128 * 128);
  for (int i = 0; i < 128 * 128; ++i) rf[i] = (float)r[i];
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* R = reinterpret_cast<float*>(ws);
  uint32_t* keys = reinterpret_cast<uint32_t*>(ws + align_up(128 * 128 * sizeof(float)));
  if (cudaMemcpyAsync(R, rf.data(), rf.size() * sizeof(float), cudaMemcpyHostToDevice, st) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  if (oscar::launch_sorted_abs_rotated(x, n_rows, R, keys, st) != cudaSuccess) return OSCAR_ERR_CUDA;
  // numpy's linear interpolation between the order statistics around p (n - 1)
  const int64_t n = n_rows * 128;
  const double pos = percentile / 100.0 * (double)(n - 1);
  int64_t lo = (int64_t)std::floor(pos);
  if (lo > n - 1) lo = n - 1;
  const int64_t hi = lo + 1 < n ? lo + 1 : lo;
  uint32_t pair[2];
  if (cudaMemcpyAsync(&pair[0], keys + lo, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(&pair[1], keys + hi, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  float a, b;
  std::memcpy(&a, &pair[0], 4);
  std::memcpy(&b, &pair[1], 4);
  const double g = pos - (double)lo;
  *tau = (double)a + g * ((double)b - (double)a);
  return OSCAR_OK;
}

oscar_status oscar_check_device_error(oscar_ctx* ctx, void* stream, uint32_t* bits) {
  if (ctx == nullptr) return OSCAR_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->cfg.device);
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return OSCAR_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, ctx->d_err, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (v != 0 && cudaMemset(ctx->d_err, 0, sizeof(unsigned)) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (bits) *bits = v;
  return v ? OSCAR_ERR_DEVICE_CHECK : OSCAR_OK;
}

oscar_status oscar_selftest_bounded_wait(oscar_ctx* ctx, uint32_t polls, void* stream) {
  if (ctx == nullptr || polls == 0 || polls > (1u << 18)) return OSCAR_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->cfg.device);
  return oscar::launch_selftest_wait(ctx->d_err, polls, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? OSCAR_OK
             : OSCAR_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decode: the same launch as oscar_decode_attention, with its
// workspace in a file-scope device array instead of caller memory.  Every GPU
// that loads this library holds the array until the process exits.  Its
// device address is looked up once per device, on the first call made with
// that device current, and cached.

static __device__ __align__(256) uint8_t g_decode_scratch[OSCAR_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxScratchDevices] = {};

// Device address of g_decode_scratch on `device` (which must be current).
cudaError_t scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxScratchDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[device] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return cudaSuccess;
}
}  // namespace

extern "C" oscar_status oscar_decode_attention_noalloc(oscar_ctx* ctx, int32_t layer, const oscar_cache_view* view,
                                                       const oscar_decode_args* args, void* stream) {
  if (ctx == nullptr || view == nullptr) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if (!ctx->loaded[layer]) return OSCAR_ERR_NOT_LOADED;
  if (!valid_view(ctx, view)) return OSCAR_ERR_INVALID_ARG;
  if (view->batch == 0) return OSCAR_OK;
  if (view->batch > 65535) return OSCAR_ERR_UNSUPPORTED;
  if (!aligned16(view->int2_pages)) return OSCAR_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->cfg.device);
  void* scratch = nullptr;
  if (scratch_address(ctx->cfg.device, &scratch) != cudaSuccess) return OSCAR_ERR_CUDA;
  DecodePlan plan;
  const oscar_status st =
      check_decode_args(ctx, args, view->batch, scratch, OSCAR_NOALLOC_SCRATCH_BYTES, 0, &plan);
  if (st != OSCAR_OK) return st;  // OSCAR_ERR_WORKSPACE when the call needs more than the array holds
  // the documented limit: what oscar_decode_workspace_bytes asks of a caller for this batch and length
  // (never below the launch's own plan), so that callers can size their calls by that function
  if (oscar_decode_workspace_bytes(ctx, view->batch, args->max_ctx_len) > OSCAR_NOALLOC_SCRATCH_BYTES)
    return OSCAR_ERR_WORKSPACE;
  DecodeLaunch d;
  d.mode = 0;
  d.c = refs_of(ctx, view);
  d.rot = rotation_of(ctx, layer);
  d.q = static_cast<const uint16_t*>(args->q);
  d.out = args->out;
  d.ctx_len = args->ctx_len;
  d.sm_scale = args->sm_scale > 0.f ? args->sm_scale : 1.0f / std::sqrt(128.0f);
  d.plan = plan;
  d.workspace = static_cast<uint8_t*>(scratch);
  d.err = ctx->d_err;
  return launch_decode(d, static_cast<cudaStream_t>(stream)) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}
