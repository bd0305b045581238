// OSCAR KV-cache write path: rotate, clip, quantise, pack; BF16 sink/ring
// writes; recent-window eviction.
//
// ainsights.it "OSCAR: Come Together AI Comprime la KV Cache a 2-bit per LLM",
// section "Architettura del Sistema di Serving e Layout di Memoria": during
// the write every token is rotated, clipped and quantised; the first 64 tokens
// and the last 256 stay BF16.  gist.science "Resumen Técnico: OSCAR ...",
// §2.2 A.3-4 (R = U H_Had P_br, per-layer clip thresholds) and §2.2 B (paged
// cache, sink/recent in BF16, INT2 history after rotation and clipping).
//
// Rotation x' = x R is computed as (x U) in fp32, then the Walsh-Hadamard
// factor as a butterfly (shuffles within a warp, shared memory across warps),
// then the bit-reversal permutation as an index map.  Quantiser per group of
// 64 rotated channels: a = min(max|x'|, tau), s = fp16(a / 1.5),
// code = [x' >= -s] + [x' >= 0] + [x' >= s].

#include "oscar_device.cuh"
#include "oscar_internal.h"
#include "oscar_quant.cuh"

namespace oscar {
namespace {

// ------------------------------------------------------------------ decode append
// One new token per request.  grid (Hkv, B), 256 threads: threads 0..127
// handle K, threads 128..255 handle V, each a channel per thread.
__global__ void __launch_bounds__(256, 1) append_one_kernel(AppendLaunch a) {
  __shared__ QuantSmem sm[2];
  griddep_wait();
  const int half = threadIdx.x >> 7;
  append_one_body(a, blockIdx.y, blockIdx.x, half, threadIdx.x & 127, a.rot.R_K, a.rot.R_V, sm[half]);
}

// ------------------------------------------------------------------ multi-token append
__device__ __forceinline__ bool request_span(const AppendLaunch& a, int b, int& p0, int& n, int& tok0) {
  if (a.cu_seqlens == nullptr) {
    tok0 = b;
    n = 1;
  } else {
    tok0 = a.cu_seqlens[b];
    n = a.cu_seqlens[b + 1] - tok0;
    if (n < 0 || tok0 < 0 || tok0 + n > a.n_tokens || n > a.max_tokens_per_req) {
      if (threadIdx.x == 0) set_error(a.err, kErrTokens);
      return false;
    }
  }
  p0 = a.pos[b];
  if (p0 < 0) {
    if (threadIdx.x == 0) set_error(a.err, kErrLength);
    return false;
  }
  // a fresh ring holds only the new tokens: the recent window must lie inside them
  if ((a.flags & 1u) && p0 > kSink && n < kRecent) {
    if (threadIdx.x == 0) set_error(a.err, kErrLength);
    return false;
  }
  return n > 0;
}

// Phase 1: ring tokens that fall out of the recent window go to the history.
// grid (256, Hkv, B), 128 threads: one token-head per block.
__global__ void __launch_bounds__(256, 1) append_evict_kernel(AppendLaunch a) {
  __shared__ QuantSmem sm[2];
  const int x = blockIdx.x, h = blockIdx.y, b = blockIdx.z, half = threadIdx.x >> 7, t = threadIdx.x & 127;
  const bool is_v = half == 1;
  int p0, n, tok0;
  if (!request_span(a, b, p0, n, tok0)) return;
  const int L = p0 + n;
  const int e0 = max(kSink, p0 - kRecent), e1 = min(p0, L - kRecent);
  const int e = e0 + x;
  if (e >= e1) return;
  const CacheRefs& c = a.c;
  const int slot = c.ring_slot[b];
  if (slot < 0 || slot >= c.num_ring) {
    if (threadIdx.x == 0) set_error(a.err, kErrRing);
    return;
  }
  uint8_t* blk = history_block(c, b, h, e, a.err);
  if (blk == nullptr) return;
  const size_t r = (((size_t)slot * c.num_kv_heads + h) * kRecent + ((e - kSink) % kRecent)) * kD + t;
  const float xv = bf16_bits_to_float((is_v ? c.v_ring : c.k_ring)[r]);
  quantize_token(xv, is_v ? a.rot.R_V : a.rot.R_K, is_v ? a.rot.tau_v : a.rot.tau_k, blk, e & 63, is_v, sm[half]);
}

// Phase 2a: new tokens that stay BF16 (sink rows, ring rows).
// grid (320, B), 128 threads; all KV heads of one position per block.
__global__ void __launch_bounds__(128) append_bf16_kernel(AppendLaunch a) {
  const int x = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  int p0, n, tok0;
  if (!request_span(a, b, p0, n, tok0)) return;
  const int L = p0 + n;
  const CacheRefs& c = a.c;
  const int Hkv = c.num_kv_heads;
  int p;
  uint16_t *kd, *vd;
  size_t row0;
  if (x < kSink) {
    p = p0 + x;
    if (p >= min(L, kSink)) return;
    const int sp = c.sink_page[b];
    if (sp < 0 || sp >= c.num_sink) {
      if (t == 0) set_error(a.err, kErrSink);
      return;
    }
    kd = c.k_sink;
    vd = c.v_sink;
    row0 = (size_t)sp * Hkv * kSink;  // + h * 64 + p
    for (int h = 0; h < Hkv; ++h) {
      const size_t s = ((size_t)(tok0 + p - p0) * Hkv + h) * kD + t;
      const size_t d = (row0 + (size_t)h * kSink + p) * kD + t;
      kd[d] = a.k[s];
      vd[d] = a.v[s];
    }
    return;
  }
  p = max(max(p0, L - kRecent), kSink) + (x - kSink);
  if (p >= L) return;
  const int slot = c.ring_slot[b];
  if (slot < 0 || slot >= c.num_ring) {
    if (t == 0) set_error(a.err, kErrRing);
    return;
  }
  kd = c.k_ring;
  vd = c.v_ring;
  for (int h = 0; h < Hkv; ++h) {
    const size_t s = ((size_t)(tok0 + p - p0) * Hkv + h) * kD + t;
    const size_t d = (((size_t)slot * Hkv + h) * kRecent + ((p - kSink) % kRecent)) * kD + t;
    kd[d] = a.k[s];
    vd[d] = a.v[s];
  }
}

// Phase 2b: new tokens that go straight into the INT2 history, one page of
// one KV head per block.  grid (pages, Hkv, B), 256 threads: threads 0..127
// quantise the K rows, 128..255 the V rows, concurrently (named barriers
// 1 and 2).  x R runs on the CUDA cores in fp32 (summed in channel order):
// warp q of a half owns rows 16 q .. 16 q + 15, lane owns channels
// 4 lane .. 4 lane + 3.
struct TileSmem {
  __align__(16) float z[2][64][kD + 4];  // K and V rows (fp32)
  uint8_t code[2][64][kD];
  __half scale[2][64][2];
};

__device__ __forceinline__ void quantize_tile_half(const AppendLaunch& a, int b, int h, int tok0, int p0, int r_lo,
                                                   int r_hi, int lp, uint8_t* blk, int half, TileSmem& sm) {
  const bool is_v = half == 1;
  const int t = threadIdx.x & 127, lane = t & 31, wq = t >> 5, bar = 1 + half;
  const int Hkv = a.c.num_kv_heads;
  const uint16_t* src = is_v ? a.v : a.k;
  const float* __restrict__ R = is_v ? a.rot.R_V : a.rot.R_K;
  const float tau = is_v ? a.rot.tau_v : a.rot.tau_k;
  float(*z)[kD + 4] = sm.z[half];
  // load the tile, 8 channels per load (rows outside [r_lo, r_hi) are zero)
  for (int i = t; i < 64 * (kD / 8); i += 128) {
    const int r = i >> 4, c8 = (i & 15) * 8;
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (r >= r_lo && r < r_hi) {
      const int p = lp * kPage + r;
      u = *reinterpret_cast<const uint4*>(src + ((size_t)(tok0 + p - p0) * Hkv + h) * kD + c8);
    }
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      z[r][c8 + 2 * k] = __uint_as_float(w[k] << 16);
      z[r][c8 + 2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
  half_sync(bar);
  float acc[16][4];
#pragma unroll
  for (int r = 0; r < 16; ++r)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[r][k] = 0.f;
#pragma unroll 2
  for (int i = 0; i < kD; i += 4) {
    const float4 r0 = __ldg(reinterpret_cast<const float4*>(R + (size_t)(i + 0) * kD) + lane);
    const float4 r1 = __ldg(reinterpret_cast<const float4*>(R + (size_t)(i + 1) * kD) + lane);
    const float4 r2 = __ldg(reinterpret_cast<const float4*>(R + (size_t)(i + 2) * kD) + lane);
    const float4 r3 = __ldg(reinterpret_cast<const float4*>(R + (size_t)(i + 3) * kD) + lane);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float4 x = *reinterpret_cast<const float4*>(&z[16 * wq + r][i]);
      acc[r][0] = fmaf(x.w, r3.x, fmaf(x.z, r2.x, fmaf(x.y, r1.x, fmaf(x.x, r0.x, acc[r][0]))));
      acc[r][1] = fmaf(x.w, r3.y, fmaf(x.z, r2.y, fmaf(x.y, r1.y, fmaf(x.x, r0.y, acc[r][1]))));
      acc[r][2] = fmaf(x.w, r3.z, fmaf(x.z, r2.z, fmaf(x.y, r1.z, fmaf(x.x, r0.z, acc[r][2]))));
      acc[r][3] = fmaf(x.w, r3.w, fmaf(x.z, r2.w, fmaf(x.y, r1.w, fmaf(x.x, r0.w, acc[r][3]))));
    }
  }
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int row = 16 * wq + r;
    const float v[4] = {acc[r][0], acc[r][1], acc[r][2], acc[r][3]};
    // group absmax: channels 0..63 on lanes 0..15, 64..127 on lanes 16..31
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float aa = fminf(m, tau);
    const __half sh = __float2half_rn(aa / 1.5f);
    const float sc = __half2float(sh);
    uint32_t packed = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      packed |= (uint32_t)((v[k] >= -sc) + (v[k] >= 0.f) + (v[k] >= sc)) << (8 * k);
    *reinterpret_cast<uint32_t*>(&sm.code[half][row][4 * lane]) = packed;
    if ((lane & 15) == 0) sm.scale[half][row][lane >> 4] = sh;
  }
  half_sync(bar);
  // pack the rows in [r_lo, r_hi) only: other rows of this page may hold
  // history tokens written by earlier appends
  for (int i = t; i < 64 * 8; i += 128) {
    const int row = i >> 3, w = i & 7;
    if (row < r_lo || row >= r_hi) continue;
    if (!is_v) {
      const int tig = w & 3, g = w >> 2, base = 64 * g + 16 * tig;
      uint32_t word = 0;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        word |= (uint32_t)sm.code[0][row][base + r] << (2 * r);
        word |= (uint32_t)sm.code[0][row][base + 8 + r] << (16 + 2 * r);
      }
      *reinterpret_cast<uint32_t*>(blk + kKCodes + k_word_offset(row, tig, g)) = word;
    } else {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int jj = 2 * w + hh;
        uint32_t hv = 0;
#pragma unroll
        for (int r = 0; r < 8; ++r) hv |= (uint32_t)sm.code[1][row][jj + 16 * r] << (2 * r);
        *reinterpret_cast<uint16_t*>(blk + kVCodes + v_half_offset(row, jj)) = (uint16_t)hv;
      }
    }
  }
  for (int i = t; i < 64 * 2; i += 128) {
    const int row = i >> 1, g = i & 1;
    if (row < r_lo || row >= r_hi) continue;
    *reinterpret_cast<__half*>(blk + (is_v ? kVScales : kKScales) + 4 * row + 2 * g) = sm.scale[half][row][g];
  }
}

__global__ void __launch_bounds__(256, 2) append_tile_kernel(AppendLaunch a) {
  extern __shared__ __align__(16) uint8_t tile_smem_raw[];
  TileSmem& sm = *reinterpret_cast<TileSmem*>(tile_smem_raw);
  const int x = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  int p0, n, tok0;
  if (!request_span(a, b, p0, n, tok0)) return;
  const int L = p0 + n;
  const int lo = max(p0, kSink), hi = L - kRecent;
  if (hi <= lo) return;
  const int lp = lo / kPage + x;
  if (lp * kPage >= hi) return;
  const int r_lo = max(lo - lp * kPage, 0), r_hi = min(hi - lp * kPage, kPage);
  uint8_t* blk = history_block(a.c, b, h, lp * kPage, a.err);
  if (blk == nullptr) return;
  quantize_tile_half(a, b, h, tok0, p0, r_lo, r_hi, lp, blk, threadIdx.x >> 7, sm);
}

}  // namespace

cudaError_t launch_append(const AppendLaunch& a, cudaStream_t stream) {
  const int B = a.c.batch, Hkv = a.c.num_kv_heads;
  if (a.cu_seqlens == nullptr) {
    append_one_kernel<<<dim3(Hkv, B), 256, 0, stream>>>(a);
    return cudaGetLastError();
  }
  if (!(a.flags & 1u)) append_evict_kernel<<<dim3(kRecent, Hkv, B), 256, 0, stream>>>(a);
  append_bf16_kernel<<<dim3(kSink + kRecent, B), 128, 0, stream>>>(a);
  const int tiles = (a.max_tokens_per_req + kPage - 1) / kPage + 1;
  const size_t smem = sizeof(TileSmem);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(append_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  append_tile_kernel<<<dim3(tiles, Hkv, B), 256, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace oscar
