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

#include <algorithm>

#include "oscar_device.cuh"
#include "oscar_internal.h"
#include "oscar_quant.cuh"

namespace oscar {
namespace {

// ------------------------------------------------------------------ decode append
// One new token per request.  grid (Hkv, B), 2 kQuantThreads threads: the
// first kQuantThreads handle K, the others V.
__global__ void __launch_bounds__(2 * kQuantThreads, 1) append_one_kernel(AppendLaunch a) {
  __shared__ QuantSmem sm[2];
  griddep_wait();
  const int half = threadIdx.x / kQuantThreads;
  append_one_body(a, blockIdx.y, blockIdx.x, half, threadIdx.x % kQuantThreads, a.rot.R_K, a.rot.R_V, sm[half],
                  1 + half);
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
// grid (256, Hkv, B), 2 kQuantThreads threads: one token-head per block, K
// by the first kQuantThreads threads, V by the others.
__global__ void __launch_bounds__(2 * kQuantThreads, 1) append_evict_kernel(AppendLaunch a) {
  __shared__ QuantSmem sm[2];
  const int x = blockIdx.x, h = blockIdx.y, b = blockIdx.z, half = threadIdx.x / kQuantThreads;
  const int u = threadIdx.x % kQuantThreads, t = u & 127;
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
  quantize_token(xv, is_v ? a.rot.R_V : a.rot.R_K, is_v ? a.rot.tau_v : a.rot.tau_k, blk, e & 63, is_v, sm[half], u,
                 1 + half);
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

// Phase 2b: new tokens that go straight into the INT2 history.
//
// x R on the tensor cores: x is a bf16 row, R^T is held as three bf16 terms
// (R = t0 + t1 + t2 to ~2^-24 relative), and each m16n8k16 product is exact
// in the MMA.  The t0 products of each 16-channel step land in a fresh
// accumulator and are summed in fp32 with round-to-nearest, so the tensor
// core's truncation of its fp32 result does not pile up; the much smaller t1,
// t2 products share one chained accumulator.  Persistent blocks of 512
// threads, one per SM, keep the six R^T terms (192 KB) in shared memory and
// run two tile slots: warps 0..7 and 8..15 each take one (request, KV head,
// page) tile at a time, K rows on their first four warps and V rows on the
// last four; each warp owns 16 rows of the tile.
constexpr int kTcSlots = 2;
constexpr int kTcThreads = 32 * 8 * kTcSlots;

struct TcSmem {
  uint16_t rt[2][3][kD][kD];          // [K, V][term][n][k], 16-byte chunks swizzled by n % 8
  uint8_t code[kTcSlots][2][64][kD];  // codes of the tile being packed
  __half scale[kTcSlots][2][64][2];
};

__device__ __forceinline__ int rt_index(int n, int k) { return n * kD + ((((k >> 3) ^ (n & 7)) << 3) | (k & 7)); }

// One (request, KV head, page) tile, rows [r_lo, r_hi) of page lp, for the
// 128 threads of (slot, matrix m) -- m = 0: K, 1: V -- synchronised by named
// barrier `bar`.
__device__ __forceinline__ void tc_quantize_tile(const AppendLaunch& a, int b, int h, int tok0, int p0, int r_lo,
                                                 int r_hi, int lp, uint8_t* blk, int slot, int m, int bar,
                                                 TcSmem& sm) {
  const int t = threadIdx.x & 127, lane = t & 31, wq = t >> 5, g = lane >> 2, tq = lane & 3;
  const int Hkv = a.c.num_kv_heads;
  const uint16_t* src = m ? a.v : a.k;
  const float tau = m ? a.rot.tau_v : a.rot.tau_k;
  // A fragments of this warp's rows 16 wq + {g, g + 8}, all 8 channel steps
  uint32_t af[8][4];
  {
    const int r0 = 16 * wq + g, r1 = r0 + 8;
    const bool v0 = r0 >= r_lo && r0 < r_hi, v1 = r1 >= r_lo && r1 < r_hi;
    const uint16_t* x0 = src + ((size_t)(tok0 + lp * kPage + r0 - p0) * Hkv + h) * kD + 2 * tq;
    const uint16_t* x1 = src + ((size_t)(tok0 + lp * kPage + r1 - p0) * Hkv + h) * kD + 2 * tq;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      af[i][0] = v0 ? *reinterpret_cast<const uint32_t*>(x0 + 16 * i) : 0u;
      af[i][1] = v1 ? *reinterpret_cast<const uint32_t*>(x1 + 16 * i) : 0u;
      af[i][2] = v0 ? *reinterpret_cast<const uint32_t*>(x0 + 16 * i + 8) : 0u;
      af[i][3] = v1 ? *reinterpret_cast<const uint32_t*>(x1 + 16 * i + 8) : 0u;
    }
  }
  const uint16_t* rtm = &sm.rt[m][0][0][0];
  // ldmatrix row of this lane: matrix q = lane / 8 covers n-block (pair base + q / 2), k half q % 2
  const int lq = lane >> 3, lr = lane & 7;
#pragma unroll 1
  for (int G = 0; G < 2; ++G) {  // quantisation group: output channels 64 G .. 64 G + 63
    float run[8][4], chn[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) run[j][e] = chn[j][e] = 0.f;
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        const int n = 64 * G + 16 * jp + 8 * (lq >> 1) + lr, k = 16 * i + 8 * (lq & 1);
        const int off = rt_index(n, k);
        uint32_t b[4];
        ldmatrix_x4(b[0], b[1], b[2], b[3], rtm + off);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float f[4];
          mma_bf16(f, af[i], b[2 * q], b[2 * q + 1], zero);
#pragma unroll
          for (int e = 0; e < 4; ++e) run[2 * jp + q][e] += f[e];
        }
#pragma unroll
        for (int term = 1; term < 3; ++term) {
          ldmatrix_x4(b[0], b[1], b[2], b[3], rtm + term * kD * kD + off);
#pragma unroll
          for (int q = 0; q < 2; ++q) mma_bf16(chn[2 * jp + q], af[i], b[2 * q], b[2 * q + 1], chn[2 * jp + q]);
        }
      }
    }
    // x' of rows 16 wq + g (elements 0, 1) and + 8 (2, 3), channels 64 G + 8 j + 2 tq + {0, 1}
    float mx0 = 0.f, mx1 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) run[j][e] += chn[j][e];
      mx0 = fmaxf(mx0, fmaxf(fabsf(run[j][0]), fabsf(run[j][1])));
      mx1 = fmaxf(mx1, fmaxf(fabsf(run[j][2]), fabsf(run[j][3])));
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const __half h0 = __float2half_rn(fminf(mx0, tau) / 1.5f), h1 = __float2half_rn(fminf(mx1, tau) / 1.5f);
    const float s0 = __half2float(h0), s1 = __half2float(h1);
    const int row0 = 16 * wq + g, row1 = row0 + 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int ch = 64 * G + 8 * j + 2 * tq;
      const float* v = run[j];
      sm.code[slot][m][row0][ch] = (uint8_t)((v[0] >= -s0) + (v[0] >= 0.f) + (v[0] >= s0));
      sm.code[slot][m][row0][ch + 1] = (uint8_t)((v[1] >= -s0) + (v[1] >= 0.f) + (v[1] >= s0));
      sm.code[slot][m][row1][ch] = (uint8_t)((v[2] >= -s1) + (v[2] >= 0.f) + (v[2] >= s1));
      sm.code[slot][m][row1][ch + 1] = (uint8_t)((v[3] >= -s1) + (v[3] >= 0.f) + (v[3] >= s1));
    }
    if (tq == 0) {
      sm.scale[slot][m][row0][G] = h0;
      sm.scale[slot][m][row1][G] = h1;
    }
  }
  half_sync(bar);
  // pack the rows in [r_lo, r_hi) only: other rows of this page may hold
  // history tokens written by earlier appends
  for (int i = t; i < 64 * 8; i += 128) {
    const int row = i >> 3, w = i & 7;
    if (row < r_lo || row >= r_hi) continue;
    const uint8_t* cr = sm.code[slot][m][row];
    if (m == 0) {
      *reinterpret_cast<uint32_t*>(blk + kKCodes + k_word_offset(row, w & 3, w >> 2)) = k_word(cr, w & 3, w >> 2);
    } else {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int jj = 2 * w + hh;
        uint32_t hv = 0;
#pragma unroll
        for (int r = 0; r < 8; ++r) hv |= (uint32_t)cr[jj + 16 * r] << (2 * r);
        *reinterpret_cast<uint16_t*>(blk + kVCodes + v_half_offset(row, jj)) = (uint16_t)hv;
      }
    }
  }
  {
    const int row = t >> 1, gg = t & 1;
    if (row >= r_lo && row < r_hi)
      *reinterpret_cast<__half*>(blk + (m ? kVScales : kKScales) + 4 * row + 2 * gg) = sm.scale[slot][m][row][gg];
  }
  half_sync(bar);  // the staging is reused by this slot's next tile
}

__global__ void __launch_bounds__(kTcThreads, 1) append_tile_kernel(AppendLaunch a, int tiles_per_req) {
  extern __shared__ __align__(16) uint8_t tile_smem_raw[];
  TcSmem& sm = *reinterpret_cast<TcSmem*>(tile_smem_raw);
  // the six R^T terms into shared memory, 16-byte chunks swizzled
  {
    const uint4* srcv = reinterpret_cast<const uint4*>(a.rot.RT_split);
    constexpr int kChunks = 2 * 3 * kD * kD / 8;
    for (int c = threadIdx.x; c < kChunks; c += kTcThreads) {
      const int row = c >> 4, chunk = c & 15, n = row & (kD - 1);
      reinterpret_cast<uint4*>(&sm.rt[0][0][0][0])[(row << 4) | (chunk ^ (n & 7))] = __ldg(srcv + c);
    }
  }
  __syncthreads();
  const int slot = threadIdx.x / 256, m = (threadIdx.x >> 7) & 1, bar = 1 + 2 * slot + m;
  const int Hkv = a.c.num_kv_heads;
  const long long n_tiles = (long long)tiles_per_req * Hkv * a.c.batch;
  for (long long tile = (long long)blockIdx.x * kTcSlots + slot; tile < n_tiles; tile += (long long)gridDim.x * kTcSlots) {
    const int x = (int)(tile % tiles_per_req);
    const int h = (int)((tile / tiles_per_req) % Hkv);
    const int b = (int)(tile / ((long long)tiles_per_req * Hkv));
    int p0, n, tok0;
    if (!request_span(a, b, p0, n, tok0)) continue;
    const int L = p0 + n;
    const int lo = max(p0, kSink), hi = L - kRecent;
    if (hi <= lo) continue;
    const int lp = lo / kPage + x;
    if (lp * kPage >= hi) continue;
    const int r_lo = max(lo - lp * kPage, 0), r_hi = min(hi - lp * kPage, kPage);
    uint8_t* blk = history_block(a.c, b, h, lp * kPage, a.err);
    if (blk == nullptr) continue;
    tc_quantize_tile(a, b, h, tok0, p0, r_lo, r_hi, lp, blk, slot, m, bar, sm);
  }
}

}  // namespace

cudaError_t launch_append(const AppendLaunch& a, cudaStream_t stream) {
  const int B = a.c.batch, Hkv = a.c.num_kv_heads;
  if (a.cu_seqlens == nullptr) {
    append_one_kernel<<<dim3(Hkv, B), 2 * kQuantThreads, 0, stream>>>(a);
    return cudaGetLastError();
  }
  if (!(a.flags & 1u)) append_evict_kernel<<<dim3(kRecent, Hkv, B), 2 * kQuantThreads, 0, stream>>>(a);
  append_bf16_kernel<<<dim3(kSink + kRecent, B), 128, 0, stream>>>(a);
  const int tiles = (a.max_tokens_per_req + kPage - 1) / kPage + 1;  // INT2 pages a request can touch
  const size_t smem = sizeof(TcSmem);
  static int sms = 0;
  if (sms == 0) {
    int dev = 0, n_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(append_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    sms = n_sm;
  }
  const long long work = (long long)tiles * Hkv * B;
  const int blocks = (int)std::min<long long>((work + kTcSlots - 1) / kTcSlots, (long long)sms);
  append_tile_kernel<<<blocks, kTcThreads, smem, stream>>>(a, tiles);
  return cudaGetLastError();
}

}  // namespace oscar
