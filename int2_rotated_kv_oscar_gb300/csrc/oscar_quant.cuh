// Rotate + clip + quantise one token into a packed INT2 block (device code
// shared by the append kernels and the fused decode-step kernel).
//
// ainsights.it "OSCAR: Come Together AI Comprime la KV Cache a 2-bit per LLM",
// "Architettura del Sistema di Serving e Layout di Memoria": each token is
// rotated, clipped and quantised on its way into the INT2 history.
// gist.science "Resumen Técnico: OSCAR ...", §2.2 A.3-4: R = U H_Had P_br and
// per-layer clip thresholds.  The rotation is applied as one dense product
// with the composite R formed on the host.
#pragma once

#include "oscar_device.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

// K codes of a 16-token tile: the 32-bit word (lane 4 (u % 8) + tq, word
// 2 (u / 8) + kp) of row u holds channels j = 32 ks + 16 kh + 4 tq + b for
// ks in {2 kp, 2 kp + 1}, kh, b in 0..3 at bit 8 b + 2 (2 (ks % 2) + kh).
// Byte offset inside a block's K code area of that word for row t.
__device__ __forceinline__ int k_word_offset(int t, int tq, int kp) {
  const int T = t >> 4, u = t & 15;
  return 512 * T + 16 * (4 * (u & 7) + tq) + 4 * (2 * (u >> 3) + kp);
}

// The K word (tq, kp) of one row from its 128 codes (one byte each).
__device__ __forceinline__ uint32_t k_word(const uint8_t* codes, int tq, int kp) {
  uint32_t w = 0;
#pragma unroll
  for (int ks2 = 0; ks2 < 2; ++ks2)
#pragma unroll
    for (int kh = 0; kh < 2; ++kh)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        w |= (uint32_t)codes[32 * (2 * kp + ks2) + 16 * kh + 4 * tq + b] << (8 * b + 2 * (2 * ks2 + kh));
  return w;
}

// Byte offset inside a block's V code area of the 16-bit half holding the
// codes of row t for the channels {jj + 16 r : r = 0..7}.
__device__ __forceinline__ int v_half_offset(int t, int jj) {
  const int T = t >> 4, u = t & 15;
  return 512 * T + 16 * (4 * (jj & 7) + ((u & 7) >> 1)) + 4 * (2 * (u >> 3) + (jj >> 3)) + 2 * (u & 1);
}

struct QuantSmem {
  __align__(16) float x[kD];
  float zq[4][kD];  // partial products over the four quarters of the rows of R
  float red[4];
  uint8_t code[kD];
};

constexpr int kQuantThreads = 512;  // threads per token: channel t = u % 128, row quarter u / 128

// The packed bytes one token adds to a block, as quantize_token stores them
// (for a reader that already holds a copy of the block from before the store).
struct RowPatch {
  uint32_t kword[8];   // K word (tq, kp) = (i % 4, i / 4) of the row
  uint16_t vhalf[16];  // V half of channels {jj + 16 r : r = 0..7}, jj = i
  uint16_t kscale[2], vscale[2];
  int row;  // the block row these bytes belong to (-1: none)
};

// Rotate + clip + quantise one token and store its codes and scale in row
// `row` of the K or V part of `block`.  Called by the kQuantThreads threads
// u of a group synchronised by named barrier `bar`; x: the token's channel
// u % 128 (read from the threads u < 128).  R: the layer's composite
// rotation (global or shared memory).  Thread u forms the partial product of
// rows [32 (u / 128), 32 (u / 128) + 32) of R for channel u % 128; the four
// partials are added in quarter order.
// rr(ii) = R[32 (u / 128) + ii][u % 128] (from memory or from registers).
// rflags: the layer's factors; without U the group's first warp applies H as
// the in-register butterfly and P as an index map instead (R is not read).
template <typename RowOf>
__device__ __forceinline__ void quantize_token(float x, RowOf rr, float tau, uint8_t* block, int row, bool is_v,
                                               QuantSmem& sm, int u, int bar, RowPatch* patch, uint32_t rflags) {
  const int t = u & 127, kq = u >> 7, lane = u & 31, warp = (u >> 5) & 3;
  const bool dense = (rflags & kRotU) != 0;
  if (kq == 0) sm.x[t] = x;
  group_sync(bar, kQuantThreads);
  if (dense) {
    float z0 = 0.f, z1 = 0.f;
#pragma unroll
    for (int ii = 0; ii < 32; ii += 4) {
      const float4 xv = *reinterpret_cast<const float4*>(&sm.x[32 * kq + ii]);
      z0 = fmaf(xv.x, rr(ii), z0);
      z1 = fmaf(xv.y, rr(ii + 1), z1);
      z0 = fmaf(xv.z, rr(ii + 2), z0);
      z1 = fmaf(xv.w, rr(ii + 3), z1);
    }
    sm.zq[kq][t] = z0 + z1;
  } else if (u < 32) {  // x' = x H P: (x H)_i lands in channel rev(i)
    float v[4];
    const float4 xv = *reinterpret_cast<const float4*>(&sm.x[4 * u]);
    v[0] = xv.x;
    v[1] = xv.y;
    v[2] = xv.z;
    v[3] = xv.w;
    if (rflags & kRotH) {
      hadamard128(v, u);
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] *= kInvSqrt128;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) sm.zq[0][(rflags & kRotP) ? brev7(4 * u + e) : 4 * u + e] = v[e];
  }
  group_sync(bar, kQuantThreads);
  float z = 0.f;
  if (kq == 0) {
    z = dense ? ((sm.zq[0][t] + sm.zq[1][t]) + sm.zq[2][t]) + sm.zq[3][t] : sm.zq[0][t];
    const float amax = warp_max(fabsf(z));
    if (lane == 0) sm.red[warp] = amax;
  }
  group_sync(bar, kQuantThreads);
  const int grp = t >> 6;
  const float a = fminf(fmaxf(sm.red[2 * grp], sm.red[2 * grp + 1]), tau);
  const __half sh = __float2half_rn(a / 1.5f);
  if (kq == 0) {
    const float s = __half2float(sh);
    sm.code[t] = (uint8_t)((z >= -s) + (z >= 0.f) + (z >= s));
  }
  group_sync(bar, kQuantThreads);
  if (kq != 0) {
  } else if (!is_v) {
    if (t < 8) {
      const uint32_t kw = k_word(sm.code, t & 3, t >> 2);
      *reinterpret_cast<uint32_t*>(block + kKCodes + k_word_offset(row, t & 3, t >> 2)) = kw;
      if (patch != nullptr) patch->kword[t] = kw;
    }
  } else {
    if (t < 16) {
      uint32_t hv = 0;
#pragma unroll
      for (int r = 0; r < 8; ++r) hv |= (uint32_t)sm.code[t + 16 * r] << (2 * r);
      *reinterpret_cast<uint16_t*>(block + kVCodes + v_half_offset(row, t)) = (uint16_t)hv;
      if (patch != nullptr) patch->vhalf[t] = (uint16_t)hv;
    }
  }
  if (kq == 0 && (t & 63) == 0) {
    *reinterpret_cast<__half*>(block + (is_v ? kVScales : kKScales) + 4 * row + 2 * grp) = sh;
    if (patch != nullptr) (is_v ? patch->vscale : patch->kscale)[grp] = __half_as_ushort(sh);
  }
  if (patch != nullptr && u == 0) patch->row = row;
  group_sync(bar, kQuantThreads);
}

// R: the layer's composite rotation, row-major in global or shared memory.
__device__ __forceinline__ void quantize_token(float x, const float* __restrict__ R, float tau, uint8_t* block,
                                               int row, bool is_v, QuantSmem& sm, int u, int bar, RowPatch* patch,
                                               uint32_t rflags) {
  const float* col = R + (size_t)32 * (u >> 7) * kD + (u & 127);
  quantize_token(x, [&](int ii) { return col[ii * kD]; }, tau, block, row, is_v, sm, u, bar, patch, rflags);
}

// Locate (and check) the INT2 block of position e of request b, head h.
// Element offset of the BF16 recent row of position p (>= 64) of request b,
// KV head h (channel 0) in k_ring / v_ring: row (p - 64) % 256 of the request's
// ring slot, or, with a recent page table, row p % 64 of the BF16 page holding
// logical page p / 64.  False (and an error bit, if report) for a bad entry.
__device__ __forceinline__ bool recent_row(const CacheRefs& c, int b, int h, int p, size_t& off, unsigned* err,
                                           bool report) {
  if (c.recent_table != nullptr) {
    const int lp = p >> 6;
    if (lp >= c.max_pages) {
      if (report) set_error(err, kErrLength);
      return false;
    }
    const int pg = c.recent_table[(size_t)b * c.max_pages + lp];
    if (pg < 0 || pg >= c.num_ring) {
      if (report) set_error(err, kErrRing);
      return false;
    }
    off = (((size_t)pg * c.num_kv_heads + h) * kPage + (p & 63)) * kD;
    return true;
  }
  const int slot = c.ring_slot[b];
  if (slot < 0 || slot >= c.num_ring) {
    if (report) set_error(err, kErrRing);
    return false;
  }
  off = (((size_t)slot * c.num_kv_heads + h) * kRecent + ((p - kSink) % kRecent)) * kD;
  return true;
}

__device__ __forceinline__ uint8_t* history_block(const CacheRefs& c, int b, int h, int e, unsigned* err) {
  const int lp = e >> 6;
  if (lp >= c.max_pages) {
    if (threadIdx.x == 0) set_error(err, kErrLength);
    return nullptr;
  }
  const int phys = c.page_table[(size_t)b * c.max_pages + lp];
  if (phys < 0 || phys >= c.num_pages) {
    if (threadIdx.x == 0) set_error(err, kErrPage);
    return nullptr;
  }
  return c.pages + ((size_t)phys * c.num_kv_heads + h) * kBlockBytes;
}

// Decode append of request b, KV head h: K (half 0) or V (half 1), by the
// kQuantThreads threads u of a group synchronised by named barrier `bar`;
// the threads u < 128 move channel u.  Writes the token into the sink page
// (position < 64) or its ring row; a position >= 320 first moves the ring
// row's old token (position - 256) into its INT2 history row.
__device__ __forceinline__ void append_one_body(const AppendLaunch& a, int b, int h, int half, int u,
                                                const float* Rk, const float* Rv, QuantSmem& sm, int bar,
                                                RowPatch* patch = nullptr) {
  const bool is_v = half == 1;
  const int t = u & 127;
  const bool mover = u < kD;
  const CacheRefs& c = a.c;
  const int Hkv = c.num_kv_heads;
  // independent loads first, so that their round trips overlap
  const int p = a.pos[b];
  const uint16_t xn = (is_v ? a.v : a.k)[((size_t)b * Hkv + h) * kD + t];
  if (p < 0 || ((a.flags & 1u) && p > kSink)) {
    if (threadIdx.x == 0) set_error(a.err, kErrLength);
    return;
  }
  if (p < kSink) {
    const int sp = c.sink_page[b];
    if (sp < 0 || sp >= c.num_sink) {
      if (threadIdx.x == 0) set_error(a.err, kErrSink);
      return;
    }
    if (mover) (is_v ? c.v_sink : c.k_sink)[(((size_t)sp * Hkv + h) * kSink + p) * kD + t] = xn;
    return;
  }
  uint16_t* ring = is_v ? c.v_ring : c.k_ring;
  size_t rdst;
  if (!recent_row(c, b, h, p, rdst, a.err, threadIdx.x == 0)) return;
  rdst += t;
  if (p >= kSink + kRecent) {
    // the token at e = p - 256 leaves the window (in the ring: the same row, read before overwrite)
    const int e = p - kRecent;
    size_t rsrc;
    if (!recent_row(c, b, h, e, rsrc, a.err, threadIdx.x == 0)) return;
    const uint16_t xo = ring[rsrc + t];  // in flight while the page table is read
    uint8_t* blk = history_block(c, b, h, e, a.err);
    if (blk != nullptr)
      quantize_token(bf16_bits_to_float(xo), is_v ? Rv : Rk, is_v ? a.rot.tau_v : a.rot.tau_k, blk, e & 63, is_v,
                     sm, u, bar, patch, a.rot.flags);
  }
  if (mover) ring[rdst] = xn;
}

// The decode append of append_one_body for K and then V of one (request b,
// KV head h), by one kQuantThreads group, with the loads of both halves
// issued together and R_K / R_V given by rk / rv as for quantize_token (the
// same arithmetic, so the same bytes); the evicted row's bytes also go to
// *patch.
template <typename RowK, typename RowV>
__device__ __forceinline__ void append_pair_body(const AppendLaunch& a, int b, int h, int u, RowK rk, RowV rv,
                                                 QuantSmem& sm, int bar, RowPatch* patch) {
  const CacheRefs& c = a.c;
  const int Hkv = c.num_kv_heads, t = u & 127;
  const bool mover = u < kD;
  const int p = a.pos[b];
  const size_t nrow = ((size_t)b * Hkv + h) * kD + t;
  const uint16_t xk = a.k[nrow], xv = a.v[nrow];
  if (p < 0 || ((a.flags & 1u) && p > kSink)) {
    if (threadIdx.x == 0) set_error(a.err, kErrLength);
    return;
  }
  if (p < kSink) {
    const int sp = c.sink_page[b];
    if (sp < 0 || sp >= c.num_sink) {
      if (threadIdx.x == 0) set_error(a.err, kErrSink);
      return;
    }
    const size_t d = (((size_t)sp * Hkv + h) * kSink + p) * kD + t;
    if (mover) {
      c.k_sink[d] = xk;
      c.v_sink[d] = xv;
    }
    return;
  }
  size_t rdst;
  if (!recent_row(c, b, h, p, rdst, a.err, threadIdx.x == 0)) return;
  rdst += t;
  if (p >= kSink + kRecent) {
    const int e = p - kRecent;
    size_t rsrc;
    if (!recent_row(c, b, h, e, rsrc, a.err, threadIdx.x == 0)) return;
    rsrc += t;
    const uint16_t ok = c.k_ring[rsrc], ov = c.v_ring[rsrc];  // in flight while the page table is read
    uint8_t* blk = history_block(c, b, h, e, a.err);
    if (blk != nullptr) {
      quantize_token(bf16_bits_to_float(ok), rk, a.rot.tau_k, blk, e & 63, false, sm, u, bar, patch, a.rot.flags);
      quantize_token(bf16_bits_to_float(ov), rv, a.rot.tau_v, blk, e & 63, true, sm, u, bar, patch, a.rot.flags);
    }
  }
  if (mover) {
    c.k_ring[rdst] = xk;
    c.v_ring[rdst] = xv;
  }
}

}  // namespace
}  // namespace oscar
