// OSCAR decode attention over the mixed-precision paged cache (sm_103a).
//
// gist.science "Resumen Técnico: OSCAR ...", §2.2 B: a fused kernel unpacks,
// de-quantises, undoes the rotation and computes attention over the INT2
// history, paged and prefix-cache compatible, with no extra memory traffic.
// ainsights.it "OSCAR: Come Together AI ...", "Architettura del Sistema di
// Serving e Layout di Memoria": sink and recent tokens stay BF16.
//
// Design (GB300):
//  * prep kernel, one block per (request, KV head): q' = q R_K (fp32 x U,
//    Walsh-Hadamard butterfly, bit reversal), times sm_scale * log2(e) and a
//    power-of-two normalisation, split into fp16 value + fp16 residual and
//    laid out as tensor-core B fragments; the plain q for the BF16 segment
//    likewise; zeroes the split counters.
//  * decode kernel, one block per (work item, KV head, request), 4 warps.
//    Work items are chunks of INT2 history pages (rotated basis) or 64-token
//    BF16 blocks (sink, ring quarters; original basis).  Each warp streams
//    its pages through a private ring of shared-memory stages filled by bulk
//    asynchronous copies (one 4608-byte copy per page), turns each pair of
//    2-bit codes into the exact fp16 levels (c - 1.5) with one LOP3 and one
//    HFMA2, runs QK^T and PV on mma.sync m16n8k16 (tokens x channels and
//    channels x tokens against the query heads) with an online softmax in
//    the log2 domain.  Warps merge in shared memory; each block writes one
//    partial (m, l, acc); the last block of a (request, KV head) merges all
//    partials (log-sum-exp), rotates the INT2 part back (acc P H U_V^T) and
//    writes the fp32 output.  No block ever waits on another.
//
// Precision: q and the softmax weights times the V scales enter the MMAs as
// fp16 value + fp16 residual (~22 significant bits).  With at most 4 query
// heads per KV head the residual rides in the MMA's otherwise unused N
// columns 4..7 (no extra MMAs); with 5..8 heads it takes a second MMA.

#include <cmath>

#include "oscar_device.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kInvSqrtD = 0.08838834764831845f;
constexpr int kWarps = 4;
constexpr int kStages = 3;
constexpr unsigned kWaitLimit = 1u << 22;
// The PV B operand is p * s * 2^k (INT2 history, s = V scale) or p * 2^k (BF16
// tiles), with p <= 2^kLazy.  k is the largest power of two that keeps it
// below 60000 for the layer's largest possible scale, so small weights stay
// clear of the fp16 subnormal range.
constexpr float kLazy = 4.0f;           // rescale only when the max grows by more than 2^4
constexpr float kPScaleBF16 = 2048.0f;  // 2^4 * 2048 < 60000

// Exact fp16 pair of the levels (c - 1.5) of the codes at index r (0..7) of
// both 16-bit halves of a code word.  One LOP3 puts the code into the low
// mantissa of the fp16 1024 ((w & mask) | 0x6400: the value 1024 + c 4^r'),
// one HFMA2 maps it to (1024 + c 4^r') 4^-r' - (1024 4^-r' + 1.5) = c - 1.5.
// r' is the code's 2-bit position in the source word: index 0 is taken from
// w << 2 (r' = 1; at r' = 0 the offset 1025.5 would not be an fp16), indices
// 1..4 from w (r' = r), indices 5..7 from w >> 6 (r' = r - 3).  The levels
// are normal fp16 numbers: tensor-core products of subnormal operands lose
// precision.
struct CodeWord {
  uint32_t lo2, w, hi6;  // w << 2, w, w >> 6
  __device__ __forceinline__ explicit CodeWord(uint32_t x) : lo2(x << 2), w(x), hi6(x >> 6) {}
};

__device__ __forceinline__ uint32_t lop_and_or(uint32_t x, uint32_t mask) {
  uint32_t y;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(y) : "r"(x), "r"(mask), "r"(0x64006400u));  // (a & b) | c
  return y;
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

template <int R>
__device__ __forceinline__ uint32_t code_level(const CodeWord& cw) {
  constexpr int rp = R == 0 ? 1 : (R < 5 ? R : R - 3);
  // fp16 constants 4^-r' and -(1024 4^-r' + 1.5) for r' = 1..4, in both halves
  constexpr uint32_t kScale = rp == 1 ? 0x34003400u : rp == 2 ? 0x2C002C00u : rp == 3 ? 0x24002400u : 0x1C001C00u;
  constexpr uint32_t kBias = rp == 1 ? 0xDC06DC06u : rp == 2 ? 0xD418D418u : rp == 3 ? 0xCC60CC60u : 0xC580C580u;
  const uint32_t src = R == 0 ? cw.lo2 : (R < 5 ? cw.w : cw.hi6);
  return hfma2_u32(lop_and_or(src, 0x00030003u << (2 * rp)), kScale, kBias);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// fp16 value of v (part 0) or the fp32 residual v - fp16(v) (part 1, rounded later)
__device__ __forceinline__ float split_part(float v, int part) {
  const float hi = __half2float(__float2half_rn(v));
  return part == 0 ? hi : v - hi;
}

struct PrepArgs {
  const uint16_t* q;
  const float* U_K;
  unsigned flags;
  float sm_scale;
  int Hq, Hkv, g;
  uint32_t* qfrag;
  uint32_t* qplain;
  float* qconst;
  int* counters;
};

// ------------------------------------------------------------------ prep
// grid (Hkv, B), 128 threads.
//
// Fragment words per (request, KV head): [32 lanes][32].  The MMA B column of
// lane L is n = L / 4.  With g <= 4 ("packed"), column n carries head n % 4
// and part n / 4 (0: fp16 value, 1: fp16 residual) in words 0..15; with
// g > 4 column n is head n, words 0..15 hold the values and 16..31 the
// residuals.
__global__ void __launch_bounds__(128) prep_kernel(PrepArgs a) {
  __shared__ float xs[kMaxG][kD];
  __shared__ float qr[kMaxG][kD];
  __shared__ float qp[kMaxG][kD];
  __shared__ float scratch[kD];
  __shared__ float red[8];
  const int h = blockIdx.x, b = blockIdx.y, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int g = a.g, bh = b * a.Hkv + h;
  const bool packed = g <= 4;
  if (t == 0) a.counters[bh] = 0;
  const float c = a.sm_scale * kLog2e;
  for (int n = 0; n < g; ++n) xs[n][t] = bf16_bits_to_float(a.q[((size_t)b * a.Hq + h * g + n) * kD + t]);
  __syncthreads();
  float z[kMaxG];
#pragma unroll
  for (int n = 0; n < kMaxG; ++n) z[n] = 0.f;
#pragma unroll 4
  for (int i = 0; i < kD; ++i) {
    const float u = __ldg(a.U_K + i * kD + t);
#pragma unroll
    for (int n = 0; n < kMaxG; ++n)
      if (n < g) z[n] = fmaf(xs[n][i], u, z[n]);
  }
#pragma unroll
  for (int n = 0; n < kMaxG; ++n) {
    if (n >= g) break;
    float v = z[n];
    if (a.flags & kRotH) v = fwht128_block(v, scratch) * kInvSqrtD;
    qr[n][t] = v;
  }
  __syncthreads();
#pragma unroll
  for (int n = 0; n < kMaxG; ++n) {
    if (n >= g) break;
    const float v = (a.flags & kRotP) ? qr[n][brev7(t)] : qr[n][t];
    z[n] = v * c;
    qp[n][t] = xs[n][t] * c;
  }
  __syncthreads();
#pragma unroll
  for (int n = 0; n < kMaxG; ++n)
    if (n < g) qr[n][t] = z[n];
  // power-of-two normalisations: max |q'| 2^-E <= 2^10, max |q| 2^-Ep <= 2^10
  float mr = 0.f, mp = 0.f;
  for (int n = 0; n < g; ++n) {
    mr = fmaxf(mr, fabsf(qr[n][t]));
    mp = fmaxf(mp, fabsf(qp[n][t]));
  }
  mr = warp_max(mr);
  mp = warp_max(mp);
  if (lane == 0) {
    red[warp] = mr;
    red[4 + warp] = mp;
  }
  __syncthreads();
  mr = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  mp = fmaxf(fmaxf(red[4], red[5]), fmaxf(red[6], red[7]));
  int er = 0, ep = 0;
  if (mr > 0.f) {
    frexpf(mr, &er);
    er -= 10;
  }
  if (mp > 0.f) {
    frexpf(mp, &ep);
    ep -= 10;
  }
  const float sr = ldexpf(1.f, -er), sp = ldexpf(1.f, -ep);
  // QK B fragments over the INT2 history: MMA i (group i / 4, r0 = 2 (i % 4))
  // takes b0 = q'[64 grp + 16 tig + {0, 8} + r0] and b1 = the same at r0 + 1.
  // BF16 segment: MMA ks = i takes channels 32 tig + 4 ks + {0,1} (b0) and {2,3} (b1).
  uint32_t* qf = a.qfrag + (size_t)bh * kQFragWords;
  uint32_t* qpl = a.qplain + (size_t)bh * kQFragWords;
  for (int e = t; e < kQFragWords; e += 128) {
    const int L = e >> 5, w = e & 31, set = w >> 4, ww = w & 15, i = ww >> 1, bs = ww & 1;
    const int n = L >> 2, tig = L & 3;
    const int head = packed ? (n & 3) : n;
    const int part = packed ? (n >> 2) : set;
    uint32_t vr = 0, vp = 0;
    if (head < g && !(packed && set == 1)) {
      const int grp = i >> 2, r = 2 * (i & 3) + bs;
      const int ch = 64 * grp + 16 * tig + r;
      vr = pack_f16x2(split_part(qr[head][ch] * sr, part), split_part(qr[head][ch + 8] * sr, part));
      const int cp = 32 * tig + 4 * i + 2 * bs;
      vp = pack_f16x2(split_part(qp[head][cp] * sp, part), split_part(qp[head][cp + 1] * sp, part));
    }
    qf[e] = vr;
    qpl[e] = vp;
  }
  if (t == 0) {
    float* qc = a.qconst + (size_t)bh * kQConstFloats;
    qc[16] = ldexpf(1.f, er);
    qc[17] = ldexpf(1.f, ep);
  }
}

// ------------------------------------------------------------------ decode
struct DecodeArgs {
  int mode;
  CacheRefs c;
  const uint16_t* kb_pages;
  const uint16_t* vb_pages;
  const int32_t* ctx_len;
  int Hq, Hkv, g;
  int n_items, n_chunks, chunk_pages;
  const uint32_t* qfrag;
  const uint32_t* qplain;
  const float* qconst;
  float* partials;
  int* counters;
  const float* U_VT;
  unsigned flags;
  float pscale, inv_pscale;
  float* out;
  unsigned* err;
};

struct WarpState {
  float m[2], l[2];
  float acc[8][4];
};

__device__ __forceinline__ void state_init(WarpState& st) {
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) st.acc[i][k] = 0.f;
}

// Update the running maxima with this tile's maxima (per lane: columns 2 tig, 2 tig + 1).
__device__ __forceinline__ void online_max(WarpState& st, float mx0, float mx1) {
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  const bool need = (mx0 > st.m[0] + kLazy) || (mx1 > st.m[1] + kLazy);
  if (__any_sync(0xffffffffu, need)) {
    const float n0 = fmaxf(st.m[0], mx0), n1 = fmaxf(st.m[1], mx1);
    const float a0 = (n0 == -INFINITY) ? 1.f : ex2(st.m[0] - n0);
    const float a1 = (n1 == -INFINITY) ? 1.f : ex2(st.m[1] - n1);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      st.acc[i][0] *= a0;
      st.acc[i][2] *= a0;
      st.acc[i][1] *= a1;
      st.acc[i][3] *= a1;
    }
    st.l[0] *= a0;
    st.l[1] *= a1;
    st.m[0] = n0;
    st.m[1] = n1;
  }
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t u) {
  return __half22float2(*reinterpret_cast<const __half2*>(&u));
}

// fp16 pair of (x0, x1) and of their rounding residuals
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_f16x2(x0, x1);
  const float2 h = half2_bits_to_float2(hi);
  lo = pack_f16x2(x0 - h.x, x1 - h.y);
}

// packed mode: lanes holding value columns take the fp16 value, lanes holding
// residual columns (tig >= 2) take the residual
__device__ __forceinline__ uint32_t pick_pair(float x0, float x1, bool residual) {
  uint32_t hi, lo;
  split_pair(x0, x1, hi, lo);
  return residual ? lo : hi;
}

// One 64-token INT2 page (K and V codes + scales) staged in shared memory.
template <bool PACK4>
__device__ __forceinline__ void int2_page(const uint8_t* __restrict__ blk, int n_valid, const uint32_t* qf,
                                          float scaleE, float pscale, WarpState& st, int lane) {
  const int q = lane >> 2;
  const bool resid = (lane & 3) >= 2;
  float lg[4][4];
#pragma unroll
  for (int T = 0; T < 4; ++T) {
    if (16 * T >= n_valid) {
#pragma unroll
      for (int k = 0; k < 4; ++k) lg[T][k] = -INFINITY;
      continue;
    }
    const uint4 kw = *reinterpret_cast<const uint4*>(blk + kKCodes + 512 * T + 16 * lane);
    const float2 sa = half2_bits_to_float2(*reinterpret_cast<const uint32_t*>(blk + kKScales + 4 * (16 * T + q)));
    const float2 sb =
        half2_bits_to_float2(*reinterpret_cast<const uint32_t*>(blk + kKScales + 4 * (16 * T + q + 8)));
    // Tensor-core f32 accumulation truncates, so each group's four MMAs run as
    // two zero-started chains that are added in fp32.
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, e0[4] = {0.f, 0.f, 0.f, 0.f};
    float d1[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
#define OSCAR_QK(D, X, Y, R, I)                                                              \
  do {                                                                                      \
    const uint32_t a0 = code_level<R>(X), a1 = code_level<R>(Y), a2 = code_level<R + 1>(X), \
                   a3 = code_level<R + 1>(Y);                                             \
    mma_f16(D, a0, a1, a2, a3, qf[2 * (I)], qf[2 * (I) + 1]);                              \
    if (!PACK4) mma_f16(D, a0, a1, a2, a3, qf[16 + 2 * (I)], qf[16 + 2 * (I) + 1]);        \
  } while (0)
    {
      const CodeWord x(kw.x), y(kw.z);  // group 0: token q, token q+8
      OSCAR_QK(d0, x, y, 0, 0);
      OSCAR_QK(e0, x, y, 2, 1);
      OSCAR_QK(d0, x, y, 4, 2);
      OSCAR_QK(e0, x, y, 6, 3);
    }
    {
      const CodeWord x(kw.y), y(kw.w);  // group 1
      OSCAR_QK(d1, x, y, 0, 4);
      OSCAR_QK(e1, x, y, 2, 5);
      OSCAR_QK(d1, x, y, 4, 6);
      OSCAR_QK(e1, x, y, 6, 7);
    }
#undef OSCAR_QK
    float l0 = fmaf(d0[0] + e0[0], sa.x, (d1[0] + e1[0]) * sa.y) * scaleE;
    float l1 = fmaf(d0[1] + e0[1], sa.x, (d1[1] + e1[1]) * sa.y) * scaleE;
    float l2 = fmaf(d0[2] + e0[2], sb.x, (d1[2] + e1[2]) * sb.y) * scaleE;
    float l3 = fmaf(d0[3] + e0[3], sb.x, (d1[3] + e1[3]) * sb.y) * scaleE;
    if (PACK4) {  // value column + residual column
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      l2 += __shfl_xor_sync(0xffffffffu, l2, 2);
      l3 += __shfl_xor_sync(0xffffffffu, l3, 2);
    }
    const bool va = 16 * T + q < n_valid, vb = 16 * T + q + 8 < n_valid;
    lg[T][0] = va ? l0 : -INFINITY;
    lg[T][1] = va ? l1 : -INFINITY;
    lg[T][2] = vb ? l2 : -INFINITY;
    lg[T][3] = vb ? l3 : -INFINITY;
  }
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int T = 0; T < 4; ++T) {
    mx0 = fmaxf(mx0, fmaxf(lg[T][0], lg[T][2]));
    mx1 = fmaxf(mx1, fmaxf(lg[T][1], lg[T][3]));
  }
  online_max(st, mx0, mx1);
#pragma unroll
  for (int T = 0; T < 4; ++T) {
    if (16 * T >= n_valid) continue;
    const float p0 = ex2(lg[T][0] - st.m[0]), p1 = ex2(lg[T][1] - st.m[1]);
    const float p2 = ex2(lg[T][2] - st.m[0]), p3 = ex2(lg[T][3] - st.m[1]);
    st.l[0] += p0 + p2;
    st.l[1] += p1 + p3;
    const bool va = 16 * T + q < n_valid, vb = 16 * T + q + 8 < n_valid;
    float2 sa = half2_bits_to_float2(*reinterpret_cast<const uint32_t*>(blk + kVScales + 4 * (16 * T + q)));
    float2 sb = half2_bits_to_float2(*reinterpret_cast<const uint32_t*>(blk + kVScales + 4 * (16 * T + q + 8)));
    sa.x = va ? sa.x * pscale : 0.f;
    sa.y = va ? sa.y * pscale : 0.f;
    sb.x = vb ? sb.x * pscale : 0.f;
    sb.y = vb ? sb.y * pscale : 0.f;
    const uint4 vw = *reinterpret_cast<const uint4*>(blk + kVCodes + 512 * T + 16 * lane);
    const CodeWord w0(vw.x), w1(vw.y), w2(vw.z), w3(vw.w);
    if (PACK4) {
      const uint32_t b00 = movmatrix_trans(pick_pair(p0 * sa.x, p1 * sa.x, resid));
      const uint32_t b01 = movmatrix_trans(pick_pair(p2 * sb.x, p3 * sb.x, resid));
      const uint32_t b10 = movmatrix_trans(pick_pair(p0 * sa.y, p1 * sa.y, resid));
      const uint32_t b11 = movmatrix_trans(pick_pair(p2 * sb.y, p3 * sb.y, resid));
#define OSCAR_PV(M, B0, B1) \
  mma_f16(st.acc[M], code_level<M>(w0), code_level<M>(w1), code_level<M>(w2), code_level<M>(w3), B0, B1)
      OSCAR_PV(0, b00, b01);
      OSCAR_PV(1, b00, b01);
      OSCAR_PV(2, b00, b01);
      OSCAR_PV(3, b00, b01);
      OSCAR_PV(4, b10, b11);
      OSCAR_PV(5, b10, b11);
      OSCAR_PV(6, b10, b11);
      OSCAR_PV(7, b10, b11);
#undef OSCAR_PV
    } else {
      uint32_t h00, l00, h01, l01, h10, l10, h11, l11;
      split_pair(p0 * sa.x, p1 * sa.x, h00, l00);
      split_pair(p2 * sb.x, p3 * sb.x, h01, l01);
      split_pair(p0 * sa.y, p1 * sa.y, h10, l10);
      split_pair(p2 * sb.y, p3 * sb.y, h11, l11);
      h00 = movmatrix_trans(h00);
      l00 = movmatrix_trans(l00);
      h01 = movmatrix_trans(h01);
      l01 = movmatrix_trans(l01);
      h10 = movmatrix_trans(h10);
      l10 = movmatrix_trans(l10);
      h11 = movmatrix_trans(h11);
      l11 = movmatrix_trans(l11);
#define OSCAR_PV2(M, H0, H1, L0, L1)                                                       \
  do {                                                                                     \
    const uint32_t a0 = code_level<M>(w0), a1 = code_level<M>(w1), a2 = code_level<M>(w2), \
                   a3 = code_level<M>(w3);                                               \
    mma_f16(st.acc[M], a0, a1, a2, a3, H0, H1);                                            \
    mma_f16(st.acc[M], a0, a1, a2, a3, L0, L1);                                            \
  } while (0)
      OSCAR_PV2(0, h00, h01, l00, l01);
      OSCAR_PV2(1, h00, h01, l00, l01);
      OSCAR_PV2(2, h00, h01, l00, l01);
      OSCAR_PV2(3, h00, h01, l00, l01);
      OSCAR_PV2(4, h10, h11, l10, l11);
      OSCAR_PV2(5, h10, h11, l10, l11);
      OSCAR_PV2(6, h10, h11, l10, l11);
      OSCAR_PV2(7, h10, h11, l10, l11);
#undef OSCAR_PV2
    }
  }
}

// One 16-token BF16 tile (rows of K and V in global memory, original basis).
template <bool PACK4>
__device__ __forceinline__ void bf16_tile(const uint16_t* __restrict__ Kt, const uint16_t* __restrict__ Vt,
                                          int n_valid, const uint32_t* qpf, float scaleEp, WarpState& st,
                                          int lane) {
  const int q = lane >> 2, tig = lane & 3;
  const bool resid = tig >= 2;
  const bool va = q < n_valid, vb = q + 8 < n_valid;
  uint32_t ka[16], kb[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint4 u = va ? __ldg(reinterpret_cast<const uint4*>(Kt + q * kD + 32 * tig) + k) : make_uint4(0, 0, 0, 0);
    ka[4 * k + 0] = bf16x2_to_f16x2(u.x);
    ka[4 * k + 1] = bf16x2_to_f16x2(u.y);
    ka[4 * k + 2] = bf16x2_to_f16x2(u.z);
    ka[4 * k + 3] = bf16x2_to_f16x2(u.w);
    u = vb ? __ldg(reinterpret_cast<const uint4*>(Kt + (q + 8) * kD + 32 * tig) + k) : make_uint4(0, 0, 0, 0);
    kb[4 * k + 0] = bf16x2_to_f16x2(u.x);
    kb[4 * k + 1] = bf16x2_to_f16x2(u.y);
    kb[4 * k + 2] = bf16x2_to_f16x2(u.z);
    kb[4 * k + 3] = bf16x2_to_f16x2(u.w);
  }
  float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    float(&acc)[4] = (ks & 1) ? e : d;  // two chains, added in fp32 (the MMA accumulation truncates)
    mma_f16(acc, ka[2 * ks], kb[2 * ks], ka[2 * ks + 1], kb[2 * ks + 1], qpf[2 * ks], qpf[2 * ks + 1]);
    if (!PACK4)
      mma_f16(acc, ka[2 * ks], kb[2 * ks], ka[2 * ks + 1], kb[2 * ks + 1], qpf[16 + 2 * ks], qpf[17 + 2 * ks]);
  }
  float l0 = (d[0] + e[0]) * scaleEp, l1 = (d[1] + e[1]) * scaleEp;
  float l2 = (d[2] + e[2]) * scaleEp, l3 = (d[3] + e[3]) * scaleEp;
  if (PACK4) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    l2 += __shfl_xor_sync(0xffffffffu, l2, 2);
    l3 += __shfl_xor_sync(0xffffffffu, l3, 2);
  }
  l0 = va ? l0 : -INFINITY;
  l1 = va ? l1 : -INFINITY;
  l2 = vb ? l2 : -INFINITY;
  l3 = vb ? l3 : -INFINITY;
  online_max(st, fmaxf(l0, l2), fmaxf(l1, l3));
  const float p0 = ex2(l0 - st.m[0]), p1 = ex2(l1 - st.m[1]), p2 = ex2(l2 - st.m[0]), p3 = ex2(l3 - st.m[1]);
  st.l[0] += p0 + p2;
  st.l[1] += p1 + p3;
  uint32_t b0h, b0l, b1h, b1l;
  if (PACK4) {
    b0h = movmatrix_trans(pick_pair(p0 * kPScaleBF16, p1 * kPScaleBF16, resid));
    b1h = movmatrix_trans(pick_pair(p2 * kPScaleBF16, p3 * kPScaleBF16, resid));
    b0l = b1l = 0u;
  } else {
    split_pair(p0 * kPScaleBF16, p1 * kPScaleBF16, b0h, b0l);
    split_pair(p2 * kPScaleBF16, p3 * kPScaleBF16, b1h, b1l);
    b0h = movmatrix_trans(b0h);
    b0l = movmatrix_trans(b0l);
    b1h = movmatrix_trans(b1h);
    b1l = movmatrix_trans(b1l);
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t a[4];
#pragma unroll
    for (int blkid = 0; blkid < 4; ++blkid) {
      const int tr = blkid >> 1, cc = blkid & 1;  // token half, channel half
      const bool ok = tr ? vb : va;
      const uint32_t u =
          ok ? __ldg(reinterpret_cast<const uint32_t*>(Vt + (8 * tr + q) * kD + 16 * mt + 8 * cc + 2 * tig)) : 0u;
      a[blkid] = movmatrix_trans(bf16x2_to_f16x2(u));
    }
    // a[0]: channels 16mt+q, tokens 2tig..; a[1]: channels +8; a[2]: tokens +8; a[3]: both
    mma_f16(st.acc[mt], a[0], a[1], a[2], a[3], b0h, b1h);
    if (!PACK4) mma_f16(st.acc[mt], a[0], a[1], a[2], a[3], b0l, b1l);
  }
}

struct MergeSmem {
  float m[kWarps][8];
  float l[kWarps][8];
  float acc[kWarps][8][kD];
};

template <int MODE, bool PACK4>
__global__ void __launch_bounds__(128, 4) decode_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int item = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, q = lane >> 2, tig = lane & 3;
  const int bh = b * a.Hkv + h;
  const CacheRefs& c = a.c;
  int L = a.ctx_len[b];
  if (L < 0) {
    if (t == 0 && item == 0) set_error(a.err, kErrLength);
    L = 0;
  }
  WarpState st;
  state_init(st);
  const bool rotated = (MODE == 0) && item < a.n_chunks;
  constexpr int kQW = PACK4 ? 16 : 32;

  if (rotated) {
    // ---------------- INT2 history pages
    const int hist_end = max(kSink, L - kRecent);
    const int n_hist = (hist_end + kPage - 1) / kPage - 1;  // logical pages 1..n_hist
    if (n_hist + 1 > c.max_pages) {
      if (t == 0 && item == 0) set_error(a.err, kErrLength);
    }
    const int n_hist_ok = min(n_hist, c.max_pages - 1);
    const int lp0 = 1 + item * a.chunk_pages;
    const int lp1 = min(lp0 + a.chunk_pages, 1 + n_hist_ok);
    const int first = lp0 + warp;
    const int n_my = first < lp1 ? (lp1 - first + kWarps - 1) / kWarps : 0;
    if (n_my > 0) {
      uint32_t qf[kQW];
      {
        const uint4* src = reinterpret_cast<const uint4*>(a.qfrag + (size_t)bh * kQFragWords + lane * 32);
#pragma unroll
        for (int k = 0; k < kQW / 4; ++k) {
          const uint4 u = __ldg(src + k);
          qf[4 * k] = u.x;
          qf[4 * k + 1] = u.y;
          qf[4 * k + 2] = u.z;
          qf[4 * k + 3] = u.w;
        }
      }
      const float scaleE = __ldg(a.qconst + (size_t)bh * kQConstFloats + 16);
      uint8_t* stages = smem + (size_t)warp * kStages * kBlockBytes;
      uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kWarps * kStages * kBlockBytes) + warp * kStages;
      const uint8_t* pool = c.pages;
      auto phys_of = [&](int k) -> int {
        const int lp = first + kWarps * k;
        const int ph = c.page_table[(size_t)b * c.max_pages + lp];
        return (ph >= 0 && ph < c.num_pages) ? ph : -1;
      };
      auto issue = [&](int k) {  // lane 0 only
        const int s = k % kStages;
        const int ph = phys_of(k);
        if (ph >= 0) {
          mbar_arrive_expect_tx(&bars[s], kBlockBytes);
          bulk_copy_g2s(stages + (size_t)s * kBlockBytes, pool + ((size_t)ph * a.Hkv + h) * kBlockBytes, kBlockBytes,
                        &bars[s]);
        } else {
          set_error(a.err, kErrPage);
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&bars[s])) : "memory");
        }
      };
      if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0)
        for (int k = 0; k < min(kStages, n_my); ++k) issue(k);
      int k = 0;
      for (; k < n_my; ++k) {
        const int s = k % kStages;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[s], (k / kStages) & 1, kWaitLimit));
        if (!ok) {
          if (lane == 0) set_error(a.err, kErrTimeout);
          break;
        }
        const int lp = first + kWarps * k;
        if (phys_of(k) >= 0) {
          const int n_valid = min(kPage, hist_end - kPage * lp);
          int2_page<PACK4>(stages + (size_t)s * kBlockBytes, n_valid, qf, scaleE, a.pscale, st, lane);
        }
        __syncwarp();
        if (lane == 0 && k + kStages < n_my) {
          fence_proxy_async_smem();
          issue(k + kStages);
        }
      }
      // after a timeout, wait (bounded) for the copies still in flight
      for (int kk = k + 1; kk < min(k + kStages, n_my); ++kk)
        mbar_wait_bounded(&bars[kk % kStages], (kk / kStages) & 1, kWaitLimit);
      if (k < n_my) mbar_wait_bounded(&bars[k % kStages], (k / kStages) & 1, kWaitLimit);
    }
  } else {
    // ---------------- BF16 tiles (original basis)
    uint32_t qpf[kQW];
    {
      const uint4* src = reinterpret_cast<const uint4*>(a.qplain + (size_t)bh * kQFragWords + lane * 32);
#pragma unroll
      for (int k = 0; k < kQW / 4; ++k) {
        const uint4 u = __ldg(src + k);
        qpf[4 * k] = u.x;
        qpf[4 * k + 1] = u.y;
        qpf[4 * k + 2] = u.z;
        qpf[4 * k + 3] = u.w;
      }
    }
    const float scaleEp = __ldg(a.qconst + (size_t)bh * kQConstFloats + 17);
    if (MODE == 0) {
      const int kb = item - a.n_chunks;  // 0: sink, 1..4: ring quarters
      const uint16_t *Kb = nullptr, *Vb = nullptr;
      int valid = 0;
      if (kb == 0) {
        valid = min(L, kSink);
        if (valid > 0) {
          const int sp = c.sink_page[b];
          if (sp < 0 || sp >= c.num_sink) {
            if (t == 0) set_error(a.err, kErrSink);
            valid = 0;
          } else {
            const size_t off = ((size_t)sp * a.Hkv + h) * kSink * kD;
            Kb = c.k_sink + off;
            Vb = c.v_sink + off;
          }
        }
      } else {
        const int q4 = kb - 1;
        valid = L >= kSink + kRecent ? kPage : max(0, min(kPage, L - kSink - kPage * q4));
        if (valid > 0) {
          const int slot = c.ring_slot[b];
          if (slot < 0 || slot >= c.num_ring) {
            if (t == 0) set_error(a.err, kErrRing);
            valid = 0;
          } else {
            const size_t off = (((size_t)slot * a.Hkv + h) * kRecent + kPage * q4) * kD;
            Kb = c.k_ring + off;
            Vb = c.v_ring + off;
          }
        }
      }
      const int nv = min(16, valid - 16 * warp);
      if (nv > 0) bf16_tile<PACK4>(Kb + 16 * warp * kD, Vb + 16 * warp * kD, nv, qpf, scaleEp, st, lane);
    } else {
      // plain BF16 paged cache: item covers pages [item*C, item*C + C); warp w takes tile w of each
      const int n_pages = (L + kPage - 1) / kPage;
      if (n_pages > c.max_pages) {
        if (t == 0 && item == 0) set_error(a.err, kErrLength);
      }
      const int pg0 = item * a.chunk_pages;
      const int pg1 = min(min(pg0 + a.chunk_pages, n_pages), c.max_pages);
      for (int pg = pg0; pg < pg1; ++pg) {
        const int ph = c.page_table[(size_t)b * c.max_pages + pg];
        if (ph < 0 || ph >= c.num_pages) {
          if (lane == 0) set_error(a.err, kErrPage);
          continue;
        }
        const int nv = min(16, L - kPage * pg - 16 * warp);
        if (nv <= 0) continue;
        const size_t off = (((size_t)ph * a.Hkv + h) * kPage + 16 * warp) * kD;
        bf16_tile<PACK4>(a.kb_pages + off, a.vb_pages + off, nv, qpf, scaleEp, st, lane);
      }
    }
  }

  // ---------------- finalise each warp's state and merge the warps
  __syncthreads();  // stage memory is reused below
  MergeSmem& ms = *reinterpret_cast<MergeSmem*>(smem);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], o);
    st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], o);
  }
  // packed mode: columns 4..7 hold the residual parts of heads 0..3
  const bool writer = PACK4 ? (tig < 2) : true;
  if (q == 0 && writer) {
    ms.m[warp][2 * tig] = st.m[0];
    ms.m[warp][2 * tig + 1] = st.m[1];
    ms.l[warp][2 * tig] = st.l[0];
    ms.l[warp][2 * tig + 1] = st.l[1];
  }
  const float inv = rotated ? a.inv_pscale : 1.0f / kPScaleBF16;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = 16 * mt + q + 8 * (i >> 1), n = 2 * tig + (i & 1);
      float v = st.acc[mt][i] * inv;
      if (PACK4) v += __shfl_xor_sync(0xffffffffu, v, 2);
      if (writer) ms.acc[warp][n][ch] = v;
    }
  }
  __syncthreads();
  float* part = a.partials + ((size_t)bh * a.n_items + item) * kPartialFloats;
  for (int n = 0; n < a.g; ++n) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ms.m[w][n]);
    float acc = 0.f, l = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = ms.m[w][n];
        const float al = (mw == -INFINITY) ? 0.f : ex2(mw - M);
        acc = fmaf(al, ms.acc[w][n][t], acc);
        l = fmaf(al, ms.l[w][n], l);
      }
    }
    part[16 + n * kD + t] = acc;
    if (t == 0) {
      part[n] = M;
      part[8 + n] = l;
    }
  }
  // ---------------- last block of this (request, KV head) merges all partials
  __shared__ int s_last;
  __syncthreads();
  if (t == 0) {
    __threadfence();
    const int ticket = atomicAdd(&a.counters[bh], 1);
    s_last = (ticket == a.n_items - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  float Mr[kMaxG], Lr[kMaxG], Ar[kMaxG], Mp[kMaxG], Lp[kMaxG], Ap[kMaxG];
#pragma unroll
  for (int n = 0; n < kMaxG; ++n) {
    Mr[n] = Mp[n] = -INFINITY;
    Lr[n] = Lp[n] = Ar[n] = Ap[n] = 0.f;
  }
  for (int x = 0; x < a.n_items; ++x) {
    const float* rec = a.partials + ((size_t)bh * a.n_items + x) * kPartialFloats;
    const bool rot = (MODE == 0) && x < a.n_chunks;
#pragma unroll
    for (int n = 0; n < kMaxG; ++n) {
      if (n >= a.g) break;
      const float m = __ldcg(rec + n);
      if (m == -INFINITY) continue;
      const float l = __ldcg(rec + 8 + n), v = __ldcg(rec + 16 + n * kD + t);
      if (rot) {
        const float Mn = fmaxf(Mr[n], m);
        const float a0 = (Mr[n] == -INFINITY) ? 0.f : ex2(Mr[n] - Mn), a1 = ex2(m - Mn);
        Ar[n] = Ar[n] * a0 + v * a1;
        Lr[n] = Lr[n] * a0 + l * a1;
        Mr[n] = Mn;
      } else {
        const float Mn = fmaxf(Mp[n], m);
        const float a0 = (Mp[n] == -INFINITY) ? 0.f : ex2(Mp[n] - Mn), a1 = ex2(m - Mn);
        Ap[n] = Ap[n] * a0 + v * a1;
        Lp[n] = Lp[n] * a0 + l * a1;
        Mp[n] = Mn;
      }
    }
  }
  float Or[kMaxG];
#pragma unroll
  for (int n = 0; n < kMaxG; ++n) Or[n] = 0.f;
  if (MODE == 0) {
    // rotate the INT2 part back: y = acc P, y = y H / sqrt(d), out = y U_V^T
    float* ys = reinterpret_cast<float*>(smem);  // [8][128]
    float* scratch = ys + kMaxG * kD;
#pragma unroll
    for (int n = 0; n < kMaxG; ++n)
      if (n < a.g) ys[n * kD + t] = Ar[n];
    __syncthreads();
    for (int n = 0; n < a.g; ++n) {
      float v = (a.flags & kRotP) ? ys[n * kD + brev7(t)] : ys[n * kD + t];
      if (a.flags & kRotH) v = fwht128_block(v, scratch) * kInvSqrtD;
      __syncthreads();
      ys[n * kD + t] = v;
      __syncthreads();
    }
#pragma unroll 4
    for (int j = 0; j < kD; ++j) {
      const float u = __ldg(a.U_VT + j * kD + t);
#pragma unroll
      for (int n = 0; n < kMaxG; ++n)
        if (n < a.g) Or[n] = fmaf(ys[n * kD + j], u, Or[n]);
    }
  }
#pragma unroll
  for (int n = 0; n < kMaxG; ++n) {
    if (n >= a.g) break;
    const float M = fmaxf(Mr[n], Mp[n]);
    float o = 0.f;
    if (M != -INFINITY) {
      const float ar = (Mr[n] == -INFINITY) ? 0.f : ex2(Mr[n] - M);
      const float ap = (Mp[n] == -INFINITY) ? 0.f : ex2(Mp[n] - M);
      const float l = ar * Lr[n] + ap * Lp[n];
      o = (ar * Or[n] + ap * Ap[n]) / l;
    }
    a.out[((size_t)b * a.Hq + h * a.g + n) * kD + t] = o;
  }
}

constexpr size_t decode_smem_bytes() {
  return (size_t)kWarps * kStages * kBlockBytes + (size_t)kWarps * kStages * sizeof(uint64_t);
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

DecodePlan plan_decode(int mode, int batch, int Hq, int Hkv, int max_ctx_len, int num_sms) {
  DecodePlan p;
  p.batch = batch;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  int pages;  // paged work per (request, KV head)
  if (mode == 0) {
    const int hist_end = max_ctx_len > kSink + kRecent ? max_ctx_len - kRecent : kSink;
    pages = (hist_end + kPage - 1) / kPage - 1;
  } else {
    pages = (max_ctx_len + kPage - 1) / kPage;
  }
  if (pages < 0) pages = 0;
  const long long total = (long long)batch * Hkv * pages;
  const long long target = 6LL * (num_sms > 0 ? num_sms : 148);
  long long C = (total + target - 1) / target;
  const int cmin = mode == 0 ? 4 : 1;
  if (C < cmin) C = cmin;
  if (C > 64) C = 64;
  p.chunk_pages = (int)C;
  p.n_chunks = pages > 0 ? (int)((pages + C - 1) / C) : 0;
  p.n_items = mode == 0 ? p.n_chunks + 5 : (p.n_chunks > 0 ? p.n_chunks : 1);
  const size_t bh = (size_t)batch * Hkv;
  size_t off = 0;
  p.off_counters = off;
  off = align256(off + bh * sizeof(int));
  p.off_qfrag = off;
  off = align256(off + bh * kQFragWords * sizeof(uint32_t));
  p.off_qplain = off;
  off = align256(off + bh * kQFragWords * sizeof(uint32_t));
  p.off_qconst = off;
  off = align256(off + bh * kQConstFloats * sizeof(float));
  p.off_partials = off;
  off = align256(off + bh * (size_t)p.n_items * kPartialFloats * sizeof(float));
  p.total = off;
  return p;
}

cudaError_t launch_decode(const DecodeLaunch& d, cudaStream_t stream) {
  const DecodePlan& p = d.plan;
  if (p.batch == 0) return cudaSuccess;
  uint8_t* ws = d.workspace;
  PrepArgs pa;
  pa.q = d.q;
  pa.U_K = d.rot.U_K;
  pa.flags = d.rot.flags;
  pa.sm_scale = d.sm_scale;
  pa.Hq = p.Hq;
  pa.Hkv = p.Hkv;
  pa.g = p.g;
  pa.qfrag = reinterpret_cast<uint32_t*>(ws + p.off_qfrag);
  pa.qplain = reinterpret_cast<uint32_t*>(ws + p.off_qplain);
  pa.qconst = reinterpret_cast<float*>(ws + p.off_qconst);
  pa.counters = reinterpret_cast<int*>(ws + p.off_counters);
  prep_kernel<<<dim3(p.Hkv, p.batch), 128, 0, stream>>>(pa);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  DecodeArgs a;
  a.mode = d.mode;
  a.c = d.c;
  a.kb_pages = d.kb_pages;
  a.vb_pages = d.vb_pages;
  a.ctx_len = d.ctx_len;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.g = p.g;
  a.n_items = p.n_items;
  a.n_chunks = p.n_chunks;
  a.chunk_pages = p.chunk_pages;
  a.qfrag = pa.qfrag;
  a.qplain = pa.qplain;
  a.qconst = pa.qconst;
  a.partials = reinterpret_cast<float*>(ws + p.off_partials);
  a.counters = pa.counters;
  a.U_VT = d.rot.U_VT;
  a.flags = d.rot.flags;
  {
    // largest V scale the layer can store: fp16(min(absmax, tau_v) / 1.5) <= 65504
    const float smax = std::isfinite(d.rot.tau_v) ? fminf(65504.f, d.rot.tau_v / 1.5f * 1.001f) : 65504.f;
    int k = (int)floorf(log2f(60000.f / (16.f * smax)));
    k = k < -20 ? -20 : (k > 20 ? 20 : k);
    a.pscale = ldexpf(1.f, k);
    a.inv_pscale = ldexpf(1.f, -k);
  }
  a.out = d.out;
  a.err = d.err;
  const size_t smem = decode_smem_bytes();
  const dim3 grid(p.n_items, p.Hkv, p.batch);
  const bool pack4 = p.g <= 4;
  void (*kern)(DecodeArgs) = d.mode == 0 ? (pack4 ? decode_kernel<0, true> : decode_kernel<0, false>)
                                         : (pack4 ? decode_kernel<1, true> : decode_kernel<1, false>);
  static bool attr_done[4] = {false, false, false, false};
  const int which = 2 * d.mode + (pack4 ? 1 : 0);
  if (!attr_done[which]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done[which] = true;
  }
  kern<<<grid, 128, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace oscar
