// OSCAR decode attention over the mixed-precision paged cache (sm_103a).
//
// gist.science "Resumen Técnico: OSCAR ...", §2.2 B: a fused kernel unpacks,
// de-quantises, undoes the rotation and computes attention over the INT2
// history, paged and prefix-cache compatible, with no extra memory traffic.
// ainsights.it "OSCAR: Come Together AI ...", "Architettura del Sistema di
// Serving e Layout di Memoria": sink and recent tokens stay BF16.
//
// Design (GB300):
//  * decode_step_kernel: one launch per layer step, one 16-warp block per
//    (work item, KV head, request).  Every block rotates its request's
//    queries, q' = q R_K (R_K rows in registers, or without U the
//    Walsh-Hadamard butterfly and the bit-reversal index map), times
//    sm_scale * log2(e) and a power-of-two normalisation, as fp16 value +
//    residual tensor-core fragments; the block whose pages hold the evicted
//    ring row appends K and V.  prep_kernel, append_one_kernel and
//    decode_kernel run the same steps as separate launches.  Work items are
//    ranges of INT2 history pages (rotated basis) from a wave cost model; two
//    warps of some items also take the BF16 sink/recent tiles (original
//    basis).  Each warp streams its pages through a private 3-stage ring of
//    bulk copies (one 4608-byte copy per page), turns each pair of 2-bit
//    codes into the exact fp16 levels (c - 1.5) with one LOP3 and one HFMA2,
//    and runs QK^T and PV on mma.sync m16n8k16 with an online softmax in the
//    log2 domain.  The block merges its warps, applies R_V^T to the INT2 part
//    and writes one record; an acq_rel ticket picks the last block of each
//    (request, KV head), which merges the records.  No block waits on another.
//
// Precision: q and the softmax weights times the V scales enter the MMAs as
// fp16 value + fp16 residual (~22 significant bits).  With at most 4 query
// heads per KV head the residual rides in the MMA's otherwise unused N
// columns 4..7 (no extra MMAs); with 5..8 heads it takes a second MMA.

#include <cmath>

#include "oscar_device.cuh"
#include "oscar_internal.h"
#include "oscar_quant.cuh"

namespace oscar {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 3;
// The PV B operand is p * s * 2^k (INT2 history, s = V scale) or p * 2^k (BF16
// tiles), with p <= 2^kLazy.  k is the largest power of two that keeps it
// below 60000 for the layer's largest possible scale, so small weights stay
// clear of the fp16 subnormal range.
constexpr float kLazy = 4.0f;           // rescale only when the max grows by more than 2^4
constexpr float kPScaleBF16 = 2048.0f;  // 2^4 * 2048 < 60000 (log2 = 11)
constexpr int kMaxChunks = 256;        // work items per (request, KV head)
constexpr int kBf16Tiles = (kSink + kRecent) / 16;  // 16-token BF16 tiles per request
constexpr int kStash = kD + 4;
constexpr int kPrefetchPages = 1;        // pages per warp pulled into L2 before the dependency wait
constexpr int kBf16Slots = 2;            // warps per work item that attend BF16 tiles (mixed cache)
// dynamic shared memory: kStages bulk-copy stages per warp, their mbarriers (+1
// for the final merge), then the BF16 warps' finished states
constexpr size_t kSlotsOffset = ((size_t)kWarps * kStages * kBlockBytes + (size_t)(kWarps * (kStages + 1) + 1) * 8 + 15) / 16 * 16;
// each warp's rows of R_V^T, copied into its last stage once that is free
constexpr int kRvRows = kD / kWarps;
constexpr unsigned kRvBytes = kRvRows * kD * 4;

// Exact fp16 pair of the levels (c - 1.5) of the codes at index r (0..7) of
// both 16-bit halves of a code word.  One LOP3 puts the code into the low
// mantissa of the fp16 1024 ((w & mask) | 0x6400: the value 1024 + c 4^r'),
// one HFMA2 maps it to (1024 + c 4^r') 4^-r' - (1024 4^-r' + 1.5) = c - 1.5.
// r' is the code's 2-bit position in the source word: indices 1..4 come
// from w (r' = r); indices 0 and 5..7 from w with the two bytes of each half
// swapped (r' = 4 and 1..3; at r' = 0 the offset 1025.5 would not be an
// fp16).  The levels are normal fp16 numbers: tensor-core products of
// subnormal operands lose precision.
__device__ __forceinline__ uint32_t swap_half_bytes(uint32_t x) {
  uint32_t y;
  asm("prmt.b32 %0, %1, 0, 0x2301;" : "=r"(y) : "r"(x));
  return y;
}

struct CodeWord {
  uint32_t w, sw;  // w, and w with the bytes of each 16-bit half swapped
  __device__ __forceinline__ explicit CodeWord(uint32_t x) : w(x), sw(swap_half_bytes(x)) {}
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
  constexpr int rp = R == 0 ? 4 : (R < 5 ? R : R - 4);
  // fp16 constants 4^-r' and -(1024 4^-r' + 1.5) for r' = 1..4, in both halves
  constexpr uint32_t kScale = rp == 1 ? 0x34003400u : rp == 2 ? 0x2C002C00u : rp == 3 ? 0x24002400u : 0x1C001C00u;
  constexpr uint32_t kBias = rp == 1 ? 0xDC06DC06u : rp == 2 ? 0xD418D418u : rp == 3 ? 0xCC60CC60u : 0xC580C580u;
  const uint32_t src = (R == 0 || R >= 5) ? cw.sw : cw.w;
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
  const float* R_K;
  float sm_scale;
  int Hq, Hkv, g;
  uint32_t rot_flags;  // the layer's factors: without U, q R_K runs as the butterfly
  uint32_t* qfrag;
  uint32_t* qplain;
  float* qconst;
  int* counters;
  int nb, per_block;  // rows (request or query) to rotate; rows per block of prep_kernel
};

// ------------------------------------------------------------------ prep
// q' = q R_K for the g query heads of (request b, KV head h), by the 128
// threads t = 0..127 of a named-barrier group `bar`; R_K may be in shared or
// global memory.
//
// Fragment words per (request, KV head): [32 lanes][32].  The MMA B column of
// lane L is n = L / 4.  With g <= 4 ("packed"), column n carries head n / 2
// and part n % 2 (0: fp16 value, 1: fp16 residual) in words 0..15, so that
// the accumulator lane holding columns 2 h and 2 h + 1 holds all of head h;
// with g > 4 column n is head n, words 0..15 hold the values and 16..31 the
// residuals.
constexpr int kPrepThreads = 512;  // channel t = u % 128, row quarter u / 128 of R_K

struct PrepSmem {
  __align__(16) float xs[kMaxG][kD];
  float zq[4][kMaxG][kD];  // partial products over the four quarters of the rows of R_K
  float qr[kMaxG][kD];     // q' times c, the partials summed (in quarter order)
  float red[kPrepThreads / 32];
};

// Partial q_n R_K over rows [32 kq, 32 kq + 32), channel t, for the first G
// heads of sm.xs, into sm.zq[kq] (two sums per head, so that the
// shared-memory loads and the multiply-adds overlap).  rk(ii) = R_K[32 kq + ii][t].
template <int G, typename RowOf>
__device__ __forceinline__ void rotate_heads(PrepSmem& sm, RowOf rk, int t, int kq) {
  float za[G], zb[G];
#pragma unroll
  for (int n = 0; n < G; ++n) za[n] = zb[n] = 0.f;
#pragma unroll
  for (int ii = 0; ii < 32; ii += 4) {
    const int i = 32 * kq + ii;
    const float r0 = rk(ii), r1 = rk(ii + 1), r2 = rk(ii + 2), r3 = rk(ii + 3);
#pragma unroll
    for (int n = 0; n < G; ++n) {
      const float4 x = *reinterpret_cast<const float4*>(&sm.xs[n][i]);
      za[n] = fmaf(x.y, r1, fmaf(x.x, r0, za[n]));
      zb[n] = fmaf(x.w, r3, fmaf(x.z, r2, zb[n]));
    }
  }
#pragma unroll
  for (int n = 0; n < G; ++n) sm.zq[kq][n][t] = za[n] + zb[n];
}

// q' = q R_K and the fragments of q' and q for (request b, KV head h), by
// the kPrepThreads threads u of a group synchronised by named barrier `bar`.
// rk(ii) = R_K[32 (u / 128) + ii][u % 128]; qbits(n) = the bf16 bits of
// q[b][h g + n][u % 128] for n = u / 128 and u / 128 + 4 below g.  Outputs:
// the history and BF16 fragment words (kQFragWords each) and the constants
// (kQConstFloats).
template <typename RowOf, typename QOf, typename Mid>
__device__ __forceinline__ void prep_body(const PrepArgs& a, int b, int h, int u, RowOf rk, QOf qbits, PrepSmem& sm,
                                          int bar, uint32_t* qf, uint32_t* qpl, float* qc, Mid mid) {
  const int t = u & 127, kq = u >> 7, lane = u & 31, warp = u >> 5;
  const int g = a.g;
  const bool packed = g <= 4;
  const float c = a.sm_scale * kLog2e;
  // heads g .. G - 1 of the padded set are zero (G = 4 when g <= 4, else 8);
  // the sum of squares over the heads: sqrt of it bounds every |q| and, the
  // rotation keeping lengths, every |q'|
  const int G = packed ? 4 : kMaxG;
  float ss = 0.f;
  for (int n = kq; n < G; n += 4) {
    const float x = n < g ? bf16_bits_to_float(qbits(n)) : 0.f;
    sm.xs[n][t] = x;
    ss = fmaf(x, x, ss);
  }
  ss = warp_sum(ss);
  constexpr int kW = kPrepThreads / 32;
  if (lane == 0) sm.red[warp] = ss;
  group_sync(bar, kPrepThreads);
  mid();  // the caller's work that may wait on loads issued before (every thread)
  const bool dense = (a.rot_flags & kRotU) != 0;
  if (dense) {
    if (packed)
      rotate_heads<4>(sm, rk, t, kq);
    else
      rotate_heads<kMaxG>(sm, rk, t, kq);
    group_sync(bar, kPrepThreads);
  }
  // one power-of-two normalisation for q' and q: their magnitudes times 2^-E stay below 2^10
  float S = 0.f;
#pragma unroll
  for (int w = 0; w < kW; ++w) S += sm.red[w];
  int er = 0;
  const float bound = sqrtf(S) * c;
  if (bound > 0.f) {
    frexpf(bound, &er);
    er -= 10;
  }
  const float sr = ldexpf(1.f, -er);
  // q' (scaled by c) of head n, channel j, from the four row-quarter partial
  // products, summed once per (head, channel) before the fragments are built;
  // without U, warp n applies H to head n as the butterfly and P as an index map
  if (dense) {
    for (int e = u; e < G * kD; e += kPrepThreads) {
      const int n = e >> 7, j = e & (kD - 1);
      sm.qr[n][j] = (((sm.zq[0][n][j] + sm.zq[1][n][j]) + sm.zq[2][n][j]) + sm.zq[3][n][j]) * c;
    }
  } else if (warp < G) {
    float v[4];
    const float4 xv = *reinterpret_cast<const float4*>(&sm.xs[warp][4 * lane]);
    v[0] = xv.x;
    v[1] = xv.y;
    v[2] = xv.z;
    v[3] = xv.w;
    float f = c;
    if (a.rot_flags & kRotH) {
      hadamard128(v, lane);
      f = kInvSqrt128 * c;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) sm.qr[warp][(a.rot_flags & kRotP) ? brev7(4 * lane + e) : 4 * lane + e] = v[e] * f;
  }
  group_sync(bar, kPrepThreads);
  auto qrot = [&](int n, int j) { return sm.qr[n][j]; };
  // QK B fragments over the INT2 history: MMA i reads the code pairs at
  // in-half position 2 R, R = 2 (i % 4) (b0) and R + 1 (b1), of word i / 4
  // (ks = 2 (i / 4) + (i % 4) % 2, byte parity pb = (i % 4) / 2), i.e.
  // channels 32 ks + 16 bs + 4 tig + pb and + 2 for b_bs.
  // BF16 segment: MMA ks = i takes channels 32 tig + 4 ks + {0,1} (b0) and {2,3} (b1).
  for (int e = u; e < kQFragWords; e += kPrepThreads) {
    const int L = e >> 5, w = e & 31, set = w >> 4, ww = w & 15, i = ww >> 1, bs = ww & 1;
    const int n = L >> 2, tig = L & 3;
    const int head = packed ? (n >> 1) : n;
    const int part = packed ? (n & 1) : set;
    uint32_t vr = 0, vp = 0;
    if (head < g && !(packed && set == 1)) {
      // MMA i of the history: group i / 4, channel step ks, byte parity pb (see the K layout)
      const int ii = i & 3, ks = 2 * (i >> 2) + (ii & 1), pb = ii >> 1;
      const int ch = 32 * ks + 16 * bs + 4 * tig + pb;
      vr = pack_f16x2(split_part(qrot(head, ch) * sr, part), split_part(qrot(head, ch + 2) * sr, part));
      const int cp = 32 * tig + 4 * i + 2 * bs;
      vp = pack_f16x2(split_part(sm.xs[head][cp] * c * sr, part), split_part(sm.xs[head][cp + 1] * c * sr, part));
    }
    // 16-byte chunk c of lane L's row stored at chunk c ^ (L % 8): the readers'
    // 16-byte loads of one chunk index spread over all banks
    const int es = (e & ~31) | ((((e >> 2) & 7) ^ (L & 7)) << 2) | (e & 3);
    qf[es] = vr;
    qpl[es] = vp;
  }
  if (u == 0) {
    qc[16] = ldexpf(1.f, er);
    qc[17] = ldexpf(1.f, er);
  }
}

// grid (Hkv, ceil(nb / per_block)), kPrepThreads threads: a block rotates rows
// per_block y .. of KV head x with its rows of R_K in registers (a constant of
// the layer, loaded before the dependency wait)
__global__ void __launch_bounds__(kPrepThreads, 1) prep_kernel(PrepArgs a) {
  __shared__ PrepSmem sm;
  const int h = blockIdx.x, u = threadIdx.x;
  float rk[32];  // R_K[32 (u / 128) + ii][u % 128]
  {
    const float* RK = a.R_K + (size_t)32 * (u >> 7) * kD + (u & 127);
#pragma unroll
    for (int ii = 0; ii < 32; ++ii) rk[ii] = __ldg(RK + ii * kD);
  }
  griddep_wait();
  griddep_launch_dependents();
  const int b0 = blockIdx.y * a.per_block, b1 = min(b0 + a.per_block, a.nb);
  for (int b = b0; b < b1; ++b) {
    const int bh = b * a.Hkv + h;
    if (u == 0) a.counters[bh] = 0;
    const uint16_t* qrow = a.q + ((size_t)b * a.Hq + h * a.g) * kD + (u & 127);
    prep_body(a, b, h, u, [&](int ii) { return rk[ii]; }, [&](int n) { return qrow[(size_t)n * kD]; }, sm, 1,
              a.qfrag + (size_t)bh * kQFragWords, a.qplain + (size_t)bh * kQFragWords,
              a.qconst + (size_t)bh * kQConstFloats, [] {});
    group_sync(1, kPrepThreads);  // the next row reuses the scratch
  }
}

// rows per prep block: about two blocks per SM
int prep_rows_per_block(int nb, int Hkv, int num_sms) {
  const long long slots = 2LL * (num_sms > 0 ? num_sms : 148);
  const long long per = ((long long)nb * Hkv + slots - 1) / slots;
  return (int)(per < 1 ? 1 : per);
}

// ------------------------------------------------------------------ decode
struct DecodeArgs {
  int mode;
  CacheRefs c;
  const uint16_t* kb_pages;
  const uint16_t* vb_pages;
  const int32_t* ctx_len;
  int Hq, Hkv, g;
  int n_items, n_chunks, chunk_pages, tiles_per_item, rec_floats;
  const uint32_t* qfrag;
  const uint32_t* qplain;
  const float* qconst;
  float* partials;
  int* counters;
  const float* R_VT;
  float pscale, inv_pscale;
  float* out;
  unsigned* err;
  const int32_t* limit;  // extend attention: per-request causal limit (nullptr otherwise)
  const uint16_t* q;     // the queries as they came in (bf16; the BF16-cache comparator reads them)
  float sm_scale;
  uint32_t rot_flags;    // the layer's factors: without U, acc R_V^T runs as an index map and the butterfly
};

// The fused decode step's other inputs: the append of this step's token and
// the q rotation.
struct StepArgs {
  AppendLaunch ap;
  PrepArgs pr;
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

// Packed mode: the lane's two accumulator columns are one head's value and
// residual parts, so a single running maximum covers all its accumulators.
__device__ __forceinline__ void online_max1(WarpState& st, float mx) {
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (__any_sync(0xffffffffu, mx > st.m[0] + kLazy)) {
    const float nm = fmaxf(st.m[0], mx);
    const float al = (nm == -INFINITY) ? 1.f : ex2(st.m[0] - nm);
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) st.acc[i][k] *= al;
    st.l[0] *= al;
    st.m[0] = nm;
  }
}

// x as an fp16 pair (value, residual): the value in the low half
__device__ __forceinline__ uint32_t value_residual(float x) {
  const float hi = __half2float(__float2half_rn(x));
  return pack_f16x2(x, x - hi);
}

// Fold one partial softmax state (m, l, acc slice) into a running one.
__device__ __forceinline__ void merge_record(float& m, float& l, float4& acc, float mx, float lx, float4 v) {
  const float M = fmaxf(m, mx);
  if (M == -INFINITY) return;
  const float so = ex2(m - M), sn = ex2(mx - M);  // an empty state (-inf) gets weight 0
  acc.x = fmaf(acc.x, so, v.x * sn);
  acc.y = fmaf(acc.y, so, v.y * sn);
  acc.z = fmaf(acc.z, so, v.z * sn);
  acc.w = fmaf(acc.w, so, v.w * sn);
  l = fmaf(l, so, lx * sn);
  m = M;
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

// The rounding residuals of an fp16 pair h = fp16(x0, x1), negated: (h0 - x0,
// h1 - x1) as an fp16 pair, by two mixed-precision subtractions (exact in
// fp32) and one pack; the MMA that reads them negates its A operand.
__device__ __forceinline__ uint32_t f16x2_negres(uint32_t h, float x0, float x1) {
  uint32_t r;
  asm("{\n .reg .b16 lo, hi;\n .reg .f32 r0, r1;\n mov.b32 {lo, hi}, %1;\n"
      " sub.rn.f32.f16 r0, lo, %2;\n sub.rn.f32.f16 r1, hi, %3;\n"
      " cvt.rn.f16x2.f32 %0, r1, r0;\n}"
      : "=r"(r)
      : "r"(h), "f"(x0), "f"(x1));
  return r;
}

// x as an fp16 pair (value, minus the residual): the value in the low half.
// One rounding, one mixed-precision subtraction (h - x is exact in fp32)
// and one pack; the consumer subtracts the residual column.
__device__ __forceinline__ uint32_t value_negres(float x) {
  unsigned short h;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(x));
  float nr;
  asm("sub.rn.f32.f16 %0, %1, %2;" : "=f"(nr) : "h"(h), "f"(x));
  uint32_t p;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(p) : "f"(nr), "f"(x));
  return p;
}

// Q.K of one 16-token tile T of a staged INT2 page: the lane's raw logits
// (packed: z[0], z[1] of head lane % 4 for tokens q, q + 8; unpacked:
// z[0..3] = (q, head 2 tig), (q, 2 tig + 1), (q + 8, 2 tig), (q + 8, 2 tig + 1)),
// sum over groups of s_K sum_j (c - 1.5) q'_j in the fragments' scale.  The
// codes enter as exact fp16 levels c - 1.5 (code_level): the operand of the
// tensor cores' products stays normal and zero-mean, which keeps the logits
// at fp32 accuracy.  Two independent chains of four MMAs (one per group).
template <bool PACK4>
__device__ __forceinline__ void qk_tile(const uint8_t* __restrict__ blk, int T, const uint32_t* qf, float (&z)[4],
                                        int lane) {
  const int q = lane >> 2;
  const uint4 kw = *reinterpret_cast<const uint4*>(blk + kKCodes + 512 * T + 16 * lane);
  const uint32_t ksa = *reinterpret_cast<const uint32_t*>(blk + kKScales + 4 * (16 * T + q));
  const uint32_t ksb = *reinterpret_cast<const uint32_t*>(blk + kKScales + 4 * (16 * T + q + 8));
  float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
  const CodeWord x0(kw.x), y0(kw.z), x1(kw.y), y1(kw.w);  // group 0 (token q, q + 8), group 1
#define OSCAR_QK2(I, R)                                                                                        \
  do {                                                                                                         \
    const uint32_t a0 = code_level<R>(x0), a1 = code_level<R>(y0), a2 = code_level<R + 1>(x0),                 \
                   a3 = code_level<R + 1>(y0);                                                                 \
    const uint32_t e0 = code_level<R>(x1), e1 = code_level<R>(y1), e2 = code_level<R + 1>(x1),                 \
                   e3 = code_level<R + 1>(y1);                                                                 \
    mma_f16(d0, a0, a1, a2, a3, qf[2 * I], qf[2 * I + 1]);                                                     \
    mma_f16(d1, e0, e1, e2, e3, qf[8 + 2 * I], qf[9 + 2 * I]);                                                 \
    if (!PACK4) {                                                                                              \
      mma_f16(d0, a0, a1, a2, a3, qf[16 + 2 * I], qf[17 + 2 * I]);                                             \
      mma_f16(d1, e0, e1, e2, e3, qf[24 + 2 * I], qf[25 + 2 * I]);                                             \
    }                                                                                                          \
  } while (0)
  OSCAR_QK2(0, 0);
  OSCAR_QK2(1, 2);
  OSCAR_QK2(2, 4);
  OSCAR_QK2(3, 6);
#undef OSCAR_QK2
  const float2 sa = half2_bits_to_float2(ksa), sb = half2_bits_to_float2(ksb);
  if (PACK4) {  // columns 2 h, 2 h + 1: value and residual parts of head h = lane % 4
    z[0] = fmaf(d0[0] + d0[1], sa.x, (d1[0] + d1[1]) * sa.y);
    z[1] = fmaf(d0[2] + d0[3], sb.x, (d1[2] + d1[3]) * sb.y);
    z[2] = z[3] = 0.f;
  } else {
    z[0] = fmaf(d0[0], sa.x, d1[0] * sa.y);
    z[1] = fmaf(d0[1], sa.x, d1[1] * sa.y);
    z[2] = fmaf(d0[2], sb.x, d1[2] * sb.y);
    z[3] = fmaf(d0[3], sb.x, d1[3] * sb.y);
  }
}

// Online softmax over N tiles' raw logits z (scaled by E into the log2
// domain): p = 2^(z E - m + kp).  The running maximum m is lazy: a warp
// rescales its state only when a logit passes m by more than kLazy (then m
// becomes the exact maximum so far), so p <= 2^(kLazy + kp).  MASKED: a
// logit of -inf (a row past the end) gives p = 0.
template <bool PACK4, bool MASKED, int N>
__device__ __forceinline__ void softmax_weights(const float (&z)[N][4], float E, float kp, WarpState& st,
                                                float (&p)[N][4]) {
  constexpr int K = PACK4 ? 2 : 4;
  const float thr = kp + kLazy;
  auto arg = [&](float zz, float m) {
    const float e = fmaf(zz, E, kp - m);
    return MASKED ? (zz == -INFINITY ? -INFINITY : e) : e;
  };
  bool need = false;
#pragma unroll
  for (int i = 0; i < N; ++i)
#pragma unroll
    for (int k = 0; k < K; ++k) {
      p[i][k] = arg(z[i][k], st.m[PACK4 ? 0 : (k & 1)]);
      need |= p[i][k] > thr;
    }
  if (__any_sync(0xffffffffu, need)) {
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < N; ++i)
#pragma unroll
      for (int k = 0; k < K; ++k) {
        if (PACK4 || (k & 1) == 0)
          mx0 = fmaxf(mx0, z[i][k] * E);
        else
          mx1 = fmaxf(mx1, z[i][k] * E);
      }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      if (!PACK4) mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float n0 = fmaxf(st.m[0], mx0), n1 = PACK4 ? n0 : fmaxf(st.m[1], mx1);
    const float a0 = (n0 == -INFINITY) ? 1.f : ex2(st.m[0] - n0);
    const float a1 = PACK4 ? a0 : ((n1 == -INFINITY) ? 1.f : ex2(st.m[1] - n1));
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
#pragma unroll
    for (int i = 0; i < N; ++i)
#pragma unroll
      for (int k = 0; k < K; ++k) p[i][k] = arg(z[i][k], st.m[PACK4 ? 0 : (k & 1)]);
  }
#pragma unroll
  for (int i = 0; i < N; ++i)
#pragma unroll
    for (int k = 0; k < K; ++k) p[i][k] = ex2(p[i][k]);
}

// P.V of one tile T with the weights p of the lane's rows (as qk_tile's z):
// B = p s_V 2^kp (value + residual) against the V codes as exact fp16
// levels c - 1.5 (code_level).  MASKED: rows at or past nv have p = 0 and
// their scales are ignored.
template <bool PACK4, bool MASKED>
__device__ __forceinline__ void pv_tile(const uint8_t* __restrict__ blk, int T, int nv, const float (&p)[4],
                                        WarpState& st, int lane) {
  const int q = lane >> 2;
  const uint4 vw = *reinterpret_cast<const uint4*>(blk + kVCodes + 512 * T + 16 * lane);
  float2 wa = half2_bits_to_float2(*reinterpret_cast<const uint32_t*>(blk + kVScales + 4 * (16 * T + q)));
  float2 wb = half2_bits_to_float2(*reinterpret_cast<const uint32_t*>(blk + kVScales + 4 * (16 * T + q + 8)));
  if (MASKED) {  // rows past the history end may hold anything
    const bool va = q < nv, vb = q + 8 < nv;
    wa.x = va ? wa.x : 0.f;
    wa.y = va ? wa.y : 0.f;
    wb.x = vb ? wb.x : 0.f;
    wb.y = vb ? wb.y : 0.f;
  }
  const CodeWord w0(vw.x), w1(vw.y), w2(vw.z), w3(vw.w);
  if constexpr (PACK4) {
    st.l[0] += p[0] + p[1];
    const uint32_t b00 = movmatrix_trans(value_negres(p[0] * wa.x));
    const uint32_t b01 = movmatrix_trans(value_negres(p[1] * wb.x));
    const uint32_t b10 = movmatrix_trans(value_negres(p[0] * wa.y));
    const uint32_t b11 = movmatrix_trans(value_negres(p[1] * wb.y));
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
    return;
  }
  st.l[0] += p[0] + p[2];
  st.l[1] += p[1] + p[3];
  uint32_t h00, l00, h01, l01, h10, l10, h11, l11;
  split_pair(p[0] * wa.x, p[1] * wa.x, h00, l00);
  split_pair(p[2] * wb.x, p[3] * wb.x, h01, l01);
  split_pair(p[0] * wa.y, p[1] * wa.y, h10, l10);
  split_pair(p[2] * wb.y, p[3] * wb.y, h11, l11);
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

// One whole, full INT2 page (64 valid rows): Q.K of its four tiles (eight
// independent MMA chains), one softmax update, P.V of the four tiles.  The
// weights come out scaled by 2^kp (undone by the caller).
template <bool PACK4>
__device__ __forceinline__ void int2_page_full(const uint8_t* __restrict__ blk, const uint32_t* qf, float E,
                                               float kp, WarpState& st, int lane) {
  // g > 4: two tiles at a time (twice the logits per tile, and twice the q' fragments)
  constexpr int NT = PACK4 ? 4 : 2;
#pragma unroll
  for (int T0 = 0; T0 < 4; T0 += NT) {
    float z[NT][4], p[NT][4];
#pragma unroll
    for (int T = 0; T < NT; ++T) qk_tile<PACK4>(blk, T0 + T, qf, z[T], lane);
    softmax_weights<PACK4, false, NT>(z, E, kp, st, p);
#pragma unroll
    for (int T = 0; T < NT; ++T) pv_tile<PACK4, false>(blk, T0 + T, 16, p[T], st, lane);
  }
}

// One 16-token tile T with rows [0, nv) valid (a page's last tile, or a
// tile of the left-over pages dealt one tile per warp).
template <bool PACK4>
__device__ __forceinline__ void int2_tile(const uint8_t* __restrict__ blk, int T, int nv, const uint32_t* qf,
                                          float E, float kp, WarpState& st, int lane) {
  const int q = lane >> 2;
  float z[1][4], p[1][4];
  qk_tile<PACK4>(blk, T, qf, z[0], lane);
  if (PACK4) {
    z[0][0] = q < nv ? z[0][0] : -INFINITY;
    z[0][1] = q + 8 < nv ? z[0][1] : -INFINITY;
  } else {
    z[0][0] = q < nv ? z[0][0] : -INFINITY;
    z[0][1] = q < nv ? z[0][1] : -INFINITY;
    z[0][2] = q + 8 < nv ? z[0][2] : -INFINITY;
    z[0][3] = q + 8 < nv ? z[0][3] : -INFINITY;
  }
  softmax_weights<PACK4, true, 1>(z, E, kp, st, p);
  pv_tile<PACK4, true>(blk, T, nv, p[0], st, lane);
}

// A BF16 tile staged in shared memory (the chunk kernel): K as 16 rows of 16
// 16-byte chunks, chunk c of row r at r * 16 + xt_kchunk(c, r); V as 16 rows of
// 64 words, word w of row r at r * 64 + xt_vword(w, r).  The swizzles keep the
// tile's MMA fragment loads free of bank conflicts.
__device__ __forceinline__ int xt_kchunk(int c, int r) { return c ^ ((c >> 3) << 1) ^ (r & 1); }
__device__ __forceinline__ int xt_vword(int w, int r) { return w ^ ((r & 7) << 2); }

// One 16-token BF16 tile (rows of K and V in global memory, original basis).
// rows: bit r set when row r of the tile is attended.
// SUB: row `sub` of the tile (-1: none) is read from knew / vnew instead.
// SMEM: Kt and Vt are a tile staged in shared memory (Kt2, Vt2, split unused).
template <bool PACK4, bool SUB = false, bool SMEM = false>
__device__ __forceinline__ void bf16_tile(const uint16_t* __restrict__ Kt, const uint16_t* __restrict__ Vt,
                                          const uint16_t* __restrict__ Kt2, const uint16_t* __restrict__ Vt2,
                                          int split, uint32_t rows, const uint32_t* qpf, float scaleEp,
                                          WarpState& st, int lane, int sub = -1, const uint16_t* knew = nullptr,
                                          const uint16_t* vnew = nullptr) {
  const int q = lane >> 2, tig = lane & 3;
  const bool va = (rows >> q) & 1u, vb = (rows >> (q + 8)) & 1u;
  // row r of the tile: (r < split ? Kt : Kt2) + r * 128 (two runs of positions in a paged recent window)
  const uint16_t* Ka = q < split ? Kt : Kt2;
  const uint16_t* Kb = q + 8 < split ? Kt : Kt2;
  const uint16_t* Va = q < split ? Vt : Vt2;
  const uint16_t* Vb = q + 8 < split ? Vt : Vt2;
  const uint16_t* krow_a = SUB && q == sub ? knew : Ka + q * kD;
  const uint16_t* krow_b = SUB && q + 8 == sub ? knew : Kb + (q + 8) * kD;
  uint32_t ka[16], kb[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4* ks = reinterpret_cast<const uint4*>(Kt);  // SMEM: chunks 4 tig + k of rows q and q + 8
    uint4 u;
    if constexpr (SMEM)
      u = va ? ks[q * 16 + xt_kchunk(4 * tig + k, q)] : make_uint4(0, 0, 0, 0);
    else
      u = va ? __ldg(reinterpret_cast<const uint4*>(krow_a + 32 * tig) + k) : make_uint4(0, 0, 0, 0);
    ka[4 * k + 0] = bf16x2_to_f16x2(u.x);
    ka[4 * k + 1] = bf16x2_to_f16x2(u.y);
    ka[4 * k + 2] = bf16x2_to_f16x2(u.z);
    ka[4 * k + 3] = bf16x2_to_f16x2(u.w);
    if constexpr (SMEM)
      u = vb ? ks[(q + 8) * 16 + xt_kchunk(4 * tig + k, q + 8)] : make_uint4(0, 0, 0, 0);
    else
      u = vb ? __ldg(reinterpret_cast<const uint4*>(krow_b + 32 * tig) + k) : make_uint4(0, 0, 0, 0);
    kb[4 * k + 0] = bf16x2_to_f16x2(u.x);
    kb[4 * k + 1] = bf16x2_to_f16x2(u.y);
    kb[4 * k + 2] = bf16x2_to_f16x2(u.z);
    kb[4 * k + 3] = bf16x2_to_f16x2(u.w);
  }
  float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    mma_f16(d, ka[2 * ks], kb[2 * ks], ka[2 * ks + 1], kb[2 * ks + 1], qpf[2 * ks], qpf[2 * ks + 1]);
    if (!PACK4) mma_f16(d, ka[2 * ks], kb[2 * ks], ka[2 * ks + 1], kb[2 * ks + 1], qpf[16 + 2 * ks], qpf[17 + 2 * ks]);
  }
  uint32_t b0h, b0l, b1h, b1l;
  if constexpr (PACK4) {  // columns 2 h, 2 h + 1: value and residual parts of head h = lane % 4
    const float lq = va ? (d[0] + d[1]) * scaleEp : -INFINITY;
    const float lq8 = vb ? (d[2] + d[3]) * scaleEp : -INFINITY;
    online_max1(st, fmaxf(lq, lq8));
    // weights scaled by 2^11 (kPScaleBF16) through the exponent
    const float ms = st.m[0] - 11.f;
    const float pq = ex2(lq - ms), pq8 = ex2(lq8 - ms);
    st.l[0] += pq + pq8;
    b0h = movmatrix_trans(value_residual(pq));
    b1h = movmatrix_trans(value_residual(pq8));
    b0l = b1l = 0u;
  } else {
  float l0 = d[0] * scaleEp, l1 = d[1] * scaleEp, l2 = d[2] * scaleEp, l3 = d[3] * scaleEp;
  l0 = va ? l0 : -INFINITY;
  l1 = va ? l1 : -INFINITY;
  l2 = vb ? l2 : -INFINITY;
  l3 = vb ? l3 : -INFINITY;
  online_max(st, fmaxf(l0, l2), fmaxf(l1, l3));
  // weights scaled by 2^11 (kPScaleBF16) through the exponent
  const float ms0 = st.m[0] - 11.f, ms1 = st.m[1] - 11.f;
  const float p0 = ex2(l0 - ms0), p1 = ex2(l1 - ms1), p2 = ex2(l2 - ms0), p3 = ex2(l3 - ms1);
  st.l[0] += p0 + p2;
  st.l[1] += p1 + p3;
  split_pair(p0, p1, b0h, b0l);
  split_pair(p2, p3, b1h, b1l);
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
      const int r = 8 * tr + q;
      uint32_t u;
      if constexpr (SMEM) {
        u = ok ? reinterpret_cast<const uint32_t*>(Vt)[r * 64 + xt_vword(8 * mt + 4 * cc + tig, r)] : 0u;
      } else {
        const uint16_t* vrow = SUB && r == sub ? vnew : (tr ? Vb : Va) + r * kD;
        u = ok ? __ldg(reinterpret_cast<const uint32_t*>(vrow + 16 * mt + 8 * cc + 2 * tig)) : 0u;
      }
      a[blkid] = movmatrix_trans(bf16x2_to_f16x2(u));
    }
    // a[0]: channels 16mt+q, tokens 2tig..; a[1]: channels +8; a[2]: tokens +8; a[3]: both
    mma_f16(st.acc[mt], a[0], a[1], a[2], a[3], b0h, b1h);
    if (!PACK4) mma_f16(st.acc[mt], a[0], a[1], a[2], a[3], b0l, b1l);
  }
}

// One 16-token tile of the plain BF16 paged cache (the comparator), rows
// [0, nv) valid, with the cached bf16 K and V rows and the query's own bf16
// values as the tensor-core operands (no conversion): Q.K against B = q
// (exact products; the softmax scale cE = sm_scale log2 e is applied to the
// fp32 logits), P.V against B = p 2^11 as a bf16 value + residual pair.  The
// lane's accumulator columns are heads 2 tig and 2 tig + 1 (store_state<false>).
// The tile's 16 K rows and 16 V rows sit in shared memory, kRawRow bytes
// apart (a row's 256 bytes plus 16, so that the fragment loads of the 16 rows
// spread over the banks).  Two halves: Q.K and the softmax give the B words
// of P.V (bw), then P.V.
// qb: the lane's B words of Q.K, word 2 ks + i = q[head lane / 4][32 tig + 4 ks + 2 i .. + 1].
constexpr int kRawRow = 2 * kD + 16;
__device__ __forceinline__ void bf16_raw_qk(const uint8_t* Ks, int nv, const uint32_t (&qb)[16], float cE,
                                            WarpState& st, int lane, uint32_t (&bw)[4]) {
  const int q = lane >> 2, tig = lane & 3;
  const bool va = q < nv, vb = q + 8 < nv;
  uint32_t ka[16], kb[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 u = va ? *reinterpret_cast<const uint4*>(Ks + q * kRawRow + 64 * tig + 16 * k) : make_uint4(0, 0, 0, 0);
    ka[4 * k] = u.x;
    ka[4 * k + 1] = u.y;
    ka[4 * k + 2] = u.z;
    ka[4 * k + 3] = u.w;
    const uint4 w =
        vb ? *reinterpret_cast<const uint4*>(Ks + (q + 8) * kRawRow + 64 * tig + 16 * k) : make_uint4(0, 0, 0, 0);
    kb[4 * k] = w.x;
    kb[4 * k + 1] = w.y;
    kb[4 * k + 2] = w.z;
    kb[4 * k + 3] = w.w;
  }
  float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) mma_bf16_acc(d, ka[2 * ks], kb[2 * ks], ka[2 * ks + 1], kb[2 * ks + 1], qb[2 * ks], qb[2 * ks + 1]);
  const float l0 = va ? d[0] * cE : -INFINITY, l1 = va ? d[1] * cE : -INFINITY;
  const float l2 = vb ? d[2] * cE : -INFINITY, l3 = vb ? d[3] * cE : -INFINITY;
  online_max(st, fmaxf(l0, l2), fmaxf(l1, l3));
  // weights scaled by 2^11 (kPScaleBF16) through the exponent
  const float ms0 = st.m[0] - 11.f, ms1 = st.m[1] - 11.f;
  const float p0 = ex2(l0 - ms0), p1 = ex2(l1 - ms1), p2 = ex2(l2 - ms0), p3 = ex2(l3 - ms1);
  st.l[0] += p0 + p2;
  st.l[1] += p1 + p3;
  auto split = [](float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16x2(x0, x1);
    lo = pack_bf16x2(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
  };
  split(p0, p1, bw[0], bw[1]);
  split(p2, p3, bw[2], bw[3]);
#pragma unroll
  for (int i = 0; i < 4; ++i) bw[i] = movmatrix_trans(bw[i]);
}

__device__ __forceinline__ void bf16_raw_pv(const uint8_t* Vs, int nv, const uint32_t (&bw)[4], WarpState& st,
                                            int lane) {
  const int q = lane >> 2, tig = lane & 3;
  const bool va = q < nv, vb = q + 8 < nv;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t a[4];
#pragma unroll
    for (int blkid = 0; blkid < 4; ++blkid) {
      const int tr = blkid >> 1, cc = blkid & 1;  // token half, channel half
      const int r = 8 * tr + q;
      const uint32_t u = (tr ? vb : va) ? *reinterpret_cast<const uint32_t*>(Vs + r * kRawRow + 32 * mt + 16 * cc + 4 * tig) : 0u;
      a[blkid] = movmatrix_trans(u);
    }
    // a[0]: channels 16mt+q, tokens 2tig..; a[1]: channels +8; a[2]: tokens +8; a[3]: both
    mma_bf16_acc(st.acc[mt], a[0], a[1], a[2], a[3], bw[0], bw[2]);
    mma_bf16_acc(st.acc[mt], a[0], a[1], a[2], a[3], bw[1], bw[3]);
  }
}

// A warp's state as written to its own stage memory: m[8], l[8], acc[8][128].
// inv undoes the B-operand scaling; packed mode adds each head's residual
// column to its value column.
template <bool PACK4>
__device__ __forceinline__ void store_state(WarpState& st, float* dst, float inv, int lane) {
  const int q = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], o);
    st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], o);
  }
  if constexpr (PACK4) {  // lane: head tig; columns 2 tig, 2 tig + 1 are its value and residual parts
    if (q == 0) {
      dst[tig] = st.m[0];
      dst[8 + tig] = st.l[0] * inv;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      dst[16 + tig * kStateStride + 16 * mt + q] = (st.acc[mt][0] + st.acc[mt][1]) * inv;
      dst[16 + tig * kStateStride + 16 * mt + q + 8] = (st.acc[mt][2] + st.acc[mt][3]) * inv;
    }
    return;
  }
  if (q == 0) {
    dst[2 * tig] = st.m[0];
    dst[2 * tig + 1] = st.m[1];
    dst[8 + 2 * tig] = st.l[0] * inv;
    dst[8 + 2 * tig + 1] = st.l[1] * inv;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = 16 * mt + q + 8 * (i >> 1), n = 2 * tig + (i & 1);
      dst[16 + n * kStateStride + ch] = st.acc[mt][i] * inv;
    }
  }
}

// A warp's INT2 (rotated-basis) state, as store_state writes it, except that
// in packed mode the residual column holds minus the residual (value_negres)
// and is subtracted from the value column.
template <bool PACK4>
__device__ __forceinline__ void store_int2_state(WarpState& st, float* dst, float inv, int lane) {
  if constexpr (PACK4) {
    const int q = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], o);
    if (q == 0) {
      dst[tig] = st.m[0];
      dst[8 + tig] = st.l[0] * inv;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      dst[16 + tig * kStateStride + 16 * mt + q] = (st.acc[mt][0] - st.acc[mt][1]) * inv;
      dst[16 + tig * kStateStride + 16 * mt + q + 8] = (st.acc[mt][2] - st.acc[mt][3]) * inv;
    }
  } else {
    store_state<false>(st, dst, inv, lane);
  }
}

// BF16 tile j (0..19) of a (request, KV head): tiles 0..3 are the sink page's
// rows 16 j .. 16 j + 15, tiles 4..19 rows 16 (j - 4) .. of the 256-row ring.
// Where the 16 ring rows rr0 .. rr0 + 15 of request b, KV head h live (element
// offsets into k_ring / v_ring): row r at (r < split ? off1 : off2) + r * 128.
// Ring row rr holds window position hist_end + ((rr - (hist_end - 64)) mod 256);
// the rows of a tile form one or two runs of consecutive positions (split where
// the oldest window position sits), each inside one 16-aligned block of
// positions, so inside one page of a paged recent window.
__device__ __forceinline__ bool recent_tile(const CacheRefs& c, int b, int h, int L, int rr0, size_t& off1,
                                            size_t& off2, int& split, unsigned* err, bool report) {
  const int hist_end = max(kSink, L - kRecent), rw = (hist_end - kSink) % kRecent;
  if (c.recent_table == nullptr) {  // the ring: contiguous rows
    split = 16;
    if (!recent_row(c, b, h, kSink + rr0, off1, err, report)) return false;
    off2 = off1;
    return true;
  }
  split = (rw > rr0 && rw < rr0 + 16) ? rw - rr0 : 16;
  const int p0 = hist_end + (((rr0 - rw) % kRecent) + kRecent) % kRecent;
  if (!recent_row(c, b, h, p0, off1, err, report)) return false;
  off2 = off1;
  if (split < 16) {
    if (!recent_row(c, b, h, hist_end, off2, err, report)) return false;
    off2 -= (size_t)split * kD;
  }
  return true;
}

__device__ __forceinline__ int bf16_tile_rows(int j, int L, size_t& row_off, bool& ring) {
  if (j < 4) {
    ring = false;
    row_off = 16 * j;
    return max(0, min(16, min(L, kSink) - 16 * j));
  }
  ring = true;
  const int rr = 16 * (j - 4);
  row_off = rr;
  const int live = L >= kSink + kRecent ? kRecent : max(0, L - kSink);
  return max(0, min(16, live - rr));
}

// Final merge of one (request, KV head): every partial record of its work
// items, the R_V^T rotation of the rotated-basis part, one normalisation.
// Run by the block that took the last ticket; kept out of line so that its
// registers are allocated apart from the page loop's.
template <bool PACK4>
__device__ __noinline__ void final_merge(const DecodeArgs& a, uint8_t* smem, int b, int h, int bh) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int X = a.n_items, g = a.g, RF = a.rec_floats;
  const float* recs = a.partials + (size_t)bh * X * RF;  // one original-basis record per item
  float* buf = reinterpret_cast<float*>(smem);            // record batch buffer
  const int cap = (int)((size_t)kWarps * kStages * kBlockBytes / 4 / RF);
  uint64_t* ubar = reinterpret_cast<uint64_t*>(smem + (size_t)kWarps * kStages * kBlockBytes) + kWarps * kStages;
  if (t == 0) {
    mbar_init(ubar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // warp (n, part): head n = warp % g merges records part, part + n_parts, ... of each batch
  const int n_parts = kWarps / g, n = warp % g, part = warp / g;
  const bool active = part < n_parts;
  float m = -INFINITY, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r0 = 0, batch = 0; r0 < X; r0 += cap, ++batch) {
    const int nb = min(cap, X - r0);
    if (warp == 0) {
      if (lane == 0) {
        fence_proxy_async_smem();  // the buffer was last used through generic loads and stores
        mbar_arrive_expect_tx(ubar, (unsigned)(nb * RF * 4));
      }
      __syncwarp();
      for (int i = lane; i < nb; i += 32)
        bulk_copy_g2s(buf + (size_t)i * RF, recs + (size_t)(r0 + i) * RF, (unsigned)(RF * 4), ubar);
    }
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(ubar, batch & 1, kWaitLimit))) {
      if (lane == 0) set_error(a.err, kErrTimeout);
      mbar_wait_bounded(ubar, batch & 1, kWaitLimit);
    }
    if (active)
      for (int i = part; i < nb; i += n_parts) {
        const float* rec = buf + (size_t)i * RF;
        merge_record(m, l, acc, rec[n], rec[8 + n], reinterpret_cast<const float4*>(rec + 16 + n * kD)[lane]);
      }
    __syncthreads();  // the buffer is refilled by the next batch, or becomes the stash
  }
  float* stash = buf;  // [kWarps][kStash]: acc[128], m, l per warp
  if (active) {
    float* s = stash + (size_t)warp * kStash;
    reinterpret_cast<float4*>(s)[lane] = acc;
    if (lane == 0) {
      s[kD] = m;
      s[kD + 1] = l;
    }
  }
  __syncthreads();
  if (warp < g) {
    const int hn = warp;
    float M = -INFINITY;
    for (int p = 0; p < n_parts; ++p) M = fmaxf(M, stash[(size_t)(p * g + hn) * kStash + kD]);
    float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      float L = 0.f;
      float4 o = res;
      for (int p = 0; p < n_parts; ++p) {
        const float* sp = stash + (size_t)(p * g + hn) * kStash;
        const float w = ex2(sp[kD] - M);
        L = fmaf(w, sp[kD + 1], L);
        const float4 v = reinterpret_cast<const float4*>(sp)[lane];
        o.x = fmaf(w, v.x, o.x);
        o.y = fmaf(w, v.y, o.y);
        o.z = fmaf(w, v.z, o.z);
        o.w = fmaf(w, v.w, o.w);
      }
      const float inv_l = 1.0f / L;
      res = make_float4(o.x * inv_l, o.y * inv_l, o.z * inv_l, o.w * inv_l);
    }
    *reinterpret_cast<float4*>(a.out + ((size_t)b * a.Hq + h * g + hn) * kD + 4 * lane) = res;
  }
  if (t == 0) a.counters[bh] = 0;  // ready for the next launch on this workspace
}

// The block merge, after every warp of the block has stored its states.
template <int MODE, bool PACK4>
__device__ __noinline__ void block_merge(const DecodeArgs& a, uint8_t* smem, const float* bf16_slots, int bh, int item) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  // warp w's rows [kRows w, kRows (w + 1)) of R_V^T (lane: output channels
  // 4 lane .. 4 lane + 3), copied into the warp's last stage during its last pages
  constexpr int kRows = kRvRows;
  float4 rv[kRows];
  if (MODE == 0) {
    uint64_t* rbar = reinterpret_cast<uint64_t*>(smem + (size_t)kWarps * kStages * kBlockBytes) + kWarps * kStages + 1 + warp;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(rbar, 0, kWaitLimit)) && lane == 0) set_error(a.err, kErrTimeout);
    const float4* src = reinterpret_cast<const float4*>(smem + ((size_t)(kStages - 1) * kWarps + warp) * kBlockBytes);
#pragma unroll
    for (int i = 0; i < kRows; ++i) rv[i] = src[i * (kD / 4) + lane];
  }
  griddep_launch_dependents();  // a dependent step kernel may start loading its constants
  __syncthreads();
  // merge the warps' states into this item's partial record:
  // the rotated-basis (INT2) states merged and multiplied by R_V^T, then
  // joined with the original-basis (BF16) states.  Thread t: head n = t / 128
  // (+ 4, + 8, ...), channel ch = t % 128.
  {
    constexpr int kG = PACK4 ? 4 : kMaxG;  // heads per KV head this variant serves
    constexpr int kHT = kG / 4;            // heads per thread
    const int ch = t & (kD - 1), n0 = t >> 7;
    float* ystage = reinterpret_cast<float*>(smem + (size_t)(kStages - 1) * kWarps * kBlockBytes);  // [kG][kD], warp 0's last stage
    float* opart = reinterpret_cast<float*>(smem);  // [kWarps][kG][kD], over the first stages once the states are merged
    const float* rot = reinterpret_cast<const float*>(smem);  // warp states, stride: a warp's stage memory
    const size_t rstride = kBlockBytes / sizeof(float);  // warp w's state: its first stage
    // original-basis states: the BF16 slots (mixed cache) or every warp's second stage
    const float* pln = MODE == 0 ? bf16_slots : rot + (size_t)kWarps * rstride;
    const size_t pstride = MODE == 0 ? (size_t)kPartialFloats : rstride;
    const int n_pln = MODE == 0 ? kBf16Slots : kWarps;
    float Mr[kHT], Lr[kHT], Mp[kHT], Lp[kHT], yp[kHT];
#pragma unroll
    for (int k = 0; k < kHT; ++k) {
      const int n = n0 + 4 * k;
      Mr[k] = Mp[k] = -INFINITY;
      Lr[k] = Lp[k] = yp[k] = 0.f;
      if (n >= a.g) continue;
      float yr = 0.f;
      if (MODE == 0) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) Mr[k] = fmaxf(Mr[k], rot[w * rstride + n]);
        if (Mr[k] != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kWarps; ++w) {
            const float* ws = rot + w * rstride;
            const float al = ex2(ws[n] - Mr[k]);  // 0 for an empty warp state (m = -inf)
            yr = fmaf(al, ws[16 + n * kStateStride + ch], yr);
            Lr[k] = fmaf(al, ws[8 + n], Lr[k]);
          }
        }
        ystage[n * kD + ch] = yr;
      }
#pragma unroll
      for (int w = 0; w < kWarps; ++w)
        if (w < n_pln) Mp[k] = fmaxf(Mp[k], pln[w * pstride + n]);
      if (Mp[k] != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          if (w >= n_pln) break;
          const float* ws = pln + w * pstride;
          const float al = ex2(ws[n] - Mp[k]);
          yp[k] = fmaf(al, ws[16 + n * kStateStride + ch], yp[k]);
          Lp[k] = fmaf(al, ws[8 + n], Lp[k]);
        }
      }
    }
    const bool dense = (a.rot_flags & kRotU) != 0;
    if (MODE == 0 && !dense) {
      // R_V^T = (H P)^T = P H: (y P) H per head, by warp hn (the product lands in opart[0])
      __syncthreads();  // ystage complete; the warp states are dead from here on
      if (warp < a.g) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = 4 * lane + e;
          v[e] = ystage[warp * kD + ((a.rot_flags & kRotP) ? brev7(i) : i)];
        }
        if (a.rot_flags & kRotH) {
          hadamard128(v, lane);
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] *= kInvSqrt128;
        }
        reinterpret_cast<float4*>(opart + warp * kD)[lane] = make_float4(v[0], v[1], v[2], v[3]);
      }
      __syncthreads();
    } else if (MODE == 0) {
      __syncthreads();  // ystage complete; the warp states are dead from here on
      // partial products y R_V^T over warp w's rows, for every head
      float o[kG][4];
#pragma unroll
      for (int hn = 0; hn < kG; ++hn) o[hn][0] = o[hn][1] = o[hn][2] = o[hn][3] = 0.f;
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const int j = kRows * warp + i;
        const float4 u = rv[i];
#pragma unroll
        for (int hn = 0; hn < kG; ++hn)
          if (hn < a.g) {
            const float yj = ystage[hn * kD + j];
            o[hn][0] = fmaf(yj, u.x, o[hn][0]);
            o[hn][1] = fmaf(yj, u.y, o[hn][1]);
            o[hn][2] = fmaf(yj, u.z, o[hn][2]);
            o[hn][3] = fmaf(yj, u.w, o[hn][3]);
          }
      }
#pragma unroll
      for (int hn = 0; hn < kG; ++hn)
        if (hn < a.g)
          reinterpret_cast<float4*>(opart + (warp * kG + hn) * kD)[lane] =
              make_float4(o[hn][0], o[hn][1], o[hn][2], o[hn][3]);
      __syncthreads();
    }
    float* part = a.partials + ((size_t)bh * a.n_items + item) * a.rec_floats;
#pragma unroll
    for (int k = 0; k < kHT; ++k) {
      const int n = n0 + 4 * k;
      if (n >= a.g) continue;
      float yr = 0.f;
      if (MODE == 0 && !dense)
        yr = opart[n * kD + ch];
      else if (MODE == 0)
#pragma unroll
        for (int w = 0; w < kWarps; ++w) yr += opart[(w * kG + n) * kD + ch];
      const float M = fmaxf(Mr[k], Mp[k]);
      float acc = 0.f, l = 0.f;
      if (M != -INFINITY) {
        const float fr = ex2(Mr[k] - M), fp = ex2(Mp[k] - M);
        acc = fmaf(fr, yr, fp * yp[k]);
        l = fmaf(fr, Lr[k], fp * Lp[k]);
      }
      part[16 + n * kD + ch] = acc;
      if (ch == 0) {
        part[n] = M;
        part[8 + n] = l;
      }
    }
  }

}

// Fused decode step (FUSED, mixed cache only): the kernel also appends this
// step's token and rotates q.  Before the dependency wait each thread loads
// its rows of R_K; after it every block rotates q itself (its warps' last
// stages serve as scratch while their first two units arrive); the block
// owning the history page that receives the evicted token moves that token
// in (and the new token into the ring or sink) and patches its own staged
// copy of the page; BF16 tiles read the new token's row from the input.
constexpr size_t kPatchOffset = (kSlotsOffset + (size_t)kBf16Slots * kPartialFloats * sizeof(float) + 15) / 16 * 16;

struct FusedScratch {  // in the warps' last stages
  PrepSmem prep;
  QuantSmem quant;
  uint32_t qf[kQFragWords];
  uint32_t qpl[kQFragWords];
  float qc[kQConstFloats];
};
static_assert(sizeof(FusedScratch) <= (size_t)kWarps * kBlockBytes, "fused scratch in the last stages");

// lanes 0..27 write the row's K words, V halves and scales into a staged block
__device__ __forceinline__ void apply_patch(uint8_t* blk, const RowPatch& pt, int row, int lane) {
  if (lane < 8) {
    *reinterpret_cast<uint32_t*>(blk + kKCodes + k_word_offset(row, lane & 3, lane >> 2)) = pt.kword[lane];
  } else if (lane < 24) {
    *reinterpret_cast<uint16_t*>(blk + kVCodes + v_half_offset(row, lane - 8)) = pt.vhalf[lane - 8];
  } else if (lane < 26) {
    *reinterpret_cast<uint16_t*>(blk + kKScales + 4 * row + 2 * (lane - 24)) = pt.kscale[lane - 24];
  } else if (lane < 28) {
    *reinterpret_cast<uint16_t*>(blk + kVScales + 4 * row + 2 * (lane - 26)) = pt.vscale[lane - 26];
  }
}

template <int MODE, bool PACK4, bool FUSED, bool LIMIT = false>
__device__ __forceinline__ void decode_body(const DecodeArgs& a, const StepArgs* f) {
  static_assert(!FUSED || MODE == 0, "the fused step serves the mixed cache");
  extern __shared__ __align__(128) uint8_t smem[];
  const int item = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int bh = b * a.Hkv + h;
  const CacheRefs& c = a.c;
  if (MODE == 0) {
    // While the kernel before this one finishes: pull this warp's first
    // pages into L2 (a hint only -- the tables read here may still change, and
    // the pages are read again, coherently, after the wait).  More than one
    // page per warp competes with the previous layer's final merge.
    if (item == 0)  // every block of this layer reads R_V^T in its block merge
      for (int i = t; i < kD * kD / 32; i += kThreads) prefetch_l2(a.R_VT + 32 * i);
    if constexpr (FUSED) {
      // the rows the q rotation and the append read first: this request's g
      // query rows and the new token's K and V rows (256 bytes each)
      const int r = t >> 1, half = t & 1;
      if (r < a.g)
        prefetch_l2(f->pr.q + ((size_t)b * f->pr.Hq + h * a.g + r) * kD + 64 * half);
      else if (r >= kMaxG && r < kMaxG + 2)
        prefetch_l2((r == kMaxG ? f->ap.k : f->ap.v) + ((size_t)b * a.Hkv + h) * kD + 64 * half);
    }
    if (lane == 0) {
      const int Lh = a.ctx_len[b];
      const int he = max(kSink, Lh - kRecent);
      const int nh = min((he + kPage - 1) / kPage - 1, c.max_pages - 1);
      const int q0 = 1 + item * a.chunk_pages, q1 = max(q0, min(q0 + a.chunk_pages, 1 + nh));
      const int rr = (q1 - q0) / kWarps, ee = (q1 - q0) - rr * kWarps;
      for (int k = 0; k <= rr && k < kPrefetchPages; ++k) {
        const int lp = k < rr ? q0 + warp + kWarps * k : (warp < ee ? q0 + kWarps * rr + warp : -1);
        if (lp < 0) break;
        const int ph = c.page_table[(size_t)b * c.max_pages + lp];
        if (ph >= 0 && ph < c.num_pages) bulk_prefetch_l2(c.pages + ((size_t)ph * a.Hkv + h) * kBlockBytes, kBlockBytes);
      }
    }
  }
  float rk[FUSED ? 32 : 1];  // fused step: R_K[32 (t / 128) + ii][t % 128] (a constant of the layer)
  if constexpr (FUSED) {
    const float* RK = f->pr.R_K + (size_t)32 * (t >> 7) * kD + (t & 127);
#pragma unroll
    for (int ii = 0; ii < 32; ++ii) rk[ii] = __ldg(RK + ii * kD);
  }
  griddep_wait();
  // fused step: the first units' page-table entries, read before the length is known (they
  // are whole pages lp0 + warp + kWarps k whenever the item has more than kStages rounds; the
  // entries are used only then)
  int spec_ph[kStages + 1];
  if constexpr (FUSED) {
    const int lps = 1 + item * a.chunk_pages + warp;
#pragma unroll
    for (int k = 0; k <= kStages; ++k)
      spec_ph[k] = lps + kWarps * k < c.max_pages ? c.page_table[(size_t)b * c.max_pages + lps + kWarps * k] : -1;
  }
  int L = a.ctx_len[b];
  if (L < 0) {
    if (t == 0 && item == 0) set_error(a.err, kErrLength);
    L = 0;
  }
  // extend attention: the query attends positions below lim only (the cache holds L)
  int lim = L;
  if constexpr (LIMIT) lim = max(0, min(a.limit[b], L));
  constexpr int kQW = PACK4 ? 16 : 32;
  // warp-private stage memory; after the warp's pages are done it holds the
  // warp's two finished states (rotated basis, original basis)
  // stage s of warp w: smem + (s kWarps + w) kBlockBytes (the warps' last
  // stages form one block)
  auto stage_ptr = [&](int s) -> uint8_t* { return smem + ((size_t)s * kWarps + warp) * kBlockBytes; };
  float* wstate = reinterpret_cast<float*>(stage_ptr(0));
  float* bf16_slots = reinterpret_cast<float*>(smem + kSlotsOffset);  // [kBf16Slots][kPartialFloats]
  WarpState st;

  if (MODE == 0) {
    // ---------------- INT2 history pages of this chunk (rotated basis)
    const int hist_end = max(kSink, L - kRecent);
    const int n_hist = (hist_end + kPage - 1) / kPage - 1;  // logical pages 1..n_hist
    if (n_hist + 1 > c.max_pages) {
      if (t == 0 && item == 0) set_error(a.err, kErrLength);
    }
    const int n_hist_ok = min(n_hist, c.max_pages - 1);
    // this item's pages [lp0, lp1): R whole rounds dealt round-robin over the
    // warps (warp w: pages lp0 + w + kWarps k, k < R), then the E left-over
    // pages as 4 E 16-token tiles (warp w: tiles w, w + kWarps, ...; tile tau
    // is tile tau % 4 of page lp0 + R kWarps + tau / 4)
    const int lp0 = 1 + item * a.chunk_pages;
    const int lp1 = max(lp0, min(lp0 + a.chunk_pages, 1 + n_hist_ok));
    const int R = (lp1 - lp0) / kWarps, E = (lp1 - lp0) - R * kWarps;
    const int n_tiles = 4 * E > warp ? (4 * E - warp + kWarps - 1) / kWarps : 0;
    const int n_my = R + n_tiles;
    // fused step: the loads the q rotation and the append wait on go first
    int p_new = -1, owner = 0, e_lp = -1, e_T = -1, e_row = -1;  // the new token; the evicted row to patch
    uint16_t qb0 = 0, qb1 = 0;
    float rvr[FUSED ? 32 : 1];  // the append block: R_V[32 (t / 128) + ii][t % 128]
    if constexpr (FUSED) {
      const int kq = t >> 7;
      const uint16_t* qrow = f->pr.q + ((size_t)b * f->pr.Hq + h * a.g) * kD + (t & 127);
      if (kq < a.g) qb0 = qrow[(size_t)kq * kD];
      if (kq + 4 < a.g) qb1 = qrow[(size_t)(kq + 4) * kD];
      p_new = f->ap.pos[b];
      if (p_new >= kSink + kRecent) {
        const int e = p_new - kRecent, lpe = e >> 6;
        if (lpe >= 1 && lpe < 1 + n_hist_ok) owner = (lpe - 1) / a.chunk_pages;
        e_lp = lpe;
        e_T = (e & 63) >> 4;
        e_row = e & 63;
      }
      if (item == owner) {
        const float* RV = f->ap.rot.R_V + (size_t)32 * kq * kD + (t & 127);
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) rvr[ii] = __ldg(RV + ii * kD);
      }
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kWarps * kStages * kBlockBytes) + warp * kStages;
    const uint8_t* pool = c.pages;
      // unit k: logical page and tile (-1: the whole page)
      auto unit_of = [&](int k, int& lp, int& T) {
        if (k < R) {
          lp = lp0 + warp + kWarps * k;
          T = -1;
        } else {
          const int tau = warp + kWarps * (k - R);
          lp = lp0 + R * kWarps + (tau >> 2);
          T = tau & 3;
        }
      };
      auto phys_of = [&](int lp) -> int {
        const int ph = c.page_table[(size_t)b * c.max_pages + lp];
        return (ph >= 0 && ph < c.num_pages) ? ph : -1;
      };
      auto phys_unit = [&](int k) -> int {  // physical page of unit k (-1: invalid)
        int lp, T;
        unit_of(k, lp, T);
        return phys_of(lp);
      };
      auto issue = [&](int k, int ph) {  // lane 0 only; ph = phys_unit(k)
        const int s = k % kStages;
        int lp, T;
        unit_of(k, lp, T);
        uint8_t* dst = stage_ptr(s);
        if (ph < 0) {
          set_error(a.err, kErrPage);
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&bars[s])) : "memory");
          return;
        }
        const uint8_t* src = pool + ((size_t)ph * a.Hkv + h) * kBlockBytes;
        if (T < 0) {
          mbar_arrive_expect_tx(&bars[s], kBlockBytes);
          bulk_copy_g2s(dst, src, kBlockBytes, &bars[s]);
        } else {  // the tile's K codes, K scales, V codes, V scales at their block offsets
          mbar_arrive_expect_tx(&bars[s], 2 * (512 + 64));
          bulk_copy_g2s(dst + kKCodes + 512 * T, src + kKCodes + 512 * T, 512, &bars[s]);
          bulk_copy_g2s(dst + kKScales + 64 * T, src + kKScales + 64 * T, 64, &bars[s]);
          bulk_copy_g2s(dst + kVCodes + 512 * T, src + kVCodes + 512 * T, 512, &bars[s]);
          bulk_copy_g2s(dst + kVScales + 64 * T, src + kVScales + 64 * T, 64, &bars[s]);
        }
      };
    // barrier of this warp's R_V^T rows (after the stage barriers and the final merge's)
    uint64_t* rbar = reinterpret_cast<uint64_t*>(smem + (size_t)kWarps * kStages * kBlockBytes) + kWarps * kStages + 1 + warp;
    bool rv_issued = false;  // lane 0
    auto issue_rv = [&]() {  // lane 0, once the last stage is free for good
      mbar_arrive_expect_tx(rbar, kRvBytes);
      bulk_copy_g2s(stage_ptr(kStages - 1), a.R_VT + (size_t)kRvRows * warp * kD, kRvBytes, rbar);
      rv_issued = true;
    };
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
      mbar_init(rbar, 1);
      fence_mbar_init();
      fence_proxy_async_smem();
    }
    __syncwarp();
    // (fused step: the last stages are scratch until the rotation and the
    // append are done; only the first kStages - 1 units are issued before)
    constexpr int kFirst = FUSED ? kStages - 1 : kStages;
    if (!FUSED && lane == 0 && n_my < kStages) issue_rv();
    // bit s: stage s holds a valid unit.  The page-table entry of unit
    // k + kStages is read during unit k - 1, so that issuing its copy after
    // unit k waits on nothing.
    uint32_t valid = 0;
    int ph_ahead = -1, ph_late = -1;
    int phs[kStages];
    // the first units' page-table entries (fused step with enough rounds: those read right
    // after the wait), then their copies -- in the fused step from inside the q rotation, so
    // that neither the entries nor the copies hold up its start
    if (n_my > 0) {
      if (FUSED && R > kStages) {
        auto checked = [&](int ph) { return (ph >= 0 && ph < c.num_pages) ? ph : -1; };
#pragma unroll
        for (int k = 0; k < kStages; ++k) phs[k] = checked(spec_ph[k]);
        ph_ahead = checked(spec_ph[kStages]);
      } else {
#pragma unroll
        for (int k = 0; k < kStages; ++k) phs[k] = k < n_my ? phys_unit(k) : -1;
        if (kStages < n_my) ph_ahead = phys_unit(kStages);
      }
    }
    auto first_copies = [&]() {
      if (n_my <= 0) return;
#pragma unroll
      for (int k = 0; k < kStages; ++k) {
        if (k >= n_my) break;
        valid |= (phs[k] >= 0 ? 1u : 0u) << k;
        if (k < kFirst) {
          if (lane == 0) issue(k, phs[k]);
        } else {
          ph_late = phs[k];
        }
      }
    };
    if (!FUSED) first_copies();
    uint32_t qf[kQW], qpf[kQW];
    float scaleE = 0.f, scaleEp = 0.f;
    const bool bf16_warp = kWarps - 1 - warp < kBf16Slots;
    if constexpr (FUSED) {
      FusedScratch& fs = *reinterpret_cast<FusedScratch*>(smem + (size_t)(kStages - 1) * kWarps * kBlockBytes);
      RowPatch* patch = reinterpret_cast<RowPatch*>(smem + kPatchOffset);
      prep_body(
          f->pr, b, h, t, [&](int ii) { return rk[ii]; }, [&](int n) { return n == (t >> 7) ? qb0 : qb1; }, fs.prep,
          1, fs.qf, fs.qpl, fs.qc, first_copies);
      // the append, by the block whose pages hold the evicted token's row (else item 0)
      if (item == owner) {
        if (t == 0) patch->row = -1;
        append_pair_body(
            f->ap, b, h, t, [&](int ii) { return rk[ii]; }, [&](int ii) { return rvr[ii]; }, fs.quant, 1, patch);
      }
      __syncthreads();
      if (item != owner || patch->row != e_row) e_lp = -1;  // no staged row to patch
      {
        const uint4* src = reinterpret_cast<const uint4*>(fs.qf + lane * 32);
        const uint4* srcp = reinterpret_cast<const uint4*>(fs.qpl + lane * 32);
#pragma unroll
        for (int k = 0; k < kQW / 4; ++k) {
          const uint4 u = src[k ^ (lane & 7)];
          qf[4 * k] = u.x;
          qf[4 * k + 1] = u.y;
          qf[4 * k + 2] = u.z;
          qf[4 * k + 3] = u.w;
          const uint4 v = bf16_warp ? srcp[k ^ (lane & 7)] : make_uint4(0, 0, 0, 0);
          qpf[4 * k] = v.x;
          qpf[4 * k + 1] = v.y;
          qpf[4 * k + 2] = v.z;
          qpf[4 * k + 3] = v.w;
        }
        scaleE = fs.qc[16];
        scaleEp = fs.qc[17];
      }
      __syncthreads();  // the scratch is released
      if (lane == 0) {
        fence_proxy_async_smem();
        if (n_my >= kStages)
          issue(kStages - 1, ph_late);
        else
          issue_rv();
      }
    }
    // BF16 sink/recent tiles (original basis) while the first pages arrive:
    // local tile k of this item goes to warp kWarps - 1 - k % kBf16Slots,
    // whose state waits in its slot until the block merge
    if (bf16_warp) {
      const int bk = kWarps - 1 - warp;
      state_init(st);
      if (bk < a.tiles_per_item && item * a.tiles_per_item + bk < kBf16Tiles) {
        if (!FUSED) {
          const uint4* src = reinterpret_cast<const uint4*>(a.qplain + (size_t)bh * kQFragWords + lane * 32);
#pragma unroll
          for (int k = 0; k < kQW / 4; ++k) {
            const uint4 u = __ldg(src + (k ^ (lane & 7)));
            qpf[4 * k] = u.x;
            qpf[4 * k + 1] = u.y;
            qpf[4 * k + 2] = u.z;
            qpf[4 * k + 3] = u.w;
          }
          scaleEp = __ldg(a.qconst + (size_t)bh * kQConstFloats + 17);
        }
        const int sp = c.sink_page[b];
        const bool sink_ok = sp >= 0 && sp < c.num_sink;
        for (int k = bk; k < a.tiles_per_item; k += kBf16Slots) {
          const int j = item * a.tiles_per_item + k;
          if (j >= kBf16Tiles) break;
          size_t row_off;
          bool ring;
          const int nv = bf16_tile_rows(j, L, row_off, ring);
          if (nv <= 0) continue;
          size_t off, off2;
          int split = 16;
          if (ring) {
            if (!recent_tile(c, b, h, L, (int)row_off, off, off2, split, a.err, lane == 0)) continue;
          } else {
            if (!sink_ok) {
              if (lane == 0) set_error(a.err, kErrSink);
              continue;
            }
            off = off2 = (((size_t)sp * a.Hkv + h) * kSink + row_off) * kD;
          }
          // fused step: the new token's row comes from the input
          int sub = -1;
          if (FUSED && p_new >= 0) {
            const int rr = p_new < kSink ? p_new : (p_new - kSink) % kRecent;
            if (ring == (p_new >= kSink) && (ring ? 4 + rr / 16 : rr / 16) == j) sub = rr % 16;
          }
          const size_t nrow = ((size_t)b * a.Hkv + h) * kD;
          uint32_t rows = (1u << nv) - 1u;
          if (LIMIT) {  // rows of positions at or past the query's limit are not attended
            if (!ring) {
              rows &= (1u << max(0, min(16, lim - (int)row_off))) - 1u;
            } else {
              // ring row rr holds position hist_end + ((rr - (hist_end - 64)) mod 256)
              const int hist_end = max(kSink, L - kRecent);
              for (int r = 0; r < nv; ++r) {
                const int rr = (int)row_off + r;
                const int p = hist_end + (((rr - (hist_end - kSink)) % kRecent) + kRecent) % kRecent;
                if (p >= lim) rows &= ~(1u << r);
              }
            }
            if (rows == 0) continue;  // nothing to attend (and a state with no max yet must stay empty)
          }
          const uint16_t* kbase = ring ? c.k_ring : c.k_sink;
          const uint16_t* vbase = ring ? c.v_ring : c.v_sink;
          bf16_tile<PACK4, FUSED>(kbase + off, vbase + off, kbase + off2, vbase + off2, split, rows, qpf, scaleEp,
                                  st, lane, sub, FUSED ? f->ap.k + nrow : nullptr, FUSED ? f->ap.v + nrow : nullptr);
        }
      }
      store_state<PACK4>(st, bf16_slots + (size_t)bk * kPartialFloats, 1.0f / kPScaleBF16, lane);
    }
    state_init(st);
    if (n_my > 0) {
      if (!FUSED) {
        const uint4* src = reinterpret_cast<const uint4*>(a.qfrag + (size_t)bh * kQFragWords + lane * 32);
#pragma unroll
        for (int k = 0; k < kQW / 4; ++k) {
          const uint4 u = __ldg(src + (k ^ (lane & 7)));
          qf[4 * k] = u.x;
          qf[4 * k + 1] = u.y;
          qf[4 * k + 2] = u.z;
          qf[4 * k + 3] = u.w;
        }
        scaleE = __ldg(a.qconst + (size_t)bh * kQConstFloats + 16);
      }
      const float kp = log2f(a.pscale);
      int k = 0;
      for (; k < n_my; ++k) {
        const int s = k % kStages;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[s], (k / kStages) & 1, kWaitLimit));
        if (!ok) {
          if (lane == 0) set_error(a.err, kErrTimeout);
          break;
        }
        int lp, T;
        unit_of(k, lp, T);
        if ((valid >> s) & 1u) {
          uint8_t* blk = stage_ptr(s);
          if (FUSED && lp == e_lp && (T < 0 || T == e_T)) {  // the row the append just evicted
            apply_patch(blk, *reinterpret_cast<const RowPatch*>(smem + kPatchOffset), e_row, lane);
            __syncwarp();
          }
          const int n_valid = min(kPage, (LIMIT ? min(hist_end, lim) : hist_end) - kPage * lp);
          if (T < 0 && n_valid == kPage) {
            int2_page_full<PACK4>(blk, qf, scaleE, kp, st, lane);
          } else {  // a partial page tile by tile, or tile T alone
            const int T0 = T < 0 ? 0 : T, T1 = T < 0 ? 4 : T + 1;
#pragma unroll 1
            for (int TT = T0; TT < T1; ++TT) {
              const int nv = min(16, n_valid - 16 * TT);
              if (nv > 0) int2_tile<PACK4>(blk, TT, nv, qf, scaleE, kp, st, lane);
            }
          }
        }
        __syncwarp();
        if (k + kStages < n_my) {
          const int ph = ph_ahead;
          ph_ahead = k + kStages + 1 < n_my ? phys_unit(k + kStages + 1) : -1;
          valid = (valid & ~(1u << s)) | ((ph >= 0 ? 1u : 0u) << s);
          if (lane == 0) {
            fence_proxy_async_smem();
            issue(k + kStages, ph);
          }
        } else if (lane == 0 && s == kStages - 1) {
          fence_proxy_async_smem();
          issue_rv();
        }
      }
      // after a timeout, wait (bounded) for the copies still in flight
      for (int kk = k + 1; kk < min(k + kStages, n_my); ++kk)
        mbar_wait_bounded(&bars[kk % kStages], (kk / kStages) & 1, kWaitLimit);
      if (k < n_my) mbar_wait_bounded(&bars[k % kStages], (k / kStages) & 1, kWaitLimit);
      if (lane == 0 && !rv_issued) {
        fence_proxy_async_smem();
        issue_rv();
      }
      __syncwarp();
    }
    store_int2_state<PACK4>(st, wstate, a.inv_pscale, lane);
  }

  // ---------------- BF16 paged cache (comparator): every warp, original basis
  if (MODE == 1) {
    state_init(st);
    // the lane's Q.K B words: head lane / 4 (columns of absent heads stay zero),
    // channels 32 tig .. 32 tig + 31 of the query as it came in (bf16)
    uint32_t qb[16];
    {
      const int n = lane >> 2;
      const uint4* src = reinterpret_cast<const uint4*>(a.q + ((size_t)b * a.Hq + h * a.g + n) * kD + 32 * (lane & 3));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 u = n < a.g ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
        qb[4 * k] = u.x;
        qb[4 * k + 1] = u.y;
        qb[4 * k + 2] = u.z;
        qb[4 * k + 3] = u.w;
      }
    }
    const float cE = a.sm_scale * kLog2e;
    {
      // plain BF16 paged cache: item covers pages [item*C, item*C + C), 4 tiles each;
      // the warp's tiles i = warp + kWarps j come through its kStages stages as units
      // 2 j (the 16 K rows) and 2 j + 1 (the 16 V rows), copied row by row (kRawRow apart)
      // kStages units ahead
      const int n_pages = (L + kPage - 1) / kPage;
      if (n_pages > c.max_pages) {
        if (t == 0 && item == 0) set_error(a.err, kErrLength);
      }
      const int pg0 = item * a.chunk_pages;
      const int pg1 = min(min(pg0 + a.chunk_pages, n_pages), c.max_pages);
      const int n_item_tiles = 4 * max(0, pg1 - pg0);
      const int n_my_t = n_item_tiles > warp ? (n_item_tiles - warp + kWarps - 1) / kWarps : 0;
      const int n_units = 2 * n_my_t;
      uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kWarps * kStages * kBlockBytes) + warp * kStages;
      if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
      }
      __syncwarp();
      auto tile_ph = [&](int j) -> int {  // physical page of the warp's tile j (-1: none or invalid)
        if (j >= n_my_t) return -1;
        const int ph = c.page_table[(size_t)b * c.max_pages + pg0 + (warp + kWarps * j) / 4];
        return (ph >= 0 && ph < c.num_pages) ? ph : -1;
      };
      // every lane: lane 0 arms the stage, lanes 0..15 copy one row each
      auto issue_u = [&](int u, int ph) {
        const int s = u % kStages, i = warp + kWarps * (u >> 1);
        if (lane == 0) {
          fence_proxy_async_smem();  // the stage's last reads came through the generic proxy
          if (ph < 0) {
            set_error(a.err, kErrPage);
            mbar_arrive(&bars[s]);
          } else {
            mbar_arrive_expect_tx(&bars[s], 16 * 2 * kD);
          }
        }
        __syncwarp();
        if (ph >= 0 && lane < 16) {
          const size_t off = (((size_t)ph * a.Hkv + h) * kPage + 16 * (i & 3) + lane) * kD;
          bulk_copy_g2s(stage_ptr(s) + lane * kRawRow, ((u & 1) ? a.vb_pages : a.kb_pages) + off, 2 * kD, &bars[s]);
        }
      };
      int ph_cur = tile_ph(0), ph_n1 = tile_ph(1);
      for (int u = 0; u < min(kStages, n_units); ++u) issue_u(u, u < 2 ? ph_cur : ph_n1);
      int j = 0;
      bool ok = true;
      for (; j < n_my_t && ok; ++j) {
        const int i = warp + kWarps * j, pg = pg0 + i / 4, tile = i & 3;
        const int ph_n2 = tile_ph(j + 2);
        const int nv = min(16, L - kPage * pg - 16 * tile);
        const bool use = ph_cur >= 0 && nv > 0;
        uint32_t bw[4];
        const int uk = 2 * j, uv = 2 * j + 1;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[uk % kStages], (uk / kStages) & 1, kWaitLimit));
        if (!ok) break;
        if (use) bf16_raw_qk(stage_ptr(uk % kStages), nv, qb, cE, st, lane, bw);
        __syncwarp();
        if (uk + kStages < n_units) issue_u(uk + kStages, ph_n1);  // V rows of tile j + 1
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[uv % kStages], (uv / kStages) & 1, kWaitLimit));
        if (!ok) break;
        if (use) bf16_raw_pv(stage_ptr(uv % kStages), nv, bw, st, lane);
        __syncwarp();
        if (uv + kStages < n_units) issue_u(uv + kStages, ph_n2);  // K rows of tile j + 2
        ph_cur = ph_n1;
        ph_n1 = ph_n2;
      }
      if (!ok) {
        if (lane == 0) set_error(a.err, kErrTimeout);
        // wait (bounded) for the copies still in flight
        for (int u = 2 * j; u < min(2 * j + kStages + 1, n_units); ++u)
          mbar_wait_bounded(&bars[u % kStages], (u / kStages) & 1, kWaitLimit);
      }
      __syncwarp();
    }
    store_state<false>(st, reinterpret_cast<float*>(stage_ptr(1)), 1.0f / kPScaleBF16, lane);
    state_init(st);
    store_state<PACK4>(st, wstate, 1.f, lane);  // the (empty) rotated-basis state
  }
  block_merge<MODE, PACK4>(a, smem, bf16_slots, bh, item);

  // ---------------- last block of this (request, KV head) merges all partials
  __shared__ int s_last;
  __syncthreads();
  if (t == 0) {
    // release this block's partial records, acquire the other blocks' ones
    int ticket;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;\n" : "=r"(ticket) : "l"(&a.counters[bh]) : "memory");
    s_last = (ticket == a.n_items - 1);
  }
  __syncthreads();
  if (!s_last) return;
  final_merge<PACK4>(a, smem, b, h, bh);
}

template <int MODE, bool PACK4, bool LIMIT = false>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ DecodeArgs a) {
  decode_body<MODE, PACK4, false, LIMIT>(a, nullptr);
}

template <bool PACK4>
__global__ void __launch_bounds__(kThreads, 1)
    decode_step_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ StepArgs f) {
  decode_body<0, PACK4, true>(a, &f);
}

// ------------------------------------------------------------------ extend (chunk) attention
// The queries of a chunk read the same cached pages: one block serves one
// (page range, KV head, group of queries) and unpacks each page once for the
// whole group (the kernel below).  Records: per (query, KV head, item) a
// rotated-basis (INT2) and an original-basis (BF16) state; a second kernel
// merges every item's records, applies R_V^T and normalises.
struct ExtendArgs {
  CacheRefs c;
  const int32_t* ctx_len;  // [B] cache lengths
  const int32_t* pos0;     // [B] chunk start positions
  int chunk, ngpr, qpg, Hq, Hkv, g;  // qpg: queries per group (one block per group, item and KV head)
  int n_items, chunk_pages, tiles_per_item;
  const uint32_t* qfrag;
  const uint32_t* qplain;
  const float* qconst;
  float* partials;  // [B chunk][Hkv][n_items][2][kPartialFloats]
  const float* R_VT;
  float pscale, inv_pscale;
  float* out;  // [B chunk][Hq][128]
  unsigned* err;
};

__device__ __forceinline__ void st_shared_u32(uint8_t* p, uint32_t v) { *reinterpret_cast<uint32_t*>(p) = v; }

// Unpack word t (< 512) of one staged INT2 block into the level tiles, and the scales (t < 64,
// as [group][token]).  The tiles are tcgen05 operands in the 128-byte swizzle -- K as [2 blocks
// of 64 channels][64 tokens][64 channels] (channels in the decode's MMA order), V as [128
// channels][64 tokens].
__device__ __forceinline__ void ext_unpack(const uint8_t* raw, uint8_t* kp, uint8_t* vp, float* ksc, float* vsc,
                                           int t) {
  const int T = t >> 7, ln = (t >> 2) & 31, wd = t & 3;
  {
    // K word t: row u, channels 32 ks + 16 kh + 4 tq + b, ks = 2 kpar + (p / 2), kh = p % 2, at bit 8 b + 2 p;
    // code_level<4 bb + p> gives channels (.. + bb, .. + bb + 2): MMA 4 (ks / 2) + 2 bb + ks % 2, columns
    // 8 kh + 2 tq and + 1 of it
    const int row = 16 * T + 8 * (wd >> 1) + (ln >> 2), tq = ln & 3, kpar = wd & 1;
    const CodeWord cw(*reinterpret_cast<const uint32_t*>(raw + kKCodes + 4 * t));
#define OSCAR_EXT_K(R)                                                                                  \
  do {                                                                                                  \
    constexpr int bb = (R) >> 2, p = (R)&3;                                                             \
    const int ks = 2 * kpar + (p >> 1), kh = p & 1;                                                     \
    const int col = 16 * (4 * (ks >> 1) + 2 * bb + (ks & 1)) + 8 * kh + 2 * tq;                         \
    st_shared_u32(kp + (col >> 6) * 8192 + sw128_elem(row, col & 63), code_level<R>(cw));             \
  } while (0)
    OSCAR_EXT_K(0);
    OSCAR_EXT_K(1);
    OSCAR_EXT_K(2);
    OSCAR_EXT_K(3);
    OSCAR_EXT_K(4);
    OSCAR_EXT_K(5);
    OSCAR_EXT_K(6);
    OSCAR_EXT_K(7);
#undef OSCAR_EXT_K
  }
  {
    // V word t: tokens u0, u0 + 1 (the halves), channels 16 r + jm at in-half index r
    const int u0 = 8 * (wd >> 1) + 2 * (ln & 3), jm = 8 * (wd & 1) + (ln >> 2);
    const int col = 16 * T + u0;
    const CodeWord cw(*reinterpret_cast<const uint32_t*>(raw + kVCodes + 4 * t));
#define OSCAR_EXT_V(R)                                                                                  \
  do {                                                                                                  \
    const int j = 16 * (R) + jm;                                                                        \
    st_shared_u32(vp + sw128_elem(j, col), code_level<R>(cw));                                        \
  } while (0)
    OSCAR_EXT_V(0);
    OSCAR_EXT_V(1);
    OSCAR_EXT_V(2);
    OSCAR_EXT_V(3);
    OSCAR_EXT_V(4);
    OSCAR_EXT_V(5);
    OSCAR_EXT_V(6);
    OSCAR_EXT_V(7);
#undef OSCAR_EXT_V
  }
  if (t < 64) {
    const float2 k2 = half2_bits_to_float2(*reinterpret_cast<const uint32_t*>(raw + kKScales + 4 * t));
    const float2 v2 = half2_bits_to_float2(*reinterpret_cast<const uint32_t*>(raw + kVScales + 4 * t));
    ksc[t] = k2.x;
    ksc[64 + t] = k2.y;
    vsc[t] = v2.x;
    vsc[64 + t] = v2.y;
  }
}

// ---------------------------------------------------------------- extend attention on tcgen05
// One block per (KV head, group of 128 / g queries, item = page range; the
// ranges sized by the plan's wave cost model): the group's (query, head)
// pairs are the 128 rows of every MMA (TMEM lane = row).  Per INT2 page:
// S = Q'_value K^T + Q'_residual K^T for each 64-channel group (f16 MMAs into
// TMEM), one softmax thread per row and half page (its query's causal limit,
// lazy rescaling of its half of the O row in TMEM), P s_v as fp16 value and
// negated residual operands, O += P V (V transposed; the residual MMAs negate
// A).  The A operands (q' and P) sit in TMEM, so an MMA reads only its B tile
// (K or V^T, 128-byte-swizzled) from shared memory.  S of the next page
// overlaps the softmax of this one.  Each block writes its rows' records;
// extend_merge_kernel merges the ranges.  Warps:
//   0-3, 9-12  softmax, two warpgroups splitting every page (tokens 0-31, 32-63) and O's
//        columns; warps 0-3 first put the q' rows into TMEM, then all eight run the
//        BF16 sink/recent tiles (per query, mma.sync, original-basis records) while
//        the first pages unpack; at the end the rows' rotated-basis records
//   4-7  the q' operands (from the prep's fragments, staged in shared memory),
//        then the pages: bulk copies (thread 128) and the unpack into the tile
//        buffers
//   8    TMEM (512 columns: S, O, q', P) and the MMA thread
constexpr int kXtThreads = 13 * 32;
constexpr uint32_t kXtQ = 0;             // q' value / residual: 2 x [2 blocks of 64 channels][128 rows][128 B]
constexpr int kXtTiles = 4;              // unpacked-page buffers (the MMAs of a page hold theirs until P V)
constexpr uint32_t kXtK = 65536;         // K tiles: kXtTiles x [2 blocks of 64 channels][64 tokens][128 B]
constexpr uint32_t kXtV = 131072;        // V^T tiles: kXtTiles x [128 channels][64 tokens]
constexpr uint32_t kXtRaw = 196608;      // raw pages: 2 x 4608
constexpr uint32_t kXtSc = kXtRaw + 2 * kBlockBytes;  // scales: kXtTiles x [K, V][group][64 tokens] float
constexpr uint32_t kXtBars = kXtSc + kXtTiles * 1024;
constexpr uint32_t kXtX = kXtBars + 256;  // softmax halves: page maxima [2][2][128], then l [2][128] (float)
constexpr uint32_t kXtTi = kXtX + 3072;   // staged BF16 tiles: [8] {valid rows, first row, ring}
constexpr int kXtStaged = 8;              // BF16 tiles an item may stage (8 KB each, in the q' staging area)
constexpr size_t kXtSmem = kXtTi + kXtStaged * 16 + 1024;  // + 1024-byte alignment slack
static_assert(kXtStaged * 8192 <= 65536, "staged BF16 tiles in the q' staging area");
static_assert(kXtK == kXtQ + 65536 && kXtV == kXtK + kXtTiles * 16384 && kXtRaw == kXtV + kXtTiles * 16384,
              "extend staging");

__global__ void __launch_bounds__(kXtThreads, 1) extend_tc_kernel(const __grid_constant__ ExtendArgs a) {
  extern __shared__ uint8_t xt_raw[];
  const uint32_t raw_s = smem_u32(xt_raw);
  uint8_t* sm = xt_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  const uint32_t sbase = smem_u32(sm);
  // blocks run KV head first and page range last: every (request, group, KV head) has its last,
  // possibly shorter, range in the last wave
  const int h = blockIdx.x, z = blockIdx.y, item = blockIdx.z;
  const int b = z / a.ngpr, grp = z % a.ngpr;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const CacheRefs& c = a.c;
  const int g = a.g, qpg = a.qpg;
  uint64_t* rawf = reinterpret_cast<uint64_t*>(sm + kXtBars);  // [2] raw page landed (tx)
  uint64_t* rawe = rawf + 2;     // [2] raw stage read by the unpack warps
  uint64_t* tfull = rawf + 4;    // [kXtTiles] tiles of buffer s unpacked
  uint64_t* tempty = rawf + 8;   // [kXtTiles] tiles of buffer s read by their MMAs (commit)
  uint64_t* sfull = rawf + 12;   // S in TMEM (commit)
  uint64_t* sfree = rawf + 13;   // S read by the softmax warps
  uint64_t* pfull = rawf + 14;   // P written, O rescaled
  uint64_t* pvdone = rawf + 15;  // P V finished (commit)
  uint64_t* done = rawf + 16;    // every MMA finished (commit)
  uint64_t* qsm = rawf + 17;     // q' operands staged in shared memory (4 warps)
  uint64_t* qtm = rawf + 18;     // q' operands in TMEM (4 warps)
  uint64_t* xm = rawf + 19;      // [2] page maxima of both softmax halves written (8 warps)
  uint64_t* xl = rawf + 21;      // the rows' l of both halves written (8 warps)
  uint32_t* tmem_at = reinterpret_cast<uint32_t*>(rawf + 22);
  uint64_t* bstg = rawf + 23;    // the item's BF16 tiles staged in shared memory (4 warps)
  // arrivals counted per warp: a lane's accesses are ordered before its
  // warp's one arrival by the warp barrier
  if (t == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&rawf[i], 1);
      mbar_init(&rawe[i], 4);
    }
    for (int i = 0; i < kXtTiles; ++i) {
      mbar_init(&tfull[i], 4);
      mbar_init(&tempty[i], 1);
    }
    mbar_init(sfull, 1);
    mbar_init(sfree, 8);
    mbar_init(pfull, 8);
    mbar_init(&xm[0], 8);
    mbar_init(&xm[1], 8);
    mbar_init(xl, 8);
    mbar_init(pvdone, 1);
    mbar_init(done, 1);
    mbar_init(qsm, 4);
    mbar_init(qtm, 4);
    mbar_init(bstg, 4);
    fence_mbar_init();
  }
  for (int i = t; i < 65536 / 16; i += kXtThreads)  // q' operands: rows without a query stay zero
    reinterpret_cast<uint4*>(sm + kXtQ)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();  // the tensor core reads them
  if (warp == 8) tmem_alloc(tmem_at, 512);
  griddep_wait();
  int L = a.ctx_len[b];
  if (L < 0) {
    if (t == 0 && item == 0) set_error(a.err, kErrLength);
    L = 0;
  }
  const int hist_end = max(kSink, L - kRecent);
  const int n_hist = (hist_end + kPage - 1) / kPage - 1;
  if (n_hist + 1 > c.max_pages && t == 0 && item == 0) set_error(a.err, kErrLength);
  const int n_hist_ok = min(n_hist, c.max_pages - 1);
  const int lp0 = 1 + item * a.chunk_pages;
  const int lp1 = max(lp0, min(lp0 + a.chunk_pages, 1 + n_hist_ok));
  const int n_units = lp1 - lp0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_at;

  // BF16 sink/recent tiles of this item (original basis, mma.sync per query).  Tile k: its
  // valid rows (0: none), positions and sources.
  const int sp = c.sink_page[b];
  const bool sink_ok = sp >= 0 && sp < c.num_sink;
  auto tile_src = [&](int k, size_t& off, size_t& off2, int& split, size_t& row_off, bool& ring) -> int {
    const int j = item * a.tiles_per_item + k;
    if (j >= kBf16Tiles) return 0;
    const int nv = bf16_tile_rows(j, L, row_off, ring);
    if (nv <= 0) return 0;
    split = 16;
    if (ring) {
      if (!recent_tile(c, b, h, L, (int)row_off, off, off2, split, a.err, lane == 0)) return 0;
    } else {
      if (!sink_ok) {
        if (lane == 0) set_error(a.err, kErrSink);
        return 0;
      }
      off = off2 = (((size_t)sp * a.Hkv + h) * kSink + row_off) * kD;
    }
    return nv;
  };
  // the rows of a tile that a query with causal limit lim attends
  auto rows_of = [&](int nv, size_t row_off, bool ring, int lim) -> uint32_t {
    uint32_t rows = (1u << nv) - 1u;
    if (!ring) {
      rows &= (1u << max(0, min(16, lim - (int)row_off))) - 1u;
    } else {
      for (int r = 0; r < nv; ++r) {
        const int rr = (int)row_off + r;
        const int p = hist_end + (((rr - (hist_end - kSink)) % kRecent) + kRecent) % kRecent;
        if (p >= lim) rows &= ~(1u << r);
      }
    }
    return rows;
  };

  if (warp >= 4 && warp < 8) {
    const int u = t - 128, w4 = warp - 4;
    auto issue = [&](int k) {  // thread u = 0: page k into raw stage k % 2
      const int st = k & 1;
      const int ph = c.page_table[(size_t)b * c.max_pages + lp0 + k];
      if (ph < 0 || ph >= c.num_pages) {
        set_error(a.err, kErrPage);
        mbar_arrive(&rawf[st]);
        return;
      }
      mbar_arrive_expect_tx(&rawf[st], kBlockBytes);
      bulk_copy_g2s(sm + kXtRaw + st * kBlockBytes, c.pages + ((size_t)ph * a.Hkv + h) * kBlockBytes, kBlockBytes,
                    &rawf[st]);
    };
    if (u == 0) {
      fence_proxy_async_smem();
      for (int k = 0; k < min(2, n_units); ++k) issue(k);
    }
    // q' rows: query ql of the group, head n, part p (value / residual) -> operand p, row ql g + n,
    // virtual channel 16 i + 8 bs + 2 tig (+1) for the word (i, bs) of lane 4 (2 n + p) + tig
    for (int ql = w4; ql < qpg; ql += 4) {
      const int qi = grp * qpg + ql;
      if (qi >= a.chunk) continue;
      const int bq = (b * a.chunk + qi) * a.Hkv + h;
      const int col = lane >> 2, tig = lane & 3, n = col >> 1, part = col & 1;
      if (n >= g) continue;
      const uint4* src = reinterpret_cast<const uint4*>(a.qfrag + (size_t)bq * kQFragWords + lane * 32);
      const int row = ql * g + n;
      uint8_t* dst = sm + kXtQ + part * 32768;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint4 v = __ldg(src + (kk ^ (lane & 7)));
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int wi = 4 * kk + x, i = wi >> 1, bs = wi & 1;
          const int vc = 16 * i + 8 * bs + 2 * tig;
          st_shared_u32(dst + (vc >> 6) * 16384 + sw128_elem(row, vc & 63), wv[x]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(qsm);
    // INT2 pages: raw stage k % 2 unpacked into the tiles of buffer k % kXtTiles
    bool timed_out = false;
    for (int k = 0; k < n_units; ++k) {
      const int rs = k & 1, st = k % kXtTiles;
      if (!mbar_wait_timed(&rawf[rs], (k >> 1) & 1, kWaitNs) ||
          !mbar_wait_timed(&tempty[st], ((k / kXtTiles) & 1) ^ 1, kWaitNs)) {
        set_error(a.err, kErrTimeout);
        timed_out = true;
        break;
      }
      const uint8_t* rp = sm + kXtRaw + rs * kBlockBytes;
      float* sc = reinterpret_cast<float*>(sm + kXtSc + st * 1024);
#pragma unroll
      for (int x = 0; x < 4; ++x)
        ext_unpack(rp, sm + kXtK + st * 16384, sm + kXtV + st * 16384, sc, sc + 128, u + 128 * x);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tfull[st]);
        mbar_arrive(&rawe[rs]);
      }
      if (u == 0 && k + 2 < n_units) {
        if (!mbar_wait_timed(&rawe[rs], (k >> 1) & 1, kWaitNs)) {
          set_error(a.err, kErrTimeout);
          timed_out = true;
          break;
        }
        issue(k + 2);
      }
    }
    if (u == 0 && timed_out)  // copies may still be in flight
      for (int k = 0; k < min(2, n_units); ++k) mbar_wait_timed(&rawf[k], 0, kWaitNs);
  } else if (warp == 8) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_f16_f32(128, 64);
      const uint64_t dhi = umma_desc_sw128(0) & 0xFFFFFFFF00000000ull;
      const uint32_t k_lo = (uint32_t)umma_desc_sw128(sbase + kXtK), v_lo = (uint32_t)umma_desc_sw128(sbase + kXtV);
      // TMEM columns: S [2 groups][64 tokens], O [128 channels], q' [part][2 blocks][32], P [group][part][32]
      const uint32_t tS = tbase, tO = tbase + 128, tQ = tbase + 256, tP = tbase + 384;
      bool ok = mbar_wait_timed(qtm, 0, kWaitNs);
      // S = q' K^T of page k (tiles of buffer k % 2) for each 64-channel group
      auto issue_s = [&](int k) {
        const int st = k % kXtTiles;
        tc_fence_after();
#pragma unroll
        for (int gr = 0; gr < 2; ++gr)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
#pragma unroll
            for (int pt = 0; pt < 2; ++pt) {
              const uint64_t bd = dhi | (k_lo + ((st * 16384 + gr * 8192 + ks * 32) >> 4));
              umma_f16_ts(tS + 64 * gr, tQ + 64 * pt + 32 * gr + 8 * ks, bd, idesc, ks > 0 || pt > 0);
            }
        umma_commit(sfull);
      };
      if (ok && n_units > 0) {
        ok = mbar_wait_timed(&tfull[0], 0, kWaitNs);
        if (ok) issue_s(0);
      }
      for (int k = 0; k < n_units && ok; ++k) {
        const int st = k % kXtTiles;
        if (k + 1 < n_units) {
          ok = mbar_wait_timed(&tfull[(k + 1) % kXtTiles], ((k + 1) / kXtTiles) & 1, kWaitNs) &&
               mbar_wait_timed(sfree, k & 1, kWaitNs);
          if (!ok) break;
          issue_s(k + 1);
        }
        ok = mbar_wait_timed(pfull, k & 1, kWaitNs);
        if (!ok) break;
        tc_fence_after();
        // O[:, 64 G ..] += P_G V^T[64 G ..]: value and residual parts, 4 steps of 16 tokens (the
        // residual matrices hold the residuals negated; bit 13 of the descriptor negates A)
#pragma unroll
        for (int gr = 0; gr < 2; ++gr)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
#pragma unroll
            for (int pt = 0; pt < 2; ++pt) {
              const uint64_t bd = dhi | (v_lo + ((st * 16384 + gr * 8192 + ks * 32) >> 4));
              umma_f16_ts(tO + 64 * gr, tP + 32 * (2 * gr + pt) + 8 * ks, bd, pt ? (idesc | (1u << 13)) : idesc,
                          k > 0 || ks > 0 || pt > 0);
            }
        umma_commit(pvdone);
        umma_commit(&tempty[st]);
      }
      if (!ok) set_error(a.err, kErrTimeout);
      umma_commit(done);
      if (!mbar_wait_timed(done, 0, kWaitNs)) set_error(a.err, kErrTimeout);
    }
    __syncwarp();
  } else {
    // softmax, two warpgroups: wg 0 (warps 0-3) takes tokens 0-31 of every page and O columns
    // 0-63, wg 1 (warps 9-12) tokens 32-63 and columns 64-127.  Row r (TMEM lane 32 (warp % 4) +
    // lane) = query ql = r / g of the group, head n = r % g; the two threads of a row swap their
    // page maxima, so both keep the same running maximum.
    const int wg = warp >= 9 ? 1 : 0;
    const int r = 32 * (warp & 3) + lane, ql = r / g, n = r % g, qi = grp * qpg + ql;
    const bool active = ql < qpg && qi < a.chunk;
    const int qg = b * a.chunk + (active ? qi : 0);
    const int lim = active ? max(0, min(a.pos0[b] + qi + 1, L)) : 0;
    const int hlim = min(hist_end, lim);
    const float scaleE = active ? __ldg(a.qconst + ((size_t)qg * a.Hkv + h) * kQConstFloats + 16) : 0.f;
    const float kpl = log2f(a.pscale);
    const uint32_t tS = tbase + ((uint32_t)(32 * (warp & 3)) << 16), tO = tS + 128, tQ = tS + 256, tP = tS + 384;
    float* pmx = reinterpret_cast<float*>(sm + kXtX);  // [page parity][wg][128 rows] page maxima, then [wg][128] l
    float m = -INFINITY;
    float2 l2 = make_float2(0.f, 0.f);  // the row's sums over even and odd tokens
    bool ok = true;
    if (wg == 0) {
      // this row's q' (both parts, K order of the staged tiles) into TMEM: the A operand of S
      ok = __all_sync(0xffffffffu, mbar_wait_timed(qsm, 0, kWaitNs));
      if (ok) {
#pragma unroll
        for (int pb = 0; pb < 4; ++pb) {  // part pb / 2, block of 64 channels pb % 2
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 v = *reinterpret_cast<const uint4*>(sm + kXtQ + pb * 16384 + sw128_elem(r, 8 * j));
            w[4 * j] = v.x;
            w[4 * j + 1] = v.y;
            w[4 * j + 2] = v.z;
            w[4 * j + 3] = v.w;
          }
          tmem_st32u(tQ + 32 * pb, w);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(qtm);
    }
    // The item's BF16 tiles, per query, while the copy warps unpack the first pages: with at most
    // kXtStaged tiles an item, the warps of warpgroup 1 stage them (warp w tiles w, w + 4) in the
    // q' staging area (free once q' is in TMEM; swizzled so the MMA fragment loads are free of bank
    // conflicts) with their rows and positions; the eight softmax warps then take queries sw,
    // sw + 8, ... of the group.
    {
      const bool staged = a.tiles_per_item <= kXtStaged;
      const int sw = 4 * wg + (warp & 3);
      uint8_t* stg = sm + kXtQ;  // [kXtStaged tiles][K 4 KB, V 4 KB]
      int4* tinfo = reinterpret_cast<int4*>(sm + kXtTi);
      if (staged) {
        if (wg == 1) {
          const bool qok = __all_sync(0xffffffffu, mbar_wait_timed(qtm, 0, kWaitNs));  // q' has left for TMEM
          if (!qok && lane == 0) set_error(a.err, kErrTimeout);
          for (int k = warp & 3; k < a.tiles_per_item; k += 4) {
            size_t off = 0, off2 = 0, row_off = 0;
            int split = 16;
            bool ring = false;
            const int nv = qok ? tile_src(k, off, off2, split, row_off, ring) : 0;
            const uint16_t* kg = ring ? c.k_ring : c.k_sink;
            const uint16_t* vg = ring ? c.v_ring : c.v_sink;
            // element e = lane + 32 i: row e / 16, 16-byte chunk e % 16
            uint4 kv[8], vv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int e = lane + 32 * i, rw = e >> 4, ch = e & 15;
              if (rw < nv) {
                const size_t o = (rw < split ? off : off2) + (size_t)rw * kD;
                kv[i] = __ldg(reinterpret_cast<const uint4*>(kg + o) + ch);
                vv[i] = __ldg(reinterpret_cast<const uint4*>(vg + o) + ch);
              }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int e = lane + 32 * i, rw = e >> 4, ch = e & 15;
              if (rw < nv) {
                reinterpret_cast<uint4*>(stg + k * 8192)[rw * 16 + xt_kchunk(ch, rw)] = kv[i];
                reinterpret_cast<uint4*>(stg + k * 8192 + 4096)[(rw * 64 + xt_vword(4 * ch, rw)) >> 2] = vv[i];
              }
            }
            if (lane == 0) tinfo[k] = make_int4(nv, (int)row_off, ring ? 1 : 0, 0);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bstg);
        }
        if (!__all_sync(0xffffffffu, mbar_wait_timed(bstg, 0, kWaitNs)) && lane == 0) set_error(a.err, kErrTimeout);
      }
      for (int qq = sw; qq < qpg && grp * qpg + qq < a.chunk; qq += 8) {
        const int qiq = grp * qpg + qq;
        const int qgq = b * a.chunk + qiq, bq = qgq * a.Hkv + h;
        const int limq = max(0, min(a.pos0[b] + qiq + 1, L));
        uint32_t qpf[16];
        {
          const uint4* srcp = reinterpret_cast<const uint4*>(a.qplain + (size_t)bq * kQFragWords + lane * 32);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint4 v = __ldg(srcp + (kk ^ (lane & 7)));
            qpf[4 * kk] = v.x;
            qpf[4 * kk + 1] = v.y;
            qpf[4 * kk + 2] = v.z;
            qpf[4 * kk + 3] = v.w;
          }
        }
        const float scaleEp = __ldg(a.qconst + (size_t)bq * kQConstFloats + 17);
        WarpState sb;
        state_init(sb);
        if (staged) {
          for (int k = 0; k < a.tiles_per_item; ++k) {
            const int4 ti = tinfo[k];
            if (ti.x == 0) continue;
            const uint32_t rows = rows_of(ti.x, (size_t)ti.y, ti.z != 0, limq);
            if (rows == 0) continue;
            const uint16_t* kt = reinterpret_cast<const uint16_t*>(stg + k * 8192);
            bf16_tile<true, false, true>(kt, kt + 2048, kt, kt + 2048, 16, rows, qpf, scaleEp, sb, lane);
          }
        } else {
          for (int k = 0; k < a.tiles_per_item; ++k) {
            size_t off = 0, off2 = 0, row_off = 0;
            int split = 16;
            bool ring = false;
            const int nv = tile_src(k, off, off2, split, row_off, ring);
            if (nv == 0) continue;
            const uint32_t rows = rows_of(nv, row_off, ring, limq);
            if (rows == 0) continue;
            const uint16_t* kbase = ring ? c.k_ring : c.k_sink;
            const uint16_t* vbase = ring ? c.v_ring : c.v_sink;
            bf16_tile<true>(kbase + off, vbase + off, kbase + off2, vbase + off2, split, rows, qpf, scaleEp, sb,
                            lane);
          }
        }
        store_state<true>(sb, a.partials + (((size_t)qgq * a.Hkv + h) * a.n_items + item) * 2 * kPartialFloats +
                                  kPartialFloats,
                          1.0f / kPScaleBF16, lane);
      }
    }
    for (int k = 0; k < n_units && ok; ++k) {
      const int st = k % kXtTiles;
      if (!__all_sync(0xffffffffu, mbar_wait_timed(sfull, k & 1, kWaitNs))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* sc = reinterpret_cast<const float*>(sm + kXtSc + st * 1024);  // K, V: [group][64 tokens]
      const int nv = min(kPage, hlim - kPage * (lp0 + k));
      // raw logits of this half page (the q' scale 2^E applied in the exponent below); a warp
      // whose rows all see the whole page skips the masking
      const bool whole = __all_sync(0xffffffffu, nv >= kPage);
      float lg[32];
      {
        float s0[32], s1[32];
        tmem_ld32x2(tS + 32 * wg, tS + 64 + 32 * wg, s0, s1);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {  // token pairs on packed fp32 pairs
          const int tk = 32 * wg + e;
          const float4 k0 = *reinterpret_cast<const float4*>(sc + tk), k1 = *reinterpret_cast<const float4*>(sc + 64 + tk);
          const float2 x0 = ffma2(make_float2(s0[e], s0[e + 1]), make_float2(k0.x, k0.y),
                                  fmul2(make_float2(s1[e], s1[e + 1]), make_float2(k1.x, k1.y)));
          const float2 x1 = ffma2(make_float2(s0[e + 2], s0[e + 3]), make_float2(k0.z, k0.w),
                                  fmul2(make_float2(s1[e + 2], s1[e + 3]), make_float2(k1.z, k1.w)));
          lg[e] = x0.x;
          lg[e + 1] = x0.y;
          lg[e + 2] = x1.x;
          lg[e + 3] = x1.y;
        }
        if (!whole) {  // rows past the query's limit or the history end
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * wg + e >= nv) lg[e] = -INFINITY;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfree);
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < 32; ++e) mq[e & 3] = fmaxf(mq[e & 3], lg[e]);
      float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * scaleE;
      // the row's page maximum over both halves
      pmx[((k & 1) * 2 + wg) * 128 + r] = mx;
      __syncwarp();
      if (lane == 0) mbar_arrive(&xm[k & 1]);
      if (!__all_sync(0xffffffffu, mbar_wait_timed(&xm[k & 1], (k >> 1) & 1, kWaitNs))) {
        ok = false;
        break;
      }
      mx = fmaxf(mx, pmx[((k & 1) * 2 + (wg ^ 1)) * 128 + r]);
      if (k > 0 && !__all_sync(0xffffffffu, mbar_wait_timed(pvdone, (k - 1) & 1, kWaitNs))) {
        ok = false;  // (the wait: P buffer free, O settled)
        break;
      }
      // lazy rescaling of this row's half of O; TMEM loads and stores are warp-wide
      // (.sync.aligned), so every lane of the warp takes part whenever one needs it
      const bool need = nv > 0 && mx > m + kLazy;
      const float nm = need ? fmaxf(m, mx) : m;
      const float al = (need && m != -INFINITY) ? ex2(m - nm) : 1.f;
      if (__any_sync(0xffffffffu, need && m != -INFINITY)) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float o[32];
          tmem_ld32(tO + 64 * wg + 32 * cc, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= al;
          tmem_st32(tO + 64 * wg + 32 * cc, o);
        }
        tmem_wait_st();
      }
      l2 = fmul2(l2, make_float2(al, al));
      m = nm;
      const float ms = nv > 0 ? m - kpl : 0.f;
      const float2 sE = make_float2(scaleE, scaleE), nms = make_float2(-ms, -ms);
      const float* vs = sc + 128;
      // P (A operand of P V) into TMEM: matrix 2 G + part (part 1: minus the residual), column =
      // token pair
#pragma unroll
      for (int c16 = 0; c16 < 2; ++c16) {
        uint32_t w[4][8];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const int el = 16 * c16 + e, tk = 32 * wg + el;
          const float4 v0 = *reinterpret_cast<const float4*>(vs + tk), v1 = *reinterpret_cast<const float4*>(vs + 64 + tk);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const float2 ar = ffma2(make_float2(lg[el + 2 * h2], lg[el + 2 * h2 + 1]), sE, nms);
            const float2 p = make_float2(ex2(ar.x), ex2(ar.y));
            l2 = fadd2(l2, p);
            const float2 a = fmul2(p, h2 ? make_float2(v0.z, v0.w) : make_float2(v0.x, v0.y));
            const float2 bq = fmul2(p, h2 ? make_float2(v1.z, v1.w) : make_float2(v1.x, v1.y));
            const int c = (e >> 1) + h2;
            w[0][c] = pack_f16x2(a.x, a.y);
            w[1][c] = f16x2_negres(w[0][c], a.x, a.y);
            w[2][c] = pack_f16x2(bq.x, bq.y);
            w[3][c] = f16x2_negres(w[2][c], bq.x, bq.y);
          }
        }
#pragma unroll
        for (int mtx = 0; mtx < 4; ++mtx) tmem_st8u(tP + 32 * mtx + 16 * wg + 8 * c16, w[mtx]);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pfull);
    }
    // the row's rotated-basis record (the TMEM loads warp-wide, the stores per row)
    if (ok && n_units > 0 && !__all_sync(0xffffffffu, mbar_wait_timed(pvdone, (n_units - 1) & 1, kWaitNs)))
      ok = false;
    // the row's l over both halves
    float l = l2.x + l2.y;
    float* pl = pmx + 512;
    pl[wg * 128 + r] = l;
    __syncwarp();
    if (lane == 0) mbar_arrive(xl);
    if (!__all_sync(0xffffffffu, mbar_wait_timed(xl, 0, kWaitNs))) ok = false;
    l += pl[(wg ^ 1) * 128 + r];
    if (!ok) set_error(a.err, kErrTimeout);
    tc_fence_after();
    float* rec = a.partials + (((size_t)qg * a.Hkv + h) * a.n_items + item) * 2 * kPartialFloats;
    if (active && wg == 0) {
      rec[n] = m;
      rec[8 + n] = l * a.inv_pscale;
    }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      float o[32];
      if (n_units > 0) {
        tmem_ld32(tO + 64 * wg + 32 * cc, o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0.f;
      }
      if (active) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(rec + 16 + n * kStateStride + 64 * wg + 32 * cc + e) =
              make_float4(o[e] * a.inv_pscale, o[e + 1] * a.inv_pscale, o[e + 2] * a.inv_pscale,
                          o[e + 3] * a.inv_pscale);
      }
    }
  }
  tc_fence_before();
  griddep_launch_dependents();  // the merge kernel may stage R_V^T
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// The merge of the chunk kernel's records: one block per (KV head, request and
// query group, slice of 16 rows; row r = query ql of the group, head n:
// r = ql g + n).  Every page range's records of both kinds are merged per
// (row, 4-channel quad), then the rotated-basis part is multiplied by R_V^T
// (staged before the dependency wait: a constant of the layer), joined with
// the original-basis part and normalised.
constexpr int kMgRows = 16;
constexpr int kMgThreads = 256;
constexpr size_t kMgSmem = (size_t)(128 * 128 + 2 * kMgRows * 128) * 4 + kMgRows * 16;

__global__ void __launch_bounds__(kMgThreads) extend_merge_kernel(const __grid_constant__ ExtendArgs a) {
  extern __shared__ float4 mg_raw[];
  float* rvt = reinterpret_cast<float*>(mg_raw);  // R_V^T [128][128]
  float* ys = rvt + 128 * 128;                   // merged rotated-basis parts [16 rows][128]
  float* ps = ys + kMgRows * 128;                // merged original-basis parts [16 rows][128]
  float4* rs = reinterpret_cast<float4*>(ps + kMgRows * 128);  // per row (M_r, L_r, M_p, L_p)
  const int h = blockIdx.x, z = blockIdx.y, r0 = blockIdx.z * kMgRows;
  const int b = z / a.ngpr, grp = z % a.ngpr;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, g = a.g, X = a.n_items;
  for (int e = t; e < 128 * 128 / 4; e += kMgThreads)
    reinterpret_cast<float4*>(rvt)[e] = __ldg(reinterpret_cast<const float4*>(a.R_VT) + e);
  griddep_wait();
  // the records, both kinds, by (row, 4-channel quad): a row's 32 quads in one warp; per eight
  // page ranges, lane i loads m and l of record i and every lane its quads of all sixteen, which
  // then merge in page-range order
  for (int task = t; task < kMgRows * 32; task += kMgThreads) {
    const int j = task >> 5, c4 = task & 31, r = r0 + j, ql = r / g, n = r % g, qi = grp * a.qpg + ql;
    float Mr = -INFINITY, Lr = 0.f, Mp = -INFINITY, Lp = 0.f;
    float4 yr = make_float4(0.f, 0.f, 0.f, 0.f), yp = yr;
    if (ql < a.qpg && qi < a.chunk) {
      const float* rec0 = a.partials + ((size_t)(b * a.chunk + qi) * a.Hkv + h) * X * 2 * kPartialFloats;
      for (int x0 = 0; x0 < X; x0 += 8) {
        const int nr = 2 * min(8, X - x0);  // records of this round: page range x0 + i / 2, kind i % 2
        float mv = -INFINITY, lv = 0.f;
        if (lane < nr) {
          const float* rc = rec0 + (size_t)(2 * x0 + lane) * kPartialFloats;
          mv = __ldcg(rc + n);
          lv = __ldcg(rc + 8 + n);
        }
        float4 v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < nr)
            v[i] = __ldcg(reinterpret_cast<const float4*>(rec0 + (size_t)(2 * x0 + i) * kPartialFloats + 16 +
                                                          n * kStateStride) + c4);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float mi = __shfl_sync(0xffffffffu, mv, i), li = __shfl_sync(0xffffffffu, lv, i);
          if (i < nr) {
            if (i & 1)
              merge_record(Mp, Lp, yp, mi, li, v[i]);
            else
              merge_record(Mr, Lr, yr, mi, li, v[i]);
          }
        }
      }
    }
    reinterpret_cast<float4*>(ys + j * 128)[c4] = yr;
    reinterpret_cast<float4*>(ps + j * 128)[c4] = yp;
    if (c4 == 0) rs[j] = make_float4(Mr, Lr, Mp, Lp);
  }
  __syncthreads();
  // y R_V^T: warp w takes rows 2 w and 2 w + 1 of the slice, lane the output channels 4 lane ..
  // 4 lane + 3; the sums run over the input channels in order
  float o[2][4];
#pragma unroll
  for (int i = 0; i < 2; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  for (int k = 0; k < 128; k += 4) {
    const float4 y0 = *reinterpret_cast<const float4*>(ys + (2 * warp) * 128 + k);
    const float4 y1 = *reinterpret_cast<const float4*>(ys + (2 * warp + 1) * 128 + k);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float4 rr = reinterpret_cast<const float4*>(rvt + (k + kk) * 128)[lane];
      const float ya = kk == 0 ? y0.x : kk == 1 ? y0.y : kk == 2 ? y0.z : y0.w;
      const float yb = kk == 0 ? y1.x : kk == 1 ? y1.y : kk == 2 ? y1.z : y1.w;
      o[0][0] = fmaf(ya, rr.x, o[0][0]);
      o[0][1] = fmaf(ya, rr.y, o[0][1]);
      o[0][2] = fmaf(ya, rr.z, o[0][2]);
      o[0][3] = fmaf(ya, rr.w, o[0][3]);
      o[1][0] = fmaf(yb, rr.x, o[1][0]);
      o[1][1] = fmaf(yb, rr.y, o[1][1]);
      o[1][2] = fmaf(yb, rr.z, o[1][2]);
      o[1][3] = fmaf(yb, rr.w, o[1][3]);
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int j = 2 * warp + i, r = r0 + j, ql = r / g, n = r % g, qi = grp * a.qpg + ql;
    if (ql >= a.qpg || qi >= a.chunk) continue;
    const float4 st = rs[j];
    const float M = fmaxf(st.x, st.z);
    float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      const float fr = ex2(st.x - M), fp = ex2(st.z - M);
      const float inv_l = 1.0f / (fr * st.y + fp * st.w);
      const float4 yp = reinterpret_cast<const float4*>(ps + j * 128)[lane];
      res = make_float4((fr * o[i][0] + fp * yp.x) * inv_l, (fr * o[i][1] + fp * yp.y) * inv_l,
                        (fr * o[i][2] + fp * yp.z) * inv_l, (fr * o[i][3] + fp * yp.w) * inv_l);
    }
    *reinterpret_cast<float4*>(a.out + ((size_t)(b * a.chunk + qi) * a.Hq + h * g + n) * kD + 4 * lane) = res;
  }
}
static_assert(kMgRows == 2 * (kMgThreads / 32), "two rows a warp in the R_V^T product");

constexpr size_t decode_smem_bytes() { return kSlotsOffset + (size_t)kBf16Slots * kPartialFloats * sizeof(float); }
// a warp state fits in one stage (the rotated-basis one in the warp's first
// stage, the comparator's original-basis one in its second); the block
// merge's partial products with R_V^T fit in the first two stages of all
// warps, below warp 0's last stage, which holds the staged accumulators; the
// final merge's stash fits in all of it
static_assert(kPartialFloats * 4 <= kBlockBytes && kRvBytes <= kBlockBytes && kMaxG * kD * 4 <= kBlockBytes,
              "states, R_V^T rows and staged accumulators in one stage");
static_assert(kWarps * kMaxG * kD * 4 <= (kStages - 1) * kWarps * kBlockBytes, "block merge products");
static_assert(kWarps * kStash * 4 <= kWarps * kStages * kBlockBytes, "final merge stash");
static_assert(kWarps * kStages * kBlockBytes / 4 / (16 + 128 * kMaxG) >= 1, "a record batch holds a record");

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
  // Pages per work item C: the split whose waves of blocks (one block per
  // SM) finish first.  A block costs a fixed amount -- the q rotation, the
  // pipeline's first copies, the block merge with its R_V^T product -- about
  // what 32 INT2 pages take its 16 warps (measured at 100K tokens: ~5 us
  // against ~2.5 us per page per warp), plus its C pages; a BF16 page streams
  // ~7x the bytes, so there the fixed part is ~5 pages.  At batch 1 this
  // gives one wave of ~num_sms blocks; at large batches a few long items per
  // (request, KV head) instead of many short ones.
  const long long bh_count = (long long)batch * Hkv;
  const long long slots = num_sms > 0 ? num_sms : 148;
  const long long fixed = mode == 0 ? 2 * kWarps : 5;
  long long C = 2;
  if (pages > 0 && bh_count > 0) {
    long long best = -1;
    for (long long n = 1; n <= kMaxChunks && n <= pages; ++n) {
      const long long c = (pages + n - 1) / n;
      if (c < 2 && n > 1) break;
      const long long items = (pages + c - 1) / c;
      const long long waves = (bh_count * items + slots - 1) / slots;
      const long long cost = waves * (fixed + c);
      if (best < 0 || cost < best) {
        best = cost;
        C = c;
      }
    }
  }
  if (C < 2) C = 2;
  if (pages > C * kMaxChunks) C = (pages + kMaxChunks - 1) / kMaxChunks;
  // The last item holds the newest history page, so in a decode step it is
  // also the block that appends the token and moves the evicted row into
  // INT2 (a few microseconds at the start).  Give it about one page per warp
  // less than the others when that keeps the item count.
  if (mode == 0 && pages > C) {
    const long long n = (pages + C - 1) / C;
    const long long C2 = (pages + kWarps + n - 1) / n;
    if (C2 > C && (pages + C2 - 1) / C2 == n) C = C2;
  }
  p.chunk_pages = (int)C;
  p.n_chunks = pages > 0 ? (int)((pages + C - 1) / C) : 0;
  p.n_items = p.n_chunks > 0 ? p.n_chunks : 1;
  // BF16 tiles go to the first items, two warps each (the last two, which
  // hold the fewest left-over INT2 tiles); they run while those warps' first
  // pages arrive
  p.tiles_per_item = max(kBf16Slots, (kBf16Tiles + p.n_items - 1) / p.n_items);
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
  p.rec_floats = partial_record_floats(p.g);
  off = align256(off + bh * (size_t)p.n_items * p.rec_floats * sizeof(float));
  p.prep_rows = prep_rows_per_block(batch, Hkv, num_sms);
  p.total = off;
  return p;
}

namespace {

PrepArgs prep_args_of(const DecodeLaunch& d) {
  const DecodePlan& p = d.plan;
  uint8_t* ws = d.workspace;
  PrepArgs pa;
  pa.q = d.q;
  pa.R_K = d.rot.R_K;
  pa.rot_flags = d.rot.flags;
  pa.sm_scale = d.sm_scale;
  pa.Hq = p.Hq;
  pa.Hkv = p.Hkv;
  pa.g = p.g;
  pa.qfrag = reinterpret_cast<uint32_t*>(ws + p.off_qfrag);
  pa.qplain = reinterpret_cast<uint32_t*>(ws + p.off_qplain);
  pa.qconst = reinterpret_cast<float*>(ws + p.off_qconst);
  pa.counters = reinterpret_cast<int*>(ws + p.off_counters);
  pa.nb = p.batch;
  pa.per_block = p.prep_rows;
  return pa;
}

DecodeArgs decode_args_of(const DecodeLaunch& d, const PrepArgs& pa) {
  const DecodePlan& p = d.plan;
  uint8_t* ws = d.workspace;
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
  a.tiles_per_item = p.tiles_per_item;
  a.rec_floats = p.rec_floats;
  a.qfrag = pa.qfrag;
  a.qplain = pa.qplain;
  a.qconst = pa.qconst;
  a.partials = reinterpret_cast<float*>(ws + p.off_partials);
  a.counters = pa.counters;
  a.R_VT = d.rot.R_VT;
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
  a.limit = d.limit;
  a.rot_flags = d.rot.flags;
  a.q = d.q;
  a.sm_scale = d.sm_scale;
  return a;
}

// the split-K decode kernel (after its prep has been queued)
cudaError_t launch_decode_kernel(const DecodeLaunch& d, const PrepArgs& pa, cudaStream_t stream) {
  const DecodePlan& p = d.plan;
  DecodeArgs a = decode_args_of(d, pa);
  const size_t smem = decode_smem_bytes();
  const dim3 grid(p.n_items, p.Hkv, p.batch);
  const bool pack4 = p.g <= 4;
  const bool lim = d.limit != nullptr;
  void (*kern)(DecodeArgs) =
      d.mode == 0 ? (lim ? (pack4 ? decode_kernel<0, true, true> : decode_kernel<0, false, true>)
                         : (pack4 ? decode_kernel<0, true> : decode_kernel<0, false>))
                  : (pack4 ? decode_kernel<1, true> : decode_kernel<1, false>);
  static std::atomic<uint64_t> attr_done[6];
  const int which = (lim ? 4 : 2 * d.mode) + (pack4 ? 1 : 0);
  const cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(kern), smem, attr_done[which]);
  if (e != cudaSuccess) return e;
  void* args[] = {&a};
  return launch_pdl(reinterpret_cast<const void*>(kern), grid, dim3(kThreads), smem, stream, args);
}

}  // namespace

ExtendPlan plan_extend(int batch, int chunk, int Hq, int Hkv, int max_ctx_len, int num_sms) {
  ExtendPlan p;
  p.batch = batch;
  p.chunk = chunk;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.qpg = 128 / p.g;  // the group's (query, head) pairs are the 128 rows of the MMAs
  p.ngpr = (chunk + p.qpg - 1) / p.qpg;
  const int hist_end = max_ctx_len > kSink + kRecent ? max_ctx_len - kRecent : kSink;
  int pages = (hist_end + kPage - 1) / kPage - 1;
  if (pages < 0) pages = 0;
  // Pages per page range C: the split whose waves of blocks (one block per SM)
  // and records' merge finish first.  In units of one page's period (~1.5 us
  // at 100K tokens): a block's fixed work (q' staging, the BF16 tiles, its
  // records) ~8, and every page range ~3 more of records to merge.
  const long long pairs = (long long)batch * p.ngpr * Hkv;
  const long long slots = num_sms > 0 ? num_sms : 148;
  long long C = 2;
  if (pages > 0 && pairs > 0) {
    long long best = -1;
    for (long long n = 1; n <= kMaxChunks && n <= pages; ++n) {
      const long long c = (pages + n - 1) / n;
      if (c < 2 && n > 1) break;
      const long long items = (pages + c - 1) / c;
      const long long waves = (pairs * items + slots - 1) / slots;
      const long long cost = waves * (8 + c) + 3 * items;
      if (best < 0 || cost < best) {
        best = cost;
        C = c;
      }
    }
  }
  if (C < 2) C = 2;
  if (pages > C * kMaxChunks) C = (pages + kMaxChunks - 1) / kMaxChunks;
  p.chunk_pages = (int)C;
  p.n_items = pages > 0 ? (int)((pages + C - 1) / C) : 1;
  p.tiles_per_item = (kBf16Tiles + p.n_items - 1) / p.n_items;
  const size_t nq = (size_t)batch * chunk, bq = nq * Hkv;
  size_t off = 0;
  p.off_counters = off;
  off = align256(off + bq * sizeof(int));
  p.off_qfrag = off;
  off = align256(off + bq * kQFragWords * sizeof(uint32_t));
  p.off_qplain = off;
  off = align256(off + bq * kQFragWords * sizeof(uint32_t));
  p.off_qconst = off;
  off = align256(off + bq * kQConstFloats * sizeof(float));
  p.off_partials = off;
  off = align256(off + bq * (size_t)p.n_items * 2 * kPartialFloats * sizeof(float));
  p.prep_rows = prep_rows_per_block(batch * chunk, Hkv, num_sms);
  p.total = off;
  return p;
}

cudaError_t launch_extend(const ExtendLaunch& e, cudaStream_t stream) {
  const ExtendPlan& p = e.plan;
  if (p.batch == 0 || p.chunk == 0) return cudaSuccess;
  uint8_t* ws = e.workspace;
  PrepArgs pa;
  pa.q = e.q;
  pa.R_K = e.rot.R_K;
  pa.rot_flags = e.rot.flags;
  pa.sm_scale = e.sm_scale;
  pa.Hq = p.Hq;
  pa.Hkv = p.Hkv;
  pa.g = p.g;
  pa.qfrag = reinterpret_cast<uint32_t*>(ws + p.off_qfrag);
  pa.qplain = reinterpret_cast<uint32_t*>(ws + p.off_qplain);
  pa.qconst = reinterpret_cast<float*>(ws + p.off_qconst);
  pa.counters = reinterpret_cast<int*>(ws + p.off_counters);
  pa.nb = p.batch * p.chunk;
  pa.per_block = p.prep_rows;
  void* pargs[] = {&pa};
  cudaError_t err = launch_pdl(reinterpret_cast<const void*>(prep_kernel),
                               dim3(p.Hkv, (pa.nb + p.prep_rows - 1) / p.prep_rows), dim3(kPrepThreads), 0, stream,
                               pargs);
  if (err != cudaSuccess) return err;
  ExtendArgs a;
  a.c = e.c;
  a.ctx_len = e.ctx_len;
  a.pos0 = e.pos0;
  a.chunk = p.chunk;
  a.ngpr = p.ngpr;
  a.qpg = p.qpg;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.g = p.g;
  a.n_items = p.n_items;
  a.chunk_pages = p.chunk_pages;
  a.tiles_per_item = p.tiles_per_item;
  a.qfrag = pa.qfrag;
  a.qplain = pa.qplain;
  a.qconst = pa.qconst;
  a.partials = reinterpret_cast<float*>(ws + p.off_partials);
  a.R_VT = e.rot.R_VT;
  {
    const float smax = std::isfinite(e.rot.tau_v) ? fminf(65504.f, e.rot.tau_v / 1.5f * 1.001f) : 65504.f;
    int k = (int)floorf(log2f(60000.f / (16.f * smax)));
    k = k < -20 ? -20 : (k > 20 ? 20 : k);
    a.pscale = ldexpf(1.f, k);
    a.inv_pscale = ldexpf(1.f, -k);
  }
  a.out = e.out;
  a.err = e.err;
  static std::atomic<uint64_t> attr_done;
  err = smem_attr_once(reinterpret_cast<const void*>(extend_tc_kernel), kXtSmem, attr_done);
  if (err != cudaSuccess) return err;
  void* args[] = {&a};
  err = launch_pdl(reinterpret_cast<const void*>(extend_tc_kernel), dim3(p.Hkv, p.batch * p.ngpr, p.n_items),
                   dim3(kXtThreads), kXtSmem, stream, args);
  if (err != cudaSuccess) return err;
  static std::atomic<uint64_t> attr_done_mg;
  err = smem_attr_once(reinterpret_cast<const void*>(extend_merge_kernel), kMgSmem, attr_done_mg);
  if (err != cudaSuccess) return err;
  return launch_pdl(reinterpret_cast<const void*>(extend_merge_kernel), dim3(p.Hkv, p.batch * p.ngpr, 128 / kMgRows),
                    dim3(kMgThreads), kMgSmem, stream, args);
}

cudaError_t launch_decode(const DecodeLaunch& d, cudaStream_t stream) {
  const DecodePlan& p = d.plan;
  if (p.batch == 0) return cudaSuccess;
  PrepArgs pa = prep_args_of(d);
  void* args[] = {&pa};
  cudaError_t e = launch_pdl(reinterpret_cast<const void*>(prep_kernel),
                             dim3(p.Hkv, (p.batch + p.prep_rows - 1) / p.prep_rows), dim3(kPrepThreads), 0, stream,
                             args);
  if (e != cudaSuccess) return e;
  return launch_decode_kernel(d, pa, stream);
}

cudaError_t launch_decode_step(const AppendLaunch& ap, const DecodeLaunch& d, cudaStream_t stream) {
  const DecodePlan& p = d.plan;
  if (p.batch == 0) return cudaSuccess;
  const PrepArgs pa = prep_args_of(d);
  DecodeArgs a = decode_args_of(d, pa);
  StepArgs sa;
  sa.ap = ap;
  sa.pr = pa;
  const size_t smem = kPatchOffset + sizeof(RowPatch);
  const bool pack4 = p.g <= 4;
  void (*kern)(DecodeArgs, StepArgs) = pack4 ? decode_step_kernel<true> : decode_step_kernel<false>;
  static std::atomic<uint64_t> attr_done[2];
  const cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(kern), smem, attr_done[pack4 ? 1 : 0]);
  if (e != cudaSuccess) return e;
  void* args[] = {&a, &sa};
  return launch_pdl(reinterpret_cast<const void*>(kern), dim3(p.n_items, p.Hkv, p.batch), dim3(kThreads), smem,
                    stream, args);
}

}  // namespace oscar
