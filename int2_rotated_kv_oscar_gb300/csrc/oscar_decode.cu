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
//    Walsh-Hadamard butterfly, bit reversal), folded with sm_scale * log2(e)
//    and a power-of-two normalisation into fp16 tensor-core B fragments whose
//    per-channel power-of-two factors match the code unpacking below; the
//    plain q for the BF16 segment likewise; zeroes the split counters.
//  * decode kernel, one block per (work item, KV head, request), 4 warps.
//    Work items are chunks of INT2 history pages (rotated basis) or 64-token
//    BF16 blocks (sink, ring quarters; original basis).  Each warp streams
//    its pages through a private ring of shared-memory stages filled by bulk
//    asynchronous copies (one 4608-byte copy per page), unpacks the 2-bit
//    codes in registers with one AND per fp16 pair (a code c masked in place
//    at bit 2r of an fp16 is the subnormal value c * 2^(2r-24); the 2^(24-2r)
//    factor lives in the other operand or is applied to the accumulator),
//    runs QK^T and PV on mma.sync m16n8k16 (tokens x channels, channels x
//    heads) with an online softmax in the log2 domain, and folds the -1.5
//    code offset in exactly (accumulator initialisation for K, a ones-row
//    MMA for V).  Warps merge in shared memory; each block writes one partial
//    (m, l, acc); the last block of a (request, KV head) merges all partials
//    (log-sum-exp), rotates the INT2 part back (acc P H U_V^T) and writes the
//    fp32 output.  No block ever waits on another.

#include "oscar_device.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kInvSqrtD = 0.08838834764831845f;
constexpr int kWarps = 4;
constexpr int kStages = 3;
constexpr unsigned kWaitLimit = 1u << 22;
constexpr uint32_t kOnesF16x2 = 0x3C003C00u;
constexpr float kPScale = 1.0f / 256.0f;  // B operand = p * s * 2^-8 keeps lazily-rescaled p in fp16 range
constexpr float kLazy = 8.0f;             // rescale only when the max grows by more than 2^8

// exponent of the fp16 value of a code masked in place at index r of a 16-bit half
__host__ __device__ constexpr int code_exp(int r) { return r < 5 ? 2 * r - 24 : 2 * r - 30; }

// fp16 pair of the codes at index r (0..7) of both halves of w, masked in place
template <int R>
__device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t ws) {
  return R < 5 ? (w & (0x00030003u << (2 * R))) : (ws & (0x00030003u << (2 * (R - 3))));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
__global__ void __launch_bounds__(128) prep_kernel(PrepArgs a) {
  __shared__ float xs[kMaxG][kD];
  __shared__ float qr[kMaxG][kD];
  __shared__ float qp[kMaxG][kD];
  __shared__ float scratch[kD];
  __shared__ float red[8];
  const int h = blockIdx.x, b = blockIdx.y, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int g = a.g, bh = b * a.Hkv + h;
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
  for (int n = 0; n < g; ++n) {
    float v = z[n];
    if (a.flags & kRotH) v = fwht128_block(v, scratch) * kInvSqrtD;
    qr[n][t] = v;
  }
  __syncthreads();
  for (int n = 0; n < g; ++n) {
    const float v = (a.flags & kRotP) ? qr[n][brev7(t)] : qr[n][t];
    z[n] = v * c;
    qp[n][t] = xs[n][t] * c;
  }
  __syncthreads();
  for (int n = 0; n < g; ++n) qr[n][t] = z[n];
  // power-of-two normalisations: max |q'| * 2^-E <= 2^-9, max |q| * 2^-Ep <= 2^10
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
    er += 9;
  }
  if (mp > 0.f) {
    frexpf(mp, &ep);
    ep -= 10;
  }
  const float sr = ldexpf(1.f, -er), sp = ldexpf(1.f, -ep);
  // B fragments for QK over the INT2 history: lane L = 4 n + tig holds, for
  // MMA i (group i / 4, r0 = 2 (i % 4)), b0 = q'[n][64 grp + 16 tig + {0, 8} + r0]
  // and b1 = the same at r0 + 1, each times 2^(-code_exp(r)).
  uint32_t* qf = a.qfrag + (size_t)bh * 512;
  uint32_t* qpl = a.qplain + (size_t)bh * 512;
  for (int e = t; e < 512; e += 128) {
    const int L = e >> 4, w = e & 15, i = w >> 1, bs = w & 1;
    const int n = L >> 2, tig = L & 3;
    uint32_t vr = 0, vp = 0;
    if (n < g) {
      const int grp = i >> 2, r = 2 * (i & 3) + bs;
      const int ch = 64 * grp + 16 * tig + r;
      const float f = sr * ldexpf(1.f, -code_exp(r));
      vr = pack_f16x2(qr[n][ch] * f, qr[n][ch + 8] * f);
      // BF16 segment: MMA ks = i covers channels 32 tig + 4 ks + {0,1} (b0), {2,3} (b1)
      const int cp = 32 * tig + 4 * i + 2 * bs;
      vp = pack_f16x2(qp[n][cp] * sp, qp[n][cp + 1] * sp);
    }
    qf[L * 16 + w] = vr;
    qpl[L * 16 + w] = vp;
  }
  // -1.5 * sum over each group of the exact fp16 values the MMA multiplies
  float* qc = a.qconst + (size_t)bh * kQConstFloats;
  for (int n = 0; n < kMaxG; ++n) {
    float v = 0.f;
    if (n < g) {
      const int r = t & 7;
      const float f = ldexpf(1.f, -code_exp(r));
      v = __half2float(__float2half_rn(qr[n][t] * sr * f)) * ldexpf(1.f, code_exp(r));
    }
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (t == 0) {
      qc[2 * n + 0] = -1.5f * (red[0] + red[1]);
      qc[2 * n + 1] = -1.5f * (red[2] + red[3]);
    }
  }
  if (t == 0) {
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
  float* out;
  unsigned* err;
};

struct WarpState {
  float m[2], l[2];
  float acc[8][4];
  float corr[2][4];
};

__device__ __forceinline__ void state_init(WarpState& st) {
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) st.acc[i][k] = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) st.corr[i][k] = 0.f;
}

// Update the running maxima with this page's maxima (per lane: heads 2 tig, 2 tig + 1).
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
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      st.corr[i][0] *= a0;
      st.corr[i][2] *= a0;
      st.corr[i][1] *= a1;
      st.corr[i][3] *= a1;
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

// One 64-token INT2 page (K and V codes + scales) staged in shared memory.
__device__ __forceinline__ void int2_page(const uint8_t* __restrict__ blk, int n_valid, const uint32_t (&qf)[16],
                                          const float (&qi)[4], float scaleE, WarpState& st, int lane) {
  const int q = lane >> 2;
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
    float d0[4] = {qi[0], qi[1], qi[0], qi[1]};
    float d1[4] = {qi[2], qi[3], qi[2], qi[3]};
    {
      const uint32_t x = kw.x, y = kw.z, xs = x >> 6, ys = y >> 6;  // group 0: token q, token q+8
      mma_f16(d0, code_pair<0>(x, xs), code_pair<0>(y, ys), code_pair<1>(x, xs), code_pair<1>(y, ys), qf[0], qf[1]);
      mma_f16(d0, code_pair<2>(x, xs), code_pair<2>(y, ys), code_pair<3>(x, xs), code_pair<3>(y, ys), qf[2], qf[3]);
      mma_f16(d0, code_pair<4>(x, xs), code_pair<4>(y, ys), code_pair<5>(x, xs), code_pair<5>(y, ys), qf[4], qf[5]);
      mma_f16(d0, code_pair<6>(x, xs), code_pair<6>(y, ys), code_pair<7>(x, xs), code_pair<7>(y, ys), qf[6], qf[7]);
    }
    {
      const uint32_t x = kw.y, y = kw.w, xs = x >> 6, ys = y >> 6;  // group 1
      mma_f16(d1, code_pair<0>(x, xs), code_pair<0>(y, ys), code_pair<1>(x, xs), code_pair<1>(y, ys), qf[8], qf[9]);
      mma_f16(d1, code_pair<2>(x, xs), code_pair<2>(y, ys), code_pair<3>(x, xs), code_pair<3>(y, ys), qf[10],
              qf[11]);
      mma_f16(d1, code_pair<4>(x, xs), code_pair<4>(y, ys), code_pair<5>(x, xs), code_pair<5>(y, ys), qf[12],
              qf[13]);
      mma_f16(d1, code_pair<6>(x, xs), code_pair<6>(y, ys), code_pair<7>(x, xs), code_pair<7>(y, ys), qf[14],
              qf[15]);
    }
    const bool va = 16 * T + q < n_valid, vb = 16 * T + q + 8 < n_valid;
    lg[T][0] = va ? fmaf(d0[0], sa.x, d1[0] * sa.y) * scaleE : -INFINITY;
    lg[T][1] = va ? fmaf(d0[1], sa.x, d1[1] * sa.y) * scaleE : -INFINITY;
    lg[T][2] = vb ? fmaf(d0[2], sb.x, d1[2] * sb.y) * scaleE : -INFINITY;
    lg[T][3] = vb ? fmaf(d0[3], sb.x, d1[3] * sb.y) * scaleE : -INFINITY;
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
    float2 va_s = half2_bits_to_float2(*reinterpret_cast<const uint32_t*>(blk + kVScales + 4 * (16 * T + q)));
    float2 vb_s = half2_bits_to_float2(*reinterpret_cast<const uint32_t*>(blk + kVScales + 4 * (16 * T + q + 8)));
    va_s.x = va ? va_s.x * kPScale : 0.f;
    va_s.y = va ? va_s.y * kPScale : 0.f;
    vb_s.x = vb ? vb_s.x * kPScale : 0.f;
    vb_s.y = vb ? vb_s.y * kPScale : 0.f;
    const uint32_t b00 = movmatrix_trans(pack_f16x2(p0 * va_s.x, p1 * va_s.x));
    const uint32_t b01 = movmatrix_trans(pack_f16x2(p2 * vb_s.x, p3 * vb_s.x));
    const uint32_t b10 = movmatrix_trans(pack_f16x2(p0 * va_s.y, p1 * va_s.y));
    const uint32_t b11 = movmatrix_trans(pack_f16x2(p2 * vb_s.y, p3 * vb_s.y));
    const uint4 vw = *reinterpret_cast<const uint4*>(blk + kVCodes + 512 * T + 16 * lane);
    const uint32_t w0 = vw.x, w1 = vw.y, w2 = vw.z, w3 = vw.w;
    const uint32_t s0 = w0 >> 6, s1 = w1 >> 6, s2 = w2 >> 6, s3 = w3 >> 6;
#define OSCAR_PV(M, B0, B1)                                                                                  \
  mma_f16(st.acc[M], code_pair<M>(w0, s0), code_pair<M>(w1, s1), code_pair<M>(w2, s2), code_pair<M>(w3, s3), \
          B0, B1)
    OSCAR_PV(0, b00, b01);
    OSCAR_PV(1, b00, b01);
    OSCAR_PV(2, b00, b01);
    OSCAR_PV(3, b00, b01);
    OSCAR_PV(4, b10, b11);
    OSCAR_PV(5, b10, b11);
    OSCAR_PV(6, b10, b11);
    OSCAR_PV(7, b10, b11);
#undef OSCAR_PV
    mma_f16(st.corr[0], kOnesF16x2, kOnesF16x2, kOnesF16x2, kOnesF16x2, b00, b01);
    mma_f16(st.corr[1], kOnesF16x2, kOnesF16x2, kOnesF16x2, kOnesF16x2, b10, b11);
  }
}

// One 16-token BF16 tile (rows of K and V in global memory, original basis).
__device__ __forceinline__ void bf16_tile(const uint16_t* __restrict__ Kt, const uint16_t* __restrict__ Vt, int n_valid,
                                          const uint32_t (&qpf)[16], float scaleEp, WarpState& st, int lane) {
  const int q = lane >> 2, tig = lane & 3;
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
  float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) mma_f16(d, ka[2 * ks], kb[2 * ks], ka[2 * ks + 1], kb[2 * ks + 1], qpf[2 * ks], qpf[2 * ks + 1]);
  const float l0 = va ? d[0] * scaleEp : -INFINITY, l1 = va ? d[1] * scaleEp : -INFINITY;
  const float l2 = vb ? d[2] * scaleEp : -INFINITY, l3 = vb ? d[3] * scaleEp : -INFINITY;
  online_max(st, fmaxf(l0, l2), fmaxf(l1, l3));
  const float p0 = ex2(l0 - st.m[0]), p1 = ex2(l1 - st.m[1]), p2 = ex2(l2 - st.m[0]), p3 = ex2(l3 - st.m[1]);
  st.l[0] += p0 + p2;
  st.l[1] += p1 + p3;
  const uint32_t b0 = movmatrix_trans(pack_f16x2(p0 * kPScale, p1 * kPScale));
  const uint32_t b1 = movmatrix_trans(pack_f16x2(p2 * kPScale, p3 * kPScale));
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t a[4];
#pragma unroll
    for (int blkid = 0; blkid < 4; ++blkid) {
      const int tr = blkid >> 1, cc = blkid & 1;  // token half, channel half
      const bool ok = tr ? vb : va;
      const uint32_t u = ok ? __ldg(reinterpret_cast<const uint32_t*>(Vt + (8 * tr + q) * kD + 16 * mt + 8 * cc + 2 * tig))
                            : 0u;
      a[blkid] = movmatrix_trans(bf16x2_to_f16x2(u));
    }
    // a[0]: channels 16mt+q, tokens 2tig..; a[1]: channels +8; a[2]: tokens +8; a[3]: both
    mma_f16(st.acc[mt], a[0], a[1], a[2], a[3], b0, b1);
  }
}

struct MergeSmem {
  float m[kWarps][8];
  float l[kWarps][8];
  float acc[kWarps][8][kD];
};

template <int MODE>
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
      uint32_t qf[16];
      {
        const uint4* src = reinterpret_cast<const uint4*>(a.qfrag + (size_t)bh * 512 + lane * 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 u = __ldg(src + k);
          qf[4 * k] = u.x;
          qf[4 * k + 1] = u.y;
          qf[4 * k + 2] = u.z;
          qf[4 * k + 3] = u.w;
        }
      }
      const float* qc = a.qconst + (size_t)bh * kQConstFloats;
      const float qi[4] = {__ldg(qc + 2 * (2 * tig) + 0), __ldg(qc + 2 * (2 * tig + 1) + 0), __ldg(qc + 2 * (2 * tig) + 1),
                           __ldg(qc + 2 * (2 * tig + 1) + 1)};
      const float scaleE = __ldg(qc + 16);
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
          int2_page(stages + (size_t)s * kBlockBytes, n_valid, qf, qi, scaleE, st, lane);
        }
        __syncwarp();
        if (lane == 0 && k + kStages < n_my) {
          fence_proxy_async_smem();
          issue(k + kStages);
        }
      }
      // after a timeout, wait (bounded) for the copies still in flight
      for (int kk = k + 1; kk < min(k + kStages, n_my); ++kk) mbar_wait_bounded(&bars[kk % kStages], (kk / kStages) & 1, kWaitLimit);
      if (k < n_my) mbar_wait_bounded(&bars[k % kStages], (k / kStages) & 1, kWaitLimit);
    }
  } else {
    // ---------------- BF16 tiles (original basis)
    uint32_t qpf[16];
    {
      const uint4* src = reinterpret_cast<const uint4*>(a.qplain + (size_t)bh * 512 + lane * 16);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
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
      if (nv > 0) bf16_tile(Kb + 16 * warp * kD, Vb + 16 * warp * kD, nv, qpf, scaleEp, st, lane);
    } else {
      // plain BF16 paged cache: item covers pages [item*C, item*C + C)
      const int n_pages = (L + kPage - 1) / kPage;
      if (n_pages > c.max_pages) {
        if (t == 0 && item == 0) set_error(a.err, kErrLength);
      }
      const int pg0 = item * a.chunk_pages;
      const int pg1 = min(min(pg0 + a.chunk_pages, n_pages), c.max_pages);
      for (int tt = warp; (pg0 + tt / 4) < pg1; tt += kWarps) {
        const int pg = pg0 + tt / 4, tile = tt & 3;
        const int ph = c.page_table[(size_t)b * c.max_pages + pg];
        if (ph < 0 || ph >= c.num_pages) {
          if (lane == 0) set_error(a.err, kErrPage);
          continue;
        }
        const int nv = min(16, L - kPage * pg - 16 * tile);
        if (nv <= 0) continue;
        const size_t off = (((size_t)ph * a.Hkv + h) * kPage + 16 * tile) * kD;
        bf16_tile(a.kb_pages + off, a.vb_pages + off, nv, qpf, scaleEp, st, lane);
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
  if (q == 0) {
    ms.m[warp][2 * tig] = st.m[0];
    ms.m[warp][2 * tig + 1] = st.m[1];
    ms.l[warp][2 * tig] = st.l[0];
    ms.l[warp][2 * tig + 1] = st.l[1];
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const float f = rotated ? ldexpf(256.f, -code_exp(mt)) : 256.f;
    const int grp = mt >> 2;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = 16 * mt + q + 8 * (i >> 1), n = 2 * tig + (i & 1);
      float v = st.acc[mt][i] * f;
      if (rotated) v = fmaf(-1.5f * 256.f, st.corr[grp][i & 1], v);
      ms.acc[warp][n][ch] = v;
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
    for (int n = 0; n < a.g; ++n) ys[n * kD + t] = Ar[n];
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
  off = align256(off + bh * 512 * sizeof(uint32_t));
  p.off_qplain = off;
  off = align256(off + bh * 512 * sizeof(uint32_t));
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
  a.out = d.out;
  a.err = d.err;
  const size_t smem = decode_smem_bytes();
  static bool attr0 = false, attr1 = false;
  const dim3 grid(p.n_items, p.Hkv, p.batch);
  if (d.mode == 0) {
    if (!attr0) {
      e = cudaFuncSetAttribute(decode_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr0 = true;
    }
    decode_kernel<0><<<grid, 128, smem, stream>>>(a);
  } else {
    if (!attr1) {
      e = cudaFuncSetAttribute(decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr1 = true;
    }
    decode_kernel<1><<<grid, 128, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace oscar
