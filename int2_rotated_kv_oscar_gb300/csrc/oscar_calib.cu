// Offline calibration on the GPU: the second-moment matrices C_Q and C_S and
// the clip thresholds of one layer (the eigendecomposition stays on the host).
//
// edge.aivizor.me "Together AI выпустила исходники OSCAR ...", paragraph
// "Техническая идея": C_Q = (1/N) sum_n q_n^T q_n for the keys' rotation and
// the score-weighted C_S = (1/N) V^T S^T S V for the values' one.
// gist.science "Resumen Técnico: OSCAR ...", §2.2 A, steps 1-4: both
// covariances on a small calibration set, spectral decomposition, R = U H P,
// and per-layer clip thresholds estimated from the rotated calibration
// activations (here: a percentile of |x R|, linearly interpolated).
#include <cstdint>
#include <cuda_runtime.h>

#include "oscar_internal.h"

namespace oscar {
namespace {

constexpr int kD = 128;

// ---------------------------------------------------------------- C = s X^T X
// Partial products of 16 x 16 output tiles over one slice of the rows, fp32
// inside a 32-row stage, fp64 across stages; grid (8, 8, parts), 256 threads.
constexpr int kGramRows = 32;

__global__ void __launch_bounds__(256) gram_partial_kernel(const float* __restrict__ X, int64_t n_rows,
                                                           int64_t rows_per_part, double* __restrict__ partial) {
  __shared__ float xi[kGramRows][16], xj[kGramRows][16];
  const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
  const int i0 = 16 * blockIdx.x, j0 = 16 * blockIdx.y;
  const int64_t r0 = (int64_t)blockIdx.z * rows_per_part;
  const int64_t r1 = r0 + rows_per_part < n_rows ? r0 + rows_per_part : n_rows;
  double acc = 0.0;
  for (int64_t rs = r0; rs < r1; rs += kGramRows) {
    for (int e = threadIdx.x; e < kGramRows * 16; e += 256) {
      const int rr = e >> 4, cc = e & 15;
      const int64_t r = rs + rr;
      xi[rr][cc] = r < r1 ? X[r * kD + i0 + cc] : 0.f;
      xj[rr][cc] = r < r1 ? X[r * kD + j0 + cc] : 0.f;
    }
    __syncthreads();
    float s = 0.f;
#pragma unroll 8
    for (int rr = 0; rr < kGramRows; ++rr) s = fmaf(xi[rr][ti], xj[rr][tj], s);
    acc += (double)s;
    __syncthreads();
  }
  partial[((int64_t)blockIdx.z * kD + i0 + ti) * kD + j0 + tj] = acc;
}

// C[i][j] = scale * (sum over parts, in part order) -- deterministic
__global__ void gram_reduce_kernel(const double* __restrict__ partial, int parts, double scale, double* __restrict__ C,
                                   int accumulate) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= kD * kD) return;
  double s = 0.0;
  for (int p = 0; p < parts; ++p) s += partial[(int64_t)p * kD * kD + e];
  C[e] = accumulate ? C[e] + scale * s : scale * s;
}

// ---------------------------------------------------------------- O = softmax(Q K^T scale) V
// One KV head and 32 queries per block (8 warps x 4 queries); keys and values
// staged 32 rows at a time; lane = key for the logits, lane + 32 c = channel
// for the output.  Online softmax in fp32 with accurate exponentials.
constexpr int kAttnQ = 32, kAttnK = 32;

__global__ void __launch_bounds__(256) calib_attention_kernel(const float* __restrict__ Q, int64_t n_q,
                                                              const float* __restrict__ K,
                                                              const float* __restrict__ V, int64_t n_k,
                                                              float sm_scale, float* __restrict__ O) {
  extern __shared__ float asm_[];  // queries [32][128], keys [32][129] (padded), values [32][128]
  float(*qs)[kD] = reinterpret_cast<float(*)[kD]>(asm_);
  float(*ks)[kD + 1] = reinterpret_cast<float(*)[kD + 1]>(asm_ + kAttnQ * kD);
  float(*vs)[kD] = reinterpret_cast<float(*)[kD]>(asm_ + kAttnQ * kD + kAttnK * (kD + 1));
  const int h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t q0 = (int64_t)blockIdx.x * kAttnQ;
  const float* Kh = K + (int64_t)h * n_k * kD;
  const float* Vh = V + (int64_t)h * n_k * kD;
  for (int e = threadIdx.x; e < kAttnQ * kD; e += 256) {
    const int r = e / kD, c = e % kD;
    qs[r][c] = q0 + r < n_q ? Q[(q0 + r) * kD + c] : 0.f;
  }
  float m[4], l[4], acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;
  }
  for (int64_t k0 = 0; k0 < n_k; k0 += kAttnK) {
    __syncthreads();  // the previous tile is consumed (and the queries are staged)
    for (int e = threadIdx.x; e < kAttnK * kD; e += 256) {
      const int r = e / kD, c = e % kD;
      const bool ok = k0 + r < n_k;
      ks[r][c] = ok ? Kh[(k0 + r) * kD + c] : 0.f;
      vs[r][c] = ok ? Vh[(k0 + r) * kD + c] : 0.f;
    }
    __syncthreads();
    const bool key_ok = k0 + lane < n_k;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int qi = 4 * warp + i;
      float z = 0.f;
#pragma unroll 16
      for (int c = 0; c < kD; ++c) z = fmaf(qs[qi][c], ks[lane][c], z);
      z = key_ok ? z * sm_scale : -INFINITY;
      float mx = z;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float mn = fmaxf(m[i], mx);  // finite: every tile holds at least one key
      const float alpha = expf(m[i] - mn);
      const float p = expf(z - mn);
      float ps = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l[i] = l[i] * alpha + ps;
      m[i] = mn;
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[i][c] *= alpha;
      for (int k = 0; k < kAttnK; ++k) {
        const float pk = __shfl_sync(0xffffffffu, p, k);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][c] = fmaf(pk, vs[k][lane + 32 * c], acc[i][c]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t qn = q0 + 4 * warp + i;
    if (qn < n_q)
#pragma unroll
      for (int c = 0; c < 4; ++c) O[((int64_t)h * n_q + qn) * kD + lane + 32 * c] = acc[i][c] / l[i];
  }
}

// ---------------------------------------------------------------- |X R| and its order statistics
// keys[r * 128 + j] = bits of |(X R)[r][j]| (non-negative floats order as
// their bit patterns); entries past n_rows * 128 up to the padded size are
// +inf, so they sort last.  8 rows per block, R staged in shared memory.
__global__ void __launch_bounds__(256) rotate_abs_kernel(const float* __restrict__ X, int64_t n_rows,
                                                         const float* __restrict__ R, uint32_t* __restrict__ keys,
                                                         int64_t n_pad) {
  extern __shared__ float rsm[];  // [128][128]
  __shared__ float xs[8][kD];
  for (int e = threadIdx.x; e < kD * kD; e += 256) rsm[e] = R[e];
  const int64_t r0 = (int64_t)blockIdx.x * 8;
  for (int e = threadIdx.x; e < 8 * kD; e += 256) {
    const int64_t r = r0 + e / kD;
    xs[e / kD][e % kD] = r < n_rows ? X[r * kD + e % kD] : 0.f;
  }
  __syncthreads();
  const int row = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r = r0 + row;
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    const int j = lane + 32 * c4;
    float y = 0.f;
#pragma unroll 16
    for (int c = 0; c < kD; ++c) y = fmaf(xs[row][c], rsm[c * kD + j], y);
    const int64_t idx = r * kD + j;
    if (r < n_rows) keys[idx] = __float_as_uint(fabsf(y));
  }
  // padding, spread over the blocks
  for (int64_t e = n_rows * kD + (int64_t)blockIdx.x * 256 + threadIdx.x; e < n_pad; e += (int64_t)gridDim.x * 256)
    keys[e] = 0x7f800000u;
}

// Bitonic sort of n (a power of two >= 2048) keys, ascending.  A block
// handles 2048 consecutive keys in shared memory for every step with
// j < 2048; the larger steps run one launch each over global memory.
constexpr int kLocal = 2048;

__device__ __forceinline__ void compare_swap(uint32_t& a, uint32_t& b, bool ascending) {
  if ((a > b) == ascending) {
    const uint32_t t = a;
    a = b;
    b = t;
  }
}

// all steps k = 2 .. 2048 (first pass) or j = 1024 .. 1 of one k > 2048
__global__ void __launch_bounds__(1024) bitonic_local_kernel(uint32_t* __restrict__ keys, int64_t k_first,
                                                             int64_t k_last) {
  __shared__ uint32_t s[kLocal];
  const int64_t base = (int64_t)blockIdx.x * kLocal;
  s[threadIdx.x] = keys[base + threadIdx.x];
  s[threadIdx.x + 1024] = keys[base + threadIdx.x + 1024];
  __syncthreads();
  for (int64_t k = k_first; k <= k_last; k <<= 1) {
    for (int64_t j = (k >> 1) < kLocal / 2 ? (k >> 1) : kLocal / 2; j > 0; j >>= 1) {
      // thread t handles the pair (i, i ^ j) with i the t-th index whose bit j is clear
      const int t = threadIdx.x;
      const int i = (int)(((t / j) * 2 * j) + (t % j));
      const int64_t gi = base + i;
      const bool ascending = (gi & k) == 0;
      uint32_t a = s[i], b = s[i + j];
      compare_swap(a, b, ascending);
      s[i] = a;
      s[i + j] = b;
      __syncthreads();
    }
  }
  keys[base + threadIdx.x] = s[threadIdx.x];
  keys[base + threadIdx.x + 1024] = s[threadIdx.x + 1024];
}

__global__ void bitonic_global_kernel(uint32_t* __restrict__ keys, int64_t n, int64_t k, int64_t j) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n / 2) return;
  const int64_t i = (t / j) * 2 * j + (t % j);
  uint32_t a = keys[i], b = keys[i + j];
  compare_swap(a, b, (i & k) == 0);
  keys[i] = a;
  keys[i + j] = b;
}

}  // namespace

int gram_parts(int64_t n_rows) {
  const int64_t per = 256;
  int64_t parts = (n_rows + per - 1) / per;
  return (int)(parts < 1 ? 1 : parts);
}

cudaError_t launch_gram(const float* X, int64_t n_rows, double scale, double* C, bool accumulate, double* partial,
                        cudaStream_t stream) {
  const int parts = gram_parts(n_rows);
  const int64_t per = (n_rows + parts - 1) / parts;
  gram_partial_kernel<<<dim3(8, 8, parts), 256, 0, stream>>>(X, n_rows, per, partial);
  gram_reduce_kernel<<<(kD * kD + 255) / 256, 256, 0, stream>>>(partial, parts, scale, C, accumulate ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_calib_attention(const float* Q, int64_t n_q, const float* K, const float* V, int64_t n_k,
                                   int n_heads, float sm_scale, float* O, cudaStream_t stream) {
  const dim3 grid((unsigned)((n_q + kAttnQ - 1) / kAttnQ), (unsigned)n_heads);
  const int smem = (kAttnQ * kD + kAttnK * (kD + 1) + kAttnK * kD) * 4;
  static std::atomic<uint64_t> attr_done;
  const cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(calib_attention_kernel), smem, attr_done);
  if (e != cudaSuccess) return e;
  calib_attention_kernel<<<grid, 256, smem, stream>>>(Q, n_q, K, V, n_k, sm_scale, O);
  return cudaGetLastError();
}

int64_t sort_size(int64_t n) {
  int64_t p = kLocal;
  while (p < n) p <<= 1;
  return p;
}

cudaError_t launch_sorted_abs_rotated(const float* X, int64_t n_rows, const float* R, uint32_t* keys,
                                      cudaStream_t stream) {
  const int64_t n = sort_size(n_rows * kD);
  static std::atomic<uint64_t> attr_done;
  const cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(rotate_abs_kernel), kD * kD * 4, attr_done);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (n_rows + 7) / 8;
  rotate_abs_kernel<<<(unsigned)(blocks > 0 ? blocks : 1), 256, kD * kD * 4, stream>>>(X, n_rows, R, keys, n);
  const unsigned nb = (unsigned)(n / kLocal);
  bitonic_local_kernel<<<nb, 1024, 0, stream>>>(keys, 2, kLocal);
  for (int64_t k = 2 * kLocal; k <= n; k <<= 1) {
    for (int64_t j = k >> 1; j >= kLocal; j >>= 1)
      bitonic_global_kernel<<<(unsigned)((n / 2 + 255) / 256), 256, 0, stream>>>(keys, n, k, j);
    bitonic_local_kernel<<<nb, 1024, 0, stream>>>(keys, k, k);
  }
  return cudaGetLastError();
}

}  // namespace oscar
