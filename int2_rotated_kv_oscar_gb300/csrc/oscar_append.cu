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
// Rotation x' = x R: the bulk path multiplies by the composite R = U H P
// (formed on the host in fp64) on the tensor cores, R as three bf16 terms;
// the one-token paths by R in fp32 on the CUDA cores, or, without U, apply H
// as an in-register butterfly and P as an index map.  Quantiser per group
// of 64 rotated channels: a = min(max|x'|, tau), s = fp16(a / 1.5),
// code = [x' >= -s] + [x' >= 0] + [x' >= s].

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>

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
// A request's new tokens; bad spans set an error bit (from the reporting thread).
__device__ __forceinline__ bool request_span(const AppendLaunch& a, int b, int& p0, int& n, int& tok0,
                                             bool report = threadIdx.x == 0) {
  if (a.cu_seqlens == nullptr) {
    tok0 = b;
    n = 1;
  } else {
    tok0 = a.cu_seqlens[b];
    n = a.cu_seqlens[b + 1] - tok0;
    if (n < 0 || tok0 < 0 || tok0 + n > a.n_tokens || n > a.max_tokens_per_req) {
      if (report) set_error(a.err, kErrTokens);
      return false;
    }
  }
  p0 = a.pos[b];
  if (p0 < 0) {
    if (report) set_error(a.err, kErrLength);
    return false;
  }
  // a fresh ring holds only the new tokens: the recent window must lie inside them
  if ((a.flags & 1u) && p0 > kSink && n < kRecent) {
    if (report) set_error(a.err, kErrLength);
    return false;
  }
  return n > 0;
}

// Phase 1: ring tokens that fall out of the recent window go to the history.
// grid (256, Hkv, B), 2 kQuantThreads threads: one token-head per block, K
// by the first kQuantThreads threads, V by the others.
__global__ void __launch_bounds__(2 * kQuantThreads, 1) append_evict_kernel(AppendLaunch a) {
  __shared__ QuantSmem sm[2];
  griddep_launch_dependents();  // the BF16-row kernel may start; it waits for this one before its writes
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
  size_t r;
  if (!recent_row(c, b, h, e, r, a.err, threadIdx.x == 0)) return;
  uint8_t* blk = history_block(c, b, h, e, a.err);
  if (blk == nullptr) return;
  const float xv = bf16_bits_to_float((is_v ? c.v_ring : c.k_ring)[r + t]);
  quantize_token(xv, is_v ? a.rot.R_V : a.rot.R_K, is_v ? a.rot.tau_v : a.rot.tau_k, blk, e & 63, is_v, sm[half], u,
                 1 + half, nullptr, a.rot.flags);
}

// Phase 2a: new tokens that stay BF16 (sink rows, ring rows).
// grid (320, B), 128 threads; all KV heads of one position per block.
// The BF16 rows of new tokens: sink positions into the sink page, the last
// 256 positions into the ring (or the recent pages).
__device__ __forceinline__ void bf16_rows(const AppendLaunch& a) {
  // block x: one position of request blockIdx.y; thread t: 16 bytes (channels
  // 8 (t % 16) ..) of KV head t / 16, t / 16 + 8, ...
  const int x = blockIdx.x, b = blockIdx.y, t = threadIdx.x, c8 = 8 * (t & 15);
  int p0, n, tok0;
  if (!request_span(a, b, p0, n, tok0)) return;
  const int L = p0 + n;
  const CacheRefs& c = a.c;
  const int Hkv = c.num_kv_heads;
  auto copy = [&](int h, int p, uint16_t* kd, uint16_t* vd, size_t d) {
    const size_t s = ((size_t)(tok0 + p - p0) * Hkv + h) * kD + c8;
    *reinterpret_cast<uint4*>(kd + d + c8) = __ldg(reinterpret_cast<const uint4*>(a.k + s));
    *reinterpret_cast<uint4*>(vd + d + c8) = __ldg(reinterpret_cast<const uint4*>(a.v + s));
  };
  if (x < kSink) {
    const int p = p0 + x;
    if (p >= min(L, kSink)) return;
    const int sp = c.sink_page[b];
    if (sp < 0 || sp >= c.num_sink) {
      if (t == 0) set_error(a.err, kErrSink);
      return;
    }
    for (int h = t >> 4; h < Hkv; h += 8) copy(h, p, c.k_sink, c.v_sink, (((size_t)sp * Hkv + h) * kSink + p) * kD);
    return;
  }
  const int p = max(max(p0, L - kRecent), kSink) + (x - kSink);
  if (p >= L) return;
  for (int h = t >> 4; h < Hkv; h += 8) {
    size_t d;
    if (!recent_row(c, b, h, p, d, a.err, (t & 15) == 0)) continue;
    copy(h, p, c.k_ring, c.v_ring, d);
  }
}

__global__ void __launch_bounds__(128) append_bf16_kernel(AppendLaunch a) {
  // Evicting: the tile kernel after this one may start (it touches no BF16
  // row), and the ring rows written here are the ones the eviction kernel
  // before this one reads, so wait for it first.  Fresh ring: this kernel
  // runs beside the tile kernel before it and waits for it at the end, so
  // that its end marks the call's.
  const bool fresh = (a.flags & 1u) != 0;
  griddep_launch_dependents();
  if (!fresh) griddep_wait();
  bf16_rows(a);
  if (fresh) griddep_wait();
}

// Phase 2b: new tokens that go straight into the INT2 history.
//
// x R on the 5th-generation tensor cores: one tile is 128 new tokens (two
// pages) of one (request, KV head) and one matrix (K or V).  D[token][n] =
// sum_k x[token][k] R^T[n][k] runs as tcgen05 MMAs (M = 128 tokens, K = 16)
// from shared memory into tensor memory.  x is bf16 (exact) and R^T is held
// as three bf16 terms (R = t0 + t1 + t2 to ~2^-24 relative), so every product
// is exact; the t0 products accumulate in one TMEM region, the much smaller
// t1, t2 products in a second, and the epilogue adds the two in fp32 (the
// codes then match the fp64 definition bit for bit outside the near-edge
// band).  Per K step one N = 256 MMA takes t0 and t1 at once (B = the t0 rows
// followed by the t1 rows, D = both regions) and one N = 128 MMA adds t2
// into the second region: 16 MMAs per tile, so that one thread issues them
// faster than the tensor cores run them.  Two TMEM buffers of 256 columns:
// the MMAs of the next tile overlap the epilogue of this one.
//
// Persistent blocks, one per SM, each for one matrix (a little more than half,
// spread evenly over the grid, for V; the others for K):
//   warps 0-15  epilogue: warp (h, g, q) = (w / 8, w / 4 % 2, w % 4) takes
//               token row 32 q + lane (its TMEM lane) of group g, channels
//               16 k + 8 h + b (k < 4, b < 8); R^T's rows are permuted in
//               shared memory so those channels come out in 32 adjacent
//               TMEM columns; the two halves of a row swap their maxima
//               through shared memory, then each writes whole K words or V
//               bytes of its row
//   warp 16     one thread loads x tiles by TMA (two 64-channel boxes of 128
//               token rows each, 128-byte swizzle, rows outside the tensor
//               read as zero) into a ring of kTcStages buffers
//   warp 17     TMEM allocation; one thread issues the MMAs
constexpr int kTcRegions = 1;
constexpr int kTcThreads = 18 * 32;
constexpr int kTcStages = 3;
constexpr uint32_t kTcCols = 512;          // TMEM columns: buffer bb = [t0: 128][t1 + t2: 128] from column 256 bb
constexpr uint32_t kTcB = 0;               // R^T terms: [2 k-blocks][3 terms][128 rows n][128 B]
constexpr uint32_t kTcA = 3 * 32768;       // x tiles: kTcStages x [2 k-blocks][128 rows][128 B]
constexpr uint32_t kTcBars = kTcA + kTcStages * 32768;
constexpr uint32_t kTcPmax = kTcBars + 512;  // [tile parity][h][g][128 rows] float: half-row maxima
constexpr double kTcVShare = 0.52;          // share of the blocks that take V tiles
constexpr int kTcDescs = 8;                  // tile descriptors the TMA thread publishes ahead
constexpr uint32_t kTcDesc = kTcPmax + 4096;
constexpr size_t kTcSmem = kTcDesc + kTcDescs * 64 + 1024;  // + 1024-byte alignment slack
// barriers (full, empty: kTcStages each; tfull, tempty: 4 each; done; 8 swaps; 2 kTcDescs; full1:
// kTcStages), TMEM address, flags
static_assert((3 * kTcStages + 8 + 1 + 8 + 2 * kTcDescs) * 8 + 4 + 4 * kTcStages <= 512, "barrier area");

// What the epilogue needs of a tile: positions [lo, hi) of page pair (lp0, lp0 + 1) get written
// to blk[0], blk[1] (null: nothing to write there); b < 0 marks the end of the block's tiles.
struct TcDesc {
  uint8_t* blk[2];
  int b, lp0, lo, hi;
};
static_assert(sizeof(TcDesc) <= 64, "descriptor slot");
static_assert(kTcRegions == 1, "the epilogue reads one t0 region and the chain");

struct TcTile {
  int b, h, lp0, lo, hi, tok0, p0;
};

// The tile-th (request, KV head, page pair) of a matrix; false: nothing to write.
__device__ __forceinline__ bool tc_tile(const AppendLaunch& a, unsigned tile, unsigned tiles2, TcTile& t) {
  const unsigned Hkv = (unsigned)a.c.num_kv_heads, r = tile / tiles2;
  t.h = (int)(r % Hkv);
  t.b = (int)(r / Hkv);
  int n;
  if (!request_span(a, t.b, t.p0, n, t.tok0, true)) return false;
  t.lo = max(t.p0, kSink);
  t.hi = t.p0 + n - kRecent;
  if (t.hi <= t.lo) return false;
  t.lp0 = t.lo / kPage + 2 * (int)(tile % tiles2);
  return t.lp0 * kPage < t.hi;
}

// Block of logical page lp (any thread may report a bad entry).
__device__ __forceinline__ uint8_t* tc_block(const CacheRefs& c, int b, int h, int lp, unsigned* err) {
  if (lp >= c.max_pages) {
    set_error(err, kErrLength);
    return nullptr;
  }
  const int phys = c.page_table[(size_t)b * c.max_pages + lp];
  if (phys < 0 || phys >= c.num_pages) {
    set_error(err, kErrPage);
    return nullptr;
  }
  return c.pages + ((size_t)phys * c.num_kv_heads + h) * kBlockBytes;
}

// Byte offset of element (row, 16-byte chunk ch of K) in a [2][rows][128 B] swizzled operand.
__device__ __forceinline__ uint32_t sw128_offset(int row, int ch) {
  return (ch >> 3) * 16384 + (row >> 3) * 1024 + (row & 7) * 128 + (((ch & 7) ^ (row & 7)) << 4);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    append_tile_kernel(const __grid_constant__ AppendLaunch a, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, unsigned tiles2, unsigned nv) {
  // the kernel after this one may start beside it (it waits before it reads what this one writes)
  griddep_launch_dependents();
  extern __shared__ uint8_t tc_raw[];
  const uint32_t raw_s = smem_u32(tc_raw);
  uint8_t* sm = tc_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  const uint32_t sbase = smem_u32(sm);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kTcBars);  // [kTcStages] k-block 0 of buffer s landed
  uint64_t* empty = full + kTcStages;                           // [kTcStages] buffer s read by its MMAs
  uint64_t* tfull = empty + kTcStages;                          // [4, 2 used] TMEM buffer bb holds its sums
  uint64_t* tempty = tfull + 4;                                 // [4, 2 used] TMEM buffer bb read
  uint64_t* done = tempty + 4;                                  // every MMA of the block finished
  uint64_t* xb = done + 1;                                      // [8] the two halves of (g, q) swapped maxima
  uint64_t* dfull = xb + 8;                                     // [kTcDescs] descriptor d written
  uint64_t* dempty = dfull + kTcDescs;                          // [kTcDescs] descriptor d read by the epilogue
  uint64_t* full1 = dempty + kTcDescs;                          // [kTcStages] k-block 1 of buffer s landed
  uint32_t* tmem_at = reinterpret_cast<uint32_t*>(full1 + kTcStages);
  TcDesc* desc = reinterpret_cast<TcDesc*>(sm + kTcDesc);
  volatile int* work = reinterpret_cast<volatile int*>(tmem_at + 1);  // [kTcStages] buffer s holds a tile (0: no more)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // nv of the blocks take V, spread evenly over the grid: block i is the v_before(i)-th V block
  // when v_before(i + 1) > v_before(i), v_before(i) = floor(i nv / blocks), else a K block
  const unsigned vb0 = blockIdx.x * nv / gridDim.x, vb1 = (blockIdx.x + 1) * nv / gridDim.x;
  const int m = vb1 > vb0 ? 1 : 0;
  const unsigned cta = m ? vb0 : blockIdx.x - vb0, n_cta = m ? nv : gridDim.x - nv;
  const int Hkv = a.c.num_kv_heads;
  const unsigned n_tiles = tiles2 * (unsigned)Hkv * (unsigned)a.c.batch;
  {  // this matrix's three R^T terms
    const uint4* src = reinterpret_cast<const uint4*>(a.rot.RT_split) + (size_t)m * 3 * 128 * 16;
    for (int c = threadIdx.x; c < 3 * 128 * 16; c += kTcThreads) {
      const int term = c >> 11, n = (c >> 4) & 127, jj = n & 63;
      const int col = (n & 64) | (jj & 8) << 2 | (jj >> 4) << 3 | (jj & 7);
      const int ch = c & 15;  // 16-byte chunk along K: k-block ch / 8
      *reinterpret_cast<uint4*>(sm + kTcB + (ch >> 3) * 49152 + term * 16384 + sw128_offset(col, ch & 7)) =
          __ldg(src + c);
    }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&full1[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 16);  // every epilogue warp, once per tile of the buffer
    }
    mbar_init(done, 1);
    for (int i = 0; i < 8; ++i) mbar_init(&xb[i], 2);
    for (int i = 0; i < kTcDescs; ++i) {
      mbar_init(&dfull[i], 1);
      mbar_init(&dempty[i], 16);  // every epilogue warp
    }
    fence_mbar_init();
  }
  if (warp == 17) tmem_alloc(tmem_at, kTcCols);
  fence_proxy_async_smem();  // R^T, for the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_at;
  // For a fresh prompt this kernel comes first in the call and may start before the stream's
  // previous work has finished: the set-up above reads only the rotation tables (written by a
  // synchronous upload), so wait here, before the inputs, tables and page blocks are touched.
  if (a.flags & 1u) griddep_wait();

  if (warp == 16) {
    // x tiles by TMA; after the last tile a buffer with work = 0 tells the MMA thread to stop.  The
    // warp looks up 32 candidate tiles at once (lane j: tile base + j n_cta, with its page blocks),
    // so that lane 0 issues each load without waiting on a table read.
    const CUtensorMap* tm = m ? &tmv : &tmk;
    if (lane == 0) prefetch_tensormap(tm);
    // x is read once: its lines go first when L2 needs room (the code writes stay)
    const uint64_t once = l2_policy_evict_first();
    int it = 0;  // lane 0: tiles whose loads were issued
    bool timed_out = false;
    for (unsigned base = cta; base < n_tiles && !timed_out; base += 32u * n_cta) {
      const unsigned tile = base + (unsigned)lane * n_cta;
      TcTile t = {};
      uint8_t* b0 = nullptr;
      uint8_t* b1 = nullptr;
      const bool valid = tile < n_tiles && tc_tile(a, tile, tiles2, t);
      int y0 = 0;
      if (valid) {
        b0 = tc_block(a.c, t.b, t.h, t.lp0, a.err);
        b1 = (t.lp0 + 1) * kPage < t.hi ? tc_block(a.c, t.b, t.h, t.lp0 + 1, a.err) : nullptr;
        y0 = t.tok0 + t.lp0 * kPage - t.p0;  // token index of the tile's first row (may be < 0)
      }
      unsigned vmask = __ballot_sync(0xffffffffu, valid);
      while (vmask != 0u) {
        const int j = __ffs(vmask) - 1;
        vmask &= vmask - 1u;
        const int th = __shfl_sync(0xffffffffu, t.h, j), ty0 = __shfl_sync(0xffffffffu, y0, j);
        const int tb = __shfl_sync(0xffffffffu, t.b, j), tlp0 = __shfl_sync(0xffffffffu, t.lp0, j);
        const int tlo = __shfl_sync(0xffffffffu, t.lo, j), thi = __shfl_sync(0xffffffffu, t.hi, j);
        const uint64_t pb0 = __shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(b0), j);
        const uint64_t pb1 = __shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(b1), j);
        if (lane == 0) {
          const int s = it % kTcStages, di = it % kTcDescs;
          if (!mbar_wait_bounded(&empty[s], ((it / kTcStages) & 1) ^ 1, kWaitLimit)) {
            timed_out = true;
          } else {
            work[s] = 1;
            // the two k-blocks land on their own barriers: the first half's MMAs start without the second
            mbar_arrive_expect_tx(&full[s], 16384);
            tma_load_3d(sm + kTcA + s * 32768, tm, 0, th, ty0, &full[s], once);
            mbar_arrive_expect_tx(&full1[s], 16384);
            tma_load_3d(sm + kTcA + s * 32768 + 16384, tm, 64, th, ty0, &full1[s], once);
            ++it;
            if (!mbar_wait_bounded(&dempty[di], (((it - 1) / kTcDescs) & 1) ^ 1, kWaitLimit)) {
              timed_out = true;
            } else {
              TcDesc& dsc = desc[di];
              dsc.b = tb;
              dsc.lp0 = tlp0;
              dsc.lo = tlo;
              dsc.hi = thi;
              dsc.blk[0] = reinterpret_cast<uint8_t*>(pb0);
              dsc.blk[1] = reinterpret_cast<uint8_t*>(pb1);
              mbar_arrive(&dfull[di]);
            }
          }
        }
        timed_out = __shfl_sync(0xffffffffu, timed_out, 0);
        if (timed_out) break;
      }
    }
    if (lane == 0) {
      if (timed_out) {
        set_error(a.err, kErrTimeout);
        // copies may still be in flight: wait for them, bounded (on the normal path the MMA thread
        // has seen every one land)
        for (int k = max(0, it - kTcStages); k < it; ++k) {
          mbar_wait_bounded(&full[k % kTcStages], (k / kTcStages) & 1, kWaitLimit);
          mbar_wait_bounded(&full1[k % kTcStages], (k / kTcStages) & 1, kWaitLimit);
        }
      } else {
        const int s = it % kTcStages, di = it % kTcDescs;
        if (!mbar_wait_bounded(&empty[s], ((it / kTcStages) & 1) ^ 1, kWaitLimit) ||
            !mbar_wait_bounded(&dempty[di], ((it / kTcDescs) & 1) ^ 1, kWaitLimit)) {
          set_error(a.err, kErrTimeout);
        } else {
          desc[di].b = -1;
          mbar_arrive(&dfull[di]);
          work[s] = 0;
          mbar_arrive(&full[s]);
        }
      }
    }
    __syncwarp();
  } else if (warp == 17) {
    if (lane == 0) {
      const uint64_t dhi = umma_desc_sw128(0) & 0xFFFFFFFF00000000ull;
      const uint32_t a_lo = (uint32_t)umma_desc_sw128(sbase + kTcA), b_lo = (uint32_t)umma_desc_sw128(sbase + kTcB);
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int s = it % kTcStages, bb = it & 1;
        if (!mbar_wait_bounded(&full[s], (it / kTcStages) & 1, kWaitLimit)) {
          ok = false;
          break;
        }
        if (work[s] == 0) break;
        const uint32_t al = a_lo + (uint32_t)s * (32768 >> 4);
        if (!mbar_wait_bounded(&tempty[bb], ((it >> 1) & 1) ^ 1, kWaitLimit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        constexpr uint32_t idesc256 = umma_idesc_bf16_f32(128, 256), idesc128 = umma_idesc_bf16_f32(128, 128);
        const uint32_t d = tbase + 256 * bb;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (i == 4 && !mbar_wait_bounded(&full1[s], (it / kTcStages) & 1, kWaitLimit)) {
            ok = false;  // the MMAs issued so far are covered by the final commit below
            break;
          }
          const uint32_t ka = (uint32_t)((i >> 2) * 16384 + (i & 3) * 32) >> 4;  // x: k-blocks 16 KB apart
          const uint32_t kb = (uint32_t)((i >> 2) * 49152 + (i & 3) * 32) >> 4;  // R^T: 48 KB apart
          const uint64_t ad = dhi | (al + ka);
          umma_f16(d, ad, dhi | (b_lo + kb), idesc256, i > 0);                          // t0 | t1
          umma_f16(d + 128, ad, dhi | (b_lo + kb + (32768 >> 4)), idesc128, true);      // + t2
        }
        if (!ok) break;
        umma_commit(&tfull[bb]);
        umma_commit(&empty[s]);
      }
      if (!ok) set_error(a.err, kErrTimeout);
      umma_commit(done);  // arrives once every MMA above has finished
      if (!mbar_wait_bounded(done, 0, kWaitLimit)) set_error(a.err, kErrTimeout);
    }
    __syncwarp();
  } else {
    // epilogue: warp (h, g, q) = (warp / 8, warp / 4 % 2, warp % 4): token row 32 q + lane, group g,
    // channels 16 k + 8 h + b (k < 4, b < 8), which the permuted R^T puts in TMEM columns 64 g + 32 h + 8 k + b
    // of the tile's buffer (t0 part; the t1 + t2 part 128 columns on)
    const int g = (warp >> 2) & 1, h = warp >> 3, q = warp & 3, row = 32 * q + lane;
    const float tau = m ? a.rot.tau_v : a.rot.tau_k;
    float* pmax = reinterpret_cast<float*>(sm + kTcPmax);
    for (int it = 0;;) {
      const int di = it % kTcDescs;
      // waits are warp-uniform: the TMEM loads below are warp-wide (.sync.aligned)
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&dfull[di], (it / kTcDescs) & 1, kWaitLimit))) {
        set_error(a.err, kErrTimeout);
        break;
      }
      const TcDesc& dsc = desc[di];
      const int b = dsc.b, p = dsc.lp0 * kPage + row;
      uint8_t* blk = (b >= 0 && p >= dsc.lo && p < dsc.hi) ? dsc.blk[row >> 6] : nullptr;
      // one arrival per warp (the lanes' reads are ordered before it by the warp barrier)
      __syncwarp();
      if (lane == 0) mbar_arrive(&dempty[di]);
      if (b < 0) break;
      const int bb = it & 1;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&tfull[bb], (it >> 1) & 1, kWaitLimit))) {
        set_error(a.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      float x[32];
      {
        float v[32], w[32];
        const uint32_t ta = tbase + ((uint32_t)(32 * q) << 16) + 256 * bb + 64 * g + 32 * h;
        tmem_ld32x2(ta, ta + 128, v, w);
        // the buffer is free once the loads have landed: the next tile's MMAs may start
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[bb]);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 s2 = fadd2(make_float2(v[e], v[e + 1]), make_float2(w[e], w[e + 1]));
          x[e] = s2.x;
          x[e + 1] = s2.y;
        }
      }
      float mq[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains
#pragma unroll
      for (int e = 0; e < 32; ++e) mq[e & 3] = fmaxf(mq[e & 3], fabsf(x[e]));
      float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      // the group maximum over both halves of the row
      float* pm = pmax + (((bb * 2 + h) * 2 + g) * 128);
      pm[row] = mx;
      __syncwarp();
      if (lane == 0) mbar_arrive(&xb[4 * g + q]);
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&xb[4 * g + q], (it & 1), kWaitLimit))) {
        set_error(a.err, kErrTimeout);
        break;
      }
      mx = fmaxf(mx, pmax[(((bb * 2 + (h ^ 1)) * 2 + g) * 128) + row]);
      ++it;
      if (blk == nullptr) continue;
      const int rp = p & 63;
      const __half hs = __float2half_rn(fminf(mx, tau) / 1.5f);
      const float sc = __half2float(hs);
      // The code (x >= -s) + (x >= 0) + (x >= s) is floor(x / s + 2) while
      // every |x| / s of the group stays below 2 (no clipped value, a normal
      // scale).  Then one fma rounding down into the units of 1.5 2^23 gives
      // it in the low bits of the result, and one multiply-add puts it at its
      // bit: sum (bits - 1.5 2^23) 2^shift over a word = sum bits 2^shift
      // minus a constant, mod 2^32.  x times the approximate reciprocal moves
      // an edge by about 2^-22 relative.
      float inv;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(sc));
      const bool fast = sc > 0.f && mx * inv < 1.99f;
      constexpr float kMagic = 12582914.0f;         // 1.5 2^23 + 2
      constexpr uint32_t kMagicBits = 0x4B400000u;  // bits of 1.5 2^23
      if (m == 0) {
        // K words tq = 2 h + b / 4: channel 16 k + 4 tq + b % 4 at bit 8 (b % 4) + 2 k
        uint32_t kw[2] = {0u, 0u};
        if (fast) {
          uint32_t part[2][4] = {{0u, 0u, 0u, 0u}, {0u, 0u, 0u, 0u}};  // short chains: by word and k
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 f = ffma2_rd(make_float2(x[e], x[e + 1]), make_float2(inv, inv), make_float2(kMagic, kMagic));
            const int kk = e >> 3, b = e & 7;
            part[b >> 2][kk] += __float_as_uint(f.x) * (1u << (8 * (b & 3) + 2 * kk));
            part[(b + 1) >> 2][kk] += __float_as_uint(f.y) * (1u << (8 * ((b + 1) & 3) + 2 * kk));
          }
          kw[0] = ((part[0][0] + part[0][1]) + (part[0][2] + part[0][3])) - kMagicBits * 0x55555555u;
          kw[1] = ((part[1][0] + part[1][1]) + (part[1][2] + part[1][3])) - kMagicBits * 0x55555555u;
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int kk = e >> 3, b = e & 7;
            const uint32_t bit = 1u << (8 * (b & 3) + 2 * kk);
            kw[b >> 2] += (x[e] >= -sc ? bit : 0u) + (x[e] >= 0.f ? bit : 0u) + (x[e] >= sc ? bit : 0u);
          }
        }
        *reinterpret_cast<uint32_t*>(blk + kKCodes + k_word_offset(rp, 2 * h, g)) = kw[0];
        *reinterpret_cast<uint32_t*>(blk + kKCodes + k_word_offset(rp, 2 * h + 1, g)) = kw[1];
      } else {
        // V: byte g of the half of channel residue 8 h + b holds channels 16 k + 8 h + b at bit 2 k
        uint32_t vb[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) vb[b] = 0u;
        if (fast) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 f = ffma2_rd(make_float2(x[e], x[e + 1]), make_float2(inv, inv), make_float2(kMagic, kMagic));
            vb[e & 7] += __float_as_uint(f.x) * (1u << (2 * (e >> 3)));
            vb[(e + 1) & 7] += __float_as_uint(f.y) * (1u << (2 * (e >> 3)));
          }
#pragma unroll
          for (int b = 0; b < 8; ++b) vb[b] -= kMagicBits * 0x55u;
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const uint32_t bit = 1u << (2 * (e >> 3));
            vb[e & 7] += (x[e] >= -sc ? bit : 0u) + (x[e] >= 0.f ? bit : 0u) + (x[e] >= sc ? bit : 0u);
          }
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) blk[kVCodes + v_half_offset(rp, 8 * h + b) + g] = (uint8_t)vb[b];
      }
      if (h == 0) *reinterpret_cast<__half*>(blk + (m ? kVScales : kKScales) + 4 * rp + 2 * g) = hs;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 17) {
    tc_fence_after();
    tmem_dealloc(tbase, kTcCols);
  }
  // this kernel may have started beside the BF16-row and eviction kernels: its
  // end also marks theirs for what comes next in the stream
  griddep_wait();
}

}  // namespace

namespace {
// The failure path of every asynchronous wait: a barrier that nothing
// completes, a bounded wait that gives up, the timeout bit, a normal return.
// Warp 0 runs the polled wait (`polls` polls), warp 1 the timed wait (polls x 4 us on the
// global timer), each on its own barrier that nothing completes; the error bit is set only
// when both give up.
__global__ void __launch_bounds__(64) selftest_wait_kernel(unsigned* err, unsigned polls) {
  __shared__ uint64_t bar[2];
  __shared__ int gave_up[2];
  const int w = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = w == 0 ? mbar_wait_bounded(&bar[0], 0, polls)
                         : mbar_wait_timed(&bar[1], 0, 4000ull * polls);
  const bool all_ok = __all_sync(0xffffffffu, ok);
  if ((threadIdx.x & 31) == 0) gave_up[w] = all_ok ? 0 : 1;
  __syncthreads();
  if (threadIdx.x == 0 && gave_up[0] && gave_up[1]) set_error(err, kErrTimeout);
}
}  // namespace

cudaError_t launch_selftest_wait(unsigned* err, unsigned polls, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 64, 0, stream>>>(err, polls);
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendLaunch& a, cudaStream_t stream) {
  const int B = a.c.batch, Hkv = a.c.num_kv_heads;
  if (a.cu_seqlens == nullptr) {
    append_one_kernel<<<dim3(Hkv, B), 2 * kQuantThreads, 0, stream>>>(a);
    return cudaGetLastError();
  }
  // The kernels after the first may start early and run beside it.  The tile
  // kernel writes only the INT2 rows of new tokens, which the eviction and
  // BF16-row kernels do not touch; the eviction reads ring rows that the
  // BF16-row kernel overwrites.
  //   evicting:     eviction -> BF16 rows (wait first) -> tiles (wait at the end)
  //   fresh ring:   tiles (set-up, then wait) -> BF16 rows (wait at the end)
  // so the last kernel of the call always ends after the others.
  AppendLaunch la = a;
  void* args1[] = {&la};
  const bool fresh = (a.flags & 1u) != 0;
  if (a.n_tokens == 0) {
    if (!fresh) append_evict_kernel<<<dim3(kRecent, Hkv, B), 2 * kQuantThreads, 0, stream>>>(a);
    append_bf16_kernel<<<dim3(kSink + kRecent, B), 128, 0, stream>>>(a);
    return cudaGetLastError();
  }
  const int pages = (a.max_tokens_per_req + kPage - 1) / kPage + 1;  // INT2 pages a request can touch
  const int tiles2 = (pages + 1) / 2;                                    // page pairs
  if ((long long)tiles2 * Hkv * B >= (1ll << 31)) return cudaErrorInvalidValue;
  int sms = 0;
  {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    static std::atomic<uint64_t> attr_done;
    if (e == cudaSuccess) e = smem_attr_once(reinterpret_cast<const void*>(append_tile_kernel), kTcSmem, attr_done);
    if (e != cudaSuccess) return e;
  }
  // tensor maps of k and v: [n_tokens][Hkv][128] bf16, boxes of 64 channels x 1 head x 128 tokens
  // (the driver entry point is looked up once; a function-local static is thread-safe to initialise)
  static const PFN_cuTensorMapEncodeTiled_v12000 encode = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess) return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap tm[2];
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)Hkv, (cuuint64_t)a.n_tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)Hkv * kD * 2};
  const cuuint32_t box[3] = {64, 1, 128}, estride[3] = {1, 1, 1};
  for (int i = 0; i < 2; ++i) {
    const CUresult r = encode(&tm[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(i ? a.v : a.k), dims,
                              strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  // one block per SM, nv of them for V and the rest for K: a V tile takes a little longer (its
  // epilogue stores bytes, K's whole words), so V gets a little more than half; neither matrix
  // gets more blocks than it has tiles
  const long long per_matrix = (long long)tiles2 * Hkv * B;
  const int blocks = (int)std::min<long long>(2 * per_matrix, std::max(2, sms));
  long long nv_ll = std::llround(blocks * kTcVShare);
  nv_ll = std::min<long long>(std::max<long long>(nv_ll, blocks - per_matrix), per_matrix);
  nv_ll = std::min<long long>(std::max<long long>(nv_ll, 1), blocks - 1);
  unsigned t2 = (unsigned)tiles2, nv = (unsigned)nv_ll;
  void* args[] = {&la, &tm[0], &tm[1], &t2, &nv};
  const void* tile_fn = reinterpret_cast<const void*>(append_tile_kernel);
  const void* bf16_fn = reinterpret_cast<const void*>(append_bf16_kernel);
  if (fresh) {
    const cudaError_t e = launch_pdl(tile_fn, dim3(blocks), dim3(kTcThreads), kTcSmem, stream, args);
    if (e != cudaSuccess) return e;
    return launch_pdl(bf16_fn, dim3(kSink + kRecent, B), dim3(128), 0, stream, args1);
  }
  append_evict_kernel<<<dim3(kRecent, Hkv, B), 2 * kQuantThreads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = launch_pdl(bf16_fn, dim3(kSink + kRecent, B), dim3(128), 0, stream, args1);
  if (e != cudaSuccess) return e;
  return launch_pdl(tile_fn, dim3(blocks), dim3(kTcThreads), kTcSmem, stream, args);
}

}  // namespace oscar
