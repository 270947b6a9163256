// fm_bounds.cu -- the bounds pass of fixed-m attention.
//
// Computes, per (batch, head): the key mean kbar (when centering), the maximum key norm
// (of k_j - kbar, or of k_j), per 128-row Q-block the maximum query norm, per row the
// centering term alpha*q_i.kbar, the global max of v^2, and from those the shift
// m = ceil(U) - C(N) and the eligibility flag v_ok && U <= gate, with
// U = alpha*sqrt(max|q|^2)*sqrt(max|k|^2).
// Sources: "feat(attention): fixed-m splash attention kernel with dynamic bounds and
// safety fallbacks" (PR #477), Summary; the fused norm reduction of "Kernel reference:
// ring_attention_const_max_fwd", section "Transpose prologue with fused norms"; the key
// mean over real tokens of PR #478, Summary.
//
// Launches (all deterministic: fixed-order sums, maxima without atomics):
//   1. ksum    (centering only) partial key sums, P row ranges per head  -> workspace
//   2. kmean   (centering only) ordered sum of the P partials / N          -> kbar
//   3. main    one grid over Q-blocks, K row-blocks and V row-blocks: row norms via warp
//              shuffles; per-block maxima -> qmax_sq (Q) and the workspace (K, V);
//              qkbar per row; with key sinks, each K block's n_sink + 1 loudest keys
//   3b. sinks  (key sinks only) per head: the n_sink + 1 loudest keys over the blocks'
//              candidates; the sinks and the max over the other keys ("Kernel reference:
//              ring_attention_const_max_fwd", section "Adapting this kernel")
//   4. finish  per head: key max, global V max, U, m, flag
//   5. shift   per row: b_i = m_i + alpha*q_i.kbar (m_i per row or per Q-block)
// Bytes: Q + K + V once each, plus K once more for the mean when centering.
#include <cuda_bf16.h>
#include <limits.h>
#include <math.h>

#include "fm_internal.h"

namespace fm {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kQRows = FM_BLOCK_Q;  // rows per Q-block
constexpr int kKVRows = 256;        // rows per K / V block of the main pass
constexpr int kMaxPartials = 64;    // row ranges per head for the key sum

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Row ranges per head for the key sum: one per 128 rows, so that short sequences still give
// enough CTAs to keep HBM busy, and at most kMaxPartials.
inline int64_t num_partials(int64_t N) {
  int64_t p = ceil_div(N, 128);
  return p < 1 ? 1 : (p > kMaxPartials ? kMaxPartials : p);
}

// A key-sink candidate: squared norm and global key index (v = -1: no candidate).
struct SinkCand {
  float v;
  int32_t idx;
};
constexpr int kCandPerBlock = FM_MAX_SINKS + 1;  // each K block keeps its top n_sink + 1

struct WsLayout {
  int64_t P, nkb, nvb;
  size_t off_part, off_kb, off_vb, off_cand, total;
};

WsLayout ws_layout(int64_t B, int64_t H, int64_t N, int64_t D) {
  WsLayout w;
  w.P = num_partials(N);
  w.nkb = ceil_div(N, kKVRows);
  w.nvb = w.nkb;
  w.off_part = 0;
  w.off_kb = w.off_part + sizeof(float) * (size_t)(B * H * w.P * D);
  w.off_vb = w.off_kb + sizeof(float) * (size_t)(B * H * w.nkb);
  w.off_cand = w.off_vb + sizeof(float) * (size_t)(B * H * w.nvb);
  w.off_cand = (w.off_cand + 15) & ~(size_t)15;
  w.total = w.off_cand + sizeof(SinkCand) * (size_t)(B * H * w.nkb * kCandPerBlock);
  w.total = (w.total + 255) & ~(size_t)255;
  return w;
}

// Load the EPL elements of row `row` that lane `lane` owns (d = lane*EPL + e) as fp32.
template <typename T, int EPL, bool CONTIG>
__device__ __forceinline__ void load_row(const T *base, int64_t sD, int lane, float (&x)[EPL]) {
  if constexpr (CONTIG && sizeof(T) == 2 && EPL == 4) {
    uint2 u = *reinterpret_cast<const uint2 *>(base + lane * 4);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&u.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&u.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    x[0] = fa.x; x[1] = fa.y; x[2] = fb.x; x[3] = fb.y;
  } else if constexpr (CONTIG && sizeof(T) == 2 && EPL == 2) {
    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(base + lane * 2);
    float2 fa = __bfloat1622float2(a);
    x[0] = fa.x; x[1] = fa.y;
  } else if constexpr (CONTIG && sizeof(T) == 4 && EPL == 4) {
    float4 f = *reinterpret_cast<const float4 *>(base + lane * 4);
    x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
  } else if constexpr (CONTIG && sizeof(T) == 4 && EPL == 2) {
    float2 f = *reinterpret_cast<const float2 *>(base + lane * 2);
    x[0] = f.x; x[1] = f.y;
  } else {
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      T t = base[(int64_t)(lane * EPL + e) * sD];
      if constexpr (sizeof(T) == 2) x[e] = __bfloat162float(t); else x[e] = (float)t;
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Key-sink order: louder first, the lower index first among equal norms.
__device__ __forceinline__ bool sink_before(float v, int32_t i, float bv, int32_t bi) {
  return v > bv || (v == bv && i < bi);
}
// (v, i) comes after the previous pick (pv, pi) in that order.
__device__ __forceinline__ bool sink_after(float v, int32_t i, float pv, int32_t pi) {
  return v < pv || (v == pv && i > pi);
}
__device__ __forceinline__ void warp_best_sink(float &bv, int32_t &bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (sink_before(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
}

// 1. Partial key sums: CTA (p, h, b) sums rows [p*len, (p+1)*len) of head (b, h).
template <typename T, int EPL, bool CONTIG>
__global__ void __launch_bounds__(kThreads) ksum_kernel(View k, int64_t P, float *part) {
  pdl_wait();  // inputs written by the kernels before this one
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t b = blockIdx.z, h = blockIdx.y, p = blockIdx.x;
  const int64_t len = ceil_div(k.S, P);
  const int64_t r0 = p * len, r1 = min(k.S, r0 + len);
  const T *base = reinterpret_cast<const T *>(k.ptr) + b * k.sB + h * k.sH;
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int64_t r = r0 + warp; r < r1; r += kWarps) {
    float x[EPL];
    load_row<T, EPL, CONTIG>(base + r * k.sS, k.sD, lane, x);
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] += x[e];
  }
  __shared__ float red[kWarps][128];
#pragma unroll
  for (int e = 0; e < EPL; ++e) red[warp][lane * EPL + e] = acc[e];
  __syncthreads();
  const int D = 32 * EPL;
  if (threadIdx.x < D) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += red[w][threadIdx.x];
    part[((b * k.H + h) * P + p) * D + threadIdx.x] = s;
  }
}

// ---- rows that start on 16-byte boundaries: 16-byte loads, several rows in flight per lane --
// A row of D elements is spread over LPR lanes with VEC consecutive elements each, so one warp
// load covers RPW = 32 / LPR rows; each lane keeps kUnroll such loads in flight before it
// reduces, which is what keeps HBM busy (one 256-byte row per warp at a time is not enough).
constexpr int kUnroll = 4;
template <typename T, int D>
struct Vec16 {
  static constexpr int VEC = 16 / (int)sizeof(T);
  static constexpr int LPR = D / VEC;
  static constexpr int RPW = 32 / LPR;
};
template <typename T, int VEC>
__device__ __forceinline__ void load16(const T *p, float (&x)[VEC]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
  if constexpr (sizeof(T) == 2) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  } else {
    x[0] = __uint_as_float(u.x);
    x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z);
    x[3] = __uint_as_float(u.w);
  }
}
// Sum over the LPR lanes of one row (lanes lane ^ o for o < LPR).
template <int LPR>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 1'. Partial key sums with 16-byte loads (the same partition of rows as ksum_kernel, a fixed
// order of additions within it).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) ksum_vec_kernel(View k, int64_t P, float *part) {
  pdl_wait();  // inputs written by the kernels before this one
  pdl_trigger();
  using V = Vec16<T, D>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / V::LPR, li = lane % V::LPR;
  const int64_t b = blockIdx.z, h = blockIdx.y, p = blockIdx.x;
  const int64_t len = ceil_div(k.S, P);
  const int64_t r0 = p * len, r1 = min(k.S, r0 + len);
  const T *base = reinterpret_cast<const T *>(k.ptr) + b * k.sB + h * k.sH + li * V::VEC;
  const int64_t step = (int64_t)kWarps * V::RPW;
  float acc[V::VEC];
#pragma unroll
  for (int e = 0; e < V::VEC; ++e) acc[e] = 0.f;
  int64_t r = r0 + warp * V::RPW + sub;
  for (; r + (kUnroll - 1) * step < r1; r += kUnroll * step) {
    float x[kUnroll][V::VEC];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) load16<T, V::VEC>(base + (r + u * step) * k.sS, x[u]);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int e = 0; e < V::VEC; ++e) acc[e] += x[u][e];
  }
  for (; r < r1; r += step) {
    float x[V::VEC];
    load16<T, V::VEC>(base + r * k.sS, x);
#pragma unroll
    for (int e = 0; e < V::VEC; ++e) acc[e] += x[e];
  }
  // the warp's sub-rows, then its warps, in a fixed order
#pragma unroll
  for (int o = V::LPR; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < V::VEC; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
  __shared__ float red[kWarps][128];
  if (sub == 0) {
#pragma unroll
    for (int e = 0; e < V::VEC; ++e) red[warp][li * V::VEC + e] = acc[e];
  }
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += red[w][threadIdx.x];
    part[((b * k.H + h) * P + p) * D + threadIdx.x] = s;
  }
}

// 2. Key mean: ordered sum of the P partials of head (b, h), divided by N.
__global__ void kmean_kernel(const float *part, int64_t H, int64_t P, int D, int64_t N, float *kbar) {
  pdl_wait();  // inputs written by the kernels before this one
  pdl_trigger();
  const int64_t bh = blockIdx.y * H + blockIdx.x;
  const int d = threadIdx.x;
  if (d >= D) return;
  float s = 0.f;
  for (int64_t p = 0; p < P; ++p) s += part[(bh * P + p) * D + d];
  kbar[bh * D + d] = N > 0 ? s / (float)N : 0.f;
}

// 3. Norms.  blockIdx.x in [0, nqb) -> Q-block; [nqb, nqb+nkb) -> K rows; then V rows.
template <typename T, int EPL, bool CONTIG>
__global__ void __launch_bounds__(kThreads)
    norms_kernel(View q, View k, View v, int64_t nqb, int64_t nkb, int centering, float alpha,
                 const float *kbar, float *qmax_sq, float *qkbar, float *qsq, float *kblk, float *vblk,
                 int n_sink, SinkCand *cand) {
  pdl_wait();  // inputs written by the kernels before this one
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t b = blockIdx.z, h = blockIdx.y, bx = blockIdx.x;
  const int64_t bh = b * q.H + h;
  const int D = 32 * EPL;
  __shared__ float wmax[kWarps];
  __shared__ float knorm[kKVRows];  // key blocks with sinks: each row's squared norm
  float kb[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) kb[e] = centering ? kbar[bh * D + lane * EPL + e] : 0.f;

  float best = 0.f;  // maxima of non-negative quantities start at 0
  if (bx < nqb) {
    // Q-block: per-row |q|^2 and alpha * q.kbar
    const T *base = reinterpret_cast<const T *>(q.ptr) + b * q.sB + h * q.sH;
    const int64_t r0 = bx * kQRows, r1 = min(q.S, r0 + kQRows);
    for (int64_t r = r0 + warp; r < r1; r += kWarps) {
      float x[EPL];
      load_row<T, EPL, CONTIG>(base + r * q.sS, q.sD, lane, x);
      float ss = 0.f, dk = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        ss = fmaf(x[e], x[e], ss);
        dk = fmaf(x[e], kb[e], dk);
      }
      ss = warp_sum(ss);
      dk = warp_sum(dk);
      best = fmaxf(best, ss);
      if (lane == 0) {
        qkbar[bh * q.S + r] = alpha * dk;
        qsq[bh * q.S + r] = ss;  // per-row |q|^2, turned into the row's shift by shift_kernel
      }
    }
  } else if (bx < nqb + nkb) {
    // K rows: |k - kbar|^2 (kbar = 0 when not centering)
    const T *base = reinterpret_cast<const T *>(k.ptr) + b * k.sB + h * k.sH;
    const int64_t r0 = (bx - nqb) * kKVRows, r1 = min(k.S, r0 + kKVRows);
    for (int64_t r = r0 + warp; r < r1; r += kWarps) {
      float x[EPL];
      load_row<T, EPL, CONTIG>(base + r * k.sS, k.sD, lane, x);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        float c = x[e] - kb[e];
        ss = fmaf(c, c, ss);
      }
      ss = warp_sum(ss);
      best = fmaxf(best, ss);
      if (n_sink > 0 && lane == 0) knorm[r - r0] = ss;
    }
  } else {
    // V rows: max element square
    const T *base = reinterpret_cast<const T *>(v.ptr) + b * v.sB + h * v.sH;
    const int64_t r0 = (bx - nqb - nkb) * kKVRows, r1 = min(v.S, r0 + kKVRows);
    for (int64_t r = r0 + warp; r < r1; r += kWarps) {
      float x[EPL];
      load_row<T, EPL, CONTIG>(base + r * v.sS, v.sD, lane, x);
#pragma unroll
      for (int e = 0; e < EPL; ++e) best = fmaxf(best, x[e] * x[e]);
    }
    best = warp_max(best);
  }
  if (lane == 0) wmax[warp] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    float mx = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, wmax[w]);
    if (bx < nqb) qmax_sq[bh * nqb + bx] = mx;
    else if (bx < nqb + nkb) kblk[bh * nkb + (bx - nqb)] = mx;
    else vblk[bh * nkb + (bx - nqb - nkb)] = mx;
  }
  if (n_sink > 0 && bx >= nqb && bx < nqb + nkb && warp == 0) {
    // this block's n_sink + 1 loudest keys, in sink order (its rows' norms are in knorm,
    // written before the barrier above)
    const int64_t r0 = (bx - nqb) * kKVRows;
    const int cnt = (int)min((int64_t)kKVRows, k.S - r0);
    SinkCand *out = cand + (bh * nkb + (bx - nqb)) * kCandPerBlock;
    float pv = INFINITY;
    int32_t pi = -1;
    for (int t = 0; t <= n_sink; ++t) {
      float bv = -1.f;
      int32_t bi = INT_MAX;
      for (int e = lane; e < cnt; e += 32) {
        const float v = knorm[e];
        const int32_t i = (int32_t)(r0 + e);
        if (sink_after(v, i, pv, pi) && sink_before(v, i, bv, bi)) {
          bv = v;
          bi = i;
        }
      }
      warp_best_sink(bv, bi);
      if (lane == 0) out[t] = SinkCand{bv, bi};
      pv = bv;
      pi = bi;
    }
  }
}

// 3'. The norms pass with 16-byte loads: the same outputs as norms_kernel, for rows that start on
// 16-byte boundaries.  A CTA streams kBlocksPerCta consecutive blocks of one kind (Q-blocks of
// 128 rows, K- or V-blocks of 256): one pass of the CTA covers at most 128 rows (8 warps x RPW
// rows x up to kRawLoads loads per lane), and the next pass's loads are issued before the current
// pass is reduced, so the loads never drain at a block boundary.  Each thread keeps one maximum
// per block; the CTA reduces them once at the end.
constexpr int kRawLoads = 8;  // most 16-byte loads per lane and pass
constexpr int kBlocksPerCta = 4;
template <typename T, int VEC>
__device__ __forceinline__ void unpack16(const uint4 &u, float (&x)[VEC]) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  } else {
    x[0] = __uint_as_float(u.x);
    x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z);
    x[3] = __uint_as_float(u.w);
  }
}

// One pass of a CTA: rows rb + sub + u*step (u < kRawLoads) that lie below r1.
template <typename T, int U>
__device__ __forceinline__ void load_pass(const T *base, int64_t sS, int64_t r, int64_t step, int64_t r1,
                                          uint4 (&raw)[U]) {
#pragma unroll
  for (int u = 0; u < U; ++u)
    if (r + u * step < r1) raw[u] = __ldg(reinterpret_cast<const uint4 *>(base + (r + u * step) * sS));
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
    norms_vec_kernel(View q, View k, View v, int64_t nqb, int64_t nkb, int centering, float alpha,
                     const float *kbar, float *qmax_sq, float *qkbar, float *qsq, float *kblk, float *vblk,
                     int n_sink, SinkCand *cand) {
  pdl_wait();  // inputs written by the kernels before this one
  pdl_trigger();
  using V = Vec16<T, D>;
  constexpr int U = kRawLoads * kWarps * V::RPW <= 128 ? kRawLoads : 128 / (kWarps * V::RPW);
  constexpr int kPass = kWarps * V::RPW * U;  // rows one pass covers (64 or 128)
  static_assert(kQRows % kPass == 0 && kKVRows % kPass == 0, "a pass stays inside one block");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / V::LPR, li = lane % V::LPR;
  const int64_t b = blockIdx.z, h = blockIdx.y;
  const int64_t bh = b * q.H + h;
  const int64_t step = (int64_t)kWarps * V::RPW;
  const int64_t nq4 = ceil_div(nqb, kBlocksPerCta), nk4 = ceil_div(nkb, kBlocksPerCta);
  const int64_t cx = blockIdx.x;
  const int kind = cx < nq4 ? 0 : (cx < nq4 + nk4 ? 1 : 2);  // Q, K or V blocks
  const int64_t blk0 = (kind == 0 ? cx : (kind == 1 ? cx - nq4 : cx - nq4 - nk4)) * kBlocksPerCta;
  const int64_t rows_per_blk = kind == 0 ? kQRows : kKVRows;
  const View &t = kind == 0 ? q : (kind == 1 ? k : v);
  const int64_t n_blk = kind == 0 ? nqb : nkb;
  const int nb = (int)min((int64_t)kBlocksPerCta, n_blk - blk0);  // blocks of this CTA
  const int64_t r0 = blk0 * rows_per_blk, r1 = min(t.S, r0 + nb * rows_per_blk);
  __shared__ float wmax[kBlocksPerCta][kWarps];
  __shared__ float knorm[kBlocksPerCta * kKVRows];  // key blocks with sinks: each row's squared norm

  float kb[V::VEC];
#pragma unroll
  for (int e = 0; e < V::VEC; ++e) kb[e] = (centering && kind < 2) ? kbar[bh * D + li * V::VEC + e] : 0.f;
  float best[kBlocksPerCta];
#pragma unroll
  for (int i = 0; i < kBlocksPerCta; ++i) best[i] = 0.f;  // maxima of non-negative quantities start at 0
  const T *base = reinterpret_cast<const T *>(t.ptr) + b * t.sB + h * t.sH + li * V::VEC;
  const int n_pass = (int)ceil_div(r1 - r0, (int64_t)kPass);
  const int pass_per_blk = (int)(rows_per_blk / kPass);

  // one pass: the rows' norms (Q: |q|^2 and alpha*q.kbar per row; K: |k - kbar|^2; V: max v^2)
  auto reduce_pass = [&](const uint4 (&raw)[U], int pass) {
    const int64_t r = r0 + (int64_t)pass * kPass + warp * V::RPW + sub;
    const int bi = pass / pass_per_blk;
    float bm = 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool ok = r + u * step < r1;
      float x[V::VEC];
      unpack16<T, V::VEC>(raw[u], x);
      if (kind == 2) {
        if (ok) {
#pragma unroll
          for (int e = 0; e < V::VEC; ++e) bm = fmaxf(bm, x[e] * x[e]);
        }
        continue;
      }
      float ss = 0.f, dk = 0.f;
      if (ok) {
#pragma unroll
        for (int e = 0; e < V::VEC; ++e) {
          const float c = x[e] - (kind == 1 ? kb[e] : 0.f);
          ss = fmaf(c, c, ss);
          dk = fmaf(x[e], kb[e], dk);
        }
      }
      ss = row_sum<V::LPR>(ss);
      if (kind == 0) dk = row_sum<V::LPR>(dk);
      if (ok) {
        bm = fmaxf(bm, ss);
        const int64_t row = r + u * step;
        if (kind == 0 && li == 0) {
          qkbar[bh * q.S + row] = alpha * dk;
          qsq[bh * q.S + row] = ss;  // per-row |q|^2, turned into the row's shift by shift_kernel
        }
        if (kind == 1 && n_sink > 0 && li == 0) knorm[row - r0] = ss;
      }
    }
#pragma unroll
    for (int i = 0; i < kBlocksPerCta; ++i)
      if (i == bi) best[i] = fmaxf(best[i], bm);
  };

  // passes two at a time, the next pass's loads in flight while the current one is reduced
  uint4 ra[U], rb2[U];
  const int64_t rw = r0 + warp * V::RPW + sub;
  if (n_pass > 0) load_pass<T, U>(base, t.sS, rw, step, r1, ra);
  for (int pass = 0; pass < n_pass; pass += 2) {
    if (pass + 1 < n_pass) load_pass<T, U>(base, t.sS, rw + (int64_t)(pass + 1) * kPass, step, r1, rb2);
    reduce_pass(ra, pass);
    if (pass + 1 < n_pass) {
      if (pass + 2 < n_pass) load_pass<T, U>(base, t.sS, rw + (int64_t)(pass + 2) * kPass, step, r1, ra);
      reduce_pass(rb2, pass + 1);
    }
  }
  // the block maxima over the CTA, once
#pragma unroll
  for (int i = 0; i < kBlocksPerCta; ++i) {
    const float m = warp_max(best[i]);
    if (lane == 0) wmax[i][warp] = m;
  }
  __syncthreads();
  if (threadIdx.x < nb) {
    const int i = threadIdx.x;
    float mx = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, wmax[i][w]);
    const int64_t blk = blk0 + i;
    if (kind == 0) qmax_sq[bh * nqb + blk] = mx;
    else if (kind == 1) kblk[bh * nkb + blk] = mx;
    else vblk[bh * nkb + blk] = mx;
  }
  if (n_sink > 0 && kind == 1 && warp < nb) {
    // key block blk0 + warp: its n_sink + 1 loudest keys, in sink order (its rows' norms are in
    // knorm, written before the barrier above)
    const int64_t blk = blk0 + warp;
    const int64_t kr0 = blk * kKVRows;
    const int cnt = (int)min((int64_t)kKVRows, k.S - kr0);
    SinkCand *out = cand + (bh * nkb + blk) * kCandPerBlock;
    float pv = INFINITY;
    int32_t pi = -1;
    for (int tt = 0; tt <= n_sink; ++tt) {
      float bv = -1.f;
      int32_t bi = INT_MAX;
      for (int e = lane; e < cnt; e += 32) {
        const float vv = knorm[warp * kKVRows + e];
        const int32_t i = (int32_t)(kr0 + e);
        if (sink_after(vv, i, pv, pi) && sink_before(vv, i, bv, bi)) {
          bv = vv;
          bi = i;
        }
      }
      warp_best_sink(bv, bi);
      if (lane == 0) out[tt] = SinkCand{bv, bi};
      pv = bv;
      pi = bi;
    }
  }
}

// 3b. Key sinks of head (b, h): the n_sink + 1 loudest keys over the blocks' candidates.
// tau = the (n_sink+1)-th norm (0 if there is none); the sinks are the picks strictly above
// tau, so the largest norm of every other key is tau.  Writes sink_idx (ascending, INT32_MAX
// pads), kmax_sq = tau, and the sinks' raw key and value rows.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    sink_select_kernel(View k, View v, int64_t nkb, int n_sink, const SinkCand *cand, int32_t *sink_idx,
                       float *sink_k, float *sink_v, float *kmax_sq) {
  pdl_wait();  // inputs written by the kernels before this one
  pdl_trigger();
  const int64_t b = blockIdx.y, h = blockIdx.x;
  const int64_t bh = b * k.H + h;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const SinkCand *c = cand + bh * nkb * kCandPerBlock;
  const int64_t M = nkb * (n_sink + 1);
  __shared__ float wv[kWarps];
  __shared__ int32_t wi[kWarps];
  __shared__ float pick_v[FM_MAX_SINKS + 1];
  __shared__ int32_t pick_i[FM_MAX_SINKS + 1];
  __shared__ int32_t list[FM_MAX_SINKS];
  float pv = INFINITY;
  int32_t pi = -1;
  for (int t = 0; t <= n_sink; ++t) {
    float bv = -1.f;
    int32_t bi = INT_MAX;
    for (int64_t e = threadIdx.x; e < M; e += kThreads) {
      const SinkCand x = c[(e / (n_sink + 1)) * kCandPerBlock + e % (n_sink + 1)];
      if (x.v >= 0.f && sink_after(x.v, x.idx, pv, pi) && sink_before(x.v, x.idx, bv, bi)) {
        bv = x.v;
        bi = x.idx;
      }
    }
    warp_best_sink(bv, bi);
    if (lane == 0) {
      wv[warp] = bv;
      wi[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float fv = wv[0];
      int32_t fi = wi[0];
      for (int w = 1; w < kWarps; ++w)
        if (sink_before(wv[w], wi[w], fv, fi)) {
          fv = wv[w];
          fi = wi[w];
        }
      pick_v[t] = fv;
      pick_i[t] = fi;
    }
    __syncthreads();
    pv = pick_v[t];
    pi = pick_i[t];
  }
  if (threadIdx.x == 0) {
    const float tau = pick_v[n_sink] >= 0.f ? pick_v[n_sink] : 0.f;
    int n = 0;
    for (int t = 0; t < n_sink; ++t)
      if (pick_v[t] >= 0.f && pick_v[t] > tau) list[n++] = pick_i[t];
    for (int i = 1; i < n; ++i)  // ascending key order
      for (int j = i; j > 0 && list[j - 1] > list[j]; --j) {
        const int32_t x = list[j];
        list[j] = list[j - 1];
        list[j - 1] = x;
      }
    for (int t = n; t < FM_MAX_SINKS; ++t) list[t] = INT_MAX;
    for (int t = 0; t < FM_MAX_SINKS; ++t) sink_idx[bh * FM_MAX_SINKS + t] = list[t];
    kmax_sq[bh] = tau;
  }
  __syncthreads();
  const int D = (int)k.D;
  const T *kp = reinterpret_cast<const T *>(k.ptr) + b * k.sB + h * k.sH;
  const T *vp = reinterpret_cast<const T *>(v.ptr) + b * v.sB + h * v.sH;
  for (int e = threadIdx.x; e < FM_MAX_SINKS * D; e += kThreads) {
    const int slot = e / D, d = e % D;
    const int32_t idx = list[slot];
    float kx = 0.f, vx = 0.f;
    if (idx != INT_MAX) {
      const T a = kp[(int64_t)idx * k.sS + (int64_t)d * k.sD];
      const T w = vp[(int64_t)idx * v.sS + (int64_t)d * v.sD];
      if constexpr (sizeof(T) == 2) {
        kx = __bfloat162float(a);
        vx = __bfloat162float(w);
      } else {
        kx = (float)a;
        vx = (float)w;
      }
    }
    sink_k[(bh * FM_MAX_SINKS + slot) * D + d] = kx;
    sink_v[(bh * FM_MAX_SINKS + slot) * D + d] = vx;
  }
}

// 4. Per head: key max, global V max, then U, m, flag for every Q-block.
__global__ void __launch_bounds__(kThreads)
    finish_kernel(int64_t H, int64_t nqb, int64_t nkb, int64_t n_heads_total, const float *kblk,
                  const float *vblk, double alpha, int C, int gate, const float *qmax_sq,
                  float *kmax_sq, float *vmax_sq, int32_t *m, uint8_t *flag, int kmax_given) {
  pdl_wait();  // inputs written by the kernels before this one
  pdl_trigger();
  const int64_t bh = blockIdx.y * H + blockIdx.x;
  __shared__ float red[2][kWarps];
  float km = 0.f, vm = 0.f;
  for (int64_t i = threadIdx.x; i < nkb; i += kThreads) km = fmaxf(km, kblk[bh * nkb + i]);
  for (int64_t i = threadIdx.x; i < n_heads_total * nkb; i += kThreads) vm = fmaxf(vm, vblk[i]);
  km = warp_max(km);
  vm = warp_max(vm);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { red[0][warp] = km; red[1][warp] = vm; }
  __syncthreads();
  km = 0.f; vm = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) { km = fmaxf(km, red[0][w]); vm = fmaxf(vm, red[1][w]); }
  if (kmax_given) km = kmax_sq[bh];  // the key sinks' pass left the max over the other keys
  __syncthreads();
  if (threadIdx.x == 0) {
    kmax_sq[bh] = km;
    if (bh == 0) vmax_sq[0] = vm;
  }
  const bool v_ok = vm <= (float)FM_VMAX * (float)FM_VMAX;
  const double ksq = sqrt((double)km);
  for (int64_t i = threadIdx.x; i < nqb; i += kThreads) {
    const double U = alpha * sqrt((double)qmax_sq[bh * nqb + i]) * ksq;
    m[bh * nqb + i] = (int32_t)ceil(U) - C;
    flag[bh * nqb + i] = (uint8_t)(v_ok && U <= (double)gate);
  }
}

// 5. Row shifts: b_i = m_i + alpha*q_i.kbar, with m_i = ceil(alpha*|q_i|*sqrt(kmax)) - C
// (per row) or the row's Q-block m.  `shift` holds |q_i|^2 on entry (from norms_kernel).
__global__ void __launch_bounds__(kThreads)
    shift_kernel(int64_t H, int64_t Sq, int64_t nqb, int per_row, double alpha, int C, const float *kmax_sq,
                 const int32_t *m, const float *qkbar, float *shift) {
  pdl_wait();  // inputs written by the kernels before this one
  pdl_trigger();
  const int64_t bh = blockIdx.z * H + blockIdx.y;
  const int64_t r = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (r >= Sq) return;
  const int64_t i = bh * Sq + r;
  int32_t mi;
  if (per_row) {
    const double U = alpha * sqrt((double)shift[i]) * sqrt((double)kmax_sq[bh]);
    mi = (int32_t)ceil(U) - C;
  } else {
    mi = m[bh * nqb + r / kQRows];
  }
  shift[i] = (float)mi + qkbar[i];
}

// ---- the bounds of a ring of ranks (each rank holds one shard of the keys and values) ----
// One rank's statistics block, exchanged (all-gathered) before the ring:
//   float    vmax_sq              (word 0 of a 16-byte header) max v^2 over the shard
//   float    kmax_sq[BH]          max |k - kbar|^2 (or |k|^2) over the shard's keys
//   SinkCand cand[BH][nc]         with key sinks (nc = n_sink + 1): the shard's nc loudest keys
//                                 in sink order, global key index; v = -1 pads
//   float    cand_k[BH][nc][D], cand_v[BH][nc][D]   their raw key and value rows
struct RingLayout {
  int nc;
  size_t off_kmax, off_cand, off_ck, off_cv, total;
};
inline size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }
RingLayout ring_layout(int64_t BH, int64_t D, int n_sink) {
  RingLayout L;
  L.nc = n_sink > 0 ? n_sink + 1 : 0;
  L.off_kmax = 16;
  L.off_cand = align16(L.off_kmax + sizeof(float) * (size_t)BH);
  L.off_ck = align16(L.off_cand + sizeof(SinkCand) * (size_t)(BH * L.nc));
  L.off_cv = L.off_ck + sizeof(float) * (size_t)(BH * L.nc * D);
  L.total = align16(L.off_cv + sizeof(float) * (size_t)(BH * L.nc * D));
  return L;
}

// Block-wide max of non-negative values held one per thread (the result in every thread).
__device__ __forceinline__ float block_max(float v, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float m = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) m = fmaxf(m, red[w]);
  return m;
}

// The nc loudest of M candidates (sink order: louder first, lower index first among equal
// norms), one pick per round over the whole CTA; candidates with v < 0 are absent.  `get(e)`
// returns candidate e.  Picks that run out are {-1, INT_MAX}.
template <typename Get>
__device__ void pick_loudest(int64_t M, int nc, Get get, float *pick_v, int32_t *pick_i, float *wv, int32_t *wi) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float pv = INFINITY;
  int32_t pi = -1;
  for (int t = 0; t < nc; ++t) {
    float bv = -1.f;
    int32_t bi = INT_MAX;
    for (int64_t e = threadIdx.x; e < M; e += kThreads) {
      const SinkCand x = get(e);
      if (x.v >= 0.f && sink_after(x.v, x.idx, pv, pi) && sink_before(x.v, x.idx, bv, bi)) {
        bv = x.v;
        bi = x.idx;
      }
    }
    warp_best_sink(bv, bi);
    if (lane == 0) {
      wv[warp] = bv;
      wi[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float fv = wv[0];
      int32_t fi = wi[0];
      for (int w = 1; w < kWarps; ++w)
        if (sink_before(wv[w], wi[w], fv, fi)) {
          fv = wv[w];
          fi = wi[w];
        }
      pick_v[t] = fv;
      pick_i[t] = fi;
    }
    __syncthreads();
    pv = pick_v[t];
    pi = pick_i[t];
  }
}

// One rank's statistics block from the norms pass over its shard: per head the key max, the V
// max over the whole shard, and (key sinks) the shard's nc loudest keys with their rows.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    ring_local_kernel(View k, View v, int64_t nkb, int64_t n_heads_total, int n_sink, int64_t key_offset,
                      const float *kblk, const float *vblk, const SinkCand *cand, uint8_t *stats, RingLayout L) {
  pdl_wait();  // inputs written by the kernels before this one
  pdl_trigger();
  const int64_t b = blockIdx.y, h = blockIdx.x;
  const int64_t bh = b * k.H + h;
  __shared__ float red[kWarps];
  __shared__ float wv[kWarps];
  __shared__ int32_t wi[kWarps];
  __shared__ float pick_v[FM_MAX_SINKS + 1];
  __shared__ int32_t pick_i[FM_MAX_SINKS + 1];
  float km = 0.f;
  for (int64_t i = threadIdx.x; i < nkb; i += kThreads) km = fmaxf(km, kblk[bh * nkb + i]);
  km = block_max(km, red);
  float *kmax = reinterpret_cast<float *>(stats + L.off_kmax);
  if (threadIdx.x == 0) kmax[bh] = km;
  if (bh == 0) {
    float vm = 0.f;
    for (int64_t i = threadIdx.x; i < n_heads_total * nkb; i += kThreads) vm = fmaxf(vm, vblk[i]);
    vm = block_max(vm, red);
    if (threadIdx.x == 0) reinterpret_cast<float *>(stats)[0] = vm;
  }
  if (L.nc == 0) return;
  const SinkCand *c = cand + bh * nkb * kCandPerBlock;
  const int per = n_sink + 1;  // candidates each K block kept
  pick_loudest(nkb * per, L.nc, [&](int64_t e) { return c[(e / per) * kCandPerBlock + e % per]; }, pick_v, pick_i,
               wv, wi);
  SinkCand *out = reinterpret_cast<SinkCand *>(stats + L.off_cand) + bh * L.nc;
  if (threadIdx.x < L.nc) {
    const int t = threadIdx.x;
    const bool have = pick_v[t] >= 0.f;
    out[t] = have ? SinkCand{pick_v[t], (int32_t)(key_offset + pick_i[t])} : SinkCand{-1.f, INT_MAX};
  }
  const int D = (int)k.D;
  const T *kp = reinterpret_cast<const T *>(k.ptr) + b * k.sB + h * k.sH;
  const T *vp = reinterpret_cast<const T *>(v.ptr) + b * v.sB + h * v.sH;
  float *ck = reinterpret_cast<float *>(stats + L.off_ck) + bh * L.nc * D;
  float *cv = reinterpret_cast<float *>(stats + L.off_cv) + bh * L.nc * D;
  for (int e = threadIdx.x; e < L.nc * D; e += kThreads) {
    const int slot = e / D, d = e % D;
    float kx = 0.f, vx = 0.f;
    if (pick_v[slot] >= 0.f) {
      const int64_t idx = pick_i[slot];
      const T a = kp[idx * k.sS + (int64_t)d * k.sD];
      const T w = vp[idx * v.sS + (int64_t)d * v.sD];
      if constexpr (sizeof(T) == 2) {
        kx = __bfloat162float(a);
        vx = __bfloat162float(w);
      } else {
        kx = (float)a;
        vx = (float)w;
      }
    }
    ck[e] = kx;
    cv[e] = vx;
  }
}

// Every rank's statistics blocks (rank order) -> the bounds over all keys for this rank's
// queries: the key max (or, with key sinks, the n_sink + 1 loudest keys of the union of the
// shards' candidates: the sinks strictly above the (n_sink+1)-th, which is the key max), the
// V max, then U, m and the flag per Q-block as fm_bounds does.
__global__ void __launch_bounds__(kThreads)
    ring_combine_kernel(const uint8_t *stats_all, size_t stats_bytes, int n_ranks, RingLayout L, int n_sink,
                        int64_t H, int64_t nqb, int D, double alpha, int C, int gate, const float *qmax_sq,
                        float *kmax_sq, float *vmax_sq, int32_t *m, uint8_t *flag, int32_t *sink_idx,
                        float *sink_k, float *sink_v) {
  pdl_wait();  // inputs written by the kernels before this one
  pdl_trigger();
  const int64_t bh = (int64_t)blockIdx.y * H + blockIdx.x;
  __shared__ float wv[kWarps];
  __shared__ int32_t wi[kWarps];
  __shared__ float pick_v[FM_MAX_SINKS + 1];
  __shared__ int32_t pick_i[FM_MAX_SINKS + 1];
  __shared__ int32_t list[FM_MAX_SINKS];
  __shared__ int src[FM_MAX_SINKS];
  __shared__ float kmv[2];
  if (threadIdx.x == 0) {
    float km = 0.f, vm = 0.f;
    for (int r = 0; r < n_ranks; ++r) {
      const uint8_t *s = stats_all + (size_t)r * stats_bytes;
      km = fmaxf(km, reinterpret_cast<const float *>(s + L.off_kmax)[bh]);
      vm = fmaxf(vm, reinterpret_cast<const float *>(s)[0]);
    }
    kmv[0] = km;
    kmv[1] = vm;
  }
  __syncthreads();
  float km = kmv[0];
  const float vm = kmv[1];
  if (n_sink > 0) {
    const int nc = L.nc;
    auto get = [&](int64_t e) {
      const uint8_t *s = stats_all + (size_t)(e / nc) * stats_bytes;
      return reinterpret_cast<const SinkCand *>(s + L.off_cand)[bh * nc + e % nc];
    };
    pick_loudest((int64_t)n_ranks * nc, n_sink + 1, get, pick_v, pick_i, wv, wi);
    if (threadIdx.x == 0) {
      const float tau = pick_v[n_sink] >= 0.f ? pick_v[n_sink] : 0.f;
      int n = 0;
      for (int t = 0; t < n_sink; ++t)
        if (pick_v[t] >= 0.f && pick_v[t] > tau) list[n++] = pick_i[t];
      for (int i = 1; i < n; ++i)  // ascending key order
        for (int j = i; j > 0 && list[j - 1] > list[j]; --j) {
          const int32_t x = list[j];
          list[j] = list[j - 1];
          list[j - 1] = x;
        }
      for (int t = n; t < FM_MAX_SINKS; ++t) list[t] = INT_MAX;
      // where each sink's rows sit among the candidates (global key indices are unique)
      for (int t = 0; t < FM_MAX_SINKS; ++t) {
        src[t] = -1;
        for (int64_t e = 0; e < (int64_t)n_ranks * nc && list[t] != INT_MAX; ++e)
          if (get(e).idx == list[t]) src[t] = (int)e;
      }
      for (int t = 0; t < FM_MAX_SINKS; ++t) sink_idx[bh * FM_MAX_SINKS + t] = list[t];
      kmv[0] = tau;
    }
    __syncthreads();
    km = kmv[0];
    for (int e = threadIdx.x; e < FM_MAX_SINKS * D; e += kThreads) {
      const int slot = e / D, d = e % D;
      float kx = 0.f, vx = 0.f;
      if (src[slot] >= 0) {
        const uint8_t *s = stats_all + (size_t)(src[slot] / nc) * stats_bytes;
        const int64_t row = bh * nc + src[slot] % nc;
        kx = reinterpret_cast<const float *>(s + L.off_ck)[row * D + d];
        vx = reinterpret_cast<const float *>(s + L.off_cv)[row * D + d];
      }
      sink_k[(bh * FM_MAX_SINKS + slot) * D + d] = kx;
      sink_v[(bh * FM_MAX_SINKS + slot) * D + d] = vx;
    }
  }
  if (threadIdx.x == 0) {
    kmax_sq[bh] = km;
    if (bh == 0) vmax_sq[0] = vm;
  }
  const bool v_ok = vm <= (float)FM_VMAX * (float)FM_VMAX;
  const double ksq = sqrt((double)km);
  for (int64_t i = threadIdx.x; i < nqb; i += kThreads) {
    const double U = alpha * sqrt((double)qmax_sq[bh * nqb + i]) * ksq;
    m[bh * nqb + i] = (int32_t)ceil(U) - C;
    flag[bh * nqb + i] = (uint8_t)(v_ok && U <= (double)gate);
  }
}

// Every row of t starts on a 16-byte boundary (unit D stride).
bool rows16(const View &t) {
  const int64_t es = t.dtype == FM_F32 ? 4 : 2;
  if (t.sD != 1 || reinterpret_cast<uintptr_t>(t.ptr) % 16) return false;
  return ((t.sB * es) % 16 == 0 || t.B <= 1) && ((t.sH * es) % 16 == 0 || t.H <= 1) &&
         ((t.sS * es) % 16 == 0 || t.S <= 1);
}

template <typename T, int EPL, bool CONTIG>
cudaError_t launch_ksum(const View &k, int64_t P, float *part, cudaStream_t st) {
  const dim3 grid((unsigned)P, (unsigned)k.H, (unsigned)k.B);
  if (CONTIG && rows16(k))
    return launch_pdl(ksum_vec_kernel<T, 32 * EPL>, grid, dim3(kThreads), 0, st, k, P, part);
  return launch_pdl(ksum_kernel<T, EPL, CONTIG>, grid, dim3(kThreads), 0, st, k, P, part);
}

template <typename T, int EPL, bool CONTIG>
cudaError_t launch_norms(const BoundsArgs &a, const WsLayout &w, float *kblk, float *vblk, SinkCand *cand,
                         cudaStream_t st) {
  const int64_t nx = a.nqb + 2 * w.nkb;
  if (nx == 0) return cudaSuccess;
  const dim3 grid((unsigned)nx, (unsigned)a.q.H, (unsigned)a.q.B);
  if (CONTIG && rows16(a.q) && rows16(a.k) && rows16(a.v)) {
    const int64_t nx4 = ceil_div(a.nqb, kBlocksPerCta) + 2 * ceil_div(w.nkb, kBlocksPerCta);
    return launch_pdl(norms_vec_kernel<T, 32 * EPL>, dim3((unsigned)nx4, (unsigned)a.q.H, (unsigned)a.q.B),
                      dim3(kThreads), 0, st, a.q, a.k, a.v, a.nqb, w.nkb, a.centering, (float)a.alpha, a.kbar,
                      a.qmax_sq, a.qkbar, a.shift, kblk, vblk, a.n_sink, cand);
  }
  return launch_pdl(norms_kernel<T, EPL, CONTIG>, grid, dim3(kThreads), 0, st, a.q, a.k, a.v, a.nqb, w.nkb,
                    a.centering, (float)a.alpha, a.kbar, a.qmax_sq, a.qkbar, a.shift, kblk, vblk, a.n_sink, cand);
}

template <typename T, int EPL, bool CONTIG>
cudaError_t launch_ring_local_typed(const BoundsArgs &a, const WsLayout &w, const float *ksum_total, int64_t N_total,
                                    int64_t key_offset, void *stats, cudaStream_t st) {
  const int64_t B = a.q.B, H = a.q.H;
  char *ws = reinterpret_cast<char *>(a.ws);
  float *kblk = reinterpret_cast<float *>(ws + w.off_kb);
  float *vblk = reinterpret_cast<float *>(ws + w.off_vb);
  SinkCand *cand = reinterpret_cast<SinkCand *>(ws + w.off_cand);
  const int D = (int)a.q.D;
  const dim3 heads((unsigned)H, (unsigned)B);
  cudaError_t e;
  // every rank divides the same ring-wide sums by the same count: one key mean for all
  if (a.centering && N_total > 0)
    e = launch_pdl(kmean_kernel, heads, dim3(128), 0, st, ksum_total, H, (int64_t)1, D, N_total, a.kbar);
  else
    e = cudaMemsetAsync(a.kbar, 0, sizeof(float) * (size_t)(B * H * D), st);
  if (e != cudaSuccess) return e;
  e = launch_norms<T, EPL, CONTIG>(a, w, kblk, vblk, cand, st);
  if (e != cudaSuccess) return e;
  const RingLayout L = ring_layout(B * H, D, a.n_sink);
  e = launch_pdl(ring_local_kernel<T>, heads, dim3(kThreads), 0, st, a.k, a.v, w.nkb, B * H, a.n_sink, key_offset, kblk,
                 vblk, cand, reinterpret_cast<uint8_t *>(stats), L);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, int EPL, bool CONTIG>
cudaError_t launch_typed(const BoundsArgs &a, const WsLayout &w, cudaStream_t st) {
  const int64_t B = a.q.B, H = a.q.H, N = a.k.S;
  char *ws = reinterpret_cast<char *>(a.ws);
  float *part = reinterpret_cast<float *>(ws + w.off_part);
  float *kblk = reinterpret_cast<float *>(ws + w.off_kb);
  float *vblk = reinterpret_cast<float *>(ws + w.off_vb);
  SinkCand *cand = reinterpret_cast<SinkCand *>(ws + w.off_cand);
  const int D = (int)a.q.D;
  const dim3 heads((unsigned)H, (unsigned)B);
  cudaError_t e = cudaSuccess;
  if (a.centering && N > 0) {
    e = launch_ksum<T, EPL, CONTIG>(a.k, w.P, part, st);
    if (e == cudaSuccess) e = launch_pdl(kmean_kernel, heads, dim3(128), 0, st, part, H, w.P, D, N, a.kbar);
  } else {
    e = cudaMemsetAsync(a.kbar, 0, sizeof(float) * (size_t)(B * H * D), st);
  }
  if (e != cudaSuccess) return e;
  e = launch_norms<T, EPL, CONTIG>(a, w, kblk, vblk, cand, st);
  if (e != cudaSuccess) return e;
  if (a.n_sink > 0) {
    e = launch_pdl(sink_select_kernel<T>, heads, dim3(kThreads), 0, st, a.k, a.v, w.nkb, a.n_sink, cand, a.sink_idx,
                   a.sink_k, a.sink_v, a.kmax_sq);
    if (e != cudaSuccess) return e;
  }
  e = launch_pdl(finish_kernel, heads, dim3(kThreads), 0, st, H, a.nqb, w.nkb, B * H, kblk, vblk, a.alpha, a.C, a.gate,
                 a.qmax_sq, a.kmax_sq, a.vmax_sq, a.m, a.flag, (int)(a.n_sink > 0));
  if (e != cudaSuccess) return e;
  if (a.q.S > 0) {
    e = launch_pdl(shift_kernel, dim3((unsigned)ceil_div(a.q.S, kThreads), (unsigned)H, (unsigned)B), dim3(kThreads),
                   0, st, H, a.q.S, a.nqb, a.per_row, a.alpha, a.C, a.kmax_sq, a.m, a.qkbar, a.shift);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

bool contiguous_rows(const View &t) {
  const size_t es = t.dtype == FM_F32 ? 4 : 2;
  const size_t vec = es * (size_t)(t.D / 32);  // bytes a lane loads
  if (t.sD != 1) return false;
  if (reinterpret_cast<uintptr_t>(t.ptr) % vec) return false;
  return ((t.sB * es) % vec == 0 || t.B == 1) && ((t.sH * es) % vec == 0 || t.H == 1) &&
         ((t.sS * es) % vec == 0 || t.S <= 1);
}

}  // namespace

size_t bounds_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t D) {
  return ws_layout(B, H, N, D).total;
}

size_t ring_stats_bytes(int64_t B, int64_t H, int64_t D, int n_sink) { return ring_layout(B * H, D, n_sink).total; }

cudaError_t launch_ring_key_sums(const View &k, float *ksum, void *ws, cudaStream_t st) {
  const int64_t B = k.B, H = k.H, N = k.S;
  const int D = (int)k.D;
  if (B * H == 0) return cudaSuccess;
  if (N == 0) return cudaMemsetAsync(ksum, 0, sizeof(float) * (size_t)(B * H * D), st);
  const WsLayout w = ws_layout(B, H, N, D);
  float *part = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + w.off_part);
  const bool contig = contiguous_rows(k);
  const dim3 heads((unsigned)H, (unsigned)B);
  cudaError_t e;
  if (k.dtype == FM_BF16)
    e = D == 128 ? (contig ? launch_ksum<__nv_bfloat16, 4, true>(k, w.P, part, st)
                           : launch_ksum<__nv_bfloat16, 4, false>(k, w.P, part, st))
                 : (contig ? launch_ksum<__nv_bfloat16, 2, true>(k, w.P, part, st)
                           : launch_ksum<__nv_bfloat16, 2, false>(k, w.P, part, st));
  else
    e = D == 128 ? (contig ? launch_ksum<float, 4, true>(k, w.P, part, st) : launch_ksum<float, 4, false>(k, w.P, part, st))
                 : (contig ? launch_ksum<float, 2, true>(k, w.P, part, st) : launch_ksum<float, 2, false>(k, w.P, part, st));
  if (e != cudaSuccess) return e;
  // the ordered sum of the partials, divided by 1
  e = launch_pdl(kmean_kernel, heads, dim3(128), 0, st, part, H, w.P, D, (int64_t)1, ksum);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_bounds_local(const BoundsArgs &a, const float *ksum_total, int64_t N_total, int64_t key_offset,
                                void *stats, cudaStream_t st) {
  const WsLayout w = ws_layout(a.q.B, a.q.H, a.k.S, a.q.D);
  const bool contig = contiguous_rows(a.q) && contiguous_rows(a.k) && contiguous_rows(a.v);
  const bool bf16 = a.q.dtype == FM_BF16;
  const bool d128 = a.q.D == 128;
#define FM_RING_LOCAL(T, E, C) launch_ring_local_typed<T, E, C>(a, w, ksum_total, N_total, key_offset, stats, st)
  if (bf16) {
    if (d128) return contig ? FM_RING_LOCAL(__nv_bfloat16, 4, true) : FM_RING_LOCAL(__nv_bfloat16, 4, false);
    return contig ? FM_RING_LOCAL(__nv_bfloat16, 2, true) : FM_RING_LOCAL(__nv_bfloat16, 2, false);
  }
  if (d128) return contig ? FM_RING_LOCAL(float, 4, true) : FM_RING_LOCAL(float, 4, false);
  return contig ? FM_RING_LOCAL(float, 2, true) : FM_RING_LOCAL(float, 2, false);
#undef FM_RING_LOCAL
}

cudaError_t launch_bounds_combine(const BoundsArgs &a, const void *stats_all, int n_ranks, cudaStream_t st) {
  const int64_t B = a.q.B, H = a.q.H;
  const int D = (int)a.q.D;
  const RingLayout L = ring_layout(B * H, D, a.n_sink);
  const dim3 heads((unsigned)H, (unsigned)B);
  cudaError_t e = launch_pdl(ring_combine_kernel, heads, dim3(kThreads), 0, st,
                             reinterpret_cast<const uint8_t *>(stats_all), L.total, n_ranks, L, a.n_sink, H, a.nqb, D,
                             a.alpha, a.C, a.gate, a.qmax_sq, a.kmax_sq, a.vmax_sq, a.m, a.flag, a.sink_idx,
                             a.sink_k, a.sink_v);
  if (e != cudaSuccess) return e;
  if (a.q.S > 0) {
    e = launch_pdl(shift_kernel, dim3((unsigned)ceil_div(a.q.S, kThreads), (unsigned)H, (unsigned)B), dim3(kThreads),
                   0, st, H, a.q.S, a.nqb, a.per_row, a.alpha, a.C, a.kmax_sq, a.m, a.qkbar, a.shift);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_bounds(const BoundsArgs &a, cudaStream_t st) {
  const WsLayout w = ws_layout(a.q.B, a.q.H, a.k.S, a.q.D);
  const bool contig = contiguous_rows(a.q) && contiguous_rows(a.k) && contiguous_rows(a.v);
  const bool bf16 = a.q.dtype == FM_BF16;
  const bool d128 = a.q.D == 128;
  if (bf16) {
    if (d128) return contig ? launch_typed<__nv_bfloat16, 4, true>(a, w, st) : launch_typed<__nv_bfloat16, 4, false>(a, w, st);
    return contig ? launch_typed<__nv_bfloat16, 2, true>(a, w, st) : launch_typed<__nv_bfloat16, 2, false>(a, w, st);
  }
  if (d128) return contig ? launch_typed<float, 4, true>(a, w, st) : launch_typed<float, 4, false>(a, w, st);
  return contig ? launch_typed<float, 2, true>(a, w, st) : launch_typed<float, 2, false>(a, w, st);
}

}  // namespace fm
