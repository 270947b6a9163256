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
// Launches (all deterministic: sums in a fixed order; maxima in shared memory or by integer
// atomicMax on the bits of non-negative floats, whose result does not depend on the order):
//   1. ksum    (centering only) partial key sums, P row ranges per head  -> workspace; the last
//              CTA of a head to finish adds the P partials in their fixed order and
//              divides by N                                                -> kbar
//   (2. kmean  the same ordered sum as a launch of its own, for the ring's key sums)
//   3. main    the norms over Q-blocks, K row-blocks and V row-blocks: row norms via warp
//              shuffles; per-block maxima -> qmax_sq (Q) and the workspace (K, V);
//              qkbar per row; with key sinks, each K block's n_sink + 1 loudest keys.  One of
//              three kernels by layout: norms_bulk_kernel (packed bf16 rows of D = 128, staged
//              through shared memory by bulk copies), norms_vec_kernel (rows on 16-byte
//              boundaries), norms_kernel (any strides)
//   3b. sinks  (key sinks only) per head: the n_sink + 1 loudest keys over the blocks'
//              candidates; the sinks and the max over the other keys ("Kernel reference:
//              ring_attention_const_max_fwd", section "Adapting this kernel")
//   4. finish  per 2048 query rows of a head: the head's key max, the global V max (folded in by
//              the norms pass with atomics on a zeroed workspace word), U, m and flag of its 16
//              Q-blocks, and every row's shift b_i = m_i + alpha*q_i.kbar (m_i per row or per
//              Q-block)
// One memset before them zeroes the V-max word and the per-head arrival counters of step 1;
// without centering the finish writes kbar as zeros.
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
  // zeroed at the start of each bounds pass: the V-max word, then one arrival counter per head
  size_t off_zero, zero_bytes;
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
  w.off_zero = w.off_cand + sizeof(SinkCand) * (size_t)(B * H * w.nkb * kCandPerBlock);
  w.off_zero = (w.off_zero + 15) & ~(size_t)15;
  w.zero_bytes = 16 + sizeof(unsigned int) * (size_t)(B * H);
  w.total = (w.off_zero + w.zero_bytes + 255) & ~(size_t)255;
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

// The key mean from the P partial sums of head bh, by the last of the head's P CTAs to write
// its partial (a counter per head, zeroed before the launch): the partials added in the order
// p = 0 .. P-1 whichever CTA arrives last, then divided by N.  count == nullptr: no mean (the
// ring's key sums, which another launch adds up).
__device__ __forceinline__ void key_mean_if_last(const float *part, int64_t bh, int64_t P, int D,
                                                 unsigned int *count, int64_t N, float *kbar) {
  if (count == nullptr) return;
  __shared__ unsigned int arrived;
  __threadfence();  // this CTA's partial, visible before its arrival is counted
  __syncthreads();
  if (threadIdx.x == 0) arrived = atomicAdd(&count[bh], 1u);
  __syncthreads();
  if (arrived != (unsigned int)(P - 1)) return;
  __threadfence();
  if (threadIdx.x < D) {
    float s = 0.f;
    for (int64_t p = 0; p < P; ++p) s += __ldcg(&part[(bh * P + p) * D + threadIdx.x]);
    kbar[bh * D + threadIdx.x] = N > 0 ? s / (float)N : 0.f;
  }
}

// 1. Partial key sums: CTA (p, h, b) sums rows [p*len, (p+1)*len) of head (b, h).
template <typename T, int EPL, bool CONTIG>
__global__ void __launch_bounds__(kThreads)
    ksum_kernel(View k, int64_t P, float *part, unsigned int *count, int64_t N, float *kbar) {
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
  key_mean_if_last(part, b * k.H + h, P, D, count, N, kbar);
}

// ---- rows that start on 16-byte boundaries: 16-byte loads, several rows in flight per lane --
// A row of D elements is spread over LPR lanes with VEC consecutive elements each, so one warp
// load covers RPW = 32 / LPR rows; each lane keeps kUnroll such loads in flight before it
// reduces, which is what keeps HBM busy (one 256-byte row per warp at a time is not enough).
constexpr int kUnroll = 8;
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
__global__ void __launch_bounds__(kThreads)
    ksum_vec_kernel(View k, int64_t P, float *part, unsigned int *count, int64_t N, float *kbar) {
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
  key_mean_if_last(part, b * k.H + h, P, D, count, N, kbar);
}

// 2. Key mean: ordered sum of the P partials of head (b, h), divided by N (the ring's key sums
// and key mean; the single-GPU pass folds this into step 1).
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
                 int n_sink, SinkCand *cand, float *vmax_all) {
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
    else {
      vblk[bh * nkb + (bx - nqb - nkb)] = mx;
      if (vmax_all) atomicMax(reinterpret_cast<int *>(vmax_all), __float_as_int(mx));  // v^2 >= 0: bits order as values
    }
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

// fp32x2 arithmetic: two floats in one 64-bit register, one instruction for both (sm_100 on).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_sum(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// One lane's part of a row's sums over its VEC consecutive elements: ss = sum (x - kb)^2
// (CENTER) or sum x^2, and dk = sum x*kb (DOT).  Two fp32x2 chains (the even and the odd
// elements) are added at the end; the kernels whose outputs must agree bit for bit all sum
// this way.
template <int VEC, bool CENTER, bool DOT>
__device__ __forceinline__ void lane_sums(const float (&x)[VEC], const float (&kb)[VEC], float &ss, float &dk) {
  uint64_t s2 = 0, d2 = 0;  // (+0, +0)
#pragma unroll
  for (int e = 0; e < VEC; e += 2) {
    const uint64_t x2 = f2(x[e], x[e + 1]);
    const uint64_t c2 = CENTER ? f2_add(x2, f2(-kb[e], -kb[e + 1])) : x2;  // x + (-kb) is x - kb
    s2 = f2_fma(c2, c2, s2);
    if (DOT) d2 = f2_fma(x2, f2(kb[e], kb[e + 1]), d2);
  }
  ss = f2_sum(s2);
  if (DOT) dk = f2_sum(d2);
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
                     int n_sink, SinkCand *cand, float *vmax_all) {
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
        if (kind == 0) lane_sums<V::VEC, false, true>(x, kb, ss, dk);
        else lane_sums<V::VEC, true, false>(x, kb, ss, dk);
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
    else {
      vblk[bh * nkb + blk] = mx;
      if (vmax_all) atomicMax(reinterpret_cast<int *>(vmax_all), __float_as_int(mx));  // v^2 >= 0: bits order as values
    }
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

// 3''. The norms pass staged through shared memory by bulk copies, for bf16 rows of D = 128 that
// lie back to back (unit D stride, row stride D, 16-byte aligned).
//
// One CTA per SM takes a contiguous run of the blocks of every head -- Q-blocks of 128 rows,
// then K-blocks and V-blocks of 256, runs cut by bytes so that every CTA streams about as much.
// One producer lane copies the run's rows into a ring of 32 KiB shared-memory stages
// (cp.async.bulk, one copy per 128 rows, completion counted in bytes on the stage's mbarrier);
// the copies run ahead of the arithmetic by the whole ring.  Each of the kNbWarps consumer warps
// takes 8 rows of every stage (16 lanes a row, 8 elements a lane), moves them to registers and
// releases the stage at once.  Per pair of rows the four rows' sums (|q|^2 and q.kbar, or
// |k - kbar|^2) are reduced over their 16 lanes together: at each of the four shuffle levels a
// lane keeps half of its remaining sums and sends the other half, so four rows take 5 shuffles
// instead of 16.  The pairs added at each level are the ones of norms_vec_kernel's row_sum, so
// the sums are the same bits.  V needs only max v^2: the max of |v| is taken on the bf16 values
// widened by a shift or a mask (no conversion), and squared once at the end -- the same value,
// since squaring is monotonic, and a NaN is skipped as fmaxf skips it.  The block's
// maximum over the warps goes through a shared-memory slot; the last warp to finish a block
// (an atomic count) writes its results, and with key sinks picks its candidates, while the
// others go on.  Eight slots: a warp can run at most kNbStages blocks ahead of the slowest.  The
// V blocks' maxima also go into one shared-memory word, which the last consumer warp to finish
// folds into the global V max (vmax_all, when given) with one atomic per CTA.
// Every wait is bounded in time; on expiry the kernel records the failure in the device error
// word and every role stops at its next wait (the producer after its own copies have landed).
constexpr int kNbWarps = 16;                     // consumer warps
constexpr int kNbThreads = 32 * (kNbWarps + 1);  // + the producer warp
constexpr int kNbStages = 6;
constexpr int kNbSlots = 8;  // > kNbStages
constexpr int kNbTileRows = 128;
constexpr int kNbRowBytes = 128 * 2;  // D = 128 bf16
constexpr int kNbTileBytes = kNbTileRows * kNbRowBytes;
constexpr int kNbRowsPerWarp = kNbTileRows / kNbWarps;       // rows of a stage per consumer warp
constexpr int kNbGroups = kNbRowsPerWarp / 8;                 // groups of four row pairs
constexpr int kNbOffBar = kNbStages * kNbTileBytes;          // full[s], then empty[s]
constexpr int kNbOffMax = kNbOffBar + 2 * kNbStages * 8;     // [kNbSlots] block maxima (fp32 bits)
constexpr int kNbOffCnt = kNbOffMax + kNbSlots * 4;          // [kNbSlots] warps done with the block
constexpr int kNbOffKnorm = kNbOffCnt + kNbSlots * 4;        // [kNbSlots][kKVRows] key norms (sinks)
constexpr int kNbOffAbort = kNbOffKnorm + kNbSlots * kKVRows * 4;
constexpr int kNbSmem = kNbOffAbort + 16 + 128;  // + slack to align the base to 128 bytes
static_assert(kNbRowsPerWarp % 8 == 0, "each consumer warp reduces whole groups of 4 row pairs per stage");
static_assert(kNbSlots > kNbStages && (kNbSlots & (kNbSlots - 1)) == 0, "slots outnumber the stages");

__device__ __forceinline__ uint32_t nb_smem(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ bool nb_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Poll until the phase of `bar` with parity `parity` completes (true), the time limit passes,
// or -- when `abort_flag` is given -- another role of the CTA has given up (false).  The first
// wait of the launch to run out records itself: role code, tag, block, thread.
__device__ __noinline__ bool nb_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned long long timeout_ns, unsigned int *err, unsigned int tag) {
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint32_t it = 1;; ++it) {
    if (nb_try(bar, parity)) return true;
    if ((it & 31) == 0) {
      if (abort_flag && *abort_flag) return false;
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > timeout_ns) {
        if (abort_flag) *abort_flag = 1;
        if (err && atomicCAS(err, 0u, kDevErrTimeoutBounds) == 0u) {
          err[1] = tag;
          err[2] = blockIdx.x;
          err[3] = blockIdx.y;
          err[4] = blockIdx.z;
          err[5] = threadIdx.x;
        }
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool nb_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                        unsigned long long timeout_ns, unsigned int *err, unsigned int tag) {
  if (nb_try(bar, parity)) return true;
  return nb_wait_slow(bar, parity, abort_flag, timeout_ns, err, tag);
}
// Sums over the 16 lanes of a row for four rows at once: v[u] is this lane's part of row u's sum;
// the result is the whole sum of row li >> 2 (li = lane % 16).  Level by level the pairs added
// are those of row_sum<16> (lane ^ 8, ^ 4, ^ 2, ^ 1), so each row's sum has the same bits.
__device__ __forceinline__ float row_sums4(const float (&v)[4], int li) {
  const bool b3 = (li & 8) != 0, b2 = (li & 4) != 0;
  const float r0 = __shfl_xor_sync(0xffffffffu, b3 ? v[0] : v[2], 8);
  const float r1 = __shfl_xor_sync(0xffffffffu, b3 ? v[1] : v[3], 8);
  const float a0 = (b3 ? v[2] : v[0]) + r0;  // row 2*b3
  const float a1 = (b3 ? v[3] : v[1]) + r1;  // row 2*b3 + 1
  const float r = __shfl_xor_sync(0xffffffffu, b2 ? a0 : a1, 4);
  float c = (b2 ? a1 : a0) + r;  // row 2*b3 + b2
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}
// max(m, |lo|, |hi|) of the two bf16 values of a word (lo in the low half), NaNs skipped.
__device__ __forceinline__ float max_abs_bf16x2(float m, uint32_t w) {
  m = fmaxf(m, fabsf(__uint_as_float(w << 16)));
  return fmaxf(m, fabsf(__uint_as_float(w & 0xffff0000u)));
}

__global__ void __launch_bounds__(kNbThreads, 1)
    norms_bulk_kernel(View q, View k, View v, int64_t nqb, int64_t nkb, int centering, float alpha,
                      const float *kbar, float *qmax_sq, float *qkbar, float *qsq, float *kblk, float *vblk,
                      int n_sink, SinkCand *cand, float *vmax_all, unsigned int *err, unsigned long long timeout_ns) {
  pdl_wait();  // inputs written by the kernels before this one
  pdl_trigger();
  extern __shared__ uint8_t nb_raw[];
  const uint32_t raw = nb_smem(nb_raw);
  const uint32_t base = (raw + 127u) & ~127u;
  uint8_t *g = nb_raw + (base - raw);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(g + kNbOffAbort);
  int *cta_vmax = reinterpret_cast<int *>(g + kNbOffAbort + 4);              // this CTA's V max (fp32 bits)
  unsigned int *warps_done = reinterpret_cast<unsigned int *>(g + kNbOffAbort + 8);
  int *smax = reinterpret_cast<int *>(g + kNbOffMax);
  unsigned int *scnt = reinterpret_cast<unsigned int *>(g + kNbOffCnt);
  float *knorm = reinterpret_cast<float *>(g + kNbOffKnorm);
  auto full = [&](int s) -> uint32_t { return base + (uint32_t)(kNbOffBar + 8 * s); };
  auto empty = [&](int s) -> uint32_t { return base + (uint32_t)(kNbOffBar + 8 * (kNbStages + s)); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t BH = q.B * q.H;
  const int64_t nQ = BH * nqb, nK = BH * nkb, n_items = nQ + 2 * nK;
  // This CTA's blocks: an even share of each kind (a contiguous run of the Q-blocks, of the
  // K-blocks and of the V-blocks), since the kinds cost different arithmetic per byte.  Items are
  // numbered Q-blocks, then K-blocks, then V-blocks; seg_range gives run `seg` as [a, e).
  const int64_t G = gridDim.x, c = blockIdx.x;
  // Where a CTA's share is a few blocks of each kind (fewer than 16 K-blocks), the block left
  // over per kind would land on the same CTAs three times (up to 15 % more bytes for them at
  // 4,096 keys): there the first n mod G CTAs of a rotated order take one block more, and the
  // rotations put those CTAs of the three kinds next to one another (Q's at CTAs [0, rQ), K's at
  // [rQ, rQ + rK), V's after, wrapping round G): the H40 S4096 pass 45.7 -> 42.7 us.  Larger
  // shares keep the plain even cut (the rotated one measured 1 % slower at Wan).
  const int64_t rQ = nQ % G, rK = nK % G;
  const bool rotate = nK < 16 * G;
  auto seg_range = [&](int seg, int64_t &a, int64_t &e) {
    const int64_t n = seg == 0 ? nQ : nK, off = seg == 0 ? 0 : (seg == 1 ? nQ : nQ + nK);
    if (!rotate) {
      a = off + c * n / G;
      e = off + (c + 1) * n / G;
      return;
    }
    const int64_t first = seg == 0 ? 0 : (seg == 1 ? rQ : rQ + rK);  // CTA of the rotated slot 0
    const int64_t cc = ((c - first) % G + G) % G;                     // this CTA's rotated slot
    const int64_t qn = n / G, r = n % G;
    a = off + cc * qn + (cc < r ? cc : r);
    e = a + qn + (cc < r ? 1 : 0);
  };
  // The runs in the order Q, K, V; with centering K, Q, V: the key sums have just read K, so at
  // sizes where K fits in L2 the K-blocks come from there (the 4,096-key pass 57.0 -> 54.9 us;
  // without centering K first was slower, 44.7 -> 47.7 us).
  auto seg_order = [centering](int si) -> int { return (centering && si < 2) ? 1 - si : si; };
  // The run's items in order: kind (0 Q, 1 K, 2 V), batch, head, block.  One division finds the
  // first; every next one is a step of the cursor (a division per item would cost about as many
  // instructions as a Q-block's arithmetic).
  struct Cursor {
    int kind;
    int64_t b, h, blk;
  };
  auto first_cursor = [&](int64_t i) -> Cursor {
    Cursor c{3, 0, 0, 0};
    if (i >= n_items) return c;  // an empty run (and no division by an empty kind's count)
    int64_t j = i, nb = nqb;
    c.kind = 0;
    if (i >= nQ) {
      c.kind = i < nQ + nK ? 1 : 2;
      j = i < nQ + nK ? i - nQ : i - nQ - nK;
      nb = nkb;
    }
    const int64_t bh = j / nb;
    c.blk = j - bh * nb;
    c.b = bh / q.H;
    c.h = bh - c.b * q.H;
    return c;
  };
  auto step = [&](Cursor &c) {
    if (++c.blk < (c.kind == 0 ? nqb : nkb)) return;
    c.blk = 0;
    if (++c.h < q.H) return;
    c.h = 0;
    if (++c.b < q.B) return;
    c.b = 0;
    ++c.kind;
  };
  // rows [r0, r1) of the cursor's block
  auto rows_of = [&](const Cursor &c, int64_t &r0, int64_t &r1) {
    if (c.kind == 0) {
      r0 = c.blk * kQRows;
      r1 = min(q.S, r0 + kQRows);
    } else {
      r0 = c.blk * kKVRows;
      r1 = min(k.S, r0 + kKVRows);
    }
  };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *cta_vmax = 0;
    *warps_done = 0;
    for (int s = 0; s < kNbStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(full(s)), "r"(1) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empty(s)), "r"(kNbWarps) : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (threadIdx.x < kNbSlots) {
    smax[threadIdx.x] = 0;  // +0.0f: maxima of non-negative quantities start at 0
    scnt[threadIdx.x] = 0;
  }
  __syncthreads();

  if (warp == kNbWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int last[kNbStages];  // phase of the last copy issued into each stage, -1: none
      for (int s = 0; s < kNbStages; ++s) last[s] = -1;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int si = 0; si < 3 && ok; ++si) {
        const int seg = seg_order(si);
        int64_t i_begin, i_end;
        seg_range(seg, i_begin, i_end);
        Cursor cur = first_cursor(i_begin);
        for (int64_t i = i_begin; i < i_end && ok; ++i, step(cur)) {
          const int kind = cur.kind;
          int64_t r0, r1;
          rows_of(cur, r0, r1);
          // the fields of q, k or v picked one by one (a reference to one of the three would put
          // the kernel parameters on the stack)
          const void *ptr = kind == 0 ? q.ptr : (kind == 1 ? k.ptr : v.ptr);
          const int64_t sB = kind == 0 ? q.sB : (kind == 1 ? k.sB : v.sB);
          const int64_t sH = kind == 0 ? q.sH : (kind == 1 ? k.sH : v.sH);
          const int64_t sS = kind == 0 ? q.sS : (kind == 1 ? k.sS : v.sS);
          const char *src = reinterpret_cast<const char *>(ptr) +
                            (cur.b * sB + cur.h * sH + r0 * sS) * (int64_t)sizeof(__nv_bfloat16);
          for (int64_t r = r0; r < r1; r += kNbTileRows) {
            ok = nb_wait(empty(s), ph ^ 1u, abort_flag, timeout_ns, err, (uint32_t)(kNbStages + s) << 16);
            if (!ok) break;
            const uint32_t bytes = (uint32_t)min((int64_t)kNbTileRows, r1 - r) * kNbRowBytes;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full(s)), "r"(bytes)
                         : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    base + (uint32_t)(s * kNbTileBytes)),
                "l"(src + (r - r0) * kNbRowBytes), "r"(bytes), "r"(full(s))
                : "memory");
            last[s] = (int)ph;
            if (++s == kNbStages) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // let every copy already issued land before the CTA can exit
        for (int st = 0; st < kNbStages; ++st)
          if (last[st] >= 0) nb_wait(full(st), (uint32_t)last[st], nullptr, timeout_ns, err, (uint32_t)st << 16);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int sub = lane >> 4, li = lane & 15;  // row of the pair, 8 elements of it
  const int my_u = li >> 2;                   // the pair whose reduced sums this lane ends with
  const bool writer = (li & 3) == 0;          // one lane per row writes the row's outputs
  int s = 0;
  uint32_t ph = 0;
  int64_t kb_head = -1;
  float kb[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) kb[e] = 0.f;
  int n_done = 0;  // items of this CTA so far: the slot of an item is n_done % kNbSlots
  for (int si = 0; si < 3; ++si) {
    const int seg = seg_order(si);
    int64_t i_begin, i_end;
    seg_range(seg, i_begin, i_end);
    Cursor cur = first_cursor(i_begin);
    for (int64_t i = i_begin; i < i_end; ++i, step(cur), ++n_done) {
      const int kind = cur.kind;
      const int64_t bh = cur.b * q.H + cur.h, blk = cur.blk;
      int64_t r0, r1;
      rows_of(cur, r0, r1);
      const int slot = n_done & (kNbSlots - 1);
      if (centering && kind < 2 && bh != kb_head) {
        kb_head = bh;
#pragma unroll
        for (int e = 0; e < 8; ++e) kb[e] = kbar[bh * 128 + li * 8 + e];
      }
      float bm = 0.f;    // Q, K: the largest row sum of this warp's rows
      float vm = 0.f;    // V: the largest |v|
      for (int64_t r = r0; r < r1; r += kNbTileRows) {
        bool ok = nb_wait(full(s), ph, abort_flag, timeout_ns, err, (uint32_t)s << 16);
        if (!__all_sync(0xffffffffu, ok)) return;  // every role stops: the error word says why
        const uint8_t *rows = g + s * kNbTileBytes + (warp * kNbRowsPerWarp + sub) * kNbRowBytes + li * 16;
        uint4 w[kNbGroups][4];
#pragma unroll
        for (int gi = 0; gi < kNbGroups; ++gi)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            w[gi][u] = *reinterpret_cast<const uint4 *>(rows + (gi * 8 + u * 2) * kNbRowBytes);
        // the rows are in registers: the stage may be refilled
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty(s)) : "memory");
        if (++s == kNbStages) {
          s = 0;
          ph ^= 1u;
        }
#pragma unroll
        for (int gi = 0; gi < kNbGroups; ++gi) {
          // this lane's row of pair u in group gi is row0 + 2u
          const int64_t row0 = r + warp * kNbRowsPerWarp + gi * 8 + sub;
          if (kind == 2) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (row0 + 2 * u < r1) {  // rows past a ragged end hold stale bytes
                vm = max_abs_bf16x2(vm, w[gi][u].x);
                vm = max_abs_bf16x2(vm, w[gi][u].y);
                vm = max_abs_bf16x2(vm, w[gi][u].z);
                vm = max_abs_bf16x2(vm, w[gi][u].w);
              }
            }
            continue;
          }
          const int64_t row = row0 + 2 * my_u;  // the row whose sums this lane ends with
          const bool valid = row < r1;
          float ss[4];
          if (kind == 0) {
            float dk[4];  // |q|^2 and q.kbar
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              float x[8];
              unpack16<__nv_bfloat16, 8>(w[gi][u], x);
              lane_sums<8, false, true>(x, kb, ss[u], dk[u]);
            }
            const float rs = row_sums4(ss, li), rd = row_sums4(dk, li);
            if (valid) {
              bm = fmaxf(bm, rs);
              if (writer) {
                qkbar[bh * q.S + row] = alpha * rd;
                qsq[bh * q.S + row] = rs;  // per-row |q|^2, turned into the row's shift by shift_kernel
              }
            }
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {  // |k - kbar|^2
              float x[8], unused;
              unpack16<__nv_bfloat16, 8>(w[gi][u], x);
              lane_sums<8, true, false>(x, kb, ss[u], unused);
            }
            const float rs = row_sums4(ss, li);
            if (valid) {
              bm = fmaxf(bm, rs);
              if (n_sink > 0 && writer) knorm[slot * kKVRows + (row - r0)] = rs;
            }
          }
        }
      }
      if (kind == 2) {
        bm = warp_max(vm * vm);
      } else {  // the four lanes of a quad end with the same row's sums: three levels suffice
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
      }
      // the block's maximum over the warps; the last warp to finish the block writes the results
      unsigned int last = 0;
      if (lane == 0) {
        atomicMax(&smax[slot], __float_as_int(bm));  // non-negative floats order as their bits
        __threadfence_block();
        last = atomicAdd(&scnt[slot], 1u) == (unsigned)(kNbWarps - 1);
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) continue;
      __threadfence_block();
      const float mx = __int_as_float(*reinterpret_cast<volatile int *>(&smax[slot]));
      if (lane == 0) {
        if (kind == 0) qmax_sq[bh * nqb + blk] = mx;
        else if (kind == 1) kblk[bh * nkb + blk] = mx;
        else {
          vblk[bh * nkb + blk] = mx;
          atomicMax(cta_vmax, __float_as_int(mx));  // v^2 >= 0: bits order as values
        }
      }
      if (n_sink > 0 && kind == 1) {
        // the block's n_sink + 1 loudest keys, in sink order
        const volatile float *kn = knorm + slot * kKVRows;
        const int cnt = (int)(r1 - r0);
        SinkCand *out = cand + (bh * nkb + blk) * kCandPerBlock;
        float pv = INFINITY;
        int32_t pi = -1;
        for (int tt = 0; tt <= n_sink; ++tt) {
          float bv = -1.f;
          int32_t bi = INT_MAX;
          for (int e = lane; e < cnt; e += 32) {
            const float vv = kn[e];
            const int32_t ix = (int32_t)(r0 + e);
            if (sink_after(vv, ix, pv, pi) && sink_before(vv, ix, bv, bi)) {
              bv = vv;
              bi = ix;
            }
          }
          warp_best_sink(bv, bi);
          if (lane == 0) out[tt] = SinkCand{bv, bi};
          pv = bv;
          pi = bi;
        }
      }
      __syncwarp();
      if (lane == 0) {
        smax[slot] = 0;
        scnt[slot] = 0;
      }
    }
  }
  // the global V max, folded in once per CTA by the last consumer warp to finish its items
  if (vmax_all && lane == 0) {
    __threadfence_block();
    if (atomicAdd(warps_done, 1u) == (unsigned)(kNbWarps - 1)) {
      __threadfence_block();
      atomicMax(reinterpret_cast<int *>(vmax_all), *reinterpret_cast<volatile int *>(cta_vmax));
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

// 4. Per block of kFinishRows query rows of one head: the head's key max (over its K blocks, or
// the key-sink pass's value), the global V max (folded in by the norms pass), then U, m and flag
// of the block's Q-blocks and every row's shift b_i = m_i + alpha*q_i.kbar (m_i per row or per
// Q-block), in one launch.  Every CTA of a head reduces the head's K-block maxima itself (nkb
// floats), so a CTA takes enough rows (8 a thread, their loads issued before that reduction) for
// the reduction's latency to be paid rarely; the first CTA of a head writes kmax_sq, the first
// CTA of all copies the V max out of the workspace into vmax_sq.
// `shift` holds |q_i|^2 on entry (from the norms pass).  Without centering the first CTA of a
// head also writes the head's key mean as zeros (kbar_zero; no memset of its own).
constexpr int kFinishRowsPerThread = 8;
constexpr int kFinishRows = kThreads * kFinishRowsPerThread;  // 2048 rows, 16 Q-blocks
constexpr int kFinishBlocks = kFinishRows / kQRows;
static_assert(kFinishRows % kQRows == 0 && kFinishBlocks <= kThreads, "whole Q-blocks per CTA");
__global__ void __launch_bounds__(kThreads)
    finish_shift_kernel(int64_t H, int64_t Sq, int64_t nqb, int64_t nkb, const float *kblk, const float *vmax_all,
                        double alpha, int C, int gate, int per_row, const float *qmax_sq, float *kmax_sq,
                        float *vmax_sq, int32_t *m, uint8_t *flag, const float *qkbar, float *shift,
                        int kmax_given, float *kbar_zero, int D) {
  pdl_wait();  // inputs written by the kernels before this one
  pdl_trigger();
  const int64_t bh = blockIdx.z * H + blockIdx.y;
  if (kbar_zero && blockIdx.x == 0 && threadIdx.x < D) kbar_zero[bh * D + threadIdx.x] = 0.f;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ float red[kWarps];
  __shared__ int32_t mblk[kFinishBlocks];
  // rows r0 + threadIdx.x + u * kThreads: coalesced, all loads of the thread in flight together,
  // and in flight while the key max is reduced
  const int64_t r0 = (int64_t)blockIdx.x * kFinishRows;
  float qk[kFinishRowsPerThread], qs[kFinishRowsPerThread];
#pragma unroll
  for (int u = 0; u < kFinishRowsPerThread; ++u) {
    const int64_t r = r0 + threadIdx.x + (int64_t)u * kThreads;
    qk[u] = r < Sq ? qkbar[bh * Sq + r] : 0.f;
    qs[u] = (per_row && r < Sq) ? shift[bh * Sq + r] : 0.f;
  }
  float km;
  if (kmax_given) {
    km = kmax_sq[bh];  // the key sinks' pass left the max over the other keys
  } else {
    float x = 0.f;
    for (int64_t i = threadIdx.x; i < nkb; i += kThreads) x = fmaxf(x, kblk[bh * nkb + i]);
    x = warp_max(x);
    if (lane == 0) red[warp] = x;
    __syncthreads();
    km = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) km = fmaxf(km, red[w]);
    if (blockIdx.x == 0 && threadIdx.x == 0) kmax_sq[bh] = km;
  }
  const float vm = *vmax_all;
  if (bh == 0 && blockIdx.x == 0 && threadIdx.x == 0) vmax_sq[0] = vm;
  const bool v_ok = vm <= (float)FM_VMAX * (float)FM_VMAX;
  const double ksq = sqrt((double)km);
  if (threadIdx.x < kFinishBlocks) {
    const int64_t qb = r0 / kQRows + threadIdx.x;
    if (qb < nqb) {
      const double U = alpha * sqrt((double)qmax_sq[bh * nqb + qb]) * ksq;
      const int32_t mv = (int32_t)ceil(U) - C;
      m[bh * nqb + qb] = mv;
      flag[bh * nqb + qb] = (uint8_t)(v_ok && U <= (double)gate);
      mblk[threadIdx.x] = mv;
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kFinishRowsPerThread; ++u) {
    const int64_t r = r0 + threadIdx.x + (int64_t)u * kThreads;
    if (r >= Sq) break;
    int32_t mi;
    if (per_row) {
      const double U = alpha * sqrt((double)qs[u]) * ksq;
      mi = (int32_t)ceil(U) - C;
    } else {
      mi = mblk[(threadIdx.x + u * kThreads) / kQRows];
    }
    shift[bh * Sq + r] = (float)mi + qk[u];
  }
}

// Row shifts alone, for the bounds of a ring (after ring_combine_kernel has written m and flag):
// b_i = m_i + alpha*q_i.kbar, with m_i = ceil(alpha*|q_i|*sqrt(kmax)) - C
// (per row) or the row's Q-block m.  `shift` holds |q_i|^2 on entry (from the norms pass).
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

// count == nullptr: partial sums only; else also the key mean (count zeroed beforehand).
template <typename T, int EPL, bool CONTIG>
cudaError_t launch_ksum(const View &k, int64_t P, float *part, unsigned int *count, int64_t N, float *kbar,
                        cudaStream_t st) {
  const dim3 grid((unsigned)P, (unsigned)k.H, (unsigned)k.B);
  if (CONTIG && rows16(k))
    return launch_pdl(ksum_vec_kernel<T, 32 * EPL>, grid, dim3(kThreads), 0, st, k, P, part, count, N, kbar);
  return launch_pdl(ksum_kernel<T, EPL, CONTIG>, grid, dim3(kThreads), 0, st, k, P, part, count, N, kbar);
}

// bf16 rows of D = 128 stored back to back within each head (the staged norms pass).
bool bulk_rows(const View &t) { return t.dtype == FM_BF16 && t.D == 128 && t.sS == t.D && rows16(t); }

cudaError_t launch_norms_bulk(const BoundsArgs &a, const WsLayout &w, float *kblk, float *vblk, SinkCand *cand,
                              float *vmax_all, cudaStream_t st) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(norms_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kNbSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int64_t n_items = a.q.B * a.q.H * (a.nqb + 2 * w.nkb);
  const int64_t grid = min(n_items, (int64_t)current_device_sm_count());
  return launch_pdl(norms_bulk_kernel, dim3((unsigned)grid), dim3(kNbThreads), (size_t)kNbSmem, st, a.q, a.k, a.v,
                    a.nqb, w.nkb, a.centering, (float)a.alpha, a.kbar, a.qmax_sq, a.qkbar, a.shift, kblk, vblk,
                    a.n_sink, cand, vmax_all, a.err, a.timeout_ns);
}

template <typename T, int EPL, bool CONTIG>
cudaError_t launch_norms(const BoundsArgs &a, const WsLayout &w, float *kblk, float *vblk, SinkCand *cand,
                         float *vmax_all, cudaStream_t st) {
  const int64_t nx = a.nqb + 2 * w.nkb;
  if (nx == 0) return cudaSuccess;
  if (CONTIG && sizeof(T) == 2 && EPL == 4 && bulk_rows(a.q) && bulk_rows(a.k) && bulk_rows(a.v))
    return launch_norms_bulk(a, w, kblk, vblk, cand, vmax_all, st);
  const dim3 grid((unsigned)nx, (unsigned)a.q.H, (unsigned)a.q.B);
  if (CONTIG && rows16(a.q) && rows16(a.k) && rows16(a.v)) {
    const int64_t nx4 = ceil_div(a.nqb, kBlocksPerCta) + 2 * ceil_div(w.nkb, kBlocksPerCta);
    return launch_pdl(norms_vec_kernel<T, 32 * EPL>, dim3((unsigned)nx4, (unsigned)a.q.H, (unsigned)a.q.B),
                      dim3(kThreads), 0, st, a.q, a.k, a.v, a.nqb, w.nkb, a.centering, (float)a.alpha, a.kbar,
                      a.qmax_sq, a.qkbar, a.shift, kblk, vblk, a.n_sink, cand, vmax_all);
  }
  return launch_pdl(norms_kernel<T, EPL, CONTIG>, grid, dim3(kThreads), 0, st, a.q, a.k, a.v, a.nqb, w.nkb,
                    a.centering, (float)a.alpha, a.kbar, a.qmax_sq, a.qkbar, a.shift, kblk, vblk, a.n_sink, cand,
                    vmax_all);
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
  e = launch_norms<T, EPL, CONTIG>(a, w, kblk, vblk, cand, nullptr, st);
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
  const dim3 heads((unsigned)H, (unsigned)B);
  // the global V max (every CTA of the norms pass folds its V max in with an integer atomicMax)
  // and the key sums' arrival counters start at zero
  float *vmax_ws = reinterpret_cast<float *>(ws + w.off_zero);
  unsigned int *count = reinterpret_cast<unsigned int *>(ws + w.off_zero + 16);
  cudaError_t e = cudaMemsetAsync(ws + w.off_zero, 0, w.zero_bytes, st);
  if (e != cudaSuccess) return e;
  // without centering no kernel reads the key mean: the finish writes it as zeros
  const bool kbar_by_finish = !a.centering && a.q.D <= kThreads;
  if (a.centering && N > 0) {
    e = launch_ksum<T, EPL, CONTIG>(a.k, w.P, part, count, N, a.kbar, st);
  } else if (!kbar_by_finish) {
    e = cudaMemsetAsync(a.kbar, 0, sizeof(float) * (size_t)(B * H * a.q.D), st);
  }
  if (e != cudaSuccess) return e;
  e = launch_norms<T, EPL, CONTIG>(a, w, kblk, vblk, cand, vmax_ws, st);
  if (e != cudaSuccess) return e;
  if (a.n_sink > 0) {
    e = launch_pdl(sink_select_kernel<T>, heads, dim3(kThreads), 0, st, a.k, a.v, w.nkb, a.n_sink, cand, a.sink_idx,
                   a.sink_k, a.sink_v, a.kmax_sq);
    if (e != cudaSuccess) return e;
  }
  // one CTA per kFinishRows query rows of each head (at least one per head, which writes kmax_sq)
  const int64_t nx = ceil_div(a.q.S, kFinishRows) > 0 ? ceil_div(a.q.S, kFinishRows) : 1;
  e = launch_pdl(finish_shift_kernel, dim3((unsigned)nx, (unsigned)H, (unsigned)B), dim3(kThreads), 0, st, H, a.q.S,
                 a.nqb, w.nkb, kblk, vmax_ws, a.alpha, a.C, a.gate, a.per_row, a.qmax_sq, a.kmax_sq, a.vmax_sq, a.m,
                 a.flag, a.qkbar, a.shift, (int)(a.n_sink > 0), kbar_by_finish ? a.kbar : nullptr,
                 (int)a.q.D);
  if (e != cudaSuccess) return e;
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
#define FM_KSUM(T, E, C) launch_ksum<T, E, C>(k, w.P, part, nullptr, 0, nullptr, st)
    e = D == 128 ? (contig ? FM_KSUM(__nv_bfloat16, 4, true) : FM_KSUM(__nv_bfloat16, 4, false))
                 : (contig ? FM_KSUM(__nv_bfloat16, 2, true) : FM_KSUM(__nv_bfloat16, 2, false));
  else
    e = D == 128 ? (contig ? FM_KSUM(float, 4, true) : FM_KSUM(float, 4, false))
                 : (contig ? FM_KSUM(float, 2, true) : FM_KSUM(float, 2, false));
#undef FM_KSUM
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
