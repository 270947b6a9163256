// fm_finalize.cu -- the single normalising divide of fixed-m attention.
//
// o = acc_o / max(acc_sum, 1e-37): "Kernel reference: ring_attention_const_max_fwd",
// section "Accumulate, then normalize once" (one divide at the end; the row sum is
// floored near the smallest fp32 normal so an all-underflow row divides by the floor).
// HBM-bound elementwise pass: each thread handles four consecutive output elements of
// a row (one 16-byte load of acc_o), grid-stride over the whole tensor.
//
// Also here: the fold of the key sinks, the few loudest keys of a head that the bounds
// pass left out of the key max and the chunks left out of their sums ("Kernel reference:
// ring_attention_const_max_fwd", section "Adapting this kernel").  One online-softmax
// merge per row, in fp32, before the divide.
#include <cuda_bf16.h>
#include <limits.h>

#include "fm_internal.h"

namespace fm {
namespace {

template <bool BF16, bool VEC, bool LSE>
__global__ void __launch_bounds__(256) finalize_kernel(const float *__restrict__ acc_o,
                                                       const float *__restrict__ acc_sum,
                                                       const float *__restrict__ acc_max, float *__restrict__ lse,
                                                       View o, int64_t n_quads) {
  pdl_wait();  // the accumulators written by the kernels before this one
  pdl_trigger();
  const int64_t D = o.D;
  const int64_t qpr = D / 4;  // quads per row
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_quads;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / qpr;  // flat row index over [B, H, Sq]
    const int64_t d0 = (i - r * qpr) * 4;
    const int64_t s = r % o.S;
    const int64_t bh = r / o.S;
    const int64_t h = bh % o.H, b = bh / o.H;
    const float sum = acc_sum[r];
    const float inv = 1.0f / fmaxf(sum, FM_SUM_CLAMP);
    // natural-log LSE of the scaled scores: acc_sum * 2^acc_max = sum_j 2^(alpha*q.k_j)
    if constexpr (LSE) {
      if (d0 == 0) lse[r] = 0.69314718055994531f * (acc_max[r] + log2f(sum));
    }
    const float4 a = *reinterpret_cast<const float4 *>(acc_o + r * D + d0);
    const float x[4] = {a.x * inv, a.y * inv, a.z * inv, a.w * inv};
    const int64_t off = b * o.sB + h * o.sH + s * o.sS + d0 * o.sD;
    if constexpr (BF16) {
      __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(const_cast<void *>(o.ptr)) + off;
      if constexpr (VEC) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(x[0], x[1]);
        __nv_bfloat162 hi = __floats2bfloat162_rn(x[2], x[3]);
        uint2 u;
        u.x = *reinterpret_cast<unsigned *>(&lo);
        u.y = *reinterpret_cast<unsigned *>(&hi);
        *reinterpret_cast<uint2 *>(dst) = u;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e * o.sD] = __float2bfloat16_rn(x[e]);
      }
    } else {
      float *dst = reinterpret_cast<float *>(const_cast<void *>(o.ptr)) + off;
      if constexpr (VEC) {
        *reinterpret_cast<float4 *>(dst) = make_float4(x[0], x[1], x[2], x[3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e * o.sD] = x[e];
      }
    }
  }
}

constexpr int kFoldWarps = 8;
constexpr int kFoldRowsPerWarp = 8;
constexpr int kFoldRows = kFoldWarps * kFoldRowsPerWarp;  // rows per CTA

// One warp per row; lane owns EPL = D/32 consecutive dimensions.  The head's sinks (raw
// key and value rows) are staged in shared memory once per CTA.  FINAL: the normalise
// follows in the same pass (o = acc / max(sum, 1e-37), and lse when given) and acc_o is
// not written back; acc_sum and acc_max are updated either way.
struct FoldOut {
  View o;
  float *lse;
};
template <typename T, int EPL, bool FINAL>
__global__ void __launch_bounds__(kFoldWarps * 32)
    fold_sinks_kernel(View q, float alpha, const int32_t *__restrict__ sink_idx, const float *__restrict__ sink_k,
                      const float *__restrict__ sink_v, float *__restrict__ acc_o, float *__restrict__ acc_sum,
                      float *__restrict__ acc_max, FoldOut fo) {
  pdl_wait();  // the accumulators written by the kernels before this one
  pdl_trigger();
  constexpr int D = 32 * EPL;
  __shared__ float sk[FM_MAX_SINKS][D];
  __shared__ float sv[FM_MAX_SINKS][D];
  const int64_t b = blockIdx.z, h = blockIdx.y;
  const int64_t bh = b * q.H + h;
  int ns = 0;
  while (ns < FM_MAX_SINKS && sink_idx[bh * FM_MAX_SINKS + ns] != INT_MAX) ++ns;  // ascending, padded
  if (!FINAL && ns == 0) return;  // no sink in this head: nothing to merge
  for (int e = threadIdx.x; e < ns * D; e += blockDim.x) {
    sk[e / D][e % D] = sink_k[(bh * FM_MAX_SINKS) * D + e];
    sv[e / D][e % D] = sink_v[(bh * FM_MAX_SINKS) * D + e];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T *qb = reinterpret_cast<const T *>(q.ptr) + b * q.sB + h * q.sH;
  for (int k = 0; k < kFoldRowsPerWarp; ++k) {
    const int64_t row = (int64_t)blockIdx.x * kFoldRows + warp * kFoldRowsPerWarp + k;
    if (row >= q.S) break;
    float qx[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const T t = qb[row * q.sS + (int64_t)(lane * EPL + e) * q.sD];
      if constexpr (sizeof(T) == 2) qx[e] = __bfloat162float(t); else qx[e] = (float)t;
    }
    float z[FM_MAX_SINKS];
    const int64_t r = bh * q.S + row;
    const float r_old = acc_max[r];
    float r_new = r_old;
#pragma unroll
    for (int s = 0; s < FM_MAX_SINKS; ++s) {
      if (s < ns) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) dot = fmaf(qx[e], sk[s][lane * EPL + e], dot);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        z[s] = alpha * dot;  // raw base-2 logit, the units of acc_max
        r_new = fmaxf(r_new, z[s]);
      }
    }
    const float c = r_old == -INFINITY ? 0.f : exp2f(r_old - r_new);
    float4 *ao = reinterpret_cast<float4 *>(acc_o + r * D) + lane * EPL / 4;
    float o[EPL];
    if constexpr (EPL == 4) {
      const float4 a = *ao;
      o[0] = a.x * c; o[1] = a.y * c; o[2] = a.z * c; o[3] = a.w * c;
    } else {
      const float2 a = *reinterpret_cast<const float2 *>(acc_o + r * D + lane * EPL);
      o[0] = a.x * c; o[1] = a.y * c;
    }
    float psum = 0.f;
#pragma unroll
    for (int s = 0; s < FM_MAX_SINKS; ++s) {
      if (s < ns) {
        const float p = exp2f(z[s] - r_new);
        psum += p;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = fmaf(p, sv[s][lane * EPL + e], o[e]);
      }
    }
    const float sum_new = fmaf(acc_sum[r], c, psum);
    if constexpr (FINAL) {
      const float inv = 1.0f / fmaxf(sum_new, FM_SUM_CLAMP);
      const int64_t off = b * fo.o.sB + h * fo.o.sH + row * fo.o.sS;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const int64_t at = off + (int64_t)(lane * EPL + e) * fo.o.sD;
        if (fo.o.dtype == FM_BF16)
          reinterpret_cast<__nv_bfloat16 *>(const_cast<void *>(fo.o.ptr))[at] = __float2bfloat16_rn(o[e] * inv);
        else
          reinterpret_cast<float *>(const_cast<void *>(fo.o.ptr))[at] = o[e] * inv;
      }
      if (fo.lse && lane == 0) fo.lse[r] = 0.69314718055994531f * (r_new + log2f(sum_new));
    } else if constexpr (EPL == 4) {
      *ao = make_float4(o[0], o[1], o[2], o[3]);
    } else {
      *reinterpret_cast<float2 *>(acc_o + r * D + lane * EPL) = make_float2(o[0], o[1]);
    }
    __syncwarp();  // every lane has read acc_sum before lane 0 replaces it
    if (lane == 0) {
      acc_sum[r] = sum_new;
      acc_max[r] = r_new;
    }
  }
}

template <bool LSE>
cudaError_t launch_typed(const float *acc_o, const float *acc_sum, const float *acc_max, const View &o,
                         float *lse, cudaStream_t st) {
  const int64_t n_quads = o.B * o.H * o.S * (o.D / 4);
  if (n_quads == 0) return cudaSuccess;
  const size_t es = o.dtype == FM_F32 ? 4 : 2;
  const size_t vb = 4 * es;  // bytes of one vector store
  const bool vec = o.sD == 1 && reinterpret_cast<uintptr_t>(o.ptr) % vb == 0 &&
                   (o.sB * es) % vb == 0 && (o.sH * es) % vb == 0 && (o.sS * es) % vb == 0;
  const int sms = current_device_sm_count();
  int64_t blocks = (n_quads + 255) / 256;
  const int64_t cap = (int64_t)sms * 16;
  if (blocks > cap) blocks = cap;
  const dim3 grid((unsigned)blocks), threads(256);
  cudaError_t e;
  if (o.dtype == FM_BF16) {
    e = vec ? launch_pdl(finalize_kernel<true, true, LSE>, grid, threads, 0, st, acc_o, acc_sum, acc_max, lse, o, n_quads)
            : launch_pdl(finalize_kernel<true, false, LSE>, grid, threads, 0, st, acc_o, acc_sum, acc_max, lse, o,
                         n_quads);
  } else {
    e = vec ? launch_pdl(finalize_kernel<false, true, LSE>, grid, threads, 0, st, acc_o, acc_sum, acc_max, lse, o,
                         n_quads)
            : launch_pdl(finalize_kernel<false, false, LSE>, grid, threads, 0, st, acc_o, acc_sum, acc_max, lse, o,
                         n_quads);
  }
  return e;
}

}  // namespace

cudaError_t launch_finalize(const float *acc_o, const float *acc_sum, const View &o, cudaStream_t st) {
  return launch_typed<false>(acc_o, acc_sum, nullptr, o, nullptr, st);
}

cudaError_t launch_finalize_lse(const float *acc_o, const float *acc_sum, const float *acc_max, const View &o,
                                float *lse, cudaStream_t st) {
  return launch_typed<true>(acc_o, acc_sum, acc_max, o, lse, st);
}

template <bool FINAL>
cudaError_t launch_fold(const View &q, float alpha, const int32_t *sink_idx, const float *sink_k, const float *sink_v,
                        float *acc_o, float *acc_sum, float *acc_max, const FoldOut &fo, cudaStream_t st) {
  if (q.B * q.H * q.S == 0) return cudaSuccess;
  const dim3 grid((unsigned)((q.S + kFoldRows - 1) / kFoldRows), (unsigned)q.H, (unsigned)q.B);
  const dim3 threads(kFoldWarps * 32);
  if (q.dtype == FM_BF16)
    return q.D == 128 ? launch_pdl(fold_sinks_kernel<__nv_bfloat16, 4, FINAL>, grid, threads, 0, st, q, alpha, sink_idx,
                                   sink_k, sink_v, acc_o, acc_sum, acc_max, fo)
                      : launch_pdl(fold_sinks_kernel<__nv_bfloat16, 2, FINAL>, grid, threads, 0, st, q, alpha, sink_idx,
                                   sink_k, sink_v, acc_o, acc_sum, acc_max, fo);
  return q.D == 128 ? launch_pdl(fold_sinks_kernel<float, 4, FINAL>, grid, threads, 0, st, q, alpha, sink_idx, sink_k,
                                 sink_v, acc_o, acc_sum, acc_max, fo)
                    : launch_pdl(fold_sinks_kernel<float, 2, FINAL>, grid, threads, 0, st, q, alpha, sink_idx, sink_k,
                                 sink_v, acc_o, acc_sum, acc_max, fo);
}

cudaError_t launch_fold_sinks(const View &q, float alpha, const int32_t *sink_idx, const float *sink_k,
                              const float *sink_v, float *acc_o, float *acc_sum, float *acc_max, cudaStream_t st) {
  return launch_fold<false>(q, alpha, sink_idx, sink_k, sink_v, acc_o, acc_sum, acc_max, FoldOut{View{}, nullptr}, st);
}

cudaError_t launch_fold_sinks_final(const View &q, float alpha, const int32_t *sink_idx, const float *sink_k,
                                    const float *sink_v, float *acc_o, float *acc_sum, float *acc_max, const View &o,
                                    float *lse, cudaStream_t st) {
  return launch_fold<true>(q, alpha, sink_idx, sink_k, sink_v, acc_o, acc_sum, acc_max, FoldOut{o, lse}, st);
}

}  // namespace fm
