// fm_finalize.cu -- the single normalising divide of fixed-m attention.
//
// o = acc_o / max(acc_sum, 1e-37): "Kernel reference: ring_attention_const_max_fwd",
// section "Accumulate, then normalize once" (one divide at the end; the row sum is
// floored near the smallest fp32 normal so an all-underflow row divides by the floor).
// HBM-bound elementwise pass: each thread handles four consecutive output elements of
// a row (one 16-byte load of acc_o), grid-stride over the whole tensor.
#include <cuda_bf16.h>

#include "fm_internal.h"

namespace fm {
namespace {

template <bool BF16, bool VEC, bool LSE>
__global__ void __launch_bounds__(256) finalize_kernel(const float *__restrict__ acc_o,
                                                       const float *__restrict__ acc_sum,
                                                       const float *__restrict__ acc_max, float *__restrict__ lse,
                                                       View o, int64_t n_quads) {
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
  if (o.dtype == FM_BF16) {
    if (vec) finalize_kernel<true, true, LSE><<<(unsigned)blocks, 256, 0, st>>>(acc_o, acc_sum, acc_max, lse, o, n_quads);
    else finalize_kernel<true, false, LSE><<<(unsigned)blocks, 256, 0, st>>>(acc_o, acc_sum, acc_max, lse, o, n_quads);
  } else {
    if (vec) finalize_kernel<false, true, LSE><<<(unsigned)blocks, 256, 0, st>>>(acc_o, acc_sum, acc_max, lse, o, n_quads);
    else finalize_kernel<false, false, LSE><<<(unsigned)blocks, 256, 0, st>>>(acc_o, acc_sum, acc_max, lse, o, n_quads);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_finalize(const float *acc_o, const float *acc_sum, const View &o, cudaStream_t st) {
  return launch_typed<false>(acc_o, acc_sum, nullptr, o, nullptr, st);
}

cudaError_t launch_finalize_lse(const float *acc_o, const float *acc_sum, const float *acc_max, const View &o,
                                float *lse, cudaStream_t st) {
  return launch_typed<true>(acc_o, acc_sum, acc_max, o, lse, st);
}

}  // namespace fm
