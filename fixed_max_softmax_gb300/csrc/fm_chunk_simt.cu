// fm_chunk_simt.cu -- CUDA-core (FFMA) chunk kernel.
//
// Serves the cases the tensor-core kernel does not: fp32 inputs (the product is exact
// fp32 arithmetic, so no TF32 or bf16 rounding of the operands), D = 64, strides that
// TMA cannot describe, and empty chunks.  Same semantics as the tensor-core kernel:
//   eligible Q-block  (flag = 1, not forced online): pure-add fixed-m accumulation,
//       p_ij = 2^(alpha*s_ij - b_i), b_i = the row's shift from fm_bounds (m + alpha*q_i.kbar)
//       ("Kernel reference: ring_attention_const_max_fwd", sections "A static bound makes
//       the ring reduction pure addition" and "Accumulate, then normalize once";
//       PR #477 Summary for m and the exp2 form; "Virtual K-centering" for the centering term)
//   other Q-blocks: online softmax with a running row max r_i kept in acc_max and
//       rescaling of the partial sums when it grows (PR #478 "Cross-Ring Safety
//       Fallback": standard online-softmax accumulation across the chunks).
// One CTA = 64 query rows of one (batch, head); each row is split over D/32 threads that
// each own 32 dimensions of q and of the output; 32-key tiles of K and V are staged in
// shared memory as fp32.  Key sinks (the loudest keys the bounds pass set aside, "Kernel
// reference: ring_attention_const_max_fwd", section "Adapting this kernel") add nothing
// here: a per-tile bit mask drops them along with the keys past the chunk's end.
#include <cuda_bf16.h>
#include <math.h>

#include "fm_internal.h"

namespace fm {
namespace {

constexpr int kRows = 64;  // query rows per CTA
constexpr int kKeys = 32;  // keys per shared-memory tile
constexpr int kDimsPerThread = 32;

template <typename T>
__device__ __forceinline__ float ld_elem(const T *p) {
  if constexpr (sizeof(T) == 2) return __bfloat162float(*p); else return (float)*p;
}

template <typename T, int D>
__global__ void __launch_bounds__(kRows *(D / kDimsPerThread))
    chunk_simt_kernel(const ChunkArgs a) {
  pdl_wait();  // bounds and accumulators written by the kernels before this one
  pdl_trigger();
  constexpr int TPR = D / kDimsPerThread;  // threads per row (2 or 4)
  constexpr int NT = kRows * TPR;
  __shared__ float Ks[kKeys][D];
  __shared__ float Vs[kKeys][D];
  __shared__ unsigned keep_bits;  // bit j: key j of the tile counts (in range, not a sink)

  const int tid = threadIdx.x;
  const int lr = tid / TPR;  // local row
  const int part = tid % TPR;
  const int64_t b = blockIdx.z, h = blockIdx.y;
  const int64_t bh = b * a.q.H + h;
  const int64_t row = (int64_t)blockIdx.x * kRows + lr;
  const bool row_ok = row < a.q.S;
  const int64_t qb = (int64_t)blockIdx.x * kRows / FM_BLOCK_Q;  // the CTA lies in one Q-block
  const bool fixed = !a.force_online && a.flag[bh * a.nqb + qb] != 0;
  const float bias = (fixed && row_ok) ? a.shift[bh * a.q.S + row] : 0.f;

  float qv[kDimsPerThread], ov[kDimsPerThread];
  const T *qp = reinterpret_cast<const T *>(a.q.ptr) + b * a.q.sB + h * a.q.sH + (row_ok ? row : 0) * a.q.sS;
#pragma unroll
  for (int d = 0; d < kDimsPerThread; ++d) {
    qv[d] = row_ok ? ld_elem(qp + (int64_t)(part * kDimsPerThread + d) * a.q.sD) : 0.f;
    ov[d] = 0.f;
  }
  float l = 0.f;
  float run = -INFINITY;  // online: running max of z = alpha*s

  const T *kp = reinterpret_cast<const T *>(a.k.ptr) + b * a.k.sB + h * a.k.sH;
  const T *vp = reinterpret_cast<const T *>(a.v.ptr) + b * a.v.sB + h * a.v.sH;
  const int64_t Nc = a.k.S;
  for (int64_t j0 = 0; j0 < Nc; j0 += kKeys) {
    const int nvalid = (int)min((int64_t)kKeys, Nc - j0);
    __syncthreads();
    for (int i = tid; i < kKeys * D; i += NT) {
      const int j = i / D, d = i % D;
      float kx = 0.f, vx = 0.f;
      if (j < nvalid) {
        kx = ld_elem(kp + (j0 + j) * a.k.sS + (int64_t)d * a.k.sD);
        vx = ld_elem(vp + (j0 + j) * a.v.sS + (int64_t)d * a.v.sD);
      }
      Ks[j][d] = kx;
      Vs[j][d] = vx;
    }
    if (tid == 0) {
      unsigned kb = nvalid >= kKeys ? 0xffffffffu : ((1u << nvalid) - 1u);
      if (a.sinks) {
        const int64_t g0 = a.key0 + j0;
        const int32_t *sk = a.sinks + bh * FM_MAX_SINKS;
        for (int t = 0; t < FM_MAX_SINKS; ++t) {
          const int64_t g = sk[t];
          if (g >= g0 && g < g0 + nvalid) kb &= ~(1u << (int)(g - g0));
        }
      }
      keep_bits = kb;
    }
    __syncthreads();
    const unsigned keep = keep_bits;
    float s[kKeys];
#pragma unroll
    for (int j = 0; j < kKeys; ++j) {
      float acc = 0.f;
#pragma unroll
      for (int d = 0; d < kDimsPerThread; ++d) acc = fmaf(qv[d], Ks[j][part * kDimsPerThread + d], acc);
#pragma unroll
      for (int o = 1; o < TPR; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      s[j] = acc;
    }
    float shift = bias;
    if (!fixed) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kKeys; ++j)
        if ((keep >> j) & 1u) mx = fmaxf(mx, s[j] * a.alpha);
      if (mx > run) {
        const float sc = exp2f(run - mx);  // 0 when run = -inf
        l *= sc;
#pragma unroll
        for (int d = 0; d < kDimsPerThread; ++d) ov[d] *= sc;
        run = mx;
      }
      shift = run;
    }
#pragma unroll
    for (int j = 0; j < kKeys; ++j) {
      const float p = ((keep >> j) & 1u) ? exp2f(fmaf(s[j], a.alpha, -shift)) : 0.f;
      l += p;
#pragma unroll
      for (int d = 0; d < kDimsPerThread; ++d) ov[d] = fmaf(p, Vs[j][part * kDimsPerThread + d], ov[d]);
    }
  }

  if (!row_ok) return;
  const int64_t r = bh * a.q.S + row;
  float *ao = a.acc_o + r * D + part * kDimsPerThread;
  if (fixed) {
    if (a.accumulate) {
#pragma unroll
      for (int d = 0; d < kDimsPerThread; ++d) ao[d] += ov[d];
    } else {
#pragma unroll
      for (int d = 0; d < kDimsPerThread; ++d) ao[d] = ov[d];
    }
    if (part == 0) {
      a.acc_sum[r] = a.accumulate ? a.acc_sum[r] + l : l;
      a.acc_max[r] = bias;
    }
    return;
  }
  // online merge with the previous chunks' state (acc_max = their running max)
  float cprev = 0.f, cnew = 1.f, nr = run;
  if (a.accumulate) {
    const float R = a.acc_max[r];
    nr = fmaxf(R, run);
    cprev = (R == -INFINITY) ? 0.f : exp2f(R - nr);
    cnew = (run == -INFINITY) ? 0.f : exp2f(run - nr);
  }
  if (a.accumulate) {
#pragma unroll
    for (int d = 0; d < kDimsPerThread; ++d) ao[d] = ao[d] * cprev + ov[d] * cnew;
  } else {
#pragma unroll
    for (int d = 0; d < kDimsPerThread; ++d) ao[d] = ov[d];
  }
  // the row's TPR threads (adjacent lanes of one warp) have all read acc_max before
  // it is overwritten; rows past Sq returned above as a whole, so the mask is exact
  const unsigned row_mask = ((1u << TPR) - 1u) << ((threadIdx.x & 31) / TPR * TPR);
  __syncwarp(row_mask);
  if (part == 0) {
    a.acc_sum[r] = a.accumulate ? a.acc_sum[r] * cprev + l * cnew : l;
    a.acc_max[r] = nr;
  }
}

template <typename T, int D>
cudaError_t launch_typed(const ChunkArgs &a, cudaStream_t st) {
  constexpr int TPR = D / kDimsPerThread;
  dim3 grid((unsigned)((a.q.S + kRows - 1) / kRows), (unsigned)a.q.H, (unsigned)a.q.B);
  if (grid.x == 0) return cudaSuccess;
  return launch_pdl(chunk_simt_kernel<T, D>, grid, dim3(kRows * TPR), 0, st, a);
}

}  // namespace

cudaError_t launch_chunk_simt(const ChunkArgs &a, cudaStream_t st) {
  if (a.q.dtype == FM_BF16)
    return a.q.D == 128 ? launch_typed<__nv_bfloat16, 128>(a, st) : launch_typed<__nv_bfloat16, 64>(a, st);
  return a.q.D == 128 ? launch_typed<float, 128>(a, st) : launch_typed<float, 64>(a, st);
}

cudaError_t launch_chunk_empty_init(const ChunkArgs &a, cudaStream_t st) {
  return launch_chunk_simt(a, st);
}

}  // namespace fm
