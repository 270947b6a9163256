// fm_internal.h -- declarations shared by the CUDA translation units of libfm.
// Not part of the public ABI (include/fm.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/fm.h"

namespace fm {

// Device error codes written to the per-GPU error word.
enum : unsigned int {
  kDevErrNone = 0,
  kDevErrTimeoutProducer = 1,
  kDevErrTimeoutMma = 2,
  kDevErrTimeoutSoftmax = 3,
  kDevErrTimeoutDrain = 4,
  kDevErrTimeoutProbe = 5,
  kDevErrTimeoutBounds = 6,
  kDevErrDebugIndex = 7,  // debug builds: an index check failed (the access was skipped)
};

// Debug builds (nvcc -DFM_DEBUG): FM_DCHECK(ok, err, site, index) is false when `ok` is, and then
// records the first failure of the launch in the error word (code, site, the index, block and
// thread) for fm_sync_status to report as FM_ERR_INDEX; the caller skips the access.  Release
// builds: always true, nothing is checked.
#ifdef FM_DEBUG
#ifdef __CUDACC__
__device__ __forceinline__ bool fm_dcheck(bool ok, unsigned int *err, unsigned int site, long long index) {
  if (ok) return true;
  if (err && atomicCAS(err, 0u, (unsigned int)kDevErrDebugIndex) == 0u) {
    err[1] = site;
    err[2] = (unsigned int)((unsigned long long)index & 0xffffffffull);
    err[3] = (unsigned int)((unsigned long long)index >> 32);
    err[4] = blockIdx.x;
    err[5] = threadIdx.x;
  }
  return false;
}
#endif
#define FM_DCHECK(ok, err, site, index) fm_dcheck((ok), (err), (site), (long long)(index))
#else
#define FM_DCHECK(ok, err, site, index) true
#endif

// Default limit of a pipeline wait inside a kernel.  One CTA of the chunk kernel runs
// for well under 10 ms at the largest sizes, so a wait that lasts seconds means a
// broken pipeline; the kernel then records the failure and returns.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

// A validated view of an fm_tensor (element strides; D stride may be any value).
struct View {
  const void *ptr;
  int dtype;
  int64_t B, H, S, D;
  int64_t sB, sH, sS, sD;
};

// ---- bounds (fm_bounds.cu) -------------------------------------------------
struct BoundsArgs {
  View q, k, v;
  int centering;
  int per_row;    // one shift per query row instead of per Q-block
  double alpha;   // softmax_scale * log2(e), fp64 for the bound
  int C, gate;
  int64_t nqb;    // ceil(Sq / 128)
  int32_t *m;
  uint8_t *flag;
  float *qmax_sq, *kmax_sq, *kbar, *qkbar, *shift, *vmax_sq;
  // key sinks: n_sink > 0 leaves that many of each head's loudest keys out of the key max
  int n_sink = 0;
  int32_t *sink_idx = nullptr;  // [B,H,FM_MAX_SINKS] ascending global key index, INT32_MAX pads
  float *sink_k = nullptr;      // [B,H,FM_MAX_SINKS,D] raw key rows of the sinks
  float *sink_v = nullptr;      // [B,H,FM_MAX_SINKS,D] their value rows
  void *ws;
  size_t ws_bytes;
  unsigned int *err = nullptr;  // device error word (bounded waits of the staged norms pass)
  unsigned long long timeout_ns = kWaitTimeoutNs;
};
size_t bounds_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t D);
cudaError_t launch_bounds(const BoundsArgs &a, cudaStream_t st);
// The bounds of a ring of ranks (each holds one shard of the keys): the shard's key sums; one
// rank's statistics block; the combine of every rank's blocks into the bounds.
size_t ring_stats_bytes(int64_t B, int64_t H, int64_t D, int n_sink);
cudaError_t launch_ring_key_sums(const View &k, float *ksum, void *ws, cudaStream_t st);
cudaError_t launch_bounds_local(const BoundsArgs &a, const float *ksum_total, int64_t N_total, int64_t key_offset,
                                void *stats, cudaStream_t st);
cudaError_t launch_bounds_combine(const BoundsArgs &a, const void *stats_all, int n_ranks, cudaStream_t st);

// ---- chunk kernels ----------------------------------------------------------
struct ChunkArgs {
  View q, k, v;            // k, v: this chunk
  float alpha;
  int force_online;
  int schedule = FM_SCHEDULE_AUTO;  // fm_opts.schedule (tensor-core kernel)
  int accumulate;
  int64_t nqb;
  const uint8_t *flag;     // [B,H,nqb]
  const float *shift;      // [B,H,Sq] the fixed-m shift of each row
  float *acc_o, *acc_sum, *acc_max;
  unsigned int *err;       // device error word
  unsigned long long timeout_ns;
  // last chunk with the normalise fused in (tensor-core path only): o = acc / sum is
  // written to `out` (and lse, when given) instead of acc_o being written back
  const View *out = nullptr;
  float *lse = nullptr;
  // several consecutive chunks in one launch (tensor-core path): n_chunks > 0 selects
  // ks/vs instead of k/v
  int n_chunks = 0;
  const View *ks = nullptr, *vs = nullptr;
  // key sinks to skip: [B,H,FM_MAX_SINKS] ascending global key indices (INT32_MAX pads),
  // or nullptr; key0 is the global index of the first chunk's first key
  const int32_t *sinks = nullptr;
  int64_t key0 = 0;
};
// SIMT path: fp32 inputs (exact fp32 arithmetic), any D in {64,128}, any strides.
cudaError_t launch_chunk_simt(const ChunkArgs &a, cudaStream_t st);
// tcgen05/TMEM/TMA path: bf16, D = 128, unit D stride, 16-byte aligned rows.  Returns
// cudaErrorNotSupported, launching nothing, when the tensor maps cannot be encoded.
bool chunk_tc_supported(const ChunkArgs &a);
cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t st);
// Can the tensor-core kernel write `o` itself (unit D stride, 16-byte aligned rows)?
bool chunk_tc_final_supported(const ChunkArgs &a, const View &o);
// One bounded wait that can never complete (the failure-detection probe).
cudaError_t launch_wait_probe(unsigned int *err, unsigned long long timeout_ns, cudaStream_t st);
// Empty chunk (Nc == 0) with accumulate == 0: write the empty state.
cudaError_t launch_chunk_empty_init(const ChunkArgs &a, cudaStream_t st);

// ---- finalize (fm_finalize.cu) ---------------------------------------------
cudaError_t launch_finalize(const float *acc_o, const float *acc_sum, const View &o,
                            cudaStream_t st);
// The same plus lse = ln2 * (acc_max + log2(acc_sum)) per row.
cudaError_t launch_finalize_lse(const float *acc_o, const float *acc_sum, const float *acc_max,
                                const View &o, float *lse, cudaStream_t st);

// Key sinks merged back into the accumulators after the last chunk (online merge per row).
cudaError_t launch_fold_sinks(const View &q, float alpha, const int32_t *sink_idx, const float *sink_k,
                              const float *sink_v, float *acc_o, float *acc_sum, float *acc_max,
                              cudaStream_t st);
// The same with the normalise in the same pass: o (and lse when given) written, acc_o not.
cudaError_t launch_fold_sinks_final(const View &q, float alpha, const int32_t *sink_idx, const float *sink_k,
                                    const float *sink_v, float *acc_o, float *acc_sum, float *acc_max, const View &o,
                                    float *lse, cudaStream_t st);

// ---- helpers shared by host code -------------------------------------------
int current_device_sm_count();
// L2 cache size of the current device in bytes (0 if unknown).
int current_device_l2_bytes();

// Programmatic dependent launch: the kernel may be scheduled while the kernel before it in
// the stream is still finishing, so its launch latency and block scheduling overlap that
// kernel's tail.  Every kernel launched this way runs pdl_wait() before it reads anything
// an earlier kernel wrote (the wait returns once the previous grid has completed and its
// memory is visible), and pdl_trigger() to let the next kernel be scheduled.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#endif

}  // namespace fm
