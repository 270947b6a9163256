// fm_api.cu -- the C ABI of libfm: argument validation, constants, dispatch.
//
// Every entry point validates its arguments on the host, returns an error code without
// enqueuing anything when they are wrong, and otherwise enqueues kernels on the caller's
// stream and returns immediately.  The only state kept is a thread-local error message
// and, per GPU, one device word where kernels record a pipeline wait that gave up.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>

#include <mutex>
#include <string>

#include "fm_internal.h"

namespace fm {

// Per-GPU error record: word 0 is set by the first kernel wait that ran past its limit
// (the role code); words 1-5 say where (barrier << 16 | tile, block x, y, z, thread).
constexpr int kErrWords = 8;
__device__ unsigned int g_dev_error[kErrWords];

namespace {

thread_local std::string t_err;

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char *what) {
  return fail(FM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

unsigned int *dev_error_ptr() {
  static unsigned int *ptrs[kMaxDevices] = {};
  static std::once_flag once[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::call_once(once[dev], [dev] {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_error) == cudaSuccess) ptrs[dev] = static_cast<unsigned int *>(p);
  });
  return ptrs[dev];
}

// ceil(log2 n) for n >= 1 (0 for n <= 1): the number of bits of n - 1.
int ceil_log2_i64(int64_t n) {
  if (n <= 1) return 0;
  uint64_t x = (uint64_t)(n - 1);
  int bits = 0;
  while (x) {
    ++bits;
    x >>= 1;
  }
  return bits;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Limit of one pipeline wait inside a kernel: kWaitTimeoutNs, or FM_WAIT_TIMEOUT_MS
// milliseconds from the environment (1 ms to 60 s).
unsigned long long wait_timeout_ns() {
  const char *s = getenv("FM_WAIT_TIMEOUT_MS");
  if (s && *s) {
    const long long ms = atoll(s);
    if (ms >= 1 && ms <= 60000) return (unsigned long long)ms * 1000000ull;
  }
  return kWaitTimeoutNs;
}

// Validate one fm_tensor and turn it into a View.  `what` names it in messages.
int to_view(const fm_tensor *t, const char *what, View *v) {
  if (!t) return fail(FM_ERR_ARG, "%s: NULL tensor", what);
  if (t->dtype == FM_F16 || t->dtype == FM_F8E4M3 || t->dtype == FM_F8E5M2)
    return fail(FM_ERR_DTYPE,
                "%s: fp16/fp8 inputs are rejected: 2^C-scale fixed-m terms overflow their exponent range",
                what);
  if (t->dtype != FM_F32 && t->dtype != FM_BF16) return fail(FM_ERR_ARG, "%s: unknown dtype %d", what, t->dtype);
  if (t->B < 0 || t->H < 0 || t->S < 0 || t->D < 0)
    return fail(FM_ERR_ARG, "%s: negative dimension [%lld,%lld,%lld,%lld]", what, (long long)t->B,
                (long long)t->H, (long long)t->S, (long long)t->D);
  for (int i = 0; i < 4; ++i)
    if (t->stride[i] < 0) return fail(FM_ERR_ARG, "%s: negative stride", what);
  if (t->D != 64 && t->D != 128)
    return fail(FM_ERR_UNSUPPORTED, "%s: head dimension %lld not supported (64 or 128)", what, (long long)t->D);
  if (t->B > 65535 || t->H > 65535) return fail(FM_ERR_UNSUPPORTED, "%s: B or H above 65535", what);
  const int64_t n = t->B * t->H * t->S * t->D;
  const size_t es = t->dtype == FM_F32 ? 4 : 2;
  if (n > 0 && !t->ptr) return fail(FM_ERR_ARG, "%s: NULL data pointer", what);
  if (reinterpret_cast<uintptr_t>(t->ptr) % es) return fail(FM_ERR_UNSUPPORTED, "%s: misaligned data", what);
  v->ptr = t->ptr;
  v->dtype = t->dtype;
  v->B = t->B;
  v->H = t->H;
  v->S = t->S;
  v->D = t->D;
  v->sB = t->stride[0];
  v->sH = t->stride[1];
  v->sS = t->stride[2];
  v->sD = t->stride[3];
  return FM_OK;
}

// softmax_scale -> alpha = scale * log2(e) (fp64), or an error.
int make_alpha(const fm_opts *opts, int64_t D, double *alpha) {
  double scale = (opts && opts->softmax_scale > 0.f) ? (double)opts->softmax_scale : 1.0 / sqrt((double)D);
  if (!(scale > 0.0) || !isfinite(scale)) return fail(FM_ERR_ARG, "softmax_scale must be finite");
  *alpha = scale * 1.4426950408889634;  // log2(e)
  return FM_OK;
}

int check_qkv(const View &q, const View &k, const View &v) {
  if (q.dtype != k.dtype || q.dtype != v.dtype) return fail(FM_ERR_DTYPE, "q, k and v must share one dtype");
  if (k.H != q.H || v.H != q.H)
    return fail(FM_ERR_UNSUPPORTED, "k/v heads (%lld/%lld) differ from q heads (%lld): GQA/MQA not supported",
                (long long)k.H, (long long)v.H, (long long)q.H);
  if (k.B != q.B || v.B != q.B) return fail(FM_ERR_SHAPE, "batch sizes of q, k, v differ");
  if (k.S != v.S) return fail(FM_ERR_SHAPE, "k and v lengths differ (%lld vs %lld)", (long long)k.S, (long long)v.S);
  if (k.D != q.D || v.D != q.D) return fail(FM_ERR_SHAPE, "head dimensions of q, k, v differ");
  return FM_OK;
}

}  // namespace

int current_device_l2_bytes() {
  static int sizes[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (!sizes[dev]) {
    int c = 0;
    cudaDeviceGetAttribute(&c, cudaDevAttrL2CacheSize, dev);
    sizes[dev] = c > 0 ? c : -1;
  }
  return sizes[dev] > 0 ? sizes[dev] : 0;
}

int current_device_sm_count() {
  static int counts[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  if (!counts[dev]) {
    int c = 0;
    cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
    counts[dev] = c > 0 ? c : 148;
  }
  return counts[dev];
}

}  // namespace fm

using namespace fm;

extern "C" {

int fm_version(void) { return (1 << 16) | 2; }

const char *fm_last_error(void) { return t_err.c_str(); }

int fm_bounds_workspace_size(int64_t B, int64_t H, int64_t N_total, int64_t D, size_t *bytes) {
  t_err.clear();
  if (!bytes) return fail(FM_ERR_ARG, "bytes is NULL");
  if (B < 0 || H < 0 || N_total < 0 || D < 0) return fail(FM_ERR_ARG, "negative size");
  *bytes = bounds_workspace_bytes(B, H, N_total, D);
  return FM_OK;
}

}  // extern "C"

namespace {
// Validation and the host-side fields that fm_bounds and fm_bounds_local share.  N_total < 0
// takes the key count of k (fm_bounds); the ring's rank gives the count over every shard.
// On success `a` is ready for the launch and *empty says that there is nothing to launch.
int setup_bounds(const fm_tensor *q, const fm_tensor *k, const fm_tensor *v, const fm_opts *opts, fm_bounds_out *out,
                 int64_t N_total, void *workspace, size_t workspace_bytes, BoundsArgs *a, bool *empty) {
  View vq, vk, vv;
  int rc;
  if ((rc = to_view(q, "q", &vq)) || (rc = to_view(k, "k", &vk)) || (rc = to_view(v, "v", &vv))) return rc;
  if ((rc = check_qkv(vq, vk, vv))) return rc;
  if (!out) return fail(FM_ERR_ARG, "out is NULL");
  if (opts && ((opts->centering != 0 && opts->centering != 1) || (opts->per_row != 0 && opts->per_row != 1)))
    return fail(FM_ERR_ARG, "centering and per_row must be 0 or 1");
  const int centering = opts ? opts->centering : 0;
  const int per_row = opts ? opts->per_row : 0;
  const int n_sink = opts ? opts->sink_keys : 0;
  if (n_sink < 0 || n_sink > FM_MAX_SINKS) return fail(FM_ERR_ARG, "sink_keys = %d outside [0, %d]", n_sink, FM_MAX_SINKS);
  double alpha;
  if ((rc = make_alpha(opts, vq.D, &alpha))) return rc;
  const int64_t B = vq.B, H = vq.H, Sq = vq.S, D = vq.D;
  const int64_t N = N_total < 0 ? vk.S : N_total;
  if (n_sink > 0 && B * H > 0 && (!out->sink_idx || !out->sink_k || !out->sink_v))
    return fail(FM_ERR_ARG, "fm_bounds_out: sink_idx, sink_k and sink_v must be set when sink_keys > 0");
  // the chunk kernels find a sink by its global key index in 32-bit arithmetic
  if (n_sink > 0 && N > (int64_t)INT32_MAX - 256)
    return fail(FM_ERR_UNSUPPORTED, "key sinks need N_total <= 2^31 - 256 (got %lld)", (long long)N);
  const int64_t nqb = ceil_div(Sq, FM_BLOCK_Q);
  // every non-empty device array must be given (torch hands out NULL for empty ones)
  if ((B * H * nqb > 0 && (!out->m || !out->flag || !out->qmax_sq)) ||
      (B * H * Sq > 0 && (!out->qkbar || !out->shift)) ||
      (B * H > 0 && (!out->kmax_sq || !out->kbar || !out->vmax_sq)))
    return fail(FM_ERR_ARG, "fm_bounds_out: every device array pointer must be set");
  const size_t need = bounds_workspace_bytes(B, H, vk.S, D);
  if (workspace_bytes < need) return fail(FM_ERR_ARG, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  if (need > 0 && !workspace) return fail(FM_ERR_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) % 16) return fail(FM_ERR_ARG, "workspace must be 16-byte aligned");

  // C(N) = 127 - ceil(log2 N) - ceil(log2 Vmax), W = C + 125, gate = floor(W / 2)
  // ("feat(attention): fixed-m splash attention kernel with dynamic bounds and safety
  // fallbacks", Summary).
  const int C = 127 - ceil_log2_i64(N) - ceil_log2_i64(FM_VMAX);
  const int W = C + 125;
  const int gate = W >= 0 ? W / 2 : -((-W + 1) / 2);

  out->B = B;
  out->H = H;
  out->Sq = Sq;
  out->D = D;
  out->n_qblocks = nqb;
  out->N_total = N;
  out->C = C;
  out->W = W;
  out->gate = gate;
  out->centered = centering;
  out->per_row = per_row;
  out->n_sink = n_sink;
  out->sinks_folded = 0;
  out->alpha = (float)alpha;
  out->dtype = vq.dtype;
  out->kv_seen = 0;
  out->next_key_offset = -1;
  out->online_lock = -1;
  out->magic = 0;
  *empty = B * H == 0;
  a->q = vq;
  a->k = vk;
  a->v = vv;
  a->err = dev_error_ptr();
  a->timeout_ns = wait_timeout_ns();
  a->centering = centering;
  a->per_row = per_row;
  a->alpha = alpha;
  a->C = C;
  a->gate = gate;
  a->nqb = nqb;
  a->m = out->m;
  a->flag = out->flag;
  a->qmax_sq = out->qmax_sq;
  a->kmax_sq = out->kmax_sq;
  a->kbar = out->kbar;
  a->qkbar = out->qkbar;
  a->shift = out->shift;
  a->vmax_sq = out->vmax_sq;
  a->n_sink = n_sink;
  a->sink_idx = out->sink_idx;
  a->sink_k = out->sink_k;
  a->sink_v = out->sink_v;
  a->ws = workspace;
  a->ws_bytes = workspace_bytes;
  return FM_OK;
}
}  // namespace

extern "C" {

int fm_bounds(const fm_tensor *q, const fm_tensor *k_full, const fm_tensor *v_full, const fm_opts *opts,
              fm_bounds_out *out, void *workspace, size_t workspace_bytes, fm_stream_t stream) {
  t_err.clear();
  BoundsArgs a;
  bool empty = false;
  int rc = setup_bounds(q, k_full, v_full, opts, out, -1, workspace, workspace_bytes, &a, &empty);
  if (rc) return rc;
  if (!empty) {
    cudaError_t e = launch_bounds(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fm_bounds launch");
  }
  out->magic = FM_BOUNDS_MAGIC;
  return FM_OK;
}

int fm_ring_stats_bytes(int64_t B, int64_t H, int64_t D, int sink_keys, size_t *bytes) {
  t_err.clear();
  if (!bytes) return fail(FM_ERR_ARG, "bytes is NULL");
  if (B < 0 || H < 0 || D < 0) return fail(FM_ERR_ARG, "negative size");
  if (sink_keys < 0 || sink_keys > FM_MAX_SINKS) return fail(FM_ERR_ARG, "sink_keys outside [0, %d]", FM_MAX_SINKS);
  *bytes = ring_stats_bytes(B, H, D, sink_keys);
  return FM_OK;
}

int fm_ring_key_sums(const fm_tensor *k_shard, float *ksum, void *workspace, size_t workspace_bytes,
                     fm_stream_t stream) {
  t_err.clear();
  View vk;
  int rc;
  if ((rc = to_view(k_shard, "k_shard", &vk))) return rc;
  if (vk.B * vk.H * vk.D > 0 && !ksum) return fail(FM_ERR_ARG, "ksum is NULL");
  const size_t need = bounds_workspace_bytes(vk.B, vk.H, vk.S, vk.D);
  if (workspace_bytes < need) return fail(FM_ERR_ARG, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  if (need > 0 && !workspace) return fail(FM_ERR_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) % 16) return fail(FM_ERR_ARG, "workspace must be 16-byte aligned");
  cudaError_t e = launch_ring_key_sums(vk, ksum, workspace, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fm_ring_key_sums launch");
  return FM_OK;
}

int fm_bounds_local(const fm_tensor *q, const fm_tensor *k_shard, const fm_tensor *v_shard, int64_t key_offset,
                    int64_t N_total, const float *ksum_total, const fm_opts *opts, fm_bounds_out *out, void *stats,
                    void *workspace, size_t workspace_bytes, fm_stream_t stream) {
  t_err.clear();
  if (!k_shard) return fail(FM_ERR_ARG, "k_shard is NULL");
  if (key_offset < 0 || N_total < 0 || k_shard->S < 0 || key_offset + k_shard->S > N_total)
    return fail(FM_ERR_ARG, "the shard's keys [%lld, %lld) must lie in [0, N_total = %lld)", (long long)key_offset,
                (long long)(key_offset + k_shard->S), (long long)N_total);
  // checked before anything of `out` is written
  const bool has_heads = q && q->B > 0 && q->H > 0;
  if (has_heads && opts && opts->centering && !ksum_total)
    return fail(FM_ERR_ARG, "centering needs ksum_total, the ring-wide key sums");
  if (has_heads && !stats) return fail(FM_ERR_ARG, "stats is NULL");
  if (reinterpret_cast<uintptr_t>(stats) % 16) return fail(FM_ERR_ARG, "stats must be 16-byte aligned");
  if (opts && opts->sink_keys > 0 && key_offset + k_shard->S > (int64_t)INT32_MAX)
    return fail(FM_ERR_UNSUPPORTED, "key sinks need global key indices below 2^31");
  BoundsArgs a;
  bool empty = false;
  int rc = setup_bounds(q, k_shard, v_shard, opts, out, N_total, workspace, workspace_bytes, &a, &empty);
  if (rc) return rc;
  if (!empty) {
    cudaError_t e = launch_bounds_local(a, ksum_total, N_total, key_offset, stats, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fm_bounds_local launch");
  }
  out->magic = FM_BOUNDS_LOCAL_MAGIC;
  return FM_OK;
}

int fm_bounds_combine(const void *stats_all, int n_ranks, const fm_opts *opts, fm_bounds_out *out,
                      fm_stream_t stream) {
  t_err.clear();
  if (!out) return fail(FM_ERR_ARG, "out is NULL");
  if (out->magic != FM_BOUNDS_LOCAL_MAGIC)
    return fail(FM_ERR_BOUNDS_MISMATCH, "out was not prepared by fm_bounds_local (magic 0x%08x)", out->magic);
  const int centering = opts ? opts->centering : 0;
  const int per_row = opts ? opts->per_row : 0;
  const int n_sink = opts ? opts->sink_keys : 0;
  double alpha;
  int rc;
  if ((rc = make_alpha(opts, out->D, &alpha))) return rc;
  if (centering != out->centered || per_row != out->per_row || n_sink != out->n_sink || (float)alpha != out->alpha)
    return fail(FM_ERR_BOUNDS_MISMATCH, "opts differ from the ones fm_bounds_local was given");
  if (n_ranks < 1) return fail(FM_ERR_ARG, "n_ranks = %d", n_ranks);
  const bool empty = out->B * out->H == 0;
  if (!empty && !stats_all) return fail(FM_ERR_ARG, "stats_all is NULL");
  if (reinterpret_cast<uintptr_t>(stats_all) % 16) return fail(FM_ERR_ARG, "stats_all must be 16-byte aligned");
  if (!empty) {
    BoundsArgs a;
    a.q = View{nullptr, out->dtype, out->B, out->H, out->Sq, out->D, 0, 0, 0, 0};
    a.k = a.v = a.q;
    a.centering = centering;
    a.per_row = per_row;
    a.alpha = alpha;
    a.C = out->C;
    a.gate = out->gate;
    a.nqb = out->n_qblocks;
    a.m = out->m;
    a.flag = out->flag;
    a.qmax_sq = out->qmax_sq;
    a.kmax_sq = out->kmax_sq;
    a.kbar = out->kbar;
    a.qkbar = out->qkbar;
    a.shift = out->shift;
    a.vmax_sq = out->vmax_sq;
    a.n_sink = n_sink;
    a.sink_idx = out->sink_idx;
    a.sink_k = out->sink_k;
    a.sink_v = out->sink_v;
    a.ws = nullptr;
    a.ws_bytes = 0;
    cudaError_t e = launch_bounds_combine(a, stats_all, n_ranks, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fm_bounds_combine launch");
  }
  out->kv_seen = 0;
  out->next_key_offset = -1;
  out->online_lock = -1;
  out->sinks_folded = 0;
  out->magic = FM_BOUNDS_MAGIC;
  return FM_OK;
}

}  // extern "C"

namespace {
// fm_attn_chunks: n consecutive chunks folded in order; with o_out given, the normalise of
// fm_attn_chunk_final follows the last one.  fm_attn_chunk and fm_attn_chunk_final are
// the n = 1 cases.
int attn_chunks_impl(const fm_tensor *q, const fm_tensor *k_chunks, const fm_tensor *v_chunks, int n_chunks,
                     fm_bounds_out *bounds, const fm_opts *opts, float *acc_o, float *acc_sum, float *acc_max,
                     int accumulate, const fm_tensor *o_out, float *lse, fm_stream_t stream) {
  t_err.clear();
  View vq;
  int rc;
  if ((rc = to_view(q, "q", &vq))) return rc;
  if (n_chunks < 1 || n_chunks > FM_MAX_CHUNKS)
    return fail(FM_ERR_ARG, "n_chunks = %d outside [1, %d]", n_chunks, FM_MAX_CHUNKS);
  if (!k_chunks || !v_chunks) return fail(FM_ERR_ARG, "k_chunks / v_chunks is NULL");
  View vk[FM_MAX_CHUNKS], vv[FM_MAX_CHUNKS];
  int64_t keys = 0;
  for (int c = 0; c < n_chunks; ++c) {
    if ((rc = to_view(&k_chunks[c], "k_chunk", &vk[c])) || (rc = to_view(&v_chunks[c], "v_chunk", &vv[c])))
      return rc;
    if ((rc = check_qkv(vq, vk[c], vv[c]))) return rc;
    keys += vk[c].S;
  }
  if (!bounds) return fail(FM_ERR_ARG, "bounds is NULL");
  if (accumulate != 0 && accumulate != 1) return fail(FM_ERR_ARG, "accumulate must be 0 or 1");
  if (opts && ((opts->centering != 0 && opts->centering != 1) || (opts->force_online != 0 && opts->force_online != 1)))
    return fail(FM_ERR_ARG, "centering and force_online must be 0 or 1");
  const int centering = opts ? opts->centering : 0;
  const int force_online = opts ? opts->force_online : 0;
  const int schedule = opts ? opts->schedule : FM_SCHEDULE_AUTO;
  if (schedule < FM_SCHEDULE_AUTO || schedule > FM_SCHEDULE_PERSISTENT)
    return fail(FM_ERR_ARG, "schedule = %d is not one of FM_SCHEDULE_AUTO, _GRID, _PERSISTENT", schedule);
  // the bounds must belong to this call
  if (bounds->magic != FM_BOUNDS_MAGIC)
    return fail(FM_ERR_BOUNDS_MISMATCH, "bounds were not produced by fm_bounds (magic 0x%08x)", bounds->magic);
  const int64_t nqb = ceil_div(vq.S, FM_BLOCK_Q);
  if (bounds->B != vq.B || bounds->H != vq.H || bounds->Sq != vq.S || bounds->n_qblocks != nqb ||
      bounds->D != vq.D)
    return fail(FM_ERR_BOUNDS_MISMATCH,
                "bounds shape [B=%lld,H=%lld,nqb=%lld] (Sq=%lld, D=%lld) does not match q [%lld,%lld,%lld] (Sq=%lld, "
                "D=%lld)",
                (long long)bounds->B, (long long)bounds->H, (long long)bounds->n_qblocks, (long long)bounds->Sq,
                (long long)bounds->D, (long long)vq.B, (long long)vq.H, (long long)nqb, (long long)vq.S,
                (long long)vq.D);
  if (bounds->centered != centering)
    return fail(FM_ERR_BOUNDS_MISMATCH,
                "bounds measured with centering=%d cannot serve a call with centering=%d: raw-key norms do not "
                "bound centered logits",
                bounds->centered, centering);
  if (bounds->dtype != vq.dtype) return fail(FM_ERR_BOUNDS_MISMATCH, "bounds were computed for another dtype");
  double alpha;
  if ((rc = make_alpha(opts, vq.D, &alpha))) return rc;
  if ((float)alpha != bounds->alpha)
    return fail(FM_ERR_BOUNDS_MISMATCH, "softmax scale differs from the one the bounds were computed with");
  const int64_t seen = accumulate ? bounds->kv_seen + keys : keys;
  if (seen > bounds->N_total)
    return fail(FM_ERR_BOUNDS_MISMATCH, "%lld keys folded in exceed the %lld keys the bounds cover",
                (long long)seen, (long long)bounds->N_total);
  if (accumulate && bounds->online_lock >= 0 && bounds->online_lock != force_online)
    return fail(FM_ERR_BOUNDS_MISMATCH, "force_online must stay the same across the chunks of one call");
  if (accumulate && bounds->online_lock < 0)
    return fail(FM_ERR_BOUNDS_MISMATCH, "accumulate=1 before any accumulate=0 chunk for these bounds");
  const int n_sink = opts ? opts->sink_keys : 0;
  if (n_sink != bounds->n_sink)
    return fail(FM_ERR_BOUNDS_MISMATCH,
                "bounds were built with sink_keys=%d, the call has sink_keys=%d: the chunks must skip exactly the "
                "keys left out of the key max",
                bounds->n_sink, n_sink);
  if (accumulate && bounds->sinks_folded)
    return fail(FM_ERR_BOUNDS_MISMATCH,
                "the key sinks were already folded in: no chunk may be added after fm_fold_sinks");
  if (n_sink > 0 && vq.B * vq.H > 0 && !bounds->sink_idx) return fail(FM_ERR_ARG, "bounds sink_idx is NULL");
  // the global index of this call's first key: given, or where the keys folded so far end
  if (bounds->next_key_offset < -1) return fail(FM_ERR_ARG, "next_key_offset = %lld", (long long)bounds->next_key_offset);
  const int64_t key_start = bounds->next_key_offset >= 0 ? bounds->next_key_offset : (accumulate ? bounds->kv_seen : 0);
  if (key_start + keys > bounds->N_total)
    return fail(FM_ERR_BOUNDS_MISMATCH, "keys [%lld, %lld) lie past the %lld keys the bounds cover",
                (long long)key_start, (long long)(key_start + keys), (long long)bounds->N_total);
  const int64_t rows = vq.B * vq.H * vq.S;
  if (rows > 0 && (!acc_o || !acc_sum || !acc_max)) return fail(FM_ERR_ARG, "accumulator pointer is NULL");
  if (rows > 0 && (!bounds->flag || !bounds->shift)) return fail(FM_ERR_ARG, "bounds flag/shift pointer is NULL");
  if (reinterpret_cast<uintptr_t>(acc_o) % 16 || reinterpret_cast<uintptr_t>(acc_sum) % 4 ||
      reinterpret_cast<uintptr_t>(acc_max) % 4)
    return fail(FM_ERR_ARG, "acc_o must be 16-byte aligned, acc_sum/acc_max 4-byte aligned");

  View vo;
  if (o_out) {
    if ((rc = to_view(o_out, "o_out", &vo))) return rc;
    if (vo.B != vq.B || vo.H != vq.H || vo.S != vq.S || vo.D != vq.D)
      return fail(FM_ERR_SHAPE, "o_out must have q's shape [B, H, Sq, D]");
  }
  unsigned int *err = dev_error_ptr();
  if (!err) return fail(FM_ERR_CUDA, "cannot resolve the device error word (no CUDA device?)");
  ChunkArgs a;
  a.q = vq;
  a.alpha = (float)alpha;
  a.force_online = force_online;
  // AUTO: the persistent schedule where a launch's work items are short (at most 8 key tiles,
  // e.g. one 1024-key chunk of a ring) and outnumber the SMs at least twice, so that its overlap
  // of the next item's Q load and first MMAs with the current epilogue pays (measured on GB300,
  // H40 S4096 in 1024-key chunks: chunk launches 778 against 761 TFLOP/s); one CTA per item
  // otherwise (2-chunk S4096: 1138 against 1153; Wan: 1483 against 1523).
  a.schedule = schedule;
  if (schedule == FM_SCHEDULE_AUTO) {
    int64_t tiles = 0;
    for (int c = 0; c < n_chunks; ++c) tiles += ceil_div(vk[c].S, 128);
    const int64_t items = vq.B * vq.H * ceil_div(nqb, 2);
    a.schedule = (tiles <= 8 && items >= 2 * (int64_t)current_device_sm_count()) ? FM_SCHEDULE_PERSISTENT
                                                                                  : FM_SCHEDULE_GRID;
  }
  a.nqb = nqb;
  a.flag = bounds->flag;
  a.shift = bounds->shift;
  a.acc_o = acc_o;
  a.acc_sum = acc_sum;
  a.acc_max = acc_max;
  a.err = err;
  a.timeout_ns = wait_timeout_ns();
  // key sinks: the chunks skip them by global key index; the first chunk of this call
  // starts where the keys folded so far end
  a.sinks = n_sink > 0 ? bounds->sink_idx : nullptr;
  a.key0 = key_start;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  bool finalize_separately = o_out != nullptr;
  if (rows > 0) {
    // chunks without keys add nothing; only the accumulators' first initialisation matters
    View ks[FM_MAX_CHUNKS], vs[FM_MAX_CHUNKS];
    int n = 0;
    for (int c = 0; c < n_chunks; ++c)
      if (vk[c].S > 0) {
        ks[n] = vk[c];
        vs[n] = vv[c];
        ++n;
      }
    a.accumulate = accumulate;
    if (n == 0) {
      if (!accumulate) {
        a.k = vk[0];
        a.v = vv[0];
        e = launch_chunk_empty_init(a, st);
      }
    } else {
      a.k = ks[0];
      a.v = vs[0];
      a.n_chunks = n;
      a.ks = ks;
      a.vs = vs;
      if (chunk_tc_supported(a)) {
        // the kernel normalises and writes o itself, unless key sinks must be folded first
        if (o_out && n_sink == 0 && chunk_tc_final_supported(a, vo)) {
          a.out = &vo;
          a.lse = lse;
          finalize_separately = false;
        }
        e = launch_chunk_tc(a, st);
        if (e == cudaErrorNotSupported) {  // tensor maps refused: the CUDA-core kernel, chunk by chunk
          finalize_separately = o_out != nullptr;
          e = cudaSuccess;
        } else {
          n = 0;  // done
        }
      }
      a.out = nullptr;
      a.lse = nullptr;
      a.n_chunks = 0;
      for (int c = 0; c < n && e == cudaSuccess; ++c) {
        a.k = ks[c];
        a.v = vs[c];
        a.accumulate = c == 0 ? accumulate : 1;
        e = launch_chunk_simt(a, st);
        a.key0 += ks[c].S;
      }
    }
  }
  if (e != cudaSuccess) return cuda_fail(e, "fm_attn_chunk launch");
  if (o_out && n_sink > 0 && rows > 0) {  // the last chunk is in: merge the sinks back and normalise
    e = launch_fold_sinks_final(vq, (float)alpha, bounds->sink_idx, bounds->sink_k, bounds->sink_v, acc_o, acc_sum,
                                acc_max, vo, lse, st);
    if (e != cudaSuccess) return cuda_fail(e, "key-sink fold launch");
    finalize_separately = false;
  }
  if (finalize_separately && rows > 0) {
    e = lse ? launch_finalize_lse(acc_o, acc_sum, acc_max, vo, lse, st) : launch_finalize(acc_o, acc_sum, vo, st);
    if (e != cudaSuccess) return cuda_fail(e, "fm_attn_chunk_final finalize launch");
  }
  bounds->kv_seen = seen;
  bounds->next_key_offset = -1;
  bounds->online_lock = force_online;
  bounds->sinks_folded = (o_out && n_sink > 0) ? 1 : 0;
  return FM_OK;
}
}  // namespace

extern "C" {

int fm_attn_chunk(const fm_tensor *q, const fm_tensor *k_chunk, const fm_tensor *v_chunk, fm_bounds_out *bounds,
                  const fm_opts *opts, float *acc_o, float *acc_sum, float *acc_max, int accumulate,
                  fm_stream_t stream) {
  return attn_chunks_impl(q, k_chunk, v_chunk, 1, bounds, opts, acc_o, acc_sum, acc_max, accumulate, nullptr,
                          nullptr, stream);
}

int fm_attn_chunks(const fm_tensor *q, const fm_tensor *k_chunks, const fm_tensor *v_chunks, int n_chunks,
                   fm_bounds_out *bounds, const fm_opts *opts, float *acc_o, float *acc_sum, float *acc_max,
                   int accumulate, const fm_tensor *o_out, float *lse, fm_stream_t stream) {
  return attn_chunks_impl(q, k_chunks, v_chunks, n_chunks, bounds, opts, acc_o, acc_sum, acc_max, accumulate, o_out,
                          lse, stream);
}

int fm_attn_chunk_final(const fm_tensor *q, const fm_tensor *k_chunk, const fm_tensor *v_chunk,
                        fm_bounds_out *bounds, const fm_opts *opts, float *acc_o, float *acc_sum, float *acc_max,
                        int accumulate, const fm_tensor *o_out, float *lse, fm_stream_t stream) {
  if (!o_out) {
    t_err.clear();
    return fail(FM_ERR_ARG, "o_out is NULL");
  }
  return attn_chunks_impl(q, k_chunk, v_chunk, 1, bounds, opts, acc_o, acc_sum, acc_max, accumulate, o_out, lse,
                          stream);
}

int fm_finalize(const float *acc_o, const float *acc_sum, const fm_tensor *o_out, fm_stream_t stream) {
  t_err.clear();
  View vo;
  int rc;
  if ((rc = to_view(o_out, "o_out", &vo))) return rc;
  const int64_t rows = vo.B * vo.H * vo.S;
  if (rows > 0 && (!acc_o || !acc_sum)) return fail(FM_ERR_ARG, "accumulator pointer is NULL");
  if (reinterpret_cast<uintptr_t>(acc_o) % 16) return fail(FM_ERR_ARG, "acc_o must be 16-byte aligned");
  cudaError_t e = launch_finalize(acc_o, acc_sum, vo, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fm_finalize launch");
  return FM_OK;
}

int fm_finalize_lse(const float *acc_o, const float *acc_sum, const float *acc_max, const fm_tensor *o_out,
                    float *lse, fm_stream_t stream) {
  t_err.clear();
  View vo;
  int rc;
  if ((rc = to_view(o_out, "o_out", &vo))) return rc;
  const int64_t rows = vo.B * vo.H * vo.S;
  if (rows > 0 && (!acc_o || !acc_sum || !acc_max || !lse)) return fail(FM_ERR_ARG, "a pointer is NULL");
  if (reinterpret_cast<uintptr_t>(acc_o) % 16) return fail(FM_ERR_ARG, "acc_o must be 16-byte aligned");
  cudaError_t e = launch_finalize_lse(acc_o, acc_sum, acc_max, vo, lse, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fm_finalize_lse launch");
  return FM_OK;
}

int fm_fold_sinks(const fm_tensor *q, fm_bounds_out *bounds, const fm_opts *opts, float *acc_o, float *acc_sum,
                  float *acc_max, fm_stream_t stream) {
  t_err.clear();
  View vq;
  int rc;
  if ((rc = to_view(q, "q", &vq))) return rc;
  if (!bounds) return fail(FM_ERR_ARG, "bounds is NULL");
  if (bounds->magic != FM_BOUNDS_MAGIC)
    return fail(FM_ERR_BOUNDS_MISMATCH, "bounds were not produced by fm_bounds (magic 0x%08x)", bounds->magic);
  if (bounds->B != vq.B || bounds->H != vq.H || bounds->Sq != vq.S || bounds->D != vq.D || bounds->dtype != vq.dtype)
    return fail(FM_ERR_BOUNDS_MISMATCH, "bounds do not belong to these queries");
  const int n_sink = opts ? opts->sink_keys : 0;
  if (n_sink != bounds->n_sink)
    return fail(FM_ERR_BOUNDS_MISMATCH, "bounds were built with sink_keys=%d, the call has sink_keys=%d",
                bounds->n_sink, n_sink);
  double alpha;
  if ((rc = make_alpha(opts, vq.D, &alpha))) return rc;
  if ((float)alpha != bounds->alpha)
    return fail(FM_ERR_BOUNDS_MISMATCH, "softmax scale differs from the one the bounds were computed with");
  if (bounds->online_lock < 0) return fail(FM_ERR_BOUNDS_MISMATCH, "no chunk has been folded in yet");
  if (bounds->sinks_folded) return fail(FM_ERR_BOUNDS_MISMATCH, "the key sinks were already folded in");
  if (n_sink == 0) return FM_OK;
  const int64_t rows = vq.B * vq.H * vq.S;
  if (rows > 0 && (!acc_o || !acc_sum || !acc_max)) return fail(FM_ERR_ARG, "accumulator pointer is NULL");
  if (rows > 0 && (!bounds->sink_idx || !bounds->sink_k || !bounds->sink_v))
    return fail(FM_ERR_ARG, "bounds sink arrays are NULL");
  if (reinterpret_cast<uintptr_t>(acc_o) % 16) return fail(FM_ERR_ARG, "acc_o must be 16-byte aligned");
  cudaError_t e = launch_fold_sinks(vq, (float)alpha, bounds->sink_idx, bounds->sink_k, bounds->sink_v, acc_o,
                                    acc_sum, acc_max, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fm_fold_sinks launch");
  bounds->sinks_folded = 1;
  return FM_OK;
}

int fm_probe_wait_timeout(unsigned int timeout_ms, fm_stream_t stream) {
  t_err.clear();
  if (timeout_ms < 1 || timeout_ms > 10000) return fail(FM_ERR_ARG, "timeout_ms must be in [1, 10000]");
  unsigned int *err = dev_error_ptr();
  if (!err) return fail(FM_ERR_CUDA, "cannot resolve the device error word (no CUDA device?)");
  cudaError_t e = launch_wait_probe(err, (unsigned long long)timeout_ms * 1000000ull,
                                    reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fm_probe_wait_timeout launch");
  return FM_OK;
}

int fm_sync_status(fm_stream_t stream) {
  t_err.clear();
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned int w[kErrWords] = {};
  e = cudaMemcpyFromSymbol(w, g_dev_error, sizeof w);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (w[0] != 0) {
    const unsigned int zero[kErrWords] = {};
    cudaMemcpyToSymbol(g_dev_error, zero, sizeof zero);
    if (w[0] == kDevErrDebugIndex)
      return fail(FM_ERR_INDEX,
                  "a debug build's index check failed and skipped the access (site %u, index %llu, block %u, "
                  "thread %u); outputs are invalid",
                  w[1], (unsigned long long)w[2] | ((unsigned long long)w[3] << 32), w[4], w[5]);
    return fail(FM_ERR_TIMEOUT,
                "a kernel pipeline wait ran past its limit (role %u, barrier %u, tile %u, block (%u,%u,%u), "
                "thread %u); outputs are invalid",
                w[0], w[1] >> 16, w[1] & 0xFFFFu, w[2], w[3], w[4], w[5]);
  }
  return FM_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------------
// fm_bounds_noalloc: fm_bounds with its scratch in a file-scope device array, for callers
// that cannot allocate.  The array is per GPU and lives as long as the process; host code
// only ever sees a stand-in for its name, so its device address is looked up once per
// device, with that device current, and that address is what the kernels receive.
namespace fm {
namespace {

__device__ __align__(256) unsigned char g_bounds_scratch[FM_NOALLOC_SCRATCH_BYTES];

int bounds_scratch_address(void **addr) {
  static void *ptrs[kMaxDevices] = {};
  static cudaError_t errs[kMaxDevices] = {};
  static std::once_flag once[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "fm_bounds_noalloc: no current device");
  if (dev < 0 || dev >= kMaxDevices) return fail(FM_ERR_UNSUPPORTED, "fm_bounds_noalloc: device index %d", dev);
  std::call_once(once[dev], [dev] {
    void *p = nullptr;
    errs[dev] = cudaGetSymbolAddress(&p, g_bounds_scratch);
    if (errs[dev] == cudaSuccess) ptrs[dev] = p;
  });
  if (errs[dev] != cudaSuccess) return cuda_fail(errs[dev], "fm_bounds_noalloc: cudaGetSymbolAddress");
  *addr = ptrs[dev];
  return FM_OK;
}

}  // namespace
}  // namespace fm

extern "C" int fm_bounds_noalloc(const fm_tensor *q, const fm_tensor *k_full, const fm_tensor *v_full,
                                 const fm_opts *opts, fm_bounds_out *out, fm_stream_t stream) {
  t_err.clear();
  if (k_full && k_full->B >= 0 && k_full->H >= 0 && k_full->S >= 0 && k_full->D >= 0) {
    const size_t need = bounds_workspace_bytes(k_full->B, k_full->H, k_full->S, k_full->D);
    if (need > FM_NOALLOC_SCRATCH_BYTES)
      return fail(FM_ERR_UNSUPPORTED,
                  "fm_bounds_noalloc: this problem needs %zu bytes of scratch; the library's static scratch "
                  "holds %zu (use fm_bounds with a workspace)",
                  need, (size_t)FM_NOALLOC_SCRATCH_BYTES);
  }
  void *scratch = nullptr;
  int rc = bounds_scratch_address(&scratch);
  if (rc != FM_OK) return rc;
  return fm_bounds(q, k_full, v_full, opts, out, scratch, FM_NOALLOC_SCRATCH_BYTES, stream);
}

// ---------------------------------------------------------------------------------
// fm_attention_host: whole forwards on host buffers, copies overlapped with the kernels.
namespace {

bool contiguous4(const fm_tensor *t) {
  return t->stride[3] == 1 && t->stride[2] == t->D && t->stride[1] == t->S * t->D && t->stride[0] == t->H * t->S * t->D;
}
size_t tensor_bytes(const fm_tensor *t) {
  return (size_t)(t->B * t->H * t->S * t->D) * (t->dtype == FM_F32 ? 4 : 2);
}
bool same_shape(const fm_tensor *a, const fm_tensor *b) {
  return a->dtype == b->dtype && a->B == b->B && a->H == b->H && a->S == b->S && a->D == b->D;
}

// Events of one call, destroyed on every return path.
struct EventSet {
  cudaEvent_t ev[6] = {};
  int n = 0;
  cudaError_t create() {
    for (; n < 6; ++n) {
      cudaError_t e = cudaEventCreateWithFlags(&ev[n], cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  ~EventSet() {
    for (int i = 0; i < n; ++i) cudaEventDestroy(ev[i]);
  }
};

}  // namespace

extern "C" int fm_attention_host(const fm_tensor *q_host, const fm_tensor *k_host, const fm_tensor *v_host,
                                 const fm_tensor *o_host, int n_batches, const int64_t *chunk_lens, int n_chunks,
                                 const fm_opts *opts, const fm_host_buffers *dev, const fm_stream_t *streams) {
  t_err.clear();
  if (!q_host || !k_host || !v_host || !o_host || !dev || !streams || !chunk_lens)
    return fail(FM_ERR_ARG, "fm_attention_host: NULL argument");
  if (n_batches < 0 || n_chunks < 1) return fail(FM_ERR_ARG, "n_batches = %d, n_chunks = %d", n_batches, n_chunks);
  if (!streams[0] || !streams[1] || !streams[2])
    return fail(FM_ERR_ARG, "fm_attention_host needs three streams (upload, compute, read-back)");
  // every buffer contiguous, the host ones shaped like the device ones
  for (int s = 0; s < 2; ++s) {
    const fm_tensor *d[4] = {&dev->q[s], &dev->k[s], &dev->v[s], &dev->o[s]};
    for (const fm_tensor *t : d)
      if (!contiguous4(t)) return fail(FM_ERR_UNSUPPORTED, "fm_attention_host: device buffers must be contiguous");
    if (!same_shape(&dev->q[s], &dev->q[0]) || !same_shape(&dev->k[s], &dev->k[0]) ||
        !same_shape(&dev->v[s], &dev->v[0]) || !same_shape(&dev->o[s], &dev->o[0]))
      return fail(FM_ERR_SHAPE, "fm_attention_host: the two buffer sets differ");
  }
  int64_t N = 0;
  for (int c = 0; c < n_chunks; ++c) {
    if (chunk_lens[c] < 0) return fail(FM_ERR_ARG, "negative chunk length");
    N += chunk_lens[c];
  }
  if (N != dev->k[0].S) return fail(FM_ERR_SHAPE, "chunk lengths sum to %lld, k has %lld keys", (long long)N,
                                    (long long)dev->k[0].S);
  for (int i = 0; i < n_batches; ++i) {
    const fm_tensor *h[4] = {&q_host[i], &k_host[i], &v_host[i], &o_host[i]};
    const fm_tensor *d[4] = {&dev->q[0], &dev->k[0], &dev->v[0], &dev->o[0]};
    for (int j = 0; j < 4; ++j) {
      if (!contiguous4(h[j])) return fail(FM_ERR_UNSUPPORTED, "fm_attention_host: host buffers must be contiguous");
      if (!same_shape(h[j], d[j])) return fail(FM_ERR_SHAPE, "fm_attention_host: batch %d's host buffer %d differs", i, j);
      if (tensor_bytes(h[j]) > 0 && !h[j]->ptr) return fail(FM_ERR_ARG, "fm_attention_host: NULL host pointer");
    }
  }
  cudaStream_t up = reinterpret_cast<cudaStream_t>(streams[0]), comp = reinterpret_cast<cudaStream_t>(streams[1]),
               down = reinterpret_cast<cudaStream_t>(streams[2]);
  EventSet es;
  cudaError_t e = es.create();
  if (e != cudaSuccess) return cuda_fail(e, "fm_attention_host: cudaEventCreate");
  cudaEvent_t *uploaded = es.ev, *computed = es.ev + 2, *read_back = es.ev + 4;
  bool used[2] = {false, false};
  fm_bounds_out *bounds = dev->bounds;
  for (int i = 0; i < n_batches; ++i) {
    const int s = i & 1;
    // upload into slot s once the batch that last used it has finished reading its inputs
    if (used[s] && (e = cudaStreamWaitEvent(up, computed[s], 0)) != cudaSuccess) return cuda_fail(e, "wait");
    const fm_tensor *src[3] = {&q_host[i], &k_host[i], &v_host[i]};
    const fm_tensor *dst[3] = {&dev->q[s], &dev->k[s], &dev->v[s]};
    for (int j = 0; j < 3; ++j)
      if (tensor_bytes(src[j]) > 0 &&
          (e = cudaMemcpyAsync(dst[j]->ptr, src[j]->ptr, tensor_bytes(src[j]),
                               cudaMemcpyHostToDevice, up)) != cudaSuccess)
        return cuda_fail(e, "fm_attention_host: upload");
    if ((e = cudaEventRecord(uploaded[s], up)) != cudaSuccess) return cuda_fail(e, "record");
    // compute once the inputs are in and the output slot has been read back
    if ((e = cudaStreamWaitEvent(comp, uploaded[s], 0)) != cudaSuccess) return cuda_fail(e, "wait");
    if (used[s] && (e = cudaStreamWaitEvent(comp, read_back[s], 0)) != cudaSuccess) return cuda_fail(e, "wait");
    int rc = fm_bounds(&dev->q[s], &dev->k[s], &dev->v[s], opts, bounds, dev->workspace, dev->workspace_bytes,
                       streams[1]);
    if (rc) return rc;
    int64_t start = 0;
    for (int c = 0; c < n_chunks; ++c) {
      fm_tensor kc = dev->k[s], vc = dev->v[s];
      const size_t es2 = kc.dtype == FM_F32 ? 4 : 2;
      kc.ptr = static_cast<char *>(kc.ptr) + (size_t)(start * kc.stride[2]) * es2;
      vc.ptr = static_cast<char *>(vc.ptr) + (size_t)(start * vc.stride[2]) * es2;
      kc.S = vc.S = chunk_lens[c];
      // the chunk's slice [start, start + len) of a contiguous K/V keeps the full tensor's strides
      bounds->next_key_offset = start;
      if (c == n_chunks - 1)
        rc = fm_attn_chunk_final(&dev->q[s], &kc, &vc, bounds, opts, dev->acc_o, dev->acc_sum, dev->acc_max, c > 0,
                                 &dev->o[s], nullptr, streams[1]);
      else
        rc = fm_attn_chunk(&dev->q[s], &kc, &vc, bounds, opts, dev->acc_o, dev->acc_sum, dev->acc_max, c > 0,
                           streams[1]);
      if (rc) return rc;
      start += chunk_lens[c];
    }
    if ((e = cudaEventRecord(computed[s], comp)) != cudaSuccess) return cuda_fail(e, "record");
    // read the output back once it is computed
    if ((e = cudaStreamWaitEvent(down, computed[s], 0)) != cudaSuccess) return cuda_fail(e, "wait");
    if (tensor_bytes(&o_host[i]) > 0 &&
        (e = cudaMemcpyAsync(o_host[i].ptr, dev->o[s].ptr, tensor_bytes(&o_host[i]),
                             cudaMemcpyDeviceToHost, down)) != cudaSuccess)
      return cuda_fail(e, "fm_attention_host: read-back");
    if ((e = cudaEventRecord(read_back[s], down)) != cudaSuccess) return cuda_fail(e, "record");
    used[s] = true;
  }
  for (cudaStream_t st : {up, comp, down})
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "fm_attention_host: synchronize");
  return FM_OK;
}
