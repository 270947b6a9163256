/*
 * fm.h -- C ABI of the fixed-m (const-max) attention forward for GB300 (sm_103a).
 *
 * The method replaces softmax's running row maximum by a shift fixed before any
 * score is computed, so that the base-2 numerator and denominator of every row
 * build up as plain fp32 sums across KV chunks, with one divide at the end.
 * Page references (title, section):
 *   [NKI]   "Kernel reference: ring_attention_const_max_fwd const-max ring attention"
 *   [PR477] "feat(attention): fixed-m splash attention kernel with dynamic bounds and
 *            safety fallbacks" (maxdiffusion PR #477)
 *   [PR478] "feat(attention): 2D Ulysses+Ring attention with Global Virtual
 *            K-Centering" (maxdiffusion PR #478)
 *
 * Call sequence for one attention forward over a key sequence split into chunks
 * (the ring's KV steps, run one after another on one GPU):
 *     fm_bounds(q, k_full, v_full)                       once
 *     fm_attn_chunk(q, k_c, v_c, accumulate = c > 0)     once per chunk c
 *     fm_finalize(acc_o, acc_sum -> o)                   once
 * or, fusing the last two: fm_attn_chunk_final(..., o) for the last chunk.
 * With key sinks (opts.sink_keys > 0) the loudest keys of each head are left out of the
 * key max and out of the chunks' fixed-m sums, and fm_fold_sinks merges them back exactly
 * after the last chunk (fm_attn_chunk_final and fm_attn_chunks with o_out do this
 * themselves).
 *
 * Conventions shared by every call:
 *   - Tensors are described by fm_tensor: a logical [B, H, S, D] array with element
 *     strides (any order, e.g. [B,H,S,D] or the pages' token-major [B,S,H,D]).
 *   - All buffers are device memory owned by the caller; the library allocates
 *     nothing and keeps no state besides a thread-local error string and one
 *     device-side error word per GPU.
 *   - Calls validate on the host, enqueue kernels on `stream` and return without
 *     synchronising.  On any error code nothing is enqueued and no output buffer is
 *     touched; fm_last_error() returns a message for the calling thread.
 *   - Device-side failures (a pipeline wait that exceeded its time limit) are
 *     reported by fm_sync_status().
 */
#ifndef FM_H_
#define FM_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FM_API __attribute__((visibility("default")))
#else
#define FM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *fm_stream_t;

/* Element types.  Only FM_F32 and FM_BF16 are accepted: [PR477]'s commit message
 * rejects fp16 (and fp8) because 2^C-scale terms overflow their exponent range
 * (Q = K = 0, V = 1 gives inf instead of 1.0); here they fail with FM_ERR_DTYPE. */
enum { FM_F32 = 0, FM_BF16 = 1, FM_F16 = 2, FM_F8E4M3 = 3, FM_F8E5M2 = 4 };

/* Return codes. */
enum {
  FM_OK = 0,
  FM_ERR_ARG = 1,             /* NULL pointer, negative size, bad flag value */
  FM_ERR_SHAPE = 2,           /* shapes of q / k / v / outputs disagree */
  FM_ERR_DTYPE = 3,           /* fp16 / fp8, or q, k, v of different types */
  FM_ERR_UNSUPPORTED = 4,     /* D not in {64, 128}; GQA (k.H != q.H); misaligned data */
  FM_ERR_BOUNDS_MISMATCH = 5, /* bounds do not belong to this call (see fm_attn_chunk) */
  FM_ERR_CUDA = 6,            /* a CUDA runtime call or kernel launch failed */
  FM_ERR_TIMEOUT = 7,         /* a kernel's pipeline wait ran past its limit */
  FM_ERR_INDEX = 8            /* debug builds only (FM_DEBUG): a kernel's index check failed */
};

#define FM_BOUNDS_MAGIC 0x314D4246u /* tag written by fm_bounds ("FBM1") */
#define FM_BOUNDS_LOCAL_MAGIC 0x314C4246u /* fm_bounds_local done, fm_bounds_combine pending ("FBL1") */
#define FM_BLOCK_Q 128              /* rows per Q-block: the granularity of m and flag */
#define FM_VMAX 256                 /* the V bound of [PR477]'s commit message */
#define FM_SUM_CLAMP 1e-37f         /* [NKI] "Accumulate, then normalize once" */
#define FM_MAX_SINKS 8              /* most key sinks per head (opts.sink_keys) */

/* A logical [B, H, S, D] tensor: element (b,h,s,d) lives at
 * ptr + (b*stride[0] + h*stride[1] + s*stride[2] + d*stride[3]) * elemsize. */
typedef struct {
  void *ptr;
  int32_t dtype; /* FM_F32 or FM_BF16 */
  int32_t reserved;
  int64_t B, H, S, D;
  int64_t stride[4]; /* element strides, >= 0 */
} fm_tensor;

typedef struct {
  float softmax_scale;  /* <= 0 selects 1/sqrt(D) ([NKI] Interface table) */
  int32_t centering;    /* 1: virtual K-centering ([PR477] "Virtual K-centering") */
  int32_t force_online; /* 1: every Q-block takes the online-softmax fallback */
  int32_t per_row;      /* 1: each query row gets its own shift m_i = ceil(U_i) - C, with
                           U_i = alpha*|q_i|*max|k| ([NKI] "Best practices": give each query
                           row its own bound); 0: one m per 128-row Q-block ([PR477]).
                           Eligibility stays per Q-block in both cases. */
  int32_t sink_keys;    /* 0..FM_MAX_SINKS: leave up to this many of each head's loudest
                           keys out of the key max ([NKI] "Adapting this kernel": attention
                           sinks inflate max|k| for every row, and excluding those few keys
                           from the max reduction recovers the bound).  The sinks are the
                           keys whose norm (|k - kbar| with centering) is strictly above the
                           (sink_keys+1)-th largest, so ties at that norm stay ordinary keys;
                           kmax_sq becomes that norm squared.  The chunks skip the sinks and
                           fm_fold_sinks merges them back exactly, so the output is still
                           plain attention over every key. */
  int32_t schedule;     /* how the tensor-core chunk kernel spreads its work (FM_SCHEDULE_*);
                           the result is the same bits either way.  Ignored by fm_bounds. */
} fm_opts;

/* fm_opts.schedule.  A work item is two 128-row Q tiles of one (batch, head) against every key
 * tile of the call.  GRID launches one CTA per item.  PERSISTENT launches one CTA per SM that
 * walks the items in turn, loading the next item's Q and K/V tiles and running its first S
 * MMAs while the softmax warps finish the current item's epilogue (its K/V ring has one stage
 * fewer; that space stages O for the bulk accumulator add; the CTAs with one item fewer start
 * spread over an item's time, so that the CTAs' epilogues do not all meet the memory system at
 * once).  AUTO takes PERSISTENT when the
 * call has at most 8 key tiles (1024 keys) and at least twice as many items as the GPU has SMs,
 * GRID otherwise: measured on GB300, the overlap pays on such short items and the simpler grid
 * wins on longer ones. */
enum { FM_SCHEDULE_AUTO = 0, FM_SCHEDULE_GRID = 1, FM_SCHEDULE_PERSISTENT = 2 };

/* Bounds of one attention call ([PR477] Summary, "Dynamic eligibility bounding").
 * The caller allocates the device arrays and fills the pointers; fm_bounds fills
 * every other field.  nqb = ceil(Sq / FM_BLOCK_Q).
 *   m       int32 [B, H, nqb]  per-(head, Q-block) shift m = ceil(U) - C(N)
 *   flag    uint8 [B, H, nqb]  1 = eligible for fixed-m: v_ok && U <= gate
 *   qmax_sq f32   [B, H, nqb]  max over the block's rows of ||q_i||^2
 *   kmax_sq f32   [B, H]       max_j ||k_j - kbar||^2 (centered) or ||k_j||^2, over the
 *                              keys that are not sinks
 *   kbar    f32   [B, H, D]    mean key over all real keys ([PR478] Summary); 0 if
 *                              not centering
 *   qkbar   f32   [B, H, Sq]   alpha * q_i . kbar, the per-row centering term; 0 if not
 *                              centering
 *   shift   f32   [B, H, Sq]   the row's whole base-2 shift b_i = m_i + qkbar_i, with m_i
 *                              the row's own ceil(U_i) - C (opts.per_row) or its Q-block's
 *                              m; the chunk kernels subtract it in registers
 *   vmax_sq f32   [1]          max over all of V of v^2 (v_ok = vmax_sq <= 256^2)
 *   sink_idx int32 [B, H, FM_MAX_SINKS]  global key indices of the head's sinks, ascending,
 *                              padded with INT32_MAX (only with opts.sink_keys > 0)
 *   sink_k, sink_v f32 [B, H, FM_MAX_SINKS, D]  the sinks' raw key and value rows (zero in
 *                              padding slots), kept for fm_fold_sinks (sink_keys > 0 only)
 * with alpha = softmax_scale * log2(e) (base-2 logits, [PR477]'s exp2 formulation)
 * and U = alpha * sqrt(qmax_sq) * sqrt(kmax_sq), the Cauchy-Schwarz bound on the
 * base-2 logit ([NKI] "Picking a max that is safe without measuring it"). */
typedef struct {
  int32_t *m;
  uint8_t *flag;
  float *qmax_sq;
  float *kmax_sq;
  float *kbar;
  float *qkbar;
  float *shift;
  float *vmax_sq;
  int32_t *sink_idx; /* required when opts.sink_keys > 0, else ignored (may be NULL) */
  float *sink_k;
  float *sink_v;
  /* filled by fm_bounds */
  int64_t B, H, Sq, D, n_qblocks;
  int64_t N_total;   /* total KV length over every chunk of the call */
  int32_t C, W, gate; /* C(N) = 127 - ceil(log2 N) - 8, W = C + 125, gate = floor(W/2) */
  int32_t centered;  /* the opts.centering the bounds were measured with */
  int32_t per_row;   /* the opts.per_row they were built with */
  int32_t n_sink;    /* the opts.sink_keys they were built with */
  float alpha;
  int32_t dtype;
  /* updated by fm_attn_chunk (host-side bookkeeping of the chunk sequence) */
  int64_t kv_seen;
  int64_t next_key_offset; /* -1 (as fm_bounds / fm_bounds_combine and every chunk call leave it):
                              the next chunk's first key has global index kv_seen (0 with
                              accumulate = 0), i.e. the chunks come in key order.  A caller that
                              folds them in another order -- a ring hands rank r the shards in
                              the rotated order r, r-1, ... -- sets it to the chunk's global offset
                              before the call.  Only key sinks depend on it (they are found by
                              global key index). */
  int32_t online_lock;
  int32_t sinks_folded; /* set by fm_fold_sinks; no chunk may follow it */
  uint32_t magic; /* FM_BOUNDS_MAGIC once fm_bounds has succeeded */
} fm_bounds_out;

/* Scratch bytes fm_bounds needs for k_full of shape [B, H, N_total, D] (partial
 * key sums for the mean, per-block key and value maxima, per-block key-sink candidates).
 * Returns FM_OK. */
FM_API int fm_bounds_workspace_size(int64_t B, int64_t H, int64_t N_total, int64_t D, size_t *bytes);

/* fm_bounds -- norms, key mean, m and the per-tile flag ([PR477] Summary; the
 * fused norm reduction of [NKI] "Transpose prologue with fused norms" and [PR478]).
 *   q      [B, H, Sq, D]  queries (all rows of the call)
 *   k_full [B, H, N, D]   ALL keys of the call (every chunk), N = N_total
 *   v_full [B, H, N, D]   all values
 *   opts   softmax_scale, centering, per_row, sink_keys (force_online is ignored here)
 *   out    caller-filled pointers; every other field is written
 *   workspace, workspace_bytes  device scratch of at least fm_bounds_workspace_size
 * Device results are deterministic (fixed-order reductions; key-sink ties broken by the
 * lower index).  Errors: FM_ERR_ARG (also sink_keys outside [0, FM_MAX_SINKS] or a missing
 * sink array), FM_ERR_SHAPE, FM_ERR_DTYPE, FM_ERR_UNSUPPORTED (also sinks with N_total
 * above 2^31 - 256), FM_ERR_CUDA. */
FM_API int fm_bounds(const fm_tensor *q, const fm_tensor *k_full, const fm_tensor *v_full,
              const fm_opts *opts, fm_bounds_out *out, void *workspace, size_t workspace_bytes,
              fm_stream_t stream);

/* fm_attn_chunk -- fold one KV chunk into the unnormalised fp32 accumulators
 * ([NKI] "A static bound makes the ring reduction pure addition", "Accumulate, then
 * normalize once").  For an eligible Q-block (flag = 1, force_online = 0) each row i
 * adds p_ij = 2^(alpha*q_i.k_j - shift_i) to acc_sum and p_ij*v_j to acc_o: pure
 * addition across chunks.  Other Q-blocks take the online-softmax fallback ([PR478]
 * "Cross-Ring Safety Fallback"): a running row max kept in acc_max, with rescaling.
 *   q        [B, H, Sq, D]   the same queries given to fm_bounds
 *   k_chunk  [B, H, Nc, D]   this chunk's keys (Nc >= 0, any Nc, ragged tails allowed)
 *   v_chunk  [B, H, Nc, D]
 *   bounds   from fm_bounds for this call; kv_seen/online_lock are updated
 *   acc_o    f32 [B, H, Sq, D] contiguous;  acc_sum, acc_max f32 [B, H, Sq] contiguous.
 *            acc_max holds each row's current base-2 shift (shift_i on fixed-m rows,
 *            the running max on fallback rows), so acc_sum * 2^acc_max is the
 *            row's sum of 2^z.
 *   accumulate  0: overwrite the accumulators (first chunk); 1: add into them
 * Key sinks (bounds->n_sink > 0): a key whose global index is in bounds->sink_idx adds
 * nothing here.  The global index of a chunk's first key is bounds->next_key_offset when the
 * caller set it (chunks in any order, e.g. a ring's rotated order), else the number of keys
 * folded before it (bounds->kv_seen: chunks in the key order fm_bounds saw).
 * Errors: FM_ERR_BOUNDS_MISMATCH when bounds->magic is wrong, the bounds' shape is
 * not [B, H, ceil(Sq/128)], bounds->centered != opts->centering (raw-key bounds must
 * never pair with centered logits: [PR477] "matched pair"), the softmax scale
 * differs, more keys arrive than bounds->N_total (or, at the chunk's offset, lie past it),
 * force_online changes within a call,
 * opts->sink_keys differs from bounds->n_sink, or the sinks were already folded in
 * (accumulate = 1 after fm_fold_sinks); plus the errors of fm_bounds. */
FM_API int fm_attn_chunk(const fm_tensor *q, const fm_tensor *k_chunk, const fm_tensor *v_chunk,
                  fm_bounds_out *bounds, const fm_opts *opts, float *acc_o, float *acc_sum,
                  float *acc_max, int accumulate, fm_stream_t stream);

/* fm_attn_chunk_final -- fold the LAST KV chunk and normalise in the same pass ([NKI]
 * "The ring loop": the last step folds and normalises, so the output write hides behind
 * attention instead of running as a separate tail).  Same arguments and checks as
 * fm_attn_chunk, plus
 *   o_out  [B, H, Sq, D] FM_F32 or FM_BF16 (any strides): o = acc / max(acc_sum, 1e-37)
 *   lse    f32 [B, H, Sq] contiguous, or NULL: as written by fm_finalize_lse
 * acc_sum and acc_max are updated as by fm_attn_chunk; acc_o is NOT (its contents are
 * unspecified afterwards).  The result equals fm_attn_chunk followed by fm_finalize (or
 * fm_finalize_lse); the tensor-core kernel does both in one launch where the layout of
 * o_out allows 16-byte stores, otherwise the two steps run back to back.  With key sinks
 * the chunk is folded as by fm_attn_chunk, then one pass merges the sinks back and
 * normalises (the result of fm_fold_sinks followed by fm_finalize(_lse)). */
FM_API int fm_attn_chunk_final(const fm_tensor *q, const fm_tensor *k_chunk, const fm_tensor *v_chunk,
                               fm_bounds_out *bounds, const fm_opts *opts, float *acc_o, float *acc_sum,
                               float *acc_max, int accumulate, const fm_tensor *o_out, float *lse,
                               fm_stream_t stream);

/* fm_attn_chunks -- fold n_chunks consecutive KV chunks (1..FM_MAX_CHUNKS) in one pass, and
 * with o_out given normalise after the last one.  The result equals fm_attn_chunk on each
 * chunk in order (the first with `accumulate`, the rest adding), followed by fm_finalize /
 * fm_finalize_lse when o_out is given; acc_o is then left unspecified, as with
 * fm_attn_chunk_final.  On the tensor-core path one launch walks every chunk's key tiles
 * (each with its own ragged end) and O and the row sums stay on chip across the chunk
 * boundaries, as the accumulator stays resident for the whole ring in [NKI] ("A static
 * bound makes the ring reduction pure addition").  k_chunks / v_chunks: arrays of n_chunks
 * fm_tensor [B, H, Nc, D].  Errors: those of fm_attn_chunk_final, FM_ERR_ARG for n_chunks
 * outside [1, FM_MAX_CHUNKS]. */
#define FM_MAX_CHUNKS 8
FM_API int fm_attn_chunks(const fm_tensor *q, const fm_tensor *k_chunks, const fm_tensor *v_chunks,
                          int n_chunks, fm_bounds_out *bounds, const fm_opts *opts, float *acc_o,
                          float *acc_sum, float *acc_max, int accumulate, const fm_tensor *o_out,
                          float *lse, fm_stream_t stream);

/* fm_finalize -- o = acc_o / max(acc_sum, 1e-37) ([NKI] "Accumulate, then normalize
 * once": one divide, sum floored near the smallest fp32 normal).
 *   acc_o f32 [B, H, Sq, D] and acc_sum f32 [B, H, Sq], contiguous
 *   o_out [B, H, Sq, D] (its B, H, S, D give the shape), FM_F32 or FM_BF16, any strides
 * Errors: FM_ERR_ARG, FM_ERR_DTYPE, FM_ERR_CUDA. */
FM_API int fm_finalize(const float *acc_o, const float *acc_sum, const fm_tensor *o_out,
                fm_stream_t stream);

/* fm_finalize_lse -- fm_finalize that also writes each row's log-sum-exp of the scaled
 * scores, lse_i = ln(sum_j exp(softmax_scale * q_i.k_j)), for training and for merging
 * partial results ([NKI] Interface: with training the kernel also returns
 * lse = c_i + log(sum_exp)).  Since acc_max holds each row's base-2 shift on both paths,
 * lse_i = ln(2) * (acc_max_i + log2(acc_sum_i)); a row that saw no key gets -inf.
 *   acc_max f32 [B, H, Sq] contiguous (as left by fm_attn_chunk)
 *   lse     f32 [B, H, Sq] contiguous, written
 * Errors: those of fm_finalize. */
FM_API int fm_finalize_lse(const float *acc_o, const float *acc_sum, const float *acc_max,
                           const fm_tensor *o_out, float *lse, fm_stream_t stream);

/* fm_fold_sinks -- merge the key sinks that fm_bounds set aside back into the accumulators,
 * exactly, after the last chunk and before fm_finalize(_lse) ([NKI] "Adapting this kernel"
 * leaves the loudest keys out of the max reduction; this is how their terms still count).
 * For each row i, with z_s = alpha * q_i.k_s the raw base-2 logit of sink s (from
 * bounds->sink_k) and r_i = acc_max_i the row's current shift:
 *   r' = max(r_i, max_s z_s),  c = 2^(r_i - r'),
 *   acc_o_i = c * acc_o_i + sum_s 2^(z_s - r') v_s,  acc_sum_i = c * acc_sum_i + sum_s 2^(z_s - r'),
 *   acc_max_i = r'
 * (an online-softmax merge in fp32), so that acc_sum * 2^acc_max stays the row's sum of 2^z
 * and fm_finalize_lse stays valid.  A no-op when bounds->n_sink == 0.
 *   q, opts  as given to the chunks;  acc_o / acc_sum / acc_max  as left by the last chunk
 * Errors: FM_ERR_BOUNDS_MISMATCH (bounds not matching q or opts, no chunk folded yet, or the
 * sinks already folded), FM_ERR_ARG, FM_ERR_CUDA. */
FM_API int fm_fold_sinks(const fm_tensor *q, fm_bounds_out *bounds, const fm_opts *opts, float *acc_o,
                         float *acc_sum, float *acc_max, fm_stream_t stream);

/* fm_sync_status -- synchronise `stream`, then report and clear this GPU's device
 * error word: FM_ERR_TIMEOUT if a kernel gave up on a pipeline wait (its outputs are
 * then invalid), FM_ERR_INDEX if a debug build's index check failed (the library built with
 * -DFM_DEBUG: the chunk kernels check their epilogue accesses to the accumulators and o, skip
 * a failing one and record the first), FM_ERR_CUDA on an asynchronous CUDA error, else FM_OK. */
FM_API int fm_sync_status(fm_stream_t stream);

/* fm_probe_wait_timeout -- exercise the failure path of the kernels' bounded waits: one
 * thread waits on a barrier phase that nothing completes and gives up after timeout_ms
 * (1..10000), recording the failure in the device error word, so that the next
 * fm_sync_status returns FM_ERR_TIMEOUT (role 5) and clears it.  Nothing faults and the
 * context stays usable.  No counterpart in the pages: it tests the library's own failure
 * detection.  Errors: FM_ERR_ARG, FM_ERR_CUDA. */
FM_API int fm_probe_wait_timeout(unsigned int timeout_ms, fm_stream_t stream);

/* Message of the last failing call on this thread ("" if none).  Valid until the
 * thread's next fm_* call. */
FM_API const char *fm_last_error(void);

/* ABI version of this header: (major << 16) | minor.  1.2 added fm_opts.schedule,
 * fm_bounds_out.next_key_offset and the ring bounds calls. */
FM_API int fm_version(void);

/* ---- The bounds of a ring of ranks ---------------------------------------------------------
 * In a multi-GPU ring each rank keeps its own query rows and holds one shard of the keys and
 * values; the shards rotate through the ranks, so no rank ever sees all keys at once.  The bounds
 * still need ring-wide key statistics, and the pages exchange them once before the ring: the key
 * mean over real tokens reduced across the ring so every rank centers against the same mean
 * ([PR478] Summary, "Global Virtual K-Centering"), then one max-reduction of the per-head key
 * norms and the V maximum ([NKI] "Global key max"; [PR478] folds the centered key max and the V
 * max into one pmax).  The library computes each rank's part and combines the exchanged parts;
 * the caller moves the bytes with its own collectives:
 *   1. (centering only) fm_ring_key_sums(k_shard) -> ksum f32 [B, H, D], the shard's key sums;
 *      the caller all-reduces (sum) ksum over the ring;
 *   2. fm_bounds_local(q, k_shard, v_shard, key_offset, N_total, ksum) -> the query-side arrays
 *      of `out` and this rank's statistics block (fm_ring_stats_bytes bytes); the caller
 *      all-gathers the blocks, in rank order, into one buffer;
 *   3. fm_bounds_combine(stats_all, n_ranks) -> the rest of `out`: kmax_sq, vmax_sq, the key
 *      sinks, m, flag and shift, as fm_bounds would give over (q, every key, every value), up to
 *      the fp32 summation order of the key mean (m and flag can then differ only where U is
 *      within fp32 rounding of an integer or of the gate).
 * Every rank then folds the shards with fm_attn_chunk in ring order, setting
 * out->next_key_offset to each shard's global offset.  The statistics block holds, per head, the
 * shard's key max and, with key sinks, its sink_keys + 1 loudest keys (norm, global index, key
 * and value rows): the ring-wide loudest keys are among the union of those. */

/* Bytes of one rank's statistics block for q of [B, H, *, D] and opts.sink_keys.  Returns FM_OK. */
FM_API int fm_ring_stats_bytes(int64_t B, int64_t H, int64_t D, int sink_keys, size_t *bytes);

/* fm_ring_key_sums -- ksum[b,h,:] = sum of this rank's keys of (b, h) in fp32 (fixed order).
 *   k_shard [B, H, Nr, D];  ksum f32 [B, H, D] device, written;
 *   workspace of fm_bounds_workspace_size(B, H, Nr, D) bytes.
 * Errors: FM_ERR_ARG, FM_ERR_DTYPE, FM_ERR_UNSUPPORTED, FM_ERR_CUDA. */
FM_API int fm_ring_key_sums(const fm_tensor *k_shard, float *ksum, void *workspace, size_t workspace_bytes,
                            fm_stream_t stream);

/* fm_bounds_local -- this rank's part of the bounds.
 *   q        [B, H, Sq, D] this rank's queries
 *   k_shard, v_shard [B, H, Nr, D] its shard of the keys and values; key_offset = the global
 *            index of the shard's first key (0 <= key_offset, key_offset + Nr <= N_total)
 *   N_total  keys over every shard of the ring (C(N) is computed from it)
 *   ksum_total f32 [B, H, D]: the ring-wide key sums (step 1) when opts->centering, else NULL
 *   out      as for fm_bounds; the query-side arrays (qmax_sq, qkbar, kbar) are written here, the
 *            rest by fm_bounds_combine; out->magic becomes FM_BOUNDS_LOCAL_MAGIC
 *   stats    device buffer of fm_ring_stats_bytes bytes, written (16-byte aligned)
 *   workspace of fm_bounds_workspace_size(B, H, Nr, D) bytes
 * Errors: those of fm_bounds, FM_ERR_ARG for a bad key_offset / N_total or a missing ksum_total. */
FM_API int fm_bounds_local(const fm_tensor *q, const fm_tensor *k_shard, const fm_tensor *v_shard, int64_t key_offset,
                           int64_t N_total, const float *ksum_total, const fm_opts *opts, fm_bounds_out *out,
                           void *stats, void *workspace, size_t workspace_bytes, fm_stream_t stream);

/* fm_bounds_combine -- finish `out` from every rank's statistics block.
 *   stats_all  device buffer of n_ranks blocks of fm_ring_stats_bytes bytes, in rank order
 *   opts       the same opts as fm_bounds_local
 *   out        as left by fm_bounds_local on this rank; becomes ready for fm_attn_chunk
 * Errors: FM_ERR_BOUNDS_MISMATCH when out was not prepared by fm_bounds_local or opts differ,
 * FM_ERR_ARG, FM_ERR_CUDA. */
FM_API int fm_bounds_combine(const void *stats_all, int n_ranks, const fm_opts *opts, fm_bounds_out *out,
                             fm_stream_t stream);

/* ---- Whole forwards on host buffers --------------------------------------------------------
 * Device buffers of fm_attention_host, all owned by the caller: two sets of inputs and outputs,
 * which consecutive batches alternate between, and one set of accumulators, bounds and workspace,
 * which the batches reuse in order. */
typedef struct {
  fm_tensor q[2], k[2], v[2]; /* device, contiguous [B, H, Sq, D] / [B, H, N, D], the inputs' dtype */
  fm_tensor o[2];             /* device, contiguous [B, H, Sq, D], the outputs' dtype */
  float *acc_o, *acc_sum, *acc_max;
  fm_bounds_out *bounds;      /* host struct whose device arrays are set, as for fm_bounds */
  void *workspace;
  size_t workspace_bytes;
} fm_host_buffers;

/* fm_attention_host -- n_batches whole forwards whose inputs and outputs live in host memory.
 * For batch i: q_host[i], k_host[i], v_host[i] are copied to the device, the path runs
 * (fm_bounds, one fm_attn_chunk per chunk of chunk_lens, the last chunk fused with the
 * normalise), and o is copied back into o_host[i].  Batch i+1's upload and batch i-1's read-back
 * run on their own streams while batch i computes, so the copies hide behind the kernels (host
 * memory must be page-locked for that; pageable memory works but does not overlap).
 *   q_host, k_host, v_host, o_host  arrays of n_batches contiguous host tensors, shaped and typed
 *                  like the device buffers
 *   chunk_lens     n_chunks >= 1 key counts summing to N (the ring steps run one after another)
 *   streams        three caller-created streams: upload, compute, read-back
 * Returns when every output is in host memory.  Creates and destroys a few CUDA events; allocates
 * no device memory.  Errors: those of the calls it makes, FM_ERR_ARG / FM_ERR_SHAPE for buffers
 * that do not match, FM_ERR_UNSUPPORTED for non-contiguous ones. */
FM_API int fm_attention_host(const fm_tensor *q_host, const fm_tensor *k_host, const fm_tensor *v_host,
                             const fm_tensor *o_host, int n_batches, const int64_t *chunk_lens, int n_chunks,
                             const fm_opts *opts, const fm_host_buffers *dev, const fm_stream_t *streams);

/* Upper bound of the scratch fm_bounds_noalloc can use: 4 MiB.  That covers, at D = 128,
 * up to 74 heads of 75,600 keys (fm_bounds_workspace_size gives the exact need). */
#define FM_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

/* fm_bounds_noalloc -- fm_bounds for callers that cannot allocate device memory.
 * The pages have no counterpart to this call: it exists for callers whose device memory
 * is planned in full before they run (an inference engine that reserves its arena up
 * front and forbids allocation afterwards, a plug-in inside another framework's memory
 * pool) and for latency-critical streams that must not pay cudaMalloc's implicit device
 * synchronisation.  Same arguments and results as fm_bounds, minus the workspace: the
 * scratch lives in a file-scope device array of FM_NOALLOC_SCRATCH_BYTES inside libfm,
 * which every GPU that loads the library holds until the process exits.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library routine.
 *   - The first call on each device looks up the array's device address with that device
 *     current (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Every call shares the one array and it keeps the last call's contents; nothing in
 *     it needs to start at zero, since every slot the kernels read is written earlier in
 *     the same call.  Calls that overlap on the GPU (other streams, other threads) race
 *     on it: serialise them.
 * Errors: those of fm_bounds, plus FM_ERR_UNSUPPORTED when the problem needs more scratch
 * than FM_NOALLOC_SCRATCH_BYTES (nothing is enqueued then). */
FM_API int fm_bounds_noalloc(const fm_tensor *q, const fm_tensor *k_full, const fm_tensor *v_full,
                             const fm_opts *opts, fm_bounds_out *out, fm_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FM_H_ */
