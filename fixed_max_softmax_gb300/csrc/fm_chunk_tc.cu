// fm_chunk_tc.cu -- tensor-core chunk kernel of fixed-m attention (sm_103a).
//
// Folds one KV chunk into the fp32 accumulators for bf16 inputs with D = 128:
//   S = Q K^T             tcgen05.mma kind::f16, A = Q and B = K from swizzled shared
//                         memory (TMA), fp32 accumulator in tensor memory (TMEM)
//   P = 2^(alpha*S - b)   softmax warps: tcgen05.ld of S, FFMA + ex2, row sums in
//                         registers, bf16 P written back over S in TMEM (tcgen05.st)
//   O += P V              tcgen05.mma with A = P read from TMEM, B = V from shared memory
//   epilogue              O and the row sums are added into (or initialise) acc_o/acc_sum;
//                         for fixed-m tiles O goes through a swizzled shared-memory tile and a
//                         TMA reduce-add (store on the first chunk), so the SM never reads acc_o
// For an eligible Q-block the shift b_i (m + alpha*q_i.kbar, from fm_bounds) is fixed before the chunk starts,
// so there is no row max, no rescale of O and the cross-chunk merge is a pure add
// ("Kernel reference: ring_attention_const_max_fwd", sections "Dropping the online max
// buys a better layout", "A static bound makes the ring reduction pure addition",
// "Accumulate, then normalize once"; PR #477 Summary for m, the exp2 form and the
// virtual centering term applied in registers).  A Q-block that failed the gate runs
// online softmax in the same pipeline (PR #478, "Cross-Ring Safety Fallback"): its
// softmax warps keep a running row max, rescale O in TMEM when the max grows by more
// than 2^8 (lazy rescale: exact, since the final shift is whatever the running max is),
// and merge with the previous chunks through acc_max.  The running max starts from the
// previous chunks' shift, so a tile whose rows never move it adds O as plainly as a fixed-m
// tile.
// Key columns that must not count -- past a chunk's ragged end, or key sinks that the
// bounds pass left out of the key max ("Kernel reference: ring_attention_const_max_fwd",
// section "Adapting this kernel") -- get -inf written over their scores in TMEM before the
// softmax reads them, so they give p = 0 with no masks in the per-element code.
//
// CTA = two 128-row Q tiles of one (batch, head) (256 rows) against every KV tile of the
// launch: one chunk, or several consecutive chunks (up to 8), whose key tiles are walked in
// order with each chunk's own tensor maps and ragged end, so that O and the row sums stay
// on chip across the chunk boundaries.  (fm_chunk_tc_persistent_kernel is the same pipeline
// with each CTA walking several such work items.)  12 warps:
//   warp 0      TMA producer: Q tiles once, then K_j, V_j into a 5-stage ring
//   warp 1      TMEM allocator; lane 0 issues every MMA and commit
//   warps 4-7   softmax + epilogue of Q tile 0 (TMEM lanes 0-127)
//   warps 8-11  softmax + epilogue of Q tile 1
// TMEM (512 columns): S0/P0 [0,128) S1/P1 [128,256) O0 [256,384) O1 [384,512).
// MMA issue order per KV tile j:  S0(j), PV1(j-1), S1(j), PV0(j) -- each softmax group
// works on its tile while the tensor core runs the other group's two MMAs.
// Every wait on an mbarrier is bounded in time; on expiry the kernel records the failure
// in the device error word, waits (bounded) for its own copies and MMAs, frees TMEM and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <limits.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#include <mutex>

#include "fm_internal.h"

namespace fm {
namespace {

constexpr int kBQ = 128;   // rows per Q tile = TMEM lanes
constexpr int kBK = 128;   // keys per KV tile
constexpr int kHD = 128;   // head dimension
constexpr int kStages = 5; // K/V ring: K_j in stage (2j)%5, V_j in stage (2j+1)%5
constexpr int kTileBytes = kBK * kHD * 2;     // 32 KiB
constexpr int kPanelBytes = 128 * 64 * 2;     // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr float kLazyRescale = 8.0f;          // online path: rescale when the max grows by > 2^8

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffKV = 2 * kTileBytes;
constexpr int kOffBar = kOffKV + kStages * kTileBytes;
constexpr int kBarQFull = 0;  // + t: Q tile t has landed
constexpr int kBarKVFull = 2;
constexpr int kBarKVEmpty = kBarKVFull + kStages;
constexpr int kBarSFull = kBarKVEmpty + kStages;
constexpr int kBarPReady = kBarSFull + 2;
constexpr int kBarODone = kBarPReady + 2;
constexpr int kBarDrain = kBarODone + 2;
constexpr int kBarQEmpty = kBarDrain + 1;  // every S MMA of an item has read Q
constexpr int kNumBars = kBarQEmpty + 1;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kOffSinks = kOffAbort + 8;  // per softmax group: its item's key sinks (FM_MAX_SINKS int32)
constexpr int kSmemUsed = kOffSinks + 2 * 4 * FM_MAX_SINKS;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base
// The persistent kernel's K/V ring has one stage fewer; the fifth stage's space holds each softmax
// group's 16 KiB box of O on its way to the bulk reduce.
constexpr int kPStages = kStages - 1;
constexpr int kOffPStage = kOffKV + kPStages * kTileBytes;
constexpr int kBoxBytes = kBQ * 128;  // 32 fp32 columns x 128 rows

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits 4-5 = 1),
// A and B bf16 (bits 7-9 = 1, bits 10-12 = 1), A K-major, B K-major (bit 16 = 0) or
// MN-major (bit 16 = 1), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdescQK = idesc_bf16(kBQ, kBK, false);  // S = Q K^T: K is [keys, D], K-major
constexpr uint32_t kIdescPV = idesc_bf16(kBQ, kHD, true);   // O = P V:   V is [keys, D], MN-major

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
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
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Slow path of wait_phase: poll until the phase completes, the time limit passes or, if
// `abort_flag` is given, another role of the CTA has already given up.  On expiry the
// first failing wait of the launch records itself in err[0..5]: role code, `tag`
// (barrier index << 16 | tile index j), block x, y, z and thread, and raises the CTA's
// abort flag.
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             unsigned long long timeout_ns, unsigned int *err,
                                             unsigned int code, unsigned int tag) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 31) == 0) {
      if (abort_flag && *abort_flag) return false;
      if (globaltimer() - t0 > timeout_ns) {
        if (abort_flag) *abort_flag = 1;
        if (atomicCAS(err, 0u, code) == 0u) {
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
// Wait for the phase of `bar` with parity `parity`; false when the wait gave up.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           unsigned long long timeout_ns, unsigned int *err,
                                           unsigned int code, unsigned int tag = 0) {
  if (mbar_test(bar, parity)) return true;
  return wait_phase_slow(bar, parity, abort_flag, timeout_ns, err, code, tag);
}
__device__ __forceinline__ unsigned int wtag(int bar_index, int j) {
  return ((unsigned int)bar_index << 16) | ((unsigned int)j & 0xFFFFu);
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *tm, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// L2 eviction priorities for bulk copies (createpolicy): evict_last for data read again soon
// (an accumulator that the next chunk adds into, when it fits in L2), evict_first for data
// read once (a Q tile of the persistent schedule).
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap *tm, uint32_t bar, int c0, int c1,
                                                 int c2, int c3, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(pol)
      : "memory");
}

// O of one Q tile from shared memory into the fp32 accumulator (3-D map over [B*H, Sq, D]):
// added to it (reduce) or written over it (store), with the L2 priority `pol`.  Rows past Sq
// are clipped by the map.
__device__ __forceinline__ void tma_acc_3d(const CUtensorMap *tm, uint32_t src, int c0, int c1, int c2, bool add,
                                           uint64_t pol) {
  if (add)
    asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group.L2::cache_hint"
                 " [%0, {%2, %3, %4}], [%1], %5;" ::"l"(reinterpret_cast<uint64_t>(tm)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
                 : "memory");
  else
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group.L2::cache_hint"
                 " [%0, {%2, %3, %4}], [%1], %5;" ::"l"(reinterpret_cast<uint64_t>(tm)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
                 : "memory");
}
// acc += v (4 consecutive fp32) as one reduction in the memory system: the same fp32 add
// as the registers would do, without reading the accumulator through the SM.
__device__ __forceinline__ void red_add_v4(float *dst, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
// Commit the bulk operations issued so far and wait until they have read their shared-memory
// source, so that it may be reused or released; their global writes complete with the grid,
// before the next kernel in the stream (or its griddepcontrol.wait) proceeds.
__device__ __forceinline__ void bulk_commit_and_wait_smem_read() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Shared-memory writes of this thread become visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier over `count` threads that also returns the AND of their `v`.
__device__ __forceinline__ bool named_barrier_and(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pin, pout;\n\t"
      "setp.ne.u32 pin, %1, 0;\n\t"
      "bar.red.and.pred pout, %2, %3, pin;\n\t"
      "selp.u32 %0, 1, 0, pout;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Shared-memory matrix descriptor: start, leading and stride byte offsets (>> 4), the
// fixed version bits (46-48 = 0b001) and the 128-byte swizzle mode (bits 61-63 = 2).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
         ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

#define FM_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                 "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
// 32 consecutive 32-bit TMEM columns of this thread's lane, waited for.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FM_R8(0), FM_R8(8), FM_R8(16), FM_R8(24)
      : "r"(taddr)
      : "memory");
}
// 16 columns of this warp's 32 TMEM lanes (one fp32 column per register), waited for.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FM_R8(0), FM_R8(8)
      : "r"(taddr)
      : "memory");
}
// The same load without waiting: the registers are valid only after tmem_ld_wait(r).
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : FM_R8(0), FM_R8(8), FM_R8(16), FM_R8(24)
      : "r"(taddr)
      : "memory");
}
#undef FM_R8
#define FM_W8(i) "+r"(r[i + 0]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), \
                 "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
// Wait for this thread's TMEM loads.  `r` (the destination of the last one) passes through
// the instruction, so the compiler cannot schedule a use of it before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : FM_W8(0), FM_W8(8), FM_W8(16), FM_W8(24) : : "memory");
}
// Ties `r` (the destination of an earlier load covered by a tmem_ld_wait just before)
// to this point, so that no use of it is scheduled above that wait.
__device__ __forceinline__ void tmem_reg_tie(uint32_t (&r)[32]) {
  asm volatile("" : FM_W8(0), FM_W8(8), FM_W8(16), FM_W8(24) : : "memory");
}
#undef FM_W8
// Two fp32 lanes in one 64-bit register (Blackwell's packed fp32x2 arithmetic).
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
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
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// two fp32 -> one bf16x2 word, `lo` in the low half (the lower column index)
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The lane index, read where it is used: arithmetic on it cannot be hoisted out of an enclosing
// loop (IN_LOOP: the epilogue helpers run once per item inside the persistent kernel's item
// loop, and their lane-dependent addresses would otherwise stay live across every key tile).
__device__ __forceinline__ int opaque_laneid() {
  int l;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

// What the debug build (FM_DEBUG) checks a warp's epilogue accesses against; unused otherwise:
// the flat row index of the warp's first row over [B, H, Sq], the rows of the accumulators, the
// offset of the warp's first row of o and the span of o, in elements.
struct EpiCheck {
  unsigned int *err;
  int64_t flat0, rows, out_off0, out_span;
};

// O of one warp's 32 rows (its TMEM lane quarter) into the fp32 accumulator, added (red) or
// stored, without reading it through the SM: each 32-column piece goes from TMEM through the
// warp's own 4 KiB of shared memory (32 rows x 128 bytes, 16-byte chunks XOR-swizzled by row,
// so that neither the row-wise writes nor the chunk-wise reads conflict on banks), so that each
// global access covers four whole 128-byte row pieces.  The reductions are posted, not waited
// for: the warp moves on while the memory system applies them.  row0 is the warp's first row and
// acc_row0 its accumulator row; rows at or past Sq are left out.
template <bool IN_LOOP = false>
__device__ __forceinline__ void o_to_acc_warp(uint8_t *slab, uint32_t tO, int lane, bool tile_ok, int64_t row0,
                                              int64_t Sq, float *acc_row0, bool add, EpiCheck ck) {
  if constexpr (IN_LOOP) lane = opaque_laneid();
  const int ch = lane & 7;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t o[32];
    tmem_ld32(tO + c * 32, o);
    uint8_t *line = slab + lane * 128;
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4)
      *reinterpret_cast<uint4 *>(line + ((q4 ^ (lane & 7)) << 4)) =
          make_uint4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = i * 4 + (lane >> 3);
      const uint4 v = *reinterpret_cast<const uint4 *>(slab + rr * 128 + ((ch ^ (rr & 7)) << 4));
      if (tile_ok && row0 + rr < Sq && FM_DCHECK(ck.flat0 + rr < ck.rows, ck.err, 1u, ck.flat0 + rr)) {
        float *dst = acc_row0 + rr * kHD + c * 32 + ch * 4;
        if (add) red_add_v4(dst, v.x, v.y, v.z, v.w);
        else *reinterpret_cast<uint4 *>(dst) = v;
      }
    }
    __syncwarp();  // the slab is read before the next piece overwrites it
  }
}

constexpr int kMaxChunks = FM_MAX_CHUNKS;  // consecutive KV chunks one launch can fold

// Tensor maps of Q and of each chunk's K and V (kernel parameter space).
struct TcMaps {
  CUtensorMap acc;  // fp32 accumulator [B*H, Sq, D], box 32 x 128 rows (valid when acc_tma)
  CUtensorMap q;
  CUtensorMap k[kMaxChunks];
  CUtensorMap v[kMaxChunks];
};

struct TcParams {
  int64_t Sq, nqb;
  int H, n_kv;                      // n_kv: key tiles over all chunks of the launch
  int n_chunks;
  int tile0[kMaxChunks + 1];        // first key tile of each chunk (prefix sums)
  int len[kMaxChunks];              // keys in each chunk
  float alpha;
  int force_online, accumulate;
  const uint8_t *flag;
  const float *shift;
  float *acc_o, *acc_sum, *acc_max;
  unsigned int *err;
  unsigned long long timeout_ns;
  // fused normalise of the last chunk: out != nullptr selects it
  void *out;
  int out_bf16;
  int64_t osB, osH, osS;
  float *lse;
  // key sinks to skip: [B,H,FM_MAX_SINKS] ascending global key indices (INT_MAX pads), or
  // nullptr; key0[c] is the global index of chunk c's first key
  const int32_t *sinks;
  int key0[kMaxChunks];
  // the persistent schedule's epilogue of a chunk that is not the last stages O in shared
  // memory and adds it into (or stores it over) acc_o with one bulk tensor operation per 32
  // columns, with L2 priority evict_last when acc_keep (the accumulator fits in L2)
  int acc_tma, acc_keep;
  // persistent schedule: each CTA walks work items (batch, head, Q-tile pair) item =
  // blockIdx.x, blockIdx.x + gridDim.x, ...; otherwise one item per CTA of a
  // (pairs, H, B) grid.  n_items = B * H * pairs.
  int persistent;
  int64_t n_items, n_pairs;
  // persistent schedule: CTAs x >= n_items mod gridDim.x, which have one item fewer than the
  // others, start (x - that) * stagger_ns later (0: no stagger)
  unsigned long long stagger_ns;
  // debug builds: the accumulator rows (B*H*Sq) and the span of `out` in elements that the
  // epilogue's index checks compare against
  int64_t dbg_rows, dbg_out_span;
};

// The epilogue that reads the accumulator, for one warp's 32 rows: x = acc + O on fixed-m rows,
// x = acc*cprev + O*cnew on online rows (x = O when !rd), then either acc = x (out == nullptr)
// or o = x * inv into `out` (bf16 or fp32; with the normalise fused in).  cprev, cnew and inv
// are this lane's row's.  As in o_to_acc_warp, every global access covers whole row pieces.
// Per 32-column piece, through the warp's 4 KiB of shared memory (32 rows x 128 bytes, 16-byte
// chunks XOR-swizzled by row):
//   1. the rows' accumulator piece comes in four rows of 128 bytes per load (the next piece's
//      loads are in flight while this one is combined) and is parked in the rows;
//   2. each lane combines its own row with O from TMEM and writes the result back into its own
//      row (fp32 in place; bf16 into the even chunks), so no lane touches another's row here;
//   3. the rows go out four (fp32) or eight (bf16) to a store.
// acc_row0 / out_row0 are the warp's first row (row0); rows at or past Sq are neither read nor
// written.
template <bool IN_LOOP = false>
__device__ __forceinline__ void acc_merge_warp(uint8_t *slab, uint32_t tO, int lane, bool tile_ok, int64_t row0,
                                               int64_t Sq, float *acc_row0, bool rd, bool fixed, float cprev,
                                               float cnew, float inv, void *out_row0, int64_t osS, bool out_bf16,
                                               EpiCheck ck) {
  if constexpr (IN_LOOP) lane = opaque_laneid();
  const int ch = lane & 7;
  const int nrows = tile_ok ? (int)max((int64_t)0, min((int64_t)32, Sq - row0)) : 0;  // valid rows of the warp
  const bool final_out = out_row0 != nullptr;
  const bool bf16_out = final_out && out_bf16;
  // this lane's row and chunk in the whole-row layout: rows lane / 8 + 4 i, 16-byte chunk lane % 8
  const float *acc_lane = acc_row0 + (lane >> 3) * kHD + ch * 4;
  uint8_t *own = slab + lane * 128;  // this lane's row
  const int sw = lane & 7;
  uint4 nxt[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    nxt[i] = (rd && i * 4 + (lane >> 3) < nrows &&
              FM_DCHECK(ck.flat0 + i * 4 + (lane >> 3) < ck.rows, ck.err, 2u, ck.flat0 + i * 4 + (lane >> 3)))
                 ? __ldcg(reinterpret_cast<const uint4 *>(acc_lane + i * 4 * kHD))
                 : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = i * 4 + (lane >> 3);
      *reinterpret_cast<uint4 *>(slab + rr * 128 + ((ch ^ (rr & 7)) << 4)) = nxt[i];
    }
    __syncwarp();
    if (c < 3) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        nxt[i] = (rd && i * 4 + (lane >> 3) < nrows &&
                  FM_DCHECK(ck.flat0 + i * 4 + (lane >> 3) < ck.rows, ck.err, 2u, ck.flat0 + i * 4 + (lane >> 3)))
                     ? __ldcg(reinterpret_cast<const uint4 *>(acc_lane + i * 4 * kHD + (c + 1) * 32))
                     : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t o[16];  // O in two 16-column halves
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if ((q & 1) == 0) tmem_ld16(tO + c * 32 + q * 8, o);
      float x[8];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint4 yy = *reinterpret_cast<const uint4 *>(own + (((2 * q + hh) ^ sw) << 4));
        const float yv[4] = {__uint_as_float(yy.x), __uint_as_float(yy.y), __uint_as_float(yy.z), __uint_as_float(yy.w)};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float ov = __uint_as_float(o[8 * (q & 1) + 4 * hh + e]);
          x[4 * hh + e] = !rd ? ov : (fixed ? ov + yv[e] : fmaf(yv[e], cprev, ov * cnew));
        }
      }
      if (bf16_out) {
        *reinterpret_cast<uint4 *>(own + (((2 * q) ^ sw) << 4)) =
            make_uint4(pack_bf16(x[0] * inv, x[1] * inv), pack_bf16(x[2] * inv, x[3] * inv),
                       pack_bf16(x[4] * inv, x[5] * inv), pack_bf16(x[6] * inv, x[7] * inv));
      } else {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float *xv = x + 4 * hh;
          *reinterpret_cast<uint4 *>(own + (((2 * q + hh) ^ sw) << 4)) =
              final_out ? make_uint4(__float_as_uint(xv[0] * inv), __float_as_uint(xv[1] * inv),
                                     __float_as_uint(xv[2] * inv), __float_as_uint(xv[3] * inv))
                        : make_uint4(__float_as_uint(xv[0]), __float_as_uint(xv[1]), __float_as_uint(xv[2]),
                                     __float_as_uint(xv[3]));
        }
      }
    }
    __syncwarp();
    if (bf16_out) {
      // 64 bytes per row piece in its even chunks: eight rows per store
      const int c4 = lane & 3;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = i * 8 + (lane >> 2);
        const uint4 v = *reinterpret_cast<const uint4 *>(slab + rr * 128 + (((2 * c4) ^ (rr & 7)) << 4));
        if (rr < nrows && FM_DCHECK(ck.out_off0 + rr * osS + c * 32 + c4 * 8 + 7 < ck.out_span, ck.err, 4u,
                                    ck.out_off0 + rr * osS + c * 32 + c4 * 8))
          *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(out_row0) + rr * osS + c * 32 + c4 * 8) = v;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = i * 4 + (lane >> 3);
        const uint4 v = *reinterpret_cast<const uint4 *>(slab + rr * 128 + ((ch ^ (rr & 7)) << 4));
        if (rr < nrows &&
            (final_out ? FM_DCHECK(ck.out_off0 + rr * osS + c * 32 + ch * 4 + 3 < ck.out_span, ck.err, 4u,
                                   ck.out_off0 + rr * osS + c * 32 + ch * 4)
                       : FM_DCHECK(ck.flat0 + rr < ck.rows, ck.err, 3u, ck.flat0 + rr))) {
          float *dst = final_out ? reinterpret_cast<float *>(out_row0) + rr * osS + c * 32 + ch * 4
                                 : acc_row0 + rr * kHD + c * 32 + ch * 4;
          *reinterpret_cast<uint4 *>(dst) = v;
        }
      }
    }
    __syncwarp();  // the slab is read before the next piece overwrites it
  }
}

// p = 2^(alpha*s - bias) for 32 scores of one full chunk, two at a time with fp32x2 FMA and
// adds; the row sum goes to two pair accumulators, P to 16 bf16x2 words pk[OFF..OFF+16).
template <int OFF, int NPK>
__device__ __forceinline__ void exp_chunk_full(const uint32_t (&s)[32], uint64_t a2, uint64_t nb2, uint64_t &acc0,
                                               uint64_t &acc1, uint32_t (&pk)[NPK]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    float z0, z1;
    f2_unpack(f2_fma(f2_pack(s[2 * e], s[2 * e + 1]), a2, nb2), z0, z1);
    const float p0 = ex2(z0), p1 = ex2(z1);
    const uint64_t pp = f2_pack(__float_as_uint(p0), __float_as_uint(p1));
    if (e & 1) acc1 = f2_add(acc1, pp); else acc0 = f2_add(acc0, pp);
    pk[OFF + e] = pack_bf16(p0, p1);
  }
}

// The smallest key sink of the head's list (in shared memory: ascending int32, INT_MAX
// pads) above `g`, or INT_MAX.
__device__ __forceinline__ int sink_after_key(const int32_t *ssk, int g) {
  int n = INT_MAX;
#pragma unroll
  for (int t = 0; t < FM_MAX_SINKS; ++t)
    if (ssk[t] > g) n = min(n, ssk[t]);
  return n;
}

// Which of a tile's 128 key columns count: the first nvalid (the rest lie past the chunk's
// end) minus the key sinks whose global index falls in the tile.  `next_sink` is the
// smallest sink index not yet passed (INT_MAX when there is none).
__device__ __forceinline__ uint32_t first_bits(int n) {
  return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
}
// Write -inf over the scores of those columns in TMEM, so that the softmax that follows
// gives them p = 2^-inf = 0 (and leaves them out of the online row max) with no masks of
// its own.  Only for the rare tiles that have such columns; warp-uniform, like every
// tcgen05.ld/st (all rows of a tile share its key columns).
__device__ __noinline__ void mask_tile(uint32_t tS, int nvalid, int g0, const int32_t *ssk, int &next_sink) {
  uint32_t k0 = first_bits(nvalid), k1 = first_bits(nvalid - 32), k2 = first_bits(nvalid - 64),
           k3 = first_bits(nvalid - 96);
  while (next_sink < g0 + nvalid) {
    const int col = next_sink - g0;
    const uint32_t bit = ~(1u << (col & 31));
    const int w = col >> 5;
    k0 &= w == 0 ? bit : 0xffffffffu;
    k1 &= w == 1 ? bit : 0xffffffffu;
    k2 &= w == 2 ? bit : 0xffffffffu;
    k3 &= w == 3 ? bit : 0xffffffffu;
    next_sink = sink_after_key(ssk, next_sink);
  }
  const uint32_t keep[4] = {k0, k1, k2, k3};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (keep[c] == 0xffffffffu) continue;
    uint32_t sc[32];
    tmem_ld32(tS + 32 * c, sc);
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (!((keep[c] >> e) & 1u)) sc[e] = 0xff800000u;  // -inf
    tmem_st32(tS + 32 * c, sc);
  }
  tmem_st_wait();
}

// Fixed-m softmax of one 128x128 S tile for this thread's row; P overwrites S.  The four
// 32-column TMEM loads are double-buffered: chunk c+1 is in flight while chunk c is
// exponentiated.  Key columns to leave out hold -inf (mask_tile) and give p = 0.  P leaves in
// 16-column stores, one per chunk, or with WIDE (the fixed-m tile loop, which has the
// registers) in one 32-column store per 64 keys: fewer TMEM stores, measured faster there.
template <bool WIDE>
__device__ __forceinline__ void softmax_fixed_tile(uint32_t tS, float alpha, float nbias, float (&l)[4]) {
  constexpr int NPK = WIDE ? 32 : 16;
  uint32_t sa[32], sb[32];
  uint32_t pk[NPK];
  tmem_ld32_async(tS, sa);
  tmem_ld_wait(sa);
  const uint64_t a2 = f2_pack(__float_as_uint(alpha), __float_as_uint(alpha));
  const uint64_t nb2 = f2_pack(__float_as_uint(nbias), __float_as_uint(nbias));
  uint64_t acc0 = 0, acc1 = 0;  // +0.0f pairs
  // P columns [16c, 16c+16) of chunk c lie in S columns already read
  tmem_ld32_async(tS + 32, sb);
  exp_chunk_full<0>(sa, a2, nb2, acc0, acc1, pk);
  if constexpr (!WIDE) tmem_st16(tS + 0, pk);
  tmem_ld_wait(sb);
  tmem_ld32_async(tS + 64, sa);
  if constexpr (WIDE) {
    exp_chunk_full<16>(sb, a2, nb2, acc0, acc1, pk);
    tmem_st32(tS + 0, pk);
  } else {
    exp_chunk_full<0>(sb, a2, nb2, acc0, acc1, pk);
    tmem_st16(tS + 16, pk);
  }
  tmem_ld_wait(sa);
  tmem_ld32_async(tS + 96, sb);
  exp_chunk_full<0>(sa, a2, nb2, acc0, acc1, pk);
  if constexpr (!WIDE) tmem_st16(tS + 32, pk);
  tmem_ld_wait(sb);
  if constexpr (WIDE) {
    exp_chunk_full<16>(sb, a2, nb2, acc0, acc1, pk);
    tmem_st32(tS + 32, pk);
  } else {
    exp_chunk_full<0>(sb, a2, nb2, acc0, acc1, pk);
    tmem_st16(tS + 48, pk);
  }
  float x0, x1, y0, y1;
  f2_unpack(acc0, x0, x1);
  f2_unpack(acc1, y0, y1);
  l[0] += x0;
  l[1] += x1;
  l[2] += y0;
  l[3] += y1;
}

// max(a, b, c) in one instruction (the three-input form of max.f32; a NaN operand is ignored,
// as fmaxf does).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// The max of 64 scores in four independent chains (one chain would put every max
// operation on the tile's critical path), two new scores per instruction.
__device__ __forceinline__ float max64(const uint32_t (&a)[32], const uint32_t (&b)[32], float mx) {
  float m0 = mx, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    m0 = max3f(m0, __uint_as_float(a[e]), __uint_as_float(a[e + 2]));
    m1 = max3f(m1, __uint_as_float(a[e + 1]), __uint_as_float(a[e + 3]));
    m2 = max3f(m2, __uint_as_float(b[e]), __uint_as_float(b[e + 2]));
    m3 = max3f(m3, __uint_as_float(b[e + 1]), __uint_as_float(b[e + 3]));
  }
  return max3f(m0, m1, fmaxf(m2, m3));
}

// Online softmax of one S tile for this thread's row, in two passes over TMEM: the first
// takes the row max of the 128 scores (two column halves, 64 registers), the second
// exponentiates exactly like the fixed-m tile (double-buffered 32-column loads) with the
// running max as the shift.  The tile max updates the running max `run` (base-2 units)
// lazily: only when it grows by more than 2^8, or on the first tile.  The row sum is
// rescaled before the new terms are added, and O in TMEM after P is out.  The rescale
// decision is per row but tcgen05.ld/st are warp-collective, so the warp rescales when any
// of its rows needs it and the other rows use a scale of 1.  Columns to leave out (past the
// chunk's end, key sinks) hold -inf (mask_tile): they drop out of the max and give p = 0;
// while every key so far was left out, run stays -inf and the shift used is 0.
__device__ __forceinline__ void softmax_online_tile(uint32_t tS, uint32_t tO, float alpha, bool have_o, float &run,
                                                    float (&l)[4]) {
  float mx;
  {
    uint32_t sa[32], sb[32];
    tmem_ld32_async(tS, sa);
    tmem_ld32_async(tS + 32, sb);
    tmem_ld_wait(sa);
    tmem_reg_tie(sb);
    mx = max64(sa, sb, -INFINITY);
    tmem_ld32_async(tS + 64, sa);
    tmem_ld32_async(tS + 96, sb);
    tmem_ld_wait(sa);
    tmem_reg_tie(sb);
    mx = max64(sa, sb, mx);
  }
  const float zmax = mx * alpha;
  const bool need = run == -INFINITY || zmax > run + kLazyRescale;
  const bool any = __any_sync(0xffffffffu, need);
  float sc = 1.0f;
  if (any) {
    const float nr = need ? fmaxf(run, zmax) : run;
    // O holds earlier tiles only when j > 0, and nothing but zeros while run is -inf
    if (have_o && need) sc = run == -INFINITY ? 0.f : ex2(run - nr);
    run = nr;
#pragma unroll
    for (int i = 0; i < 4; ++i) l[i] *= sc;
  }
  softmax_fixed_tile<false>(tS, alpha, run == -INFINITY ? 0.f : -run, l);
  if (any && have_o) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + c * 32, o);
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * sc);
      tmem_st32(tO + c * 32, o);
    }
  }
}

// One CTA per work item (grid (pairs, H, B)): the schedule every launch takes unless the
// persistent one is asked for.
__global__ void __launch_bounds__(kThreads, 1)
    fm_chunk_tc_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
  pdl_wait();  // bounds and accumulators written by the kernels before this one
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + kOffAbort);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kOffTmemSlot);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, h = blockIdx.y;
  const int64_t qb0 = 2 * (int64_t)blockIdx.x;
  auto bar = [&](int i) -> uint32_t { return base + (uint32_t)(kOffBar + 8 * i); };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(kBarQFull + 0), 1);
    mbar_init(bar(kBarQFull + 1), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKVFull + s), 1);
      mbar_init(bar(kBarKVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarPReady + t), 128);
      mbar_init(bar(kBarODone + t), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    fence_mbar_init();
    int32_t *ssk = reinterpret_cast<int32_t *>(gbase + kOffSinks);
    for (int t = 0; t < FM_MAX_SINKS; ++t)
      ssk[t] = p.sinks ? p.sinks[((int64_t)b * p.H + h) * FM_MAX_SINKS + t] : INT_MAX;
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_kv = p.n_kv;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int last_round[kStages];
      for (int s = 0; s < kStages; ++s) last_round[s] = -1;
      // one barrier per Q tile, so that S0 can start before tile 1 has landed
      for (int t = 0; t < 2; ++t) {
        mbar_expect_tx(bar(kBarQFull + t), 2 * kPanelBytes);
        for (int pn = 0; pn < 2; ++pn)
          tma_load_4d(base + kOffQ + t * kTileBytes + pn * kPanelBytes, &maps.q, bar(kBarQFull + t), pn * 64,
                      (int)((qb0 + t) * kBQ), h, b);
      }
      bool ok = true;
      int c = 0;  // chunk of key tile j
      for (int j = 0; j < n_kv && ok; ++j) {
        while (j >= p.tile0[c + 1]) ++c;
        const int jl = j - p.tile0[c];  // tile within its chunk
        for (int w = 0; w < 2 && ok; ++w) {
          const int idx = 2 * j + w, s = idx % kStages, round = idx / kStages;
          ok = wait_phase(bar(kBarKVEmpty + s), (uint32_t)((round & 1) ^ 1), abort_flag, p.timeout_ns, p.err,
                          kDevErrTimeoutProducer, wtag(kBarKVEmpty + s, j));
          if (!ok) break;
          mbar_expect_tx(bar(kBarKVFull + s), kTileBytes);
          const CUtensorMap *tm = w ? &maps.v[c] : &maps.k[c];
          for (int pn = 0; pn < 2; ++pn)
            tma_load_4d(base + kOffKV + s * kTileBytes + pn * kPanelBytes, tm, bar(kBarKVFull + s), pn * 64,
                        jl * kBK, h, b);
          last_round[s] = round;
        }
      }
      if (!ok) {
        // let every copy already issued land before the CTA can exit
        for (int t = 0; t < 2; ++t)
          wait_phase(bar(kBarQFull + t), 0, nullptr, p.timeout_ns, p.err, kDevErrTimeoutDrain, wtag(kBarQFull + t, 0));
        for (int s = 0; s < kStages; ++s)
          if (last_round[s] >= 0)
            wait_phase(bar(kBarKVFull + s), (uint32_t)(last_round[s] & 1), nullptr, p.timeout_ns, p.err,
                       kDevErrTimeoutDrain, wtag(kBarKVFull + s, 0));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t tS0 = tmem + 0, tS1 = tmem + 128, tO0 = tmem + 256, tO1 = tmem + 384;
      auto q_desc = [&](int t, int kk) {
        return smem_desc(base + kOffQ + t * kTileBytes + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
      };
      auto k_desc = [&](int s, int kk) {
        return smem_desc(base + kOffKV + s * kTileBytes + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
      };
      auto v_desc = [&](int s, int kk) {
        return smem_desc(base + kOffKV + s * kTileBytes + kk * 2048, kPanelBytes, 1024);
      };
      bool ok = wait_phase(bar(kBarQFull + 0), 0, abort_flag, p.timeout_ns, p.err, kDevErrTimeoutMma,
                           wtag(kBarQFull + 0, 0));
      int vs_prev = 0;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int ki = 2 * j, ks = ki % kStages;
        ok = wait_phase(bar(kBarKVFull + ks), (uint32_t)((ki / kStages) & 1), abort_flag, p.timeout_ns, p.err,
                        kDevErrTimeoutMma, wtag(kBarKVFull + ks, j));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tS0, q_desc(0, kk), k_desc(ks, kk), kIdescQK, kk > 0);
        mma_commit(bar(kBarSFull + 0));
        if (j > 0) {
          ok = wait_phase(bar(kBarPReady + 1), (uint32_t)((j - 1) & 1), abort_flag, p.timeout_ns, p.err,
                          kDevErrTimeoutMma, wtag(kBarPReady + 1, j));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tO1, tS1 + kk * 8, v_desc(vs_prev, kk), kIdescPV, (j - 1 > 0 || kk > 0));
          mma_commit(bar(kBarKVEmpty + vs_prev));
        }
        if (j == 0) {  // Q tile 1 may land after tile 0
          ok = wait_phase(bar(kBarQFull + 1), 0, abort_flag, p.timeout_ns, p.err, kDevErrTimeoutMma,
                          wtag(kBarQFull + 1, 0));
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tS1, q_desc(1, kk), k_desc(ks, kk), kIdescQK, kk > 0);
        mma_commit(bar(kBarSFull + 1));
        mma_commit(bar(kBarKVEmpty + ks));
        const int vi = 2 * j + 1, vs = vi % kStages;
        ok = wait_phase(bar(kBarKVFull + vs), (uint32_t)((vi / kStages) & 1), abort_flag, p.timeout_ns, p.err,
                        kDevErrTimeoutMma, wtag(kBarKVFull + vs, j)) &&
             wait_phase(bar(kBarPReady + 0), (uint32_t)(j & 1), abort_flag, p.timeout_ns, p.err,
                        kDevErrTimeoutMma, wtag(kBarPReady + 0, j));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ts(tO0, tS0 + kk * 8, v_desc(vs, kk), kIdescPV, (j > 0 || kk > 0));
        if (j == n_kv - 1) mma_commit(bar(kBarODone + 0));
        vs_prev = vs;
      }
      if (ok) {
        ok = wait_phase(bar(kBarPReady + 1), (uint32_t)((n_kv - 1) & 1), abort_flag, p.timeout_ns, p.err,
                        kDevErrTimeoutMma, wtag(kBarPReady + 1, n_kv));
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tO1, tS1 + kk * 8, v_desc(vs_prev, kk), kIdescPV, (n_kv - 1 > 0 || kk > 0));
          mma_commit(bar(kBarKVEmpty + vs_prev));
          mma_commit(bar(kBarODone + 1));
        }
      }
      if (!ok) {
        // every MMA issued so far must finish reading shared memory and TMEM before exit
        mma_commit(bar(kBarDrain));
        wait_phase(bar(kBarDrain), 0, nullptr, p.timeout_ns, p.err, kDevErrTimeoutDrain, wtag(kBarDrain, 0));
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax groups
    const int t = (warp - 4) >> 2;   // Q tile of this group
    const int wq = warp & 3;         // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;    // row within the tile
    const int64_t qb = qb0 + t;
    const bool tile_ok = qb < p.nqb;
    const int64_t row = qb * kBQ + r;
    const bool row_ok = tile_ok && row < p.Sq;
    const int64_t bh = (int64_t)b * p.H + h;
    const bool fixed = !tile_ok || (!p.force_online && p.flag[bh * p.nqb + qb] != 0);
    // the row's shift: fixed-m rows subtract b_i from fm_bounds; online rows their running
    // max (one register serves both, the kernel is at its register limit)
    float shv = -INFINITY;
    if (fixed) shv = row_ok ? p.shift[bh * p.Sq + row] : 0.f;
    // an online row that adds into earlier chunks starts from their shift: as long as this
    // chunk's scores stay within 2^8 of it, O comes out at the accumulator's own shift and the
    // merge is a plain add
    else if (p.accumulate && row_ok) shv = p.acc_max[bh * p.Sq + row];
    const float shift_prev = shv;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + (uint32_t)(t * 128);
    const uint32_t tO = tmem + lane_off + 256u + (uint32_t)(t * 128);
    float l[4] = {0.f, 0.f, 0.f, 0.f};
    // key sinks of this head (ascending global key indices, INT_MAX pads): columns to drop
    int next_sink = sink_after_key(reinterpret_cast<const int32_t *>(gbase + kOffSinks), INT_MIN);
    bool ok = true;
    // the tile loop, instantiated once per kind of group (fixed-m or online), so that each copy
    // keeps only its own values live across the tiles
    auto tile_loop = [&](auto softmax_tile) {
      int c = 0;  // chunk of key tile j
      for (int j = 0; j < n_kv; ++j) {
        while (j >= p.tile0[c + 1]) ++c;
        ok = wait_phase(bar(kBarSFull + t), (uint32_t)(j & 1), abort_flag, p.timeout_ns, p.err,
                        kDevErrTimeoutSoftmax, wtag(kBarSFull + t, j));
        ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld/st below are warp-collective
        if (!ok) break;
        tc_fence_after();
        const int jl = (j - p.tile0[c]) * kBK;  // first key of the tile within its chunk
        const int nvalid = min(kBK, p.len[c] - jl);  // ragged end of each chunk
        const int g0 = p.key0[c] + jl;               // global index of the tile's first key
        if (next_sink < g0)  // sinks before this tile
          next_sink = sink_after_key(reinterpret_cast<const int32_t *>(gbase + kOffSinks), g0 - 1);
        // -inf over the key sinks in this tile and over the columns past the chunk's end
        if (next_sink < g0 + nvalid || nvalid < kBK)
          mask_tile(tS, nvalid, g0, reinterpret_cast<const int32_t *>(gbase + kOffSinks), next_sink);
        softmax_tile(j);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(kBarPReady + t));
      }
    };
    // the earlier chunks' row sum: a fixed-m group loads it before its tiles, so that the load's
    // latency hides behind them; an online group after them (a register held across its tiles,
    // which need more of them, slows the online tiles)
    float sum_prev = 0.f;
    if (fixed) {
      if (p.accumulate && row_ok) sum_prev = p.acc_sum[bh * p.Sq + row];
      tile_loop([&](int) { softmax_fixed_tile<true>(tS, p.alpha, -shv, l); });
    } else {
      tile_loop([&](int j) { softmax_online_tile(tS, tO, p.alpha, j > 0, shv, l); });
      if (ok && p.accumulate && row_ok) sum_prev = p.acc_sum[bh * p.Sq + row];
    }
    if (ok) {
      ok = wait_phase(bar(kBarODone + t), 0, abort_flag, p.timeout_ns, p.err, kDevErrTimeoutSoftmax,
                      wtag(kBarODone + t, n_kv));
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const float lsum = (l[0] + l[1]) + (l[2] + l[3]);
      const int64_t rflat = bh * p.Sq + row;
      float cprev = 0.f, cnew = 1.f, nr = shv;
      if (!fixed && row_ok && p.accumulate) {
        const float R = shift_prev;  // the previous chunks' shift (acc_max)
        nr = fmaxf(R, shv);
        cprev = (R == -INFINITY) ? 0.f : exp2f(R - nr);
        cnew = (shv == -INFINITY) ? 0.f : exp2f(shv - nr);
      }
      // the row's sum and shift after this chunk
      float sum_new = lsum;
      if (row_ok && p.accumulate) sum_new = fixed ? sum_prev + lsum : fmaf(sum_prev, cprev, lsum * cnew);
      const float shift_new = nr;  // b_i on fixed-m rows
      const bool final_out = p.out != nullptr;
      // A chunk that is not the last, on a tile whose O needs no rescale of the accumulator
      // (fixed-m; any tile of a first chunk, whose O is simply stored; an online tile whose
      // every row kept the accumulator's shift, so that cprev = cnew = 1): each warp posts its
      // rows' O as whole-row reductions (or stores) through 4 KiB of shared memory, so the SM
      // never reads the accumulator and the CTA need not wait for them before it exits (which
      // measured 1 % faster per step than staging the tile for bulk tensor reductions).  The
      // slabs are the Q region for tile 0, free once the last S MMA is done, which the O-done
      // commit covers, and the first K/V stage for tile 1, free once every MMA is done.
      bool plain_add = fixed || !p.accumulate;
      if (!plain_add && !final_out)
        plain_add = named_barrier_and(1 + t, 128, !row_ok || (shift_prev != -INFINITY && shv == shift_prev));
      if (plain_add && !final_out) {
        // the warp's first row is row - lane
        o_to_acc_warp(gbase + (t == 0 ? kOffQ : kOffKV) + wq * 4096, tO, lane, tile_ok, row - lane, p.Sq,
                      p.acc_o + (rflat - lane) * kHD, p.accumulate != 0,
                      EpiCheck{p.err, rflat - lane, p.dbg_rows, 0, 0});
        if (row_ok && FM_DCHECK(rflat < p.dbg_rows, p.err, 5u, rflat)) {
          p.acc_sum[rflat] = sum_new;
          p.acc_max[rflat] = shift_new;
        }
      } else {
      // the accumulator is read: the last chunk (o = (acc + O) / sum goes to `out`; "Kernel
      // reference: ring_attention_const_max_fwd": the last ring step folds and normalises, and
      // acc_o itself is not written back) or an online tile whose shift moved (acc = acc*cprev +
      // O*cnew); whole-row accesses per warp through its 4 KiB slab
      const float inv = final_out ? 1.0f / fmaxf(sum_new, FM_SUM_CLAMP) : 1.0f;
      void *out_row0 = nullptr;
      int64_t out_off0 = 0;
      if (final_out) {
        const int64_t ooff0 = (bh / p.H) * p.osB + (bh % p.H) * p.osH + (row - lane) * p.osS;
        out_off0 = ooff0;
        out_row0 = p.out_bf16 ? static_cast<void *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + ooff0)
                              : static_cast<void *>(reinterpret_cast<float *>(p.out) + ooff0);
      }
      acc_merge_warp(gbase + (t == 0 ? kOffQ : kOffKV) + wq * 4096, tO, lane, tile_ok, row - lane, p.Sq,
                     p.acc_o + (rflat - lane) * kHD, p.accumulate != 0, fixed, cprev, cnew, inv, out_row0, p.osS,
                     p.out_bf16 != 0,
                     EpiCheck{p.err, rflat - lane, p.dbg_rows, out_off0, p.dbg_out_span});
      if (row_ok && FM_DCHECK(rflat < p.dbg_rows, p.err, 5u, rflat)) {
        p.acc_sum[rflat] = sum_new;
        p.acc_max[rflat] = shift_new;
        if (final_out && p.lse) p.lse[rflat] = 0.69314718055994531f * (shift_new + log2f(sum_new));
      }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The persistent schedule (fm_opts.schedule = FM_SCHEDULE_PERSISTENT): one CTA per SM walks work
// items blockIdx.x, blockIdx.x + gridDim.x, ...; barrier phases and the K/V ring position carry
// over from item to item, and a Q-empty commit after an item's last S MMA lets the producer load
// the next item's Q while the softmax warps run the epilogue.  Its K/V ring has one stage fewer
// than the grid schedule's: that stage's space stages O for the bulk tensor reductions into the
// accumulator, one 16 KiB box per softmax group, while the next item's Q and K/V load.
__global__ void __launch_bounds__(kThreads, 1)
    fm_chunk_tc_persistent_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
  pdl_wait();  // bounds and accumulators written by the kernels before this one
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + kOffAbort);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kOffTmemSlot);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return base + (uint32_t)(kOffBar + 8 * i); };
  // this CTA's work items: every gridDim.x-th from blockIdx.x on.  Item -> (b, h, Q-tile pair);
  // consecutive items share a head and so its K/V tiles in L2.
  const int64_t item0 = blockIdx.x;
  const int64_t item_step = gridDim.x;
  auto item_bh = [&](int64_t item) -> int64_t { return item / p.n_pairs; };
  auto item_qb0 = [&](int64_t item) -> int64_t { return 2 * (item % p.n_pairs); };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(kBarQFull + 0), 1);
    mbar_init(bar(kBarQFull + 1), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKVFull + s), 1);
      mbar_init(bar(kBarKVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarPReady + t), 128);
      mbar_init(bar(kBarODone + t), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarQEmpty), 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_kv = p.n_kv;
  // Every item takes the same time, so without this every CTA would reach its epilogue at the
  // same moment and all their accumulator write-backs would meet in the memory system at once.
  // The CTAs with one item fewer have an item's time to spare: they start spread over it.
  if (p.stagger_ns) {
    const int64_t R = p.n_items % (int64_t)gridDim.x;
    if (R > 0 && (int64_t)blockIdx.x >= R) {
      const uint64_t d = p.stagger_ns * (uint64_t)((int64_t)blockIdx.x - R);
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < d) __nanosleep(256);
    }
  }

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int last_phase[kStages];  // phase of the last load issued into each stage, -1: none
      for (int s = 0; s < kStages; ++s) last_phase[s] = -1;
      bool ok = true;
      uint32_t q_loads = 0;      // Q tile pairs issued
      int st = 0;                // ring position of the next K/V load (carries over items)
      uint32_t ph = 0;
      const uint64_t q_pol = policy_evict_first();  // each Q tile is read once per launch
      for (int64_t item = item0; item < p.n_items && ok; item += item_step) {
        const int64_t bh = item_bh(item), qb0 = item_qb0(item);
        const int h = (int)(bh % p.H), b = (int)(bh / p.H);
        // Q of the previous item must have been read by all of its S MMAs
        if (q_loads > 0)
          ok = wait_phase(bar(kBarQEmpty), (q_loads - 1) & 1u, abort_flag, p.timeout_ns, p.err,
                          kDevErrTimeoutProducer, wtag(kBarQEmpty, 0));
        if (!ok) break;
        // one barrier per Q tile, so that S0 can start before tile 1 has landed
        for (int t = 0; t < 2; ++t) {
          mbar_expect_tx(bar(kBarQFull + t), 2 * kPanelBytes);
          for (int pn = 0; pn < 2; ++pn)
            tma_load_4d_hint(base + kOffQ + t * kTileBytes + pn * kPanelBytes, &maps.q, bar(kBarQFull + t),
                             pn * 64, (int)((qb0 + t) * kBQ), h, b, q_pol);
        }
        ++q_loads;
        int c = 0;  // chunk of key tile j
        for (int j = 0; j < n_kv && ok; ++j) {
          while (j >= p.tile0[c + 1]) ++c;
          const int jl = j - p.tile0[c];  // tile within its chunk
          for (int w = 0; w < 2 && ok; ++w) {
            ok = wait_phase(bar(kBarKVEmpty + st), ph ^ 1u, abort_flag, p.timeout_ns, p.err, kDevErrTimeoutProducer,
                            wtag(kBarKVEmpty + st, j));
            if (!ok) break;
            mbar_expect_tx(bar(kBarKVFull + st), kTileBytes);
            const CUtensorMap *tm = w ? &maps.v[c] : &maps.k[c];
            for (int pn = 0; pn < 2; ++pn)
              tma_load_4d(base + kOffKV + st * kTileBytes + pn * kPanelBytes, tm, bar(kBarKVFull + st), pn * 64,
                          jl * kBK, h, b);
            last_phase[st] = (int)ph;
            if (++st == kPStages) {
              st = 0;
              ph ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // let every copy already issued land before the CTA can exit
        for (int t = 0; t < 2 && q_loads > 0; ++t)
          wait_phase(bar(kBarQFull + t), (q_loads - 1) & 1u, nullptr, p.timeout_ns, p.err, kDevErrTimeoutDrain,
                     wtag(kBarQFull + t, 0));
        for (int s = 0; s < kPStages; ++s)
          if (last_phase[s] >= 0)
            wait_phase(bar(kBarKVFull + s), (uint32_t)last_phase[s], nullptr, p.timeout_ns, p.err,
                       kDevErrTimeoutDrain, wtag(kBarKVFull + s, 0));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t tS0 = tmem + 0, tS1 = tmem + 128, tO0 = tmem + 256, tO1 = tmem + 384;
      auto q_desc = [&](int t, int kk) {
        return smem_desc(base + kOffQ + t * kTileBytes + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
      };
      auto k_desc = [&](int s, int kk) {
        return smem_desc(base + kOffKV + s * kTileBytes + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
      };
      auto v_desc = [&](int s, int kk) {
        return smem_desc(base + kOffKV + s * kTileBytes + kk * 2048, kPanelBytes, 1024);
      };
      bool ok = true;
      uint32_t k = 0;    // items done by this CTA
      uint32_t tix = 0;  // key tiles consumed so far: the phase of the S-full / P-ready barriers
      int st = 0;        // ring position of the next K/V tile to consume
      uint32_t ph = 0;
      for (int64_t item = item0; item < p.n_items && ok; item += item_step, ++k) {
        // MMAs of one CTA run in issue order, so S(j) of this item may overwrite the S/P
        // columns that the previous item's last PV MMAs read; O is overwritten only by PV(0),
        // issued after the softmax group's P-ready arrival, which follows its epilogue reads.
        ok = wait_phase(bar(kBarQFull + 0), k & 1u, abort_flag, p.timeout_ns, p.err, kDevErrTimeoutMma,
                        wtag(kBarQFull + 0, 0));
        int vs_prev = 0;
        for (int j = 0; j < n_kv && ok; ++j, ++tix) {
          const int ks = st;
          const uint32_t kph = ph;
          if (++st == kPStages) {
            st = 0;
            ph ^= 1u;
          }
          ok = wait_phase(bar(kBarKVFull + ks), kph, abort_flag, p.timeout_ns, p.err, kDevErrTimeoutMma,
                          wtag(kBarKVFull + ks, j));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tS0, q_desc(0, kk), k_desc(ks, kk), kIdescQK, kk > 0);
          mma_commit(bar(kBarSFull + 0));
          if (j > 0) {
            ok = wait_phase(bar(kBarPReady + 1), (tix - 1) & 1u, abort_flag, p.timeout_ns, p.err,
                            kDevErrTimeoutMma, wtag(kBarPReady + 1, j));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tO1, tS1 + kk * 8, v_desc(vs_prev, kk), kIdescPV, (j - 1 > 0 || kk > 0));
            mma_commit(bar(kBarKVEmpty + vs_prev));
          }
          if (j == 0) {  // Q tile 1 may land after tile 0
            ok = wait_phase(bar(kBarQFull + 1), k & 1u, abort_flag, p.timeout_ns, p.err, kDevErrTimeoutMma,
                            wtag(kBarQFull + 1, 0));
            if (!ok) break;
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tS1, q_desc(1, kk), k_desc(ks, kk), kIdescQK, kk > 0);
          mma_commit(bar(kBarSFull + 1));
          mma_commit(bar(kBarKVEmpty + ks));
          if (j == n_kv - 1) mma_commit(bar(kBarQEmpty));  // the producer may load the next Q
          const int vs = st;
          const uint32_t vph = ph;
          if (++st == kPStages) {
            st = 0;
            ph ^= 1u;
          }
          ok = wait_phase(bar(kBarKVFull + vs), vph, abort_flag, p.timeout_ns, p.err, kDevErrTimeoutMma,
                          wtag(kBarKVFull + vs, j)) &&
               wait_phase(bar(kBarPReady + 0), tix & 1u, abort_flag, p.timeout_ns, p.err, kDevErrTimeoutMma,
                          wtag(kBarPReady + 0, j));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ts(tO0, tS0 + kk * 8, v_desc(vs, kk), kIdescPV, (j > 0 || kk > 0));
          if (j == n_kv - 1) mma_commit(bar(kBarODone + 0));
          vs_prev = vs;
        }
        if (ok) {
          ok = wait_phase(bar(kBarPReady + 1), (tix - 1) & 1u, abort_flag, p.timeout_ns, p.err,
                          kDevErrTimeoutMma, wtag(kBarPReady + 1, n_kv));
          if (ok) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tO1, tS1 + kk * 8, v_desc(vs_prev, kk), kIdescPV, (n_kv - 1 > 0 || kk > 0));
            mma_commit(bar(kBarKVEmpty + vs_prev));
            mma_commit(bar(kBarODone + 1));
          }
        }
      }
      if (!ok) {
        // every MMA issued so far must finish reading shared memory and TMEM before exit
        mma_commit(bar(kBarDrain));
        wait_phase(bar(kBarDrain), 0, nullptr, p.timeout_ns, p.err, kDevErrTimeoutDrain, wtag(kBarDrain, 0));
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax groups
    const int t = (warp - 4) >> 2;   // Q tile of this group
    const int wq = warp & 3;         // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;    // row within the tile
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + (uint32_t)(t * 128);
    const uint32_t tO = tmem + lane_off + 256u + (uint32_t)(t * 128);
    int32_t *ssk = reinterpret_cast<int32_t *>(gbase + kOffSinks) + t * FM_MAX_SINKS;
    bool ok = true;
    uint32_t g = 0;  // key tiles of earlier items: the phase of the S-full barrier carries over
    uint32_t k = 0;
    // Every thread of the group takes the same named barriers in the same order: a wait that
    // gave up ends this thread's tile loop, and the group agrees on the outcome at one barrier
    // that each of its threads reaches, before any other barrier of the item.
    for (int64_t item = item0; item < p.n_items; item += item_step, g += (uint32_t)n_kv, ++k) {
      const int64_t bh = item_bh(item);
      const int64_t qb = item_qb0(item) + t;
      const bool tile_ok = qb < p.nqb;
      const int64_t row = qb * kBQ + r;
      const bool row_ok = tile_ok && row < p.Sq;
      const bool fixed = !tile_ok || (!p.force_online && p.flag[bh * p.nqb + qb] != 0);
      // the row's shift: fixed-m rows subtract b_i from fm_bounds; online rows their running
      // max (one register serves both, the kernel is at its register limit)
      float shv = -INFINITY;
      if (fixed) shv = row_ok ? p.shift[bh * p.Sq + row] : 0.f;
      // an online row that adds into earlier chunks starts from their shift: as long as this
      // chunk's scores stay within 2^8 of it, O comes out at the accumulator's own shift and the
      // merge is a plain add
      else if (p.accumulate && row_ok) shv = p.acc_max[bh * p.Sq + row];
      const float shift_prev = shv;
      // the earlier chunks' row sum, loaded now so that its memory latency hides behind the tiles
      const float sum_prev = (p.accumulate && row_ok) ? p.acc_sum[bh * p.Sq + row] : 0.f;
      float l[4] = {0.f, 0.f, 0.f, 0.f};
      // key sinks of this item's head (ascending global key indices, INT_MAX pads): columns to
      // drop.  Every thread of the group finished the previous item's tiles (their P-ready
      // arrivals preceded its O-done) before any thread gets here, so the list can be replaced.
      // Without sinks the list is never read (next_sink stays INT_MAX).
      int next_sink = INT_MAX;
      if (p.sinks) {
        if (wq == 0 && lane < FM_MAX_SINKS) ssk[lane] = p.sinks[bh * FM_MAX_SINKS + lane];
        named_barrier(1 + t, 128);
        next_sink = sink_after_key(ssk, INT_MIN);
      }
      int c = 0;  // chunk of key tile j
      for (int j = 0; j < n_kv; ++j) {
        while (j >= p.tile0[c + 1]) ++c;
        ok = wait_phase(bar(kBarSFull + t), (g + (uint32_t)j) & 1u, abort_flag, p.timeout_ns, p.err,
                        kDevErrTimeoutSoftmax, wtag(kBarSFull + t, j));
        ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld/st below are warp-collective
        if (!ok) break;
        tc_fence_after();
        const int jl = (j - p.tile0[c]) * kBK;  // first key of the tile within its chunk
        const int nvalid = min(kBK, p.len[c] - jl);  // ragged end of each chunk
        const int g0 = p.key0[c] + jl;               // global index of the tile's first key
        if (next_sink < g0)  // sinks before this tile
          next_sink = sink_after_key(ssk, g0 - 1);
        // -inf over the key sinks in this tile and over the columns past the chunk's end
        if (next_sink < g0 + nvalid || nvalid < kBK) mask_tile(tS, nvalid, g0, ssk, next_sink);
        if (fixed) softmax_fixed_tile<false>(tS, p.alpha, -shv, l);
        else softmax_online_tile(tS, tO, p.alpha, j > 0, shv, l);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(kBarPReady + t));
      }
      if (ok) {
        ok = wait_phase(bar(kBarODone + t), k & 1u, abort_flag, p.timeout_ns, p.err, kDevErrTimeoutSoftmax,
                        wtag(kBarODone + t, n_kv));
        ok = __all_sync(0xffffffffu, ok);
      }
      ok = named_barrier_and(1 + t, 128, ok);
      if (!ok) break;
      tc_fence_after();
      const float lsum = (l[0] + l[1]) + (l[2] + l[3]);
      const int64_t rflat = bh * p.Sq + row;
      float cprev = 0.f, cnew = 1.f, nr = shv;
      if (!fixed && row_ok && p.accumulate) {
        const float R = shift_prev;  // the previous chunks' shift (acc_max)
        nr = fmaxf(R, shv);
        cprev = (R == -INFINITY) ? 0.f : exp2f(R - nr);
        cnew = (shv == -INFINITY) ? 0.f : exp2f(shv - nr);
      }
      // the row's sum and shift after this chunk
      float sum_new = lsum;
      if (row_ok && p.accumulate) sum_new = fixed ? sum_prev + lsum : fmaf(sum_prev, cprev, lsum * cnew);
      const float shift_new = nr;  // b_i on fixed-m rows
      const bool final_out = p.out != nullptr;
      // A chunk that is not the last, on a tile whose O needs no rescale of the accumulator
      // (fixed-m; any tile of a first chunk, whose O is simply stored; an online tile whose
      // every row kept the accumulator's shift, so that cprev = cnew = 1), adds O into acc_o
      // (or stores it there) without reading the accumulator through the SM: one 32-column box
      // at a time through the group's 16 KiB in the ring's fifth stage, with bulk tensor
      // reductions (the next item's Q and K/V load meanwhile), or, without an accumulator map,
      // with whole-row vector reductions per warp through the same box.
      bool plain_add = fixed || !p.accumulate;
      if (!plain_add && !final_out)
        plain_add = named_barrier_and(1 + t, 128, !row_ok || (shift_prev != -INFINITY && shv == shift_prev));
      if (p.acc_tma && plain_add && !final_out) {
        uint8_t *box = gbase + kOffPStage + t * kBoxBytes;
        const uint32_t sbox = base + (uint32_t)(kOffPStage + t * kBoxBytes);
        // an accumulator that fits in L2 stays there for the next chunk to add into
        const uint64_t acc_pol = p.acc_keep ? policy_evict_last() : policy_evict_normal();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c > 0) named_barrier(1 + t, 128);  // the previous box has been read
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          const int rl = wq * 32 + opaque_laneid();  // r, computed here (see opaque_laneid)
          uint8_t *line = box + rl * 128;
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            *reinterpret_cast<uint4 *>(line + ((q4 ^ (rl & 7)) << 4)) =
                make_uint4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
          fence_proxy_async_smem();
          named_barrier(1 + t, 128);
          if (wq == 0 && lane == 0) {
            if (tile_ok) tma_acc_3d(&maps.acc, sbox, c * 32, (int)(qb * kBQ), (int)bh, p.accumulate != 0, acc_pol);
            bulk_commit_and_wait_smem_read();
          }
        }
        if (row_ok && FM_DCHECK(rflat < p.dbg_rows, p.err, 5u, rflat)) {
          p.acc_sum[rflat] = sum_new;
          p.acc_max[rflat] = shift_new;
        }
      } else if (plain_add && !final_out) {
        o_to_acc_warp<true>(gbase + kOffPStage + t * kBoxBytes + wq * 4096, tO, lane, tile_ok, row - lane, p.Sq,
                            p.acc_o + (rflat - lane) * kHD, p.accumulate != 0,
                            EpiCheck{p.err, rflat - lane, p.dbg_rows, 0, 0});
        if (row_ok && FM_DCHECK(rflat < p.dbg_rows, p.err, 5u, rflat)) {
          p.acc_sum[rflat] = sum_new;
          p.acc_max[rflat] = shift_new;
        }
      } else {
      // the accumulator is read: the last chunk (o = (acc + O) / sum goes to `out`; "Kernel
      // reference: ring_attention_const_max_fwd": the last ring step folds and normalises, and
      // acc_o itself is not written back) or an online tile whose shift moved (acc = acc*cprev +
      // O*cnew); whole-row accesses per warp through its 4 KiB slab
      const float inv = final_out ? 1.0f / fmaxf(sum_new, FM_SUM_CLAMP) : 1.0f;
      void *out_row0 = nullptr;
      int64_t out_off0 = 0;
      if (final_out) {
        const int64_t ooff0 = (bh / p.H) * p.osB + (bh % p.H) * p.osH + (row - lane) * p.osS;
        out_off0 = ooff0;
        out_row0 = p.out_bf16 ? static_cast<void *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + ooff0)
                              : static_cast<void *>(reinterpret_cast<float *>(p.out) + ooff0);
      }
      acc_merge_warp<true>(gbase + kOffPStage + t * kBoxBytes + wq * 4096, tO, lane, tile_ok, row - lane, p.Sq,
                     p.acc_o + (rflat - lane) * kHD, p.accumulate != 0, fixed, cprev, cnew, inv, out_row0, p.osS,
                     p.out_bf16 != 0,
                     EpiCheck{p.err, rflat - lane, p.dbg_rows, out_off0, p.dbg_out_span});
      if (row_ok && FM_DCHECK(rflat < p.dbg_rows, p.err, 5u, rflat)) {
        p.acc_sum[rflat] = sum_new;
        p.acc_max[rflat] = shift_new;
        if (final_out && p.lse) p.lse[rflat] = 0.69314718055994531f * (shift_new + log2f(sum_new));
      }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The failure path of the bounded waits, on its own: one thread waits on an mbarrier
// phase that nothing completes, gives up after `timeout_ns` and records the failure in the
// error word exactly as the chunk kernel's waits do.
__global__ void wait_probe_kernel(unsigned int *err, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar_storage;
  const uint32_t bar = smem_u32(&bar_storage);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_phase(bar, 0, nullptr, timeout_ns, err, kDevErrTimeoutProbe, 0);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [B, H, S, D] bf16 view -> 4-D tensor map (D, S, H, B) with 64 x 128 boxes, 128-byte swizzle.
bool encode_map(CUtensorMap *map, const View &t) {
  auto enc = get_encode();
  if (!enc) return false;
  const uint64_t es = 2;
  cuuint64_t dims[4] = {(cuuint64_t)t.D, (cuuint64_t)t.S, (cuuint64_t)t.H, (cuuint64_t)t.B};
  // strides of size-1 dimensions are never stepped; give them a well-formed value
  const int64_t sS = t.S > 1 ? t.sS : t.D;
  const int64_t sH = t.H > 1 ? t.sH : t.S * sS;
  const int64_t sB = t.B > 1 ? t.sB : t.H * sH;
  cuuint64_t strides[3] = {(cuuint64_t)(sS * es), (cuuint64_t)(sH * es), (cuuint64_t)(sB * es)};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(t.ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The fp32 accumulator [B, H, Sq, 128] (contiguous) as a 3-D map over [B*H, Sq, 128] with a
// 32-column x 128-row box, 128-byte swizzle (the staging layout of the epilogue).
bool encode_acc_map(CUtensorMap *map, float *acc_o, const View &q) {
  auto enc = get_encode();
  if (!enc || q.S < 1 || q.B * q.H < 1) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kHD, (cuuint64_t)q.S, (cuuint64_t)(q.B * q.H)};
  cuuint64_t strides[2] = {(cuuint64_t)kHD * 4, (cuuint64_t)q.S * kHD * 4};
  cuuint32_t box[3] = {32, (cuuint32_t)kBQ, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, acc_o, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Schedule of a launch: fm_opts.schedule, with AUTO already resolved by the caller into one of
// the two (the persistent schedule for launches of short work items, fm_api.cu).
bool use_persistent(int schedule) { return schedule == FM_SCHEDULE_PERSISTENT; }

bool tma_view_ok(const View &t) {
  if (t.dtype != FM_BF16 || t.D != kHD || t.sD != 1) return false;
  if (reinterpret_cast<uintptr_t>(t.ptr) % 16) return false;
  if (t.S < 1 || t.B < 1 || t.H < 1) return false;
  auto ok16 = [](int64_t s, int64_t n) { return n <= 1 || ((s * 2) % 16 == 0 && s > 0); };
  return ok16(t.sS, t.S) && ok16(t.sH, t.H) && ok16(t.sB, t.B);
}

}  // namespace

bool chunk_tc_supported(const ChunkArgs &a) {
  if (a.n_chunks > kMaxChunks) return false;
  for (int c = 0; c < a.n_chunks; ++c)
    if (!tma_view_ok(a.ks[c]) || !tma_view_ok(a.vs[c]) || a.ks[c].S > ((int64_t)1 << 30)) return false;
  if (a.n_chunks > 0) {
    int64_t total = 0;
    for (int c = 0; c < a.n_chunks; ++c) total += a.ks[c].S;
    if (total > ((int64_t)1 << 30)) return false;
  }
  return tma_view_ok(a.q) && (a.n_chunks > 0 || (tma_view_ok(a.k) && tma_view_ok(a.v))) &&
         reinterpret_cast<uintptr_t>(a.acc_o) % 16 == 0 && a.q.B <= 65535 && a.q.H <= 65535 &&
         a.k.S <= (int64_t)1 << 30 && a.q.S <= (int64_t)1 << 30;
}

bool chunk_tc_final_supported(const ChunkArgs &a, const View &o) {
  const int64_t es = o.dtype == FM_F32 ? 4 : 2;
  const int64_t vec = 16;  // bytes of one vector store (4 fp32 or 8 bf16 elements)
  return o.D == kHD && o.sD == 1 && reinterpret_cast<uintptr_t>(o.ptr) % 16 == 0 &&
         (o.sS * es) % vec == 0 && (o.sH * es) % vec == 0 && (o.sB * es) % vec == 0 && o.B == a.q.B &&
         o.H == a.q.H && o.S == a.q.S;
}

cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t st) {
  const int nc = a.n_chunks > 0 ? a.n_chunks : 1;
  if (nc > kMaxChunks) return cudaErrorNotSupported;
  const View *ks = a.n_chunks > 0 ? a.ks : &a.k;
  const View *vs = a.n_chunks > 0 ? a.vs : &a.v;
  TcMaps maps;
  memset(&maps, 0, sizeof maps);
  // a layout the driver's tensor-map encoder refuses is reported so the caller can use
  // the CUDA-core kernel instead; nothing has been launched then
  if (!encode_map(&maps.q, a.q)) return cudaErrorNotSupported;
  for (int c = 0; c < nc; ++c)
    if (!encode_map(&maps.k[c], ks[c]) || !encode_map(&maps.v[c], vs[c])) return cudaErrorNotSupported;
  // once per device (and so never while a stream is being captured into a graph, as long
  // as the first call on a device comes before any capture)
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(fm_chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fm_chunk_tc_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  TcParams p;
  p.Sq = a.q.S;
  p.nqb = a.nqb;
  p.H = (int)a.q.H;
  p.n_chunks = nc;
  p.tile0[0] = 0;
  for (int c = 0; c < kMaxChunks; ++c) {
    p.len[c] = c < nc ? (int)ks[c].S : 0;
    p.tile0[c + 1] = p.tile0[c] + (c < nc ? (int)((ks[c].S + kBK - 1) / kBK) : 0);
  }
  p.n_kv = p.tile0[nc];
  p.sinks = a.sinks;
  int64_t g = a.sinks ? a.key0 : 0;  // without sinks the global offsets are not needed
  for (int c = 0; c < kMaxChunks; ++c) {
    p.key0[c] = (int)g;
    if (c < nc) g += ks[c].S;
  }
  p.alpha = a.alpha;
  p.force_online = a.force_online;
  p.accumulate = a.accumulate;
  p.flag = a.flag;
  p.shift = a.shift;
  p.acc_o = a.acc_o;
  p.acc_sum = a.acc_sum;
  p.acc_max = a.acc_max;
  p.err = a.err;
  p.timeout_ns = a.timeout_ns;
  p.out = nullptr;
  p.out_bf16 = 0;
  p.osB = p.osH = p.osS = 0;
  p.lse = a.lse;
  if (a.out) {
    p.out = const_cast<void *>(a.out->ptr);
    p.out_bf16 = a.out->dtype == FM_BF16;
    p.osB = a.out->sB;
    p.osH = a.out->sH;
    p.osS = a.out->sS;
  }
  p.n_pairs = (a.nqb + 1) / 2;
  p.n_items = p.n_pairs * a.q.H * a.q.B;
  // what the debug build's epilogue index checks compare against: the accumulator rows, and
  // the elements from o's first one to one past its last (positive strides on the fused path)
  p.dbg_rows = a.q.B * a.q.H * a.q.S;
  p.dbg_out_span = a.out ? (a.out->B - 1) * a.out->sB + (a.out->H - 1) * a.out->sH + (a.out->S - 1) * a.out->sS +
                               (a.out->D - 1) * a.out->sD + 1
                         : 0;
#ifdef FM_DEBUG
  // test hook of debug builds: FM_DEBUG_SHRINK_ROWS=n declares the accumulators n rows short,
  // so that the checks must catch (and skip) the last rows' accesses
  if (const char *shrink = getenv("FM_DEBUG_SHRINK_ROWS")) p.dbg_rows -= atoll(shrink);
#endif
  const int sms = current_device_sm_count();
  p.persistent = use_persistent(a.schedule) ? 1 : 0;
  // non-final chunks of the persistent schedule add O into acc_o with bulk tensor operations
  // where the map encodes (the one-item-per-CTA schedule posts whole-row reductions instead);
  // an accumulator within three quarters of L2 is kept there for the next chunk
  p.acc_tma = (p.persistent && !a.out && a.q.B * a.q.H <= INT_MAX && encode_acc_map(&maps.acc, a.acc_o, a.q)) ? 1 : 0;
  const double acc_bytes = 4.0 * (double)kHD * (double)a.q.S * (double)(a.q.B * a.q.H);
  p.acc_keep = acc_bytes <= 0.75 * (double)current_device_l2_bytes() ? 1 : 0;
  const dim3 grid = p.persistent ? dim3((unsigned)(p.n_items < sms ? p.n_items : sms))
                                 : dim3((unsigned)p.n_pairs, (unsigned)a.q.H, (unsigned)a.q.B);
  // the persistent CTAs with one item fewer start spread over an item's time, estimated low
  // (1.7 us a key tile and 4 us of prologue and epilogue) so that none ends later than the rest:
  // the 1024-key chunks' step went 785 -> 807 TFLOP/s, same bits
  p.stagger_ns = 0;
  if (p.persistent) {
    const int64_t G = grid.x, R = p.n_items % G;
    if (R > 0 && G > R)
      p.stagger_ns = (unsigned long long)((1700.0 * p.n_kv + 4000.0) / (double)(G - R));
  }
  return p.persistent ? launch_pdl(fm_chunk_tc_persistent_kernel, grid, dim3(kThreads), kSmemBytes, st, maps, p)
                      : launch_pdl(fm_chunk_tc_kernel, grid, dim3(kThreads), kSmemBytes, st, maps, p);
}

cudaError_t launch_wait_probe(unsigned int *err, unsigned long long timeout_ns, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fm
