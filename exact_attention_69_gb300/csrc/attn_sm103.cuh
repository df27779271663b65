// attn_sm103.cuh -- the fused exact-attention forward kernel for sm_103a.
//
// One CTA per SM (persistent). A task is a pair of 128-row Q tiles of one
// (batch, head); the CTA streams the K/V tiles that the pair needs and keeps
// the two Q tiles in flight at once, so that the tensor core works on one tile
// while the softmax warps work on the other.
//
//   warp 0      loader: TMA of Q (once per task) and of K_j, V_j into
//               multi-stage shared-memory rings (mbarrier full/empty pairs)
//   warp 1      MMA issuer (one elected lane of the converged warp): S_h = Q_h K_j^T into TMEM
//               (tcgen05.mma, both operands in shared memory), then
//               O_h += P_h V_j (A operand P_h read from TMEM)
//   warps 2-3   idle (they complete warpgroup 0, which gives its registers
//               to the softmax warpgroups with setmaxnreg)
//   warps 4-7   softmax of Q tile 0, warps 8-11 softmax of Q tile 1: one thread
//               per query row reads its S row from TMEM, applies the mask,
//               keeps the running maximum and row sum, writes P as bf16 back
//               over S in two halves of 64 keys (each announced on its own
//               barrier so that P V starts on the first half while the second
//               is computed), rescales O when the maximum grew, and finally
//               divides O by the row sum and stores O and the log-sum-exp.
//
// The method: "Fused Self Attention" (NKI tutorial) -- one strip of query rows
// at a time ("Fusion to Save SBUF Space"), row maxima and row sums with the
// division delayed until after the product with V ("Softmax implementation");
// the xformers memory-efficient attention post -- K tiles read in turn with a
// running softmax, only the end result written to memory; NATTEN issue #142
// -- a CTA loads a Q tile, loops over the K/V tiles it needs, skips the tiles
// that no window touches and masks the rest inside the tile.
//
// TMEM (512 columns, fp32 per 32-bit cell, one row per lane):
//   [0,128)   S_0 (P_0 as packed bf16 pairs in columns [0,64))
//   [128,256) S_1 (P_1 likewise)
//   [256,256+D) O_0, [256+D,256+2D) O_1
//
// Every wait is bounded: when one runs out the kernel records the failure in
// the device status word, raises a CTA-wide abort flag, lets every role leave
// its loop, waits (bounded) for its own copies and MMAs in flight, frees TMEM
// and returns.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "attn_kernel.h"

namespace attn {
namespace dev {

constexpr uint32_t kStatusTimeout = 5;  // same value as ATTN_ERR_TIMEOUT in attn.h
constexpr uint32_t kSleepHintNs = 200000;  // longest park per try_wait (also the abort latency)

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// The loader and MMA warps run converged: every lane executes the same
// instruction stream and `elect.sync` picks the one lane that acts. (Issued
// from a lone diverged lane, each tcgen05.mma costs ~190 cycles of issue
// instead of running back to back at the tensor core's rate.)
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

// True once the phase of `bar` with parity `parity` has completed.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_test, but lets the hardware park the thread until the phase
// completes or `hint_ns` passes, instead of returning at once: waiting
// threads then take no issue slots from the warps that share their scheduler.
__device__ __forceinline__ bool mbar_test_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 4-D tiled TMA load into shared memory, completion counted on `bar`
// (warp-wide; one elected lane issues it).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// As tma_load_4d, with an L2 eviction-priority policy for the tile (from
// l2_policy_evict_first / l2_policy_evict_last).
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                                 int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
      : "memory");
}

// L2 policies: data read once (Q) goes first when L2 needs room; data read by
// every task of a head (K, V) goes last.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// --- tcgen05: tensor memory and the 5th-generation tensor core

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (TMEM) = A (smem) * B (smem) [+ D]   (warp-wide; one elected lane issues it)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (TMEM) = A (TMEM) * B (smem) [+ D]   (warp-wide; one elected lane issues it)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Groups of MMAs along K in one statement, one election for the group: the
// first MMA accumulates iff `accumulate`, the others always do. The start
// address fields of consecutive k-steps' descriptors differ by the
// compile-time steps O1.. (address >> 4; no step carries out of the field,
// shared memory being below 256 KB). A group costs the issuing warp a
// fraction of the instructions of separately elected MMAs, which keeps the
// MMA warp's loop small.
template <int O1>
__device__ __forceinline__ void mma_ss2(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e, t;\n\t.reg .b64 a1, b1;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "add.s64 a1, %1, %5;\n\tadd.s64 b1, %2, %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(O1)
      : "memory");
}

template <int O1, int O2, int O3>
__device__ __forceinline__ void mma_ss4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e, t;\n\t.reg .b64 a1, b1;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "add.s64 a1, %1, %5;\n\tadd.s64 b1, %2, %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
      "add.s64 a1, %1, %6;\n\tadd.s64 b1, %2, %6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
      "add.s64 a1, %1, %7;\n\tadd.s64 b1, %2, %7;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(O1), "n"(O2), "n"(O3)
      : "memory");
}

// Four MMAs with A in TMEM: A steps 8 columns (16 bf16 keys) per k-step, B
// by the descriptor steps O1, O2, O3.
template <int O1, int O2, int O3>
__device__ __forceinline__ void mma_ts4(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e, t;\n\t.reg .b32 a1;\n\t.reg .b64 b1;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.u32 a1, %1, 8;\n\tadd.s64 b1, %2, %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
      "add.u32 a1, %1, 16;\n\tadd.s64 b1, %2, %6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
      "add.u32 a1, %1, 24;\n\tadd.s64 b1, %2, %7;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(O1), "n"(O2), "n"(O3)
      : "memory");
}

// One arrive on `bar` once every tcgen05 operation issued so far by the
// elected lane is complete (warp-wide; the same lane that issued the MMAs).
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

// Per-warpgroup register budget (all threads of the warpgroup execute it).
template <int N>
__device__ __forceinline__ void set_max_regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void set_max_regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#include "tmem_ldst.inc"

// --- arithmetic helpers (single PTX instructions)

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two floats to a bf16 pair (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor of tcgen05.mma: start address, leading and
// stride byte offsets (all >> 4), the fixed descriptor version bit 46, and
// the swizzle layout code in bits 61-63 (2 = 128-byte, 4 = 64-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(layout) << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: f32 accumulator, bf16 A
// and B, A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------- layout

template <int D>
struct Cfg {
  static_assert(D == 32 || D == 64 || D == 128, "head dimension");
  // A K/V/Q tile of 128 rows x D bf16 is stored as D / kBoxCols column chunks;
  // each chunk is 128 rows of kSwizzle bytes, swizzled the same way by TMA and
  // by the MMA descriptor, and lands 1024-byte aligned.
  static constexpr int kSwizzle = D >= 64 ? 128 : 64;
  static constexpr int kBoxCols = kSwizzle / 2;
  static constexpr int kChunks = D / kBoxCols;
  static constexpr int kChunkBytes = kBN * kSwizzle;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kKStages = D == 128 ? 2 : (D == 64 ? 3 : 4);
  static constexpr int kVStages = kKStages;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
  static constexpr int kBarBytes = 512;
  static_assert(8 * (15 + 2 * kKStages + 2 * kVStages) + 8 <= kBarBytes, "barrier area");
  // first unit of every CTA of a split schedule (kMaxSplitCtas + 1 int64),
  // then this CTA's first (task, K/V tile) packed in one int64
  static constexpr int kOffTbl = kOffBar + kBarBytes;
  static constexpr int kTblBytes = 8 * (kMaxSplitCtas + 2);
  static_assert(kTblBytes >= 2 * kBM * 4, "the twin exchange (m and l of 128 rows) shares the table");
  static constexpr int kSmemBytes = kOffTbl + kTblBytes + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static constexpr uint32_t kLayout = D >= 64 ? 2u : 4u;
  static constexpr uint32_t kIdescS = make_idesc(kBM, kBN, false);
  static constexpr uint32_t kIdescO = make_idesc(kBM, D, true);
  static constexpr uint32_t kTmemCols = 512;
  // S of Q tile h, its bf16 P (written over the first 64 columns of S) and O.
  __host__ __device__ static constexpr uint32_t tm_s(int h) { return 128u * h; }
  __host__ __device__ static constexpr uint32_t tm_p(int h) { return tm_s(h); }
  __host__ __device__ static constexpr uint32_t tm_o(int h) { return 256u + static_cast<uint32_t>(D) * h; }
};

// Barrier slots (8 bytes each) after the tiles.
struct Bars {
  uint32_t base;
  int kst, vst;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t q_empty() const { return base + 8; }
  __device__ uint32_t s_full(int h) const { return base + 16 + 8 * h; }
  // P of Q tile h, keys [64 * part, 64 * part + 64) written to TMEM
  __device__ uint32_t p_full(int h, int part) const { return base + 32 + 8 * (2 * h + part); }
  __device__ uint32_t o_full(int h) const { return base + 64 + 8 * h; }
  __device__ uint32_t o_empty(int h) const { return base + 80 + 8 * h; }
  __device__ uint32_t done() const { return base + 96; }
  __device__ uint32_t k_full(int s) const { return base + 104 + 8 * s; }
  __device__ uint32_t k_empty(int s) const { return base + 104 + 8 * (kst + s); }
  __device__ uint32_t v_full(int s) const { return base + 104 + 8 * (2 * kst + s); }
  __device__ uint32_t v_empty(int s) const { return base + 104 + 8 * (2 * kst + vst + s); }
  // twin tasks: warpgroup 1's m and l handed to warpgroup 0, and handed back
  __device__ uint32_t x_full() const { return base + 104 + 8 * (2 * kst + 2 * vst); }
  __device__ uint32_t x_empty() const { return base + 112 + 8 * (2 * kst + 2 * vst); }
  __device__ int count() const { return 15 + 2 * kst + 2 * vst; }
};

// ------------------------------------------------------------- bounded waits

struct Ctl {
  volatile uint32_t* abort;   // CTA-wide abort flag in shared memory
  uint32_t* status;           // device status word (4 x u32)
  uint64_t timeout_ns;
};

// Records the first failure in the device status word and raises the CTA's
// abort flag. Out of line: it runs only when a wait has run out.
static __device__ __noinline__ void report_timeout(volatile uint32_t* abort, uint32_t* status,
                                                   uint32_t role, int tile) {
  if (atomicCAS(status, 0u, kStatusTimeout) == 0u) {
    status[1] = role;
    status[2] = static_cast<uint32_t>(tile);
    status[3] = blockIdx.x;
    __threadfence();
  }
  *abort = 1u;
}

// The waiting part of warp_wait, out of line so that each wait site inlines
// only its first poll and vote: the control warps' loops stay small enough
// to run from the instruction cache. Called by all 32 lanes.
static __device__ __forceinline__ bool warp_wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                                   uint32_t* status, uint64_t timeout_ns, int tile,
                                                   uint32_t role, bool honour_abort) {
  const uint64_t t0 = global_ns();
  for (uint32_t n = 1;; ++n) {
    const bool ok = mbar_test_sleep(bar, parity, kSleepHintNs);
    if (__all_sync(0xffffffffu, ok)) return true;
    if (honour_abort && __any_sync(0xffffffffu, *abort != 0u)) return false;
    if ((n & 3u) == 0u &&
        __any_sync(0xffffffffu, global_ns() - t0 > timeout_ns || n >= (1u << 28))) {
      if ((threadIdx.x & 31) == 0) report_timeout(abort, status, role, tile);
      __syncwarp();
      return false;
    }
  }
}

// Warp-uniform wait for the phase of parity `parity` of `bar`: every lane
// polls the barrier and warp votes make each decision (done, abort, time out)
// the same for all lanes, so the warp never diverges. (Polling from one lane
// while the others wait at a shuffle costs the warps that share the scheduler
// measurably.) False: the CTA is aborting. Used by the softmax warps, whose
// live S row would have to be saved around a call.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Ctl& c, int tile,
                                          uint32_t role = kRoleSoftmax, bool honour_abort = true) {
  if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
  return warp_wait_slow(bar, parity, c.abort, c.status, c.timeout_ns, tile, role, honour_abort);
}

static __device__ __noinline__ bool ctl_wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                                  uint32_t* status, uint64_t timeout_ns, int tile,
                                                  uint32_t role, bool honour_abort) {
  return warp_wait_slow(bar, parity, abort, status, timeout_ns, tile, role, honour_abort);
}

// warp_wait for the loader and MMA warps: the same protocol with the waiting
// part out of line. Each of their many wait sites then inlines one poll and
// one vote, which keeps their loops a few KB long: measured on GB300, with
// every wait inlined whole the MMA warp's loop took ~50 KB of code and ran at
// instruction-fetch speed, hundreds of cycles per MMA issued.
__device__ __forceinline__ bool ctl_wait(uint32_t bar, uint32_t parity, const Ctl& c, int tile,
                                         uint32_t role, bool honour_abort = true) {
  if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
  return ctl_wait_slow(bar, parity, c.abort, c.status, c.timeout_ns, tile, role, honour_abort);
}

// Waits until the kernel this launch depends on (the previous one on the
// stream, under programmatic dependent launch) has completed and its memory
// operations are visible; returns at once without such a dependency.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------- work and masks

// The causal key bound's shift: key k allowed iff k <= q + shift (0 for
// top-left, a compile-time constant there; Nk - Nq for bottom-right).
template <int MASK>
__host__ __device__ __forceinline__ int causal_shift(const KernelParams& p) {
  return MASK == kMaskCausalBR ? p.causal_off : 0;
}

struct Task {
  int b, h, bh;
  int q0[2];
  bool live[2];
};

// Neighbourhood launches with one Q tile per task and long K/V chains run each
// task as a twin task (the host sets p.twin): both softmax warpgroups hold the
// same 128 queries and take its K/V tiles in turn (each with its own S, P, O,
// running maximum and row sum), and warpgroup 0 merges the two halves at the
// end, as the split schedule merges parts: M = max(m0, m1),
// L = l0 2^(m0 - M) + l1 2^(m1 - M), O = (O0 2^(m0 - M) + O1 2^(m1 - M)) / L.
// The K/V chain of a task is then half as long, and the tensor core runs one
// half's S while the other's softmax works.
template <int MASK>
__host__ __device__ __forceinline__ bool twin_mode(const KernelParams& p) {
  return mask_is_na(MASK) && p.twin != 0;
}

// Task t -> (batch, head, Q tiles: a pair, or one when p.q_tiles == 1). Causal:
// tasks in decreasing length order across all heads (longest first);
// otherwise head-major so that CTAs working at the same time share a head's
// K/V in L2.
template <int MASK>
__host__ __device__ __forceinline__ Task decode_task(int t, const KernelParams& p) {
  const int BH = p.B * p.H;
  int bh, qp;
  if (mask_is_causal(MASK)) {
    bh = t % BH;
    qp = p.n_qtasks - 1 - t / BH;
  } else {
    bh = t / p.n_qtasks;
    qp = t - bh * p.n_qtasks;
  }
  Task k;
  k.bh = bh;
  k.b = bh / p.H;
  k.h = bh - k.b * p.H;
  k.q0[0] = qp * p.q_tiles * kBM;
  k.q0[1] = k.q0[0] + kBM;
  k.live[0] = k.q0[0] < p.Nq;
  k.live[1] = p.q_tiles == 2 && k.q0[1] < p.Nq;
  if (twin_mode<MASK>(p)) {  // both warpgroups on the one Q tile
    k.q0[1] = k.q0[0];
    k.live[1] = k.live[0];
  }
  return k;
}

// Along one axis of length G with window w: does some query coordinate in
// [c0, c1] have a window that meets the key coordinates [e0, e1]?
template <bool WRAP>
__host__ __device__ __forceinline__ bool axis_meets(int c0, int c1, int e0, int e1, int G, int w) {
  const int half = w >> 1;
  if (!WRAP) {
    // clamped windows start at clamp(c - w/2, 0, G - w); starts grow with c
    const int lo = min(max(c0 - half, 0), G - w);
    const int hi = min(max(c1 - half, 0), G - w) + w - 1;
    return hi >= e0 && lo <= e1;
  }
  const int span = c1 - c0 + w;  // positions covered, counted circularly
  if (span >= G) return true;
  int a = c0 - half;
  if (a < 0) a += G;
  const int b = a + span - 1;
  if (b < G) return b >= e0 && a <= e1;
  return a <= e1 || b - G >= e0;  // covered: [a, G-1] and [0, b-G]
}

// As axis_meets for a dilated window (stride dl > 1). Every key coordinate
// of a dilated window lies within dl * (w - 1) of its query (clamp; the window
// holds the query) or dl * (w / 2) circularly (wrap): the test is whether
// that neighbourhood of [c0, c1] meets [e0, e1], a superset of the exact
// answer. A tile it keeps that no window touches is fully masked: wasted
// work, never a wrong result.
template <bool WRAP>
__host__ __device__ __forceinline__ bool axis_meets_dilated(int c0, int c1, int e0, int e1, int G,
                                                            int w, int dl) {
  if (!WRAP) {
    const int lo = max(c0 - dl * (w - 1), 0), hi = min(c1 + dl * (w - 1), G - 1);
    return hi >= e0 && lo <= e1;
  }
  const int reach = dl * (w >> 1);
  const int span = c1 - c0 + 1 + 2 * reach;
  if (span >= G) return true;
  int a = c0 - reach;
  if (a < 0) a += G;
  const int b = a + span - 1;
  if (b < G) return b >= e0 && a <= e1;
  return a <= e1 || b - G >= e0;
}

template <bool WRAP, bool DIL>
__host__ __device__ __forceinline__ bool axis_meets_nd(int c0, int c1, int e0, int e1, int G, int w,
                                                       int dl) {
  if (DIL) return axis_meets_dilated<WRAP>(c0, c1, e0, e1, G, w, dl);
  return axis_meets<WRAP>(c0, c1, e0, e1, G, w);
}

// Does any query in rows [q0, q1) attend any key in [k0, k1)? The Q and K
// ranges are cut into their grid-row segments; exact for dilation 1, a
// superset for dilation > 1 (see axis_meets_dilated).
template <bool WRAP_H, bool WRAP_W, bool DIL>
__host__ __device__ __forceinline__ bool na_tile_meets(int q0, int q1, int k0, int k1, const KernelParams& p) {
  const int W = p.grid_w;
  const int kr0 = k0 / W, kr1 = (k1 - 1) / W;
  // rows advance one by one: no division inside the loops
  for (int qa = q0, qr = q0 / W; qa < q1; ++qr) {
    const int qb = min(q1, (qr + 1) * W);
    if (axis_meets_nd<WRAP_H, DIL>(qr, qr, kr0, kr1, p.grid_h, p.window_h, p.dilation)) {
      for (int ka = k0, kr = kr0; ka < k1; ++kr) {
        const int kb = min(k1, (kr + 1) * W);
        if (axis_meets_nd<WRAP_H, DIL>(qr, qr, kr, kr, p.grid_h, p.window_h, p.dilation) &&
            axis_meets_nd<WRAP_W, DIL>(qa - qr * W, qb - 1 - qr * W, ka - kr * W, kb - 1 - kr * W,
                                       W, p.window_w, p.dilation))
          return true;
        ka = kb;
      }
    }
    qa = qb;
  }
  return false;
}

// axis_meets_nd with the wrap choice and the dilation read at run time.
__host__ __device__ __forceinline__ bool axis_meets_rt(bool wrap, int c0, int c1, int e0, int e1,
                                                       int G, int w, int dl) {
  if (dl > 1)
    return wrap ? axis_meets_dilated<true>(c0, c1, e0, e1, G, w, dl)
                : axis_meets_dilated<false>(c0, c1, e0, e1, G, w, dl);
  return wrap ? axis_meets<true>(c0, c1, e0, e1, G, w) : axis_meets<false>(c0, c1, e0, e1, G, w);
}

// na_tile_meets for a volume (depth, rows, columns; depth slowest). A line of
// the volume (fixed depth and row) holds grid_w consecutive tokens; the Q and
// K ranges are cut into line segments and each pair of segments is tested
// axis by axis (depth first, for the cheap rejection of far slices).
__host__ __device__ __forceinline__ bool na3_tile_meets(int q0, int q1, int k0, int k1,
                                                        const KernelParams& p) {
  const int W = p.grid_w, Gh = p.grid_h, dl = p.dilation;
  const bool wd = (p.na_wrap & kNa3WrapDepth) != 0, wh = (p.na_wrap & kNa3WrapRows) != 0,
             ww = (p.na_wrap & kNa3WrapCols) != 0;
  const int kr0 = k0 / W, kt0 = kr0 / Gh, ky0 = kr0 - kt0 * Gh, kt1 = ((k1 - 1) / W) / Gh;
  int qr = q0 / W;
  int qt = qr / Gh, qy = qr - qt * Gh;
  // lines advance one by one (row, then depth): no division inside the loops
  for (int qa = q0; qa < q1;) {
    const int qb = min(q1, (qr + 1) * W);
    if (axis_meets_rt(wd, qt, qt, kt0, kt1, p.grid_d, p.window_d, dl)) {
      int kt = kt0, ky = ky0;
      for (int ka = k0, kr = kr0; ka < k1; ++kr) {
        const int kb = min(k1, (kr + 1) * W);
        if (axis_meets_rt(wd, qt, qt, kt, kt, p.grid_d, p.window_d, dl) &&
            axis_meets_rt(wh, qy, qy, ky, ky, Gh, p.window_h, dl) &&
            axis_meets_rt(ww, qa - qr * W, qb - 1 - qr * W, ka - kr * W, kb - 1 - kr * W, W,
                          p.window_w, dl))
          return true;
        ka = kb;
        if (++ky == Gh) {
          ky = 0;
          ++kt;
        }
      }
    }
    qa = qb;
    ++qr;
    if (++qy == Gh) {
      qy = 0;
      ++qt;
    }
  }
  return false;
}

// Tiles (128 tokens, for K/V and for Q alike) that can hold a partner of some
// token in [a, b] (inclusive): at most two half-open intervals [lo0, hi0) and
// [lo1, hi1), in increasing order. A superset, from the slowest grid axis that
// is longer than one: a clamped window keeps every key within dl * (w - 1) of
// its query on each axis and a wrapped one within dl * (w / 2) circularly;
// both bounds hold in either direction (the keys of a query, the queries of a
// key), so the forward and the backward passes share the band.
struct Band {
  int lo0, hi0, lo1, hi1;
};

template <int MASK>
__host__ __device__ __forceinline__ Band na_band(int a, int b, const KernelParams& p) {
  int unit, G, w;
  bool wrap;
  if (MASK == kMaskNa3 && p.grid_d > 1) {
    unit = p.grid_h * p.grid_w;
    G = p.grid_d;
    w = p.window_d;
    wrap = (p.na_wrap & kNa3WrapDepth) != 0;
  } else if (p.grid_h > 1) {
    unit = p.grid_w;
    G = p.grid_h;
    w = p.window_h;
    wrap = MASK == kMaskNa3 ? (p.na_wrap & kNa3WrapRows) != 0 : mask_na_wrap_rows(MASK);
  } else {
    unit = 1;
    G = p.grid_w;
    w = p.window_w;
    wrap = MASK == kMaskNa3 ? (p.na_wrap & kNa3WrapCols) != 0 : mask_na_wrap_cols(MASK);
  }
  const int dl = (MASK == kMaskNa3 || mask_na_dilated(MASK)) ? p.dilation : 1;
  const int c0 = a / unit, c1 = b / unit;
  int x0, x1, y0 = 0, y1 = -1;  // coordinate intervals [x0, x1] then [y0, y1]
  if (wrap) {
    const int reach = dl * (w >> 1);
    const int lo = c0 - reach, hi = c1 + reach;
    if (c1 - c0 + 1 + 2 * reach >= G) {
      x0 = 0;
      x1 = G - 1;
    } else if (lo < 0) {
      x0 = 0;
      x1 = hi;
      y0 = lo + G;
      y1 = G - 1;
    } else if (hi >= G) {
      x0 = 0;
      x1 = hi - G;
      y0 = lo;
      y1 = G - 1;
    } else {
      x0 = lo;
      x1 = hi;
    }
  } else {
    const int reach = dl * (w - 1);
    x0 = max(c0 - reach, 0);
    x1 = min(c1 + reach, G - 1);
  }
  Band r;
  r.lo0 = x0 * unit / kBN;
  r.hi0 = ((x1 + 1) * unit - 1) / kBN + 1;
  r.lo1 = r.hi1 = 0;
  if (y1 >= y0) {
    r.lo1 = y0 * unit / kBN;
    r.hi1 = ((y1 + 1) * unit - 1) / kBN + 1;
  }
  return r;
}

// The first tile of the band after tile j (a large number if none).
__host__ __device__ __forceinline__ int band_next(const Band& b, int j) {
  ++j;
  if (j < b.lo0) return b.lo0;
  if (j < b.hi0) return j;
  if (j < b.lo1) j = b.lo1;
  return j < b.hi1 ? j : 0x7fffffff;
}

// K/V tiles a task may visit: the band of its queries (every tile without a
// neighbourhood mask).
template <int MASK>
__host__ __device__ __forceinline__ Band task_band(const Task& tk, const KernelParams& p) {
  if constexpr (mask_is_na(MASK)) {
    return na_band<MASK>(tk.q0[0], min(tk.q0[tk.live[1] ? 1 : 0] + kBM, p.Nq) - 1, p);
  } else {
    Band b;
    b.lo0 = 0;
    b.hi0 = p.n_kv;
    b.lo1 = b.hi1 = 0;
    return b;
  }
}

// 0: no query of the tile attends any key of KV tile j (skip it);
// 1: every (query, key) pair is allowed (no mask); 2: mask inside the tile.
template <int MASK>
__host__ __device__ __forceinline__ int tile_class(int q0, int j, const KernelParams& p) {
  const int k0 = j * kBN;
  const bool ragged = k0 + kBN > p.Nk;
  if (MASK == kMaskNone) return ragged ? 2 : 1;
  const int q1 = min(q0 + kBM, p.Nq);
  if (mask_is_causal(MASK)) {  // key k allowed iff k <= q + off
    const int off = causal_shift<MASK>(p);
    if (k0 > q1 - 1 + off) return 0;
    return (!ragged && k0 + kBN - 1 <= q0 + off) ? 1 : 2;
  }
  if (MASK == kMaskNa3) return na3_tile_meets(q0, q1, k0, min(k0 + kBN, p.Nk), p) ? 2 : 0;
  return na_tile_meets<mask_na_wrap_rows(MASK), mask_na_wrap_cols(MASK), mask_na_dilated(MASK)>(
             q0, q1, k0, min(k0 + kBN, p.Nk), p)
             ? 2 : 0;
}

template <int MASK>
__host__ __device__ __forceinline__ bool tile_active(const Task& tk, int h, int j, const KernelParams& p) {
  return tk.live[h] && tile_class<MASK>(tk.q0[h], j, p) != 0;
}

// Next KV tile after j and before `end` that some live Q tile of the task
// needs (`end` if none); neighbourhood masks look only inside the task's band.
template <int MASK>
__host__ __device__ __forceinline__ int next_tile(const Task& tk, const Band& band, int j, int end,
                                                  const KernelParams& p) {
  if constexpr (mask_is_na(MASK)) {
    for (j = band_next(band, j); j < end; j = band_next(band, j))
      if (tile_active<MASK>(tk, 0, j, p) || tile_active<MASK>(tk, 1, j, p)) return j;
  } else {
    for (++j; j < end; ++j)
      if (tile_active<MASK>(tk, 0, j, p) || tile_active<MASK>(tk, 1, j, p)) return j;
  }
  return end;
}

// Successive K/V tiles of a neighbourhood task inside its band, with the Q
// tiles each one is active for. A whole warp searches 32 band positions at a
// time (lane i runs the exact tile test on position base + i; ballots collect
// the answers), so one warp pays one test per 32 tiles instead of one per
// tile. `which` = 0 or 1: only that Q tile's tiles are wanted (the other's
// tests are skipped); 2: both. Every lane of the warp must call next().
template <int MASK>
struct TileCursor {
  Band b;
  int len0, lo1s, len, base, pos, which, cnt;
  uint32_t m0, m1;
  bool twin;
  __device__ __forceinline__ TileCursor(const Band& band, int w, bool tw = false)
      : b(band), which(w), cnt(0), twin(tw) {
    len0 = b.hi0 - b.lo0;
    lo1s = max(b.lo1, b.hi0);  // the second interval may share a tile with the first
    len = len0 + max(b.hi1 - lo1s, 0);
    base = -32;
    pos = -1;
    m0 = m1 = 0u;
  }
  __device__ __forceinline__ int tile_at(int q) const {
    return q < len0 ? b.lo0 + q : lo1s + (q - len0);
  }
  // The next active tile (`end` if none) and, in a, whether each Q tile needs it.
  __device__ __forceinline__ int next(const Task& tk, int end, bool (&a)[2], const KernelParams& p) {
    for (++pos; pos < len;) {
      if (pos >= base + 32) {
        base = pos & ~31;
        const int q = base + static_cast<int>(threadIdx.x & 31);
        const int t = q < len ? tile_at(q) : -1;
        const bool x0 = t >= 0 && which != 1 && tile_active<MASK>(tk, 0, t, p);
        const bool x1 = t >= 0 && which != 0 && tile_active<MASK>(tk, 1, t, p);
        m0 = __ballot_sync(0xffffffffu, x0);
        m1 = __ballot_sync(0xffffffffu, x1);
      }
      const uint32_t m = (m0 | m1) >> (pos - base);
      if (m != 0u) {
        pos += __ffs(static_cast<int>(m)) - 1;
        if (twin) {
          // a twin task's tiles go to its two warpgroups in turn
          const int owner = cnt & 1;
          ++cnt;
          if (which != 2 && which != owner) {
            ++pos;
            continue;
          }
          a[0] = owner == 0;
          a[1] = owner == 1;
        } else {
          a[0] = ((m0 >> (pos - base)) & 1u) != 0u;
          a[1] = ((m1 >> (pos - base)) & 1u) != 0u;
        }
        const int t = tile_at(pos);
        return t < end ? t : end;
      }
      pos = base + 32;
    }
    return end;
  }
};

// ------------------------------------------------------------- work split

// A segment: KV tiles [kv0, kv1) of task t; `head` marks the CTA's first one.
struct Seg {
  int t, kv0, kv1;
  bool head;
};

// First unit of CTA c when the units are split evenly over `ctas` CTAs.
__host__ __device__ __forceinline__ int64_t unit_lo(int64_t units, int ctas, int c) {
  return static_cast<int64_t>(c) * units / ctas;
}

// The split schedule's segments of this CTA, walked without division: the
// first (task, K/V tile) comes from the prologue's table, then the position
// advances by each segment's length. (A 64-bit division per segment is a
// call into a library routine, and the call made the MMA warp, which runs
// with few registers, spill its loop state to local memory.)
template <int MASK>
struct SegIter {
  int rest;  // units of this CTA not yet handed out (< 2^31: the host splits no larger share)
  int t_rr, kv;
  int rnd = 0;  // causal: tasks taken so far
  bool first;
  __device__ __forceinline__ SegIter(const KernelParams& p, const int64_t* lo) : first(true) {
    if (MASK == kMaskNone && p.split) {
      rest = static_cast<int>(lo[blockIdx.x + 1] - lo[blockIdx.x]);
      const int64_t f = lo[kMaxSplitCtas + 1];
      t_rr = static_cast<int>(f >> 32);
      kv = static_cast<int>(f & 0xffffffff);
    } else {
      t_rr = blockIdx.x;
    }
  }
  __device__ __forceinline__ bool next(const KernelParams& p, Seg& s) {
    if (MASK == kMaskNone && p.split) {
      if (rest <= 0) return false;
      s.t = t_rr;
      s.kv0 = kv;
      const int len = min(rest, p.n_kv - kv);
      s.kv1 = kv + len;
      rest -= len;
      kv += len;
      if (kv == p.n_kv) {
        kv = 0;
        ++t_rr;
      }
    } else if constexpr (mask_is_causal(MASK)) {
      // Causal tasks come longest first; dealt back and forth (CTA c takes
      // task c of the first round, task G - 1 - c of the second, ...), the
      // CTAs' total lengths come out nearly equal, where a plain round robin
      // gives CTA 0 the longest task of every round. A CTA past the last
      // task in one round is past it in every later one.
      const int G = static_cast<int>(gridDim.x);
      const int t = rnd * G + ((rnd & 1) ? G - 1 - static_cast<int>(blockIdx.x)
                                         : static_cast<int>(blockIdx.x));
      if (t >= p.n_tasks) return false;
      ++rnd;
      s.t = t;
      s.kv0 = 0;
      s.kv1 = p.n_kv;
    } else {
      if (t_rr >= p.n_tasks) return false;
      s.t = t_rr;
      s.kv0 = 0;
      s.kv1 = p.n_kv;
      t_rr += gridDim.x;
    }
    s.head = first;
    first = false;
    return true;
  }
};

// First key coordinate of the window of query coordinate c on an axis of
// length G (window w odd, dilation dl): the window's keys are f + dl * t,
// t in [0, w) (modulo G for wrap). Clamp: the keys share c's residue modulo
// dl, and inside that residue class the w-wide window is centred on c and
// shifted inward at the borders. Wrap: centred on c, circular.
template <bool WRAP, bool DIL>
__host__ __device__ __forceinline__ int na_window_first(int c, int G, int w, int dl) {
  const int half = w >> 1;
  if (!DIL) dl = 1;
  if (WRAP) {
    const int f = c - dl * half;  // > -G since dl * w <= G
    return f < 0 ? f + G : f;
  }
  if (dl == 1) return min(max(c - half, 0), G - w);
  const int r = c % dl;
  const int len = (G - r + dl - 1) / dl;  // positions of residue r
  const int start = min(max(c / dl - half, 0), len - w);
  return r + dl * start;
}

// Grid coordinates of query token q and the first key coordinates of its
// window along each axis.
template <bool WRAP_H, bool WRAP_W, bool DIL>
__host__ __device__ __forceinline__ void na_query_coords(const KernelParams& p, int q, int& qy,
                                                         int& qx, int& wy, int& wx) {
  qy = q / p.grid_w;
  qx = q - qy * p.grid_w;
  wy = na_window_first<WRAP_H, DIL>(qy, p.grid_h, p.window_h, p.dilation);
  wx = na_window_first<WRAP_W, DIL>(qx, p.grid_w, p.window_w, p.dilation);
}

// Is key coordinate k in the window that starts at f (stride dl, w keys)?
template <bool WRAP, bool DIL>
__host__ __device__ __forceinline__ bool na_in_window(int k, int f, int G, int w, int dl) {
  int d = k - f;
  if (WRAP) d += d < 0 ? G : 0;
  if (d < 0) return false;
  if (!DIL) return d < w;
  return d % dl == 0 && d / dl < w;
}

// Sets bits [lo, hi) (0 <= lo <= hi <= 128) of a 128-bit mask.
__host__ __device__ __forceinline__ void set_bits(uint32_t (&bits)[4], int lo, int hi) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int a = max(lo - 32 * w, 0), b = min(hi - 32 * w, 32);
    if (a < b) {
      const uint32_t upto = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
      bits[w] |= upto & ~((1u << a) - 1u);
    }
  }
}

// Columns of one key line that the window's columns cover: the line's
// columns [kx0, kx0 + len) sit at bits base + kx0 ... (base = bit of column 0).
// With dilation 1 they form one interval (two when a wrapped window crosses
// the last column); with dilation > 1 they are set one by one.
template <bool WRAP_W, bool DIL>
__host__ __device__ __forceinline__ void na_line_cols(uint32_t (&bits)[4], int base, int kx0, int len,
                                                      int wx, int G_w, int w, int dl) {
  if (!DIL) {
    const int e1 = min(wx + w, G_w);
    int lo = max(wx, kx0), hi = min(e1, kx0 + len);
    if (lo < hi) set_bits(bits, base + lo, base + hi);
    if (WRAP_W && wx + w > G_w) {  // the window wraps past the last column
      lo = kx0;
      hi = min(wx + w - G_w, kx0 + len);
      if (lo < hi) set_bits(bits, base + lo, base + hi);
    }
  } else {
    for (int t = 0; t < w; ++t) {
      int cx = wx + dl * t;
      if (WRAP_W && cx >= G_w) cx -= G_w;
      if (cx >= kx0 && cx < kx0 + len) {
        const int bit = base + cx;
        bits[bit >> 5] |= 1u << (bit & 31);
      }
    }
  }
}

// Allowed keys of query (qy, qx) in the K/V tile starting at key k0, as bits
// of a 128-bit mask (bit i: key k0 + i). The window's rows are wy + dl * t,
// t in [0, w_h), and its columns wx + dl * t, t in [0, w_w) (modulo the grid
// side along an axis that wraps). With dilation 1 a row's allowed columns
// form one interval (two when a wrapped window crosses the last column); with
// dilation > 1 they are set one by one.
template <bool WRAP_H, bool WRAP_W, bool DIL>
__host__ __device__ __forceinline__ void na_tile_bits(const KernelParams& p, int k0, int qy, int qx, int wy,
                                             int wx, uint32_t (&bits)[4]) {
  const int G_h = p.grid_h, G_w = p.grid_w, w_h = p.window_h, w = p.window_w, dl = p.dilation;
  bits[0] = bits[1] = bits[2] = bits[3] = 0u;
  const int nvalid = min(kBN, p.Nk - k0);
  int ky = k0 / G_w;
  int kx0 = k0 - ky * G_w;
  for (int i = 0; i < nvalid; ++ky) {
    const int len = min(G_w - kx0, nvalid - i);  // this row's columns [kx0, kx0 + len)
    if (na_in_window<WRAP_H, DIL>(ky, wy, G_h, w_h, dl))
      na_line_cols<WRAP_W, DIL>(bits, i - kx0, kx0, len, wx, G_w, w, dl);
    i += len;
    kx0 = 0;
  }
}

// ---- volumes (kMaskNa3): the same rules with the wrap choice and dilation
// read at run time, and a depth axis slower than the rows ----

__host__ __device__ __forceinline__ int na_first_rt(int c, int G, int w, int dl, bool wrap) {
  return wrap ? na_window_first<true, true>(c, G, w, dl) : na_window_first<false, true>(c, G, w, dl);
}

__host__ __device__ __forceinline__ bool na_in_rt(int k, int f, int G, int w, int dl, bool wrap) {
  if (dl == 1) return wrap ? na_in_window<true, false>(k, f, G, w, 1) : na_in_window<false, false>(k, f, G, w, 1);
  return wrap ? na_in_window<true, true>(k, f, G, w, dl) : na_in_window<false, true>(k, f, G, w, dl);
}

// A query's grid coordinates and the first key coordinate of its window on
// each axis (depth only for volumes).
struct NaQuery {
  int qy = 0, qx = 0, wy = 0, wx = 0, qt = 0, wt = 0;
};

template <int MASK>
__host__ __device__ __forceinline__ NaQuery na_query(const KernelParams& p, int q) {
  NaQuery n;
  if constexpr (MASK == kMaskNa3) {
    const int plane = p.grid_h * p.grid_w;
    n.qt = q / plane;
    const int r = q - n.qt * plane;
    n.qy = r / p.grid_w;
    n.qx = r - n.qy * p.grid_w;
    n.wt = na_first_rt(n.qt, p.grid_d, p.window_d, p.dilation, (p.na_wrap & kNa3WrapDepth) != 0);
    n.wy = na_first_rt(n.qy, p.grid_h, p.window_h, p.dilation, (p.na_wrap & kNa3WrapRows) != 0);
    n.wx = na_first_rt(n.qx, p.grid_w, p.window_w, p.dilation, (p.na_wrap & kNa3WrapCols) != 0);
  } else if constexpr (mask_is_na2(MASK)) {
    na_query_coords<mask_na_wrap_rows(MASK), mask_na_wrap_cols(MASK), mask_na_dilated(MASK)>(
        p, q, n.qy, n.qx, n.wy, n.wx);
  }
  return n;
}

// na_tile_bits for a volume: a key line (fixed depth and row) is kept when
// both its depth and its row are in the query's window, then its columns are
// set as in two dimensions.
__host__ __device__ __forceinline__ void na3_tile_bits(const KernelParams& p, int k0, const NaQuery& n,
                                                       uint32_t (&bits)[4]) {
  const int G_h = p.grid_h, G_w = p.grid_w, dl = p.dilation;
  const bool wd = (p.na_wrap & kNa3WrapDepth) != 0, wh = (p.na_wrap & kNa3WrapRows) != 0,
             ww = (p.na_wrap & kNa3WrapCols) != 0;
  bits[0] = bits[1] = bits[2] = bits[3] = 0u;
  const int nvalid = min(kBN, p.Nk - k0);
  const int r0 = k0 / G_w;
  int kt = r0 / G_h, ky = r0 - kt * G_h;
  int kx0 = k0 - r0 * G_w;
  for (int i = 0; i < nvalid;) {
    const int len = min(G_w - kx0, nvalid - i);
    if (na_in_rt(kt, n.wt, p.grid_d, p.window_d, dl, wd) && na_in_rt(ky, n.wy, G_h, p.window_h, dl, wh)) {
      const int base = i - kx0;
      if (dl == 1) {
        if (ww) na_line_cols<true, false>(bits, base, kx0, len, n.wx, G_w, p.window_w, 1);
        else na_line_cols<false, false>(bits, base, kx0, len, n.wx, G_w, p.window_w, 1);
      } else {
        if (ww) na_line_cols<true, true>(bits, base, kx0, len, n.wx, G_w, p.window_w, dl);
        else na_line_cols<false, true>(bits, base, kx0, len, n.wx, G_w, p.window_w, dl);
      }
    }
    i += len;
    kx0 = 0;
    if (++ky == G_h) {
      ky = 0;
      ++kt;
    }
  }
}

// ---------------------------------------------------------------- roles

template <int D, int MASK>
__device__ void loader_role(const KernelParams& p, uint32_t sbase, const Bars& bars,
                            const int64_t* cta_lo, const Ctl& ctl) {
  using C = Cfg<D>;
  uint32_t q_it = 0, k_it = 0, v_it = 0;
  // Stage bookkeeping for the drain, as bit masks (bit s: stage s holds an
  // armed copy; its phase parity), so that it stays in registers.
  int q_armed = -1;
  uint32_t k_armed = 0, k_par = 0, v_armed = 0, v_par = 0;
  bool injected = false;
  const uint64_t pol_once = l2_policy_evict_first(), pol_reuse = l2_policy_evict_last();
  SegIter<MASK> it(p, cta_lo);
  Seg sg;
  bool dep_waited = false;
  while (it.next(p, sg)) {
    const Task tk = decode_task<MASK>(sg.t, p);
    const Band band = task_band<MASK>(tk, p);
    constexpr bool kNa = mask_is_na(MASK);
    TileCursor<MASK> cur(band, 2, twin_mode<MASK>(p));
    bool act[2];
    // the first tile is found (kernel parameters only) before the previous
    // kernel's completion is awaited
    const int j0 = kNa ? cur.next(tk, sg.kv1, act, p) : next_tile<MASK>(tk, band, sg.kv0 - 1, sg.kv1, p);
    if (!dep_waited) {
      grid_dep_wait();
      dep_waited = true;
    }
    if (!ctl_wait(bars.q_empty(), (q_it & 1u) ^ 1u, ctl, -1, kRoleLoader)) goto drain;
    mbar_expect_tx(bars.q_full(), 2 * C::kTileBytes);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_4d_hint(sbase + C::kOffQ + h * C::kTileBytes + c * C::kChunkBytes, &p.tm_q,
                         bars.q_full(), c * C::kBoxCols, tk.q0[h], tk.h, tk.b, pol_once);
    q_armed = static_cast<int>(q_it & 1u);
    ++q_it;
    int nth = 0;
    for (int j = j0;
         j < sg.kv1;
         j = kNa ? cur.next(tk, sg.kv1, act, p) : next_tile<MASK>(tk, band, j, sg.kv1, p), ++nth) {
      const int ks = static_cast<int>(k_it % C::kKStages);
      if (!ctl_wait(bars.k_empty(ks), ((k_it / C::kKStages) & 1u) ^ 1u, ctl, j, kRoleLoader))
        goto drain;
      if (p.inject && !injected && nth == 1) {
        injected = true;  // withhold this K tile: the MMA issuer's wait must run out
      } else {
        mbar_expect_tx(bars.k_full(ks), C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d_hint(sbase + C::kOffK + ks * C::kTileBytes + c * C::kChunkBytes, &p.tm_k,
                           bars.k_full(ks), c * C::kBoxCols, j * kBN, tk.h, tk.b, pol_reuse);
        k_armed |= 1u << ks;
        k_par = (k_par & ~(1u << ks)) | (((k_it / C::kKStages) & 1u) << ks);
      }
      ++k_it;
      const int vs = static_cast<int>(v_it % C::kVStages);
      if (!ctl_wait(bars.v_empty(vs), ((v_it / C::kVStages) & 1u) ^ 1u, ctl, j, kRoleLoader))
        goto drain;
      mbar_expect_tx(bars.v_full(vs), C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_4d_hint(sbase + C::kOffV + vs * C::kTileBytes + c * C::kChunkBytes, &p.tm_v,
                         bars.v_full(vs), c * C::kBoxCols, j * kBN, tk.h, tk.b, pol_reuse);
      v_armed |= 1u << vs;
      v_par = (v_par & ~(1u << vs)) | (((v_it / C::kVStages) & 1u) << vs);
      ++v_it;
    }
  }
drain:
  // The last copy armed on each barrier must have landed before the CTA exits.
  if (q_armed >= 0) ctl_wait(bars.q_full(), q_armed, ctl, -1, kRoleLoader, false);
  for (int s = 0; s < C::kKStages; ++s)
    if ((k_armed >> s) & 1u) ctl_wait(bars.k_full(s), (k_par >> s) & 1u, ctl, -1, kRoleLoader, false);
  for (int s = 0; s < C::kVStages; ++s)
    if ((v_armed >> s) & 1u) ctl_wait(bars.v_full(s), (v_par >> s) & 1u, ctl, -1, kRoleLoader, false);
}

// An opaque copy of a value: keeps the compiler from hoisting every per-step
// value derived from it out of a loop (used where registers are scarce).
__device__ __forceinline__ uint32_t opaque(uint32_t x) {
  asm volatile("mov.b32 %0, %0;" : "+r"(x));
  return x;
}

// Shared-memory descriptors of the MMA operands, built once per CTA. Stage s
// of the K (V) ring is the stage-0 descriptor plus s * (kTileBytes >> 4) in
// the start-address field (bits 0-13, address >> 4); shared memory is below
// 256 KB, so no step carries out of the field. The MMA warp is the kernel's
// critical path and every instruction of its loop shows in the launch time,
// so nothing of this is recomputed per tile.
template <int D>
struct Descs {
  uint64_t q0, q1;  // Q tiles 0 and 1 (K-major)
  uint64_t k0;      // K ring stage 0 (K-major)
  uint64_t v0;      // V ring stage 0 (MN-major)
  __device__ __forceinline__ explicit Descs(uint32_t sbase) {
    using C = Cfg<D>;
    q0 = smem_desc(sbase + C::kOffQ, 16, 8 * C::kSwizzle, C::kLayout);
    q1 = smem_desc(sbase + C::kOffQ + C::kTileBytes, 16, 8 * C::kSwizzle, C::kLayout);
    k0 = smem_desc(sbase + C::kOffK, 16, 8 * C::kSwizzle, C::kLayout);
    v0 = smem_desc(sbase + C::kOffV, C::kChunkBytes, 8 * C::kSwizzle, C::kLayout);
  }
  static constexpr uint64_t kStageStep = static_cast<uint64_t>(Cfg<D>::kTileBytes >> 4);
};

// S_h = Q_h K^T: k-steps of 16 columns (32 bytes) inside a swizzle row; d =
// 128 has two 64-column chunks, kChunkBytes apart.
template <int D>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint64_t a0, uint64_t b0) {
  using C = Cfg<D>;
  if constexpr (D == 32) {
    mma_ss2<2>(d_tmem, a0, b0, C::kIdescS, 0u);
  } else {
    mma_ss4<2, 4, 6>(d_tmem, a0, b0, C::kIdescS, 0u);
    if constexpr (D == 128)
      mma_ss4<2, 4, 6>(d_tmem, a0 + (C::kChunkBytes >> 4), b0 + (C::kChunkBytes >> 4), C::kIdescS,
                       1u);
  }
}

// O_h += P_h[:, keys of `part`] V_j[keys of `part`, :], part 0 = keys 0-63, 1 =
// keys 64-127. V is [key, d] with d contiguous: the B operand (K = keys, N = d)
// is MN-major; 16 keys = 16 rows of kSwizzle bytes (k-step ks: P columns
// 8 * ks, V descriptor + ks * kSwizzle).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t t_o, uint32_t t_p, uint64_t v_desc, int part,
                                         uint32_t accumulate) {
  using C = Cfg<D>;
  constexpr int kStep = C::kSwizzle;
  const int ks0 = part * (kBN / 32);
  mma_ts4<kStep, 2 * kStep, 3 * kStep>(t_o, t_p + ks0 * 8, v_desc + ks0 * kStep, C::kIdescO,
                                       accumulate);
}

// A ring position: stage index and the parity of its current phase, advanced
// without division.
template <int N>
struct RingPos {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void advance() {
    if (++s == N) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// One warp issues both products. P_h overwrites the first half of S_h, so
// S_h of the next tile follows P V of this one: per tile, P V_h(j) then
// S_h(j + 1) for each Q tile. The loops over the two Q tiles are unrolled, so
// that every per-Q-tile quantity (descriptors, TMEM columns, barrier
// addresses, phase bits) is a constant or a register of its own.
template <int D, int MASK>
__device__ void mma_role(const KernelParams& p, uint32_t sbase, const Bars& bars, uint32_t tmem,
                         const int64_t* cta_lo, const Ctl& ctl) {
  using C = Cfg<D>;
  constexpr bool kNa = mask_is_na(MASK);
  const Descs<D> dsc(sbase);
  uint32_t q_ph = 0;
  RingPos<C::kKStages> kr;
  RingPos<C::kVStages> vr;
  uint32_t p_par = 0;  // bit h: parity of Q tile h's next P phases
  uint32_t o_par = 0;  // bit h: parity of Q tile h's next O phase
  const bool twin = mask_is_na(MASK) && p.twin != 0;
  SegIter<MASK> it(p, cta_lo);
  Seg sg;
  while (it.next(p, sg)) {
    const Task tk = decode_task<MASK>(sg.t, p);
    const Band band = task_band<MASK>(tk, p);
    if (!ctl_wait(bars.q_full(), q_ph, ctl, -1, kRoleMma)) goto drain;
    q_ph ^= 1u;
    tc_fence_after();
    uint32_t o_ready = 0;  // bit h: O_h holds this task's partial sum
    // The next K/V tile after `from` and, in `act`, the Q tiles that need it
    // (bit h). Unmasked: every tile of the segment, for every live Q tile.
    // Neighbourhood masks: the cursor's search; others: the tile test.
    TileCursor<MASK> cur(band, 2, twin_mode<MASK>(p));
    const uint32_t live = (tk.live[0] ? 1u : 0u) | (tk.live[1] ? 2u : 0u);
    auto step = [&](int from, uint32_t& act) -> int {
      if constexpr (MASK == kMaskNone) {
        act = live;
        return from + 1;
      } else if constexpr (kNa) {
        bool a[2];
        const int t = cur.next(tk, sg.kv1, a, p);
        act = (a[0] ? 1u : 0u) | (a[1] ? 2u : 0u);
        return t;
      } else {
        const int t = next_tile<MASK>(tk, band, from, sg.kv1, p);
        act = t < sg.kv1 ? ((tile_active<MASK>(tk, 0, t, p) ? 1u : 0u) |
                            (tile_active<MASK>(tk, 1, t, p) ? 2u : 0u))
                         : 0u;
        return t;
      }
    };
    uint32_t aj = 0, an = 0;
    int j = step(sg.kv0 - 1, aj);
    if constexpr (MASK != kMaskNone) {
      // a task without a K/V tile (a Q tile of rows that see no key) is done with Q at once
      if (j >= sg.kv1) mma_commit(bars.q_empty());
    }
    if (j < sg.kv1) {
      if (!ctl_wait(bars.k_full(kr.s), kr.ph, ctl, j, kRoleMma)) goto drain;
      tc_fence_after();
      const uint64_t kd = dsc.k0 + kr.s * Descs<D>::kStageStep;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        if ((aj >> h) & 1u) {
          issue_s<D>(tmem + C::tm_s(h), h ? dsc.q1 : dsc.q0, kd);
          mma_commit(bars.s_full(h));
        }
      mma_commit(bars.k_empty(kr.s));
      kr.advance();
    }
    while (j < sg.kv1) {
      const int jn = step(j, an);
      const bool has_next = jn < sg.kv1;
      if (!has_next) mma_commit(bars.q_empty());  // every S of the task is issued
      bool k_taken = false;
      uint32_t early = 0;
      if constexpr (kNa) {
        // Twin tasks: this tile is one warpgroup's, the next the other's, so
        // the next S waits for nothing of this tile's softmax; it goes first,
        // and the tensor core runs it while this tile's P is computed.
        if (twin && has_next) {
          early = an;
          if (!ctl_wait(bars.k_full(kr.s), kr.ph, ctl, jn, kRoleMma)) goto drain;
          tc_fence_after();
          k_taken = true;
          const bool h1 = an == 2u;
          issue_s<D>(tmem + (h1 ? C::tm_s(1) : C::tm_s(0)), h1 ? dsc.q1 : dsc.q0,
                     dsc.k0 + kr.s * Descs<D>::kStageStep);
          mma_commit(h1 ? bars.s_full(1) : bars.s_full(0));
        }
      }
      if (!ctl_wait(bars.v_full(vr.s), vr.ph, ctl, j, kRoleMma)) goto drain;
      tc_fence_after();
      const uint64_t vd = dsc.v0 + vr.s * Descs<D>::kStageStep;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if ((aj >> h) & 1u) {
          if (!((o_ready >> h) & 1u)) {
            if (!ctl_wait(bars.o_empty(h), ((o_par >> h) & 1u) ^ 1u, ctl, j, kRoleMma)) goto drain;
          }
          const uint32_t par = (p_par >> h) & 1u;
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            if (!ctl_wait(bars.p_full(h, part), par, ctl, j, kRoleMma)) goto drain;
            tc_fence_after();
            issue_pv<D>(tmem + C::tm_o(h), tmem + C::tm_p(h), vd, part,
                        (((o_ready >> h) & 1u) != 0u || part > 0) ? 1u : 0u);
          }
          p_par ^= 1u << h;
          o_ready |= 1u << h;
        }
        if (has_next && ((an >> h) & 1u) && !((early >> h) & 1u)) {
          if (!k_taken) {
            if (!ctl_wait(bars.k_full(kr.s), kr.ph, ctl, jn, kRoleMma)) goto drain;
            tc_fence_after();
            k_taken = true;
          }
          issue_s<D>(tmem + C::tm_s(h), h ? dsc.q1 : dsc.q0, dsc.k0 + kr.s * Descs<D>::kStageStep);
          mma_commit(bars.s_full(h));
        }
      }
      mma_commit(bars.v_empty(vr.s));
      vr.advance();
      if (k_taken) {
        mma_commit(bars.k_empty(kr.s));
        kr.advance();
      }
      j = jn;
      aj = an;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (!tk.live[h]) continue;
      if (!((o_ready >> h) & 1u)) {  // keeps the o_empty phases in step even without a PV
        if (!ctl_wait(bars.o_empty(h), ((o_par >> h) & 1u) ^ 1u, ctl, -1, kRoleMma)) goto drain;
      }
      mma_commit(bars.o_full(h));
      o_par ^= 1u << h;
    }
  }
drain:
  // Every MMA this thread issued must be complete before TMEM is freed.
  mma_commit(bars.done());
  ctl_wait(bars.done(), 0, ctl, -1, kRoleMma, false);
}

// ------------------------------------------------------------- partial results

// Orders this thread's earlier global writes before, or its later global
// reads after, a flag observed by another CTA (release / acquire, GPU scope).
__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// A 64-bit load with acquire semantics at GPU scope.
__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* a) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
  return v;
}

// A 64-bit load with relaxed semantics at GPU scope (an acquire fence after it
// orders the reads that depend on what it saw).
__device__ __forceinline__ unsigned long long ld_relaxed_gpu(const unsigned long long* a) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
  return v;
}

// Stores a warp's block of 32 output rows x 32 bf16 columns (64 bytes per
// row; the lane's own row in pk). Storing each lane's row as it stands would
// make every 16-byte store instruction touch 32 rows; instead the four lanes
// 4g..4g+3 first trade 16-byte chunks (a rotation by the lane's index, four
// shuffle rounds, the opposite rotation), after which lane 4g + c holds
// chunk c of rows 4g..4g+3, and store k writes eight whole 64-byte row
// segments (row 4g + k of each group). `seg` points at column 0 of the
// block's row 0, `stride` is the row stride in elements; rows from `rows`
// on are not written. Called by all 32 lanes.
__device__ __forceinline__ void store_rows32(const uint32_t (&pk)[16], __nv_bfloat16* seg,
                                             int64_t stride, int rows) {
  const int lane = threadIdx.x & 31, c = lane & 3, g4 = lane & ~3;
  uint32_t a[4][4], b[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int w = 0; w < 4; ++w) a[i][w] = pk[4 * i + w];
  // chunk i of the rotated row: chunk (i + c) mod 4
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int w = 0; w < 4; ++w) b[i][w] = (c & 1) ? a[(i + 1) & 3][w] : a[i][w];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int w = 0; w < 4; ++w) a[i][w] = (c & 2) ? b[(i + 2) & 3][w] : b[i][w];
  // round i: from lane g4 + (c - i) mod 4, whose rotated chunk i is its chunk c
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int src = g4 | ((c - i) & 3);
#pragma unroll
    for (int w = 0; w < 4; ++w) b[i][w] = __shfl_sync(0xffffffffu, a[i][w], src);
  }
  // b[i] is chunk c of row g4 + (c - i) mod 4; put row g4 + k at index k
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int w = 0; w < 4; ++w) a[r][w] = (c & 1) ? b[(1 - r) & 3][w] : b[(4 - r) & 3][w];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int w = 0; w < 4; ++w) b[r][w] = (c & 2) ? a[(r + 2) & 3][w] : a[r][w];
#pragma unroll
  for (int r = 0; r < 4; ++r)
    if (g4 + r < rows)
      __stcs(reinterpret_cast<uint4*>(seg + (g4 + r) * stride + c * 8),
             make_uint4(b[r][0], b[r][1], b[r][2], b[r][3]));
}

// A 32-row quarter of a part slot: [D/4][32 rows] float4, then m[32], l[32].
// CTA `cta` keeps two slots per Q tile: one for its first segment (`head`),
// one for its last.
template <int D>
__device__ __forceinline__ float* part_slot(const KernelParams& p, int cta, bool head, int hh,
                                            int quarter) {
  return p.ws_part + static_cast<int64_t>((2 * cta + (head ? 0 : 1)) * 2 + hh) * 128 * (D + 2) +
         quarter * 32 * (D + 2);
}

// Arrival word of (task t, Q tile hh, 32-row quarter).
__device__ __forceinline__ unsigned long long* arrival_word(const KernelParams& p, int t, int hh,
                                                            int quarter) {
  return p.ws_count + (2 * static_cast<int64_t>(t) + hh) * 4 + quarter;
}

// The CTAs [c_lo, c_hi] holding the parts of task t under the split
// schedule: they are adjacent (CTA c covers units [cta_lo[c], cta_lo[c + 1]),
// and no range is empty), so walk out from this CTA to the first and last.
__device__ __forceinline__ void cut_span(const KernelParams& p, const int64_t* cta_lo, int t,
                                         int& c_lo, int& c_hi) {
  const int64_t t_first = static_cast<int64_t>(t) * p.n_kv;
  c_lo = c_hi = blockIdx.x;
  while (c_lo > 0 && cta_lo[c_lo] > t_first) --c_lo;
  while (c_hi + 1 < static_cast<int>(gridDim.x) && cta_lo[c_hi + 1] < t_first + p.n_kv) ++c_hi;
}

// The merge of a task cut in two parts, by the part that finishes last: this
// part's unnormalised O (TMEM), maximum m_ref and row sum l, with the other
// part's mi, li and O row (float4 column group g from oth(g)); the lower
// CTA's part comes first in every sum, so either part computes the same
// bits. Writes the bf16 row and the log-sum-exp and hands O_h back to the
// MMA warp. O_h must be complete (o_full seen).
template <int D, typename Oth>
__device__ __forceinline__ void merge_two(const KernelParams& p, const Bars& bars, const Task& tk,
                                          int hh, int row, uint32_t t_o, float m_ref, float l,
                                          float mi, float li, bool me_lo, Oth oth) {
  const int lane = threadIdx.x & 31;
  const int q = tk.q0[hh] + row;
  const bool row_ok = q < p.Nq;
  const int q_blk = q - lane;  // the warp's first row
  __nv_bfloat16* seg = reinterpret_cast<__nv_bfloat16*>(p.o) + tk.b * p.o_sb + tk.h * p.o_sh +
                       static_cast<int64_t>(q_blk) * p.o_sn;
  const float M = fmaxf(m_ref, mi);
  const float w_me = m_ref == -CUDART_INF_F ? 0.f : ex2(m_ref - M);
  const float w_ot = mi == -CUDART_INF_F ? 0.f : ex2(mi - M);
  const float w_lo = me_lo ? w_me : w_ot, w_hi = me_lo ? w_ot : w_me;
  const float L = __fmaf_rn(me_lo ? li : l, w_hi, __fmul_rn(me_lo ? l : li, w_lo));
  const float inv_L = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int ch = 0; ch < D / 32; ++ch) {
    uint32_t ov[32];
    tmem_ld32(t_o + ch * 32, ov);
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = oth(ch * 8 + i);
    auto mix = [&](float own, float other) {
      return __fmaf_rn(w_hi, me_lo ? other : own, __fmul_rn(w_lo, me_lo ? own : other)) * inv_L;
    };
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      packed[2 * i] = pack_bf16(mix(__uint_as_float(ov[4 * i]), v[i].x),
                                mix(__uint_as_float(ov[4 * i + 1]), v[i].y));
      packed[2 * i + 1] = pack_bf16(mix(__uint_as_float(ov[4 * i + 2]), v[i].z),
                                    mix(__uint_as_float(ov[4 * i + 3]), v[i].w));
    }
    store_rows32(packed, seg + ch * 32, p.o_sn, p.Nq - q_blk);
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bars.o_empty(hh));
  if (row_ok && p.lse != nullptr) {
    const float lse = L > 0.f ? (M + __log2f(L)) * 0.69314718055994530942f : -CUDART_INF_F;
    __stcs(p.lse + static_cast<int64_t>(tk.bh) * p.Nq + q, lse);
  }
}

// One arrival on a (task, Q tile) word tagged with this call's epoch; returns
// the number of parts arrived so far in this call, or 0 if the CAS loop ran
// past its bound (recorded as a timeout). The first attempt assumes this is
// the call's first arrival, which saves a round trip for the first part.
__device__ __forceinline__ uint32_t arrive_part(unsigned long long* w, uint32_t epoch,
                                                const Ctl& c) {
  unsigned long long assumed = static_cast<unsigned long long>(epoch) << 32;
  for (int n = 0; n < (1 << 20); ++n) {
    const uint32_t cnt = static_cast<uint32_t>(assumed >> 32) == epoch
                             ? static_cast<uint32_t>(assumed) : 0u;
    const unsigned long long nv = (static_cast<unsigned long long>(epoch) << 32) | (cnt + 1u);
    const unsigned long long old = atomicCAS(w, assumed, nv);
    if (old == assumed) return cnt + 1u;
    assumed = old;
  }
  report_timeout(c.abort, c.status, kRoleSoftmax, -2);
  return 0u;
}

// Epilogue of a task cut between CTAs. Each warp handles its 32 rows on its
// own. It first reads the rows' arrival word: if every other part has
// arrived already (the usual case for the part a CTA works on last), it
// merges at once, without storing its own part. Otherwise it writes this part
// (unnormalised O, the running maximum m in log2 units, the row sum l),
// counts the part on the arrival word, and if that makes it the last part of
// those rows, merges all parts:
//   M = max_i m_i,  L = sum_i 2^(m_i - M) l_i,  O = sum_i 2^(m_i - M) O_i / L,
//   LSE = ln 2 (M + log2 L).
// No CTA waits for another: the last part to finish does the merge, reading
// its own O from TMEM (o_empty is arrived only at the end, which costs
// nothing: the next task's first P V also needs this warpgroup's next P).
// A part is stored per 32-row quarter, [d/4][32 rows] of float4, then m[32]
// and l[32], so that every warp access is one contiguous 512-byte run.
// Inlined into the softmax loop: as a call, the softmax warps saved their
// live registers to local memory around it and reloaded them from L2 after
// the epilogue's stores, measured ~2000 cycles per cut on GB300.
// False: the CTA is aborting.
template <int D>
__device__ __forceinline__ bool partial_epilogue(const KernelParams& p, const Bars& bars, const Seg& sg,
                                              const Task& tk, int hh, int row, uint32_t t_o,
                                              float m_ref, float l, const int64_t* cta_lo,
                                              uint32_t& o_par, const Ctl& ctl) {
  const int lane = threadIdx.x & 31;
  const int quarter = row >> 5;
  auto slot_of = [&](int cta, bool head) { return part_slot<D>(p, cta, head, hh, quarter); };
  auto release_o = [&]() {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.o_empty(hh));
  };
  const int64_t t_first = static_cast<int64_t>(sg.t) * p.n_kv;
  const int me = blockIdx.x;
  int c_lo, c_hi;
  cut_span(p, cta_lo, sg.t, c_lo, c_hi);
  const uint32_t n_parts = static_cast<uint32_t>(c_hi - c_lo + 1);
  // a part of CTA c is that CTA's first segment iff its range starts in this task
  auto part = [&](int c) -> const float* { return slot_of(c, cta_lo[c] >= t_first); };
  // Another part (every other part has been written by the time it is read)
  // stands in for the unused slots of a merge round, so that all of its loads
  // are in flight together and read this call's finite values; this CTA's
  // own slot may hold a previous call's data.
  const int stand_in = c_lo != me ? c_lo : c_hi;
  unsigned long long* word = arrival_word(p, sg.t, hh, quarter);
  // Every lane reads the arrival word (relaxed, one broadcast load) before O
  // is complete, so the read overlaps the last P V; if every other part is
  // in, an acquire fence orders the reads of those parts after it.
  const unsigned long long w0 = ld_relaxed_gpu(word);
  uint32_t seen = static_cast<uint32_t>(w0 >> 32) == p.epoch ? static_cast<uint32_t>(w0) : 0u;
  bool claim = seen + 1u == n_parts;
  if (!claim && sg.kv0 == 0) {
    // The first part of its task is this CTA's last segment, and the task's
    // other parts began earlier (at their CTAs' starts): read again, now
    // that this part is complete, before handing it on.
    const unsigned long long w1 = ld_relaxed_gpu(word);
    seen = static_cast<uint32_t>(w1 >> 32) == p.epoch ? static_cast<uint32_t>(w1) : 0u;
    claim = seen + 1u == n_parts;
  }
  if (claim) fence_gpu();
  const int q = tk.q0[hh] + row;
  const bool row_ok = q < p.Nq;
  if (claim && n_parts == 2) {
    // The usual cut: the other part is complete; fetch its m, l and its
    // first 64 columns of O while the last P V finishes, then merge.
    const float* sl = part(stand_in);
    const float mi = __ldcg(sl + 32 * D + lane);
    const float li = __ldcg(sl + 32 * D + 32 + lane);
    constexpr int kPre = D < 64 ? D / 4 : 16;  // float4 columns fetched ahead
    const float4* src = reinterpret_cast<const float4*>(sl);
    float4 pre[kPre];
#pragma unroll
    for (int i = 0; i < kPre; ++i) pre[i] = __ldcg(src + i * 32 + lane);
    if (!warp_wait(bars.o_full(hh), o_par, ctl, -1)) return false;
    o_par ^= 1u;
    tc_fence_after();
    merge_two<D>(p, bars, tk, hh, row, t_o, m_ref, l, mi, li, me == c_lo, [&](int g) {
      return g < kPre ? pre[g % kPre] : __ldcg(src + g * 32 + lane);
    });
    return !*ctl.abort;
  }
  if (!warp_wait(bars.o_full(hh), o_par, ctl, -1)) return false;
  o_par ^= 1u;
  tc_fence_after();
  if (!claim) {
    float* mine = slot_of(blockIdx.x, sg.head);
    float4* mine4 = reinterpret_cast<float4*>(mine);
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t ov[32];
      tmem_ld32(t_o + ch * 32, ov);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        mine4[(ch * 8 + i) * 32 + lane] =
            make_float4(__uint_as_float(ov[4 * i]), __uint_as_float(ov[4 * i + 1]),
                        __uint_as_float(ov[4 * i + 2]), __uint_as_float(ov[4 * i + 3]));
    }
    mine[32 * D + lane] = m_ref;
    mine[32 * D + 32 + lane] = l;
    fence_gpu();
    __syncwarp();
    uint32_t n = 0;
    if (lane == 0) n = arrive_part(word, p.epoch, ctl);
    n = __shfl_sync(0xffffffffu, n, 0);
    if (n != n_parts) {
      release_o();
      return !*ctl.abort;
    }
    fence_gpu();  // the other lanes' reads of the other parts come after lane 0's arrival
  }
  // The merge sums the parts in CTA order (this part at its own place), so
  // the result has the same bits whichever part does it. M first: the
  // largest m of all parts (exact in any order); then L.
  float M = m_ref;
  float L = 0.f;
  if (c_hi - c_lo < 8) {  // every part in one round: m and l stay in registers
    float mi[8], li[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = c_lo + u;
      const float* sl = part(c <= c_hi && c != me ? c : stand_in);
      mi[u] = __ldcg(sl + 32 * D + lane);
      li[u] = __ldcg(sl + 32 * D + 32 + lane);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (c_lo + u <= c_hi && c_lo + u != me) M = fmaxf(M, mi[u]);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = c_lo + u;
      const float mc = c == me ? m_ref : mi[u];
      if (c <= c_hi && mc != -CUDART_INF_F) L = __fmaf_rn(c == me ? l : li[u], ex2(mc - M), L);
    }
  } else {  // more parts: the maximum first, then L
    for (int c0 = c_lo; c0 <= c_hi; c0 += 8) {
      float mi[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u;
        mi[u] = __ldcg(part(c <= c_hi && c != me ? c : stand_in) + 32 * D + lane);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c0 + u <= c_hi && c0 + u != me) M = fmaxf(M, mi[u]);
    }
    for (int c0 = c_lo; c0 <= c_hi; c0 += 8) {
      float mi[8], li[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u;
        const float* sl = part(c <= c_hi && c != me ? c : stand_in);
        mi[u] = __ldcg(sl + 32 * D + lane);
        li[u] = __ldcg(sl + 32 * D + 32 + lane);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u;
        const float mc = c == me ? m_ref : mi[u];
        if (c <= c_hi && mc != -CUDART_INF_F) L = __fmaf_rn(c == me ? l : li[u], ex2(mc - M), L);
      }
    }
  }
  const float inv_L = L > 0.f ? 1.f / L : 0.f;
  const float w_me = (m_ref == -CUDART_INF_F) ? 0.f : ex2(m_ref - M);
  __nv_bfloat16* seg = reinterpret_cast<__nv_bfloat16*>(p.o) + tk.b * p.o_sb + tk.h * p.o_sh +
                       static_cast<int64_t>(q - lane) * p.o_sn;  // the warp's first row
  // O in chunks of 32 columns: this part's from TMEM, four parts' rows per round.
#pragma unroll 1
  for (int ch = 0; ch < D / 32; ++ch) {
    float acc[32], own[32];
    {
      uint32_t ov[32];
      tmem_ld32(t_o + ch * 32, ov);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        own[i] = __uint_as_float(ov[i]);
        acc[i] = 0.f;
      }
    }
#pragma unroll 1
    for (int c0 = c_lo; c0 <= c_hi; c0 += 4) {
      float4 v[4][8];
      float wgt[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u;
        const bool in = c <= c_hi && c != me;
        const float* sl = part(in ? c : stand_in);
        const float mi = __ldcg(sl + 32 * D + lane);
        wgt[u] = c == me ? w_me : (in && mi != -CUDART_INF_F) ? ex2(mi - M) : 0.f;
        const float4* src = reinterpret_cast<const float4*>(sl);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[u][i] = __ldcg(src + (ch * 8 + i) * 32 + lane);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool is_me = c0 + u == me;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[4 * i] = __fmaf_rn(wgt[u], is_me ? own[4 * i] : v[u][i].x, acc[4 * i]);
          acc[4 * i + 1] = __fmaf_rn(wgt[u], is_me ? own[4 * i + 1] : v[u][i].y, acc[4 * i + 1]);
          acc[4 * i + 2] = __fmaf_rn(wgt[u], is_me ? own[4 * i + 2] : v[u][i].z, acc[4 * i + 2]);
          acc[4 * i + 3] = __fmaf_rn(wgt[u], is_me ? own[4 * i + 3] : v[u][i].w, acc[4 * i + 3]);
        }
      }
    }
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) packed[i] = pack_bf16(acc[2 * i] * inv_L, acc[2 * i + 1] * inv_L);
    store_rows32(packed, seg + ch * 32, p.o_sn, p.Nq - (q - lane));
  }
  release_o();
  if (row_ok && p.lse != nullptr) {
    const float lse = L > 0.f ? (M + __log2f(L)) * 0.69314718055994530942f : -CUDART_INF_F;
    __stcs(p.lse + static_cast<int64_t>(tk.bh) * p.Nq + q, lse);
  }
  return !*ctl.abort;
}

// Warpgroup 0's end of a twin task: both halves' O (TMEM; O_1 from the
// other warpgroup's columns, same lanes), this half's m and l, the other's
// from the exchange. A half with no tile (m = -inf) is left out by a select,
// not a zero weight: its O columns may hold an earlier task's values.
// False: the CTA is aborting.
template <int D>
__device__ __forceinline__ bool twin_epilogue(const KernelParams& p, const Bars& bars, const Task& tk,
                                           int row, uint32_t t_o0, uint32_t t_o1, float m0,
                                           float l0, const float* xch, uint32_t& o_par,
                                           uint32_t& o_par1, uint32_t& x_par, const Ctl& ctl) {
  const int lane = threadIdx.x & 31;
  if (!warp_wait(bars.o_full(0), o_par, ctl, -1)) return false;
  o_par ^= 1u;
  if (!warp_wait(bars.o_full(1), o_par1, ctl, -1)) return false;
  o_par1 ^= 1u;
  if (!warp_wait(bars.x_full(), x_par, ctl, -1)) return false;
  x_par ^= 1u;
  tc_fence_after();
  const float m1 = xch[row], l1 = xch[kBM + row];
  __syncwarp();
  if (lane == 0) mbar_arrive(bars.x_empty());
  const float M = fmaxf(m0, m1);
  const bool h0 = m0 != -CUDART_INF_F, h1 = m1 != -CUDART_INF_F;
  const float w0 = h0 ? ex2(m0 - M) : 0.f, w1 = h1 ? ex2(m1 - M) : 0.f;
  const float L = __fmaf_rn(l1, w1, __fmul_rn(l0, w0));
  const float inv_L = L > 0.f ? 1.f / L : 0.f;
  const bool empty = !(L > 0.f);
  const int q = tk.q0[0] + row;
  __nv_bfloat16* seg = reinterpret_cast<__nv_bfloat16*>(p.o) + tk.b * p.o_sb + tk.h * p.o_sh +
                       static_cast<int64_t>(q - lane) * p.o_sn;  // the warp's first row
  auto mix = [&](uint32_t a, uint32_t b) {
    const float x = h0 ? __fmul_rn(__uint_as_float(a), w0) : 0.f;
    return (h1 ? __fmaf_rn(__uint_as_float(b), w1, x) : x) * inv_L;
  };
#pragma unroll
  for (int ch = 0; ch < D / 32; ++ch) {
    uint32_t oa[32], ob[32];
    tmem_ld32(t_o0 + ch * 32, oa);
    tmem_ld32(t_o1 + ch * 32, ob);
    if (ch == D / 32 - 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bars.o_empty(0));
        mbar_arrive(bars.o_empty(1));
      }
    }
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      packed[i] = empty ? 0u : pack_bf16(mix(oa[2 * i], ob[2 * i]), mix(oa[2 * i + 1], ob[2 * i + 1]));
    store_rows32(packed, seg + ch * 32, p.o_sn, p.Nq - (q - lane));
  }
  if (q < p.Nq && p.lse != nullptr) {
    const float lse = L > 0.f ? (M + __log2f(L)) * 0.69314718055994530942f : -CUDART_INF_F;
    __stcs(p.lse + static_cast<int64_t>(tk.bh) * p.Nq + q, lse);
  }
  return !*ctl.abort;
}

// Keys of a partial tile (class 2) that the query may not see become -inf.
template <int MASK>
__device__ __forceinline__ void mask_tile(uint32_t (&s)[128], const KernelParams& p, int j, int q,
                                          const NaQuery& nq) {
  const uint32_t neg_inf = __float_as_uint(-CUDART_INF_F);
  const int k0 = j * kBN;
  if (MASK == kMaskNone || mask_is_causal(MASK)) {
    int lim = p.Nk - 1 - k0;                       // last valid key column
    if (mask_is_causal(MASK)) lim = min(lim, q + causal_shift<MASK>(p) - k0);
#pragma unroll
    for (int i = 0; i < 128; ++i)
      if (i > lim) s[i] = neg_inf;
  } else {
    // The window is a product of a row set and a column set, and a K/V
    // tile covers whole grid-row segments: build the tile's allowed
    // keys as a 128-bit mask, one column interval per row segment,
    // then clear the rest with independent selects.
    uint32_t bits[4];
    if constexpr (MASK == kMaskNa3)
      na3_tile_bits(p, k0, nq, bits);
    else
      na_tile_bits<mask_na_wrap_rows(MASK), mask_na_wrap_cols(MASK), mask_na_dilated(MASK)>(
          p, k0, nq.qy, nq.qx, nq.wy, nq.wx, bits);
#pragma unroll
    for (int i = 0; i < 128; ++i)
      if (((bits[i >> 5] >> (i & 31)) & 1u) == 0u) s[i] = neg_inf;
  }
}

// Row maximum of a tile (fp32 bit patterns): 8 independent chains of 3-input max.
__device__ __forceinline__ float row_max128(const uint32_t (&s)[128]) {
  float mx8[8];
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    mx8[ch] = fmaxf(__uint_as_float(s[ch]), __uint_as_float(s[ch + 8]));
#pragma unroll
    for (int i = 16; i < 128; i += 16)
      mx8[ch] = fmax3(mx8[ch], __uint_as_float(s[ch + i]), __uint_as_float(s[ch + i + 8]));
  }
  return fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
}

// O row *= alpha (the accumulated P V of earlier tiles, brought to a new maximum).
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t t_o, float alpha) {
#pragma unroll
  for (int ch = 0; ch < D / 32; ++ch) {
    uint32_t ov[32];
    tmem_ld32(t_o + ch * 32, ov);
#pragma unroll
    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
    tmem_st32(t_o + ch * 32, ov);
  }
}

template <int D, int MASK>
__device__ void softmax_role(const KernelParams& p, const Bars& bars, uint32_t tmem,
                             const int64_t* cta_lo, float* xch, const Ctl& ctl) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hh = (warp - 4) >> 2;          // which Q tile of the pair
  const int quarter = warp & 3;            // TMEM lanes this warp may access
  const int row = quarter * 32 + lane;     // query row inside the Q tile
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  const uint32_t t_s = lane_base + C::tm_s(hh);
  const uint32_t t_o = lane_base + C::tm_o(hh);
  const uint32_t t_p = lane_base + C::tm_p(hh);
  const float c = p.c;
  uint32_t s_par = 0, o_par = 0;
  const bool twin = twin_mode<MASK>(p);
  uint32_t o_par1 = 0, x_par = 0;  // twin tasks: warpgroup 0's view of O_1, the exchange

  grid_dep_wait();  // before the first global store (O, LSE, partial results)
  SegIter<MASK> it(p, cta_lo);
  Seg sg;
  while (it.next(p, sg)) {
    const Task tk = decode_task<MASK>(sg.t, p);
    if (!tk.live[hh]) continue;
    const int q0 = tk.q0[hh];
    const int q = q0 + row;
    // neighbourhood: this query's grid coordinates and window starts
    const NaQuery nq = na_query<MASK>(p, q);
    const bool cut = MASK == kMaskNone && p.split && (sg.kv0 > 0 || sg.kv1 < p.n_kv);
    float m_ref = -CUDART_INF_F;  // running maximum in log2 units (possibly stale by < 2^8)
    float l = 0.f;                // running row sum relative to m_ref
    bool first = true;
    // P overwrites the first half of S, and each half of P is announced on
    // its own so that P V starts on the first.
    // neighbourhood masks: the tiles the cursor finds for this Q tile (class 2)
    constexpr bool kNa = mask_is_na(MASK);
    TileCursor<MASK> cur(task_band<MASK>(tk, p), hh, twin);
    bool act[2];
    for (int j = kNa ? cur.next(tk, sg.kv1, act, p) : sg.kv0; j < sg.kv1;
         j = kNa ? cur.next(tk, sg.kv1, act, p) : j + 1) {
      const int cls = kNa ? 2 : tile_class<MASK>(q0, j, p);
      if (cls == 0) continue;
      if (!warp_wait(bars.s_full(hh), s_par, ctl, j)) return;
      s_par ^= 1u;
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld128(t_s, sr);
      if (cls == 2) mask_tile<MASK>(sr, p, j, q, nq);
      const float mx = row_max128(sr);
      float s[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(sr[i]);
      const float m_tile = (mx == -CUDART_INF_F) ? -CUDART_INF_F : mx * c;
      const bool grow = m_tile > m_ref + kRescaleLog2;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2(m_ref - m_tile);  // 0 while m_ref is still -inf
        l *= alpha;
        m_ref = m_tile;
      }
      // O holds the previous tiles' P V, whose MMAs completed before this S
      // was committed: bring it to the new maximum before the next P V.
      if (__any_sync(0xffffffffu, grow && !first)) rescale_o<D>(t_o, alpha);
      const float neg_m = (m_ref == -CUDART_INF_F) ? 0.f : -m_ref;
      const float2 c2 = make_float2(c, c), nm2 = make_float2(neg_m, neg_m);
      float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
      // The first half's store completes while the second half's
      // exponentials are computed (tcgen05.wait::st waits for every store of
      // the thread); then each half is announced on its own barrier.
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = 64 * part + 2 * i;
          const float2 x = __ffma2_rn(make_float2(s[e], s[e + 1]), c2, nm2);
          const float2 pe = make_float2(ex2(x.x), ex2(x.y));
          sum4[i & 3] = __fadd2_rn(sum4[i & 3], pe);
          pk[i] = pack_bf16(pe.x, pe.y);
        }
        if (part == 1) {
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.p_full(hh, 0));
        }
        tmem_st32(t_p + 32 * part, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.p_full(hh, 1));
      const float2 sa = __fadd2_rn(sum4[0], sum4[1]), sb = __fadd2_rn(sum4[2], sum4[3]);
      l += (sa.x + sa.y) + (sb.x + sb.y);
      first = false;
    }
    if (twin) {
      if (hh == 1) {
        // this half's m and l to warpgroup 0, which merges both halves and
        // hands O_1 back to the MMA warp
        if (!warp_wait(bars.x_empty(), x_par ^ 1u, ctl, -1)) return;
        x_par ^= 1u;
        xch[row] = m_ref;
        xch[kBM + row] = l;
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.x_full());
        continue;
      }
      if (!twin_epilogue<D>(p, bars, tk, row, t_o, lane_base + C::tm_o(1), m_ref, l, xch, o_par,
                            o_par1, x_par, ctl))
        return;
      continue;
    }
    // epilogue: O / l, bf16 store, log-sum-exp
    if (cut) {
      if (!partial_epilogue<D>(p, bars, sg, tk, hh, row, t_o, m_ref, l, cta_lo, o_par, ctl)) return;
      continue;
    }
    if (!warp_wait(bars.o_full(hh), o_par, ctl, -1)) return;
    o_par ^= 1u;
    tc_fence_after();
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    // a row that saw no key (bottom-right causal with Nq > Nk) is 0: O in
    // TMEM may never have been written for it
    const bool empty = !(l > 0.f);
    const bool row_ok = q < p.Nq;
    __nv_bfloat16* seg = reinterpret_cast<__nv_bfloat16*>(p.o) + tk.b * p.o_sb + tk.h * p.o_sh +
                         static_cast<int64_t>(q - lane) * p.o_sn;  // the warp's first row
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t ov[32];
      tmem_ld32(t_o + ch * 32, ov);
      if (ch == D / 32 - 1) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.o_empty(hh));
      }
      uint32_t packed[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        packed[i] = empty ? 0u
                          : pack_bf16(__uint_as_float(ov[2 * i]) * inv_l,
                                      __uint_as_float(ov[2 * i + 1]) * inv_l);
      store_rows32(packed, seg + ch * 32, p.o_sn, p.Nq - (q - lane));
    }
    if (row_ok && p.lse != nullptr) {
      const float lse = l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994530942f : -CUDART_INF_F;
      __stcs(p.lse + static_cast<int64_t>(tk.bh) * p.Nq + q, lse);
    }
  }
}

// ---------------------------------------------------------------- kernel

template <int D, int MASK>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ KernelParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  Bars bars{sbase + C::kOffBar, C::kKStages, C::kVStages};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 8 * bars.count());
  volatile uint32_t* abort_flag = tmem_slot + 1;
  int64_t* cta_lo = reinterpret_cast<int64_t*>(smem + C::kOffTbl);
  if (MASK == kMaskNone && p.split) {
    for (int c = threadIdx.x; c <= static_cast<int>(gridDim.x); c += blockDim.x)
      cta_lo[c] = unit_lo(p.units, gridDim.x, c);  // ordered by the __syncthreads below
    if (threadIdx.x == 0) {
      const int64_t u0 = unit_lo(p.units, gridDim.x, blockIdx.x);
      const int64_t t0 = u0 / p.n_kv;
      cta_lo[kMaxSplitCtas + 1] = (t0 << 32) | (u0 - t0 * p.n_kv);
    }
  }

  if (threadIdx.x == 0) {
    mbar_init(bars.q_full(), 1);
    mbar_init(bars.q_empty(), 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(bars.s_full(h), 1);
      mbar_init(bars.p_full(h, 0), 4);   // one arrive per softmax warp
      mbar_init(bars.p_full(h, 1), 4);
      mbar_init(bars.o_full(h), 1);
      mbar_init(bars.o_empty(h), 4);
    }
    mbar_init(bars.done(), 1);
    mbar_init(bars.x_full(), 4);   // one arrive per warp of warpgroup 1
    mbar_init(bars.x_empty(), 4);  // one arrive per warp of warpgroup 0
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(bars.k_full(s), 1);
      mbar_init(bars.k_empty(s), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(bars.v_full(s), 1);
      mbar_init(bars.v_empty(s), 1);
    }
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};
  // Everything above touches only this CTA's shared memory and TMEM; the next
  // launch's CTAs may start on the SMs this grid leaves. The loader and the
  // softmax warps wait for the previous kernel on the stream to complete
  // before their first global access (grid_dep_wait); the MMA warp reads only
  // what the loader's copies brought in.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp < 4) {
    // warpgroup 0 needs few registers; the softmax warpgroups take them
    set_max_regs_dec<kRegsControl>();
    if (warp == 0) {
      loader_role<D, MASK>(p, sbase, bars, cta_lo, ctl);    // whole warp, elected lane issues
    } else if (warp == 1) {
      mma_role<D, MASK>(p, sbase, bars, tmem, cta_lo, ctl);  // whole warp, elected lane issues
    }
    __syncwarp();
  } else {
    set_max_regs_inc<kRegsSoftmax>();
    softmax_role<D, MASK>(p, bars, tmem, cta_lo, reinterpret_cast<float*>(cta_lo), ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- launch

constexpr int kMinSmemBytes = 116 * 1024;  // more than half an SM: one CTA (and one TMEM owner) per SM

template <int D>
constexpr int smem_request() {
  return Cfg<D>::kSmemBytes > kMinSmemBytes ? Cfg<D>::kSmemBytes : kMinSmemBytes;
}

// A twin task pays an exchange and a merge (~2K cycles) to halve its K/V
// chain. Measured on GB300: a gain with ~10 tiles a Q tile (16^3 volume,
// window 5: 8 %), a loss with 5 (64 x 64 grid, window 7: 2-3 %).
constexpr int kTwinMinTiles = 8;

// Whether a neighbourhood launch with one Q tile per task runs its tasks as
// twins: the K/V tiles of a task from the middle of head 0, counted on the host.
template <int MASK>
bool twin_worthwhile(const KernelParams& p) {
  if (!mask_is_na(MASK) || p.q_tiles != 1 || p.n_qtasks <= 0 || p.twin != 0) return false;
  const Task tk = decode_task<MASK>(p.n_qtasks / 2, p);
  const Band band = task_band<MASK>(tk, p);
  int n = 0;
  for (int j = next_tile<MASK>(tk, band, -1, p.n_kv, p); j < p.n_kv && n < kTwinMinTiles;
       j = next_tile<MASK>(tk, band, j, p.n_kv, p))
    ++n;
  return n >= kTwinMinTiles;
}

template <int D, int MASK>
cudaError_t launch_mask(const KernelParams& p, int grid, cudaStream_t s) {
  auto kern = attn_fwd_kernel<D, MASK>;
  const int smem = smem_request<D>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: the CTAs of this launch may start (shared
  // memory, barriers, TMEM) while the previous kernel on the stream finishes;
  // they wait for its completion before their first global memory access.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

inline int twin_dim(const KernelParams& p, int mask) {
  switch (mask) {
    case kMaskNa + 0: return twin_worthwhile<kMaskNa + 0>(p);
    case kMaskNa + 1: return twin_worthwhile<kMaskNa + 1>(p);
    case kMaskNa + 2: return twin_worthwhile<kMaskNa + 2>(p);
    case kMaskNa + 3: return twin_worthwhile<kMaskNa + 3>(p);
    case kMaskNa + 4: return twin_worthwhile<kMaskNa + 4>(p);
    case kMaskNa + 5: return twin_worthwhile<kMaskNa + 5>(p);
    case kMaskNa + 6: return twin_worthwhile<kMaskNa + 6>(p);
    case kMaskNa + 7: return twin_worthwhile<kMaskNa + 7>(p);
    case kMaskNa3: return twin_worthwhile<kMaskNa3>(p);
    default: return 0;
  }
}

template <int D>
cudaError_t launch_dim(const KernelParams& p, int mask, int grid, cudaStream_t s) {
  switch (mask) {
    case kMaskNone: return launch_mask<D, kMaskNone>(p, grid, s);
    case kMaskCausal: return launch_mask<D, kMaskCausal>(p, grid, s);
    case kMaskCausalBR: return launch_mask<D, kMaskCausalBR>(p, grid, s);
    case kMaskNa + 0: return launch_mask<D, kMaskNa + 0>(p, grid, s);
    case kMaskNa + 1: return launch_mask<D, kMaskNa + 1>(p, grid, s);
    case kMaskNa + 2: return launch_mask<D, kMaskNa + 2>(p, grid, s);
    case kMaskNa + 3: return launch_mask<D, kMaskNa + 3>(p, grid, s);
    case kMaskNa + 4: return launch_mask<D, kMaskNa + 4>(p, grid, s);
    case kMaskNa + 5: return launch_mask<D, kMaskNa + 5>(p, grid, s);
    case kMaskNa + 6: return launch_mask<D, kMaskNa + 6>(p, grid, s);
    case kMaskNa + 7: return launch_mask<D, kMaskNa + 7>(p, grid, s);
    case kMaskNa3: return launch_mask<D, kMaskNa3>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dev
}  // namespace attn
