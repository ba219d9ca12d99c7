// device_common.cuh -- loads, conversions and workspace layout shared by the
// verify kernels (sm_103a).  Host-visible parts are plain structs.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace specv {

constexpr int kThreads = 256;           // threads per CTA in every kernel
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;          // portable cluster size
constexpr int kMaxTiles = 1024;         // tiles of kThreads vectors per CTA segment

// Device status bits (same values as the public header's SPEC_DATA_* and
// SPEC_DEVICE_WAIT_TIMEOUT).
constexpr int kDataTokenRange = 1;
constexpr int kDataNonfiniteLogit = 2;
constexpr int kDataUniformRange = 4;
constexpr int kWaitTimeout = 8;
// Bound on the polls of one mbarrier wait (each poll may suspend the thread
// for a short hardware-defined time); past it the kernel reports
// kWaitTimeout instead of waiting forever.
constexpr unsigned int kMaxPolls = 1u << 22;
// Debug builds (-DSPEC_DEBUG) only: an index check on a kernel's global
// access failed; the access was skipped (public SPEC_DEBUG_BOUNDS).
constexpr int kDebugBounds = 32;
// Per-sequence boundary flags (public SPEC_FLAG_*).
constexpr uint32_t kFlagRatio = 1;
constexpr uint32_t kFlagCdf = 2;

// Per-sequence state in the workspace.  Zero at rest: the kernel that
// finalises a sequence puts every field back to zero.
struct __align__(32) SeqState {
  unsigned int arrivals;          // rows (sampling) or CTAs (greedy) done
  unsigned int pad0;
  unsigned long long reject_mask; // bit i: draft position i was rejected
  unsigned long long near_mask;   // bit i: accept test i was within 1e-6
  unsigned long long row_word;    // greedy, one CTA per row: rows done << 48 | mismatch bits
};
static_assert(sizeof(SeqState) == 32, "SeqState layout");

// One per row (B*(K+1) of them) after SeqState[B].  Zero at rest.
struct __align__(16) RowSlot {
  unsigned long long value;  // sampling: candidate token (low 31 bits) | CDF-near bit 31
                             // greedy:   packed (orderable max, ~index) argmax key
  unsigned int spare;        // unused (zero)
  unsigned int pad;
};
static_assert(sizeof(RowSlot) == 16, "RowSlot layout");

// Partial softmax normalisers of one work unit (a segment of a target row
// and of the matching draft row) of the sampling kernel, relative to scaled
// offsets: target (ms_t, z_t), draft (ms_d, z_d).
struct __align__(16) Partial {
  float ms_t, z_t, ms_d, z_d;
};

// Work units of the fused sampling kernel: each draft position's (target,
// draft) row pair is cut into segments of kFusedSeg 16-byte vectors, the bonus
// target row into segments of twice that; a sequence has
// fused_tasks_per_seq(K, nvec) of them and the workspace one Partial each.
constexpr int kFusedSeg = 4096;
inline long long fused_tasks_per_seq(long long K, long long nvec) {
  const long long segs = (nvec + kFusedSeg - 1) / kFusedSeg;
  const long long segs_b = (nvec + 2 * kFusedSeg - 1) / (2 * kFusedSeg);
  return K * segs + segs_b;
}

// Claim counters of the fused sampling kernel.  Zero at rest: the last CTA
// to finish puts them back.
struct __align__(16) FusedCtl {
  unsigned long long next_task;  // next work unit to hand out
  unsigned long long done_ctas;  // CTAs that have taken their last unit
  unsigned int pending;          // early exit: sequences that accepted x_0
  unsigned int pad[3];           // pad[0]: early exit, phase-2 CTAs finished
};

// Most ranges the two-kernel sampler's streaming pass cuts the rows into.
// Its partials need at most kMaxStreamCtas + rows slots (range c of row pair
// p writes slot c + p).
constexpr long long kMaxStreamCtas = 4096;

// Workspace layout: SeqState[B] | units | FusedCtl, 16-byte aligned parts,
// where `units` is RowSlot[B*(K+1)] (greedy kernel, streaming sampler),
// Partial[B * tasks_per_seq] (fused sampler) or Partial[kMaxStreamCtas +
// B*(K+1) + 1] (two-kernel sampler).  One call uses one view and leaves
// everything zero-filled, so the views can share the region.  Sizes use
// 16-byte vectors of the row (ceil(V*bytes/16)).
struct WorkspaceLayout {
  size_t seq, units, ctl, total;
};
inline WorkspaceLayout workspace_layout(long long B, long long K, long long V, int elem_bytes) {
  const size_t R = (size_t)B * (size_t)(K + 1);
  const long long nvec = (V * elem_bytes + 15) / 16;
  const size_t P = (size_t)B * (size_t)fused_tasks_per_seq(K, nvec);
  WorkspaceLayout l;
  l.seq = 0;
  l.units = l.seq + (size_t)B * sizeof(SeqState);
  size_t ub = R * sizeof(RowSlot);
  if (P * sizeof(Partial) > ub) ub = P * sizeof(Partial);
  if (((size_t)kMaxStreamCtas + R + 1) * sizeof(Partial) > ub) ub = ((size_t)kMaxStreamCtas + R + 1) * sizeof(Partial);
  l.ctl = (l.units + ub + 15) & ~(size_t)15;
  l.total = ((l.ctl + sizeof(FusedCtl)) + 255) & ~(size_t)255;
  return l;
}
inline size_t workspace_bytes(long long B, long long K, long long V, int elem_bytes) {
  return workspace_layout(B, K, V, elem_bytes).total;
}

// Division by a divisor fixed at launch, as one multiply-high: q = floor(n *
// m / 2^64) with m = floor(2^64 / d) + 1 (2^64 / d when d is a power of two).
// Writing m * d = 2^64 + e with 0 <= e <= d, the product is n / d + n*e /
// (d * 2^64), whose floor is floor(n / d) whenever n * d < 2^64.  Every
// quotient taken here has n * d < 2^60 for logits that fit in device memory.
// (This GPU's 64-bit integer division is a ~500-cycle subroutine, its 32-bit
// division ~140 cycles; a 64-bit multiply-high is ~40.)
struct DivU64 {
  unsigned long long m = 0;  // 0: divide by 1
  static DivU64 make(unsigned long long d) {
    DivU64 r;
    r.m = d <= 1 ? 0ull : (~0ull / d) + 1ull;
    return r;
  }
#ifdef __CUDACC__
  __device__ __forceinline__ unsigned long long operator()(unsigned long long n) const {
    return m ? __umul64hi(n, m) : n;
  }
#endif
};

#ifdef __CUDACC__

// ---- debug-build index checks ----------------------------------------------
// SPEC_IN(i, n, status): whether 0 <= i < n.  In a -DSPEC_DEBUG build a
// failed check ORs kDebugBounds into the status word (when given) and the
// caller skips the access instead of faulting; release builds compile every
// check to `true`.
#ifdef SPEC_DEBUG
__device__ __forceinline__ bool spec_in(long long i, long long n, int32_t* status) {
  if (i >= 0 && i < n) return true;
  if (status) atomicOr(status, kDebugBounds);
  return false;
}
#define SPEC_IN(i, n, status) ::specv::spec_in(static_cast<long long>(i), static_cast<long long>(n), (status))
#else
#define SPEC_IN(i, n, status) true
#endif

// ---- loads ---------------------------------------------------------------
// 16-byte streaming load through the read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Element types: float (fp32) or the raw 16-bit pattern of a bf16.
struct F32 {
  using raw = float;
  static constexpr int kBytes = 4;
};
struct BF16 {
  using raw = uint16_t;
  static constexpr int kBytes = 2;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// VEC consecutive elements starting at element v*VEC of `row`, as floats.
// VEC is 16 bytes worth (4 fp32 / 8 bf16) for 16-byte aligned rows, else 1.
template <typename E, int VEC>
struct VecLoad;

template <>
struct VecLoad<F32, 4> {
  static __device__ __forceinline__ void load(const void* row, long long v, float (&x)[4]) {
    uint4 r = ld_stream_v4(static_cast<const float*>(row) + v * 4);
    x[0] = __uint_as_float(r.x); x[1] = __uint_as_float(r.y);
    x[2] = __uint_as_float(r.z); x[3] = __uint_as_float(r.w);
  }
};
template <>
struct VecLoad<BF16, 8> {
  static __device__ __forceinline__ void load(const void* row, long long v, float (&x)[8]) {
    uint4 r = ld_stream_v4(static_cast<const uint16_t*>(row) + v * 8);
    x[0] = bf16_lo(r.x); x[1] = bf16_hi(r.x); x[2] = bf16_lo(r.y); x[3] = bf16_hi(r.y);
    x[4] = bf16_lo(r.z); x[5] = bf16_hi(r.z); x[6] = bf16_lo(r.w); x[7] = bf16_hi(r.w);
  }
};
template <>
struct VecLoad<F32, 1> {
  static __device__ __forceinline__ void load(const void* row, long long v, float (&x)[1]) {
    x[0] = __ldg(static_cast<const float*>(row) + v);
  }
};
template <>
struct VecLoad<BF16, 1> {
  static __device__ __forceinline__ void load(const void* row, long long v, float (&x)[1]) {
    uint16_t h = __ldg(static_cast<const unsigned short*>(row) + v);
    x[0] = __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
};

// One element of a row, as float (t[x], d[x] at a draft token x).
template <typename E>
__device__ __forceinline__ float load_one(const void* row, long long j);
template <>
__device__ __forceinline__ float load_one<F32>(const void* row, long long j) {
  return __ldg(static_cast<const float*>(row) + j);
}
template <>
__device__ __forceinline__ float load_one<BF16>(const void* row, long long j) {
  uint16_t h = __ldg(static_cast<const unsigned short*>(row) + j);
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// ---- TMA bulk copies and mbarriers ---------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once on `bar` and announce `bytes` of transactions for this phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Global -> shared bulk copy (16-byte aligned addresses, size a multiple of
// 16), completing `bytes` transactions on `bar`.  No multicast.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// The same copy with an L2 cache policy (from make_policy_*): the lines it
// brings into L2 are kept there longer (evict_last) or dropped first
// (evict_first) when L2 needs room.
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               unsigned long long* bar, unsigned long long pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ unsigned long long make_policy_evict_last() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ unsigned long long make_policy_evict_first() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test: has phase `parity` of `bar` completed?
__device__ __forceinline__ bool mbar_test(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// One poll that may suspend the thread for up to `ns` nanoseconds while the
// phase is incomplete (the hardware wakes it when the phase completes).
__device__ __forceinline__ bool mbar_try_wait_sleep(unsigned long long* bar, uint32_t parity,
                                                    uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` from ONE thread, sleeping between polls
// instead of spinning (other threads of the CTA wait at a barrier and take
// no issue slots).  At most 2^16 polls of <= 20 us each (~1.3 s), then false.
__device__ __forceinline__ bool mbar_wait_one(unsigned long long* bar, uint32_t parity) {
  for (unsigned int i = 0; i < (1u << 16); ++i)
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  return false;
}

// Wait for phase `parity` of `bar` from any number of threads; each blocks
// in hardware between polls (no spinning).  At most 2^16 polls of <= 20 us.
__device__ __forceinline__ bool mbar_wait_sleep(unsigned long long* bar, uint32_t parity) {
  for (unsigned int i = 0; i < (1u << 16); ++i)
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  return false;
}

// Plain arrival (count 1) on `bar`.
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Wait for phase `parity` of `bar` to complete, polling at most kMaxPolls
// times.  Returns false on timeout (the caller reports kWaitTimeout).
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, uint32_t parity) {
  for (unsigned int i = 0; i < kMaxPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// The GPU's nanosecond clock (%globaltimer), for waits bounded in time.
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- cluster barrier, split -----------------------------------------------
// Every thread of every CTA of the cluster arrives early and waits just
// before its first access to another CTA's shared memory: that access must
// not come before all CTAs of the cluster have started.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// ---- arithmetic ----------------------------------------------------------
// 2^x on the SFU (PTX ex2.approx, flush-to-zero): 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Merge two partial softmax normalisers (m = max logit, z = sum 2^((x-m)s)).
__device__ __forceinline__ void merge_mz(float& m, float& z, float m2, float z2, float s) {
  float mn = fmaxf(m, m2);
  if (mn == -INFINITY) {  // both empty so far
    m = mn;
    z = 0.f;
    return;
  }
  float a = (m == -INFINITY) ? 0.f : z * ex2((m - mn) * s);
  float b = (m2 == -INFINITY) ? 0.f : z2 * ex2((m2 - mn) * s);
  m = mn;
  z = a + b;
}

// Add to a counter in global memory with acquire-release semantics at GPU
// scope: this thread's earlier writes are visible to whoever observes the
// new value, and what the earlier adders wrote is visible to this thread.
__device__ __forceinline__ unsigned int atom_add_acq_rel_gpu(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

// ---- workspace arrival ---------------------------------------------------
// Count one arrival for sequence b with acquire-release semantics: this
// thread's earlier writes (and atomics) are visible to whoever arrives later,
// and the last of `total` arrivals -- the one call that returns true -- sees
// everything the earlier arrivals wrote.
__device__ __forceinline__ unsigned long long atom_add_acq_rel_gpu(unsigned long long* p,
                                                                   unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;"
               : "=l"(old)
               : "l"(p), "l"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ void red_add_release_gpu(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ bool arrive_last(SeqState* seq, int b, unsigned int total) {
  return atom_add_acq_rel_gpu(&seq[b].arrivals, 1u) + 1u == total;
}

#endif  // __CUDACC__

}  // namespace specv
