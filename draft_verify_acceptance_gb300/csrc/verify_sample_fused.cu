// verify_sample_fused.cu -- speculative-sampling verification on sm_103a in
// one persistent kernel that reads every logit once from HBM and overlaps
// each sequence's accept decision and replacement draw with the streaming of
// later sequences.
//
// Sources (page title, section):
//   "推测性拒绝采样", 技术原理与步骤 steps 2-4: the target's K+1 rows come from
//     one parallel pass; x_i is accepted when p(x_i) >= q(x_i), else with
//     probability p(x_i)/q(x_i); everything after the first rejection is
//     dropped and one replacement token is drawn there.  关键保证: the output
//     follows the target distribution exactly, which makes the replacement
//     law normalize(max(0, p - q)).
//   "논문 리뷰 [Speculative Contrastive Decoding]", Speculative Decoding: with
//     all K accepted, the target supplies token K+1 (drawn from p_K).
//
// Work units.  Each draft position's (target row, draft row) pair is cut into
// segments of kFusedSeg 16-byte vectors and the bonus target row into
// segments of twice that; units are numbered sequence-major, so at any moment
// the GPU works on a narrow window of consecutive sequences.  One CTA runs on
// each SM (a cooperative launch: all of them resident) and takes units from a
// global counter as it goes, so a CTA that spends time on a draw simply takes
// fewer units.  Sequence b is decided and drawn by CTA b mod grid, whichever
// CTAs streamed it: the draws are spread evenly and never pile up on the CTAs
// that happen to finish sequences.
//
// Warp roles in a CTA:
//   producer (one thread): claims units (one ahead) and moves their rows into
//     a ring of shared-memory stages with cp.async.bulk, and on request moves
//     the row pair of a decided sequence through the same ring, ahead of the
//     next unit;
//   16 consumer warps: per stage, online normalisers (max and sum of
//     2^(x*s - offset)) of the target and draft segment; at a unit's end each
//     warp folds its lanes and leaves one value per warp.  For a draw stage
//     they compute the fixed-point residual mass of every 16-byte vector and
//     store the mass of each run of 32 vectors.  Consumers never wait on one
//     another or on the other roles, only on the ring;
//   arrivals (one warp): folds the 16 warp values of each unit in a fixed
//     order, writes the unit's Partial to the workspace and counts it on its
//     sequence with a release add (no round trip);
//   decisions (one warp): for each of its sequences (b = blockIdx.x, + grid,
//     ...), waits with an acquire load until all of the sequence's units are
//     counted, merges its partials row by row in unit order, runs the K
//     accept tests, finds the first rejection n and asks the producer for row
//     pair n (or the bonus row), streamed moments ago.  When the consumers
//     have reduced it, the warp locates the crossing run of the inverse CDF,
//     recomputes that run's 32 vectors from global memory and writes the
//     outputs.
// Only the decision warp waits on other CTAs (their unit counts), and the
// cooperative launch guarantees those CTAs are running; every wait is bounded.
#include <climits>

#include "device_common.cuh"
#include "launch.h"
#include "sample_common.cuh"

namespace specv {
namespace {

constexpr int kCW = 16;                     // consumer warps
constexpr int kCT = kCW * 32;               // consumer threads
constexpr int kProdWarp = kCW;
constexpr int kArrWarp = kCW + 1;
constexpr int kDecWarp = kCW + 2;
constexpr int kThreadsF = (kCW + 3) * 32;
constexpr int kLs = 2 * kCT;                // vectors per row per stage (16 KiB)
constexpr int kStageVec = 2 * kLs;          // vectors per stage (32 KiB)
constexpr int kStagesF = 6;
constexpr int kMaxEntries = static_cast<int>(kFusedMaxVec / 32);  // 32-vector runs per row
constexpr int kScratch = 512;               // partials per decision window
constexpr int kPartBuf = 16;                // unit ends the consumers may run ahead
constexpr int kUQ = 64;                     // producer -> arrivals: units issued
constexpr int kBatch = 8;                   // unit ends the arrival warp takes at once
constexpr int kRounds = (64 + 1 + 31) / 32; // rows per lane in a decision (K <= 64)
// Decisions -> producer draw requests.  At most 2 are issued and unfinished
// (two run-mass tables); the decision warp posts at most one request per
// sequence it owns.
constexpr int kReq = 64;
static_assert(kFusedSeg % kLs == 0, "a pair segment is a whole number of stages");
static_assert(kBatch <= kPartBuf, "batched tests must not alias");
static_assert(kUQ > kStagesF + 2 + kPartBuf, "issued units fit");

constexpr size_t kSmemF = static_cast<size_t>(kStagesF) * kStageVec * 16 +
                          2 * static_cast<size_t>(kMaxEntries) * 8 +
                          static_cast<size_t>(kScratch) * sizeof(Partial);

enum : int { kStream = 0, kDraw = 1, kExit = 3 };

// What a stage holds: a 16-byte head every consumer reads, and the
// normalisers that only draw stages need.
struct __align__(16) StageInfo {
  int kind;                       // kStream, kDraw, kExit
  int len;                        // vectors per row (pair) or of the target row
  int off;                        // first vector of the stage in its row
  int flags;                      // kPair | kLast | table << 2
  float MSt, invZt, MSd, invZd;   // draw: normalisers of the drawn rows
};
constexpr int kPair = 1;          // target half + draft half (else target only)
constexpr int kLast = 2;          // last stage of its unit / draw

// A decided sequence: the draw it needs and what its outputs depend on.
struct __align__(16) Job {
  int b, n, residual, ratio_near;
  float uK, MSt, invZt, MSd;
  float invZd;
  int pad[3];
};

struct FusedShared {
  unsigned long long full[kStagesF], empty[kStagesF];
  unsigned long long part_full[kPartBuf], part_free[kPartBuf];
  unsigned long long drawn[2];                // a draw's run masses are all in its table
  StageInfo info[kStagesF];
  float4 part[kPartBuf][kCW];                 // one value per consumer warp per unit end
  long long utau[kUQ];                        // units in issue order
  int ub[kUQ];
  Job jobs[kReq];
  long long units_issued, units_final, units_folded;  // units_final: -1 until known
  long long req_posted, draws_finished;       // written by the decision warp
  int exit_flag, abort_flag;
};

struct FusedGeom {
  int nvec;         // 16-byte vectors per row
  int segs;         // units per draft pair
  int segs_b;       // units of the bonus row
  int tps;          // units per sequence
  int ne;           // 32-vector runs per row
  int K, B;
  long long total;  // B * tps
  DivU64 by_tps, by_segs;  // divisions by tps and segs as multiply-highs
};

template <typename T>
__device__ __forceinline__ T vld(const T& x) {
  return *const_cast<const volatile T*>(&x);
}
template <typename T>
__device__ __forceinline__ void vst(T& x, T v) {
  *const_cast<volatile T*>(&x) = v;
}

__device__ __forceinline__ void set_abort(FusedShared& sh, const VerifyArgs& a) {
  vst(sh.abort_flag, 1);
  if (a.status) atomicOr(a.status, kWaitTimeout);
}

// Polling for work of other warps or thread blocks, bounded in time:
// expired() answers true once the caller has polled for longer than the
// call's wait limit since its last progress().
struct WaitClock {
  unsigned long long since = 0, limit;
  __device__ explicit WaitClock(unsigned long long l) : limit(l) {}
  __device__ __forceinline__ void progress() { since = 0; }
  __device__ __forceinline__ bool expired() {
    const unsigned long long t = global_ns();
    if (since == 0) {
      since = t;
      return false;
    }
    return t - since > limit;
  }
};

// Waits for phase `parity` of `bar`, the thread sleeping in hardware between
// polls.  False when the CTA aborts or the wait limit passes first.
__device__ __forceinline__ bool wait_phase(unsigned long long* bar, uint32_t parity,
                                           const FusedShared& sh, unsigned long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait_sleep(bar, parity, 5000u)) {
    if (vld(sh.abort_flag) || global_ns() - t0 > limit) return false;
  }
  return true;
}

// Position in the ring of stages: slot q, the parity of the slot's current
// round, and whether the ring has wrapped once (32-bit, no division).
struct RingPos {
  int q = 0;
  uint32_t ph = 0;
  bool wrapped = false;
  __device__ __forceinline__ void advance() {
    if (++q == kStagesF) {
      q = 0;
      ph ^= 1u;
      wrapped = true;
    }
  }
};

// ---------------------------------------------------------------------------
// producer

// The producer may refill slot p.q once the consumers released its previous
// round.
__device__ __forceinline__ bool acquire_slot(FusedShared& sh, const RingPos& p,
                                             unsigned long long limit) {
  if (!p.wrapped) return true;
  return wait_phase(&sh.empty[p.q], p.ph ^ 1u, sh, limit);
}

// Copies vectors [off, off+len) of target row `trow` (and of draft row
// `drow` when non-null, into the stage's second half) into stage q.
__device__ __forceinline__ void issue_copies(FusedShared& sh, uint4* ring, int q, const uint4* trow,
                                             const uint4* drow, int off, int len) {
  uint4* dst = ring + static_cast<size_t>(q) * kStageVec;
  const uint32_t bytes = static_cast<uint32_t>(len) * 16u;
  if (drow) {
    mbar_arrive_expect_tx(&sh.full[q], 2u * bytes);
    bulk_load(dst, trow + off, bytes, &sh.full[q]);
    bulk_load(dst + kLs, drow + off, bytes, &sh.full[q]);
  } else {
    mbar_arrive_expect_tx(&sh.full[q], bytes);
    bulk_load(dst, trow + off, bytes, &sh.full[q]);
  }
}

template <typename E>
__device__ __forceinline__ void run_producer(const VerifyArgs& a, const FusedGeom& g, FusedCtl* ctl,
                                             FusedShared& sh, uint4* ring) {
  const int nvec = g.nvec, K = g.K;
  const uint4* T = static_cast<const uint4*>(a.target);
  const uint4* D = static_cast<const uint4*>(a.draft);
  long long k = 0, taken = 0, units = 0;  // k: stages issued
  RingPos pos;
  bool ok = true, exhausted = false;
  // the unit being issued: rows, vector range, next stage offset
  bool in_unit = false;
  const uint4* ctrow = nullptr;
  const uint4* cdrow = nullptr;
  int cb = 0, cend = 0, cnext = 0;
  // one unit is claimed ahead of its use
  unsigned long long next = atomicAdd(&ctl->next_task, 1ull);
  bool have_next = true;
  WaitClock idle(a.wait_ns);

  while (true) {
    if (vld(sh.abort_flag)) break;
    if (in_unit) {  // finish the current unit first
      const int per = cdrow ? kLs : kStageVec;
      const int len = min(per, cend - cnext);
      if (!acquire_slot(sh, pos, a.wait_ns)) {
        ok = false;
        break;
      }
      const int q = pos.q;
      StageInfo& in = sh.info[q];
      in.kind = kStream;
      in.off = cnext;
      in.len = len;
      in.flags = (cdrow ? kPair : 0) | (cnext + len >= cend ? kLast : 0);
      issue_copies(sh, ring, q, ctrow, cdrow, cnext, len);
      ++k;
      pos.advance();
      cnext += len;
      if (cnext >= cend) in_unit = false;
      idle.progress();
      continue;
    }
    const long long posted = vld(sh.req_posted);
    const bool want_draw = posted > taken;
    // a requested draw goes ahead of the next unit; request `taken` uses
    // table taken & 1, free once request taken-2 is done
    if (want_draw && (taken < 2 || vld(sh.draws_finished) >= taken - 1)) {
      __threadfence_block();
      const Job j = sh.jobs[taken % kReq];
      if (!(SPEC_IN(j.b, g.B, a.status) && SPEC_IN(j.n, K + 1, a.status))) {
        ok = false;  // (debug builds) a draw outside the batch: stop this CTA
        break;
      }
      const int per = j.residual ? kLs : kStageVec;
      const uint4* trow = T + (static_cast<size_t>(j.b) * (K + 1) + j.n) * nvec;
      const uint4* drow = j.residual ? D + (static_cast<size_t>(j.b) * K + j.n) * nvec : nullptr;
      for (int off = 0; off < nvec; off += per) {
        const int len = min(per, nvec - off);
        if (!acquire_slot(sh, pos, a.wait_ns)) {
          ok = false;
          break;
        }
        const int q = pos.q;
        StageInfo& in = sh.info[q];
        in.kind = kDraw;
        in.off = off;
        in.len = len;
        in.flags = (j.residual ? kPair : 0) | (off + per >= nvec ? kLast : 0) |
                   (static_cast<int>(taken & 1) << 2);
        in.MSt = j.MSt;
        in.invZt = j.invZt;
        in.MSd = j.MSd;
        in.invZd = j.invZd;
        issue_copies(sh, ring, q, trow, drow, off, len);
        ++k;
        pos.advance();
      }
      if (!ok) break;
      ++taken;
      idle.progress();
      continue;
    }
    if (have_next) {  // start the unit claimed ahead
      const unsigned long long t = next;
      if (t >= static_cast<unsigned long long>(g.total)) {
        have_next = false;
        exhausted = true;
        vst(sh.units_final, units);
        // the last CTA to take its final unit puts the counters back to zero
        if (atomicAdd(&ctl->done_ctas, 1ull) == static_cast<unsigned long long>(gridDim.x) - 1ull) {
          ctl->next_task = 0ull;
          ctl->done_ctas = 0ull;
        }
        continue;
      }
      if (units - vld(sh.units_folded) >= kUQ) {  // the arrival warp is kUQ units behind
        if (idle.expired()) {
          ok = false;
          break;
        }
        __nanosleep(64);
        continue;
      }
      have_next = false;
      const long long b = static_cast<long long>(g.by_tps(t));
      const int jj = static_cast<int>(static_cast<long long>(t) - b * g.tps);
      cb = static_cast<int>(b);
      int i, coff;
      if (jj < K * g.segs) {
        i = static_cast<int>(g.by_segs(static_cast<unsigned long long>(jj)));
        coff = (jj - i * g.segs) * kFusedSeg;
        cend = min(coff + kFusedSeg, nvec);
        cdrow = D + (static_cast<size_t>(cb) * K + i) * nvec;
      } else {
        i = K;
        coff = (jj - K * g.segs) * 2 * kFusedSeg;
        cend = min(coff + 2 * kFusedSeg, nvec);
        cdrow = nullptr;
      }
      if (!(SPEC_IN(cb, g.B, a.status) && SPEC_IN(i, K + 1, a.status) &&
            SPEC_IN(cend - 1, nvec, a.status))) {
        ok = false;  // (debug builds) a unit outside the batch: stop this CTA
        break;
      }
      ctrow = T + (static_cast<size_t>(cb) * (K + 1) + i) * nvec;
      cnext = coff;
      in_unit = true;
      // tell the arrival warp which unit ends next
      sh.ub[units % kUQ] = cb;
      sh.utau[units % kUQ] = static_cast<long long>(t);
      __threadfence_block();
      vst(sh.units_issued, ++units);
      next = atomicAdd(&ctl->next_task, 1ull);  // the next unit, claimed ahead
      have_next = true;
      idle.progress();
      continue;
    }
    if (exhausted && !want_draw && vld(sh.exit_flag)) {
      if (acquire_slot(sh, pos, a.wait_ns)) {
        sh.info[pos.q].kind = kExit;
        mbar_arrive(&sh.full[pos.q]);
        ++k;
        pos.advance();
      } else {
        ok = false;
      }
      break;
    }
    if (idle.expired()) {
      ok = false;
      break;
    }
    __nanosleep(128);
  }
  if (!ok) set_abort(sh, a);
  if (!ok || vld(sh.abort_flag)) {
    // an early exit (this warp's or another's): the consumers may leave
    // without reading the stages still in flight, so the copies already
    // issued must land before the CTA can exit
    for (long long kk = (k > kStagesF ? k - kStagesF : 0); kk < k; ++kk)
      mbar_wait_sleep(&sh.full[kk % kStagesF], static_cast<uint32_t>((kk / kStagesF) & 1));
  }
}

// ---------------------------------------------------------------------------
// consumers

template <typename E>
__device__ __forceinline__ void run_consumers(const VerifyArgs& a, FusedShared& sh,
                                              const uint4* ring, unsigned long long* tables) {
  constexpr int VEC = Staged<E>::kVec;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float s = a.scale;
  // At: the target row; Ad: the draft row of a pair unit, or the second half
  // of each stage of a bonus-row unit (folded into At at the unit's end)
  RowAcc At{-INFINITY, 0.f}, Ad{-INFINITY, 0.f};
  unsigned int u = 0;  // unit ends seen
  RingPos pos;
  bool ok = true;
  for (;; pos.advance()) {
    const int q = pos.q;
    if (!wait_phase(&sh.full[q], pos.ph, sh, a.wait_ns)) {
      ok = false;  // the producer stopped (abort) or a copy never landed
      break;
    }
    const int4 in = *reinterpret_cast<const int4*>(&sh.info[q]);  // kind, len, off, flags
    const int in_kind = in.x, in_len = in.y, in_off = in.z;
    const bool in_pair = (in.w & kPair) != 0, in_last = (in.w & kLast) != 0;
    const uint4* st = ring + static_cast<size_t>(q) * kStageVec;
    if (in_kind == kStream) {
      uint4 w0[2], w1[2];
      if (in_len == (in_pair ? kLs : kStageVec)) {  // a full stage
        w0[0] = st[tid];
        w0[1] = st[tid + kCT];
        w1[0] = st[kLs + tid];
        w1[1] = st[kLs + tid + kCT];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[q]);  // this warp is done reading the stage
        acc_vectors_full<E>(At, w0, s);
        acc_vectors_full<E>(Ad, w1, s);
      } else {
        const int h = in_pair ? in_len : min(in_len, kLs), r = in_pair ? in_len : in_len - kLs;
        const int n0 = (tid < h ? 1 : 0) + (tid + kCT < h ? 1 : 0);
        const int n1 = (tid < r ? 1 : 0) + (tid + kCT < r ? 1 : 0);
        if (n0 > 0) w0[0] = st[tid];
        if (n0 > 1) w0[1] = st[tid + kCT];
        if (n1 > 0) w1[0] = st[kLs + tid];
        if (n1 > 1) w1[1] = st[kLs + tid + kCT];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[q]);
        acc_vectors<E>(At, w0, n0, s);
        acc_vectors<E>(Ad, w1, n1, s);
      }
      if (in_last) {  // end of a unit: this warp's value for the arrival warp
        float mt = At.ms, zt = At.z, md = Ad.ms, zd = Ad.z;
        if (!in_pair) {  // both halves belong to the target row
          merge_scaled(mt, zt, md, zd);
          md = -INFINITY;
          zd = 0.f;
        }
        warp_merge_scaled(mt, zt);
        warp_merge_scaled(md, zd);
        const unsigned int buf = u % kPartBuf;
        if (lane == 0) {
          if (u >= kPartBuf &&
              !wait_phase(&sh.part_free[buf], ((u / kPartBuf) - 1u) & 1u, sh, a.wait_ns))
            ok = false;
          sh.part[buf][warp] = make_float4(mt, zt, md, zd);
          mbar_arrive(&sh.part_full[buf]);
        }
        ++u;
        At = RowAcc{-INFINITY, 0.f};
        Ad = RowAcc{-INFINITY, 0.f};
      }
    } else if (in_kind == kDraw) {
      const int table = in.w >> 2;
      const float4 nz = *reinterpret_cast<const float4*>(&sh.info[q].MSt);
      unsigned long long* tab = tables + static_cast<size_t>(table) * kMaxEntries;
      uint4 v[4];
      if (in_pair) {
        if (tid < in_len) {
          v[0] = st[tid];
          v[1] = st[kLs + tid];
        }
        if (tid + kCT < in_len) {
          v[2] = st[tid + kCT];
          v[3] = st[kLs + tid + kCT];
        }
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h)
          if (h * kCT + tid < in_len) v[h] = st[h * kCT + tid];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[q]);
      if (in_pair) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int base = h * kCT + warp * 32;
          if (base < in_len) {  // warp-uniform
            float xt[VEC], xd[VEC], r[VEC];
            if (h * kCT + tid < in_len) {
              Staged<E>::unpack(v[2 * h], xt);
              Staged<E>::unpack(v[2 * h + 1], xd);
            } else {
#pragma unroll
              for (int e = 0; e < VEC; ++e) xt[e] = xd[e] = -INFINITY;
            }
            const unsigned long long m = warp_sum_mass(
                vec_weight_scaled<VEC>(xt, xd, nz.x, nz.y, nz.z, nz.w, s, true, r));
            if (lane == 0) tab[(in_off + base) >> 5] = m;
          }
        }
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int base = h * kCT + warp * 32;
          if (base < in_len) {
            float xt[VEC], xd[VEC], r[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) xd[e] = -INFINITY;
            if (h * kCT + tid < in_len) {
              Staged<E>::unpack(v[h], xt);
            } else {
#pragma unroll
              for (int e = 0; e < VEC; ++e) xt[e] = -INFINITY;
            }
            const unsigned long long m = warp_sum_mass(
                vec_weight_scaled<VEC>(xt, xd, nz.x, nz.y, nz.z, nz.w, s, false, r));
            if (lane == 0) tab[(in_off + base) >> 5] = m;
          }
        }
      }
      // every warp's run masses of the draw are in the table
      if (in_last && lane == 0) mbar_arrive(&sh.drawn[table]);
    } else {
      break;  // kExit
    }
  }
  if (!ok) set_abort(sh, a);
}

// ---------------------------------------------------------------------------
// arrivals

// Folds each unit's 16 warp values, publishes the unit's Partial and counts it
// on its sequence; hands completed sequences (then -1) to the decision warp.
__device__ __forceinline__ void run_arrivals(const VerifyArgs& a, const FusedGeom& g, FusedShared& sh) {
  const int lane = threadIdx.x & 31;
  Partial* partials = static_cast<Partial*>(a.partials);
  long long u = 0;
  bool ok = true;
  WaitClock idle(a.wait_ns);
  while (true) {
    if (vld(sh.abort_flag)) break;
    const long long issued = vld(sh.units_issued);
    const long long fin = vld(sh.units_final);
    if (fin >= 0 && u >= fin) break;  // every unit of this CTA is counted
    // the unit ends that are already folded by the consumers (up to kBatch)
    int rdy = 0;
    if (lane < kBatch && u + lane < issued)
      rdy = mbar_test(&sh.part_full[(u + lane) % kPartBuf], static_cast<uint32_t>(((u + lane) / kPartBuf) & 1)) ? 1 : 0;
    int nb = __ffs(~__ballot_sync(0xffffffffu, rdy)) - 1;
    if (nb == 0) {
      if (u < issued) {  // wait for the next unit end
        int got = 0;
        if (lane == 0)
          got = wait_phase(&sh.part_full[u % kPartBuf], static_cast<uint32_t>((u / kPartBuf) & 1), sh, a.wait_ns) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
        nb = 1;
      } else {  // nothing issued yet
        if (idle.expired()) {
          ok = false;
          break;
        }
        __nanosleep(256);
        continue;
      }
    }
    idle.progress();
    __syncwarp();
    // fold each ready unit (lanes 0..15 hold its 16 warp values); lane j keeps unit u+j
    Partial mine{-INFINITY, 0.f, -INFINITY, 0.f};
    for (int j = 0; j < nb; ++j) {
      const int buf = static_cast<int>((u + j) % kPartBuf);
      float4 v = lane < kCW ? sh.part[buf][lane] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
      warp_merge_scaled(v.x, v.y);
      warp_merge_scaled(v.z, v.w);
      if (lane == j) mine = Partial{v.x, v.y, v.z, v.w};
    }
    __syncwarp();
    if (lane < nb) {
      const long long uu = u + lane;
      mbar_arrive(&sh.part_free[uu % kPartBuf]);
      const int b = sh.ub[uu % kUQ];
      const long long tau = sh.utau[uu % kUQ];
      if (SPEC_IN(tau, a.ws_units, a.status) && SPEC_IN(b, g.B, a.status)) {
        partials[tau] = mine;
        red_add_release_gpu(&a.seq[b].arrivals, 1u);  // the Partial is published first
      }
    }
    u += nb;
    if (lane == 0) vst(sh.units_folded, u);
  }
  if (!__all_sync(0xffffffffu, ok) && lane == 0) set_abort(sh, a);
}

// ---------------------------------------------------------------------------
// decisions

__device__ __forceinline__ const void* row_ptr(const void* base, size_t row, long long V, int bytes) {
  return static_cast<const char*>(base) + row * static_cast<size_t>(V) * bytes;
}

// The accept decision of sequence b (whole warp).  Each lane owns the rows
// i = r*32 + lane; a row's partials are merged in unit order, so the result
// does not depend on which CTA streamed which unit.  Writes p(x_i), q(x_i)
// and the data-error bits; puts the sequence's partials back to zero.
template <typename E>
__device__ __noinline__ Job decide(const VerifyArgs& a, const FusedGeom& g, int b, Partial* scratch, int lane) {
  const int K = g.K, K1 = K + 1;
  const float s = a.scale;
  const float* u = a.uniforms + static_cast<size_t>(b) * K1;
  Partial* parts = static_cast<Partial*>(a.partials) + static_cast<size_t>(b) * g.tps;
  if (!SPEC_IN(static_cast<long long>(b + 1) * g.tps - 1, a.ws_units, a.status)) parts = nullptr;
  float MSt[kRounds], Zt[kRounds], MSd[kRounds], Zd[kRounds], gx[kRounds], gy[kRounds], ui[kRounds];
  int xr[kRounds];
  // one lane's acquire saw every unit's partial; order every lane's loads
  // after it
  __syncwarp();
  __threadfence();
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int i = r * 32 + lane;
    MSt[r] = -INFINITY;
    Zt[r] = 0.f;
    MSd[r] = -INFINITY;
    Zd[r] = 0.f;
    gx[r] = 0.f;
    gy[r] = 0.f;
    ui[r] = 0.f;
    xr[r] = 0;
    if (i <= K) ui[r] = u[i];
    if (i < K) xr[r] = a.tokens[static_cast<size_t>(b) * K + i];
  }
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int i = r * 32 + lane;
    if (i < K) {
      const long long x = min(max(xr[r], 0), a.V - 1);
      gx[r] = load_one<E>(row_ptr(a.target, static_cast<size_t>(b) * K1 + i, a.V, E::kBytes), x);
      gy[r] = load_one<E>(row_ptr(a.draft, static_cast<size_t>(b) * K + i, a.V, E::kBytes), x);
    }
  }
  for (int w0 = 0; w0 < g.tps; w0 += kScratch) {
    const int cnt = min(kScratch, g.tps - w0);
    for (int j = lane; j < cnt; j += 32) {
      const float4 v = parts ? __ldcg(reinterpret_cast<const float4*>(parts + w0 + j))
                             : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
      scratch[j] = Partial{v.x, v.y, v.z, v.w};
    }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int i = r * 32 + lane;
      if (i <= K) {
        const int lo0 = i < K ? i * g.segs : K * g.segs;
        const int hi0 = lo0 + (i < K ? g.segs : g.segs_b);
        const int lo = max(lo0, w0), hi = min(hi0, w0 + cnt);
        for (int j = lo; j < hi; ++j) {
          const Partial p = scratch[j - w0];
          merge_scaled(MSt[r], Zt[r], p.ms_t, p.z_t);
          if (i < K) merge_scaled(MSd[r], Zd[r], p.ms_d, p.z_d);
        }
      }
    }
    __syncwarp();
  }
  for (int j = lane; parts && j < g.tps; j += 32)
    reinterpret_cast<float4*>(parts)[j] = make_float4(0.f, 0.f, 0.f, 0.f);

  int n = K, bad = 0;
  bool ratio_near = false, decided = false;
  float nMSt = 0.f, nZt = 0.f, nMSd = 0.f, nZd = 0.f;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int i = r * 32 + lane;
    bool rej = false, nr = false;
    if (i <= K) {
      if (!(isfinite(MSt[r]) && isfinite(Zt[r]) && Zt[r] > 0.f)) bad |= kDataNonfiniteLogit;
      if (!(ui[r] >= 0.f && ui[r] < 1.f)) bad |= kDataUniformRange;
      if (i < K) {
        if (xr[r] < 0 || xr[r] >= a.V) bad |= kDataTokenRange;
        if (!(isfinite(MSd[r]) && isfinite(Zd[r]) && Zd[r] > 0.f)) bad |= kDataNonfiniteLogit;
        const float px = ex2(fmaf(gx[r], s, -MSt[r])) / Zt[r];
        const float qx = ex2(fmaf(gy[r], s, -MSd[r])) / Zd[r];
        if (SPEC_IN(static_cast<long long>(b) * K + i, static_cast<long long>(a.B) * K, a.status)) {
          if (a.p_at) a.p_at[static_cast<size_t>(b) * K + i] = px;
          if (a.q_at) a.q_at[static_cast<size_t>(b) * K + i] = qx;
        }
        rej = !(ui[r] * qx < px);
        nr = qx > 0.f && fabsf(ui[r] - fminf(1.f, px / qx)) < kBandF;
      }
    }
    const unsigned int rb = __ballot_sync(0xffffffffu, rej);
    const unsigned int nb = __ballot_sync(0xffffffffu, nr);
    if (!decided) {  // warp-uniform
      int pick = -1;
      if (rb) {
        pick = __ffs(rb) - 1;
        n = r * 32 + pick;
        ratio_near |= (nb & (pick == 31 ? 0xffffffffu : ((2u << pick) - 1u))) != 0u;
        decided = true;
      } else {
        ratio_near |= nb != 0u;
        if (K - r * 32 < 32) {  // the bonus row is in this round
          pick = K - r * 32;
          decided = true;
        }
      }
      if (pick >= 0) {
        nMSt = __shfl_sync(0xffffffffu, MSt[r], pick);
        nZt = __shfl_sync(0xffffffffu, Zt[r], pick);
        nMSd = __shfl_sync(0xffffffffu, MSd[r], pick);
        nZd = __shfl_sync(0xffffffffu, Zd[r], pick);
      }
    }
  }
  bad = __reduce_or_sync(0xffffffffu, bad);
  if (lane == 0 && bad && a.status) atomicOr(a.status, bad);
  Job j;
  j.b = b;
  j.n = n;
  j.residual = n < K ? 1 : 0;
  j.ratio_near = ratio_near ? 1 : 0;
  j.uK = u[K];
  j.MSt = nMSt;
  j.invZt = 1.f / nZt;
  j.MSd = nMSd;
  j.invZd = n < K ? 1.f / nZd : 0.f;
  j.pad[0] = j.pad[1] = j.pad[2] = 0;
  return j;
}

// Finishes a draw (whole warp) from the run masses in `tab`: S, the run and
// then the element where the fixed-point CDF passes floor(u_K * S), and the
// sequence's outputs.  Returns true, writing nothing, when a residual row has
// no mass (p == q there): the draw must be redone from p.
template <typename E>
__device__ __noinline__ bool finish_draw(const VerifyArgs& a, const FusedGeom& g, const Job& j,
                            const unsigned long long* tab, int lane) {
  constexpr int VEC = Staged<E>::kVec;
  const int ne = g.ne;
  const int per = (ne + 31) >> 5;
  const int e0 = min(lane * per, ne), e1 = min(e0 + per, ne);
  unsigned long long bs = 0;
  for (int e = e0; e < e1; ++e) bs += tab[e];
  const unsigned long long incl = warp_scan_u64(bs, lane);
  const unsigned long long S = __shfl_sync(0xffffffffu, incl, 31);
  const bool residual = j.residual != 0;
  if (S == 0 && residual) return true;
  const int K = g.K, K1 = K + 1, b = j.b, n = j.n;
  int token = 0, near = 0;
  if (S != 0) {
    const unsigned long long theta = draw_threshold(j.uK, S);
    // the lane block holding the crossing, then the run inside it
    const int lb = __ffs(__ballot_sync(0xffffffffu, incl > theta)) - 1;
    unsigned long long base = __shfl_sync(0xffffffffu, incl - bs, lb);
    const int s0 = __shfl_sync(0xffffffffu, e0, lb), s1 = __shfl_sync(0xffffffffu, e1, lb);
    int estar = s1 - 1;
    for (int c0 = s0; c0 < s1; c0 += 32) {
      const int e = c0 + lane;
      const unsigned long long m = e < s1 ? tab[e] : 0ull;
      const unsigned long long ii = warp_scan_u64(m, lane);
      const unsigned int h = __ballot_sync(0xffffffffu, e < s1 && base + ii > theta);
      if (h) {
        const int l = __ffs(h) - 1;
        base += __shfl_sync(0xffffffffu, ii - m, l);
        estar = c0 + l;
        break;
      }
      base += __shfl_sync(0xffffffffu, ii, 31);
    }
    // the run's 32 vectors again, from global memory (L2)
    const long long v = static_cast<long long>(estar) * 32 + lane;
    const uint4* trow = static_cast<const uint4*>(a.target) +
                        (static_cast<size_t>(b) * K1 + n) * g.nvec;
    float xt[VEC], xd[VEC], r[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) xt[e] = xd[e] = -INFINITY;
    if (v < g.nvec) {
      Staged<E>::unpack(__ldg(trow + v), xt);
      if (residual) {
        const uint4* drow = static_cast<const uint4*>(a.draft) +
                            (static_cast<size_t>(b) * K + n) * g.nvec;
        Staged<E>::unpack(__ldg(drow + v), xd);
      }
    }
    const unsigned long long w =
        vec_weight_scaled<VEC, true>(xt, xd, j.MSt, j.invZt, j.MSd, j.invZd, a.scale, residual, r);
    const unsigned long long wi = warp_scan_u64(w, lane);
    const unsigned int h3 = __ballot_sync(0xffffffffu, base + wi > theta);
    const int lstar = h3 ? __ffs(h3) - 1 : 31;
    int tok = 0, nr = 0;
    if (lane == lstar) {
      const unsigned long long before = base + wi - w;
      unsigned long long c_prev, c_cur;
      const int mstar = pick_in_vector<VEC>(r, w, theta - before, c_prev, c_cur);
      const long long t = v * VEC + mstar;
      nr = near_step(theta, before + c_prev, before + c_cur, S) ? 1 : 0;
      tok = static_cast<int>(t < a.V ? t : a.V - 1);
    }
    token = __shfl_sync(0xffffffffu, tok, lstar);
    near = __shfl_sync(0xffffffffu, nr, lstar);
  }
  if (!SPEC_IN(b, g.B, a.status) || !SPEC_IN(n, K1, a.status)) return false;
  const int32_t* x = a.tokens + static_cast<size_t>(b) * K;
  int32_t* out = a.out_tokens + static_cast<size_t>(b) * K1;
  for (int jj = lane; jj < K1; jj += 32)
    out[jj] = (jj < n) ? min(max(x[jj], 0), a.V - 1) : (jj == n ? token : -1);
  if (lane == 0) {
    if (a.accepted_len) a.accepted_len[b] = n;
    if (a.flags) a.flags[b] = (j.ratio_near ? kFlagRatio : 0u) | (near ? kFlagCdf : 0u);
    if (a.p_emit) {  // p_n(token) from the drawn row's normaliser
      const float xt = load_one<E>(a.target, (static_cast<long long>(b) * K1 + n) * a.V + token);
      a.p_emit[b] = ex2(fmaf(xt, a.scale, -j.MSt)) * j.invZt;
    }
  }
  return false;
}

// Decision warp: waits for each of this CTA's sequences (b = blockIdx.x,
// blockIdx.x + gridDim.x, ...) to be counted complete, decides it, requests
// its draw and finishes the draws in order.
template <typename E>
__device__ __forceinline__ void run_decisions(const VerifyArgs& a, const FusedGeom& g, FusedShared& sh,
                                              const unsigned long long* tables, Partial* scratch) {
  const int lane = threadIdx.x & 31;
  long long posted = 0, finished = 0;
  int nb = blockIdx.x;  // the next sequence this CTA owns
  bool ok = true;
  WaitClock idle(a.wait_ns);
  while (nb < g.B || finished < posted) {
    if (vld(sh.abort_flag)) break;
    // the oldest outstanding draw is reduced: finish it (frees its table)
    int r2 = 0;
    if (finished < posted && lane == 0 &&
        mbar_test(&sh.drawn[finished & 1], static_cast<uint32_t>((finished >> 1) & 1)))
      r2 = 1;
    if (__shfl_sync(0xffffffffu, r2, 0)) {
      __syncwarp();
      const long long rq = finished;
      Job j = sh.jobs[rq % kReq];
      const bool redo = finish_draw<E>(a, g, j, tables + static_cast<size_t>(rq & 1) * kMaxEntries, lane);
      ++finished;
      if (redo) {  // residual mass zero: draw from p_n instead
        j.residual = 0;
        j.invZd = 0.f;
        if (lane == 0) {
          sh.jobs[posted % kReq] = j;
          __threadfence_block();
        }
        ++posted;
      }
      if (lane == 0) {
        vst(sh.draws_finished, finished);
        if (redo) vst(sh.req_posted, posted);
      }
      idle.progress();
      continue;
    }
    // the next owned sequence complete: decide it and request its draw
    int r3 = 0;
    if (nb < g.B && lane == 0)
      r3 = ld_acquire_gpu(&a.seq[nb].arrivals) == static_cast<unsigned int>(g.tps) ? 1 : 0;
    if (__shfl_sync(0xffffffffu, r3, 0)) {
      __syncwarp();  // lane 0's acquire orders every lane's reads of the partials
      if (lane == 0) a.seq[nb].arrivals = 0u;  // complete: back to zero
      const Job j = decide<E>(a, g, nb, scratch, lane);
      if (posted - finished >= kReq) {  // cannot happen: at most one request per owned sequence
        ok = false;
        break;
      }
      if (lane == 0) {
        sh.jobs[posted % kReq] = j;
        __threadfence_block();
        vst(sh.req_posted, posted + 1);
      }
      ++posted;
      nb += gridDim.x;
      idle.progress();
      continue;
    }
    if (idle.expired()) {
      ok = false;
      break;
    }
    __nanosleep(128);
  }
  if (lane == 0) vst(sh.exit_flag, 1);
  if (!ok && lane == 0) set_abort(sh, a);
}

template <typename E>
__global__ void __launch_bounds__(kThreadsF, 1)
fused_sample_kernel(VerifyArgs a, FusedGeom g, FusedCtl* ctl) {
  extern __shared__ __align__(128) uint4 dsm[];
  __shared__ FusedShared sh;
  uint4* ring = dsm;
  unsigned long long* tables = reinterpret_cast<unsigned long long*>(dsm + static_cast<size_t>(kStagesF) * kStageVec);
  Partial* scratch = reinterpret_cast<Partial*>(tables + 2 * kMaxEntries);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    for (int q = 0; q < kStagesF; ++q) {
      mbar_init(&sh.full[q], 1);
      mbar_init(&sh.empty[q], kCW);
    }
    for (int q = 0; q < kPartBuf; ++q) {
      mbar_init(&sh.part_full[q], kCW);
      mbar_init(&sh.part_free[q], 1);
    }
    mbar_init(&sh.drawn[0], kCW);
    mbar_init(&sh.drawn[1], kCW);
    sh.units_issued = 0;
    sh.units_final = -1;
    sh.units_folded = 0;
    sh.req_posted = 0;
    sh.draws_finished = 0;
    sh.exit_flag = 0;
    sh.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == kProdWarp) {
    if ((tid & 31) == 0) run_producer<E>(a, g, ctl, sh, ring);
  } else if (warp == kArrWarp) {
    run_arrivals(a, g, sh);
  } else if (warp == kDecWarp) {
    run_decisions<E>(a, g, sh, tables, scratch);
  } else {
    run_consumers<E>(a, sh, ring, tables);
  }
}

}  // namespace

cudaError_t sample_fused_prepare() {
  cudaError_t e = cudaFuncSetAttribute(fused_sample_kernel<BF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemF));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused_sample_kernel<F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemF));
  return e;
}

cudaError_t launch_sample_fused(const VerifyArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  FusedGeom g;
  const long long nvec = static_cast<long long>(a.V) * (a.bf16 ? 2 : 4) / 16;
  if (!a.vec || nvec < 1 || nvec > kFusedMaxVec) return cudaErrorInvalidValue;
  g.nvec = static_cast<int>(nvec);
  g.segs = static_cast<int>((nvec + kFusedSeg - 1) / kFusedSeg);
  g.segs_b = static_cast<int>((nvec + 2 * kFusedSeg - 1) / (2 * kFusedSeg));
  g.tps = static_cast<int>(fused_tasks_per_seq(a.K, nvec));
  g.ne = static_cast<int>((nvec + 31) / 32);
  g.K = a.K;
  g.B = a.B;
  g.total = static_cast<long long>(a.B) * g.tps;
  g.by_tps = DivU64::make(static_cast<unsigned long long>(g.tps));
  g.by_segs = DivU64::make(static_cast<unsigned long long>(g.segs));
  long long G = dev.sm_count > 0 ? dev.sm_count : 1;
  if (G > g.total) G = g.total;
  FusedCtl* ctl = static_cast<FusedCtl*>(a.ctl);
  // cooperative: every CTA is resident, since decision warps wait on the
  // unit counts that other CTAs' arrival warps publish
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(G));
  cfg.blockDim = dim3(kThreadsF);
  cfg.dynamicSmemBytes = kSmemF;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.bf16 ? cudaLaunchKernelEx(&cfg, fused_sample_kernel<BF16>, a, g, ctl)
                : cudaLaunchKernelEx(&cfg, fused_sample_kernel<F32>, a, g, ctl);
}

}  // namespace specv
