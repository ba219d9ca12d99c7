// verify_sample_2p.cu -- speculative-sampling verification on sm_103a in two
// kernels with no cross-CTA atomics on either critical path.
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
// Kernel A (normaliser stream): a persistent grid of G CTAs streams every
// (target row i, draft row i) pair once from HBM through a ring of shared-
// memory stages filled by cp.async.bulk.  The pairs, position-major, form one
// flat space of 16-byte vectors weighted by their bytes (32 per draft pair
// vector, 16 per bonus-row vector); CTA c owns a byte-balanced contiguous
// range of it.  Each thread keeps online normalisers of both rows relative to
// scaled offsets; at a row change the warps fold them into shared memory, and
// at the end warp 0 writes one Partial per (CTA, pair) to slot c + pair -- a
// plain store.  The CTA that streams the vector holding x_i stores t[x_i] and
// d[x_i].
// Kernel B (decide and sample), launched as a programmatic dependent of A:
// one cluster per sequence.  Warp 0 of every CTA merges each row's partials
// in contributor order, runs the K accept tests in parallel lanes and finds
// the first rejection n with a ballot; every CTA of the cluster then reads its
// slice of row pair n (or of the bonus row) from global memory and computes
// its fixed-point residual mass, the CTAs exchange slice masses through
// distributed shared memory, and the CTA holding the crossing finds the
// token.  Rank 0 writes the outputs.  Kernel B re-reads one row pair per
// sequence.
#include <cooperative_groups.h>

#include <cfloat>
#include <climits>

#include "device_common.cuh"
#include "launch.h"
#include "sample_common.cuh"

namespace cg = cooperative_groups;

namespace specv {

// Byte-weighted partition of the pair-vector space over G CTAs.  Vectors
// [0, P) belong to draft pairs (positions 0..K-1, weight 2), [P, P + Q) to
// bonus rows (position K, weight 1); pair p = i*B + b covers vectors
// [p*nvec, (p+1)*nvec).  CTA c streams the weight range [W*c/G, W*(c+1)/G).
// (Handing out smaller ranges dynamically was measured: it evens out the
// CTAs' finishing times but not the last one, since the pass is bound by the
// GPU's total throughput, not by its slowest CTA.)
struct StreamPartition {
  long long nvec, P, Q, W;
  int G;
  // 0: a whole verify; 1: early exit, position 0 only (a sequence that
  // accepts x_0 is counted in *pending and left to phase 2); 2: early exit,
  // the whole verify, skipped when *pending is 0
  int phase = 0;
  unsigned int* pending = nullptr;
  // launch-time constants of the division-free index arithmetic: W = qw*G + rw
  long long qw;
  int rw;
  float fw;                                // G / W (estimate)
  DivU64 by_G, by_nvec, by_B;
  __device__ long long vec_of_w(long long w) const {
    return w <= 2 * P ? (w >> 1) : P + (w - 2 * P);
  }
  __device__ long long w_of_vec(long long v) const {
    return v <= P ? 2 * v : 2 * P + (v - P);
  }
  // first vector of CTA c (c = G gives the end): weight floor(W*c/G)
  __device__ long long lo(int c) const {
    if (c >= G) return P + Q;
    return vec_of_w(qw * c + static_cast<long long>(by_G(static_cast<unsigned long long>(rw) * c)));
  }
  // the CTA whose range holds vector v: the largest c with lo(c) <= v (a
  // float estimate, corrected against lo())
  __device__ int cta_of(long long v) const {
    const long long w1 = w_of_vec(v + 1);  // lo(c) <= v  <=>  start weight of c < w1
    int c = static_cast<int>(static_cast<float>(w1 - 1) * fw);
    c = c < 0 ? 0 : (c > G - 1 ? G - 1 : c);
    while (c > 0 && lo(c) > v) --c;
    while (c + 1 < G && lo(c + 1) <= v) ++c;
    return c;
  }
};

namespace {

constexpr int kStages2 = 4;
constexpr int kChunk2 = 512;              // vectors per row per stage (8 KiB)
constexpr int kMaxPending2 = 32;

// Walks [pos, hi) in chunks of at most kChunk2 vectors that never cross a
// pair; the pair and its (position i, sequence b) are tracked incrementally,
// so the loop has no division.
struct PairCursor {
  long long pos, hi, nvec, pair_end;
  int i, b, B;
  __device__ PairCursor(long long lo, long long hi_, const StreamPartition& pt, int B_)
      : pos(lo), hi(hi_), nvec(pt.nvec), B(B_) {
    const long long p = static_cast<long long>(pt.by_nvec(lo));
    pair_end = (p + 1) * nvec;
    i = static_cast<int>(pt.by_B(p));
    b = static_cast<int>(p - static_cast<long long>(i) * B_);
  }
  // next chunk: start, length, the pair's (i, b) and the offset in the pair.
  // A chunk of a draft pair holds kChunk2 vectors of each row; a chunk of a
  // bonus row (i == K, target only) holds 2 * kChunk2, so every stage carries
  // the same bytes and the byte-balanced partition balances chunks too.
  __device__ bool next(long long& start, int& len, int& pi, int& pb, long long& off, int K) {
    if (pos >= hi) return false;
    if (pos >= pair_end) {
      pair_end += nvec;
      if (++b == B) {
        b = 0;
        ++i;
      }
    }
    long long end = pos + (i < K ? kChunk2 : 2 * kChunk2);
    if (end > hi) end = hi;
    if (end > pair_end) end = pair_end;
    start = pos;
    len = static_cast<int>(end - pos);
    pi = i;
    pb = b;
    off = pos - (pair_end - nvec);
    pos = end;
    return true;
  }
};

__device__ __forceinline__ void issue_chunk(const VerifyArgs& a, long long nvec, int i, int b,
                                           long long off, int len, uint4* stage,
                                           unsigned long long* bar, unsigned long long pol_keep,
                                           unsigned long long pol_drop) {
  const uint32_t bytes = static_cast<uint32_t>(len) * 16u;
  if (!(SPEC_IN(static_cast<long long>(b) * (a.K + 1) + i, static_cast<long long>(a.B) * (a.K + 1),
                a.status) &&
        SPEC_IN(off + len - 1, nvec, a.status))) {
    mbar_arrive(bar);  // (debug builds) nothing copied: the stage keeps stale data
    return;
  }
  const uint4* trow = static_cast<const uint4*>(a.target) +
                      (static_cast<size_t>(b) * (a.K + 1) + i) * nvec + off;
  // the row pairs of draft position 0 -- the likeliest first rejection --
  // are kept in L2 in preference to the others (streamed evict-first), so
  // that the decide-and-draw kernel's re-read of the drawn pair more often
  // finds them there.  Measured: position 0 alone beats positions 0-1 and
  // position 0 plus the bonus rows (more than L2 keeps under the stream)
  const unsigned long long pol = i < 1 ? pol_keep : pol_drop;
  if (i < a.K) {
    const uint4* drow = static_cast<const uint4*>(a.draft) +
                        (static_cast<size_t>(b) * a.K + i) * nvec + off;
    mbar_arrive_expect_tx(bar, 2u * bytes);
    bulk_load_hint(stage, trow, bytes, bar, pol);
    bulk_load_hint(stage + kChunk2, drow, bytes, bar, pol);
  } else {
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load_hint(stage, trow, bytes, bar, pol);
  }
}

constexpr int kThreadsA = kThreads + 32;  // 8 consumer warps + 1 producer warp
constexpr int kHalfA = kThreads / 2;      // consumer threads per row of a stage

// Fold up to four 16-byte vectors of one row into a row accumulator (the
// same steps as acc_vectors_impl on two): one offset update and rescale per
// 4 * VEC logits.  kFull: all four are valid.
template <typename E, bool kFull>
__device__ __forceinline__ void acc4(RowAcc& A, const uint4 (&w)[4], int nvalid, float s) {
  constexpr int VEC = Staged<E>::kVec;
  constexpr int NP = 2 * VEC;  // pairs in four vectors
  typename Staged<E>::Max pm = Staged<E>::max_init();
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (kFull || j < nvalid) Staged<E>::max_update(pm, w[j]);
  const float nm = fmaxf(A.ms, Staged<E>::max_value(pm) * s);
  const float f = (A.ms == nm) ? 1.f : ex2(A.ms - nm);
  const float2 s2 = make_float2(s, s), nm2 = make_float2(-nm, -nm);
  float2 e[NP];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float2 x[VEC / 2];
    unpack_pairs<E>(w[j], x);
#pragma unroll
    for (int k = 0; k < VEC / 2; ++k) {
      const float2 t = ffma2(x[k], s2, nm2);
      e[j * (VEC / 2) + k] = (kFull || j < nvalid) ? make_float2(ex2(t.x), ex2(t.y))
                                                   : make_float2(0.f, 0.f);
    }
  }
#pragma unroll
  for (int h = NP / 2; h > 0; h >>= 1)
#pragma unroll
    for (int k = 0; k < h; ++k) e[k] = fadd2(e[k], e[k + h]);
  const float zn = fmaf(A.z, f, e[0].x + e[0].y);
  A.z = (nm == -INFINITY) ? 0.f : zn;
  A.ms = nm;
}

// Consumer warps only (named barrier 1): warp 0 merges the parked partials of
// each (range, pair) over the 8 warps and stores one Partial at its slot
// (range + pair).
__device__ __forceinline__ void flush_partials(const VerifyArgs& a, Partial* partials,
                                               const float4* s_pend, const long long* s_slot,
                                               int npend, int warp, int lane) {
  asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
  if (warp == 0) {
    for (int j = lane; j < npend; j += 32) {
      float4 v = s_pend[j * kWarps];
      for (int w = 1; w < kWarps; ++w) {
        const float4 u = s_pend[j * kWarps + w];
        merge_scaled(v.x, v.y, u.x, u.y);
        merge_scaled(v.z, v.w, u.z, u.w);
      }
      Partial out;
      out.ms_t = v.x; out.z_t = v.y; out.ms_d = v.z; out.z_d = v.w;
      if (SPEC_IN(s_slot[j], a.ws_units, a.status)) partials[s_slot[j]] = out;
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}
static_assert(kChunk2 == 4 * kHalfA, "four vectors per consumer thread of a row per stage");

template <typename E>
__global__ void __launch_bounds__(kThreadsA)
norm_stream_kernel(VerifyArgs a, StreamPartition pt) {
  constexpr int VEC = Staged<E>::kVec;
  extern __shared__ __align__(128) uint4 ring2[];  // [kStages2][target, draft][kChunk2]
  __shared__ __align__(8) unsigned long long full[kStages2];   // copies landed
  __shared__ __align__(8) unsigned long long empty[kStages2];  // consumers done
  __shared__ long long s_slot[kMaxPending2];  // partial slot (range + pair) of each parked entry
  __shared__ float4 s_pend[kMaxPending2 * kWarps];

  // early exit: nothing left to verify after position 0
  if (pt.phase == 2 && *static_cast<volatile unsigned int*>(pt.pending) == 0u) return;
  // the decide-and-sample kernel may be scheduled as soon as SMs free up;
  // it waits for this grid's results before reading them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int c = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long nvec = pt.nvec;
  const long long vlo = pt.lo(c), vhi = pt.lo(c + 1);
  const float s = a.scale;

  if (tid == 0) {
    for (int q = 0; q < kStages2; ++q) {
      mbar_init(&full[q], 1);
      mbar_init(&empty[q], kWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  // ---- producer warp: one thread keeps kStages2 chunks in flight ---------
  if (warp == kWarps) {
    if (lane == 0) {
      const unsigned long long pol_keep = make_policy_evict_last();
      const unsigned long long pol_drop = make_policy_evict_first();
      PairCursor prod(vlo, vhi, pt, a.B);
      bool ok = true;
      long long st, off;
      int len, pi, pb;
      for (int k = 0; prod.next(st, len, pi, pb, off, a.K); ++k) {
        const int q = k % kStages2;
        if (k >= kStages2 && !mbar_wait_sleep(&empty[q], static_cast<uint32_t>((k / kStages2 - 1) & 1)))
          ok = false;
        issue_chunk(a, nvec, pi, pb, off, len, ring2 + static_cast<size_t>(q) * 2 * kChunk2, &full[q],
                    pol_keep, pol_drop);
      }
      if (!ok && a.status) atomicOr(a.status, kWaitTimeout);
    }
    return;
  }

  // ---- consumer warps -----------------------------------------------------
  // Warps 0-3 fold the stage's target vectors, warps 4-7 its draft vectors
  // (for a bonus row: the first and the second half of the double-length
  // target chunk), four vectors a thread, into one accumulator per thread.
  // Per-pair facts are set once per pair; per chunk only 32-bit arithmetic.
  Partial* partials = static_cast<Partial*>(a.partials);
  const int grp = warp >> 2, gtid = tid & (kHalfA - 1);  // row group, thread in group
  long long pos = vlo;
  long long p = static_cast<long long>(pt.by_nvec(vlo));  // current pair
  long long pair_end = (p + 1) * nvec;                     // its end in the flat space
  int ci = static_cast<int>(pt.by_B(p));                   // (position, sequence) of pair p
  int cb = static_cast<int>(p - static_cast<long long>(ci) * a.B);
  int npend = 0;
  RowAcc A{-INFINITY, 0.f};
  bool ok = true;
  // this warp's parked normaliser: the draft row's for group 1 of a draft pair
  auto park = [&](bool draft_pair) {
    float m = A.ms, z = A.z;
    warp_merge_scaled(m, z);
    if (lane == 0)
      s_pend[npend * kWarps + warp] = (grp == 1 && draft_pair) ? make_float4(-INFINITY, 0.f, m, z)
                                                               : make_float4(m, z, -INFINITY, 0.f);
    if (tid == 0) s_slot[npend] = c + p;
    ++npend;
  };

  for (int k = 0; pos < vhi; ++k) {
    if (pos == pair_end) {  // pair change: park the finished pair's partial
      park(ci < a.K);
      if (npend == kMaxPending2) {
        flush_partials(a, partials, s_pend, s_slot, npend, warp, lane);
        npend = 0;
      }
      ++p;
      pair_end += nvec;
      if (++cb == a.B) {
        cb = 0;
        ++ci;
      }
      A = RowAcc{-INFINITY, 0.f};
    }
    const bool has_draft = ci < a.K;  // a (target, draft) pair, else a bonus row
    long long end = pos + (has_draft ? kChunk2 : 2 * kChunk2);
    if (end > vhi) end = vhi;
    if (end > pair_end) end = pair_end;
    const int len = static_cast<int>(end - pos);
    const int q = k % kStages2;
    if (!mbar_wait_sleep(&full[q], static_cast<uint32_t>((k / kStages2) & 1))) ok = false;
    // draft pair: group 0 reads the target half of the stage, group 1 the
    // draft half, len vectors each; bonus row: the two halves of the chunk
    const uint4* src = ring2 + static_cast<size_t>(q) * 2 * kChunk2 + grp * kChunk2;
    const int half = has_draft ? len : (len < kChunk2 ? len : kChunk2);
    const int cnt = grp == 0 ? half : (has_draft ? len : len - half);
    uint4 w[4];
    if (cnt == kChunk2) {  // a full half-stage (warp-uniform): no per-element selects
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = src[gtid + j * kHalfA];
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[q]);  // this warp is done reading stage q
      acc4<E, true>(A, w, 4, s);
    } else {
      int nvalid = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (gtid + j * kHalfA < cnt) {
          w[j] = src[gtid + j * kHalfA];
          nvalid = j + 1;
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[q]);
      acc4<E, false>(A, w, nvalid, s);
    }
    pos = end;
  }
  park(ci < a.K);  // the last pair
  flush_partials(a, partials, s_pend, s_slot, npend, warp, lane);
  if (!ok && a.status) atomicOr(a.status, kWaitTimeout);
}

constexpr int kMaxCB = 8;                // largest cluster of kernel B
constexpr int kMaxK1 = 65;               // K + 1 <= 65 (the API's largest K is 64)
constexpr int kSliceB = 2048;            // vectors per row that one CTA of kernel B aims for

// t[b, i, x] and d[b, i, x] (x clamped into the vocabulary) as fp32.
template <typename E>
__device__ __forceinline__ float2 logits_at(const VerifyArgs& a, int b, int i, int x) {
  const long long xc = min(max(x, 0), a.V - 1);
  const long long ti = (static_cast<long long>(b) * (a.K + 1) + i) * a.V + xc;
  const long long di = (static_cast<long long>(b) * a.K + i) * a.V + xc;
  return make_float2(load_one<E>(a.target, ti), load_one<E>(a.draft, di));
}

// Decision of one sequence, pushed from rank 0 to every CTA of its cluster.
struct Decision {
  float MSt, Zt, MSd, Zd;  // normalisers of the row pair that is drawn from
  float uK;
  int n;                   // number of accepted draft tokens
  int ratio_near;          // a ratio test at a position <= n was within the band
  int pad;
};

template <typename E, int NT>
__global__ void __launch_bounds__(NT, 1024 / NT)  // <= 64 registers
decide_sample_kernel(VerifyArgs a, StreamPartition pt) {
  constexpr int kTB = NT, kWB = NT / 32;  // threads, warps
  constexpr int VEC = Staged<E>::kVec;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int lgC = __ffs(C) - 1;  // C is a power of two
  const int b = static_cast<int>(blockIdx.x >> lgC);
  const int K = a.K, K1 = K + 1;
  const int Klast = pt.phase == 1 ? 0 : K;  // the last position merged and tested
  const long long nvec = pt.nvec;
  const float s = a.scale;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // early exit: nothing left to verify after position 0 (the whole cluster
  // reads the same word)
  if (pt.phase == 2 && *static_cast<volatile unsigned int*>(pt.pending) == 0u) return;

  extern __shared__ __align__(16) unsigned long long tws[];  // [tiles][warps] slice masses
  __shared__ Decision s_dec;                           // this CTA's decision
  __shared__ unsigned long long s_mass[2][kMaxCB];     // pushed by each rank
  __shared__ int s_tok[2];                             // pushed by the crossing CTA to rank 0
  __shared__ float4 s_norm[kMaxK1];                    // per position: (MSt, Zt, MSd, Zd)

  cluster_arrive_relaxed();  // matched by cluster_wait() before the first DSMEM push

  // The call's inputs are complete before the normaliser stream starts, so
  // warp 0 reads the first 32 positions' uniforms, draft tokens and the two
  // logits at each token now, while the stream may still be running.
  const float* u = a.uniforms + static_cast<size_t>(b) * K1;
  float2 g0 = make_float2(0.f, 0.f);
  int x0 = 0;
  float u0 = 0.f;
  if (warp == 0 && lane <= Klast) {
    u0 = u[lane];
    if (lane < K) {
      x0 = a.tokens[static_cast<size_t>(b) * K + lane];
      g0 = logits_at<E>(a, b, lane, x0);
    }
  }

  // everything below reads what the normaliser stream wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- row normalisers (all warps; identical in every CTA) --------------
  // Warp w merges positions w, w + kWB, ...: one lane per contributing range
  // (the loads of up to four positions in flight at once), then a butterfly.
  const Partial* partials = static_cast<const Partial*>(a.partials);
  for (int i0 = warp; i0 <= Klast; i0 += 4 * kWB) {
    Partial q[4];
    int f[4], l[4];
    long long pp[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int i = i0 + t * kWB;
      q[t] = Partial{-INFINITY, 0.f, -INFINITY, 0.f};
      f[t] = 0;
      l[t] = -1;
      pp[t] = 0;
      if (i <= Klast) {
        pp[t] = static_cast<long long>(i) * a.B + b;
        f[t] = pt.cta_of(pp[t] * nvec);
        l[t] = pt.cta_of((pp[t] + 1) * nvec - 1);
        if (f[t] + lane <= l[t] && SPEC_IN(f[t] + lane + pp[t], a.ws_units, a.status))
          q[t] = partials[f[t] + lane + pp[t]];
      }
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int i = i0 + t * kWB;
      if (i <= Klast) {  // warp-uniform
        float mt = q[t].ms_t, zt = q[t].z_t, md = q[t].ms_d, zd = q[t].z_d;
        warp_merge_scaled(mt, zt);
        warp_merge_scaled(md, zd);
        for (int j0 = f[t] + 32; j0 <= l[t]; j0 += 32) {  // rows over more than 32 ranges
          Partial r = Partial{-INFINITY, 0.f, -INFINITY, 0.f};
          if (j0 + lane <= l[t] && SPEC_IN(j0 + lane + pp[t], a.ws_units, a.status))
            r = partials[j0 + lane + pp[t]];
          warp_merge_scaled(r.ms_t, r.z_t);
          warp_merge_scaled(r.ms_d, r.z_d);
          merge_scaled(mt, zt, r.ms_t, r.z_t);
          merge_scaled(md, zd, r.ms_d, r.z_d);
        }
        if (lane == 0) s_norm[i] = make_float4(mt, zt, md, zd);
      }
    }
  }
  __syncthreads();

  // ---- decision (warp 0 of every CTA; identical in all of them) ----------
  // One lane per position: the ratio test, then a ballot gives the first
  // rejection n.  Only rank 0 writes p(x_i), q(x_i) and the status.
  if (warp == 0) {
    const bool writer = rank == 0;
    int n = K, bad = 0, ratio_near = 0;
    float nMSt = 0.f, nZt = 0.f, nMSd = 0.f, nZd = 0.f;
    for (int i0 = 0; i0 <= Klast; i0 += 32) {
      const int i = i0 + lane;
      float MSt = -INFINITY, Zt = 0.f, MSd = -INFINITY, Zd = 0.f;
      bool rej = false, nr = false;
      if (i <= Klast) {
        const float4 nz = s_norm[i];
        MSt = nz.x; Zt = nz.y; MSd = nz.z; Zd = nz.w;
        float2 g = g0;
        int xr = x0;
        float ui = u0;
        if (i0 > 0) {
          ui = u[i];
          if (i < K) {
            xr = a.tokens[static_cast<size_t>(b) * K + i];
            g = logits_at<E>(a, b, i, xr);
          }
        }
        if (!(isfinite(MSt) && isfinite(Zt) && Zt > 0.f)) bad |= kDataNonfiniteLogit;
        if (!(ui >= 0.f && ui < 1.f)) bad |= kDataUniformRange;
        if (i < K) {
          if (xr < 0 || xr >= a.V) bad |= kDataTokenRange;
          if (!(isfinite(MSd) && isfinite(Zd) && Zd > 0.f)) bad |= kDataNonfiniteLogit;
          const float px = ex2(fmaf(g.x, s, -MSt)) / Zt;
          const float qx = ex2(fmaf(g.y, s, -MSd)) / Zd;
          if (writer && a.p_at) a.p_at[static_cast<size_t>(b) * K + i] = px;
          if (writer && a.q_at) a.q_at[static_cast<size_t>(b) * K + i] = qx;
          rej = !(ui * qx < px);
          nr = qx > 0.f && fabsf(ui - fminf(1.f, px / qx)) < kBandF;
        }
      }
      const unsigned rb = __ballot_sync(0xffffffffu, rej);
      const unsigned nb = __ballot_sync(0xffffffffu, nr);
      if (n == K) {  // still no rejection before this round (warp-uniform)
        int pick = -1;
        if (rb) {
          pick = __ffs(rb) - 1;
          n = i0 + pick;
          ratio_near |= (nb & (pick == 31 ? 0xffffffffu : ((2u << pick) - 1u))) != 0u;
        } else {
          ratio_near |= nb != 0u;
          if (Klast == K && K - i0 < 32) pick = K - i0;  // the bonus row is in this round
        }
        if (pick >= 0) {
          nMSt = __shfl_sync(0xffffffffu, MSt, pick);
          nZt = __shfl_sync(0xffffffffu, Zt, pick);
          nMSd = __shfl_sync(0xffffffffu, MSd, pick);
          nZd = __shfl_sync(0xffffffffu, Zd, pick);
        }
      }
    }
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0) {
      if (writer && bad && a.status) atomicOr(a.status, bad);
      Decision d;
      d.MSt = nMSt; d.Zt = nZt; d.MSd = nMSd; d.Zd = nZd;
      d.uK = u[K];
      d.n = n;
      d.ratio_near = ratio_near;
      d.pad = 0;
      s_dec = d;
    }
  }
  __syncthreads();

  if (pt.phase == 1 && s_dec.n == K) {
    // x_0 accepted: this sequence waits for phase 2.  Every CTA of the
    // cluster has read the partials once all have passed the barrier.
    cluster_wait();
    cluster.sync();
    if (rank == 0 && warp == 0) {
      Partial* parts = static_cast<Partial*>(a.partials);
      const long long p = b;  // pair (0, b)
      const int f = pt.cta_of(p * nvec), l = pt.cta_of((p + 1) * nvec - 1);
      for (int c = f + lane; c <= l; c += 32) parts[c + p] = Partial{0.f, 0.f, 0.f, 0.f};
      if (lane == 0) atomicAdd(pt.pending, 1u);
    }
    return;
  }

  // ---- this CTA's slice of row pair n (or of the bonus row) -------------
  // read straight from global memory (the rows were streamed moments ago;
  // no staging, so four CTAs fit on an SM and the grid is one wave)
  const Decision dec = s_dec;
  const int n = dec.n;
  bool residual = n < K;
  const long long v0 = (nvec * rank) >> lgC;
  const int nv = static_cast<int>(((nvec * (rank + 1)) >> lgC) - v0);
  const int ntl = (nv + kTB - 1) / kTB;
  const uint4* trow = static_cast<const uint4*>(a.target) + (static_cast<size_t>(b) * K1 + n) * nvec + v0;
  const uint4* drow = residual
      ? static_cast<const uint4*>(a.draft) + (static_cast<size_t>(b) * K + n) * nvec + v0
      : nullptr;

  // ---- pass 2: fixed-point mass of the slice, per (tile, warp) ------------
  const float MSt = dec.MSt, MSd = dec.MSd;
  const float invZt = 1.f / dec.Zt;
  const float invZd = residual ? 1.f / dec.Zd : 0.f;
  int rnd = 0;
  unsigned long long S = 0;
  for (;; ++rnd) {
    for (int k0 = 0; k0 < ntl; k0 += 4) {  // four tiles of loads in flight
      uint4 wt[4], wd[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = (k0 + j) * kTB + tid;
        if (k0 + j < ntl && v < nv) {
          wt[j] = ld_stream_v4(trow + v);
          if (residual) wd[j] = ld_stream_v4(drow + v);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k = k0 + j;
        if (k < ntl) {  // block-uniform
          const int v = k * kTB + tid;
          float xt[VEC], xd[VEC], r[VEC];
          if (v < nv) {
            Staged<E>::unpack(wt[j], xt);
            if (residual) Staged<E>::unpack(wd[j], xd);
            else {
#pragma unroll
              for (int q = 0; q < VEC; ++q) xd[q] = -INFINITY;
            }
          } else {
#pragma unroll
            for (int q = 0; q < VEC; ++q) xt[q] = xd[q] = -INFINITY;
          }
          const unsigned long long w = warp_sum_mass(
              vec_weight_scaled<VEC>(xt, xd, MSt, invZt, MSd, invZd, s, residual, r));
          if (lane == 0) tws[k * kWB + warp] = w;
        }
      }
    }
    __syncthreads();
    if (rnd == 0) cluster_wait();  // every CTA of the cluster has started
    if (warp == 0) {
      unsigned long long t = 0;
      for (int k = lane; k < ntl * kWB; k += 32) t += tws[k];
      t = warp_sum_u64(t);
      if (lane < C) *cluster.map_shared_rank(&s_mass[rnd][rank], lane) = t;
    }
    cluster.sync();
    S = 0;
    for (int r = 0; r < C; ++r) S += s_mass[rnd][r];
    if (S != 0 || !residual || rnd == 1) break;
    residual = false;  // p == q at this row: the draw falls back to p
  }

  // every CTA of the cluster has read the partials (before the first cluster
  // barrier): rank 0 puts its sequence's slots back to zero, keeping the
  // workspace zero-filled between calls
  if (rank == 0 && warp == 0) {
    Partial* partials = static_cast<Partial*>(a.partials);
    for (int i = lane; i <= Klast; i += 32) {
      const long long p = static_cast<long long>(i) * a.B + b;
      const int f = pt.cta_of(p * nvec), l = pt.cta_of((p + 1) * nvec - 1);
      for (int c = f; c <= l; ++c)
        if (SPEC_IN(c + p, a.ws_units, a.status)) partials[c + p] = Partial{0.f, 0.f, 0.f, 0.f};
    }
  }

  int token = 0, near = 0;
  if (S != 0) {
    const unsigned long long theta = draw_threshold(dec.uK, S);
    int cstar = C - 1;
    unsigned long long off = 0;
    for (int r = 0; r < C; ++r) {
      const unsigned long long m = s_mass[rnd][r];
      if (off + m > theta) { cstar = r; break; }
      off += m;
    }
    // ---- pass 3: the crossing inside the slice of rank cstar (warp 0) ----
    if (rank == cstar && warp == 0 && ntl > 0) {
      const unsigned long long tl = theta - off;
      unsigned long long base = 0;
      int kstar = ntl - 1;
      for (int k0 = 0; k0 < ntl; k0 += 32) {
        const int k = k0 + lane;
        unsigned long long tt = 0;
        if (k < ntl)
          for (int w = 0; w < kWB; ++w) tt += tws[k * kWB + w];
        unsigned long long incl = tt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += o;
        }
        const unsigned int hit = __ballot_sync(0xffffffffu, k < ntl && base + incl > tl);
        if (hit) {
          const int l = __ffs(hit) - 1;
          base += __shfl_sync(0xffffffffu, incl - tt, l);
          kstar = k0 + l;
          break;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
      int wstar = kWB - 1;
      {  // the crossing warp of tile kstar: one lane per warp, scan and ballot
        const unsigned long long m = lane < kWB ? tws[kstar * kWB + lane] : 0ull;
        unsigned long long incl = m;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += o;
        }
        const unsigned int hit = __ballot_sync(0xffffffffu, lane < kWB && base + incl > tl);
        if (hit) wstar = __ffs(hit) - 1;
        base += __shfl_sync(0xffffffffu, incl - m, wstar);
      }
      const int v = kstar * kTB + wstar * 32 + lane;
      float xt[VEC], xd[VEC], r[VEC];
      if (v < nv) {
        Staged<E>::unpack(ld_stream_v4(trow + v), xt);
        if (residual) Staged<E>::unpack(ld_stream_v4(drow + v), xd);
        else {
#pragma unroll
          for (int q = 0; q < VEC; ++q) xd[q] = -INFINITY;
        }
      } else {
#pragma unroll
        for (int q = 0; q < VEC; ++q) xt[q] = xd[q] = -INFINITY;
      }
      const unsigned long long w =
          vec_weight_scaled<VEC, true>(xt, xd, MSt, invZt, MSd, invZd, s, residual, r);
      unsigned long long incl = w;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
      }
      const unsigned int hit = __ballot_sync(0xffffffffu, base + incl > tl);
      const int lstar = hit ? (__ffs(hit) - 1) : 31;
      if (lane == lstar) {
        const unsigned long long before = base + incl - w;
        const unsigned long long rem = tl - before;
        float acc = 0.f;
        int mstar = VEC - 1;
        unsigned long long c_prev = 0, c_cur = w;
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
          acc = __fadd_rn(acc, r[k]);
          const unsigned long long cc = fix56(acc);
          if (cc > rem) { mstar = k; c_cur = cc; break; }
          c_prev = cc;
        }
        const long long t = (v0 + v) * VEC + mstar;
        const bool nr = near_step(theta, off + before + c_prev, off + before + c_cur, S);
        int* dst = cluster.map_shared_rank(&s_tok[0], 0);
        dst[0] = static_cast<int>(t < a.V ? t : a.V - 1);
        dst[1] = nr ? 1 : 0;
      }
    }
    cluster.sync();  // the token has reached rank 0
    token = s_tok[0];
    near = s_tok[1];
  }

  // ---- outputs (warp 0 of rank 0) ----------------------------------------
  if (rank == 0 && warp == 0 && SPEC_IN(b, a.B, a.status) && SPEC_IN(n, K1, a.status)) {
    const int32_t* x = a.tokens + static_cast<size_t>(b) * K;
    int32_t* out = a.out_tokens + static_cast<size_t>(b) * K1;
    for (int j = lane; j < K1; j += 32)
      out[j] = (j < n) ? min(max(x[j], 0), a.V - 1) : (j == n ? token : -1);
    if (lane == 0) {
      if (a.accepted_len) a.accepted_len[b] = n;
      if (a.flags) a.flags[b] = (dec.ratio_near ? kFlagRatio : 0u) | (near ? kFlagCdf : 0u);
      if (a.p_emit) {  // p_n(token) from the drawn row's normaliser
        const float xt = load_one<E>(a.target, (static_cast<long long>(b) * K1 + n) * a.V + token);
        a.p_emit[b] = ex2(fmaf(xt, s, -dec.MSt)) / dec.Zt;
      }
    }
  }
  // early exit, phase 2 (it ran, so *pending > 0): the last CTA to finish --
  // every CTA of the grid has read *pending by then -- puts it back to zero
  if (pt.phase == 2 && tid == 0) {
    FusedCtl* ctl = static_cast<FusedCtl*>(a.ctl);
    if (atom_add_acq_rel_gpu(&ctl->pad[0], 1u) + 1u == gridDim.x) {
      ctl->pending = 0u;
      ctl->pad[0] = 0u;
    }
  }
}

size_t smem_b(long long nvec, int C, int nt) {
  const long long nvs = (nvec + C - 1) / C;
  const long long ntiles = (nvs + nt - 1) / nt;
  return static_cast<size_t>(ntiles * (nt / 32) * 8);
}

// Threads per CTA of kernel B: few clusters (few, long sequences) get larger
// CTAs, so that every SM keeps as many slice loads in flight as when four
// 256-thread CTAs share it -- provided all B clusters of that shape fit on the
// GPU at once.
int threads_b(long long B, int C, const DeviceInfo& dev) {
  int c = 0;
  while ((1 << c) < C && c < 3) ++c;
  const long long ctas = B * C;
  if (ctas <= dev.sm_count && B <= dev.decide_clusters[2][c]) return 1024;
  if (ctas <= 2LL * dev.sm_count && B <= dev.decide_clusters[1][c]) return 512;
  return kThreads;
}

constexpr int kSmemA = kStages2 * 2 * kChunk2 * 16;

}  // namespace

// Cluster size of kernel B: the smallest C in {1, 2, 4, 8} whose slices are
// at most kSliceB vectors per row, else 8; 0 when the slice masses would not
// fit the default shared memory of a CTA.
int sample_2p_cluster(long long nvec) {
  int C = 1;
  while (C < kMaxCB && (nvec + C - 1) / C > kSliceB) C *= 2;
  return smem_b(nvec, C, kThreads) <= 48 * 1024 ? C : 0;
}

cudaError_t sample_2p_prepare(DeviceInfo* d) {
  cudaError_t e = cudaFuncSetAttribute(norm_stream_kernel<BF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemA);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(norm_stream_kernel<F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemA);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d->stream_ctas_per_sm,
                                                      norm_stream_kernel<BF16>, kThreadsA, kSmemA);
  // how many clusters of kernel B fit at once, per (threads, cluster size)
  for (int t = 0; t < 3 && e == cudaSuccess; ++t) {
    for (int c = 0; c < 4 && e == cudaSuccess; ++c) {
      const int nt = 256 << t, C = 1 << c;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned int>(C));
      cfg.blockDim = dim3(nt);
      cfg.dynamicSmemBytes = 4096;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = C;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      e = nt == 1024 ? cudaOccupancyMaxActiveClusters(&n, decide_sample_kernel<BF16, 1024>, &cfg)
          : nt == 512 ? cudaOccupancyMaxActiveClusters(&n, decide_sample_kernel<BF16, 512>, &cfg)
                      : cudaOccupancyMaxActiveClusters(&n, decide_sample_kernel<BF16, kThreads>, &cfg);
      d->decide_clusters[t][c] = n;
    }
  }
  return e;
}

// positions: draft positions streamed (0..positions-1); bonus: the bonus rows too
StreamPartition stream_partition(const VerifyArgs& a, const DeviceInfo& dev, int positions,
                                 bool bonus) {
  StreamPartition pt;
  pt.nvec = static_cast<long long>(a.V) * (a.bf16 ? 2 : 4) / 16;
  pt.P = static_cast<long long>(positions) * a.B * pt.nvec;
  pt.Q = bonus ? static_cast<long long>(a.B) * pt.nvec : 0;
  pt.W = 2 * pt.P + pt.Q;
  // two CTAs per SM: 8 stages of 16 KiB in flight per SM, and room to compute
  const int per_sm = dev.stream_ctas_per_sm < 2 ? (dev.stream_ctas_per_sm > 0 ? dev.stream_ctas_per_sm : 1) : 2;
  long long G = static_cast<long long>(dev.sm_count) * per_sm;
  if (G > kMaxStreamCtas) G = kMaxStreamCtas;
  if (G > pt.W / 4) G = pt.W / 4;  // every CTA owns at least one vector
  if (G < 1) G = 1;
  pt.G = static_cast<int>(G);
  pt.qw = pt.W / G;
  pt.rw = static_cast<int>(pt.W % G);
  pt.fw = static_cast<float>(static_cast<double>(G) / static_cast<double>(pt.W));
  pt.by_G = DivU64::make(static_cast<unsigned long long>(G));
  pt.by_nvec = DivU64::make(static_cast<unsigned long long>(pt.nvec));
  pt.by_B = DivU64::make(static_cast<unsigned long long>(a.B));
  return pt;
}

// The two kernels over partition pt (the second as a programmatic dependent).
cudaError_t launch_2p(const VerifyArgs& a, const DeviceInfo& dev, int C, const StreamPartition& pt,
                      cudaStream_t stream) {
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned int>(pt.G));
    cfg.blockDim = dim3(kThreadsA);
    cfg.dynamicSmemBytes = kSmemA;
    cfg.stream = stream;
    const cudaError_t e = a.bf16 ? cudaLaunchKernelEx(&cfg, norm_stream_kernel<BF16>, a, pt)
                                 : cudaLaunchKernelEx(&cfg, norm_stream_kernel<F32>, a, pt);
    if (e != cudaSuccess) return e;
  }
  const long long grid = static_cast<long long>(a.B) * C;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(grid));
  const int nt = threads_b(a.B, C, dev);
  cfg.blockDim = dim3(nt);
  cfg.dynamicSmemBytes = smem_b(pt.nvec, C, nt);
  if (cfg.dynamicSmemBytes > 48 * 1024) return cudaErrorInvalidConfiguration;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (nt == 1024)
    return a.bf16 ? cudaLaunchKernelEx(&cfg, decide_sample_kernel<BF16, 1024>, a, pt)
                  : cudaLaunchKernelEx(&cfg, decide_sample_kernel<F32, 1024>, a, pt);
  if (nt == 512)
    return a.bf16 ? cudaLaunchKernelEx(&cfg, decide_sample_kernel<BF16, 512>, a, pt)
                  : cudaLaunchKernelEx(&cfg, decide_sample_kernel<F32, 512>, a, pt);
  return a.bf16 ? cudaLaunchKernelEx(&cfg, decide_sample_kernel<BF16, kThreads>, a, pt)
                : cudaLaunchKernelEx(&cfg, decide_sample_kernel<F32, kThreads>, a, pt);
}

cudaError_t launch_sample_2p(const VerifyArgs& a, const DeviceInfo& dev, int C,
                             cudaStream_t stream) {
  return launch_2p(a, dev, C, stream_partition(a, dev, a.K, true), stream);
}

cudaError_t launch_sample_early_exit(const VerifyArgs& a, const DeviceInfo& dev, int C,
                                     cudaStream_t stream) {
  unsigned int* pending = &static_cast<FusedCtl*>(a.ctl)->pending;
  // phase 1: position 0's row pairs; rejecting sequences are drawn and done
  StreamPartition p1 = stream_partition(a, dev, 1, false);
  p1.phase = 1;
  p1.pending = pending;
  cudaError_t e = launch_2p(a, dev, C, p1, stream);
  if (e != cudaSuccess) return e;
  // phase 2: the whole verify, which both kernels skip on the device when
  // no sequence accepted x_0; it recomputes every sequence, the phase-1 ones
  // included (same result, up to the flagged boundary cases)
  StreamPartition p2 = stream_partition(a, dev, a.K, true);
  p2.phase = 2;
  p2.pending = pending;
  // (*pending is zero at rest again: untouched when phase 2 is skipped,
  // reset by phase 2's last CTA otherwise)
  return launch_2p(a, dev, C, p2, stream);
}

}  // namespace specv
