// verify_scd.cu -- speculative contrastive decoding's verify step on sm_103a:
// speculative sampling against the contrastive target P_n of an expert
// (target) and an amateur (drafter), with the bonus token drawn from P_n.
//
// Sources (page title, section):
//   "논문 리뷰 [Speculative Contrastive Decoding]", Speculative Contrastive
//     Decoding: the amateur drafts gamma tokens; the expert checks them
//     against the contrastive-decoding distribution P_n instead of its own;
//     when all are accepted the extra token comes from P_n too.
//   "推测性拒绝采样", 技术原理与步骤 steps 3-4 and 关键保证: the accept test,
//     the first rejection, and the residual law normalize(max(0, P - q)) that
//     keeps the output distributed as the target (here P_n).
// The page lost P_n's formula; this file reads it as contrastive decoding's
//   P_n(j) ~ exp((t_j - a_j) / T)  on the head { t_j >= max t + T ln alpha }
// (p_e(j) >= alpha * max p_e, p_e = softmax(t / T)), 0 elsewhere.  The head
// test is taken exactly: thr = the double M + T ln alpha rounded up to fp32,
// and t_j >= thr in fp32 (thr is the smallest float >= M + T ln alpha).
//
// Design: one cluster of C CTAs per row (b, i), i = 0..K, each CTA a slice
// of at most 2048 16-byte vectors of both rows.  (1) One streaming pass
// reads the slice of the expert row and of the amateur row once from HBM:
// the expert row's maximum (packed NaN-propagating maxima, which also catch
// NaN / +inf), the amateur's online normaliser, and the few vectors that may
// hold head tokens -- a vector is remembered when its maximum is within
// T ln(1/alpha) of the thread's running maximum, a superset of the final
// head since the row maximum is at least the running one.  The cluster
// exchanges maxima and normalisers through DSMEM, which fixes the head.
// (2) Only remembered vectors at or above the head threshold are read again
// (from L2) for the contrast's normaliser, merged in rank order; rank 0 runs
// the accept test of x_i and decides whether the row draws (a rejected draft
// position with no earlier rejection, or the bonus row).  (3) The fixed-
// point masses of max(0, P_n - q) (or of P_n) are non-zero only on head
// vectors, summed per (tile, warp) and per slice, exchanged over the
// cluster; (4) the CTA holding the draw's threshold finds the token and
// stores it as the row's candidate.  The rows of a sequence meet through its
// arrival counter; the last one writes the outputs (the same protocol as the
// streaming sampler).  A thread that meets more candidate vectors than it
// can remember (alpha near 0, where the head is most of the row) makes its
// CTA read its slice again in (2) and (3) instead.
#include <cooperative_groups.h>

#include <cfloat>
#include <climits>
#include <cmath>

#include "../../include/spec_verify.h"
#include "device_common.cuh"
#include "launch.h"
#include "sample_common.cuh"

namespace cg = cooperative_groups;

namespace specv {
namespace {

constexpr int kThreadsS = 256;
constexpr int kWarpsS = kThreadsS / 32;
constexpr int kMaxCS = 8;
constexpr int kSliceVecS = 2048;  // vectors of each row per CTA (8 tiles) when the cluster allows
constexpr int kMaxTilesS = 64;    // tiles of kThreadsS vectors per slice at most
constexpr int kCand = 8;          // head-candidate vectors remembered per thread
constexpr int kU = 4;             // vectors of each row in flight per thread

struct __align__(16) Norm4 {
  float msc, zc, msa, za;
};

// Online normaliser of VEC values relative to a scaled offset: terms
// 2^(x * s - ms).  -inf values add nothing.
template <int VEC>
__device__ __forceinline__ void acc_floats(RowAcc& A, const float (&x)[VEC], float s) {
  float mx = x[0];
#pragma unroll
  for (int k = 1; k < VEC; ++k) mx = fmaxf(mx, x[k]);
  const float nm = fmaxf(A.ms, mx * s);
  if (nm == -INFINITY) return;
  const float f = (A.ms == nm) ? 1.f : ex2(A.ms - nm);
  float e = 0.f;
#pragma unroll
  for (int k = 0; k < VEC; ++k) e += ex2(__fmaf_rn(x[k], s, -nm));
  A.z = fmaf(A.z, f, e);
  A.ms = nm;
}

// Maximum that propagates NaN.
__device__ __forceinline__ float nan_max(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// Largest element of a 16-byte vector, NaN if it holds one.
template <typename E>
__device__ __forceinline__ float vec_max_nan(const uint4 w);
template <>
__device__ __forceinline__ float vec_max_nan<BF16>(const uint4 w) {
  uint32_t m;
  asm("{\n\t.reg .b32 t0, t1;\n\t"
      "max.NaN.bf16x2 t0, %1, %2;\n\tmax.NaN.bf16x2 t1, %3, %4;\n\t"
      "max.NaN.bf16x2 %0, t0, t1;\n\t}"
      : "=r"(m) : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w));
  return nan_max(bf16_lo(m), bf16_hi(m));
}
template <>
__device__ __forceinline__ float vec_max_nan<F32>(const uint4 w) {
  return nan_max(nan_max(__uint_as_float(w.x), __uint_as_float(w.y)),
                 nan_max(__uint_as_float(w.z), __uint_as_float(w.w)));
}

// Largest element of a 16-byte vector (rows already known to hold no NaN).
template <typename E>
__device__ __forceinline__ float vec_max(const uint4 w) {
  typename Staged<E>::Max m = Staged<E>::max_init();
  Staged<E>::max_update(m, w);
  return Staged<E>::max_value(m);
}

// Contrast of one element: t - a on the head, -inf elsewhere.
__device__ __forceinline__ float contrast(float t, float a, float thr) {
  return (t >= thr && t > -INFINITY) ? __fsub_rn(t, a) : -INFINITY;
}

template <typename E>
__global__ void __launch_bounds__(kThreadsS, 5)
scd_row_kernel(VerifyArgs a, const void* amateur, long long nvec, float s, double L, float Lmag) {
  constexpr int VEC = Staged<E>::kVec;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int lgC = __ffs(C) - 1;  // C is a power of two
  const int row = static_cast<int>(blockIdx.x >> lgC);
  const int K = a.K, K1 = K + 1;
  const int b = row / K1, i = row - b * K1;
  const bool has_draft = i < K;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long v0 = (nvec * rank) >> lgC;
  const int nv = static_cast<int>(((nvec * (rank + 1)) >> lgC) - v0);
  const int ntl = (nv + kThreadsS - 1) / kThreadsS;

  extern __shared__ unsigned long long tws[];  // [ntl][warps] masses
  __shared__ uint16_t s_ck[kCand][kThreadsS];  // head-candidate tiles of each thread
  __shared__ float s_cm[kCand][kThreadsS];     // and their vectors' maxima
  __shared__ float s_wmax[kWarpsS];
  __shared__ Norm4 s_warp[kWarpsS];
  __shared__ Norm4 s_part1[kMaxCS];            // (row max, amateur normaliser), pushed by each rank
  __shared__ Norm4 s_part[kMaxCS];             // contrast normaliser, pushed by each rank
  __shared__ unsigned long long s_mass[kMaxCS];
  __shared__ int s_need, s_bad, s_rescan;

  const size_t roff = static_cast<size_t>(row) * nvec;
  const uint4* trow = static_cast<const uint4*>(a.target) + roff + v0;
  const uint4* arow = static_cast<const uint4*>(amateur) + roff + v0;
  if (tid == 0) {
    s_bad = 0;
    s_rescan = 0;
  }
  // the draft token and its two logits, read early by the thread that takes
  // the accept test
  int xr = 0, xcl = 0;
  float tx = 0.f, ax = 0.f;
  if (has_draft && rank == 0 && tid == 0) {
    xr = a.tokens[static_cast<size_t>(b) * K + i];
    xcl = min(max(xr, 0), a.V - 1);
    tx = load_one<E>(static_cast<const uint4*>(a.target) + roff, xcl);
    ax = load_one<E>(static_cast<const uint4*>(amateur) + roff, xcl);
  }
  __syncthreads();
  cluster_arrive_relaxed();  // matched before the first DSMEM push

  // ---- (1) one streaming pass over both rows ------------------------------
  // The expert row's maximum and NaN checks (packed NaN-propagating maxima),
  // the amateur's online normaliser, and the vectors that may hold head
  // tokens: a vector is remembered when its maximum is within T ln(1/alpha)
  // of this thread's running maximum (rounded down: every vector of the
  // final head is remembered, since the row maximum is at least the running
  // one).  A thread with more than kCand of them makes its CTA rescan.
  float mt = -INFINITY, ma = -INFINITY;
  RowAcc Aa{-INFINITY, 0.f};
  int nc = 0;
  for (int k0 = 0; k0 < ntl; k0 += kU) {
    uint4 wt[kU], wa[kU];
    int nval = 0;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = (k0 + u) * kThreadsS + tid;
      if (k0 + u < ntl && v < nv) {
        wt[u] = ld_stream_v4(trow + v);
        wa[u] = ld_stream_v4(arow + v);
        nval = u + 1;
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (u < nval) {
        const float vm = vec_max_nan<E>(wt[u]);
        mt = nan_max(mt, vm);
        ma = nan_max(ma, vec_max_nan<E>(wa[u]));
        if (vm >= __fsub_rd(mt, Lmag)) {
          if (nc < kCand) {
            s_ck[nc][tid] = static_cast<uint16_t>(k0 + u);
            s_cm[nc][tid] = vm;
          }
          ++nc;
        }
      }
    }
    if (has_draft) {
#pragma unroll
      for (int u = 0; u < kU; u += 2) {
        const int n2 = min(max(nval - u, 0), 2);
        if (n2 > 0) {
          const uint4 w2[2] = {wa[u], wa[u + 1]};
          acc_vectors<E>(Aa, w2, n2, s);
        }
      }
    }
  }
  const bool bad = isnan(mt) || mt == INFINITY || isnan(ma) || ma == INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mt = nan_max(mt, __shfl_xor_sync(0xffffffffu, mt, o));
  warp_merge_scaled(Aa.ms, Aa.z);
  if (lane == 0) {
    s_wmax[warp] = mt;
    s_warp[warp] = Norm4{-INFINITY, 0.f, Aa.ms, Aa.z};
  }
  if (__syncthreads_or(bad) && tid == 0) s_bad = 1;
  if (__syncthreads_or(nc > kCand) && tid == 0) s_rescan = 1;
  cluster_wait();  // every CTA of the cluster has started
  if (warp == 0) {
    float m = lane < kWarpsS ? s_wmax[lane] : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = nan_max(m, __shfl_xor_sync(0xffffffffu, m, o));
    Norm4 p = lane < kWarpsS ? s_warp[lane] : Norm4{-INFINITY, 0.f, -INFINITY, 0.f};
    warp_merge_scaled(p.msa, p.za);
    p.msc = m;  // the slice's maximum rides in the first field
    if (lane < C) *cluster.map_shared_rank(&s_part1[rank], lane) = p;
  }
  cluster.sync();
  float M = -INFINITY, MSa = -INFINITY, Za = 0.f;
  for (int r = 0; r < C; ++r) {  // rank order: the same bits in every CTA
    M = nan_max(M, s_part1[r].msc);
    merge_scaled(MSa, Za, s_part1[r].msa, s_part1[r].za);
  }
  const float thr = __double2float_ru(__dadd_rn(static_cast<double>(M), L));
  const bool rescan = s_rescan != 0;
  const int ncs = min(nc, kCand);

  // ---- (2) the contrast's normaliser on the head --------------------------
  // Only remembered vectors at or above the threshold are read again (from
  // L2, shortly after the stream); a rescanning CTA reads its slice again.
  RowAcc Ac{-INFINITY, 0.f};
  bool unbounded = false;  // a head token the amateur gives no mass
  for (int c = 0; c < (rescan ? ntl : ncs); ++c) {
    int v;
    if (rescan) {
      v = c * kThreadsS + tid;
      if (v >= nv) break;
    } else {
      if (!(s_cm[c][tid] >= thr)) continue;
      v = s_ck[c][tid] * kThreadsS + tid;
    }
    const uint4 wt = __ldg(trow + v);
    if (!(vec_max<E>(wt) >= thr)) continue;
    float xt[VEC], xa[VEC], xc[VEC];
    Staged<E>::unpack(wt, xt);
    Staged<E>::unpack(__ldg(arow + v), xa);
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      xc[k] = contrast(xt[k], xa[k], thr);
      unbounded |= xc[k] == INFINITY;
    }
    acc_floats<VEC>(Ac, xc, s);
  }
  warp_merge_scaled(Ac.ms, Ac.z);
  if (lane == 0) {
    s_warp[warp].msc = Ac.ms;
    s_warp[warp].zc = Ac.z;
  }
  if (__syncthreads_or(unbounded) && tid == 0) s_bad = 1;
  if (warp == 0) {
    Norm4 m = lane < kWarpsS ? s_warp[lane] : Norm4{-INFINITY, 0.f, -INFINITY, 0.f};
    warp_merge_scaled(m.msc, m.zc);
    if (lane < C) *cluster.map_shared_rank(&s_part[rank], lane) = m;
  }
  cluster.sync();
  float MSc = -INFINITY, Zc = 0.f;
  for (int r = 0; r < C; ++r) merge_scaled(MSc, Zc, s_part[r].msc, s_part[r].zc);
  const bool norm_ok = isfinite(MSc) && isfinite(Zc) && Zc > 0.f &&
                       (!has_draft || (isfinite(MSa) && isfinite(Za) && Za > 0.f));
  const float invZc = norm_ok ? 1.f / Zc : 0.f;
  const float invZa = (norm_ok && has_draft) ? 1.f / Za : 0.f;
  const float uK = a.uniforms[static_cast<size_t>(b) * K1 + K];

  // ---- accept test and whether this row needs a draw (rank 0) -------------
  // A row draws when its draft token is rejected and no earlier position has
  // been rejected yet, and the bonus row always; the sequence's last arrival
  // picks the first rejected row's candidate.
  if (rank == 0 && tid == 0) {
    SeqState* st = a.seq + b;
    int err = norm_ok ? 0 : kDataNonfiniteLogit;
    bool need = true;
    if (has_draft) {
      const float ui = a.uniforms[static_cast<size_t>(b) * K1 + i];
      const float cx = contrast(tx, ax, thr);
      const float px = __fmul_rn(ex2(__fmaf_rn(cx, s, -MSc)), invZc);
      const float qx = __fmul_rn(ex2(__fmaf_rn(ax, s, -MSa)), invZa);
      const bool accept = ui * qx < px;
      if (a.p_at) a.p_at[static_cast<size_t>(b) * K + i] = px;
      if (a.q_at) a.q_at[static_cast<size_t>(b) * K + i] = qx;
      if (xr != xcl) err |= kDataTokenRange;
      if (!(ui >= 0.f && ui < 1.f)) err |= kDataUniformRange;
      if (qx > 0.f && fabsf(ui - fminf(1.f, px / qx)) < kBandF)
        atomicOr(&st->near_mask, 1ull << i);
      if (!accept) atomicOr(&st->reject_mask, 1ull << i);
      need = !accept;
    } else if (!(uK >= 0.f && uK < 1.f)) {
      err |= kDataUniformRange;
    }
    if (err && a.status) atomicOr(a.status, err);
    __threadfence();
    if (need) {
      const unsigned long long m = *reinterpret_cast<volatile unsigned long long*>(&st->reject_mask);
      const unsigned long long earlier = (i >= 64) ? ~0ull : ((1ull << i) - 1ull);
      if (m & earlier) need = false;  // an earlier position already rejected
    }
    for (int r = 0; r < C; ++r) *cluster.map_shared_rank(&s_need, r) = need ? 1 : 0;
  }
  // any CTA that saw a bad element reports it
  if (tid == 0 && s_bad && a.status) atomicOr(a.status, kDataNonfiniteLogit);
  cluster.sync();
  if (!s_need) {
    if (rank == 0 && warp == 0) warp_arrive_and_finalize(a, b);
    return;
  }

  // ---- (3) fixed-point masses of max(0, P_n - q) (or P_n) -----------------
  // P_n is 0 off the head, and so is max(0, P_n - q): only head vectors have
  // mass; the per-(tile, warp) sums keep the slice's order for the crossing.
  bool residual = has_draft;
  unsigned long long S = 0;
  for (int rnd = 0; rnd < 2; ++rnd) {
    int ci = 0;
    for (int k = 0; k < ntl; ++k) {
      const int v = k * kThreadsS + tid;
      bool look = false;
      if (rescan) {
        look = v < nv;
      } else {
        while (ci < ncs && s_ck[ci][tid] < k) ++ci;
        look = ci < ncs && s_ck[ci][tid] == k && s_cm[ci][tid] >= thr;
      }
      unsigned long long w = 0;
      if (!__any_sync(0xffffffffu, look)) {  // no head vector in this warp's tile
        if (lane == 0) tws[k * kWarpsS + warp] = 0ull;
        continue;
      }
      if (look) {
        const uint4 wt = __ldg(trow + v);
        if (vec_max<E>(wt) >= thr) {
          float xt[VEC], xa[VEC], xc[VEC], r[VEC];
          Staged<E>::unpack(wt, xt);
          Staged<E>::unpack(__ldg(arow + v), xa);
#pragma unroll
          for (int q = 0; q < VEC; ++q) xc[q] = contrast(xt[q], xa[q], thr);
          w = vec_weight_scaled<VEC>(xc, xa, MSc, invZc, MSa, invZa, s, residual, r);
        }
      }
      w = warp_sum_mass(w);
      if (lane == 0) tws[k * kWarpsS + warp] = w;
    }
    __syncthreads();
    if (warp == 0) {
      unsigned long long t = 0;
      for (int k = lane; k < ntl * kWarpsS; k += 32) t += tws[k];
      t = warp_sum_u64(t);
      if (lane < C) *cluster.map_shared_rank(&s_mass[rank], lane) = t;
    }
    cluster.sync();
    S = 0;
    for (int r = 0; r < C; ++r) S += s_mass[r];
    if (S != 0 || !residual) break;
    residual = false;  // P_n == q at this row: the draw falls back to P_n
    cluster.sync();    // every CTA has read s_mass before it is pushed again
  }

  // ---- (4) the crossing, in the CTA that holds it (warp 0) ----------------
  const unsigned long long theta = draw_threshold(uK, S);
  int cstar = C - 1;
  unsigned long long off = 0;
  for (int r = 0; r < C; ++r) {
    if (off + s_mass[r] > theta) {
      cstar = r;
      break;
    }
    off += s_mass[r];
  }
  if (rank != cstar || warp != 0) return;
  int32_t cand = 0;
  if (S != 0 && ntl > 0) {
    const unsigned long long tl = theta - off;
    unsigned long long base = 0;
    int kstar = ntl - 1;
    for (int k0 = 0; k0 < ntl; k0 += 32) {
      const int k = k0 + lane;
      unsigned long long tt = 0;
      if (k < ntl)
        for (int w = 0; w < kWarpsS; ++w) tt += tws[k * kWarpsS + w];
      const unsigned long long incl = warp_scan_u64(tt, lane);
      const unsigned int hit = __ballot_sync(0xffffffffu, k < ntl && base + incl > tl);
      if (hit) {
        const int l = __ffs(hit) - 1;
        base += __shfl_sync(0xffffffffu, incl - tt, l);
        kstar = k0 + l;
        break;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    int wstar = kWarpsS - 1;
    {
      const unsigned long long m = lane < kWarpsS ? tws[kstar * kWarpsS + lane] : 0ull;
      const unsigned long long incl = warp_scan_u64(m, lane);
      const unsigned int hit = __ballot_sync(0xffffffffu, lane < kWarpsS && base + incl > tl);
      if (hit) wstar = __ffs(hit) - 1;
      base += __shfl_sync(0xffffffffu, incl - m, wstar);
    }
    const int v = kstar * kThreadsS + wstar * 32 + lane;
    float xc[VEC], xa[VEC], r[VEC];
    if (v < nv) {
      float xt[VEC];
      Staged<E>::unpack(__ldg(trow + v), xt);
      Staged<E>::unpack(__ldg(arow + v), xa);
#pragma unroll
      for (int q = 0; q < VEC; ++q) xc[q] = contrast(xt[q], xa[q], thr);
    } else {
#pragma unroll
      for (int q = 0; q < VEC; ++q) xc[q] = xa[q] = -INFINITY;
    }
    const unsigned long long w =
        vec_weight_scaled<VEC, true>(xc, xa, MSc, invZc, MSa, invZa, s, residual, r);
    const unsigned long long incl = warp_scan_u64(w, lane);
    const unsigned int hit = __ballot_sync(0xffffffffu, base + incl > tl);
    const int lstar = hit ? __ffs(hit) - 1 : 31;
    if (lane == lstar) {
      const unsigned long long before = base + incl - w;
      unsigned long long c_prev, c_cur;
      const int mstar = pick_in_vector<VEC>(r, w, tl - before, c_prev, c_cur);
      const long long t = (v0 + v) * VEC + mstar;
      const int32_t tok = static_cast<int32_t>(t < a.V ? t : a.V - 1);
      const bool near = near_step(theta, off + before + c_prev, off + before + c_cur, S);
      cand = near ? static_cast<int32_t>(static_cast<uint32_t>(tok) | 0x80000000u) : tok;
    }
    cand = __shfl_sync(0xffffffffu, cand, lstar);
  }
  if (lane == 0) {
    *candidate_slot(a, b, i) = cand;
    __threadfence();
  }
  __syncwarp();
  warp_arrive_and_finalize(a, b);
}

}  // namespace

// Cluster size for row pairs of nvec vectors: the smallest C in {1, 2, 4, 8}
// whose slices hold at most kSliceVecS vectors, else 8 while a slice stays
// within kMaxTilesS tiles; 0 when the rows are too long.
int scd_cluster(long long nvec) {
  for (int C = 1; C <= kMaxCS; C *= 2)
    if ((nvec + C - 1) / C <= kSliceVecS) return C;
  if ((nvec + kMaxCS - 1) / kMaxCS <= static_cast<long long>(kMaxTilesS) * kThreadsS) return kMaxCS;
  return 0;
}

static size_t scd_smem(long long nvec, int C) {
  const long long nvs = (nvec + C - 1) / C;
  const long long ntl = (nvs + kThreadsS - 1) / kThreadsS;
  return static_cast<size_t>(ntl * kWarpsS * 8);
}

cudaError_t scd_prepare() { return cudaSuccess; }

cudaError_t launch_scd(const VerifyArgs& a, const void* amateur, double L, int C,
                       cudaStream_t stream) {
  const int esz = a.bf16 ? 2 : 4;
  const long long nvec = static_cast<long long>(a.V) * esz / 16;
  const long long grid = static_cast<long long>(a.B) * (a.K + 1) * C;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  // |L| rounded up to fp32, for the candidates' conservative test
  float Lmag = static_cast<float>(-L);
  if (static_cast<double>(Lmag) < -L) Lmag = std::nextafter(Lmag, INFINITY);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(grid));
  cfg.blockDim = dim3(kThreadsS);
  cfg.dynamicSmemBytes = scd_smem(nvec, C);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.bf16
             ? cudaLaunchKernelEx(&cfg, scd_row_kernel<BF16>, a, amateur, nvec, a.scale, L, Lmag)
             : cudaLaunchKernelEx(&cfg, scd_row_kernel<F32>, a, amateur, nvec, a.scale, L, Lmag);
}

}  // namespace specv
