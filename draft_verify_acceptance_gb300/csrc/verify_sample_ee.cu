// verify_sample_ee.cu -- early-exit speculative sampling on sm_103a: one
// cluster of C CTAs per sequence walks the draft positions in order and
// stops reading rows at the first rejection.
//
// Sources (page title, section):
//   "推测性拒绝采样", 技术原理与步骤 steps 2-4 and 关键保证: x_i is accepted
//     when u_i * q_i(x_i) < p_i(x_i); once a token is rejected every later
//     one is dropped and one token is drawn from normalize(max(0, p - q))
//     there, which keeps the output distributed as the target.
//   "논문 리뷰 [Speculative Contrastive Decoding]", Speculative Decoding: with
//     all K accepted the target supplies token K+1, drawn from p_K.
//
// Design: each CTA stages its slice of the position's target row and draft
// row in shared memory (TMA bulk copies of 32 KiB, one mbarrier each), so a
// row crosses HBM once and the draw at the rejected position reads nothing
// again.  Per position: (1) both rows' online normalisers as the copies land
// (max and sum of 2^(x*s - offset)), exchanged over the cluster through DSMEM
// in one step; (2) every CTA takes the same accept decision from the same
// values (the token's two logits are read once from global memory).  At the
// first rejection (or at the bonus row): the fixed-point masses of
// max(0, p - q) (or of p) per 16-byte vector, the verifier's scheme, summed
// per lane with a checkpoint every four steps of 32 vectors; slice masses
// over DSMEM; the CTA holding u_K * S finds the warp range, the checkpoint
// group, the step, the lane and the element, and writes the outputs.  Two
// cluster exchanges per draw plus one per accepted position; no workspace,
// no global atomics; every wait is bounded.
#include <cooperative_groups.h>

#include <cfloat>
#include <climits>

#include "device_common.cuh"
#include "launch.h"
#include "launch_ee.h"
#include "sample_common.cuh"

namespace cg = cooperative_groups;

namespace specv {
namespace {

constexpr int kThreadsE = 512;
constexpr int kWarpsE = kThreadsE / 32;
constexpr int kMaxCE = 8;
constexpr int kChunkE = 2048;                  // vectors per bulk copy (32 KiB)
constexpr long long kBudgetE = 200 * 1024;     // slices and checkpoints of one CTA
constexpr int kMaxChunksE = static_cast<int>(kBudgetE / 2 / 16 / kChunkE) + 1;
constexpr int kGroupE = 4;                     // 32-vector steps between a lane's checkpoints
static_assert(kGroupE <= kWarpsE, "one warp per step of the crossing group");
static_assert(kChunkE % kThreadsE == 0, "whole vectors per thread in a full chunk");

__host__ __device__ __forceinline__ int ee_steps(int nv) {
  return ((nv + kWarpsE - 1) / kWarpsE + 31) / 32;
}
__host__ __device__ __forceinline__ int ee_groups(int nv) {
  return (ee_steps(nv) + kGroupE - 1) / kGroupE;
}
__host__ __device__ __forceinline__ long long ee_smem(long long nvec, int C) {
  const long long nvs = (nvec + C - 1) / C;
  return 2 * nvs * 16 + static_cast<long long>(ee_groups(static_cast<int>(nvs))) * kWarpsE * 32 * 8;
}

// The fixed-point residual mass of staged vector v (max(0, p - q), or p).
template <typename E, bool kInt = false>
__device__ __forceinline__ unsigned long long vec_mass(const uint4* st, const uint4* sd, int v,
                                                       float MSt, float invZt, float MSd,
                                                       float invZd, float s, bool residual,
                                                       float (&r)[Staged<E>::kVec]) {
  constexpr int VEC = Staged<E>::kVec;
  float xt[VEC], xd[VEC];
  Staged<E>::unpack(st[v], xt);
  if (residual) {
    Staged<E>::unpack(sd[v], xd);
  } else {
#pragma unroll
    for (int q = 0; q < VEC; ++q) xd[q] = -INFINITY;
  }
  return vec_weight_scaled<VEC, kInt>(xt, xd, MSt, invZt, MSd, invZd, s, residual, r);
}

template <typename E>
__global__ void __launch_bounds__(kThreadsE, 1)
ee_cluster_kernel(VerifyArgs a, long long nvec) {
  constexpr int VEC = Staged<E>::kVec;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int lgC = __ffs(C) - 1;  // C is a power of two
  const int b = static_cast<int>(blockIdx.x >> lgC);
  const int K = a.K, K1 = K + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float s = a.scale;
  const bool solo = C == 1;  // a one-CTA cluster: CTA barriers stand in for the cluster's
  const long long v0 = (nvec * rank) >> lgC;
  const int nv = static_cast<int>(((nvec * (rank + 1)) >> lgC) - v0);
  const int nvs = static_cast<int>((nvec + C - 1) >> lgC);
  const int nch = (nv + kChunkE - 1) / kChunkE;
  const int steps = ee_steps(nv), ngr = ee_groups(nv);
  const int lo = (nv * warp) / kWarpsE, hi = (nv * (warp + 1)) / kWarpsE;  // this warp's range

  extern __shared__ __align__(128) uint4 smem[];
  uint4* st = smem;        // [nvs] the position's target slice
  uint4* sd = smem + nvs;  // [nvs] its draft slice
  unsigned long long* cp = reinterpret_cast<unsigned long long*>(smem + 2 * static_cast<size_t>(nvs));
  __shared__ __align__(8) unsigned long long bar_t[kMaxChunksE], bar_d[kMaxChunksE];
  __shared__ float4 s_wn[kWarpsE];                 // per-warp (target, draft) normalisers
  __shared__ float4 s_n[2][kMaxCE];                // pushed by each rank, per position parity
  __shared__ unsigned long long s_wm[kWarpsE];     // per-warp masses
  __shared__ unsigned long long s_mass[2][kMaxCE]; // pushed by each rank, per round
  __shared__ int s_tok[2];                         // the drawn token and its near flag
  __shared__ int s_dec[3];                         // the position's rejection, near flag, errors
  __shared__ int s_sel[2];                         // crossing warp and group
  __shared__ unsigned long long s_tl;              // threshold left inside the group
  __shared__ unsigned long long s_cm[kGroupE][32]; // lane masses of the crossing group
  __shared__ unsigned long long s_ct[kGroupE];     // its steps' masses
  __shared__ int s_fail;                           // a copy never landed

  if (tid == 0) {
    for (int c = 0; c < nch; ++c) {
      mbar_init(&bar_t[c], 1);
      mbar_init(&bar_d[c], 1);
    }
    fence_barrier_init();
    s_fail = 0;
    s_tok[0] = 0;
    s_tok[1] = 0;
  }
  __syncthreads();
  if (!solo) cluster_arrive_relaxed();  // matched before the first DSMEM push

  const size_t esz = E::kBytes;
  const char* tbase = static_cast<const char*>(a.target) + static_cast<size_t>(b) * K1 * a.V * esz;
  const char* dbase = static_cast<const char*>(a.draft) + static_cast<size_t>(b) * K * a.V * esz;
  const float* ub = a.uniforms + static_cast<size_t>(b) * K1;
  const float uK = ub[K];

  int n = K;           // first rejected position (K: all accepted)
  int ratio_near = 0;  // a ratio test at a position <= n was within the band
  int bad = 0;         // data-error bits
  float MSt = 0.f, Zt = 1.f, MSd = 0.f, Zd = 1.f;
  bool waited = solo;  // the cluster's start barrier has been passed
  for (int i = 0; i <= K; ++i) {
    const bool pair = i < K;
    const uint32_t par = static_cast<uint32_t>(i & 1);  // every barrier completes once per position
    // ---- stage position i's slices (thread 0) -----------------------------
    if (tid == 0 && !s_fail) {
      // the CTA's reads of the previous position are done (barrier below):
      // order them before the async proxy writes the same shared memory
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const uint4* tr = reinterpret_cast<const uint4*>(tbase + static_cast<size_t>(i) * a.V * esz) + v0;
      const uint4* dr = reinterpret_cast<const uint4*>(dbase + static_cast<size_t>(i) * a.V * esz) + v0;
      for (int c = 0; c < nch; ++c) {
        const uint32_t bytes = static_cast<uint32_t>(min(kChunkE, nv - c * kChunkE)) * 16u;
        mbar_arrive_expect_tx(&bar_t[c], bytes);
        bulk_load(st + c * kChunkE, tr + c * kChunkE, bytes, &bar_t[c]);
        if (pair) {
          mbar_arrive_expect_tx(&bar_d[c], bytes);
          bulk_load(sd + c * kChunkE, dr + c * kChunkE, bytes, &bar_d[c]);
        }
      }
    }
    // the draft token, its two logits and u_i (thread 0; the same in every CTA)
    int xr = 0;
    float tx = 0.f, dx = 0.f, ui = uK;
    if (tid == 0 && pair) {
      ui = ub[i];
      xr = a.tokens[static_cast<size_t>(b) * K + i];
      const int xc = min(max(xr, 0), a.V - 1);
      tx = load_one<E>(tbase + static_cast<size_t>(i) * a.V * esz, xc);
      dx = load_one<E>(dbase + static_cast<size_t>(i) * a.V * esz, xc);
    }

    // ---- (1) online normalisers as the copies land, one exchange ----------
    RowAcc At{-INFINITY, 0.f}, Ad{-INFINITY, 0.f};
    // after a copy that never landed the barriers' phases are lost: every
    // later wait is skipped (the outputs are unspecified, the status says so)
    bool ok = s_fail == 0;
    for (int c = 0; ok && c < nch; ++c) {
      if (!mbar_wait_sleep(&bar_t[c], par) || (pair && !mbar_wait_sleep(&bar_d[c], par))) {
        ok = false;
        break;
      }
      const int c0 = c * kChunkE, cend = min(c0 + kChunkE, nv);
      if (cend - c0 == kChunkE) {  // a full chunk: pairs of vectors of each row a thread
#pragma unroll
        for (int k = 0; k < kChunkE / kThreadsE; k += 2) {
          const uint4 wt[2] = {st[c0 + k * kThreadsE + tid], st[c0 + (k + 1) * kThreadsE + tid]};
          acc_vectors_full<E>(At, wt, s);
          if (pair) {
            const uint4 wd[2] = {sd[c0 + k * kThreadsE + tid], sd[c0 + (k + 1) * kThreadsE + tid]};
            acc_vectors_full<E>(Ad, wd, s);
          }
        }
      } else {
        for (int v = c0 + tid; v < cend; v += 2 * kThreadsE) {
          const int n2 = 1 + (v + kThreadsE < cend ? 1 : 0);
          uint4 wt[2], wd[2];
          wt[0] = st[v];
          if (pair) wd[0] = sd[v];
          if (n2 > 1) {
            wt[1] = st[v + kThreadsE];
            if (pair) wd[1] = sd[v + kThreadsE];
          }
          acc_vectors<E>(At, wt, n2, s);
          if (pair) acc_vectors<E>(Ad, wd, n2, s);
        }
      }
    }
    warp_merge_scaled(At.ms, At.z);
    warp_merge_scaled(Ad.ms, Ad.z);
    if (lane == 0) s_wn[warp] = make_float4(At.ms, At.z, Ad.ms, Ad.z);
    if (__syncthreads_or(!ok) && tid == 0) s_fail = 1;
    if (!waited) {
      cluster_wait();  // every CTA of the cluster has started
      waited = true;
    }
    float4* s_nb = s_n[i & 1];  // one buffer per position parity: a peer a
                                // position ahead never overwrites a value in use
    if (warp == 0) {
      float4 m = lane < kWarpsE ? s_wn[lane] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
      warp_merge_scaled(m.x, m.y);
      warp_merge_scaled(m.z, m.w);
      if (solo) {
        if (lane == 0) s_nb[0] = m;
      } else if (lane < C) {
        *cluster.map_shared_rank(&s_nb[rank], lane) = m;
      }
    }
    if (solo) __syncthreads();
    else cluster.sync();
    MSt = -INFINITY;
    Zt = 0.f;
    MSd = -INFINITY;
    Zd = 0.f;
    for (int r = 0; r < C; ++r) {  // rank order: the same bits in every CTA
      merge_scaled(MSt, Zt, s_nb[r].x, s_nb[r].y);
      merge_scaled(MSd, Zd, s_nb[r].z, s_nb[r].w);
    }

    // ---- (2) the accept test, the same in every CTA -----------------------
    if (tid == 0) {
      int err = 0, rej = 1, nr = 0;
      if (!(isfinite(MSt) && isfinite(Zt) && Zt > 0.f)) err |= kDataNonfiniteLogit;
      if (!(ui >= 0.f && ui < 1.f)) err |= kDataUniformRange;
      if (pair) {
        if (xr < 0 || xr >= a.V) err |= kDataTokenRange;
        if (!(isfinite(MSd) && isfinite(Zd) && Zd > 0.f)) err |= kDataNonfiniteLogit;
        const float px = ex2(fmaf(tx, s, -MSt)) / Zt;
        const float qx = ex2(fmaf(dx, s, -MSd)) / Zd;
        if (rank == 0 && a.p_at) a.p_at[static_cast<size_t>(b) * K + i] = px;
        if (rank == 0 && a.q_at) a.q_at[static_cast<size_t>(b) * K + i] = qx;
        rej = !(ui * qx < px) ? 1 : 0;
        nr = (qx > 0.f && fabsf(ui - fminf(1.f, px / qx)) < kBandF) ? 1 : 0;
      }
      s_dec[0] = rej;
      s_dec[1] = nr;
      s_dec[2] = err;
    }
    __syncthreads();
    ratio_near |= s_dec[1];
    bad |= s_dec[2];
    if (s_dec[0]) {  // the first rejection (or the bonus row): draw here
      n = i;
      break;
    }
    __syncthreads();  // every read of s_dec and of the slices is done before they change
  }

  // ---- the draw from position n: fixed-point masses, lane checkpoints ------
  bool residual = n < K;
  const float invZt = (isfinite(Zt) && Zt > 0.f) ? 1.f / Zt : 0.f;
  float invZd = (residual && isfinite(Zd) && Zd > 0.f) ? 1.f / Zd : 0.f;
  unsigned long long S = 0;
  int rnd = 0;
  for (;; ++rnd) {
    unsigned long long run = 0;
    unsigned long long* mycp = cp + static_cast<size_t>(warp) * ngr * 32 + lane;
    for (int g = 0; g < ngr; ++g) {
      for (int jj = 0; jj < kGroupE; ++jj) {
        const int v = lo + (g * kGroupE + jj) * 32 + lane;
        if (v < hi) {
          float r[VEC];
          run += vec_mass<E>(st, sd, v, MSt, invZt, MSd, invZd, s, residual, r);
        }
      }
      mycp[g * 32] = run;
    }
    const unsigned long long wm = warp_sum_u64(run);
    if (lane == 0) s_wm[warp] = wm;
    __syncthreads();
    if (warp == 0) {
      const unsigned long long t = warp_sum_u64(lane < kWarpsE ? s_wm[lane] : 0ull);
      if (solo) {
        if (lane == 0) s_mass[rnd][0] = t;
      } else if (lane < C) {
        *cluster.map_shared_rank(&s_mass[rnd][rank], lane) = t;
      }
    }
    if (solo) __syncthreads();
    else cluster.sync();
    S = 0;
    for (int r = 0; r < C; ++r) S += s_mass[rnd][r];
    if (S != 0 || !residual || rnd == 1) break;
    residual = false;  // p == q at this position: the draw falls back to p
    invZd = 0.f;
    __syncthreads();   // the checkpoints are read again only after this round
  }

  // ---- the crossing, in the CTA that holds it ------------------------------
  const unsigned long long theta = draw_threshold(uK, S);
  int cstar = C - 1;
  unsigned long long off = 0;
  for (int r = 0; r < C; ++r) {
    const unsigned long long m = s_mass[rnd][r];
    if (off + m > theta) {
      cstar = r;
      break;
    }
    off += m;
  }
  if (S != 0 && rank == cstar && nv > 0) {
    // warp 0: the warp range (lane w holds the prefix through warp w), then
    // the checkpoint group in it (lane g holds the prefix through group g)
    if (warp == 0) {
      unsigned long long tl = theta - off;
      const unsigned long long m = lane < kWarpsE ? s_wm[lane] : 0ull;
      const unsigned long long incl = warp_scan_u64(m, lane);
      unsigned int hit = __ballot_sync(0xffffffffu, lane < kWarpsE && incl > tl);
      const int ws = hit ? __ffs(hit) - 1 : kWarpsE - 1;
      tl -= min(__shfl_sync(0xffffffffu, incl - m, ws), tl);
      unsigned long long mine = 0;
      for (int g = 0; g < ngr; ++g) {
        const unsigned long long gp = warp_sum_u64(cp[(static_cast<size_t>(ws) * ngr + g) * 32 + lane]);
        if (lane == g) mine = gp;
      }
      hit = __ballot_sync(0xffffffffu, lane < ngr && mine > tl);
      const int gs = hit ? __ffs(hit) - 1 : ngr - 1;
      const unsigned long long before = gs > 0 ? __shfl_sync(0xffffffffu, mine, gs - 1) : 0ull;
      if (lane == 0) {
        s_sel[0] = ws;
        s_sel[1] = gs;
        s_tl = tl - min(before, tl);
      }
    }
    __syncthreads();
    const int ws = s_sel[0], gs = s_sel[1];
    const int wlo = (nv * ws) / kWarpsE, whi = (nv * (ws + 1)) / kWarpsE;
    if (warp < kGroupE) {  // warp j recomputes step gs * kGroupE + j of warp ws's range
      const int j = gs * kGroupE + warp;
      const int v = wlo + j * 32 + lane;
      unsigned long long m = 0;
      if (j < steps && v < whi) {
        float r[VEC];
        m = vec_mass<E>(st, sd, v, MSt, invZt, MSd, invZd, s, residual, r);
      }
      s_cm[warp][lane] = m;
      const unsigned long long t = warp_sum_u64(m);
      if (lane == 0) s_ct[warp] = t;
    }
    __syncthreads();
    if (warp == 0) {
      const unsigned long long tl0 = theta - off;  // the threshold inside this slice
      unsigned long long tl = s_tl;
      const unsigned long long c = lane < kGroupE ? s_ct[lane] : 0ull;
      const unsigned long long cincl = warp_scan_u64(c, lane);
      unsigned int hit = __ballot_sync(0xffffffffu, lane < kGroupE && cincl > tl);
      const int js = hit ? __ffs(hit) - 1 : kGroupE - 1;
      tl -= min(__shfl_sync(0xffffffffu, cincl - c, js), tl);
      const unsigned long long m = s_cm[js][lane];
      const unsigned long long incl = warp_scan_u64(m, lane);
      hit = __ballot_sync(0xffffffffu, incl > tl);
      const int ls = hit ? __ffs(hit) - 1 : 31;
      if (lane == ls) {
        const int v = min(wlo + (gs * kGroupE + js) * 32 + lane, nv - 1);
        float r[VEC];
        const unsigned long long w = vec_mass<E, true>(st, sd, v, MSt, invZt, MSd, invZd, s, residual, r);
        const unsigned long long rem = tl - min(incl - m, tl);
        unsigned long long c_prev, c_cur;
        const int ks = pick_in_vector<VEC>(r, w, rem, c_prev, c_cur);
        const unsigned long long before = tl0 - rem;  // the slice's mass before this vector
        const long long t = (v0 + v) * VEC + ks;
        const int tok = static_cast<int>(t < a.V ? t : a.V - 1);
        const int nr = near_step(theta, off + before + c_prev, off + before + c_cur, S) ? 1 : 0;
        s_tok[0] = tok;
        s_tok[1] = nr;
      }
    }
    __syncthreads();
  }

  // ---- outputs (warp 0 of the CTA that drew; rank 0 when nothing was drawn)
  // No DSMEM access after the mass exchange: the other CTAs may have left.
  const int writer = S != 0 ? cstar : 0;
  if (rank == writer && warp == 0 && SPEC_IN(b, a.B, a.status) && SPEC_IN(n, K1, a.status)) {
    const int token = s_tok[0], near = s_tok[1];
    const int32_t* x = a.tokens + static_cast<size_t>(b) * K;
    int32_t* out = a.out_tokens + static_cast<size_t>(b) * K1;
    for (int j = lane; j < K1; j += 32)
      out[j] = (j < n) ? min(max(x[j], 0), a.V - 1) : (j == n ? token : -1);
    if (lane == 0) {
      if (a.accepted_len) a.accepted_len[b] = n;
      if (a.flags) a.flags[b] = (ratio_near ? kFlagRatio : 0u) | (near ? kFlagCdf : 0u);
      const int st_bits = bad | (s_fail ? kWaitTimeout : 0);
      if (st_bits && a.status) atomicOr(a.status, st_bits);
    }
  } else if (rank != writer && tid == 0 && s_fail && a.status) {
    atomicOr(a.status, kWaitTimeout);
  }
}

}  // namespace

// Cluster size for early-exit sequences of nvec-vector rows: the smallest C
// in {1, 2, 4, 8} whose two slices and checkpoints fit kBudgetE; 0 if none.
int ee_cluster(long long nvec) {
  for (int C = 1; C <= kMaxCE; C *= 2)
    if (ee_smem(nvec, C) <= kBudgetE) return C;
  return 0;
}

cudaError_t sample_ee_prepare() {
  const int smem = static_cast<int>(kBudgetE);
  cudaError_t e = cudaFuncSetAttribute(ee_cluster_kernel<BF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ee_cluster_kernel<F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
  return e;
}

cudaError_t launch_sample_ee(const VerifyArgs& a, int C, cudaStream_t stream) {
  const long long nvec = static_cast<long long>(a.V) * (a.bf16 ? 2 : 4) / 16;
  const long long smem = ee_smem(nvec, C);
  if (C < 1 || C > kMaxCE || smem > kBudgetE) return cudaErrorInvalidValue;
  const long long grid = static_cast<long long>(a.B) * C;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(grid));
  cfg.blockDim = dim3(kThreadsE);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.bf16 ? cudaLaunchKernelEx(&cfg, ee_cluster_kernel<BF16>, a, nvec)
                : cudaLaunchKernelEx(&cfg, ee_cluster_kernel<F32>, a, nvec);
}

}  // namespace specv
