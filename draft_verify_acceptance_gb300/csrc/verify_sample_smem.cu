// verify_sample_smem.cu -- speculative-sampling verification on sm_103a with
// each row slice staged in shared memory by one TMA bulk copy.
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
// Design: one thread-block cluster of C CTAs (C in {1,2,4,8}, chosen so a
// CTA's slice of both rows fits in ~72 KiB, three CTAs per SM) per
// (position i, sequence b) row pair, positions launched in order.  Each CTA
// stages its 1/C slice of target row i and draft row i with cp.async.bulk
// into shared memory and never reads them from global memory again:
//   pass 1  per-thread max, then sum 2^((x - max) * log2e/T), merged across
//           the block and, through DSMEM, across the cluster in rank order
//           (identical normalisers in every CTA).  The CTA whose slice holds
//           x_i pushes t[x_i], d[x_i] to rank 0 at the same time.
//   accept  rank 0 tests u_i * q(x_i) < p(x_i) and records a rejection with
//           one atomicOr, whose returned mask says whether an earlier
//           position of the sequence has already rejected; only a row that
//           may still be the first rejection (or a bonus row with no known
//           rejection) goes on.
//   pass 2  the residual max(0, p - q) (or p) of every staged vector as a
//           2^-56 fixed-point mass; tile/warp masses in shared memory, CTA
//           masses exchanged through DSMEM.  Integer sums agree exactly in
//           every order.
//   pass 3  warp 0 of the CTA holding the crossing of u_K * S walks tile ->
//           warp -> lane -> element over the staged data.
// The warp that completes a sequence's last row finalises it.
#include <cooperative_groups.h>

#include <cfloat>
#include <climits>

#include "device_common.cuh"
#include "launch.h"
#include "sample_common.cuh"

namespace cg = cooperative_groups;

namespace specv {

namespace {

constexpr int kMaxC = 8;                  // largest cluster (portable size)
constexpr int kProducer = kThreads - 32;  // issues the bulk copies
constexpr int kSmemTarget = 72 * 1024;    // slice bytes for three CTAs per SM

// Per-thread normaliser of a slice relative to the scaled offset
// ms = round(max(x) * s): z = sum 2^fma(x, s, -ms).
template <typename E>
__device__ __forceinline__ void slice_normaliser(const uint4* slice, int nv, float s, float& ms,
                                                 float& z) {
  constexpr int VEC = Staged<E>::kVec;
  typename Staged<E>::Max pm = Staged<E>::max_init();
  for (int v = threadIdx.x; v < nv; v += kThreads) Staged<E>::max_update(pm, slice[v]);
  const float m = Staged<E>::max_value(pm);
  z = 0.f;
  if (m == -INFINITY) {  // nothing finite here (or nothing at all)
    ms = -INFINITY;
    return;
  }
  ms = m * s;
  float z0 = 0.f, z1 = 0.f;
  for (int v = threadIdx.x; v < nv; v += kThreads) {
    float x[VEC];
    Staged<E>::unpack(slice[v], x);
#pragma unroll
    for (int k = 0; k < VEC; k += 2) {
      z0 += ex2(fmaf(x[k], s, -ms));
      z1 += ex2(fmaf(x[k + 1], s, -ms));
    }
  }
  z = z0 + z1;
}

template <typename E>
__global__ void __launch_bounds__(kThreads)
sample_smem_kernel(VerifyArgs a, long long nvec, int nvs) {
  constexpr int VEC = Staged<E>::kVec;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const long long pair = blockIdx.x / C;  // position-major: earlier positions launch first
  const int K = a.K, K1 = K + 1;
  const int i = static_cast<int>(pair / a.B);
  const int b = static_cast<int>(pair - static_cast<long long>(i) * a.B);
  const bool has_draft = i < K;
  const uint4* trow = static_cast<const uint4*>(a.target) + (static_cast<size_t>(b) * K1 + i) * nvec;
  const uint4* drow = has_draft
      ? static_cast<const uint4*>(a.draft) + (static_cast<size_t>(b) * K + i) * nvec
      : trow;
  const long long v0 = nvec * rank / C;
  const int nv = static_cast<int>(nvec * (rank + 1) / C - v0);
  const int ntl = (nv + kThreads - 1) / kThreads;  // tiles of kThreads vectors in this slice
  const float s = a.scale;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ __align__(128) uint4 smem[];
  uint4* st = smem;                                                     // target slice
  uint4* sd = smem + nvs;                                               // draft slice
  unsigned long long* tws = reinterpret_cast<unsigned long long*>(smem + 2 * static_cast<size_t>(nvs));
  __shared__ __align__(8) unsigned long long bar;
  __shared__ float s_part[kMaxC][4];                   // pushed by each rank
  __shared__ float s_gx[2];                            // t[x_i], d[x_i], pushed to rank 0
  __shared__ float s_red[kWarps][4];
  __shared__ int s_need;                               // pushed by rank 0
  __shared__ unsigned long long s_mass[2][kMaxC];      // pushed by each rank
  __shared__ float s_uK;

  cluster_arrive_relaxed();  // matched by cluster_wait() before the first DSMEM push
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == kProducer) {
    const uint32_t bytes = static_cast<uint32_t>(nv) * 16u;
    mbar_arrive_expect_tx(&bar, has_draft ? 2u * bytes : bytes);
    bulk_load(st, trow + v0, bytes, &bar);
    if (has_draft) bulk_load(sd, drow + v0, bytes, &bar);
  }
  // while the slice lands: this row's token and uniforms
  int xr = 0;
  float ui = 0.f, uK = 0.f;
  if (tid == 0) {
    if (has_draft) {
      xr = a.tokens[static_cast<size_t>(b) * K + i];
      ui = a.uniforms[static_cast<size_t>(b) * K1 + i];
    }
    uK = a.uniforms[static_cast<size_t>(b) * K1 + K];
    s_uK = uK;  // every thread needs it for the draw (read after the next barrier)
  }
  const int x = min(max(xr, 0), a.V - 1);
  // thread 0 sleeps on the barrier; the others park at __syncthreads
  int ok = 1;
  if (tid == 0) {
    ok = mbar_wait_one(&bar, 0) ? 1 : 0;
    if (!ok) ok = mbar_wait_one(&bar, 0) ? 1 : 0;  // a second bounded wait before giving up
    if (!ok && a.status) atomicOr(a.status, kWaitTimeout);
  }
  __syncthreads();

  // ---- pass 1: normalisers of both rows over the staged slice -----------
  float mt, zt, md = -INFINITY, zd = 0.f;
  slice_normaliser<E>(st, nv, s, mt, zt);
  if (has_draft) slice_normaliser<E>(sd, nv, s, md, zd);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    merge_scaled(mt, zt, __shfl_xor_sync(0xffffffffu, mt, o), __shfl_xor_sync(0xffffffffu, zt, o));
    merge_scaled(md, zd, __shfl_xor_sync(0xffffffffu, md, o), __shfl_xor_sync(0xffffffffu, zd, o));
  }
  if (lane == 0) {
    s_red[warp][0] = mt; s_red[warp][1] = zt; s_red[warp][2] = md; s_red[warp][3] = zd;
  }
  __syncthreads();
  cluster_wait();  // every CTA of the cluster has started
  if (tid < C) {
    float m0 = s_red[0][0], z0 = s_red[0][1], m1 = s_red[0][2], z1 = s_red[0][3];
    for (int w = 1; w < kWarps; ++w) {
      merge_scaled(m0, z0, s_red[w][0], s_red[w][1]);
      merge_scaled(m1, z1, s_red[w][2], s_red[w][3]);
    }
    float* dst = cluster.map_shared_rank(&s_part[rank][0], tid);
    dst[0] = m0; dst[1] = z0; dst[2] = m1; dst[3] = z1;
  }
  // the CTA whose slice holds x_i hands t[x_i], d[x_i] to rank 0
  if (tid == 0 && has_draft && x >= v0 * VEC && x < (v0 + nv) * VEC) {
    const int j = static_cast<int>(x - v0 * VEC);
    float* dst = cluster.map_shared_rank(&s_gx[0], 0);
    dst[0] = staged_elem<E>(st, j);
    dst[1] = staged_elem<E>(sd, j);
  }
  cluster.sync();
  // Mt, Md: scaled offsets (round(max * s)); Zt, Zd relative to them
  float Mt = s_part[0][0], Zt = s_part[0][1], Md = s_part[0][2], Zd = s_part[0][3];
  for (int r = 1; r < C; ++r) {
    merge_scaled(Mt, Zt, s_part[r][0], s_part[r][1]);
    merge_scaled(Md, Zd, s_part[r][2], s_part[r][3]);
  }

  // ---- accept test; does this row still need a draw? ---------------------
  if (rank == 0 && tid == 0) {
    SeqState* sq = a.seq + b;
    int bad = 0;
    if (!(isfinite(Mt) && isfinite(Zt) && Zt > 0.f)) bad |= kDataNonfiniteLogit;
    bool need;
    if (has_draft) {
      const float px = ex2(fmaf(s_gx[0], s, -Mt)) / Zt;
      const float qx = ex2(fmaf(s_gx[1], s, -Md)) / Zd;
      const bool accept = ui * qx < px;
      if (a.p_at) a.p_at[static_cast<size_t>(b) * K + i] = px;
      if (a.q_at) a.q_at[static_cast<size_t>(b) * K + i] = qx;
      if (xr != x) bad |= kDataTokenRange;
      if (!(ui >= 0.f && ui < 1.f)) bad |= kDataUniformRange;
      if (!(isfinite(Md) && isfinite(Zd) && Zd > 0.f)) bad |= kDataNonfiniteLogit;
      if (qx > 0.f && fabsf(ui - fminf(1.f, px / qx)) < kBandF) atomicOr(&sq->near_mask, 1ull << i);
      if (accept) {
        need = false;
      } else {
        // the mask before this rejection says whether an earlier one exists
        const unsigned long long before = atomicOr(&sq->reject_mask, 1ull << i);
        need = (before & ((1ull << i) - 1ull)) == 0ull;
      }
    } else {
      if (!(uK >= 0.f && uK < 1.f)) bad |= kDataUniformRange;
      need = atomicOr(&sq->reject_mask, 0ull) == 0ull;  // bonus row: no rejection known
    }
    if (bad && a.status) atomicOr(a.status, bad);
    for (int r = 0; r < C; ++r) *cluster.map_shared_rank(&s_need, r) = need ? 1 : 0;
  }
  cluster.sync();
  if (!s_need) {
    if (rank == 0 && warp == 0) warp_arrive_and_finalize(a, b);
    return;
  }

  // ---- pass 2: fixed-point mass of the staged slice, per tile and warp ---
  const float invZt = 1.f / Zt;
  const float invZd = has_draft ? 1.f / Zd : 0.f;
  bool residual = has_draft;
  int rnd = 0;
  unsigned long long S = 0;
  for (;; ++rnd) {
    for (int k = 0; k < ntl; ++k) {
      const int v = k * kThreads + tid;
      float xt[VEC], xd[VEC], r[VEC];
      if (v < nv) {
        Staged<E>::unpack(st[v], xt);
        if (residual) Staged<E>::unpack(sd[v], xd);
      } else {
#pragma unroll
        for (int q = 0; q < VEC; ++q) xt[q] = xd[q] = -INFINITY;
      }
      const unsigned long long w =
          warp_sum_u64(vec_weight_scaled<VEC>(xt, xd, Mt, invZt, Md, invZd, s, residual, r));
      if (lane == 0) tws[k * kWarps + warp] = w;
    }
    __syncthreads();
    if (warp == 0) {
      unsigned long long t = 0;
      for (int k = lane; k < ntl * kWarps; k += 32) t += tws[k];
      t = warp_sum_u64(t);
      if (lane < C) *cluster.map_shared_rank(&s_mass[rnd][rank], lane) = t;
    }
    cluster.sync();
    S = 0;
    for (int r = 0; r < C; ++r) S += s_mass[rnd][r];
    if (S != 0 || !residual || rnd == 1) break;
    residual = false;  // p == q at this row: the draw falls back to p
  }

  if (S == 0) {  // no mass at all: only with non-finite data (already flagged)
    if (rank == 0 && warp == 0) {
      if (lane == 0) *candidate_slot(a, b, i) = 0;
      warp_arrive_and_finalize(a, b);
    }
    return;
  }
  const float uKs = s_uK;
  double th = static_cast<double>(uKs) * static_cast<double>(S);
  if (!(th >= 0.0)) th = 0.0;
  const unsigned long long theta =
      (th >= static_cast<double>(S)) ? S - 1 : static_cast<unsigned long long>(th);
  int cstar = C - 1;
  unsigned long long off = 0;
  for (int r = 0; r < C; ++r) {
    const unsigned long long m = s_mass[rnd][r];
    if (off + m > theta) { cstar = r; break; }
    off += m;
  }
  if (rank != cstar || warp != 0) return;

  // ---- pass 3: the crossing inside this slice (warp 0 of that CTA) ------
  int token = 0;
  bool near = false;
  if (ntl > 0) {
    const unsigned long long tl = theta - off;
    unsigned long long base = 0;
    int kstar = ntl - 1;
    for (int k0 = 0; k0 < ntl; k0 += 32) {
      const int k = k0 + lane;
      unsigned long long tt = 0;
      if (k < ntl)
        for (int w = 0; w < kWarps; ++w) tt += tws[k * kWarps + w];
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
    int wstar = kWarps - 1;
    for (int w = 0; w < kWarps; ++w) {
      const unsigned long long m = tws[kstar * kWarps + w];
      if (base + m > tl) { wstar = w; break; }
      base += m;
    }
    const int v = kstar * kThreads + wstar * 32 + lane;
    float xt[VEC], xd[VEC], r[VEC];
    if (v < nv) {
      Staged<E>::unpack(st[v], xt);
      if (residual) Staged<E>::unpack(sd[v], xd);
    } else {
#pragma unroll
      for (int q = 0; q < VEC; ++q) xt[q] = xd[q] = -INFINITY;
    }
    const unsigned long long w = vec_weight_scaled<VEC>(xt, xd, Mt, invZt, Md, invZd, s, residual, r);
    unsigned long long incl = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    const unsigned int hit = __ballot_sync(0xffffffffu, base + incl > tl);
    const int lstar = hit ? (__ffs(hit) - 1) : 31;
    if (lane == lstar) {
      const unsigned long long before = base + incl - w;  // slice prefix before this vector
      const unsigned long long rem = tl - before;
      float acc = 0.f;
      int mstar = VEC - 1;
      unsigned long long c_prev = 0, c_cur = w;
#pragma unroll
      for (int k = 0; k < VEC; ++k) {
        acc = __fadd_rn(acc, r[k]);
        const unsigned long long c = __float2ull_rn(__fmul_rn(acc, kFix));
        if (c > rem) { mstar = k; c_cur = c; break; }
        c_prev = c;
      }
      const long long t = (v0 + v) * VEC + mstar;
      token = static_cast<int>(t < a.V ? t : a.V - 1);
      const double band = 1e-6 * static_cast<double>(S);
      near = fabs(th - static_cast<double>(off + before + c_prev)) < band ||
             fabs(static_cast<double>(off + before + c_cur) - th) < band;
    }
    token = __shfl_sync(0xffffffffu, token, lstar);
    near = __shfl_sync(0xffffffffu, near ? 1 : 0, lstar) != 0;
  }
  if (lane == 0)
    *candidate_slot(a, b, i) = near ? static_cast<int32_t>(static_cast<uint32_t>(token) | 0x80000000u)
                                    : token;
  warp_arrive_and_finalize(a, b);
}

// Dynamic shared memory of one CTA: both slices and the tile/warp masses.
size_t smem_bytes(long long nvec, int C) {
  const long long nvs = (nvec + C - 1) / C;
  const long long ntiles = (nvs + kThreads - 1) / kThreads;
  return static_cast<size_t>(2 * nvs * 16 + ntiles * kWarps * 8);
}

}  // namespace

// Cluster size for the staged kernel: the smallest C in {1, 2, 4, 8} whose
// slices fit three CTAs per SM, else 0 (the rows are too long to stage; the
// streaming kernel takes them).
int sample_smem_cluster(long long nvec) {
  for (int C = 1; C <= kMaxC; C *= 2)
    if (smem_bytes(nvec, C) <= static_cast<size_t>(kSmemTarget)) return C;
  return 0;
}

cudaError_t sample_smem_prepare() {
  cudaError_t e = cudaFuncSetAttribute(sample_smem_kernel<BF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTarget);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(sample_smem_kernel<F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemTarget);
  return e;
}

cudaError_t launch_sample_smem(const VerifyArgs& a, int C, cudaStream_t stream) {
  const long long nvec = static_cast<long long>(a.V) * (a.bf16 ? 2 : 4) / 16;
  const long long pairs = static_cast<long long>(a.B) * (a.K + 1);
  const long long grid = pairs * C;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  const int nvs = static_cast<int>((nvec + C - 1) / C);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes(nvec, C);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.bf16 ? cudaLaunchKernelEx(&cfg, sample_smem_kernel<BF16>, a, nvec, nvs)
                : cudaLaunchKernelEx(&cfg, sample_smem_kernel<F32>, a, nvec, nvs);
}

}  // namespace specv
