// verify_draft_sample.cu -- the drafter's sampling step on sm_103a: one
// token per row of logits, x ~ softmax(row / T), by the same inverse CDF and
// fixed-point scheme as the verifier's draws, plus q(x).
//
// Sources (page title, section):
//   "推测性拒绝采样", 技术原理与步骤 step 1: the draft model proposes its K
//     tokens, each sampled from its own distribution q_i;
//   "논문 리뷰 [Speculative Contrastive Decoding]", Speculative Decoding: the
//     verifier needs q_i(x_i) of the sampled tokens.
//
// Design: one cluster of C CTAs per row; each CTA copies its slice of the row
// into shared memory once (TMA bulk copies), so the row crosses HBM exactly
// once.  From shared memory: (1) the slice's online normaliser, merged over
// the cluster through DSMEM in rank order (every CTA then holds the row's
// (M, Z)); (2) the fixed-point mass round(2^56 * sum) of p over every
// 16-byte vector, summed per (tile, warp) and per slice, the slice masses
// exchanged through DSMEM; (3) in the CTA holding u * S, one warp finds the
// crossing vector and element.  No workspace, no global atomics; every wait
// is bounded.
#include <cooperative_groups.h>

#include <cfloat>
#include <climits>

#include "device_common.cuh"
#include "launch.h"
#include "sample_common.cuh"

namespace cg = cooperative_groups;

namespace specv {
namespace {

constexpr int kThreadsR = 256;
constexpr int kWarpsR = kThreadsR / 32;
constexpr int kMaxCR = 8;
constexpr long long kSliceBytesR = 96 * 1024;  // two CTAs per SM
constexpr int kCopyVec = 2048;                 // vectors per bulk copy (32 KiB)

struct __align__(8) MsZ {
  float ms, z;
};

template <typename E>
__global__ void __launch_bounds__(kThreadsR, 2)
row_sample_kernel(const void* logits, const float* uniforms, int R, int V, long long nvec,
                  float s, int32_t* tokens, float* q_at, int32_t* status) {
  constexpr int VEC = Staged<E>::kVec;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int lgC = __ffs(C) - 1;  // C is a power of two
  const int row = static_cast<int>(blockIdx.x >> lgC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long v0 = (nvec * rank) >> lgC;
  const int nv = static_cast<int>(((nvec * (rank + 1)) >> lgC) - v0);
  const int ntl = (nv + kThreadsR - 1) / kThreadsR;

  extern __shared__ __align__(128) uint4 slice[];  // [nvs] staged vectors, then tws
  unsigned long long* tws = reinterpret_cast<unsigned long long*>(
      slice + ((nvec + C - 1) >> lgC));              // [tiles][warps] masses
  __shared__ __align__(8) unsigned long long bar;
  __shared__ MsZ s_warp[kWarpsR];
  __shared__ MsZ s_part[kMaxCR];                     // pushed by each rank
  __shared__ unsigned long long s_mass[kMaxCR];      // pushed by each rank
  __shared__ int s_bad;

  // ---- stage the slice ------------------------------------------------
  const uint4* src = static_cast<const uint4*>(logits) + static_cast<size_t>(row) * nvec + v0;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    s_bad = 0;
  }
  __syncthreads();
  if (tid == 0 && nv > 0) {
    mbar_arrive_expect_tx(&bar, static_cast<uint32_t>(nv) * 16u);
    for (int c0 = 0; c0 < nv; c0 += kCopyVec) {
      const int len = min(kCopyVec, nv - c0);
      bulk_load(slice + c0, src + c0, static_cast<uint32_t>(len) * 16u, &bar);
    }
  }
  cluster_arrive_relaxed();  // matched before the first DSMEM push
  const float u = uniforms[row];
  bool ok = true;
  if (nv > 0 && !mbar_wait_sleep(&bar, 0u)) ok = false;

  // ---- pass 1: the row's normaliser ------------------------------------
  RowAcc A{-INFINITY, 0.f};
  bool bad = false;
  for (int v = tid; v < nv; v += 2 * kThreadsR) {
    uint4 w[2];
    w[0] = slice[v];
    const int n2 = v + kThreadsR < nv ? 2 : 1;
    if (n2 > 1) w[1] = slice[v + kThreadsR];
    float x[VEC];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (j < n2) {
        Staged<E>::unpack(w[j], x);
#pragma unroll
        for (int k = 0; k < VEC; ++k) bad |= !(x[k] <= FLT_MAX) && !(x[k] == -INFINITY);
      }
    }
    acc_vectors<E>(A, w, n2, s);
  }
  float ms = A.ms, z = A.z;
  warp_merge_scaled(ms, z);
  if (lane == 0) s_warp[warp] = MsZ{ms, z};
  if (__syncthreads_or(bad) && tid == 0) s_bad = 1;
  cluster_wait();  // every CTA of the cluster has started
  if (warp == 0) {
    MsZ m = lane < kWarpsR ? s_warp[lane] : MsZ{-INFINITY, 0.f};
    warp_merge_scaled(m.ms, m.z);
    if (lane < C) *cluster.map_shared_rank(&s_part[rank], lane) = m;
  }
  cluster.sync();
  float M = -INFINITY, Z = 0.f;
  for (int r = 0; r < C; ++r) merge_scaled(M, Z, s_part[r].ms, s_part[r].z);  // rank order
  const bool row_ok = isfinite(M) && isfinite(Z) && Z > 0.f;
  const float invZ = row_ok ? 1.f / Z : 0.f;

  // ---- pass 2: fixed-point masses per (tile, warp) and per slice ---------
  for (int k = 0; k < ntl; ++k) {
    const int v = k * kThreadsR + tid;
    float xt[VEC], xd[VEC], r[VEC];
    if (v < nv) {
      Staged<E>::unpack(slice[v], xt);
    } else {
#pragma unroll
      for (int q = 0; q < VEC; ++q) xt[q] = -INFINITY;
    }
#pragma unroll
    for (int q = 0; q < VEC; ++q) xd[q] = -INFINITY;
    const unsigned long long w =
        warp_sum_mass(vec_weight_scaled<VEC>(xt, xd, M, invZ, 0.f, 0.f, s, false, r));
    if (lane == 0) tws[k * kWarpsR + warp] = w;
  }
  __syncthreads();
  if (warp == 0) {
    unsigned long long t = 0;
    for (int k = lane; k < ntl * kWarpsR; k += 32) t += tws[k];
    t = warp_sum_u64(t);
    if (lane < C) *cluster.map_shared_rank(&s_mass[rank], lane) = t;
  }
  cluster.sync();
  unsigned long long S = 0;
  for (int r = 0; r < C; ++r) S += s_mass[r];

  // ---- pass 3: the crossing, in the CTA that holds it (warp 0) -----------
  const unsigned long long theta = draw_threshold(u, S);
  int cstar = C - 1;
  unsigned long long off = 0;
  for (int r = 0; r < C; ++r) {
    if (off + s_mass[r] > theta) {
      cstar = r;
      break;
    }
    off += s_mass[r];
  }
  if (rank == cstar && warp == 0) {
    int token = 0;
    float qx = 0.f;
    if (S != 0 && ntl > 0) {
      const unsigned long long tl = theta - off;
      unsigned long long base = 0;
      int kstar = ntl - 1;
      for (int k0 = 0; k0 < ntl; k0 += 32) {
        const int k = k0 + lane;
        unsigned long long tt = 0;
        if (k < ntl)
          for (int w = 0; w < kWarpsR; ++w) tt += tws[k * kWarpsR + w];
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
      int wstar = kWarpsR - 1;
      {
        const unsigned long long m = lane < kWarpsR ? tws[kstar * kWarpsR + lane] : 0ull;
        const unsigned long long incl = warp_scan_u64(m, lane);
        const unsigned int hit = __ballot_sync(0xffffffffu, lane < kWarpsR && base + incl > tl);
        if (hit) wstar = __ffs(hit) - 1;
        base += __shfl_sync(0xffffffffu, incl - m, wstar);
      }
      const int v = kstar * kThreadsR + wstar * 32 + lane;
      float xt[VEC], xd[VEC], r[VEC];
      if (v < nv) {
        Staged<E>::unpack(slice[v], xt);
      } else {
#pragma unroll
        for (int q = 0; q < VEC; ++q) xt[q] = -INFINITY;
      }
#pragma unroll
      for (int q = 0; q < VEC; ++q) xd[q] = -INFINITY;
      const unsigned long long w =
          vec_weight_scaled<VEC, true>(xt, xd, M, invZ, 0.f, 0.f, s, false, r);
      const unsigned long long incl = warp_scan_u64(w, lane);
      const unsigned int hit = __ballot_sync(0xffffffffu, base + incl > tl);
      const int lstar = hit ? __ffs(hit) - 1 : 31;
      int tok = 0;
      float q = 0.f;
      if (lane == lstar) {
        const unsigned long long before = base + incl - w;
        unsigned long long c_prev, c_cur;
        const int mstar = pick_in_vector<VEC>(r, w, tl - before, c_prev, c_cur);
        const long long t = (v0 + v) * VEC + mstar;
        tok = static_cast<int>(t < V ? t : V - 1);
        q = ex2(fmaf(xt[mstar], s, -M)) * invZ;
      }
      token = __shfl_sync(0xffffffffu, tok, lstar);
      qx = __shfl_sync(0xffffffffu, q, lstar);
    }
    if (lane == 0) {
      tokens[row] = token;
      if (q_at) q_at[row] = qx;
      int st = (s_bad || !row_ok || S == 0) ? kDataNonfiniteLogit : 0;
      if (!(u >= 0.f && u < 1.f)) st |= kDataUniformRange;
      if (!ok) st |= kWaitTimeout;
      if (st && status) atomicOr(status, st);
    }
  }
  // flag a bad row from every CTA of the cluster that saw it
  if (rank != cstar && tid == 0 && (s_bad || !ok) && status)
    atomicOr(status, (s_bad ? kDataNonfiniteLogit : 0) | (ok ? 0 : kWaitTimeout));
}

}  // namespace

// Cluster size for rows of nvec vectors: the smallest C in {1, 2, 4, 8}
// whose slices fit kSliceBytesR; 0 when none does (the caller falls back).
int row_sample_cluster(long long nvec) {
  for (int C = 1; C <= kMaxCR; C *= 2)
    if (((nvec + C - 1) / C) * 16 <= kSliceBytesR) return C;
  return 0;
}

cudaError_t row_sample_prepare() {
  const int smem = static_cast<int>(kSliceBytesR) + 8 * 1024;
  cudaError_t e = cudaFuncSetAttribute(row_sample_kernel<BF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(row_sample_kernel<F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
  return e;
}

cudaError_t launch_row_sample(const void* logits, const float* uniforms, int R, int V, bool bf16,
                              float scale, int32_t* tokens, float* q_at, int32_t* status, int C,
                              cudaStream_t stream) {
  const long long nvec = static_cast<long long>(V) * (bf16 ? 2 : 4) / 16;
  const long long nvs = (nvec + C - 1) / C;
  const long long ntiles = (nvs + kThreadsR - 1) / kThreadsR;
  const size_t smem = static_cast<size_t>(nvs * 16 + ntiles * kWarpsR * 8);
  const long long grid = static_cast<long long>(R) * C;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(grid));
  cfg.blockDim = dim3(kThreadsR);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return bf16 ? cudaLaunchKernelEx(&cfg, row_sample_kernel<BF16>, logits, uniforms, R, V, nvec,
                                   scale, tokens, q_at, status)
              : cudaLaunchKernelEx(&cfg, row_sample_kernel<F32>, logits, uniforms, R, V, nvec,
                                   scale, tokens, q_at, status);
}

}  // namespace specv
