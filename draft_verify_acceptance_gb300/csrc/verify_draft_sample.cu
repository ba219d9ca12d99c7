// verify_draft_sample.cu -- the drafter's sampling step on sm_103a: one
// token per row of logits, x ~ softmax(row / T), by the inverse CDF of the
// verifier's draws on an exact fixed-point running sum, plus q(x).
//
// Sources (page title, section):
//   "推测性拒绝采样", 技术原理与步骤 step 1: the draft model proposes its K
//     tokens, each sampled from its own distribution q_i;
//   "논문 리뷰 [Speculative Contrastive Decoding]", Speculative Decoding: the
//     verifier needs q_i(x_i) of the sampled tokens.
//
// Design: one cluster of C CTAs per row; each CTA copies its slice of the row
// into shared memory (TMA bulk copies of 16 KiB, one mbarrier each), so the
// row crosses HBM exactly once.  (1) As the copies land, each thread keeps a
// packed running maximum; the cluster exchanges the slices' maxima through
// DSMEM (a one-CTA cluster uses CTA barriers only).  (2) With the row's
// maximum M known, every logit costs one fused multiply-add and one 2^x:
// each warp walks its own contiguous range of the slice, 32 vectors per step
// (lane l takes the step's vector l), four steps at a time unrolled, and
// adds the vector's terms 2^(x*s - M*s) to a float normaliser Z and, as the
// fixed-point mass round(2^40 * sum), to the lane's running integer sum; the
// lane stores that sum after every four steps (a checkpoint).  The slices'
// masses and normalisers are exchanged through DSMEM.  (3) In the CTA holding
// u * S, warp 0 finds the warp range and the checkpoint group by prefix sums
// across lanes, four warps recompute the group's four steps, and warp 0 finds
// the step, the lane and (one element per lane) the element.  The masses are
// unnormalised (the largest term is 1), so nothing waits for Z before the
// sums.  No workspace, no global atomics; every wait is bounded.
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
constexpr long long kSliceBytesR = 96 * 1024;
constexpr int kChunkVecR = 1024;  // vectors per bulk copy (16 KiB), one mbarrier each
constexpr int kMaxChunksR = static_cast<int>(kSliceBytesR / 16 / kChunkVecR);
constexpr int kGroupR = 4;       // 32-vector steps between a lane's checkpoints
static_assert(kGroupR <= kWarpsR, "one warp per step of the crossing group");
// a warp's range holds at most ceil(6144 / 8) = 768 vectors: 24 steps, 6 groups
constexpr int kMaxGroupsR = 8;
static_assert((kSliceBytesR / 16 + kWarpsR - 1) / kWarpsR <= 32 * kGroupR * kMaxGroupsR, "groups");

// round(2^40 * acc), to nearest even, for acc in [0, 2^8).  Below 2^23 the
// integer is read off the float sum 2^40 * acc + 2^23, whose unit in the
// last place is 1; from 2^23 up, 2^40 * acc is already an integer and its
// mantissa is shifted into place (a shift of 64 or more gives 0, as the PTX
// shift defines it, so NaN and infinity give 0).
__device__ __forceinline__ unsigned long long fix40(float acc) {
  const float y = __fmul_rn(acc, 1099511627776.0f);  // exact
  const unsigned int small = __float_as_uint(__fadd_rn(y, 8388608.0f)) - 0x4b000000u;
  const unsigned int b = __float_as_uint(y);
  const unsigned long long m = static_cast<unsigned long long>((b & 0x7fffffu) | 0x800000u);
  const unsigned int sh = (b >> 23) - 150u;
  unsigned long long big;
  asm("shl.b64 %0, %1, %2;" : "=l"(big) : "l"(m), "r"(sh));
  return y < 8388608.0f ? static_cast<unsigned long long>(small) : big;
}

// The terms e_k = 2^(x_k * s - ms) of one vector and their fp32 sum in
// element order (explicitly rounded: every recomputation gives the same bits).
template <typename E>
__device__ __forceinline__ float vec_terms(const uint4 w, float s, float ms,
                                           float (&e)[Staged<E>::kVec]) {
  constexpr int VEC = Staged<E>::kVec;
  float2 x[VEC / 2];
  unpack_pairs<E>(w, x);
  const float2 s2 = make_float2(s, s), m2 = make_float2(-ms, -ms);
#pragma unroll
  for (int k = 0; k < VEC / 2; ++k) {
    const float2 t = ffma2(x[k], s2, m2);
    e[2 * k] = ex2(t.x);
    e[2 * k + 1] = ex2(t.y);
  }
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < VEC; ++k) acc = __fadd_rn(acc, e[k]);
  return acc;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Butterfly sum: every lane ends with the same bits.
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Checkpoint groups of a slice of nv vectors (the same for every warp).
__host__ __device__ __forceinline__ int row_sample_steps(int nv) {
  return ((nv + kWarpsR - 1) / kWarpsR + 31) / 32;
}
__host__ __device__ __forceinline__ int row_sample_groups(int nv) {
  return (row_sample_steps(nv) + kGroupR - 1) / kGroupR;
}

template <typename E>
__global__ void __launch_bounds__(kThreadsR, 3)
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
  const int nch = (nv + kChunkVecR - 1) / kChunkVecR;
  const int steps = row_sample_steps(nv), ngr = row_sample_groups(nv);

  extern __shared__ __align__(128) uint4 slice[];  // [nvs] staged vectors, then cp
  unsigned long long* cp = reinterpret_cast<unsigned long long*>(
      slice + ((nvec + C - 1) >> lgC));              // [warps][groups][32] checkpoints
  __shared__ __align__(8) unsigned long long bars[kMaxChunksR];
  __shared__ float s_wf[kWarpsR];                    // per-warp maxima, then normalisers
  __shared__ unsigned long long s_wm[kWarpsR];       // per-warp masses
  __shared__ float s_pm[kMaxCR], s_pz[kMaxCR];       // pushed by each rank
  __shared__ unsigned long long s_mass[kMaxCR];      // pushed by each rank
  __shared__ int s_sel[2];                           // crossing warp and group
  __shared__ unsigned long long s_tl;                // threshold left inside the group
  __shared__ unsigned long long s_cm[kGroupR][32];   // lane masses of the crossing group
  __shared__ unsigned long long s_ct[kGroupR];       // its steps' masses

  // ---- stage the slice ------------------------------------------------
  const uint4* src = static_cast<const uint4*>(logits) + static_cast<size_t>(row) * nvec + v0;
  if (tid == 0) {
    for (int c = 0; c < nch; ++c) mbar_init(&bars[c], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int c = 0; c < nch; ++c) {
      const int len = min(kChunkVecR, nv - c * kChunkVecR);
      mbar_arrive_expect_tx(&bars[c], static_cast<uint32_t>(len) * 16u);
      bulk_load(slice + c * kChunkVecR, src + c * kChunkVecR, static_cast<uint32_t>(len) * 16u,
                &bars[c]);
    }
  }
  // a cluster of one CTA exchanges nothing: CTA barriers stand in for the
  // cluster's (C is the same for the whole grid)
  const bool solo = C == 1;
  if (!solo) cluster_arrive_relaxed();  // matched before the first DSMEM push
  const float u = uniforms[row];

  // ---- pass 1: the row's maximum, as the copies land -------------------
  bool ok = true;
  typename Staged<E>::Max pm = Staged<E>::max_init();
  for (int c = 0; c < nch; ++c) {
    if (!mbar_wait_sleep(&bars[c], 0u)) {
      ok = false;
      break;
    }
    const int cend = min((c + 1) * kChunkVecR, nv);
    if (cend - c * kChunkVecR == kChunkVecR) {  // a full chunk: four vectors a thread
      static_assert(kChunkVecR == 4 * kThreadsR, "four vectors a thread");
      uint4 w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) w[k] = slice[c * kChunkVecR + k * kThreadsR + tid];
#pragma unroll
      for (int k = 0; k < 4; ++k) Staged<E>::max_update(pm, w[k]);
    } else {
      for (int v = c * kChunkVecR + tid; v < cend; v += kThreadsR) Staged<E>::max_update(pm, slice[v]);
    }
  }
  const float wmax = warp_max(Staged<E>::max_value(pm));  // NaN-ignoring
  if (lane == 0) s_wf[warp] = wmax;
  const int failed = __syncthreads_or(!ok);
  if (!solo) cluster_wait();  // every CTA of the cluster has started
  if (warp == 0) {
    const float m = warp_max(lane < kWarpsR ? s_wf[lane] : -INFINITY);
    if (solo) {
      if (lane == 0) s_pm[0] = m;
    } else if (lane < C) {
      *cluster.map_shared_rank(&s_pm[rank], lane) = m;
    }
  }
  if (solo) __syncthreads();
  else cluster.sync();
  float M = -INFINITY;
  for (int r = 0; r < C; ++r) M = fmaxf(M, s_pm[r]);
  const float MS = M * s;  // p_k = 2^(x_k * s - MS) / Z

  // ---- pass 2: normaliser, masses, lane checkpoints -----------------------
  const int lo = (nv * warp) / kWarpsR, hi = (nv * (warp + 1)) / kWarpsR;
  unsigned long long run = 0;
  float zs = 0.f;
  unsigned long long* mycp = cp + static_cast<size_t>(warp) * ngr * 32 + lane;
  // groups whose kGroupR steps are all full run unrolled and unpredicated;
  // the rest (at most the warp's last group) checks each vector
  const int nfull = (hi - lo) / (32 * kGroupR);
  for (int g = 0; g < ngr; ++g) {
    const uint4* src_g = slice + lo + g * kGroupR * 32 + lane;
    if (g < nfull) {
      uint4 w[kGroupR];
#pragma unroll
      for (int jj = 0; jj < kGroupR; ++jj) w[jj] = src_g[jj * 32];
#pragma unroll
      for (int jj = 0; jj < kGroupR; ++jj) {
        float e[VEC];
        const float acc = vec_terms<E>(w[jj], s, MS, e);
        zs = __fadd_rn(zs, acc);
        run += fix40(acc);
      }
    } else {
      for (int jj = 0; jj < kGroupR; ++jj) {
        if (lo + (g * kGroupR + jj) * 32 + lane < hi) {
          float e[VEC];
          const float acc = vec_terms<E>(src_g[jj * 32], s, MS, e);
          zs = __fadd_rn(zs, acc);
          run += fix40(acc);
        }
      }
    }
    mycp[g * 32] = run;
  }
  const unsigned long long wm = warp_sum_u64(run);
  const float wz = warp_sum_f(zs);
  if (lane == 0) {
    s_wm[warp] = wm;
    s_wf[warp] = wz;
  }
  __syncthreads();
  if (warp == 0) {
    const unsigned long long t = warp_sum_u64(lane < kWarpsR ? s_wm[lane] : 0ull);
    const float z = warp_sum_f(lane < kWarpsR ? s_wf[lane] : 0.f);
    if (solo) {
      if (lane == 0) {
        s_mass[0] = t;
        s_pz[0] = z;
      }
    } else if (lane < C) {
      *cluster.map_shared_rank(&s_mass[rank], lane) = t;
      *cluster.map_shared_rank(&s_pz[rank], lane) = z;
    }
  }
  if (solo) __syncthreads();
  else cluster.sync();  // no DSMEM access after this point: CTAs may leave
  unsigned long long S = 0;
  float Z = 0.f;
  for (int r = 0; r < C; ++r) {  // rank order: the same bits on every CTA
    S += s_mass[r];
    Z += s_pz[r];
  }
  const bool row_ok = isfinite(M) && isfinite(Z) && Z > 0.f && S != 0;

  // ---- pass 3: the crossing, in the CTA that holds it ---------------------
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
  if (rank != cstar) {
    if (tid == 0 && failed && status) atomicOr(status, kWaitTimeout);
    return;
  }
  int token = 0;
  float qx = 0.f;
  if (row_ok && nv > 0) {
    // warp 0: the warp whose range holds the crossing (lane w holds the
    // prefix through warp w), then the checkpoint group inside it (lane g
    // holds the prefix through group g)
    if (warp == 0) {
      unsigned long long tl = theta - off;
      const unsigned long long m = lane < kWarpsR ? s_wm[lane] : 0ull;
      const unsigned long long incl = warp_scan_u64(m, lane);
      unsigned int hit = __ballot_sync(0xffffffffu, lane < kWarpsR && incl > tl);
      const int ws = hit ? __ffs(hit) - 1 : kWarpsR - 1;
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
    const int wlo = (nv * ws) / kWarpsR, whi = (nv * (ws + 1)) / kWarpsR;
    if (warp < kGroupR) {  // warp j recomputes step gs * kGroupR + j of warp ws's range
      const int j = gs * kGroupR + warp;
      const int v = wlo + j * 32 + lane;
      unsigned long long m = 0;
      if (j < steps && v < whi) {
        float e[VEC];
        m = fix40(vec_terms<E>(slice[v], s, MS, e));
      }
      s_cm[warp][lane] = m;
      const unsigned long long t = warp_sum_u64(m);
      if (lane == 0) s_ct[warp] = t;
    }
    __syncthreads();
    if (warp == 0) {
      unsigned long long tl = s_tl;
      const unsigned long long c = lane < kGroupR ? s_ct[lane] : 0ull;
      const unsigned long long cincl = warp_scan_u64(c, lane);
      unsigned int hit = __ballot_sync(0xffffffffu, lane < kGroupR && cincl > tl);
      const int js = hit ? __ffs(hit) - 1 : kGroupR - 1;
      tl -= min(__shfl_sync(0xffffffffu, cincl - c, js), tl);
      const unsigned long long m = s_cm[js][lane];
      const unsigned long long incl = warp_scan_u64(m, lane);
      hit = __ballot_sync(0xffffffffu, incl > tl);
      const int ls = hit ? __ffs(hit) - 1 : 31;
      const unsigned long long rem = tl - min(__shfl_sync(0xffffffffu, incl - m, ls), tl);
      // the element: every lane recomputes the crossing vector's terms; lane
      // k < VEC tests the running sum through element k (element order,
      // rounded as the masses are: its last value is the vector's mass, > rem)
      const int v = min(wlo + (gs * kGroupR + js) * 32 + ls, nv - 1);
      float e[VEC];
      vec_terms<E>(slice[v], s, MS, e);
      float acc = 0.f, ek = 0.f;
#pragma unroll
      for (int k = 0; k < VEC; ++k) {
        if (k <= lane) acc = __fadd_rn(acc, e[k]);
        if (k == lane) ek = e[k];
      }
      hit = __ballot_sync(0xffffffffu, lane < VEC && fix40(acc) > rem);
      const int ks = hit ? __ffs(hit) - 1 : VEC - 1;
      const long long t = (v0 + v) * VEC + ks;
      token = static_cast<int>(t < V ? t : V - 1);
      qx = __shfl_sync(0xffffffffu, ek, ks) * (1.f / Z);
    }
  }
  if (tid == 0) {
    tokens[row] = token;
    if (q_at) q_at[row] = qx;
    int st = row_ok ? 0 : kDataNonfiniteLogit;
    if (!(u >= 0.f && u < 1.f)) st |= kDataUniformRange;
    if (failed) st |= kWaitTimeout;
    if (st && status) atomicOr(status, st);
  }
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
  const int smem = static_cast<int>(kSliceBytesR) + 16 * 1024;
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
  const size_t smem = static_cast<size_t>(nvs * 16) +
                      static_cast<size_t>(row_sample_groups(static_cast<int>(nvs))) * kWarpsR * 32 * 8;
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
