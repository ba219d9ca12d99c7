// verify_sample_seq.cu -- speculative-sampling verification of small batches
// on sm_103a: one CTA per sequence with the whole sequence in shared memory.
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
// A decode step with a handful of sequences moves little data; what costs is
// the chain of steps.  Here one CTA takes one sequence: two bulk copies bring
// its K+1 target rows and K draft rows (contiguous in the batch layout) into
// shared memory; each warp reduces whole rows to their normalisers; warp 0
// runs the K accept tests in parallel lanes and finds the first rejection n
// with a ballot; all warps then compute the fixed-point masses of the drawn
// row(s) per run of 32 vectors, straight from shared memory, and warp 0
// locates the crossing of floor(u_K * S) and writes the outputs.  Every row
// is read once from HBM, the draw reads nothing more, and no CTA depends on
// another or on a workspace.
#include "device_common.cuh"
#include "launch.h"
#include "sample_common.cuh"

namespace specv {
namespace {

constexpr int kSeqThreads = 256;
constexpr int kSeqWarps = kSeqThreads / 32;
constexpr int kSeqK1 = 65;                       // K + 1 <= 65
constexpr int kSeqRuns = kSeqMaxBytes / 16 / 32; // 32-vector runs of the longest row
constexpr int kCopyVecS = 2048;                  // vectors per bulk copy (32 KiB)

template <typename E>
__global__ void __launch_bounds__(kSeqThreads)
seq_sample_kernel(VerifyArgs a, int nvec) {
  constexpr int VEC = Staged<E>::kVec;
  extern __shared__ __align__(128) uint4 rows[];  // [K+1 target rows][K draft rows] x nvec
  __shared__ __align__(8) unsigned long long bar;
  __shared__ float4 s_norm[2 * kSeqK1];           // row r: (offset, z, -, -)
  __shared__ unsigned long long s_run[kSeqRuns];
  __shared__ float s_u[kSeqK1];
  __shared__ int s_x[kSeqK1];
  __shared__ int s_n, s_near, s_tok, s_cnear, s_redo;

  const int b = blockIdx.x;
  const int K = a.K, K1 = K + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float s = a.scale;
  const int nrows = 2 * K + 1;
  const int ne = (nvec + 31) >> 5;

  // ---- stage the sequence ----------------------------------------------
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    const long long tvec = static_cast<long long>(K1) * nvec, dvec = static_cast<long long>(K) * nvec;
    mbar_arrive_expect_tx(&bar, static_cast<uint32_t>((tvec + dvec) * 16));
    const uint4* tsrc = static_cast<const uint4*>(a.target) + static_cast<size_t>(b) * tvec;
    for (long long c0 = 0; c0 < tvec; c0 += kCopyVecS)
      bulk_load(rows + c0, tsrc + c0, static_cast<uint32_t>(min(static_cast<long long>(kCopyVecS), tvec - c0)) * 16u, &bar);
    if (K > 0) {
      const uint4* dsrc = static_cast<const uint4*>(a.draft) + static_cast<size_t>(b) * dvec;
      for (long long c0 = 0; c0 < dvec; c0 += kCopyVecS)
        bulk_load(rows + tvec + c0, dsrc + c0, static_cast<uint32_t>(min(static_cast<long long>(kCopyVecS), dvec - c0)) * 16u, &bar);
    }
  }
  // the uniforms and draft tokens while the rows land
  for (int j = tid; j < K1; j += kSeqThreads) {
    s_u[j] = a.uniforms[static_cast<size_t>(b) * K1 + j];
    if (j < K) s_x[j] = a.tokens[static_cast<size_t>(b) * K + j];
  }
  if (!mbar_wait_sleep(&bar, 0u)) {
    // a copy that never completes: report it, and leave only once the copies
    // are done writing this CTA's shared memory
    if (tid == 0 && a.status) atomicOr(a.status, kWaitTimeout);
    mbar_wait_sleep(&bar, 0u);
    return;
  }

  // ---- normalisers: warp w reduces rows w, w + 8, ... --------------------
  for (int r = warp; r < nrows; r += kSeqWarps) {
    const uint4* row = rows + static_cast<size_t>(r) * nvec;
    RowAcc A{-INFINITY, 0.f};
    for (int v = lane; v < nvec; v += 64) {
      uint4 w[2];
      w[0] = row[v];
      const int n2 = v + 32 < nvec ? 2 : 1;
      if (n2 > 1) w[1] = row[v + 32];
      acc_vectors<E>(A, w, n2, s);
    }
    warp_merge_scaled(A.ms, A.z);
    if (lane == 0) s_norm[r] = make_float4(A.ms, A.z, 0.f, 0.f);
  }
  __syncthreads();

  // ---- accept tests and the first rejection (warp 0) ---------------------
  if (warp == 0) {
    int n = K, bad = 0;
    bool ratio_near = false;
    for (int i0 = 0; i0 < K1; i0 += 32) {
      const int i = i0 + lane;
      bool rej = false, nr = false;
      if (i <= K) {
        const float4 nt = s_norm[i];
        if (!(isfinite(nt.x) && isfinite(nt.y) && nt.y > 0.f)) bad |= kDataNonfiniteLogit;
        if (!(s_u[i] >= 0.f && s_u[i] < 1.f)) bad |= kDataUniformRange;
        if (i < K) {
          const float4 nd = s_norm[K1 + i];
          const int x = s_x[i];
          if (x < 0 || x >= a.V) bad |= kDataTokenRange;
          if (!(isfinite(nd.x) && isfinite(nd.y) && nd.y > 0.f)) bad |= kDataNonfiniteLogit;
          const int xc = min(max(x, 0), a.V - 1);
          const float gx = staged_elem<E>(rows + static_cast<size_t>(i) * nvec, xc);
          const float gy = staged_elem<E>(rows + static_cast<size_t>(K1 + i) * nvec, xc);
          const float px = ex2(fmaf(gx, s, -nt.x)) / nt.y;
          const float qx = ex2(fmaf(gy, s, -nd.x)) / nd.y;
          if (SPEC_IN(static_cast<long long>(b) * K + i, static_cast<long long>(a.B) * K, a.status)) {
            if (a.p_at) a.p_at[static_cast<size_t>(b) * K + i] = px;
            if (a.q_at) a.q_at[static_cast<size_t>(b) * K + i] = qx;
          }
          rej = !(s_u[i] * qx < px);
          nr = qx > 0.f && fabsf(s_u[i] - fminf(1.f, px / qx)) < kBandF;
        }
      }
      const unsigned int rb = __ballot_sync(0xffffffffu, rej);
      const unsigned int nb = __ballot_sync(0xffffffffu, nr);
      if (n == K) {  // no rejection before this round (warp-uniform)
        if (rb) {
          const int pick = __ffs(rb) - 1;
          n = i0 + pick;
          ratio_near |= (nb & (pick == 31 ? 0xffffffffu : ((2u << pick) - 1u))) != 0u;
        } else {
          ratio_near |= nb != 0u;
        }
      }
    }
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0) {
      if (bad && a.status) atomicOr(a.status, bad);
      s_n = n;
      s_near = ratio_near ? 1 : 0;
    }
  }
  __syncthreads();

  // ---- the draw from row n (residual) or the bonus row, from shared memory
  const int n = s_n;
  bool residual = n < K;
  const uint4* trow = rows + static_cast<size_t>(n) * nvec;
  const uint4* drow = rows + static_cast<size_t>(K1 + (residual ? n : 0)) * nvec;
  const float4 nt = s_norm[n];
  const float4 nd = residual ? s_norm[K1 + n] : make_float4(0.f, 1.f, 0.f, 0.f);
  const float MSt = nt.x, invZt = 1.f / nt.y, MSd = nd.x;
  for (int rnd = 0; rnd < 2; ++rnd) {
    const float invZd = residual ? 1.f / nd.y : 0.f;
    // fixed-point mass of every run of 32 vectors (warp w: runs w, w + 8, ...)
    for (int e = warp; e < ne; e += kSeqWarps) {
      const int v = e * 32 + lane;
      float xt[VEC], xd[VEC], r[VEC];
#pragma unroll
      for (int q = 0; q < VEC; ++q) xt[q] = xd[q] = -INFINITY;
      if (v < nvec) {
        Staged<E>::unpack(trow[v], xt);
        if (residual) Staged<E>::unpack(drow[v], xd);
      }
      const unsigned long long m = warp_sum_mass(
          vec_weight_scaled<VEC>(xt, xd, MSt, invZt, MSd, invZd, s, residual, r));
      if (lane == 0) s_run[e] = m;
    }
    __syncthreads();
    bool redo = false;
    if (warp == 0) {  // (in the second round residual is false, so redo stays false)
      // S, then the run holding the crossing: each lane sums a block of runs
      const int per = (ne + 31) >> 5;
      const int e0 = min(lane * per, ne), e1 = min(e0 + per, ne);
      unsigned long long bs = 0;
      for (int e = e0; e < e1; ++e) bs += s_run[e];
      const unsigned long long incl = warp_scan_u64(bs, lane);
      const unsigned long long S = __shfl_sync(0xffffffffu, incl, 31);
      int token = 0, cnear = 0;
      if (S == 0 && residual) {
        redo = true;  // p == q on the whole row: the draw falls back to p_n
      } else if (S != 0) {
        const unsigned long long theta = draw_threshold(s_u[K], S);
        const int lb = __ffs(__ballot_sync(0xffffffffu, incl > theta)) - 1;
        unsigned long long base = __shfl_sync(0xffffffffu, incl - bs, lb);
        const int s0 = __shfl_sync(0xffffffffu, e0, lb), s1 = __shfl_sync(0xffffffffu, e1, lb);
        int estar = s1 - 1;
        for (int c0 = s0; c0 < s1; c0 += 32) {
          const int e = c0 + lane;
          const unsigned long long m = e < s1 ? s_run[e] : 0ull;
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
        // the crossing run's 32 vectors again (same arithmetic, integer rounding)
        const int v = estar * 32 + lane;
        float xt[VEC], xd[VEC], r[VEC];
#pragma unroll
        for (int q = 0; q < VEC; ++q) xt[q] = xd[q] = -INFINITY;
        if (v < nvec) {
          Staged<E>::unpack(trow[v], xt);
          if (residual) Staged<E>::unpack(drow[v], xd);
        }
        const unsigned long long w =
            vec_weight_scaled<VEC, true>(xt, xd, MSt, invZt, MSd, invZd, s, residual, r);
        const unsigned long long wi = warp_scan_u64(w, lane);
        const unsigned int h3 = __ballot_sync(0xffffffffu, base + wi > theta);
        const int lstar = h3 ? __ffs(h3) - 1 : 31;
        int tok = 0, nr = 0;
        if (lane == lstar) {
          const unsigned long long before = base + wi - w;
          unsigned long long c_prev, c_cur;
          const int mstar = pick_in_vector<VEC>(r, w, theta - before, c_prev, c_cur);
          const long long t = static_cast<long long>(v) * VEC + mstar;
          nr = near_step(theta, before + c_prev, before + c_cur, S) ? 1 : 0;
          tok = static_cast<int>(t < a.V ? t : a.V - 1);
        }
        token = __shfl_sync(0xffffffffu, tok, lstar);
        cnear = __shfl_sync(0xffffffffu, nr, lstar);
      }
      if (lane == 0) {
        s_tok = token;
        s_cnear = cnear;
        s_redo = redo ? 1 : 0;
      }
    }
    __syncthreads();
    if (!s_redo) break;  // block-uniform; the second round never redoes
    residual = false;
  }

  // ---- outputs (warp 0) ------------------------------------------------
  if (warp == 0 && SPEC_IN(b, a.B, a.status) && SPEC_IN(n, K1, a.status)) {
    const int token = s_tok;
    for (int j = lane; j < K1; j += 32) {
      int o = -1;
      if (j < n) o = min(max(s_x[j], 0), a.V - 1);
      else if (j == n) o = token;
      a.out_tokens[static_cast<size_t>(b) * K1 + j] = o;
    }
    if (lane == 0) {
      if (a.accepted_len) a.accepted_len[b] = n;
      if (a.flags) a.flags[b] = (s_near ? kFlagRatio : 0u) | (s_cnear ? kFlagCdf : 0u);
      if (a.p_emit) a.p_emit[b] = ex2(fmaf(staged_elem<E>(trow, token), s, -MSt)) * invZt;
    }
  }
}

}  // namespace

long long seq_sample_bytes(int K, long long nvec) {
  return static_cast<long long>(2 * K + 1) * nvec * 16;
}

cudaError_t seq_sample_prepare() {
  cudaError_t e = cudaFuncSetAttribute(seq_sample_kernel<BF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSeqMaxBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(seq_sample_kernel<F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSeqMaxBytes);
  return e;
}

cudaError_t launch_sample_seq(const VerifyArgs& a, cudaStream_t stream) {
  const long long nvec = static_cast<long long>(a.V) * (a.bf16 ? 2 : 4) / 16;
  const long long bytes = seq_sample_bytes(a.K, nvec);
  if (!a.vec || a.K + 1 > kSeqK1 || bytes > kSeqMaxBytes || a.B < 1) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(a.B));
  cfg.blockDim = dim3(kSeqThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(bytes);
  cfg.stream = stream;
  return a.bf16 ? cudaLaunchKernelEx(&cfg, seq_sample_kernel<BF16>, a, static_cast<int>(nvec))
                : cudaLaunchKernelEx(&cfg, seq_sample_kernel<F32>, a, static_cast<int>(nvec));
}

}  // namespace specv
