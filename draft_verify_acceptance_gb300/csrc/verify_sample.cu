// verify_sample.cu -- speculative-sampling verification on sm_103a.
//
// Sources (page title, section):
//   "推测性拒绝采样", 技术原理与步骤 steps 2-4: all K+1 target rows come from one
//     parallel pass; x_i is accepted when p(x_i) >= q(x_i), else with
//     probability p(x_i)/q(x_i); everything after the first rejection is
//     dropped and one replacement token is drawn there.  关键保证: the output
//     follows the target distribution exactly, which makes the replacement
//     law normalize(max(0, p - q)).
//   "논문 리뷰 [Speculative Contrastive Decoding]", Speculative Decoding: with
//     all K accepted, the target supplies token K+1 (drawn from p_K).
//
// Design (one thread-block cluster per (position i, sequence b) row pair):
//   pass 1  each CTA of the cluster streams its 1/C slice of target row i
//           and draft row i once from HBM (16-byte non-allocating loads) and
//           keeps an online (max, sum 2^((x-max)*log2e/T)) per row;
//           partials are pushed to every CTA's shared memory (DSMEM) and
//           merged in rank order, so all CTAs hold identical normalisers.
//   accept  p(x_i), q(x_i) from two gathered logits; accept iff u_i*q < p.
//           Rank 0 records a rejection in the sequence's reject mask.  A row
//           that accepts, or that sees an earlier rejection of its sequence
//           already recorded, is done: its replacement can never be used.
//   pass 2  rows that still may be the first rejection (and the bonus row)
//           re-read their slice (normally an L2 hit: it was read a few
//           microseconds earlier) and form r_j = max(0, p_j - q_j) (or p_j).
//           Each 16-byte vector's fp32 sum is converted to a 2^-56 fixed-
//           point integer; integer sums are exact in any order, so the
//           per-tile, per-warp, per-CTA and cluster totals all agree
//           bit-for-bit with one another.
//   pass 3  the CTA holding the crossing of u_K * S walks its per-tile/per-
//           warp sums, re-reads the 32 vectors of the crossing warp, scans
//           them and walks the crossing vector's elements in token order.
//   finalise  the CTA that completes the last row of sequence b (an atomic
//           counter, no waiting) reads the reject mask, picks n and the
//           candidate of row n, writes the outputs and zeroes its workspace.
#include <cooperative_groups.h>

#include <climits>

#include "device_common.cuh"
#include "launch.h"
#include "launch_ee.h"
#include "sample_common.cuh"

namespace cg = cooperative_groups;

namespace specv {

namespace {

// Online update of (m, z) with a register chunk.
template <int N>
__device__ __forceinline__ void online_chunk(float& m, float& z, const float* x, float s) {
  float cm = x[0];
#pragma unroll
  for (int k = 1; k < N; ++k) cm = fmaxf(cm, x[k]);
  const float nm = fmaxf(m, cm);
  if (nm != -INFINITY) {
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < N; ++k) acc += ex2((x[k] - nm) * s);
    z = z * ex2((m - nm) * s) + acc;  // ex2(0) = 1, ex2(-inf) = 0
    m = nm;
  }
}

// Finalise sequence b (called by the single last arrival).
__device__ void finalize_sequence(const VerifyArgs& a, int b) {
  const int K = a.K, K1 = K + 1;
  SeqState* st = a.seq + b;
  const unsigned long long mask = *reinterpret_cast<volatile unsigned long long*>(&st->reject_mask);
  const unsigned long long near = *reinterpret_cast<volatile unsigned long long*>(&st->near_mask);
  const int n = mask ? (__ffsll(static_cast<long long>(mask)) - 1) : K;
  const volatile int32_t* slots = static_cast<const volatile int32_t*>(a.slots);
  const int32_t c = slots[4 * (static_cast<size_t>(b) * K1 + n)];
  const int32_t* x = a.tokens + static_cast<size_t>(b) * K;
  int32_t* out = a.out_tokens + static_cast<size_t>(b) * K1;
  for (int j = 0; j < n; ++j) out[j] = min(max(x[j], 0), a.V - 1);
  out[n] = c & 0x7fffffff;
  for (int j = n + 1; j < K1; ++j) out[j] = -1;
  if (a.accepted_len) a.accepted_len[b] = n;
  if (a.flags) {
    const unsigned long long evaluated = (n >= 63) ? ~0ull : ((2ull << n) - 1ull);
    a.flags[b] = ((near & evaluated) ? kFlagRatio : 0u) | ((c < 0) ? kFlagCdf : 0u);
  }
  // leave this sequence's part of the workspace zero-filled for the next call
  volatile int32_t* wslots = static_cast<volatile int32_t*>(a.slots);
  for (int j = 0; j < K1; ++j) wslots[4 * (static_cast<size_t>(b) * K1 + j)] = 0;
  st->reject_mask = 0ull;
  st->near_mask = 0ull;
  st->arrivals = 0u;
}

// Load the VEC-element vector vv of a row slice, or -inf past its end.
template <typename E, int VEC>
__device__ __forceinline__ void load_or_pad(const void* row, long long vv, long long v1,
                                            float (&x)[VEC]) {
  if (vv < v1) {
    VecLoad<E, VEC>::load(row, vv, x);
  } else {
#pragma unroll
    for (int q = 0; q < VEC; ++q) x[q] = -INFINITY;
  }
}

template <typename E, int VEC, int U, int U2>
__global__ void __launch_bounds__(kThreads)
sample_kernel(VerifyArgs a, long long nvec, int ntiles) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const long long pair = blockIdx.x / C;  // position-major: earlier positions launch first
  const int K = a.K, K1 = K + 1;
  const int i = static_cast<int>(pair / a.B);
  const int b = static_cast<int>(pair - static_cast<long long>(i) * a.B);
  const bool has_draft = i < K;
  const size_t rowbytes = static_cast<size_t>(a.V) * E::kBytes;
  const char* trow = static_cast<const char*>(a.target) + (static_cast<size_t>(b) * K1 + i) * rowbytes;
  const char* drow = has_draft
      ? static_cast<const char*>(a.draft) + (static_cast<size_t>(b) * K + i) * rowbytes
      : trow;
  const long long v0 = nvec * rank / C;
  const long long v1 = nvec * (rank + 1) / C;
  const int ntl = static_cast<int>((v1 - v0 + kThreads - 1) / kThreads);  // tiles here (<= ntiles)
  const float s = a.scale;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t* slots = static_cast<int32_t*>(a.slots);
  const size_t my_slot = 4 * (static_cast<size_t>(b) * K1 + i);

  __shared__ float s_part[kMaxCluster][4];               // pushed by each rank
  __shared__ float s_red[kWarps][4];
  __shared__ int s_need;                                  // pushed by rank 0
  __shared__ unsigned long long s_mass[2][kMaxCluster];   // pushed by each rank
  extern __shared__ unsigned long long s_tws[];           // [ntiles][kWarps]

  cluster_arrive_relaxed();  // matched by cluster_wait() before the first DSMEM push
  // ---- pass 1: online normalisers of target row i and draft row i -------
  float mt = -INFINITY, zt = 0.f, md = -INFINITY, zd = 0.f;
  for (long long v = v0 + tid; v < v1; v += static_cast<long long>(kThreads) * U) {
    float xt[U * VEC], xd[U * VEC];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long vv = v + static_cast<long long>(u) * kThreads;
      load_or_pad<E, VEC>(trow, vv, v1, *reinterpret_cast<float(*)[VEC]>(&xt[u * VEC]));
      if (has_draft)
        load_or_pad<E, VEC>(drow, vv, v1, *reinterpret_cast<float(*)[VEC]>(&xd[u * VEC]));
    }
    online_chunk<U * VEC>(mt, zt, xt, s);
    if (has_draft) online_chunk<U * VEC>(md, zd, xd, s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    merge_mz(mt, zt, __shfl_xor_sync(0xffffffffu, mt, o), __shfl_xor_sync(0xffffffffu, zt, o), s);
    merge_mz(md, zd, __shfl_xor_sync(0xffffffffu, md, o), __shfl_xor_sync(0xffffffffu, zd, o), s);
  }
  if (lane == 0) {
    s_red[warp][0] = mt; s_red[warp][1] = zt; s_red[warp][2] = md; s_red[warp][3] = zd;
  }
  __syncthreads();
  cluster_wait();  // every CTA of the cluster has started
  if (tid < C) {
    float m0 = s_red[0][0], z0 = s_red[0][1], m1 = s_red[0][2], z1 = s_red[0][3];
    for (int w = 1; w < kWarps; ++w) {
      merge_mz(m0, z0, s_red[w][0], s_red[w][1], s);
      merge_mz(m1, z1, s_red[w][2], s_red[w][3], s);
    }
    float* dst = cluster.map_shared_rank(&s_part[rank][0], tid);
    dst[0] = m0; dst[1] = z0; dst[2] = m1; dst[3] = z1;
  }
  cluster.sync();
  // identical merge order in every CTA -> identical normalisers everywhere
  float Mt = s_part[0][0], Zt = s_part[0][1], Md = s_part[0][2], Zd = s_part[0][3];
  for (int r = 1; r < C; ++r) {
    merge_mz(Mt, Zt, s_part[r][0], s_part[r][1], s);
    merge_mz(Md, Zd, s_part[r][2], s_part[r][3], s);
  }
  const float uK = a.uniforms[static_cast<size_t>(b) * K1 + K];

  // ---- accept test and the decision whether this row needs a draw -------
  if (rank == 0 && tid == 0) {
    SeqState* st = a.seq + b;
    int bad = 0;
    if (!(isfinite(Mt) && isfinite(Zt) && Zt > 0.f)) bad |= kDataNonfiniteLogit;
    bool need = true;
    if (has_draft) {
      const int xr = a.tokens[static_cast<size_t>(b) * K + i];
      const int x = min(max(xr, 0), a.V - 1);
      const float ui = a.uniforms[static_cast<size_t>(b) * K1 + i];
      const float px = ex2((load_one<E>(trow, x) - Mt) * s) / Zt;
      const float qx = ex2((load_one<E>(drow, x) - Md) * s) / Zd;
      const bool accept = ui * qx < px;
      if (a.p_at) a.p_at[static_cast<size_t>(b) * K + i] = px;
      if (a.q_at) a.q_at[static_cast<size_t>(b) * K + i] = qx;
      if (xr != x) bad |= kDataTokenRange;
      if (!(ui >= 0.f && ui < 1.f)) bad |= kDataUniformRange;
      if (!(isfinite(Md) && isfinite(Zd) && Zd > 0.f)) bad |= kDataNonfiniteLogit;
      if (qx > 0.f && fabsf(ui - fminf(1.f, px / qx)) < kBandF)
        atomicOr(&st->near_mask, 1ull << i);
      if (!accept) atomicOr(&st->reject_mask, 1ull << i);
      need = !accept;
    } else if (!(uK >= 0.f && uK < 1.f)) {
      bad |= kDataUniformRange;
    }
    if (bad && a.status) atomicOr(a.status, bad);
    if (need) {
      __threadfence();
      const unsigned long long m = *reinterpret_cast<volatile unsigned long long*>(&st->reject_mask);
      const unsigned long long earlier = (i >= 64) ? ~0ull : ((1ull << i) - 1ull);
      if (m & earlier) need = false;  // an earlier position already rejected
    }
    for (int r = 0; r < C; ++r) *cluster.map_shared_rank(&s_need, r) = need ? 1 : 0;
  }
  cluster.sync();
  if (!s_need) {
    if (rank == 0 && tid == 0 && arrive_last(a.seq, b, static_cast<unsigned int>(K1)))
      finalize_sequence(a, b);
    return;
  }

  // ---- pass 2: fixed-point mass of this slice, per tile and warp --------
  const float invZt = 1.f / Zt;
  const float invZd = has_draft ? 1.f / Zd : 0.f;
  bool residual = has_draft;
  int rnd = 0;
  unsigned long long S = 0;
  for (;; ++rnd) {
    for (int kb = 0; kb < ntl; kb += U2) {
      float xt[U2][VEC], xd[U2][VEC];
#pragma unroll
      for (int uu = 0; uu < U2; ++uu) {
        const long long vv = v0 + static_cast<long long>(kb + uu) * kThreads + tid;
        load_or_pad<E, VEC>(trow, vv, v1, xt[uu]);
        if (residual) load_or_pad<E, VEC>(drow, vv, v1, xd[uu]);
      }
#pragma unroll
      for (int uu = 0; uu < U2; ++uu) {
        float r[VEC];
        const unsigned long long w =
            warp_sum_u64(vec_weight<VEC>(xt[uu], xd[uu], Mt, invZt, Md, invZd, s, residual, r));
        if (lane == 0 && kb + uu < ntl) s_tws[(kb + uu) * kWarps + warp] = w;
      }
    }
    __syncthreads();
    if (warp == 0) {
      unsigned long long t = 0;
      for (int k = lane; k < ntl * kWarps; k += 32) t += s_tws[k];
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
    if (rank == 0 && tid == 0) {
      slots[my_slot] = 0;
      if (arrive_last(a.seq, b, static_cast<unsigned int>(K1))) finalize_sequence(a, b);
    }
    return;
  }
  const unsigned long long theta = draw_threshold(uK, S);
  // the slice holding the crossing: first rank whose running total passes theta
  int cstar = C - 1;
  unsigned long long off = 0;
  for (int r = 0; r < C; ++r) {
    const unsigned long long m = s_mass[rnd][r];
    if (off + m > theta) { cstar = r; break; }
    off += m;
  }
  if (rank != cstar || warp != 0) return;
  if (ntl <= 0) {  // cannot hold the crossing (its mass is 0); keeps indexing in bounds
    if (lane == 0) {
      slots[my_slot] = 0;
      if (arrive_last(a.seq, b, static_cast<unsigned int>(K1))) finalize_sequence(a, b);
    }
    return;
  }

  // ---- pass 3: the crossing inside this slice (warp 0 of that CTA) ------
  const unsigned long long tl = theta - off;
  unsigned long long base = 0;
  int kstar = ntl - 1;
  for (int k0 = 0; k0 < ntl; k0 += 32) {
    const int k = k0 + lane;
    unsigned long long tt = 0;
    if (k < ntl)
      for (int w = 0; w < kWarps; ++w) tt += s_tws[k * kWarps + w];
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
    const unsigned long long m = s_tws[kstar * kWarps + w];
    if (base + m > tl) { wstar = w; break; }
    base += m;
  }
  const long long vv = v0 + static_cast<long long>(kstar) * kThreads + wstar * 32 + lane;
  float xt[VEC], xd[VEC], r[VEC];
  load_or_pad<E, VEC>(trow, vv, v1, xt);
  if (residual) load_or_pad<E, VEC>(drow, vv, v1, xd);
  const unsigned long long w = vec_weight<VEC, true>(xt, xd, Mt, invZt, Md, invZd, s, residual, r);
  unsigned long long incl = w;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  const unsigned int hit = __ballot_sync(0xffffffffu, base + incl > tl);
  const int lstar = hit ? (__ffs(hit) - 1) : 31;
  if (lane != lstar) return;
  const unsigned long long before = base + incl - w;  // slice prefix before this vector
  const unsigned long long rem = tl - before;
  float acc = 0.f;
  int mstar = VEC - 1;
  unsigned long long c_prev = 0, c_cur = w;
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    acc = __fadd_rn(acc, r[k]);
    const unsigned long long c = fix56(acc);
    if (c > rem) { mstar = k; c_cur = c; break; }
    c_prev = c;
  }
  const long long token = vv * VEC + mstar;
  const bool near = near_step(theta, off + before + c_prev, off + before + c_cur, S);
  const int32_t tok = static_cast<int32_t>(token < a.V ? token : a.V - 1);
  slots[my_slot] = near ? static_cast<int32_t>(static_cast<uint32_t>(tok) | 0x80000000u) : tok;
  if (arrive_last(a.seq, b, static_cast<unsigned int>(K1))) finalize_sequence(a, b);
}

template <typename E, int VEC, int U>
cudaError_t launch_sample_t(const VerifyArgs& a, cudaStream_t stream) {
  const long long nvec = a.V / VEC;
  const int C = sample_cluster_size(a.V, E::kBytes);
  const long long ntiles = sample_tiles(nvec, C);
  if (ntiles > kMaxTiles) return cudaErrorInvalidConfiguration;
  const long long pairs = static_cast<long long>(a.B) * (a.K + 1);
  const long long grid = pairs * C;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(ntiles) * kWarps * sizeof(unsigned long long);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sample_kernel<E, VEC, U, (U > 2 ? 2 : U)>, a, nvec, static_cast<int>(ntiles));
}

template <typename E, int VEC, int U>
cudaError_t prepare_t() {
  return cudaFuncSetAttribute(sample_kernel<E, VEC, U, (U > 2 ? 2 : U)>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kMaxTiles * kWarps * static_cast<int>(sizeof(unsigned long long)));
}

}  // namespace

// Cluster size: about 32 KiB of each row per CTA, at most 8 CTAs.
int sample_cluster_size(long long V, int elem_bytes) {
  const long long bytes = V * elem_bytes;
  long long C = (bytes + 32767) / 32768;
  if (C < 1) C = 1;
  if (C > kMaxCluster) C = kMaxCluster;
  return static_cast<int>(C);
}

// Tiles of kThreads vectors in the largest slice of a row.
long long sample_tiles(long long nvec, int cluster) {
  const long long per = (nvec + cluster - 1) / cluster;
  const long long t = (per + kThreads - 1) / kThreads;
  return t < 1 ? 1 : t;
}

cudaError_t sample_prepare() {
  cudaError_t e;
  if ((e = prepare_t<BF16, 8, 4>()) != cudaSuccess) return e;
  if ((e = prepare_t<BF16, 1, 8>()) != cudaSuccess) return e;
  if ((e = prepare_t<F32, 4, 4>()) != cudaSuccess) return e;
  return prepare_t<F32, 1, 8>();
}

cudaError_t launch_sample(const VerifyArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  if (a.vec) {
    const long long nvec = static_cast<long long>(a.V) * (a.bf16 ? 2 : 4) / 16;
    // a draw that fits one segment: the fused kernel draws as it streams;
    // longer rows: the two-kernel sampler, whose per-sequence clusters finish
    // the last draws sooner (measured: the fused kernel takes 59 / 106 us on
    // the 128256-row bf16 and 152064-row fp32 batches, against 47 / 65)
    // a batch of at most one sequence per SM whose sequences fit one CTA's
    // shared memory: one CTA per sequence, everything on chip (early-exit
    // mode included: every row is read anyway, and the outputs are the same)
    if (a.B <= dev.sm_count && seq_sample_bytes(a.K, nvec) <= kSeqMaxBytes)
      return launch_sample_seq(a, stream);
    // early exit: one cluster per sequence walks its positions in order and
    // reads no row after the first rejection (clusters that do not fit at
    // once run in waves; nothing waits across clusters).  Measured against
    // the two-phase schedule below: 3.2x faster when a few sequences accept
    // x_0 and force its second phase, 1.7x when none does, 1.2x when most
    // accept every position; rows too long for a cluster take the two phases
    if (a.early_exit && a.K >= 1) {
      const int Ce = ee_cluster(nvec);
      if (Ce > 0) return launch_sample_ee(a, Ce, stream);
    }
    const int C = sample_2p_cluster(nvec);
    if (a.early_exit && a.K >= 1 && C > 0) return launch_sample_early_exit(a, dev, C, stream);
    if (nvec <= kFusedSeg) return launch_sample_fused(a, dev, stream);
    if (C > 0) return launch_sample_2p(a, dev, C, stream);
  }
  // unaligned rows, or rows too long for the fused kernel: the streaming
  // kernel below
  if (a.bf16) {
    return a.vec ? launch_sample_t<BF16, 8, 4>(a, stream)
                 : launch_sample_t<BF16, 1, 8>(a, stream);
  }
  return a.vec ? launch_sample_t<F32, 4, 4>(a, stream)
               : launch_sample_t<F32, 1, 8>(a, stream);
}

}  // namespace specv
