// rejection_cut.cu -- Speculative Rejection's cut ("Speculative Rejection"
// review, section 4.2 "算法", the speculative-rejection phase): for each of G
// prompts, r_cut = the alpha-quantile of its N partial reward scores, and the
// sequences scoring at least r_cut are kept.
//
// Quantile: linear interpolation between the order statistics s_j and
// s_{j+1} (0-based, j = floor(alpha (N-1)), g = alpha (N-1) - j, j+1 clamped
// to N-1):  r_cut = s_j + g (s_{j+1} - s_j)  in IEEE double without FMA.
//
// The two order statistics come from a most-significant-digit radix select
// on order-preserving 32-bit keys of the fp32 scores (four 8-bit digits, a
// 256-bin shared-memory histogram per pass): exact, no sort, and each pass
// touches only the keys still matching the selected prefix.  The keep test
// compares keys against the key of c = r_cut rounded up to fp32, which keeps
// exactly the scores x with (double)x >= r_cut (c is the smallest float
// >= r_cut, and keys order as the values do).
//
//  - N <= 1024: one warp per prompt, the row held in registers (up to 32
//    scores a lane), read once from HBM; its kept indices are written with
//    warp ballots in ascending order.  No block-wide barrier.
//  - N > 1024: one CTA per prompt; every pass re-reads the row (from L2).
#include <climits>
#include <cmath>
#include <cstdint>

#include "../../include/spec_verify.h"
#include "launch.h"

namespace specv {
namespace {

constexpr int kDataNonfiniteScore = 16;  // SPEC_DATA_NONFINITE_SCORE
constexpr int kCutWarps = 8;             // prompts per CTA, one-warp-per-prompt kernel
constexpr int kCutBlock = 512;           // threads per CTA, one-CTA-per-prompt kernel
constexpr int kWarpMaxN = 1024;          // rows the warp kernel holds in registers

// Unsigned keys that order like the floats: negative values have all bits
// flipped, the others the sign bit set.  -0 is keyed as +0 (v + 0 is +0 for
// v = -0), so that keys compare exactly as the values do.  Finite values get
// keys in [0x00800000, 0xff7fffff].
__device__ __forceinline__ unsigned int ord_key(float v) {
  const unsigned int b = __float_as_uint(v + 0.f);
  return b ^ (static_cast<unsigned int>(static_cast<int>(b) >> 31) | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned int k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}
__device__ __forceinline__ bool nonfinite(float v) {
  return (__float_as_uint(v) & 0x7f800000u) == 0x7f800000u;
}

// s_j + g (s_{j+1} - s_j), each operation rounded on its own.
__device__ __forceinline__ double cut_value(float lo, float hi, double g) {
  const double dlo = static_cast<double>(lo);
  return __dadd_rn(dlo, __dmul_rn(g, __dsub_rn(static_cast<double>(hi), dlo)));
}

// One warp finds the bin of a 256-bin histogram that holds rank r (0-based,
// counting from bin 0) and the count of the bins before it.  Lane l owns bins
// 8l .. 8l+7.  Every lane returns the same values.
__device__ __forceinline__ int select_bin(const unsigned int* h, unsigned int r, int lane,
                                          unsigned int* before_out, unsigned int* count_out) {
  const uint4 a = reinterpret_cast<const uint4*>(h)[lane * 2];
  const uint4 b = reinterpret_cast<const uint4*>(h)[lane * 2 + 1];
  const unsigned int c[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  unsigned int tot = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += c[i];
  unsigned int incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const unsigned int excl = incl - tot;
  int bin = lane * 8;
  unsigned int before = excl, cnt = 0, run = excl;
  bool found = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (!found && r < run + c[i]) {
      bin = lane * 8 + i;
      before = run;
      cnt = c[i];
      found = true;
    }
    run += c[i];
  }
  const unsigned int own = __ballot_sync(0xffffffffu, r >= excl && r < incl);
  const int src = own ? __ffs(own) - 1 : 0;  // rank r < total always has an owner
  *before_out = __shfl_sync(0xffffffffu, before, src);
  *count_out = __shfl_sync(0xffffffffu, cnt, src);
  return __shfl_sync(0xffffffffu, bin, src);
}

// One warp per prompt; lane l holds scores l, l+32, ... (KPL of them).
// Slots past N hold key 0, below every finite score's key (pads), so rank j
// of the scores is rank j + npad of the slots and no later step has to skip
// the pads: they are never kept and never above a selected key.
template <int KPL>
__global__ void __launch_bounds__(kCutWarps * 32, 4)
    cut_warp_kernel(const float* __restrict__ scores, int G, int N, int j, double g,
                    double* __restrict__ r_cut, int32_t* __restrict__ n_accepted,
                    int32_t* __restrict__ accepted, int32_t* status) {
  __shared__ __align__(16) unsigned int hist_all[kCutWarps][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long pr = static_cast<long long>(blockIdx.x) * kCutWarps + warp;
  if (pr >= G) return;
  unsigned int* h = hist_all[warp];
  const float* row = scores + pr * N;
  int32_t* out = accepted + pr * N;

  unsigned int key[KPL];
  float nf = 0.f;  // becomes NaN once a score is NaN or infinite (x * 0)
#pragma unroll
  for (int k = 0; k < KPL; ++k) {
    const int i = k * 32 + lane;
    const float v = i < N ? __ldg(row + i) : 0.f;
    nf = fmaf(v, 0.f, nf);
    key[k] = i < N ? ord_key(v) : 0u;
  }
  if (__any_sync(0xffffffffu, nf != nf)) {
    if (lane == 0) {
      r_cut[pr] = __longlong_as_double(0x7ff8000000000000LL);
      n_accepted[pr] = 0;
      if (status) atomicOr(status, kDataNonfiniteScore);
    }
    for (int i = lane; i < N; i += 32) out[i] = -1;
    return;
  }
  const unsigned int jj = static_cast<unsigned int>(j + (KPL * 32 - N));  // rank among slots

  // radix select of slot rank jj
  unsigned int prefix = 0, pmask = 0, r = jj, cnt = 0;
  bool unique = false;
#pragma unroll 1
  for (int shift = 24; shift >= 0 && !unique; shift -= 8) {
    reinterpret_cast<uint4*>(h)[lane * 2] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(h)[lane * 2 + 1] = make_uint4(0, 0, 0, 0);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < KPL; ++k)
      if ((key[k] & pmask) == prefix) atomicAdd(&h[(key[k] >> shift) & 255u], 1u);
    __syncwarp();
    unsigned int before;
    const int bin = select_bin(h, r, lane, &before, &cnt);
    r -= before;
    prefix |= static_cast<unsigned int>(bin) << shift;
    pmask |= 255u << shift;
    unique = cnt == 1;  // one key left with this prefix: it is rank jj
    __syncwarp();
  }
  // Selected key: with one key left in the bin it is the smallest key >=
  // prefix (keys below prefix wrap around in key - prefix); after all four
  // digits it is the prefix itself, held by cnt keys of which r rank before.
  unsigned int klo = prefix;
  if (unique) {
    unsigned int m = 0xffffffffu;
#pragma unroll
    for (int k = 0; k < KPL; ++k) m = min(m, key[k] - prefix);
    klo = prefix + __reduce_min_sync(0xffffffffu, m);
  }
  // rank jj + 1: klo again while copies of klo remain, else the next larger
  // key (keys <= klo wrap around in key - klo - 1)
  unsigned int khi = klo;
  const bool repeats = !unique && r + 1 < cnt;
  if (j + 1 < N && !repeats) {
    unsigned int m = 0xffffffffu;
#pragma unroll
    for (int k = 0; k < KPL; ++k) m = min(m, key[k] - klo - 1u);
    khi = klo + 1u + __reduce_min_sync(0xffffffffu, m);
  }
  const double rc = cut_value(key_value(klo), key_value(khi), g);
  const unsigned int kc = ord_key(__double2float_ru(rc));

  // kept indices in ascending order, then -1
  int base = 0;
  const unsigned int lt = (1u << lane) - 1u;
#pragma unroll
  for (int k = 0; k < KPL; ++k) {
    const bool keep = key[k] >= kc;
    const unsigned int bal = __ballot_sync(0xffffffffu, keep);
    if (keep) out[base + __popc(bal & lt)] = k * 32 + lane;
    base += __popc(bal);
  }
  for (int i = base + lane; i < N; i += 32) out[i] = -1;
  if (lane == 0) {
    r_cut[pr] = rc;
    n_accepted[pr] = base;
  }
}

// One CTA per prompt, for rows longer than the warp kernel holds.
__global__ void __launch_bounds__(kCutBlock)
    cut_block_kernel(const float* __restrict__ scores, int G, int N, int j, double g,
                     double* __restrict__ r_cut, int32_t* __restrict__ n_accepted,
                     int32_t* __restrict__ accepted, int32_t* status) {
  constexpr int kW = kCutBlock / 32;
  __shared__ __align__(16) unsigned int h[256];
  __shared__ unsigned int s_bin, s_before, s_le, s_above;
  __shared__ unsigned int s_wsum[kW];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long pr = blockIdx.x;
  const float* row = scores + pr * N;
  int32_t* out = accepted + pr * N;

  bool bad = false;
  for (int i = tid; i < N; i += kCutBlock) bad |= nonfinite(__ldg(row + i));
  if (__syncthreads_or(bad)) {
    if (tid == 0) {
      r_cut[pr] = __longlong_as_double(0x7ff8000000000000LL);
      n_accepted[pr] = 0;
      if (status) atomicOr(status, kDataNonfiniteScore);
    }
    for (int i = tid; i < N; i += kCutBlock) out[i] = -1;
    return;
  }

  unsigned int prefix = 0, pmask = 0, r = static_cast<unsigned int>(j);
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) h[tid] = 0;
    __syncthreads();
    for (int i = tid; i < N; i += kCutBlock) {
      const unsigned int k = ord_key(__ldg(row + i));
      if ((k & pmask) == prefix) atomicAdd(&h[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      unsigned int before, cnt;
      const int bin = select_bin(h, r, lane, &before, &cnt);
      if (lane == 0) {
        s_bin = static_cast<unsigned int>(bin);
        s_before = before;
      }
    }
    __syncthreads();
    r -= s_before;
    prefix |= s_bin << shift;
    pmask |= 255u << shift;
    __syncthreads();  // s_bin / s_before are read before the next pass rewrites them
  }
  const unsigned int klo = prefix;
  if (tid == 0) {
    s_le = 0;
    s_above = 0xffffffffu;
  }
  __syncthreads();
  unsigned int le = 0, above = 0xffffffffu;
  for (int i = tid; i < N; i += kCutBlock) {
    const unsigned int k = ord_key(__ldg(row + i));
    le += k <= klo ? 1u : 0u;
    if (k > klo) above = min(above, k);
  }
  le = __reduce_add_sync(0xffffffffu, le);
  above = __reduce_min_sync(0xffffffffu, above);
  if (lane == 0) {
    atomicAdd(&s_le, le);
    atomicMin(&s_above, above);
  }
  __syncthreads();
  const unsigned int khi =
      (j + 1 >= N || s_le >= static_cast<unsigned int>(j) + 2u) ? klo : s_above;
  const double rc = cut_value(key_value(klo), key_value(khi), g);
  const unsigned int kc = ord_key(__double2float_ru(rc));

  const unsigned int lt = (1u << lane) - 1u;
  int base = 0;
  for (int c0 = 0; c0 < N; c0 += kCutBlock) {
    const int i = c0 + tid;
    const bool keep = i < N && ord_key(__ldg(row + i)) >= kc;
    const unsigned int bal = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) s_wsum[warp] = __popc(bal);
    __syncthreads();
    int off = base, tot = 0;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const int n = static_cast<int>(s_wsum[w]);
      off += w < warp ? n : 0;
      tot += n;
    }
    if (keep) out[off + __popc(bal & lt)] = i;
    base += tot;
    __syncthreads();  // s_wsum is read before the next chunk rewrites it
  }
  for (int i = base + tid; i < N; i += kCutBlock) out[i] = -1;
  if (tid == 0) {
    r_cut[pr] = rc;
    n_accepted[pr] = base;
  }
}

}  // namespace

cudaError_t launch_rejection_cut(const float* scores, int G, int N, int j, double g,
                                 double* r_cut, int32_t* n_accepted, int32_t* accepted,
                                 int32_t* status, cudaStream_t stream) {
  if (N > kWarpMaxN) {
    cut_block_kernel<<<G, kCutBlock, 0, stream>>>(scores, G, N, j, g, r_cut, n_accepted,
                                                  accepted, status);
    return cudaGetLastError();
  }
  const int grid = (G + kCutWarps - 1) / kCutWarps;
  if (N <= 128)
    cut_warp_kernel<4><<<grid, kCutWarps * 32, 0, stream>>>(scores, G, N, j, g, r_cut,
                                                            n_accepted, accepted, status);
  else if (N <= 256)
    cut_warp_kernel<8><<<grid, kCutWarps * 32, 0, stream>>>(scores, G, N, j, g, r_cut,
                                                            n_accepted, accepted, status);
  else if (N <= 512)
    cut_warp_kernel<16><<<grid, kCutWarps * 32, 0, stream>>>(scores, G, N, j, g, r_cut,
                                                             n_accepted, accepted, status);
  else
    cut_warp_kernel<32><<<grid, kCutWarps * 32, 0, stream>>>(scores, G, N, j, g, r_cut,
                                                             n_accepted, accepted, status);
  return cudaGetLastError();
}

}  // namespace specv

extern "C" {

spec_status_t spec_rejection_cut(const float* scores, int G, int N, double alpha, double* r_cut,
                                 int32_t* n_accepted, int32_t* accepted, spec_stream_t stream,
                                 int32_t* device_status) {
  SPEC_RANGE("spec_rejection_cut");
  if (G < 0 || N < 0 || !(alpha >= 0.0 && alpha <= 1.0)) return SPEC_ERR_INVALID_ARG;
  if (G == 0) return SPEC_OK;
  if (N < 1 || !scores || !r_cut || !n_accepted || !accepted) return SPEC_ERR_INVALID_ARG;
  const auto misaligned = [](const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) != 0;
  };
  if (misaligned(scores, 4) || misaligned(r_cut, 8) || misaligned(n_accepted, 4) ||
      misaligned(accepted, 4) || (device_status && misaligned(device_status, 4)))
    return SPEC_ERR_INVALID_ARG;
  // the same double arithmetic as the definition: h = alpha (N - 1)
  const double h = alpha * static_cast<double>(N - 1);
  const double jf = std::floor(h);
  const int j = static_cast<int>(jf);
  const double g = h - jf;
  const cudaError_t e = specv::launch_rejection_cut(scores, G, N, j, g, r_cut, n_accepted,
                                                    accepted, device_status,
                                                    reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"
