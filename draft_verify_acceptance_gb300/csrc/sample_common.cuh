// sample_common.cuh -- pieces shared by the two sampling kernels: the
// fixed-point residual weights of one vector, and the warp-parallel
// finalisation of a sequence.
#pragma once

#include "device_common.cuh"
#include "launch.h"

namespace specv {

constexpr float kBandF = 1e-6f;               // boundary band of the ratio test

// round(2^56 * acc) to nearest, ties to even, for a finite acc in [0, 2^7),
// with integer operations only: acc = m * 2^(e - 150) (m with its implicit
// bit), so 2^56 * acc = m * 2^(e - 94).  The same value as fix56_cvt (the
// hardware conversion of the exact product 2^56 * acc), with a shorter
// latency: the 64-bit float-to-integer conversion runs on a narrow pipe of
// this GPU (about 100 cycles, 2 results per clock per SM).  Latency-bound
// steps (one lane walking a vector's elements) use this form; bulk passes,
// where the conversions overlap with other work, use fix56_cvt.
__device__ __forceinline__ unsigned long long fix56(float acc) {
  const unsigned int u = __float_as_uint(acc);
  const int e = static_cast<int>(u >> 23);  // acc >= +0: no sign bit
  const unsigned int m = (u & 0x7fffffu) | 0x800000u;
  if (e >= 94) return static_cast<unsigned long long>(m) << (e - 94);
  const int sh = 94 - e;                    // 2^56 * acc < 0.5 when sh >= 25
  if (sh >= 25) return 0ull;
  const unsigned int q = m >> sh;
  const unsigned int rem = m & ((1u << sh) - 1u), half = 1u << (sh - 1);
  return q + ((rem > half || (rem == half && (q & 1u))) ? 1u : 0u);
}

__device__ __forceinline__ unsigned long long fix56_cvt(float acc) {
  return __float2ull_rn(__fmul_rn(acc, 72057594037927936.0f));  // 2^56 * acc is exact
}

// The draw's threshold floor(u * S), exactly, for u in [0, 1): u = m * 2^(e -
// 150), so u * S = (m * S) >> (150 - e) with the 88-bit product m * S formed
// in two 64-bit halves.  u <= 0 or NaN gives 0, u >= 1 gives S - 1.
__device__ __forceinline__ unsigned long long draw_threshold(float u, unsigned long long S) {
  if (!(u > 0.f)) return 0ull;
  if (!(u < 1.f)) return S - 1;
  const unsigned int b = __float_as_uint(u);
  const int e = static_cast<int>(b >> 23);
  if (e == 0) return 0ull;                  // subnormal u: u * S < 1
  const unsigned long long m = (b & 0x7fffffu) | 0x800000u;
  const int sh = 150 - e;                   // >= 24 since u < 1
  const unsigned long long lo = m * S, hi = __umul64hi(m, S);
  if (sh >= 64) return sh >= 128 ? 0ull : hi >> (sh - 64);
  return (lo >> sh) | (hi << (64 - sh));
}

// Whether the threshold lies within 1e-6 * S of either end [lo, hi) of the
// chosen element's step of the fixed-point CDF.
__device__ __forceinline__ bool near_step(unsigned long long theta, unsigned long long lo,
                                          unsigned long long hi, unsigned long long S) {
  const unsigned long long band = __umul64hi(S, 18446744073710ull);  // 1e-6 * 2^64
  const unsigned long long dl = theta >= lo ? theta - lo : lo - theta;
  const unsigned long long dh = hi >= theta ? hi - theta : theta - hi;
  return dl < band || dh < band;
}

// The residual weights r_k = max(0, p_k - q_k) (or p_k when `residual` is
// false) of one vector and the vector's fixed-point mass round(2^56 * sum r).
// The fp32 sum runs in element order with explicitly rounded operations, so
// every recomputation is bit-identical and integer sums of masses agree
// exactly in any order.  kInt: round with fix56 (latency-bound callers).
template <int VEC, bool kInt = false>
__device__ __forceinline__ unsigned long long vec_weight(const float (&xt)[VEC],
                                                         const float (&xd)[VEC], float Mt,
                                                         float invZt, float Md, float invZd,
                                                         float s, bool residual,
                                                         float (&r)[VEC]) {
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const float pt = __fmul_rn(ex2(__fmul_rn(__fsub_rn(xt[k], Mt), s)), invZt);
    float rk = pt;
    if (residual) {
      const float qd = __fmul_rn(ex2(__fmul_rn(__fsub_rn(xd[k], Md), s)), invZd);
      rk = fmaxf(0.f, __fsub_rn(pt, qd));
    }
    r[k] = rk;
    acc = __fadd_rn(acc, rk);
  }
  return kInt ? fix56(acc) : fix56_cvt(acc);
}

// The same weights with the normalisers kept relative to scaled offsets
// MSt = round(Mt * s), MSd = round(Md * s): p_k = 2^fma(x_k, s, -MSt) / Zt.
// One fused multiply-add per logit; the offset's rounding is common to every
// term of the row and to its normaliser, so it cancels.
template <int VEC, bool kInt = false>
__device__ __forceinline__ unsigned long long vec_weight_scaled(
    const float (&xt)[VEC], const float (&xd)[VEC], float MSt, float invZt, float MSd,
    float invZd, float s, bool residual, float (&r)[VEC]) {
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const float pt = __fmul_rn(ex2(__fmaf_rn(xt[k], s, -MSt)), invZt);
    float rk = pt;
    if (residual) {
      const float qd = __fmul_rn(ex2(__fmaf_rn(xd[k], s, -MSd)), invZd);
      rk = fmaxf(0.f, __fsub_rn(pt, qd));
    }
    r[k] = rk;
    acc = __fadd_rn(acc, rk);
  }
  return kInt ? fix56(acc) : fix56_cvt(acc);
}

// Merge two normalisers kept relative to scaled offsets (ms, z): the result
// is relative to the larger offset.  Subtracting two close offsets is exact.
__device__ __forceinline__ void merge_scaled(float& ms, float& z, float ms2, float z2) {
  const float mn = fmaxf(ms, ms2);
  if (mn == -INFINITY) {
    ms = mn;
    z = 0.f;
    return;
  }
  const float a = (ms == -INFINITY) ? 0.f : z * ex2(ms - mn);
  const float b = (ms2 == -INFINITY) ? 0.f : z2 * ex2(ms2 - mn);
  ms = mn;
  z = a + b;
}

// Warp-wide merge of (ms, z) normalisers: the warp's largest offset, one
// rescale per lane, then a butterfly sum (every lane ends with the same bits:
// each step adds the same two values on both partners).
__device__ __forceinline__ void warp_merge_scaled(float& ms, float& z) {
  float M = ms;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float zz = (ms == -INFINITY) ? 0.f : z * ex2(ms - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) zz += __shfl_xor_sync(0xffffffffu, zz, o);
  ms = M;
  z = (M == -INFINITY) ? 0.f : zz;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Exact warp-wide sum of fixed-point masses below 2^59 with three 32-bit
// reductions (redux.sync): the 22-bit limbs of 32 lanes sum below 2^27, so
// no limb carries out.
__device__ __forceinline__ unsigned long long warp_sum_mass(unsigned long long v) {
  const unsigned int l0 = static_cast<unsigned int>(v & 0x3fffffull);
  const unsigned int l1 = static_cast<unsigned int>((v >> 22) & 0x3fffffull);
  const unsigned int l2 = static_cast<unsigned int>(v >> 44);
  const unsigned long long s0 = __reduce_add_sync(0xffffffffu, l0);
  const unsigned long long s1 = __reduce_add_sync(0xffffffffu, l1);
  const unsigned long long s2 = __reduce_add_sync(0xffffffffu, l2);
  return s0 + (s1 << 22) + (s2 << 44);
}

// Inclusive prefix sum over the lanes of a warp.
__device__ __forceinline__ unsigned long long warp_scan_u64(unsigned long long v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned long long o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

// The element of a vector at which the fixed-point residual CDF passes
// `rem` (the draw's threshold minus the mass before the vector): the running
// fp32 sum of r in element order, rounded to fixed point exactly as the
// vector's mass w was, so the last element's value equals w > rem and the
// search always ends inside the vector.  c_prev / c_cur are the in-vector
// CDF values just below and at the chosen element.
template <int VEC>
__device__ __forceinline__ int pick_in_vector(const float (&r)[VEC], unsigned long long w,
                                              unsigned long long rem,
                                              unsigned long long& c_prev,
                                              unsigned long long& c_cur) {
  float acc = 0.f;
  int mstar = VEC - 1;
  c_prev = 0;
  c_cur = w;
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    acc = __fadd_rn(acc, r[k]);
    const unsigned long long cc = fix56(acc);
    if (cc > rem) {
      mstar = k;
      c_cur = cc;
      break;
    }
    c_prev = cc;
  }
  return mstar;
}

// 16-byte staged vectors: unpacking and a NaN-ignoring running maximum.
template <typename E>
struct Staged;

template <>
struct Staged<BF16> {
  static constexpr int kVec = 8;
  using Max = uint32_t;  // packed bf16x2 running maximum
  static __device__ __forceinline__ Max max_init() { return 0xff80ff80u; }  // (-inf, -inf)
  static __device__ __forceinline__ uint32_t bmax(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  static __device__ __forceinline__ void max_update(Max& m, const uint4 w) {
    m = bmax(m, bmax(bmax(w.x, w.y), bmax(w.z, w.w)));
  }
  static __device__ __forceinline__ float max_value(Max m) { return fmaxf(bf16_lo(m), bf16_hi(m)); }
  static __device__ __forceinline__ void unpack(const uint4 w, float (&x)[8]) {
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
  }
};

template <>
struct Staged<F32> {
  static constexpr int kVec = 4;
  using Max = float;
  static __device__ __forceinline__ Max max_init() { return -INFINITY; }
  static __device__ __forceinline__ void max_update(Max& m, const uint4 w) {
    m = fmaxf(fmaxf(m, fmaxf(__uint_as_float(w.x), __uint_as_float(w.y))),
              fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
  }
  static __device__ __forceinline__ float max_value(Max m) { return m; }
  static __device__ __forceinline__ void unpack(const uint4 w, float (&x)[4]) {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
};

// Online normaliser of one row relative to a scaled offset: the row's terms
// are 2^(x*s - ms), summed in z.
struct RowAcc {
  float ms, z;
};

// Packed fp32 pair arithmetic (two lanes per instruction, each rounded as the
// scalar operation would be).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\t"
      "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\tmov.b64 pc, {%6, %7};\n\t"
      "fma.rn.f32x2 pd, pa, pb, pc;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
      "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
      "add.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// The VEC elements of a 16-byte vector as VEC/2 fp32 pairs, in element order.
template <typename E>
__device__ __forceinline__ void unpack_pairs(const uint4 w, float2 (&x)[Staged<E>::kVec / 2]) {
  if constexpr (Staged<E>::kVec == 8) {
    x[0] = make_float2(bf16_lo(w.x), bf16_hi(w.x));
    x[1] = make_float2(bf16_lo(w.y), bf16_hi(w.y));
    x[2] = make_float2(bf16_lo(w.z), bf16_hi(w.z));
    x[3] = make_float2(bf16_lo(w.w), bf16_hi(w.w));
  } else {
    x[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
    x[1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
  }
}

// Fold up to two 16-byte vectors held in registers into a row accumulator
// without branches (so independent rows of a stage interleave): the new
// offset is the larger of the old one and the vectors' packed maximum, the
// old sum is rescaled by 2^(old - new) (exactly 1 when unchanged), and each
// logit adds 2^(x*s - new), summed as a tree.  The FFMAs and the tree's adds
// run on fp32 pairs (same roundings, same order as the scalar form).  An
// accumulator that has seen no finite logit stays at (-inf, 0).  kFull: both
// vectors are valid (nvalid == 2), so there are no per-element selects.
template <typename E, bool kFull>
__device__ __forceinline__ void acc_vectors_impl(RowAcc& A, const uint4 (&w)[2], int nvalid, float s) {
  constexpr int VEC = Staged<E>::kVec;
  constexpr int NP = VEC;  // pairs in two vectors
  typename Staged<E>::Max pm = Staged<E>::max_init();
  if (kFull || nvalid > 0) Staged<E>::max_update(pm, w[0]);
  if (kFull || nvalid > 1) Staged<E>::max_update(pm, w[1]);
  const float nm = fmaxf(A.ms, Staged<E>::max_value(pm) * s);
  const float f = (A.ms == nm) ? 1.f : ex2(A.ms - nm);
  const float2 s2 = make_float2(s, s), nm2 = make_float2(-nm, -nm);
  float2 e[NP];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
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
template <typename E>
__device__ __forceinline__ void acc_vectors(RowAcc& A, const uint4 (&w)[2], int nvalid, float s) {
  acc_vectors_impl<E, false>(A, w, nvalid, s);
}
template <typename E>
__device__ __forceinline__ void acc_vectors_full(RowAcc& A, const uint4 (&w)[2], float s) {
  acc_vectors_impl<E, true>(A, w, 2, s);
}

// One element of a staged slice.
template <typename E>
__device__ __forceinline__ float staged_elem(const uint4* slice, int j) {
  if constexpr (Staged<E>::kVec == 8)
    return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(slice)[j]) << 16);
  else
    return reinterpret_cast<const float*>(slice)[j];
}

// Candidate slot of row (b, i): the token in the low 31 bits, bit 31 set
// when the draw was within the boundary band of a CDF step.
__device__ __forceinline__ volatile int32_t* candidate_slot(const VerifyArgs& a, int b, int i) {
  return reinterpret_cast<volatile int32_t*>(static_cast<RowSlot*>(a.slots) +
                                             static_cast<size_t>(b) * (a.K + 1) + i);
}

// Counts one finished row of sequence b and, for the last of its K+1 rows,
// finalises the sequence with the whole calling warp: n is the lowest
// rejected position (K if none), the outputs are x_0..x_{n-1}, the candidate
// of row n, then -1, and the sequence's workspace goes back to zero.  All 32
// lanes of one warp must call this; lane 0 has already written the row's
// candidate (if any) before the call.
__device__ __forceinline__ void warp_arrive_and_finalize(const VerifyArgs& a, int b) {
  const int lane = threadIdx.x & 31;
  const int K = a.K, K1 = K + 1;
  // (debug builds) the sequence and its K+1 candidate slots lie in the batch
  // and the workspace
  if (!(SPEC_IN(b, a.B, a.status) &&
        SPEC_IN((static_cast<long long>(b) + 1) * K1 - 1, a.ws_units, a.status)))
    return;
  int last = 0;
  if (lane == 0) last = arrive_last(a.seq, b, static_cast<unsigned int>(K1)) ? 1 : 0;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();  // every lane reads what the other rows published
  __syncwarp();
  SeqState* st = a.seq + b;
  const unsigned long long mask = *reinterpret_cast<volatile unsigned long long*>(&st->reject_mask);
  const unsigned long long near = *reinterpret_cast<volatile unsigned long long*>(&st->near_mask);
  const int n = mask ? (__ffsll(static_cast<long long>(mask)) - 1) : K;
  const int32_t c = *candidate_slot(a, b, n);
  const int32_t* x = a.tokens + static_cast<size_t>(b) * K;
  int32_t* out = a.out_tokens + static_cast<size_t>(b) * K1;
  for (int j = lane; j < K1; j += 32)
    out[j] = (j < n) ? min(max(x[j], 0), a.V - 1) : (j == n ? (c & 0x7fffffff) : -1);
  __syncwarp();
  for (int j = lane; j < K1; j += 32) *candidate_slot(a, b, j) = 0;
  if (lane == 0) {
    if (a.accepted_len) a.accepted_len[b] = n;
    if (a.flags) {
      const unsigned long long evaluated = (n >= 63) ? ~0ull : ((2ull << n) - 1ull);
      a.flags[b] = ((near & evaluated) ? kFlagRatio : 0u) | ((c < 0) ? kFlagCdf : 0u);
    }
    st->reject_mask = 0ull;
    st->near_mask = 0ull;
    st->arrivals = 0u;
  }
}

}  // namespace specv
