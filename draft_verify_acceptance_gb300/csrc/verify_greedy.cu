// verify_greedy.cu -- greedy (blockwise-parallel) verification on sm_103a.
//
// "Garden | Blockwise Parallel Decoding", sections 3.2 (Accept) and 3.5:
// the target's argmax g_i at each of the K+1 positions is compared with the
// draft token x_i; the longest matching prefix is kept and the target's own
// token g_n is emitted at the first mismatch n (or at K when all match).
//
// Design: the [B*(K+1), V] logit rows are streamed once from HBM with 16-byte
// non-allocating loads, the next batch in flight while the current one is
// reduced.  Each row is split into S segments, one CTA each, so that the
// whole grid is resident in about one wave.  A thread keeps the first 16-byte
// vector holding its largest value (one NaN-propagating packed max per
// vector, no per-element index bookkeeping) and finds the element inside it
// at the end; the CTA reduces to (max value, lowest index).
//   One CTA per row (S == 1, K + 1 <= 48): the CTA writes g_i to its output
//   slot and adds (1 << 48 | mismatch bit i) to its sequence's word with one
//   acquire-release atomic; the CTA that completes the count knows n from the
//   mismatch bits and only overwrites the padding and writes n.
//   Several CTAs per row: each folds its result into the row's packed 64-bit
//   key with one atomicMax and counts itself on the sequence; the last CTA
//   loads the K+1 keys, compares them with the draft tokens and writes the
//   outputs.
// Either way no CTA waits, and the workspace is put back to zero.
#include <cfloat>
#include <climits>

#include "device_common.cuh"
#include "launch.h"

namespace specv {

namespace {

// Total order on floats for atomicMax: larger float -> larger key; -0 == +0.
__device__ __forceinline__ unsigned int orderable(float f) {
  unsigned int u = __float_as_uint(__fadd_rn(f, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Larger key wins: higher value first, then the LOWER index.
__device__ __forceinline__ unsigned long long pack_key(float v, int idx) {
  return (static_cast<unsigned long long>(orderable(v)) << 32) |
         static_cast<unsigned long long>(0xffffffffu - static_cast<unsigned int>(idx));
}

__device__ __forceinline__ int key_index(unsigned long long key) {
  return static_cast<int>(0xffffffffu - static_cast<unsigned int>(key & 0xffffffffull));
}

// NaN-propagating maximum of a 16-byte vector, as fp32 (NaN if it holds a NaN).
template <typename E>
struct VecMax;
template <>
struct VecMax<BF16> {
  static constexpr uint32_t kNegInf = 0xff80ff80u;
  static __device__ __forceinline__ uint32_t mx(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  static __device__ __forceinline__ float of(const uint4 w) {
    uint32_t m = mx(mx(w.x, w.y), mx(w.z, w.w));
    m = mx(m, __byte_perm(m, 0u, 0x1032));  // both halves: the vector's maximum
    return bf16_hi(m);
  }
  static __device__ __forceinline__ void unpack(const uint4 w, float (&x)[8]) {
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
  }
};
template <>
struct VecMax<F32> {
  static constexpr uint32_t kNegInf = 0xff800000u;
  static __device__ __forceinline__ float mx(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
  }
  static __device__ __forceinline__ float of(const uint4 w) {
    return mx(mx(__uint_as_float(w.x), __uint_as_float(w.y)),
              mx(__uint_as_float(w.z), __uint_as_float(w.w)));
  }
  static __device__ __forceinline__ void unpack(const uint4 w, float (&x)[4]) {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
};

// Largest value of this thread's vectors v0 + tid + j*kThreads (< v1) and the
// lowest index holding it; a vector with a NaN is skipped (and flagged).
// Vector indices within a row fit in int (V <= 2^22).
template <typename E, int VEC, int U>
__device__ __forceinline__ void thread_argmax_vec(const uint4* row, int v0, int v1,
                                                 float& best, int& bidx, bool& bad) {
  constexpr uint32_t ni = VecMax<E>::kNegInf;
  constexpr int kStep = kThreads * U;
  const int tid = threadIdx.x;
  int bv = -1;
  uint4 bw = make_uint4(ni, ni, ni, ni);
  uint4 cur[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int vv = v0 + tid + u * kThreads;
    cur[u] = vv < v1 ? ld_stream_v4(row + vv) : make_uint4(ni, ni, ni, ni);
  }
  for (int v = v0 + tid; v < v1; v += kStep) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      // reduce vector u of this batch, then put the next batch's vector u in
      // flight in its place (the loads of a batch overlap the reduction)
      const float f = VecMax<E>::of(cur[u]);
      bad |= !(f <= FLT_MAX);  // NaN or +inf
      if (f > best) {
        best = f;
        bv = v + u * kThreads;
        bw = cur[u];
      }
      const int vv = v + kStep + u * kThreads;
      cur[u] = vv < v1 ? ld_stream_v4(row + vv) : make_uint4(ni, ni, ni, ni);
    }
  }
  if (bv >= 0) {
    float x[VEC];
    VecMax<E>::unpack(bw, x);
    int k = VEC - 1;
#pragma unroll
    for (int j = VEC - 1; j >= 0; --j)
      if (x[j] == best) k = j;
    bidx = bv * VEC + k;
  }
}

template <typename E, int VEC, int U>
__global__ void __launch_bounds__(kThreads, 4)  // <= 64 registers: four CTAs per SM
greedy_kernel(VerifyArgs a, int nvec, int S, DivU64 by_S, DivU64 by_K1, bool one_word) {
  // 32-bit index arithmetic (the grid fits int and nvec * S <= 2^22 * 64);
  // divisions by S and K + 1 as multiply-highs
  const int K1 = a.K + 1;
  const int row = static_cast<int>(by_S(blockIdx.x));
  const int seg = static_cast<int>(blockIdx.x) - row * S;
  const int v0 = static_cast<int>(by_S(static_cast<unsigned long long>(nvec) * seg));
  const int v1 = static_cast<int>(by_S(static_cast<unsigned long long>(nvec) * (seg + 1)));
  const char* base = static_cast<const char*>(a.target) +
                     static_cast<size_t>(row) * static_cast<size_t>(a.V) * E::kBytes;

  const int tid = threadIdx.x;
  const int b = static_cast<int>(by_K1(row));  // sequence, before the stream
  // the draft token this row is compared with, fetched while the row streams
  int xtok = 0;
  if (one_word && tid == 0) {
    const int pos = row - b * K1;
    if (pos < a.K) xtok = a.tokens[static_cast<size_t>(b) * a.K + pos];
  }

  float best = -INFINITY;
  int bidx = (v0 + tid < v1) ? (v0 + tid) * VEC : INT_MAX;
  bool bad = false;

  if constexpr (VEC > 1) {
    thread_argmax_vec<E, VEC, U>(reinterpret_cast<const uint4*>(base), v0, v1, best, bidx, bad);
  } else {
    for (int v = v0 + tid; v < v1; v += kThreads * U) {
      float x[U][VEC];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int vv = v + u * kThreads;
        if (vv < v1) {
          VecLoad<E, VEC>::load(base, vv, x[u]);
        } else {
#pragma unroll
          for (int k = 0; k < VEC; ++k) x[u][k] = -INFINITY;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
          const float e = x[u][k];
          bad |= !(e <= FLT_MAX);  // NaN or +inf
          if (e > best) {
            best = e;
            bidx = (v + u * kThreads) * VEC + k;
          }
        }
      }
    }
  }

  // block argmax (larger value, then lower index, wins): per warp, the
  // largest orderable value and then the lowest index holding it, two
  // redux.sync each; then the same over the kWarps warp results in warp 0
  const int warp = tid >> 5, lane = tid & 31;
  unsigned int ov = orderable(best);
  unsigned int oi = static_cast<unsigned int>(bidx);
  unsigned int m = __reduce_max_sync(0xffffffffu, ov);
  oi = __reduce_min_sync(0xffffffffu, ov == m ? oi : 0xffffffffu);
  __shared__ unsigned int s_v[kWarps], s_i[kWarps];
  if (lane == 0) {
    s_v[warp] = m;
    s_i[warp] = oi;
  }
  const int any_bad = __syncthreads_or(bad);
  if (warp != 0) return;
  ov = lane < kWarps ? s_v[lane] : 0u;
  oi = lane < kWarps ? s_i[lane] : 0xffffffffu;
  m = __reduce_max_sync(0xffffffffu, ov);
  oi = __reduce_min_sync(0xffffffffu, ov == m ? oi : 0xffffffffu);
  const unsigned long long key =
      (static_cast<unsigned long long>(m) << 32) | (0xffffffffu - oi);  // as pack_key

  if (one_word) {  // one CTA per row: g_i to its slot, one atomic on the sequence
    if (lane == 0) {
      const int pos = row - b * K1;
      bidx = key_index(key);
      int flags = any_bad ? kDataNonfiniteLogit : 0;
      bool mism = true;  // the bonus position always ends the prefix
      if (pos < a.K) {
        mism = xtok != bidx;
        if (xtok < 0 || xtok >= a.V) flags |= kDataTokenRange;
      }
      if (flags && a.status) atomicOr(a.status, flags);
      int32_t* out = a.out_tokens + static_cast<size_t>(b) * K1;
      if (!(SPEC_IN(b, a.B, a.status) && SPEC_IN(pos, K1, a.status))) return;
      out[pos] = bidx;  // x_i when it matches, g_n at the first mismatch
      const unsigned long long add = (1ull << 48) | (mism ? (1ull << pos) : 0ull);
      const unsigned long long now = atom_add_acq_rel_gpu(&a.seq[b].row_word, add) + add;
      if (static_cast<int>(now >> 48) == K1) {  // every row of the sequence is done
        const int n = __ffsll(static_cast<long long>(now & ((1ull << 48) - 1))) - 1;
        for (int i = n + 1; i < K1; ++i) out[i] = -1;
        a.accepted_len[b] = n;
        if (a.flags) a.flags[b] = 0;
        a.seq[b].row_word = 0ull;
      }
    }
    return;
  }

  // warp 0: the block's argmax into the row's key; the last CTA of the
  // sequence finalises it with the whole warp (all loads at once)
  unsigned int last = 0;
  if (lane == 0) {
    if (any_bad && a.status) atomicOr(a.status, kDataNonfiniteLogit);
    RowSlot* slots = static_cast<RowSlot*>(a.slots);
    if (SPEC_IN(row, a.ws_units, a.status) && SPEC_IN(b, a.B, a.status)) {
      if (S == 1) slots[row].value = key;
      else atomicMax(&slots[row].value, key);
      last = arrive_last(a.seq, b, static_cast<unsigned int>(K1) * static_cast<unsigned int>(S)) ? 1u : 0u;
    }
  }
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();  // every lane reads what the other CTAs published

  // last arrival for sequence b: longest matching prefix, outputs, reset.
  // Lane l holds positions l, 32 + l, 64 + l (K + 1 <= 65): all loads first.
  volatile RowSlot* vslots = static_cast<RowSlot*>(a.slots) + static_cast<size_t>(b) * K1;
  const int32_t* x = a.tokens + static_cast<size_t>(b) * a.K;
  int32_t* out = a.out_tokens + static_cast<size_t>(b) * K1;
  constexpr int kR = (64 + 1 + 31) / 32;
  int gk[kR], xt[kR];
  bool bad_tok = false;
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    const int i = r * 32 + lane;
    gk[r] = (i < K1) ? key_index(vslots[i].value) : 0;
    xt[r] = (i < a.K) ? x[i] : 0;
    bad_tok |= (i < a.K) && (xt[r] < 0 || xt[r] >= a.V);
  }
  int n = a.K;
#pragma unroll
  for (int r = 0; r < kR; ++r) {  // the first position whose draft token differs
    const int i = r * 32 + lane;
    const unsigned int mism = __ballot_sync(0xffffffffu, i < a.K && xt[r] != gk[r]);
    if (n == a.K && mism) n = r * 32 + __ffs(mism) - 1;
  }
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    const int i = r * 32 + lane;
    if (i < K1) {
      out[i] = (i < n) ? xt[r] : (i == n ? gk[r] : -1);
      vslots[i].value = 0ull;
    }
  }
  bad_tok = __any_sync(0xffffffffu, bad_tok);
  if (lane == 0) {
    a.accepted_len[b] = n;
    if (a.flags) a.flags[b] = 0;
    if (bad_tok && a.status) atomicOr(a.status, kDataTokenRange);
    a.seq[b].arrivals = 0u;
  }
}

// Sequences of at most this many rows keep their mismatch bits and row count
// in one 64-bit word (count in the top 16 bits).
constexpr int kOneWordRows = 48;

template <typename E, int VEC, int U>
cudaError_t launch_greedy_t(const VerifyArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  const long long nvec = a.V / VEC;
  const long long rows = static_cast<long long>(a.B) * (a.K + 1);
  const int S = greedy_segments(rows, nvec, dev.sm_count, dev.greedy_ctas_per_sm);
  const long long grid = rows * S;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  const bool one_word = S == 1 && a.K + 1 <= kOneWordRows;
  return cudaLaunchKernelEx(&cfg, greedy_kernel<E, VEC, U>, a, static_cast<int>(nvec), S,
                            DivU64::make(static_cast<unsigned long long>(S)),
                            DivU64::make(static_cast<unsigned long long>(a.K + 1)), one_word);
}

}  // namespace

// Segments per row: enough CTAs to fill every SM once (one resident wave),
// but never fewer than ~2 loads of 16 bytes per thread in a segment.
int greedy_segments(long long rows, long long nvec, int sm_count, int ctas_per_sm) {
  if (rows <= 0 || nvec <= 0) return 1;
  const long long slots = static_cast<long long>(sm_count > 0 ? sm_count : 1) *
                          (ctas_per_sm > 0 ? ctas_per_sm : 1);
  long long S = slots / rows;
  const long long max_s = nvec / (2LL * kThreads);
  if (S > max_s) S = max_s;
  if (S < 1) S = 1;
  if (S > 64) S = 64;
  return static_cast<int>(S);
}

cudaError_t greedy_occupancy(int* ctas_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm,
                                                       greedy_kernel<BF16, 8, 8>, kThreads, 0);
}

cudaError_t launch_greedy(const VerifyArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  if (a.bf16) {
    return a.vec ? launch_greedy_t<BF16, 8, 8>(a, dev, stream)
                 : launch_greedy_t<BF16, 1, 8>(a, dev, stream);
  }
  return a.vec ? launch_greedy_t<F32, 4, 8>(a, dev, stream)
               : launch_greedy_t<F32, 1, 8>(a, dev, stream);
}

}  // namespace specv
