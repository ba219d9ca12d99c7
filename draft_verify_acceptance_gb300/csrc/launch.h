// launch.h -- internal host interface between the C ABI (spec_verify.cu)
// and the kernel translation units.  Not part of the public API.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

// Optional NVTX ranges around every entry point (build with -DSPEC_NVTX; the
// NVTX3 headers are header-only and cost nothing without a profiler).
#ifdef SPEC_NVTX
#include <nvtx3/nvToolsExt.h>
namespace specv {
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
}  // namespace specv
#define SPEC_RANGE(name) ::specv::NvtxRange spec_nvtx_range_(name)
#else
#define SPEC_RANGE(name) \
  do {                   \
  } while (0)
#endif

namespace specv {

struct SeqState;

// Everything a verify launch needs, already validated by the C ABI layer.
struct VerifyArgs {
  const void* target;          // [B, K+1, V]
  const void* draft;           // [B, K, V] (sampling, K > 0)
  const int32_t* tokens;       // [B, K]
  const float* uniforms;       // [B, K+1] (sampling)
  int B, K, V;
  bool bf16;                   // element type of both logit tensors
  bool vec;                    // rows are 16-byte aligned: 16-byte vector loads
  float scale;                 // log2(e) / T (sampling)
  int32_t* accepted_len;       // [B] (null: not written; the draft sampler)
  int32_t* out_tokens;         // [B, K+1]
  float* p_at;                 // [B, K] or null
  float* q_at;                 // [B, K] or null
  uint32_t* flags;             // [B] or null
  int32_t* status;             // device status word or null
  SeqState* seq;               // workspace: [B]
  void* slots;                 // workspace: [B*(K+1)] RowSlot (greedy, streaming sampler)
  void* partials;              // workspace: Partial per work unit (fused sampler); same
                               // region as `slots`
  void* ctl;                   // workspace: FusedCtl (work counters)
  long long ws_units = 0;      // 16-byte slots in the `slots` / `partials` region (index checks
                               // of debug builds)
  bool early_exit = false;     // sampling: verify position 0 first (SPEC_MODE_SAMPLE_EARLY_EXIT)
  float* p_emit = nullptr;     // [B] or null: p_n of the token emitted at position n
                               // (fused and two-kernel samplers; the draft sampler's q(x))
  // Longest a kernel waits, without progress, on work of other warps or
  // thread blocks before it gives up and reports SPEC_DEVICE_WAIT_TIMEOUT.
  unsigned long long wait_ns = 2000000000ull;
};

// Per-device facts gathered once.
struct DeviceInfo {
  int sm_count = 0;
  int greedy_ctas_per_sm = 0;  // occupancy of the greedy kernel
  int stream_ctas_per_sm = 0;  // occupancy of the two-kernel sampler's streaming pass
  // clusters of the two-kernel sampler's second kernel that fit at once:
  // [256, 512, 1024 threads][cluster size 1, 2, 4, 8]
  int decide_clusters[3][4] = {};
};

cudaError_t device_info(int device, DeviceInfo* out);

// Launch configuration choices, exposed so the host logic can be tested.
int greedy_segments(long long rows, long long nvec, int sm_count, int ctas_per_sm);
int sample_cluster_size(long long V, int elem_bytes);
long long sample_tiles(long long nvec, int cluster);

cudaError_t launch_greedy(const VerifyArgs& a, const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_sample(const VerifyArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// The fused sampling kernel (16-byte aligned rows of at most kFusedMaxVec
// vectors: one draw segment); launch_sample dispatches to it.
constexpr long long kFusedMaxVec = 4096;
cudaError_t sample_fused_prepare();
cudaError_t launch_sample_fused(const VerifyArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// Small batches: one CTA per sequence with its K+1 target rows and K draft
// rows staged in shared memory (at most kSeqMaxBytes of them); no workspace.
constexpr int kSeqMaxBytes = 192 * 1024;
long long seq_sample_bytes(int K, long long nvec);
cudaError_t seq_sample_prepare();
cudaError_t launch_sample_seq(const VerifyArgs& a, cudaStream_t stream);

// The two-kernel sampler (normaliser stream, then decide and draw with one
// cluster per sequence) for rows whose draw spans several draw segments.
int sample_2p_cluster(long long nvec);
cudaError_t sample_2p_prepare(DeviceInfo* d);
cudaError_t launch_sample_2p(const VerifyArgs& a, const DeviceInfo& dev, int C,
                             cudaStream_t stream);
// Early-exit schedule (aligned rows, K >= 1): position 0 of every sequence,
// then -- only if some sequence accepted x_0 -- the full two-kernel sampler.
cudaError_t launch_sample_early_exit(const VerifyArgs& a, const DeviceInfo& dev, int C,
                                     cudaStream_t stream);

// The drafter's sampling step: one cluster of C CTAs per row, the row staged
// in shared memory (rows of up to 8 * 96 KiB).
int row_sample_cluster(long long nvec);
cudaError_t row_sample_prepare();
cudaError_t launch_row_sample(const void* logits, const float* uniforms, int R, int V, bool bf16,
                              float scale, int32_t* tokens, float* q_at, int32_t* status, int C,
                              cudaStream_t stream);

// Speculative contrastive decoding: one cluster of C CTAs per row pair
// (target, amateur), both rows streamed once; L = T ln(alpha).
int scd_cluster(long long nvec);
cudaError_t scd_prepare();
cudaError_t launch_scd(const VerifyArgs& a, const void* amateur, double L, int C,
                       cudaStream_t stream);

// Speculative Rejection's cut: r_cut and the kept indices per prompt
// (j, g from alpha (N - 1) on the host).
cudaError_t launch_rejection_cut(const float* scores, int G, int N, int j, double g,
                                 double* r_cut, int32_t* n_accepted, int32_t* accepted,
                                 int32_t* status, cudaStream_t stream);

}  // namespace specv
