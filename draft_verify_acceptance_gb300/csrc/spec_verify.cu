// spec_verify.cu -- the C ABI of libspecverify.so (declared in
// include/spec_verify.h): argument validation on the host, one-time per-
// device set-up, and dispatch to the greedy or sampling kernel.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/spec_verify.h"
#include "device_common.cuh"
#include "launch.h"
#include "launch_ee.h"


namespace specv {

cudaError_t greedy_occupancy(int* ctas_per_sm);
cudaError_t sample_prepare();

namespace {
constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
DeviceInfo g_info[kMaxDevices];
cudaError_t g_err[kMaxDevices];
}  // namespace

// Gathered once per device, with that device current (the caller's).
cudaError_t device_info(int device, DeviceInfo* out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_once[device], [device]() {
    DeviceInfo d;
    cudaError_t e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = greedy_occupancy(&d.greedy_ctas_per_sm);
    if (e == cudaSuccess) e = sample_prepare();
    if (e == cudaSuccess) e = sample_fused_prepare();
    if (e == cudaSuccess) e = seq_sample_prepare();
    if (e == cudaSuccess) e = sample_2p_prepare(&d);
    if (e == cudaSuccess) e = row_sample_prepare();
    if (e == cudaSuccess) e = sample_ee_prepare();
    if (e == cudaSuccess) e = scd_prepare();
    g_info[device] = d;
    g_err[device] = e;
  });
  *out = g_info[device];
  return g_err[device];
}

}  // namespace specv

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Bound on a kernel's waits for work of other warps or thread blocks
// (spec_set_wait_limit); read at every launch.
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

}  // namespace

extern "C" {

size_t spec_verify_workspace_size(int B, int K, int V, int dtype, int mode) {
  if (B < 0 || K < 0 || K > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return 0;
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return 0;
  if (mode != SPEC_MODE_SAMPLE && mode != SPEC_MODE_GREEDY && mode != SPEC_MODE_SAMPLE_EARLY_EXIT)
    return 0;
  return specv::workspace_bytes(B, K, V, dtype == SPEC_DTYPE_BF16 ? 2 : 4);
}

spec_status_t spec_verify_ex(const void* target_logits, const void* draft_logits,
                             const int32_t* draft_tokens, const float* uniforms, int B,
                             int K, int V, int dtype, float temperature, int mode,
                             int32_t* accepted_len, int32_t* out_tokens, void* workspace,
                             size_t workspace_bytes, spec_stream_t stream,
                             float* p_at_draft, float* q_at_draft, uint32_t* flags,
                             int32_t* device_status) {
  SPEC_RANGE("spec_verify_ex");
  // ---- sizes, enums ------------------------------------------------------
  if (B < 0 || K < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_INVALID_ARG;
  if (mode != SPEC_MODE_SAMPLE && mode != SPEC_MODE_GREEDY && mode != SPEC_MODE_SAMPLE_EARLY_EXIT)
    return SPEC_ERR_INVALID_ARG;
  if (K > SPEC_MAX_K || V > SPEC_MAX_V) return SPEC_ERR_UNSUPPORTED;
  const bool sample = mode != SPEC_MODE_GREEDY;
  if (sample && !(temperature > 0.f && std::isfinite(temperature))) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;

  // ---- pointers ----------------------------------------------------------
  const int esz = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  if (!target_logits || !aligned(target_logits, esz)) return SPEC_ERR_INVALID_ARG;
  if (K > 0 && (!draft_tokens || !aligned(draft_tokens, 4))) return SPEC_ERR_INVALID_ARG;
  if (!accepted_len || !aligned(accepted_len, 4)) return SPEC_ERR_INVALID_ARG;
  if (!out_tokens || !aligned(out_tokens, 4)) return SPEC_ERR_INVALID_ARG;
  if (sample) {
    if (K > 0 && (!draft_logits || !aligned(draft_logits, esz))) return SPEC_ERR_INVALID_ARG;
    if (!uniforms || !aligned(uniforms, 4)) return SPEC_ERR_INVALID_ARG;
  }
  if ((p_at_draft && !aligned(p_at_draft, 4)) || (q_at_draft && !aligned(q_at_draft, 4)) ||
      (flags && !aligned(flags, 4)) || (device_status && !aligned(device_status, 4)))
    return SPEC_ERR_INVALID_ARG;
  const size_t need = specv::workspace_bytes(B, K, V, esz);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return SPEC_ERR_INVALID_ARG;

  // ---- launch ------------------------------------------------------------
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  specv::DeviceInfo info;
  if (specv::device_info(dev, &info) != cudaSuccess) return SPEC_ERR_CUDA;

  specv::VerifyArgs a;
  a.target = target_logits;
  a.draft = (sample && K > 0) ? draft_logits : nullptr;
  a.tokens = draft_tokens;
  a.uniforms = sample ? uniforms : nullptr;
  a.B = B;
  a.K = K;
  a.V = V;
  a.bf16 = dtype == SPEC_DTYPE_BF16;
  const long long rowbytes = static_cast<long long>(V) * esz;
  a.vec = (rowbytes % 16 == 0) && aligned(target_logits, 16) && (!a.draft || aligned(a.draft, 16));
  a.scale = sample ? static_cast<float>(1.4426950408889634 / static_cast<double>(temperature)) : 0.f;
  a.accepted_len = accepted_len;
  a.out_tokens = out_tokens;
  a.p_at = sample ? p_at_draft : nullptr;
  a.q_at = sample ? q_at_draft : nullptr;
  a.flags = flags;
  a.status = device_status;
  const specv::WorkspaceLayout lay = specv::workspace_layout(B, K, V, esz);
  a.seq = reinterpret_cast<specv::SeqState*>(static_cast<char*>(workspace) + lay.seq);
  a.slots = static_cast<char*>(workspace) + lay.units;
  a.partials = static_cast<char*>(workspace) + lay.units;
  a.ctl = static_cast<char*>(workspace) + lay.ctl;
  a.ws_units = static_cast<long long>((lay.ctl - lay.units) / 16);
  a.early_exit = mode == SPEC_MODE_SAMPLE_EARLY_EXIT;
  a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);

  const long long rows = static_cast<long long>(B) * (K + 1);
  if (rows * specv::kMaxCluster > INT32_MAX) return SPEC_ERR_UNSUPPORTED;
  // aligned rows go to the fused or the two-kernel sampler; the streaming
  // sampler takes the rest
  const bool streaming = !a.vec || (rowbytes / 16 > specv::kFusedMaxVec &&
                                    specv::sample_2p_cluster(rowbytes / 16) == 0);
  if (sample && streaming) {  // limits of the streaming sampler
    const long long nvec = a.vec ? rowbytes / 16 : V;
    const int C = specv::sample_cluster_size(V, esz);
    if (specv::sample_tiles(nvec, C) > specv::kMaxTiles) return SPEC_ERR_UNSUPPORTED;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = sample ? specv::launch_sample(a, info, s) : specv::launch_greedy(a, info, s);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_verify(const void* target_logits, const void* draft_logits,
                          const int32_t* draft_tokens, const float* uniforms, int B, int K,
                          int V, int dtype, float temperature, int mode,
                          int32_t* accepted_len, int32_t* out_tokens, void* workspace,
                          size_t workspace_bytes, spec_stream_t stream) {
  return spec_verify_ex(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype,
                        temperature, mode, accepted_len, out_tokens, workspace,
                        workspace_bytes, stream, nullptr, nullptr, nullptr, nullptr);
}

spec_status_t spec_draft_sample(const void* logits, const float* uniforms, int R, int V, int dtype,
                                float temperature, int32_t* tokens, float* q_at, void* workspace,
                                size_t workspace_bytes, spec_stream_t stream,
                                int32_t* device_status) {
  SPEC_RANGE("spec_draft_sample");
  if (R < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_INVALID_ARG;
  if (V > SPEC_MAX_V) return SPEC_ERR_UNSUPPORTED;
  if (!(temperature > 0.f && std::isfinite(temperature))) return SPEC_ERR_INVALID_ARG;
  if (R == 0) return SPEC_OK;
  const int esz = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  if (!logits || !aligned(logits, esz)) return SPEC_ERR_INVALID_ARG;
  if (!uniforms || !aligned(uniforms, 4)) return SPEC_ERR_INVALID_ARG;
  if (!tokens || !aligned(tokens, 4)) return SPEC_ERR_INVALID_ARG;
  if ((q_at && !aligned(q_at, 4)) || (device_status && !aligned(device_status, 4)))
    return SPEC_ERR_INVALID_ARG;
  const size_t need = specv::workspace_bytes(R, 0, V, esz);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return SPEC_ERR_INVALID_ARG;
  const long long rowbytes = static_cast<long long>(V) * esz;
  if (rowbytes % 16 != 0 || !aligned(logits, 16)) return SPEC_ERR_UNSUPPORTED;
  if (static_cast<long long>(R) * specv::kMaxCluster > INT32_MAX) return SPEC_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  specv::DeviceInfo info;
  if (specv::device_info(dev, &info) != cudaSuccess) return SPEC_ERR_CUDA;

  const float scale = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  const int C = specv::row_sample_cluster(rowbytes / 16);
  if (C > 0) {  // rows that fit a cluster's shared memory: read once
    const cudaError_t e = specv::launch_row_sample(
        logits, uniforms, R, V, dtype == SPEC_DTYPE_BF16, scale, tokens, q_at, device_status, C,
        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
  }
  // longer rows: a verify of R sequences with K = 0, whose one draw is the
  // bonus draw from p_0 = softmax(row / T) with u[r]; p_emit is p_0 there
  specv::VerifyArgs a;
  a.target = logits;
  a.draft = nullptr;
  a.tokens = nullptr;
  a.uniforms = uniforms;
  a.B = R;
  a.K = 0;
  a.V = V;
  a.bf16 = dtype == SPEC_DTYPE_BF16;
  a.vec = true;
  a.scale = scale;
  a.accepted_len = nullptr;
  a.out_tokens = tokens;
  a.p_at = nullptr;
  a.q_at = nullptr;
  a.flags = nullptr;
  a.status = device_status;
  a.p_emit = q_at;
  a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  const specv::WorkspaceLayout lay = specv::workspace_layout(R, 0, V, esz);
  a.seq = reinterpret_cast<specv::SeqState*>(static_cast<char*>(workspace) + lay.seq);
  a.slots = static_cast<char*>(workspace) + lay.units;
  a.partials = static_cast<char*>(workspace) + lay.units;
  a.ctl = static_cast<char*>(workspace) + lay.ctl;
  a.ws_units = static_cast<long long>((lay.ctl - lay.units) / 16);
  const cudaError_t e = specv::launch_sample(a, info, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_verify_scd(const void* target_logits, const void* amateur_logits,
                              const int32_t* draft_tokens, const float* uniforms, int B, int K,
                              int V, int dtype, float temperature, double alpha,
                              int32_t* accepted_len, int32_t* out_tokens, void* workspace,
                              size_t workspace_bytes, spec_stream_t stream, float* p_at_draft,
                              float* q_at_draft, uint32_t* flags, int32_t* device_status) {
  SPEC_RANGE("spec_verify_scd");
  if (B < 0 || K < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_INVALID_ARG;
  if (!(temperature > 0.f && std::isfinite(temperature))) return SPEC_ERR_INVALID_ARG;
  if (!(alpha >= 0.0 && alpha <= 1.0)) return SPEC_ERR_INVALID_ARG;
  if (K > SPEC_MAX_K || V > SPEC_MAX_V) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  const int esz = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  if (!target_logits || !aligned(target_logits, esz)) return SPEC_ERR_INVALID_ARG;
  if (!amateur_logits || !aligned(amateur_logits, esz)) return SPEC_ERR_INVALID_ARG;
  if (K > 0 && (!draft_tokens || !aligned(draft_tokens, 4))) return SPEC_ERR_INVALID_ARG;
  if (!uniforms || !aligned(uniforms, 4)) return SPEC_ERR_INVALID_ARG;
  if (!accepted_len || !aligned(accepted_len, 4)) return SPEC_ERR_INVALID_ARG;
  if (!out_tokens || !aligned(out_tokens, 4)) return SPEC_ERR_INVALID_ARG;
  if ((p_at_draft && !aligned(p_at_draft, 4)) || (q_at_draft && !aligned(q_at_draft, 4)) ||
      (flags && !aligned(flags, 4)) || (device_status && !aligned(device_status, 4)))
    return SPEC_ERR_INVALID_ARG;
  const size_t need = specv::workspace_bytes(B, K, V, esz);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return SPEC_ERR_INVALID_ARG;
  const long long rowbytes = static_cast<long long>(V) * esz;
  if (rowbytes % 16 != 0 || !aligned(target_logits, 16) || !aligned(amateur_logits, 16))
    return SPEC_ERR_UNSUPPORTED;
  const int C = specv::scd_cluster(rowbytes / 16);
  if (C == 0) return SPEC_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * (K + 1) * C > INT32_MAX) return SPEC_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  specv::DeviceInfo info;
  if (specv::device_info(dev, &info) != cudaSuccess) return SPEC_ERR_CUDA;

  specv::VerifyArgs a;
  a.target = target_logits;
  a.draft = nullptr;
  a.tokens = draft_tokens;
  a.uniforms = uniforms;
  a.B = B;
  a.K = K;
  a.V = V;
  a.bf16 = dtype == SPEC_DTYPE_BF16;
  a.vec = true;
  a.scale = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  a.accepted_len = accepted_len;
  a.out_tokens = out_tokens;
  a.p_at = p_at_draft;
  a.q_at = q_at_draft;
  a.flags = flags;
  a.status = device_status;
  const specv::WorkspaceLayout lay = specv::workspace_layout(B, K, V, esz);
  a.seq = reinterpret_cast<specv::SeqState*>(static_cast<char*>(workspace) + lay.seq);
  a.slots = static_cast<char*>(workspace) + lay.units;
  a.partials = static_cast<char*>(workspace) + lay.units;
  a.ctl = static_cast<char*>(workspace) + lay.ctl;
  a.ws_units = static_cast<long long>((lay.ctl - lay.units) / 16);
  // the head's log-threshold T ln(alpha), in double (alpha = 0: no cut)
  const double L = alpha > 0.0 ? static_cast<double>(temperature) * std::log(alpha) : -INFINITY;
  const cudaError_t e =
      specv::launch_scd(a, amateur_logits, L, C, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_set_wait_limit(unsigned int microseconds) {
  g_wait_ns.store(microseconds == 0 ? kDefaultWaitNs : 1000ull * microseconds,
                  std::memory_order_relaxed);
  return SPEC_OK;
}

const char* spec_status_string(int status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported size";
    case SPEC_ERR_CUDA: return "CUDA error";
    case SPEC_ERR_SCRATCH_LIMIT: return "batch needs more scratch than the static no-allocation buffer holds";
    default: return "unknown status";
  }
}

}  // extern "C"
