// spec_verify_static.cu -- the verify step for callers that cannot allocate
// device memory.
//
// spec_verify needs a caller-provided workspace.  Some callers have no way to
// provide one at the point where they verify: a host program that only holds
// the logits and output buffers handed to it by another runtime's memory
// pool (an inference server that reserves all device memory up front and
// forbids outside allocations), or a latency-critical decode loop where
// cudaMalloc / cudaFree are not allowed because they can synchronise the
// device and take unbounded time.  This entry point serves them from a
// fixed scratch array that lives in the library itself.
//
// The scratch is a file-scope __device__ array of SPEC_STATIC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address (on the host it is
// only a stand-in), so the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device.
#include <mutex>

#include "../../include/spec_verify.h"
#include "device_common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[SPEC_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
void* g_addr[kMaxDevices];
cudaError_t g_err[kMaxDevices];

// Device address of the scratch array on `device` (the current device).
cudaError_t scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_once[device], [device]() {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    g_addr[device] = (e == cudaSuccess) ? p : nullptr;
    g_err[device] = e;
  });
  *out = g_addr[device];
  return g_err[device];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The pointer and temperature checks of spec_verify, done here as well so
// that a call with bad arguments queues nothing (not even the clearing).
bool args_ok(const void* target, const void* draft, const int32_t* tokens, const float* uniforms,
             int K, int dtype, float temperature, int mode, const int32_t* acc,
             const int32_t* out) {
  const uintptr_t esz = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  const bool sample = mode != SPEC_MODE_GREEDY;
  if (!target || !aligned(target, esz)) return false;
  if (K > 0 && (!tokens || !aligned(tokens, 4))) return false;
  if (!acc || !aligned(acc, 4) || !out || !aligned(out, 4)) return false;
  if (sample) {
    if (K > 0 && (!draft || !aligned(draft, esz))) return false;
    if (!uniforms || !aligned(uniforms, 4)) return false;
    if (!(temperature > 0.f && temperature <= 3.4e38f)) return false;
  }
  return true;
}

}  // namespace

extern "C" {

SPEC_API spec_status_t spec_verify_static(const void* target_logits, const void* draft_logits,
                                          const int32_t* draft_tokens, const float* uniforms,
                                          int B, int K, int V, int dtype, float temperature,
                                          int mode, int32_t* accepted_len, int32_t* out_tokens,
                                          spec_stream_t stream) {
  const size_t need = spec_verify_workspace_size(B, K, V, dtype, mode);
  if (need == 0) {
    // an empty batch, or invalid sizes: the full argument check answers
    // (it returns before touching any workspace or launching anything)
    return spec_verify(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype,
                       temperature, mode, accepted_len, out_tokens, nullptr, 0, stream);
  }
  if (need > SPEC_STATIC_SCRATCH_BYTES) return SPEC_ERR_SCRATCH_LIMIT;
  if (!args_ok(target_logits, draft_logits, draft_tokens, uniforms, K, dtype, temperature, mode,
               accepted_len, out_tokens))
    return SPEC_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  void* scratch = nullptr;
  if (scratch_address(dev, &scratch) != cudaSuccess || scratch == nullptr) return SPEC_ERR_CUDA;
  // The array keeps whatever the previous call left; the kernels need the
  // part they use zero-filled, so clear it on this call's stream first.
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess) return SPEC_ERR_CUDA;
  return spec_verify(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype,
                     temperature, mode, accepted_len, out_tokens, scratch,
                     SPEC_STATIC_SCRATCH_BYTES, stream);
}

}  // extern "C"
