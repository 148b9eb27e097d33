// spec_verify_greedy_noalloc: spec_verify_greedy with the library's own
// built-in device scratch instead of a caller-provided workspace.
//
// The scratch is one file-scope device array of kStaticScratchBytes. Its
// device address is looked up once per device with cudaGetSymbolAddress (the
// first call on a device does that setup, which may load the module) and
// cached; every call then hands that address to spec_verify_greedy as its
// workspace. Nothing is allocated: no cudaMalloc, no cudaFree, no library
// routine that allocates. Of the scratch, the header, row counters and work
// queue must start at zero for every launch; spec_verify_greedy clears them
// itself with cudaMemsetAsync on the caller's stream, so no state carries
// over between calls.
//
// All calls on one device share the one scratch: two calls whose launches
// can overlap on the device (different streams without ordering, several
// host threads) race on it and produce wrong results. Callers must order
// them, e.g. issue them on one stream.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/specverify.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_scratch[kStaticScratchBytes];

void* g_scratch_ptr[kMaxDevices];  // per-device address, set on first use

}  // namespace

extern "C" {

size_t spec_verify_greedy_noalloc_max_bytes(void) { return kStaticScratchBytes; }

int spec_verify_greedy_noalloc(const void* target_logits, const int32_t* draft_tokens, int B,
                               int K, int V, int32_t* out_tokens, int32_t* out_num_accepted,
                               void* stream, int dtype, int32_t* err_flag) {
  const size_t need = spec_verify_workspace_bytes(B, K, V, dtype);
  if (need == 0) {
    // arguments spec_verify_greedy rejects: let it report why
    return spec_verify_greedy(target_logits, draft_tokens, B, K, V, out_tokens, out_num_accepted,
                              stream, dtype, err_flag, nullptr, 0, nullptr);
  }
  if (need > kStaticScratchBytes) return SPEC_ENOTSUP;  // larger than the built-in scratch
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ECUDA;
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return SPEC_ECUDA;
    g_scratch_ptr[dev] = p;
  }
  return spec_verify_greedy(target_logits, draft_tokens, B, K, V, out_tokens, out_num_accepted,
                            stream, dtype, err_flag, g_scratch_ptr[dev], kStaticScratchBytes,
                            nullptr);
}

}  // extern "C"
