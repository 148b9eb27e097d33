// spec_verify_greedy_noalloc: spec_verify_greedy with the library's own
// built-in device scratch instead of a caller-provided workspace.
//
// The scratch is one file-scope device array of kStaticScratchBytes; every
// GPU that loads the library holds it until the process exits. Host code
// cannot use the array's name as a device address, so every call looks the
// address up with cudaGetSymbolAddress on the current device and checks the
// result. The first call on a device may load the library's module there,
// so that first call should come before any stream capture. Looking the
// address up on every call (instead of caching it) keeps it right after a
// context is torn down and re-created, and leaves no shared host state for
// concurrent callers to race on. Nothing is allocated: no cudaMalloc, no
// cudaFree, no library routine that allocates. Of the scratch, the header,
// row counters and work queue must start at zero for every launch;
// spec_verify_greedy clears them itself with a small zeroing kernel on the
// caller's stream, so no state carries over between calls.
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

__device__ __align__(256) uint8_t g_scratch[kStaticScratchBytes];

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
  void* scratch = nullptr;  // the array's device address on the current device
  if (cudaGetSymbolAddress(&scratch, g_scratch) != cudaSuccess || scratch == nullptr)
    return SPEC_ECUDA;
  return spec_verify_greedy(target_logits, draft_tokens, B, K, V, out_tokens, out_num_accepted,
                            stream, dtype, err_flag, scratch, kStaticScratchBytes, nullptr);
}

}  // extern "C"
