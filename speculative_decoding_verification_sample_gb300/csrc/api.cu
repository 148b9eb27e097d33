// C-ABI entry points: host-side argument validation, then asynchronous launch
// on the caller's stream. No allocation, no synchronisation.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/specverify.h"
#include "launch.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(int dtype) { return dtype == SPEC_BF16 ? 2 : (dtype == SPEC_F32 ? 4 : 0); }

}  // namespace

extern "C" {

int spec_version(void) { return 100; }

const char* spec_status_string(int status) {
  switch (status) {
    case SPEC_OK:
      return "ok";
    case SPEC_EINVAL:
      return "invalid argument";
    case SPEC_ECUDA:
      return "CUDA launch failed";
    case SPEC_ENOTSUP:
      return "unsupported configuration";
    default:
      return "unknown status";
  }
}

size_t spec_verify_workspace_bytes(int B, int K, int V, int dtype) {
  const int eb = elem_bytes(dtype);
  if (eb == 0 || B < 1 || K < 1 || K > 31 || V < 1 || (int64_t(V) * eb) % 16 != 0) return 0;
  const size_t a = sv::sample_workspace_bytes(B, K, V, dtype);
  const size_t g = sv::greedy_workspace_bytes(B, K, V, dtype);
  return a > g ? a : g;
}

static int check_workspace(void* ws, size_t bytes, int B, int K, int V, int dtype) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SPEC_EINVAL;
  if (bytes < spec_verify_workspace_bytes(B, K, V, dtype)) return SPEC_EINVAL;
  return SPEC_OK;
}

int spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B, int K,
                       int V, int32_t* out_tokens, int32_t* out_num_accepted, void* stream,
                       int dtype, int32_t* err_flag, void* workspace, size_t workspace_bytes,
                       uint64_t* accept_counters) {
  const int eb = elem_bytes(dtype);
  if (!target_logits || !draft_tokens || !out_tokens || !out_num_accepted) return SPEC_EINVAL;
  if (eb == 0 || B < 1 || K < 1 || K > 31 || V < 1) return SPEC_EINVAL;
  if (!aligned16(target_logits)) return SPEC_EINVAL;
  if ((int64_t(V) * eb) % 16 != 0) return SPEC_ENOTSUP;
  if (int64_t(B) * (V / (16 / eb)) > INT32_MAX) return SPEC_EINVAL;
  if (check_workspace(workspace, workspace_bytes, B, K, V, dtype) != SPEC_OK) return SPEC_EINVAL;
  sv::GreedyLaunch g{target_logits, draft_tokens, B, K, V, dtype, out_tokens, out_num_accepted,
                     err_flag, stream, workspace,
                     reinterpret_cast<unsigned long long*>(accept_counters), nullptr, nullptr};
  return sv::launch_verify_greedy(g);
}

int spec_verify_tree_greedy(const void* target_logits, const int32_t* tree_parents,
                            const int32_t* tree_tokens, int B, int N, int V, int32_t* out_tokens,
                            int32_t* out_num_accepted, int32_t* out_slots, void* stream,
                            int dtype, int32_t* err_flag, void* workspace,
                            size_t workspace_bytes) {
  const int eb = elem_bytes(dtype);
  if (!target_logits || !tree_parents || !tree_tokens || !out_tokens || !out_num_accepted)
    return SPEC_EINVAL;
  if (eb == 0 || B < 1 || N < 1 || N > 31 || V < 1) return SPEC_EINVAL;
  if (!aligned16(target_logits)) return SPEC_EINVAL;
  if ((int64_t(V) * eb) % 16 != 0) return SPEC_ENOTSUP;
  if (int64_t(B) * (V / (16 / eb)) > INT32_MAX) return SPEC_EINVAL;
  if (check_workspace(workspace, workspace_bytes, B, N, V, dtype) != SPEC_OK) return SPEC_EINVAL;
  sv::GreedyLaunch g{target_logits, tree_tokens, B, N, V, dtype, out_tokens, out_num_accepted,
                     err_flag, stream, workspace, nullptr, tree_parents, out_slots};
  return sv::launch_verify_greedy(g);
}

int spec_verify_sample(const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, const float* uniforms, float temperature,
                       int B, int K, int V, int32_t* out_tokens, int32_t* out_num_accepted,
                       void* stream, int dtype, int32_t* err_flag, int32_t* row_info,
                       float* q_at_d, float* p_at_d, void* workspace, size_t workspace_bytes,
                       uint64_t* accept_counters, const float* target_threshold,
                       const float* draft_threshold) {
  if (std::isnan(temperature) || temperature < 0.0f || std::isinf(temperature)) return SPEC_EINVAL;
  if (temperature == 0.0f) {
    const int st = spec_verify_greedy(target_logits, draft_tokens, B, K, V, out_tokens,
                                      out_num_accepted, stream, dtype, err_flag, workspace,
                                      workspace_bytes, accept_counters);
    if (st == SPEC_OK && row_info)
      if (cudaMemsetAsync(row_info, 0, size_t(B) * sizeof(int32_t),
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SPEC_ECUDA;
    return st;
  }
  const int eb = elem_bytes(dtype);
  if (!target_logits || !draft_logits || !draft_tokens || !uniforms || !out_tokens ||
      !out_num_accepted)
    return SPEC_EINVAL;
  if ((q_at_d == nullptr) != (p_at_d == nullptr)) return SPEC_EINVAL;
  if (eb == 0 || B < 1 || K < 1 || K > 31 || V < 1) return SPEC_EINVAL;
  if (!aligned16(target_logits) || !aligned16(draft_logits)) return SPEC_EINVAL;
  if ((int64_t(V) * eb) % 16 != 0) return SPEC_ENOTSUP;
  if (int64_t(B) * (V / (16 / eb)) > INT32_MAX) return SPEC_EINVAL;
  if (check_workspace(workspace, workspace_bytes, B, K, V, dtype) != SPEC_OK) return SPEC_EINVAL;
  sv::SampleLaunch s{target_logits, draft_logits, draft_tokens, uniforms, temperature, B, K, V,
                     dtype, out_tokens, out_num_accepted, err_flag, row_info, q_at_d, p_at_d,
                     stream, workspace, reinterpret_cast<unsigned long long*>(accept_counters),
                     target_threshold, draft_threshold};
  return sv::launch_verify_sample(s);
}

int spec_filter_thresholds(const void* logits, int R, int V, int dtype, float temperature,
                           int top_k, float top_p, float* out_threshold, void* stream,
                           int32_t* err_flag) {
  const int eb = elem_bytes(dtype);
  if (!logits || !out_threshold) return SPEC_EINVAL;
  if (eb == 0 || R < 1 || V < 1 || top_k < 0) return SPEC_EINVAL;
  if (!(top_p > 0.0f) || top_p > 1.0f) return SPEC_EINVAL;
  if (std::isnan(temperature) || !(temperature > 0.0f) || std::isinf(temperature)) return SPEC_EINVAL;
  if (!aligned16(logits)) return SPEC_EINVAL;
  if ((int64_t(V) * eb) % 16 != 0) return SPEC_ENOTSUP;
  if (V > (1 << 24)) return SPEC_ENOTSUP;
  sv::FilterLaunch f{logits, R, V, dtype, top_k, temperature, top_p, out_threshold, err_flag,
                     stream};
  return sv::launch_filter(f);
}

int kv_commit_rollback(int32_t* block_table, int32_t* seq_lens, const int32_t* num_accepted,
                       int32_t* prov_blocks, void* kv_pool, int num_blocks, int num_layers,
                       int num_kv_heads, int head_dim, int kv_elem_bytes, int block_size, int B,
                       int K, int max_blocks, int P, int32_t* free_stack, int32_t* free_top,
                       int32_t* status, void* stream, const int32_t* slot_map) {
  if (!block_table || !seq_lens || !num_accepted || !prov_blocks || !kv_pool || !free_stack ||
      !free_top || !status)
    return SPEC_EINVAL;
  if (num_blocks < 1 || num_layers < 1 || num_kv_heads < 1 || head_dim < 1 || kv_elem_bytes < 1 ||
      block_size < 1 || B < 1 || K < 0 || K > 31 || max_blocks < 1 || P < 1 || P > 512)
    return SPEC_EINVAL;
  const int64_t slot = int64_t(num_kv_heads) * head_dim * kv_elem_bytes;
  if (slot % 16 != 0 || !aligned16(kv_pool)) return SPEC_ENOTSUP;
  sv::KvLaunch k{block_table, seq_lens, num_accepted, prov_blocks, kv_pool, num_blocks,
                 num_layers,  num_kv_heads, head_dim, kv_elem_bytes, block_size, B, K,
                 max_blocks,  P, free_stack, free_top, status, stream, slot_map};
  return sv::launch_kv_commit(k);
}

static int kv_truncate(int32_t* block_table, int32_t* seq_lens, const int32_t* num_accepted,
                       int num_blocks, int block_size, int B, int K, int max_blocks,
                       int32_t* free_stack, int32_t* free_top, int32_t* status, void* stream) {
  if (!block_table || !seq_lens || !free_stack || !free_top || !status) return SPEC_EINVAL;
  if (num_blocks < 1 || block_size < 1 || B < 1 || K < 0 || K > 31 || max_blocks < 1)
    return SPEC_EINVAL;
  sv::KvTruncLaunch k{block_table, seq_lens, num_accepted, num_blocks, block_size, B, K,
                      max_blocks, free_stack, free_top, status, stream};
  return sv::launch_kv_truncate(k);
}

int kv_commit_inplace(int32_t* block_table, int32_t* seq_lens, const int32_t* num_accepted,
                      int num_blocks, int block_size, int B, int K, int max_blocks,
                      int32_t* free_stack, int32_t* free_top, int32_t* status, void* stream) {
  if (!num_accepted) return SPEC_EINVAL;
  return kv_truncate(block_table, seq_lens, num_accepted, num_blocks, block_size, B, K,
                     max_blocks, free_stack, free_top, status, stream);
}

int kv_evict_provisional(int32_t* block_table, int32_t* seq_lens, int num_blocks,
                         int block_size, int B, int K, int max_blocks, int32_t* free_stack,
                         int32_t* free_top, int32_t* status, void* stream) {
  return kv_truncate(block_table, seq_lens, nullptr, num_blocks, block_size, B, K, max_blocks,
                     free_stack, free_top, status, stream);
}

}  // extern "C"
