// Host-side launch descriptors shared by the C-ABI layer (api.cu) and the
// kernel translation units. Plain structs of pointers and sizes.
#pragma once
#include <cstdint>

namespace sv {

// Bound on the relative error of ex2.approx.ftz.f32 for arguments in
// [-126, 127], used by the certification of the fp32 fast path (the raw bonus
// draw's arguments reach up to 100). An exhaustive sweep of every fp32
// argument in [-126, 1] against an fp64 reference on GB300 measured a maximum
// of 1.4584e-7; the bound adds a 10% margin, and the GPU tests re-measure
// the whole range [-126, 127] against it.
constexpr double kEx2RelErrBound = 1.6e-7;

struct SampleLaunch {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const float* uniforms;
  float temperature;
  int B, K, V, dtype;
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* err;
  int32_t* row_info;
  float* q_at_d;
  float* p_at_d;
  void* stream;
  void* workspace;
  unsigned long long* counters;
  const float* thr_t;  // optional [B, K + 1] target-row logit thresholds
  const float* thr_d;  // optional [B, K] draft-row logit thresholds
};

struct GreedyLaunch {
  const void* target;
  const int32_t* tokens;
  int B, K, V, dtype;
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* err;
  void* stream;
  void* workspace;
  unsigned long long* counters;
  const int32_t* parents;  // tree mode: [B, K] node parents; null for a chain
  int32_t* out_slots;      // tree mode: [B, K + 1]
};

struct KvLaunch {
  int32_t* block_table;
  int32_t* seq_lens;
  const int32_t* num_accepted;
  int32_t* prov_blocks;
  void* kv_pool;
  int num_blocks, num_layers, num_kv_heads, head_dim, elem_bytes, block_size;
  int B, K, max_blocks, P;
  int32_t* free_stack;
  int32_t* free_top;
  int32_t* status;
  void* stream;
  const int32_t* slot_map;  // [B, K + 1] provisional slot of each kept position; null: identity
};

struct KvTruncLaunch {
  int32_t* block_table;
  int32_t* seq_lens;
  const int32_t* num_accepted;  // null: evict the provisional slots
  int num_blocks, block_size, B, K, max_blocks;
  int32_t* free_stack;
  int32_t* free_top;
  int32_t* status;
  void* stream;
};

struct FilterLaunch {
  const void* logits;
  int R, V, dtype, top_k;
  float temperature, top_p;
  float* out;
  int32_t* err;
  void* stream;
};

int launch_verify_sample(const SampleLaunch& s);
int launch_filter(const FilterLaunch& f);
size_t sample_workspace_bytes(int B, int K, int V, int dtype);
size_t greedy_workspace_bytes(int B, int K, int V, int dtype);
int launch_verify_greedy(const GreedyLaunch& g);
int launch_kv_commit(const KvLaunch& k);
int launch_kv_truncate(const KvTruncLaunch& k);

}  // namespace sv
