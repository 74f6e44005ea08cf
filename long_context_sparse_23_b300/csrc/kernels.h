// Internal launch interface between the C ABI (csa_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace csa {

// ---- (1) compression -------------------------------------------------------
struct CompressArgs {
  const void* x[3];
  const void* g[3];
  void* out[3];
  int D[3];
  int n_streams;
  int B, T, m;
  int out_f32;
};
cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s);

// ---- (2) indexer scores ----------------------------------------------------
struct IndexerArgs {
  const void* q_idx;  // [B, Tq, H_I, d_I] bf16
  const void* k_idx;  // [B, N, d_I] bf16
  const float* w;     // [H_I]
  const int32_t* q_pos;
  float* scores;
  long long ld;
  int B, Tq, N, H_I, d_I, m;
  uint32_t* errw;
  long long budget;
};
// returns cudaErrorNotSupported for shapes outside the instantiated set
cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s);

// ---- (3) top-k --------------------------------------------------------------
struct TopkArgs {
  const float* scores;
  long long ld;
  const int32_t* q_pos;
  int B, Tq, N, m, k;
  int32_t* idx_out;
  float* score_out;
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s);
bool topk_supported(int N);

// ---- (4) attention ----------------------------------------------------------
struct AttendArgs {
  const void* q;
  const void* k_cmp;
  const void* v_cmp;
  const int32_t* idx;  // nullptr: HCA mode (every visible entry)
  const void* k_raw;
  const void* v_raw;
  const int32_t* raw_base;
  const int32_t* q_pos;
  int B, Tq, N, T_raw, H, d, k, W, m;
  float scale;
  void* out;
  int out_f32;
  float* lse;
  float* part;  // split partials (workspace), may be nullptr when nsplit == 1
  uint32_t* errw;
};
struct AttendPlan {
  int nsplit;
  int tiles_per_split;
  size_t part_bytes;
};
AttendPlan plan_attend(int Tq, long long nq, int n_keys_max, int H, int d);
cudaError_t launch_attend(const AttendArgs& a, const AttendPlan& plan, cudaStream_t s);

}  // namespace csa
