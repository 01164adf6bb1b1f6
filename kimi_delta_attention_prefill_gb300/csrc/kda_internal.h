// kda_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace kda {

constexpr int kHeadDim = 128;
constexpr int kChunk = 64;
constexpr int kMaxDecodeTokens = 4;

// Device-side error report: the first non-zero code wins.
__device__ __forceinline__ void report_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

cudaError_t launch_decode(const void* q, const void* k, const void* v, const float* g, const float* beta, float* S,
                          const int32_t* n_commit, float* o, int B, int n_tok, int H, int* status,
                          cudaStream_t stream);

struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* S_in;
  const int32_t* cu_seqlens;
  int n_seq;
  int64_t total_tokens;
  const int32_t* ckpt_off;
  const int32_t* ckpt_pos;
  int64_t n_ckpt;
  void* o;
  float* S_out;
  float* ckpts;
  int H;
  int n_segments;  // 0 = planner, k >= 1 forced
  void* workspace;
  size_t workspace_bytes;
  int* status;
  cudaStream_t stream;
};

// Workspace bytes for the segment split; 0 when it cannot be taken.
size_t prefill_workspace_bytes(int n_seq, int H, int64_t total_tokens, int n_segments, int num_sms);
cudaError_t launch_prefill(const PrefillArgs& a, int num_sms);

}  // namespace kda
