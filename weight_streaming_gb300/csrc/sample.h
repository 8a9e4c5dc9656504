// Sampled acceptance over given logits (sample.cu): workspace carving and the launch.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace vp {

// Largest vocabulary (the workspace holds 32 candidates per 4096-wide chunk of every row).
constexpr int kSampleMaxV = 1 << 20;

struct SampleWs {
  int n_chunks;
  size_t cand, tok, prob, count, cnt, total;
};
SampleWs sample_ws_layout(int M, int V);

cudaError_t launch_sample_accept(const float* logits, int M, int V, float temperature, int top_k, float top_p,
                                 const int32_t* pending, const int32_t* draft_tokens, const float* draft_probs,
                                 const float* uniforms, int32_t* n_commit, int32_t* committed, void* ws,
                                 cudaStream_t s);

}  // namespace vp
