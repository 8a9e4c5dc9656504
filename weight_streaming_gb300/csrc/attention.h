// Verify attention over a BF16 KV cache (attention.cu): arguments, workspace carving, the launch.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace vp {

constexpr int kAttnPart = 1024;       // keys per partition at most (the pages' 32K-tier partition size)
constexpr int kAttnTargetCtas = 152;  // one CTA per SM fits (160 KB of shared memory): one wave on GB300

struct AttnArgs {
  const uint16_t* q;      // bf16 [M][Hq][256]
  const uint16_t* k_new;  // bf16 [M][Hkv][256]
  const uint16_t* v_new;
  uint16_t* k_cache;      // bf16 [L][Hkv][cap][256]
  uint16_t* v_cache;
  const int32_t* ctx;     // [L] cached positions per lane (device)
  const uint16_t* gate;   // bf16 [M][Hq][256] or null
  uint16_t* out;          // bf16 [M][Hq][256]
  int Hq, Hkv, cap, n_part, part_len;
  float* part_o;          // [L][Hkv][n_part][64][256] unnormalised partial outputs
  float* part_ml;         // [L][Hkv][n_part][64][2] (max in log2 units, sum)
  int* status;            // the workspace's status word: set when a lane's ctx is out of range
};

struct AttnWs {
  int n_part, part_len;
  size_t status, part_o, part_ml, total;
};
AttnWs attn_ws_layout(int M, int Hkv, int cap);

// status: the word a lane out of range is reported in (null: the workspace's own status word).
cudaError_t launch_attention_verify(AttnArgs a, int M, void* ws, cudaStream_t s, int* status = nullptr);

}  // namespace vp
