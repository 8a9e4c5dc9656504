// Launches of the mixer cores' producer and consumer steps (mixer.cu); each returns the launch's
// error.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace vp {

// The gates alpha[t][j] = exp(-exp(a_log[j]) softplus(a + dt_bias[j])), beta[t][j] = sigmoid(b) of
// a = bf16(RMSNorm(h_t)) . wa[j], b = ... . wb[j] (fp32 [M][n_v]); h bf16 [M][hidden], hidden % 8 == 0,
// hidden <= 8192, h / wa / wb 16-byte aligned.
cudaError_t launch_ab_gates(const uint16_t* h, int hidden, int M, float eps, const uint16_t* wa, const uint16_t* wb,
                            int n_v, const float* a_log, const float* dt_bias, float* alpha, float* beta,
                            cudaStream_t s);
// Short convolution + SiLU + Q / K L2 norm (q, k expanded to the n_v heads, v) bf16 [M][n_v][d], the
// conv history [lanes][11][C] and rows8[lane] = 8.
cudaError_t launch_gdn_prep(const uint16_t* u, int ld_u, int M, const uint16_t* window_a, const uint16_t* taps,
                            int n_qk, int n_v, int d, uint16_t* q, uint16_t* k, uint16_t* v, uint16_t* conv_hist,
                            int32_t* rows8, cudaStream_t s);
// out[t][h d + i] = bf16(gated RMSNorm of the scan output o with silu(z)), z = u[t][z0 + h d + i].
cudaError_t launch_gated_norm(const float* o, const uint16_t* u, int ld_u, int z0, const float* w, int M, int n_v,
                              int d, uint16_t* out, cudaStream_t s);
// The rotary embedding's inverse frequencies 10000^(-2j / D), j < D / 2 (formed on the host in fp64).
struct RopeTable {
  double inv_freq[256];
};
RopeTable rope_table(int D);
// Q / K head RMSNorm + RoPE at ctx[lane] + t % 8, and dense copies of V and the gate.  D <= 512, even.
cudaError_t launch_attn_prep(const uint16_t* uq, int ld_q, const uint16_t* ukv, int ld_kv, int M, int Hq, int Hkv,
                             int D, const float* q_norm, const float* k_norm, const int32_t* ctx, const RopeTable& rt,
                             uint16_t* q, uint16_t* k, uint16_t* v, uint16_t* gate, cudaStream_t s);

}  // namespace vp
