// Launches of the mixer cores' producer and consumer steps (mixer.cu); each returns the launch's
// error.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace vp {

// The Gated DeltaNet core of one layer for all lanes (8 rows each), one launch (mixer.cu).
struct GdnCoreArgs {
  const uint16_t* h;         // bf16 [M][hidden]: the residual (the A / B projections' input)
  int hidden;                // % 128 == 0, <= 8192
  float eps;                 // RMSNorm eps of the A / B projections' input
  const uint16_t* u;         // bf16 [M][ld_u]: the in-projection (q, k, v, z)
  int ld_u, z0;              // row stride; first column of z
  const uint16_t* window_a;  // bf16 [lanes][3][C], C = (2 n_qk + n_v) 128
  const uint16_t* taps;      // bf16 [C][4]
  const uint16_t* wa;        // bf16 [n_v][hidden], 16-byte aligned
  const uint16_t* wb;        // bf16 [n_v][hidden], 16-byte aligned
  const float* a_log;        // fp32 [n_v]
  const float* dt_bias;      // fp32 [n_v]
  const float* norm_w;       // fp32 [128]
  const float* state_in;     // fp32 [lanes][n_v][128][128]
  float* state_out;          // fp32 [lanes][n_v][128][128]
  uint16_t* conv_hist;       // bf16 [lanes][11][C]
  uint16_t* out;             // bf16 [M][n_v 128]: the out-projection's input
  uint16_t* rec_qk;          // bf16 [M][2][n_qk][128]: the scan's q then k per q/k head (recorded)
  uint16_t* rec_v;           // bf16 [M][n_v][128]: the scan's v (recorded)
  float* rec_ab;             // fp32 [M][n_v][2]: alpha, beta (recorded)
  int n_qk, n_v;
};
cudaError_t launch_gdn_core(const GdnCoreArgs& a, int lanes, cudaStream_t s);

// The commit re-scan of up to kCommitLayers Gated DeltaNet layers in one launch (mixer.cu).
constexpr int kCommitLayers = 48;
struct GdnCommitLayer {
  const float* state_in;     // the intact parity buffer
  float* state_out;          // the other one: the state after the committed rows
  const uint16_t* conv_hist; // bf16 [lanes][11][C] of the pass
  uint16_t* window;          // bf16 [lanes][3][C]: rows n .. n + 2 of the history
  const uint16_t* rec_qk;    // the pass's record (GdnCoreArgs)
  const uint16_t* rec_v;
  const float* rec_ab;
};
struct GdnCommitArgs {
  GdnCommitLayer layer[kCommitLayers];
  const int32_t* n_commit;   // int32 [lanes], rows kept per lane (clamped to 0 .. 8)
  int lanes, n_qk, n_v;
};
cudaError_t launch_gdn_commit(const GdnCommitArgs& a, int n_layers, cudaStream_t s);
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
