// Internal definitions shared by the host API (api.cu) and the kernels (gemm.cuh).
#pragma once
#include <cstddef>
#include <cstdint>

namespace vp {

// ---------------------------------------------------------------- packed layout constants
constexpr int kRowsPerBlock = 16;   // one MMA A tile: 16 weight rows
constexpr int kBlocksPerSlab = 16;  // 256 rows per slab (one stage of the copy ring)
constexpr int kSlabRows = kRowsPerBlock * kBlocksPerSlab;
constexpr int kQuadK = 64;          // K chunk of one packed block (four k16 MMA steps)
constexpr int kNvfp4BlockBytes = 576;  // 512 code bytes + 64 scale bytes (9 bytes per 16 weights)
constexpr int kFp8BlockBytes = 1024;   // 16 x 64 E4M3 bytes

enum Fmt : int { kFmtNvfp4 = 0, kFmtFp8 = 1 };

// ---------------------------------------------------------------- kernel geometry
constexpr int kConsumerWarps = 8;                      // each owns 2 row-blocks of a 256-row group
constexpr int kThreads = (kConsumerWarps + 1) * 32;    // + one bulk-copy producer warp
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kXBufBytes = 104 * 1024;                 // staged activation fragments
constexpr int kNvfp4Stages = 12;                       // 12 x 9216 B ring
constexpr int kFp8Stages = 7;                          // 7 x 16384 B ring
constexpr int kMaxM = 32;

enum Epi : int {
  kEpiF32 = 0,        // y[m][n] = scale * acc (fp32)
  kEpiBf16Prefix = 1, // out[m][n] = bf16(scale * acc) for n < out_cols (segment 0 only)
  kEpiSiluMul = 2,    // out[m][f] = bf16(silu(ts0 * gate) * ts1 * up)  (interleaved segments)
  kEpiResid = 3,      // h[m][n] = bf16(h[m][n] + scale * acc); finisher writes 1/rms(h) per row
  kEpiHead = 4,       // per-row argmax over n, then greedy acceptance per lane
};

struct GemmParams {
  // weights: one or two packed matrices ("segments") forming the virtual output rows
  const uint8_t* w[2];
  int seg_rows[2];    // rows of each segment (multiple of 16; seg_rows[1] = 0 if unused)
  float wscale[2];    // fp32 scale (NVFP4 tensor scale / FP8 per-tensor scale) per segment
  int interleave;     // 1: each 256-row group = 8 row-blocks of seg 0 + the same 8 of seg 1
  int K, M;
  int nq;             // K / 64
  int n_groups;       // virtual 256-row groups
  int seg0_groups;    // groups belonging to segment 0 (non-interleaved)
  long long units;    // n_groups * nq
  // activation source: bf16 [M][ld]; optional per-row multiplier (RMSNorm: 1/rms)
  const uint16_t* x;
  int x_ld;
  const float* x_rowscale;
  // epilogue
  int epi;
  float* y;  int y_ld;                 // kEpiF32
  uint16_t* out; int out_ld; int out_cols;  // kEpiBf16Prefix / kEpiSiluMul
  uint16_t* resid; int resid_ld; int resid_cols;  // kEpiResid (in/out)
  float* rms_out; float rms_eps;       // kEpiResid finisher
  const int32_t* pending; int32_t* argmax; int32_t* n_commit; int32_t* committed;  // kEpiHead
  float* logits; int logits_ld;        // kEpiHead (optional)
  // workspace
  int* status;
  unsigned* task_cnt;
  unsigned* group_cnt;  // [n_groups]
  float* group_aux;     // [n_groups][kMaxM][2]
  float* partials;      // [grid][2][kConsumerThreads][8 * MT]
};

// Workspace carving shared by the host-side size query and the launch code.
struct WsLayout {
  size_t status, task_cnt, group_cnt, group_aux, partials, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsLayout gemm_ws_layout(int n_groups, int grid, int mt) {
  WsLayout L;
  L.status = 0;
  L.task_cnt = 64;
  L.group_cnt = 256;
  L.group_aux = align_up(L.group_cnt + sizeof(unsigned) * (size_t)n_groups, 256);
  L.partials = align_up(L.group_aux + sizeof(float) * 2 * kMaxM * (size_t)n_groups, 256);
  L.total = align_up(L.partials + sizeof(float) * (size_t)grid * 2 * kConsumerThreads * 8 * mt, 256);
  return L;
}

}  // namespace vp
