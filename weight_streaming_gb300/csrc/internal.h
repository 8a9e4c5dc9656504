// Definitions shared by the host API (api.cu) and the streaming executor (exec.cuh): the packed
// weight layout, the phase program the executor runs, and the workspace carving.
#pragma once
#include <cstddef>
#include <cstdint>

struct vp_model;

namespace vp {

// Hidden size of a model handle (the width of x0 and of the residual stream); api.cu.
int model_hidden(const vp_model* model);

// ---------------------------------------------------------------- packed weight layout
// A matrix [N][K] (N % 16 == 0) is stored as row blocks of 16 rows; each row block as K chunks
// (256 weights wide for NVFP4, 128 for FP8); each chunk as two 8-row strips (rows 0-7, then 8-15 of
// the block).  Row block rb, chunk kc, strip t starts at ((rb * KC + kc) * 2 + t) * strip bytes, so
// a row block's stream along K is contiguous: one chunk of a row block is 2304 (NVFP4) or 2048
// (FP8) contiguous bytes, and so is any run of consecutive chunks.
//
// Inside a strip, thread (g = lane / 4, c = lane % 4) of a warp owns row g and, in every 16-wide k
// step s of the chunk, the four weights k = 16 s + 4 c .. + 3 (the mma.sync A fragment with the k
// order permuted inside each step; the activations are staged with the same permutation):
//   NVFP4 strip (1152 B): codes [half h = 0..1][g][c][16 B] -- the 16 bytes are steps 8h .. 8h + 7,
//                         two bytes per step (k, k+1 in the first byte, low nibble first; k+2, k+3
//                         in the second) -- then block scales [g][16 B], byte s = E4M3 scale of step s.
//   FP8 strip (1024 B):   [half h = 0..1][g][c][16 B] -- steps 4h .. 4h + 3, four bytes per step.
//   Q4 strip (1152 B):    codes [h][g][c][16 B] as NVFP4, but each 32-bit word w of the 16 bytes holds
//                         steps s = 8h + 2w and s + 1 with its eight 4-bit codes in the order the
//                         f16 magic-number conversion reads them: nibbles 0, 4 = step s, k + 0 / k + 1;
//                         nibbles 2, 6 = step s, k + 2 / k + 3; nibbles 1, 5 and 3, 7 = the same of step
//                         s + 1 -- then [g][16 B]: word G = bf16 scale | bf16 bias << 16 of the 64-wide
//                         group G of the chunk (steps 4G .. 4G + 3).
// Every warp-wide 16-byte shared-memory read of a strip is one contiguous 512-byte row.
constexpr int kRowBlock = 16;
constexpr int kStripRows = 8;
constexpr int kMaxM = 32;
// Rows a wide verify call takes (vp_verify_pass_rows and its kin): more than kMaxM run as passes of
// kMaxM rows, whole lanes each.
constexpr int kMaxRows = 128;

enum Fmt : int { kFmtNvfp4 = 0, kFmtFp8 = 1, kFmtQ4 = 2 };

__host__ __device__ constexpr int chunk_k(int fmt) { return fmt == kFmtFp8 ? 128 : 256; }
__host__ __device__ constexpr int strip_bytes(int fmt) { return fmt == kFmtFp8 ? 1024 : 1152; }
__host__ __device__ inline size_t strip_offset(int fmt, int KC, int rb, int kc, int t) {
  return (((size_t)rb * KC + kc) * 2 + t) * (size_t)strip_bytes(fmt);
}

// ---------------------------------------------------------------- executor geometry
// One persistent CTA per SM, 16 warps.  Every warp streams its own contiguous range of units
// through a private 2-slot shared-memory ring filled by bulk copies it issues itself, and runs the
// dequantisation + warp MMAs of each unit from there.  A unit is one "group" of K chunks of a
// virtual row block: two consecutive chunks of one row block (plain layout: one 4608 / 4096-byte
// copy), or one chunk of a gate row block and the same chunk of the matching up row block
// (interleaved layout: two 2304-byte copies).  Copies of this size keep a warp's ring streaming at
// full DRAM rate (many smaller copies queue up and lengthen the latency).  The rest of shared
// memory holds the activations of the CTA's K slice as f16 MMA fragments.
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 2;
constexpr int kSlotBytes = 4608;
constexpr int kRingBytes = kWarps * kSlots * kSlotBytes;  // 147,456
constexpr int kMiscBytes = 2560;
constexpr int kSmemBytes = 232448;  // 227 KB: the per-CTA maximum
constexpr int kXBytes = kSmemBytes - kRingBytes - kMiscBytes;
constexpr int kMaxGrid = 256;

// Widest K slice whose activations fit in kXBytes (16 NT bytes per k, NT n-tiles of 8 tokens) and
// that the staging threads hold in registers (128 k per thread of a row): a multiple of 512.
__host__ __device__ constexpr int ks_max(int NT) { return NT == 1 ? 5120 : NT == 2 ? 2560 : NT == 3 ? 1536 : 1024; }
static_assert(16 * 1 * ks_max(1) <= kXBytes && 16 * 2 * ks_max(2) <= kXBytes && 16 * 3 * ks_max(3) <= kXBytes &&
                  16 * 4 * ks_max(4) <= kXBytes,
              "activation slices fit the shared memory left by the ring");

enum Layout : int {
  kPlain = 0,        // virtual row blocks = the row blocks of w0, then of w1 (from row block rb1); groups of 2 chunks
  kInterleaved = 1,  // virtual row block rb = row block rb of w0 and of w1 (gate and up); groups of 1 chunk
};
enum Epi : int {
  kEpiF32 = 0,    // y[m][n] = s * acc
  kEpiZ = 1,      // z[m][n] = bf16(s * acc) for segment-0 rows n < out_cols (the rest is computed, unused)
  kEpiSilu = 2,   // a[m][f] = bf16(silu(s0 * gate) * s1 * up) (interleaved)
  kEpiResid = 3,  // h[m][n] = bf16(h[m][n] + s * acc) (and the trace copy)
  kEpiHead = 4,   // logits -> per-row argmax -> greedy acceptance
  kEpiU = 5,      // u[m][v] = bf16(s * acc) for every virtual row v (both segments): the in-projection
                  // kept whole for the real mixer cores
};
// Row-block sums of squares of the residual stream: a kEpiResid phase with kSsWrite stores, per token
// and 16-column row block of its output, the sum of the squares of the stored bf16 values; an RMSNorm
// phase with kSsRead whose K slice is narrower than the row takes the row's statistic from them (a
// fixed-order sum, the same in every CTA) instead of loading the whole row.  Used at 2+ n-tiles.
enum : int { kSsRead = 1, kSsWrite = 2 };
// Buffers a phase reads or writes, resolved per launch through Io::buf.
enum Buf : int { kBufX = 0, kBufY, kBufH, kBufZ, kBufA, kBufLogits, kBufTrace, kBufU, kNumBufs };

struct Phase {
  const uint8_t* w0;
  const uint8_t* w1;
  float s0, s1;     // fp32 scale of w0 / w1 (NVFP4 tensor scale or FP8 per-tensor scale)
  int K, KC;        // reduction length and its chunk count
  int grp, KG;      // chunks per unit (2 plain, 1 interleaved) and groups along K (ceil(KC / grp))
  int RB, rb1;      // virtual row blocks; first row block of w1 (plain; RB if none)
  int8_t fmt, layout, epi, ks;  // ks: K slices
  int8_t x_src, x_rms, out, ss;  // ss: kSsRead | kSsWrite (row-block sums of squares, see Io::rss)
  int x_ld, out_ld, out_cols, trace_slot;
};

constexpr int kMaxPhases = 160;
struct Program {
  int n, M;
  float eps;
  int q4;  // 1: every phase is Q4 (the executor instantiation with the Q4 unit)
  int rows;  // verify rows per lane of the head's acceptance (anchor + rows - 1 drafts)
  Phase ph[kMaxPhases];
};

struct Io {
  void* buf[kNumBufs];
  const int32_t* pending;
  int32_t* argmax;
  int32_t* n_commit;
  int32_t* committed;
  size_t trace_stride;  // elements between trace slots
  // workspace
  int* status;
  unsigned* bar;       // [0] barrier arrivals (monotonic within a launch), [1] CTAs that finished
  unsigned* head_cnt;
  float* head_aux;     // [kMaxGrid][kMaxM][2]
  // Split-K partials, in floats of 32 lanes x cs_lane (cs_lane = 4 NT, or 8 NT when the program has an
  // interleaved phase: its gate and up rows travel together):
  float* cslots;       // within a CTA: [kMaxGrid][kWarps][2] (a warp's first / last row block)
  float* xslots;       // across K slices: [RB][ks] (phases with ks > 1)
  int cs_lane;
  float* rss;          // row-block sums of squares [kMaxM][rss_ld] (or null)
  int rss_ld;
};

// ---------------------------------------------------------------- workspace carving
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Byte offset, from the status word, of the wait-test hook word (read only by the wait-test build:
// a nonzero value v makes CTA v - 1 leave its first grid-barrier arrival out).  It lies in the
// padding between the status word and the barrier counters.
constexpr size_t kWsTestSkip = 32;

struct WsLayout {
  size_t status, bar, head_cnt, head_aux, cslots, xslots, total;
};

// cs_lane: floats per lane of one partial (4 NT, or 8 NT with an interleaved phase); x_floats: the
// largest RB * ks * 32 * cs_lane of the program's phases with ks > 1 (0 if none); grid: the CTAs the
// in-CTA slots are sized for (kMaxGrid, so that a workspace size does not depend on the device,
// except where the caller knows the grid).
inline WsLayout ws_layout(int cs_lane, size_t x_floats, int grid = kMaxGrid) {
  WsLayout L;
  L.status = 0;
  L.bar = 64;
  L.head_cnt = 128;
  L.head_aux = 256;
  L.cslots = align_up(L.head_aux + sizeof(float) * 2 * kMaxM * kMaxGrid, 256);
  L.xslots = align_up(L.cslots + sizeof(float) * (size_t)grid * kWarps * 2 * 32 * cs_lane, 256);
  L.total = align_up(L.xslots + sizeof(float) * x_floats, 256);
  return L;
}

}  // namespace vp
