// The streaming executor of the verify pass: one persistent kernel that runs a program of
// weight-streaming GEMM phases  Y = X W^T  (M = 1..32 activation rows, NVFP4 or FP8 weights, fp32
// accumulation) with their fused epilogues, separated by grid-wide barriers.
//
// Sources: "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max" -- "What one token
// costs the bus" (the NVFP4/FP8 weight groups a pass streams), "Formats, and what runs where"
// (NVFP4 = E2M1 code x E4M3 scale per 16 weights x fp32 tensor scale; weight-only arithmetic with
// BF16 activations and wide accumulation) and "The megakernel is per layer, not per step" (greedy
// acceptance); "Beating Splash on an M5 Max" -- "The kernels were not the gap" (split-K for narrow
// projections) and "The bugs a second reviewer found" (one argmax tie rule everywhere).
//
// GB300 design (not the pages' Metal tiles):
//  * One CTA per SM, 16 independent warps.  Each phase's units (a virtual row block x a group of K
//    chunks: 4608 B NVFP4 / 4096 B FP8) are split into equal contiguous ranges, one per warp.  A
//    warp streams its range through a private 2-slot ring with 1-D bulk copies that its lane 0
//    issues (evict-first), so no warp ever waits for another inside a phase, and it keeps
//    prefetching across phase ends: the next phase's first units are in flight while the grid
//    barrier and the activation staging of the phase boundary run.
//  * Dequantisation is exact in f16 (E2M1 x E4M3 products have <= 5 significant bits), done in
//    registers straight into mma.sync.m16n8k16 A fragments; the activations (B) are staged once per
//    phase as f16 fragments scaled per row by an exact power of two, which un-scales the fp32
//    accumulators.  At M <= 8 a 16x16 weight tile costs one MMA per 8 tokens, so the SM's issue
//    slots, not the tensor pipe, carry the dequantisation (about 8 TB/s-equivalent per GPU).
//  * K slices: when a phase's activations do not fit shared memory, its K chunks are cut into ks
//    slices with CTAs assigned in proportion.  Row blocks that several warps share are reduced by
//    the last contributor (atomic counter, no waiting) in a fixed order, so every result is
//    bit-reproducible; it then runs the epilogue.  The partials pass through tensor memory between
//    warps of one lane quarter (the warps' ranges are handed out quarter by quarter), else through
//    L2.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "internal.h"
#include "ptx.cuh"
#include "trace.cuh"

namespace vp {

enum : int { kStatusTimeout = 6 };

// ---------------------------------------------------------------- tensor memory (the in-CTA fixups)
// Warp w reaches lanes 32 (w % 4) .. + 31 of the SM's tensor memory.  The fixups keep each warp's
// partials there too, in its lane quarter, so that a warp of the same quarter can sum them without
// an L2 round trip: 4 warps x 2 slots x cs_lane columns (cs_lane <= 8 NT).
template <int NT>
constexpr uint32_t kTmemCols = NT == 1 ? 64u : NT == 2 ? 128u : 256u;
// The range of units a warp takes within its CTA: warps 0, 4, 8, 12 the first four, then 1, 5, 9,
// 13, ...: consecutive ranges (which share row blocks) then mostly sit in one lane quarter.
__device__ __forceinline__ int range_of(int warp) { return 4 * (warp & 3) + (warp >> 2); }

static_assert(kSlotBytes >= 2 * 2304 && kSlotBytes >= 2 * 2048, "a slot holds one unit");

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }
__device__ __forceinline__ uint16_t bf16_bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

// ---------------------------------------------------------------- argmax helpers
// Lowest index among the largest values; callers map NaN to -inf first, and -0 == +0.
__device__ __forceinline__ bool am_better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }
__device__ __forceinline__ void am_shfl_xor(float& v, int& i, int off) {
  const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
  const int i2 = __shfl_xor_sync(0xffffffffu, i, off);
  if (am_better(v2, i2, v, i)) {
    v = v2;
    i = i2;
  }
}
// Greedy acceptance of lane l of R verify rows given the target tokens tok[R l .. R l + R - 1] (the
// anchor pending[R l] is not compared): the longest prefix of drafts equal to the target's tokens
// plus the target's token after it.  The pages' verify has R = 8; lookup drafts verify up to 32.
__device__ __forceinline__ void accept_lane(int l, int R, const int* tok, const int32_t* pending, int32_t* n_commit,
                                            int32_t* committed) {
  int acc = 0;
  while (acc < R - 1 && tok[R * l + acc] == pending[R * l + acc + 1]) ++acc;
  n_commit[l] = acc + 1;
  for (int j = 0; j < R; ++j) committed[R * l + j] = j <= acc ? tok[R * l + j] : -1;
}

// ---------------------------------------------------------------- phase geometry
// K slice s of a phase: chunk groups [kg0, kg0 + kgn), CTAs [cta0, cta0 + ctan) in proportion to
// the groups.  Within a slice every CTA owns whole row blocks: CTA c of the slice owns row blocks
// [c RB / ctan, (c + 1) RB / ctan), so a (row block, slice) task never leaves its CTA.  The CTA's
// units (row-block major, kgn per row block) are cut into equal contiguous ranges over
// W = min(16, U) warps, so every warp with a range owns at least one unit and the contributors of
// a row block are consecutive warps.
struct Slice {
  int kg0, kgn, cta0, ctan;
};
// (a * b + d) / c for non-negative ints with a quotient that fits an int: 32-bit unsigned division
// when the dividend fits (the usual case), else 64-bit.
__device__ __forceinline__ int muldiv(int a, int b, int d, int c) {
  const long long n = (long long)a * b + d;
  return n < (1LL << 32) ? (int)((unsigned)n / (unsigned)c) : (int)(n / c);
}
__device__ __forceinline__ Slice slice_geom(const Phase& ph, int G, int s) {
  Slice S;
  const int kg0 = muldiv(s, ph.KG, 0, ph.ks), kg1 = muldiv(s + 1, ph.KG, 0, ph.ks);
  const int c0 = muldiv(G, kg0, ph.KG / 2, ph.KG);
  const int c1 = s + 1 == ph.ks ? G : muldiv(G, kg1, ph.KG / 2, ph.KG);
  S.kg0 = kg0;
  S.kgn = kg1 - kg0;
  S.cta0 = c0;
  S.ctan = c1 - c0;
  return S;
}
// A CTA's share of a phase: its slice, its row blocks [rb0, rb0 + nrb), U = nrb * kgn units over W
// warps.
struct Part {
  Slice S;
  int sidx, rb0, nrb, U, W;
};
__device__ __forceinline__ Part part_of_cta(const Phase& ph, int G, int cta) {
  Part P;
  P.sidx = ph.ks - 1;
  for (int s = 0; s < ph.ks; ++s) {
    P.S = slice_geom(ph, G, s);
    if (cta < P.S.cta0 + P.S.ctan) {
      P.sidx = s;
      break;
    }
  }
  const int c = cta - P.S.cta0;
  P.rb0 = muldiv(c, ph.RB, 0, P.S.ctan);
  P.nrb = muldiv(c + 1, ph.RB, 0, P.S.ctan) - P.rb0;
  P.U = P.nrb * P.S.kgn;
  P.W = min(kWarps, P.U);
  return P;
}
// Warp w of a CTA owns its units [wbegin(w), wbegin(w + 1)); wowner(u) inverts it.
__device__ __forceinline__ int wbegin(const Part& P, int w) { return w >= P.W ? P.U : muldiv(w, P.U, 0, P.W); }
__device__ __forceinline__ int wowner(const Part& P, int u) { return muldiv(u + 1, P.W, -1, P.U); }

// A phase's descriptor, the CTA's share of it and the warps' unit ranges, kept in shared memory.
// Slot p % 3 holds phase p.  Phases 0 and 1 are filled at the start; phase p + 2 by the first warp
// of the CTA to finish its units of phase p, so that neither the phase loop nor the weight
// producers (which cross into the next phase while the current one streams) read the kernel
// parameters or divide on their critical paths.  The slot's phase index is written last with a
// CTA-scope release and read with an acquire.
constexpr int kPhaseSlots = 3;
struct PhaseSlot {
  Phase ph;
  Part part;
  int idx;                // the phase held (-1: none)
  int wb[kWarps + 1];     // warp w's units: [wb[w], wb[w + 1])
  const void* x;          // the phase's activation source
};
static __device__ __noinline__ void fill_slot(PhaseSlot& sl, const Program& prog, const Io& io, int p, int G, int cta,
                                          int lane) {
  static_assert(sizeof(Phase) % 4 == 0 && sizeof(Phase) <= 32 * 4, "a phase descriptor is at most 32 words");
  const uint32_t* src = reinterpret_cast<const uint32_t*>(&prog.ph[p]);
  uint32_t* dst = reinterpret_cast<uint32_t*>(&sl.ph);
  if (lane < (int)(sizeof(Phase) / 4)) dst[lane] = src[lane];
  __syncwarp();
  const Part P = part_of_cta(sl.ph, G, cta);
  if (lane <= kWarps) sl.wb[lane] = wbegin(P, lane);
  if (lane == 0) {
    sl.part = P;
    sl.x = io.buf[sl.ph.x_src];
  }
  __syncwarp();
  if (lane == 0) st_release_cta_smem(&sl.idx, p);
}
__device__ __forceinline__ bool slot_holds(const PhaseSlot& sl, int p) { return ld_acquire_cta_smem(&sl.idx) == p; }

// ---------------------------------------------------------------- weight producer (lane 0 of a warp)
// Walks the warp's units across all phases of the program, in consumption order, keeping the
// source addresses of the current unit: within a row block the next unit is the next K chunk
// (2 strips further on), so a step is two pointer increments; the phase descriptor is read only
// when the row block or the phase changes.
struct __align__(16) Cursor {
  int p;             // phase (== prog.n when done)
  int left;          // units left in the phase's range, including the current one
  int rb, kgl;       // row block and group position within the slice of the current unit
  int kg0, kgn;      // the slice's groups
  int kc, KC, grp;   // first chunk of the current unit; the phase's chunks and group width
  uint32_t chunk;    // bytes of one chunk of one row block (two strips)
  const uint8_t* a;
  const uint8_t* b;  // the up row block's chunk (interleaved layout), else nullptr
  uint32_t bytes;    // per source
};
static_assert(sizeof(Cursor) == 64, "a cursor is four 16-byte words");
// The warp's cursor moves between shared memory and registers as four 16-byte words.
__device__ __forceinline__ void cursor_load(Cursor& dst, const Cursor& src) {
  const uint4* s = reinterpret_cast<const uint4*>(&src);
  uint4* d = reinterpret_cast<uint4*>(&dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = s[i];
}
// Source addresses of the cursor's unit (read from the phase descriptor).
__device__ __forceinline__ void cursor_locate_in(Cursor& c, const Phase& ph) {
  c.KC = ph.KC;
  c.grp = ph.grp;
  c.chunk = 2u * strip_bytes(ph.fmt);
  c.kc = (c.kg0 + c.kgl) * ph.grp;
  if (ph.layout == kPlain) {
    const bool s1 = c.rb >= ph.rb1;
    c.a = (s1 ? ph.w1 : ph.w0) + strip_offset(ph.fmt, ph.KC, s1 ? c.rb - ph.rb1 : c.rb, c.kc, 0);
    c.b = nullptr;
    c.bytes = (uint32_t)min(ph.grp, ph.KC - c.kc) * c.chunk;
  } else {
    const size_t off = strip_offset(ph.fmt, ph.KC, c.rb, c.kc, 0);
    c.a = ph.w0 + off;
    c.b = ph.w1 + off;
    c.bytes = c.chunk;
  }
}
// Out of line: called when the row block or the phase changes, which keeps the unit loop's
// registers for the unit.
__device__ __forceinline__ void cursor_locate(Cursor& c, const Program& prog, const PhaseSlot*) {
  cursor_locate_in(c, prog.ph[c.p]);
}
__device__ __forceinline__ void cursor_seek(Cursor& c, const Program& prog, const PhaseSlot* slots, int G, int cta,
                                            int warp) {
  while (c.p < prog.n) {
    const PhaseSlot& sl = slots[c.p % kPhaseSlots];
    Part P;
    int u;
    const int q = range_of(warp);
    if (slot_holds(sl, c.p)) {
      P = sl.part;
      u = sl.wb[q];
      c.left = sl.wb[q + 1] - u;
    } else {
      P = part_of_cta(prog.ph[c.p], G, cta);
      u = wbegin(P, q);
      c.left = wbegin(P, q + 1) - u;
    }
    if (c.left > 0) {
      c.kg0 = P.S.kg0;
      c.kgn = P.S.kgn;
      c.rb = P.rb0 + u / P.S.kgn;
      c.kgl = u - (c.rb - P.rb0) * P.S.kgn;
      cursor_locate(c, prog, slots);
      return;
    }
    ++c.p;
  }
}
// Next unit: within a row block the next group follows contiguously (grp chunks further on).
__device__ __forceinline__ void cursor_next(Cursor& c, const Program& prog, const PhaseSlot* slots, int G, int cta,
                                            int warp) {
  if (--c.left == 0) {
    ++c.p;
    cursor_seek(c, prog, slots, G, cta, warp);
  } else if (++c.kgl == c.kgn) {
    c.kgl = 0;
    ++c.rb;
    cursor_locate(c, prog, slots);
  } else {
    const uint32_t step = (uint32_t)c.grp * c.chunk;
    c.kc += c.grp;
    c.a += step;
    if (c.b)
      c.b += step;
    else
      c.bytes = (uint32_t)min(c.grp, c.KC - c.kc) * c.chunk;
  }
}

struct SmemMisc {
  uint64_t full[kWarps][kSlots];
  Cursor cur[kWarps];  // the producer state of each warp (used by its lane 0 only)
  unsigned tcnt[kWarps];  // arrivals at a row block shared by warps, indexed by its first contributor
  PhaseSlot ps[kPhaseSlots];  // phase p in slot p % 3
  int fillp;                  // the phase whose slot is filled next, minus 2
  float red[kThreads / 16];
  float xscale[kMaxM];
  int tok[kMaxM];
  int abort;
  int flag;
  uint32_t tmem;  // the CTA's tensor-memory allocation
};
static_assert(sizeof(SmemMisc) + 16 <= (size_t)kMiscBytes, "SmemMisc exceeds its shared-memory budget (the last word is the trace parity)");

// Bulk copy of the cursor's unit into the slot at shared address dst, completing on bar.
__device__ __forceinline__ void issue_unit(const Cursor& c, uint32_t dst, uint64_t* bar, uint64_t pol) {
  const uint32_t b = smem_addr(bar);
  mbar_arrive_expect_tx(bar, c.b ? 2u * c.bytes : c.bytes);
  bulk_g2s(dst, c.a, c.bytes, b, pol);
  if (c.b) bulk_g2s(dst + c.bytes, c.b, c.bytes, b, pol);
}

// ---------------------------------------------------------------- activation staging
// Shared layout of the K slice's activations: for every pair of 16-wide k steps p, n-tile j and lane
// (g, c): 16 bytes = the f16 values of token 8j + g at k = 32p + 4c .. +3 (step 2p) and
// 32p + 16 + 4c .. +3 (step 2p + 1) -- exactly the thread's two B fragments.
template <int NT>
__device__ __forceinline__ uint32_t xfrag_offset(int p, int n, int c) {
  return (uint32_t)((((p * NT + (n >> 3)) * 32 + (n & 7) * 4 + c) * 16));
}

__device__ __forceinline__ float sumsq8(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = bf16_bits_to_float(w[i] & 0xFFFFu), b = bf16_bits_to_float(w[i] >> 16);
    s = fmaf(a, a, s);
    s = fmaf(b, b, s);
  }
  return s;
}

// Exponent e of a row whose largest magnitude is mx: the row enters the tensor core as x * 2^-e,
// below 2^15 (f16 holds every bf16 value exactly there, down to 2^-24 of that scale).
__device__ __forceinline__ int exp_of_max(float mx) {
  if (!(mx > 0.0f) || !(mx < INFINITY)) return 0;
  int ex;
  frexpf(mx, &ex);  // mx in [2^(ex-1), 2^ex)
  return ex - 1 - 14;
}

// Stages the CTA's K slice [kbase, kbase + Ks) of phase `trace_phase`'s activation rows: x, or
// bf16(RMSNorm(x)) (unit weight) when the phase asks for it, with the row statistics taken over
// the whole row.
//
// Work items: (token n, 64-wide k block, its 32-wide half p, h) -> the thread loads the 16-byte chunks
// k = 32 p + 8 h .. + 7 and 32 p + 16 + 8 h .. + 7 and writes the two whole fragment entries they fill
// (lanes c = 2 h and 2 h + 1 of token n for k-step pair p: 32 contiguous bytes).  Lane l of a warp
// takes token 2 (l >> 3) + (l & 1) of an 8-token tile, h = (l >> 1) & 1 and the parity of p
// (l >> 2) & 1, and writes first the entry c = 2 h + (p & 1): the 8 lanes of a quarter warp then hit
// 8 different 4-bank groups (token parity x c), so the 16-byte stores have no bank conflicts.  Each
// warp takes (tile, 64-wide block) pairs warp, warp + 16, ... (at most 5: Ks <= ks_max(NT)).
template <int NT>
__device__ __forceinline__ void stage_x(const Program& prog, const Phase& ph, const Io& io, int kbase, int Ks,
                                        uint8_t* xs, SmemMisc& sm, int trace_phase) {
  constexpr int kIt = 5;
  static_assert(NT * ks_max(NT) / 64 <= kIt * kWarps, "every (tile, k block) pair has a warp iteration");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, M = prog.M;
  const int g = 2 * (lane >> 3) + (lane & 1), h = (lane >> 1) & 1, pp = (lane >> 2) & 1;
  const int blocks = Ks >> 6, items = NT * blocks;
  const uint16_t* xsrc = static_cast<const uint16_t*>(sm.ps[trace_phase % kPhaseSlots].x);
  const bool rms = ph.x_rms != 0;
  uint4 va[kIt], vb[kIt];
  float stat[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) stat[j] = 0.0f;
  // All of the thread's chunks are loaded at once (one memory round trip).
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    const int item = warp + kWarps * it, tile = item % NT, n = 8 * tile + g, p = 2 * (item / NT) + pp;
    const bool ok = item < items && n < M;
    const uint16_t* a = xsrc + (size_t)(ok ? n : 0) * ph.x_ld + kbase + 32 * p + 8 * h;
    va[it] = ok ? ldcg128(a) : make_uint4(0u, 0u, 0u, 0u);
    vb[it] = ok ? ldcg128(a + 16) : make_uint4(0u, 0u, 0u, 0u);
  }
  // The thread's statistic per tile (sum of squares for RMSNorm, else the largest magnitude).
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    const int tile = (warp + kWarps * it) % NT;
    const uint32_t w[8] = {va[it].x, va[it].y, va[it].z, va[it].w, vb[it].x, vb[it].y, vb[it].z, vb[it].w};
    float st = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float a = __uint_as_float(w[k] << 16), b = __uint_as_float(w[k] & 0xFFFF0000u);
      st = rms ? fmaf(b, b, fmaf(a, a, st)) : fmaxf(st, fmaxf(fabsf(a), fabsf(b)));
    }
#pragma unroll
    for (int j = 0; j < NT; ++j)
      if (j == tile) stat[j] = rms ? stat[j] + st : fmaxf(stat[j], st);
  }
  // The row's statistic, summed in a fixed order (the same in every CTA): per warp over the lanes of
  // a token (xor 2, 4), then over the warps in order.  Scratch: the start of the activation area,
  // which the fragments overwrite only after the next barrier.
  float* red = reinterpret_cast<float*>(xs);  // [kWarps][kMaxM]
  bool from_rss = false, whole_row = false;
  if (rms && Ks < ph.K) {
    if constexpr (NT > 1) from_rss = (ph.ss & kSsRead) && io.rss;
    whole_row = !from_rss;
  }
  if (from_rss || whole_row) {
    // The statistic of the whole row, not only the slice: thread 16 n + i sums its share of token n's
    // row -- the producer's 16-wide row-block sums of squares, or the row itself -- with 8 loads in
    // flight at a time, then a fixed xor tree over the token's 16 threads.
    const int n = tid >> 4, i = tid & 15;
    float sum = 0.0f;
    if (n < M) {
      if (from_rss) {
        const float4* r4 = reinterpret_cast<const float4*>(io.rss + (size_t)n * io.rss_ld);
        const int nq = ph.K >> 6;
        for (int q0 = i; q0 < nq; q0 += 16 * 8) {
          float4 a[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            a[k] = q0 + 16 * k < nq ? __ldcg(r4 + q0 + 16 * k) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
          for (int k = 0; k < 8; ++k) sum += (a[k].x + a[k].y) + (a[k].z + a[k].w);
        }
      } else {
        const uint16_t* row = xsrc + (size_t)n * ph.x_ld;
        const int nq = ph.K >> 3;
        for (int q0 = i; q0 < nq; q0 += 16 * 8) {
          uint4 a[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) a[k] = q0 + 16 * k < nq ? ldcg128(row + 8 * (q0 + 16 * k)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int k = 0; k < 8; ++k) sum += sumsq8(a[k]);
        }
      }
    }
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (i == 0) red[n] = sum;
  } else {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      float x = stat[j];
      const float y2 = __shfl_xor_sync(0xffffffffu, x, 2);
      x = rms ? x + y2 : fmaxf(x, y2);
      const float y4 = __shfl_xor_sync(0xffffffffu, x, 4);
      x = rms ? x + y4 : fmaxf(x, y4);
      // the warp's partial for tile j: its lanes' statistic over the pairs of that tile (zero if none)
      if ((lane & 6) == 0) red[warp * kMaxM + 8 * j + g] = x;
    }
    if (NT * 8 < kMaxM && lane < kMaxM - 8 * NT) red[warp * kMaxM + 8 * NT + lane] = 0.0f;
  }
  __syncthreads();
  if (tid < kMaxM) {
    float tot = 0.0f;
    if (from_rss || whole_row)
      tot = red[tid];
    else
      for (int w = 0; w < kWarps; ++w) tot = rms ? tot + red[w * kMaxM + tid] : fmaxf(tot, red[w * kMaxM + tid]);
    int e;
    float inv = 1.0f;
    if (rms) {
      inv = 1.0f / sqrtf(tot / (float)ph.K + prog.eps);
      // RMSNorm output has |r| <= sqrt(K) (no element exceeds the root of the row's sum of squares;
      // 1% covers the fp32 1/rms and the bf16 rounding): the exponent of that bound.
      e = exp_of_max(1.01f * sqrtf((float)ph.K));
    } else {
      e = exp_of_max(tot);
    }
    sm.xscale[tid] = tid < M ? pow2f(e) : 0.0f;
    sm.red[tid] = inv;
    sm.tok[tid] = e;
  }
  __syncthreads();
  VP_TRACE(tid == 0, trace_phase, 36);
  // x * 2^-e exactly (two power-of-two steps when 2^-e is not a normal float); for RMSNorm the
  // 2^-e folds into 1/rms: bf16(x * inv) * 2^-e == bf16(x * (inv * 2^-e)) (no under/overflow).
  const uint32_t xb = smem_addr(xs);
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    const int item = warp + kWarps * it, tile = item % NT, n = 8 * tile + g, p = 2 * (item / NT) + pp;
    if (item >= items) continue;
    const int ne = -sm.tok[n];
    float sc1 = ne > 127 ? pow2f(127) : ne < -126 ? pow2f(-126) : pow2f(ne);
    const float sc2 = ne > 127 ? pow2f(ne - 127) : ne < -126 ? pow2f(ne + 126) : 1.0f;
    if (rms) sc1 *= sm.red[n];
    const uint32_t w[8] = {va[it].x, va[it].y, va[it].z, va[it].w, vb[it].x, vb[it].y, vb[it].z, vb[it].w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float a = __uint_as_float(w[k] << 16) * sc1, b = __uint_as_float(w[k] & 0xFFFF0000u) * sc1;
      if (rms) {
        const __nv_bfloat162 r = __floats2bfloat162_rn(a, b);  // the RMSNorm output, rounded once
        a = __low2float(r);
        b = __high2float(r);
      } else {
        a *= sc2;
        b *= sc2;
      }
      const __half2 hh = __floats2half2_rn(a, b);
      o[k] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    // entry c = 2h: k = 32p + 8h + 0..3 (chunk a words 0, 1) and 32p + 16 + 8h + 0..3 (chunk b words
    // 0, 1); entry c = 2h + 1: the upper halves (words 2, 3 of each chunk).
    const uint32_t e0 = xb + xfrag_offset<NT>(p, n, 2 * h);
    const uint4 lo = make_uint4(o[0], o[1], o[4], o[5]), hi = make_uint4(o[2], o[3], o[6], o[7]);
    if (pp) {
      sts128(e0 + 16, hi);
      sts128(e0, lo);
    } else {
      sts128(e0, lo);
      sts128(e0 + 16, hi);
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------- one unit of a warp
// One K chunk of one row block.  acc[j] (16 rows x 8 tokens, the mma.sync C fragment): rows g, g + 8
// of the row block, tokens 8j + 2c, 8j + 2c + 1; even k steps accumulate into acc, odd ones into
// acc2 (the caller passes the same array twice for one chain).  ua: the chunk in the slot; xa: this
// lane's fragments of the chunk's first k-step pair.
template <int NT>
__device__ __forceinline__ void unit_nvfp4(uint32_t ua, uint32_t xa, int lane, float (&acc)[NT][4],
                                           float (&acc2)[NT][4]) {
  const int g = lane >> 2;
  const uint4 c0a = lds128(ua + lane * 16), c0b = lds128(ua + 512 + lane * 16);
  const uint4 c1a = lds128(ua + 1152 + lane * 16), c1b = lds128(ua + 1152 + 512 + lane * 16);
  const uint4 s0 = lds128(ua + 1024 + g * 16), s1 = lds128(ua + 1152 + 1024 + g * 16);
  const uint32_t w0[8] = {c0a.x, c0a.y, c0a.z, c0a.w, c0b.x, c0b.y, c0b.z, c0b.w};
  const uint32_t w1[8] = {c1a.x, c1a.y, c1a.z, c1a.w, c1b.x, c1b.y, c1b.z, c1b.w};
  const uint32_t sw0[4] = {s0.x, s0.y, s0.z, s0.w}, sw1[4] = {s1.x, s1.y, s1.z, s1.w};
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    uint4 b[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) b[j] = lds128(xa + (p * NT + j) * 512);
    // block scales of steps 2p, 2p + 1 for rows g and g + 8
    const uint32_t sc0 = e4m3x2_to_f16x2((p & 1) ? (sw0[p >> 1] >> 16) : sw0[p >> 1]);
    const uint32_t sc1 = e4m3x2_to_f16x2((p & 1) ? (sw1[p >> 1] >> 16) : sw1[p >> 1]);
    uint32_t o0[4], o1[4];
    e2m1x8_to_f16x2x4(w0[p], o0);
    e2m1x8_to_f16x2x4(w1[p], o1);
    {
      const uint32_t d0 = dup_lo16(sc0), d1 = dup_lo16(sc1);
      const uint32_t a0 = hmul2_u32(o0[0], d0), a1 = hmul2_u32(o1[0], d1);
      const uint32_t a2 = hmul2_u32(o0[1], d0), a3 = hmul2_u32(o1[1], d1);
#pragma unroll
      for (int j = 0; j < NT; ++j) mma_f16_16816(acc[j], a0, a1, a2, a3, b[j].x, b[j].y);
    }
    {
      const uint32_t d0 = dup_hi16(sc0), d1 = dup_hi16(sc1);
      const uint32_t a0 = hmul2_u32(o0[2], d0), a1 = hmul2_u32(o1[2], d1);
      const uint32_t a2 = hmul2_u32(o0[3], d0), a3 = hmul2_u32(o1[3], d1);
#pragma unroll
      for (int j = 0; j < NT; ++j) mma_f16_16816(acc2[j], a0, a1, a2, a3, b[j].z, b[j].w);
    }
  }
}

// The same K chunk of two row blocks (chunk u0 -> acc0, chunk u1 -> acc1) against the same
// activations: each B fragment is loaded from shared memory once for both row blocks' MMAs.  The
// code words are loaded per half chunk (steps 0-7, then 8-15) to keep fewer registers live.
template <int NT>
__device__ __forceinline__ void unit_nvfp4_pair(uint32_t u0, uint32_t u1, uint32_t xa, int lane, float (&acc0)[NT][4],
                                                float (&acc1)[NT][4]) {
  const int g = lane >> 2;
  const uint4 s00 = lds128(u0 + 1024 + g * 16), s01 = lds128(u0 + 1152 + 1024 + g * 16);
  const uint4 s10 = lds128(u1 + 1024 + g * 16), s11 = lds128(u1 + 1152 + 1024 + g * 16);
  const uint32_t sw00[4] = {s00.x, s00.y, s00.z, s00.w}, sw01[4] = {s01.x, s01.y, s01.z, s01.w};
  const uint32_t sw10[4] = {s10.x, s10.y, s10.z, s10.w}, sw11[4] = {s11.x, s11.y, s11.z, s11.w};
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint4 c00 = lds128(u0 + 512 * half + lane * 16), c01 = lds128(u0 + 1152 + 512 * half + lane * 16);
    const uint4 c10 = lds128(u1 + 512 * half + lane * 16), c11 = lds128(u1 + 1152 + 512 * half + lane * 16);
    const uint32_t w00[4] = {c00.x, c00.y, c00.z, c00.w}, w01[4] = {c01.x, c01.y, c01.z, c01.w};
    const uint32_t w10[4] = {c10.x, c10.y, c10.z, c10.w}, w11[4] = {c11.x, c11.y, c11.z, c11.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int p = 4 * half + q;
      uint4 b[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) b[j] = lds128(xa + (p * NT + j) * 512);
#pragma unroll
      for (int r = 0; r < 2; ++r) {  // row block r of the pair
        const uint32_t* sa = r ? sw10 : sw00;
        const uint32_t* sb = r ? sw11 : sw01;
        const uint32_t sc0 = e4m3x2_to_f16x2((p & 1) ? (sa[p >> 1] >> 16) : sa[p >> 1]);
        const uint32_t sc1 = e4m3x2_to_f16x2((p & 1) ? (sb[p >> 1] >> 16) : sb[p >> 1]);
        uint32_t o0[4], o1[4];
        e2m1x8_to_f16x2x4(r ? w10[q] : w00[q], o0);
        e2m1x8_to_f16x2x4(r ? w11[q] : w01[q], o1);
        float (&acc)[NT][4] = r ? acc1 : acc0;
        {
          const uint32_t d0 = dup_lo16(sc0), d1 = dup_lo16(sc1);
          const uint32_t a0 = hmul2_u32(o0[0], d0), a1 = hmul2_u32(o1[0], d1);
          const uint32_t a2 = hmul2_u32(o0[1], d0), a3 = hmul2_u32(o1[1], d1);
#pragma unroll
          for (int j = 0; j < NT; ++j) mma_f16_16816(acc[j], a0, a1, a2, a3, b[j].x, b[j].y);
        }
        {
          const uint32_t d0 = dup_hi16(sc0), d1 = dup_hi16(sc1);
          const uint32_t a0 = hmul2_u32(o0[2], d0), a1 = hmul2_u32(o1[2], d1);
          const uint32_t a2 = hmul2_u32(o0[3], d0), a3 = hmul2_u32(o1[3], d1);
#pragma unroll
          for (int j = 0; j < NT; ++j) mma_f16_16816(acc[j], a0, a1, a2, a3, b[j].z, b[j].w);
        }
      }
    }
  }
}

// One Q4 chunk (w = scale * q + bias per 64-wide group): for each group, the codes q (exact f16
// integers) times the staged activations on the tensor core into a group accumulator t, and a
// ones operand times the same activations into sx, the group's activation sums of the C fragment's
// tokens (every row of that product is the column sum); then acc += scale * t + bias * sx in fp32.
// t and sx are both in the staged (row-scaled) units.
template <int NT>
__device__ __forceinline__ void unit_q4(uint32_t ua, uint32_t xa, int lane, float (&acc)[NT][4]) {
  const int g = lane >> 2;
  const uint4 c0a = lds128(ua + lane * 16), c0b = lds128(ua + 512 + lane * 16);
  const uint4 c1a = lds128(ua + 1152 + lane * 16), c1b = lds128(ua + 1152 + 512 + lane * 16);
  const uint4 s0 = lds128(ua + 1024 + g * 16), s1 = lds128(ua + 1152 + 1024 + g * 16);
  const uint32_t w0[8] = {c0a.x, c0a.y, c0a.z, c0a.w, c0b.x, c0b.y, c0b.z, c0b.w};
  const uint32_t w1[8] = {c1a.x, c1a.y, c1a.z, c1a.w, c1b.x, c1b.y, c1b.z, c1b.w};
  const uint32_t sb0[4] = {s0.x, s0.y, s0.z, s0.w}, sb1[4] = {s1.x, s1.y, s1.z, s1.w};
  constexpr uint32_t kOnes = 0x3C003C00u;  // f16x2 (1, 1)
#pragma unroll
  for (int G = 0; G < 4; ++G) {
    float t[NT][4], sx[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) t[j][r] = sx[j][r] = 0.0f;
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
      const int p = 2 * G + pp;  // steps 2p, 2p + 1
      uint4 b[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) b[j] = lds128(xa + (p * NT + j) * 512);
      uint32_t o0[4], o1[4];
      q4x8_to_f16x2x4(w0[p], o0);
      q4x8_to_f16x2x4(w1[p], o1);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        mma_f16_16816(t[j], o0[0], o1[0], o0[1], o1[1], b[j].x, b[j].y);
        mma_f16_16816(t[j], o0[2], o1[2], o0[3], o1[3], b[j].z, b[j].w);
        mma_f16_16816(sx[j], kOnes, kOnes, kOnes, kOnes, b[j].x, b[j].y);
        mma_f16_16816(sx[j], kOnes, kOnes, kOnes, kOnes, b[j].z, b[j].w);
      }
    }
    const float sc0 = __uint_as_float(sb0[G] << 16), bi0 = __uint_as_float(sb0[G] & 0xFFFF0000u);
    const float sc1 = __uint_as_float(sb1[G] << 16), bi1 = __uint_as_float(sb1[G] & 0xFFFF0000u);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      acc[j][0] = fmaf(bi0, sx[j][0], fmaf(sc0, t[j][0], acc[j][0]));
      acc[j][1] = fmaf(bi0, sx[j][1], fmaf(sc0, t[j][1], acc[j][1]));
      acc[j][2] = fmaf(bi1, sx[j][2], fmaf(sc1, t[j][2], acc[j][2]));
      acc[j][3] = fmaf(bi1, sx[j][3], fmaf(sc1, t[j][3], acc[j][3]));
    }
  }
}

template <int NT>
__device__ __forceinline__ void unit_fp8(uint32_t ua, uint32_t xa, int lane, float (&acc)[NT][4],
                                         float (&acc2)[NT][4]) {
  const uint4 c0a = lds128(ua + lane * 16), c0b = lds128(ua + 512 + lane * 16);
  const uint4 c1a = lds128(ua + 1024 + lane * 16), c1b = lds128(ua + 1024 + 512 + lane * 16);
  const uint32_t w0[8] = {c0a.x, c0a.y, c0a.z, c0a.w, c0b.x, c0b.y, c0b.z, c0b.w};
  const uint32_t w1[8] = {c1a.x, c1a.y, c1a.z, c1a.w, c1b.x, c1b.y, c1b.z, c1b.w};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint4 b[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) b[j] = lds128(xa + (p * NT + j) * 512);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t a0, a1, a2, a3;
      e4m3x4_to_f16x2x2(w0[2 * p + h], a0, a2);
      e4m3x4_to_f16x2x2(w1[2 * p + h], a1, a3);
#pragma unroll
      for (int j = 0; j < NT; ++j) mma_f16_16816(h ? acc2[j] : acc[j], a0, a1, a2, a3, h ? b[j].z : b[j].x, h ? b[j].w : b[j].y);
    }
  }
}

// ---------------------------------------------------------------- epilogues
template <int NT>
struct HeadBest {
  float v[NT][2];
  int i[NT][2];
};

// Residual inputs h[t][n] of the thread's elements of row block rb (plain layout) for token tile j:
// element [2r + h] = row g + 8r, token 8j + 2c + h.
__device__ __forceinline__ void load_resid_tile(const Phase& ph, const Io& io, int M, int rb, int j, uint16_t (&hold)[4],
                                                int lane) {
  const int g = lane >> 2, c = lane & 3;
  const uint16_t* hp = static_cast<const uint16_t*>(io.buf[ph.out]);
  const int nb = rb * kRowBlock + g;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int t = 8 * j + 2 * c + h;
      unsigned short b = 0;
      if (t < M) asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(b) : "l"(hp + (size_t)t * ph.out_ld + nb + 8 * r));
      hold[2 * r + h] = b;
    }
}
template <int NT>
__device__ __forceinline__ void load_resid(const Phase& ph, const Io& io, int M, int rb, uint16_t (&hold)[NT][4],
                                           int lane) {
#pragma unroll
  for (int j = 0; j < NT; ++j) load_resid_tile(ph, io, M, rb, j, hold[j], lane);
}

// Token tile j of the finished row block rb: v (fp32, un-scaled activations, before the weight
// scale); interleaved layout: v = the gate rows, u = the up rows (else u is unused).
template <int NT, bool kHead>
__device__ __forceinline__ void epilogue_tile(const Phase& ph, const Io& io, int M, int rb, int j, const float (&v)[4],
                                              const float (&u)[4], const uint16_t (&hold)[4], HeadBest<NT>& hb,
                                              int lane) {
  const int g = lane >> 2, c = lane & 3;
  if (ph.layout == kInterleaved) {  // a = bf16(silu(s0 * gate) * s1 * up)
    uint16_t* out = static_cast<uint16_t*>(io.buf[ph.out]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = 8 * j + 2 * c + h;
      if (t >= M) continue;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int f = rb * kRowBlock + g + 8 * r;
        const float gt = ph.s0 * v[2 * r + h], up = ph.s1 * u[2 * r + h];
        out[(size_t)t * ph.out_ld + f] = bf16_bits(gt / (1.0f + expf(-gt)) * up);
      }
    }
    return;
  }
  const bool seg1 = rb >= ph.rb1;
  const float s = seg1 ? ph.s1 : ph.s0;
  const int nb = (seg1 ? rb - ph.rb1 : rb) * kRowBlock + g;
  float sq[2] = {0.0f, 0.0f};  // kSsWrite: this lane's squares of the stored values, per token
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = 8 * j + 2 * c + h;
    if (t >= M) continue;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int n = nb + 8 * r;
      const float val = s * v[2 * r + h];
      const size_t o = (size_t)t * ph.out_ld + n;
      switch (ph.epi) {
        case kEpiF32:
          static_cast<float*>(io.buf[ph.out])[o] = val;
          break;
        case kEpiZ:
          if (!seg1 && n < ph.out_cols) static_cast<uint16_t*>(io.buf[ph.out])[o] = bf16_bits(val);
          break;
        case kEpiU:  // column = the virtual row: segment 1 follows segment 0
          static_cast<uint16_t*>(io.buf[ph.out])[(size_t)t * ph.out_ld + rb * kRowBlock + g + 8 * r] = bf16_bits(val);
          break;
        case kEpiResid: {
          uint16_t* hp = static_cast<uint16_t*>(io.buf[ph.out]);
          const uint16_t nv = bf16_bits(bf16_bits_to_float(hold[2 * r + h]) + val);
          hp[o] = nv;
          if constexpr (NT > 1) {
            const float f = bf16_bits_to_float(nv);
            sq[h] = fmaf(f, f, sq[h]);
          }
          if (ph.trace_slot >= 0 && io.buf[kBufTrace])
            static_cast<uint16_t*>(io.buf[kBufTrace])[(size_t)ph.trace_slot * io.trace_stride + o] = nv;
          break;
        }
        case kEpiHead: {
          if constexpr (kHead) {  // only the head phase's instantiation carries the argmax state
            if (io.buf[kBufLogits]) static_cast<float*>(io.buf[kBufLogits])[o] = val;
            const float key = isnan(val) ? -INFINITY : val;
            if (am_better(key, n, hb.v[j][h], hb.i[j][h])) {
              hb.v[j][h] = key;
              hb.i[j][h] = n;
            }
          }
          break;
        }
        default:
          break;
      }
    }
  }
  if constexpr (NT > 1) {
    if (ph.epi == kEpiResid && (ph.ss & kSsWrite)) {  // the row block's 16 rows: lanes g = 0..7 (xor 4, 8, 16)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float q = sq[h];
        q += __shfl_xor_sync(0xffffffffu, q, 4);
        q += __shfl_xor_sync(0xffffffffu, q, 8);
        q += __shfl_xor_sync(0xffffffffu, q, 16);
        const int t = 8 * j + 2 * c + h;
        if (g == 0 && t < M) io.rss[(size_t)t * io.rss_ld + (seg1 ? rb - ph.rb1 : rb)] = q;
      }
    }
  }
}

// The finished row block rb, every token tile.
template <int NT, bool kHead>
__device__ void epilogue(const Phase& ph, const Io& io, int M, int rb, const float (&v)[NT][4],
                         const float (&u)[NT][4], const uint16_t (&hold)[NT][4], HeadBest<NT>& hb, int lane) {
#pragma unroll
  for (int j = 0; j < NT; ++j) epilogue_tile<NT, kHead>(ph, io, M, rb, j, v[j], u[j], hold[j], hb, lane);
}

// A partial of a row block (one slot: 32 lanes x cs_lane floats) is laid out token tile major:
// sub-block j (v) and NT + j (u, interleaved) of 32 lanes x 4 floats each, so that one tile's 32
// lanes read or write 512 contiguous bytes.  slot: the slot's first float; this lane's float4 of
// sub-block b is at slot + (32 b + lane) * 4.
template <int NT>
__device__ __forceinline__ void store_partial(float* slot, int lane, bool two, const float (&v)[NT][4],
                                              const float (&u)[NT][4]) {
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    *reinterpret_cast<float4*>(slot + (32 * j + lane) * 4) = make_float4(v[j][0], v[j][1], v[j][2], v[j][3]);
    if (two)
      *reinterpret_cast<float4*>(slot + (32 * (NT + j) + lane) * 4) = make_float4(u[j][0], u[j][1], u[j][2], u[j][3]);
  }
}

// Finishes the warp's part of row block rb (the task of this CTA's K slice): v = its sum over the
// slice (plain: acc + acc2, two MMA chains; interleaved: acc = gate rows, acc2 = up rows, in u).
//  * Several warps of the CTA share the row block: each stores its partial in the CTA's slot of its
//    first or last row block and arrives on a shared-memory counter (CTA scope); the last to arrive
//    sums the slots in warp order, so the result does not depend on who arrives last.
//  * One K slice (ks == 1): the finished row block runs its epilogue here.  Several K slices: its
//    sum over this slice goes to the cross-slice slot, summed after the next grid barrier.
// Register budget: at 3-4 token tiles the per-token scales are read from shared memory here (tsc is
// unused), so that they do not stay live through the unit loop; at 1-2 tiles the caller's copy is
// cheaper.
template <int NT>
constexpr bool kScalesFromSmem = NT >= 3;
template <int NT, bool kHead>
__device__ void flush(const Phase& ph, const Part& P, const Io& io, int M, int G, int w, int rb, const float (&acc)[NT][4],
                      const float (&acc2)[NT][4], const float (&tsc)[NT][2], HeadBest<NT>& hb, SmemMisc& sm,
                      int lane) {
  // P is the shared-memory copy: nothing of it stays live in the unit loop
  const bool two = ph.layout == kInterleaved;
  const int c = lane & 3;
  float v[NT][4], u[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float sc;
      if constexpr (kScalesFromSmem<NT>)
        sc = sm.xscale[8 * j + 2 * c + (r & 1)];
      else
        sc = tsc[j][r & 1];
      v[j][r] = (two ? acc[j][r] : acc[j][r] + acc2[j][r]) * sc;
      u[j][r] = two ? acc2[j][r] * sc : 0.0f;
    }
  const size_t slot_floats = 32 * (size_t)io.cs_lane;
  const int kgn = P.S.kgn, r0 = (rb - P.rb0) * kgn;
  const int wf = wowner(P, r0), wl = wowner(P, r0 + kgn - 1);
  // The residual inputs of a row block this warp finishes, loaded ahead of the partials' round trip.
  uint16_t hold[NT][4];
  const bool resid = ph.ks == 1 && ph.epi == kEpiResid;
  if (resid && wf == wl) load_resid<NT>(ph, io, M, rb, hold, lane);
  if (wf != wl) {
    const size_t cta_slots = (size_t)blockIdx.x * kWarps * 2;
    const int sel = wbegin(P, w) >= r0 ? 0 : 1;
    store_partial<NT>(io.cslots + (cta_slots + 2 * w + sel) * slot_floats, lane, two, v, u);
    // the same partial in the warp's lane quarter of tensor memory, for a contributor of that quarter
    const uint32_t tq = sm.tmem + ((uint32_t)(32 * (w >> 2)) << 16);
    {
      const uint32_t col = (uint32_t)((2 * (w & 3) + sel) * io.cs_lane);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        tmem_st4(tq + col + 4 * j, v[j]);
        if (two) tmem_st4(tq + col + 4 * (NT + j), u[j]);
      }
      tmem_wait_st();
      tmem_fence_before();
    }
    // Release (CTA scope): the warp's stores, ordered before by the warp barrier, are visible to the
    // warp that finishes the row block; acquire: that warp then sees every contributor's partial.
    __syncwarp();
    unsigned old = 0;
    if (lane == 0) old = atom_add_acq_rel_cta_smem(&sm.tcnt[wf], 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old + 1 != (unsigned)(wl - wf + 1)) return;
    __syncwarp();
    tmem_fence_after();
    if (resid) load_resid<NT>(ph, io, M, rb, hold, lane);
    float ov[NT][4], ou[NT][4];  // this warp's own partial
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        ov[j][r] = v[j][r];
        ou[j][r] = u[j][r];
        v[j][r] = u[j][r] = 0.0f;
      }
    for (int c = wf; c <= wl; ++c) {
      const int sel_c = wbegin(P, c) >= r0 ? 0 : 1;
      if (c == w) {
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            v[j][r] += ov[j][r];
            if (two) u[j][r] += ou[j][r];
          }
      } else if ((c >> 2) == (w >> 2)) {  // the same lane quarter: from tensor memory
        const uint32_t col = (uint32_t)((2 * (c & 3) + sel_c) * io.cs_lane);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          float q[4];
          tmem_ld4(tq + col + 4 * j, q);
#pragma unroll
          for (int r = 0; r < 4; ++r) v[j][r] += q[r];
          if (two) {
            tmem_ld4(tq + col + 4 * (NT + j), q);
#pragma unroll
            for (int r = 0; r < 4; ++r) u[j][r] += q[r];
          }
        }
      } else {
        const float* sl = io.cslots + (cta_slots + 2 * c + sel_c) * slot_floats + lane * 4;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const float4 q = *reinterpret_cast<const float4*>(sl + 128 * j);
          v[j][0] += q.x;
          v[j][1] += q.y;
          v[j][2] += q.z;
          v[j][3] += q.w;
          if (two) {
            const float4 q2 = *reinterpret_cast<const float4*>(sl + 128 * (NT + j));
            u[j][0] += q2.x;
            u[j][1] += q2.y;
            u[j][2] += q2.z;
            u[j][3] += q2.w;
          }
        }
      }
    }
    if (lane == 0) sm.tcnt[wf] = 0u;
  }
  if (ph.ks > 1) {
    store_partial<NT>(io.xslots + ((size_t)rb * ph.ks + P.sidx) * slot_floats, lane, two, v, u);
    return;
  }
  epilogue<NT, kHead>(ph, io, M, rb, v, u, hold, hb, lane);
}

// Phases with several K slices, after the grid barrier that follows the units: token tile j of
// row block rb is summed over its slices in slice order by one warp (items (rb, j) spread over the
// CTAs first), its slice partials loaded 8 slices at a time, then its epilogue runs.
template <int NT, bool kHead>
__device__ void cross_slice_fixup(const Phase& ph, const Io& io, int M, int G, HeadBest<NT>& hb, int warp,
                                  int lane) {
  const bool two = ph.layout == kInterleaved;
  const size_t slot_floats = 32 * (size_t)io.cs_lane;
  const int ks = ph.ks;
  for (int item = warp * G + (int)blockIdx.x; item < ph.RB * NT; item += G * kWarps) {
    const int rb = item / NT, j = item - rb * NT;
    uint16_t hold[4];
    if (ph.epi == kEpiResid) load_resid_tile(ph, io, M, rb, j, hold, lane);
    float v[4] = {0.0f, 0.0f, 0.0f, 0.0f}, u[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const float* base = io.xslots + (size_t)rb * ks * slot_floats + (32 * j + lane) * 4;
    for (int s0 = 0; s0 < ks; s0 += 8) {
      float4 q[8], q2[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float* sl = base + (size_t)(s0 + i) * slot_floats;
        q[i] = s0 + i < ks ? ldcg_f4(sl) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        q2[i] = two && s0 + i < ks ? ldcg_f4(sl + 128 * NT) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (s0 + i >= ks) break;
        v[0] += q[i].x;
        v[1] += q[i].y;
        v[2] += q[i].z;
        v[3] += q[i].w;
        u[0] += q2[i].x;
        u[1] += q2[i].y;
        u[2] += q2[i].z;
        u[3] += q2[i].w;
      }
    }
    epilogue_tile<NT, kHead>(ph, io, M, rb, j, v, u, hold, hb, lane);
  }
}

// Head phase end: per-token argmax of the CTA, then the last CTA to finish reduces all CTAs in a
// fixed order and runs the acceptance.
template <int NT>
__device__ __noinline__ void head_finish(const Program& prog, const Io& io, int G, HeadBest<NT>& hb, uint8_t* xs,
                                         SmemMisc& sm, int warp, int lane) {
  const int M = prog.M, tid = threadIdx.x;
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      am_shfl_xor(hb.v[j][h], hb.i[j][h], 4);
      am_shfl_xor(hb.v[j][h], hb.i[j][h], 8);
      am_shfl_xor(hb.v[j][h], hb.i[j][h], 16);
    }
  __syncthreads();  // every warp is done with the activation fragments: reuse that space
  float* rv = reinterpret_cast<float*>(xs);
  int* ri = reinterpret_cast<int*>(xs + kWarps * kMaxM * sizeof(float));
  if (lane < 4)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int t = 8 * j + 2 * lane + h;
        rv[warp * kMaxM + t] = hb.v[j][h];
        ri[warp * kMaxM + t] = hb.i[j][h];
      }
  __syncthreads();
  if (tid < M) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int w = 0; w < kWarps; ++w)
      if (am_better(rv[w * kMaxM + tid], ri[w * kMaxM + tid], bv, bi)) {
        bv = rv[w * kMaxM + tid];
        bi = ri[w * kMaxM + tid];
      }
    io.head_aux[((size_t)blockIdx.x * kMaxM + tid) * 2] = bv;
    io.head_aux[((size_t)blockIdx.x * kMaxM + tid) * 2 + 1] = __int_as_float(bi);
    __threadfence();
  }
  __syncthreads();
  if (tid == 0) sm.flag = atomicAdd(io.head_cnt, 1u) + 1 == (unsigned)G;
  __syncthreads();
  if (!sm.flag) return;
  __threadfence();
  // Warp w reduces tokens w, w + 16 (its lanes stride over the CTAs, then a warp reduction); the
  // winner (largest value, then lowest index) is the same in any order.
  for (int t = warp; t < M; t += kWarps) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int c = lane; c < G; c += 32) {
      const float2 e = __ldcg(reinterpret_cast<const float2*>(io.head_aux) + (size_t)c * kMaxM + t);
      const int ei = __float_as_int(e.y);
      if (am_better(e.x, ei, bv, bi)) {
        bv = e.x;
        bi = ei;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) am_shfl_xor(bv, bi, o);
    if (lane == 0) {
      if (bi == 0x7fffffff) bi = 0;
      sm.tok[t] = bi;
      io.argmax[t] = bi;
    }
  }
  __syncthreads();
  if (tid < M / prog.rows) accept_lane(tid, prog.rows, sm.tok, io.pending, io.n_commit, io.committed);
  if (tid == 0) *io.head_cnt = 0u;
}

// ---------------------------------------------------------------- grid barrier
// One monotonic arrival counter per launch: barrier b releases once it reaches G * (b + 1), so the
// last CTA to arrive has nothing more to do (its atomic is the release) and the others poll one
// word.  The last CTA to leave the kernel resets the counter (and the exit counter) for the next
// launch.
__device__ __forceinline__ void grid_barrier(const Io& io, int G, unsigned target, SmemMisc& sm) {
  __syncthreads();
  bool skip = false;
#ifdef VP_WAIT_TEST
  // Wait-test hook (workspace word kWsTestSkip): CTA (value - 1) leaves its first arrival out, so
  // that every other CTA's wait runs out.
  skip = target == (unsigned)G && ((const volatile int*)io.status)[kWsTestSkip / sizeof(int)] == (int)blockIdx.x + 1;
#endif
  if (threadIdx.x == 0 && !skip) {
    __threadfence();
    const unsigned arrived = atomicAdd(io.bar, 1u) + 1u;
    if (arrived < target && !sm.abort) {
      uint32_t n = 0;
      while (ld_acquire_gpu(io.bar) < target) {
        if (++n > kBarrierPolls) {  // about 1-2 s (milliseconds in the wait-test build)
          sm.abort = 1;
          atomicExch(io.status, kStatusTimeout);
          break;
        }
        if (n > 256) __nanosleep(32);
      }
    }
  }
  __syncthreads();
}
__device__ __forceinline__ void grid_exit(const Io& io, int G) {
  __syncthreads();
  if (threadIdx.x == 0 && atomicAdd(io.bar + 1, 1u) + 1u == (unsigned)G) {
    atomicExch(io.bar, 0u);
    atomicExch(io.bar + 1, 0u);
    VP_TRACE_LAUNCH_DONE();
  }
}

// The streaming part of phase p (after its staging): the warp's units, its row blocks' fixups, the
// cross-slice sums and the head's argmax and acceptance.  Instantiated twice: only the head phase's
// copy (kHead) keeps the running argmax in registers through the unit loop.
template <int NT, bool kQ4, bool kHead>
__device__ __forceinline__ void phase_units(const Program& prog, const Io& io, const Phase& ph, const PhaseSlot& sl,
                                            int p, uint8_t* xs, SmemMisc& sm, uint32_t ring_w, uint64_t pol,
                                            unsigned& issued, unsigned& seq, unsigned& nbar) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  Cursor& pc = sm.cur[warp];
  const Part P = sl.part;
  const int ck = chunk_k(ph.fmt);
  float tsc[NT][2];  // per-token scales (unused at 3-4 tiles: see flush)
  if constexpr (!kScalesFromSmem<NT>) {
    const int c = lane & 3;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      tsc[j][0] = sm.xscale[8 * j + 2 * c];
      tsc[j][1] = sm.xscale[8 * j + 2 * c + 1];
    }
  }
  HeadBest<NT> hb;
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      hb.v[j][h] = -INFINITY;
      hb.i[j][h] = 0x7fffffff;
    }
  const int wr = range_of(warp);  // the warp's range index within the CTA
  const int ub = sl.wb[wr], ue = sl.wb[wr + 1];
  const uint32_t xlane = smem_addr(xs) + lane * 16;
  const int pair_stride = (ck / 32) * NT * 512;  // bytes of fragments per chunk
  const uint32_t chunk_bytes = 2u * strip_bytes(ph.fmt);
  const bool two = ph.layout == kInterleaved;
  int rb = ub < ue ? P.rb0 + ub / P.S.kgn : 0, kgl = ub < ue ? ub % P.S.kgn : 0;
  float acc[NT][4], acc2[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[j][r] = acc2[j][r] = 0.0f;
  int cur = -1;
  for (int u = ub; u < ue; ++u) {
    if (rb != cur) {
      if (cur >= 0) {
        flush<NT, kHead>(ph, sl.part, io, prog.M, G, wr, cur, acc, acc2, tsc, hb, sm, lane);
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[j][r] = acc2[j][r] = 0.0f;
      }
      cur = rb;
    }
    const int slot = (int)(seq % kSlots);
    if (!sm.abort && !mbar_wait_bounded(&sm.full[warp][slot], (seq / kSlots) & 1u)) {
      sm.abort = 1;
      atomicExch(io.status, kStatusTimeout);
    }
    const uint32_t ua = ring_w + slot * kSlotBytes, xa = xlane + kgl * ph.grp * pair_stride;
    if constexpr (kQ4) {  // one or two consecutive chunks of the row block, 4 groups each
      unit_q4<NT>(ua, xa, lane, acc);
      if ((P.S.kg0 + kgl) * 2 + 1 < ph.KC) unit_q4<NT>(ua + chunk_bytes, xa + pair_stride, lane, acc);
    } else if (two) {  // gate chunk -> acc, up chunk -> acc2, same activations (NVFP4 only)
      unit_nvfp4_pair<NT>(ua, ua + chunk_bytes, xa, lane, acc, acc2);
    } else {  // one or two consecutive chunks of the row block (one chain per n-tile, two if NT = 1)
      const bool second = ph.grp == 2 && (P.S.kg0 + kgl) * 2 + 1 < ph.KC;
      if (ph.fmt == kFmtNvfp4) {
        unit_nvfp4<NT>(ua, xa, lane, acc, NT == 1 ? acc2 : acc);
        if (second) unit_nvfp4<NT>(ua + chunk_bytes, xa + pair_stride, lane, acc, NT == 1 ? acc2 : acc);
      } else {
        unit_fp8<NT>(ua, xa, lane, acc, NT == 1 ? acc2 : acc);
        if (second) unit_fp8<NT>(ua + chunk_bytes, xa + pair_stride, lane, acc, NT == 1 ? acc2 : acc);
      }
    }
    __syncwarp();
    if (lane == 0) {  // the producer works on a register copy of its cursor
      Cursor c;
      cursor_load(c, pc);
      if (c.p < prog.n && !sm.abort) {
        fence_proxy_async_smem();
        issue_unit(c, ua, &sm.full[warp][slot], pol);
        cursor_next(c, prog, sm.ps, G, cta, warp);
        ++issued;
        cursor_load(pc, c);
      }
    }
    ++seq;
    if (++kgl == P.S.kgn) {
      kgl = 0;
      ++rb;
    }
  }
  VP_TRACE(lane == 0, p, 2 + warp);
  if (cur >= 0) flush<NT, kHead>(ph, sl.part, io, prog.M, G, wr, cur, acc, acc2, tsc, hb, sm, lane);
  if (p + 2 < prog.n) {  // the first warp of the CTA done with this phase fills phase p + 2's slot
    int won = 0;
    if (lane == 0) won = atomicCAS(&sm.fillp, p, p + 1) == p;
    if (__shfl_sync(0xffffffffu, won, 0)) fill_slot(sm.ps[(p + 2) % kPhaseSlots], prog, io, p + 2, G, cta, lane);
  }
  VP_TRACE(lane == 0, p, 18 + warp);
  if (ph.ks > 1) {  // every row block's slices meet after a grid barrier
    grid_barrier(io, G, (unsigned)G * ++nbar, sm);
    cross_slice_fixup<NT, kHead>(ph, io, prog.M, G, hb, warp, lane);
    VP_TRACE(threadIdx.x == 0, p, 35);
  }
  if (kHead && ph.epi == kEpiHead) head_finish<NT>(prog, io, G, hb, xs, sm, warp, lane);
}

// ---------------------------------------------------------------- the kernel
template <int NT, bool kQ4>
__global__ void __launch_bounds__(kThreads, 1) exec_kernel(const __grid_constant__ Program prog,
                                                           const __grid_constant__ Io io) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* xs = smem + kRingBytes;
  SmemMisc& sm = *reinterpret_cast<SmemMisc*>(smem + kRingBytes + kXBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, c = lane & 3;
  const int G = gridDim.x, cta = blockIdx.x;

  if (lane == 0) {
    for (int s = 0; s < kSlots; ++s) mbar_init(&sm.full[warp][s], 1);
    sm.tcnt[warp] = 0u;
  }
  if (threadIdx.x == 0) {
    sm.abort = 0;
    sm.fillp = 0;
    sm.ps[2].idx = -1;
  }
  VP_TRACE_INIT();
  if (warp == 0) tmem_alloc(&sm.tmem, kTmemCols<NT>);
  if (warp == 1) fill_slot(sm.ps[0], prog, io, 0, G, cta, lane);
  if (warp == 2) {
    if (prog.n > 1)
      fill_slot(sm.ps[1], prog, io, 1, G, cta, lane);
    else if (lane == 0)
      sm.ps[1].idx = -1;
  }
  fence_mbar_init();
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();

  const uint32_t ring_w = smem_addr(smem) + warp * kSlots * kSlotBytes;
  uint64_t pol = 0;
  Cursor& pc = sm.cur[warp];  // next unit to copy into the ring (lane 0)
  unsigned issued = 0;
  if (lane == 0) {
    pol = l2_evict_first_policy();
    pc.p = 0;
    cursor_seek(pc, prog, sm.ps, G, cta, warp);
    for (; issued < (unsigned)kSlots && pc.p < prog.n; ++issued) {
      issue_unit(pc, ring_w + issued * kSlotBytes, &sm.full[warp][issued], pol);
      cursor_next(pc, prog, sm.ps, G, cta, warp);
    }
  }

  unsigned seq = 0, nbar = 0;
  for (int p = 0; p < prog.n; ++p) {
    const PhaseSlot& sl = sm.ps[p % kPhaseSlots];
    const Phase& ph = prog.ph[p];
    VP_TRACE(threadIdx.x == 0, p, 0);
    const Part P = sl.part;
    const int ck = chunk_k(ph.fmt), kc0 = P.S.kg0 * ph.grp;
    stage_x<NT>(prog, ph, io, kc0 * ck, (min(kc0 + P.S.kgn * ph.grp, ph.KC) - kc0) * ck, xs, sm, p);
    VP_TRACE(threadIdx.x == 0, p, 1);
    // the streaming part of the phase
    // (at 4 tiles the other phases use an instantiation without the running argmax: registers)
    if (NT == 4 && ph.epi != kEpiHead)
      phase_units<NT, kQ4, false>(prog, io, ph, sl, p, xs, sm, ring_w, pol, issued, seq, nbar);
    else
      phase_units<NT, kQ4, true>(prog, io, ph, sl, p, xs, sm, ring_w, pol, issued, seq, nbar);
    if (p + 1 < prog.n) grid_barrier(io, G, (unsigned)G * ++nbar, sm);
    VP_TRACE(threadIdx.x == 0, p, 34);
  }
  // Copies still in flight (only after a timeout, when the units are consumed without waiting):
  // wait for the last copy issued into each slot before the CTA's memory goes away.  A copy goes
  // into a slot only after the wait for that slot's previous copy, so the last one is the only one
  // that can be pending, and waiting on its phase parity is exact whether or not it has landed.
  if (lane == 0)
    for (unsigned s = 0; s < (unsigned)kSlots && s < issued; ++s) {
      const unsigned k = issued - 1 - ((issued - 1 - s) % kSlots);  // the last copy into slot s
      mbar_wait_bounded(&sm.full[warp][s], (k / kSlots) & 1u);
    }
  // Every CTA takes the same barriers; a program that took any (several phases, or one phase cut
  // into K slices) resets the counter on the way out, so the workspace is ready for the next call.
  if (nbar > 0) grid_exit(io, G);
  tmem_fence_before();
  __syncthreads();  // no warp touches tensor memory any more
  tmem_fence_after();
  if (warp == 0) tmem_dealloc(sm.tmem, kTmemCols<NT>);
}

// ---------------------------------------------------------------- launch (host)
// One instantiation per translation unit that uses it (exec_nt12.cu, exec_nt34.cu, exec_q4.cu), so
// the kernels compile in parallel.
template <int NT, bool kQ4>
cudaError_t launch_exec_kernel(const Program& prog, const Io& io, int grid, cudaStream_t s, bool coop) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(exec_kernel<NT, kQ4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = coop ? at : nullptr;
  cfg.numAttrs = coop ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, exec_kernel<NT, kQ4>, prog, io);
}

}  // namespace vp
