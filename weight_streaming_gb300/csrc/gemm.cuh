// The skinny block-quantized GEMM of the verify pass: Y[M][N] = X[M][K] * W[N][K]^T for
// M = 1..32 rows, with NVFP4 (E2M1 code x E4M3 scale per 16) or FP8 E4M3 weights, and fused
// epilogues (fp32 store, bf16 prefix store, SiLU(gate)*up, residual add + RMS statistics, and the
// vocabulary head's argmax + greedy acceptance).
//
// Sources: "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max" -- "What one token
// costs the bus" (the NVFP4/FP8 weight groups one pass reads) and "Formats, and what runs where"
// (NVFP4 dequantisation, tensor scale as a multiplier, weight-only arithmetic with BF16
// activations and wide accumulation); "Beating Splash on an M5 Max" -- "The kernels were not the
// gap" (split-K across threadgroups for the narrow 5120-wide projections) and "The bugs a second
// reviewer found" (one argmax tie rule everywhere).
//
// GB300 design (not the pages' Metal tiles):
//  * One persistent CTA per SM: 8 consumer warps + 1 producer warp.  The (256-row group, 64-wide K
//    quad) units of the whole matrix are split into equal contiguous ranges, one per CTA (stream-K),
//    so every SM streams the same number of bytes.
//  * The producer warp moves each unit's packed weights (a contiguous 9 KB NVFP4 / 16 KB FP8 slab
//    chunk) into a deep shared-memory ring with 1-D bulk copies (cp.async.bulk, evict-first L2
//    policy) completing on mbarriers.  Weights never depend on the previous kernel, so under
//    programmatic dependent launch the ring fills while the previous kernel drains.
//  * Consumer warps stage the activation rows they need once per batch as f16 MMA fragments, each
//    row scaled by an exact power of two (so bf16 values fit f16 exactly), then per unit dequantise
//    the weights in registers (cvt e2m1x2/e4m3x2 -> f16x2, times the f16 block scale: exact) and run
//    m16n8k16 MMAs with fp32 accumulation: weights are the 16-row A operand, the M tokens the n = 8
//    columns, so no MMA work is wasted at M = 8.
//  * Partial sums of a group that several CTAs share go to the workspace; the last CTA to arrive
//    (atomic counter, no waiting) adds them in CTA order -- a fixed order, so results are
//    bit-reproducible -- and runs the epilogue.  A per-task counter lets the last group run the
//    cross-group finisher (1/rms per row, or argmax + acceptance).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace vp {

enum : int { kStatusOk = 0, kStatusTimeout = 6 };

template <int FMT>
struct FmtTraits;
template <>
struct FmtTraits<kFmtNvfp4> {
  static constexpr int kBlock = kNvfp4BlockBytes;
  static constexpr int kStages = kNvfp4Stages;
};
template <>
struct FmtTraits<kFmtFp8> {
  static constexpr int kBlock = kFp8BlockBytes;
  static constexpr int kStages = kFp8Stages;
};

template <int FMT>
__host__ __device__ constexpr int stage_bytes() {
  return FmtTraits<FMT>::kBlock * kBlocksPerSlab;
}
template <int FMT>
__host__ __device__ constexpr int ring_bytes() {
  return stage_bytes<FMT>() * FmtTraits<FMT>::kStages;
}

struct SmemMisc {
  uint64_t full[16];
  uint64_t empty[16];
  int xexp[kMaxM];
  int xmax[kMaxM];
  float red_v[kConsumerWarps][kMaxM];
  int red_i[kConsumerWarps][kMaxM];
  int tok[kMaxM];
  int flag_last;
  int flag_task_last;
  volatile int abort;
};

template <int FMT>
__host__ __device__ constexpr size_t gemm_smem_bytes() {
  return (size_t)ring_bytes<FMT>() + kXBufBytes + sizeof(SmemMisc);
}

// ---------------------------------------------------------------- stream-K decomposition
__device__ __forceinline__ long long unit_begin(long long U, int G, int c) { return (long long)c * U / G; }
// The CTA whose range holds unit u (grid <= U, so every CTA's range is non-empty).
__device__ __forceinline__ int cta_of_unit(long long U, int G, long long u) {
  return (int)(((u + 1) * (long long)G + U - 1) / U - 1);
}

// Geometry of a 256-row virtual group.
struct GroupGeom {
  int seg;       // segment (non-interleaved)
  int row0;      // first segment-local row of the group (non-interleaved) / first feature (interleaved)
  int nrb;       // valid 16-row blocks in the group (interleaved: per segment, <= 8)
  const uint8_t* src[2];  // packed address of this group's quad 0 for each copy
  int src_stride[2];      // bytes between consecutive quads of this group
  int copy_bytes[2];      // bytes per quad per copy (0 = no copy)
  int dst_slot[2];        // first stage slot of each copy
};

template <int FMT>
__device__ __forceinline__ GroupGeom group_geom(const GemmParams& p, int g) {
  constexpr int B = FmtTraits<FMT>::kBlock;
  GroupGeom gg;
  const int nq = p.nq;
  if (p.interleave) {
    // group g = features [128 g, 128 g + 128): row-blocks 8(g%2).. of slab g/2 of each segment
    const int rows = p.seg_rows[0];
    const int slab = g >> 1;
    const int slab_rb = min(kBlocksPerSlab, (rows - slab * kSlabRows) / kRowsPerBlock);
    const int rb_in = (g & 1) * 8;
    gg.seg = 0;
    gg.row0 = g * 128;
    gg.nrb = min(8, slab_rb - rb_in);
    for (int s = 0; s < 2; ++s) {
      gg.src[s] = p.w[s] + ((size_t)slab * kBlocksPerSlab * nq + rb_in) * B;
      gg.src_stride[s] = slab_rb * B;
      gg.copy_bytes[s] = gg.nrb * B;
      gg.dst_slot[s] = 8 * s;
    }
  } else {
    const int seg = g < p.seg0_groups ? 0 : 1;
    const int gl = seg ? g - p.seg0_groups : g;
    const int rows = p.seg_rows[seg];
    gg.seg = seg;
    gg.row0 = gl * kSlabRows;
    gg.nrb = min(kBlocksPerSlab, (rows - gg.row0) / kRowsPerBlock);
    gg.src[0] = p.w[seg] + (size_t)gl * kBlocksPerSlab * nq * B;
    gg.src_stride[0] = gg.nrb * B;
    gg.copy_bytes[0] = gg.nrb * B;
    gg.dst_slot[0] = 0;
    gg.src[1] = nullptr;
    gg.src_stride[1] = 0;
    gg.copy_bytes[1] = 0;
    gg.dst_slot[1] = 0;
  }
  return gg;
}

// ---------------------------------------------------------------- activation staging
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// Stages rows m < MT*8 of X for the quads [qa0, qb0) and [qa1, qb1) into f16 MMA B fragments at
// slot (q - origin).  Each row m is scaled by 2^-xexp[m], chosen from the row's largest magnitude
// over the staged quads so that it lies in [2^14, 2^15): every bf16 value then converts to f16
// exactly (f16 has more significand bits) unless it is over 2^31 times smaller than that maximum.
// Pass 1 reads X once (16-byte loads, all consumer threads), applies the optional row multiplier
// (bf16-rounded, as RMSNorm's output), stores the bf16 pairs straight into their fragment slots and
// takes the row maxima; pass 2 rescales every fragment word in place to f16.
template <int MT>
__device__ void stage_x(const GemmParams& p, uint32_t* xbuf, SmemMisc& sm, int origin, int qa0, int qb0,
                        int qa1, int qb1, int ctid) {
  if (ctid < MT * 8) sm.xmax[ctid] = 0;
  named_bar_sync(1, kConsumerThreads);
  const int n0 = (qb0 - qa0) * 8, n1 = (qb1 - qa1) * 8;  // 8-element chunks per row
  const int per_row = n0 + n1;
  const int total = MT * 8 * per_row;
  const bool use_rs = p.x_rowscale != nullptr;
#pragma unroll 4
  for (int c = ctid; c < total; c += kConsumerThreads) {
    const int m = c / per_row, jj = c - m * per_row;
    const int kc = jj < n0 ? qa0 * 8 + jj : qa1 * 8 + (jj - n0);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (m < p.M) {
      const uint4 raw = ldcg128(p.x + (size_t)m * p.x_ld + (size_t)kc * 8);
      w[0] = raw.x;
      w[1] = raw.y;
      w[2] = raw.z;
      w[3] = raw.w;
      float mx = 0.0f;
      const float rs = use_rs ? p.x_rowscale[m] : 1.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float v0 = bf16_bits_to_float(w[i] & 0xFFFFu), v1 = bf16_bits_to_float(w[i] >> 16);
        if (use_rs) {
          v0 = round_bf16(v0 * rs);
          v1 = round_bf16(v1 * rs);
          w[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v0)) |
                 ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v1)) << 16);
        }
        mx = fmaxf(mx, fmaxf(fabsf(v0), fabsf(v1)));
      }
      atomicMax(&sm.xmax[m], __float_as_int(mx));  // non-negative floats order like their bits
    }
    const int k0 = kc * 8, q = k0 >> 6, kl = k0 & 63;
    const int slot = q - origin, j16 = kl >> 4, reg = (kl & 15) >> 3;
    const int nt = m >> 3, g = m & 7;
    uint32_t* dst = xbuf + (((slot * 4 + j16) * MT + nt) * 32 + g * 4) * 2 + reg;
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[2 * i] = w[i];
  }
  named_bar_sync(1, kConsumerThreads);
  if (ctid < MT * 8) {
    const float mx = __int_as_float(sm.xmax[ctid]);
    int e = 0;
    if (mx > 0.0f) {
      const int ef = (__float_as_uint(mx) >> 23) & 0xFF;
      e = (ef ? ef - 127 : -127) - 14;  // floor(log2(mx)) - 14 (subnormal maxima: -127 - 14)
    }
    sm.xexp[ctid] = e;
  }
  named_bar_sync(1, kConsumerThreads);
  for (int iv = 0; iv < 2; ++iv) {
    const int qa = iv ? qa1 : qa0, qb = iv ? qb1 : qb0;
    if (qb <= qa) continue;
    uint32_t* base = xbuf + (size_t)(qa - origin) * (256 * MT);
    const int nwords = (qb - qa) * 256 * MT;
#pragma unroll 4
    for (int wi = ctid; wi < nwords; wi += kConsumerThreads) {
      const int nt = (wi >> 6) % MT, m = nt * 8 + ((wi >> 3) & 7);
      if (m >= p.M) continue;
      const uint32_t wv = base[wi];
      const int e = sm.xexp[m];
      const __half2 h = __floats2half2_rn(mul_pow2(bf16_bits_to_float(wv & 0xFFFFu), -e),
                                          mul_pow2(bf16_bits_to_float(wv >> 16), -e));
      base[wi] = *reinterpret_cast<const uint32_t*>(&h);
    }
  }
}

// ---------------------------------------------------------------- one unit of MMA work
template <int FMT, int MT>
__device__ __forceinline__ void compute_unit(const uint8_t* stage, const uint32_t* xq, int sA, int sB, bool vA,
                                             bool vB, int lane, float (&acc)[2][MT][4]) {
  if constexpr (FMT == kFmtNvfp4) {
    const int gq = lane >> 2;
    uint4 cw[2];
    uint2 sw[2];
    cw[0] = lds128(stage + sA * kNvfp4BlockBytes + lane * 16);
    sw[0] = lds64(stage + sA * kNvfp4BlockBytes + 512 + gq * 8);
    cw[1] = lds128(stage + sB * kNvfp4BlockBytes + lane * 16);
    sw[1] = lds64(stage + sB * kNvfp4BlockBytes + 512 + gq * 8);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t b0[MT], b1[MT];
#pragma unroll
      for (int nt = 0; nt < MT; ++nt) {
        const uint2 bb = lds64(xq + ((j * MT + nt) * 32 + lane) * 2);
        b0[nt] = bb.x;
        b1[nt] = bb.y;
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (r == 0 ? !vA : !vB) continue;
        const uint32_t cword = j == 0 ? cw[r].x : j == 1 ? cw[r].y : j == 2 ? cw[r].z : cw[r].w;
        uint32_t a[4];
        e2m1x8_to_f16x2x4(cword, a);
        const uint32_t sp = ((j < 2) ? sw[r].x : sw[r].y) >> (16 * (j & 1));
        const uint32_t s2 = e4m3x2_to_f16x2(sp);  // low half: row g scale, high half: row g+8
        const uint32_t slo = dup_lo16(s2), shi = dup_hi16(s2);
        a[0] = hmul2_u32(a[0], slo);
        a[1] = hmul2_u32(a[1], shi);
        a[2] = hmul2_u32(a[2], slo);
        a[3] = hmul2_u32(a[3], shi);
#pragma unroll
        for (int nt = 0; nt < MT; ++nt) mma_f16_16816(acc[r][nt], a, b0[nt], b1[nt]);
      }
    }
  } else {
    uint4 wv[2][2];
    wv[0][0] = lds128(stage + sA * kFp8BlockBytes + lane * 32);
    wv[0][1] = lds128(stage + sA * kFp8BlockBytes + lane * 32 + 16);
    wv[1][0] = lds128(stage + sB * kFp8BlockBytes + lane * 32);
    wv[1][1] = lds128(stage + sB * kFp8BlockBytes + lane * 32 + 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t b0[MT], b1[MT];
#pragma unroll
      for (int nt = 0; nt < MT; ++nt) {
        const uint2 bb = lds64(xq + ((j * MT + nt) * 32 + lane) * 2);
        b0[nt] = bb.x;
        b1[nt] = bb.y;
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (r == 0 ? !vA : !vB) continue;
        const uint4& h = wv[r][j >> 1];
        const uint32_t w0 = (j & 1) ? h.z : h.x;
        const uint32_t w1 = (j & 1) ? h.w : h.y;
        uint32_t a[4];
        a[0] = e4m3x2_to_f16x2(w0 & 0xFFFFu);
        a[1] = e4m3x2_to_f16x2(w0 >> 16);
        a[2] = e4m3x2_to_f16x2(w1 & 0xFFFFu);
        a[3] = e4m3x2_to_f16x2(w1 >> 16);
#pragma unroll
        for (int nt = 0; nt < MT; ++nt) mma_f16_16816(acc[r][nt], a, b0[nt], b1[nt]);
      }
    }
  }
}

// ---------------------------------------------------------------- argmax helpers
// (v, i) beats (bv, bi) when v is larger, or equal with a lower index (lowest index wins ties;
// -0 == +0 under IEEE compare).  Callers map NaN to -inf first.
__device__ __forceinline__ bool am_better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

__device__ __forceinline__ void am_shfl_reduce(float& v, int& i, int mask_bits_from, int mask_bits_to) {
  for (int o = mask_bits_from; o <= mask_bits_to; o <<= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (am_better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

// Cross-group argmax (fixed group order) and greedy acceptance, run by the last group of a head
// task.  aux[g][m] = (value, index bits).  `nthr` threads participate (tid < nthr).
__device__ __forceinline__ void argmax_accept_finish(const float* aux, int n_groups, int M, const int32_t* pending,
                                                     int32_t* argmax, int32_t* n_commit, int32_t* committed,
                                                     float* red_v, int* red_i, int* tok, int tid, int nthr,
                                                     int bar_id) {
  const int tpt = nthr / M;  // threads per token
  if (tid < tpt * M) {
    const int m = tid / tpt, part = tid % tpt;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int g = part; g < n_groups; g += tpt) {
      const float v = __ldcg(aux + ((size_t)g * kMaxM + m) * 2);
      const int i = __float_as_int(__ldcg(aux + ((size_t)g * kMaxM + m) * 2 + 1));
      if (am_better(v, i, bv, bi)) {
        bv = v;
        bi = i;
      }
    }
    red_v[tid] = bv;
    red_i[tid] = bi;
  }
  named_bar_sync(bar_id, nthr);
  if (tid < M) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int part = 0; part < tpt; ++part) {
      const float v = red_v[tid * tpt + part];
      const int i = red_i[tid * tpt + part];
      if (am_better(v, i, bv, bi)) {
        bv = v;
        bi = i;
      }
    }
    if (bi == 0x7fffffff) bi = 0;
    tok[tid] = bi;
    argmax[tid] = bi;
  }
  named_bar_sync(bar_id, nthr);
  if (tid < M / 8) {
    const int base = 8 * tid;
    int acc = 0;
    while (acc < 7 && tok[base + acc] == pending[base + acc + 1]) acc++;
    n_commit[tid] = acc + 1;
    for (int j = 0; j < 8; ++j) committed[base + j] = (j <= acc) ? tok[base + j] : -1;
  }
}

// ---------------------------------------------------------------- epilogue for one finished group
template <int FMT, int MT>
__device__ void group_epilogue(const GemmParams& p, int g, const float (&v)[2][MT][4], SmemMisc& sm, int warp,
                               int lane) {
  const int gq = lane >> 2, tq = lane & 3;
  const int ctid = warp * 32 + lane;
  const GroupGeom gg = group_geom<FMT>(p, g);
  const int sA = p.interleave ? warp : 2 * warp;
  const int sB = p.interleave ? 8 + warp : 2 * warp + 1;
  const bool vA = p.interleave ? (warp < gg.nrb) : (sA < gg.nrb);
  const bool vB = p.interleave ? (warp < gg.nrb) : (sB < gg.nrb);

  if (p.epi == kEpiSiluMul) {
    if (vA) {
#pragma unroll
      for (int nt = 0; nt < MT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int m = nt * 8 + 2 * tq + (i & 1);
          if (m >= p.M) continue;
          const int f = gg.row0 + warp * 16 + gq + 8 * (i >> 1);
          const float gt = v[0][nt][i] * p.wscale[0];
          const float up = v[1][nt][i] * p.wscale[1];
          const float a = gt / (1.0f + expf(-gt)) * up;
          p.out[(size_t)m * p.out_ld + f] = __bfloat16_as_ushort(__float2bfloat16_rn(a));
        }
    }
    return;
  }

  const float wsc = p.wscale[gg.seg];
  if (p.epi == kEpiF32 || p.epi == kEpiBf16Prefix) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r == 0 ? !vA : !vB) continue;
      const int slot = r ? sB : sA;
#pragma unroll
      for (int nt = 0; nt < MT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int m = nt * 8 + 2 * tq + (i & 1);
          if (m >= p.M) continue;
          const int n = gg.row0 + slot * 16 + gq + 8 * (i >> 1);
          const float val = v[r][nt][i] * wsc;
          if (p.epi == kEpiF32) {
            p.y[(size_t)m * p.y_ld + (gg.seg ? p.seg_rows[0] : 0) + n] = val;
          } else if (gg.seg == 0 && n < p.out_cols) {
            p.out[(size_t)m * p.out_ld + n] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
          }
        }
    }
    return;
  }

  if (p.epi == kEpiResid) {
    float ss[MT][2];
#pragma unroll
    for (int nt = 0; nt < MT; ++nt) ss[nt][0] = ss[nt][1] = 0.0f;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r == 0 ? !vA : !vB) continue;
      const int slot = r ? sB : sA;
#pragma unroll
      for (int nt = 0; nt < MT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int m = nt * 8 + 2 * tq + (i & 1);
          if (m >= p.M) continue;
          const int n = gg.row0 + slot * 16 + gq + 8 * (i >> 1);
          uint16_t* hp = p.resid + (size_t)m * p.resid_ld + n;
          const float hn = round_bf16(bf16_bits_to_float(*hp) + v[r][nt][i] * wsc);
          *hp = __bfloat16_as_ushort(__float2bfloat16_rn(hn));
          ss[nt][i & 1] += hn * hn;
        }
    }
#pragma unroll
    for (int nt = 0; nt < MT; ++nt)
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        float s = ss[nt][b];
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        s += __shfl_xor_sync(0xffffffffu, s, 8);
        s += __shfl_xor_sync(0xffffffffu, s, 16);
        const int m = nt * 8 + 2 * tq + b;
        if (gq == 0 && m < kMaxM) sm.red_v[warp][m] = s;
      }
    named_bar_sync(1, kConsumerThreads);
    if (ctid < p.M) {
      float s = 0.0f;
      for (int w = 0; w < kConsumerWarps; ++w) s += sm.red_v[w][ctid];
      p.group_aux[((size_t)g * kMaxM + ctid) * 2] = s;
    }
  } else {  // kEpiHead
    float bv[MT][2];
    int bi[MT][2];
#pragma unroll
    for (int nt = 0; nt < MT; ++nt)
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        bv[nt][b] = -INFINITY;
        bi[nt][b] = 0x7fffffff;
      }
    const int nbase = (gg.seg ? p.seg_rows[0] : 0) + gg.row0;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r == 0 ? !vA : !vB) continue;
      const int slot = r ? sB : sA;
#pragma unroll
      for (int nt = 0; nt < MT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int m = nt * 8 + 2 * tq + (i & 1);
          const int n = nbase + slot * 16 + gq + 8 * (i >> 1);
          const float val = v[r][nt][i] * wsc;
          if (p.logits && m < p.M) p.logits[(size_t)m * p.logits_ld + n] = val;
          const float key = isnan(val) ? -INFINITY : val;
          if (am_better(key, n, bv[nt][i & 1], bi[nt][i & 1])) {
            bv[nt][i & 1] = key;
            bi[nt][i & 1] = n;
          }
        }
    }
#pragma unroll
    for (int nt = 0; nt < MT; ++nt)
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        am_shfl_reduce(bv[nt][b], bi[nt][b], 4, 16);
        const int m = nt * 8 + 2 * tq + b;
        if (gq == 0 && m < kMaxM) {
          sm.red_v[warp][m] = bv[nt][b];
          sm.red_i[warp][m] = bi[nt][b];
        }
      }
    named_bar_sync(1, kConsumerThreads);
    if (ctid < p.M) {
      float b_v = -INFINITY;
      int b_i = 0x7fffffff;
      for (int w = 0; w < kConsumerWarps; ++w)
        if (am_better(sm.red_v[w][ctid], sm.red_i[w][ctid], b_v, b_i)) {
          b_v = sm.red_v[w][ctid];
          b_i = sm.red_i[w][ctid];
        }
      p.group_aux[((size_t)g * kMaxM + ctid) * 2] = b_v;
      p.group_aux[((size_t)g * kMaxM + ctid) * 2 + 1] = __int_as_float(b_i);
    }
  }

  // ---- cross-group finisher: run by the CTA that completes the task's last group
  __threadfence();
  named_bar_sync(1, kConsumerThreads);
  if (ctid == 0) {
    const unsigned old = atomicAdd(p.task_cnt, 1u);
    sm.flag_task_last = (old == (unsigned)p.n_groups - 1u);
  }
  named_bar_sync(1, kConsumerThreads);
  if (!sm.flag_task_last) return;
  __threadfence();
  if (p.epi == kEpiResid) {
    if (ctid < p.M) {
      float s = 0.0f;
      for (int gg2 = 0; gg2 < p.n_groups; ++gg2) s += __ldcg(p.group_aux + ((size_t)gg2 * kMaxM + ctid) * 2);
      p.rms_out[ctid] = 1.0f / sqrtf(s / (float)p.resid_cols + p.rms_eps);
    }
  } else {
    argmax_accept_finish(p.group_aux, p.n_groups, p.M, p.pending, p.argmax, p.n_commit, p.committed, &sm.red_v[0][0],
                         &sm.red_i[0][0], sm.tok, ctid, kConsumerThreads, 1);
  }
  if (ctid == 0) *p.task_cnt = 0u;
}

// ---------------------------------------------------------------- the kernel
template <int FMT, int MT>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  constexpr int S = FmtTraits<FMT>::kStages;
  constexpr int SB = stage_bytes<FMT>();
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  uint32_t* xbuf = reinterpret_cast<uint32_t*>(smem + ring_bytes<FMT>());
  SmemMisc& sm = *reinterpret_cast<SmemMisc*>(smem + ring_bytes<FMT>() + kXBufBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const long long U = p.units;
  const long long u0 = unit_begin(U, G, blockIdx.x), u1 = unit_begin(U, G, blockIdx.x + 1);
  const int nq = p.nq;

  // Let the next kernel of the stream start its (weight-only) prologue as early as possible.
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumerWarps);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer: weights -> ring
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      long long issued = 0;
      int cur_g = -1;
      GroupGeom gg{};
      for (long long u = u0; u < u1; ++u, ++issued) {
        const int st = (int)(issued % S);
        const uint32_t ph = (uint32_t)((issued / S) & 1);
        if (issued >= S && !sm.abort) {
          if (!mbar_wait_bounded(&sm.empty[st], ph ^ 1u)) {
            sm.abort = 1;
            atomicExch(p.status, kStatusTimeout);
          }
        }
        if (sm.abort) break;
        const int g = (int)(u / nq), q = (int)(u % nq);
        if (g != cur_g) {
          gg = group_geom<FMT>(p, g);
          cur_g = g;
        }
        uint8_t* dst = ring + (size_t)st * SB;
        mbar_arrive_expect_tx(&sm.full[st], (uint32_t)(gg.copy_bytes[0] + gg.copy_bytes[1]));
        for (int c = 0; c < 2; ++c)
          if (gg.copy_bytes[c])
            bulk_g2s(dst + gg.dst_slot[c] * FmtTraits<FMT>::kBlock, gg.src[c] + (size_t)q * gg.src_stride[c],
                     (uint32_t)gg.copy_bytes[c], &sm.full[st], pol);
      }
      // Do not leave the CTA with copies in flight: wait (bounded) for the last issued stages.
      const long long last = issued;
      for (long long k = (last > S ? last - S : 0); k < last; ++k) {
        const int st = (int)(k % S);
        const uint32_t ph = (uint32_t)((k / S) & 1);
        if (!mbar_wait_bounded(&sm.full[st], ph)) atomicExch(p.status, kStatusTimeout);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // Everything below reads the previous kernel's outputs or writes outputs: wait for it.
  pdl_wait();
  const int capq = kXBufBytes / (1024 * MT);
  const bool all_k = capq >= nq;
  const int sA = p.interleave ? warp : 2 * warp;
  const int sB = p.interleave ? 8 + warp : 2 * warp + 1;
  const int first_group = (int)(u0 / nq);

  float acc[2][MT][4], tot[2][MT][4];
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int nt = 0; nt < MT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[r][nt][i] = tot[r][nt][i] = 0.0f;

  auto fold = [&]() {
#pragma unroll
    for (int nt = 0; nt < MT; ++nt)
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int e = sm.xexp[nt * 8 + 2 * (lane & 3) + b];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tot[r][nt][2 * h + b] += mul_pow2(acc[r][nt][2 * h + b], e);
            acc[r][nt][2 * h + b] = 0.0f;
          }
      }
  };

  long long u = u0, it = 0;
  while (u < u1) {
    long long ub;
    int origin, qa0, qb0, qa1 = 0, qb1 = 0;
    if (all_k) {
      ub = u1;
      origin = 0;
      if (u1 - u0 >= nq) {
        qa0 = 0;
        qb0 = nq;
      } else if (u0 / nq == (u1 - 1) / nq) {
        qa0 = (int)(u0 % nq);
        qb0 = (int)((u1 - 1) % nq) + 1;
      } else {
        qa0 = (int)(u0 % nq);
        qb0 = nq;
        qa1 = 0;
        qb1 = (int)((u1 - 1) % nq) + 1;
      }
    } else {
      const long long gend = (u / nq + 1) * nq;
      ub = min(u1, min(gend, u + capq));
      origin = (int)(u % nq);
      qa0 = origin;
      qb0 = origin + (int)(ub - u);
    }
    named_bar_sync(1, kConsumerThreads);
    stage_x<MT>(p, xbuf, sm, origin, qa0, qb0, qa1, qb1, warp * 32 + lane);
    named_bar_sync(1, kConsumerThreads);

    int cur_g = -1;
    int nrb = 0;
    for (; u < ub; ++u, ++it) {
      const int st = (int)(it % S);
      const uint32_t ph = (uint32_t)((it / S) & 1);
      if (!sm.abort && !mbar_wait_bounded(&sm.full[st], ph)) {
        sm.abort = 1;
        if (lane == 0) atomicExch(p.status, kStatusTimeout);
      }
      const int g = (int)(u / nq), q = (int)(u % nq);
      if (g != cur_g) {
        nrb = group_geom<FMT>(p, g).nrb;
        cur_g = g;
      }
      const bool vA = p.interleave ? (warp < nrb) : (sA < nrb);
      const bool vB = p.interleave ? (warp < nrb) : (sB < nrb);
      compute_unit<FMT, MT>(ring + (size_t)st * SB, xbuf + (size_t)(q - origin) * (256 * MT), sA, sB, vA, vB, lane,
                            acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[st]);

      const bool group_end = ((u + 1) % nq == 0) || (u + 1 == u1);
      if (group_end) {
        fold();
        const int ctid = warp * 32 + lane;
        const bool cover = ((long long)g * nq >= u0) && ((long long)(g + 1) * nq <= u1);
        if (cover) {
          group_epilogue<FMT, MT>(p, g, tot, sm, warp, lane);
        } else {
          const int slot_p = (g == first_group) ? 0 : 1;
          float* dst = p.partials + (((size_t)blockIdx.x * 2 + slot_p) * kConsumerThreads + ctid) * (8 * MT);
#pragma unroll
          for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int nt = 0; nt < MT; ++nt)
              reinterpret_cast<float4*>(dst)[r * MT + nt] =
                  make_float4(tot[r][nt][0], tot[r][nt][1], tot[r][nt][2], tot[r][nt][3]);
          __threadfence();
          named_bar_sync(1, kConsumerThreads);
          const int c_first = cta_of_unit(U, G, (long long)g * nq);
          const int c_last = cta_of_unit(U, G, (long long)(g + 1) * nq - 1);
          if (ctid == 0) {
            const unsigned old = atomicAdd(p.group_cnt + g, 1u);
            sm.flag_last = (old == (unsigned)(c_last - c_first));
          }
          named_bar_sync(1, kConsumerThreads);
          if (sm.flag_last) {
            __threadfence();
            float sum[2][MT][4];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
              for (int nt = 0; nt < MT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) sum[r][nt][i] = 0.0f;
            for (int c = c_first; c <= c_last; ++c) {
              const int fg = (int)(unit_begin(U, G, c) / nq);
              const int sp = (g == fg) ? 0 : 1;
              const float4* src = reinterpret_cast<const float4*>(
                  p.partials + (((size_t)c * 2 + sp) * kConsumerThreads + ctid) * (8 * MT));
#pragma unroll
              for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int nt = 0; nt < MT; ++nt) {
                  const float4 f = __ldcg(src + r * MT + nt);
                  sum[r][nt][0] += f.x;
                  sum[r][nt][1] += f.y;
                  sum[r][nt][2] += f.z;
                  sum[r][nt][3] += f.w;
                }
            }
            group_epilogue<FMT, MT>(p, g, sum, sm, warp, lane);
            if (ctid == 0) p.group_cnt[g] = 0u;
          }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int nt = 0; nt < MT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) tot[r][nt][i] = 0.0f;
      }
    }
    if (u < u1 && (u % nq) != 0) fold();  // batch ended inside a group
  }
}

}  // namespace vp
