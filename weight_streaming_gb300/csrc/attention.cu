// Verify attention over a BF16 KV cache (vp_attention_verify): the attention core of the pages'
// full-attention layers for the 8 verify rows of each lane.
//
// Source: "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max", section "The megakernel
// is per layer, not per step" (the full-attention figure and the text after it): the core reads and
// appends a BF16 KV cache, runs a causal softmax of q k^T weighting V, and multiplies by the sigmoid
// of the gate; the KV range is split into partitions (1,024 keys at the 32K tier) whose online-softmax
// partials m' = max(m, max s), a = e^(m - m'), l' = a l + sum e^(s - m'), o' = a o + e^(s - m') V are
// merged.  Geometry (24 q heads, 4 kv heads, head dim 256): "144 tok/s needs 502 GB/s", section "The
// engine hard-codes the model".
//
// GB300 design:
//  * attn_append: the verify rows' keys and values go into the cache at ctx[l] .. ctx[l] + 7.
//  * attn_partition, grid (partitions, kv heads, lanes): one CTA per partition (at most 1,024 keys;
//    shorter when that fills the GPU in one wave) of one kv head of one lane computes the partials of all its query rows (the G = Hq / Hkv heads that share
//    the kv head x 8 verify rows, padded to 64).  Key and value tiles of 64 positions stream through
//    a two-stage cp.async ring in shared memory (16-byte chunks XOR-swizzled by row, so every
//    ldmatrix is conflict-free); S = Q K^T on the tensor core in bf16 (q and k exact), the online
//    softmax in fp32 (exp2 with the 1/sqrt(D) log2(e) scale folded in), then O += P V on the tensor
//    core in bf16 with the values as cached (exact over bf16's whole range) and P in [0, 1] split into
//    two bf16 parts, P = hi + lo (hi = bf16(P), lo = bf16(P - hi): P to about 2^-17 relative), one
//    MMA each.  Warps w and w + 4 share m-tile w % 4: each computes S for half of the tile's keys, they
//    exchange the row maxima and their halves of P through shared memory (named barrier per pair),
//    and each accumulates output dims 128 (w / 4) .. + 127 over all keys.
//  * attn_merge: per output row and head, the partitions' partials in a fixed order, then the sigmoid
//    gate and one bf16 rounding.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>
#include <cstdint>

#include "attention.h"
#include "internal.h"

namespace vp {

namespace {

constexpr int kD = 256;          // head dim
constexpr int kTile = 64;        // keys per tile
constexpr int kRows = 64;        // query rows per CTA (G heads x 8 rows, padded)
constexpr int kRowBytes = kD * 2;
constexpr int kTileBytes = kTile * kRowBytes;  // 32 KB
constexpr int kThreadsA = 256;
constexpr int kSmemA = kRows * kRowBytes + 4 * kTileBytes;  // Q + 2 x (K, V) = 160 KB

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
// Byte offset of 16-byte chunk c of row r in a swizzled [rows][256] 16-bit tile.
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * kRowBytes + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Byte offset of (row, key) in a [rows][64] 16-bit P tile, 16-byte chunks XOR-swizzled by row.
__device__ __forceinline__ uint32_t pswz(int r, int key) {
  return (uint32_t)(r * 128 + ((((key >> 3) ^ (r & 7)) << 4) | ((key & 7) << 1)));
}
// The two warps of m-tile mt (warps mt and mt + 4) meet at named barrier 1 + mt.
__device__ __forceinline__ void pair_sync(int mt) { asm volatile("bar.sync %0, 64;" ::"r"(1 + mt) : "memory"); }
// Two fp32 values as bf16 pairs: hi = bf16(x) (a in the low half), lo = bf16(x - hi).
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - __low2float(h), b - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

constexpr int kStatusShape = 2;  // VP_ERR_SHAPE

// A lane's cached length is usable when its 8 new positions fit the cache.
__device__ __forceinline__ bool ctx_ok(int c, int cap) { return c >= 0 && c <= cap - 8; }

__global__ void attn_append(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                            uint16_t* __restrict__ k_cache, uint16_t* __restrict__ v_cache,
                            const int32_t* __restrict__ ctx, int Hkv, int cap, int* status) {
  const int r = blockIdx.x, g = blockIdx.y, l = r / 8, j = r % 8, t = threadIdx.x;  // 32 threads x 16 B
  if (!ctx_ok(ctx[l], cap)) {
    if (t == 0) atomicExch(status, kStatusShape);
    return;
  }
  const size_t src = ((size_t)r * Hkv + g) * kD + 8 * t;
  const size_t dst = (((size_t)l * Hkv + g) * cap + ctx[l] + j) * kD + 8 * t;
  *reinterpret_cast<uint4*>(k_cache + dst) = *reinterpret_cast<const uint4*>(k_new + src);
  *reinterpret_cast<uint4*>(v_cache + dst) = *reinterpret_cast<const uint4*>(v_new + src);
}

__global__ void __launch_bounds__(kThreadsA, 1) attn_partition(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const uint32_t sQ = smem_u32(sm);
  const uint32_t sK0 = sQ + kRows * kRowBytes, sV0 = sK0 + 2 * kTileBytes;  // buffer b at + b * kTileBytes
  const int part = blockIdx.x, g = blockIdx.y, l = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, cq = lane & 3;
  const int G = a.Hq / a.Hkv, rows = 8 * G;
  const int ctx = a.ctx[l], n_keys = ctx + 8;
  const int k0 = part * a.part_len, k1 = min(k0 + a.part_len, n_keys);
  float* pO = a.part_o + ((((size_t)l * a.Hkv + g) * a.n_part + part) * kRows) * kD;
  float* pML = a.part_ml + (((size_t)l * a.Hkv + g) * a.n_part + part) * kRows * 2;
  if (k0 >= n_keys || !ctx_ok(ctx, a.cap)) {  // beyond this lane's keys (or a bad ctx): an empty partial
    for (int i = tid; i < kRows; i += blockDim.x) {
      pML[2 * i] = -INFINITY;
      pML[2 * i + 1] = 0.0f;
    }
    return;
  }
  const uint16_t* kc = a.k_cache + ((size_t)l * a.Hkv + g) * a.cap * kD;
  const uint16_t* vc = a.v_cache + ((size_t)l * a.Hkv + g) * a.cap * kD;
  // Q: row i = hg * 8 + j (head g * G + hg, verify row j); rows >= 8 G are zero.
  for (int c = tid; c < kRows * 32; c += blockDim.x) {
    const int i = c >> 5, ch = c & 31;
    const bool ok = i < rows;
    const uint16_t* src = a.q + (((size_t)(8 * l + (ok ? i % 8 : 0)) * a.Hq + g * G + (ok ? i / 8 : 0)) * kD) + 8 * ch;
    cp_async16(sQ + swz(i, ch), src, ok);
  }
  const int n_tiles = (k1 - k0 + kTile - 1) / kTile;
  // Copies of key / value tile t into buffer b; positions past the partition's end are zero-filled.
#define ATTN_ISSUE(t, b)                                                                         \
  for (int c = tid; c < kTile * 32; c += blockDim.x) {                                           \
    const int r = c >> 5, ch = c & 31, pos = k0 + (t) * kTile + r;                               \
    const bool ok = pos < k1;                                                                    \
    cp_async16(sK0 + (b) * kTileBytes + swz(r, ch), kc + (size_t)(ok ? pos : 0) * kD + 8 * ch, ok); \
    cp_async16(sV0 + (b) * kTileBytes + swz(r, ch), vc + (size_t)(ok ? pos : 0) * kD + 8 * ch, ok); \
  }
  ATTN_ISSUE(0, 0)
  cp_async_commit();  // group 0: Q and tile 0

  __shared__ float xmax[4][2][16];                // per m-tile, per warp of the pair: row maxima, then sums
  // per m-tile: P [16 rows][64 keys] as bf16 hi parts, then (at + kPLo) the lo parts, swizzled
  constexpr int kPLo = 4 * 16 * 128;
  __shared__ __align__(16) uint8_t sP[2 * kPLo];
  const int mt = warp & 3, dh = warp >> 2;
  const bool live = mt * 16 < rows;
  const float sl2 = 1.4426950408889634f / sqrtf((float)kD);  // log2(e) / sqrt(D)
  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.0f, 0.0f};  // rows gq, gq + 8 of the m-tile (log2 units)
  const int row0 = mt * 16 + gq;
  const int lim[2] = {ctx + (row0 % 8), ctx + ((row0 + 8) % 8)};  // last visible position per row

  for (int t = 0; t < n_tiles; ++t) {
    const int b = t & 1;
    if (t + 1 < n_tiles) ATTN_ISSUE(t + 1, b ^ 1)
    cp_async_commit();
    cp_async_wait<1>();  // this thread's copies of tile t (and Q) have landed
    __syncthreads();     // and every other thread's
    if (live) {
      // S = Q K^T for the m-tile and this warp's 32 keys of the tile (4 n-tiles); the pair's other
      // warp takes the other 32.
      float s[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sQ + swz(mt * 16 + (lane & 15), 2 * ks + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(sK0 + b * kTileBytes + swz(dh * 32 + np * 16 + (lane >> 4) * 8 + (lane & 7), 2 * ks + ((lane >> 3) & 1)),
                  b0, b1, b2, b3);
          mma_bf16(s[2 * np], a0, a1, a2, a3, b0, b1);
          mma_bf16(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      // online softmax (log2 units), causal mask per row; the row maximum over both halves
      const int base = k0 + t * kTile + dh * 32;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pos = base + n * 8 + 2 * cq + (e & 1), h = e >> 1;
          const float v = pos <= lim[h] ? s[n][e] * sl2 : -INFINITY;
          s[n][e] = v;
          mx[h] = fmaxf(mx[h], v);
        }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      }
      if (cq == 0) {
        xmax[mt][dh][gq] = mx[0];
        xmax[mt][dh][gq + 8] = mx[1];
      }
      pair_sync(mt);
      float alpha[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float mn = fmaxf(m_r[h], fmaxf(mx[h], xmax[mt][dh ^ 1][gq + 8 * h]));
        alpha[h] = mn == -INFINITY ? 1.0f : exp2f(m_r[h] - mn);
        m_r[h] = mn;
      }
      float rs[2] = {0.0f, 0.0f};
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          const float p = m_r[h] == -INFINITY ? 0.0f : exp2f(s[n][e] - m_r[h]);
          s[n][e] = p;
          rs[h] += p;
        }
#pragma unroll
      for (int h = 0; h < 2; ++h) l_r[h] = alpha[h] * l_r[h] + rs[h];  // this warp's keys only
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
      // this warp's half of P (bf16 hi and lo parts) for the other warp of the pair
      uint32_t ph[2][4], pl[2][4];  // A fragments of this warp's two 16-key steps
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        split_bf16(s[2 * kk][0], s[2 * kk][1], ph[kk][0], pl[kk][0]);
        split_bf16(s[2 * kk][2], s[2 * kk][3], ph[kk][1], pl[kk][1]);
        split_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[kk][2], pl[kk][2]);
        split_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[kk][3], pl[kk][3]);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // n-tile 2 kk + hh: keys dh * 32 + 16 kk + 8 hh + 2 cq
          const int key = dh * 32 + 16 * kk + 8 * hh + 2 * cq;
          const uint32_t o0 = pswz(mt * 16 + gq, key), o1 = pswz(mt * 16 + gq + 8, key);
          *reinterpret_cast<uint32_t*>(sP + o0) = ph[kk][2 * hh];
          *reinterpret_cast<uint32_t*>(sP + o1) = ph[kk][2 * hh + 1];
          *reinterpret_cast<uint32_t*>(sP + kPLo + o0) = pl[kk][2 * hh];
          *reinterpret_cast<uint32_t*>(sP + kPLo + o1) = pl[kk][2 * hh + 1];
        }
      }
      pair_sync(mt);
      // O += (P_hi + P_lo) V for this warp's 128 output dims: 4 key steps of 16 (two from registers,
      // two from the other warp through shared memory), 16 n-tiles of 8 dims
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t a[4], c[4];
        if ((kk >> 1) == dh) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            a[e] = ph[kk & 1][e];
            c[e] = pl[kk & 1][e];
          }
        } else {
          const uint32_t at = smem_u32(sP) + pswz(mt * 16 + (lane & 15), 16 * kk + 8 * (lane >> 4));
          ldsm_x4(at, a[0], a[1], a[2], a[3]);
          ldsm_x4(at + kPLo, c[0], c[1], c[2], c[3]);
        }
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sV0 + b * kTileBytes + swz(kk * 16 + (lane & 15), dh * 16 + 2 * np + (lane >> 4)), b0, b1, b2, b3);
          mma_bf16(o[2 * np], a[0], a[1], a[2], a[3], b0, b1);
          mma_bf16(o[2 * np], c[0], c[1], c[2], c[3], b0, b1);
          mma_bf16(o[2 * np + 1], a[0], a[1], a[2], a[3], b2, b3);
          mma_bf16(o[2 * np + 1], c[0], c[1], c[2], c[3], b2, b3);
        }
      }
    }
    __syncthreads();  // tile buffer b is free for tile t + 2
  }
#undef ATTN_ISSUE
  cp_async_wait<0>();
  if (!live) return;
  // partials: m (log2 units), l (the row's full sum over both warps of the pair), o unnormalised
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 1);
    l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 2);
  }
  if (cq == 0) {
    xmax[mt][dh][gq] = l_r[0];
    xmax[mt][dh][gq + 8] = l_r[1];
  }
  pair_sync(mt);
  l_r[0] += xmax[mt][dh ^ 1][gq];
  l_r[1] += xmax[mt][dh ^ 1][gq + 8];
  const int r0 = mt * 16 + gq, r1 = r0 + 8;
  if (cq == 0 && dh == 0) {
    pML[2 * r0] = m_r[0];
    pML[2 * r0 + 1] = l_r[0];
    pML[2 * r1] = m_r[1];
    pML[2 * r1 + 1] = l_r[1];
  }
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const int d = dh * 128 + n * 8 + 2 * cq;
    *reinterpret_cast<float2*>(pO + (size_t)r0 * kD + d) = make_float2(o[n][0], o[n][1]);
    *reinterpret_cast<float2*>(pO + (size_t)r1 * kD + d) = make_float2(o[n][2], o[n][3]);
  }
}

// One CTA per (verify row, q head), one thread per output dim: the partitions in order.  The
// partitions' maxima and sums are the same for every thread of the CTA: they are read once per CTA
// (thread p reads partition p of each chunk of kD) and each partition's weight exp2(m - M) is formed
// once, in shared memory; every thread then adds the partitions in order.
__global__ void attn_merge(const AttnArgs a) {
  __shared__ float sw[kD], sl[kD], red[kD / 32];
  const int r = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const int G = a.Hq / a.Hkv, g = h / G, l = r / 8, i = (h % G) * 8 + r % 8;
  const size_t pb = ((size_t)l * a.Hkv + g) * a.n_part;
  if (!ctx_ok(a.ctx[l], a.cap)) {  // reported through the status word; the output is zero
    a.out[((size_t)r * a.Hq + h) * kD + d] = 0;
    return;
  }
  float M = -INFINITY;
  for (int p = d; p < a.n_part; p += kD) M = fmaxf(M, a.part_ml[((pb + p) * kRows + i) * 2]);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if ((d & 31) == 0) red[d >> 5] = M;
  __syncthreads();
  M = red[0];
  for (int w = 1; w < kD / 32; ++w) M = fmaxf(M, red[w]);
  float den = 0.0f, num = 0.0f;
  for (int p0 = 0; p0 < a.n_part; p0 += kD) {
    if (p0 + d < a.n_part) {
      const float* ml = a.part_ml + ((pb + p0 + d) * kRows + i) * 2;
      const float m = ml[0];
      sw[d] = m == -INFINITY ? -1.0f : exp2f(m - M);  // -1: an empty partition, skipped
      sl[d] = ml[1];
    }
    __syncthreads();
    const int n = min(kD, a.n_part - p0);
    const float* po = a.part_o + ((pb + p0) * kRows + i) * kD + d;
#pragma unroll 8
    for (int q = 0; q < n; ++q) {
      const float w = sw[q];
      if (w < 0.0f) continue;
      den += w * sl[q];
      num += w * po[(size_t)q * kRows * kD];
    }
    __syncthreads();
  }
  float v = num / den;
  if (a.gate) v /= 1.0f + expf(-__uint_as_float((uint32_t)a.gate[((size_t)r * a.Hq + h) * kD + d] << 16));
  a.out[((size_t)r * a.Hq + h) * kD + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

}  // namespace

AttnWs attn_ws_layout(int M, int Hkv, int cap) {
  AttnWs L;
  // Partitions per (lane, kv head) so that the grid is one wave of kAttnTargetCtas CTAs, each a
  // multiple of the 64-key tile and at most kAttnPart keys (longer contexts take several waves).
  const int per = std::max(1, kAttnTargetCtas / std::max(1, (M / 8) * Hkv));
  const int len = (cap + per - 1) / per;
  L.part_len = std::min(kAttnPart, std::max(kTile, (len + kTile - 1) / kTile * kTile));
  L.n_part = (cap + L.part_len - 1) / L.part_len;
  const size_t units = (size_t)(M / 8) * Hkv * L.n_part * kRows;
  L.status = 0;
  L.part_o = 256;
  L.part_ml = align_up(L.part_o + sizeof(float) * units * kD, 256);
  L.total = align_up(L.part_ml + sizeof(float) * units * 2, 256);
  return L;
}

cudaError_t launch_attention_verify(AttnArgs a, int M, void* ws, cudaStream_t s, int* status) {
  const AttnWs L = attn_ws_layout(M, a.Hkv, a.cap);
  uint8_t* b = static_cast<uint8_t*>(ws);
  a.n_part = L.n_part;
  a.part_len = L.part_len;
  a.part_o = reinterpret_cast<float*>(b + L.part_o);
  a.part_ml = reinterpret_cast<float*>(b + L.part_ml);
  a.status = status ? status : reinterpret_cast<int*>(b + L.status);
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(attn_partition, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemA);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  attn_append<<<dim3((unsigned)M, (unsigned)a.Hkv), 32, 0, s>>>(a.k_new, a.v_new, a.k_cache, a.v_cache, a.ctx, a.Hkv,
                                                                 a.cap, a.status);
  attn_partition<<<dim3((unsigned)L.n_part, (unsigned)a.Hkv, (unsigned)(M / 8)), kThreadsA, kSmemA, s>>>(a);
  attn_merge<<<dim3((unsigned)M, (unsigned)a.Hq), kD, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace vp
