// Producer and consumer steps of the pass's real mixer cores, between the executor's projections:
// the Gated DeltaNet layer's A / B projections, short convolution, Q / K normalisation and gates
// ahead of its delta-rule scan (gdn.cu) and its gated RMSNorm after it; the attention layer's Q / K
// RMSNorm and rotary embedding ahead of its core over the KV cache (attention.cu).
//
// Sources: "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max" -- "The megakernel is
// per layer, not per step" (the GDN layer: RMSNorm, FP8 QKV and Z projections, BF16 A / B
// projections, short convolution, Q / K norm, gates, the recurrence, gated RMSNorm with SiLU of Z, FP8
// out-projection with the residual; the full-attention layer: FP8 Q / K / V and gate projections, Q /
// K RMSNorm, RoPE, the causal softmax over a read-and-appended BF16 cache, times the sigmoid of the
// gate, FP8 o-projection with the residual) and "What one token costs the bus" (the A / B
// projections, norms and convolution taps are small BF16 tensors); "144 tok/s needs 502 GB/s" -- "The
// engine hard-codes the model" (4-tap convolutions, decays and time biases).  The formulas the pages
// leave open are the readings stated with each kernel: the plainest ones the names support.
//
// All arithmetic is fp32 with every rounding to bf16 where the layer keeps bf16 values.  Every kernel
// is one launch on the caller's stream, reads only device memory and synchronises nothing.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mixer.h"

namespace vp {

namespace {

__device__ __forceinline__ float bfv(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t to_bf(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

// Sum of x over the block's threads (blockDim.x a multiple of 32, at most 1024), in a fixed order;
// every thread gets the result.
__device__ __forceinline__ float block_sum(float x, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = x;
  __syncthreads();
  float s = 0.0f;
  for (int i = 0; i < nw; ++i) s += red[i];
  return s;
}

// A / B projections of a Gated DeltaNet layer on r = bf16(RMSNorm(h)) (unit weight), with the gates:
// alpha[t][j] = exp(-exp(A_log[j]) softplus(r_t . A[j] + dt_bias[j])), beta[t][j] = sigmoid(r_t . B[j])
// (fp32 [M][n_v]).  Block (j, g): weight row j (rows 0 .. n_v - 1 of A, then those of B) against rows
// 4g .. 4g + 3.  Thread i holds 16-byte chunks i and i + 512 of K of the 4 rows in registers (all
// loads issued at once), so the rows' statistic and the dot products read h once; both sums meet in a
// fixed order (shuffle tree, then the 16 warps in order).  hidden % 8 == 0, hidden <= 8192.
constexpr int kAbThreads = 512, kAbPer = 2, kAbRows = 4;
__device__ __forceinline__ void ab_block_sum(float (&v)[kAbRows], float (*red)[kAbRows], float* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < kAbRows; ++t) {
    float x = v[t];
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) red[warp][t] = x;
  }
  __syncthreads();
  if (threadIdx.x < kAbRows) {
    float x = 0.0f;
    for (int w = 0; w < kAbThreads / 32; ++w) x += red[w][threadIdx.x];
    out[threadIdx.x] = x;
  }
  __syncthreads();
}
__global__ void __launch_bounds__(kAbThreads) ab_gates_kernel(
    const uint16_t* __restrict__ h, int hidden, int M, float eps, const uint16_t* __restrict__ wa,
    const uint16_t* __restrict__ wb, int n_v, const float* __restrict__ a_log, const float* __restrict__ dt_bias,
    float* __restrict__ alpha, float* __restrict__ beta) {
  __shared__ float red[kAbThreads / 32][kAbRows];
  __shared__ float sums[kAbRows];
  const int j = blockIdx.x, t0 = blockIdx.y * kAbRows, tid = threadIdx.x, chunks = hidden / 8;
  const uint16_t* w = j < n_v ? wa + (size_t)j * hidden : wb + (size_t)(j - n_v) * hidden;
  uint4 hv[kAbPer][kAbRows], wv[kAbPer];
#pragma unroll
  for (int p = 0; p < kAbPer; ++p) {
    const int c = tid + p * kAbThreads;
    const bool ok = c < chunks;
    wv[p] = ok ? *reinterpret_cast<const uint4*>(w + 8 * c) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int t = 0; t < kAbRows; ++t)
      hv[p][t] = ok && t0 + t < M ? *reinterpret_cast<const uint4*>(h + (size_t)(t0 + t) * hidden + 8 * c)
                                  : make_uint4(0, 0, 0, 0);
  }
  float acc[kAbRows];
#pragma unroll
  for (int t = 0; t < kAbRows; ++t) {
    acc[t] = 0.0f;
#pragma unroll
    for (int p = 0; p < kAbPer; ++p) {
      const uint32_t x4[4] = {hv[p][t].x, hv[p][t].y, hv[p][t].z, hv[p][t].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(x4[e] << 16), hi = __uint_as_float(x4[e] & 0xFFFF0000u);
        acc[t] = fmaf(lo, lo, acc[t]);
        acc[t] = fmaf(hi, hi, acc[t]);
      }
    }
  }
  ab_block_sum(acc, red, sums);
  float inv[kAbRows];
#pragma unroll
  for (int t = 0; t < kAbRows; ++t) inv[t] = 1.0f / sqrtf(sums[t] / (float)hidden + eps);
  __syncthreads();  // sums is rewritten below
#pragma unroll
  for (int t = 0; t < kAbRows; ++t) {
    acc[t] = 0.0f;
#pragma unroll
    for (int p = 0; p < kAbPer; ++p) {
      const uint32_t x4[4] = {hv[p][t].x, hv[p][t].y, hv[p][t].z, hv[p][t].w};
      const uint32_t w4[4] = {wv[p].x, wv[p].y, wv[p].z, wv[p].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float r0 = bfv(to_bf(__uint_as_float(x4[e] << 16) * inv[t]));
        const float r1 = bfv(to_bf(__uint_as_float(x4[e] & 0xFFFF0000u) * inv[t]));
        acc[t] = fmaf(r0, __uint_as_float(w4[e] << 16), acc[t]);
        acc[t] = fmaf(r1, __uint_as_float(w4[e] & 0xFFFF0000u), acc[t]);
      }
    }
  }
  ab_block_sum(acc, red, sums);
  if (tid < kAbRows && t0 + tid < M) {
    const float x = sums[tid];
    const int t = t0 + tid;
    if (j < n_v) {
      const float z = x + dt_bias[j];
      const float sp = z > 20.0f ? z : log1pf(expf(z));
      alpha[(size_t)t * n_v + j] = expf(-expf(a_log[j]) * sp);
    } else {
      beta[(size_t)t * n_v + (j - n_v)] = 1.0f / (1.0f + expf(-x));
    }
  }
}

// The Gated DeltaNet producer steps, block (row t, head) of d threads (one channel each):
//  * the conv input of channel c: e = [window_a rows 0..2 (the lane's three earlier rows), the
//    lane's 8 rows of u (the in-projection's q, k, v part)]; row t's output is
//    y = silu(sum_j taps[c][j] e[t + j]) (tap 3 on the current row), in fp32 in tap order;
//  * q and k heads: y over its L2 norm (eps 1e-6 inside the root), then bf16; v: bf16(y);
//  * q / k head i serves v heads i * rep .. (i + 1) * rep - 1 (rep = n_v / n_qk): written there;
//  * conv_hist[lane] = e (11 rows): the window after n accepted rows is rows n .. n + 2.
// Heads: 0 .. n_qk - 1 q, n_qk .. 2 n_qk - 1 k, then n_v v heads.
__global__ void gdn_prep_kernel(const uint16_t* __restrict__ u, int ld_u, const uint16_t* __restrict__ window_a,
                                const uint16_t* __restrict__ taps, int n_qk, int n_v, int d,
                                uint16_t* __restrict__ q, uint16_t* __restrict__ k, uint16_t* __restrict__ v,
                                uint16_t* __restrict__ conv_hist, int32_t* __restrict__ rows8) {
  __shared__ float red[8];
  const int t = blockIdx.x, head = blockIdx.y, i = threadIdx.x;
  const int lane = t >> 3, tl = t & 7, C = (2 * n_qk + n_v) * d;
  const int c = head * d + i;
  const uint16_t* wa = window_a + (size_t)lane * 3 * C;
  float e[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = tl + j;  // row of e
    e[j] = r < 3 ? bfv(wa[(size_t)r * C + c]) : bfv(u[(size_t)(8 * lane + r - 3) * ld_u + c]);
  }
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) acc = fmaf(bfv(taps[(size_t)c * 4 + j]), e[j], acc);
  const float y = silu(acc);
  if (tl == 0) {  // the lane's conv history: its window, then its 8 rows
    uint16_t* hist = conv_hist + (size_t)lane * 11 * C;
    for (int r = 0; r < 3; ++r) hist[(size_t)r * C + c] = wa[(size_t)r * C + c];
    for (int r = 0; r < 8; ++r) hist[(size_t)(3 + r) * C + c] = u[(size_t)(8 * lane + r) * ld_u + c];
    if (head == 0 && i == 0) rows8[lane] = 8;
  }
  const int rep = n_v / n_qk;
  if (head < 2 * n_qk) {
    const float n2 = block_sum(y * y, red);
    const uint16_t o = to_bf(y / sqrtf(n2 + 1e-6f));
    uint16_t* dst = head < n_qk ? q : k;
    const int qh = head < n_qk ? head : head - n_qk;
    for (int r = 0; r < rep; ++r) dst[((size_t)t * n_v + qh * rep + r) * d + i] = o;
  } else {
    v[((size_t)t * n_v + (head - 2 * n_qk)) * d + i] = to_bf(y);
  }
}

// Gated RMSNorm, block (row t, v head) of d threads: bf16(o / sqrt(mean(o^2) + eps) * w * silu(z)),
// o the scan's output (fp32 [M][n_v][d]), z = u[t][z0 + head * d + i] (bf16 in-projection output).
__global__ void gated_norm_kernel(const float* __restrict__ o, const uint16_t* __restrict__ u, int ld_u, int z0,
                                  const float* __restrict__ w, int n_v, int d, uint16_t* __restrict__ out) {
  __shared__ float red[8];
  const int t = blockIdx.x, hh = blockIdx.y, i = threadIdx.x;
  const float x = o[((size_t)t * n_v + hh) * d + i];
  const float ms = block_sum(x * x, red) / (float)d;
  const float z = bfv(u[(size_t)t * ld_u + z0 + hh * d + i]);
  out[(size_t)t * n_v * d + hh * d + i] = to_bf(x / sqrtf(ms + 1e-6f) * w[i] * silu(z));
}

// Attention producer steps, block (row t, group of kPrepHeads heads) of D threads: heads 0 .. Hq - 1
// the queries (uq[t][h D + i]), Hq .. Hq + Hkv - 1 the keys (ukv[t][h D + i]): each over its root
// mean square (eps 1e-6) times the shared weight (q_norm / k_norm), then the rotary embedding over
// the whole head at the row's cache position ctx[lane] + t % 8 (pairs (2j, 2j + 1) rotated by
// pos * 10000^(-2j / D)), then bf16.  The angle is formed in fp64 from the host's fp64 inverse
// frequencies and reduced to [-pi, pi] in fp64 (a - 2 pi rint(a / 2 pi) with one fma; the error of
// the fp64 2 pi, under 1e-9 rad for positions below 2^24, is far below bf16), then sine and cosine in
// fp32 -- once per block for the row.  Then Hkv value heads and Hq gate heads, copied to dense
// [M][heads][D] rows.  Every head's element is loaded up front, the group's sums of squares meet in
// one fixed-order reduction, and a pair's partner comes from the neighbouring lane.  D <= 512, even.
constexpr int kPrepHeads = 8;
__global__ void attn_prep_kernel(const uint16_t* __restrict__ uq, int ld_q, const uint16_t* __restrict__ ukv,
                                 int ld_kv, int Hq, int Hkv, int D, const float* __restrict__ q_norm,
                                 const float* __restrict__ k_norm, const int32_t* __restrict__ ctx,
                                 const __grid_constant__ RopeTable rt, uint16_t* __restrict__ q,
                                 uint16_t* __restrict__ k, uint16_t* __restrict__ v, uint16_t* __restrict__ gate) {
  __shared__ float red[16][kPrepHeads];
  __shared__ float cs_t[256], sn_t[256];
  const int t = blockIdx.x, i = threadIdx.x, warp = i >> 5, lane = i & 31;
  const int h0 = blockIdx.y * kPrepHeads, nh = min(kPrepHeads, 2 * Hq + 2 * Hkv - h0), nr = Hq + Hkv - h0;
  float x[kPrepHeads];
#pragma unroll
  for (int e = 0; e < kPrepHeads; ++e) {
    const int hh = h0 + e;
    x[e] = 0.0f;
    if (e >= nh) continue;
    if (hh < Hq) {
      x[e] = bfv(uq[(size_t)t * ld_q + hh * D + i]);
    } else if (hh < Hq + Hkv) {
      x[e] = bfv(ukv[(size_t)t * ld_kv + (hh - Hq) * D + i]);
    } else if (hh < Hq + 2 * Hkv) {
      const int h = hh - Hq - Hkv;
      v[((size_t)t * Hkv + h) * D + i] = ukv[(size_t)t * ld_kv + (Hkv + h) * D + i];
    } else {
      const int h = hh - Hq - 2 * Hkv;
      gate[((size_t)t * Hq + h) * D + i] = uq[(size_t)t * ld_q + (Hq + h) * D + i];
    }
  }
  if (nr <= 0) return;  // a group of copies only
  if (i < D / 2) {
    const double a = ((double)ctx[t >> 3] + (double)(t & 7)) * rt.inv_freq[i];
    const double r = fma(-rint(a * 0.15915494309189535), 6.283185307179586, a);  // a mod 2 pi
    sincosf((float)r, &sn_t[i], &cs_t[i]);
  }
#pragma unroll
  for (int e = 0; e < kPrepHeads; ++e) {
    float s2 = x[e] * x[e];
#pragma unroll
    for (int o = 16; o; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    if (lane == 0) red[warp][e] = s2;
  }
  __syncthreads();
  const int j = i >> 1;
  const float sn = sn_t[j], cs = cs_t[j];
#pragma unroll
  for (int e = 0; e < kPrepHeads; ++e) {
    float ms = 0.0f;
    for (int w = 0; w < (D >> 5); ++w) ms += red[w][e];
    const int hh = h0 + e;
    const bool isq = hh < Hq;
    const float y = e < nr ? x[e] / sqrtf(ms / (float)D + 1e-6f) * (isq ? q_norm[i] : k_norm[i]) : 0.0f;
    const float yp = __shfl_xor_sync(0xffffffffu, y, 1);  // the pair's other element
    if (e >= nr) continue;
    const float x0 = (i & 1) ? yp : y, x1 = (i & 1) ? y : yp;
    const float r = (i & 1) ? fmaf(x0, sn, x1 * cs) : fmaf(x0, cs, -(x1 * sn));
    (isq ? q + ((size_t)t * Hq + hh) * D : k + ((size_t)t * Hkv + (hh - Hq)) * D)[i] = to_bf(r);
  }
}

}  // namespace

cudaError_t launch_ab_gates(const uint16_t* h, int hidden, int M, float eps, const uint16_t* wa, const uint16_t* wb,
                            int n_v, const float* a_log, const float* dt_bias, float* alpha, float* beta,
                            cudaStream_t s) {
  ab_gates_kernel<<<dim3(2 * n_v, (M + kAbRows - 1) / kAbRows), kAbThreads, 0, s>>>(h, hidden, M, eps, wa, wb, n_v,
                                                                                    a_log, dt_bias, alpha, beta);
  return cudaGetLastError();
}

cudaError_t launch_gdn_prep(const uint16_t* u, int ld_u, int M, const uint16_t* window_a, const uint16_t* taps,
                            int n_qk, int n_v, int d, uint16_t* q, uint16_t* k, uint16_t* v, uint16_t* conv_hist,
                            int32_t* rows8, cudaStream_t s) {
  gdn_prep_kernel<<<dim3(M, 2 * n_qk + n_v), d, 0, s>>>(u, ld_u, window_a, taps, n_qk, n_v, d, q, k, v, conv_hist,
                                                        rows8);
  return cudaGetLastError();
}

cudaError_t launch_gated_norm(const float* o, const uint16_t* u, int ld_u, int z0, const float* w, int M, int n_v,
                              int d, uint16_t* out, cudaStream_t s) {
  gated_norm_kernel<<<dim3(M, n_v), d, 0, s>>>(o, u, ld_u, z0, w, n_v, d, out);
  return cudaGetLastError();
}

RopeTable rope_table(int D) {
  RopeTable rt;
  for (int j = 0; j < 256; ++j) rt.inv_freq[j] = 2 * j < D ? pow(10000.0, -2.0 * (double)j / (double)D) : 0.0;
  return rt;
}

cudaError_t launch_attn_prep(const uint16_t* uq, int ld_q, const uint16_t* ukv, int ld_kv, int M, int Hq, int Hkv,
                             int D, const float* q_norm, const float* k_norm, const int32_t* ctx, const RopeTable& rt,
                             uint16_t* q, uint16_t* k, uint16_t* v, uint16_t* gate, cudaStream_t s) {
  attn_prep_kernel<<<dim3(M, (2 * Hq + 2 * Hkv + kPrepHeads - 1) / kPrepHeads), D, 0, s>>>(uq, ld_q, ukv, ld_kv, Hq, Hkv, D, q_norm, k_norm, ctx, rt, q, k,
                                                           v, gate);
  return cudaGetLastError();
}

}  // namespace vp
