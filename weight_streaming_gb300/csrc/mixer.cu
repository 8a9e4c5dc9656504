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

// A / B projections of a Gated DeltaNet layer on r = bf16(RMSNorm(h)) (unit weight): block j < n_v
// computes a[t][j] = r_t . A[j], block n_v + j computes b[t][j] = r_t . B[j], for every row t, in fp32.
// Each block recomputes the rows' statistic (the same fixed-order sum as every other block).
__global__ void __launch_bounds__(256) ab_proj_kernel(const uint16_t* __restrict__ h, int hidden, int M, float eps,
                                                      const uint16_t* __restrict__ wa, const uint16_t* __restrict__ wb,
                                                      int n_v, float* __restrict__ a, float* __restrict__ b) {
  __shared__ float red[8];
  const int j = blockIdx.x, tid = threadIdx.x;
  const uint16_t* w = j < n_v ? wa + (size_t)j * hidden : wb + (size_t)(j - n_v) * hidden;
  for (int t = 0; t < M; ++t) {
    const uint16_t* x = h + (size_t)t * hidden;
    float ss = 0.0f;
    for (int k = tid; k < hidden; k += blockDim.x) ss = fmaf(bfv(x[k]), bfv(x[k]), ss);
    const float inv = 1.0f / sqrtf(block_sum(ss, red) / (float)hidden + eps);
    float acc = 0.0f;
    for (int k = tid; k < hidden; k += blockDim.x) acc = fmaf(bfv(to_bf(bfv(x[k]) * inv)), bfv(w[k]), acc);
    const float s = block_sum(acc, red);
    if (tid == 0) (j < n_v ? a + (size_t)t * n_v + j : b + (size_t)t * n_v + (j - n_v))[0] = s;
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

// Gates per row and v head: alpha = exp(-exp(A_log) * softplus(a + dt_bias)), beta = sigmoid(b).
__global__ void gdn_gates_kernel(const float* __restrict__ a, const float* __restrict__ b,
                                 const float* __restrict__ a_log, const float* __restrict__ dt_bias, int n_v, int M,
                                 float* __restrict__ alpha, float* __restrict__ beta) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= M * n_v) return;
  const int j = idx % n_v;
  const float x = a[idx] + dt_bias[j];
  const float sp = x > 20.0f ? x : log1pf(expf(x));
  alpha[idx] = expf(-expf(a_log[j]) * sp);
  beta[idx] = 1.0f / (1.0f + expf(-b[idx]));
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

// Attention producer steps, block (row t, head) of D threads: heads 0 .. Hq - 1 the queries
// (uq[t][h D + i]), Hq .. Hq + Hkv - 1 the keys (ukv[t][h D + i]): each over its root mean square
// (eps 1e-6) times the shared weight (q_norm / k_norm), then the rotary embedding over the whole
// head at the row's cache position ctx[lane] + t % 8 (pairs (2j, 2j + 1) rotated by
// pos * 10000^(-2j / D); angle in fp64), then bf16.  Then Hkv value heads and Hq gate heads, copied
// to dense [M][heads][D] rows.
__global__ void attn_prep_kernel(const uint16_t* __restrict__ uq, int ld_q, const uint16_t* __restrict__ ukv,
                                 int ld_kv, int Hq, int Hkv, int D, const float* __restrict__ q_norm,
                                 const float* __restrict__ k_norm, const int32_t* __restrict__ ctx,
                                 uint16_t* __restrict__ q, uint16_t* __restrict__ k, uint16_t* __restrict__ v,
                                 uint16_t* __restrict__ gate) {
  __shared__ float red[8];
  __shared__ float xs[512];
  const int t = blockIdx.x, hh = blockIdx.y, i = threadIdx.x;
  if (hh < Hq + Hkv) {
    const bool isq = hh < Hq;
    const int h = isq ? hh : hh - Hq;
    const float x = bfv(isq ? uq[(size_t)t * ld_q + h * D + i] : ukv[(size_t)t * ld_kv + h * D + i]);
    const float ms = block_sum(x * x, red) / (float)D;
    xs[i] = x / sqrtf(ms + 1e-6f) * (isq ? q_norm[i] : k_norm[i]);
    __syncthreads();
    const int j = i >> 1;
    const double pos = (double)ctx[t >> 3] + (double)(t & 7);
    const double ang = pos * pow(10000.0, -2.0 * (double)j / (double)D);
    double sn, cs;
    sincos(ang, &sn, &cs);
    const float x0 = xs[2 * j], x1 = xs[2 * j + 1];
    const float r = (i & 1) ? (float)((double)x0 * sn + (double)x1 * cs) : (float)((double)x0 * cs - (double)x1 * sn);
    (isq ? q + ((size_t)t * Hq + h) * D : k + ((size_t)t * Hkv + h) * D)[i] = to_bf(r);
  } else if (hh < Hq + 2 * Hkv) {
    const int h = hh - Hq - Hkv;
    v[((size_t)t * Hkv + h) * D + i] = ukv[(size_t)t * ld_kv + (Hkv + h) * D + i];
  } else {
    const int h = hh - Hq - 2 * Hkv;
    gate[((size_t)t * Hq + h) * D + i] = uq[(size_t)t * ld_q + (Hq + h) * D + i];
  }
}

}  // namespace

cudaError_t launch_ab_proj(const uint16_t* h, int hidden, int M, float eps, const uint16_t* wa, const uint16_t* wb,
                           int n_v, float* a, float* b, cudaStream_t s) {
  ab_proj_kernel<<<2 * n_v, 256, 0, s>>>(h, hidden, M, eps, wa, wb, n_v, a, b);
  return cudaGetLastError();
}

cudaError_t launch_gdn_prep(const uint16_t* u, int ld_u, int M, const uint16_t* window_a, const uint16_t* taps,
                            int n_qk, int n_v, int d, uint16_t* q, uint16_t* k, uint16_t* v, uint16_t* conv_hist,
                            int32_t* rows8, const float* a, const float* b, const float* a_log, const float* dt_bias,
                            float* alpha, float* beta, cudaStream_t s) {
  gdn_prep_kernel<<<dim3(M, 2 * n_qk + n_v), d, 0, s>>>(u, ld_u, window_a, taps, n_qk, n_v, d, q, k, v, conv_hist,
                                                        rows8);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  gdn_gates_kernel<<<(M * n_v + 127) / 128, 128, 0, s>>>(a, b, a_log, dt_bias, n_v, M, alpha, beta);
  return cudaGetLastError();
}

cudaError_t launch_gated_norm(const float* o, const uint16_t* u, int ld_u, int z0, const float* w, int M, int n_v,
                              int d, uint16_t* out, cudaStream_t s) {
  gated_norm_kernel<<<dim3(M, n_v), d, 0, s>>>(o, u, ld_u, z0, w, n_v, d, out);
  return cudaGetLastError();
}

cudaError_t launch_attn_prep(const uint16_t* uq, int ld_q, const uint16_t* ukv, int ld_kv, int M, int Hq, int Hkv,
                             int D, const float* q_norm, const float* k_norm, const int32_t* ctx, uint16_t* q,
                             uint16_t* k, uint16_t* v, uint16_t* gate, cudaStream_t s) {
  attn_prep_kernel<<<dim3(M, 2 * Hq + 2 * Hkv), D, 0, s>>>(uq, ld_q, ukv, ld_kv, Hq, Hkv, D, q_norm, k_norm, ctx, q, k,
                                                           v, gate);
  return cudaGetLastError();
}

}  // namespace vp
