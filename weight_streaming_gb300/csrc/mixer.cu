// The pass's real mixer cores between the executor's projections: the whole Gated DeltaNet core in one
// launch (A / B projections and gates, short convolution, Q / K normalisation, the delta-rule scan of
// gdn_step.cuh, the gated RMSNorm), and the attention layer's Q / K RMSNorm and rotary embedding
// ahead of its core over the KV cache (attention.cu).
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

#include "gdn_step.cuh"

#include <cstdint>

#include "mixer.h"

namespace vp {

namespace {

__device__ __forceinline__ float bfv(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t to_bf(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

// ---------------------------------------------------------------- the Gated DeltaNet core
// One cluster of 4 CTAs per (v head hv, lane); CTA rank rb of the cluster owns rows rb * 32 .. + 31
// of the head's 128 x 128 state and quarter rb of K for the A / B projections.  The CTAs exchange
// partial sums through distributed shared memory at cluster barriers (every CTA then adds the four
// partials in rank order, so all four hold the same values):
//  1. r_t = bf16(RMSNorm(h_t)) (unit weight): sums of squares of the rows' K quarters, exchanged;
//     then the K quarter's dot products with A[hv] and B[hv], exchanged; alpha_t = exp(-exp(A_log)
//     softplus(a + dt_bias)), beta_t = sigmoid(b);
//  2. the causal depthwise 4-tap convolution of u's q, k, v channels over the lane's window (3 earlier
//     rows) and its 8 rows (tap 3 on the current row), SiLU; q, k of q/k head hv / (n_v / n_qk) over
//     their L2 norm (eps 1e-6 inside the root), bf16; v of the CTA's 32 channels, bf16; the
//     convolution history (the window, then the 8 rows' inputs) of the channels the CTA owns;
//  3. the delta rule over the 8 rows (gdn_step.cuh) from state_in into state_out; the scan's inputs
//     (q, k per q/k head, v, alpha, beta) are recorded for the commit re-scan;
//  4. the gated RMSNorm per row and head: o / sqrt(mean(o^2) + 1e-6) * norm_w * silu(z), the sum of
//     squares over the head's 128 outputs exchanged, then bf16 into the out-projection's input.
constexpr int kCoreThreads = 256, kCoreRows = 32, kCoreCta = 4;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of all CTAs of the cluster: writes to shared memory before it are visible after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// p in CTA rank's shared memory (the same variable as p in this CTA's).
__device__ __forceinline__ float ld_cluster(const float* p, uint32_t rank) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
  return v;
}
// Per-warp partial sums of n values (n <= 24) into red[warp][.], then thread i < n adds the warps
// [w0, w1) in order; the caller synchronises before reading the result.
template <int N>
__device__ __forceinline__ void warp_partials(const float (&v)[N], float (*red)[24]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int e = 0; e < N; ++e) {
    float x = v[e];
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) red[warp][e] = x;
  }
}

__global__ void __cluster_dims__(kCoreCta, 1, 1) __launch_bounds__(kCoreThreads) gdn_core_kernel(const GdnCoreArgs a) {
  __shared__ float sk[8][kGdnDk], sq[8][kGdnDk], sab[8][2], sv[8][kCoreRows], so[8][kCoreRows];
  __shared__ float red[kCoreThreads / 32][24];
  __shared__ float xp[8 + 16 + 8];  // exchanged partials: sums of squares of h, a and b, sums of o^2
  __shared__ float inv[8], onorm[8];
  const uint32_t rb = cluster_rank();
  const int hv = blockIdx.y, l = blockIdx.z, tid = threadIdx.x, warp = tid >> 5;
  const int n_qk = a.n_qk, n_v = a.n_v, C = (2 * n_qk + n_v) * kGdnDk, head_qk = hv / (n_v / n_qk);
  const int i = rb * kCoreRows + tid / kGdnTpr, c0 = tid % kGdnTpr;  // state row and column phase
  const size_t so_off = (((size_t)l * n_v + hv) * kGdnDv + i) * kGdnDk + c0;
  float s[kGdnSeg];
#pragma unroll
  for (int e = 0; e < kGdnSeg; ++e) s[e] = a.state_in[so_off + kGdnTpr * e];

  // 1. A / B projections and gates: chunk (8 values) rb * qc + tid of K, for the lane's 8 rows
  const int qc = a.hidden / 32, ch = rb * qc + tid;
  const bool kin = tid < qc;
  uint4 hx[8];
#pragma unroll
  for (int t = 0; t < 8; ++t)
    hx[t] = kin ? *reinterpret_cast<const uint4*>(a.h + (size_t)(8 * l + t) * a.hidden + 8 * ch) : make_uint4(0, 0, 0, 0);
  {
    float p[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t x4[4] = {hx[t].x, hx[t].y, hx[t].z, hx[t].w};
      p[t] = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(x4[e] << 16), hi = __uint_as_float(x4[e] & 0xFFFF0000u);
        p[t] = fmaf(lo, lo, p[t]);
        p[t] = fmaf(hi, hi, p[t]);
      }
    }
    warp_partials(p, red);
  }
  __syncthreads();
  if (tid < 8) {
    float x = 0.0f;
    for (int w = 0; w < kCoreThreads / 32; ++w) x += red[w][tid];
    xp[tid] = x;
  }
  cluster_sync();
  if (tid < 8) {
    float x = 0.0f;
    for (uint32_t r = 0; r < kCoreCta; ++r) x += ld_cluster(&xp[tid], r);
    inv[tid] = 1.0f / sqrtf(x / (float)a.hidden + a.eps);
  }
  __syncthreads();
  {
    const uint4 wa = kin ? *reinterpret_cast<const uint4*>(a.wa + (size_t)hv * a.hidden + 8 * ch) : make_uint4(0, 0, 0, 0);
    const uint4 wb = kin ? *reinterpret_cast<const uint4*>(a.wb + (size_t)hv * a.hidden + 8 * ch) : make_uint4(0, 0, 0, 0);
    const uint32_t a4[4] = {wa.x, wa.y, wa.z, wa.w}, b4[4] = {wb.x, wb.y, wb.z, wb.w};
    float p[16];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t x4[4] = {hx[t].x, hx[t].y, hx[t].z, hx[t].w};
      p[t] = p[8 + t] = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float r0 = bfv(to_bf(__uint_as_float(x4[e] << 16) * inv[t]));
        const float r1 = bfv(to_bf(__uint_as_float(x4[e] & 0xFFFF0000u) * inv[t]));
        p[t] = fmaf(r0, __uint_as_float(a4[e] << 16), p[t]);
        p[t] = fmaf(r1, __uint_as_float(a4[e] & 0xFFFF0000u), p[t]);
        p[8 + t] = fmaf(r0, __uint_as_float(b4[e] << 16), p[8 + t]);
        p[8 + t] = fmaf(r1, __uint_as_float(b4[e] & 0xFFFF0000u), p[8 + t]);
      }
    }
    __syncthreads();  // red is reused
    warp_partials(p, red);
  }
  __syncthreads();
  if (tid < 16) {
    float x = 0.0f;
    for (int w = 0; w < kCoreThreads / 32; ++w) x += red[w][tid];
    xp[8 + tid] = x;
  }
  cluster_sync();
  if (tid < 16) {
    float x = 0.0f;
    for (uint32_t r = 0; r < kCoreCta; ++r) x += ld_cluster(&xp[8 + tid], r);
    float g;
    if (tid < 8) {
      const float z = x + a.dt_bias[hv];
      const float sp = z > 20.0f ? z : log1pf(expf(z));
      g = expf(-expf(a.a_log[hv]) * sp);
    } else {
      g = 1.0f / (1.0f + expf(-x));
    }
    sab[tid & 7][tid >> 3] = g;
    if (rb == 0) a.rec_ab[((size_t)(8 * l + (tid & 7)) * n_v + hv) * 2 + (tid >> 3)] = g;
  }

  // 2. convolution: threads 0..127 the q channel, 128..255 the k channel of q/k head head_qk;
  //    threads 0..31 also the CTA's 32 v channels
  const uint16_t* win = a.window_a + (size_t)l * 3 * C;
  uint16_t* hist = a.conv_hist + (size_t)l * 11 * C;
  auto conv = [&](int c, float (&y)[8], bool keep) {
    float e[11];
    uint16_t eb[11];
#pragma unroll
    for (int r = 0; r < 11; ++r) {
      eb[r] = r < 3 ? win[(size_t)r * C + c] : a.u[(size_t)(8 * l + r - 3) * a.ld_u + c];
      e[r] = bfv(eb[r]);
    }
    float tp[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) tp[j] = bfv(a.taps[(size_t)c * 4 + j]);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      float acc = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) acc = fmaf(tp[j], e[t + j], acc);
      y[t] = silu(acc);
    }
    if (keep)
#pragma unroll
      for (int r = 0; r < 11; ++r) hist[(size_t)r * C + c] = eb[r];
  };
  {
    const bool isk = tid >= kGdnDk;
    const int c = (isk ? n_qk + head_qk : head_qk) * kGdnDk + (tid & (kGdnDk - 1));
    float y[8];
    conv(c, y, rb == 0 && hv % (n_v / n_qk) == 0);  // one CTA keeps each q / k channel's history
    float p[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) p[t] = y[t] * y[t];
    warp_partials(p, red);
    __syncthreads();
    const bool rec_qk = rb == 0 && hv % (n_v / n_qk) == 0;  // one CTA records each q / k head
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int w0 = isk ? 4 : 0;
      const float n2 = red[w0][t] + red[w0 + 1][t] + red[w0 + 2][t] + red[w0 + 3][t];
      const uint16_t b = to_bf(y[t] / sqrtf(n2 + 1e-6f));
      (isk ? sk : sq)[t][tid & (kGdnDk - 1)] = bfv(b);
      if (rec_qk) a.rec_qk[(((size_t)(8 * l + t) * 2 + isk) * n_qk + head_qk) * kGdnDk + (tid & (kGdnDk - 1))] = b;
    }
    if (tid < kCoreRows) {
      float yv[8];
      conv((2 * n_qk + hv) * kGdnDv + rb * kCoreRows + tid, yv, true);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const uint16_t b = to_bf(yv[t]);
        sv[t][tid] = bfv(b);
        a.rec_v[((size_t)(8 * l + t) * n_v + hv) * kGdnDv + rb * kCoreRows + tid] = b;
      }
    }
  }
  __syncthreads();

  // 3. the delta rule over the 8 rows
  float vi[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) vi[t] = sv[t][tid / kGdnTpr];
  gdn_scan_rows(s, sk, sq, sab, vi, 8, c0, [&](int t, float o) {
    if (c0 == 0) so[t][tid / kGdnTpr] = o;
  });
#pragma unroll
  for (int e = 0; e < kGdnSeg; ++e) a.state_out[so_off + kGdnTpr * e] = s[e];
  __syncthreads();

  // 4. gated RMSNorm: the head's sum of o^2 per row from the four CTAs' 32 rows each
  if (tid < 8) {
    float x = 0.0f;
    for (int r = 0; r < kCoreRows; ++r) x = fmaf(so[tid][r], so[tid][r], x);
    xp[24 + tid] = x;
  }
  cluster_sync();
  if (tid < 8) {
    float x = 0.0f;
    for (uint32_t r = 0; r < kCoreCta; ++r) x += ld_cluster(&xp[24 + tid], r);
    onorm[tid] = x / (float)kGdnDv;
  }
  __syncthreads();
  {
    const int t = tid / kCoreRows, r = tid % kCoreRows, ch = rb * kCoreRows + r;
    const float z = bfv(a.u[(size_t)(8 * l + t) * a.ld_u + a.z0 + hv * kGdnDv + ch]);
    a.out[(size_t)(8 * l + t) * n_v * kGdnDv + hv * kGdnDv + ch] =
        to_bf(so[t][r] / sqrtf(onorm[t] + 1e-6f) * a.norm_w[ch] * silu(z));
  }
  cluster_sync();  // no CTA leaves while another may still read its shared memory
}

// The commit re-scan of every Gated DeltaNet layer: CTA (rb, hv, layer x lane) re-runs the delta
// rule of gdn_step.cuh over the lane's first n = n_commit[lane] rows from the intact state_in into
// state_out, from the inputs the pass recorded (the same values, the same arithmetic: n = 8
// reproduces the pass's state bit for bit), and writes the next pass's window, rows n .. n + 2 of
// the convolution history, for the channels it owns (its 32 v channels; the q / k head's channels
// in the CTAs with rb == 0 and hv % (n_v / n_qk) == 0).
__global__ void __launch_bounds__(kCoreThreads) gdn_commit_kernel(const __grid_constant__ GdnCommitArgs a) {
  __shared__ float sk[8][kGdnDk], sq[8][kGdnDk], sab[8][2];
  const int rb = blockIdx.x, hv = blockIdx.y, li = blockIdx.z / a.lanes, l = blockIdx.z % a.lanes, tid = threadIdx.x;
  const int n_qk = a.n_qk, n_v = a.n_v, C = (2 * n_qk + n_v) * kGdnDk, head_qk = hv / (n_v / n_qk);
  const GdnCommitLayer& L = a.layer[li];
  int n = a.n_commit[l];
  n = n < 0 ? 0 : (n > 8 ? 8 : n);
  const int i = rb * kCoreRows + tid / kGdnTpr, c0 = tid % kGdnTpr;
  const size_t so_off = (((size_t)l * n_v + hv) * kGdnDv + i) * kGdnDk + c0;
  const uint16_t* rqk = L.rec_qk;
  for (int t = 0; t < n; ++t) {
    const int isk = tid >> 7, c = tid & (kGdnDk - 1);
    (isk ? sk : sq)[t][c] = bfv(rqk[(((size_t)(8 * l + t) * 2 + isk) * n_qk + head_qk) * kGdnDk + c]);
    if (tid < 2) sab[t][tid] = L.rec_ab[((size_t)(8 * l + t) * n_v + hv) * 2 + tid];
  }
  float vi[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) vi[t] = t < n ? bfv(L.rec_v[((size_t)(8 * l + t) * n_v + hv) * kGdnDv + i]) : 0.0f;
  float s[kGdnSeg];
#pragma unroll
  for (int e = 0; e < kGdnSeg; ++e) s[e] = L.state_in[so_off + kGdnTpr * e];
  __syncthreads();
  gdn_scan_rows(s, sk, sq, sab, vi, n, c0, [](int, float) {});
#pragma unroll
  for (int e = 0; e < kGdnSeg; ++e) L.state_out[so_off + kGdnTpr * e] = s[e];
  // the window after n rows
  const uint16_t* hist = L.conv_hist + (size_t)l * 11 * C;
  uint16_t* win = L.window + (size_t)l * 3 * C;
  auto copy = [&](int c) {
#pragma unroll
    for (int r = 0; r < 3; ++r) win[(size_t)r * C + c] = hist[(size_t)(n + r) * C + c];
  };
  if (tid < kCoreRows) copy((2 * n_qk + hv) * kGdnDv + rb * kCoreRows + tid);
  if (rb == 0 && hv % (n_v / n_qk) == 0) copy(((tid >> 7) ? n_qk + head_qk : head_qk) * kGdnDk + (tid & (kGdnDk - 1)));
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

cudaError_t launch_gdn_commit(const GdnCommitArgs& a, int n_layers, cudaStream_t s) {
  gdn_commit_kernel<<<dim3(kCoreCta, (unsigned)a.n_v, (unsigned)(n_layers * a.lanes)), kCoreThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gdn_core(const GdnCoreArgs& a, int lanes, cudaStream_t s) {
  gdn_core_kernel<<<dim3(kCoreCta, (unsigned)a.n_v, (unsigned)lanes), kCoreThreads, 0, s>>>(a);
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
