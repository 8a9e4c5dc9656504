// One thread's share of the gated delta rule (Yang, Kautz and Hatamizadeh, "Gated Delta Networks",
// 2024) for a head with state S (dv x dk, fp32):
//   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,   o_t = S_t q_t.
// Rows of S evolve independently; a thread keeps kSeg entries of one row (columns c0 + kTpr e) and
// its kTpr-thread group reduces S[i, :] . k and S[i, :] . q with a fixed shuffle tree.  Every kernel
// that advances the state calls this function, so the pass's scan and the commit re-scan perform the
// same arithmetic in the same order (their states agree bit for bit).
#pragma once
#include <cuda_runtime.h>

namespace vp {

constexpr int kGdnDk = 128, kGdnDv = 128;
constexpr int kGdnSeg = 16;                  // entries of a row per thread
constexpr int kGdnTpr = kGdnDk / kGdnSeg;    // 8 threads per row

// s: the thread's entries of row i; sk / sq: k and q of rows 0 .. 7 (fp32 values of bf16);
// sab[j] = (alpha_j, beta_j); vi[j] = v_j[i]; n rows (<= 8).  out(j, o) receives o_j[i] (every thread
// of the row holds it).
template <typename Out>
__device__ __forceinline__ void gdn_scan_rows(float (&s)[kGdnSeg], const float (*sk)[kGdnDk],
                                              const float (*sq)[kGdnDk], const float (*sab)[2], const float (&vi)[8],
                                              int n, int c0, Out out) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= n) break;
    const float a = sab[j][0], b = sab[j][1];
    float u = 0.0f;
#pragma unroll
    for (int e = 0; e < kGdnSeg; ++e) u = fmaf(s[e], sk[j][c0 + kGdnTpr * e], u);
#pragma unroll
    for (int m = 1; m < kGdnTpr; m <<= 1) u += __shfl_xor_sync(0xffffffffu, u, m);
    const float d = b * (vi[j] - a * u);
    float o = 0.0f;
#pragma unroll
    for (int e = 0; e < kGdnSeg; ++e) {
      s[e] = fmaf(d, sk[j][c0 + kGdnTpr * e], a * s[e]);
      o = fmaf(s[e], sq[j][c0 + kGdnTpr * e], o);
    }
#pragma unroll
    for (int m = 1; m < kGdnTpr; m <<= 1) o += __shfl_xor_sync(0xffffffffu, o, m);
    out(j, o);
  }
}

}  // namespace vp
