// Gated DeltaNet verify scan (vp_gdn_scan): the recurrent core of the pages' 48 Gated DeltaNet layers
// for the verify rows, with the state double-buffered by step parity.
//
// Sources: "Beating Splash on an M5 Max", section "What actually moved the needle" (the fused GDN
// step writes out of place from parity buffer A to parity buffer B; a partly rejected round re-scans
// only the committed rows from the intact A; the state after every possible number of kept tokens
// must match a reference scan exactly); "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5
// Max", sections "What one token costs the bus" (fp32 state (v_heads, dk, dv), 48 x 128 x 128 per
// layer, read and written once per pass) and "The megakernel is per layer, not per step" (the commit
// pass recomputes the recurrence over the committed tokens).  The recurrence is the published gated
// delta rule (Yang, Kautz and Hatamizadeh, "Gated Delta Networks", 2024), per head with S dv x dk:
//   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,   o_t = S_t q_t.
//
// GB300 design: the rows of S evolve independently (row i needs only S[i, :], k, q, v_i), so a head's
// 128 x 128 fp32 state is cut into four 32-row blocks, one CTA each, grid (4, heads, lanes); a thread
// keeps 16 entries of one row (every 8th column) in registers for the whole scan, its 8-thread group
// reduces S[i, :] . k and S[i, :] . q with a fixed shuffle tree, and the k, q of all rows sit in
// shared memory (loaded with the state, so the scan itself waits on no memory).  The state is read
// once and written once: the kernel streams 2 x 64 KB per head.
// The verify scan (8 rows) and the commit re-scan (the committed count) are the same code, so a
// re-scan of n rows reproduces the verify scan's state after n rows bit for bit.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "errors.h"
#include "gdn_step.cuh"
#include "internal.h"
#include "verify.h"

namespace vp {

namespace {

constexpr int kDk = kGdnDk, kDv = kGdnDv;
constexpr int kRowsPerCta = 32;   // rows of S per CTA
constexpr int kSeg = kGdnSeg;     // entries of a row per thread (8 threads per row)
constexpr int kThreadsG = kRowsPerCta * (kDk / kSeg);  // 256
constexpr int kTpr = kGdnTpr;     // threads per row

__device__ __forceinline__ float bf(const uint16_t* p, size_t i) { return __uint_as_float((uint32_t)p[i] << 16); }

__global__ void __launch_bounds__(kThreadsG) gdn_scan_kernel(const float* __restrict__ state_in,
                                                            float* __restrict__ state_out,
                                                            const uint16_t* __restrict__ q,
                                                            const uint16_t* __restrict__ k,
                                                            const uint16_t* __restrict__ v,
                                                            const float* __restrict__ alpha,
                                                            const float* __restrict__ beta,
                                                            const int32_t* __restrict__ rows, int H,
                                                            float* __restrict__ out) {
  __shared__ float sk[8][kDk], sq[8][kDk], sab[8][2];
  const int rb = blockIdx.x, h = blockIdx.y, l = blockIdx.z, t = threadIdx.x;
  // thread t holds columns c0 + 8 e (e = 0..15) of row i: the 8 threads of a row read 8 consecutive
  // shared-memory words per step (conflict-free) and 32 consecutive bytes of the state per load
  const int i = rb * kRowsPerCta + t / kTpr, c0 = t % kTpr;
  const size_t so = (((size_t)l * H + h) * kDv + i) * kDk + c0;
  int n = rows[l];
  n = n < 0 ? 0 : (n > 8 ? 8 : n);  // a lane scans at most its 8 verify rows
  // Every row's k, q, alpha, beta and this thread's v_i are loaded up front, with the state: one
  // memory round trip, then the scan runs from registers and shared memory.
  float vi[8];
  for (int j = 0; j < n; ++j) {
    const size_t rh = (size_t)(8 * l + j) * H + h;
    if (t < kDk)
      sk[j][t] = bf(k, rh * kDk + t);
    else if (t < 2 * kDk)
      sq[j][t - kDk] = bf(q, rh * kDk + (t - kDk));
    if (t < 2) sab[j][t] = t == 0 ? alpha[rh] : beta[rh];
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) vi[j] = j < n ? bf(v, ((size_t)(8 * l + j) * H + h) * kDv + i) : 0.0f;
  float s[kSeg];
#pragma unroll
  for (int e = 0; e < kSeg; ++e) s[e] = state_in[so + kTpr * e];
  __syncthreads();
  gdn_scan_rows(s, sk, sq, sab, vi, n, c0, [&](int j, float o) {
    if (out && c0 == 0) out[((size_t)(8 * l + j) * H + h) * kDv + i] = o;
  });
#pragma unroll
  for (int e = 0; e < kSeg; ++e) state_out[so + kTpr * e] = s[e];
}

bool aligned_to(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

}  // namespace vp

extern "C" vp_status vp_gdn_scan(const float* state_in, float* state_out, const void* q, const void* k, const void* v,
                                 const float* alpha, const float* beta, const int32_t* rows, int M, int H, int dk,
                                 int dv, float* out, void* stream) {
  using namespace vp;
  if (!state_in || !state_out || !q || !k || !v || !alpha || !beta || !rows) return VP_ERR_INVALID_ARG;
  if (M < 8 || M > kMaxM || M % 8 || H < 1 || H > 4096 || dk != kDk || dv != kDv) return VP_ERR_SHAPE;
  if (!aligned_to(state_in, 4) || !aligned_to(state_out, 4) || !aligned_to(q, 2) || !aligned_to(k, 2) ||
      !aligned_to(v, 2) || !aligned_to(alpha, 4) || !aligned_to(beta, 4) || !aligned_to(rows, 4) ||
      (out && !aligned_to(out, 4)))
    return VP_ERR_ALIGNMENT;
  gdn_scan_kernel<<<dim3(kDv / kRowsPerCta, (unsigned)H, (unsigned)(M / 8)), kThreadsG, 0, (cudaStream_t)stream>>>(
      state_in, state_out, static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
      static_cast<const uint16_t*>(v), alpha, beta, rows, H, out);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}
