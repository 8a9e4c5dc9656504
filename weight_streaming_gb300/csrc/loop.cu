// A device-resident decode loop around the verify pass: the embedding gather of the pass's rows, the
// history append of the committed tokens, lookup drafts from the history, and vp_decode_steps, which
// enqueues any number of rounds with no host synchronisation (so the whole loop can be one CUDA
// graph).
//
// Sources: "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max", section "What one token
// costs the bus" (the embedding is a gather of the 4-bit table; the pass streams everything else)
// and section "The megakernel is per layer, not per step" (a round commits 1..8 tokens: the accepted
// drafts, then the target's token after them); "Speculative decoding" (mlx-dspark), sections "Lookup
// (no drafter)" and "Lookup drafts" (when the text being written already appeared earlier in the
// context, the continuation of that earlier match is a free draft); "Beating Splash on an M5 Max",
// section "The kernels were not the gap" (host synchronisations per round were the cost, the GPU sat
// idle between command buffers).
//
// Per lane the state lives on the device: the token history hist[l][0 .. T_l) (T_l = hist_len[l]; its
// last token is the anchor, already committed) and a status word.  One round: x0 = embed(pending),
// the verify pass (argmax + greedy accept), append the committed tokens, lookup drafts -> pending.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "errors.h"
#include "internal.h"
#include "ptx.cuh"
#include "verify.h"

namespace vp {

namespace {

constexpr int kStatusShapeL = 2;  // VP_ERR_SHAPE

// x[m][k] = bf16(e2m1(code) * e4m3(scale) * ts) of row tokens[m] of a canonical NVFP4 table
// (codes [V][K/2], low nibble first; scales [V][K/16]), rounded once (the product is exact in fp64).
__global__ void embed_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, float ts,
                             const int32_t* __restrict__ tokens, int V, int K, uint16_t* __restrict__ x,
                             int* status) {
  const int m = blockIdx.x;
  const int t = tokens[m];
  uint16_t* row = x + (size_t)m * K;
  if (t < 0 || t >= V) {  // an out-of-range token: a zero row and VP_ERR_SHAPE
    for (int k = threadIdx.x; k < K; k += blockDim.x) row[k] = 0;
    if (threadIdx.x == 0 && status) atomicExch(status, kStatusShapeL);
    return;
  }
  for (int j = threadIdx.x; j < K / 2; j += blockDim.x) {
    const uint32_t byte = codes[(size_t)t * (K / 2) + j];
    const uint32_t sc = e4m3x2_to_f16x2(scales[(size_t)t * (K / 16) + (2 * j) / 16]);
    uint32_t pair[4];
    e2m1x8_to_f16x2x4(byte, pair);  // byte 0 -> pair[0]: (low nibble, high nibble)
    const __half2 w = *reinterpret_cast<const __half2*>(&pair[0]);
    const float s = __half2float(*reinterpret_cast<const __half*>(&sc));
    row[2 * j] = __bfloat16_as_ushort(__double2bfloat16((double)(__low2float(w) * s) * (double)ts));
    row[2 * j + 1] = __bfloat16_as_ushort(__double2bfloat16((double)(__high2float(w) * s) * (double)ts));
  }
}

// Appends committed[l][0 .. n_commit[l]) (rows of R entries) to lane l's history (one thread per
// lane); a lane whose history would overflow is left as it is and VP_ERR_SHAPE is reported.
__global__ void append_kernel(int32_t* __restrict__ hist, int32_t* __restrict__ hist_len, int L, int cap, int R,
                              const int32_t* __restrict__ n_commit, const int32_t* __restrict__ committed,
                              int* status) {
  const int l = threadIdx.x;
  if (l >= L) return;
  const int n = n_commit[l], T = hist_len[l];
  if (n < 1 || n > R || T < 0 || T + n > cap) {
    if (status) atomicExch(status, kStatusShapeL);
    return;
  }
  for (int j = 0; j < n; ++j) hist[(size_t)l * cap + T + j] = committed[R * l + j];
  hist_len[l] = T + n;
}

// Lookup drafts, one CTA per lane: every earlier position p (continuation hist[p..]) scores the
// number of tokens before it that match the history's last tokens (up to max_match); the best score
// wins, the latest p among equals (one key: score * 2^24 + p, reduced by maximum).
// The anchor and R - 1 drafts go to pending[R l .. R l + R - 1].
__global__ void __launch_bounds__(256) lookup_kernel(const int32_t* __restrict__ hist,
                                                    const int32_t* __restrict__ hist_len, int cap, int max_match,
                                                    int R, int32_t* __restrict__ pending, int* status) {
  __shared__ int red[8];
  const int l = blockIdx.x, tid = threadIdx.x;
  const int32_t* h = hist + (size_t)l * cap;
  const int T = hist_len[l];
  if (T < 1 || T > cap) {
    if (tid < R) pending[R * l + tid] = 0;
    if (tid == 0 && status) atomicExch(status, kStatusShapeL);
    return;
  }
  int best = 0;
  for (int p = 1 + tid; p < T; p += blockDim.x) {
    int len = 0;
    while (len < max_match && p - 1 - len >= 0 && h[p - 1 - len] == h[T - 1 - len]) ++len;
    if (len >= 1) best = max(best, (len << 24) | p);
  }
  for (int o = 16; o; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  if ((tid & 31) == 0) red[tid >> 5] = best;
  __syncthreads();
  if (tid != 0) return;
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) best = max(best, red[w]);
  const int p = best ? (best & 0xFFFFFF) : -1;
  const int32_t anchor = h[T - 1];
  pending[R * l] = anchor;
  int32_t last = anchor;
  for (int j = 0; j < R - 1; ++j) {
    if (p >= 0 && p + j < T) last = h[p + j];
    pending[R * l + 1 + j] = last;
  }
}

bool al(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

}  // namespace vp

using namespace vp;

extern "C" {

vp_status vp_embed_nvfp4(const void* codes, const void* scales, float ts, const int32_t* tokens, int M, int V, int K,
                         void* x, int* status, void* stream) {
  if (!codes || !scales || !tokens || !x) return VP_ERR_INVALID_ARG;
  if (M < 1 || V < 1 || K < 16 || K % 16 || (long long)V * K >= (1LL << 40)) return VP_ERR_SHAPE;
  if (!al(tokens, 4) || !al(x, 2) || (status && !al(status, 4))) return VP_ERR_ALIGNMENT;
  embed_kernel<<<M, 256, 0, (cudaStream_t)stream>>>(static_cast<const uint8_t*>(codes),
                                                    static_cast<const uint8_t*>(scales), ts, tokens, V, K,
                                                    static_cast<uint16_t*>(x), status);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

vp_status vp_lookup_drafts_rows(const int32_t* hist, const int32_t* hist_len, int lanes, int rows, int cap,
                                int max_match, int32_t* pending, int* status, void* stream) {
  if (!hist || !hist_len || !pending) return VP_ERR_INVALID_ARG;
  if (rows < 1 || rows > kMaxM || lanes < 1 || lanes > kMaxM || lanes * rows > kMaxRows || cap < 1 ||
      cap >= (1 << 24) || max_match < 1 || max_match > 127)
    return VP_ERR_SHAPE;
  if (!al(hist, 4) || !al(hist_len, 4) || !al(pending, 4) || (status && !al(status, 4))) return VP_ERR_ALIGNMENT;
  lookup_kernel<<<lanes, 256, 0, (cudaStream_t)stream>>>(hist, hist_len, cap, max_match, rows, pending, status);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

vp_status vp_lookup_drafts(const int32_t* hist, const int32_t* hist_len, int lanes, int cap, int max_match,
                           int32_t* pending, int* status, void* stream) {
  if (lanes > kMaxM / 8) return VP_ERR_SHAPE;
  return vp_lookup_drafts_rows(hist, hist_len, lanes, 8, cap, max_match, pending, status, stream);
}

vp_status vp_commit_append_rows(int32_t* hist, int32_t* hist_len, int lanes, int rows, int cap,
                                const int32_t* n_commit, const int32_t* committed, int* status, void* stream) {
  if (!hist || !hist_len || !n_commit || !committed) return VP_ERR_INVALID_ARG;
  if (rows < 1 || rows > kMaxM || lanes < 1 || lanes > kMaxM || lanes * rows > kMaxRows || cap < 1) return VP_ERR_SHAPE;
  if (!al(hist, 4) || !al(hist_len, 4) || !al(n_commit, 4) || !al(committed, 4) || (status && !al(status, 4)))
    return VP_ERR_ALIGNMENT;
  append_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(hist, hist_len, lanes, cap, rows, n_commit, committed, status);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

vp_status vp_commit_append(int32_t* hist, int32_t* hist_len, int lanes, int cap, const int32_t* n_commit,
                           const int32_t* committed, int* status, void* stream) {
  if (lanes > kMaxM / 8) return VP_ERR_SHAPE;
  return vp_commit_append_rows(hist, hist_len, lanes, 8, cap, n_commit, committed, status, stream);
}

vp_status vp_decode_steps_rows(const vp_model* model, int steps, int rows, const void* emb_codes,
                               const void* emb_scales, float emb_ts, int vocab, int hidden, int32_t* hist,
                               int32_t* hist_len, int cap, int lanes, int max_match, int32_t* pending, void* x0,
                               int32_t* argmax, int32_t* n_commit, int32_t* committed, void* ws, size_t ws_bytes,
                               int* status, void* stream) {
  if (!model || !emb_codes || !emb_scales || !hist || !hist_len || !pending || !x0 || !argmax || !n_commit ||
      !committed || !ws)
    return VP_ERR_INVALID_ARG;
  if (steps < 0 || rows < 1 || rows > kMaxM || lanes < 1 || lanes * rows > kMaxRows) return VP_ERR_SHAPE;
  const int M = rows * lanes;
  if (M > kMaxM && (M % kMaxM || kMaxM % rows)) return VP_ERR_SHAPE;  // passes of 32 rows, whole lanes
  // Every argument of the four steps is checked before the first launch, so a bad call enqueues
  // nothing.  (The pass's own per-phase checks still run inside vp_verify_pass.)
  if (vocab < 1 || hidden < 16 || hidden % 16 || (long long)vocab * hidden >= (1LL << 40) || cap < 1 ||
      cap >= (1 << 24) || max_match < 1 || max_match > 127)
    return VP_ERR_SHAPE;
  // The embedding writes x0 rows of `hidden` values and the pass reads rows of the model's width.
  if (hidden != vp::model_hidden(model)) return VP_ERR_SHAPE;
  if (!al(hist, 4) || !al(hist_len, 4) || !al(pending, 4) || !al(x0, 16) || !al(argmax, 4) || !al(n_commit, 4) ||
      !al(committed, 4) || !al(ws, 256) || (status && !al(status, 4)))
    return VP_ERR_ALIGNMENT;
  const size_t need = vp_pass_workspace_bytes(model, M);
  if (need == 0) return VP_ERR_SHAPE;
  if (ws_bytes < need) return VP_ERR_WORKSPACE;
  for (int s = 0; s < steps; ++s) {
    vp_status st = vp_embed_nvfp4(emb_codes, emb_scales, emb_ts, pending, M, vocab, hidden, x0, status, stream);
    if (st != VP_OK) return st;
    st = vp_verify_pass_rows(model, x0, M, rows, pending, argmax, n_commit, committed, nullptr, nullptr, ws,
                             ws_bytes, stream);
    if (st != VP_OK) return st;
    st = vp_commit_append_rows(hist, hist_len, lanes, rows, cap, n_commit, committed, status, stream);
    if (st != VP_OK) return st;
    st = vp_lookup_drafts_rows(hist, hist_len, lanes, rows, cap, max_match, pending, status, stream);
    if (st != VP_OK) return st;
  }
  return VP_OK;
}

vp_status vp_decode_steps(const vp_model* model, int steps, const void* emb_codes, const void* emb_scales,
                          float emb_ts, int vocab, int hidden, int32_t* hist, int32_t* hist_len, int cap,
                          int lanes, int max_match, int32_t* pending, void* x0, int32_t* argmax, int32_t* n_commit,
                          int32_t* committed, void* ws, size_t ws_bytes, int* status, void* stream) {
  if (lanes > kMaxM / 8) return VP_ERR_SHAPE;
  return vp_decode_steps_rows(model, steps, 8, emb_codes, emb_scales, emb_ts, vocab, hidden, hist, hist_len, cap,
                              lanes, max_match, pending, x0, argmax, n_commit, committed, ws, ws_bytes, status,
                              stream);
}

}  // extern "C"
