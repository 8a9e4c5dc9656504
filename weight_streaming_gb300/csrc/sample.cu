// Sampled acceptance over given verify logits (vp_sample_accept): per row the target distribution
// (top_k <= 32 candidates, temperature, top_p truncation, renormalised), then per lane standard
// speculative sampling of the 7 drafts (accept when u * q < p, else a draw from max(p - q, 0)) and the
// bonus draw.
//
// Sources: "144 tok/s needs 502 GB/s" -- "Exact, up to top-32" (the acceptance test u * q < p with
// a residual max(p - q, 0) draw; the target contributes its first top_k <= 32 entries, temperature
// over them, truncated by top_p, renormalised; a token outside them has probability zero);
// "lithos-metal ..." -- "How DSpark is wired in" (a greedy drafter is a point mass); "Beating Splash
// on an M5 Max" -- "What actually moved the needle" (one GPU pass over the verify logits applies
// top-k and top-p, samples and runs the acceptance rule; no logit readback).
//
// One launch on the caller's stream, grid (chunks x M), in three stages:
//  1. every CTA: the top 32 of one 4096-wide chunk of one row.  Candidates are 64-bit keys
//     (order-preserving logit bits, then the complemented token index: a larger key is a larger
//     logit and, among equal logits, the lower index).  Each warp keeps a descending run of 32 keys
//     across its lanes and folds in 32 new keys at a time (warp bitonic sort, then a bitonic merge
//     keeping the larger half); only keys at or above a lower bound of the warp's 32nd largest key
//     are folded in.
//  2. the CTA that finishes a row's last chunk: folds the row's chunk runs the same way and turns
//     the first top_k into the row's distribution (fp32: exp of (l - l_max) / T, top_p prefix,
//     renormalised).
//  3. the CTA that finishes a lane's last row: the acceptance scan over the lane's 8 rows.
#include <cuda_runtime.h>
#include <math.h>

#include <cstdint>

#include "internal.h"
#include "sample.h"

namespace vp {

namespace {

constexpr int kChunk = 4096;   // logits per chunk CTA
constexpr int kCand = 32;      // candidates kept per chunk (= the largest top_k)

// Order-preserving map of a logit to 32 bits (NaN as -inf, -0 as +0), then the token index
// complemented: a larger key is a better candidate.
__device__ __forceinline__ uint64_t cand_key(float v, int idx) {
  if (isnan(v)) v = -INFINITY;
  if (v == 0.0f) v = 0.0f;
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)u << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)idx);
}
__device__ __forceinline__ int key_index(uint64_t k) { return (int)(0xFFFFFFFFu - (uint32_t)k); }

__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m), hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
  return ((uint64_t)hi << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)v, src), hi = __shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src);
  return ((uint64_t)hi << 32) | lo;
}
// Bitonic stages k = kmin .. 32 over the warp's 32 keys (one per lane): lane i ends with the i-th
// largest.  kmin = 2 sorts any input; kmin = 32 (the last stage) sorts a bitonic sequence.
__device__ __forceinline__ uint64_t warp_bitonic(uint64_t key, int lane, int kmin) {
  for (int k = kmin; k <= 32; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t o = shfl_xor64(key, j);
      const bool desc = (lane & k) == 0, lower = (lane & j) == 0;
      key = (lower == desc) ? (key > o ? key : o) : (key < o ? key : o);
    }
  return key;
}
// The largest 32 of two descending runs a, b (lane i holds element i of each), descending.
__device__ __forceinline__ uint64_t warp_merge_top(uint64_t a, uint64_t b, int lane) {
  const uint64_t br = shfl64(b, 31 - lane);
  return warp_bitonic(a > br ? a : br, lane, 32);  // max(a_i, b_31-i) is bitonic
}
// Adds the 32 keys of `col` (one per lane, any order) to the descending top-32 run `best`; a column
// with no key above the run's last one is skipped.
__device__ __forceinline__ uint64_t warp_add_column(uint64_t best, uint64_t col, int lane) {
  const uint64_t thr = shfl64(best, 31);
  if (!__any_sync(0xffffffffu, col > thr)) return best;
  return warp_merge_top(best, warp_bitonic(col, lane, 2), lane);
}
// Adds a descending run (lane i holds element i) to `best`; skipped when its largest key is not above
// best's last.
__device__ __forceinline__ uint64_t warp_add_run(uint64_t best, uint64_t run, int lane) {
  if (!(shfl64(run, 0) > shfl64(best, 31))) return best;
  return warp_merge_top(best, run, lane);
}

constexpr int kPerLane = kChunk / 8 / 32;  // keys per lane of a chunk warp (16)

// First i with u * sum(w) < w_0 + .. + w_i (the last one if rounding leaves none).
__device__ int draw(const float* w, int n, float u) {
  float W = 0.0f;
  for (int i = 0; i < n; ++i) W += w[i];
  const float t = u * W;
  float cum = 0.0f;
  for (int i = 0; i < n; ++i) {
    cum += w[i];
    if (t < cum) return i;
  }
  return n - 1;
}

struct SampleArgs {
  const float* logits;
  int M, V, n_chunks, top_k;
  float temperature, top_p;
  const int32_t* pending;
  const int32_t* draft_tokens;
  const float* draft_probs;
  const float* uniforms;
  int32_t* n_commit;
  int32_t* committed;
  uint64_t* cand;  // [M][n_chunks][32] chunk runs
  int32_t* tok;    // [M][32] row candidates (-1 past the kept ones)
  float* prob;     // [M][32]
  int32_t* count;  // [M]
  unsigned* cnt;   // [M] chunks done per row, then [M / 8] rows done per lane
};

// Stage 1: top 32 of one chunk of one row.  Each warp holds 512 keys, 16 per lane.  The smallest of
// the 32 lane maxima is a lower bound of the warp's 32nd largest key (the 32 maxima are all at least
// it), so only keys at or above it are folded into the warp's run, 32 at a time through shared memory.
__device__ void chunk_topk(const SampleArgs& a, int c, int m, uint64_t (*wtop)[kCand], uint64_t (*buf)[kChunk / 8]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* row = a.logits + (size_t)m * a.V;
  const int base = c * kChunk + warp * (kChunk / 8);
  uint64_t key[kPerLane];
  uint64_t mx = 0;  // 0: below every real key
#pragma unroll
  for (int col = 0; col < kPerLane; ++col) {
    const int idx = base + col * 32 + lane;
    key[col] = idx < a.V ? cand_key(row[idx], idx) : 0ull;
    mx = key[col] > mx ? key[col] : mx;
  }
  uint64_t thr = mx;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const uint64_t t = shfl_xor64(thr, o);
    thr = t < thr ? t : thr;
  }
  int n = 0;  // candidates (keys >= thr) packed into the warp's buffer in a fixed order
#pragma unroll
  for (int col = 0; col < kPerLane; ++col) {
    const bool take = key[col] >= thr && key[col] != 0ull;
    const unsigned bal = __ballot_sync(0xffffffffu, take);
    if (take) buf[warp][n + __popc(bal & ((1u << lane) - 1u))] = key[col];
    n += __popc(bal);
  }
  __syncwarp();
  uint64_t best = 0;
  for (int i = 0; i < n; i += 32) best = warp_add_column(best, i + lane < n ? buf[warp][i + lane] : 0ull, lane);
  wtop[warp][lane] = best;
  __syncthreads();
  if (warp == 0) {
    for (int w = 1; w < 8; ++w) best = warp_add_run(best, wtop[w][lane], lane);
    a.cand[((size_t)m * a.n_chunks + c) * kCand + lane] = best;
  }
}

// Stage 2 (the CTA that finished a row's last chunk): the row's top_k from its chunk runs, then the
// distribution -- the arithmetic follows the definition in order, one thread, fp32.
__device__ void row_dist(const SampleArgs& a, int m, uint64_t (*wtop)[kCand]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t best = 0;
  for (int c0 = warp; c0 < a.n_chunks; c0 += 8 * 4) {  // four runs in flight per warp
    uint64_t r[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = c0 + 8 * q;
      r[q] = c < a.n_chunks ? __ldcg(a.cand + ((size_t)m * a.n_chunks + c) * kCand + lane) : 0ull;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) best = warp_add_run(best, r[q], lane);
  }
  __syncthreads();  // wtop is free again
  wtop[warp][lane] = best;
  __syncthreads();
  if (warp == 0) {
    for (int w = 1; w < 8; ++w) best = warp_add_run(best, wtop[w][lane], lane);
    wtop[0][lane] = best;
    __syncwarp();
    if (lane == 0) {
      const float* row = a.logits + (size_t)m * a.V;
      float l[kCand], e[kCand];
      int id[kCand];
      for (int i = 0; i < a.top_k; ++i) {
        id[i] = key_index(wtop[0][i]);
        const float v = row[id[i]];
        l[i] = isnan(v) ? -INFINITY : v;
      }
      float sum = 0.0f;
      for (int i = 0; i < a.top_k; ++i) {
        e[i] = expf((l[i] - l[0]) / a.temperature);
        sum += e[i];
      }
      int keep = a.top_k;
      float cum = 0.0f;
      for (int i = 0; i < a.top_k; ++i) {
        cum += e[i] / sum;
        if (cum >= a.top_p) {
          keep = i + 1;
          break;
        }
      }
      float ksum = 0.0f;
      for (int i = 0; i < keep; ++i) ksum += e[i];
      for (int i = 0; i < kCand; ++i) {
        a.tok[m * kCand + i] = i < keep ? id[i] : -1;
        a.prob[m * kCand + i] = i < keep ? e[i] / ksum : 0.0f;
      }
      a.count[m] = keep;
    }
  }
}

// Stage 3 (the CTA that finished a lane's last row): the lane's 8 distributions, its drafts'
// distributions and its uniforms are copied to shared memory, q of every candidate (and of every
// draft) looked up by all threads; thread 0 then runs the acceptance scan.
__device__ void accept_scan(const SampleArgs& a, int l) {
  __shared__ int32_t st[8][kCand];
  __shared__ float sp[8][kCand], sq[8][kCand], sqd[8], su[8][2];
  __shared__ int32_t sn[8], sd[8];
  const int tid = threadIdx.x;
  {
    const int j = tid / kCand, i = tid % kCand, r = 8 * l + j;  // 8 rows x 32 candidates = 256 threads
    const int32_t t = __ldcg(a.tok + r * kCand + i);
    st[j][i] = t;
    sp[j][i] = __ldcg(a.prob + r * kCand + i);
    const int32_t d = j < 7 ? a.pending[8 * l + j + 1] : -1;
    float q = 0.0f, qd = 0.0f;
    if (j < 7) {
      if (!a.draft_probs) {
        q = t == d ? 1.0f : 0.0f;
        qd = 1.0f;
      } else {
        bool ft = false, fd = false;  // the first listed entry of a token counts
        for (int c = 0; c < 16; ++c) {
          const int32_t dt = a.draft_tokens[r * 16 + c];
          const float dp = a.draft_probs[r * 16 + c];
          if (dt == t && !ft) {
            q = dp;
            ft = true;
          }
          if (dt == d && !fd) {
            qd = dp;
            fd = true;
          }
        }
      }
    }
    sq[j][i] = q;  // q of candidate i at row j
    if (i == 0) {
      sqd[j] = qd;  // q of the draft checked at row j
      sd[j] = d;
      sn[j] = __ldcg(a.count + r);
      su[j][0] = a.uniforms[2 * r];
      su[j][1] = a.uniforms[2 * r + 1];
    }
  }
  __syncthreads();
  if (tid != 0) return;
  int acc = 0, last = -1;
  for (int j = 0; j <= 7; ++j) {
    const int n = sn[j];
    if (j == 7) {
      last = st[j][draw(sp[j], n, su[j][1])];
      break;
    }
    float pd = 0.0f;
    for (int i = 0; i < n; ++i)
      if (st[j][i] == sd[j]) pd = sp[j][i];
    if (su[j][0] * sqd[j] < pd) {
      ++acc;
      continue;
    }
    float w[kCand], W = 0.0f;
    for (int i = 0; i < n; ++i) {
      w[i] = fmaxf(sp[j][i] - sq[j][i], 0.0f);
      W += w[i];
    }
    last = st[j][W > 0.0f ? draw(w, n, su[j][1]) : draw(sp[j], n, su[j][1])];
    break;
  }
  a.n_commit[l] = acc + 1;
  for (int j = 0; j < 8; ++j) a.committed[8 * l + j] = j < acc ? sd[j] : (j == acc ? last : -1);
}

// One launch, grid (chunks, M): every CTA runs stage 1; the last CTA to finish a row (a counter per
// row) runs stage 2 for it, and the last row of a lane (a counter per lane) stage 3.  The counters
// count with release / acquire fences, as the grid's other fixed-order hand-offs do, and are reset by
// their last user.
__global__ void __launch_bounds__(256) sa_kernel(const SampleArgs a) {
  __shared__ uint64_t wtop[8][kCand];
  __shared__ uint64_t buf[8][kChunk / 8];
  __shared__ int last;
  const int c = blockIdx.x, m = blockIdx.y;
  chunk_topk(a, c, m, wtop, buf);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last = atomicAdd(a.cnt + m, 1u) + 1 == (unsigned)a.n_chunks;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  row_dist(a, m, wtop);
  __syncthreads();
  const int l = m / 8;
  if (threadIdx.x == 0) {
    a.cnt[m] = 0u;
    __threadfence();
    last = atomicAdd(a.cnt + a.M + l, 1u) + 1 == 8u;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  accept_scan(a, l);
  if (threadIdx.x == 0) a.cnt[a.M + l] = 0u;
}

}  // namespace

SampleWs sample_ws_layout(int M, int V) {
  SampleWs L;
  L.n_chunks = (V + kChunk - 1) / kChunk;
  L.cand = 0;
  L.tok = align_up(L.cand + sizeof(uint64_t) * (size_t)M * L.n_chunks * kCand, 256);
  L.prob = align_up(L.tok + sizeof(int32_t) * (size_t)M * kCand, 256);
  L.count = align_up(L.prob + sizeof(float) * (size_t)M * kCand, 256);
  L.cnt = align_up(L.count + sizeof(int32_t) * (size_t)M, 256);
  L.total = align_up(L.cnt + sizeof(unsigned) * (size_t)(M + M / 8), 256);
  return L;
}

cudaError_t launch_sample_accept(const float* logits, int M, int V, float temperature, int top_k, float top_p,
                                 const int32_t* pending, const int32_t* draft_tokens, const float* draft_probs,
                                 const float* uniforms, int32_t* n_commit, int32_t* committed, void* ws,
                                 cudaStream_t s) {
  const SampleWs L = sample_ws_layout(M, V);
  uint8_t* b = static_cast<uint8_t*>(ws);
  SampleArgs a;
  a.logits = logits;
  a.M = M;
  a.V = V;
  a.n_chunks = L.n_chunks;
  a.top_k = top_k;
  a.temperature = temperature;
  a.top_p = top_p;
  a.pending = pending;
  a.draft_tokens = draft_tokens;
  a.draft_probs = draft_probs;
  a.uniforms = uniforms;
  a.n_commit = n_commit;
  a.committed = committed;
  a.cand = reinterpret_cast<uint64_t*>(b + L.cand);
  a.tok = reinterpret_cast<int32_t*>(b + L.tok);
  a.prob = reinterpret_cast<float*>(b + L.prob);
  a.count = reinterpret_cast<int32_t*>(b + L.count);
  a.cnt = reinterpret_cast<unsigned*>(b + L.cnt);
  sa_kernel<<<dim3((unsigned)L.n_chunks, (unsigned)M), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace vp
