// Host side of libverify: argument validation, packers, workspace carving and the verify-pass
// driver.  Every entry point is declared (with its source passage) in include/verify.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "verify.h"
#include "gemm.cuh"
#include "internal.h"
#include "launch_decl.h"

using namespace vp;

namespace {

thread_local int g_last_cuda_error = 0;

vp_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return VP_ERR_CUDA;
}

constexpr int kMaxGrid = 256;  // workspace is sized for grids up to this many CTAs
constexpr int kArgmaxChunk = 8192;

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// SM count of the current device (cached per ordinal); also checks for an sm_103 device.
vp_status device_sms(int* sms) {
  static int cache[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev >= 0 && dev < 64 && cache[dev] > 0) {
    *sms = cache[dev];
    return VP_OK;
  }
  int major = 0, minor = 0, n = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return cuda_fail(e);
  if (major != 10 || minor != 3) return VP_ERR_UNSUPPORTED;
  if (n > kMaxGrid) n = kMaxGrid;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  *sms = n;
  return VP_OK;
}

bool linear_shape_ok(int M, int N, int K) {
  return M >= 1 && M <= kMaxM && N >= 16 && N % kRowsPerBlock == 0 && K >= kQuadK && K % kQuadK == 0 &&
         (long long)N * K < (1LL << 40);
}

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

struct GemmWs {
  WsLayout L;
  int* status;
  unsigned* task_cnt;
  unsigned* group_cnt;
  float* group_aux;
  float* partials;
};

GemmWs carve_gemm_ws(void* ws, int n_groups, int mt) {
  GemmWs w;
  w.L = gemm_ws_layout(n_groups, kMaxGrid, mt);
  uint8_t* b = (uint8_t*)ws;
  w.status = (int*)(b + w.L.status);
  w.task_cnt = (unsigned*)(b + w.L.task_cnt);
  w.group_cnt = (unsigned*)(b + w.L.group_cnt);
  w.group_aux = (float*)(b + w.L.group_aux);
  w.partials = (float*)(b + w.L.partials);
  return w;
}

void fill_ws(GemmParams& p, const GemmWs& w) {
  p.status = w.status;
  p.task_cnt = w.task_cnt;
  p.group_cnt = w.group_cnt;
  p.group_aux = w.group_aux;
  p.partials = w.partials;
}

// Plain single-matrix GEMM parameters.
GemmParams single(const void* w, int N, int K, int M, float scale) {
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.w[0] = (const uint8_t*)w;
  p.seg_rows[0] = N;
  p.wscale[0] = scale;
  p.wscale[1] = 1.0f;
  p.K = K;
  p.M = M;
  p.nq = K / kQuadK;
  p.n_groups = ceil_div(N, kSlabRows);
  p.seg0_groups = p.n_groups;
  p.units = (long long)p.n_groups * p.nq;
  return p;
}

vp_status launch(int fmt, const GemmParams& p, int sms, cudaStream_t s, bool pdl) {
  const int mt = (p.M + 7) / 8;
  const int grid = (int)((p.units < (long long)sms) ? p.units : (long long)sms);
  cudaError_t e = fmt == kFmtNvfp4 ? launch_gemm_nvfp4(p, mt, grid, s, pdl) : launch_gemm_fp8(p, mt, grid, s, pdl);
  if (e != cudaSuccess) return cuda_fail(e);
  return VP_OK;
}

// ------------------------------------------------------------------ packers
// Packed NVFP4 block (16 rows x 64 K, 576 bytes) of row-block rb, quad q:
//   byte 16*L + 4*j + i (L = lane 0..31, g = L/4, t = L%4, j = k16 step, i = MMA A register):
//     the canonical code byte holding weights (row rb*16 + g + 8*(i&1), k = 64q + 16j + 2t + 8*(i>>1))
//     and k + 1 (low nibble = k).
//   byte 512 + 8*g + 2*j + h: block scale of row rb*16 + g + 8h for k16 step j (scale column 4q + j).
// Blocks are ordered slab by slab (256 rows); within a slab, quad-major then row-block.
__global__ void pack_nvfp4_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, int N, int K,
                                  uint8_t* __restrict__ out, long long total) {
  const int nq = K / kQuadK;
  const int nrb_total = N / kRowsPerBlock;
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total; o += (long long)gridDim.x * blockDim.x) {
    const long long b = o / kNvfp4BlockBytes;
    const int bb = (int)(o % kNvfp4BlockBytes);
    const long long slab = b / ((long long)kBlocksPerSlab * nq);
    const long long r = b % ((long long)kBlocksPerSlab * nq);
    const int nrb_s = min(kBlocksPerSlab, nrb_total - (int)slab * kBlocksPerSlab);
    const int q = (int)(r / nrb_s), rb = (int)slab * kBlocksPerSlab + (int)(r % nrb_s);
    uint8_t v;
    if (bb < 512) {
      const int L = bb >> 4, j = (bb >> 2) & 3, i = bb & 3;
      const int g = L >> 2, t = L & 3;
      const long long row = (long long)rb * kRowsPerBlock + g + 8 * (i & 1);
      const int k = q * kQuadK + 16 * j + 2 * t + 8 * (i >> 1);
      v = codes[row * (K / 2) + k / 2];
    } else {
      const int x = bb - 512, g = x >> 3, j = (x >> 1) & 3, h = x & 1;
      const long long row = (long long)rb * kRowsPerBlock + g + 8 * h;
      v = scales[row * (K / 16) + 4 * q + j];
    }
    out[o] = v;
  }
}

// Packed FP8 block (16 rows x 64 K, 1024 bytes): byte 32*L + 8*j + 2*i + e holds
// w[rb*16 + g + 8*(i&1)][64q + 16j + 2t + 8*(i>>1) + e] (g = L/4, t = L%4).
__global__ void pack_fp8_kernel(const uint8_t* __restrict__ w, int N, int K, uint8_t* __restrict__ out, long long total) {
  const int nq = K / kQuadK;
  const int nrb_total = N / kRowsPerBlock;
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total; o += (long long)gridDim.x * blockDim.x) {
    const long long b = o / kFp8BlockBytes;
    const int bb = (int)(o % kFp8BlockBytes);
    const long long slab = b / ((long long)kBlocksPerSlab * nq);
    const long long r = b % ((long long)kBlocksPerSlab * nq);
    const int nrb_s = min(kBlocksPerSlab, nrb_total - (int)slab * kBlocksPerSlab);
    const int q = (int)(r / nrb_s), rb = (int)slab * kBlocksPerSlab + (int)(r % nrb_s);
    const int L = bb >> 5, j = (bb >> 3) & 3, i = (bb >> 1) & 3, e = bb & 1;
    const int g = L >> 2, t = L & 3;
    const long long row = (long long)rb * kRowsPerBlock + g + 8 * (i & 1);
    const int k = q * kQuadK + 16 * j + 2 * t + 8 * (i >> 1) + e;
    out[o] = w[row * K + k];
  }
}

int pack_grid(long long total) {
  long long b = (total + 255) / 256;
  if (b > 152LL * 32) b = 152LL * 32;
  return (int)(b < 1 ? 1 : b);
}

// ------------------------------------------------------------------ argmax + accept over given logits
__global__ void __launch_bounds__(256) argmax_accept_kernel(const float* __restrict__ logits, int M, int V, int chunk,
                                                            int n_chunks, const int32_t* pending, int32_t* argmax,
                                                            int32_t* n_commit, int32_t* committed, float* aux,
                                                            unsigned* task_cnt) {
  __shared__ float red_v[256];
  __shared__ int red_i[256];
  __shared__ int tok[kMaxM];
  __shared__ int last;
  const int c = blockIdx.x, m = blockIdx.y;
  const int lo = c * chunk, hi = min(V, lo + chunk);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  const float* row = logits + (size_t)m * V;
  for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
    float v = row[i];
    if (isnan(v)) v = -INFINITY;
    if (am_better(v, i, bv, bi)) {
      bv = v;
      bi = i;
    }
  }
  am_shfl_reduce(bv, bi, 1, 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red_v[warp] = bv;
    red_i[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float v0 = -INFINITY;
    int i0 = 0x7fffffff;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
      if (am_better(red_v[w], red_i[w], v0, i0)) {
        v0 = red_v[w];
        i0 = red_i[w];
      }
    aux[((size_t)c * kMaxM + m) * 2] = v0;
    aux[((size_t)c * kMaxM + m) * 2 + 1] = __int_as_float(i0);
    __threadfence();
    const unsigned old = atomicAdd(task_cnt, 1u);
    last = (old == (unsigned)(n_chunks * M) - 1u);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  argmax_accept_finish(aux, n_chunks, M, pending, argmax, n_commit, committed, red_v, red_i, tok, threadIdx.x, 256, 1);
  if (threadIdx.x == 0) *task_cnt = 0u;
}

// ------------------------------------------------------------------ pass prologue
// h = x0 and inv_rms[m] = 1 / sqrt(mean(h[m]^2) + eps), one CTA per row.
__global__ void __launch_bounds__(256) pass_prep_kernel(const uint16_t* __restrict__ x0, uint16_t* __restrict__ h, int H,
                                                        float eps, float* __restrict__ inv_rms) {
  pdl_trigger();
  __shared__ float red[8];
  const int m = blockIdx.x;
  float s = 0.0f;
  for (int k = threadIdx.x; k < H; k += blockDim.x) {
    const uint16_t b = x0[(size_t)m * H + k];
    h[(size_t)m * H + k] = b;
    const float v = __uint_as_float((uint32_t)b << 16);
    s += v * v;
  }
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.0f;
    for (int w = 0; w < 8; ++w) t += red[w];
    inv_rms[m] = 1.0f / sqrtf(t / (float)H + eps);
  }
}

size_t argmax_ws_bytes(int V) {
  const int n_chunks = ceil_div(V, kArgmaxChunk);
  return align_up(256 + sizeof(float) * 2 * kMaxM * (size_t)n_chunks, 256);
}

}  // namespace

// ======================================================================== C ABI

extern "C" {

const char* vp_status_string(int s) {
  switch (s) {
    case VP_OK: return "VP_OK";
    case VP_ERR_INVALID_ARG: return "VP_ERR_INVALID_ARG";
    case VP_ERR_SHAPE: return "VP_ERR_SHAPE";
    case VP_ERR_ALIGNMENT: return "VP_ERR_ALIGNMENT";
    case VP_ERR_WORKSPACE: return "VP_ERR_WORKSPACE";
    case VP_ERR_CUDA: return "VP_ERR_CUDA";
    case VP_ERR_TIMEOUT: return "VP_ERR_TIMEOUT";
    case VP_ERR_UNSUPPORTED: return "VP_ERR_UNSUPPORTED";
    default: return "VP_ERR_UNKNOWN";
  }
}

int vp_get_last_cuda_error(void) { return g_last_cuda_error; }

vp_status vp_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws) return VP_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return VP_ERR_ALIGNMENT;
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream);
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

vp_status vp_read_status(const void* ws, int* status, void* stream) {
  if (!ws || !status) return VP_ERR_INVALID_ARG;
  cudaError_t e = cudaMemcpyAsync(status, ws, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

size_t vp_packed_bytes_nvfp4(int N, int K) {
  if (N < 16 || N % 16 || K < 64 || K % 64) return 0;
  return (size_t)N * (size_t)K / 16 * 9;
}

size_t vp_packed_bytes_fp8(int N, int K) {
  if (N < 16 || N % 16 || K < 64 || K % 64) return 0;
  return (size_t)N * (size_t)K;
}

vp_status vp_pack_nvfp4(const void* codes, const void* scales, int N, int K, void* packed, size_t packed_bytes,
                        void* stream) {
  if (!codes || !scales || !packed) return VP_ERR_INVALID_ARG;
  const size_t need = vp_packed_bytes_nvfp4(N, K);
  if (need == 0) return VP_ERR_SHAPE;
  if (packed_bytes < need) return VP_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(scales, 16) || !aligned(packed, 16)) return VP_ERR_ALIGNMENT;
  int sms = 0;
  vp_status st = device_sms(&sms);
  if (st != VP_OK) return st;
  pack_nvfp4_kernel<<<pack_grid((long long)need), 256, 0, (cudaStream_t)stream>>>(
      (const uint8_t*)codes, (const uint8_t*)scales, N, K, (uint8_t*)packed, (long long)need);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

vp_status vp_pack_fp8(const void* w, int N, int K, void* packed, size_t packed_bytes, void* stream) {
  if (!w || !packed) return VP_ERR_INVALID_ARG;
  const size_t need = vp_packed_bytes_fp8(N, K);
  if (need == 0) return VP_ERR_SHAPE;
  if (packed_bytes < need) return VP_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(packed, 16)) return VP_ERR_ALIGNMENT;
  int sms = 0;
  vp_status st = device_sms(&sms);
  if (st != VP_OK) return st;
  pack_fp8_kernel<<<pack_grid((long long)need), 256, 0, (cudaStream_t)stream>>>((const uint8_t*)w, N, K,
                                                                               (uint8_t*)packed, (long long)need);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

size_t vp_workspace_bytes(int op, int M, int N, int K) {
  if (op == VP_OP_ARGMAX) {
    if (M < 8 || M > kMaxM || M % 8 || N < 1) return 0;
    return argmax_ws_bytes(N);
  }
  if (op != VP_OP_NVFP4 && op != VP_OP_FP8 && op != VP_OP_HEAD) return 0;
  if (!linear_shape_ok(M, N, K)) return 0;
  if (op == VP_OP_HEAD && M % 8) return 0;
  return gemm_ws_layout(ceil_div(N, kSlabRows), kMaxGrid, (M + 7) / 8).total;
}

static vp_status linear_common(int fmt, const void* w, float scale, const void* x, float* y, int M, int N, int K,
                               void* ws, size_t ws_bytes, void* stream) {
  if (!w || !x || !y || !ws) return VP_ERR_INVALID_ARG;
  if (!linear_shape_ok(M, N, K)) return VP_ERR_SHAPE;
  if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 4) || !aligned(ws, 256)) return VP_ERR_ALIGNMENT;
  const size_t need = vp_workspace_bytes(fmt == kFmtNvfp4 ? VP_OP_NVFP4 : VP_OP_FP8, M, N, K);
  if (ws_bytes < need) return VP_ERR_WORKSPACE;
  int sms = 0;
  vp_status st = device_sms(&sms);
  if (st != VP_OK) return st;
  GemmParams p = single(w, N, K, M, scale);
  p.x = (const uint16_t*)x;
  p.x_ld = K;
  p.epi = kEpiF32;
  p.y = y;
  p.y_ld = N;
  fill_ws(p, carve_gemm_ws(ws, p.n_groups, (M + 7) / 8));
  return launch(fmt, p, sms, (cudaStream_t)stream, false);
}

vp_status vp_linear_nvfp4(const void* w_packed, float tensor_scale, const void* x, float* y, int M, int N, int K,
                          void* ws, size_t ws_bytes, void* stream) {
  return linear_common(kFmtNvfp4, w_packed, tensor_scale, x, y, M, N, K, ws, ws_bytes, stream);
}

vp_status vp_linear_fp8(const void* w_packed, float scale, const void* x, float* y, int M, int N, int K, void* ws,
                        size_t ws_bytes, void* stream) {
  return linear_common(kFmtFp8, w_packed, scale, x, y, M, N, K, ws, ws_bytes, stream);
}

vp_status vp_head_argmax_accept(const void* w_packed, float tensor_scale, const void* x, int M, int V, int K,
                                const int32_t* pending, int32_t* argmax, int32_t* n_commit, int32_t* committed,
                                float* logits, void* ws, size_t ws_bytes, void* stream) {
  if (!w_packed || !x || !pending || !argmax || !n_commit || !committed || !ws) return VP_ERR_INVALID_ARG;
  if (!linear_shape_ok(M, V, K) || M % 8) return VP_ERR_SHAPE;
  if (!aligned(w_packed, 16) || !aligned(x, 16) || !aligned(ws, 256) || !aligned(pending, 4) || !aligned(argmax, 4) ||
      !aligned(n_commit, 4) || !aligned(committed, 4) || (logits && !aligned(logits, 4)))
    return VP_ERR_ALIGNMENT;
  if (ws_bytes < vp_workspace_bytes(VP_OP_HEAD, M, V, K)) return VP_ERR_WORKSPACE;
  int sms = 0;
  vp_status st = device_sms(&sms);
  if (st != VP_OK) return st;
  GemmParams p = single(w_packed, V, K, M, tensor_scale);
  p.x = (const uint16_t*)x;
  p.x_ld = K;
  p.epi = kEpiHead;
  p.pending = pending;
  p.argmax = argmax;
  p.n_commit = n_commit;
  p.committed = committed;
  p.logits = logits;
  p.logits_ld = V;
  fill_ws(p, carve_gemm_ws(ws, p.n_groups, (M + 7) / 8));
  return launch(kFmtNvfp4, p, sms, (cudaStream_t)stream, false);
}

vp_status vp_argmax_accept(const float* logits, int M, int V, const int32_t* pending, int32_t* argmax,
                           int32_t* n_commit, int32_t* committed, void* ws, size_t ws_bytes, void* stream) {
  if (!logits || !pending || !argmax || !n_commit || !committed || !ws) return VP_ERR_INVALID_ARG;
  if (M < 8 || M > kMaxM || M % 8 || V < 1) return VP_ERR_SHAPE;
  if (!aligned(logits, 4) || !aligned(ws, 256) || !aligned(pending, 4) || !aligned(argmax, 4) ||
      !aligned(n_commit, 4) || !aligned(committed, 4))
    return VP_ERR_ALIGNMENT;
  if (ws_bytes < argmax_ws_bytes(V)) return VP_ERR_WORKSPACE;
  int sms = 0;
  vp_status st = device_sms(&sms);
  if (st != VP_OK) return st;
  const int n_chunks = ceil_div(V, kArgmaxChunk);
  uint8_t* b = (uint8_t*)ws;
  argmax_accept_kernel<<<dim3(n_chunks, M), 256, 0, (cudaStream_t)stream>>>(
      logits, M, V, kArgmaxChunk, n_chunks, pending, argmax, n_commit, committed, (float*)(b + 256),
      (unsigned*)(b + 64));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

}  // extern "C"

// ======================================================================== the verify pass

struct vp_model {
  int hidden, inter;
  float eps;
  std::vector<vp_layer_desc> layers;
  vp_head_desc head;
  int max_groups;
  int zmax;
};

namespace {

struct PassWs {
  GemmWs g;
  float* inv_rms;
  uint16_t* h;
  uint16_t* z;
  uint16_t* a;
  size_t counters_bytes;
  size_t total;
};

PassWs carve_pass_ws(const vp_model* md, int M, void* ws) {
  PassWs w;
  const int mt = (M + 7) / 8;
  w.g = carve_gemm_ws(ws, md->max_groups, mt);
  size_t off = w.g.L.total;
  const size_t inv_off = off;
  off = align_up(off + sizeof(float) * kMaxM, 256);
  const size_t h_off = off;
  off = align_up(off + sizeof(uint16_t) * (size_t)M * md->hidden, 256);
  const size_t z_off = off;
  off = align_up(off + sizeof(uint16_t) * (size_t)M * md->zmax, 256);
  const size_t a_off = off;
  off = align_up(off + sizeof(uint16_t) * (size_t)M * md->inter, 256);
  uint8_t* b = (uint8_t*)ws;
  w.inv_rms = (float*)(b + inv_off);
  w.h = (uint16_t*)(b + h_off);
  w.z = (uint16_t*)(b + z_off);
  w.a = (uint16_t*)(b + a_off);
  w.counters_bytes = w.g.L.group_aux;
  w.total = off;
  return w;
}

bool fp8_ok(const void* w, int N, int K) { return w && aligned(w, 16) && vp_packed_bytes_fp8(N, K) > 0; }
bool nvfp4_ok(const void* w, int N, int K) { return w && aligned(w, 16) && vp_packed_bytes_nvfp4(N, K) > 0; }

}  // namespace

extern "C" {

vp_status vp_model_create(int hidden, int inter, float rms_eps, const vp_layer_desc* layers, int n_layers,
                          const vp_head_desc* head, vp_model** out) {
  if (!layers || !head || !out || n_layers < 1 || !(rms_eps >= 0.0f)) return VP_ERR_INVALID_ARG;
  if (hidden < 64 || hidden % 64 || inter < 64 || inter % 64) return VP_ERR_SHAPE;
  int max_groups = ceil_div(head->vocab, kSlabRows);
  int zmax = 64;
  for (int l = 0; l < n_layers; ++l) {
    const vp_layer_desc& d = layers[l];
    if (d.kind != VP_LAYER_GDN && d.kind != VP_LAYER_ATTN) return VP_ERR_INVALID_ARG;
    if (!fp8_ok(d.w_in, d.n_in, hidden) || !fp8_ok(d.w_out, hidden, d.k_out)) return VP_ERR_SHAPE;
    if (d.k_out > d.n_in) return VP_ERR_SHAPE;
    if (d.kind == VP_LAYER_ATTN && !fp8_ok(d.w_kv, d.n_kv, hidden)) return VP_ERR_SHAPE;
    if (d.kind == VP_LAYER_GDN && (d.w_kv || d.n_kv)) return VP_ERR_INVALID_ARG;
    if (!nvfp4_ok(d.w_gate, inter, hidden) || !nvfp4_ok(d.w_up, inter, hidden) || !nvfp4_ok(d.w_down, hidden, inter))
      return VP_ERR_SHAPE;
    int gin = ceil_div(d.n_in, kSlabRows) + (d.kind == VP_LAYER_ATTN ? ceil_div(d.n_kv, kSlabRows) : 0);
    if (gin > max_groups) max_groups = gin;
    if (d.k_out > zmax) zmax = d.k_out;
  }
  if (!nvfp4_ok(head->w, head->vocab, hidden)) return VP_ERR_SHAPE;
  max_groups = std::max(max_groups, ceil_div(inter, 128));
  max_groups = std::max(max_groups, ceil_div(hidden, kSlabRows));
  vp_model* m = new (std::nothrow) vp_model;
  if (!m) return VP_ERR_INVALID_ARG;
  m->hidden = hidden;
  m->inter = inter;
  m->eps = rms_eps;
  m->layers.assign(layers, layers + n_layers);
  m->head = *head;
  m->max_groups = max_groups;
  m->zmax = zmax;
  *out = m;
  return VP_OK;
}

void vp_model_destroy(vp_model* model) { delete model; }

size_t vp_pass_workspace_bytes(const vp_model* model, int M) {
  if (!model || M < 8 || M > kMaxM || M % 8) return 0;
  return carve_pass_ws(model, M, nullptr).total;
}

int vp_pass_launch_count(const vp_model* model) { return model ? 2 + 4 * (int)model->layers.size() : 0; }

}  // extern "C"

namespace {

// Enqueues blocks [b0, b1) of the pass (block 2l = mixer of layer l, 2l + 1 = MLP of layer l) on
// the residual stream h (bf16 [M][hidden], updated in place).  inv_rms must hold 1/rms of h's rows
// on entry and holds 1/rms of the result on exit.  Optional trace: h after each block.
vp_status enqueue_blocks(const vp_model* md, const PassWs& w, uint16_t* h, int M, int b0, int b1, void* trace,
                         int sms, cudaStream_t s) {
  const int H = md->hidden, I = md->inter;
  const size_t hbytes = sizeof(uint16_t) * (size_t)M * H;
  vp_status st;
  cudaError_t e;
  for (int b = b0; b < b1; ++b) {
    const vp_layer_desc& d = md->layers[b / 2];
    if ((b & 1) == 0) {
      // mixer in-projection (GDN in, or attention q + kv): z = bf16(first k_out columns of RMSNorm(h) W^T)
      GemmParams p = single(d.w_in, d.n_in, H, M, d.s_in);
      if (d.kind == VP_LAYER_ATTN) {
        p.w[1] = (const uint8_t*)d.w_kv;
        p.seg_rows[1] = d.n_kv;
        p.wscale[1] = d.s_kv;
        p.n_groups = p.seg0_groups + ceil_div(d.n_kv, kSlabRows);
        p.units = (long long)p.n_groups * p.nq;
      }
      p.x = h;
      p.x_ld = H;
      p.x_rowscale = w.inv_rms;
      p.epi = kEpiBf16Prefix;
      p.out = w.z;
      p.out_ld = d.k_out;
      p.out_cols = d.k_out;
      fill_ws(p, w.g);
      if ((st = launch(kFmtFp8, p, sms, s, true)) != VP_OK) return st;
      // mixer out-projection + residual: h = bf16(h + z W_out^T); 1/rms(h) for the next block
      p = single(d.w_out, H, d.k_out, M, d.s_out);
      p.x = w.z;
      p.x_ld = d.k_out;
      p.epi = kEpiResid;
      p.resid = h;
      p.resid_ld = H;
      p.resid_cols = H;
      p.rms_out = w.inv_rms;
      p.rms_eps = md->eps;
      fill_ws(p, w.g);
      if ((st = launch(kFmtFp8, p, sms, s, true)) != VP_OK) return st;
    } else {
      // MLP gate + up (interleaved row-blocks) -> a = bf16(silu(gate) * up)
      GemmParams p = single(d.w_gate, I, H, M, d.ts_gate);
      p.w[1] = (const uint8_t*)d.w_up;
      p.seg_rows[1] = I;
      p.wscale[1] = d.ts_up;
      p.interleave = 1;
      p.n_groups = ceil_div(I, 128);
      p.seg0_groups = p.n_groups;
      p.units = (long long)p.n_groups * p.nq;
      p.x = h;
      p.x_ld = H;
      p.x_rowscale = w.inv_rms;
      p.epi = kEpiSiluMul;
      p.out = w.a;
      p.out_ld = I;
      fill_ws(p, w.g);
      if ((st = launch(kFmtNvfp4, p, sms, s, true)) != VP_OK) return st;
      // MLP down + residual
      p = single(d.w_down, H, I, M, d.ts_down);
      p.x = w.a;
      p.x_ld = I;
      p.epi = kEpiResid;
      p.resid = h;
      p.resid_ld = H;
      p.resid_cols = H;
      p.rms_out = w.inv_rms;
      p.rms_eps = md->eps;
      fill_ws(p, w.g);
      if ((st = launch(kFmtNvfp4, p, sms, s, true)) != VP_OK) return st;
    }
    if (trace &&
        (e = cudaMemcpyAsync((uint8_t*)trace + (size_t)(b - b0) * hbytes, h, hbytes, cudaMemcpyDeviceToDevice, s)) !=
            cudaSuccess)
      return cuda_fail(e);
  }
  return VP_OK;
}

vp_status pass_args_ok(const vp_model* md, int M, void* ws, size_t ws_bytes) {
  if (!md || !ws) return VP_ERR_INVALID_ARG;
  if (M < 8 || M > kMaxM || M % 8) return VP_ERR_SHAPE;
  if (!aligned(ws, 256)) return VP_ERR_ALIGNMENT;
  if (ws_bytes < vp_pass_workspace_bytes(md, M)) return VP_ERR_WORKSPACE;
  return VP_OK;
}

}  // namespace

extern "C" {

vp_status vp_verify_pass(const vp_model* md, const void* x0, int M, const int32_t* pending, int32_t* argmax,
                         int32_t* n_commit, int32_t* committed, void* trace, float* logits, void* ws, size_t ws_bytes,
                         void* stream) {
  vp_status st = pass_args_ok(md, M, ws, ws_bytes);
  if (st != VP_OK) return st;
  if (!x0 || !pending || !argmax || !n_commit || !committed) return VP_ERR_INVALID_ARG;
  if (!aligned(x0, 16) || (trace && !aligned(trace, 16)) || (logits && !aligned(logits, 4)) || !aligned(pending, 4) ||
      !aligned(argmax, 4) || !aligned(n_commit, 4) || !aligned(committed, 4))
    return VP_ERR_ALIGNMENT;
  int sms = 0;
  if ((st = device_sms(&sms)) != VP_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const int H = md->hidden;
  const PassWs w = carve_pass_ws(md, M, ws);
  cudaError_t e;
  pass_prep_kernel<<<M, 256, 0, s>>>((const uint16_t*)x0, w.h, H, md->eps, w.inv_rms);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
  if ((st = enqueue_blocks(md, w, w.h, M, 0, 2 * (int)md->layers.size(), trace, sms, s)) != VP_OK) return st;
  // head + argmax + acceptance on RMSNorm(h)
  GemmParams p = single(md->head.w, md->head.vocab, H, M, md->head.ts);
  p.x = w.h;
  p.x_ld = H;
  p.x_rowscale = w.inv_rms;
  p.epi = kEpiHead;
  p.pending = pending;
  p.argmax = argmax;
  p.n_commit = n_commit;
  p.committed = committed;
  p.logits = logits;
  p.logits_ld = md->head.vocab;
  fill_ws(p, w.g);
  return launch(kFmtNvfp4, p, sms, s, true);
}

vp_status vp_verify_blocks(const vp_model* md, void* h, int M, int block_begin, int block_end, void* trace, void* ws,
                           size_t ws_bytes, void* stream) {
  vp_status st = pass_args_ok(md, M, ws, ws_bytes);
  if (st != VP_OK) return st;
  if (!h) return VP_ERR_INVALID_ARG;
  const int nb = 2 * (int)md->layers.size();
  if (block_begin < 0 || block_end > nb || block_begin > block_end) return VP_ERR_INVALID_ARG;
  if (!aligned(h, 16) || (trace && !aligned(trace, 16))) return VP_ERR_ALIGNMENT;
  int sms = 0;
  if ((st = device_sms(&sms)) != VP_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const PassWs w = carve_pass_ws(md, M, ws);
  cudaError_t e;
  // 1/rms of the incoming rows (the copy onto itself is a no-op)
  pass_prep_kernel<<<M, 256, 0, s>>>((const uint16_t*)h, (uint16_t*)h, md->hidden, md->eps, w.inv_rms);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
  return enqueue_blocks(md, w, (uint16_t*)h, M, block_begin, block_end, trace, sms, s);
}

}  // extern "C"
