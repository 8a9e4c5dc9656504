// Host side of libverify: argument validation, packers, workspace carving, the phase programs of
// the linear / head calls and of the verify pass, and the argmax + accept kernel over given logits.
// Every entry point is declared (with its source passage) in include/verify.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <new>
#include <vector>

#include "exec.cuh"
#include "exec_launch.h"
#include "internal.h"
#include "attention.h"
#include "errors.h"
#include "mixer.h"
#include "sample.h"
#include "verify.h"

using namespace vp;

namespace {


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

constexpr int kMaxK = 65536;

bool weight_shape_ok(int fmt, int N, int K) {
  const int ck = chunk_k(fmt);
  return N >= kRowBlock && N % kRowBlock == 0 && K >= ck && K % ck == 0 && K <= kMaxK &&
         (long long)N * K < (1LL << 40);
}

int nt_of(int M) { return (M + 7) / 8; }

// ------------------------------------------------------------------ phases
struct PhaseSpec {
  int fmt = kFmtNvfp4, layout = kPlain;
  const void* w0 = nullptr;
  const void* w1 = nullptr;
  float s0 = 1.0f, s1 = 1.0f;
  int rows0 = 0, rows1 = 0, K = 0;
  int epi = kEpiF32, x_src = kBufX, x_ld = 0, x_rms = 0, out = kBufY, out_ld = 0, out_cols = 0, trace_slot = -1;
  int ss = 0;
};

Phase make_phase(const PhaseSpec& s, int NT) {
  Phase ph;
  memset(&ph, 0, sizeof(ph));
  ph.w0 = static_cast<const uint8_t*>(s.w0);
  ph.w1 = static_cast<const uint8_t*>(s.w1);
  ph.s0 = s.s0;
  ph.s1 = s.s1;
  ph.K = s.K;
  ph.KC = s.K / chunk_k(s.fmt);
  ph.RB = (s.rows0 + s.rows1) / kRowBlock;
  if (s.layout == kPlain) {
    ph.grp = 2;  // units of two chunks: one 4096 / 4608-byte copy (smaller copies stream slower)
    ph.rb1 = s.rows0 / kRowBlock;
  } else {
    ph.grp = 1;
    ph.RB = s.rows0 / kRowBlock;
    ph.rb1 = ph.RB;
  }
  ph.KG = (ph.KC + ph.grp - 1) / ph.grp;
  const int per = ks_max(NT) / chunk_k(s.fmt) / ph.grp;  // groups per slice at most
  ph.ks = (int8_t)((ph.KG + per - 1) / per);
  ph.fmt = (int8_t)s.fmt;
  ph.layout = (int8_t)s.layout;
  ph.epi = (int8_t)s.epi;
  ph.x_src = (int8_t)s.x_src;
  ph.x_rms = (int8_t)s.x_rms;
  ph.ss = (int8_t)s.ss;
  ph.out = (int8_t)s.out;
  ph.x_ld = s.x_ld;
  ph.out_ld = s.out_ld;
  ph.out_cols = s.out_cols;
  ph.trace_slot = s.trace_slot;
  return ph;
}

// Every K slice gets at least one CTA (the same integer formula as the device's slice_geom).
bool slices_ok(const Phase& ph, int G) {
  int prev = 0;
  for (int s = 1; s <= ph.ks; ++s) {
    const int kg = (int)((long long)s * ph.KG / ph.ks);
    const int c = s == ph.ks ? G : (int)(((long long)G * kg + ph.KG / 2) / ph.KG);
    if (c <= prev) return false;
    prev = c;
  }
  return true;
}

// The split-K bookkeeping a program needs: floats per lane of a partial (4 NT; 8 NT when a phase is
// interleaved) and the largest cross-slice slot area (RB * ks partials of the phases with ks > 1).
struct Needs {
  int NT = 1;
  bool two = false;
  size_t x_parts = 0;
  explicit Needs(int nt = 1) : NT(nt) {}
  void add(const Phase& ph) {
    two = two || ph.layout == kInterleaved;
    if (ph.ks > 1) x_parts = std::max(x_parts, (size_t)ph.RB * ph.ks);
  }
  int cs_lane() const { return 4 * NT * (two ? 2 : 1); }
  WsLayout layout(int grid = kMaxGrid) const { return ws_layout(cs_lane(), x_parts * 32 * (size_t)cs_lane(), grid); }
};

Io make_io(void* ws, const WsLayout& L, int cs_lane) {
  Io io;
  memset(&io, 0, sizeof(io));
  uint8_t* b = static_cast<uint8_t*>(ws);
  io.status = reinterpret_cast<int*>(b + L.status);
  io.bar = reinterpret_cast<unsigned*>(b + L.bar);
  io.head_cnt = reinterpret_cast<unsigned*>(b + L.head_cnt);
  io.head_aux = reinterpret_cast<float*>(b + L.head_aux);
  io.cslots = reinterpret_cast<float*>(b + L.cslots);
  io.xslots = reinterpret_cast<float*>(b + L.xslots);
  io.cs_lane = cs_lane;
  return io;
}

// Launches phases [0, n) of `phases` as programs of at most kMaxPhases phases each.
vp_status run_phases(const std::vector<Phase>& phases, int M, float eps, const Io& io, int G, cudaStream_t s,
                     int rows = 8) {
  const int n = (int)phases.size();
  const int launches = (n + kMaxPhases - 1) / kMaxPhases;
  static thread_local Program prog;  // ~12 KB: kept off the stack
  for (int l = 0; l < launches; ++l) {
    const int p0 = (int)((long long)l * n / launches), p1 = (int)((long long)(l + 1) * n / launches);
    prog.n = p1 - p0;
    prog.M = M;
    prog.eps = eps;
    prog.q4 = phases[p0].fmt == kFmtQ4;  // a program is all Q4 or has none (checked by the callers)
    prog.rows = rows;
    for (int i = p0; i < p1; ++i) prog.ph[i - p0] = phases[i];
    cudaError_t e = launch_exec(prog, io, G, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return VP_OK;
}

int program_launches(int n_phases) { return (n_phases + kMaxPhases - 1) / kMaxPhases; }

// ------------------------------------------------------------------ packers
// Canonical row-major weights -> the packed layout of internal.h.  One thread per 16-byte piece of
// a strip: NVFP4 strips have 64 code pieces ([h][g][c]) and 8 scale pieces ([g]); FP8 strips 64.
__global__ void pack_nvfp4_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, int N, int K,
                                  uint8_t* __restrict__ out) {
  const int KC = K / 256;
  const long long pieces = (long long)(N / 8) * KC * 72;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < pieces;
       i += (long long)gridDim.x * blockDim.x) {
    const long long strip = i / 72;
    const int piece = (int)(i % 72);
    const int t = (int)(strip & 1), kc = (int)((strip >> 1) % KC);
    const long long rb = (strip >> 1) / KC;
    uint8_t b[16];
    if (piece < 64) {
      const int h = piece >> 5, g = (piece >> 2) & 7, c = piece & 3;
      const uint8_t* src = codes + (size_t)(rb * 16 + t * 8 + g) * (K / 2) + (size_t)kc * 128;
#pragma unroll
      for (int ss = 0; ss < 8; ++ss) {
        const int s = 8 * h + ss;
        b[2 * ss] = src[8 * s + 2 * c];
        b[2 * ss + 1] = src[8 * s + 2 * c + 1];
      }
    } else {
      const int g = piece - 64;
      const uint8_t* src = scales + (size_t)(rb * 16 + t * 8 + g) * (K / 16) + (size_t)kc * 16;
#pragma unroll
      for (int s = 0; s < 16; ++s) b[s] = src[s];
    }
    uint4 v;
    memcpy(&v, b, 16);
    *reinterpret_cast<uint4*>(out + strip * 1152 + piece * 16) = v;
  }
}

__global__ void pack_fp8_kernel(const uint8_t* __restrict__ w, int N, int K, uint8_t* __restrict__ out) {
  const int KC = K / 128;
  const long long pieces = (long long)(N / 8) * KC * 64;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < pieces;
       i += (long long)gridDim.x * blockDim.x) {
    const long long strip = i / 64;
    const int piece = (int)(i % 64);
    const int t = (int)(strip & 1), kc = (int)((strip >> 1) % KC);
    const long long rb = (strip >> 1) / KC;
    const int h = piece >> 5, g = (piece >> 2) & 7, c = piece & 3;
    const uint8_t* src = w + (size_t)(rb * 16 + t * 8 + g) * K + (size_t)kc * 128;
    uint32_t q[4];
#pragma unroll
    for (int ss = 0; ss < 4; ++ss) q[ss] = *reinterpret_cast<const uint32_t*>(src + 16 * (4 * h + ss) + 4 * c);
    *reinterpret_cast<uint4*>(out + strip * 1024 + piece * 16) = make_uint4(q[0], q[1], q[2], q[3]);
  }
}

// Q4: codes [N][K/2] (low nibble first), scales and biases bf16 [N][K/64].  Code pieces hold, per
// 32-bit word, steps s and s + 1 of the piece's lane in the nibble order of internal.h; scale piece g
// holds the four (scale, bias) pairs of row g's groups in the chunk.
__global__ void pack_q4_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                               const uint16_t* __restrict__ biases, int N, int K, uint8_t* __restrict__ out) {
  const int KC = K / 256;
  const long long pieces = (long long)(N / 8) * KC * 72;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < pieces;
       i += (long long)gridDim.x * blockDim.x) {
    const long long strip = i / 72;
    const int piece = (int)(i % 72);
    const int t = (int)(strip & 1), kc = (int)((strip >> 1) % KC);
    const long long rb = (strip >> 1) / KC;
    uint32_t wd[4];
    if (piece < 64) {
      const int h = piece >> 5, g = (piece >> 2) & 7, c = piece & 3;
      const uint8_t* src = codes + (size_t)(rb * 16 + t * 8 + g) * (K / 2) + (size_t)kc * 128;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int s0 = 8 * h + 2 * w;
        uint32_t q[2][4];  // [step][k within the lane's four]
#pragma unroll
        for (int d = 0; d < 2; ++d) {
          const uint8_t b0 = src[8 * (s0 + d) + 2 * c], b1 = src[8 * (s0 + d) + 2 * c + 1];
          q[d][0] = b0 & 15u;
          q[d][1] = b0 >> 4;
          q[d][2] = b1 & 15u;
          q[d][3] = b1 >> 4;
        }
        wd[w] = q[0][0] | q[1][0] << 4 | q[0][2] << 8 | q[1][2] << 12 | q[0][1] << 16 | q[1][1] << 20 |
                q[0][3] << 24 | q[1][3] << 28;
      }
    } else {
      const int g = piece - 64;
      const size_t row = (size_t)(rb * 16 + t * 8 + g) * (K / 64) + (size_t)kc * 4;
#pragma unroll
      for (int G = 0; G < 4; ++G) wd[G] = (uint32_t)scales[row + G] | (uint32_t)biases[row + G] << 16;
    }
    *reinterpret_cast<uint4*>(out + strip * 1152 + piece * 16) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
  }
}

int pack_grid(long long total) {
  long long b = (total + 255) / 256;
  if (b > 152LL * 32) b = 152LL * 32;
  return (int)(b < 1 ? 1 : b);
}

// ------------------------------------------------------------------ argmax + accept over given logits
// Grid (chunks, M): each CTA reduces one chunk of one row, the last CTA reduces the chunks in order
// and runs the acceptance.
__global__ void __launch_bounds__(256) argmax_accept_kernel(const float* __restrict__ logits, int M, int V, int chunk,
                                                            int n_chunks, int rows, const int32_t* pending, int32_t* argmax,
                                                            int32_t* n_commit, int32_t* committed, float* aux,
                                                            unsigned* cnt) {
  __shared__ float red_v[8];
  __shared__ int red_i[8];
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
  for (int o = 1; o < 32; o <<= 1) am_shfl_xor(bv, bi, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red_v[warp] = bv;
    red_i[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float v0 = -INFINITY;
    int i0 = 0x7fffffff;
    for (int w = 0; w < 8; ++w)
      if (am_better(red_v[w], red_i[w], v0, i0)) {
        v0 = red_v[w];
        i0 = red_i[w];
      }
    aux[((size_t)c * kMaxM + m) * 2] = v0;
    aux[((size_t)c * kMaxM + m) * 2 + 1] = __int_as_float(i0);
    __threadfence();
    last = atomicAdd(cnt, 1u) + 1 == (unsigned)(n_chunks * M);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (threadIdx.x < M) {
    float v0 = -INFINITY;
    int i0 = 0x7fffffff;
    for (int cc = 0; cc < n_chunks; ++cc) {
      const float2 e = __ldcg(reinterpret_cast<const float2*>(aux) + (size_t)cc * kMaxM + threadIdx.x);
      if (am_better(e.x, __float_as_int(e.y), v0, i0)) {
        v0 = e.x;
        i0 = __float_as_int(e.y);
      }
    }
    if (i0 == 0x7fffffff) i0 = 0;
    tok[threadIdx.x] = i0;
    argmax[threadIdx.x] = i0;
  }
  __syncthreads();
  if ((int)threadIdx.x < M / rows) accept_lane(threadIdx.x, rows, tok, pending, n_commit, committed);
  if (threadIdx.x == 0) *cnt = 0u;
}

void argmax_chunking(int V, int* chunk, int* n_chunks) {
  int ch = 8192;
  if ((V + ch - 1) / ch > kMaxGrid) ch = (V + kMaxGrid - 1) / kMaxGrid;
  *chunk = ch;
  *n_chunks = (V + ch - 1) / ch;
}

Needs single_needs(const Phase& ph, int NT) {
  Needs n(NT);
  n.add(ph);
  return n;
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

int vp_get_last_cuda_error(void) { return vp::last_cuda_error(); }

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
  if (!weight_shape_ok(kFmtNvfp4, N, K)) return 0;
  return (size_t)N * (size_t)K / 16 * 9;
}

size_t vp_packed_bytes_fp8(int N, int K) {
  if (!weight_shape_ok(kFmtFp8, N, K)) return 0;
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
  pack_nvfp4_kernel<<<pack_grid((long long)(N / 8) * (K / 256) * 72), 256, 0, (cudaStream_t)stream>>>(
      (const uint8_t*)codes, (const uint8_t*)scales, N, K, (uint8_t*)packed);
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
  pack_fp8_kernel<<<pack_grid((long long)(N / 8) * (K / 128) * 64), 256, 0, (cudaStream_t)stream>>>(
      (const uint8_t*)w, N, K, (uint8_t*)packed);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

size_t vp_packed_bytes_q4(int N, int K) {
  if (!weight_shape_ok(kFmtQ4, N, K)) return 0;
  return (size_t)N * (size_t)K / 16 * 9;
}

vp_status vp_pack_q4(const void* codes, const void* scales, const void* biases, int N, int K, void* packed,
                     size_t packed_bytes, void* stream) {
  if (!codes || !scales || !biases || !packed) return VP_ERR_INVALID_ARG;
  const size_t need = vp_packed_bytes_q4(N, K);
  if (need == 0) return VP_ERR_SHAPE;
  if (packed_bytes < need) return VP_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(scales, 2) || !aligned(biases, 2) || !aligned(packed, 16))
    return VP_ERR_ALIGNMENT;
  int sms = 0;
  vp_status st = device_sms(&sms);
  if (st != VP_OK) return st;
  pack_q4_kernel<<<pack_grid((long long)(N / 8) * (K / 256) * 72), 256, 0, (cudaStream_t)stream>>>(
      (const uint8_t*)codes, (const uint16_t*)scales, (const uint16_t*)biases, N, K, (uint8_t*)packed);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

size_t vp_workspace_bytes(int op, int M, int N, int K) {
  if (op == VP_OP_ARGMAX) {
    if (M < 8 || M > kMaxM || M % 8 || N < 1) return 0;
    return ws_layout(4, 0).cslots;  // the counter and the per-chunk maxima
  }
  if (op == VP_OP_ATTN) {  // N = kv heads, K = cache capacity (positions per lane)
    if (M < 8 || M > kMaxM || M % 8 || N < 1 || K < 8 || K > (1 << 24)) return 0;
    return attn_ws_layout(M, N, K).total;
  }
  if (op == VP_OP_SAMPLE) {
    if (M < 8 || M > kMaxM || M % 8 || N < 1 || N > kSampleMaxV) return 0;
    return sample_ws_layout(M, N).total;
  }
  if (op != VP_OP_NVFP4 && op != VP_OP_FP8 && op != VP_OP_HEAD && op != VP_OP_Q4) return 0;
  const int fmt = op == VP_OP_FP8 ? kFmtFp8 : op == VP_OP_Q4 ? kFmtQ4 : kFmtNvfp4;
  if (M < 1 || M > kMaxM || !weight_shape_ok(fmt, N, K)) return 0;
  if (op == VP_OP_HEAD && M % 8) return 0;
  PhaseSpec s;
  s.fmt = fmt;
  s.rows0 = N;
  s.K = K;
  return single_needs(make_phase(s, nt_of(M)), nt_of(M)).layout().total;
}

static vp_status run_single(const PhaseSpec& s, int M, const void* x, void* ws, size_t ws_bytes, Io io_extra,
                            cudaStream_t stream) {
  const int NT = nt_of(M);
  const Phase ph = make_phase(s, NT);
  const Needs nd = single_needs(ph, NT);
  const WsLayout L = nd.layout();
  if (ws_bytes < L.total) return VP_ERR_WORKSPACE;
  int sms = 0;
  vp_status st = device_sms(&sms);
  if (st != VP_OK) return st;
  if (!slices_ok(ph, sms)) return VP_ERR_SHAPE;
  Io io = make_io(ws, L, nd.cs_lane());
  for (int b = 0; b < kNumBufs; ++b) io.buf[b] = io_extra.buf[b];
  io.buf[kBufX] = const_cast<void*>(x);
  io.pending = io_extra.pending;
  io.argmax = io_extra.argmax;
  io.n_commit = io_extra.n_commit;
  io.committed = io_extra.committed;
  std::vector<Phase> phases(1, ph);
  return run_phases(phases, M, 0.0f, io, sms, stream);
}

static vp_status linear_common(int fmt, const void* w, float scale, const void* x, float* y, int M, int N, int K,
                               void* ws, size_t ws_bytes, void* stream) {
  if (!w || !x || !y || !ws) return VP_ERR_INVALID_ARG;
  if (M < 1 || M > kMaxM || !weight_shape_ok(fmt, N, K)) return VP_ERR_SHAPE;
  if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 4) || !aligned(ws, 256)) return VP_ERR_ALIGNMENT;
  PhaseSpec s;
  s.fmt = fmt;
  s.w0 = w;
  s.s0 = scale;
  s.rows0 = N;
  s.K = K;
  s.epi = kEpiF32;
  s.x_src = kBufX;
  s.x_ld = K;
  s.out = kBufY;
  s.out_ld = N;
  Io extra;
  memset(&extra, 0, sizeof(extra));
  extra.buf[kBufY] = y;
  return run_single(s, M, x, ws, ws_bytes, extra, (cudaStream_t)stream);
}

vp_status vp_linear_nvfp4(const void* w_packed, float tensor_scale, const void* x, float* y, int M, int N, int K,
                          void* ws, size_t ws_bytes, void* stream) {
  return linear_common(kFmtNvfp4, w_packed, tensor_scale, x, y, M, N, K, ws, ws_bytes, stream);
}

vp_status vp_linear_fp8(const void* w_packed, float scale, const void* x, float* y, int M, int N, int K, void* ws,
                        size_t ws_bytes, void* stream) {
  return linear_common(kFmtFp8, w_packed, scale, x, y, M, N, K, ws, ws_bytes, stream);
}

vp_status vp_sample_accept(const float* logits, int M, int V, float temperature, int top_k, float top_p,
                           const int32_t* pending, const int32_t* draft_tokens, const float* draft_probs,
                           const float* uniforms, int32_t* n_commit, int32_t* committed, void* ws, size_t ws_bytes,
                           void* stream) {
  if (!logits || !pending || !uniforms || !n_commit || !committed || !ws) return VP_ERR_INVALID_ARG;
  if ((draft_tokens == nullptr) != (draft_probs == nullptr)) return VP_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !(temperature < INFINITY) || !(top_p > 0.0f) || !(top_p <= 1.0f))
    return VP_ERR_INVALID_ARG;
  if (M < 8 || M > kMaxM || M % 8 || V < 1 || V > kSampleMaxV || top_k < 1 || top_k > 32 || top_k > V)
    return VP_ERR_SHAPE;
  if (!aligned(logits, 4) || !aligned(pending, 4) || !aligned(uniforms, 4) || !aligned(n_commit, 4) ||
      !aligned(committed, 4) || !aligned(ws, 256) || (draft_tokens && (!aligned(draft_tokens, 4) || !aligned(draft_probs, 4))))
    return VP_ERR_ALIGNMENT;
  if (ws_bytes < sample_ws_layout(M, V).total) return VP_ERR_WORKSPACE;
  cudaError_t e = launch_sample_accept(logits, M, V, temperature, top_k, top_p, pending, draft_tokens, draft_probs,
                                       uniforms, n_commit, committed, ws, (cudaStream_t)stream);
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

vp_status vp_attention_verify(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                              const int32_t* ctx, int cap, const void* gate, void* out, int M, int Hq, int Hkv, int D,
                              void* ws, size_t ws_bytes, void* stream) {
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !ctx || !out || !ws) return VP_ERR_INVALID_ARG;
  if (M < 8 || M > kMaxM || M % 8 || D != 256 || Hkv < 1 || Hq < Hkv || Hq % Hkv || Hq / Hkv > 8 || cap < 8 ||
      cap > (1 << 24))
    return VP_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(ctx, 4) || (gate && !aligned(gate, 16)) || !aligned(out, 16) ||
      !aligned(ws, 256))
    return VP_ERR_ALIGNMENT;
  if (ws_bytes < attn_ws_layout(M, Hkv, cap).total) return VP_ERR_WORKSPACE;
  int sms = 0;
  vp_status st = device_sms(&sms);
  if (st != VP_OK) return st;
  AttnArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.k_cache = static_cast<uint16_t*>(k_cache);
  a.v_cache = static_cast<uint16_t*>(v_cache);
  a.ctx = ctx;
  a.gate = static_cast<const uint16_t*>(gate);
  a.out = static_cast<uint16_t*>(out);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.cap = cap;
  cudaError_t e = launch_attention_verify(a, M, ws, (cudaStream_t)stream);
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

vp_status vp_linear_q4(const void* w_packed, const void* x, float* y, int M, int N, int K, void* ws, size_t ws_bytes,
                       void* stream) {
  return linear_common(kFmtQ4, w_packed, 1.0f, x, y, M, N, K, ws, ws_bytes, stream);
}

vp_status vp_head_argmax_accept(const void* w_packed, float tensor_scale, const void* x, int M, int V, int K,
                                const int32_t* pending, int32_t* argmax, int32_t* n_commit, int32_t* committed,
                                float* logits, void* ws, size_t ws_bytes, void* stream) {
  if (!w_packed || !x || !pending || !argmax || !n_commit || !committed || !ws) return VP_ERR_INVALID_ARG;
  if (M < 8 || M > kMaxM || M % 8 || !weight_shape_ok(kFmtNvfp4, V, K)) return VP_ERR_SHAPE;
  if (!aligned(w_packed, 16) || !aligned(x, 16) || !aligned(ws, 256) || !aligned(pending, 4) || !aligned(argmax, 4) ||
      !aligned(n_commit, 4) || !aligned(committed, 4) || (logits && !aligned(logits, 4)))
    return VP_ERR_ALIGNMENT;
  PhaseSpec s;
  s.fmt = kFmtNvfp4;
  s.w0 = w_packed;
  s.s0 = tensor_scale;
  s.rows0 = V;
  s.K = K;
  s.epi = kEpiHead;
  s.x_src = kBufX;
  s.x_ld = K;
  s.out = kBufLogits;
  s.out_ld = V;
  Io extra;
  memset(&extra, 0, sizeof(extra));
  extra.buf[kBufLogits] = logits;
  extra.pending = pending;
  extra.argmax = argmax;
  extra.n_commit = n_commit;
  extra.committed = committed;
  return run_single(s, M, x, ws, ws_bytes, extra, (cudaStream_t)stream);
}

}  // extern "C"

// ------------------------------------------------------------------ linear layer without a workspace
// Some callers cannot hand the library a workspace: a plugin hook or a custom-op interface with a
// fixed signature that has no scratch argument, or a decode loop that must never stall, where a
// device allocation is ruled out because cudaMalloc and cudaFree synchronise the device.  For them
// vp_linear_nvfp4_noalloc runs the same streaming executor as vp_linear_nvfp4 on a scratch area
// that lives in the library itself: a fixed-size device array, zero at load time, whose address is
// looked up once per device.
namespace {

constexpr size_t kNoallocScratchBytes = (size_t)8 << 20;  // 8 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

// Address of the scratch array on the current device, looked up on the first call per device (with
// that device current) and kept.  Host threads may race on the first call: each lookup yields the
// same address, and the atomic slot makes the store and the later loads well defined.
vp_status noalloc_scratch(void** out) {
  static std::atomic<void*> addr[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return VP_ERR_UNSUPPORTED;
  void* p = addr[dev].load(std::memory_order_acquire);
  if (!p) {
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return VP_OK;
}

}  // namespace

extern "C" {

vp_status vp_linear_nvfp4_noalloc(const void* w_packed, float tensor_scale, const void* x, float* y, int M, int N,
                                  int K, void* stream) {
  if (!w_packed || !x || !y) return VP_ERR_INVALID_ARG;
  if (M < 1 || M > kMaxM || !weight_shape_ok(kFmtNvfp4, N, K)) return VP_ERR_SHAPE;
  if (!aligned(w_packed, 16) || !aligned(x, 16) || !aligned(y, 4)) return VP_ERR_ALIGNMENT;
  PhaseSpec s;
  s.fmt = kFmtNvfp4;
  s.w0 = w_packed;
  s.s0 = tensor_scale;
  s.rows0 = N;
  s.K = K;
  s.epi = kEpiF32;
  s.x_src = kBufX;
  s.x_ld = K;
  s.out = kBufY;
  s.out_ld = N;
  const int NT = nt_of(M);
  const Phase ph = make_phase(s, NT);
  int sms = 0;
  vp_status st = device_sms(&sms);
  if (st != VP_OK) return st;
  const Needs nd = single_needs(ph, NT);
  const WsLayout L = nd.layout(sms);  // in-CTA slots for this device's grid only
  if (L.total > kNoallocScratchBytes) return VP_ERR_WORKSPACE;  // the shape needs more than the fixed scratch
  if (!slices_ok(ph, sms)) return VP_ERR_SHAPE;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != VP_OK) return st;
  cudaStream_t cs = (cudaStream_t)stream;
  // The status word, the barrier and the counters must start at zero: clear them on every call
  // (the split-K slots and the head maxima are written before they are read).
  cudaError_t e = cudaMemsetAsync(scratch, 0, L.head_aux, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  Io io = make_io(scratch, L, nd.cs_lane());
  io.buf[kBufX] = const_cast<void*>(x);
  io.buf[kBufY] = y;
  static thread_local Program prog;
  prog.n = 1;
  prog.M = M;
  prog.eps = 0.0f;
  prog.q4 = 0;
  prog.rows = 8;
  prog.ph[0] = ph;
  e = launch_exec(prog, io, sms, cs);
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

vp_status vp_noalloc_read_status(int* status, void* stream) {
  if (!status) return VP_ERR_INVALID_ARG;
  void* scratch = nullptr;
  vp_status st = noalloc_scratch(&scratch);
  if (st != VP_OK) return st;
  // The status word is the first word of the scratch (the workspace layout's status offset is 0).
  cudaError_t e = cudaMemcpyAsync(status, scratch, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

vp_status vp_argmax_accept_rows(const float* logits, int M, int V, int rows, const int32_t* pending,
                                int32_t* argmax, int32_t* n_commit, int32_t* committed, void* ws, size_t ws_bytes,
                                void* stream) {
  if (!logits || !pending || !argmax || !n_commit || !committed || !ws) return VP_ERR_INVALID_ARG;
  if (rows < 1 || rows > kMaxM || M < rows || M > kMaxRows || M % rows || V < 1) return VP_ERR_SHAPE;
  if (M > kMaxM && (M % kMaxM || kMaxM % rows)) return VP_ERR_SHAPE;  // runs of 32 rows, whole lanes each
  if (!aligned(logits, 4) || !aligned(ws, 256) || !aligned(pending, 4) || !aligned(argmax, 4) ||
      !aligned(n_commit, 4) || !aligned(committed, 4))
    return VP_ERR_ALIGNMENT;
  const int Mp = M > kMaxM ? kMaxM : M;
  if (ws_bytes < vp_workspace_bytes(VP_OP_ARGMAX, Mp, V, 0)) return VP_ERR_WORKSPACE;
  int sms = 0;
  vp_status st = device_sms(&sms);
  if (st != VP_OK) return st;
  int chunk = 0, n_chunks = 0;
  argmax_chunking(V, &chunk, &n_chunks);
  const WsLayout L = ws_layout(4, 0);
  uint8_t* b = (uint8_t*)ws;
  for (int r0 = 0; r0 < M; r0 += Mp) {  // runs of at most 32 rows, whole lanes each
    const int l0 = r0 / rows;
    argmax_accept_kernel<<<dim3(n_chunks, Mp), 256, 0, (cudaStream_t)stream>>>(
        logits + (size_t)r0 * V, Mp, V, chunk, n_chunks, rows, pending + r0, argmax + r0, n_commit + l0,
        committed + (size_t)l0 * rows, (float*)(b + L.head_aux), (unsigned*)(b + L.head_cnt));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return VP_OK;
}

vp_status vp_argmax_accept(const float* logits, int M, int V, const int32_t* pending, int32_t* argmax,
                           int32_t* n_commit, int32_t* committed, void* ws, size_t ws_bytes, void* stream) {
  if (M < 8 || M % 8) return VP_ERR_SHAPE;
  return vp_argmax_accept_rows(logits, M, V, 8, pending, argmax, n_commit, committed, ws, ws_bytes, stream);
}

}  // extern "C"

// ======================================================================== the verify pass

struct vp_model {
  int hidden, inter;
  float eps;
  std::vector<vp_layer_desc> layers;
  vp_head_desc head;
  int zmax;
  std::vector<Phase> phases[4];  // per NT: 4 phases per layer (in, out, gate+up, down), then the head
  Needs needs[4] = {Needs(1), Needs(2), Needs(3), Needs(4)};
  // the real mixer cores (vp_model_set_cores): the same program with the in-projections kept whole
  bool has_cores = false;
  vp_core_geom cg{};
  std::vector<vp_core_desc> cores;
  int umax = 0;  // widest in-projection (both segments)
  std::vector<Phase> cphases[4];
  Needs cneeds[4] = {Needs(1), Needs(2), Needs(3), Needs(4)};
  RopeTable rope{};
};

namespace vp {
int model_hidden(const vp_model* model) { return model ? model->hidden : 0; }
}  // namespace vp

namespace {

// The pass's phases at NT n-tiles.  Block 2l (mixer of layer l) = phases 4l, 4l + 1; block 2l + 1
// (its MLP) = phases 4l + 2, 4l + 3; the head is the last phase.  cores: the in-projections keep
// every row (kEpiU into the U buffer) for the real mixer cores.
void build_pass(vp_model* md, int NT, bool cores = false) {
  const int H = md->hidden, I = md->inter;
  std::vector<Phase>& out = cores ? md->cphases[NT - 1] : md->phases[NT - 1];
  Needs& nd = cores ? md->cneeds[NT - 1] : md->needs[NT - 1];
  out.clear();
  for (int l = 0; l < (int)md->layers.size(); ++l) {
    const vp_layer_desc& d = md->layers[l];
    PhaseSpec in;  // mixer in-projection (GDN in, or attention q + kv): z = bf16(u[:, :k_out])
    in.fmt = kFmtFp8;
    in.w0 = d.w_in;
    in.s0 = d.s_in;
    in.rows0 = d.n_in;
    if (d.kind == VP_LAYER_ATTN) {
      in.w1 = d.w_kv;
      in.s1 = d.s_kv;
      in.rows1 = d.n_kv;
    }
    in.K = H;
    in.epi = kEpiZ;
    in.x_src = kBufH;
    in.x_ld = H;
    in.x_rms = 1;
    in.ss = l > 0 ? kSsRead : 0;  // layer 0 reads x0, which no phase produced
    in.out = kBufZ;
    in.out_ld = d.k_out;
    in.out_cols = d.k_out;
    if (cores) {
      in.epi = kEpiU;
      in.out = kBufU;
      in.out_ld = d.n_in + (d.kind == VP_LAYER_ATTN ? d.n_kv : 0);
    }
    out.push_back(make_phase(in, NT));
    PhaseSpec o;  // mixer out-projection + residual
    o.fmt = kFmtFp8;
    o.w0 = d.w_out;
    o.s0 = d.s_out;
    o.rows0 = H;
    o.K = d.k_out;
    o.epi = kEpiResid;
    o.x_src = kBufZ;
    o.x_ld = d.k_out;
    o.out = kBufH;
    o.out_ld = H;
    o.ss = kSsWrite;
    o.trace_slot = 2 * l;
    out.push_back(make_phase(o, NT));
    PhaseSpec gu;  // MLP gate + up, interleaved strips -> a = bf16(silu(gate) * up)
    gu.fmt = kFmtNvfp4;
    gu.layout = kInterleaved;
    gu.w0 = d.w_gate;
    gu.s0 = d.ts_gate;
    gu.w1 = d.w_up;
    gu.s1 = d.ts_up;
    gu.rows0 = I;
    gu.K = H;
    gu.epi = kEpiSilu;
    gu.x_src = kBufH;
    gu.x_ld = H;
    gu.x_rms = 1;
    gu.ss = kSsRead;
    gu.out = kBufA;
    gu.out_ld = I;
    out.push_back(make_phase(gu, NT));
    PhaseSpec dn;  // MLP down + residual
    dn.fmt = kFmtNvfp4;
    dn.w0 = d.w_down;
    dn.s0 = d.ts_down;
    dn.rows0 = H;
    dn.K = I;
    dn.epi = kEpiResid;
    dn.x_src = kBufA;
    dn.x_ld = I;
    dn.out = kBufH;
    dn.out_ld = H;
    dn.ss = kSsWrite;
    dn.trace_slot = 2 * l + 1;
    out.push_back(make_phase(dn, NT));
  }
  PhaseSpec hd;
  hd.fmt = kFmtNvfp4;
  hd.w0 = md->head.w;
  hd.s0 = md->head.ts;
  hd.rows0 = md->head.vocab;
  hd.K = H;
  hd.epi = kEpiHead;
  hd.x_src = kBufH;
  hd.x_ld = H;
  hd.x_rms = 1;
  hd.ss = kSsRead;
  hd.out = kBufLogits;
  hd.out_ld = md->head.vocab;
  out.push_back(make_phase(hd, NT));
  nd = Needs(NT);
  for (const Phase& ph : out) nd.add(ph);
}

struct PassWs {
  WsLayout L;
  size_t h, z, a, rss, total;
};

PassWs pass_ws(const vp_model* md, int M) {
  const int NT = nt_of(M);
  PassWs w;
  w.L = md->needs[NT - 1].layout();
  size_t off = w.L.total;
  w.h = off;
  off = align_up(off + sizeof(uint16_t) * (size_t)M * md->hidden, 256);
  w.z = off;
  off = align_up(off + sizeof(uint16_t) * (size_t)M * md->zmax, 256);
  w.a = off;
  off = align_up(off + sizeof(uint16_t) * (size_t)M * md->inter, 256);
  w.rss = off;
  off = align_up(off + sizeof(float) * (size_t)M * (md->hidden / kRowBlock), 256);
  w.total = off;
  return w;
}

// The cores pass's workspace: the pass's, then the in-projections kept whole and the cores' scratch.
struct CoresWs {
  PassWs P;
  size_t u, aq, ak, av, ag, attn, rec, rec_qk, rec_v, rec_ab, rec_layer, total;
};
CoresWs cores_ws(const vp_model* md, int M) {
  CoresWs w;
  w.P = pass_ws(md, M);
  const vp_core_geom& g = md->cg;
  const size_t hq = (size_t)M * g.Hq * g.D, hk = (size_t)M * g.Hkv * g.D;
  size_t off = w.P.total;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  w.u = take(sizeof(uint16_t) * (size_t)M * md->umax);
  w.aq = take(sizeof(uint16_t) * hq);
  w.ag = take(sizeof(uint16_t) * hq);
  w.ak = take(sizeof(uint16_t) * hk);
  w.av = take(sizeof(uint16_t) * hk);
  w.attn = take(g.Hkv > 0 && g.cap >= 8 ? attn_ws_layout(M, g.Hkv, g.cap).total : 0);
  // per Gated DeltaNet layer, the scan's recorded inputs for the commit re-scan
  w.rec_qk = 0;
  w.rec_v = align_up(sizeof(uint16_t) * (size_t)M * 2 * g.n_qk * g.d, 256);
  w.rec_ab = align_up(w.rec_v + sizeof(uint16_t) * (size_t)M * g.n_v * g.d, 256);
  w.rec_layer = align_up(w.rec_ab + sizeof(float) * (size_t)M * g.n_v * 2, 256);
  int n_gdn = 0;
  for (const vp_layer_desc& d : md->layers) n_gdn += d.kind == VP_LAYER_GDN;
  w.rec = take(w.rec_layer * n_gdn);
  w.total = off;
  return w;
}

bool fp8_ok(const void* w, int N, int K) { return w && aligned(w, 16) && vp_packed_bytes_fp8(N, K) > 0; }
bool nvfp4_ok(const void* w, int N, int K) { return w && aligned(w, 16) && vp_packed_bytes_nvfp4(N, K) > 0; }

// lanes: the call ends in the head's acceptance, so M must be whole lanes of 8 rows.
vp_status pass_args_ok(const vp_model* md, int M, void* ws, size_t ws_bytes, bool lanes) {
  if (!md || !ws) return VP_ERR_INVALID_ARG;
  if (M < 1 || M > kMaxM || (lanes && M % 8)) return VP_ERR_SHAPE;
  if (!aligned(ws, 256)) return VP_ERR_ALIGNMENT;
  if (ws_bytes < pass_ws(md, M).total) return VP_ERR_WORKSPACE;
  return VP_OK;
}

}  // namespace

extern "C" {

vp_status vp_model_create(int hidden, int inter, float rms_eps, const vp_layer_desc* layers, int n_layers,
                          const vp_head_desc* head, vp_model** out) {
  if (!layers || !head || !out || n_layers < 1 || !(rms_eps >= 0.0f)) return VP_ERR_INVALID_ARG;
  if (hidden < 256 || hidden % 256 || inter < 256 || inter % 256) return VP_ERR_SHAPE;
  int zmax = 128;
  for (int l = 0; l < n_layers; ++l) {
    const vp_layer_desc& d = layers[l];
    if (d.kind != VP_LAYER_GDN && d.kind != VP_LAYER_ATTN) return VP_ERR_INVALID_ARG;
    if (!fp8_ok(d.w_in, d.n_in, hidden) || !fp8_ok(d.w_out, hidden, d.k_out)) return VP_ERR_SHAPE;
    if (d.k_out > d.n_in) return VP_ERR_SHAPE;
    if (d.kind == VP_LAYER_ATTN && !fp8_ok(d.w_kv, d.n_kv, hidden)) return VP_ERR_SHAPE;
    if (d.kind == VP_LAYER_GDN && (d.w_kv || d.n_kv)) return VP_ERR_INVALID_ARG;
    if (!nvfp4_ok(d.w_gate, inter, hidden) || !nvfp4_ok(d.w_up, inter, hidden) || !nvfp4_ok(d.w_down, hidden, inter))
      return VP_ERR_SHAPE;
    if (d.k_out > zmax) zmax = d.k_out;
  }
  if (!nvfp4_ok(head->w, head->vocab, hidden)) return VP_ERR_SHAPE;
  vp_model* m = new (std::nothrow) vp_model;
  if (!m) return VP_ERR_INVALID_ARG;
  m->hidden = hidden;
  m->inter = inter;
  m->eps = rms_eps;
  m->layers.assign(layers, layers + n_layers);
  m->head = *head;
  m->zmax = zmax;
  for (int nt = 1; nt <= 4; ++nt) build_pass(m, nt);
  *out = m;
  return VP_OK;
}

void vp_model_destroy(vp_model* model) { delete model; }

size_t vp_pass_workspace_bytes(const vp_model* model, int M) {
  if (!model || M < 1 || M > kMaxRows || (M > kMaxM && M % kMaxM)) return 0;
  return pass_ws(model, M > kMaxM ? kMaxM : M).total;  // more rows run as passes of 32
}

vp_status vp_trace_read(int M, void* dst, size_t bytes, unsigned* launches) {
  if (!dst || !launches) return VP_ERR_INVALID_ARG;
  if (M < 1 || M > kMaxM) return VP_ERR_SHAPE;
  const cudaError_t e = nt_of(M) <= 2 ? trace_read_nt12(dst, bytes, launches) : trace_read_nt34(dst, bytes, launches);
  if (e == cudaErrorNotSupported) return VP_ERR_UNSUPPORTED;
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

int vp_pass_launch_count(const vp_model* model) {
  return model ? program_launches((int)model->phases[0].size()) : 0;
}

}  // extern "C"

namespace {

// The pass's launches once its arguments are checked: the x0 copy, then the phase program.
vp_status enqueue_pass(const vp_model* md, const void* x0, int M, const int32_t* pending, int32_t* argmax,
                       int32_t* n_commit, int32_t* committed, void* trace, float* logits, void* ws, int sms,
                       cudaStream_t s, int rows = 8) {
  const std::vector<Phase>& phases = md->phases[nt_of(M) - 1];
  const PassWs w = pass_ws(md, M);
  uint8_t* b = (uint8_t*)ws;
  Io io = make_io(ws, w.L, md->needs[nt_of(M) - 1].cs_lane());
  io.buf[kBufH] = b + w.h;
  io.buf[kBufZ] = b + w.z;
  io.buf[kBufA] = b + w.a;
  io.rss = reinterpret_cast<float*>(b + w.rss);
  io.rss_ld = md->hidden / kRowBlock;
  io.buf[kBufLogits] = logits;
  io.buf[kBufTrace] = trace;
  io.trace_stride = (size_t)M * md->hidden;
  io.pending = pending;
  io.argmax = argmax;
  io.n_commit = n_commit;
  io.committed = committed;
  cudaError_t e = cudaMemcpyAsync(io.buf[kBufH], x0, sizeof(uint16_t) * (size_t)M * md->hidden,
                                  cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return run_phases(phases, M, md->eps, io, sms, s, rows);
}

vp_status pass_io_ok(const vp_model* md, const void* x0, int M, const int32_t* pending, int32_t* argmax,
                     int32_t* n_commit, int32_t* committed, void* trace, float* logits, void* ws, size_t ws_bytes,
                     int* sms) {
  vp_status st = pass_args_ok(md, M, ws, ws_bytes, true);
  if (st != VP_OK) return st;
  if (!x0 || !pending || !argmax || !n_commit || !committed) return VP_ERR_INVALID_ARG;
  if (!aligned(x0, 16) || (trace && !aligned(trace, 16)) || (logits && !aligned(logits, 4)) || !aligned(pending, 4) ||
      !aligned(argmax, 4) || !aligned(n_commit, 4) || !aligned(committed, 4))
    return VP_ERR_ALIGNMENT;
  if ((st = device_sms(sms)) != VP_OK) return st;
  for (const Phase& ph : md->phases[nt_of(M) - 1])
    if (!slices_ok(ph, *sms)) return VP_ERR_SHAPE;
  return VP_OK;
}

// The sampled pass's workspace: the pass's, then the greedy acceptance it does not report (n_commit,
// committed of up to 4 lanes), the logits [M][vocab] fp32, the sampling kernel's.
struct SampledWs {
  size_t greedy, logits, sample, total;
};
SampledWs sampled_ws(const vp_model* md, int M) {
  SampledWs w;
  w.greedy = align_up(pass_ws(md, M).total, 256);
  w.logits = align_up(w.greedy + sizeof(int32_t) * 9 * (kMaxM / 8), 256);
  w.sample = align_up(w.logits + sizeof(float) * (size_t)M * md->head.vocab, 256);
  w.total = align_up(w.sample + sample_ws_layout(M, md->head.vocab).total, 256);
  return w;
}

}  // namespace

extern "C" {

vp_status vp_verify_pass(const vp_model* md, const void* x0, int M, const int32_t* pending, int32_t* argmax,
                         int32_t* n_commit, int32_t* committed, void* trace, float* logits, void* ws, size_t ws_bytes,
                         void* stream) {
  int sms = 0;
  vp_status st = pass_io_ok(md, x0, M, pending, argmax, n_commit, committed, trace, logits, ws, ws_bytes, &sms);
  if (st != VP_OK) return st;
  return enqueue_pass(md, x0, M, pending, argmax, n_commit, committed, trace, logits, ws, sms, (cudaStream_t)stream);
}

vp_status vp_verify_pass_rows(const vp_model* md, const void* x0, int M, int rows, const int32_t* pending,
                              int32_t* argmax, int32_t* n_commit, int32_t* committed, void* trace, float* logits,
                              void* ws, size_t ws_bytes, void* stream) {
  if (!md || !ws) return VP_ERR_INVALID_ARG;
  if (rows < 1 || rows > kMaxM || M < rows || M > kMaxRows || M % rows) return VP_ERR_SHAPE;
  // More than 32 rows: passes of 32 rows (whole lanes each) one after the other on the stream.
  if (M > kMaxM && (M % kMaxM || kMaxM % rows || trace)) return VP_ERR_SHAPE;
  const int Mp = M > kMaxM ? kMaxM : M;
  int sms = 0;
  vp_status st = pass_args_ok(md, Mp, ws, ws_bytes, false);
  if (st != VP_OK) return st;
  if (!x0 || !pending || !argmax || !n_commit || !committed) return VP_ERR_INVALID_ARG;
  if (!aligned(x0, 16) || (trace && !aligned(trace, 16)) || (logits && !aligned(logits, 4)) || !aligned(pending, 4) ||
      !aligned(argmax, 4) || !aligned(n_commit, 4) || !aligned(committed, 4))
    return VP_ERR_ALIGNMENT;
  if ((st = device_sms(&sms)) != VP_OK) return st;
  for (const Phase& ph : md->phases[nt_of(Mp) - 1])
    if (!slices_ok(ph, sms)) return VP_ERR_SHAPE;
  for (int r0 = 0; r0 < M; r0 += Mp) {
    const int l0 = r0 / rows;
    st = enqueue_pass(md, static_cast<const uint16_t*>(x0) + (size_t)r0 * md->hidden, Mp, pending + r0, argmax + r0,
                      n_commit + l0, committed + (size_t)l0 * rows, trace, logits ? logits + (size_t)r0 * md->head.vocab : nullptr,
                      ws, sms, (cudaStream_t)stream, rows);
    if (st != VP_OK) return st;
  }
  return VP_OK;
}

vp_status vp_model_set_cores(vp_model* md, const vp_core_geom* g, const vp_core_desc* cores, int n_layers) {
  if (!md || !g || !cores || n_layers != (int)md->layers.size()) return VP_ERR_INVALID_ARG;
  if (g->d != 128 || g->n_qk < 1 || g->n_v < g->n_qk || g->n_v % g->n_qk || g->n_v > 4096) return VP_ERR_SHAPE;
  if (md->hidden > 8192) return VP_ERR_SHAPE;  // the A / B projections hold two 16-byte chunks of K per thread
  if (g->D != 256 || g->Hkv < 1 || g->Hq < g->Hkv || g->Hq % g->Hkv || g->Hq / g->Hkv > 8 || g->cap < 8 ||
      g->cap > (1 << 24))
    return VP_ERR_SHAPE;
  int umax = 0;
  for (int l = 0; l < n_layers; ++l) {
    const vp_layer_desc& d = md->layers[l];
    const vp_core_desc& c = cores[l];
    if (d.kind == VP_LAYER_GDN) {
      if (d.n_in != (2 * g->n_qk + 2 * g->n_v) * g->d || d.k_out != g->n_v * g->d) return VP_ERR_SHAPE;
      if (!c.w_a || !c.w_b || !c.conv_taps || !c.a_log || !c.dt_bias || !c.norm_w || !c.state_a || !c.state_b ||
          !c.window_a || !c.conv_hist)
        return VP_ERR_INVALID_ARG;
      if (!aligned(c.state_a, 16) || !aligned(c.state_b, 16) || !aligned(c.w_a, 16) || !aligned(c.w_b, 16) ||
          !aligned(c.conv_taps, 2) || !aligned(c.window_a, 2) || !aligned(c.conv_hist, 2))
        return VP_ERR_ALIGNMENT;
      umax = std::max(umax, d.n_in);
    } else {
      if (d.n_in != 2 * g->Hq * g->D || d.n_kv != 2 * g->Hkv * g->D || d.k_out != g->Hq * g->D) return VP_ERR_SHAPE;
      if (!c.q_norm || !c.k_norm || !c.k_cache || !c.v_cache) return VP_ERR_INVALID_ARG;
      if (!aligned(c.k_cache, 16) || !aligned(c.v_cache, 16)) return VP_ERR_ALIGNMENT;
      umax = std::max(umax, d.n_in + d.n_kv);
    }
  }
  md->cg = *g;
  md->cores.assign(cores, cores + n_layers);
  md->umax = umax;
  md->rope = rope_table(g->D);
  for (int nt = 1; nt <= 4; ++nt) build_pass(md, nt, true);
  md->has_cores = true;
  return VP_OK;
}

size_t vp_pass_cores_workspace_bytes(const vp_model* model, int M) {
  if (!model || !model->has_cores || M < 8 || M > kMaxM || M % 8) return 0;
  return cores_ws(model, M).total;
}

vp_status vp_verify_pass_cores(const vp_model* md, const void* x0, int M, const int32_t* ctx, int parity,
                               const int32_t* pending, int32_t* argmax, int32_t* n_commit, int32_t* committed,
                               void* trace, float* logits, void* ws, size_t ws_bytes, void* stream) {
  if (!md || !md->has_cores || !ctx || (parity != 0 && parity != 1)) return VP_ERR_INVALID_ARG;
  if (!aligned(ctx, 4)) return VP_ERR_ALIGNMENT;
  if (M >= 8 && M <= kMaxM && M % 8 == 0 && ws_bytes < cores_ws(md, M).total) return VP_ERR_WORKSPACE;
  int sms = 0;
  vp_status st = pass_io_ok(md, x0, M, pending, argmax, n_commit, committed, trace, logits, ws, ws_bytes, &sms);
  if (st != VP_OK) return st;
  const int NT = nt_of(M), L = (int)md->layers.size();
  const std::vector<Phase>& all = md->cphases[NT - 1];
  for (const Phase& ph : all)
    if (!slices_ok(ph, sms)) return VP_ERR_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  const CoresWs w = cores_ws(md, M);
  uint8_t* b = (uint8_t*)ws;
  Io io = make_io(ws, w.P.L, md->needs[NT - 1].cs_lane());
  io.buf[kBufH] = b + w.P.h;
  io.buf[kBufZ] = b + w.P.z;
  io.buf[kBufA] = b + w.P.a;
  io.buf[kBufU] = b + w.u;
  io.rss = reinterpret_cast<float*>(b + w.P.rss);
  io.rss_ld = md->hidden / kRowBlock;
  io.buf[kBufLogits] = logits;
  io.buf[kBufTrace] = trace;
  io.trace_stride = (size_t)M * md->hidden;
  io.pending = pending;
  io.argmax = argmax;
  io.n_commit = n_commit;
  io.committed = committed;
  cudaError_t e = cudaMemcpyAsync(io.buf[kBufH], x0, sizeof(uint16_t) * (size_t)M * md->hidden,
                                  cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e);
  const vp_core_geom& g = md->cg;
  const uint16_t* h = static_cast<const uint16_t*>(io.buf[kBufH]);
  const uint16_t* u = reinterpret_cast<const uint16_t*>(b + w.u);
  uint16_t* zb = static_cast<uint16_t*>(io.buf[kBufZ]);
  // Program segments: [in(0)], then per layer l: its core, then [out(l), gate+up(l), down(l), in(l + 1)]
  // (the head after the last layer's down).
  int gdn_index = 0;
  for (int l = 0; l <= L; ++l) {
    const int p0 = l == 0 ? 0 : 4 * (l - 1) + 1, p1 = l == 0 ? 1 : 4 * l + 1;
    std::vector<Phase> seg(all.begin() + p0, all.begin() + p1);
    if ((st = run_phases(seg, M, md->eps, io, sms, s)) != VP_OK) return st;
    if (l == L) break;
    const vp_layer_desc& d = md->layers[l];
    const vp_core_desc& c = md->cores[l];
    const int ld_u = d.n_in + (d.kind == VP_LAYER_ATTN ? d.n_kv : 0);
    if (d.kind == VP_LAYER_GDN) {
      GdnCoreArgs ga;
      ga.h = h;
      ga.hidden = md->hidden;
      ga.eps = md->eps;
      ga.u = u;
      ga.ld_u = ld_u;
      ga.z0 = (2 * g.n_qk + g.n_v) * g.d;
      ga.window_a = static_cast<const uint16_t*>(c.window_a);
      ga.taps = static_cast<const uint16_t*>(c.conv_taps);
      ga.wa = static_cast<const uint16_t*>(c.w_a);
      ga.wb = static_cast<const uint16_t*>(c.w_b);
      ga.a_log = c.a_log;
      ga.dt_bias = c.dt_bias;
      ga.norm_w = c.norm_w;
      ga.state_in = parity ? c.state_b : c.state_a;
      ga.state_out = parity ? c.state_a : c.state_b;
      ga.conv_hist = static_cast<uint16_t*>(c.conv_hist);
      ga.out = zb;
      uint8_t* rec = b + w.rec + w.rec_layer * gdn_index++;
      ga.rec_qk = reinterpret_cast<uint16_t*>(rec + w.rec_qk);
      ga.rec_v = reinterpret_cast<uint16_t*>(rec + w.rec_v);
      ga.rec_ab = reinterpret_cast<float*>(rec + w.rec_ab);
      ga.n_qk = g.n_qk;
      ga.n_v = g.n_v;
      if ((e = launch_gdn_core(ga, M / 8, s)) != cudaSuccess) return cuda_fail(e);
    } else {
      uint16_t *aq = reinterpret_cast<uint16_t*>(b + w.aq), *ag = reinterpret_cast<uint16_t*>(b + w.ag);
      uint16_t *ak = reinterpret_cast<uint16_t*>(b + w.ak), *av = reinterpret_cast<uint16_t*>(b + w.av);
      if ((e = launch_attn_prep(u, ld_u, u + d.n_in, ld_u, M, g.Hq, g.Hkv, g.D, c.q_norm, c.k_norm, ctx, md->rope, aq,
                                ak, av, ag, s)) != cudaSuccess)
        return cuda_fail(e);
      AttnArgs aa;
      memset(&aa, 0, sizeof(aa));
      aa.q = aq;
      aa.k_new = ak;
      aa.v_new = av;
      aa.k_cache = static_cast<uint16_t*>(c.k_cache);
      aa.v_cache = static_cast<uint16_t*>(c.v_cache);
      aa.ctx = ctx;
      aa.gate = ag;
      aa.out = zb;
      aa.Hq = g.Hq;
      aa.Hkv = g.Hkv;
      aa.cap = g.cap;
      if ((e = launch_attention_verify(aa, M, b + w.attn, s, io.status)) != cudaSuccess) return cuda_fail(e);
    }
  }
  return VP_OK;
}

vp_status vp_commit_cores(const vp_model* md, int M, const int32_t* n_commit, int parity, void* ws, size_t ws_bytes,
                          void* stream) {
  if (!md || !md->has_cores || !n_commit || !ws || (parity != 0 && parity != 1)) return VP_ERR_INVALID_ARG;
  if (M < 8 || M > kMaxM || M % 8) return VP_ERR_SHAPE;
  if (!aligned(ws, 256) || !aligned(n_commit, 4)) return VP_ERR_ALIGNMENT;
  const CoresWs w = cores_ws(md, M);
  if (ws_bytes < w.total) return VP_ERR_WORKSPACE;
  uint8_t* b = static_cast<uint8_t*>(ws);
  static thread_local GdnCommitArgs ca;  // ~2.7 KB: kept off the stack
  ca.n_commit = n_commit;
  ca.lanes = M / 8;
  ca.n_qk = md->cg.n_qk;
  ca.n_v = md->cg.n_v;
  int n = 0, gdn_index = 0;
  for (int l = 0; l < (int)md->layers.size(); ++l) {
    if (md->layers[l].kind != VP_LAYER_GDN) continue;
    const vp_core_desc& c = md->cores[l];
    GdnCommitLayer& L = ca.layer[n++];
    L.state_in = parity ? c.state_b : c.state_a;
    L.state_out = parity ? c.state_a : c.state_b;
    L.conv_hist = static_cast<const uint16_t*>(c.conv_hist);
    L.window = static_cast<uint16_t*>(c.window_a);
    const uint8_t* rec = b + w.rec + w.rec_layer * gdn_index++;
    L.rec_qk = reinterpret_cast<const uint16_t*>(rec + w.rec_qk);
    L.rec_v = reinterpret_cast<const uint16_t*>(rec + w.rec_v);
    L.rec_ab = reinterpret_cast<const float*>(rec + w.rec_ab);
    if (n == kCommitLayers) {
      const cudaError_t e = launch_gdn_commit(ca, n, (cudaStream_t)stream);
      if (e != cudaSuccess) return cuda_fail(e);
      n = 0;
    }
  }
  if (n > 0) {
    const cudaError_t e = launch_gdn_commit(ca, n, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return VP_OK;
}

int vp_pass_cores_launch_count(const vp_model* md) {
  if (!md || !md->has_cores) return 0;
  // one executor program per segment (the in-projection of layer 0, then 4 phases per layer, the
  // last with the head), then per Gated DeltaNet layer its whole core (one cluster launch); per
  // attention layer the prep, the cache append, the partitions and the merge
  int n = program_launches(1);
  for (const vp_layer_desc& d : md->layers) n += program_launches(4) + (d.kind == VP_LAYER_GDN ? 1 : 4);
  return n;
}

size_t vp_pass_sampled_workspace_bytes(const vp_model* model, int M) {
  if (!model || M < 8 || M > kMaxM || M % 8 || model->head.vocab > kSampleMaxV) return 0;
  return sampled_ws(model, M).total;
}

vp_status vp_verify_pass_sampled(const vp_model* md, const void* x0, int M, const int32_t* pending, float temperature,
                                 int top_k, float top_p, const int32_t* draft_tokens, const float* draft_probs,
                                 const float* uniforms, int32_t* argmax, int32_t* n_commit, int32_t* committed,
                                 float* logits, void* ws, size_t ws_bytes, void* stream) {
  if (!md || !uniforms) return VP_ERR_INVALID_ARG;
  if ((draft_tokens == nullptr) != (draft_probs == nullptr)) return VP_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !(temperature < INFINITY) || !(top_p > 0.0f) || !(top_p <= 1.0f))
    return VP_ERR_INVALID_ARG;
  const int V = md->head.vocab;
  if (top_k < 1 || top_k > 32 || top_k > V || V > kSampleMaxV) return VP_ERR_SHAPE;
  if (!aligned(uniforms, 4) || (draft_tokens && (!aligned(draft_tokens, 4) || !aligned(draft_probs, 4))))
    return VP_ERR_ALIGNMENT;
  if (M >= 8 && M <= kMaxM && M % 8 == 0 && ws_bytes < sampled_ws(md, M).total) return VP_ERR_WORKSPACE;
  int sms = 0;
  vp_status st = pass_io_ok(md, x0, M, pending, argmax, n_commit, committed, nullptr, logits, ws, ws_bytes, &sms);
  if (st != VP_OK) return st;
  const SampledWs w = sampled_ws(md, M);
  uint8_t* b = (uint8_t*)ws;
  float* lg = logits ? logits : reinterpret_cast<float*>(b + w.logits);
  int32_t* greedy = reinterpret_cast<int32_t*>(b + w.greedy);
  cudaStream_t s = (cudaStream_t)stream;
  // The head phase writes the logits (and the argmax); its greedy acceptance goes to scratch, the
  // sampled acceptance over the same logits to the caller.
  st = enqueue_pass(md, x0, M, pending, argmax, greedy, greedy + kMaxM / 8, nullptr, lg, ws, sms, s);
  if (st != VP_OK) return st;
  cudaError_t e = launch_sample_accept(lg, M, V, temperature, top_k, top_p, pending, draft_tokens, draft_probs,
                                       uniforms, n_commit, committed, b + w.sample, s);
  return e == cudaSuccess ? VP_OK : cuda_fail(e);
}

vp_status vp_verify_blocks(const vp_model* md, void* h, int M, int block_begin, int block_end, void* trace, void* ws,
                           size_t ws_bytes, void* stream) {
  vp_status st = pass_args_ok(md, M, ws, ws_bytes, false);
  if (st != VP_OK) return st;
  if (!h) return VP_ERR_INVALID_ARG;
  const int nb = 2 * (int)md->layers.size();
  if (block_begin < 0 || block_end > nb || block_begin > block_end) return VP_ERR_INVALID_ARG;
  if (!aligned(h, 16) || (trace && !aligned(trace, 16))) return VP_ERR_ALIGNMENT;
  if (block_begin == block_end) return VP_OK;
  int sms = 0;
  if ((st = device_sms(&sms)) != VP_OK) return st;
  const std::vector<Phase>& all = md->phases[nt_of(M) - 1];
  std::vector<Phase> phases(all.begin() + 2 * block_begin, all.begin() + 2 * block_end);
  for (Phase& ph : phases) {
    if (!slices_ok(ph, sms)) return VP_ERR_SHAPE;
    if (ph.trace_slot >= 0) ph.trace_slot -= block_begin;
  }
  phases[0].ss &= ~kSsRead;  // the caller's h: no producer left its row-block sums
  const PassWs w = pass_ws(md, M);
  uint8_t* b = (uint8_t*)ws;
  Io io = make_io(ws, w.L, md->needs[nt_of(M) - 1].cs_lane());
  io.buf[kBufH] = h;
  io.buf[kBufZ] = b + w.z;
  io.buf[kBufA] = b + w.a;
  io.rss = reinterpret_cast<float*>(b + w.rss);
  io.rss_ld = md->hidden / kRowBlock;
  io.buf[kBufTrace] = trace;
  io.trace_stride = (size_t)M * md->hidden;
  return run_phases(phases, M, md->eps, io, sms, (cudaStream_t)stream);
}

}  // extern "C"
