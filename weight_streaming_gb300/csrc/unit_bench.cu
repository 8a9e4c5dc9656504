// Cost breakdown of the executor's unit loop (a measurement build, libverify_unitbench.so; not part of
// the verify pass).  Every warp keeps two NVFP4 units (16 rows x 512 K, 4608 bytes each, the packed
// layout of internal.h) and the activation fragments of their K range resident in shared memory and
// runs the unit computation over them `reps` times, so no memory traffic is timed: the rate is the
// SM's compute rate for the unit at NT n-tiles of 8 tokens, in weight bytes per second.  Variants
// take parts of the computation out:
//   0 full: code and scale loads, E2M1 / E4M3 conversion and block scaling, activation-fragment
//     loads, mma.sync (the executor's unit_nvfp4);
//   1 no MMA: as 0 with the MMAs replaced by one integer add per A register (the conversion results
//     stay live);
//   2 no conversion: the code words go to the MMAs as they are (code and activation loads, MMAs);
//   3 conversion only: code and scale loads and the conversion and scaling, no activation loads, no
//     MMA;
//   4 pairs: the gate+up unit (unit_nvfp4_pair): two row blocks' chunks share each activation load.
// The split shows how much of a unit's time a tensor-core path (tcgen05, whose MMAs read the
// activations from shared memory themselves) could remove: the activation loads and the MMAs, but not
// the conversion, which any path from 4-bit codes to a 16-bit operand keeps.
//
// Sources: "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max" -- "Formats, and what runs
// where" (NVFP4: E2M1 codes, one E4M3 scale per 16 weights).
#include <cuda_runtime.h>

#include "exec.cuh"

namespace vp {
namespace {

template <int NT, int kVar>
__device__ __forceinline__ void unit_variant(uint32_t ua, uint32_t xa, int lane, float (&acc)[NT][4], uint32_t& sink) {
  if constexpr (kVar == 0) {
    unit_nvfp4<NT>(ua, xa, lane, acc, acc);
  } else {
    const int g = lane >> 2;
    const uint4 c0a = lds128(ua + lane * 16), c0b = lds128(ua + 512 + lane * 16);
    const uint4 c1a = lds128(ua + 1152 + lane * 16), c1b = lds128(ua + 1152 + 512 + lane * 16);
    const uint4 s0 = lds128(ua + 1024 + g * 16), s1 = lds128(ua + 1152 + 1024 + g * 16);
    const uint32_t w0[8] = {c0a.x, c0a.y, c0a.z, c0a.w, c0b.x, c0b.y, c0b.z, c0b.w};
    const uint32_t w1[8] = {c1a.x, c1a.y, c1a.z, c1a.w, c1b.x, c1b.y, c1b.z, c1b.w};
    const uint32_t sw0[4] = {s0.x, s0.y, s0.z, s0.w}, sw1[4] = {s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      uint4 b[NT];
      if constexpr (kVar != 3) {
#pragma unroll
        for (int j = 0; j < NT; ++j) b[j] = lds128(xa + (p * NT + j) * 512);
      }
      uint32_t A[8];
      if constexpr (kVar == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          A[i] = w0[p] ^ (i * 0x01010101u);
          A[4 + i] = w1[p] ^ (i * 0x01010101u);
        }
      } else {
        const uint32_t sc0 = e4m3x2_to_f16x2((p & 1) ? (sw0[p >> 1] >> 16) : sw0[p >> 1]);
        const uint32_t sc1 = e4m3x2_to_f16x2((p & 1) ? (sw1[p >> 1] >> 16) : sw1[p >> 1]);
        uint32_t o0[4], o1[4];
        e2m1x8_to_f16x2x4(w0[p], o0);
        e2m1x8_to_f16x2x4(w1[p], o1);
        const uint32_t d0 = dup_lo16(sc0), d1 = dup_lo16(sc1), e0 = dup_hi16(sc0), e1 = dup_hi16(sc1);
        A[0] = hmul2_u32(o0[0], d0);
        A[1] = hmul2_u32(o1[0], d1);
        A[2] = hmul2_u32(o0[1], d0);
        A[3] = hmul2_u32(o1[1], d1);
        A[4] = hmul2_u32(o0[2], e0);
        A[5] = hmul2_u32(o1[2], e1);
        A[6] = hmul2_u32(o0[3], e0);
        A[7] = hmul2_u32(o1[3], e1);
      }
      if constexpr (kVar == 1 || kVar == 3) {
#pragma unroll
        for (int i = 0; i < 8; ++i) sink += A[i];
        if constexpr (kVar == 1) {
#pragma unroll
          for (int j = 0; j < NT; ++j) sink += b[j].x ^ b[j].y ^ b[j].z ^ b[j].w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_f16_16816(acc[j], A[0], A[1], A[2], A[3], b[j].x, b[j].y);
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_f16_16816(acc[j], A[4], A[5], A[6], A[7], b[j].z, b[j].w);
      }
    }
  }
}

// smem: 16 warps x 2 units x 4608 B, then the activation fragments of 512 K (NT x 16 KB).
template <int NT, int kVar>
__global__ void __launch_bounds__(kThreads, 1) unit_bench_kernel(const uint8_t* units, int reps, float* out) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + warp * 2 * 4608;
  uint8_t* xs = smem + kWarps * 2 * 4608;
  // the warp's two units (the same 9216 bytes for every warp) and f16 activations of small integers
  for (int i = lane; i < 2 * 4608 / 16; i += 32)
    reinterpret_cast<uint4*>(ring)[i] = reinterpret_cast<const uint4*>(units)[i];
  for (int i = threadIdx.x; i < NT * 512 * 16 / 16; i += kThreads) {
    const uint32_t h = 0x3C003C00u + ((i & 7) << 10);  // f16 pairs 1, 2, 3 ... (exact)
    reinterpret_cast<uint4*>(xs)[i] = make_uint4(h, h, h, h);
  }
  __syncthreads();
  float acc[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[j][r] = 0.0f;
  uint32_t sink = 0;
  const uint32_t ua = smem_addr(ring), xa = smem_addr(xs) + lane * 16;
  const int pair_stride = 8 * NT * 512;
  float acc2[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc2[j][r] = 0.0f;
  for (int it = 0; it < reps; ++it) {
#pragma unroll 1
    for (int u = 0; u < 2; ++u) {
      if constexpr (kVar == 4) {  // the same bytes: two chunk pairs of two row blocks
        unit_nvfp4_pair<NT>(ua + u * 4608, ua + u * 4608 + 2304, xa, lane, acc, acc2);
      } else {
        unit_variant<NT, kVar>(ua + u * 4608, xa, lane, acc, sink);
        unit_variant<NT, kVar>(ua + u * 4608 + 2304, xa + pair_stride, lane, acc, sink);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[j][r] += acc2[j][r];
  float s = __uint_as_float(sink & 0x007FFFFFu);
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) s += acc[j][r];
  out[blockIdx.x * kThreads + threadIdx.x] = s;
}

template <int NT, int kVar>
cudaError_t launch_unit_bench(const uint8_t* units, int reps, float* out, int grid, cudaStream_t st) {
  const int smem = kWarps * 2 * 4608 + NT * 512 * 16;
  cudaError_t e = cudaFuncSetAttribute(unit_bench_kernel<NT, kVar>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  unit_bench_kernel<NT, kVar><<<grid, kThreads, smem, st>>>(units, reps, out);
  return cudaGetLastError();
}

template <int NT>
cudaError_t dispatch_variant(int variant, const uint8_t* units, int reps, float* out, int grid, cudaStream_t st) {
  switch (variant) {
    case 0: return launch_unit_bench<NT, 0>(units, reps, out, grid, st);
    case 1: return launch_unit_bench<NT, 1>(units, reps, out, grid, st);
    case 2: return launch_unit_bench<NT, 2>(units, reps, out, grid, st);
    case 3: return launch_unit_bench<NT, 3>(units, reps, out, grid, st);
    case 4: return launch_unit_bench<NT, 4>(units, reps, out, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

// The ring alone, streaming from device memory: W warps per CTA, each streaming its own contiguous
// range of `src` through S slots of B bytes (one bulk copy per slot, evict-first, mbarrier
// completion), refilling a slot as soon as it is consumed -- the executor's producer.  kUnit = 0:
// consuming a slot is one shared-memory load (the ring's own rate); kUnit = 1: the executor's NVFP4
// unit at NT n-tiles on the slot's two 2304-byte chunks (B = 4608), activations resident in shared
// memory.  A wait that runs out sets *err and ends the warp's stream.
template <int NT, int kUnit>
__global__ void __launch_bounds__(kThreads, 1) ring_bench_kernel(const uint8_t* src, long long units_per_warp, int S,
                                                                  int B, int* err, float* out) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bars[kWarps][8];
  const int W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0)
    for (int s = 0; s < S; ++s) mbar_init(&bars[warp][s], 1);
  uint8_t* xs = smem + (size_t)W * S * B;
  if (kUnit)
    for (int i = threadIdx.x; i < NT * 512; i += blockDim.x)
      reinterpret_cast<uint4*>(xs)[i] = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
  fence_mbar_init();
  __syncthreads();
  const uint8_t* base = src + ((long long)blockIdx.x * W + warp) * units_per_warp * B;
  const uint32_t ring = smem_addr(smem) + warp * S * B, xa = smem_addr(xs) + lane * 16;
  const uint64_t pol = l2_evict_first_policy();
  long long issued = 0;
  if (lane == 0)
    for (; issued < S && issued < units_per_warp; ++issued) {
      mbar_arrive_expect_tx(&bars[warp][issued], (uint32_t)B);
      bulk_g2s(ring + (uint32_t)issued * B, base + issued * B, (uint32_t)B, smem_addr(&bars[warp][issued]), pol);
    }
  float acc[NT][4], acc2[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[j][r] = acc2[j][r] = 0.0f;
  uint32_t sink = 0;
  for (long long u = 0; u < units_per_warp; ++u) {
    const int s = (int)(u % S);
    if (!mbar_wait_bounded(&bars[warp][s], (uint32_t)((u / S) & 1))) {
      if (lane == 0) atomicExch(err, 1);
      break;
    }
    const uint32_t ua = ring + s * B;
    if constexpr (kUnit) {
      unit_nvfp4<NT>(ua, xa, lane, acc, NT == 1 ? acc2 : acc);
      unit_nvfp4<NT>(ua + 2304, xa + 8 * NT * 512, lane, acc, NT == 1 ? acc2 : acc);
    } else {
      sink += lds128(ua + lane * 16).x;
    }
    __syncwarp();
    if (lane == 0 && issued < units_per_warp) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bars[warp][s], (uint32_t)B);
      bulk_g2s(ua, base + issued * B, (uint32_t)B, smem_addr(&bars[warp][s]), pol);
      ++issued;
    }
  }
  float v = __uint_as_float(sink & 0x007FFFFFu);
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) v += acc[j][r] + acc2[j][r];
  out[blockIdx.x * kThreads + threadIdx.x] = v;
}

template <int NT, int kUnit>
cudaError_t launch_ring(const uint8_t* src, long long upw, int W, int S, int B, int grid, int* err, float* out,
                        cudaStream_t st) {
  const int smem = W * S * B + (kUnit ? NT * 8192 : 0);
  cudaError_t e =
      cudaFuncSetAttribute(ring_bench_kernel<NT, kUnit>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ring_bench_kernel<NT, kUnit><<<grid, W * 32, smem, st>>>(src, upw, S, B, err, out);
  return cudaGetLastError();
}

}  // namespace
}  // namespace vp

// src: device, src_bytes (16-byte aligned); warps W (1..16), slots S (1..8) of B bytes (multiple of
// 16; unit mode: B = 4608); grid CTAs each stream W ranges of src_bytes / (grid W B) slots.  nt = 0:
// the ring alone; nt = 1..4: the NVFP4 unit at nt n-tiles per slot.  out: device float [grid][512];
// err: device int, set to 1 if a wait ran out.  Returns a cudaError_t.
extern "C" int vp_ring_bench(int nt, int warps, int slots, int slot_bytes, const void* src, long long src_bytes,
                             int grid, int* err, float* out, void* stream) {
  if (!src || !err || !out || warps < 1 || warps > vp::kWarps || slots < 1 || slots > 8 || slot_bytes < 16 ||
      slot_bytes % 16 || grid < 1 || grid > 1024 || nt < 0 || nt > 4 || (nt > 0 && slot_bytes != 4608))
    return (int)cudaErrorInvalidValue;
  const long long smem = (long long)warps * slots * slot_bytes + (nt ? nt * 8192 : 0);
  if (smem > vp::kSmemBytes - 1024) return (int)cudaErrorInvalidValue;
  const long long upw = src_bytes / ((long long)grid * warps * slot_bytes);
  if (upw < 1) return (int)cudaErrorInvalidValue;
  const uint8_t* s = static_cast<const uint8_t*>(src);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (nt) {
    case 0: return (int)vp::launch_ring<1, 0>(s, upw, warps, slots, slot_bytes, grid, err, out, st);
    case 1: return (int)vp::launch_ring<1, 1>(s, upw, warps, slots, slot_bytes, grid, err, out, st);
    case 2: return (int)vp::launch_ring<2, 1>(s, upw, warps, slots, slot_bytes, grid, err, out, st);
    case 3: return (int)vp::launch_ring<3, 1>(s, upw, warps, slots, slot_bytes, grid, err, out, st);
    default: return (int)vp::launch_ring<4, 1>(s, upw, warps, slots, slot_bytes, grid, err, out, st);
  }
}

// units: device, 9216 bytes (two packed NVFP4 units); out: device float [grid][512]; one launch of
// `grid` CTAs of 16 warps, each warp running 4 x reps unit chunks.  Returns a cudaError_t.
extern "C" int vp_unit_bench(int nt, int variant, const void* units, int reps, float* out, int grid, void* stream) {
  if (!units || !out || reps < 1 || grid < 1 || grid > 1024) return (int)cudaErrorInvalidValue;
  const uint8_t* u = static_cast<const uint8_t*>(units);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (nt) {
    case 1: return (int)vp::dispatch_variant<1>(variant, u, reps, out, grid, st);
    case 2: return (int)vp::dispatch_variant<2>(variant, u, reps, out, grid, st);
    case 3: return (int)vp::dispatch_variant<3>(variant, u, reps, out, grid, st);
    case 4: return (int)vp::dispatch_variant<4>(variant, u, reps, out, grid, st);
    default: return (int)cudaErrorInvalidValue;
  }
}
