// KV append into ring slots: BF16 copy and FP8-E4M3 absmax quantisation.
//
// A new chunk's K and V (token-major [B, Lc, H, D], as a QKV projection writes
// them) are written into the ring slot chunk mod R of one layer, head-major
// [B, H, rows, D], overwriting the oldest chunk in place ("Matrix-Game 4.0:
// Harnessing Video Models for Real-Time Playable Game Worlds", section
// "技术新颖性": the ring overwrites the oldest slot instead of copying the
// window).  Both layouts keep each (b, t, h) row of D elements contiguous, so
// the transpose is a permutation of 128/256-byte rows: every thread moves
// 16-byte vectors, reads and writes are fully coalesced, and the kernel is a
// pure HBM stream (bytes in = bytes out = 2 * B * Lc * H * D * 2).
//
// The FP8 variant quantises each (b, h) block of Lc x D values with one fp32
// scale = amax / 448 (IEEE round-to-nearest division) and E4M3 codes rounded
// to nearest even with saturation ("Matrix-Game 4.0", section "技术新颖性":
// 8-bit keys/values per window interval, only the changed interval is
// re-quantised -- here the changed interval is the appended chunk).  An
// INT8-key ring quantises K with scale = amax / 127 and codes rounded half to
// even, clamped to [-127, 127] (the same section: INT8 keys, FP8 values).
#include "ptx.cuh"
#include "sab_internal.h"

namespace sab {
namespace {

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads)
append_bf16_kernel(const __grid_constant__ AppendParams p) {
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();  // the slot may still be read by the previous kernel
  int slot_row0 = p.slot_row0;
  if (p.d_chunk != nullptr) {  // graph mode: the chunk index lives on the device
    const long long c = *p.d_chunk;
    slot_row0 = (p.has_sink + (int)((c < 0 ? 0 : c) % p.ring_slots)) * p.Lc;
  }
  const int vec_per_row = p.D / 8;  // 16-byte vectors per row
  const long long per_tensor = (long long)p.B * p.H * p.Lc * vec_per_row;
  const long long total = 2 * per_tensor;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int tensor = (int)(i / per_tensor);
    long long r = i - tensor * per_tensor;
    // destination order (b, h, t, vec): consecutive threads write consecutive bytes
    const int vec = (int)(r % vec_per_row); r /= vec_per_row;
    const int t = (int)(r % p.Lc); r /= p.Lc;
    const int h = (int)(r % p.H);
    const int b = (int)(r / p.H);
    const uint4* src = reinterpret_cast<const uint4*>(
        p.src[tensor] + (((long long)b * p.Lc + t) * p.H + h) * p.D) + vec;
    uint4* dst = reinterpret_cast<uint4*>(
        static_cast<uint16_t*>(p.dst[tensor]) +
        (((long long)b * p.H + h) * p.rows + slot_row0 + t) * p.D) + vec;
    *dst = __ldg(src);
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> two E4M3 codes (RNE, satfinite); `lo` lands in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One fp32 -> INT8 code: round half to even, clamp to the symmetric range.
__device__ __forceinline__ uint32_t s8_code(float y) {
  int q;
  asm("cvt.rni.s32.f32 %0, %1;" : "=r"(q) : "f"(y));
  return (uint32_t)(min(max(q, -127), 127)) & 0xFFu;
}

__global__ void __launch_bounds__(kAppendThreads)
append_fp8_kernel(const __grid_constant__ AppendParams p) {
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();  // the slot may still be read by the previous kernel
  const int tensor = blockIdx.x;
  const bool int8 = p.k_int8 && tensor == 0;  // block-uniform
  int slot_row0 = p.slot_row0, scale_idx = p.scale_idx;
  if (p.d_chunk != nullptr) {  // graph mode: the chunk index lives on the device
    const long long c = *p.d_chunk;
    const int slot = (int)((c < 0 ? 0 : c) % p.ring_slots);
    slot_row0 = (p.has_sink + slot) * p.Lc;
    scale_idx = p.has_sink + slot;
  }
  const int bh = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H;
  const int vec_per_row = p.D / 8;
  const int nvec = p.Lc * vec_per_row;
  const uint16_t* src = p.src[tensor];
  auto src_vec = [&](int v) -> uint4 {
    const int t = v / vec_per_row, c = v % vec_per_row;
    return __ldg(reinterpret_cast<const uint4*>(src + (((long long)b * p.Lc + t) * p.H + h) * p.D) + c);
  };
  // pass 1: amax over the (b, h) block
  float amax = 0.f;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    const uint4 x = src_vec(v);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[kAppendThreads / 32];
  __shared__ float s_scale;
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
    const float sc = (m == 0.f) ? 1.0f : __fdiv_rn(m, int8 ? 127.0f : 448.0f);
    s_scale = sc;
    p.scale[tensor][(long long)bh * p.scale_stride + scale_idx] = sc;
  }
  __syncthreads();
  const float sc = s_scale;
  // pass 2: quantise (the block is re-read from L2)
  uint8_t* dst = static_cast<uint8_t*>(p.dst[tensor]) + ((long long)bh * p.rows + slot_row0) * p.D;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    const uint4 x = src_vec(v);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t out[2];
    if (int8) {
#pragma unroll
      for (int k = 0; k < 2; ++k)
        out[k] = s8_code(__fdiv_rn(bf16_lo(w[2 * k]), sc)) | (s8_code(__fdiv_rn(bf16_hi(w[2 * k]), sc)) << 8) |
                 (s8_code(__fdiv_rn(bf16_lo(w[2 * k + 1]), sc)) << 16) |
                 (s8_code(__fdiv_rn(bf16_hi(w[2 * k + 1]), sc)) << 24);
    } else {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint16_t c0 = e4m3x2(__fdiv_rn(bf16_lo(w[2 * k]), sc), __fdiv_rn(bf16_hi(w[2 * k]), sc));
        const uint16_t c1 = e4m3x2(__fdiv_rn(bf16_lo(w[2 * k + 1]), sc), __fdiv_rn(bf16_hi(w[2 * k + 1]), sc));
        out[k] = (uint32_t)c0 | ((uint32_t)c1 << 16);
      }
    }
    const int t = v / vec_per_row, c = v % vec_per_row;
    *reinterpret_cast<uint2*>(dst + (long long)t * p.D + c * 8) = make_uint2(out[0], out[1]);
  }
}

// Launch with programmatic dependent launch allowed (the kernel itself waits
// for its predecessor before touching global memory).
cudaError_t launch_pdl(void (*kernel)(AppendParams), dim3 grid, const AppendParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kAppendThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Graph mode: advance the device-side chunk index at the end of a chunk step.
__global__ void counter_add_kernel(long long* counter, long long delta) {
  ptx::griddep_wait();
  *counter += delta;
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

}  // namespace

cudaError_t launch_append_bf16(const AppendParams& p, cudaStream_t s) {
  const long long vecs = 2LL * p.B * p.H * p.Lc * (p.D / 8);
  long long blocks = (vecs + kAppendThreads - 1) / kAppendThreads;
  const long long cap = (long long)num_sms() * 8;  // grid-stride beyond 8 CTAs per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(append_bf16_kernel, dim3((unsigned)blocks), p, s);
}

cudaError_t launch_append_fp8(const AppendParams& p, cudaStream_t s) {
  return launch_pdl(append_fp8_kernel, dim3(2, p.B * p.H), p, s);
}

cudaError_t launch_counter_add(long long* counter, long long delta, cudaStream_t s) {
  counter_add_kernel<<<1, 1, 0, s>>>(counter, delta);
  return cudaGetLastError();
}

}  // namespace sab
