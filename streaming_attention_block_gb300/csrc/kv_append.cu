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

// Debug builds: the destination slot lies inside the (b, h) block, on a slot
// boundary, and its scale entry inside the scale row; else the error word
// records it and the caller returns before any load or store (uniform over
// the CTA).
__device__ bool slot_in_bounds(const AppendParams& p, int bh, int slot_row0, int scale_idx) {
  const bool ok = bh < p.B * p.H && p.Lc > 0 && slot_row0 >= 0 && slot_row0 % p.Lc == 0 &&
                  slot_row0 + p.Lc <= p.rows && scale_idx >= 0 && scale_idx < p.scale_stride;
  if (!ok && threadIdx.x == 0 && p.err_word != nullptr) atomicOr(p.err_word, kErrBoundsBit);
  return ok;
}

// One CTA moves kAppendVecs 16-byte vectors of one (tensor, b, h) block:
// the destination block is one contiguous run of Lc * D elements, the source
// rows are D-element runs H * D apart.  Each thread issues all its loads
// before its stores, so every thread keeps kAppendUnroll vectors in flight.
constexpr int kAppendUnroll = 4;
constexpr int kAppendVecs = kAppendThreads * kAppendUnroll;

__global__ void __launch_bounds__(kAppendThreads)
append_bf16_kernel(const __grid_constant__ AppendParams p) {
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();  // the slot may still be read by the previous kernel
  int slot_row0 = p.slot_row0;
  if (p.d_chunk != nullptr) {  // graph mode: the chunk index lives on the device
    const long long c = *p.d_chunk;
    slot_row0 = (p.has_sink + (int)((c < 0 ? 0 : c) % p.ring_slots)) * p.Lc;
  }
  const int tensor = blockIdx.y & 1;
  const int bh = blockIdx.y >> 1;
  const int b = bh / p.H, h = bh - b * p.H;
  if constexpr (kDebugBounds) {
    if (!slot_in_bounds(p, bh, slot_row0, slot_row0 / (p.Lc > 0 ? p.Lc : 1))) return;
  }
  const int lvpr = p.D == 128 ? 4 : 3;  // log2 of the 16-byte vectors per row (D / 8)
  const int nvec = p.Lc << lvpr;
  const uint4* src = reinterpret_cast<const uint4*>(p.src[tensor] + ((long long)b * p.Lc * p.H + h) * p.D);
  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dst[tensor]) +
                                        ((long long)bh * p.rows + slot_row0) * p.D);
  const long long src_row = (long long)p.H * (p.D / 8);  // source row pitch in vectors
  const int i0 = blockIdx.x * kAppendVecs + threadIdx.x;
  uint4 v[kAppendUnroll];
#pragma unroll
  for (int k = 0; k < kAppendUnroll; ++k) {
    const int i = i0 + k * kAppendThreads;
    if (i < nvec) v[k] = __ldg(src + (i >> lvpr) * src_row + (i & ((1 << lvpr) - 1)));
  }
#pragma unroll
  for (int k = 0; k < kAppendUnroll; ++k) {
    const int i = i0 + k * kAppendThreads;
    if (i < nvec) dst[i] = v[k];
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
  if constexpr (kDebugBounds) {
    if (!slot_in_bounds(p, bh, slot_row0, scale_idx) || scale_idx * p.Lc != slot_row0) return;
  }
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

// 8-bit append with one cluster of kQCluster CTAs per (tensor, b, h) block:
// each CTA loads its share of the block into registers (NV 16-byte vectors a
// thread), the partial absmax values meet through distributed shared memory,
// and every CTA quantises the values it holds with the common scale -- the
// block is read from HBM once and the grid is kQCluster times wider than one
// CTA per block.  Same arithmetic as append_fp8_kernel (scale = amax / 448 or
// / 127 by IEEE division, codes of x / scale).
constexpr int kQCluster = 8;

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

template <int NV>
__global__ void __launch_bounds__(kAppendThreads)
append_q_cluster_kernel(const __grid_constant__ AppendParams p) {
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();  // the slot may still be read by the previous kernel
  const int tensor = blockIdx.y & 1;
  const int bh = blockIdx.y >> 1;
  const bool int8 = p.k_int8 && tensor == 0;  // uniform over the cluster
  int slot_row0 = p.slot_row0, scale_idx = p.scale_idx;
  if (p.d_chunk != nullptr) {  // graph mode: the chunk index lives on the device
    const long long c = *p.d_chunk;
    const int slot = (int)((c < 0 ? 0 : c) % p.ring_slots);
    slot_row0 = (p.has_sink + slot) * p.Lc;
    scale_idx = p.has_sink + slot;
  }
  if constexpr (kDebugBounds) {  // uniform over the cluster: all of it returns, before any barrier
    if (!slot_in_bounds(p, bh, slot_row0, scale_idx) || scale_idx * p.Lc != slot_row0) return;
  }
  const int b = bh / p.H, h = bh - b * p.H;
  const uint32_t rank = ptx::cluster_ctarank();
  const int lvpr = p.D == 128 ? 4 : 3;  // log2 of the 16-byte vectors per row
  const int nvec = p.Lc << lvpr;
  const int per = (nvec + kQCluster - 1) / kQCluster;
  const int v0 = (int)rank * per, v1 = min(nvec, v0 + per);
  const uint4* src = reinterpret_cast<const uint4*>(p.src[tensor] + ((long long)b * p.Lc * p.H + h) * p.D);
  const long long src_row = (long long)p.H * (p.D / 8);
  uint4 x[NV];
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = v0 + (int)threadIdx.x + k * kAppendThreads;
    if (i < v1) {
      x[k] = __ldg(src + (i >> lvpr) * src_row + (i & ((1 << lvpr) - 1)));
      const uint32_t w[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[kAppendThreads / 32];
  __shared__ float s_part, s_scale;
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int w = 0; w < kAppendThreads / 32; ++w) m = fmaxf(m, red[w]);
    s_part = m;
  }
  ptx::cluster_sync_all();  // every CTA's partial absmax is visible to the cluster
  if (threadIdx.x < 32) {
    float m = threadIdx.x < kQCluster ? ld_cluster_f32(ptx::mapa(ptx::smem_u32(&s_part), threadIdx.x)) : 0.f;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) {
      const float sc = (m == 0.f) ? 1.0f : __fdiv_rn(m, int8 ? 127.0f : 448.0f);
      s_scale = sc;
      if (rank == 0) p.scale[tensor][(long long)bh * p.scale_stride + scale_idx] = sc;
    }
  }
  __syncthreads();
  // the peers' partials have been read: a CTA may leave once all have arrived
  ptx::cluster_arrive_relaxed();
  const float sc = s_scale;
  uint8_t* dst = static_cast<uint8_t*>(p.dst[tensor]) + ((long long)bh * p.rows + slot_row0) * p.D;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = v0 + (int)threadIdx.x + k * kAppendThreads;
    if (i < v1) {
      const uint32_t w[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
      uint32_t out[2];
      if (int8) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
          out[q] = s8_code(__fdiv_rn(bf16_lo(w[2 * q]), sc)) | (s8_code(__fdiv_rn(bf16_hi(w[2 * q]), sc)) << 8) |
                   (s8_code(__fdiv_rn(bf16_lo(w[2 * q + 1]), sc)) << 16) |
                   (s8_code(__fdiv_rn(bf16_hi(w[2 * q + 1]), sc)) << 24);
      } else {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint16_t c0 = e4m3x2(__fdiv_rn(bf16_lo(w[2 * q]), sc), __fdiv_rn(bf16_hi(w[2 * q]), sc));
          const uint16_t c1 = e4m3x2(__fdiv_rn(bf16_lo(w[2 * q + 1]), sc), __fdiv_rn(bf16_hi(w[2 * q + 1]), sc));
          out[q] = (uint32_t)c0 | ((uint32_t)c1 << 16);
        }
      }
      reinterpret_cast<uint2*>(dst)[i] = make_uint2(out[0], out[1]);  // vector i = 8 codes at byte 8 i
    }
  }
  ptx::cluster_wait();
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
  const long long vecs = (long long)p.Lc * (p.D / 8);  // per (tensor, b, h) block
  const long long gx = (vecs + kAppendVecs - 1) / kAppendVecs;
  const long long gy = 2LL * p.B * p.H;
  if ((p.D != 64 && p.D != 128) || gx > 0x7fffffffLL || gy > 65535) return cudaErrorInvalidValue;
  return launch_pdl(append_bf16_kernel, dim3((unsigned)gx, (unsigned)gy), p, s);
}

template <int NV>
cudaError_t launch_q_cluster(const AppendParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kQCluster, 2 * p.B * p.H, 1);
  cfg.blockDim = dim3(kAppendThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kQCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, append_q_cluster_kernel<NV>, p);
}

cudaError_t launch_append_fp8(const AppendParams& p, cudaStream_t s) {
  // vectors a thread holds when a cluster shares one (tensor, b, h) block
  const long long per = ((long long)p.Lc * (p.D / 8) + kQCluster - 1) / kQCluster;
  const long long nv = (per + kAppendThreads - 1) / kAppendThreads;
  if ((p.D == 64 || p.D == 128) && 2LL * p.B * p.H <= 65535) {
    if (nv <= 2) return launch_q_cluster<2>(p, s);
    if (nv <= 4) return launch_q_cluster<4>(p, s);
    if (nv <= 8) return launch_q_cluster<8>(p, s);
    if (nv <= 16) return launch_q_cluster<16>(p, s);
  }
  // larger blocks: one CTA per block, the block re-read from L2 for the codes
  return launch_pdl(append_fp8_kernel, dim3(2, p.B * p.H), p, s);
}

cudaError_t launch_counter_add(long long* counter, long long delta, cudaStream_t s) {
  counter_add_kernel<<<1, 1, 0, s>>>(counter, delta);
  return cudaGetLastError();
}

}  // namespace sab
