// Fused Q/K RMSNorm + rotary embedding producer for one chunk, optionally
// writing the chunk's K and V straight into the ring slot (BF16 ring).
//
// "WorldPlay2: Extending Real-Time Interactive World Models in Control and
// Horizon", section 方法步骤详情 (inference: QKRoPE and QKV fusion) and
// "Matrix-Game 4.0: Harnessing Video Models for Real-Time Playable Game
// Worlds", section 实验结果 (a fused RoPE kernel) name the step; the formulas
// are the plain ones of a Wan-style video DiT:
//   RMSNorm over each token's H*D vector: y = x * rsqrt(mean(x^2) + eps) * gamma
//   rotary embedding per head on interleaved pairs (2i, 2i+1): three bands of
//   the head dimension (frame, row, column of the chunk's latent grid), each
//   rotated by pos * base^(-2i / band).
// One warp per token: a lane holds the same 8 head dimensions of every head
// (D / 8 divides 32 for D = 64, 128), so it computes the sine and cosine of
// its 4 pairs once and reuses them for all heads and for both q and k.
// Reads Q, K, V and writes Q', K', V once each: an HBM stream.
#include <math.h>

#include "ptx.cuh"
#include "sab_internal.h"

namespace sab {
namespace {

constexpr int kRopeWarps = 2;  // tokens per CTA (small CTAs spread a chunk over every SM)

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int VPL>
__global__ void __launch_bounds__(32 * kRopeWarps)
qk_rope_kernel(const __grid_constant__ RopeParams p) {
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  const int lane = threadIdx.x & 31;
  if constexpr (kDebugBounds) {
    // the appended chunk's ring rows lie inside each (b, h) block, on a slot
    // boundary; checked by the whole CTA before any load or store
    if (p.ring_k != nullptr &&
        !(p.Lc > 0 && p.slot_row0 >= 0 && p.slot_row0 % p.Lc == 0 && p.slot_row0 + p.Lc <= p.rows)) {
      if (threadIdx.x == 0 && p.err_word != nullptr) atomicOr(p.err_word, kErrBoundsBit);
      return;
    }
  }
  const long long tok = (long long)blockIdx.x * kRopeWarps + (threadIdx.x >> 5);  // b * Lc + t
  if (tok >= (long long)p.B * p.Lc) return;
  const int t = (int)(tok % p.Lc);
  const int b = (int)(tok / p.Lc);
  const int HD = p.H * p.D;
  const int nvec = HD / 8;  // 16-byte vectors per token and tensor

  // rotation of this lane's 4 pairs (head dimensions d0 .. d0 + 7)
  const int d0 = (lane * 8) % p.D;
  const float pos_f = (float)(p.chunk * p.F + t / (p.Hp * p.Wp));
  const float pos_h = (float)((t / p.Wp) % p.Hp), pos_w = (float)(t % p.Wp);
  float cs[4], sn[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int d = d0 + 2 * k;  // even dimension of the pair
    float pos = pos_f;
    int i = d / 2, band = p.bt;
    if (d >= p.bt + p.bh) {
      pos = pos_w; i = (d - p.bt - p.bh) / 2; band = p.bw;
    } else if (d >= p.bt) {
      pos = pos_h; i = (d - p.bt) / 2; band = p.bh;
    }
    const float theta = exp2f(-2.0f * (float)i / (float)band * p.log2_base);
    sincosf(pos * theta, &sn[k], &cs[k]);
  }

  const uint4* q4 = reinterpret_cast<const uint4*>(p.q_in + tok * HD);
  const uint4* k4 = reinterpret_cast<const uint4*>(p.k_in + tok * HD);
  const uint4* v4 = reinterpret_cast<const uint4*>(p.v_in + tok * HD);
  // VPL > 0: the token's q, k, v vectors of this lane stay in registers (one
  // HBM round trip); VPL == 0: any H*D, second pass re-reads q, k from L1
  constexpr int kR = VPL > 0 ? VPL : 1;
  uint4 qa[kR], ka[kR], va[kR];
  float sq = 0.f, sk = 0.f;
  auto sumsq = [&](const uint4& a, float& acc) {
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) acc = fmaf(bf_lo(wa[j]), bf_lo(wa[j]), fmaf(bf_hi(wa[j]), bf_hi(wa[j]), acc));
  };
  if constexpr (VPL > 0) {
#pragma unroll
    for (int r = 0; r < VPL; ++r) {
      qa[r] = q4[lane + 32 * r];
      ka[r] = k4[lane + 32 * r];
      va[r] = v4[lane + 32 * r];
    }
#pragma unroll
    for (int r = 0; r < VPL; ++r) {
      sumsq(qa[r], sq);
      sumsq(ka[r], sk);
    }
  } else {
    for (int v = lane; v < nvec; v += 32) {
      sumsq(q4[v], sq);
      sumsq(k4[v], sk);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sq += __shfl_xor_sync(0xffffffffu, sq, o);
    sk += __shfl_xor_sync(0xffffffffu, sk, o);
  }
  const float rq = rsqrtf(sq / (float)HD + p.eps), rk = rsqrtf(sk / (float)HD + p.eps);

  auto emit = [&](int v, const uint4& a, const uint4& c, const uint4& vv) {
    const int e = v * 8, h = e / p.D, d = e - h * p.D;  // d == d0
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wc[4] = {c.x, c.y, c.z, c.w};
    float gq[8], gk[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      gq[j] = p.gamma_q ? __ldg(p.gamma_q + e + j) : 1.f;
      gk[j] = p.gamma_k ? __ldg(p.gamma_k + e + j) : 1.f;
    }
    uint32_t oq[4], ok[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float q0 = bf_lo(wa[k]) * rq * gq[2 * k], q1 = bf_hi(wa[k]) * rq * gq[2 * k + 1];
      const float k0 = bf_lo(wc[k]) * rk * gk[2 * k], k1 = bf_hi(wc[k]) * rk * gk[2 * k + 1];
      oq[k] = ptx::pack_bf16(q0 * cs[k] - q1 * sn[k], q0 * sn[k] + q1 * cs[k]);
      ok[k] = ptx::pack_bf16(k0 * cs[k] - k1 * sn[k], k0 * sn[k] + k1 * cs[k]);
    }
    const uint4 vq = make_uint4(oq[0], oq[1], oq[2], oq[3]), vk = make_uint4(ok[0], ok[1], ok[2], ok[3]);
    reinterpret_cast<uint4*>(p.q_out + tok * HD)[v] = vq;
    if (p.k_out) reinterpret_cast<uint4*>(p.k_out + tok * HD)[v] = vk;
    if (p.v_out) reinterpret_cast<uint4*>(p.v_out + tok * HD)[v] = vv;
    if (p.ring_k) {  // head-major ring rows [B, H, rows, D]
      const long long row = ((long long)b * p.H + h) * p.rows + p.slot_row0 + t;
      reinterpret_cast<uint4*>(p.ring_k + row * p.D + d)[0] = vk;
      reinterpret_cast<uint4*>(p.ring_v + row * p.D + d)[0] = vv;
    }
  };
  if constexpr (VPL > 0) {
#pragma unroll
    for (int r = 0; r < VPL; ++r) emit(lane + 32 * r, qa[r], ka[r], va[r]);
  } else {
    for (int v = lane; v < nvec; v += 32) emit(v, q4[v], k4[v], v4[v]);
  }
}

}  // namespace

cudaError_t launch_qk_rope(const RopeParams& p, cudaStream_t s) {
  const long long tokens = (long long)p.B * p.Lc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((tokens + kRopeWarps - 1) / kRopeWarps), 1, 1);
  cfg.blockDim = dim3(32 * kRopeWarps, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch ((p.H * p.D) / 256 * ((p.H * p.D) % 256 == 0)) {  // 16-byte vectors per lane
    case 2: return cudaLaunchKernelEx(&cfg, qk_rope_kernel<2>, p);
    case 4: return cudaLaunchKernelEx(&cfg, qk_rope_kernel<4>, p);
    case 6: return cudaLaunchKernelEx(&cfg, qk_rope_kernel<6>, p);
    default: return cudaLaunchKernelEx(&cfg, qk_rope_kernel<0>, p);  // larger H*D: two passes
  }
}

}  // namespace sab
