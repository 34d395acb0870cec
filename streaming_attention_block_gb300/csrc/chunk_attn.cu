// Chunk attention over a ring KV cache (streaming) or a whole sequence
// (block-causal), for sm_103a: TMA tile loads, tcgen05 MMAs with TMEM
// accumulators, online softmax in registers, split-KV with an in-kernel
// log-sum-exp merge.
//
// What it computes (see include/sab.h): for every query row i of a (b, h)
// and its visible key set J, O_i = softmax_j(scale * q_i.k_j) V and
// LSE_i = ln sum_j exp(scale * q_i.k_j).  Visibility follows the block-causal
// chunk rule of "WanToFight: Real-Time Generative Game Engine for
// Multi-Player Combat Interaction" (section 三, table "模型组件", row
// "Block-Causal Attention"): bidirectional inside a chunk, causal over the W
// previous chunks, plus an optional sink ("Matrix-Game 4.0: Harnessing Video
// Models for Real-Time Playable Game Worlds", section "前置知识 / 因果自回归与
// KV 缓存").  The mask is never materialised: in streaming mode every key the
// host planner hands over is visible and only the ragged end of a key run is
// masked; in block-causal mode each row derives its key interval from its
// chunk index.
//
// One forward kernel, chunk_attn_kh_kernel (below): one CTA = one tile of
// 128 query rows x one (b, h) x one KV split; each 128-key tile's scores are
// handled by two softmax warpgroups, one per 64-key half, double-buffered S
// in TMEM.  With more than one split, each split writes its normalised
// partial rows and LSE to the workspace and the last split of a query tile
// to finish (atomic ticket) merges them by log-sum-exp ("Matrix-Game 4.0",
// section "技术新颖性": KV window intervals computed in parallel and merged
// with log-sum-exp).  Further down: the backward kernels.
//
// Every mbarrier wait is bounded: on expiry the kernel records the wait site
// in a device error word, raises a CTA-wide abort flag, drains its own TMA
// copies and MMAs (again with bounded waits), frees TMEM and returns.
#include <math.h>

#include <mutex>

#include "ptx.cuh"
#include "sab_internal.h"

namespace sab {

__device__ unsigned int g_sab_error_word = 0;

namespace {

using namespace ptx;

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per pipeline wait
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8
// E4M3 P: by > 2^5.75, so that P' = P * 2^3 * vs / vs_ref <= 2^8.75 ~ 430.5
// stays below the largest code 448 = 2^8.807
constexpr float kRescaleThresholdF8 = 5.75f;
constexpr int kScaleTab = 64;  // per-chunk coefficient table entries (1 KB of shared memory)

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded mbarrier wait.  try_wait already suspends the thread in hardware
// until the phase completes (or a short system limit passes), so the loop
// spins without sleeping -- a sleep would delay the wake-up of this
// latency-critical pipeline.  Every 256 polls it checks the CTA abort flag and
// the elapsed time; after kTimeoutNs it records the wait site, raises the
// abort flag and gives up.
template <bool kClusterScope = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned site, uint64_t timeout_ns = kTimeoutNs) {
  if (!kClusterScope && mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
#pragma unroll 1
  for (uint32_t it = 1;; ++it) {
    if (kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > timeout_ns) {
        atomicOr(&g_sab_error_word, 1u << site);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Bounded wait used while draining after an abort (ignores the abort flag).
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
#pragma unroll 1
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kTimeoutNs) {
      atomicOr(&g_sab_error_word, 1u << 31);
      return;
    }
  }
}

struct Tile {
  int src;    // tensor-map index
  int row;    // first key row of the tile in the map's row axis
  int valid;  // keys of the run inside this tile (streaming); 128 otherwise
};

__device__ __forceinline__ Tile stream_tile(const KeyPlan& kp, int g) {
  int s = 0;
#pragma unroll
  for (int i = 1; i < kMaxSegments; ++i)
    if (i < kp.nseg && g >= kp.seg[i].tile0) s = i;
  const int t = g - kp.seg[s].tile0;
  Tile ti;
  ti.src = kp.seg[s].src;
  ti.row = kp.seg[s].row0 + t * kTileN;
  ti.valid = min(kTileN, kp.seg[s].nrows - t * kTileN);
  return ti;
}

__device__ __forceinline__ Tile tile_at(const AttnParams& p, const KeyPlan& kp, int g) {
  if (p.mode != kModeBlockCausal) return stream_tile(kp, g);
  Tile ti;
  ti.src = 0;
  ti.row = g * kTileN;
  ti.valid = kTileN;
  return ti;
}

// KV tiles of this CTA: [first, first + count).
__device__ __forceinline__ void kv_range(const AttnParams& p, const KeyPlan& kp, int q0, int qrows, int split,
                                         int& first, int& count) {
  int total = 0, base = 0;
  if (p.mode != kModeBlockCausal) {
    total = kp.total_tiles;
  } else {
    const int q_last = min(p.Lq, q0 + qrows) - 1;
    if (q_last >= q0) {
      const int c_lo = q0 / p.chunk_tokens, c_hi = q_last / p.chunk_tokens;
      const int klo = max(0, c_lo - p.window) * p.chunk_tokens;
      const int khi = min(p.Lk, (c_hi + 1) * p.chunk_tokens);
      base = klo / kTileN;
      total = (khi + kTileN - 1) / kTileN - base;
    }
  }
  const long long a = (long long)total * split / p.splits;
  const long long e = (long long)total * (split + 1) / p.splits;
  first = base + (int)a;
  count = (int)(e - a);
}

// Debug builds: every global index a forward CTA will form, checked before it
// issues any copy or store.  Uniform over the CTA (it depends on the launch
// parameters, the block index and the key plan only).
__device__ bool attn_indices_ok(const AttnParams& p, const KeyPlan& kp, int b, int q0, int split, int first,
                                int n_tiles) {
  if (b >= p.B || q0 >= p.Lq || (int)blockIdx.x >= p.n_qtiles || split >= p.splits) return false;
  if (first < 0 || n_tiles < 0) return false;
  for (int g = first; g < first + n_tiles; ++g) {
    const Tile t = tile_at(p, kp, g);
    if (t.src < 0 || t.src > 1 || (t.src == 1 && !(p.mode == kModeStreaming && p.kcur))) return false;
    if (t.row < 0 || t.row >= p.src_rows[t.src] || t.valid < 1) return false;
    // streaming key runs end inside their source (block-causal tiles may run
    // past the last key: the copy fills zeros and the mask drops them)
    if (p.mode != kModeBlockCausal && t.row + t.valid > p.src_rows[t.src]) return false;
    if (p.fp8 && (t.row + t.valid - 1) / p.chunk_tokens >= p.scale_stride) return false;
  }
  if (p.splits > 1) {
    const long long tile = ((long long)split * p.B * p.H + blockIdx.y) * p.n_qtiles + blockIdx.x;
    if (tile >= p.ws_tiles || (long long)blockIdx.y * p.n_qtiles + blockIdx.x >= (long long)p.B * p.H * p.n_qtiles)
      return false;
  }
  return true;
}

// Key runs of the query rows [q0, q0 + qrows) behind a memory prefix
// ("WorldPlay2", Figure 3 and section 方法步骤详情, training stage 3): the
// first P = mem_len[b] positions are real memory that every real query sees;
// target chunk c (tokens from mem_pad on) also sees target chunks c - W .. c.
// Run 0: the real memory [0, P), when any row of the tile sees it; run 1:
// the union of the target rows' chunk windows.  Padding is in neither.
__device__ __forceinline__ void plan_prefix_runs(const AttnParams& p, int b, int q0, int qrows, KeyPlan& kp) {
  const int M = p.mem_pad;
  const int P = min(max(__ldg(p.mem_len + b), 0), M);
  const int q_last = min(p.Lq, q0 + qrows) - 1;
  const bool any_target = q_last >= M;
  const int nmem = (q0 < P || any_target) ? P : 0;
  int klo = M, khi = M;
  if (any_target) {
    const int c_lo = (max(q0, M) - M) / p.chunk_tokens, c_hi = (q_last - M) / p.chunk_tokens;
    klo = M + max(0, c_lo - p.window) * p.chunk_tokens;
    khi = min(p.Lk, M + (c_hi + 1) * p.chunk_tokens);
  }
  const int t1 = (nmem + kTileN - 1) / kTileN;
  kp.nseg = 2;
  kp.seg[0] = KvSegment{0, 0, nmem, 0};
  kp.seg[1] = KvSegment{0, klo, khi - klo, t1};
#pragma unroll
  for (int i = 2; i < kMaxSegments; ++i) kp.seg[i] = KvSegment{0, 0, 0, 0x7fffffff};
  kp.total_tiles = t1 + (khi - klo + kTileN - 1) / kTileN;
}

// Expand two key/value rows (both K rows or both V rows of one tile) of 128
// 8-bit codes each in place into 128 fp16 values (the operand type of the
// 8-bit-cache path).  The codes sit in the second 128-byte box of a row
// (where its upper 16-bit half goes); every code of both rows is read before
// any fp16 chunk is written (the two rows' shared-memory latencies overlap),
// and the rows are written in the 128-byte-swizzled layout of the MMA
// operands.  A row's 16-byte code chunks are visited from chunk (row mod 8),
// so the eight rows a quarter-warp touches read eight different bank groups
// and write eight different ones through the swizzle.  One conversion
// instruction per pair of E4M3 codes; two integer and two half-precision
// instructions per four INT8 codes.  Exact for every code.
template <bool K8>
__device__ __forceinline__ void expand_code_rows2_f16(uint8_t* tile, int ra, int rb, uint32_t box_bytes) {
  const int rot[2] = {ra & 7, rb & 7};
  const int rr[2] = {ra, rb};
  uint4 raw[2][8];
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const uint8_t* src = tile + box_bytes + rr[w] * 128;
#pragma unroll
    for (int i = 0; i < 8; ++i) raw[w][i] = *reinterpret_cast<const uint4*>(src + (((i + rot[w]) & 7) << 4));
  }
#pragma unroll
  for (int w = 0; w < 2; ++w) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = (i + rot[w]) & 7;  // codes 16c .. 16c + 15
      const uint32_t wd[4] = {raw[w][i].x, raw[w][i].y, raw[w][i].z, raw[w][i].w};
      uint32_t out[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (K8) {
          s8x4_to_f16x4(wd[q], out[2 * q], out[2 * q + 1]);
        } else {
          out[2 * q] = e4m3x2_to_f16x2((uint16_t)(wd[q] & 0xFFFFu));
          out[2 * q + 1] = e4m3x2_to_f16x2((uint16_t)(wd[q] >> 16));
        }
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int k = 2 * c + hh;
        *reinterpret_cast<uint4*>(tile + (k >> 3) * box_bytes + rr[w] * 128 + (((k & 7) ^ rot[w]) << 4)) =
            make_uint4(out[4 * hh], out[4 * hh + 1], out[4 * hh + 2], out[4 * hh + 3]);
      }
    }
  }
}

// ===========================================================================
// Key-half kernel: one CTA = one query tile of 128 rows x one (b, h), no KV
// split.  Each 128-key tile's scores are processed by two softmax
// warpgroups, one per 64-key half; each half keeps its own running max, row
// sum and output accumulator O_h in TMEM (O_0 + O_1 combined by log-sum-exp
// in the epilogue), so the halves never exchange data inside the loop.  S is
// double-buffered in TMEM, so the MMA warp issues S(j+2) right after PV(j),
// while the softmax of tile j+1 runs: the tensor pipe sees PV_0(j), PV_1(j),
// S(j+2) per tile and the softmax has a whole tile period to finish.
//   warp 0        TMA producer (Q once, then stage u holds K(u) and V(u-1):
//                 a stage is released by PV(u-1), which the MMA warp issues
//                 after S(u), and K(u) arrives two tile periods before S(u))
//   warp 1        TMEM allocator, tcgen05 MMA issuer (one elected lane)
//   warps 2-3     E4M3 -> bf16 expansion (FP8 cache only)
//   8 warps       softmax: half h = keys [64h, 64h + 64) of every tile
// TMEM: S/P buffers at columns 0 and 128 (P_h packed bf16 in the first 32
// columns of its half), O_h at column 256 + h * D.
template <int D_, bool FP8_, bool F8MMA_ = false>
struct KhCfg {
  static constexpr int D = D_;
  // F8MMA: E4M3 K/V tiles go to the tensor core as stored (no expansion);
  // Q is quantised per row on chip and P is rounded to E4M3
  // 8-bit cache with 16-bit products: the codes are expanded to fp16 on
  // chip (exact), Q is converted to fp16 with a per-row power-of-two scale
  // (exact) and P is rounded to fp16; kind::f16 products with fp16 operands
  static constexpr bool kConv = FP8_ && !F8MMA_;  // 8-bit -> fp16 expansion warps
  static constexpr int kBoxes = D / 64;
  static constexpr uint32_t kBoxBytes = 128u * 128u;
  static constexpr uint32_t kTileBytes = kBoxBytes * kBoxes;                  // bf16 tile of 128 rows
  static constexpr uint32_t kKVTileBytes = F8MMA_ ? 128u * D : kTileBytes;   // one K or V stage tile
  static constexpr int kStages = F8MMA_ ? 5 : ((D == 128) ? 3 : 4);
  static constexpr uint32_t kKOff = 0;
  static constexpr uint32_t kVOff = kKOff + kStages * kKVTileBytes;
  static constexpr uint32_t kQOff = kVOff + kStages * kKVTileBytes;
  static constexpr uint32_t kQ8Off = kQOff + kTileBytes;                        // E4M3 Q (F8MMA)
  static constexpr uint32_t kQmaxOff = kQ8Off + (F8MMA_ ? 128u * D : 0u);       // 2 x 128 row maxima
  static constexpr uint32_t kBarOff = kQmaxOff + (FP8_ ? 1024u : 0u);
  static constexpr int kBarQ = 0;
  static constexpr int kBarKFull = 1;                         // [kStages]
  static constexpr int kBarKVEmpty = kBarKFull + kStages;     // [kStages]
  static constexpr int kBarRawFull = kBarKVEmpty + kStages;   // [kStages] FP8 codes landed
  static constexpr int kBarSFull = kBarRawFull + kStages;     // [2 buffers]
  static constexpr int kBarPFull = kBarSFull + 2;             // [2 buffers][2 halves]
  static constexpr int kBarPVLast = kBarPFull + 4;            // PV of the last tile but one complete
  static constexpr int kBarOFinal = kBarPVLast + 1;           // every MMA complete
  static constexpr int kBarDrain = kBarOFinal + 1;
  static constexpr int kBarQ8 = kBarDrain + 1;                // 8-bit cache: converted Q written
  static constexpr int kBarMerge = kBarQ8 + 1;                // split merge: partial tiles landed
  static constexpr int kNumBars = kBarMerge + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;
  // 8-bit cache: warps 2 and 3 expand codes, softmax warps 4..11
  static constexpr int kConvThreads = kConv ? 64 : 0;
  static constexpr int kSoftmaxWarp0 = kConv ? 4 : 2;
  static constexpr int kThreads = 32 * (kSoftmaxWarp0 + 8);
  static constexpr uint32_t kTmemO = 256;
  static constexpr uint32_t kTmemCols = 512;
  // epilogue scratch in the dead operand region: (m, l) of every row and
  // half, and the bf16 output tile (Q slot) for the TMA store
  static constexpr uint32_t kXchOff = kKOff;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <int D, bool FP8, bool F8MMA, bool K8>
__global__ void __launch_bounds__(KhCfg<D, FP8, F8MMA>::kThreads, 1)
chunk_attn_kh_kernel(const __grid_constant__ AttnParams p) {
  using C = KhCfg<D, FP8, F8MMA>;
  static_assert(!F8MMA || (FP8 && D == 128), "E4M3 products: 8-bit cache, D = 128");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t sQ = base_u32 + C::kQOff;
  const uint32_t sK = base_u32 + C::kKOff;
  const uint32_t sV = base_u32 + C::kVOff;
  const uint32_t bars = base_u32 + C::kBarOff;
  uint32_t* misc = reinterpret_cast<uint32_t*>(base + C::kMiscOff);  // [0] tmem, [1] abort
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int b = bh / p.H;
  const int h = bh - b * p.H;
  const int q0 = blockIdx.x * kTileM;
  const int split = blockIdx.z;  // KV partition (p.splits of them, merged through the workspace)


  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBarQ), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarKFull + s), C::kConv ? C::kConvThreads : 1);
      mbar_init(bar(C::kBarKVEmpty + s), 1);
      mbar_init(bar(C::kBarRawFull + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::kBarSFull + i), 1);
      mbar_init(bar(C::kBarPFull + 2 * i), 128);
      mbar_init(bar(C::kBarPFull + 2 * i + 1), 128);
    }
    mbar_init(bar(C::kBarPVLast), 1);
    mbar_init(bar(C::kBarOFinal), 1);
    mbar_init(bar(C::kBarDrain), 1);
    mbar_init(bar(C::kBarQ8), 256);
    mbar_init(bar(C::kBarMerge), 1);
    misc[1] = 0;
    misc[2] = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.q_map);
    prefetch_tmap(&p.k_map[0]);
    prefetch_tmap(&p.v_map[0]);
    prefetch_tmap(&p.o_map);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  griddep_launch_dependents();
  griddep_wait();
  // key runs: planned on the host, or (graph mode) by every thread from the
  // chunk index in device memory, read only after the previous grid completed
  KeyPlan kp;
  if (p.mode == kModeStreaming && p.d_chunk != nullptr)
    plan_key_runs(*p.d_chunk, p.window, p.ring_slots, p.chunk_tokens, p.has_sink, p.use_sink, p.kcur, kp);
  else if (p.mode == kModeMemPrefix)
    plan_prefix_runs(p, b, q0, kTileM, kp);
  else
    kp = p.plan;
  int first = 0, n_tiles = 0;
  kv_range(p, kp, q0, kTileM, split, first, n_tiles);
  if constexpr (kDebugBounds) {
    if (!attn_indices_ok(p, kp, b, q0, split, first, n_tiles)) {  // the whole CTA takes this branch
      n_tiles = 0;
      if (threadIdx.x == 0) {
        atomicOr(&g_sab_error_word, kErrBoundsBit);
        *abort_flag = 1;  // every role leaves as after a wait that gave up
      }
      __syncthreads();
    }
  }

  // Roles: softmax warps (and their epilogue); producer, MMA issuer and
  // (8-bit cache) conversion warps.
  if (warp >= C::kSoftmaxWarp0) {
    // ---------------------------------------------- softmax + epilogue
    const int hf = (warp - C::kSoftmaxWarp0) >> 2;  // key half of every tile
    const int quad = warp & 3;                        // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;
    const int q_row = q0 + row;
    const bool row_valid = q_row < p.Lq;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tSh = tmem + lane_off + (uint32_t)hf * 64u;  // + buffer * 128
    const uint32_t tO = tmem + lane_off + C::kTmemO + (uint32_t)hf * D;
    const int kofs = hf * 64;  // first key of this half inside a tile
    // visible keys of this row: block-causal window [klo, khi); behind a
    // memory prefix also the memory run [0, mhi)
    int klo = 0, khi = 0, mhi = 0;
    if (p.mode != kModeStreaming && row_valid) {
      const int tq = q_row - p.mem_pad;  // position among the target tokens
      if (tq >= 0) {
        const int qc = tq / p.chunk_tokens;
        klo = p.mem_pad + max(0, qc - p.window) * p.chunk_tokens;
        khi = min(p.Lk, p.mem_pad + (qc + 1) * p.chunk_tokens);
      }
      if (p.mode == kModeMemPrefix) mhi = (tq >= 0 || q_row < kp.seg[0].nrows) ? kp.seg[0].nrows : 0;
    }
    const float sl = p.scale_log2;
    int seg_tile0[kMaxSegments], seg_rows[kMaxSegments], seg_row0[kMaxSegments];
#pragma unroll
    for (int i = 0; i < kMaxSegments; ++i) {
      seg_tile0[i] = (i < kp.nseg) ? kp.seg[i].tile0 : 0x7fffffff;
      seg_rows[i] = kp.seg[i].nrows;
      seg_row0[i] = kp.seg[i].row0;
    }
    const long long srow = (long long)bh * p.scale_stride;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    // 8-bit cache: this thread converts its half of the row's Q in shared
    // memory before the first product (the two halves of a row agree on the
    // row's absmax through shared memory).
    //  * E4M3 products: Q quantised to E4M3 with one absmax scale per row (as
    //    the cache's quantiser does per chunk; the division in fp32), into a
    //    separate buffer; P is formed as P * (vs / vs_ref) * 2^3 so that the
    //    codes of V are used as stored and P stays out of the subnormals (the
    //    running max lags by at most 2^5.75, so P' <= 2^8.75 < 448).
    //  * 16-bit products: Q converted in place to fp16 times 2^e, with e
    //    chosen per row so that the row's absmax lands in [2^14, 2^15): exact
    //    for every value down to 2^-28 of the row's absmax (and below that an
    //    error under 2^-39 of it); 2^-e goes into the score coefficient.  P is
    //    formed as P * (vs / vs_ref) * 2^6 <= 2^14 (the running max lags by at
    //    most 2^8) and rounded to fp16.
    float slq = sl, vgain = 1.f, ofac = 1.f;
    if constexpr (FP8) {
      ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarQ), 0, abort_flag, 10));
      float* qmax = reinterpret_cast<float*>(base + C::kQmaxOff);
      uint8_t* qrow = base + C::kQOff + hf * C::kBoxBytes + row * 128;  // bf16 columns 64hf ..
      uint4 qv[8];
      float amax = 0.f;
      if (ok) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          qv[c] = *reinterpret_cast<const uint4*>(qrow + ((c ^ (row & 7)) << 4));
          const uint32_t w[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
#pragma unroll
          for (int k = 0; k < 4; ++k)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[k] << 16)), fabsf(__uint_as_float(w[k] & 0xFFFF0000u))));
        }
      }
      qmax[hf * 128 + row] = amax;
      named_bar_sync(1, 256);
      amax = fmaxf(amax, qmax[(1 - hf) * 128 + row]);
      if constexpr (F8MMA) {
        const float qs = amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
        if (ok) {
          uint8_t* q8row = base + C::kQ8Off + row * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {  // 16 codes: bf16 chunks 2i, 2i + 1 of this half
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint4 src = qv[2 * i + (k >> 1)];
              const uint32_t wa = (k & 1) ? src.z : src.x, wb = (k & 1) ? src.w : src.y;
              o[k] = pack_e4m3x2(__fdiv_rn(__uint_as_float(wa << 16), qs),
                                 __fdiv_rn(__uint_as_float(wa & 0xFFFF0000u), qs)) |
                     (pack_e4m3x2(__fdiv_rn(__uint_as_float(wb << 16), qs),
                                  __fdiv_rn(__uint_as_float(wb & 0xFFFF0000u), qs))
                      << 16);
            }
            *reinterpret_cast<uint4*>(q8row + (((4 * hf + i) ^ (row & 7)) << 4)) =
                make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        slq = sl * qs;
      } else {
        int e = 0;
        if (amax > 0.f) e = min(max(14 - ((int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127), -126), 126);
        const float up = __uint_as_float((uint32_t)(127 + e) << 23);    // 2^e
        const float down = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
        if (ok) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // in place: the same 16-byte chunk, bf16 -> fp16
            const uint32_t w[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
              o[k] = pack_f16(__uint_as_float(w[k] << 16) * up, __uint_as_float(w[k] & 0xFFFF0000u) * up);
            *reinterpret_cast<uint4*>(qrow + ((c ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        slq = sl * down;
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(C::kBarQ8));
      // largest V scale over the chunks of the key runs
      float vmax = 0.f;
#pragma unroll 1
      for (int i = 0; i < kp.nseg; ++i) {
        if (kp.seg[i].nrows <= 0) continue;
        const int c_hi = min((kp.seg[i].row0 + kp.seg[i].nrows - 1) / p.chunk_tokens, p.scale_stride - 1);
#pragma unroll 1
        for (int c = kp.seg[i].row0 / p.chunk_tokens; c <= c_hi; ++c) vmax = fmaxf(vmax, __ldg(p.v_scale + srow + c));
      }
      const float vref = vmax > 0.f ? vmax : 1.f;
      constexpr float kGain = F8MMA ? 8.f : 64.f;
      vgain = __fdiv_rn(kGain, vref);
      ofac = vref * (1.f / kGain);
      // The per-chunk coefficients of this (b, h) go to a shared table (over
      // the row maxima, dead now) so that no tile waits on a global load:
      // {K scale, V scale * gain, log2 of it, its reciprocal}
      if (p.scale_stride <= kScaleTab) {
        named_bar_sync(1, 256);  // every thread has read the row maxima
        float4* tab = reinterpret_cast<float4*>(base + C::kQmaxOff);
        const int t = hf * 128 + row;
        if (t < p.scale_stride) {
          const float ks = __ldg(p.k_scale + srow + t), vs = __ldg(p.v_scale + srow + t);
          const float v = vs * vgain;
          tab[t] = make_float4(ks, v, vs > 0.f ? __log2f(v) : 0.f, vs > 0.f ? 1.f / v : 0.f);
        }
        named_bar_sync(1, 256);
      }
    }
    int rec_si = 0, rec_end = 0;  // 8-bit cache: lane L's record of tile 32 * (j / 32) + L
    for (int j = 0; ok && j < n_tiles; ++j) {
      ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarSFull + (j & 1)), (uint32_t)(j >> 1) & 1u,
                                                abort_flag, 6 + hf));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tSh + (uint32_t)(j & 1) * 128u;
      uint32_t s0[32], s1[32];
      tmem_ld32(tS + 0, s0);
      tmem_ld32(tS + 32, s1);  // both loads in flight while the key range is worked out
      int lo, hi;
      int tile_row0 = 0;
      const int g = first + j;
      // key run of plan tile gg: its index, first plan tile, rows and first row
      auto seg_of = [&](int gg, int& sg, int& t0, int& nr, int& r0) {
        sg = 0;
#pragma unroll
        for (int i = 1; i < kMaxSegments; ++i) sg = (gg >= seg_tile0[i]) ? i : sg;
        t0 = seg_tile0[0], nr = seg_rows[0], r0 = seg_row0[0];
#pragma unroll
        for (int i = 1; i < kMaxSegments; ++i) {
          t0 = (sg == i) ? seg_tile0[i] : t0;
          nr = (sg == i) ? seg_rows[i] : nr;
          r0 = (sg == i) ? seg_row0[i] : r0;
        }
      };
      if (p.mode != kModeBlockCausal) {
        int sg, t0, nr, r0;
        seg_of(g, sg, t0, nr, r0);
        tile_row0 = r0 + (g - t0) * kTileN;
        if (p.mode == kModeStreaming) {
          lo = 0;
          hi = nr - (g - t0) * kTileN;
        } else {  // memory run, then the chunk window
          lo = (sg == 0 ? 0 : klo) - tile_row0;
          hi = (sg == 0 ? mhi : khi) - tile_row0;
        }
      } else {
        lo = klo - g * kTileN;
        hi = khi - g * kTileN;
      }
      lo -= kofs;
      hi -= kofs;
      // FP8 cache: the tile's keys belong to at most two chunks; columns of
      // this half before `bnd` to the first, the rest to the next
      float c0 = slq, c1 = slq, d0 = 0.f, v0 = 1.f, v1 = 1.f, iv0 = 1.f;
      int bnd = 64;
      if constexpr (FP8) {
        if ((j & 31) == 0) {
          // lane L works out the first chunk of tile j + L and where it ends
          // (rows from the tile's first), once for the next 32 tiles
          int sg, t0, nr, r0;
          seg_of(g + lane, sg, t0, nr, r0);
          const int tr = r0 + (g + lane - t0) * kTileN;
          rec_si = min(tr / p.chunk_tokens, p.scale_stride - 1);
          rec_end = (rec_si + 1) * p.chunk_tokens - tr;
        }
        const int si0 = __shfl_sync(0xffffffffu, rec_si, j & 31);
        const int si1 = min(si0 + 1, p.scale_stride - 1);
        bnd = __shfl_sync(0xffffffffu, rec_end, j & 31) - kofs;
        // the half's keys before `bnd` belong to chunk si0, the rest to si1
        float4 e0, e1;
        if (p.scale_stride <= kScaleTab) {
          const float4* tab = reinterpret_cast<const float4*>(base + C::kQmaxOff);
          e0 = tab[bnd <= 0 ? si1 : si0];  // the whole half in the second chunk
          e1 = tab[si1];
        } else {
          const int a = bnd <= 0 ? si1 : si0;
          const float ks0 = __ldg(p.k_scale + srow + a), ks1 = __ldg(p.k_scale + srow + si1);
          const float vs0 = __ldg(p.v_scale + srow + a), vs1 = __ldg(p.v_scale + srow + si1);
          e0 = make_float4(ks0, vs0 * vgain, vs0 > 0.f ? __log2f(vs0 * vgain) : 0.f, vs0 > 0.f ? 1.f / (vs0 * vgain) : 0.f);
          e1 = make_float4(ks1, vs1 * vgain, 0.f, 0.f);
        }
        // a zero scale marks a slot never written, whose keys are all masked:
        // keep the coefficients finite and non-zero so that -inf stays -inf
        c0 = e0.x > 0.f ? slq * e0.x : slq;
        c1 = e1.x > 0.f ? slq * e1.x : slq;
        v0 = e0.y;  // V scale times the P gain of the 8-bit paths
        v1 = e1.y;
        d0 = e0.z;
        iv0 = e0.w;
      }
      const bool straddle = FP8 && bnd > 0 && bnd < 64;
      const bool masked = !(lo <= 0 && hi >= 64);
      // per-column scaling (straddling FP8 tile) and masking of 32 columns
      // starting at column cb of this half
      auto prep = [&](uint32_t (&sv)[32], int cb) {
        if (straddle) {
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[c] = __float_as_uint(__uint_as_float(sv[c]) * (cb + c < bnd ? c0 : c1));
        }
        if (masked) {
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[c] = (cb + c >= lo && cb + c < hi) ? sv[c] : 0xff800000u;
        }
      };
      auto max32 = [&](const uint32_t (&sv)[32]) -> float {
        float pm[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float m = fmax3(__uint_as_float(sv[k]), __uint_as_float(sv[k + 4]), __uint_as_float(sv[k + 8]));
          m = fmax3(m, __uint_as_float(sv[k + 12]), __uint_as_float(sv[k + 16]));
          m = fmax3(m, __uint_as_float(sv[k + 20]), __uint_as_float(sv[k + 24]));
          pm[k] = fmaxf(m, __uint_as_float(sv[k + 28]));
        }
        return fmax3(fmaxf(pm[0], pm[1]), pm[2], pm[3]);
      };
      // P of 32 columns: e = 2^(s*xa + xs); packed bf16 pairs into pko[0..15]
      // (E4M3 products: four codes a word into pko[0..7]), row-sum terms into
      // ps (before any per-column V scale)
      auto exps32 = [&](const uint32_t (&sv)[32], int cb, float xa, float xs, uint32_t* pko, float2& ps) {
        const float2 xa2 = make_float2(xa, xa), xs2 = make_float2(xs, xs);
        uint32_t lo16 = 0;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), xa2, xs2);
          float e0 = ex2(x.x), e1 = ex2(x.y);
          ps = __fadd2_rn(ps, make_float2(e0, e1));
          if (straddle) {
            e0 *= (cb + 2 * c < bnd ? v0 : v1);
            e1 *= (cb + 2 * c + 1 < bnd ? v0 : v1);
          }
          if constexpr (F8MMA) {
            const uint32_t h2 = pack_e4m3x2(e0, e1);
            if (c & 1) pko[c >> 1] = lo16 | (h2 << 16);
            else lo16 = h2;
          } else if constexpr (C::kConv) {
            pko[c] = pack_f16(e0, e1);
          } else {
            pko[c] = pack_bf16(e0, e1);
          }
        }
      };
      // 16-bit P: exponentials are taken against the running max m_run right
      // away, in parallel with the row max; only when the max grows by more
      // than the rescale threshold (always on a row's first visible tile) are
      // they recomputed against the new max, with O and l rescaled.  E4M3 P:
      // the narrow range makes rescales frequent (a warp rescales when any of
      // its 32 rows does), so the max comes first and the exponentials are
      // taken once.
      constexpr bool kSpeculate = !F8MMA;
      const float mb0 = (m_run == -INFINITY) ? 0.f : m_run;
      const float xa = straddle ? 1.f : c0;
      uint32_t pk[32];
      float2 psa = make_float2(0.f, 0.f), psb = make_float2(0.f, 0.f);
      tmem_wait_ld();
      prep(s0, 0);
      const float mx0 = max32(s0);
      if constexpr (kSpeculate) exps32(s0, 0, xa, straddle ? -mb0 : d0 - mb0, pk, psa);
      prep(s1, 32);
      const float mx1 = max32(s1);
      if constexpr (kSpeculate) exps32(s1, 32, xa, straddle ? -mb0 : d0 - mb0, pk + 16, psb);
      const float mx = fmaxf(mx0, mx1);
      const float m_new = fmaxf(m_run, straddle ? mx : mx * c0);
      const bool need = m_new > m_run + (F8MMA ? kRescaleThresholdF8 : kRescaleThreshold);
      if (__any_sync(0xffffffffu, need)) {
        float alpha = 1.f;
        if (need) {
          alpha = ex2(m_run - m_new);  // 0 when m_run is -inf
          l_run *= alpha;
          m_run = m_new;
        }
        if (j > 0) {
          // O_hf holds PV_hf(j-1) only once that MMA group has completed:
          // S(j+1) was issued after it (one tensor pipe, in order), and for
          // the last tile a commit follows PV(j-1) itself
          const uint32_t wb = j + 1 < n_tiles ? bar(C::kBarSFull + ((j + 1) & 1)) : bar(C::kBarPVLast);
          const uint32_t wp = j + 1 < n_tiles ? (uint32_t)((j + 1) >> 1) & 1u : 0u;
          ok = __all_sync(0xffffffffu, wait_bounded(wb, wp, abort_flag, 8 + hf));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 32) {
            uint32_t o[32];
            tmem_ld32(tO + cc, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(tO + cc, o);
          }
        }
        if constexpr (kSpeculate) {
          const float mb = (m_run == -INFINITY) ? 0.f : m_run;
          psa = psb = make_float2(0.f, 0.f);
          exps32(s0, 0, xa, straddle ? -mb : d0 - mb, pk, psa);
          exps32(s1, 32, xa, straddle ? -mb : d0 - mb, pk + 16, psb);
        }
      }
      if constexpr (!kSpeculate) {
        const float mb = (m_run == -INFINITY) ? 0.f : m_run;
        exps32(s0, 0, xa, straddle ? -mb : d0 - mb, pk, psa);
        exps32(s1, 32, xa, straddle ? -mb : d0 - mb, pk + 8, psb);
      }
      if constexpr (F8MMA) tmem_st16(tS, *reinterpret_cast<const uint32_t(*)[16]>(pk));
      else tmem_st32(tS, pk);
      l_run += ((psa.x + psa.y) + (psb.x + psb.y)) * (straddle ? 1.f : iv0);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::kBarPFull + 2 * (j & 1) + hf));
    }
    // ------------------------------------------------------------ epilogue
    // (the other half's softmax may still be a tile behind, so completion is
    // read from the single-phase final barrier, not from the per-tile ones)
    if (ok) ok = wait_bounded(bar(C::kBarOFinal), 0, abort_flag, 8);
    // a completed barrier does not clear an abort raised elsewhere in the CTA
    // (another role's wait, or a failed index check): nothing is stored then
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    // every MMA is complete: the operand region is free.  Exchange (m, l) of
    // the two halves of each row, then each half finishes D/2 columns.
    float2* xch = reinterpret_cast<float2*>(base + C::kXchOff);
    xch[hf * 128 + row] = make_float2(m_run, l_run);
    named_bar_sync(1, 256);
    const float2 other = xch[(1 - hf) * 128 + row];
    const float m0 = hf == 0 ? m_run : other.x, l0 = hf == 0 ? l_run : other.y;
    const float m1 = hf == 0 ? other.x : m_run, l1 = hf == 0 ? other.y : l_run;
    const float M = fmaxf(m0, m1);
    const float w0 = (M == -INFINITY) ? 0.f : ex2(m0 - M);
    const float w1 = (M == -INFINITY) ? 0.f : ex2(m1 - M);
    const float L = l0 * w0 + l1 * w1;
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const float sc0 = w0 * inv * ofac, sc1 = w1 * inv * ofac;  // ofac undoes the 8-bit paths' P gain
    constexpr int kHalfCols = D / 2;
    uint8_t* stage = base + C::kQOff;
    if (ok) {
      tc_fence_after();
      uint32_t oa[kHalfCols], ob[kHalfCols];
      if (n_tiles > 0) {
        const uint32_t tO0 = tmem + lane_off + C::kTmemO + (uint32_t)(hf * kHalfCols);
#pragma unroll
        for (int cc = 0; cc < kHalfCols; cc += 32) {
          tmem_ld32(tO0 + cc, *reinterpret_cast<uint32_t(*)[32]>(oa + cc));
          tmem_ld32(tO0 + D + cc, *reinterpret_cast<uint32_t(*)[32]>(ob + cc));
        }
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int c = 0; c < kHalfCols; ++c) oa[c] = ob[c] = 0u;
      }
      const float lse = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
      if (p.splits == 1) {
#pragma unroll
        for (int i = 0; i < kHalfCols / 8; ++i) {
          float v[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            v[c] = fmaf(__uint_as_float(oa[8 * i + c]), sc0, __uint_as_float(ob[8 * i + c]) * sc1);
          uint4 w;
          w.x = pack_bf16(v[0], v[1]);
          w.y = pack_bf16(v[2], v[3]);
          w.z = pack_bf16(v[4], v[5]);
          w.w = pack_bf16(v[6], v[7]);
          const int k = hf * (kHalfCols / 8) + i;  // 16-byte chunk of the output row
          *reinterpret_cast<uint4*>(stage + (k >> 3) * C::kBoxBytes + row * 128 + (((k & 7) ^ (row & 7)) << 4)) = w;
        }
        if (hf == 0 && row_valid && p.LSE != nullptr) p.LSE[(long long)bh * p.Lq + q_row] = lse;
      } else {
        // this split's normalised partial tile (fp32) and its LSEs go to the
        // workspace: a tile is 128 x D floats stored as [D / 4][128 rows]
        // float4s, so the 32 rows of a warp write 512 contiguous bytes
        const long long tile = ((long long)split * p.B * p.H + bh) * p.n_qtiles + blockIdx.x;
        float4* dst = reinterpret_cast<float4*>(p.ws_o) + tile * (kTileM * D / 4) + hf * (kHalfCols / 4) * kTileM + row;
#pragma unroll
        for (int i = 0; i < kHalfCols / 4; ++i)
          __stcg(dst + i * kTileM,
                 make_float4(fmaf(__uint_as_float(oa[4 * i]), sc0, __uint_as_float(ob[4 * i]) * sc1),
                             fmaf(__uint_as_float(oa[4 * i + 1]), sc0, __uint_as_float(ob[4 * i + 1]) * sc1),
                             fmaf(__uint_as_float(oa[4 * i + 2]), sc0, __uint_as_float(ob[4 * i + 2]) * sc1),
                             fmaf(__uint_as_float(oa[4 * i + 3]), sc0, __uint_as_float(ob[4 * i + 3]) * sc1)));
        if (hf == 0) __stcg(p.ws_lse + tile * kTileM + row, lse);
        fence_proxy_async_global();  // the merging CTA reads the partials with bulk copies
      }
    }
    bool store = p.splits == 1;
    if (p.splits > 1) {
      // ------------------------------ log-sum-exp merge of the KV splits
      // ("Matrix-Game 4.0", section 技术新颖性: window intervals computed in
      // parallel, merged by log-sum-exp).  Every split of the query tile
      // arrives on its counter, also one that gave up on a wait: the low 16
      // bits count arrivals, the high 16 bits aborts.  The last arriver resets
      // the counter (the workspace stays usable after a reported timeout) and,
      // if no split aborted, merges the partial rows and stores the tile.
      __threadfence();
      fence_proxy_async_smem();  // the operand region may be overwritten by bulk copies below
      named_bar_sync(1, 256);
      volatile uint32_t* ticket = misc + 2;
      if (warp == C::kSoftmaxWarp0 && lane == 0) {
        unsigned* cnt = &p.ws_count[(long long)bh * p.n_qtiles + blockIdx.x];
        if (split + 1 == p.inject_abort) {  // self-test: behave as a split whose wait gave up
          atomicOr(&g_sab_error_word, kErrInjectedAbortBit);
          *abort_flag = 1;
        }
        const bool aborted = *abort_flag != 0;
        const unsigned old = atomicAdd(cnt, aborted ? 0x10001u : 1u);
        const bool last = (old & 0xFFFFu) == (unsigned)(p.splits - 1);
        if (last) *cnt = 0u;
        *ticket = (last && !aborted && (old >> 16) == 0u) ? 1u : 0u;
      }
      named_bar_sync(1, 256);
      store = *ticket == 1u;
      if (store) {
        __threadfence();
        fence_proxy_async_global();
        // partial tiles of this query tile: split sp at tile index t0 + sp * tstride
        const long long tstride = (long long)p.B * p.H * p.n_qtiles;
        const long long t0 = (long long)bh * p.n_qtiles + blockIdx.x;
        auto lse_of = [&](int sp) { return __ldcg(p.ws_lse + (t0 + sp * tstride) * kTileM + row); };
        float Mx = -INFINITY;
        for (int s8 = 0; s8 < p.splits; s8 += 8) {  // eight loads in flight
          float l8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) l8[k] = s8 + k < p.splits ? lse_of(s8 + k) : -INFINITY;
#pragma unroll
          for (int k = 0; k < 8; ++k) Mx = fmaxf(Mx, l8[k]);
        }
        float tot = 0.f;
        if (Mx != -INFINITY) {
          for (int s8 = 0; s8 < p.splits; s8 += 8) {
            float l8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) l8[k] = s8 + k < p.splits ? lse_of(s8 + k) : -INFINITY;
#pragma unroll
            for (int k = 0; k < 8; ++k) tot += l8[k] == -INFINITY ? 0.f : ex2((l8[k] - Mx) * kLog2e);
          }
        }
        const float Lm = (Mx == -INFINITY) ? -INFINITY : Mx + __logf(tot);
        float acc[kHalfCols];
#pragma unroll
        for (int c = 0; c < kHalfCols; ++c) acc[c] = 0.f;
        // The partial tiles come into the (dead) K/V stage region by bulk
        // copies, as many at a time as it holds; each thread then reads its
        // row's half from shared memory (a warp's 32 rows: 512 contiguous bytes).
        constexpr uint32_t kPartBytes = kTileM * D * 4;
        constexpr int kBatch = (int)((2u * C::kStages * C::kKVTileBytes) / kPartBytes);
        static_assert(kBatch >= 1, "one partial tile fits in the operand region");
        const bool leader = warp == C::kSoftmaxWarp0 && lane == 0;
        bool got = true;
        int batch = 0;
        for (int b0 = 0; got && b0 < p.splits; b0 += kBatch, ++batch) {
          const int nb = min(kBatch, p.splits - b0);
          if (leader) {
            mbar_arrive_expect_tx(bar(C::kBarMerge), (uint32_t)nb * kPartBytes);
            for (int k = 0; k < nb; ++k)
              bulk_copy_g2s(base_u32 + C::kKOff + (uint32_t)k * kPartBytes,
                            reinterpret_cast<const float4*>(p.ws_o) + (t0 + (b0 + k) * tstride) * (kTileM * D / 4),
                            kPartBytes, bar(C::kBarMerge));
          }
          float lb[kBatch];
#pragma unroll
          for (int k = 0; k < kBatch; ++k) lb[k] = k < nb ? lse_of(b0 + k) : -INFINITY;
          got = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarMerge), (uint32_t)batch & 1u, abort_flag, 13));
          if (got) {
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
              if (k >= nb || lb[k] == -INFINITY || Lm == -INFINITY) continue;
              const float wgt = ex2((lb[k] - Lm) * kLog2e);
              const float4* src = reinterpret_cast<const float4*>(base + C::kKOff + k * kPartBytes) +
                                  hf * (kHalfCols / 4) * kTileM + row;
#pragma unroll
              for (int i = 0; i < kHalfCols / 4; ++i) {
                const float4 x = src[i * kTileM];
                acc[4 * i] = fmaf(wgt, x.x, acc[4 * i]);
                acc[4 * i + 1] = fmaf(wgt, x.y, acc[4 * i + 1]);
                acc[4 * i + 2] = fmaf(wgt, x.z, acc[4 * i + 2]);
                acc[4 * i + 3] = fmaf(wgt, x.w, acc[4 * i + 3]);
              }
            }
          }
          named_bar_sync(1, 256);  // the batch is read before the next one lands
        }
        if (!got) {
          // a bulk copy did not land in time: drain it before the CTA exits
          if (leader) wait_drain(bar(C::kBarMerge), (uint32_t)(batch - 1) & 1u);
          store = false;
        }
#pragma unroll
        for (int i = 0; i < kHalfCols / 8; ++i) {
          uint4 w;
          w.x = pack_bf16(acc[8 * i + 0], acc[8 * i + 1]);
          w.y = pack_bf16(acc[8 * i + 2], acc[8 * i + 3]);
          w.z = pack_bf16(acc[8 * i + 4], acc[8 * i + 5]);
          w.w = pack_bf16(acc[8 * i + 6], acc[8 * i + 7]);
          const int k = hf * (kHalfCols / 8) + i;
          *reinterpret_cast<uint4*>(stage + (k >> 3) * C::kBoxBytes + row * 128 + (((k & 7) ^ (row & 7)) << 4)) = w;
        }
        if (hf == 0 && row_valid && p.LSE != nullptr) p.LSE[(long long)bh * p.Lq + q_row] = Lm;
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 256);
    if (store && warp == C::kSoftmaxWarp0 && lane == 0 && !*abort_flag) {
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx)
        tma_store_4d(&p.o_map, base_u32 + C::kQOff + bx * C::kBoxBytes, bx * 64, q0, h, b);
      tma_store_commit_and_wait_read();
    }
  } else {
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::kBarQ), C::kTileBytes);
  #pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_4d(sQ + bx * C::kBoxBytes, &p.q_map, bar(C::kBarQ), bx * 64, q0, h, b);
        int u = 0;
        for (; u <= n_tiles && n_tiles > 0; ++u) {
          const int st = u % C::kStages;
          if (u >= C::kStages &&
              !wait_bounded(bar(C::kBarKVEmpty + st), (uint32_t)(u / C::kStages - 1) & 1u, abort_flag, 0))
            break;
          // the first product's operands (Q, K(0)) land before the later
          // stages are requested
          if (!FP8 && u == 1 && !wait_bounded(bar(C::kBarKFull + 0), 0, abort_flag, 0)) break;
          const bool has_k = u < n_tiles, has_v = u > 0;
          const Tile tk = tile_at(p, kp, first + (has_k ? u : u - 1));
          const Tile tv = tile_at(p, kp, first + (has_v ? u - 1 : u));
          if constexpr (F8MMA) {  // E4M3 code tiles, used by the MMA as stored
            mbar_arrive_expect_tx(bar(C::kBarKFull + st),
                                  (has_k ? C::kKVTileBytes : 0u) + (has_v ? C::kKVTileBytes : 0u));
            if (has_k)
              tma_load_4d(sK + st * C::kKVTileBytes, &p.k_map[0], bar(C::kBarKFull + st), 0, tk.row, h, b);
            if (has_v)
              tma_load_4d(sV + st * C::kKVTileBytes, &p.v_map[0], bar(C::kBarKFull + st), 0, tv.row, h, b);
          } else if (FP8) {
            mbar_arrive_expect_tx(bar(C::kBarRawFull + st), (has_k ? 128 * D : 0) + (has_v ? 128 * D : 0));
            if (has_k)
              tma_load_4d(sK + st * C::kTileBytes + C::kBoxBytes, &p.k_map[0], bar(C::kBarRawFull + st), 0, tk.row,
                          h, b);
            if (has_v)
              tma_load_4d(sV + st * C::kTileBytes + C::kBoxBytes, &p.v_map[0], bar(C::kBarRawFull + st), 0, tv.row,
                          h, b);
          } else {
            mbar_arrive_expect_tx(bar(C::kBarKFull + st), (has_k ? C::kTileBytes : 0) + (has_v ? C::kTileBytes : 0));
            if (has_k) {
  #pragma unroll
              for (int bx = 0; bx < C::kBoxes; ++bx)
                tma_load_4d(sK + st * C::kTileBytes + bx * C::kBoxBytes, &p.k_map[tk.src], bar(C::kBarKFull + st),
                            bx * 64, tk.row, h, b);
            }
            if (has_v) {
  #pragma unroll
              for (int bx = 0; bx < C::kBoxes; ++bx)
                tma_load_4d(sV + st * C::kTileBytes + bx * C::kBoxBytes, &p.v_map[tv.src], bar(C::kBarKFull + st),
                            bx * 64, tv.row, h, b);
            }
          }
        }
        if (*abort_flag) {
          wait_drain(bar(C::kBarQ), 0);
          for (int uu = max(0, u - C::kStages); uu < u; ++uu)
            wait_drain(bar((C::kConv ? C::kBarRawFull : C::kBarKFull) + uu % C::kStages),
                       (uint32_t)(uu / C::kStages) & 1u);
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc_qk = F8MMA ? idesc_e4m3_f32(128, kTileN, 0)
                                          : (C::kConv ? idesc_f16_f32(128, kTileN, 0) : idesc_bf16_f32(128, kTileN, 0));
      constexpr uint32_t idesc_pv = F8MMA ? idesc_e4m3_f32(128, D, 1)
                                          : (C::kConv ? idesc_f16_f32(128, D, 1) : idesc_bf16_f32(128, D, 1));
      // 8-bit cache: the A operand is the converted Q the softmax warps write
      bool ok = __all_sync(0xffffffffu, wait_bounded(bar(FP8 ? C::kBarQ8 : C::kBarQ), 0, abort_flag, 1));
      if (ok) tc_fence_after();
      const uint64_t dq = smem_desc_sw128(F8MMA ? base_u32 + C::kQ8Off : sQ, 16, 1024);
      const uint64_t dk = smem_desc_sw128(sK, 16, 1024);
      const uint64_t dv = smem_desc_sw128(sV, C::kBoxBytes, 1024);
      const uint32_t q_lo = (uint32_t)dq, k_lo = (uint32_t)dk, v_lo = (uint32_t)dv;
      const uint32_t kq_hi = (uint32_t)(dq >> 32), v_hi = (uint32_t)(dv >> 32);
      constexpr uint32_t kTileStep = C::kKVTileBytes >> 4;
      // As in the two-tile kernel, the barrier needed next is probed without
      // blocking in the middle of the preceding MMA group.
      auto issue_s = [&](int j, uint32_t pb, uint32_t pp, bool& pout) {
        const uint32_t d = tmem + (uint32_t)(j & 1) * 128u;
        const uint32_t b0 = k_lo + (uint32_t)(j % C::kStages) * kTileStep;
        if constexpr (F8MMA) {  // 128-byte code rows: K = 32 codes (32 bytes) a step
  #pragma unroll
          for (int kk = 0; kk < D / 32; ++kk) {
            const uint32_t koff = (uint32_t)(kk * 32) >> 4;
            mma_ss_f8_e(d, make_desc(q_lo + koff, kq_hi), make_desc(b0 + koff, kq_hi), idesc_qk, kk > 0 ? 1u : 0u);
            if (kk == D / 64 && pb != 0) pout = mbar_test_wait(pb, pp);
          }
        } else {
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
            mma_ss_e(d, make_desc(q_lo + koff, kq_hi), make_desc(b0 + koff, kq_hi), idesc_qk, kk > 0 ? 1u : 0u);
            if (kk == D / 32 && pb != 0) pout = mbar_test_wait(pb, pp);
          }
        }
      };
      // O_hf += P_hf V[64 hf .. 64 hf + 63]
      auto issue_pv = [&](int j, int hf, uint32_t pb, uint32_t pp, bool& pout) {
        const uint32_t d = tmem + C::kTmemO + (uint32_t)hf * D;
        const uint32_t b0 = v_lo + (uint32_t)((j + 1) % C::kStages) * kTileStep;
        const uint32_t a0 = tmem + (uint32_t)(j & 1) * 128u + (uint32_t)hf * 64u;
        if constexpr (F8MMA) {  // P_hf: 64 E4M3 keys in 16 columns, 32 keys (8 columns) a step
  #pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const int kr = hf * 64 + kk * 32;  // first key row of the step
            mma_ts_f8_e(d, a0 + kk * 8, make_desc(b0 + ((kr * 128) >> 4), v_hi), idesc_pv,
                        (kk > 0 || j > 0) ? 1u : 0u);
            if (kk == 0 && pb != 0) pout = mbar_test_wait(pb, pp);
          }
        } else {
  #pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int kg = hf * 4 + kk;  // group of 16 keys
            mma_ts_e(d, a0 + kk * 8, make_desc(b0 + ((kg * 16 * 128) >> 4), v_hi), idesc_pv,
                     (kk > 0 || j > 0) ? 1u : 0u);
            if (kk == 1 && pb != 0) pout = mbar_test_wait(pb, pp);
          }
        }
      };
      auto wait_probed = [&](uint32_t bb, uint32_t par, bool probed, unsigned site) -> bool {
        if (probed) return true;
        return __all_sync(0xffffffffu, wait_bounded(bb, par, abort_flag, site));
      };
      auto kbar = [&](int j) { return bar(C::kBarKFull + j % C::kStages); };
      auto kpar = [&](int j) { return (uint32_t)(j / C::kStages) & 1u; };
      auto pbar = [&](int j, int hf) { return bar(C::kBarPFull + 2 * (j & 1) + hf); };
      auto ppar = [&](int j) { return (uint32_t)(j >> 1) & 1u; };
      bool pr = false;
      // prologue: S(0), S(1)
      for (int j = 0; ok && j < 2 && j < n_tiles; ++j) {
        if (!(ok = wait_probed(kbar(j), kpar(j), pr, 5))) break;
        tc_fence_after();
        pr = false;
        if (j + 1 < 2 && j + 1 < n_tiles) issue_s(j, kbar(j + 1), kpar(j + 1), pr);
        else issue_s(j, pbar(0, 0), ppar(0), pr);
        mma_commit_e(bar(C::kBarSFull + (j & 1)));
        if (j == 0) mma_commit_e(bar(C::kBarKVEmpty + 0));  // stage 0 holds K(0) only
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        // V(j) sits in stage j + 1 with K(j + 1): already waited for before
        // S(j + 1), except after the last tile
        if (j + 1 >= n_tiles && !(ok = wait_probed(kbar(j + 1), kpar(j + 1), false, 5))) break;
        if (!(ok = wait_probed(pbar(j, 0), ppar(j), pr, 2))) break;
        tc_fence_after();
        pr = false;
        issue_pv(j, 0, pbar(j, 1), ppar(j), pr);
        if (!(ok = wait_probed(pbar(j, 1), ppar(j), pr, 3))) break;
        tc_fence_after();
        pr = false;
        if (j + 2 < n_tiles) issue_pv(j, 1, kbar(j + 2), kpar(j + 2), pr);
        else issue_pv(j, 1, 0u, 0u, pr);
        // the softmax of the last tile learns from this that O holds every
        // earlier tile (other tiles learn it from the next tile's S)
        if (j + 2 == n_tiles) mma_commit_e(bar(C::kBarPVLast));
        // stage j + 1 (K(j + 1), V(j)) is free once PV(j) completes: S(j + 1)
        // was issued before it
        mma_commit_e(bar(C::kBarKVEmpty + (j + 1) % C::kStages));
        if (j + 2 < n_tiles) {
          if (!(ok = wait_probed(kbar(j + 2), kpar(j + 2), pr, 5))) break;
          tc_fence_after();
          pr = false;
          issue_s(j + 2, pbar(j + 1, 0), ppar(j + 1), pr);
          mma_commit_e(bar(C::kBarSFull + (j & 1)));
        } else {
          pr = false;
        }
      }
      if (ok) mma_commit_e(bar(C::kBarOFinal));
      if (!ok) {
        mma_commit_e(bar(C::kBarDrain));
        if (lane == 0) wait_drain(bar(C::kBarDrain), 0);
      }
      __syncwarp();
    } else if (C::kConv) {
      // ----------------------------------------- 8-bit -> fp16 expansion
      const int ct = threadIdx.x - 64;
      for (int u = 0; u <= n_tiles && n_tiles > 0; ++u) {
        const int st = u % C::kStages;
        if (!wait_bounded(bar(C::kBarRawFull + st), (uint32_t)(u / C::kStages) & 1u, abort_flag, 12)) break;
        const int job0 = u < n_tiles ? 0 : kTileN, job1 = u > 0 ? 2 * kTileN : kTileN;  // K rows, then V rows
        // rows job and job + 64 of the same tensor (the job range is a
        // multiple of 128 long)
  #pragma unroll 1
        for (int job = job0 + ct; job < job1; job += 2 * C::kConvThreads) {
          const int r = job & (kTileN - 1);
          const bool isv = job >= kTileN;
          uint8_t* tile = base + (isv ? C::kVOff : C::kKOff) + st * C::kTileBytes;
          if (K8 && !isv) expand_code_rows2_f16<true>(tile, r, r + C::kConvThreads, C::kBoxBytes);  // INT8 keys
          else expand_code_rows2_f16<false>(tile, r, r + C::kConvThreads, C::kBoxBytes);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(C::kBarKFull + st));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool FP8, bool F8MMA = false, bool K8 = false>
cudaError_t launch_kh_impl(const AttnParams& p, cudaStream_t s) {
  using C = KhCfg<D, FP8, F8MMA>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(chunk_attn_kh_kernel<D, FP8, F8MMA, K8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_qtiles, p.B * p.H, p.splits);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chunk_attn_kh_kernel<D, FP8, F8MMA, K8>, p);
}

// ===========================================================================
// Backward of block-causal attention ("WanToFight", section 训练流程 / Stage 2:
// training with the block-causal mask).  With P = softmax(scale * Q K^T) over
// the visible keys (recomputed from the forward's LSE), delta_i = sum_d dO O:
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - delta),
//   dK = scale * dS^T Q,  dQ = scale * dS K.
// Two kernels with the pipeline of the forward: the key-tile kernel keeps K,
// V of 128 keys resident and streams the visible query tiles (S^T = K Q^T and
// dP^T = V dO^T into TMEM; the softmax warps write P^T and dS^T back as bf16;
// dV += P^T dO and dK += dS^T Q read them from TMEM); the query-tile kernel
// keeps Q, dO resident and streams the visible key tiles (S, dP; dS back to
// TMEM; dQ += dS K).  Every MMA operand layout is one the forward uses.
template <int D_>
struct BwdCfg {
  static constexpr int D = D_;
  static constexpr int kBoxes = D / 64;
  static constexpr uint32_t kBoxBytes = 128u * 128u;
  static constexpr uint32_t kTileBytes = kBoxBytes * kBoxes;
  static constexpr int kStages = 2;
  static constexpr uint32_t kR0Off = 0;                   // resident tile 0 (K, or Q)
  static constexpr uint32_t kR1Off = kTileBytes;          // resident tile 1 (V, or dO)
  static constexpr uint32_t kStageOff = 2 * kTileBytes;
  // stage: streamed tile 0 (Q_j, or K_j), streamed tile 1 (dO_j, or V_j), then
  // 128 fp32 lse * log2(e) and 128 fp32 delta of the stage's queries
  static constexpr uint32_t kStageBytes = 2 * kTileBytes + 1024;
  static constexpr uint32_t kBarOff = kStageOff + kStages * kStageBytes;
  static constexpr int kBarRes = 0;
  // a stage fills and frees per 64-row half of the streamed tiles: half h of
  // a stage is read by S_h, dP_h and the accumulations of half h only
  static constexpr int kBarFull = 1;                          // [kStages][2 halves]
  static constexpr int kBarEmpty = kBarFull + 2 * kStages;    // [kStages][2 halves]
  static constexpr int kBarSFull = kBarEmpty + 2 * kStages;   // [2 halves]
  static constexpr int kBarPFull = kBarSFull + 2;         // [2 halves]
  static constexpr int kBarFinal = kBarPFull + 2;
  static constexpr int kBarDrain = kBarFinal + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;
  static constexpr int kThreads = 320;                    // producer, MMA, 8 softmax warps
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// delta = rowsum(dO * O) per (b, h, token): one warp per token, D / 8 lanes per head
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __grid_constant__ BwdParams p) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const long long tok = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (tok >= (long long)p.B * p.L) return;
  const int b = (int)(tok / p.L), t = (int)(tok % p.L);
  const int HD = p.H * p.D, lph = p.D / 8;  // lanes per head
  const uint4* o4 = reinterpret_cast<const uint4*>(p.O + tok * HD);
  const uint4* d4 = reinterpret_cast<const uint4*>(p.dO + tok * HD);
  for (int v0 = 0; v0 < HD / 8; v0 += 32) {
    const int v = v0 + lane;
    float acc = 0.f;
    if (v < HD / 8) {
      const uint4 a = o4[v], c = d4[v];
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wc[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        acc = fmaf(__uint_as_float(wa[j] << 16), __uint_as_float(wc[j] << 16),
                   fmaf(__uint_as_float(wa[j] & 0xFFFF0000u), __uint_as_float(wc[j] & 0xFFFF0000u), acc));
    }
    for (int o = lph >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    const int h = (v * 8) / p.D;
    if (v < HD / 8 && (lane % lph) == 0) p.delta[((long long)b * p.H + h) * p.L + t] = acc;
  }
}

// Streamed tiles of a resident tile of rows [r0, r0 + 128): run 0 = n0
// tiles from row 0 (the real memory [0, P) behind a memory prefix), run 1 =
// n1 tiles from row1.  Query i sees key j iff both are real memory, or i is
// a target token and j real memory, or both are target tokens with
// 0 <= chunk(i) - chunk(j) <= window (target chunks counted from mem_pad;
// mem_pad = P = 0 is plain block-causal attention).
struct BwdRuns {
  int n0, row1, n1;
};
template <bool KQ>
__device__ __forceinline__ BwdRuns bwd_runs(const BwdParams& p, int P, int r0) {
  const int M = p.mem_pad, Lc = p.chunk_tokens;
  const int r_last = min(p.L, r0 + kTileM) - 1;
  const bool any_target = r_last >= M;
  const int c_lo = (max(r0, M) - M) / Lc, c_hi = (r_last - M) / Lc;  // target chunks of the tile
  BwdRuns u{0, M, 0};
  int lo = M, hi = M;
  if (KQ) {  // keys: the queries that see them
    if (r0 < P) {
      u.n0 = (P + kTileM - 1) / kTileM;
      hi = p.L;  // every target query sees the real memory
    } else if (any_target) {
      lo = M + c_lo * Lc;
      hi = min(p.L, M + (c_hi + p.window + 1) * Lc);
    }
  } else {   // queries: the keys they see
    if (r0 < P || any_target) u.n0 = (P + kTileN - 1) / kTileN;
    if (any_target) {
      lo = M + max(0, c_lo - p.window) * Lc;
      hi = min(p.L, M + (c_hi + 1) * Lc);
    }
  }
  u.row1 = lo;
  u.n1 = (hi - lo + kTileN - 1) / kTileN;
  return u;
}

// KQ == true: key-tile kernel (dK, dV); false: query-tile kernel (dQ).
template <int D, bool KQ>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
attn_bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t bars = base_u32 + C::kBarOff;
  uint32_t* misc = reinterpret_cast<uint32_t*>(base + C::kMiscOff);  // [0] tmem, [1] abort
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y, b = bh / p.H, h = bh - b * p.H;
  const int r0 = blockIdx.x * 128;  // first row of the resident tile (keys, or queries)

  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBarRes), 1);
    for (int s = 0; s < C::kStages; ++s) {
      for (int hh = 0; hh < 2; ++hh) {
        mbar_init(bar(C::kBarFull + 2 * s + hh), KQ ? 2 : 1);  // key-tile kernel: copies + LSE/delta
        mbar_init(bar(C::kBarEmpty + 2 * s + hh), 1);
      }
    }
    mbar_init(bar(C::kBarSFull + 0), 1);
    mbar_init(bar(C::kBarSFull + 1), 1);
    mbar_init(bar(C::kBarPFull + 0), 128);
    mbar_init(bar(C::kBarPFull + 1), 128);
    mbar_init(bar(C::kBarFinal), 1);
    mbar_init(bar(C::kBarDrain), 1);
    misc[1] = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  griddep_launch_dependents();
  griddep_wait();
  const int P = p.mem_pad > 0 ? min(max(__ldg(p.mem_len + b), 0), p.mem_pad) : 0;  // real memory
  const BwdRuns u = bwd_runs<KQ>(p, P, r0);
  int nt = u.n0 + u.n1;  // streamed tiles
  auto tile_row = [&](int j) { return j < u.n0 ? j * 128 : u.row1 + (j - u.n0) * 128; };
  if constexpr (kDebugBounds) {
    // the resident tile and every streamed tile start inside [0, L) of an
    // existing (b, h); checked by the whole CTA before any copy or store
    bool in = b < p.B && r0 < p.L && u.n0 >= 0 && u.n1 >= 0;
    for (int j = 0; in && j < nt; ++j) in = tile_row(j) >= 0 && tile_row(j) < p.L;
    if (!in) {
      nt = 0;
      if (threadIdx.x == 0) {
        atomicOr(&g_sab_error_word, kErrBoundsBit);
        *abort_flag = 1;
      }
      __syncthreads();
    }
  }
  // resident: K, V (key-tile kernel) or Q, dO (query-tile kernel);
  // streamed: Q_j, dO_j or K_j, V_j
  const CUtensorMap* res0 = KQ ? &p.k_map : &p.q_map;
  const CUtensorMap* res1 = KQ ? &p.v_map : &p.do_map;
  const CUtensorMap* str0 = KQ ? &p.q_map : &p.k_map;
  const CUtensorMap* str1 = KQ ? &p.do_map : &p.v_map;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::kBarRes), 2 * C::kTileBytes);
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        tma_load_4d(base_u32 + C::kR0Off + bx * C::kBoxBytes, res0, bar(C::kBarRes), bx * 64, r0, h, b);
        tma_load_4d(base_u32 + C::kR1Off + bx * C::kBoxBytes, res1, bar(C::kBarRes), bx * 64, r0, h, b);
      }
    }
    // key-tile kernel: the 128 LSE * log2(e) and delta values of a streamed
    // tile are loaded into registers (four of each per lane) one tile ahead,
    // so their global-memory latency passes while the producer waits for a
    // free stage; they go to the stage after its tile copies are issued
    float lsr[4], dlr[4];
    auto load_lse = [&](int jj) {
      const int row = tile_row(jj);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int q = row + lane + 32 * i;
        const bool in = q < p.L;
        lsr[i] = in ? -__ldg(p.LSE + (long long)bh * p.L + q) * kLog2e : -INFINITY;  // stored negated
        dlr[i] = in ? -__ldg(p.delta + (long long)bh * p.L + q) : 0.f;
      }
    };
    if (KQ && nt > 0) load_lse(0);
    // streamed rows come in 64-row halves (their own tensor maps), each as
    // soon as the same half of the stage is free
    const CUtensorMap* str0h = KQ ? &p.q_map_h : &p.k_map_h;
    const CUtensorMap* str1h = KQ ? &p.do_map_h : &p.v_map_h;
    int nh = 0;  // half-stage loads issued
    bool ok = true;
    for (int j = 0; ok && j < nt; ++j) {
      const int st = j % C::kStages;
      const uint32_t so = C::kStageOff + st * C::kStageBytes;
      const int row = tile_row(j);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t fb = bar(C::kBarFull + 2 * st + hh);
        if (j >= C::kStages)
          ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarEmpty + 2 * st + hh),
                                                    (uint32_t)(j / C::kStages - 1) & 1u, abort_flag, 0));
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, 2u * C::kBoxes * (C::kBoxBytes / 2));
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx) {
            const uint32_t off = so + bx * C::kBoxBytes + hh * (C::kBoxBytes / 2);
            tma_load_4d(base_u32 + off, str0h, fb, bx * 64, row + 64 * hh, h, b);
            tma_load_4d(base_u32 + off + C::kTileBytes, str1h, fb, bx * 64, row + 64 * hh, h, b);
          }
        }
        if (KQ) {
          float* ls = reinterpret_cast<float*>(base + so + 2 * C::kTileBytes);
          float* dl = ls + 128;
#pragma unroll
          for (int i = 2 * hh; i < 2 * hh + 2; ++i) {
            ls[lane + 32 * i] = lsr[i];
            dl[lane + 32 * i] = dlr[i];
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(fb);  // second arrival: the half's LSE and delta
        }
        ++nh;
        __syncwarp();
      }
      if (KQ && ok && j + 1 < nt) load_lse(j + 1);
    }
    if (lane == 0 && *abort_flag) {
      wait_drain(bar(C::kBarRes), 0);
      for (int k = max(0, nh - 2 * C::kStages); k < nh; ++k)
        wait_drain(bar(C::kBarFull + 2 * ((k >> 1) % C::kStages) + (k & 1)), (uint32_t)((k >> 1) / C::kStages) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The streamed tile is taken in two halves of 64 rows, each with its own
    // TMEM buffer (columns 128h .. 128h + 127: scores in the first 64, dP in
    // the next 64), so the gradient products of one half and the scores of
    // the next tile's same half run while the other half's softmax works.
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, 0);   // scores: N = 64 rows of a streamed half
    constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, 1);  // accumulators: B MN-major, N = D
    constexpr uint32_t kStageStep = C::kStageBytes >> 4;
    bool ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarRes), 0, abort_flag, 1));
    if (ok) tc_fence_after();
    const uint64_t dr0 = smem_desc_sw128(base_u32 + C::kR0Off, 16, 1024);
    const uint64_t dr1 = smem_desc_sw128(base_u32 + C::kR1Off, 16, 1024);
    const uint64_t ds0 = smem_desc_sw128(base_u32 + C::kStageOff, 16, 1024);
    const uint64_t ds1 = smem_desc_sw128(base_u32 + C::kStageOff + C::kTileBytes, 16, 1024);
    const uint64_t dm0 = smem_desc_sw128(base_u32 + C::kStageOff, C::kBoxBytes, 1024);  // streamed tile 0, MN-major
    const uint64_t dm1 = smem_desc_sw128(base_u32 + C::kStageOff + C::kTileBytes, C::kBoxBytes, 1024);
    const uint32_t hi_k = (uint32_t)(dr0 >> 32), hi_mn = (uint32_t)(dm0 >> 32);
    // scores of the resident tile against rows [64h, 64h + 64) of a streamed
    // tile: d = A_res . B_str^T (the half starts 64 rows = 8 KB into each box)
    auto scores = [&](uint32_t d, uint64_t a, uint64_t bdesc, uint32_t st, int h) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
        mma_ss_e(d, make_desc((uint32_t)a + koff, hi_k),
                 make_desc((uint32_t)bdesc + st * kStageStep + (uint32_t)h * ((64u * 128u) >> 4) + koff, hi_k),
                 idesc_s, kk > 0 ? 1u : 0u);
      }
    };
    // acc += X_h . rows [64h, 64h + 64) of a streamed tile (X_h: bf16 rows
    // of 64 written to TMEM from column a_col; the streamed tile as the
    // MN-major B operand, K = 64)
    auto accum = [&](uint32_t d, uint32_t a_col, uint64_t bmn, uint32_t st, int h, bool first) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_ts_e(d, tmem + a_col + kk * 8,
                 make_desc((uint32_t)bmn + st * kStageStep + (((64 * h + 16 * kk) * 128) >> 4), hi_mn), idesc_acc,
                 (first && kk == 0) ? 0u : 1u);
      }
    };
    auto issue_scores = [&](int j, int h) {
      const uint32_t st = (uint32_t)(j % C::kStages);
      scores(tmem + 128u * h, dr0, ds0, st, h);        // S^T = K Q^T  (or S = Q K^T)
      scores(tmem + 128u * h + 64u, dr1, ds1, st, h);  // dP^T = V dO^T (or dP = dO V^T)
      mma_commit_e(bar(C::kBarSFull + h));
    };
    auto issue_accum = [&](int j, int h) {
      const uint32_t st = (uint32_t)(j % C::kStages);
      const bool first = j == 0 && h == 0;
      if (KQ) {
        accum(tmem + 256, 128u * h, dm1, st, h, first);           // dV += P^T dO
        accum(tmem + 256 + D, 128u * h + 64u, dm0, st, h, first);  // dK += dS^T Q
      } else {
        accum(tmem + 256, 128u * h, dm0, st, h, first);           // dQ += dS K
      }
    };
    auto wait_full = [&](int j, int hh) -> bool {
      const bool r = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarFull + 2 * (j % C::kStages) + hh),
                                                          (uint32_t)(j / C::kStages) & 1u, abort_flag, 5));
      if (r) tc_fence_after();
      return r;
    };
    // order: S_0(0), S_1(0), then per tile j: G_0(j), S_0(j+1), G_1(j), S_1(j+1)
    if (ok && nt > 0 && (ok = wait_full(0, 0))) {
      issue_scores(0, 0);
      if ((ok = wait_full(0, 1))) issue_scores(0, 1);
    }
    for (int j = 0; ok && j < nt; ++j) {
      const int st = j % C::kStages;
      if (!(ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarPFull + 0), (uint32_t)j & 1u, abort_flag, 2))))
        break;
      tc_fence_after();
      issue_accum(j, 0);
      mma_commit_e(bar(C::kBarEmpty + 2 * st + 0));  // half 0 of tile j's stage is read for the last time
      if (j + 1 < nt) {
        if (!(ok = wait_full(j + 1, 0))) break;
        issue_scores(j + 1, 0);
      }
      if (!(ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarPFull + 1), (uint32_t)j & 1u, abort_flag, 3))))
        break;
      tc_fence_after();
      issue_accum(j, 1);
      mma_commit_e(bar(C::kBarEmpty + 2 * st + 1));
      if (j + 1 < nt) {
        if (!(ok = wait_full(j + 1, 1))) break;
        issue_scores(j + 1, 1);
      }
    }
    if (ok) mma_commit_e(bar(C::kBarFinal));
    if (!ok) {
      mma_commit_e(bar(C::kBarDrain));
      if (lane == 0) wait_drain(bar(C::kBarDrain), 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------- probabilities + epilogue
    const int hf = (warp - 2) >> 2;  // half of the streamed tile's 128 rows
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // row of the resident tile
    const int r = r0 + row;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + hf * 128, tdP = tS + 64;  // this half's buffer
    // visible streamed rows of this resident row: [lo0, hi0) in run 0 (real
    // memory) and [lo1, hi1) in run 1
    int hi0 = 0, lo1 = 0, hi1 = 0;
    float lse2 = 0.f, dlt = 0.f;
    if (r < p.L) {
      const int M = p.mem_pad, Lc = p.chunk_tokens, t = r - M;
      if (KQ) {
        if (r < P) {           // real memory key: real memory and every target query
          hi0 = P;
          lo1 = M;
          hi1 = p.L;
        } else if (t >= 0) {   // target key of chunk c: queries of chunks c .. c + W
          const int c = t / Lc;
          lo1 = M + c * Lc;
          hi1 = min(p.L, M + (c + p.window + 1) * Lc);
        }
      } else {
        if (r < P || t >= 0) hi0 = P;  // real queries see the real memory
        if (t >= 0) {                  // target query of chunk c: keys of chunks c - W .. c
          const int c = t / Lc;
          lo1 = M + max(0, c - p.window) * Lc;
          hi1 = min(p.L, M + (c + 1) * Lc);
        }
        lse2 = -__ldg(p.LSE + (long long)bh * p.L + r) * kLog2e;  // negated, as the stages hold them
        dlt = -__ldg(p.delta + (long long)bh * p.L + r);
      }
    }
    const float sc = p.scale_log2;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarSFull + hf), (uint32_t)j & 1u, abort_flag, 6 + hf));
      if (!ok) break;
      tc_fence_after();
      const int c0 = tile_row(j) + hf * 64;  // first streamed row of this half
      const int lo = (j < u.n0 ? 0 : lo1) - c0, hi = (j < u.n0 ? hi0 : hi1) - c0;
      const float* ls = reinterpret_cast<const float*>(base + C::kStageOff + (j % C::kStages) * C::kStageBytes +
                                                       2 * C::kTileBytes) + hf * 64;
      const float* dl = ls + 128;
      // ls, dl (and lse2, dlt) hold -lse * log2(e) and -delta
      auto one = [&](uint32_t s, uint32_t dpv, int c, float& pv, float& dsv) {
        const bool vis = c >= lo && c < hi;
        const float nl2 = KQ ? ls[c] : lse2;
        const float nde = KQ ? dl[c] : dlt;
        pv = vis ? ex2(fmaf(__uint_as_float(s), sc, nl2)) : 0.f;
        dsv = pv * (__uint_as_float(dpv) + nde);
      };
      // every row of this warp sees all 64 columns of the half: no mask,
      // pairs of columns in packed fp32 arithmetic
      const bool whole = __all_sync(0xffffffffu, lo <= 0 && hi >= 64);
      const float2 sc2 = make_float2(sc, sc);
      // two passes of 32 columns (the packed results of a pass go over
      // columns its own loads have already read, so the passes never clash)
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        uint32_t sv[32], dv[32];
        tmem_ld32(tS + 32 * pass, sv);
        tmem_ld32(tdP + 32 * pass, dv);
        tmem_wait_ld();
        uint32_t pk[16], dk[16];
        if (whole) {
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {  // four columns: one 16-byte read of the stage's values
            float4 nl4, nd4;
            if (KQ) {
              nl4 = *reinterpret_cast<const float4*>(ls + 32 * pass + 4 * c4);
              nd4 = *reinterpret_cast<const float4*>(dl + 32 * pass + 4 * c4);
            } else {
              nl4 = make_float4(lse2, lse2, lse2, lse2);
              nd4 = make_float4(dlt, dlt, dlt, dlt);
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = 2 * c4 + e;
              const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), sc2,
                                          e ? make_float2(nl4.z, nl4.w) : make_float2(nl4.x, nl4.y));
              const float2 pv = make_float2(ex2(x.x), ex2(x.y));
              const float2 dd = __fadd2_rn(make_float2(__uint_as_float(dv[2 * c]), __uint_as_float(dv[2 * c + 1])),
                                           e ? make_float2(nd4.z, nd4.w) : make_float2(nd4.x, nd4.y));
              const float2 ds = __fmul2_rn(pv, dd);
              pk[c] = pack_bf16(pv.x, pv.y);
              dk[c] = pack_bf16(ds.x, ds.y);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            float pa, pb, da, db;
            one(sv[2 * c], dv[2 * c], 32 * pass + 2 * c, pa, da);
            one(sv[2 * c + 1], dv[2 * c + 1], 32 * pass + 2 * c + 1, pb, db);
            pk[c] = pack_bf16(pa, pb);
            dk[c] = pack_bf16(da, db);
          }
        }
        if (KQ) {
          tmem_st16(tS + 16 * pass, pk);   // P^T over S^T
          tmem_st16(tdP + 16 * pass, dk);  // dS^T over dP^T
        } else {
          tmem_st16(tS + 16 * pass, dk);   // dS over S
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::kBarPFull + hf));
    }
    // ------------------------------------------------------------ epilogue
    if (ok) ok = wait_bounded(bar(C::kBarFinal), 0, abort_flag, 8);
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);  // an abort anywhere in the CTA: no store
    if (ok) {  // warp-uniform: tcgen05.ld is warp-collective, rows past L only skip the store
      tc_fence_after();
      // key-tile kernel: half 0 writes the dV row, half 1 the dK row;
      // query-tile kernel: half h writes columns [h D/2, (h + 1) D/2) of dQ
      constexpr int kCols = KQ ? D : D / 2;
      const uint32_t src = tmem + lane_off + 256 + (KQ ? hf * D : hf * (D / 2));
      uint16_t* dst = (KQ ? (hf == 0 ? p.dV : p.dK) : p.dQ) + (((long long)b * p.L + r) * p.H + h) * D +
                      (KQ ? 0 : hf * (D / 2));
      const float mul = (KQ && hf == 0) ? 1.f : p.scale;  // dK, dQ carry the softmax scale
#pragma unroll
      for (int cc = 0; cc < kCols; cc += 32) {
        uint32_t o[32];
        if (nt > 0) {
          tmem_ld32(src + cc, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = 0u;
        }
        if (r >= p.L) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * mul, __uint_as_float(o[8 * v + 1]) * mul);
          w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * mul, __uint_as_float(o[8 * v + 3]) * mul);
          w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * mul, __uint_as_float(o[8 * v + 5]) * mul);
          w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * mul, __uint_as_float(o[8 * v + 7]) * mul);
          reinterpret_cast<uint4*>(dst + cc)[v] = w;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool KQ>
cudaError_t launch_bwd_impl(const BwdParams& p, cudaStream_t s) {
  using C = BwdCfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D, KQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.L + 127) / 128, p.B * p.H, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_bwd_kernel<D, KQ>, p);
}

// Self-test of the failure detection: one CTA waits, with the pipeline's own
// bounded wait, on an mbarrier that nothing ever completes.  The wait gives
// up after timeout_ns, records its site (bit 30) in the device error word and
// the kernel returns: no fault, no hang.
__global__ void wait_timeout_probe_kernel(uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar_;
  __shared__ int abort_;
  const uint32_t bar = smem_u32(&bar_);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    abort_ = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)wait_bounded(bar, 0, reinterpret_cast<volatile int*>(&abort_), kErrProbeSite, timeout_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_attention_backward(const BwdParams& p, cudaStream_t s) {
  const long long tokens = (long long)p.B * p.L;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((tokens + 7) / 8), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, bwd_delta_kernel, p);
  if (e != cudaSuccess) return e;
  if (p.D == 128) {
    e = launch_bwd_impl<128, true>(p, s);
    return e != cudaSuccess ? e : launch_bwd_impl<128, false>(p, s);
  }
  if (p.D == 64) {
    e = launch_bwd_impl<64, true>(p, s);
    return e != cudaSuccess ? e : launch_bwd_impl<64, false>(p, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_wait_timeout_probe(unsigned long long timeout_ns, cudaStream_t s) {
  wait_timeout_probe_kernel<<<1, 32, 0, s>>>(timeout_ns);
  return cudaGetLastError();
}

cudaError_t launch_chunk_attention_kh(const AttnParams& p, cudaStream_t s) {
  if (p.splits < 1 || p.splits > 65535 || (p.splits > 1 && (p.ws_o == nullptr || p.ws_lse == nullptr ||
                                                             p.ws_count == nullptr)))
    return cudaErrorInvalidValue;
  if (p.f8mma) return (p.fp8 && !p.k_int8 && p.D == 128) ? launch_kh_impl<128, true, true>(p, s) : cudaErrorInvalidValue;
  if (p.fp8 && p.D != 128) return cudaErrorInvalidValue;
  if (p.fp8) return p.k_int8 ? launch_kh_impl<128, true, false, true>(p, s) : launch_kh_impl<128, true, false, false>(p, s);
  if (p.D == 128) return launch_kh_impl<128, false>(p, s);
  if (p.D == 64) return launch_kh_impl<64, false>(p, s);
  return cudaErrorInvalidValue;
}

// Scratch of the allocation-free entry point: the split partials, partial
// LSEs and arrival counters of the workspace merge live in this file-scope
// array instead of caller-provided memory.  Every GPU that loads the library
// holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

cudaError_t noalloc_scratch(void** ptr, size_t* bytes) {
  // In host code the array's name is only a stand-in: the device address is
  // looked up with the device current and cached per device together with
  // the context it belongs to.  A call under another context (the primary
  // context was reset and re-created, which reloads the module) looks the
  // address up again; a lock keeps concurrent first calls from racing.
  constexpr int kMaxDevices = 64;
  struct Entry {
    CUcontext ctx;
    void* addr;
  };
  static std::mutex mu;
  static Entry cache[kMaxDevices] = {};
  static CtxGetCurrentFn get_ctx = nullptr;
  static bool get_ctx_tried = false;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!get_ctx_tried) {
    get_ctx_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_ctx = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  CUcontext ctx = nullptr;
  if (cache[dev].addr != nullptr && get_ctx != nullptr && get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  if (cache[dev].addr == nullptr || ctx != cache[dev].ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes the device's context current
    if (e != cudaSuccess) return e;
    CUcontext now = nullptr;
    if (get_ctx != nullptr && get_ctx(&now) != CUDA_SUCCESS) now = nullptr;
    cache[dev] = Entry{now, p};
  }
  *ptr = cache[dev].addr;
  *bytes = kNoAllocScratchBytes;
  return cudaSuccess;
}

unsigned int* device_error_word() {
  static unsigned int* ptr = nullptr;
  if (ptr == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_sab_error_word) == cudaSuccess) ptr = static_cast<unsigned int*>(a);
  }
  return ptr;
}

cudaError_t read_and_clear_device_error(unsigned int* value) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_sab_error_word, sizeof(v));
  if (e != cudaSuccess) return e;
  *value = v;
  if (v != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_sab_error_word, &zero, sizeof(zero));
  }
  return e;
}

}  // namespace sab
