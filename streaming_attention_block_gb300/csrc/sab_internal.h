// Internal interface between the host API (sab_api.cu) and the kernels.
// Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sab {

constexpr int kTileM = 128;    // query rows per tile (one TMEM lane per row)
constexpr int kTileN = 128;    // keys per KV tile
constexpr int kMaxSegments = 4;

// Device error word bits: bit k < 16, a bounded wait at site k gave up; bit
// 28, the bounded-wait self-test's wait gave up; bit 29, a split reported
// itself as aborted on request (self-test); bit 30, a debug-build index check
// failed; bit 31, a drain after an abort gave up.
constexpr unsigned kErrProbeSite = 28;
constexpr unsigned kErrInjectedAbortBit = 1u << 29;
constexpr unsigned kErrBoundsBit = 1u << 30;
#ifdef SAB_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

// One contiguous run of key rows inside one K/V source.
//   src 0: the layer's ring (rows along the [B,H,rows,D] row axis),
//   src 1: the current chunk passed in (token axis of [B,L,H,D]).
struct KvSegment {
  int src;
  int row0;    // first row of the run in the source's row axis
  int nrows;   // rows in the run
  int tile0;   // global index of the run's first 128-key tile
};

// kModeMemPrefix: block-causal target chunks behind a per-sample memory
// prefix of mem_pad positions, the first mem_len[b] of them real; the key
// runs of a query tile (memory, then the chunk window) are planned by each
// CTA on the device.
enum AttnMode : int { kModeStreaming = 0, kModeBlockCausal = 1, kModeMemPrefix = 2 };

// Key runs of one streaming call, in physical row order.
struct KeyPlan {
  int nseg;
  int total_tiles;
  KvSegment seg[kMaxSegments];
};

// Key set of chunk c ("WanToFight", table "模型组件", row "Rolling KV Cache";
// "Matrix-Game 4.0", section "前置知识 / 因果自回归与 KV 缓存"): the sink rows
// [0, Lc) when used, the ring chunks max(0, c - W) .. c - 1 (and c itself when
// the current chunk was appended first, kcur == 0) at rows
// (has_sink + chunk mod R) * Lc, physically adjacent runs merged (softmax does
// not depend on key order), then the current chunk's own tensor (kcur == 1).
// The host planner and the graph-mode kernels (chunk index read on the
// device) share this function.  At most R ring chunks are taken.
__host__ __device__ inline void plan_key_runs(long long c, int W, int R, int Lc, int has_sink, int use_sink,
                                              int kcur, KeyPlan& kp) {
  int r0[3], nr[3], n = 0;
  if (use_sink) {
    r0[n] = 0;
    nr[n] = Lc;
    ++n;
  }
  if (c < 0) c = 0;
  const long long lo = c - W > 0 ? c - W : 0;
  const long long hi = kcur ? c - 1 : c;
  if (hi >= lo && R > 0) {
    long long cnt = hi - lo + 1;
    if (cnt > R) cnt = R;
    const int s_lo = (int)(lo % R), s_end = s_lo + (int)cnt;
    const int base = has_sink * Lc;
    if (s_end <= R) {
      r0[n] = base + s_lo * Lc;
      nr[n] = (int)cnt * Lc;
      ++n;
    } else {  // wraps: the low slots come first in row order
      r0[n] = base;
      nr[n] = (s_end - R) * Lc;
      ++n;
      r0[n] = base + s_lo * Lc;
      nr[n] = (R - s_lo) * Lc;
      ++n;
    }
  }
  int tiles = 0, m = 0;
  for (int i = 0; i < n; ++i) {
    if (m > 0 && kp.seg[m - 1].row0 + kp.seg[m - 1].nrows == r0[i]) {
      tiles -= (kp.seg[m - 1].nrows + kTileN - 1) / kTileN;
      kp.seg[m - 1].nrows += nr[i];
      tiles += (kp.seg[m - 1].nrows + kTileN - 1) / kTileN;
    } else {
      kp.seg[m] = KvSegment{0, r0[i], nr[i], tiles};
      tiles += (nr[i] + kTileN - 1) / kTileN;
      ++m;
    }
  }
  if (kcur) {
    kp.seg[m] = KvSegment{1, 0, Lc, tiles};
    tiles += (Lc + kTileN - 1) / kTileN;
    ++m;
  }
  for (int i = m; i < kMaxSegments; ++i) kp.seg[i] = KvSegment{0, 0, 0, 0x7fffffff};
  kp.nseg = m;
  kp.total_tiles = tiles;
}

struct AttnParams {
  CUtensorMap q_map;      // dims (D, Lq, H, B), box (64, 128, 1, 1), SW128
  CUtensorMap k_map[2];   // per source, dims (D, rows, H, B)
  CUtensorMap v_map[2];
  CUtensorMap o_map;      // output, dims (D, Lq, H, B), box (64, 128, 1, 1), SW128
  int mode;
  int fp8;                // 1: the ring holds 8-bit codes (k_map[0]/v_map[0] are uint8 maps)
  int k_int8;             // with fp8: keys are INT8 codes (values stay E4M3)
  int f8mma;              // with fp8 (E4M3 keys and values): Q and P in E4M3, kind::f8f6f4 products
  const float* k_scale;   // FP8: [B*H][scale_stride] fp32 scales, index = ring row / chunk_tokens
  const float* v_scale;
  int scale_stride;
  int B, H, D;
  int Lq;                 // query rows per (b, h)
  int n_qtiles;           // ceil(Lq / 128)
  int splits;
  float scale_log2;       // softmax_scale * log2(e)
  // streaming: key runs planned on the host, or (d_chunk != null: graph mode)
  // planned by every CTA from the chunk index in device memory
  KeyPlan plan;
  const long long* d_chunk;
  int ring_slots, has_sink, use_sink, kcur;
  // block-causal (and memory prefix)
  int chunk_tokens;
  int window;
  int Lk;
  int mem_pad;            // memory positions ahead of the first target chunk
  const int* mem_len;     // device [B]: real memory positions per sample
  // outputs
  uint16_t* O;            // bf16 [B, Lq, H, D]
  float* LSE;             // [B, H, Lq] or null
  // failure-detection self-test: 0, or 1 + the index of a split that
  // reports itself at the workspace merge as if one of its waits had given up
  int inject_abort;
  // split workspace: tile t = (split * B*H + bh) * n_qtiles + query tile
  float* ws_o;            // [tiles][D / 4][128 rows] float4: normalised partial rows
  float* ws_lse;          // [tiles][128 rows]: partial LSEs
  unsigned int* ws_count; // [B*H][n_qtiles] arrival counters
  // debug-build index checks: rows of each key source's row axis, and the
  // partial tiles the workspace holds
  int src_rows[2];
  long long ws_tiles;
};

// FP8 append: per (b, h) block of one chunk.
struct AppendParams {
  const uint16_t* src[2];   // K, V token-major [B, Lc, H, D] bf16
  void* dst[2];             // ring K, V region base of the layer
  float* scale[2];          // FP8 only: ring K, V scale base of the layer
  int B, H, D, Lc;
  int rows;                 // rows per (b, h) in the ring
  int slot_row0;            // first row of the destination slot
  int scale_idx;            // (has_sink + slot) or 0 for the sink
  int scale_stride;         // has_sink + R
  int k_int8;               // 8-bit ring: K as INT8 (amax / 127) instead of E4M3
  // graph mode: the slot is chunk mod R with the chunk read on the device
  const long long* d_chunk;
  int ring_slots, has_sink;
  unsigned int* err_word;   // the library's device error word (debug-build index checks)
};

// Fused Q/K RMSNorm + rotary embedding of one chunk (token-major [B, Lc, H, D]).
struct RopeParams {
  const uint16_t* q_in;
  const uint16_t* k_in;
  const uint16_t* v_in;
  const float* gamma_q;     // [H*D] or null (1)
  const float* gamma_k;
  uint16_t* q_out;
  uint16_t* k_out;          // token-major K', or null
  uint16_t* v_out;          // token-major V copy, or null
  uint16_t* ring_k;         // BF16 ring K/V region of the layer, or null (no append)
  uint16_t* ring_v;
  int B, H, D, Lc;
  int rows;                 // ring rows per (b, h)
  int slot_row0;            // first ring row of the chunk's slot
  long long chunk;
  int F, Hp, Wp;            // latent grid of a chunk: Lc = F * Hp * Wp
  int bt, bh, bw;           // rotary bands of the head dimension (even, sum D)
  float log2_base;          // log2(rotary base)
  float eps;
  unsigned int* err_word;   // the library's device error word (debug-build index checks)
};

// Backward of block-causal attention (token-major [B, L, H, D] tensors).
struct BwdParams {
  CUtensorMap q_map, k_map, v_map, do_map;  // dims (D, L, H, B), box (64, 128, 1, 1), SW128
  CUtensorMap q_map_h, k_map_h, v_map_h, do_map_h;  // the same with 64-row boxes (streamed halves)
  const uint16_t* O;      // forward output
  const uint16_t* dO;
  const float* LSE;       // [B, H, L] natural-log LSE of the forward
  float* delta;           // [B, H, L] workspace: sum_d dO * O
  uint16_t* dQ;
  uint16_t* dK;
  uint16_t* dV;
  int B, H, D, L;
  int chunk_tokens, window;
  int mem_pad;            // memory prefix (0: plain block-causal), as in AttnParams
  const int* mem_len;     // device [B] (read only when mem_pad > 0)
  float scale;            // softmax scale
  float scale_log2;       // scale * log2(e)
};

// Launchers (return cudaError_t of the launch).
cudaError_t launch_append_bf16(const AppendParams& p, cudaStream_t s);
cudaError_t launch_append_fp8(const AppendParams& p, cudaStream_t s);
cudaError_t launch_counter_add(long long* counter, long long delta, cudaStream_t s);
cudaError_t launch_qk_rope(const RopeParams& p, cudaStream_t s);
cudaError_t launch_attention_backward(const BwdParams& p, cudaStream_t s);
cudaError_t launch_wait_timeout_probe(unsigned long long timeout_ns, cudaStream_t s);
// One query tile per CTA, key-half softmax warpgroups; unsplit KV only.
cudaError_t launch_chunk_attention_kh(const AttnParams& p, cudaStream_t s);
cudaError_t read_and_clear_device_error(unsigned int* value);
// Device address of the error word (for kernels of other translation units).
unsigned int* device_error_word();
// Device address and size of the library's own split-merge scratch.
cudaError_t noalloc_scratch(void** ptr, size_t* bytes);

}  // namespace sab
